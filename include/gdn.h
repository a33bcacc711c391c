/*
 * gdn.h -- C ABI of the gated delta rule library (libgdn.so, sm_103a).
 *
 * The operation (value-major storage; S is dv x dk fp32 per value head):
 *
 *   per token t of a request, for each value head h (query/key head
 *   qh = h * Hq / Hv):
 *     alpha = exp(g_t)                      (scalar, or a dk-vector per key)
 *     S     = S * Diag(alpha)               (decay; rules gated, gated_delta, gdn2)
 *     u     = S kappa                       (retrieval; rules delta, gated_delta, gdn2)
 *     d     = beta_t (v_t - u)              (delta, gated_delta)
 *     d     = beta_t (w_t .* v_t) - u       (gdn2; kappa = b_t .* k_t; beta_t = 1
 *                                            when the erase gate rides in beta,
 *                                            w_t = 1 without a write gate)
 *     d     = v_t                           (linear, gated)
 *     S     = S + d k_t^T
 *     o_t   = scale * S q_t
 *
 * Sources: "com.microsoft.GatedDeltaNet" README (Description, Inputs,
 * Outputs, Attributes); "com.microsoft.LinearAttentionGate" (Description);
 * "aclnnRecurrentGatedDeltaRule" (Formula; two-phase workspace query);
 * "gatedDeltaUpdate" (CLIKA runtime: slot_ids slab, raw-gate arm, per-key
 * gate, key-major state slab); ONNX issue "Spec gap: LinearAttention
 * (opset 27) cannot represent Gated DeltaNet-2 channel-wise erase gate"
 * (proposals A and B, and the write gate of its first display).
 *
 * Conventions for every entry point:
 *  - Every tensor pointer is DEVICE memory owned by the caller, row-major and
 *    contiguous in the layout stated, aligned at least to its element size.
 *    The library allocates no device memory and keeps no pointer after the
 *    call returns.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and runs asynchronously: no entry point synchronises.  Inputs
 *    must stay valid and outputs must not be read until the stream reaches
 *    the work.
 *  - Arguments are validated on the host before anything is launched; a
 *    non-OK status means nothing was enqueued and no output was touched.
 *    gdn_last_error_message() then describes the first failed check.
 *  - All entry points are thread-safe (the message is thread-local).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *gdn_stream;

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID = 1,     /* the arguments break the op contract */
    GDN_ERR_UNSUPPORTED = 2, /* a valid request this library declines (typed) */
    GDN_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned */
    GDN_ERR_CUDA = 4         /* a CUDA launch or runtime call failed */
} gdn_status;

typedef enum gdn_dtype {
    GDN_DTYPE_F32 = 0,
    GDN_DTYPE_F16 = 1,
    GDN_DTYPE_BF16 = 2 /* named so it can be declined: GDN_ERR_UNSUPPORTED */
} gdn_dtype;

/* "com.microsoft.GatedDeltaNet", Attributes, update_rule; GDN2 is the rule
 * of the ONNX "Spec gap ... Gated DeltaNet-2" issue (its erase gate in beta,
 * proposal A, or in erase_gate, proposal B). */
typedef enum gdn_rule {
    GDN_RULE_LINEAR = 0,      /* no decay, no retrieval: S += v k^T */
    GDN_RULE_GATED = 1,       /* decay only */
    GDN_RULE_DELTA = 2,       /* retrieval only */
    GDN_RULE_GATED_DELTA = 3, /* both (the default of the op) */
    GDN_RULE_GDN2 = 4         /* decay, then erase with kappa = b .* k, write k v^T */
} gdn_rule;

/* Flags (gdn_problem.flags). */
#define GDN_FLAG_L2NORM_Q 0x1u      /* q <- q / sqrt(sum q^2 + 1e-12) first (qk_l2_norm) */
#define GDN_FLAG_L2NORM_K 0x2u      /* same for k */
#define GDN_FLAG_BETA_SIGMOID 0x4u  /* beta <- sigmoid(beta) in fp32 (beta_activation) */
#define GDN_FLAG_DECAY_PER_KEY 0x8u /* decay is [.., Hv, dk]: one log-decay per key channel */
#define GDN_FLAG_BETA_SHARED 0x10u  /* beta is [total_tokens]: one per token, shared by every value head */
#define GDN_FLAG_STATE_KMAJOR 0x20u /* states are key-major [num_state_rows, Hv, dk, dv] ("gatedDeltaUpdate") */

/* Bits OR-ed into *error_word by the device (never reset by the library). */
#define GDN_DEVERR_BAD_SLOT 0x1 /* a slot id outside [0, num_state_rows): request skipped */
#define GDN_DEVERR_TIMEOUT 0x2  /* a bounded wait on an asynchronous copy ran out: the CTA gave up */
#define GDN_DEVERR_OVERLAP 0x4  /* chunked prefill: the requests' chunks outgrew the workspace, which only
                                   requests sharing tokens can do; the requests past it were skipped */
#define GDN_DEVERR_DECAY_RANGE 0x8 /* chunked prefill, per-key decay on the tensor cores: a log decay above 0
                                      (a decay above 1) was given; that path needs decays in (0, 1] and the
                                      results of the chunks concerned are not valid */

/*
 * One call of the recurrence over a batch of requests.
 *
 * Token layout.  Rank-3 packed form (seq_len == 0): q, k are
 * [total_tokens, Hq, dk], v and o are [total_tokens, Hv, dv].  Request b owns
 * tokens [clamp(cu_seqlens[b]), clamp(cu_seqlens[b+1])), each clamped to
 * [0, total_tokens]; a decreasing pair gives an empty request (GatedDeltaNet
 * Inputs table, cu_seqlens).  cu_seqlens NULL means uniform packing:
 * total_tokens / batch tokens each (total_tokens must divide).  Output tokens
 * that no request covers are not written.
 * Rank-4 form (seq_len > 0): q, k are [batch, seq_len, Hq, dk] (the same
 * memory layout), total_tokens must equal batch * seq_len, and cu_seqlens must
 * be NULL (the op allows cu_seqlens with the rank-3 spelling only).  seq_lens
 * (rank-4 form only; "gatedDeltaUpdate", seq_lens bounds the rows of a ragged
 * prefill) makes the batch padded-ragged: request b owns the first
 * clamp(seq_lens[b], 0, seq_len) tokens of its row, [b * seq_len,
 * b * seq_len + that); the padding tokens take no part in any result and
 * are not written (their contents may be anything, NaN included).
 * seq_lens NULL means every row is full.
 *
 * Heads.  num_heads_v is a positive multiple of num_heads_q; value head h
 * reads query/key head h * Hq / Hv.
 *
 * Gate (decay).  Present exactly for rules GATED, GATED_DELTA and GDN2.
 *  - gate_bias == gate_scale == NULL: `decay` is the log-space decay g.
 *  - both non-NULL (raw-gate arm, gatedDeltaUpdate): `decay` is the raw gate
 *    projection and g = gate_scale[h] * softplus(decay + gate_bias) is formed
 *    in fp32 inside the kernel.  gate_bias is [Hv] (or [Hv, dk] with
 *    GDN_FLAG_DECAY_PER_KEY), gate_scale is [Hv] (the folded -exp(A_log)).
 *  - exactly one of them non-NULL: GDN_ERR_INVALID.
 *  decay is [total_tokens, Hv], or [total_tokens, Hv, dk] with
 *  GDN_FLAG_DECAY_PER_KEY; decay_dtype is F32 or act_dtype.
 *
 * Beta.  Present exactly for rules DELTA, GATED_DELTA (shape [total_tokens,
 * Hv], or [total_tokens] with GDN_FLAG_BETA_SHARED: beta's last dimension 1,
 * broadcast over the value heads, as the LinearAttention schema allows) and
 * GDN2 (the erase gate b, [total_tokens, Hv, dk], when erase_gate is NULL;
 * GDN_FLAG_BETA_SHARED is then rejected); beta_dtype is F32 or act_dtype;
 * GDN_FLAG_BETA_SIGMOID applies the logistic sigmoid first.
 *
 * GDN2 gates (ONNX GDN-2 issue).  erase_gate (proposal B) is the erase gate b
 * as an input of its own, fp32 [total_tokens, Hv, dk], taken as given (no
 * activation); beta is then the scalar write rate of DELTA / GATED_DELTA
 * ([total_tokens, Hv], or [total_tokens] with GDN_FLAG_BETA_SHARED; the
 * sigmoid flag applies to it), so erase_gate = beta * 1 gives GATED_DELTA.
 * write_gate is the write gate w, fp32 [total_tokens, Hv, dv], multiplied
 * into v inside the kernels (NULL: w = 1, or already folded into v by the
 * caller).  Both are GDN2 only (GDN_ERR_INVALID otherwise).
 *
 * State.  initial_state and final_state are fp32, value-major
 * [num_state_rows, Hv, dv, dk], or key-major [num_state_rows, Hv, dk, dv]
 * with GDN_FLAG_STATE_KMAJOR (the slab layout of "gatedDeltaUpdate"; the
 * recurrence is the same).  Request b reads and writes row
 * slot_ids[b] if slot_ids is non-NULL (the slab of gatedDeltaUpdate), else
 * row b.  initial_state NULL means a zero state.  final_state may equal
 * initial_state (in-place update); otherwise the two must not overlap.  Rows
 * no request names are not touched.  An empty request leaves its final
 * state equal to its initial state ("com.microsoft.GatedDeltaNet",
 * Outputs).  Slot ids must be distinct (caller's contract); a slot id outside [0, num_state_rows) makes every CTA of that request skip it
 * and OR GDN_DEVERR_BAD_SLOT into *error_word (if error_word is non-NULL).
 *
 * scale == 0 selects 1/sqrt(dk).  state_update_capacity must be 0 (compact
 * transition capture is not part of this library).
 */
typedef struct gdn_problem {
    int32_t batch;          /* B: number of requests (0: nothing to do) */
    int32_t total_tokens;   /* T */
    int32_t seq_len;        /* 0: rank-3 packed; > 0: rank-4 uniform */
    int32_t num_heads_q;    /* Hq */
    int32_t num_heads_v;    /* Hv */
    int32_t head_dim_k;     /* dk */
    int32_t head_dim_v;     /* dv */
    int32_t num_state_rows; /* rows of the state tensors; 0 means batch */
    int32_t act_dtype;      /* gdn_dtype of q, k, v, o: F32 or F16 */
    int32_t decay_dtype;    /* gdn_dtype of decay: F32 or act_dtype */
    int32_t beta_dtype;     /* gdn_dtype of beta: F32 or act_dtype */
    int32_t rule;           /* gdn_rule */
    uint32_t flags;         /* GDN_FLAG_* */
    float scale;            /* 0: 1/sqrt(dk) */
    int32_t state_update_capacity; /* must be 0 */
    const void *q;
    const void *k;
    const void *v;
    void *o;
    const void *decay;
    const float *gate_bias;
    const float *gate_scale;
    const void *beta;
    const int32_t *cu_seqlens; /* [batch + 1] or NULL */
    const int32_t *slot_ids;   /* [batch] or NULL */
    const float *initial_state;
    float *final_state;
    int32_t *error_word; /* optional device int32 */
    const int32_t *seq_lens; /* [batch] or NULL: rank-4 form only (see Token layout) */
    const float *erase_gate; /* GDN2 only: [total_tokens, Hv, dk] fp32, or NULL (see GDN2 gates) */
    const float *write_gate; /* GDN2 only: [total_tokens, Hv, dv] fp32, or NULL (see GDN2 gates) */
} gdn_problem;

/*
 * gdn_gate -- "com.microsoft.LinearAttentionGate", Description:
 *   decay = decay_scale * softplus(a + dt_bias)   and, if beta_out != NULL,
 *   beta  = sigmoid(b).
 * a (and b) are [n, heads]: any leading axes folded into n, heads last.
 * dt_bias and decay_scale are fp32 [heads].  a, b, decay_out and beta_out
 * share `dtype` (F32 or F16).  Arithmetic is fp32, rounded once on store.
 * beta_out requires b (GDN_ERR_INVALID otherwise); b without beta_out is
 * accepted and unused.  n == 0 is a no-op.
 */
typedef struct gdn_gate_args {
    int64_t n;
    int32_t heads;
    int32_t dtype;
    const void *a;
    const float *dt_bias;
    const float *decay_scale;
    const void *b;
    void *decay_out;
    void *beta_out;
} gdn_gate_args;

gdn_status gdn_gate(const gdn_gate_args *args, gdn_stream stream);

/*
 * gdn_recurrent_step -- token-serial recurrence ("aclnnRecurrentGatedDeltaRule":
 * the variable-step-size form, designed for L_i <= 8 tokens per request, the
 * decode / multi-token-prediction step).  Any request length is accepted;
 * time grows linearly with the longest request.  Supports every rule, both
 * gate arms, per-key decay, GDN2, 1 <= dk, dv <= 256 (larger:
 * GDN_ERR_UNSUPPORTED).  fp32 arithmetic throughout; the state tile of each
 * (request, value head) crosses HBM once each way.
 */
gdn_status gdn_recurrent_step(const gdn_problem *p, gdn_stream stream);

/*
 * gdn_chunked_prefill_workspace_size -- bytes of device workspace that
 * gdn_chunked_prefill needs for this problem and chunk size (the first phase
 * of the two-phase style of "aclnnRecurrentGatedDeltaRule").  Returns 0 when
 * no workspace is needed, and (size_t)-1 when the problem is rejected (the
 * reason is then in gdn_last_error_message()).
 */
size_t gdn_chunked_prefill_workspace_size(const gdn_problem *p, int32_t chunk_size);

/*
 * gdn_chunked_prefill_workspace_size_min -- the least workspace
 * gdn_chunked_prefill accepts for this problem (0, (size_t)-1 as above).  It
 * holds one chunk of every request at a time, so it does not grow with the
 * request lengths (the fp32-activation and fp16-gate copies aside).  With any
 * workspace from this size up to gdn_chunked_prefill_workspace_size() the call
 * runs in windows of as many chunks per request as fit, one after another on
 * the stream: each window reads the state the previous one left in
 * final_state (fp32, so the result is the same, bit for bit, as a single pass)
 * and writes its tokens' outputs.  Not an operation of the pages: a bound on
 * the library's own scratch ("aclnnRecurrentGatedDeltaRule" asks for its
 * workspace in a first phase; this is the least of it).
 */
size_t gdn_chunked_prefill_workspace_size_min(const gdn_problem *p, int32_t chunk_size);

/*
 * gdn_chunked_prefill -- the same result as gdn_recurrent_step, computed
 * chunk-parallel: within a chunk the delta rule becomes a unit-lower-
 * triangular system solved once per chunk, and the intra-chunk attention and
 * the state carry-in/carry-out become dense fp16 tensor-core products with
 * fp32 accumulation; the state itself stays fp32 across chunks.
 * ("com.microsoft.GatedDeltaNet", Attributes, chunk_size: any value is
 * accepted and none changes the result beyond rounding; <= 0 selects 64.)
 * Extra constraints (GDN_ERR_UNSUPPORTED otherwise): dk in {16, 32, 64, 128},
 * dv a multiple of 16 (<= 256), q, k, v, o and the state 16-byte aligned.
 * fp32 activations are rounded to fp16 for the products (at dk = dv = 128
 * through fp16 copies of q, k and v that the library writes into the
 * workspace; o is still written in fp32).  Per-key decay (gated, gated_delta)
 * and GDN2 run on the tensor cores when dk = dv = 128 and the per-key gate
 * rows are 16-byte aligned (fp16 per-key log decays, and GDN2's fp16 per-key
 * beta, through fp32 copies that the library writes into the workspace);
 * per-key log decays are expected <= 0 there (decays in (0, 1], as the
 * raw-gate arm always gives).  Per-key problems at other head sizes run the
 * token-serial form (same result).
 *
 * Workspace: owned by the caller, device memory of at least
 * gdn_chunked_prefill_workspace_size_min() bytes, 256-byte aligned (NULL
 * allowed when that is 0); GDN_ERR_WORKSPACE otherwise.  Below
 * gdn_chunked_prefill_workspace_size() the call runs in windows (see
 * gdn_chunked_prefill_workspace_size_min).  It is non-zero whenever the
 * tensor-core path runs (every rule with dk = dv = 128, per-key problems as
 * above), and 0 otherwise.  Layout, for T / 64 + B + 1 chunk slots:
 * per-request chunk offsets, a chunk-slot -> request table and the requests
 * ordered by length (rounded up to 1 KB); then one 88 KB image per (chunk
 * slot, value head) of the chunk's state-independent operands (fp16); with
 * fp32 activations, the fp16 copies of q, k and v (each rounded up to 256
 * bytes); last, fp32 copies [total_tokens, Hv, 128] of fp16 per-key gate rows
 * (the log decay; GDN2's per-key beta), each rounded up to 256 bytes.
 * Its contents are scratch, rewritten by every call on the stream; two calls
 * in flight at once need two workspaces.  Requests that share tokens can need
 * more slots than that; the ones past the capacity are skipped and
 * GDN_DEVERR_OVERLAP is set.
 */
gdn_status gdn_chunked_prefill(const gdn_problem *p, int32_t chunk_size, void *workspace,
                               size_t workspace_bytes, gdn_stream stream);

/*
 * gdn_chunked_prefill_noalloc -- gdn_chunked_prefill with the library's own
 * scratch instead of a caller workspace.  None of the reference pages has a
 * counterpart of this entry point; it exists for callers that cannot allocate
 * device memory around the call.
 *
 * The scratch is one static device array of 768 MiB per device (set aside
 * when libgdn loads; this entry point allocates nothing).  Each process that
 * loads libgdn reserves its own 768 MiB on every device it uses, so calls
 * from different processes never share it.  Problems whose
 * gdn_chunked_prefill_workspace_size() exceeds it are rejected on the host
 * with GDN_ERR_WORKSPACE before anything is enqueued (the long and ragged
 * prefill configurations, about 745-765 MB, fit).  Within a process, every
 * call on a device shares the array: two calls in flight at the same time on
 * that device (different streams or threads) race on it, so the caller
 * serialises them.  Every call looks the array's address up on the current
 * device (cudaGetSymbolAddress), so the address stays right after a device
 * reset; the first call on each device also sets kernel attributes: make it
 * outside any stream capture.  Same arguments, constraints, results and
 * error bits as gdn_chunked_prefill.
 */
gdn_status gdn_chunked_prefill_noalloc(const gdn_problem *p, int32_t chunk_size, gdn_stream stream);

/* Static description of a status code ("ok", "invalid argument", ...). */
const char *gdn_status_string(gdn_status status);

/* Detail of the most recent non-OK status returned on this thread ("" if none). */
const char *gdn_last_error_message(void);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* GDN_H_ */
