/*
 * gdn_oracle.c -- CPU oracle for the gated delta rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, token-serial
 * definition that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg load it.  It shares no
 * code, header, table or helper with the CUDA path, and the CUDA path never
 * calls it.
 *
 * Everything is computed in double precision.  Inputs arrive as doubles that
 * the caller converted exactly from the activation dtype (fp16 and fp32 both
 * embed exactly in double); rounding to an output dtype is the caller's
 * business and happens once.
 *
 * Sources (page title, section):
 *  - "com.microsoft.GatedDeltaNet" README, Description: per value head,
 *    S_t = exp(g_t) S_{t-1} + k_t (beta_t (v_t - exp(g_t) S_{t-1}^T k_t))^T,
 *    o_t = scale * S_t^T q_t (state written key-major there).  Value head h
 *    reads query/key head h * Hq / Hv.
 *  - same page, Inputs table: cu_seqlens are exclusive prefix sums clamped to
 *    [0, total_tokens]; a decreasing entry yields an empty request; absent
 *    means uniform packing.  initial_state absent means zeros.
 *  - same page, Outputs table (final_state row): when a request is empty,
 *    its final state equals its initial state.
 *  - ONNX issue "Spec gap ... Gated DeltaNet-2", "What LinearAttention
 *    currently does": beta's last dimension is kv_num_heads or 1; with 1,
 *    one beta per token serves every value head.
 *  - "gatedDeltaUpdate": seq_lens [B] bounds the rows of a ragged prefill in
 *    the [B, T, ...] layout: request b takes the first seq_lens[b] tokens of
 *    its row (clamped to [0, row length]; the rest is padding, neither read
 *    nor written).
 *  - same page, Attributes: beta_activation (sigmoid in float), qk_l2_norm
 *    (eps 1e-12), scale (0 selects 1/sqrt(head_size_qk)), update_rule
 *    (linear drops decay and retrieval, gated keeps only decay, delta keeps
 *    only retrieval, gated_delta keeps both), gate_activation "qwen"
 *    (-exp(a_log) * softplus(decay + dt_bias)).
 *  - "aclnnRecurrentGatedDeltaRule", Formula: the value-major form
 *    S_t = alpha_t Diag(alpha_kt) S_{t-1} + beta_t (v_t - ... S_{t-1} k_t) k_t^T,
 *    o = S_t q_t / sqrt(d_k), with S in R^{dv x dk}.
 *  - "gatedDeltaUpdate" (CLIKA runtime): grouped heads, slot_ids addressing a
 *    state slab in place, the raw-gate arm gate_scale * softplus(g + gate_bias)
 *    with gate_bias [HV] or [HV, K] beside a per-head or per-key gate.
 *  - ONNX issue "Spec gap: LinearAttention (opset 27) cannot represent Gated
 *    DeltaNet-2 channel-wise erase gate", proposal (A): decay first, then the
 *    erase with retrieval key (b_t .* k_t) on the key side, then the write
 *    k_t v_t^T; the write gate w_t is folded into v by the caller.
 *  - same issue, proposal (B): the erase gate b_t is an input of its own,
 *    [T, Hv * dk], beside the scalar beta; with b_t = beta_t * 1 the update is
 *    gated_delta again.  Reading taken here: beta keeps the write role, so
 *    delta = beta (w .* v) - D S (b .* k); the write gate w_t of the first
 *    display of that issue may be passed in (w .* v formed here) instead of
 *    being folded into v by the caller.
 *  - "gatedDeltaUpdate": the state may be stored key-major, [B, HV, K, V]
 *    (slab [num_slots, HV, K, V]); the recurrence is the same, only the
 *    layout of initial_state and final_state changes.
 *
 * Storage here is value-major: M (dv x dk) is the transpose of the key-major
 * state of the first page, row i = value channel i, contiguous over dk.  With
 * that, per token (after the optional L2 norms and the gate):
 *     M    <- M * Diag(alpha)                 (decay; alpha = exp(g))
 *     u     = M kappa                         (retrieval; delta rules only)
 *     delta = beta (v - u)    (delta, gated_delta; GDN-2: v - u, beta == 1)
 *     delta = v               (linear, gated)
 *     M    <- M + delta k^T
 *     o     = scale * M q                     (readout of the updated state)
 * where kappa = k for the v1 rules and kappa = b .* k for GDN-2.  For GDN-2,
 * delta = beta (w .* v) - u, with beta == 1 when the erase gate rides in
 * beta (proposal A) and w == 1 when no write gate is passed.
 */
#include <tgmath.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* The arithmetic type.  The definition is the double build (parity); the same
 * source compiled with -DORACLE_REAL=float is a float instantiation that the
 * benchmark times beside it (tgmath.h sends exp, log1p and sqrt to the
 * function of the argument's type). */
#ifndef ORACLE_REAL
#define ORACLE_REAL double
#endif
typedef ORACLE_REAL real;

#define ORACLE_RULE_LINEAR 0
#define ORACLE_RULE_GATED 1
#define ORACLE_RULE_DELTA 2
#define ORACLE_RULE_GATED_DELTA 3
#define ORACLE_RULE_GDN2 4

#define ORACLE_ERR_BAD_SLOT 1

typedef struct {
    int32_t batch;         /* B */
    int32_t total_tokens;  /* T */
    int32_t hq, hv, dk, dv;
    int32_t rule;
    int32_t l2norm_q, l2norm_k;
    int32_t beta_sigmoid;  /* apply the logistic sigmoid to beta */
    int32_t decay_per_key; /* decay is [T, Hv, dk] instead of [T, Hv] */
    int32_t raw_gate;      /* decay holds the raw gate; gate_bias/gate_scale set */
    int32_t num_state_rows;
    int32_t threads;
    real scale;                /* 0 selects 1/sqrt(dk) */
    const real *q, *k, *v;     /* [T,Hq,dk], [T,Hq,dk], [T,Hv,dv] */
    const real *decay;         /* [T,Hv] or [T,Hv,dk] */
    const real *gate_bias;     /* [Hv] or [Hv,dk] (raw arm) */
    const real *gate_scale;    /* [Hv] (raw arm) */
    const real *beta;          /* [T,Hv]; GDN-2: [T,Hv,dk] */
    const int32_t *cu_seqlens;   /* [B+1] or NULL */
    const int32_t *slot_ids;     /* [B] or NULL */
    const real *initial_state; /* [rows,Hv,dv,dk] or NULL */
    real *final_state;         /* [rows,Hv,dv,dk] */
    real *o;                   /* [T,Hv,dv] */
    int32_t *error_word;         /* may be NULL */
    const int32_t *seq_lens;     /* [B] or NULL: rows of the uniform layout shortened */
    int32_t beta_shared;         /* scalar beta is [T]: one per token for every value head */
    int32_t state_kmajor;        /* states are [rows,Hv,dk,dv] (key-major) instead of [rows,Hv,dv,dk] */
    const real *erase_gate;    /* GDN-2 proposal (B): [T,Hv,dk]; beta is then scalar */
    const real *write_gate;    /* GDN-2: [T,Hv,dv] or NULL (w == 1) */
} oracle_problem;

/* softplus(x) = ln(1 + e^x), evaluated without overflow. */
static real softplus(real x) {
    return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

static real sigmoid(real x) { return 1.0 / (1.0 + exp(-x)); }

/* "com.microsoft.LinearAttentionGate", Description:
 * decay = decay_scale * softplus(a + dt_bias); beta = sigmoid(b) when asked.
 * a and b are [n, h] with the head axis last. */
int oracle_gate(int64_t n, int32_t h, const real *a, const real *dt_bias,
                const real *decay_scale, const real *b, real *decay_out,
                real *beta_out) {
    if (n < 0 || h <= 0 || !a || !dt_bias || !decay_scale || !decay_out) return 1;
    if (beta_out && !b) return 1;
    for (int64_t i = 0; i < n; ++i) {
        for (int32_t j = 0; j < h; ++j) {
            int64_t e = i * h + j;
            decay_out[e] = decay_scale[j] * softplus(a[e] + dt_bias[j]);
            if (beta_out) beta_out[e] = sigmoid(b[e]);
        }
    }
    return 0;
}

static int32_t clamp_i32(int32_t x, int32_t lo, int32_t hi) {
    return x < lo ? lo : (x > hi ? hi : x);
}

/* Token range of request b: clamped exclusive prefix sums, or uniform rows,
 * each shortened to its clamped seq_lens entry when those are given. */
static void request_range(const oracle_problem *p, int32_t b, int32_t *t0, int32_t *t1) {
    if (p->cu_seqlens) {
        *t0 = clamp_i32(p->cu_seqlens[b], 0, p->total_tokens);
        *t1 = clamp_i32(p->cu_seqlens[b + 1], 0, p->total_tokens);
        if (*t1 < *t0) *t1 = *t0; /* decreasing entry: empty request */
    } else {
        int32_t len = p->total_tokens / p->batch;
        *t0 = b * len;
        *t1 = *t0 + (p->seq_lens ? clamp_i32(p->seq_lens[b], 0, len) : len);
    }
}

static void l2_normalise(real *x, int32_t n) {
    real ss = 0.0;
    for (int32_t i = 0; i < n; ++i) ss += x[i] * x[i];
    real inv = 1.0 / sqrt(ss + 1e-12);
    for (int32_t i = 0; i < n; ++i) x[i] *= inv;
}

static int rule_has_decay(int32_t r) {
    return r == ORACLE_RULE_GATED || r == ORACLE_RULE_GATED_DELTA || r == ORACLE_RULE_GDN2;
}
static int rule_has_retrieval(int32_t r) {
    return r == ORACLE_RULE_DELTA || r == ORACLE_RULE_GATED_DELTA || r == ORACLE_RULE_GDN2;
}

/* One (request, value head) pair, token by token. */
static void run_pair(const oracle_problem *p, int32_t b, int32_t h, real *work) {
    const int32_t dk = p->dk, dv = p->dv, hq = p->hq, hv = p->hv;
    const int32_t qh = (int32_t)((int64_t)h * hq / hv); /* grouped heads */
    const int32_t row = p->slot_ids ? p->slot_ids[b] : b;
    if (row < 0 || row >= p->num_state_rows) {
        if (p->error_word) {
#pragma omp atomic
            *p->error_word |= ORACLE_ERR_BAD_SLOT;
        }
        return;
    }
    real *M = work;                 /* dv * dk */
    real *kv = M + (size_t)dv * dk; /* dk */
    real *qv = kv + dk;             /* dk */
    real *alpha = qv + dk;          /* dk */
    real *kappa = alpha + dk;       /* dk */
    real *u = kappa + dk;           /* dv */
    real *delta = u + dv;           /* dv */

    const size_t state_off = (((size_t)row * hv) + h) * (size_t)dv * dk;
    if (!p->initial_state)
        memset(M, 0, sizeof(real) * (size_t)dv * dk);
    else if (p->state_kmajor) /* stored [dk][dv]: element (i, c) of M at c * dv + i */
        for (int32_t i = 0; i < dv; ++i)
            for (int32_t c = 0; c < dk; ++c) M[(size_t)i * dk + c] = p->initial_state[state_off + (size_t)c * dv + i];
    else
        memcpy(M, p->initial_state + state_off, sizeof(real) * (size_t)dv * dk);

    const real scale = p->scale != 0.0 ? p->scale : 1.0 / sqrt((real)dk);
    int32_t t0, t1;
    request_range(p, b, &t0, &t1);

    for (int32_t t = t0; t < t1; ++t) {
        const real *kin = p->k + ((size_t)t * hq + qh) * dk;
        const real *qin = p->q + ((size_t)t * hq + qh) * dk;
        const real *vin = p->v + ((size_t)t * hv + h) * dv;
        memcpy(kv, kin, sizeof(real) * dk);
        memcpy(qv, qin, sizeof(real) * dk);
        if (p->l2norm_k) l2_normalise(kv, dk);
        if (p->l2norm_q) l2_normalise(qv, dk);

        /* decay: alpha_c = exp(g_c); scalar decay broadcasts over c */
        if (rule_has_decay(p->rule)) {
            for (int32_t c = 0; c < dk; ++c) {
                real g;
                if (p->decay_per_key) {
                    real raw = p->decay[((size_t)t * hv + h) * dk + c];
                    g = p->raw_gate ? p->gate_scale[h] * softplus(raw + p->gate_bias[(size_t)h * dk + c])
                                    : raw;
                } else {
                    real raw = p->decay[(size_t)t * hv + h];
                    g = p->raw_gate ? p->gate_scale[h] * softplus(raw + p->gate_bias[h]) : raw;
                }
                alpha[c] = exp(g);
            }
            for (int32_t i = 0; i < dv; ++i)
                for (int32_t c = 0; c < dk; ++c) M[(size_t)i * dk + c] *= alpha[c];
        }

        if (p->rule == ORACLE_RULE_GDN2) {
            /* erase gate b: its own input (proposal B, taken as given) or the
             * per-key beta (proposal A, through the sigmoid when asked) */
            for (int32_t c = 0; c < dk; ++c) {
                real bc;
                if (p->erase_gate) {
                    bc = p->erase_gate[((size_t)t * hv + h) * dk + c];
                } else {
                    bc = p->beta[((size_t)t * hv + h) * dk + c];
                    if (p->beta_sigmoid) bc = sigmoid(bc);
                }
                kappa[c] = bc * kv[c];
            }
            /* the write's scalar: beta under proposal B, 1 under proposal A */
            real beta = 1.0;
            if (p->erase_gate) {
                beta = p->beta[p->beta_shared ? (size_t)t : (size_t)t * hv + h];
                if (p->beta_sigmoid) beta = sigmoid(beta);
            }
            for (int32_t i = 0; i < dv; ++i) {
                real s = 0.0;
                for (int32_t c = 0; c < dk; ++c) s += M[(size_t)i * dk + c] * kappa[c];
                u[i] = s;
            }
            for (int32_t i = 0; i < dv; ++i) {
                const real w = p->write_gate ? p->write_gate[((size_t)t * hv + h) * dv + i] : 1.0;
                delta[i] = beta * (w * vin[i]) - u[i];
            }
        } else if (rule_has_retrieval(p->rule)) {
            real beta = p->beta[p->beta_shared ? (size_t)t : (size_t)t * hv + h];
            if (p->beta_sigmoid) beta = sigmoid(beta);
            memcpy(kappa, kv, sizeof(real) * dk);
            for (int32_t i = 0; i < dv; ++i) {
                real s = 0.0;
                for (int32_t c = 0; c < dk; ++c) s += M[(size_t)i * dk + c] * kappa[c];
                u[i] = s;
            }
            for (int32_t i = 0; i < dv; ++i) delta[i] = beta * (vin[i] - u[i]);
        } else {
            memcpy(delta, vin, sizeof(real) * dv);
        }

        for (int32_t i = 0; i < dv; ++i)
            for (int32_t c = 0; c < dk; ++c) M[(size_t)i * dk + c] += delta[i] * kv[c];

        real *out = p->o + ((size_t)t * hv + h) * dv;
        for (int32_t i = 0; i < dv; ++i) {
            real s = 0.0;
            for (int32_t c = 0; c < dk; ++c) s += M[(size_t)i * dk + c] * qv[c];
            out[i] = scale * s;
        }
    }
    if (p->state_kmajor)
        for (int32_t i = 0; i < dv; ++i)
            for (int32_t c = 0; c < dk; ++c) p->final_state[state_off + (size_t)c * dv + i] = M[(size_t)i * dk + c];
    else
        memcpy(p->final_state + state_off, M, sizeof(real) * (size_t)dv * dk);
}

/* Runs every (request, value head) pair.  Returns 0, or 1 on bad arguments. */
int oracle_gdn(const oracle_problem *p) {
    if (!p || p->batch <= 0 || p->total_tokens < 0 || p->hq <= 0 || p->hv <= 0 ||
        p->dk <= 0 || p->dv <= 0 || p->hv % p->hq != 0)
        return 1;
    if (!p->q || !p->k || !p->v || !p->o || !p->final_state) return 1;
    if (rule_has_decay(p->rule) && !p->decay) return 1;
    if (rule_has_retrieval(p->rule) && !p->beta) return 1;
    if (p->raw_gate && (!p->gate_bias || !p->gate_scale)) return 1;
    if (!p->cu_seqlens && p->total_tokens % p->batch != 0) return 1;
    if (p->cu_seqlens && p->seq_lens) return 1;
    if (p->beta_shared && p->rule != ORACLE_RULE_DELTA && p->rule != ORACLE_RULE_GATED_DELTA &&
        !(p->rule == ORACLE_RULE_GDN2 && p->erase_gate))
        return 1;
    if ((p->erase_gate || p->write_gate) && p->rule != ORACLE_RULE_GDN2) return 1;

    const int64_t pairs = (int64_t)p->batch * p->hv;
    const size_t per = (size_t)p->dv * p->dk + 4 * (size_t)p->dk + 2 * (size_t)p->dv;
    int nthreads = p->threads > 0 ? p->threads : 1;
    real *work = (real *)malloc(sizeof(real) * per * (size_t)nthreads);
    if (!work) return 2;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t i = 0; i < pairs; ++i) {
#ifdef _OPENMP
        int tid = omp_get_thread_num();
#else
        int tid = 0;
#endif
        run_pair(p, (int32_t)(i / p->hv), (int32_t)(i % p->hv), work + per * (size_t)tid);
    }
    free(work);
    return 0;
}
