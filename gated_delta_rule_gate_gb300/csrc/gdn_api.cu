// gdn_api.cu -- the C ABI of libgdn: host-side validation and kernel dispatch.
//
// Every check runs before anything is enqueued, so a rejected call touches
// no memory.  The rules come from the op contracts: "com.microsoft.GatedDeltaNet"
// (Inputs: decay present exactly for gated rules, beta exactly for delta
// rules, cu_seqlens only with the rank-3 spelling; Attributes:
// state_update_capacity 0 only; Type constraints: fp32/fp16, no bf16),
// "com.microsoft.LinearAttentionGate" (beta requires b) and
// "gatedDeltaUpdate" (Hv a multiple of Hq; gate_bias and gate_scale together
// or not at all).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/gdn.h"
#include "launch.h"

namespace {

thread_local char g_msg[512] = "";

gdn_status fail(gdn_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

gdn_status ok() {
    g_msg[0] = '\0';
    return GDN_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Library-owned scratch of gdn_chunked_prefill_noalloc: one per device, set
// aside when the module loads, so that entry point allocates nothing.  Every
// call on a device shares it (see the header).
constexpr size_t kNoAllocBytes = (size_t)768 << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Its address on the current device, looked up on every call: after a
// device reset the module is loaded again and the array may move, so a
// cached address could be stale.
cudaError_t noalloc_scratch(void **ptr) {
    *ptr = nullptr;
    return cudaGetSymbolAddress(ptr, g_noalloc_scratch);
}

size_t dtype_size(int dt) { return dt == GDN_DTYPE_F16 || dt == GDN_DTYPE_BF16 ? 2 : 4; }

gdn_status check_dtype(int dt, const char *what) {
    if (dt == GDN_DTYPE_BF16) return fail(GDN_ERR_UNSUPPORTED, "%s: bfloat16 is not implemented", what);
    if (dt != GDN_DTYPE_F32 && dt != GDN_DTYPE_F16)
        return fail(GDN_ERR_INVALID, "%s: unknown dtype %d", what, dt);
    return GDN_OK;
}

// Validates a problem and fills the device-side description.
gdn_status validate(const gdn_problem *p, gdn::Problem *out) {
    if (!p) return fail(GDN_ERR_INVALID, "problem is NULL");
    if (p->batch < 0) return fail(GDN_ERR_INVALID, "batch must be >= 0 (got %d)", p->batch);
    if (p->total_tokens < 0) return fail(GDN_ERR_INVALID, "total_tokens must be >= 0");
    if (p->num_heads_q <= 0 || p->num_heads_v <= 0)
        return fail(GDN_ERR_INVALID, "head counts must be positive (Hq=%d, Hv=%d)", p->num_heads_q,
                    p->num_heads_v);
    if (p->num_heads_v % p->num_heads_q != 0)
        return fail(GDN_ERR_INVALID, "num_heads_v (%d) must be a multiple of num_heads_q (%d)",
                    p->num_heads_v, p->num_heads_q);
    if (p->head_dim_k <= 0 || p->head_dim_v <= 0)
        return fail(GDN_ERR_INVALID, "head sizes must be positive (dk=%d, dv=%d)", p->head_dim_k,
                    p->head_dim_v);
    if (p->head_dim_k > 256 || p->head_dim_v > 256)
        return fail(GDN_ERR_UNSUPPORTED, "head sizes above 256 are not supported (dk=%d, dv=%d)",
                    p->head_dim_k, p->head_dim_v);
    gdn_status st;
    if ((st = check_dtype(p->act_dtype, "act_dtype")) != GDN_OK) return st;
    if (p->rule < GDN_RULE_LINEAR || p->rule > GDN_RULE_GDN2)
        return fail(GDN_ERR_INVALID, "unknown update rule %d", p->rule);
    static_assert(GDN_FLAG_L2NORM_Q == gdn::kL2q && GDN_FLAG_L2NORM_K == gdn::kL2k &&
                      GDN_FLAG_BETA_SIGMOID == gdn::kBetaSigmoid && GDN_FLAG_DECAY_PER_KEY == gdn::kPerKey &&
                      GDN_FLAG_BETA_SHARED == gdn::kBetaShared && GDN_FLAG_STATE_KMAJOR == gdn::kKMajor,
                  "flag mirror");
    static_assert(GDN_DEVERR_BAD_SLOT == gdn::kErrBadSlot && GDN_DEVERR_TIMEOUT == gdn::kErrTimeout &&
                      GDN_DEVERR_OVERLAP == gdn::kErrOverlap && GDN_DEVERR_DECAY_RANGE == gdn::kErrDecayRange,
                  "error bit mirror");
    if (p->flags & ~(GDN_FLAG_L2NORM_Q | GDN_FLAG_L2NORM_K | GDN_FLAG_BETA_SIGMOID | GDN_FLAG_DECAY_PER_KEY |
                     GDN_FLAG_BETA_SHARED | GDN_FLAG_STATE_KMAJOR))
        return fail(GDN_ERR_INVALID, "unknown flag bits 0x%x", p->flags);
    if ((p->erase_gate || p->write_gate) && p->rule != GDN_RULE_GDN2)
        return fail(GDN_ERR_INVALID, "erase_gate and write_gate belong to rule GDN2");
    if ((p->flags & GDN_FLAG_BETA_SHARED) && p->rule != GDN_RULE_DELTA && p->rule != GDN_RULE_GATED_DELTA &&
        !(p->rule == GDN_RULE_GDN2 && p->erase_gate))
        return fail(GDN_ERR_INVALID,
                    "GDN_FLAG_BETA_SHARED applies to a scalar beta (rules DELTA, GATED_DELTA, GDN2 with erase_gate)");
    if (p->state_update_capacity != 0)
        return fail(GDN_ERR_INVALID, "state_update_capacity must be 0 (compact capture is not provided)");
    if (!isfinite(p->scale)) return fail(GDN_ERR_INVALID, "scale must be finite");
    if (p->seq_len < 0) return fail(GDN_ERR_INVALID, "seq_len must be >= 0");
    if (p->seq_len > 0) {
        if (p->cu_seqlens)
            return fail(GDN_ERR_INVALID, "cu_seqlens requires the rank-3 (packed) form; seq_len must be 0");
        if ((long long)p->batch * p->seq_len != p->total_tokens)
            return fail(GDN_ERR_INVALID, "rank-4 form: total_tokens (%d) != batch * seq_len (%d * %d)",
                        p->total_tokens, p->batch, p->seq_len);
    } else if (p->seq_lens) {
        return fail(GDN_ERR_INVALID, "seq_lens requires the rank-4 (padded) form; seq_len must be > 0");
    } else if (!p->cu_seqlens && p->batch > 0 && p->total_tokens % p->batch != 0) {
        return fail(GDN_ERR_INVALID, "uniform packing: total_tokens (%d) is not a multiple of batch (%d)",
                    p->total_tokens, p->batch);
    }
    const bool has_decay = gdn::rule_has_decay(p->rule);
    const bool has_beta = gdn::rule_has_retrieval(p->rule);
    if (has_decay != (p->decay != nullptr))
        return fail(GDN_ERR_INVALID, has_decay ? "this update rule needs decay" : "decay given for a rule without decay");
    if (has_beta != (p->beta != nullptr))
        return fail(GDN_ERR_INVALID, has_beta ? "this update rule needs beta" : "beta given for a rule without retrieval");
    if ((p->gate_bias == nullptr) != (p->gate_scale == nullptr))
        return fail(GDN_ERR_INVALID, "gate_bias and gate_scale must be given together (raw-gate arm) or not at all");
    if (p->gate_bias && !has_decay) return fail(GDN_ERR_INVALID, "raw-gate parameters given for a rule without decay");
    if ((p->flags & GDN_FLAG_DECAY_PER_KEY) && !has_decay)
        return fail(GDN_ERR_INVALID, "GDN_FLAG_DECAY_PER_KEY given for a rule without decay");
    if (has_decay) {
        if ((st = check_dtype(p->decay_dtype, "decay_dtype")) != GDN_OK) return st;
        if (p->decay_dtype != GDN_DTYPE_F32 && p->decay_dtype != p->act_dtype)
            return fail(GDN_ERR_INVALID, "decay_dtype must be F32 or the activation dtype");
    }
    if (has_beta) {
        if ((st = check_dtype(p->beta_dtype, "beta_dtype")) != GDN_OK) return st;
        if (p->beta_dtype != GDN_DTYPE_F32 && p->beta_dtype != p->act_dtype)
            return fail(GDN_ERR_INVALID, "beta_dtype must be F32 or the activation dtype");
    }
    const int rows = p->num_state_rows ? p->num_state_rows : p->batch;
    if (p->num_state_rows < 0) return fail(GDN_ERR_INVALID, "num_state_rows must be >= 0");
    if (!p->slot_ids && rows < p->batch)
        return fail(GDN_ERR_INVALID, "num_state_rows (%d) < batch (%d) without slot_ids", rows, p->batch);
    if (p->batch > 0) {
        if (!p->q || !p->k || !p->v || !p->o) return fail(GDN_ERR_INVALID, "q, k, v and o are required");
        if (!p->final_state) return fail(GDN_ERR_INVALID, "final_state is required");
    }
    const size_t ea = dtype_size(p->act_dtype);
    if (!aligned(p->q, ea) || !aligned(p->k, ea) || !aligned(p->v, ea) || !aligned(p->o, ea) ||
        !aligned(p->decay, dtype_size(p->decay_dtype)) || !aligned(p->beta, dtype_size(p->beta_dtype)) ||
        !aligned(p->gate_bias, 4) || !aligned(p->gate_scale, 4) || !aligned(p->cu_seqlens, 4) ||
        !aligned(p->slot_ids, 4) || !aligned(p->initial_state, 4) || !aligned(p->final_state, 4) ||
        !aligned(p->error_word, 4) || !aligned(p->seq_lens, 4) || !aligned(p->erase_gate, 4) ||
        !aligned(p->write_gate, 4))
        return fail(GDN_ERR_INVALID, "a pointer is not aligned to its element size");
    const long long grid_bound = (long long)p->batch * p->num_heads_v * p->head_dim_v;
    if (grid_bound > (1LL << 31) - 1) return fail(GDN_ERR_UNSUPPORTED, "batch * Hv * dv exceeds 2^31 - 1");

    gdn::Problem &d = *out;
    d.B = p->batch;
    d.T = p->total_tokens;
    d.seq_len = p->seq_len;
    d.Hq = p->num_heads_q;
    d.Hv = p->num_heads_v;
    d.dk = p->head_dim_k;
    d.dv = p->head_dim_v;
    d.rows = rows;
    d.rule = p->rule;
    d.flags = p->flags;
    d.scale = p->scale != 0.f ? p->scale : (float)(1.0 / sqrt((double)p->head_dim_k));
    d.act_f16 = p->act_dtype == GDN_DTYPE_F16;
    d.decay_f16 = has_decay && p->decay_dtype == GDN_DTYPE_F16;
    d.beta_f16 = has_beta && p->beta_dtype == GDN_DTYPE_F16;
    d.raw_gate = p->gate_bias != nullptr;
    d.q = p->q;
    d.k = p->k;
    d.v = p->v;
    d.o = p->o;
    d.decay = p->decay;
    d.gate_bias = p->gate_bias;
    d.gate_scale = p->gate_scale;
    d.beta = p->beta;
    d.cu = p->cu_seqlens;
    d.seqlens = p->seq_lens;
    d.slots = p->slot_ids;
    d.init = p->initial_state;
    d.fin = p->final_state;
    d.err = p->error_word;
    d.erase_gate = p->erase_gate;
    d.write_gate = p->write_gate;
    d.o_f32 = 0;
    d.win = nullptr;
    return GDN_OK;
}

gdn_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return ok();
    return fail(GDN_ERR_CUDA, "CUDA error: %s", cudaGetErrorString(e));
}

}  // namespace

namespace gdn {

// Kernel attributes and occupancy, set or queried once per (device, kernel,
// size) under a lock, so that threads making their first calls at the same
// time do not race on the caches.
namespace {
std::mutex g_attr_mu;
std::map<std::tuple<int, const void *, size_t>, int> g_attr;  // value: blocks per SM (0: attribute only)
}  // namespace

cudaError_t smem_attr(const void *fn, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_attr_mu);
    const auto key = std::make_tuple(dev, fn, (size_t)bytes | ((size_t)1 << 62));
    if (g_attr.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) g_attr[key] = 0;
    return e;
}

cudaError_t blocks_per_sm(const void *fn, int threads, size_t smem, int *n) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_attr_mu);
    const auto key = std::make_tuple(dev, fn, smem * 4096 + (size_t)threads);
    auto it = g_attr.find(key);
    if (it != g_attr.end()) {
        *n = it->second;
        return cudaSuccess;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    g_attr[key] = per_sm;
    *n = per_sm;
    return cudaSuccess;
}

int sm_count() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace gdn

extern "C" {

const char *gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported by this library";
        case GDN_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case GDN_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

const char *gdn_last_error_message(void) { return g_msg; }

gdn_status gdn_gate(const gdn_gate_args *a, gdn_stream stream) {
    if (!a) return fail(GDN_ERR_INVALID, "args is NULL");
    gdn_status st;
    if ((st = check_dtype(a->dtype, "dtype")) != GDN_OK) return st;
    if (a->n < 0) return fail(GDN_ERR_INVALID, "n must be >= 0");
    if (a->heads <= 0) return fail(GDN_ERR_INVALID, "heads must be positive");
    if (a->beta_out && !a->b) return fail(GDN_ERR_INVALID, "beta requested without b");
    if (a->n == 0) return ok();
    if (!a->a || !a->dt_bias || !a->decay_scale || !a->decay_out)
        return fail(GDN_ERR_INVALID, "a, dt_bias, decay_scale and decay_out are required");
    const size_t e = dtype_size(a->dtype);
    if (!aligned(a->a, e) || !aligned(a->b, e) || !aligned(a->decay_out, e) || !aligned(a->beta_out, e) ||
        !aligned(a->dt_bias, 4) || !aligned(a->decay_scale, 4))
        return fail(GDN_ERR_INVALID, "a pointer is not aligned to its element size");
    gdn::GateLaunch g{a->n, a->heads, a->dtype == GDN_DTYPE_F16, a->a, a->dt_bias, a->decay_scale,
                      a->beta_out ? a->b : nullptr, a->decay_out, a->beta_out};
    return cuda_status(gdn::launch_gate(g, (cudaStream_t)stream));
}

gdn_status gdn_recurrent_step(const gdn_problem *p, gdn_stream stream) {
    gdn::Problem d;
    gdn_status st = validate(p, &d);
    if (st != GDN_OK) return st;
    if (d.B == 0) return ok();
    return cuda_status(gdn::launch_recurrent(d, (cudaStream_t)stream));
}

size_t gdn_chunked_prefill_workspace_size(const gdn_problem *p, int32_t chunk_size) {
    gdn::Problem d;
    if (validate(p, &d) != GDN_OK) return (size_t)-1;
    const char *why = nullptr;
    if (!gdn::chunked_supported(d, chunk_size, &why)) {
        fail(GDN_ERR_UNSUPPORTED, "chunked prefill: %s", why);
        return (size_t)-1;
    }
    ok();
    return gdn::chunked_workspace_bytes(d, chunk_size);
}

size_t gdn_chunked_prefill_workspace_size_min(const gdn_problem *p, int32_t chunk_size) {
    gdn::Problem d;
    if (validate(p, &d) != GDN_OK) return (size_t)-1;
    const char *why = nullptr;
    if (!gdn::chunked_supported(d, chunk_size, &why)) {
        fail(GDN_ERR_UNSUPPORTED, "chunked prefill: %s", why);
        return (size_t)-1;
    }
    ok();
    return gdn::chunked_workspace_min_bytes(d, chunk_size);
}

gdn_status gdn_chunked_prefill(const gdn_problem *p, int32_t chunk_size, void *ws, size_t ws_bytes,
                               gdn_stream stream) {
    gdn::Problem d;
    gdn_status st = validate(p, &d);
    if (st != GDN_OK) return st;
    const char *why = nullptr;
    if (!gdn::chunked_supported(d, chunk_size, &why)) return fail(GDN_ERR_UNSUPPORTED, "chunked prefill: %s", why);
    const size_t need = gdn::chunked_workspace_bytes(d, chunk_size);
    const size_t least = gdn::chunked_workspace_min_bytes(d, chunk_size);
    if (need > 0 && (ws == nullptr || ws_bytes < least || !aligned(ws, 256)))
        return fail(GDN_ERR_WORKSPACE,
                    "workspace needs at least %zu bytes (%zu for a single pass), 256-byte aligned (got %zu)", least,
                    need, ws_bytes);
    if (d.B == 0) return ok();
    return cuda_status(gdn::launch_chunked(d, chunk_size, ws, ws_bytes, (cudaStream_t)stream));
}

gdn_status gdn_chunked_prefill_noalloc(const gdn_problem *p, int32_t chunk_size, gdn_stream stream) {
    gdn::Problem d;
    gdn_status st = validate(p, &d);
    if (st != GDN_OK) return st;
    const char *why = nullptr;
    if (!gdn::chunked_supported(d, chunk_size, &why)) return fail(GDN_ERR_UNSUPPORTED, "chunked prefill: %s", why);
    const size_t need = gdn::chunked_workspace_bytes(d, chunk_size);
    if (need > kNoAllocBytes)
        return fail(GDN_ERR_WORKSPACE, "needs %zu bytes of scratch, the library's static scratch holds %zu", need,
                    kNoAllocBytes);
    if (d.B == 0) return ok();
    void *ws = nullptr;
    if (need > 0) {
        const cudaError_t e = noalloc_scratch(&ws);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return cuda_status(gdn::launch_chunked(d, chunk_size, ws, need, (cudaStream_t)stream));
}

}  // extern "C"
