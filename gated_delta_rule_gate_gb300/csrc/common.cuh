// common.cuh -- device helpers shared by the CUDA kernels of libgdn.
//
// Nothing here is shared with the CPU oracle: the oracle is a separate C
// program, and this header is included by the CUDA translation units only.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// Rules and flags, mirrored from include/gdn.h for device code.
enum : int { kLinear = 0, kGated = 1, kDelta = 2, kGatedDelta = 3, kGdn2 = 4 };
enum : unsigned { kL2q = 0x1u, kL2k = 0x2u, kBetaSigmoid = 0x4u, kPerKey = 0x8u, kBetaShared = 0x10u, kKMajor = 0x20u };
// Device error bits, mirrored from include/gdn.h.
enum : int { kErrBadSlot = 0x1, kErrTimeout = 0x2, kErrOverlap = 0x4, kErrDecayRange = 0x8 };

__host__ __device__ inline bool rule_has_decay(int r) {
    return r == kGated || r == kGatedDelta || r == kGdn2;
}
__host__ __device__ inline bool rule_has_retrieval(int r) {
    return r == kDelta || r == kGatedDelta || r == kGdn2;
}

// Validated problem, passed by value to every recurrence kernel.
struct Problem {
    int B, T, seq_len, Hq, Hv, dk, dv, rows;
    int rule;
    unsigned flags;
    float scale;  // already resolved (0 -> 1/sqrt(dk))
    int act_f16, decay_f16, beta_f16;
    int raw_gate;
    const void *q, *k, *v;
    void *o;
    const void *decay;
    const float *gate_bias, *gate_scale;
    const void *beta;
    const int32_t *cu, *slots, *seqlens;
    const float *init;
    float *fin;
    int32_t *err;
    const float *erase_gate;  // GDN-2 erase gate as its own input [T, Hv, dk], or null
    const float *write_gate;  // GDN-2 write gate [T, Hv, dv], or null
    int o_f32;                // tensor-core prefill on fp16 copies of fp32 inputs: o is fp32
    // windowed tensor-core prefill: per request the [t0, t1) of the current window (device,
    // 2 B ints), which then replaces the request's own range; null otherwise
    const int32_t *win;
};

// GDN-2 with the erase gate in its own input: beta is then a scalar per
// (token, head) that scales the write, d = beta (w .* v) - u.
__host__ __device__ inline bool erase_input(const Problem &p) { return p.erase_gate != nullptr; }
// Rules whose beta is one scalar per (token, head) (or per token, shared).
__host__ __device__ inline bool beta_is_scalar(const Problem &p) {
    return p.rule == kDelta || p.rule == kGatedDelta || (p.rule == kGdn2 && p.erase_gate != nullptr);
}
// GDN-2 with its value rows scaled inside the kernel (v' = beta w .* v).
__host__ __device__ inline bool scales_v(const Problem &p) {
    return p.rule == kGdn2 && (p.erase_gate != nullptr || p.write_gate != nullptr);
}

// Element index of the scalar beta of token t and value head h: [T, Hv], or
// [T] when one beta per token serves every value head (kBetaShared).
__device__ __forceinline__ size_t beta_at(const Problem &p, size_t t, int h) {
    return (p.flags & kBetaShared) ? t : t * p.Hv + h;
}

__device__ __forceinline__ float ld_any(const void *p, size_t i, int f16) {
    return f16 ? __half2float(static_cast<const __half *>(p)[i]) : static_cast<const float *>(p)[i];
}

// softplus(x) = ln(1 + e^x) in fp32; above 20 the correction is below fp32
// resolution of x, so x itself is returned.
__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// Token range [t0, t1) of request b: cu_seqlens clamped to [0, T] (a
// decreasing pair gives an empty request), or uniform packing, whose rows
// seq_lens (clamped to [0, seq_len]) can shorten.
__device__ __forceinline__ void request_range(const Problem &p, int b, int &t0, int &t1) {
    if (p.win) {
        t0 = p.win[2 * b];
        t1 = p.win[2 * b + 1];
        return;
    }
    if (p.cu) {
        int a = p.cu[b], c = p.cu[b + 1];
        a = a < 0 ? 0 : (a > p.T ? p.T : a);
        c = c < 0 ? 0 : (c > p.T ? p.T : c);
        t0 = a;
        t1 = c < a ? a : c;
    } else {
        int L = p.seq_len ? p.seq_len : p.T / p.B;
        t0 = b * L;
        int n = L;
        if (p.seqlens) {
            n = p.seqlens[b];
            n = n < 0 ? 0 : (n > L ? L : n);
        }
        t1 = t0 + n;
    }
}

// State row of request b, or -1 (and the error bit) for an out-of-range slot.
__device__ __forceinline__ int state_row(const Problem &p, int b, bool report) {
    int r = p.slots ? p.slots[b] : b;
    if (r < 0 || r >= p.rows) {
        if (report && p.err) atomicOr(p.err, 1);
        return -1;
    }
    return r;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace gdn
