// recurrent.cu -- token-serial gated delta rule ("aclnnRecurrentGatedDeltaRule":
// the variable-step form for L_i <= 8 tokens per request; the decode and
// multi-token-prediction step).
//
// Design (HBM-bound: the fp32 state tile dominates the bytes):
//  * One CTA per (request, value head, slice of 32 value rows).  The slice of
//    the V-major state is 32 contiguous rows of dk floats, so a CTA streams one
//    contiguous 32*dk*4-byte block in and out, once.
//  * Fast path (dk in {32, 64, 128, 256}): 8 warps x 4 rows; the 8 lanes of a
//    row each hold dk/8 columns as float4s (column 32*j + 4*lane8), so every
//    load/store instruction moves 128 contiguous bytes per row.  Row dot
//    products reduce over those 8 lanes with 3 xor-shuffles.
//  * All state loads are issued first; while they are in flight the CTA stages
//    up to 8 tokens of per-token data in shared memory: the (optionally
//    L2-normalised) key and query in fp32, q.k, alpha = exp(g) from the fused
//    raw-gate arm, beta (optionally through the sigmoid), the per-key alpha
//    vector and the GDN-2 retrieval key b .* k.  One warp per token does this
//    with full-warp reductions, so the per-row loop only does FMAs.
//  * Per token and row i:  u = S_i . kappa,  w = S_i . q (one pass), then
//      d = beta (v_i - alpha u),  S_i <- alpha S_i + d k,
//      o_i = scale (alpha w + d (k . q))   (= scale * S_i^new . q exactly)
//    With per-key decay S_i is first scaled column-wise and alpha = 1 above.
//  * Generic path (any dk, dv <= 256 or unaligned pointers): one warp per row,
//    lane c holds columns c + 32 i, full-warp reductions.
#include "common.cuh"
#include "launch.h"

namespace gdn {

constexpr int kTB = 8;           // tokens staged per step
constexpr int kFastRows = 32;    // value rows per CTA, fast path
constexpr int kGenericRows = 8;  // value rows per CTA, generic path (one per warp)
constexpr int kThreads = 256;

struct Stage {
    float *k, *q, *a, *x, *v, *alpha, *beta, *kq;
    int dkp;
};

__device__ __forceinline__ Stage carve(float *smem, int dkp, int rows) {
    Stage s;
    s.dkp = dkp;
    s.k = smem;
    s.q = s.k + kTB * dkp;
    s.a = s.q + kTB * dkp;
    s.x = s.a + kTB * dkp;
    s.v = s.x + kTB * dkp;
    s.alpha = s.v + kTB * rows;
    s.beta = s.alpha + kTB;
    s.kq = s.beta + kTB;
    return s;
}

static size_t stage_bytes(int dkp, int rows) {
    return sizeof(float) * ((size_t)4 * kTB * dkp + (size_t)kTB * rows + 3 * kTB);
}

// Stages tokens [tb, tb + nt) of (request's head h / key head qh) and the v
// entries of rows [r0, r0 + rows).  All warps of the CTA take part.
__device__ void stage_tokens(const Problem &p, const Stage &s, int h, int qh, int tb, int nt,
                             int r0, int rows) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const bool has_decay = rule_has_decay(p.rule);
    const bool perkey = (p.flags & kPerKey) != 0;
    const bool gdn2 = p.rule == kGdn2;
    const bool beta_scalar = p.rule == kDelta || p.rule == kGatedDelta;
    const bool sig = (p.flags & kBetaSigmoid) != 0;
    for (int idx = threadIdx.x; idx < nt * rows; idx += blockDim.x) {
        const int tt = idx / rows, r = idx % rows;
        const int i = r0 + r;
        s.v[tt * rows + r] = i < p.dv ? ld_any(p.v, ((size_t)(tb + tt) * p.Hv + h) * p.dv + i, p.act_f16) : 0.f;
    }
    for (int tt = warp; tt < nt; tt += nw) {
        const int t = tb + tt;
        const size_t qko = ((size_t)t * p.Hq + qh) * p.dk;
        float kv[8], qv[8];
        float ssk = 0.f, ssq = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = lane + 32 * i;
            kv[i] = c < p.dk ? ld_any(p.k, qko + c, p.act_f16) : 0.f;
            qv[i] = c < p.dk ? ld_any(p.q, qko + c, p.act_f16) : 0.f;
            ssk += kv[i] * kv[i];
            ssq += qv[i] * qv[i];
        }
        const float ik = (p.flags & kL2k) ? rsqrtf(warp_sum(ssk) + 1e-12f) : 1.f;
        const float iq = (p.flags & kL2q) ? rsqrtf(warp_sum(ssq) + 1e-12f) : 1.f;
        float kq = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            kv[i] *= ik;
            qv[i] *= iq;
            kq += kv[i] * qv[i];
        }
        kq = warp_sum(kq);
        const size_t th = (size_t)t * p.Hv + h;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = lane + 32 * i;
            if (c < p.dk) {
                s.k[tt * s.dkp + c] = kv[i];
                s.q[tt * s.dkp + c] = qv[i];
                if (has_decay && perkey) {
                    float g = ld_any(p.decay, th * p.dk + c, p.decay_f16);
                    if (p.raw_gate) g = p.gate_scale[h] * softplus_f(g + p.gate_bias[(size_t)h * p.dk + c]);
                    s.a[tt * s.dkp + c] = expf(g);
                }
                if (gdn2) {
                    float bb = ld_any(p.beta, th * p.dk + c, p.beta_f16);
                    if (sig) bb = sigmoid_f(bb);
                    s.x[tt * s.dkp + c] = bb * kv[i];
                }
            }
        }
        if (lane == 0) {
            float alpha = 1.f, beta = 1.f;
            if (has_decay && !perkey) {
                float g = ld_any(p.decay, th, p.decay_f16);
                if (p.raw_gate) g = p.gate_scale[h] * softplus_f(g + p.gate_bias[h]);
                alpha = expf(g);
            }
            if (beta_scalar) {
                beta = ld_any(p.beta, th, p.beta_f16);
                if (sig) beta = sigmoid_f(beta);
            }
            s.alpha[tt] = alpha;
            s.beta[tt] = beta;
            s.kq[tt] = kq;
        }
    }
}

__device__ __forceinline__ void st_out(const Problem &p, size_t idx, float x) {
    if (p.act_f16)
        static_cast<__half *>(p.o)[idx] = __float2half_rn(x);
    else
        static_cast<float *>(p.o)[idx] = x;
}

__device__ __forceinline__ float dot4(const float4 &a, const float4 &b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}
__device__ __forceinline__ float4 ld_f4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

template <int DK>
__global__ void __launch_bounds__(kThreads) recurrent_fast_kernel(Problem p, int slices) {
    constexpr int NV = DK / 32;  // float4s per lane per row
    extern __shared__ __align__(16) float smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cg = lane & 7;
    const int sidx = blockIdx.x % slices;
    const int bh = blockIdx.x / slices;
    const int h = bh % p.Hv, b = bh / p.Hv;
    const int r0 = sidx * kFastRows;
    const int i_row = r0 + warp * 4 + (lane >> 3);
    const bool active = i_row < p.dv;

    const int row = state_row(p, b, h == 0 && sidx == 0 && threadIdx.x == 0);
    if (row < 0) return;
    int t0, t1;
    request_range(p, b, t0, t1);

    const size_t soff = (((size_t)row * p.Hv + h) * p.dv + i_row) * DK + 4 * cg;
    float4 S[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) S[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active && p.init) {
#pragma unroll
        for (int j = 0; j < NV; ++j) S[j] = __ldcs(reinterpret_cast<const float4 *>(p.init + soff + 32 * j));
    }
    if (t1 == t0) {  // empty request: the incoming state goes through unchanged
        if (active && p.fin != p.init) {
#pragma unroll
            for (int j = 0; j < NV; ++j) __stcs(reinterpret_cast<float4 *>(p.fin + soff + 32 * j), S[j]);
        }
        return;
    }

    const Stage s = carve(smem, DK, kFastRows);
    const int qh = (int)((long long)h * p.Hq / p.Hv);
    const bool perkey = (p.flags & kPerKey) != 0 && rule_has_decay(p.rule);
    const bool retrieval = rule_has_retrieval(p.rule);
    const float *kap = p.rule == kGdn2 ? s.x : s.k;
    const int rloc = i_row - r0;

    for (int tb = t0; tb < t1; tb += kTB) {
        const int nt = min(kTB, t1 - tb);
        if (tb != t0) __syncthreads();
        stage_tokens(p, s, h, qh, tb, nt, r0, kFastRows);
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            const float *kk = s.k + tt * DK + 4 * cg;
            const float *qq = s.q + tt * DK + 4 * cg;
            const float *xx = kap + tt * DK + 4 * cg;
            if (perkey) {
                const float *aa = s.a + tt * DK + 4 * cg;
#pragma unroll
                for (int j = 0; j < NV; ++j) {
                    const float4 a4 = ld_f4(aa + 32 * j);
                    S[j].x *= a4.x, S[j].y *= a4.y, S[j].z *= a4.z, S[j].w *= a4.w;
                }
            }
            float u = 0.f, w = 0.f;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                u += dot4(S[j], ld_f4(xx + 32 * j));
                w += dot4(S[j], ld_f4(qq + 32 * j));
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                u += __shfl_xor_sync(0xffffffffu, u, o);
                w += __shfl_xor_sync(0xffffffffu, w, o);
            }
            const float alpha = perkey ? 1.f : s.alpha[tt];
            const float vi = s.v[tt * kFastRows + rloc];
            const float d = retrieval ? s.beta[tt] * (vi - alpha * u) : vi;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const float4 k4 = ld_f4(kk + 32 * j);
                S[j].x = fmaf(alpha, S[j].x, d * k4.x);
                S[j].y = fmaf(alpha, S[j].y, d * k4.y);
                S[j].z = fmaf(alpha, S[j].z, d * k4.z);
                S[j].w = fmaf(alpha, S[j].w, d * k4.w);
            }
            if (cg == 0 && active)
                st_out(p, ((size_t)(tb + tt) * p.Hv + h) * p.dv + i_row,
                       p.scale * fmaf(alpha, w, d * s.kq[tt]));
        }
    }
    if (active) {
#pragma unroll
        for (int j = 0; j < NV; ++j) __stcs(reinterpret_cast<float4 *>(p.fin + soff + 32 * j), S[j]);
    }
}

// Any dk, dv <= 256: one warp per value row, lane c holds columns c + 32 i.
__global__ void __launch_bounds__(kThreads) recurrent_generic_kernel(Problem p, int slices) {
    extern __shared__ __align__(16) float smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sidx = blockIdx.x % slices;
    const int bh = blockIdx.x / slices;
    const int h = bh % p.Hv, b = bh / p.Hv;
    const int r0 = sidx * kGenericRows;
    const int i_row = r0 + warp;
    const bool active = i_row < p.dv;
    const int row = state_row(p, b, h == 0 && sidx == 0 && threadIdx.x == 0);
    if (row < 0) return;
    int t0, t1;
    request_range(p, b, t0, t1);
    const size_t soff = (((size_t)row * p.Hv + h) * p.dv + i_row) * p.dk;
    float S[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = lane + 32 * i;
        S[i] = (active && p.init && c < p.dk) ? p.init[soff + c] : 0.f;
    }
    if (t1 == t0) {
        if (active && p.fin != p.init) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = lane + 32 * i;
                if (c < p.dk) p.fin[soff + c] = S[i];
            }
        }
        return;
    }
    const int dkp = (p.dk + 3) & ~3;
    const Stage s = carve(smem, dkp, kGenericRows);
    const int qh = (int)((long long)h * p.Hq / p.Hv);
    const bool perkey = (p.flags & kPerKey) != 0 && rule_has_decay(p.rule);
    const bool retrieval = rule_has_retrieval(p.rule);
    const float *kap = p.rule == kGdn2 ? s.x : s.k;
    for (int tb = t0; tb < t1; tb += kTB) {
        const int nt = min(kTB, t1 - tb);
        if (tb != t0) __syncthreads();
        stage_tokens(p, s, h, qh, tb, nt, r0, kGenericRows);
        __syncthreads();
        for (int tt = 0; tt < nt; ++tt) {
            float u = 0.f, w = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = lane + 32 * i;
                if (c < p.dk) {
                    if (perkey) S[i] *= s.a[tt * dkp + c];
                    u += S[i] * kap[tt * dkp + c];
                    w += S[i] * s.q[tt * dkp + c];
                }
            }
            u = warp_sum(u);
            w = warp_sum(w);
            const float alpha = perkey ? 1.f : s.alpha[tt];
            const float vi = s.v[tt * kGenericRows + warp];
            const float d = retrieval ? s.beta[tt] * (vi - alpha * u) : vi;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = lane + 32 * i;
                if (c < p.dk) S[i] = fmaf(alpha, S[i], d * s.k[tt * dkp + c]);
            }
            if (lane == 0 && active)
                st_out(p, ((size_t)(tb + tt) * p.Hv + h) * p.dv + i_row,
                       p.scale * fmaf(alpha, w, d * s.kq[tt]));
        }
    }
    if (active) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = lane + 32 * i;
            if (c < p.dk) p.fin[soff + c] = S[i];
        }
    }
}

static bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

cudaError_t launch_recurrent(const Problem &p, cudaStream_t stream) {
    const bool fast_dk = p.dk == 32 || p.dk == 64 || p.dk == 128 || p.dk == 256;
    const bool fast = fast_dk && aligned16(p.fin) && (p.init == nullptr || aligned16(p.init));
    const long long pairs = (long long)p.B * p.Hv;
    if (fast) {
        const int slices = (p.dv + kFastRows - 1) / kFastRows;
        const long long grid = pairs * slices;
        const size_t smem = stage_bytes(p.dk, kFastRows);
        switch (p.dk) {
            case 32: recurrent_fast_kernel<32><<<(unsigned)grid, kThreads, smem, stream>>>(p, slices); break;
            case 64: recurrent_fast_kernel<64><<<(unsigned)grid, kThreads, smem, stream>>>(p, slices); break;
            case 128: recurrent_fast_kernel<128><<<(unsigned)grid, kThreads, smem, stream>>>(p, slices); break;
            default: recurrent_fast_kernel<256><<<(unsigned)grid, kThreads, smem, stream>>>(p, slices); break;
        }
    } else {
        const int slices = (p.dv + kGenericRows - 1) / kGenericRows;
        const long long grid = pairs * slices;
        const size_t smem = stage_bytes((p.dk + 3) & ~3, kGenericRows);
        recurrent_generic_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(p, slices);
    }
    return cudaGetLastError();
}

}  // namespace gdn
