// chunked.cu -- chunk-parallel prefill of the gated delta rule.
//
// "com.microsoft.GatedDeltaNet" (key input; chunk_size attribute) states that
// a chunk-parallel prefill exists, that its per-chunk system needs unit keys,
// and that the chunk size never changes the result.  The per-chunk algebra is
// derived from the token recurrence (value-major M, in-chunk log-decay
// cumulants G_r = sum_{j<=r} g_j, chunk of C tokens, incoming state M0):
//
//   A_rj  = beta_r e^{G_r - G_j} (kappa_r . k_j)  (j < r),   T = (I + A)^-1
//   U'    = T diag(beta) V,        W = T diag(beta e^G) Kappa
//   Delta = U' - W M0^T            (rows = the per-token corrections d_t)
//   O     = scale (diag(e^G) Q M0^T + P Delta),  P_rj = e^{G_r - G_j} (q_r . k_j), j <= r
//   M_C   = e^{G_C} M0 + Delta^T diag(e^{G_C - G}) K
//
// kappa = k for the v1 rules; kappa = b .* k with beta = 1 for GDN-2.  Rules
// without retrieval take Delta = V.  Every exponent is a difference G_r - G_j
// with j <= r (or G_C - G_j, or G_r), so nothing overflows however strong the
// decay (cumulants of -165 per chunk occur with the ragged-prefill gates).
//
// Kernel layout: one CTA of 4 warps per (request, value head, 64-row slice of
// dv).  Warp w owns 16 value rows of the state, held in registers as fp32
// m16n8 accumulator tiles for the whole request; those tiles are also exactly
// the B fragments of M0^T that the Delta and Q M0^T products need (after a
// pack to fp16), so the state never leaves registers between chunks.  The
// chunk's K, Q, V tiles are fetched with cp.async into padded shared memory.
// All products are fp16 x fp16 -> fp32 warp-level tensor-core MMAs
// (m16n8k16); the triangular solve runs in fp32 on the CUDA cores as 16x16
// diagonal-block inverses plus blocked off-diagonal updates.
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int C = 64;        // tokens per chunk
constexpr int VS = 64;       // value rows per CTA
constexpr int NW = 4;        // warps per CTA
constexpr int NTH = NW * 32;

template <int DK, bool GDN2>
struct Lay {
    static constexpr int KS = DK + 8;   // halfs per row, [C][DK] tiles
    static constexpr int VSS = VS + 8;  // halfs per row, [C][VS] tiles
    static constexpr int CS = C + 8;    // halfs per row, [C][C] tiles
    static constexpr int FS = C + 1;    // floats per row, fp32 [C][C] tiles
    static constexpr int bK = C * KS * 2;
    static constexpr int bV = C * VSS * 2;
    static constexpr int bC = C * CS * 2;
    static constexpr int bF = C * FS * 4;
    static constexpr int oK = 0;
    static constexpr int oQ = oK + bK;
    static constexpr int oV = oQ + bK;
    // region 1: {Af, Tf} during the solve, then {W, D, Dt}
    static constexpr int oU1 = oV + bV;
    static constexpr int szU1 = (2 * bF > bK + 2 * bV) ? 2 * bF : bK + 2 * bV;
    static constexpr int oAf = oU1, oTf = oU1 + bF;
    static constexpr int oW = oU1, oD = oU1 + bK, oDt = oD + bV;
    // region 2: {Ta, Tb}, then {P}
    static constexpr int oU2 = oU1 + szU1;
    static constexpr int oTa = oU2, oTb = oU2 + bC, oP = oU2;
    static constexpr int oG = oU2 + 2 * bC;
    static constexpr int oB = oG + C * 4;
    static constexpr int oEG = oB + C * 4;
    static constexpr int oEGC = oEG + C * 4;
    static constexpr int oX16 = oEGC + C * 4;
    static constexpr int oKap = oX16 + NW * 16 * 17 * 4;
    static constexpr int oVB = oKap + (GDN2 ? bK : 0);  // GDN-2: beta of the write, per token
    static constexpr int total = oVB + (GDN2 ? C * 4 : 0);
};

__device__ __forceinline__ float2 ld_f2(const float *p) { return *reinterpret_cast<const float2 *>(p); }

template <int DK, bool GDN2>
__global__ void __launch_bounds__(NTH, 2) chunked_mma_kernel(Problem p, int slices) {
    using Ly = Lay<DK, GDN2>;
    constexpr int KS = Ly::KS, VSS = Ly::VSS, CS = Ly::CS, FS = Ly::FS;
    constexpr int NT8 = DK / 8;   // n-tiles across dk
    constexpr int KST = DK / 16;  // k-steps across dk
    extern __shared__ __align__(128) unsigned char sm[];
    __half *sK = reinterpret_cast<__half *>(sm + Ly::oK);
    __half *sQ = reinterpret_cast<__half *>(sm + Ly::oQ);
    __half *sV = reinterpret_cast<__half *>(sm + Ly::oV);
    float *sAf = reinterpret_cast<float *>(sm + Ly::oAf);
    float *sTf = reinterpret_cast<float *>(sm + Ly::oTf);
    __half *sW = reinterpret_cast<__half *>(sm + Ly::oW);
    __half *sD = reinterpret_cast<__half *>(sm + Ly::oD);
    __half *sDt = reinterpret_cast<__half *>(sm + Ly::oDt);
    __half *sTa = reinterpret_cast<__half *>(sm + Ly::oTa);
    __half *sTb = reinterpret_cast<__half *>(sm + Ly::oTb);
    __half *sP = reinterpret_cast<__half *>(sm + Ly::oP);
    float *sG = reinterpret_cast<float *>(sm + Ly::oG);
    float *sBt = reinterpret_cast<float *>(sm + Ly::oB);
    float *sEG = reinterpret_cast<float *>(sm + Ly::oEG);
    float *sEGC = reinterpret_cast<float *>(sm + Ly::oEGC);
    float *sX16 = reinterpret_cast<float *>(sm + Ly::oX16);
    __half *sKap = reinterpret_cast<__half *>(sm + Ly::oKap);
    float *sVB = reinterpret_cast<float *>(sm + Ly::oVB);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int sidx = blockIdx.x % slices;
    const int bh = blockIdx.x / slices;
    const int h = bh % p.Hv, b = bh / p.Hv;
    const int vs0 = sidx * VS;
    const int wrow0 = vs0 + 16 * warp;

    const int row = state_row(p, b, h == 0 && sidx == 0 && tid == 0);
    if (row < 0) return;
    int t0, t1;
    request_range(p, b, t0, t1);
    const int qh = (int)((long long)h * p.Hq / p.Hv);
    const bool retrieval = rule_has_retrieval(p.rule);
    const bool has_decay = rule_has_decay(p.rule);
    const bool beta_scalar = p.rule == kDelta || p.rule == kGatedDelta;
    const bool sig = (p.flags & kBetaSigmoid) != 0;

    // ---- the state: rows rlo = wrow0 + g and rhi = rlo + 8, columns 8 nt + 2 t4 + {0,1}
    float S[NT8][4];
    // element (r, c) of the state tile: value-major at r * DK + c, key-major at c * dv + r
    const bool km = (p.flags & kKMajor) != 0;
    const size_t tile = ((size_t)row * p.Hv + h) * p.dv * DK;
    const int rlo = wrow0 + g, rhi = rlo + 8;
    const bool lo_ok = rlo < p.dv, hi_ok = rhi < p.dv;
    auto ld_pair = [&](int r, int col) {
        return km ? make_float2(p.init[tile + (size_t)col * p.dv + r], p.init[tile + (size_t)(col + 1) * p.dv + r])
                  : ld_f2(p.init + tile + (size_t)r * DK + col);
    };
    auto st_pair = [&](int r, int col, float x, float y) {
        if (km) {
            p.fin[tile + (size_t)col * p.dv + r] = x;
            p.fin[tile + (size_t)(col + 1) * p.dv + r] = y;
        } else {
            *reinterpret_cast<float2 *>(p.fin + tile + (size_t)r * DK + col) = make_float2(x, y);
        }
    };
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) {
        const int col = 8 * nt + 2 * t4;
        float2 a = make_float2(0.f, 0.f), c = make_float2(0.f, 0.f);
        if (p.init && lo_ok) a = ld_pair(rlo, col);
        if (p.init && hi_ok) c = ld_pair(rhi, col);
        S[nt][0] = a.x, S[nt][1] = a.y, S[nt][2] = c.x, S[nt][3] = c.y;
    }
    if (t1 == t0) {  // empty request: the final state is the initial one
        if (p.fin != p.init) {
#pragma unroll
            for (int nt = 0; nt < NT8; ++nt) {
                const int col = 8 * nt + 2 * t4;
                if (lo_ok) st_pair(rlo, col, S[nt][0], S[nt][1]);
                if (hi_ok) st_pair(rhi, col, S[nt][2], S[nt][3]);
            }
        }
        return;
    }

    for (int c0 = t0; c0 < t1; c0 += C) {
        const int n = min(C, t1 - c0);
        __syncthreads();  // the previous chunk is done with shared memory

        // ---------------------------------------------------------------- load
        if (p.act_f16) {
            const __half *kg = static_cast<const __half *>(p.k);
            const __half *qg = static_cast<const __half *>(p.q);
            const __half *vg = static_cast<const __half *>(p.v);
            for (int idx = tid; idx < C * (DK / 8); idx += NTH) {
                const int r = idx / (DK / 8), sg = idx % (DK / 8);
                const bool ok = r < n;
                const size_t off = ok ? ((size_t)(c0 + r) * p.Hq + qh) * DK + sg * 8 : 0;
                ptx::cp_async16(sK + r * KS + sg * 8, kg + off, ok ? 16 : 0);
                ptx::cp_async16(sQ + r * KS + sg * 8, qg + off, ok ? 16 : 0);
            }
            for (int idx = tid; idx < C * (VS / 8); idx += NTH) {
                const int r = idx / (VS / 8), sg = idx % (VS / 8);
                const int col = vs0 + sg * 8;
                const bool ok = r < n && col < p.dv;
                const size_t off = ok ? ((size_t)(c0 + r) * p.Hv + h) * p.dv + col : 0;
                ptx::cp_async16(sV + r * VSS + sg * 8, vg + off, ok ? 16 : 0);
            }
        } else {
            const float *kg = static_cast<const float *>(p.k);
            const float *qg = static_cast<const float *>(p.q);
            const float *vg = static_cast<const float *>(p.v);
            for (int idx = tid; idx < C * DK; idx += NTH) {
                const int r = idx / DK, c = idx % DK;
                const bool ok = r < n;
                const size_t off = ((size_t)(c0 + r) * p.Hq + qh) * DK + c;
                sK[r * KS + c] = __float2half_rn(ok ? kg[off] : 0.f);
                sQ[r * KS + c] = __float2half_rn(ok ? qg[off] : 0.f);
            }
            for (int idx = tid; idx < C * VS; idx += NTH) {
                const int r = idx / VS, c = idx % VS;
                const int col = vs0 + c;
                const bool ok = r < n && col < p.dv;
                sV[r * VSS + c] = __float2half_rn(ok ? vg[((size_t)(c0 + r) * p.Hv + h) * p.dv + col] : 0.f);
            }
        }
        if (tid < C) {
            const int r = tid;
            float gr = 0.f, br = 0.f;
            if (r < n) {
                const size_t th = (size_t)(c0 + r) * p.Hv + h;
                if (has_decay) {
                    gr = ld_any(p.decay, th, p.decay_f16);
                    if (p.raw_gate) gr = p.gate_scale[h] * softplus_f(gr + p.gate_bias[h]);
                }
                br = 1.f;
                if (beta_scalar || (GDN2 && p.erase_gate)) {
                    br = ld_any(p.beta, beta_at(p, c0 + r, h), p.beta_f16);
                    if (sig) br = sigmoid_f(br);
                }
            }
            sG[r] = gr;
            // GDN-2: beta (its own erase gate given) scales the value rows, not the system
            sBt[r] = GDN2 ? 1.f : br;
            if (GDN2) sVB[r] = br;
        }
        ptx::cp_async_wait_all();
        __syncthreads();

        // ------------------------------------------- L2 norms, kappa, cumulants
        {
            constexpr int EPL = DK >= 32 ? DK / 32 : 1;
            const bool nk = (p.flags & kL2k) != 0, nq = (p.flags & kL2q) != 0;
            if (nk || nq || GDN2) {
                for (int r = warp; r < C; r += NW) {
                    float kv[EPL], qv[EPL];
                    float ssk = 0.f, ssq = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) {
                        const int c = lane * EPL + e;
                        kv[e] = c < DK ? __half2float(sK[r * KS + c]) : 0.f;
                        qv[e] = c < DK ? __half2float(sQ[r * KS + c]) : 0.f;
                        ssk += kv[e] * kv[e];
                        ssq += qv[e] * qv[e];
                    }
                    const float ik = nk ? rsqrtf(warp_sum(ssk) + 1e-12f) : 1.f;
                    const float iq = nq ? rsqrtf(warp_sum(ssq) + 1e-12f) : 1.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) {
                        const int c = lane * EPL + e;
                        if (c < DK) {
                            const float kn = kv[e] * ik;
                            if (nk) sK[r * KS + c] = __float2half_rn(kn);
                            if (nq) sQ[r * KS + c] = __float2half_rn(qv[e] * iq);
                            if (GDN2) {
                                float bb = 0.f;
                                if (r < n) {
                                    const size_t e = ((size_t)(c0 + r) * p.Hv + h) * DK + c;
                                    if (p.erase_gate) {
                                        bb = p.erase_gate[e];
                                    } else {
                                        bb = ld_any(p.beta, e, p.beta_f16);
                                        if (sig) bb = sigmoid_f(bb);
                                    }
                                }
                                sKap[r * KS + c] = __float2half_rn(bb * kn);
                            }
                        }
                    }
                }
            }
            if (GDN2 && scales_v(p)) {
                // v' = beta w .* v (beta of the write when the erase gate is its own input)
                for (int idx = tid; idx < n * VS; idx += NTH) {
                    const int r = idx / VS, c = idx % VS, col = vs0 + c;
                    if (col < p.dv) {
                        float f = sVB[r];
                        if (p.write_gate) f *= p.write_gate[((size_t)(c0 + r) * p.Hv + h) * p.dv + col];
                        sV[r * VSS + c] = __float2half_rn(__half2float(sV[r * VSS + c]) * f);
                    }
                }
            }
            if (warp == 0) {
                // inclusive scan of g over the 64 tokens (2 per lane)
                const float g0 = sG[2 * lane], g1 = sG[2 * lane + 1];
                float s = g0 + g1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, s, o);
                    if (lane >= o) s += y;
                }
                const float G1 = s, G0 = s - g1;
                const float GC = __shfl_sync(0xffffffffu, s, 31);
                sG[2 * lane] = G0;
                sG[2 * lane + 1] = G1;
                sEG[2 * lane] = expf(G0);
                sEG[2 * lane + 1] = expf(G1);
                sEGC[2 * lane] = expf(GC - G0);
                sEGC[2 * lane + 1] = expf(GC - G1);
            }
        }
        __syncthreads();

        const __half *Dp = sV;  // Delta (rows = tokens), V for rules without retrieval
        if (retrieval) {
            // ------------------------------------ A = Kappa K^T (rows of this warp)
            const __half *Xs = GDN2 ? sKap : sK;
            {
                float acc[8][4];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < KST; ++ks) {
                    uint32_t a[4];
                    ptx::ldsm_x4(a, Xs + (16 * warp + (lane & 15)) * KS + 16 * ks + (lane >> 4) * 8);
#pragma unroll
                    for (int np = 0; np < 4; ++np) {
                        if (np <= warp) {
                            uint32_t bb[4];
                            ptx::ldsm_x4(bb, sK + (16 * np + (lane & 7) + ((lane >> 4) << 3)) * KS + 16 * ks +
                                                 ((lane >> 3) & 1) * 8);
                            ptx::mma16816(acc[2 * np], a, bb[0], bb[1]);
                            ptx::mma16816(acc[2 * np + 1], a, bb[2], bb[3]);
                        }
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int r = 16 * warp + g + 8 * hf, j = 8 * nt + 2 * t4 + e;
                            float v = 0.f;
                            if (j < r) v = sBt[r] * expf(sG[r] - sG[j]) * acc[nt][2 * hf + e];
                            sAf[r * FS + j] = v;
                        }
            }
            __syncthreads();

            // ------------------------------------ T = (I + A)^-1, 16x16 blocks
            if (lane < 16) {
                float x[16];
                const float *Ab = sAf + (16 * warp) * FS + 16 * warp;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float s = (i == lane) ? 1.f : 0.f;
#pragma unroll
                    for (int j = 0; j < i; ++j) s -= Ab[i * FS + j] * x[j];
                    x[i] = s;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) sTf[(16 * warp + i) * FS + 16 * warp + lane] = x[i];
            }
            __syncthreads();
            for (int d = 1; d < 4; ++d) {
                const int jb = warp, ib = warp + d;
                if (ib < 4) {
                    const int rr = lane >> 1, cc0 = (lane & 1) * 8;
                    float xs[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) xs[e] = 0.f;
                    for (int m = jb; m < ib; ++m) {
#pragma unroll 4
                        for (int q = 0; q < 16; ++q) {
                            const float a = sAf[(16 * ib + rr) * FS + 16 * m + q];
                            const float *tr = sTf + (16 * m + q) * FS + 16 * jb + cc0;
#pragma unroll
                            for (int e = 0; e < 8; ++e) xs[e] += a * tr[e];
                        }
                    }
                    float *X = sX16 + warp * 16 * 17;
#pragma unroll
                    for (int e = 0; e < 8; ++e) X[rr * 17 + cc0 + e] = xs[e];
                    __syncwarp();
                    float ts[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) ts[e] = 0.f;
                    for (int q = 0; q <= rr; ++q) {
                        const float t = sTf[(16 * ib + rr) * FS + 16 * ib + q];
#pragma unroll
                        for (int e = 0; e < 8; ++e) ts[e] += t * X[q * 17 + cc0 + e];
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) sTf[(16 * ib + rr) * FS + 16 * jb + cc0 + e] = -ts[e];
                    __syncwarp();
                }
                __syncthreads();
            }
            for (int idx = tid; idx < C * C; idx += NTH) {
                const int r = idx / C, j = idx % C;
                const float t = j <= r ? sTf[r * FS + j] : 0.f;
                const float bj = GDN2 ? 1.f : sBt[j];
                sTa[r * CS + j] = __float2half_rn(t * bj * sEG[j]);
                sTb[r * CS + j] = __float2half_rn(t * bj);
            }
            __syncthreads();

            // ------------------------------------ W (rows of this warp) and U' (own columns)
            {
                float accW[NT8][4];
#pragma unroll
                for (int i = 0; i < NT8; ++i) accW[i][0] = accW[i][1] = accW[i][2] = accW[i][3] = 0.f;
                const __half *Bs = GDN2 ? sKap : sK;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    if (ks <= warp) {
                        uint32_t a[4];
                        ptx::ldsm_x4(a, sTa + (16 * warp + (lane & 15)) * CS + 16 * ks + (lane >> 4) * 8);
#pragma unroll
                        for (int np = 0; np < KST; ++np) {
                            uint32_t bb[4];
                            ptx::ldsm_x4_t(bb, Bs + (16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8) * KS + 16 * np +
                                                   (lane >> 4) * 8);
                            ptx::mma16816(accW[2 * np], a, bb[0], bb[1]);
                            ptx::mma16816(accW[2 * np + 1], a, bb[2], bb[3]);
                        }
                    }
                }
                // stored negated, so that Delta = U' + (-W) M0^T accumulates in place
#pragma unroll
                for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int r = 16 * warp + g + 8 * hf, col = 8 * nt + 2 * t4;
                        *reinterpret_cast<uint32_t *>(sW + r * KS + col) =
                            ptx::pack_h2(-accW[nt][2 * hf], -accW[nt][2 * hf + 1]);
                    }
            }
            float accU[4][2][4];
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int i = 0; i < 2; ++i) accU[mt][i][0] = accU[mt][i][1] = accU[mt][i][2] = accU[mt][i][3] = 0.f;
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int ks = 0; ks <= mt; ++ks) {
                    uint32_t a[4], bb[4];
                    ptx::ldsm_x4(a, sTb + (16 * mt + (lane & 15)) * CS + 16 * ks + (lane >> 4) * 8);
                    ptx::ldsm_x4_t(bb, sV + (16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8) * VSS + 16 * warp +
                                           (lane >> 4) * 8);
                    ptx::mma16816(accU[mt][0], a, bb[0], bb[1]);
                    ptx::mma16816(accU[mt][1], a, bb[2], bb[3]);
                }
            __syncthreads();  // sW complete

            // ------------------------------------ Delta = U' - W M0^T (own columns)
#pragma unroll
            for (int ks = 0; ks < KST; ++ks) {
                const uint32_t b0lo = ptx::pack_h2(S[2 * ks][0], S[2 * ks][1]);
                const uint32_t b1lo = ptx::pack_h2(S[2 * ks + 1][0], S[2 * ks + 1][1]);
                const uint32_t b0hi = ptx::pack_h2(S[2 * ks][2], S[2 * ks][3]);
                const uint32_t b1hi = ptx::pack_h2(S[2 * ks + 1][2], S[2 * ks + 1][3]);
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    uint32_t a[4];
                    ptx::ldsm_x4(a, sW + (16 * mt + (lane & 15)) * KS + 16 * ks + (lane >> 4) * 8);
                    ptx::mma16816(accU[mt][0], a, b0lo, b1lo);
                    ptx::mma16816(accU[mt][1], a, b0hi, b1hi);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int r = 16 * mt + g + 8 * hf, col = 16 * warp + 8 * nt + 2 * t4;
                        const float d0 = accU[mt][nt][2 * hf], d1 = accU[mt][nt][2 * hf + 1];
                        *reinterpret_cast<uint32_t *>(sD + r * VSS + col) = ptx::pack_h2(d0, d1);
                        const float e = sEGC[r];
                        *reinterpret_cast<uint32_t *>(sDt + r * VSS + col) = ptx::pack_h2(d0 * e, d1 * e);
                    }
            Dp = sD;
        } else {
            // Delta = V: only the decayed copy is needed for the state update
            for (int idx = tid; idx < C * (VS / 2); idx += NTH) {
                const int r = idx / (VS / 2), c = 2 * (idx % (VS / 2));
                const __half2 v2 = *reinterpret_cast<const __half2 *>(sV + r * VSS + c);
                const float2 vf = __half22float2(v2);
                const float e = sEGC[r];
                *reinterpret_cast<uint32_t *>(sDt + r * VSS + c) = ptx::pack_h2(vf.x * e, vf.y * e);
            }
        }

        // ------------------------------------ P = (Q K^T) masked and decayed
        {
            float acc[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KST; ++ks) {
                uint32_t a[4];
                ptx::ldsm_x4(a, sQ + (16 * warp + (lane & 15)) * KS + 16 * ks + (lane >> 4) * 8);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    if (np <= warp) {
                        uint32_t bb[4];
                        ptx::ldsm_x4(bb, sK + (16 * np + (lane & 7) + ((lane >> 4) << 3)) * KS + 16 * ks +
                                             ((lane >> 3) & 1) * 8);
                        ptx::mma16816(acc[2 * np], a, bb[0], bb[1]);
                        ptx::mma16816(acc[2 * np + 1], a, bb[2], bb[3]);
                    }
                }
            }
            __syncthreads();  // region 2 (Ta/Tb) is free; Delta tiles are complete
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int r = 16 * warp + g + 8 * hf, j = 8 * nt + 2 * t4;
                    const float v0 = j <= r ? expf(sG[r] - sG[j]) * acc[nt][2 * hf] : 0.f;
                    const float v1 = j + 1 <= r ? expf(sG[r] - sG[j + 1]) * acc[nt][2 * hf + 1] : 0.f;
                    *reinterpret_cast<uint32_t *>(sP + r * CS + j) = ptx::pack_h2(v0, v1);
                }
        }
        __syncthreads();

        // ------------------------------------ O = scale (diag(e^G) Q M0^T + P Delta)
        {
            float accO[4][2][4];
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int i = 0; i < 2; ++i) accO[mt][i][0] = accO[mt][i][1] = accO[mt][i][2] = accO[mt][i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KST; ++ks) {
                const uint32_t b0lo = ptx::pack_h2(S[2 * ks][0], S[2 * ks][1]);
                const uint32_t b1lo = ptx::pack_h2(S[2 * ks + 1][0], S[2 * ks + 1][1]);
                const uint32_t b0hi = ptx::pack_h2(S[2 * ks][2], S[2 * ks][3]);
                const uint32_t b1hi = ptx::pack_h2(S[2 * ks + 1][2], S[2 * ks + 1][3]);
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    uint32_t a[4];
                    ptx::ldsm_x4(a, sQ + (16 * mt + (lane & 15)) * KS + 16 * ks + (lane >> 4) * 8);
                    ptx::mma16816(accO[mt][0], a, b0lo, b1lo);
                    ptx::mma16816(accO[mt][1], a, b0hi, b1hi);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const float elo = sEG[16 * mt + g], ehi = sEG[16 * mt + g + 8];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    accO[mt][nt][0] *= elo, accO[mt][nt][1] *= elo;
                    accO[mt][nt][2] *= ehi, accO[mt][nt][3] *= ehi;
                }
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int ks = 0; ks <= mt; ++ks) {
                    uint32_t a[4], bb[4];
                    ptx::ldsm_x4(a, sP + (16 * mt + (lane & 15)) * CS + 16 * ks + (lane >> 4) * 8);
                    ptx::ldsm_x4_t(bb, Dp + (16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8) * VSS + 16 * warp +
                                           (lane >> 4) * 8);
                    ptx::mma16816(accO[mt][0], a, bb[0], bb[1]);
                    ptx::mma16816(accO[mt][1], a, bb[2], bb[3]);
                }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int r = 16 * mt + g + 8 * hf;
                        const int col = wrow0 + 8 * nt + 2 * t4;
                        if (r < n && col < p.dv) {
                            const float o0 = p.scale * accO[mt][nt][2 * hf], o1 = p.scale * accO[mt][nt][2 * hf + 1];
                            const size_t oi = ((size_t)(c0 + r) * p.Hv + h) * p.dv + col;
                            if (p.act_f16)
                                *reinterpret_cast<__half2 *>(static_cast<__half *>(p.o) + oi) = __floats2half2_rn(o0, o1);
                            else
                                *reinterpret_cast<float2 *>(static_cast<float *>(p.o) + oi) = make_float2(o0, o1);
                        }
                    }
        }

        // ------------------------------------ M <- e^{G_C} M + Delta^T diag(e^{G_C - G}) K
        {
            const float eC = sEG[C - 1];
#pragma unroll
            for (int nt = 0; nt < NT8; ++nt) S[nt][0] *= eC, S[nt][1] *= eC, S[nt][2] *= eC, S[nt][3] *= eC;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t a[4];
                ptx::ldsm_x4_t(a, sDt + (16 * ks + (lane & 7) + (lane >> 4) * 8) * VSS + 16 * warp +
                                      ((lane >> 3) & 1) * 8);
#pragma unroll
                for (int np = 0; np < KST; ++np) {
                    uint32_t bb[4];
                    ptx::ldsm_x4_t(bb, sK + (16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8) * KS + 16 * np +
                                           (lane >> 4) * 8);
                    ptx::mma16816(S[2 * np], a, bb[0], bb[1]);
                    ptx::mma16816(S[2 * np + 1], a, bb[2], bb[3]);
                }
            }
        }
    }

#pragma unroll
    for (int nt = 0; nt < NT8; ++nt) {
        const int col = 8 * nt + 2 * t4;
        if (lo_ok) st_pair(rlo, col, S[nt][0], S[nt][1]);
        if (hi_ok) st_pair(rhi, col, S[nt][2], S[nt][3]);
    }
}

template <int DK, bool GDN2>
cudaError_t launch_mma(const Problem &p, cudaStream_t stream) {
    using Ly = Lay<DK, GDN2>;
    const int slices = (p.dv + VS - 1) / VS;
    const long long grid = (long long)p.B * p.Hv * slices;
    const cudaError_t e = smem_attr((const void *)chunked_mma_kernel<DK, GDN2>, Ly::total);
    if (e != cudaSuccess) return e;
    chunked_mma_kernel<DK, GDN2><<<(unsigned)grid, NTH, Ly::total, stream>>>(p, slices);
    return cudaGetLastError();
}

bool al16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

size_t chunked_workspace_bytes(const Problem &p, int) {
    return chunked_tc_eligible(p) ? chunked_tc_workspace_bytes(p) : 0;
}

size_t chunked_workspace_min_bytes(const Problem &p, int) {
    return chunked_tc_eligible(p) ? chunked_tc_workspace_min_bytes(p) : 0;
}

bool chunked_supported(const Problem &p, int, const char **why) {
    if (!(p.dk == 16 || p.dk == 32 || p.dk == 64 || p.dk == 128)) {
        *why = "head_dim_k must be 16, 32, 64 or 128";
        return false;
    }
    if (p.dv % 16 != 0) {
        *why = "head_dim_v must be a multiple of 16";
        return false;
    }
    if (!al16(p.q) || !al16(p.k) || !al16(p.v) || !al16(p.o) || !al16(p.fin) || (p.init && !al16(p.init))) {
        *why = "q, k, v, o and the state tensors must be 16-byte aligned";
        return false;
    }
    return true;
}

cudaError_t launch_chunked(const Problem &p, int chunk, void *ws, size_t ws_bytes, cudaStream_t stream) {
    (void)chunk;
    if (chunked_tc_eligible(p)) return launch_chunked_tc(p, ws, ws_bytes, stream);
    if ((p.flags & kPerKey) && rule_has_decay(p.rule)) {
        // Per-key decay outside the tcgen05 path's shapes (head sizes other
        // than dk = dv = 128, unaligned rows) runs through the token-serial
        // kernel (same result).
        return launch_recurrent(p, stream);
    }
    const bool g2 = p.rule == kGdn2;
    switch (p.dk) {
        case 16: return g2 ? launch_mma<16, true>(p, stream) : launch_mma<16, false>(p, stream);
        case 32: return g2 ? launch_mma<32, true>(p, stream) : launch_mma<32, false>(p, stream);
        case 64: return g2 ? launch_mma<64, true>(p, stream) : launch_mma<64, false>(p, stream);
        default: return g2 ? launch_mma<128, true>(p, stream) : launch_mma<128, false>(p, stream);
    }
}

}  // namespace gdn
