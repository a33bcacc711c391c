// chunked_tc_perkey.cu -- the prepare pass of the tcgen05 chunked prefill for
// decay per key channel ("aclnnRecurrentGatedDeltaRule" Formula, second form;
// "gatedDeltaUpdate" per-key gate) and for the GDN-2 key-channel erase gate
// (ONNX issue "Spec gap: LinearAttention ... Gated DeltaNet-2", section "The
// GDN-2 recurrence", options A and B of "Proposed extension").  Under option
// B (the erase gate as its own input beside a scalar beta) and with a write
// gate w, GDN-2 is option A on the value rows beta_r w_r .* v_r, which this
// kernel scales in shared memory before the U product.
//
// With per-channel log decay g_t[c], in-chunk cumulants Gamma_t[c] (one per
// key channel), retrieval key kappa_t (= k_t for gated_delta, = b_t .* k_t
// for GDN-2 with beta = 1), normalised keys Kn and queries Qn, the chunk
// algebra of the scalar case keeps its shape once every decay factor is taken
// per channel:
//
//   A_rj = beta_r sum_c kappa_r[c] kn_j[c] e^{Gamma_r[c] - Gamma_j[c]}  (j < r),  T = (I + A)^-1
//   P_rj = scale  sum_c qn_r[c]    kn_j[c] e^{Gamma_r[c] - Gamma_j[c]}  (j <= r)
//   U  = T diag(beta) V,     Wn = -T diag(beta) (e^Gamma .* kappa)
//   Kt = e^{Gamma_C - Gamma} .* Kn,       Qh = scale e^Gamma .* Qn
//   Q' = Qh + P Wn,          E  = Wn^T Kt + Diag(e^{Gamma_C} - 1)   (written as E^T = Kt^T Wn + ...)
//
// and the chain kernel's two lines S <- S + U^T Kt + S E, O^T = U^T P^T + S Q'^T
// are unchanged, so this kernel writes the same operand image as the scalar
// prepare kernel and the same chain kernel consumes it.
//
// The only new difficulty is A and P: a per-channel factor e^{Gamma_r - Gamma_j}
// does not pull out of the channel sum.  The 64 tokens split into four blocks
// of 16.  For row r in block s >= 1 and column j in an earlier block, with the
// reference token rho = 16 s - 1 (j <= rho < r),
//   e^{Gamma_r - Gamma_j} = e^{Gamma_r - Gamma_rho} e^{Gamma_rho - Gamma_j},
// both factors at most 1, so these blocks are plain products of two scaled
// fp16 operands (three tcgen05 products, one per s, M = 128 key and query rows,
// N = 16 s).  The four diagonal 16 x 16 blocks are summed in fp32 on the CUDA
// cores with the factor carried as a running product of per-token decays
// (e^{Gamma_r - Gamma_{j-1}} = e^{Gamma_r - Gamma_j} alpha_j), so nothing
// overflows or loses range however strong the decay.
//
// The gated rule with per-key decay (no retrieval: W = 0) takes the same pass
// without the solve: U = V, Q' = Qh and E = Diag(e^{Gamma_C} - 1), so the
// chain's S E applies the per-channel decay of the chunk.
#include <algorithm>
#include <type_traits>

#include "chunk_image.cuh"
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace gdn {
namespace {

using namespace img;

// ---------------------------------------------------------------------------
// Shared memory (one CTA per SM), offsets from a 1024-byte-aligned base.
constexpr int PK_WORK = 256;
constexpr int PK_THREADS = PK_WORK + 32;
constexpr int kFA = kSolveStride;      // fp32 row stride of At and T
constexpr int pKQ = 0;                 // 32 KB: key / query tiles (TMA); later Wn over the key rows
constexpr int pV = 32768;              // 16 KB: value tile (TMA); later U
constexpr int pG = 49152;              // 32 KB: fp32 [64 t][128 c] log decay -> Gamma -> alpha
constexpr int pXo = 81920;             // 32 KB: A operand of the off-block products; later At, T, Tb, Ta', E
constexpr int pYo = pXo + 32768;       // 24 KB: B operands of the off-block products (16 + 32 + 48 key rows)
constexpr int pXp = pYo + 24576;       // 16 KB: X' = e^Gamma .* kappa_n (B operand of Wn); with pKt the erase-gate landing
constexpr int pKt = pXp + 16384;       // 16 KB: Kt (image layout)
constexpr int pQh = pKt + 16384;       // 16 KB: Qh, then Q' (image layout)
constexpr int pP = pQh + 16384;        //  8 KB: P (image layout)
constexpr int pKap = pP + 8192;        // 16 KB: b .* k (raw keys), GDN-2; [2 c-blocks][64 t][64 c]
constexpr int pSc = pKap + 16384;      // per-token and per-channel factors
constexpr int pGin = pSc + 320 * 4;    // 2 x (scalar log decay, beta, value-row factor) of 64 tokens
constexpr int pHdr = pGin + 2 * 192 * 4;  // 2 x {slot, head, first token, tokens, gate scale}
constexpr int pBar = pHdr + 2 * 8 * 4;    // seven mbarriers, TMEM address
constexpr int pGb = pBar + 96;            // the head's per-key gate bias (raw arm), 128 floats
constexpr int PK_SMEM = pGb + 512 + 1024;
constexpr int pAt = pXo, pTf = pXo + 64 * kFA * 4, pTb = pXo, pTa = pXo + 8192;
static_assert(pTf + 64 * kFA * 4 <= pXp, "perkey layout: solve area");
static_assert(pYo % 1024 == 0 && pXp % 1024 == 0 && pKt % 1024 == 0 && pQh % 1024 == 0 && pP % 1024 == 0 &&
                  pKap % 1024 == 0,
              "perkey layout: swizzled tiles");
static_assert(PK_SMEM <= 227 * 1024, "perkey layout: one CTA per SM");
// factor arrays (offsets in floats from pSc)
constexpr int fB = 0, fIK = 64, fIQ = 128, fGC = 192;  // beta, 1/|k|, 1/|q| per token; Gamma_C per channel
// first row of each off-block B operand group (s = 1, 2, 3) and its tensor-memory column
__device__ __forceinline__ int ystart(int s) { return s == 1 ? 0 : (s == 2 ? 16 : 48); }
constexpr int kYBlk = 96 * 128;        // bytes per 64-channel block of the off-block B operands

// shared-memory offset of 16-byte chunk `ch` (0..15) of key row r / query row r
__device__ __forceinline__ int kq_at(int r, int ch, bool query) {
    return (ch >> 3) * 16384 + (query ? 8192 : 0) + sw(r, ch & 7);
}
// the same for a [2 c-blocks][64 t][64 c] tile (value, Kt, Qh, X', b .* k)
__device__ __forceinline__ int t64(int r, int ch) { return (ch >> 3) * 8192 + sw(r, ch & 7); }

// ln(1 + e^x) for the per-key raw gate, 8192 of them per task: x itself above
// 15 (the correction, below 3.1e-7, is under fp32 resolution of x);
// y (1 - y / 2) with y = e^x below y = 1e-3 (the dropped terms are below
// 3.4e-7 relative); otherwise the fast logarithm of 1 + y, whose error stays
// below 2e-4 relative near y = 1e-3 and near fp32 resolution for y ~ 1.  The
// log decay it feeds is then exact to a few 1e-7 absolute.
__device__ __forceinline__ float softplus_fast(float x) {
    const float y = __expf(x);
    const float r = y < 1e-3f ? y * fmaf(-0.5f, y, 1.f) : __logf(1.f + y);
    return x > 15.f ? x : r;
}
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }

__device__ __forceinline__ void ld8f(const float *p, float *x) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
__device__ __forceinline__ float2 h2f(const unsigned char *p) {
    return __half22float2(*reinterpret_cast<const __half2 *>(p));
}
__device__ __forceinline__ void unpack8(uint4 u, float *x) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 f = __half22float2(h[w]);
        x[2 * w] = f.x, x[2 * w + 1] = f.y;
    }
}

// ---------------------------------------------------------------------------
// chunk_prepare_perkey_kernel: the operand image of every (chunk slot, value
// head).  Persistent CTAs, one per SM: a producer warp and eight worker warps.
// The producer looks up the next task and loads its scalar gates one task
// ahead.  It lands the per-key log-decay rows and the head's gate bias as soon
// as the previous task has finished its diagonal blocks (gfree).  The key,
// query and value tiles (TMA; the gated rule takes no value tile, its chain
// reads v itself) and the erase-gate rows follow once that task's
// last products have read their buffers (tfree), and the task after that is
// prefetched into L2.  So the next task's loads overlap the solve and the
// epilogues of the current one.  Per task the workers
//   1. zero the rows past a short last chunk, apply the raw gate and take the
//      per-channel cumulants Gamma, 1/|k|, 1/|q| and b .* k;
//   2. write Kt, Qh, X' and the scaled operands of the off-block products;
//      issue those products (tensor memory columns [0, 96));
//   3. turn Gamma into per-token decays and sum the diagonal blocks of A and P
//      on the CUDA cores while the products run; then A (fp32, transposed) and
//      P (image layout) from both parts;
//   4. solve T = (I + A)^-1 in fp32 (as the scalar prepare kernel), products
//      U = Tb V and Wn = Ta' X', then Wn^T Kt and P Wn;
//   5. Q' = Qh + P Wn and E = Wn^T Kt + Diag(e^{Gamma_C} - 1) to the image.
// Padding tokens of a short last chunk get zero keys, queries, values, log
// decay and beta, so every operand row or column that belongs to them is zero.
// Waits are bounded; a failed wait sets bit 2 of the error word.
template <bool GDN2>
__global__ void __launch_bounds__(PK_THREADS, 1)
    chunk_prepare_perkey_kernel(Problem p, const __grid_constant__ CUtensorMap tmK,
                                const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmV,
                                const int *offs, const int *slot_req, unsigned char *img, int cap) {
    extern __shared__ unsigned char smraw[];
    const uint32_t sb0 = ptx::smem_u32(smraw);
    unsigned char *sm = smraw + (((sb0 + 1023u) & ~1023u) - sb0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = min(offs[p.B], cap);
    const long long ntasks = (long long)total * p.Hv;
    const bool perkey = (p.flags & kPerKey) != 0;
    float *F = reinterpret_cast<float *>(sm + pSc);
    float *G = reinterpret_cast<float *>(sm + pG);
    // land / tfree: key, query, value tiles and erase-gate rows landed / free again;
    // landG / gfree: the same for the log-decay rows; MMA completions bar2, bar3, barO
    uint64_t *land = reinterpret_cast<uint64_t *>(sm + pBar);
    uint64_t *tfree = land + 1, *bar2 = land + 2, *bar3 = land + 3, *barO = land + 4;
    uint64_t *landG = land + 5, *gfree = land + 6;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + pBar + 64);
    if (tid == 0) {
        for (int i = 0; i < 7; ++i) ptx::mbar_init(&land[i], 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tslot, 256);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    const long long NG = gridDim.x;
    // the GDN-2 erase gate rows (fp32): its own input, or the per-key beta
    const float *erase_rows = p.erase_gate ? p.erase_gate : static_cast<const float *>(p.beta);

    if (warp == 8) {
        // ===================== producer
        struct Next {
            int slot, h, c0, n;
            float gs, g[2], bt[2], bv[2];
        };
        auto fetch = [&](long long t) {
            Next x;
            x.slot = (int)(t / p.Hv), x.h = (int)(t % p.Hv);
            const int b = slot_req[x.slot];
            int t0, t1;
            request_range(p, b, t0, t1);
            x.c0 = t0 + TC_C * (x.slot - offs[b]);
            x.n = min(TC_C, t1 - x.c0);
            x.gs = p.raw_gate ? p.gate_scale[x.h] : 0.f;
            const float gb = (p.raw_gate && !perkey) ? p.gate_bias[x.h] : 0.f;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tt = lane + 32 * e;
                const size_t th = (size_t)(x.c0 + tt) * p.Hv + x.h;
                float g = 0.f, bt = 0.f, bv = 1.f;
                if (tt < x.n) {
                    if (!perkey) {
                        g = ld_any(p.decay, th, p.decay_f16);
                        if (p.raw_gate) g = x.gs * softplus_f(g + gb);
                    }
                    if (GDN2 && !p.erase_gate) {
                        bt = 1.f;
                    } else if (!GDN2 && p.rule == kGated) {
                        bt = 0.f;  // no retrieval: no beta, and the A parts come out zero
                    } else {
                        bt = ld_any(p.beta, beta_at(p, x.c0 + tt, x.h), p.beta_f16);
                        if (p.flags & kBetaSigmoid) bt = sigmoid_f(bt);
                    }
                    // GDN-2 with its own erase gate: beta scales the value row, not the system
                    if (GDN2) bv = bt, bt = 1.f;
                }
                x.g[e] = g, x.bt[e] = bt, x.bv[e] = bv;
            }
            return x;
        };
        // the per-key rows of one task into L2 (two rows of each tensor per lane)
        auto prefetch_rows = [&](const Next &x) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int rr = lane + 32 * e;
                if (rr < x.n) {
                    const size_t th = (size_t)(x.c0 + rr) * p.Hv + x.h;
                    if (perkey) ptx::prefetch_l2(static_cast<const float *>(p.decay) + th * 128, 512);
                    if (GDN2) ptx::prefetch_l2(erase_rows + th * 128, 512);
                    if (GDN2 && p.write_gate) ptx::prefetch_l2(p.write_gate + th * 128, 512);
                }
            }
        };
        Next nx;
        if (blockIdx.x < ntasks) nx = fetch(blockIdx.x);
        if (blockIdx.x < ntasks) prefetch_rows(nx);
        int i = 0;
        for (long long t = blockIdx.x; t < ntasks; t += NG, ++i) {
            // the log-decay rows land once the previous task has finished its diagonal blocks
            if (i > 0 && !ptx::mbar_wait_sleep(gfree, (i - 1) & 1)) {
                if (p.err && lane == 0) atomicOr(p.err, 2);
                break;
            }
            float *gin = reinterpret_cast<float *>(sm + pGin) + (i & 1) * 192;
            int *hdr = reinterpret_cast<int *>(sm + pHdr) + (i & 1) * 8;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                gin[lane + 32 * e] = nx.g[e];
                gin[64 + lane + 32 * e] = nx.bt[e];
                gin[128 + lane + 32 * e] = nx.bv[e];
            }
            if (lane == 0) {
                hdr[0] = nx.slot, hdr[1] = nx.h, hdr[2] = nx.c0, hdr[3] = nx.n;
                hdr[4] = __float_as_int(nx.gs);
            }
            __syncwarp();
            const bool gbias = perkey && p.raw_gate;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(landG, (perkey ? (uint32_t)nx.n * 512u : 0u) + (gbias ? 512u : 0u));
                if (gbias) ptx::bulk_g2s(sm + pGb, p.gate_bias + (size_t)nx.h * 128, 512, landG);
            }
            __syncwarp();
            if (perkey) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int rr = lane + 32 * e;
                    if (rr < nx.n) {
                        const size_t th = (size_t)(nx.c0 + rr) * p.Hv + nx.h;
                        ptx::bulk_g2s(sm + pG + rr * 512, static_cast<const float *>(p.decay) + th * 128, 512, landG);
                    }
                }
            }
            // the other tiles once the previous task's last products have read them
            if (i > 0 && !ptx::mbar_wait_sleep(tfree, (i - 1) & 1)) {
                if (p.err && lane == 0) atomicOr(p.err, 2);
                break;
            }
            if (lane == 0) {
                const int qh = (int)((long long)nx.h * p.Hq / p.Hv);
                // the gated rule's chain loads U = V from the value input itself
                const bool needv = GDN2 || p.rule != kGated;
                ptx::mbar_arrive_expect_tx(land, (needv ? 3 : 2) * 16384 + (GDN2 ? (uint32_t)nx.n * 512u : 0u));
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    ptx::tma_load_3d(sm + pKQ + kb * 16384, &tmK, 64 * kb, qh, nx.c0, land);
                    ptx::tma_load_3d(sm + pKQ + kb * 16384 + 8192, &tmQ, 64 * kb, qh, nx.c0, land);
                    if (needv) ptx::tma_load_3d(sm + pV + kb * 8192, &tmV, 64 * kb, nx.h, nx.c0, land);
                }
            }
            __syncwarp();
            if (GDN2) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int rr = lane + 32 * e;
                    if (rr < nx.n) {
                        const size_t th = (size_t)(nx.c0 + rr) * p.Hv + nx.h;
                        ptx::bulk_g2s(sm + pXp + rr * 512, erase_rows + th * 128, 512, land);
                    }
                }
            }
            if (t + NG < ntasks) {
                nx = fetch(t + NG);
                prefetch_rows(nx);
                if (lane == 0) {
                    const int qh = (int)((long long)nx.h * p.Hq / p.Hv);
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb) {
                        ptx::prefetch_tile_3d(&tmK, 64 * kb, qh, nx.c0);
                        ptx::prefetch_tile_3d(&tmQ, 64 * kb, qh, nx.c0);
                        ptx::prefetch_tile_3d(&tmV, 64 * kb, nx.h, nx.c0);
                    }
                }
            }
        }
    } else {
        // ===================== workers (256 threads)
        const int q = warp & 3;    // tensor-memory lane quarter of this warp
        const int hh = warp >> 2;  // column half of this warp in the epilogues
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const int ra = 16 * q + (lane >> 2), rb = ra + 8, cp = 2 * (lane & 3);
        const uint32_t aKQ = ptx::smem_u32(sm + pKQ), aV = ptx::smem_u32(sm + pV);
        const uint32_t aKt = ptx::smem_u32(sm + pKt), aP = ptx::smem_u32(sm + pP);
        const uint32_t aTb = ptx::smem_u32(sm + pTb), aTa = ptx::smem_u32(sm + pTa);
        const uint32_t aXo = ptx::smem_u32(sm + pXo), aYo = ptx::smem_u32(sm + pYo);
        const uint32_t aXp = ptx::smem_u32(sm + pXp);
        // shared-memory descriptors built once; each product advances them (desc_adv)
        const uint64_t d_aKQ_16384 = tc::desc_sw128(aKQ, 16384);
        const uint64_t d_aKt_8192 = tc::desc_sw128(aKt, 8192);
        const uint64_t d_aP = tc::desc_sw128(aP);
        const uint64_t d_aTa = tc::desc_sw128(aTa);
        const uint64_t d_aTb = tc::desc_sw128(aTb);
        const uint64_t d_aV_8192 = tc::desc_sw128(aV, 8192);
        const uint64_t d_aXo = tc::desc_sw128(aXo);
        const uint64_t d_aXp_8192 = tc::desc_sw128(aXp, 8192);
        const uint64_t d_aYo = tc::desc_sw128(aYo);
        float *At = reinterpret_cast<float *>(sm + pAt);
        float *Tf = reinterpret_cast<float *>(sm + pTf);
        const bool nk = (p.flags & kL2k) != 0, nq = (p.flags & kL2q) != 0;
        bool ok = true;
        uint32_t ph = 0;
        int i = 0;
        for (long long t = blockIdx.x; t < ntasks; t += NG, ++i) {
            // the previous task's last image copies (Q', E) have read their staging areas
            if (tid == 0) ptx::bulk_wait_read();
            ok = ptx::named_bar_and(3, PK_WORK,
                                    ptx::mbar_wait_sleep(landG, i & 1) && ptx::mbar_wait_sleep(land, i & 1));
            if (!ok) break;
            const float *gin = reinterpret_cast<const float *>(sm + pGin) + (i & 1) * 192;
            const int *hdr = reinterpret_cast<const int *>(sm + pHdr) + (i & 1) * 8;
            const int slot = hdr[0], h = hdr[1], n = hdr[3];
            const float gs = __int_as_float(hdr[4]);
            unsigned char *dst = img + ((size_t)slot * p.Hv + h) * IM_BYTES;
            // ---- 1. rows past a short last chunk hold other tokens (or nothing): clear them
            if (n < TC_C) {
                const int nz = (TC_C - n) * 16;  // 16-byte chunks of one fp16 tile's cleared rows
                for (int idx = tid; idx < 3 * nz; idx += PK_WORK) {
                    const int which = idx / nz, rem = idx % nz, r = n + (rem >> 4), ch = rem & 15;
                    const int off = which == 2 ? pV + t64(r, ch) : pKQ + kq_at(r, ch, which == 1);
                    *reinterpret_cast<uint4 *>(sm + off) = make_uint4(0, 0, 0, 0);
                }
                const int ng = (TC_C - n) * 32;  // the same for the fp32 [64][128] row tiles
                for (int idx = tid; idx < 2 * ng; idx += PK_WORK) {
                    const int which = idx / ng, rem = idx % ng, r = n + (rem >> 5), cc = rem & 31;
                    if (which == 0 ? perkey : GDN2)
                        *reinterpret_cast<uint4 *>(sm + (which == 0 ? pG : pXp) + r * 512 + cc * 16) =
                            make_uint4(0, 0, 0, 0);
                }
                ptx::named_bar_sync(3, PK_WORK);
            }
            if (GDN2 && scales_v(p)) {
                // v' = beta_r w_r .* v_r in the value tile (fp16, image layout); thread = four
                // 16-byte chunks (8 value channels each) of the rows below n
                const int c0 = hdr[2];
                for (int idx = tid; idx < n * 16; idx += PK_WORK) {
                    const int r = idx >> 4, ch = idx & 15;
                    const float f = gin[128 + r];
                    float x[8];
                    uint4 *cell = reinterpret_cast<uint4 *>(sm + pV + t64(r, ch));
                    unpack8(*cell, x);
                    if (p.write_gate) {
                        float w[8];
                        ld8f(p.write_gate + ((size_t)(c0 + r) * p.Hv + h) * 128 + 8 * ch, w);
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] *= f * w[e];
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] *= f;
                    }
                    uint4 u;
                    u.x = ptx::pack_h2(x[0], x[1]), u.y = ptx::pack_h2(x[2], x[3]);
                    u.z = ptx::pack_h2(x[4], x[5]), u.w = ptx::pack_h2(x[6], x[7]);
                    *cell = u;
                }
                // (the U product reads the tile after several barriers of the workers)
            }
            // gates: thread = (channel c, half of the tokens); the inclusive cumulative sum
            // Gamma of the log decays per channel, in place
            const int gc = tid & 127, ghf = tid >> 7;
            {
                float gv[32];
                if (perkey) {
                    const float gb = p.raw_gate ? reinterpret_cast<const float *>(sm + pGb)[gc] : 0.f;
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt) gv[tt] = G[(32 * ghf + tt) * 128 + gc];
                    if (p.raw_gate) {
#pragma unroll
                        for (int tt = 0; tt < 32; ++tt) gv[tt] = gs * softplus_fast(gv[tt] + gb);
                    }
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt)
                        if (32 * ghf + tt >= n) gv[tt] = 0.f;
                    if (!p.raw_gate && p.err) {
                        // this path needs log decays <= 0 (its operand factors are then at most 1)
                        bool bad = false;
#pragma unroll
                        for (int tt = 0; tt < 32; ++tt) bad |= gv[tt] > 0.f;
                        if (bad) atomicOr(p.err, kErrDecayRange);
                    }
                } else {
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt) gv[tt] = gin[32 * ghf + tt];
                }
                float run = 0.f;
#pragma unroll
                for (int tt = 0; tt < 32; ++tt) {
                    run += gv[tt];
                    G[(32 * ghf + tt) * 128 + gc] = run;
                }
                if (warp == 0) {
                    F[fB + lane] = gin[64 + lane];
                    F[fB + 32 + lane] = gin[96 + lane];
                }
            }
            // 1 / |k| and 1 / |q| per row (warp = 16 of the 128 key and query rows: warps 0-3 keys,
            // 4-7 queries; lane = 4 channels); for GDN-2 also b .* k of the key rows (raw keys),
            // fp16.  All loads first, then the sums, then the stores.
            {
                const bool qrow = warp >= 4;
                uint2 u[16];
#pragma unroll
                for (int k8 = 0; k8 < 16; ++k8) {
                    const int r = (16 * warp + k8) & 63;
                    u[k8] = *reinterpret_cast<const uint2 *>(sm + pKQ + kq_at(r, lane >> 1, qrow) + (lane & 1) * 8);
                }
                float inv[16];
#pragma unroll
                for (int k8 = 0; k8 < 16; ++k8) {
                    const float2 x0 = __half22float2(*reinterpret_cast<const __half2 *>(&u[k8].x));
                    const float2 x1 = __half22float2(*reinterpret_cast<const __half2 *>(&u[k8].y));
                    inv[k8] = x0.x * x0.x + x0.y * x0.y + x1.x * x1.x + x1.y * x1.y;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int k8 = 0; k8 < 16; ++k8) inv[k8] += __shfl_xor_sync(0xffffffffu, inv[k8], o);
                if (GDN2 && !qrow) {
                    float4 bb[16];
#pragma unroll
                    for (int k8 = 0; k8 < 16; ++k8)
                        bb[k8] = *reinterpret_cast<const float4 *>(sm + pXp + (16 * warp + k8) * 512 + lane * 16);
                    const bool sg = (p.flags & kBetaSigmoid) != 0 && !p.erase_gate;
#pragma unroll
                    for (int k8 = 0; k8 < 16; ++k8) {
                        float4 c = bb[k8];
                        if (sg) {
                            c.x = sigmoid_fast(c.x), c.y = sigmoid_fast(c.y);
                            c.z = sigmoid_fast(c.z), c.w = sigmoid_fast(c.w);
                        }
                        const float2 x0 = __half22float2(*reinterpret_cast<const __half2 *>(&u[k8].x));
                        const float2 x1 = __half22float2(*reinterpret_cast<const __half2 *>(&u[k8].y));
                        u[k8].x = ptx::pack_h2(c.x * x0.x, c.y * x0.y);
                        u[k8].y = ptx::pack_h2(c.z * x1.x, c.w * x1.y);
                    }
#pragma unroll
                    for (int k8 = 0; k8 < 16; ++k8)
                        *reinterpret_cast<uint2 *>(sm + pKap + t64(16 * warp + k8, lane >> 1) + (lane & 1) * 8) = u[k8];
                }
                const bool nrm = qrow ? nq : nk;
                if (lane < 16) {
                    float x = inv[0];
#pragma unroll
                    for (int k8 = 1; k8 < 16; ++k8) x = lane == k8 ? inv[k8] : x;
                    F[(qrow ? fIQ : fIK) + ((16 * warp + lane) & 63)] = nrm ? rsqrtf(x + 1e-12f) : 1.f;
                }
            }
            ptx::named_bar_sync(3, PK_WORK);
            if (ghf == 1) {  // the second half of the tokens continues the first half's sums
                const float add = G[31 * 128 + gc];
#pragma unroll 8
                for (int tk = 32; tk < 64; ++tk) G[tk * 128 + gc] += add;
                F[fGC + gc] = G[63 * 128 + gc];
            }
            ptx::named_bar_sync(3, PK_WORK);

            // ---- 2. Kt, Qh, X' and the operands of the off-block products, thread = (row, 8 channels)
            {
                const float sc = p.scale;
#pragma unroll 1
                for (int w = 0; w < 4; ++w) {
                    const int idx = tid + PK_WORK * w, R = idx >> 4, ch = idx & 15, c0 = 8 * ch;
                    const int s = R >> 4;
                    float gR[8], gC[8], kr[8], qr[8], xr[8];
                    ld8f(G + R * 128 + c0, gR);
                    ld8f(F + fGC + c0, gC);
                    unpack8(*reinterpret_cast<const uint4 *>(sm + pKQ + kq_at(R, ch, false)), kr);
                    unpack8(*reinterpret_cast<const uint4 *>(sm + pKQ + kq_at(R, ch, true)), qr);
                    if (GDN2) {
                        unpack8(*reinterpret_cast<const uint4 *>(sm + pKap + t64(R, ch)), xr);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) xr[e] = kr[e];
                    }
                    const float ik = F[fIK + R], iq = F[fIQ + R], bR = F[fB + R];
                    float a[8], b[8], c[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float eg = __expf(gR[e]);
                        a[e] = __expf(gC[e] - gR[e]) * ik * kr[e];  // Kt
                        b[e] = sc * iq * eg * qr[e];                 // Qh
                        c[e] = eg * ik * xr[e];                      // X'
                    }
                    st_chunk(sm + pKt + (ch >> 3) * 8192, R, ch & 7, a);
                    st_chunk(sm + pQh + (ch >> 3) * 8192, R, ch & 7, b);
                    st_chunk(sm + pXp + (ch >> 3) * 8192, R, ch & 7, c);
                    // A operand rows: beta_r kappa_r and scale q_r, both times e^{Gamma_r - Gamma_rho},
                    // rho = 16 s - 1 (zero in block 0, which has no earlier block)
                    if (s > 0) {
                        float gr0[8];
                        ld8f(G + (16 * s - 1) * 128 + c0, gr0);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float f = __expf(gR[e] - gr0[e]);
                            a[e] = bR * ik * xr[e] * f;
                            b[e] = sc * iq * qr[e] * f;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) a[e] = b[e] = 0.f;
                    }
                    st_chunk(sm + pXo + (ch >> 3) * 16384, R, ch & 7, a);
                    st_chunk(sm + pXo + (ch >> 3) * 16384 + 8192, R, ch & 7, b);
                    // B operand rows: k_j e^{Gamma_rho - Gamma_j} for every later block's reference
                    for (int s2 = s + 1; s2 <= 3; ++s2) {
                        float gr2[8];
                        ld8f(G + (16 * s2 - 1) * 128 + c0, gr2);
#pragma unroll
                        for (int e = 0; e < 8; ++e) c[e] = ik * kr[e] * __expf(gr2[e] - gR[e]);
                        st_chunk(sm + pYo + (ch >> 3) * kYBlk, ystart(s2) + R, ch & 7, c);
                    }
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, PK_WORK);
            if (tid == 0) {
                tc::fence_after();
                // off-block products: for s = 1, 2, 3, [A rows; P rows] (M = 128) times the 16 s key
                // rows of group s (N = 16 s), K = 128 channels, into columns [ystart(s), + 16 s)
#pragma unroll
                for (int s2 = 1; s2 <= 3; ++s2) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t ao = (ks >> 2) * 16384 + (ks & 3) * 32;
                        const uint32_t bo = (ks >> 2) * kYBlk + ystart(s2) * 128 + (ks & 3) * 32;
                        tc::mma_f16(tmem + (uint32_t)ystart(s2), tc::desc_adv(d_aXo, ao), tc::desc_adv(d_aYo, bo),
                                    tc::idesc_f16(128, 16 * s2), ks > 0);
                    }
                }
                tc::commit(barO);
            }

            // ---- 3. Gamma -> per-token decays alpha_t = e^{Gamma_t - Gamma_{t-1}}, in place
            {
                float gv[33];
                gv[0] = ghf ? G[31 * 128 + gc] : 0.f;
#pragma unroll
                for (int tt = 0; tt < 32; ++tt) gv[tt + 1] = G[(32 * ghf + tt) * 128 + gc];
                ptx::named_bar_sync(3, PK_WORK);
#pragma unroll
                for (int tt = 0; tt < 32; ++tt) G[(32 * ghf + tt) * 128 + gc] = __expf(gv[tt + 1] - gv[tt]);
                ptx::named_bar_sync(3, PK_WORK);
            }
            // diagonal blocks of A and P: thread = (block s, rows rp and rp + 8 of it, channel group
            // cg: the pairs 16 m + 2 cg, + 1 for m = 0..7), so every thread has one short and one
            // long row; the factor e^{Gamma_R - Gamma_J} runs down J from R as a product of
            // per-token decays, two channels at a time (packed fp32x2)
            const int ds = warp >> 1, drp = 4 * (warp & 1) + (lane >> 3), dcg = lane & 7;
            const int dR1 = 16 * ds + drp, dR2 = dR1 + 8;
            float2 A1[8], P1[8], A2[16], P2[16];
            // the gated rule has no retrieval: its A parts are zero, so its loop sums P alone
            const bool with_a = GDN2 || p.rule != kGated;
            auto diag = [&](auto wa_tag) {
                constexpr bool WA = decltype(wa_tag)::value;
#pragma unroll
                for (int e = 0; e < 8; ++e) A1[e] = P1[e] = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < 16; ++e) A2[e] = P2[e] = make_float2(0.f, 0.f);
                const int bo = 4 * (dcg & 3);
#pragma unroll 1
                for (int m = 0; m < 8; ++m) {
                    const int ic = 2 * m + (dcg >> 2);  // the 16-byte chunk of channels 16 m + 2 cg, + 1
                    const int xo1 = GDN2 ? pKap + t64(dR1, ic) : pKQ + kq_at(dR1, ic, false);
                    const int xo2 = GDN2 ? pKap + t64(dR2, ic) : pKQ + kq_at(dR2, ic, false);
                    const float2 xk1 = WA ? h2f(sm + xo1 + bo) : make_float2(0.f, 0.f);
                    const float2 xk2 = WA ? h2f(sm + xo2 + bo) : make_float2(0.f, 0.f);
                    const float2 xq1 = h2f(sm + pKQ + kq_at(dR1, ic, true) + bo);
                    const float2 xq2 = h2f(sm + pKQ + kq_at(dR2, ic, true) + bo);
                    // e = 0 above the row's diagonal, 1 on it, then the running product: no branches,
                    // so the loads of every step can run ahead of the product chain
                    float2 e1 = make_float2(0.f, 0.f), e2 = e1;
                    const float2 one = make_float2(1.f, 1.f);
#pragma unroll
                    for (int jl = 15; jl >= 0; --jl) {
                        const int J = 16 * ds + jl;
                        const float2 kk = h2f(sm + pKQ + kq_at(J, ic, false) + bo);
                        const float2 a2 = *reinterpret_cast<const float2 *>(G + J * 128 + 16 * m + 2 * dcg);
                        e2 = jl == drp + 8 ? one : e2;
                        const float2 t2 = __fmul2_rn(kk, e2);
                        if (WA) A2[jl] = __ffma2_rn(xk2, t2, A2[jl]);
                        P2[jl] = __ffma2_rn(xq2, t2, P2[jl]);
                        e2 = __fmul2_rn(e2, a2);
                        if (jl < 8) {
                            e1 = jl == drp ? one : e1;
                            const float2 t1 = __fmul2_rn(kk, e1);
                            if (WA) A1[jl & 7] = __ffma2_rn(xk1, t1, A1[jl & 7]);
                            P1[jl & 7] = __ffma2_rn(xq1, t1, P1[jl & 7]);
                            e1 = __fmul2_rn(e1, a2);
                        }
                    }
                }
            };
            if (with_a)
                diag(std::true_type{});
            else
                diag(std::false_type{});
            // sums over the channel pair and the eight channel groups
            float a1[8], p1[8], a2s[16], p2s[16];
#pragma unroll
            for (int e = 0; e < 8; ++e) a1[e] = A1[e].x + A1[e].y, p1[e] = P1[e].x + P1[e].y;
#pragma unroll
            for (int e = 0; e < 16; ++e) a2s[e] = A2[e].x + A2[e].y, p2s[e] = P2[e].x + P2[e].y;
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (with_a) a1[e] += __shfl_xor_sync(0xffffffffu, a1[e], o);
                    p1[e] += __shfl_xor_sync(0xffffffffu, p1[e], o);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    if (with_a) a2s[e] += __shfl_xor_sync(0xffffffffu, a2s[e], o);
                    p2s[e] += __shfl_xor_sync(0xffffffffu, p2s[e], o);
                }
            }
            // the off-block products are done: their operand area takes A
            ok = ptx::named_bar_and(3, PK_WORK, ptx::mbar_wait_sleep(barO, ph));
            if (!ok) break;
            if (tid == 0) ptx::mbar_arrive(gfree);  // nothing reads the decays of this task any more
            tc::fence_after();
            {
                const float sc = p.scale;
                const float f1 = F[fB + dR1] * F[fIK + dR1], f2 = F[fB + dR2] * F[fIK + dR2];
                const float g1 = sc * F[fIQ + dR1], g2 = sc * F[fIQ + dR2];
                float ikb[16];  // 1 / |k_J| of this block's columns, read before any store below
#pragma unroll
                for (int jl = 0; jl < 16; ++jl) ikb[jl] = F[fIK + 16 * ds + jl];
                // A[R][J] of this block for both rows, stored transposed: lane cg takes columns 2 cg, + 1
#pragma unroll
                for (int jl = 0; jl < 16; ++jl)
                    if ((jl >> 1) == dcg) {
                        const int J = 16 * ds + jl;
                        const float ikJ = ikb[jl];
                        At[J * kFA + dR1] = (jl < 8 && jl < drp) ? f1 * ikJ * a1[jl & 7] : 0.f;
                        At[J * kFA + dR2] = jl < drp + 8 ? f2 * ikJ * a2s[jl] : 0.f;
                    }
                // P rows: this block's two chunks of each row (lanes 0-3), the zero chunks right of
                // the block (lanes 4-7)
                if (dcg < 4) {
                    const bool second = dcg >= 2;
                    const int c = dcg & 1;
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int jl = 8 * c + e;
                        const float ikJ = c == 0 ? ikb[e] : ikb[8 + e];
                        const float v1 = (c == 0 && e <= drp) ? g1 * ikJ * p1[e] : 0.f;
                        const float v2 = c == 0 ? p2s[e] : p2s[8 + e];
                        x[e] = second ? (jl <= drp + 8 ? g2 * ikJ * v2 : 0.f) : v1;
                    }
                    st_chunk(sm + pP, second ? dR2 : dR1, 2 * ds + c, x);
                } else {
                    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    const int row = (dcg & 1) ? dR2 : dR1;
                    for (int ch = 2 * ds + 2 + ((dcg >> 1) & 1); ch < 8; ch += 2) st_chunk(sm + pP, row, ch, z);
                }
            }
            if (warp < 4) {
                // off-block parts: lane = row R (key rows for warps 0, 1: A; query rows for 2, 3: P),
                // its block s >= 1 reads columns [ystart(s), ystart(s) + 16 s)
                const int R = 32 * (q & 1) + lane, s = R >> 4;
                float v[32], w[64];
                tc::ld32(tmem + lane_off, v);
                tc::ld64(tmem + lane_off + 32, w);
#define PK_COL(x) ((x) < 32 ? v[(x)] : w[(x) - 32])
#define PK_OFF(J) (s == 1 ? PK_COL(J) : (s == 2 ? PK_COL(16 + (J)) : PK_COL(48 + (J))))
                if (q < 2) {
#pragma unroll
                    for (int J = 0; J < 48; ++J)
                        if (J < 16 * s) At[J * kFA + R] = PK_OFF(J);
                } else {
#pragma unroll
                    for (int cc = 0; cc < 6; ++cc) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = PK_OFF(8 * cc + e);
                        if (cc < 2 * s) st_chunk(sm + pP, R, cc, x);
                    }
                }
#undef PK_OFF
#undef PK_COL
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, PK_WORK);
            if (tid == 0) {
                ptx::bulk_s2g(dst + IM_P, sm + pP, 8192);
                ptx::bulk_s2g(dst + IM_KT, sm + pKt, 16384);
                ptx::bulk_commit();
            }
            if (!GDN2 && p.rule == kGated) {
                // no retrieval (W = 0): U = V (which the chain loads from the value input), Q' = Qh
                // and E = Diag(e^{Gamma_C} - 1), so the chain's S E scales the state per key channel.  E^T is staged over the solve
                // area (row j = 32 q + lane, columns [64 hh, 64 hh + 64)).
                const int ii = 32 * q + lane;
                float v[64];
#pragma unroll
                for (int e = 0; e < 64; ++e) v[e] = 0.f;
                if (hh == (q >> 1)) {
                    const float gm1 = expm1f(F[fGC + ii]);
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (e == ii - 64 * hh) v[e] = gm1;
                }
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) st_chunk(sm + pXo + hh * 16384, ii, cc, v + 8 * cc);
                tc::fence_async_smem();
                ptx::named_bar_sync(3, PK_WORK);
                if (tid == 0) {
                    ptx::bulk_s2g(dst + im_q(0), sm + pQh, 8192);
                    ptx::bulk_s2g(dst + im_q(1), sm + pQh + 8192, 8192);
                    ptx::bulk_s2g(dst + im_e(0), sm + pXo, 16384);
                    ptx::bulk_s2g(dst + im_e(1), sm + pXo + 16384, 16384);
                    ptx::bulk_commit();
                    // the copies have read their staging areas: the next task's tiles may land
                    ptx::bulk_wait_read();
                    ptx::mbar_arrive(tfree);
                }
                ph ^= 1u;
                continue;
            }

            // ---- 4. T = (I + A)^-1; Tb = T diag(beta) and Ta' = -T diag(beta) (j <= r), fp16,
            // K-major, over the solve area (At is no longer read); thread = (row, 16 columns)
            solve_unit_lower64(At, Tf, tid);
            {
                const int r = tid & 63, j0 = 16 * (tid >> 6);
                float x[16], y[16];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 tv = *reinterpret_cast<const float4 *>(Tf + r * kFA + j0 + 4 * m);
                    const float4 bv = *reinterpret_cast<const float4 *>(F + fB + j0 + 4 * m);
                    const float t4[4] = {tv.x, tv.y, tv.z, tv.w}, b4[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        x[4 * m + e] = j0 + 4 * m + e <= r ? t4[e] * b4[e] : 0.f;
                        y[4 * m + e] = -x[4 * m + e];
                    }
                }
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    st_chunk(sm + pTb, r, (j0 >> 3) + cc, x + 8 * cc);
                    st_chunk(sm + pTa, r, (j0 >> 3) + cc, y + 8 * cc);
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, PK_WORK);
            if (tid == 0) {
                tc::fence_after();
                // U = Tb V -> [0, 128) and Wn = Ta' X' -> [128, 256): M = 64, N = 128, K = 64
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    tc::mma_f16(tmem, tc::desc_adv(d_aTb, s * 32), tc::desc_adv(d_aV_8192, s * 2048),
                                tc::idesc_f16(64, 128, false, true), s > 0);
                    tc::mma_f16(tmem + 128, tc::desc_adv(d_aTa, s * 32), tc::desc_adv(d_aXp_8192, s * 2048),
                                tc::idesc_f16(64, 128, false, true), s > 0);
                }
                tc::commit(bar2);
            }
            ok = ptx::named_bar_and(3, PK_WORK, ptx::mbar_wait_sleep(bar2, ph));
            if (!ok) break;
            tc::fence_after();
            {
                // warps 0-3: U rows into the value tile (image layout); warps 4-7: Wn rows over the
                // key rows (the operand of Wn^T Kt and P Wn)
                const uint32_t col = hh == 0 ? 0u : 128u;
                unsigned char *tile = sm + (hh == 0 ? pV : pKQ);
                const int bstride = hh == 0 ? 8192 : 16384;
                float v[64];
                tc::ld16x256x16(tmem + lane_off + col, v);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    *reinterpret_cast<uint32_t *>(tile + (k >> 3) * bstride + sw(ra, k & 7) + 2 * cp) =
                        ptx::pack_h2(v[4 * k], v[4 * k + 1]);
                    *reinterpret_cast<uint32_t *>(tile + (k >> 3) * bstride + sw(rb, k & 7) + 2 * cp) =
                        ptx::pack_h2(v[4 * k + 2], v[4 * k + 3]);
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, PK_WORK);
            if (tid == 0) {
                ptx::bulk_s2g(dst + IM_U, sm + pV, 16384);
                ptx::bulk_commit();
                tc::fence_after();
                // Kt^T Wn = E^T - Diag(...) -> [0, 128): M = 128 (j), N = 128 (i), K = 64 (t), both
                // operands M/N-major
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tc::mma_f16(tmem, tc::desc_adv(d_aKt_8192, s * 2048), tc::desc_adv(d_aKQ_16384, s * 2048),
                                tc::idesc_f16(128, 128, true, true), s > 0);
                // P Wn -> [128, 256): M = 64 (r), N = 128 (i), K = 64 (t)
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tc::mma_f16(tmem + 128, tc::desc_adv(d_aP, s * 32), tc::desc_adv(d_aKQ_16384, s * 2048),
                                tc::idesc_f16(64, 128, false, true), s > 0);
                tc::commit(bar3);
            }
            ok = ptx::named_bar_and(3, PK_WORK, ptx::mbar_wait_sleep(bar3, ph));
            if (!ok) break;
            if (tid == 0) {
                // the last products have read the key rows (Wn), X' and Kt, and the copies of U, P
                // and Kt their staging areas: the next task's tiles may land
                ptx::bulk_wait_read();
                ptx::mbar_arrive(tfree);
            }
            tc::fence_after();

            // ---- 5. Q' = Qh + P Wn in place (columns [64 hh, 64 hh + 64) of i), and
            // E = Wn^T Kt + Diag(e^{Gamma_C} - 1) staged over the solve area
            {
                float v[32];
                tc::ld16x256<8>(tmem + lane_off + 128 + 64 * hh, v);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    __half2 *pa = reinterpret_cast<__half2 *>(sm + pQh + hh * 8192 + sw(ra, k) + 2 * cp);
                    __half2 *pb = reinterpret_cast<__half2 *>(sm + pQh + hh * 8192 + sw(rb, k) + 2 * cp);
                    const float2 xa = __half22float2(*pa), xb = __half22float2(*pb);
                    *pa = __floats2half2_rn(xa.x + v[4 * k], xa.y + v[4 * k + 1]);
                    *pb = __floats2half2_rn(xb.x + v[4 * k + 2], xb.y + v[4 * k + 3]);
                }
            }
            {
                const int ii = 32 * q + lane;
                float v[64];
                tc::ld64(tmem + lane_off + 64 * hh, v);
                if (hh == (q >> 1)) {  // this warp's rows meet the diagonal at column ii
                    const float gm1 = expm1f(F[fGC + ii]);
                    if (q & 1) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e == lane) v[32 + e] += gm1;
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e == lane) v[e] += gm1;
                    }
                }
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) st_chunk(sm + pXo + hh * 16384, ii, cc, v + 8 * cc);
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, PK_WORK);
            if (tid == 0) {
                ptx::bulk_s2g(dst + im_q(0), sm + pQh, 8192);
                ptx::bulk_s2g(dst + im_q(1), sm + pQh + 8192, 8192);
                ptx::bulk_s2g(dst + im_e(0), sm + pXo, 16384);
                ptx::bulk_s2g(dst + im_e(1), sm + pXo + 16384, 16384);
                ptx::bulk_commit();
            }
            ph ^= 1u;
        }
        if (tid == 0) ptx::bulk_wait();  // every image copy has landed before the CTA leaves
        if (!ok && p.err && tid == 0) atomicOr(p.err, 2);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

}  // namespace
}  // namespace gdn

namespace gdn {

bool chunk_prepare_perkey_eligible(const Problem &p) {
    const bool perkey = (p.flags & kPerKey) != 0;
    const bool rule_ok = p.rule == kGdn2 || ((p.rule == kGatedDelta || p.rule == kGated) && perkey);
    auto al = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    // GDN-2's erase-gate rows land by 512-byte bulk copies: fp32, 16-byte aligned
    const bool erase_ok = p.erase_gate ? al(p.erase_gate) : (!p.beta_f16 && al(p.beta));
    return rule_ok && p.dk == 128 && p.dv == 128 && (!perkey || (!p.decay_f16 && al(p.decay))) &&
           (!perkey || !p.raw_gate || al(p.gate_bias)) && (p.rule != kGdn2 || erase_ok) &&
           (p.write_gate == nullptr || al(p.write_gate));
}

cudaError_t launch_chunk_prepare_perkey(const Problem &p, const CUtensorMap &tk, const CUtensorMap &tq,
                                        const CUtensorMap &tv, const int *offs, const int *slot_req,
                                        unsigned char *img, int cap, cudaStream_t stream) {
    cudaError_t e = smem_attr((const void *)chunk_prepare_perkey_kernel<true>, PK_SMEM);
    if (e != cudaSuccess) return e;
    e = smem_attr((const void *)chunk_prepare_perkey_kernel<false>, PK_SMEM);
    if (e != cudaSuccess) return e;
    // persistent CTAs, one per SM (shared memory), at most one per task
    const long long tasks = (long long)cap * p.Hv;
    const unsigned grid = (unsigned)std::min<long long>(tasks, sm_count());
    if (grid == 0) return cudaSuccess;
    if (p.rule == kGdn2)
        chunk_prepare_perkey_kernel<true><<<grid, PK_THREADS, PK_SMEM, stream>>>(p, tk, tq, tv, offs, slot_req, img,
                                                                                 cap);
    else
        chunk_prepare_perkey_kernel<false><<<grid, PK_THREADS, PK_SMEM, stream>>>(p, tk, tq, tv, offs, slot_req, img,
                                                                                  cap);
    return cudaGetLastError();
}

}  // namespace gdn
