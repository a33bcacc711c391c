// chunked_tc.cu -- chunk-parallel prefill on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), for dk = dv = 128: the offsets
// kernel, the prepare pass for scalar decay (rules linear / gated / delta /
// gated_delta), the chain kernel for every rule (chunked_tc_perkey.cu holds
// the prepare pass for per-key decay and GDN-2) and the launcher, which first
// writes fp16 copies of fp32 activations and fp32 copies of fp16 per-key gate
// rows into the workspace when the problem has them.
//
// Same per-chunk algebra as chunked.cu (derived from the token recurrence;
// see the comment there).  For one chunk of C = 64 tokens, with normalised
// keys Kn, A = strict-lower(diag(beta) e^{G_r - G_j} Kn Kn^T), T = (I + A)^-1,
// Tb = T diag(beta), W = T diag(beta e^G) Kn, U = Tb V:
//
//   D = U - W S^T                 (the token corrections, D^T = U^T - S W^T)
//   O = Qh S^T + P D,             Qh = scale diag(e^G) Qn,  P = decayed causal scale Qn Kn^T
//   S <- e^{G_C} S + D^T Kt,      Kt = diag(e^{G_C - G}) Kn
//
// Substituting D turns one chunk into an affine map of the state:
//
//   S <- S + U^T Kt + S E,        E  = (e^{G_C} - 1) I - W^T Kt     (dk x dk)
//   O^T = U^T P^T + S Q'^T,       Q' = Qh - P W                     (C x dk)
//
// Everything but S in those two lines is state-independent.  So the work
// splits into two kernels: chunk_prepare_kernel builds E, Q', U, P and Kt for
// every (chunk, value head) at once (including the triangular solve), and
// writes them to the workspace already in the 128-byte-swizzled layout the
// tensor cores read; chunk_chain_kernel then walks each (request, value head)
// chunk by chunk with one dependent tensor-core product per chunk (S E; the
// other three do not wait for the state's previous step).  The fp32 state
// lives in tensor memory and is only ever accumulated into: the fp16 copy of
// S enters the products, so the rounding of the old state is scaled by
// (e^{G_C} - 1) and stays at fp16 resolution of one chunk's change.  The
// rules without retrieval take U = V and W = 0.
#include <algorithm>
#include <cuda.h>  // CUtensorMap (the encoder is fetched through the runtime)
#include <cuda_fp16.h>

#include "chunk_image.cuh"
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace gdn {
namespace {

using namespace img;

// number of chunks of request b
__device__ __forceinline__ int request_chunks(const Problem &p, int b) {
    int t0, t1;
    request_range(p, b, t0, t1);
    return (t1 - t0 + TC_C - 1) / TC_C;
}

// ---------------------------------------------------------------------------
// Workspace slots: chunk j of request b has slot offs[b] + j, offs being the
// exclusive prefix sum of the requests' chunk counts (offs[B] = the total);
// slot_req[slot] is the request owning a slot.  order[] lists the requests by
// decreasing chunk count (ties by index) when B <= kSortMax, else in index
// order: the chain kernel starts the longest chains first.  One CTA.
constexpr int kSortMax = 2048;
__global__ void __launch_bounds__(1024) chunk_offsets_kernel(Problem p, int *offs, int *slot_req, int *order, int cap,
                                                             int win_w, int win_W) {
    __shared__ int wsum[32];
    __shared__ int snch[kSortMax];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (p.win) {
        // windowed call: first the window's range of every request, chunks [w W, (w + 1) W) of
        // it, for this kernel and the ones after it (p.win is the output here)
        Problem po = p;
        po.win = nullptr;
        for (int b = tid; b < p.B; b += 1024) {
            int t0, t1;
            request_range(po, b, t0, t1);
            const long long a = (long long)t0 + (long long)win_w * win_W * TC_C, c = a + (long long)win_W * TC_C;
            const_cast<int32_t *>(p.win)[2 * b] = (int)(a < t1 ? a : t1);
            const_cast<int32_t *>(p.win)[2 * b + 1] = (int)(c < t1 ? c : t1);
        }
        __syncthreads();
    }
    const int per = (p.B + 1023) / 1024;
    const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
    int s = 0;
    for (int b = b0; b < b1; ++b) {
        const int nb = request_chunks(p, b);
        s += nb;
        if (p.B <= kSortMax) snch[b] = nb;
    }
    // exclusive block scan of s
    int x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int base = x - s + (warp > 0 ? wsum[warp - 1] : 0);
    for (int b = b0; b < b1; ++b) {
        offs[b] = base;
        const int nb = request_chunks(p, b);
        for (int j = 0; j < nb && base + j < cap; ++j) slot_req[base + j] = b;
        base += nb;
    }
    if (tid == 1023) offs[p.B] = wsum[31];
    if (p.B <= kSortMax) {
        for (int b = tid; b < p.B; b += 1024) {
            const int nb = snch[b];
            int rank = 0;
            for (int b2 = 0; b2 < p.B; ++b2) {
                const int n2 = snch[b2];
                rank += (n2 > nb) || (n2 == nb && b2 < b);
            }
            order[rank] = b;
        }
    } else {
        for (int b = tid; b < p.B; b += 1024) order[b] = b;
    }
}

// ---------------------------------------------------------------------------
// chunk_prepare_kernel: the operand image of every (chunk slot, value head).
//
// Per task, in order (an M = 64 product puts row m on tensor-memory lane
// 32 (m / 16) + m % 16, where the 16x256b load gives thread t of a warp rows
// t / 4 and t / 4 + 8 and the column pairs 2 (t % 4) of every 8; an M = 128
// product puts row m on lane m):
//   1. gates, G = cumulative log decay, beta, 1 / |k|, 1 / |q|; per-token
//      factors; the key rows scaled into Kt (to the image);
//   2. one product [K; Q] K^T (M = 128: the key rows of the delta rules' system
//      and the query rows of P);
//   3. warps on lanes 0-63: A from K K^T;  warps on lanes 64-127: P from Q K^T
//      (to the image);
//   4. all eight warps: the fp32 solve T = (I + A)^-1 (16 x 16 diagonal blocks
//      by substitution, four threads per column, then two recursive-doubling
//      merges [[T0, 0], [L, T1]], L = -T1 A10 T0), written as fp16
//      Tb = T diag(beta) and Ta' = -T diag(beta e^G / |k|);
//   5. products U = Tb V and Wn = Ta' K (= -W);
//   6. U to the image, Wn over the key rows;
//   7. products Wn^T Kt and P Wn;
//   8. Q' = Qh + P Wn (staged over Kt) and E = Wn^T Kt + (e^{G_C} - 1) I to the image.
// The rules without retrieval stop after step 3, with Q' = Qh (U = V, which the
// chain loads from the value input itself); for
// the gated rule the image's E area holds only e^{G_C}.  Padding tokens of a short last chunk get
// zero keys, queries, values, log decay and beta, so every operand row or
// column that belongs to them is zero.
//
// Persistent CTAs, two per SM: a producer warp (task lookup and gates in fp32
// one task ahead, the key / query / value tiles by TMA as soon as the
// previous task releases them; the rules without retrieval take no value tile)
// and eight worker warps.  Waits are bounded.
constexpr int PR_WORK = 256;
constexpr int PR_THREADS = PR_WORK + 32;
constexpr int FA = 68;  // fp32 row stride of At (16-byte rows; lanes = consecutive r, conflict-free)
constexpr int FT = 68;  // fp32 row stride of T (16-byte rows for vector reads)
constexpr int rKQ = 0;                   // 32 KB: 2 blocks (64 channels each) of [64 key rows; 64 query rows]
constexpr int rV = 32768;                // 16 KB: V tile, 2 blocks [64 t][64 v]; later U
constexpr int rAt = 49152;               // fp32 [64][FA], At[j][r] = A[r][j]; later Tb, Ta'; later E
constexpr int rTf = rAt + 64 * FA * 4;   // fp32 [64][FT], T (its unused upper-right block holds Y)
constexpr int rTb = rAt, rTa = rAt + 8192;
constexpr int rKt = 83968;               // 16 KB: Kt, 2 blocks [64 t][64 j]
constexpr int rP = rKt + 16384;          // 8 KB: P [64 r][64 t]
constexpr int rSc = rP + 8192;           // 8 x 64 fp32 per-token factors
constexpr int rGin = rSc + 8 * 64 * 4;   // 2 x (log decay, beta of the 64 tokens), from the producer
constexpr int rHdr = rGin + 2 * 128 * 4; // 2 x {slot, head, first token, tokens}
constexpr int rBar = rHdr + 32;          // land, tiles free, three MMA barriers, TMEM address
constexpr int PR_SMEM = rBar + 64 + 1024;
static_assert(rTf + 64 * FT * 4 <= rKt, "prepare layout");
static_assert(FA == kSolveStride && FT == kSolveStride && PR_WORK == kSolveThreads, "prepare layout: solve");
static_assert(rAt + 32768 <= rKt, "prepare layout: E staging");
static_assert(rKt % 1024 == 0 && rP % 1024 == 0, "prepare layout: swizzled tiles");
static_assert(2 * (PR_SMEM + 1024) <= 228 * 1024, "prepare: two CTAs per SM");
// per-token factor arrays (offsets in floats from rSc)
constexpr int fG = 0, fB = 64, fIK = 128, fIQ = 192, fKF = 256, fTF = 320, fQF = 384, fQS = 448;
// shared-memory offset of 16-byte chunk `ch` (0..15) of key row r / query row r / value row r
__device__ __forceinline__ int kq_off(int r, int ch, bool query) {
    return (ch >> 3) * 16384 + (query ? 8192 : 0) + sw(r, ch & 7);
}

template <bool RETR>
__global__ void __launch_bounds__(PR_THREADS, 2)
    chunk_prepare_kernel(Problem p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmV, const int *offs, const int *slot_req,
                         unsigned char *img, int cap) {
    extern __shared__ unsigned char smraw[];
    const uint32_t sb0 = ptx::smem_u32(smraw);
    unsigned char *sm = smraw + (((sb0 + 1023u) & ~1023u) - sb0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = min(offs[p.B], cap);
    const long long ntasks = (long long)total * p.Hv;
    float *At = reinterpret_cast<float *>(sm + rAt);
    float *Tf = reinterpret_cast<float *>(sm + rTf);
    float *F = reinterpret_cast<float *>(sm + rSc);
    uint64_t *land = reinterpret_cast<uint64_t *>(sm + rBar);
    uint64_t *tfree = land + 1, *bar1 = land + 2, *bar2 = land + 3, *bar3 = land + 4;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + rBar + 48);
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) ptx::mbar_init(&land[i], 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tslot, 256);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    const long long G = gridDim.x;

    if (warp == 8) {
        // ===================== producer.  The task's lookups and gates are loaded into
        // registers while the previous task runs; its tiles are loaded as soon as the
        // previous task has released the key, query and value tiles.
        struct Next {
            int slot, h, c0, n;
            float g[2], bt[2];
        };
        auto fetch = [&](long long t) {
            Next x;
            x.slot = (int)(t / p.Hv), x.h = (int)(t % p.Hv);
            const int b = slot_req[x.slot];
            int t0, t1;
            request_range(p, b, t0, t1);
            x.c0 = t0 + TC_C * (x.slot - offs[b]);
            x.n = min(TC_C, t1 - x.c0);
            const bool raw = rule_has_decay(p.rule) && p.raw_gate;
            const float gs = raw ? p.gate_scale[x.h] : 0.f, gb = raw ? p.gate_bias[x.h] : 0.f;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tt = lane + 32 * e;
                const size_t th = (size_t)(x.c0 + tt) * p.Hv + x.h;
                x.g[e] = (rule_has_decay(p.rule) && tt < x.n) ? ld_any(p.decay, th, p.decay_f16) : 0.f;
                x.bt[e] = (RETR && tt < x.n) ? ld_any(p.beta, beta_at(p, x.c0 + tt, x.h), p.beta_f16) : 0.f;
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if (raw && lane + 32 * e < x.n) x.g[e] = gs * softplus_f(x.g[e] + gb);
                if (RETR && (p.flags & kBetaSigmoid) && lane + 32 * e < x.n) x.bt[e] = sigmoid_f(x.bt[e]);
            }
            return x;
        };
        Next nx;
        if (blockIdx.x < ntasks) nx = fetch(blockIdx.x);
        int i = 0;
        for (long long t = blockIdx.x; t < ntasks; t += G, ++i) {
            if (i > 0 && !ptx::mbar_wait_sleep(tfree, (i - 1) & 1)) {
                if (p.err && lane == 0) atomicOr(p.err, 2);
                break;
            }
            float *gin = reinterpret_cast<float *>(sm + rGin) + (i & 1) * 128;
            int *hdr = reinterpret_cast<int *>(sm + rHdr) + (i & 1) * 4;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                gin[lane + 32 * e] = nx.g[e];
                gin[64 + lane + 32 * e] = nx.bt[e];
            }
            if (lane == 0) hdr[0] = nx.slot, hdr[1] = nx.h, hdr[2] = nx.c0, hdr[3] = nx.n;
            __syncwarp();
            if (lane == 0) {
                const int qh = (int)((long long)nx.h * p.Hq / p.Hv);
                // the rules without retrieval never read the value tile here (U = V)
                ptx::mbar_arrive_expect_tx(land, (RETR ? 3 : 2) * 16384);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    ptx::tma_load_3d(sm + rKQ + kb * 16384, &tmK, 64 * kb, qh, nx.c0, land);
                    ptx::tma_load_3d(sm + rKQ + kb * 16384 + 8192, &tmQ, 64 * kb, qh, nx.c0, land);
                    if (RETR) ptx::tma_load_3d(sm + rV + kb * 8192, &tmV, 64 * kb, nx.h, nx.c0, land);
                }
            }
            if (t + G < ntasks) {
                nx = fetch(t + G);
                if (lane == 0) {  // its tiles into L2 while this task runs
                    const int qh = (int)((long long)nx.h * p.Hq / p.Hv);
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb) {
                        ptx::prefetch_tile_3d(&tmK, 64 * kb, qh, nx.c0);
                        ptx::prefetch_tile_3d(&tmQ, 64 * kb, qh, nx.c0);
                        if (RETR) ptx::prefetch_tile_3d(&tmV, 64 * kb, nx.h, nx.c0);
                    }
                }
            }
        }
    } else {
        // ===================== workers (256 threads)
        const bool nq = (p.flags & kL2q) != 0;
        const bool decay = rule_has_decay(p.rule);
        const int q = warp & 3;    // tensor-memory lane quarter of this warp
        const int hh = warp >> 2;  // column half of this warp in the epilogues
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const int ra = 16 * q + (lane >> 2), rb = ra + 8, cp = 2 * (lane & 3);
        const uint32_t aKQ = ptx::smem_u32(sm + rKQ), aV = ptx::smem_u32(sm + rV);
        const uint32_t aKt = ptx::smem_u32(sm + rKt), aP = ptx::smem_u32(sm + rP);
        const uint32_t aTb = ptx::smem_u32(sm + rTb), aTa = ptx::smem_u32(sm + rTa);
        // shared-memory descriptors built once; each product advances them (desc_adv)
        const uint64_t d_aKQ = tc::desc_sw128(aKQ);
        const uint64_t d_aKQ_16384 = tc::desc_sw128(aKQ, 16384);
        const uint64_t d_aKt_8192 = tc::desc_sw128(aKt, 8192);
        const uint64_t d_aP = tc::desc_sw128(aP);
        const uint64_t d_aTa = tc::desc_sw128(aTa);
        const uint64_t d_aTb = tc::desc_sw128(aTb);
        const uint64_t d_aV_8192 = tc::desc_sw128(aV, 8192);
        bool ok = true;
        uint32_t ph = 0;
        int i = 0;
        for (long long t = blockIdx.x; t < ntasks; t += G, ++i) {
            ok = ptx::named_bar_and(3, PR_WORK, ptx::mbar_wait_sleep(land, i & 1));
            if (!ok) break;
            const float *gin = reinterpret_cast<const float *>(sm + rGin) + (i & 1) * 128;
            const int *hdr = reinterpret_cast<const int *>(sm + rHdr) + (i & 1) * 4;
            const int slot = hdr[0], h = hdr[1], n = hdr[3];
            unsigned char *dst = img + ((size_t)slot * p.Hv + h) * IM_BYTES;
            if (n < TC_C) {  // the boxes run past this request: clear the rows beyond it
                const int nz = (TC_C - n) * 16;
                for (int idx = tid; idx < (RETR ? 3 : 2) * nz; idx += PR_WORK) {
                    const int which = idx / nz, rem = idx % nz, r = n + (rem >> 4), ch = rem & 15;
                    const int off = which == 2 ? rV + (ch >> 3) * 8192 + sw(r, ch & 7) : kq_off(r, ch, which == 1);
                    *reinterpret_cast<uint4 *>(sm + off) = make_uint4(0, 0, 0, 0);
                }
                ptx::named_bar_sync(3, PR_WORK);
            }
            if (warp == 0) {  // G = inclusive cumulative sum of the log decays; beta
                const float x0 = gin[2 * lane], x1 = gin[2 * lane + 1];
                float sacc = x0 + x1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, sacc, o);
                    if (lane >= o) sacc += y;
                }
                F[fG + 2 * lane] = sacc - x1;
                F[fG + 2 * lane + 1] = sacc;
                F[fB + 2 * lane] = gin[64 + 2 * lane];
                F[fB + 2 * lane + 1] = gin[64 + 2 * lane + 1];
            }
            // the previous task's image copies have read their staging areas
            if (tid == 0) ptx::bulk_wait_read();
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, PR_WORK);
            if (tid == 0) {
                tc::fence_after();
                // [K; Q] [K; Q]^T -> columns [0, 128): M = N = 128, K = 128.  Columns [0, 64) hold
                // K K^T over Q K^T; the diagonal holds the squared norms of the key and query rows.
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t o = (s >> 2) * 16384 + (s & 3) * 32;
                    tc::mma_f16(tmem, tc::desc_adv(d_aKQ, o), tc::desc_adv(d_aKQ, o), tc::idesc_f16(128, 128), s > 0);
                }
                tc::commit(bar1);
            }
            ok = ptx::named_bar_and(3, PR_WORK, ptx::mbar_wait_sleep(bar1, ph));
            if (!ok) break;
            tc::fence_after();
            if (warp < 4) {
                // 1 / |k_r| and 1 / |q_r| from the diagonal: row m = 32 q + lane sits on lane m
                float v[32];
                tc::ld32(tmem + lane_off + 32 * q, v);
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (e == lane) d = v[e];
                const int m = 32 * q + lane;
                if (m < TC_C) F[fIK + m] = (p.flags & kL2k) ? rsqrtf(d + 1e-12f) : 1.f;
                else F[fIQ + m - TC_C] = nq ? rsqrtf(d + 1e-12f) : 1.f;
            }
            ptx::named_bar_sync(3, PR_WORK);
            if (tid < TC_C) {
                const float Gt = F[fG + tid], ik = F[fIK + tid], iq = F[fIQ + tid], eg = __expf(Gt);
                F[fKF + tid] = __expf(F[fG + TC_C - 1] - Gt) * ik;  // e^{G_C - G} <= 1
                F[fTF + tid] = -eg * ik;
                F[fQF + tid] = p.scale * eg * iq;
                F[fQS + tid] = p.scale * iq;
            }
            ptx::named_bar_sync(3, PR_WORK);
            // Kt rows = e^{G_C - G_t} k_t / |k_t| into their tile (image layout; the operand of E);
            // without retrieval also Q' = Qh straight to the image
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int idx = tid + PR_WORK * w, tr = idx >> 4, ch = idx & 15;
                const int io = (ch >> 3) * 8192 + sw(tr, ch & 7);  // image (and Kt / V tile) offset
                *reinterpret_cast<uint4 *>(sm + rKt + io) =
                    scale_chunk(*reinterpret_cast<const uint4 *>(sm + kq_off(tr, ch, false)), F[fKF + tr]);
                if (!RETR) {  // (U = V: the chain loads it from the value input)
                    *reinterpret_cast<uint4 *>(dst + im_q(ch >> 3) + sw(tr, ch & 7)) =
                        scale_chunk(*reinterpret_cast<const uint4 *>(sm + kq_off(tr, ch, true)), F[fQF + tr]);
                }
            }
            tc::fence_async_smem();
            if (!RETR) {
                // the gated rule's chain scales the state by e^{G_C} itself: only that goes to the image
                if (decay && tid == 0) *reinterpret_cast<float *>(dst + IM_EQ) = __expf(F[fG + TC_C - 1]);
                ptx::named_bar_sync(3, PR_WORK);
                if (tid == 0) {
                    ptx::bulk_s2g(dst + IM_KT, sm + rKt, 16384);
                    ptx::bulk_commit();
                    // without retrieval nothing reads the key and query tiles any more
                    ptx::mbar_arrive(tfree);
                }
            }
            {
                // thread = row 32 (q % 2) + lane of K K^T (q < 2) or of Q K^T (q >= 2), columns
                // [32 hh, 32 hh + 32)
                const int r = 32 * (q & 1) + lane, j0 = 32 * hh;
                float v[32];
                tc::ld32(tmem + lane_off + j0, v);
                const float Gr = F[fG + r];
                // the factors e^{G_r - G_j} / |k_j| of this thread's 32 columns
                float w[32];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(F + fG + j0 + 4 * m);
                    const float4 i4 = *reinterpret_cast<const float4 *>(F + fIK + j0 + 4 * m);
                    w[4 * m] = __expf(Gr - g4.x) * i4.x;
                    w[4 * m + 1] = __expf(Gr - g4.y) * i4.y;
                    w[4 * m + 2] = __expf(Gr - g4.z) * i4.z;
                    w[4 * m + 3] = __expf(Gr - g4.w) * i4.w;
                }
                if (q >= 2) {
                    // P[r][t] = scale e^{G_r - G_t} q_r . k_t / (|q_r| |k_t|) for t <= r
                    const float qr = F[fQS + r];
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = j0 + e <= r ? qr * w[e] * v[e] : 0.f;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) st_chunk(sm + rP, r, 4 * hh + cc, v + 8 * cc);
                } else if (RETR) {
                    // A[r][j] = beta_r e^{G_r - G_j} k_r . k_j / (|k_r| |k_j|), j < r, stored transposed
                    const float fr = F[fB + r] * F[fIK + r];
#pragma unroll
                    for (int e = 0; e < 32; ++e) At[(j0 + e) * FA + r] = j0 + e < r ? fr * w[e] * v[e] : 0.f;
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, PR_WORK);
            if (tid == 0) {
                ptx::bulk_s2g(dst + IM_P, sm + rP, 8192);
                if (RETR) ptx::bulk_s2g(dst + IM_KT, sm + rKt, 16384);
                ptx::bulk_commit();
            }
            if (!RETR) {
                ph ^= 1u;
                continue;
            }
            solve_unit_lower64(At, Tf, tid);
            {
                // Tb[r][j] = T[r][j] beta_j and Ta'[r][j] = -T[r][j] beta_j e^{G_j} / |k_j| (j <= r),
                // fp16, K-major (the At rows are no longer read); thread = (row, 16 columns)
                const int r = tid & 63, j0 = 16 * (tid >> 6);
                float x[16], y[16];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 tv = *reinterpret_cast<const float4 *>(Tf + r * FT + j0 + 4 * m);
                    const float4 bv = *reinterpret_cast<const float4 *>(F + fB + j0 + 4 * m);
                    const float4 fv = *reinterpret_cast<const float4 *>(F + fTF + j0 + 4 * m);
                    const float t4[4] = {tv.x, tv.y, tv.z, tv.w}, b4[4] = {bv.x, bv.y, bv.z, bv.w};
                    const float f4[4] = {fv.x, fv.y, fv.z, fv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        x[4 * m + e] = j0 + 4 * m + e <= r ? t4[e] * b4[e] : 0.f;
                        y[4 * m + e] = x[4 * m + e] * f4[e];
                    }
                }
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    st_chunk(sm + rTb, r, (j0 >> 3) + cc, x + 8 * cc);
                    st_chunk(sm + rTa, r, (j0 >> 3) + cc, y + 8 * cc);
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, PR_WORK);
            if (tid == 0) {
                tc::fence_after();
                // U = Tb V -> [0, 128) and Wn = Ta' K -> [128, 256): M = 64, N = 128, K = 64
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    tc::mma_f16(tmem, tc::desc_adv(d_aTb, s * 32), tc::desc_adv(d_aV_8192, s * 2048),
                                tc::idesc_f16(64, 128, false, true), s > 0);
                    tc::mma_f16(tmem + 128, tc::desc_adv(d_aTa, s * 32), tc::desc_adv(d_aKQ_16384, s * 2048),
                                tc::idesc_f16(64, 128, false, true), s > 0);
                }
                tc::commit(bar2);
            }
            ok = ptx::named_bar_and(3, PR_WORK, ptx::mbar_wait_sleep(bar2, ph));
            if (!ok) break;
            tc::fence_after();
            {
                // warps 0-3: U rows into the freed value tile (image layout); warps 4-7: Wn rows
                // over the key rows (the operand of Wn^T Kt and P Wn)
                const uint32_t col = hh == 0 ? 0u : 128u;
                unsigned char *tile = sm + (hh == 0 ? rV : rKQ);
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
            ptx::named_bar_sync(3, PR_WORK);
            if (tid == 0) {
                // U to the image (while the last two products run)
                ptx::bulk_s2g(dst + IM_U, sm + rV, 16384);
                ptx::bulk_commit();
                tc::fence_after();
                // Kt^T Wn = (Wn^T Kt)^T -> [0, 128): M = 128 (j), N = 128 (i), K = 64 (t), both
                // operands M/N-major (E^T, the K-major B operand of the chain's S E)
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
            // the copies of Kt and P have read their tiles (Q' goes into the Kt tile)
            if (tid == 0) ptx::bulk_wait_read_all_but_last();
            ok = ptx::named_bar_and(3, PR_WORK, ptx::mbar_wait_sleep(bar3, ph));
            if (!ok) break;
            tc::fence_after();
            {
                // Q' = scale e^{G_r} q_r / |q_r| + (P Wn)_r into the Kt tile, in image layout
                // (columns [64 hh, 64 hh + 64) of i)
                const float fa = F[fQF + ra], fb = F[fQF + rb];
                float v[32];
                tc::ld16x256<8>(tmem + lane_off + 128 + 64 * hh, v);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 xa = __half22float2(
                        *reinterpret_cast<const __half2 *>(sm + rKQ + hh * 16384 + 8192 + sw(ra, k) + 2 * cp));
                    const float2 xb = __half22float2(
                        *reinterpret_cast<const __half2 *>(sm + rKQ + hh * 16384 + 8192 + sw(rb, k) + 2 * cp));
                    *reinterpret_cast<__half2 *>(sm + rKt + hh * 8192 + sw(ra, k) + 2 * cp) =
                        __floats2half2_rn(fmaf(fa, xa.x, v[4 * k]), fmaf(fa, xa.y, v[4 * k + 1]));
                    *reinterpret_cast<__half2 *>(sm + rKt + hh * 8192 + sw(rb, k) + 2 * cp) =
                        __floats2half2_rn(fmaf(fb, xb.x, v[4 * k + 2]), fmaf(fb, xb.y, v[4 * k + 3]));
                }
            }
            tc::fence_async_smem();
            ptx::named_bar_sync(3, PR_WORK);
            if (tid == 0) {
                // the key, query and value tiles are free for the producer's next loads once the
                // copy of U has read the value tile
                ptx::bulk_wait_read();
                ptx::mbar_arrive(tfree);
                ptx::bulk_s2g(dst + im_q(0), sm + rKt, 8192);
                ptx::bulk_s2g(dst + im_q(1), sm + rKt + 8192, 8192);
                ptx::bulk_commit();
            }
            {
                // E^T = Kt^T Wn + (e^{G_C} - 1) I: row j = 32 q + lane, columns i in
                // [64 hh, 64 hh + 64), staged in the At region as [2 i-blocks][128 j][64 i]
                const int ii = 32 * q + lane;
                float v[64];
                tc::ld64(tmem + lane_off + 64 * hh, v);
                if (decay && hh == (q >> 1)) {  // this warp's rows meet the diagonal at column ii
                    const float gm1 = expm1f(F[fG + TC_C - 1]);
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
                for (int cc = 0; cc < 8; ++cc) st_chunk(sm + rAt + hh * 16384, ii, cc, v + 8 * cc);
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(3, PR_WORK);
            if (tid == 0) {
                ptx::bulk_s2g(dst + im_e(0), sm + rAt, 16384);
                ptx::bulk_s2g(dst + im_e(1), sm + rAt + 16384, 16384);
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

// ---------------------------------------------------------------------------
// chunk_chain_kernel: one CTA per (request, value head), longest requests
// first.  The fp32 state S (128 value rows = tensor-memory lanes x 128
// columns) is accumulated in tensor memory; its fp16 copy Sh (K-major, shared
// memory) is the A operand.  Per chunk c, with the chunk's image landed by
// bulk copies (two buffers):
//   UK:    S   += U^T Kt          (state-independent; issued once S_c has been read)
//   UP:    O^T  = U^T P^T         (state-independent; once O^T of chunk c - 1 is read)
//   SE+SQ: [S | O^T] += Sh [E^T; Q']^T   (once Sh = S_c is in shared memory)
// S (columns 0-127) and O^T (columns 128-191) sit side by side in tensor
// memory and the image stores E^T and Q' as one K-major B operand of 192
// rows, so the delta rules' S E and S Q'^T are a single N = 192 product: 8
// instructions where they were 16, with the descriptors built once per chunk
// and advanced per K-step.  What sets the pace, as measured: one K = 16
// instruction costs about max(47, N / 2) cycles on its own, for M = 64 and
// 128 alike, but in this kernel the products run at about 100 cycles per
// N = 128 instruction while the 88 KB image of the next chunk lands in
// shared memory and the state warps write Sh, and a chunk takes about 2.5 K
// cycles whether S E and S Q'^T are fused or issued apart, in either order,
// and whether M is 64 or 128.  The rules without retrieval have no E: SQ
// alone (N = 64), and the gated rule's state warps scale S by e^{G_C} in
// tensor memory when they read it (the prepare kernel leaves e^{G_C} at the
// start of the image's E^T area).  Roles (14 warps): warps 0-7 read S after
// each chunk (thread = value row 32 (warp % 4) + lane, column half warp / 4),
// write Sh and, after the last chunk, the final state; warps 8-11 read O^T
// and store the outputs; warp 12 loads the images; warp 13 issues the
// products.  Hand-overs are mbarriers with bounded, sleeping waits; each role
// makes a failed wait uniform before leaving.
//
// Value rows never mix (S <- S + U^T Kt + S E and O^T = U^T P^T + S Q'^T act
// row by row), so with ROWS = 64 a chain is split over two CTAs, each with
// half the value rows: every product has M = 64 (row m of an M = 64 result
// sits on tensor-memory lane 32 (m / 16) + m % 16, so lanes 16-31 of each
// quarter carry nothing), each CTA loads only its half of U, and twice as
// many SMs work on the same chains.  The launcher splits when there are fewer
// chains than SMs.
constexpr int CH_THREADS = 448;
constexpr int cImg = 0;                       // 2 x IM_BYTES
constexpr int cS = 2 * IM_BYTES;              // 32 KB: Sh, 2 blocks [128 v][64 i]
constexpr int cBar = cS + 32768;              // 12 mbarriers, TMEM address
constexpr int CH_SMEM = cBar + 128 + 1024;
static_assert(cS % 1024 == 0, "chain layout");
// tensor-memory columns: S [0, 128), O^T [128, 192) (and [192, 256): the second O^T buffer of the
// rules without E)
constexpr uint32_t tS = 0, tO = 128;
// what the state step of a rule needs beyond U^T Kt
enum : int { kStepPlain = 0, kStepDecay = 1, kStepE = 2 };

template <int STEP, int ROWS>
__global__ void __launch_bounds__(CH_THREADS, 1)
    chunk_chain_kernel(Problem p, const __grid_constant__ CUtensorMap tmV, const int *offs, const int *order,
                       const unsigned char *img, int cap) {
    constexpr bool HALF = ROWS == 64;
    // Rules without E, split chains: the state S_{c+1} = S_c + U^T Kt (gated: scaled as it is
    // read) does not wait for Sh, so S is published right after U^T Kt and the readout of
    // chunk c runs while the state warps copy S_{c+1}; Sh then alternates between two buffers
    // (they fit in the 32 KB area at ROWS = 64) and its hand-over between two barriers.
    constexpr bool PIPE = HALF && STEP != kStepE;
    // Rules without E: O^T alternates between two tensor-memory buffers, so the readout product
    // of chunk c + 1 does not wait for the output warps to read chunk c (the delta rules' fused
    // product needs O^T beside S: one buffer)
    constexpr bool O2 = STEP != kStepE;
    constexpr int SHB = ROWS * 128;  // bytes per 64-column block of Sh
    extern __shared__ unsigned char smraw[];
    const uint32_t sb0 = ptx::smem_u32(smraw);
    unsigned char *sm = smraw + (((sb0 + 1023u) & ~1023u) - sb0);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + cBar);
    uint64_t *land = bars + 0;    // [2] image landed
    uint64_t *freeb = bars + 2;   // [2] image buffer no longer read
    uint64_t *rsread = bars + 4;  // S_c read by the state warps (one phase per chunk, from c = 0)
    uint64_t *shready = bars + 5; // Sh = S_c written
    uint64_t *barS = bars + 6;    // every product of chunk c done
    uint64_t *barO = bars + 7;    // O^T of chunk c done
    uint64_t *shready2 = bars + 8; // PIPE: Sh of the odd chunks written (shready: the even ones)
    uint64_t *ofree = bars + 9;   // O^T of chunk c read by the output warps (O2: the even chunks)
    uint64_t *ofree2 = bars + 10; // O2: O^T of the odd chunks read
    uint64_t *barO2 = bars + 11;  // O2: O^T of the odd chunks done (barO: the even ones)
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + cBar + 96);
    unsigned char *sS = sm + cS;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int vh = HALF ? (int)(blockIdx.x & 1) : 0;  // which half of the value rows (ROWS = 64)
    const int cid = HALF ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int h = cid % p.Hv, b = order[cid / p.Hv];
    const int row = state_row(p, b, h == 0 && vh == 0 && tid == 0);
    if (row < 0) return;
    int t0, t1;
    request_range(p, b, t0, t1);
    const int nch = (t1 - t0 + TC_C - 1) / TC_C;
    int slot0 = 0;
    if (nch > 0) {
        slot0 = offs[b];
        if (slot0 + nch > cap) {
            // only overlapping requests can outgrow the workspace: skip this one
            if (p.err && tid == 0) atomicOr(p.err, 4);
            return;
        }
    }
    // the state tile; value row i_g, key column c at i_g * 128 + c (value-major) or
    // c * 128 + i_g (key-major, GDN_FLAG_STATE_KMAJOR)
    const bool km = (p.flags & kKMajor) != 0;
    const size_t tile = ((size_t)row * p.Hv + h) * 128 * 128;
    const size_t sbase = tile + (size_t)64 * vh * 128;  // this CTA's rows (value-major)
    if (nch == 0) {  // empty request: the final state is the initial one
        if (p.fin != p.init) {
            for (int idx = tid; idx < ROWS * 32; idx += CH_THREADS) {
                // key-major: key row c, four of this CTA's value columns
                const size_t off = km ? tile + (size_t)(idx / (ROWS / 4)) * 128 + 64 * vh + 4 * (idx % (ROWS / 4))
                                      : sbase + 4 * (size_t)idx;
                *reinterpret_cast<float4 *>(p.fin + off) =
                    p.init ? *reinterpret_cast<const float4 *>(p.init + off) : make_float4(0, 0, 0, 0);
            }
        }
        return;
    }

    if (tid == 0) {
        // rsread, shready and shready2 take one arrival from each of the eight state warps
        for (int i = 0; i < 12; ++i) ptx::mbar_init(&bars[i], (i == 4 || i == 5 || i == 8) ? 8 : 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tslot, 256);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;

    if (warp < 8) {
        // ===================== state: S_c -> Sh after every chunk (256 threads)
        const int q4 = warp & 3, hc = warp >> 2, i = (HALF ? 16 : 32) * q4 + lane;
        const bool live = !HALF || lane < 16;  // lanes that hold a row of this CTA's state
        const uint32_t lo = tmem + ((uint32_t)(32 * q4) << 16) + tS + 64 * hc;
        const size_t srow = sbase + (size_t)i * 128 + 64 * hc;
        // key-major: element (value row 64 vh + i, key column 64 hc + c) at kcol + c * 128
        const size_t kcol = tile + (size_t)(64 * hc) * 128 + 64 * vh + i;
        // e^{G_C} of chunk c, as the prepare kernel left it in the chunk's image
        auto gamma = [&](int c) {
            return *reinterpret_cast<const float *>(img + ((size_t)(slot0 + c) * p.Hv + h) * IM_BYTES + IM_EQ);
        };
        {
            const float g0 = STEP == kStepDecay ? gamma(0) : 1.f;
            float v[32];
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (p.init && live) {
                        if (km) {
                            const float *b = p.init + kcol + (size_t)(32 * pc + 4 * j) * 128;
                            f = make_float4(b[0], b[128], b[256], b[384]);
                        } else {
                            f = *reinterpret_cast<const float4 *>(p.init + srow + 32 * pc + 4 * j);
                        }
                    }
                    v[4 * j] = f.x, v[4 * j + 1] = f.y, v[4 * j + 2] = f.z, v[4 * j + 3] = f.w;
                }
                if (live) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) st_chunk(sS + hc * SHB, i, 4 * pc + cc, v + 8 * cc);
                }
                if (STEP == kStepDecay) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= g0;
                }
                tc::st32(lo + 32 * pc, v);
            }
            tc::wait_st();
        }
        // each warp hands over its rows itself (the barriers count the eight warps)
        tc::fence_async_smem();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) {
            ptx::mbar_arrive(rsread);
            ptx::mbar_arrive(shready);
        }
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const float gn = (STEP == kStepDecay && c + 1 < nch) ? gamma(c + 1) : 1.f;
            ok = ptx::named_bar_and(1, 256, ptx::mbar_wait_sleep(barS, c & 1));
            if (!ok) break;
            tc::fence_after();
            if (HALF) {
                // M = 64: the 16 rows of this warp's lane quarter over all 32 lanes (16x256b
                // shape): rows ra and ra + 8, columns 8 k + cq and + 1 of this warp's half
                const int ra = 16 * q4 + (lane >> 2), rb = ra + 8, cq = 2 * (lane & 3);
                float hv[32];
                tc::ld16x256<8>(lo, hv);
                if (STEP == kStepDecay && c + 1 < nch) {
                    // S <- e^{G_C} S of the next chunk before its U^T Kt lands
                    float w[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) w[e] = hv[e] * gn;
                    tc::st16x256_8(lo, w);
                    tc::wait_st();
                }
                tc::fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(rsread);
                if (c + 1 < nch) {
                    unsigned char *shb = sS + (PIPE ? ((c + 1) & 1) * 2 * SHB : 0) + hc * SHB;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        *reinterpret_cast<uint32_t *>(shb + sw(ra, k) + 2 * cq) = ptx::pack_h2(hv[4 * k], hv[4 * k + 1]);
                        *reinterpret_cast<uint32_t *>(shb + sw(rb, k) + 2 * cq) =
                            ptx::pack_h2(hv[4 * k + 2], hv[4 * k + 3]);
                    }
                    tc::fence_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(PIPE && ((c + 1) & 1) ? shready2 : shready);
                } else if (km) {
                    const size_t kc = tile + (size_t)(64 * hc) * 128 + 64 * vh;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const size_t c0 = kc + (size_t)(8 * k + cq) * 128;
                        p.fin[c0 + ra] = hv[4 * k];
                        p.fin[c0 + 128 + ra] = hv[4 * k + 1];
                        p.fin[c0 + rb] = hv[4 * k + 2];
                        p.fin[c0 + 128 + rb] = hv[4 * k + 3];
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const size_t c0 = sbase + 64 * hc + 8 * k + cq;
                        *reinterpret_cast<float2 *>(p.fin + c0 + (size_t)ra * 128) = make_float2(hv[4 * k], hv[4 * k + 1]);
                        *reinterpret_cast<float2 *>(p.fin + c0 + (size_t)rb * 128) =
                            make_float2(hv[4 * k + 2], hv[4 * k + 3]);
                    }
                }
                continue;
            }
            float sv[64];  // both column blocks in one load (one wait)
            tc::ld64(lo, sv);
            const float *v0 = sv, *v1 = sv + 32;
            if (STEP == kStepDecay && c + 1 < nch) {
                // S <- e^{G_C} S of the next chunk before its U^T Kt lands
                float w[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = v0[j] * gn;
                tc::st32(lo, w);
#pragma unroll
                for (int j = 0; j < 32; ++j) w[j] = v1[j] * gn;
                tc::st32(lo + 32, w);
                tc::wait_st();
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(rsread);
            if (c + 1 < nch) {
                // PIPE: chunk c + 1 writes buffer (c + 1) % 2 (the readout of chunk c may still
                // read the other) and publishes it on the barrier of its parity
                unsigned char *shb = sS + (PIPE ? ((c + 1) & 1) * 2 * SHB : 0) + hc * SHB;
                if (live) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) st_chunk(shb, i, cc, v0 + 8 * cc);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) st_chunk(shb, i, 4 + cc, v1 + 8 * cc);
                }
                tc::fence_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(PIPE && ((c + 1) & 1) ? shready2 : shready);
            } else if (live && km) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    p.fin[kcol + (size_t)j * 128] = v0[j];
                    p.fin[kcol + (size_t)(32 + j) * 128] = v1[j];
                }
            } else if (live) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    *reinterpret_cast<float4 *>(p.fin + srow + 4 * j) =
                        make_float4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
                    *reinterpret_cast<float4 *>(p.fin + srow + 32 + 4 * j) =
                        make_float4(v1[4 * j], v1[4 * j + 1], v1[4 * j + 2], v1[4 * j + 3]);
                }
            }
        }
        if (!ok && p.err && tid == 0) atomicOr(p.err, 2);
    } else if (warp < 12) {
        // ===================== outputs (128 threads): O^T[i][t] -> O[t][h][i]
        const int q4 = warp & 3, i = (HALF ? 16 : 32) * q4 + lane, ot = tid - 256;
        const bool live = !HALF || lane < 16;
        const size_t rstride = (size_t)p.Hv * 128;
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const bool odd = O2 && (c & 1);
            const uint32_t lo = tmem + ((uint32_t)(32 * q4) << 16) + tO + (odd ? 64u : 0u);
            ok = ptx::named_bar_and(2, 128, ptx::mbar_wait_sleep(odd ? barO2 : barO, O2 ? (c >> 1) & 1 : c & 1));
            if (!ok) break;
            tc::fence_after();
            if (HALF) {
                // M = 64: the 16 rows of this quarter over all 32 lanes (16x256b shape): value
                // rows ra and ra + 8, tokens 8 k + cq and + 1
                const int ra = 16 * q4 + (lane >> 2), rb = ra + 8, cq = 2 * (lane & 3);
                float hv[32];
                tc::ld16x256<8>(lo, hv);
                tc::fence_before();
                ptx::named_bar_sync(2, 128);
                if (ot == 0) ptx::mbar_arrive(odd ? ofree2 : ofree);
                const int n = min(TC_C, t1 - (t0 + TC_C * c));
                const size_t ob = ((size_t)(t0 + TC_C * c) * p.Hv + h) * 128 + 64 * vh;
#pragma unroll
                for (int k = 0; k < 8; ++k)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int t = 8 * k + cq + e;
                        if (t < n) {
                            const size_t o_t = ob + (size_t)t * rstride;
                            if (p.o_f32) {
                                static_cast<float *>(p.o)[o_t + ra] = hv[4 * k + e];
                                static_cast<float *>(p.o)[o_t + rb] = hv[4 * k + 2 + e];
                            } else {
                                static_cast<__half *>(p.o)[o_t + ra] = __float2half_rn(hv[4 * k + e]);
                                static_cast<__half *>(p.o)[o_t + rb] = __float2half_rn(hv[4 * k + 2 + e]);
                            }
                        }
                    }
                continue;
            }
            float ov[64];  // both column blocks in one load (one wait)
            tc::ld64(lo, ov);
            const float *o0 = ov, *o1 = ov + 32;
            tc::fence_before();
            ptx::named_bar_sync(2, 128);
            if (ot == 0) ptx::mbar_arrive(odd ? ofree2 : ofree);
            const int n = live ? min(TC_C, t1 - (t0 + TC_C * c)) : 0;
            const size_t obase = ((size_t)(t0 + TC_C * c) * p.Hv + h) * 128 + 64 * vh + i;
            if (p.o_f32) {  // fp32 activations (the products ran on fp16 copies)
                float *orow = static_cast<float *>(p.o) + obase;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    if (jj < n) orow[jj * rstride] = o0[jj];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    if (32 + jj < n) orow[(32 + jj) * rstride] = o1[jj];
            } else {
                __half *orow = static_cast<__half *>(p.o) + obase;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    if (jj < n) orow[jj * rstride] = __float2half_rn(o0[jj]);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    if (32 + jj < n) orow[(32 + jj) * rstride] = __float2half_rn(o1[jj]);
            }
        }
        if (!ok && p.err && ot == 0) atomicOr(p.err, 2);
    } else if (warp == 12) {
        // ===================== image loads, two buffers
        if (lane == 0) {
            const uint32_t skip = STEP == kStepE ? 0u : (uint32_t)(IM_U - 16384);  // only the delta rules load E^T
            const uint32_t ubytes = HALF ? 8192u : 16384u;               // U: this CTA's value rows
            // U = V, from the value input: the rules without retrieval (the per-key gated rule's
            // image carries E^T but no U)
            const bool u_from_v = STEP != kStepE || p.rule == kGated;
            for (int c = 0; c < nch; ++c) {
                const int bf = c & 1;
                if (c >= 2 && !ptx::mbar_wait_sleep(&freeb[bf], ((c - 2) >> 1) & 1)) {
                    if (p.err) atomicOr(p.err, 2);
                    break;
                }
                const unsigned char *src = img + ((size_t)(slot0 + c) * p.Hv + h) * IM_BYTES;
                unsigned char *dstb = sm + cImg + bf * IM_BYTES;
                ptx::mbar_arrive_expect_tx(&land[bf], IM_BYTES - skip - (16384u - ubytes));
                // the image two chunks ahead into L2, so that its load from there is short
                if (c + 2 < nch) {
                    const unsigned char *nxt = src + 2 * (size_t)p.Hv * IM_BYTES;
                    if (STEP == kStepE && !u_from_v) {
                        ptx::prefetch_l2(nxt, IM_BYTES);
                    } else if (STEP == kStepE) {
                        ptx::prefetch_l2(nxt, IM_U);
                        ptx::prefetch_l2(nxt + IM_P, IM_BYTES - IM_P);
#pragma unroll
                        for (int kb = 0; kb < 2; ++kb)
                            if (!HALF || kb == vh) ptx::prefetch_tile_3d(&tmV, 64 * kb, h, t0 + TC_C * (c + 2));
                    } else {
                        ptx::prefetch_l2(nxt + im_q(0), 8192);
                        ptx::prefetch_l2(nxt + im_q(1), 8192);
                        ptx::prefetch_l2(nxt + IM_P, IM_BYTES - IM_P);
#pragma unroll
                        for (int kb = 0; kb < 2; ++kb)
                            if (!HALF || kb == vh) ptx::prefetch_tile_3d(&tmV, 64 * kb, h, t0 + TC_C * (c + 2));
                    }
                }
                if (STEP == kStepE) {
                    ptx::bulk_g2s(dstb, src, IM_U, &land[bf]);  // E^T and Q'
                    if (!u_from_v) ptx::bulk_g2s(dstb + IM_U, src + IM_U + 8192 * vh, ubytes, &land[bf]);  // U (its rows)
                } else {
                    ptx::bulk_g2s(dstb + im_q(0), src + im_q(0), 8192, &land[bf]);  // Q'
                    ptx::bulk_g2s(dstb + im_q(1), src + im_q(1), 8192, &land[bf]);
                }
                if (u_from_v) {
                    // without retrieval U = V: its rows straight from the value input (the box
                    // lands in the image's U layout; rows past the request meet zero Kt rows and
                    // causally masked P entries only)
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb)
                        if (!HALF || kb == vh)
                            ptx::tma_load_3d(dstb + IM_U + (HALF ? 0 : 8192 * kb), &tmV, 64 * kb, h, t0 + TC_C * c,
                                             &land[bf]);
                }
                ptx::bulk_g2s(dstb + IM_P, src + IM_P, IM_BYTES - IM_P, &land[bf]);  // P, Kt
            }
        }
    } else {
        // ===================== products
        if (lane == 0) {
            const uint32_t aS = ptx::smem_u32(sS);
            // descriptors built once; each product advances them (desc_adv)
            const uint64_t dSh0 = tc::desc_sw128(aS);
            constexpr uint32_t idUK = tc::idesc_f16(ROWS, 128, true, true), idUP = tc::idesc_f16(ROWS, 64, true, false);
            constexpr uint32_t idSQ = tc::idesc_f16(ROWS, 64), idSEQ = tc::idesc_f16(ROWS, 192);
            bool ok = true;
            for (int c = 0; c < nch; ++c) {
                const int bf = c & 1;
                const uint32_t base = ptx::smem_u32(sm + cImg + bf * IM_BYTES);
                const uint64_t dU = tc::desc_sw128(base + IM_U, 8192), dKt = tc::desc_sw128(base + IM_KT, 8192);
                const uint64_t dP = tc::desc_sw128(base + IM_P), dEQ = tc::desc_sw128(base + IM_EQ);
                // (the issuing thread polls its waits on the chain's serial path: one lane, and
                // a poll wakes sooner than a suspended wait)
                ok = ptx::mbar_wait_spin(&land[bf], (c >> 1) & 1) && ptx::mbar_wait_spin(rsread, c & 1);
                if (!ok) break;
                tc::fence_after();
                if ((STEP != kStepE || p.rule == kGated) && c == nch - 1) {
                    // U came straight from the value input: in a short last chunk its rows past the
                    // request hold other tokens (or whatever the caller keeps there) and are cleared
                    const int n = t1 - (t0 + TC_C * c);
                    if (n < TC_C) {
                        unsigned char *ub = sm + cImg + bf * IM_BYTES + IM_U;
                        for (int r = n; r < TC_C; ++r)
#pragma unroll
                            for (int kb = 0; kb < (HALF ? 1 : 2); ++kb)
#pragma unroll
                                for (int q16 = 0; q16 < 8; ++q16)
                                    *reinterpret_cast<uint4 *>(ub + kb * 8192 + r * 128 + q16 * 16) = make_uint4(0, 0, 0, 0);
                        tc::fence_async_smem();
                    }
                }
                // UK: S += U^T Kt (M = 128 v, N = 128 j, K = 64 t; A and B M/N-major)
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tc::mma_f16(tmem + tS, tc::desc_adv(dU, s * 2048), tc::desc_adv(dKt, s * 2048), idUK, true);
                if (PIPE) tc::commit(barS);  // S_{c+1} is complete

                // the output warps have read the O^T buffer of this chunk: of chunk c - 1 (one
                // buffer) or c - 2 (O2)
                const bool odd = O2 && (c & 1);
                const uint32_t tOc = tO + (odd ? 64u : 0u);
                if (c >= (O2 ? 2 : 1)) {
                    ok = O2 ? ptx::mbar_wait_sleep(odd ? ofree2 : ofree, ((c - 2) >> 1) & 1)
                            : ptx::mbar_wait_sleep(ofree, (c - 1) & 1);
                    if (!ok) break;
                    tc::fence_after();
                }
                // UP: O^T = U^T P^T (N = 64 r, K = 64 t; B K-major)
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tc::mma_f16(tmem + tOc, tc::desc_adv(dU, s * 2048), tc::desc_adv(dP, s * 32), idUP, s > 0);
                if (PIPE) {
                    ok = ptx::mbar_wait_spin((c & 1) ? shready2 : shready, (c >> 1) & 1);
                    if (!ok) break;
                    tc::fence_after();
                    const uint64_t dSh = tc::desc_adv(dSh0, (c & 1) * 2 * SHB);
                    // SQ: O^T += Sh Q'^T (N = 64 t, K = 128 i; both K-major)
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        tc::mma_f16(tmem + tOc, tc::desc_adv(dSh, (s >> 2) * SHB + (s & 3) * 32),
                                    tc::desc_adv(dEQ, (s >> 2) * IM_EQ_BLK + IM_EQ_Q + (s & 3) * 32), idSQ, true);
                    tc::commit(odd ? barO2 : barO);
                    tc::commit(&freeb[bf]);
                    continue;
                }
                ok = ptx::mbar_wait_spin(shready, c & 1);
                if (!ok) break;
                tc::fence_after();
                if (STEP == kStepE) {
                    // SE and SQ as one product: [S | O^T] += Sh [E^T; Q']^T (N = 128 j + 64 t = 192,
                    // K = 128 i; A and B K-major; S and O^T are adjacent in tensor memory)
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        tc::mma_f16(tmem + tS, tc::desc_adv(dSh0, (s >> 2) * SHB + (s & 3) * 32),
                                    tc::desc_adv(dEQ, (s >> 2) * IM_EQ_BLK + (s & 3) * 32), idSEQ, true);
                } else {
                    // SQ: O^T += Sh Q'^T (N = 64 t, K = 128 i; both K-major)
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        tc::mma_f16(tmem + tOc, tc::desc_adv(dSh0, (s >> 2) * SHB + (s & 3) * 32),
                                    tc::desc_adv(dEQ, (s >> 2) * IM_EQ_BLK + IM_EQ_Q + (s & 3) * 32), idSQ, true);
                }
                tc::commit(odd ? barO2 : barO);
                // every product of chunk c is done: S_{c+1} is complete and Sh is free
                tc::commit(barS);
                tc::commit(&freeb[bf]);
            }
            if (!ok && p.err) atomicOr(p.err, 2);
        }
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

bool al16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// fp32 -> fp16 copy of n elements (n a multiple of 4, both pointers 16-byte aligned): the
// tensor-core prefill takes fp32 activations through fp16 copies in its workspace (its
// products round their operands to fp16 anyway).
__global__ void __launch_bounds__(256) f16_to_f32_kernel(const __half *src, float *dst, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = __half2float(src[i]);
}

__global__ void __launch_bounds__(256) f32_to_f16_kernel(const float4 *src, uint2 *dst, size_t n4) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 f = src[i];
        dst[i] = make_uint2(ptx::pack_h2(f.x, f.y), ptx::pack_h2(f.z, f.w));
    }
}

// bytes of each fp16 copy (256-byte aligned) for fp32 activations: q, k [T, Hq, 128], v [T, Hv, 128]
size_t copy_bytes(const Problem &p, int heads) { return (((size_t)p.T * heads * 128 * 2) + 255) & ~(size_t)255; }
// fp16 per-key gate rows that the per-key prepare pass lands by bulk copies get fp32 copies:
// the log decay (or raw gate) and GDN-2's per-key beta (its erase gate)
bool decay_copy(const Problem &p) { return (p.flags & kPerKey) && rule_has_decay(p.rule) && p.decay_f16; }
bool erase_copy(const Problem &p) { return p.rule == kGdn2 && p.erase_gate == nullptr && p.beta_f16; }
size_t gate_copy_bytes(const Problem &p) { return (((size_t)p.T * p.Hv * 128 * 4) + 255) & ~(size_t)255; }
size_t copies_bytes(const Problem &p) {
    return (p.act_f16 ? 0 : 2 * copy_bytes(p, p.Hq) + copy_bytes(p, p.Hv)) +
           (decay_copy(p) ? gate_copy_bytes(p) : 0) + (erase_copy(p) ? gate_copy_bytes(p) : 0);
}

// slots for every chunk of pairwise disjoint requests: sum ceil(len / C) <= T / C + B
int slot_capacity(const Problem &p) { return (int)((long long)p.T / TC_C + p.B + 1); }
// workspace head: chunk offsets (B + 1 ints), the slot -> request table (one int
// per slot) and the request order (B ints), rounded up to 1 KB
// offsets [B + 1], slot -> request [cap], order [B], rounded to 1 KB
size_t head_bytes(const Problem &p, int cap) {
    return (((size_t)2 * p.B + 1 + (size_t)cap) * sizeof(int) + 1023) & ~(size_t)1023;
}
size_t head_bytes(const Problem &p) { return head_bytes(p, slot_capacity(p)); }
// the windowed call: the per-request window ranges [B][2] (rounded to 256 bytes), then a head
// and images for W chunks of every request: at most window_fixed + W * window_per_chunk bytes
size_t window_bytes(const Problem &p) { return ((size_t)2 * p.B * sizeof(int) + 255) & ~(size_t)255; }
size_t window_fixed(const Problem &p) { return window_bytes(p) + ((size_t)2 * p.B + 1) * sizeof(int) + 1023; }
size_t window_per_chunk(const Problem &p) { return (size_t)p.B * ((size_t)p.Hv * IM_BYTES + sizeof(int)); }



}  // namespace

bool chunked_tc_eligible(const Problem &p) {
    // scalar decay, v1 rules: the scalar prepare kernel; per-key decay of gated_delta and
    // GDN-2: the per-key prepare kernel.  Both feed the same chain kernel.
    const bool rule_ok = p.rule == kLinear || p.rule == kGated || p.rule == kDelta || p.rule == kGatedDelta;
    const bool scalar_ok = rule_ok && !((p.flags & kPerKey) && rule_has_decay(p.rule));
    // fp32 activations run on fp16 copies made in the workspace, fp16 per-key gate rows on
    // fp32 copies
    Problem pg = p;
    if (decay_copy(p)) pg.decay_f16 = 0, pg.decay = p.q;  // (a 16-byte aligned stand-in for the copy)
    if (erase_copy(p)) pg.beta_f16 = 0, pg.beta = p.q;
    return (scalar_ok || chunk_prepare_perkey_eligible(pg)) && p.dk == 128 && p.dv == 128 &&
           al16(p.q) && al16(p.k) && al16(p.v) && al16(p.fin) && (p.init == nullptr || al16(p.init));
}

// workspace: [offsets | slot table | order] [one operand image per (slot, head)]
size_t chunked_tc_workspace_bytes(const Problem &p) {
    if (p.B == 0) return 0;
    return head_bytes(p) + (size_t)slot_capacity(p) * p.Hv * IM_BYTES + copies_bytes(p);
}

// one chunk per request at a time (the windowed call with W = 1)
size_t chunked_tc_workspace_min_bytes(const Problem &p) {
    if (p.B == 0) return 0;
    const size_t full = chunked_tc_workspace_bytes(p);
    const size_t one = ((window_fixed(p) + window_per_chunk(p) + 255) & ~(size_t)255) + copies_bytes(p);
    return one < full ? one : full;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

bool make_kqv_map(CUtensorMap *m, const void *base, int heads, int tokens) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static cudaError_t launch_tc_f16(const Problem &p, void *ws, size_t ws_bytes, int cap, cudaStream_t stream,
                                 int win_w = 0, int win_W = 0);

cudaError_t launch_chunked_tc(const Problem &p, void *ws, size_t ws_bytes, cudaStream_t stream) {
    const void *fns[8] = {(const void *)chunk_prepare_kernel<true>,
                          (const void *)chunk_prepare_kernel<false>,
                          (const void *)chunk_chain_kernel<kStepPlain, 128>,
                          (const void *)chunk_chain_kernel<kStepDecay, 128>,
                          (const void *)chunk_chain_kernel<kStepE, 128>,
                          (const void *)chunk_chain_kernel<kStepPlain, 64>,
                          (const void *)chunk_chain_kernel<kStepDecay, 64>,
                          (const void *)chunk_chain_kernel<kStepE, 64>};
    cudaError_t e;
    for (int f = 0; f < 8; ++f) {
        e = smem_attr(fns[f], f < 2 ? PR_SMEM : CH_SMEM);
        if (e != cudaSuccess) return e;
    }
    const size_t cb = copies_bytes(p);
    if (p.B == 0) return cudaSuccess;
    // fp32 activations: fp16 copies of q, k and v at the end of the workspace, the chain writing o
    // in fp32; fp16 per-key gate rows: fp32 copies after them.  Then the same kernels on them.
    if (ws == nullptr || ws_bytes < chunked_tc_workspace_min_bytes(p)) return cudaErrorInvalidValue;
    const size_t avail = (ws_bytes - cb) & ~(size_t)255;  // the copies sit above it, 256-byte aligned
    unsigned char *cp = static_cast<unsigned char *>(ws) + avail;
    Problem pc = p;
    if (!p.act_f16) {
        const void *src[3] = {p.q, p.k, p.v};
        const int heads[3] = {p.Hq, p.Hq, p.Hv};
        const void **dstp[3] = {&pc.q, &pc.k, &pc.v};
        for (int t = 0; t < 3; ++t) {
            const size_t n4 = (size_t)p.T * heads[t] * 128 / 4;
            const long long blocks = std::min<long long>((long long)(n4 + 255) / 256, 8LL * sm_count());
            if (blocks > 0)
                f32_to_f16_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const float4 *>(src[t]),
                                                                       reinterpret_cast<uint2 *>(cp), n4);
            *dstp[t] = cp;
            cp += copy_bytes(p, heads[t]);
        }
        pc.act_f16 = 1;
        pc.o_f32 = 1;
    }
    const bool cdec = decay_copy(p), cera = erase_copy(p);
    for (int t = 0; t < 2; ++t) {
        if (!(t == 0 ? cdec : cera)) continue;
        const size_t n = (size_t)p.T * p.Hv * 128;
        const long long blocks = std::min<long long>((long long)(n + 255) / 256, 8LL * sm_count());
        if (blocks > 0)
            f16_to_f32_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
                static_cast<const __half *>(t == 0 ? p.decay : p.beta), reinterpret_cast<float *>(cp), n);
        if (t == 0)
            pc.decay = cp, pc.decay_f16 = 0;
        else
            pc.beta = cp, pc.beta_f16 = 0;
        cp += gate_copy_bytes(p);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int full_cap = slot_capacity(p);
    if (avail >= head_bytes(p, full_cap) + (size_t)full_cap * p.Hv * IM_BYTES)
        return launch_tc_f16(pc, ws, avail, full_cap, stream);
    // Windowed: W chunks of every request at a time, as many as the workspace holds.  Window w
    // reads the state window w - 1 left in final_state (fp32, so the carry is exact) and writes
    // its outputs in place; a request past its end is empty in a window and keeps its state.
    const size_t wb = window_bytes(p), fixed = window_fixed(p);
    const long long W = avail > fixed ? (long long)((avail - fixed) / window_per_chunk(p)) : 0;
    if (W < 1) return cudaErrorInvalidValue;
    // the longest a request can be: the uniform length, else every token
    const long long L = p.cu ? p.T : (p.seq_len ? p.seq_len : (long long)p.T / p.B);
    const long long nwin = ((L + TC_C - 1) / TC_C + W - 1) / W;
    int32_t *win = static_cast<int32_t *>(ws);
    unsigned char *rest = static_cast<unsigned char *>(ws) + wb;
    for (long long w = 0; w < nwin; ++w) {
        // (the offsets kernel of each window first writes the window's request ranges)
        Problem pw = pc;
        pw.win = win;
        if (w > 0) pw.init = pc.fin;
        e = launch_tc_f16(pw, rest, avail - wb, (int)(p.B * W), stream, (int)w, (int)W);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// the tensor-core prefill proper, on fp16 activations (its workspace: offsets, tables, images)
static cudaError_t launch_tc_f16(const Problem &p, void *ws, size_t ws_bytes, int cap, cudaStream_t stream,
                                 int win_w, int win_W) {
    cudaError_t e;
    CUtensorMap tk, tq, tv;
    if (!make_kqv_map(&tk, p.k, p.Hq, p.T) || !make_kqv_map(&tq, p.q, p.Hq, p.T) ||
        !make_kqv_map(&tv, p.v, p.Hv, p.T))
        return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)((long long)p.B * p.Hv);
    if (grid == 0) return cudaSuccess;
    if (ws == nullptr || ws_bytes < head_bytes(p, cap) + (size_t)cap * p.Hv * IM_BYTES) return cudaErrorInvalidValue;
    const bool retr = rule_has_retrieval(p.rule);
    int *offs = static_cast<int *>(ws);
    int *slot_req = offs + p.B + 1;
    int *order = slot_req + cap;
    unsigned char *img = static_cast<unsigned char *>(ws) + head_bytes(p, cap);
    chunk_offsets_kernel<<<1, 1024, 0, stream>>>(p, offs, slot_req, order, cap, win_w, win_W);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // persistent prepare CTAs: two per SM (shared and tensor memory), at most one per task
    const long long tasks = (long long)cap * p.Hv;
    const long long pgrid = std::min<long long>(tasks, 2LL * sm_count());
    const bool perkey_prep = chunk_prepare_perkey_eligible(p);
    if (perkey_prep) {
        e = launch_chunk_prepare_perkey(p, tk, tq, tv, offs, slot_req, img, cap, stream);
    } else {
        if (retr)
            chunk_prepare_kernel<true><<<(unsigned)pgrid, PR_THREADS, PR_SMEM, stream>>>(p, tk, tq, tv, offs, slot_req,
                                                                                       img, cap);
        else
            chunk_prepare_kernel<false><<<(unsigned)pgrid, PR_THREADS, PR_SMEM, stream>>>(p, tk, tq, tv, offs, slot_req,
                                                                                        img, cap);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    // fewer chains than SMs: two CTAs per chain, one per half of the value rows
    if ((long long)grid < sm_count()) {
        if (p.rule == kLinear)
            chunk_chain_kernel<kStepPlain, 64><<<2 * grid, CH_THREADS, CH_SMEM, stream>>>(p, tv, offs, order, img, cap);
        else if (p.rule == kGated && !perkey_prep)  // (per-key decay: E carries it)
            chunk_chain_kernel<kStepDecay, 64><<<2 * grid, CH_THREADS, CH_SMEM, stream>>>(p, tv, offs, order, img, cap);
        else
            chunk_chain_kernel<kStepE, 64><<<2 * grid, CH_THREADS, CH_SMEM, stream>>>(p, tv, offs, order, img, cap);
    } else {
        if (p.rule == kLinear)
            chunk_chain_kernel<kStepPlain, 128><<<grid, CH_THREADS, CH_SMEM, stream>>>(p, tv, offs, order, img, cap);
        else if (p.rule == kGated && !perkey_prep)
            chunk_chain_kernel<kStepDecay, 128><<<grid, CH_THREADS, CH_SMEM, stream>>>(p, tv, offs, order, img, cap);
        else
            chunk_chain_kernel<kStepE, 128><<<grid, CH_THREADS, CH_SMEM, stream>>>(p, tv, offs, order, img, cap);
    }
    return cudaGetLastError();
}

}  // namespace gdn
