// chunked_tc.cu -- chunk-parallel prefill on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), for dk = dv = 128, fp16
// activations, scalar decay, rules linear / gated / delta / gated_delta.
//
// Same per-chunk algebra as chunked.cu (derived from the token recurrence;
// see the comment there).  For one chunk of C = 64 tokens, with
// A = strict-lower(diag(beta) e^{G_r - G_j} K K^T), T = (I + A)^-1,
// Ta = T diag(beta e^G), Tb = T diag(beta), W = Ta K, U = Tb V:
//
//   D = U - W S^T                 (the token corrections, D^T = U^T - S W^T)
//   O = scale (diag(e^G) Q S^T + P D),   P = decayed causal Q K^T
//   S <- e^{G_C} S + D^T diag(e^{G_C - G}) K
//
// Two kernels run the delta rules.  The key-side system does not depend on
// the state, so chunk_solve_kernel builds A with one tensor-core product and
// solves it in fp32 for every (chunk, head), all chunks in parallel, and
// writes Tb (fp16) to the workspace.  chunked_pipe_kernel then walks each
// (request, value head) chunk by chunk, with the state in tensor memory; it
// loads Tb by TMA together with the chunk's keys, queries and values.  The
// rules without retrieval (D = V) need no solve.  The layout of each kernel
// is described above it.
#include <algorithm>
#include <cuda.h>  // CUtensorMap (the encoder is fetched through the runtime)
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int TC_C = 64;  // tokens per chunk
constexpr int TC_TMEM_COLS = 512;
constexpr int kTbBytes = TC_C * TC_C * 2;  // one fp16 Tb tile
constexpr int kFacFloats = 2 * TC_C;       // per (chunk, head): G and 1 / |k| of the 64 tokens

constexpr uint32_t kLandBytes = 3 * 16384;  // K, Q and V boxes of one chunk

// shared memory layout of chunk_solve_kernel (persistent: a producer warp and
// four solver warps, two task buffers)
constexpr int SV_SOLVERS = 128;
constexpr int SV_THREADS = SV_SOLVERS + 32;
constexpr int FA = 68;  // fp32 row stride of At (16-byte rows; lanes = consecutive r, conflict-free)
constexpr int FT = 68;  // fp32 row stride of T (16-byte rows for vector reads)
constexpr int sK = 0;                      // 2 x 16 KB: K, 2 blocks of [64 tokens][64 dk], K-major
constexpr int sAt = 32768;                 // fp32 [64][FA], At[j][r] = A[r][j]
constexpr int sTf = sAt + 64 * FA * 4;     // fp32 [64][FT], T
constexpr int sY = sTf + 64 * FT * 4;      // fp32 [32][36] product scratch
constexpr int sGin = sY + 32 * 36 * 4;     // 2 x (log decay, beta) of 64 tokens, from the producer
constexpr int sSc = sGin + 2 * 128 * 4;    // fp32 G, beta, 1/|k| of the current task: 3 x 64
constexpr int sHdr = sSc + 3 * 64 * 4;     // 2 x {request, head, first token, tokens}
constexpr int sBar = sHdr + 2 * 16;        // full[2], empty[2], MMA barrier, TMEM address
constexpr int SV_SMEM = sBar + 64 + 1024;  // + alignment slack

// writes 8 consecutive fp16 values (one 16-byte chunk) of row `row`, chunk
// `ch` (0..7) of a 64-column block
__device__ __forceinline__ void st_chunk(unsigned char *tile, int row, int ch, const float *x) {
    uint4 u;
    u.x = ptx::pack_h2(x[0], x[1]);
    u.y = ptx::pack_h2(x[2], x[3]);
    u.z = ptx::pack_h2(x[4], x[5]);
    u.w = ptx::pack_h2(x[6], x[7]);
    *reinterpret_cast<uint4 *>(tile + row * 128 + ((ch ^ (row & 7)) << 4)) = u;
}

// number of chunks of request b
__device__ __forceinline__ int request_chunks(const Problem &p, int b) {
    int t0, t1;
    request_range(p, b, t0, t1);
    return (t1 - t0 + TC_C - 1) / TC_C;
}

// ---------------------------------------------------------------------------
// Workspace slots: chunk j of request b has slot offs[b] + j, offs being the
// exclusive prefix sum of the requests' chunk counts (offs[B] = the total);
// slot_req[slot] is the request owning a slot.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) chunk_offsets_kernel(Problem p, int *offs, int *slot_req, int cap) {
    __shared__ int wsum[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (p.B + 1023) / 1024;
    const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
    int s = 0;
    for (int b = b0; b < b1; ++b) s += request_chunks(p, b);
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
}

// ---------------------------------------------------------------------------
// Tb = (I + A)^-1 diag(beta) for every (chunk slot, value head) task.
// A = strict-lower(diag(beta) e^{G_r - G_j} Kn Kn^T), Kn the key rows after
// the optional L2 norm, from one M = 64 tensor-core product of the raw fp16
// keys (the norms are applied to the fp32 result).  The solve is fp32
// recursive doubling: the four 16 x 16 diagonal blocks by substitution, then
// [[T0, 0], [L, T1]] with L = -T1 A10 T0 twice.  Padding tokens of a short
// last chunk get beta = 0 and zero keys, so their rows and columns of Tb are
// zero.
//
// Persistent CTAs: a producer warp walks the CTA's tasks (slot, head) two
// ahead of the solvers (request lookup, the gates in fp32, the key tile by
// TMA) into two buffers; four solver warps run the product, the system and
// its solve.  Waits are bounded.
template <bool RETR>
__global__ void __launch_bounds__(SV_THREADS) chunk_solve_kernel(Problem p, const __grid_constant__ CUtensorMap tmK,
                                                                 const int *offs, const int *slot_req, __half *tb,
                                                                 float *fac, int cap) {
    extern __shared__ unsigned char smraw[];
    const uint32_t sb0 = ptx::smem_u32(smraw);
    unsigned char *sm = smraw + (((sb0 + 1023u) & ~1023u) - sb0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = min(offs[p.B], cap);
    const long long ntasks = (long long)total * p.Hv;
    float *At = reinterpret_cast<float *>(sm + sAt);
    float *Tf = reinterpret_cast<float *>(sm + sTf);
    float *Y = reinterpret_cast<float *>(sm + sY);
    float *gin = reinterpret_cast<float *>(sm + sGin);
    float *sG = reinterpret_cast<float *>(sm + sSc);
    float *sB = sG + 64, *sInv = sG + 128;
    int *hdr = reinterpret_cast<int *>(sm + sHdr);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + sBar);
    uint64_t *empty = full + 2;
    uint64_t *mbar = full + 4;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + sBar + 40);
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) ptx::mbar_init(&full[i], 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tslot, 64);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    const long long G = gridDim.x;

    if (warp == 4) {
        // ===================== producer
        int i = 0;
        for (long long t = blockIdx.x; t < ntasks; t += G, ++i) {
            const int bf = i & 1;
            if (!ptx::mbar_wait_sleep(&empty[bf], ((i >> 1) & 1) ^ 1)) {
                if (p.err && lane == 0) atomicOr(p.err, 2);
                break;
            }
            const int slot = (int)(t / p.Hv), h = (int)(t % p.Hv);
            const int b = slot_req[slot];
            int t0, t1;
            request_range(p, b, t0, t1);
            const int c0 = t0 + TC_C * (slot - offs[b]);
            const int n = min(TC_C, t1 - c0);
            float *g2 = gin + bf * 128;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tt = lane + 32 * e;
                float g = 0.f, bt = 0.f;
                if (tt < n) {
                    const size_t th = (size_t)(c0 + tt) * p.Hv + h;
                    if (rule_has_decay(p.rule)) {
                        g = ld_any(p.decay, th, p.decay_f16);
                        if (p.raw_gate) g = p.gate_scale[h] * softplus_f(g + p.gate_bias[h]);
                    }
                    if (RETR) {
                        bt = ld_any(p.beta, th, p.beta_f16);
                        if (p.flags & kBetaSigmoid) bt = sigmoid_f(bt);
                    }
                }
                g2[tt] = g;
                g2[64 + tt] = bt;
            }
            if (lane == 0) {
                int *hd = hdr + 4 * bf;
                hd[0] = b, hd[1] = h, hd[2] = c0, hd[3] = n;
            }
            __syncwarp();
            if (lane == 0) {
                const int qh = (int)((long long)h * p.Hq / p.Hv);
                unsigned char *kt = sm + sK + bf * 16384;
                ptx::mbar_arrive_expect_tx(&full[bf], 16384);
                ptx::tma_load_3d(kt, &tmK, 0, qh, c0, &full[bf]);
                ptx::tma_load_3d(kt + 8192, &tmK, 64, qh, c0, &full[bf]);
            }
        }
    } else {
        // ===================== solvers (128 threads)
        bool ok = true;
        uint32_t mphase = 0;
        int i = 0;
        for (long long t = blockIdx.x; t < ntasks; t += G, ++i) {
            const int bf = i & 1;
            ok = ptx::named_bar_and(1, SV_SOLVERS, ptx::mbar_wait_sleep(&full[bf], (i >> 1) & 1));
            if (!ok) break;
            const int *hd = hdr + 4 * bf;
            const int slot = (int)(t / p.Hv), h = hd[1], n = hd[3];
            unsigned char *sKt = sm + sK + bf * 16384;
            const float *g2 = gin + bf * 128;
            if (n < TC_C) {  // the boxes run past this request: clear the rows beyond it
                for (int idx = tid; idx < (TC_C - n) * 16; idx += SV_SOLVERS) {
                    const int r = n + (idx >> 4), ch = idx & 15;
                    *reinterpret_cast<uint4 *>(sKt + (ch >> 3) * 8192 + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            if (warp == 0) {  // G = inclusive cumulative sum of the log decays; beta
                const float x0 = g2[2 * lane], x1 = g2[2 * lane + 1];
                float sacc = x0 + x1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, sacc, o);
                    if (lane >= o) sacc += y;
                }
                sG[2 * lane] = sacc - x1;
                sG[2 * lane + 1] = sacc;
                sB[2 * lane] = g2[64 + 2 * lane];
                sB[2 * lane + 1] = g2[64 + 2 * lane + 1];
            }
            ptx::named_bar_sync(1, SV_SOLVERS);
            {  // 1 / |k_r|: thread pair (2r, 2r + 1), one 64-column block each
                const int r = tid >> 1, kb = tid & 1;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(sKt + kb * 8192 + r * 128 + ((c ^ (r & 7)) << 4));
                    const __half2 *hp = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float2 f = __half22float2(hp[w]);
                        s0 = fmaf(f.x, f.x, s0);
                        s1 = fmaf(f.y, f.y, s1);
                    }
                }
                float ss = s0 + s1;
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (kb == 0) sInv[r] = (p.flags & kL2k) ? rsqrtf(ss + 1e-12f) : 1.f;
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(1, SV_SOLVERS);
            {
                // the chunk's per-token factors for the chain kernel: G (cumulative log
                // decay) and 1 / |k|
                float *fd = fac + ((size_t)slot * p.Hv + h) * kFacFloats;
                fd[tid] = tid < 64 ? sG[tid] : sInv[tid - 64];
            }
            if (!RETR) {
                // no system to solve: the key tile and gate buffer are free again
                ptx::named_bar_sync(1, SV_SOLVERS);
                if (tid == 0) ptx::mbar_arrive(&empty[bf]);
                continue;
            }
            if (tid == 0) {
                tc::fence_after();
                // K K^T: M = 64 tokens, N = 64 tokens, K = 128 channels
                const uint32_t aK = ptx::smem_u32(sKt);
#pragma unroll
                for (int s2 = 0; s2 < 8; ++s2) {
                    const uint64_t d = tc::desc_sw128(aK + (s2 >> 2) * 8192 + (s2 & 3) * 32);
                    tc::mma_f16(tmem, d, d, tc::idesc_f16(64, 64), s2 > 0);
                }
                tc::commit(mbar);
            }
            ok = ptx::named_bar_and(1, SV_SOLVERS, ptx::mbar_wait_sleep(mbar, mphase));
            mphase ^= 1u;
            if (!ok) break;
            tc::fence_after();
            // the key tile and the gate buffer are free for the producer
            if (tid == 0) ptx::mbar_arrive(&empty[bf]);
            {
                // rows 16 warp .. 16 warp + 15 sit on tensor-memory lanes 32 warp .. + 15 (M = 64);
                // the 16x256b shape gives thread `lane` rows ra, ra + 8 and column pairs 2 (lane % 4)
                const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
                const int ra = 16 * warp + (lane >> 2), rb = ra + 8, cp = 2 * (lane & 3);
                const float fa = sB[ra] * sInv[ra], fb = sB[rb] * sInv[rb], Ga = sG[ra], Gb = sG[rb];
                float v[32];
                tc::ld16x256<8>(tmem + lane_off, v);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = 8 * k + cp;
                    const float2 gj = *reinterpret_cast<const float2 *>(sG + j);
                    const float2 ij = *reinterpret_cast<const float2 *>(sInv + j);
                    At[j * FA + ra] = j < ra ? fa * __expf(Ga - gj.x) * ij.x * v[4 * k] : 0.f;
                    At[(j + 1) * FA + ra] = j + 1 < ra ? fa * __expf(Ga - gj.y) * ij.y * v[4 * k + 1] : 0.f;
                    At[j * FA + rb] = j < rb ? fb * __expf(Gb - gj.x) * ij.x * v[4 * k + 2] : 0.f;
                    At[(j + 1) * FA + rb] = j + 1 < rb ? fb * __expf(Gb - gj.y) * ij.y * v[4 * k + 3] : 0.f;
                }
            }
            tc::fence_before();
            ptx::named_bar_sync(1, SV_SOLVERS);
            if (lane < 16) {
                // column `lane` of the inverse of diagonal block `warp`, right-looking:
                // once x[j] is final it updates every later row at once
                float x[16];
                const float *Ab = At + (16 * warp) * FA + 16 * warp;  // Ab[j][i] = A[i][j]
#pragma unroll
                for (int q = 0; q < 16; ++q) x[q] = (q == lane) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < 15; ++j) {
                    float a[16];
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) {
                        const float4 tv = *reinterpret_cast<const float4 *>(Ab + j * FA + 4 * w4);
                        a[4 * w4] = tv.x, a[4 * w4 + 1] = tv.y, a[4 * w4 + 2] = tv.z, a[4 * w4 + 3] = tv.w;
                    }
#pragma unroll
                    for (int q = j + 1; q < 16; ++q) x[q] = fmaf(-a[q], x[j], x[q]);
                }
#pragma unroll
                for (int q = 0; q < 16; ++q) Tf[(16 * warp + q) * FT + 16 * warp + lane] = x[q];
            }
            // the strictly upper blocks (0,1) and (2,3) that the 32x32 products read are zero
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int idx = 4 * tid + e, blk = idx >> 8, rr = (idx >> 4) & 15, cc = idx & 15;
                Tf[(32 * blk + rr) * FT + 32 * blk + 16 + cc] = 0.f;
            }
            ptx::named_bar_sync(1, SV_SOLVERS);
            {
                // level 1: blocks (1,0) and (3,2): Y = A_{b,b-1} T_{b-1}, then L = -T_b Y
                const int r = tid >> 3, c = 2 * (tid & 7);  // row 0..15, columns c, c+1
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    const int o0 = 32 * blk;
                    float y0 = 0.f, y1 = 0.f;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float a = At[(o0 + k) * FA + o0 + 16 + r];
                        y0 = fmaf(a, Tf[(o0 + k) * FT + o0 + c], y0);
                        y1 = fmaf(a, Tf[(o0 + k) * FT + o0 + c + 1], y1);
                    }
                    Y[blk * 16 * 36 + r * 36 + c] = y0;
                    Y[blk * 16 * 36 + r * 36 + c + 1] = y1;
                }
                ptx::named_bar_sync(1, SV_SOLVERS);
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    const int o0 = 32 * blk;
                    float l0 = 0.f, l1 = 0.f;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float tv = Tf[(o0 + 16 + r) * FT + o0 + 16 + k];
                        l0 = fmaf(tv, Y[blk * 16 * 36 + k * 36 + c], l0);
                        l1 = fmaf(tv, Y[blk * 16 * 36 + k * 36 + c + 1], l1);
                    }
                    Tf[(o0 + 16 + r) * FT + o0 + c] = -l0;
                    Tf[(o0 + 16 + r) * FT + o0 + c + 1] = -l1;
                }
            }
            ptx::named_bar_sync(1, SV_SOLVERS);
            {
                // level 2: Y = A_10 T_0 (32 x 32), then L = -T_1 Y; thread = (row, 2 x 4 columns).
                // T_0 and T_1 are lower triangular: Y[r][c] sums k >= c, L[r][c] sums k <= r.
                const int r = tid >> 2;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int c = 4 * (tid & 3) + 16 * half;
                    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                    for (int k = c; k < 32; ++k) {
                        const float a = At[k * FA + 32 + r];
                        const float4 tv = *reinterpret_cast<const float4 *>(Tf + k * FT + c);
                        y.x = fmaf(a, tv.x, y.x), y.y = fmaf(a, tv.y, y.y), y.z = fmaf(a, tv.z, y.z),
                        y.w = fmaf(a, tv.w, y.w);
                    }
                    *reinterpret_cast<float4 *>(Y + r * 36 + c) = y;
                }
                ptx::named_bar_sync(1, SV_SOLVERS);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int c = 4 * (tid & 3) + 16 * half;
                    float4 l = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                    for (int k = 0; k <= r; ++k) {
                        const float tv = Tf[(32 + r) * FT + 32 + k];
                        const float4 yy = *reinterpret_cast<const float4 *>(Y + k * 36 + c);
                        l.x = fmaf(tv, yy.x, l.x), l.y = fmaf(tv, yy.y, l.y), l.z = fmaf(tv, yy.z, l.z),
                        l.w = fmaf(tv, yy.w, l.w);
                    }
                    *reinterpret_cast<float4 *>(Tf + (32 + r) * FT + c) = make_float4(-l.x, -l.y, -l.z, -l.w);
                }
            }
            ptx::named_bar_sync(1, SV_SOLVERS);
            {
                // Tb[r][j] = T[r][j] beta_j (j <= r), fp16 rows of 128 bytes
                const int r = tid >> 1, j0 = 32 * (tid & 1);
                __half *dst = tb + (((size_t)slot * p.Hv + h) * TC_C + r) * TC_C + j0;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = j0 + 8 * w + e;
                        x[e] = j <= r ? Tf[r * FT + j] * sB[j] : 0.f;
                    }
                    uint4 u;
                    u.x = ptx::pack_h2(x[0], x[1]);
                    u.y = ptx::pack_h2(x[2], x[3]);
                    u.z = ptx::pack_h2(x[4], x[5]);
                    u.w = ptx::pack_h2(x[6], x[7]);
                    *reinterpret_cast<uint4 *>(dst + 8 * w) = u;
                }
            }
            // At, Tf, Y and the task scalars are rewritten by the next task
            ptx::named_bar_sync(1, SV_SOLVERS);
        }
        if (!ok && p.err && tid == 0) atomicOr(p.err, 2);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 64);
}

// ---------------------------------------------------------------------------
// Pipelined chain kernel: the same per-chunk algebra with the state-free work
// of chunk c + 1 overlapped with the state chain of chunk c, and the chain
// reduced to two tensor-core rounds per chunk:
//
//   C12: [D^T | O^T]  = S [-W; Qh]^T                  (N = 128, K-major B)
//   C34: [O^T | S  ] += D^T [P^T | Kt]                 (N = 192, MN-major B)
//
// where D^T starts from U^T = V^T Tb^T (computed ahead into its own tensor
// memory, added in the epilogue), Kt = diag(e^{G_C - G}) K, P^T comes from
// the product K Q^T, and the fp32 state S lives in tensor memory: the
// epilogue of C12 scales it by e^{G_C} in place and C34 accumulates
// X = D^T Kt into it.  The rules without retrieval use Tb = I and W = 0
// (D = V).
//
// Roles (16 warps): warps 0..7 run the state chain (thread = value row
// 32 (warp % 4) + lane, column half warp / 4); their thread 0 issues the
// loads, U, C12 and C34.  Warps 8..15 prepare the next chunk: gates and their
// cumulants, L2 norms with the decay-scaled copy Kt, Ta = Tb diag(e^G); their
// thread 0 then issues K Q^T and W (and signals that U's operands are ready),
// and P^T, -W and Qh follow once those products are done ("chunk ready").
// Each issuing thread commits only its own products.  Roles hand over through
// mbarriers (bounded waits); each role makes a failed wait uniform before
// leaving.
constexpr int PQ_THREADS = 512;
constexpr int kPrep = 256;    // preparation threads
constexpr int qKQ = 0;        // 2 x 32 KB: [K; Q] landing tiles (K rows become -W, Q rows Qh)
constexpr int qV = 65536;     // 2 x 16 KB: V landing tiles (MN-major V^T operand)
constexpr int qTb = 98304;    // 2 x 8 KB: Tb tiles
constexpr int qPK = 114688;   // 2 x 24 KB: MN-major blocks [64 j][64]: P^T, Kt (d < 64), Kt (d >= 64)
constexpr int qTa = 163840;   // 8 KB
constexpr int qDT = 172032;   // 16 KB: D^T [128 i][64 j]
constexpr int qS = 188416;    // 32 KB: fp16 mirror of the state
constexpr int qSc = 221184;   // 3 slots (chunk % 3) of per-token factors, 7 x 64 fp32 each
constexpr int kScal = 7 * 64 * 4;
constexpr int qBar = qSc + 3 * kScal;  // mbarriers, TMEM address
constexpr int PQ_SMEM = qBar + 256 + 1024;
// tensor memory columns
constexpr uint32_t pU = 0, pD = 64, pO = 128, pS = 192, pI1 = 320, pW = 384;
// per-token factors of one chunk (offsets in floats): G (cumulative log decay) and IK = 1 / |k|
// as the solve kernel wrote them (one bulk copy), then e^G, KF = e^{G_C - G} / |k| (rows of Kt),
// TF = -e^G / |k| (columns of Ta), QF = scale e^G / |q| (rows of Qh), QS = scale / |q|
// (columns of P^T)
constexpr int fG = 0, fIK = 64, fEG = 128, fKF = 192, fTF = 256, fQF = 320, fQS = 384;

// byte offset of 16-byte chunk `ch` of row `r` in a 128-byte-swizzled block
__device__ __forceinline__ int sw(int r, int ch) { return r * 128 + ((ch ^ (r & 7)) << 4); }

// Scales the eight fp16 values of one 16-byte chunk by f: fp16 products while
// the factor is well inside the fp16 range, fp32 products beyond it (the
// factor 1 / |x| of an all-zero padding row is 1e6: 0 x 1e6 must stay 0).
constexpr float kHalfSafe = 8192.f;
__device__ __forceinline__ uint4 scale_chunk(uint4 u, float f) {
    __half2 *hp = reinterpret_cast<__half2 *>(&u);
    if (fabsf(f) <= kHalfSafe) {
        const __half2 f2 = __float2half2_rn(f);
#pragma unroll
        for (int w = 0; w < 4; ++w) hp[w] = __hmul2(hp[w], f2);
    } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float2 x = __half22float2(hp[w]);
            hp[w] = __floats2half2_rn(x.x * f, x.y * f);
        }
    }
    return u;
}
// scales the eight fp16 values of one chunk by eight factors (same rule)
__device__ __forceinline__ uint4 scale_chunk8(uint4 u, const float *f) {
    const float4 a = *reinterpret_cast<const float4 *>(f), b = *reinterpret_cast<const float4 *>(f + 4);
    const float fv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(fv[e]));
    __half2 *hp = reinterpret_cast<__half2 *>(&u);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        if (m <= kHalfSafe) {
            hp[w] = __hmul2(hp[w], __floats2half2_rn(fv[2 * w], fv[2 * w + 1]));
        } else {
            const float2 x = __half22float2(hp[w]);
            hp[w] = __floats2half2_rn(x.x * fv[2 * w], x.y * fv[2 * w + 1]);
        }
    }
    return u;
}

template <bool RETR>
__global__ void __launch_bounds__(PQ_THREADS, 1)
    chunked_pipe_kernel(Problem p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmT,
                        const int *offs, const float *fac, int cap) {
    extern __shared__ unsigned char smraw[];
    const uint32_t sb0 = ptx::smem_u32(smraw);
    unsigned char *sm = smraw + (((sb0 + 1023u) & ~1023u) - sb0);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + qBar);
    uint64_t *land = bars + 0;    // [2] TMA landed
    uint64_t *barU = bars + 2;    // U^T = V^T Tb^T done
    uint64_t *prepA = bars + 3;   // operands of K Q^T, W and U ready (one phase per chunk)
    uint64_t *prepB = bars + 4;   // [2] -W and Qh ready (C12's operands)
    uint64_t *prepC = bars + 11;  // [2] P^T and Kt ready (C34's operands)
    uint64_t *barPM = bars + 6;   // [2] K Q^T and W done
    uint64_t *barD = bars + 8;    // C12 done
    uint64_t *barX = bars + 9;    // [2] C34 done
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + qBar + 128);
    unsigned char *sS = sm + qS, *sTa = sm + qTa, *sDT = sm + qDT;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % p.Hv, b = blockIdx.x / p.Hv;
    const int row = state_row(p, b, h == 0 && tid == 0);
    if (row < 0) return;
    int t0, t1;
    request_range(p, b, t0, t1);
    const int qh = (int)((long long)h * p.Hq / p.Hv);
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
    const size_t sbase = ((size_t)row * p.Hv + h) * 128 * 128;
    if (nch == 0) {  // empty request: copy the incoming state through
        if (p.fin != p.init) {
            for (int idx = tid; idx < 128 * 32; idx += PQ_THREADS)
                reinterpret_cast<float4 *>(p.fin + sbase)[idx] =
                    p.init ? reinterpret_cast<const float4 *>(p.init + sbase)[idx] : make_float4(0, 0, 0, 0);
        }
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < 13; ++i) ptx::mbar_init(&bars[i], 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tslot, TC_TMEM_COLS);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
// ---- loads and products (each issued by one thread of the role that needs it)
    const uint32_t aS = ptx::smem_u32(sS), aTa = ptx::smem_u32(sTa), aDT = ptx::smem_u32(sDT);
    auto tma = [&](int c) {
        const int bf = c & 1;
        ptx::mbar_arrive_expect_tx(&land[bf], kLandBytes + kFacFloats * 4 + (RETR ? (uint32_t)kTbBytes : 0u));
        // the chunk's G and 1 / |k| into the factor slot of chunk c
        ptx::bulk_g2s(sm + qSc + (c % 3) * kScal, fac + ((size_t)(slot0 + c) * p.Hv + h) * kFacFloats,
                      kFacFloats * 4, &land[bf]);
        unsigned char *kq = sm + qKQ + bf * 32768, *vt = sm + qV + bf * 16384;
        const int c0 = t0 + TC_C * c;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
            ptx::tma_load_3d(kq + kb * 16384, &tmK, 64 * kb, qh, c0, &land[bf]);
            ptx::tma_load_3d(kq + kb * 16384 + 8192, &tmQ, 64 * kb, qh, c0, &land[bf]);
            ptx::tma_load_3d(vt + kb * 8192, &tmV, 64 * kb, h, c0, &land[bf]);
        }
        if (RETR) ptx::tma_load_2d(sm + qTb + bf * kTbBytes, &tmT, 0, ((slot0 + c) * p.Hv + h) * TC_C, &land[bf]);
    };
    // K Q^T (M = 64) and W = Ta K (M = 64, N = 128)
    auto prep_mma = [&](int c) {
        const int bf = c & 1;
        const uint32_t aKQ = ptx::smem_u32(sm + qKQ + bf * 32768);
#pragma unroll
        for (int s = 0; s < 8; ++s)
            tc::mma_f16(tmem + pI1, tc::desc_sw128(aKQ + (s >> 2) * 16384 + (s & 3) * 32),
                        tc::desc_sw128(aKQ + 8192 + (s >> 2) * 16384 + (s & 3) * 32), tc::idesc_f16(64, 64),
                        s > 0);
        if (RETR) {
#pragma unroll
            for (int s = 0; s < 4; ++s)
                tc::mma_f16(tmem + pW, tc::desc_sw128(aTa + s * 32), tc::desc_sw128(aKQ + s * 2048, 16384),
                            tc::idesc_f16(64, 128, false, true), s > 0);
        }
        tc::commit(&barPM[bf]);
    };
    // U^T = V^T Tb^T (M = 128, N = 64)
    auto u_mma = [&](int c) {
        const int bf = c & 1;
        const uint32_t aV = ptx::smem_u32(sm + qV + bf * 16384), aTb = ptx::smem_u32(sm + qTb + bf * kTbBytes);
#pragma unroll
        for (int s = 0; s < 4; ++s)
            tc::mma_f16(tmem + pU, tc::desc_sw128(aV + s * 2048, 8192), tc::desc_sw128(aTb + s * 32),
                        tc::idesc_f16(128, 64, true, false), s > 0);
        tc::commit(barU);
    };
    // U of chunk c once its V and Tb tiles are ready (U's tensor memory was read by
    // the D^T epilogue of chunk c - 1 before this is called)
    auto u_product = [&](int c) -> bool {
        if (!ptx::mbar_wait_sleep(prepA, c & 1)) return false;
        tc::fence_after();
        u_mma(c);
        return true;
    };
    // C12: [D^T | O^T] = S [-W; Qh]^T once the preparation of chunk c is done
    auto c12 = [&](int c) -> bool {
        const int bf = c & 1;
        if (!ptx::mbar_wait_sleep(&prepB[bf], (c >> 1) & 1)) return false;
        tc::fence_after();
        const uint32_t aKQ = ptx::smem_u32(sm + qKQ + bf * 32768);
#pragma unroll
        for (int s = 0; s < 8; ++s)
            tc::mma_f16(tmem + pD, tc::desc_sw128(aS + (s >> 2) * 16384 + (s & 3) * 32),
                        tc::desc_sw128(aKQ + (s >> 2) * 16384 + (s & 3) * 32), tc::idesc_f16(128, 128), s > 0);
        tc::commit(barD);
        return true;
    };
    // C34: [O^T | S] += D^T [P^T | Kt]   (B MN-major: three 64-wide blocks)
    auto c34 = [&](int c) -> bool {
        const int bf = c & 1;
        if (!ptx::mbar_wait_sleep(&prepC[bf], (c >> 1) & 1)) return false;
        tc::fence_after();
        const uint32_t aPK = ptx::smem_u32(sm + qPK + bf * 24576);
#pragma unroll
        for (int s = 0; s < 4; ++s)
            tc::mma_f16(tmem + pO, tc::desc_sw128(aDT + s * 32), tc::desc_sw128(aPK + s * 2048, 8192),
                        tc::idesc_f16(128, 192, false, true), true);
        tc::commit(&barX[bf]);
        return true;
    };

    if (warp < 8) {
        // ===================== state chain (256 threads)
        const int q4 = warp & 3, hc = warp >> 2, i = 32 * q4 + lane, ct = tid;
        const uint32_t lo = tmem + ((uint32_t)(32 * q4) << 16);
        const size_t srow = sbase + (size_t)i * 128 + 64 * hc;
        {
            float v[32];
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 f = p.init ? *reinterpret_cast<const float4 *>(p.init + srow + 32 * pc + 4 * j)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[4 * j] = f.x, v[4 * j + 1] = f.y, v[4 * j + 2] = f.z, v[4 * j + 3] = f.w;
                }
                tc::st32(lo + pS + 64 * hc + 32 * pc, v);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) st_chunk(sS + hc * 16384, i, 4 * pc + cc, v + 8 * cc);
            }
            tc::wait_st();
        }
        tc::fence_async_smem();
        tc::fence_before();
        ptx::named_bar_sync(1, 256);
        bool ok = true;
        if (ct == 0) {
            tc::fence_after();
            tma(0);
            if (nch > 1) tma(1);
            ok = u_product(0) && c12(0);
        }
        for (int c = 0; c < nch; ++c) {
            const int bf = c & 1;
            const float *scal = reinterpret_cast<const float *>(sm + qSc + (c % 3) * kScal);
            const int n = min(TC_C, t1 - (t0 + TC_C * c));
            // ---- C12 and U done: D^T = U^T + (-S W^T) -> fp16 operand; S *= e^{G_C}
            ok = ptx::named_bar_and(1, 256, ok && ptx::mbar_wait_sleep(barD, c & 1) && ptx::mbar_wait_sleep(barU, c & 1));
            if (!ok) break;
            tc::fence_after();
            {
                float u[32], d[32];
                tc::ld32(lo + pU + 32 * hc, u);
                tc::ld32(lo + pD + 32 * hc, d);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) u[jj] += d[jj];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) st_chunk(sDT, i, 4 * hc + cc, u + 8 * cc);
                if (rule_has_decay(p.rule)) {
                    const float eC = scal[fEG + TC_C - 1];
#pragma unroll
                    for (int pc = 0; pc < 2; ++pc) {
                        tc::ld32(lo + pS + 64 * hc + 32 * pc, d);
#pragma unroll
                        for (int jj = 0; jj < 32; ++jj) d[jj] *= eC;
                        tc::st32(lo + pS + 64 * hc + 32 * pc, d);
                    }
                    tc::wait_st();
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(1, 256);
            if (ct == 0) {
                tc::fence_after();
                ok = c34(c);
                // chunk c's landing buffer is free: C12, U and the preparation have run
                if (c + 2 < nch) tma(c + 2);
                if (c + 1 < nch) ok = ok && u_product(c + 1);
            }
            // ---- C34 done: mirror the state, read O^T, start C12 of the next chunk
            ok = ptx::named_bar_and(1, 256, ok && ptx::mbar_wait_sleep(&barX[bf], (c >> 1) & 1));
            if (!ok) break;
            tc::fence_after();
            float o[32];
            {
                float v[32];
#pragma unroll
                for (int pc = 0; pc < 2; ++pc) {
                    tc::ld32(lo + pS + 64 * hc + 32 * pc, v);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) st_chunk(sS + hc * 16384, i, 4 * pc + cc, v + 8 * cc);
                }
                tc::ld32(lo + pO + 32 * hc, o);
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(1, 256);
            if (ct == 0 && c + 1 < nch) ok = c12(c + 1);
            // ---- outputs of chunk c: O^T[i][r] straight to O[r][i] (a warp writes 64 contiguous
            // bytes of each token row)
            {
                __half *orow = static_cast<__half *>(p.o) + ((size_t)(t0 + TC_C * c + 32 * hc) * p.Hv + h) * 128 + i;
                const size_t rstride = (size_t)p.Hv * 128;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    if (32 * hc + jj < n) orow[jj * rstride] = __float2half_rn(o[jj]);
            }
        }
        if (!ok && p.err && ct == 0) atomicOr(p.err, 2);
        if (ok) {
            float v[32];
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
                tc::ld32(lo + pS + 64 * hc + 32 * pc, v);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4 *>(p.fin + srow + 32 * pc + 4 * j) =
                        make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
        }
    } else if (warp < 16) {
        // ===================== next-chunk preparation (256 threads)
        // The key and query tiles stay as loaded.  The decays, the L2 norms and the
        // output scale enter through per-token factors (the solve kernel supplies G and
        // 1 / |k|): Kt rows, Ta columns (which also carry the sign of -W), Qh rows and
        // the rows / columns of P^T.  Two signals per chunk: C12's operands (-W, Qh),
        // then C34's (P^T; Kt is written earlier).
        const int pt = tid - 256, pw = warp - 8, pq = pw & 3, ph = pw >> 2;
        const uint32_t lo = tmem + ((uint32_t)(32 * pq) << 16);
        const bool nq = (p.flags & kL2q) != 0;
        if (!RETR) {
            // Tb = I (U^T = V^T), in both buffers, once
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int idx = pt + kPrep * w, bf = idx >> 9, r = (idx >> 3) & 63, ch = idx & 7;
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = (8 * ch + e == r) ? 1.f : 0.f;
                st_chunk(sm + qTb + bf * kTbBytes, r, ch, x);
            }
        }
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int bf = c & 1;
            const int c0 = t0 + TC_C * c, n = min(TC_C, t1 - c0);
            unsigned char *sKQ = sm + qKQ + bf * 32768, *sV = sm + qV + bf * 16384;
            unsigned char *sTb = sm + qTb + bf * kTbBytes, *sPK = sm + qPK + bf * 24576;
            float *F = reinterpret_cast<float *>(sm + qSc + (c % 3) * kScal);
            // landed (tiles and factors); PK[bf] was last read by C34 of chunk c - 2
            bool okw = ptx::mbar_wait_sleep(&land[bf], (c >> 1) & 1);
            if (c >= 2) okw = okw && ptx::mbar_wait_sleep(&barX[bf], ((c - 2) >> 1) & 1);
            ok = ptx::named_bar_and(2, kPrep, okw);
            if (!ok) break;
            if (n < TC_C) {  // the boxes run past this request: clear the rows beyond it
                const int nz = (TC_C - n) * 16;
                for (int idx = pt; idx < 3 * nz; idx += kPrep) {
                    const int which = idx / nz, rem = idx % nz, r = n + (rem >> 4), ch = rem & 15;
                    unsigned char *base = which == 2 ? sV + (ch >> 3) * 8192
                                                     : sKQ + (ch >> 3) * 16384 + (which == 1 ? 8192 : 0);
                    *reinterpret_cast<uint4 *>(base + sw(r, ch & 7)) = make_uint4(0, 0, 0, 0);
                }
            }
            if (nq) {
                // 1 / |q_r|, four threads per query row (kept in QS until the factors below)
                ptx::named_bar_sync(2, kPrep);
                const int r = pt >> 2, part = pt & 3;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int ch = 4 * part + w;
                    const uint4 uq = *reinterpret_cast<const uint4 *>(sKQ + (ch >> 3) * 16384 + sw(64 + r, ch & 7));
                    const __half2 *hp = reinterpret_cast<const __half2 *>(&uq);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __half22float2(hp[e]);
                        s0 = fmaf(f.x, f.x, s0);
                        s1 = fmaf(f.y, f.y, s1);
                    }
                }
                float ss = s0 + s1;
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                if (part == 0) F[fQS + r] = rsqrtf(ss + 1e-12f);
                ptx::named_bar_sync(2, kPrep);
            }
            if (pt < TC_C) {
                const float G = F[fG + pt], ik = F[fIK + pt], eg = __expf(G);
                const float iq = nq ? F[fQS + pt] : 1.f;
                F[fEG + pt] = eg;
                F[fKF + pt] = __expf(F[fG + TC_C - 1] - G) * ik;  // e^{G_C - G} <= 1
                F[fTF + pt] = -eg * ik;
                F[fQF + pt] = p.scale * eg * iq;
                F[fQS + pt] = p.scale * iq;
            }
            ptx::named_bar_sync(2, kPrep);
            if (RETR) {
                // Ta = -Tb diag(e^G / |k|): W = Ta K comes out as -W (the K rows stay unnormalised)
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int idx = 2 * pt + w, tr = idx >> 3, ch = idx & 7;
                    const uint4 u = *reinterpret_cast<const uint4 *>(sTb + sw(tr, ch));
                    *reinterpret_cast<uint4 *>(sTa + sw(tr, ch)) = scale_chunk8(u, F + fTF + 8 * ch);
                }
            }
            // the operands of K Q^T, W and U are ready: issue the first two, signal U
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(2, kPrep);
            if (pt == 0) {
                tc::fence_after();
                prep_mma(c);
                ptx::mbar_arrive(prepA);
            }
            // Kt[j][d] = e^{G_C - G_j} k_j[d] / |k_j| into PK blocks 1 and 2, while those run
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int idx = pt + kPrep * w, j = idx >> 4, ch = idx & 15;
                const uint4 u = *reinterpret_cast<const uint4 *>(sKQ + (ch >> 3) * 16384 + sw(j, ch & 7));
                *reinterpret_cast<uint4 *>(sPK + 8192 + (ch >> 3) * 8192 + sw(j, ch & 7)) = scale_chunk(u, F[fKF + j]);
            }
            // ---- K Q^T and W = Ta K done (and every thread is past its Kt rows)
            ok = ptx::named_bar_and(2, kPrep, ptx::mbar_wait_sleep(&barPM[bf], (c >> 1) & 1));
            if (!ok) break;
            tc::fence_after();
            // M = 64 results: rows 16 pq .. 16 pq + 15 sit on lanes 32 pq .. 32 pq + 15; the
            // 16x256b shape spreads them over the warp: rows ja, ja + 8, column pairs 2 (lane % 4)
            const int ja = 16 * pq + (lane >> 2), jb = ja + 8, cp = 2 * (lane & 3);
            float vp[16];
            tc::ld16x256<4>(lo + pI1 + 32 * ph, vp);
            if (RETR) {
                // -W over the key rows: columns [64 ph, 64 ph + 64) = key block ph
                float v[32];
                tc::ld16x256<8>(lo + pW + 64 * ph, v);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    *reinterpret_cast<uint32_t *>(sKQ + ph * 16384 + sw(ja, k) + 2 * cp) =
                        ptx::pack_h2(v[4 * k], v[4 * k + 1]);
                    *reinterpret_cast<uint32_t *>(sKQ + ph * 16384 + sw(jb, k) + 2 * cp) =
                        ptx::pack_h2(v[4 * k + 2], v[4 * k + 3]);
                }
            }
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int idx = pt + kPrep * w, r = idx >> 4, ch = idx & 15;
                if (!RETR)  // W = 0: clear the key rows
                    *reinterpret_cast<uint4 *>(sKQ + (ch >> 3) * 16384 + sw(r, ch & 7)) = make_uint4(0, 0, 0, 0);
                // query rows -> scale e^{G_r} q_r / |q_r| in place (K Q^T has read the raw rows)
                uint4 *ptr = reinterpret_cast<uint4 *>(sKQ + (ch >> 3) * 16384 + sw(64 + r, ch & 7));
                *ptr = scale_chunk(*ptr, F[fQF + r]);
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(2, kPrep);
            if (pt == 0) ptx::mbar_arrive(&prepB[bf]);
            {
                // P^T[j][r] = scale e^{G_r - G_j} k_j . q_r / (|k_j| |q_r|) for r >= j
                const float Ga = F[fG + ja], Gb = F[fG + jb], ka = F[fIK + ja], kb = F[fIK + jb];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r0 = 32 * ph + 8 * k + cp;
                    const float2 g = *reinterpret_cast<const float2 *>(F + fG + r0);
                    const float2 qs = *reinterpret_cast<const float2 *>(F + fQS + r0);
                    const float a0 = r0 >= ja ? __expf(g.x - Ga) * ka * qs.x * vp[4 * k] : 0.f;
                    const float a1 = r0 + 1 >= ja ? __expf(g.y - Ga) * ka * qs.y * vp[4 * k + 1] : 0.f;
                    const float b0 = r0 >= jb ? __expf(g.x - Gb) * kb * qs.x * vp[4 * k + 2] : 0.f;
                    const float b1 = r0 + 1 >= jb ? __expf(g.y - Gb) * kb * qs.y * vp[4 * k + 3] : 0.f;
                    const int ch = 4 * ph + k;
                    *reinterpret_cast<uint32_t *>(sPK + sw(ja, ch) + 2 * cp) = ptx::pack_h2(a0, a1);
                    *reinterpret_cast<uint32_t *>(sPK + sw(jb, ch) + 2 * cp) = ptx::pack_h2(b0, b1);
                }
            }
            tc::fence_async_smem();
            tc::fence_before();
            ptx::named_bar_sync(2, kPrep);
            if (pt == 0) ptx::mbar_arrive(&prepC[bf]);
        }
        if (!ok && p.err && pt == 0) atomicOr(p.err, 2);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, TC_TMEM_COLS);
}

bool al16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// slots for every chunk of pairwise disjoint requests: sum ceil(len / C) <= T / C + B
int slot_capacity(const Problem &p) { return (int)((long long)p.T / TC_C + p.B + 1); }
// workspace: chunk offsets (B + 1 ints) and the slot -> request table (one int per
// slot), rounded up to 1 KB, then the Tb tiles
size_t offs_bytes(const Problem &p) {
    return (((size_t)p.B + 1 + (size_t)slot_capacity(p)) * sizeof(int) + 1023) & ~(size_t)1023;
}

}  // namespace

bool chunked_tc_eligible(const Problem &p) {
    const bool rule_ok = p.rule == kLinear || p.rule == kGated || p.rule == kDelta || p.rule == kGatedDelta;
    return rule_ok && p.dk == 128 && p.dv == 128 && p.act_f16 && !((p.flags & kPerKey) && rule_has_decay(p.rule)) &&
           al16(p.q) && al16(p.k) && al16(p.v) && al16(p.fin) && (p.init == nullptr || al16(p.init));
}

// workspace: [offsets | slot table] [Tb tiles (delta rules)] [per-chunk factors]
size_t tb_bytes(const Problem &p) {
    return rule_has_retrieval(p.rule) ? (size_t)slot_capacity(p) * p.Hv * kTbBytes : 0;
}
size_t chunked_tc_workspace_bytes(const Problem &p) {
    if (p.B == 0) return 0;
    return offs_bytes(p) + tb_bytes(p) + (size_t)slot_capacity(p) * p.Hv * kFacFloats * 4;
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

// [T, H, 128] fp16 rows -> boxes of 64 channels x 1 head x 64 tokens, 128-byte swizzle.
static bool make_map(CUtensorMap *m, const void *base, int heads, int tokens) {
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

// Tb tiles: rows of 64 fp16, one 64 x 64 box per (slot, head), 128-byte swizzle.
static bool make_map_tb(CUtensorMap *m, const void *base, long long rows) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {64, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {64 * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_chunked_tc(const Problem &p, void *ws, size_t ws_bytes, cudaStream_t stream) {
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(chunk_solve_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SV_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chunk_solve_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SV_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chunked_pipe_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, PQ_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chunked_pipe_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, PQ_SMEM);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_done[dev] = 1;
    }
    CUtensorMap tk, tq, tv, tt;
    if (!make_map(&tk, p.k, p.Hq, p.T) || !make_map(&tq, p.q, p.Hq, p.T) || !make_map(&tv, p.v, p.Hv, p.T))
        return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)((long long)p.B * p.Hv);
    if (grid == 0) return cudaSuccess;
    if (ws == nullptr || ws_bytes < chunked_tc_workspace_bytes(p)) return cudaErrorInvalidValue;
    const bool retr = rule_has_retrieval(p.rule);
    int *offs = static_cast<int *>(ws);
    int *slot_req = offs + p.B + 1;
    unsigned char *wsb = static_cast<unsigned char *>(ws);
    __half *tb = reinterpret_cast<__half *>(wsb + offs_bytes(p));
    float *fac = reinterpret_cast<float *>(wsb + offs_bytes(p) + tb_bytes(p));
    const int cap = slot_capacity(p);
    if (retr) {
        if (!make_map_tb(&tt, tb, (long long)cap * p.Hv * TC_C)) return cudaErrorInvalidValue;
    } else {
        tt = tk;  // unused without retrieval
    }
    chunk_offsets_kernel<<<1, 1024, 0, stream>>>(p, offs, slot_req, cap);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // persistent solver CTAs: three per SM (shared memory), at most one per task
    const long long tasks = (long long)cap * p.Hv;
    const long long sgrid = std::min<long long>(tasks, 3LL * sm_count());
    if (retr)
        chunk_solve_kernel<true><<<(unsigned)sgrid, SV_THREADS, SV_SMEM, stream>>>(p, tk, offs, slot_req, tb, fac, cap);
    else
        chunk_solve_kernel<false><<<(unsigned)sgrid, SV_THREADS, SV_SMEM, stream>>>(p, tk, offs, slot_req, tb, fac,
                                                                                   cap);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (retr)
        chunked_pipe_kernel<true><<<grid, PQ_THREADS, PQ_SMEM, stream>>>(p, tk, tq, tv, tt, offs, fac, cap);
    else
        chunked_pipe_kernel<false><<<grid, PQ_THREADS, PQ_SMEM, stream>>>(p, tk, tq, tv, tt, offs, fac, cap);
    return cudaGetLastError();
}

}  // namespace gdn
