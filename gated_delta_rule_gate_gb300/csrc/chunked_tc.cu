// chunked_tc.cu -- chunk-parallel prefill on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory), for dk = dv = 128, fp16
// activations, scalar decay, rules linear / gated / delta / gated_delta.
//
// Same per-chunk algebra as chunked.cu (derived from the token recurrence;
// see the comment there), written "transposed" so that the M = 128 side of
// every tensor-core product is the value axis of the V-major state: lane i
// of tensor memory is value row i.  For one chunk of C = 64 tokens:
//
//   I1:  [K; Q] K^T      -> rows 0..63: K K^T (the system), rows 64..127: Q K^T
//   I2:  W^T  = K^T Ta^T       Ta = T diag(beta e^G),  T = (I + A)^-1
//   C1:  D^T  = V^T Tb^T - S W^T   Tb = T diag(beta)   (D = the token corrections)
//   C2:  O^T  = S Qh^T + D^T P^T   Qh = diag(e^G) Q,  P = decayed causal Q K^T
//   C4:  X    = (D^T diag(e^{G_C - G})) K
//   S   <- e^{G_C} S + X                               (fp32, in registers)
//
// Operands are fp16 tiles in shared memory with the 128-byte swizzle.  The
// key/query chunk lands (cp.async) as a 128-row K-major tile [K; Q]; its key
// rows double as the MN-major K^T operand of I2 and C4, and the value chunk
// lands as the MN-major V^T operand, so nothing is transposed by hand.  The
// fp32 state lives in registers of the 8 warps (row i, 64 columns each) and
// is mirrored each chunk into an fp16 K-major tile, the A operand of C1/C2.
// The unit-lower-triangular solve runs in fp32 on the CUDA cores.  The next
// chunk's loads are in flight while the current chunk computes.  One CTA of
// 256 threads per (request, value head); one thread issues every MMA and
// tracks completion through an mbarrier (bounded waits).
#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace gdn {
namespace {

constexpr int TC_C = 64;        // tokens per chunk
constexpr int TC_THREADS = 256;  // 8 warps
constexpr int TC_TMEM_COLS = 512;

// shared memory layout (bytes from a 1024-aligned base)
constexpr int oKQ = 0;            // 2 x 32 KB: [K; Q] landing tiles, 128 rows x 128 dk, K-major
constexpr int oV = 65536;         // 2 x 16 KB: V landing tiles, MN-major (rows = tokens)
constexpr int oS = 98304;         // 32 KB: fp16 state, 128 rows x 128 dk, K-major
constexpr int oTa = 131072;       // 8 KB: [64 r][64 j]
constexpr int oTb = 139264;       // 8 KB
constexpr int oP = 147456;        // 8 KB
constexpr int oR = 155648;        // 48 KB region: solve scratch, then W | DT | DTs
constexpr int oW = oR;            // 16 KB: [64 r][128 c], K-major
constexpr int oDT = oR + 16384;   // 16 KB: [128 i][64 j]
constexpr int oDTs = oR + 32768;  // 16 KB
constexpr int oAf = oR;           // fp32 [64][65]
constexpr int oTf = oR + 16640;   // fp32 [64][65]
constexpr int oX16 = oR + 33280;  // fp32 [4][16][17]
constexpr int oScal = oR + 49152; // fp32 G, beta, e^G, e^{G_C - G}: 4 x 64
constexpr int oBar = oScal + 1024;
constexpr int TC_SMEM = oBar + 16 + 1024;  // + alignment slack

constexpr int FS = 65;

// byte offset of element (row, k) in a K-major 128B-swizzled tile with `rows`
// rows per 64-column block
__device__ __forceinline__ int swz(int row, int k, int rows) {
    return (k >> 6) * rows * 128 + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) + (k & 7) * 2;
}
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

__device__ __forceinline__ void sync_tc() {
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
}

__device__ __forceinline__ bool wait_mma(uint64_t *bar, uint32_t &phase, int32_t *err) {
    const bool ok = ptx::mbar_wait(bar, phase);
    phase ^= 1u;
    if (!ok && err && threadIdx.x == 0) atomicOr(err, 2);
    tc::fence_after();
    return ok;
}

__device__ __forceinline__ void issue_loads(const Problem &p, unsigned char *kq, unsigned char *vt, int c0, int n,
                                            int h, int qh) {
    const __half *kg = static_cast<const __half *>(p.k);
    const __half *qg = static_cast<const __half *>(p.q);
    const __half *vg = static_cast<const __half *>(p.v);
    for (int idx = threadIdx.x; idx < 128 * 16; idx += TC_THREADS) {
        const int row = idx >> 4, ch = idx & 15, rr = row & 63;
        const bool ok = rr < n;
        const __half *src = ok ? (row < 64 ? kg : qg) + (((size_t)(c0 + rr) * p.Hq + qh) * 128 + ch * 8) : kg;
        ptx::cp_async16(kq + (ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ (row & 7)) << 4), src, ok ? 16 : 0);
    }
    for (int idx = threadIdx.x; idx < 64 * 16; idx += TC_THREADS) {
        const int j = idx >> 4, ch = idx & 15;
        const bool ok = j < n;
        const __half *src = ok ? vg + (((size_t)(c0 + j) * p.Hv + h) * 128 + ch * 8) : vg;
        ptx::cp_async16(vt + (ch >> 3) * 8192 + j * 128 + (((ch & 7) ^ (j & 7)) << 4), src, ok ? 16 : 0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <bool RETR>
__global__ void __launch_bounds__(TC_THREADS, 1) chunked_tc_kernel(Problem p) {
    extern __shared__ unsigned char smraw[];
    const uint32_t sb0 = ptx::smem_u32(smraw);
    unsigned char *sm = smraw + (((sb0 + 1023u) & ~1023u) - sb0);
    unsigned char *sS = sm + oS, *sTa = sm + oTa, *sTb = sm + oTb, *sP = sm + oP;
    unsigned char *sW = sm + oW, *sDT = sm + oDT, *sDTs = sm + oDTs;
    float *sAf = reinterpret_cast<float *>(sm + oAf);
    float *sTf = reinterpret_cast<float *>(sm + oTf);
    float *sX16 = reinterpret_cast<float *>(sm + oX16);
    float *sG = reinterpret_cast<float *>(sm + oScal);
    float *sB = sG + 64, *sEG = sG + 128, *sEGC = sG + 192;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + oBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + oBar + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hc = warp >> 2;
    const int ell = 32 * q4 + lane;  // tensor-memory lane = row served by this thread
    const int h = blockIdx.x % p.Hv, b = blockIdx.x / p.Hv;
    const int row = state_row(p, b, h == 0 && tid == 0);
    if (row < 0) return;
    int t0, t1;
    request_range(p, b, t0, t1);
    const int qh = (int)((long long)h * p.Hq / p.Hv);
    const bool has_decay = rule_has_decay(p.rule);
    const bool sig = (p.flags & kBetaSigmoid) != 0;

    // ---- the fp32 state: row ell, columns [64 hc, 64 hc + 64)
    float Sr[64];
    const size_t srow = (((size_t)row * p.Hv + h) * 128 + ell) * 128 + 64 * hc;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float4 v = p.init ? *reinterpret_cast<const float4 *>(p.init + srow + 4 * j) : make_float4(0, 0, 0, 0);
        Sr[4 * j] = v.x, Sr[4 * j + 1] = v.y, Sr[4 * j + 2] = v.z, Sr[4 * j + 3] = v.w;
    }
    if (t1 == t0) {  // empty request: copy the incoming state through
        if (p.fin != p.init) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                *reinterpret_cast<float4 *>(p.fin + srow + 4 * j) =
                    make_float4(Sr[4 * j], Sr[4 * j + 1], Sr[4 * j + 2], Sr[4 * j + 3]);
        }
        return;
    }

    if (tid == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tslot, TC_TMEM_COLS);
    // the fp16 mirror of the state
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) st_chunk(sS + hc * 16384, ell, ch, Sr + 8 * ch);
    issue_loads(p, sm + oKQ, sm + oV, t0, min(TC_C, t1 - t0), h, qh);
    float graw = 0.f, braw = 0.f;
    if (tid < TC_C && tid < t1 - t0) {
        const size_t th = (size_t)(t0 + tid) * p.Hv + h;
        if (has_decay) graw = ld_any(p.decay, th, p.decay_f16);
        if (RETR) braw = ld_any(p.beta, th, p.beta_f16);
    }
    tc::fence_async_smem();
    sync_tc();
    const uint32_t tmem = *tslot;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const uint32_t tI1 = tmem, tWT = tmem + 64, tD = tmem + 128, tO = tmem + 192, tX = tmem + 256;
    uint32_t phase = 0;
    bool ok = true;
    const uint32_t IDN64 = tc::idesc_f16(128, 64);
    const uint32_t IDN64_AMN = tc::idesc_f16(128, 64, true, false);
    const uint32_t IDN64_NEGB = tc::idesc_f16(128, 64, false, false, true);
    const uint32_t IDN128_BMN = tc::idesc_f16(128, 128, false, true);
    const uint32_t aS = ptx::smem_u32(sS), aTa = ptx::smem_u32(sTa), aTb = ptx::smem_u32(sTb);
    const uint32_t aP = ptx::smem_u32(sP), aW = ptx::smem_u32(sW), aDT = ptx::smem_u32(sDT);
    const uint32_t aDTs = ptx::smem_u32(sDTs);

    int buf = 0;
    for (int c0 = t0; c0 < t1 && ok; c0 += TC_C, buf ^= 1) {
        const int n = min(TC_C, t1 - c0);
        unsigned char *sKQ = sm + oKQ + buf * 32768;
        unsigned char *sV = sm + oV + buf * 16384;
        const uint32_t aKQ = ptx::smem_u32(sKQ), aV = ptx::smem_u32(sV);
        ptx::cp_async_wait_all();
        __syncthreads();  // this chunk's tiles have landed; the other buffer is free
        if (c0 + TC_C < t1) issue_loads(p, sm + oKQ + (buf ^ 1) * 32768, sm + oV + (buf ^ 1) * 16384, c0 + TC_C,
                                        min(TC_C, t1 - c0 - TC_C), h, qh);
        if (tid < TC_C) {
            float g = 0.f, bt = 0.f;
            if (tid < n) {
                if (has_decay) g = p.raw_gate ? p.gate_scale[h] * softplus_f(graw + p.gate_bias[h]) : graw;
                bt = RETR ? (sig ? sigmoid_f(braw) : braw) : 1.f;
            }
            sG[tid] = g;
            sB[tid] = bt;
            graw = braw = 0.f;
            if (c0 + TC_C + tid < t1) {
                const size_t th = (size_t)(c0 + TC_C + tid) * p.Hv + h;
                if (has_decay) graw = ld_any(p.decay, th, p.decay_f16);
                if (RETR) braw = ld_any(p.beta, th, p.beta_f16);
            }
        }
        __syncthreads();
        // ---- cumulants (warp 0) and the L2 norms of the key / query rows
        if (warp == 0) {
            const float g0 = sG[2 * lane], g1 = sG[2 * lane + 1];
            float s = g0 + g1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            const float G1 = s, G0 = s - g1, GC = __shfl_sync(0xffffffffu, s, 31);
            sG[2 * lane] = G0, sG[2 * lane + 1] = G1;
            sEG[2 * lane] = expf(G0), sEG[2 * lane + 1] = expf(G1);
            sEGC[2 * lane] = expf(GC - G0), sEGC[2 * lane + 1] = expf(GC - G1);
        }
        {
            const bool nk = (p.flags & kL2k) != 0, nq = (p.flags & kL2q) != 0;
            if (nk || nq) {
                const int kb = lane >> 4, c = (4 * lane) & 63;
                for (int rr = warp; rr < 128; rr += 8) {
                    if ((rr < 64 && !nk) || (rr >= 64 && !nq)) continue;
                    uint2 *ptr = reinterpret_cast<uint2 *>(sKQ + kb * 16384 + rr * 128 +
                                                           ((((c >> 3)) ^ (rr & 7)) << 4) + (c & 7) * 2);
                    uint2 u = *ptr;
                    float2 a = __half22float2(*reinterpret_cast<__half2 *>(&u.x));
                    float2 d = __half22float2(*reinterpret_cast<__half2 *>(&u.y));
                    const float inv = rsqrtf(warp_sum(a.x * a.x + a.y * a.y + d.x * d.x + d.y * d.y) + 1e-12f);
                    u.x = ptx::pack_h2(a.x * inv, a.y * inv);
                    u.y = ptx::pack_h2(d.x * inv, d.y * inv);
                    *ptr = u;
                }
            }
        }
        tc::fence_async_smem();
        sync_tc();

        // ---- I1: [K; Q] K^T
        if (tid == 0) {
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint64_t d = tc::desc_sw128(aKQ + (s >> 2) * 16384 + (s & 3) * 32);
                tc::mma_f16(tI1, d, d, IDN64, s > 0);
            }
            tc::commit(bar);
        }
        ok = wait_mma(bar, phase, p.err);
        {
            float v[32];
            tc::ld32(tI1 + lane_off + 32 * hc, v);
            if (ell < 64) {
                if (RETR) {
                    const int r = ell;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        const int j = 32 * hc + jj;
                        sAf[r * FS + j] = j < r ? sB[r] * expf(sG[r] - sG[j]) * v[jj] : 0.f;
                    }
                }
            } else {
                const int r = ell - 64;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = 32 * hc + jj;
                    v[jj] = j <= r ? expf(sG[r] - sG[j]) * v[jj] : 0.f;
                }
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) st_chunk(sP, r, 4 * hc + cc, v + 8 * cc);
            }
        }
        // query rows -> e^{G_r} q_r in place (I1 has consumed the raw rows)
        for (int idx = tid; idx < 64 * 16; idx += TC_THREADS) {
            const int r = idx >> 4, ch = idx & 15, rr = 64 + r;
            uint4 *ptr = reinterpret_cast<uint4 *>(sKQ + (ch >> 3) * 16384 + rr * 128 + (((ch & 7) ^ (rr & 7)) << 4));
            uint4 u = *ptr;
            const float e = sEG[r];
            __half2 *hp = reinterpret_cast<__half2 *>(&u);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                float2 f = __half22float2(hp[w]);
                hp[w] = __floats2half2_rn(f.x * e, f.y * e);
            }
            *ptr = u;
        }
        tc::fence_async_smem();
        sync_tc();

        if (RETR) {
            // ---- T = (I + A)^-1 in fp32: 16x16 diagonal blocks, then blocked updates
            if (warp < 4 && lane < 16) {
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
                if (warp < 4 && ib < 4) {
                    const int rr = lane >> 1, cc0 = (lane & 1) * 8;
                    float xs[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) xs[e] = 0.f;
                    for (int m = jb; m < ib; ++m) {
#pragma unroll 4
                        for (int qq = 0; qq < 16; ++qq) {
                            const float a = sAf[(16 * ib + rr) * FS + 16 * m + qq];
                            const float *tr = sTf + (16 * m + qq) * FS + 16 * jb + cc0;
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
                    for (int qq = 0; qq <= rr; ++qq) {
                        const float t = sTf[(16 * ib + rr) * FS + 16 * ib + qq];
#pragma unroll
                        for (int e = 0; e < 8; ++e) ts[e] += t * X[qq * 17 + cc0 + e];
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) sTf[(16 * ib + rr) * FS + 16 * jb + cc0 + e] = -ts[e];
                    __syncwarp();
                }
                __syncthreads();
            }
            {
                const int r = tid >> 2, qq = tid & 3;
                float ta[16], tb[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int j = 16 * qq + e;
                    const float t = j <= r ? sTf[r * FS + j] : 0.f;
                    tb[e] = t * sB[j];
                    ta[e] = tb[e] * sEG[j];
                }
                st_chunk(sTa, r, 2 * qq, ta);
                st_chunk(sTa, r, 2 * qq + 1, ta + 8);
                st_chunk(sTb, r, 2 * qq, tb);
                st_chunk(sTb, r, 2 * qq + 1, tb + 8);
            }
            tc::fence_async_smem();
            sync_tc();

            // ---- I2 (W^T = K^T Ta^T), C1a (V^T Tb^T), C2 (S Qh^T)
            if (tid == 0) {
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tc::mma_f16(tWT, tc::desc_sw128(aKQ + s * 2048, 16384), tc::desc_sw128(aTa + s * 32), IDN64_AMN,
                                s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tc::mma_f16(tD, tc::desc_sw128(aV + s * 2048, 8192), tc::desc_sw128(aTb + s * 32), IDN64_AMN,
                                s > 0);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    tc::mma_f16(tO, tc::desc_sw128(aS + (s >> 2) * 16384 + (s & 3) * 32),
                                tc::desc_sw128(aKQ + 8192 + (s >> 2) * 16384 + (s & 3) * 32), IDN64, s > 0);
                tc::commit(bar);
            }
            ok = wait_mma(bar, phase, p.err) && ok;
            {
                // W^T[c][r] (lane = key channel c) -> W tile [r][c]
                float v[32];
                tc::ld32(tWT + lane_off + 32 * hc, v);
                const int c = ell;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int r = 32 * hc + jj;
                    *reinterpret_cast<__half *>(sW + swz(r, c, 64)) = __float2half_rn(v[jj]);
                }
            }
            tc::fence_async_smem();
            sync_tc();
            // ---- C1b: D^T += S (-W)^T
            if (tid == 0) {
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    tc::mma_f16(tD, tc::desc_sw128(aS + (s >> 2) * 16384 + (s & 3) * 32),
                                tc::desc_sw128(aW + (s >> 2) * 8192 + (s & 3) * 32), IDN64_NEGB, true);
                tc::commit(bar);
            }
            ok = wait_mma(bar, phase, p.err) && ok;
            {
                float v[32], vs[32];
                tc::ld32(tD + lane_off + 32 * hc, v);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) vs[jj] = v[jj] * sEGC[32 * hc + jj];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    st_chunk(sDT, ell, 4 * hc + cc, v + 8 * cc);
                    st_chunk(sDTs, ell, 4 * hc + cc, vs + 8 * cc);
                }
            }
            tc::fence_async_smem();
            sync_tc();
            // ---- C3 (O^T += D^T P^T) and C4 (X = DTs K)
            if (tid == 0) {
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tc::mma_f16(tO, tc::desc_sw128(aDT + s * 32), tc::desc_sw128(aP + s * 32), IDN64, true);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tc::mma_f16(tX, tc::desc_sw128(aDTs + s * 32), tc::desc_sw128(aKQ + s * 2048, 16384),
                                IDN128_BMN, s > 0);
                tc::commit(bar);
            }
        } else {
            // rules without retrieval: D = V.  DTs = V^T diag(e^{G_C - G}) by hand.
            {
                const int i = ell;
                float vs[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = 32 * hc + jj;
                    const __half hv = *reinterpret_cast<const __half *>(
                        sV + (i >> 6) * 8192 + j * 128 + (((((i & 63) >> 3)) ^ (j & 7)) << 4) + (i & 7) * 2);
                    vs[jj] = __half2float(hv) * sEGC[j];
                }
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) st_chunk(sDTs, i, 4 * hc + cc, vs + 8 * cc);
            }
            tc::fence_async_smem();
            sync_tc();
            if (tid == 0) {
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    tc::mma_f16(tO, tc::desc_sw128(aS + (s >> 2) * 16384 + (s & 3) * 32),
                                tc::desc_sw128(aKQ + 8192 + (s >> 2) * 16384 + (s & 3) * 32), IDN64, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tc::mma_f16(tO, tc::desc_sw128(aV + s * 2048, 8192), tc::desc_sw128(aP + s * 32), IDN64_AMN,
                                true);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    tc::mma_f16(tX, tc::desc_sw128(aDTs + s * 32), tc::desc_sw128(aKQ + s * 2048, 16384),
                                IDN128_BMN, s > 0);
                tc::commit(bar);
            }
        }
        ok = wait_mma(bar, phase, p.err) && ok;

        // ---- S <- e^{G_C} S + X;  O stores
        {
            const float eC = sEG[TC_C - 1];
            float v[32];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                tc::ld32(tX + lane_off + 64 * hc + 32 * hh, v);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) Sr[32 * hh + jj] = fmaf(eC, Sr[32 * hh + jj], v[jj]);
            }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) st_chunk(sS + hc * 16384, ell, ch, Sr + 8 * ch);
            tc::ld32(tO + lane_off + 32 * hc, v);
            __half *og = static_cast<__half *>(p.o);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int r = 32 * hc + jj;
                if (r < n) og[((size_t)(c0 + r) * p.Hv + h) * 128 + ell] = __float2half_rn(p.scale * v[jj]);
            }
        }
        tc::fence_async_smem();
        tc::fence_before();
    }

    // ---- final state, then release tensor memory
#pragma unroll
    for (int j = 0; j < 16; ++j)
        *reinterpret_cast<float4 *>(p.fin + srow + 4 * j) = make_float4(Sr[4 * j], Sr[4 * j + 1], Sr[4 * j + 2], Sr[4 * j + 3]);
    ptx::cp_async_wait_all();
    sync_tc();
    if (warp == 0) tc::tmem_dealloc(*tslot, TC_TMEM_COLS);
}

bool al16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

bool chunked_tc_eligible(const Problem &p) {
    const bool rule_ok = p.rule == kLinear || p.rule == kGated || p.rule == kDelta || p.rule == kGatedDelta;
    return rule_ok && p.dk == 128 && p.dv == 128 && p.act_f16 && !((p.flags & kPerKey) && rule_has_decay(p.rule)) &&
           al16(p.q) && al16(p.k) && al16(p.v) && al16(p.fin) && (p.init == nullptr || al16(p.init));
}

cudaError_t launch_chunked_tc(const Problem &p, cudaStream_t stream) {
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(chunked_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chunked_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_done[dev] = 1;
    }
    const unsigned grid = (unsigned)((long long)p.B * p.Hv);
    if (rule_has_retrieval(p.rule))
        chunked_tc_kernel<true><<<grid, TC_THREADS, TC_SMEM, stream>>>(p);
    else
        chunked_tc_kernel<false><<<grid, TC_THREADS, TC_SMEM, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
