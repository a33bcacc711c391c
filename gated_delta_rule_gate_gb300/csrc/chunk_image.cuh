// chunk_image.cuh -- the operand image shared by the tcgen05 chunked-prefill
// kernels (internal to libgdn): its layout and the helpers that write it.
//
// A prepare kernel writes, for every (chunk, value head), the
// state-independent operands of one chunk of the chunk-parallel prefill; the
// chain kernel then reads them chunk by chunk.  Both sides see the same
// 128-byte-swizzled shared-memory layout, so an image moves between global
// and shared memory with plain bulk copies.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace gdn {
namespace img {

constexpr int TC_C = 64;  // tokens per chunk

// ---------------------------------------------------------------------------
// Chunk operand image: the state-independent operands of one (chunk, value
// head), in shared-memory layout (128-byte swizzle; 64 fp16 per 128-byte row;
// 16-byte chunk c of row r stored at chunk position c ^ (r % 8)):
//   EQ  [2 i-blocks][192 rows][64 i] B operand, K-major: rows 0-127 hold E^T
//                                    (row = N index j), rows 128-191 hold Q'
//                                    (row = N index t), so that S E and S Q'^T
//                                    are one N = 192 product over the shared A
//   U   [2 v-blocks][64 t][64 v]     A operand of U^T, M-major (row = K index t)
//   P   [64 r][64 t]                 B operand, K-major (row = N index r)
//   Kt  [2 j-blocks][64 t][64 j]     B operand, N-major (row = K index t)
// (The gated rule keeps e^{G_C}, one float, at the start of the EQ area.)
constexpr int IM_EQ = 0, IM_EQ_BLK = 24576, IM_EQ_Q = 16384;
constexpr int IM_U = 49152, IM_P = 65536, IM_KT = 73728;
constexpr int IM_BYTES = 90112;
// byte offsets of i-block b of E^T and of Q'
__host__ __device__ constexpr int im_e(int b) { return IM_EQ + b * IM_EQ_BLK; }
__host__ __device__ constexpr int im_q(int b) { return IM_EQ + b * IM_EQ_BLK + IM_EQ_Q; }

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


// T = (I + A)^-1 of a unit lower-triangular 64 x 64 system in fp32, by the 256
// worker threads of a prepare kernel (named barrier 3): the 16 x 16 diagonal
// blocks by substitution (four threads per column), then two
// recursive-doubling merges [[T0, 0], [L, T1]], L = -T1 A10 T0.  At holds the
// strictly lower part of A transposed (At[j][r] = A[r][j]); T is written to
// Tf (row-major); Y = Tf + 32, the unused upper-right 32 x 32 block of T, is
// scratch.  Both arrays have row stride kSolveStride floats.  Only entries
// j < r of At are read.  Ends with a barrier of the 256 threads.
constexpr int kSolveThreads = 256;
constexpr int kSolveStride = 68;
__device__ __forceinline__ void solve_unit_lower64(const float *At, float *Tf, int tid) {
    const int lane = tid & 31;
    float *Y = Tf + 32;
    {
        // diagonal blocks: column c of the inverse of block b, rows 4 s .. 4 s + 3 of it,
        // right-looking (once x[j] is final it updates every later row at once)
        const int b = tid >> 6, c = (tid >> 2) & 15, s4 = 4 * (tid & 3);
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = (s4 + e == c) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < 15; ++j) {
            const float xj = __shfl_sync(0xffffffffu, x[j & 3], (lane & ~3) | (j >> 2));
            const float4 a = *reinterpret_cast<const float4 *>(At + (16 * b + j) * kSolveStride + 16 * b + s4);
            x[0] = s4 > j ? fmaf(-a.x, xj, x[0]) : x[0];
            x[1] = s4 + 1 > j ? fmaf(-a.y, xj, x[1]) : x[1];
            x[2] = s4 + 2 > j ? fmaf(-a.z, xj, x[2]) : x[2];
            x[3] = s4 + 3 > j ? fmaf(-a.w, xj, x[3]) : x[3];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) Tf[(16 * b + s4 + e) * kSolveStride + 16 * b + c] = x[e];
        // the strictly upper blocks (0,1) and (2,3) that the 32x32 products read are zero
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int idx = 2 * tid + e, blk = idx >> 8, rr = (idx >> 4) & 15, cc = idx & 15;
            Tf[(32 * blk + rr) * kSolveStride + 32 * blk + 16 + cc] = 0.f;
        }
    }
    ptx::named_bar_sync(3, kSolveThreads);
    {
        // level 1: blocks (1,0) and (3,2): Y = A_{b,b-1} T_{b-1}, then L = -T_b Y
        const int blk = tid >> 7, r = (tid >> 3) & 15, c = 2 * (tid & 7), o0 = 32 * blk;
        float y0 = 0.f, y1 = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float a = At[(o0 + k) * kSolveStride + o0 + 16 + r];
            const float2 tv = *reinterpret_cast<const float2 *>(Tf + (o0 + k) * kSolveStride + o0 + c);
            y0 = fmaf(a, tv.x, y0);
            y1 = fmaf(a, tv.y, y1);
        }
        *reinterpret_cast<float2 *>(Y + (16 * blk + r) * kSolveStride + c) = make_float2(y0, y1);
        ptx::named_bar_sync(3, kSolveThreads);
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float tv = Tf[(o0 + 16 + r) * kSolveStride + o0 + 16 + k];
            const float2 yy = *reinterpret_cast<const float2 *>(Y + (16 * blk + k) * kSolveStride + c);
            l0 = fmaf(tv, yy.x, l0);
            l1 = fmaf(tv, yy.y, l1);
        }
        *reinterpret_cast<float2 *>(Tf + (o0 + 16 + r) * kSolveStride + o0 + c) = make_float2(-l0, -l1);
    }
    ptx::named_bar_sync(3, kSolveThreads);
    {
        // level 2: Y = A_10 T_0 (32 x 32), then L = -T_1 Y; thread = (row, 4 columns).
        // T_0 and T_1 are lower triangular and their upper parts are stored as zeros, so
        // both sums run over every k: the same k in every lane (broadcast loads, no bank
        // conflicts) and no divergent trip counts.
        const int r = tid >> 3, c = 4 * (tid & 7);
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int k = 0; k < 32; ++k) {
            const float a = At[k * kSolveStride + 32 + r];
            const float4 tv = *reinterpret_cast<const float4 *>(Tf + k * kSolveStride + c);
            y.x = fmaf(a, tv.x, y.x), y.y = fmaf(a, tv.y, y.y), y.z = fmaf(a, tv.z, y.z), y.w = fmaf(a, tv.w, y.w);
        }
        *reinterpret_cast<float4 *>(Y + r * kSolveStride + c) = y;
        ptx::named_bar_sync(3, kSolveThreads);
        float4 l = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int k = 0; k < 32; ++k) {
            const float tv = Tf[(32 + r) * kSolveStride + 32 + k];
            const float4 yy = *reinterpret_cast<const float4 *>(Y + k * kSolveStride + c);
            l.x = fmaf(tv, yy.x, l.x), l.y = fmaf(tv, yy.y, l.y), l.z = fmaf(tv, yy.z, l.z), l.w = fmaf(tv, yy.w, l.w);
        }
        *reinterpret_cast<float4 *>(Tf + (32 + r) * kSolveStride + c) = make_float4(-l.x, -l.y, -l.z, -l.w);
    }
    ptx::named_bar_sync(3, kSolveThreads);
}

}  // namespace img

// [T, H, 128] fp16 rows -> a tensor map of boxes of 64 channels x 1 head x
// 64 tokens with the 128-byte swizzle (the key, query and value tiles).
bool make_kqv_map(CUtensorMap *m, const void *base, int heads, int tokens);

// Launches the per-key-decay prepare kernel (chunked_tc_perkey.cu): the
// operand image of every (chunk slot, value head) for the rules with
// per-key-channel decay or the GDN-2 erase gate.
cudaError_t launch_chunk_prepare_perkey(const Problem &p, const CUtensorMap &tk, const CUtensorMap &tq,
                                        const CUtensorMap &tv, const int *offs, const int *slot_req,
                                        unsigned char *img, int cap, cudaStream_t stream);
bool chunk_prepare_perkey_eligible(const Problem &p);

}  // namespace gdn
