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
#include "ptx.cuh"

namespace gdn {

constexpr int kTB = 8;           // tokens staged per step
constexpr int kFastRows = 32;    // value rows per state slice, fast path
constexpr int kGenericRows = 8;  // value rows per CTA, generic path (one per warp)
constexpr int kThreads = 256;    // compute threads per CTA (both paths)
constexpr int kStages = 4;       // state slices in flight per CTA, fast path

struct Stage {
    float *k, *q, *a, *x, *v, *alpha, *beta, *kq;
    int *hdr;  // pipe kernel: row, t0, t1 of the staged pair
    int dkp, vrows;
};

__device__ __forceinline__ Stage carve(float *smem, int dkp, int vrows) {
    Stage s;
    s.dkp = dkp;
    s.vrows = vrows;
    s.k = smem;
    s.q = s.k + kTB * dkp;
    s.a = s.q + kTB * dkp;
    s.x = s.a + kTB * dkp;
    s.v = s.x + kTB * dkp;
    s.alpha = s.v + kTB * vrows;
    s.beta = s.alpha + kTB;
    s.kq = s.beta + kTB;
    s.hdr = nullptr;
    return s;
}

__host__ __device__ constexpr size_t stage_bytes(int dkp, int vrows) {
    return sizeof(float) * ((size_t)4 * kTB * dkp + (size_t)kTB * vrows + 3 * kTB);
}

// GDN-2 erase gate b of element e = (token, head) * dk + channel: its own
// input (taken as given) or the per-key beta (through the sigmoid if asked).
__device__ __forceinline__ float erase_at(const Problem &p, size_t e) {
    if (p.erase_gate) return p.erase_gate[e];
    const float b = ld_any(p.beta, e, p.beta_f16);
    return (p.flags & kBetaSigmoid) ? sigmoid_f(b) : b;
}

// GDN-2 factor on value entry vi = (token t, head h) * dv + i: the scalar
// beta of the write when the erase gate is its own input, times the write gate.
__device__ __forceinline__ float write_scale(const Problem &p, int t, int h, size_t vi) {
    float f = 1.f;
    if (p.erase_gate) {
        f = ld_any(p.beta, beta_at(p, t, h), p.beta_f16);
        if (p.flags & kBetaSigmoid) f = sigmoid_f(f);
    }
    if (p.write_gate) f *= p.write_gate[vi];
    return f;
}

// Stages tokens [tb, tb + nt) of value head h (key head qh) and the v entries
// of rows [r0, r0 + s.vrows).  Threads [0, nthreads) of the CTA take part.
__device__ void stage_tokens(const Problem &p, const Stage &s, int h, int qh, int tb, int nt,
                             int r0, int tid, int nthreads) {
    const int lane = tid & 31, warp = tid >> 5, nw = nthreads >> 5;
    const bool has_decay = rule_has_decay(p.rule);
    const bool perkey = (p.flags & kPerKey) != 0;
    const bool gdn2 = p.rule == kGdn2;
    const bool beta_scalar = p.rule == kDelta || p.rule == kGatedDelta;
    const bool sig = (p.flags & kBetaSigmoid) != 0;
    const bool vscale = scales_v(p);
    const int rows = s.vrows;
    for (int idx = tid; idx < nt * rows; idx += nthreads) {
        const int tt = idx / rows, r = idx % rows;
        const int i = r0 + r;
        const size_t vi = ((size_t)(tb + tt) * p.Hv + h) * p.dv + i;
        float x = i < p.dv ? ld_any(p.v, vi, p.act_f16) : 0.f;
        if (vscale && i < p.dv) x *= write_scale(p, tb + tt, h, vi);
        s.v[tt * rows + r] = x;
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
                if (gdn2) s.x[tt * s.dkp + c] = erase_at(p, th * p.dk + c) * kv[i];
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
                beta = ld_any(p.beta, beta_at(p, t, h), p.beta_f16);
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
// The same as an explicit shared-space load (the key-major consumers: measured 3 % faster
// there); volatile keeps it in order with the barriers and waits
__device__ __forceinline__ float4 lds_f4(const float *p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(ptx::smem_u32(p)));
    return v;
}

// Applies the staged tokens [0, nt) to one row slice held in registers.
// Lane group cg (8 lanes per row) owns columns 32 j + 4 cg + [0, 4).
template <int NV>
__device__ __forceinline__ void apply_tokens(const Problem &p, const Stage &s, float4 (&S)[NV], int nt,
                                             int tb, int h, int i_row, int vcol, int cg, bool active) {
    const bool perkey = (p.flags & kPerKey) != 0 && rule_has_decay(p.rule);
    const bool retrieval = rule_has_retrieval(p.rule);
    const float *kap = p.rule == kGdn2 ? s.x : s.k;
    const int dk = s.dkp;
    for (int tt = 0; tt < nt; ++tt) {
        const float *kk = s.k + tt * dk + 4 * cg;
        const float *qq = s.q + tt * dk + 4 * cg;
        const float *xx = kap + tt * dk + 4 * cg;
        if (perkey) {
            const float *aa = s.a + tt * dk + 4 * cg;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const float4 a4 = ld_f4(aa + 32 * j);
                S[j].x *= a4.x, S[j].y *= a4.y, S[j].z *= a4.z, S[j].w *= a4.w;
            }
        }
        // independent partial sums (one per float4 lane component) keep the
        // FMA chains short
        float4 uu = make_float4(0.f, 0.f, 0.f, 0.f), ww = uu;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const float4 x4 = ld_f4(xx + 32 * j), q4 = ld_f4(qq + 32 * j);
            uu.x = fmaf(S[j].x, x4.x, uu.x), uu.y = fmaf(S[j].y, x4.y, uu.y);
            uu.z = fmaf(S[j].z, x4.z, uu.z), uu.w = fmaf(S[j].w, x4.w, uu.w);
            ww.x = fmaf(S[j].x, q4.x, ww.x), ww.y = fmaf(S[j].y, q4.y, ww.y);
            ww.z = fmaf(S[j].z, q4.z, ww.z), ww.w = fmaf(S[j].w, q4.w, ww.w);
        }
        float u = (uu.x + uu.y) + (uu.z + uu.w), w = (ww.x + ww.y) + (ww.z + ww.w);
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            u += __shfl_xor_sync(0xffffffffu, u, o);
            w += __shfl_xor_sync(0xffffffffu, w, o);
        }
        const float alpha = perkey ? 1.f : s.alpha[tt];
        const float vi = active ? s.v[tt * s.vrows + vcol] : 0.f;
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
            st_out(p, ((size_t)(tb + tt) * p.Hv + h) * p.dv + i_row, p.scale * fmaf(alpha, w, d * s.kq[tt]));
    }
}

// Applies the staged tokens [0, nt) to R row slices at once (R = 1 or 2): the
// staged key/query loads are shared by the R rows and their reduction chains
// interleave.  A scalar decay is kept as a lazy factor, S = c * S~, so each
// token updates the state with one FMA per element:
//   u = c' (S~ . kappa),  d = beta (v - u),  o = scale (c' (S~ . q) + d (k . q)),
//   S~ += (d / c') k,  c' = c alpha
// (renormalised into S~ when c' < 1e-20, and folded back before returning).
template <int NV, int R>
__device__ __forceinline__ void apply_tokens_multi(const Problem &p, const Stage &s, float4 (&S)[R][NV], int nt,
                                                   int tb, int h, const int (&i_row)[R], const int (&vcol)[R],
                                                   int cg, const bool (&active)[R]) {
    const bool perkey = (p.flags & kPerKey) != 0 && rule_has_decay(p.rule);
    const bool retrieval = rule_has_retrieval(p.rule);
    const float *kap = p.rule == kGdn2 ? s.x : s.k;
    const int dk = s.dkp;
    float c = 1.f;
    const size_t ostride = (size_t)p.Hv * p.dv;
    unsigned char *obase = static_cast<unsigned char *>(p.o) +
                           ((size_t)tb * p.Hv + h) * p.dv * (p.act_f16 ? 2 : 4);
    for (int tt = 0; tt < nt; ++tt) {
        const float *kk = s.k + tt * dk + 4 * cg;
        const float *qq = s.q + tt * dk + 4 * cg;
        const float *xx = kap + tt * dk + 4 * cg;
        if (perkey) {
            const float *aa = s.a + tt * dk + 4 * cg;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const float4 a4 = ld_f4(aa + 32 * j);
#pragma unroll
                for (int r = 0; r < R; ++r)
                    S[r][j].x *= a4.x, S[r][j].y *= a4.y, S[r][j].z *= a4.z, S[r][j].w *= a4.w;
            }
        }
        // packed fp32x2 FMAs (two lanes of a float4 per instruction)
        float2 ua[R], ub[R], wa[R], wb[R];
#pragma unroll
        for (int r = 0; r < R; ++r) ua[r] = ub[r] = wa[r] = wb[r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const float4 x4 = ld_f4(xx + 32 * j), q4 = ld_f4(qq + 32 * j);
            const float2 xlo = make_float2(x4.x, x4.y), xhi = make_float2(x4.z, x4.w);
            const float2 qlo = make_float2(q4.x, q4.y), qhi = make_float2(q4.z, q4.w);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 slo = make_float2(S[r][j].x, S[r][j].y), shi = make_float2(S[r][j].z, S[r][j].w);
                ua[r] = __ffma2_rn(slo, xlo, ua[r]);
                ub[r] = __ffma2_rn(shi, xhi, ub[r]);
                wa[r] = __ffma2_rn(slo, qlo, wa[r]);
                wb[r] = __ffma2_rn(shi, qhi, wb[r]);
            }
        }
        // Butterfly over the 8 lanes of a row group: each exchange halves the set
        // of partial sums a lane carries (4 shuffles for R = 2 instead of 12),
        // leaving u (cg 0-1), w (cg 2-3) of row 0 and u (cg 4-5), w (cg 6-7)
        // of row 1 (R = 2), or u (cg 0-3), w (cg 4-7) (R = 1); u is then
        // broadcast to the whole group and the lane holding w writes o.
        float val;
        if (R == 2) {
            const float u0 = (ua[0].x + ua[0].y) + (ub[0].x + ub[0].y), w0 = (wa[0].x + wa[0].y) + (wb[0].x + wb[0].y);
            const float u1 = (ua[R - 1].x + ua[R - 1].y) + (ub[R - 1].x + ub[R - 1].y);
            const float w1 = (wa[R - 1].x + wa[R - 1].y) + (wb[R - 1].x + wb[R - 1].y);
            const bool hi = (cg & 4) != 0;
            const float ra = __shfl_xor_sync(0xffffffffu, hi ? u0 : u1, 4);
            const float rb = __shfl_xor_sync(0xffffffffu, hi ? w0 : w1, 4);
            const float ka = (hi ? u1 : u0) + ra, kb = (hi ? w1 : w0) + rb;
            const bool b1 = (cg & 2) != 0;
            val = (b1 ? kb : ka) + __shfl_xor_sync(0xffffffffu, b1 ? ka : kb, 2);
        } else {
            const float u0 = (ua[0].x + ua[0].y) + (ub[0].x + ub[0].y), w0 = (wa[0].x + wa[0].y) + (wb[0].x + wb[0].y);
            const bool hi = (cg & 4) != 0;
            val = (hi ? w0 : u0) + __shfl_xor_sync(0xffffffffu, hi ? u0 : w0, 4);
            val += __shfl_xor_sync(0xffffffffu, val, 2);
        }
        val += __shfl_xor_sync(0xffffffffu, val, 1);
        const int gbase = (threadIdx.x & 31) & ~7;
        float u[R];
        u[0] = __shfl_sync(0xffffffffu, val, gbase);
        if (R == 2) u[R - 1] = __shfl_sync(0xffffffffu, val, gbase + 4);
        float cn = c * s.alpha[tt];  // alpha is 1 without scalar decay
        const float bt = s.beta[tt], kq = s.kq[tt];
        float d[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float vi = active[r] ? s.v[tt * s.vrows + vcol[r]] : 0.f;
            d[r] = retrieval ? bt * (vi - cn * u[r]) : vi;
            // the lane that holds this row's w writes its output
            const int wl = R == 2 ? (r == 0 ? 2 : 6) : 4;
            if (cg == wl && active[r]) {
                const float ov = p.scale * fmaf(cn, val, d[r] * kq);
                if (p.act_f16)
                    reinterpret_cast<__half *>(obase)[(size_t)tt * ostride + i_row[r]] = __float2half_rn(ov);
                else
                    reinterpret_cast<float *>(obase)[(size_t)tt * ostride + i_row[r]] = ov;
            }
        }
        if (cn < 1e-20f) {  // fold the factor in before it underflows (uniform across the CTA)
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int j = 0; j < NV; ++j) S[r][j].x *= cn, S[r][j].y *= cn, S[r][j].z *= cn, S[r][j].w *= cn;
            cn = 1.f;
        }
        const float rc = __frcp_rn(cn);
        float e[R];
#pragma unroll
        for (int r = 0; r < R; ++r) e[r] = d[r] * rc;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const float4 k4 = ld_f4(kk + 32 * j);
            const float2 klo = make_float2(k4.x, k4.y), khi = make_float2(k4.z, k4.w);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 ee = make_float2(e[r], e[r]);
                const float2 lo = __ffma2_rn(ee, klo, make_float2(S[r][j].x, S[r][j].y));
                const float2 hi = __ffma2_rn(ee, khi, make_float2(S[r][j].z, S[r][j].w));
                S[r][j] = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
        c = cn;
    }
    if (c != 1.f) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int j = 0; j < NV; ++j) S[r][j].x *= c, S[r][j].y *= c, S[r][j].z *= c, S[r][j].w *= c;
    }
}

// ---------------------------------------------------------------------------
// Fast path: persistent, warp-specialised (dk in {32, 64, 128, 256}).
//
// Work item = one (request, value head) pair, processed as ceil(dv/32) row
// slices of the state.  Three roles share each CTA:
//  * warp 8, the state producer: one lane streams every slice (32 contiguous
//    rows, 32*dk*4 bytes) into a kStages-deep shared-memory ring with bulk
//    async copies (TMA), completing `full[s]`;
//  * warp 9, the token stager: for the NEXT pair it reads the request range
//    and slot, pulls the raw key/query/value rows in with cp.async, then
//    writes the staged fp32 tokens (L2-normalised k and q, q.k, alpha, beta,
//    per-key alpha, GDN-2 kappa) into one of two staging buffers
//    (`tok_full[b]`);
//  * warps 0-7, the consumers: per slice they wait on `full[s]`, copy the
//    slice into registers, release the slot (`empty[s]`), apply the staged
//    tokens and store the new state straight from registers; after the last
//    slice of a pair they release the staging buffer (`tok_empty[b]`).
// Requests longer than kTB tokens are staged by the consumers themselves,
// kTB tokens at a time.  Every wait is bounded; one that runs out ORs
// GDN_DEVERR_TIMEOUT into the error word and the CTA returns.
// ---------------------------------------------------------------------------
struct PipeLayout {
    int dvp;          // staged value rows (dv)
    int stage_floats; // floats per staging buffer
    int raw_bytes;    // cp.async landing area of the stager
    int ring_bytes;
    int stages;       // state slices in flight
    int nbuf;         // staging buffers
    int nstg;         // stager warps (each with its own landing area)
    int total_bytes;
    int xes;          // bytes per element of the GDN-2 erase-gate rows
    bool has_a, has_x, has_w;
};

// Key-major state in the decode kernel: its consumers hold a whole 128 x 128
// tile (each warp 16 columns of all key rows), so one CTA per SM, with twice
// the ring (when the staging area leaves room for it), two stager warps taking
// alternate pairs and three staging buffers, so that one CTA stages pairs as
// fast as the two CTAs per SM of the value-major kernel.
constexpr int kStagesKM = 8;
constexpr int kMaxStagers = 2;
constexpr int kMaxStageBufs = 3;

__host__ __device__ inline PipeLayout pipe_layout(const Problem &p) {
    PipeLayout L;
    const bool km = (p.flags & kKMajor) != 0;
    L.has_a = (p.flags & kPerKey) != 0 && rule_has_decay(p.rule);
    L.has_x = p.rule == kGdn2;
    L.has_w = p.rule == kGdn2 && p.write_gate != nullptr;
    L.xes = p.erase_gate ? 4 : (p.beta_f16 ? 2 : 4);
    L.dvp = (p.dv + 3) & ~3;
    L.stage_floats = kTB * p.dk * (2 + (L.has_a ? 1 : 0) + (L.has_x ? 1 : 0)) + kTB * L.dvp + 3 * kTB + 4;
    const int es = p.act_f16 ? 2 : 4;
    const int des = p.decay_f16 ? 2 : 4;
    L.raw_bytes = kTB * (2 * p.dk * es + p.dv * es + (L.has_a ? p.dk * des : 0) + (L.has_x ? p.dk * L.xes : 0) +
                         (L.has_w ? p.dv * 4 : 0));
    L.raw_bytes = (L.raw_bytes + 15) & ~15;
    L.nbuf = km ? kMaxStageBufs : 2;
    L.nstg = km ? kMaxStagers : 1;
    // a slice is 32 stored rows: value rows of dk floats, or key rows of dv floats (key-major)
    const int slice_bytes = kFastRows * (km ? p.dv : p.dk) * 4;
    auto total = [&](int stages) {
        return stages * slice_bytes + L.nbuf * L.stage_floats * 4 + L.nstg * L.raw_bytes +
               (2 * stages + 2 * L.nbuf) * 8;
    };
    L.stages = km && total(kStagesKM) <= 200 * 1024 ? kStagesKM : kStages;
    L.ring_bytes = L.stages * slice_bytes;
    L.total_bytes = total(L.stages);
    return L;
}

__device__ __forceinline__ Stage carve_pipe(float *base, const Problem &p, const PipeLayout &L) {
    Stage s;
    s.dkp = p.dk;
    s.vrows = L.dvp;
    s.k = base;
    s.q = s.k + kTB * p.dk;
    float *nx = s.q + kTB * p.dk;
    s.a = L.has_a ? nx : nullptr;
    nx += L.has_a ? kTB * p.dk : 0;
    s.x = L.has_x ? nx : nullptr;
    nx += L.has_x ? kTB * p.dk : 0;
    s.v = nx;
    nx += kTB * L.dvp;
    s.alpha = nx;
    s.beta = nx + kTB;
    s.kq = nx + 2 * kTB;
    s.hdr = reinterpret_cast<int *>(s.kq + kTB);
    return s;
}

__device__ __forceinline__ float ld_raw(const unsigned char *base, int idx, int f16) {
    return f16 ? __half2float(reinterpret_cast<const __half *>(base)[idx]) : reinterpret_cast<const float *>(base)[idx];
}

// Per-lane scalars the stager loads together with its copies: lane tt < L
// holds token tt's decay input and beta as loaded (fp16 in the low half, or
// fp32 bits; converted after the copies have landed, so the loads overlap
// them); gs, gb are the head's gate scale and bias.
struct TokScalars {
    uint32_t g, b;
    float gs, gb;
};

__device__ __forceinline__ uint32_t ld_bits(const void *p, size_t i, int f16) {
    return f16 ? (uint32_t) reinterpret_cast<const unsigned short *>(p)[i] : reinterpret_cast<const uint32_t *>(p)[i];
}
__device__ __forceinline__ float bits_to_f(uint32_t x, int f16) {
    return f16 ? __half2float(__ushort_as_half((unsigned short)x)) : __uint_as_float(x);
}

// cp.async of L token rows of row_bytes each (a multiple of 16): row tt comes
// from row first + tt * step of src and lands at dst + tt * row_bytes.
__device__ __forceinline__ void copy_token_rows(unsigned char *dst, const void *src, size_t first, size_t step,
                                                int row_bytes, int L, int lane) {
    const int ch = row_bytes / 16;
    const unsigned char *s0 = static_cast<const unsigned char *>(src) + first * row_bytes;
    const size_t sstep = step * row_bytes;
    for (int tt = 0; tt < L; ++tt, dst += row_bytes, s0 += sstep)
        for (int c = lane; c < ch; c += 32) ptx::cp_async16(dst + 16 * c, s0 + 16 * c, 16);
}

// The stager's copies for one pair with 0 < L <= kTB tokens starting at t0:
// raw key/query/value rows (and per-key decay, erase gate) land in `raw` by
// cp.async; the per-token scalars come back in `ts`.
template <int DK>
__device__ __forceinline__ void issue_pair(const Problem &p, const PipeLayout &Ly, unsigned char *raw, int h, int qh,
                                           int t0, int L, int lane, TokScalars &ts) {
    const int es = p.act_f16 ? 2 : 4;
    const int des = p.decay_f16 ? 2 : 4, bes = Ly.xes;
    unsigned char *rk = raw;
    unsigned char *rq = rk + kTB * DK * es;
    unsigned char *rv = rq + kTB * DK * es;
    unsigned char *ra = rv + kTB * p.dv * es;
    unsigned char *rx = ra + (Ly.has_a ? kTB * DK * des : 0);
    const int kch = DK * es / 16, vch = p.dv * es / 16;
    for (int idx = lane; idx < L * kch; idx += 32) {
        const int tt = idx / kch, c = idx % kch;
        const size_t off = (((size_t)(t0 + tt) * p.Hq + qh) * DK) * es + 16 * c;
        ptx::cp_async16(rk + tt * DK * es + 16 * c, static_cast<const unsigned char *>(p.k) + off, 16);
        ptx::cp_async16(rq + tt * DK * es + 16 * c, static_cast<const unsigned char *>(p.q) + off, 16);
    }
    for (int idx = lane; idx < L * vch; idx += 32) {
        const int tt = idx / vch, c = idx % vch;
        const size_t off = (((size_t)(t0 + tt) * p.Hv + h) * p.dv) * es + 16 * c;
        ptx::cp_async16(rv + tt * p.dv * es + 16 * c, static_cast<const unsigned char *>(p.v) + off, 16);
    }
    if (Ly.has_a) {
        const int ach = DK * des / 16;
        for (int idx = lane; idx < L * ach; idx += 32) {
            const int tt = idx / ach, c = idx % ach;
            const size_t off = (((size_t)(t0 + tt) * p.Hv + h) * DK) * des + 16 * c;
            ptx::cp_async16(ra + tt * DK * des + 16 * c, static_cast<const unsigned char *>(p.decay) + off, 16);
        }
    }
    // the GDN-2 write gate rows (fp32)
    if (Ly.has_w) copy_token_rows(rx + kTB * DK * Ly.xes, p.write_gate, (size_t)t0 * p.Hv + h, p.Hv, p.dv * 4, L, lane);
    if (Ly.has_x) {  // the GDN-2 erase gate: its own input, or the per-key beta
        const unsigned char *xsrc = static_cast<const unsigned char *>(p.erase_gate ? (const void *)p.erase_gate : p.beta);
        const int xch = DK * bes / 16;
        for (int idx = lane; idx < L * xch; idx += 32) {
            const int tt = idx / xch, c = idx % xch;
            const size_t off = (((size_t)(t0 + tt) * p.Hv + h) * DK) * bes + 16 * c;
            ptx::cp_async16(rx + tt * DK * bes + 16 * c, xsrc + off, 16);
        }
    }
    ts.g = ts.b = 0u;
    ts.gs = ts.gb = 0.f;
    if (lane < L) {
        const size_t th = (size_t)(t0 + lane) * p.Hv + h;
        if (rule_has_decay(p.rule) && !Ly.has_a) {
            ts.g = ld_bits(p.decay, th, p.decay_f16);
            if (p.raw_gate) {
                ts.gs = p.gate_scale[h];
                ts.gb = p.gate_bias[h];
            }
        }
        if (beta_is_scalar(p)) ts.b = ld_bits(p.beta, beta_at(p, t0 + lane, h), p.beta_f16);
    }
}

// L2 normalisation and k . q of staged tokens g0 .. g0 + TG - 1 (those below
// L), written as the fp32 rows the consumers read.  The TG tokens' warp
// reductions are interleaved.
// N consecutive raw elements (fp16 or fp32) starting at element e, as floats;
// e * element size is a multiple of N * element size (vector loads).
template <int N>
__device__ __forceinline__ void ld_raw_vec(const unsigned char *base, int e, int f16, float (&x)[N]) {
    if (f16) {
        const __half *hp = reinterpret_cast<const __half *>(base) + e;
        if (N == 8) {
            const uint4 u = *reinterpret_cast<const uint4 *>(hp);
            const __half2 *h2 = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float2 f = __half22float2(h2[i]);
                x[2 * i] = f.x, x[2 * i + 1] = f.y;
            }
        } else if (N == 4) {
            const uint2 u = *reinterpret_cast<const uint2 *>(hp);
            const __half2 *h2 = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float2 f = __half22float2(h2[i]);
                x[2 * i] = f.x, x[2 * i + 1] = f.y;
            }
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) x[i] = __half2float(hp[i]);
        }
    } else {
        const float *fp = reinterpret_cast<const float *>(base) + e;
        if (N % 4 == 0) {
#pragma unroll
            for (int i = 0; i < N; i += 4) {
                const float4 f = *reinterpret_cast<const float4 *>(fp + i);
                x[i] = f.x, x[i + 1] = f.y, x[i + 2] = f.z, x[i + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < N; ++i) x[i] = fp[i];
        }
    }
}

// stores N floats at dst (16-byte aligned when N is a multiple of 4)
template <int N>
__device__ __forceinline__ void st_vec(float *dst, const float (&x)[N]) {
    if (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) dst[i] = x[i];
    }
}

// L2 normalisation and k . q of staged tokens g0 .. g0 + TG - 1 (those below
// L), written as the fp32 rows the consumers read.  Lane l owns the DK / 32
// consecutive channels l * DK / 32 + [0, DK / 32) (vector loads and stores);
// the TG tokens' warp reductions are interleaved.
template <int DK, int TG>
__device__ __forceinline__ void stage_token_group(const Problem &p, const Stage &st, const PipeLayout &Ly,
                                                  const unsigned char *rk, const unsigned char *rq,
                                                  const unsigned char *ra, const unsigned char *rx, int h, int g0,
                                                  int L, int lane) {
    constexpr int EPL = DK / 32;
    const bool sig = (p.flags & kBetaSigmoid) != 0;
    const int c0 = lane * EPL;
    float ssk[TG], ssq[TG], kq[TG];
#pragma unroll
    for (int u = 0; u < TG; ++u) {
        const int tt = g0 + u;
        ssk[u] = ssq[u] = kq[u] = 0.f;
        if (tt < L) {
            float kx[EPL], qx[EPL];
            ld_raw_vec<EPL>(rk, tt * DK + c0, p.act_f16, kx);
            ld_raw_vec<EPL>(rq, tt * DK + c0, p.act_f16, qx);
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                ssk[u] = fmaf(kx[i], kx[i], ssk[u]);
                ssq[u] = fmaf(qx[i], qx[i], ssq[u]);
                kq[u] = fmaf(kx[i], qx[i], kq[u]);
            }
        }
    }
    const bool l2k = (p.flags & kL2k) != 0, l2q = (p.flags & kL2q) != 0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int u = 0; u < TG; ++u) {
            if (l2k) ssk[u] += __shfl_xor_sync(0xffffffffu, ssk[u], off);
            if (l2q) ssq[u] += __shfl_xor_sync(0xffffffffu, ssq[u], off);
            kq[u] += __shfl_xor_sync(0xffffffffu, kq[u], off);
        }
#pragma unroll
    for (int u = 0; u < TG; ++u) {
        const int tt = g0 + u;
        if (tt >= L) break;
        const float ik = l2k ? rsqrtf(ssk[u] + 1e-12f) : 1.f;
        const float iq = l2q ? rsqrtf(ssq[u] + 1e-12f) : 1.f;
        float kn[EPL], qn[EPL];
        ld_raw_vec<EPL>(rk, tt * DK + c0, p.act_f16, kn);
        ld_raw_vec<EPL>(rq, tt * DK + c0, p.act_f16, qn);
#pragma unroll
        for (int i = 0; i < EPL; ++i) kn[i] *= ik, qn[i] *= iq;
        st_vec<EPL>(st.k + tt * DK + c0, kn);
        st_vec<EPL>(st.q + tt * DK + c0, qn);
        if (Ly.has_a) {
            float g[EPL];
            ld_raw_vec<EPL>(ra, tt * DK + c0, p.decay_f16, g);
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                if (p.raw_gate) g[i] = p.gate_scale[h] * softplus_f(g[i] + p.gate_bias[(size_t)h * DK + c0 + i]);
                g[i] = expf(g[i]);
            }
            st_vec<EPL>(st.a + tt * DK + c0, g);
        }
        if (Ly.has_x) {
            float bb[EPL];
            ld_raw_vec<EPL>(rx, tt * DK + c0, p.erase_gate ? 0 : p.beta_f16, bb);
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                if (sig && !p.erase_gate) bb[i] = sigmoid_f(bb[i]);
                bb[i] *= kn[i];
            }
            st_vec<EPL>(st.x + tt * DK + c0, bb);
        }
        if (lane == 0) st.kq[tt] = kq[u] * ik * iq;
    }
}

// The stager's processing of one pair once its copies have landed: L2
// normalisation, k . q, the decay and beta scalars, and the staged fp32
// token rows the consumers read.
template <int DK>
__device__ void finish_pair(const Problem &p, const Stage &st, const PipeLayout &Ly, const unsigned char *raw, int h,
                            int L, int lane, const TokScalars &ts) {
    const int es = p.act_f16 ? 2 : 4;
    const int des = p.decay_f16 ? 2 : 4;
    const bool beta_scalar = p.rule == kDelta || p.rule == kGatedDelta;  // d = beta (v - alpha u)
    const bool vscale = scales_v(p);  // GDN-2: v' = beta w .* v, d = v' - alpha u
    const bool sig = (p.flags & kBetaSigmoid) != 0;
    const unsigned char *rk = raw;
    const unsigned char *rq = rk + kTB * DK * es;
    const unsigned char *rv = rq + kTB * DK * es;
    const unsigned char *ra = rv + kTB * p.dv * es;
    const unsigned char *rx = ra + (Ly.has_a ? kTB * DK * des : 0);
    const unsigned char *rw = rx + (Ly.has_x ? kTB * DK * Ly.xes : 0);
    int g0 = 0;
    for (; g0 + 4 <= L; g0 += 4) stage_token_group<DK, 4>(p, st, Ly, rk, rq, ra, rx, h, g0, L, lane);
    if (L - g0 == 1)
        stage_token_group<DK, 1>(p, st, Ly, rk, rq, ra, rx, h, g0, L, lane);
    else if (L - g0 == 2)
        stage_token_group<DK, 2>(p, st, Ly, rk, rq, ra, rx, h, g0, L, lane);
    else if (L - g0 == 3)
        stage_token_group<DK, 4>(p, st, Ly, rk, rq, ra, rx, h, g0, L, lane);
    // per-token scalars (lane tt holds token tt's)
    float vb = 1.f;  // GDN-2 with its own erase gate: beta scales the value row
    if (lane < L) {
        float alpha = 1.f;
        if (rule_has_decay(p.rule) && !Ly.has_a) {
            const float graw = bits_to_f(ts.g, p.decay_f16);
            const float g = p.raw_gate ? ts.gs * softplus_f(graw + ts.gb) : graw;
            alpha = expf(g);
        }
        const float b0 = bits_to_f(ts.b, p.beta_f16);
        const float bs = sig ? sigmoid_f(b0) : b0;
        st.alpha[lane] = alpha;
        st.beta[lane] = beta_scalar ? bs : 1.f;
        if (p.erase_gate) vb = bs;
    }
    // value rows: 16-byte chunks (dv * element size is a multiple of 16)
    const int vch = p.dv * es / 16;
    if (!vscale) {
        for (int idx = lane; idx < L * vch; idx += 32) {
            const int tt = idx / vch, c = idx % vch;
            const uint4 w = *reinterpret_cast<const uint4 *>(rv + tt * p.dv * es + 16 * c);
            float *dst = st.v + tt * st.vrows;
            if (p.act_f16) {
                const __half2 *hp = reinterpret_cast<const __half2 *>(&w);
                const float2 f0 = __half22float2(hp[0]), f1 = __half22float2(hp[1]);
                const float2 f2 = __half22float2(hp[2]), f3 = __half22float2(hp[3]);
                *reinterpret_cast<float4 *>(dst + 8 * c) = make_float4(f0.x, f0.y, f1.x, f1.y);
                *reinterpret_cast<float4 *>(dst + 8 * c + 4) = make_float4(f2.x, f2.y, f3.x, f3.y);
            } else {
                *reinterpret_cast<uint4 *>(dst + 4 * c) = w;
            }
        }
        return;
    }
    // GDN-2: v' = beta w .* v.  The trip count is the same in every lane so that
    // the shuffle (beta of token tt from lane tt) sees all of them.
    for (int base = 0; base < L * vch; base += 32) {
        const int idx = base + lane;
        const int tt = idx / vch, c = idx % vch;
        const float f = __shfl_sync(0xffffffffu, vb, min(tt, 31));
        if (idx < L * vch) {
            const uint4 w = *reinterpret_cast<const uint4 *>(rv + tt * p.dv * es + 16 * c);
            float *dst = st.v + tt * st.vrows;
            const float *wr = reinterpret_cast<const float *>(rw + tt * p.dv * 4);
            if (p.act_f16) {
                const __half2 *hp = reinterpret_cast<const __half2 *>(&w);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x = __half22float2(hp[e]);
                    const int col = 8 * c + 2 * e;
                    dst[col] = x.x * (Ly.has_w ? f * wr[col] : f);
                    dst[col + 1] = x.y * (Ly.has_w ? f * wr[col + 1] : f);
                }
            } else {
                const float x[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                                    __uint_as_float(w.w)};
#pragma unroll
                for (int e = 0; e < 4; ++e) dst[4 * c + e] = x[e] * (Ly.has_w ? f * wr[4 * c + e] : f);
            }
        }
    }
}

// The consumer side of one (request, head) pair: waits for each state slice in
// the ring, applies the staged tokens R slices at a time and stores the result.
// `j` counts ring uses across the CTA's pairs; it is set to -1 if a wait runs out.
template <int DK, int R>
__device__ __forceinline__ void consume_slices(const Problem &p, const Stage &st, const float *ring, uint64_t *full,
                                               uint64_t *empty, int &j, int slices, int row, int h, int qh, int t0,
                                               int t1, int tid, int lane, int cg, int rloc) {
    constexpr int NV = DK / 32;
    constexpr int kSlice = kFastRows * DK;
    const int L = t1 - t0;
    const bool one_block = L <= kTB;
    for (int sl = 0; sl < slices; sl += R) {
        float4 S[R][NV];
        int i_row[R];
        bool active[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int s = j % kStages;
            if (!ptx::mbar_wait(&full[s], (j / kStages) & 1)) {
                if (p.err && tid == 0) atomicOr(p.err, 2);
                j = -1;
                return;
            }
            ++j;
            i_row[r] = (sl + r) * kFastRows + rloc;
            active[r] = i_row[r] < p.dv;
            const bool have = active[r] && row >= 0 && p.init != nullptr;
            const float *src = ring + s * kSlice + rloc * DK + 4 * cg;
#pragma unroll
            for (int jj = 0; jj < NV; ++jj) S[r][jj] = have ? ld_f4(src + 32 * jj) : make_float4(0.f, 0.f, 0.f, 0.f);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty[s]);
        }
        if (row < 0) continue;
        if (L > 0) {
            for (int tb = t0; tb < t1; tb += kTB) {
                const int nt = min(kTB, t1 - tb);
                if (!one_block) {  // long request: stage kTB tokens at a time ourselves
                    ptx::named_bar_sync(1, kThreads);
                    stage_tokens(p, st, h, qh, tb, nt, 0, tid, kThreads);
                    ptx::named_bar_sync(1, kThreads);
                }
                apply_tokens_multi<NV, R>(p, st, S, nt, tb, h, i_row, i_row, cg, active);
            }
        } else if (p.fin == p.init) {
            continue;  // empty request, in place: nothing changes
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (active[r]) {
                float *dst = p.fin + (((size_t)row * p.Hv + h) * p.dv + i_row[r]) * DK + 4 * cg;
#pragma unroll
                for (int jj = 0; jj < NV; ++jj) __stcs(reinterpret_cast<float4 *>(dst + 32 * jj), S[r][jj]);
            }
    }
}


// ---------------------------------------------------------------------------
// Key-major state ("gatedDeltaUpdate": [rows, Hv, dk, dv]; dk = dv = 128).
// The stored rows are key rows, so a slice is 32 key rows of 128 value
// columns, and the dot products S^T kappa and S^T q of a value column run
// over all four slices.  The consumers hold the whole tile in registers (the
// layout is described at apply_tokens_km).  The scalar decay is kept as a lazy
// factor as in apply_tokens_multi.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 f4_fma(float a, const float4 &x, const float4 &y) {
    return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}
__device__ __forceinline__ float4 f4_add(const float4 &x, const float4 &y) {
    return make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
}
__device__ __forceinline__ float4 f4_scale(float a, const float4 &x) {
    return make_float4(a * x.x, a * x.y, a * x.z, a * x.w);
}

// Key-major consumers.  Warp w holds the state columns 16 w + [0, 16) of
// all 128 key rows, so every sum over key rows stays inside the warp: lane
// (rg = lane / 4, cq = lane % 4) keeps the float4 of columns 16 w + 4 cq of key
// rows 32 s + 4 rg + e (S[s][e]: slice s, e < 4).  The staged key / query
// entries a thread needs are one float4 per slice and vector (the four lanes
// of a row group read the same one), and the sums are the thread's 16 rows and
// then three shuffle levels over the eight row groups.

__device__ __forceinline__ void apply_tokens_km(const Problem &p, const Stage &s, float4 (&S)[4][4], int nt, int tb,
                                                int h, int warp, int lane) {
    constexpr int DK = 128;
    const bool perkey = (p.flags & kPerKey) != 0 && rule_has_decay(p.rule);
    const bool retrieval = rule_has_retrieval(p.rule);
    const float *kap = p.rule == kGdn2 ? s.x : s.k;
    const int rg = lane >> 2, col = 16 * warp + 4 * (lane & 3);
    float c = 1.f;
    for (int tt = 0; tt < nt; ++tt) {
        const int ro = tt * DK + 4 * rg;  // staged entry of key row 4 rg (+ 32 s + e)
        if (perkey) {
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) {
                const float4 a4 = lds_f4(s.a + ro + 32 * sl);
                S[sl][0] = f4_scale(a4.x, S[sl][0]);
                S[sl][1] = f4_scale(a4.y, S[sl][1]);
                S[sl][2] = f4_scale(a4.z, S[sl][2]);
                S[sl][3] = f4_scale(a4.w, S[sl][3]);
            }
        }
        float4 ua = make_float4(0.f, 0.f, 0.f, 0.f), ub = ua, wa = ua, wb = ua;
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
            const float4 x4 = lds_f4(kap + ro + 32 * sl), q4 = lds_f4(s.q + ro + 32 * sl);
            ua = f4_fma(x4.x, S[sl][0], ua), ub = f4_fma(x4.y, S[sl][1], ub);
            ua = f4_fma(x4.z, S[sl][2], ua), ub = f4_fma(x4.w, S[sl][3], ub);
            wa = f4_fma(q4.x, S[sl][0], wa), wb = f4_fma(q4.y, S[sl][1], wb);
            wa = f4_fma(q4.z, S[sl][2], wa), wb = f4_fma(q4.w, S[sl][3], wb);
        }
        float4 U = f4_add(ua, ub), W = f4_add(wa, wb);
        // over the eight row groups: every lane of a column quad ends with the same sums
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            U.x += __shfl_xor_sync(0xffffffffu, U.x, o), U.y += __shfl_xor_sync(0xffffffffu, U.y, o);
            U.z += __shfl_xor_sync(0xffffffffu, U.z, o), U.w += __shfl_xor_sync(0xffffffffu, U.w, o);
            W.x += __shfl_xor_sync(0xffffffffu, W.x, o), W.y += __shfl_xor_sync(0xffffffffu, W.y, o);
            W.z += __shfl_xor_sync(0xffffffffu, W.z, o), W.w += __shfl_xor_sync(0xffffffffu, W.w, o);
        }
        float cn = c * s.alpha[tt];  // alpha is 1 without scalar decay
        const float bt = s.beta[tt], kq = s.kq[tt];
        const float4 v4 = lds_f4(s.v + tt * s.vrows + col);
        float4 d;
        if (retrieval) {
            d.x = bt * (v4.x - cn * U.x), d.y = bt * (v4.y - cn * U.y);
            d.z = bt * (v4.z - cn * U.z), d.w = bt * (v4.w - cn * U.w);
        } else {
            d = v4;
        }
        if (rg == 0) {
            const float4 ov = make_float4(p.scale * fmaf(cn, W.x, d.x * kq), p.scale * fmaf(cn, W.y, d.y * kq),
                                          p.scale * fmaf(cn, W.z, d.z * kq), p.scale * fmaf(cn, W.w, d.w * kq));
            const size_t oi = ((size_t)(tb + tt) * p.Hv + h) * p.dv + col;
            if (p.act_f16) {
                __half2 *o2 = reinterpret_cast<__half2 *>(static_cast<__half *>(p.o) + oi);
                o2[0] = __floats2half2_rn(ov.x, ov.y);
                o2[1] = __floats2half2_rn(ov.z, ov.w);
            } else {
                *reinterpret_cast<float4 *>(static_cast<float *>(p.o) + oi) = ov;
            }
        }
        if (cn < 1e-20f) {  // fold the factor in before it underflows (uniform across the CTA)
#pragma unroll
            for (int sl = 0; sl < 4; ++sl)
#pragma unroll
                for (int e = 0; e < 4; ++e) S[sl][e] = f4_scale(cn, S[sl][e]);
            cn = 1.f;
        }
        const float rc = __frcp_rn(cn);
        const float4 ev = f4_scale(rc, d);
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
            const float4 k4 = lds_f4(s.k + ro + 32 * sl);
            S[sl][0] = f4_fma(k4.x, ev, S[sl][0]);
            S[sl][1] = f4_fma(k4.y, ev, S[sl][1]);
            S[sl][2] = f4_fma(k4.z, ev, S[sl][2]);
            S[sl][3] = f4_fma(k4.w, ev, S[sl][3]);
        }
        c = cn;
    }
    if (c != 1.f) {
#pragma unroll
        for (int sl = 0; sl < 4; ++sl)
#pragma unroll
            for (int e = 0; e < 4; ++e) S[sl][e] = f4_scale(c, S[sl][e]);
    }
}

// The key-major consumer side of one (request, head) pair.  `j` counts ring
// uses (set to -1 if a wait runs out).
__device__ __forceinline__ void consume_tile_km(const Problem &p, const Stage &st, const float *ring, uint64_t *full,
                                                uint64_t *empty, int &j, int row, int h,
                                                int qh, int t0, int t1, int tid, int warp, int lane, int NST) {
    constexpr int kSlice = kFastRows * 128;
    const int rg = lane >> 2, col = 16 * warp + 4 * (lane & 3);
    float4 S[4][4];
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
        const int slot = j % NST;
        if (!ptx::mbar_wait(&full[slot], (j / NST) & 1)) {
            if (p.err && tid == 0) atomicOr(p.err, kErrTimeout);
            j = -1;
            return;
        }
        ++j;
        const bool have = row >= 0 && p.init != nullptr;
        const float *src = ring + slot * kSlice + 4 * rg * 128 + col;
#pragma unroll
        for (int e = 0; e < 4; ++e) S[sl][e] = have ? lds_f4(src + e * 128) : make_float4(0.f, 0.f, 0.f, 0.f);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&empty[slot]);
    }
    if (row < 0) return;
    const int L = t1 - t0;
    if (L > 0) {
        for (int tb = t0; tb < t1; tb += kTB) {
            const int nt = min(kTB, t1 - tb);
            if (L > kTB) {  // long request: stage kTB tokens at a time ourselves
                ptx::named_bar_sync(1, kThreads);
                stage_tokens(p, st, h, qh, tb, nt, 0, tid, kThreads);
                ptx::named_bar_sync(1, kThreads);
            }
            apply_tokens_km(p, st, S, nt, tb, h, warp, lane);
        }
    } else if (p.fin == p.init) {
        return;  // empty request, in place: nothing changes
    }
    float *dst = p.fin + ((size_t)row * p.Hv + h) * 128 * 128 + 4 * rg * 128 + col;
#pragma unroll
    for (int sl = 0; sl < 4; ++sl)
#pragma unroll
        for (int e = 0; e < 4; ++e) __stcs(reinterpret_cast<float4 *>(dst + (32 * sl + e) * 128), S[sl][e]);
}

template <int DK, bool KM>
__global__ void __launch_bounds__(kThreads + 32 + 32 * (KM ? kMaxStagers : 1), KM ? 1 : 2)
    recurrent_pipe_kernel(Problem p, int slices, int pairs) {
    // KM: key-major state (dk = dv = DK = 128); a slice is 32 key rows
    constexpr int NSTG = KM ? kMaxStagers : 1;   // stager warps
    constexpr int NBUF = KM ? kMaxStageBufs : 2; // staging buffers
    constexpr int kSlice = kFastRows * DK;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const PipeLayout Ly = pipe_layout(p);
    const int NST = Ly.stages;
    float *ring = reinterpret_cast<float *>(smem_raw);
    float *stage_base = reinterpret_cast<float *>(smem_raw + Ly.ring_bytes);
    unsigned char *raw0 = smem_raw + Ly.ring_bytes + NBUF * Ly.stage_floats * 4;
    uint64_t *full = reinterpret_cast<uint64_t *>(raw0 + NSTG * Ly.raw_bytes);
    uint64_t *empty = full + NST;
    uint64_t *tok_full = empty + NST;
    uint64_t *tok_empty = tok_full + NBUF;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kCW = kThreads / 32;  // consumer warps
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], kCW);
        }
        for (int s = 0; s < NBUF; ++s) {
            ptx::mbar_init(&tok_full[s], 1);
            ptx::mbar_init(&tok_empty[s], kCW);
        }
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kCW) {  // ---- state producer
        if (lane == 0) {
            int j = 0;
            for (int pair = blockIdx.x; pair < pairs; pair += gridDim.x) {
                const int b = pair / p.Hv, h = pair % p.Hv;
                const int row = p.slots ? p.slots[b] : b;
                const bool valid = row >= 0 && row < p.rows && p.init != nullptr;
                for (int sl = 0; sl < slices; ++sl, ++j) {
                    const int s = j % NST;
                    if (!ptx::mbar_wait(&empty[s], ((j / NST) & 1) ^ 1)) {
                        if (p.err) atomicOr(p.err, 2);
                        return;
                    }
                    const int r0 = sl * kFastRows;
                    // stored rows: value rows of DK floats (or key rows of dv = DK floats)
                    const int nrows = min(kFastRows, (KM ? p.dk : p.dv) - r0);
                    if (valid) {
                        const uint32_t bytes = (uint32_t)nrows * DK * 4u;
                        ptx::mbar_arrive_expect_tx(&full[s], bytes);
                        ptx::bulk_g2s(ring + s * kSlice, p.init + (((size_t)row * p.Hv + h) * p.dv + r0) * DK,
                                      bytes, &full[s]);
                    } else {
                        ptx::mbar_arrive(&full[s]);
                    }
                }
            }
        }
        return;
    }
    if (warp > kCW) {  // ---- token stagers: stager s takes the CTA's pairs k = s, s + NSTG, ...
        const int sid = warp - kCW - 1;
        unsigned char *raw = raw0 + sid * Ly.raw_bytes;
        const int gstep = NSTG * (int)gridDim.x;
        // request range and slot of the next pair are read one pair ahead
        auto header = [&](int pair, int &row, int &t0, int &t1) {
            const int b = pair / p.Hv, h = pair % p.Hv;
            row = state_row(p, b, h == 0 && lane == 0);
            request_range(p, b, t0, t1);
        };
        int nrow = -1, nt0 = 0, nt1 = 0;
        const int first = blockIdx.x + sid * (int)gridDim.x;
        if (first < pairs) header(first, nrow, nt0, nt1);
        int k = sid;
        for (int pair = first; pair < pairs; pair += gstep, k += NSTG) {
            // buffer k % NBUF, used for the (k / NBUF)-th time
            const int buf = k % NBUF;
            const int row = nrow, t0 = nt0, t1 = nt1;
            if (pair + gstep < pairs) header(pair + gstep, nrow, nt0, nt1);
            if (!ptx::mbar_wait(&tok_empty[buf], ((k / NBUF) & 1) ^ 1)) {
                if (p.err && lane == 0) atomicOr(p.err, 2);
                return;
            }
            const Stage st = carve_pipe(stage_base + buf * Ly.stage_floats, p, Ly);
            const int h = pair % p.Hv;
            const int L = t1 - t0;
            if (row >= 0 && L > 0 && L <= kTB) {
                TokScalars ts;
                issue_pair<DK>(p, Ly, raw, h, (int)((long long)h * p.Hq / p.Hv), t0, L, lane, ts);
                // key-major: the next pair's key, query and value rows into L2 while this one
                // lands (measured: helps the one-CTA-per-SM key-major kernel, not the other)
                const int nL = nt1 - nt0;
                if (KM && pair + gstep < pairs && nrow >= 0 && nL > 0 && nL <= kTB && lane < 3 * nL) {
                    const int nh = (pair + gstep) % p.Hv, nqh = (int)((long long)nh * p.Hq / p.Hv);
                    const int tt = lane / 3, which = lane % 3, es = p.act_f16 ? 2 : 4;
                    const unsigned char *src =
                        which == 2 ? static_cast<const unsigned char *>(p.v) + (((size_t)(nt0 + tt) * p.Hv + nh) * p.dv) * es
                                   : static_cast<const unsigned char *>(which ? p.q : p.k) +
                                         (((size_t)(nt0 + tt) * p.Hq + nqh) * DK) * es;
                    const int bytes = (which == 2 ? p.dv : DK) * es;
                    if (bytes % 16 == 0) ptx::prefetch_l2(src, (uint32_t)bytes);
                }
                ptx::cp_async_wait_all();
                __syncwarp();
                finish_pair<DK>(p, st, Ly, raw, h, L, lane, ts);
            }
            if (lane == 0) {
                st.hdr[0] = row;
                st.hdr[1] = t0;
                st.hdr[2] = t1;
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tok_full[buf]);
        }
        return;
    }

    // ---- consumer warps
    const int cg = lane & 7;
    const int rloc = warp * 4 + (lane >> 3);
    int j = 0, k = 0;
    for (int pair = blockIdx.x; pair < pairs; pair += gridDim.x, ++k) {
        const int buf = k % NBUF;
        if (!ptx::mbar_wait(&tok_full[buf], (k / NBUF) & 1)) {
            if (p.err && tid == 0) atomicOr(p.err, 2);
            return;
        }
        const Stage st = carve_pipe(stage_base + buf * Ly.stage_floats, p, Ly);
        const int *hdr = st.hdr;
        const int row = hdr[0], t0 = hdr[1], t1 = hdr[2];
        const int h = pair % p.Hv;
        const int L = t1 - t0;
        const int qh = (int)((long long)h * p.Hq / p.Hv);
        const bool one_block = L <= kTB;
        // R state slices per pass (2 when the slice count is even): the staged
        // key/query loads are shared and the rows' reduction chains interleave
        if (KM)
            consume_tile_km(p, st, ring, full, empty, j, row, h, qh, t0, t1, tid, warp, lane, NST);
        else if ((slices & 1) == 0)
            consume_slices<DK, 2>(p, st, ring, full, empty, j, slices, row, h, qh, t0, t1, tid, lane, cg, rloc);
        else
            consume_slices<DK, 1>(p, st, ring, full, empty, j, slices, row, h, qh, t0, t1, tid, lane, cg, rloc);
        if (j < 0) return;  // a wait ran out
        if (!one_block) ptx::named_bar_sync(1, kThreads);  // every consumer is done with the buffer
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&tok_empty[buf]);
    }
}

// ---------------------------------------------------------------------------
// Long requests (prefill through the token-serial form): one CTA per
// (request, value head, 32-row slice), so a few long sequences still spread
// over many SMs.  The state slice stays in registers for the whole request;
// tokens go through in blocks of kTB: while block b is applied, the raw
// key/query/value (and per-key decay / erase gate) rows of block b+1 are
// already in flight with cp.async, and its scalar gates in registers.
// ---------------------------------------------------------------------------
struct LongLayout {
    int stage_floats, raw_bytes, total_bytes;
    bool has_a, has_x;
};

__host__ __device__ inline LongLayout long_layout(const Problem &p) {
    LongLayout L;
    L.has_a = (p.flags & kPerKey) != 0 && rule_has_decay(p.rule);
    L.has_x = p.rule == kGdn2;
    L.stage_floats = kTB * p.dk * (2 + (L.has_a ? 1 : 0) + (L.has_x ? 1 : 0)) + kTB * kFastRows + 3 * kTB + 4;
    const int es = p.act_f16 ? 2 : 4, des = p.decay_f16 ? 2 : 4, xes = p.erase_gate ? 4 : (p.beta_f16 ? 2 : 4);
    L.raw_bytes = kTB * (2 * p.dk * es + kFastRows * es + (L.has_a ? p.dk * des : 0) + (L.has_x ? p.dk * xes : 0));
    L.raw_bytes = (L.raw_bytes + 15) & ~15;
    L.total_bytes = L.stage_floats * 4 + 2 * L.raw_bytes;
    return L;
}

template <int DK>
__device__ void issue_block_raw(const Problem &p, const LongLayout &Ly, unsigned char *raw, int h, int qh, int r0,
                                int tb, int nt) {
    const int es = p.act_f16 ? 2 : 4, des = p.decay_f16 ? 2 : 4, xes = p.erase_gate ? 4 : (p.beta_f16 ? 2 : 4);
    unsigned char *rk = raw, *rq = rk + kTB * DK * es, *rv = rq + kTB * DK * es;
    unsigned char *ra = rv + kTB * kFastRows * es, *rx = ra + (Ly.has_a ? kTB * DK * des : 0);
    const int kch = DK * es / 16;
    const int vrows = min(kFastRows, p.dv - r0), vch = vrows * es / 16;
    for (int idx = threadIdx.x; idx < nt * kch; idx += blockDim.x) {
        const int tt = idx / kch, c = idx % kch;
        const size_t off = (((size_t)(tb + tt) * p.Hq + qh) * DK) * es + 16 * c;
        ptx::cp_async16(rk + tt * DK * es + 16 * c, static_cast<const unsigned char *>(p.k) + off, 16);
        ptx::cp_async16(rq + tt * DK * es + 16 * c, static_cast<const unsigned char *>(p.q) + off, 16);
    }
    for (int idx = threadIdx.x; idx < nt * vch; idx += blockDim.x) {
        const int tt = idx / vch, c = idx % vch;
        const size_t off = (((size_t)(tb + tt) * p.Hv + h) * p.dv + r0) * es + 16 * c;
        ptx::cp_async16(rv + tt * kFastRows * es + 16 * c, static_cast<const unsigned char *>(p.v) + off, 16);
    }
    if (Ly.has_a) {
        const int ach = DK * des / 16;
        for (int idx = threadIdx.x; idx < nt * ach; idx += blockDim.x) {
            const int tt = idx / ach, c = idx % ach;
            const size_t off = (((size_t)(tb + tt) * p.Hv + h) * DK) * des + 16 * c;
            ptx::cp_async16(ra + tt * DK * des + 16 * c, static_cast<const unsigned char *>(p.decay) + off, 16);
        }
    }
    if (Ly.has_x) {  // the GDN-2 erase gate: its own input, or the per-key beta
        const int xch = DK * xes / 16;
        const unsigned char *xsrc = static_cast<const unsigned char *>(p.erase_gate ? (const void *)p.erase_gate : p.beta);
        for (int idx = threadIdx.x; idx < nt * xch; idx += blockDim.x) {
            const int tt = idx / xch, c = idx % xch;
            const size_t off = (((size_t)(tb + tt) * p.Hv + h) * DK) * xes + 16 * c;
            ptx::cp_async16(rx + tt * DK * xes + 16 * c, xsrc + off, 16);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int DK>
__global__ void __launch_bounds__(kThreads, 2) recurrent_long_kernel(Problem p, int slices) {
    constexpr int NV = DK / 32;
    constexpr int EPL = DK / 32;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const LongLayout Ly = long_layout(p);
    float *stage_mem = reinterpret_cast<float *>(smem_raw);
    unsigned char *raw0 = smem_raw + Ly.stage_floats * 4;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = lane & 7;
    const int sidx = blockIdx.x % slices, bh = blockIdx.x / slices;
    const int h = bh % p.Hv, b = bh / p.Hv;
    const int r0 = sidx * kFastRows;
    const int rloc = warp * 4 + (lane >> 3), i_row = r0 + rloc;
    const bool active = i_row < p.dv;
    const int row = state_row(p, b, h == 0 && sidx == 0 && tid == 0);
    if (row < 0) return;
    int t0, t1;
    request_range(p, b, t0, t1);
    // value-major: row i_row is contiguous; key-major: element (i, c) sits at c * dv + i
    const bool km = (p.flags & kKMajor) != 0;
    const size_t tbase = ((size_t)row * p.Hv + h) * p.dv * DK;
    const size_t soff = tbase + (size_t)i_row * DK + 4 * cg;
    auto load_state = [&](float4(&S)[NV]) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if (!active || !p.init) {
                S[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            } else if (km) {
                const float *b = p.init + tbase + (size_t)(4 * cg + 32 * j) * p.dv + i_row;
                S[j] = make_float4(b[0], b[p.dv], b[2 * p.dv], b[3 * p.dv]);
            } else {
                S[j] = *reinterpret_cast<const float4 *>(p.init + soff + 32 * j);
            }
        }
    };
    auto store_state = [&](const float4(&S)[NV]) {
        if (!active) return;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if (km) {
                float *b = p.fin + tbase + (size_t)(4 * cg + 32 * j) * p.dv + i_row;
                b[0] = S[j].x, b[p.dv] = S[j].y, b[2 * p.dv] = S[j].z, b[3 * p.dv] = S[j].w;
            } else {
                *reinterpret_cast<float4 *>(p.fin + soff + 32 * j) = S[j];
            }
        }
    };
    float4 S[NV];
    load_state(S);
    if (t1 == t0) {
        if (p.fin != p.init) store_state(S);
        return;
    }
    Stage st;
    st.dkp = DK;
    st.vrows = kFastRows;
    st.k = stage_mem;
    st.q = st.k + kTB * DK;
    float *nx = st.q + kTB * DK;
    st.a = Ly.has_a ? nx : nullptr;
    nx += Ly.has_a ? kTB * DK : 0;
    st.x = Ly.has_x ? nx : nullptr;
    nx += Ly.has_x ? kTB * DK : 0;
    st.v = nx;
    nx += kTB * kFastRows;
    st.alpha = nx;
    st.beta = nx + kTB;
    st.kq = nx + 2 * kTB;
    st.hdr = nullptr;

    const int qh = (int)((long long)h * p.Hq / p.Hv);
    const bool has_decay = rule_has_decay(p.rule);
    const bool beta_scalar = p.rule == kDelta || p.rule == kGatedDelta;
    const bool sig = (p.flags & kBetaSigmoid) != 0;
    const int es = p.act_f16 ? 2 : 4, des = p.decay_f16 ? 2 : 4;
    auto prefetch_scalars = [&](int tb, int nt, float &g, float &bb) {
        g = 0.f, bb = 1.f;
        if (tid < nt) {
            const size_t th = (size_t)(tb + tid) * p.Hv + h;
            if (has_decay && !Ly.has_a) g = ld_any(p.decay, th, p.decay_f16);
            if (beta_scalar) bb = ld_any(p.beta, beta_at(p, tb + tid, h), p.beta_f16);
        }
    };
    float sg, sb;
    issue_block_raw<DK>(p, Ly, raw0, h, qh, r0, t0, min(kTB, t1 - t0));
    prefetch_scalars(t0, min(kTB, t1 - t0), sg, sb);
    int blk = 0;
    for (int tb = t0; tb < t1; tb += kTB, ++blk) {
        const int nt = min(kTB, t1 - tb);
        unsigned char *raw = raw0 + (blk & 1) * Ly.raw_bytes;
        ptx::cp_async_wait_all();
        __syncthreads();  // this block's rows landed; the previous block is fully applied
        const float my_g = sg, my_b = sb;
        if (tb + kTB < t1) {
            const int nn = min(kTB, t1 - tb - kTB);
            issue_block_raw<DK>(p, Ly, raw0 + ((blk + 1) & 1) * Ly.raw_bytes, h, qh, r0, tb + kTB, nn);
            prefetch_scalars(tb + kTB, nn, sg, sb);
        }
        // stage: warp w takes token w
        if (warp < nt) {
            const int tt = warp;
            const unsigned char *rk = raw, *rq = rk + kTB * DK * es, *rv = rq + kTB * DK * es;
            const unsigned char *ra = rv + kTB * kFastRows * es, *rx = ra + (Ly.has_a ? kTB * DK * des : 0);
            (void)rv;
            float kv[EPL], qv[EPL];
            float ssk = 0.f, ssq = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int c = lane + 32 * i;
                kv[i] = ld_raw(rk, tt * DK + c, p.act_f16);
                qv[i] = ld_raw(rq, tt * DK + c, p.act_f16);
                ssk += kv[i] * kv[i];
                ssq += qv[i] * qv[i];
            }
            const float ik = (p.flags & kL2k) ? rsqrtf(warp_sum(ssk) + 1e-12f) : 1.f;
            const float iq = (p.flags & kL2q) ? rsqrtf(warp_sum(ssq) + 1e-12f) : 1.f;
            float kq = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                kv[i] *= ik;
                qv[i] *= iq;
                kq += kv[i] * qv[i];
            }
            kq = warp_sum(kq);
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int c = lane + 32 * i;
                st.k[tt * DK + c] = kv[i];
                st.q[tt * DK + c] = qv[i];
                if (Ly.has_a) {
                    float g = ld_raw(ra, tt * DK + c, p.decay_f16);
                    if (p.raw_gate) g = p.gate_scale[h] * softplus_f(g + p.gate_bias[(size_t)h * DK + c]);
                    st.a[tt * DK + c] = expf(g);
                }
                if (Ly.has_x) {
                    float bb = ld_raw(rx, tt * DK + c, p.erase_gate ? 0 : p.beta_f16);
                    if (sig && !p.erase_gate) bb = sigmoid_f(bb);
                    st.x[tt * DK + c] = bb * kv[i];
                }
            }
            if (lane == 0) st.kq[tt] = kq;
        }
        {
            const unsigned char *rv = raw + 2 * kTB * DK * es;
            const int vrows = min(kFastRows, p.dv - r0);
            const bool vscale = scales_v(p);
            for (int idx = tid; idx < nt * kFastRows; idx += kThreads) {
                const int tt = idx / kFastRows, r = idx % kFastRows;
                float x = r < vrows ? ld_raw(rv, tt * kFastRows + r, p.act_f16) : 0.f;
                if (vscale && r < vrows) x *= write_scale(p, tb + tt, h, ((size_t)(tb + tt) * p.Hv + h) * p.dv + r0 + r);
                st.v[tt * kFastRows + r] = x;
            }
        }
        if (tid < nt) {
            float alpha = 1.f;
            if (has_decay && !Ly.has_a) alpha = expf(p.raw_gate ? p.gate_scale[h] * softplus_f(my_g + p.gate_bias[h]) : my_g);
            st.alpha[tid] = alpha;
            st.beta[tid] = beta_scalar ? (sig ? sigmoid_f(my_b) : my_b) : 1.f;
        }
        __syncthreads();
        apply_tokens<NV>(p, st, S, nt, tb, h, i_row, rloc, cg, active);
    }
    store_state(S);
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
    // element (i_row, c) of the state tile: value-major at i_row * dk + c, key-major at c * dv + i_row
    const bool km = (p.flags & kKMajor) != 0;
    const size_t tbase = ((size_t)row * p.Hv + h) * p.dv * p.dk;
    auto sat = [&](int c) { return tbase + (km ? (size_t)c * p.dv + i_row : (size_t)i_row * p.dk + c); };
    float S[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = lane + 32 * i;
        S[i] = (active && p.init && c < p.dk) ? p.init[sat(c)] : 0.f;
    }
    if (t1 == t0) {
        if (active && p.fin != p.init) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = lane + 32 * i;
                if (c < p.dk) p.fin[sat(c)] = S[i];
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
        stage_tokens(p, s, h, qh, tb, nt, r0, threadIdx.x, blockDim.x);
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
            if (c < p.dk) p.fin[sat(c)] = S[i];
        }
    }
}

static bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

template <int DK, bool KM>
static cudaError_t launch_pipe(const Problem &p, cudaStream_t stream) {
    const int slices = ((KM ? p.dk : p.dv) + kFastRows - 1) / kFastRows;
    const int pairs = p.B * p.Hv;
    const size_t smem = (size_t)pipe_layout(p).total_bytes;
    const void *fn = (const void *)recurrent_pipe_kernel<DK, KM>;
    cudaError_t e = smem_attr(fn, 220 * 1024);
    if (e != cudaSuccess) return e;
    int per_sm = 1;
    const int threads = kThreads + 32 + 32 * (KM ? kMaxStagers : 1);
    e = blocks_per_sm(fn, threads, smem, &per_sm);
    if (e != cudaSuccess) return e;
    long long grid = (long long)sm_count() * per_sm;
    if (grid > pairs) grid = pairs;
    recurrent_pipe_kernel<DK, KM><<<(unsigned)grid, threads, smem, stream>>>(p, slices, pairs);
    return cudaGetLastError();
}

template <int DK>
static cudaError_t launch_long(const Problem &p, cudaStream_t stream) {
    const int slices = (p.dv + kFastRows - 1) / kFastRows;
    const long long grid = (long long)p.B * p.Hv * slices;
    const size_t smem = (size_t)long_layout(p).total_bytes;
    cudaError_t e = smem_attr((const void *)recurrent_long_kernel<DK>, 120 * 1024);
    if (e != cudaSuccess) return e;
    recurrent_long_kernel<DK><<<(unsigned)grid, kThreads, smem, stream>>>(p, slices);
    return cudaGetLastError();
}

cudaError_t launch_recurrent(const Problem &p, cudaStream_t stream) {
    const bool fast_dk = p.dk == 32 || p.dk == 64 || p.dk == 128 || p.dk == 256;
    const int es = p.act_f16 ? 2 : 4;
    const bool per_key = (p.flags & kPerKey) != 0 && rule_has_decay(p.rule);
    // the stager's cp.async copies need 16-byte aligned rows
    // the GDN-2 erase-gate rows: the erase-gate input, or the per-key beta
    const void *xrows = p.erase_gate ? (const void *)p.erase_gate : p.beta;
    const bool gates16 = (!per_key || aligned16(p.decay)) && (p.rule != kGdn2 || aligned16(xrows)) &&
                         (p.write_gate == nullptr || aligned16(p.write_gate));
    const bool rows16 = aligned16(p.q) && aligned16(p.k) && aligned16(p.v) && (p.dv * es) % 16 == 0 && gates16;
    const bool km = (p.flags & kKMajor) != 0;
    // key-major state: the decode kernel's consumers hold whole 128 x 128 tiles
    const bool fast = fast_dk && rows16 && aligned16(p.fin) && (p.init == nullptr || aligned16(p.init)) &&
                      pipe_layout(p).total_bytes <= 200 * 1024 && (!km || (p.dk == 128 && p.dv == 128));
    // Requests longer than a few token blocks on average: spread the slices of
    // each (request, head) over their own CTAs instead of one persistent CTA.
    const long long avg_len = p.seq_len ? p.seq_len : (p.B ? (long long)p.T / p.B : 0);
    const bool long_rows = (p.dv * es) % 16 == 0 && aligned16(p.q) && aligned16(p.k) && aligned16(p.v) && gates16;
    if (fast_dk && long_rows && avg_len > 4 * kTB && aligned16(p.fin) && (p.init == nullptr || aligned16(p.init))) {
        switch (p.dk) {
            case 32: return launch_long<32>(p, stream);
            case 64: return launch_long<64>(p, stream);
            case 128: return launch_long<128>(p, stream);
            default: return launch_long<256>(p, stream);
        }
    }
    if (fast && km) return launch_pipe<128, true>(p, stream);
    if (fast) {
        switch (p.dk) {
            case 32: return launch_pipe<32, false>(p, stream);
            case 64: return launch_pipe<64, false>(p, stream);
            case 128: return launch_pipe<128, false>(p, stream);
            default: return launch_pipe<256, false>(p, stream);
        }
    }
    const long long pairs = (long long)p.B * p.Hv;
    const int slices = (p.dv + kGenericRows - 1) / kGenericRows;
    const long long grid = pairs * slices;
    const size_t smem = stage_bytes((p.dk + 3) & ~3, kGenericRows);
    recurrent_generic_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(p, slices);
    return cudaGetLastError();
}

}  // namespace gdn
