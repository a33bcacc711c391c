// gate.cu -- the gate-fusion op ("com.microsoft.LinearAttentionGate",
// Description): decay = decay_scale * softplus(a + dt_bias) and, when asked,
// beta = sigmoid(b).  fp32 arithmetic, one rounding on store.
//
// Elementwise and HBM-bound: each thread handles kVec consecutive elements
// with one vector load/store per operand, grid-stride over the flattened
// [n, heads] tensor; the per-head parameters come from L1/L2.
#include "common.cuh"
#include "launch.h"

namespace gdn {

template <typename T>
struct Vec4;
template <>
struct Vec4<float> {
    using type = float4;
};
template <>
struct Vec4<__half> {
    using type = uint2;  // four halves
};

__device__ __forceinline__ void unpack4(const float4 &v, float *x) {
    x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
}
__device__ __forceinline__ void unpack4(const uint2 &v, float *x) {
    __half2 a = *reinterpret_cast<const __half2 *>(&v.x);
    __half2 b = *reinterpret_cast<const __half2 *>(&v.y);
    float2 fa = __half22float2(a), fb = __half22float2(b);
    x[0] = fa.x, x[1] = fa.y, x[2] = fb.x, x[3] = fb.y;
}
__device__ __forceinline__ float4 pack4f(const float *x) { return make_float4(x[0], x[1], x[2], x[3]); }
__device__ __forceinline__ uint2 pack4h(const float *x) {
    __half2 a = __floats2half2_rn(x[0], x[1]);
    __half2 b = __floats2half2_rn(x[2], x[3]);
    uint2 r;
    r.x = *reinterpret_cast<uint32_t *>(&a);
    r.y = *reinterpret_cast<uint32_t *>(&b);
    return r;
}

template <typename T>
__global__ void __launch_bounds__(256) gate_kernel(int64_t total, int heads, const T *__restrict__ a,
                                                   const float *__restrict__ dt_bias,
                                                   const float *__restrict__ decay_scale,
                                                   const T *__restrict__ b, T *__restrict__ decay_out,
                                                   T *__restrict__ beta_out, int vec_ok) {
    using V = typename Vec4<T>::type;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (vec_ok) {
        // total % 4 == 0 and every pointer 4-element aligned.
        const int64_t nv = total / 4;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
            float x[4], y[4];
            unpack4(reinterpret_cast<const V *>(a)[i], x);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int h = (int)((i * 4 + e) % heads);
                y[e] = decay_scale[h] * softplus_f(x[e] + dt_bias[h]);
            }
            if constexpr (sizeof(T) == 4)
                reinterpret_cast<V *>(decay_out)[i] = pack4f(y);
            else
                reinterpret_cast<V *>(decay_out)[i] = pack4h(y);
            if (beta_out) {
                unpack4(reinterpret_cast<const V *>(b)[i], x);
#pragma unroll
                for (int e = 0; e < 4; ++e) y[e] = sigmoid_f(x[e]);
                if constexpr (sizeof(T) == 4)
                    reinterpret_cast<V *>(beta_out)[i] = pack4f(y);
                else
                    reinterpret_cast<V *>(beta_out)[i] = pack4h(y);
            }
        }
        return;
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int h = (int)(i % heads);
        float x;
        if constexpr (sizeof(T) == 4) x = a[i]; else x = __half2float(a[i]);
        float y = decay_scale[h] * softplus_f(x + dt_bias[h]);
        if constexpr (sizeof(T) == 4) decay_out[i] = y; else decay_out[i] = __float2half_rn(y);
        if (beta_out) {
            if constexpr (sizeof(T) == 4) x = b[i]; else x = __half2float(b[i]);
            y = sigmoid_f(x);
            if constexpr (sizeof(T) == 4) beta_out[i] = y; else beta_out[i] = __float2half_rn(y);
        }
    }
}

cudaError_t launch_gate(const GateLaunch &g, cudaStream_t stream) {
    const int64_t total = g.n * (int64_t)g.heads;
    const size_t esz = g.f16 ? 2 : 4;
    auto al = [&](const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % (4 * esz)) == 0; };
    const int vec_ok = (total % 4 == 0) && al(g.a) && al(g.b) && al(g.decay_out) && al(g.beta_out);
    const int64_t work = vec_ok ? total / 4 : total;
    const int threads = 256;
    int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = 152 * 16;  // a few waves of the 152 SMs; grid-stride beyond
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (g.f16) {
        gate_kernel<__half><<<(unsigned)blocks, threads, 0, stream>>>(
            total, g.heads, (const __half *)g.a, g.dt_bias, g.decay_scale, (const __half *)g.b,
            (__half *)g.decay_out, (__half *)g.beta_out, vec_ok);
    } else {
        gate_kernel<float><<<(unsigned)blocks, threads, 0, stream>>>(
            total, g.heads, (const float *)g.a, g.dt_bias, g.decay_scale, (const float *)g.b,
            (float *)g.decay_out, (float *)g.beta_out, vec_ok);
    }
    return cudaGetLastError();
}

}  // namespace gdn
