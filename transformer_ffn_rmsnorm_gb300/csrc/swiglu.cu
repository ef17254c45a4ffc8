// swiglu.cu -- h[i] = silu(gate[i]) * up[i], the activation in fp32.
//
// "When to hand-write a GPU kernel on Apple Silicon", Rung 1: for
// memory-bound elementwise work the optimum is one pass (read gate and up
// once, write h once), with the activation upcast to fp32.
//
// GB300 design: 16-byte vector loads and stores with streaming cache hints
// (nothing is reused), several vectors in flight per thread, a grid of a
// few CTAs per SM striding over the array; the ragged tail (count not a
// multiple of the vector width) is done by one scalar pass.
#include "ffn_internal.cuh"

namespace ffn {
namespace {

constexpr int kUnroll = 4;

template <typename T>
__global__ void __launch_bounds__(256) swiglu_vec_kernel(const T *gate, const T *up, T *h,
                                                         int64_t nvec) {
    constexpr int EPV = 16 / sizeof(T);
    const uint4 *gv = reinterpret_cast<const uint4 *>(gate);
    const uint4 *uv = reinterpret_cast<const uint4 *>(up);
    uint4 *hv = reinterpret_cast<uint4 *>(h);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < nvec; i += kUnroll * stride) {
        uint4 a[kUnroll], b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            a[u] = __ldcs(gv + i + u * stride);
            b[u] = __ldcs(uv + i + u * stride);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float fg[EPV], fu[EPV];
            Vec16<T>::unpack(a[u], fg);
            Vec16<T>::unpack(b[u], fu);
#pragma unroll
            for (int e = 0; e < EPV; ++e) fg[e] = silu_f32(fg[e]) * fu[e];
            __stcs(hv + i + u * stride, Vec16<T>::pack(fg));
        }
    }
    for (; i < nvec; i += stride) {
        float fg[EPV], fu[EPV];
        Vec16<T>::unpack(__ldcs(gv + i), fg);
        Vec16<T>::unpack(__ldcs(uv + i), fu);
#pragma unroll
        for (int e = 0; e < EPV; ++e) fg[e] = silu_f32(fg[e]) * fu[e];
        __stcs(hv + i, Vec16<T>::pack(fg));
    }
}

template <typename T>
__global__ void swiglu_tail_kernel(const T *gate, const T *up, T *h, int64_t begin,
                                   int64_t count) {
    const int64_t i = begin + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < count) h[i] = from_f32<T>(silu_f32(to_f32(gate[i])) * to_f32(up[i]));
}

// h = silu(gate) * up with fp32 inputs and 16-bit output (the unfused arm of
// the prefill block keeps G and U in fp32 so h is rounded exactly once).  With
// h_lo, also the residual h - round(h), rounded once.
template <typename T>
__global__ void __launch_bounds__(256) swiglu_f32in_kernel(const float *gate, const float *up, T *h,
                                                           T *h_lo, int64_t count, float out_scale) {
    ptx::griddep_launch_dependents();   // the down projection may start its weight loads
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t nvec = count / 8;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        const float4 *gv = reinterpret_cast<const float4 *>(gate) + 2 * i;
        const float4 *uv = reinterpret_cast<const float4 *>(up) + 2 * i;
        const float4 g0 = __ldcs(gv), g1 = __ldcs(gv + 1), u0 = __ldcs(uv), u1 = __ldcs(uv + 1);
        float f[8] = {silu_f32(g0.x) * u0.x, silu_f32(g0.y) * u0.y, silu_f32(g0.z) * u0.z,
                      silu_f32(g0.w) * u0.w, silu_f32(g1.x) * u1.x, silu_f32(g1.y) * u1.y,
                      silu_f32(g1.z) * u1.z, silu_f32(g1.w) * u1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] *= out_scale;
        const uint4 hv = Vec16<T>::pack(f);
        __stcs(reinterpret_cast<uint4 *>(h) + i, hv);
        if (h_lo) {
            float hf[8];
            Vec16<T>::unpack(hv, hf);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] -= hf[e];
            __stcs(reinterpret_cast<uint4 *>(h_lo) + i, Vec16<T>::pack(f));
        }
    }
    for (int64_t i = nvec * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
         i += stride) {
        const float v = silu_f32(gate[i]) * up[i] * out_scale;
        const T hi = from_f32<T>(v);
        h[i] = hi;
        if (h_lo) h_lo[i] = from_f32<T>(v - to_f32(hi));
    }
}

template <typename T>
cudaError_t launch_typed(const void *gate, const void *up, void *h, int64_t count,
                         cudaStream_t s) {
    constexpr int EPV = 16 / sizeof(T);
    const int64_t nvec = count / EPV;
    const T *g = static_cast<const T *>(gate);
    const T *u = static_cast<const T *>(up);
    T *o = static_cast<T *>(h);
    if (nvec > 0) {
        const int threads = 256;
        int64_t blocks = static_cast<int64_t>(sm_count()) * 8;
        const int64_t need = (nvec + threads - 1) / threads;
        if (blocks > need) blocks = need;
        LaunchScope scope(K_SWIGLU, s);
        swiglu_vec_kernel<T><<<static_cast<unsigned>(blocks), threads, 0, s>>>(g, u, o, nvec);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int64_t done = nvec * EPV;
    if (done < count) {
        LaunchScope scope(K_SWIGLU, s);
        swiglu_tail_kernel<T><<<1, 32, 0, s>>>(g, u, o, done, count);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

template <typename T>
cudaError_t launch_f32in(const float *gate, const float *up, void *h, void *h_lo, int64_t count,
                         float out_scale, cudaStream_t s) {
    const int threads = 256;
    int64_t blocks = static_cast<int64_t>(sm_count()) * 8;
    const int64_t need = (count / 8 + threads - 1) / threads;
    if (blocks > need) blocks = need < 1 ? 1 : need;
    LaunchScope scope(K_SWIGLU, s);
    swiglu_f32in_kernel<T><<<static_cast<unsigned>(blocks), threads, 0, s>>>(
        gate, up, static_cast<T *>(h), static_cast<T *>(h_lo), count, out_scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_swiglu_f32in(const float *gate, const float *up, void *h, void *h_lo,
                                int64_t count, int dt, float out_scale, cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    return dt == DT_F16 ? launch_f32in<__half>(gate, up, h, h_lo, count, out_scale, s)
                        : launch_f32in<__nv_bfloat16>(gate, up, h, h_lo, count, out_scale, s);
}

cudaError_t launch_swiglu(const void *gate, const void *up, void *h, int64_t count, int dt,
                          cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    switch (dt) {
        case DT_F32: return launch_typed<float>(gate, up, h, count, s);
        case DT_F16: return launch_typed<__half>(gate, up, h, count, s);
        default: return launch_typed<__nv_bfloat16>(gate, up, h, count, s);
    }
}

}  // namespace ffn
