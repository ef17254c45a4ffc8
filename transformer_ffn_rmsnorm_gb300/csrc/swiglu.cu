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

}  // namespace

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
