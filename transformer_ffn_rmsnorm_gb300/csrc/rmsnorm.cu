// rmsnorm.cu -- n[r,c] = x[r,c] * rsqrt(mean_c(x[r,c]^2) + eps) * g[c]
//
// "When to hand-write a GPU kernel on Apple Silicon", Rung 2 (a reduction
// needs threads to share partial sums: per-thread sums of squares, combined,
// then rsqrt(sum/d + eps)) and Rung 4 (wide vector loads and a hardware warp
// reduction, then a small combine of per-warp partials).
//
// GB300 design: the row is read once into registers with 16-byte loads
// (coalesced: for a fixed vector slot, a warp reads 512 contiguous bytes),
// squares are summed in fp32, reduced with __shfl_xor_sync, combined across
// the warps of the row in shared memory, and the scaled row is written from
// the same registers -- one HBM read and one HBM write per element.
#include "ffn_internal.cuh"

namespace ffn {
namespace {

constexpr int kMaxVPT = 8;

// Stores v rounded once; with SPLIT also the residual v - hi rounded once, so
// that hi + lo carries about twice the storage type's significant bits.
template <typename T, int EPV, bool SPLIT>
__device__ __forceinline__ void store_vec(T *hi, T *lo, int64_t i, const float (&f)[EPV]) {
    const uint4 hv = Vec16<T>::pack(f);
    reinterpret_cast<uint4 *>(hi)[i] = hv;
    if constexpr (SPLIT) {
        float hf[EPV], r[EPV];
        Vec16<T>::unpack(hv, hf);
#pragma unroll
        for (int e = 0; e < EPV; ++e) r[e] = f[e] - hf[e];
        reinterpret_cast<uint4 *>(lo)[i] = Vec16<T>::pack(r);
    }
}

// One row per group of WPR warps; each thread holds VPT 16-byte vectors.
// T: storage of x and g; TO: storage of n (same element size).
template <typename T, typename TO, int VPT, int WPR, bool SPLIT>
__global__ void __launch_bounds__(256) rmsnorm_reg_kernel(const T *x,
                                                          const T *__restrict__ g,
                                                          TO *n, TO *nlo, int64_t rows,
                                                          int d, float eps) {
    static_assert(sizeof(T) == sizeof(TO), "input and output element sizes must match");
    constexpr int EPV = 16 / sizeof(T);
    __shared__ float partial[256 / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows_per_cta = (blockDim.x >> 5) / WPR;
    const int row_in_cta = warp / WPR, wr = warp % WPR;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * rows_per_cta + row_in_cta;
    const bool valid = row < rows;
    const int nvec = d / EPV;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (valid ? row : 0) * d);

    uint4 v[VPT];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int vi = (i * WPR + wr) * 32 + lane;
        if (valid && vi < nvec) {
            v[i] = xr[vi];
            float f[EPV];
            Vec16<T>::unpack(v[i], f);
#pragma unroll
            for (int e = 0; e < EPV; ++e) ss = fmaf(f[e], f[e], ss);
        } else {
            v[i] = make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if constexpr (WPR > 1) {
        if (lane == 0) partial[warp] = ss;
        __syncthreads();
        ss = 0.f;
#pragma unroll
        for (int w = 0; w < WPR; ++w) ss += partial[row_in_cta * WPR + w];
    }
    if (!valid) return;
    const float inv = rsqrtf(ss / static_cast<float>(d) + eps);
    const uint4 *gv = reinterpret_cast<const uint4 *>(g);
    TO *nr = n + row * d;
    TO *lr = SPLIT ? nlo + row * d : nullptr;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int vi = (i * WPR + wr) * 32 + lane;
        if (vi < nvec) {
            float f[EPV], gf[EPV];
            Vec16<T>::unpack(v[i], f);
            Vec16<T>::unpack(gv[vi], gf);
#pragma unroll
            for (int e = 0; e < EPV; ++e) f[e] = f[e] * inv * gf[e];
            store_vec<TO, EPV, SPLIT>(nr, lr, vi, f);
        }
    }
}

// Any d (including rows whose length is not a whole number of 16-byte
// vectors): one CTA per row, scalar loads, two passes over the row.
template <typename T, typename TO, bool SPLIT>
__global__ void __launch_bounds__(256) rmsnorm_generic_kernel(const T *x,
                                                              const T *__restrict__ g,
                                                              TO *n, TO *nlo, int64_t rows,
                                                              int64_t d, float eps) {
    __shared__ float partial[8];
    const int64_t row = blockIdx.x;
    if (row >= rows) return;
    const T *xr = x + row * d;
    float ss = 0.f;
    for (int64_t c = threadIdx.x; c < d; c += blockDim.x) {
        const float v = to_f32(xr[c]);
        ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) partial[threadIdx.x >> 5] = ss;
    __syncthreads();
    ss = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) ss += partial[w];
    const float inv = rsqrtf(ss / static_cast<float>(d) + eps);
    TO *nr = n + row * d;
    for (int64_t c = threadIdx.x; c < d; c += blockDim.x) {
        const float v = to_f32(xr[c]) * inv * to_f32(g[c]);
        const TO hi = from_f32<TO>(v);
        nr[c] = hi;
        if constexpr (SPLIT) nlo[row * d + c] = from_f32<TO>(v - to_f32(hi));
    }
}

template <typename T, typename TO, int VPT, int WPR, bool SPLIT>
cudaError_t launch_reg(const void *x, const void *g, void *n, void *nlo, int64_t rows, int d,
                       float eps, cudaStream_t s) {
    const int threads = 256;
    const int rows_per_cta = (threads / 32) / WPR;
    const int64_t blocks = (rows + rows_per_cta - 1) / rows_per_cta;
    LaunchScope scope(K_RMSNORM, s);
    rmsnorm_reg_kernel<T, TO, VPT, WPR, SPLIT><<<static_cast<unsigned>(blocks), threads, 0, s>>>(
        static_cast<const T *>(x), static_cast<const T *>(g), static_cast<TO *>(n),
        static_cast<TO *>(nlo), rows, d, eps);
    return cudaGetLastError();
}

template <typename T, typename TO, int WPR, bool SPLIT>
cudaError_t dispatch_vpt(int vpt, const void *x, const void *g, void *n, void *nlo, int64_t rows,
                         int d, float eps, cudaStream_t s) {
    switch (vpt) {
        case 1: return launch_reg<T, TO, 1, WPR, SPLIT>(x, g, n, nlo, rows, d, eps, s);
        case 2: return launch_reg<T, TO, 2, WPR, SPLIT>(x, g, n, nlo, rows, d, eps, s);
        case 4: return launch_reg<T, TO, 4, WPR, SPLIT>(x, g, n, nlo, rows, d, eps, s);
        default: return launch_reg<T, TO, 8, WPR, SPLIT>(x, g, n, nlo, rows, d, eps, s);
    }
}

template <typename T, typename TO, bool SPLIT>
cudaError_t launch_typed(const void *x, const void *g, void *n, void *nlo, int64_t rows,
                         int64_t d, float eps, cudaStream_t s) {
    constexpr int EPV = 16 / sizeof(T);
    const bool aligned = (d % EPV) == 0;
    const int64_t nvec = d / EPV;
    // registers hold the row when nvec <= 32 lanes * 8 warps * kMaxVPT
    if (aligned && nvec <= 32 * 8 * kMaxVPT) {
        int wpr = 1;
        while (nvec > static_cast<int64_t>(32) * wpr * kMaxVPT) wpr <<= 1;
        const int64_t per_thread = (nvec + 32 * wpr - 1) / (32 * wpr);
        int vpt = 1;
        while (vpt < per_thread) vpt <<= 1;
        const int di = static_cast<int>(d);
        switch (wpr) {
            case 1: return dispatch_vpt<T, TO, 1, SPLIT>(vpt, x, g, n, nlo, rows, di, eps, s);
            case 2: return dispatch_vpt<T, TO, 2, SPLIT>(vpt, x, g, n, nlo, rows, di, eps, s);
            case 4: return dispatch_vpt<T, TO, 4, SPLIT>(vpt, x, g, n, nlo, rows, di, eps, s);
            default: return dispatch_vpt<T, TO, 8, SPLIT>(vpt, x, g, n, nlo, rows, di, eps, s);
        }
    }
    LaunchScope scope(K_RMSNORM, s);
    rmsnorm_generic_kernel<T, TO, SPLIT><<<static_cast<unsigned>(rows), 256, 0, s>>>(
        static_cast<const T *>(x), static_cast<const T *>(g), static_cast<TO *>(n),
        static_cast<TO *>(nlo), rows, d, eps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm(const void *x, const void *g, void *n, int64_t rows, int64_t d,
                           float eps, int dt, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    switch (dt) {
        case DT_F32: return launch_typed<float, float, false>(x, g, n, nullptr, rows, d, eps, s);
        case DT_F16: return launch_typed<__half, __half, false>(x, g, n, nullptr, rows, d, eps, s);
        default:
            return launch_typed<__nv_bfloat16, __nv_bfloat16, false>(x, g, n, nullptr, rows, d, eps, s);
    }
}

cudaError_t launch_rmsnorm_split(const void *x, const void *g, void *n_hi, void *n_lo,
                                 int64_t rows, int64_t d, float eps, int dt, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    switch (dt) {
        case DT_F16: return launch_typed<__half, __half, true>(x, g, n_hi, n_lo, rows, d, eps, s);
        case DT_BF16:
            return launch_typed<__nv_bfloat16, __nv_bfloat16, true>(x, g, n_hi, n_lo, rows, d, eps, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_rmsnorm_to_f16(const void *x, const void *g, void *n, int64_t rows, int64_t d,
                                  float eps, int dt_in, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    switch (dt_in) {
        case DT_F16: return launch_typed<__half, __half, false>(x, g, n, nullptr, rows, d, eps, s);
        case DT_BF16: return launch_typed<__nv_bfloat16, __half, false>(x, g, n, nullptr, rows, d, eps, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ffn
