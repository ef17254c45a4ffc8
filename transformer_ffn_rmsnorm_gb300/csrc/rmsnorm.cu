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
                                                          int d, float eps, const float *ss_in) {
    static_assert(sizeof(T) == sizeof(TO), "input and output element sizes must match");
    constexpr int EPV = 16 / sizeof(T);
    __shared__ float partial[256 / 32];
    // launched as a programmatic dependent: nothing is read before the
    // previous kernel has finished; only then may the projection after this
    // one start (it requests weights at once, which that kernel may have written)
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
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
    if (ss_in) ss = ss_in[row];   // the row's sum of squares, handed on by the block before
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
                                                              int64_t d, float eps, const float *ss_in) {
    __shared__ float partial[8];
    // launched as a programmatic dependent: nothing is read before the
    // previous kernel has finished; only then may the projection after this
    // one start (it requests weights at once, which that kernel may have written)
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
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
    if (ss_in) ss = ss_in[row];
    const float inv = rsqrtf(ss / static_cast<float>(d) + eps);
    TO *nr = n + row * d;
    for (int64_t c = threadIdx.x; c < d; c += blockDim.x) {
        const float v = to_f32(xr[c]) * inv * to_f32(g[c]);
        const TO hi = from_f32<TO>(v);
        nr[c] = hi;
        if constexpr (SPLIT) nlo[row * d + c] = from_f32<TO>(v - to_f32(hi));
    }
}

// ---------------------------------------------------------------------------
// Streaming variant for many rows: in a persistent CTA a producer thread
// keeps one shared-memory slot per consumer warp filled with whole rows by
// 1-D bulk copies (cp.async.bulk); each of the eight consumer warps owns one
// slot and normalises its rows on its own (fp32 squares, __shfl_xor_sync, no
// cross-warp barrier), scaling by rsqrt(ms + eps) * g with g staged in shared
// memory once per CTA, and writes 16-byte streaming stores.  Loads stay in
// flight continuously and sixteen rows are in process per SM.  Every mbarrier
// wait is bounded (1 s) and sets the device status word when it gives up.
constexpr int kNormWarps = 8;
constexpr int kNormThreads = 32 * (kNormWarps + 1);
constexpr uint64_t kNormWaitNs = 1000000000ull;

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

template <typename T, typename TO, bool SPLIT>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_stream_kernel(
    const T *x, const T *__restrict__ g, TO *n, TO *nlo, int64_t rows, int d, float eps,
    uint32_t row_bytes, unsigned *err, const float *ss_in) {
    constexpr int EPV = 16 / sizeof(T);
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kNormWarps], bar_empty[kNormWarps], bar_g;
    __shared__ int s_abort, s_never;
    // launched as a programmatic dependent: nothing is read before the
    // previous kernel has finished; only then may the projection after this
    // one start (it requests weights at once, which that kernel may have written)
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t stride = (row_bytes + 127u) & ~127u;
    const uint32_t gsm = (ptx::smem_u32(smem_raw) + 127u) & ~127u;   // g, one row's worth
    const uint32_t ring = gsm + stride;                               // slot w: warp w's rows
    auto full = [&](int s) { return ptx::smem_u32(&bar_full[s]); };
    auto empty = [&](int s) { return ptx::smem_u32(&bar_empty[s]); };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kNormWarps; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&bar_g), 1);
        s_abort = 0;
        s_never = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    volatile int *abort_flag = &s_abort;
    volatile int *never = &s_never;
    int64_t issued = 0;
    const int nvec = d / EPV;

    if (warp == kNormWarps) {
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(ptx::smem_u32(&bar_g), row_bytes);
            ptx::bulk_load(gsm, g, row_bytes, ptx::smem_u32(&bar_g));
            bool ok = true;
            // the i-th row of this CTA goes to slot i % kNormWarps (its k-th use)
            for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, ++issued) {
                const int s = static_cast<int>(issued % kNormWarps);
                const uint32_t ph = static_cast<uint32_t>((issued / kNormWarps) & 1);
                if (!ptx::mbar_wait(empty(s), ph ^ 1u, abort_flag, kNormWaitNs)) {
                    ok = false;
                    break;
                }
                ptx::mbar_arrive_expect_tx(full(s), row_bytes);
                ptx::bulk_load(ring + s * stride, x + r * d, row_bytes, full(s));
            }
            if (!ok) {
                atomicOr(err, DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else {
        const bool gok = ptx::mbar_wait(ptx::smem_u32(&bar_g), 0, abort_flag, kNormWaitNs);
        bool ok = __all_sync(0xffffffffu, gok);
        const uint32_t slot = ring + warp * stride;
        for (int64_t k = 0; ok; ++k) {
            const int64_t i = warp + k * kNormWarps;                      // this CTA's i-th row
            const int64_t r = blockIdx.x + i * gridDim.x;
            if (r >= rows) break;
            const bool got = ptx::mbar_wait(full(warp), static_cast<uint32_t>(k & 1), abort_flag, kNormWaitNs);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            float ss = 0.f;
            if (ss_in) {
                ss = ss_in[r];   // the row's sum of squares, handed on by the block before
            } else {
                for (int v = lane; v < nvec; v += 32) {
                    float f[EPV];
                    Vec16<T>::unpack(lds128(slot + v * 16), f);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) ss = fmaf(f[e], f[e], ss);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            }
            const float inv = rsqrtf(ss / static_cast<float>(d) + eps);
            TO *nr = n + r * d;
            TO *lr = SPLIT ? nlo + r * d : nullptr;
            for (int v = lane; v < nvec; v += 32) {
                float f[EPV], gf[EPV];
                Vec16<T>::unpack(lds128(slot + v * 16), f);
                Vec16<T>::unpack(lds128(gsm + v * 16), gf);
#pragma unroll
                for (int e = 0; e < EPV; ++e) f[e] = f[e] * inv * gf[e];
                const uint4 hv = Vec16<TO>::pack(f);
                __stcs(reinterpret_cast<uint4 *>(nr) + v, hv);
                if constexpr (SPLIT) {
                    float hf[EPV];
                    Vec16<TO>::unpack(hv, hf);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) f[e] -= hf[e];
                    __stcs(reinterpret_cast<uint4 *>(lr) + v, Vec16<TO>::pack(f));
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty(warp));
        }
        if (!ok && lane == 0) {
            atomicOr(err, DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }
    __syncthreads();
    if (warp == kNormWarps && lane == 0) {
        ptx::mbar_wait(ptx::smem_u32(&bar_g), 0, never, kNormWaitNs);
        for (int s = 0; s < kNormWarps; ++s)
            if (issued > s) {
                const int64_t armed = (issued - s + kNormWarps - 1) / kNormWarps;
                ptx::mbar_wait(full(s), static_cast<uint32_t>((armed - 1) & 1), never, kNormWaitNs);
            }
    }
}

// Rows up to 16 KB: g plus one slot per consumer warp fit in ~144 KB.
constexpr uint32_t kNormMaxRowBytes = 16 * 1024;

template <typename T, typename TO, bool SPLIT>
cudaError_t launch_stream(const void *x, const void *g, void *n, void *nlo, int64_t rows, int d, float eps,
                          const float *ss_in, cudaStream_t s) {
    const uint32_t row_bytes = static_cast<uint32_t>(d) * sizeof(T);
    const uint32_t stride = (row_bytes + 127u) & ~127u;
    const size_t smem = static_cast<size_t>(stride) * (kNormWarps + 1) + 128;
    static int configured = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured != dev) {
        e = cudaFuncSetAttribute(rmsnorm_stream_kernel<T, TO, SPLIT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kNormMaxRowBytes * (kNormWarps + 1) + 128));
        if (e != cudaSuccess) return e;
        configured = dev;
    }
    unsigned *err = device_status_word();
    if (!err) return cudaErrorUnknown;
    // as many CTAs as fit, persistent over rows: three per SM at 8 KB rows
    // (24 rows in flight an SM; two per SM measured 47.8 against 46.1 us on
    // 16384 x 4096 fp16, same bits)
    int per_sm = static_cast<int>((227 * 1024) / (smem + 1024));
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 3) per_sm = 3;
    int64_t grid = static_cast<int64_t>(sm_count()) * per_sm;
    if (grid > rows) grid = rows;
    LaunchScope scope(K_RMSNORM, s);
    e = launch_dependent(rmsnorm_stream_kernel<T, TO, SPLIT>, dim3(static_cast<unsigned>(grid)), dim3(kNormThreads),
                         smem, s, static_cast<const T *>(x), static_cast<const T *>(g), static_cast<TO *>(n),
                         static_cast<TO *>(nlo), rows, d, eps, row_bytes, err, ss_in);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, typename TO, int VPT, int WPR, bool SPLIT>
cudaError_t launch_reg(const void *x, const void *g, void *n, void *nlo, int64_t rows, int d,
                       float eps, const float *ss_in, cudaStream_t s) {
    const int threads = 256;
    const int rows_per_cta = (threads / 32) / WPR;
    const int64_t blocks = (rows + rows_per_cta - 1) / rows_per_cta;
    LaunchScope scope(K_RMSNORM, s);
    const cudaError_t e = launch_dependent(rmsnorm_reg_kernel<T, TO, VPT, WPR, SPLIT>,
                                           dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s,
                                           static_cast<const T *>(x), static_cast<const T *>(g),
                                           static_cast<TO *>(n), static_cast<TO *>(nlo), rows, d, eps, ss_in);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T, typename TO, int WPR, bool SPLIT>
cudaError_t dispatch_vpt(int vpt, const void *x, const void *g, void *n, void *nlo, int64_t rows,
                         int d, float eps, const float *ss_in, cudaStream_t s) {
    switch (vpt) {
        case 1: return launch_reg<T, TO, 1, WPR, SPLIT>(x, g, n, nlo, rows, d, eps, ss_in, s);
        case 2: return launch_reg<T, TO, 2, WPR, SPLIT>(x, g, n, nlo, rows, d, eps, ss_in, s);
        case 4: return launch_reg<T, TO, 4, WPR, SPLIT>(x, g, n, nlo, rows, d, eps, ss_in, s);
        default: return launch_reg<T, TO, 8, WPR, SPLIT>(x, g, n, nlo, rows, d, eps, ss_in, s);
    }
}

template <typename T, typename TO, bool SPLIT>
cudaError_t launch_typed(const void *x, const void *g, void *n, void *nlo, int64_t rows,
                         int64_t d, float eps, const float *ss_in, cudaStream_t s) {
    constexpr int EPV = 16 / sizeof(T);
    const bool aligned = (d % EPV) == 0;
    const int64_t nvec = d / EPV;
    // many rows: stream whole rows through shared memory
    if (aligned && rows >= 4 * static_cast<int64_t>(sm_count()) && d * sizeof(T) <= kNormMaxRowBytes)
        return launch_stream<T, TO, SPLIT>(x, g, n, nlo, rows, static_cast<int>(d), eps, ss_in, s);
    // registers hold the row when nvec <= 32 lanes * 8 warps * kMaxVPT
    if (aligned && nvec <= 32 * 8 * kMaxVPT) {
        int wpr = 1;
        while (nvec > static_cast<int64_t>(32) * wpr * kMaxVPT) wpr <<= 1;
        const int64_t per_thread = (nvec + 32 * wpr - 1) / (32 * wpr);
        int vpt = 1;
        while (vpt < per_thread) vpt <<= 1;
        const int di = static_cast<int>(d);
        switch (wpr) {
            case 1: return dispatch_vpt<T, TO, 1, SPLIT>(vpt, x, g, n, nlo, rows, di, eps, ss_in, s);
            case 2: return dispatch_vpt<T, TO, 2, SPLIT>(vpt, x, g, n, nlo, rows, di, eps, ss_in, s);
            case 4: return dispatch_vpt<T, TO, 4, SPLIT>(vpt, x, g, n, nlo, rows, di, eps, ss_in, s);
            default: return dispatch_vpt<T, TO, 8, SPLIT>(vpt, x, g, n, nlo, rows, di, eps, ss_in, s);
        }
    }
    LaunchScope scope(K_RMSNORM, s);
    const cudaError_t e = launch_dependent(rmsnorm_generic_kernel<T, TO, SPLIT>, dim3(static_cast<unsigned>(rows)),
                                           dim3(256), 0, s, static_cast<const T *>(x), static_cast<const T *>(g),
                                           static_cast<TO *>(n), static_cast<TO *>(nlo), rows, d, eps, ss_in);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm(const void *x, const void *g, void *n, int64_t rows, int64_t d,
                           float eps, int dt, cudaStream_t s, const float *ss_in) {
    if (rows <= 0) return cudaSuccess;
    switch (dt) {
        case DT_F32: return launch_typed<float, float, false>(x, g, n, nullptr, rows, d, eps, ss_in, s);
        case DT_F16: return launch_typed<__half, __half, false>(x, g, n, nullptr, rows, d, eps, ss_in, s);
        default:
            return launch_typed<__nv_bfloat16, __nv_bfloat16, false>(x, g, n, nullptr, rows, d, eps, ss_in, s);
    }
}

cudaError_t launch_rmsnorm_split(const void *x, const void *g, void *n_hi, void *n_lo,
                                 int64_t rows, int64_t d, float eps, int dt, cudaStream_t s, const float *ss_in) {
    if (rows <= 0) return cudaSuccess;
    switch (dt) {
        case DT_F16: return launch_typed<__half, __half, true>(x, g, n_hi, n_lo, rows, d, eps, ss_in, s);
        case DT_BF16:
            return launch_typed<__nv_bfloat16, __nv_bfloat16, true>(x, g, n_hi, n_lo, rows, d, eps, ss_in, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_rmsnorm_to_f16(const void *x, const void *g, void *n, int64_t rows, int64_t d,
                                  float eps, int dt_in, cudaStream_t s, const float *ss_in) {
    if (rows <= 0) return cudaSuccess;
    switch (dt_in) {
        case DT_F16: return launch_typed<__half, __half, false>(x, g, n, nullptr, rows, d, eps, ss_in, s);
        case DT_BF16: return launch_typed<__nv_bfloat16, __half, false>(x, g, n, nullptr, rows, d, eps, ss_in, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ffn
