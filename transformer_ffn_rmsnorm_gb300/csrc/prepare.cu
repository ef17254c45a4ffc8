// prepare.cu -- one-time re-encoding of 16-bit weights for fp16 tensor operands.
//
// dst[i] = fp16(src[i] * 2^8).  The power-of-two factor moves the weights'
// usual range into fp16's normal range without changing any value: a bf16
// weight w keeps all 8 of its significant bits when 2^-25 <= |w| < 256, and
// below 2^-25 it rounds by at most 2^-33 absolute.  |w| * 2^8 beyond fp16's
// largest finite value becomes infinite and sets DEVERR_RANGE in the device
// status word.  Tensor-core kernels undo the factor in fp32 (exactly).
#include "ffn_internal.cuh"

namespace ffn {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) prepare_kernel(const T *__restrict__ src, __half *__restrict__ dst,
                                                      int64_t count, unsigned *status) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t nvec = count / 8;
    bool bad = false;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        float f[8];
        Vec16<T>::unpack(__ldcs(reinterpret_cast<const uint4 *>(src) + i), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float v = f[e] * kPreparedScale;
            bad |= isfinite(f[e]) && !isfinite(__half2float(__float2half_rn(v)));
            f[e] = v;
        }
        __stcs(reinterpret_cast<uint4 *>(dst) + i, Vec16<__half>::pack(f));
    }
    for (int64_t i = nvec * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
         i += stride) {
        const float w = to_f32(src[i]);
        const __half h = __float2half_rn(w * kPreparedScale);
        bad |= isfinite(w) && !isfinite(__half2float(h));
        dst[i] = h;
    }
    if (bad) atomicOr(status, DEVERR_RANGE);
}

}  // namespace

cudaError_t launch_prepare_weights(const void *src, void *dst, int64_t count, int dt, cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    unsigned *status = device_status_word();
    if (!status) return cudaErrorUnknown;
    const int threads = 256;
    int64_t blocks = static_cast<int64_t>(sm_count()) * 8;
    const int64_t need = (count / 8 + threads - 1) / threads;
    if (blocks > need) blocks = need < 1 ? 1 : need;
    LaunchScope scope(K_PREPARE, s);
    if (dt == DT_BF16)
        prepare_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), threads, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(src), static_cast<__half *>(dst), count, status);
    else
        prepare_kernel<__half><<<static_cast<unsigned>(blocks), threads, 0, s>>>(
            static_cast<const __half *>(src), static_cast<__half *>(dst), count, status);
    return cudaGetLastError();
}

}  // namespace ffn
