// prepare.cu -- one-time re-encoding of weights for fp16 tensor operands.
//
// dst[i] = fp16(w[i] * 2^8), from 16-bit weights, e4m3 codes with row scales,
// or Q4 blocks (the last two turn a quantised model's weights into the
// prepared form the tensor-core GEMMs of ffn_block_forward stream).  The power-of-two factor moves the weights'
// usual range into fp16's normal range without changing any value: a bf16
// weight w keeps all 8 of its significant bits when 2^-25 <= |w| < 256, and
// below 2^-25 it rounds by at most 2^-33 absolute.  |w| * 2^8 beyond fp16's
// largest finite value becomes infinite and sets DEVERR_RANGE in the device
// status word.  Tensor-core kernels undo the factor in fp32 (exactly).
#include "gemv_common.cuh"

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

// e4m3 codes [rows x cols] with a float scale per row: w = e4m3 * scale.
// e4m3 -> fp16 is exact, and e4m3 * scale * 2^8 (4 + 24 significant bits) is
// exact in double, so each output is one correct rounding.  One thread per 16
// codes (cols % 16 == 0).
__global__ void __launch_bounds__(256) prepare_fp8_kernel(const uint8_t *__restrict__ codes,
                                                          const float *__restrict__ scales, __half *__restrict__ dst,
                                                          int64_t rows, int64_t cols, unsigned *status) {
    const int64_t per_row = cols / 16, nvec = rows * per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    bool bad = false;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        const double sc = static_cast<double>(scales[i / per_row]) * static_cast<double>(kPreparedScale);
        const uint4 c = __ldcs(reinterpret_cast<const uint4 *>(codes) + i);
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
        uint32_t out[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t pair = words[q >> 1] >> (16 * (q & 1));
            const uint32_t h2 = gemv::e4m3x2_to_f16x2(pair);
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
            const __half lo = __double2half(static_cast<double>(f.x) * sc), hi = __double2half(static_cast<double>(f.y) * sc);
            bad |= (isfinite(f.x) && !isfinite(__half2float(lo))) || (isfinite(f.y) && !isfinite(__half2float(hi)));
            const __half2 o = __halves2half2(lo, hi);
            out[q] = *reinterpret_cast<const uint32_t *>(&o);
        }
        uint4 *d = reinterpret_cast<uint4 *>(dst) + 2 * i;
        __stcs(d, make_uint4(out[0], out[1], out[2], out[3]));
        __stcs(d + 1, make_uint4(out[4], out[5], out[6], out[7]));
    }
    if (bad) atomicOr(status, DEVERR_RANGE);
}

// Q4 in the device layout (include/ffn.h) [rows x cols]: w = (u - 8) * s.  The
// product (u - 8) * s * 2^8 (4 + 11 significant bits) is exact in fp32, so
// each output is one rounding.  One thread per 64-byte group of four blocks
// (128 weights); byte 16 t + 4 b + e of the group is canonical byte 4 t + e of
// block b, whose low nibble is weight 4 t + e of the block and whose high
// nibble is weight 4 t + e + 16.  A row holds ceil(cols / 128) groups; the
// blocks of a last, partial group past cols are padding and write nothing.
__global__ void __launch_bounds__(256) prepare_q4_kernel(const uint8_t *__restrict__ qs,
                                                         const uint16_t *__restrict__ sc, __half *__restrict__ dst,
                                                         int64_t rows, int64_t cols, unsigned *status) {
    const int64_t per_row = (cols + 127) / 128, ngroups = rows * per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    bool bad = false;
    for (int64_t gi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; gi < ngroups; gi += stride) {
        uint8_t bytes[64];
#pragma unroll
        for (int v = 0; v < 4; ++v)
            *reinterpret_cast<uint4 *>(bytes + 16 * v) = __ldcs(reinterpret_cast<const uint4 *>(qs) + 4 * gi + v);
        const uint2 sraw = *reinterpret_cast<const uint2 *>(sc + 4 * gi);
        const uint16_t sbits[4] = {static_cast<uint16_t>(sraw.x), static_cast<uint16_t>(sraw.x >> 16),
                                   static_cast<uint16_t>(sraw.y), static_cast<uint16_t>(sraw.y >> 16)};
        const int64_t col0 = 128 * (gi % per_row);
        __half *out = dst + (gi / per_row) * cols + col0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            if (col0 + 32 * b >= cols) break;
            const float s = __half2float(__ushort_as_half(sbits[b])) * kPreparedScale;
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                float f[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int jj = j + k, i = jj & 15;
                    const uint8_t byte = bytes[16 * (i >> 2) + 4 * b + (i & 3)];
                    const int u = jj < 16 ? (byte & 15) : (byte >> 4);
                    f[k] = static_cast<float>(u - 8) * s;
                }
                const __half2 o = __floats2half2_rn(f[0], f[1]);
                bad |= isfinite(s) && (!isfinite(__low2float(o)) || !isfinite(__high2float(o)));
                w[j / 2] = *reinterpret_cast<const uint32_t *>(&o);
            }
            uint4 *d = reinterpret_cast<uint4 *>(out + 32 * b);
#pragma unroll
            for (int v = 0; v < 4; ++v) __stcs(d + v, make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]));
        }
    }
    if (bad) atomicOr(status, DEVERR_RANGE);
}

// Q8_0 codes [rows x cols] with fp16 scales per 32: w = q * s.  q * s * 2^8
// (8 + 11 significant bits) is exact in fp32, so each output is one rounding.
// One thread per 16 codes (cols % 32 == 0).
__global__ void __launch_bounds__(256) prepare_q8_kernel(const int8_t *__restrict__ codes,
                                                         const uint16_t *__restrict__ sc, __half *__restrict__ dst,
                                                         int64_t rows, int64_t cols, unsigned *status) {
    const int64_t nvec = rows * (cols / 16);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    bool bad = false;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        // 16 codes of one block: element 16 i is column (16 i) % cols of row (16 i) / cols
        const float s = __half2float(__ushort_as_half(sc[(16 * i) / 32])) * kPreparedScale;
        const uint4 c = __ldcs(reinterpret_cast<const uint4 *>(codes) + i);
        const int8_t *q = reinterpret_cast<const int8_t *>(&c);
        uint32_t out[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const __half2 o = __floats2half2_rn(static_cast<float>(q[2 * k]) * s, static_cast<float>(q[2 * k + 1]) * s);
            bad |= isfinite(s) && (!isfinite(__low2float(o)) || !isfinite(__high2float(o)));
            out[k] = *reinterpret_cast<const uint32_t *>(&o);
        }
        uint4 *d = reinterpret_cast<uint4 *>(dst) + 2 * i;
        __stcs(d, make_uint4(out[0], out[1], out[2], out[3]));
        __stcs(d + 1, make_uint4(out[4], out[5], out[6], out[7]));
    }
    if (bad) atomicOr(status, DEVERR_RANGE);
}

int64_t prepare_grid(int64_t units) {
    int64_t blocks = static_cast<int64_t>(sm_count()) * 8;
    const int64_t need = (units + 255) / 256;
    return blocks > need ? (need < 1 ? 1 : need) : blocks;
}

}  // namespace

cudaError_t launch_prepare_fp8(const uint8_t *codes, const float *scales, void *dst, int64_t rows, int64_t cols,
                               cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    unsigned *status = device_status_word();
    if (!status) return cudaErrorUnknown;
    LaunchScope scope(K_PREPARE, s);
    prepare_fp8_kernel<<<static_cast<unsigned>(prepare_grid(rows * (cols / 16))), 256, 0, s>>>(
        codes, scales, static_cast<__half *>(dst), rows, cols, status);
    return cudaGetLastError();
}

cudaError_t launch_prepare_q4(const uint8_t *qs, const uint16_t *scales, void *dst, int64_t rows, int64_t cols,
                              cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    unsigned *status = device_status_word();
    if (!status) return cudaErrorUnknown;
    LaunchScope scope(K_PREPARE, s);
    prepare_q4_kernel<<<static_cast<unsigned>(prepare_grid(rows * ((cols + 127) / 128))), 256, 0, s>>>(
        qs, scales, static_cast<__half *>(dst), rows, cols, status);
    return cudaGetLastError();
}

cudaError_t launch_prepare_q8(const int8_t *codes, const uint16_t *scales, void *dst, int64_t rows, int64_t cols,
                              cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    unsigned *status = device_status_word();
    if (!status) return cudaErrorUnknown;
    LaunchScope scope(K_PREPARE, s);
    prepare_q8_kernel<<<static_cast<unsigned>(prepare_grid(rows * (cols / 16))), 256, 0, s>>>(
        codes, scales, static_cast<__half *>(dst), rows, cols, status);
    return cudaGetLastError();
}

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
