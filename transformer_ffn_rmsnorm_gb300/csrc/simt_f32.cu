// simt_f32.cu -- the FFN block in fp32 storage with fp32 FFMA arithmetic.
//
// The fp32 path must land within 1e-4 * rms(y) of the float64 result, which
// rules out TF32 tensor cores (10-bit mantissa, about 5e-4 relative per
// product).  The projections therefore run as shared-memory tiled SIMT
// GEMMs of the form C = A * B^T with both operands K-contiguous, as the
// weights are stored [out x in].  The gate/up GEMM computes the gate and up
// tiles side by side and applies silu(G)*U in its epilogue ("Unfusing a
// Kernel Made It 1.63x Faster", Finding 1: one pass over the activations;
// on this path there is no accumulator budget to trade against).
#include "ffn_internal.cuh"

namespace ffn {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

template <bool GATEUP>
__global__ void __launch_bounds__(256) simt_gemm_nt_kernel(const float *__restrict__ A,
                                                           const float *__restrict__ B0,
                                                           const float *__restrict__ B1,
                                                           float *__restrict__ C, int64_t M,
                                                           int64_t N, int64_t K,
                                                           const float *__restrict__ R) {
    constexpr int NB = GATEUP ? 2 : 1;
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[NB][BK][BN + 4];
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * BN;
    const int lr = tid >> 2, lk = (tid & 3) * 4;
    float acc[NB][4][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[b][i][j] = 0.f;

    for (int64_t k0 = 0; k0 < K; k0 += BK) {
        const bool kok = k0 + lk < K;  // K % 4 == 0, so the float4 is whole
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        if (kok && m0 + lr < M) a = *reinterpret_cast<const float4 *>(A + (m0 + lr) * K + k0 + lk);
        As[lk + 0][lr] = a.x;
        As[lk + 1][lr] = a.y;
        As[lk + 2][lr] = a.z;
        As[lk + 3][lr] = a.w;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float *B = b == 0 ? B0 : B1;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kok && n0 + lr < N) v = *reinterpret_cast<const float4 *>(B + (n0 + lr) * K + k0 + lk);
            Bs[b][lk + 0][lr] = v.x;
            Bs[b][lk + 1][lr] = v.y;
            Bs[b][lk + 2][lr] = v.z;
            Bs[b][lk + 3][lr] = v.w;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float ar[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) ar[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float br[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) br[j] = Bs[b][kk][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[b][i][j] = fmaf(ar[i], br[j], acc[b][i][j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t n = n0 + tx * 4 + j;
            if (n >= N) continue;
            float v = acc[0][i][j];
            if constexpr (GATEUP) v = silu_f32(v) * acc[NB - 1][i][j];
            else if (R) v += R[m * N + n];   // the block's skip connection
            C[m * N + n] = v;
        }
    }
}

}  // namespace

cudaError_t launch_simt_block(const float *x, const float *g, const float *wg, const float *wu,
                              const float *wd, float *y, int64_t rows, int64_t d, int64_t ffn,
                              float eps, float *n, float *h, cudaStream_t s, const float *res) {
    cudaError_t e = launch_rmsnorm(x, g, n, rows, d, eps, DT_F32, s);
    if (e != cudaSuccess) return e;
    {
        dim3 grid(static_cast<unsigned>((rows + BM - 1) / BM), static_cast<unsigned>((ffn + BN - 1) / BN));
        LaunchScope scope(K_SIMT_GATEUP, s);
        simt_gemm_nt_kernel<true><<<grid, 256, 0, s>>>(n, wg, wu, h, rows, ffn, d, nullptr);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        dim3 grid(static_cast<unsigned>((rows + BM - 1) / BM), static_cast<unsigned>((d + BN - 1) / BN));
        LaunchScope scope(K_SIMT_DOWN, s);
        simt_gemm_nt_kernel<false><<<grid, 256, 0, s>>>(h, wd, nullptr, y, rows, d, ffn, res);
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace ffn
