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
//
// Each CTA stages k-chunks of its A rows and B rows in shared memory with
// cp.async (16-byte copies, zero-filled past M, N and K), two chunks in
// flight, so the next chunk's global loads overlap the current chunk's
// FFMAs.  Two tile shapes:
//   wide  64 x 64 outputs, 4 x 4 per thread, for grids that fill the SMs;
//   small 16 x 32 outputs, 2 x 2 per thread, the CTA's threads split into
//         KG groups that take disjoint k ranges of every chunk and add their
//         sums in group order at the end (deterministic) -- few-row batches
//         (a 64-row block: 88 gate/up and 32 down CTAs instead of 11 and 4)
//         then spread over more SMs and more warps per SM.
// All three kernels of the block are programmatic dependents of the kernel
// before them: weights (inputs of the call) are requested before
// griddepcontrol.wait, activations after it.
#include "ffn_internal.cuh"

namespace ffn {
namespace {

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
    const int n = pred ? 16 : 0;   // 0 source bytes: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int BM_, int BN_, int TM_, int TN_, int KG_, int KC_, bool GATEUP>
struct Simt {
    static constexpr int BM = BM_, BN = BN_, TM = TM_, TN = TN_, KG = KG_, KC = KC_;
    static constexpr int NB = GATEUP ? 2 : 1;
    static constexpr int TX = BN / TN, TY = BM / TM;
    static constexpr int GT = TX * TY;              // threads of one k group
    static constexpr int THREADS = GT * KG;
    static constexpr int KS = KC / KG;              // k values of a chunk per group
    static constexpr int LD = KC + 4;               // padded row (floats): rows 16 bytes apart mod 128
    static constexpr int ROWS = BM + NB * BN;       // staged rows: A, then B (gate rows, up rows)
    static constexpr int STAGE = ROWS * LD;         // floats
    static constexpr size_t SMEM = 2 * STAGE * sizeof(float);
    static constexpr int ACC = TM * TN * NB;
    static_assert(KS % 4 == 0 && BM % TM == 0 && BN % TN == 0, "tile");
    static_assert(KG == 1 || (KG - 1) * GT * ACC <= 2 * STAGE, "group sums fit the staging buffers");
};

// C[m][n] = sum_k A[m][k] B[n][k]; GATEUP: C = silu(A B0^T) * (A B1^T).
// R (optional, plain): added to C (the block's skip connection).
template <typename S, bool GATEUP>
__global__ void __launch_bounds__(S::THREADS) simt_gemm_nt_kernel(const float *__restrict__ A,
                                                                  const float *__restrict__ B0,
                                                                  const float *__restrict__ B1,
                                                                  float *__restrict__ C, int64_t M, int64_t N,
                                                                  int64_t K, const float *__restrict__ R) {
    extern __shared__ __align__(16) float smem[];
    const int tid = threadIdx.x;
    const int kg = tid / S::GT, t = tid % S::GT;
    const int tx = t % S::TX, ty = t / S::TX;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * S::BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * S::BN;
    const int64_t nchunks = (K + S::KC - 1) / S::KC;
    const uint32_t sbase = ptx::smem_u32(smem);

    // rows [r0, r1) of the staged tile of chunk c into buffer b
    auto stage_rows = [&](int64_t c, int b, int r0, int r1) {
        constexpr int V = S::KC / 4;   // 16-byte pieces per row
        const int64_t k0 = c * S::KC;
        for (int i = tid; i < (r1 - r0) * V; i += S::THREADS) {
            const int r = r0 + i / V, v = i % V;
            const int64_t k = k0 + 4 * v;
            const float *src;
            bool ok;
            if (r < S::BM) {
                ok = m0 + r < M && k < K;
                src = A + (ok ? (m0 + r) * K + k : 0);
            } else {
                const int rb = r - S::BM, mat = rb / S::BN, rr = rb % S::BN;
                const float *B = mat ? B1 : B0;
                ok = n0 + rr < N && k < K;
                src = B + (ok ? (n0 + rr) * K + k : 0);
            }
            cp_async16(sbase + static_cast<uint32_t>((b * S::STAGE + r * S::LD + 4 * v) * 4), src, ok);
        }
    };

    // chunk 0: the weight rows before the wait (inputs of the call), the
    // activation rows after it
    stage_rows(0, 0, S::BM, S::ROWS);
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    stage_rows(0, 0, 0, S::BM);
    cp_async_commit();

    float acc[S::NB][S::TM][S::TN];
#pragma unroll
    for (int b = 0; b < S::NB; ++b)
#pragma unroll
        for (int i = 0; i < S::TM; ++i)
#pragma unroll
            for (int j = 0; j < S::TN; ++j) acc[b][i][j] = 0.f;

    for (int64_t c = 0; c < nchunks; ++c) {
        const int buf = static_cast<int>(c & 1);
        if (c + 1 < nchunks) {
            stage_rows(c + 1, buf ^ 1, 0, S::ROWS);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float *As = smem + buf * S::STAGE;
        const float *Bs = As + S::BM * S::LD;
        const int kbeg = kg * S::KS;
#pragma unroll 4
        for (int kk = kbeg; kk < kbeg + S::KS; kk += 4) {
            float4 a[S::TM];
#pragma unroll
            for (int i = 0; i < S::TM; ++i)
                a[i] = *reinterpret_cast<const float4 *>(As + (ty + i * S::TY) * S::LD + kk);
#pragma unroll
            for (int b = 0; b < S::NB; ++b)
#pragma unroll
                for (int j = 0; j < S::TN; ++j) {
                    const float4 w = *reinterpret_cast<const float4 *>(Bs + (b * S::BN + tx + j * S::TX) * S::LD + kk);
#pragma unroll
                    for (int i = 0; i < S::TM; ++i) {
                        float v = acc[b][i][j];
                        v = fmaf(a[i].x, w.x, v);
                        v = fmaf(a[i].y, w.y, v);
                        v = fmaf(a[i].z, w.z, v);
                        v = fmaf(a[i].w, w.w, v);
                        acc[b][i][j] = v;
                    }
                }
        }
        __syncthreads();   // buffer buf is refilled by the next iteration's copies
    }

    if constexpr (S::KG > 1) {
        // the k groups' sums, added in group order by group 0
        float *red = smem;
        if (kg > 0) {
            float *dst = red + ((kg - 1) * S::GT + t) * S::ACC;
#pragma unroll
            for (int b = 0; b < S::NB; ++b)
#pragma unroll
                for (int i = 0; i < S::TM; ++i)
#pragma unroll
                    for (int j = 0; j < S::TN; ++j) dst[(b * S::TM + i) * S::TN + j] = acc[b][i][j];
        }
        __syncthreads();
        if (kg > 0) return;
        for (int q = 0; q < S::KG - 1; ++q) {
            const float *src = red + (q * S::GT + t) * S::ACC;
#pragma unroll
            for (int b = 0; b < S::NB; ++b)
#pragma unroll
                for (int i = 0; i < S::TM; ++i)
#pragma unroll
                    for (int j = 0; j < S::TN; ++j) acc[b][i][j] += src[(b * S::TM + i) * S::TN + j];
        }
    }
#pragma unroll
    for (int i = 0; i < S::TM; ++i) {
        const int64_t m = m0 + ty + i * S::TY;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < S::TN; ++j) {
            const int64_t n = n0 + tx + j * S::TX;
            if (n >= N) continue;
            float v = acc[0][i][j];
            if constexpr (GATEUP) v = silu_f32(v) * acc[S::NB - 1][i][j];
            else if (R) v += R[m * N + n];   // the block's skip connection
            C[m * N + n] = v;
        }
    }
}

template <typename S, bool GATEUP>
cudaError_t launch_simt(const float *A, const float *B0, const float *B1, float *C, int64_t M, int64_t N,
                        int64_t K, const float *R, cudaStream_t s) {
    constexpr auto kern = simt_gemm_nt_kernel<S, GATEUP>;
    static int configured = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(S::SMEM));
        if (e != cudaSuccess) return e;
        configured = dev;
    }
    const dim3 grid(static_cast<unsigned>((M + S::BM - 1) / S::BM), static_cast<unsigned>((N + S::BN - 1) / S::BN));
    e = launch_dependent(kern, grid, dim3(S::THREADS), S::SMEM, s, A, B0, B1, C, M, N, K, R);
    return e != cudaSuccess ? e : cudaGetLastError();
}

using WideGateUp = Simt<64, 64, 4, 4, 1, 32, true>;
using WideDown = Simt<64, 64, 4, 4, 1, 32, false>;
using SmallGateUp = Simt<16, 32, 2, 2, 2, 128, true>;
using SmallDown = Simt<16, 32, 2, 2, 4, 256, false>;

// ss[r] = sum over the row of y[r,c]^2: one CTA a row, a fixed reduction
// tree (the same bits every run).  The fp32 path's rows' sums of squares for
// the next block's RMSNorm: a pass over y after the down projection (on this
// path, whose outputs carry no rounding, the tile epilogues would have to
// combine across CTAs for the same sums).
__global__ void __launch_bounds__(256) row_sumsq_kernel(const float *y, int64_t d, float *ss) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    __shared__ float red[8];
    const float *yr = y + static_cast<int64_t>(blockIdx.x) * d;
    float acc = 0.f;
    for (int64_t c = threadIdx.x; c < d; c += 256) acc = fmaf(yr[c], yr[c], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += red[w];
        ss[blockIdx.x] = t;
    }
}

// The wide tiles once their grid covers every SM; the small ones before.
bool wide_tiles(int64_t M, int64_t N) { return ((M + 63) / 64) * ((N + 63) / 64) >= sm_count(); }

}  // namespace

cudaError_t launch_simt_block(const float *x, const float *g, const float *wg, const float *wu,
                              const float *wd, float *y, int64_t rows, int64_t d, int64_t ffn,
                              float eps, float *n, float *h, cudaStream_t s, const float *res,
                              const float *ss_in, float *ss_out) {
    cudaError_t e = launch_rmsnorm(x, g, n, rows, d, eps, DT_F32, s, ss_in);
    if (e != cudaSuccess) return e;
    {
        LaunchScope scope(K_SIMT_GATEUP, s);
        e = wide_tiles(rows, ffn) ? launch_simt<WideGateUp, true>(n, wg, wu, h, rows, ffn, d, nullptr, s)
                                  : launch_simt<SmallGateUp, true>(n, wg, wu, h, rows, ffn, d, nullptr, s);
        if (e != cudaSuccess) return e;
    }
    {
        LaunchScope scope(K_SIMT_DOWN, s);
        e = wide_tiles(rows, d) ? launch_simt<WideDown, false>(h, wd, nullptr, y, rows, d, ffn, res, s)
                                : launch_simt<SmallDown, false>(h, wd, nullptr, y, rows, d, ffn, res, s);
        if (e != cudaSuccess || !ss_out) return e;
    }
    LaunchScope scope(K_SIMT_DOWN, s);
    e = launch_dependent(row_sumsq_kernel, dim3(static_cast<unsigned>(rows)), dim3(256), 0, s,
                         static_cast<const float *>(y), d, ss_out);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ffn
