// gemm_tcgen05.cu -- the prefill projections on the 5th-generation tensor cores.
//
//   gate/up:  [G | U] = n * [W_gate ; W_up]^T   (n [M x K], W [F x K])
//             fused epilogue:   h = silu(G) * U            -> h [M x F]
//             unfused epilogue: G and U stored in fp32     -> a SwiGLU pass
//   down:     y = h * W_down^T                  (h [M x F], W_down [d x F])
//
// "Unfusing a Kernel Made It 1.63x Faster", Finding 1: on the Apple part the
// fused gate/up kernel lost because its two accumulators cost 64 registers
// per thread and with them occupancy.  On sm_103a the accumulators live in
// tensor memory (TMEM), not registers: one 128 x 256 fp32 accumulator holds
// 128 gate columns and the 128 up columns of the same features side by side
// (the B tile is 128 rows of W_gate stacked on 128 rows of W_up), so the
// fused epilogue costs no extra accumulator space.  Both arms share this
// kernel's main loop, tiles and schedule ("How Megakernels Work", section
// "Packing and geometry in the unfused control"); only the epilogue differs.
//
// Kernel structure (one CTA per SM, persistent over output tiles):
//   warp 0      one thread issues TMA loads of A (128 x 64) and B (256 x 64)
//               bf16/fp16 tiles, 128-byte swizzled, into a 4-stage ring;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators);
//               one thread issues tcgen05.mma (M=128, N=256, K=16) and
//               tcgen05.commit to release ring slots and publish accumulators;
//   warps 2-5   epilogue: tcgen05.ld rows of the finished accumulator, apply
//               the epilogue, store 16-byte vectors, release the accumulator
//               so the next tile's MMAs overlap this tile's epilogue.
// Every mbarrier wait is bounded (1 s of wall time).  A wait that gives up
// sets the device status word, tells the other roles to stop, waits (again
// bounded) for its own TMA loads and MMAs in flight, and frees TMEM.
#include <cudaTypedefs.h>

#include <type_traits>

#include "ffn_internal.cuh"

namespace ffn {
namespace {

constexpr int BM = 128, BK = 64, UMMA_K = 16;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;

// A_TERMS = 2: the A operand is given as two bf16 matrices whose sum is the
// fp32 value (hi + lo); both are multiplied by the same B tile and accumulate
// into the same TMEM accumulator, so A carries ~16 significant bits.
// BN: accumulator columns per tile (256, or 224 for the plain GEMM when it
// evens out the waves); the B tile is BN rows of 64 k values.
template <int A_TERMS, int BN> struct Ring {
    static constexpr uint32_t B_BYTES = BN * BK * 2;
    static constexpr int STAGES = A_TERMS == 1 ? 4 : 3;
    static constexpr uint32_t STAGE_BYTES = A_TERMS * A_BYTES + B_BYTES;
    static constexpr size_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
};
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

enum Mode { MODE_PLAIN = 0, MODE_GATEUP_FUSED = 1, MODE_GATEUP_SPLIT = 2 };

struct GemmParams {
    int64_t M, N, K;          // N: output columns (ffn for gate/up, d for down)
    int64_t num_m_blocks, num_tiles;
    int num_k_blocks;
    void *out0, *out1;        // plain: C; fused: h (and its residual, or null); split: G, U
    int64_t ldo;              // output row stride in elements
    unsigned *err;
    uint64_t wait_limit_ns;
    float acc_scale;          // applied to every accumulator value (exact powers of two)
    float out_scale;          // fused: applied to h before rounding
};

// Stores 32 values rounded once; with `lo` also the rounding residual
// v - round(v), rounded once, so that hi + lo carries ~16 significant bits.
template <typename T>
__device__ __forceinline__ void store_row32(T *dst, T *lo, int64_t col, int64_t ncols,
                                            const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (col + 8 * j < ncols) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = v[8 * j + e];
            const uint4 hv = Vec16<T>::pack(f);
            *reinterpret_cast<uint4 *>(dst + col + 8 * j) = hv;
            if (lo) {
                float hf[8];
                Vec16<T>::unpack(hv, hf);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] -= hf[e];
                *reinterpret_cast<uint4 *>(lo + col + 8 * j) = Vec16<T>::pack(f);
            }
        }
    }
}

__device__ __forceinline__ void store_row32_f32(float *dst, int64_t col, int64_t ncols,
                                               const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (col + 4 * j < ncols)
            *reinterpret_cast<float4 *>(dst + col + 4 * j) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

// BF16: operand type (bf16 or fp16); OUT_BF16: type of the stored output
// (plain mode; the fused h has the operand type, it feeds the next GEMM).
template <int MODE, bool BF16, int A_TERMS, bool OUT_BF16, int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_a2,
                        const __grid_constant__ CUtensorMap map_b0,
                        const __grid_constant__ CUtensorMap map_b1, const GemmParams p) {
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    using TOut = typename std::conditional<OUT_BF16, __nv_bfloat16, __half>::type;
    static_assert(BN % 32 == 0 && BN <= 256 && (MODE == MODE_PLAIN || BN == 256), "tile width");
    constexpr int STAGES = Ring<A_TERMS, BN>::STAGES;
    constexpr uint32_t STAGE_BYTES = Ring<A_TERMS, BN>::STAGE_BYTES;
    constexpr uint32_t B_BYTES = Ring<A_TERMS, BN>::B_BYTES;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[STAGES], bar_empty[STAGES];
    __shared__ __align__(8) uint64_t bar_tfull[2], bar_tempty[2], bar_drain;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort, s_never;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
    // stage s: A term 0 | A term 1 (if any) | B, each 1024-byte aligned
    auto sA = [&](uint32_t s, int t) { return base + s * STAGE_BYTES + t * A_BYTES; };
    auto sB = [&](uint32_t s) { return base + s * STAGE_BYTES + A_TERMS * A_BYTES; };
    auto full = [&](uint32_t s) { return ptx::smem_u32(&bar_full[s]); };
    auto empty = [&](uint32_t s) { return ptx::smem_u32(&bar_empty[s]); };
    auto tfull = [&](uint32_t a) { return ptx::smem_u32(&bar_tfull[a]); };
    auto tempty = [&](uint32_t a) { return ptx::smem_u32(&bar_tempty[a]); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(tfull(a), 1);
            ptx::mbar_init(tempty(a), 4);
        }
        ptx::mbar_init(ptx::smem_u32(&bar_drain), 1);
        s_abort = 0;
        s_never = 0;
        ptx::fence_mbar_init();
        ptx::tma_prefetch_map(&map_a);
        if (A_TERMS == 2) ptx::tma_prefetch_map(&map_a2);
        ptx::tma_prefetch_map(&map_b0);
        if (MODE != MODE_PLAIN) ptx::tma_prefetch_map(&map_b1);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&s_tmem_base), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = s_tmem_base;
    volatile int *abort_flag = &s_abort;
    volatile int *never = &s_never;
    const uint64_t limit = p.wait_limit_ns;
    uint64_t produced = 0;   // k-blocks whose TMA loads were issued (producer thread)

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ TMA producer
        bool ok = true;
        for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
            const int m0 = static_cast<int>((t % p.num_m_blocks) * BM);
            const int64_t n_blk = t / p.num_m_blocks;
            for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                const uint32_t s = static_cast<uint32_t>(produced % STAGES);
                const uint32_t ph = static_cast<uint32_t>((produced / STAGES) & 1);
                if (!ptx::mbar_wait(empty(s), ph ^ 1u, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                ptx::mbar_arrive_expect_tx(full(s), STAGE_BYTES);
                const int k0 = kb * BK;
                ptx::tma_load_2d(sA(s, 0), &map_a, full(s), k0, m0);
                if (A_TERMS == 2) ptx::tma_load_2d(sA(s, 1), &map_a2, full(s), k0, m0);
                if (MODE == MODE_PLAIN) {
                    ptx::tma_load_2d(sB(s), &map_b0, full(s), k0, static_cast<int>(n_blk * BN));
                } else {
                    const int f0 = static_cast<int>(n_blk * (BN / 2));
                    ptx::tma_load_2d(sB(s), &map_b0, full(s), k0, f0);
                    ptx::tma_load_2d(sB(s) + B_BYTES / 2, &map_b1, full(s), k0, f0);
                }
                ++produced;
            }
        }
        if (!ok) {
            atomicOr(p.err, DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp == 1 && lane == 0) {
        // -------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = ptx::idesc_f16(BM, BN, BF16);
        bool ok = true;
        uint64_t consumed = 0;
        uint32_t acc = 0, acc_ph = 0;
        for (int64_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
            if (!ptx::mbar_wait(tempty(acc), acc_ph ^ 1u, abort_flag, limit)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                const uint32_t s = static_cast<uint32_t>(consumed % STAGES);
                const uint32_t ph = static_cast<uint32_t>((consumed / STAGES) & 1);
                if (!ptx::mbar_wait(full(s), ph, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t b0 = sB(s);
#pragma unroll
                for (int t = 0; t < A_TERMS; ++t) {
                    const uint32_t a0 = sA(s, t);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        ptx::tc_mma_f16(d_tmem, ptx::sdesc_k_sw128(a0 + k * UMMA_K * 2),
                                        ptx::sdesc_k_sw128(b0 + k * UMMA_K * 2), idesc,
                                        (kb | k | t) != 0 ? 1u : 0u);
                }
                ptx::tc_commit(empty(s));
                ++consumed;
            }
            if (!ok) break;
            ptx::tc_commit(tfull(acc));
            acc ^= 1u;
            if (acc == 0) acc_ph ^= 1u;
        }
        if (!ok) {
            atomicOr(p.err, DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
        // every MMA issued above must finish before TMEM is freed
        ptx::tc_commit(ptx::smem_u32(&bar_drain));
        ptx::mbar_wait(ptx::smem_u32(&bar_drain), 0, never, limit);
    } else if (warp >= 2) {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;   // this warp may read TMEM lanes 32q .. 32q+31
        bool ok = true;
        uint32_t acc = 0, acc_ph = 0;
        T *out0 = static_cast<T *>(p.out0);
        T *out1 = static_cast<T *>(p.out1);
        for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
            const int64_t m_blk = t % p.num_m_blocks, n_blk = t / p.num_m_blocks;
            // every lane waits (each gets its own acquire); the vote keeps the
            // warp converged and in agreement before the warp-wide tcgen05.ld
            const bool got = ptx::mbar_wait(tfull(acc), acc_ph, abort_flag, limit);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const int64_t row = m_blk * BM + q * 32 + lane;
            const bool live = row < p.M;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            if (MODE == MODE_PLAIN) {
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(taddr + c, r);
                    ptx::tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * p.acc_scale;
                    if (live)
                        store_row32<TOut>(static_cast<TOut *>(p.out0) + row * p.ldo, nullptr,
                                          n_blk * BN + c, p.N, v);
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 32) {
                    uint32_t rg[32], ru[32];
                    ptx::tmem_ld_32x32b_x32(taddr + c, rg);
                    ptx::tmem_ld_32x32b_x32(taddr + BN / 2 + c, ru);
                    ptx::tmem_ld_wait();
                    const int64_t col = n_blk * (BN / 2) + c;
                    if (MODE == MODE_GATEUP_FUSED) {
                        float h[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            h[j] = silu_f32(__uint_as_float(rg[j]) * p.acc_scale) *
                                   (__uint_as_float(ru[j]) * p.acc_scale) * p.out_scale;
                        if (live)
                            store_row32<T>(out0 + row * p.ldo, out1 ? out1 + row * p.ldo : nullptr,
                                           col, p.N, h);
                    } else {
                        float g[32], u[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            g[j] = __uint_as_float(rg[j]) * p.acc_scale;
                            u[j] = __uint_as_float(ru[j]) * p.acc_scale;
                        }
                        // G and U stay fp32 so that h is rounded exactly
                        // once, as in the fused arm
                        if (live) {
                            store_row32_f32(static_cast<float *>(p.out0) + row * p.ldo, col, p.N, g);
                            store_row32_f32(static_cast<float *>(p.out1) + row * p.ldo, col, p.N, u);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty(acc));
            acc ^= 1u;
            if (acc == 0) acc_ph ^= 1u;
        }
        if (!ok && lane == 0) {
            atomicOr(p.err, DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    __syncthreads();
    if (warp == 0 && lane == 0) {
        // TMA loads still in flight (only after an abandoned wait) must land
        // before this CTA's shared memory is released.
        for (uint32_t s = 0; s < STAGES; ++s) {
            if (produced > s) {
                const uint64_t armed = (produced - s + STAGES - 1) / STAGES;
                ptx::mbar_wait(full(s), static_cast<uint32_t>((armed - 1) & 1), never, limit);
            }
        }
    }
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

bool encode_tma_2d(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, int64_t inner,
                   int64_t rows, int64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// A row-major [rows x inner] 16-bit matrix, boxes of 64 x box_rows, 128B swizzle.
bool make_map(CUtensorMap *m, const void *ptr, bool bf16, int64_t inner, int64_t rows,
              uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                     const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int MODE, bool BF16, int A_TERMS, bool OUT_BF16 = BF16, int BN = 256>
cudaError_t launch_impl(const void *A, const void *A2, const void *B0, const void *B1, void *out0,
                        void *out1, int64_t M, int64_t K, int64_t N, int kind, float acc_scale,
                        float out_scale, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    constexpr size_t SMEM_BYTES = Ring<A_TERMS, BN>::SMEM_BYTES;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(gemm_tcgen05_kernel<MODE, BF16, A_TERMS, OUT_BF16, BN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(SMEM_BYTES));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    CUtensorMap ma, ma2, mb0, mb1;
    if (!make_map(&ma, A, BF16, K, M, BM)) return cudaErrorInvalidValue;
    ma2 = ma;
    if (A_TERMS == 2 && !make_map(&ma2, A2, BF16, K, M, BM)) return cudaErrorInvalidValue;
    if (MODE == MODE_PLAIN) {
        if (!make_map(&mb0, B0, BF16, K, N, BN)) return cudaErrorInvalidValue;
        mb1 = mb0;
    } else {
        if (!make_map(&mb0, B0, BF16, K, N, BN / 2)) return cudaErrorInvalidValue;
        if (!make_map(&mb1, B1, BF16, K, N, BN / 2)) return cudaErrorInvalidValue;
    }
    GemmParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_m_blocks = (M + BM - 1) / BM;
    const int64_t ncols = MODE == MODE_PLAIN ? BN : BN / 2;
    const int64_t num_n_blocks = (N + ncols - 1) / ncols;
    p.num_tiles = p.num_m_blocks * num_n_blocks;
    p.num_k_blocks = static_cast<int>((K + BK - 1) / BK);
    p.out0 = out0;
    p.out1 = out1;
    p.ldo = N;
    p.err = device_status_word();
    p.wait_limit_ns = WAIT_LIMIT_NS;
    p.acc_scale = acc_scale;
    p.out_scale = out_scale;
    if (!p.err) return cudaErrorUnknown;
    int64_t grid = sm_count();
    if (grid > p.num_tiles) grid = p.num_tiles;
    LaunchScope scope(kind, s);
    gemm_tcgen05_kernel<MODE, BF16, A_TERMS, OUT_BF16, BN>
        <<<static_cast<unsigned>(grid), NUM_THREADS, SMEM_BYTES, s>>>(ma, ma2, mb0, mb1, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_gateup(int dt, const void *A, const void *A_lo, const void *Wg,
                               const void *Wu, void *H, void *H_lo, void *G, void *U, int64_t M,
                               int64_t K, int64_t F, bool fused, float acc_scale, float out_scale,
                               cudaStream_t s) {
    const bool bf = dt == DT_BF16;
    const int k = K_GEMM_GATEUP;
    const float a = acc_scale, o = out_scale;
    if (A_lo) {
        if (fused)
            return bf ? launch_impl<MODE_GATEUP_FUSED, true, 2>(A, A_lo, Wg, Wu, H, H_lo, M, K, F, k, a, o, s)
                      : launch_impl<MODE_GATEUP_FUSED, false, 2>(A, A_lo, Wg, Wu, H, H_lo, M, K, F, k, a, o, s);
        return bf ? launch_impl<MODE_GATEUP_SPLIT, true, 2>(A, A_lo, Wg, Wu, G, U, M, K, F, k, a, o, s)
                  : launch_impl<MODE_GATEUP_SPLIT, false, 2>(A, A_lo, Wg, Wu, G, U, M, K, F, k, a, o, s);
    }
    if (fused)
        return bf ? launch_impl<MODE_GATEUP_FUSED, true, 1>(A, nullptr, Wg, Wu, H, H_lo, M, K, F, k, a, o, s)
                  : launch_impl<MODE_GATEUP_FUSED, false, 1>(A, nullptr, Wg, Wu, H, H_lo, M, K, F, k, a, o, s);
    return bf ? launch_impl<MODE_GATEUP_SPLIT, true, 1>(A, nullptr, Wg, Wu, G, U, M, K, F, k, a, o, s)
              : launch_impl<MODE_GATEUP_SPLIT, false, 1>(A, nullptr, Wg, Wu, G, U, M, K, F, k, a, o, s);
}

// Tile width for the plain GEMM: waves of tiles times the width of a tile
// (time per wave scales with it); e.g. 4096 columns on 152 SMs with 32 row
// blocks: 256 wide -> 512 tiles, 4 waves (the last 37 % full); 224 wide ->
// 608 tiles, exactly 4 full waves.
int plain_tile_width(int64_t M, int64_t N) {
    const int64_t mb = (M + BM - 1) / BM;
    const int64_t sms = sm_count();
    int best = 256;
    int64_t best_cost = 0;
    for (int bn : {256, 224}) {
        const int64_t tiles = mb * ((N + bn - 1) / bn);
        const int64_t cost = ((tiles + sms - 1) / sms) * bn;
        if (best_cost == 0 || cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

template <bool BF16, int A_TERMS, bool OUT_BF16>
cudaError_t launch_plain_bn(const void *A, const void *A_lo, const void *B, void *C, int64_t M,
                            int64_t K, int64_t N, float acc_scale, cudaStream_t s) {
    if (plain_tile_width(M, N) == 224)
        return launch_impl<MODE_PLAIN, BF16, A_TERMS, OUT_BF16, 224>(A, A_lo, B, nullptr, C, nullptr, M, K,
                                                                     N, K_GEMM_DOWN, acc_scale, 1.f, s);
    return launch_impl<MODE_PLAIN, BF16, A_TERMS, OUT_BF16, 256>(A, A_lo, B, nullptr, C, nullptr, M, K, N,
                                                                 K_GEMM_DOWN, acc_scale, 1.f, s);
}

cudaError_t launch_gemm_plain(int dt, int dt_out, const void *A, const void *A_lo, const void *B,
                              void *C, int64_t M, int64_t K, int64_t N, float acc_scale,
                              cudaStream_t s) {
    const float a = acc_scale;
    if (dt == DT_BF16) {
        if (A_lo) return launch_plain_bn<true, 2, true>(A, A_lo, B, C, M, K, N, a, s);
        return launch_plain_bn<true, 1, true>(A, nullptr, B, C, M, K, N, a, s);
    }
    if (dt_out == DT_BF16) {   // fp16 operands, bf16 output (prepared-weights path)
        if (A_lo) return launch_plain_bn<false, 2, true>(A, A_lo, B, C, M, K, N, a, s);
        return launch_plain_bn<false, 1, true>(A, nullptr, B, C, M, K, N, a, s);
    }
    if (A_lo) return launch_plain_bn<false, 2, false>(A, A_lo, B, C, M, K, N, a, s);
    return launch_plain_bn<false, 1, false>(A, nullptr, B, C, M, K, N, a, s);
}

}  // namespace ffn
