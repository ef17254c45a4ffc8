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
// kernel's main loop, tiles and schedule ("Megakernels on Mac: What Fusion Saves and What It Costs", section
// "Packing and geometry in the unfused control"); only the epilogue differs.
//
// Kernel structure (one CTA per SM, persistent over output tiles):
//   warp 0      one thread issues TMA loads of A (128 x 64) and B (BN x 64)
//               bf16/fp16 tiles, 128-byte swizzled, into a ring of as many
//               stages as fit (4-5);
//   warp 1      allocates 512 TMEM columns (two 128 x BN fp32 accumulators);
//               one thread issues tcgen05.mma (M=128, N=BN, K=16) and
//               tcgen05.commit to release ring slots and publish accumulators;
//   warps 2-5   epilogue: tcgen05.ld rows of the finished accumulator, apply
//               the epilogue, store 16-byte vectors, release the accumulator
//               so the next tile's MMAs overlap this tile's epilogue.
// CTAs run in clusters of two over row blocks 2i and 2i+1 of the same column
// block, and the even CTA issues tcgen05.mma.cta_group::2 over both: each
// CTA loads its own 128-row A tile and one half of the B tile
// (cp.async.bulk.tensor ... .cta_group::2) into its OWN ring, the two copies'
// byte counts completing on the even CTA's ring barrier; the pair MMA reads
// the A rows and the B half from each CTA's shared memory.  No copy is
// multicast: every B byte leaves L2 once per pair because each CTA fetches a
// different half.  A ring slot is reused once the pair's MMAs have released
// it (the commit arrives on the barriers of both CTAs).
// The kernel is launched as a programmatic dependent of the kernel before it:
// the first ring's worth of B (weights) is requested before that kernel has
// finished, A (its output) only after.
// Every mbarrier wait is bounded (1 s of wall time).  A wait that gives up
// sets the device status word, tells the other roles to stop, waits (again
// bounded) for its own TMA loads and MMAs in flight, and frees TMEM; the two
// CTAs of a cluster leave together.
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
// BN: accumulator columns per tile (256; 224 for the plain GEMM when it
// evens out the waves; with few row blocks 192, or 64 for a down GEMM whose
// reduction is too short to split); the B tile is BN rows of 64 k values, all of them in
// this CTA's ring, or (PAIR) BN/2 of them, the peer CTA holding the others.
// The ring takes as many stages as fit in 225 KB; a CTA therefore always
// holds more than half of the SM's shared memory, so two of these CTAs
// (each allocating all of TMEM) never share an SM, not even while one kernel
// overlaps the tail of the one before it.
// KSUB: 64-wide k blocks per ring stage.  A pair stage holds two (one
// barrier wait and one release per 8 MMAs instead of 4): the MMA thread's
// per-stage overhead is not hidden by the tensor pipe's queue.
template <int A_TERMS, int BN, bool PAIR> struct Ring {
    static constexpr int KSUB = (PAIR && A_TERMS == 1) ? 2 : 1;
    static constexpr uint32_t B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;   // this CTA's part of B, per k block
    static constexpr uint32_t SUB_BYTES = A_TERMS * A_BYTES + B_BYTES;
    static constexpr uint32_t STAGE_BYTES = KSUB * SUB_BYTES;
    static constexpr int FIT = static_cast<int>((225u * 1024u) / STAGE_BYTES);
    static constexpr int STAGES = FIT > 8 ? 8 : FIT;
    static constexpr size_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
    static_assert(STAGES >= 3 && SMEM_BYTES > 114 * 1024, "ring");
};
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

enum Mode { MODE_PLAIN = 0, MODE_GATEUP_FUSED = 1, MODE_GATEUP_SPLIT = 2 };

struct GemmParams {
    int64_t M, N, K;          // N: output columns (ffn for gate/up, d for down)
    int64_t num_m_blocks, num_n_blocks;
    int num_k_blocks;
    // split-K (plain mode, too few tiles to fill the SMs): unit u sums ring
    // stages [kst_per_split * s, kst_per_split * (s + 1)) of its tile, s =
    // u / (pairs x column blocks), and stores the fp32 sum in part[s]; a
    // second kernel adds the splits in order.  Unsplit: kst_per_split covers
    // all stages and part is null.
    int kst_per_split;
    float *part;
    // CTAs per unit of work: 1, or 2 for a CTA pair (rows of row blocks 2i
    // and 2i+1 against one column block, one M=256 MMA over both SMs)
    int cluster;
    int64_t num_m_pairs, num_units;
    void *out0, *out1;        // plain: C; fused: h (and its residual, or null); split: G, U
    int64_t ldo;              // output row stride in elements
    unsigned *err;
    uint64_t wait_limit_ns;
    float acc_scale;          // applied to every accumulator value (exact powers of two)
    float out_scale;          // fused: applied to h before rounding
    int a_keep;               // keep A in L2 (evict-last): every wave of tiles re-reads it
    const void *res;          // plain: added to C before rounding (same type and layout as C), or null
    // plain, unsplit, with ss_out: each row's sum of squares of the stored C,
    // through per-column-block parts ss_part[n_blk][M] and per-row-block
    // arrival counters ss_ctr[m_blk] (zero at the start; the last arrival
    // adds the parts in column-block order)
    float *ss_part;
    unsigned *ss_ctr;
    float *ss_out;
    unsigned *zero;           // counters of a later kernel of the call, zeroed once the wait returns
    int nzero;
};

// What a launch adds to the plain GEMM's output, and what it clears for a
// later kernel (see GemmParams).
struct GemmRowSS {
    float *part = nullptr;
    unsigned *ctr = nullptr;
    float *out = nullptr;
    unsigned *zero = nullptr;
    int nzero = 0;
};

// Stores NV (16 or 32) values rounded once; with `lo` also the rounding
// residual v - round(v), rounded once, so that hi + lo carries ~16
// significant bits.  Columns at or past ncols (a multiple of 8) are skipped.
template <typename T, int NV>
__device__ __forceinline__ void store_row(T *dst, T *lo, int64_t col, int64_t ncols, const float (&v)[NV]) {
#pragma unroll
    for (int j = 0; j < NV / 8; ++j) {
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

// Sum of the squares of v rounded to T (the values store_row writes), over
// the columns below ncols, in column order.
template <typename T, int NV>
__device__ __forceinline__ float stored_sumsq(int64_t col, int64_t ncols, const float (&v)[NV]) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < NV / 8; ++j)
        if (col + 8 * j < ncols)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float r = to_f32(from_f32<T>(v[8 * j + e]));
                s = fmaf(r, r, s);
            }
    return s;
}

// v[e] += src[col + e] for the NV (16 or 32) columns from col that are
// below ncols (a multiple of 8), 16-byte loads.
template <typename T, int NV>
__device__ __forceinline__ void add_row(const T *src, int64_t col, int64_t ncols, float (&v)[NV]) {
#pragma unroll
    for (int j = 0; j < NV / 8; ++j) {
        if (col + 8 * j < ncols) {
            float f[8];
            Vec16<T>::unpack(*reinterpret_cast<const uint4 *>(src + col + 8 * j), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[8 * j + e] += f[e];
        }
    }
}

template <int NV>
__device__ __forceinline__ void store_row_f32(float *dst, int64_t col, int64_t ncols, const float (&v)[NV]) {
#pragma unroll
    for (int j = 0; j < NV / 4; ++j)
        if (col + 4 * j < ncols)
            *reinterpret_cast<float4 *>(dst + col + 4 * j) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

// BF16: operand type (bf16 or fp16); OUT_BF16: type of the stored output
// (plain mode; the fused h has the operand type, it feeds the next GEMM).
// PAIR: clusters of two CTAs on two SMs compute 256 x BN tiles with
// tcgen05 .cta_group::2 MMAs issued by the even CTA.  Each CTA's ring holds
// its own 128 rows of A and half of B (W_gate rows in the even CTA and W_up
// rows in the odd one for gate/up; the two column halves for the plain
// GEMM), so per flop an SM stores and feeds a third fewer operand bytes than
// with one CTA per 128 x BN tile, and each B byte leaves L2 once per pair.
// The pair's producers report their bytes to the even CTA's ring barriers;
// the even CTA's MMA thread releases ring slots and publishes accumulators
// to both CTAs; both epilogues (each reading its own TMEM rows) report to
// the even CTA's accumulator barriers.
template <int MODE, bool BF16, int A_TERMS, bool OUT_BF16, int BN, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_a2,
                        const __grid_constant__ CUtensorMap map_b0,
                        const __grid_constant__ CUtensorMap map_b1, const GemmParams p) {
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    using TOut = typename std::conditional<OUT_BF16, __nv_bfloat16, __half>::type;
    using RG = Ring<A_TERMS, BN, PAIR>;
    static_assert(BN % 32 == 0 && BN <= 256 && (BN / 2) % 16 == 0, "tile width");
    // epilogue chunk: 32 accumulator columns, or 16 when a half tile (gate
    // or up part of a fused tile) is not a multiple of 32 wide
    constexpr int CW = (MODE == MODE_PLAIN || (BN / 2) % 32 == 0) ? 32 : 16;
    constexpr int STAGES = RG::STAGES, KSUB = RG::KSUB;
    constexpr uint32_t STAGE_BYTES = RG::STAGE_BYTES, SUB_BYTES = RG::SUB_BYTES;
    constexpr uint32_t B_BYTES = RG::B_BYTES;
    constexpr int NCTA = PAIR ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[STAGES], bar_empty[STAGES];
    __shared__ __align__(8) uint64_t bar_tfull[2], bar_tempty[2], bar_drain;
    __shared__ uint32_t s_tmem_base;
    __shared__ int s_abort, s_never;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
    // stage s, k block j of it: A term 0 | A term 1 (if any) | B (or this
    // CTA's half), each 1024-byte aligned
    auto sA = [&](uint32_t s, int j, int t) { return base + s * STAGE_BYTES + j * SUB_BYTES + t * A_BYTES; };
    auto sB = [&](uint32_t s, int j) { return base + s * STAGE_BYTES + j * SUB_BYTES + A_TERMS * A_BYTES; };
    const int nst = (p.num_k_blocks + KSUB - 1) / KSUB;   // ring stages per tile
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
            ptx::mbar_init(tempty(a), 4 * NCTA);   // the epilogue warps of every CTA of the unit
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
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_u32(&s_tmem_base), TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_u32(&s_tmem_base), TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised before either reports to the other
    if constexpr (PAIR) ptx::cluster_sync();
    ptx::tc_fence_after();
    // the next kernel on the stream may be scheduled once every CTA is running
    ptx::griddep_launch_dependents();
    const uint32_t tmem_base = s_tmem_base;
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int64_t unit0 = blockIdx.x / NCTA, unit_step = gridDim.x / NCTA;
    auto m_blk_of = [&](int64_t u) { return (u % p.num_m_pairs) * NCTA + rank; };
    auto n_blk_of = [&](int64_t u) { return (u / p.num_m_pairs) % p.num_n_blocks; };
    auto split_of = [&](int64_t u) { return static_cast<int>(u / (p.num_m_pairs * p.num_n_blocks)); };
    auto kst_lo = [&](int64_t u) { return split_of(u) * p.kst_per_split; };
    auto kst_hi = [&](int64_t u) {
        const int e = kst_lo(u) + p.kst_per_split;
        return e < nst ? e : nst;
    };
    // the barriers the pair shares live in the even CTA
    auto lead = [&](uint32_t bar) { return PAIR ? ptx::mapa_shared(bar, 0) : bar; };
    volatile int *abort_flag = &s_abort;
    volatile int *never = &s_never;
    const uint64_t limit = p.wait_limit_ns;
    uint64_t produced = 0;   // k-blocks whose TMA loads were issued (producer thread)

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ TMA producer
        const uint64_t keep = ptx::l2_policy_evict_last();
        auto load = [&](uint32_t dst, const CUtensorMap *map, uint32_t s, int x, int y, bool hint) {
            if constexpr (PAIR) {
                if (hint) ptx::tma_load_2d_pair_hint(dst, map, lead(full(s)), x, y, keep);
                else ptx::tma_load_2d_pair(dst, map, lead(full(s)), x, y);
            } else {
                if (hint) ptx::tma_load_2d_hint(dst, map, full(s), x, y, keep);
                else ptx::tma_load_2d(dst, map, full(s), x, y);
            }
        };
        // stage s holds k blocks KSUB * kst .. (a block past K is TMA zero fill)
        auto load_a = [&](uint32_t s, int kst, int m0) {
#pragma unroll
            for (int j = 0; j < KSUB; ++j) {
                const int k0 = (kst * KSUB + j) * BK;
                load(sA(s, j, 0), &map_a, s, k0, m0, p.a_keep != 0);
                if (A_TERMS == 2) load(sA(s, j, 1), &map_a2, s, k0, m0, p.a_keep != 0);
            }
        };
        auto load_b = [&](uint32_t s, int kst, int64_t n_blk) {
#pragma unroll
            for (int j = 0; j < KSUB; ++j) {
                const int k0 = (kst * KSUB + j) * BK;
                if constexpr (PAIR) {
                    // plain: columns BN/2 * rank .. of the tile; gate/up: the
                    // W_gate rows (even CTA) or the W_up rows (odd CTA)
                    if (MODE == MODE_PLAIN)
                        load(sB(s, j), &map_b0, s, k0, static_cast<int>(n_blk * BN + rank * (BN / 2)), false);
                    else
                        load(sB(s, j), rank ? &map_b1 : &map_b0, s, k0, static_cast<int>(n_blk * (BN / 2)), false);
                } else if (MODE == MODE_PLAIN) {
                    load(sB(s, j), &map_b0, s, k0, static_cast<int>(n_blk * BN), false);
                } else {
                    const int f0 = static_cast<int>(n_blk * (BN / 2));
                    load(sB(s, j), &map_b0, s, k0, f0, false);
                    load(sB(s, j) + B_BYTES / 2, &map_b1, s, k0, f0, false);
                }
            }
        };
        // the even CTA expects the bytes of the whole pair on its barrier
        auto arm = [&](uint32_t s) {
            if (leader) ptx::mbar_arrive_expect_tx(full(s), NCTA * STAGE_BYTES);
        };
        // The first ring's worth of B (weights: inputs of the call) is
        // requested before the kernel that writes A has finished; A only
        // after it has.  The grid never exceeds the unit count, so every CTA
        // has a first unit.
        const int kfirst = kst_lo(unit0), nfirst = kst_hi(unit0) - kfirst;
        const int npre = nfirst < STAGES ? nfirst : STAGES;
        for (int kb = 0; kb < npre; ++kb) {
            arm(kb);
            load_b(kb, kfirst + kb, n_blk_of(unit0));
        }
        ptx::griddep_wait();
        for (int kb = 0; kb < npre; ++kb) load_a(kb, kfirst + kb, static_cast<int>(m_blk_of(unit0) * BM));
        produced = npre;
        bool ok = true;
        for (int64_t u = unit0; u < p.num_units && ok; u += unit_step) {
            const int m0 = static_cast<int>(m_blk_of(u) * BM);
            const int64_t n_blk = n_blk_of(u);
            for (int kb = (u == unit0) ? kfirst + npre : kst_lo(u), ke = kst_hi(u); kb < ke; ++kb) {
                const uint32_t s = static_cast<uint32_t>(produced % STAGES);
                const uint32_t ph = static_cast<uint32_t>((produced / STAGES) & 1);
                if (!ptx::mbar_wait(empty(s), ph ^ 1u, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                arm(s);
                load_a(s, kb, m0);
                load_b(s, kb, n_blk);
                ++produced;
            }
        }
        if (!ok) {
            atomicOr(p.err, DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // -------------------------------------------------------- MMA issuer
        constexpr uint32_t idesc = ptx::idesc_f16(BM * NCTA, BN, BF16);
        bool ok = true;
        uint64_t consumed = 0;
        uint32_t acc = 0, acc_ph = 0;
        for (int64_t u = unit0; u < p.num_units && ok; u += unit_step) {
            if (!ptx::mbar_wait(tempty(acc), acc_ph ^ 1u, abort_flag, limit)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            const int kb0 = kst_lo(u), ke = kst_hi(u);
            for (int kb = kb0; kb < ke; ++kb) {
                const uint32_t s = static_cast<uint32_t>(consumed % STAGES);
                const uint32_t ph = static_cast<uint32_t>((consumed / STAGES) & 1);
                if (!ptx::mbar_wait(full(s), ph, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
#pragma unroll
                for (int j = 0; j < KSUB; ++j) {
                    const uint32_t b0 = sB(s, j);
#pragma unroll
                    for (int t = 0; t < A_TERMS; ++t) {
                        const uint32_t a0 = sA(s, j, t);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            const uint64_t ad = ptx::sdesc_k_sw128(a0 + k * UMMA_K * 2);
                            const uint64_t bd = ptx::sdesc_k_sw128(b0 + k * UMMA_K * 2);
                            const uint32_t accumulate = ((kb - kb0) | j | k | t) != 0 ? 1u : 0u;
                            if constexpr (PAIR) ptx::tc_mma_f16_pair(d_tmem, ad, bd, idesc, accumulate);
                            else ptx::tc_mma_f16(d_tmem, ad, bd, idesc, accumulate);
                        }
                    }
                }
                // the slot is free again in every CTA of the unit
                if constexpr (PAIR) ptx::tc_commit_pair(empty(s), 0x3);
                else ptx::tc_commit(empty(s));
                ++consumed;
            }
            if (!ok) break;
            if constexpr (PAIR) ptx::tc_commit_pair(tfull(acc), 0x3);
            else ptx::tc_commit(tfull(acc));
            acc ^= 1u;
            if (acc == 0) acc_ph ^= 1u;
        }
        if (!ok) {
            atomicOr(p.err, DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
        // every MMA issued above must finish before TMEM is freed
        if constexpr (PAIR) ptx::tc_commit_pair(ptx::smem_u32(&bar_drain), 0x1);
        else ptx::tc_commit(ptx::smem_u32(&bar_drain));
        ptx::mbar_wait(ptx::smem_u32(&bar_drain), 0, never, limit);
    } else if (warp >= 2) {
        // ---------------------------------------------------------- epilogue
        ptx::griddep_wait();   // outputs may be read by the kernel before this one
        if (blockIdx.x == 0 && warp == 2)
            for (int i = lane; i < p.nzero; i += 32) p.zero[i] = 0u;
        const int q = warp & 3;   // this warp may read TMEM lanes 32q .. 32q+31
        bool ok = true;
        uint32_t acc = 0, acc_ph = 0;
        T *out0 = static_cast<T *>(p.out0);
        T *out1 = static_cast<T *>(p.out1);
        for (int64_t u = unit0; u < p.num_units; u += unit_step) {
            const int64_t m_blk = m_blk_of(u), n_blk = n_blk_of(u);
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
            float ss = 0.f;   // this row's stored values squared, over the tile's columns
            if (MODE == MODE_PLAIN) {
#pragma unroll 1
                for (int c = 0; c < BN; c += CW) {
                    uint32_t r[CW];
                    ptx::tmem_ld_cols<CW>(taddr + c, r);
                    ptx::tmem_ld_wait();
                    float v[CW];
#pragma unroll
                    for (int j = 0; j < CW; ++j) v[j] = __uint_as_float(r[j]) * p.acc_scale;
                    if (live) {
                        const int64_t col = n_blk * BN + c;
                        if (p.part) {
                            float *dst = p.part + (static_cast<int64_t>(split_of(u)) * p.M + row) * p.ldo;
                            store_row_f32<CW>(dst, col, p.N, v);
                        } else {
                            if (p.res)
                                add_row<TOut, CW>(static_cast<const TOut *>(p.res) + row * p.ldo, col, p.N, v);
                            store_row<TOut, CW>(static_cast<TOut *>(p.out0) + row * p.ldo, nullptr, col, p.N, v);
                            if (p.ss_out) ss += stored_sumsq<TOut, CW>(col, p.N, v);
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += CW) {
                    uint32_t rg[CW], ru[CW];
                    ptx::tmem_ld_cols<CW>(taddr + c, rg);
                    ptx::tmem_ld_cols<CW>(taddr + BN / 2 + c, ru);
                    ptx::tmem_ld_wait();
                    const int64_t col = n_blk * (BN / 2) + c;
                    if (MODE == MODE_GATEUP_FUSED) {
                        float h[CW];
#pragma unroll
                        for (int j = 0; j < CW; ++j)
                            h[j] = silu_f32(__uint_as_float(rg[j]) * p.acc_scale) *
                                   (__uint_as_float(ru[j]) * p.acc_scale) * p.out_scale;
                        if (live)
                            store_row<T, CW>(out0 + row * p.ldo, out1 ? out1 + row * p.ldo : nullptr, col, p.N, h);
                    } else {
                        float gv[CW], uv[CW];
#pragma unroll
                        for (int j = 0; j < CW; ++j) {
                            gv[j] = __uint_as_float(rg[j]) * p.acc_scale;
                            uv[j] = __uint_as_float(ru[j]) * p.acc_scale;
                        }
                        // G and U stay fp32 so that h is rounded exactly
                        // once, as in the fused arm
                        if (live) {
                            store_row_f32<CW>(static_cast<float *>(p.out0) + row * p.ldo, col, p.N, gv);
                            store_row_f32<CW>(static_cast<float *>(p.out1) + row * p.ldo, col, p.N, uv);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && !leader) ptx::mbar_arrive_cluster(lead(tempty(acc)));
                else ptx::mbar_arrive(tempty(acc));
            }
            acc ^= 1u;
            if (acc == 0) acc_ph ^= 1u;
            if (MODE == MODE_PLAIN && p.ss_out && !p.part) {
                // "Megakernels on Mac: What Fusion Saves and What It Costs",
                // "Dependencies and synchronization": the next RMSNorm needs
                // the whole row's sum of squares; each warp leaves its rows'
                // part for this column block, and the last of the row block's
                // arrivals (4 warps per column block) adds them in order
                if (live) p.ss_part[n_blk * p.M + row] = ss;
                __syncwarp();
                unsigned last = 0;
                if (lane == 0) {
                    __threadfence();
                    last = atomicAdd(&p.ss_ctr[m_blk], 1u) == static_cast<unsigned>(4 * p.num_n_blocks - 1);
                }
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __threadfence();
                    for (int r = lane; r < BM; r += 32) {
                        const int64_t rr = m_blk * BM + r;
                        if (rr >= p.M) continue;
                        float t = 0.f;
                        for (int64_t nb = 0; nb < p.num_n_blocks; ++nb) t += __ldcg(p.ss_part + nb * p.M + rr);
                        p.ss_out[rr] = t;
                    }
                    if (lane == 0) p.ss_ctr[m_blk] = 0u;
                }
            }
        }
        if (!ok && lane == 0) {
            atomicOr(p.err, DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    __syncthreads();
    if (warp == 0 && lane == 0 && leader) {
        // TMA loads still in flight (only after an abandoned wait) must land
        // before shared memory is released; the even CTA's ring barriers
        // count the bytes of both CTAs of a pair.
        for (uint32_t s = 0; s < STAGES; ++s) {
            if (produced > s) {
                const uint64_t armed = (produced - s + STAGES - 1) / STAGES;
                ptx::mbar_wait(full(s), static_cast<uint32_t>((armed - 1) & 1), never, limit);
            }
        }
    }
    if constexpr (PAIR) {
        // neither CTA of the pair leaves (or frees TMEM) while the other may
        // still copy into its shared memory, arrive on its barriers or
        // read the accumulators
        __syncthreads();
        ptx::cluster_sync();
    }
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        if constexpr (PAIR) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else ptx::tmem_dealloc(tmem_base, TMEM_COLS);
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

template <int MODE, bool BF16, int A_TERMS, bool OUT_BF16, int BN, bool PAIR>
cudaError_t launch_kernel(const void *A, const void *A2, const void *B0, const void *B1, void *out0,
                          void *out1, int64_t M, int64_t K, int64_t N, int kind, float acc_scale,
                          float out_scale, const void *res, float *part, int kst_per_split, int splits,
                          GemmRowSS ex, cudaStream_t s) {
    constexpr size_t SMEM_BYTES = Ring<A_TERMS, BN, PAIR>::SMEM_BYTES;
    constexpr int NCTA = PAIR ? 2 : 1;
    using RG = Ring<A_TERMS, BN, PAIR>;
    const auto kern = &gemm_tcgen05_kernel<MODE, BF16, A_TERMS, OUT_BF16, BN, PAIR>;
    static int configured_device = -1, slots = 0;   // co-resident units (CTAs or pairs)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
        if (e != cudaSuccess) return e;
        slots = sm_count();
        if (PAIR) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * static_cast<unsigned>(sm_count()));
            cfg.blockDim = dim3(NUM_THREADS);
            cfg.dynamicSmemBytes = SMEM_BYTES;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&slots, kern, &cfg);
            if (e != cudaSuccess) return e;
        }
        if (slots < 1) return cudaErrorLaunchOutOfResources;
        configured_device = dev;
    }
    const int64_t num_m_blocks = (M + BM - 1) / BM;
    const int64_t ncols = MODE == MODE_PLAIN ? BN : BN / 2;
    const int64_t num_n_blocks = (N + ncols - 1) / ncols;
    CUtensorMap ma, ma2, mb0, mb1;
    if (!make_map(&ma, A, BF16, K, M, BM)) return cudaErrorInvalidValue;
    ma2 = ma;
    if (A_TERMS == 2 && !make_map(&ma2, A2, BF16, K, M, BM)) return cudaErrorInvalidValue;
    if (MODE == MODE_PLAIN) {
        // with a pair, each CTA loads half of the B tile
        if (!make_map(&mb0, B0, BF16, K, N, static_cast<uint32_t>(BN / NCTA))) return cudaErrorInvalidValue;
        mb1 = mb0;
    } else {
        if (!make_map(&mb0, B0, BF16, K, N, BN / 2)) return cudaErrorInvalidValue;
        if (!make_map(&mb1, B1, BF16, K, N, BN / 2)) return cudaErrorInvalidValue;
    }
    GemmParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.num_m_blocks = num_m_blocks;
    p.num_n_blocks = num_n_blocks;
    p.num_k_blocks = static_cast<int>((K + BK - 1) / BK);
    p.kst_per_split = splits > 1 ? kst_per_split : (p.num_k_blocks + RG::KSUB - 1) / RG::KSUB;
    p.part = splits > 1 ? part : nullptr;
    p.cluster = NCTA;
    p.num_m_pairs = (num_m_blocks + NCTA - 1) / NCTA;
    p.num_units = p.num_m_pairs * num_n_blocks * (splits > 1 ? splits : 1);
    p.out0 = out0;
    p.out1 = out1;
    p.ldo = N;
    p.err = device_status_word();
    p.wait_limit_ns = WAIT_LIMIT_NS;
    p.acc_scale = acc_scale;
    p.out_scale = out_scale;
    // every wave of tiles re-reads all of A (tiles are ordered row block
    // fastest); ask L2 to keep it when it fits comfortably
    p.a_keep = (num_n_blocks > 1 && M * K * 2 * A_TERMS <= (int64_t{96} << 20)) ? 1 : 0;
    p.res = res;
    p.ss_part = ex.part;
    p.ss_ctr = ex.ctr;
    p.ss_out = ex.out;
    p.zero = ex.zero;
    p.nzero = ex.nzero;
    if (!p.err) return cudaErrorUnknown;
    // persistent: one unit of CTAs per co-resident slot, never more units
    // than there is work for
    int64_t units = slots;
    if (units > p.num_units) units = p.num_units;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * NCTA));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(NCTA);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 2 : 1;
    LaunchScope scope(kind, s);
    e = cudaLaunchKernelEx(&cfg, kern, ma, ma2, mb0, mb1, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// CTA pairs whenever there are at least two row blocks to pair up.
template <int MODE, bool BF16, int A_TERMS, bool OUT_BF16 = BF16, int BN = 256>
cudaError_t launch_impl(const void *A, const void *A2, const void *B0, const void *B1, void *out0,
                        void *out1, int64_t M, int64_t K, int64_t N, int kind, float acc_scale,
                        float out_scale, cudaStream_t s, const void *res = nullptr, float *part = nullptr,
                        int kst_per_split = 0, int splits = 1, GemmRowSS ex = {}) {
    if (M <= 0) return cudaSuccess;
    if (M > BM)
        return launch_kernel<MODE, BF16, A_TERMS, OUT_BF16, BN, true>(A, A2, B0, B1, out0, out1, M, K, N, kind,
                                                                       acc_scale, out_scale, res, part,
                                                                       kst_per_split, splits, ex, s);
    return launch_kernel<MODE, BF16, A_TERMS, OUT_BF16, BN, false>(A, A2, B0, B1, out0, out1, M, K, N, kind,
                                                                    acc_scale, out_scale, res, part,
                                                                    kst_per_split, splits, ex, s);
}

// Waves of tiles times the width of a tile (the time of a wave scales with
// it), for units of `ncta` CTAs each covering `cols` output columns.
int64_t wave_cost(int64_t M, int64_t N, int cols, int width) {
    const int64_t mb = (M + BM - 1) / BM;
    const int64_t ncta = mb > 1 ? 2 : 1;
    const int64_t units = ((mb + ncta - 1) / ncta) * ((N + cols - 1) / cols);
    const int64_t slots = sm_count() / ncta > 0 ? sm_count() / ncta : 1;
    return ((units + slots - 1) / slots) * width;
}

// Tile width of the plain GEMM.  E.g. 4096 rows onto 4096 columns: 224-wide
// tiles make 608 tiles, exactly 4 waves on 152 SMs (256 wide: 512 tiles, the
// 4th wave 37 % full).
int tile_width(int64_t M, int64_t N) {
    return wave_cost(M, N, 224, 224) < wave_cost(M, N, 256, 256) ? 224 : 256;
}

// Gate/up tile width: 128 + 128 features, or 96 + 96 when the 256-wide tiles
// take at most two waves and the narrower ones take less time.  Small batches
// stream the weights, and the tile count sets how many SMs do it: ffn 14336
// on one row block makes 150 tiles of 96 + 96 on 152 SMs against 112 of 128 +
// 128; on two row blocks (one CTA pair each tile) 2 waves of 192 against 2 of
// 256.  Long prefill keeps 256 even where 192 evens the waves: on 4096 x
// 11008, 112 + 112 tiles ran 6 % slower, a narrower tile moving more operand
// bytes from L2 per flop.
int gateup_width(int64_t M, int64_t N) {
    const int64_t wide = wave_cost(M, N, 128, 256);
    return (wide <= 2 * 256 && wave_cost(M, N, 96, 192) < wide) ? 192 : 256;
}

// Split-K plan of the plain GEMM (the down projection).  With fewer 256-wide
// tiles than half the CTA slots (d 4096 on up to 512 rows: 16-64 CTAs of
// 152), each CTA would stream a whole K-long strip of W_down through one SM.
// Instead the reduction is cut into `splits` runs of whole ring stages
// (at least kMinSplitKBlocks 64-wide k blocks each) that together fill the
// SMs; each run stores an fp32 partial tile, and splitk_reduce_kernel adds
// them in split order (deterministic) with the residual, rounding once.
// Tiles are 192 wide when those can be split (fewer splits, so less partial
// traffic: 4096 columns at 64-256 rows 1-3 % faster than 256 wide), else 256.
// Returns the split count (1: no split), the stages per run and the width.
constexpr int kMinSplitKBlocks = 8, kMaxSplits = 16;
int plain_split_plan(int64_t M, int64_t K, int64_t N, int a_terms, int *kst_per_split, int *width) {
    const int64_t mb = (M + BM - 1) / BM;
    const bool pair = mb > 1;
    const int64_t ncta = pair ? 2 : 1;
    const int64_t slots = sm_count() / ncta;
    const int64_t kblocks = (K + BK - 1) / BK;
    const int64_t ksub = (pair && a_terms == 1) ? 2 : 1;   // Ring<a_terms, BN, pair>::KSUB
    const int64_t nst = (kblocks + ksub - 1) / ksub;
    if (M <= 0) return 1;
    for (int bn : {192, 256}) {
        const int64_t units = ((mb + ncta - 1) / ncta) * ((N + bn - 1) / bn);
        if (2 * units > slots) continue;
        int64_t sp = slots / units;
        if (sp > kblocks / kMinSplitKBlocks) sp = kblocks / kMinSplitKBlocks;
        if (sp > kMaxSplits) sp = kMaxSplits;
        if (sp < 2) return 1;
        const int64_t per = (nst + sp - 1) / sp;
        if (kst_per_split) *kst_per_split = static_cast<int>(per);
        if (width) *width = bn;
        return static_cast<int>((nst + per - 1) / per);
    }
    return 1;
}
static_assert(Ring<1, 256, true>::KSUB == 2 && Ring<2, 256, true>::KSUB == 1 && Ring<1, 256, false>::KSUB == 1 &&
                  Ring<1, 192, true>::KSUB == 2 && Ring<1, 192, false>::KSUB == 1,
              "plain_split_plan's stage size");

// out = sum over s of part[s] (s = 0, 1, ...) + res, rounded once to TOut.
// part: [splits][count] fp32; count (M x N) is a multiple of 8.  One float4
// a thread; the loads of up to four splits are in flight at once (the
// partials sit in L2: the kernel is bound by their latency, not bandwidth).
template <typename TOut>
__device__ __forceinline__ uint2 pack4(float a, float b, float c, float d) {
    uint2 v;
    if constexpr (std::is_same<TOut, __nv_bfloat16>::value) {
        *reinterpret_cast<__nv_bfloat162 *>(&v.x) = __floats2bfloat162_rn(a, b);
        *reinterpret_cast<__nv_bfloat162 *>(&v.y) = __floats2bfloat162_rn(c, d);
    } else {
        *reinterpret_cast<__half2 *>(&v.x) = __floats2half2_rn(a, b);
        *reinterpret_cast<__half2 *>(&v.y) = __floats2half2_rn(c, d);
    }
    return v;
}

template <typename TOut>
__device__ __forceinline__ float4 unpack4(uint2 v) {
    float2 lo, hi;
    if constexpr (std::is_same<TOut, __nv_bfloat16>::value) {
        lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
        hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
    } else {
        lo = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
        hi = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
    }
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

template <typename TOut>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *part, int splits, int64_t count,
                                                            const TOut *res, TOut *out) {
    // the partials are the previous kernel's output; only once they are
    // complete may the kernel after this one start
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int64_t n4 = count / 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const float4 *p4 = reinterpret_cast<const float4 *>(part);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int sp = 0;
        for (; sp + 4 <= splits; sp += 4) {
            float4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) v[k] = __ldcs(p4 + (sp + k) * n4 + i);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc.x += v[k].x;
                acc.y += v[k].y;
                acc.z += v[k].z;
                acc.w += v[k].w;
            }
        }
        for (; sp < splits; ++sp) {
            const float4 v = __ldcs(p4 + sp * n4 + i);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        if (res) {
            const float4 r = unpack4<TOut>(reinterpret_cast<const uint2 *>(res)[i]);
            acc.x += r.x;
            acc.y += r.y;
            acc.z += r.z;
            acc.w += r.w;
        }
        reinterpret_cast<uint2 *>(out)[i] = pack4<TOut>(acc.x, acc.y, acc.z, acc.w);
    }
}

// The same sums a row per CTA, also writing the row's sum of squares of the
// stored values (fixed thread-to-column map and reduction tree: the same bits
// every run).  N is a multiple of 8.
template <typename TOut>
__global__ void __launch_bounds__(256) splitk_reduce_rows_kernel(const float *part, int splits, int64_t M, int64_t N,
                                                                 const TOut *res, TOut *out, float *ss_out) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    __shared__ float red[8];
    const int64_t row = blockIdx.x, n4 = N / 4, count4 = M * n4;
    const float4 *p4 = reinterpret_cast<const float4 *>(part);
    float ss = 0.f;
    for (int64_t c = threadIdx.x; c < n4; c += 256) {
        const int64_t i = row * n4 + c;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < splits; ++sp) {
            const float4 v = __ldcs(p4 + sp * count4 + i);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        if (res) {
            const float4 r = unpack4<TOut>(reinterpret_cast<const uint2 *>(res)[i]);
            acc.x += r.x;
            acc.y += r.y;
            acc.z += r.z;
            acc.w += r.w;
        }
        const uint2 pk = pack4<TOut>(acc.x, acc.y, acc.z, acc.w);
        reinterpret_cast<uint2 *>(out)[i] = pk;
        const float4 r = unpack4<TOut>(pk);
        ss = fmaf(r.x, r.x, ss);
        ss = fmaf(r.y, r.y, ss);
        ss = fmaf(r.z, r.z, ss);
        ss = fmaf(r.w, r.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += red[w];
        ss_out[row] = t;
    }
}

template <typename TOut>
cudaError_t launch_splitk_reduce(const float *part, int splits, int64_t count, const void *res, void *out,
                                 cudaStream_t s, int64_t M = 0, float *ss_out = nullptr) {
    if (ss_out) {
        LaunchScope scope(K_SPLITK_REDUCE, s);
        cudaError_t e = launch_dependent(splitk_reduce_rows_kernel<TOut>, dim3(static_cast<unsigned>(M)), dim3(256),
                                         0, s, part, splits, M, count / M, static_cast<const TOut *>(res),
                                         static_cast<TOut *>(out), ss_out);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int64_t n4 = count / 4;
    int64_t blocks = static_cast<int64_t>(sm_count()) * 8;
    const int64_t need = (n4 + 255) / 256;
    if (blocks > need) blocks = need;
    if (blocks < 1) return cudaSuccess;
    LaunchScope scope(K_SPLITK_REDUCE, s);
    cudaError_t e = launch_dependent(splitk_reduce_kernel<TOut>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                     s, part, splits, count, static_cast<const TOut *>(res),
                                     static_cast<TOut *>(out));
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int MODE, bool BF16, int A_TERMS>
cudaError_t launch_gateup_bn(const void *A, const void *A2, const void *B0, const void *B1, void *out0,
                             void *out1, int64_t M, int64_t K, int64_t N, float acc_scale, float out_scale,
                             GemmRowSS ex, cudaStream_t s) {
    if (gateup_width(M, N) == 192)
        return launch_impl<MODE, BF16, A_TERMS, BF16, 192>(A, A2, B0, B1, out0, out1, M, K, N, K_GEMM_GATEUP,
                                                           acc_scale, out_scale, s, nullptr, nullptr, 0, 1, ex);
    return launch_impl<MODE, BF16, A_TERMS, BF16, 256>(A, A2, B0, B1, out0, out1, M, K, N, K_GEMM_GATEUP,
                                                       acc_scale, out_scale, s, nullptr, nullptr, 0, 1, ex);
}

// One row block and a reduction too short to split: 64-wide tiles (d 4096:
// 64 CTAs instead of 16).
template <bool BF16, int A_TERMS, bool OUT_BF16>
cudaError_t launch_plain_bn(const void *A, const void *A_lo, const void *B, void *C, int64_t M, int64_t K,
                            int64_t N, float acc_scale, const void *res, float *part, GemmRowSS ex, cudaStream_t s) {
    using TOut = typename std::conditional<OUT_BF16, __nv_bfloat16, __half>::type;
    int per = 0, bn = 256;
    const int splits = plain_split_plan(M, K, N, A_TERMS, &per, &bn);
    if (splits > 1) {
        if (!part) return cudaErrorInvalidValue;
        cudaError_t e =
            bn == 192 ? launch_impl<MODE_PLAIN, BF16, A_TERMS, OUT_BF16, 192>(A, A_lo, B, nullptr, C, nullptr, M, K, N,
                                                                              K_GEMM_DOWN, acc_scale, 1.f, s, nullptr,
                                                                              part, per, splits)
                      : launch_impl<MODE_PLAIN, BF16, A_TERMS, OUT_BF16, 256>(A, A_lo, B, nullptr, C, nullptr, M, K, N,
                                                                              K_GEMM_DOWN, acc_scale, 1.f, s, nullptr,
                                                                              part, per, splits);
        if (e != cudaSuccess) return e;
        return launch_splitk_reduce<TOut>(part, splits, M * N, res, C, s, M, ex.out);
    }
    if (M <= BM)
        return launch_impl<MODE_PLAIN, BF16, A_TERMS, OUT_BF16, 64>(A, A_lo, B, nullptr, C, nullptr, M, K, N,
                                                                    K_GEMM_DOWN, acc_scale, 1.f, s, res, nullptr, 0,
                                                                    1, ex);
    if (tile_width(M, N) == 224)
        return launch_impl<MODE_PLAIN, BF16, A_TERMS, OUT_BF16, 224>(A, A_lo, B, nullptr, C, nullptr, M, K,
                                                                     N, K_GEMM_DOWN, acc_scale, 1.f, s, res, nullptr,
                                                                     0, 1, ex);
    return launch_impl<MODE_PLAIN, BF16, A_TERMS, OUT_BF16, 256>(A, A_lo, B, nullptr, C, nullptr, M, K, N,
                                                                 K_GEMM_DOWN, acc_scale, 1.f, s, res, nullptr, 0, 1,
                                                                 ex);
}

}  // namespace

// The largest partial-sum buffer any M' <= M needs, so that a workspace sized
// for a batch also serves every smaller one.  Splits only occur while the
// tiles fill less than half the SMs, and they are fixed per row-block count,
// so the maximum is over the first few row-block counts at their full rows.
size_t gemm_plain_partial_bytes(int64_t M, int64_t K, int64_t N, int a_terms) {
    size_t most = 0;
    for (int64_t mb = 1; mb <= (M + BM - 1) / BM; ++mb) {
        const int64_t rows = mb * BM < M ? mb * BM : M;
        const int splits = plain_split_plan(rows, K, N, a_terms, nullptr, nullptr);
        if (splits <= 1) {
            if (mb > 1) break;   // more row blocks, more tiles: no split from here on
            continue;
        }
        const size_t bytes = static_cast<size_t>(splits) * static_cast<size_t>(rows) * static_cast<size_t>(N) * 4;
        if (bytes > most) most = bytes;
    }
    return most;
}

cudaError_t launch_gemm_gateup(int dt, const void *A, const void *A_lo, const void *Wg,
                               const void *Wu, void *H, void *H_lo, void *G, void *U, int64_t M,
                               int64_t K, int64_t F, bool fused, float acc_scale, float out_scale,
                               cudaStream_t s, unsigned *zero, int nzero) {
    const bool bf = dt == DT_BF16;
    const float a = acc_scale, o = out_scale;
    GemmRowSS ex;
    ex.zero = zero;
    ex.nzero = nzero;
    if (A_lo) {
        if (fused)
            return bf ? launch_gateup_bn<MODE_GATEUP_FUSED, true, 2>(A, A_lo, Wg, Wu, H, H_lo, M, K, F, a, o, ex, s)
                      : launch_gateup_bn<MODE_GATEUP_FUSED, false, 2>(A, A_lo, Wg, Wu, H, H_lo, M, K, F, a, o, ex, s);
        return bf ? launch_gateup_bn<MODE_GATEUP_SPLIT, true, 2>(A, A_lo, Wg, Wu, G, U, M, K, F, a, o, ex, s)
                  : launch_gateup_bn<MODE_GATEUP_SPLIT, false, 2>(A, A_lo, Wg, Wu, G, U, M, K, F, a, o, ex, s);
    }
    if (fused)
        return bf ? launch_gateup_bn<MODE_GATEUP_FUSED, true, 1>(A, nullptr, Wg, Wu, H, H_lo, M, K, F, a, o, ex, s)
                  : launch_gateup_bn<MODE_GATEUP_FUSED, false, 1>(A, nullptr, Wg, Wu, H, H_lo, M, K, F, a, o, ex, s);
    return bf ? launch_gateup_bn<MODE_GATEUP_SPLIT, true, 1>(A, nullptr, Wg, Wu, G, U, M, K, F, a, o, ex, s)
              : launch_gateup_bn<MODE_GATEUP_SPLIT, false, 1>(A, nullptr, Wg, Wu, G, U, M, K, F, a, o, ex, s);
}

cudaError_t launch_gemm_plain(int dt, int dt_out, const void *A, const void *A_lo, const void *B,
                              void *C, int64_t M, int64_t K, int64_t N, float acc_scale,
                              const void *res, float *part, cudaStream_t s, float *ss_part,
                              unsigned *ss_ctr, float *ss_out) {
    const float a = acc_scale;
    GemmRowSS ex;
    ex.part = ss_part;
    ex.ctr = ss_ctr;
    ex.out = ss_out;
    if (dt == DT_BF16) {
        if (A_lo) return launch_plain_bn<true, 2, true>(A, A_lo, B, C, M, K, N, a, res, part, ex, s);
        return launch_plain_bn<true, 1, true>(A, nullptr, B, C, M, K, N, a, res, part, ex, s);
    }
    if (dt_out == DT_BF16) {   // fp16 operands, bf16 output (prepared-weights path)
        if (A_lo) return launch_plain_bn<false, 2, true>(A, A_lo, B, C, M, K, N, a, res, part, ex, s);
        return launch_plain_bn<false, 1, true>(A, nullptr, B, C, M, K, N, a, res, part, ex, s);
    }
    if (A_lo) return launch_plain_bn<false, 2, false>(A, A_lo, B, C, M, K, N, a, res, part, ex, s);
    return launch_plain_bn<false, 1, false>(A, nullptr, B, C, M, K, N, a, res, part, ex, s);
}

}  // namespace ffn
