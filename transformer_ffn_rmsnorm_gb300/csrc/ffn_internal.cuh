// ffn_internal.cuh -- shared declarations of the sm_103a kernels behind include/ffn.h.
//
// Everything here is internal: launchers return cudaError_t and assume the
// C-ABI layer (api.cu) has validated their arguments.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ffn {

enum DType : int { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };

// Kernel kinds, for launch counting and event timing.
enum KernelKind : int {
    K_PREPARE = 0,
    K_RMSNORM,
    K_SWIGLU,
    K_SIMT_GATEUP,
    K_SIMT_DOWN,
    K_GEMV_NORM,
    K_GEMV_GATEUP,
    K_GEMV_DOWN,
    K_GEMM_GATEUP,
    K_GEMM_DOWN,
    K_SELFTEST,
    K_SPLITK_REDUCE,
    K_GEMV_FUSED,
    K_NUM_KINDS
};
const char *kernel_name(int kind);

// Brackets one launch: counts it and, when timing is on, records events on
// the launch stream around it.
struct LaunchScope {
    int kind;
    cudaStream_t stream;
    void *ev0;
    LaunchScope(int kind, cudaStream_t s);
    ~LaunchScope();
};

// Launches kern<<<grid, block, smem, s>>>(args...) allowed to overlap the
// tail of the kernel before it on s (programmatic stream serialization); the
// kernel must call ptx::griddep_wait() before touching that kernel's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Device status word bits (bounded waits that gave up; weights out of range).
enum : unsigned { DEVERR_TIMEOUT = 1u, DEVERR_RANGE = 2u };

// Prepared weights are fp16 values of w * 2^8 (exact for 2^-25 <= |w| < 256).
constexpr float kPreparedScale = 256.0f;
unsigned *device_status_word();   // device address, for the current device
int sm_count();                   // multiprocessors on the current device

// ---------------------------------------------------------------- launchers
// ss_in (optional): each row's sum of squares of x, used instead of reducing
// the row (the block before handed it on).
cudaError_t launch_rmsnorm(const void *x, const void *g, void *n, int64_t rows, int64_t d,
                           float eps, int dt, cudaStream_t s, const float *ss_in = nullptr);
// As launch_rmsnorm, for 16-bit storage, also writing the rounding residual:
// n_hi = round(v), n_lo = round(v - n_hi), so n_hi + n_lo carries ~16 bits.
cudaError_t launch_rmsnorm_split(const void *x, const void *g, void *n_hi, void *n_lo,
                                 int64_t rows, int64_t d, float eps, int dt, cudaStream_t s,
                                 const float *ss_in = nullptr);
// 16-bit x and g of type dt_in, n written as fp16 (operand of fp16 tensor ops).
cudaError_t launch_rmsnorm_to_f16(const void *x, const void *g, void *n, int64_t rows, int64_t d,
                                  float eps, int dt_in, cudaStream_t s, const float *ss_in = nullptr);
// dst[i] = fp16(src[i] * 2^8) for 16-bit src of type dt; out-of-range values
// set DEVERR_RANGE in the device status word.
cudaError_t launch_prepare_weights(const void *src, void *dst, int64_t count, int dt, cudaStream_t s);
// fp16(w * 2^8) from e4m3 codes with row scales / from Q4 in the device layout
cudaError_t launch_prepare_fp8(const uint8_t *codes, const float *scales, void *dst, int64_t rows, int64_t cols,
                               cudaStream_t s);
cudaError_t launch_prepare_q4(const uint8_t *qs, const uint16_t *scales, void *dst, int64_t rows, int64_t cols,
                              cudaStream_t s);
cudaError_t launch_prepare_q8(const int8_t *codes, const uint16_t *scales, void *dst, int64_t rows, int64_t cols,
                              cudaStream_t s);
cudaError_t launch_swiglu(const void *gate, const void *up, void *h, int64_t count, int dt,
                          cudaStream_t s);
// One CTA whose bounded wait on a never-completed barrier gives up after
// limit_ns and records DEVERR_TIMEOUT (selftest.cu).
cudaError_t launch_bounded_wait_probe(uint64_t limit_ns, cudaStream_t s);

// fp32 G, U -> 16-bit h = silu(G) * U * out_scale, and its residual h_lo
// when non-null (unfused arm of the tensor-core path)
cudaError_t launch_swiglu_f32in(const float *gate, const float *up, void *h, void *h_lo,
                                int64_t count, int dt, float out_scale, cudaStream_t s);

// fp32 SIMT block: n (rows x d) and h (rows x ffn) are fp32 scratch.
cudaError_t launch_simt_block(const float *x, const float *g, const float *wg, const float *wu,
                              const float *wd, float *y, int64_t rows, int64_t d, int64_t ffn,
                              float eps, float *n, float *h, cudaStream_t s,
                              const float *res = nullptr, const float *ss_in = nullptr, float *ss_out = nullptr);

// Decode (weight-streaming) block for rows <= 16.
struct GemvWorkspace {
    void *nfrag;        // normalised activations in mma B-fragment order
    void *hfrag;        // hidden activations in mma B-fragment order
    void *nfrag_lo;     // their rounding residuals (two-term operands), or null
    void *hfrag_lo;
    float *partials;    // [splits][rows][d] fp32
    unsigned *counters; // [d / 64] arrival counters, then one for the rows' sums of squares
    float *ss_part;     // [d / 64][rows] parts of the rows' sums of squares of y
    float *ncorr;       // Q4 streaming kernels: block offsets of n and of h
    float *hcorr;
};
// The block's RMSNorm reduction handed from one block to the next: ss_in (or
// null) holds each row's sum of squares of x, used instead of reducing the
// row; ss_out (or null) receives each row's sum of squares of the stored y.
struct RowStats {
    const float *ss_in = nullptr;
    float *ss_out = nullptr;
};
size_t gemv_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, bool two_terms);
void gemv_carve(void *base, int64_t rows, int64_t d, int64_t ffn, bool two_terms, GemvWorkspace *ws);
// wfmt: 0 f16, 1 bf16, 2 q4 (bf16 x/y, fp16 operands), 3 prepared fp16 weights
// (bf16 x/y, fp16 operands), 4 e4m3 weights with per-row scales (bf16 x/y,
// fp16 operands), 5 Q8_0 (int8 codes, fp16 scale per 32; bf16 x/y, fp16
// operands)
enum { WF_F16 = 0, WF_BF16 = 1, WF_Q4 = 2, WF_F16P = 3, WF_FP8 = 4, WF_Q8 = 5 };
struct GemvWeights {
    const void *w;          // f16/bf16 [out x in]; e4m3 or int8 codes [out x in]
    const uint8_t *qs;      // q4 device layout
    const uint16_t *sc;     // q4 / Q8_0 block scales [out x in/32]
    const float *rs;        // e4m3: float scale of each output row [out]
};
// one_kernel: the whole block as one persistent kernel where the streaming
// kernels run (FFN_DECODE_ONE_KERNEL), else the norm, gate/up and down kernels.
cudaError_t launch_gemv_block(int wfmt, const void *x, const void *g, GemvWeights wg,
                              GemvWeights wu, GemvWeights wd, void *y, int64_t rows, int64_t d,
                              int64_t ffn, float eps, const GemvWorkspace &ws, cudaStream_t s,
                              const void *res = nullptr, RowStats rs = {}, bool one_kernel = false);

// A 2D tiled TMA descriptor over a row-major array of `rows` rows, `inner`
// elements a row, rows `row_bytes` apart; boxes of box_inner x box_rows.
bool encode_tma_2d(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, int64_t inner,
                   int64_t rows, int64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle);

// Prefill tensor-core GEMMs (tcgen05 + TMEM + TMA).
//   gate/up: A = n [M x K] (plus its residual A_lo, or nullptr), B = W_gate,
//            W_up [F x K]; G, U = accumulator * acc_scale;
//            fused -> h = silu(G) U out_scale [M x F] (plus residual H_lo if
//            non-null); unfused -> G, U [M x F] fp32 each
//   down:    A = h [M x F] (plus residual A_lo, or nullptr), B = W_down [N x F]
//            -> C = accumulator * acc_scale [M x N] stored as dt_out
// dt: the operand type (bf16 or fp16); h has the operand type.
// zero, nzero: counters the down projection of the same call uses, zeroed
// once the kernel before this one has completed.
cudaError_t launch_gemm_gateup(int dt, const void *A, const void *A_lo, const void *Wg,
                               const void *Wu, void *H, void *H_lo, void *G, void *U, int64_t M,
                               int64_t K, int64_t F, bool fused, float acc_scale, float out_scale,
                               cudaStream_t s, unsigned *zero = nullptr, int nzero = 0);
// res (optional): added to C before its one rounding (same type and layout as C).
// part: fp32 scratch of gemm_plain_partial_bytes(M, K, N, A_lo ? 2 : 1) bytes
// (16-byte aligned) for the split-K partial sums of short, wide-K products;
// may be null when that size is 0.  That size never decreases with M.
// ss_out (optional): each row's sum of squares of the stored C, through
// ss_part [ceil(N / 64)][M] fp32 and ss_ctr [ceil(M / 128)] counters (zero
// when the GEMM starts) -- or, when the reduction is split, by the kernel
// that adds the splits.
cudaError_t launch_gemm_plain(int dt, int dt_out, const void *A, const void *A_lo, const void *B,
                              void *C, int64_t M, int64_t K, int64_t N, float acc_scale,
                              const void *res, float *part, cudaStream_t s, float *ss_part = nullptr,
                              unsigned *ss_ctr = nullptr, float *ss_out = nullptr);
size_t gemm_plain_partial_bytes(int64_t M, int64_t K, int64_t N, int a_terms);

}  // namespace ffn

// ====================================================================== PTX
// Thin wrappers over inline PTX used by the kernels.
namespace ffn {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Suspends the thread until the phase completes or about 1 ms has passed
// (the hint), so waiting warps leave their scheduler's issue slots to the
// warps that work: on the GEMM's MMA thread the barrier polls of the other
// roles had cost 5-7 % of tensor throughput.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000000;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase of parity `parity` to complete.  Gives up (returns
// false) after `limit_ns` of wall time or as soon as *abort is non-zero.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ---- programmatic dependent launch
// A kernel launched with launch_dependent() may start while the kernel before
// it on the stream is still running.  Before griddep_wait() it may only read
// what no earlier kernel of the stream writes (weights, its own shared
// memory); griddep_wait() returns once the earlier kernel has completed and
// its writes are visible.  griddep_launch_dependents() lets the next such
// kernel start once every CTA of this grid has issued it (or exited).  Both
// are no-ops when there is no programmatic dependency.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- TMA
__device__ __forceinline__ void tma_prefetch_map(const void *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// L2 eviction priority for data that later loads of the same kernel re-read.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void *map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster: release this CTA's prior shared
// memory writes (barrier initialisation included) to the others, acquire theirs.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// ---- CTA pairs (tcgen05 .cta_group::2: one MMA over the tensor cores of two SMs)
// A kernel uses either these forms or the .cta_group::1 ones, never both.
// The copy lands in this CTA's shared memory; its complete_tx goes to the
// mbarrier at bar, a shared::cluster address in this CTA or its peer.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const void *map, uint32_t bar, int x, int y,
                                                      uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
        : "memory");
}
// One warp of each CTA of the pair executes these together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Issued by one thread of the even CTA: D (rows 0-127 in this CTA's TMEM,
// 128-255 in the peer's) (+)= A (rows 0-127 from this CTA's shared memory,
// 128-255 from the peer's, same offsets) * B^T (columns 0..N/2-1 from this
// CTA, N/2..N-1 from the peer).
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives on the mbarrier at offset bar of every CTA in cta_mask once the
// pair MMAs issued so far have completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, uint32_t bar, int x,
                                            int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// 1-D bulk copy global -> shared, completing bytes on an mbarrier (both
// addresses and the size multiples of 16 bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// ---- tcgen05 (cta_group::1)
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 or fp16 inputs, fp32 accumulate)
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread t gets lane (base lane + t)
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// Loads CW (16 or 32) consecutive columns of this warp's 32 TMEM lanes.
template <int CW>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[CW]) {
    static_assert(CW == 16 || CW == 32, "tcgen05.ld width");
    if constexpr (CW == 32) tmem_ld_32x32b_x32(taddr, r);
    else tmem_ld_32x32b_x16(taddr, r);
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major tile written by TMA with
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
    return d;
}
// Instruction descriptor, kind::f16: fp32 accumulate, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---- warp-level mma (m16n8k16, fp32 accumulate); pure functions of their
// operands (no volatile), so the compiler may interleave them with the
// dequantisation around them
template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (BF16) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// d += a * b on tf32 operands, m16n8k8: a0 (row g, k t), a1 (row g + 8, k t),
// a2 (row g, k t + 4), a3 (row g + 8, k t + 4); b0 (k t, column g), b1 (k t
// + 4, column g); d as for m16n8k16 (g = lane / 4, t = lane % 4).
__device__ __forceinline__ void mma_1688_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp32 rounded to tf32 (10 fraction bits, nearest, ties away), as fp32 bits
__device__ __forceinline__ float round_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// d = a * b (a zero accumulator that the compiler need not materialise in
// registers: C is an input-only zero)
template <bool BF16>
__device__ __forceinline__ void mma_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (BF16) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
    }
}

// ---- streaming global loads
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

}  // namespace ptx

// ------------------------------------------------------------ conversions
template <int DT> struct Storage;
template <> struct Storage<DT_F32> { using T = float; };
template <> struct Storage<DT_F16> { using T = __half; };
template <> struct Storage<DT_BF16> { using T = __nv_bfloat16; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// 16 bytes <-> floats (paired conversions for the 16-bit types)
template <typename T> struct Vec16 {
    static constexpr int N = 16 / sizeof(T);
    __device__ static __forceinline__ void unpack(const uint4 &v, float (&f)[16 / sizeof(T)]) {
        const T *e = reinterpret_cast<const T *>(&v);
#pragma unroll
        for (int i = 0; i < N; ++i) f[i] = to_f32(e[i]);
    }
    __device__ static __forceinline__ uint4 pack(const float (&f)[16 / sizeof(T)]) {
        uint4 v;
        T *e = reinterpret_cast<T *>(&v);
#pragma unroll
        for (int i = 0; i < N; ++i) e[i] = from_f32<T>(f[i]);
        return v;
    }
};
template <> struct Vec16<__half> {
    static constexpr int N = 8;
    __device__ static __forceinline__ void unpack(const uint4 &v, float (&f)[8]) {
        const __half2 *e = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __half22float2(e[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    __device__ static __forceinline__ uint4 pack(const float (&f)[8]) {
        uint4 v;
        __half2 *e = reinterpret_cast<__half2 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) e[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        return v;
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static __forceinline__ void unpack(const uint4 &v, float (&f)[8]) {
        const __nv_bfloat162 *e = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __bfloat1622float2(e[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    __device__ static __forceinline__ uint4 pack(const float (&f)[8]) {
        uint4 v;
        __nv_bfloat162 *e = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) e[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        return v;
    }
};

// silu(z) = z / (1 + exp(-z)) in fp32, as z times the correctly rounded
// reciprocal of 1 + exp(-z) (within 1.5 ulp of the quotient; the limit 0 for
// very negative z comes out of exp overflowing to +inf).  Not the IEEE
// division: its quotient routine leaves the fast path for some operands, a
// zero numerator among them, and rows of zeros (the copy engine's fill past
// the end of a batch that is not a whole number of tiles, or padding tokens)
// then made the fused gate/up epilogue the bottleneck of its GEMM: 15-20 %
// slower gate/up on 320-448-row batches onto 14336 features.
__device__ __forceinline__ float silu_f32(float z) { return z * __frcp_rn(1.0f + __expf(-z)); }

}  // namespace ffn
