// noalloc.cu -- the decode block with its scratch in library-owned device memory.
//
// ffn_block_forward needs a caller-provided workspace.  Some callers cannot
// provide one: a serving runtime that plans all device memory at start-up and
// forbids allocation once requests flow, a plugin that a host framework hands
// only its input and output buffers, or a latency-critical decode loop that
// must not call cudaMalloc (which can synchronise the device).  For them this
// file keeps the decode path's scratch in one file-scope device array.
//
// The array lives in every GPU that loads the library, for the life of the
// process.  Its size bounds the shapes this entry point accepts.  All calls
// share it and it keeps whatever the last call left there, so the kernels
// rewrite every byte they read before reading it and zero the split-K arrival
// counters at the start of each call.  Two calls that run at the same time on
// the GPU (different streams, or different host threads) race on the array.
#include <algorithm>

#include "../../include/ffn.h"
#include "ffn_internal.cuh"

namespace {

constexpr int64_t kStaticMaxRows = 16;
constexpr int64_t kStaticMaxD = 8192;
constexpr int64_t kStaticMaxFfn = 32768;
constexpr size_t kStaticScratchBytes = size_t(12) << 20;   // 12 MiB

}  // namespace

// Host code must never use this name as an address: on the host it is only a
// stand-in for the device symbol.  The device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

namespace {

// Device address of g_decode_scratch in the current device's context, looked
// up on every call.  The lookup allocates nothing and, once the module is
// loaded in a context, is a host-side table query; not caching it keeps the
// address right after cudaDeviceReset or a context rebuilt in the same
// process (the module is then loaded again, perhaps elsewhere) and needs no
// lock between host threads.  The first call in a context loads the module,
// so make it before any stream capture.
void *static_scratch(cudaError_t *err) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_decode_scratch);
    return *err == cudaSuccess ? p : nullptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return na && nb && a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace

extern "C" ffn_status ffn_block_forward_decode_static(const void *x, const void *g,
                                                      const void *w_gate, const void *w_up,
                                                      const void *w_down, void *y, int64_t rows,
                                                      int64_t d, int64_t ffn, float eps,
                                                      ffn_dtype dtype, void *stream) {
    if (!g || !w_gate || !w_up || !w_down || (rows != 0 && (!x || !y))) return FFN_ERR_NULL;
    if (dtype != FFN_F16 && dtype != FFN_BF16) return FFN_ERR_DTYPE;
    if (rows < 0 || d < 1 || ffn < 1 || d % 8 || ffn % 8) return FFN_ERR_SHAPE;
    if (rows > kStaticMaxRows || d > kStaticMaxD || ffn > kStaticMaxFfn) return FFN_ERR_SHAPE;
    // same operand precision as ffn_block_forward's defaults: bf16 activations
    // enter the tensor ops as hi + lo terms, fp16 as one rounding
    const bool two = dtype == FFN_BF16;
    const int64_t grp = std::max<int64_t>(rows, 1);
    if (ffn::gemv_workspace_bytes(grp, d, ffn, two) > kStaticScratchBytes) return FFN_ERR_SHAPE;
    const void *ptrs[] = {x, g, w_gate, w_up, w_down, y};
    for (const void *p : ptrs)
        if (!aligned16(p)) return FFN_ERR_ALIGN;
    const size_t act = static_cast<size_t>(rows) * d * 2, wb = static_cast<size_t>(ffn) * d * 2;
    if (overlaps(y, act, x, act) || overlaps(y, act, g, static_cast<size_t>(d) * 2) ||
        overlaps(y, act, w_gate, wb) || overlaps(y, act, w_up, wb) || overlaps(y, act, w_down, wb))
        return FFN_ERR_ALIAS;
    if (rows == 0) return FFN_OK;

    cudaError_t e = cudaSuccess;
    void *scratch = static_scratch(&e);
    if (!scratch) return FFN_ERR_CUDA;
    ffn::GemvWorkspace ws;
    ffn::gemv_carve(scratch, rows, d, ffn, two, &ws);
    ffn::GemvWeights a{w_gate, nullptr, nullptr}, b{w_up, nullptr, nullptr}, c{w_down, nullptr, nullptr};
    e = ffn::launch_gemv_block(dtype == FFN_BF16 ? 1 : 0, x, g, a, b, c, y, rows, d, ffn, eps, ws,
                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FFN_OK : FFN_ERR_CUDA;
}
