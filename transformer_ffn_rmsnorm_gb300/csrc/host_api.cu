// host_api.cu -- the FFN block with x and y in host memory.
//
// ffn_block_forward_host copies x in, runs the block and copies y out, with
// the copies overlapped with the compute: the rows are split into chunks;
// every chunk's host-to-device copy is queued at once on a copy stream of the
// library's own, each chunk's block runs on the caller's stream as soon as its
// rows have landed, and its device-to-host copy runs on a second copy stream
// while the next chunk computes.  The caller's stream finally waits for the
// last copy, so synchronising that stream means y is in host memory.  Only
// the first chunk's input copy and the last chunk's output copy are exposed.
//
// Chunks are 1024 rows for batches above 1024 rows.  On the host link of a
// GB300 (about 200 GB/s each way for page-locked memory) the exposed copies
// are the first chunk's input and the last chunk's output, so chunks should
// be short; but each chunk's GEMMs run in whole waves of 76 CTA pairs.  At
// 1024 rows (4 pairs of 128-row blocks) the down projection of d = 4096 is
// exactly one wave (4 x 19 tiles of 224 columns) and gate/up (ffn 11008, 4 x
// 86 tile pairs) fills 4.5 of 5 waves; 1536-row chunks fill gate/up better
// (6.8 of 7) but leave the down projection's second wave half empty, and
// cost 50 % more exposed copy time.
#include <cstring>
#include <mutex>

#include "../../include/ffn.h"
#include "ffn_internal.cuh"

namespace ffn {
namespace {

constexpr int kMaxChunks = 16;
constexpr int kMaxDevices = 64;

struct Chunks {
    int64_t rows;    // rows per chunk (the last may be fewer)
    int count;
};

Chunks plan_chunks(int64_t rows) {
    Chunks c;
    if (rows <= 1024) {
        c.rows = rows;
        c.count = rows > 0 ? 1 : 0;
        return c;
    }
    c.rows = 1024;
    if ((rows + c.rows - 1) / c.rows > kMaxChunks) c.rows = ((rows + kMaxChunks - 1) / kMaxChunks + 255) / 256 * 256;
    c.count = static_cast<int>((rows + c.rows - 1) / c.rows);
    return c;
}

int64_t elem_bytes(ffn_dtype dt) { return dt == FFN_F32 ? 4 : 2; }
size_t align256(size_t v) { return (v + 255) & ~size_t{255}; }

struct Layout {
    size_t x_stage, y_stage, block, total;   // byte sizes; block = scratch of the largest chunk
};

ffn_status layout(int64_t rows, int64_t d, int64_t ffn, ffn_dtype dt, uint32_t flags, Layout *l) {
    const Chunks c = plan_chunks(rows);
    size_t block = 0;
    if (c.count > 0) {
        size_t a = 0, b = 0;
        ffn_status st = ffn_block_workspace_bytes(c.rows, d, ffn, dt, flags, &a);
        if (st != FFN_OK) return st;
        const int64_t last = rows - c.rows * (c.count - 1);
        st = ffn_block_workspace_bytes(last, d, ffn, dt, flags, &b);
        if (st != FFN_OK) return st;
        block = a > b ? a : b;
    } else {
        size_t a = 0;
        ffn_status st = ffn_block_workspace_bytes(0, d, ffn, dt, flags, &a);
        if (st != FFN_OK) return st;
    }
    l->x_stage = align256(static_cast<size_t>(rows) * d * elem_bytes(dt));
    l->y_stage = l->x_stage;
    l->block = align256(block);
    l->total = l->x_stage + l->y_stage + l->block;
    return FFN_OK;
}

// Copy streams and events of one device, created on first use and kept for
// the life of the process.
struct Pipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, end = nullptr, landed[kMaxChunks] = {}, computed[kMaxChunks] = {};
    bool ready = false;
};
std::mutex g_pipe_mu;
Pipe g_pipes[kMaxDevices];

bool make_pipe(Pipe &p) {
    if (p.ready) return true;
    const unsigned ev = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&p.start, ev) != cudaSuccess) return false;
    if (cudaEventCreateWithFlags(&p.end, ev) != cudaSuccess) return false;
    for (int i = 0; i < kMaxChunks; ++i) {
        if (cudaEventCreateWithFlags(&p.landed[i], ev) != cudaSuccess) return false;
        if (cudaEventCreateWithFlags(&p.computed[i], ev) != cudaSuccess) return false;
    }
    p.ready = true;
    return true;
}

}  // namespace
}  // namespace ffn

extern "C" {

ffn_status ffn_block_host_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, ffn_dtype dtype, uint32_t flags,
                                          size_t *bytes) {
    if (!bytes) return FFN_ERR_NULL;
    ffn::Layout l;
    ffn_status st = ffn::layout(rows, d, ffn, dtype, flags, &l);
    if (st != FFN_OK) return st;
    *bytes = rows == 0 ? 0 : l.total;
    return FFN_OK;
}

ffn_status ffn_block_forward_host(const void *x_host, const void *g, const void *w_gate, const void *w_up,
                                  const void *w_down, void *y_host, int64_t rows, int64_t d, int64_t ffn,
                                  float eps, ffn_dtype dtype, uint32_t flags, void *workspace,
                                  size_t workspace_bytes, void *stream) {
    using namespace ffn;
    if (!g || !w_gate || !w_up || !w_down || (rows != 0 && (!x_host || !y_host))) return FFN_ERR_NULL;
    Layout l;
    ffn_status st = layout(rows, d, ffn, dtype, flags, &l);
    if (st != FFN_OK) return st;
    if (rows == 0) return FFN_OK;
    if (!workspace || workspace_bytes < l.total) return FFN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return FFN_ERR_ALIGN;
    const int64_t row_bytes = d * elem_bytes(dtype);
    {
        const uintptr_t xa = reinterpret_cast<uintptr_t>(x_host), ya = reinterpret_cast<uintptr_t>(y_host);
        const uintptr_t n = static_cast<uintptr_t>(rows * row_bytes);
        if (xa < ya + n && ya < xa + n) return FFN_ERR_ALIAS;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FFN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_pipe_mu);   // the events are shared by calls on this device
    Pipe &p = g_pipes[dev];
    if (!make_pipe(p)) return FFN_ERR_CUDA;

    char *ws = static_cast<char *>(workspace);
    char *x_dev = ws, *y_dev = ws + l.x_stage, *block_ws = ws + l.x_stage + l.y_stage;
    const char *xh = static_cast<const char *>(x_host);
    char *yh = static_cast<char *>(y_host);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Chunks c = plan_chunks(rows);

    // the staging buffers may still be in use by work queued before this call
    if (cudaEventRecord(p.start, s) != cudaSuccess) return FFN_ERR_CUDA;
    if (cudaStreamWaitEvent(p.h2d, p.start, 0) != cudaSuccess) return FFN_ERR_CUDA;
    if (cudaStreamWaitEvent(p.d2h, p.start, 0) != cudaSuccess) return FFN_ERR_CUDA;
    for (int i = 0; i < c.count; ++i) {
        const int64_t r0 = c.rows * i, nr = (i + 1 < c.count) ? c.rows : rows - r0;
        if (cudaMemcpyAsync(x_dev + r0 * row_bytes, xh + r0 * row_bytes, nr * row_bytes, cudaMemcpyHostToDevice,
                            p.h2d) != cudaSuccess)
            return FFN_ERR_CUDA;
        if (cudaEventRecord(p.landed[i], p.h2d) != cudaSuccess) return FFN_ERR_CUDA;
    }
    for (int i = 0; i < c.count; ++i) {
        const int64_t r0 = c.rows * i, nr = (i + 1 < c.count) ? c.rows : rows - r0;
        if (cudaStreamWaitEvent(s, p.landed[i], 0) != cudaSuccess) return FFN_ERR_CUDA;
        st = ffn_block_forward(x_dev + r0 * row_bytes, g, w_gate, w_up, w_down, y_dev + r0 * row_bytes, nr, d, ffn,
                               eps, dtype, flags, block_ws, l.block, stream);
        if (st != FFN_OK) return st;
        if (cudaEventRecord(p.computed[i], s) != cudaSuccess) return FFN_ERR_CUDA;
        if (cudaStreamWaitEvent(p.d2h, p.computed[i], 0) != cudaSuccess) return FFN_ERR_CUDA;
        if (cudaMemcpyAsync(yh + r0 * row_bytes, y_dev + r0 * row_bytes, nr * row_bytes, cudaMemcpyDeviceToHost,
                            p.d2h) != cudaSuccess)
            return FFN_ERR_CUDA;
    }
    if (cudaEventRecord(p.end, p.d2h) != cudaSuccess) return FFN_ERR_CUDA;
    if (cudaStreamWaitEvent(s, p.end, 0) != cudaSuccess) return FFN_ERR_CUDA;
    return FFN_OK;
}

}  // extern "C"
