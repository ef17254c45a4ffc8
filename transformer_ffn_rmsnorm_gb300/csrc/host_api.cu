// host_api.cu -- the FFN block with x and y in host memory.
//
// ffn_block_forward_host copies x in, runs the block and copies y out, with
// the copies overlapped with the compute: the rows are split into chunks;
// every chunk's host-to-device copy is queued at once on a copy stream of the
// library's own, each chunk's block runs on the caller's stream as soon as its
// rows have landed, and its device-to-host copy runs on a second copy stream
// while the next chunk computes.  The caller's stream finally waits for the
// last copy, so synchronising that stream means y is in host memory.  The
// staging buffers come in two sets used by consecutive calls in turn, so one
// call's input copies run while the call before it still computes.
//
// With calls back to back, every input copy runs while the call before
// computes, and only the last chunk's output copy is exposed (the host link
// of a GB300 moves about 200 GB/s each way for page-locked memory, 160 GB/s
// each way when both directions run).  Each chunk's GEMMs pay a ramp, a
// drain and a partly filled last wave, so few, long chunks compute fastest;
// the last one is short because its output copy is exposed.  Measured on
// 4096 x 4096 -> 11008 (prepared weights, burst clocks), calls back to back,
// x and y on the host (in brackets the same chunks computed from device
// memory):
//   3072, 1024                 722 us (646-654 us)
//   1024, 2048, 1024           766 us (689 us)
//   3584, 512                  753-765 us;  2048, 2048  793-805 us
//   2048, 1024, 1024           781-819 us;  3072, 512, 512  787-838 us
// A single call, with nothing before it to overlap, also pays the first
// chunk's input copy (3072 rows: ~125 us).
#include <cstring>
#include <mutex>

#include "../../include/ffn.h"
#include "ffn_internal.cuh"

namespace ffn {
namespace {

constexpr int kMaxChunks = 16;
constexpr int kMaxDevices = 64;

struct Chunks {
    int64_t start[kMaxChunks + 1];   // chunk i holds rows start[i] .. start[i+1]-1
    int count;
    int64_t rows(int i) const { return start[i + 1] - start[i]; }
};

// A last chunk of kLastRows (its output copy is the one exposed), the rows
// before it in near-equal chunks of at most kFrontRows (multiples of 256),
// at most kMaxChunks in all.
constexpr int64_t kLastRows = 1024, kFrontRows = 4096;
Chunks plan_chunks(int64_t rows) {
    Chunks c;
    c.count = 0;
    c.start[0] = 0;
    if (rows <= 0) return c;
    auto push = [&](int64_t n) {
        c.start[c.count + 1] = c.start[c.count] + n;
        ++c.count;
    };
    if (rows <= kLastRows) {
        push(rows);
        return c;
    }
    const int64_t front = rows - kLastRows;
    int64_t pieces = (front + kFrontRows - 1) / kFrontRows;
    if (pieces > kMaxChunks - 1) pieces = kMaxChunks - 1;
    const int64_t each = ((front + pieces - 1) / pieces + 255) / 256 * 256;
    for (int64_t left = front; left > 0; left -= each) push(left < each ? left : each);
    push(kLastRows);
    return c;
}

int64_t elem_bytes(ffn_dtype dt) { return dt == FFN_F32 ? 4 : 2; }
size_t align256(size_t v) { return (v + 255) & ~size_t{255}; }

// The workspace holds two sets of x and y staging buffers, used by calls in
// turn, and the block's scratch (sized for the largest chunk).
struct Layout {
    size_t x_stage, y_stage, block, total;   // byte sizes of one x and one y staging buffer, scratch, all
};

ffn_status layout(int64_t rows, int64_t d, int64_t ffn, ffn_dtype dt, uint32_t flags, Layout *l) {
    const Chunks c = plan_chunks(rows);
    size_t block = 0;
    if (c.count > 0) {
        for (int i = 0; i < c.count; ++i) {
            size_t a = 0;
            ffn_status st = ffn_block_workspace_bytes(c.rows(i), d, ffn, dt, flags, &a);
            if (st != FFN_OK) return st;
            if (a > block) block = a;
        }
    } else {
        size_t a = 0;
        ffn_status st = ffn_block_workspace_bytes(0, d, ffn, dt, flags, &a);
        if (st != FFN_OK) return st;
    }
    l->x_stage = align256(static_cast<size_t>(rows) * d * elem_bytes(dt));
    l->y_stage = l->x_stage;
    l->block = align256(block);
    l->total = 2 * (l->x_stage + l->y_stage) + l->block;
    return FFN_OK;
}

// Copy streams and events of one device, created on first use and kept for
// the life of the process.
// Calls alternate between the two staging sets: a call's input copies wait
// only until the call before the previous one has finished computing from
// that set's x (x_free), and its compute until that call's output copies
// have drained that set's y (y_free), so the input copies of a call overlap
// the compute of the call before it.
struct Pipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t landed[kMaxChunks] = {}, computed[kMaxChunks] = {};
    cudaEvent_t x_free[2] = {}, y_free[2] = {};
    int next = 0;   // staging set of the next call
    bool ready = false;
};
std::mutex g_pipe_mu;
Pipe g_pipes[kMaxDevices];

bool make_pipe(Pipe &p) {
    if (p.ready) return true;
    const unsigned ev = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) != cudaSuccess) return false;
    for (int b = 0; b < 2; ++b) {
        if (cudaEventCreateWithFlags(&p.x_free[b], ev) != cudaSuccess) return false;
        if (cudaEventCreateWithFlags(&p.y_free[b], ev) != cudaSuccess) return false;
    }
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

    const int b = p.next;
    char *ws = static_cast<char *>(workspace);
    char *x_dev = ws + b * (l.x_stage + l.y_stage), *y_dev = x_dev + l.x_stage;
    char *block_ws = ws + 2 * (l.x_stage + l.y_stage);
    const char *xh = static_cast<const char *>(x_host);
    char *yh = static_cast<char *>(y_host);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Chunks c = plan_chunks(rows);

    // A call that fails part way has queued some copies and blocks on this
    // staging set.  Its free events are then re-recorded behind everything
    // queued so far (s after h2d, d2h after s), and the set is not handed on,
    // so the next call on it waits for this one's work before overwriting
    // the buffers.  Best effort: the error being reported comes first.
    auto fail = [&](ffn_status why) {
        if (cudaEventRecord(p.landed[0], p.h2d) == cudaSuccess) cudaStreamWaitEvent(s, p.landed[0], 0);
        cudaEventRecord(p.x_free[b], s);
        if (cudaEventRecord(p.computed[0], s) == cudaSuccess) cudaStreamWaitEvent(p.d2h, p.computed[0], 0);
        cudaEventRecord(p.y_free[b], p.d2h);
        return why;
    };

    // this staging set's x may still be read, and its y still be copied out,
    // by the call before the previous one
    if (cudaStreamWaitEvent(p.h2d, p.x_free[b], 0) != cudaSuccess) return FFN_ERR_CUDA;
    if (cudaStreamWaitEvent(s, p.y_free[b], 0) != cudaSuccess) return FFN_ERR_CUDA;
    for (int i = 0; i < c.count; ++i) {
        const int64_t r0 = c.start[i], nr = c.rows(i);
        if (cudaMemcpyAsync(x_dev + r0 * row_bytes, xh + r0 * row_bytes, nr * row_bytes, cudaMemcpyHostToDevice,
                            p.h2d) != cudaSuccess)
            return fail(FFN_ERR_CUDA);
        if (cudaEventRecord(p.landed[i], p.h2d) != cudaSuccess) return fail(FFN_ERR_CUDA);
    }
    for (int i = 0; i < c.count; ++i) {
        const int64_t r0 = c.start[i], nr = c.rows(i);
        if (cudaStreamWaitEvent(s, p.landed[i], 0) != cudaSuccess) return fail(FFN_ERR_CUDA);
        st = ffn_block_forward(x_dev + r0 * row_bytes, g, w_gate, w_up, w_down, y_dev + r0 * row_bytes, nr, d, ffn,
                               eps, dtype, flags, block_ws, l.block, stream);
        if (st != FFN_OK) return fail(st);
        if (cudaEventRecord(p.computed[i], s) != cudaSuccess) return fail(FFN_ERR_CUDA);
        if (cudaStreamWaitEvent(p.d2h, p.computed[i], 0) != cudaSuccess) return fail(FFN_ERR_CUDA);
        if (cudaMemcpyAsync(yh + r0 * row_bytes, y_dev + r0 * row_bytes, nr * row_bytes, cudaMemcpyDeviceToHost,
                            p.d2h) != cudaSuccess)
            return fail(FFN_ERR_CUDA);
    }
    if (cudaEventRecord(p.x_free[b], s) != cudaSuccess) return fail(FFN_ERR_CUDA);
    if (cudaEventRecord(p.y_free[b], p.d2h) != cudaSuccess) return fail(FFN_ERR_CUDA);
    if (cudaStreamWaitEvent(s, p.y_free[b], 0) != cudaSuccess) return fail(FFN_ERR_CUDA);
    p.next = b ^ 1;   // the next call uses the other staging set
    return FFN_OK;
}

}  // extern "C"
