// api.cu -- the extern "C" boundary declared in include/ffn.h.
//
// Host-side validation happens before any CUDA call; a rejected call launches
// nothing.  Path choice for ffn_block_forward:
//   fp32                      -> SIMT FFMA kernels (TF32 cannot meet 1e-4*rms)
//   fp16/bf16, rows <= 16     -> weight-streaming decode kernels (gemv.cu)
//   fp16/bf16, rows >  16     -> RMSNorm + tcgen05 gate/up GEMM + tcgen05 down GEMM
// Operands of the tensor ops: bf16 activations enter as hi + lo terms unless
// FFN_ACT_SINGLE; with FFN_PREPARED_WEIGHTS everything runs on fp16 operands
// (weights re-encoded once by ffn_prepare_weights).
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/ffn.h"
#include "ffn_internal.cuh"

__device__ unsigned g_ffn_status_word;

namespace ffn {
namespace {

// rows up to which the weight-streaming (decode) kernels can run the block
// (FFN_PATH_GEMV: eight token tiles), and up to which they do by default;
// the quantised entries run their rows in groups of kQuantGroupRows
constexpr int64_t kGemvMaxRows = 64;
constexpr int64_t kGemvAutoRows = 16;
constexpr int64_t kQuantGroupRows = 16;
constexpr int kMaxDevices = 64;

std::atomic<uint64_t> g_launch_count{0};

struct TimingRecord {
    int kind;
    cudaEvent_t a, b;
};
std::mutex g_mu;
std::atomic<bool> g_timing{false};
std::vector<TimingRecord> g_pending;
std::vector<cudaEvent_t> g_spare;
uint64_t g_timed_launches[K_NUM_KINDS];
double g_timed_ms[K_NUM_KINDS];

cudaEvent_t take_event() {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_spare.empty()) {
            cudaEvent_t e = g_spare.back();
            g_spare.pop_back();
            return e;
        }
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

size_t dtype_size(ffn_dtype dt) { return dt == FFN_F32 ? 4 : 2; }

bool valid_dtype(ffn_dtype dt) { return dt == FFN_F32 || dt == FFN_F16 || dt == FFN_BF16; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 64-byte groups of four Q4 blocks in a device-layout row of `in` weights
int64_t q4_groups(int64_t in) { return (in + 127) / 128; }

struct Range {
    const void *p;
    size_t bytes;
};
bool overlaps(Range a, Range b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

enum Path { PATH_SIMT, PATH_GEMV, PATH_GEMM };

struct Plan {
    Path path;
    bool fused;
    bool split_act;    // 16-bit paths: n and h enter the tensor ops as hi + lo terms
    bool prepared;     // weights are fp16 * 2^8 (ffn_prepare_weights); fp16 operands
    size_t workspace;
};

ffn_status check_block_shape(int64_t rows, int64_t d, int64_t ffn, ffn_dtype dt) {
    if (!valid_dtype(dt)) return FFN_ERR_DTYPE;
    if (rows < 0 || d < 1 || ffn < 1) return FFN_ERR_SHAPE;
    if (rows > INT32_MAX || d > INT32_MAX || ffn > INT32_MAX) return FFN_ERR_SHAPE;
    const int64_t vec = dt == FFN_F32 ? 4 : 8;
    if (d % vec || ffn % vec) return FFN_ERR_SHAPE;
    return FFN_OK;
}

ffn_status plan_block(int64_t rows, int64_t d, int64_t ffn, ffn_dtype dt, uint32_t flags,
                      Plan *plan) {
    ffn_status st = check_block_shape(rows, d, ffn, dt);
    if (st != FFN_OK) return st;
    const uint32_t known = FFN_GATEUP_FUSED | FFN_GATEUP_UNFUSED | FFN_PATH_GEMM | FFN_PATH_GEMV |
                           FFN_ACT_SINGLE | FFN_ACT_SPLIT | FFN_PREPARED_WEIGHTS | FFN_RESIDUAL |
                           FFN_DECODE_ONE_KERNEL;
    if (flags & ~known) return FFN_ERR_FLAGS;
    if ((flags & FFN_GATEUP_FUSED) && (flags & FFN_GATEUP_UNFUSED)) return FFN_ERR_FLAGS;
    if ((flags & FFN_PATH_GEMM) && (flags & FFN_PATH_GEMV)) return FFN_ERR_FLAGS;
    if ((flags & FFN_ACT_SINGLE) && (flags & FFN_ACT_SPLIT)) return FFN_ERR_FLAGS;
    plan->fused = !(flags & FFN_GATEUP_UNFUSED);
    // bf16 keeps 8 significant bits: rounding n and h once each costs more
    // than the block's error budget allows, so by default they enter the
    // tensor ops as hi + lo (about 16 bits).
    plan->prepared = (flags & FFN_PREPARED_WEIGHTS) != 0;
    if (plan->prepared && (dt == FFN_F32 || (flags & FFN_ACT_SPLIT))) return FFN_ERR_FLAGS;
    plan->split_act = !plan->prepared &&
                      ((flags & FFN_ACT_SPLIT) || (dt == FFN_BF16 && !(flags & FFN_ACT_SINGLE)));
    if (dt == FFN_F32 && (flags & (FFN_PATH_GEMM | FFN_PATH_GEMV))) return FFN_ERR_FLAGS;
    if ((flags & FFN_PATH_GEMV) && rows > kGemvMaxRows) return FFN_ERR_SHAPE;
    // rows up to which these flags take the decode kernels.  Measured
    // crossover on 4096 -> 14336 (graph-replayed block, one-term / hi + lo
    // operands): the GEMMs (one-row-block tiles, split-K down projection)
    // take 84 / 97 us at 12 rows, 73 / 78 us at 16-32, 75-79 / 81-86 us at
    // 64-128; the weight-streaming kernels 65 / 79 us at 12, 66 / 80 us at
    // 16, 75 / 104 us at 17, 79 / 107 us at 32 (four token tiles).
    // Two-term operands double their MMAs.
    int64_t gemv_rows = 0;
    if (dt != FFN_F32 && !(flags & FFN_PATH_GEMM))
        gemv_rows = (flags & FFN_PATH_GEMV) ? kGemvMaxRows : kGemvAutoRows;
    if (dt == FFN_F32)
        plan->path = PATH_SIMT;
    else
        plan->path = rows <= gemv_rows ? PATH_GEMV : PATH_GEMM;
    const size_t es = dtype_size(dt);
    const size_t r = static_cast<size_t>(rows);
    switch (plan->path) {
        case PATH_SIMT:
            plan->workspace = align256(r * d * 4) + align256(r * ffn * 4);
            break;
        case PATH_GEMV:
            plan->workspace = rows == 0 ? 0 : gemv_workspace_bytes(rows, d, ffn, plan->split_act);
            break;
        case PATH_GEMM:   // n and h (and their residuals); both 2 bytes when prepared
            plan->workspace = align256(r * d * es) + align256(r * ffn * es);
            if (plan->split_act) plan->workspace += align256(r * d * es) + align256(r * ffn * es);
            if (!plan->fused) plan->workspace += 2 * align256(r * ffn * 4);
            // split-K partial sums of the down GEMM (few rows)
            plan->workspace += align256(gemm_plain_partial_bytes(rows, ffn, d, plan->split_act ? 2 : 1));
            // the rows' sums of squares of y (ffn_block_forward_chained): parts per
            // 64-column block (the narrowest down tile) and counters per 128 rows
            plan->workspace += align256(static_cast<size_t>((d + 63) / 64) * r * 4) +
                               align256(static_cast<size_t>((rows + 127) / 128) * 4);
            // a workspace sized for these rows also serves every smaller
            // batch, those that take the decode kernels included
            if (gemv_rows > 0)
                plan->workspace = std::max(plan->workspace, gemv_workspace_bytes(std::min(rows, gemv_rows), d, ffn,
                                                                                  plan->split_act));
            break;
    }
    return FFN_OK;
}

ffn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FFN_OK : FFN_ERR_CUDA; }

}  // namespace

// ------------------------------------------------------------ shared helpers
const char *kernel_name(int kind) {
    static const char *names[K_NUM_KINDS] = {
        "prepare", "rmsnorm", "swiglu", "simt_gateup", "simt_down", "gemv_norm",
        "gemv_gateup", "gemv_down", "gemm_gateup", "gemm_down", "selftest", "splitk_reduce",
        "gemv_fused"};
    return (kind >= 0 && kind < K_NUM_KINDS) ? names[kind] : "unknown";
}

LaunchScope::LaunchScope(int k, cudaStream_t s) : kind(k), stream(s), ev0(nullptr) {
    g_launch_count.fetch_add(1, std::memory_order_relaxed);
    if (g_timing.load(std::memory_order_relaxed)) {
        cudaEvent_t e = take_event();
        if (e && cudaEventRecord(e, s) == cudaSuccess) ev0 = e;
    }
}

LaunchScope::~LaunchScope() {
    if (!ev0) return;
    cudaEvent_t e1 = take_event();
    if (!e1) return;
    if (cudaEventRecord(e1, stream) != cudaSuccess) return;
    std::lock_guard<std::mutex> lk(g_mu);
    g_pending.push_back({kind, static_cast<cudaEvent_t>(ev0), e1});
}

// Looked up on every call, not cached: after a cudaDeviceReset (or a context
// rebuilt in the same process) the module loads again and the word may sit
// elsewhere; once the module is loaded the lookup is a host-side query that
// allocates nothing, and it needs no lock between host threads.
unsigned *device_status_word() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ffn_status_word) != cudaSuccess) return nullptr;
    return static_cast<unsigned *>(p);
}

int sm_count() {
    static int count[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    if (!count[dev]) {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c < 1) c = 1;
        count[dev] = c;
    }
    return count[dev];
}

}  // namespace ffn

using namespace ffn;

extern "C" {

const char *ffn_status_string(ffn_status s) {
    switch (s) {
        case FFN_OK: return "ok";
        case FFN_ERR_NULL: return "a required pointer is NULL";
        case FFN_ERR_SHAPE: return "a size is out of range or breaks a divisibility rule";
        case FFN_ERR_DTYPE: return "unknown or unsupported storage type";
        case FFN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case FFN_ERR_WORKSPACE: return "workspace missing or too small";
        case FFN_ERR_ALIAS: return "an output overlaps an input";
        case FFN_ERR_CUDA: return "a CUDA runtime call failed";
        case FFN_ERR_TIMEOUT: return "a kernel abandoned a bounded wait";
        case FFN_ERR_FLAGS: return "contradictory or unknown flags";
        case FFN_ERR_RANGE: return "a weight is outside the prepared format's range";
    }
    return "unknown status";
}

uint64_t ffn_launch_count(void) { return g_launch_count.load(); }

ffn_status ffn_rmsnorm(const void *x, const void *g, void *n, int64_t rows, int64_t d, float eps,
                       ffn_dtype dtype, void *stream) {
    if (!g || (rows != 0 && (!x || !n))) return FFN_ERR_NULL;
    if (!valid_dtype(dtype)) return FFN_ERR_DTYPE;
    if (rows < 0 || d < 1 || rows > INT32_MAX || d > INT32_MAX) return FFN_ERR_SHAPE;
    if (rows == 0) return FFN_OK;
    if (!aligned16(x) || !aligned16(g) || !aligned16(n)) return FFN_ERR_ALIGN;
    const size_t es = dtype_size(dtype);
    const Range rx{x, static_cast<size_t>(rows) * d * es}, rg{g, static_cast<size_t>(d) * es},
        rn{n, static_cast<size_t>(rows) * d * es};
    if (n != x && overlaps(rn, rx)) return FFN_ERR_ALIAS;
    if (overlaps(rn, rg)) return FFN_ERR_ALIAS;
    if (rows == 0) return FFN_OK;
    return from_cuda(launch_rmsnorm(x, g, n, rows, d, eps, dtype, static_cast<cudaStream_t>(stream)));
}

ffn_status ffn_swiglu(const void *gate, const void *up, void *h, int64_t count, ffn_dtype dtype,
                      void *stream) {
    if (count != 0 && (!gate || !up || !h)) return FFN_ERR_NULL;
    if (!valid_dtype(dtype)) return FFN_ERR_DTYPE;
    if (count < 0) return FFN_ERR_SHAPE;
    if (count == 0) return FFN_OK;
    if (!aligned16(gate) || !aligned16(up) || !aligned16(h)) return FFN_ERR_ALIGN;
    const size_t bytes = static_cast<size_t>(count) * dtype_size(dtype);
    const Range rg{gate, bytes}, ru{up, bytes}, rh{h, bytes};
    if (h != gate && overlaps(rh, rg)) return FFN_ERR_ALIAS;
    if (h != up && overlaps(rh, ru)) return FFN_ERR_ALIAS;
    if (count == 0) return FFN_OK;
    return from_cuda(launch_swiglu(gate, up, h, count, dtype, static_cast<cudaStream_t>(stream)));
}

ffn_status ffn_block_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, ffn_dtype dtype,
                                     uint32_t flags, size_t *bytes) {
    if (!bytes) return FFN_ERR_NULL;
    Plan plan;
    ffn_status st = plan_block(rows, d, ffn, dtype, flags, &plan);
    if (st != FFN_OK) return st;
    *bytes = plan.workspace;
    return FFN_OK;
}

static ffn_status block_forward(const void *x, const float *x_sumsq, const void *g, const void *w_gate,
                                const void *w_up, const void *w_down, void *y, float *y_sumsq, int64_t rows,
                                int64_t d, int64_t ffn, float eps, ffn_dtype dtype, uint32_t flags,
                                void *workspace, size_t workspace_bytes, void *stream) {
    if (!g || !w_gate || !w_up || !w_down || (rows != 0 && (!x || !y))) return FFN_ERR_NULL;
    Plan plan;
    ffn_status st = plan_block(rows, d, ffn, dtype, flags, &plan);
    if (st != FFN_OK) return st;
    if (rows == 0) return FFN_OK;
    if (plan.workspace > 0 && !workspace) return FFN_ERR_WORKSPACE;
    if (workspace_bytes < plan.workspace) return FFN_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(g) || !aligned16(w_gate) || !aligned16(w_up) ||
        !aligned16(w_down) || !aligned16(y) || (workspace && !aligned16(workspace)))
        return FFN_ERR_ALIGN;
    const size_t es = dtype_size(dtype);
    const Range rx{x, static_cast<size_t>(rows) * d * es}, rg{g, static_cast<size_t>(d) * es},
        rwg{w_gate, static_cast<size_t>(ffn) * d * es}, rwu{w_up, static_cast<size_t>(ffn) * d * es},
        rwd{w_down, static_cast<size_t>(ffn) * d * es}, ry{y, static_cast<size_t>(rows) * d * es},
        rws{workspace, plan.workspace};
    for (const Range &in : {rx, rg, rwg, rwu, rwd})
        if (overlaps(ry, in) || overlaps(rws, in)) return FFN_ERR_ALIAS;
    if (overlaps(ry, rws)) return FFN_ERR_ALIAS;
    if ((x_sumsq && !aligned16(x_sumsq)) || (y_sumsq && !aligned16(y_sumsq))) return FFN_ERR_ALIGN;
    if (y_sumsq) {   // written last: may overlap nothing the call reads or writes
        const Range rso{y_sumsq, static_cast<size_t>(rows) * 4}, rsi{x_sumsq, static_cast<size_t>(rows) * 4};
        for (const Range &o : {rx, rg, rwg, rwu, rwd, ry, rws, rsi})
            if (overlaps(rso, o)) return FFN_ERR_ALIAS;
    }
    if (rows == 0) return FFN_OK;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    const void *res = (flags & FFN_RESIDUAL) ? x : nullptr;   // the skip connection adds x back
    switch (plan.path) {
        case PATH_SIMT: {
            float *n = reinterpret_cast<float *>(ws);
            float *h = reinterpret_cast<float *>(ws + align256(static_cast<size_t>(rows) * d * 4));
            return from_cuda(launch_simt_block(
                static_cast<const float *>(x), static_cast<const float *>(g),
                static_cast<const float *>(w_gate), static_cast<const float *>(w_up),
                static_cast<const float *>(w_down), static_cast<float *>(y), rows, d, ffn, eps, n, h, s,
                static_cast<const float *>(res), x_sumsq, y_sumsq));
        }
        case PATH_GEMV: {
            GemvWorkspace gw;
            gemv_carve(workspace, rows, d, ffn, plan.split_act, &gw);
            GemvWeights a{w_gate, nullptr, nullptr}, b{w_up, nullptr, nullptr}, c{w_down, nullptr, nullptr};
            const int wf = plan.prepared ? (dtype == FFN_BF16 ? WF_F16P : WF_F16)
                                         : (dtype == FFN_BF16 ? WF_BF16 : WF_F16);
            RowStats rs;
            rs.ss_in = x_sumsq;
            rs.ss_out = y_sumsq;
            return from_cuda(launch_gemv_block(wf, x, g, a, b, c, y, rows, d, ffn, eps, gw, s, res, rs,
                                               (flags & FFN_DECODE_ONE_KERNEL) != 0));
        }
        case PATH_GEMM: {
            const size_t nb = align256(static_cast<size_t>(rows) * d * es);
            const size_t hb = align256(static_cast<size_t>(rows) * ffn * es);
            char *p = ws;
            void *n = p;
            p += nb;
            void *n_lo = nullptr;
            void *h = nullptr;
            void *h_lo = nullptr;
            if (plan.split_act) {
                n_lo = p;
                p += nb;
            }
            h = p;
            p += hb;
            if (plan.split_act) {
                h_lo = p;
                p += hb;
            }
            // prepared weights: fp16 operands; the weights' 2^8 is undone on
            // G and U, h is stored times 2^-8 and the two cancel in the down GEMM
            const int op = plan.prepared ? static_cast<int>(DT_F16) : static_cast<int>(dtype);
            const float w_unscale = plan.prepared ? 1.f / kPreparedScale : 1.f;
            const float h_scale = plan.prepared ? 1.f / 256.f : 1.f;
            cudaError_t e;
            if (plan.prepared)
                e = launch_rmsnorm_to_f16(x, g, n, rows, d, eps, dtype, s, x_sumsq);
            else if (plan.split_act)
                e = launch_rmsnorm_split(x, g, n, n_lo, rows, d, eps, dtype, s, x_sumsq);
            else
                e = launch_rmsnorm(x, g, n, rows, d, eps, dtype, s, x_sumsq);
            if (e != cudaSuccess) return FFN_ERR_CUDA;
            // split-K partials: after h, or after G and U when unfused; then
            // the parts and counters of the rows' sums of squares of y
            char *pp = plan.fused ? p : p + 2 * align256(static_cast<size_t>(rows) * ffn * 4);
            float *part = reinterpret_cast<float *>(pp);
            pp += align256(gemm_plain_partial_bytes(rows, ffn, d, plan.split_act ? 2 : 1));
            float *ss_part = reinterpret_cast<float *>(pp);
            pp += align256(static_cast<size_t>((d + 63) / 64) * rows * 4);
            unsigned *ss_ctr = reinterpret_cast<unsigned *>(pp);
            const int nctr = y_sumsq ? static_cast<int>((rows + 127) / 128) : 0;
            if (plan.fused) {
                e = launch_gemm_gateup(op, n, n_lo, w_gate, w_up, h, h_lo, nullptr, nullptr, rows, d,
                                       ffn, true, w_unscale, h_scale, s, ss_ctr, nctr);
            } else {
                float *G = reinterpret_cast<float *>(p);
                float *U = reinterpret_cast<float *>(p + align256(static_cast<size_t>(rows) * ffn * 4));
                e = launch_gemm_gateup(op, n, n_lo, w_gate, w_up, nullptr, nullptr, G, U, rows, d, ffn,
                                       false, w_unscale, 1.f, s, ss_ctr, nctr);
                if (e == cudaSuccess) e = launch_swiglu_f32in(G, U, h, h_lo, rows * ffn, op, h_scale, s);
            }
            if (e != cudaSuccess) return FFN_ERR_CUDA;
            return from_cuda(launch_gemm_plain(op, dtype, h, h_lo, w_down, y, rows, ffn, d,
                                               w_unscale / h_scale, res, part, s, ss_part, ss_ctr, y_sumsq));
        }
    }
    return FFN_ERR_SHAPE;
}

ffn_status ffn_block_forward(const void *x, const void *g, const void *w_gate, const void *w_up,
                             const void *w_down, void *y, int64_t rows, int64_t d, int64_t ffn,
                             float eps, ffn_dtype dtype, uint32_t flags, void *workspace,
                             size_t workspace_bytes, void *stream) {
    return block_forward(x, nullptr, g, w_gate, w_up, w_down, y, nullptr, rows, d, ffn, eps, dtype, flags,
                         workspace, workspace_bytes, stream);
}

ffn_status ffn_block_forward_chained(const void *x, const float *x_sumsq, const void *g, const void *w_gate,
                                     const void *w_up, const void *w_down, void *y, float *y_sumsq, int64_t rows,
                                     int64_t d, int64_t ffn, float eps, ffn_dtype dtype, uint32_t flags,
                                     void *workspace, size_t workspace_bytes, void *stream) {
    return block_forward(x, x_sumsq, g, w_gate, w_up, w_down, y, y_sumsq, rows, d, ffn, eps, dtype, flags,
                         workspace, workspace_bytes, stream);
}

ffn_status ffn_block_q4_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, size_t *bytes) {
    if (!bytes) return FFN_ERR_NULL;
    if (rows < 0 || d < 32 || ffn < 32 || d % 32 || ffn % 32) return FFN_ERR_SHAPE;
    if (rows > INT32_MAX || d > INT32_MAX || ffn > INT32_MAX) return FFN_ERR_SHAPE;
    *bytes = rows == 0 ? 0 : gemv_workspace_bytes(std::min<int64_t>(rows, kQuantGroupRows), d, ffn, false);
    return FFN_OK;
}

ffn_status ffn_block_forward_q4(const void *x, const void *g, ffn_q4_weight w_gate,
                                ffn_q4_weight w_up, ffn_q4_weight w_down, void *y, int64_t rows,
                                int64_t d, int64_t ffn, float eps, uint32_t flags, void *workspace,
                                size_t workspace_bytes, void *stream) {
    if (!g || !w_gate.qs || !w_gate.scales || !w_up.qs || !w_up.scales || !w_down.qs ||
        !w_down.scales || (rows != 0 && (!x || !y)))
        return FFN_ERR_NULL;
    if (flags & ~(FFN_RESIDUAL | FFN_DECODE_ONE_KERNEL)) return FFN_ERR_FLAGS;
    size_t need = 0;
    ffn_status st = ffn_block_q4_workspace_bytes(rows, d, ffn, &need);
    if (st != FFN_OK) return st;
    if (need > 0 && !workspace) return FFN_ERR_WORKSPACE;
    if (workspace_bytes < need) return FFN_ERR_WORKSPACE;
    const void *ptrs[] = {x, g, y, w_gate.qs, w_gate.scales, w_up.qs, w_up.scales, w_down.qs,
                          w_down.scales};
    for (const void *p : ptrs)
        if (!aligned16(p)) return FFN_ERR_ALIGN;
    if (workspace && !aligned16(workspace)) return FFN_ERR_ALIGN;
    // device-layout bytes: rows of ceil(in/128) 64-byte groups, 4 scales a group
    const size_t qb = static_cast<size_t>(ffn) * q4_groups(d) * 64, sb = static_cast<size_t>(ffn) * q4_groups(d) * 8;
    const size_t qbd = static_cast<size_t>(d) * q4_groups(ffn) * 64, sbd = static_cast<size_t>(d) * q4_groups(ffn) * 8;
    const Range ry{y, static_cast<size_t>(rows) * d * 2}, rws{workspace, need};
    const Range ins[] = {{x, static_cast<size_t>(rows) * d * 2}, {g, static_cast<size_t>(d) * 2},
                         {w_gate.qs, qb}, {w_gate.scales, sb}, {w_up.qs, qb}, {w_up.scales, sb},
                         {w_down.qs, qbd}, {w_down.scales, sbd}};
    for (const Range &in : ins)
        if (overlaps(ry, in) || overlaps(rws, in)) return FFN_ERR_ALIAS;
    if (overlaps(ry, rws)) return FFN_ERR_ALIAS;
    if (rows == 0) return FFN_OK;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t grp = std::min<int64_t>(rows, kQuantGroupRows);
    GemvWorkspace gw;
    gemv_carve(workspace, grp, d, ffn, false, &gw);
    GemvWeights a{nullptr, w_gate.qs, w_gate.scales}, b{nullptr, w_up.qs, w_up.scales},
        c{nullptr, w_down.qs, w_down.scales};
    for (int64_t r0 = 0; r0 < rows; r0 += kQuantGroupRows) {
        const int64_t nr = std::min<int64_t>(kQuantGroupRows, rows - r0);
        const char *xr = static_cast<const char *>(x) + r0 * d * 2;
        char *yr = static_cast<char *>(y) + r0 * d * 2;
        cudaError_t e = launch_gemv_block(WF_Q4, xr, g, a, b, c, yr, nr, d, ffn, eps, gw, s,
                                          (flags & FFN_RESIDUAL) ? xr : nullptr, RowStats{},
                                          (flags & FFN_DECODE_ONE_KERNEL) != 0);
        if (e != cudaSuccess) return FFN_ERR_CUDA;
    }
    return FFN_OK;
}

ffn_status ffn_block_fp8_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, size_t *bytes) {
    if (!bytes) return FFN_ERR_NULL;
    if (rows < 0 || d < 256 || ffn < 256 || d % 256 || ffn % 256) return FFN_ERR_SHAPE;
    if (rows > INT32_MAX || d > INT32_MAX || ffn > INT32_MAX) return FFN_ERR_SHAPE;
    *bytes = rows == 0 ? 0 : gemv_workspace_bytes(std::min<int64_t>(rows, kQuantGroupRows), d, ffn, false);
    return FFN_OK;
}

ffn_status ffn_block_forward_fp8(const void *x, const void *g, ffn_fp8_weight w_gate,
                                 ffn_fp8_weight w_up, ffn_fp8_weight w_down, void *y, int64_t rows,
                                 int64_t d, int64_t ffn, float eps, uint32_t flags, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    if (!g || !w_gate.codes || !w_gate.scales || !w_up.codes || !w_up.scales || !w_down.codes ||
        !w_down.scales || (rows != 0 && (!x || !y)))
        return FFN_ERR_NULL;
    if (flags & ~(FFN_RESIDUAL | FFN_DECODE_ONE_KERNEL)) return FFN_ERR_FLAGS;
    size_t need = 0;
    ffn_status st = ffn_block_fp8_workspace_bytes(rows, d, ffn, &need);
    if (st != FFN_OK) return st;
    if (need > 0 && !workspace) return FFN_ERR_WORKSPACE;
    if (workspace_bytes < need) return FFN_ERR_WORKSPACE;
    const void *ptrs[] = {x, g, y, w_gate.codes, w_gate.scales, w_up.codes, w_up.scales, w_down.codes,
                          w_down.scales};
    for (const void *p : ptrs)
        if (!aligned16(p)) return FFN_ERR_ALIGN;
    if (workspace && !aligned16(workspace)) return FFN_ERR_ALIGN;
    const size_t cb = static_cast<size_t>(ffn) * d;
    const Range ry{y, static_cast<size_t>(rows) * d * 2}, rws{workspace, need};
    const Range ins[] = {{x, static_cast<size_t>(rows) * d * 2}, {g, static_cast<size_t>(d) * 2},
                         {w_gate.codes, cb}, {w_gate.scales, static_cast<size_t>(ffn) * 4},
                         {w_up.codes, cb}, {w_up.scales, static_cast<size_t>(ffn) * 4},
                         {w_down.codes, cb}, {w_down.scales, static_cast<size_t>(d) * 4}};
    for (const Range &in : ins)
        if (overlaps(ry, in) || overlaps(rws, in)) return FFN_ERR_ALIAS;
    if (overlaps(ry, rws)) return FFN_ERR_ALIAS;
    if (rows == 0) return FFN_OK;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t grp = std::min<int64_t>(rows, kQuantGroupRows);
    GemvWorkspace gw;
    gemv_carve(workspace, grp, d, ffn, false, &gw);
    GemvWeights a{w_gate.codes, nullptr, nullptr, w_gate.scales}, b{w_up.codes, nullptr, nullptr, w_up.scales},
        c{w_down.codes, nullptr, nullptr, w_down.scales};
    for (int64_t r0 = 0; r0 < rows; r0 += kQuantGroupRows) {
        const int64_t nr = std::min<int64_t>(kQuantGroupRows, rows - r0);
        const char *xr = static_cast<const char *>(x) + r0 * d * 2;
        char *yr = static_cast<char *>(y) + r0 * d * 2;
        cudaError_t e = launch_gemv_block(WF_FP8, xr, g, a, b, c, yr, nr, d, ffn, eps, gw, s,
                                          (flags & FFN_RESIDUAL) ? xr : nullptr, RowStats{},
                                          (flags & FFN_DECODE_ONE_KERNEL) != 0);
        if (e != cudaSuccess) return FFN_ERR_CUDA;
    }
    return FFN_OK;
}

ffn_status ffn_block_q8_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, size_t *bytes) {
    if (!bytes) return FFN_ERR_NULL;
    if (rows < 0 || d < 256 || ffn < 256 || d % 256 || ffn % 256) return FFN_ERR_SHAPE;
    if (rows > INT32_MAX || d > INT32_MAX || ffn > INT32_MAX) return FFN_ERR_SHAPE;
    *bytes = rows == 0 ? 0 : gemv_workspace_bytes(std::min<int64_t>(rows, kQuantGroupRows), d, ffn, false);
    return FFN_OK;
}

ffn_status ffn_block_forward_q8(const void *x, const void *g, ffn_q8_weight w_gate,
                                 ffn_q8_weight w_up, ffn_q8_weight w_down, void *y, int64_t rows,
                                 int64_t d, int64_t ffn, float eps, uint32_t flags, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    if (!g || !w_gate.codes || !w_gate.scales || !w_up.codes || !w_up.scales || !w_down.codes ||
        !w_down.scales || (rows != 0 && (!x || !y)))
        return FFN_ERR_NULL;
    if (flags & ~(FFN_RESIDUAL | FFN_DECODE_ONE_KERNEL)) return FFN_ERR_FLAGS;
    size_t need = 0;
    ffn_status st = ffn_block_q8_workspace_bytes(rows, d, ffn, &need);
    if (st != FFN_OK) return st;
    if (need > 0 && !workspace) return FFN_ERR_WORKSPACE;
    if (workspace_bytes < need) return FFN_ERR_WORKSPACE;
    const void *ptrs[] = {x, g, y, w_gate.codes, w_gate.scales, w_up.codes, w_up.scales, w_down.codes,
                          w_down.scales};
    for (const void *p : ptrs)
        if (!aligned16(p)) return FFN_ERR_ALIGN;
    if (workspace && !aligned16(workspace)) return FFN_ERR_ALIGN;
    const size_t cb = static_cast<size_t>(ffn) * d, sb = cb / 16;
    const Range ry{y, static_cast<size_t>(rows) * d * 2}, rws{workspace, need};
    const Range ins[] = {{x, static_cast<size_t>(rows) * d * 2}, {g, static_cast<size_t>(d) * 2},
                         {w_gate.codes, cb}, {w_gate.scales, sb}, {w_up.codes, cb}, {w_up.scales, sb},
                         {w_down.codes, cb}, {w_down.scales, sb}};
    for (const Range &in : ins)
        if (overlaps(ry, in) || overlaps(rws, in)) return FFN_ERR_ALIAS;
    if (overlaps(ry, rws)) return FFN_ERR_ALIAS;
    if (rows == 0) return FFN_OK;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t grp = std::min<int64_t>(rows, kQuantGroupRows);
    GemvWorkspace gw;
    gemv_carve(workspace, grp, d, ffn, false, &gw);
    GemvWeights a{w_gate.codes, nullptr, w_gate.scales}, b{w_up.codes, nullptr, w_up.scales},
        c{w_down.codes, nullptr, w_down.scales};
    for (int64_t r0 = 0; r0 < rows; r0 += kQuantGroupRows) {
        const int64_t nr = std::min<int64_t>(kQuantGroupRows, rows - r0);
        const char *xr = static_cast<const char *>(x) + r0 * d * 2;
        char *yr = static_cast<char *>(y) + r0 * d * 2;
        cudaError_t e = launch_gemv_block(WF_Q8, xr, g, a, b, c, yr, nr, d, ffn, eps, gw, s,
                                          (flags & FFN_RESIDUAL) ? xr : nullptr, RowStats{},
                                          (flags & FFN_DECODE_ONE_KERNEL) != 0);
        if (e != cudaSuccess) return FFN_ERR_CUDA;
    }
    return FFN_OK;
}

ffn_status ffn_q4_pack_host(const int8_t *q, const uint16_t *scales, int64_t out, int64_t in,
                            uint8_t *qs_out, uint16_t *scales_out) {
    if (!q || !scales || !qs_out || !scales_out) return FFN_ERR_NULL;
    if (out < 0 || in < 0 || in % 32) return FFN_ERR_SHAPE;
    const int64_t nblk = in / 32, ngrp = q4_groups(in);
    for (int64_t o = 0; o < out; ++o) {
        const int8_t *qr = q + o * in;
        for (int64_t i = 0; i < in; ++i)
            if (qr[i] < -8 || qr[i] > 7) return FFN_ERR_SHAPE;
        uint8_t *dst = qs_out + o * ngrp * 64;
        // a last, partial group's padding: zero bytes, zero scales
        std::memset(dst, 0, static_cast<size_t>(ngrp) * 64);
        std::memset(scales_out + o * ngrp * 4, 0, static_cast<size_t>(ngrp) * 8);
        for (int64_t blk = 0; blk < nblk; ++blk) {
            const int64_t grp = blk / 4;
            const int b = static_cast<int>(blk % 4);
            for (int i = 0; i < 16; ++i) {
                const uint8_t lo = static_cast<uint8_t>(qr[blk * 32 + i] + 8);
                const uint8_t hi = static_cast<uint8_t>(qr[blk * 32 + 16 + i] + 8);
                const int t = i / 4, e = i % 4;
                dst[grp * 64 + 16 * t + 4 * b + e] = static_cast<uint8_t>(lo | (hi << 4));
            }
        }
        std::memcpy(scales_out + o * ngrp * 4, scales + o * nblk, static_cast<size_t>(nblk) * 2);
    }
    return FFN_OK;
}

ffn_status ffn_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return FFN_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpyFromSymbol(&word, g_ffn_status_word, sizeof(word)) != cudaSuccess) return FFN_ERR_CUDA;
    if (word) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_ffn_status_word, &zero, sizeof(zero)) != cudaSuccess) return FFN_ERR_CUDA;
    }
    if (word & DEVERR_TIMEOUT) return FFN_ERR_TIMEOUT;
    return (word & DEVERR_RANGE) ? FFN_ERR_RANGE : FFN_OK;
}

ffn_status ffn_selftest_bounded_wait(uint64_t limit_ns, void *stream) {
    if (limit_ns < 1000) limit_ns = 1000;
    if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
    return from_cuda(launch_bounded_wait_probe(limit_ns, static_cast<cudaStream_t>(stream)));
}

ffn_status ffn_prepare_weights(const void *src, void *dst, int64_t count, ffn_dtype src_dtype,
                               void *stream) {
    if (count != 0 && (!src || !dst)) return FFN_ERR_NULL;
    if (src_dtype != FFN_BF16 && src_dtype != FFN_F16) return FFN_ERR_DTYPE;
    if (count < 0) return FFN_ERR_SHAPE;
    if (count == 0) return FFN_OK;
    if (!aligned16(src) || !aligned16(dst)) return FFN_ERR_ALIGN;
    const size_t bytes = static_cast<size_t>(count) * 2;
    if (overlaps({src, bytes}, {dst, bytes}) && src != dst) return FFN_ERR_ALIAS;
    return from_cuda(launch_prepare_weights(src, dst, count, src_dtype, static_cast<cudaStream_t>(stream)));
}

ffn_status ffn_prepare_weights_fp8(ffn_fp8_weight w, void *dst, int64_t out, int64_t in, void *stream) {
    if (out < 0 || in < 0 || in % 16) return FFN_ERR_SHAPE;
    if (out == 0 || in == 0) return FFN_OK;
    if (!w.codes || !w.scales || !dst) return FFN_ERR_NULL;
    if (!aligned16(w.codes) || !aligned16(w.scales) || !aligned16(dst)) return FFN_ERR_ALIGN;
    const size_t n = static_cast<size_t>(out) * in;
    const Range rd{dst, 2 * n};
    if (overlaps(rd, {w.codes, n}) || overlaps(rd, {w.scales, static_cast<size_t>(out) * 4})) return FFN_ERR_ALIAS;
    return from_cuda(launch_prepare_fp8(w.codes, w.scales, dst, out, in, static_cast<cudaStream_t>(stream)));
}

ffn_status ffn_prepare_weights_q4(ffn_q4_weight w, void *dst, int64_t out, int64_t in, void *stream) {
    if (out < 0 || in < 0 || in % 32) return FFN_ERR_SHAPE;
    if (out == 0 || in == 0) return FFN_OK;
    if (!w.qs || !w.scales || !dst) return FFN_ERR_NULL;
    if (!aligned16(w.qs) || !aligned16(w.scales) || !aligned16(dst)) return FFN_ERR_ALIGN;
    const size_t n = static_cast<size_t>(out) * in, grp = static_cast<size_t>(out) * q4_groups(in);
    const Range rd{dst, 2 * n};
    if (overlaps(rd, {w.qs, grp * 64}) || overlaps(rd, {w.scales, grp * 8})) return FFN_ERR_ALIAS;
    return from_cuda(launch_prepare_q4(w.qs, w.scales, dst, out, in, static_cast<cudaStream_t>(stream)));
}

ffn_status ffn_prepare_weights_q8(ffn_q8_weight w, void *dst, int64_t out, int64_t in, void *stream) {
    if (out < 0 || in < 0 || in % 32) return FFN_ERR_SHAPE;
    if (out == 0 || in == 0) return FFN_OK;
    if (!w.codes || !w.scales || !dst) return FFN_ERR_NULL;
    if (!aligned16(w.codes) || !aligned16(w.scales) || !aligned16(dst)) return FFN_ERR_ALIGN;
    const size_t n = static_cast<size_t>(out) * in;
    const Range rd{dst, 2 * n};
    if (overlaps(rd, {w.codes, n}) || overlaps(rd, {w.scales, n / 16})) return FFN_ERR_ALIAS;
    return from_cuda(launch_prepare_q8(w.codes, w.scales, dst, out, in, static_cast<cudaStream_t>(stream)));
}

ffn_status ffn_timing_enable(int on) {
    g_timing.store(on != 0);
    return FFN_OK;
}

ffn_status ffn_timing_collect(void) {
    std::vector<TimingRecord> pending;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        pending.swap(g_pending);
    }
    ffn_status st = FFN_OK;
    for (const TimingRecord &r : pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
            st = FFN_ERR_CUDA;
            continue;
        }
        std::lock_guard<std::mutex> lk(g_mu);
        g_timed_launches[r.kind] += 1;
        g_timed_ms[r.kind] += ms;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    for (const TimingRecord &r : pending) {
        g_spare.push_back(r.a);
        g_spare.push_back(r.b);
    }
    return st;
}

ffn_status ffn_timing_reset(void) {
    ffn_status st = ffn_timing_collect();
    std::lock_guard<std::mutex> lk(g_mu);
    for (int k = 0; k < K_NUM_KINDS; ++k) {
        g_timed_launches[k] = 0;
        g_timed_ms[k] = 0.0;
    }
    return st;
}

int ffn_kernel_kinds(void) { return K_NUM_KINDS; }

const char *ffn_kernel_name(int kind) { return kernel_name(kind); }

ffn_status ffn_timing_read(int kind, uint64_t *launches, double *total_ms) {
    if (!launches || !total_ms) return FFN_ERR_NULL;
    if (kind < 0 || kind >= K_NUM_KINDS) return FFN_ERR_SHAPE;
    std::lock_guard<std::mutex> lk(g_mu);
    *launches = g_timed_launches[kind];
    *total_ms = g_timed_ms[kind];
    return FFN_OK;
}

}  // extern "C"
