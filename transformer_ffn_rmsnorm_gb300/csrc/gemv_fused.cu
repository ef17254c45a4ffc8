// gemv_fused.cu -- the decode block (up to 64 token rows) as ONE persistent
// kernel: RMSNorm, gate/up with silu(G) * U, down projection.
//
// "Megakernels on Mac: What Fusion Saves and What It Costs" (sections
// "Dependencies and synchronization", "Small gaps between dispatches"): when
// the stages of a step run as one resident grid, the hand-off from one stage
// to the next is a counter in memory instead of the end of one dispatch and
// the start of the next, and a worker that is done with one stage goes on to
// the next stage's work that does not depend on the first.  Here:
//
//   * one cooperative launch: every CTA is resident for the whole call;
//   * norm    -- 8 x NT CTAs, one token slot each, write the normalised row
//                in fragment order (the same fragments as the three-kernel
//                path); the last of them raises every CTA's norm flag;
//   * gate/up -- CTA c owns the groups of 32 features c, c + G, ...; its
//                producer requests W_gate / W_up k-blocks at once and the
//                activation fragments of each stage once its norm flag is
//                up; silu(G) * U goes to the h fragments; the last CTA past
//                its gate/up work raises every CTA's gate/up flag;
//   * down    -- CTA c owns the units (64 output rows, one split of ffn) c,
//                c + G, ...; its producer requests W_down k-blocks as soon as
//                the ring has room -- while other CTAs still finish gate/up,
//                so HBM keeps streaming through the gate/up tail -- and the
//                h fragments of each stage once its gate/up flag is up.
//                Split partials are added in split order by the unit's last
//                CTA (bitwise reproducible), which also leaves the rows' sums
//                of squares of y when asked.
//
// The ring, its stage layout and the MMAs of one stage are those of the
// three-kernel path (gemv_stage.cuh): a gate/up stage (2 x 32 rows) and a
// down stage (64 rows) have the same size, so one ring serves both.
//
// Opt-in (FFN_DECODE_ONE_KERNEL): on GB300 the three-kernel chain is faster
// (8 x 4096 -> 14336 bf16 61.6 against 69.0 us, Q4 8 x 5120 -> 17408 38.1
// against 51.2 us, same session).  Its programmatic launches already request
// the next kernel's weights while the one before finishes, and the in-grid
// hand-off of the normalised row (stores, fence, arrival, flag, poll, bulk
// copy) takes longer than the kernel boundary it replaces.
//
// Synchronisation: through the stream's control block (library-owned device
// memory, below): arrival counters that their last arrival resets, and go
// flags stamped with the call's epoch, so nothing has to clear them between
// calls and no grid-wide barrier is needed (a cooperative-groups grid sync
// at the start measured 5 us).  Each CTA polls only its own go flags, not a
// word that every CTA reads.  A writer publishes with __threadfence() before
// its arrival; the last arriver fences again before raising the flags; a
// producer polls its flag with relaxed loads, fences (acquire) once it sees
// it, and issues fence.proxy.async before its bulk copies read the fragments
// other CTAs wrote with ordinary stores.  Every wait on a flag or an mbarrier
// is bounded (1 s): a wait that gives up records FFN_ERR_TIMEOUT, the CTA's
// other warps stop waiting but walk the same units (so their named barriers
// and arrivals still happen), and the producer lets the copies it issued
// land before the CTA exits.
#include <map>
#include <mutex>
#include <utility>

#include "gemv_stage.cuh"

namespace ffn {
namespace gemv {
namespace {

constexpr int kDone = 2;   // cursor role once a CTA has no more units

struct FusedParams {
    int64_t d, ffn;
    int rows;
    float eps;
    // RMSNorm
    const void *x, *gain;
    const float *ss_in;     // given rows' sums of squares of x, or null
    int nslots;             // token slots (8 x NT)
    int norm_cta0;          // CTA of slot 0
    // fragments
    uint16_t *nfrag, *nfrag_lo;
    int64_t nchK, nchF;     // 32-wide chunks along d and along ffn
    uint16_t *hfrag, *hfrag_lo;
    // gate/up
    int64_t ngu, nkb_gu;    // groups of 32 features; k-blocks over d
    const float *rs_g, *rs_u;
    // down
    int64_t ndn, nkb_dn;    // groups of 64 outputs; k-blocks over ffn
    int64_t splits, kb_per_split;
    void *y;
    const void *res;
    float *partials;        // [splits][rows][d]
    const float *rs_d;
    float *ss_part;         // [ndn][rows], with y_sumsq
    float *y_sumsq;         // [rows] or null
    unsigned long long *ctl;   // the stream's control block
    unsigned *err;
};

// A CTA's walk over its stages: its gate/up groups, then its down units.
struct Cursor {
    int role;
    int64_t unit, grp, kb, kb_end;
};

__device__ __forceinline__ void cursor_set(Cursor &c, const FusedParams &p) {
    if (c.role == ROLE_GATEUP) {
        if (c.unit < p.ngu) {
            c.grp = c.unit;
            c.kb = 0;
            c.kb_end = p.nkb_gu;
            return;
        }
        c.role = ROLE_DOWN;
        c.unit = blockIdx.x;
    }
    if (c.role == ROLE_DOWN) {
        if (c.unit < p.ndn * p.splits) {
            c.grp = c.unit / p.splits;
            c.kb = (c.unit % p.splits) * p.kb_per_split;
            c.kb_end = c.kb + p.kb_per_split < p.nkb_dn ? c.kb + p.kb_per_split : p.nkb_dn;
            return;
        }
        c.role = kDone;
    }
}
__device__ __forceinline__ void cursor_begin(Cursor &c, const FusedParams &p) {
    c.role = ROLE_GATEUP;
    c.unit = blockIdx.x;
    cursor_set(c, p);
}
__device__ __forceinline__ void cursor_next(Cursor &c, const FusedParams &p) {
    if (++c.kb == c.kb_end) {
        c.unit += gridDim.x;
        cursor_set(c, p);
    }
}

// Control blocks: library-owned device memory (a module array, zero when
// the module loads), one block a stream (calls on one stream run one after another; calls on
// different streams may overlap).  Arrival counters are plain atomicAdd
// counters that their last arrival sets back to zero, so every call finds
// them at zero.  Go flags carry the call's epoch (one more than the last
// completed call's, which that call's last CTA to exit stores), so they need
// no clearing: a flag of an earlier call is simply not this call's value.
// (Counters stamped with the epoch and updated by compare-and-swap convoyed
// when hundreds of CTAs arrived together: ~3 arrivals a microsecond.)
// Layout (words): the epoch, and the counters of norm slots done, CTAs past
// gate/up, CTAs done and groups with their row sums in, one 128-byte line
// each; then two go flags a CTA (norm done, gate/up done), eight CTAs a line;
// then a split counter a group of 64 outputs.
constexpr int kCtlSlots = 64;
constexpr int kMaxGrid = 4 * 152;
constexpr int kMaxGroups = 1024;   // d <= 65536
enum : int {
    W_EPOCH = 0,
    W_NORM = 16,
    W_GATEUP = 32,
    W_EXIT = 48,
    W_ROWS = 64,
    W_FLAGS0 = 80,
    W_SPLIT0 = W_FLAGS0 + 2 * kMaxGrid,
    kCtlWords = W_SPLIT0 + kMaxGroups
};
static_assert(kCtlWords % 16 == 0, "blocks of whole 128-byte lines");
__device__ __align__(128) unsigned long long g_fused_ctl[kCtlSlots * kCtlWords];
enum { GO_NORM = 0, GO_GATEUP = 1 };

// Polls read relaxed (an acquire load on every poll held up the SM's other
// memory traffic); the one that sees the flag is followed by an acquire fence.
__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long *ptr) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ptr) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// One arrival of n at counter c: true for the last, which sets the counter
// back to zero for the next call.
__device__ __forceinline__ bool arrive_last(unsigned long long *c, unsigned long long n) {
    if (atomicAdd(c, 1ull) != n - 1) return false;
    atomicExch(c, 0ull);
    return true;
}

// True once *flag holds `value` (then with acquire ordering); false after
// limit_ns of wall time or once *abort is set.
__device__ bool wait_flag(const unsigned long long *flag, unsigned long long value, volatile int *abort,
                          uint64_t limit_ns) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ld_relaxed64(flag) != value) {
        if (*abort) return false;
        if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
        __nanosleep(200);
    }
    fence_acquire_gpu();
    return true;
}

// Bulk copies issued after this read what this thread's earlier acquire made
// visible (ordinary stores of other CTAs).
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over the four consumer warps of every thread's v, returned to all.
__device__ __forceinline__ float consumer_sum(float v, float (&part)[kConsumers]) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
    consumer_sync();
    v = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) v += part[w];
    return v;
}

// RMSNorm of one token slot by the 128 consumer threads, into fragment order
// ("When to hand-write a GPU kernel on Apple Silicon", Rung 2: the row's sum
// of squares, the reciprocal root of its mean plus eps, times the gain).
// Rows of up to 4096 values stay in registers (one round trip for x and g);
// longer rows are read twice.  Slots >= rows (and k >= d) are written as 0.
template <int WF, bool TWO>
__device__ void norm_slot(const FusedParams &p, int token, float (&part)[kConsumers]) {
    using T = typename Fmt<WF>::TIn;
    constexpr int VPT = 4;
    const int64_t K = p.d, nv = K / 8, ngroups = p.nchK * 4;
    const bool live = token < p.rows;
    const uint4 *x = reinterpret_cast<const uint4 *>(static_cast<const T *>(p.x) + static_cast<int64_t>(token) * K);
    const uint4 *g = static_cast<const uint4 *>(p.gain);
    const int t = threadIdx.x;
    if (ngroups <= VPT * 32 * kConsumers) {
        uint4 xv[VPT], gv[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t v = t + 32 * kConsumers * i;
            const bool in = live && v < nv;
            xv[i] = in ? x[v] : make_uint4(0, 0, 0, 0);
            gv[i] = in ? g[v] : make_uint4(0, 0, 0, 0);
        }
        float ss = 0.f;
        if (p.ss_in) {
            ss = live ? p.ss_in[token] : 0.f;
        } else {
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                float f[8];
                Vec16<T>::unpack(xv[i], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
            }
            ss = consumer_sum(ss, part);
        }
        const float inv = rsqrtf(ss / static_cast<float>(K) + p.eps);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t v = t + 32 * kConsumers * i;
            if (v >= ngroups) break;
            float f[8], gf[8];
            Vec16<T>::unpack(xv[i], f);
            Vec16<T>::unpack(gv[i], gf);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = f[e] * inv * gf[e];
            store_group<WF, TWO>(p.nfrag, p.nfrag_lo, p.nchK, token, 8 * v, f);
        }
    } else {
        float ss = 0.f;
        if (p.ss_in) {
            ss = live ? p.ss_in[token] : 0.f;
        } else {
            for (int64_t v = t; live && v < nv; v += 32 * kConsumers) {
                float f[8];
                Vec16<T>::unpack(x[v], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
            }
            ss = consumer_sum(ss, part);
        }
        const float inv = rsqrtf(ss / static_cast<float>(K) + p.eps);
        for (int64_t v = t; v < ngroups; v += 32 * kConsumers) {
            float f[8];
            if (live && v < nv) {
                float gf[8];
                Vec16<T>::unpack(x[v], f);
                Vec16<T>::unpack(g[v], gf);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = f[e] * inv * gf[e];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = 0.f;
            }
            store_group<WF, TWO>(p.nfrag, p.nfrag_lo, p.nchK, token, 8 * v, f);
        }
    }
}

// CTAs a SM that the ring's shared memory allows (plus ~3 KB of static and
// reserved shared memory, out of 228 KB; at most four): the registers are
// held to that occupancy too.
template <int WF, int NT, bool TWO>
constexpr int fused_fit() {
    constexpr int fit = static_cast<int>((228 * 1024) / (Tile<WF, ROLE_GATEUP, NT, TWO>::smem_bytes + 3 * 1024));
    return fit < 1 ? 1 : fit > 4 ? 4 : fit;
}

template <int WF, int NT, bool TWO>
__global__ void __launch_bounds__(kThreads, fused_fit<WF, NT, TWO>()) gemv_fused_kernel(
    const __grid_constant__ CUtensorMap map_wg, const __grid_constant__ CUtensorMap map_wu,
    const __grid_constant__ CUtensorMap map_wd, const __grid_constant__ CUtensorMap map_sg,
    const __grid_constant__ CUtensorMap map_su, const __grid_constant__ CUtensorMap map_sd,
    const FusedParams p) {
    using TG = Tile<WF, ROLE_GATEUP, NT, TWO>;
    using TD = Tile<WF, ROLE_DOWN, NT, TWO>;
    static_assert(TG::stage_bytes == TD::stage_bytes && TG::b_off == TD::b_off && TG::kb == TD::kb &&
                      TG::stages == TD::stages && TG::b_bytes == TD::b_bytes,
                  "one ring serves both projections");
    using TO = typename Fmt<WF>::TOp;
    using TIn = typename Fmt<WF>::TIn;
    constexpr bool fp8 = TG::fp8;
    constexpr int kStages = TG::stages;
    constexpr int T = 8 * NT;   // token slots
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages], bar_empty[kStages];
    __shared__ float red[2][32][NT * 4];   // up sums handed to the gate warps
    __shared__ float half_ss[T][2];        // halves of a row's sum of squares within a group
    __shared__ float part[kConsumers];
    __shared__ int2 pend[kStages];         // producer: (k-block, role) of stages whose activations wait
    __shared__ int s_abort, s_never, s_last;
    __shared__ unsigned s_epoch;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
    auto full = [&](int s) { return ptx::smem_u32(&bar_full[s]); };
    auto empty = [&](int s) { return ptx::smem_u32(&bar_empty[s]); };
    auto stage_of = [&](int64_t i) { return base + static_cast<uint32_t>(i % kStages) * TG::stage_bytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), kConsumers);
        }
        s_abort = 0;
        s_never = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    volatile int *abort_flag = &s_abort;
    volatile int *never = &s_never;
    int64_t issued = 0;   // stages armed by the producer
    int64_t npend = 0;    // the last npend of them still wait for their activations
    Cursor pc;

    // ------------------------------------------------ producer helpers
    auto nvalid = [&](int role, int64_t kb) {   // activation chunks of a k range that exist
        const int64_t left = (role == ROLE_GATEUP ? p.nchK : p.nchF) - kb * TG::chunks;
        return static_cast<uint32_t>(left < TG::chunks ? left : TG::chunks);
    };
    auto arm = [&](int64_t i, int role, int64_t kb) {
        ptx::mbar_arrive_expect_tx(full(static_cast<int>(i % kStages)),
                                   TG::b_off + NT * TG::terms * nvalid(role, kb) * kFragBytes);
    };
    auto load_weights = [&](int64_t i, const Cursor &c) {
        const uint32_t st = stage_of(i), bar = full(static_cast<int>(i % kStages));
        const int x = static_cast<int>(c.kb * TG::x_per_kb);
        if (c.role == ROLE_GATEUP) {
            const int y = static_cast<int>(c.grp * TG::box_rows);
            ptx::tma_load_2d(st, &map_wg, bar, x, y);
            ptx::tma_load_2d(st + TG::w_bytes, &map_wu, bar, x, y);
            if (TG::boxes == 2) {
                ptx::tma_load_2d(st + TG::box_bytes, &map_wg, bar, x + TG::box_x, y);
                ptx::tma_load_2d(st + TG::w_bytes + TG::box_bytes, &map_wu, bar, x + TG::box_x, y);
            }
            if (TG::blocks) {
                const uint32_t sc = st + 2 * TG::w_bytes;
                ptx::tma_load_2d(sc, &map_sg, bar, static_cast<int>(c.kb * 8), y);
                ptx::tma_load_2d(sc + TG::s_bytes, &map_su, bar, static_cast<int>(c.kb * 8), y);
            }
        } else {
            const int y = static_cast<int>(c.grp * TD::box_rows);
            ptx::tma_load_2d(st, &map_wd, bar, x, y);
            if (TD::boxes == 2) ptx::tma_load_2d(st + TD::box_bytes, &map_wd, bar, x + TD::box_x, y);
            if (TD::blocks) ptx::tma_load_2d(st + TD::w_bytes, &map_sd, bar, static_cast<int>(c.kb * 8), y);
        }
    };
    auto load_acts = [&](int64_t i, int role, int64_t kb) {
        const uint32_t st = stage_of(i), bar = full(static_cast<int>(i % kStages));
        const uint32_t nv = nvalid(role, kb);
        const uint16_t *src = role == ROLE_GATEUP ? p.nfrag : p.hfrag;
        const uint16_t *src_lo = role == ROLE_GATEUP ? p.nfrag_lo : p.hfrag_lo;
        const int64_t nch = role == ROLE_GATEUP ? p.nchK : p.nchF;
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int t = 0; t < TG::terms; ++t)
                ptx::bulk_load(st + TG::b_off + (n * TG::terms + t) * TG::chunks * kFragBytes,
                               reinterpret_cast<const uint4 *>(t ? src_lo : src) + (n * nch + kb * TG::chunks) * 32,
                               nv * kFragBytes, bar);
    };

    // ---------- the first stages' weights, before the previous kernel ends
    if (warp == kConsumers && lane == 0) {
        ptx::tma_prefetch_map(&map_wg);
        ptx::tma_prefetch_map(&map_wu);
        ptx::tma_prefetch_map(&map_wd);
        cursor_begin(pc, p);
        while (issued < kStages && pc.role != kDone) {
            arm(issued, pc.role, pc.kb);
            load_weights(issued, pc);
            pend[issued % kStages] = make_int2(static_cast<int>(pc.kb), pc.role);
            ++issued;
            ++npend;
            cursor_next(pc, p);
        }
    }
    // the previous kernel's writes (x, the control block) are visible and its
    // reads of this call's buffers are done
    ptx::griddep_wait();
    if (threadIdx.x == 0)
        s_epoch = static_cast<unsigned>(*reinterpret_cast<volatile unsigned long long *>(p.ctl + W_EPOCH)) + 1u;
    __syncthreads();
    const unsigned ep = s_epoch;
    const unsigned long long go_value = (static_cast<unsigned long long>(ep) << 32) | 1ull;
    unsigned long long *const go = p.ctl + W_FLAGS0 + 2 * blockIdx.x;   // this CTA's flags
    ptx::griddep_launch_dependents();

    if (warp == kConsumers) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true, a_ok = false, b_ok = false;
            // may the activations of `role` be requested?  (block: wait for it)
            auto ready = [&](int role, bool block) -> bool {
                bool &flag = role == ROLE_GATEUP ? a_ok : b_ok;
                if (flag) return true;
                const unsigned long long *f = go + (role == ROLE_GATEUP ? GO_NORM : GO_GATEUP);
                if (block) {
                    if (!wait_flag(f, go_value, abort_flag, kWaitNs)) {
                        ok = false;
                        return false;
                    }
                    flag = true;
                } else {
                    flag = ld_relaxed64(f) == go_value;
                    if (flag) fence_acquire_gpu();
                }
                if (flag) fence_proxy_async_global();
                return flag;
            };
            while (ok) {
                // activations held back, oldest first; wait for them only when
                // the ring is all held-back stages or nothing else is left
                while (npend > 0) {
                    const int64_t i = issued - npend;
                    const int2 pe = pend[i % kStages];
                    if (!ready(pe.y, npend == kStages || pc.role == kDone)) break;
                    load_acts(i, pe.y, pe.x);
                    --npend;
                }
                if (!ok || pc.role == kDone) break;
                const int s = static_cast<int>(issued % kStages);
                const uint32_t ph = static_cast<uint32_t>((issued / kStages) & 1);
                if (!ptx::mbar_wait(empty(s), ph ^ 1u, abort_flag, kWaitNs)) {
                    ok = false;
                    break;
                }
                arm(issued, pc.role, pc.kb);
                load_weights(issued, pc);
                if (npend == 0 && ready(pc.role, false)) {
                    load_acts(issued, pc.role, pc.kb);
                } else {
                    pend[s] = make_int2(static_cast<int>(pc.kb), pc.role);
                    ++npend;
                }
                ++issued;
                cursor_next(pc, p);
            }
            if (!ok) {
                atomicOr(p.err, DEVERR_TIMEOUT);
                *abort_flag = 1;
                // complete the armed stages (workspace reads, whatever their
                // contents) so that no copy is left in flight
                for (; npend > 0; --npend) {
                    const int64_t i = issued - npend;
                    load_acts(i, pend[i % kStages].y, pend[i % kStages].x);
                }
            }
        }
    } else {
        // ------------------------------------------------------ MMA warps
        const int t = threadIdx.x;
        // This CTA's writes so far are published and it counts itself into
        // the counter at `word`; the last of `target` arrivals (returns true)
        // raises go flag `which` of every CTA (which < 0: none).
        auto arrive = [&](int64_t word, unsigned target, int which) -> bool {
            __threadfence();
            consumer_sync();
            if (t == 0) s_last = arrive_last(p.ctl + word, target);
            consumer_sync();
            const bool last = s_last != 0;
            if (last) {
                __threadfence();
                if (which >= 0)
                    for (int64_t cta = t; cta < gridDim.x; cta += 32 * kConsumers)
                        p.ctl[W_FLAGS0 + 2 * cta + which] = go_value;
            }
            return last;
        };
        const int slot = static_cast<int>(blockIdx.x) - p.norm_cta0;
        if (slot >= 0 && slot < p.nslots) {
            norm_slot<WF, TWO>(p, slot, part);
            arrive(W_NORM, static_cast<unsigned>(p.nslots), GO_NORM);
        }
        if (static_cast<int64_t>(blockIdx.x) >= p.ngu) arrive(W_GATEUP, gridDim.x, GO_GATEUP);   // no gate/up work

        const int g = lane >> 2, tid = lane & 3;
        float acc[NT][4];
        bool ok = true, fresh = true;
        Cursor c;
        cursor_begin(c, p);
        for (int64_t it = 0; c.role != kDone; ++it) {
            const int s = static_cast<int>(it % kStages);
            if (ok) {
                const uint32_t ph = static_cast<uint32_t>((it / kStages) & 1);
                const bool got = ptx::mbar_wait(full(s), ph, abort_flag, kWaitNs);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    if (lane == 0) {
                        atomicOr(p.err, DEVERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                }
            }
            if (fresh) {
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;
                fresh = false;
            }
            if (ok) {
                if (c.role == ROLE_GATEUP)
                    stage_mma<WF, NT, TWO, ROLE_GATEUP>(acc, stage_of(it), c.kb, p.nchK, warp, lane);
                else
                    stage_mma<WF, NT, TWO, ROLE_DOWN>(acc, stage_of(it), c.kb, p.nchF, warp, lane);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(empty(s));
            }
            if (c.kb + 1 < c.kb_end) {
                cursor_next(c, p);
                continue;
            }
            fresh = true;
            if (c.role == ROLE_GATEUP) {
                // ------------------------------- silu(G) * U of 32 features
                const int64_t row0 = c.grp * 32;
                const int r0 = 16 * (warp & 1);
                if (warp >= 2) {   // up tiles hand their sums to the gate warps
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int i = 0; i < 4; ++i) red[warp - 2][lane][n * 4 + i] = acc[n][i];
                }
                consumer_sync();
                if (warp < 2) {
                    constexpr float ws = Fmt<WF>::w_unscale;
                    float rsg[2] = {ws, ws}, rsu[2] = {ws, ws};   // weight scales of rows ra and rb
                    if constexpr (fp8) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int64_t feat = row0 + r0 + g + 8 * h;
                            rsg[h] = feat < p.ffn ? p.rs_g[feat] : 0.f;
                            rsu[h] = feat < p.ffn ? p.rs_u[feat] : 0.f;
                        }
                    }
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int64_t feat = row0 + r0 + g + 8 * (i >> 1);
                            const int token = 8 * n + 2 * tid + (i & 1);
                            const float hv = silu_f32(acc[n][i] * rsg[i >> 1]) *
                                             (red[warp][lane][n * 4 + i] * rsu[i >> 1]) * Fmt<WF>::h_scale;
                            const TO hq = from_f32<TO>(hv);
                            const int64_t at = frag_elem(frag_order<WF>(), p.nchF, token, feat);
                            p.hfrag[at] = *reinterpret_cast<const uint16_t *>(&hq);
                            if (TWO) {
                                const TO hl = from_f32<TO>(hv - to_f32(hq));
                                p.hfrag_lo[at] = *reinterpret_cast<const uint16_t *>(&hl);
                            }
                        }
                }
                if (c.unit + gridDim.x >= p.ngu)   // the CTA's last group: count it past gate/up
                    arrive(W_GATEUP, gridDim.x, GO_GATEUP);
                else
                    consumer_sync();   // red is free again
            } else {
                // -------------------- one split of 64 outputs: partial sums
                const int64_t row0 = c.grp * 64;
                const int64_t split = c.unit % p.splits;
                const int r0 = 16 * warp;
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int64_t feat = row0 + r0 + g + 8 * (i >> 1);
                        const int token = 8 * n + 2 * tid + (i & 1);
                        if (token < p.rows && feat < p.d)
                            p.partials[(split * p.rows + token) * p.d + feat] = acc[n][i];
                    }
                if (arrive(W_SPLIT0 + c.grp, static_cast<unsigned>(p.splits), -1)) {
                    // the unit's last split: add the splits in order, four
                    // outputs a thread and four splits at a time (16 loads in
                    // flight), and round y once
                    __threadfence();
                    TIn *y = static_cast<TIn *>(p.y);
                    constexpr int kStep = 32 * kConsumers;
                    constexpr float out_scale = Fmt<WF>::w_unscale / Fmt<WF>::h_scale;
                    const int nout = p.rows * 64;
                    const int64_t stride = static_cast<int64_t>(p.rows) * p.d;
                    const int nsplit = static_cast<int>(p.splits);
                    for (int b0 = 0; b0 < nout; b0 += 4 * kStep) {
                        bool live[4];
                        const float *src[4];
                        float sum[4];
#pragma unroll
                        for (int o = 0; o < 4; ++o) {
                            const int i = b0 + t + o * kStep;
                            const int64_t feat = row0 + (i & 63);
                            live[o] = i < nout && feat < p.d;
                            src[o] = p.partials + static_cast<int64_t>(i >> 6) * p.d + feat;
                            sum[o] = 0.f;
                        }
                        for (int sp0 = 0; sp0 < nsplit; sp0 += 4) {
                            float v[4][4];
#pragma unroll
                            for (int o = 0; o < 4; ++o)
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    v[o][q] = (live[o] && sp0 + q < nsplit) ? __ldcg(src[o] + (sp0 + q) * stride) : 0.f;
#pragma unroll
                            for (int o = 0; o < 4; ++o)
#pragma unroll
                                for (int q = 0; q < 4; ++q) sum[o] += v[o][q];
                        }
#pragma unroll
                        for (int o = 0; o < 4; ++o) {
                            const int i = b0 + t + o * kStep;
                            const int token = i >> 6;
                            const int64_t feat = row0 + (i & 63);
                            float sq = 0.f;
                            if (live[o]) {
                                float v = fp8 ? (sum[o] * p.rs_d[feat]) * out_scale : sum[o] * out_scale;
                                if (p.res) v += to_f32(static_cast<const TIn *>(p.res)[static_cast<int64_t>(token) * p.d + feat]);
                                const TIn yv = from_f32<TIn>(v);
                                y[static_cast<int64_t>(token) * p.d + feat] = yv;
                                const float r = to_f32(yv);
                                sq = r * r;
                            }
                            if (p.y_sumsq) {
                                // the 32 lanes hold 32 consecutive outputs of one token
                                sq = warp_sum(sq);
                                if (lane == 0 && token < p.rows) half_ss[token][warp & 1] = sq;
                            }
                        }
                    }
                    if (p.y_sumsq) {
                        // "Megakernels on Mac: What Fusion Saves and What It
                        // Costs", "Dependencies and synchronization": the next
                        // RMSNorm needs the sum of squares of the whole row, so
                        // each group's last split leaves its part, and the last
                        // group to finish adds the parts in group order
                        consumer_sync();
                        if (t < p.rows) p.ss_part[c.grp * p.rows + t] = half_ss[t][0] + half_ss[t][1];
                        if (arrive(W_ROWS, static_cast<unsigned>(p.ndn), -1)) {
                            if (t < p.rows) {
                                float ss = 0.f;
                                for (int64_t gi = 0; gi < p.ndn; ++gi) ss += __ldcg(p.ss_part + gi * p.rows + t);
                                p.y_sumsq[t] = ss;
                            }
                        }
                    }
                }
                consumer_sync();   // half_ss is free again
            }
            cursor_next(c, p);
        }
    }

    __syncthreads();
    if (threadIdx.x == 0 && arrive_last(p.ctl + W_EXIT, gridDim.x)) {
        // every CTA is past its last use of the control block: the next call
        // takes the next epoch
        __threadfence();
        *reinterpret_cast<volatile unsigned long long *>(p.ctl + W_EPOCH) = ep;
    }
    if (warp == kConsumers && lane == 0) {
        // copies still in flight (only after an abandoned wait) land before exit
        for (int s = 0; s < kStages; ++s) {
            if (issued > s) {
                const int64_t armed = (issued - s + kStages - 1) / kStages;
                ptx::mbar_wait(full(s), static_cast<uint32_t>((armed - 1) & 1), never, kWaitNs);
            }
        }
    }
}

// CTAs of the fused kernel that fit on 152 SMs at once: an upper bound of the
// grid, a function of the shape alone so that workspace queries agree with
// launches.
template <int WF, int NT, bool TWO>
constexpr int64_t fused_slots() {
    return 152 * static_cast<int64_t>(fused_fit<WF, NT, TWO>());
}

// Splits of ffn for the down units: as many as the grid has CTAs for (every
// unit one CTA), never finer than one k-block; then the k-blocks per split.
void fused_splits(int64_t ndn, int64_t nkb, int64_t grid, int64_t *splits, int64_t *per) {
    int64_t s = grid / ndn;
    if (s < 1) s = 1;
    if (s > nkb) s = nkb;
    *per = cdiv(nkb, s);
    *splits = cdiv(nkb, *per);
}

template <int WF, int NT, bool TWO>
int64_t fused_partial_floats(int64_t rows, int64_t d, int64_t ffn) {
    using TD = Tile<WF, ROLE_DOWN, NT, TWO>;
    int64_t splits, per;
    fused_splits(cdiv(d, 64), cdiv(ffn, TD::kb), fused_slots<WF, NT, TWO>(), &splits, &per);
    return splits * rows * d;
}

}  // namespace

unsigned long long *fused_control(int64_t d, cudaStream_t s) {
    if (cdiv(d, 64) > kMaxGroups) return nullptr;
    static std::mutex mu;
    static std::map<std::pair<int, cudaStream_t>, int> slot_of;
    constexpr int kDevices = 64;
    static int used[kDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return nullptr;
    // the blocks' address in the current context, looked up every call (a
    // host-side query once the module is loaded): right after a
    // cudaDeviceReset too, when the module loads again with its blocks zero
    void *base = nullptr;
    if (cudaGetSymbolAddress(&base, g_fused_ctl) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(dev, s);
    auto it = slot_of.find(key);
    if (it == slot_of.end()) {
        if (used[dev] == kCtlSlots) return nullptr;
        it = slot_of.emplace(key, used[dev]++).first;
    }
    return static_cast<unsigned long long *>(base) + static_cast<size_t>(it->second) * kCtlWords;
}

int64_t fused_partial_floats(int wfmt, int64_t rows, int64_t d, int64_t ffn, int nt, bool two) {
    switch (wfmt) {
        case WF_Q4: return nt == 1 ? fused_partial_floats<WF_Q4, 1, false>(rows, d, ffn)
                                   : fused_partial_floats<WF_Q4, 2, false>(rows, d, ffn);
        case WF_FP8: return nt == 1 ? fused_partial_floats<WF_FP8, 1, false>(rows, d, ffn)
                                    : fused_partial_floats<WF_FP8, 2, false>(rows, d, ffn);
        case WF_Q8: return nt == 1 ? fused_partial_floats<WF_Q8, 1, false>(rows, d, ffn)
                                   : fused_partial_floats<WF_Q8, 2, false>(rows, d, ffn);
        default: break;
    }
    if (two) {
        switch (nt) {
            case 1: return fused_partial_floats<WF_BF16, 1, true>(rows, d, ffn);
            case 2: return fused_partial_floats<WF_BF16, 2, true>(rows, d, ffn);
            case 4: return fused_partial_floats<WF_BF16, 4, true>(rows, d, ffn);
            default: return fused_partial_floats<WF_BF16, 8, true>(rows, d, ffn);
        }
    }
    switch (nt) {
        case 1: return fused_partial_floats<WF_BF16, 1, false>(rows, d, ffn);
        case 2: return fused_partial_floats<WF_BF16, 2, false>(rows, d, ffn);
        case 4: return fused_partial_floats<WF_BF16, 4, false>(rows, d, ffn);
        default: return fused_partial_floats<WF_BF16, 8, false>(rows, d, ffn);
    }
}

template <int WF, int NT, bool TWO>
cudaError_t launch_fused(GemvWeights wg, GemvWeights wu, GemvWeights wd, const void *x, const void *gain, void *y,
                         int rows, int64_t d, int64_t ffn, float eps, const GemvWorkspace &ws, const void *res,
                         const float *ss_in, float *y_sumsq, unsigned long long *ctl, cudaStream_t s) {
    using TG = Tile<WF, ROLE_GATEUP, NT, TWO>;
    constexpr auto kern = gemv_fused_kernel<WF, NT, TWO>;
    cudaError_t e = set_smem<kern>(TG::smem_bytes);
    if (e != cudaSuccess) return e;
    // grid: every CTA resident at once (a cooperative launch checks it)
    static int dev_seen = -1, per_sm = 0;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev != dev_seen) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, TG::smem_bytes);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        per_sm = n > 4 ? 4 : n;
        dev_seen = dev;
    }
    int64_t grid = static_cast<int64_t>(per_sm) * sm_count();
    if (grid > fused_slots<WF, NT, TWO>()) grid = fused_slots<WF, NT, TWO>();
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (grid < 8 * NT) return cudaErrorInvalidConfiguration;

    CUtensorMap mwg, mwu, mwd, msg, msu, msd;
    if (!weight_maps<WF, ROLE_GATEUP>(&mwg, &msg, wg, ffn, d) || !weight_maps<WF, ROLE_GATEUP>(&mwu, &msu, wu, ffn, d) ||
        !weight_maps<WF, ROLE_DOWN>(&mwd, &msd, wd, d, ffn))
        return cudaErrorInvalidValue;
    FusedParams p{};
    p.d = d;
    p.ffn = ffn;
    p.rows = rows;
    p.eps = eps;
    p.x = x;
    p.gain = gain;
    p.ss_in = ss_in;
    p.nslots = 8 * NT;
    p.nfrag = static_cast<uint16_t *>(ws.nfrag);
    p.nfrag_lo = static_cast<uint16_t *>(ws.nfrag_lo);
    p.nchK = cdiv(d, kChunk);
    p.nchF = cdiv(ffn, kChunk);
    p.hfrag = static_cast<uint16_t *>(ws.hfrag);
    p.hfrag_lo = static_cast<uint16_t *>(ws.hfrag_lo);
    p.ngu = p.nchF;   // groups of 32 features; covering nchF * 32 writes every slot of h
    p.nkb_gu = cdiv(d, TG::kb);
    p.rs_g = wg.rs;
    p.rs_u = wu.rs;
    p.ndn = cdiv(d, 64);
    p.nkb_dn = cdiv(ffn, TG::kb);
    fused_splits(p.ndn, p.nkb_dn, grid, &p.splits, &p.kb_per_split);
    // the norm slots on CTAs without gate/up work when there are enough
    p.norm_cta0 = grid - p.ngu >= p.nslots ? static_cast<int>(grid - p.nslots) : 0;
    p.y = y;
    p.res = res;
    p.partials = ws.partials;
    p.rs_d = wd.rs;
    p.ss_part = ws.ss_part;
    p.y_sumsq = y_sumsq;
    p.ctl = ctl;
    p.err = device_status_word();
    if (!p.err) return cudaErrorUnknown;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = TG::smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // as a programmatic dependent too (the first stages' weights requested
    // while the kernel before still runs), unless the runtime refuses that
    // together with a cooperative launch
    static bool pdl = true;
    cfg.numAttrs = pdl ? 2 : 1;
    LaunchScope scope(K_GEMV_FUSED, s);
    e = cudaLaunchKernelEx(&cfg, kern, mwg, mwu, mwd, msg, msu, msd, p);
    if (e != cudaSuccess && pdl) {
        (void)cudaGetLastError();
        pdl = false;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, mwg, mwu, mwd, msg, msu, msd, p);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

#define FFN_FUSED_INSTANTIATE(WF, NT, TWO)                                                                     \
    template cudaError_t launch_fused<WF, NT, TWO>(GemvWeights, GemvWeights, GemvWeights, const void *,          \
                                                   const void *, void *, int, int64_t, int64_t, float,           \
                                                   const GemvWorkspace &, const void *, const float *, float *, \
                                                   unsigned long long *, cudaStream_t);
FFN_FUSED_INSTANTIATE(WF_F16, 1, false)
FFN_FUSED_INSTANTIATE(WF_F16, 2, false)
FFN_FUSED_INSTANTIATE(WF_F16, 4, false)
FFN_FUSED_INSTANTIATE(WF_F16, 8, false)
FFN_FUSED_INSTANTIATE(WF_F16, 1, true)
FFN_FUSED_INSTANTIATE(WF_F16, 2, true)
FFN_FUSED_INSTANTIATE(WF_F16, 4, true)
FFN_FUSED_INSTANTIATE(WF_F16, 8, true)
FFN_FUSED_INSTANTIATE(WF_BF16, 1, false)
FFN_FUSED_INSTANTIATE(WF_BF16, 2, false)
FFN_FUSED_INSTANTIATE(WF_BF16, 4, false)
FFN_FUSED_INSTANTIATE(WF_BF16, 8, false)
FFN_FUSED_INSTANTIATE(WF_BF16, 1, true)
FFN_FUSED_INSTANTIATE(WF_BF16, 2, true)
FFN_FUSED_INSTANTIATE(WF_BF16, 4, true)
FFN_FUSED_INSTANTIATE(WF_BF16, 8, true)
FFN_FUSED_INSTANTIATE(WF_F16P, 1, false)
FFN_FUSED_INSTANTIATE(WF_F16P, 2, false)
FFN_FUSED_INSTANTIATE(WF_F16P, 4, false)
FFN_FUSED_INSTANTIATE(WF_F16P, 8, false)
FFN_FUSED_INSTANTIATE(WF_Q4, 1, false)
FFN_FUSED_INSTANTIATE(WF_Q4, 2, false)
FFN_FUSED_INSTANTIATE(WF_FP8, 1, false)
FFN_FUSED_INSTANTIATE(WF_FP8, 2, false)
FFN_FUSED_INSTANTIATE(WF_Q8, 1, false)
FFN_FUSED_INSTANTIATE(WF_Q8, 2, false)

}  // namespace gemv
}  // namespace ffn
