// gemv_stream.cu -- decode (few-row) projections with the weight stream decoupled
// from the math.
//
// The register-streaming kernels (gemv.cu) load weights straight into MMA
// fragments: each warp issues a burst of loads, waits, computes, and only
// then issues the next burst, so HBM idles between bursts (ncu: stalled on
// the long scoreboard, 1.6-4.4 TB/s).  Here one producer thread per CTA keeps
// a 6-stage shared-memory ring full with TMA bulk tensor copies of 64 weight
// rows x one k-block (16-bit: 128 values in two 128-byte boxes a row; Q4: 256 values,
// 128 bytes of nibbles plus 16 bytes of fp16 scales a row; e4m3: 256 codes
// in two 128-byte boxes a row; Q8_0: the same plus 16 bytes of scales a
// row), 128-byte swizzled, plus -- by 1-D bulk copies -- the pre-arranged activation
// fragments of the same k range, while four MMA warps read everything from
// shared memory.  (Reading the activations through L1 instead stalls: the
// rings leave too little L1 to hold them.)
//
// Roles: gate/up -- a CTA owns 32 features (32 rows of W_gate and of W_up)
// over the whole of d and applies silu(G)*U; down -- a CTA owns 64 rows of
// W_down over one split of ffn and hands its partial sums to the same
// deterministic last-CTA reduction as the register kernels.
//
// Q4 ("Unfusing a Kernel Made It 1.63x Faster", "The finding that keeps us
// honest about microbenchmarks": the unpacking must hide under the stream):
// the nibbles enter the MMAs as the LOP3s leave them (unpack_word_biased),
// and each stage's per-block offsets, written beside the activations by the
// kernel that wrote them (store_block_corr), come off through two tf32 MMAs
// on the block scales; the gate/up epilogue writes h and its offsets in the
// same form for the down kernel.
//
// Both kernels are launched as programmatic dependents of the kernel before
// them: a CTA starts while that kernel is still running, requests its first
// ring's worth of weights (inputs of the call) at once, and waits for that
// kernel to complete before it requests any activation or writes anything.
//
// Every mbarrier wait is bounded (1 s); a wait that gives up records
// FFN_ERR_TIMEOUT in the device status word, stops the other roles, and the
// producer waits (bounded) for its copies in flight before the CTA exits.
#include <algorithm>
#include <cstdlib>

#include "gemv_stage.cuh"

namespace ffn {
namespace gemv {
namespace {

struct StreamParams {
    int64_t K;              // reduction length
    int64_t rows_w;         // rows of each weight matrix (ffn for gate/up, d for down)
    int64_t nkb;            // k-blocks over K
    int64_t kb_per_split;   // down: k-blocks per CTA split
    const uint4 *bfrag, *bfrag_lo;
    int64_t nch_b;          // fragment chunks of the activation operand
    uint16_t *hfrag, *hfrag_lo;
    int64_t nch_h;          // gate/up: fragment chunks of h
    void *y;
    float *partials;
    unsigned *counters;
    int ncounters;
    int rows;               // token rows (<= 16)
    int64_t D;              // down: output features
    unsigned *err;
    const void *res;        // down: added to y before its rounding ([rows x D] of y's type), or null
    const float *rs0, *rs1; // e4m3: row scales of the weight matrices (gate and up, or down)
    int pre_stages;         // weight stages requested before the wait (at most the ring)
    float *ss_part;         // down, with y_sumsq: [feature groups][rows] sums of squares of stored y
    float *y_sumsq;         // down: [rows] sum over the row of the stored y squared, or null
    const float *bcorr;     // Q4: block offsets of the activation operand (store_q4_corr)
    float *hcorr;           // Q4 gate/up: block offsets of h, written here
};

template <int WF, int NT, bool TWO, int ROLE>
__global__ void __launch_bounds__(kThreads) gemv_stream_kernel(
    const __grid_constant__ CUtensorMap map_w0, const __grid_constant__ CUtensorMap map_w1,
    const __grid_constant__ CUtensorMap map_s0, const __grid_constant__ CUtensorMap map_s1,
    const StreamParams p) {
    // Q4 operands take the biased form (unpack_word_biased) here
    constexpr bool BIAS = WF == WF_Q4;
    using TL = Tile<WF, ROLE, NT, TWO, BIAS>;
    using TO = typename Fmt<WF>::TOp;
    constexpr bool fp8 = TL::fp8;
    constexpr int kStages = TL::stages;
    // h is stored times hs (the biased Q4 form: low positions 2^-4, high
    // ones a further 2^-4, so both keep the precision of the plain form's
    // 2^-8 where it matters and |h| up to 2^20 stays finite)
    constexpr float hs = BIAS ? 0.0625f : Fmt<WF>::h_scale;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages], bar_empty[kStages];
    __shared__ float s_bias[2][BIAS ? 8 * NT : 1];
    __shared__ int s_abort, s_never, s_last, s_last_row;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t cbase = base + kStages * TL::stage_bytes;   // the ring of block offsets (BIAS)
    // generic address of the ring, for epilogue scratch once every stage is consumed
    uint8_t *const ring = smem_raw + (base - ptx::smem_u32(smem_raw));
    auto full = [&](int s) { return ptx::smem_u32(&bar_full[s]); };
    auto empty = [&](int s) { return ptx::smem_u32(&bar_empty[s]); };

    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * (ROLE == ROLE_GATEUP ? 32 : 64);
    const int64_t kb0 = ROLE == ROLE_DOWN ? blockIdx.y * p.kb_per_split : 0;
    const int64_t kb1 = ROLE == ROLE_DOWN ? min(p.nkb, kb0 + p.kb_per_split) : p.nkb;

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
    // the next kernel on the stream may be scheduled once every CTA is running
    ptx::griddep_launch_dependents();
    volatile int *abort_flag = &s_abort;
    volatile int *never = &s_never;
    int64_t issued = 0;

    if (warp == kConsumers) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            ptx::tma_prefetch_map(&map_w0);
            if (TL::nmat == 2) ptx::tma_prefetch_map(&map_w1);
            // Stage slots and phases are running 32-bit counters, and every
            // address below is one multiply-add from a per-CTA base: the
            // producer shares its SM's issue slots with the MMA warps of up to
            // four CTAs (64-bit stage arithmetic here had cost ~120
            // instructions per stage, 9 % of the Q4 gate/up kernel's).
            const int nkb = static_cast<int>(kb1 - kb0);
            const int nch_b = static_cast<int>(p.nch_b);
            const int y = static_cast<int>(row0);
            const uint4 *act[NT * TL::terms];
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int t = 0; t < TL::terms; ++t)
                    act[n * TL::terms + t] = (t ? p.bfrag_lo : p.bfrag) + (n * p.nch_b + kb0 * TL::chunks) * 32;
            // activation chunks of k-block j that exist (the last 64-wide
            // block can hang one chunk past the buffer)
            auto nvalid = [&](int j) {
                const int left = nch_b - static_cast<int>(kb0 + j) * TL::chunks;
                return static_cast<uint32_t>(left < TL::chunks ? left : TL::chunks);
            };
            auto arm = [&](int s, int j) {
                ptx::mbar_arrive_expect_tx(full(s), TL::b_off + NT * TL::terms * nvalid(j) * kFragBytes +
                                                        TL::corr_bytes);
            };
            auto load_weights = [&](int s, int j) {
                const uint32_t st = base + s * TL::stage_bytes, bar = full(s);
                const int kb = static_cast<int>(kb0) + j;
                const int x = kb * TL::x_per_kb;   // bytes of nibbles or codes / elements
                ptx::tma_load_2d(st, &map_w0, bar, x, y);
                if (TL::nmat == 2) ptx::tma_load_2d(st + TL::w_bytes, &map_w1, bar, x, y);
                if (TL::boxes == 2) {   // the second 128 bytes of each row
                    ptx::tma_load_2d(st + TL::box_bytes, &map_w0, bar, x + TL::box_x, y);
                    if (TL::nmat == 2)
                        ptx::tma_load_2d(st + TL::w_bytes + TL::box_bytes, &map_w1, bar, x + TL::box_x, y);
                }
                if (TL::blocks) {
                    const uint32_t sc = st + TL::nmat * TL::w_bytes;
                    ptx::tma_load_2d(sc, &map_s0, bar, kb * 8, y);
                    if (TL::nmat == 2) ptx::tma_load_2d(sc + TL::s_bytes, &map_s1, bar, kb * 8, y);
                }
            };
            auto load_acts = [&](int s, int j) {
                const uint32_t st = base + s * TL::stage_bytes, bar = full(s);
                const uint32_t nv = nvalid(j);
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int t = 0; t < TL::terms; ++t)
                        ptx::bulk_load(st + TL::b_off + (n * TL::terms + t) * TL::chunks * kFragBytes,
                                       act[n * TL::terms + t] + j * (TL::chunks * 32), nv * kFragBytes, bar);
                if constexpr (TL::corr_bytes != 0)   // the stage's block offsets: NT x 512 contiguous bytes
                    ptx::bulk_load(cbase + s * TL::corr_bytes, p.bcorr + (kb0 + j) * (TL::corr_bytes / 4),
                                   TL::corr_bytes, bar);
            };
            // The first ring's worth of weights is requested before the kernel
            // that writes the activations has finished (weights are inputs of
            // the call); the activations only after it has.
            int npre = nkb < kStages ? nkb : kStages;
            if (npre > p.pre_stages) npre = p.pre_stages;
            for (int j = 0; j < npre; ++j) {
                arm(j, j);
                load_weights(j, j);
            }
            issued = npre;
            ptx::griddep_wait();
            for (int j = 0; j < npre; ++j) load_acts(j, j);
            bool ok = true;
            int s = npre == kStages ? 0 : npre;
            uint32_t ph = npre == kStages ? 1u : 0u;   // parity of the slot's current use
            for (int j = npre; j < nkb; ++j) {
                if (!ptx::mbar_wait(empty(s), ph ^ 1u, abort_flag, kWaitNs)) {
                    ok = false;
                    break;
                }
                arm(s, j);
                load_acts(s, j);
                load_weights(s, j);
                issued = j + 1;
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) {
                atomicOr(p.err, DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
        }
    } else {
        // ------------------------------------------------------ MMA warps
        ptx::griddep_wait();
        if (ROLE == ROLE_GATEUP && blockIdx.x == 0)   // arrival counters of this call's down projection
            for (int i = threadIdx.x; i < p.ncounters; i += 32 * kConsumers) p.counters[i] = 0u;
        const int g = lane >> 2, tid = lane & 3;
        const int r0 = 16 * (ROLE == ROLE_GATEUP ? (warp & 1) : warp);   // row tile inside the box
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[n][i] = 0.f;
        bool ok = true;
        int s = 0;
        uint32_t ph = 0;   // slot and parity of the stage consumed next
        for (int64_t kb = kb0; kb < kb1; ++kb) {
            const bool got = ptx::mbar_wait(full(s), ph, abort_flag, kWaitNs);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            stage_mma<WF, NT, TWO, ROLE, BIAS>(acc, base + s * TL::stage_bytes, kb, p.nch_b, warp, lane,
                                               cbase + s * TL::corr_bytes);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty(s));
            if (++s == kStages) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!ok) {
            if (lane == 0) {
                atomicOr(p.err, DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
        }

        // ------------------------------------------------------- epilogues
        if constexpr (ROLE == ROLE_GATEUP) {
            // scratch in the ring, once every MMA warp is past its last stage
            float (*red)[32][NT * 4] = reinterpret_cast<float (*)[32][NT * 4]>(ring);
            consumer_sync();
            if (warp >= 2) {   // up tiles hand their fragments to the gate warps
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
                        rsg[h] = feat < p.rows_w ? p.rs0[feat] : 0.f;
                        rsu[h] = feat < p.rows_w ? p.rs1[feat] : 0.f;
                    }
                }
                // (BIAS: this CTA's 32 features are one Q4 block of the down
                // projection's K, warp 0's its low half, warp 1's its high half)
                float bsum[NT][2];
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int64_t feat = row0 + r0 + g + 8 * (i >> 1);
                        const int token = 8 * n + 2 * tid + (i & 1);
                        float hv = silu_f32(acc[n][i] * rsg[i >> 1]) * (red[warp][lane][n * 4 + i] * rsu[i >> 1]) * hs;
                        if (BIAS && warp == 1) hv *= 0.0625f;
                        const TO t = from_f32<TO>(hv);
                        const int64_t at = frag_elem(frag_order<WF>(), p.nch_h, token, feat);
                        p.hfrag[at] = *reinterpret_cast<const uint16_t *>(&t);
                        if (TWO) {
                            const TO tl = from_f32<TO>(hv - to_f32(t));
                            p.hfrag_lo[at] = *reinterpret_cast<const uint16_t *>(&tl);
                        }
                        if (BIAS) bsum[n][i & 1] = (i < 2 ? 0.f : bsum[n][i & 1]) + to_f32(t);
                    }
                if constexpr (BIAS) {
                    // per token, the sum of the stored h over the warp's 16
                    // features (lanes of one t share the tokens), weighted by
                    // the half's offset
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            float v = bsum[n][e];
                            v += __shfl_xor_sync(0xffffffffu, v, 4);
                            v += __shfl_xor_sync(0xffffffffu, v, 8);
                            v += __shfl_xor_sync(0xffffffffu, v, 16);
                            if (g == 0) s_bias[warp][8 * n + 2 * tid + e] = v * (warp ? 1152.f : 1032.f);
                        }
                }
            }
            if constexpr (BIAS) {
                consumer_sync();
                if (threadIdx.x < 8 * NT)
                    store_q4_corr(p.hcorr, NT, threadIdx.x, blockIdx.x, s_bias[0][threadIdx.x] + s_bias[1][threadIdx.x]);
            }
        } else {
            using T = typename Fmt<WF>::TIn;
            constexpr float out_scale = Fmt<WF>::w_unscale / hs;
            const int split = blockIdx.y, nsplit = gridDim.y;
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t feat = row0 + r0 + g + 8 * (i >> 1);
                    const int token = 8 * n + 2 * tid + (i & 1);
                    if (token < p.rows && feat < p.D)
                        p.partials[(static_cast<int64_t>(split) * p.rows + token) * p.D + feat] = acc[n][i];
                }
            __threadfence();
            consumer_sync();
            if (threadIdx.x == 0)
                s_last = atomicAdd(&p.counters[blockIdx.x], 1u) == static_cast<unsigned>(nsplit - 1);
            consumer_sync();
            if (s_last) {
                __threadfence();
                T *y = static_cast<T *>(p.y);
                // four outputs a thread at a time, their partials four splits at a
                // time (16 loads in flight), each output summed in split order
                constexpr int kStep = 32 * kConsumers;
                const int nout = p.rows * 64;
                const int64_t stride = static_cast<int64_t>(p.rows) * p.D;
                for (int i0 = threadIdx.x; i0 < nout; i0 += 4 * kStep) {
                    bool live[4];
                    const float *src[4];
                    float sum[4];
#pragma unroll
                    for (int o = 0; o < 4; ++o) {
                        const int i = i0 + o * kStep;
                        const int64_t feat = row0 + i % 64;
                        live[o] = i < nout && feat < p.D;
                        src[o] = p.partials + static_cast<int64_t>(i / 64) * p.D + feat;
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
                        if (!live[o]) continue;
                        const int i = i0 + o * kStep;
                        const int token = i / 64;
                        const int64_t feat = row0 + i % 64;
                        float v = fp8 ? (sum[o] * p.rs0[feat]) * out_scale : sum[o] * out_scale;
                        if (p.res) v += to_f32(static_cast<const T *>(p.res)[static_cast<int64_t>(token) * p.D + feat]);
                        const T yv = from_f32<T>(v);
                        y[static_cast<int64_t>(token) * p.D + feat] = yv;
                        if (p.y_sumsq) {   // the stored value squared, for the row's sum (ring memory is free now)
                            const float r = to_f32(yv);
                            reinterpret_cast<float *>(ring)[i] = r * r;
                        }
                    }
                }
                if (threadIdx.x == 0) p.counters[blockIdx.x] = 0u;
                if (p.y_sumsq) {
                    // "Megakernels on Mac: What Fusion Saves and What It Costs",
                    // "Dependencies and synchronization": the next RMSNorm needs
                    // the sum of squares of every element of the row, so each
                    // feature group's closing CTA leaves its part of it, and the
                    // last group to finish adds the parts in group order
                    const float *sq = reinterpret_cast<const float *>(ring);
                    consumer_sync();
                    const int64_t nf = p.D - row0 < 64 ? p.D - row0 : 64;
                    if (threadIdx.x < p.rows) {
                        float ss = 0.f;
                        for (int j = 0; j < nf; ++j) ss += sq[threadIdx.x * 64 + j];
                        p.ss_part[static_cast<int64_t>(blockIdx.x) * p.rows + threadIdx.x] = ss;
                    }
                    consumer_sync();
                    if (threadIdx.x == 0) {
                        __threadfence();
                        s_last_row = atomicAdd(&p.counters[gridDim.x], 1u) == gridDim.x - 1;
                    }
                    consumer_sync();
                    if (s_last_row) {
                        __threadfence();
                        if (threadIdx.x < p.rows) {
                            float ss = 0.f;
                            for (unsigned gi = 0; gi < gridDim.x; ++gi)
                                ss += __ldcg(p.ss_part + static_cast<int64_t>(gi) * p.rows + threadIdx.x);
                            p.y_sumsq[threadIdx.x] = ss;
                        }
                        if (threadIdx.x == 0) p.counters[gridDim.x] = 0u;
                    }
                }
            }
        }
    }

    __syncthreads();
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

}  // namespace

// Launch-shape choices of the decode kernels, measured on GB300 (per-CTA
// globaltimer traces of graph-replayed 8 x 4096 -> 14336 bf16 and 8 x 5120 ->
// 17408 Q4 calls):
//  - the norm kernel releases the gate/up kernel right after its own wait,
//    so the gate/up kernel is resident and requesting weights while the norm
//    runs (Q4 call 38.2 us against 39.3 us when released at its end);
//  - gate/up requests ONE stage of weights before its wait, not its whole
//    ring: the wait returns once the norm kernel has completed, and that
//    completion takes longer while megabytes of loads are in flight (3.1 us
//    against 4.7 us after the call starts; Q4 call 38.2 against 38.9 us);
//  - down requests all of its ring but one stage before its wait (-1 below):
//    the whole ring competes with the gate/up tail it overlaps for HBM, none
//    leaves the ring to fill after the wait.  Calls, us (Q4 / bf16 / e4m3 /
//    Q8_0): whole ring 36.9 / 62.2 / 36.3 / 37.7; ring less one 37.0 / 61.4
//    / 36.0 / 37.0 (Q4's ring has four stages, the others three); one stage
//    37.5 / 62.0 / 36.7 / 37.6; none 39.3 / 62.9 / 37.3 / 38.9.
// FFN_NORM_RELEASE_EARLY, FFN_PRE_STAGES_GATEUP and FFN_PRE_STAGES_DOWN in the
// environment override them (read once per process, for measurement).
int decode_tuning(int knob) {
    static int v[TUNE_COUNT];
    static bool read[TUNE_COUNT];
    static const char *names[TUNE_COUNT] = {"FFN_NORM_RELEASE_EARLY", "FFN_PRE_STAGES_GATEUP", "FFN_PRE_STAGES_DOWN",
                                            "FFN_NORM_SLICES"};
    static const int defaults[TUNE_COUNT] = {1, 1, -1, 1};
    if (!read[knob]) {
        const char *e = getenv(names[knob]);
        v[knob] = e ? std::max(0, atoi(e)) : defaults[knob];
        read[knob] = true;
    }
    return v[knob];
}

bool stream_supported(int wfmt, int64_t d, int64_t ffn) {
    if (wfmt == WF_Q4) return d % 256 == 0 && ffn % 256 == 0;
    if (wfmt == WF_FP8) return d % 256 == 0 && ffn % 256 == 0;
    if (wfmt == WF_Q8) return d % 256 == 0 && ffn % 256 == 0;
    return d % 8 == 0 && ffn % 8 == 0;
}

template <int WF, int NT, bool TWO>
cudaError_t launch_stream_gateup(GemvWeights wg, GemvWeights wu, const void *nfrag, const void *nfrag_lo,
                                 void *hfrag, void *hfrag_lo, int64_t d, int64_t ffn, int64_t nchK,
                                 int64_t nchF, unsigned *counters, int ncounters, const float *ncorr, float *hcorr,
                                 cudaStream_t s) {
    using TL = Tile<WF, ROLE_GATEUP, NT, TWO, WF == WF_Q4>;
    constexpr auto kern = gemv_stream_kernel<WF, NT, TWO, ROLE_GATEUP>;
    cudaError_t e = set_smem<kern>(TL::smem_bytes);
    if (e != cudaSuccess) return e;
    CUtensorMap w0, w1, s0, s1;
    if (!weight_maps<WF, ROLE_GATEUP>(&w0, &s0, wg, ffn, d) || !weight_maps<WF, ROLE_GATEUP>(&w1, &s1, wu, ffn, d))
        return cudaErrorInvalidValue;
    StreamParams p{};
    p.K = d;
    p.rows_w = ffn;
    p.nkb = cdiv(d, TL::kb);
    p.kb_per_split = p.nkb;
    p.bfrag = static_cast<const uint4 *>(nfrag);
    p.bfrag_lo = static_cast<const uint4 *>(nfrag_lo);
    p.nch_b = nchK;
    p.hfrag = static_cast<uint16_t *>(hfrag);
    p.hfrag_lo = static_cast<uint16_t *>(hfrag_lo);
    p.nch_h = nchF;
    p.counters = counters;
    p.ncounters = ncounters;
    p.err = device_status_word();
    if (!p.err) return cudaErrorUnknown;
    p.res = nullptr;
    p.rs0 = wg.rs;
    p.rs1 = wu.rs;
    p.bcorr = ncorr;
    p.hcorr = hcorr;
    p.pre_stages = decode_tuning(TUNE_PRE_STAGES_GATEUP);
    // 32 features per CTA; covering nchF * 32 features writes every slot of h
    const int64_t blocks = nchF;
    LaunchScope scope(K_GEMV_GATEUP, s);
    e = launch_dependent(kern, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), TL::smem_bytes, s, w0, w1,
                         s0, s1, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int WF, int NT, bool TWO>
cudaError_t launch_stream_down(GemvWeights wd, const void *hfrag, const void *hfrag_lo, void *y,
                               float *partials, unsigned *counters, int rows, int64_t d, int64_t ffn,
                               int64_t nchF, int64_t splits, const void *res, float *ss_part, float *y_sumsq,
                               const float *hcorr, cudaStream_t s) {
    using TL = Tile<WF, ROLE_DOWN, NT, TWO, WF == WF_Q4>;
    constexpr auto kern = gemv_stream_kernel<WF, NT, TWO, ROLE_DOWN>;
    cudaError_t e = set_smem<kern>(TL::smem_bytes);
    if (e != cudaSuccess) return e;
    CUtensorMap w0, s0;
    if (!weight_maps<WF, ROLE_DOWN>(&w0, &s0, wd, d, ffn)) return cudaErrorInvalidValue;
    StreamParams p{};
    p.K = ffn;
    p.rows_w = d;
    p.nkb = cdiv(ffn, TL::kb);
    p.kb_per_split = cdiv(p.nkb, splits);
    (void)nchF;
    p.bfrag = static_cast<const uint4 *>(hfrag);
    p.bfrag_lo = static_cast<const uint4 *>(hfrag_lo);
    p.nch_b = nchF;
    p.y = y;
    p.partials = partials;
    p.counters = counters;
    p.rows = rows;
    p.D = d;
    p.res = res;
    p.rs0 = wd.rs;
    p.rs1 = nullptr;
    const int pre = decode_tuning(TUNE_PRE_STAGES_DOWN);
    p.pre_stages = pre < 0 ? TL::stages - 1 : pre;   // (default: the ring less one stage)
    p.ss_part = ss_part;
    p.y_sumsq = y_sumsq;
    p.bcorr = hcorr;
    p.err = device_status_word();
    if (!p.err) return cudaErrorUnknown;
    const int64_t nsplit = cdiv(p.nkb, p.kb_per_split);
    dim3 grid(static_cast<unsigned>(cdiv(d, 64)), static_cast<unsigned>(nsplit));
    LaunchScope scope(K_GEMV_DOWN, s);
    e = launch_dependent(kern, grid, dim3(kThreads), TL::smem_bytes, s, w0, w0, s0, s0, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Down-projection CTAs that fit in one wave: the CTAs per SM that the
// format's ring allows (its shared memory plus ~3 KB of static and reserved
// shared memory, out of 228 KB; Q4: its ring of block offsets, and 1.5 KB,
// its epilogue scratch living in the ring) times 152 SMs, less a small
// margin.
template <int WF>
constexpr int64_t down_cta_budget() {
    constexpr size_t per_cta = WF == WF_Q4 ? Tile<WF, ROLE_DOWN, 1, false, true>::smem_bytes + 1536
                                           : Tile<WF, ROLE_DOWN, 1, false>::smem_bytes + 3 * 1024;
    return 152 * static_cast<int64_t>((228 * 1024) / per_cta) - 8;
}

// Down-projection splits for the streaming kernel: at most one wave of CTAs
// of 64 rows (600 with the four CTAs per SM of most formats, 448 for Q8_0's
// larger ring), never finer than one k-block.  A function of the shape
// alone, so workspace queries agree with launches.
int64_t stream_down_splits(int wfmt, int64_t d, int64_t ffn) {
    const int64_t groups = cdiv(d, 64);
    const int64_t kb = (wfmt == WF_Q4 || wfmt == WF_Q8 || wfmt == WF_FP8) ? 256 : 128;
    const int64_t nkb = cdiv(ffn, kb);
    const int64_t budget = wfmt == WF_Q8 ? down_cta_budget<WF_Q8>() : wfmt == WF_Q4 ? down_cta_budget<WF_Q4>()
                         : wfmt == WF_FP8 ? down_cta_budget<WF_FP8>() : down_cta_budget<WF_BF16>();
    int64_t splits = budget / groups;
    if (splits < 1) splits = 1;
    if (splits > nkb) splits = nkb;
    return cdiv(nkb, cdiv(nkb, splits));   // the splits the kernel will actually run
}

#define FFN_STREAM_INSTANTIATE(WF, NT, TWO)                                                            \
    template cudaError_t launch_stream_gateup<WF, NT, TWO>(GemvWeights, GemvWeights, const void *,      \
                                                           const void *, void *, void *, int64_t,       \
                                                           int64_t, int64_t, int64_t, unsigned *, int,   \
                                                           const float *, float *, cudaStream_t);        \
    template cudaError_t launch_stream_down<WF, NT, TWO>(GemvWeights, const void *, const void *, void *, \
                                                         float *, unsigned *, int, int64_t, int64_t,     \
                                                         int64_t, int64_t, const void *, float *, float *, \
                                                         const float *, cudaStream_t);
FFN_STREAM_INSTANTIATE(WF_F16, 1, false)
FFN_STREAM_INSTANTIATE(WF_F16, 2, false)
FFN_STREAM_INSTANTIATE(WF_F16, 1, true)
FFN_STREAM_INSTANTIATE(WF_F16, 2, true)
FFN_STREAM_INSTANTIATE(WF_BF16, 1, false)
FFN_STREAM_INSTANTIATE(WF_BF16, 2, false)
FFN_STREAM_INSTANTIATE(WF_BF16, 1, true)
FFN_STREAM_INSTANTIATE(WF_BF16, 2, true)
FFN_STREAM_INSTANTIATE(WF_Q4, 1, false)
FFN_STREAM_INSTANTIATE(WF_Q4, 2, false)
FFN_STREAM_INSTANTIATE(WF_F16P, 1, false)
FFN_STREAM_INSTANTIATE(WF_F16P, 2, false)
// four and eight token tiles (17 to 64 rows): 16-bit weights only
FFN_STREAM_INSTANTIATE(WF_F16, 4, false)
FFN_STREAM_INSTANTIATE(WF_F16, 8, false)
FFN_STREAM_INSTANTIATE(WF_F16, 4, true)
FFN_STREAM_INSTANTIATE(WF_F16, 8, true)
FFN_STREAM_INSTANTIATE(WF_BF16, 4, false)
FFN_STREAM_INSTANTIATE(WF_BF16, 8, false)
FFN_STREAM_INSTANTIATE(WF_BF16, 4, true)
FFN_STREAM_INSTANTIATE(WF_BF16, 8, true)
FFN_STREAM_INSTANTIATE(WF_F16P, 4, false)
FFN_STREAM_INSTANTIATE(WF_F16P, 8, false)
FFN_STREAM_INSTANTIATE(WF_FP8, 1, false)
FFN_STREAM_INSTANTIATE(WF_FP8, 2, false)
FFN_STREAM_INSTANTIATE(WF_Q8, 1, false)
FFN_STREAM_INSTANTIATE(WF_Q8, 2, false)
#undef FFN_STREAM_INSTANTIATE

}  // namespace gemv
}  // namespace ffn
