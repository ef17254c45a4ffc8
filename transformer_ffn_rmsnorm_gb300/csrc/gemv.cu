// gemv.cu -- the FFN block for few token rows (decode): weight streaming.
//
// With at most 16 token rows every weight byte is used for at most 16
// multiply-adds, far below the GB300's ridge point, so the time is the HBM
// stream of W_gate, W_up and W_down ("Megakernels on Mac: What Fusion Saves and What It Costs", section
// "Projection shape changes the achieved rate": eight-row projections, and
// a deeper K split for the long-K down projection).  Design:
//
// * The weights are the M side of a warp-level m16n8k16 tensor-core MMA and
//   the (<= 8 per n-tile) token rows are the N side, so no MMA lane is wasted
//   on padding.  Each lane loads 16 contiguous weight bytes per row straight
//   from HBM into the A fragment.  Because K is only summed over, the k
//   index inside one MMA can be permuted freely as long as A and B agree;
//   the activations are therefore pre-arranged once per call ("fragment
//   order") so that each lane's B operand is one 16-byte load.  fp32 FFMA
//   would need 8-16 issue slots per weight pair at these row counts, about
//   as long as the weight stream itself; the MMA needs one per 256 weights.
// * Q4 weights ("Unfusing a Kernel Made It 1.63x Faster", section "The
//   finding that keeps us honest about microbenchmarks": repacked so every
//   block is read once, coalesced; "Megakernels on Mac: What Fusion Saves and What It Costs", section
//   "Threadgroup staging": no shared-memory staging) are dequantised in
//   registers: nibbles become (u - 8) exactly in bf16, one block's two MMAs
//   accumulate into a fresh fp32 fragment, and the block scale multiplies
//   that fragment (w = (u - 8) * s applied exactly in fp32).
// * gate/up: 4 warps split K for each 16-feature tile and combine their
//   partial fragments in shared memory in a fixed order; the epilogue applies
//   silu(G)*U and writes h already in the down projection's fragment order.
// * down: K (= ffn) is split across CTAs; each CTA writes fp32 partials and
//   the last CTA to arrive for a feature group sums the partials in split
//   order and writes y.  No CTA ever waits for another, and the sum order is
//   fixed, so results are bitwise reproducible.
#include <algorithm>

#include "gemv_common.cuh"

namespace ffn {
namespace {

using namespace gemv;
constexpr int kSplitK = 2048;           // down projection: k values per CTA split
constexpr int kGuKS = 4;                // gate/up: warps along K per tile
constexpr int kGuTPC = 2;               // gate/up: 16-feature tiles per CTA
constexpr int kDnTPC = 4;               // down: 16-feature tiles per CTA (one per warp)
constexpr int kDnFeat = 16 * kDnTPC;    // features per down CTA

// ---------------------------------------------------------------------------
// 1. RMSNorm of <= 16 token rows, written in fragment order.
//
// Sum over the CTA (256 threads) of every thread's v, returned to all.
__device__ __forceinline__ float cta_sum256(float v, float (&partial)[8]) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) partial[threadIdx.x >> 5] = v;
    __syncthreads();
    v = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += partial[w];
    return v;
}

// grid = (token slots, slices): every CTA reads its token's row (VPT
// 16-byte vectors of x per thread) for the sum of squares, and with it, in
// the same round trip, x and g of its slice of whole 32-value blocks (at
// most one 8-value group per thread); then the reciprocal root and the
// slice's fragments.  Slots >= rows (and k >= K) are written as zeros.  The
// call's first kernel: it waits for the kernel before it, then lets the
// projection kernel after it start its weight stream, at once
// (release_early) or when it has finished (its reads then do not queue
// behind that stream).  Slices: as few as give every thread one group at
// most (FFN_NORM_SLICES asks for more; 2 to 8 a token measured the same
// per call for bf16, e4m3, Q8_0 and Q4 blocks).
// With BIAS (Q4 for the streaming kernels) the fragments take the biased
// form (store_group_q4_biased) and each block's offset goes to corr: a
// block's four 8-value groups sit on four adjacent lanes.
template <int WF, bool TWO, int VPT, bool BIAS>
__global__ void __launch_bounds__(256) gemv_norm_frag_reg_kernel(const void *x_, const void *g_,
                                                                 uint16_t *nfrag, uint16_t *nlo, int rows,
                                                                 int64_t K, int64_t nch, float eps,
                                                                 int release_early, const float *ss_in,
                                                                 float *corr) {
    using T = typename Fmt<WF>::TIn;
    __shared__ float partial[8];
    ptx::griddep_wait();
    if (release_early) ptx::griddep_launch_dependents();
    const int token = blockIdx.x;
    const int64_t nv = K / 8;
    const int64_t v0 = 4 * (nch * blockIdx.y / gridDim.y), v1 = 4 * (nch * (blockIdx.y + 1) / gridDim.y);
    const uint4 *x = reinterpret_cast<const uint4 *>(static_cast<const T *>(x_) + static_cast<int64_t>(token) * K);
    const uint4 *g = static_cast<const uint4 *>(g_);
    const bool live = token < rows;
    uint4 xv[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int64_t v = threadIdx.x + 256 * i;
        xv[i] = (live && !ss_in && v < nv) ? x[v] : make_uint4(0, 0, 0, 0);
    }
    const int64_t vs = v0 + threadIdx.x;   // this thread's group of the slice
    const bool in = vs < v1, ld = live && in && vs < nv;
    const uint4 xs = ld ? x[vs] : make_uint4(0, 0, 0, 0), gs = ld ? g[vs] : make_uint4(0, 0, 0, 0);
    float ss = 0.f;
    if (ss_in) {   // the row's sum of squares, handed on by the block before
        ss = live ? ss_in[token] : 0.f;
    } else {
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            float f[8];
            Vec16<T>::unpack(xv[i], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
        }
        ss = cta_sum256(ss, partial);
    }
    const float inv = rsqrtf(ss / static_cast<float>(K) + eps);
    float f[8], gf[8];
    Vec16<T>::unpack(xs, f);
    Vec16<T>::unpack(gs, gf);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = f[e] * inv * gf[e];
    if constexpr (BIAS) {
        // (v0 and v1 are multiples of 4: a lane quad is in or out as a whole)
        float part = in ? store_group_q4_biased(nfrag, nch, token, 8 * vs, f) : 0.f;
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (in && (vs & 3) == 0) store_q4_corr(corr, gridDim.x / 8, token, vs >> 2, part);
    } else if (in) {
        store_group<WF, TWO>(nfrag, nlo, nch, token, 8 * vs, f);
    }
}

// The same for rows too long for registers (d > 16384): grid = (token slots,
// slices); every CTA reduces its token's whole row and writes one slice.
template <int WF, bool TWO, bool BIAS>
__global__ void __launch_bounds__(256) gemv_norm_frag_kernel(const void *x_, const void *g_,
                                                             uint16_t *nfrag, uint16_t *nlo,
                                                             int rows, int64_t K, int64_t nch,
                                                             float eps, const float *ss_in, float *corr) {
    using T = typename Fmt<WF>::TIn;
    __shared__ float partial[8];
    // launched as a programmatic dependent: nothing is read or written before
    // the previous kernel has finished; only then may the projection kernel
    // after this one start its weight stream (weights that kernel may have written)
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int token = blockIdx.x;
    const T *x = static_cast<const T *>(x_) + static_cast<int64_t>(token) * K;
    const T *g = static_cast<const T *>(g_);
    // slices of whole 32-value blocks (four 8-element groups), the zero tail included
    const int64_t v0 = 4 * (nch * blockIdx.y / gridDim.y), v1 = 4 * (nch * (blockIdx.y + 1) / gridDim.y);
    const int64_t nv = K / 8;
    float ss = 0.f;
    if (token < rows) {
        for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
            float f[8];
            Vec16<T>::unpack(reinterpret_cast<const uint4 *>(x)[v], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
        }
    }
    ss = cta_sum256(ss, partial);
    if (ss_in) ss = token < rows ? ss_in[token] : 0.f;
    const float inv = rsqrtf(ss / static_cast<float>(K) + eps);
    // every thread takes the same number of turns (the biased form reduces
    // over lane quads)
    for (int64_t vb = v0; vb < v1; vb += blockDim.x) {
        const int64_t v = vb + threadIdx.x;
        float f[8];
        if (token < rows && v < nv && v < v1) {
            float gf[8];
            Vec16<T>::unpack(reinterpret_cast<const uint4 *>(x)[v], f);
            Vec16<T>::unpack(reinterpret_cast<const uint4 *>(g)[v], gf);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = f[e] * inv * gf[e];
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = 0.f;
        }
        if constexpr (BIAS) {
            float part = v < v1 ? store_group_q4_biased(nfrag, nch, token, 8 * v, f) : 0.f;
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            if (v < v1 && (v & 3) == 0) store_q4_corr(corr, gridDim.x / 8, token, v >> 2, part);
        } else if (v < v1) {
            store_group<WF, TWO>(nfrag, nlo, nch, token, 8 * v, f);
        }
    }
}

// ---------------------------------------------------------------------------
// Accumulate RT row tiles (16 weight rows each) x NT token tiles over a
// range of K for one warp.  For f16/bf16, [c0, c1) are 32-wide chunks; for
// Q4, [c0, c1) are 128-wide groups (four blocks; a row holds ceil(K / 128),
// the padding of a last, partial group being zero bytes and zero scales that
// meet zero activations).
// With TWO, the activation operand is given as two fragments (value and
// rounding residual) and every weight fragment is multiplied by both.
template <int WF, int RT, int NT, int U, bool TWO>
__device__ __forceinline__ void warp_accumulate(const void *const (&w)[RT],
                                                const uint16_t *const (&sc)[RT],
                                                const int64_t (&row)[RT][2],
                                                const bool (&rowok)[RT][2], int64_t K,
                                                const uint4 *__restrict__ bfrag,
                                                const uint4 *__restrict__ bfrag_lo, int64_t nch,
                                                int64_t c0, int64_t c1, float (&acc)[RT][NT][4]) {
    constexpr bool bf = Fmt<WF>::op_bf16;
    const int lane = threadIdx.x & 31, tid = lane & 3;
    if constexpr (WF != WF_Q4) {
        const uint16_t *W[RT];
#pragma unroll
        for (int r = 0; r < RT; ++r) W[r] = static_cast<const uint16_t *>(w[r]);
        for (int64_t c = c0; c < c1; c += U) {
            uint4 a[U][RT][2], b[U][NT], bl[U][TWO ? NT : 1];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t cc = c + u;
                const int64_t k = cc * kChunk + 8 * tid;
                const bool ok = cc < c1 && k < K;
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        a[u][r][h] = (ok && rowok[r][h]) ? ptx::ld_stream_v4(W[r] + row[r][h] * K + k)
                                                         : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    b[u][n] = (cc < c1) ? __ldg(bfrag + (n * nch + cc) * 32 + lane) : make_uint4(0, 0, 0, 0);
                    if constexpr (TWO)
                        bl[u][n] = (cc < c1) ? __ldg(bfrag_lo + (n * nch + cc) * 32 + lane)
                                             : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        ptx::mma_16816<bf>(acc[r][n], a[u][r][0].x, a[u][r][1].x, a[u][r][0].y,
                                           a[u][r][1].y, b[u][n].x, b[u][n].y);
                        ptx::mma_16816<bf>(acc[r][n], a[u][r][0].z, a[u][r][1].z, a[u][r][0].w,
                                           a[u][r][1].w, b[u][n].z, b[u][n].w);
                        if constexpr (TWO) {
                            ptx::mma_16816<bf>(acc[r][n], a[u][r][0].x, a[u][r][1].x, a[u][r][0].y,
                                               a[u][r][1].y, bl[u][n].x, bl[u][n].y);
                            ptx::mma_16816<bf>(acc[r][n], a[u][r][0].z, a[u][r][1].z, a[u][r][0].w,
                                               a[u][r][1].w, bl[u][n].z, bl[u][n].w);
                        }
                    }
        }
    } else {
        const int64_t qrow = cdiv(K, 128) * 64;   // bytes per weight row
        const int64_t srow = cdiv(K, 128) * 4;    // scales per weight row
        for (int64_t gi = c0; gi < c1; gi += U) {
            uint4 q[U][RT][2];
            uint2 s[U][RT][2];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t gg = gi + u;
                const bool ok = gg < c1;
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const bool live = ok && rowok[r][h];
                        const uint8_t *qp = static_cast<const uint8_t *>(w[r]) + row[r][h] * qrow + gg * 64 + 16 * tid;
                        q[u][r][h] = live ? ptx::ld_stream_v4(qp) : make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
                        s[u][r][h] = live ? ptx::ld_stream_v2(sc[r] + row[r][h] * srow + gg * 4) : make_uint2(0, 0);
                    }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t gg = gi + u;
                if (gg >= c1) break;
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    uint4 b[NT], bl[TWO ? NT : 1];
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        b[n] = __ldg(bfrag + (n * nch + gg * 4 + blk) * 32 + lane);
                        if constexpr (TWO) bl[n] = __ldg(bfrag_lo + (n * nch + gg * 4 + blk) * 32 + lane);
                    }
#pragma unroll
                    for (int r = 0; r < RT; ++r) {
                        uint32_t lo[4], hi[4];
                        dequant_word(word_of(q[u][r][0], blk), lo);
                        dequant_word(word_of(q[u][r][1], blk), hi);
                        const uint32_t s0 = (blk < 2 ? s[u][r][0].x : s[u][r][0].y) >> (16 * (blk & 1));
                        const uint32_t s1 = (blk < 2 ? s[u][r][1].x : s[u][r][1].y) >> (16 * (blk & 1));
                        const float f0 = __half2float(__ushort_as_half(static_cast<unsigned short>(s0 & 0xFFFFu)));
                        const float f1 = __half2float(__ushort_as_half(static_cast<unsigned short>(s1 & 0xFFFFu)));
#pragma unroll
                        for (int n = 0; n < NT; ++n) {
                            float t[4];   // this block's products alone, scaled below
                            ptx::mma_16816_z<bf>(t, lo[0], hi[0], lo[2], hi[2], b[n].x, b[n].y);
                            ptx::mma_16816<bf>(t, lo[1], hi[1], lo[3], hi[3], b[n].z, b[n].w);
                            if constexpr (TWO) {
                                ptx::mma_16816<bf>(t, lo[0], hi[0], lo[2], hi[2], bl[n].x, bl[n].y);
                                ptx::mma_16816<bf>(t, lo[1], hi[1], lo[3], hi[3], bl[n].z, bl[n].w);
                            }
                            acc[r][n][0] = fmaf(f0, t[0], acc[r][n][0]);
                            acc[r][n][1] = fmaf(f0, t[1], acc[r][n][1]);
                            acc[r][n][2] = fmaf(f1, t[2], acc[r][n][2]);
                            acc[r][n][3] = fmaf(f1, t[3], acc[r][n][3]);
                        }
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 2. gate/up: h = silu(W_gate n) * (W_up n), written in fragment order for
//    the down projection.  CTA = kGuTPC tiles x kGuKS warps along K.
template <int WF, int NT, bool TWO>
__global__ void __launch_bounds__(256) gemv_gateup_kernel(
    const void *wg, const void *wu, const uint16_t *sg, const uint16_t *su,
    const uint4 *__restrict__ nfrag, const uint4 *__restrict__ nfrag_lo, uint16_t *hfrag,
    uint16_t *hfrag_lo, int64_t K, int64_t F, int64_t nchK, int64_t nchF, int64_t nunits,
    unsigned *counters, int ncounters) {
    using TO = typename Fmt<WF>::TOp;
    constexpr bool q4 = WF == WF_Q4;
    constexpr int U = q4 ? 2 : 4;
    __shared__ float red[kGuTPC][kGuKS - 1][32][2 * NT * 4];
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < ncounters; i += blockDim.x) counters[i] = 0u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tl = warp / kGuKS, ks = warp % kGuKS;
    const int64_t tile = static_cast<int64_t>(blockIdx.x) * kGuTPC + tl;
    const int64_t f0 = tile * 16;
    const int gq = lane >> 2, tid = lane & 3;
    const int64_t c0 = nunits * ks / kGuKS, c1 = nunits * (ks + 1) / kGuKS;

    const void *const w[2] = {wg, wu};
    const uint16_t *const sc[2] = {sg, su};
    int64_t row[2][2];
    bool rowok[2][2];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            row[r][h] = f0 + gq + 8 * h;
            rowok[r][h] = row[r][h] < F;
        }
    float acc[2][NT][4];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[r][n][i] = 0.f;
    warp_accumulate<WF, 2, NT, U, TWO>(w, sc, row, rowok, K, nfrag, nfrag_lo, nchK, c0, c1, acc);

    if (ks > 0) {
        float *dst = red[tl][ks - 1][lane];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[(r * NT + n) * 4 + i] = acc[r][n][i];
    }
    __syncthreads();
    if (ks != 0) return;
#pragma unroll
    for (int j = 0; j < kGuKS - 1; ++j) {
        const float *src = red[tl][j][lane];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[r][n][i] += src[(r * NT + n) * 4 + i];
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t feat = f0 + gq + 8 * (i >> 1);
            const int token = 8 * n + 2 * tid + (i & 1);
            constexpr float ws = Fmt<WF>::w_unscale;
            const float hv = silu_f32(acc[0][n][i] * ws) * (acc[1][n][i] * ws) * Fmt<WF>::h_scale;
            const TO t = from_f32<TO>(hv);
            const int64_t at = frag_elem(frag_order<WF>(), nchF, token, feat);
            hfrag[at] = *reinterpret_cast<const uint16_t *>(&t);
            if (TWO) {
                const TO tl = from_f32<TO>(hv - to_f32(t));
                hfrag_lo[at] = *reinterpret_cast<const uint16_t *>(&tl);
            }
        }
}

// ---------------------------------------------------------------------------
// 3. down: y = W_down h.  grid = (feature groups of 64, K splits).
template <int WF, int NT, bool TWO>
__global__ void __launch_bounds__(128) gemv_down_kernel(
    const void *wd, const uint16_t *sd, const uint4 *__restrict__ hfrag,
    const uint4 *__restrict__ hfrag_lo, void *y_, float *partials,
    unsigned *counters, int rows, int64_t D, int64_t F, int64_t nchF, int64_t units_per_split,
    const void *res, float *ss_part, float *y_sumsq) {
    using T = typename Fmt<WF>::TIn;
    constexpr bool q4 = WF == WF_Q4;
    constexpr int U = q4 ? 2 : 8;
    constexpr float out_scale = Fmt<WF>::w_unscale / Fmt<WF>::h_scale;
    __shared__ int s_last, s_last_row;
    __shared__ float sq[16 * kDnFeat];   // stored y squared (rows <= 16 on this path)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tid = lane & 3;
    const int64_t f0 = (static_cast<int64_t>(blockIdx.x) * kDnTPC + warp) * 16;
    const int split = blockIdx.y, nsplit = gridDim.y;
    const int64_t nunits = q4 ? cdiv(F, 128) : nchF;
    const int64_t c0 = split * units_per_split;
    const int64_t c1 = (c0 + units_per_split < nunits) ? c0 + units_per_split : nunits;

    const void *const w[1] = {wd};
    const uint16_t *const sc[1] = {sd};
    int64_t row[1][2];
    bool rowok[1][2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        row[0][h] = f0 + gq + 8 * h;
        rowok[0][h] = row[0][h] < D;
    }
    float acc[1][NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[0][n][i] = 0.f;
    warp_accumulate<WF, 1, NT, U, TWO>(w, sc, row, rowok, F, hfrag, hfrag_lo, nchF, c0, c1, acc);

#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t feat = f0 + gq + 8 * (i >> 1);
            const int token = 8 * n + 2 * tid + (i & 1);
            if (token < rows && feat < D)
                partials[(static_cast<int64_t>(split) * rows + token) * D + feat] = acc[0][n][i];
        }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&counters[blockIdx.x], 1u) == static_cast<unsigned>(nsplit - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    T *y = static_cast<T *>(y_);
    const int64_t fbase = static_cast<int64_t>(blockIdx.x) * kDnFeat;
    for (int i = threadIdx.x; i < rows * kDnFeat; i += blockDim.x) {
        const int token = i / kDnFeat;
        const int64_t feat = fbase + i % kDnFeat;
        if (feat >= D) continue;
        float sum = 0.f;
        for (int sp = 0; sp < nsplit; ++sp)
            sum += __ldcg(partials + (static_cast<int64_t>(sp) * rows + token) * D + feat);
        float v = sum * out_scale;
        if (res) v += to_f32(static_cast<const T *>(res)[static_cast<int64_t>(token) * D + feat]);
        const T yv = from_f32<T>(v);
        y[static_cast<int64_t>(token) * D + feat] = yv;
        const float r = to_f32(yv);
        sq[i] = r * r;
    }
    if (threadIdx.x == 0) counters[blockIdx.x] = 0u;
    if (!y_sumsq) return;
    // the row's sum of squares of the stored y ("Megakernels on Mac: What
    // Fusion Saves and What It Costs", "Dependencies and synchronization"):
    // this group's part, then the last group adds the parts in group order
    __syncthreads();
    const int64_t nf = D - fbase < kDnFeat ? D - fbase : kDnFeat;
    if (threadIdx.x < rows) {
        float ss = 0.f;
        for (int j = 0; j < nf; ++j) ss += sq[threadIdx.x * kDnFeat + j];
        ss_part[static_cast<int64_t>(blockIdx.x) * rows + threadIdx.x] = ss;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last_row = atomicAdd(&counters[gridDim.x], 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last_row) return;
    __threadfence();
    if (threadIdx.x < rows) {
        float ss = 0.f;
        for (unsigned gi = 0; gi < gridDim.x; ++gi) ss += __ldcg(ss_part + static_cast<int64_t>(gi) * rows + threadIdx.x);
        y_sumsq[threadIdx.x] = ss;
    }
    if (threadIdx.x == 0) counters[gridDim.x] = 0u;
}

// ---------------------------------------------------------------------------
struct Geometry {
    int nt;            // token tiles of 8
    int64_t nchK;      // chunks of 32 along d (gate/up K)
    int64_t nchF;      // chunks of 32 along ffn (down K)
    int64_t splits;    // down-projection K splits
    int64_t ups;       // units (chunks or Q4 groups) per split
    int64_t groups;    // down feature groups of 64
};

Geometry geometry(int64_t rows, int64_t d, int64_t ffn, bool q4) {
    Geometry g;
    g.nt = rows <= 8 ? 1 : rows <= 16 ? 2 : rows <= 32 ? 4 : 8;   // token tiles of 8 (16-bit weights: up to 8)
    // (Q4 rows hold whole 128-wide groups: the chunk counts round up to them,
    // the chunks past K being zeros)
    g.nchK = q4 ? 4 * cdiv(d, 128) : cdiv(d, kChunk);
    g.nchF = q4 ? 4 * cdiv(ffn, 128) : cdiv(ffn, kChunk);
    g.ups = q4 ? kSplitK / 128 : kSplitK / kChunk;
    const int64_t units = q4 ? cdiv(ffn, 128) : g.nchF;
    g.splits = cdiv(units, g.ups);
    g.groups = cdiv(d, kDnFeat);
    return g;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// The call's norm kernel: one CTA per token slot holding its row in
// registers, or (rows past 16384 values) slices of the row per CTA.
template <int WF, bool TWO, bool BIAS, int NT>
cudaError_t launch_norm(const void *x, const void *gain, int rows, int64_t d, float eps, const GemvWorkspace &ws,
                        const Geometry &geo, cudaStream_t s, RowStats rs) {
    uint16_t *nf = static_cast<uint16_t *>(ws.nfrag), *nl = static_cast<uint16_t *>(ws.nfrag_lo);
    const int64_t vpt = cdiv(geo.nchK * 4, 256);   // 16-byte vectors of the row per thread
    // slices a token: at least one 8-value group a thread, at most one block a slice
    int64_t slices = std::max<int64_t>(decode_tuning(TUNE_NORM_SLICES), vpt);
    slices = std::max<int64_t>(1, std::min<int64_t>(slices, geo.nchK));
    const dim3 grid(8 * NT, static_cast<unsigned>(slices));
    const int early = decode_tuning(TUNE_NORM_RELEASE_EARLY);
    if (vpt <= 1)
        return launch_dependent(gemv_norm_frag_reg_kernel<WF, TWO, 1, BIAS>, grid, dim3(256), 0, s, x, gain, nf, nl,
                                rows, d, geo.nchK, eps, early, rs.ss_in, ws.ncorr);
    if (vpt <= 2)
        return launch_dependent(gemv_norm_frag_reg_kernel<WF, TWO, 2, BIAS>, grid, dim3(256), 0, s, x, gain, nf, nl,
                                rows, d, geo.nchK, eps, early, rs.ss_in, ws.ncorr);
    if (vpt <= 4)
        return launch_dependent(gemv_norm_frag_reg_kernel<WF, TWO, 4, BIAS>, grid, dim3(256), 0, s, x, gain, nf, nl,
                                rows, d, geo.nchK, eps, early, rs.ss_in, ws.ncorr);
    if (vpt <= 8)
        return launch_dependent(gemv_norm_frag_reg_kernel<WF, TWO, 8, BIAS>, grid, dim3(256), 0, s, x, gain, nf, nl,
                                rows, d, geo.nchK, eps, early, rs.ss_in, ws.ncorr);
    return launch_dependent(gemv_norm_frag_kernel<WF, TWO, BIAS>,
                            dim3(8 * NT, static_cast<unsigned>(std::min<int64_t>(16, cdiv(vpt, 4)))), dim3(256), 0, s,
                            x, gain, nf, nl, rows, d, geo.nchK, eps, rs.ss_in, ws.ncorr);
}

template <int WF, int NT, bool TWO>
cudaError_t launch_typed(const void *x, const void *gain, GemvWeights wg, GemvWeights wu,
                         GemvWeights wd, void *y, int rows, int64_t d, int64_t ffn, float eps,
                         const GemvWorkspace &ws, const Geometry &geo, cudaStream_t s, const void *res,
                         RowStats rs, bool one_kernel) {
    constexpr bool q4 = WF == WF_Q4;
    if (one_kernel && stream_supported(WF, d, ffn))
        if (unsigned long long *ctl = fused_control(d, s))
            return launch_fused<WF, NT, TWO>(wg, wu, wd, x, gain, y, rows, d, ffn, eps, ws, res, rs.ss_in, rs.ss_out,
                                             ctl, s);
    {
        LaunchScope scope(K_GEMV_NORM, s);
        cudaError_t e;
        // Q4 activations for the streaming kernels take the biased form
        if constexpr (q4)
            e = stream_supported(WF, d, ffn) ? launch_norm<WF, TWO, true, NT>(x, gain, rows, d, eps, ws, geo, s, rs)
                                             : launch_norm<WF, TWO, false, NT>(x, gain, rows, d, eps, ws, geo, s, rs);
        else
            e = launch_norm<WF, TWO, false, NT>(x, gain, rows, d, eps, ws, geo, s, rs);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (stream_supported(WF, d, ffn)) {
        cudaError_t e = launch_stream_gateup<WF, NT, TWO>(wg, wu, ws.nfrag, ws.nfrag_lo, ws.hfrag, ws.hfrag_lo, d,
                                                          ffn, geo.nchK, geo.nchF, ws.counters,
                                                          static_cast<int>(geo.groups + 1), ws.ncorr, ws.hcorr, s);
        if (e != cudaSuccess) return e;
        return launch_stream_down<WF, NT, TWO>(wd, ws.hfrag, ws.hfrag_lo, y, ws.partials, ws.counters, rows, d,
                                               ffn, geo.nchF, stream_down_splits(WF, d, ffn), res, ws.ss_part,
                                               rs.ss_out, ws.hcorr, s);
    }
    if constexpr (WF == WF_FP8 || WF == WF_Q8 || NT > 2) {
        // e4m3 and Q8_0 weights, and more than two token tiles, stream through
        // the TMA kernels only
        return cudaErrorInvalidValue;
    } else {
        {
            const int64_t tiles = 2 * geo.nchF;  // covers every fragment slot of h
            const int64_t blocks = cdiv(tiles, kGuTPC);
            const int64_t units = q4 ? cdiv(d, 128) : geo.nchK;
            LaunchScope scope(K_GEMV_GATEUP, s);
            gemv_gateup_kernel<WF, NT, TWO><<<static_cast<unsigned>(blocks), 32 * kGuTPC * kGuKS, 0, s>>>(
                q4 ? static_cast<const void *>(wg.qs) : wg.w, q4 ? static_cast<const void *>(wu.qs) : wu.w,
                wg.sc, wu.sc, static_cast<const uint4 *>(ws.nfrag), static_cast<const uint4 *>(ws.nfrag_lo),
                static_cast<uint16_t *>(ws.hfrag), static_cast<uint16_t *>(ws.hfrag_lo), d, ffn, geo.nchK,
                geo.nchF, units, ws.counters, static_cast<int>(geo.groups + 1));
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        dim3 grid(static_cast<unsigned>(geo.groups), static_cast<unsigned>(geo.splits));
        LaunchScope scope(K_GEMV_DOWN, s);
        gemv_down_kernel<WF, NT, TWO><<<grid, 32 * kDnTPC, 0, s>>>(
            q4 ? static_cast<const void *>(wd.qs) : wd.w, wd.sc, static_cast<const uint4 *>(ws.hfrag),
            static_cast<const uint4 *>(ws.hfrag_lo), y, ws.partials, ws.counters, rows, d, ffn, geo.nchF,
            geo.ups, res, ws.ss_part, rs.ss_out);
        return cudaGetLastError();
    }
}

template <int WF, bool TWO>
cudaError_t launch_nt(int nt, const void *x, const void *g, GemvWeights wg, GemvWeights wu,
                      GemvWeights wd, void *y, int rows, int64_t d, int64_t ffn, float eps,
                      const GemvWorkspace &ws, const Geometry &geo, cudaStream_t s, const void *res,
                      RowStats rs, bool one_kernel) {
#define FFN_TYPED_ARGS x, g, wg, wu, wd, y, rows, d, ffn, eps, ws, geo, s, res, rs, one_kernel
    if (nt == 1) return launch_typed<WF, 1, TWO>(FFN_TYPED_ARGS);
    if (nt == 2) return launch_typed<WF, 2, TWO>(FFN_TYPED_ARGS);
    // 17 to 64 rows: 16-bit weights only (the quantised entries go in groups of 16)
    if constexpr (WF == WF_F16 || WF == WF_BF16 || WF == WF_F16P) {
        if (nt == 4) return launch_typed<WF, 4, TWO>(FFN_TYPED_ARGS);
        return launch_typed<WF, 8, TWO>(FFN_TYPED_ARGS);
    }
#undef FFN_TYPED_ARGS
    return cudaErrorInvalidValue;
}

struct Layout {
    size_t frag_n, frag_h, partials, counters, ss_part, corr_n, corr_h;
};

Layout layout(int64_t rows, int64_t d, int64_t ffn) {
    // sized for the Q4 or 16-bit geometry and for the register or streaming
    // down kernel, whichever needs most split-K partials
    const Geometry a = geometry(rows, d, ffn, false);
    const Geometry b = geometry(rows, d, ffn, (d % 32 == 0) && (ffn % 32 == 0));
    int64_t splits = a.splits > b.splits ? a.splits : b.splits;
    for (int wf : {WF_BF16, WF_Q4, WF_FP8, WF_Q8})
        if (stream_supported(wf, d, ffn)) splits = std::max(splits, stream_down_splits(wf, d, ffn));
    // (and the one-kernel decode's split partials)
    const int64_t r = rows > 64 ? 64 : rows;
    int64_t floats = splits * r * d;
    for (int wf : {WF_BF16, WF_Q4, WF_FP8, WF_Q8})
        if (stream_supported(wf, d, ffn))
            for (bool two : {false, true}) floats = std::max(floats, fused_partial_floats(wf, r, d, ffn, a.nt, two));
    Layout l;
    // (Q4 fragments cover whole 128-wide groups)
    l.frag_n = align256(static_cast<size_t>(a.nt) * std::max(a.nchK, b.nchK) * 32 * 16);
    l.frag_h = align256(static_cast<size_t>(a.nt) * std::max(a.nchF, b.nchF) * 32 * 16);
    l.partials = align256(static_cast<size_t>(floats) * 4);
    l.counters = align256(static_cast<size_t>(a.groups + 1) * 4);   // arrivals per group, then for the row sums
    l.ss_part = align256(static_cast<size_t>(a.groups) * (rows > 64 ? 64 : rows) * 4);
    l.corr_n = align256(static_cast<size_t>(q4_corr_floats(a.nt, a.nchK)) * 4);
    l.corr_h = align256(static_cast<size_t>(q4_corr_floats(a.nt, a.nchF)) * 4);
    return l;
}

}  // namespace

size_t gemv_workspace_bytes(int64_t rows, int64_t d, int64_t ffn, bool two_terms) {
    const Layout l = layout(rows, d, ffn);
    const size_t frags = l.frag_n + l.frag_h;
    return (two_terms ? 2 * frags : frags) + l.partials + l.counters + l.ss_part + l.corr_n + l.corr_h;
}

void gemv_carve(void *base, int64_t rows, int64_t d, int64_t ffn, bool two_terms, GemvWorkspace *ws) {
    const Layout l = layout(rows, d, ffn);
    char *p = static_cast<char *>(base);
    ws->nfrag = p;
    p += l.frag_n;
    ws->hfrag = p;
    p += l.frag_h;
    ws->nfrag_lo = nullptr;
    ws->hfrag_lo = nullptr;
    if (two_terms) {
        ws->nfrag_lo = p;
        p += l.frag_n;
        ws->hfrag_lo = p;
        p += l.frag_h;
    }
    ws->partials = reinterpret_cast<float *>(p);
    p += l.partials;
    ws->counters = reinterpret_cast<unsigned *>(p);
    p += l.counters;
    ws->ss_part = reinterpret_cast<float *>(p);
    p += l.ss_part;
    ws->ncorr = reinterpret_cast<float *>(p);
    p += l.corr_n;
    ws->hcorr = reinterpret_cast<float *>(p);
}

cudaError_t launch_gemv_block(int wfmt, const void *x, const void *g, GemvWeights wg,
                              GemvWeights wu, GemvWeights wd, void *y, int64_t rows, int64_t d,
                              int64_t ffn, float eps, const GemvWorkspace &ws, cudaStream_t s,
                              const void *res, RowStats rs, bool one_kernel) {
    if (rows <= 0) return cudaSuccess;
    const Geometry geo = geometry(rows, d, ffn, wfmt == WF_Q4);
    const int r = static_cast<int>(rows);
    const bool two = ws.nfrag_lo != nullptr;
#define FFN_GEMV_ARGS geo.nt, x, g, wg, wu, wd, y, r, d, ffn, eps, ws, geo, s, res, rs, one_kernel
    switch (wfmt) {
        case WF_F16:
            return two ? launch_nt<WF_F16, true>(FFN_GEMV_ARGS) : launch_nt<WF_F16, false>(FFN_GEMV_ARGS);
        case WF_BF16:
            return two ? launch_nt<WF_BF16, true>(FFN_GEMV_ARGS) : launch_nt<WF_BF16, false>(FFN_GEMV_ARGS);
        case WF_Q4:   // fp16 operands: one term is enough
            return launch_nt<WF_Q4, false>(FFN_GEMV_ARGS);
        case WF_FP8:  // fp16 operands, as for Q4
            return launch_nt<WF_FP8, false>(FFN_GEMV_ARGS);
        case WF_Q8:
            return launch_nt<WF_Q8, false>(FFN_GEMV_ARGS);
        default:      // prepared fp16 weights
            return launch_nt<WF_F16P, false>(FFN_GEMV_ARGS);
    }
#undef FFN_GEMV_ARGS
}

}  // namespace ffn
