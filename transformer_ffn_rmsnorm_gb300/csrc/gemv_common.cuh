// gemv_common.cuh -- pieces shared by the decode (few-row) kernels.
#pragma once

#include "ffn_internal.cuh"

namespace ffn {
namespace gemv {

constexpr int kChunk = 32;   // k values per MMA pair

__host__ __device__ inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Fragment order of an activation vector of length K for one token:
//   16-bit element index = ((nt * nch + c) * 32 + lane) * 8 + slot
//   lane = 4 * (token % 8) + tid, nt = token / 8.
// Natural order (f16/bf16 weights): c = k / 32, k % 32 = 8 * tid + slot.
// Q4 order: c = k / 32; position p = k % 32, hi = p / 16, q = p % 16,
//   tid = q / 4, slot = 4 * hi + perm[q % 4] with perm = {0, 2, 1, 3}; this
//   matches the nibble unpacking in dequant_word below.
// e4m3 order: groups of 64 k, one group = two chunks; position p = k % 64,
//   tid = p / 16, j = p % 16, c = 2 * (k / 64) + j / 8, slot = j % 8.  A
//   lane reads 16 consecutive weight bytes of a row (k = 16 tid .. 16 tid +
//   15 of the group) and feeds four MMAs with them, four k each; its B
//   values for those MMAs are these 16 k in order, split over the group's
//   two chunks.
enum { FRAG_NATURAL = 0, FRAG_Q4 = 1, FRAG_FP8 = 2 };
template <int WF> __host__ __device__ constexpr int frag_order() {
    return WF == WF_Q4 ? FRAG_Q4 : WF == WF_FP8 ? FRAG_FP8 : FRAG_NATURAL;
}
__device__ __forceinline__ int64_t frag_elem(int order, int64_t nch, int token, int64_t k) {
    int64_t c;
    int tid, slot;
    if (order == FRAG_FP8) {
        const int p = static_cast<int>(k & 63), j = p & 15;
        tid = p >> 4;
        c = 2 * (k >> 6) + (j >> 3);
        slot = j & 7;
    } else {
        c = k / kChunk;
        const int p = static_cast<int>(k % kChunk);
        if (order == FRAG_Q4) {
            const int hi = p >> 4, q = p & 15;
            tid = q >> 2;
            const int e = q & 3;
            slot = 4 * hi + ((e == 1) ? 2 : (e == 2) ? 1 : e);
        } else {
            tid = p >> 3;
            slot = p & 7;
        }
    }
    const int lane = 4 * (token & 7) + tid;
    return (((token >> 3) * nch + c) * 32 + lane) * 8 + slot;
}

// Per weight format: TIn stores x, g and y; TOp is the MMA operand type of the
// activation fragments; the weights carry a factor w_scale (undone on the
// fp32 accumulator) and h is stored times h_scale (undone after the down
// projection).  All factors are powers of two, so they change no bits.
template <int WF> struct Fmt;
template <> struct Fmt<WF_F16> {
    using TIn = __half; using TOp = __half;
    static constexpr bool op_bf16 = false;
    static constexpr float w_unscale = 1.f, h_scale = 1.f;
};
template <> struct Fmt<WF_BF16> {
    using TIn = __nv_bfloat16; using TOp = __nv_bfloat16;
    static constexpr bool op_bf16 = true;
    static constexpr float w_unscale = 1.f, h_scale = 1.f;
};
// Q4 codes (u - 8) are exact in fp16; activations go in as fp16 (11 bits),
// h scaled by 2^-8 to keep fp16 clear of overflow.
template <> struct Fmt<WF_Q4> {
    using TIn = __nv_bfloat16; using TOp = __half;
    static constexpr bool op_bf16 = false;
    static constexpr float w_unscale = 1.f, h_scale = 1.f / 256.f;
};
// Prepared weights: fp16 values of w * 2^8.
template <> struct Fmt<WF_F16P> {
    using TIn = __nv_bfloat16; using TOp = __half;
    static constexpr bool op_bf16 = false;
    static constexpr float w_unscale = 1.f / kPreparedScale, h_scale = 1.f / 256.f;
};
// Q8_0: the codes (-128..127) are exact in fp16 and times an fp16 block scale
// exact in fp32; activations as for Q4.
template <> struct Fmt<WF_Q8> {
    using TIn = __nv_bfloat16; using TOp = __half;
    static constexpr bool op_bf16 = false;
    static constexpr float w_unscale = 1.f, h_scale = 1.f / 256.f;
};

// e4m3 weights: every code is exact in fp16 (3 fraction bits, exponents
// 2^-9 .. 2^8), so the MMA multiplies the codes themselves and the row scale
// multiplies each output once; activations as for Q4.
template <> struct Fmt<WF_FP8> {
    using TIn = __nv_bfloat16; using TOp = __half;
    static constexpr bool op_bf16 = false;
    static constexpr float w_unscale = 1.f, h_scale = 1.f / 256.f;
};

// Q4: one 32-bit word = canonical bytes 4*tid .. 4*tid+3 of a block.
// Returns (u - 8) as fp16 pairs:
//   r[0] = (e0, e2), r[1] = (e16, e18), r[2] = (e1, e3), r[3] = (e17, e19)
// relative to element 4*tid of the block.  0x6400 is fp16 1024.0, whose ulp
// is 1: OR-ing a low nibble u into its mantissa gives exactly 1024 + u, and
// subtracting 1032 gives u - 8.  A high nibble is OR-ed in where it sits
// (mantissa bits 4-7), giving 1024 + 16u exactly; (1024 + 16u) / 16 - 72 =
// u - 8 is one fp16 FMA whose exact result is representable.  One shift and
// four LOP3s per word on the integer pipe, four fp16 ops on the FMA pipe.
__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t mask, uint32_t bits) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(bits));   // (a & mask) | bits
    return r;
}

__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t (&r)[4]) {
    const __half2 k1032 = __floats2half2_rn(1032.f, 1032.f);
    const __half2 k16th = __floats2half2_rn(0.0625f, 0.0625f);
    const __half2 k72 = __floats2half2_rn(-72.f, -72.f);
    const uint32_t w8 = w >> 8;
    uint32_t v[4] = {lop_and_or(w, 0x000F000Fu, 0x64006400u), lop_and_or(w, 0x00F000F0u, 0x64006400u),
                     lop_and_or(w8, 0x000F000Fu, 0x64006400u), lop_and_or(w8, 0x00F000F0u, 0x64006400u)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 b = *reinterpret_cast<__half2 *>(&v[i]);
        b = (i & 1) ? __hfma2(b, k16th, k72) : __hsub2(b, k1032);
        r[i] = *reinterpret_cast<uint32_t *>(&b);
    }
}

// The same unpacking with the offsets left in (the streaming kernels): r[0]
// and r[2] hold 1024 + u, r[1] and r[3] hold 1024 + 16u, exactly, from one
// shift and four LOP3s.  The high-nibble activations are stored divided by
// 16, so a weight meets its stored activation a as ((u - 8) + 1032) a in a
// low position and as ((u - 8) + 72) (16 a) in a high one: every block's
// products carry 1032 * (sum of its low stored values) + 1152 * (sum of its
// high ones), a per-(block, token) constant that the activation writer
// stores beside the fragments (store_q4_corr) and one tf32 MMA a stage
// takes off again, weighted by the block scales.
__device__ __forceinline__ void unpack_word_biased(uint32_t w, uint32_t (&r)[4]) {
    const uint32_t w8 = w >> 8;
    r[0] = lop_and_or(w, 0x000F000Fu, 0x64006400u);
    r[1] = lop_and_or(w, 0x00F000F0u, 0x64006400u);
    r[2] = lop_and_or(w8, 0x000F000Fu, 0x64006400u);
    r[3] = lop_and_or(w8, 0x00F000F0u, 0x64006400u);
}

// Offsets of the biased Q4 operands (unpack_word_biased), per block of 32
// and token: C = 1032 * sum(low stored values) + 1152 * sum(high stored
// values), stored negated as two tf32 terms (hi + lo = -C to ~2^-22) in the
// order of the stage's correction MMA: per stage of 8 blocks and token tile
// (nt tiles), lane 4 * (token % 8) + t holds {hi(2t), hi(2t + 1), lo(2t),
// lo(2t + 1)} for blocks 2t and 2t + 1 of the stage (16 bytes a lane, 512 a
// tile, nt x 512 contiguous bytes a stage).
__host__ __device__ constexpr int64_t q4_corr_floats(int nt, int64_t nch) { return static_cast<int64_t>(nt) * nch * 16; }
__device__ __forceinline__ void store_q4_corr(float *corr, int nt, int token, int64_t blk, float c) {
    const float hi = ptx::round_tf32(-c);
    const float lo = ptx::round_tf32(-c - hi);
    float *p = corr + ((((blk >> 3) * nt + (token >> 3)) * 32 + 4 * (token & 7) + ((blk & 7) >> 1)) * 4 +
                       (blk & 1));
    p[0] = hi;
    p[2] = lo;
}

// Four signed bytes (the low byte first) as two fp16 pairs, exactly: each
// byte q + 128 (the sign bit flipped) goes into the low mantissa byte of
// fp16 1024 (ulp 1), giving 1024 + 128 + q; one fp16 subtraction of 1152
// leaves q.  One LOP3, two PRMT and two HSUB2.
__device__ __forceinline__ void s8x4_to_f16x2(uint32_t w, uint32_t &h01, uint32_t &h23) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));   // [u0, 0x64, u1, 0x64]
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));   // [u2, 0x64, u3, 0x64]
    const __half2 k1152 = __floats2half2_rn(1152.f, 1152.f);
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), k1152);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), k1152);
    h01 = *reinterpret_cast<const uint32_t *>(&ha);
    h23 = *reinterpret_cast<const uint32_t *>(&hb);
}

// Two e4m3 codes (the low byte is the first) as an fp16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    uint32_t r;
    const uint16_t v = static_cast<uint16_t>(two_codes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int b) {
    return b == 0 ? v.x : b == 1 ? v.y : b == 2 ? v.z : v.w;
}

// Eight normalised values n[k .. k+7] of one token (k a multiple of 8) into
// their fragment slots; with TWO, nlo receives the rounding residual of every
// value (same order).
template <int WF, bool TWO>
__device__ __forceinline__ void store_group(uint16_t *nfrag, uint16_t *nlo, int64_t nch, int token, int64_t k,
                                            const float (&f)[8]) {
    using TO = typename Fmt<WF>::TOp;
    float r[8];   // residuals v - round(v)
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = f[e] - to_f32(from_f32<TO>(f[e]));
    if constexpr (WF == WF_Q4) {
        // two runs of 4 consecutive k; each lands in one 8-byte half of a
        // lane's fragment with its elements in order {0, 2, 1, 3}
#pragma unroll
        for (int run = 0; run < 2; ++run) {
            TO o[4], ol[4];
            const int src[4] = {0, 2, 1, 3};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                o[e] = from_f32<TO>(f[4 * run + src[e]]);
                ol[e] = from_f32<TO>(r[4 * run + src[e]]);
            }
            const int64_t base = frag_elem(FRAG_Q4, nch, token, k + 4 * run);
            *reinterpret_cast<uint2 *>(nfrag + base) = *reinterpret_cast<const uint2 *>(o);
            if (TWO) *reinterpret_cast<uint2 *>(nlo + base) = *reinterpret_cast<const uint2 *>(ol);
        }
    } else {
        const int64_t base = frag_elem(frag_order<WF>(), nch, token, k);
        *reinterpret_cast<uint4 *>(nfrag + base) = Vec16<TO>::pack(f);
        if (TWO) *reinterpret_cast<uint4 *>(nlo + base) = Vec16<TO>::pack(r);
    }
}

// Q4 for the streaming kernels: eight values n[k .. k+7] (k a multiple of 8)
// into their fragment slots as store_group does, the high-nibble positions
// of a block (k % 32 >= 16) divided by 16; returns those stored values
// summed and weighted by their offset (1032 low, 1152 high).
__device__ __forceinline__ float store_group_q4_biased(uint16_t *nfrag, int64_t nch, int token, int64_t k,
                                                       const float (&f)[8]) {
    const bool hi = (k & 31) >= 16;
    const float scale = hi ? 0.0625f : 1.f;
    float sum = 0.f;
#pragma unroll
    for (int run = 0; run < 2; ++run) {
        __half o[4];
        const int src[4] = {0, 2, 1, 3};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            o[e] = __float2half_rn(f[4 * run + src[e]] * scale);
            sum += __half2float(o[e]);
        }
        const int64_t base = frag_elem(FRAG_Q4, nch, token, k + 4 * run);
        *reinterpret_cast<uint2 *>(nfrag + base) = *reinterpret_cast<const uint2 *>(o);
    }
    return sum * (hi ? 1152.f : 1032.f);
}

// Launch-shape knobs of the decode kernels.
enum {
    TUNE_NORM_RELEASE_EARLY = 0,
    TUNE_PRE_STAGES_GATEUP = 1,
    TUNE_PRE_STAGES_DOWN = 2,
    TUNE_NORM_SLICES = 3,
    TUNE_COUNT = 4
};
int decode_tuning(int knob);

// TMA-streamed decode kernels (gemv_stream.cu)
bool stream_supported(int wfmt, int64_t d, int64_t ffn);
int64_t stream_down_splits(int wfmt, int64_t d, int64_t ffn);
template <int WF, int NT, bool TWO>
cudaError_t launch_stream_gateup(GemvWeights wg, GemvWeights wu, const void *nfrag, const void *nfrag_lo,
                                 void *hfrag, void *hfrag_lo, int64_t d, int64_t ffn, int64_t nchK,
                                 int64_t nchF, unsigned *counters, int ncounters, const float *ncorr,
                                 float *hcorr, cudaStream_t s);
template <int WF, int NT, bool TWO>
// ss_part, y_sumsq (y_sumsq may be null): the rows' sums of squares of the
// stored y, through [ceil(d/64)][rows] partial sums and counters[ceil(d/64)];
// Q4: ncorr / hcorr the block offsets of n (read) and h (written, then read)
cudaError_t launch_stream_down(GemvWeights wd, const void *hfrag, const void *hfrag_lo, void *y,
                               float *partials, unsigned *counters, int rows, int64_t d, int64_t ffn,
                               int64_t nchF, int64_t splits, const void *res, float *ss_part, float *y_sumsq,
                               const float *hcorr, cudaStream_t s);

// The decode block as one cooperative persistent kernel (gemv_fused.cu,
// FFN_DECODE_ONE_KERNEL): norm, gate/up and down handing over through the
// stream's control block; ws.partials holds fused_partial_floats(...) fp32
// split partials.  The shapes of stream_supported().
int64_t fused_partial_floats(int wfmt, int64_t rows, int64_t d, int64_t ffn, int nt, bool two);
// The control block of stream s on the current device, or null (d above
// 65536, or 64 streams of this device already hold one): then the three
// kernels run instead.
unsigned long long *fused_control(int64_t d, cudaStream_t s);
template <int WF, int NT, bool TWO>
cudaError_t launch_fused(GemvWeights wg, GemvWeights wu, GemvWeights wd, const void *x, const void *gain, void *y,
                         int rows, int64_t d, int64_t ffn, float eps, const GemvWorkspace &ws, const void *res,
                         const float *ss_in, float *y_sumsq, unsigned long long *ctl, cudaStream_t s);

}  // namespace gemv
}  // namespace ffn
