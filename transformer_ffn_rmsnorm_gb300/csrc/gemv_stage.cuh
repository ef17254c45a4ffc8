// gemv_stage.cuh -- the ring stage shared by the TMA-streamed decode kernels:
// its layout, the MMAs of one stage for each weight format, and the tensor
// maps that fill it.
#pragma once

#include <cudaTypedefs.h>

#include "gemv_common.cuh"

namespace ffn {
namespace gemv {
namespace {

constexpr int kConsumers = 4;
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint32_t kFragBytes = 32 * 16;   // one 32-value chunk of fragments for 8 tokens

enum { ROLE_GATEUP = 0, ROLE_DOWN = 1 };

// Stage layout: [weights of each matrix][their scales (Q4)][activation
// fragments: NT tiles x terms x chunks x 512 B].  Every format but Q8_0
// moves 128 bytes of each weight row per stage (Q8_0: 256).  With BIAS (Q4
// on the streaming kernels) each stage also has NT x 512 bytes of block
// offsets (store_q4_corr), kept in a ring of their own after the stages so
// that the stages keep their 1 KB multiple.
template <int WF, int ROLE, int NT, bool TWO, bool BIAS = false> struct Tile {
    static constexpr bool q4 = WF == WF_Q4;
    static constexpr bool fp8 = WF == WF_FP8;
    static constexpr bool q8 = WF == WF_Q8;
    static constexpr bool blocks = q4 || q8;                     // fp16 scales per 32 weights
    static constexpr int nmat = ROLE == ROLE_GATEUP ? 2 : 1;     // weight matrices per stage
    static constexpr int box_rows = ROLE == ROLE_GATEUP ? 32 : 64;
    // 128-byte boxes per row and stage: two, but one for Q4 (its 128 bytes
    // hold 256 weights) and for four or more token tiles, whose activation
    // fragments would otherwise outgrow the weights in the stage
    static constexpr int boxes = (q4 || (NT >= 4 && !q8)) ? 1 : 2;
    static constexpr int box_x = (q8 || fp8) ? 128 : 64;         // TMA inner coordinate per box (bytes / elements)
    static constexpr int kb = (q4 || q8) ? 256 : boxes * box_x;  // k values per stage
    static constexpr int x_per_kb = q4 ? 128 : boxes * box_x;   // TMA inner coordinate per stage
    static constexpr int chunks = kb / kChunk;                   // fragment chunks per stage
    static constexpr int terms = TWO ? 2 : 1;
    static constexpr uint32_t box_bytes = box_rows * 128;        // one 128-byte-wide TMA box
    static constexpr uint32_t w_bytes = boxes * box_bytes;       // one matrix' rows of a stage
    static constexpr uint32_t s_bytes = blocks ? box_rows * 16 : 0; // its scales
    static constexpr uint32_t b_off = nmat * (w_bytes + s_bytes);
    static constexpr uint32_t b_bytes = NT * terms * chunks * kFragBytes;
    static constexpr uint32_t stage_bytes = (b_off + b_bytes + 1023) & ~1023u;
    static constexpr int stages_fit = (52 * 1024) / stage_bytes;
    // (large stages of many token tiles run with two, keeping three CTAs a SM)
    static constexpr int min_stages = (NT >= 4 && stage_bytes > 20 * 1024) ? 2 : 3;
    static constexpr int stages = stages_fit < min_stages ? min_stages : stages_fit > 6 ? 6 : stages_fit;
    static constexpr uint32_t corr_bytes = (q4 && BIAS) ? NT * 512 : 0;
    static constexpr size_t smem_bytes = stages * (stage_bytes + corr_bytes) + 1024;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// One ring stage of MMAs for one consumer warp: the stage at shared address
// st holds k-block kb of the warp's weight rows (gate/up: warp / 2 picks the
// matrix, warp % 2 the 16-row tile of the box's 32 rows; down: warp picks the
// 16-row tile of 64) and of the activation fragments; acc gathers the
// products for NT token tiles.  With BIAS, cst is the stage's block offsets.
template <int WF, int NT, bool TWO, int ROLE, bool BIAS = false>
__device__ __forceinline__ void stage_mma(float (&acc)[NT][4], uint32_t st, int64_t kb, int64_t nch_b, int warp,
                                          int lane, uint32_t cst = 0) {
    using TL = Tile<WF, ROLE, NT, TWO, BIAS>;
    constexpr bool bf = Fmt<WF>::op_bf16;
    constexpr bool q4 = TL::q4;
    constexpr bool fp8 = TL::fp8;
    const int g = lane >> 2, tid = lane & 3;
    const int mat = ROLE == ROLE_GATEUP ? (warp >> 1) : 0;
    const int r0 = 16 * (ROLE == ROLE_GATEUP ? (warp & 1) : warp);   // row tile inside the box
    const int ra = r0 + g, rb = r0 + g + 8;                             // (ra & 7) == (rb & 7) == g
    const uint32_t wbase = st + mat * TL::w_bytes;
    if constexpr (fp8) {
        // 256 k = four groups of 64, two in each 128-byte box of a row; in
        // each, this lane's 16 codes of rows ra and rb (k = 16 tid .. 16
        // tid + 15) feed four MMAs, four k each, against the group's two
        // fragment chunks
        const uint32_t bbase = st + TL::b_off + lane * 16;
#pragma unroll
        for (int grp = 0; grp < 2 * TL::boxes; ++grp) {
            uint4 b0[NT], b1[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                b0[n] = lds128(bbase + (n * TL::chunks + 2 * grp) * kFragBytes);
                b1[n] = lds128(bbase + (n * TL::chunks + 2 * grp + 1) * kFragBytes);
            }
            const uint32_t box = wbase + static_cast<uint32_t>(grp >> 1) * TL::box_bytes;
            const uint32_t off = static_cast<uint32_t>(((4 * (grp & 1) + tid) ^ g) << 4);
            const uint4 qa = lds128(box + ra * 128 + off);
            const uint4 qb = lds128(box + rb * 128 + off);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t wa = word_of(qa, m), wb = word_of(qb, m);
                const uint32_t a0 = e4m3x2_to_f16x2(wa), a2 = e4m3x2_to_f16x2(wa >> 16);
                const uint32_t a1 = e4m3x2_to_f16x2(wb), a3 = e4m3x2_to_f16x2(wb >> 16);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint4 &bv = m < 2 ? b0[n] : b1[n];
                    const uint32_t x0 = (m & 1) ? bv.z : bv.x, x1 = (m & 1) ? bv.w : bv.y;
                    ptx::mma_16816<bf>(acc[n], a0, a1, a2, a3, x0, x1);
                }
            }
        }
    } else if constexpr (TL::q8) {
        // 256 k = eight 32-value blocks, 0-3 in the first 128-byte box of a
        // row, 4-7 in the second; in block b this lane owns k = 8 tid .. 8
        // tid + 7 (natural fragment order) of rows ra and rb
        const uint32_t sbase = st + TL::nmat * TL::w_bytes + mat * TL::s_bytes;
        const uint32_t bbase = st + TL::b_off + lane * 16;
        const uint4 sa = lds128(sbase + ra * 16), sb = lds128(sbase + rb * 16);
        float2 fsa[4], fsb[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t a = word_of(sa, j), b = word_of(sb, j);
            fsa[j] = __half22float2(*reinterpret_cast<const __half2 *>(&a));
            fsb[j] = __half22float2(*reinterpret_cast<const __half2 *>(&b));
        }
#pragma unroll
        for (int bi = 0; bi < 8; ++bi) {
            const uint32_t box = wbase + static_cast<uint32_t>(bi >> 2) * TL::box_bytes;
            const int bl = bi & 3;
            // bytes 32 bl + 8 tid .. + 7 of the row: 16-byte granule 2 bl + tid / 2
            const uint32_t off = static_cast<uint32_t>((((2 * bl + (tid >> 1)) ^ g) << 4) + ((tid & 1) << 3));
            const uint2 qa = lds64(box + ra * 128 + off), qb = lds64(box + rb * 128 + off);
            uint4 b[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) b[n] = lds128(bbase + (n * TL::chunks + bi) * kFragBytes);
            uint32_t a01x, a23x, a01y, a23y, c01x, c23x, c01y, c23y;
            s8x4_to_f16x2(qa.x, a01x, a23x);
            s8x4_to_f16x2(qa.y, a01y, a23y);
            s8x4_to_f16x2(qb.x, c01x, c23x);
            s8x4_to_f16x2(qb.y, c01y, c23y);
            const float fa = (bi & 1) ? fsa[bi >> 1].y : fsa[bi >> 1].x;
            const float fb = (bi & 1) ? fsb[bi >> 1].y : fsb[bi >> 1].x;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                float t[4];   // this block's products alone, scaled below
                ptx::mma_16816_z<bf>(t, a01x, c01x, a23x, c23x, b[n].x, b[n].y);
                ptx::mma_16816<bf>(t, a01y, c01y, a23y, c23y, b[n].z, b[n].w);
                acc[n][0] = fmaf(fa, t[0], acc[n][0]);
                acc[n][1] = fmaf(fa, t[1], acc[n][1]);
                acc[n][2] = fmaf(fb, t[2], acc[n][2]);
                acc[n][3] = fmaf(fb, t[3], acc[n][3]);
            }
        }
    } else if constexpr (!q4) {
        // 32-wide chunks, two in each 128-byte box of a row: this lane's 16
        // bytes of rows ra, rb at granule 4 (j % 2) + tid of box j / 2
        const uint32_t bbase = st + TL::b_off + lane * 16;
#pragma unroll
        for (int j = 0; j < TL::chunks; ++j) {
            const int64_t c = kb * TL::chunks + j;
            // the last k-block can run past the fragment buffer (K a
            // multiple of 8 only); the weights there are TMA zero fill,
            // the operand must be 0
            const bool cin = c < nch_b;
            const uint32_t box = wbase + static_cast<uint32_t>(j >> 1) * TL::box_bytes;
            const uint32_t off = static_cast<uint32_t>(((4 * (j & 1) + tid) ^ g) << 4);
            const uint4 a0 = lds128(box + ra * 128 + off);
            const uint4 a1 = lds128(box + rb * 128 + off);
            // one token tile's operand at a time (eight tiles' would
            // cost 64 registers)
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const uint4 b = cin ? lds128(bbase + ((n * TL::terms) * TL::chunks + j) * kFragBytes)
                                    : make_uint4(0, 0, 0, 0);
                ptx::mma_16816<bf>(acc[n], a0.x, a1.x, a0.y, a1.y, b.x, b.y);
                ptx::mma_16816<bf>(acc[n], a0.z, a1.z, a0.w, a1.w, b.z, b.w);
                if constexpr (TWO) {
                    const uint4 bl = cin ? lds128(bbase + ((n * TL::terms + 1) * TL::chunks + j) * kFragBytes)
                                         : make_uint4(0, 0, 0, 0);
                    ptx::mma_16816<bf>(acc[n], a0.x, a1.x, a0.y, a1.y, bl.x, bl.y);
                    ptx::mma_16816<bf>(acc[n], a0.z, a1.z, a0.w, a1.w, bl.z, bl.w);
                }
            }
        }
    } else {
        // 256 k = two groups of four 32-value blocks; scales follow the nibbles
        const uint32_t sbase = st + TL::nmat * TL::w_bytes + mat * TL::s_bytes;
        const uint32_t bbase = st + TL::b_off + lane * 16;
        const uint4 sa = lds128(sbase + ra * 16), sb = lds128(sbase + rb * 16);
        // the stage's eight block scales of rows ra and rb, widened in pairs
        float2 fsa[4], fsb[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t a = word_of(sa, j), b = word_of(sb, j);
            fsa[j] = __half22float2(*reinterpret_cast<const __half2 *>(&a));
            fsb[j] = __half22float2(*reinterpret_cast<const __half2 *>(&b));
        }
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
            const uint32_t off = static_cast<uint32_t>(((4 * grp + tid) ^ g) << 4);
            const uint4 qa = lds128(wbase + ra * 128 + off);
            const uint4 qb = lds128(wbase + rb * 128 + off);
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                const int bi = 4 * grp + blk;            // block inside the stage, 0..7
                uint4 b[NT];
#pragma unroll
                for (int n = 0; n < NT; ++n) b[n] = lds128(bbase + (n * TL::chunks + bi) * kFragBytes);
                uint32_t lo[4], hi[4];
                if constexpr (BIAS) {
                    unpack_word_biased(word_of(qa, blk), lo);
                    unpack_word_biased(word_of(qb, blk), hi);
                } else {
                    dequant_word(word_of(qa, blk), lo);
                    dequant_word(word_of(qb, blk), hi);
                }
                const float fa = (bi & 1) ? fsa[bi >> 1].y : fsa[bi >> 1].x;
                const float fb = (bi & 1) ? fsb[bi >> 1].y : fsb[bi >> 1].x;
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    float t[4];   // this block's products alone, scaled below
                    ptx::mma_16816_z<bf>(t, lo[0], hi[0], lo[2], hi[2], b[n].x, b[n].y);
                    ptx::mma_16816<bf>(t, lo[1], hi[1], lo[3], hi[3], b[n].z, b[n].w);
                    acc[n][0] = fmaf(fa, t[0], acc[n][0]);
                    acc[n][1] = fmaf(fa, t[1], acc[n][1]);
                    acc[n][2] = fmaf(fb, t[2], acc[n][2]);
                    acc[n][3] = fmaf(fb, t[3], acc[n][3]);
                }
            }
        }
        if constexpr (BIAS) {
            // the offsets of the stage's 8 blocks: acc += s(row, block) x
            // (-C(block, token)) summed over the blocks, one tf32 MMA per term
            // of -C (k = block: this lane's k t and t + 4 are blocks 2t and
            // 2t + 1, whose scales are one 4-byte load a row)
            uint32_t s2a, s2b;
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(s2a) : "r"(sbase + ra * 16 + 4 * tid));
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(s2b) : "r"(sbase + rb * 16 + 4 * tid));
            const float2 ca = __half22float2(*reinterpret_cast<const __half2 *>(&s2a));
            const float2 cb = __half22float2(*reinterpret_cast<const __half2 *>(&s2b));
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const uint4 c = lds128(cst + n * 512 + lane * 16);
                ptx::mma_1688_tf32(acc[n], __float_as_uint(ca.x), __float_as_uint(cb.x), __float_as_uint(ca.y),
                                   __float_as_uint(cb.y), c.x, c.y);
                ptx::mma_1688_tf32(acc[n], __float_as_uint(ca.x), __float_as_uint(cb.x), __float_as_uint(ca.y),
                                   __float_as_uint(cb.y), c.z, c.w);
            }
        }
    }
}

// ------------------------------------------------------------------ host side
bool map_rows(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, int64_t inner, int64_t rows,
              int64_t row_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle) {
    return encode_tma_2d(m, ptr, dt, inner, rows, row_bytes, box_inner, box_rows,
                         swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Weight (and scale) maps of one matrix [rows x K] in format WF.
template <int WF, int ROLE>
bool weight_maps(CUtensorMap *w, CUtensorMap *sc, const GemvWeights &wt, int64_t rows, int64_t K) {
    using TL = Tile<WF, ROLE, 1, false>;
    if (TL::q8) {
        if (!map_rows(w, wt.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, rows, K, 128, TL::box_rows, true)) return false;
        return map_rows(sc, wt.sc, CU_TENSOR_MAP_DATA_TYPE_UINT16, K / 32, rows, K / 16, 8, TL::box_rows, false);
    }
    if (TL::fp8) {
        *sc = CUtensorMap{};
        return map_rows(w, wt.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, rows, K, 128, TL::box_rows, true);
    }
    if (TL::q4) {
        if (!map_rows(w, wt.qs, CU_TENSOR_MAP_DATA_TYPE_UINT8, K / 2, rows, K / 2, 128, TL::box_rows, true))
            return false;
        return map_rows(sc, wt.sc, CU_TENSOR_MAP_DATA_TYPE_UINT16, K / 32, rows, K / 16, 8, TL::box_rows, false);
    }
    *sc = CUtensorMap{};
    return map_rows(w, wt.w, CU_TENSOR_MAP_DATA_TYPE_UINT16, K, rows, K * 2, 64, TL::box_rows, true);
}

// Opt one kernel (the template argument itself, so every instantiation has
// its own flag) into more than 48 KB of dynamic shared memory on this device.
template <auto KERN>
cudaError_t set_smem(size_t bytes) {
    static int configured = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured != dev) {
        e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
        if (e != cudaSuccess) return e;
        configured = dev;
    }
    return cudaSuccess;
}

}  // namespace
}  // namespace gemv
}  // namespace ffn
