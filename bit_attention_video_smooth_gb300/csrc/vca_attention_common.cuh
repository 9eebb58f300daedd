// vca_attention_common.cuh -- pieces both attention kernels (E4M3 residual V
// with FP8 P, NVFP4 residual V with NVFP4 P) share: the softmax warps' named
// barriers, the lazy reference-max threshold, the mean-restore operands, the
// output epilogue and the host-side tensor maps.
//
// Mean restore (paper page, "method": the block means come back through the
// row sums online softmax keeps): O_acc accumulates P (V - mu)/s_v per block;
// the means come back as sum_b rowsum_b (x) mu_b.  Every kMeanJ key blocks one
// bf16 MMA adds [rs hi | rs lo | rs hi | rs lo] . [mu' hi | mu' hi | mu' lo | mu' lo]^T
// (mu' = mu / s_v) to O_acc: the hi/lo bf16 splits keep ~16 bits of both
// factors and the products are exact in the fp32 accumulator.
#pragma once

#include <cuda.h>

#include "vca_device.cuh"

namespace vca {
namespace attn {

// Eight softmax warps, two per TMEM lane quarter: the two take alternate key
// blocks (one thread per query row and block) and hold a row in registers
// kCols columns at a time.
constexpr int kParts = 2;
constexpr int kCols = kBlk / kParts;       // S columns held in registers at a time
constexpr int kSoftmaxWarps = 4 * kParts;
constexpr int kMeanJ = 16;                 // key blocks per mean-restore MMA
constexpr float kLazyTau = 8.0f;           // log2 units: the reference max moves by more than 2^8 only

constexpr uint32_t kBarSoftmax = 1;        // all softmax warps
constexpr uint32_t kBarHand0 = 2;          // + 2 * quarter + parity: the reference-max hand-over

// Wait ignoring the abort flag (used only to drain work this thread issued).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Largest of a thread's kCols raw scores.
__device__ __forceinline__ float row_part_max(const uint32_t (&S)[kCols]) {
    float a[4] = {__uint_as_float(S[0]), __uint_as_float(S[1]), __uint_as_float(S[2]), __uint_as_float(S[3])};
#pragma unroll
    for (int j = 4; j < kCols; j += 2)
        a[(j >> 1) & 3] = max3(a[(j >> 1) & 3], __uint_as_float(S[j]), __uint_as_float(S[j + 1]));
    return fmaxf(max3(a[0], a[1], a[2]), a[3]);
}

// Named barrier that also ANDs a flag over its `count` threads.
__device__ __forceinline__ bool bar_and(bool v, uint32_t id, uint32_t count) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Signal a named barrier without waiting (the producer side of bar.sync).
// When the barrier completes, the memory accesses this thread made before
// bar.arrive are performed relative to every thread taking part in it (the
// PTX barrier rule covers arrive as well as sync), so the shared-memory writes
// before it are visible to the threads that complete it with bar.sync; a
// separate CTA fence is not needed (it cost ~0.8 % of the 8-bit kernel).
__device__ __forceinline__ void bar_arrive_release(uint32_t id, uint32_t count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// One row of a mean-restore operand from kMeanJ values split as hi + lo bf16,
// into the 128-byte-swizzled K-major tile `dst`:
//   A (query row): [hi | lo | hi | lo]   (chunks 0,1 hi; 2,3 lo; 4,5 hi; 6,7 lo)
//   B (channel):   [hi | hi | lo | lo]   (chunks 0-3 hi; 4-7 lo)
__device__ __forceinline__ void store_mean_row(unsigned char *dst, int row, const float (&x)[kMeanJ], bool a_operand) {
    uint32_t h[kMeanJ / 2], l[kMeanJ / 2];
#pragma unroll
    for (int k = 0; k < kMeanJ / 2; ++k) split_pack_bf16x2(x[2 * k], x[2 * k + 1], h[k], l[k]);
    const uint4 hv[2] = {make_uint4(h[0], h[1], h[2], h[3]), make_uint4(h[4], h[5], h[6], h[7])};
    const uint4 lv[2] = {make_uint4(l[0], l[1], l[2], l[3]), make_uint4(l[4], l[5], l[6], l[7])};
#pragma unroll
    for (int ck = 0; ck < 8; ++ck) {
        const bool use_lo = a_operand ? (((ck >> 1) & 1) != 0) : (ck >= 4);
        *reinterpret_cast<uint4 *>(dst + sw128_offset(row, ck)) = use_lo ? lv[ck & 1] : hv[ck & 1];
    }
}


// O row part = O_acc s_v / l for this thread's kCols channels starting at
// col0 (every block's mean term is in O_acc by then): tO is the TMEM address
// of those accumulator columns in this thread's lane, orow the output row at
// col0.  sSV is 16-byte aligned and read four channels at a time.
constexpr int kRsSlots = 32;   // row-sum slots per query row (a ring)
__device__ __forceinline__ void store_output(uint32_t tO, const float *sSV, int col0, float inv_l, uint16_t *orow) {
#pragma unroll 1
    for (int i = 0; i < kCols / 32; ++i) {
        uint32_t o[32];
        VCA_TMEM_LD32(tO + 32 * i, o);
        tmem_ld_wait();
        const float4 *sv4 = reinterpret_cast<const float4 *>(sSV + col0 + 32 * i);
        float acc[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float4 v = sv4[e];
            acc[4 * e] = __fmul_rn(__uint_as_float(o[4 * e]), v.x);
            acc[4 * e + 1] = __fmul_rn(__uint_as_float(o[4 * e + 1]), v.y);
            acc[4 * e + 2] = __fmul_rn(__uint_as_float(o[4 * e + 2]), v.z);
            acc[4 * e + 3] = __fmul_rn(__uint_as_float(o[4 * e + 3]), v.w);
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(__fmul_rn(acc[2 * e], inv_l), __fmul_rn(acc[2 * e + 1], inv_l));
#pragma unroll
        for (int e = 0; e < 4; ++e)
            reinterpret_cast<uint4 *>(orow + 32 * i)[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
    }
}

// A mean-restore MMA follows PV(b) for b = 19, 35, 51, ...: it adds the terms
// of blocks b-19 .. b-4.  Their row sums are all visible to the thread that
// stages them at block b (b is odd, so that thread takes the odd blocks): the
// sum of an odd block j is written by the thread itself at block j+2 <= b-2,
// the sum of an even block j <= b-5 by its partner at block j+2, before the
// partner hands over the reference max at block j+4 <= b-1.
constexpr int kMeanLag = 3;
__host__ __device__ constexpr bool flush_after(int b) {
    return b >= kMeanJ + kMeanLag && (b % kMeanJ) == kMeanLag;
}

// Operands of the mean-restore MMA for blocks b0 .. b0+n-1, n <= kMeanJ (row /
// channel `row`): A row = the row sums from their ring slots, each brought
// from the reference max it was taken against to m; B row = mean / s_v; the
// K entries of the kMeanJ - n missing blocks are zero in both.  sMeanGroup
// holds the means of the group's blocks, block b0 + i at i * kD.
__device__ __forceinline__ void stage_mean_sums(int row, const float *sRS, const float *sRSM, float m, int b0,
                                                unsigned char *sMA, int n = kMeanJ) {
    float x[kMeanJ];
#pragma unroll
    for (int i = 0; i < kMeanJ; ++i) {
        x[i] = 0.0f;
        if (i < n) {
            const int slot = ((b0 + i) & (kRsSlots - 1)) * kBlk + row;
            float rs = sRS[slot];
            const float mt = sRSM[slot];
            if (mt != m) rs = __fmul_rn(rs, ex2_approx(__fsub_rn(mt, m)));
            x[i] = rs;
        }
    }
    store_mean_row(sMA, row, x, true);
}
__device__ __forceinline__ void stage_mean_values(int row, const uint16_t *sMeanGroup, const float *sSV,
                                                  unsigned char *sMB, int n = kMeanJ) {
    float x[kMeanJ];
    const float inv_sv = 1.0f / sSV[row];
#pragma unroll
    for (int i = 0; i < kMeanJ; ++i)
        x[i] = i < n ? __fmul_rn(bf16_bits_to_f32(sMeanGroup[i * kD + row]), inv_sv) : 0.0f;
    store_mean_row(sMB, row, x, false);
}
__device__ __forceinline__ void stage_means(int row, const float *sRS, const float *sRSM, float m, int b0,
                                            const uint16_t *sMeanGroup, const float *sSV, unsigned char *sMA,
                                            unsigned char *sMB) {
    stage_mean_sums(row, sRS, sRSM, m, b0, sMA);
    stage_mean_values(row, sMeanGroup, sSV, sMB);
}

// The epilogue's mean terms: blocks tail0 .. tail0 + rs_cnt - 1 (those after
// the last in-loop mean MMA's range; rs_cnt <= 2 kMeanJ) are added into O by
// one more mean-restore MMA group, two when rs_cnt > kMeanJ, instead of on
// CUDA cores (there every thread reads every mean: shared-memory broadcast
// bound).  Called by all softmax threads once every PV has completed: blocks
// tail0 .. tail0 + 15 go to tiles0 (A, B), the rest to tiles1; the even-block
// threads stage the A rows (row sums), the odd-block threads the B rows
// (means).  tail0 is a multiple of kMeanJ, so the two groups' means are in
// buffers (tail0 / kMeanJ) & 1 and the other.
// One thread issues the MMAs and commits them to `bar` (phase 0, count 1);
// every thread waits for it.  Returns false when that wait gave up (the
// issuing thread then still waits for its MMAs, so that TMEM outlives them).
__device__ __forceinline__ bool restore_tail_means(int par, int row, bool issuer, const float *sRS, const float *sRSM,
                                                   float mf, int tail0, int rs_cnt, const uint16_t *sMean,
                                                   const float *sSV, unsigned char *tiles0, unsigned char *tiles1,
                                                   uint32_t tO, uint64_t *bar, int *abort_flag, uint64_t limit_ns) {
    const int n0 = rs_cnt < kMeanJ ? rs_cnt : kMeanJ, n1 = rs_cnt - n0;
    const int g0 = tail0 / kMeanJ;
    constexpr uint32_t kTile = kBlk * kD;   // one staged operand: 128 rows x 64 bf16
    if (par == 0) {
        stage_mean_sums(row, sRS, sRSM, mf, tail0, tiles0, n0);
        if (n1 > 0) stage_mean_sums(row, sRS, sRSM, mf, tail0 + kMeanJ, tiles1, n1);
    } else {
        stage_mean_values(row, sMean + (g0 & 1) * (kMeanJ * kD), sSV, tiles0 + kTile, n0);
        if (n1 > 0) stage_mean_values(row, sMean + ((g0 + 1) & 1) * (kMeanJ * kD), sSV, tiles1 + kTile, n1);
    }
    fence_proxy_async_smem();   // read by the tensor core
    bar_sync(kBarSoftmax, 32 * kSoftmaxWarps);
    if (issuer) {
        tc_fence_after();
        constexpr uint32_t idesc_bf16 = make_idesc(128, 128, 1, 1);
        for (int g = 0; g < (n1 > 0 ? 2 : 1); ++g) {
            const uint32_t base = smem_u32(g == 0 ? tiles0 : tiles1);
            const uint64_t da = sdesc_k_sw128(base), db = sdesc_k_sw128(base + kTile);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_f16(tO, da + 2 * kk, db + 2 * kk, idesc_bf16, 1u);
        }
        tc_commit(bar);
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, 0, abort_flag, limit_ns));
    if (!ok && issuer) drain_wait(bar, 0, limit_ns);
    if (ok) tc_fence_after();
    return ok;
}

// One Q tile row (the A operand of QK) into registers: `row`'s 128 E4M3
// codes as 32 words, in the column order of its TMEM lane.
__device__ __forceinline__ void load_q_regs(const uint8_t *q8row, uint32_t (&qv)[32]) {
    const uint4 *qrow = reinterpret_cast<const uint4 *>(q8row);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 u = qrow[i];
        qv[4 * i] = u.x;
        qv[4 * i + 1] = u.y;
        qv[4 * i + 2] = u.z;
        qv[4 * i + 3] = u.w;
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// 2-D byte matrix [rows][128] with 128 x 128 boxes and the 128-byte swizzle.
inline bool make_tile_map(CUtensorMap *map, const void *base, uint64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte matrix [rows][64] with 64 x 128 boxes and the 64-byte swizzle (the
// NVFP4 V codes: one 128-channel block per box).
inline bool make_tile_map_sw64(CUtensorMap *map, const void *base, uint64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {64, rows};
    cuuint64_t strides[1] = {64};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace attn
}  // namespace vca
