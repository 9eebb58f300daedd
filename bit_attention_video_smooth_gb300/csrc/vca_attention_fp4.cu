// vca_attention_fp4.cu -- the 4-bit VC-Attention kernel (paper page, "method":
// the residual left after demeaning is quantised to NVFP4 for the 4-bit
// path): V residual as NVFP4 (E2M1 codes, one E4M3 scale per 16 tokens of a
// channel, one fp32 scale g per head) and P as NVFP4 (E2M1 codes, one E4M3
// scale per 16 keys of a row), with the V-Smooth mean restore of the 8-bit
// kernel.
//
// PV runs on the tensor core as the block-scaled FP4 MMA (kind::mxf4nvf4,
// scale_vec::4X): P (A, E2M1 codes from TMEM) times V (B, E2M1 codes from
// shared memory), each 16 keys of a row of either operand scaled by its E4M3
// scale factor, which the MMA reads from TMEM; fp32 accumulation.  QK stays
// E4M3 (kind::f8f6f4).  Layouts (measured on the hardware with a probe): P key k
// at TMEM column k / 8, nibble k % 8; row m's four scales of a 64-key MMA in
// lane m, column sfa + m / 32; B row n's, for the D rows of lane quarter q,
// in lane 32 q + n % 32, column sfb + n / 32, so the V scales (and the ones'
// scales of the row-sum MMA) are present in all four lane quarters; the V
// codes as a 128-byte-swizzled K-major tile whose 128-byte rows (one per
// channel) carry the block's 128 keys in their first 64 bytes.
//
// One CTA owns a 128-row query tile of one (batch, head).  Warp roles:
//   warp 11      TMA producer: K tiles into a 3-stage ring
//   warp 1       TMEM owner and MMA issuer (one thread); per key block j:
//                  O += P_j V_j, E_{j&1} = P_j ones  (two block-scaled MMAs
//                                 each, K = 64; the second gives P_j's row sums)
//                  then the mean-restore MMA when due, then
//                  S[j&1] = Q8 K8_{j+2}^T               (kind::f8f6f4)
//   warps 0, 10  V layout: each block's packed codes (8 KB) into the swizzled
//                tile, two channels per thread, and its scale factors into
//                the 32-row matrices the MMA issuer copies into TMEM (one
//                copy fills all four lane quarters); warp 0's lane 0
//                bulk-copies block j+3's codes and scales into a 4-stage ring.
//   warps 2-9    softmax, two threads per query row (column halves): running
//                max with the lazy threshold, NVFP4 P of the row against it,
//                P codes and scales into TMEM once PV(j-1) is done, row sum of
//                block j-1 from its TMEM slot, O rescale, mean-restore
//                operands, epilogue.
// P has a single TMEM buffer, so P_j is written after PV(j-1) completes; the
// softmax computes it while PV(j-1) runs.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384), E0 [384,400),
// E1 [400,416), P [416,432) (eight E2M1 codes per column), P scales
// [432,440), V scales [440,456) (two buffers), ones' scales 456, Q [480,512).
// Every wait is bounded; a wait that runs out raises a CTA-wide abort, the CTA
// drains its copies and MMAs, frees TMEM and reports VCA_ERR_TIMEOUT.
#include "vca_attention_common.cuh"
#include "vca_internal.h"

namespace vca {

namespace {

using namespace attn;

constexpr int kKStages = 3;                  // K tiles in flight
constexpr int kRawStages = 4;                // packed V blocks in flight
constexpr int kVStages = 2;                  // swizzled V code tiles
constexpr int kLayWarp0 = 0;                 // V layout; its lane 0 copies
constexpr int kLayWarp1 = 2 + kSoftmaxWarps; // V layout
constexpr int kLayWarps = 2;                 // two channels per thread
constexpr int kKWarp = kLayWarp1 + 1;        // K producer
// 12 warps: at most three per SM sub-partition, so up to 168 registers a thread
constexpr int kThreads = 32 * (kKWarp + 1);
constexpr int kRsCap = kMeanJ;               // buffered row sums per row

constexpr uint32_t kTileBytes = kBlk * kD;              // one 128 x 128 FP8 K tile
constexpr uint32_t kCodeBytes = kD * kBlk / 2;          // a block's E2M1 codes, [ch][64 bytes]
constexpr uint32_t kSfBytes = kD * kBlk / 16;           // a block's E4M3 scales, [ch][8]
constexpr uint32_t kRawStageBytes = kCodeBytes + kSfBytes;
constexpr uint32_t kVStageBytes = kD * 128;             // 128 channel rows of 128 bytes (codes in the first 64)
constexpr uint32_t kOnesRows = 16;
constexpr uint32_t kOnesBytes = kOnesRows * 128;        // 16 rows of E2M1 1.0: the row-sum MMA's B
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256, kTmemE0 = 384, kTmemE1 = 400, kTmemP = 416, kTmemSFA = 432, kTmemSFB = 440,
                   kTmemSF1 = 456, kTmemQ = 480;

constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffOnes = kOffV + kVStages * kVStageBytes;
constexpr uint32_t kSfbBytes = 32 * 16;                  // V scales of one MMA: 32 rows x 4 words
constexpr uint32_t kOffSfb = kOffOnes + kOnesBytes;        // [kVStages][2][kSfbBytes]
constexpr uint32_t kOffRaw = kOffSfb + kVStages * 2 * kSfbBytes;
constexpr uint32_t kOffMA = (kOffRaw + kRawStages * kRawStageBytes + 1023) & ~1023u;
constexpr uint32_t kOffMB = kOffMA + kTileBytes;
constexpr uint32_t kOffRS = kOffMB + kTileBytes;            // fp32 [kRsCap][128] buffered row sums
constexpr uint32_t kOffSV = kOffRS + kRsCap * kBlk * 4;     // fp32 [128]: g for every channel
constexpr uint32_t kOffPM = kOffSV + kBlk * 4;              // fp32 [2][kParts][128] part-row maxima
constexpr uint32_t kOffL = kOffPM + 2 * kParts * kBlk * 4;  // fp32 [128] final row sums
constexpr uint32_t kOffLg = kOffL + kBlk * 4;               // fp32 [128]: -log2(dec(E4M3 code)), -inf for code 0
constexpr uint32_t kOffBar = kOffLg + kBlk * 4;
constexpr int kNumBars = 1 + 2 * kKStages + 2 + kVStages + 2 * kRawStages + 1 + 2 + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;       // tmem address, abort flag
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;       // + alignment slack
static_assert(kOffV % 1024 == 0 && kVStageBytes % 1024 == 0 && kOffOnes % 1024 == 0 && kOffMA % 1024 == 0 &&
                  kOffMB % 1024 == 0,
              "swizzled operand tiles need 1024-byte alignment");
static_assert(kRawStageBytes % 16 == 0 && kOffRaw % 16 == 0, "bulk copies need 16-byte alignment");
static_assert(kOffSfb % 128 == 0, "scale-factor copies start on a 16-byte boundary");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kD % (kLayWarps * 32) == 0, "layout threads cover the channels evenly");
static_assert(kTmemSF1 < kTmemQ && kTmemSFB + 2 * 8 <= kTmemSF1, "TMEM plan");

// Instruction descriptor of the block-scaled FP4 MMA: A and B E2M1, UE4M3 scale
// factors (one per 16 elements, scale_vec::4X), scale-factor IDs 0, K = 64.
__host__ __device__ constexpr uint32_t make_idesc_mxf4(int M, int N) {
    return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D (+)= A B^T with A (E2M1 codes) in TMEM, B described in shared memory, and
// the scale factors of A and B in TMEM.
__device__ __forceinline__ void mma_mxf4_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], [%1], %2, %3, [%4], [%5], p;\n\t}\n"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Shared-memory descriptor of a plain (no swizzle) matrix of 16-byte rows
// stored one after another: 8-row groups 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(16 >> 4) << 16;              // leading byte offset (one 16-byte column)
    d |= static_cast<uint64_t>(128 >> 4) << 32;             // stride byte offset: next 8 rows
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version for tcgen05
    return d;                                               // layout type 0: no swizzle
}

// 32 rows x 128 bits from shared memory into TMEM columns taddr .. taddr + 3,
// row r into lane r of every lane quarter (asynchronous, ordered before the
// MMAs this thread issues after it).
__device__ __forceinline__ void tc_cp_rows_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

struct Bars {
    uint64_t *q_full, *k_full, *k_empty, *s_ready, *v_full, *raw_full, *raw_empty, *p_full, *pv_done, *drain;
};

struct Params {
    const uint8_t *q8, *v_code, *v_sf;
    const float *sq, *sk, *v_scale;
    const uint16_t *v_mean;
    uint16_t *O;
    int32_t *dev_status;
    int N;
    float scale_log2;
    uint64_t limit_ns;
};

// The mean-restore MMA for key blocks j-16 .. j-1 follows PV(j); the softmax
// stages its operands in step j, once block j-1's row sums are read.
__host__ __device__ constexpr bool flush_after(int j) { return j >= kMeanJ && (j % kMeanJ) == 0; }

// Largest raw score of each group of 16 of the thread's kCols keys.
__device__ __forceinline__ void group_max(const uint32_t (&S)[kCols], float (&gm)[kCols / 16]) {
#pragma unroll
    for (int g = 0; g < kCols / 16; ++g) {
        const uint32_t *s = S + 16 * g;
        const float a = max3(__uint_as_float(s[0]), __uint_as_float(s[1]), __uint_as_float(s[2]));
        const float b = max3(__uint_as_float(s[3]), __uint_as_float(s[4]), __uint_as_float(s[5]));
        const float c = max3(__uint_as_float(s[6]), __uint_as_float(s[7]), __uint_as_float(s[8]));
        const float d = max3(__uint_as_float(s[9]), __uint_as_float(s[10]), __uint_as_float(s[11]));
        const float e = max3(__uint_as_float(s[12]), __uint_as_float(s[13]), __uint_as_float(s[14]));
        gm[g] = fmaxf(max3(a, b, c), max3(d, e, __uint_as_float(s[15])));
    }
}

// NVFP4 P of this thread's kCols keys against the reference max m: per group
// of 16 keys p = 2^(fma(S, c, -m)), scale sf = E4M3(amax16 / 6), code =
// E2M1(p / dec(sf)); P gets the codes (key k of the thread's keys at word
// k / 8, nibble k % 8), sfa the four scale bytes (group g in byte g).
// With c > 0, S -> 2^(fma(S, c, -m)) does not decrease, so amax16 is 2 to
// the power of the group's largest score term (gm, from group_max).  The
// quotient amax16 / 6 is corrected by one FMA step,
// q = RN(a r), q' = RN(q + RN(a - 6q) r) with r = RN(1/6): equal to the IEEE
// quotient for every a in [2^-120, 2^30] (checked exhaustively), and below
// that both round to the E4M3 code 0.  p / dec(sf) is evaluated as
// 2^(fma(S, c, lg(sf) - m)) with lg(sf) = -log2(dec(sf)) from a per-CTA
// table of the 127 codes (sLg; -inf for code 0, whose group codes are 0):
// one FMA and one exp per key, the same hardware-exp accuracy as p itself.
__device__ __forceinline__ void nvfp4_p(const uint32_t (&S)[kCols], const float (&gm)[kCols / 16], float c, float m,
                                        const float *sLg, uint32_t (&P)[kCols / 8], uint32_t &sfa) {
    constexpr float kSixth = 1.0f / 6.0f;
    const float negm = -m;
    const uint64_t cx2 = pk2(__float_as_uint(c), __float_as_uint(c));
    sfa = 0u;
#pragma unroll
    for (int g = 0; g < kCols / 16; ++g) {
        const float amax = ex2_approx(__fmaf_rn(gm[g], c, negm));
        const float q0 = __fmul_rn(amax, kSixth);
        const float q1 = __fmaf_rn(__fmaf_rn(-q0, 6.0f, amax), kSixth, q0);
        const uint32_t sf = e4m3x2(q1, 0.0f) & 0xFFu;
        sfa |= sf << (8 * g);
        const float bias = __fadd_rn(sLg[sf], negm);
        const uint64_t bx2 = pk2(__float_as_uint(bias), __float_as_uint(bias));
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            float x[8];
#pragma unroll
            for (int q = 0; q < 8; q += 2) {
                float t0, t1;
                upk2(fma2(pk2(S[16 * g + 8 * w + q], S[16 * g + 8 * w + q + 1]), cx2, bx2), t0, t1);
                x[q] = ex2_approx(t0);
                x[q + 1] = ex2_approx(t1);
            }
            P[2 * g + w] = e2m1x8(x);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_nvfp4_kernel(const __grid_constant__ CUtensorMap tmK, const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    Bars B;
    B.q_full = bars;
    B.k_full = B.q_full + 1;
    B.k_empty = B.k_full + kKStages;
    B.s_ready = B.k_empty + kKStages;
    B.v_full = B.s_ready + 2;
    B.raw_full = B.v_full + kVStages;
    B.raw_empty = B.raw_full + kRawStages;
    B.p_full = B.raw_empty + kRawStages;
    B.pv_done = B.p_full + 1;
    B.drain = B.pv_done + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    int *abort_flag = reinterpret_cast<int *>(smem + kOffMisc + 4);
    float *sRS = reinterpret_cast<float *>(smem + kOffRS);
    float *sSV = reinterpret_cast<float *>(smem + kOffSV);
    float *sPM = reinterpret_cast<float *>(smem + kOffPM);
    float *sL = reinterpret_cast<float *>(smem + kOffL);
    float *sLg = reinterpret_cast<float *>(smem + kOffLg);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qtile = blockIdx.x, bh = blockIdx.y;
    const int N = p.N, nb = N / kBlk;

    if (threadIdx.x == 0) {
        mbar_init(B.q_full, 4);   // the four warps that store Q into TMEM
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(B.k_full + s, 1);
            mbar_init(B.k_empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(B.s_ready + i, 1);
            mbar_init(B.pv_done + i, 1);
        }
        for (int i = 0; i < kVStages; ++i) mbar_init(B.v_full + i, kLayWarps);
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(B.raw_full + s, 1);
            mbar_init(B.raw_empty + s, kLayWarps);
        }
        mbar_init(B.p_full, kSoftmaxWarps);
        mbar_init(B.drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp >= 2 && warp < 6) {
        const int t = threadIdx.x - 64;
        sSV[t] = p.v_scale[bh];
        // scale tables for the E4M3 codes (127 = NaN is never produced)
        sLg[t] = (t == 0 || t == 127) ? __int_as_float(0xff800000) : -log2f(e4m3_to_f32(static_cast<uint32_t>(t)));
        // the row-sum MMA's B: 16 rows of E2M1 1.0 (every nibble 2)
        const uint4 ones = make_uint4(0x22222222u, 0x22222222u, 0x22222222u, 0x22222222u);
        *reinterpret_cast<uint4 *>(smem + kOffOnes + 16 * t) = ones;
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kKWarp) {
        // ------------------------------------------------------------ K producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            int armed[kKStages];
            for (int s = 0; s < kKStages; ++s) armed[s] = 0;
            for (int b = 0; b < nb; ++b) {
                const int s = b % kKStages, use = b / kKStages;
                if (use > 0 && !mbar_wait(B.k_empty + s, (use - 1) & 1, abort_flag, p.limit_ns)) break;
                mbar_expect_tx(B.k_full + s, kTileBytes);
                tma_load_2d(smem + kOffK + s * kTileBytes, &tmK, B.k_full + s, 0, bh * N + b * kBlk);
                armed[s] = use + 1;
            }
            for (int s = 0; s < kKStages; ++s)
                if (armed[s] > 0) drain_wait(B.k_full + s, (armed[s] - 1) & 1, p.limit_ns);
        }
    } else if (warp == kLayWarp0 || warp == kLayWarp1) {
        // ------------------------------------------------------------ V layout
        // Per channel ch: the 64 bytes of its 128 E2M1 codes (token 2i in the
        // low nibble of byte i) as the first four 16-byte chunks of row ch of
        // the swizzled tile.  The block's V scales are staged for the MMA
        // issuer's copy into TMEM: for keys 64h.. (MMA h), row r of matrix
        // (v, h) holds the four scales of channels r, r + 32, r + 64, r + 96
        // (the MMA reads channel n's from lane n % 32 of the D row's lane
        // quarter, column n / 32).
        const bool lanes0 = warp == kLayWarp0;
        const int t0 = (lanes0 ? 0 : 32) + lane;
        const bool copier = (lanes0 && lane == 0);
        int armed[kRawStages];
        for (int s = 0; s < kRawStages; ++s) armed[s] = 0;
        // block b's codes and scales into raw stage b % kRawStages, which the
        // layout of block b - kRawStages (both warps) has released
        auto copy_block = [&](int b) -> bool {
            const int s = b % kRawStages, use = b / kRawStages;
            if (use > 0 && !mbar_wait(B.raw_empty + s, (use - 1) & 1, abort_flag, p.limit_ns)) return false;
            const int64_t blk = static_cast<int64_t>(bh) * nb + b;
            unsigned char *dst = smem + kOffRaw + s * kRawStageBytes;
            mbar_expect_tx(B.raw_full + s, kRawStageBytes);
            bulk_load(dst, p.v_code + blk * kCodeBytes, kCodeBytes, B.raw_full + s);
            bulk_load(dst + kCodeBytes, p.v_sf + blk * kSfBytes, kSfBytes, B.raw_full + s);
            armed[s] = use + 1;
            return true;
        };
        bool cok = true;
        if (copier)
            for (int b = 0; cok && b < kRawStages - 1 && b < nb; ++b) cok = copy_block(b);
        for (int j = 0; j < nb; ++j) {
            const int s = j % kRawStages, v = j & 1;
            if (copier && cok && j + kRawStages - 1 < nb) cok = copy_block(j + kRawStages - 1);
            bool ok = cok && mbar_wait(B.raw_full + s, (j / kRawStages) & 1, abort_flag, p.limit_ns);
            // tile v and the V-scale buffer v were last read by PV(j-2)
            if (ok && j >= 2) ok = mbar_wait(B.pv_done + (j & 1), ((j - 2) >> 1) & 1, abort_flag, p.limit_ns);
            if (!__all_sync(0xffffffffu, ok)) break;
            const unsigned char *raw = smem + kOffRaw + s * kRawStageBytes;
            unsigned char *vs = smem + kOffV + v * kVStageBytes;
#pragma unroll
            for (int t = t0; t < kD; t += 32 * kLayWarps) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<uint4 *>(vs + sw128_offset(t, i)) =
                        reinterpret_cast<const uint4 *>(raw + t * (kBlk / 2))[i];
            }
            {
                const int h = t0 >> 5;   // thread t0 stages row lane of matrix (v, h)
                const unsigned char *sf = raw + kCodeBytes + 4 * h;
                uint4 w;
                w.x = *reinterpret_cast<const uint32_t *>(sf + (lane + 0) * (kBlk / 16));
                w.y = *reinterpret_cast<const uint32_t *>(sf + (lane + 32) * (kBlk / 16));
                w.z = *reinterpret_cast<const uint32_t *>(sf + (lane + 64) * (kBlk / 16));
                w.w = *reinterpret_cast<const uint32_t *>(sf + (lane + 96) * (kBlk / 16));
                *reinterpret_cast<uint4 *>(smem + kOffSfb + (2 * v + h) * kSfbBytes + 16 * lane) = w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(B.raw_empty + s);
            fence_proxy_async_smem();   // the tile is read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(B.v_full + v);
        }
        // every copy this thread issued has landed before the CTA can exit
        if (copier)
            for (int s = 0; s < kRawStages; ++s)
                if (armed[s] > 0) drain_wait(B.raw_full + s, (armed[s] - 1) & 1, p.limit_ns);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = make_idesc(128, 128, 0, 0);    // E4M3 x E4M3
            constexpr uint32_t idesc_pv = make_idesc_mxf4(128, 128);     // NVFP4 x NVFP4
            constexpr uint32_t idesc_rs = make_idesc_mxf4(128, kOnesRows);
            constexpr uint32_t idesc_bf16 = make_idesc(128, 128, 1, 1);  // BF16 x BF16
            const uint32_t sbase = smem_u32(smem);
            const uint64_t dma = sdesc_k_sw128(sbase + kOffMA);
            const uint64_t dmb = sdesc_k_sw128(sbase + kOffMB);
            const uint32_t tO = tmem + kTmemO;
            // QK(b) into S[b & 1]; S(b-2) was read before P(b-2) was released
            auto issue_qk = [&](int b) -> bool {
                const int s = b % kKStages;
                if (!mbar_wait(B.k_full + s, (b / kKStages) & 1, abort_flag, p.limit_ns)) return false;
                tc_fence_after();
                const uint64_t dk = sdesc_k_sw128(sbase + kOffK + s * kTileBytes);
#pragma unroll
                for (int kk = 0; kk < kD / 32; ++kk)
                    mma_f8f6f4_ts(tmem + (b & 1) * 128, tmem + kTmemQ + 8 * kk, dk + 2 * kk, idesc_qk, kk > 0);
                tc_commit(B.k_empty + s);
                tc_commit(B.s_ready + (b & 1));
                return true;
            };
            bool ok = mbar_wait(B.q_full, 0, abort_flag, p.limit_ns);
            for (int b = 0; ok && b < 2 && b < nb; ++b) ok = issue_qk(b);
            for (int j = 0; ok && j < nb; ++j) {
                if (!mbar_wait(B.v_full + (j & 1), (j >> 1) & 1, abort_flag, p.limit_ns)) break;
                tc_fence_after();
                // block j's V scales into every lane quarter (buffer j & 1 was
                // last read by PV(j-2), which finished before tile j was laid out)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    tc_cp_rows_x4(tmem + kTmemSFB + 8 * (j & 1) + 4 * h,
                                  sdesc_rows16(sbase + kOffSfb + (2 * (j & 1) + h) * kSfbBytes));
                if (!mbar_wait(B.p_full, j & 1, abort_flag, p.limit_ns)) break;
                tc_fence_after();
                // O += P V and E_{j&1} = P ones, keys 64h .. 64h+63 per MMA
                // (A columns 8h.., B bytes 32h.. of every row, scales at +4h)
                const uint64_t dv = sdesc_k_sw128(sbase + kOffV + (j & 1) * kVStageBytes);
                const uint64_t d1 = sdesc_k_sw128(sbase + kOffOnes);
                const uint32_t te = tmem + ((j & 1) ? kTmemE1 : kTmemE0);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    mma_mxf4_ts(tO, tmem + kTmemP + 8 * h, dv + 2 * h, idesc_pv, tmem + kTmemSFA + 4 * h,
                                tmem + kTmemSFB + 8 * (j & 1) + 4 * h, (j > 0 || h > 0) ? 1u : 0u);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    mma_mxf4_ts(te, tmem + kTmemP + 8 * h, d1 + 2 * h, idesc_rs, tmem + kTmemSFA + 4 * h, tmem + kTmemSF1,
                                h > 0 ? 1u : 0u);
                if (flush_after(j)) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma_f16(tO, dma + 2 * kk, dmb + 2 * kk, idesc_bf16, 1u);
                }
                tc_commit(B.pv_done + (j & 1));
                if (j + 2 < nb) ok = issue_qk(j + 2);
            }
            tc_commit(B.drain);
            drain_wait(B.drain, 0, p.limit_ns);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3;                              // TMEM lane quarter
        const int half = (warp - 2) >> 2;                          // column half: keys kCols*half ..
        const int row = quarter * 32 + lane;                       // query row in the tile == TMEM lane
        const uint32_t pair_bar = kBarPair0 + quarter;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t col0 = static_cast<uint32_t>(kCols) * half;
        const uint32_t tO = tmem + lane_base + kTmemO + col0;
        const uint32_t tP = tmem + lane_base + kTmemP + (kCols / 8) * half;       // this half's codes
        // its scales: the MMA reads row m's from lane m, column base + m / 32
        const uint32_t tSFA = tmem + lane_base + kTmemSFA + 4 * half + quarter;
        const float sqv = p.sq[static_cast<int64_t>(bh) * nb + qtile];
        const float *skh = p.sk + static_cast<int64_t>(bh) * nb;
        const uint16_t *vmh = p.v_mean + static_cast<int64_t>(bh) * nb * kD;
        unsigned char *sMA = smem + kOffMA;
        unsigned char *sMB = smem + kOffMB;
        const float kNegInf = __int_as_float(0xff800000);
        float m = kNegInf;    // reference max
        float l = 0.0f;       // kept by the half-0 thread of the row
        int rs_cnt = 0;
        bool ok = true;
        float sk_next = skh[0];
        if (half == 0) {
            load_q_row(p.q8 + (static_cast<int64_t>(bh) * N + static_cast<int64_t>(qtile) * kBlk + row) * kD,
                       tmem + lane_base + kTmemQ);
            // the row-sum MMA's B scales (E4M3 1.0), read in every lane quarter
            asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tmem + lane_base + kTmemSF1),
                         "r"(0x38383838u) : "memory");
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.q_full);
        }
        for (int b = 0; b < nb; ++b) {
            const int sb = b & 1;
            const float sk_b = sk_next;
            if (b + 1 < nb) sk_next = skh[b + 1];
            const float c = __fmul_rn(__fmul_rn(sqv, sk_b), p.scale_log2);
            bool wok = mbar_wait(B.s_ready + sb, (b >> 1) & 1, abort_flag, p.limit_ns);
            wok = __all_sync(0xffffffffu, wok) && ok;
            uint32_t S[kCols];
            float gm[kCols / 16];
            float pm = kNegInf;
            if (wok) {
                tc_fence_after();
                const uint32_t tS = tmem + lane_base + sb * 128 + col0;
#pragma unroll
                for (int i = 0; i < kCols / 32; ++i) VCA_TMEM_LD32(tS + 32 * i, (S + 32 * i));
                tmem_ld_wait();
                group_max(S, gm);
                pm = gm[0];
#pragma unroll
                for (int g = 1; g < kCols / 16; ++g) pm = fmaxf(pm, gm[g]);
                sPM[(sb * kParts + half) * kBlk + row] = pm;
            }
            ok = bar_and(wok, pair_bar, 32 * kParts);
            if (!ok) break;
            float smax = pm;
#pragma unroll
            for (int q = 1; q < kParts; ++q) smax = fmaxf(smax, sPM[(sb * kParts + ((half + q) % kParts)) * kBlk + row]);
            const float bm = __fmul_rn(smax, c);
            // lazy reference-max update: only when the block's max exceeds it by tau
            float alpha = 1.0f;
            if (bm > __fadd_rn(m, kLazyTau)) {
                if (b > 0) alpha = ex2_approx(__fsub_rn(m, bm));
                m = bm;
            }
            uint32_t P[kCols / 8], sfa;
            nvfp4_p(S, gm, c, m, sLg, P, sfa);
            // PV(b-1) is done: the P buffer and O are free, block b-1's row sums
            // are in their slot
            if (b >= 1) ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done + ((b - 1) & 1), ((b - 1) >> 1) & 1, abort_flag,
                                                                p.limit_ns));
            if (ok) {
                tc_fence_after();
                if (half == 0 && b >= 1) {
                    // read block b-1's sums (taken against the max before this
                    // block's update); PV(b)'s row-sum MMA overwrites this
                    // block's slot
                    const uint32_t te_prev = tmem + lane_base + (sb ? kTmemE0 : kTmemE1);
                    uint32_t rs_raw;
                    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(rs_raw) : "r"(te_prev));
                    tmem_ld_wait();
                    const float rs = __uint_as_float(rs_raw);
                    l = __fadd_rn(l, rs);
                    sRS[rs_cnt * kBlk + row] = rs;
                }
                if (b >= 1) ++rs_cnt;
                if (__any_sync(0xffffffffu, alpha != 1.0f)) {
                    if (half == 0 && alpha != 1.0f) {
                        l = __fmul_rn(l, alpha);
#pragma unroll 1
                        for (int i = 0; i < rs_cnt; ++i) sRS[i * kBlk + row] = __fmul_rn(sRS[i * kBlk + row], alpha);
                    }
#pragma unroll 1
                    for (int i = 0; i < kCols / 32; ++i) {
                        uint32_t o[32];
                        VCA_TMEM_LD32(tO + 32 * i, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__fmul_rn(__uint_as_float(o[e]), alpha));
                        VCA_TMEM_ST32(tO + 32 * i, o);
                    }
                }
                if (flush_after(b)) {
                    // row sums of blocks b-16 .. b-1 (all at the current max)
                    stage_mean_operands(half, row, sRS, vmh, b - kMeanJ, sSV, sMA, sMB);
                    rs_cnt = 0;
                    fence_proxy_async_smem();   // the mean operands are read by the tensor core
                }
                VCA_TMEM_ST8(tP, P);
                asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tSFA), "r"(sfa) : "memory");
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(B.p_full);
            }
        }
        // ------------------------------------------------------------ epilogue
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done + ((nb - 1) & 1), ((nb - 1) >> 1) & 1, abort_flag,
                                                        p.limit_ns));
        // every softmax warp arrives here, whether it finished or gave up; the
        // epilogue (and its barriers) runs only if all of them finished
        ok = bar_and(ok, kBarSoftmax, 32 * kSoftmaxWarps);
        if (ok) {
            tc_fence_after();
            if (half == 0) {
                // the last block's row sums, taken against m itself
                uint32_t r1;
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                             : "=r"(r1)
                             : "r"(tmem + lane_base + (((nb - 1) & 1) ? kTmemE1 : kTmemE0)));
                tmem_ld_wait();
                const float rs = __uint_as_float(r1);
                l = __fadd_rn(l, rs);
                sRS[rs_cnt * kBlk + row] = rs;
                sL[row] = l;
            }
            ++rs_cnt;
            // the blocks since the last mean MMA: stage their means (fp32) in the
            // mean-B buffer, whose last reader (the final mean MMA) has finished
            const int tail0 = nb - rs_cnt;
            float *sMu = reinterpret_cast<float *>(sMB);
            bar_sync(kBarSoftmax, 32 * kSoftmaxWarps);
            for (int i = threadIdx.x - 64; i < rs_cnt * kD; i += 32 * kSoftmaxWarps)
                sMu[i] = bf16_bits_to_f32(vmh[(tail0 + i / kD) * kD + (i % kD)]);
            bar_sync(kBarSoftmax, 32 * kSoftmaxWarps);
            const float inv_l = 1.0f / sL[row];
            uint16_t *orow = p.O + (static_cast<int64_t>(bh) * N + static_cast<int64_t>(qtile) * kBlk + row) * kD + col0;
            store_output(tO, sSV, sRS, sMu, rs_cnt, 0, row, static_cast<int>(col0), inv_l, orow);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 0 && *reinterpret_cast<volatile int *>(abort_flag) && p.dev_status)
        atomicExch(p.dev_status, kErrTimeout);
}

}  // namespace

cudaError_t launch_attention_nvfp4(const AttentionArgs &a, cudaStream_t st) {
    CUtensorMap mk;
    const uint64_t rows = static_cast<uint64_t>(a.BH) * a.N;
    if (!make_tile_map(&mk, a.k8, rows)) return cudaErrorInvalidValue;
    Params p;
    p.q8 = a.q8;
    p.v_code = a.v_res;
    p.v_sf = a.v_sf;
    p.sq = a.sq;
    p.sk = a.sk;
    p.v_scale = a.v_scale;
    p.v_mean = a.v_mean;
    p.O = a.O;
    p.dev_status = a.dev_status;
    p.N = a.N;
    p.scale_log2 = a.scale_log2;
    p.limit_ns = a.wait_limit_ns;
    const cudaError_t e =
        cudaFuncSetAttribute(attention_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attention_nvfp4_kernel<<<dim3(a.N / kBlk, a.BH), kThreads, kSmemBytes, st>>>(mk, p);
    return cudaGetLastError();
}

}  // namespace vca
