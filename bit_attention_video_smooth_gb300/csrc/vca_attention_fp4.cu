// vca_attention_fp4.cu -- the 4-bit VC-Attention kernel (paper page, "method":
// the residual left after demeaning is quantised to NVFP4 for the 4-bit
// path): V residual as NVFP4 (E2M1 codes, one E4M3 scale per 16 tokens of a
// channel, one fp32 scale g per head) and P as NVFP4 (E2M1 codes, one E4M3
// scale per 16 keys of a row), with the V-Smooth mean restore of the 8-bit
// kernel.
//
// PV runs on the tensor core as kind::f16 on the decoded operands: an E2M1
// value times an E4M3 scale has at most 6 significant bits and lies in
// [2^-10, 2688] (V) or [2^-10, 256] (P), so decoded P and decoded V are exact
// in f16 and the MMA forms exactly the products a block-scaled FP4 MMA forms,
// summed in fp32.  QK stays E4M3 (kind::f8f6f4).
//
// One CTA owns a 128-row query tile of one (batch, head).  Warp roles:
//   warp 0       TMA producer: K tiles into a 3-stage ring
//   warp 1       TMEM owner and MMA issuer (one thread); per key block j:
//                  [E | O] += P_j [ones ; Vhat_j]   (kind::f16, N = 144: the 16
//                             extra columns are P_j's row sums), then the
//                             mean-restore MMA when due, then
//                  S[j&1] = Q8 K8_{j+2}^T             (kind::f8f6f4)
//   warps 10-11  V decode: two channels per thread; E2M1 x E4M3 -> f16 in the
//                128-byte-swizzled K-major layout of the PV B operand.  Lane 0
//                of warp 10 also bulk-copies block j+3's packed codes (8 KB)
//                and scales (1 KB) into a 4-stage ring.
//   warps 2-9    softmax, two threads per query row (column halves): running
//                max with the lazy threshold, NVFP4 P of the row against it,
//                P into TMEM once PV(j-1) is done, row sum of block j-1 from
//                its TMEM slot, O rescale, mean-restore operands, epilogue.
// P has a single TMEM buffer (the budget holds no second one), so P_j is
// written after PV(j-1) completes; the softmax computes P_j while PV(j-1) runs.
// TMEM columns: S0 [0,128), S1 [128,256), E0 [256,272), O [272,400),
// E1 [400,416), P [416,480) (f16, two keys per column), Q [480,512).
// Every wait is bounded; a wait that runs out raises a CTA-wide abort, the CTA
// drains its copies and MMAs, frees TMEM and reports VCA_ERR_TIMEOUT.
#include "vca_attention_common.cuh"
#include "vca_internal.h"

namespace vca {

namespace {

using namespace attn;

constexpr int kKStages = 3;                  // K tiles in flight
constexpr int kRawStages = 4;                // packed V blocks in flight
constexpr int kVStages = 2;                  // decoded f16 V tiles
constexpr int kDecWarp0 = 2 + kSoftmaxWarps; // first V-decode warp (its lane 0 also copies)
constexpr int kDecWarps = 2;                 // two channels per thread
// 12 warps: at most three per SM sub-partition, so up to 168 registers a thread
constexpr int kThreads = 32 * (kDecWarp0 + kDecWarps);
constexpr int kRsCap = kMeanJ;               // buffered row sums per row

constexpr uint32_t kTileBytes = kBlk * kD;              // one 128 x 128 FP8 K tile
constexpr uint32_t kCodeBytes = kD * kBlk / 2;          // a block's E2M1 codes, [ch][64 bytes]
constexpr uint32_t kSfBytes = kD * kBlk / 16;           // a block's E4M3 scales, [ch][8]
constexpr uint32_t kRawStageBytes = kCodeBytes + kSfBytes;
constexpr uint32_t kOnesRows = 16;
// A decoded V tile is two K panels (keys 0-63, 64-127) of 128-byte rows (64
// f16), each [16 rows of 1.0 | 128 channel rows | 16 rows of 1.0].
constexpr uint32_t kPanelBytes = (kOnesRows + kD + kOnesRows) * 128;
constexpr uint32_t kVStageBytes = 2 * kPanelBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemE0 = 256, kTmemO = 272, kTmemE1 = 400, kTmemP = 416, kTmemQ = 480;

constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffRaw = kOffV + kVStages * kVStageBytes;
constexpr uint32_t kOffMA = kOffRaw + kRawStages * kRawStageBytes;
constexpr uint32_t kOffMB = kOffMA + kTileBytes;
constexpr uint32_t kOffRS = kOffMB + kTileBytes;            // fp32 [kRsCap][128] buffered row sums
constexpr uint32_t kOffSV = kOffRS + kRsCap * kBlk * 4;     // fp32 [128]: g for every channel
constexpr uint32_t kOffPM = kOffSV + kBlk * 4;              // fp32 [2][kParts][128] part-row maxima
constexpr uint32_t kOffL = kOffPM + 2 * kParts * kBlk * 4;  // fp32 [128] final row sums
constexpr uint32_t kOffRcp = kOffL + kBlk * 4;              // fp32 [128]: 1 / dec(E4M3 code), 0 for code 0
constexpr uint32_t kOffSf2 = kOffRcp + kBlk * 4;            // u32 [128]: dec(E4M3 code) as f16 in both halves
constexpr uint32_t kOffBar = kOffSf2 + kBlk * 4;
constexpr int kNumBars = 1 + 2 * kKStages + 2 + kVStages + 2 * kRawStages + 1 + 2 + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;       // tmem address, abort flag
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;       // + alignment slack
static_assert(kOffV % 1024 == 0 && kPanelBytes % 1024 == 0 && kOffMA % 1024 == 0 && kOffMB % 1024 == 0,
              "swizzled operand tiles need 1024-byte alignment");
static_assert(kRawStageBytes % 16 == 0 && kOffRaw % 16 == 0, "bulk copies need 16-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kD % (kDecWarps * 32) == 0, "decode threads cover the channels evenly");

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

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// f16 pattern of an E4M3 byte, in both halves of a word.
__device__ __forceinline__ uint32_t e4m3_f16x2_splat(uint32_t code) {
    const uint32_t h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3).x;
    return h | (h << 16);
}

// The four bytes of w, each two E2M1 nibbles -> f16x2 (the low nibble in the
// low half): d[i] from byte i.
__device__ __forceinline__ void e2m1x8_f16x2(uint32_t w, uint32_t &d0, uint32_t &d1, uint32_t &d2, uint32_t &d3) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
        : "r"(w));
}

// (lo, hi) rounded to E2M1 (nearest even, saturating at 6) and decoded back,
// as f16x2 (lo in the low half).
__device__ __forceinline__ uint32_t e2m1_round_f16x2(float lo, float hi) {
    uint32_t d;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(d)
        : "f"(lo), "f"(hi));
    return d;
}

// NVFP4 P of this thread's kCols keys against the reference max m: per group
// of 16 keys p = 2^(fma(S, c, -m)), scale sf = E4M3(amax16 / 6), code =
// E2M1(p * (1 / dec(sf))), decoded value code * dec(sf) as f16 (exact), two
// keys per word.  amax16 / 6 is the quotient corrected by one FMA step,
// q = RN(a r), q' = RN(q + RN(a - 6q) r) with r = RN(1/6): equal to the IEEE
// quotient for every a in [2^-120, 2^30] (checked exhaustively), and below
// that both round to the E4M3 code 0.  The reciprocal and the f16 pattern of
// the scale come from per-CTA tables of the 127 codes (sRcp, sSf2).
__device__ __forceinline__ void nvfp4_p(const uint32_t (&S)[kCols], float c, float m, const float *sRcp,
                                        const uint32_t *sSf2, uint32_t (&P)[kCols / 2]) {
    constexpr float kSixth = 1.0f / 6.0f;
    const float negm = -m;
    const uint64_t cx2 = pk2(__float_as_uint(c), __float_as_uint(c));
    const uint64_t nx2 = pk2(__float_as_uint(negm), __float_as_uint(negm));
#pragma unroll
    for (int g = 0; g < kCols / 16; ++g) {
        float pv[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float t0, t1;
            upk2(fma2(pk2(S[16 * g + 2 * q], S[16 * g + 2 * q + 1]), cx2, nx2), t0, t1);
            pv[2 * q] = ex2_approx(t0);
            pv[2 * q + 1] = ex2_approx(t1);
        }
        float a[4] = {pv[0], pv[1], pv[2], pv[3]};
#pragma unroll
        for (int j = 4; j < 16; j += 2) a[(j >> 1) & 3] = max3(a[(j >> 1) & 3], pv[j], pv[j + 1]);
        const float amax = fmaxf(max3(a[0], a[1], a[2]), a[3]);
        const float q0 = __fmul_rn(amax, kSixth);
        const float q1 = __fmaf_rn(__fmaf_rn(-q0, 6.0f, amax), kSixth, q0);
        const uint32_t sf = e4m3x2(q1, 0.0f) & 0xFFu;
        const float inv = sRcp[sf];
        const uint32_t sf2 = sSf2[sf];
        const uint64_t inv2 = pk2(__float_as_uint(inv), __float_as_uint(inv));
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            float x0, x1;
            upk2(mul2(pk2(__float_as_uint(pv[2 * q]), __float_as_uint(pv[2 * q + 1])), inv2), x0, x1);
            P[8 * g + q] = f16x2_mul(e2m1_round_f16x2(x0, x1), sf2);
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
    float *sRcp = reinterpret_cast<float *>(smem + kOffRcp);
    uint32_t *sSf2 = reinterpret_cast<uint32_t *>(smem + kOffSf2);

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
        for (int i = 0; i < kVStages; ++i) mbar_init(B.v_full + i, kDecWarps);
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(B.raw_full + s, 1);
            mbar_init(B.raw_empty + s, kDecWarps);
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
        sRcp[t] = (t == 0 || t == 127) ? 0.0f : __frcp_rn(e4m3_to_f32(static_cast<uint32_t>(t)));
        sSf2[t] = e4m3_f16x2_splat(static_cast<uint32_t>(t));
        // the rows of f16 1.0 at both ends of every panel
        const uint4 ones = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
        for (int st = 0; st < kVStages; ++st)
            for (int pn = 0; pn < 2; ++pn) {
                unsigned char *panel = smem + kOffV + st * kVStageBytes + pn * kPanelBytes;
                *reinterpret_cast<uint4 *>(panel + 16 * t) = ones;
                *reinterpret_cast<uint4 *>(panel + (kOnesRows + kD) * 128 + 16 * t) = ones;
            }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
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
    } else if (warp >= kDecWarp0) {
        // ------------------------------------------------------------ V decode
        // Per channel ch: 128 E2M1 codes (token 2i in the low nibble of byte
        // i) and 8 E4M3 scales -> 128 f16 values, written as 16-byte chunks
        // (8 keys) of row 16 + ch of the two K panels.
        const int t0 = threadIdx.x - 32 * kDecWarp0;
        const bool copier = (warp == kDecWarp0 && lane == 0);
        int armed[kRawStages];
        for (int s = 0; s < kRawStages; ++s) armed[s] = 0;
        // block b's codes and scales into raw stage b % kRawStages, which the
        // decode of block b - kRawStages (both warps) has released
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
            // decoded stage v was last read by PV(j-2)
            if (ok && j >= 2) ok = mbar_wait(B.pv_done + (j & 1), ((j - 2) >> 1) & 1, abort_flag, p.limit_ns);
            if (!__all_sync(0xffffffffu, ok)) break;
            const unsigned char *raw = smem + kOffRaw + s * kRawStageBytes;
            unsigned char *vs = smem + kOffV + v * kVStageBytes;
#pragma unroll 1
            for (int t = t0; t < kD; t += 32 * kDecWarps) {
                uint32_t code[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 u = reinterpret_cast<const uint4 *>(raw + t * (kBlk / 2))[i];
                    code[4 * i] = u.x;
                    code[4 * i + 1] = u.y;
                    code[4 * i + 2] = u.z;
                    code[4 * i + 3] = u.w;
                }
                const uint2 sfw = *reinterpret_cast<const uint2 *>(raw + kCodeBytes + t * (kBlk / 16));
#pragma unroll
                for (int g = 0; g < kBlk / 16; ++g) {
                    const uint32_t sf2 = e4m3_f16x2_splat(((g < 4 ? sfw.x : sfw.y) >> (8 * (g & 3))) & 0xFFu);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t w = code[2 * g + h];   // keys 16g + 8h .. +7
                        uint4 o;
                        e2m1x8_f16x2(w, o.x, o.y, o.z, o.w);
                        o.x = f16x2_mul(o.x, sf2);
                        o.y = f16x2_mul(o.y, sf2);
                        o.z = f16x2_mul(o.z, sf2);
                        o.w = f16x2_mul(o.w, sf2);
                        const int panel = g >> 2, chunk = (2 * g + h) & 7;
                        *reinterpret_cast<uint4 *>(vs + panel * kPanelBytes + sw128_offset(kOnesRows + t, chunk)) = o;
                    }
                }
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
            constexpr uint32_t idesc_pv = make_idesc(128, 144, 0, 0);    // F16 x F16
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
                if (!mbar_wait(B.p_full, j & 1, abort_flag, p.limit_ns)) break;
                tc_fence_after();
                // even j: B = [ones ; V], D = [E0 | O]; odd j: B = [V ; ones], D = [O | E1]
                const uint32_t vstage = sbase + kOffV + (j & 1) * kVStageBytes + ((j & 1) ? kOnesRows * 128 : 0);
                const uint32_t td = tmem + ((j & 1) ? kTmemO : kTmemE0);
#pragma unroll
                for (int kk = 0; kk < kBlk / 16; ++kk)
                    mma_f16_ts(td, tmem + kTmemP + 8 * kk, sdesc_k_sw128(vstage + (kk >> 2) * kPanelBytes) + 2 * (kk & 3),
                               idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
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
        const uint32_t tP = tmem + lane_base + kTmemP + (kCols / 2) * half;
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
            float pm = kNegInf;
            if (wok) {
                tc_fence_after();
                const uint32_t tS = tmem + lane_base + sb * 128 + col0;
#pragma unroll
                for (int i = 0; i < kCols / 32; ++i) VCA_TMEM_LD32(tS + 32 * i, (S + 32 * i));
                tmem_ld_wait();
                pm = row_part_max(S);
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
            uint32_t P[kCols / 2];
            nvfp4_p(S, c, m, sRcp, sSf2, P);
            // PV(b-1) is done: the P buffer and O are free, block b-1's row sums
            // are in their slot
            if (b >= 1) ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done + ((b - 1) & 1), ((b - 1) >> 1) & 1, abort_flag,
                                                                p.limit_ns));
            if (ok) {
                tc_fence_after();
                if (half == 0 && b >= 1) {
                    // read block b-1's sums (taken against the max before this
                    // block's update) and clear this block's slot for PV(b)
                    const uint32_t te_prev = tmem + lane_base + (sb ? kTmemE0 : kTmemE1);
                    const uint32_t te_cur = tmem + lane_base + (sb ? kTmemE1 : kTmemE0);
                    uint32_t rs_raw;
                    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(rs_raw) : "r"(te_prev));
                    tmem_ld_wait();
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};"
                        ::"r"(te_cur), "r"(0u) : "memory");
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
                VCA_TMEM_ST32(tP, P);
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
