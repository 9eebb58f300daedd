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
// E4M3 (kind::f8f6f4).  Layouts (measured on the hardware with probes): P key
// k at TMEM column k / 8, nibble k % 8; row m's four scales of a 64-key MMA in
// lane m, column sfa + m / 32; B row n's, for the D rows of lane quarter q, in
// lane 32 q + n % 32, column sfb + n / 32, so the V scales (and the ones'
// scales of the row-sum MMA) are present in all four lane quarters; the V
// codes of a block as TMA writes them with the 64-byte swizzle (64-byte
// channel rows, the block's 128 keys), a K-major B operand whose second
// 64-key half starts 32 bytes into the rows.
//
// One CTA owns a 128-row query tile of one (batch, head); the organisation is
// the 8-bit kernel's.  Warp roles:
//   warp 0     TMA producer: the Q tile once, then K tiles into a 3-stage ring
//   warp 10    V producer: lane 0 loads each block's codes (TMA) and scales
//              (bulk copy) into a 4-stage ring, three blocks ahead; the warp
//              then lays the block's scales out as the two 32-row matrices the
//              PV issuer copies into TMEM (one copy fills all four lane
//              quarters) and marks the stage ready
//   warp 11    QK issuer (one thread): S[b&1] = Q8 K8_b^T (kind::f8f6f4, both
//              operands in shared memory) once K(b) has landed and S(b-2)
//              has been read
//   warp 1     TMEM owner and PV issuer (one thread), per key block j:
//                the V scales into TMEM (two buffers, by block parity),
//                O += P_j V_j, E_{j&1} = P_j ones   (two block-scaled MMAs
//                                  each, K = 64; the second gives the row sums)
//              and every 16 key blocks the bf16 mean-restore MMA
//   warps 2-9  softmax, one thread per query row and key block: warps w and
//              w+4 share a TMEM lane quarter and take the even and the odd key
//              blocks.  Per block: the row max from the group maxima of the
//              raw scores, the reference max handed over by the partner and
//              updated with the lazy threshold, NVFP4 P of the row (codes and
//              scales) into the P buffer of the block's parity, the row sum of
//              block b-2 from its TMEM slot, O rescaled when the max moves,
//              mean-restore operands when due, epilogue.
// Barriers between the softmax and the MMA threads, per parity of b: s_full
// (QK(b) committed), s_free (S(b) read), p_full (P(b) written), pv_done
// (PV(b), its row sums and the mean MMA after it committed).
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384), E0 [384,400),
// E1 [400,416), P0 [416,432), P1 [432,448) (eight E2M1 codes per column),
// P scales [448,456) and [456,464) per parity, V scales [464,472) and
// [472,480) per parity, the ones' scales 480 (Q stays in shared memory: TMEM
// has no room for it beside a second V-scale buffer).
// Every wait on an mbarrier is bounded; a wait that runs out raises a CTA-wide
// abort, the CTA drains its copies and MMAs, frees TMEM and reports
// VCA_ERR_TIMEOUT.  Each named-barrier wait is matched by an arrival on every
// path: a thread that gives up still hands on a reference max (NaN, which
// makes its partner give up at its next block) before leaving the loop.
#include "vca_attention_common.cuh"
#include "vca_internal.h"

namespace vca {

namespace {

using namespace attn;

constexpr int kKStages = 3;                  // K tiles in flight (released after their QK MMA)
constexpr int kVStages = 4;                  // V blocks in flight (released after their PV MMA)
constexpr int kVAhead = kVStages - 1;        // blocks the V loads run ahead of the layout
constexpr int kVWarp = 2 + kSoftmaxWarps;    // the V producer
constexpr int kQKWarp = kVWarp + 1;          // the QK issuer (the PV issuer is warp 1)
constexpr int kThreads = 32 * (kQKWarp + 1);

constexpr uint32_t kTileBytes = kBlk * kD;              // one 128 x 128 FP8 K tile
constexpr uint32_t kCodeBytes = kD * kBlk / 2;          // a block's E2M1 codes, [ch][64 bytes]
constexpr uint32_t kSfBytes = kD * kBlk / 16;           // a block's E4M3 scales, [ch][8]
constexpr uint32_t kSfbBytes = 32 * 16;                 // V scales of one 64-key MMA: 32 rows x 4 words
constexpr uint32_t kVStageBytes = kCodeBytes + kSfBytes + 2 * kSfbBytes;   // [codes | scales | laid-out scales]
constexpr uint32_t kOnesRows = 16;
constexpr uint32_t kOnesBytes = kOnesRows * 128;        // 16 rows of E2M1 1.0: the row-sum MMA's B
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256, kTmemE0 = 384, kTmemP0 = 416, kTmemSFA0 = 448, kTmemSFB = 464, kTmemSF1 = 480;

// shared-memory layout (bytes from a 1024-aligned base)
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffQ = kOffK + kKStages * kTileBytes;     // the Q tile (QK's A operand)
constexpr uint32_t kOffV = kOffQ + kTileBytes;
constexpr uint32_t kOffOnes = kOffV + kVStages * kVStageBytes;
constexpr uint32_t kOffMA = kOffOnes + kOnesBytes;
constexpr uint32_t kOffMB = kOffMA + kTileBytes;
constexpr uint32_t kMeanGroupBytes = kMeanJ * kD * 2;        // bf16 means of 16 key blocks
constexpr uint32_t kOffMean = kOffMB + kTileBytes;           // bf16 [2][16][128]: group g in buffer g & 1
constexpr uint32_t kOffRS = kOffMean + 2 * kMeanGroupBytes;  // fp32 [kRsSlots][128] row sums (block j in slot j % 32)
constexpr uint32_t kOffRSM = kOffRS + kRsSlots * kBlk * 4;   // fp32 [kRsSlots][128] the max each sum is taken against
constexpr uint32_t kOffSV = kOffRSM + kRsSlots * kBlk * 4;   // fp32 [128] g for every channel
constexpr uint32_t kOffMX = kOffSV + kBlk * 4;               // fp32 [2][128] reference max handed over, per parity
constexpr uint32_t kOffL = kOffMX + 2 * kBlk * 4;            // fp32 [128] l, [2][128] partial l, [2][128] their max
constexpr uint32_t kOffLg = kOffL + 5 * kBlk * 4;            // fp32 [128]: -log2(dec(E4M3 code)), -inf for code 0
constexpr uint32_t kOffBar = kOffLg + kBlk * 4;
constexpr int kNumBars = 1 + 2 * kKStages + 3 * kVStages + 2 * 4 + 2 + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;       // tmem address, abort flag
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;       // + alignment slack
static_assert(kOffQ % 1024 == 0 && kOffV % 1024 == 0 && kVStageBytes % 1024 == 0 && kOffOnes % 1024 == 0 && kOffMA % 1024 == 0 &&
                  kOffMB % 1024 == 0,
              "swizzled operand tiles need 1024-byte alignment");
static_assert(kCodeBytes % 16 == 0 && kSfBytes % 16 == 0 && kSfbBytes % 16 == 0, "copies need 16-byte alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kTmemSF1 < kTmemCols && kTmemSFB + 16 <= kTmemSF1 && kTmemSFA0 + 16 <= kTmemSFB, "TMEM plan");

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
    uint64_t *q_full, *k_full, *k_empty, *v_full, *v_ready, *v_empty, *s_full, *s_free, *p_full, *pv_done, *drain, *tail;
};

struct Params {
    const uint8_t *v_sf;
    const float *sq, *sk, *v_scale;
    const uint16_t *v_mean;
    uint16_t *O;
    int32_t *dev_status;
    int N;
    float scale_log2;
    uint64_t limit_ns;
};

// Largest raw score of each group of 16 of the kCols scores in X, into
// gm[kG0 .. kG0 + kCols / 16).
template <int kG0>
__device__ __forceinline__ void group_max(const uint32_t (&X)[kCols], float (&gm)[kBlk / 16]) {
#pragma unroll
    for (int g = 0; g < kCols / 16; ++g) {
        const uint32_t *s = X + 16 * g;
        const float a = max3(__uint_as_float(s[0]), __uint_as_float(s[1]), __uint_as_float(s[2]));
        const float b = max3(__uint_as_float(s[3]), __uint_as_float(s[4]), __uint_as_float(s[5]));
        const float c = max3(__uint_as_float(s[6]), __uint_as_float(s[7]), __uint_as_float(s[8]));
        const float d = max3(__uint_as_float(s[9]), __uint_as_float(s[10]), __uint_as_float(s[11]));
        const float e = max3(__uint_as_float(s[12]), __uint_as_float(s[13]), __uint_as_float(s[14]));
        gm[kG0 + g] = fmaxf(max3(a, b, c), max3(d, e, __uint_as_float(s[15])));
    }
}

// NVFP4 P of a row against the reference max m (negm = -m): per group of 16
// keys p = 2^(fma(S, c, -m)), scale sf = E4M3(amax16 / 6), code =
// E2M1(p / dec(sf)); P's codes go to W (key k at word k / 8, nibble k % 8),
// the scale bytes to a word per 64 keys (group g in byte g).
// With c > 0, S -> 2^(fma(S, c, -m)) does not decrease, so amax16 is 2 to the
// power of the group's largest score term (gm, from group_max or the reducing
// loads).  The quotient amax16 / 6 is corrected by one FMA step,
// q = RN(a r), q' = RN(q + RN(a - 6q) r) with r = RN(1/6): equal to the IEEE
// quotient for every a in [2^-120, 2^30] (checked exhaustively), and below
// that both round to the E4M3 code 0.  p / dec(sf) is evaluated as
// 2^(fma(S, c, lg(sf) - m)) with lg(sf) = -log2(dec(sf)) from a per-CTA table
// of the 127 codes (sLg; -inf for code 0, whose group codes are 0): one FMA and
// one exp per key, the same hardware-exp accuracy as p itself.
//
// Scales of the four groups kG .. kG + 3 (maxima gm[kG + i]): the scale word
// (group i in byte i) is returned, bias[kB + i] = lg(sf_i) - m; two groups per
// packed instruction and per E4M3 convert, each rounded as alone.
template <int kG, int kB>
__device__ __forceinline__ uint32_t nvfp4_scales4(const float (&gm)[kBlk / 16], float c, float negm, const float *sLg,
                                                  float (&bias)[kBlk / 16]) {
    constexpr float kSixth = 1.0f / 6.0f;
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = ex2_approx(__fmaf_rn(gm[kG + i], c, negm));
    const uint64_t r6 = pk2(__float_as_uint(kSixth), __float_as_uint(kSixth));
    const uint64_t m6 = pk2(__float_as_uint(-6.0f), __float_as_uint(-6.0f));
    float q[4];
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
        const uint64_t a2 = pk2(__float_as_uint(a[i]), __float_as_uint(a[i + 1]));
        const uint64_t q0 = mul2(a2, r6);
        upk2(fma2(fma2(q0, m6, a2), r6, q0), q[i], q[i + 1]);
    }
    const uint32_t sfa = e4m3x4(q[0], q[1], q[2], q[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) bias[kB + i] = __fadd_rn(sLg[(sfa >> (8 * i)) & 0xFFu], negm);
    return sfa;
}

// E2M1 codes of one group of 16 keys X[kOff .. kOff + 15] into W[kW], W[kW + 1]:
// E2M1(2^(fma(S, c, bias))) with bias = lg(sf) - m.
template <int kOff, int kW>
__device__ __forceinline__ void nvfp4_codes16(const uint32_t (&X)[kCols], float bias, uint64_t cx2,
                                              uint32_t (&W)[kBlk / 8]) {
    const uint64_t bx2 = pk2(__float_as_uint(bias), __float_as_uint(bias));
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        float x[8];
#pragma unroll
        for (int q = 0; q < 8; q += 2) {
            float t0, t1;
            upk2(fma2(pk2(X[kOff + 8 * w + q], X[kOff + 8 * w + q + 1]), cx2, bx2), t0, t1);
            x[q] = ex2_approx(t0);
            x[q + 1] = ex2_approx(t1);
        }
        W[kW + w] = e2m1x8(x);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    attention_nvfp4_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    Bars B;
    B.q_full = bars;
    B.k_full = bars + 1;
    B.k_empty = B.k_full + kKStages;
    B.v_full = B.k_empty + kKStages;
    B.v_ready = B.v_full + kVStages;
    B.v_empty = B.v_ready + kVStages;
    B.s_full = B.v_empty + kVStages;
    B.s_free = B.s_full + 2;
    B.p_full = B.s_free + 2;
    B.pv_done = B.p_full + 2;
    B.drain = B.pv_done + 2;   // [0]: QK thread, [1]: PV thread
    B.tail = B.drain + 2;      // the epilogue's mean-restore MMAs
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    int *abort_flag = reinterpret_cast<int *>(smem + kOffMisc + 4);
    float *sRS = reinterpret_cast<float *>(smem + kOffRS);
    float *sRSM = reinterpret_cast<float *>(smem + kOffRSM);
    float *sSV = reinterpret_cast<float *>(smem + kOffSV);
    float *sMX = reinterpret_cast<float *>(smem + kOffMX);
    float *sL = reinterpret_cast<float *>(smem + kOffL);
    float *sLp = sL + kBlk;        // [2][128] partial row sums, per parity
    float *sMp = sL + 3 * kBlk;    // [2][128] the reference max they are taken against
    float *sLg = reinterpret_cast<float *>(smem + kOffLg);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qtile = blockIdx.x, bh = blockIdx.y;
    const int N = p.N, nb = N / kBlk;

    if (threadIdx.x == 0) {
        mbar_init(B.q_full, 1);   // the Q tile's TMA load
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(B.k_full + s, 1);
            mbar_init(B.k_empty + s, 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(B.v_full + s, 1);
            mbar_init(B.v_ready + s, 1);
            mbar_init(B.v_empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(B.s_full + i, 1);
            mbar_init(B.s_free + i, kSoftmaxWarps / 2);
            mbar_init(B.p_full + i, kSoftmaxWarps / 2);
            mbar_init(B.pv_done + i, 1);
            mbar_init(B.drain + i, 1);
        }
        mbar_init(B.tail, 1);
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
        // lg of the E4M3 codes (127 = NaN is never produced)
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

    if (warp == 0) {
        // ------------------------------------------------------------ K producer
        // a stage is refilled as soon as the QK MMA that read it has finished
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            mbar_expect_tx(B.q_full, kTileBytes);
            tma_load_2d(smem + kOffQ, &tmQ, B.q_full, 0, bh * N + qtile * kBlk);
            int armed[kKStages];
            for (int s = 0; s < kKStages; ++s) armed[s] = 0;
            for (int b = 0; b < nb; ++b) {
                const int s = b % kKStages, use = b / kKStages;
                if (use > 0 && !mbar_wait(B.k_empty + s, (use - 1) & 1, abort_flag, p.limit_ns)) break;
                mbar_expect_tx(B.k_full + s, kTileBytes);
                tma_load_2d(smem + kOffK + s * kTileBytes, &tmK, B.k_full + s, 0, bh * N + b * kBlk);
                armed[s] = use + 1;
            }
            // every copy this thread issued has landed before the CTA can exit
            drain_wait(B.q_full, 0, p.limit_ns);
            for (int s = 0; s < kKStages; ++s)
                if (armed[s] > 0) drain_wait(B.k_full + s, (armed[s] - 1) & 1, p.limit_ns);
        }
    } else if (warp == kVWarp) {
        // ------------------------------------------------------------ V producer
        // Lane 0 loads block b (codes by TMA with the 64-byte swizzle, scales,
        // and with V(16 g) the bf16 means of group g into buffer g & 1) into
        // stage b % kVStages once PV(b - kVStages) has released it.  The warp
        // lays out block j's scales: row r of matrix h holds the scale words
        // (keys 64h ..) of channels r, r + 32, r + 64, r + 96, the order in
        // which the MMA reads B's scales from a lane quarter's columns.  The
        // means group g - 2 that a buffer held was staged at block 16 g - 13,
        // before PV(16 g - 4) completed, which the load of V(16 g) waited for.
        int armed[kVStages];
        for (int s = 0; s < kVStages; ++s) armed[s] = 0;
        auto issue = [&](int b) -> bool {
            const int s = b % kVStages, use = b / kVStages;
            if (use > 0 && !mbar_wait(B.v_empty + s, (use - 1) & 1, abort_flag, p.limit_ns)) return false;
            unsigned char *st = smem + kOffV + s * kVStageBytes;
            const int64_t blk = static_cast<int64_t>(bh) * nb + b;
            const bool with_means = (b % kMeanJ) == 0;
            const uint32_t mean_bytes =
                with_means ? static_cast<uint32_t>(nb - b < kMeanJ ? nb - b : kMeanJ) * kD * 2 : 0u;
            mbar_expect_tx(B.v_full + s, kCodeBytes + kSfBytes + mean_bytes);
            tma_load_2d(st, &tmV, B.v_full + s, 0, static_cast<int>(blk * kD));
            bulk_load(st + kCodeBytes, p.v_sf + blk * kSfBytes, kSfBytes, B.v_full + s);
            if (with_means)
                bulk_load(smem + kOffMean + ((b / kMeanJ) & 1) * kMeanGroupBytes, p.v_mean + blk * kD, mean_bytes,
                          B.v_full + s);
            armed[s] = use + 1;
            return true;
        };
        bool lok = true;   // lane 0: every load so far issued
        if (lane == 0) {
            tma_prefetch_desc(&tmV);
            for (int b = 0; lok && b < kVAhead && b < nb; ++b) lok = issue(b);
        }
        for (int j = 0; j < nb; ++j) {
            const int s = j % kVStages;
            const bool landed = (lane != 0 || lok) && mbar_wait(B.v_full + s, (j / kVStages) & 1, abort_flag, p.limit_ns);
            if (!__all_sync(0xffffffffu, landed)) break;
            unsigned char *st = smem + kOffV + s * kVStageBytes;
            const unsigned char *sf = st + kCodeBytes;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint4 w;
                w.x = *reinterpret_cast<const uint32_t *>(sf + (lane + 0) * (kBlk / 16) + 4 * h);
                w.y = *reinterpret_cast<const uint32_t *>(sf + (lane + 32) * (kBlk / 16) + 4 * h);
                w.z = *reinterpret_cast<const uint32_t *>(sf + (lane + 64) * (kBlk / 16) + 4 * h);
                w.w = *reinterpret_cast<const uint32_t *>(sf + (lane + 96) * (kBlk / 16) + 4 * h);
                *reinterpret_cast<uint4 *>(st + kCodeBytes + kSfBytes + h * kSfbBytes + 16 * lane) = w;
            }
            fence_proxy_async_smem();   // read by the scale copy into TMEM
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(B.v_ready + s);
                if (lok && j + kVAhead < nb) lok = issue(j + kVAhead);
            }
        }
        // every copy lane 0 issued has landed before the CTA can exit
        if (lane == 0)
            for (int s = 0; s < kVStages; ++s)
                if (armed[s] > 0) drain_wait(B.v_full + s, (armed[s] - 1) & 1, p.limit_ns);
    } else if (warp == kQKWarp) {
        // ------------------------------------------------------------ QK issuer
        // QK(b) into S[b & 1] once K(b) has landed and the softmax has read
        // S(b-2) out of that buffer; commits for the K stage and for s_full.
        if (lane == 0) {
            constexpr uint32_t idesc_qk = make_idesc(128, 128, 0, 0);
            const uint32_t sbase = smem_u32(smem);
            const uint64_t dq = sdesc_k_sw128(sbase + kOffQ);
            bool ok = mbar_wait(B.q_full, 0, abort_flag, p.limit_ns);
            for (int b = 0; ok && b < nb; ++b) {
                const int s = b % kKStages, sb = b & 1;
                if (b >= 2 && !mbar_wait_spin(B.s_free + sb, ((b - 2) >> 1) & 1, abort_flag, p.limit_ns)) break;
                if (!mbar_wait(B.k_full + s, (b / kKStages) & 1, abort_flag, p.limit_ns)) break;
                tc_fence_after();
                const uint64_t dk = sdesc_k_sw128(sbase + kOffK + s * kTileBytes);
#pragma unroll
                for (int kk = 0; kk < kD / 32; ++kk)
                    mma_f8f6f4(tmem + sb * 128, dq + 2 * kk, dk + 2 * kk, idesc_qk, kk > 0);
                tc_commit(B.k_empty + s);
                tc_commit(B.s_full + sb);
            }
            tc_commit(B.drain);
            drain_wait(B.drain, 0, p.limit_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ PV issuer
        // PV(j) once V(j) is laid out and P(j) is written: block j's V scales
        // into TMEM buffer j & 1 (last read by PV(j-2), which this thread
        // waits for), O += P V and the row sums E_{j&1} = P ones, two K = 64
        // halves each, the mean-restore MMA when due, then commits for the V
        // stage and for pv_done.
        if (lane == 0) {
            constexpr uint32_t idesc_pv = make_idesc_mxf4(128, 128);
            constexpr uint32_t idesc_rs = make_idesc_mxf4(128, kOnesRows);
            constexpr uint32_t idesc_bf16 = make_idesc(128, 128, 1, 1);
            const uint32_t sbase = smem_u32(smem);
            const uint64_t dma = sdesc_k_sw128(sbase + kOffMA);
            const uint64_t dmb = sdesc_k_sw128(sbase + kOffMB);
            const uint64_t d1 = sdesc_k_sw128(sbase + kOffOnes);
            const uint32_t tO = tmem + kTmemO;
            for (int j = 0; j < nb; ++j) {
                const int s = j % kVStages, pb = j & 1;
                if (!mbar_wait(B.v_ready + s, (j / kVStages) & 1, abort_flag, p.limit_ns)) break;
                // V-scale buffer j & 1 was last read by PV(j-2): in the steady state long done
                if (j >= 2 && !mbar_wait_spin(B.pv_done + pb, ((j - 2) >> 1) & 1, abort_flag, p.limit_ns)) break;
                tc_fence_after();
                const uint32_t vst = sbase + kOffV + s * kVStageBytes;
                const uint32_t tsfb = tmem + kTmemSFB + 8 * pb;
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    tc_cp_rows_x4(tsfb + 4 * h, sdesc_rows16(vst + kCodeBytes + kSfBytes + h * kSfbBytes));
                if (!mbar_wait_spin(B.p_full + pb, (j >> 1) & 1, abort_flag, p.limit_ns)) break;
                tc_fence_after();
                const uint64_t dv = sdesc_k_sw64(vst);
                const uint32_t tp = tmem + kTmemP0 + 16 * pb;
                const uint32_t tsfa = tmem + kTmemSFA0 + 8 * pb;
                const uint32_t te = tmem + kTmemE0 + 16 * pb;
                // keys 64h .. 64h + 63: A columns 8h.., B bytes 32h.. of every row, scales at +4h
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    mma_mxf4_ts(tO, tp + 8 * h, dv + 2 * h, idesc_pv, tsfa + 4 * h, tsfb + 4 * h, (j > 0 || h > 0) ? 1u : 0u);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    mma_mxf4_ts(te, tp + 8 * h, d1 + 2 * h, idesc_rs, tsfa + 4 * h, tmem + kTmemSF1, h > 0 ? 1u : 0u);
                if (flush_after(j)) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma_f16(tO, dma + 2 * kk, dmb + 2 * kk, idesc_bf16, 1u);
                }
                tc_commit(B.v_empty + s);
                tc_commit(B.pv_done + pb);
            }
            tc_commit(B.drain + 1);
            drain_wait(B.drain + 1, 0, p.limit_ns);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3;                              // TMEM lane quarter
        const int par = (warp - 2) >> 2;                           // this warp's key blocks: par, par + 2, ...
        const int row = quarter * 32 + lane;                       // query row in the tile == TMEM lane
        const uint32_t bar_out = kBarHand0 + 2 * quarter + par;    // hands the reference max on
        const uint32_t bar_in = kBarHand0 + 2 * quarter + (par ^ 1);
        const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const float sqv = p.sq[static_cast<int64_t>(bh) * nb + qtile];
        const float *skh = p.sk + static_cast<int64_t>(bh) * nb;
        unsigned char *sMA = smem + kOffMA;
        unsigned char *sMB = smem + kOffMB;
        const float kNegInf = __int_as_float(0xff800000);
        float m = kNegInf;   // reference max after this thread's latest block
        float l = 0.0f;      // row sum of this thread's blocks, taken against m
        bool ok = true;
        if (par == 0) {
            // the row-sum MMA's B scales (E4M3 1.0), read in every lane quarter;
            // stored before this warp's first P, which PV(0) waits for
            asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tl + kTmemSF1), "r"(0x38383838u)
                         : "memory");
            tmem_st_wait();
        }
        float sk_next = par < nb ? skh[par] : 0.0f;
        for (int b = par; b < nb; b += 2) {
            const int sb = b & 1;
            const float sk_b = sk_next;
            const float c = __fmul_rn(__fmul_rn(sqv, sk_b), p.scale_log2);
            const uint32_t tS = tl + sb * 128;
            // the group maxima of S(b); X keeps keys 64..127
            uint32_t X[kCols];
            float gm[kBlk / 16];
            float pm = kNegInf;
            const bool wok = ok && __all_sync(0xffffffffu, mbar_wait(B.s_full + sb, (b >> 1) & 1, abort_flag, p.limit_ns));
            if (wok) {
                tc_fence_after();
                VCA_TMEM_LD32(tS, X);
                VCA_TMEM_LD32(tS + 32, (X + 32));
                tmem_ld_wait();
                group_max<0>(X, gm);
                // keys 64..127 by reducing loads, which return each 16 keys' max
                // with the data (for keys 0..63 as well they cost more in spills)
                VCA_TMEM_LDMAX16(tS + 64, X, gm[4]);
                VCA_TMEM_LDMAX16(tS + 80, (X + 16), gm[5]);
                VCA_TMEM_LDMAX16(tS + 96, (X + 32), gm[6]);
                VCA_TMEM_LDMAX16(tS + 112, (X + 48), gm[7]);
                tmem_ld_wait();
                pm = max3(max3(gm[0], gm[1], gm[2]), max3(gm[3], gm[4], gm[5]), fmaxf(gm[6], gm[7]));
            }
            // reference max after block b-1 (from the partner), after block b
            // (handed on); NaN marks a partner that gave up
            float m_in = kNegInf;
            if (b >= 1) {
                bar_sync(bar_in, 64);
                m_in = sMX[(sb ^ 1) * kBlk + row];
            }
            const bool valid = wok && !(m_in != m_in);
            const float bm = __fmul_rn(pm, c);
            const bool moved = valid && bm > __fadd_rn(m_in, kLazyTau);
            const float m_new = moved ? bm : m_in;
            if (b + 1 < nb) {
                sMX[sb * kBlk + row] = valid ? m_new : __int_as_float(0x7fc00000);
                bar_arrive_release(bar_out, 64);
            }
            // the next block's key scale, loaded after the hand-over so that the
            // fence before it never waits for this load
            if (b + 2 < nb) sk_next = skh[b + 2];
            if (!__all_sync(0xffffffffu, valid)) {
                ok = false;
                break;
            }
            // NVFP4 P of all 128 keys: keys 64..127 from X while keys 0..63 are
            // reloaded behind them; sfa0 / sfa1 the scale bytes of keys 0..63 / 64..127
            const float negm = -m_new;
            const uint64_t cx2 = pk2(__float_as_uint(c), __float_as_uint(c));
            uint32_t W[kBlk / 8];
            float bias[kBlk / 16];
            const uint32_t sfa1 = nvfp4_scales4<4, 4>(gm, c, negm, sLg, bias);
            nvfp4_codes16<0, 8>(X, bias[4], cx2, W);
            nvfp4_codes16<16, 10>(X, bias[5], cx2, W);
            VCA_TMEM_LD32(tS, X);
            nvfp4_codes16<32, 12>(X, bias[6], cx2, W);
            nvfp4_codes16<48, 14>(X, bias[7], cx2, W);
            VCA_TMEM_LD32(tS + 32, (X + 32));
            tmem_ld_wait();
            // S(b) is read: QK(b+2) may overwrite the buffer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.s_free + sb);
            const uint32_t sfa0 = nvfp4_scales4<0, 0>(gm, c, negm, sLg, bias);
            nvfp4_codes16<0, 0>(X, bias[0], cx2, W);
            nvfp4_codes16<16, 2>(X, bias[1], cx2, W);
            nvfp4_codes16<32, 4>(X, bias[2], cx2, W);
            nvfp4_codes16<48, 6>(X, bias[3], cx2, W);
            // P buffer b&1 and row-sum slot b&1 are free once PV(b-2) completed
            if (b >= 2) ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done + sb, ((b - 2) >> 1) & 1, abort_flag, p.limit_ns));
            if (ok) {
                tc_fence_after();
                // block b-2's row sum from the slot of this parity, then P(b):
                // the codes, and the row's scales in lane `row`, column
                // sfa + 4h + quarter (PV(b)'s row-sum MMA rewrites the slot)
                const uint32_t te = tl + kTmemE0 + 16 * sb;
                uint32_t rs_raw = 0;
                if (b >= 2) {
                    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(rs_raw) : "r"(te));
                    tmem_ld_wait();
                }
                VCA_TMEM_ST16(tl + kTmemP0 + 16 * sb, W);
                const uint32_t tsfa = tl + kTmemSFA0 + 8 * sb + quarter;
                asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tsfa), "r"(sfa0) : "memory");
                asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tsfa + 4), "r"(sfa1) : "memory");
                if (b >= 2) {
                    // block b-2's sum, taken against m (this thread's max after b-2)
                    const float rs = __uint_as_float(rs_raw);
                    const int slot = ((b - 2) & (kRsSlots - 1)) * kBlk + row;
                    sRS[slot] = rs;
                    sRSM[slot] = m;
                    l = __fadd_rn(l, rs);
                    if (m != m_new) l = __fmul_rn(l, ex2_approx(__fsub_rn(m, m_new)));
                }
                // the reference max moved at block b: O (after PV(b-1)) from m_in to m_new
                const float alpha = (moved && b > 0) ? ex2_approx(__fsub_rn(m_in, m_new)) : 1.0f;
                if (__any_sync(0xffffffffu, alpha != 1.0f)) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(B.pv_done + (sb ^ 1), ((b - 1) >> 1) & 1, abort_flag, p.limit_ns));
                    if (ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int i = 0; i < kD / 32; ++i) {
                            uint32_t o[32];
                            VCA_TMEM_LD32(tl + kTmemO + 32 * i, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__fmul_rn(__uint_as_float(o[e]), alpha));
                            VCA_TMEM_ST32(tl + kTmemO + 32 * i, o);
                        }
                    }
                }
                if (ok && flush_after(b)) {
                    // mean-restore operands of blocks b-19 .. b-4 (the MMA follows PV(b))
                    // the group's means landed with V(b0), before PV(b0) could run
                    const int b0 = b - kMeanJ - kMeanLag;
                    stage_means(row, sRS, sRSM, m_new, b0,
                                reinterpret_cast<const uint16_t *>(smem + kOffMean) + ((b0 / kMeanJ) & 1) * (kMeanJ * kD),
                                sSV, sMA, sMB);
                    fence_proxy_async_smem();   // read by the tensor core
                }
                if (ok) {
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B.p_full + sb);
                }
            }
            m = m_new;
        }
        // ------------------------------------------------------------ epilogue
        // this thread's last block lb: once PV(lb) has completed, its row sum
        // is in the slot of this parity.  The wait is on this parity's barrier,
        // whose previous phase (PV(lb-2)) this thread has seen complete.
        const int lb = (((nb - 1) & 1) == par) ? nb - 1 : nb - 2;
        if (ok && lb >= 0)
            ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done + par, (lb >> 1) & 1, abort_flag, p.limit_ns));
        if (ok && lb >= 0) {
            tc_fence_after();
            uint32_t r = 0;
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(tl + kTmemE0 + 16 * par));
            tmem_ld_wait();
            const float rs = __uint_as_float(r);
            const int slot = (lb & (kRsSlots - 1)) * kBlk + row;
            sRS[slot] = rs;
            sRSM[slot] = m;
            l = __fadd_rn(l, rs);
        }
        sLp[par * kBlk + row] = l;
        sMp[par * kBlk + row] = lb >= 0 ? m : kNegInf;
        // every softmax warp arrives here, whether it finished or gave up; the
        // epilogue (and its barriers) runs only if all of them finished.
        // PV(nb-1), and with it every MMA, has completed once the threads of
        // its parity have passed their wait above
        ok = bar_and(ok, kBarSoftmax, 32 * kSoftmaxWarps);
        if (ok) {
            tc_fence_after();
            // the blocks after the last mean MMA's range
            const int bf = nb - 1 >= kMeanJ + kMeanLag ? kMeanLag + kMeanJ * ((nb - 1 - kMeanLag) / kMeanJ) : -1;
            const int tail0 = bf >= 0 ? bf - kMeanLag : 0;
            const float mf = sMp[((nb - 1) & 1) * kBlk + row];   // the final reference max
            if (par == 0) {
                float lt = 0.0f;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float mq = sMp[q * kBlk + row];
                    if (mq != kNegInf)
                        lt = __fadd_rn(lt, mq == mf ? sLp[q * kBlk + row]
                                                    : __fmul_rn(sLp[q * kBlk + row], ex2_approx(__fsub_rn(mq, mf))));
                }
                sL[row] = lt;
            }
            // the tail's mean terms by the tensor core: staged into the mean
            // tiles (whose last reader, the final in-loop mean MMA, has
            // finished) and the K ring's first two tiles (every QK has
            // completed); sL is written before the staging barrier
            ok = restore_tail_means(par, row, warp == 2 && lane == 0, sRS, sRSM, mf, tail0, nb - tail0,
                                    reinterpret_cast<const uint16_t *>(smem + kOffMean), sSV, sMA, smem + kOffK,
                                    tl + kTmemO, B.tail, abort_flag, p.limit_ns);
        }
        if (ok) {
            const float inv_l = 1.0f / sL[row];
            const int col0 = kCols * par;
            uint16_t *orow = p.O + (static_cast<int64_t>(bh) * N + static_cast<int64_t>(qtile) * kBlk + row) * kD + col0;
            store_output(tl + kTmemO + col0, sSV, col0, inv_l, orow);
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
    CUtensorMap mq, mk, mv;
    const uint64_t rows = static_cast<uint64_t>(a.BH) * a.N;
    // Q, K: [BH N][128] FP8 rows; V codes: [BH nb 128][64] bytes, one channel row per 128 keys
    if (!make_tile_map(&mq, a.q8, rows) || !make_tile_map(&mk, a.k8, rows) || !make_tile_map_sw64(&mv, a.v_res, rows))
        return cudaErrorInvalidValue;
    Params p;
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
    attention_nvfp4_kernel<<<dim3(a.N / kBlk, a.BH), kThreads, kSmemBytes, st>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

}  // namespace vca
