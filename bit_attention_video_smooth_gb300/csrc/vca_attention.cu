// vca_attention.cu -- non-causal FP8 attention with the V-Smooth mean restore
// and ExpCast-FP8 ("VC-Attention", paper page, section "method"): QK and PV on
// FP8 tensor cores, online softmax whose per-block row sums bring the block
// means back as one outer product rowsum_b (x) mean_b, and ExpCast writing the
// E4M3 probability bytes with one FMA (news page, "ExpCast-FP8").
//
// One CTA owns a 128-row query tile of one (batch, head) and streams the key
// blocks of that head in increasing (permuted) order.  Warp roles:
//   warp 0     TMA producer: K tiles into a 3-stage ring
//   warp 10    TMA producer: V-residual tiles into a 3-stage ring
//   warp 11    QK issuer (one thread): S[b&1] = Q8 K8_b^T (kind::f8f6f4,
//              N = 128) once K(b) has landed and S(b-2) has been read
//   warp 1     TMEM owner and PV issuer (one thread):
//                [E | O] += P_b [ones ; V8_b]       (kind::f8f6f4, N = 144): the
//                         16 extra output columns are the block's row sums of the
//                         decoded P, so the softmax threads never add them up
//              and every 16 key blocks O += [rowsum hi|lo] [mean/s_v hi|lo]^T (bf16).
//   warps 2-9  softmax, one thread per query row and key block: the warps w and
//              w+4 share a TMEM lane quarter (and a sub-partition) and take the
//              even and the odd key blocks, whole rows of 128 scores each, so
//              one of them computes while the other waits for its next block.
//              The reference max is sequential over blocks: after its row max
//              of block b, a thread takes the reference max after block b-1
//              from its partner (shared memory + a named barrier), decides the
//              max after block b (lazy threshold: it moves only when the block
//              max exceeds it by 8) and hands it on before computing the codes,
//              so every code is taken against its block's final reference max.
//              O is rescaled in TMEM when the max moves; the row sum of block
//              b-2 is read from its TMEM slot and kept, with the reference max
//              it was taken against, for the mean restore; epilogue
//              O = (O s_v + the last, partial group of mean terms) / l.
// Barriers between the softmax and the MMA threads, per parity of b:
//   s_full  QK(b) committed: S(b) is in S[b&1]
//   s_free  the four warps of the parity have read S(b): QK(b+2) may start
//   p_full  the four warps have written P(b) (and cleared the row-sum slot)
//   pv_done PV(b) (and the mean MMA after it) committed: P buffer b&1 and the
//           row-sum slot b&1 are free, and the slot holds block b's sums.
// A parity wait is only exact when the waiter is at most one phase behind the
// barrier and has seen the phase before the one it waits for complete: each
// thread waits on a barrier phase by phase (or, for the other parity's
// pv_done, only after PV(b-2) and so PV(b-3) completed).  The MMA threads wait
// with non-suspending polls (they are on the critical path).
// TMEM columns: S0 [0,128), S1 [128,256), E0 [256,272), O [272,400), E1 [400,416),
// P0 [416,448), P1 [448,480), Q [480,512).  Q and P, the A operands of the two
// contractions, live in TMEM (four FP8 codes per column), so the tensor core
// reads only K and V from shared memory.
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

constexpr int kKStages = 3;               // K tiles in flight (released after their QK MMA)
constexpr int kVStages = 3;               // V tiles in flight (released after their PV MMA)
constexpr int kVWarp = 2 + kSoftmaxWarps;  // the V producer
constexpr int kQKWarp = kVWarp + 1;        // the QK issuer (the PV issuer is warp 1)
constexpr int kThreads = 32 * (kQKWarp + 1);
constexpr uint32_t kTileBytes = kBlk * kD; // one 128 x 128 FP8 tile (16 KB)
constexpr uint32_t kTmemCols = 512;
// TMEM: S0 [0,128), S1 [128,256), row-sum slot E0 [256,272), O [272,400), E1 [400,416).
// PV of an even block writes [E0 | O] (B = [ones ; V]), of an odd block [O | E1]
// (B = [V ; ones]): the 16 extra output columns are the block's row sums.
constexpr uint32_t kTmemE0 = 256, kTmemO = 272, kTmemE1 = 400, kTmemP0 = 416, kTmemQ = 480;

// shared-memory layout (bytes from a 1024-aligned base)
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOnesBytes = 16 * 128;            // 16 rows of E4M3 1.0
constexpr uint32_t kVStageBytes = kOnesBytes + kTileBytes + kOnesBytes;   // [ones | V | ones]
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffMA = kOffV + kVStages * kVStageBytes;
constexpr uint32_t kOffMB = kOffMA + kTileBytes;
constexpr uint32_t kMeanGroupBytes = kMeanJ * kD * 2;        // bf16 means of 16 key blocks
constexpr uint32_t kOffMean = kOffMB + kTileBytes;           // bf16 [2][16][128]: group g in buffer g & 1
constexpr uint32_t kOffRS = kOffMean + 2 * kMeanGroupBytes;  // fp32 [kRsSlots][128] row sums (block j in slot j % 32)
constexpr uint32_t kOffRSM = kOffRS + kRsSlots * kBlk * 4;   // fp32 [kRsSlots][128] the max each sum is taken against
constexpr uint32_t kOffSV = kOffRSM + kRsSlots * kBlk * 4;   // fp32 [128] residual scales
constexpr uint32_t kOffMX = kOffSV + kBlk * 4;               // fp32 [2][128] reference max handed over, per parity
constexpr uint32_t kOffL = kOffMX + 2 * kBlk * 4;            // fp32 [128] l, [2][128] partial l, [2][128] their max
constexpr uint32_t kOffBar = kOffL + 5 * kBlk * 4;
constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 2 * 4 + 2 + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;       // tmem address, abort flag
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;       // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Bars {
    uint64_t *q_full, *k_full, *k_empty, *v_full, *v_empty, *s_full, *s_free, *p_full, *pv_done, *drain, *tail;
};

struct Params {
    const uint8_t *q8;
    const float *sq, *sk, *v_scale;
    const uint16_t *v_mean;
    uint16_t *O;
    int32_t *dev_status;
    int N;
    float scale_log2;
    uint64_t limit_ns;
    uint32_t one;   // 1: an opaque multiplier for integer adds on the FMA pipe
};


// exp2 then E4M3 for four raw scores: p = 2^(fma(S, c, -m)).
__device__ __forceinline__ uint32_t expconv4(uint64_t s01, uint64_t s23, uint64_t cx2, uint64_t negmx2) {
    float a[4];
    upk2(fma2(s01, cx2, negmx2), a[0], a[1]);
    upk2(fma2(s23, cx2, negmx2), a[2], a[3]);
    return e4m3x4(ex2_approx(a[0]), ex2_approx(a[1]), ex2_approx(a[2]), ex2_approx(a[3]));
}

// P codes of 32 keys (X[kOff .. kOff+31]) against the reference max m of the
// block, four codes per word, into W[kW .. kW+7] (the word order of the P
// buffer's TMEM columns).  `fast` (warp-uniform) says |m| < 2^22, so that the
// ExpCast codes need no clip: m is the block's final reference max, so every
// score satisfies s c <= m + 8.
// The clipped ExpCast codes of 32 scores (taken only when |m| >= 2^22, i.e.
// never for finite attention inputs of any realistic scale): out of line, so
// the hot loop holds one copy of the code arithmetic per call site.
__device__ __noinline__ void expcast32_clip(const uint32_t *sv, float c8s, float bs, uint32_t one, uint32_t *w) {
    for (int q = 0; q < 8; ++q) {
        const uint32_t s4[4] = {sv[4 * q], sv[4 * q + 1], sv[4 * q + 2], sv[4 * q + 3]};
        w[q] = expcast4<true>(s4, c8s, bs, one);
    }
}

template <bool kExpcast, int kOff, int kW>
__device__ __forceinline__ void codes32(const uint32_t (&X)[kCols], float c, float m, bool fast, uint32_t one,
                                        uint32_t (&W)[32]) {
    if constexpr (kExpcast) {
        // t = fma(S, 8c, 55.65 - 8m); the clipped form takes t / 256 (both
        // scalings exact)
        const float c8 = __fmul_rn(8.0f, c);
        const float b = __fsub_rn(kExpcastOffset, __fmul_rn(8.0f, m));
        if (fast) {
            const uint64_t c8x2 = pk2(__float_as_uint(c8), __float_as_uint(c8));
            const uint64_t bx2 = pk2(__float_as_uint(b), __float_as_uint(b));
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t sv[4] = {X[kOff + 4 * q], X[kOff + 4 * q + 1], X[kOff + 4 * q + 2], X[kOff + 4 * q + 3]};
                W[kW + q] = expcast4_fast(sv, c8x2, bx2, one);
            }
        } else {
            const float c8s = __fmul_rn(c8, 1.0f / 256.0f);
            const float bs = __fmul_rn(b, 1.0f / 256.0f);
            // copies, so that X and W themselves never need an address
            uint32_t sv[32], w[8];
#pragma unroll
            for (int e = 0; e < 32; ++e) sv[e] = X[kOff + e];
            expcast32_clip(sv, c8s, bs, one, w);
#pragma unroll
            for (int q = 0; q < 8; ++q) W[kW + q] = w[q];
        }
    } else {
        const float negm = -m;
        const uint64_t cx2 = pk2(__float_as_uint(c), __float_as_uint(c));
        const uint64_t nx2 = pk2(__float_as_uint(negm), __float_as_uint(negm));
#pragma unroll
        for (int q = 0; q < 8; ++q)
            W[kW + q] = expconv4(pk2(X[kOff + 4 * q], X[kOff + 4 * q + 1]), pk2(X[kOff + 4 * q + 2], X[kOff + 4 * q + 3]),
                                 cx2, nx2);
    }
}


template <bool kExpcast>
__global__ void __launch_bounds__(kThreads, 1)
    attention_e4m3_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    Bars B;
    B.q_full = bars;
    B.k_full = bars + 1;
    B.k_empty = B.k_full + kKStages;
    B.v_full = B.k_empty + kKStages;
    B.v_empty = B.v_full + kVStages;
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

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qtile = blockIdx.x, bh = blockIdx.y;
    const int N = p.N, nb = N / kBlk;

    if (threadIdx.x == 0) {
        mbar_init(B.q_full, 4);   // the four warps that store Q into TMEM
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(B.k_full + s, 1);
            mbar_init(B.k_empty + s, 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(B.v_full + s, 1);
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
    // the Q tile: warps 2-5 (the even-block softmax warps, one query row per
    // thread) load their rows now and store them into TMEM once it is allocated
    uint32_t qv[32];
    if (warp >= 2 && warp < 6) {
        const int t = threadIdx.x - 64;
        load_q_regs(p.q8 + (static_cast<int64_t>(bh) * N + static_cast<int64_t>(qtile) * kBlk + (warp & 3) * 32 + lane) * kD,
                    qv);
        sSV[t] = p.v_scale[static_cast<int64_t>(bh) * kD + t];
        // the ones rows around every V stage: 16 x 128 bytes of E4M3 1.0 (0x38)
        const uint4 ones = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
        for (int st = 0; st < kVStages; ++st) {
            unsigned char *vs = smem + kOffV + st * kVStageBytes;
            *reinterpret_cast<uint4 *>(vs + 16 * t) = ones;
            *reinterpret_cast<uint4 *>(vs + kOnesBytes + kTileBytes + 16 * t) = ones;
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 || warp == kVWarp) {
        // ------------------------------------------------------------ producers
        // warp 0: the K ring; warp kVWarp: the V ring.  A stage is refilled
        // as soon as the MMA that read it has finished (the issuing thread's
        // commit onto k_empty / v_empty).
        if (lane == 0) {
            const bool is_k = (warp == 0);
            const int stages = is_k ? kKStages : kVStages;
            uint64_t *full = is_k ? B.k_full : B.v_full;
            uint64_t *empty = is_k ? B.k_empty : B.v_empty;
            unsigned char *ring = smem + (is_k ? kOffK : kOffV + kOnesBytes);
            const uint32_t stride = is_k ? kTileBytes : kVStageBytes;
            const void *tm = is_k ? static_cast<const void *>(&tmK) : static_cast<const void *>(&tmV);
            tma_prefetch_desc(tm);
            int armed[kKStages > kVStages ? kKStages : kVStages];
            for (int s = 0; s < stages; ++s) armed[s] = 0;
            for (int b = 0; b < nb; ++b) {
                const int s = b % stages, use = b / stages;
                if (use > 0 && !mbar_wait(empty + s, (use - 1) & 1, abort_flag, p.limit_ns)) break;
                // with V(16 g) the bf16 means of group g (blocks 16 g .. 16 g + 15), on
                // the same barrier, into buffer g & 1: PV(16 g) complete implies they
                // have landed.  The group that buffer held (g - 2) was staged at block
                // 16 g - 13, before PV(16 g - 3) completed, which this refill waited for.
                const bool with_means = !is_k && (b % kMeanJ) == 0;
                const uint32_t mean_bytes =
                    with_means ? static_cast<uint32_t>(nb - b < kMeanJ ? nb - b : kMeanJ) * kD * 2 : 0u;
                mbar_expect_tx(full + s, kTileBytes + mean_bytes);
                tma_load_2d(ring + s * stride, tm, full + s, 0, is_k ? bh * N + b * kBlk : (bh * nb + b) * kBlk);
                if (with_means)
                    bulk_load(smem + kOffMean + ((b / kMeanJ) & 1) * kMeanGroupBytes,
                              p.v_mean + (static_cast<int64_t>(bh) * nb + b) * kD, mean_bytes, full + s);
                armed[s] = use + 1;
            }
            // every copy this thread issued has landed before the CTA can exit
            for (int s = 0; s < stages; ++s)
                if (armed[s] > 0) drain_wait(full + s, (armed[s] - 1) & 1, p.limit_ns);
        }
    } else if (warp == kQKWarp) {
        // ------------------------------------------------------------ QK issuer
        // QK(b) into S[b & 1] once K(b) has landed and the softmax has read
        // S(b-2) out of that buffer; commits for the K stage and for s_full.
        if (lane == 0) {
            constexpr uint32_t idesc_qk = make_idesc(128, 128, 0, 0);
            const uint32_t sbase = smem_u32(smem);
            bool ok = mbar_wait(B.q_full, 0, abort_flag, p.limit_ns);
            for (int b = 0; ok && b < nb; ++b) {
                const int s = b % kKStages, sb = b & 1;
                if (b >= 2 && !mbar_wait_spin(B.s_free + sb, ((b - 2) >> 1) & 1, abort_flag, p.limit_ns)) break;
                if (!mbar_wait(B.k_full + s, (b / kKStages) & 1, abort_flag, p.limit_ns)) break;
                tc_fence_after();
                const uint64_t dk = sdesc_k_sw128(sbase + kOffK + s * kTileBytes);
#pragma unroll
                for (int kk = 0; kk < kD / 32; ++kk)
                    mma_f8f6f4_ts(tmem + sb * 128, tmem + kTmemQ + 8 * kk, dk + 2 * kk, idesc_qk, kk > 0);
                tc_commit(B.k_empty + s);
                tc_commit(B.s_full + sb);
            }
            tc_commit(B.drain);
            drain_wait(B.drain, 0, p.limit_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ PV issuer
        // PV(j) once P(j) is written and V(j) has landed: [E | O] += P [ones ; V]
        // (the 16 extra columns receive the row sums), the mean-restore MMA when
        // due, then commits for the V stage and for pv_done.
        if (lane == 0) {
            constexpr uint32_t idesc_pv = make_idesc(128, 144, 0, 0);
            constexpr uint32_t idesc_bf16 = make_idesc(128, 128, 1, 1);
            const uint32_t sbase = smem_u32(smem);
            const uint64_t dma = sdesc_k_sw128(sbase + kOffMA);
            const uint64_t dmb = sdesc_k_sw128(sbase + kOffMB);
            const uint32_t tO = tmem + kTmemO;
            for (int j = 0; j < nb; ++j) {
                const int s = j % kVStages, pb = j & 1;
                if (!mbar_wait(B.v_full + s, (j / kVStages) & 1, abort_flag, p.limit_ns)) break;
                if (!mbar_wait_spin(B.p_full + pb, (j >> 1) & 1, abort_flag, p.limit_ns)) break;
                tc_fence_after();
                const uint32_t vstage = sbase + kOffV + s * kVStageBytes;
                const uint64_t dv = sdesc_k_sw128(pb == 0 ? vstage : vstage + kOnesBytes);
                const uint32_t td = tmem + (pb == 0 ? kTmemE0 : kTmemO);
                const uint32_t tp = tmem + kTmemP0 + 32 * pb;
#pragma unroll
                for (int kk = 0; kk < kBlk / 32; ++kk)
                    mma_f8f6f4_ts(td, tp + 8 * kk, dv + 2 * kk, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
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
            // Q tile into TMEM (the A operand of QK): this row's 128 codes, 32 columns
            VCA_TMEM_ST32(tl + kTmemQ, qv);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.q_full);
        }
        float sk_next = par < nb ? skh[par] : 0.0f;
        for (int b = par; b < nb; b += 2) {
            const int sb = b & 1;
            const float sk_b = sk_next;
            const float c = __fmul_rn(__fmul_rn(sqv, sk_b), p.scale_log2);
            const uint32_t tS = tl + sb * 128;
            // the row max of S(b); X keeps columns 64..127
            uint32_t X[kCols];
            float pm = kNegInf;
            const bool wok = ok && __all_sync(0xffffffffu, mbar_wait(B.s_full + sb, (b >> 1) & 1, abort_flag, p.limit_ns));
            if (wok) {
                tc_fence_after();
                if constexpr (kExpcast) {
                    // the reducing loads return each 32 columns' max with the
                    // data (the exp-path build takes them for columns 64..127
                    // only: for both halves they cost it more in spills than
                    // the max instructions they save)
                    float r0, r1, r2, r3;
                    VCA_TMEM_LDMAX32(tS, X, r0);
                    VCA_TMEM_LDMAX32(tS + 32, (X + 32), r1);
                    tmem_ld_wait();
                    VCA_TMEM_LDMAX32(tS + 64, X, r2);
                    VCA_TMEM_LDMAX32(tS + 96, (X + 32), r3);
                    tmem_ld_wait();
                    pm = fmaxf(fmaxf(r0, r1), fmaxf(r2, r3));
                } else {
                    VCA_TMEM_LD32(tS, X);
                    VCA_TMEM_LD32(tS + 32, (X + 32));
                    tmem_ld_wait();
                    pm = row_part_max(X);
                    float r2, r3;
                    VCA_TMEM_LDMAX32(tS + 64, X, r2);
                    VCA_TMEM_LDMAX32(tS + 96, (X + 32), r3);
                    tmem_ld_wait();
                    pm = fmaxf(pm, fmaxf(r2, r3));
                }
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
            // all 128 codes into registers: columns 64..127 from X while
            // columns 0..63 are reloaded behind them.  The ExpCast build takes
            // the give-up test from the fast-path vote (one vote per block).
            bool fast;
            if constexpr (kExpcast) {
                fast = __all_sync(0xffffffffu, valid && fabsf(m_new) < kExpcastFastMax);
                if (!fast && !__all_sync(0xffffffffu, valid)) {
                    ok = false;
                    break;
                }
            } else {
                fast = true;
                if (!__all_sync(0xffffffffu, valid)) {
                    ok = false;
                    break;
                }
            }
            const uint32_t tp = tl + kTmemP0 + 32 * sb;
            uint32_t W[32];
            codes32<kExpcast, 0, 16>(X, c, m_new, fast, p.one, W);
            VCA_TMEM_LD32(tS, X);
            codes32<kExpcast, 32, 24>(X, c, m_new, fast, p.one, W);
            VCA_TMEM_LD32(tS + 32, (X + 32));
            tmem_ld_wait();
            // S(b) is read: QK(b+2) may overwrite the buffer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.s_free + sb);
            codes32<kExpcast, 0, 0>(X, c, m_new, fast, p.one, W);
            codes32<kExpcast, 32, 8>(X, c, m_new, fast, p.one, W);
            // P buffer b&1 and row-sum slot b&1 are free once PV(b-2) completed
            if (b >= 2) ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done + sb, ((b - 2) >> 1) & 1, abort_flag, p.limit_ns));
            if (ok) {
                tc_fence_after();
                // block b-2's row sum from the slot of this parity, then P(b) and
                // the cleared slot for PV(b) (PV(0) initialises E0)
                const uint32_t te = tl + (sb == 0 ? kTmemE0 : kTmemE1);
                // the exp-path build stores P before reading the slot, the
                // ExpCast build after (each order measured faster for its build)
                if constexpr (!kExpcast) VCA_TMEM_ST32(tp, W);
                uint32_t rs_raw = 0;
                if (b >= 2) {
                    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(rs_raw) : "r"(te));
                    tmem_ld_wait();
                }
                if constexpr (kExpcast) VCA_TMEM_ST32(tp, W);
                if (b >= 1)
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};"
                        ::"r"(te), "r"(0u) : "memory");
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
        // whose previous phase (PV(lb-2)) this thread has seen complete: a
        // parity wait for a phase two ahead of the barrier would return at once.
        const int lb = (((nb - 1) & 1) == par) ? nb - 1 : nb - 2;
        if (ok && lb >= 0)
            ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done + par, (lb >> 1) & 1, abort_flag, p.limit_ns));
        if (ok && lb >= 0) {
            tc_fence_after();
            uint32_t r = 0;
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                         : "=r"(r)
                         : "r"(tl + (par == 0 ? kTmemE0 : kTmemE1)));
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
        // epilogue (and its barriers) runs only if all of them finished
        // PV(nb-1), and with it every MMA, has completed once the threads of its
        // parity have passed their wait above
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

// ExpCast map alone, for bit-exact tests of the device function.
// Four elements per thread through the same packed path the attention kernel
// uses.  The unclipped variant is taken where the attention kernel would take
// it: |m| < 2^22 and fp32(s_raw * c) <= fp32(m + 8) (m is the lazily updated
// reference max there).
__global__ void expcast_codes_kernel(const float *__restrict__ s_raw, const float *__restrict__ c,
                                     const float *__restrict__ m, int64_t n, uint8_t *__restrict__ out) {
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; 4 * g < n;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // the kernel's arithmetic, one scale per element: 8c and 55.65 - 8m,
        // and for the clipped form t / 256 from the exactly scaled factors
        uint32_t w = 0;
        bool fast = true;
        uint32_t sv[4];
        float c8[4], b[4];
        for (int e = 0; e < 4; ++e) {
            const int64_t i = (4 * g + e < n) ? 4 * g + e : n - 1;
            sv[e] = __float_as_uint(s_raw[i]);
            c8[e] = __fmul_rn(8.0f, c[i]);
            b[e] = __fsub_rn(kExpcastOffset, __fmul_rn(8.0f, m[i]));
            fast = fast && fabsf(m[i]) < kExpcastFastMax && __fmul_rn(s_raw[i], c[i]) <= __fadd_rn(m[i], 8.0f);
        }
        for (int e = 0; e < 4; ++e) {
            const uint32_t one[4] = {sv[e], sv[e], sv[e], sv[e]};
            const uint32_t code =
                (fast ? expcast4_fast(one, pk2(__float_as_uint(c8[e]), __float_as_uint(c8[e])),
                                      pk2(__float_as_uint(b[e]), __float_as_uint(b[e])), 1u)
                      : expcast4<true>(one, __fmul_rn(c8[e], 1.0f / 256.0f), __fmul_rn(b[e], 1.0f / 256.0f), 1u)) &
                0xFFu;
            w |= code << (8 * e);
        }
        for (int e = 0; e < 4; ++e)
            if (4 * g + e < n) out[4 * g + e] = static_cast<uint8_t>((w >> (8 * e)) & 0xFFu);
    }
}

__global__ void e4m3_bits_kernel(uint32_t start, int64_t n, uint8_t *__restrict__ out) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out[i] = static_cast<uint8_t>(e4m3(__uint_as_float(start + static_cast<uint32_t>(i))));
}

// One bounded wait on a barrier nothing completes: exercises the give-up path.
__global__ void selftest_timeout_kernel(int32_t *dev_status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, &abort_flag, limit_ns);
    __syncthreads();
    if (threadIdx.x == 0 && !ok) atomicExch(dev_status, kErrTimeout);
}

}  // namespace

cudaError_t launch_attention(const AttentionArgs &a, cudaStream_t st) {
    CUtensorMap mk, mv;
    const uint64_t rows = static_cast<uint64_t>(a.BH) * a.N;
    if (!make_tile_map(&mk, a.k8, rows) || !make_tile_map(&mv, a.v_res, rows)) return cudaErrorInvalidValue;
    Params p;
    p.q8 = a.q8;
    p.sq = a.sq;
    p.sk = a.sk;
    p.v_scale = a.v_scale;
    p.v_mean = a.v_mean;
    p.O = a.O;
    p.dev_status = a.dev_status;
    p.N = a.N;
    p.scale_log2 = a.scale_log2;
    p.limit_ns = a.wait_limit_ns;
    p.one = 1u;
    const dim3 grid(a.N / kBlk, a.BH);
    cudaError_t e;
    if (a.expcast) {
        e = cudaFuncSetAttribute(attention_e4m3_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attention_e4m3_kernel<true><<<grid, kThreads, kSmemBytes, st>>>(mk, mv, p);
    } else {
        e = cudaFuncSetAttribute(attention_e4m3_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attention_e4m3_kernel<false><<<grid, kThreads, kSmemBytes, st>>>(mk, mv, p);
    }
    return cudaGetLastError();
}

cudaError_t launch_expcast_codes(const float *s_raw, const float *c, const float *m, int64_t n, uint8_t *out,
                                 cudaStream_t st) {
    expcast_codes_kernel<<<1024, 256, 0, st>>>(s_raw, c, m, n, out);
    return cudaGetLastError();
}

cudaError_t launch_e4m3_encode_bits(uint32_t start, int64_t n, uint8_t *out, cudaStream_t st) {
    e4m3_bits_kernel<<<4096, 256, 0, st>>>(start, n, out);
    return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(int32_t *dev_status, uint64_t limit_ns, cudaStream_t st) {
    selftest_timeout_kernel<<<1, 32, 0, st>>>(dev_status, limit_ns);
    return cudaGetLastError();
}

}  // namespace vca
