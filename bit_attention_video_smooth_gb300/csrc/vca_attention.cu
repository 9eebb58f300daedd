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
//              N = 128) once K(b) has landed and P(b-2) has been released
//   warp 1     TMEM owner and PV issuer (one thread):
//                [E | O] += P_b [ones ; V8_b]       (kind::f8f6f4, N = 144): the
//                         16 extra output columns are the block's row sums of the
//                         decoded P, so the softmax threads never add them up
//              and every 16 key blocks O += [rowsum hi|lo] [mean/s_v hi|lo]^T (bf16).
//              Two issuing threads keep each one's serial work (barrier
//              checks, MMA issue, commits) off the other's critical path.
//   warps 2-9  softmax: two threads per query row -- the warps w and w+4 share
//              a TMEM lane quarter and take the S columns 0-63 and 64-127; the
//              pair exchanges its half-row maxima through shared memory at a
//              64-thread named barrier.  Reference max with the lazy threshold
//              (it moves only when a block's max exceeds it by 8), O rescaled in
//              TMEM when it moves, P codes stored to TMEM (the A operand of PV);
//              the row sum of block b-2 is read from its TMEM slot, brought to
//              the current max and buffered for the mean restore; epilogue
//              O = (O s_v + the last, partial group of mean terms) / l.
// The issuing threads wait for P with non-suspending polls (they are on the
// critical path); S[b&1] needs no signal of its own: every softmax warp reads
// S(b-2) before it releases P(b-2), which the QK thread waits for.
// TMEM columns: S0 [0,128), S1 [128,256), E0 [256,272), O [272,400), E1 [400,416),
// P0 [416,448), P1 [448,480), Q [480,512).  Q and P, the A operands of the two
// contractions, live in TMEM (four FP8 codes per column), so the tensor core
// reads only K and V from shared memory.
// Every wait is bounded; a wait that runs out raises a CTA-wide abort, the CTA
// drains its copies and MMAs, frees TMEM and reports VCA_ERR_TIMEOUT.
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
constexpr int kRsCap = 32;                 // buffered row sums per row (<= 17 in use)
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
constexpr uint32_t kOffRS = kOffMB + kTileBytes;            // fp32 [kRsCap][128] buffered row sums
constexpr uint32_t kOffSV = kOffRS + kRsCap * kBlk * 4;     // fp32 [128] residual scales
constexpr uint32_t kOffPM = kOffSV + kBlk * 4;              // fp32 [2][kParts][128] part-row maxima
constexpr uint32_t kOffL = kOffPM + 2 * kParts * kBlk * 4;  // fp32 [128] final row sums
constexpr uint32_t kOffBar = kOffL + kBlk * 4;
constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 2 + 2 + 2;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;       // tmem address, abort flag
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;       // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Bars {
    uint64_t *q_full, *k_full, *k_empty, *v_full, *v_empty, *p_full, *s_ready, *drain;
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

// Two threads issue the MMAs: the QK thread (S(b) = Q K_b^T) and the PV thread
// (O += P_j V_j and the mean-restore MMAs).  The softmax of block b waits on
// s_ready[b & 1], whose phase completes on two tcgen05.commit arrivals: the QK
// thread's after QK(b) (S(b) is in TMEM) and the PV thread's after PV(b-2)
// (P buffer and row-sum slot b & 1 are free, and the slot holds block b-2's
// sums).  Every waiter is at most one phase behind: the next phase of
// s_ready[b & 1] needs PV(b), which needs the softmax's P(b).
__device__ __forceinline__ bool wait_s_ready(const Bars &B, int b, int *abort, uint64_t limit_ns) {
    return mbar_wait(B.s_ready + (b & 1), (b >> 1) & 1, abort, limit_ns);
}

// A mean-restore MMA follows PV(b) when the row sums of blocks b-17 .. b-2 are
// all buffered (they are read two blocks late).
__host__ __device__ constexpr bool flush_after(int b) { return b >= kMeanJ + 1 && (b % kMeanJ) == 1; }

// exp2 then E4M3 for four raw scores: p = 2^(fma(S, c, -m)).
__device__ __forceinline__ uint32_t expconv4(uint64_t s01, uint64_t s23, uint64_t cx2, uint64_t negmx2) {
    float a[4];
    upk2(fma2(s01, cx2, negmx2), a[0], a[1]);
    upk2(fma2(s23, cx2, negmx2), a[2], a[3]);
    return e4m3x2(ex2_approx(a[0]), ex2_approx(a[1])) | (e4m3x2(ex2_approx(a[2]), ex2_approx(a[3])) << 16);
}

// P codes of this thread's half row (64 keys) against the reference max m,
// stored as 16 TMEM columns (four codes per column) of the P buffer at `tp`.
template <bool kExpcast>
__device__ __forceinline__ void write_codes(const uint32_t (&S)[kCols], float c, float m, uint32_t tp, uint32_t one) {
    uint32_t w[kCols / 4];
    if constexpr (kExpcast) {
        // t / 256 = fma(S, 8c / 256, (55.65 - 8m) / 256), both scalings exact
        const float c8s = __fmul_rn(c, 1.0f / 32.0f);
        const float bs = __fmul_rn(__fsub_rn(kExpcastOffset, __fmul_rn(8.0f, m)), 1.0f / 256.0f);
        if (__all_sync(0xffffffffu, fabsf(m) < kExpcastFastMax)) {
#pragma unroll
            for (int q = 0; q < kCols / 4; ++q) {
                const uint32_t sv[4] = {S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]};
                w[q] = expcast4<false>(sv, c8s, bs, one);
            }
        } else {
#pragma unroll
            for (int q = 0; q < kCols / 4; ++q) {
                const uint32_t sv[4] = {S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]};
                w[q] = expcast4<true>(sv, c8s, bs, one);
            }
        }
    } else {
        const float negm = -m;
        const uint64_t cx2 = pk2(__float_as_uint(c), __float_as_uint(c));
        const uint64_t nx2 = pk2(__float_as_uint(negm), __float_as_uint(negm));
#pragma unroll
        for (int q = 0; q < kCols / 4; ++q)
            w[q] = expconv4(pk2(S[4 * q], S[4 * q + 1]), pk2(S[4 * q + 2], S[4 * q + 3]), cx2, nx2);
    }
    if constexpr (kCols == 64) {
        VCA_TMEM_ST16(tp, w);
    } else {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(tp), "r"(w[0]),
                     "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
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
    B.p_full = B.v_empty + kVStages;
    B.s_ready = B.p_full + 2;
    B.drain = B.s_ready + 2;   // [0]: QK thread, [1]: PV thread
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    int *abort_flag = reinterpret_cast<int *>(smem + kOffMisc + 4);
    float *sRS = reinterpret_cast<float *>(smem + kOffRS);
    float *sSV = reinterpret_cast<float *>(smem + kOffSV);
    float *sPM = reinterpret_cast<float *>(smem + kOffPM);
    float *sL = reinterpret_cast<float *>(smem + kOffL);

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
            mbar_init(B.p_full + i, kSoftmaxWarps);
            mbar_init(B.s_ready + i, 2);   // QK(b) and PV(b-2)
            mbar_init(B.drain + i, 1);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp >= 2 && warp < 6) {
        const int t = threadIdx.x - 64;
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
                mbar_expect_tx(full + s, kTileBytes);
                tma_load_2d(ring + s * stride, tm, full + s, 0, is_k ? bh * N + b * kBlk : (bh * nb + b) * kBlk);
                armed[s] = use + 1;
            }
            // every copy this thread issued has landed before the CTA can exit
            for (int s = 0; s < stages; ++s)
                if (armed[s] > 0) drain_wait(full + s, (armed[s] - 1) & 1, p.limit_ns);
        }
    } else if (warp == kQKWarp) {
        // ------------------------------------------------------------ QK issuer
        // QK(b) into S[b & 1] once K(b) has landed and the softmax has released
        // P(b-2) (it reads S(b-2) out of S[b & 1] before that); then commits
        // for the K stage and for s_ready.  Steps nb and nb+1 issue no MMA but
        // still wait for P(b-2) and commit, so that the last two phases of
        // s_ready (the epilogue waits for them) complete, each only after the
        // phase before it on the same barrier.
        if (lane == 0) {
            constexpr uint32_t idesc_qk = make_idesc(128, 128, 0, 0);
            const uint32_t sbase = smem_u32(smem);
            bool ok = mbar_wait(B.q_full, 0, abort_flag, p.limit_ns);
            for (int b = 0; ok && b < nb + 2; ++b) {
                if (b >= 2 && !mbar_wait_spin(B.p_full + (b & 1), ((b - 2) >> 1) & 1, abort_flag, p.limit_ns)) break;
                if (b < nb) {
                    const int s = b % kKStages, sb = b & 1;
                    if (!mbar_wait(B.k_full + s, (b / kKStages) & 1, abort_flag, p.limit_ns)) break;
                    tc_fence_after();
                    const uint64_t dk = sdesc_k_sw128(sbase + kOffK + s * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < kD / 32; ++kk)
                        mma_f8f6f4_ts(tmem + sb * 128, tmem + kTmemQ + 8 * kk, dk + 2 * kk, idesc_qk, kk > 0);
                    tc_commit(B.k_empty + s);
                }
                tc_commit(B.s_ready + (b & 1));
            }
            tc_commit(B.drain);
            drain_wait(B.drain, 0, p.limit_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ PV issuer
        // PV(j) once P(j) is written and V(j) has landed: [E | O] += P [ones ; V]
        // (the 16 extra columns receive the row sums), the mean-restore MMA when
        // due, then commits for the V stage and for s_ready (phase of block j+2).
        if (lane == 0) {
            constexpr uint32_t idesc_pv = make_idesc(128, 144, 0, 0);
            constexpr uint32_t idesc_bf16 = make_idesc(128, 128, 1, 1);
            const uint32_t sbase = smem_u32(smem);
            const uint64_t dma = sdesc_k_sw128(sbase + kOffMA);
            const uint64_t dmb = sdesc_k_sw128(sbase + kOffMB);
            const uint32_t tO = tmem + kTmemO;
            // blocks 0 and 1 have no PV(b-2): their s_ready phases take a plain arrival
            mbar_arrive(B.s_ready);
            mbar_arrive(B.s_ready + 1);
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
                tc_commit(B.s_ready + pb);
            }
            tc_commit(B.drain + 1);
            drain_wait(B.drain + 1, 0, p.limit_ns);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3;                              // TMEM lane quarter
        const int half = (warp - 2) >> 2;                          // column part: S columns kCols*half ..
        const int row = quarter * 32 + lane;                       // query row in the tile == TMEM lane
        const uint32_t pair_bar = kBarPair0 + quarter;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t col0 = static_cast<uint32_t>(kCols) * half;
        const uint32_t tO = tmem + lane_base + kTmemO + col0;
        const float sqv = p.sq[static_cast<int64_t>(bh) * nb + qtile];
        const float *skh = p.sk + static_cast<int64_t>(bh) * nb;
        const uint16_t *vmh = p.v_mean + static_cast<int64_t>(bh) * nb * kD;
        unsigned char *sMA = smem + kOffMA;
        unsigned char *sMB = smem + kOffMB;
        const float kNegInf = __int_as_float(0xff800000);
        float m = kNegInf, mh1 = kNegInf, mh2 = kNegInf;   // running max; the max of blocks b-1, b-2
        float l = 0.0f;                                    // kept by the half-0 thread of the row
        int rs_cnt = 0;
        bool ok = true;
        float sk_next = skh[0];
        if (half == 0) {
            // Q tile into TMEM (the A operand of QK): this row's 128 codes, 32 columns
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
            // S(b) is ready, and with it PV(b-2): P buffer sb is free and the
            // row-sum slot of this parity holds block b-2's sums
            bool wok = wait_s_ready(B, b, abort_flag, p.limit_ns);
            wok = __all_sync(0xffffffffu, wok) && ok;
            uint32_t S[kCols];
            uint32_t rs_raw = 0;
            float pm = kNegInf;
            const float c = __fmul_rn(__fmul_rn(sqv, sk_b), p.scale_log2);
            const uint32_t tp = tmem + lane_base + kTmemP0 + 32 * sb + (kCols / 4) * half;
            if (wok) {
                tc_fence_after();
                const uint32_t tS = tmem + lane_base + sb * 128 + col0;
#pragma unroll
                for (int i = 0; i < kCols / 32; ++i) VCA_TMEM_LD32(tS + 32 * i, (S + 32 * i));
                // half 0 owns the row-sum slot of this parity: read block b-2's
                // sum, then clear the slot for PV(b) (PV(0) initialises E0 itself)
                const uint32_t te = tmem + lane_base + (sb == 0 ? kTmemE0 : kTmemE1);
                if (half == 0 && b >= 2)
                    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(rs_raw) : "r"(te));
                tmem_ld_wait();
                if (half == 0 && b >= 1)   // completes before P(b) is released
                    asm volatile(
                        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1,%1};"
                        ::"r"(te), "r"(0u) : "memory");
                pm = row_part_max(S);
                // codes against the current reference max, on the bet that this
                // block does not move it (rewritten below when it does)
                if (b > 0) write_codes<kExpcast>(S, c, m, tp, p.one);
            }
            // Lazy reference-max update: only when the block's max exceeds m by
            // tau.  The block max moves m exactly when one part's max does
            // (scaling by c >= 0 is monotone), so the common case takes one pair
            // barrier: every thread of the row finished its wait and no part
            // moves m.  Otherwise the parts exchange their maxima.
            const float lim = __fadd_rn(m, kLazyTau);
            const bool quiet = bar_and(wok && !(__fmul_rn(pm, c) > lim), pair_bar, 32 * kParts);
            float alpha = 1.0f;
            bool rescale = false;
            if (!quiet) {
                sPM[(sb * kParts + half) * kBlk + row] = pm;
                ok = bar_and(wok, pair_bar, 32 * kParts);
                if (!ok) break;
                float smax = pm;
#pragma unroll
                for (int q = 1; q < kParts; ++q)
                    smax = fmaxf(smax, sPM[(sb * kParts + ((half + q) % kParts)) * kBlk + row]);
                const float bm = __fmul_rn(smax, c);
                const bool moved = bm > lim;
                if (moved) {
                    if (b > 0) alpha = ex2_approx(__fsub_rn(m, bm));
                    m = bm;
                }
                if (__any_sync(0xffffffffu, moved)) {
                    // S(b) is still in TMEM (S[b&1] is rewritten only after P(b) is
                    // released): reload it rather than keep 64 registers live
                    // through the code computation for this rare path
                    tmem_st_wait();   // the optimistic codes land before they are replaced
                    uint32_t S2[kCols];
                    const uint32_t tS = tmem + lane_base + sb * 128 + col0;
#pragma unroll
                    for (int i = 0; i < kCols / 32; ++i) VCA_TMEM_LD32(tS + 32 * i, (S2 + 32 * i));
                    tmem_ld_wait();
                    write_codes<kExpcast>(S2, c, m, tp, p.one);
                }
                rescale = __any_sync(0xffffffffu, alpha != 1.0f);
                if (half == 0 && alpha != 1.0f) {
                    l = __fmul_rn(l, alpha);
#pragma unroll 1
                    for (int i = 0; i < rs_cnt; ++i) sRS[i * kBlk + row] = __fmul_rn(sRS[i * kBlk + row], alpha);
                }
            }
            if (half == 0 && b >= 2) {
                // row sum of block b-2, taken against that block's max: bring it to m
                float rs = __uint_as_float(rs_raw);
                if (mh2 != m) rs = __fmul_rn(rs, ex2_approx(__fsub_rn(mh2, m)));
                l = __fadd_rn(l, rs);
                sRS[rs_cnt * kBlk + row] = rs;
            }
            if (b >= 2) ++rs_cnt;

            // rescale this half of the O accumulator after PV(b-1) (and any mean
            // MMA after it) finished
            if (rescale) {
                const int jb = b - 1;
                ok = __all_sync(0xffffffffu, wait_s_ready(B, jb + 2, abort_flag, p.limit_ns));
                if (ok) {
                    tc_fence_after();
#pragma unroll 1
                    for (int i = 0; i < kCols / 32; ++i) {
                        uint32_t o[32];
                        VCA_TMEM_LD32(tO + 32 * i, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__fmul_rn(__uint_as_float(o[e]), alpha));
                        VCA_TMEM_ST32(tO + 32 * i, o);
                    }
                    tmem_st_wait();
                }
            }

            if (ok && flush_after(b)) {
                // row sums of blocks b0 .. b0+15 (all at the current max)
                stage_mean_operands(half, row, sRS, vmh, b - kMeanJ - 1, sSV, sMA, sMB);
                rs_cnt = 0;
                fence_proxy_async_smem();   // the mean operands are read by the tensor core
            }
            if (ok) {
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(B.p_full + sb);
            }
            mh2 = mh1;
            mh1 = m;
        }
        // ------------------------------------------------------------ epilogue
        if (ok) {
            const int jb = nb - 1;
            ok = __all_sync(0xffffffffu, wait_s_ready(B, jb + 2, abort_flag, p.limit_ns));
        }
        // every softmax warp arrives here, whether it finished or gave up; the
        // epilogue (and its barriers) runs only if all of them finished
        ok = bar_and(ok, kBarSoftmax, 32 * kSoftmaxWarps);
        if (ok) {
            tc_fence_after();
            if (half == 0) {
                // the last two blocks' row sums
                uint32_t r2 = 0, r1 = 0;
                const uint32_t te0 = tmem + lane_base + kTmemE0, te1 = tmem + lane_base + kTmemE1;
                const uint32_t te_last = ((nb - 1) & 1) ? te1 : te0, te_prev = ((nb - 1) & 1) ? te0 : te1;
                if (nb >= 2)
                    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r2) : "r"(te_prev));
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r1) : "r"(te_last));
                tmem_ld_wait();
                int cnt = rs_cnt;
                if (nb >= 2) {
                    float rs = __uint_as_float(r2);
                    if (mh2 != m) rs = __fmul_rn(rs, ex2_approx(__fsub_rn(mh2, m)));
                    l = __fadd_rn(l, rs);
                    sRS[cnt * kBlk + row] = rs;
                    ++cnt;
                }
                const float rs = __uint_as_float(r1);   // taken against m itself
                l = __fadd_rn(l, rs);
                sRS[cnt * kBlk + row] = rs;
                sL[row] = l;
            }
            rs_cnt += (nb >= 2) ? 2 : 1;
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
            store_output(tO, sSV, sRS, sMu, rs_cnt, row, static_cast<int>(col0), inv_l, orow);
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

// --------------------------------------------------------------------------
// Host side: tensor maps and launch
// --------------------------------------------------------------------------
// ExpCast map alone, for bit-exact tests of the device function.
// Four elements per thread through the same packed path the attention kernel
// uses.  The unclipped variant is taken where the attention kernel would take
// it: |m| < 2^22 and fp32(s_raw * c) <= fp32(m + 8) (m is the lazily updated
// reference max there).
__global__ void expcast_codes_kernel(const float *__restrict__ s_raw, const float *__restrict__ c,
                                     const float *__restrict__ m, int64_t n, uint8_t *__restrict__ out) {
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; 4 * g < n;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // the kernel's arithmetic, one scale per element: t / 256 from the
        // exactly scaled factors
        uint32_t w = 0;
        bool fast = true;
        uint32_t sv[4];
        float c8s[4], bs[4];
        for (int e = 0; e < 4; ++e) {
            const int64_t i = (4 * g + e < n) ? 4 * g + e : n - 1;
            sv[e] = __float_as_uint(s_raw[i]);
            c8s[e] = __fmul_rn(c[i], 1.0f / 32.0f);
            bs[e] = __fmul_rn(__fsub_rn(kExpcastOffset, __fmul_rn(8.0f, m[i])), 1.0f / 256.0f);
            fast = fast && fabsf(m[i]) < kExpcastFastMax && __fmul_rn(s_raw[i], c[i]) <= __fadd_rn(m[i], 8.0f);
        }
        for (int e = 0; e < 4; ++e) {
            const uint32_t one[4] = {sv[e], sv[e], sv[e], sv[e]};
            const uint32_t code = (fast ? expcast4<false>(one, c8s[e], bs[e], 1u) : expcast4<true>(one, c8s[e], bs[e], 1u)) & 0xFFu;
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
