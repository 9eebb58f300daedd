// vca_attention.cu -- non-causal FP8 attention with the V-Smooth mean restore
// and ExpCast-FP8 ("VC-Attention", paper page, section "method"): QK and PV on
// FP8 tensor cores, online softmax whose per-block row sums bring the block
// means back as one outer product rowsum_b (x) mean_b, and ExpCast writing the
// E4M3 probability bytes with one FMA (news page, "ExpCast-FP8").
//
// One CTA owns a 128-row query tile of one (batch, head) and streams the key
// blocks of that head in increasing (permuted) order.  Warp roles:
//   warp 0     TMA producer: Q once, then K / V-residual tiles into a 3-stage ring
//   warp 1     TMEM owner and MMA issuer (one thread), per key block b:
//                S[b&1] = Q8 K8_b^T                       (kind::f8f6f4, N = 128)
//                O     += P_{b-1} V8_{b-1}                 (kind::f8f6f4, N = 128)
//                RS[(b-1)%8] = P_{b-1} 1                   (kind::f8f6f4, N = 16)
//              the last one writes the block's row sums of the decoded P into a
//              rotating TMEM slot, so the softmax threads never add them up; and
//              every 16 key blocks O += [rowsum hi|lo] [mean/s_v hi|lo]^T (bf16).
//   warps 2-5  softmax: one thread per query row (its TMEM lane); running max,
//              O rescale in TMEM when the max grows, P codes straight to shared
//              memory in the 128-byte-swizzled K-major layout the MMAs read; the
//              row sum of block b-2 is read from its TMEM slot, brought to the
//              current max and buffered for the mean restore; epilogue
//              O = (O s_v + the last, partial group of mean terms) / l.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384), row-sum slots [384,512).
// Every wait is bounded; a wait that runs out raises a CTA-wide abort, the CTA
// drains its copies and MMAs, frees TMEM and reports VCA_ERR_TIMEOUT.
#include <cuda.h>

#include "vca_device.cuh"
#include "vca_internal.h"

namespace vca {

namespace {

constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr int kMeanJ = 16;                 // key blocks per mean-restore MMA
constexpr int kRsSlots = 8;                // rotating TMEM row-sum slots (16 columns each)
constexpr int kRsCap = 32;                 // buffered row sums per thread (<= 17 in use)
constexpr uint32_t kTileBytes = kBlk * kD; // one 128 x 128 FP8 tile (16 KB)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256, kTmemRS = 384;

// shared-memory layout (bytes from a 1024-aligned base)
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
constexpr uint32_t kOffP = kOffV + kStages * kTileBytes;
constexpr uint32_t kOffMA = kOffP + 2 * kTileBytes;
constexpr uint32_t kOffMB = kOffMA + kTileBytes;
constexpr uint32_t kOffOnes = kOffMB + kTileBytes;          // 16 x 128 E4M3 ones (B of the row-sum MMA)
constexpr uint32_t kOffRS = kOffOnes + 16 * 128;            // fp32 [kRsCap][128] buffered row sums
constexpr uint32_t kOffSV = kOffRS + kRsCap * kBlk * 4;     // fp32 [128] residual scales
constexpr uint32_t kOffBar = kOffSV + kBlk * 4;
constexpr int kNumBars = 1 + 3 * kStages + 2 * 4 + 1;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;       // tmem address, abort flag
constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;       // + alignment slack

struct Bars {
    uint64_t *q_full, *k_full, *v_full, *kv_empty, *s_full, *s_free, *p_full, *pv_done, *drain;
};

struct Params {
    const float *sq, *sk, *v_scale;
    const uint16_t *v_mean;
    uint16_t *O;
    int32_t *dev_status;
    int N;
    float scale_log2;
    uint64_t limit_ns;
};

// A mean-restore MMA follows PV(b) when the row sums of blocks b-17 .. b-2 are
// all buffered (they are read two blocks late).
__host__ __device__ constexpr bool flush_after(int b) { return b >= kMeanJ + 1 && (b % kMeanJ) == 1; }

// Wait ignoring the abort flag (used only to drain work this thread issued).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// hi + lo split of x into two bf16 values (x ~= hi + lo to ~16 bits).
__device__ __forceinline__ void split_bf16(float x, float &hi, float &lo) {
    hi = __bfloat162float(__float2bfloat16_rn(x));
    lo = __fsub_rn(x, hi);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// packed fp32 pairs (two lanes per instruction on sm_100+)
__device__ __forceinline__ uint64_t pk2(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ void upk2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ExpCast for four raw scores -> four E4M3 bytes in one word (the same
// arithmetic as expcast_rounded(): one fp32 FMA, magic-constant rounding,
// flush below code 8, clip above 126).
__device__ __forceinline__ uint32_t expcast4(uint32_t s0, uint32_t s1, uint32_t s2, uint32_t s3, uint64_t c8x2,
                                             uint64_t biasx2, uint64_t magicx2) {
    float x[4];
    upk2(add2(fma2(pk2(s0, s1), c8x2, biasx2), magicx2), x[0], x[1]);
    upk2(add2(fma2(pk2(s2, s3), c8x2, biasx2), magicx2), x[2], x[3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[e] = (x[e] >= kMagic + 8.0f) ? x[e] : kMagic;
        x[e] = fminf(x[e], kMagic + 126.0f);
    }
    return __byte_perm(__byte_perm(__float_as_uint(x[0]), __float_as_uint(x[1]), 0x0040),
                       __byte_perm(__float_as_uint(x[2]), __float_as_uint(x[3]), 0x0040), 0x5410);
}

// exp2 then E4M3 for four raw scores: p = 2^(fma(S, c, -m)).
__device__ __forceinline__ uint32_t expconv4(uint32_t s0, uint32_t s1, uint32_t s2, uint32_t s3, uint64_t cx2,
                                             uint64_t negmx2) {
    float a[4];
    upk2(fma2(pk2(s0, s1), cx2, negmx2), a[0], a[1]);
    upk2(fma2(pk2(s2, s3), cx2, negmx2), a[2], a[3]);
    return e4m3x2(ex2_approx(a[0]), ex2_approx(a[1])) | (e4m3x2(ex2_approx(a[2]), ex2_approx(a[3])) << 16);
}

__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Named barrier over the four softmax warps that also ANDs a flag across them.
__device__ __forceinline__ bool softmax_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v))
        : "memory");
    return r != 0;
}

template <bool kExpcast>
__global__ void __launch_bounds__(kThreads, 1)
    attention_e4m3_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    Bars B;
    B.q_full = bars;
    B.k_full = bars + 1;
    B.v_full = B.k_full + kStages;
    B.kv_empty = B.v_full + kStages;
    B.s_full = B.kv_empty + kStages;
    B.s_free = B.s_full + 2;
    B.p_full = B.s_free + 2;
    B.pv_done = B.p_full + 2;
    B.drain = B.pv_done + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    int *abort_flag = reinterpret_cast<int *>(smem + kOffMisc + 4);
    float *sRS = reinterpret_cast<float *>(smem + kOffRS);
    float *sSV = reinterpret_cast<float *>(smem + kOffSV);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qtile = blockIdx.x, bh = blockIdx.y;
    const int N = p.N, nb = N / kBlk;

    if (threadIdx.x == 0) {
        mbar_init(B.q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(B.k_full + s, 1);
            mbar_init(B.v_full + s, 1);
            mbar_init(B.kv_empty + s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(B.s_full + i, 1);
            mbar_init(B.s_free + i, 4);
            mbar_init(B.p_full + i, 4);
            mbar_init(B.pv_done + i, 1);
        }
        mbar_init(B.drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp >= 2) {
        const int t = threadIdx.x - 64;
        sSV[t] = p.v_scale[static_cast<int64_t>(bh) * kD + t];
        // the ones tile: 16 rows x 128 bytes of E4M3 1.0 (0x38)
        *reinterpret_cast<uint4 *>(smem + kOffOnes + 16 * t) = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int armed[kStages];
            for (int s = 0; s < kStages; ++s) armed[s] = 0;
            mbar_expect_tx(B.q_full, kTileBytes);
            tma_load_2d(smem + kOffQ, &tmQ, B.q_full, 0, bh * N + qtile * kBlk);
            for (int b = 0; b < nb; ++b) {
                const int s = b % kStages, use = b / kStages;
                if (use > 0 && !mbar_wait(B.kv_empty + s, (use - 1) & 1, abort_flag, p.limit_ns)) break;
                mbar_expect_tx(B.k_full + s, kTileBytes);
                tma_load_2d(smem + kOffK + s * kTileBytes, &tmK, B.k_full + s, 0, bh * N + b * kBlk);
                mbar_expect_tx(B.v_full + s, kTileBytes);
                tma_load_2d(smem + kOffV + s * kTileBytes, &tmV, B.v_full + s, 0, (bh * nb + b) * kBlk);
                armed[s] = use + 1;
            }
            // every copy this thread issued has landed before the CTA can exit
            drain_wait(B.q_full, 0, p.limit_ns);
            for (int s = 0; s < kStages; ++s)
                if (armed[s] > 0) {
                    drain_wait(B.k_full + s, (armed[s] - 1) & 1, p.limit_ns);
                    drain_wait(B.v_full + s, (armed[s] - 1) & 1, p.limit_ns);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_f8 = make_idesc(128, 128, 0, 0);
            constexpr uint32_t idesc_rs = make_idesc(128, 16, 0, 0);
            constexpr uint32_t idesc_bf16 = make_idesc(128, 128, 1, 1);
            const uint32_t sbase = smem_u32(smem);
            const uint64_t dq = sdesc_k_sw128(sbase + kOffQ);
            const uint64_t dma = sdesc_k_sw128(sbase + kOffMA);
            const uint64_t dmb = sdesc_k_sw128(sbase + kOffMB);
            const uint64_t dones = sdesc_k_sw128(sbase + kOffOnes);
            const uint32_t tO = tmem + kTmemO;
            bool ok = mbar_wait(B.q_full, 0, abort_flag, p.limit_ns);
            for (int b = 0; ok && b <= nb; ++b) {
                if (b < nb) {
                    const int s = b % kStages, sb = b & 1;
                    if (!mbar_wait(B.k_full + s, (b / kStages) & 1, abort_flag, p.limit_ns)) break;
                    if (b >= 2 && !mbar_wait(B.s_free + sb, ((b >> 1) - 1) & 1, abort_flag, p.limit_ns)) break;
                    tc_fence_after();
                    const uint64_t dk = sdesc_k_sw128(sbase + kOffK + s * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < kD / 32; ++kk)
                        mma_f8f6f4(tmem + sb * 128, dq + 2 * kk, dk + 2 * kk, idesc_f8, kk > 0);
                    tc_commit(B.s_full + sb);
                }
                if (b >= 1) {
                    const int j = b - 1, s = j % kStages, pb = j & 1;
                    if (!mbar_wait(B.v_full + s, (j / kStages) & 1, abort_flag, p.limit_ns)) break;
                    if (!mbar_wait(B.p_full + pb, (j >> 1) & 1, abort_flag, p.limit_ns)) break;
                    tc_fence_after();
                    const uint64_t dp = sdesc_k_sw128(sbase + kOffP + pb * kTileBytes);
                    const uint64_t dv = sdesc_k_sw128(sbase + kOffV + s * kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < kBlk / 32; ++kk)
                        mma_f8f6f4(tO, dp + 2 * kk, dv + 2 * kk, idesc_f8, (j > 0 || kk > 0) ? 1u : 0u);
                    const uint32_t trs = tmem + kTmemRS + 16 * (j % kRsSlots);
#pragma unroll
                    for (int kk = 0; kk < kBlk / 32; ++kk)
                        mma_f8f6f4(trs, dp + 2 * kk, dones + 2 * kk, idesc_rs, kk > 0 ? 1u : 0u);
                    if (flush_after(j)) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) mma_f16(tO, dma + 2 * kk, dmb + 2 * kk, idesc_bf16, 1u);
                    }
                    tc_commit(B.kv_empty + s);
                    tc_commit(B.pv_done + pb);
                }
            }
            tc_commit(B.drain);
            drain_wait(B.drain, 0, p.limit_ns);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;                       // query row in the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_base + kTmemO;
        const float sqv = p.sq[static_cast<int64_t>(bh) * nb + qtile];
        const float *skh = p.sk + static_cast<int64_t>(bh) * nb;
        const uint16_t *vmh = p.v_mean + static_cast<int64_t>(bh) * nb * kD;
        unsigned char *sP = smem + kOffP;
        unsigned char *sMA = smem + kOffMA;
        unsigned char *sMB = smem + kOffMB;
        const float kNegInf = __int_as_float(0xff800000);
        float m = kNegInf, mh1 = kNegInf, mh2 = kNegInf;   // running max; the max of blocks b-1, b-2
        float l = 0.0f;
        int rs_cnt = 0;
        bool ok = true;
        float sk_next = skh[0];
        for (int b = 0; b < nb; ++b) {
            const int sb = b & 1;
            const float sk_b = sk_next;
            if (b + 1 < nb) sk_next = skh[b + 1];
            ok = __all_sync(0xffffffffu, mbar_wait(B.s_full + sb, (b >> 1) & 1, abort_flag, p.limit_ns));
            if (!ok) break;
            // PV(b-2) and its row sums are done (also frees P buffer sb)
            if (b >= 2) {
                ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done + sb, ((b >> 1) - 1) & 1, abort_flag, p.limit_ns));
                if (!ok) break;
            }
            tc_fence_after();
            uint32_t S[128];
            uint32_t rs_raw = 0;
            const uint32_t tS = tmem + lane_base + sb * 128;
            VCA_TMEM_LD32(tS + 0, (S + 0));
            VCA_TMEM_LD32(tS + 32, (S + 32));
            VCA_TMEM_LD32(tS + 64, (S + 64));
            VCA_TMEM_LD32(tS + 96, (S + 96));
            if (b >= 2) {
                const uint32_t trs = tmem + lane_base + kTmemRS + 16 * ((b - 2) % kRsSlots);
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(rs_raw) : "r"(trs));
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.s_free + sb);

            const float c = __fmul_rn(__fmul_rn(sqv, sk_b), p.scale_log2);
            float a0 = __uint_as_float(S[0]), a1 = __uint_as_float(S[1]);
            float a2 = __uint_as_float(S[2]), a3 = __uint_as_float(S[3]);
#pragma unroll
            for (int j = 4; j < 128; j += 8) {
                a0 = max3(a0, __uint_as_float(S[j + 0]), __uint_as_float(S[j + 1]));
                a1 = max3(a1, __uint_as_float(S[j + 2]), __uint_as_float(S[j + 3]));
                a2 = max3(a2, __uint_as_float(S[j + 4]), __uint_as_float(S[j + 5]));
                a3 = max3(a3, __uint_as_float(S[j + 6]), __uint_as_float(S[j + 7]));
            }
            const float smax = fmaxf(max3(a0, a1, a2), a3);
            const float m_new = fmaxf(m, __fmul_rn(smax, c));
            float alpha = 1.0f;
            if (m_new > m && b > 0) alpha = ex2_approx(__fsub_rn(m, m_new));
            m = m_new;
            const bool rescale = __any_sync(0xffffffffu, alpha != 1.0f);
            if (alpha != 1.0f) {
                l = __fmul_rn(l, alpha);
#pragma unroll 1
                for (int i = 0; i < rs_cnt; ++i) sRS[i * kBlk + row] = __fmul_rn(sRS[i * kBlk + row], alpha);
            }
            if (b >= 2) {
                // row sum of block b-2, taken against that block's max: bring it to m
                float rs = __uint_as_float(rs_raw);
                if (mh2 != m) rs = __fmul_rn(rs, ex2_approx(__fsub_rn(mh2, m)));
                l = __fadd_rn(l, rs);
                sRS[rs_cnt * kBlk + row] = rs;
                ++rs_cnt;
            }

            unsigned char *prow = sP + sb * kTileBytes;
            if constexpr (kExpcast) {
                const float c8 = __fmul_rn(8.0f, c);
                const float bias = __fsub_rn(kExpcastOffset, __fmul_rn(8.0f, m));
                const uint64_t c8x2 = pk2(__float_as_uint(c8), __float_as_uint(c8));
                const uint64_t bx2 = pk2(__float_as_uint(bias), __float_as_uint(bias));
                const uint64_t mx2 = pk2(__float_as_uint(kMagic), __float_as_uint(kMagic));
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint32_t *s = S + ch * 16;
                    const uint32_t w0 = expcast4(s[0], s[1], s[2], s[3], c8x2, bx2, mx2);
                    const uint32_t w1 = expcast4(s[4], s[5], s[6], s[7], c8x2, bx2, mx2);
                    const uint32_t w2 = expcast4(s[8], s[9], s[10], s[11], c8x2, bx2, mx2);
                    const uint32_t w3 = expcast4(s[12], s[13], s[14], s[15], c8x2, bx2, mx2);
                    *reinterpret_cast<uint4 *>(prow + sw128_offset(row, ch)) = make_uint4(w0, w1, w2, w3);
                }
            } else {
                const float negm = -m;
                const uint64_t cx2 = pk2(__float_as_uint(c), __float_as_uint(c));
                const uint64_t nx2 = pk2(__float_as_uint(negm), __float_as_uint(negm));
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint32_t *s = S + ch * 16;
                    const uint32_t w0 = expconv4(s[0], s[1], s[2], s[3], cx2, nx2);
                    const uint32_t w1 = expconv4(s[4], s[5], s[6], s[7], cx2, nx2);
                    const uint32_t w2 = expconv4(s[8], s[9], s[10], s[11], cx2, nx2);
                    const uint32_t w3 = expconv4(s[12], s[13], s[14], s[15], cx2, nx2);
                    *reinterpret_cast<uint4 *>(prow + sw128_offset(row, ch)) = make_uint4(w0, w1, w2, w3);
                }
            }

            // rescale the O accumulator after PV(b-1) (and any mean MMA after it) finished
            if (rescale) {
                const int jb = b - 1;
                ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done + (jb & 1), (jb >> 1) & 1, abort_flag, p.limit_ns));
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
                    uint32_t o[32];
                    VCA_TMEM_LD32(tO + 32 * i, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__fmul_rn(__uint_as_float(o[e]), alpha));
                    VCA_TMEM_ST32(tO + 32 * i, o);
                }
                tmem_st_wait();
            }

            if (flush_after(b)) {
                // row sums of blocks b0 .. b0+15 (all at the current max):
                // A row (this query row): [rs hi | rs lo | rs hi | rs lo]
                // B row (channel `row`):  [mu hi | mu hi | mu lo | mu lo], mu = mean / s_v
                const int b0 = b - kMeanJ - 1;
                const float inv_sv = 1.0f / sSV[row];
                float rh[kMeanJ], rl[kMeanJ], mh[kMeanJ], ml[kMeanJ];
#pragma unroll
                for (int i = 0; i < kMeanJ; ++i) {
                    split_bf16(sRS[i * kBlk + row], rh[i], rl[i]);
                    split_bf16(__fmul_rn(bf16_bits_to_f32(vmh[(b0 + i) * kD + row]), inv_sv), mh[i], ml[i]);
                }
#pragma unroll
                for (int ck = 0; ck < 8; ++ck) {
                    const float *srcA = ((ck >> 1) & 1) ? rl : rh;   // chunks 0,1 hi; 2,3 lo; 4,5 hi; 6,7 lo
                    const float *srcB = (ck < 4) ? mh : ml;          // chunks 0-3 hi; 4-7 lo
                    const int i0 = (ck & 1) * 8;
                    uint4 a, bv;
                    a.x = pack_bf16x2(srcA[i0 + 0], srcA[i0 + 1]);
                    a.y = pack_bf16x2(srcA[i0 + 2], srcA[i0 + 3]);
                    a.z = pack_bf16x2(srcA[i0 + 4], srcA[i0 + 5]);
                    a.w = pack_bf16x2(srcA[i0 + 6], srcA[i0 + 7]);
                    bv.x = pack_bf16x2(srcB[i0 + 0], srcB[i0 + 1]);
                    bv.y = pack_bf16x2(srcB[i0 + 2], srcB[i0 + 3]);
                    bv.z = pack_bf16x2(srcB[i0 + 4], srcB[i0 + 5]);
                    bv.w = pack_bf16x2(srcB[i0 + 6], srcB[i0 + 7]);
                    *reinterpret_cast<uint4 *>(sMA + sw128_offset(row, ck)) = a;
                    *reinterpret_cast<uint4 *>(sMB + sw128_offset(row, ck)) = bv;
                }
                rs_cnt = 0;
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.p_full + sb);
            mh2 = mh1;
            mh1 = m;
        }
        // ------------------------------------------------------------ epilogue
        if (ok) {
            const int jb = nb - 1;
            ok = __all_sync(0xffffffffu, mbar_wait(B.pv_done + (jb & 1), (jb >> 1) & 1, abort_flag, p.limit_ns));
        }
        // every softmax warp arrives here, whether it finished or gave up; the
        // epilogue (and its named barrier) runs only if all four finished
        ok = softmax_all(ok);
        if (ok) {
            tc_fence_after();
            // the last two blocks' row sums
            uint32_t r2 = 0, r1 = 0;
            const uint32_t tr = tmem + lane_base + kTmemRS;
            if (nb >= 2)
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                             : "=r"(r2) : "r"(tr + 16 * ((nb - 2) % kRsSlots)));
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                         : "=r"(r1) : "r"(tr + 16 * ((nb - 1) % kRsSlots)));
            tmem_ld_wait();
            if (nb >= 2) {
                float rs = __uint_as_float(r2);
                if (mh2 != m) rs = __fmul_rn(rs, ex2_approx(__fsub_rn(mh2, m)));
                l = __fadd_rn(l, rs);
                sRS[rs_cnt * kBlk + row] = rs;
                ++rs_cnt;
            }
            {
                const float rs = __uint_as_float(r1);   // taken against m itself
                l = __fadd_rn(l, rs);
                sRS[rs_cnt * kBlk + row] = rs;
                ++rs_cnt;
            }
            // the blocks since the last mean MMA: stage their means (fp32) in the
            // mean-B buffer, whose last reader (the final mean MMA) has finished
            const int tail0 = nb - rs_cnt;
            float *sMu = reinterpret_cast<float *>(sMB);
            softmax_bar();
            for (int i = threadIdx.x - 64; i < rs_cnt * kD; i += 128)
                sMu[i] = bf16_bits_to_f32(vmh[(tail0 + i / kD) * kD + (i % kD)]);
            softmax_bar();
            const float inv_l = 1.0f / l;
            uint16_t *orow = p.O + (static_cast<int64_t>(bh) * N + static_cast<int64_t>(qtile) * kBlk + row) * kD;
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                uint32_t o[32];
                VCA_TMEM_LD32(tO + 32 * i, o);
                tmem_ld_wait();
                float acc[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) acc[e] = __fmul_rn(__uint_as_float(o[e]), sSV[32 * i + e]);
#pragma unroll 1
                for (int t = 0; t < rs_cnt; ++t) {
                    const float r = sRS[t * kBlk + row];
                    const float *mu = sMu + t * kD + 32 * i;
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[e] = __fmaf_rn(r, mu[e], acc[e]);
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack_bf16x2(__fmul_rn(acc[2 * e], inv_l), __fmul_rn(acc[2 * e + 1], inv_l));
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    reinterpret_cast<uint4 *>(orow + 32 * i)[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
            }
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
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 2-D byte matrix [rows][128] with 128 x 128 boxes and the 128-byte swizzle.
bool make_tile_map(CUtensorMap *map, const void *base, uint64_t rows) {
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

// ExpCast map alone, for bit-exact tests of the device function.
__global__ void expcast_codes_kernel(const float *__restrict__ s_raw, const float *__restrict__ c,
                                     const float *__restrict__ m, int64_t n, uint8_t *__restrict__ out) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float c8 = __fmul_rn(8.0f, c[i]);
        const float bias = __fsub_rn(kExpcastOffset, __fmul_rn(8.0f, m[i]));
        out[i] = static_cast<uint8_t>(expcast_code(s_raw[i], c8, bias));
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
    CUtensorMap mq, mk, mv;
    const uint64_t rows = static_cast<uint64_t>(a.BH) * a.N;
    if (!make_tile_map(&mq, a.q8, rows) || !make_tile_map(&mk, a.k8, rows) || !make_tile_map(&mv, a.v_res, rows))
        return cudaErrorInvalidValue;
    Params p;
    p.sq = a.sq;
    p.sk = a.sk;
    p.v_scale = a.v_scale;
    p.v_mean = a.v_mean;
    p.O = a.O;
    p.dev_status = a.dev_status;
    p.N = a.N;
    p.scale_log2 = a.scale_log2;
    p.limit_ns = a.wait_limit_ns;
    const dim3 grid(a.N / kBlk, a.BH);
    cudaError_t e;
    if (a.expcast) {
        e = cudaFuncSetAttribute(attention_e4m3_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attention_e4m3_kernel<true><<<grid, kThreads, kSmemBytes, st>>>(mq, mk, mv, p);
    } else {
        e = cudaFuncSetAttribute(attention_e4m3_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attention_e4m3_kernel<false><<<grid, kThreads, kSmemBytes, st>>>(mq, mk, mv, p);
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
