// vca_group.cu -- V-Smooth "Group": per-(batch, head) k-means on the Value
// tokens and the stable permutation of the tokens by cluster label
// ("VC-Attention", paper page, section "method": online k-means per batch and
// head, then Key and Value are permuted together by cluster label).
//
// One Lloyd round is two launches:
//   assign  grid (chunks, BH): each CTA takes chunk_tokens tokens in 128-token
//           tiles (TMA, 128-byte swizzle), forms the tile's dot products with
//           all centroids on the tensor core (tcgen05, accumulators in TMEM),
//           assigns each token to its nearest centroid (|c|^2 - 2 v.c in fp32,
//           ties to the lowest index) and accumulates per-cluster sums and
//           counts of its tokens in a fixed order (no float atomics);
//   reduce  grid (k, BH): sums the chunk partials in chunk order and divides by
//           the count (an empty cluster keeps its centroid).
// V is read once per round (the HBM-bound part); the partials are small.
// After the last round, `scatter` turns labels into the stable permutation:
// slot = (tokens with a smaller label) + (same label, earlier chunk) + (same
// label, earlier in the chunk), the last term from warp match/ballot ranks.
#include "vca_device.cuh"
#include "vca_internal.h"

namespace vca {

namespace {

constexpr int kThreads = 192;          // warp 0 TMA, warp 1 MMA, warps 2-5 assign
constexpr uint32_t kTileBytes = kBlk * kD * 2;       // 128 tokens x 128 bf16 channels
constexpr uint32_t kPanelBytes = kTileBytes / 2;     // channels 0-63 or 64-127 of the tile

// Sum of x over the block's 128 threads (one value per channel), in a fixed
// order: a butterfly within each warp, then the four warp sums in order.
__device__ __forceinline__ float block_sum_128(float x, float *red4) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red4[threadIdx.x >> 5] = x;
    __syncthreads();
    return __fadd_rn(__fadd_rn(red4[0], red4[1]), __fadd_rn(red4[2], red4[3]));
}

// Centroid c starts at V row floor((c + 1/2) N / k); norm[c] = |C_c|^2.
__global__ void __launch_bounds__(kBlk) group_init_kernel(const uint16_t *V, int N, int k, float *C, float *norm) {
    __shared__ float red4[4];
    const int bh = blockIdx.x, ch = threadIdx.x;
    for (int c = 0; c < k; ++c) {
        const int64_t src = (static_cast<int64_t>(2 * c + 1) * N) / (2 * static_cast<int64_t>(k));
        const float x = bf16_bits_to_f32(V[(static_cast<int64_t>(bh) * N + src) * kD + ch]);
        C[(static_cast<int64_t>(bh) * k + c) * kD + ch] = x;
        const float n2 = block_sum_128(__fmul_rn(x, x), red4);
        if (ch == 0) norm[static_cast<int64_t>(bh) * k + c] = n2;
    }
}

// Shared-memory and TMEM layout of the assign kernel for up to KPAD centroids.
template <int KPAD>
struct AssignLayout {
    static constexpr int kStages = KPAD <= 64 ? 4 : 2;           // V tiles in flight
    static constexpr int kN = 2 * KPAD;                            // distance MMA N: centroid hi rows, then lo rows
    static constexpr int kDBufs = KPAD <= 64 ? 2 : 1;              // distance accumulators in TMEM
    static constexpr uint32_t kBPanel = kN * 128;                  // one 64-channel panel of the centroid operand
    static constexpr uint32_t kOhPanel = kBlk * 128;               // one-hot rows of 64 clusters for 128 tokens
    static constexpr uint32_t kOhBytes = (KPAD / 64) * kOhPanel;   // one tile's one-hot operand
    static constexpr uint32_t kOffV = 0;
    static constexpr uint32_t kOffB = kOffV + kStages * kTileBytes;
    static constexpr uint32_t kOffOh = kOffB + 2 * kBPanel;        // two one-hot buffers
    static constexpr uint32_t kOffNorm = kOffOh + 2 * kOhBytes;    // fp32 [KPAD]
    static constexpr uint32_t kOffCnt = kOffNorm + KPAD * 4;       // int [KPAD]
    static constexpr uint32_t kOffBar = kOffCnt + KPAD * 4;
    static constexpr int kNumBars = 2 * kStages + 2 * kDBufs + 4 + 1;   // v_full, v_empty; d_full, d_free; oh_full, oh_free; done
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kBytes = kOffMisc + 16 + 1024;
    static constexpr uint32_t kTmemSum = kDBufs * kN;              // cluster sums: KPAD columns, lane = channel
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kTmemSum + KPAD <= kTmemCols, "TMEM budget");
    static_assert(kOffB % 1024 == 0 && kBPanel % 1024 == 0 && kOffOh % 1024 == 0 && kOhPanel % 1024 == 0,
                  "swizzled operands need 1024-byte alignment");
    static_assert(kBytes <= 232448, "shared memory budget");
};

// One Lloyd round over a chunk of chunk_tokens tokens of one (batch, head):
// assign every token to its nearest centroid and accumulate the chunk's
// per-cluster sums and counts, both contractions on the tensor core
// (kind::f16, bf16 operands, fp32 accumulators in TMEM):
//   distances: D[token][j] = V_tile . [c_hi ; c_lo]^T.  V is exact in bf16 and
//              each centroid is split c = c_hi + c_lo into two bf16 rows, so
//              the dot product keeps ~16 bits of every centroid coordinate;
//   assign:    one thread per token reads its TMEM lane, |c_j|^2 - 2 (hi + lo)
//              in fp32, lowest index on ties, and writes the token's one-hot
//              row (bf16 1.0 at its label);
//   sums:      Sum[channel][j] += V_tile^T . onehot, the V tile read in place
//              as an MN-major operand; the products are exact and the chunk's
//              sums accumulate in TMEM over its tiles in a fixed order.
template <int KPAD>
__global__ void __launch_bounds__(kThreads, 1)
    group_assign_kernel(const __grid_constant__ CUtensorMap tmV, int N, int k, int nchunk, int chunk_tokens, const float *C,
                        const float *norm, int32_t *labels, float *part_sum, int32_t *part_cnt, int32_t *dev_status,
                        uint64_t limit_ns) {
    using L = AssignLayout<KPAD>;
    constexpr int S = L::kStages;
    constexpr int NB = L::kDBufs;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *sNorm = reinterpret_cast<float *>(smem + L::kOffNorm);
    int *sCnt = reinterpret_cast<int *>(smem + L::kOffCnt);
    uint64_t *v_full = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint64_t *v_empty = v_full + S;
    uint64_t *d_full = v_empty + S;
    uint64_t *d_free = d_full + NB;
    uint64_t *oh_full = d_free + NB;
    uint64_t *oh_free = oh_full + 2;
    uint64_t *done = oh_free + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    int *abort_flag = reinterpret_cast<int *>(smem + L::kOffMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = blockIdx.x, bh = blockIdx.y;
    const int tok0 = chunk * chunk_tokens;
    const int ntiles = min(chunk_tokens, N - tok0) / kBlk;
    const float *Cb = C + static_cast<int64_t>(bh) * k * kD;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(v_full + s, 1);
            mbar_init(v_empty + s, 1);    // the commit after the tile's sum MMA
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(d_full + i, 1);
            mbar_init(d_free + i, 4);     // the assign warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(oh_full + i, 4);    // the assign warps
            mbar_init(oh_free + i, 1);    // the commit after the tile's sum MMA
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    // centroid operand: row c = hi(c), row KPAD + c = lo(c), 8 channels per item
    for (int i = tid; i < KPAD * (kD / 8); i += kThreads) {
        const int c = i / (kD / 8), x0 = (i % (kD / 8)) * 8;
        float v[8];
        if (c < k) {
            const float4 a = *reinterpret_cast<const float4 *>(Cb + c * kD + x0);
            const float4 b = *reinterpret_cast<const float4 *>(Cb + c * kD + x0 + 4);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.0f;
        }
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_pack_bf16x2(v[2 * e], v[2 * e + 1], wh[e], wl[e]);
        unsigned char *panel = smem + L::kOffB + (x0 / 64) * L::kBPanel;
        const uint32_t chunk16 = (x0 % 64) / 8;
        *reinterpret_cast<uint4 *>(panel + sw128_offset(c, chunk16)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4 *>(panel + sw128_offset(KPAD + c, chunk16)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    }
    for (int c = tid; c < KPAD; c += kThreads) {
        sCnt[c] = 0;
        sNorm[c] = (c < k) ? norm[static_cast<int64_t>(bh) * k + c] : __int_as_float(0x7f800000);   // padding never wins
    }
    fence_proxy_async_smem();   // the centroid operand is read by the tensor core
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmV);
            int armed[S];
            for (int s = 0; s < S; ++s) armed[s] = 0;
            for (int i = 0; i < ntiles; ++i) {
                const int s = i % S, use = i / S;
                if (use > 0 && !mbar_wait(v_empty + s, (use - 1) & 1, abort_flag, limit_ns)) break;
                unsigned char *dst = smem + L::kOffV + s * kTileBytes;
                const int row = bh * N + tok0 + i * kBlk;
                mbar_expect_tx(v_full + s, kTileBytes);
                tma_load_2d(dst, &tmV, v_full + s, 0, row);
                tma_load_2d(dst + kPanelBytes, &tmV, v_full + s, 64, row);
                armed[s] = use + 1;
            }
            for (int s = 0; s < S; ++s)
                if (armed[s] > 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(v_full + s, (armed[s] - 1) & 1))
                        if (globaltimer_ns() - t0 > limit_ns) break;
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_dist = make_idesc(128, L::kN, 1, 1);        // bf16, both K-major
            constexpr uint32_t idesc_sum = make_idesc(128, KPAD, 1, 1, 1, 1);    // bf16, both MN-major
            const uint32_t sbase = smem_u32(smem);
            // distances of tile i into accumulator i % NB
            auto issue_dist = [&](int i) -> bool {
                const int s = i % S, buf = i % NB;
                if (!mbar_wait(v_full + s, (i / S) & 1, abort_flag, limit_ns)) return false;
                if (i >= NB && !mbar_wait(d_free + buf, ((i / NB) - 1) & 1, abort_flag, limit_ns)) return false;
                tc_fence_after();
                const uint32_t va = sbase + L::kOffV + s * kTileBytes;
                const uint32_t cb = sbase + L::kOffB;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    mma_f16(tmem + buf * L::kN, sdesc_k_sw128(va + (kk >> 2) * kPanelBytes) + 2 * (kk & 3),
                            sdesc_k_sw128(cb + (kk >> 2) * L::kBPanel) + 2 * (kk & 3), idesc_dist, kk > 0 ? 1u : 0u);
                tc_commit(d_full + buf);
                return true;
            };
            bool ok = ntiles > 0 && issue_dist(0);
            for (int i = 0; ok && i < ntiles; ++i) {
                if (i + 1 < ntiles && !issue_dist(i + 1)) break;
                const int s = i % S, ob = i & 1;
                if (!mbar_wait(oh_full + ob, (i >> 1) & 1, abort_flag, limit_ns)) break;
                tc_fence_after();
                // Sum[ch][j] += sum over the tile's tokens t of V[t][ch] onehot[t][j]
                const uint32_t va = sbase + L::kOffV + s * kTileBytes;
                const uint32_t oh = sbase + L::kOffOh + ob * L::kOhBytes;
#pragma unroll
                for (int kk = 0; kk < kBlk / 16; ++kk)
                    mma_f16(tmem + L::kTmemSum, sdesc_mn_sw128(va + kk * 2048, kPanelBytes),
                            sdesc_mn_sw128(oh + kk * 2048, L::kOhPanel), idesc_sum, (i > 0 || kk > 0) ? 1u : 0u);
                tc_commit(v_empty + s);
                tc_commit(oh_free + ob);
            }
            // every MMA this thread issued has finished: the sums are final
            tc_commit(done);
        }
    } else {
        // ------------------------------------------------------------ assign
        const int quarter = warp & 3;
        const int tok = quarter * 32 + lane;   // token in the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        bool ok = true;
        for (int i = 0; i < ntiles; ++i) {
            const int buf = i % NB, ob = i & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(d_full + buf, (i / NB) & 1, abort_flag, limit_ns));
            if (!ok) break;
            tc_fence_after();
            float best = __int_as_float(0x7f800000);
            int bi = 0;
#pragma unroll 1
            for (int c0 = 0; c0 < KPAD; c0 += 32) {
                uint32_t h[32], l[32];
                VCA_TMEM_LD32(tmem + lane_base + buf * L::kN + c0, h);
                VCA_TMEM_LD32(tmem + lane_base + buf * L::kN + KPAD + c0, l);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float dot = __fadd_rn(__uint_as_float(h[e]), __uint_as_float(l[e]));
                    const float dist = __fmaf_rn(-2.0f, dot, sNorm[c0 + e]);
                    if (dist < best) {
                        best = dist;
                        bi = c0 + e;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(d_free + buf);
            if (bi >= k) bi = 0;   // unreachable for finite inputs; keeps the label in range
            labels[static_cast<int64_t>(bh) * N + tok0 + i * kBlk + tok] = bi;
            atomicAdd(&sCnt[bi], 1);
            // the token's one-hot row, once the sum MMA of tile i-2 has read the buffer
            if (i >= 2) ok = __all_sync(0xffffffffu, mbar_wait(oh_free + ob, ((i >> 1) - 1) & 1, abort_flag, limit_ns));
            if (!ok) break;
            unsigned char *oh = smem + L::kOffOh + ob * L::kOhBytes;
#pragma unroll
            for (int j = 0; j < KPAD / 8; ++j) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if ((bi >> 3) == j) {
                    const uint32_t one = 0x3F80u << (16 * (bi & 1));   // bf16 1.0 in the label's half-word
                    const int word = (bi & 7) >> 1;
                    w.x = word == 0 ? one : 0u;
                    w.y = word == 1 ? one : 0u;
                    w.z = word == 2 ? one : 0u;
                    w.w = word == 3 ? one : 0u;
                }
                *reinterpret_cast<uint4 *>(oh + (j >> 3) * L::kOhPanel + sw128_offset(tok, j & 7)) = w;
            }
            fence_proxy_async_smem();   // the one-hot rows are read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(oh_full + ob);
        }
        // the chunk's sums: lane = channel, column j = cluster
        ok = __all_sync(0xffffffffu, ok && mbar_wait(done, 0, abort_flag, limit_ns));
        if (ok) {
            tc_fence_after();
            const int ch = quarter * 32 + lane;
            float *ps = part_sum + (static_cast<int64_t>(bh) * nchunk + chunk) * k * kD;
#pragma unroll 1
            for (int c0 = 0; c0 < KPAD; c0 += 32) {
                uint32_t v[32];
                VCA_TMEM_LD32(tmem + lane_base + L::kTmemSum + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (c0 + e < k) ps[(c0 + e) * kD + ch] = __uint_as_float(v[e]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // every MMA has finished before TMEM is freed (the assign warps waited
        // for `done` unless the CTA gave up; then wait here, bounded)
        if (lane == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(done, 0))
                if (globaltimer_ns() - t0 > limit_ns) break;
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
    const int64_t pbase = static_cast<int64_t>(bh) * nchunk + chunk;
    for (int i = tid; i < k; i += kThreads) part_cnt[pbase * k + i] = sCnt[i];
    if (tid == 0 && *reinterpret_cast<volatile int *>(abort_flag) && dev_status) atomicExch(dev_status, kErrTimeout);
}

__global__ void __launch_bounds__(kBlk) group_reduce_kernel(int k, int nchunk, const float *__restrict__ part_sum,
                                                            const int32_t *__restrict__ part_cnt,
                                                            float *__restrict__ C, float *__restrict__ norm,
                                                            int32_t *__restrict__ counts) {
    __shared__ float red4[4];
    const int c = blockIdx.x, bh = blockIdx.y, ch = threadIdx.x;
    float s = 0.0f;
    int n = 0;
    for (int j = 0; j < nchunk; ++j) {
        const int64_t pb = static_cast<int64_t>(bh) * nchunk + j;
        s = __fadd_rn(s, part_sum[(pb * k + c) * kD + ch]);
        n += part_cnt[pb * k + c];
    }
    float *cc = C + (static_cast<int64_t>(bh) * k + c) * kD + ch;
    const float x = (n > 0) ? __fdiv_rn(s, static_cast<float>(n)) : *cc;   // an empty cluster keeps its centroid
    *cc = x;
    const float n2 = block_sum_128(__fmul_rn(x, x), red4);
    if (ch == 0) {
        norm[static_cast<int64_t>(bh) * k + c] = n2;
        if (counts) counts[static_cast<int64_t>(bh) * k + c] = n;
    }
}

__global__ void __launch_bounds__(32) group_scatter_kernel(int N, int k, int nchunk, int chunk_tokens,
                                                           const int32_t *__restrict__ labels,
                                                           const int32_t *__restrict__ part_cnt,
                                                           int32_t *__restrict__ perm) {
    __shared__ int sBase[kMaxK];
    const int chunk = blockIdx.x, bh = blockIdx.y, lane = threadIdx.x;
    const int32_t *pc = part_cnt + static_cast<int64_t>(bh) * nchunk * k;
    for (int l = lane; l < k; l += 32) {
        int before = 0;   // tokens with a smaller label (all chunks)
        for (int j = 0; j < nchunk; ++j)
            for (int l2 = 0; l2 < l; ++l2) before += pc[j * k + l2];
        int earlier = 0;  // same label, earlier chunks
        for (int j = 0; j < chunk; ++j) earlier += pc[j * k + l];
        sBase[l] = before + earlier;
    }
    __syncwarp();
    const int tok0 = chunk * chunk_tokens;
    const int tok1 = min(N, tok0 + chunk_tokens);
    const int32_t *lab = labels + static_cast<int64_t>(bh) * N;
    int32_t *out = perm + static_cast<int64_t>(bh) * N;
    for (int t = tok0; t < tok1; t += 32) {
        const int l = lab[t + lane];
        const unsigned same = __match_any_sync(0xffffffffu, l);
        const int rank = __popc(same & ((1u << lane) - 1u));
        const int slot = sBase[l] + rank;
        __syncwarp();
        out[slot] = t + lane;
        if (rank == 0) sBase[l] += __popc(same);
        __syncwarp();
    }
}

// V as a 2-D bf16 matrix [rows][128] loaded in 64-channel x 128-token boxes
// with the 128-byte swizzle (the K-major A operand of the distance MMA).
bool make_v_map(CUtensorMap *map, const uint16_t *V, uint64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), rows};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlk)};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(V), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KPAD>
cudaError_t launch_assign(const CUtensorMap &tmV, int BH, int N, int k, int nchunk, int chunk_tokens, const float *C,
                          const float *norm, int32_t *labels, float *psum, int32_t *pcnt, int32_t *dev_status,
                          uint64_t limit_ns, cudaStream_t st) {
    constexpr uint32_t smem = AssignLayout<KPAD>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(group_assign_kernel<KPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    group_assign_kernel<KPAD><<<dim3(nchunk, BH), kThreads, smem, st>>>(tmV, N, k, nchunk, chunk_tokens, C, norm,
                                                                         labels, psum, pcnt, dev_status, limit_ns);
    return cudaGetLastError();
}

}  // namespace

// Chunks per head for the assign kernel: the count c that minimises the
// launch's modelled makespan, ceil(BH c / SMs) waves of ceil(tiles / c) + 6
// tile times each (6 for a CTA's fixed start-up -- centroid staging, the first
// V tile's latency -- and its drain of the partial sums), with at least 8
// tiles per chunk; ties go to fewer chunks.  For B=1, H=40, N=70,656 that is
// 7 chunks of 79 tiles (280 CTAs, two waves); measured there: 7 chunks
// 1.48 ms per group step, 11: 1.50, 15: 1.52, 18 (4096 tokens each, a fifth
// partly filled wave): 1.66.
constexpr int kSmCount = 152;
constexpr int kMinChunkTiles = 8;
constexpr int kChunkStartTiles = 6;
static int group_chunks_per_head(int BH, int tiles) {
    int best = 1;
    long best_cost = -1;
    for (int c = 1; c <= tiles; ++c) {
        const int per = (tiles + c - 1) / c;
        if (per < kMinChunkTiles && c > 1) break;
        if ((tiles + per - 1) / per != c) continue;   // c chunks of `per` tiles must all be non-empty
        const long waves = (static_cast<long>(BH) * c + kSmCount - 1) / kSmCount;
        const long cost = waves * (per + kChunkStartTiles);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = c;
        }
    }
    return best;
}

GroupWorkspace group_workspace_layout(int BH, int N, int k) {
    GroupWorkspace w;
    const int tiles = (N + kBlk - 1) / kBlk;
    const int c = group_chunks_per_head(BH, tiles);
    w.chunk_tokens = ((tiles + c - 1) / c) * kBlk;
    w.nchunk = (N + w.chunk_tokens - 1) / w.chunk_tokens;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += (bytes + 255) & ~size_t(255); return o; };
    w.off_centroids = take(sizeof(float) * BH * k * kD);
    w.off_norm = take(sizeof(float) * BH * k);
    w.off_psum = take(sizeof(float) * static_cast<size_t>(BH) * w.nchunk * k * kD);
    w.off_pcnt = take(sizeof(int32_t) * static_cast<size_t>(BH) * w.nchunk * k);
    w.bytes = off;
    return w;
}

cudaError_t launch_group(const uint16_t *V, int BH, int N, int k, int iters, int32_t *labels, int32_t *perm,
                         int32_t *counts, float *centroids, void *ws, int32_t *dev_status, uint64_t limit_ns,
                         cudaStream_t st) {
    const GroupWorkspace w = group_workspace_layout(BH, N, k);
    unsigned char *base = static_cast<unsigned char *>(ws);
    float *C = centroids ? centroids : reinterpret_cast<float *>(base + w.off_centroids);
    float *psum = reinterpret_cast<float *>(base + w.off_psum);
    int32_t *pcnt = reinterpret_cast<int32_t *>(base + w.off_pcnt);
    float *norm = reinterpret_cast<float *>(base + w.off_norm);

    CUtensorMap tmV;
    if (!make_v_map(&tmV, V, static_cast<uint64_t>(BH) * N)) return cudaErrorInvalidValue;
    group_init_kernel<<<BH, kBlk, 0, st>>>(V, N, k, C, norm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    for (int it = 0; it < iters; ++it) {
        e = (k <= 64)
                ? launch_assign<64>(tmV, BH, N, k, w.nchunk, w.chunk_tokens, C, norm, labels, psum, pcnt, dev_status,
                                    limit_ns, st)
                : launch_assign<128>(tmV, BH, N, k, w.nchunk, w.chunk_tokens, C, norm, labels, psum, pcnt, dev_status,
                                     limit_ns, st);
        if (e != cudaSuccess) return e;
        group_reduce_kernel<<<dim3(k, BH), kBlk, 0, st>>>(k, w.nchunk, psum, pcnt, C, norm, counts);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    group_scatter_kernel<<<dim3(w.nchunk, BH), 32, 0, st>>>(N, k, w.nchunk, w.chunk_tokens, labels, pcnt, perm);
    return cudaGetLastError();
}

}  // namespace vca
