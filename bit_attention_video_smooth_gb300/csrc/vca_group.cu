// vca_group.cu -- V-Smooth "Group": per-(batch, head) k-means on the Value
// tokens and the stable permutation of the tokens by cluster label
// ("VC-Attention", paper page, section "method": online k-means per batch and
// head, then Key and Value are permuted together by cluster label).
//
// One Lloyd round is two launches:
//   assign_update  grid (chunks, BH): each CTA takes kChunk tokens, assigns each
//                  to its nearest centroid (|c|^2 - 2 v.c in fp32, ties to the
//                  lowest index) and accumulates per-cluster sums and counts of
//                  its tokens in a fixed order (no float atomics);
//   reduce         grid (k, BH): sums the chunk partials in chunk order and
//                  divides by the count (an empty cluster keeps its centroid).
// V is read once per round (the HBM-bound part); the partials are small.
// After the last round, `scatter` turns labels into the stable permutation:
// slot = (tokens with a smaller label) + (same label, earlier chunk) + (same
// label, earlier in the chunk), the last term from warp match/ballot ranks.
#include "vca_device.cuh"
#include "vca_internal.h"

namespace vca {

namespace {

constexpr int kThreads = 256;
constexpr int kTilePad = 4;                    // bf16 pad per transposed row: keeps 8-byte row alignment
constexpr int kTileStride = kBlk + kTilePad;   // elements per channel row of the tile

__global__ void __launch_bounds__(kBlk) group_init_kernel(const uint16_t *__restrict__ V, int N, int k,
                                                          float *__restrict__ C) {
    const int bh = blockIdx.x, ch = threadIdx.x;
    for (int c = 0; c < k; ++c) {
        const int64_t src = (static_cast<int64_t>(2 * c + 1) * N) / (2 * static_cast<int64_t>(k));
        C[(static_cast<int64_t>(bh) * k + c) * kD + ch] =
            bf16_bits_to_f32(V[(static_cast<int64_t>(bh) * N + src) * kD + ch]);
    }
}

// Centroids per thread along the centroid axis: kpad / 8 (8 warps).
template <int CPT>
__global__ void __launch_bounds__(kThreads) group_assign_update_kernel(
    const uint16_t *__restrict__ V, int N, int k, int nchunk, const float *__restrict__ C,
    int32_t *__restrict__ labels, float *__restrict__ part_sum, int32_t *__restrict__ part_cnt) {
    constexpr int KPAD = CPT * 8;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *sC = reinterpret_cast<float *>(smem_raw);                    // [KPAD][kD]
    float *sSum = sC + KPAD * kD;                                       // [KPAD][kD]
    float *sNorm = sSum + KPAD * kD;                                    // [KPAD]
    float *sBestD = sNorm + KPAD;                                       // [8][kBlk]
    int *sBestI = reinterpret_cast<int *>(sBestD + 8 * kBlk);           // [8][kBlk]
    int *sLab = sBestI + 8 * kBlk;                                      // [kBlk]
    int *sCnt = sLab + kBlk;                                            // [KPAD]
    uint16_t *sV = reinterpret_cast<uint16_t *>(sCnt + KPAD);           // [kD][kTileStride] (transposed)

    const int tid = threadIdx.x;
    const int chunk = blockIdx.x, bh = blockIdx.y;
    const float *Cb = C + static_cast<int64_t>(bh) * k * kD;

    for (int i = tid; i < KPAD * kD; i += kThreads) {
        const int c = i / kD;
        sC[i] = (c < k) ? Cb[i] : 0.0f;
        sSum[i] = 0.0f;
    }
    for (int i = tid; i < KPAD; i += kThreads) sCnt[i] = 0;
    __syncthreads();
    if (tid < KPAD) {
        float s = 0.0f;
        for (int x = 0; x < kD; ++x) s = __fmaf_rn(sC[tid * kD + x], sC[tid * kD + x], s);
        sNorm[tid] = (tid < k) ? s : __int_as_float(0x7f800000);   // padded centroids never win
    }

    const int tok0 = chunk * kChunkTokens;
    const int ntiles = min(kChunkTokens, N - tok0) / kBlk;
    const int tg = tid & 31;          // token group: tokens 4*tg .. 4*tg+3
    const int cg = tid >> 5;          // centroid group: centroids CPT*cg .. CPT*cg+CPT-1

    for (int tile = 0; tile < ntiles; ++tile) {
        const int t0 = tok0 + tile * kBlk;
        __syncthreads();   // previous tile fully consumed
        // load 128 tokens x 128 channels, transposed into sV[ch][tok]
        const uint4 *src = reinterpret_cast<const uint4 *>(V + (static_cast<int64_t>(bh) * N + t0) * kD);
        for (int u = tid; u < kBlk * kD / 8; u += kThreads) {
            const int t = u >> 4, c8 = (u & 15) * 8;
            const uint4 val = src[u];
            const uint16_t *h = reinterpret_cast<const uint16_t *>(&val);
#pragma unroll
            for (int j = 0; j < 8; ++j) sV[(c8 + j) * kTileStride + t] = h[j];
        }
        __syncthreads();

        // dot products for 4 tokens x CPT centroids
        float acc[4][CPT];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < CPT; ++j) acc[i][j] = 0.0f;
#pragma unroll 4
        for (int x = 0; x < kD; ++x) {
            const uint2 vv = *reinterpret_cast<const uint2 *>(&sV[x * kTileStride + 4 * tg]);
            const float v0 = __uint_as_float(vv.x << 16), v1 = __uint_as_float(vv.x & 0xFFFF0000u);
            const float v2 = __uint_as_float(vv.y << 16), v3 = __uint_as_float(vv.y & 0xFFFF0000u);
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                const float c = sC[(cg * CPT + j) * kD + x];
                acc[0][j] = __fmaf_rn(v0, c, acc[0][j]);
                acc[1][j] = __fmaf_rn(v1, c, acc[1][j]);
                acc[2][j] = __fmaf_rn(v2, c, acc[2][j]);
                acc[3][j] = __fmaf_rn(v3, c, acc[3][j]);
            }
        }
        // local argmin of |c|^2 - 2 v.c, lowest index on ties
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float best = __int_as_float(0x7f800000);
            int bi = 0x7fffffff;
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                const float dist = __fmaf_rn(-2.0f, acc[i][j], sNorm[cg * CPT + j]);
                if (dist < best) { best = dist; bi = cg * CPT + j; }
            }
            sBestD[cg * kBlk + 4 * tg + i] = best;
            sBestI[cg * kBlk + 4 * tg + i] = bi;
        }
        __syncthreads();
        if (tid < kBlk) {
            float best = sBestD[tid];
            int bi = sBestI[tid];
            for (int g = 1; g < 8; ++g) {
                const float dd = sBestD[g * kBlk + tid];
                if (dd < best) { best = dd; bi = sBestI[g * kBlk + tid]; }
            }
            if (bi >= k) bi = 0;   // unreachable for finite inputs; keeps the label in range
            sLab[tid] = bi;
            labels[static_cast<int64_t>(bh) * N + t0 + tid] = bi;
            atomicAdd(&sCnt[bi], 1);
        }
        __syncthreads();
        // per-cluster sums, channel per thread, tokens in order (deterministic)
        if (tid < kD) {
            const uint16_t *row = sV + tid * kTileStride;
            for (int t = 0; t < kBlk; ++t) {
                float *dst = &sSum[sLab[t] * kD + tid];
                *dst = __fadd_rn(*dst, bf16_bits_to_f32(row[t]));
            }
        }
    }
    __syncthreads();
    const int64_t pbase = (static_cast<int64_t>(bh) * nchunk + chunk);
    for (int i = tid; i < k * kD; i += kThreads) part_sum[pbase * k * kD + i] = sSum[i];
    for (int i = tid; i < k; i += kThreads) part_cnt[pbase * k + i] = sCnt[i];
}

__global__ void __launch_bounds__(kBlk) group_reduce_kernel(int k, int nchunk, const float *__restrict__ part_sum,
                                                            const int32_t *__restrict__ part_cnt,
                                                            float *__restrict__ C, int32_t *__restrict__ counts) {
    const int c = blockIdx.x, bh = blockIdx.y, ch = threadIdx.x;
    float s = 0.0f;
    int n = 0;
    for (int j = 0; j < nchunk; ++j) {
        const int64_t pb = static_cast<int64_t>(bh) * nchunk + j;
        s = __fadd_rn(s, part_sum[(pb * k + c) * kD + ch]);
        n += part_cnt[pb * k + c];
    }
    if (n > 0) C[(static_cast<int64_t>(bh) * k + c) * kD + ch] = __fdiv_rn(s, static_cast<float>(n));
    if (ch == 0 && counts) counts[static_cast<int64_t>(bh) * k + c] = n;
}

__global__ void __launch_bounds__(32) group_scatter_kernel(int N, int k, int nchunk,
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
    const int tok0 = chunk * kChunkTokens;
    const int tok1 = min(N, tok0 + kChunkTokens);
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

template <int CPT>
size_t assign_smem_bytes() {
    constexpr int KPAD = CPT * 8;
    return sizeof(float) * (2 * KPAD * kD + KPAD + 8 * kBlk) + sizeof(int) * (8 * kBlk + kBlk + KPAD) +
           sizeof(uint16_t) * kD * kTileStride;
}

template <int CPT>
cudaError_t launch_assign(const uint16_t *V, int BH, int N, int k, int nchunk, const float *C, int32_t *labels,
                          float *psum, int32_t *pcnt, cudaStream_t st) {
    const size_t smem = assign_smem_bytes<CPT>();
    cudaError_t e = cudaFuncSetAttribute(group_assign_update_kernel<CPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    group_assign_update_kernel<CPT><<<dim3(nchunk, BH), kThreads, smem, st>>>(V, N, k, nchunk, C, labels, psum, pcnt);
    return cudaGetLastError();
}

}  // namespace

GroupWorkspace group_workspace_layout(int BH, int N, int k) {
    GroupWorkspace w;
    w.nchunk = (N + kChunkTokens - 1) / kChunkTokens;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += (bytes + 255) & ~size_t(255); return o; };
    w.off_centroids = take(sizeof(float) * BH * k * kD);
    w.off_psum = take(sizeof(float) * static_cast<size_t>(BH) * w.nchunk * k * kD);
    w.off_pcnt = take(sizeof(int32_t) * static_cast<size_t>(BH) * w.nchunk * k);
    w.bytes = off;
    return w;
}

cudaError_t launch_group(const uint16_t *V, int BH, int N, int k, int iters, int32_t *labels, int32_t *perm,
                         int32_t *counts, float *centroids, void *ws, cudaStream_t st) {
    const GroupWorkspace w = group_workspace_layout(BH, N, k);
    unsigned char *base = static_cast<unsigned char *>(ws);
    float *C = centroids ? centroids : reinterpret_cast<float *>(base + w.off_centroids);
    float *psum = reinterpret_cast<float *>(base + w.off_psum);
    int32_t *pcnt = reinterpret_cast<int32_t *>(base + w.off_pcnt);

    group_init_kernel<<<BH, kBlk, 0, st>>>(V, N, k, C);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int kpad8 = (k + 7) / 8;   // centroids per thread
    for (int it = 0; it < iters; ++it) {
        if (kpad8 <= 1) e = launch_assign<1>(V, BH, N, k, w.nchunk, C, labels, psum, pcnt, st);
        else if (kpad8 <= 2) e = launch_assign<2>(V, BH, N, k, w.nchunk, C, labels, psum, pcnt, st);
        else if (kpad8 <= 4) e = launch_assign<4>(V, BH, N, k, w.nchunk, C, labels, psum, pcnt, st);
        else if (kpad8 <= 8) e = launch_assign<8>(V, BH, N, k, w.nchunk, C, labels, psum, pcnt, st);
        else e = launch_assign<16>(V, BH, N, k, w.nchunk, C, labels, psum, pcnt, st);
        if (e != cudaSuccess) return e;
        group_reduce_kernel<<<dim3(k, BH), kBlk, 0, st>>>(k, w.nchunk, psum, pcnt, C, counts);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    group_scatter_kernel<<<dim3(w.nchunk, BH), 32, 0, st>>>(N, k, w.nchunk, labels, pcnt, perm);
    return cudaGetLastError();
}

}  // namespace vca
