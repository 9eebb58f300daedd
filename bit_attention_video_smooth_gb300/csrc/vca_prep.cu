// vca_prep.cu -- the fused V-Smooth prep ("VC-Attention", paper page, section
// "method": each 128-token hardware block subtracts its own mean, stored as a
// 16-bit vector, and only the residual is quantised -- per-channel E4M3 for the
// 8-bit path, NVFP4 for the 4-bit path; the preprocessing chain is fused so no
// high-precision intermediate goes back to device memory).
//
// A per-channel residual scale over the whole sequence needs the sequence-wide
// amax before any residual byte can be written, so the prep is three launches:
//   prep_stats  grid (nb, BH): Q and K blocks (K gathered by perm) -> FP8 with a
//               per-block absmax scale; the gathered V block -> its bf16 mean and
//               the per-channel amax of the residual (a small partial);
//   prep_scale  grid (BH): reduce the partials -> per-channel scales (E4M3) or
//               the per-(b,h) scale (NVFP4);
//   prep_vquant grid (nb, BH): gather V again (L2-resident when a head's blocks
//               run close together), subtract the stored mean, quantise, and
//               write the residual channel-major (tokens contiguous per channel,
//               the K-major operand layout of the PV contraction).
// With K smoothing (SageAttention's treatment of the keys' channel bias: the
// channel mean of K over the sequence is subtracted, which moves every score
// of a query row by the same amount) the K quantisation moves to prep_vquant:
// prep_stats writes each permuted block's channel sums, prep_scale adds them
// in block order into the mean, prep_vquant quantises K - mean.
#include "vca_device.cuh"
#include "vca_internal.h"

namespace vca {

namespace {

constexpr int kThreads = 256;
constexpr int kRowPad = 8;                      // bf16 pad per token row of the V tile
constexpr int kRowStride = kD + kRowPad;

__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float r = red[0];
    for (int i = 1; i < kThreads / 32; ++i) r = fmaxf(r, red[i]);
    return r;
}

// Quantise one 128 x 128 bf16 block (rows given by `rows`, or contiguous from
// `row0` when rows == nullptr) to E4M3 with the block's absmax scale.  With
// kShift every value first has its channel's shift[c] subtracted (one fp32
// rounding): the K smoothing.
template <bool kShift>
__device__ __forceinline__ float qk_value(uint32_t w, int half, int c, const float *shift) {
    const float x = __uint_as_float(half ? (w & 0xFFFF0000u) : (w << 16));
    if constexpr (kShift) return __fsub_rn(x, shift[c]);
    return x;
}

template <bool kShift>
__device__ __forceinline__ void quant_qk_block(const uint16_t *__restrict__ X, int64_t head_row0,
                                               const int32_t *__restrict__ rows, int row0, const float *shift,
                                               uint8_t *__restrict__ out, float *__restrict__ scale, float *red) {
    const int tid = threadIdx.x;
    uint4 v[8];
    float amax = 0.0f;
    const int c8 = (tid & 15) * 8;   // this thread's 8 channels (the same for every i)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int u = i * kThreads + tid;
        const int r = u >> 4;
        const int64_t src = head_row0 + (rows ? rows[r] : row0 + r);
        v[i] = *reinterpret_cast<const uint4 *>(X + src * kD + c8);
        const uint32_t *w = reinterpret_cast<const uint32_t *>(&v[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            amax = fmaxf(amax, fabsf(qk_value<kShift>(w[j], 0, c8 + 2 * j, shift)));
            amax = fmaxf(amax, fabsf(qk_value<kShift>(w[j], 1, c8 + 2 * j + 1, shift)));
        }
    }
    amax = block_max(amax, red);
    float inv = 1.0f, s = 1.0f;
    if (amax > 0.0f) {
        inv = __fdiv_rn(448.0f, amax);
        s = __fdiv_rn(amax, 448.0f);
    }
    if (tid == 0) *scale = s;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int u = i * kThreads + tid;
        const uint32_t *w = reinterpret_cast<const uint32_t *>(&v[i]);
        uint32_t packed[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = c8 + 4 * j;
            packed[j] = e4m3x4(__fmul_rn(qk_value<kShift>(w[2 * j], 0, c, shift), inv),
                               __fmul_rn(qk_value<kShift>(w[2 * j], 1, c + 1, shift), inv),
                               __fmul_rn(qk_value<kShift>(w[2 * j + 1], 0, c + 2, shift), inv),
                               __fmul_rn(qk_value<kShift>(w[2 * j + 1], 1, c + 3, shift), inv));
        }
        *reinterpret_cast<uint2 *>(out + static_cast<int64_t>(u) * 8) = make_uint2(packed[0], packed[1]);
    }
}

// The same block after rotating every row by the unnormalised 128-point
// Walsh-Hadamard transform (the QK Hadamard option): fp32 butterflies in the
// fixed order bit 0, 1, ..., 6 of the channel index, each pair (c, c + 2^k)
// with bit k clear becoming (a + b, a - b).  A row's 128 channels sit in 16
// consecutive lanes, 8 per lane: bits 0-2 are butterflied in registers, bits
// 3-6 (the lane's bits 0-3) across lanes.  The stored scale is amax / 448
// times `post` (a power of two: 1 for Q, 1/128 for K, so that sq sk q8 . k8
// still approximates q . k).  With kShift the channel shift (K smoothing) is
// subtracted before the rotation.
template <bool kShift>
__device__ __forceinline__ void quant_qk_block_hadamard(const uint16_t *__restrict__ X, int64_t head_row0,
                                                        const int32_t *__restrict__ rows, int row0, float post,
                                                        const float *shift, uint8_t *__restrict__ out,
                                                        float *__restrict__ scale, float *red) {
    const int tid = threadIdx.x, lane = tid & 31;
    float x[8][8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int u = i * kThreads + tid;
        const int r = u >> 4, c8 = (u & 15) * 8;
        const int64_t src = head_row0 + (rows ? rows[r] : row0 + r);
        const uint4 v = *reinterpret_cast<const uint4 *>(X + src * kD + c8);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[i][2 * j] = qk_value<kShift>(w[j], 0, c8 + 2 * j, shift);
            x[i][2 * j + 1] = qk_value<kShift>(w[j], 1, c8 + 2 * j + 1, shift);
        }
#pragma unroll
        for (int h = 1; h < 8; h <<= 1)
#pragma unroll
            for (int c = 0; c < 8; ++c)
                if (!(c & h)) {
                    const float a = x[i][c], b = x[i][c + h];
                    x[i][c] = __fadd_rn(a, b);
                    x[i][c + h] = __fsub_rn(a, b);
                }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const bool upper = (lane >> m) & 1;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float y = __shfl_xor_sync(0xffffffffu, x[i][c], 1 << m);
                x[i][c] = upper ? __fsub_rn(y, x[i][c]) : __fadd_rn(x[i][c], y);
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) amax = fmaxf(amax, fabsf(x[i][c]));
    }
    amax = block_max(amax, red);
    float inv = 1.0f, s = 1.0f;
    if (amax > 0.0f) {
        inv = __fdiv_rn(448.0f, amax);
        s = __fdiv_rn(amax, 448.0f);
    }
    if (tid == 0) *scale = __fmul_rn(s, post);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int u = i * kThreads + tid;
        const uint32_t lo = e4m3x4(__fmul_rn(x[i][0], inv), __fmul_rn(x[i][1], inv), __fmul_rn(x[i][2], inv),
                                   __fmul_rn(x[i][3], inv));
        const uint32_t hi = e4m3x4(__fmul_rn(x[i][4], inv), __fmul_rn(x[i][5], inv), __fmul_rn(x[i][6], inv),
                                   __fmul_rn(x[i][7], inv));
        *reinterpret_cast<uint2 *>(out + static_cast<int64_t>(u) * 8) = make_uint2(lo, hi);
    }
}

// K smoothing: the channel sums of one permuted 128-token K block in a fixed
// fp32 order, a halving tree (token i plus token i + 64 for i < 64, then
// i + 32, ..., i + 1).  Thread (t16 = tid / 16) holds tokens 16 i + t16 of
// eight channels, so the first three levels stay in its registers
// ((x_0 + x_4) + (x_2 + x_6)) + ((x_1 + x_5) + (x_3 + x_7)) over its i = 0..7;
// the last four (over t16) run per channel from shared memory.
__device__ __forceinline__ void k_block_tree_sums(const uint16_t *__restrict__ K, int64_t head_row0,
                                                  const int32_t *__restrict__ rows, float *sPart,
                                                  float *__restrict__ out) {
    const int tid = threadIdx.x, t16 = tid >> 4, c8 = (tid & 15) * 8;
    float x[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = *reinterpret_cast<const uint4 *>(K + (head_row0 + rows[16 * i + t16]) * kD + c8);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[i][2 * j] = __uint_as_float(w[j] << 16);
            x[i][2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float a0 = __fadd_rn(x[0][c], x[4][c]), a1 = __fadd_rn(x[1][c], x[5][c]);
        const float a2 = __fadd_rn(x[2][c], x[6][c]), a3 = __fadd_rn(x[3][c], x[7][c]);
        sPart[t16 * kD + c8 + c] = __fadd_rn(__fadd_rn(a0, a2), __fadd_rn(a1, a3));
    }
    __syncthreads();
    if (tid < kD) {
        float p[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) p[t] = sPart[t * kD + tid];
#pragma unroll
        for (int h = 8; h >= 1; h >>= 1)
#pragma unroll
            for (int t = 0; t < h; ++t) p[t] = __fadd_rn(p[t], p[t + h]);
        out[tid] = p[0];
    }
}

// Gather the block's 128 V rows into shared memory (token-major, padded rows)
// as asynchronous 16-byte copies (cp.async): all of a thread's copies are in
// flight at once, and the gather can run while the thread works on something
// else; cp_async_wait_all() + a barrier before the tile is read.
__device__ __forceinline__ void load_v_tile_async(const uint16_t *__restrict__ V, int64_t head_row0,
                                                  const int32_t *__restrict__ rows, uint16_t *sV) {
    for (int u = threadIdx.x; u < kBlk * kD / 8; u += kThreads) {
        const int r = u >> 4, c8 = (u & 15) * 8;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sV + r * kRowStride + c8)),
                     "l"(V + (head_row0 + rows[r]) * kD + c8)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Error-free transformation: a + b = s + e exactly (Knuth's two-sum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

template <bool kHadamard, bool kSmooth>
__global__ void __launch_bounds__(kThreads) prep_stats_kernel(const uint16_t *__restrict__ Q,
                                                              const uint16_t *__restrict__ K,
                                                              const uint16_t *__restrict__ V,
                                                              const int32_t *__restrict__ perm, int N,
                                                              uint8_t *__restrict__ q8, float *__restrict__ sq,
                                                              uint8_t *__restrict__ k8, float *__restrict__ sk,
                                                              uint16_t *__restrict__ v_mean,
                                                              float *__restrict__ amax_part,
                                                              float *__restrict__ ksum) {
    // the V tile, then 2 x 2 x 128 floats of per-half partial results
    __shared__ __align__(16) uint16_t sV[kBlk * kRowStride + 4 * kD * 2];
    __shared__ float red[kThreads / 32];
    const int b = blockIdx.x, bh = blockIdx.y, nb = gridDim.x;
    const int64_t head_row0 = static_cast<int64_t>(bh) * N;
    const int32_t *rows = perm + head_row0 + static_cast<int64_t>(b) * kBlk;
    const int64_t blk_off = (head_row0 + static_cast<int64_t>(b) * kBlk) * kD;

    // V's gather runs in the background while Q and K are quantised (K, with
    // smoothing, waits for the sequence's mean: here only its block sums)
    load_v_tile_async(V, head_row0, rows, sV);
    if constexpr (kHadamard)
        quant_qk_block_hadamard<false>(Q, head_row0, nullptr, b * kBlk, 1.0f, nullptr, q8 + blk_off,
                                       sq + static_cast<int64_t>(bh) * nb + b, red);
    else
        quant_qk_block<false>(Q, head_row0, nullptr, b * kBlk, nullptr, q8 + blk_off,
                              sq + static_cast<int64_t>(bh) * nb + b, red);
    if constexpr (kSmooth) {
        __shared__ float sPart[16 * kD];
        k_block_tree_sums(K, head_row0, rows, sPart, ksum + (static_cast<int64_t>(bh) * nb + b) * kD);
    } else if constexpr (kHadamard) {
        quant_qk_block_hadamard<false>(K, head_row0, rows, 0, 1.0f / kD, nullptr, k8 + blk_off,
                                       sk + static_cast<int64_t>(bh) * nb + b, red);
    } else {
        quant_qk_block<false>(K, head_row0, rows, 0, nullptr, k8 + blk_off, sk + static_cast<int64_t>(bh) * nb + b,
                              red);
    }
    cp_async_wait_all();
    __syncthreads();

    // Thread (ch, g) takes tokens 64g .. 64g+63 of channel ch: four compensated
    // (two-sum) partial sums over interleaved tokens, merged in a fixed order;
    // the two halves meet in shared memory.  The mean is fp32(sum) / 128 ->
    // bf16, the residual amax max |v - mean| over the block.
    const int ch = threadIdx.x & (kD - 1), g = threadIdx.x >> 7;
    const uint16_t *col = sV + (g * 64) * kRowStride + ch;
    float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
    for (int t = 0; t < 64; t += 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float e;
            two_sum(s4[k], bf16_bits_to_f32(col[(t + k) * kRowStride]), s4[k], e);
            c4[k] = __fadd_rn(c4[k], e);
        }
    }
    float sh, ch_c;
    {
        float e0, e1, e2;
        float s01, s23;
        two_sum(s4[0], s4[1], s01, e0);
        two_sum(s4[2], s4[3], s23, e1);
        two_sum(s01, s23, sh, e2);
        ch_c = __fadd_rn(__fadd_rn(__fadd_rn(c4[0], c4[1]), __fadd_rn(c4[2], c4[3])), __fadd_rn(__fadd_rn(e0, e1), e2));
    }
    float *sHalf = reinterpret_cast<float *>(sV + kBlk * kRowStride);   // [2][128] sums, [2][128] compensations
    __shared__ float sMu[kD];
    if (g == 1) {
        sHalf[ch] = sh;
        sHalf[kD + ch] = ch_c;
    }
    __syncthreads();
    if (g == 0) {
        float s, e;
        two_sum(sh, sHalf[ch], s, e);
        const float comp = __fadd_rn(__fadd_rn(ch_c, sHalf[kD + ch]), e);
        const float mean = __fdiv_rn(__fadd_rn(s, comp), 128.0f);
        const __nv_bfloat16 mu = __float2bfloat16_rn(mean);
        v_mean[(static_cast<int64_t>(bh) * nb + b) * kD + ch] = __bfloat16_as_ushort(mu);
        sMu[ch] = __bfloat162float(mu);
    }
    __syncthreads();
    const float muf = sMu[ch];
    float a4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
    for (int t = 0; t < 64; t += 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            a4[k] = fmaxf(a4[k], fabsf(__fsub_rn(bf16_bits_to_f32(col[(t + k) * kRowStride]), muf)));
    }
    const float a = fmaxf(fmaxf(a4[0], a4[1]), fmaxf(a4[2], a4[3]));
    if (g == 1) sHalf[ch] = a;
    __syncthreads();
    if (g == 0) amax_part[(static_cast<int64_t>(bh) * nb + b) * kD + ch] = fmaxf(a, sHalf[ch]);
}

// E4M3: per channel a_c -> v_scale = a_c / 448, inv_c = 448 / a_c.
// NVFP4: g = max_c a_c / (6 * 448) -> v_scale[bh]; inv[bh][0] = 6 g, inv[bh][1] = g.
// K smoothing (ksum != nullptr): the channel mean of K = the block sums added
// in block order, divided by N (fp32).
__global__ void __launch_bounds__(kD) prep_scale_kernel(int nb, int vmode, const float *__restrict__ amax_part,
                                                        float *__restrict__ v_scale, float *__restrict__ inv,
                                                        const float *__restrict__ ksum, float *__restrict__ kmean,
                                                        int N) {
    __shared__ float red[kD / 32];
    const int bh = blockIdx.x, ch = threadIdx.x;
    if (ksum) {
        float total = 0.0f;
        for (int b = 0; b < nb; ++b) total = __fadd_rn(total, ksum[(static_cast<int64_t>(bh) * nb + b) * kD + ch]);
        kmean[static_cast<int64_t>(bh) * kD + ch] = __fdiv_rn(total, static_cast<float>(N));
    }
    float a = 0.0f;
    for (int b = 0; b < nb; ++b) a = fmaxf(a, amax_part[(static_cast<int64_t>(bh) * nb + b) * kD + ch]);
    if (vmode == 0) {
        float s = 1.0f, iv = 1.0f;
        if (a > 0.0f) { s = __fdiv_rn(a, 448.0f); iv = __fdiv_rn(448.0f, a); }
        v_scale[static_cast<int64_t>(bh) * kD + ch] = s;
        inv[static_cast<int64_t>(bh) * kD + ch] = iv;
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if ((ch & 31) == 0) red[ch >> 5] = a;
        __syncthreads();
        if (ch == 0) {
            float m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
            const float g = (m > 0.0f) ? __fdiv_rn(m, 2688.0f) : 1.0f;   // 6 * 448
            v_scale[bh] = g;
            inv[static_cast<int64_t>(bh) * kD + 0] = __fmul_rn(6.0f, g);
            inv[static_cast<int64_t>(bh) * kD + 1] = g;
        }
    }
}

template <bool kSmooth, bool kHadamard>
__global__ void __launch_bounds__(kThreads) prep_vquant_kernel(const uint16_t *__restrict__ V,
                                                               const int32_t *__restrict__ perm, int N, int vmode,
                                                               const uint16_t *__restrict__ v_mean,
                                                               const float *__restrict__ inv,
                                                               uint8_t *__restrict__ v_res,
                                                               uint8_t *__restrict__ v_sf,
                                                               const uint16_t *__restrict__ K,
                                                               const float *__restrict__ kmean,
                                                               uint8_t *__restrict__ k8, float *__restrict__ sk) {
    __shared__ __align__(16) uint16_t sV[kBlk * kRowStride];
    const int b = blockIdx.x, bh = blockIdx.y, nb = gridDim.x;
    const int64_t head_row0 = static_cast<int64_t>(bh) * N;
    const int32_t *rows = perm + head_row0 + static_cast<int64_t>(b) * kBlk;
    load_v_tile_async(V, head_row0, rows, sV);
    if constexpr (kSmooth) {
        // K smoothing: the permuted K block minus the channel mean, quantised
        // while V's gather is in flight
        __shared__ float sShift[kD];
        __shared__ float red[kThreads / 32];
        if (threadIdx.x < kD) sShift[threadIdx.x] = kmean[static_cast<int64_t>(bh) * kD + threadIdx.x];
        __syncthreads();
        const int64_t blk_off = (head_row0 + static_cast<int64_t>(b) * kBlk) * kD;
        if constexpr (kHadamard)
            quant_qk_block_hadamard<true>(K, head_row0, rows, 0, 1.0f / kD, sShift, k8 + blk_off,
                                          sk + static_cast<int64_t>(bh) * nb + b, red);
        else
            quant_qk_block<true>(K, head_row0, rows, 0, sShift, k8 + blk_off, sk + static_cast<int64_t>(bh) * nb + b,
                                 red);
    }
    cp_async_wait_all();
    __syncthreads();
    const int ch = threadIdx.x & (kD - 1);
    const int half = threadIdx.x >> 7;                  // tokens 64*half .. 64*half+63
    const float muf = bf16_bits_to_f32(v_mean[(static_cast<int64_t>(bh) * nb + b) * kD + ch]);
    const int64_t cb = (static_cast<int64_t>(bh) * nb + b) * kD + ch;   // (block, channel) index
    if (vmode == 0) {
        const float iv = inv[static_cast<int64_t>(bh) * kD + ch];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int t0 = half * 64 + g * 16;
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float r[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    r[q] = __fmul_rn(__fsub_rn(bf16_bits_to_f32(sV[(t0 + 4 * j + q) * kRowStride + ch]), muf), iv);
                w[j] = e4m3x4(r[0], r[1], r[2], r[3]);
            }
            *reinterpret_cast<uint4 *>(v_res + cb * kBlk + t0) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        const float g6 = inv[static_cast<int64_t>(bh) * kD + 0];
        const float gs = inv[static_cast<int64_t>(bh) * kD + 1];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int t0 = half * 64 + g * 16;
            float r[16];
            float a16 = 0.0f;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                r[q] = __fsub_rn(bf16_bits_to_f32(sV[(t0 + q) * kRowStride + ch]), muf);
                a16 = fmaxf(a16, fabsf(r[q]));
            }
            const uint32_t sf = e4m3(__fdiv_rn(a16, g6));
            float iv = 0.0f;
            if (sf != 0) iv = __fdiv_rn(1.0f, __fmul_rn(e4m3_to_f32(sf), gs));
            uint32_t w[2];
            const uint64_t iv2 = pk2(__float_as_uint(iv), __float_as_uint(iv));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float x[8];
#pragma unroll
                for (int q = 0; q < 8; q += 2)
                    upk2(mul2(pk2(__float_as_uint(r[8 * h + q]), __float_as_uint(r[8 * h + q + 1])), iv2), x[q], x[q + 1]);
                w[h] = e2m1x8(x);
            }
            *reinterpret_cast<uint2 *>(v_res + cb * (kBlk / 2) + t0 / 2) = make_uint2(w[0], w[1]);
            v_sf[cb * (kBlk / 16) + t0 / 16] = static_cast<uint8_t>(sf);
        }
    }
}

}  // namespace

PrepWorkspace prep_workspace_layout(int BH, int N, uint32_t flags) {
    PrepWorkspace w;
    const size_t nb = static_cast<size_t>(N) / kBlk;
    const size_t per_block = (sizeof(float) * BH * nb * kD + 255) & ~size_t(255);
    const size_t per_head = (sizeof(float) * BH * kD + 255) & ~size_t(255);
    w.off_amax = 0;
    w.off_inv = per_block;
    w.bytes = per_block + per_head;
    w.off_ksum = w.off_kmean = 0;
    if (flags & kPrepKSmooth) {   // the K block sums and the K mean
        w.off_ksum = w.bytes;
        w.off_kmean = w.off_ksum + per_block;
        w.bytes = w.off_kmean + per_head;
    }
    return w;
}

cudaError_t launch_prep(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *perm, int BH, int N,
                        int vmode, uint32_t flags, uint8_t *q8, float *sq, uint8_t *k8, float *sk, uint8_t *v_res,
                        uint8_t *v_sf, float *v_scale, uint16_t *v_mean, void *ws, cudaStream_t st) {
    const PrepWorkspace w = prep_workspace_layout(BH, N, flags);
    unsigned char *base = static_cast<unsigned char *>(ws);
    float *amax = reinterpret_cast<float *>(base + w.off_amax);
    float *inv = reinterpret_cast<float *>(base + w.off_inv);
    const bool smooth = (flags & kPrepKSmooth) != 0, had = (flags & kPrepQkHadamard) != 0;
    float *ksum = smooth ? reinterpret_cast<float *>(base + w.off_ksum) : nullptr;
    float *kmean = smooth ? reinterpret_cast<float *>(base + w.off_kmean) : nullptr;
    const int nb = N / kBlk;
    const dim3 grid(nb, BH);
    if (had && smooth)
        prep_stats_kernel<true, true><<<grid, kThreads, 0, st>>>(Q, K, V, perm, N, q8, sq, k8, sk, v_mean, amax, ksum);
    else if (had)
        prep_stats_kernel<true, false><<<grid, kThreads, 0, st>>>(Q, K, V, perm, N, q8, sq, k8, sk, v_mean, amax, ksum);
    else if (smooth)
        prep_stats_kernel<false, true><<<grid, kThreads, 0, st>>>(Q, K, V, perm, N, q8, sq, k8, sk, v_mean, amax, ksum);
    else
        prep_stats_kernel<false, false><<<grid, kThreads, 0, st>>>(Q, K, V, perm, N, q8, sq, k8, sk, v_mean, amax, ksum);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prep_scale_kernel<<<BH, kD, 0, st>>>(nb, vmode, amax, v_scale, inv, ksum, kmean, N);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (smooth && had)
        prep_vquant_kernel<true, true><<<grid, kThreads, 0, st>>>(V, perm, N, vmode, v_mean, inv, v_res, v_sf, K, kmean,
                                                                  k8, sk);
    else if (smooth)
        prep_vquant_kernel<true, false><<<grid, kThreads, 0, st>>>(V, perm, N, vmode, v_mean, inv, v_res, v_sf, K,
                                                                   kmean, k8, sk);
    else
        prep_vquant_kernel<false, false><<<grid, kThreads, 0, st>>>(V, perm, N, vmode, v_mean, inv, v_res, v_sf, K,
                                                                    kmean, k8, sk);
    return cudaGetLastError();
}

}  // namespace vca
