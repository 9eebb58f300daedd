/*
 * vca.h -- C ABI of the VC-Attention hot path on GB300 (sm_103a).
 *
 * VC-Attention ("VC-Attention: Value Smoothing and Softmax Casting for Low-bit
 * Attention", agihunt.info/papers/2609.15810, section "method") changes two steps
 * of a FlashAttention-style FP8 kernel:
 *   V-Smooth   -- per (batch, head), k-means on the Value tokens; K and V are
 *                 permuted together by cluster label; every 128-token block
 *                 subtracts its mean (a 16-bit vector), only the residual is
 *                 quantised (per-channel E4M3 or NVFP4) and the mean is added
 *                 back through the row sums online softmax already keeps.
 *   ExpCast-FP8 -- one FMA writes the E4M3 byte of the softmax probability
 *                 straight from the log2-domain score:
 *                 byte = rne(8 log2 p + 56 + beta), beta = -0.35, clipped to the
 *                 normal range (codes below 8 flush to 0).
 *
 * The library computes on the device only; there is no CPU fallback.  Every
 * entry point is asynchronous on the caller's CUDA stream (`stream` is a
 * cudaStream_t; NULL is the legacy default stream).  The library allocates no
 * device memory: the caller owns every buffer (inputs, outputs and the scratch
 * workspace sized by vca_workspace_bytes).  Device pointers must be 16-byte
 * aligned.  No C++ exception crosses this boundary.
 *
 * Layouts (all contiguous, row-major, little-endian; BH = B*H, nb = N/128):
 *   Q, K, V       bf16 (uint16 bit patterns) [B][H][N][d], d = 128
 *   labels, perm  int32 [BH][N]; perm[i] = source token placed in slot i
 *   counts        int32 [BH][k];  centroids fp32 [BH][k][d]
 *   q8, k8        E4M3 bytes [BH][N][d] (q8 in original order, k8 permuted)
 *   sq, sk        fp32 [BH][nb]  (one dequantisation scale per 128-token block)
 *   v_mean        bf16 [BH][nb][d] (block means of the permuted V)
 *   E4M3 mode:  v_res E4M3 [BH][nb][d][128] (residual, channel-major per block),
 *               v_scale fp32 [BH][d] (one scale per channel), v_sf unused (NULL)
 *   NVFP4 mode: v_res [BH][nb][d][64] packed E2M1 (token 2i in the low nibble),
 *               v_sf E4M3 [BH][nb][d][8] (one scale per 16 tokens of a channel),
 *               v_scale fp32 [BH] (the per-(b,h) scale above the E4M3 scales)
 *   O             bf16 [B][H][N][d], rows in the original query order
 *
 * Sizes accepted by every entry point: B >= 1, H >= 1, B*H <= 65,535 (one grid
 * row of CTAs per head), N a positive multiple of 128, B*H*N <= 2^31 - 1
 * tokens, d = 128.  Anything else is VCA_ERR_INVALID_ARG.
 *
 * Return value: a vca_status.  Invalid arguments are reported synchronously and
 * launch nothing.  Device-side failures (a bounded wait that ran out) are
 * written to the optional `dev_status` word, which the caller reads after the
 * stream has synchronised.
 */
#ifndef VCA_H
#define VCA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VCA_OK = 0,
    VCA_ERR_INVALID_ARG = 1,   /* bad size, null or misaligned pointer */
    VCA_ERR_UNSUPPORTED = 2,   /* a combination the method does not define */
    VCA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    VCA_ERR_TIMEOUT = 4,       /* a bounded device wait ran out (dev_status) */
    VCA_ERR_WORKSPACE = 5      /* workspace missing or smaller than required */
} vca_status;

typedef enum { VCA_V_E4M3 = 0, VCA_V_NVFP4 = 1 } vca_vmode;
/* VCA_OP_PREP_KSMOOTH: the prep's workspace when VCA_PREP_K_SMOOTH is set. */
typedef enum { VCA_OP_GROUP = 0, VCA_OP_PREP = 1, VCA_OP_ATTENTION = 2, VCA_OP_PREP_KSMOOTH = 3 } vca_op;

/* Human-readable name of a vca_status value (static string, never NULL). */
const char *vca_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int vca_version(void);

/* Scratch bytes the caller must pass as `ws` for `op` at this problem size
 * (0 if none).  Returns 0 as well for invalid sizes. */
size_t vca_workspace_bytes(int op, int B, int H, int N, int d, int k, int vmode);

/*
 * vca_group -- V-Smooth "Group" step (paper page, "method"; news page,
 * "V-Smooth" bullet "Group"): per (b,h), Lloyd k-means on the N Value tokens
 * (d = 128 channels), then a stable counting sort of the tokens by label.
 *   init     centroid c = V row floor((c + 1/2) N / k)
 *   assign   label = argmin_c |v - C_c|^2, ties to the lowest c
 *   update   C_c = mean of its tokens (fp32); an empty cluster keeps C_c
 *   `iters` rounds of (assign, update); labels are those of the last assign.
 * Outputs: labels [BH][N], perm [BH][N] (tokens ordered by (label, index)),
 * counts [BH][k] (tokens per label), centroids [BH][k][d] (may be NULL).
 * The distances are taken on the tensor core from bf16 V and the centroids
 * split into bf16 hi + lo parts (fp32 accumulation): labels equal those of an
 * exact computation except where two centroids are within ~2^-16 relative of
 * each other.
 * Requires 1 <= k <= min(N, 128), 1 <= iters <= 1000,
 * ws_bytes >= vca_workspace_bytes(VCA_OP_GROUP, ...).
 * dev_status (optional, device int32): set to VCA_ERR_TIMEOUT if a bounded
 * wait inside the kernels ran out; left untouched otherwise.
 */
int vca_group(const uint16_t *V, int B, int H, int N, int d, int k, int iters,
              int32_t *labels, int32_t *perm, int32_t *counts, float *centroids,
              void *ws, size_t ws_bytes, int32_t *dev_status, void *stream);

/*
 * vca_prep_quant -- the fused V-Smooth prep (paper page, "method": demean each
 * 128-token hardware block, quantise only the residual, 16-bit mean per block;
 * Q/K to FP8; no high-precision intermediate is written to device memory):
 *   K and V are gathered by perm (perm may be reused across calls);
 *   v_mean[b] = bf16(fp32(sum of the block's 128 tokens) / 128);
 *   residual R = fp32(v) - fp32(v_mean);
 *   E4M3:  a_c = max |R[:, c]| over the sequence, v_scale[c] = a_c / 448,
 *          v_res = E4M3_rne_sat(R * (448 / a_c));
 *   NVFP4: g = max |R| / (6 * 448) per (b,h) (v_scale), per 16 tokens of a
 *          channel sf = E4M3(amax16 / (6 g)) (v_sf),
 *          v_res = E2M1_rne_sat(R * (1 / (sf * g)));
 *   Q (original order) and K (permuted) per 128-token block:
 *          s = amax / 448, x8 = E4M3_rne_sat(x * (448 / amax)).
 * An all-zero block or channel gets scale 1.
 */
int vca_prep_quant(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *perm,
                   int B, int H, int N, int d, int vmode,
                   uint8_t *q8, float *sq, uint8_t *k8, float *sk,
                   uint8_t *v_res, uint8_t *v_sf, float *v_scale, uint16_t *v_mean,
                   void *ws, size_t ws_bytes, void *stream);

/*
 * vca_prep_quant_ex -- vca_prep_quant with option flags (flags = 0 is exactly
 * vca_prep_quant; unknown bits return VCA_ERR_INVALID_ARG):
 *   VCA_PREP_QK_HADAMARD  rotate every Q and K row by the unnormalised 128-point
 *          Walsh-Hadamard transform H before the FP8 quantisation (the QK
 *          Hadamard of the Q/K prior art the insight page discusses, which
 *          spreads outlier channels over all channels).  H is symmetric with
 *          H H = 128 I, so (H q) . (H k) = 128 q . k: sk carries the factor
 *          1/128 (exact) and vca_attention needs no change.  The transform is
 *          defined as fp32 butterflies in a fixed order -- for bit k = 0..6 of
 *          the channel index, every pair (c, c + 2^k) with bit k of c clear
 *          becomes (a + b, a - b) -- so its rounding is reproducible; then
 *          s = amax / 448 and x8 = E4M3_rne_sat(x * (448 / amax)) as usual.
 *   VCA_PREP_K_SMOOTH  subtract the keys' channel mean over the sequence of
 *          each (b,h) before the FP8 quantisation (SageAttention's treatment
 *          of the keys' channel bias, the handling of Q/K outliers the paper
 *          page's motivation and the insight page's section "Value Is the
 *          Error Source Earlier Methods Underestimated" refer to).  Every score
 *          of a query row moves by the same amount, so softmax attention is
 *          unchanged and vca_attention needs no change.  The mean is fp32 in a
 *          fixed order, so it is reproducible: per permuted 128-token block a
 *          halving tree (token i plus token i + 64 for i < 64, then i + 32, ...,
 *          i + 1), the block sums added in block order, divided by N; each key
 *          value becomes fp32(k) - mean (one rounding), before the Hadamard
 *          rotation when both flags are set.  Needs ws_bytes >=
 *          vca_workspace_bytes(VCA_OP_PREP_KSMOOTH, ...).
 */
#define VCA_PREP_QK_HADAMARD 1u
#define VCA_PREP_K_SMOOTH 2u
int vca_prep_quant_ex(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *perm,
                      int B, int H, int N, int d, int vmode, uint32_t flags,
                      uint8_t *q8, float *sq, uint8_t *k8, float *sk,
                      uint8_t *v_res, uint8_t *v_sf, float *v_scale, uint16_t *v_mean,
                      void *ws, size_t ws_bytes, void *stream);

/*
 * vca_prep_quant_noalloc -- the same computation and outputs as vca_prep_quant,
 * for callers that cannot pass the library any scratch device memory (a host
 * program that owns all device memory and gives an operator only its tensors,
 * or a code path where a cudaMalloc and its possible device synchronisation are
 * not allowed).  The paper has no counterpart to this entry point.
 * Scratch: a buffer of VCA_NOALLOC_SCRATCH_BYTES built into the library, which
 * every GPU that loads the library holds until the process exits.  Problems
 * whose prep workspace (vca_workspace_bytes(VCA_OP_PREP, ...)) exceeds it return
 * VCA_ERR_WORKSPACE and launch nothing.  That workspace is 512 bytes per
 * 128-token block plus 512 bytes per head, so 16 MiB covers exactly the
 * problems with B*H*(N/128) + B*H <= 32,768 (B=1, H=40, N=70,656 needs 22,120
 * of those units, 11.3 MB).  The first call on a device looks
 * up the buffer's device address (make it before any stream capture).  Every
 * call shares the one buffer: calls that overlap on the GPU race and must be
 * ordered by the caller.  Nothing in the buffer needs clearing between calls.
 * This entry point allocates no device memory.
 */
#define VCA_NOALLOC_SCRATCH_BYTES (16u << 20)
int vca_prep_quant_noalloc(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *perm,
                           int B, int H, int N, int d, int vmode,
                           uint8_t *q8, float *sq, uint8_t *k8, float *sk,
                           uint8_t *v_res, uint8_t *v_sf, float *v_scale, uint16_t *v_mean,
                           void *stream);

/*
 * vca_attention -- non-causal FP8 attention over the prepared operands (paper
 * page, "method": online softmax; ExpCast; the block means come back as one
 * outer product rowsum_b x mean_b per key block, no second pass).  For every
 * query row, key blocks are visited in increasing (permuted) order; with
 * c = (sq * sk_b) * (softmax_scale * log2 e), S the raw FP8 product q8 . k8
 * and m the reference max (log2 units), which moves to the block's max
 * max_j(S_j * c) only when that exceeds m + 8 (the first block always sets it):
 *   expcast = 1:  P = E4M3 byte rne(fma(S, 8c, 55.65 - 8m)), flushed below 8
 *   expcast = 0:  P = E4M3_rne_sat(exp2(fma(S, c, -m)))
 *   NVFP4 mode (expcast must be 0): per 16 keys p = exp2(fma(S, c, -m)),
 *                 sf = E4M3(amax16 / 6), P = E2M1(p * (1 / sf)) * sf; the V
 *                 residual decodes to E2M1 * its 16-token E4M3 scale
 *   rowsum_b = sum of the decoded P of block b; l = sum_b rowsum_b
 *   O = (sum_b P_b . v_res_b * v_scale + sum_b rowsum_b (x) v_mean_b) / l
 * with accumulators rescaled by 2^(m_old - m_new) whenever m moves.
 * softmax_scale <= 0 selects 1/sqrt(d).  expcast = 1 with VCA_V_NVFP4 returns
 * VCA_ERR_UNSUPPORTED (NVFP4 has no single affine log-to-code map).
 * dev_status (optional, device int32): set to VCA_ERR_TIMEOUT if a bounded
 * wait inside the kernel ran out; left untouched otherwise.
 */
int vca_attention(const uint8_t *q8, const float *sq, const uint8_t *k8, const float *sk,
                  const uint8_t *v_res, const uint8_t *v_sf, const float *v_scale,
                  const uint16_t *v_mean, int B, int H, int N, int d,
                  float softmax_scale, int expcast, int vmode,
                  uint16_t *O, int32_t *dev_status, void *stream);

/*
 * vca_expcast_codes -- the device ExpCast map on its own (the same inline
 * function the attention kernel uses), for bit-exact testing:
 *   out[i] = clip(rne(fma(s_raw[i], 8 c[i], 55.65 - 8 m[i]))), codes < 8 -> 0,
 *   codes > 126 -> 126.  Device arrays of n elements.
 */
int vca_expcast_codes(const float *s_raw, const float *c, const float *m, int64_t n,
                      uint8_t *out, void *stream);

/*
 * vca_e4m3_encode_bits -- the device's E4M3 conversion (round to nearest even,
 * saturating to +-448) applied to the fp32 bit patterns start .. start+n-1;
 * out is a device array of n bytes.  Used to compare the hardware conversion
 * with a software one over every fp32 input.
 */
int vca_e4m3_encode_bits(uint32_t start, int64_t n, uint8_t *out, void *stream);

/*
 * vca_selftest_timeout -- launches one bounded wait on a barrier that nothing
 * completes, with the given limit in nanoseconds (1e3 .. 1e10); the kernel gives
 * up, writes VCA_ERR_TIMEOUT to dev_status and returns, leaving the context
 * usable.  Exercises the failure path every kernel wait uses.
 */
int vca_selftest_timeout(int32_t *dev_status, uint64_t limit_ns, void *stream);

/* Upper bound on every bounded device wait, in nanoseconds (default 2e9). */
void vca_set_wait_limit_ns(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* VCA_H */
