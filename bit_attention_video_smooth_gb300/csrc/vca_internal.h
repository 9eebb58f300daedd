// vca_internal.h -- launch functions and workspace layouts shared by the
// kernel translation units and the C-ABI layer (vca_api.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace vca {

constexpr int kMaxK = 128;           // largest supported cluster count

// The k-means assign kernel's work split: each CTA takes one chunk of
// chunk_tokens tokens (a multiple of 128) of one (batch, head), nchunk chunks
// per head (the last one ragged); group_workspace_layout picks the split.
struct GroupWorkspace {
    int nchunk, chunk_tokens;
    size_t off_centroids, off_norm, off_psum, off_pcnt, bytes;
};
GroupWorkspace group_workspace_layout(int BH, int N, int k);
cudaError_t launch_group(const uint16_t *V, int BH, int N, int k, int iters, int32_t *labels, int32_t *perm,
                         int32_t *counts, float *centroids, void *ws, int32_t *dev_status, uint64_t limit_ns,
                         cudaStream_t st);

constexpr uint32_t kPrepQkHadamard = 1u;   // VCA_PREP_QK_HADAMARD
constexpr uint32_t kPrepKSmooth = 2u;      // VCA_PREP_K_SMOOTH
struct PrepWorkspace {
    size_t off_amax, off_inv, off_ksum, off_kmean, bytes;
};
PrepWorkspace prep_workspace_layout(int BH, int N, uint32_t flags);
cudaError_t launch_prep(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *perm, int BH, int N,
                        int vmode, uint32_t flags, uint8_t *q8, float *sq, uint8_t *k8, float *sk, uint8_t *v_res,
                        uint8_t *v_sf, float *v_scale, uint16_t *v_mean, void *ws, cudaStream_t st);

struct AttentionArgs {
    const uint8_t *q8, *k8, *v_res, *v_sf;
    const float *sq, *sk, *v_scale;
    const uint16_t *v_mean;
    uint16_t *O;
    int32_t *dev_status;
    int BH, N;
    float scale_log2;      // softmax_scale * log2(e), fp32
    int expcast, vmode;
    uint64_t wait_limit_ns;
};
cudaError_t launch_attention(const AttentionArgs &a, cudaStream_t st);         // E4M3 residual V
cudaError_t launch_attention_nvfp4(const AttentionArgs &a, cudaStream_t st);   // NVFP4 residual V and P

cudaError_t launch_expcast_codes(const float *s_raw, const float *c, const float *m, int64_t n, uint8_t *out,
                                 cudaStream_t st);
cudaError_t launch_e4m3_encode_bits(uint32_t start, int64_t n, uint8_t *out, cudaStream_t st);
cudaError_t launch_selftest_timeout(int32_t *dev_status, uint64_t limit_ns, cudaStream_t st);

}  // namespace vca
