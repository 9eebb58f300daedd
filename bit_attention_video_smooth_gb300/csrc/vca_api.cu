// vca_api.cu -- the C ABI declared in include/vca.h: argument validation,
// workspace sizing and kernel launches.  No device memory is allocated here.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/vca.h"
#include "vca_internal.h"

namespace {

uint64_t g_wait_limit_ns = 2000000000ull;   // 2 s

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool shape_ok(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 128 || d != 128 || (N % 128) != 0) return false;
    const int64_t BH = static_cast<int64_t>(B) * H;
    return BH <= 65535 && BH * N <= (static_cast<int64_t>(1) << 31) - 1;   // BH is a grid y extent
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? VCA_OK : VCA_ERR_CUDA; }

}  // namespace

extern "C" {

const char *vca_status_string(int status) {
    switch (status) {
        case VCA_OK: return "ok";
        case VCA_ERR_INVALID_ARG: return "invalid argument";
        case VCA_ERR_UNSUPPORTED: return "unsupported combination";
        case VCA_ERR_CUDA: return "CUDA error";
        case VCA_ERR_TIMEOUT: return "device wait timed out";
        case VCA_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

int vca_version(void) { return 100; }

size_t vca_workspace_bytes(int op, int B, int H, int N, int d, int k, int vmode) {
    if (!shape_ok(B, H, N, d)) return 0;
    const int BH = B * H;
    switch (op) {
        case VCA_OP_GROUP:
            if (k < 1 || k > vca::kMaxK || k > N) return 0;
            return vca::group_workspace_layout(BH, N, k).bytes;
        case VCA_OP_PREP:
        case VCA_OP_PREP_KSMOOTH:
            if (vmode != VCA_V_E4M3 && vmode != VCA_V_NVFP4) return 0;
            return vca::prep_workspace_layout(BH, N, op == VCA_OP_PREP_KSMOOTH ? vca::kPrepKSmooth : 0u).bytes;
        default:
            return 0;
    }
}

int vca_group(const uint16_t *V, int B, int H, int N, int d, int k, int iters, int32_t *labels, int32_t *perm,
              int32_t *counts, float *centroids, void *ws, size_t ws_bytes, int32_t *dev_status, void *stream) {
    if (!shape_ok(B, H, N, d) || k < 1 || k > vca::kMaxK || k > N || iters < 1 || iters > 1000) return VCA_ERR_INVALID_ARG;
    if (!V || !labels || !perm || !aligned16(V) || !aligned16(labels) || !aligned16(perm)) return VCA_ERR_INVALID_ARG;
    if ((counts && !aligned16(counts)) || (centroids && !aligned16(centroids))) return VCA_ERR_INVALID_ARG;
    if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return VCA_ERR_INVALID_ARG;
    const size_t need = vca_workspace_bytes(VCA_OP_GROUP, B, H, N, d, k, 0);
    if (!ws || ws_bytes < need || !aligned16(ws)) return VCA_ERR_WORKSPACE;
    return from_cuda(vca::launch_group(V, B * H, N, k, iters, labels, perm, counts, centroids, ws, dev_status,
                                       g_wait_limit_ns, static_cast<cudaStream_t>(stream)));
}

int vca_prep_quant(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *perm, int B, int H, int N,
                   int d, int vmode, uint8_t *q8, float *sq, uint8_t *k8, float *sk, uint8_t *v_res, uint8_t *v_sf,
                   float *v_scale, uint16_t *v_mean, void *ws, size_t ws_bytes, void *stream) {
    return vca_prep_quant_ex(Q, K, V, perm, B, H, N, d, vmode, 0u, q8, sq, k8, sk, v_res, v_sf, v_scale, v_mean, ws,
                             ws_bytes, stream);
}

int vca_prep_quant_ex(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *perm, int B, int H,
                      int N, int d, int vmode, uint32_t flags, uint8_t *q8, float *sq, uint8_t *k8, float *sk,
                      uint8_t *v_res, uint8_t *v_sf, float *v_scale, uint16_t *v_mean, void *ws, size_t ws_bytes,
                      void *stream) {
    if (!shape_ok(B, H, N, d) || (vmode != VCA_V_E4M3 && vmode != VCA_V_NVFP4)) return VCA_ERR_INVALID_ARG;
    if (flags & ~(VCA_PREP_QK_HADAMARD | VCA_PREP_K_SMOOTH)) return VCA_ERR_INVALID_ARG;
    const void *ptrs[] = {Q, K, V, perm, q8, sq, k8, sk, v_res, v_scale, v_mean};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return VCA_ERR_INVALID_ARG;
    if (vmode == VCA_V_NVFP4 && (!v_sf || !aligned16(v_sf))) return VCA_ERR_INVALID_ARG;
    const size_t need = vca_workspace_bytes((flags & VCA_PREP_K_SMOOTH) ? VCA_OP_PREP_KSMOOTH : VCA_OP_PREP, B, H, N, d, 1,
                                            vmode);
    if (!ws || ws_bytes < need || !aligned16(ws)) return VCA_ERR_WORKSPACE;
    return from_cuda(vca::launch_prep(Q, K, V, perm, B * H, N, vmode, flags, q8, sq, k8, sk, v_res, v_sf, v_scale,
                                      v_mean, ws, static_cast<cudaStream_t>(stream)));
}

int vca_attention(const uint8_t *q8, const float *sq, const uint8_t *k8, const float *sk, const uint8_t *v_res,
                  const uint8_t *v_sf, const float *v_scale, const uint16_t *v_mean, int B, int H, int N, int d,
                  float softmax_scale, int expcast, int vmode, uint16_t *O, int32_t *dev_status, void *stream) {
    if (!shape_ok(B, H, N, d) || (vmode != VCA_V_E4M3 && vmode != VCA_V_NVFP4) || (expcast != 0 && expcast != 1))
        return VCA_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale)) return VCA_ERR_INVALID_ARG;
    const void *ptrs[] = {q8, sq, k8, sk, v_res, v_scale, v_mean, O};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return VCA_ERR_INVALID_ARG;
    if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return VCA_ERR_INVALID_ARG;
    if (vmode == VCA_V_NVFP4) {
        if (expcast) return VCA_ERR_UNSUPPORTED;   // no single affine log -> E2M1 code map
        if (!v_sf || !aligned16(v_sf)) return VCA_ERR_INVALID_ARG;
    }
    if (softmax_scale <= 0.0f) softmax_scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
    vca::AttentionArgs a;
    a.q8 = q8;
    a.k8 = k8;
    a.v_res = v_res;
    a.v_sf = v_sf;
    a.sq = sq;
    a.sk = sk;
    a.v_scale = v_scale;
    a.v_mean = v_mean;
    a.O = O;
    a.dev_status = dev_status;
    a.BH = B * H;
    a.N = N;
    a.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634);
    a.expcast = expcast;
    a.vmode = vmode;
    a.wait_limit_ns = g_wait_limit_ns;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    return from_cuda(vmode == VCA_V_NVFP4 ? vca::launch_attention_nvfp4(a, st) : vca::launch_attention(a, st));
}

int vca_expcast_codes(const float *s_raw, const float *c, const float *m, int64_t n, uint8_t *out, void *stream) {
    if (n < 0 || (n > 0 && (!s_raw || !c || !m || !out))) return VCA_ERR_INVALID_ARG;
    if (n == 0) return VCA_OK;
    return from_cuda(vca::launch_expcast_codes(s_raw, c, m, n, out, static_cast<cudaStream_t>(stream)));
}

int vca_e4m3_encode_bits(uint32_t start, int64_t n, uint8_t *out, void *stream) {
    if (n < 0 || (n > 0 && !out) || static_cast<uint64_t>(start) + static_cast<uint64_t>(n) > (1ull << 32))
        return VCA_ERR_INVALID_ARG;
    if (n == 0) return VCA_OK;
    return from_cuda(vca::launch_e4m3_encode_bits(start, n, out, static_cast<cudaStream_t>(stream)));
}

int vca_selftest_timeout(int32_t *dev_status, uint64_t limit_ns, void *stream) {
    if (!dev_status || limit_ns < 1000ull || limit_ns > 10000000000ull) return VCA_ERR_INVALID_ARG;
    return from_cuda(vca::launch_selftest_timeout(dev_status, limit_ns, static_cast<cudaStream_t>(stream)));
}

void vca_set_wait_limit_ns(uint64_t limit_ns) {
    if (limit_ns < 1000ull) limit_ns = 1000ull;
    if (limit_ns > 10000000000ull) limit_ns = 10000000000ull;
    g_wait_limit_ns = limit_ns;
}

}  // extern "C"
