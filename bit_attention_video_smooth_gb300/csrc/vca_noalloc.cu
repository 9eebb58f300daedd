// vca_noalloc.cu -- vca_prep_quant_noalloc: the fused prep with its scratch in a
// buffer that lives inside this library, for callers that cannot hand the
// library any device memory beyond their own inputs and outputs.
//
// Who needs this: code that runs inside a host program which owns every byte of
// device memory (an inference server or plugin host that reserves the GPU's
// memory up front and passes an operator only its tensors), and code paths that
// must not call cudaMalloc because it can synchronise the device or fail under
// memory pressure at a point where failure cannot be handled.
//
// The scratch is a file-scope __device__ array of kNoallocScratchBytes, which
// every GPU that loads libvca.so keeps until the process exits.  Host code
// cannot use the array's name as a device pointer, so the first call on each
// device looks up its device address with cudaGetSymbolAddress (with that
// device current) and caches it; that first call should come before any stream
// capture on the device.  All calls share the one buffer: two calls whose work
// overlaps on the GPU (different streams, or different host threads) race on it
// and must be ordered by the caller.  The prep writes every scratch element it
// later reads, so nothing needs clearing between calls.
#include <mutex>

#include "../../include/vca.h"
#include "vca_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = VCA_NOALLOC_SCRATCH_BYTES;
static_assert(kNoallocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_prep_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_prep_scratch on the current device (looked up once).
cudaError_t scratch_for_current_device(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_prep_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int vca_prep_quant_noalloc(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int32_t *perm,
                                      int B, int H, int N, int d, int vmode, uint8_t *q8, float *sq, uint8_t *k8,
                                      float *sk, uint8_t *v_res, uint8_t *v_sf, float *v_scale, uint16_t *v_mean,
                                      void *stream) {
    const size_t need = vca_workspace_bytes(VCA_OP_PREP, B, H, N, d, 1, vmode);
    if (need == 0) return VCA_ERR_INVALID_ARG;                 // bad shape or mode
    if (need > kNoallocScratchBytes) return VCA_ERR_WORKSPACE; // problem too large for the built-in scratch
    const void *ptrs[] = {Q, K, V, perm, q8, sq, k8, sk, v_res, v_scale, v_mean};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return VCA_ERR_INVALID_ARG;
    if (vmode == VCA_V_NVFP4 && (!v_sf || !aligned16(v_sf))) return VCA_ERR_INVALID_ARG;
    void *ws = nullptr;
    if (scratch_for_current_device(&ws) != cudaSuccess) return VCA_ERR_CUDA;
    const cudaError_t e = vca::launch_prep(Q, K, V, perm, B * H, N, vmode, 0u, q8, sq, k8, sk, v_res, v_sf, v_scale,
                                           v_mean, ws, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VCA_OK : VCA_ERR_CUDA;
}
