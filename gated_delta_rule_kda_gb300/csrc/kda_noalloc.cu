// kda_layer_core_noalloc: the layer core for callers that cannot allocate device
// memory.
//
// kda_layer_core needs a scratch workspace (the fp32 q^, k^, v, log_alpha, beta
// and o~ handed from stage to stage) that its caller allocates.  Some callers
// cannot do that: a plugin running inside a host application that owns every
// device allocation and hands out no scratch, or a latency-critical path where
// an allocation (and the synchronisation it may imply) is not acceptable.  For
// them this entry point uses a fixed scratch array that lives in the library's
// own device memory instead: a file-scope __device__ array of
// KDA_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the library holds
// until the process exits.
//
// In host code the array's name is only a host-side stand-in for the device
// object, so the device address is obtained with cudaGetSymbolAddress, once per
// device, on the first call made with that device current.  The address is cached
// for the life of the process and is not looked up again after a device reset.
#include <atomic>

#include "kda_common.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (set up on first use).
void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev].store(addr, std::memory_order_release);
        p = addr;
    }
    return p;
}

}  // namespace

extern "C" kda_status kda_layer_core_noalloc(
    int32_t num_seqs, int32_t total_tokens, int32_t num_heads, const void *qp, const void *kp,
    const void *vp, const float *conv_w, const void *z, const float *A, const float *b,
    const void *beta_logit, const void *g, const int32_t *cu_seqlens, const float *S0,
    float scale, float l2_eps, float rms_eps, kda_dtype out_dtype, void *o_gated, float *S_final,
    void *stream) {
    if (num_seqs < 1 || total_tokens < 0 || num_heads < 1) return KDA_ERR_INVALID_ARGUMENT;
    const size_t need = kda_layer_core_workspace_size(num_seqs, total_tokens, num_heads);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_UNSUPPORTED;
    void *scratch = scratch_address();
    if (scratch == nullptr) return KDA_ERR_CUDA;
    return kda_layer_core(num_seqs, total_tokens, num_heads, qp, kp, vp, conv_w, z, A, b,
                          beta_logit, g, cu_seqlens, S0, scale, l2_eps, rms_eps, out_dtype,
                          o_gated, S_final, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES, stream);
}
