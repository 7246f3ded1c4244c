// kda_prefill_noalloc.cu -- kda_prefill for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) around a prefill: code
// running inside a CUDA-graph capture or under a caching allocator that owns every byte of the
// device, runtimes that pre-reserve a fixed memory budget before serving starts, and C hosts
// that have no allocator of their own.  kda_prefill needs a scratch workspace; this entry point
// uses a fixed region compiled into the library instead of a caller buffer.
//
// The region is a file-scope __device__ array of kda::kNoAllocScratchBytes (64 MiB); every GPU
// that loads the library holds it until the process exits.  In host code the array's name is
// only a host-side stand-in, so its device address is obtained per device with
// cudaGetSymbolAddress the first time this entry point runs with that device current, and that
// address is what the kernels receive.  Under lazy module loading that first call is also when
// the device reserves the region (it can fail for want of memory); a cudaDeviceReset
// invalidates the cached address.  All calls share the region and it keeps the last
// call's contents; the prefill fully writes every scratch byte it later reads, so nothing has
// to be cleared between calls.  Two calls whose kernels overlap on the GPU (different streams,
// no ordering between them) race on the region.
#include <mutex>
#include <stdio.h>

#include "kda_internal.cuh"
#include "kda_prefill.cuh"

void kda_set_last_error(const char *msg);

namespace kda {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_prefill_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch region on the current device (set up on first use).
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_prefill_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace kda

extern "C" {

size_t kda_prefill_noalloc_max_bytes(void) { return kda::kNoAllocScratchBytes; }

kda_status kda_prefill_noalloc(const kda_layer *layer, const kda_pool *pool, const int32_t *slot_ids,
                               int32_t B, int32_t L, int32_t chunk, const void *q, const void *k,
                               const void *v, const void *f_a, const void *beta_logit,
                               const void *gate, void *out, void *stream)
{
    const size_t need = kda_prefill_workspace_size(layer, B, L, chunk);
    if (need > kda::kNoAllocScratchBytes) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "kda_prefill_noalloc: B=%d, L=%d, H=%d need %zu bytes of scratch, more than the %zu built in",
                 B, L, layer ? layer->num_heads : 0, need, kda::kNoAllocScratchBytes);
        kda_set_last_error(msg);
        return KDA_ERR_UNSUPPORTED;
    }
    void *ws = nullptr;
    const cudaError_t e = kda::scratch_address(&ws);
    if (e != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof msg, "kda_prefill_noalloc: scratch set-up failed: %s", cudaGetErrorString(e));
        kda_set_last_error(msg);
        return KDA_ERR_CUDA;
    }
    return kda_prefill(layer, pool, slot_ids, B, L, chunk, q, k, v, f_a, beta_logit, gate, out, ws,
                       kda::kNoAllocScratchBytes, stream);
}

}  // extern "C"
