// decode_noalloc.cu -- vtmu_attention_decode_noalloc: the split-KV decode
// kernel with its scratch in a static device array instead of a
// caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory of their own --
// for example a plug-in whose host process owns every byte of device memory
// through its own pool, or a latency-critical decode loop that must never
// call cudaMalloc (which can synchronise the device and stall other streams).
// Those callers still pass q, k, v, bias and out; the only memory this call
// needs beyond them is the decode kernel's per-split partial results and its
// arrival counters, and those live in `g_decode_scratch` below.
//
// The array is part of the library image: every GPU that loads the library
// holds VTMU_NOALLOC_SCRATCH_BYTES of device memory for it until the process
// exits.  Host code cannot use the array's name as a device address (in host
// code it names a host-side stand-in), so the first call on each device
// looks the address up with cudaGetSymbolAddress while that device is
// current, checks the result and caches it; later calls on that device reuse
// it.  Make that first call before any stream capture.
//
// All calls share the one array and each call leaves its contents behind:
// the arrival counters are cleared on the stream before every launch, and
// calls whose work overlaps on the GPU (two streams, or two host threads at
// once) race on the array and give wrong results.  Serialise them.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "vtmu_attention.h"

namespace vtmu {
vtmu_status report_error(vtmu_status status, const char* message);  // vtmu_api.cpp
}

// The decode scratch: arrival counters first, then the split partials.
static __device__ __align__(256) unsigned char g_decode_scratch[VTMU_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Address of g_decode_scratch on the current device, looked up once per
// device while it is current.  Returns nullptr and fills `msg` on failure.
void* scratch_address(char* msg, size_t n) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        std::snprintf(msg, n, "decode_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        std::snprintf(msg, n, "decode_noalloc: device %d outside 0..%d", dev, kMaxDevices - 1);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess || !ptr) {
            std::snprintf(msg, n, "decode_noalloc: cudaGetSymbolAddress: %s",
                          e != cudaSuccess ? cudaGetErrorString(e) : "null address");
            return nullptr;
        }
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" VTMU_API vtmu_status vtmu_attention_decode_noalloc(const float* q, const float* k, const float* v,
                                                              const float* bias, float* out,
                                                              const vtmu_attention_params* p,
                                                              cudaStream_t stream) {
    if (!p) return vtmu::report_error(VTMU_ERR_INVALID, "params is NULL");
    if (p->T != 1) return vtmu::report_error(VTMU_ERR_INVALID, "decode_noalloc: T must be 1");
    vtmu_attention_params dp = *p;
    dp.kernel = VTMU_KERNEL_DECODE;
    size_t need = 0;
    vtmu_status st = vtmu_attention_workspace_size(&dp, &need);  // checks the parameters
    if (st != VTMU_OK) return st;
    char msg[256];
    if (need > (size_t)VTMU_NOALLOC_SCRATCH_BYTES) {
        std::snprintf(msg, sizeof(msg),
                      "decode_noalloc: this shape needs %zu bytes of decode scratch; the static scratch "
                      "holds %zu (use vtmu_attention with a workspace)",
                      need, (size_t)VTMU_NOALLOC_SCRATCH_BYTES);
        return vtmu::report_error(VTMU_ERR_WORKSPACE, msg);
    }
    void* scratch = scratch_address(msg, sizeof(msg));
    if (!scratch) return vtmu::report_error(VTMU_ERR_CUDA, msg);
    // The arrival counters sit at the start of the scratch and must read zero
    // when the kernel starts; clear them on the caller's stream.
    const int kv_heads = dp.kv_heads ? dp.kv_heads : dp.heads;
    const size_t counter_bytes = ((size_t)kv_heads * 4 + 255) / 256 * 256;
    cudaError_t e = cudaMemsetAsync(scratch, 0, counter_bytes, stream);
    if (e != cudaSuccess) {
        std::snprintf(msg, sizeof(msg), "decode_noalloc: clearing counters: %s", cudaGetErrorString(e));
        return vtmu::report_error(VTMU_ERR_CUDA, msg);
    }
    return vtmu_attention(q, k, v, bias, out, &dp, scratch, (size_t)VTMU_NOALLOC_SCRATCH_BYTES, stream);
}
