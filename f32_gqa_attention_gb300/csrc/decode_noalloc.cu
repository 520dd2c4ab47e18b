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
// code it names a host-side stand-in), so every call looks the address up
// with cudaGetSymbolAddress while the caller's device is current and checks
// the result.  Nothing is cached: after cudaDeviceReset, or under another
// CUDA context of the same device, the library's module is loaded anew and
// the array has a new address, which the next call picks up.  The first call
// in a context may load the module (lazy loading), so make it before any
// stream capture.
//
// All calls share the one array and each call leaves its contents behind:
// the arrival counters are cleared on the stream before every launch (after
// every host-side check has passed), and calls whose work overlaps on the
// GPU (two streams, or two host threads at once) race on the array and give
// wrong results.  Serialise them.
#include <cstdio>

#include <cuda_runtime.h>

#include "vtmu_attention.h"

namespace vtmu {
vtmu_status report_error(vtmu_status status, const char* message);  // vtmu_api.cpp
vtmu_status check_decode_call(const vtmu_attention_params* p, const float* q, const float* k, const float* v,
                              const float* bias, const float* out, size_t* scratch_bytes);  // vtmu_api.cpp
}

// The decode scratch: arrival counters first, then the split partials.
static __device__ __align__(256) unsigned char g_decode_scratch[VTMU_NOALLOC_SCRATCH_BYTES];

extern "C" VTMU_API vtmu_status vtmu_attention_decode_noalloc(const float* q, const float* k, const float* v,
                                                              const float* bias, float* out,
                                                              const vtmu_attention_params* p,
                                                              cudaStream_t stream) {
    if (!p) return vtmu::report_error(VTMU_ERR_INVALID, "params is NULL");
    if (p->T != 1) return vtmu::report_error(VTMU_ERR_INVALID, "decode_noalloc: T must be 1");
    if (p->kernel != VTMU_KERNEL_AUTO && p->kernel != VTMU_KERNEL_DECODE)
        return vtmu::report_error(VTMU_ERR_INVALID,
                                  "decode_noalloc: kernel must be VTMU_KERNEL_AUTO or VTMU_KERNEL_DECODE");
    vtmu_attention_params dp = *p;
    dp.kernel = VTMU_KERNEL_DECODE;
    // Every check of the regular entry point, before anything touches the
    // shared array.
    size_t need = 0;
    vtmu_status st = vtmu::check_decode_call(&dp, q, k, v, bias, out, &need);
    if (st != VTMU_OK) return st;
    char msg[256];
    if (need > (size_t)VTMU_NOALLOC_SCRATCH_BYTES) {
        std::snprintf(msg, sizeof(msg),
                      "decode_noalloc: this shape needs %zu bytes of decode scratch; the static scratch "
                      "holds %zu (use vtmu_attention with a workspace)",
                      need, (size_t)VTMU_NOALLOC_SCRATCH_BYTES);
        return vtmu::report_error(VTMU_ERR_WORKSPACE, msg);
    }
    void* scratch = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&scratch, g_decode_scratch);
    if (e != cudaSuccess || !scratch) {
        std::snprintf(msg, sizeof(msg), "decode_noalloc: cudaGetSymbolAddress: %s",
                      e != cudaSuccess ? cudaGetErrorString(e) : "null address");
        return vtmu::report_error(VTMU_ERR_CUDA, msg);
    }
    // The arrival counters sit at the start of the scratch and must read zero
    // when the kernel starts; clear them on the caller's stream.
    const int kv_heads = dp.kv_heads ? dp.kv_heads : dp.heads;
    const size_t counter_bytes = ((size_t)kv_heads * 4 + 255) / 256 * 256;
    e = cudaMemsetAsync(scratch, 0, counter_bytes, stream);
    if (e != cudaSuccess) {
        std::snprintf(msg, sizeof(msg), "decode_noalloc: clearing counters: %s", cudaGetErrorString(e));
        return vtmu::report_error(VTMU_ERR_CUDA, msg);
    }
    return vtmu_attention(q, k, v, bias, out, &dp, scratch, (size_t)VTMU_NOALLOC_SCRATCH_BYTES, stream);
}
