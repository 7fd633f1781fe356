// xq_layer_mixed_static: the layer entry point for callers that cannot
// allocate device memory.
//
// xq_layer_mixed asks its caller for a workspace (the layer's Q8 buffers and
// the grouped matmul's scheduling state). Some callers have no way to get
// one: an engine that hands all device memory to its own pool at start-up
// and forbids allocation afterwards, a plugin running inside a host
// application that owns the allocator, or a latency-critical decode loop
// that must not pay for cudaMalloc, which can synchronize the whole device
// and fail under memory pressure in the middle of a request. This file gives
// them a fixed workspace instead: a file-scope device array that every GPU
// loading the library holds until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it
// is only a stand-in symbol). Every call asks the runtime for the real
// address with cudaGetSymbolAddress, with the caller's device current, and
// checks the result. The address belongs to the current context (the
// module instance loaded into it), so it is not cached across calls: after
// cudaDeviceReset, or under a caller's own driver-API context, a cached
// address could point into a module that is gone. Once the module is loaded
// the lookup is a host-side table lookup; the first call on a device may
// load it, so make that first call before any stream capture on the device.
//
// Nothing here allocates: no cudaMalloc, no cudaFree, no library allocator.
// Every call on a device shares the one array and leaves its contents
// behind. The only part that must start at zero, the scheduling state, is
// cleared by the quantize kernel of every call. Calls whose work overlaps on
// the GPU (different streams, or different host threads without ordering)
// race on the array: order them on one stream or synchronize between them.
#include "xq.h"
#include "xq_common.cuh"

namespace {

// XQ_LAYER_STATIC_SCRATCH_BYTES (4 MiB) covers one decode layer of an
// 8B-class model at M <= 8 (the Llama-3-8B-shaped layer needs about
// 1.3 MB); larger requests are refused.
constexpr size_t kStaticScratchBytes = XQ_LAYER_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_layer_scratch[kStaticScratchBytes];

// Device address of the scratch array in the current context.
xq_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_layer_scratch) != cudaSuccess || !p) return XQ_ERR_CUDA;
  *out = p;
  return XQ_OK;
}

}  // namespace

extern "C" {

xq_status xq_layer_mixed_static(const xq_proj* proj, int n_proj, const float* const* inputs, int n_inputs,
                                int M, xq_stream stream) {
  const size_t need = xq_layer_workspace_bytes(proj, n_proj, n_inputs, M);
  if (need == 0) {
    // Bad arguments: let the regular entry point report the precise code
    // (it returns before touching the workspace).
    return xq_layer_mixed(proj, n_proj, inputs, n_inputs, M, nullptr, 0, stream);
  }
  if (need > kStaticScratchBytes) return XQ_ERR_WORKSPACE;
  void* ws = nullptr;
  const xq_status st = scratch_address(&ws);
  if (st != XQ_OK) return st;
  return xq_layer_mixed(proj, n_proj, inputs, n_inputs, M, ws, kStaticScratchBytes, stream);
}

}  // extern "C"
