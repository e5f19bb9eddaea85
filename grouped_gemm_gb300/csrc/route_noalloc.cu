// route_noalloc.cu -- the routing permutation for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc, or own no spare device buffer to hand
// us: code running while a CUDA graph is being captured under an allocator
// that forbids new allocations, runtimes that plan every byte of device memory
// ahead of time, or plain C hosts without a memory allocator of their own on
// the device.  For them, moe_ffn_route_noalloc keeps its scratch (the per-block
// histograms, padded offsets, row tables and status words) in one file-scope
// device array instead of a caller workspace.  The caller still passes the
// inputs and the output arrays.
//
// The array is loaded with the library on every device that uses it and stays
// there until the process exits.  Every call on a device shares it and it keeps
// the previous call's contents, so two calls that overlap on the GPU (different
// streams, or host threads racing on one device) corrupt each other.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe_ffn.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

// Limits of the allocation-free routing call.
constexpr int64_t kNoAllocMaxPairs = 131072;          // T * k
constexpr size_t kNoAllocScratchBytes = 6u << 20;     // 6 MiB

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device, looked up once per
// device.  In host code the symbol itself is only a host-side stand-in.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_ffn_route_noalloc(const int32_t* topk_ids, const float* topk_w, int T, int E, int k,
                                              int32_t* counts, int32_t* offsets, int32_t* slot_of_pair,
                                              int32_t* status_bits, void* stream) {
  if (T < 0 || E < 1 || E > kMaxExperts || k < 1) return MOE_ERR_INVALID_ARG;
  if ((int64_t)T * k > kNoAllocMaxPairs) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (T > 0 && (!topk_ids || !topk_w)) return MOE_ERR_INVALID_ARG;
  const Workspace probe = plan_workspace(nullptr, T, E, 128, 128, k, kRouteOnly);
  if (probe.bytes > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Workspace ws = plan_workspace(scratch, T, E, 128, 128, k, kRouteOnly);
  // The status words accumulate error bits: they must start at zero.
  cudaError_t e = cudaMemsetAsync(ws.err, 0, 32, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (T == 0) {
    if (counts) e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, st);
    if (e == cudaSuccess && offsets) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st);
  } else {
    e = launch_route(ws, topk_ids, topk_w, T, E, k, st);
    if (e == cudaSuccess && counts)
      e = cudaMemcpyAsync(counts, ws.counts, sizeof(int32_t) * E, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && offsets)
      e = cudaMemcpyAsync(offsets, ws.offsets, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && slot_of_pair)
      e = cudaMemcpyAsync(slot_of_pair, ws.slot_of_pair, sizeof(int32_t) * T * k, cudaMemcpyDeviceToDevice, st);
  }
  if (e == cudaSuccess && status_bits)
    e = cudaMemcpyAsync(status_bits, ws.err, sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
