// Segmented prefill whose scratch memory lives inside the library, for callers that cannot allocate.
//
// Some callers cannot hand this library a workspace: a plugin inside an inference server that owns all
// device memory through its own pool and gives plugins no allocation hook, or a serving loop that may
// not call cudaMalloc after start-up (cudaMalloc can synchronise the device and its latency is not
// bounded).  kda_prefill_segmented_noalloc serves them: it runs exactly the kernels of
// kda_prefill_segmented (on the tensor-core path four: operand records, fragments, scan, outputs), with
// that call's whole workspace taken from the fixed array below.  The workspace is laid out as
// [per-chunk operand records][segment fragments][entry states] (kda_segmented_workspace_size); the
// records, 145 KiB per 64-token chunk and head, are most of it.
//
// The array is 32 MiB.  Every GPU that loads this code holds it until the process exits.  Calls share
// it and it keeps the last call's contents; nothing in it needs to start at zero (every byte the kernels
// read was written earlier in the same call).  Calls whose kernels overlap on the GPU (other streams,
// other host threads) race on it.
#include <mutex>

#include "../../include/kda.h"
#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

// In host code this name is a host-side stand-in, not a device address: only the address obtained from
// cudaGetSymbolAddress below may be handed to a kernel.
__device__ __align__(256) unsigned char g_segment_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev >= 0 && dev < kMaxDevices && g_addr[dev]) {
    *out = g_addr[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_segment_scratch);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) g_addr[dev] = p;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" kda_status kda_prefill_segmented_noalloc(const kda_prefill_args* a, int32_t segment_len,
                                                    kda_stream_t stream) {
  if (!a) return KDA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
  kda_prefill_args b = *a;
  b.workspace = scratch;
  b.workspace_bytes = kScratchBytes;
  return kda_prefill_segmented(&b, segment_len, stream);  // KDA_ERR_WORKSPACE if it needs more than 32 MiB
}
