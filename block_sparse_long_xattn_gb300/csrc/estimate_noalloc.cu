// bsx_xattn_estimate_noalloc: the estimate entry point for callers that cannot
// allocate device memory.
//
// Some hosts own every byte of device memory: an inference engine that hands
// its plugins fixed buffers from its own pool and forbids them to call
// cudaMalloc, or a real-time loop that may not call an allocator (cudaMalloc
// and cudaFree can block on the device).  Such a caller may also have no spare
// buffer to lend as the estimator's scratch.  This entry point takes the same
// inputs and outputs as bsx_xattn_estimate but uses a scratch array of fixed
// size that lives in the library's own device code.
//
// The array is a file-scope __device__ variable; every GPU that uses the
// library keeps it until the process exits.  Host code may not use the
// variable's name as a device address, so the first call on each device looks
// its address up with cudaGetSymbolAddress (with that device current) and
// caches it.  CUDA loads device code lazily: the array is committed on the
// device by that first lookup, which can therefore fail for lack of device
// memory; it should come before the caller's engine fills its memory pool and
// before any stream capture.  The cache belongs to the primary context of
// each device and does not survive cudaDeviceReset.
// Calls share the one array: two calls whose kernels overlap on the GPU (on
// different streams, or from different host threads) race on it.  Nothing in
// the array needs to start at zero: the estimate writes every scratch cell it
// later reads.
#include <stdio.h>

#include <atomic>

#include "../../include/bsxattn.h"
#include "common.cuh"

namespace {

// 32 MiB: enough for 32 q-heads x 1024 key blocks x 256 reshaped rows (a
// 4096-token chunk of a 128K context at stride 16) or a 4096-token chunk of a
// 32K context at stride 8.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (looked up on the
// first call per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return BSX_ERR_CUDA;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      fprintf(stderr, "bsxattn: scratch lookup failed: %s\n", cudaGetErrorString(e));
      return BSX_ERR_CUDA;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return BSX_OK;
}

}  // namespace

extern "C" {

int bsx_xattn_estimate_noalloc(bsx_shape s, const void* q, const void* k, int q_len,
                               int q_start_pos, int stride, float threshold,
                               uint8_t* mask, float* block_sums, void* stream) {
  const size_t need = bsx_estimate_workspace_bytes(s, q_len, q_start_pos, stride);
  // invalid shape or stride: let the regular entry point report which (it
  // returns before touching the device)
  if (need == 0)
    return bsx_xattn_estimate(s, q, k, q_len, q_start_pos, stride, threshold, mask,
                              block_sums, nullptr, 0, stream);
  if (need > kNoAllocScratchBytes) return BSX_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != BSX_OK) return rc;
  return bsx_xattn_estimate(s, q, k, q_len, q_start_pos, stride, threshold, mask,
                            block_sums, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
