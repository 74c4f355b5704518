// photon_noalloc.cu -- photon_paged_decode_noalloc: the paged decode with its
// split-KV scratch taken from a fixed array inside the library instead of a
// caller-allocated workspace.
//
// Who needs it: code that runs the decode but cannot hand it device memory.
// Serving engines usually reserve nearly all of HBM for the KV pool when they
// start, so a later cudaMalloc either fails or eats into that reservation;
// plugins and extension points inside such a host often get no allocator
// handle at all; and some callers must not make a cudaMalloc/cudaFree call on
// their decode path at all, since those calls can synchronise the device.
// Such callers pass only their inputs and outputs here.
//
// The scratch array is a file-scope __device__ array of kNoAllocScratchBytes
// (32 MiB).  Every GPU that loads the library holds it until the process exits.
// In host code the array's name is only a host-side stand-in, so the device
// address is looked up once per device with cudaGetSymbolAddress (on the first
// call made with that device current) and cached.
#include <atomic>
#include <cstddef>

#include <cuda_runtime.h>

#include "../../include/photon_paged.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::atomic<void*> g_noalloc_scratch_addr[kNoAllocMaxDevices];

// Device address of the scratch array on the current device (set-up on the
// first call per device).
photon_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PHOTON_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return PHOTON_ERR_UNSUPPORTED;
  void* p = g_noalloc_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PHOTON_ERR_CUDA;
    g_noalloc_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return PHOTON_OK;
}

}  // namespace

extern "C" photon_status_t photon_paged_decode_noalloc(const void* q, const void* k_cache,
                                                       const void* v_cache,
                                                       const int32_t* block_tables,
                                                       const int32_t* context_lens, float scale,
                                                       void* out,
                                                       const photon_paged_shape_t* shape,
                                                       photon_stream_t stream) {
  const size_t need = photon_paged_decode_workspace_size(shape);
  if (need == 0)  // invalid shape or an empty batch: the regular entry point reports it
    return photon_paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                               nullptr, 0, shape, stream);
  if (need > kNoAllocScratchBytes) return PHOTON_ERR_WORKSPACE;
  void* scratch = nullptr;
  const photon_status_t st = noalloc_scratch(&scratch);
  if (st != PHOTON_OK) return st;
  return photon_paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, scratch,
                             kNoAllocScratchBytes, shape, stream);
}
