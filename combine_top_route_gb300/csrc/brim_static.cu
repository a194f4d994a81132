// occult_build_brim_noalloc: the BRIM build with its scratch in a static device
// array, for callers that cannot allocate device memory.
//
// occult_build_brim needs a small caller-provided workspace (per-tile column
// counts).  Some callers cannot call cudaMalloc to provide it: code whose device
// memory belongs to another allocator it cannot reach from plain C, serving
// loops that forbid allocation after start-up (cudaMalloc and cudaFree may
// synchronise the device), and processes that must keep a fixed device
// footprint.  This entry point takes the same inputs and outputs and uses the
// file-scope array below instead.  It allocates nothing.
//
// The array is loaded with the library on every GPU that uses the library and
// stays allocated until the process exits.  Every call on a device uses the same
// array, and a call leaves its contents behind.  The three BRIM kernels write
// every entry they read before reading it, so nothing has to start at zero.
// Calls that overlap on the GPU (different streams, no ordering between them)
// race on the array and give wrong results.  Order them on one stream or with
// events.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace occult {

namespace {

// Enough for any layer with T <= 32768 tokens and Ne <= 256 experts:
// ceil(T/32) tiles x (32 + Ne + 1) int32 columns.
static __device__ __align__(256) int32_t g_brim_scratch[OCCULT_STATIC_SCRATCH_BYTES / sizeof(int32_t)];

constexpr int kMaxDevices = 64;

// Device address of the array on each device, once it has been looked up.
std::mutex g_slots_mutex;
void* g_slots[kMaxDevices] = {};

// Device address of the array on the current device, looked up with that device
// current (a host-side name of the array is not an address the GPU can use).
// Only a successful lookup is kept: after a failed one (say, the device was not
// usable yet) the next call asks again.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OCCULT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_slots_mutex);
  if (g_slots[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_brim_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();  // the failure is reported here, not to a later call
      return OCCULT_ERR_CUDA;
    }
    g_slots[dev] = p;
  }
  *out = g_slots[dev];
  return OCCULT_OK;
}

}  // namespace

}  // namespace occult

using namespace occult;

extern "C" int occult_build_brim_noalloc(const occult_desc_t* desc, const int32_t* ids,
                                         const float* gates, const uint32_t* vmask,
                                         const int32_t* placement, int32_t* brim0,
                                         int32_t* seg_off, int32_t* brim1, int32_t* exp_off,
                                         int32_t* epd_src, float* epd_gate, int32_t* counts,
                                         occult_stream_t stream) {
  const int rc = occult_check_desc(desc);
  if (rc) return rc;
  if (!placement || !seg_off || !exp_off || !counts) return OCCULT_ERR_INVALID_ARG;
  if (desc->T > 0 && !(ids && gates && vmask && brim0 && brim1 && epd_src && epd_gate))
    return OCCULT_ERR_INVALID_ARG;
  // the layer's scratch must fit in the static array
  if (brim_ws_bytes(*desc) > static_cast<size_t>(OCCULT_STATIC_SCRATCH_BYTES))
    return OCCULT_ERR_WORKSPACE;
  void* scratch = nullptr;
  int r = scratch_address(&scratch);
  if (r) return r;
  LaunchCtx ctx;
  r = launch_ctx(stream, &ctx);
  if (r) return r;
  return launch_build_brim(ctx, *desc, ids, gates, vmask, placement, brim0, seg_off, brim1,
                           exp_off, epd_src, epd_gate, counts, scratch);
}
