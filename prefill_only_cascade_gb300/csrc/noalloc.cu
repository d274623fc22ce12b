// noalloc.cu - quail_cascade_attn_noalloc: the cascade attention without a caller
// workspace, for callers that may not allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) around this library: a serving
// engine whose device memory is carved up once at start-up and may not grow afterwards, a
// host framework whose plugin interface only hands over input and output buffers, or
// code on a latency path where an allocation (which can synchronise the device) is not
// allowed. For them the scratch that the cascade kernels need (offset-check flag, anchor
// order, work-item prefix, per-token suffix starts, one record per work item and, with FP8
// anchor KV, the anchors widened to bf16) lives in a file-scope device array of fixed size
// instead of a caller workspace.
//
// Cost and limits:
//   - Every GPU on which the library's kernels are loaded holds kScratchBytes (64 MiB)
//     for this array until the process exits, whether or not this entry point is used.
//   - Batches whose scratch would exceed kScratchBytes are rejected with
//     QUAIL_ERR_UNSUPPORTED (quail_cascade_workspace_size() tells the need).
//   - All calls share the one array, which keeps the previous call's contents. The only
//     word that has to start at zero (the offset-check flag) is cleared on the stream by
//     every call; everything else is written before it is read. Calls whose work
//     overlaps on the GPU (different streams, or other threads, without ordering) race
//     on the array and give wrong results.
//   - The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current); make that first call before any
//     stream capture begins.
#include <mutex>

#include "kernels.h"
#include "quail.h"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(QUAIL_NOALLOC_SCRATCH_BYTES);
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

// In host code this name is only a host-side stand-in for the device array; its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_cascade_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch[kMaxDevices];  // device address per device once a lookup has succeeded

// Device address of the scratch array on the current device. The device is checked first
// (a device other than a GB300 gets QUAIL_ERR_UNSUPPORTED, as from every entry point);
// only a successful lookup is kept, so a failed one (for example a first call made while
// the stream is being captured) is tried again on the next call.
quail_status scratch_address(void** out) {
  const quail_status dev_status = static_cast<quail_status>(quail::current_device_status());
  if (dev_status != QUAIL_OK) return dev_status;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QUAIL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_cascade_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // clear the error so that later calls start clean
      return QUAIL_ERR_CUDA;
    }
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return QUAIL_OK;
}

}  // namespace

extern "C" quail_status quail_cascade_attn_noalloc(
    const quail_cascade_desc* desc, const void* q_suf, const void* k_anc, const void* v_anc,
    const void* k_suf, const void* v_suf, const int32_t* anchor_offsets,
    const int32_t* anchor_suffix_ptr, const int32_t* suffix_offsets, const float* k_scale,
    const float* v_scale, void* out, float* lse, quail_stream_t stream) {
  if (desc == nullptr) return QUAIL_ERR_INVALID_ARG;
  const size_t need = quail_cascade_workspace_size(desc);
  if (need > kScratchBytes) return QUAIL_ERR_UNSUPPORTED;  // batch too large for the array
  void* scratch = nullptr;
  const quail_status st = scratch_address(&scratch);
  if (st != QUAIL_OK) return st;
  return quail_cascade_attn(desc, q_suf, k_anc, v_anc, k_suf, v_suf, anchor_offsets,
                            anchor_suffix_ptr, suffix_offsets, k_scale, v_scale, out, lse,
                            scratch, kScratchBytes, stream);
}
