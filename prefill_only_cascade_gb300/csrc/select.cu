// select.cu - the join's verdicts from the restricted head's argmax. "Motor de inferência
// Quail atinge 1 bilhão de tokens por minuto por GPU", section "Como funciona": a boolean
// AI.IF needs only the one token of the last prefill pass, chosen among 8 options; the
// AI_JOIN of "Quail: یک میلیارد توکن در دقیقه روی یک GPU" keeps the pairs for which it
// holds. Suffix s passes when argmax[s] == true_index.
//
// Order-preserving compaction in three launches over chunks of kChunk suffixes:
//   1. select_count_kernel  per-chunk count of passing suffixes
//   2. select_scan_kernel   (1 CTA) exclusive scan of the chunk counts; total -> num_selected
//   3. select_scatter_kernel verdicts, and the passing ids written in increasing order
//   4. select_anchor_kernel  (optional) passing suffixes per anchor: two binary searches of
//                            the anchor's suffix range in the sorted list
#include <cstdint>

#include "kernels.h"

namespace quail {

namespace {

constexpr int kSelThreads = 256;
constexpr int kPerThread = 16;
constexpr int kChunk = kSelThreads * kPerThread;  // suffixes per CTA

// Exclusive scan of one int per thread over the block (blockDim.x a multiple of 32, at
// most 1024); `total` receives the block's sum.
__device__ int block_scan_excl(int v, int& total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  total = warp_sums[nw - 1];
  const int before = warp > 0 ? warp_sums[warp - 1] : 0;
  __syncthreads();  // warp_sums is reused by the next call
  return before + x - v;
}

__global__ void __launch_bounds__(kSelThreads) select_count_kernel(const int32_t* argmax,
                                                                   int64_t S, int32_t t,
                                                                   int32_t* chunk_count) {
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kChunk;
  int c = 0;
  for (int i = threadIdx.x; i < kChunk; i += kSelThreads) {
    const int64_t s = base + i;
    if (s < S && __ldg(argmax + s) == t) ++c;
  }
  int total;
  block_scan_excl(c, total);
  if (threadIdx.x == 0) chunk_count[blockIdx.x] = total;
}

__global__ void __launch_bounds__(1024) select_scan_kernel(int32_t* chunk_count, int n,
                                                           int32_t* num_selected) {
  int carry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int v = i < n ? chunk_count[i] : 0;
    int total;
    const int ex = block_scan_excl(v, total);
    if (i < n) chunk_count[i] = carry + ex;  // now the chunk's first output position
    carry += total;
  }
  if (threadIdx.x == 0) *num_selected = carry;
}

// Thread j of chunk b owns suffixes b * kChunk + 16 j .. + 15, so a block scan of the
// per-thread counts gives every passing suffix its position in increasing order.
__global__ void __launch_bounds__(kSelThreads) select_scatter_kernel(
    const int32_t* argmax, int64_t S, int32_t t, const int32_t* chunk_base, uint8_t* verdict,
    int32_t* selected) {
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kChunk +
                     static_cast<int64_t>(threadIdx.x) * kPerThread;
  uint32_t bits = 0;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k)
    if (s0 + k < S && __ldg(argmax + s0 + k) == t) bits |= 1u << k;
  int total;
  int pos = chunk_base[blockIdx.x] + block_scan_excl(__popc(bits), total);
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    if (s0 + k >= S) break;
    const bool pass = (bits >> k) & 1u;
    if (verdict != nullptr) verdict[s0 + k] = pass ? 1 : 0;
    if (pass) selected[pos++] = static_cast<int32_t>(s0 + k);
  }
}

// first position in sorted[0, n) whose value is >= key
__device__ __forceinline__ int lower_bound_dev(const int32_t* sorted, int n, int32_t key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(sorted + mid) < key) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(256) select_anchor_kernel(const int32_t* selected,
                                                            const int32_t* num_selected,
                                                            const int32_t* anchor_suffix_ptr,
                                                            int A, int32_t* anchor_count) {
  const int a = blockIdx.x * blockDim.x + threadIdx.x;
  if (a >= A) return;
  const int n = *num_selected;
  anchor_count[a] = lower_bound_dev(selected, n, __ldg(anchor_suffix_ptr + a + 1)) -
                    lower_bound_dev(selected, n, __ldg(anchor_suffix_ptr + a));
}

}  // namespace

size_t join_select_workspace_bytes(int64_t num_suffixes) {
  return static_cast<size_t>((num_suffixes + kChunk - 1) / kChunk) * 4 + 16;
}

cudaError_t launch_join_select(const JoinSelectArgs& j, cudaStream_t stream) {
  cudaError_t e;
  const int64_t chunks = (j.num_suffixes + kChunk - 1) / kChunk;
  if (chunks == 0) {
    e = cudaMemsetAsync(j.num_selected, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
  } else {
    select_count_kernel<<<static_cast<unsigned>(chunks), kSelThreads, 0, stream>>>(
        j.argmax, j.num_suffixes, j.true_index, j.chunk_work);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    select_scan_kernel<<<1, 1024, 0, stream>>>(j.chunk_work, static_cast<int>(chunks),
                                               j.num_selected);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    select_scatter_kernel<<<static_cast<unsigned>(chunks), kSelThreads, 0, stream>>>(
        j.argmax, j.num_suffixes, j.true_index, j.chunk_work, j.verdict, j.selected);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (j.anchor_count != nullptr && j.num_anchors > 0) {
    select_anchor_kernel<<<(j.num_anchors + 255) / 256, 256, 0, stream>>>(
        j.selected, j.num_selected, j.anchor_suffix_ptr, j.num_anchors, j.anchor_count);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace quail
