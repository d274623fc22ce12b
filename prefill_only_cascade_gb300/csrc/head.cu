// head.cu - fused RMSNorm + 8-column unembedding + argmax (the restricted head of the
// zero-decode step: "Motor de inferência Quail atinge 1 bilhão de tokens por minuto por
// GPU", section "Como funciona", zero-decode and cascade-attention bullets; "Quail: یک
// میلیارد توکن در دقیقه روی یک GPU", key points on the 8-token head).
//
// The kernel is bound by the HBM read of h (2 bytes per element, read once). Per element
// it needs 8 multiply-adds for the logits and one for the sum of squares. The 8 dot
// products run on the tensor cores (mma.sync m16n8k16 bf16 -> fp32: N = 8 is exactly the
// retained vocabulary) so that the FP32 pipes only square and add; gamma is folded into
// the head weights in fp32 and split into a bf16 high part and a bf16 low part, both
// multiplied, so the folded weights keep ~16 significant bits.
//
// Work split: a warp owns 16 rows at a time. Lane (g = lane / 4, t = lane % 4) loads
// 16 bytes of rows g and g + 8 at column 32c + 8t for every 32-column chunk c; these two
// vectors are exactly the A fragments of two k16 MMA steps once the k index inside a
// chunk is permuted the same way for A and B (a dot product does not depend on the
// order of k). The weights are stored in shared memory in that fragment order, so a warp
// reads 512 contiguous bytes per chunk.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace quail {

namespace {

constexpr int kHeadThreads = 256;

__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float sq_sum_bf16x8(const uint4& v, float acc) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16);
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u);
    acc = fmaf(lo, lo, acc);
    acc = fmaf(hi, hi, acc);
  }
  return acc;
}

__global__ void __launch_bounds__(kHeadThreads)
restricted_head_kernel(int64_t n_rows, int hidden, float eps, const __nv_bfloat16* __restrict__ h,
                       int64_t h_rows, int64_t stride, const int32_t* __restrict__ row_index,
                       const __nv_bfloat16* __restrict__ gamma,
                       const __nv_bfloat16* __restrict__ w8, float* __restrict__ logits,
                       int32_t* __restrict__ argmax, unsigned* err_word) {
  extern __shared__ __align__(16) uint4 wfrag[];  // [chunks][32 lanes] hi, then the same lo
  const int nchunks = hidden / 32;
  uint4* whi = wfrag;
  uint4* wlo = wfrag + nchunks * 32;

  // Fold gamma into W8 (fp32, exact for bf16 x bf16), split hi/lo, store in fragment order:
  // entry (c, lane) holds W[lane / 4][32c + 8(lane % 4) .. + 7].
  for (int e = threadIdx.x; e < nchunks * 32; e += blockDim.x) {
    const int c = e >> 5, ln = e & 31;
    const int n = ln >> 2, k0 = 32 * c + 8 * (ln & 3);
    uint32_t hi_w[4], lo_w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int k = k0 + 2 * i + j;
        f[j] = __bfloat162float(gamma[k]) * __bfloat162float(w8[n * hidden + k]);
      }
      const __nv_bfloat162 hi2 = __floats2bfloat162_rn(f[0], f[1]);
      const __nv_bfloat162 lo2 =
          __floats2bfloat162_rn(f[0] - __low2float(hi2), f[1] - __high2float(hi2));
      hi_w[i] = *reinterpret_cast<const uint32_t*>(&hi2);
      lo_w[i] = *reinterpret_cast<const uint32_t*>(&lo2);
    }
    whi[e] = make_uint4(hi_w[0], hi_w[1], hi_w[2], hi_w[3]);
    wlo[e] = make_uint4(lo_w[0], lo_w[1], lo_w[2], lo_w[3]);
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t ngroups = (n_rows + 15) / 16;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const float inv_hidden = 1.0f / static_cast<float>(hidden);

  for (int64_t grp = warp0; grp < ngroups; grp += nwarps) {
    const int64_t rowA = grp * 16 + g, rowB = rowA + 8;
    const bool outA = rowA < n_rows, outB = rowB < n_rows;  // output rows that exist
    int64_t srcA = outA ? (row_index ? static_cast<int64_t>(row_index[rowA]) : rowA) : 0;
    int64_t srcB = outB ? (row_index ? static_cast<int64_t>(row_index[rowB]) : rowB) : 0;
    // a gathered source row outside h is never read: its row gets NaN logits, argmax -1
    const bool badA = outA && (srcA < 0 || srcA >= h_rows);
    const bool badB = outB && (srcB < 0 || srcB >= h_rows);
    if (badA) srcA = 0;
    if (badB) srcB = 0;
    if ((badA || badB) && t == 0) atomicOr(err_word, kErrDeviceBounds);
    const bool okA = outA && !badA, okB = outB && !badB;  // rows that are read
    const __nv_bfloat16* pA = h + srcA * stride + 8 * t;
    const __nv_bfloat16* pB = h + srcB * stride + 8 * t;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float ssA = 0.f, ssB = 0.f;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    // Software pipeline over batches of kB chunks with two register buffers: the loads of
    // the next batch are in flight while the current batch is multiplied.
    constexpr int kB = 4;
    uint4 xa[2][kB], xb[2][kB];
    auto load = [&](int buf, int c0) {
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        const bool in = c0 + i < nchunks;
        xa[buf][i] = (okA && in) ? ld_stream_16(pA + 32 * (c0 + i)) : zero;
        xb[buf][i] = (okB && in) ? ld_stream_16(pB + 32 * (c0 + i)) : zero;
      }
    };
    auto compute = [&](int buf, int c0) {
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        if (c0 + i < nchunks) {
          const uint4 a = xa[buf][i], b = xb[buf][i];
          const uint4 wh = whi[(c0 + i) * 32 + lane];
          const uint4 wl = wlo[(c0 + i) * 32 + lane];
          mma_bf16_16816(acc, a.x, b.x, a.y, b.y, wh.x, wh.y);
          mma_bf16_16816(acc, a.z, b.z, a.w, b.w, wh.z, wh.w);
          mma_bf16_16816(acc, a.x, b.x, a.y, b.y, wl.x, wl.y);
          mma_bf16_16816(acc, a.z, b.z, a.w, b.w, wl.z, wl.w);
          ssA = sq_sum_bf16x8(a, ssA);
          ssB = sq_sum_bf16x8(b, ssB);
        }
      }
    };
    load(0, 0);
    for (int c = 0; c < nchunks; c += 2 * kB) {
      if (c + kB < nchunks) load(1, c + kB);
      compute(0, c);
      if (c + 2 * kB < nchunks) load(0, c + 2 * kB);
      if (c + kB < nchunks) compute(1, c + kB);
    }
    // The four lanes of a quad share rows g and g + 8.
    ssA += __shfl_xor_sync(0xFFFFFFFFu, ssA, 1);
    ssA += __shfl_xor_sync(0xFFFFFFFFu, ssA, 2);
    ssB += __shfl_xor_sync(0xFFFFFFFFu, ssB, 1);
    ssB += __shfl_xor_sync(0xFFFFFFFFu, ssB, 2);
    const float rA = 1.0f / sqrtf(ssA * inv_hidden + eps);
    const float rB = 1.0f / sqrtf(ssB * inv_hidden + eps);
    // acc: (row g, cols 2t, 2t+1), (row g+8, cols 2t, 2t+1)
    const float lA0 = acc[0] * rA, lA1 = acc[1] * rA;
    const float lB0 = acc[2] * rB, lB1 = acc[3] * rB;
    // argmax over the 8 columns of each row: the lowest index wins ties
    float vA = lA0;
    int iA = 2 * t;
    if (lA1 > vA) { vA = lA1; iA = 2 * t + 1; }
    float vB = lB0;
    int iB = 2 * t;
    if (lB1 > vB) { vB = lB1; iB = 2 * t + 1; }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      const float ovA = __shfl_xor_sync(0xFFFFFFFFu, vA, off);
      const int oiA = __shfl_xor_sync(0xFFFFFFFFu, iA, off);
      const float ovB = __shfl_xor_sync(0xFFFFFFFFu, vB, off);
      const int oiB = __shfl_xor_sync(0xFFFFFFFFu, iB, off);
      if (ovA > vA || (ovA == vA && oiA < iA)) { vA = ovA; iA = oiA; }
      if (ovB > vB || (ovB == vB && oiB < iB)) { vB = ovB; iB = oiB; }
    }
    const float nan = __int_as_float(0x7fc00000);
    if (outA) {
      *reinterpret_cast<float2*>(logits + rowA * 8 + 2 * t) =
          badA ? make_float2(nan, nan) : make_float2(lA0, lA1);
      if (t == 0) argmax[rowA] = badA ? -1 : iA;
    }
    if (outB) {
      *reinterpret_cast<float2*>(logits + rowB * 8 + 2 * t) =
          badB ? make_float2(nan, nan) : make_float2(lB0, lB1);
      if (t == 0) argmax[rowB] = badB ? -1 : iB;
    }
  }
}

}  // namespace

size_t restricted_head_smem_bytes(int hidden) { return static_cast<size_t>(hidden) * 32; }

cudaError_t launch_restricted_head(const HeadArgs& a, int num_sms, cudaStream_t stream) {
  if (a.n_rows == 0) return cudaSuccess;
  const size_t smem = restricted_head_smem_bytes(a.hidden);
  cudaError_t e = cudaFuncSetAttribute(restricted_head_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, restricted_head_kernel,
                                                    kHeadThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t groups = (a.n_rows + 15) / 16;
  const int64_t need = (groups + (kHeadThreads / 32) - 1) / (kHeadThreads / 32);
  const int64_t grid = need < static_cast<int64_t>(num_sms) * per_sm
                           ? need
                           : static_cast<int64_t>(num_sms) * per_sm;
  restricted_head_kernel<<<static_cast<unsigned>(grid), kHeadThreads, smem, stream>>>(
      a.n_rows, a.hidden, a.eps, static_cast<const __nv_bfloat16*>(a.h), a.h_rows,
      a.h_row_stride, a.row_index, static_cast<const __nv_bfloat16*>(a.gamma),
      static_cast<const __nv_bfloat16*>(a.w8), a.logits, a.argmax, a.err_word);
  return cudaGetLastError();
}

}  // namespace quail
