// quantize.cu - per-(anchor, KV head) E4M3 quantisation of anchor K or V (the FP8 KV of
// the qwen3-4b-fp8 model in the key points of "Quail: یک میلیارد توکن در دقیقه روی یک
// GPU"). scale = amax / 448 (1 when amax == 0, IEEE fp32 division); code =
// e4m3_rn_satfinite(y) with y the correctly rounded fp32 quotient x / scale.
//
// Two calls:
//  * quail_quantize_kv_fp8 (kv_quantize_kernel): the scales are not known. Persistent
//    clusters of 8 CTAs (two CTAs of different clusters per SM, 8 warps each) take slabs
//    = (anchor, group of KV heads with up to 256 contiguous bytes of every token row);
//    the cluster splits the slab's rows into 8 contiguous parts of up to 512 rows. A
//    CTA holds its part on chip: 14 chunks of 32 rows in shared memory (TMA loads, 112
//    KB) and 2 chunks in registers (4 x 16 bytes per thread). Each warp forms the max
//    |x| of its chunks as they land, the CTA maxima meet in CTA 0's shared memory
//    (distributed shared memory), and one cluster barrier later every thread quantises
//    its chunks from shared memory and registers and stores the codes. HBM sees one read
//    and one write per element (anchors up to 4,096 tokens at 256-byte rows; longer
//    ones are read twice, in rounds of 512 rows per CTA). Each warp issues the first
//    round of its next slab as soon as it has quantised the current one; the two CTAs
//    on an SM belong to different clusters, so one's loads overlap the other's compute.
//    (8-CTA clusters of one 200 KB CTA per SM reach only 15 resident clusters - 120
//    SMs - on GB300; with 112 KB per CTA, 36 clusters fit on 144 SMs.)
//  * quail_quantize_kv_fp8_with_scales (kv_quantize_scaled_kernel): the amax of every
//    (anchor, KV head) is given (as the causal prefill emits it); a grid-stride stream of
//    16-byte loads and 8-byte stores, one read and one write per element.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace quail {

namespace {

constexpr int kMaxHeadsPerSlab = 2;  // heads per 256-byte row (d >= 64)

// 8-byte store of codes with an L2 eviction policy (the codes are not re-read here)
__device__ __forceinline__ void st_hint_8(uint2* p, uint2 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p), "r"(v.x),
               "r"(v.y), "l"(policy)
               : "memory");
}
// A plain shared-memory load (not volatile asm): the compiler may issue a warp's loads
// of a chunk together, ahead of the arithmetic that uses them. The chunks are written
// by TMA and read only after their mbarrier wait, whose asm carries a memory clobber.
__device__ __forceinline__ uint4 ld_shared_16(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// packed running max |x| over 8 bf16 (see absmax_bf16x2)
__device__ __forceinline__ uint32_t absmax_bf16x8(uint32_t acc, const uint4& raw) {
  acc = absmax_bf16x2(acc, raw.x);
  acc = absmax_bf16x2(acc, raw.y);
  acc = absmax_bf16x2(acc, raw.z);
  return absmax_bf16x2(acc, raw.w);
}

inline bool hkv_divides(int hkv, int n) { return hkv % n == 0; }

__device__ __forceinline__ float scale_from_amax(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

// x / s correctly rounded in fp32, given r = RN(1/s): q = RN(x r), then one correction
// with the exact residual x - q s (Markstein's division by reciprocal with an FMA
// correction: P. Markstein, "IA-64 and Elementary Functions", 2000). It can differ from
// the IEEE quotient only when the quotient underflows fp32, where the E4M3 code is a
// signed zero either way; the GPU tests compare it bit for bit with the oracle's IEEE
// division over every bf16 input for many scales. Eight bf16 -> eight E4M3 codes
// (e4m3_rn_satfinite of the fp32 quotient), the arithmetic on fp32 pairs (each lane
// rounds exactly as the scalar instruction). For s > 0 the quotient has the sign of x,
// so OR-ing x's sign bit in restores -0 / s = -0, the one case the FMAs round to +0.
__device__ __forceinline__ uint2 quantize_bf16x8(const uint4& raw, float s, float r) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  const uint64_t r2 = f2(r, r), ns2 = f2(-s, -s);
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t lo_bits = w[k] << 16, hi_bits = w[k] & 0xFFFF0000u;
    const uint64_t x = f2(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    const uint64_t q = f2_mul(x, r2);
    const uint64_t e = f2_fma(q, ns2, x);  // x - q s, rounded once
    float a, b;
    f2_split(f2_fma(e, r2, q), a, b);
    a = __uint_as_float(__float_as_uint(a) | (lo_bits & 0x80000000u));
    b = __uint_as_float(__float_as_uint(b) | (hi_bits & 0x80000000u));
    const __nv_fp8x2_storage_t c =
        __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    packed[k >> 1] |= static_cast<uint32_t>(c) << (16 * (k & 1));
  }
  return make_uint2(packed[0], packed[1]);
}

constexpr int kCluster = 8;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCtasPerSm = 2;                     // two clusters' CTAs share each SM
constexpr int kRows = 32;                         // rows per chunk
constexpr int kChunkBytes = kRows * 256;          // 8 KB at 256-byte rows
constexpr int kSmemChunks = 14;                   // chunks held in shared memory
constexpr int kRegChunks = 2;                     // chunks held in registers
constexpr int kChunksPerRound = kSmemChunks + kRegChunks;  // per CTA: 512 rows
constexpr int kRegVecs = kRegChunks * kRows * 16 / kThreads;  // 16-byte vectors / thread
constexpr int kSmemBytes = kSmemChunks * kChunkBytes + 128;  // + alignment slack

struct __align__(8) QBars {
  uint64_t full[kSmemChunks];
  float warp_max[kWarps][kMaxHeadsPerSlab];
  float part[2][kCluster][kMaxHeadsPerSlab];  // CTA maxima, in CTA 0
  int abort_flag;
};

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* m, uint64_t* bar, void* dst, int x,
                                            int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint4 ld_global_16(const uint4* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

// Geometry of slab `slab` for CTA `rank` of the cluster.
struct Slab {
  int a, c;          // anchor, head group
  int64_t lo;        // first row of this CTA's part
  int rows;          // rows of this CTA's part
  int chunks;        // ceil(rows / kRows)
  int rounds;        // ceil(chunks / kChunksPerRound)
};
__device__ __forceinline__ Slab slab_geometry(int64_t slab, int groups, uint32_t rank,
                                              const int32_t* ao, int64_t T) {
  Slab g;
  g.a = static_cast<int>(slab / groups);
  g.c = static_cast<int>(slab % groups);
  // offsets clamped into [0, T]: inconsistent ones cannot address out of bounds
  const int64_t lo = min(max(static_cast<int64_t>(__ldg(ao + g.a)), int64_t{0}), T);
  const int64_t hi = min(max(static_cast<int64_t>(__ldg(ao + g.a + 1)), lo), T);
  const int64_t len = hi - lo;
  // rows per CTA: a multiple of kRows so that chunks never straddle two CTAs' parts
  const int64_t per = ((len + kCluster - 1) / kCluster + kRows - 1) / kRows * kRows;
  const int64_t start = min(static_cast<int64_t>(rank) * per, len);
  g.lo = lo + start;
  g.rows = static_cast<int>(min(per, len - start));
  g.chunks = (g.rows + kRows - 1) / kRows;
  g.rounds = (g.chunks + kChunksPerRound - 1) / kChunksPerRound;
  return g;
}

// A round of a CTA's part is 16 chunks of 32 rows: chunks 0..13 go to shared memory by
// TMA (chunk j is owned by warp j % 8: warps 0-5 own two, warps 6-7 one), chunks 14 and
// 15 are loaded into registers, kRegVecs (256-byte rows) or kRegVecs / 2 (128-byte rows)
// 16-byte vectors per thread: thread t holds vectors t + 256 i of the two chunks.
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, kCtasPerSm)
kv_quantize_kernel(const __grid_constant__ CUtensorMap map, int num_anchors, int64_t T,
                   int hkv, int d, int hg, const int32_t* __restrict__ ao,
                   const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
                   float* __restrict__ scale, unsigned* err_word, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* buf0 = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  __shared__ QBars bars;
  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_bytes = hg * d * 2;         // 128 or 256
  const int vpr = row_bytes / 16;           // 16-byte vectors per row: 8 or 16
  const int vph = d / 8;                    // vectors per head
  const int chunk_bytes = kRows * row_bytes;
  const int vec_per_lane = kRows * vpr / 32;  // 8 or 16
  const int col = lane & (vpr - 1);          // vpr divides 32: the lane's column is fixed
  const int my_head = col / vph;             // within the slab
  const int row_step = 32 / vpr;             // rows between a lane's vectors
  const int lane_row = lane / vpr;
  const int nreg = kRegChunks * kRows * vpr / kThreads;  // register vectors: 4 or 2
  const int reg_row0 = threadIdx.x / vpr;    // row (in the register chunks) of vector 0
  const int reg_row_step = kThreads / vpr;   // rows between a thread's register vectors
  const int groups = hkv / hg;
  const int64_t slabs = static_cast<int64_t>(num_anchors) * groups;
  const int64_t n_clusters = gridDim.x / kCluster;
  const int64_t row_codes = static_cast<int64_t>(hkv) * d;  // code bytes per token row
  const int64_t row_vec = row_codes / 8;                    // 16-byte vectors of x per row
  const uint64_t pol = l2_policy_evict_first();             // each byte is read once
  const uint4* xv = reinterpret_cast<const uint4*>(x);

  if (threadIdx.x == 0) {
    for (int b = 0; b < kSmemChunks; ++b) mbar_init(&bars.full[b], 1);
    bars.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map);
  }
  __syncthreads();
  WaitCtl wc;
  wc.timeout_ns = timeout_ns;
  wc.abort_flag = &bars.abort_flag;
  wc.err_word = err_word;

  uint32_t fills[2] = {0, 0};  // loads issued into this warp's chunk slots warp, warp + 8
  uint4 rv[kRegVecs];           // this thread's register-chunk vectors of the current round
  auto buf = [&](int slot) { return buf0 + slot * kChunkBytes; };
  // global vector index of row `row` (of the CTA's part) at the thread's column
  auto gvec = [&](const Slab& g, int row) {
    return (g.lo + row) * row_vec + static_cast<int64_t>(g.c) * vpr + col;
  };
  // Issue round r of slab g: this warp's shared-memory chunk slot warp + 8 k (TMA), and
  // this thread's register vectors (plain loads; their first use waits for them).
  auto issue_slot = [&](const Slab& g, int r, int k) {
    const int slot = warp + kWarps * k;
    const int j = r * kChunksPerRound + slot;
    if (slot < kSmemChunks && j < g.chunks) {
      __syncwarp();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier reads first
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars.full[slot], chunk_bytes);
        tma_load_2d(&map, &bars.full[slot], buf(slot), g.c * hg * d,
                    static_cast<int>(g.lo + static_cast<int64_t>(j) * kRows), pol);
      }
      ++fills[k];
      __syncwarp();
    }
  };
  auto issue_regs = [&](const Slab& g, int r) {
    const int row_base = (r * kChunksPerRound + kSmemChunks) * kRows;
#pragma unroll
    for (int i = 0; i < kRegVecs; ++i) {
      const int row = row_base + reg_row0 + i * reg_row_step;
      if (i < nreg && row < g.rows) rv[i] = ld_global_16(xv + gvec(g, row), pol);
    }
  };
  auto issue_round = [&](const Slab& g, int r) {
    issue_slot(g, r, 0);
    issue_slot(g, r, 1);
    issue_regs(g, r);
  };
  auto wait_slot = [&](int k) {
    return wait_parity_warp(wc, &bars.full[warp + kWarps * k], (fills[k] - 1) & 1u);
  };

  int64_t slab = blockIdx.x / kCluster;
  if (slab < slabs) issue_round(slab_geometry(slab, groups, rank, ao, T), 0);
  int parity = 0;
  for (; slab < slabs; slab += n_clusters) {
    const Slab g = slab_geometry(slab, groups, rank, ao, T);
    // pass 1: max |x| of this lane's head over this warp's chunks and this thread's
    // register vectors (packed bf16 maxima)
    uint32_t mp = 0;
    for (int r = 0; r < g.rounds; ++r) {
      if (r > 0) issue_round(g, r);  // round 0 was issued ahead
      // the register vectors were issued first (see pass 2)
      const int row_base = (r * kChunksPerRound + kSmemChunks) * kRows;
#pragma unroll
      for (int i = 0; i < kRegVecs; ++i)
        if (i < nreg && row_base + reg_row0 + i * reg_row_step < g.rows)
          mp = absmax_bf16x8(mp, rv[i]);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int slot = warp + kWarps * k;
        const int j = r * kChunksPerRound + slot;
        if (slot >= kSmemChunks || j >= g.chunks) continue;
        wait_slot(k);
        const int nrows = min(kRows, g.rows - j * kRows);
        const uint8_t* base = buf(slot);
        for (int i = 0; i < vec_per_lane; ++i) {
          const int row = lane_row + i * row_step;
          if (row < nrows) mp = absmax_bf16x8(mp, ld_shared_16(base + (row * vpr + col) * 16));
        }
      }
    }
    // lanes with the same head: the vph-lane group, repeated every vpr lanes
    for (int off = 1; off < vph; off <<= 1)
      mp = absmax_bf16x2(mp, __shfl_xor_sync(0xFFFFFFFFu, mp, off));
    for (int off = vpr; off < 32; off <<= 1)
      mp = absmax_bf16x2(mp, __shfl_xor_sync(0xFFFFFFFFu, mp, off));
    if (lane < vpr && lane % vph == 0) bars.warp_max[warp][my_head] = absmax_bf16x2_value(mp);
    __syncthreads();
    if (threadIdx.x < hg) {
      float cm = bars.warp_max[0][threadIdx.x];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) cm = fmaxf(cm, bars.warp_max[w][threadIdx.x]);
      st_cluster_f32(cluster_map(&bars.part[parity][rank][threadIdx.x], 0), cm);
    }
    cluster_sync();
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < kCluster; ++r)
      amax = fmaxf(amax, ld_cluster_f32(cluster_map(&bars.part[parity][r][my_head], 0)));
    const float s = scale_from_amax(amax);
    const float rs = __frcp_rn(s);
    if (rank == 0 && warp == 0 && lane < vpr && lane % vph == 0)
      scale[static_cast<int64_t>(g.a) * hkv + g.c * hg + my_head] = s;
    // pass 2: quantise from shared memory and registers (a slab held on chip), or read
    // again round by round. In the last round each chunk slot takes the first round of
    // the cluster's next slab as soon as it is quantised.
    const bool more = slab + n_clusters < slabs;
    const Slab ng = more ? slab_geometry(slab + n_clusters, groups, rank, ao, T) : g;
    for (int r = 0; r < g.rounds; ++r) {
      if (g.rounds > 1) issue_round(g, r);
      const bool last = r == g.rounds - 1;
      // the register vectors first, so that the next slab's register loads go out at the
      // start of this pass rather than its end (their latency was exposed in the next
      // slab's max pass)
      const int row_base = (r * kChunksPerRound + kSmemChunks) * kRows;
#pragma unroll
      for (int i = 0; i < kRegVecs; ++i) {
        const int row = row_base + reg_row0 + i * reg_row_step;
        if (i < nreg && row < g.rows)
          st_hint_8(reinterpret_cast<uint2*>(codes) + gvec(g, row),
                    quantize_bf16x8(rv[i], s, rs), pol);
      }
      if (last && more) issue_regs(ng, 0);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int slot = warp + kWarps * k;
        const int j = r * kChunksPerRound + slot;
        if (slot < kSmemChunks && j < g.chunks) {
          if (g.rounds > 1) wait_slot(k);
          const int nrows = min(kRows, g.rows - j * kRows);
          const uint8_t* base = buf(slot);
          uint2* dst = reinterpret_cast<uint2*>(codes) + gvec(g, j * kRows);
          for (int i = 0; i < vec_per_lane; ++i) {
            const int row = lane_row + i * row_step;
            if (row < nrows)
              st_hint_8(dst + row * row_vec,
                        quantize_bf16x8(ld_shared_16(base + (row * vpr + col) * 16), s, rs),
                        pol);
          }
        }
        if (last && more) issue_slot(ng, 0, k);
      }
    }
    if (g.rounds == 0 && more) issue_round(ng, 0);  // this CTA's part was empty
    parity ^= 1;  // the next slab's maxima go to the other buffer (see the barrier note)
  }
  // CTA 0's shared memory must outlive every CTA's reads of it. (Within the loop, the
  // partials of slab k + 2 reuse slab k's buffer only after every CTA has passed slab
  // k + 1's barrier, hence after its reads of slab k.)
  cluster_sync();
}

// Given amax: one read and one write per element, a grid-stride stream of 16-byte loads
// and 8-byte stores. Each block takes chunks of 2,048 consecutive 16-byte vectors (8 per
// thread, thread t holding vectors t + 256 i, so every load and store instruction of a
// warp is contiguous): 128 bytes in flight per thread, 96 KB per SM. (A stream of 16 KB
// bulk copies through a shared-memory ring, one producer lane per SM, read only 5.1-5.4
// TB/s on GB300 against 6.6-6.8 for plain loads, and quantised at 38 % of the copy
// bandwidth.) The scales and their reciprocals of all
// (anchor, KV head) pairs are formed once per block in shared memory when they fit; a
// thread's column is the same for all its vectors when a token row's vector count divides
// 256, and the anchor of a row (binary search of the offsets) and its scale are cached per
// thread.
constexpr int kScaledThreads = 256;
constexpr int kScaledVecs = 8;
// 3 blocks of 256 threads per SM: the compiler's 80 registers a thread, no spills (a
// bound of 4 blocks forces 64 registers and spills, and measured slower)
constexpr int kScaledBlocksPerSm = 3;
constexpr int kScaleTable = 4096;  // (anchor, KV head) pairs kept in shared memory

__global__ void __launch_bounds__(kScaledThreads, kScaledBlocksPerSm) kv_quantize_scaled_kernel(
    int num_anchors, int64_t T, int hkv, int d, const int32_t* __restrict__ ao,
    const float* __restrict__ amax, const __nv_bfloat16* __restrict__ x,
    uint8_t* __restrict__ codes, float* __restrict__ scale) {
  __shared__ float2 table[kScaleTable];  // (scale, RN(1 / scale))
  const int64_t pairs = static_cast<int64_t>(num_anchors) * hkv;
  const bool cached = pairs <= kScaleTable;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t i = tid; i < pairs; i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    scale[i] = amax != nullptr ? scale_from_amax(__ldg(amax + i)) : 1.0f;  // no rows: 1
  const int64_t row_vec = static_cast<int64_t>(hkv) * d / 8;  // vectors per token row
  const int64_t total = T * row_vec;
  if (total == 0 || amax == nullptr) return;
  if (cached) {
    for (int i = threadIdx.x; i < pairs; i += blockDim.x) {
      const float sc = scale_from_amax(__ldg(amax + i));
      table[i] = make_float2(sc, __frcp_rn(sc));
    }
    __syncthreads();
  }
  const uint64_t pol = l2_policy_evict_first();
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint2* cv = reinterpret_cast<uint2*>(codes);
  const int64_t chunk = static_cast<int64_t>(kScaledThreads) * kScaledVecs;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * chunk;
  const uint32_t rv32 = static_cast<uint32_t>(row_vec);
  const uint32_t vph = static_cast<uint32_t>(d / 8);
  const bool even = rv32 <= kScaledThreads && kScaledThreads % rv32 == 0;
  const uint32_t rstep = even ? kScaledThreads / rv32 : 0;
  int a = 0;
  int64_t a_lo = 0, a_hi = -1;  // rows of the anchor of the cached scale
  int64_t pr_cur = -1;
  float sc = 1.0f, rc = 1.0f;
  auto anchor_of = [&](int64_t row) {  // anchors are sorted
    if (row < a_lo || row >= a_hi) {
      int lo = 0, hi = num_anchors - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(ao + mid) <= row) lo = mid; else hi = mid - 1;
      }
      a = lo;
      a_lo = __ldg(ao + a);
      a_hi = __ldg(ao + a + 1);
    }
  };
  auto scale_of = [&](int64_t pr) {
    if (pr != pr_cur) {
      pr_cur = pr;
      if (cached) {
        const float2 t2 = table[pr];
        sc = t2.x;
        rc = t2.y;
      } else {
        sc = scale_from_amax(__ldg(amax + pr));
        rc = __frcp_rn(sc);
      }
    }
  };
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * chunk; base < total; base += stride) {
    uint4 v[kScaledVecs];
#pragma unroll
    for (int i = 0; i < kScaledVecs; ++i) {
      const int64_t e = base + i * kScaledThreads + threadIdx.x;
      if (e < total) v[i] = ld_global_16(xv + e, pol);
    }
    // one 64-bit division per chunk; 32-bit arithmetic within it
    const int64_t base_row = base / row_vec;
    const uint32_t base_col = static_cast<uint32_t>(base - base_row * row_vec);
    if (even) {
      const uint32_t o0 = base_col + threadIdx.x;
      const uint32_t col = o0 % rv32;
      const int64_t row0 = base_row + o0 / rv32;
#pragma unroll
      for (int i = 0; i < kScaledVecs; ++i) {
        const int64_t e = base + i * kScaledThreads + threadIdx.x;
        if (e >= total) continue;
        anchor_of(row0 + static_cast<int64_t>(i) * rstep);
        scale_of(static_cast<int64_t>(a) * hkv + col / vph);
        st_hint_8(cv + e, quantize_bf16x8(v[i], sc, rc), pol);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kScaledVecs; ++i) {
        const int64_t e = base + i * kScaledThreads + threadIdx.x;
        if (e >= total) continue;
        const uint32_t o = base_col + static_cast<uint32_t>(i * kScaledThreads + threadIdx.x);
        const uint32_t orow = o / rv32;
        anchor_of(base_row + orow);
        scale_of(static_cast<int64_t>(a) * hkv + (o - orow * rv32) / vph);
        st_hint_8(cv + e, quantize_bf16x8(v[i], sc, rc), pol);
      }
    }
  }
}

}  // namespace

int quantize_heads_per_slab(int num_kv_heads, int head_dim) {
  // the largest power of two dividing Hkv with HG * d * 2 <= 256 bytes per token row
  int hg = 1;
  while (hg * 2 <= kMaxHeadsPerSlab && hkv_divides(num_kv_heads, hg * 2) &&
         hg * 2 * head_dim * 2 <= 256)
    hg *= 2;
  return hg;
}

cudaError_t launch_quantize_kv_fp8(const QuantArgs& q, int num_sms, cudaStream_t stream) {
  if (q.num_anchors == 0) return cudaSuccess;
  const int hg = quantize_heads_per_slab(q.num_kv_heads, q.head_dim);
  const int64_t slabs = static_cast<int64_t>(q.num_anchors) * (q.num_kv_heads / hg);
  cudaError_t e = cudaFuncSetAttribute(kv_quantize_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // persistent: as many clusters as can be resident at once (one CTA per SM)
  int max_clusters = 0;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms * kCtasPerSm / kCluster * kCluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kv_quantize_kernel, &cfg) != cudaSuccess ||
        max_clusters <= 0) {
      cudaGetLastError();
      max_clusters = num_sms * kCtasPerSm / kCluster;
    }
  }
  const int64_t clusters = slabs < max_clusters ? slabs : max_clusters;
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  kv_quantize_kernel<<<static_cast<unsigned>(clusters * kCluster), kThreads, kSmemBytes,
                       stream>>>(q.map, q.num_anchors, q.total_tokens, q.num_kv_heads,
                                 q.head_dim, hg, q.anchor_offsets,
                                 static_cast<const __nv_bfloat16*>(q.kv),
                                 static_cast<uint8_t*>(q.codes), q.scale, q.err_word,
                                 q.timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_quantize_kv_fp8_scaled(const QuantArgs& q, const float* amax, int num_sms,
                                          cudaStream_t stream) {
  if (q.num_anchors == 0) return cudaSuccess;
  const int64_t vecs = q.total_tokens * q.num_kv_heads * q.head_dim / 8;
  const int64_t chunk = int64_t{kScaledThreads} * kScaledVecs;
  const int64_t need = std::max<int64_t>(
      (vecs + chunk - 1) / chunk, (int64_t{q.num_anchors} * q.num_kv_heads + 255) / 256);
  // one wave of resident blocks (grid-stride): no tail of late blocks
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kv_quantize_scaled_kernel,
                                                    kScaledThreads, 0) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    per_sm = 1;
  }
  const int blocks = static_cast<int>(std::min<int64_t>(need, int64_t{num_sms} * per_sm));
  kv_quantize_scaled_kernel<<<blocks, kScaledThreads, 0, stream>>>(
      q.num_anchors, q.total_tokens, q.num_kv_heads, q.head_dim, q.anchor_offsets, amax,
      static_cast<const __nv_bfloat16*>(q.kv), static_cast<uint8_t*>(q.codes), q.scale);
  return cudaGetLastError();
}

}  // namespace quail
