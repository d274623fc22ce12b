// cascade.cu - simplified cascade attention for the prefill-only AI.IF / AI_JOIN step
// ("Motor de inferência Quail atinge 1 bilhão de tokens por minuto por GPU", section
// "Como funciona", cascade-attention bullet: suffixes attend to the anchor, then to
// themselves, and the two results are combined by LSE rescaling).
//
// One persistent kernel computes, for every suffix token and query head, softmax
// attention over [all anchor keys ; its own suffix keys up to itself]. The anchor part
// and the suffix part are two groups of KV tiles folded into one online softmax, which
// is the LSE merge done incrementally: after the anchor tiles the running (max, sum, O)
// is the anchor partial, and each suffix tile merges into it by rescaling.
//
// Work item = (anchor a, KV head g, 2 x 128 query rows). A query tile packs 128/G
// consecutive suffix tokens of anchor a times the G query heads that share KV head g
// (row r = token r / G, head g*G + r % G). Every suffix of the anchor sees the same
// anchor keys with no mask, so any tokens of the anchor's suffixes can share a tile; the
// suffix part uses a per-row key window [start of the row's suffix, the row's token].
//
// Launch sequence on the caller's stream (all scratch lives in the caller's workspace):
//   1. memset of the check flag
//   2. cascade_segments_kernel  (grid)   per-suffix offset checks; seg[t] = start of the
//                                        suffix holding token t
//   3. cascade_schedule_kernel  (1 CTA)  anchor checks; anchors ordered by decreasing
//                                        anchor-tile count; prefix sum of work items
//   4. cascade_items_kernel     (grid)   one record per work item (a quad of four query
//                                        tiles for the CTA-pair kernel)
//   5. anchor_e4m3_to_bf16_kernel (grid, FP8 anchor KV only) stages the anchor codes as
//                                        bf16 in the workspace
//   6. the fast kernel - cascade_attn_kernel (persistent, one CTA per SM) or, for d = 128
//      fused calls, cascade_pair_kernel (persistent clusters of two CTAs, 256-row tcgen05
//      MMAs over an SM pair, a 3- or 4-stage K/V ring) - then cascade_attn_kernel's exact
//      instance over the items the fast kernel listed
//
// Per CTA of the attention kernel:
//   warp 8      TMA producer: a ring of K / V tiles (128 keys each)
//   warp 9      MMA issuer:   S_q = Q_q K^T (SMEM x SMEM -> TMEM), O_q += P_q V
//                             (P from TMEM, V from SMEM), tcgen05 kind::f16, M = 128
//   warp 10     fill checker: folds the V and next-K fills into the P-ready barrier
//   warp 11     query loader: each item's two query tiles, as soon as their buffers free
//   warps 0-3   softmax of query tile 0, one thread per TMEM lane (= query row), and its
//               epilogue (O / l through shared memory and TMA tensor stores)
//   warps 4-7   softmax and epilogue of query tile 1
// TMEM (512 columns): tile q uses S/P at columns 256q .. +127 and O at 256q+128 .. +255.
// The two query tiles share every anchor KV tile loaded into shared memory and ping-pong:
// while one warpgroup exponentiates its scores the tensor core works on the other tile.
//
// FP8 anchor KV (e4m3 codes with one fp32 scale per (anchor, KV head) for K and for V):
// every e4m3 value is a bf16 value, so the codes are widened to bf16 once per call into
// the workspace (exact; 2 bytes written per code) and the same bf16 kernel runs with
// FP8 = true. The K scale folds into the score scale of anchor tiles and the V scale into
// their P (P = p * v_scale, while the row sum keeps p), so O accumulates true values.
// Converting once per call instead of once per work item keeps the tensor core fed: a
// (anchor, KV head) is read by hundreds of work items.
#include <atomic>
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace quail {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 384;             // three warpgroups
// Register split (setmaxnreg): the two softmax warpgroups grow to Cfg::kRegsSoftmax, the
// producer/MMA warpgroup shrinks to Cfg::kRegsOther; 256 * softmax + 128 * other =
// 64,512 registers, which must not exceed the 384 * (registers at launch) the block
// holds; the host checks the compiled register count before launching.
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpFillCheck = 10;
constexpr int kWarpQLoad = 11;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: O is rescaled only past 2^8
// Fast kernel bounds (P = 2^(s c) with no max subtracted); outside them the item goes to
// the exact kernel. The row sum l = sum P must lie in [2^-64, 2^32]: every P <= l <= 2^32
// keeps O and l far from fp32 overflow (an infinite P makes l infinite, so it is caught),
// and l >= 2^-64 keeps the largest P >= 2^-64 / (keys), far inside the bf16/fp32 range.
// Testing l needs no row max at all. With FP8 anchor KV, P also carries v_scale; a scale
// above 2^64 (or NaN) sends the item to the exact kernel as well, so P * v_scale and O
// stay finite.
constexpr float kSpecSumLow = 5.421010862427522e-20f;   // 2^-64
constexpr float kSpecSumHigh = 4294967296.0f;            // 2^32
constexpr float kSpecScaleHigh = 1.8446744073709552e19f;  // 2^64
constexpr int kSortBins = 1024;
constexpr uint32_t kTmemCols = 512;

// Shared-memory staging of the epilogue: two 2 KB buffers per softmax warp.
constexpr int kStageWarpBytes = 2 * 2048;
constexpr int kSmemStage = 8 * kStageWarpBytes;

template <int D>
struct Cfg {
  static constexpr int kKB = D / 64;                   // 128-byte column blocks per row
  static constexpr int kBlockBytes = 128 * 128;        // 128 rows x 128 bytes
  static constexpr int kTileBytes = kKB * kBlockBytes;  // one 128-row bf16 tile
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kSmemQ = 2 * kTileBytes;
  static constexpr int kSmemKV = kStages * 2 * kTileBytes;
  // queries, K/V ring, barriers (1 KB), epilogue staging, alignment slack (1 KB)
  static constexpr int kSmemBytes = kSmemQ + kSmemKV + 1024 + kSmemStage + 1024;
  static constexpr int kRegsSoftmax = (D == 128) ? 176 : 184;
  static constexpr int kRegsOther = (D == 128) ? 152 : 136;
  static_assert(256 * kRegsSoftmax + 128 * kRegsOther <= 384 * 168, "register split");
};
struct __align__(8) Bars {
  uint64_t q_full[4], q_empty[4];  // the single-CTA kernel uses [0, 2)
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  uint32_t peer_abort;  // CTA pairs: the other CTA of the pair gave up on a wait
  // AMAX: the tile each K/V slot holds - its first row, the own rows of query tiles 0
  // and 1 ([lo, hi) each), its KV head
  int rec[4][6];
};
static_assert(sizeof(Bars) <= 1024, "barriers fit in the last kilobyte of shared memory");

// One work item as written by cascade_items_kernel (two int4).
struct Item {
  int a_tok0, la;   // anchor token start (into k_anc/v_anc) and length
  int t0, ag;       // first suffix token of query tile 0; anchor * Hkv + KV head
  int ws0, ws1;     // suffix key window start of query tile 0 / 1
  int tend0, tend1; // one past the last valid token of query tile 0 / 1 (tend == start: empty)
  __device__ __forceinline__ int ws(int q) const { return q ? ws1 : ws0; }
  __device__ __forceinline__ int tend(int q) const { return q ? tend1 : tend0; }
  __device__ __forceinline__ int n_anchor_tiles() const { return (la + kBN - 1) / kBN; }
  __device__ __forceinline__ int window() const { return max(tend0 - ws0, tend1 - ws1); }
  __device__ __forceinline__ int n_sfx_tiles() const { return (window() + kBN - 1) / kBN; }
  __device__ __forceinline__ int nk_sfx() const {
    return (n_sfx_tiles() == 1 && window() <= 64) ? 64 : 128;
  }
  // Both query tiles' suffix windows start at the same token (both inside one suffix, or
  // q1 inside the suffix where q0 ends): then they share their suffix tiles as they share
  // the anchor tiles (q0 masks the keys past its rows).
  __device__ __forceinline__ bool sfx_shared() const { return ws0 == ws1; }
  __device__ __forceinline__ int n_tiles() const {
    return n_anchor_tiles() + (sfx_shared() ? 1 : 2) * n_sfx_tiles();
  }
};

__device__ __forceinline__ int4 ld_nc_v4(const int32_t* p) {
  int4 v;
  asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// QUADS: the caller may walk quad halves (the exact kernel; the fast single-CTA kernel
// always runs with two-tile items, and leaves the branch out).
template <bool QUADS>
__device__ __forceinline__ Item load_item(const CascadeParams& p, int item) {
  if (QUADS && p.tiles_per_item == 4) {
    // half h of quad item / 2 (the exact kernel after the CTA-pair kernel): its query
    // tiles 2h and 2h + 1, each with its own key window
    const int quad = item >> 1, h = item & 1;
    const int4 a = ld_nc_v4(p.items + 12 * static_cast<int64_t>(quad));
    const int4 b = ld_nc_v4(p.items + 12 * static_cast<int64_t>(quad) + 4);
    const int4 c = ld_nc_v4(p.items + 12 * static_cast<int64_t>(quad) + 8);
    const int tok = p.tok_per_tile;
    Item it;
    it.a_tok0 = a.x; it.la = a.y; it.ag = a.w;
    it.t0 = a.z + 2 * h * tok;
    it.tend0 = h ? c.x : b.z;
    it.tend1 = h ? c.y : b.w;
    const int t1 = it.t0 + tok;
    it.ws0 = it.t0 < it.tend0 ? __ldg(p.seg + it.t0) : it.t0;
    it.ws1 = t1 < it.tend1 ? __ldg(p.seg + t1) : t1;
    return it;
  }
  const int4 a = ld_nc_v4(p.items + 8 * static_cast<int64_t>(item));
  const int4 b = ld_nc_v4(p.items + 8 * static_cast<int64_t>(item) + 4);
  Item it;
  it.a_tok0 = a.x; it.la = a.y; it.t0 = a.z; it.ag = a.w;
  it.ws0 = b.x; it.ws1 = b.y; it.tend0 = b.z; it.tend1 = b.w;
  return it;
}

// Ring position -> what it holds: anchor tile k (k < nA), then the suffix tiles: shared,
// suffix tile i at position nA + i; else suffix tile i of query tile q at nA + 2i + q.
__device__ __forceinline__ int pos_of(int nA, bool shared, int q, int k) {
  return (k < nA || shared) ? k : nA + 2 * (k - nA) + q;
}

__device__ __forceinline__ bool drain_wait(uint64_t* bar, uint32_t parity, uint64_t deadline) {
  const uint32_t a = smem_u32(bar);
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() > deadline) return false;
  }
  return true;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// 32-byte global store (sm_100+); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// Epilogue of one warp whose 32 rows are all valid output rows: O / l as bf16 through
// shared memory and TMA tensor stores. The warp's TMEM lanes are 32 / G consecutive
// tokens x G heads, which is one box (32 columns of d, G heads, 32 / G tokens) of the
// output map. Each 64-column half of the row (128 bytes a row) is staged as two 32-column
// boxes in the warp's two 2 KB buffers with the 64-byte swizzle (16-byte chunk c of row r
// at c ^ ((r >> 1) & 3), so each st.shared of the warp takes the minimum four wavefronts),
// made visible to the async proxy by one fence and written by two TMA stores; the buffers
// are rewritten only once the stores issued from them before have read them. The
// per-thread 32-byte row stores this replaces touch 32 cache lines per warp instruction.
template <int D>
__device__ __forceinline__ void store_rows_tma(const CUtensorMap* map, uint32_t t_o, uint64_t il,
                                               uint32_t stage, int lane, int head0, int tok0,
                                               uint64_t policy) {
  const uint32_t row_addr = stage + static_cast<uint32_t>(lane) * 64u;
  const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
  for (int ch2 = 0; ch2 < D / 64; ++ch2) {
    uint32_t r[2][32];
    tmem_ld32(t_o + ch2 * 64, r[0]);
    tmem_ld32(t_o + ch2 * 64 + 32, r[1]);
    tmem_wait_ld_dep(r[0]);
    reg_dep(r[1]);
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float lo, hi;
        f2_split(f2_mul(f2(__uint_as_float(r[h][2 * e]), __uint_as_float(r[h][2 * e + 1])), il),
                 lo, hi);
        pk[e] = pack_bf16(lo, hi);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st_shared_v4(row_addr + static_cast<uint32_t>(h) * 2048u +
                         16u * (static_cast<uint32_t>(c) ^ sw),
                     pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d_hint(map, stage, ch2 * 64, head0, tok0, policy);
      tma_store_3d_hint(map, stage + 2048u, ch2 * 64 + 32, head0, tok0, policy);
      bulk_commit_group();
    }
    __syncwarp();  // converged again before the next .sync.aligned tcgen05.ld
  }
}

// The same with all D columns staged (4 KB per 64 columns) before one proxy fence and the
// stores: one wait, before the staging is written, for the previous item's stores to have
// read it.
template <int D>
__device__ __forceinline__ void store_rows_tma_all(const CUtensorMap* map, uint32_t t_o,
                                                   uint64_t il, uint32_t stage, int lane,
                                                   int head0, int tok0, uint64_t policy) {
  const uint32_t row_addr = stage + static_cast<uint32_t>(lane) * 64u;
  const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
  if (lane == 0) bulk_wait_group_read<0>();
  __syncwarp();
#pragma unroll
  for (int ch2 = 0; ch2 < D / 64; ++ch2) {
    uint32_t r[2][32];
    tmem_ld32(t_o + ch2 * 64, r[0]);
    tmem_ld32(t_o + ch2 * 64 + 32, r[1]);
    tmem_wait_ld_dep(r[0]);
    reg_dep(r[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float lo, hi;
        f2_split(f2_mul(f2(__uint_as_float(r[h][2 * e]), __uint_as_float(r[h][2 * e + 1])), il),
                 lo, hi);
        pk[e] = pack_bf16(lo, hi);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st_shared_v4(row_addr + static_cast<uint32_t>(ch2) * 4096u +
                         static_cast<uint32_t>(h) * 2048u + 16u * (static_cast<uint32_t>(c) ^ sw),
                     pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
#pragma unroll
    for (int b = 0; b < 2 * (D / 64); ++b)
      tma_store_3d_hint(map, stage + 2048u * b, 32 * b, head0, tok0, policy);
    bulk_commit_group();
  }
  __syncwarp();  // converged again before the next .sync.aligned tcgen05.ld
}

// ---------------------------------------------------------------------------------
// Softmax of one S tile: one thread per row, NC columns; P = 2^(s c - m) is written back
// to TMEM as bf16 pairs (times pscale = v_scale on the anchor tiles of the FP8 variant)
// over the upper half of the S columns, and l accumulates the unscaled P.
//
// Two kernels share this code:
//  * the fast kernel uses m = 0 throughout: no max pass and no rescale of O. An item with
//    a valid row outside the fast-kernel bounds (P could overflow, or all of it
//    underflow: tested on l) is listed for the exact kernel, which writes its output
//    rows again;
//  * the exact kernel recomputes those items with the usual online softmax (lazy rescale
//    of O past 2^kRescaleThreshold).

template <int NC>
__device__ __forceinline__ void load_s(uint32_t t_s, bool masked, int lo_c, int hi_c,
                                       float (&s)[NC]) {
  uint32_t r[NC / 32][32];
#pragma unroll
  for (int ch = 0; ch < NC / 32; ++ch) tmem_ld32(t_s + ch * 32, r[ch]);
  tmem_wait_ld_dep(r[0]);
#pragma unroll
  for (int ch = 1; ch < NC / 32; ++ch) reg_dep(r[ch]);
#pragma unroll
  for (int j = 0; j < NC; ++j) s[j] = __uint_as_float(r[j / 32][j % 32]);
  if (masked) {
#pragma unroll
    for (int j = 0; j < NC; ++j)
      if (j < lo_c || j > hi_c) s[j] = -INFINITY;
  }
}

// P = 2^(s c - m_safe) for all NC columns, packed in bf16 pairs (times pscale if SCALED)
// and stored to TMEM at t_p 32 columns (16 packed) at a time as they are made; returns
// the row sum of the unscaled P.
template <int NC, bool SCALED>
__device__ __forceinline__ float exp_store(const float (&s)[NC], float c, float m_safe,
                                           float pscale, uint32_t t_p) {
  const uint64_t cc = f2(c, c);
  const uint64_t nm = f2(-m_safe, -m_safe);
  const uint64_t ps = f2(pscale, pscale);
  uint64_t acc[4] = {0, 0, 0, 0};  // four packed partial sums (+0.0f bit patterns)
#pragma unroll
  for (int ch = 0; ch < NC / 32; ++ch) {
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int e = ch * 32 + 2 * j;
      const uint64_t x = f2_fma(f2(s[e], s[e + 1]), cc, nm);
      float x0, x1;
      f2_split(x, x0, x1);
      const uint64_t pp = f2(ex2(x0), ex2(x1));
      acc[j & 3] = f2_add(acc[j & 3], pp);
      float p0, p1;
      f2_split(SCALED ? f2_mul(pp, ps) : pp, p0, p1);
      pk[j] = pack_bf16(p0, p1);
    }
    tmem_st16(t_p + ch * 16, pk);
  }
  const uint64_t acc2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
  float sa, sb;
  f2_split(acc2, sa, sb);
  return sa + sb;
}

template <int NC>
__device__ __forceinline__ float row_max(const float (&s)[NC]) {
  float m8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
  for (int j = 8; j + 16 <= NC; j += 16)
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = max3(m8[i], s[j + i], s[j + 8 + i]);
  if ((NC - 8) % 16) {
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], s[NC - 8 + i]);
  }
  return fmaxf(max3(m8[0], m8[1], m8[2]), fmaxf(max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])));
}

// Exact online softmax (the recompute kernel).
template <int NC, int D, bool SCALED>
__device__ __forceinline__ void softmax_tile_exact(uint32_t t_s, uint32_t t_o, bool first_tile,
                                                   bool masked, int lo_c, int hi_c, float c,
                                                   float pscale, float& m_used, float& l) {
  float s[NC];
  load_s<NC>(t_s, masked, lo_c, hi_c, s);
  const float m_tile = row_max<NC>(s) * c;
  float alpha = 1.0f;
  bool rescale = false;
  if (first_tile) {
    m_used = m_tile;
  } else if (m_tile > m_used + kRescaleThreshold) {
    alpha = ex2(m_used - m_tile);
    m_used = m_tile;
    rescale = true;
  }
  const float m_safe = (m_used == -INFINITY) ? 0.0f : m_used;
  const float sum = exp_store<NC, SCALED>(s, c, m_safe, pscale, t_s + NC / 2);
  l = l * alpha + sum;
  // The PV of the previous tile is complete (the commit that signalled this S tile
  // tracks every earlier MMA), and the PV of this tile waits for this warpgroup's P,
  // so O can be rescaled in place here.
  if (__any_sync(0xFFFFFFFFu, rescale)) {
    const uint64_t aa = f2(alpha, alpha);
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t o[32];
      tmem_ld32(t_o + ch * 32, o);
      tmem_wait_ld_dep(o);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float lo, hi;
        f2_split(f2_mul(f2(__uint_as_float(o[2 * j]), __uint_as_float(o[2 * j + 1])), aa), lo, hi);
        o[2 * j] = __float_as_uint(lo);
        o[2 * j + 1] = __float_as_uint(hi);
      }
      tmem_st32(t_o + ch * 32, o);
    }
  }
  tmem_wait_st();
}

// Fast kernel: P = 2^(s c - m_ref) against a fixed reference m_ref, the row max of the
// item's first tile (0 when the row sees no key of that tile): one max pass per item
// instead of one per tile, and no rescale of O afterwards. Wide logit ranges stay on the
// fast path as long as no later tile exceeds the first one's max by ~2^32 in P.
template <int NC, bool SCALED>
__device__ __forceinline__ void softmax_tile_spec(uint32_t t_s, bool first, bool masked,
                                                  int lo_c, int hi_c, float c, float pscale,
                                                  float& m_ref, float& l) {
  float s[NC];
  load_s<NC>(t_s, masked, lo_c, hi_c, s);
  if (first) {
    const float m = row_max<NC>(s) * c;
    m_ref = (m == -INFINITY) ? 0.0f : m;
  }
  l += exp_store<NC, SCALED>(s, c, m_ref, pscale, t_s + NC / 2);
  tmem_wait_st();
}

// ---------------------------------------------------------------------------------
// EXACT = false: the fast kernel over all work items. EXACT = true: the exact kernel over
// the items the fast kernel listed in redo_list (its CTAs return at once if none).
// AMAX (fast kernel of the causal prefill only): the producer also takes max |k| and
// max |v| of every suffix token row, from each tile it is about to overwrite.
template <int D, bool FP8, bool EXACT, bool AMAX>
__global__ void __launch_bounds__(kThreads, 1)
cascade_attn_kernel(const __grid_constant__ CascadeParams p,
                    const __grid_constant__ CascadeMaps maps) {
  using C = Cfg<D>;
  // work items this kernel walks; position i of the walk is item item_id(i)
  const int total_items = EXACT ? *p.redo_count : __ldg(p.prefix + p.num_anchors);
  if (EXACT && static_cast<int>(blockIdx.x) >= total_items) return;
  auto item_id = [&](int i) { return EXACT ? __ldg(p.redo_list + i) : i; };
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::kSmemQ;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kSmemQ + C::kSmemKV);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int q = 0; q < 2; ++q) {
      mbar_init(&bars->q_full[q], 1);
      mbar_init(&bars->q_empty[q], 1);
      mbar_init(&bars->s_full[q], 1);
      // one arrival per softmax warp and one from the fill checker
      mbar_init(&bars->p_full[q], 5);
      mbar_init(&bars->o_done[q], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  WaitCtl wc;
  wc.timeout_ns = p.timeout_ns;
  wc.abort_flag = &bars->abort_flag;
  wc.err_word = p.err_word;

  const int tok = p.tok_per_tile;
  const int G = p.group;
  const int hkv = p.hkv;
  const int stride = gridDim.x;

  if (warp >= 8) {
   // ------------------------------------ warpgroup 2: producer, MMA, fill checker, idle
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg<D>::kRegsOther));
   if (warp == kWarpProducer) {
    // The whole warp walks the schedule (so every operand is warp-uniform); one elected
    // lane issues the TMA copies and the expect-tx arrivals.
    {
      const bool leader = elect_one();
      if (leader) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k_anc);
        tma_prefetch_desc(&maps.v_anc);
        tma_prefetch_desc(&maps.k_suf);
        tma_prefetch_desc(&maps.v_suf);
      }
      const uint64_t keep = l2_policy_evict_last(), stream_pol = l2_policy_evict_first();
      uint32_t kv_seq = 0, it_count = 0;
      uint32_t k_arm[4] = {0, 0, 0, 0}, v_arm[4] = {0, 0, 0, 0};
      bool skip_pending = p.inject_skip_first_kv != 0;
      bool ok = true;
      // AMAX: per-row max |x| of the K (kv = 0) or V (kv = 1) tile in `slot`, over the rows
      // that are query tokens of the item that loaded it (each suffix token row is one of
      // those exactly once per KV head). One lane per row: the row's 2 D bytes are D / 64
      // 128-byte rows of the swizzled tile (the swizzle permutes 16-byte chunks within a
      // row only, and a max does not care about order), read as 2 D / 16 independent
      // 16-byte loads; rows r..r+31 fall on 8 bank groups, so each load takes the minimum
      // 4 wavefronts.
      auto read_own = [&](int slot, int kv) {
        if (!AMAX) return;
        const int* rc = bars->rec[slot];
        const uint8_t* tile = sKV + slot * 2 * C::kTileBytes + kv * C::kTileBytes;
        const int base = rc[0], g_rec = rc[5];
        for (int qq = 0; qq < 2; ++qq) {
          const int lo = rc[1 + 2 * qq], hi = rc[2 + 2 * qq];
          for (int r0 = lo; r0 < hi; r0 += 32) {
            const int r = r0 + lane;
            if (r < hi) {
              const uint8_t* row = tile + (r - base) * 128;
              uint32_t m = 0;
              // plain loads (not volatile asm), so that all of the row's loads are issued
              // before the first max waits on one
              uint4 w[C::kKB * 8];
#pragma unroll
              for (int kb = 0; kb < C::kKB; ++kb)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  w[kb * 8 + c] = *reinterpret_cast<const uint4*>(row + kb * C::kBlockBytes + c * 16);
#pragma unroll
              for (int i = 0; i < C::kKB * 8; ++i) {
                m = absmax_bf16x2(m, w[i].x);
                m = absmax_bf16x2(m, w[i].y);
                m = absmax_bf16x2(m, w[i].z);
                m = absmax_bf16x2(m, w[i].w);
              }
              p.rowmax[(static_cast<int64_t>(r) * hkv + g_rec) * 2 + kv] =
                  static_cast<uint16_t>(max(m & 0xFFFFu, m >> 16));
            }
          }
        }
      };
      // AMAX: slots whose K / V tile still has own rows to read (bit per slot). They are
      // read while the producer would otherwise wait (a tile that has landed, polled
      // without blocking, before each wait for a free slot), and at the latest just
      // before the slot is overwritten.
      uint32_t pend_k = 0, pend_v = 0;
      auto landed = [&](uint64_t* bar, uint32_t parity) {
        return __shfl_sync(0xFFFFFFFFu, mbar_test_wait(smem_u32(bar), parity) ? 1 : 0, 0) != 0;
      };
      auto service = [&]() {
        if constexpr (AMAX) {
          for (int s2 = 0; s2 < C::kStages; ++s2) {
            if ((pend_k >> s2 & 1u) && landed(&bars->k_full[s2], (k_arm[s2] - 1) & 1u)) {
              read_own(s2, 0);
              pend_k &= ~(1u << s2);
            }
            if ((pend_v >> s2 & 1u) && landed(&bars->v_full[s2], (v_arm[s2] - 1) & 1u)) {
              read_own(s2, 1);
              pend_v &= ~(1u << s2);
            }
          }
        }
      };
      int item = blockIdx.x;
      Item it = item < total_items ? load_item<EXACT>(p, item_id(item)) : Item{};
      for (; ok && item < total_items; item += stride, ++it_count) {
        const Item nxt = item + stride < total_items ? load_item<EXACT>(p, item_id(item + stride)) : it;
        const int nA = it.n_anchor_tiles();
        const int n_tiles = it.n_tiles();
        const bool sh = it.sfx_shared();
        const int g = it.ag % hkv;
        // Suffix tiles of a window longer than one tile (a long sequence) are re-read by
        // every later query tile of that sequence: keep them in L2 like anchor tiles.
        // Short windows (join) are read by one or two items: stream them.
        const uint64_t sfx_pol = it.n_sfx_tiles() > 1 ? keep : stream_pol;
        for (int pos = 0; pos < n_tiles; ++pos, ++kv_seq) {
          const int slot = kv_seq % C::kStages;
          const uint32_t ph = (kv_seq / C::kStages) & 1u;
          const CUtensorMap* mk;
          const CUtensorMap* mv;
          int row;
          uint64_t pol;
          if (pos < nA) {
            mk = &maps.k_anc;
            mv = &maps.v_anc;
            row = it.a_tok0 + pos * kBN;
            pol = keep;
          } else {
            const int rel = pos - nA;
            mk = &maps.k_suf;
            mv = &maps.v_suf;
            row = sh ? it.ws0 + rel * kBN : it.ws(rel & 1) + (rel >> 1) * kBN;
            pol = sfx_pol;
          }
          uint8_t* k_dst = sKV + slot * 2 * C::kTileBytes;
          uint8_t* v_dst = k_dst + C::kTileBytes;
          service();
          if (!(ok = wait_parity_warp(wc, &bars->k_empty[slot], ph ^ 1u))) break;
          // the slot's previous tile is consumed and has landed: its own K rows, if not
          // read yet, before the load below overwrites them
          if (AMAX && (pend_k >> slot & 1u)) {
            read_own(slot, 0);
            pend_k &= ~(1u << slot);
          }
          if (skip_pending) {
            skip_pending = false;  // fault injection: this tile's K never arrives
          } else {
            ++k_arm[slot];
            if (leader) {
              mbar_arrive_expect_tx(&bars->k_full[slot], C::kTileBytes);
              for (int kb = 0; kb < C::kKB; ++kb)
                tma_load_3d_hint(mk, &bars->k_full[slot], k_dst + kb * C::kBlockBytes, kb * 64, g,
                                 row, pol);
            }
            __syncwarp();
          }
          service();
          if (!(ok = wait_parity_warp(wc, &bars->v_empty[slot], ph ^ 1u))) break;
          if (AMAX) {
            if (pend_v >> slot & 1u) read_own(slot, 1);
            // record this tile: own rows of the query tiles whose window it covers
            bool own = false;
            for (int qq = 0; qq < 2; ++qq) {
              const int rel = pos - nA;
              const bool mine = pos >= nA && (sh || (rel & 1) == qq);
              own |= mine && min(it.tend(qq), row + kBN) > max(it.t0 + qq * tok, row);
            }
            __syncwarp();
            if (lane == 0) {
              int* rc = bars->rec[slot];
              rc[0] = row;
              rc[5] = g;
              for (int qq = 0; qq < 2; ++qq) {
                const int rel = pos - nA;
                const bool mine = pos >= nA && (sh || (rel & 1) == qq);
                rc[1 + 2 * qq] = mine ? max(it.t0 + qq * tok, row) : 0;
                rc[2 + 2 * qq] = mine ? min(it.tend(qq), row + kBN) : 0;
              }
            }
            __syncwarp();
            // the K half of this slot is being loaded too (above)
            pend_k = own ? (pend_k | (1u << slot)) : (pend_k & ~(1u << slot));
            pend_v = own ? (pend_v | (1u << slot)) : (pend_v & ~(1u << slot));
          }
          ++v_arm[slot];
          if (leader) {
            mbar_arrive_expect_tx(&bars->v_full[slot], C::kTileBytes);
            for (int kb = 0; kb < C::kKB; ++kb)
              tma_load_3d_hint(mv, &bars->v_full[slot], v_dst + kb * C::kBlockBytes, kb * 64, g,
                               row, pol);
          }
          __syncwarp();
        }
        it = nxt;
      }
      // Let every load that was issued land before the CTA can exit.
      const uint64_t dl = global_timer_ns() + 100000000ull;
      for (int s = 0; s < C::kStages; ++s) {
        bool landed = true;
        if (k_arm[s]) landed &= drain_wait(&bars->k_full[s], (k_arm[s] - 1) & 1u, dl);
        if (v_arm[s]) landed &= drain_wait(&bars->v_full[s], (v_arm[s] - 1) & 1u, dl);
        // AMAX: the tiles still in the ring were never overwritten; read them now
        if (AMAX && ok && landed && k_arm[s] && v_arm[s]) {
          if (pend_k >> s & 1u) read_own(s, 0);
          if (pend_v >> s & 1u) read_own(s, 1);
        }
      }
    }
   } else if (warp == kWarpQLoad) {
    // ------------------------------------------------ query loader
    // Each item's two query tiles load as soon as their buffers are free (the commit after
    // the previous item's last S of that tile), apart from the K/V ring: a producer that
    // issued them in ring order held them back until a K/V slot freed, and the next item's
    // first S then waited for the query tile at every item boundary.
    const bool leader = elect_one();
    const uint64_t stream_pol = l2_policy_evict_first();
    uint32_t it_count = 0, q_arm[2] = {0, 0};
    bool ok = true;
    int item = blockIdx.x;
    Item it = item < total_items ? load_item<EXACT>(p, item_id(item)) : Item{};
    for (; ok && item < total_items; item += stride, ++it_count) {
      const Item nxt = item + stride < total_items ? load_item<EXACT>(p, item_id(item + stride)) : it;
      const int g = it.ag % hkv;
      for (int q = 0; q < 2 && ok; ++q) {
        if (!(ok = wait_parity_warp(wc, &bars->q_empty[q], (it_count & 1u) ^ 1u))) break;
        ++q_arm[q];
        if (leader) {
          mbar_arrive_expect_tx(&bars->q_full[q], C::kTileBytes);
          for (int kb = 0; kb < C::kKB; ++kb)
            tma_load_3d_hint(&maps.q, &bars->q_full[q], sQ + q * C::kTileBytes + kb * C::kBlockBytes,
                             kb * 64, g * G, it.t0 + q * tok, stream_pol);
        }
        __syncwarp();
      }
      it = nxt;
    }
    const uint64_t dl = global_timer_ns() + 100000000ull;
    for (int q = 0; q < 2; ++q)
      if (q_arm[q]) drain_wait(&bars->q_full[q], (q_arm[q] - 1) & 1u, dl);
   } else if (warp == kWarpFillCheck) {
    // ------------------------------------------------ fill checker
    // For every group {PV(q,k), S(q,k+1)}: wait until the V(q,k) and K(q,k+1) fills it
    // reads have landed, then add the fifth arrival on p_full[q]. Before arriving for a
    // group it waits for the previous phase of p_full[q] to complete, so it never gives
    // two arrivals to one phase.
    uint32_t kv_base = 0, arrived[2] = {0, 0};
    bool ok = true;
    int item = blockIdx.x;
    Item it = item < total_items ? load_item<EXACT>(p, item_id(item)) : Item{};
    for (; ok && item < total_items; item += stride) {
      const Item nxt = item + stride < total_items ? load_item<EXACT>(p, item_id(item + stride)) : it;
      const int nA = it.n_anchor_tiles();
      const int nS = it.n_sfx_tiles();
      const int n = nA + nS;
      const bool sh = it.sfx_shared();
      for (int k = 0; ok && k < n; ++k) {
        for (int q = 0; ok && q < 2; ++q) {
          // shared tiles are checked once, for query tile 0 (whose group runs first)
          if ((k >= nA && !sh) || q == 0) {
            const uint32_t seq = kv_base + pos_of(nA, sh, q, k);
            ok = wait_parity_warp(wc, &bars->v_full[seq % C::kStages], (seq / C::kStages) & 1u);
          }
          if (ok && k + 1 < n && ((k + 1 >= nA && !sh) || q == 0)) {
            const uint32_t seq = kv_base + pos_of(nA, sh, q, k + 1);
            ok = wait_parity_warp(wc, &bars->k_full[seq % C::kStages], (seq / C::kStages) & 1u);
          }
          if (ok && arrived[q] > 0)
            ok = wait_parity_warp(wc, &bars->p_full[q], (arrived[q] - 1) & 1u);
          if (!ok) break;
          ++arrived[q];
          if (lane == 0) mbar_arrive(&bars->p_full[q]);
          __syncwarp();
        }
      }
      kv_base += it.n_tiles();
      it = nxt;
    }
   } else if (warp == kWarpMma) {
    // Whole warp walks the schedule; one elected lane issues tcgen05.mma / commit.
    {
      const bool leader = elect_one();
      constexpr uint32_t kAB = 1u;  // operand type bf16 (A and B)
      constexpr uint32_t kIdescS128 = idesc_f16(kBM, 128, kAB, 0);
      constexpr uint32_t kIdescS64 = idesc_f16(kBM, 64, kAB, 0);
      constexpr uint32_t kIdescPV = idesc_f16(kBM, D, kAB, 1);
      constexpr uint32_t kDescHi = sw128_desc_hi(1024);  // 8-row groups 1024 bytes apart
      const uint32_t q_lo0 = sw128_desc_lo(smem_u32(sQ), 16);
      const uint32_t k_lo0 = sw128_desc_lo(smem_u32(sKV), 16);
      // V is the MN-major B operand: 64-column blocks (128 rows x 128 bytes) 16 KB apart
      const uint32_t v_lo0 = sw128_desc_lo(smem_u32(sKV + C::kTileBytes), C::kBlockBytes);
      uint32_t kv_base = 0, it_count = 0;
      uint32_t p_cnt[2] = {0, 0};
      bool ok = true;
      int item = blockIdx.x;
      Item it = item < total_items ? load_item<EXACT>(p, item_id(item)) : Item{};
      for (; ok && item < total_items; item += stride, ++it_count) {
        const Item nxt = item + stride < total_items ? load_item<EXACT>(p, item_id(item + stride)) : it;
        const int nA = it.n_anchor_tiles();
        const int nS = it.n_sfx_tiles();
        const int nk_sfx = it.nk_sfx();
        const int n = nA + nS;
        const bool sh = it.sfx_shared();

        // Waits (K fill, Q fill) for S(q, k) and (V fill, P ready) for PV(q, k); the MMAs
        // are issued only after every wait of the next pair of groups is done, so PV(q, k)
        // and S(q, k + 1) go to the tensor pipe back to back. The fill checker warp folds
        // the V(q,k) and K(q,k+1) fills into p_full[q], so after the first group of an
        // item the MMA warp waits once per group: an mbarrier wait costs
        // it a few hundred cycles while the tensor pipe reads shared memory, and the pipe's
        // queue holds only about two MMAs.
        auto wait_s = [&](int q, int k) -> bool {
          const uint32_t seq = kv_base + pos_of(nA, sh, q, k);
          const int slot = seq % C::kStages;
          const uint32_t ph = (seq / C::kStages) & 1u;
          const bool own = k >= nA && !sh;  // the query tile's own suffix tile
          if ((own || q == 0) && !wait_parity_warp(wc, &bars->k_full[slot], ph))
            return false;
          if (k == 0 && !wait_parity_warp(wc, &bars->q_full[q], it_count & 1u)) return false;
          return true;
        };
        auto wait_pv = [&](int q) -> bool {
          if (!wait_parity_warp(wc, &bars->p_full[q], p_cnt[q] & 1u)) return false;
          ++p_cnt[q];
          return true;
        };
        // Issue parts: called by the elected lane only.
        auto mma_s = [&](int q, int k) {
          const uint32_t seq = kv_base + pos_of(nA, sh, q, k);
          const int slot = seq % C::kStages;
          const bool sfx = k >= nA;
          const uint32_t k_lo = k_lo0 + slot * (2 * C::kTileBytes >> 4);
          const uint32_t q_lo = q_lo0 + q * (C::kTileBytes >> 4);
          const uint32_t idesc = (!sfx || nk_sfx == 128) ? kIdescS128 : kIdescS64;
          const uint32_t d_s = tmem + 256u * q;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // K step kk: 128-byte block kk / 4, 32-byte column offset (kk % 4) inside it
            const uint32_t adv = (kk >> 2) * (C::kBlockBytes >> 4) + (kk & 3) * 2;
            mma_ss_lohi(d_s, q_lo + adv, kDescHi, k_lo + adv, kDescHi, idesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[q]);
          if ((k >= nA && !sh) || q == 1) mma_commit(&bars->k_empty[slot]);
          if (k == n - 1) mma_commit(&bars->q_empty[q]);
        };
        auto mma_pv = [&](int q, int k) {
          const uint32_t seq = kv_base + pos_of(nA, sh, q, k);
          const int slot = seq % C::kStages;
          const bool sfx = k >= nA;
          const uint32_t v_lo = v_lo0 + slot * (2 * C::kTileBytes >> 4);
          const uint32_t d_o = tmem + 256u * q + 128u;
          // P sits over the upper half of the S columns (64 of 128, or 32 of 64)
          const uint32_t a_p = tmem + 256u * q + ((sfx && nk_sfx == 64) ? 32u : 64u);
          const uint32_t acc0 = k > 0 ? 1u : 0u;
          // 16 keys per step: 16 rows of 128 bytes of V; P columns advance by 8 (2 x bf16)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts_lohi(d_o, a_p + 8u * kk, v_lo + kk * 128, kDescHi, kIdescPV, kk > 0 ? 1u : acc0);
          if (!sfx || nk_sfx == 128) {
#pragma unroll
            for (int kk = 4; kk < 8; ++kk)
              mma_ts_lohi(d_o, a_p + 8u * kk, v_lo + kk * 128, kDescHi, kIdescPV, 1u);
          }
          if ((k >= nA && !sh) || q == 1) mma_commit(&bars->v_empty[slot]);
          if (k == n - 1) mma_commit(&bars->o_done[q]);
        };

        // S(0,0) goes as soon as its own K and Q fills are in (the Q fills of an item land
        // one after the other).
        for (int q = 0; q < 2 && ok; ++q) {
          ok = wait_s(q, 0);
          if (ok) {
            tc_fence_after();
            if (leader) mma_s(q, 0);
            __syncwarp();
          }
        }
        for (int k = 0; ok && k < n; ++k) {
          for (int q = 0; q < 2 && ok; ++q) {
            // the fill checker's arrival on p_full covers V(q,k) and K(q,k+1)
            ok = wait_pv(q);
            if (!ok) break;
            tc_fence_after();
            if (leader) {
              mma_pv(q, k);
              if (k + 1 < n) mma_s(q, k + 1);
            }
            __syncwarp();
          }
        }
        kv_base += it.n_tiles();
        it = nxt;
      }
      // Every MMA issued so far has completed once this barrier flips.
      if (leader) mma_commit(&bars->drain);
      __syncwarp();
      drain_wait(&bars->drain, 0, global_timer_ns() + 100000000ull);
    }
   }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg<D>::kRegsSoftmax));
    const int q = warp >> 2;
    const int row = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + 256u * q;
    const uint32_t t_o = t_s + 128u;
    const uint32_t stage = smem_u32(smem + C::kSmemQ + C::kSmemKV + 1024) + warp * kStageWarpBytes;
    const uint64_t out_pol = l2_policy_evict_first();
    uint32_t s_cnt = 0, it_count = 0;
    bool ok = true;
    const float c = p.scale_log2;
    int item = blockIdx.x;
    Item it = item < total_items ? load_item<EXACT>(p, item_id(item)) : Item{};
    for (; ok && item < total_items; item += stride, ++it_count) {
      const Item nxt = item + stride < total_items ? load_item<EXACT>(p, item_id(item + stride)) : it;
      const int nA = it.n_anchor_tiles();
      const int n = nA + it.n_sfx_tiles();
      const int nk_sfx = it.nk_sfx();
      const int g = it.ag % hkv;
      const int t = it.t0 + q * tok + row / G;
      const bool valid = t < it.tend(q);
      // visible suffix keys of this row: [vis_lo, t] (first used on the suffix tiles)
      const int vis_lo = valid ? __ldg(p.seg + t) : t;
      const int ws_q = it.ws(q);
      // FP8 anchor tiles: scores use c * k_scale, and P carries v_scale
      const float c_anc = FP8 ? c * __ldg(p.k_scale + it.ag) : c;
      const float v_sc = FP8 ? __ldg(p.v_scale + it.ag) : 1.0f;
      float m_used = EXACT ? -INFINITY : 0.0f, l = 0.0f;  // fast: set by the first tile
      for (int k = 0; k < n; ++k) {
        if (!(ok = wait_parity(wc, &bars->s_full[q], s_cnt & 1u))) break;
        ++s_cnt;
        tc_fence_after();
        if (k < nA) {
          const int rem = it.la - k * kBN;
          if (EXACT)
            softmax_tile_exact<128, D, FP8>(t_s, t_o, k == 0, rem < kBN, 0, rem - 1, c_anc,
                                            v_sc, m_used, l);
          else
            softmax_tile_spec<128, FP8>(t_s, k == 0, rem < kBN, 0, rem - 1, c_anc, v_sc,
                                        m_used, l);
        } else {
          const int base = ws_q + (k - nA) * kBN;
          const int lo_c = vis_lo - base, hi_c = t - base;
          // the column mask is skipped when every row of the warp sees the whole tile
          // (the tiles below the diagonal of a long suffix)
          const bool mk = __any_sync(0xFFFFFFFFu, lo_c > 0 || hi_c < nk_sfx - 1);
          if (EXACT) {
            if (nk_sfx == 64)
              softmax_tile_exact<64, D, false>(t_s, t_o, k == 0, mk, lo_c, hi_c, c, 1.0f,
                                               m_used, l);
            else
              softmax_tile_exact<128, D, false>(t_s, t_o, k == 0, mk, lo_c, hi_c, c, 1.0f,
                                                m_used, l);
          } else {
            if (nk_sfx == 64)
              softmax_tile_spec<64, false>(t_s, k == 0, mk, lo_c, hi_c, c, 1.0f, m_used, l);
            else
              softmax_tile_spec<128, false>(t_s, k == 0, mk, lo_c, hi_c, c, 1.0f, m_used, l);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[q]);
      }
      if (!ok) break;
      // Fast kernel: hand the item to the exact kernel if a valid row left the bounds
      // (its output rows are then written again).
      const bool broke = !(l >= kSpecSumLow && l <= kSpecSumHigh) ||
                         (FP8 && it.la > 0 && !(fabsf(v_sc) <= kSpecScaleHigh));
      if (!EXACT && __any_sync(0xFFFFFFFFu, broke && valid) && lane == 0) {
        const int id = item_id(item);
        if (atomicExch(p.redo_flag + id, 1) == 0) p.redo_list[atomicAdd(p.redo_count, 1)] = id;
      }
      __syncwarp();  // reconverge after the lane-0 branch (the TMEM loads are .aligned)
      if (!(ok = wait_parity(wc, &bars->o_done[q], it_count & 1u))) break;
      tc_fence_after();
      const int64_t orow = static_cast<int64_t>(t) * p.hq + g * G + (row % G);
      // This launch's partial: lse_own (natural log) and O / l. The suffix pass of the
      // two-pass variant may merge it with the anchor partial here (A4: LSE rescaling).
      const float lse_own = (m_used + __log2f(l)) * 0.69314718055994531f;
      float w_own = __fdividef(1.0f, l), w_part = 0.0f, lse_out = lse_own;
      const float* part = nullptr;
      if (p.mode == kSuffixPass && p.merge && valid) {
        const float lse_a = __ldg(p.lse_part + orow);
        if (lse_a > -INFINITY) {  // -inf: the anchor is empty, nothing to merge
          const float mx = fmaxf(lse_a, lse_own);
          const float ea = expf(lse_a - mx), es = expf(lse_own - mx);
          const float inv = 1.0f / (ea + es);
          lse_out = mx + logf(ea + es);
          w_part = ea * inv;
          w_own = es * inv / l;
          part = p.o_part + orow * D;
        }
      }
      const uint64_t wo = f2(w_own, w_own), wp = f2(w_part, w_part);
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + orow * D;
      float* out32 = p.mode == kAnchorPass ? p.o_part + orow * D : nullptr;
      if (p.mode == kFused && __all_sync(0xFFFFFFFFu, valid)) {
        store_rows_tma<D>(&maps.out, t_o, wo, stage, lane, g * G,
                          it.t0 + q * tok + (warp & 3) * (32 / G), out_pol);
      } else {
      // Two 32-column chunks of O per TMEM wait; each thread writes its row with 32-byte
      // stores (one full sector each): the rows of a partly valid warp and the
      // two-pass variant's outputs.
#pragma unroll
      for (int ch2 = 0; ch2 < D / 64; ++ch2) {
        uint32_t r[2][32];
        tmem_ld32(t_o + ch2 * 64, r[0]);
        tmem_ld32(t_o + ch2 * 64 + 32, r[1]);
        tmem_wait_ld_dep(r[0]);
        reg_dep(r[1]);
        if (valid) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col0 = ch2 * 64 + h * 32;
            if (out32 != nullptr) {  // anchor pass: fp32 normalised partial
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                uint32_t v[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  float lo, hi;
                  f2_split(f2_mul(f2(__uint_as_float(r[h][8 * j + 2 * e]),
                                     __uint_as_float(r[h][8 * j + 2 * e + 1])), wo), lo, hi);
                  v[2 * e] = __float_as_uint(lo);
                  v[2 * e + 1] = __float_as_uint(hi);
                }
                st_global_v8(out32 + col0 + 8 * j, v);
              }
              continue;
            }
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              uint64_t o = f2_mul(f2(__uint_as_float(r[h][2 * j]),
                                     __uint_as_float(r[h][2 * j + 1])), wo);
              if (part != nullptr) {
                const float2 a2 = *reinterpret_cast<const float2*>(part + col0 + 2 * j);
                o = f2_fma(f2(a2.x, a2.y), wp, o);
              }
              float lo, hi;
              f2_split(o, lo, hi);
              pk[j] = pack_bf16(lo, hi);
            }
            st_global_v8(out + col0, pk);
            st_global_v8(out + col0 + 16, pk + 8);
          }
        }
      }
      }
      if (valid) {
        if (p.mode == kAnchorPass)
          p.lse_part[orow] = lse_own;
        else if (p.lse != nullptr)
          p.lse[orow] = lse_out;
      }
      it = nxt;
    }
    // the output stores have read their staging buffers and written global memory
    if (lane == 0) bulk_wait_group_all();
    tc_fence_before();
  }

  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// =================================================================================
// The fast kernel on CTA pairs (d = 128): tcgen05.mma.cta_group::2, M = 256.
//
// A cluster of two CTAs takes a "quad" work item: (anchor, KV head, four 128-row query
// tiles over 4 x 128 / G consecutive suffix tokens). Query tile j of the quad is held by
// CTA j % 2 as its pair tile q = j / 2: pair tile q is one M = 256 MMA over query tiles 2q
// (rank 0) and 2q + 1 (rank 1), and each CTA still ping-pongs two pair tiles between its
// softmax warpgroups. Every K/V tile (128 keys) serves all four query tiles; each CTA
// loads and holds half of it: keys 64 r .. 64 r + 63 of the K tile (the N half of the B
// operand of S = Q K^T) and d columns 64 r .. 64 r + 63 of the V tile (the N half of the B
// operand of O += P V). Per SM and K16 step, S then reads 4 KB (its own query rows) + 2 KB
// (its K half) of shared memory instead of 8 KB, and each SM loads half of every K/V tile.
// Synchronisation: rank 0's MMA warp issues every MMA for both CTAs, and its commits
// arrive on the barrier of the same name in both CTAs (slot free, S ready, query tile
// free, O done). Both CTAs' TMA loads complete on rank 0's full barriers, for which rank 0
// expects both halves' bytes; both CTAs' softmax warps arrive on rank 0's P-ready barrier
// (9 arrivals: 2 x 4 softmax warps + rank 0's fill checker). Rank 1's MMA warp takes part
// only in the TMEM allocation and release. Barrier waits and remote arrivals keep the
// default CTA-scope semantics (no data moves through generic memory between the CTAs).
// Suffix tiles always use N = 128 (a 64-key tile would split 32 / 32 between the CTAs, not
// as the 64-row K halves are loaded).
template <int STAGES>
struct PairCfgT {
  static constexpr int kKB = 2;                          // 128-byte column blocks (d = 128)
  static constexpr int kBlockBytes = 128 * 128;          // 128 rows x 128 bytes
  static constexpr int kQTileBytes = 2 * kBlockBytes;    // one 128-row query tile
  static constexpr int kKHalfBlock = 64 * 128;           // 64 key rows x 128 bytes
  static constexpr int kKHalfBytes = 2 * kKHalfBlock;    // 64 keys x d
  static constexpr int kVHalfBytes = kBlockBytes;        // 128 keys x 64 d columns
  static constexpr int kStageBytes = kKHalfBytes + kVHalfBytes;
  // Query-tile buffers: query tile qq of the quad with walk count ic is query slot
  // j = 2 ic + qq, held in buffer j % kQBufs (its use j / kQBufs). A third or fourth
  // buffer (the next quad's queries loading a whole quad ahead, at the cost of a K/V
  // stage) measured no faster, nor did an L2 prefetch of the next quad's query rows.
  static constexpr int kQBufs = 2;  // the query loader puts slot 2 ic + qq in buffer qq
  // K/V ring depth: 4 stages, or 3 where the K/V stream is served from L2 (anchor K/V
  // well inside L2, one suffix tile per pair tile); the 32 KB that frees doubles each
  // softmax warp's epilogue staging, so all its output columns go out after one proxy
  // fence instead of two halves in turn.
  static constexpr int kStages = STAGES;
  static constexpr int kStageWarpBytes = STAGES == 4 ? 2 * 2048 : 4 * 2048;
  static constexpr int kSmemQ = kQBufs * kQTileBytes;
  static constexpr int kSmemKV = kStages * kStageBytes;
  static constexpr int kSmemBytes = kSmemQ + kSmemKV + 1024 + 8 * kStageWarpBytes + 1024;
};
static_assert(PairCfgT<4>::kSmemBytes <= 232448 && PairCfgT<3>::kSmemBytes <= 232448,
              "shared memory of one CTA");

struct Quad {
  int a_tok0, la, t0, ag;
  int wsp0, wsp1;          // key window start of pair tile 0 / 1 (its first token's suffix)
  int te0, te1, te2, te3;  // one past the last token of query tile j (its start when empty)
  // selects, not indexing: a dynamically indexed array would live in local memory
  __device__ __forceinline__ int wsp(int q) const { return q ? wsp1 : wsp0; }
  __device__ __forceinline__ int tend(int j) const {
    return j < 2 ? (j ? te1 : te0) : (j == 3 ? te3 : te2);
  }
  __device__ __forceinline__ int n_anchor_tiles() const { return (la + kBN - 1) / kBN; }
  __device__ __forceinline__ int n_sfx_tiles() const {
    const int w = max(max(max(te0, te1) - wsp0, max(te2, te3) - wsp1), 0);
    return (w + kBN - 1) / kBN;
  }
  __device__ __forceinline__ bool sfx_shared() const { return wsp0 == wsp1; }
  __device__ __forceinline__ int n_tiles() const {
    return n_anchor_tiles() + (sfx_shared() ? 1 : 2) * n_sfx_tiles();
  }
};
__device__ __forceinline__ Quad load_quad(const CascadeParams& p, int item) {
  const int4 a = ld_nc_v4(p.items + 12 * static_cast<int64_t>(item));
  const int4 b = ld_nc_v4(p.items + 12 * static_cast<int64_t>(item) + 4);
  const int4 c = ld_nc_v4(p.items + 12 * static_cast<int64_t>(item) + 8);
  Quad it;
  it.a_tok0 = a.x; it.la = a.y; it.t0 = a.z; it.ag = a.w;
  it.wsp0 = b.x; it.wsp1 = b.y; it.te0 = b.z; it.te1 = b.w;
  it.te2 = c.x; it.te3 = c.y;
  return it;
}

template <bool FP8, int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
cascade_pair_kernel(const __grid_constant__ CascadeParams p,
                    const __grid_constant__ CascadeMaps maps) {
  using C = PairCfgT<STAGES>;
  constexpr int D = 128;
  const int total_items = __ldg(p.prefix + p.num_anchors);  // quads
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::kSmemQ;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kSmemQ + C::kSmemKV);
  const uint32_t rank = cluster_ctarank();
  const bool lead = rank == 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b = 0; b < C::kQBufs; ++b) {
      mbar_init(&bars->q_full[b], 1);
      mbar_init(&bars->q_empty[b], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&bars->s_full[q], 1);
      mbar_init(&bars->p_full[q], 9);  // 2 x 4 softmax warps + the fill checker
      mbar_init(&bars->o_done[q], 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    bars->peer_abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc_pair(&bars->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrival or transfer
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  WaitCtl wc;
  wc.timeout_ns = p.timeout_ns;
  wc.abort_flag = &bars->abort_flag;
  wc.err_word = p.err_word;

  const int tok = p.tok_per_tile;
  const int G = p.group;
  const int hkv = p.hkv;
  const int stride = gridDim.x / 2;  // clusters
  const int first = blockIdx.x / 2;
  // rank 0's copy of a barrier, as a shared::cluster address
  auto lead_bar = [&](uint64_t* b) { return cluster_map(b, 0); };

  if (warp >= 8) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg<D>::kRegsOther));
   if (warp == kWarpProducer) {
    // both CTAs: their query tiles and their halves of every K/V tile
    const bool elect = elect_one();
    if (elect) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k_anc64);
      tma_prefetch_desc(&maps.v_anc);
      tma_prefetch_desc(&maps.k_suf64);
      tma_prefetch_desc(&maps.v_suf);
    }
    const uint64_t keep = l2_policy_evict_last(), stream_pol = l2_policy_evict_first();
    uint32_t kv_seq = 0, it_count = 0;
    uint32_t k_arm[4] = {0, 0, 0, 0}, v_arm[4] = {0, 0, 0, 0};
    bool skip_pending = lead && p.inject_skip_first_kv != 0;
    bool ok = true;
    int item = first;
    Quad it = item < total_items ? load_quad(p, item) : Quad{};
    for (; ok && item < total_items; item += stride, ++it_count) {
      const Quad nxt = item + stride < total_items ? load_quad(p, item + stride) : it;
      const int nA = it.n_anchor_tiles();
      const int n_tiles = it.n_tiles();
      const bool sh = it.sfx_shared();
      const int g = it.ag % hkv;
      const uint64_t sfx_pol = it.n_sfx_tiles() > 1 ? keep : stream_pol;
      for (int pos = 0; pos < n_tiles; ++pos, ++kv_seq) {
        const int slot = kv_seq % C::kStages;
        const uint32_t ph = (kv_seq / C::kStages) & 1u;
        const CUtensorMap* mk;
        const CUtensorMap* mv;
        int row;
        uint64_t pol;
        if (pos < nA) {
          mk = &maps.k_anc64;
          mv = &maps.v_anc;
          row = it.a_tok0 + pos * kBN;
          pol = keep;
        } else {
          const int rel = pos - nA;
          mk = &maps.k_suf64;
          mv = &maps.v_suf;
          row = sh ? it.wsp0 + rel * kBN : it.wsp(rel & 1) + (rel >> 1) * kBN;
          pol = sfx_pol;
        }
        uint8_t* k_dst = sKV + slot * C::kStageBytes;
        uint8_t* v_dst = k_dst + C::kKHalfBytes;
        if (!(ok = wait_parity_warp(wc, &bars->k_empty[slot], ph ^ 1u))) break;
        if (skip_pending) {
          skip_pending = false;  // fault injection: this K half never arrives
        } else {
          if (lead) ++k_arm[slot];
          if (elect) {
            if (lead) mbar_arrive_expect_tx(&bars->k_full[slot], 2 * C::kKHalfBytes);
            for (int kb = 0; kb < C::kKB; ++kb)
              tma_load_3d_pair(mk, lead_bar(&bars->k_full[slot]), k_dst + kb * C::kKHalfBlock,
                               kb * 64, g, row + 64 * static_cast<int>(rank), pol);
          }
          __syncwarp();
        }
        if (!(ok = wait_parity_warp(wc, &bars->v_empty[slot], ph ^ 1u))) break;
        if (lead) ++v_arm[slot];
        if (elect) {
          if (lead) mbar_arrive_expect_tx(&bars->v_full[slot], 2 * C::kVHalfBytes);
          tma_load_3d_pair(mv, lead_bar(&bars->v_full[slot]), v_dst,
                           64 * static_cast<int>(rank), g, row, pol);
        }
        __syncwarp();
      }
      it = nxt;
    }
    // rank 0: every load of the pair that was issued has landed before the CTAs exit
    // (rank 1's loads complete on rank 0's barriers)
    if (lead) {
      const uint64_t dl = global_timer_ns() + 100000000ull;
      for (int s = 0; s < C::kStages; ++s) {
        if (k_arm[s]) drain_wait(&bars->k_full[s], (k_arm[s] - 1) & 1u, dl);
        if (v_arm[s]) drain_wait(&bars->v_full[s], (v_arm[s] - 1) & 1u, dl);
      }
    }
   } else if (warp == kWarpQLoad) {
    // both CTAs: their query tiles. Query tile qq of the quad with walk count ic is query
    // slot 2 ic + qq, in buffer qq; each loads as soon as its buffer is free (the commit
    // after the previous quad's last S of that pair tile), apart from the K/V ring. The
    // waits run in slot order, so a buffer's empty barrier is at most one phase short of
    // the release a wait asks for.
    const bool elect = elect_one();
    const uint64_t stream_pol = l2_policy_evict_first();
    uint32_t it_count = 0, q_arm[2] = {0, 0};
    bool ok = true;
    int item = first;
    Quad it = item < total_items ? load_quad(p, item) : Quad{};
    for (; ok && item < total_items; item += stride, ++it_count) {
      const Quad nxt = item + stride < total_items ? load_quad(p, item + stride) : it;
      for (int qq = 0; qq < 2 && ok; ++qq) {
        if (!(ok = wait_parity_warp(wc, &bars->q_empty[qq], (it_count & 1u) ^ 1u))) break;
        if (lead) ++q_arm[qq];
        if (elect) {
          if (lead) mbar_arrive_expect_tx(&bars->q_full[qq], 2 * C::kQTileBytes);
          for (int kb = 0; kb < C::kKB; ++kb)
            tma_load_3d_pair(&maps.q, lead_bar(&bars->q_full[qq]),
                             sQ + qq * C::kQTileBytes + kb * C::kBlockBytes, kb * 64,
                             (it.ag % hkv) * G, it.t0 + (2 * qq + static_cast<int>(rank)) * tok,
                             stream_pol);
        }
        __syncwarp();
      }
      it = nxt;
    }
    // rank 0: every query load of the pair that was issued has landed before the CTAs exit
    if (lead) {
      const uint64_t dl = global_timer_ns() + 100000000ull;
      for (int b = 0; b < 2; ++b)
        if (q_arm[b]) drain_wait(&bars->q_full[b], (q_arm[b] - 1) & 1u, dl);
    }
   } else if (warp == kWarpFillCheck && lead) {
    // rank 0: the fill checker, as in the single-CTA kernel, on rank 0's full barriers
    uint32_t kv_base = 0, arrived[2] = {0, 0};
    bool ok = true;
    int item = first;
    Quad it = item < total_items ? load_quad(p, item) : Quad{};
    for (; ok && item < total_items; item += stride) {
      const Quad nxt = item + stride < total_items ? load_quad(p, item + stride) : it;
      const int nA = it.n_anchor_tiles();
      const int n = nA + it.n_sfx_tiles();
      const bool sh = it.sfx_shared();
      for (int k = 0; ok && k < n; ++k) {
        for (int q = 0; ok && q < 2; ++q) {
          if ((k >= nA && !sh) || q == 0) {
            const uint32_t seq = kv_base + pos_of(nA, sh, q, k);
            ok = wait_parity_warp(wc, &bars->v_full[seq % C::kStages], (seq / C::kStages) & 1u);
          }
          if (ok && k + 1 < n && ((k + 1 >= nA && !sh) || q == 0)) {
            const uint32_t seq = kv_base + pos_of(nA, sh, q, k + 1);
            ok = wait_parity_warp(wc, &bars->k_full[seq % C::kStages], (seq / C::kStages) & 1u);
          }
          if (ok && arrived[q] > 0)
            ok = wait_parity_warp(wc, &bars->p_full[q], (arrived[q] - 1) & 1u);
          if (!ok) break;
          ++arrived[q];
          if (lane == 0) mbar_arrive(&bars->p_full[q]);
          __syncwarp();
        }
      }
      kv_base += it.n_tiles();
      it = nxt;
    }
   } else if (warp == kWarpMma && lead) {
    // rank 0: every MMA of the pair
    const bool elect = elect_one();
    constexpr uint32_t kAB = 1u;  // bf16 A and B
    constexpr uint32_t kIdescS = idesc_f16(256, 128, kAB, 0);
    constexpr uint32_t kIdescPV = idesc_f16(256, D, kAB, 1);
    constexpr uint32_t kDescHi = sw128_desc_hi(1024);  // 8-row groups 1024 bytes apart
    const uint32_t q_lo0 = sw128_desc_lo(smem_u32(sQ), 16);
    const uint32_t k_lo0 = sw128_desc_lo(smem_u32(sKV), 16);
    // each CTA's V half is one 64-column block (128 rows x 128 bytes)
    const uint32_t v_lo0 = sw128_desc_lo(smem_u32(sKV + C::kKHalfBytes), C::kBlockBytes);
    uint32_t kv_base = 0, it_count = 0;
    uint32_t p_cnt[2] = {0, 0};
    bool ok = true;
    int item = first;
    Quad it = item < total_items ? load_quad(p, item) : Quad{};
    for (; ok && item < total_items; item += stride, ++it_count) {
      const Quad nxt = item + stride < total_items ? load_quad(p, item + stride) : it;
      const int nA = it.n_anchor_tiles();
      const int n = nA + it.n_sfx_tiles();
      const bool sh = it.sfx_shared();
      // this quad's query buffers (query slots 2 it_count and 2 it_count + 1, which the
      // query-loader warp fills)
      auto qbuf = [&](int q) { return static_cast<int>((2 * it_count + q) % C::kQBufs); };
      auto quse = [&](int q) { return ((2 * it_count + q) / C::kQBufs) & 1u; };
      auto wait_s = [&](int q, int k) -> bool {
        const uint32_t seq = kv_base + pos_of(nA, sh, q, k);
        const bool own = k >= nA && !sh;
        if ((own || q == 0) &&
            !wait_parity_warp(wc, &bars->k_full[seq % C::kStages], (seq / C::kStages) & 1u))
          return false;
        if (k == 0 &&
            !wait_parity_warp(wc, &bars->q_full[qbuf(q)], quse(q)))
          return false;
        return true;
      };
      auto wait_pv = [&](int q) -> bool {
        if (!wait_parity_warp(wc, &bars->p_full[q], p_cnt[q] & 1u)) return false;
        ++p_cnt[q];
        return true;
      };
      auto mma_s = [&](int q, int k) {
        const uint32_t seq = kv_base + pos_of(nA, sh, q, k);
        const int slot = seq % C::kStages;
        const uint32_t k_lo = k_lo0 + slot * (C::kStageBytes >> 4);
        const uint32_t q_lo = q_lo0 + qbuf(q) * (C::kQTileBytes >> 4);
        const uint32_t d_s = tmem + 256u * q;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K step kk: 128-byte block kk / 4 (16 KB apart for Q, 8 KB for the K half),
          // 32-byte column offset (kk % 4) inside it
          const uint32_t a_adv = (kk >> 2) * (C::kBlockBytes >> 4) + (kk & 3) * 2;
          const uint32_t b_adv = (kk >> 2) * (C::kKHalfBlock >> 4) + (kk & 3) * 2;
          mma_pair_ss(d_s, q_lo + a_adv, kDescHi, k_lo + b_adv, kDescHi, kIdescS,
                      kk > 0 ? 1u : 0u);
        }
        mma_commit_pair(&bars->s_full[q]);
        if ((k >= nA && !sh) || q == 1) mma_commit_pair(&bars->k_empty[slot]);
        if (k == n - 1) mma_commit_pair(&bars->q_empty[qbuf(q)]);
      };
      // 16-key steps of PV(q, k): keys past the last one that any row of pair tile q sees
      // have P = 0 (the anchor's last tile; the last tile of the pair tile's suffix
      // window), and their steps are left out
      auto pv_steps = [&](int q, int k) {
        const int vis = k < nA ? (k == nA - 1 ? it.la - k * kBN : kBN)
                               : max(it.tend(2 * q), it.tend(2 * q + 1)) - it.wsp(q) -
                                     (k - nA) * kBN;
        return min(8, max(1, (vis + 15) / 16));
      };
      auto mma_pv = [&](int q, int k, int nkk) {
        const uint32_t seq = kv_base + pos_of(nA, sh, q, k);
        const int slot = seq % C::kStages;
        const uint32_t v_lo = v_lo0 + slot * (C::kStageBytes >> 4);
        const uint32_t d_o = tmem + 256u * q + 128u;
        const uint32_t a_p = tmem + 256u * q + 64u;  // P over the upper half of S's columns
        const uint32_t acc0 = k > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (kk < nkk)
            mma_pair_ts(d_o, a_p + 8u * kk, v_lo + kk * 128, kDescHi, kIdescPV,
                        kk > 0 ? 1u : acc0);
        if ((k >= nA && !sh) || q == 1) mma_commit_pair(&bars->v_empty[slot]);
        if (k == n - 1) mma_commit_pair(&bars->o_done[q]);
      };
      for (int q = 0; q < 2 && ok; ++q) {
        ok = wait_s(q, 0);
        if (ok) {
          tc_fence_after();
          if (elect) mma_s(q, 0);
          __syncwarp();
        }
      }
      for (int k = 0; ok && k < n; ++k) {
        for (int q = 0; q < 2 && ok; ++q) {
          const int nkk = pv_steps(q, k);
          ok = wait_pv(q);
          if (!ok) break;
          tc_fence_after();
          if (elect) {
            mma_pv(q, k, nkk);
            if (k + 1 < n) mma_s(q, k + 1);
          }
          __syncwarp();
        }
      }
      kv_base += it.n_tiles();
      it = nxt;
    }
    if (elect) mma_commit_pair_local(&bars->drain);
    __syncwarp();
    drain_wait(&bars->drain, 0, global_timer_ns() + 100000000ull);
   }
  } else {
    // ------------------------------------------------------ softmax warpgroups (both CTAs)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg<D>::kRegsSoftmax));
    const int q = warp >> 2;                        // pair tile
    const int j = 2 * q + static_cast<int>(rank);   // query tile of the quad
    const int row = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + 256u * q;
    const uint32_t t_o = t_s + 128u;
    const uint32_t p_full_lead = lead_bar(&bars->p_full[q]);
    const uint32_t stage = smem_u32(smem + C::kSmemQ + C::kSmemKV + 1024) + warp * C::kStageWarpBytes;
    const uint64_t out_pol = l2_policy_evict_first();
    uint32_t s_cnt = 0, it_count = 0;
    bool ok = true;
    const float c = p.scale_log2;
    // What this warp needs of a quad. The next quad's record is loaded at the start of the
    // current one and decoded at its end: decoding it at once would wait for the load at
    // the item boundary, on the critical path.
    struct Part {
      int nA, n, la, ag, t0, ws_q, tend_j;
      bool half1;  // query tiles 2 and 3 are not empty
    };
    auto part_of = [&](int i, const Quad& x) {
      Part r{};
      if (i < total_items) {
        r.nA = x.n_anchor_tiles();
        r.n = r.nA + x.n_sfx_tiles();
        r.la = x.la;
        r.ag = x.ag;
        r.t0 = x.t0;
        r.ws_q = x.wsp(q);
        r.tend_j = x.tend(j);
        r.half1 = x.te2 > x.t0 + 2 * tok;
      }
      return r;
    };
    // This row's loads for a quad: the start of its suffix (visible suffix keys of the row:
    // [vis_lo, t]) and, with FP8 anchor KV, the quad's K and V scales. Issued for the next
    // quad after the current one's first tile, used at the next quad.
    struct RowIn {
      int vis_lo;
      float k_sc, v_sc;
    };
    auto row_in = [&](const Part& x, int i) {
      RowIn r{0, 1.0f, 1.0f};
      if (i < total_items) {
        const int tt = x.t0 + j * tok + row / G;
        r.vis_lo = tt < x.tend_j ? __ldg(p.seg + tt) : tt;
        if (FP8) {
          r.k_sc = __ldg(p.k_scale + x.ag);
          r.v_sc = __ldg(p.v_scale + x.ag);
        }
      }
      return r;
    };
    int item = first;
    Part it = part_of(item, item < total_items ? load_quad(p, item) : Quad{});
    RowIn in = row_in(it, item);
    for (; ok && item < total_items; item += stride, ++it_count) {
      const Quad nxt_raw = item + stride < total_items ? load_quad(p, item + stride) : Quad{};
      Part nxt{};
      RowIn nxt_in{0, 1.0f, 1.0f};
      const int nA = it.nA;
      const int n = it.n;
      const int g = it.ag % hkv;
      const int t = it.t0 + j * tok + row / G;
      const bool valid = t < it.tend_j;
      const int vis_lo = in.vis_lo;
      const int ws_q = it.ws_q;
      const float c_anc = FP8 ? c * in.k_sc : c;
      const float v_sc = FP8 ? in.v_sc : 1.0f;
      float m_ref = 0.0f, l = 0.0f;
      for (int k = 0; k < n; ++k) {
        if (!(ok = wait_parity(wc, &bars->s_full[q], s_cnt & 1u))) break;
        ++s_cnt;
        tc_fence_after();
        if (k < nA) {
          const int rem = it.la - k * kBN;
          softmax_tile_spec<128, FP8>(t_s, k == 0, rem < kBN, 0, rem - 1, c_anc, v_sc, m_ref, l);
        } else {
          const int base = ws_q + (k - nA) * kBN;
          const int lo_c = vis_lo - base, hi_c = t - base;
          const bool mk = __any_sync(0xFFFFFFFFu, lo_c > 0 || hi_c < kBN - 1);
          softmax_tile_spec<128, false>(t_s, k == 0, mk, lo_c, hi_c, c, 1.0f, m_ref, l);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(p_full_lead);
        if (k == 0) {  // the next quad's record has arrived by now
          nxt = part_of(item + stride, nxt_raw);
          nxt_in = row_in(nxt, item + stride);
        }
      }
      if (!ok) break;
      // a valid row outside the fast-kernel bounds: the quad's non-empty halves go to the
      // exact kernel (as items 2 x quad and 2 x quad + 1)
      const bool broke = !(l >= kSpecSumLow && l <= kSpecSumHigh) ||
                         (FP8 && it.la > 0 && !(fabsf(v_sc) <= kSpecScaleHigh));
      if (__any_sync(0xFFFFFFFFu, broke && valid) && lane == 0) {
        if (atomicExch(p.redo_flag + item, 1) == 0) {
          const int at = atomicAdd(p.redo_count, it.half1 ? 2 : 1);
          p.redo_list[at] = 2 * item;
          if (it.half1) p.redo_list[at + 1] = 2 * item + 1;
        }
      }
      __syncwarp();
      if (!(ok = wait_parity(wc, &bars->o_done[q], it_count & 1u))) break;
      tc_fence_after();
      const float inv_l = __fdividef(1.0f, l);
      const uint64_t il = f2(inv_l, inv_l);
      const int64_t orow = static_cast<int64_t>(t) * p.hq + g * G + (row % G);
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + orow * D;
      if (__all_sync(0xFFFFFFFFu, valid)) {
        if constexpr (C::kStageWarpBytes >= 2 * 2048 * (D / 64))
          store_rows_tma_all<D>(&maps.out, t_o, il, stage, lane, g * G,
                                it.t0 + j * tok + (warp & 3) * (32 / G), out_pol);
        else
          store_rows_tma<D>(&maps.out, t_o, il, stage, lane, g * G,
                            it.t0 + j * tok + (warp & 3) * (32 / G), out_pol);
      } else {
#pragma unroll
      for (int ch2 = 0; ch2 < D / 64; ++ch2) {
        uint32_t r[2][32];
        tmem_ld32(t_o + ch2 * 64, r[0]);
        tmem_ld32(t_o + ch2 * 64 + 32, r[1]);
        tmem_wait_ld_dep(r[0]);
        reg_dep(r[1]);
        if (valid) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float lo, hi;
              f2_split(f2_mul(f2(__uint_as_float(r[h][2 * e]), __uint_as_float(r[h][2 * e + 1])),
                              il),
                       lo, hi);
              pk[e] = pack_bf16(lo, hi);
            }
            st_global_v8(out + ch2 * 64 + h * 32, pk);
            st_global_v8(out + ch2 * 64 + h * 32 + 16, pk + 8);
          }
        }
      }
      }
      if (valid && p.lse != nullptr)
        p.lse[orow] = (m_ref + __log2f(l)) * 0.69314718055994531f;
      it = nxt;
      in = nxt_in;
    }
    if (lane == 0) bulk_wait_group_all();
    tc_fence_before();
  }

  __syncthreads();
  // Each CTA tells the other whether it gave up on a wait. Rank 1's copies complete on
  // rank 0's barriers, and after an abort nothing waits for those that were issued: then
  // both CTAs give copies in flight 50 us to land before either exits.
  if (threadIdx.x == 0 && bars->abort_flag)
    st_cluster_u32(cluster_map(&bars->peer_abort, rank ^ 1u), 1u);
  cluster_sync();  // also: rank 0's MMAs on rank 1's shared memory and TMEM are complete
  if (bars->abort_flag || bars->peer_abort) {
    const uint64_t until = global_timer_ns() + 50000ull;
    while (global_timer_ns() < until) {
    }
    __syncthreads();
    cluster_sync();
  }
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------
// Per-suffix offset checks and the per-token suffix start. Each suffix is checked on its
// own (0 <= start <= end <= T_S, length <= max_suffix_len) before any write, so nothing
// outside seg[0, T_S) is ever written; a failed check raises the flag that the schedule
// kernel turns into QUAIL_ERR_DEVICE_BOUNDS.
__global__ void __launch_bounds__(256) cascade_segments_kernel(const CascadeParams p) {
  const int S = p.num_suffixes;
  const int64_t T = p.total_suffix_tokens;
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  // one warp per suffix: its lanes write the suffix's tokens
  for (int s = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; s < S; s += warps) {
    const int lo = __ldg(p.suffix_offsets + s), hi = __ldg(p.suffix_offsets + s + 1);
    if (lo < 0 || hi < lo || hi > T || hi - lo > p.max_suffix_len) {
      if (lane == 0) atomicOr(p.flag, 1);
      continue;
    }
    for (int t = lo + lane; t < hi; t += 32) p.seg[t] = lo;
  }
}

// Work-item schedule: validate the anchor offsets and the end points, order anchors by
// decreasing anchor-tile count (longest work first, so the static round-robin over CTAs
// approximates longest-processing-time-first) and write the prefix sum of work items
// over that order.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = warp > 0 ? warp_sums[warp - 1] : 0;
  total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(1024) cascade_schedule_kernel(const CascadeParams p) {
  __shared__ int hist[kSortBins];
  __shared__ int warp_sums[32];
  __shared__ int bad;
  const int A = p.num_anchors, S = p.num_suffixes;
  const int32_t* ao = p.anchor_offsets;
  const int32_t* asp = p.anchor_suffix_ptr;
  const int32_t* so = p.suffix_offsets;
  int32_t* prefix = p.prefix;
  int32_t* order = p.order;
  const int tid = threadIdx.x;
  if (tid == 0) {
    bad = 0;
    *p.redo_count = 0;
  }
  for (int i = tid; i < kSortBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  int my_bad = 0;
  if (tid == 0) {
    my_bad |= *p.flag != 0;  // a per-suffix check failed
    my_bad |= ao[0] != 0 || static_cast<int64_t>(ao[A]) != p.total_anchor_tokens;
    my_bad |= asp[0] != 0 || asp[A] != S;
    my_bad |= so[0] != 0 || static_cast<int64_t>(so[S]) != p.total_suffix_tokens;
  }
  for (int a = tid; a < A; a += blockDim.x) {
    const int la = ao[a + 1] - ao[a];
    my_bad |= la < 0 || la > p.max_anchor_len || asp[a + 1] < asp[a];
  }
  if (my_bad) atomicOr(&bad, 1);
  __syncthreads();
  if (bad) {
    if (tid == 0) atomicOr(p.err_word, kErrDeviceBounds);
    for (int i = tid; i <= A; i += blockDim.x) prefix[i] = 0;
    return;
  }
  const int pair_tok = p.tiles_per_item * p.tok_per_tile;  // suffix tokens per work item
  for (int a = tid; a < A; a += blockDim.x) {
    const int key = min((ao[a + 1] - ao[a] + kBN - 1) / kBN, kSortBins - 1);
    atomicAdd(&hist[kSortBins - 1 - key], 1);
  }
  __syncthreads();
  {
    int total;
    const int v = tid < kSortBins ? hist[tid] : 0;
    const int ex = block_exclusive_scan(v, warp_sums, total);
    if (tid < kSortBins) hist[tid] = ex;  // now the cursor of each bin
    __syncthreads();
  }
  for (int a = tid; a < A; a += blockDim.x) {
    const int key = min((ao[a + 1] - ao[a] + kBN - 1) / kBN, kSortBins - 1);
    const int pos = atomicAdd(&hist[kSortBins - 1 - key], 1);
    order[pos] = a;
  }
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < A; base += blockDim.x) {
    const int i = base + tid;
    int v = 0;
    if (i < A) {
      const int a = order[i];
      const int ntok = so[asp[a + 1]] - so[asp[a]];
      // the anchor pass of the two-pass variant has nothing to do for an empty anchor
      const bool none = p.mode == kAnchorPass && ao[a + 1] == ao[a];
      v = none ? 0 : p.hkv * ((ntok + pair_tok - 1) / pair_tok);
    }
    int total;
    const int ex = block_exclusive_scan(v, warp_sums, total);
    if (i < A) prefix[i] = carry + ex;
    carry += total;
  }
  if (tid == 0) prefix[A] = carry;
}

// One record per work item: (a_tok0, la, t0, a * Hkv + g, ws0, ws1, tend0, tend1); for
// the CTA-pair kernel one per quad: (a_tok0, la, t0, a * Hkv + g, wsp0, wsp1, tend0,
// tend1, tend2, tend3).
__global__ void __launch_bounds__(256) cascade_items_kernel(const CascadeParams p) {
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  const int A = p.num_anchors;
  const int total = p.prefix[A];
  if (item >= total) return;
  p.redo_flag[item] = 0;
  int lo = 0, hi = A - 1;  // largest sorted position with prefix <= item
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int a = p.order[lo];
  const int local = item - p.prefix[lo];
  const int s_begin = p.suffix_offsets[p.anchor_suffix_ptr[a]];
  const int s_end = p.suffix_offsets[p.anchor_suffix_ptr[a + 1]];
  const int tok = p.tok_per_tile;
  if (p.tiles_per_item == 4) {
    const int quads = (s_end - s_begin + 4 * tok - 1) / (4 * tok);
    const int g = local / quads;
    const int t0 = s_begin + (local % quads) * 4 * tok;
    int tend[4];
    for (int j = 0; j < 4; ++j) {
      const int start = t0 + j * tok;
      tend[j] = start < s_end ? min(start + tok, s_end) : start;
    }
    int4* dst = reinterpret_cast<int4*>(p.items + 12 * static_cast<int64_t>(item));
    dst[0] = make_int4(p.anchor_offsets[a], p.anchor_offsets[a + 1] - p.anchor_offsets[a], t0,
                       a * p.hkv + g);
    const int s2 = t0 + 2 * tok;
    dst[1] = make_int4(p.seg[t0], s2 < s_end ? p.seg[s2] : s2, tend[0], tend[1]);
    dst[2] = make_int4(tend[2], tend[3], 0, 0);
    return;
  }
  const int pairs = (s_end - s_begin + 2 * tok - 1) / (2 * tok);
  const int g = local / pairs;
  const int t0 = s_begin + (local % pairs) * 2 * tok;
  const int tend0 = min(t0 + tok, s_end);
  const int t1 = t0 + tok;
  const bool has1 = s_end > t1;
  int4 r0, r1;
  r0.x = p.anchor_offsets[a];
  r0.y = p.anchor_offsets[a + 1] - r0.x;
  r0.z = t0;
  r0.w = a * p.hkv + g;
  r1.x = p.seg[t0];
  r1.y = has1 ? p.seg[t1] : t1;
  r1.z = tend0;
  r1.w = has1 ? min(t1 + tok, s_end) : t1;
  if (p.mode == kAnchorPass) {  // anchor keys only: empty suffix windows
    r1.x = r1.z;
    r1.y = r1.w;
  } else if (p.mode == kSuffixPass) {  // suffix keys only: no anchor tiles
    r0.y = 0;
  }
  int4* dst = reinterpret_cast<int4*>(p.items + 8 * static_cast<int64_t>(item));
  dst[0] = r0;
  dst[1] = r1;
}

// FP8 anchor KV staging: e4m3 codes -> bf16, exact (every e4m3 value, subnormals
// included, is a bf16 value; the NaN codes stay NaN). Both tensors [T_A, Hkv, D] are
// walked as one range of 16-code units: one 16-byte load and two 16-byte stores each,
// two units per thread in flight.
__device__ __forceinline__ uint4 ld_stream_u4(const uint8_t* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ void st_u4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
// Two f16 values of at most 4 significant bits and exponents in [-9, 8] -> bf16x2, exact
// (f16 -> f32 is exact, and so is f32 -> bf16 for such values).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  float lo, hi;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
  return pack_bf16(lo, hi);
}
// Four e4m3 codes (bytes 0..3 of w) -> four bf16 in two words, the lower code in the
// lower half (memory order kept).
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t& a, uint32_t& b) {
  uint32_t h0, h1;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(h0), "=r"(h1)
      : "r"(w));
  a = f16x2_to_bf16x2(h0);
  b = f16x2_to_bf16x2(h1);
}
__device__ __forceinline__ void convert_unit(const uint4 c, uint8_t* dst) {
  uint32_t o[8];
  e4m3x4_to_bf16x4(c.x, o[0], o[1]);
  e4m3x4_to_bf16x4(c.y, o[2], o[3]);
  e4m3x4_to_bf16x4(c.z, o[4], o[5]);
  e4m3x4_to_bf16x4(c.w, o[6], o[7]);
  st_u4(dst, o[0], o[1], o[2], o[3]);
  st_u4(dst + 16, o[4], o[5], o[6], o[7]);
}
__global__ void __launch_bounds__(256) anchor_e4m3_to_bf16_kernel(const CascadeParams p,
                                                                   int64_t units) {
  const uint8_t* kc = static_cast<const uint8_t*>(p.k_anc);
  const uint8_t* vc = static_cast<const uint8_t*>(p.v_anc);
  uint8_t* kb = static_cast<uint8_t*>(p.k_anc_bf16);
  uint8_t* vb = static_cast<uint8_t*>(p.v_anc_bf16);
  const uint64_t pol = l2_policy_evict_first();
  const int64_t total = 2 * units;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  auto src = [&](int64_t u) { return u < units ? kc + 16 * u : vc + 16 * (u - units); };
  auto dst = [&](int64_t u) { return u < units ? kb + 32 * u : vb + 32 * (u - units); };
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += 2 * step) {
    const bool two = u + step < total;
    const uint4 c0 = ld_stream_u4(src(u), pol);
    const uint4 c1 = two ? ld_stream_u4(src(u + step), pol) : make_uint4(0u, 0u, 0u, 0u);
    convert_unit(c0, dst(u));
    if (two) convert_unit(c1, dst(u + step));
  }
}

// Causal prefill with K/V amax: per (suffix, KV head), the max of the per-row maxima the
// producer stored (bf16 bit patterns of non-negative values order like integers). One
// block per suffix; suffixes whose offsets fail the checks are skipped.
__global__ void __launch_bounds__(256) kv_amax_reduce_kernel(const CascadeParams p) {
  // one warp per (suffix, KV head); lanes stride over the suffix's rows
  const int hkv = p.hkv;
  const int lane = threadIdx.x & 31;
  const int64_t pairs = static_cast<int64_t>(p.num_suffixes) * hkv;
  const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       w < pairs; w += warps) {
    const int s = static_cast<int>(w / hkv), g = static_cast<int>(w % hkv);
    const int lo = __ldg(p.suffix_offsets + s), hi = __ldg(p.suffix_offsets + s + 1);
    uint32_t m = 0;  // packed (max |k|, max |v|) bf16 patterns
    if (lo >= 0 && hi >= lo && hi <= p.total_suffix_tokens) {
      const uint32_t* rm = reinterpret_cast<const uint32_t*>(p.rowmax);
      for (int r = lo + lane; r < hi; r += 32) {
        uint32_t v = __ldg(rm + static_cast<int64_t>(r) * hkv + g);
        asm("max.u16x2 %0, %0, %1;" : "+r"(m) : "r"(v));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint32_t v = __shfl_xor_sync(0xFFFFFFFFu, m, o);
      asm("max.u16x2 %0, %0, %1;" : "+r"(m) : "r"(v));
    }
    if (lane == 0) {
      p.k_amax[w] = __uint_as_float((m & 0xFFFFu) << 16);
      p.v_amax[w] = __uint_as_float(m & 0xFFFF0000u);
    }
  }
}

// Two-pass variant, A4 as its own kernel: the LSE merge of the anchor partial (fp32 O_a,
// lse_a) with the suffix partial (out holds O_s in bf16, lse_s) for every (token, query
// head) row, in place: lse = log(e^lse_a + e^lse_s), out = e^(lse_a - lse) O_a +
// e^(lse_s - lse) O_s. lse_a = -inf (an empty anchor) leaves O_s as it is. One warp per
// row, D / 32 elements per lane (16-byte fp32 and 8-byte bf16 accesses for D = 128).
template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(int64_t rows, const float* o_part,
                                                        const float* lse_part,
                                                        const float* lse_s,
                                                        __nv_bfloat16* out, float* lse) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       r < rows; r += warps) {
    const float la = __ldg(lse_part + r), ls = __ldg(lse_s + r);
    float wa = 0.0f, ws = 1.0f, lm = ls;
    if (la > -INFINITY) {
      const float mx = fmaxf(la, ls);
      const float ea = expf(la - mx), es = expf(ls - mx);
      const float inv = 1.0f / (ea + es);
      wa = ea * inv;
      ws = es * inv;
      lm = mx + logf(ea + es);
    }
    __nv_bfloat16* o = out + r * D + lane * E;
    const float* a = o_part + r * D + lane * E;
    float va[E];
    __nv_bfloat16 vs[E];
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 x = *reinterpret_cast<const float2*>(a + e);
      va[e] = x.x;
      va[e + 1] = x.y;
      const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(o + e);
      vs[e] = y.x;
      vs[e + 1] = y.y;
    }
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float lo = wa * va[e] + ws * __bfloat162float(vs[e]);
      const float hi = wa * va[e + 1] + ws * __bfloat162float(vs[e + 1]);
      *reinterpret_cast<__nv_bfloat162*>(o + e) = __floats2bfloat162_rn(lo, hi);
    }
    if (lane == 0 && lse != nullptr) lse[r] = lm;
  }
}

__global__ void __launch_bounds__(256) fill_neg_inf_kernel(float* x, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    x[i] = -INFINITY;
}

}  // namespace

cudaError_t launch_fill_neg_inf(float* x, int64_t n, int num_sms, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, int64_t{num_sms} * 8));
  fill_neg_inf_kernel<<<blocks, 256, 0, stream>>>(x, n);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(int64_t rows, int head_dim, const float* o_part,
                             const float* lse_part, const float* lse_s, void* out, float* lse,
                             int num_sms, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((rows + 7) / 8, int64_t{num_sms} * 8));
  auto* o = static_cast<__nv_bfloat16*>(out);
  if (head_dim == 128)
    lse_merge_kernel<128><<<blocks, 256, 0, stream>>>(rows, o_part, lse_part, lse_s, o, lse);
  else
    lse_merge_kernel<64><<<blocks, 256, 0, stream>>>(rows, o_part, lse_part, lse_s, o, lse);
  return cudaGetLastError();
}

int64_t cascade_item_bound(int num_anchors, int64_t total_suffix_tokens, int hkv, int group) {
  const int64_t pair_tok = 2 * (128 / group);
  return static_cast<int64_t>(hkv) * ((total_suffix_tokens + pair_tok - 1) / pair_tok + num_anchors);
}

CascadeWorkspace cascade_workspace_layout(int num_anchors, int64_t total_suffix_tokens,
                                          int64_t item_bound, int64_t anchor_bf16_bytes) {
  auto up = [](size_t x, size_t a) { return (x + a - 1) / a * a; };
  CascadeWorkspace w;
  w.flag = 0;
  w.redo_count = 4;
  w.prefix = 16;
  w.order = w.prefix + 4 * (static_cast<size_t>(num_anchors) + 1);
  w.seg = up(w.order + 4 * static_cast<size_t>(num_anchors), 16);
  w.items = up(w.seg + 4 * static_cast<size_t>(total_suffix_tokens), 32);
  w.redo_flag = w.items + 48 * static_cast<size_t>(item_bound);  // records of up to 12 ints
  w.redo_list = w.redo_flag + 4 * static_cast<size_t>(item_bound);
  w.k_anc_bf16 = up(w.redo_list + 4 * static_cast<size_t>(item_bound), 256);
  w.v_anc_bf16 = up(w.k_anc_bf16 + static_cast<size_t>(anchor_bf16_bytes), 256);
  w.total = up(w.v_anc_bf16 + static_cast<size_t>(anchor_bf16_bytes), 256);
  return w;
}

template <int D, bool FP8, bool EXACT, bool AMAX = false>
static cudaError_t launch_attn_kernel(const CascadeParams& p, const CascadeMaps& maps,
                                      int num_sms, cudaStream_t stream) {
  using C = Cfg<D>;
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, cascade_attn_kernel<D, FP8, EXACT, AMAX>);
  if (e != cudaSuccess) return e;
  // the register split must fit in what the block is launched with (else setmaxnreg.inc
  // would wait forever)
  if (static_cast<int64_t>(attr.numRegs) * kThreads <
      256 * Cfg<D>::kRegsSoftmax + 128 * Cfg<D>::kRegsOther)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(cascade_attn_kernel<D, FP8, EXACT, AMAX>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = p.item_bound < num_sms ? p.item_bound : num_sms;
  if (grid <= 0) return cudaSuccess;
  cascade_attn_kernel<D, FP8, EXACT, AMAX><<<grid, kThreads, C::kSmemBytes, stream>>>(p, maps);
  return cudaGetLastError();
}

// Clusters of two CTAs (one per SM) that can be resident at once, per device.
template <bool FP8, int STAGES>
static int pair_clusters(int num_sms, cudaStream_t stream) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::atomic<int>* slot = dev >= 0 && dev < 64 ? &cache[dev] : nullptr;
  if (slot != nullptr && slot->load() > 0) return slot->load();
  if (cudaFuncSetAttribute(cascade_pair_kernel<FP8, STAGES>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PairCfgT<STAGES>::kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int clusters = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms / 2 * 2), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = PairCfgT<STAGES>::kSmemBytes;
  cfg.stream = stream;
  if (cudaOccupancyMaxActiveClusters(&clusters, cascade_pair_kernel<FP8, STAGES>, &cfg) !=
          cudaSuccess ||
      clusters <= 0) {
    cudaGetLastError();
    return 0;
  }
  if (slot != nullptr) slot->store(clusters);
  return clusters;
}

template <bool FP8, int STAGES>
static cudaError_t launch_pair_kernel(const CascadeParams& p, const CascadeMaps& maps,
                                      int num_sms, cudaStream_t stream) {
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, cascade_pair_kernel<FP8, STAGES>);
  if (e != cudaSuccess) return e;
  if (static_cast<int64_t>(attr.numRegs) * kThreads <
      256 * Cfg<128>::kRegsSoftmax + 128 * Cfg<128>::kRegsOther)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(cascade_pair_kernel<FP8, STAGES>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PairCfgT<STAGES>::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int clusters = pair_clusters<FP8, STAGES>(num_sms, stream);
  if (clusters <= 0) return cudaErrorInvalidConfiguration;
  // quads <= item_bound (the bound on two-tile items)
  const int grid = 2 * (p.item_bound < clusters ? p.item_bound : clusters);
  if (grid <= 0) return cudaSuccess;
  cascade_pair_kernel<FP8, STAGES><<<grid, kThreads, PairCfgT<STAGES>::kSmemBytes, stream>>>(p, maps);
  return cudaGetLastError();
}

// Ring depth of the pair kernel: 3 K/V stages (and all output columns staged at once) when
// the anchor K/V is well inside L2 (<= 64 MB, K and V in bf16, so that every quad of an
// anchor finds its tiles there) and each pair tile's suffix window is one 128-key tile (2
// tokens-per-tile + the longest suffix - 1 <= 128 keys); else 4. Measured: join (33.6 MB
// of anchor K/V, windows of at most 87 keys) 1-3 % faster with 3; ragged, fp8_long and
// the causal prefill (anchor K/V or windows beyond that) unchanged or slower.
static bool pair_shallow_ring(const CascadeParams& p) {
  const int64_t anchor_kv_bytes = p.total_anchor_tokens * p.hkv * 128 * 2 * 2;
  return anchor_kv_bytes <= (int64_t{64} << 20) &&
         2 * p.tok_per_tile + p.max_suffix_len - 1 <= 128;
}

// The fast kernel (single CTAs, or CTA pairs over quads), then the exact kernel over the
// items it handed over (none: its CTAs return at once).
template <int D, bool FP8>
static cudaError_t launch_attn_d(const CascadeParams& p, const CascadeMaps& maps, int num_sms,
                                 cudaStream_t stream) {
  // the K/V amax (causal prefill) is formed by the fast kernel, which sees every item
  const bool amax = !FP8 && p.k_amax != nullptr;
  cudaError_t e;
  if (D == 128 && p.tiles_per_item == 4)
    e = pair_shallow_ring(p) ? launch_pair_kernel<FP8, 3>(p, maps, num_sms, stream)
                             : launch_pair_kernel<FP8, 4>(p, maps, num_sms, stream);
  else
    e = amax ? launch_attn_kernel<D, false, false, true>(p, maps, num_sms, stream)
             : launch_attn_kernel<D, FP8, false>(p, maps, num_sms, stream);
  if (e != cudaSuccess) return e;
  e = launch_attn_kernel<D, FP8, true>(p, maps, num_sms, stream);
  if (e != cudaSuccess || !amax || p.num_suffixes == 0) return e;
  const int64_t pairs = static_cast<int64_t>(p.num_suffixes) * p.hkv;
  const int blocks = static_cast<int>(std::min<int64_t>((pairs + 7) / 8, int64_t{num_sms} * 8));
  kv_amax_reduce_kernel<<<blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

namespace {
std::atomic<int> g_cta_pairs{QUAIL_CTA_PAIRS_AUTO};
}
void set_cta_pairs(int mode) { g_cta_pairs.store(mode); }

cudaError_t launch_cascade(const CascadeParams& params, const CascadeMaps& maps, int head_dim,
                           bool fp8, int num_sms, cudaStream_t stream) {
  // The CTA-pair kernel takes d = 128 calls with both parts fused and no K/V amax (with
  // the fault-injection switch on, only when forced: then its own timeout path runs, else
  // the single-CTA kernel's). The automatic choice takes it for all of them: its pair
  // tiles load a short suffix window as a 128-key tile where the single-CTA kernel loads
  // 64 keys, but its PV stops at the window's last key and its anchor tiles move half the
  // operand bytes per SM, and it measured faster on every shape tried (join with 4, 8 and
  // 16 query heads per KV head and suffixes of 1 to 24 tokens included).
  CascadeParams p = params;
  const int mode = g_cta_pairs.load();
  bool pairs = mode != QUAIL_CTA_PAIRS_OFF && head_dim == 128 && p.mode == kFused &&
               p.k_amax == nullptr && num_sms >= 2 &&
               (p.inject_skip_first_kv == 0 || mode == QUAIL_CTA_PAIRS_ALWAYS);
  // no resident pair of SMs (e.g. a partition of the GPU): the single-CTA kernel
  if (pairs && (fp8 ? pair_clusters<true, 4>(num_sms, stream)
                    : pair_clusters<false, 4>(num_sms, stream)) <= 0)
    pairs = false;
  p.tiles_per_item = pairs ? 4 : 2;
  cudaError_t e = cudaMemsetAsync(p.flag, 0, sizeof(int32_t), stream);
  if (e != cudaSuccess) return e;
  if (p.num_suffixes > 0) {
    const int blocks = static_cast<int>(
        std::min<int64_t>((p.num_suffixes + 7) / 8, static_cast<int64_t>(num_sms) * 8));
    cascade_segments_kernel<<<blocks, 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  cascade_schedule_kernel<<<1, 1024, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.item_bound > 0) {
    cascade_items_kernel<<<(p.item_bound + 255) / 256, 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (fp8 && p.total_anchor_tokens > 0) {
    const int64_t units = p.total_anchor_tokens * p.hkv * head_dim / 16;
    const int blocks = static_cast<int>(
        std::min<int64_t>((units + 255) / 256, static_cast<int64_t>(num_sms) * 8));
    anchor_e4m3_to_bf16_kernel<<<blocks, 256, 0, stream>>>(p, units);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (head_dim == 128)
    return fp8 ? launch_attn_d<128, true>(p, maps, num_sms, stream)
               : launch_attn_d<128, false>(p, maps, num_sms, stream);
  return fp8 ? launch_attn_d<64, true>(p, maps, num_sms, stream)
             : launch_attn_d<64, false>(p, maps, num_sms, stream);
}

}  // namespace quail
