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
// Per CTA (one per SM, persistent):
//   warp 8      TMA producer: Q tiles, then a ring of K / V tiles (128 keys each)
//   warp 9      MMA issuer:   S_q = Q_q K^T (SMEM x SMEM -> TMEM), O_q += P_q V
//                             (P from TMEM, V from SMEM), tcgen05 kind::f16, M = 128
//   warps 0-3   softmax of query tile 0, one thread per TMEM lane (= query row)
//   warps 4-7   softmax of query tile 1
// TMEM (512 columns): tile q uses S/P at columns 256q .. +127 and O at 256q+128 .. +255.
// The two query tiles share every anchor KV tile loaded into shared memory and ping-pong:
// while one warpgroup exponentiates its scores the tensor core works on the other tile.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace quail {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 320;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: O is rescaled only past 2^8
constexpr int kSortBins = 1024;
constexpr uint32_t kTmemCols = 512;

template <int D>
struct Cfg {
  static constexpr int kKB = D / 64;                   // 128-byte column blocks per row
  static constexpr int kBlockBytes = 128 * 128;        // 128 rows x 128 bytes
  static constexpr int kTileBytes = kKB * kBlockBytes;  // one 128-row bf16 tile
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kSmemQ = 2 * kTileBytes;
  static constexpr int kSmemKV = kStages * 2 * kTileBytes;
  static constexpr int kSmemBytes = kSmemQ + kSmemKV + 1024 + 1024;
};

struct __align__(8) Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct Item {
  int a, g;
  int a_tok0, la;      // anchor token start (into k_anc/v_anc) and length
  int s_lo, s_hi;      // suffix index range of the anchor
  int t0;              // first suffix token of query tile 0
  int n_anchor_tiles;  // ceil(la / 128)
  int n_sfx_tiles;     // suffix-window tiles per query tile
  int nk_sfx;          // keys per suffix tile (64 or 128)
  int ws0, ws1;        // suffix window start of query tile 0 / 1
  int tend0, tend1;    // one past the last valid token of query tile 0 / 1
  __device__ __forceinline__ int ws(int q) const { return q ? ws1 : ws0; }
  __device__ __forceinline__ int tend(int q) const { return q ? tend1 : tend0; }
};

// Start token of the suffix (of the anchor's range [s_lo, s_hi)) that contains token t.
__device__ __forceinline__ int seg_start(const int32_t* __restrict__ so, int s_lo, int s_hi,
                                         int t) {
  int lo = s_lo, hi = s_hi - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(so + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return __ldg(so + lo);
}

__device__ __forceinline__ void decode_item(const CascadeParams& p, int item, Item& it) {
  const int A = p.num_anchors;
  const int32_t* prefix = p.sched;
  const int32_t* order = p.sched + A + 1;
  int lo = 0, hi = A - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(prefix + mid) <= item) lo = mid; else hi = mid - 1;
  }
  const int a = __ldg(order + lo);
  const int local = item - __ldg(prefix + lo);
  it.a = a;
  it.s_lo = __ldg(p.anchor_suffix_ptr + a);
  it.s_hi = __ldg(p.anchor_suffix_ptr + a + 1);
  const int s_begin = __ldg(p.suffix_offsets + it.s_lo);
  const int s_end = __ldg(p.suffix_offsets + it.s_hi);
  const int tok = p.tok_per_tile;
  const int pairs = (s_end - s_begin + 2 * tok - 1) / (2 * tok);
  it.g = local / pairs;
  it.t0 = s_begin + (local % pairs) * 2 * tok;
  it.a_tok0 = __ldg(p.anchor_offsets + a);
  it.la = __ldg(p.anchor_offsets + a + 1) - it.a_tok0;
  it.n_anchor_tiles = (it.la + kBN - 1) / kBN;
  // query tile 0 always holds at least one token of the anchor
  it.tend0 = min(it.t0 + tok, s_end);
  it.ws0 = seg_start(p.suffix_offsets, it.s_lo, it.s_hi, it.t0);
  int wmax = it.tend0 - it.ws0;
  const int t1 = it.t0 + tok;
  if (s_end > t1) {
    it.tend1 = min(t1 + tok, s_end);
    it.ws1 = seg_start(p.suffix_offsets, it.s_lo, it.s_hi, t1);
    wmax = max(wmax, it.tend1 - it.ws1);
  } else {
    it.tend1 = t1;
    it.ws1 = t1;
  }
  it.n_sfx_tiles = (wmax + kBN - 1) / kBN;
  it.nk_sfx = (it.n_sfx_tiles == 1 && wmax <= 64) ? 64 : 128;
}

// Ring position -> what it holds: anchor tile k (k < nA) or the suffix tile i of query
// tile q at position nA + 2i + q.
__device__ __forceinline__ int pos_of(const Item& it, int q, int k) {
  return k < it.n_anchor_tiles ? k : it.n_anchor_tiles + 2 * (k - it.n_anchor_tiles) + q;
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

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ---------------------------------------------------------------------------------
// Softmax of one S tile held in registers: mask, row max, lazy rescale of O, P = 2^(s c - m)
// written back to TMEM as bf16 (columns 0 .. NC/2 of the S region), row sum update.
template <int NC, int D>
__device__ __forceinline__ void softmax_tile(uint32_t t_s, uint32_t t_o, bool first_tile,
                                             bool masked, int lo_c, int hi_c, float c,
                                             float& m_used, float& l) {
  float s[NC];
  {
    uint32_t r[NC / 32][32];
#pragma unroll
    for (int ch = 0; ch < NC / 32; ++ch) tmem_ld32(t_s + ch * 32, r[ch]);
    tmem_wait_ld_dep(r[0]);
#pragma unroll
    for (int ch = 1; ch < NC / 32; ++ch) reg_dep(r[ch]);
#pragma unroll
    for (int ch = 0; ch < NC / 32; ++ch)
#pragma unroll
      for (int j = 0; j < 32; ++j) s[ch * 32 + j] = __uint_as_float(r[ch][j]);
  }
  if (masked) {
#pragma unroll
    for (int j = 0; j < NC; ++j)
      if (j < lo_c || j > hi_c) s[j] = -INFINITY;
  }
  float mx = s[0];
#pragma unroll
  for (int j = 1; j < NC; ++j) mx = fmaxf(mx, s[j]);
  const float m_tile = mx * c;
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
  float sum = 0.0f;
#pragma unroll
  for (int ch = 0; ch < NC / 32; ++ch) {
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float p0 = ex2(fmaf(s[ch * 32 + 2 * j], c, -m_safe));
      const float p1 = ex2(fmaf(s[ch * 32 + 2 * j + 1], c, -m_safe));
      sum += p0 + p1;
      pk[j] = pack_bf16(p0, p1);
    }
    tmem_st16(t_s + ch * 16, pk);
  }
  l = l * alpha + sum;
  // The PV of the previous tile is complete (the commit that signalled this S tile
  // tracks every earlier MMA), and the PV of this tile waits for this warpgroup's P,
  // so O can be rescaled in place here.
  if (__any_sync(0xFFFFFFFFu, rescale)) {
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t r[32];
      tmem_ld32(t_o + ch * 32, r);
      tmem_wait_ld_dep(r);
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
      tmem_st32(t_o + ch * 32, r);
    }
  }
  tmem_wait_st();
}

// ---------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
cascade_attn_kernel(const __grid_constant__ CascadeParams p,
                    const __grid_constant__ CascadeMaps maps) {
  using C = Cfg<D>;
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
      mbar_init(&bars->p_full[q], kBM);
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

  const int total_items = __ldg(p.sched + p.num_anchors);
  const int tok = p.tok_per_tile;
  const int G = p.group;

  if (warp == kWarpProducer) {
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k_anc);
      tma_prefetch_desc(&maps.v_anc);
      tma_prefetch_desc(&maps.k_suf);
      tma_prefetch_desc(&maps.v_suf);
      uint32_t kv_seq = 0, it_count = 0;
      uint32_t q_arm[2] = {0, 0}, k_arm[4] = {0, 0, 0, 0}, v_arm[4] = {0, 0, 0, 0};
      bool skip_pending = p.inject_skip_first_kv != 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < total_items; item += gridDim.x, ++it_count) {
        Item it;
        decode_item(p, item, it);
        const int n_tiles = it.n_anchor_tiles + 2 * it.n_sfx_tiles;
        for (int pos = 0; pos < n_tiles; ++pos, ++kv_seq) {
          const int slot = kv_seq % C::kStages;
          const uint32_t ph = (kv_seq / C::kStages) & 1u;
          const CUtensorMap* mk;
          const CUtensorMap* mv;
          int row;
          if (pos < it.n_anchor_tiles) {
            mk = &maps.k_anc;
            mv = &maps.v_anc;
            row = it.a_tok0 + pos * kBN;
          } else {
            const int rel = pos - it.n_anchor_tiles;
            mk = &maps.k_suf;
            mv = &maps.v_suf;
            row = it.ws(rel & 1) + (rel >> 1) * kBN;
          }
          uint8_t* k_dst = sKV + slot * 2 * C::kTileBytes;
          uint8_t* v_dst = k_dst + C::kTileBytes;
          if (!(ok = wait_parity(wc, &bars->k_empty[slot], ph ^ 1u))) break;
          if (skip_pending) {
            skip_pending = false;  // fault injection: this tile's K never arrives
          } else {
            mbar_arrive_expect_tx(&bars->k_full[slot], C::kTileBytes);
            ++k_arm[slot];
            for (int kb = 0; kb < C::kKB; ++kb)
              tma_load_3d(mk, &bars->k_full[slot], k_dst + kb * C::kBlockBytes, kb * 64, it.g,
                          row);
          }
          if (pos == 0) {
            for (int q = 0; q < 2 && ok; ++q) {
              if (!(ok = wait_parity(wc, &bars->q_empty[q], (it_count & 1u) ^ 1u))) break;
              mbar_arrive_expect_tx(&bars->q_full[q], C::kTileBytes);
              ++q_arm[q];
              for (int kb = 0; kb < C::kKB; ++kb)
                tma_load_3d(&maps.q, &bars->q_full[q], sQ + q * C::kTileBytes + kb * C::kBlockBytes,
                            kb * 64, it.g * G, it.t0 + q * tok);
            }
            if (!ok) break;
          }
          if (!(ok = wait_parity(wc, &bars->v_empty[slot], ph ^ 1u))) break;
          mbar_arrive_expect_tx(&bars->v_full[slot], C::kTileBytes);
          ++v_arm[slot];
          for (int kb = 0; kb < C::kKB; ++kb)
            tma_load_3d(mv, &bars->v_full[slot], v_dst + kb * C::kBlockBytes, kb * 64, it.g, row);
        }
      }
      // Let every load that was issued land before the CTA can exit.
      const uint64_t dl = global_timer_ns() + 100000000ull;
      for (int q = 0; q < 2; ++q)
        if (q_arm[q]) drain_wait(&bars->q_full[q], (q_arm[q] - 1) & 1u, dl);
      for (int s = 0; s < C::kStages; ++s) {
        if (k_arm[s]) drain_wait(&bars->k_full[s], (k_arm[s] - 1) & 1u, dl);
        if (v_arm[s]) drain_wait(&bars->v_full[s], (v_arm[s] - 1) & 1u, dl);
      }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      constexpr uint32_t kIdescS128 = idesc_f16(kBM, 128, 1, 0);
      constexpr uint32_t kIdescS64 = idesc_f16(kBM, 64, 1, 0);
      constexpr uint32_t kIdescPV = idesc_f16(kBM, D, 1, 1);
      const uint32_t sQa = smem_u32(sQ);
      const uint32_t sKVa = smem_u32(sKV);
      uint32_t kv_base = 0, it_count = 0;
      uint32_t p_cnt[2] = {0, 0};
      bool ok = true;
      for (int item = blockIdx.x; ok && item < total_items; item += gridDim.x, ++it_count) {
        Item it;
        decode_item(p, item, it);
        const int nA = it.n_anchor_tiles;
        const int n = nA + it.n_sfx_tiles;

        auto issue_s = [&](int q, int k) -> bool {
          const uint32_t seq = kv_base + pos_of(it, q, k);
          const int slot = seq % C::kStages;
          const uint32_t ph = (seq / C::kStages) & 1u;
          const bool sfx = k >= nA;
          if ((sfx || q == 0) && !wait_parity(wc, &bars->k_full[slot], ph)) return false;
          if (k == 0 && !wait_parity(wc, &bars->q_full[q], it_count & 1u)) return false;
          tc_fence_after();
          const uint32_t kaddr = sKVa + slot * 2 * C::kTileBytes;
          const uint32_t qaddr = sQa + q * C::kTileBytes;
          const uint32_t idesc = (!sfx || it.nk_sfx == 128) ? kIdescS128 : kIdescS64;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBlockBytes + (kk & 3) * 32;
            mma_ss(tmem + 256u * q, smem_desc_sw128(qaddr + off, 16, 1024),
                   smem_desc_sw128(kaddr + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[q]);
          if (sfx || q == 1) mma_commit(&bars->k_empty[slot]);
          if (k == n - 1) mma_commit(&bars->q_empty[q]);
          return true;
        };
        auto issue_pv = [&](int q, int k) -> bool {
          const uint32_t seq = kv_base + pos_of(it, q, k);
          const int slot = seq % C::kStages;
          const uint32_t ph = (seq / C::kStages) & 1u;
          const bool sfx = k >= nA;
          if ((sfx || q == 0) && !wait_parity(wc, &bars->v_full[slot], ph)) return false;
          if (!wait_parity(wc, &bars->p_full[q], p_cnt[q] & 1u)) return false;
          ++p_cnt[q];
          tc_fence_after();
          const uint32_t vaddr = sKVa + slot * 2 * C::kTileBytes + C::kTileBytes;
          const int nk = sfx ? it.nk_sfx : kBN;
          for (int kk = 0; kk < nk / 16; ++kk) {
            mma_ts(tmem + 256u * q + 128u, tmem + 256u * q + 8u * kk,
                   smem_desc_sw128(vaddr + kk * 2048, C::kBlockBytes, 1024), kIdescPV,
                   (k > 0 || kk > 0) ? 1u : 0u);
          }
          if (sfx || q == 1) mma_commit(&bars->v_empty[slot]);
          if (k == n - 1) mma_commit(&bars->o_done[q]);
          return true;
        };

        ok = issue_s(0, 0) && issue_s(1, 0);
        for (int k = 0; ok && k < n; ++k) {
          ok = issue_pv(0, k) && (k + 1 >= n || issue_s(0, k + 1)) && issue_pv(1, k) &&
               (k + 1 >= n || issue_s(1, k + 1));
        }
        kv_base += nA + 2 * it.n_sfx_tiles;
      }
      // Every MMA issued so far has completed once this barrier flips.
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, global_timer_ns() + 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int q = warp >> 2;
    const int row = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + 256u * q;
    const uint32_t t_o = t_s + 128u;
    uint32_t s_cnt = 0, it_count = 0;
    bool ok = true;
    const float c = p.scale_log2;
    for (int item = blockIdx.x; ok && item < total_items; item += gridDim.x, ++it_count) {
      Item it;
      decode_item(p, item, it);
      const int nA = it.n_anchor_tiles;
      const int n = nA + it.n_sfx_tiles;
      const int t = it.t0 + q * tok + row / G;
      const bool valid = t < it.tend(q);
      // visible suffix keys of this row: [vis_lo, t]
      const int vis_lo = valid ? seg_start(p.suffix_offsets, it.s_lo, it.s_hi, t) : t;
      float m_used = -INFINITY, l = 0.0f;
      for (int k = 0; k < n; ++k) {
        if (!(ok = wait_parity(wc, &bars->s_full[q], s_cnt & 1u))) break;
        ++s_cnt;
        tc_fence_after();
        if (k < nA) {
          const int rem = it.la - k * kBN;
          softmax_tile<128, D>(t_s, t_o, k == 0, rem < kBN, 0, rem - 1, c, m_used, l);
        } else {
          const int base = it.ws(q) + (k - nA) * kBN;
          const int lo_c = vis_lo - base, hi_c = t - base;
          if (it.nk_sfx == 64)
            softmax_tile<64, D>(t_s, t_o, k == 0, true, lo_c, hi_c, c, m_used, l);
          else
            softmax_tile<128, D>(t_s, t_o, k == 0, true, lo_c, hi_c, c, m_used, l);
        }
        tc_fence_before();
        mbar_arrive(&bars->p_full[q]);
      }
      if (!ok) break;
      if (!(ok = wait_parity(wc, &bars->o_done[q], it_count & 1u))) break;
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const int64_t orow = static_cast<int64_t>(t) * p.hq + it.g * G + (row % G);
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + orow * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(t_o + ch * 32, r);
        tmem_wait_ld_dep(r);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(out + ch * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r[8 * j + 0]) * inv_l, __uint_as_float(r[8 * j + 1]) * inv_l);
            v.y = pack_bf16(__uint_as_float(r[8 * j + 2]) * inv_l, __uint_as_float(r[8 * j + 3]) * inv_l);
            v.z = pack_bf16(__uint_as_float(r[8 * j + 4]) * inv_l, __uint_as_float(r[8 * j + 5]) * inv_l);
            v.w = pack_bf16(__uint_as_float(r[8 * j + 6]) * inv_l, __uint_as_float(r[8 * j + 7]) * inv_l);
            dst[j] = v;
          }
        }
      }
      if (valid && p.lse != nullptr)
        p.lse[orow] = (m_used + __log2f(l)) * 0.69314718055994531f;
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------
// Tile schedule: validate the offsets, order anchors by decreasing anchor-tile count
// (longest work first, so the static round-robin over CTAs approximates LPT) and write
// the prefix sum of work items over that order.
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
  int32_t* prefix = p.sched;
  int32_t* order = p.sched + A + 1;
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  for (int i = tid; i < kSortBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  // offsets must be monotone, start at 0, end at the totals, and respect the maxima
  int my_bad = 0;
  if (tid == 0) {
    my_bad |= ao[0] != 0 || static_cast<int64_t>(ao[A]) != p.total_anchor_tokens;
    my_bad |= asp[0] != 0 || asp[A] != S;
    my_bad |= so[0] != 0 || static_cast<int64_t>(so[S]) != p.total_suffix_tokens;
  }
  for (int a = tid; a < A; a += blockDim.x) {
    const int la = ao[a + 1] - ao[a];
    my_bad |= la < 0 || la > p.max_anchor_len || asp[a + 1] < asp[a];
  }
  for (int s = tid; s < S; s += blockDim.x) {
    const int ls = so[s + 1] - so[s];
    my_bad |= ls < 0 || ls > p.max_suffix_len;
  }
  if (my_bad) atomicOr(&bad, 1);
  __syncthreads();
  if (bad) {
    if (tid == 0) atomicOr(p.err_word, kErrDeviceBounds);
    for (int i = tid; i <= A; i += blockDim.x) prefix[i] = 0;
    return;
  }
  const int pair_tok = 2 * p.tok_per_tile;
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
  __threadfence_block();
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < A; base += blockDim.x) {
    const int i = base + tid;
    int v = 0;
    if (i < A) {
      const int a = order[i];
      const int ntok = so[asp[a + 1]] - so[asp[a]];
      v = p.hkv * ((ntok + pair_tok - 1) / pair_tok);
    }
    int total;
    const int ex = block_exclusive_scan(v, warp_sums, total);
    if (i < A) prefix[i] = carry + ex;
    carry += total;
  }
  if (tid == 0) prefix[A] = carry;
}

}  // namespace

size_t cascade_workspace_bytes(int num_anchors) {
  const size_t words = 2 * static_cast<size_t>(num_anchors) + 1;
  return (words * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
}

template <int D>
static cudaError_t launch_cascade_d(const CascadeParams& p, const CascadeMaps& maps,
                                    int num_sms, cudaStream_t stream) {
  using C = Cfg<D>;
  cudaError_t e = cudaFuncSetAttribute(cascade_attn_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t pair_tok = 2 * p.tok_per_tile;
  const int64_t bound =
      static_cast<int64_t>(p.hkv) * ((p.total_suffix_tokens + pair_tok - 1) / pair_tok + p.num_anchors);
  const int grid = static_cast<int>(bound < num_sms ? bound : num_sms);
  if (grid <= 0) return cudaSuccess;
  cascade_attn_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(p, maps);
  return cudaGetLastError();
}

cudaError_t launch_cascade(const CascadeParams& p, const CascadeMaps& maps, int head_dim,
                           int num_sms, cudaStream_t stream) {
  cascade_schedule_kernel<<<1, 1024, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (head_dim == 128) return launch_cascade_d<128>(p, maps, num_sms, stream);
  return launch_cascade_d<64>(p, maps, num_sms, stream);
}

}  // namespace quail
