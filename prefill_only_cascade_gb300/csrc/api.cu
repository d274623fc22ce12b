// api.cu - the C ABI of libquail (declared in include/quail.h): argument validation on
// the host, tensor-map encoding, and launches on the caller's stream. No call allocates.
#include <cmath>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "quail.h"

namespace {

// The library's device error word (one per device context). Kernels OR bits into it;
// quail_get_device_error() reads and clears it.
__device__ unsigned g_quail_error_word;

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

struct DeviceState {
  bool ready = false;
  quail_status status = QUAIL_ERR_CUDA;
  int num_sms = 0;
  unsigned* err_word = nullptr;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
uint64_t g_timeout_ns = kDefaultTimeoutNs;
int g_inject_skip = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device set-up: the device must be a GB300 (compute capability 10.3).
quail_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QUAIL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    st.ready = true;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      st.status = QUAIL_ERR_CUDA;
    } else if (prop.major != 10 || prop.minor != 3) {
      st.status = QUAIL_ERR_UNSUPPORTED;
    } else if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err_word),
                                    g_quail_error_word) != cudaSuccess) {
      st.status = QUAIL_ERR_CUDA;
    } else {
      st.num_sms = prop.multiProcessorCount;
      st.status = QUAIL_OK;
      if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
          st.status = QUAIL_ERR_CUDA;
        } else {
          g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
      }
    }
  }
  *out = &st;
  return st.status;
}

}  // namespace

int quail::current_device_status() {
  DeviceState* st = nullptr;
  return static_cast<int>(device_state(&st));
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D tensor map over [tokens, heads, d] (innermost d), box (box_inner elements of d,
// box_heads, box_rows), 128-byte swizzle unless given; out-of-range rows read as zero.
bool encode_3d(CUtensorMap* m, const void* base, int64_t tokens, int heads, int d,
               int box_heads, int box_rows, CUtensorMapDataType dt, int elem_bytes, int box_inner,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem_bytes,
                                 static_cast<cuuint64_t>(heads) * d * elem_bytes};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner),
                             static_cast<cuuint32_t>(box_heads),
                             static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool valid_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

}  // namespace

extern "C" {

const char* quail_version(void) { return "quail-gb300 0.1"; }

const char* quail_status_string(quail_status s) {
  switch (s) {
    case QUAIL_OK: return "QUAIL_OK";
    case QUAIL_ERR_INVALID_ARG: return "QUAIL_ERR_INVALID_ARG";
    case QUAIL_ERR_UNSUPPORTED: return "QUAIL_ERR_UNSUPPORTED";
    case QUAIL_ERR_CUDA: return "QUAIL_ERR_CUDA";
    case QUAIL_ERR_TIMEOUT: return "QUAIL_ERR_TIMEOUT";
    case QUAIL_ERR_DEVICE_BOUNDS: return "QUAIL_ERR_DEVICE_BOUNDS";
  }
  return "QUAIL_ERR_UNKNOWN";
}

void quail_set_wait_timeout_ns(uint64_t ns) {
  std::lock_guard<std::mutex> lock(g_mutex);
  g_timeout_ns = ns == 0 ? kDefaultTimeoutNs : ns;
}

quail_status quail_set_cta_pairs(int32_t mode) {
  if (mode != QUAIL_CTA_PAIRS_OFF && mode != QUAIL_CTA_PAIRS_AUTO && mode != QUAIL_CTA_PAIRS_ALWAYS)
    return QUAIL_ERR_INVALID_ARG;
  quail::set_cta_pairs(mode);
  return QUAIL_OK;
}

void quail_debug_inject(int32_t skip_first_kv_load) {
  std::lock_guard<std::mutex> lock(g_mutex);
  g_inject_skip = skip_first_kv_load != 0;
}

// FP8 anchor KV: bytes of each bf16 copy of the anchor codes staged in the workspace.
static int64_t anchor_bf16_bytes(const quail_cascade_desc& d) {
  if (d.kv_anchor_dtype != QUAIL_FP8_E4M3 || d.total_anchor_tokens <= 0 ||
      (d.head_dim != 64 && d.head_dim != 128))
    return 0;
  return d.total_anchor_tokens * d.num_kv_heads * d.head_dim * 2;
}

size_t quail_cascade_workspace_size(const quail_cascade_desc* desc) {
  if (desc == nullptr || desc->num_anchors < 0 || desc->total_suffix_tokens < 0 ||
      desc->num_q_heads <= 0 || desc->num_kv_heads <= 0 ||
      desc->num_q_heads % desc->num_kv_heads != 0 ||
      !valid_group(desc->num_q_heads / desc->num_kv_heads))
    return 0;
  const int64_t bound = quail::cascade_item_bound(
      desc->num_anchors, desc->total_suffix_tokens, desc->num_kv_heads,
      desc->num_q_heads / desc->num_kv_heads);
  return quail::cascade_workspace_layout(desc->num_anchors, desc->total_suffix_tokens, bound,
                                         anchor_bf16_bytes(*desc))
      .total;
}

quail_status quail_get_device_error(quail_stream_t stream) {
  DeviceState* st = nullptr;
  const quail_status s = device_state(&st);
  if (s != QUAIL_OK) return s;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return QUAIL_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, st->err_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return QUAIL_ERR_CUDA;
  if (word == 0) return QUAIL_OK;
  if (cudaMemset(st->err_word, 0, sizeof(unsigned)) != cudaSuccess) return QUAIL_ERR_CUDA;
  if (word & quail::kErrTimeout) return QUAIL_ERR_TIMEOUT;
  return QUAIL_ERR_DEVICE_BOUNDS;
}

}  // extern "C"

namespace {

// Validation of one cascade call and the kernels' parameters. `extra_bytes` is workspace
// that the caller's variant needs after the cascade's own (256-byte aligned start).
// Returns QUAIL_OK with *nothing = true when there is no work (T_S = 0).
quail_status prepare_cascade(const quail_cascade_desc* desc, const void* q_suf, const void* k_anc,
                             const void* v_anc, const void* k_suf, const void* v_suf,
                             const int32_t* anchor_offsets, const int32_t* anchor_suffix_ptr,
                             const int32_t* suffix_offsets, const float* k_scale,
                             const float* v_scale, void* out, float* lse, void* workspace,
                             size_t workspace_bytes, size_t extra_bytes, quail::CascadeParams* pp,
                             quail::CascadeMaps* mp, DeviceState** stp, size_t* ws_used,
                             bool* nothing) {
  *nothing = false;
  if (desc == nullptr) return QUAIL_ERR_INVALID_ARG;
  const quail_cascade_desc& d = *desc;
  const int64_t kMaxTok = (1ll << 31) - 1;
  if (d.num_anchors < 0 || d.num_suffixes < 0 || d.total_anchor_tokens < 0 ||
      d.total_suffix_tokens < 0 || d.total_anchor_tokens > kMaxTok ||
      d.total_suffix_tokens > kMaxTok || d.max_anchor_len < 0 || d.max_suffix_len < 0)
    return QUAIL_ERR_INVALID_ARG;
  if (d.num_q_heads <= 0 || d.num_kv_heads <= 0 || d.num_q_heads % d.num_kv_heads != 0)
    return QUAIL_ERR_INVALID_ARG;
  if (!(d.softmax_scale >= 0.0f) || !std::isfinite(d.softmax_scale)) return QUAIL_ERR_INVALID_ARG;
  if (d.kv_anchor_dtype != QUAIL_BF16 && d.kv_anchor_dtype != QUAIL_FP8_E4M3)
    return QUAIL_ERR_INVALID_ARG;
  const bool fp8 = d.kv_anchor_dtype == QUAIL_FP8_E4M3;
  if (fp8 ? (k_scale == nullptr || v_scale == nullptr) : (k_scale != nullptr || v_scale != nullptr))
    return QUAIL_ERR_INVALID_ARG;
  if (d.num_suffixes == 0 && d.total_suffix_tokens != 0) return QUAIL_ERR_INVALID_ARG;
  if (d.num_anchors == 0 && (d.num_suffixes != 0 || d.total_anchor_tokens != 0))
    return QUAIL_ERR_INVALID_ARG;
  const int group = d.num_q_heads / d.num_kv_heads;
  if (d.head_dim != 64 && d.head_dim != 128) return QUAIL_ERR_UNSUPPORTED;
  if (!valid_group(group)) return QUAIL_ERR_UNSUPPORTED;
  if (anchor_offsets == nullptr || anchor_suffix_ptr == nullptr || suffix_offsets == nullptr)
    return QUAIL_ERR_INVALID_ARG;
  if (d.total_suffix_tokens > 0) {
    if (q_suf == nullptr || k_suf == nullptr || v_suf == nullptr || out == nullptr)
      return QUAIL_ERR_INVALID_ARG;
    if (!aligned16(q_suf) || !aligned16(k_suf) || !aligned16(v_suf) ||
        (reinterpret_cast<uintptr_t>(out) & 31u))  // out rows are written with 32-byte stores
      return QUAIL_ERR_INVALID_ARG;
  }
  if (d.total_anchor_tokens > 0) {
    if (k_anc == nullptr || v_anc == nullptr) return QUAIL_ERR_INVALID_ARG;
    if (!aligned16(k_anc) || !aligned16(v_anc)) return QUAIL_ERR_INVALID_ARG;
  }
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return QUAIL_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(anchor_offsets) | reinterpret_cast<uintptr_t>(anchor_suffix_ptr) |
       reinterpret_cast<uintptr_t>(suffix_offsets)) & 3u)
    return QUAIL_ERR_INVALID_ARG;
  const int64_t item_bound =
      quail::cascade_item_bound(d.num_anchors, d.total_suffix_tokens, d.num_kv_heads, group);
  if (item_bound > (1ll << 31) - 1) return QUAIL_ERR_UNSUPPORTED;
  const quail::CascadeWorkspace wl = quail::cascade_workspace_layout(
      d.num_anchors, d.total_suffix_tokens, item_bound, anchor_bf16_bytes(d));
  *ws_used = wl.total;
  if (workspace == nullptr || workspace_bytes < wl.total + extra_bytes || !aligned16(workspace))
    return QUAIL_ERR_INVALID_ARG;

  DeviceState* st = nullptr;
  const quail_status ds = device_state(&st);
  if (ds != QUAIL_OK) return ds;
  *stp = st;
  if (d.total_suffix_tokens == 0) {  // nothing to compute
    *nothing = true;
    return QUAIL_OK;
  }

  const int D = d.head_dim;
  const int tok = 128 / group;
  quail::CascadeMaps& maps = *mp;
  std::memset(&maps, 0, sizeof(maps));
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  // FP8 anchor KV: the kernels read the bf16 copies that the staging kernel writes into
  // the workspace.
  const void* k_anc_tiles = fp8 ? static_cast<const void*>(wsb + wl.k_anc_bf16) : k_anc;
  const void* v_anc_tiles = fp8 ? static_cast<const void*>(wsb + wl.v_anc_bf16) : v_anc;
  bool ok =
      encode_3d(&maps.q, q_suf, d.total_suffix_tokens, d.num_q_heads, D, group, tok, bf, 2, 64) &&
      encode_3d(&maps.k_suf, k_suf, d.total_suffix_tokens, d.num_kv_heads, D, 1, 128, bf, 2, 64) &&
      encode_3d(&maps.v_suf, v_suf, d.total_suffix_tokens, d.num_kv_heads, D, 1, 128, bf, 2, 64);
  // K with 64-row boxes: the halves of a key tile that the two CTAs of a pair load
  ok = ok && encode_3d(&maps.k_suf64, k_suf, d.total_suffix_tokens, d.num_kv_heads, D, 1, 64,
                       bf, 2, 64);
  if (d.total_anchor_tokens > 0) {
    ok = ok &&
         encode_3d(&maps.k_anc, k_anc_tiles, d.total_anchor_tokens, d.num_kv_heads, D, 1, 128, bf, 2, 64) &&
         encode_3d(&maps.v_anc, v_anc_tiles, d.total_anchor_tokens, d.num_kv_heads, D, 1, 128, bf, 2, 64) &&
         encode_3d(&maps.k_anc64, k_anc_tiles, d.total_anchor_tokens, d.num_kv_heads, D, 1, 64, bf, 2, 64);
  } else {
    maps.k_anc = maps.k_suf;  // never read: every anchor is empty
    maps.v_anc = maps.v_suf;
    maps.k_anc64 = maps.k_suf64;
  }
  // the output, for the epilogue's TMA stores: one warp's 32 rows (32 / G tokens x G heads)
  // by 32 columns of d, 64 bytes a row (64-byte swizzle)
  ok = ok && encode_3d(&maps.out, out, d.total_suffix_tokens, d.num_q_heads, D, group, 32 / group,
                       bf, 2, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok) return QUAIL_ERR_CUDA;

  quail::CascadeParams& p = *pp;
  std::memset(&p, 0, sizeof(p));
  p.num_anchors = d.num_anchors;
  p.num_suffixes = d.num_suffixes;
  p.total_anchor_tokens = d.total_anchor_tokens;
  p.total_suffix_tokens = d.total_suffix_tokens;
  p.max_anchor_len = d.max_anchor_len;
  p.max_suffix_len = d.max_suffix_len;
  p.hq = d.num_q_heads;
  p.hkv = d.num_kv_heads;
  p.group = group;
  p.tok_per_tile = tok;
  const float scale = d.softmax_scale > 0.0f ? d.softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  p.scale_log2 = scale * 1.4426950408889634f;
  p.fp8 = fp8;
  p.anchor_offsets = anchor_offsets;
  p.anchor_suffix_ptr = anchor_suffix_ptr;
  p.suffix_offsets = suffix_offsets;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.q_suf = q_suf;
  p.k_anc = k_anc;
  p.v_anc = v_anc;
  p.k_suf = k_suf;
  p.v_suf = v_suf;
  p.out = out;
  p.lse = lse;
  p.item_bound = static_cast<int>(item_bound);
  p.flag = reinterpret_cast<int32_t*>(wsb + wl.flag);
  p.prefix = reinterpret_cast<int32_t*>(wsb + wl.prefix);
  p.order = reinterpret_cast<int32_t*>(wsb + wl.order);
  p.seg = reinterpret_cast<int32_t*>(wsb + wl.seg);
  p.items = reinterpret_cast<int32_t*>(wsb + wl.items);
  p.redo_count = reinterpret_cast<int32_t*>(wsb + wl.redo_count);
  p.redo_flag = reinterpret_cast<int32_t*>(wsb + wl.redo_flag);
  p.redo_list = reinterpret_cast<int32_t*>(wsb + wl.redo_list);
  p.k_anc_bf16 = fp8 ? wsb + wl.k_anc_bf16 : nullptr;
  p.v_anc_bf16 = fp8 ? wsb + wl.v_anc_bf16 : nullptr;
  p.mode = quail::kFused;
  p.merge = 0;
  p.tiles_per_item = 2;  // launch_cascade picks the item shape for the kernel it runs
  p.o_part = nullptr;
  p.lse_part = nullptr;
  p.err_word = st->err_word;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    p.timeout_ns = g_timeout_ns;
    p.inject_skip_first_kv = g_inject_skip;
  }
  return QUAIL_OK;
}

// Extra workspace of the two-pass variant after the cascade's own: fp32 O_a [T_S, Hq, d],
// lse_a and lse_s [T_S, Hq].
struct TwoPassLayout {
  size_t o_part, lse_part, lse_s, total;
};
TwoPassLayout two_pass_layout(const quail_cascade_desc& d, size_t base) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = static_cast<size_t>(d.total_suffix_tokens) * d.num_q_heads;
  TwoPassLayout t;
  t.o_part = up(base);
  t.lse_part = up(t.o_part + rows * d.head_dim * 4);
  t.lse_s = up(t.lse_part + rows * 4);
  t.total = up(t.lse_s + rows * 4);
  return t;
}

}  // namespace

extern "C" {

quail_status quail_cascade_attn(const quail_cascade_desc* desc, const void* q_suf,
                                const void* k_anc, const void* v_anc, const void* k_suf,
                                const void* v_suf, const int32_t* anchor_offsets,
                                const int32_t* anchor_suffix_ptr,
                                const int32_t* suffix_offsets, const float* k_scale,
                                const float* v_scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes,
                                quail_stream_t stream) {
  quail::CascadeParams p;
  quail::CascadeMaps maps;
  DeviceState* st = nullptr;
  size_t used = 0;
  bool nothing = false;
  const quail_status s = prepare_cascade(desc, q_suf, k_anc, v_anc, k_suf, v_suf,
                                         anchor_offsets, anchor_suffix_ptr, suffix_offsets,
                                         k_scale, v_scale, out, lse, workspace, workspace_bytes,
                                         0, &p, &maps, &st, &used, &nothing);
  if (s != QUAIL_OK || nothing) return s;
  const cudaError_t e = quail::launch_cascade(p, maps, desc->head_dim, p.fp8, st->num_sms,
                                              reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QUAIL_OK : QUAIL_ERR_CUDA;
}

}  // extern "C"

// quail_cascade_attn that also forms the max |x| of the suffix K and V per (suffix, KV
// head) into k_amax / v_amax ([S, Hkv] fp32, zeroed here): the causal prefill's path.
quail_status quail::cascade_attn_with_amax(const quail_cascade_desc* desc, const void* q_suf,
                                           const void* k_anc, const void* v_anc,
                                           const void* k_suf, const void* v_suf,
                                           const int32_t* anchor_offsets,
                                           const int32_t* anchor_suffix_ptr,
                                           const int32_t* suffix_offsets, void* out, float* lse,
                                           float* k_amax, float* v_amax, uint16_t* rowmax,
                                           void* workspace, size_t workspace_bytes,
                                           quail_stream_t stream) {
  quail::CascadeParams p;
  quail::CascadeMaps maps;
  DeviceState* st = nullptr;
  size_t used = 0;
  bool nothing = false;
  const quail_status s = prepare_cascade(desc, q_suf, k_anc, v_anc, k_suf, v_suf,
                                         anchor_offsets, anchor_suffix_ptr, suffix_offsets,
                                         nullptr, nullptr, out, lse, workspace, workspace_bytes,
                                         0, &p, &maps, &st, &used, &nothing);
  if (s != QUAIL_OK) return s;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (nothing) {  // no tokens: every sequence is empty, its amax 0
    const size_t n = static_cast<size_t>(desc->num_suffixes) * desc->num_kv_heads * sizeof(float);
    if (n > 0 && (cudaMemsetAsync(k_amax, 0, n, cs) != cudaSuccess ||
                  cudaMemsetAsync(v_amax, 0, n, cs) != cudaSuccess))
      return QUAIL_ERR_CUDA;
    return QUAIL_OK;
  }
  p.k_amax = k_amax;
  p.v_amax = v_amax;
  p.rowmax = rowmax;
  const cudaError_t e = quail::launch_cascade(p, maps, desc->head_dim, false, st->num_sms, cs);
  return e == cudaSuccess ? QUAIL_OK : QUAIL_ERR_CUDA;
}

extern "C" {

size_t quail_cascade_two_pass_workspace_size(const quail_cascade_desc* desc) {
  const size_t base = quail_cascade_workspace_size(desc);
  if (base == 0 || desc->total_suffix_tokens < 0 ||
      (desc->head_dim != 64 && desc->head_dim != 128))
    return 0;
  return two_pass_layout(*desc, base).total;
}

quail_status quail_cascade_attn_two_pass(const quail_cascade_desc* desc, const void* q_suf,
                                         const void* k_anc, const void* v_anc,
                                         const void* k_suf, const void* v_suf,
                                         const int32_t* anchor_offsets,
                                         const int32_t* anchor_suffix_ptr,
                                         const int32_t* suffix_offsets, const float* k_scale,
                                         const float* v_scale, int32_t merge_in_suffix_pass,
                                         void* out, float* lse, void* workspace,
                                         size_t workspace_bytes, quail_stream_t stream) {
  if (desc == nullptr || (merge_in_suffix_pass != 0 && merge_in_suffix_pass != 1))
    return QUAIL_ERR_INVALID_ARG;
  const size_t base = quail_cascade_workspace_size(desc);
  const size_t need = quail_cascade_two_pass_workspace_size(desc);
  quail::CascadeParams p;
  quail::CascadeMaps maps;
  DeviceState* st = nullptr;
  size_t used = 0;
  bool nothing = false;
  const quail_status s = prepare_cascade(
      desc, q_suf, k_anc, v_anc, k_suf, v_suf, anchor_offsets, anchor_suffix_ptr,
      suffix_offsets, k_scale, v_scale, out, lse, workspace, workspace_bytes,
      need > base ? need - base : 0, &p, &maps, &st, &used, &nothing);
  if (s != QUAIL_OK || nothing) return s;
  const TwoPassLayout tl = two_pass_layout(*desc, used);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  float* lse_a = reinterpret_cast<float*>(wsb + tl.lse_part);
  float* lse_s = reinterpret_cast<float*>(wsb + tl.lse_s);
  const int64_t rows = desc->total_suffix_tokens * desc->num_q_heads;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  p.o_part = reinterpret_cast<float*>(wsb + tl.o_part);
  p.lse_part = lse_a;
  // A2: anchor keys only (empty anchors get no items: their lse_a stays -inf)
  cudaError_t e = quail::launch_fill_neg_inf(lse_a, rows, st->num_sms, cs);
  p.mode = quail::kAnchorPass;
  if (e == cudaSuccess) e = quail::launch_cascade(p, maps, desc->head_dim, p.fp8, st->num_sms, cs);
  // A3: the suffix's own keys; A4 merged in its epilogue, or by the merge kernel
  p.mode = quail::kSuffixPass;
  p.merge = merge_in_suffix_pass;
  if (!merge_in_suffix_pass) p.lse = lse_s;
  if (e == cudaSuccess) e = quail::launch_cascade(p, maps, desc->head_dim, false, st->num_sms, cs);
  if (e == cudaSuccess && !merge_in_suffix_pass)
    e = quail::launch_lse_merge(rows, desc->head_dim, p.o_part, lse_a, lse_s, out, lse,
                                st->num_sms, cs);
  return e == cudaSuccess ? QUAIL_OK : QUAIL_ERR_CUDA;
}

size_t quail_join_select_workspace_size(int32_t num_suffixes) {
  return num_suffixes < 0 ? 0 : quail::join_select_workspace_bytes(num_suffixes);
}

quail_status quail_join_select(int32_t num_anchors, int32_t num_suffixes,
                               const int32_t* anchor_suffix_ptr, const int32_t* argmax,
                               int32_t true_index, uint8_t* verdict, int32_t* selected,
                               int32_t* num_selected, int32_t* anchor_count, void* workspace,
                               size_t workspace_bytes, quail_stream_t stream) {
  if (num_anchors < 0 || num_suffixes < 0 || true_index < 0 || true_index > 7)
    return QUAIL_ERR_INVALID_ARG;
  if (num_selected == nullptr || (reinterpret_cast<uintptr_t>(num_selected) & 3u))
    return QUAIL_ERR_INVALID_ARG;
  if (num_suffixes > 0 &&
      (argmax == nullptr || selected == nullptr ||
       ((reinterpret_cast<uintptr_t>(argmax) | reinterpret_cast<uintptr_t>(selected)) & 3u)))
    return QUAIL_ERR_INVALID_ARG;
  if (anchor_count != nullptr && num_anchors > 0 &&
      (anchor_suffix_ptr == nullptr ||
       ((reinterpret_cast<uintptr_t>(anchor_count) |
         reinterpret_cast<uintptr_t>(anchor_suffix_ptr)) & 3u)))
    return QUAIL_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < quail::join_select_workspace_bytes(num_suffixes) ||
      (reinterpret_cast<uintptr_t>(workspace) & 15u))
    return QUAIL_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  const quail_status ds = device_state(&st);
  if (ds != QUAIL_OK) return ds;
  quail::JoinSelectArgs j{num_anchors, num_suffixes, anchor_suffix_ptr, argmax, true_index,
                          verdict, selected, num_selected, anchor_count,
                          static_cast<int32_t*>(workspace)};
  const cudaError_t e = quail::launch_join_select(j, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QUAIL_OK : QUAIL_ERR_CUDA;
}

quail_status quail_restricted_head(int64_t n_rows, int32_t hidden, float eps, const void* h,
                                   int64_t h_rows, int64_t h_row_stride,
                                   const int32_t* row_index, const void* gamma, const void* w8,
                                   float* logits, int32_t* argmax, quail_stream_t stream) {
  if (n_rows < 0 || hidden <= 0 || hidden % 32 != 0 || !(eps >= 0.0f) || !std::isfinite(eps))
    return QUAIL_ERR_INVALID_ARG;
  // without a gather every output row reads the source row of the same index
  if (h_rows < 0 || (row_index == nullptr && n_rows > h_rows)) return QUAIL_ERR_INVALID_ARG;
  if (hidden > 6144) return QUAIL_ERR_UNSUPPORTED;
  if (h_row_stride < hidden || (h_row_stride * 2) % 16 != 0) return QUAIL_ERR_INVALID_ARG;
  if (n_rows > 0) {
    if (h == nullptr || gamma == nullptr || w8 == nullptr || logits == nullptr || argmax == nullptr)
      return QUAIL_ERR_INVALID_ARG;
    if (!aligned16(h) || !aligned16(logits) || (reinterpret_cast<uintptr_t>(argmax) & 3u) ||
        (reinterpret_cast<uintptr_t>(gamma) & 1u) || (reinterpret_cast<uintptr_t>(w8) & 1u) ||
        (reinterpret_cast<uintptr_t>(row_index) & 3u))
      return QUAIL_ERR_INVALID_ARG;
  }
  DeviceState* st = nullptr;
  const quail_status ds = device_state(&st);
  if (ds != QUAIL_OK) return ds;
  quail::HeadArgs a{n_rows, hidden, eps, h, h_rows, h_row_stride, row_index, gamma, w8,
                    logits, argmax, st->err_word};
  const cudaError_t e =
      quail::launch_restricted_head(a, st->num_sms, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QUAIL_OK : QUAIL_ERR_CUDA;
}

static quail_status quantize_checks(int32_t num_anchors, const int32_t* anchor_offsets,
                                    int64_t total_anchor_tokens, int32_t num_kv_heads,
                                    int32_t head_dim, const void* kv_bf16, void* kv_e4m3,
                                    float* scale) {
  if (num_anchors < 0 || total_anchor_tokens < 0 || total_anchor_tokens > (1ll << 31) - 1 ||
      num_kv_heads <= 0)
    return QUAIL_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return QUAIL_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_kv_heads) * head_dim > 4096) return QUAIL_ERR_UNSUPPORTED;
  if (num_anchors == 0 && total_anchor_tokens != 0) return QUAIL_ERR_INVALID_ARG;
  if (num_anchors > 0 && (anchor_offsets == nullptr || scale == nullptr)) return QUAIL_ERR_INVALID_ARG;
  if (total_anchor_tokens > 0 &&
      (kv_bf16 == nullptr || kv_e4m3 == nullptr || !aligned16(kv_bf16) || !aligned16(kv_e4m3)))
    return QUAIL_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scale) | reinterpret_cast<uintptr_t>(anchor_offsets)) & 3u)
    return QUAIL_ERR_INVALID_ARG;
  return QUAIL_OK;
}

quail_status quail_quantize_kv_fp8(int32_t num_anchors, const int32_t* anchor_offsets,
                                   int64_t total_anchor_tokens, int32_t num_kv_heads,
                                   int32_t head_dim, const void* kv_bf16, void* kv_e4m3,
                                   float* scale, quail_stream_t stream) {
  const quail_status c = quantize_checks(num_anchors, anchor_offsets, total_anchor_tokens,
                                         num_kv_heads, head_dim, kv_bf16, kv_e4m3, scale);
  if (c != QUAIL_OK) return c;
  DeviceState* st = nullptr;
  const quail_status ds = device_state(&st);
  if (ds != QUAIL_OK) return ds;
  quail::QuantArgs q{};
  q.num_anchors = num_anchors;
  q.anchor_offsets = anchor_offsets;
  q.total_tokens = total_anchor_tokens;
  q.num_kv_heads = num_kv_heads;
  q.head_dim = head_dim;
  q.kv = kv_bf16;
  q.codes = kv_e4m3;
  q.scale = scale;
  q.err_word = st->err_word;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    q.timeout_ns = g_timeout_ns;
  }
  if (total_anchor_tokens > 0) {
    // [T_A, Hkv * d] bf16, box (hg * d, 32 rows), no swizzle; rows past T_A read as zero
    const int hg = quail::quantize_heads_per_slab(num_kv_heads, head_dim);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(num_kv_heads) * head_dim,
                                static_cast<cuuint64_t>(total_anchor_tokens)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(num_kv_heads) * head_dim * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(hg * head_dim), 32};
    const cuuint32_t estr[2] = {1, 1};
    if (g_encode(&q.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_bf16), dims,
                 strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QUAIL_ERR_CUDA;
  } else {
    // no rows: only the scales (1 each) are written
    const cudaError_t e = quail::launch_quantize_kv_fp8_scaled(
        q, nullptr, st->num_sms, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QUAIL_OK : QUAIL_ERR_CUDA;
  }
  const cudaError_t e =
      quail::launch_quantize_kv_fp8(q, st->num_sms, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QUAIL_OK : QUAIL_ERR_CUDA;
}

quail_status quail_quantize_kv_fp8_with_scales(int32_t num_anchors,
                                               const int32_t* anchor_offsets,
                                               int64_t total_anchor_tokens,
                                               int32_t num_kv_heads, int32_t head_dim,
                                               const void* kv_bf16, const float* amax,
                                               void* kv_e4m3, float* scale,
                                               quail_stream_t stream) {
  const quail_status c = quantize_checks(num_anchors, anchor_offsets, total_anchor_tokens,
                                         num_kv_heads, head_dim, kv_bf16, kv_e4m3, scale);
  if (c != QUAIL_OK) return c;
  if (num_anchors > 0 && (amax == nullptr || (reinterpret_cast<uintptr_t>(amax) & 3u)))
    return QUAIL_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  const quail_status ds = device_state(&st);
  if (ds != QUAIL_OK) return ds;
  quail::QuantArgs q{};
  q.num_anchors = num_anchors;
  q.anchor_offsets = anchor_offsets;
  q.total_tokens = total_anchor_tokens;
  q.num_kv_heads = num_kv_heads;
  q.head_dim = head_dim;
  q.kv = kv_bf16;
  q.codes = kv_e4m3;
  q.scale = scale;
  q.err_word = st->err_word;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    q.timeout_ns = g_timeout_ns;
  }
  const cudaError_t e = quail::launch_quantize_kv_fp8_scaled(
      q, amax, st->num_sms, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QUAIL_OK : QUAIL_ERR_CUDA;
}

}  // extern "C"
