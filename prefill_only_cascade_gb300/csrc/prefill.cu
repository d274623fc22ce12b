// prefill.cu - causal self-attention over packed sequences (the anchors' own prefill,
// the step before the cascade of "Motor de inferência Quail atinge 1 bilhão de tokens por
// minuto por GPU", section "Como funciona", cascade-attention bullet). It is the cascade
// with one anchor of length 0 whose suffixes are the sequences: the same kernels run, and
// the two query tiles of a work item share their key tiles whenever both lie in one
// sequence.
#include <cstdint>

#include <cmath>

#include <cuda_runtime.h>

#include "kernels.h"
#include "quail.h"

namespace {

constexpr size_t kMetaBytes = 256;  // [0, 0] anchor offsets, [0, S] anchor->suffix map

// Workspace: meta, then the per-row K/V maxima [T, Hkv, 2] uint16 (used when the K/V
// amax is formed), then the cascade's own workspace.
size_t rowmax_bytes(int64_t total_tokens, int32_t num_kv_heads) {
  return (static_cast<size_t>(total_tokens) * num_kv_heads * 4 + 255) / 256 * 256;
}

__global__ void prefill_meta_kernel(int32_t* meta, int32_t num_seqs) {
  meta[0] = 0;  // anchor_offsets: one anchor of length 0
  meta[1] = 0;
  meta[2] = 0;  // anchor_suffix_ptr: its suffixes are all the sequences
  meta[3] = num_seqs;
}

quail_cascade_desc prefill_desc(int32_t num_seqs, int64_t total_tokens, int32_t max_seq_len,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                float softmax_scale) {
  quail_cascade_desc d{};
  d.num_anchors = num_seqs > 0 ? 1 : 0;
  d.num_suffixes = num_seqs;
  d.total_anchor_tokens = 0;
  d.total_suffix_tokens = total_tokens;
  d.max_anchor_len = 0;
  d.max_suffix_len = max_seq_len;
  d.num_q_heads = num_q_heads;
  d.num_kv_heads = num_kv_heads;
  d.head_dim = head_dim;
  d.softmax_scale = softmax_scale;
  d.kv_anchor_dtype = QUAIL_BF16;
  return d;
}

}  // namespace

extern "C" {

size_t quail_causal_prefill_workspace_size(int32_t num_seqs, int64_t total_tokens,
                                           int32_t max_seq_len, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim) {
  if (num_seqs < 0 || total_tokens < 0 || max_seq_len < 0) return 0;
  const quail_cascade_desc d = prefill_desc(num_seqs, total_tokens, max_seq_len, num_q_heads,
                                            num_kv_heads, head_dim, 0.0f);
  const size_t inner = quail_cascade_workspace_size(&d);
  return inner == 0 ? 0 : kMetaBytes + rowmax_bytes(total_tokens, num_kv_heads) + inner;
}

quail_status quail_causal_prefill_attn(int32_t num_seqs, int64_t total_tokens,
                                       int32_t max_seq_len, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim,
                                       float softmax_scale, const void* q, const void* k,
                                       const void* v, const int32_t* seq_offsets, void* out,
                                       float* lse, float* k_amax, float* v_amax,
                                       void* workspace, size_t workspace_bytes,
                                       quail_stream_t stream) {
  // Host checks first (the cascade's, for this shape), so that nothing is launched when
  // the arguments are rejected.
  if (num_seqs < 0 || total_tokens < 0 || total_tokens > (1ll << 31) - 1 || max_seq_len < 0)
    return QUAIL_ERR_INVALID_ARG;
  if (num_seqs == 0) return total_tokens == 0 ? QUAIL_OK : QUAIL_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return QUAIL_ERR_INVALID_ARG;
  if (!(softmax_scale >= 0.0f) || !(softmax_scale < INFINITY)) return QUAIL_ERR_INVALID_ARG;
  const int group = num_q_heads / num_kv_heads;
  if (head_dim != 64 && head_dim != 128) return QUAIL_ERR_UNSUPPORTED;
  if (group != 1 && group != 2 && group != 4 && group != 8 && group != 16)
    return QUAIL_ERR_UNSUPPORTED;
  if (seq_offsets == nullptr || (reinterpret_cast<uintptr_t>(seq_offsets) & 3u))
    return QUAIL_ERR_INVALID_ARG;
  if (total_tokens > 0 &&
      (q == nullptr || k == nullptr || v == nullptr || out == nullptr ||
       ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v)) & 15u) ||
       (reinterpret_cast<uintptr_t>(out) & 31u)))
    return QUAIL_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return QUAIL_ERR_INVALID_ARG;
  if ((k_amax == nullptr) != (v_amax == nullptr) ||
      ((reinterpret_cast<uintptr_t>(k_amax) | reinterpret_cast<uintptr_t>(v_amax)) & 3u))
    return QUAIL_ERR_INVALID_ARG;
  const size_t need = quail_causal_prefill_workspace_size(num_seqs, total_tokens, max_seq_len,
                                                          num_q_heads, num_kv_heads, head_dim);
  if (need == 0 || workspace == nullptr || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & (kMetaBytes - 1)))
    return QUAIL_ERR_INVALID_ARG;
  if (quail::cascade_item_bound(1, total_tokens, num_kv_heads, group) > (1ll << 31) - 1)
    return QUAIL_ERR_UNSUPPORTED;

  const quail_cascade_desc d = prefill_desc(num_seqs, total_tokens, max_seq_len, num_q_heads,
                                            num_kv_heads, head_dim, softmax_scale);
  int32_t* meta = static_cast<int32_t*>(workspace);
  prefill_meta_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(meta, num_seqs);
  if (cudaGetLastError() != cudaSuccess) return QUAIL_ERR_CUDA;
  // k and v double as the (empty) anchor key/value tensors: T_A = 0, nothing is read
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  const size_t front = kMetaBytes + rowmax_bytes(total_tokens, num_kv_heads);
  if (k_amax != nullptr)
    return quail::cascade_attn_with_amax(&d, q, k, v, k, v, meta, meta + 2, seq_offsets, out,
                                         lse, k_amax, v_amax,
                                         reinterpret_cast<uint16_t*>(wsb + kMetaBytes),
                                         wsb + front, workspace_bytes - front, stream);
  return quail_cascade_attn(&d, q, k, v, k, v, meta, meta + 2, seq_offsets, nullptr, nullptr,
                            out, lse, wsb + front, workspace_bytes - front, stream);
}

}  // extern "C"
