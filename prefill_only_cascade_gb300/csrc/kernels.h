// kernels.h - internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "quail.h"

namespace quail {

// Status (a quail_status value) of the current device for the library: QUAIL_OK on a
// GB300 after the one-time set-up, else the same code every entry point returns.
int current_device_status();

struct HeadArgs {
  int64_t n_rows;
  int hidden;
  float eps;
  const void* h;
  int64_t h_rows;
  int64_t h_row_stride;
  const int32_t* row_index;
  const void* gamma;
  const void* w8;
  float* logits;
  int32_t* argmax;
  unsigned* err_word;  // the library's device error word (bounds failures)
};
size_t restricted_head_smem_bytes(int hidden);
cudaError_t launch_restricted_head(const HeadArgs& a, int num_sms, cudaStream_t stream);

struct QuantArgs {
  int num_anchors;
  const int32_t* anchor_offsets;
  int64_t total_tokens;
  int num_kv_heads;
  int head_dim;
  const void* kv;
  void* codes;
  float* scale;
  CUtensorMap map;     // 2-D bf16 map over kv [T_A, Hkv * d], box (hg * d, 32 rows)
  unsigned* err_word;
  uint64_t timeout_ns;
};
// Heads per slab of the quantiser (the tensor map's box is hg * d wide).
int quantize_heads_per_slab(int num_kv_heads, int head_dim);
cudaError_t launch_quantize_kv_fp8(const QuantArgs& q, int num_sms, cudaStream_t stream);
// With the amax of every (anchor, KV head) given ([A, Hkv] fp32, device).
cudaError_t launch_quantize_kv_fp8_scaled(const QuantArgs& q, const float* amax, int num_sms,
                                          cudaStream_t stream);

struct JoinSelectArgs {
  int num_anchors;
  int64_t num_suffixes;
  const int32_t* anchor_suffix_ptr;
  const int32_t* argmax;
  int32_t true_index;
  uint8_t* verdict;
  int32_t* selected;
  int32_t* num_selected;
  int32_t* anchor_count;
  int32_t* chunk_work;  // workspace: one int32 per chunk of suffixes
};
size_t join_select_workspace_bytes(int64_t num_suffixes);
cudaError_t launch_join_select(const JoinSelectArgs& j, cudaStream_t stream);

// Everything the cascade kernels need besides the tensor maps.
struct CascadeParams {
  int num_anchors, num_suffixes;
  int64_t total_anchor_tokens, total_suffix_tokens;
  int max_anchor_len, max_suffix_len;
  int hq, hkv, group;        // group = hq / hkv
  int tok_per_tile;          // 128 / group suffix tokens per 128-row query tile
  int item_bound;            // host-known upper bound of work items
  float scale_log2;          // softmax_scale * log2(e)
  bool fp8;
  const int32_t* anchor_offsets;
  const int32_t* anchor_suffix_ptr;
  const int32_t* suffix_offsets;
  const float* k_scale;
  const float* v_scale;
  const void* q_suf;
  const void* k_anc;         // bf16, or e4m3 codes with FP8 anchor KV
  const void* v_anc;
  const void* k_suf;
  const void* v_suf;
  void* out;
  float* lse;
  // workspace (see cascade_workspace_layout)
  int32_t* flag;             // nonzero: a suffix offset check failed
  int32_t* prefix;           // [A+1] work-item prefix over the anchor order; [A] = total
  int32_t* order;            // [A] anchors by decreasing anchor-tile count
  int32_t* seg;              // [T_S] first token of the suffix that holds each token
  int32_t* items;            // [item_bound][12] one record per work item (8 or 12 ints)
  int32_t* redo_count;       // items the speculative kernel handed to the exact one
  int32_t* redo_flag;        // [item_bound] nonzero: item is in redo_list
  int32_t* redo_list;        // [item_bound] item indices, redo_count of them valid
  void* k_anc_bf16;          // FP8 anchor KV: [T_A, Hkv, D] bf16 copies of the codes
  void* v_anc_bf16;
  // Which part of the cascade one launch sequence computes:
  //   kFused       anchor and suffix keys in one online softmax (out, lse)
  //   kAnchorPass  anchor keys only: fp32 normalised O_a -> o_part, lse_a -> lse_part
  //                (anchors of length 0 get no work items; lse_part must hold -inf there)
  //   kSuffixPass  the suffix's own keys only: out / lse as kFused, or with merge != 0
  //                the LSE merge with (o_part, lse_part) done in the epilogue
  int mode;
  int merge;
  // 2: work items of two 128-row query tiles (one CTA each); 4: "quads" of four query
  // tiles for the CTA-pair kernel (the exact kernel then walks quad halves)
  int tiles_per_item;
  float* o_part;             // [T_S, Hq, D] fp32
  float* lse_part;           // [T_S, Hq] fp32 (natural log)
  // Optional (causal prefill): max |x| of the suffix K and V per (suffix, KV head),
  // [S, Hkv] fp32, formed from the K/V tiles already in shared memory via per-row
  // maxima rowmax [T_S, Hkv, 2] (bf16 bit patterns of max |k|, max |v|).
  float* k_amax;
  float* v_amax;
  uint16_t* rowmax;
  unsigned* err_word;
  uint64_t timeout_ns;
  int inject_skip_first_kv;
};

// Byte offsets of the workspace regions; `total` is the size to allocate.
struct CascadeWorkspace {
  size_t flag, redo_count, prefix, order, seg, items, redo_flag, redo_list, k_anc_bf16,
      v_anc_bf16, total;
};
// anchor_bf16_bytes: T_A * Hkv * D * 2 with FP8 anchor KV (each of the two staged
// copies), else 0.
CascadeWorkspace cascade_workspace_layout(int num_anchors, int64_t total_suffix_tokens,
                                          int64_t item_bound, int64_t anchor_bf16_bytes);
int64_t cascade_item_bound(int num_anchors, int64_t total_suffix_tokens, int hkv, int group);

// Tensor maps over q_suf, k/v anchor and k/v suffix (bf16, 3-D: d, head, token).
struct CascadeMaps {
  CUtensorMap q, k_anc, v_anc, k_suf, v_suf;
  CUtensorMap k_anc64, k_suf64;  // the same K tensors with 64-row boxes (CTA-pair halves)
  // bf16 output [T_S, Hq, d] for the epilogue's TMA stores: box (32 of d, G heads, 32 / G
  // tokens) = one warp's rows, 64-byte swizzle (fused mode only)
  CUtensorMap out;
};

// Which d = 128 fused calls run the CTA-pair kernel: QUAIL_CTA_PAIRS_OFF / _AUTO (the
// default) / _ALWAYS.
void set_cta_pairs(int mode);

constexpr int kFused = 0, kAnchorPass = 1, kSuffixPass = 2;

// quail_cascade_attn plus the max |x| of the suffix K and V per (suffix, KV head) into
// k_amax / v_amax ([S, Hkv] fp32), formed by the fast kernel from the tiles it loads.
// rowmax: [T_S, Hkv, 2] uint16 scratch for the per-row maxima.
quail_status cascade_attn_with_amax(const quail_cascade_desc* desc, const void* q_suf,
                                    const void* k_anc, const void* v_anc, const void* k_suf,
                                    const void* v_suf, const int32_t* anchor_offsets,
                                    const int32_t* anchor_suffix_ptr,
                                    const int32_t* suffix_offsets, void* out, float* lse,
                                    float* k_amax, float* v_amax, uint16_t* rowmax,
                                    void* workspace, size_t workspace_bytes,
                                    quail_stream_t stream);

cudaError_t launch_cascade(const CascadeParams& p, const CascadeMaps& maps, int head_dim,
                           bool fp8, int num_sms, cudaStream_t stream);

// Two-pass helpers: lse_part[0, n) = -inf; and the LSE merge of the anchor partial
// (o_part, lse_part) with the suffix partial (out, lse_s) in place into out (and lse).
cudaError_t launch_fill_neg_inf(float* x, int64_t n, int num_sms, cudaStream_t stream);
cudaError_t launch_lse_merge(int64_t rows, int head_dim, const float* o_part,
                             const float* lse_part, const float* lse_s, void* out, float* lse,
                             int num_sms, cudaStream_t stream);

}  // namespace quail
