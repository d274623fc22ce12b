"""Float64 CPU oracle for the prefill-only cascade attention and the restricted head.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links this
package: only the tests, the smoke check and the benchmark's CPU-baseline leg do. It
shares no code with the CUDA library and does not import it.

Sources (page titles and sections; the pages print no equations):
  [P1] "Motor de inferência Quail atinge 1 bilhão de tokens por minuto por GPU",
       section "Como funciona": the zero-decode bullet (a boolean AI.IF needs only the last
       prefill pass, which emits one token) and the simplified cascade attention bullet
       (suffixes attend to the anchor, then to themselves; the two results are combined
       by LSE rescaling; the output vocabulary is cut to 8 options, shrinking the final
       unembedding matrix).
  [P2] "Quail: یک میلیارد توکن در دقیقه روی یک GPU", the paragraph on the missing decode
       phase and the key-points list (the model head is restricted to 8 output tokens).
  [P2-SQL] the same page's AI.IF join example: PROMPT("{customers.profile} might buy
       this: {products.description}"), i.e. a shared anchor text followed by a per-pair
       suffix, which fixes "anchor fully visible, suffix causal".

Readings where the pages are silent (each also listed in the design notes):
  softmax scale 1/sqrt(d); natural-log LSE of the scaled scores; query head h uses KV
  head h // (Hq/Hkv); inputs are already rotated (positions are not the kernel's
  concern); RMSNorm y = h * (mean(h^2) + eps)^(-1/2) * gamma with no intermediate
  rounding; argmax takes the lowest index among equal maxima; FP8 is OCP E4M3FN with one
  fp32 scale per (anchor, KV head) = amax / 448 (1 when amax == 0), codes by
  round-to-nearest-even with saturation from the fp32 quotient x / scale.

kv_plan.py: the anchor-KV cache plan of a known query plan (LRU, furthest-next-use,
and the exhaustive minimum regret); pins in tests/test_oracle_kv_plan.py (a hand-worked
plan, furthest-next-use equal to the exhaustive minimum for equal sizes, bounds).

shard.py: sharding one batch over ranks by anchor (visible-pair work per anchor,
longest-processing-time-first, the exhaustive optimum); pins in tests/test_oracle_shard.py
(pair counts from the mask, Graham's bound against the optimum, a textbook worst case).

join.py: the join's verdicts from the head's argmax (verdict per suffix, the passing
suffixes in order, a count per anchor); pins in tests/test_oracle_join.py.

Pins (tests/test_oracle.py): brute-force loops, the cascade-merge = monolithic identity,
closed forms, a library SDPA with an explicit mask, RMSNorm closed forms, all 256 E4M3
codes against the OCP formula and against torch's float8_e4m3fn. No function here is
"parity unpinned".
"""
from .attention import (anchor_partial, cascade_attention, cascade_suffix, lse_merge,
                        suffix_attention, suffix_partial)
from .fp8 import dequantize_kv_fp8, e4m3_decode, e4m3_encode, quantize_kv_fp8
from .head import restricted_head, rmsnorm, top2_margin
from .join import join_select

__all__ = [
    "anchor_partial", "cascade_attention", "cascade_suffix", "lse_merge", "suffix_attention",
    "suffix_partial", "dequantize_kv_fp8", "e4m3_decode", "e4m3_encode", "quantize_kv_fp8", "restricted_head",
    "rmsnorm", "top2_margin",
]
