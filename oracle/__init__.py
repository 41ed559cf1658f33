"""CPU oracle for the tree-verification path — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct numpy float64 restatement of what the path
computes, used to prove the CUDA path right. Only `tests/`,
`__graft_entry__.smoke()` and `bench.py`'s CPU-baseline / reference leg may
import it. The product (the CUDA library and its binding) never imports,
links or runs anything here, and this package shares no code with it.

Modules and the passages they follow (page title, then section):
  tree_mask   "EAGLE-2 deep dive" (techknowgenie), section on the core engineering
              implementation: the draft-tree construction ends by marking, for each
              node, the node itself and every ancestor up to the root in a 2-D tree
              mask; the architecture section injects that mask into attention.
  attention   same page, architecture section ("one target forward over all tree
              tokens ... 2-D tree mask injected into the FlashAttention kernel") and
              production section (paged tree attention); "Accelerating Sonar through
              speculation" (Perplexity), EAGLE section (tree verification needs a
              custom mask). The oracle is the plain definition: softmax over the
              allowed keys with an explicit dense boolean mask.
  accept      "EAGLE-2 deep dive", architecture section (target logits contrasted with
              the draft tokens; the longest accepted path is fixed) and benchmark
              section (rejection sampling, lossless at temperature 0 and under
              sampling); "Accelerating Sonar", speculative-decoding section (n draft
              tokens give up to n+1 output tokens; the target's logits at the
              mismatch or end give the extra token) and draft-target section
              (acceptance compares the full draft and target distributions).
  commit      "EAGLE-2 deep dive", architecture section (verification must not
              contaminate the target KV cache); "Accelerating Sonar", draft-target and
              MTP-schedule sections (KV entries filled for accepted tokens; a kernel
              inserts the next token after the shift, with no CPU sync: token_insert).

  draft_tree  "EAGLE-2 deep dive", section on the dynamic draft-tree algorithm (confidence =
              product of draft probabilities along the path; a priority queue pops the
              best candidate; nodes below the depth limit are expanded into top-k).
  fp8         "EAGLE-3 paper explainer" (0h-n0), operations section, model-optimisation list
              (quantisation and PagedAttention KV-cache tuning to cut GPU memory): the E4M3
              codes and per-KV-head scales of an FP8 paged KV cache, used by attention and
              commit when a `kv_scale` is given.

Readings where the pages are silent are stated in each function's docstring.
Every function here is pinned by `tests/test_oracle_*.py` against brute force,
closed forms, textbook routines or hand-worked examples in `tests/golden/`.
"""

from .tree_mask import ancestor_mask, ancestor_mask_batch, pack_mask_words
from .attention import tree_verify_attention, tree_verify_attention_rows, gather_prefix
from .accept import greedy_accept, stochastic_accept, AcceptResult
from .commit import kv_commit, token_insert
from .draft_tree import best_first_tree, topk_softmax
from .fp8 import e4m3_decode, e4m3_encode, kv_quantize, kv_dequantize

__all__ = [
    "ancestor_mask",
    "ancestor_mask_batch",
    "pack_mask_words",
    "tree_verify_attention",
    "tree_verify_attention_rows",
    "gather_prefix",
    "greedy_accept",
    "stochastic_accept",
    "AcceptResult",
    "kv_commit",
    "token_insert",
    "best_first_tree",
    "topk_softmax",
    "e4m3_decode",
    "e4m3_encode",
    "kv_quantize",
    "kv_dequantize",
]
