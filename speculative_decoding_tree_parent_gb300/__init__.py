"""GB300-native verification hot path of tree speculative decoding.

Four steps, each a hand-written sm_103a CUDA kernel family behind a C ABI
(`include/spec_verify.h`, library `libspecverify.so`):

  spec_build_tree_mask   parent array -> per-node ancestor bitmasks (+ depth)
  spec_tree_verify_attn  paged, GQA tree-verify attention (prefix unmasked,
                         in-tree tile bit-masked)
  spec_accept            greedy / stochastic acceptance of the longest path + bonus
  spec_kv_commit         copy of the accepted path's K/V into the paged cache

`binding` is the thin ctypes layer over the library (argument marshalling only);
`workloads` draws the seeded synthetic inputs. Importing the package loads
nothing: the library is opened on first use of `binding`.
"""

__all__ = ["binding", "workloads"]
