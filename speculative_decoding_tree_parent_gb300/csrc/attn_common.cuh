// Shared pieces of the tree-verify attention kernels: key-split plan, workspace
// layout of the split partials, and the log-sum-exp merge of the splits.
//
// Key space of sequence b: blocks of kb keys; first ceil(P_b / kb) prefix blocks
// (slots read through the page table, never masked; the last one is cut at P_b),
// then ceil(N_b / kb) tree blocks (tree K/V, filtered by the ancestor mask bits).
// Split s of S takes the contiguous run [s*total/S, (s+1)*total/S) of that combined
// block list, so the tree blocks fall in the last split(s) and split sizes differ by
// at most one block.
// ("Accelerating Sonar through speculation", EAGLE section: a custom mask over the
// whole sequence is what slows attention, so only tree blocks are masked.)
#pragma once

#include "common.cuh"

namespace specv {

struct SplitRange {
  int blk_lo, blk_hi;   // combined block indices [lo, hi)
  int n_prefix_blocks;  // blocks before this index are prefix blocks
};

__device__ __forceinline__ SplitRange split_range(int P, int N, int kb, int splits, int s) {
  SplitRange r;
  r.n_prefix_blocks = (P + kb - 1) / kb;
  const int total = r.n_prefix_blocks + (N + kb - 1) / kb;
  r.blk_lo = (int)((long)s * total / splits);        // sizes differ by at most one block
  r.blk_hi = (int)((long)(s + 1) * total / splits);
  return r;
}

// Workspace of the key-split partials: per split s and output row (t * Hq + h):
// unnormalised O (fp32, D values) and (m, l) with m the running max of the scores
// in log2 units and l = sum 2^(score - m).
struct AttnWs {
  float* o;   // [S][rows][D]
  float2* ml; // [S][rows]
  static size_t bytes(int splits, int rows, int d) {
    return align_up((size_t)splits * rows * d * sizeof(float), 256) +
           align_up((size_t)splits * rows * sizeof(float2), 256);
  }
  static AttnWs at(void* ws, int splits, int rows, int d) {
    AttnWs w;
    w.o = static_cast<float*>(ws);
    w.ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) +
                                     align_up((size_t)splits * rows * d * sizeof(float), 256));
    return w;
  }
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Split counts (host side; the workspace size and the launch use the same rule).
int attn_splits_simt(int batch, int max_nodes, int hq, int hkv, int max_prefix);
int attn_splits_tc(int batch, int max_nodes, int hq, int hkv, int max_prefix);

int launch_attn_combine(int dtype, const AttnWs& w, int splits, int total_nodes, int hq, int d,
                        void* out, float* lse, cudaStream_t stream);

}  // namespace specv
