// Host/device interface of the draft-tree kernels (draft_tree.cu).
#pragma once

#include "common.cuh"

namespace specv {

struct TreeArgs {
  uint8_t* state;        // per-sequence construction state (tree_state_bytes)
  int max_nodes, topk, max_depth;
  double threshold;      // candidates scoring at or below it are dropped; <= 0: none
  int32_t* parent_out;   // [batch][max_nodes]
  int32_t* tokens_out;   // [batch][max_nodes]
  int32_t* n_nodes_out;  // [batch]
  int32_t* next_node;    // [batch]: node awaiting its expansion, -1 once the tree is complete
  uint8_t* flags;        // [batch] (nullable): bit 0 = a near-tie pop
  int32_t* status;
};

size_t tree_state_bytes(int batch, int max_nodes);
int launch_tree_init(const int32_t* root_tokens, int batch, const TreeArgs& a, cudaStream_t stream);
int launch_tree_expand(const float* logits, int vocab, long row_stride, long node_stride, int batch,
                       const TreeArgs& a, cudaStream_t stream);

}  // namespace specv
