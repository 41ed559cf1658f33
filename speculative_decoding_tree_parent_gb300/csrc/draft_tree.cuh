// Host/device interface of the draft-tree kernels (draft_tree.cu).
#pragma once

#include "common.cuh"

namespace specv {

constexpr int kTreeMaxW = 8;  // rows per sequence of one multi-row expansion call

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
  // multi-row call only: at most `width` requests per sequence for the next call
  int width;
  int32_t* req_parent;   // [batch][width]: parent node of request j (-1: the root; past req_n: -1)
  int32_t* req_token;    // [batch][width]: its token
  int32_t* req_n;        // [batch]: requests listed (0 once the tree is complete)
};

size_t tree_state_bytes(int batch, int max_nodes);
int launch_tree_init(const int32_t* root_tokens, int batch, const TreeArgs& a, cudaStream_t stream);
int launch_tree_expand(const float* logits, int vocab, long row_stride, long node_stride, int batch,
                       const TreeArgs& a, cudaStream_t stream);
int launch_tree_expand_multi(const float* logits, int vocab, long row_stride, long req_stride, int batch,
                             const TreeArgs& a, cudaStream_t stream);

}  // namespace specv
