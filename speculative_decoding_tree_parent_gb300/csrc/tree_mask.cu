// K-MASK: ancestor bitmask of every draft-tree node.
//
// "EAGLE-2 deep dive" (techknowgenie), core-implementation section: a node's row
// of the tree mask marks the node and each ancestor, found by following parent
// links to the root; node ids are assigned in creation order so parent[i] < i.
//
// One thread per node. The walk is at most depth+1 steps, each a 4-byte load
// that hits L1 (the whole parent array of a tree is a few hundred bytes). The
// row (W <= 16 words) is built in registers and written once.
#include "common.cuh"

namespace specv {

constexpr int kMaskMaxWords = 16;  // max_nodes <= 1024

template <int W>
__global__ void __launch_bounds__(128) tree_mask_kernel(const int32_t* __restrict__ parent,
                                                        const int32_t* __restrict__ qo, int batch,
                                                        int total_nodes, int max_nodes,
                                                        uint64_t* __restrict__ mask,
                                                        int32_t* __restrict__ depth,
                                                        int32_t* status) {
  pdl_trigger();  // the attention kernel may start its mask-independent prologue
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= total_nodes) return;
  const int b = seq_of_row(qo, batch, t);
  const int base = __ldg(qo + b);
  const int n = __ldg(qo + b + 1) - base;
  const int i = t - base;
  uint64_t row[W];
#pragma unroll
  for (int w = 0; w < W; ++w) row[w] = 0;
  int dep = 0;
  bool ok = true;
  int cur = i;
  // a sequence longer than max_nodes: its rows are written all-zero with depth -1 (no
  // stale bits from an earlier call survive for a later attention to read)
  const bool fits = n <= max_nodes;
  if (!fits) report(status, SPEC_ERR_CAPACITY);
  while (fits) {
#pragma unroll
    for (int w = 0; w < W; ++w)
      if ((cur >> 6) == w) row[w] |= 1ull << (cur & 63);
    const int p = __ldg(parent + base + cur);
    if (cur == 0) {
      if (p != -1) ok = false;
      break;
    }
    if (p < 0 || p >= cur) {
      ok = false;
      break;
    }
    cur = p;
    ++dep;
  }
  if (!fits || !ok) {
    if (fits) report(status, SPEC_ERR_PARENT);
#pragma unroll
    for (int w = 0; w < W; ++w) row[w] = 0;
    dep = -1;
  }
  const int words = (max_nodes + 63) >> 6;
  uint64_t* out = mask + (size_t)t * words;
#pragma unroll
  for (int w = 0; w < W; ++w)
    if (w < words) out[w] = row[w];
  if (depth != nullptr) depth[t] = dep;
}

int launch_tree_mask(const int32_t* parent, const int32_t* qo, int batch, int total_nodes,
                     int max_nodes, uint64_t* mask, int32_t* depth, int32_t* status,
                     cudaStream_t stream) {
  const int words = (max_nodes + 63) >> 6;
  const dim3 grid(ceil_div(total_nodes, 128));
  if (words <= 1)
    tree_mask_kernel<1><<<grid, 128, 0, stream>>>(parent, qo, batch, total_nodes, max_nodes, mask, depth, status);
  else if (words <= 2)
    tree_mask_kernel<2><<<grid, 128, 0, stream>>>(parent, qo, batch, total_nodes, max_nodes, mask, depth, status);
  else if (words <= 4)
    tree_mask_kernel<4><<<grid, 128, 0, stream>>>(parent, qo, batch, total_nodes, max_nodes, mask, depth, status);
  else
    tree_mask_kernel<kMaskMaxWords><<<grid, 128, 0, stream>>>(parent, qo, batch, total_nodes, max_nodes, mask, depth, status);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace specv
