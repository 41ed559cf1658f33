// K-TREE: the EAGLE-2 dynamic draft tree, built on the device one expansion at a time.
//
// "EAGLE-2 deep dive" (techknowgenie), section on the dynamic draft-tree algorithm: the
// confidence of a node is the product of the draft probabilities along its path from the
// root; a priority queue holds the candidates; the best one is popped and becomes the next
// node; unless it sits at the depth limit it is expanded -- the draft head runs on it and
// its top-k tokens become candidates scored by the product (those at or below a threshold
// are dropped) -- and construction stops at the node budget.
//
// The draft model is not part of this library: between two calls it writes the logits row
// of the node awaiting expansion. spec_tree_expand consumes that row -- the softmax
// statistics and the top-k tokens over the vocabulary, by a cluster of 8 CTAs per sequence,
// each on an eighth of the row: pass 1 takes the slice's max and a threshold (the k-th
// largest of a warp's lane maxima, so at least k elements reach it), the cluster shares both
// through distributed shared memory; pass 2 (the slice again, from L2) sums exp(x - max) and
// keeps the few elements at or above the threshold; each CTA selects its top-k from those and
// rank 0 merges the eight lists -- then rank 0 pushes the k
// candidates and pops until a popped node needs the draft model or the budget is met. The
// candidates, scores and depths live in a caller state buffer, so a whole tree is built with
// one launch per expansion and no host round trip.
//
// Pop order: the largest score, ties to the earliest pushed candidate (the queue's order).
// Scores are fp64 products; a token's probability is exp(x - max) in fp32 times 1 / Z, Z the
// softmax normaliser summed in double-float. A pop whose best two scores lie within a
// relative 1e-6 sets flags bit 0 (fp32 rounding could have ordered them the other way).
#include <cooperative_groups.h>
#include <limits.h>

#include "draft_tree.cuh"

namespace specv {

constexpr int kTreeThreads = 512;
constexpr int kTreeCluster = 8;  // CTAs per sequence, each on an eighth of the vocabulary
constexpr int kTreeMaxK = 16;
constexpr int kTreeCand = 2048;  // candidate buffer of a row scan (shared memory)
constexpr double kTreeTieRel = 1e-6;

// Per-sequence state: a header, then node scores and depths [N], then the candidate
// arrays [N * kTreeMaxK] (scores; parents; tokens). A candidate score < 0 marks a slot
// already popped (scores are probabilities products: >= 0).
struct TreeHeader {
  int n_nodes, n_cand, cur, flags;
};
struct TreeLayout {
  size_t score, depth, cscore, cparent, ctoken, per_seq;
  __host__ __device__ static TreeLayout make(int max_nodes) {
    TreeLayout l;
    const size_t C = (size_t)max_nodes * kTreeMaxK;
    size_t off = align_up(sizeof(TreeHeader), 16);
    l.score = off;   off = align_up(off + sizeof(double) * max_nodes, 16);
    l.depth = off;   off = align_up(off + sizeof(int) * max_nodes, 16);
    l.cscore = off;  off = align_up(off + sizeof(double) * C, 16);
    l.cparent = off; off = align_up(off + sizeof(int) * C, 16);
    l.ctoken = off;  off = align_up(off + sizeof(int) * C, 16);
    l.per_seq = align_up(off, 256);
    return l;
  }
};

size_t tree_state_bytes(int batch, int max_nodes) { return (size_t)batch * TreeLayout::make(max_nodes).per_seq; }

__global__ void tree_init_kernel(const int32_t* __restrict__ root_tokens, int batch, TreeArgs a) {
  const int b = blockIdx.x;
  const TreeLayout l = TreeLayout::make(a.max_nodes);
  uint8_t* st = a.state + (size_t)b * l.per_seq;
  pdl_wait();
  for (int i = threadIdx.x; i < a.max_nodes; i += blockDim.x) {
    a.parent_out[(size_t)b * a.max_nodes + i] = -1;
    a.tokens_out[(size_t)b * a.max_nodes + i] = i == 0 ? __ldg(root_tokens + b) : -1;
  }
  if (threadIdx.x == 0) {
    TreeHeader* h = reinterpret_cast<TreeHeader*>(st);
    h->n_nodes = 1;
    h->n_cand = 0;
    h->cur = a.max_nodes > 1 ? 0 : -1;  // the root awaits its expansion
    h->flags = 0;
    reinterpret_cast<double*>(st + l.score)[0] = 1.0;
    reinterpret_cast<int*>(st + l.depth)[0] = 0;
    a.n_nodes_out[b] = 1;
    a.next_node[b] = h->cur;
    if (a.flags != nullptr) a.flags[b] = 0;
  }
}

// (value, index) order of the top-k: larger value first, then the lower token id.
__device__ __forceinline__ bool tk_better(float v, int i, float v2, int i2) { return v > v2 || (v == v2 && i < i2); }

// Candidate score as an integer key: the bits of a non-negative double order like the
// value, so the pops compare integers (a dependent fp64 operation costs hundreds of cycles
// here). Popped slots hold -1.0, a negative key.
__device__ __forceinline__ long long score_key(double s) { return __double_as_longlong(s); }
__device__ __forceinline__ bool key_better(long long s, int i, long long s2, int i2) {
  return s > s2 || (s == s2 && i < i2);
}

template <int KMAX, bool kVec>
__global__ void __cluster_dims__(kTreeCluster, 1, 1) __launch_bounds__(kTreeThreads, 1)
    tree_expand_kernel(const float* __restrict__ logits, int vocab, long row_stride, long node_stride, TreeArgs a) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int b = blockIdx.y;
  const int rank = (int)cl.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kTreeThreads / 32;
  const TreeLayout l = TreeLayout::make(a.max_nodes);
  uint8_t* st = a.state + (size_t)b * l.per_seq;
  TreeHeader* h = reinterpret_cast<TreeHeader*>(st);
  double* score = reinterpret_cast<double*>(st + l.score);
  int* depth = reinterpret_cast<int*>(st + l.depth);
  double* cscore = reinterpret_cast<double*>(st + l.cscore);
  int* cparent = reinterpret_cast<int*>(st + l.cparent);
  int* ctoken = reinterpret_cast<int*>(st + l.ctoken);
  __shared__ float s_m[kWarps], s_th[kWarps], s_hi[kWarps], s_lo[kWarps];
  __shared__ float s_cv[kTreeCand];  // the row's elements >= theta (the top-k is among them)
  __shared__ int s_ci[kTreeCand];
  __shared__ int s_cnt;
  __shared__ float s_wv[kWarps];
  __shared__ int s_wi[kWarps];
  __shared__ float s_topv[KMAX];
  __shared__ int s_topi[KMAX];
  __shared__ long long s_k1[kWarps], s_k2[kWarps];
  __shared__ int s_i1[kWarps];
  __shared__ double s_inv_z;
  __shared__ int s_u, s_stop;
  __shared__ float s_gv[KMAX];                 // rank 0: the merged top-k
  __shared__ int s_gi[KMAX];
  __shared__ float s_allv[kTreeCluster * KMAX];  // rank 0: every slice's list, pushed to it
  __shared__ int s_alli[kTreeCluster * KMAX];
  __shared__ float s_allz[2 * kTreeCluster];
  __shared__ float s_allM[kTreeCluster], s_allT[kTreeCluster];  // every slice's max, threshold
  pdl_wait();  // the logits row (the draft model) and the state (the previous call)
  if (threadIdx.x == 0) s_u = h->cur;
  __syncthreads();
  const int u = s_u;
  if (u < 0) return;  // this sequence's tree is complete (the same answer in every rank)
  // every rank of the cluster is running before any writes into another's shared memory:
  // arrive now, wait just before the first such write (after pass 1)
  cl.barrier_arrive();
  const int k = a.topk;
  // this CTA's slice of the row: tokens [c_lo, c_lo + n_sl) (a multiple of 4 long, but the last)
  const int per = ((vocab + kTreeCluster - 1) / kTreeCluster + 3) & ~3;
  const int c_lo = rank * per;
  const int n_sl = max(0, min(vocab, c_lo + per) - c_lo);
  const float* row = logits + (long)b * row_stride + (long)u * node_stride + c_lo;

  // Every element of the row goes through `visit(x, t)`, eight loads per thread in flight.
  constexpr int kU = 8;
  auto scan_row = [&](auto&& visit, bool stream) {
    if (kVec) {
      const float4* r4 = reinterpret_cast<const float4*>(row);
      const int n4 = n_sl >> 2;
      for (int i0 = threadIdx.x; i0 < n4; i0 += kU * kTreeThreads) {
        float4 xv[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
          const int i4 = i0 + q * kTreeThreads;
          xv[q] = i4 < n4 ? (stream ? __ldcs(r4 + i4) : __ldg(r4 + i4)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
          const int i4 = i0 + q * kTreeThreads;
          if (i4 < n4) {
            visit(xv[q].x, c_lo + 4 * i4);
            visit(xv[q].y, c_lo + 4 * i4 + 1);
            visit(xv[q].z, c_lo + 4 * i4 + 2);
            visit(xv[q].w, c_lo + 4 * i4 + 3);
          }
        }
      }
    } else {
      for (int i0 = threadIdx.x; i0 < n_sl; i0 += kU * kTreeThreads) {
        float xv[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
          const int t = i0 + q * kTreeThreads;
          xv[q] = t < n_sl ? (stream ? __ldcs(row + t) : __ldg(row + t)) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
          const int t = i0 + q * kTreeThreads;
          if (t < n_sl) visit(xv[q], c_lo + t);
        }
      }
    }
  };

  // ---- pass 1: the row max, and theta: the k-th largest of a warp's 32 lane maxima (so at
  // least k elements are >= theta), the largest such over the warps. The row stays in L2.
  float tmax = -INFINITY;
  scan_row([&](float x, int) { tmax = fmaxf(tmax, x); }, false);
  {
    float mine = tmax, th = -INFINITY, wmax = -INFINITY;
    for (int r = 0; r < k; ++r) {
      float v = mine;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (r == 0) wmax = v;
      th = v;
      const unsigned who = __ballot_sync(0xffffffffu, mine == v);
      if (lane == __ffs(who) - 1) mine = -INFINITY;
    }
    if (lane == 0) {
      s_m[warp] = wmax;
      s_th[warp] = th;
    }
    if (threadIdx.x == 0) s_cnt = 0;
  }
  __syncthreads();
  cl.barrier_wait();
  if (warp == 0) {  // this slice's max and threshold, written into every CTA of the cluster
    float cm = s_m[0], ct = s_th[0];
    for (int w = 1; w < kWarps; ++w) {
      cm = fmaxf(cm, s_m[w]);
      ct = fmaxf(ct, s_th[w]);
    }
    if (lane < kTreeCluster) {
      *cl.map_shared_rank(&s_allM[rank], lane) = cm;
      *cl.map_shared_rank(&s_allT[rank], lane) = ct;
    }
  }
  cl.sync();  // (A) every slice's max and threshold are here
  float M = -INFINITY, theta = -INFINITY;
  for (int r = 0; r < kTreeCluster; ++r) {
    M = fmaxf(M, s_allM[r]);
    theta = fmaxf(theta, s_allT[r]);
  }
  // ---- pass 2: the normaliser sum of exp(x - M) (compensated, no branch) and the elements
  // >= theta into the candidate buffer
  float s = 0.f, comp = 0.f;
  scan_row(
      [&](float x, int t) {
        const float y = expf(x - M) - comp, z = s + y;
        comp = (z - s) - y;
        s = z;
        if (x >= theta) {
          const int at = atomicAdd(&s_cnt, 1);
          if (at < kTreeCand) {
            s_cv[at] = x;
            s_ci[at] = t;
          }
        }
      },
      true);
  const F2 zs = f2_warp_sum(F2{s, -comp});
  if (lane == 0) {
    s_hi[warp] = zs.hi;
    s_lo[warp] = zs.lo;
  }
  __syncthreads();
  // ---- top-k of this slice: k rounds, round r taking the best element strictly after round
  // r-1's winner in the (value, lower id) order. Up to 256 candidates: warp 0 alone, from
  // registers; more (many ties at theta): the whole CTA, from the buffer or, past its
  // capacity, from the slice.
  const int cnt = s_cnt;
  constexpr int kLane = 8;
  if (cnt <= 32 * kLane) {
    if (warp == 0) {
      float cv[kLane];
      int ci[kLane];
#pragma unroll
      for (int q = 0; q < kLane; ++q) {
        const int c = lane + 32 * q;
        cv[q] = c < cnt ? s_cv[c] : -INFINITY;
        ci[q] = c < cnt ? s_ci[c] : INT_MAX;
      }
      float prev_v = INFINITY;
      int prev_i = -1;
      for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int q = 0; q < kLane; ++q)
          if (ci[q] != INT_MAX && tk_better(prev_v, prev_i, cv[q], ci[q]) && tk_better(cv[q], ci[q], bv, bi)) {
            bv = cv[q];
            bi = ci[q];
          }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
          if (tk_better(v2, i2, bv, bi)) {
            bv = v2;
            bi = i2;
          }
        }
        if (lane == 0) {
          s_topv[r] = bv;
          s_topi[r] = bi;
        }
        prev_v = bv;
        prev_i = bi;
      }
    }
  } else {
    float prev_v = INFINITY;
    int prev_i = -1;
    for (int r = 0; r < k; ++r) {
      float bv = -INFINITY;
      int bi = INT_MAX;
      auto offer = [&](float x, int t) {
        if (x >= theta && tk_better(prev_v, prev_i, x, t) && tk_better(x, t, bv, bi)) {
          bv = x;
          bi = t;
        }
      };
      if (cnt <= kTreeCand) {
        for (int c = threadIdx.x; c < cnt; c += kTreeThreads) offer(s_cv[c], s_ci[c]);
      } else {
        scan_row(offer, false);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        if (tk_better(v2, i2, bv, bi)) {
          bv = v2;
          bi = i2;
        }
      }
      if (lane == 0) {
        s_wv[warp] = bv;
        s_wi[warp] = bi;
      }
      __syncthreads();
      bv = s_wv[0];
      bi = s_wi[0];
      for (int w = 1; w < kWarps; ++w)
        if (tk_better(s_wv[w], s_wi[w], bv, bi)) {
          bv = s_wv[w];
          bi = s_wi[w];
        }
      if (threadIdx.x == 0) {
        s_topv[r] = bv;
        s_topi[r] = bi;
      }
      prev_v = bv;
      prev_i = bi;
      __syncthreads();  // (s_wv is rewritten next round)
    }
  }
  __syncthreads();  // (this slice's list and the warps' partial sums are complete)
  if (warp == 0) {  // this slice's list and normaliser partial, written into rank 0
    F2 z{0.f, 0.f};
    for (int w = 0; w < kWarps; ++w) z = f2_add(z, F2{s_hi[w], s_lo[w]});
    for (int j = lane; j < k; j += 32) {
      *cl.map_shared_rank(&s_allv[rank * k + j], 0) = s_topv[j];
      *cl.map_shared_rank(&s_alli[rank * k + j], 0) = s_topi[j];
    }
    if (lane == 0) {
      *cl.map_shared_rank(&s_allz[rank], 0) = z.hi;
      *cl.map_shared_rank(&s_allz[kTreeCluster + rank], 0) = z.lo;
    }
  }
  cl.sync();  // (B) every slice's list and partial are in rank 0; the other CTAs are done
  if (rank != 0) return;
  if (warp == 0) {  // the slices' k best each (up to 8 x 16 entries): k rounds over the warp
    constexpr int kPer = (kTreeCluster * KMAX + 31) / 32;
    float ev[kPer];
    int ei[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = lane + 32 * q;
      ev[q] = e < kTreeCluster * k ? s_allv[e] : -INFINITY;
      ei[q] = e < kTreeCluster * k ? s_alli[e] : INT_MAX;
    }
    float prev_v = INFINITY;
    int prev_i = -1;
    for (int r = 0; r < k; ++r) {
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int q = 0; q < kPer; ++q)
        if (ei[q] != INT_MAX && tk_better(prev_v, prev_i, ev[q], ei[q]) && tk_better(ev[q], ei[q], bv, bi)) {
          bv = ev[q];
          bi = ei[q];
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        if (tk_better(v2, i2, bv, bi)) {
          bv = v2;
          bi = i2;
        }
      }
      if (lane == 0) {
        s_gv[r] = bv;
        s_gi[r] = bi;
      }
      prev_v = bv;
      prev_i = bi;
    }
    if (lane == 0) {
      F2 z{0.f, 0.f};
      for (int r = 0; r < kTreeCluster; ++r) z = f2_add(z, F2{s_allz[r], s_allz[kTreeCluster + r]});
      // 1 / (hi + lo) from an fp32 reciprocal refined once (the probabilities carry fp32 error
      // already; no fp64 division on this path)
      const float rcp = 1.0f / z.hi;
      const float e1 = fmaf(-z.hi, rcp, 1.0f) - z.lo * rcp;  // 1 - (hi + lo) * rcp
      s_inv_z = (double)rcp + (double)(rcp * e1);
    }
  }
  __syncthreads();
  if (warp == 0) {
    // ---- push the k children of u: lane r scores candidate r; a ballot keeps the order
    const int nc0 = h->n_cand;
    double c = 0.0;
    bool keep = false;
    if (lane < k) {
      const int tok = s_gi[lane];
      if (tok != INT_MAX && tok < vocab) {
        c = score[u] * ((double)expf(s_gv[lane] - M) * s_inv_z);
        keep = !(a.threshold > 0.0) || c > a.threshold;
      }
    }
    const unsigned kb = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int at = nc0 + __popc(kb & ((1u << lane) - 1u));
      cscore[at] = c;
      cparent[at] = u;
      ctoken[at] = s_gi[lane];
    }
    if (lane == 0) {
      h->n_cand = nc0 + __popc(kb);
      s_stop = 0;
    }
  }
  __syncthreads();

  // ---- pops: the best candidate becomes the next node, until one needs its expansion
  const int nc = h->n_cand;
  while (true) {
    long long k1 = -1, k2 = -1;
    int i1 = INT_MAX;
    for (int c = threadIdx.x; c < nc; c += kTreeThreads) {
      const long long key = score_key(cscore[c]);
      if (key < 0) continue;  // popped
      if (key_better(key, c, k1, i1)) {
        k2 = k1;
        k1 = key;
        i1 = c;
      } else if (key > k2) {
        k2 = key;
      }
    }
    auto merge = [&](long long ok1, int oi1, long long ok2) {
      if (key_better(ok1, oi1, k1, i1)) {
        k2 = k1 > ok2 ? k1 : ok2;
        k1 = ok1;
        i1 = oi1;
      } else if (ok1 > k2) {
        k2 = ok1;
      }
    };
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      merge(__shfl_xor_sync(0xffffffffu, k1, o), __shfl_xor_sync(0xffffffffu, i1, o),
            __shfl_xor_sync(0xffffffffu, k2, o));
    if (lane == 0) {
      s_k1[warp] = k1;
      s_k2[warp] = k2;
      s_i1[warp] = i1;
    }
    __syncthreads();
    if (warp == 0) {
      k1 = lane < kWarps ? s_k1[lane] : -1;
      k2 = lane < kWarps ? s_k2[lane] : -1;
      i1 = lane < kWarps ? s_i1[lane] : INT_MAX;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        merge(__shfl_xor_sync(0xffffffffu, k1, o), __shfl_xor_sync(0xffffffffu, i1, o),
              __shfl_xor_sync(0xffffffffu, k2, o));
      if (lane == 0) {
        int stop = 1;
        if (i1 != INT_MAX && k1 >= 0) {
          const double b1 = __longlong_as_double(k1);
          if (k2 >= 0) {  // near tie: the gap relative to the best, in fp32 (ample for 1e-6)
            const float f1 = (float)b1, f2 = (float)__longlong_as_double(k2);
            if (f1 - f2 <= (float)kTreeTieRel * f1) h->flags |= 1;
          }
          const int nid = h->n_nodes;
          const int par = cparent[i1];
          cscore[i1] = -1.0;  // popped
          a.parent_out[(size_t)b * a.max_nodes + nid] = par;
          a.tokens_out[(size_t)b * a.max_nodes + nid] = ctoken[i1];
          score[nid] = b1;
          depth[nid] = depth[par] + 1;
          h->n_nodes = nid + 1;
          if (depth[nid] < a.max_depth && nid + 1 < a.max_nodes) {
            h->cur = nid;  // its logits come next
          } else if (nid + 1 < a.max_nodes) {
            stop = 0;  // at the depth limit: the next candidate
          } else {
            h->cur = -1;  // budget met
          }
        } else {
          h->cur = -1;  // no candidate left
        }
        s_stop = stop;
      }
    }
    __syncthreads();
    if (s_stop) break;
  }
  if (threadIdx.x == 0) {
    a.n_nodes_out[b] = h->n_nodes;
    a.next_node[b] = h->cur;
    if (a.flags != nullptr) a.flags[b] = (uint8_t)h->flags;
  }
}

int launch_tree_init(const int32_t* root_tokens, int batch, const TreeArgs& a, cudaStream_t stream) {
  if (launch_pdl(tree_init_kernel, dim3(batch), dim3(128), 0, stream, root_tokens, batch, a) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

int launch_tree_expand(const float* logits, int vocab, long row_stride, long node_stride, int batch,
                       const TreeArgs& a, cudaStream_t stream) {
  const bool vec = (reinterpret_cast<uintptr_t>(logits) & 15) == 0 && vocab % 4 == 0 && row_stride % 4 == 0 &&
                   node_stride % 4 == 0;
  cudaError_t e;
#define SPECV_TREE_LAUNCH(K)                                                                              \
  e = vec ? launch_pdl(tree_expand_kernel<K, true>, dim3(kTreeCluster, batch), dim3(kTreeThreads), 0, stream, \
                       logits, vocab, row_stride, node_stride, a)                                          \
          : launch_pdl(tree_expand_kernel<K, false>, dim3(kTreeCluster, batch), dim3(kTreeThreads), 0, stream, \
                       logits, vocab, row_stride, node_stride, a)
  if (a.topk <= 4)
    SPECV_TREE_LAUNCH(4);
  else if (a.topk <= 10)
    SPECV_TREE_LAUNCH(10);
  else
    SPECV_TREE_LAUNCH(kTreeMaxK);
#undef SPECV_TREE_LAUNCH
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace specv
