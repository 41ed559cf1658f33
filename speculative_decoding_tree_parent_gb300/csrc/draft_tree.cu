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
// the multi-row call's queue goes to shared memory up to this size (with the row scan's ~19 KB
// static shared memory it stays under the default 48 KB dynamic limit)
constexpr size_t kTreeFastSmemMax = 28 * 1024;

// Per-sequence state: a header, then node scores and depths [N], then the candidate
// arrays [N * kTreeMaxK] (scores; parents; tokens; result index), then the expansion
// results of the multi-row call [N * kTreeMaxW][kTreeMaxK] (tokens; probabilities). A
// candidate score < 0 marks a slot already popped (scores are probabilities products: >= 0).
struct TreeHeader {
  int n_nodes, n_cand, cur, flags;
  // multi-row call: the current request list is result entries [req_base, req_base + nreq);
  // n_res entries are assigned; arrive counts the request clusters of the running call
  int nreq, req_base, n_res, arrive;
};
struct TreeLayout {
  size_t score, depth, cscore, cparent, ctoken, cres, rtok, rp, per_seq;
  int n_res_max;
  __host__ __device__ static TreeLayout make(int max_nodes) {
    TreeLayout l;
    const size_t C = (size_t)max_nodes * kTreeMaxK;
    const size_t R = (size_t)max_nodes * kTreeMaxW;
    l.n_res_max = (int)R;
    size_t off = align_up(sizeof(TreeHeader), 16);
    l.score = off;   off = align_up(off + sizeof(double) * max_nodes, 16);
    l.depth = off;   off = align_up(off + sizeof(int) * max_nodes, 16);
    l.cscore = off;  off = align_up(off + sizeof(double) * C, 16);
    l.cparent = off; off = align_up(off + sizeof(int) * C, 16);
    l.ctoken = off;  off = align_up(off + sizeof(int) * C, 16);
    l.cres = off;    off = align_up(off + sizeof(int) * C, 16);
    l.rtok = off;    off = align_up(off + sizeof(int) * R * kTreeMaxK, 16);
    l.rp = off;      off = align_up(off + sizeof(double) * R * kTreeMaxK, 16);
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
    h->nreq = a.max_nodes > 1 ? 1 : 0;  // the multi-row call's first request: the root (entry 0)
    h->req_base = 0;
    h->n_res = 1;
    h->arrive = 0;
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

// The softmax statistics and the top-k tokens of one draft row (row_base: its first logit),
// by the 8 CTAs of the calling cluster, each on an eighth of the vocabulary (the passes and the
// cluster exchange described at the top of this file). Every rank must call it. Returns false
// in ranks 1-7, which are then done with the row; true in rank 0, with out.gv / out.gi the
// row's top-k in shared memory (largest logit first, lower token id on ties; INT_MAX when the
// row has fewer than k tokens), out.M the row max and out.inv_z the normaliser's reciprocal.
struct RowTopk {
  const float* gv;
  const int* gi;
  float M;
  double inv_z;
};

template <int KMAX, bool kVec>
__device__ __forceinline__ bool tree_row_topk(const float* __restrict__ row_base, int vocab, int k, RowTopk& out) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kTreeThreads / 32;
  __shared__ float s_m[kWarps], s_th[kWarps], s_hi[kWarps], s_lo[kWarps];
  __shared__ float s_cv[kTreeCand];  // the row's elements >= theta (the top-k is among them)
  __shared__ int s_ci[kTreeCand];
  __shared__ int s_cnt;
  __shared__ float s_wv[kWarps];
  __shared__ int s_wi[kWarps];
  __shared__ float s_topv[KMAX];
  __shared__ int s_topi[KMAX];
  __shared__ double s_inv_z;
  __shared__ float s_gv[KMAX];                 // rank 0: the merged top-k
  __shared__ int s_gi[KMAX];
  __shared__ float s_allv[kTreeCluster * KMAX];  // rank 0: every slice's list, pushed to it
  __shared__ int s_alli[kTreeCluster * KMAX];
  __shared__ float s_allz[2 * kTreeCluster];
  __shared__ float s_allM[kTreeCluster], s_allT[kTreeCluster];  // every slice's max, threshold
  // every rank of the cluster is running before any writes into another's shared memory:
  // arrive now, wait just before the first such write (after pass 1)
  cl.barrier_arrive();
  // this CTA's slice of the row: tokens [c_lo, c_lo + n_sl) (a multiple of 4 long, but the last)
  const int per = ((vocab + kTreeCluster - 1) / kTreeCluster + 3) & ~3;
  const int c_lo = rank * per;
  const int n_sl = max(0, min(vocab, c_lo + per) - c_lo);
  const float* row = row_base + c_lo;

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
    // each lane's place among the warp's 32 maxima (larger first, ties by lane: all distinct),
    // from 32 independent shuffles; theta is the value in place k - 1 (k <= 16)
    const float mine = tmax;
    int ahead = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float o = __shfl_sync(0xffffffffu, mine, j);
      ahead += (o > mine || (o == mine && j < lane)) ? 1 : 0;
    }
    const float th = __shfl_sync(0xffffffffu, mine, __ffs(__ballot_sync(0xffffffffu, ahead == k - 1)) - 1);
    const float wmax = __shfl_sync(0xffffffffu, mine, __ffs(__ballot_sync(0xffffffffu, ahead == 0)) - 1);
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
  // ---- top-k of this slice. The buffer (up to kTreeCand elements, usually a few dozen): every
  // element counts the elements ahead of it in the (value, lower id) order -- a strict order,
  // the ids being distinct -- and one whose count is below k is the count-th best. More
  // elements than the buffer holds (many ties at theta): k rounds over the slice, round r
  // taking the best element strictly after round r-1's winner.
  const int cnt = s_cnt;
  const int cnt8 = (min(cnt, kTreeCand) + 7) & ~7;
  for (int r = threadIdx.x; r < k; r += kTreeThreads) {  // (slots no element reaches: none)
    s_topv[r] = -INFINITY;
    s_topi[r] = INT_MAX;
  }
  for (int c = cnt + threadIdx.x; c < cnt8; c += kTreeThreads) {  // padding: never ahead of anything
    s_cv[c] = -INFINITY;
    s_ci[c] = INT_MAX;
  }
  __syncthreads();
  if (cnt <= kTreeCand) {
    for (int c = threadIdx.x; c < cnt; c += kTreeThreads) {
      const float v = s_cv[c];
      const int i = s_ci[c];
      int ahead = 0;
      for (int e0 = 0; e0 < cnt8; e0 += 8) {  // eight loads in flight, then eight tests
        float vv[8];
        int ii[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          vv[q] = s_cv[e0 + q];
          ii[q] = s_ci[e0 + q];
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) ahead += tk_better(vv[q], ii[q], v, i) ? 1 : 0;
      }
      if (ahead < k) {
        s_topv[ahead] = v;
        s_topi[ahead] = i;
      }
    }
  } else {
    float prev_v = INFINITY;
    int prev_i = -1;
    for (int r = 0; r < k; ++r) {
      float bv = -INFINITY;
      int bi = INT_MAX;
      scan_row(
          [&](float x, int t) {
            if (x >= theta && tk_better(prev_v, prev_i, x, t) && tk_better(x, t, bv, bi)) {
              bv = x;
              bi = t;
            }
          },
          false);
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
  if (rank != 0) return false;
  // the slices' k best each (up to 8 x 16 entries, ids distinct across slices): ranked as
  // above; entries a short slice left empty (-inf, INT_MAX) tie among themselves, but rank
  // behind every real one and write only what the slots already hold
  if (threadIdx.x < k) {
    s_gv[threadIdx.x] = -INFINITY;
    s_gi[threadIdx.x] = INT_MAX;
  }
  __syncthreads();
  if (threadIdx.x < kTreeCluster * k) {
    const int ne = kTreeCluster * k;
    const float v = s_allv[threadIdx.x];
    const int i = s_alli[threadIdx.x];
    int ahead = 0;
    for (int e0 = 0; e0 < ne; e0 += 8) {  // (ne = 8 k)
      float vv[8];
      int ii[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        vv[q] = s_allv[e0 + q];
        ii[q] = s_alli[e0 + q];
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) ahead += tk_better(vv[q], ii[q], v, i) ? 1 : 0;
    }
    if (ahead < k) {
      s_gv[ahead] = v;
      s_gi[ahead] = i;
    }
  }
  if (warp == 0) {
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
  out.gv = s_gv;
  out.gi = s_gi;
  out.M = M;
  out.inv_z = s_inv_z;
  return true;
}

// The best candidate (largest key, then lowest slot) among the slots c < nc with a
// non-negative key that ok(c) admits, and the second-best key, reduced over the CTA: the
// answer is in every lane of warp 0 (k1 = -1 / i1 = INT_MAX: none). Every thread must call it;
// the caller synchronises before calling it again.
template <class Ok>
__device__ __forceinline__ void cand_best(const double* cscore, int nc, Ok ok, long long& k1, int& i1,
                                          long long& k2) {
  constexpr int kWarps = kTreeThreads / 32;
  __shared__ long long s_k1[kWarps], s_k2[kWarps];
  __shared__ int s_i1[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  k1 = -1;
  k2 = -1;
  i1 = INT_MAX;
  for (int c = threadIdx.x; c < nc; c += kTreeThreads) {
    const long long key = score_key(cscore[c]);
    if (key < 0 || !ok(c)) continue;  // popped, or not admitted
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
  }
}

// Whether a pop's best two scores (their keys) lie within a relative 1e-6, in fp32. Keys 2^36
// or more apart (same sign, non-negative doubles) differ by more than 2^-17 relative, which
// no fp32 rounding brings under 1e-6: those skip the conversions (fp64 pipe, slow here).
__device__ __forceinline__ bool near_tie(long long k1, long long k2) {
  if (k2 < 0 || k1 - k2 >= (1ll << 36)) return false;
  const float f1 = (float)__longlong_as_double(k1), f2 = (float)__longlong_as_double(k2);
  return f1 - f2 <= (float)kTreeTieRel * f1;
}

// Pops the best candidate as node n_nodes (by lane 0 of warp 0, with k1 / i1 / k2 from
// cand_best): writes its parent, token, score and depth and marks the slot popped. Returns the
// new node id, or -1 when no candidate is left. Sets flags bit 0 on a near tie.
__device__ __forceinline__ int pop_node(TreeHeader* h, double* score, int* depth, double* cscore, const int* cparent,
                                        const int* ctoken, const TreeArgs& a, int b, long long k1, int i1, long long k2) {
  if (i1 == INT_MAX || k1 < 0) return -1;
  const double b1 = __longlong_as_double(k1);
  if (near_tie(k1, k2)) h->flags |= 1;  // (the gap relative to the best, in fp32: ample for 1e-6)
  const int nid = h->n_nodes;
  const int par = cparent[i1];
  cscore[i1] = -1.0;  // popped
  a.parent_out[(size_t)b * a.max_nodes + nid] = par;
  a.tokens_out[(size_t)b * a.max_nodes + nid] = ctoken[i1];
  score[nid] = b1;
  depth[nid] = depth[par] + 1;
  h->n_nodes = nid + 1;
  return nid;
}

template <int KMAX, bool kVec>
__global__ void __cluster_dims__(kTreeCluster, 1, 1) __launch_bounds__(kTreeThreads, 1)
    tree_expand_kernel(const float* __restrict__ logits, int vocab, long row_stride, long node_stride, TreeArgs a) {
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TreeLayout l = TreeLayout::make(a.max_nodes);
  uint8_t* st = a.state + (size_t)b * l.per_seq;
  TreeHeader* h = reinterpret_cast<TreeHeader*>(st);
  double* score = reinterpret_cast<double*>(st + l.score);
  int* depth = reinterpret_cast<int*>(st + l.depth);
  double* cscore = reinterpret_cast<double*>(st + l.cscore);
  int* cparent = reinterpret_cast<int*>(st + l.cparent);
  int* ctoken = reinterpret_cast<int*>(st + l.ctoken);
  __shared__ int s_u, s_stop;
  pdl_wait();  // the logits row (the draft model) and the state (the previous call)
  if (threadIdx.x == 0) s_u = h->cur;
  __syncthreads();
  const int u = s_u;
  if (u < 0) return;  // this sequence's tree is complete (the same answer in every rank)
  const int k = a.topk;
  RowTopk rt;
  if (!tree_row_topk<KMAX, kVec>(logits + (long)b * row_stride + (long)u * node_stride, vocab, k, rt)) return;
  const float M = rt.M;
  if (warp == 0) {
    // ---- push the k children of u: lane r scores candidate r; a ballot keeps the order
    const int nc0 = h->n_cand;
    double c = 0.0;
    bool keep = false;
    if (lane < k) {
      const int tok = rt.gi[lane];
      if (tok != INT_MAX && tok < vocab) {
        c = score[u] * ((double)expf(rt.gv[lane] - M) * rt.inv_z);
        keep = !(a.threshold > 0.0) || c > a.threshold;
      }
    }
    const unsigned kb = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int at = nc0 + __popc(kb & ((1u << lane) - 1u));
      cscore[at] = c;
      cparent[at] = u;
      ctoken[at] = rt.gi[lane];
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
    long long k1, k2;
    int i1;
    cand_best(cscore, nc, [](int) { return true; }, k1, i1, k2);
    if (threadIdx.x == 0) {
      int stop = 1;
      const int nid = pop_node(h, score, depth, cscore, cparent, ctoken, a, b, k1, i1, k2);
      if (nid < 0) {
        h->cur = -1;  // no candidate left
      } else if (depth[nid] < a.max_depth && nid + 1 < a.max_nodes) {
        h->cur = nid;  // its logits come next
      } else if (nid + 1 < a.max_nodes) {
        stop = 0;  // at the depth limit: the next candidate
      } else {
        h->cur = -1;  // budget met
      }
      s_stop = stop;
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

// The pops and the next requests of the multi-row call with the tree's queue staged in shared
// memory and walked by one warp: no CTA barrier and no L2 round trip per pop (the CTA-wide form
// in the kernel below pays both, about 1.7 us a pop). Every thread stages the candidates
// (key = score bits, parent, token, result entry), the node depths and this call's result
// entries; warp 0 pops, pushes and selects exactly as the CTA-wide form; every thread writes
// the candidates back. Shared memory: cap * 20 + max_nodes * 4 + width * kTreeMaxK * 12 bytes,
// cap = max_nodes * topk (the most candidates one tree can hold) + 256 slots of padding, so
// that a lane's eight-slot loads never need a bounds test (padding keys are -1: popped).
// The warp's best two (key, slot) pairs from every lane's own best two (keys >= -1, -1 for
// none; slots distinct, INT_MAX for none): the larger key first, the lower slot on equal keys.
// Each step is one redux.sync over 32-bit halves, so no lane waits on a chain of shuffles.
__device__ __forceinline__ void warp_top2(long long& k1, int& i1, long long& k2, int& i2) {
  auto best = [](long long k, int i, long long& km, int& im) {
    const unsigned long long u = (unsigned long long)(k + 1);  // -1 -> 0
    const unsigned hi = __reduce_max_sync(0xffffffffu, (unsigned)(u >> 32));
    const unsigned lo = __reduce_max_sync(0xffffffffu, (unsigned)(u >> 32) == hi ? (unsigned)u : 0u);
    const unsigned long long m = ((unsigned long long)hi << 32) | lo;
    im = (int)__reduce_min_sync(0xffffffffu, u == m ? (unsigned)i : 0xffffffffu);
    km = (long long)m - 1;
  };
  long long m1, m2;
  int j1, j2;
  best(k1, i1, m1, j1);
  const bool won = i1 == j1;  // this lane held the winner: it offers its second
  best(won ? k2 : k1, won ? i2 : i1, m2, j2);
  k1 = m1;
  i1 = j1;
  k2 = m2;
  i2 = j2;
}

constexpr int kTreePad = 256;
struct FastReplay {
  long long* key;
  int *par, *tok, *res, *dep, *rtk;
  double* rpp;
};

__device__ __forceinline__ FastReplay fast_replay_carve(uint8_t* smem, int cap, int max_nodes) {
  FastReplay f;
  f.key = reinterpret_cast<long long*>(smem);
  f.rpp = reinterpret_cast<double*>(smem + (size_t)cap * 8);
  f.par = reinterpret_cast<int*>(smem + (size_t)cap * 8 + (size_t)kTreeMaxW * kTreeMaxK * 8);
  f.tok = f.par + cap;
  f.res = f.tok + cap;
  f.dep = f.res + cap;
  f.rtk = f.dep + max_nodes;
  return f;
}

size_t tree_fast_smem_bytes(int max_nodes, int topk) {
  const size_t cap = (size_t)max_nodes * topk + kTreePad;
  return cap * 20 + (size_t)max_nodes * 4 + (size_t)kTreeMaxW * kTreeMaxK * 12;
}

__device__ __noinline__ void tree_replay_fast(TreeHeader* h, double* score, int* depth, double* cscore, int* cparent,
                                              int* ctoken, int* cres, const int* rtok, const double* rp,
                                              const TreeArgs& a_ref, int b, int base, int nreq, int n_res_max,
                                              int cap) {
  extern __shared__ __align__(16) uint8_t tree_dsmem[];
  const TreeArgs a = a_ref;  // (in registers: the stores below cannot alias it)
  const FastReplay f = fast_replay_carve(tree_dsmem, cap, a.max_nodes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = a.topk;
  const int nc0 = h->n_cand, nn0 = h->n_nodes;
  for (int c = threadIdx.x; c < cap; c += blockDim.x) {  // (slots past the queue: padding)
    const bool in = c < nc0;
    f.key[c] = in ? score_key(cscore[c]) : -1;
    f.par[c] = in ? cparent[c] : 0;
    f.tok[c] = in ? ctoken[c] : -1;
    f.res[c] = in ? cres[c] : -1;
  }
  for (int u = threadIdx.x; u < nn0; u += blockDim.x) f.dep[u] = depth[u];
  for (int i = threadIdx.x; i < nreq * kTreeMaxK; i += blockDim.x) {  // this call's entries (other SMs wrote them)
    f.rtk[i] = __ldcg(rtok + (size_t)base * kTreeMaxK + i);
    f.rpp[i] = __ldcg(rp + (size_t)base * kTreeMaxK + i);
  }
  __shared__ int s_nc;
  __syncthreads();
  if (warp == 0) {
    int nc = nc0, nn = nn0, flags = h->flags, cur = h->cur;
    int node = cur, r = base;
    double node_score = score[cur];
    // Each lane keeps the best two of its own slots (c = lane mod 32): (ck1, ci1) the best
    // alive one, ck2 the second-best key. A pop reduces the 32 over the warp, and the warp
    // rescans the winning lane's slots together (lane j takes the j-th of them): every step
    // has 32 independent loads or shuffles behind it, not a chain of one lane's.
    long long ck1 = -1, ck2 = -1;
    int ci1 = INT_MAX;
    auto offer = [](long long key, int c, long long& k1, int& i1, long long& k2) {
      if (key < 0) return;  // popped (or not admitted)
      if (key_better(key, c, k1, i1)) {
        k2 = k1;
        k1 = key;
        i1 = c;
      } else if (key > k2) {
        k2 = key;
      }
    };
    // the best two of a lane's values (slot of the second too)
    auto offer2 = [](long long key, int c, long long& k1, int& i1, long long& k2, int& i2) {
      if (key < 0) return;
      if (key_better(key, c, k1, i1)) {
        k2 = k1;
        i2 = i1;
        k1 = key;
        i1 = c;
      } else if (key_better(key, c, k2, i2)) {
        k2 = key;
        i2 = c;
      }
    };
    // lane w's slots, scanned by the warp (lane j takes the j-th of them), with their best two;
    // sel: only the slots the selection admits
    auto scan_lane = [&](int w, bool sel, long long& k1, int& i1, long long& k2, int& i2) {
      k1 = -1;
      k2 = -1;
      i1 = INT_MAX;
      i2 = INT_MAX;
      for (int c = w + 32 * lane; c < nc; c += 32 * 32) {
        const long long key = f.key[c];
        const bool ok = !sel || (f.res[c] < 0 && f.dep[f.par[c]] + 1 < a.max_depth);
        offer2(ok ? key : -1, c, k1, i1, k2, i2);
      }
      warp_top2(k1, i1, k2, i2);
    };
    // this lane's own slots, eight loads in flight at a time (no bounds test: the slots past
    // the queue hold padding keys)
    auto scan_own = [&](bool sel, long long& k1, int& i1, long long& k2) {
      k1 = -1;
      k2 = -1;
      i1 = INT_MAX;
      for (int c0 = lane; c0 < nc; c0 += 32 * 8) {
        long long kk[8];
        int rs[8], ps[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          kk[q] = f.key[c0 + 32 * q];
          rs[q] = f.res[c0 + 32 * q];
          ps[q] = f.par[c0 + 32 * q];
        }
        if (sel) {
          int dd[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) dd[q] = f.dep[ps[q]];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (!(rs[q] < 0 && dd[q] + 1 < a.max_depth)) kk[q] = -1;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) offer(kk[q], c0 + 32 * q, k1, i1, k2);
      }
    };
    const bool use_thr = a.threshold > 0.0;
    scan_own(false, ck1, ci1, ck2);
    while (true) {
      // push the children of `node` from result entry r (lane q: child q)
      {
        const bool local = r >= base && r < base + nreq;
        double c = 0.0;
        bool keep = false;
        int tok = -1;
        if (lane < k) {
          const size_t at = (size_t)(local ? r - base : r) * kTreeMaxK + lane;
          tok = local ? f.rtk[at] : __ldcg(rtok + at);
          if (tok >= 0) {
            c = node_score * (local ? f.rpp[at] : __ldcg(rp + at));
            keep = !use_thr || c > a.threshold;
          }
        }
        const unsigned kb = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          const int at = nc + __popc(kb & ((1u << lane) - 1u));
          f.key[at] = score_key(c);
          f.par[at] = node;
          f.tok[at] = tok;
          f.res[at] = -1;
        }
        __syncwarp();
        const int nc_new = nc + __popc(kb);
        for (int c2 = nc + ((lane - nc) & 31); c2 < nc_new; c2 += 32) offer(f.key[c2], c2, ck1, ci1, ck2);
        nc = nc_new;
      }
      int stop = 2;
      while (stop == 2) {  // pops until one needs a row (1) or has its result (0)
        long long k1 = ck1, k2 = ck2;
        int i1 = ci1, i2 = INT_MAX;  // (i2: the runner-up's slot, unused: ck2 is a key alone)
        warp_top2(k1, i1, k2, i2);
        if (i1 == INT_MAX || k1 < 0) {
          cur = -1;  // no candidate left
          stop = 1;
          break;
        }
        const double b1 = __longlong_as_double(k1);
        if (near_tie(k1, k2)) flags |= 1;
        const int nid = nn, par = f.par[i1], tk = f.tok[i1], rr = f.res[i1];
        const int d = f.dep[par] + 1;
        __syncwarp();
        if (lane == 0) {
          f.key[i1] = -1;  // popped
          f.dep[nid] = d;
          a.parent_out[(size_t)b * a.max_nodes + nid] = par;
          a.tokens_out[(size_t)b * a.max_nodes + nid] = tk;
          score[nid] = b1;
          depth[nid] = d;
        }
        __syncwarp();
        {  // the winner's lane, rescanned
          const int w = i1 & 31;
          long long n1, n2;
          int ni, ni2;
          scan_lane(w, false, n1, ni, n2, ni2);
          if (lane == w) {
            ck1 = n1;
            ci1 = ni;
            ck2 = n2;
          }
        }
        nn = nid + 1;
        if (d < a.max_depth && nid + 1 < a.max_nodes) {
          if (rr >= 0) {  // its row came with an earlier request: expand it now
            node = nid;
            node_score = b1;
            r = rr;
            stop = 0;
          } else {
            cur = nid;  // its row is the next call's first request
            stop = 1;
          }
        } else if (nid + 1 >= a.max_nodes) {
          cur = -1;  // budget met
          stop = 1;
        }  // else: at the depth limit, the next candidate
      }
      if (stop == 1) break;
    }
    // the next requests: per-lane caches of the best admitted slot, reduced per round
    int nr = 0;
    const int n_res = h->n_res;
    if (cur >= 0) {
      const int room = min(a.width, n_res_max - n_res);
      if (room <= 0) {
        if (lane == 0) report(a.status, SPEC_ERR_CAPACITY);
        cur = -1;
      } else {
        if (lane == 0) {
          a.req_parent[(size_t)b * a.width] = a.parent_out[(size_t)b * a.max_nodes + cur];
          a.req_token[(size_t)b * a.width] = a.tokens_out[(size_t)b * a.max_nodes + cur];
        }
        nr = 1;
        // Each lane keeps its best two admitted slots with their indices; a round reduces the
        // bests, the winning lane promotes its second, and only a lane that wins without a
        // known second rescans (with the warp).
        long long sk1 = -1, sk2 = -1;
        int si1 = INT_MAX, si2 = INT_MAX;
        bool sec = true;  // (sk2, si2) is this lane's true second
        if (room > 1) {
          for (int c0 = lane; c0 < nc; c0 += 32 * 8) {
            long long kk[8];
            int rs[8], ps[8], dd[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              kk[q] = f.key[c0 + 32 * q];
              rs[q] = f.res[c0 + 32 * q];
              ps[q] = f.par[c0 + 32 * q];
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) dd[q] = f.dep[ps[q]];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              offer2(rs[q] < 0 && dd[q] + 1 < a.max_depth ? kk[q] : -1, c0 + 32 * q, sk1, si1, sk2, si2);
          }
        }
        for (int q = 1; q < room; ++q) {
          long long k1 = sk1, k2 = sk2;
          int i1 = si1, i2 = si2;
          warp_top2(k1, i1, k2, i2);
          if (i1 == INT_MAX || k1 < 0) break;
          __syncwarp();
          if (lane == 0) {
            f.res[i1] = n_res + q;
            a.req_parent[(size_t)b * a.width + q] = f.par[i1];
            a.req_token[(size_t)b * a.width + q] = f.tok[i1];
          }
          __syncwarp();
          nr = q + 1;
          const int w = i1 & 31;
          const bool resc = __shfl_sync(0xffffffffu, sec ? 0 : 1, w) != 0;
          if (lane == w && !resc) {  // promote the known second
            sk1 = sk2;
            si1 = si2;
            sk2 = -1;
            si2 = INT_MAX;
            sec = false;
          }
          if (resc && q + 1 < room) {  // lane w's slots, by the warp: its best two
            long long n1, n2;
            int ni1, ni2;
            scan_lane(w, true, n1, ni1, n2, ni2);
            if (lane == w) {
              sk1 = n1;
              si1 = ni1;
              sk2 = n2;
              si2 = ni2;
              sec = true;
            }
          }
        }
      }
    }
    if (lane == 0) {
      for (int q = nr; q < a.width; ++q) {
        a.req_parent[(size_t)b * a.width + q] = -1;
        a.req_token[(size_t)b * a.width + q] = -1;
      }
      h->n_nodes = nn;
      h->n_cand = nc;
      h->cur = cur;
      h->flags = flags;
      h->nreq = nr;
      if (nr > 0) {
        h->req_base = n_res;
        h->n_res = n_res + nr;
      }
      a.req_n[b] = nr;
      a.n_nodes_out[b] = nn;
      a.next_node[b] = cur;
      if (a.flags != nullptr) a.flags[b] = (uint8_t)flags;
      s_nc = nc;
    }
  }
  __syncthreads();
  const int nc = s_nc;
  for (int c = threadIdx.x; c < nc; c += blockDim.x) {  // the queue back to the state
    const long long key = f.key[c];
    cscore[c] = key < 0 ? -1.0 : __longlong_as_double(key);
    cparent[c] = f.par[c];
    ctoken[c] = f.tok[c];
    cres[c] = f.res[c];
  }
}

// ------------------------------------------------------------------ the multi-row call
// Exact batching of the construction above. A queued candidate's expansion (its draft row's
// top-k tokens and probabilities) depends on the candidate alone -- its parent and token --
// not on when it leaves the queue. So one call takes the rows of the node awaiting its
// expansion and of up to width - 1 of the best queued candidates (the requests the previous
// call listed), keeps each row's result with its candidate, and then pops exactly as the
// one-row call would: a popped node whose result is at hand has its children pushed at once
// and the pops go on; the first popped node that needs a row it has not got ends the call.
// The tree is the one-row call's, node for node; only the number of calls falls.
//
// Grid: one 8-CTA cluster per (request slot, sequence), width slots. A cluster with a request
// reduces its row (as above) and rank 0 stores the result in the state's entry for that
// request; every cluster's rank 0 then counts itself in with one acq_rel atomic (a cluster
// without a request only after all its ranks have read the header), and the one that counts
// in last runs the pops and lists the next requests. So the header is rewritten only after
// every CTA has read it, and nothing waits: the other clusters are done when they count in.
template <int KMAX, bool kVec>
__global__ void __cluster_dims__(kTreeCluster, 1, 1) __launch_bounds__(kTreeThreads, 1)
    tree_expand_multi_kernel(const float* __restrict__ logits, int vocab, long row_stride, long req_stride,
                             TreeArgs a, int fast_cap) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int j = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TreeLayout l = TreeLayout::make(a.max_nodes);
  uint8_t* st = a.state + (size_t)b * l.per_seq;
  TreeHeader* h = reinterpret_cast<TreeHeader*>(st);
  double* score = reinterpret_cast<double*>(st + l.score);
  int* depth = reinterpret_cast<int*>(st + l.depth);
  double* cscore = reinterpret_cast<double*>(st + l.cscore);
  int* cparent = reinterpret_cast<int*>(st + l.cparent);
  int* ctoken = reinterpret_cast<int*>(st + l.ctoken);
  int* cres = reinterpret_cast<int*>(st + l.cres);
  int* rtok = reinterpret_cast<int*>(st + l.rtok);
  double* rp = reinterpret_cast<double*>(st + l.rp);
  __shared__ int s_nreq, s_base, s_last, s_stop, s_node, s_res, s_nr;
  pdl_wait();  // the rows (the draft model) and the state (the previous call)
  if (threadIdx.x == 0) {
    s_nreq = h->nreq;
    s_base = h->req_base;
  }
  __syncthreads();
  const int nreq = s_nreq;
  if (nreq == 0) return;  // the tree is complete: no CTA counts in, nothing changes
  if (nreq > (int)gridDim.y) {  // listed by a call of a larger width: refused, nothing changes
    if (j == 0 && cl.block_rank() == 0 && threadIdx.x == 0) report(a.status, SPEC_ERR_ARG);
    return;
  }
  const int k = a.topk;
  if (j < nreq) {
    RowTopk rt;
    if (!tree_row_topk<KMAX, kVec>(logits + (long)b * row_stride + (long)j * req_stride, vocab, k, rt)) return;
    // rank 0: the row's result into entry req_base + j
    const int e = s_base + j;
    if (warp == 0 && lane < k) {
      const int tok = rt.gi[lane];
      const bool ok = tok != INT_MAX && tok < vocab;
      rtok[(size_t)e * kTreeMaxK + lane] = ok ? tok : -1;
      rp[(size_t)e * kTreeMaxK + lane] = ok ? (double)expf(rt.gv[lane] - rt.M) * rt.inv_z : 0.0;
    }
    __syncthreads();  // the entry is written before thread 0's release
  } else {
    cl.sync();  // every rank has read the header before rank 0 counts in
    if (cl.block_rank() != 0) return;
  }
  if (threadIdx.x == 0) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(old) : "l"(&h->arrive) : "memory");
    s_last = old == (int)gridDim.y - 1;
    if (s_last) h->arrive = 0;  // every slot has counted in: ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  if (fast_cap > 0) {  // the queue fits in shared memory: one warp pops
    tree_replay_fast(h, score, depth, cscore, cparent, ctoken, cres, rtok, rp, a, b, s_base, nreq, l.n_res_max,
                     fast_cap);
    return;
  }

  // ---- the last cluster: expand the awaiting node from entry req_base, then pop
  // (the other clusters' entries are read from L2: they were written on other SMs)
  auto push_children = [&](int u, int r) {  // warp 0: the children of node u from entry r
    const int nc0 = h->n_cand;
    double c = 0.0;
    bool keep = false;
    int tok = -1;
    if (lane < k) {
      tok = __ldcg(rtok + (size_t)r * kTreeMaxK + lane);
      if (tok >= 0) {
        c = score[u] * __ldcg(rp + (size_t)r * kTreeMaxK + lane);
        keep = !(a.threshold > 0.0) || c > a.threshold;
      }
    }
    const unsigned kb = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int at = nc0 + __popc(kb & ((1u << lane) - 1u));
      cscore[at] = c;
      cparent[at] = u;
      ctoken[at] = tok;
      cres[at] = -1;  // no row yet
    }
    if (lane == 0) h->n_cand = nc0 + __popc(kb);
  };
  if (threadIdx.x == 0) {
    s_node = h->cur;
    s_res = s_base;
  }
  __syncthreads();
  while (true) {
    if (warp == 0) push_children(s_node, s_res);
    __syncthreads();
    const int nc = h->n_cand;
    int stop;
    while (true) {  // pops until one needs a row (stop 1) or has its result (stop 0)
      long long k1, k2;
      int i1;
      cand_best(cscore, nc, [](int) { return true; }, k1, i1, k2);
      if (threadIdx.x == 0) {
        int sp = 1;
        const int r = i1 != INT_MAX ? cres[i1] : -1;
        const int nid = pop_node(h, score, depth, cscore, cparent, ctoken, a, b, k1, i1, k2);
        if (nid < 0) {
          h->cur = -1;  // no candidate left
        } else if (depth[nid] < a.max_depth && nid + 1 < a.max_nodes) {
          if (r >= 0) {  // its row came with an earlier request: expand it now
            s_node = nid;
            s_res = r;
            sp = 0;
          } else {
            h->cur = nid;  // its row is the next call's first request
          }
        } else if (nid + 1 < a.max_nodes) {
          sp = 2;  // at the depth limit: the next candidate
        } else {
          h->cur = -1;  // budget met
        }
        s_stop = sp;
      }
      __syncthreads();
      stop = s_stop;
      if (stop != 2) break;
    }
    if (stop == 1) break;
  }

  // ---- the next requests: the awaiting node, then the best queued candidates that have no
  // row yet and would be expanded (below the depth limit), best first
  const int cur = h->cur;
  const int nc = h->n_cand;
  if (threadIdx.x == 0) s_nr = 0;
  if (cur >= 0) {
    const int n_res = h->n_res;
    // Entries suffice: a call with requests consumes one awaiting node and the next awaiting
    // node is a new node, so at most max_nodes - 1 such calls follow the root's, each taking
    // at most width <= kTreeMaxW entries. Checked all the same: short, it reports and stops.
    const int room = min(a.width, l.n_res_max - n_res);
    if (threadIdx.x == 0 && room <= 0) {
      report(a.status, SPEC_ERR_CAPACITY);
      h->cur = -1;
    }
    if (threadIdx.x == 0 && room > 0) {
      a.req_parent[(size_t)b * a.width] = a.parent_out[(size_t)b * a.max_nodes + cur];
      a.req_token[(size_t)b * a.width] = a.tokens_out[(size_t)b * a.max_nodes + cur];
      s_nr = 1;
    }
    __syncthreads();
    for (int q = 1; q < room; ++q) {
      long long k1, k2;
      int i1;
      cand_best(
          cscore, nc, [&](int c) { return cres[c] < 0 && depth[cparent[c]] + 1 < a.max_depth; }, k1, i1, k2);
      if (threadIdx.x == 0) {
        if (i1 != INT_MAX && k1 >= 0) {
          cres[i1] = n_res + q;
          a.req_parent[(size_t)b * a.width + q] = cparent[i1];
          a.req_token[(size_t)b * a.width + q] = ctoken[i1];
          s_nr = q + 1;
        }
      }
      __syncthreads();
      if (s_nr != q + 1) break;
    }
    if (threadIdx.x == 0) {
      h->req_base = n_res;
      h->n_res = n_res + s_nr;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    h->nreq = s_nr;
    for (int q = s_nr; q < a.width; ++q) {
      a.req_parent[(size_t)b * a.width + q] = -1;
      a.req_token[(size_t)b * a.width + q] = -1;
    }
    a.req_n[b] = s_nr;
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

int launch_tree_expand_multi(const float* logits, int vocab, long row_stride, long req_stride, int batch,
                             const TreeArgs& a, cudaStream_t stream) {
  const bool vec = (reinterpret_cast<uintptr_t>(logits) & 15) == 0 && vocab % 4 == 0 && row_stride % 4 == 0 &&
                   req_stride % 4 == 0;
  const dim3 grid(kTreeCluster, a.width, batch);
  // the queue in shared memory when it fits beside the row scan's own (no raised limit needed)
  const size_t fsm = tree_fast_smem_bytes(a.max_nodes, a.topk);
  const bool fast = fsm <= kTreeFastSmemMax;
  const size_t dsm = fast ? fsm : 0;
  const int cap = fast ? a.max_nodes * a.topk + kTreePad : 0;
  cudaError_t e;
#define SPECV_TREE_LAUNCH(K)                                                                                 \
  e = vec ? launch_pdl(tree_expand_multi_kernel<K, true>, grid, dim3(kTreeThreads), dsm, stream, logits, vocab,  \
                       row_stride, req_stride, a, cap)                                                       \
          : launch_pdl(tree_expand_multi_kernel<K, false>, grid, dim3(kTreeThreads), dsm, stream, logits, vocab, \
                       row_stride, req_stride, a, cap)
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
