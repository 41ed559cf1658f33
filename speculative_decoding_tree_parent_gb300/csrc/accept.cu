// K-ACCEPT: longest accepted path of every draft tree + the bonus token.
//
// Greedy ("EAGLE-2 deep dive", architecture section: the target's logits are
// contrasted with the draft tokens and the longest accepted path is fixed;
// "Accelerating Sonar through speculation", speculative-decoding section: n
// drafts give up to n+1 tokens, the extra one from the target's logits where
// the walk stops). Stochastic ("EAGLE-2 deep dive", benchmark section:
// rejection sampling on the target distribution; "Accelerating Sonar",
// draft-target section: full draft and target distributions are compared),
// with the rule of the speculative-sampling works those pages cite applied to
// the children of a node one after another.
//
// Greedy, one launch:
//   accept_greedy_kernel   one wave of CTAs streams every logits row in 4096-logit
//                          tasks (16-byte loads, the next task's loads in flight while
//                          the current one is reduced); each task folds its (max, first
//                          index) into its row's slot with one 64-bit atomicMax. The
//                          last CTA to finish (atomic counter, no waiting) reads every
//                          row's argmax from the slots and walks every sequence, one
//                          warp each.
// Stochastic, one launch:
//   accept_walk_kernel     one 8-CTA cluster per sequence, each CTA on an eighth of the
//                          vocabulary. At each node the walk visits (the root, then each
//                          accepted child) it loads the node's target and draft rows, takes
//                          their max and sum of exp((x - max) / T) (fp32 elements, Kahan per
//                          thread, double-float across threads, warps and the CTAs of the
//                          cluster, exchanged through distributed shared memory) and keeps p
//                          and q of its slice in shared memory; the children's tests and the
//                          residual passes then read those. Only the visited nodes' rows are
//                          read: the method needs no other node's distributions. Every CTA of
//                          the cluster takes the same decisions from bitwise-identical sums.
//
// Residual in closed form. Starting from r_1 = p, the update
// r <- max(r - q, 0) / sum(max(r - q, 0)) keeps r of the form
// max(p - c q, 0) / s with scalars c and s:  c_1 = 0, s_1 = 1, and after a
// rejection c' = c + s, s' = sum_t max(p(t) - c' q(t), 0) (if s' = 0, r is kept).
// The test of a child with token x is then u < max(p(x) - c q(x), 0) / (s q(x)).
// Only the scalar pair (c, s) travels between passes; each rejection costs one
// pass over the vocabulary and the bonus draw one more (an inverse-CDF search).
#include <cooperative_groups.h>
#include <float.h>
#include <limits.h>

#include <mutex>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace specv {

constexpr int kAcceptThreads = 256;
constexpr int kWalkThreads = 512;
constexpr int kWalkCluster = 8;
constexpr double kTieEps = 1e-6;    // ratio test near-tie band (absolute)
constexpr double kBonusEps = 1e-8;  // bonus draw near-tie band (relative to the residual's total)

struct alignas(8) ArgPartial {
  float v;
  int i;
};
struct NodeStats {  // a row's max and the reciprocal of its softmax normaliser (fp32)
  float m_p, m_q;
  float inv_zp, inv_zq;
};

// Workspace layout for spec_accept (offsets in bytes, each 256-aligned). The greedy
// kernel's counter (finished CTAs) and its per-row argmax slots sit in a fixed area at
// the start, the same for every size and mode, that holds nothing else; every call leaves
// them at zero, so no size change can hand them stale partial data.
constexpr int kArgSlots = 8192;  // rows whose argmax is folded in a slot (more: task partials)
struct AcceptWs {
  size_t counter, slots, partials, results, total;
  static AcceptWs make(int batch, int total_nodes, int chunks) {
    (void)batch;
    AcceptWs w;
    size_t off = 0;
    w.counter = off;  off = align_up(off + sizeof(unsigned), 256);
    w.slots = off;    off = align_up(off + sizeof(unsigned long long) * kArgSlots, 256);
    w.partials = off; off = align_up(off + sizeof(ArgPartial) * (size_t)total_nodes * chunks, 256);
    w.results = off;  off = align_up(off + sizeof(int) * (size_t)total_nodes, 256);
    w.total = off;
    return w;
  }
};

constexpr int kGreedyVec = 4;                                  // float4 per thread per task
constexpr int kGreedyChunk = kAcceptThreads * kGreedyVec * 4;  // 4096 logits
int greedy_chunks(int vocab) { return ceil_div(vocab, kGreedyChunk); }

// the greedy per-task partials (past kArgSlots rows): one per 4096-logit piece of a row
int accept_chunks(int total_nodes, int vocab) {
  (void)total_nodes;
  return greedy_chunks(vocab);
}

size_t accept_ws_bytes(int batch, int total_nodes, int vocab) {
  return AcceptWs::make(batch, total_nodes, accept_chunks(total_nodes, vocab)).total;
}

__device__ __forceinline__ void arg_better(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// (value, index) as one 64-bit key whose unsigned order is the argmax order: larger
// value first, then the lower index (the index is stored complemented). Every real key
// is > 0, so 0 marks an empty slot. -0.0 is keyed as +0.0: the two compare equal, so a
// row whose maximum is zero takes the lowest index holding either (the order bits alone
// would put -0.0 below +0.0 and let a later task's +0.0 win).
__device__ __forceinline__ unsigned long long arg_key(float v, int i) {
  unsigned u = __float_as_uint(v == 0.f ? 0.f : v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned)(~i);
}
__device__ __forceinline__ int arg_key_index(unsigned long long key) { return (int)~(unsigned)key; }

__device__ __forceinline__ void warp_arg_reduce(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    arg_better(v, i, v2, i2);
  }
}

// Greedy walk of one sequence by one warp: from the root, move to the first child
// (lowest id) whose draft token equals the node's target argmax. The three arrays hold
// the sequence's nodes 0..n-1 (staged in shared memory by the caller).
__device__ void greedy_walk_warp(int b, int n, const int* parent, const int* tokens, const int* argmax,
                                 int path_cap, int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                                 uint8_t* flags, int32_t* status) {
  const int lane = threadIdx.x & 31;
  int v = 0, L = 0, bonus = 0;
  int32_t* prow = path + (size_t)b * path_cap;
  int32_t* trow = out_tokens + (size_t)b * path_cap;
  if (lane == 0) prow[0] = 0;
  while (true) {
    const int a = argmax[v];
    int found = -1;
    for (int c0 = v + 1; c0 < n; c0 += 32) {
      const int c = c0 + lane;
      const bool m = c < n && parent[c] == v && tokens[c] == a;
      const unsigned bal = __ballot_sync(0xffffffffu, m);
      if (bal) {
        found = c0 + __ffs(bal) - 1;
        break;
      }
    }
    if (found < 0) {
      bonus = a;
      break;
    }
    if (L + 1 >= path_cap) {  // accepted path does not fit: truncate here
      if (lane == 0) report(status, SPEC_ERR_CAPACITY);
      bonus = a;
      break;
    }
    ++L;
    if (lane == 0) {
      prow[L] = found;
      trow[L - 1] = tokens[found];
    }
    v = found;
  }
  if (lane == 0) {
    trow[L] = bonus;
    accept_len[b] = L;
    if (flags != nullptr) flags[b] = 0;
  }
  for (int k = L + 1 + lane; k < path_cap; k += 32) {
    prow[k] = -1;
    trow[k] = -1;
  }
}

// Greedy argmax + walk, one launch. A task is one chunk of kGreedyChunk logits of one
// row; the grid is one wave of CTAs (as many as fit on the SMs at once) and CTA i takes
// tasks i, i + grid, ... with the loads of its next task issued before the current one
// is reduced, so every SM keeps two tasks of loads in flight until the stream ends. A
// task folds its (max, first index) into its row's slot (64-bit atomicMax on an
// order-preserving key; beyond kArgSlots rows it leaves a partial instead). The last CTA
// to finish (one counter, no waiting) reads every row's argmax (or merges the partials)
// and walks every sequence, one warp per sequence, on the tree staged in shared memory.
constexpr int kGreedyStage = 2048;  // nodes the final CTA stages
constexpr int kCommitCta = 4;          // fused commit: up to this many sequences, one at a time by the CTA
constexpr int kCommitPathStage = 128;  // path rows up to this long kept in shared memory for it


// The same walk on a tree staged in shared memory, in two steps: every node c > 0 whose
// draft token equals its parent's argmax offers itself to the parent (atomicMin keeps the
// lowest id), then the warp follows the offers from the root. `child` is scratch of n
// entries.
// `spath` (nullable) receives a shared-memory copy of the path row's first L + 1
// entries (room for path_cap). Returns L on every lane.
__device__ int greedy_walk_warp_staged(int b, int n, const int* parent, const int* tokens, const int* argmax,
                                       int* child, int path_cap, int32_t* accept_len, int32_t* path,
                                       int32_t* out_tokens, uint8_t* flags, int32_t* status, int* spath) {
  const int lane = threadIdx.x & 31;
  for (int c = lane; c < n; c += 32) child[c] = INT_MAX;
  __syncwarp();
  for (int c = 1 + lane; c < n; c += 32) {
    const int v = parent[c];
    if (v >= 0 && v < c && tokens[c] == argmax[v]) atomicMin(child + v, c);
  }
  __syncwarp();
  int32_t* prow = path + (size_t)b * path_cap;
  int32_t* trow = out_tokens + (size_t)b * path_cap;
  if (lane == 0) {
    int v = 0, L = 0;
    prow[0] = 0;
    if (spath != nullptr) spath[0] = 0;
    while (child[v] != INT_MAX) {
      if (L + 1 >= path_cap) {  // accepted path does not fit: truncate here
        report(status, SPEC_ERR_CAPACITY);
        break;
      }
      const int c = child[v];
      ++L;
      prow[L] = c;
      if (spath != nullptr) spath[L] = c;
      trow[L - 1] = tokens[c];
      v = c;
    }
    trow[L] = argmax[v];
    accept_len[b] = L;
    if (flags != nullptr) flags[b] = 0;
    child[0] = L;  // hand L to the lanes through shared memory
  }
  __syncwarp();
  const int L = child[0];
  for (int k = L + 1 + lane; k < path_cap; k += 32) {
    prow[k] = -1;
    trow[k] = -1;
  }
  return L;
}

// Commit of sequence b (the rules of kv_commit_kernel) by a team: the whole CTA
// (kCta) or one warp. L and the path come from this CTA's walk: `spath` in shared
// memory (nullable: then the global row `gpath`, written before a barrier). Every slot
// is validated and the first rows' K/V are loaded before the team's vote, so a valid
// commit costs one memory round trip; a sequence with an error is reported and left
// unwritten.
// Rows `first` .. L are copied (first = 1 when the root row went early, see
// commit_root_early, whose P is then passed as P_pre; P_pre < 0: P is read here).
template <bool kCta, bool kIns>
__device__ void commit_sequence(const CommitArgs& ca, int b, int base, int n, int L, const int* spath,
                                const int32_t* gpath, int path_cap, int32_t* status, int first = 0,
                                int P_pre = -1) {
  const int rank = kCta ? (int)threadIdx.x : (int)(threadIdx.x & 31);
  const int size = kCta ? (int)blockDim.x : 32;
  const int P = P_pre >= 0 ? P_pre : __ldg(ca.prefix_len + b);
  const int32_t* prow_pt = ca.page_table + (size_t)b * ca.max_pages;
  auto node_at = [&](int i) { return spath != nullptr ? spath[i] : gpath[i]; };
  int code = 0;
  if (L < 0 || L >= path_cap || L >= n || P < 0) {
    code = SPEC_ERR_INDEX;
  } else if (kIns && P + L + 1 >= ca.ins.token_stride) {
    code = SPEC_ERR_CAPACITY;  // the token row has no room for L + 1 tokens after P
  } else {
    for (int i = first + rank; i <= L; i += size) {
      const int node = node_at(i);
      const int lp = (P + i) / ca.page_size;
      const int page = lp < ca.max_pages ? __ldg(prow_pt + lp) : -1;
      int c = 0;
      if (node < 0 || node >= n || (i == 0 && node != 0)) c = SPEC_ERR_INDEX;
      else if (lp >= ca.max_pages) c = SPEC_ERR_CAPACITY;
      else if (page < 0 || page >= ca.num_pages) c = SPEC_ERR_PAGE;
      if (code == 0) code = c;
    }
  }
  const int row_bytes = ca.d * ca.elem_bytes;
  const int vecs = row_bytes >> 4;
  const int total = code == 0 && L >= first ? (L + 1 - first) * ca.hkv * vecs : 0;
  // the first rows' loads go out with the checks (a row only if its node is in range)
  constexpr int kPer = 2;
  uint4 kb[kPer], vb[kPer];
  size_t dsts[kPer];
  auto locate = [&](int e, size_t& src, size_t& dst) {
    const int r = e / vecs, vi = e - (e / vecs) * vecs;
    const int i = first + r / ca.hkv, g = r - (r / ca.hkv) * ca.hkv;
    const int slot = P + i;
    const int node = node_at(i);
    const int lp = slot / ca.page_size;
    const int page = lp < ca.max_pages ? __ldg(prow_pt + lp) : -1;  // another slot's check may have failed
    src = ((size_t)(base + node) * ca.hkv + g) * row_bytes + ((size_t)vi << 4);
    dst = (((size_t)page * ca.hkv + g) * ca.page_size + (slot % ca.page_size)) * row_bytes + ((size_t)vi << 4);
    return node >= 0 && node < n && page >= 0 && page < ca.num_pages;
  };
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = rank + u * size;
    size_t src = 0;
    dsts[u] = 0;
    if (e < total && locate(e, src, dsts[u])) {
      kb[u] = __ldg(reinterpret_cast<const uint4*>(ca.k_tree + src));
      vb[u] = __ldg(reinterpret_cast<const uint4*>(ca.v_tree + src));
    }
  }
  const bool bad = kCta ? __syncthreads_or(code != 0) : __any_sync(0xffffffffu, code != 0);
  if (bad) {
    if (code != 0) report(status, code);
    return;
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    if (rank + u * size < total) {
      *reinterpret_cast<uint4*>(ca.k_pool + dsts[u]) = kb[u];
      *reinterpret_cast<uint4*>(ca.v_pool + dsts[u]) = vb[u];
    }
  }
  for (int e = rank + kPer * size; e < total; e += size) {
    size_t src, dst;
    locate(e, src, dst);
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(ca.k_tree + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(ca.v_tree + src));
    *reinterpret_cast<uint4*>(ca.k_pool + dst) = kv;
    *reinterpret_cast<uint4*>(ca.v_pool + dst) = vv;
  }
  if (kIns)  // the accepted tokens and the bonus after the root
    for (int i = rank; i <= L; i += size)
      ca.ins.token_buf[(size_t)b * ca.ins.token_stride + P + 1 + i] = ca.ins.out_tokens[(size_t)b * path_cap + i];
  if (rank == 0 && ca.seq_len_out != nullptr) ca.seq_len_out[b] = P + L + 1;
}

// The same commit in two halves, for the walk from the root (the whole CTA, rows 0 .. L).
// walk_commit_load reads inputs only: the first rows' K/V (their sources need only the
// path, so they load alongside the prefix length), then every slot's page entry, checked;
// two dependent memory round trips in all, and the walk may run it before its
// grid-dependency wait. walk_commit_store votes (a sequence with an error is reported and
// left unwritten) and writes.
constexpr int kCommitPer = 1;  // 16-byte pieces of the rows a thread holds in registers
struct CommitLoad {
  int P, code, total;
  uint4 kb[kCommitPer], vb[kCommitPer];
  size_t dst[kCommitPer];
};

__device__ __forceinline__ void walk_commit_load(const CommitArgs& ca, int b, int base, int n, int L,
                                                 const int* spath, int path_cap, CommitLoad& c) {
  const int rank = threadIdx.x, size = blockDim.x;
  const int row_bytes = ca.d * ca.elem_bytes;
  const int vecs = row_bytes >> 4;
  const bool shape_ok = L >= 0 && L < path_cap && L < n;
  const int total = shape_ok ? (L + 1) * ca.hkv * vecs : 0;
  int slot_i[kCommitPer];
#pragma unroll
  for (int u = 0; u < kCommitPer; ++u) {  // the rows: addressed by the path alone
    const int e = rank + u * size;
    slot_i[u] = -1;
    if (e < total) {
      const int r = e / vecs, vi = e - (e / vecs) * vecs;
      const int i = r / ca.hkv, g = r - (r / ca.hkv) * ca.hkv;
      const int node = spath[i];
      if (node >= 0 && node < n) {
        const size_t src = ((size_t)(base + node) * ca.hkv + g) * row_bytes + ((size_t)vi << 4);
        c.kb[u] = __ldg(reinterpret_cast<const uint4*>(ca.k_tree + src));
        c.vb[u] = __ldg(reinterpret_cast<const uint4*>(ca.v_tree + src));
        slot_i[u] = i;
        c.dst[u] = (size_t)g * ca.page_size * row_bytes + ((size_t)vi << 4);  // + the page and slot below
      }
    }
  }
  const int P = __ldg(ca.prefix_len + b);
  const int32_t* prow_pt = ca.page_table + (size_t)b * ca.max_pages;
  int code = 0;
  if (!shape_ok || P < 0) {
    code = SPEC_ERR_INDEX;
  } else if (ca.ins.token_buf != nullptr && P + L + 1 >= ca.ins.token_stride) {
    code = SPEC_ERR_CAPACITY;  // the token row has no room for L + 1 tokens after P
  } else {
    for (int i = rank; i <= L; i += size) {
      const int node = spath[i];
      const int lp = (P + i) / ca.page_size;
      const int page = lp < ca.max_pages ? __ldg(prow_pt + lp) : -1;
      int cc = 0;
      if (node < 0 || node >= n || (i == 0 && node != 0)) cc = SPEC_ERR_INDEX;
      else if (lp >= ca.max_pages) cc = SPEC_ERR_CAPACITY;
      else if (page < 0 || page >= ca.num_pages) cc = SPEC_ERR_PAGE;
      if (code == 0) code = cc;
    }
  }
#pragma unroll
  for (int u = 0; u < kCommitPer; ++u) {  // each held piece's destination (used once the vote passes)
    if (slot_i[u] >= 0 && code == 0) {
      const int slot = P + slot_i[u];
      const int lp = slot / ca.page_size;
      const int page = lp < ca.max_pages ? __ldg(prow_pt + lp) : 0;
      c.dst[u] += (((size_t)page * ca.hkv) * ca.page_size + (slot % ca.page_size)) * row_bytes;
    }
  }
  c.P = P;
  c.code = code;
  c.total = code == 0 ? total : 0;
}

template <bool kIns>
__device__ __forceinline__ void walk_commit_store(const CommitArgs& ca, int b, int base, int L, const int* spath,
                                                  int path_cap, int32_t* status, const CommitLoad& c) {
  const int rank = threadIdx.x, size = blockDim.x;
  if (__syncthreads_or(c.code != 0)) {
    if (c.code != 0) report(status, c.code);
    return;
  }
  // every slot and node checked above is valid from here on
#pragma unroll
  for (int u = 0; u < kCommitPer; ++u) {
    if (rank + u * size < c.total) {
      *reinterpret_cast<uint4*>(ca.k_pool + c.dst[u]) = c.kb[u];
      *reinterpret_cast<uint4*>(ca.v_pool + c.dst[u]) = c.vb[u];
    }
  }
  const int P = c.P;
  const int row_bytes = ca.d * ca.elem_bytes;
  const int vecs = row_bytes >> 4;
  const int32_t* prow_pt = ca.page_table + (size_t)b * ca.max_pages;
  for (int e = rank + kCommitPer * size; e < c.total; e += size) {  // long paths: the rest
    const int r = e / vecs, vi = e - (e / vecs) * vecs;
    const int i = r / ca.hkv, g = r - (r / ca.hkv) * ca.hkv;
    const int slot = P + i;
    const int page = __ldg(prow_pt + slot / ca.page_size);
    const size_t src = ((size_t)(base + spath[i]) * ca.hkv + g) * row_bytes + ((size_t)vi << 4);
    const size_t dst =
        (((size_t)page * ca.hkv + g) * ca.page_size + (slot % ca.page_size)) * row_bytes + ((size_t)vi << 4);
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(ca.k_tree + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(ca.v_tree + src));
    *reinterpret_cast<uint4*>(ca.k_pool + dst) = kv;
    *reinterpret_cast<uint4*>(ca.v_pool + dst) = vv;
  }
  if (kIns)  // the accepted tokens and the bonus after the root
    for (int i = rank; i <= L; i += size)
      ca.ins.token_buf[(size_t)b * ca.ins.token_stride + P + 1 + i] = ca.ins.out_tokens[(size_t)b * path_cap + i];
  if (rank == 0 && ca.seq_len_out != nullptr) ca.seq_len_out[b] = P + L + 1;
}

// ---- the root row committed while the walk runs (fused greedy commit, few sequences)
// The root (node 0, the last accepted token) always goes to slot P, whatever the walk
// decides; only rows 1 .. L wait for it. One warp of the final CTA stages the root rows
// with asynchronous copies into shared memory the walk leaves unused (root_stage), then,
// while the walk runs, checks every slot the walk could reach (P .. P + path_cap - 1):
// when all lie in valid pages nothing after the walk can fail, so the row is written at
// once and the result is that of committing after the walk (root_write); otherwise the
// commit after the walk copies it (and reports the error).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((unsigned)__cvta_generic_to_shared(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Root K/V rows of the sequence whose node 0 is global row `base` into buf (K, then V).
__device__ void root_stage(const CommitArgs& ca, int base, uint4* buf) {
  const int lane = threadIdx.x & 31;
  const int row_bytes = ca.d * ca.elem_bytes, chunks = ca.hkv * row_bytes / 16;
  const size_t src = (size_t)base * ca.hkv * row_bytes;  // node 0: its heads back to back
  for (int e = lane; e < chunks; e += 32) {
    cp_async16(buf + e, ca.k_tree + src + ((size_t)e << 4));
    cp_async16(buf + chunks + e, ca.v_tree + src + ((size_t)e << 4));
  }
}

// The staged root rows of sequence b to slot P, when every reachable slot's page is valid
// (each lane stores the chunks its own copies staged). Returns P when written, else -1.
template <bool kIns>
__device__ int root_write(const CommitArgs& ca, int b, int P, int n, int path_cap, const uint4* buf) {
  const int lane = threadIdx.x & 31;
  if (P < 0 || n < 1 || path_cap < 1) return -1;
  if (kIns && P + path_cap >= ca.ins.token_stride) return -1;  // token room too
  const int lp0 = P / ca.page_size, lp1 = (P + path_cap - 1) / ca.page_size;
  if (lp1 - lp0 >= 32) return -1;
  int page = -1;
  bool ok = true;
  if (lp0 + lane <= lp1) {
    const int lp = lp0 + lane;
    page = lp < ca.max_pages ? __ldg(ca.page_table + (size_t)b * ca.max_pages + lp) : -1;
    ok = page >= 0 && page < ca.num_pages;
  }
  if (!__all_sync(0xffffffffu, ok)) return -1;
  const int pg = __shfl_sync(0xffffffffu, page, 0);
  const int row_bytes = ca.d * ca.elem_bytes, vecs = row_bytes >> 4, chunks = ca.hkv * vecs;
  const size_t dst0 = ((size_t)pg * ca.hkv * ca.page_size + P % ca.page_size) * row_bytes;
  for (int e = lane; e < chunks; e += 32) {
    const int g = e / vecs, vi = e - g * vecs;
    const size_t dst = dst0 + (size_t)g * ca.page_size * row_bytes + ((size_t)vi << 4);
    *reinterpret_cast<uint4*>(ca.k_pool + dst) = buf[e];
    *reinterpret_cast<uint4*>(ca.v_pool + dst) = buf[chunks + e];
  }
  return P;
}

// (five CTAs per SM: the streaming loop needs the occupancy, the final CTA's epilogue may spill)
template <bool kVec, bool kIns>
__global__ void __launch_bounds__(kAcceptThreads, 5) accept_greedy_kernel(
    const float* __restrict__ logits, int vocab, int gchunks, int tasks, const int32_t* __restrict__ qo,
    int batch, int total_nodes, const int32_t* __restrict__ parent, const int32_t* __restrict__ tokens,
    int path_cap, int32_t* accept_len, int32_t* path, int32_t* out_tokens, uint8_t* flags, unsigned* done,
    unsigned long long* slots, ArgPartial* partials, int* argmax, int32_t* status, const CommitArgs ca) {
  __shared__ float sv[2][kAcceptThreads / 32];
  __shared__ int si[2][kAcceptThreads / 32];
  __shared__ bool s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();  // stream order: nothing is read before the previous kernel has finished
  if (blockIdx.x == gridDim.x - 1) {  // what the last CTA reads at the end: into L2 early
    for (int i = threadIdx.x * 32; i < total_nodes; i += kAcceptThreads * 32) {
      asm volatile("prefetch.global.L2 [%0];" ::"l"(parent + i));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(tokens + i));
    }
    if (ca.k_tree != nullptr) {  // each sequence's page-table entries from its prefix end on
      for (int bb = threadIdx.x; bb < batch; bb += kAcceptThreads) {
        const int P = __ldg(ca.prefix_len + bb);
        const int lp = P >= 0 ? P / ca.page_size : 0;
        if (lp < ca.max_pages)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(ca.page_table + (size_t)bb * ca.max_pages + lp));
      }
    }
    if (ca.k_tree != nullptr) {  // the tree K/V rows the commit copies (a few MB at most)
      const size_t bytes = (size_t)total_nodes * ca.hkv * ca.d * ca.elem_bytes;
      if (bytes <= (size_t(4) << 20))
        for (size_t off = (size_t)threadIdx.x * 128; off < bytes; off += (size_t)kAcceptThreads * 128) {
          asm volatile("prefetch.global.L2 [%0];" ::"l"(ca.k_tree + off));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(ca.v_tree + off));
        }
    }
  }

  auto bounds = [&](int task, int& t, int& lo, int& hi) {
    t = task / gchunks;
    lo = (task - t * gchunks) * kGreedyChunk;
    hi = lo + kGreedyChunk < vocab ? lo + kGreedyChunk : vocab;
  };
  auto load = [&](int task, float4* x) {
    int t, lo, hi;
    bounds(task, t, lo, hi);
    const float4* r4 = reinterpret_cast<const float4*>(logits + (size_t)t * vocab);
    const int q1 = hi >> 2;  // vocab % 4 == 0 on this path
#pragma unroll
    for (int u = 0; u < kGreedyVec; ++u) {
      const int j = (lo >> 2) + threadIdx.x + u * kAcceptThreads;
      x[u] = j < q1 ? __ldcs(r4 + j) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
  };
  float4 cur[kGreedyVec], nxt[kGreedyVec];
  if (kVec && (int)blockIdx.x < tasks) load(blockIdx.x, cur);
  int k = 0;
  for (int task = blockIdx.x; task < tasks; task += gridDim.x, ++k) {
    int t, lo, hi;
    bounds(task, t, lo, hi);
    float bv = -INFINITY;
    int bi = INT_MAX;
    if (kVec) {
      if (task + (int)gridDim.x < tasks) load(task + gridDim.x, nxt);
#pragma unroll
      for (int u = 0; u < kGreedyVec; ++u) {
        const int e = lo + ((threadIdx.x + u * kAcceptThreads) << 2);
        if (e < hi) {
          arg_better(bv, bi, cur[u].x, e);
          arg_better(bv, bi, cur[u].y, e + 1);
          arg_better(bv, bi, cur[u].z, e + 2);
          arg_better(bv, bi, cur[u].w, e + 3);
        }
      }
#pragma unroll
      for (int u = 0; u < kGreedyVec; ++u) cur[u] = nxt[u];
    } else {
      const float* row = logits + (size_t)t * vocab;
      for (int e = lo + threadIdx.x; e < hi; e += kAcceptThreads) arg_better(bv, bi, __ldcs(row + e), e);
    }
    warp_arg_reduce(bv, bi);
    if (lane == 0) {  // two slots: task k+1 writes the other one, so one barrier per task
      sv[k & 1][warp] = bv;
      si[k & 1][warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kAcceptThreads / 32; ++w) arg_better(bv, bi, sv[k & 1][w], si[k & 1][w]);
      if (slots != nullptr) atomicMax(slots + t, arg_key(bv, bi));  // the row's running argmax
      else partials[task] = ArgPartial{bv, bi};
    }
  }
  if (threadIdx.x == 0) {
    // this CTA has streamed its tasks: the next kernel may be scheduled -- unless this
    // launch also commits K/V, which a next kernel may read before it waits
    if (ca.k_tree == nullptr) pdl_trigger();
    unsigned prev;  // one release-acquire RMW: this CTA's slot updates are visible before its count
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(prev) : "l"(done) : "memory");
    s_last = prev == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;

  // ---- the last CTA: argmax of every row, then the walk of every sequence
  __shared__ __align__(16) int s_stage[4][kGreedyStage];
  int* const s_par = s_stage[0];
  int* const s_tok = s_stage[1];
  int* const s_am = s_stage[2];
  int* const s_child = s_stage[3];
  __shared__ int s_len[kCommitCta];                     // L of sequences 0 .. 3 (fused commit)
  __shared__ int s_root_P[kCommitCta];                  // P when their root row went early, else -1
  __shared__ int s_cpath[kCommitCta][kCommitPathStage];  // their paths, when path_cap fits
  const bool staged = total_nodes <= kGreedyStage;
  if (threadIdx.x == 0) done[0] = 0u;  // every CTA has counted itself: ready for the next call
  // root rows of the fused commit: staged by the last warp (warps 0 .. batch - 1 walk) in
  // the upper halves of the staging arrays, which hold nothing when the trees are small
  constexpr int kRootWarp = kAcceptThreads / 32 - 1;
  const int root_chunks = ca.k_tree != nullptr ? ca.hkv * ca.d * ca.elem_bytes / 16 : 0;
  const bool early = ca.k_tree != nullptr && batch <= kCommitCta && total_nodes <= kGreedyStage / 2 &&
                     2 * root_chunks * 16 <= (kGreedyStage / 2) * (int)sizeof(int);
  auto root_buf = [&](int b) { return reinterpret_cast<uint4*>(s_stage[b] + kGreedyStage / 2); };
  int root_P = -1, root_n = 0;  // lane b of the root warp: sequence b's prefix length, node count
  if (early && warp == kRootWarp) {
    int base = 0;
    if (lane < batch) {
      base = __ldg(qo + lane);
      root_n = __ldg(qo + lane + 1) - base;
      root_P = __ldg(ca.prefix_len + lane);  // not waited for before the walk
    }
    for (int b = 0; b < batch; ++b) root_stage(ca, __shfl_sync(0xffffffffu, base, b), root_buf(b));
  }
  if (staged) {
    for (int i = threadIdx.x; i < total_nodes; i += kAcceptThreads) {
      s_par[i] = __ldg(parent + i);
      s_tok[i] = __ldg(tokens + i);
    }
  }
  if (slots != nullptr) {  // each row's argmax is already folded into its slot
    for (int t = threadIdx.x; t < total_nodes; t += kAcceptThreads) {
      const unsigned long long key = __ldcg(slots + t);
      slots[t] = 0ull;  // empty again for the next call
      const int ix = arg_key_index(key);
      const int a = (key == 0ull || ix < 0 || ix >= vocab) ? 0 : ix;
      if (staged) s_am[t] = a;
      else argmax[t] = a;
    }
  }
  // warp w: rows w, w + 8, ...; eight rows' partials loaded before any is reduced
  constexpr int kRowsPerPass = 8;
  for (int t0 = warp; slots == nullptr && t0 < total_nodes; t0 += kRowsPerPass * (kAcceptThreads / 32)) {
    float v[kRowsPerPass];
    int ix[kRowsPerPass];
#pragma unroll
    for (int r = 0; r < kRowsPerPass; ++r) {
      v[r] = -INFINITY;
      ix[r] = INT_MAX;
    }
    for (int c0 = 0; c0 < gchunks; c0 += 32) {
      const int c = c0 + lane;
      float2 pv[kRowsPerPass];  // (value, index bits): all loads issued before any compare
#pragma unroll
      for (int r = 0; r < kRowsPerPass; ++r) {
        const int t = t0 + r * (kAcceptThreads / 32);
        pv[r] = (t < total_nodes && c < gchunks)
                    ? __ldcg(reinterpret_cast<const float2*>(partials + (size_t)t * gchunks + c))
                    : make_float2(-INFINITY, __int_as_float(INT_MAX));
      }
#pragma unroll
      for (int r = 0; r < kRowsPerPass; ++r) arg_better(v[r], ix[r], pv[r].x, __float_as_int(pv[r].y));
    }
#pragma unroll
    for (int r = 0; r < kRowsPerPass; ++r) {
      const int t = t0 + r * (kAcceptThreads / 32);
      warp_arg_reduce(v[r], ix[r]);
      if (lane == 0 && t < total_nodes) {
        const int a = ix[r] == INT_MAX ? 0 : ix[r];
        if (staged) s_am[t] = a;
        else argmax[t] = a;
      }
    }
  }
  __syncthreads();
  for (int b = warp; b < batch; b += kAcceptThreads / 32) {
    const int base = __ldg(qo + b);
    const int n = min(__ldg(qo + b + 1) - base, kMaxTreeNodes);
    if (staged) {
      int* sp = (ca.k_tree != nullptr && b < kCommitCta && path_cap <= kCommitPathStage) ? s_cpath[b] : nullptr;
      const int L = greedy_walk_warp_staged(b, n, s_par + base, s_tok + base, s_am + base, s_child + base, path_cap,
                                            accept_len, path, out_tokens, flags, status, sp);
      if (b < kCommitCta && lane == 0) s_len[b] = L;
    }
    else
      greedy_walk_warp(b, n, parent + base, tokens + base, argmax + base, path_cap, accept_len, path, out_tokens,
                       flags, status);
  }
  if (early && warp == kRootWarp) {  // while warps 0 .. batch - 1 walk
    cp_async_wait_all();
    for (int b = 0; b < batch; ++b) {
      const int r = root_write<kIns>(ca, b, __shfl_sync(0xffffffffu, root_P, b), __shfl_sync(0xffffffffu, root_n, b),
                               path_cap, root_buf(b));
      if (lane == 0) s_root_P[b] = r;
    }
  }
  if (ca.k_tree == nullptr) return;
  // ---- fused commit of every sequence's accepted path
  __syncthreads();  // accept_len and the path rows written above are visible to the CTA
  if (batch <= kCommitCta) {  // few sequences: the whole CTA on each in turn
    const bool in_smem = staged && path_cap <= kCommitPathStage;
    for (int b = 0; b < batch; ++b) {
      const int base = __ldg(qo + b);
      const int rootP = early ? s_root_P[b] : -1;
      commit_sequence<true, kIns>(ca, b, base, __ldg(qo + b + 1) - base, staged ? s_len[b] : accept_len[b],
                            in_smem ? s_cpath[b] : nullptr, path + (size_t)b * path_cap, path_cap, status,
                            rootP >= 0 ? 1 : 0, rootP);
      __syncthreads();
    }
  } else {
    for (int b = warp; b < batch; b += kAcceptThreads / 32) {
      const int base = __ldg(qo + b);
      commit_sequence<false, kIns>(ca, b, base, __ldg(qo + b + 1) - base, accept_len[b], nullptr,
                             path + (size_t)b * path_cap, path_cap, status);
    }
  }
}

// ---------------------------------------------------------------- greedy: walk from the root
// Greedy acceptance needs the target argmax of the nodes the walk visits only: the root, then
// each accepted child. For many sequences of many nodes, reading just those rows beats
// streaming every row: one 8-CTA cluster per sequence walks from the root, each CTA takes the
// argmax of its eighth of the visited row (eight float4 loads in flight per thread), the eight
// (max, index) pairs meet through distributed shared memory, and every CTA finds the same
// child (the lowest id whose token is the argmax) in the sequence's staged tree. The outputs
// are the stream kernel's bit for bit (the same (value, lower index) order). The commit, when
// asked for, follows in the same launch: rank 0 of each cluster copies its sequence's path.
constexpr int kLazyCluster = 8;
constexpr int kLazyThreads = 512;

// Whether greedy acceptance walks from the root (true) or streams every row. The walk reads
// at most path_cap rows per sequence, one after another; the stream reads every row at the
// copy rate. A model of both (a step: ~1.5 us of latency plus an eighth of a row at ~50 GB/s
// per SM, two clusters' CTAs per SM; the stream: ~6 TB/s and a ~3.5 us tail) picks the walk
// only where it is clearly cheaper: many rows per sequence, several sequences.
bool greedy_walks(int batch, int total_nodes, int vocab, int path_cap, int sms) {
  if (batch > kMaxGridYZ || sms <= 0) return false;
  const double stream_us = (double)total_nodes * vocab * 4.0 / 6.0e6 + 3.5;
  const long clusters = (sms * 2L) / kLazyCluster > 0 ? (sms * 2L) / kLazyCluster : 1;
  const long waves = (batch + clusters - 1) / clusters;
  const double step_us = 1.5 + (double)vocab * 4.0 / kLazyCluster / 50.0e3;
  return (double)waves * path_cap * step_us < stream_us;
}

__global__ void __cluster_dims__(kLazyCluster, 1, 1) __launch_bounds__(kLazyThreads, 2)
    accept_greedy_lazy_kernel(const float* __restrict__ logits, int vocab, const int32_t* __restrict__ qo,
                              const int32_t* __restrict__ parent, const int32_t* __restrict__ tokens, int path_cap,
                              int32_t* accept_len, int32_t* path, int32_t* out_tokens, uint8_t* flags,
                              int32_t* status, bool vec, bool early, const CommitArgs ca) {
  cg::cluster_group cl = cg::this_cluster();
  constexpr int kWarps = kLazyThreads / 32;
  __shared__ int s_par[kMaxTreeNodes], s_tok[kMaxTreeNodes];
  __shared__ float s_wv[2][kWarps];  // each warp's (max, index) of the step, by step parity
  __shared__ int s_wi[2][kWarps];
  __shared__ int s_path[kMaxTreeNodes];  // the accepted nodes, written out after the wait below
  // The walk reads inputs only (the tree, the logits, qo_indptr). Where the caller has
  // declared that the kernel enqueued before this one writes none of them (early), it runs
  // before the grid-dependency wait, which then comes just before its first write, so its
  // reads overlap that kernel's tail; otherwise it waits first.
  if (!early) pdl_wait();
  const int b = blockIdx.y;
  const int rank = (int)cl.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int base = __ldg(qo + b);
  const int n = min(__ldg(qo + b + 1) - base, kMaxTreeNodes);
  int32_t* prow = path + (size_t)b * path_cap;
  int32_t* trow = out_tokens + (size_t)b * path_cap;
  const bool writer = rank == 0 && threadIdx.x == 0;
  if (n < 1) {  // the same in every CTA of the cluster: all leave here
    pdl_wait();
    if (writer) report(status, SPEC_ERR_CAPACITY);
    return;
  }
  for (int c = threadIdx.x; c < n; c += kLazyThreads) {
    s_par[c] = __ldg(parent + base + c);
    s_tok[c] = __ldg(tokens + base + c);
  }
  if (threadIdx.x == 0) s_path[0] = 0;  // the root
  const int per = ((vocab + kLazyCluster - 1) / kLazyCluster + 3) & ~3;
  const int c_lo = rank * per;
  const int n_sl = max(0, min(vocab, c_lo + per) - c_lo);
  int v = 0, L = 0, bonus = 0, parity = 0;
  bool truncated = false;
  __syncthreads();
  while (true) {
    const float* row = logits + (size_t)(base + v) * vocab + c_lo;
    float bv = -INFINITY;
    int bi = INT_MAX;
    if (vec) {
      const float4* r4 = reinterpret_cast<const float4*>(row);
      const int n4 = n_sl >> 2;  // (n_sl is a multiple of 4 when the vocabulary is)
      for (int i0 = threadIdx.x; i0 < n4; i0 += 8 * kLazyThreads) {
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {  // every load issued (clamped into the slice), then used
          const int i = i0 + u * kLazyThreads;
          x[u] = __ldcs(r4 + (i < n4 ? i : n4 - 1));
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * kLazyThreads;
          if (i < n4) {
            const int e = c_lo + 4 * i;
            arg_better(bv, bi, x[u].x, e);
            arg_better(bv, bi, x[u].y, e + 1);
            arg_better(bv, bi, x[u].z, e + 2);
            arg_better(bv, bi, x[u].w, e + 3);
          }
        }
      }
    } else {
      for (int i = threadIdx.x; i < n_sl; i += kLazyThreads) arg_better(bv, bi, __ldcs(row + i), c_lo + i);
    }
    warp_arg_reduce(bv, bi);
    if (lane == 0) {
      s_wv[parity][warp] = bv;
      s_wi[parity][warp] = bi;
    }
    // One barrier per step: every warp of every CTA publishes its pair, then every warp reads
    // all kLazyCluster x kWarps pairs itself (kPer per lane, every load issued first) and finds
    // the child on its own, so no block barrier follows. (A pair of this parity is written
    // again two steps on, after the next step's barrier, which no thread passes before it has
    // finished reading this step's pairs.)
    cl.sync();
    constexpr int kPairs = kLazyCluster * kWarps, kPer = kPairs / 32;
    static_assert(kPairs % 32 == 0, "the pairs split evenly over a warp's lanes");
    float ov[kPer];
    int oi[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int e = lane + 32 * k, r = e / kWarps, w = e - r * kWarps;
      ov[k] = *cl.map_shared_rank(&s_wv[parity][w], r);
      oi[k] = *cl.map_shared_rank(&s_wi[parity][w], r);
    }
    float av = ov[0];
    int ai = oi[0];
#pragma unroll
    for (int k = 1; k < kPer; ++k) arg_better(av, ai, ov[k], oi[k]);
    warp_arg_reduce(av, ai);  // (a total order: every warp of every CTA gets the same pair)
    const int a = ai == INT_MAX ? 0 : ai;  // (an empty or all-NaN row: token 0, as the stream kernel)
    // the child of v whose token is a, lowest id first: each lane's first match, then the
    // warp's minimum
    int mine = INT_MAX;
    for (int c = v + 1 + lane; c < n; c += 32)
      if (s_par[c] == v && s_tok[c] == a) {
        mine = c;
        break;
      }
    const int c = (int)__reduce_min_sync(0xffffffffu, (unsigned)mine);
    if (c == INT_MAX) {
      bonus = a;
      break;
    }
    if (L + 1 >= path_cap) {  // accepted path does not fit: truncate here
      truncated = true;
      bonus = a;
      break;
    }
    ++L;
    if (threadIdx.x == 0) s_path[L] = c;  // (L < n: the path visits distinct nodes)
    v = c;
    parity ^= 1;
  }
  // The commit's reads (the path's K/V rows, the prefix length, the slots' page entries) are
  // inputs too: with early reads they go out before the wait, and only stores follow it.
  const bool commit = ca.k_tree != nullptr && rank == 0;
  CommitLoad pre;
  if (commit && early) {
    __syncthreads();  // (s_path complete)
    walk_commit_load(ca, b, base, n, L, s_path, path_cap, pre);
  }
  pdl_wait();  // the kernel before has finished: the outputs may be written
  __syncthreads();  // (s_path complete)
  if (rank == 0) {
    for (int k = threadIdx.x; k < path_cap; k += kLazyThreads) {
      const int node = k == 0 ? 0 : k <= L ? s_path[k] : -1;
      prow[k] = node;
      trow[k] = k < L ? s_tok[s_path[k + 1]] : k == L ? bonus : -1;
    }
    if (threadIdx.x == 0) {
      accept_len[b] = L;
      if (flags != nullptr) flags[b] = 0;
      if (truncated) report(status, SPEC_ERR_CAPACITY);
    }
  }
  cl.sync();  // no CTA leaves while another may still read its shared memory
  if (commit) {  // the commit of this sequence's path (the whole CTA)
    __syncthreads();  // (the path and tokens written above are visible to the CTA)
    if (!early) walk_commit_load(ca, b, base, n, L, s_path, path_cap, pre);
    if (ca.ins.token_buf != nullptr)
      walk_commit_store<true>(ca, b, base, L, s_path, path_cap, status, pre);
    else
      walk_commit_store<false>(ca, b, base, L, s_path, path_cap, status, pre);
  }
}

// ---------------------------------------------------------------- stochastic: walk

// The CTA's slice [c_lo, c_hi) of the vocabulary (a multiple of 4 tokens long, so rows
// with 16-byte alignment stage with float4 loads) is cut into kWalkWarps contiguous
// segments, one per warp (a multiple of 256 tokens each); lane l of a warp takes the
// segment's tokens l, l + 32, ... At a node's first pass p and q of the slice are staged
// in shared memory as fp32 values, zero past the slice up to kWalkWarps whole segments
// (a zero p and q add nothing), so the passes load eight tokens at a time without a
// bounds test (dynamic shared memory: kWalkStage of each at most, i.e. vocabularies up to
// about 8 x kWalkStage tokens; larger ones are evaluated from global memory on every pass,
// with the same arithmetic). Sums: fp32 Kahan per lane, then
// double-float (an fp32 pair, error-free adds, about 48 significant bits) across lanes,
// warps and the CTAs of the cluster. The decisions are taken in double-float as well, with no
// fp64: on this part a dependent fp64 operation costs hundreds of cycles.
constexpr int kWalkWarps = kWalkThreads / 32;
constexpr int kWalkKids = 32;  // children listed per batch
static_assert(kMaxTreeNodes == 32 * 32, "the children bitmap is one word per lane of a warp");
static_assert((kWalkWarps * 256) % (8 * kWalkThreads) == 0, "a staged slice is whole steps of eight");
constexpr int kWalkStage = 24576;

struct WalkShared {
  float row_max[2];                   // this CTA's max of the visited row (target, draft)
  float row_sum[4];                   // this CTA's sums of exp((x - max) / T) (hi, lo; target, draft)
  float red[2][kWalkWarps];           // per-warp maxima
  float red_hi[2][kWalkWarps], red_lo[2][kWalkWarps];  // per-warp sums
  float part_hi[kWalkWarps], part_lo[kWalkWarps];  // this pass's segment sums (double-float)
  float pre_hi[kWalkWarps], pre_lo[kWalkWarps];    // their exclusive prefix (bonus draw)
  float cta_hi[2], cta_lo[2];         // this CTA's pass total (double-buffered by pass parity)
  unsigned kids[kMaxTreeNodes / 32];  // children bitmap of the current node
  // the next children to test (ascending id) with what their tests read: loaded together,
  // so the tests do not each wait on a token load and then on its logits
  int kid_c[kWalkKids], kid_x[kWalkKids];
  float kid_p[kWalkKids], kid_q[kWalkKids], kid_u[kWalkKids];
  int nkids;
  int found;                          // bonus token found by this CTA (-1 = none)
  int found_flag;
};

// p(t) and q(t) of the visited node in fp32, from global memory (the staging source and
// the path for vocabularies too large to stage).
struct RowEval {
  const float* tl;
  const float* dl;
  float m_p, m_q, invT, inv_zp, inv_zq;
  __device__ __forceinline__ float pv(float x) const { return expf((x - m_p) * invT) * inv_zp; }
  __device__ __forceinline__ float qv(float x) const { return expf((x - m_q) * invT) * inv_zq; }
  __device__ __forceinline__ float p(int t) const { return pv(__ldg(tl + t)); }
  __device__ __forceinline__ float q(int t) const { return qv(__ldg(dl + t)); }
};

struct WalkSlice {
  int c_lo, n, seg;  // slice start, its length, the segment length
  float* sp;         // staged p and q (nullptr: not staged for this vocabulary)
  float* sq;
  __device__ __forceinline__ float p(const RowEval& ev, int i) const { return sp ? sp[i] : ev.p(c_lo + i); }
  __device__ __forceinline__ float q(const RowEval& ev, int i) const { return sq ? sq[i] : ev.q(c_lo + i); }
  __device__ __forceinline__ float resid(const RowEval& ev, int i, float c) const {
    const float pt = p(ev, i);
    return c == 0.f ? pt : fmaxf(pt - c * q(ev, i), 0.f);
  }
};

// A CTA's slice length, its segment length, and the floats staged per row (p, and q after
// it): the kernel's layout and the launch's dynamic shared memory both come from here.
__host__ __device__ __forceinline__ int walk_per_cta(int vocab) {
  return ((vocab + kWalkCluster - 1) / kWalkCluster + 3) & ~3;
}
__host__ __device__ __forceinline__ int walk_seg(int vocab) {
  return ((walk_per_cta(vocab) + kWalkWarps - 1) / kWalkWarps + 255) & ~255;
}
__host__ __device__ __forceinline__ int walk_stage_floats(int vocab) {  // 0: not staged
  const int padded = kWalkWarps * walk_seg(vocab);
  return padded <= kWalkStage ? padded : 0;
}

__device__ __forceinline__ WalkSlice walk_slice(int vocab, int rank, float* smem) {
  const int per_cta = walk_per_cta(vocab);
  WalkSlice s;
  s.c_lo = rank * per_cta;
  s.n = max(0, min(vocab, s.c_lo + per_cta) - s.c_lo);
  s.seg = walk_seg(vocab);  // (the same in every CTA)
  const int staged = walk_stage_floats(vocab);
  s.sp = staged > 0 ? smem : nullptr;
  s.sq = staged > 0 ? smem + staged : nullptr;
  return s;
}

// The visited row's statistics, by the cluster (every CTA gets the same bits): the max of the
// target and of the draft logits, then their sums of exp((x - max) / T), each CTA over its
// slice, exchanged through distributed shared memory. When the slice is staged, its logits go
// into the staging arrays once (-inf past the slice, so no test is needed in the loops), the
// sum pass leaves exp((x - max) / T) there and the last pass scales it into p and q (the
// padding then holds 0). The tests' p(x) = RowEval::p gives the same bits.
__device__ NodeStats walk_row_stats(cg::cluster_group& cl, WalkShared& sh, const WalkSlice& sl, const float* trow,
                                    const float* drow, float invT, bool vec) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pad = kWalkWarps * sl.seg;
  float mp = -INFINITY, mq = -INFINITY;
  if (sl.sp != nullptr) {
    const int n4 = sl.n >> 2, pad4 = pad >> 2;
    const float4 neg = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4* p4 = reinterpret_cast<float4*>(sl.sp);
    float4* q4 = reinterpret_cast<float4*>(sl.sq);
    if (vec && n4 > 0) {  // (n is a multiple of 4 when the vocabulary is)
      const float4* t4 = reinterpret_cast<const float4*>(trow + sl.c_lo);
      const float4* d4 = reinterpret_cast<const float4*>(drow + sl.c_lo);
      for (int i0 = threadIdx.x; i0 < pad4; i0 += 8 * kWalkThreads) {
        float4 a[8], d[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {  // every load issued (clamped into the slice), then used
          const int i = i0 + u * kWalkThreads;
          const int ic = i < n4 ? i : n4 - 1;
          a[u] = __ldg(t4 + ic);
          d[u] = __ldg(d4 + ic);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * kWalkThreads;
          if (i < pad4) {
            const float4 x = i < n4 ? a[u] : neg, y = i < n4 ? d[u] : neg;
            p4[i] = x;
            q4[i] = y;
            mp = fmaxf(mp, fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
            mq = fmaxf(mq, fmaxf(fmaxf(y.x, y.y), fmaxf(y.z, y.w)));
          }
        }
      }
    } else {
      for (int i = threadIdx.x; i < pad; i += kWalkThreads) {
        const float x = i < sl.n ? __ldg(trow + sl.c_lo + i) : -INFINITY;
        const float y = i < sl.n ? __ldg(drow + sl.c_lo + i) : -INFINITY;
        sl.sp[i] = x;
        sl.sq[i] = y;
        mp = fmaxf(mp, x);
        mq = fmaxf(mq, y);
      }
    }
  } else {
    for (int i = threadIdx.x; i < sl.n; i += kWalkThreads) {
      mp = fmaxf(mp, __ldg(trow + sl.c_lo + i));
      mq = fmaxf(mq, __ldg(drow + sl.c_lo + i));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, o));
    mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
  }
  if (lane == 0) {
    sh.red[0][warp] = mp;
    sh.red[1][warp] = mq;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = sh.red[0][0], d = sh.red[1][0];
    for (int w = 1; w < kWalkWarps; ++w) {
      a = fmaxf(a, sh.red[0][w]);
      d = fmaxf(d, sh.red[1][w]);
    }
    sh.row_max[0] = a;
    sh.row_max[1] = d;
  }
  cl.sync();  // every CTA's max is in place
  float xm[kWalkCluster], ym[kWalkCluster];
#pragma unroll
  for (int r = 0; r < kWalkCluster; ++r) {
    xm[r] = *cl.map_shared_rank(&sh.row_max[0], r);
    ym[r] = *cl.map_shared_rank(&sh.row_max[1], r);
  }
  float Mp = xm[0], Mq = ym[0];
#pragma unroll
  for (int r = 1; r < kWalkCluster; ++r) {
    Mp = fmaxf(Mp, xm[r]);
    Mq = fmaxf(Mq, ym[r]);
  }
  // sums of exp((x - M) / T): Kahan per thread, double-float across threads, warps and CTAs
  float sp = 0.f, cp = 0.f, sq = 0.f, cq = 0.f;
  auto kahan = [](float e, float& sum, float& comp) {
    const float y = e - comp, z = sum + y;
    comp = (z - sum) - y;
    sum = z;
  };
  const bool okp = Mp != -INFINITY, okq = Mq != -INFINITY;  // (a row of -inf has no mass)
  if (sl.sp != nullptr) {  // (pad is a multiple of 8 x kWalkThreads: no bounds test)
    for (int i0 = threadIdx.x; i0 < pad; i0 += 8 * kWalkThreads) {
      float x[8], y[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        x[u] = sl.sp[i0 + u * kWalkThreads];
        y[u] = sl.sq[i0 + u * kWalkThreads];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float ep = okp ? expf((x[u] - Mp) * invT) : 0.f, eq = okq ? expf((y[u] - Mq) * invT) : 0.f;
        sl.sp[i0 + u * kWalkThreads] = ep;
        sl.sq[i0 + u * kWalkThreads] = eq;
        kahan(ep, sp, cp);
        kahan(eq, sq, cq);
      }
    }
  } else {
    for (int i = threadIdx.x; i < sl.n; i += kWalkThreads) {
      if (okp) kahan(expf((__ldg(trow + sl.c_lo + i) - Mp) * invT), sp, cp);
      if (okq) kahan(expf((__ldg(drow + sl.c_lo + i) - Mq) * invT), sq, cq);
    }
  }
  const F2 wp = f2_warp_sum(F2{sp, -cp}), wq = f2_warp_sum(F2{sq, -cq});
  if (lane == 0) {
    sh.red_hi[0][warp] = wp.hi;
    sh.red_lo[0][warp] = wp.lo;
    sh.red_hi[1][warp] = wq.hi;
    sh.red_lo[1][warp] = wq.lo;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    F2 tp{0.f, 0.f}, tq{0.f, 0.f};
    for (int w = 0; w < kWalkWarps; ++w) {
      tp = f2_add(tp, F2{sh.red_hi[0][w], sh.red_lo[0][w]});
      tq = f2_add(tq, F2{sh.red_hi[1][w], sh.red_lo[1][w]});
    }
    sh.row_sum[0] = tp.hi;
    sh.row_sum[1] = tp.lo;
    sh.row_sum[2] = tq.hi;
    sh.row_sum[3] = tq.lo;
  }
  cl.sync();  // every CTA's sums are in place
  float zs[4][kWalkCluster];
#pragma unroll
  for (int r = 0; r < kWalkCluster; ++r)
#pragma unroll
    for (int k = 0; k < 4; ++k) zs[k][r] = *cl.map_shared_rank(&sh.row_sum[k], r);
  F2 Zp{0.f, 0.f}, Zq{0.f, 0.f};
#pragma unroll
  for (int r = 0; r < kWalkCluster; ++r) {
    Zp = f2_add(Zp, F2{zs[0][r], zs[1][r]});
    Zq = f2_add(Zq, F2{zs[2][r], zs[3][r]});
  }
  const NodeStats st{Mp, Mq, f2_rcp(Zp), f2_rcp(Zq)};
  if (sl.sp != nullptr) {  // exp((x - M) / T) into p and q
    for (int i = threadIdx.x; i < pad; i += kWalkThreads) {
      sl.sp[i] *= st.inv_zp;
      sl.sq[i] *= st.inv_zq;
    }
  }
  __syncthreads();
  return st;
}

// One pass: sum over the whole vocabulary (all CTAs of the cluster) of the residual with
// coefficient c, identical bitwise in every CTA (double-float). Leaves the segment sums in
// sh.part_hi / part_lo and, when `prefix`, their exclusive prefix in sh.pre_hi / pre_lo;
// *cta_pre receives the sum over the CTAs ranked before this one.
__device__ F2 walk_pass(cg::cluster_group& cl, WalkShared& sh, const WalkSlice& sl, const RowEval& ev, float c,
                        int parity, bool prefix, F2* cta_pre) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s_lo = warp * sl.seg, s_hi = min(sl.n, s_lo + sl.seg);
  float s = 0.f, comp = 0.f;
  auto add = [&](float x) {  // fp32 Kahan step
    const float y = x - comp;
    const float z = s + y;
    comp = (z - s) - y;
    s = z;
  };
  if (sl.sp != nullptr) {  // staged and padded: whole segments, eight tokens in flight
    for (int i0 = s_lo + lane; i0 < s_lo + sl.seg; i0 += 32 * 8) {
      float pv[8], qv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        pv[u] = sl.sp[i0 + 32 * u];
        qv[u] = sl.sq[i0 + 32 * u];
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) add(c == 0.f ? pv[u] : fmaxf(pv[u] - c * qv[u], 0.f));
    }
  } else {
    for (int i = s_lo + lane; i < s_hi; i += 32) add(sl.resid(ev, i, c));
  }
  const F2 w = f2_warp_sum(F2{s, -comp});
  if (lane == 0) {
    sh.part_hi[warp] = w.hi;
    sh.part_lo[warp] = w.lo;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    F2 tot{0.f, 0.f};
    for (int k = 0; k < kWalkWarps; ++k) {
      if (prefix) {
        sh.pre_hi[k] = tot.hi;
        sh.pre_lo[k] = tot.lo;
      }
      tot = f2_add(tot, F2{sh.part_hi[k], sh.part_lo[k]});
    }
    sh.cta_hi[parity] = tot.hi;
    sh.cta_lo[parity] = tot.lo;
  }
  cl.sync();
  const int rank = (int)cl.block_rank();
  float xh[kWalkCluster], xl[kWalkCluster];  // every CTA's total: all sixteen loads first
#pragma unroll
  for (int r = 0; r < kWalkCluster; ++r) {
    xh[r] = *cl.map_shared_rank(&sh.cta_hi[parity], r);
    xl[r] = *cl.map_shared_rank(&sh.cta_lo[parity], r);
  }
  F2 all{0.f, 0.f}, pre{0.f, 0.f};
#pragma unroll
  for (int r = 0; r < kWalkCluster; ++r) {
    if (r == rank) pre = all;
    all = f2_add(all, F2{xh[r], xl[r]});
  }
  if (cta_pre != nullptr) *cta_pre = pre;
  return all;
}

__global__ void __cluster_dims__(kWalkCluster, 1, 1) __launch_bounds__(kWalkThreads)
    accept_walk_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ tokens,
                       const float* __restrict__ tl, const float* __restrict__ dl,
                       const float* __restrict__ uniforms, float temperature, int vocab,
                       const int32_t* __restrict__ qo, int path_cap, int32_t* accept_len, int32_t* path,
                       int32_t* out_tokens, uint8_t* flags,
                       int32_t* status, bool vec) {
  cg::cluster_group cl = cg::this_cluster();
  __shared__ WalkShared sh;
  extern __shared__ __align__(16) float walk_smem[];
  pdl_wait();  // stream order: the inputs may come from the kernel before
  const int b = blockIdx.y;
  const int rank = (int)cl.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int base = __ldg(qo + b);
  const int n = __ldg(qo + b + 1) - base;
  const float invT = 1.0f / temperature;
  int32_t* prow = path + (size_t)b * path_cap;
  int32_t* trow = out_tokens + (size_t)b * path_cap;
  const bool writer = rank == 0 && threadIdx.x == 0;
  if (n < 1 || n > kMaxTreeNodes) {  // same answer in every CTA of the cluster: all leave here
    if (writer) report(status, SPEC_ERR_CAPACITY);
    return;
  }
  const WalkSlice sl = walk_slice(vocab, rank, walk_smem);
  if (writer) prow[0] = 0;
  int v = 0, L = 0, flag = 0, bonus = 0;
  int parity = 0;
  while (true) {
    // children bitmap of v (its loads in flight with the row's), then v's row statistics and,
    // when staged, p and q of the slice
    for (int w = threadIdx.x; w < kMaxTreeNodes / 32; w += blockDim.x) sh.kids[w] = 0u;
    __syncthreads();
    for (int c = v + 1 + threadIdx.x; c < n; c += blockDim.x)
      if (__ldg(parent + base + c) == v) atomicOr(&sh.kids[c >> 5], 1u << (c & 31));
    const float* trow_v = tl + (size_t)(base + v) * vocab;
    const float* drow_v = dl + (size_t)(base + v) * vocab;
    const NodeStats st = walk_row_stats(cl, sh, sl, trow_v, drow_v, invT, vec);  // (syncs the CTA)
    const RowEval ev{trow_v, drow_v, st.m_p, st.m_q, invT, st.inv_zp, st.inv_zq};
    F2 cc{0.f, 0.f}, ss{1.f, 0.f};  // residual r = max(p - cc q, 0) / ss (double-float)
    int accepted = -1;
    int next_c = v + 1;  // children with ids >= next_c are not listed yet
    while (accepted < 0) {
      // list the next children (ascending id): warp 0, one bitmap word per lane
      if (warp == 0) {
        unsigned bits = sh.kids[lane];
        const int w0 = next_c >> 5;
        if (lane < w0) bits = 0u;
        if (lane == w0) bits &= ~((1u << (next_c & 31)) - 1u);
        const int cnt = __popc(bits);
        int incl = cnt;  // inclusive prefix of the counts over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        int at = incl - cnt;
        while (bits && at < kWalkKids) {
          sh.kid_c[at++] = (lane << 5) + __ffs(bits) - 1;
          bits &= bits - 1;
        }
        if (lane == 31) sh.nkids = min(incl, kWalkKids);
      }
      __syncthreads();
      const int nk = sh.nkids;
      if (nk == 0) break;
      // their tokens, then p(x), q(x) (the fp32 values the passes use) and u: one round trip each
      for (int j = threadIdx.x; j < nk; j += blockDim.x) {
        const int c = sh.kid_c[j];
        const int x = __ldg(tokens + base + c);
        sh.kid_x[j] = x;
        const bool okx = x >= 0 && x < vocab;
        sh.kid_p[j] = okx ? ev.p(x) : 0.f;
        sh.kid_q[j] = okx ? ev.q(x) : 0.f;
        sh.kid_u[j] = __ldg(uniforms + 2 * (size_t)(base + c));
      }
      __syncthreads();
      for (int j = 0; j < nk; ++j) {
        const int c = sh.kid_c[j];
        const int x = sh.kid_x[j];
        if (x < 0 || x >= vocab) {
          if (writer) report(status, SPEC_ERR_INDEX);
          continue;
        }
        // the test u < max(p - cc q, 0) / (ss q) as u ss q < max(p - cc q, 0) in double-float
        // (about 48 bits: a decision it could take otherwise than fp64 lies far inside the
        // flagged band), with no exponential or division there
        const float px = sh.kid_p[j], qx = sh.kid_q[j], u = sh.kid_u[j];
        const F2 cq = f2_mul_f(cc, qx);
        F2 num = f2_add(F2{px, 0.f}, F2{-cq.hi, -cq.lo});
        if (!f2_gt(num, F2{0.f, 0.f})) num = F2{0.f, 0.f};
        bool ok;
        if (qx > 0.f) {
          const F2 den = f2_mul_f(ss, qx);
          const F2 lhs = f2_mul_f(den, u);
          const F2 gap = f2_add(lhs, F2{-num.hi, -num.lo});
          if (fabsf(gap.hi + gap.lo) <= (float)kTieEps * (den.hi + den.lo)) flag |= 1;
          ok = f2_gt(num, lhs);
        } else {
          ok = f2_gt(num, F2{0.f, 0.f});
        }
        if (ok) {
          accepted = c;
          break;
        }
        const F2 cn = f2_add(cc, ss);
        const F2 sn = walk_pass(cl, sh, sl, ev, cn.hi + cn.lo, parity, false, nullptr);
        parity ^= 1;
        if (f2_gt(sn, F2{0.f, 0.f})) {
          cc = cn;
          ss = sn;
        }
      }
      next_c = sh.kid_c[nk - 1] + 1;
      __syncthreads();  // (the list is rewritten next round)
    }
    __syncthreads();  // everyone done with sh.kids before the next node rebuilds it
    if (accepted >= 0) {
      if (L + 1 >= path_cap) {
        if (writer) report(status, SPEC_ERR_CAPACITY);
        accepted = -1;  // truncate: fall through to the bonus draw at v
      } else {
        ++L;
        if (writer) {
          prow[L] = accepted;
          trow[L - 1] = __ldg(tokens + base + accepted);
        }
        v = accepted;
        continue;
      }
    }
    // bonus: inverse-CDF draw from r = max(p - cc q, 0) / ss with u_bonus of v: the smallest
    // token whose cumulative residual exceeds u * total. The segment sums locate the
    // segment holding the threshold; its warp scans it 32 tokens at a time.
    {
      const float cf = cc.hi + cc.lo;
      F2 cta_pre{0.f, 0.f};
      const F2 total2 = walk_pass(cl, sh, sl, ev, cf, parity, true, &cta_pre);
      parity ^= 1;
      if (threadIdx.x == 0) {
        sh.found = -1;
        sh.found_flag = 0;
      }
      __syncthreads();
      // threshold and segment bounds in double-float: the segment intervals tile the line
      const F2 thr = f2_mul_f(total2, __ldg(uniforms + 2 * (size_t)(base + v) + 1));
      const int s_lo = warp * sl.seg, s_hi = min(sl.n, s_lo + sl.seg);
      const F2 seg_start = f2_add(cta_pre, F2{sh.pre_hi[warp], sh.pre_lo[warp]});
      const F2 seg_end = f2_add(seg_start, F2{sh.part_hi[warp], sh.part_lo[warp]});
      if (s_hi > s_lo && !f2_gt(seg_start, thr) && f2_gt(seg_end, thr)) {  // (warp-uniform)
        // The segment holds the threshold. Lane l sums its own contiguous run of sub = seg / 32
        // tokens (read in a rotated order, so the lanes hit distinct banks), a double-float scan
        // over the lanes finds the run where the cumulative residual crosses, and that run's
        // lane walks it in order for the token.
        const F2 loc = f2_add(thr, F2{-seg_start.hi, -seg_start.lo});
        const float band = (float)kBonusEps * (total2.hi + total2.lo);
        const int sub = sl.seg >> 5;
        const int r_lo = s_lo + lane * sub, r_hi = min(s_hi, r_lo + sub);
        float rs = 0.f, rc = 0.f;
        int lp = -1;  // the run's last token with positive residual
        const int rot = lane % sub;
        auto take = [&](int i, float rv) {  // fp32 Kahan step; the last positive token
          const float y = rv - rc, z = rs + y;
          rc = (z - rs) - y;
          rs = z;
          if (rv > 0.f && i > lp) lp = i;
        };
        if (sl.sp != nullptr) {  // staged: padded with zeros, eight tokens in flight (sub % 8 == 0)
          for (int t0 = 0; t0 < sub; t0 += 8) {
            float pv[8], qv[8];
            int ix[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int o = t0 + u + rot;
              ix[u] = r_lo + (o < sub ? o : o - sub);
              pv[u] = sl.sp[ix[u]];
              qv[u] = sl.sq[ix[u]];
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) take(ix[u], cf == 0.f ? pv[u] : fmaxf(pv[u] - cf * qv[u], 0.f));
          }
        } else {
          for (int t = 0; t < sub; ++t) {
            const int o = t + rot;
            const int i = r_lo + (o < sub ? o : o - sub);
            take(i, i < r_hi ? sl.resid(ev, i, cf) : 0.f);
          }
        }
        F2 inc{rs, -rc};  // inclusive scan of the runs' sums over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const F2 y{__shfl_up_sync(0xffffffffu, inc.hi, o), __shfl_up_sync(0xffffffffu, inc.lo, o)};
          if (lane >= o) inc = f2_add(y, inc);
        }
        F2 exc{__shfl_up_sync(0xffffffffu, inc.hi, 1), __shfl_up_sync(0xffffffffu, inc.lo, 1)};
        if (lane == 0) exc = F2{0.f, 0.f};
        const unsigned hit = __ballot_sync(0xffffffffu, r_hi > r_lo && f2_gt(inc, loc));
        int tok = -1, fl = 0;
        if (hit) {
          // the crossing run, in order, 32 tokens a round: lane j takes the round's j-th token,
          // an inclusive double-float scan over the lanes, the first lane past the threshold
          const int l = __ffs(hit) - 1;
          const int c_lo = s_lo + l * sub, c_hi = min(s_hi, c_lo + sub);
          F2 carry{__shfl_sync(0xffffffffu, exc.hi, l), __shfl_sync(0xffffffffu, exc.lo, l)};
          for (int i0 = c_lo; i0 < c_hi && tok < 0; i0 += 32) {
            const int i = i0 + lane;
            const float rv = i < c_hi ? sl.resid(ev, i, cf) : 0.f;
            F2 in2{rv, 0.f};
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const F2 y{__shfl_up_sync(0xffffffffu, in2.hi, o), __shfl_up_sync(0xffffffffu, in2.lo, o)};
              if (lane >= o) in2 = f2_add(y, in2);
            }
            const F2 cum = f2_add(carry, in2);
            const unsigned h2 = __ballot_sync(0xffffffffu, i < c_hi && f2_gt(cum, loc));
            if (h2) {
              const int j = __ffs(h2) - 1;
              tok = sl.c_lo + i0 + j;
              // distances of the crossing token's two CDF edges from the threshold
              const F2 da = f2_add(cum, F2{-loc.hi, -loc.lo});
              const F2 db = f2_add(da, F2{-rv, 0.f});
              const float d_after = __shfl_sync(0xffffffffu, da.hi + da.lo, j);
              const float d_before = __shfl_sync(0xffffffffu, db.hi + db.lo, j);
              if (fabsf(d_after) <= band || fabsf(d_before) <= band) fl = 2;
            }
            carry = F2{__shfl_sync(0xffffffffu, cum.hi, 31), __shfl_sync(0xffffffffu, cum.lo, 31)};
          }
          if (tok < 0) {  // the in-order sum fell short of the run's total: at its last mass
            const int lpl = __shfl_sync(0xffffffffu, lp, l);
            tok = sl.c_lo + (lpl >= 0 ? lpl : c_lo);
            fl = 2;
          }
        } else {  // rounding put the crossing just past this segment's last mass
          const int last = __reduce_max_sync(0xffffffffu, (unsigned)(lp + 1)) - 1;
          tok = sl.c_lo + (last >= 0 ? last : s_lo);
          fl = 2;
        }
        if (lane == 0) {
          sh.found = tok;
          sh.found_flag = fl;
        }
      }
      cl.sync();
      if (rank == 0 && threadIdx.x == 0) {
        int fs[kWalkCluster], ffl[kWalkCluster];  // all sixteen loads first
#pragma unroll
        for (int r = 0; r < kWalkCluster; ++r) {
          fs[r] = *cl.map_shared_rank(&sh.found, r);
          ffl[r] = *cl.map_shared_rank(&sh.found_flag, r);
        }
        int tok = -1;
#pragma unroll
        for (int r = 0; r < kWalkCluster; ++r)
          if (tok < 0 && fs[r] >= 0) {
            tok = fs[r];
            flag |= ffl[r];
          }
        if (tok < 0) flag |= 2;  // (no segment held the threshold: an fp64 rounding gap, flagged)
        bonus = tok < 0 ? 0 : tok;
      }
      cl.sync();  // keep every CTA's shared memory alive until rank 0 has read it
      break;
    }
  }
  if (writer) {
    trow[L] = bonus;
    accept_len[b] = L;
    for (int k = L + 1; k < path_cap; ++k) {
      prow[k] = -1;
      trow[k] = -1;
    }
    if (flags != nullptr) flags[b] = (uint8_t)flag;
  }
}

int launch_kv_commit(int elem_bytes, const void* k_tree, const void* v_tree, const int32_t* path, int path_cap,
                     const int32_t* accept_len, const int32_t* qo, const int32_t* page_table, int max_pages,
                     int num_pages, int page_size, const int32_t* prefix_len, int32_t* seq_len_out, void* k_pool,
                     void* v_pool, int batch, int hkv, int d, int32_t* status, cudaStream_t stream, TokenInsert ins);

// `commit` (nullable): also commit the accepted paths' K/V, as spec_kv_commit would right
// after; greedy does it inside the acceptance kernel, stochastic with the commit kernel.
int launch_accept(int mode, const int32_t* parent, const int32_t* tokens, const float* tl,
                  const float* dl, const float* uniforms, float temperature, int vocab,
                  const int32_t* qo, int batch, int total_nodes, int path_cap, int32_t* accept_len,
                  int32_t* path, int32_t* out_tokens, uint8_t* flags, void* ws, int32_t* status,
                  cudaStream_t stream, const CommitArgs* commit, bool host_logits) {
  CommitArgs ca = {};
  if (commit != nullptr) ca = *commit;
  const bool vec = (vocab % 4 == 0) && ((reinterpret_cast<uintptr_t>(tl) & 15) == 0) &&
                   (dl == nullptr || (reinterpret_cast<uintptr_t>(dl) & 15) == 0);
  if (mode == SPEC_GREEDY && vec && batch <= kMaxGridYZ) {  // the walk from the root, commit fused
    static PerDevice sm_walk;
    const int sms = per_device(sm_walk, [](int dev) {
      int v = 0;
      return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0 ? v : 0;
    });
    if (sms == 0) return SPEC_ERR_CUDA;
    // logits in host memory: the walk, whose reads cross the host link for the visited rows only
    if (host_logits || greedy_walks(batch, total_nodes, vocab, path_cap, sms)) {
      if (launch_pdl(accept_greedy_lazy_kernel, dim3(kLazyCluster, batch), dim3(kLazyThreads), 0, stream, tl, vocab,
                     qo, parent, tokens, path_cap, accept_len, path, out_tokens, flags, status, vec, early_reads(), ca) !=
          cudaSuccess)
        return SPEC_ERR_CUDA;
      return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
    }
  }
  // Greedy commits inside the acceptance kernel only for a few sequences: its final CTA does
  // them one after another. More sequences are committed by the commit kernel (one CTA per
  // sequence, launched to start as the acceptance grid drains), like the stochastic path.
  if (mode == SPEC_GREEDY && ca.k_tree != nullptr && batch > kCommitCta) {
    const int e = launch_accept(mode, parent, tokens, tl, dl, uniforms, temperature, vocab, qo, batch, total_nodes,
                                path_cap, accept_len, path, out_tokens, flags, ws, status, stream, nullptr,
                                host_logits);
    if (e != SPEC_OK) return e;
    return launch_kv_commit(ca.elem_bytes, ca.k_tree, ca.v_tree, path, path_cap, accept_len, qo, ca.page_table,
                            ca.max_pages, ca.num_pages, ca.page_size, ca.prefix_len, ca.seq_len_out, ca.k_pool,
                            ca.v_pool, batch, ca.hkv, ca.d, status, stream, ca.ins);
  }
  const int chunks = accept_chunks(total_nodes, vocab);
  const AcceptWs w = AcceptWs::make(batch, total_nodes, chunks);
  uint8_t* wb = static_cast<uint8_t*>(ws);
  unsigned* counter = reinterpret_cast<unsigned*>(wb + w.counter);
  if (mode == SPEC_GREEDY) {
    // the partials (8 bytes per 4096-logit task) when the rows pass the slots
    ArgPartial* part = reinterpret_cast<ArgPartial*>(wb + w.partials);
    int* am = reinterpret_cast<int*>(wb + w.results);
    const int gch = greedy_chunks(vocab);
    const int tasks = total_nodes * gch;
    static PerDevice per_sm[4], sm_n;
    // (the token insert is a separate instance: calls without a token buffer run code that
    // carries none of it, which keeps the streaming kernel's registers as they were)
    const bool ins = ca.ins.token_buf != nullptr;
    auto kern = vec ? (ins ? accept_greedy_kernel<true, true> : accept_greedy_kernel<true, false>)
                    : (ins ? accept_greedy_kernel<false, true> : accept_greedy_kernel<false, false>);
    const int occ = per_device(per_sm[(vec ? 1 : 0) + (ins ? 2 : 0)], [kern](int) {
      int o = 0;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, kAcceptThreads, 0) == cudaSuccess && o > 0 ? o
                                                                                                               : 1;
    });
    const int sms = per_device(sm_n, [](int dev) {
      int v = 0;
      return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0 ? v : 0;
    });
    if (occ == 0 || sms == 0) return SPEC_ERR_CUDA;
    // one wave with the same number of CTAs on every SM: tasks go round-robin to the CTAs, so
    // each SM's share differs from another's by at most one task per CTA it holds (a grid that
    // is not a multiple of the SM count leaves some SMs with one CTA -- and its tasks -- more)
    const int ctas_sm = occ < ceil_div(tasks, sms) ? occ : ceil_div(tasks, sms);
    const int grid_n = ctas_sm * sms;
    if (launch_pdl(kern, dim3((unsigned)grid_n), dim3(kAcceptThreads), 0, stream, tl, vocab, gch, tasks, qo, batch,
                   total_nodes, parent, tokens, path_cap, accept_len, path, out_tokens, flags, counter,
                   total_nodes <= kArgSlots ? reinterpret_cast<unsigned long long*>(wb + w.slots) : nullptr, part, am,
                   status, ca) != cudaSuccess)
      return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  // dynamic shared memory of the walk: each CTA's slice of p and q (when it fits)
  const size_t walk_smem = 2 * sizeof(float) * (size_t)walk_stage_floats(vocab);  // (p, then q)
  static PerDevice walk_attr;  // the raised shared-memory limit, set once per device
  if (per_device(walk_attr, [](int) {
        return cudaFuncSetAttribute(accept_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(2 * sizeof(float) * kWalkStage)) == cudaSuccess
                   ? 1
                   : 0;
      }) == 0)
    return SPEC_ERR_CUDA;
  if (launch_pdl(accept_walk_kernel, dim3(kWalkCluster, batch), dim3(kWalkThreads), walk_smem, stream, parent,
                 tokens, tl, dl, uniforms, temperature, vocab, qo, path_cap, accept_len, path, out_tokens, flags,
                 status, vec) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (ca.k_tree == nullptr) return SPEC_OK;
  return launch_kv_commit(ca.elem_bytes, ca.k_tree, ca.v_tree, path, path_cap, accept_len, qo, ca.page_table,
                          ca.max_pages, ca.num_pages, ca.page_size, ca.prefix_len, ca.seq_len_out, ca.k_pool,
                          ca.v_pool, batch, ca.hkv, ca.d, status, stream, ca.ins);
}

}  // namespace specv

// ------------------------------------------------------------------------------------
// Acceptance without caller-provided scratch.
//
// Some callers cannot allocate device memory at all: a runtime that hands out only the
// tensors it owns, a plugin host with no allocator of its own, a serving loop that
// forbids allocation once it is running. For them spec_accept_noalloc (api.cu) runs the
// same kernels as spec_accept with its scratch (counters, chunk partials, per-node
// results) in the file-scope array below, of fixed size kNoAllocScratchBytes. Every GPU
// that loads the library holds that array until the process exits.
namespace specv {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_accept_scratch[kNoAllocScratchBytes];

// Device address of g_accept_scratch for the current device. The symbol's host-side
// name is only a stand-in, so the address is asked of the runtime, once per device,
// with that device current (the answer stays valid until the device's context is
// destroyed, e.g. by cudaDeviceReset). Returns nullptr when the lookup fails.
static void* noalloc_scratch() {
  static void* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

// The fixed scratch as the workspace of an acceptance call of these sizes: SPEC_ERR_WORKSPACE
// when they need more than it holds, SPEC_ERR_CUDA when its address cannot be had. Its
// counters and argmax slots are zeroed on `stream` (the array keeps the previous call's
// contents), so the kernels find them as a fresh workspace would have them.
int accept_noalloc_scratch(int batch, int total_nodes, int vocab, cudaStream_t stream, void** ws) {
  const AcceptWs w = AcceptWs::make(batch, total_nodes, accept_chunks(total_nodes, vocab));
  if (w.total > kNoAllocScratchBytes) return SPEC_ERR_WORKSPACE;
  void* p = noalloc_scratch();
  if (p == nullptr) return SPEC_ERR_CUDA;
  if (cudaMemsetAsync(p, 0, w.partials, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  *ws = p;
  return SPEC_OK;
}

}  // namespace specv
