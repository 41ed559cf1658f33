// C ABI of libspecverify: argument checks on the host, then kernel dispatch.
// Every entry point is asynchronous on the caller's stream and allocates nothing.
#include <atomic>

#include "attn_common.cuh"
#include "draft_tree.cuh"

namespace specv {
bool greedy_walks(int batch, int total_nodes, int vocab, int path_cap, int sms);
int launch_tree_mask(const int32_t* parent, const int32_t* qo, int batch, int total_nodes, int max_nodes,
                     uint64_t* mask, int32_t* depth, int32_t* status, cudaStream_t stream);
int launch_kv_commit(int elem_bytes, const void* k_tree, const void* v_tree, const int32_t* path, int path_cap,
                     const int32_t* accept_len, const int32_t* qo, const int32_t* page_table, int max_pages,
                     int num_pages, int page_size, const int32_t* prefix_len, int32_t* seq_len_out, void* k_pool,
                     void* v_pool, int batch, int hkv, int d, int32_t* status, cudaStream_t stream, TokenInsert ins,
                     const float* kv_scale);
int launch_accept(int mode, const int32_t* parent, const int32_t* tokens, const float* tl, const float* dl,
                  const float* uniforms, float temperature, int vocab, const int32_t* qo, int batch,
                  int total_nodes, int path_cap, int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                  uint8_t* flags, void* ws, int32_t* status, cudaStream_t stream, const CommitArgs* commit,
                  bool host_logits);
size_t accept_ws_bytes(int batch, int total_nodes, int vocab);
int accept_noalloc_scratch(int batch, int total_nodes, int vocab, cudaStream_t stream, void** ws);
int launch_attn_simt(int dtype, const void* q, const void* k_pool, const void* v_pool, int num_pages, int ps,
                     const int32_t* page_table, int max_pages, const int32_t* prefix_len, int max_prefix,
                     const void* k_tree, const void* v_tree, const uint64_t* mask, const int32_t* qo, int batch,
                     int total_nodes, int max_nodes, int hq, int hkv, int d, float sm_scale, void* out, float* lse,
                     void* ws, int32_t* status, cudaStream_t stream);
bool attn_tc_shape(int dtype, int hq, int hkv, int d, int page_size, int max_nodes);
bool attn_tc_ready();
size_t attn_tc_ws_bytes(int batch, int max_nodes, int hq, int hkv, int max_prefix);
int launch_attn_tc(const void* q, const void* k_pool, const void* v_pool, int num_pages, int ps,
                   const int32_t* page_table, int max_pages, const int32_t* prefix_len, int max_prefix,
                   const void* k_tree, const void* v_tree, const uint64_t* mask, const int32_t* qo, int batch,
                   int total_nodes, int max_nodes, int hq, int hkv, int d, float sm_scale, void* out, float* lse,
                   void* ws, int32_t* status, cudaStream_t stream, const float* kv_scale, const int32_t* parent);

constexpr int kMaxNodes = kMaxTreeNodes;

static size_t attn_ws_bytes(int batch, int total_nodes, int max_nodes, int hq, int hkv, int d, int max_prefix) {
  const int rows = total_nodes * hq;
  const int s1 = attn_splits_simt(batch, max_nodes, hq, hkv, max_prefix);
  const size_t b1 = s1 > 1 ? AttnWs::bytes(s1, rows, d) : 0;
  const size_t b2 = d == 128 ? attn_tc_ws_bytes(batch, max_nodes, hq, hkv, max_prefix) : 0;
  return b1 > b2 ? b1 : b2;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// bf16 inputs with head dim 128 run on the tensor-core kernel and nowhere else; the
// CUDA-core kernel serves fp32 inputs and head dim 64.
static bool attn_wants_tc(int dtype, int d) { return dtype == SPEC_BF16 && d == 128; }
// Grids put (sequence, KV head) pairs, or sequences, on a launch's y or z dimension.
static bool grid_fits(long n) { return n <= kMaxGridYZ; }

static std::atomic<int> g_early_reads{0};
bool early_reads() { return g_early_reads.load(std::memory_order_relaxed) != 0; }

}  // namespace specv

using namespace specv;

extern "C" {

int spec_version(void) { return 112; }

int spec_set_early_reads(int enable) { return g_early_reads.exchange(enable ? 1 : 0); }

const char* spec_status_string(int status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_ARG: return "invalid argument (null pointer or bad size)";
    case SPEC_ERR_PARENT: return "parent array is not a tree (root must be -1, 0 <= parent[i] < i)";
    case SPEC_ERR_PAGE: return "page table entry outside the KV pool";
    case SPEC_ERR_CAPACITY: return "capacity exceeded (nodes, pages or path slots)";
    case SPEC_ERR_WORKSPACE: return "workspace smaller than spec_workspace_size()";
    case SPEC_ERR_UNSUPPORTED: return "unsupported dtype / head dim / shape";
    case SPEC_ERR_CUDA: return "CUDA runtime or launch error";
    case SPEC_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
    case SPEC_ERR_INDEX: return "token or node index out of range";
    default: return "unknown status";
  }
}

size_t spec_workspace_size(int op, int batch, int total_nodes, int max_nodes, int hq, int hkv, int d,
                           int max_prefix, int vocab) {
  if (batch < 0 || total_nodes < 0) return 0;
  switch (op) {
    case SPEC_OP_ATTN:
      if (hq <= 0 || hkv <= 0 || hq % hkv || d <= 0 || max_nodes <= 0 || max_prefix < 0) return 0;
      return attn_ws_bytes(batch, total_nodes, max_nodes, hq, hkv, d, max_prefix);
    case SPEC_OP_ACCEPT:
      if (vocab <= 0) return 0;
      return accept_ws_bytes(batch, total_nodes, vocab);
    case SPEC_OP_TREE:
      if (max_nodes < 1 || max_nodes > kMaxNodes) return 0;
      return tree_state_bytes(batch, max_nodes);
    default:
      return 0;
  }
}

int spec_attn_plan(int dtype, int batch, int max_nodes, int hq, int hkv, int d, int page_size, int max_prefix,
                   int* splits, int* tensor_cores) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (batch < 0 || max_nodes < 1 || max_nodes > kMaxNodes || max_prefix < 0 || hq <= 0 || hkv <= 0 ||
      hq % hkv != 0 || !splits || !tensor_cores)
    return SPEC_ERR_ARG;
  if (d != 64 && d != 128) return SPEC_ERR_UNSUPPORTED;
  if (page_size <= 0 || page_size % 8 != 0) return SPEC_ERR_UNSUPPORTED;
  if (!grid_fits((long)batch * hkv)) return SPEC_ERR_UNSUPPORTED;
  const bool tc = attn_wants_tc(dtype, d);
  if (tc && !attn_tc_shape(dtype, hq, hkv, d, page_size, max_nodes)) return SPEC_ERR_UNSUPPORTED;
  *tensor_cores = tc ? 1 : 0;
  *splits = tc ? attn_splits_tc(batch, max_nodes, hq, hkv, max_prefix)
               : attn_splits_simt(batch, max_nodes, hq, hkv, max_prefix);
  return SPEC_OK;
}

int spec_accept_plan(int mode, int batch, int total_nodes, int vocab, int path_cap, int sm_count, int* walk) {
  if (mode != SPEC_GREEDY && mode != SPEC_STOCHASTIC) return SPEC_ERR_ARG;
  if (batch < 0 || total_nodes < batch || vocab <= 0 || path_cap < 1 || sm_count < 0 || !walk) return SPEC_ERR_ARG;
  if (mode == SPEC_STOCHASTIC) {
    *walk = 1;
    return SPEC_OK;
  }
  int sms = sm_count;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return SPEC_ERR_CUDA;
  }
  *walk = (vocab % 4 == 0 && greedy_walks(batch, total_nodes, vocab, path_cap, sms)) ? 1 : 0;
  return SPEC_OK;
}

int spec_build_tree_mask(const int32_t* parent, const int32_t* qo_indptr, int batch, int total_nodes,
                         int max_nodes, uint64_t* mask, int32_t* depth, int32_t* dev_status, void* stream) {
  if (batch < 0 || total_nodes < 0 || max_nodes < 1 || max_nodes > kMaxNodes) return SPEC_ERR_ARG;
  if (batch == 0 || total_nodes == 0) return SPEC_OK;
  if (!parent || !qo_indptr || !mask) return SPEC_ERR_ARG;
  return launch_tree_mask(parent, qo_indptr, batch, total_nodes, max_nodes, mask, depth, dev_status,
                          static_cast<cudaStream_t>(stream));
}

int spec_tree_verify_attn(int dtype, const void* q, const void* k_pool, const void* v_pool, int num_pages,
                          int page_size, const int32_t* page_table, int max_pages, const int32_t* prefix_len,
                          int max_prefix, const void* k_tree, const void* v_tree, const uint64_t* mask,
                          const int32_t* qo_indptr, int batch, int total_nodes, int max_nodes, int hq, int hkv,
                          int d, float sm_scale, void* out, float* lse, void* ws, size_t ws_bytes,
                          int32_t* dev_status, void* stream) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (batch < 0 || total_nodes < 0 || max_nodes < 1 || max_nodes > kMaxNodes || max_prefix < 0 ||
      num_pages < 0 || max_pages < 0)
    return SPEC_ERR_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return SPEC_ERR_ARG;
  if (d != 64 && d != 128) return SPEC_ERR_UNSUPPORTED;
  if (page_size <= 0 || page_size % 8 != 0) return SPEC_ERR_UNSUPPORTED;
  if (!grid_fits((long)batch * hkv)) return SPEC_ERR_UNSUPPORTED;
  const bool tc = attn_wants_tc(dtype, d);
  if (tc && !attn_tc_shape(dtype, hq, hkv, d, page_size, max_nodes)) return SPEC_ERR_UNSUPPORTED;
  if (batch == 0 || total_nodes == 0) return SPEC_OK;
  if (!q || !k_tree || !v_tree || !mask || !qo_indptr || !prefix_len || !out) return SPEC_ERR_ARG;
  if (max_prefix > 0 && (!k_pool || !v_pool || !page_table || max_pages <= 0 || num_pages <= 0))
    return SPEC_ERR_ARG;
  if ((long)max_pages * page_size < max_prefix) return SPEC_ERR_ARG;
  if (tc && (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(out) ||
             (max_prefix > 0 && (!aligned16(k_pool) || !aligned16(v_pool)))))
    return SPEC_ERR_ARG;  // TMA copies need 16-byte aligned tensors
  const size_t need = spec_workspace_size(SPEC_OP_ATTN, batch, total_nodes, max_nodes, hq, hkv, d, max_prefix, 0);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return SPEC_ERR_WORKSPACE;
  if (sm_scale <= 0.f) sm_scale = 1.0f / sqrtf((float)d);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (tc) {
    if (!attn_tc_ready()) return SPEC_ERR_CUDA;
    return launch_attn_tc(q, k_pool, v_pool, num_pages, page_size, page_table, max_pages, prefix_len, max_prefix,
                          k_tree, v_tree, mask, qo_indptr, batch, total_nodes, max_nodes, hq, hkv, d, sm_scale,
                          out, lse, ws, dev_status, st, nullptr, nullptr);
  }
  return launch_attn_simt(dtype, q, k_pool, v_pool, num_pages, page_size, page_table, max_pages, prefix_len,
                          max_prefix, k_tree, v_tree, mask, qo_indptr, batch, total_nodes, max_nodes, hq, hkv, d,
                          sm_scale, out, lse, ws, dev_status, st);
}

// Host checks of spec_accept's arguments other than the workspace (SPEC_OK when they pass);
// spec_accept_noalloc makes the same checks.
// Where logits live: device memory, or host memory the device reads at the same address
// (pinned by cudaHostAlloc or cudaHostRegister under unified addressing; on a Grace-Blackwell
// part the rows then cross NVLink-C2C as the kernels read them). Anything else -- pageable or
// unregistered host memory, or pinned memory the device sees at another address -- is refused,
// so no kernel is handed an address it cannot read.
static int logits_where(const void* p, bool* host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return SPEC_ERR_ARG;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *host = false;
    return SPEC_OK;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer == p) {
    *host = true;
    return SPEC_OK;
  }
  return SPEC_ERR_ARG;
}

static int check_accept_args(int mode, const int32_t* parent, const int32_t* draft_tokens,
                             const float* target_logits, const float* draft_logits, const float* uniforms,
                             float temperature, int vocab, const int32_t* qo_indptr, int batch, int total_nodes,
                             int max_nodes, int path_cap, const int32_t* accept_len, const int32_t* path,
                             const int32_t* out_tokens) {
  if (mode != SPEC_GREEDY && mode != SPEC_STOCHASTIC) return SPEC_ERR_ARG;
  if (batch < 0 || total_nodes < 0 || vocab <= 0 || path_cap < 1 || max_nodes < 1 || max_nodes > kMaxNodes)
    return SPEC_ERR_ARG;
  if (batch == 0) return SPEC_OK;
  if (total_nodes < batch) return SPEC_ERR_ARG;  // every sequence has at least its root
  if (!parent || !draft_tokens || !target_logits || !qo_indptr || !accept_len || !path || !out_tokens)
    return SPEC_ERR_ARG;
  if (mode == SPEC_STOCHASTIC && (!draft_logits || !uniforms || !(temperature > 0.f))) return SPEC_ERR_ARG;
  if (mode == SPEC_STOCHASTIC && !grid_fits(batch)) return SPEC_ERR_UNSUPPORTED;  // one cluster row each
  return SPEC_OK;
}

// The last host check of an acceptance call (after every other): where its logits live.
static int accept_logits_where(int mode, const float* target_logits, const float* draft_logits, bool* host) {
  bool ht = false, hd = false;
  int rc = logits_where(target_logits, &ht);
  if (rc == SPEC_OK && mode == SPEC_STOCHASTIC) rc = logits_where(draft_logits, &hd);
  *host = ht || hd;
  return rc;
}

// Host checks of spec_accept's arguments (SPEC_OK when they pass).
static int check_accept(int mode, const int32_t* parent, const int32_t* draft_tokens, const float* target_logits,
                        const float* draft_logits, const float* uniforms, float temperature, int vocab,
                        const int32_t* qo_indptr, int batch, int total_nodes, int max_nodes, int path_cap,
                        const int32_t* accept_len, const int32_t* path, const int32_t* out_tokens, const void* ws,
                        size_t ws_bytes) {
  const int rc = check_accept_args(mode, parent, draft_tokens, target_logits, draft_logits, uniforms, temperature,
                                   vocab, qo_indptr, batch, total_nodes, max_nodes, path_cap, accept_len, path,
                                   out_tokens);
  if (rc != SPEC_OK || batch == 0) return rc;
  const size_t need = spec_workspace_size(SPEC_OP_ACCEPT, batch, total_nodes, max_nodes, 0, 0, 0, 0, vocab);
  if (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255)) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
}

// Host checks of spec_kv_commit's arguments (SPEC_OK when they pass).
static int check_commit(int dtype, const void* k_tree, const void* v_tree, const int32_t* path, int path_cap,
                        const int32_t* accept_len, const int32_t* qo_indptr, const int32_t* page_table,
                        int max_pages, int num_pages, int page_size, const int32_t* prefix_len, const void* k_pool,
                        const void* v_pool, int batch, int total_nodes, int hkv, int d) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
  if (batch < 0 || total_nodes < 0 || path_cap < 1 || max_pages < 0 || num_pages < 0 || page_size <= 0 ||
      hkv <= 0 || d <= 0)
    return SPEC_ERR_ARG;
  const int elem = dtype == SPEC_F32 ? 4 : 2;
  if ((d * elem) % 16 != 0) return SPEC_ERR_UNSUPPORTED;
  if (batch == 0) return SPEC_OK;
  if (!k_tree || !v_tree || !path || !accept_len || !qo_indptr || !page_table || !prefix_len || !k_pool || !v_pool)
    return SPEC_ERR_ARG;
  if (!aligned16(k_tree) || !aligned16(v_tree) || !aligned16(k_pool) || !aligned16(v_pool)) return SPEC_ERR_ARG;
  return SPEC_OK;
}

int spec_accept(int mode, const int32_t* parent, const int32_t* draft_tokens, const float* target_logits,
                const float* draft_logits, const float* uniforms, float temperature, int vocab,
                const int32_t* qo_indptr, int batch, int total_nodes, int max_nodes, int path_cap,
                int32_t* accept_len, int32_t* path, int32_t* out_tokens, uint8_t* flags, void* ws,
                size_t ws_bytes, int32_t* dev_status, void* stream) {
  bool host = false;
  int rc = check_accept(mode, parent, draft_tokens, target_logits, draft_logits, uniforms, temperature, vocab,
                        qo_indptr, batch, total_nodes, max_nodes, path_cap, accept_len, path, out_tokens, ws,
                        ws_bytes);
  if (rc != SPEC_OK || batch == 0) return rc;
  rc = accept_logits_where(mode, target_logits, draft_logits, &host);
  if (rc != SPEC_OK) return rc;
  return launch_accept(mode, parent, draft_tokens, target_logits, draft_logits, uniforms, temperature, vocab,
                       qo_indptr, batch, total_nodes, path_cap, accept_len, path, out_tokens, flags, ws,
                       dev_status, static_cast<cudaStream_t>(stream), nullptr, host);
}

int spec_accept_noalloc(int mode, const int32_t* parent, const int32_t* draft_tokens, const float* target_logits,
                        const float* draft_logits, const float* uniforms, float temperature, int vocab,
                        const int32_t* qo_indptr, int batch, int total_nodes, int max_nodes, int path_cap,
                        int32_t* accept_len, int32_t* path, int32_t* out_tokens, uint8_t* flags,
                        int32_t* dev_status, void* stream) {
  bool host = false;
  int rc = check_accept_args(mode, parent, draft_tokens, target_logits, draft_logits, uniforms, temperature, vocab,
                             qo_indptr, batch, total_nodes, max_nodes, path_cap, accept_len, path, out_tokens);
  if (rc != SPEC_OK || batch == 0) return rc;
  rc = accept_logits_where(mode, target_logits, draft_logits, &host);
  if (rc != SPEC_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  rc = accept_noalloc_scratch(batch, total_nodes, vocab, st, &ws);
  if (rc != SPEC_OK) return rc;
  return launch_accept(mode, parent, draft_tokens, target_logits, draft_logits, uniforms, temperature, vocab,
                       qo_indptr, batch, total_nodes, path_cap, accept_len, path, out_tokens, flags, ws,
                       dev_status, st, nullptr, host);
}

int spec_accept_commit(int mode, const int32_t* parent, const int32_t* draft_tokens, const float* target_logits,
                       const float* draft_logits, const float* uniforms, float temperature, int vocab,
                       const int32_t* qo_indptr, int batch, int total_nodes, int max_nodes, int path_cap,
                       int32_t* accept_len, int32_t* path, int32_t* out_tokens, uint8_t* flags, int dtype,
                       const void* k_tree, const void* v_tree, const int32_t* page_table, int max_pages,
                       int num_pages, int page_size, const int32_t* prefix_len, int32_t* seq_len_out, void* k_pool,
                       void* v_pool, int hkv, int d, int32_t* token_buf, int token_stride, void* ws,
                       size_t ws_bytes, int32_t* dev_status, void* stream) {
  bool host = false;
  int rc = check_accept(mode, parent, draft_tokens, target_logits, draft_logits, uniforms, temperature, vocab,
                        qo_indptr, batch, total_nodes, max_nodes, path_cap, accept_len, path, out_tokens, ws, ws_bytes);
  if (rc != SPEC_OK) return rc;
  rc = check_commit(dtype, k_tree, v_tree, path, path_cap, accept_len, qo_indptr, page_table, max_pages, num_pages,
                    page_size, prefix_len, k_pool, v_pool, batch, total_nodes, hkv, d);
  if (rc != SPEC_OK || batch == 0) return rc;
  if (token_buf != nullptr && token_stride < 1) return SPEC_ERR_ARG;
  rc = accept_logits_where(mode, target_logits, draft_logits, &host);
  if (rc != SPEC_OK) return rc;
  CommitArgs ca;
  ca.k_tree = static_cast<const uint8_t*>(k_tree);
  ca.v_tree = static_cast<const uint8_t*>(v_tree);
  ca.page_table = page_table;
  ca.max_pages = max_pages;
  ca.num_pages = num_pages;
  ca.page_size = page_size;
  ca.prefix_len = prefix_len;
  ca.seq_len_out = seq_len_out;
  ca.k_pool = static_cast<uint8_t*>(k_pool);
  ca.v_pool = static_cast<uint8_t*>(v_pool);
  ca.hkv = hkv;
  ca.d = d;
  ca.elem_bytes = dtype == SPEC_F32 ? 4 : 2;
  ca.ins = TokenInsert{out_tokens, token_buf, token_stride};
  return launch_accept(mode, parent, draft_tokens, target_logits, draft_logits, uniforms, temperature, vocab,
                       qo_indptr, batch, total_nodes, path_cap, accept_len, path, out_tokens, flags, ws,
                       dev_status, static_cast<cudaStream_t>(stream), &ca, host);
}

int spec_kv_commit(int dtype, const void* k_tree, const void* v_tree, const int32_t* path, int path_cap,
                   const int32_t* accept_len, const int32_t* qo_indptr, const int32_t* page_table, int max_pages,
                   int num_pages, int page_size, const int32_t* prefix_len, int32_t* seq_len_out, void* k_pool,
                   void* v_pool, int batch, int total_nodes, int hkv, int d, int32_t* dev_status, void* stream) {
  const int rc = check_commit(dtype, k_tree, v_tree, path, path_cap, accept_len, qo_indptr, page_table, max_pages,
                              num_pages, page_size, prefix_len, k_pool, v_pool, batch, total_nodes, hkv, d);
  if (rc != SPEC_OK || batch == 0) return rc;
  const int elem = dtype == SPEC_F32 ? 4 : 2;
  return launch_kv_commit(elem, k_tree, v_tree, path, path_cap, accept_len, qo_indptr, page_table, max_pages,
                          num_pages, page_size, prefix_len, seq_len_out, k_pool, v_pool, batch, hkv, d, dev_status,
                          static_cast<cudaStream_t>(stream), TokenInsert{nullptr, nullptr, 0}, nullptr);
}

int spec_tree_verify_attn_kv8(const void* q, const uint8_t* k_pool, const uint8_t* v_pool, const float* kv_scale,
                              int num_pages, int page_size, const int32_t* page_table, int max_pages,
                              const int32_t* prefix_len, int max_prefix, const void* k_tree, const void* v_tree,
                              const uint64_t* mask, const int32_t* qo_indptr, int batch, int total_nodes,
                              int max_nodes, int hq, int hkv, int d, float sm_scale, void* out, float* lse, void* ws,
                              size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (batch < 0 || total_nodes < 0 || max_nodes < 1 || max_nodes > kMaxNodes || max_prefix < 0 ||
      num_pages < 0 || max_pages < 0)
    return SPEC_ERR_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return SPEC_ERR_ARG;
  if (!attn_tc_shape(SPEC_BF16, hq, hkv, d, page_size, max_nodes)) return SPEC_ERR_UNSUPPORTED;
  if (!grid_fits((long)batch * hkv)) return SPEC_ERR_UNSUPPORTED;
  if (batch == 0 || total_nodes == 0) return SPEC_OK;
  if (!q || !k_tree || !v_tree || !mask || !qo_indptr || !prefix_len || !out || !kv_scale) return SPEC_ERR_ARG;
  if (max_prefix > 0 && (!k_pool || !v_pool || !page_table || max_pages <= 0 || num_pages <= 0))
    return SPEC_ERR_ARG;
  if ((long)max_pages * page_size < max_prefix) return SPEC_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(out) ||
      (max_prefix > 0 && (!aligned16(k_pool) || !aligned16(v_pool))))
    return SPEC_ERR_ARG;
  const size_t need = spec_workspace_size(SPEC_OP_ATTN, batch, total_nodes, max_nodes, hq, hkv, d, max_prefix, 0);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return SPEC_ERR_WORKSPACE;
  if (sm_scale <= 0.f) sm_scale = 1.0f / sqrtf((float)d);
  if (!attn_tc_ready()) return SPEC_ERR_CUDA;
  return launch_attn_tc(q, k_pool, v_pool, num_pages, page_size, page_table, max_pages, prefix_len, max_prefix,
                        k_tree, v_tree, mask, qo_indptr, batch, total_nodes, max_nodes, hq, hkv, d, sm_scale, out,
                        lse, ws, dev_status, static_cast<cudaStream_t>(stream), kv_scale, nullptr);
}

int spec_tree_verify_attn_parents(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                                  int page_size, const int32_t* page_table, int max_pages,
                                  const int32_t* prefix_len, int max_prefix, const void* k_tree,
                                  const void* v_tree, const int32_t* parent, const int32_t* qo_indptr, int batch,
                                  int total_nodes, int max_nodes, int hq, int hkv, int d, float sm_scale,
                                  void* out, float* lse, void* ws, size_t ws_bytes, int32_t* dev_status,
                                  void* stream) {
  if (batch < 0 || total_nodes < 0 || max_nodes < 1 || max_nodes > kMaxNodes || max_prefix < 0 ||
      num_pages < 0 || max_pages < 0)
    return SPEC_ERR_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return SPEC_ERR_ARG;
  if (!attn_tc_shape(SPEC_BF16, hq, hkv, d, page_size, max_nodes)) return SPEC_ERR_UNSUPPORTED;
  if (!grid_fits((long)batch * hkv)) return SPEC_ERR_UNSUPPORTED;
  if (batch == 0 || total_nodes == 0) return SPEC_OK;
  if (!q || !k_tree || !v_tree || !parent || !qo_indptr || !prefix_len || !out) return SPEC_ERR_ARG;
  if (max_prefix > 0 && (!k_pool || !v_pool || !page_table || max_pages <= 0 || num_pages <= 0))
    return SPEC_ERR_ARG;
  if ((long)max_pages * page_size < max_prefix) return SPEC_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_tree) || !aligned16(v_tree) || !aligned16(out) ||
      (max_prefix > 0 && (!aligned16(k_pool) || !aligned16(v_pool))))
    return SPEC_ERR_ARG;
  const size_t need = spec_workspace_size(SPEC_OP_ATTN, batch, total_nodes, max_nodes, hq, hkv, d, max_prefix, 0);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return SPEC_ERR_WORKSPACE;
  if (sm_scale <= 0.f) sm_scale = 1.0f / sqrtf((float)d);
  if (!attn_tc_ready()) return SPEC_ERR_CUDA;
  return launch_attn_tc(q, k_pool, v_pool, num_pages, page_size, page_table, max_pages, prefix_len, max_prefix,
                        k_tree, v_tree, nullptr, qo_indptr, batch, total_nodes, max_nodes, hq, hkv, d, sm_scale, out,
                        lse, ws, dev_status, static_cast<cudaStream_t>(stream), nullptr, parent);
}

int spec_kv_commit_kv8(const void* k_tree, const void* v_tree, const float* kv_scale, const int32_t* path,
                       int path_cap, const int32_t* accept_len, const int32_t* qo_indptr, const int32_t* page_table,
                       int max_pages, int num_pages, int page_size, const int32_t* prefix_len, int32_t* seq_len_out,
                       uint8_t* k_pool, uint8_t* v_pool, int batch, int total_nodes, int hkv, int d,
                       int32_t* dev_status, void* stream) {
  // the tree rows are bf16 (d * 2 bytes), the pool rows d codes: d a multiple of 16
  const int rc = check_commit(SPEC_BF16, k_tree, v_tree, path, path_cap, accept_len, qo_indptr, page_table,
                              max_pages, num_pages, page_size, prefix_len, k_pool, v_pool, batch, total_nodes, hkv, d);
  if (rc != SPEC_OK || batch == 0) return rc;
  if (d % 16 != 0) return SPEC_ERR_UNSUPPORTED;
  if (!kv_scale) return SPEC_ERR_ARG;
  return launch_kv_commit(2, k_tree, v_tree, path, path_cap, accept_len, qo_indptr, page_table, max_pages, num_pages,
                          page_size, prefix_len, seq_len_out, k_pool, v_pool, batch, hkv, d, dev_status,
                          static_cast<cudaStream_t>(stream), TokenInsert{nullptr, nullptr, 0}, kv_scale);
}


int spec_tree_init(const int32_t* root_tokens, int batch, int max_nodes, void* state, size_t state_bytes,
                   int32_t* parent_out, int32_t* tokens_out, int32_t* n_nodes_out, int32_t* next_node,
                   uint8_t* flags, void* stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > kMaxNodes) return SPEC_ERR_ARG;
  if (!grid_fits(batch)) return SPEC_ERR_UNSUPPORTED;
  if (batch == 0) return SPEC_OK;
  if (!root_tokens || !state || !parent_out || !tokens_out || !n_nodes_out || !next_node) return SPEC_ERR_ARG;
  if (state_bytes < tree_state_bytes(batch, max_nodes)) return SPEC_ERR_WORKSPACE;
  TreeArgs a{static_cast<uint8_t*>(state), max_nodes, 1, 1, 0.0, parent_out, tokens_out, n_nodes_out, next_node,
             flags, nullptr, 1, nullptr, nullptr, nullptr};
  return launch_tree_init(root_tokens, batch, a, static_cast<cudaStream_t>(stream));
}

int spec_tree_expand(const float* draft_logits, int vocab, long long row_stride, long long node_stride, int batch,
                     int max_nodes, int topk, int max_depth, double threshold, void* state, size_t state_bytes,
                     int32_t* parent_out, int32_t* tokens_out, int32_t* n_nodes_out, int32_t* next_node,
                     uint8_t* flags, int32_t* dev_status, void* stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > kMaxNodes || vocab < 1 || topk < 1 || topk > 16 ||
      max_depth < 1 || row_stride < 0 || node_stride < 0)
    return SPEC_ERR_ARG;
  if (!grid_fits(batch)) return SPEC_ERR_UNSUPPORTED;
  if (batch == 0) return SPEC_OK;
  if (!draft_logits || !state || !parent_out || !tokens_out || !n_nodes_out || !next_node) return SPEC_ERR_ARG;
  if (state_bytes < tree_state_bytes(batch, max_nodes)) return SPEC_ERR_WORKSPACE;
  TreeArgs a{static_cast<uint8_t*>(state), max_nodes, topk, max_depth, threshold, parent_out, tokens_out,
             n_nodes_out, next_node, flags, dev_status, 1, nullptr, nullptr, nullptr};
  return launch_tree_expand(draft_logits, vocab, (long)row_stride, (long)node_stride, batch, a,
                            static_cast<cudaStream_t>(stream));
}

int spec_tree_expand_multi(const float* draft_logits, int vocab, long long row_stride, long long req_stride,
                           int batch, int max_nodes, int width, int topk, int max_depth, double threshold,
                           void* state, size_t state_bytes, int32_t* parent_out, int32_t* tokens_out,
                           int32_t* n_nodes_out, int32_t* next_node, int32_t* req_parent, int32_t* req_token,
                           int32_t* req_n, uint8_t* flags, int32_t* dev_status, void* stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > kMaxNodes || vocab < 1 || topk < 1 || topk > 16 ||
      max_depth < 1 || width < 1 || width > kTreeMaxW || row_stride < 0 || req_stride < 0)
    return SPEC_ERR_ARG;
  if (!grid_fits(batch)) return SPEC_ERR_UNSUPPORTED;
  if (batch == 0) return SPEC_OK;
  if (!draft_logits || !state || !parent_out || !tokens_out || !n_nodes_out || !next_node || !req_parent ||
      !req_token || !req_n)
    return SPEC_ERR_ARG;
  if (state_bytes < tree_state_bytes(batch, max_nodes)) return SPEC_ERR_WORKSPACE;
  TreeArgs a{static_cast<uint8_t*>(state), max_nodes, topk, max_depth, threshold, parent_out, tokens_out,
             n_nodes_out, next_node, flags, dev_status, width, req_parent, req_token, req_n};
  return launch_tree_expand_multi(draft_logits, vocab, (long)row_stride, (long)req_stride, batch, a,
                                  static_cast<cudaStream_t>(stream));
}

}  // extern "C"
