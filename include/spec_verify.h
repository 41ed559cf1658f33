/*
 * spec_verify.h — C ABI of the tree-speculative-decoding verification path
 * (library: libspecverify.so, sm_103a / GB300).
 *
 * Four operations, in the order a verification step runs them:
 *
 *   spec_build_tree_mask   draft tree (parent array) -> ancestor bitmasks + depths
 *   spec_tree_verify_attn  one attention pass of every tree node over the paged
 *                          prefix and the tree's own K/V, ancestors only
 *   spec_accept            longest accepted path + bonus token (greedy / stochastic)
 *   spec_kv_commit         the accepted path's K/V written into the paged cache
 *
 * spec_accept_commit runs the last two as one call (the same results, one kernel
 * boundary fewer). spec_tree_verify_attn_parents runs the first two as one call (the mask
 * built inside the attention from the parent array). spec_tree_verify_attn_kv8 and
 * spec_kv_commit_kv8 are the attention and the commit over an FP8 (E4M3) paged cache;
 * spec_tree_init / spec_tree_expand (/ spec_tree_expand_multi) build the draft tree on
 * the device;
 * spec_accept_noalloc is spec_accept without a workspace argument.
 *
 * Sources of the operations (page title, then section):
 *   "EAGLE-2 deep dive" (techknowgenie): architecture section (all tree tokens
 *     verified in one target forward with a 2-D tree mask injected into
 *     attention; target logits contrasted with draft tokens; longest accepted
 *     path; the target KV cache must not be contaminated), core-implementation
 *     section (tree mask = node + ancestors up to the root; node ids in
 *     creation order), production section (paged tree attention indexing the
 *     mask over paged KV), benchmark section (rejection sampling, lossless).
 *   "Accelerating Sonar through speculation" (Perplexity): speculative-decoding
 *     section (n drafts -> up to n+1 tokens; the extra token from the target's
 *     logits at the stop position), draft-target section (acceptance compares
 *     full draft and target distributions; KV filled for accepted tokens),
 *     EAGLE section (a custom mask over the whole sequence slows attention by
 *     up to 50% — so the prefix here is never masked), MTP-schedule section (a
 *     kernel inserts the next token after the shift, no CPU-GPU sync — so
 *     every length stays on the device here).
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless stated otherwise; the caller owns
 *     every buffer. No call allocates, frees or synchronises with the host:
 *     each enqueues its kernels on `stream` (a cudaStream_t passed as void*,
 *     NULL = legacy default stream) and returns.
 *   - Layouts are row-major, C order. Tree node ids are sequence-local:
 *     sequence b owns global rows [qo_indptr[b], qo_indptr[b+1]) of every
 *     per-node array; its node i is global row qo_indptr[b] + i.
 *   - Errors the host can see (null pointer, bad size, unsupported shape,
 *     workspace too small) return a negative spec_status at once and enqueue
 *     nothing. Errors that depend on device data (bad parent, page id outside
 *     the pool, path longer than its buffer, timeout of a bounded wait) are
 *     written to *dev_status with first-error-wins semantics (the word is
 *     only changed while it holds SPEC_OK); the kernels then skip the bad
 *     item and finish cleanly — no trap, assert or unbounded wait. dev_status
 *     may be NULL (device errors are then not reported). The caller zeroes
 *     it when it wants a fresh report.
 *   - Workspace: `ws` is scratch of at least spec_workspace_size(...) bytes,
 *     256-byte aligned. It must be zero-filled before its first use with
 *     spec_accept (it keeps arrival counters there); every call leaves the
 *     counters it uses at zero again. One workspace must not serve two calls
 *     that may run concurrently.
 *   - Early start: the kernels are launched with programmatic stream
 *     serialization, so a call may begin while the kernel enqueued before it
 *     is still running. By default every kernel waits for that predecessor
 *     before it reads or writes anything (a predecessor's writes are visible
 *     only after that wait, whether or not it signals early). A caller whose
 *     preceding kernel writes none of the inputs listed below can let two
 *     kernels read them before the wait with spec_set_early_reads(1):
 *     spec_tree_verify_attn (and its _kv8 and _parents forms) then reads q,
 *     k_pool, v_pool, k_tree, v_tree, page_table, prefix_len, qo_indptr and
 *     kv_scale (everything but the mask or parent array) before it waits, and
 *     greedy spec_accept (and spec_accept_commit), when it walks from the root
 *     (spec_accept_plan), reads parent, draft_tokens, target_logits and
 *     qo_indptr before it waits (spec_accept_commit also the commit's k_tree,
 *     v_tree, page_table and prefix_len); both still wait before their first
 *     write.
 *     (In a target model's forward pass the kernel before the attention
 *     writes q and the tree's K/V, and the one before the acceptance writes
 *     the logits: keep the switch off there, or put an event between.) Of
 *     this library's kernels, the ones that signal early write only mask and
 *     depth (spec_build_tree_mask), out, lse and the workspace (the attention
 *     and its split merge) and the acceptance results (greedy spec_accept when
 *     it streams every row); the commit kernels and the acceptance walks,
 *     which may write the pool, never do.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_ARG = -1,         /* host: null pointer, negative or inconsistent size            */
  SPEC_ERR_PARENT = -2,      /* device: parent array is not a tree (root != -1, parent >= i) */
  SPEC_ERR_PAGE = -3,        /* device: page table entry outside [0, num_pages)              */
  SPEC_ERR_CAPACITY = -4,    /* device: a sequence needs more nodes/pages/path slots than given */
  SPEC_ERR_WORKSPACE = -5,   /* host: ws_bytes smaller than spec_workspace_size()            */
  SPEC_ERR_UNSUPPORTED = -6, /* host: dtype / head dim / group size not implemented, or a
                                batch past a launch's grid: batch x hkv > 65535 for the
                                attention calls, batch > 65535 for stochastic acceptance
                                and the draft-tree calls                                      */
  SPEC_ERR_CUDA = -7,        /* host: a CUDA runtime call or kernel launch failed            */
  SPEC_ERR_TIMEOUT = -8,     /* device: a bounded wait inside a kernel gave up               */
  SPEC_ERR_INDEX = -9        /* device: token id / path node id out of range                 */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;
typedef enum { SPEC_GREEDY = 0, SPEC_STOCHASTIC = 1 } spec_mode;
typedef enum { SPEC_OP_MASK = 0, SPEC_OP_ATTN = 1, SPEC_OP_ACCEPT = 2, SPEC_OP_COMMIT = 3,
               SPEC_OP_TREE = 4 } spec_op;

/* Bytes of workspace `op` needs for these sizes (0 when it needs none).
 * For SPEC_OP_ATTN the result depends on (batch, max_nodes, hq, hkv, d,
 * max_prefix, total_nodes); for SPEC_OP_ACCEPT on (batch, total_nodes, vocab); for
 * SPEC_OP_TREE (the draft-tree state of spec_tree_init / spec_tree_expand) on
 * (batch, max_nodes).
 * Unused arguments may be 0. Returns 0 for invalid sizes. */
size_t spec_workspace_size(int op, int batch, int total_nodes, int max_nodes, int hq, int hkv,
                           int d, int max_prefix, int vocab);

/* Launch plan spec_tree_verify_attn uses for these sizes (informational; the pages
 * have no counterpart): *splits = number of key splits (> 1 adds a merge kernel),
 * *tensor_cores = 1 when the tcgen05 kernel runs (every bf16 call with d = 128), 0 for
 * the CUDA-core kernel (fp32 inputs, or d = 64). Returns SPEC_OK or SPEC_ERR_ARG /
 * SPEC_ERR_UNSUPPORTED like the call would. */
int spec_attn_plan(int dtype, int batch, int max_nodes, int hq, int hkv, int d, int page_size,
                   int max_prefix, int* splits, int* tensor_cores);

/* Read plan spec_accept uses for these sizes (informational; the pages have no
 * counterpart): *walk = 1 when the call reads only the rows of the nodes its walk visits
 * (the root and each accepted node) -- always for SPEC_STOCHASTIC; for SPEC_GREEDY when a
 * model of the two ways (a walk from the root, one 8-CTA cluster per sequence, at most
 * path_cap rows each, against streaming every row at the copy rate) finds the walk
 * cheaper, which needs many rows per sequence -- and 0 when it streams every row (logits
 * in host memory always walk, whatever this says). The results are the same either way.
 * sm_count: the GPU's SMs (0: the current device's).
 * Assumes 16-byte aligned logits rows (the walk needs them). Returns SPEC_OK,
 * SPEC_ERR_ARG, or SPEC_ERR_CUDA when sm_count is 0 and no device answers. */
int spec_accept_plan(int mode, int batch, int total_nodes, int vocab, int path_cap, int sm_count, int* walk);

/* Whether the attention and the greedy walk may read their inputs before waiting for
 * the kernel enqueued just before them (the early-start rule above). enable != 0 turns
 * it on for the whole process, 0 (the default) off; each later call reads the setting
 * when it is made (a captured CUDA graph keeps the setting it was captured with).
 * Thread-safe. Results do not depend on it. Returns the previous setting (0 or 1). */
int spec_set_early_reads(int enable);

/* Static, NUL-terminated description of a spec_status value. */
const char* spec_status_string(int status);

/* Library version as an integer (major * 10000 + minor * 100 + patch). */
int spec_version(void);

/*
 * spec_build_tree_mask — ancestor bitmask of every draft-tree node.
 *   ("EAGLE-2 deep dive", core-implementation section: a node's row of the tree
 *   mask marks the node itself and every ancestor, walking parent links to the
 *   root; nodes are numbered after their parents.)
 *
 *   parent     int32 [total_nodes]  sequence-local parent id; the root (node 0 of
 *                                   each sequence) holds -1; node i > 0 needs
 *                                   0 <= parent[i] < i.
 *   qo_indptr  int32 [batch+1]      node ranges; qo_indptr[0] = 0, non-decreasing,
 *                                   qo_indptr[batch] = total_nodes.
 *   max_nodes  >= every sequence's node count; fixes the mask row width
 *              W = ceil(max_nodes / 64) words.
 *   mask       uint64 [total_nodes][W] (out)  bit (j & 63) of word (j >> 6) of row
 *              t = node j of t's sequence is t itself or an ancestor of t. Bits of
 *              node ids >= the sequence's node count are 0.
 *   depth      int32 [total_nodes] (out, nullable)  parent links to the root (root 0).
 *   Device errors: SPEC_ERR_PARENT (that row written all-zero, depth -1),
 *   SPEC_ERR_CAPACITY (sequence longer than max_nodes: its rows written all-zero,
 *   depth -1, so no earlier call's bits remain for a later attention to read).
 */
int spec_build_tree_mask(const int32_t* parent, const int32_t* qo_indptr, int batch,
                         int total_nodes, int max_nodes, uint64_t* mask, int32_t* depth,
                         int32_t* dev_status, void* stream);

/*
 * spec_tree_verify_attn — tree-verify attention with GQA over a paged prefix.
 *   ("EAGLE-2 deep dive", architecture and production sections: one target
 *   forward over all tree tokens, 2-D tree mask inside attention, mask indexed
 *   over paged KV. "Accelerating Sonar", EAGLE section: a mask over the whole
 *   sequence costs up to 50% — here the prefix is never masked.)
 *
 *   For sequence b, node i, query head h (KV head g = h / (hq / hkv)):
 *     keys  = prefix slots 0 .. prefix_len[b]-1  (read through page_table)
 *             ++ tree nodes j of b with mask bit j of row i set
 *     out[t][h] = softmax(sm_scale * q[t][h] . K^T) V,  lse[t][h] = ln sum exp(scores)
 *
 *   dtype      SPEC_F32 or SPEC_BF16: element type of q, k_pool, v_pool, k_tree,
 *              v_tree and out (accumulation is fp32 in both cases).
 *   q          [total_nodes][hq][d]
 *   k_pool, v_pool  [num_pages][hkv][page_size][d]  the paged KV cache ("HND" pages)
 *   page_table int32 [batch][max_pages]  page id of logical page p of sequence b;
 *              entries past ceil(prefix_len[b] / page_size) are not read.
 *   prefix_len int32 [batch]   verified prefix length per sequence (>= 0).
 *   max_prefix >= every prefix_len[b]; used on the host to size the key split.
 *   k_tree, v_tree  [total_nodes][hkv][d]  K/V of the tree tokens themselves.
 *   mask       uint64 [total_nodes][ceil(max_nodes/64)]  from spec_build_tree_mask.
 *   qo_indptr  int32 [batch+1]; max_nodes >= every sequence's node count.
 *   hq % hkv == 0; d in {64, 128}; sm_scale <= 0 selects 1/sqrt(d).
 *   Kernels: bf16 with d = 128 runs on the tensor-core kernel and on nothing else. It
 *   needs page_size 16 and hq / hkv dividing 128 (else SPEC_ERR_UNSUPPORTED), q, k_pool,
 *   v_pool, k_tree, v_tree and out 16-byte aligned (else SPEC_ERR_ARG), and the driver's
 *   tensor-map encoder (else SPEC_ERR_CUDA). fp32 inputs, and d = 64, run on the
 *   CUDA-core kernel (page_size a multiple of 8).
 *   out        [total_nodes][hq][d] (out)
 *   lse        float [total_nodes][hq] (out, nullable)  natural-log log-sum-exp.
 *   ws         workspace of spec_workspace_size(SPEC_OP_ATTN, ...) bytes (key-split
 *              partial results; any contents).
 *   Device errors: SPEC_ERR_PAGE (page id outside [0, num_pages): the page is read
 *   as zeros), SPEC_ERR_TIMEOUT.
 */
int spec_tree_verify_attn(int dtype, const void* q, const void* k_pool, const void* v_pool,
                          int num_pages, int page_size, const int32_t* page_table, int max_pages,
                          const int32_t* prefix_len, int max_prefix, const void* k_tree,
                          const void* v_tree, const uint64_t* mask, const int32_t* qo_indptr,
                          int batch, int total_nodes, int max_nodes, int hq, int hkv, int d,
                          float sm_scale, void* out, float* lse, void* ws, size_t ws_bytes,
                          int32_t* dev_status, void* stream);

/*
 * spec_accept — longest accepted root-to-node path of each tree + the bonus token.
 *   Greedy ("EAGLE-2 deep dive", architecture section; "Accelerating Sonar",
 *   speculative-decoding section): a[v] = argmax of target_logits[v] (lowest
 *   token id on ties); from the root, move to the first child (lowest node id)
 *   whose draft token equals a[v]; stop when none does; bonus = a[stop node].
 *   Stochastic ("EAGLE-2 deep dive", benchmark section; "Accelerating Sonar",
 *   draft-target section; rule of the speculative-sampling works they cite):
 *   p_v = softmax(target_logits[v] / T), q_v = softmax(draft_logits[v] / T);
 *   at node v, r = p_v; each child c (increasing id, token x) is accepted iff
 *   uniforms[c][0] < r(x) / q_v(x); a rejection replaces r by
 *   max(r - q_v, 0) normalised; if no child is accepted the bonus is the
 *   inverse-CDF draw from r with uniforms[v][1].
 *   Rows read: both modes need the logits of the nodes the walk visits only (the
 *   root and each accepted node). Stochastic acceptance always reads just those;
 *   greedy acceptance either streams every row (one wave of CTAs, a last-CTA walk)
 *   or walks from the root reading just those, whichever spec_accept_plan's model
 *   finds cheaper for the sizes. The results are the same either way.
 *
 *   parent, draft_tokens  int32 [total_nodes]  (root's token = last accepted token)
 *   target_logits  float [total_nodes][vocab]
 *   draft_logits   float [total_nodes][vocab]  (stochastic only; NULL for greedy)
 *                  Either may sit in device memory or in pinned host memory the
 *                  device reads at the same address (cudaHostAlloc, or
 *                  cudaHostRegister, under unified addressing). From host memory
 *                  only the visited rows cross the host link (NVLink-C2C on a
 *                  Grace-Blackwell part): greedy acceptance then always walks from
 *                  the root. Any other pointer (pageable host memory, pinned
 *                  memory mapped elsewhere) returns SPEC_ERR_ARG.
 *   uniforms       float [total_nodes][2]      (stochastic only) (u_accept, u_bonus) in [0,1)
 *   temperature    > 0 (stochastic only)
 *   path_cap       row length of path / out_tokens (>= deepest accepted path + 1; the
 *                  trees' depth + 1 always suffices). It also bounds the greedy walk's
 *                  rows per sequence in spec_accept_plan's model.
 *   accept_len int32 [batch] (out)  L = accepted draft nodes (root excluded).
 *   path       int32 [batch][path_cap] (out)  root (0) then the accepted node ids; -1 after.
 *   out_tokens int32 [batch][path_cap] (out)  the L accepted tokens, then the bonus; -1 after.
 *   flags      uint8 [batch] (out, nullable)  stochastic near-ties seen by the GPU:
 *              bit 0 a ratio test with |u - ratio| <= 1e-6, bit 1 a bonus draw within
 *              1e-8 (relative to the residual's total) of a CDF boundary. Greedy writes 0.
 *   ws         workspace of spec_workspace_size(SPEC_OP_ACCEPT, ...) bytes, zeroed
 *              before first use (see the conventions above).
 *   Device errors: SPEC_ERR_PARENT, SPEC_ERR_INDEX (draft token outside [0, vocab)),
 *   SPEC_ERR_CAPACITY (accepted path longer than path_cap - 1: truncated).
 */
int spec_accept(int mode, const int32_t* parent, const int32_t* draft_tokens,
                const float* target_logits, const float* draft_logits, const float* uniforms,
                float temperature, int vocab, const int32_t* qo_indptr, int batch,
                int total_nodes, int max_nodes, int path_cap, int32_t* accept_len, int32_t* path,
                int32_t* out_tokens, uint8_t* flags, void* ws, size_t ws_bytes,
                int32_t* dev_status, void* stream);

/*
 * spec_kv_commit — write the accepted path's K/V into each sequence's cache.
 *   ("EAGLE-2 deep dive", architecture section: verification must not
 *   contaminate the target KV cache; "Accelerating Sonar", draft-target and
 *   MTP-schedule sections: KV of accepted tokens is filled, the next token is
 *   placed after the shift on the device with no CPU sync.)
 *   For i = 0 .. accept_len[b]: tree row qo_indptr[b] + path[b][i] (all hkv heads)
 *   is copied to logical slot prefix_len[b] + i of sequence b (page
 *   page_table[b][slot / page_size], row slot % page_size). Then
 *   seq_len_out[b] = prefix_len[b] + accept_len[b] + 1. accept_len and path are
 *   read on the device (straight from spec_accept), so no host sync is needed.
 *   The tree buffers must not alias the pool.
 *
 *   dtype       element type of k_tree, v_tree, k_pool, v_pool.
 *   k_tree, v_tree  [total_nodes][hkv][d];  k_pool, v_pool  [num_pages][hkv][page_size][d] (in/out)
 *   path        int32 [batch][path_cap];  accept_len int32 [batch]
 *   seq_len_out int32 [batch] (out, nullable)
 *   Device errors: SPEC_ERR_INDEX (path node outside the sequence's tree, or
 *   accept_len outside [0, path_cap)), SPEC_ERR_CAPACITY (slot beyond max_pages),
 *   SPEC_ERR_PAGE (page id outside the pool). A sequence with an error is
 *   left unwritten.
 */
int spec_kv_commit(int dtype, const void* k_tree, const void* v_tree, const int32_t* path,
                   int path_cap, const int32_t* accept_len, const int32_t* qo_indptr,
                   const int32_t* page_table, int max_pages, int num_pages, int page_size,
                   const int32_t* prefix_len, int32_t* seq_len_out, void* k_pool, void* v_pool,
                   int batch, int total_nodes, int hkv, int d, int32_t* dev_status, void* stream);

/*
 * spec_accept_commit — spec_accept, then spec_kv_commit of the paths it accepted, in one
 *   call: the results (accept_len, path, out_tokens, flags, the written pool rows,
 *   seq_len_out, device errors) are those of the two calls made back to back on
 *   `stream`. Greedy acceptance commits inside its own kernel where it can: walking from
 *   the root (spec_accept_plan), each sequence's cluster commits that sequence after its
 *   walk; streaming every row, the last CTA commits up to 4 sequences right after its
 *   walk. More sequences when streaming, and stochastic acceptance, launch the commit
 *   kernel after the acceptance kernels.
 *   Arguments: those of spec_accept (mode ... flags, ws, ws_bytes) and of spec_kv_commit
 *   (dtype ... d); path_cap, path and accept_len serve both. The same host errors, the
 *   same layouts; ws as for spec_accept.
 *   Next-step tokens on the device ("Accelerating Sonar", MTP-schedule section: a kernel
 *   places the next token after the shift, with no CPU-GPU sync):
 *   token_buf  int32 [batch][token_stride] (in/out, nullable)  each sequence's tokens by
 *              position, the root (the last accepted token) at prefix_len[b]. With every
 *              commit of sequence b the call also writes out_tokens[b][0 .. L] (the L
 *              accepted tokens, then the bonus token, the next step's root) to
 *              token_buf[b][P + 1 .. P + L + 1], P = prefix_len[b]; nothing else of the row
 *              changes. A row without room (P + L + 1 >= token_stride) is a device error
 *              SPEC_ERR_CAPACITY, and that sequence is left unwritten (K/V and tokens).
 *   token_stride  row length of token_buf (>= 1 when token_buf is given).
 */
int spec_accept_commit(int mode, const int32_t* parent, const int32_t* draft_tokens,
                       const float* target_logits, const float* draft_logits, const float* uniforms,
                       float temperature, int vocab, const int32_t* qo_indptr, int batch,
                       int total_nodes, int max_nodes, int path_cap, int32_t* accept_len,
                       int32_t* path, int32_t* out_tokens, uint8_t* flags, int dtype,
                       const void* k_tree, const void* v_tree, const int32_t* page_table,
                       int max_pages, int num_pages, int page_size, const int32_t* prefix_len,
                       int32_t* seq_len_out, void* k_pool, void* v_pool, int hkv, int d,
                       int32_t* token_buf, int token_stride, void* ws, size_t ws_bytes,
                       int32_t* dev_status, void* stream);

/*
 * spec_tree_init / spec_tree_expand -- the EAGLE-2 dynamic draft tree, built on the device.
 *   ("EAGLE-2 deep dive", section on the dynamic draft-tree algorithm: a node's confidence
 *   is the product of the draft probabilities along its path; a priority queue pops the
 *   best candidate as the next node; a node below the depth limit is expanded into its
 *   top-k tokens, scored by the product, those at or below a threshold dropped; the tree
 *   stops at the node budget.)
 *   The draft model is the caller's: between two spec_tree_expand calls it writes the
 *   logits row of each sequence's node awaiting expansion (next_node). A call reads that
 *   row, computes p = softmax(row) and the top-k tokens (largest logit first, lower token
 *   id on ties), pushes the k candidates with score = score(node) * p(token), then pops the
 *   best candidate (largest score, the earlier push on ties) as node n_nodes (its parent and
 *   token in parent_out / tokens_out); a popped node at the depth limit is not expanded and
 *   the next best is popped, until one needs its expansion or max_nodes nodes exist. Node
 *   ids therefore grow in pop order and parent[i] < i: parent_out / tokens_out feed
 *   spec_build_tree_mask and the verification calls directly (row b = sequence b).
 *
 *   spec_tree_init: root_tokens int32 [batch] (the last accepted token of each sequence);
 *     sets node 0 (parent -1, score 1), every other entry of parent_out / tokens_out to -1,
 *     n_nodes_out = 1 and next_node = 0 (the root awaits its expansion; -1 if max_nodes = 1).
 *   spec_tree_expand:
 *     draft_logits  float; the row of sequence b for node u starts at
 *                   draft_logits + b * row_stride + u * node_stride (elements). With the
 *                   draft model writing one row per sequence: row_stride = vocab,
 *                   node_stride = 0. Sequences whose next_node is -1 are skipped.
 *     topk in [1, 16]; max_depth >= 1 (a node of that depth is not expanded);
 *     threshold    candidates with score <= threshold are dropped (<= 0: none).
 *     state        spec_workspace_size(SPEC_OP_TREE, batch, 0, max_nodes, ...) bytes,
 *                  written by spec_tree_init; one state per tree under construction.
 *     parent_out, tokens_out  int32 [batch][max_nodes] (in/out);  n_nodes_out, next_node
 *                  int32 [batch] (out);  flags uint8 [batch] (out, nullable): bit 0 set
 *                  when a pop's best two scores were within a relative 1e-6 (the
 *                  probabilities are exp in fp32: such a pop could be ordered either way).
 *   Scores: fp64 products of p(token) = exp(x - max) (fp32) / Z, Z summed in double-float.
 *   Host errors as for the other calls; no device errors.
 */
int spec_tree_init(const int32_t* root_tokens, int batch, int max_nodes, void* state, size_t state_bytes,
                   int32_t* parent_out, int32_t* tokens_out, int32_t* n_nodes_out, int32_t* next_node,
                   uint8_t* flags, void* stream);
int spec_tree_expand(const float* draft_logits, int vocab, long long row_stride, long long node_stride,
                     int batch, int max_nodes, int topk, int max_depth, double threshold, void* state,
                     size_t state_bytes, int32_t* parent_out, int32_t* tokens_out, int32_t* n_nodes_out,
                     int32_t* next_node, uint8_t* flags, int32_t* dev_status, void* stream);

/*
 * spec_tree_expand_multi -- the same construction, several draft rows per call.
 *   ("EAGLE-2 deep dive", section on the dynamic draft-tree algorithm, as above; the batching
 *   is this library's and leaves the tree unchanged.)
 *   A queued candidate's expansion (its draft row's top-k and probabilities) depends only on
 *   the candidate -- its parent node and its token -- not on when it is popped. So each call
 *   lists up to `width` requests per sequence for the next call: request 0 is the node
 *   awaiting its expansion (the last node created), requests 1.. are the best queued
 *   candidates (largest score first, earlier push on ties) that have no row yet and sit
 *   below the depth limit. The caller's draft model writes one row per request (for a
 *   candidate: the row of the node it would become, given its parent and token). The next
 *   call reduces every row, keeps each candidate's result, expands the awaiting node and
 *   pops exactly as spec_tree_expand would, expanding at once every popped node whose result
 *   it holds; it stops at the first popped node that needs a row it has not got, or when the
 *   tree is complete. The tree (parent_out, tokens_out, n_nodes_out, flags) is therefore
 *   spec_tree_expand's, node for node, for every width; width 1 is spec_tree_expand.
 *
 *   After spec_tree_init the request list is the root alone (row 0).
 *   draft_logits  float; row j of sequence b starts at draft_logits + b * row_stride +
 *                 j * req_stride (elements); rows j >= req_n[b] are not read.
 *   width         in [1, 8]: the same for every call on one state (a state listing more
 *                 requests than the call's width is refused: SPEC_ERR_ARG in *dev_status,
 *                 nothing changes). topk, max_depth and threshold as for spec_tree_expand,
 *                 also the same for every call on one state.
 *   state         as for spec_tree_expand (spec_tree_init's), driven by this call only.
 *   req_parent, req_token  int32 [batch][width] (out): the parent node id (-1 for the root)
 *                 and token of each request; -1 past req_n[b].
 *   req_n         int32 [batch] (out): requests listed; 0 once the tree is complete.
 *   next_node     int32 [batch] (out): the awaiting node (request 0), -1 once complete.
 *   A sequence whose tree is complete is skipped: its outputs keep their last values.
 *   Device errors: SPEC_ERR_ARG as above; SPEC_ERR_CAPACITY if the state's result entries
 *   ran out (they cannot: max_nodes * 8 entries, and each call takes at most width while
 *   creating at least one node), the tree then ends.
 */
int spec_tree_expand_multi(const float* draft_logits, int vocab, long long row_stride, long long req_stride,
                           int batch, int max_nodes, int width, int topk, int max_depth, double threshold,
                           void* state, size_t state_bytes, int32_t* parent_out, int32_t* tokens_out,
                           int32_t* n_nodes_out, int32_t* next_node, int32_t* req_parent, int32_t* req_token,
                           int32_t* req_n, uint8_t* flags, int32_t* dev_status, void* stream);

/*
 * spec_accept_noalloc — spec_accept for callers that cannot allocate device memory.
 *   (No counterpart on the pages: this is a deployment convenience of this library.)
 *   Some callers have no way to obtain scratch memory: a runtime that only lends out
 *   the tensors it owns, a plugin host without an allocator, a serving loop that
 *   forbids allocation once it runs. This entry point takes the same arguments as
 *   spec_accept minus the workspace and computes the same results; its scratch is a
 *   fixed 4 MiB array inside the library (a file-scope __device__ array that every GPU
 *   loading the library holds until the process exits). It allocates and frees nothing.
 *   - Limit: sizes whose workspace (spec_workspace_size(SPEC_OP_ACCEPT, ...)) exceeds
 *     4 MiB return SPEC_ERR_WORKSPACE at once (e.g. 128256-token rows: up to ~10K nodes).
 *   - Set-up: the first call on a device, with that device current, looks up the array's
 *     device address; make that first call before any stream capture. The address is
 *     kept for the life of the process: do not use this entry point on a device after
 *     cudaDeviceReset (the array is then reloaded elsewhere).
 *   - Host checks are spec_accept's (the same argument errors, the same limits).
 *   - Every call zeroes the array's counters on `stream` first, then runs the kernels.
 *   - All calls share the one array: calls that may overlap on the GPU (different
 *     streams, or different host threads) race and must be serialised by the caller.
 */
int spec_accept_noalloc(int mode, const int32_t* parent, const int32_t* draft_tokens,
                        const float* target_logits, const float* draft_logits, const float* uniforms,
                        float temperature, int vocab, const int32_t* qo_indptr, int batch,
                        int total_nodes, int max_nodes, int path_cap, int32_t* accept_len,
                        int32_t* path, int32_t* out_tokens, uint8_t* flags, int32_t* dev_status,
                        void* stream);

/*
 * spec_tree_verify_attn_parents — spec_tree_verify_attn with the tree given as its parent
 *   array instead of a mask: the mask step runs inside the attention call.
 *   ("EAGLE-2 deep dive", core-implementation section: a node's mask row is the node and
 *   every ancestor up to the root.)
 *   Arguments: those of spec_tree_verify_attn, minus dtype (bf16 only) and mask, plus
 *   parent  int32 [total_nodes]  sequence-local parents, as for spec_build_tree_mask.
 *   The result equals spec_build_tree_mask followed by spec_tree_verify_attn on the same
 *   stream: for each in-tree key block, every query row derives its ancestor bits by
 *   walking parent links (staged in shared memory), with no mask buffer in between.
 *   - Device error SPEC_ERR_PARENT for a parent array that is not a tree; the affected
 *     rows then see no tree keys.
 *   - The tensor-core path only: d = 128, page_size = 16, hq / hkv dividing 128; other
 *     shapes return SPEC_ERR_UNSUPPORTED (use the two calls).
 *   - The parent array is read after the PDL wait, so it may come from the kernel just
 *     before. No depth output.
 */
int spec_tree_verify_attn_parents(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                                  int page_size, const int32_t* page_table, int max_pages,
                                  const int32_t* prefix_len, int max_prefix, const void* k_tree,
                                  const void* v_tree, const int32_t* parent, const int32_t* qo_indptr,
                                  int batch, int total_nodes, int max_nodes, int hq, int hkv, int d,
                                  float sm_scale, void* out, float* lse, void* ws, size_t ws_bytes,
                                  int32_t* dev_status, void* stream);

/*
 * FP8 KV cache: spec_tree_verify_attn_kv8 / spec_kv_commit_kv8.
 *   ("EAGLE-3 paper explainer" (0h-n0), operations section, model-optimisation list:
 *   quantisation and PagedAttention KV-cache tuning to cut GPU memory. The page names no
 *   format; this library reads it as follows.)
 *   The paged pool holds E4M3 codes, as the OCP 8-bit floating-point format defines them:
 *   1 sign, 4 exponent (bias 7) and 3 mantissa bits, subnormals at exponent 0, S.1111.111
 *   = NaN, largest magnitude 448. Code c of KV head g stands for
 *   value(c) * kv_scale[0][g] in K and value(c) * kv_scale[1][g] in V.
 *   kv_scale   float32 [2][hkv], device memory: K scales, then V scales. Each scale must
 *              be positive, finite and normal. A scale is read on the device at every
 *              call, so it may change between replays of a captured graph.
 *   k_pool, v_pool  uint8 [num_pages][hkv][page_size][d] codes, 16-byte aligned.
 *   The tree's own K/V (k_tree, v_tree), q and out stay bf16.
 *
 * spec_tree_verify_attn_kv8 — spec_tree_verify_attn (same arguments minus dtype, plus
 *   kv_scale) over an FP8 pool. The result is the attention of the definition with every
 *   prefix key and value replaced by its dequantised value; the tree keys are used as
 *   given. The tensor-core path only: d = 128, page_size = 16, hq / hkv dividing 128;
 *   other shapes return SPEC_ERR_UNSUPPORTED. The workspace is spec_workspace_size(
 *   SPEC_OP_ATTN, ...) for the same sizes. Errors as for spec_tree_verify_attn; q, k_tree,
 *   v_tree, out and (with a prefix) the pools must be 16-byte aligned (else SPEC_ERR_ARG).
 *   The pool must hold finite codes: a NaN code (S.1111.111) is read as +-480.
 */
int spec_tree_verify_attn_kv8(const void* q, const uint8_t* k_pool, const uint8_t* v_pool,
                              const float* kv_scale, int num_pages, int page_size,
                              const int32_t* page_table, int max_pages, const int32_t* prefix_len,
                              int max_prefix, const void* k_tree, const void* v_tree,
                              const uint64_t* mask, const int32_t* qo_indptr, int batch,
                              int total_nodes, int max_nodes, int hq, int hkv, int d, float sm_scale,
                              void* out, float* lse, void* ws, size_t ws_bytes, int32_t* dev_status,
                              void* stream);

/*
 * spec_kv_commit_kv8 — spec_kv_commit from bf16 tree rows into an FP8 pool.
 *   Every element x of a committed row of KV head g is written as the E4M3 code nearest to
 *   x / scale (the division in IEEE fp32, then round to nearest, ties to the even code).
 *   Finite quotients beyond +-448 saturate to +-448. scale = kv_scale[0][g] for K,
 *   kv_scale[1][g] for V. Arguments, checks and device errors are those of spec_kv_commit
 *   with dtype = SPEC_BF16 for the tree rows. d must be a multiple of 16 (else
 *   SPEC_ERR_UNSUPPORTED). kv_scale must not be NULL (SPEC_ERR_ARG).
 *   For a fused greedy acceptance + commit into an FP8 pool, call spec_accept and then
 *   this call on the same stream.
 */
int spec_kv_commit_kv8(const void* k_tree, const void* v_tree, const float* kv_scale,
                       const int32_t* path, int path_cap, const int32_t* accept_len,
                       const int32_t* qo_indptr, const int32_t* page_table, int max_pages,
                       int num_pages, int page_size, const int32_t* prefix_len, int32_t* seq_len_out,
                       uint8_t* k_pool, uint8_t* v_pool, int batch, int total_nodes, int hkv, int d,
                       int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
