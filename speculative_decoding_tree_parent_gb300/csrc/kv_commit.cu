// K-COMMIT: copy the accepted path's tree K/V rows into the sequence's paged cache.
//
// "EAGLE-2 deep dive", architecture section (the target KV cache must not be
// contaminated by verification) and "Accelerating Sonar through speculation",
// draft-target / MTP-schedule sections (KV of accepted tokens is filled; the
// next token is placed after the shift on the device, without a CPU sync).
//
// One CTA per sequence. The CTA first validates every slot of the commit
// (accept_len range, path node ids, page capacity and page ids), then moves the
// (L+1) x Hkv rows of D elements for K and V with 16-byte loads/stores. The
// rows are independent, so the copy is a flat loop over 16-byte vectors.
#include "common.cuh"

namespace specv {

__global__ void __launch_bounds__(256) kv_commit_kernel(
    const uint8_t* __restrict__ k_tree, const uint8_t* __restrict__ v_tree,
    const int32_t* __restrict__ path, int path_cap, const int32_t* __restrict__ accept_len,
    const int32_t* __restrict__ qo, const int32_t* __restrict__ page_table, int max_pages,
    int num_pages, int page_size, const int32_t* __restrict__ prefix_len,
    int32_t* __restrict__ seq_len_out, uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
    int hkv, int row_bytes, int32_t* status, const TokenInsert ins) {
  const int b = blockIdx.x;
  __shared__ int s_ok;
  __shared__ int s_L;
  // Everything the acceptance kernel does not write is read (or pulled into L2) before
  // waiting for it: the sequence's bounds, its page-table entries past the prefix and
  // its tree K/V rows (a few KB), so only accept_len / path remain on the critical path.
  const int base = __ldg(qo + b);
  const int n = __ldg(qo + b + 1) - base;
  const int P = __ldg(prefix_len + b);
  {
    const int span = n < path_cap ? n : path_cap;
    const int lp0 = P / page_size, lp1 = (P + span - 1) / page_size;
    for (int lp = lp0 + (int)threadIdx.x; lp <= lp1 && lp < max_pages; lp += blockDim.x)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(page_table + (size_t)b * max_pages + lp));
    const size_t bytes = (size_t)n * hkv * row_bytes;
    const uint8_t* k0 = k_tree + (size_t)base * hkv * row_bytes;
    const uint8_t* v0 = v_tree + (size_t)base * hkv * row_bytes;
    for (size_t off = (size_t)threadIdx.x * 128; off < bytes; off += (size_t)blockDim.x * 128) {
      asm volatile("prefetch.global.L2 [%0];" ::"l"(k0 + off));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(v0 + off));
    }
  }
  pdl_wait();  // accept_len / path come from the acceptance kernel just before
  if (threadIdx.x == 0) {
    int L = __ldg(accept_len + b);
    int ok = 1;
    if (L < 0 || L >= path_cap || L >= n || P < 0) {
      report(status, SPEC_ERR_INDEX);
      ok = 0;
    } else if (ins.token_buf != nullptr && P + L + 1 >= ins.token_stride) {
      report(status, SPEC_ERR_CAPACITY);  // the token row has no room for L + 1 tokens after P
      ok = 0;
    }
    s_L = L;
    s_ok = ok;
  }
  __syncthreads();
  const int L = s_L;
  if (!s_ok) return;
  // validation of every slot (L + 1 <= path_cap entries, one thread each)
  for (int i = threadIdx.x; i <= L; i += blockDim.x) {
    const int node = __ldg(path + (size_t)b * path_cap + i);
    const int slot = P + i;
    const int lp = slot / page_size;
    int code = 0;
    if (node < 0 || node >= n || (i == 0 && node != 0)) code = SPEC_ERR_INDEX;
    else if (lp >= max_pages) code = SPEC_ERR_CAPACITY;
    else {
      const int page = __ldg(page_table + (size_t)b * max_pages + lp);
      if (page < 0 || page >= num_pages) code = SPEC_ERR_PAGE;
    }
    if (code) {
      report(status, code);
      s_ok = 0;
    }
  }
  __syncthreads();
  if (!s_ok) return;
  // copy: vector v of the (i, g) row, for K and V
  const int vecs_per_row = row_bytes >> 4;
  const int rows = (L + 1) * hkv;
  const int total = rows * vecs_per_row;
  for (int e = threadIdx.x; e < total; e += blockDim.x) {
    const int r = e / vecs_per_row;
    const int vi = e - r * vecs_per_row;
    const int i = r / hkv;
    const int g = r - i * hkv;
    const int node = __ldg(path + (size_t)b * path_cap + i);
    const int slot = P + i;
    const int page = __ldg(page_table + (size_t)b * max_pages + slot / page_size);
    const int prow = slot - (slot / page_size) * page_size;
    const size_t src = ((size_t)(base + node) * hkv + g) * row_bytes + ((size_t)vi << 4);
    const size_t dst = (((size_t)page * hkv + g) * page_size + prow) * row_bytes + ((size_t)vi << 4);
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(k_tree + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(v_tree + src));
    *reinterpret_cast<uint4*>(k_pool + dst) = kv;
    *reinterpret_cast<uint4*>(v_pool + dst) = vv;
  }
  if (ins.token_buf != nullptr)  // the accepted tokens and the bonus after the root (room checked above)
    for (int i = threadIdx.x; i <= L; i += blockDim.x)
      ins.token_buf[(size_t)b * ins.token_stride + P + 1 + i] = __ldg(ins.out_tokens + (size_t)b * path_cap + i);
  if (threadIdx.x == 0 && seq_len_out != nullptr) seq_len_out[b] = P + L + 1;
}

int launch_kv_commit(int elem_bytes, const void* k_tree, const void* v_tree, const int32_t* path,
                     int path_cap, const int32_t* accept_len, const int32_t* qo,
                     const int32_t* page_table, int max_pages, int num_pages, int page_size,
                     const int32_t* prefix_len, int32_t* seq_len_out, void* k_pool, void* v_pool,
                     int batch, int hkv, int d, int32_t* status, cudaStream_t stream, TokenInsert ins) {
  const int row_bytes = d * elem_bytes;
  if (launch_pdl(kv_commit_kernel, dim3(batch), dim3(256), 0, stream, static_cast<const uint8_t*>(k_tree),
                 static_cast<const uint8_t*>(v_tree), path, path_cap, accept_len, qo, page_table, max_pages,
                 num_pages, page_size, prefix_len, seq_len_out, static_cast<uint8_t*>(k_pool),
                 static_cast<uint8_t*>(v_pool), hkv, row_bytes, status, ins) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace specv
