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
//
// FP8 cache (kQuant): the tree rows are bf16 and the pool holds E4M3 codes ("EAGLE-3 paper
// explainer", operations section: quantisation and KV-cache tuning to cut memory). Code i
// of a row of KV head g is the nearest E4M3 value to x_i / scale[g] (one IEEE fp32
// division), ties to even, saturated to +-448 (cvt.rn.satfinite). A thread turns 32 bytes
// of bf16 into one 16-byte vector of codes.
#include "common.cuh"

namespace specv {

// 16 bf16 (two 16-byte vectors) divided by s -> 16 E4M3 codes, element i in byte i
__device__ __forceinline__ uint32_t quant4(uint32_t a, uint32_t b, float s) {
  const float x0 = __fdiv_rn(__uint_as_float(a << 16), s), x1 = __fdiv_rn(__uint_as_float(a & 0xFFFF0000u), s);
  const float x2 = __fdiv_rn(__uint_as_float(b << 16), s), x3 = __fdiv_rn(__uint_as_float(b & 0xFFFF0000u), s);
  uint16_t lo, hi;
  // the first source operand lands in the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ uint4 quant16(const uint4& u, const uint4& v, float s) {
  return make_uint4(quant4(u.x, u.y, s), quant4(u.z, u.w, s), quant4(v.x, v.y, s), quant4(v.z, v.w, s));
}

template <bool kQuant>
__global__ void __launch_bounds__(256) kv_commit_kernel(
    const uint8_t* __restrict__ k_tree, const uint8_t* __restrict__ v_tree,
    const int32_t* __restrict__ path, int path_cap, const int32_t* __restrict__ accept_len,
    const int32_t* __restrict__ qo, const int32_t* __restrict__ page_table, int max_pages,
    int num_pages, int page_size, const int32_t* __restrict__ prefix_len,
    int32_t* __restrict__ seq_len_out, uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
    int hkv, int row_bytes, int32_t* status, const TokenInsert ins, const float* __restrict__ kv_scale) {
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
    const int src_row = kQuant ? 2 * row_bytes : row_bytes;  // bf16 rows feed a code row
    const size_t bytes = (size_t)n * hkv * src_row;
    const uint8_t* k0 = k_tree + (size_t)base * hkv * src_row;
    const uint8_t* v0 = v_tree + (size_t)base * hkv * src_row;
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
    const size_t dst = (((size_t)page * hkv + g) * page_size + prow) * row_bytes + ((size_t)vi << 4);
    if (kQuant) {
      const size_t src = ((size_t)(base + node) * hkv + g) * (2 * row_bytes) + ((size_t)vi << 5);
      const uint4* ks = reinterpret_cast<const uint4*>(k_tree + src);
      const uint4* vs = reinterpret_cast<const uint4*>(v_tree + src);
      const uint4 k0v = __ldg(ks), k1v = __ldg(ks + 1), v0v = __ldg(vs), v1v = __ldg(vs + 1);
      *reinterpret_cast<uint4*>(k_pool + dst) = quant16(k0v, k1v, __ldg(kv_scale + g));
      *reinterpret_cast<uint4*>(v_pool + dst) = quant16(v0v, v1v, __ldg(kv_scale + hkv + g));
    } else {
      const size_t src = ((size_t)(base + node) * hkv + g) * row_bytes + ((size_t)vi << 4);
      const uint4 kv = __ldg(reinterpret_cast<const uint4*>(k_tree + src));
      const uint4 vv = __ldg(reinterpret_cast<const uint4*>(v_tree + src));
      *reinterpret_cast<uint4*>(k_pool + dst) = kv;
      *reinterpret_cast<uint4*>(v_pool + dst) = vv;
    }
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
                     int batch, int hkv, int d, int32_t* status, cudaStream_t stream, TokenInsert ins,
                     const float* kv_scale) {
  // the pool's row: d codes for an FP8 cache (bf16 tree rows), else d elements
  const int row_bytes = kv_scale != nullptr ? d : d * elem_bytes;
  const uint8_t* kt = static_cast<const uint8_t*>(k_tree);
  const uint8_t* vt = static_cast<const uint8_t*>(v_tree);
  uint8_t* kp = static_cast<uint8_t*>(k_pool);
  uint8_t* vp = static_cast<uint8_t*>(v_pool);
  const cudaError_t e =
      kv_scale != nullptr
          ? launch_pdl(kv_commit_kernel<true>, dim3(batch), dim3(256), 0, stream, kt, vt, path, path_cap, accept_len,
                       qo, page_table, max_pages, num_pages, page_size, prefix_len, seq_len_out, kp, vp, hkv,
                       row_bytes, status, ins, kv_scale)
          : launch_pdl(kv_commit_kernel<false>, dim3(batch), dim3(256), 0, stream, kt, vt, path, path_cap,
                       accept_len, qo, page_table, max_pages, num_pages, page_size, prefix_len, seq_len_out, kp, vp,
                       hkv, row_bytes, status, ins, kv_scale);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// a cache of the tree's own element type (plain copy)
int launch_kv_commit(int elem_bytes, const void* k_tree, const void* v_tree, const int32_t* path,
                     int path_cap, const int32_t* accept_len, const int32_t* qo,
                     const int32_t* page_table, int max_pages, int num_pages, int page_size,
                     const int32_t* prefix_len, int32_t* seq_len_out, void* k_pool, void* v_pool,
                     int batch, int hkv, int d, int32_t* status, cudaStream_t stream, TokenInsert ins) {
  return launch_kv_commit(elem_bytes, k_tree, v_tree, path, path_cap, accept_len, qo, page_table, max_pages,
                          num_pages, page_size, prefix_len, seq_len_out, k_pool, v_pool, batch, hkv, d, status,
                          stream, ins, nullptr);
}

}  // namespace specv
