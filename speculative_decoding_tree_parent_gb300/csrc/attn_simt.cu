// Tree-verify attention on the CUDA cores (FFMA), fp32 or bf16 inputs, fp32 math.
//
// This is the path for fp32 inputs (tf32 tensor-core products would miss the
// 1e-4 fp32 tolerance) and for head dims / group sizes the tensor-core kernel
// does not take. Same split-KV structure and partial format as the tcgen05
// kernel, so both share the combine kernel.
//
// CTA = (key split s, block of 16 query rows, sequence b x KV head g). Query
// rows of (b, g) are ordered node-major: row r -> node r / G, head g*G + r % G.
// Keys arrive in tiles of 32 (converted to fp32 in shared memory); a warp owns
// 4 rows, lane j scores key j, the online softmax runs in the log2 domain with
// warp shuffles, and lane l accumulates output dims l, l+32, ...
#include "attn_common.cuh"

namespace specv {

constexpr int kSimtKeys = 32;
constexpr int kSimtRows = 16;
constexpr int kSimtWarps = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kSimtWarps * 32) attn_simt_kernel(
    const T* __restrict__ q, const T* __restrict__ k_pool, const T* __restrict__ v_pool, int num_pages,
    int ps, const int32_t* __restrict__ page_table, int max_pages, const int32_t* __restrict__ prefix_len,
    const T* __restrict__ k_tree, const T* __restrict__ v_tree, const uint64_t* __restrict__ mask,
    int mask_words, const int32_t* __restrict__ qo, int hq, int hkv, float scale_log2, int splits,
    int total_rows, T* __restrict__ out, float* __restrict__ lse, AttnWs ws, int32_t* status) {
  constexpr int KB = kSimtKeys, R = kSimtRows, RPW = R / kSimtWarps, DL = D / 32;
  __shared__ float sq[R][D];
  __shared__ float sk[KB][D + 1];
  __shared__ float sv[KB][D];
  __shared__ uint32_t smask[R];
  const int s = blockIdx.x, rb = blockIdx.y, bg = blockIdx.z;
  const int G = hq / hkv;
  const int b = bg / hkv, g = bg - (bg / hkv) * hkv;
  const int base = __ldg(qo + b);
  const int N = __ldg(qo + b + 1) - base;
  int P = __ldg(prefix_len + b);
  if (N > mask_words * 64 || P > max_pages * ps || P < 0) {  // sizes beyond what the caller declared
    if (threadIdx.x == 0 && s == 0 && rb == 0) report(status, SPEC_ERR_CAPACITY);
    return;
  }
  const int rows = N * G;
  const int row0 = rb * R;
  if (row0 >= rows) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SplitRange sr = split_range(P, N, KB, splits, s);

  for (int idx = tid; idx < R * D; idx += blockDim.x) {
    const int r = idx / D, d = idx - (idx / D) * D;
    const int row = row0 + r;
    float val = 0.f;
    if (row < rows) {
      const int i = row / G, h = g * G + (row - (row / G) * G);
      val = to_f32(q[((size_t)(base + i) * hq + h) * D + d]) * scale_log2;
    }
    sq[r][d] = val;
  }

  float m[RPW], l[RPW], o[RPW][DL];
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
#pragma unroll
    for (int k = 0; k < DL; ++k) o[rr][k] = 0.f;
  }

  for (int blk = sr.blk_lo; blk < sr.blk_hi; ++blk) {
    const bool is_tree = blk >= sr.n_prefix_blocks;
    const int key0 = is_tree ? (blk - sr.n_prefix_blocks) * KB : blk * KB;
    const int nvalid = is_tree ? min(KB, N - key0) : min(KB, P - key0);
    // the tile's K/V into registers (every load of the tile in flight at once), then shared memory
    constexpr int kPer = KB * D / (kSimtWarps * 32);
    float kr[kPer], vr[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = tid + u * kSimtWarps * 32;
      const int j = idx / D, d = idx - (idx / D) * D;
      kr[u] = 0.f;
      vr[u] = 0.f;
      if (j < nvalid) {
        size_t off;
        bool ok = true;
        if (!is_tree) {
          const int k = key0 + j;
          const int page = __ldg(page_table + (size_t)b * max_pages + k / ps);
          if (page < 0 || page >= num_pages) {
            ok = false;
            if (d == 0) report(status, SPEC_ERR_PAGE);
          }
          off = (((size_t)page * hkv + g) * ps + (k - (k / ps) * ps)) * D + d;
        } else {
          off = ((size_t)(base + key0 + j) * hkv + g) * D + d;
        }
        if (ok) {
          kr[u] = to_f32(is_tree ? k_tree[off] : k_pool[off]);
          vr[u] = to_f32(is_tree ? v_tree[off] : v_pool[off]);
        }
      }
    }
    __syncthreads();  // previous tile fully consumed
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = tid + u * kSimtWarps * 32;
      const int j = idx / D, d = idx - (idx / D) * D;
      sk[j][d] = kr[u];
      sv[j][d] = vr[u];
    }
    if (is_tree && tid < R) {
      const int row = row0 + tid;
      uint32_t bits = 0u;
      if (row < rows) {
        const int i = row / G;
        const uint64_t w = __ldg(mask + (size_t)(base + i) * mask_words + (key0 >> 6));
        bits = (uint32_t)(w >> (key0 & 63));
      }
      smask[tid] = bits;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
      const int r = warp * RPW + rr;
      float sc = 0.f;
#pragma unroll 16
      for (int d = 0; d < D; ++d) sc = fmaf(sq[r][d], sk[lane][d], sc);
      const bool ok = lane < nvalid && (!is_tree || ((smask[r] >> lane) & 1u));
      sc = ok ? sc : -INFINITY;
      float mx = sc;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mnew = fmaxf(m[rr], mx);
      const float p = (mnew == -INFINITY) ? 0.f : exp2f(sc - mnew);
      const float alpha = (mnew == -INFINITY) ? 1.f : exp2f(m[rr] - mnew);
      float ps_ = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps_ += __shfl_xor_sync(0xffffffffu, ps_, off);
      l[rr] = l[rr] * alpha + ps_;
      m[rr] = mnew;
#pragma unroll
      for (int k = 0; k < DL; ++k) o[rr][k] *= alpha;
#pragma unroll 8
      for (int j = 0; j < KB; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int k = 0; k < DL; ++k) o[rr][k] = fmaf(pj, sv[j][lane + 32 * k], o[rr][k]);
      }
    }
  }

#pragma unroll
  for (int rr = 0; rr < RPW; ++rr) {
    const int row = row0 + warp * RPW + rr;
    if (row >= rows) continue;
    const int i = row / G, h = g * G + (row - (row / G) * G);
    const size_t orow = (size_t)(base + i) * hq + h;
    if (splits == 1) {
      const float inv = l[rr] > 0.f ? 1.f / l[rr] : 0.f;
#pragma unroll
      for (int k = 0; k < DL; ++k) out[orow * D + lane + 32 * k] = from_f32<T>(o[rr][k] * inv);
      if (lse != nullptr && lane == 0) lse[orow] = (m[rr] + log2f(l[rr])) * kLn2;
    } else {
      float* dst = ws.o + ((size_t)s * total_rows + orow) * D;
#pragma unroll
      for (int k = 0; k < DL; ++k) dst[lane + 32 * k] = o[rr][k];
      if (lane == 0) ws.ml[(size_t)s * total_rows + orow] = make_float2(m[rr], l[rr]);
    }
  }
}

// Merge of the key-split partials: one warp per output row.
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ wo,
                                                           const float2* __restrict__ wml, int splits,
                                                           int total_rows, T* __restrict__ out,
                                                           float* __restrict__ lse) {
  constexpr int DL = D / 32;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= total_rows) return;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, __ldg(&wml[(size_t)s * total_rows + row].x));
  float L = 0.f, acc[DL];
#pragma unroll
  for (int k = 0; k < DL; ++k) acc[k] = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float2 ml = __ldg(&wml[(size_t)s * total_rows + row]);
    if (ml.x == -INFINITY) continue;
    const float f = exp2f(ml.x - M);
    L = fmaf(ml.y, f, L);
    const float* src = wo + ((size_t)s * total_rows + row) * D;
#pragma unroll
    for (int k = 0; k < DL; ++k) acc[k] = fmaf(__ldg(src + lane + 32 * k), f, acc[k]);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int k = 0; k < DL; ++k) out[(size_t)row * D + lane + 32 * k] = from_f32<T>(acc[k] * inv);
  if (lse != nullptr && lane == 0) lse[row] = (M + log2f(L)) * kLn2;
}

int attn_splits_simt(int batch, int max_nodes, int hq, int hkv, int max_prefix) {
  const int G = hq / hkv;
  const int row_blocks = ceil_div(max_nodes * G, kSimtRows);
  const long base = (long)batch * hkv * row_blocks;
  const int blocks = ceil_div(max_prefix, kSimtKeys) + ceil_div(max_nodes, kSimtKeys);
  int s = (int)((2L * 152 + base - 1) / (base > 0 ? base : 1));
  // at least four 32-key tiles per split, except for grids far too small to fill the GPU
  // (a handful of row blocks): there one tile per split, as the tiles are the only parallelism
  const int per = base * 4 <= 152 ? 1 : 4;
  const int cap = blocks / per > 1 ? blocks / per : 1;
  if (s > cap) s = cap;
  if (s > 64) s = 64;
  return s < 1 ? 1 : s;
}

template <typename T, int D>
static int launch_simt_t(const void* q, const void* k_pool, const void* v_pool, int num_pages, int ps,
                         const int32_t* page_table, int max_pages, const int32_t* prefix_len,
                         const void* k_tree, const void* v_tree, const uint64_t* mask, int mask_words,
                         const int32_t* qo, int batch, int total_nodes, int max_nodes, int hq, int hkv,
                         float sm_scale, int splits, void* out, float* lse, void* ws, int32_t* status,
                         cudaStream_t stream) {
  const int rows = total_nodes * hq;
  const AttnWs w = AttnWs::at(ws, splits, rows, D);
  const int G = hq / hkv;
  const dim3 grid(splits, ceil_div(max_nodes * G, kSimtRows), batch * hkv);
  attn_simt_kernel<T, D><<<grid, kSimtWarps * 32, 0, stream>>>(
      static_cast<const T*>(q), static_cast<const T*>(k_pool), static_cast<const T*>(v_pool), num_pages, ps,
      page_table, max_pages, prefix_len, static_cast<const T*>(k_tree), static_cast<const T*>(v_tree), mask,
      mask_words, qo, hq, hkv, sm_scale * kLog2e, splits, rows, static_cast<T*>(out), lse, w, status);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (splits > 1) {
    attn_combine_kernel<T, D><<<ceil_div(rows, 8), 256, 0, stream>>>(w.o, w.ml, splits, rows,
                                                                      static_cast<T*>(out), lse);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

int launch_attn_simt(int dtype, const void* q, const void* k_pool, const void* v_pool, int num_pages, int ps,
                     const int32_t* page_table, int max_pages, const int32_t* prefix_len, int max_prefix,
                     const void* k_tree, const void* v_tree, const uint64_t* mask, const int32_t* qo,
                     int batch, int total_nodes, int max_nodes, int hq, int hkv, int d, float sm_scale,
                     void* out, float* lse, void* ws, int32_t* status, cudaStream_t stream) {
  const int splits = attn_splits_simt(batch, max_nodes, hq, hkv, max_prefix);
  const int mw = (max_nodes + 63) >> 6;
#define SPECV_SIMT(T, D)                                                                                   \
  return launch_simt_t<T, D>(q, k_pool, v_pool, num_pages, ps, page_table, max_pages, prefix_len, k_tree,  \
                             v_tree, mask, mw, qo, batch, total_nodes, max_nodes, hq, hkv, sm_scale, splits, \
                             out, lse, ws, status, stream)
  if (dtype == SPEC_F32) {
    if (d == 64) SPECV_SIMT(float, 64);
    if (d == 128) SPECV_SIMT(float, 128);
  } else {
    if (d == 64) SPECV_SIMT(__nv_bfloat16, 64);
    if (d == 128) SPECV_SIMT(__nv_bfloat16, 128);
  }
#undef SPECV_SIMT
  return SPEC_ERR_UNSUPPORTED;
}

int launch_attn_combine(int dtype, const AttnWs& w, int splits, int total_nodes, int hq, int d, void* out,
                        float* lse, cudaStream_t stream) {
  const int rows = total_nodes * hq;
  const dim3 grid(ceil_div(rows, 8));
  if (dtype == SPEC_F32) {
    if (d == 64) attn_combine_kernel<float, 64><<<grid, 256, 0, stream>>>(w.o, w.ml, splits, rows, (float*)out, lse);
    else attn_combine_kernel<float, 128><<<grid, 256, 0, stream>>>(w.o, w.ml, splits, rows, (float*)out, lse);
  } else {
    if (d == 64)
      attn_combine_kernel<__nv_bfloat16, 64><<<grid, 256, 0, stream>>>(w.o, w.ml, splits, rows, (__nv_bfloat16*)out, lse);
    else
      attn_combine_kernel<__nv_bfloat16, 128><<<grid, 256, 0, stream>>>(w.o, w.ml, splits, rows, (__nv_bfloat16*)out, lse);
  }
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace specv
