// Shared device/host helpers of libspecverify (no kernel lives here).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "spec_verify.h"

namespace specv {

// Most nodes one draft tree may have (every entry point refuses larger max_nodes).
constexpr int kMaxTreeNodes = 1024;
constexpr long kMaxGridYZ = 65535;  // a launch's y and z extents

// First-error-wins report into the caller's status word (nullable).
__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Sequence that owns global node row t: largest b with qo_indptr[b] <= t.
__device__ __forceinline__ int seq_of_row(const int32_t* __restrict__ qo, int batch, int t) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(qo + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor in the stream still runs; it must
// call pdl_wait() before reading anything the predecessor writes. pdl_trigger() lets
// the successor be scheduled early. A predecessor's writes are visible only after
// pdl_wait(), whether or not it signals early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The process-wide choice of spec_set_early_reads, taken when a call is made: whether the
// attention and the greedy walk may read their inputs before pdl_wait() (off: they wait first).
bool early_reads();

// Device-side insert of a step's tokens into each sequence's token buffer (the next step's
// input, no host round trip): out_tokens[b][0 .. L] (the L accepted tokens, then the bonus,
// which is the next root) go to token_buf[b][P + 1 .. P + L + 1], after the root at P.
// token_buf == nullptr: no insert.
struct TokenInsert {
  const int32_t* out_tokens;  // [batch][path_cap]
  int32_t* token_buf;         // [batch][token_stride]
  int token_stride;
};

// Arguments of the KV commit when it runs fused after the acceptance (spec_accept_commit).
struct CommitArgs {
  const uint8_t* k_tree;  // nullptr: no commit
  const uint8_t* v_tree;
  const int32_t* page_table;
  int max_pages, num_pages, page_size;
  const int32_t* prefix_len;
  int32_t* seq_len_out;
  uint8_t* k_pool;
  uint8_t* v_pool;
  int hkv, d, elem_bytes;
  TokenInsert ins;
};

// Double-float arithmetic: an fp32 pair (hi, lo) carrying about 48 significant bits,
// for sums that must stay accurate without fp64 in loops (its rate is low on this part).
struct F2 {
  float hi, lo;
};
// Double-float sum. Its first step is exact (two-sum), so a + b and b + a give the same
// bits: every lane of a butterfly ends with the same total.
__host__ __device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  const float s = a.hi + b.hi;
  const float v = s - a.hi;
  float e = (a.hi - (s - v)) + (b.hi - v);
  e += a.lo + b.lo;
  const float hi = s + e;
  return F2{hi, e - (hi - s)};
}
__device__ __forceinline__ F2 f2_warp_sum(F2 x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    x = f2_add(x, F2{__shfl_xor_sync(0xffffffffu, x.hi, o), __shfl_xor_sync(0xffffffffu, x.lo, o)});
  return x;
}

// a > b for normalised double-float values (|lo| at most half an ulp of hi).
__host__ __device__ __forceinline__ bool f2_gt(F2 a, F2 b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
// a * b for a double-float a and an fp32 b: the product of the high parts exactly (fma), the
// low part's product added, renormalised.
__host__ __device__ __forceinline__ F2 f2_mul_f(F2 a, float b) {
  const float p = a.hi * b;
  const float e = fmaf(a.lo, b, fmaf(a.hi, b, -p));
  const float hi = p + e;
  return F2{hi, e - (hi - p)};
}
// 1 / (hi + lo) in fp32: the fp32 reciprocal of hi refined once with the residual of both
// parts (Newton's step r + r (1 - x r)); 0 for a zero or negative input.
__host__ __device__ __forceinline__ float f2_rcp(F2 x) {
  if (!(x.hi > 0.f)) return 0.f;
  const float r = 1.0f / x.hi;
  const float e = fmaf(-x.hi, r, 1.0f) - x.lo * r;
  return fmaf(r, e, r);
}

// Host-side values that belong to one device: a kernel's raised shared-memory limit
// (cudaFuncSetAttribute applies to the current device only), its occupancy, the SM count.
// Kept per device index and read and written under one mutex, so several devices and
// several host threads each see their own device's value.
constexpr int kMaxDevices = 64;
struct PerDevice {
  std::mutex mu;
  int val[kMaxDevices] = {};  // 0: not known yet
};
// The current device's entry, computed by f() (> 0 on success, 0 on failure: asked again on
// the next call) the first time. Returns 0 when no device is current or f() failed.
template <typename F>
inline int per_device(PerDevice& c, F f) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(c.mu);
  if (c.val[dev] == 0) c.val[dev] = f(dev);
  return c.val[dev];
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

}  // namespace specv

// Launch `kernel` on `stream` with programmatic stream serialization (see pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Host-side launch check used by the entry points.
#define SPECV_LAUNCH_CHECK()                              \
  do {                                                    \
    cudaError_t e__ = cudaGetLastError();                 \
    if (e__ != cudaSuccess) return SPEC_ERR_CUDA;         \
  } while (0)
