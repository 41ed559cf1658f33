// Tree-verify attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "EAGLE-2 deep dive" (techknowgenie), architecture and production sections: every
// tree token is verified in one attention pass; a node sees the verified prefix and
// only its ancestors (the 2-D tree mask), indexed over paged KV memory.
// "Accelerating Sonar through speculation", EAGLE section: applying a custom mask
// over the whole sequence is what slows attention (up to 50%), so here prefix
// tiles run with no mask at all (only a length bound on the ragged last block) and
// the ancestor bits are tested on the in-tree tiles only.
//
// CTA = (key split s, M-tile of 128 query rows, sequence b x KV head g); rows are
// node-major (row r -> node r / G, head g*G + r % G), so the G query heads of a KV
// head share every K/V tile (GQA). Keys come in blocks of 64: prefix blocks are 4
// pages of 16 tokens, TMA-loaded page by page through the page table
// ([page][Hkv][16][128] bf16, so a (page, head) is one 4 KB tile); tree blocks are
// 64 rows of the dense tree K/V. Warp roles:
//   warp 0     TMA producer: Q once, then K/V blocks into a 4-stage ring
//   warp 1     TMEM allocation; one lane issues the MMAs:
//                S[j%2] = Q K_j^T   (M 128, N 64, K 128; both operands K-major)
//                O     += P_j V_j   (M 128, N 128, K 64; V is MN-major)
//   warps 2-5  softmax, one thread per query row (its TMEM lane): S row -> max /
//              exp2 / row sum in registers, P row -> bf16 in shared memory
//              (128-byte swizzle), O rescale in TMEM only when the running max
//              grows by more than 2^8; finally O / l to global memory (or the
//              unnormalised split partial for the LSE merge).
// S is double-buffered in TMEM (2 x 64 columns) next to O (128 columns), so QK of
// block j+1 runs while the softmax of block j does. Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "tc_ptx.cuh"

namespace specv {

constexpr int kTcRows = 128;
constexpr int kTcKeys = 64;
constexpr int kTcD = 128;
constexpr int kTcStages = 4;
constexpr int kTcThreads = 192;
constexpr float kRescaleThr = 8.0f;            // log2 units: P entries stay <= 2^8
constexpr long long kWaitLimit = 4000000000LL;  // cycles (about 2 s) before a wait gives up

constexpr uint32_t kQSlab = kTcRows * 128;                  // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kKVSlab = kTcKeys * 128;                 // 8 KB: 64 keys x 64 bf16
constexpr uint32_t kStageBytes = 4 * kKVSlab;               // K (2 slabs) + V (2 slabs)
constexpr uint32_t kPBuf = kTcRows * 128;                   // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + 2 * kQSlab;
constexpr uint32_t kOffP = kOffKV + kTcStages * kStageBytes;
constexpr uint32_t kOffBar = kOffP + 2 * kPBuf;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;       // barriers + alignment slack
constexpr uint32_t kTmemCols = 256;                         // S0 | S1 | O
constexpr uint32_t kIdescQK = tc::idesc_bf16(kTcRows, kTcKeys, 0);
constexpr uint32_t kIdescPV = tc::idesc_bf16(kTcRows, kTcD, 1);

struct TcParams {
  const int32_t* page_table;
  int max_pages, num_pages;
  const int32_t* prefix_len;
  const uint64_t* mask;
  int mask_words;
  const int32_t* qo;
  int hq, hkv, G, splits, total_rows;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  AttnWs ws;
  int32_t* status;
};

struct TcBars {
  uint64_t q_full, kv_full[kTcStages], kv_empty[kTcStages], s_full[2], p_full[2], pv_done, mma_fin;
  uint32_t tmem_base;
  int abort;
};

// One lane waits, the whole warp gets the answer: keeps warp-collective tcgen05.ld/st
// and __syncwarp on a converged warp even when a wait gives up.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, abort, kWaitLimit) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
                   const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kt,
                   const __grid_constant__ CUtensorMap tm_vt, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcBars& bars = *reinterpret_cast<TcBars*>(smem + kOffBar);
  const uint32_t s_base = tc::smem_u32(smem);

  const int split = blockIdx.x, mt = blockIdx.y, bg = blockIdx.z;
  const int G = p.G;
  const int b = bg / p.hkv, g = bg - (bg / p.hkv) * p.hkv;
  const int base = __ldg(p.qo + b);
  const int N = __ldg(p.qo + b + 1) - base;
  const int P = __ldg(p.prefix_len + b);
  const int npt = kTcRows / G;  // tree nodes per M-tile
  const int node0 = mt * npt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (node0 >= N) return;  // whole CTA: this M-tile is past the sequence's tree
  if (N > p.mask_words * 64 || P < 0 || P > p.max_pages * 16) {
    if (threadIdx.x == 0 && split == 0) report(p.status, SPEC_ERR_CAPACITY);
    return;
  }
  const SplitRange sr = split_range(P, N, kTcKeys, p.splits, split);
  const int nb = sr.blk_hi - sr.blk_lo;
  const int npb = sr.n_prefix_blocks;

  // softmax-thread row bookkeeping (warps 2-5; quarter q of TMEM lanes = warp % 4)
  const int row = (warp & 3) * 32 + lane;
  const int node_l = node0 + row / G;
  const int head = g * G + (row - (row / G) * G);
  const bool row_valid = node_l < N;
  const size_t orow = (size_t)(base + node_l) * p.hq + head;

  if (nb == 0) {  // empty key split: an empty partial (only possible when splits > 1)
    if (warp >= 2 && row_valid) {
      float* dst = p.ws.o + ((size_t)split * p.total_rows + orow) * kTcD;
      for (int d = 0; d < kTcD; d += 4) *reinterpret_cast<float4*>(dst + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      p.ws.ml[(size_t)split * p.total_rows + orow] = make_float2(-INFINITY, 0.f);
    }
    return;
  }

  const uint32_t bar_q = tc::smem_u32(&bars.q_full);
  const uint32_t bar_pv = tc::smem_u32(&bars.pv_done);
  const uint32_t bar_fin = tc::smem_u32(&bars.mma_fin);
  auto bar_kvf = [&](int s) { return tc::smem_u32(&bars.kv_full[s]); };
  auto bar_kve = [&](int s) { return tc::smem_u32(&bars.kv_empty[s]); };
  auto bar_sf = [&](int s) { return tc::smem_u32(&bars.s_full[s]); };
  auto bar_pf = [&](int s) { return tc::smem_u32(&bars.p_full[s]); };
  volatile int* abort = &bars.abort;

  if (threadIdx.x == 0) {
    tc::mbar_init(bar_q, 1);
    for (int s = 0; s < kTcStages; ++s) {
      tc::mbar_init(bar_kvf(s), 1);
      tc::mbar_init(bar_kve(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar_sf(s), 1);
      tc::mbar_init(bar_pf(s), 128);
    }
    tc::mbar_init(bar_pv, 1);
    tc::mbar_init(bar_fin, 1);
    bars.abort = 0;
    tc::mbar_fence_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(&bars.tmem_base), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = bars.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    int issued = 0;
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_kp);
      tc::prefetch_tmap(&tm_vp);
      tc::prefetch_tmap(&tm_kt);
      tc::prefetch_tmap(&tm_vt);
      tc::mbar_arrive_expect_tx(bar_q, 2 * kQSlab);
      tc::tma_load_3d(s_base + kOffQ, &tm_q, bar_q, 0, g * G, base + node0);
      tc::tma_load_3d(s_base + kOffQ + kQSlab, &tm_q, bar_q, 64, g * G, base + node0);
    }
    for (int j = 0; j < nb; ++j) {
      const int st = j % kTcStages;
      if (!warp_wait(bar_kve(st), ((j / kTcStages) & 1) ^ 1, abort)) {
        if (lane == 0) report(p.status, SPEC_ERR_TIMEOUT);
        break;
      }
      const uint32_t dst0 = s_base + kOffKV + st * kStageBytes;
      const int blk = sr.blk_lo + j;
      if (lane == 0) tc::mbar_arrive_expect_tx(bar_kvf(st), kStageBytes);
      __syncwarp();
      if (blk < npb) {
        if (lane < 16) {
          const int pp = lane >> 2, which = lane & 3;
          const int lp = blk * 4 + pp;
          int page = p.num_pages;  // out of range: TMA fills zeros
          if (lp * 16 < P) {
            const int pg = __ldg(p.page_table + (size_t)b * p.max_pages + lp);
            if (pg >= 0 && pg < p.num_pages) page = pg;
            else report(p.status, SPEC_ERR_PAGE);
          }
          const int slab = which & 1, isv = which >> 1;
          const uint32_t dst = dst0 + isv * 2 * kKVSlab + slab * kKVSlab + pp * 2048;
          tc::tma_load_4d(dst, isv ? &tm_vp : &tm_kp, bar_kvf(st), slab * 64, 0, g, page);
        }
      } else {
        if (lane < 4) {
          const int tb = blk - npb;
          const int slab = lane & 1, isv = lane >> 1;
          const uint32_t dst = dst0 + isv * 2 * kKVSlab + slab * kKVSlab;
          tc::tma_load_3d(dst, isv ? &tm_vt : &tm_kt, bar_kvf(st), slab * 64, g, base + tb * 64);
        }
      }
      issued = j + 1;
    }
    // leave no copy in flight: the last stages issued must have landed
    if (lane == 0 && *abort) {
      int zero = 0;
      for (int j = max(0, issued - kTcStages); j < issued; ++j)
        tc::mbar_wait(bar_kvf(j % kTcStages), (j / kTcStages) & 1, &zero, kWaitLimit);
      tc::mbar_wait(bar_q, 0, &zero, kWaitLimit);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t t_s[2] = {tbase, tbase + 64};
      const uint32_t t_o = tbase + 128;
      auto pv = [&](int i) -> bool {
        if (!tc::mbar_wait(bar_pf(i & 1), (i >> 1) & 1, abort, kWaitLimit)) return false;
        tc::fence_after_sync();
        const uint32_t pbuf = s_base + kOffP + (i & 1) * kPBuf;
        const uint32_t vbuf = s_base + kOffKV + (i % kTcStages) * kStageBytes + 2 * kKVSlab;
#pragma unroll
        for (int k = 0; k < kTcKeys / 16; ++k) {
          const uint64_t a = tc::sdesc_sw128(pbuf + k * 32, 16, 1024);
          const uint64_t bdesc = tc::sdesc_sw128(vbuf + k * 2048, kKVSlab, 1024);
          tc::mma_bf16(t_o, a, bdesc, kIdescPV, (i > 0 || k > 0) ? 1u : 0u);
        }
        tc::mma_commit(bar_kve(i % kTcStages));
        tc::mma_commit(bar_pv);
        return true;
      };
      bool ok = tc::mbar_wait(bar_q, 0, abort, kWaitLimit);
      int j = 0;
      for (; ok && j < nb; ++j) {
        const int st = j % kTcStages;
        if (!tc::mbar_wait(bar_kvf(st), (j / kTcStages) & 1, abort, kWaitLimit)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t kbuf = s_base + kOffKV + st * kStageBytes;
#pragma unroll
        for (int k = 0; k < kTcD / 16; ++k) {
          const uint64_t a = tc::sdesc_sw128(s_base + kOffQ + (k >> 2) * kQSlab + (k & 3) * 32, 16, 1024);
          const uint64_t bdesc = tc::sdesc_sw128(kbuf + (k >> 2) * kKVSlab + (k & 3) * 32, 16, 1024);
          tc::mma_bf16(t_s[j & 1], a, bdesc, kIdescQK, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar_sf(j & 1));
        if (j >= 1 && !pv(j - 1)) {
          ok = false;
          break;
        }
      }
      if (ok) ok = pv(nb - 1);
      if (!ok) report(p.status, SPEC_ERR_TIMEOUT);
      // every MMA issued has completed before TMEM is released
      tc::mma_commit(bar_fin);
      int zero = 0;
      tc::mbar_wait(bar_fin, 0, &zero, kWaitLimit);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax warps
    const uint32_t t_lane = tbase + ((uint32_t)((warp & 3) * 32) << 16);
    const uint64_t* mrow = p.mask + (size_t)(base + node_l) * p.mask_words;
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      if (!warp_wait(bar_sf(j & 1), (j >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      float sv[kTcKeys];
      tc::tmem_ld32(t_lane + (j & 1) * 64, sv);
      tc::tmem_ld32(t_lane + (j & 1) * 64 + 32, sv + 32);
      tc::tmem_wait_ld();
      const int blk = sr.blk_lo + j;
      float mx = -INFINITY;
      if (blk < npb) {
        const int nvalid = min(kTcKeys, P - blk * kTcKeys);  // length bound only, no mask
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c) {
          sv[c] = c < nvalid ? sv[c] * p.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sv[c]);
        }
      } else {
        const uint64_t bits = row_valid ? __ldg(mrow + (blk - npb)) : 0ull;
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c) {
          sv[c] = ((bits >> c) & 1ull) ? sv[c] * p.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sv[c]);
        }
      }
      float alpha = 1.f;
      bool rescale = false;
      if (mx > -INFINITY && (m_run == -INFINITY || mx > m_run + kRescaleThr)) {
        alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - mx);
        m_run = mx;
        rescale = j > 0;
      }
      uint32_t packed[kTcKeys / 2];
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kTcKeys; c += 2) {
        const float p0 = m_run == -INFINITY ? 0.f : exp2f(sv[c] - m_run);
        const float p1 = m_run == -INFINITY ? 0.f : exp2f(sv[c + 1] - m_run);
        rs += p0 + p1;
        packed[c >> 1] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;
      if (j >= 1) {  // PV of the previous block done: O is stable and P[j%2] is free
        if (!warp_wait(bar_pv, (j - 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
      }
      if (__any_sync(0xffffffffu, rescale)) {  // tcgen05.ld/st are warp-collective
#pragma unroll
        for (int ch = 0; ch < kTcD / 32; ++ch) {
          float o[32];
          tc::tmem_ld32(t_lane + 128 + ch * 32, o);
          tc::tmem_wait_ld();
          const float f = rescale ? alpha : 1.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tc::tmem_st32(t_lane + 128 + ch * 32, o);
        }
        tc::tmem_wait_st();
      }
      uint8_t* prow = smem + kOffP + (j & 1) * kPBuf + row * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const int phys = cc ^ (row & 7);
        *reinterpret_cast<uint4*>(prow + phys * 16) =
            make_uint4(packed[4 * cc], packed[4 * cc + 1], packed[4 * cc + 2], packed[4 * cc + 3]);
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(bar_pf(j & 1));
    }
    if (ok && warp_wait(bar_pv, (nb - 1) & 1, abort)) {
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      for (int ch = 0; ch < kTcD / 32; ++ch) {
        float o[32];
        __syncwarp();
        tc::tmem_ld32(t_lane + 128 + ch * 32, o);
        tc::tmem_wait_ld();
        if (!row_valid) {
        } else if (p.splits == 1) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kTcD + ch * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pack_bf16x2(o[8 * v] * inv, o[8 * v + 1] * inv),
                                pack_bf16x2(o[8 * v + 2] * inv, o[8 * v + 3] * inv),
                                pack_bf16x2(o[8 * v + 4] * inv, o[8 * v + 5] * inv),
                                pack_bf16x2(o[8 * v + 6] * inv, o[8 * v + 7] * inv));
        } else {
          float4* dst = reinterpret_cast<float4*>(p.ws.o + ((size_t)split * p.total_rows + orow) * kTcD + ch * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v) dst[v] = make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        }
      }
      if (row_valid) {
        if (p.splits == 1) {
          if (p.lse != nullptr) p.lse[orow] = (m_run + log2f(l)) * kLn2;
        } else {
          p.ws.ml[(size_t)split * p.total_rows + orow] = make_float2(m_run, l);
        }
      }
    } else if (threadIdx.x == 64) {
      report(p.status, SPEC_ERR_TIMEOUT);
    }
    __syncwarp();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, kTmemCols);
  }
}

// ------------------------------------------------------------------------------ host

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// bf16 tensor map, 128-byte swizzle, zero fill out of bounds; dims/box innermost first.
static bool encode_bf16(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                        const cuuint32_t* box) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool attn_tc_supported(int dtype, int hq, int hkv, int d, int page_size, int max_nodes) {
  if (dtype != SPEC_BF16 || d != kTcD || page_size != 16 || hkv <= 0 || hq % hkv) return false;
  const int G = hq / hkv;
  return G >= 1 && G <= kTcRows && kTcRows % G == 0 && max_nodes >= 1 && max_nodes <= 1024 &&
         tensor_map_encoder() != nullptr;
}

int attn_splits_tc(int batch, int max_nodes, int hq, int hkv, int max_prefix) {
  if (hkv <= 0 || hq % hkv) return 1;
  const int G = hq / hkv;
  const int mtiles = ceil_div(max_nodes * G, kTcRows);
  const long base = (long)batch * hkv * mtiles;
  const int blocks = ceil_div(max_prefix, kTcKeys) + ceil_div(max_nodes, kTcKeys);
  const int cap = blocks / 2 > 1 ? blocks / 2 : 1;
  int s = 1;
  if (base < 152) {
    s = (int)(152 / (base > 0 ? base : 1));
  } else {  // several waves: take a second split when it evens out the last wave
    const double e1 = (double)base / (double)(((base + 151) / 152) * 152);
    const double e2 = (double)(2 * base) / (double)(((2 * base + 151) / 152) * 152);
    if (e1 < 0.9 && e2 > e1 + 0.05) s = 2;
  }
  if (s > cap) s = cap;
  if (s > 64) s = 64;
  return s < 1 ? 1 : s;
}

int launch_attn_tc(const void* q, const void* k_pool, const void* v_pool, int num_pages, int ps,
                   const int32_t* page_table, int max_pages, const int32_t* prefix_len, int max_prefix,
                   const void* k_tree, const void* v_tree, const uint64_t* mask, const int32_t* qo, int batch,
                   int total_nodes, int max_nodes, int hq, int hkv, int d, float sm_scale, void* out, float* lse,
                   void* ws, int32_t* status, cudaStream_t stream) {
  (void)ps;
  (void)d;
  const int G = hq / hkv;
  CUtensorMap tm_q, tm_kp, tm_vp, tm_kt, tm_vt;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kTcD, (cuuint64_t)hq, (cuuint64_t)total_nodes};
    const cuuint64_t str[2] = {(cuuint64_t)kTcD * 2, (cuuint64_t)hq * kTcD * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(kTcRows / G)};
    if (!encode_bf16(&tm_q, q, 3, dims, str, box)) return SPEC_ERR_CUDA;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kTcD, (cuuint64_t)hkv, (cuuint64_t)total_nodes};
    const cuuint64_t str[2] = {(cuuint64_t)kTcD * 2, (cuuint64_t)hkv * kTcD * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kTcKeys};
    if (!encode_bf16(&tm_kt, k_tree, 3, dims, str, box)) return SPEC_ERR_CUDA;
    if (!encode_bf16(&tm_vt, v_tree, 3, dims, str, box)) return SPEC_ERR_CUDA;
  }
  if (max_prefix > 0 && num_pages > 0 && k_pool != nullptr && v_pool != nullptr) {
    const cuuint64_t dims[4] = {(cuuint64_t)kTcD, 16, (cuuint64_t)hkv, (cuuint64_t)num_pages};
    const cuuint64_t str[3] = {(cuuint64_t)kTcD * 2, (cuuint64_t)16 * kTcD * 2, (cuuint64_t)hkv * 16 * kTcD * 2};
    const cuuint32_t box[4] = {64, 16, 1, 1};
    if (!encode_bf16(&tm_kp, k_pool, 4, dims, str, box)) return SPEC_ERR_CUDA;
    if (!encode_bf16(&tm_vp, v_pool, 4, dims, str, box)) return SPEC_ERR_CUDA;
  } else {  // no prefix anywhere: the pool maps are never used
    tm_kp = tm_kt;
    tm_vp = tm_vt;
  }
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
      return SPEC_ERR_CUDA;
    attr_set = true;
  }
  const int splits = attn_splits_tc(batch, max_nodes, hq, hkv, max_prefix);
  const int rows = total_nodes * hq;
  TcParams prm;
  prm.page_table = page_table;
  prm.max_pages = max_pages;
  prm.num_pages = num_pages;
  prm.prefix_len = prefix_len;
  prm.mask = mask;
  prm.mask_words = (max_nodes + 63) >> 6;
  prm.qo = qo;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.G = G;
  prm.splits = splits;
  prm.total_rows = rows;
  prm.scale_log2 = sm_scale * kLog2e;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.ws = AttnWs::at(ws, splits, rows, kTcD);
  prm.status = status;
  const dim3 grid(splits, ceil_div(max_nodes * G, kTcRows), batch * hkv);
  attn_tc_kernel<<<grid, kTcThreads, kSmemBytes, stream>>>(tm_q, tm_kp, tm_vp, tm_kt, tm_vt, prm);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (splits > 1) return launch_attn_combine(SPEC_BF16, prm.ws, splits, total_nodes, hq, kTcD, out, lse, stream);
  return SPEC_OK;
}

}  // namespace specv
