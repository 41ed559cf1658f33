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
// Query rows of (sequence b, KV head g) are node-major (row r -> node r / G, head
// g*G + r % G), so the G query heads of a KV head share every K/V tile (GQA); they
// are cut into M-tiles of 128 rows. A CTA = (key split s, pair of M-tiles, b x g):
// both tiles share each K/V block, which halves K/V traffic into shared memory and
// lets two softmax warp groups hide each other's latency (ping-pong). Keys come in
// blocks of 64: prefix blocks are 4 pages of 16 tokens, TMA-loaded page by page
// through the page table ([page][Hkv][16][128] bf16: a (page, head) is one 4 KB
// tile; page ids are fetched a batch of 8 blocks ahead); tree blocks are 64 rows of
// the dense tree K/V. Warp roles (352 threads):
//   warp 0      TMA producer: Q of both tiles, then K/V blocks into a 4-stage ring
//   warp 1      TMEM allocation (512 columns); lane 0 issues the MMAs of tile 0,
//   warp 10     lane 0 those of tile 1 (one issuing thread sustains only about one
//               tcgen05.mma per 100 cycles, so each tile gets its own):
//                 S_t[j%2] = Q_t K_j^T  (M 128, N 64, K 128; both operands K-major)
//                 O_t     += P_t V_j    (M 128, N 128, K 64; P from TMEM, V MN-major)
//   warps 2-5   softmax of tile 0, warps 6-9 softmax of tile 1: one query row per
//               thread (its TMEM lane); S row -> max / exp2 / row sum in registers,
//               P row -> bf16 pairs in TMEM over the S it came from, O rescaled in
//               TMEM only when the running max grows by more than 2^8.
// S is double-buffered in TMEM, so QK of block j+1 runs while the softmax of block j
// does. Every wait is bounded.
// The kernel has three forms: attn_tc_kernel<false, false, *> (bf16 cache, mask given),
// <true, false, *> (FP8 cache) and <false, true, *> (bf16 cache; the ancestor bits come
// from a walk of the parent array, staged in shared memory, instead of a mask). The last
// parameter selects longest-first dispatch: an unsplit launch over sequences of unequal
// length runs in waves, and ranking the work items by length before they are taken turns
// the in-order CTA dispatch into longest-first list scheduling (batch 32, prefixes of
// 512-8192: 190 -> 152 us).
// FP8 cache: the pool holds E4M3 codes ([page][Hkv][16][128] bytes, a 2 KB tile per
// (page, head)) with an fp32 scale per KV head for K and for V. The producer TMA-loads the
// prefix pages into a 3-stage ring of 16 KB code stages (half the bytes of bf16). Four
// more warps (11-14) widen each stage into a 3-stage bf16 ring, in the swizzled layout TMA
// would have written, with integer ops and a packed multiply (no conversion-pipe
// instructions); they also TMA-load the bf16 tree blocks, so one party fills every bf16
// stage and waits for each of its phases in order. The conversion is exact: every E4M3
// value is a bf16 value. The scales never touch the operands. The K scale multiplies the
// prefix blocks' score scale. The V scale is folded into the exponent of those blocks' P
// (2^(s - m + log2 v_scale)), and their row sum is divided by it.
// Keys are split when a short batch cannot fill 152 SMs otherwise, and for larger batches
// when the waves of CTAs end better split (the host's wave model). Each split CTA
// writes a partial per tile (O / l rounded to bf16 plus the split's log2-sum-exp;
// coalesced, L2-resident) and a small merge kernel, launched with programmatic
// serialization so it is resident before this grid ends, combines them by log-sum-exp.
// Rounding the normalised partials to bf16 adds at most 2^-9 max|v| to the output error
// (the merge is a convex combination of them).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "tc_ptx.cuh"

namespace specv {

constexpr int kTcRows = 128;
constexpr int kTcKeys = 64;
constexpr int kTcD = 128;
constexpr int kTcStages = 4;
constexpr int kTiles = 2;
constexpr int kTcThreads = 64 + kTiles * 128 + 32;  // + one more MMA-issuing warp
constexpr int kMma1Warp = kTcThreads / 32 - 1;     // the MMA issuer of tile 1
constexpr int kCvtWarps = 4;                       // FP8 cache: code -> bf16 converters
constexpr int kF8Stages = 3;
constexpr int kParMax = kMaxTreeNodes;             // nodes per tree (parent array staged in smem)
constexpr float kRescaleThr = 8.0f;            // log2 units: P entries stay <= 2^8
constexpr long long kWaitLimit = 4000000000LL;  // cycles (about 2 s) before a wait gives up

constexpr uint32_t kQSlab = kTcRows * 128;                  // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kQTile = 2 * kQSlab;
constexpr uint32_t kKVSlab = kTcKeys * 128;                 // 8 KB: 64 keys x 64 bf16
constexpr uint32_t kStageBytes = 4 * kKVSlab;               // K (2 slabs) + V (2 slabs)
constexpr uint32_t kF8Stage = 2 * kTcKeys * kTcD;           // 16 KB: K codes, then V codes
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kTiles * kQTile;
constexpr uint32_t kTmemCols = 512;                         // per tile: S0 | S1 | O (P aliases S)
constexpr uint32_t kIdescQK = tc::idesc_bf16(kTcRows, kTcKeys, 0);
constexpr uint32_t kIdescPV = tc::idesc_bf16(kTcRows, kTcD, 1);

// Shared-memory plan and block size of the bf16-cache (false) and FP8-cache (true) kernels;
// kPar: the variant that builds the ancestor bits from the parent array (bf16 cache).
template <bool kFp8, bool kPar = false>
struct TcCfg {
  static constexpr int kStages = kFp8 ? 3 : kTcStages;      // bf16 K/V ring
  static constexpr int kThreads = kTcThreads + (kFp8 ? 32 * kCvtWarps : 0);
  static constexpr uint32_t kOffF8 = kOffKV + kStages * kStageBytes;
  static constexpr uint32_t kOffBar = kOffF8 + (kFp8 ? kF8Stages * kF8Stage : 0);
  static constexpr uint32_t kOffPar = kOffBar + 256;          // parent arrays, one per tile
  static constexpr uint32_t kSmem = kOffPar + (kPar ? kTiles * kParMax * 4 : 0) + 1024;  // + alignment slack
  static constexpr int kFullCount = kFp8 ? kCvtWarps : 1;   // arrivals that fill a bf16 stage
};
static_assert(TcCfg<false>::kSmem <= 232448 && TcCfg<true>::kSmem <= 232448 && TcCfg<false, true>::kSmem <= 232448,
              "shared memory over the per-CTA limit");

struct TcParams {
  const int32_t* page_table;
  int max_pages, num_pages;
  const int32_t* prefix_len;
  const uint64_t* mask;   // ancestor bitsets [T][mask_words], or
  const int32_t* parent;  // the parent array (mask == nullptr): the bits come from a walk
  int mask_words;
  const int32_t* qo;
  int hq, hkv, G, splits, mtiles;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  uint4* part_o;       // split partials [tile group][S][128 rows][16 chunks]: O / l in bf16, 8 per chunk,
                       // chunk c of row r at position c ^ (r % 16)
  float* part_lse;     // [tile group][S][128 rows]: log2-sum-exp of the split's scores (-inf: empty)
  const float* kv_scale;  // FP8 cache: [2][Hkv] K then V scales (unused with a bf16 cache)
  int32_t* status;
  int batch;
  int early_reads;  // the inputs may be read before the grid-dependency wait (spec_set_early_reads)
};

// Longest-first order (kLpt instances) applies to unsplit launches of 2 .. kLptMax sequences
// that run in at most four waves.
constexpr int kLptMax = 256;

struct TcBars {
  uint64_t q_full, kv_full[kTcStages], kv_empty[kTcStages];
  uint64_t s_full[kTiles][2], p_full[kTiles], pv_done[kTiles], mma_fin[kTiles];
  uint64_t f8_full[kF8Stages], f8_empty[kF8Stages];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(TcBars) <= 256, "barrier block over its reserved bytes");

// One lane waits, the whole warp gets the answer: keeps warp-collective tcgen05.ld/st
// and __syncwarp on a converged warp even when a wait gives up.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = tc::mbar_wait(bar, parity, abort, kWaitLimit) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// the 128 softmax threads of one tile (barrier 1 + tile; 0 is __syncthreads)
__device__ __forceinline__ void tile_bar_sync(int tile) {
  if (tile == 0) asm volatile("bar.sync 1, 128;" ::: "memory");
  else asm volatile("bar.sync 2, 128;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Four E4M3 codes (byte i = element i) -> four bf16 (lo: elements 0, 1; hi: 2, 3), exactly.
// One byte permute puts each code in the low byte of a 16-bit lane with its sign replicated
// in the high byte; a shift and a mask then leave s | eeee << 7 | mmm << 4, the bf16 whose
// value is the code's times 2^-120 (the exponent biases, 127 and 7, differ by 120; zero and
// the subnormals line up as zero and subnormals). One packed bf16 multiply by 2^120 gives
// the value: every E4M3 value is a bf16 value, so the product is exact. (A NaN code, which
// a cache does not hold, reads as +-480.)
__device__ __forceinline__ uint32_t e4m3x2_lanes_to_bf16x2(uint32_t h) {
  const uint32_t x = (h << 4) & 0x87F087F0u;
  uint32_t y;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(x), "r"(0x7B807B80u));  // 2^120 in both lanes
  return y;
}

__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  uint32_t a, b;
  asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(a) : "r"(w));  // [sgn b1, b1, sgn b0, b0]
  asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(b) : "r"(w));  // [sgn b3, b3, sgn b2, b2]
  lo = e4m3x2_lanes_to_bf16x2(a);
  hi = e4m3x2_lanes_to_bf16x2(b);
}

// Two fp32 lanes per instruction (packed f32x2 on this architecture); each lane is the
// scalar operation, rounded to nearest.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rc, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5}; mov.b64 rc, {%6, %7};"
      " fma.rn.f32x2 rd, ra, rb, rc; mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5}; add.rn.f32x2 rd, ra, rb;"
      " mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Key split of a sequence, balanced to the 16-token page: the work units are the prefix
// pages, then each tree block as 4 units; split s takes units [s U / S, (s+1) U / S).
// Its prefix pages become blocks of up to 4 pages (the last one may hold fewer); a tree
// block belongs to the split holding its first unit.
struct TcSplit {
  int pg_lo, pg_hi;  // prefix pages [lo, hi)
  int npb;           // prefix blocks
  int tb_lo;         // first tree block
  int nb;            // blocks in all: prefix blocks, then tree blocks tb_lo, tb_lo + 1, ...
};

__device__ __forceinline__ TcSplit tc_split(int P, int N, int splits, int s) {
  const int np = (P + 15) >> 4;
  const int nt = (N + kTcKeys - 1) / kTcKeys;
  const long units = np + 4L * nt;
  const int lo = (int)((long)s * units / splits), hi = (int)((long)(s + 1) * units / splits);
  TcSplit r;
  r.pg_lo = min(lo, np);
  r.pg_hi = min(hi, np);
  r.npb = (r.pg_hi - r.pg_lo + 3) >> 2;
  const int t_lo = lo <= np ? 0 : (lo - np + 3) >> 2;            // first i with np + 4i >= lo
  const int t_hi = hi <= np ? 0 : min(nt, (hi - np + 3) >> 2);   // first i with np + 4i >= hi
  r.tb_lo = t_lo;
  r.nb = r.npb + max(0, t_hi - t_lo);
  return r;
}

template <bool kFp8, bool kPar, bool kLpt>
__global__ void __launch_bounds__(TcCfg<kFp8, kPar>::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kp,
                   const __grid_constant__ CUtensorMap tm_vp, const __grid_constant__ CUtensorMap tm_kt,
                   const __grid_constant__ CUtensorMap tm_vt, const TcParams p) {
  static_assert(!(kFp8 && kPar), "the FP8-cache kernel takes a mask");
  using Cfg = TcCfg<kFp8, kPar>;
  constexpr int kStages = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcBars& bars = *reinterpret_cast<TcBars*>(smem + Cfg::kOffBar);
  const uint32_t s_base = tc::smem_u32(smem);

  const int split = blockIdx.x, pair = blockIdx.y, bg = blockIdx.z;
  // the split merge (launched next) may be scheduled now: it waits for this grid to end
  pdl_trigger();
  if (threadIdx.x == 0) {  // descriptor fetches overlap the first loads of qo / prefix_len
    tc::prefetch_tmap(&tm_q);
    tc::prefetch_tmap(&tm_kp);
    tc::prefetch_tmap(&tm_vp);
    tc::prefetch_tmap(&tm_kt);
    tc::prefetch_tmap(&tm_vt);
  }
  // Unless the caller has declared that the kernel enqueued before this one writes none of
  // the inputs (everything but the mask or parent array), nothing is read before it ends.
  if (!p.early_reads) pdl_wait();
  const int G = p.G;
  int b = bg / p.hkv;
  const int g = bg - b * p.hkv;
  if (kLpt) {
    // Unsplit launch over sequences of unequal length: the grid runs in waves, and CTAs are
    // dispatched in index order, so CTA rank r takes the sequence with the r-th most work
    // (prefix + tree keys; ties by sequence id). The hardware's in-order dispatch then
    // places the longest items first and fills the last wave with the shortest.
    __shared__ int s_key[kLptMax];
    __shared__ int s_seq;
    for (int t = threadIdx.x; t < p.batch; t += blockDim.x)
      s_key[t] = __ldg(p.prefix_len + t) + (__ldg(p.qo + t + 1) - __ldg(p.qo + t));
    __syncthreads();
    for (int t = threadIdx.x; t < p.batch; t += blockDim.x) {
      const int k = s_key[t];
      int r = 0;
      for (int u = 0; u < p.batch; ++u) {
        const int ku = s_key[u];
        r += (ku > k || (ku == k && u < t)) ? 1 : 0;
      }
      if (r == b) s_seq = t;  // ranks are distinct: exactly one thread writes
    }
    __syncthreads();
    b = s_seq;
  }
  if (threadIdx.x < 32) {  // the sequence's page-table row into L2 while qo / prefix_len load
    for (int i = (threadIdx.x & 31) * 32; i < p.max_pages; i += 32 * 32)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.page_table + (size_t)b * p.max_pages + i));
  }
  const int base = __ldg(p.qo + b);
  const int N = __ldg(p.qo + b + 1) - base;
  const int P = __ldg(p.prefix_len + b);
  const int npt = kTcRows / G;  // tree nodes per M-tile
  const int node0 = 2 * pair * npt;
  const bool has1 = node0 + npt < N;  // tile 1 holds rows of this sequence
  const int ntiles = has1 ? 2 : 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the two exits below are taken by every split CTA of a tile alike (they depend on b, g, pair)
  if (node0 >= N) return;  // this pair of M-tiles is past the sequence's tree
  if (N > p.mask_words * 64 || P < 0 || P > p.max_pages * 16) {
    if (threadIdx.x == 0 && split == 0) {
      pdl_wait();  // (the status word is written in stream order)
      report(p.status, SPEC_ERR_CAPACITY);
    }
    return;
  }
  const TcSplit sr = tc_split(P, N, p.splits, split);
  const int nb = sr.nb;
  const int npb = sr.npb;

  // softmax-thread bookkeeping: warps 2-5 tile 0, warps 6-9 tile 1; TMEM lane quarter = warp % 4
  const int tile = warp >= 6 ? 1 : 0;
  const int row = (warp & 3) * 32 + lane;
  const int node_l = node0 + tile * npt + row / G;
  const int head = g * G + (row - (row / G) * G);
  const bool row_valid = node_l < N;
  const size_t orow = (size_t)(base + node_l) * p.hq + head;
  const int grp = (2 * pair + tile) + p.mtiles * bg;  // tile group of the key splits

  if (nb > 0) {
    const uint32_t bar_q = tc::smem_u32(&bars.q_full);
    auto bar_kvf = [&](int s) { return tc::smem_u32(&bars.kv_full[s]); };
    auto bar_kve = [&](int s) { return tc::smem_u32(&bars.kv_empty[s]); };
    auto bar_sf = [&](int t, int s) { return tc::smem_u32(&bars.s_full[t][s]); };
    auto bar_pf = [&](int t) { return tc::smem_u32(&bars.p_full[t]); };
    auto bar_pv = [&](int t) { return tc::smem_u32(&bars.pv_done[t]); };
    auto bar_f8f = [&](int s) { return tc::smem_u32(&bars.f8_full[s]); };
    auto bar_f8e = [&](int s) { return tc::smem_u32(&bars.f8_empty[s]); };
    volatile int* abort = &bars.abort;

    // Page ids of the producer's next 8 blocks, one per lane (lane l: block 8k + l/4,
    // page l%4), fetched a batch ahead so the page-table latency is paid once per 8 blocks.
    // Pages past the split (and invalid ids, reported) become the out-of-range id
    // num_pages, which TMA reads as zeros.
    auto fetch_pages = [&](int k) -> int {
      const int blk = 8 * k + (lane >> 2);
      const int lp = sr.pg_lo + blk * 4 + (lane & 3);
      int page = p.num_pages;
      if (blk < npb && lp < sr.pg_hi) {
        const int pg = __ldg(p.page_table + (size_t)b * p.max_pages + lp);
        if (pg >= 0 && pg < p.num_pages) page = pg;
        else report(p.status, SPEC_ERR_PAGE);
      }
      return page;
    };
    int pg_cur = 0, pg_nxt = 0;

    // K/V block j into ring stage j % kStages (the warp's lanes each issue one copy);
    // called for j = 0, 1, 2, ... in order by the whole producer warp. With an FP8 cache the
    // producer loads only the prefix blocks, into code stage j % kF8Stages; the converter
    // warps fill every bf16 stage (the tree blocks by TMA), so each ring has one filler that
    // waits for every phase of its "empty" barriers in order (a filler running two uses
    // ahead of a barrier would pass a parity wait one phase early).
    auto load_block = [&](int j) {
      const int st = j % kStages;
      const uint32_t dst0 = s_base + kOffKV + st * kStageBytes;
      if ((j & 7) == 0 && j > 0) {
        pg_cur = pg_nxt;
        pg_nxt = fetch_pages((j >> 3) + 1);
      }
      const int page_here = __shfl_sync(0xffffffffu, pg_cur, ((j & 7) << 2) + ((lane >> 2) & 3));
      if (kFp8 && j < npb) {
        const int s8 = j % kF8Stages;
        if (lane == 0) tc::mbar_arrive_expect_tx(bar_f8f(s8), kF8Stage);
        __syncwarp();
        if (lane < 16 && (lane & 3) < 2) {  // page lane >> 2, K (lane & 1 == 0) or V
          const int pp = lane >> 2, isv = lane & 1;
          const uint32_t dst = s_base + Cfg::kOffF8 + s8 * kF8Stage + isv * (kF8Stage / 2) + pp * 2048;
          tc::tma_load_4d(dst, isv ? &tm_vp : &tm_kp, bar_f8f(s8), 0, 0, g, page_here);
        }
        return;
      }
      if (lane == 0) tc::mbar_arrive_expect_tx(bar_kvf(st), kStageBytes);
      __syncwarp();
      if (j < npb) {
        if (lane < 16) {
          const int pp = lane >> 2, which = lane & 3;
          const int slab = which & 1, isv = which >> 1;
          const uint32_t dst = dst0 + isv * 2 * kKVSlab + slab * kKVSlab + pp * 2048;
          tc::tma_load_4d(dst, isv ? &tm_vp : &tm_kp, bar_kvf(st), slab * 64, 0, g, page_here);
        }
      } else if (lane < 4) {
        const int tb = sr.tb_lo + (j - npb);
        const int slab = lane & 1, isv = lane >> 1;
        const uint32_t dst = dst0 + isv * 2 * kKVSlab + slab * kKVSlab;
        tc::tma_load_3d(dst, isv ? &tm_vt : &tm_kt, bar_kvf(st), slab * 64, g, base + tb * 64);
      }
    };

    if (warp == 0) {
      // page ids (in flight while the barriers are set up), Q and the first block before
      // the CTA-wide sync: their latency overlaps the TMEM allocation
      pg_cur = fetch_pages(0);
      pg_nxt = fetch_pages(1);
      if (lane == 0) {
        tc::mbar_init(bar_q, 1);
        for (int s = 0; s < kStages; ++s) {
          tc::mbar_init(bar_kvf(s), Cfg::kFullCount);
          tc::mbar_init(bar_kve(s), ntiles);  // released by each tile's PV
        }
        if (kFp8)
          for (int s = 0; s < kF8Stages; ++s) {
            tc::mbar_init(bar_f8f(s), 1);
            tc::mbar_init(bar_f8e(s), kCvtWarps);  // released by each converter warp
          }
        for (int t = 0; t < kTiles; ++t) {
          tc::mbar_init(bar_sf(t, 0), 1);
          tc::mbar_init(bar_sf(t, 1), 1);
          tc::mbar_init(bar_pf(t), 128);
          tc::mbar_init(bar_pv(t), 1);
          tc::mbar_init(tc::smem_u32(&bars.mma_fin[t]), 1);
        }
        bars.abort = 0;
        tc::mbar_fence_init();
        tc::mbar_arrive_expect_tx(bar_q, ntiles * kQTile);
        for (int t = 0; t < ntiles; ++t) {
          const int n0 = base + node0 + t * npt;
          tc::tma_load_3d(s_base + kOffQ + t * kQTile, &tm_q, bar_q, 0, g * G, n0);
          tc::tma_load_3d(s_base + kOffQ + t * kQTile + kQSlab, &tm_q, bar_q, 64, g * G, n0);
        }
      }
      __syncwarp();
      if (!kFp8 || npb > 0) load_block(0);
    } else if (warp == 1) {
      tc::tmem_alloc(tc::smem_u32(&bars.tmem_base), kTmemCols);
      tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = bars.tmem_base;

    if (warp == 0) {
      // ---------------------------------------------------------------- TMA producer
      const int n_own = kFp8 ? npb : nb;  // blocks this warp loads
      int issued = n_own > 0 ? 1 : 0;
      for (int j = 1; j < n_own; ++j) {
        const uint32_t bar_free = kFp8 ? bar_f8e(j % kF8Stages) : bar_kve(j % kStages);
        const int parity = kFp8 ? ((j / kF8Stages) & 1) ^ 1 : ((j / kStages) & 1) ^ 1;
        if (!warp_wait(bar_free, parity, abort)) {
          if (lane == 0) report(p.status, SPEC_ERR_TIMEOUT);
          break;
        }
        load_block(j);
        issued = j + 1;
      }
      // leave no copy in flight: the last stages issued must have landed (the last
      // kF8Stages code stages, or the last kStages bf16 stages, are all distinct)
      if (lane == 0 && *abort) {
        int zero = 0;
        const int win = kFp8 ? kF8Stages : kStages;
        for (int j = max(0, issued - win); j < issued; ++j) {
          if (kFp8) tc::mbar_wait(bar_f8f(j % kF8Stages), (j / kF8Stages) & 1, &zero, kWaitLimit);
          else tc::mbar_wait(bar_kvf(j % kStages), (j / kStages) & 1, &zero, kWaitLimit);
        }
        tc::mbar_wait(bar_q, 0, &zero, kWaitLimit);
      }
    } else if (warp == 1 || warp == kMma1Warp) {
      // ---------------------------------------------------------------- MMA issuers
      // One issuing thread per M-tile (warp 1: tile 0, the last warp: tile 1): a thread
      // issues one tcgen05.mma about every 100 cycles whatever the shape, so two issuers
      // keep the tensor pipe twice as busy as one.
      const int t = warp == 1 ? 0 : 1;
      if (lane == 0 && t < ntiles) {
        const uint32_t qbuf = s_base + kOffQ + t * kQTile;
        auto qk = [&](int j) {
          const uint32_t kbuf = s_base + kOffKV + (j % kStages) * kStageBytes;
#pragma unroll
          for (int k = 0; k < kTcD / 16; ++k) {
            const uint64_t a = tc::sdesc_sw128(qbuf + (k >> 2) * kQSlab + (k & 3) * 32, 16, 1024);
            const uint64_t bdesc = tc::sdesc_sw128(kbuf + (k >> 2) * kKVSlab + (k & 3) * 32, 16, 1024);
            tc::mma_bf16(tbase + t * 256 + (j & 1) * 64, a, bdesc, kIdescQK, k > 0 ? 1u : 0u);
          }
          tc::mma_commit(bar_sf(t, j & 1));
        };
        bool ok = tc::mbar_wait(bar_q, 0, abort, kWaitLimit) &&
                  tc::mbar_wait(bar_kvf(0), 0, abort, kWaitLimit);
        if (ok) {
          tc::fence_after_sync();
          qk(0);
        }
        for (int j = 0; ok && j < nb; ++j) {
          if (j + 1 < nb) {  // S of the next block while the softmax works on this one
            const int st = (j + 1) % kStages;
            if (!tc::mbar_wait(bar_kvf(st), ((j + 1) / kStages) & 1, abort, kWaitLimit)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            qk(j + 1);
          }
          const uint32_t vbuf = s_base + kOffKV + (j % kStages) * kStageBytes + 2 * kKVSlab;
          if (!tc::mbar_wait(bar_pf(t), j & 1, abort, kWaitLimit)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          // P(j) sits in the first 32 columns of S buffer j % 2 (bf16 pairs); the QK that
          // next overwrites that buffer is issued after this PV by this thread (in order)
#pragma unroll
          for (int k = 0; k < kTcKeys / 16; ++k) {
            const uint64_t bdesc = tc::sdesc_sw128(vbuf + k * 2048, kKVSlab, 1024);
            tc::mma_bf16_ts(tbase + t * 256 + 128, tbase + t * 256 + (j & 1) * 64 + 8 * k, bdesc, kIdescPV,
                            (j > 0 || k > 0) ? 1u : 0u);
          }
          tc::mma_commit(bar_pv(t));
          tc::mma_commit(bar_kve(j % kStages));
        }
        if (!ok) report(p.status, SPEC_ERR_TIMEOUT);
        // every MMA this thread issued has completed before TMEM is released
        const uint32_t bar_fin = tc::smem_u32(&bars.mma_fin[t]);
        tc::mma_commit(bar_fin);
        int zero = 0;
        tc::mbar_wait(bar_fin, 0, &zero, kWaitLimit);
      }
      __syncwarp();
    } else if (kFp8 && warp >= kTcThreads / 32) {
      // ---------------------------------------------------------------- FP8 converters
      // The four warps fill every bf16 stage, block by block; each warp first waits for the
      // stage's previous use to be consumed (every phase in order), then adds its arrival.
      // Prefix block j: its 16 KB of codes (TMA, 128-byte swizzle: 16-byte chunk c of key
      // row r at c ^ (r % 8)) become the bf16 stage the MMAs read (slab d / 64, row r,
      // chunk (d % 64) / 8 at chunk ^ (r % 8)). A thread widens one 16-code chunk into two
      // bf16 chunks per step; the 8 lanes of a quarter-warp take 8 consecutive rows, so
      // their loads and stores land in 8 distinct bank groups. Tree block j: the first
      // converter warp TMA-loads the bf16 rows (expecting their bytes), the others arrive.
      const int ct = threadIdx.x - kTcThreads;
      const bool tma_warp = warp == kTcThreads / 32;
      int tree_issued = npb;  // tree blocks npb .. tree_issued - 1 were loaded by this warp
      for (int j = 0; j < nb; ++j) {
        const int st = j % kStages;
        if (j >= kStages && !warp_wait(bar_kve(st), ((j / kStages) & 1) ^ 1, abort)) {
          if (lane == 0) report(p.status, SPEC_ERR_TIMEOUT);
          break;
        }
        if (j >= npb) {
          if (tma_warp) {
            if (lane == 0) tc::mbar_arrive_expect_tx(bar_kvf(st), kStageBytes);
            __syncwarp();
            if (lane < 4) {
              const int tb = sr.tb_lo + (j - npb);
              const int slab = lane & 1, isv = lane >> 1;
              const uint32_t dst = s_base + kOffKV + st * kStageBytes + isv * 2 * kKVSlab + slab * kKVSlab;
              tc::tma_load_3d(dst, isv ? &tm_vt : &tm_kt, bar_kvf(st), slab * 64, g, base + tb * 64);
            }
            tree_issued = j + 1;
          } else if (lane == 0) {
            tc::mbar_arrive(bar_kvf(st));
          }
          continue;
        }
        const int s8 = j % kF8Stages;
        if (!warp_wait(bar_f8f(s8), (j / kF8Stages) & 1, abort)) {
          if (lane == 0) report(p.status, SPEC_ERR_TIMEOUT);
          break;
        }
        const uint8_t* src = smem + Cfg::kOffF8 + s8 * kF8Stage;
        uint8_t* dst = smem + kOffKV + st * kStageBytes;
#pragma unroll
        for (int it = 0; it < (int)(kF8Stage / 16) / (32 * kCvtWarps); ++it) {
          const int id = it * (32 * kCvtWarps) + ct;
          const int isv = id >> 9, cid = id & 511;
          const int r = (cid & 7) | ((cid >> 6) << 3);  // key row of the block
          const int cc = (cid >> 3) & 7;                // codes 16 cc .. 16 cc + 15
          const uint4 w = *reinterpret_cast<const uint4*>(src + isv * (kF8Stage / 2) + r * 128 + ((cc ^ (r & 7)) << 4));
          uint4 a, b2;
          e4m3x4_to_bf16x4(w.x, a.x, a.y);
          e4m3x4_to_bf16x4(w.y, a.z, a.w);
          e4m3x4_to_bf16x4(w.z, b2.x, b2.y);
          e4m3x4_to_bf16x4(w.w, b2.z, b2.w);
          uint8_t* row = dst + isv * 2 * kKVSlab + (cc >> 2) * kKVSlab + r * 128;
          const int ch = (cc & 3) * 2;
          *reinterpret_cast<uint4*>(row + ((ch ^ (r & 7)) << 4)) = a;
          *reinterpret_cast<uint4*>(row + (((ch + 1) ^ (r & 7)) << 4)) = b2;
        }
        tc::fence_proxy_async_smem();  // the tensor cores read these stores through the async proxy
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(bar_kvf(st));
          tc::mbar_arrive(bar_f8e(s8));
        }
      }
      // leave no tree copy in flight (the last kStages blocks use distinct stages)
      if (tma_warp && lane == 0 && *abort) {
        int zero = 0;
        for (int j = max(npb, tree_issued - kStages); j < tree_issued; ++j)
          tc::mbar_wait(bar_kvf(j % kStages), (j / kStages) & 1, &zero, kWaitLimit);
      }
    } else if (tile < ntiles) {
      // ---------------------------------------------------------------- softmax warps
      const uint32_t t_lane = tbase + tile * 256 + ((uint32_t)((warp & 3) * 32) << 16);
      const uint64_t* mrow = p.mask != nullptr ? p.mask + (size_t)(base + node_l) * p.mask_words : nullptr;
      const float sl2 = p.scale_log2;
      // FP8 cache: prefix scores scale by the K scale; prefix P carries the V scale in its
      // exponent and its row sum is divided by it
      float sl2_pre = sl2, lvs_pre = 0.f, ivs_pre = 1.f;
      if (kFp8) {
        const float ks = __ldg(p.kv_scale + g), vs = __ldg(p.kv_scale + p.hkv + g);
        sl2_pre = sl2 * ks;
        lvs_pre = log2f(vs);
        ivs_pre = 1.f / vs;
      }
      float m_run = -INFINITY, l = 0.f;
      bool ok = true;
      // The first tree block's mask word, fetched while the prefix blocks stream (the mask
      // may come from the kernel launched just before this one: wait for it first). Given
      // the parent array instead, the tile's 128 threads stage it in shared memory and each
      // row's bits for a tree block come from a walk up its ancestors ("EAGLE-2 deep
      // dive", core-implementation section: a node's mask row is the node and every
      // ancestor up to the root), checked as the mask kernel checks them.
      uint64_t bits_next = 0ull;
      const int32_t* spar = reinterpret_cast<const int32_t*>(smem + Cfg::kOffPar) + tile * kParMax;
      if (nb > npb) {
        pdl_wait();
        if (kPar) {
          int32_t* sp = const_cast<int32_t*>(spar);
          for (int i = threadIdx.x & 127; i < N; i += 128) sp[i] = __ldcg(p.parent + base + i);
          tile_bar_sync(tile);  // every softmax thread of the tile reaches this
        } else if (row_valid) {
          bits_next = __ldcg(mrow + sr.tb_lo);
        }
      }
      // ancestor bits of this row among tree keys 64 tb .. 64 tb + 63 (ids fall along the
      // walk, so it stops below the block; the walk for block 0 reaches the root)
      auto walk_bits = [&](int tb) -> uint64_t {
        const int lo = tb * kTcKeys;
        uint64_t bits = 0ull;
        int cur = node_l;
        while (true) {
          if (cur < lo) break;
          if (cur < lo + kTcKeys) bits |= 1ull << (cur - lo);
          const int pp = spar[cur];
          if (cur == 0 ? pp != -1 : (pp < 0 || pp >= cur)) {
            report(p.status, SPEC_ERR_PARENT);
            return 0ull;
          }
          if (cur == 0) break;
          cur = pp;
        }
        return bits;
      };
      for (int j = 0; j < nb; ++j) {
        if (!warp_wait(bar_sf(tile, j & 1), (j >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        float sv[kTcKeys];
        tc::tmem_ld32(t_lane + (j & 1) * 64, sv);
        tc::tmem_ld32(t_lane + (j & 1) * 64 + 32, sv + 32);
        tc::tmem_wait_ld();
        if (j < npb) {  // prefix: a length bound (the split's last page, P), never a mask
          const int nvalid = min(P, sr.pg_hi * 16) - (sr.pg_lo + 4 * j) * 16;
          if (nvalid < kTcKeys) {
#pragma unroll
            for (int c = 0; c < kTcKeys; ++c) sv[c] = c < nvalid ? sv[c] : -INFINITY;
          }
        } else {  // tree block: ancestor bits
          uint64_t bits;
          if (kPar) {
            bits = row_valid ? walk_bits(sr.tb_lo + (j - npb)) : 0ull;
          } else {
            bits = bits_next;
            if (row_valid && j + 1 < nb) bits_next = __ldcg(mrow + sr.tb_lo + (j + 1 - npb));
          }
#pragma unroll
          for (int c = 0; c < kTcKeys; ++c) sv[c] = ((bits >> c) & 1ull) ? sv[c] : -INFINITY;
        }
        // row max in four chains of three-input maxima (exact, any order)
        float mxc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float* v = sv + 16 * q;
          float m = fmax3(v[0], v[1], v[2]);
#pragma unroll
          for (int c = 3; c < 15; c += 2) m = fmax3(m, v[c], v[c + 1]);
          mxc[q] = fmaxf(m, v[15]);
        }
        const float mx0 = mxc[0], mx1 = mxc[1], mx2 = mxc[2], mx3 = mxc[3];
        const bool pre8 = kFp8 && j < npb;
        const float sc = pre8 ? sl2_pre : sl2;
        const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sc;  // sm_scale, scales > 0
        float alpha = 1.f;
        bool rescale = false;
        if (mx > -INFINITY && (m_run == -INFINITY || mx > m_run + kRescaleThr)) {
          alpha = m_run == -INFINITY ? 0.f : ex2_approx(m_run - mx);
          m_run = mx;
          rescale = j > 0;
        }
        float negm = m_run == -INFINITY ? 0.f : -m_run;  // all scores are -inf then
        if (pre8) negm += lvs_pre;
        uint32_t packed[kTcKeys / 2];
        // exponent arguments and row sums two lanes at a time (packed f32x2); per lane the
        // same roundings, in the same order, as the scalar form
        const float2 sc2 = make_float2(sc, sc), nm2 = make_float2(negm, negm);
        float2 r01 = make_float2(0.f, 0.f), r23 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kTcKeys; c += 4) {
          const float2 x01 = ffma2(make_float2(sv[c], sv[c + 1]), sc2, nm2);
          const float2 x23 = ffma2(make_float2(sv[c + 2], sv[c + 3]), sc2, nm2);
          const float2 p01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
          const float2 p23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
          r01 = fadd2(r01, p01);
          r23 = fadd2(r23, p23);
          packed[c >> 1] = pack_bf16x2(p01.x, p01.y);
          packed[(c >> 1) + 1] = pack_bf16x2(p23.x, p23.y);
        }
        float rsum = (r01.x + r01.y) + (r23.x + r23.y);
        if (pre8) rsum *= ivs_pre;
        l = l * alpha + rsum;
        if (j >= 1) {  // PV of the previous block done: O is stable
          if (!warp_wait(bar_pv(tile), (j - 1) & 1, abort)) {
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
        // P(j) into the S buffer it came from (S(j) is in registers now)
        tc::tmem_st32_u(t_lane + (j & 1) * 64, packed);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::mbar_arrive(bar_pf(tile));
      }
      ok = ok && warp_wait(bar_pv(tile), (nb - 1) & 1, abort);
      if (!ok && (threadIdx.x & 127) == 0) report(p.status, SPEC_ERR_TIMEOUT);
      tc::fence_after_sync();
      // O row out of TMEM: final output when unsplit, else this split's partial (O / l in
      // bf16, 8 values per 16-byte chunk, chunk-major) and its log2-sum-exp m + log2(l)
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // nothing is written before the previous kernel in the stream has finished (it may
      // still be reading the buffers this one is about to write)
      pdl_wait();
      uint4* po = p.part_o + ((size_t)grp * p.splits + split) * (kTcRows * kTcD / 8);
#pragma unroll 1
      for (int ch = 0; ch < kTcD / 32; ch += 2) {  // two 32-column loads per wait
        float o[64];
        __syncwarp();
        tc::tmem_ld32(t_lane + 128 + ch * 32, o);
        tc::tmem_ld32(t_lane + 128 + ch * 32 + 32, o + 32);
        tc::tmem_wait_ld();
        if (!ok) {
#pragma unroll
          for (int i = 0; i < 64; ++i) o[i] = 0.f;
        }
        uint4 c8[8];
#pragma unroll
        for (int v = 0; v < 8; ++v)
          c8[v] = make_uint4(pack_bf16x2(o[8 * v] * inv, o[8 * v + 1] * inv),
                             pack_bf16x2(o[8 * v + 2] * inv, o[8 * v + 3] * inv),
                             pack_bf16x2(o[8 * v + 4] * inv, o[8 * v + 5] * inv),
                             pack_bf16x2(o[8 * v + 6] * inv, o[8 * v + 7] * inv));
        if (p.splits == 1) {
          if (row_valid) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kTcD + ch * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v) dst[v] = c8[v];
          }
        } else {  // chunk-major: a warp's 32 rows write 512 contiguous bytes per chunk
#pragma unroll
          for (int v = 0; v < 8; ++v) po[(ch * 4 + v) * kTcRows + row] = c8[v];
        }
      }
      const float lse2 = (ok && l > 0.f) ? m_run + log2f(l) : -INFINITY;
      if (p.splits == 1) {
        if (row_valid && p.lse != nullptr) p.lse[orow] = lse2 * kLn2;
      } else {
        p.part_lse[((size_t)grp * p.splits + split) * kTcRows + row] = lse2;
      }
      __syncwarp();
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
      tc::fence_after_sync();
      tc::tmem_dealloc(tbase, kTmemCols);
    }
  } else if (warp >= 2 && warp < 2 + 4 * kTiles && tile < ntiles) {  // empty key split: contributes nothing to the merge
    pdl_wait();
    p.part_lse[((size_t)grp * p.splits + split) * kTcRows + row] = -INFINITY;
  }
}

// ------------------------------------------------------------------ merge of the key splits
// One thread per (tile group, 16-byte chunk, row): a warp reads 32 consecutive rows of one
// chunk, 512 contiguous bytes per split. Launched with programmatic serialization right
// after the attention kernel (which lets it start at once): it waits for that grid to
// finish, then O = sum_s 2^(lse_s - M) O_s / L with M = max_s lse_s, L = sum_s 2^(lse_s - M),
// and the row's log-sum-exp M + log2 L (natural log on output).
struct TcMergeParams {
  const uint4* part_o;
  const float* part_lse;
  const int32_t* qo;
  int splits, mtiles, hkv, hq, G;
  long groups;
  __nv_bfloat16* out;
  float* lse;
};

constexpr int kMergeThreads = 64;  // small CTAs: one fits beside an attention CTA on an SM
constexpr int kMaxSplits = 32;  // attn_splits_tc never returns more

// MAXS >= splits: the unrolled load batch, sized to the launch so the registers stay few
// enough for a merge CTA to sit beside an attention CTA on one SM.
template <int MAXS>
__global__ void __launch_bounds__(kMergeThreads) attn_tc_merge_kernel(const TcMergeParams p) {
  pdl_trigger();  // the next kernel may be scheduled: whatever it reads, it waits for this grid
  const long idx = (long)blockIdx.x * kMergeThreads + threadIdx.x;
  if (idx >= p.groups * 16 * kTcRows) return;
  const int gt = (int)(idx / (16 * kTcRows));
  const int rem = (int)(idx - (long)gt * 16 * kTcRows);
  const int c = rem / kTcRows, r = rem - (rem / kTcRows) * kTcRows;
  const int tt = gt % p.mtiles, bg = gt / p.mtiles;
  const int b = bg / p.hkv, g = bg - (bg / p.hkv) * p.hkv;
  const int G = p.G;
  const int node_l = tt * (kTcRows / G) + r / G;
  const int base = __ldg(p.qo + b);  // qo is an input: safe to read before the wait
  if (node_l >= __ldg(p.qo + b + 1) - base) return;
  pdl_wait();  // the attention grid has finished: its partials are visible
  // every load (split statistics and partial rows) is issued before any is used: one
  // round trip to L2
  const int S = p.splits;  // <= MAXS
  const float* ls = p.part_lse + (size_t)gt * S * kTcRows + r;
  const uint4* po = p.part_o + (size_t)gt * S * (kTcRows * kTcD / 8) + c * kTcRows + r;
  float lv[MAXS];
  uint4 q[MAXS];
#pragma unroll
  for (int s = 0; s < MAXS; ++s) {
    lv[s] = s < S ? __ldcg(ls + (size_t)s * kTcRows) : -INFINITY;
    q[s] = s < S ? __ldcg(po + (size_t)s * (kTcRows * kTcD / 8)) : make_uint4(0, 0, 0, 0);
  }
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < MAXS; ++s) M = fmaxf(M, lv[s]);
  float L = 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < MAXS; ++s) {
    if (lv[s] == -INFINITY) continue;  // an empty split (or s >= S): its row holds no partial
    const float w = ex2_approx(lv[s] - M);
    L += w;
    const uint32_t uu[4] = {q[s].x, q[s].y, q[s].z, q[s].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc[2 * k] = fmaf(__uint_as_float(uu[k] << 16), w, acc[2 * k]);
      acc[2 * k + 1] = fmaf(__uint_as_float(uu[k] & 0xFFFF0000u), w, acc[2 * k + 1]);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int head = g * G + (r - (r / G) * G);
  const size_t orow = (size_t)(base + node_l) * p.hq + head;
  *reinterpret_cast<uint4*>(p.out + orow * kTcD + c * 8) =
      make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                 pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
  if (c == 0 && p.lse != nullptr) p.lse[orow] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

// ------------------------------------------------------------------------------ host

// The driver's tensor-map encoder, looked up once per process (a thread-safe static; the
// entry point is the same for every device). nullptr when there is no driver.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return nullptr;
  }();
  return fn;
}

// Tensor map with 128-byte swizzle and zero fill out of bounds; dims/box innermost first.
static bool encode_tiled(CUtensorMap* m, CUtensorMapDataType type, const void* ptr, int rank,
                         const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, type, rank, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool encode_bf16(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                        const cuuint32_t* box) {
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, rank, dims, strides, box);
}

// The shapes the tensor-core kernel serves (every bf16 call with d = 128 must be one of
// them: such a call never runs on the CUDA-core kernel instead).
bool attn_tc_shape(int dtype, int hq, int hkv, int d, int page_size, int max_nodes) {
  if (dtype != SPEC_BF16 || d != kTcD || page_size != 16 || hkv <= 0 || hq % hkv) return false;
  const int G = hq / hkv;
  return G >= 1 && G <= kTcRows && kTcRows % G == 0 && max_nodes >= 1 && max_nodes <= kMaxTreeNodes;
}

// The driver entry point that encodes tensor maps was found (false on a host without a
// CUDA driver): a tensor-core call without it fails with SPEC_ERR_CUDA.
bool attn_tc_ready() { return tensor_map_encoder() != nullptr; }

static int sm_count() {
  static PerDevice cache;
  const int n = per_device(cache, [](int dev) {
    int v = 0;
    return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0 ? v : 0;
  });
  return n > 0 ? n : 152;  // no device visible (sizing on a build machine): the GB300 count
}

static int tc_mtiles(int max_nodes, int G) { return ceil_div(max_nodes * G, kTcRows); }

// Key splits per CTA work item (sequence, KV head, pair of M-tiles), from the sizes alone
// (the per-sequence lengths stay on the device). One CTA fits on an SM (over 197 KB of
// shared memory).
// - Fewer items than SMs: enough splits that the items x splits CTAs cover the SMs, never
//   more CTAs than SMs.
// - Otherwise the CTAs run in waves. The count S in 1..8 minimises
//   ceil(items * S / SMs) * (ceil(blocks / S) + 4), where blocks = the longest sequence's
//   key blocks and 4 blocks stand for a CTA's fixed cost (prologue, partials, merge share).
//   A batch of long sequences of equal length then stops losing its last, partly filled
//   wave. The keys are split only when that modelled cost falls at least 8% below the
//   unsplit one: the merge kernel is not in the model, and a split that gains less loses
//   to it (batch 64, 2048-token prefixes, 64-node trees: 2 splits modelled 1% better,
//   measured 6% slower).
// At least two key blocks per split, at most 32 splits. The split merge waits for the
// whole attention grid (programmatic launch releases it only once every attention CTA
// has started), so any number of waves is safe.
int attn_splits_tc(int batch, int max_nodes, int hq, int hkv, int max_prefix) {
  if (hkv <= 0 || hq % hkv) return 1;
  const int G = hq / hkv;
  const long items = (long)batch * hkv * ceil_div(tc_mtiles(max_nodes, G), kTiles);
  const int blocks = ceil_div(max_prefix, kTcKeys) + ceil_div(max_nodes, kTcKeys);
  const long sms = sm_count();
  long s = 1;
  if (items > 0 && items < sms) {
    s = sms / items;
  } else if (items > 0) {
    long best = -1;
    for (long c = 1; c <= 8; ++c) {
      const long cost = ((items * c + sms - 1) / sms) * ((blocks + c - 1) / c + 4);
      if (best < 0 || cost < best) {
        best = cost;
        s = c;
      }
    }
    const long unsplit = ((items + sms - 1) / sms) * (blocks + 4);
    if (s > 1 && best * 100 > unsplit * 92) s = 1;  // less than an 8% modelled gain
  }
  if (s > blocks / 2) s = blocks / 2;
  if (s > kMaxSplits) s = kMaxSplits;
  return s < 1 ? 1 : (int)s;
}

struct TcWs {
  size_t ml, o, total;
  static TcWs make(long groups, int splits) {
    TcWs w;
    size_t off = 0;
    w.ml = off;       off = align_up(off + sizeof(float) * groups * splits * kTcRows, 256);
    w.o = off;        off = align_up(off + sizeof(__nv_bfloat16) * groups * splits * kTcRows * kTcD, 256);
    w.total = off;
    return w;
  }
};

size_t attn_tc_ws_bytes(int batch, int max_nodes, int hq, int hkv, int max_prefix) {
  const int s = attn_splits_tc(batch, max_nodes, hq, hkv, max_prefix);
  if (s <= 1) return 0;
  const long groups = (long)batch * hkv * tc_mtiles(max_nodes, hq / hkv);
  return TcWs::make(groups, s).total;
}

using TcKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TcParams);

// The instance for a cache kind (0 bf16 with a mask, 1 FP8, 2 bf16 with the parent array)
// and dispatch order (lpt: longest sequence first).
static TcKernel tc_kernel_for(int variant, bool lpt) {
  switch (variant * 2 + (lpt ? 1 : 0)) {
    case 0: return attn_tc_kernel<false, false, false>;
    case 1: return attn_tc_kernel<false, false, true>;
    case 2: return attn_tc_kernel<true, false, false>;
    case 3: return attn_tc_kernel<true, false, true>;
    case 4: return attn_tc_kernel<false, true, false>;
    default: return attn_tc_kernel<false, true, true>;
  }
}

int launch_attn_tc(const void* q, const void* k_pool, const void* v_pool, int num_pages, int ps,
                   const int32_t* page_table, int max_pages, const int32_t* prefix_len, int max_prefix,
                   const void* k_tree, const void* v_tree, const uint64_t* mask, const int32_t* qo, int batch,
                   int total_nodes, int max_nodes, int hq, int hkv, int d, float sm_scale, void* out, float* lse,
                   void* ws, int32_t* status, cudaStream_t stream, const float* kv_scale, const int32_t* parent) {
  (void)ps;
  const bool fp8 = kv_scale != nullptr;
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
  if (max_prefix > 0 && num_pages > 0 && k_pool != nullptr && v_pool != nullptr && !fp8) {
    const cuuint64_t dims[4] = {(cuuint64_t)kTcD, 16, (cuuint64_t)hkv, (cuuint64_t)num_pages};
    const cuuint64_t str[3] = {(cuuint64_t)kTcD * 2, (cuuint64_t)16 * kTcD * 2, (cuuint64_t)hkv * 16 * kTcD * 2};
    const cuuint32_t box[4] = {64, 16, 1, 1};
    if (!encode_bf16(&tm_kp, k_pool, 4, dims, str, box)) return SPEC_ERR_CUDA;
    if (!encode_bf16(&tm_vp, v_pool, 4, dims, str, box)) return SPEC_ERR_CUDA;
  } else if (max_prefix > 0 && num_pages > 0 && k_pool != nullptr && v_pool != nullptr) {
    // E4M3 codes: one 16-token x 128-code tile (2 KB) per (page, head), 128-byte rows
    const cuuint64_t dims[4] = {(cuuint64_t)kTcD, 16, (cuuint64_t)hkv, (cuuint64_t)num_pages};
    const cuuint64_t str[3] = {(cuuint64_t)kTcD, (cuuint64_t)16 * kTcD, (cuuint64_t)hkv * 16 * kTcD};
    const cuuint32_t box[4] = {(cuuint32_t)kTcD, 16, 1, 1};
    if (!encode_tiled(&tm_kp, CU_TENSOR_MAP_DATA_TYPE_UINT8, k_pool, 4, dims, str, box)) return SPEC_ERR_CUDA;
    if (!encode_tiled(&tm_vp, CU_TENSOR_MAP_DATA_TYPE_UINT8, v_pool, 4, dims, str, box)) return SPEC_ERR_CUDA;
  } else {  // no prefix anywhere: the pool maps are never used
    tm_kp = tm_kt;
    tm_vp = tm_vt;
  }
  const bool par = mask == nullptr && parent != nullptr;
  const int variant = fp8 ? 1 : par ? 2 : 0;
  const int splits = attn_splits_tc(batch, max_nodes, hq, hkv, max_prefix);
  // (past four waves the last one is a small share of the grid: no ranking then)
  const bool lpt = splits == 1 && batch > 1 && batch <= kLptMax &&
                   (long)batch * hkv * ceil_div(tc_mtiles(max_nodes, G), kTiles) <= 4L * sm_count();
  const TcKernel kern = tc_kernel_for(variant, lpt);
  const int smem = variant == 1 ? TcCfg<true>::kSmem : variant == 2 ? TcCfg<false, true>::kSmem : TcCfg<false>::kSmem;
  static PerDevice attr_set[6];  // the raised shared-memory limit, set once per device and instance
  if (per_device(attr_set[variant * 2 + (lpt ? 1 : 0)], [kern, smem](int) {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess ? 1 : 0;
      }) == 0)
    return SPEC_ERR_CUDA;
  const int mtiles = tc_mtiles(max_nodes, G);
  TcParams prm;
  prm.page_table = page_table;
  prm.max_pages = max_pages;
  prm.num_pages = num_pages;
  prm.prefix_len = prefix_len;
  prm.mask = mask;
  prm.parent = par ? parent : nullptr;
  prm.mask_words = (max_nodes + 63) >> 6;
  prm.qo = qo;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.G = G;
  prm.splits = splits;
  prm.mtiles = mtiles;
  prm.scale_log2 = sm_scale * kLog2e;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  const long groups = (long)batch * hkv * mtiles;
  const TcWs w = TcWs::make(groups, splits);
  uint8_t* wb = static_cast<uint8_t*>(ws);
  prm.part_o = splits > 1 ? reinterpret_cast<uint4*>(wb + w.o) : nullptr;
  prm.part_lse = splits > 1 ? reinterpret_cast<float*>(wb + w.ml) : nullptr;
  prm.kv_scale = kv_scale;
  prm.status = status;
  prm.batch = batch;
  prm.early_reads = early_reads() ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(splits, ceil_div(mtiles, kTiles), batch * hkv);
  cfg.blockDim = dim3(fp8 ? TcCfg<true>::kThreads : TcCfg<false>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // programmatic serialization: the prologue (barriers, TMEM, Q and first K/V loads)
  // overlaps the mask kernel; the softmax waits for it before the first tree block
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = cudaLaunchKernelEx(&cfg, kern, tm_q, tm_kp, tm_vp, tm_kt, tm_vt, prm);
  if (le != cudaSuccess) return SPEC_ERR_CUDA;
  if (splits > 1) {
    TcMergeParams mp;
    mp.part_o = prm.part_o;
    mp.part_lse = prm.part_lse;
    mp.qo = qo;
    mp.splits = splits;
    mp.mtiles = mtiles;
    mp.hkv = hkv;
    mp.hq = hq;
    mp.G = G;
    mp.groups = groups;
    mp.out = prm.out;
    mp.lse = lse;
    const long threads = groups * 16 * kTcRows;
    const dim3 grid((unsigned)ceil_div(threads, (long)kMergeThreads)), block(kMergeThreads);
    cudaError_t e;
    if (splits <= 8) e = launch_pdl(attn_tc_merge_kernel<8>, grid, block, 0, stream, mp);
    else if (splits <= 16) e = launch_pdl(attn_tc_merge_kernel<16>, grid, block, 0, stream, mp);
    else if (splits <= 24) e = launch_pdl(attn_tc_merge_kernel<24>, grid, block, 0, stream, mp);
    else e = launch_pdl(attn_tc_merge_kernel<kMaxSplits>, grid, block, 0, stream, mp);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace specv
