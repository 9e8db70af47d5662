// Internal definitions shared by the planner, decode and reduce kernels and the C ABI:
// the kernel variant chosen for a configuration, the workspace layout, and thin
// wrappers over the sm_100-family PTX used for staging (mbarrier, TMA, cp.async).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pa.h"

namespace pa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kFull = 0xffffffffu;

enum KvKind { KV_BF16 = 0, KV_FP16 = 1, KV_FP8 = 2 };
enum QKind { Q_BF16 = 0, Q_FP16 = 1 };

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int round_up(int a, int b) { return ceil_div(a, b) * b; }
__host__ __device__ constexpr size_t round_up_sz(size_t a, size_t b) { return (a + b - 1) / b * b; }

// ---------------------------------------------------------------------------------
// Kernel variant.  M = G * Sq query rows share one kv head.  Rows are processed in
// tiles of `mp` (a power of two); a unit of work is one (sequence, kv head, row
// tile), and `tt` is the number of tokens staged per pipeline stage.
struct Variant {
  int path;         // 0: CUDA-core kernel, 1: mma.sync kernel, 2: tcgen05 kernel
  int rows;         // M = G * Sq
  int mp;           // rows per unit (padded to a power of two)
  int rb;           // row tiles per kv head
  int tt;           // tokens per stage (tile)
  int units;        // B * Hkv * rb
  int ctas;         // persistent grid size C
  int ctas_per_sm;  // decode CTAs resident per SM
  int bpe;          // bytes per cache element
  int item_cost;    // tokens of work a unit costs on top of its own (a tile multiple)
  int ns_dec;       // the decode merges a split unit of at most this many pieces itself
  int sms;          // SMs of the device when the grid was sized from it, else 0
};

// Largest row tile of the CUDA-core decode kernel.
constexpr int kSimtMaxRows = 8;
// Bytes of one K (or V) tile of a stage.
constexpr int kTileBytes = 16384;
// Tokens of one tile of the tcgen05 kernel (one MMA step: 16 KB of K at head dim 128, 32 KB
// at 256).
constexpr int kTcStepTokens = 64;
// Fixed cost of a work item, in tiles of streaming: a CTA that starts a unit pays for the
// unit's epilogue and for refilling its copy pipeline (about 5 us at the ~22 GB/s one CTA
// streams, or three tiles of K and V), so the planner counts every unit that long.
constexpr int kItemCostTiles = 3;
// The same for the tcgen05 kernel, in 64-token steps.  Per-CTA exit times against the number
// of items a CTA holds put an extra item at about 5 us on the long-context Sq = 4 decode
// (head dim 128, bf16) and 9-10 us on the head-dim-256 Sq = 64 one, both about 430 tokens of
// the CTA's own streaming (the query rows into tensor memory, the last PVs, the two token
// streams' merge and the output or partial); seven steps balance the CTAs' exits there (the
// long-context decode went from 37.5 to 35.0 us), and on the fp8 decodes too.
constexpr int kTcItemCostSteps = 7;

inline int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// CTAs of the decode instance for these parameters that fit on one SM.
int simt_ctas_per_sm(int head_dim, int mp, int kvk, bool toks);
int mma_ctas_per_sm(int head_dim, int mp, int kvk, bool toks);
// Largest row tile of the tensor-core decode kernel.
constexpr int kMmaMaxRows = 64;

// The most pieces of a split unit the decode kernel merges itself (1: none).  Under
// PA_MERGE_AUTO every split unit is left to the reduce kernel: a merge inside the decode runs
// on one SM after that CTA's own work (on the tcgen05 kernel, on the softmax warps, holding
// the tensor-memory accumulator), so it lengthens the decode's tail, while the reduce kernel
// spreads the rows of all split units over the GPU, a warp per row for units of few pieces
// (measured on GB300, step times with the merge in the reduce kernel against two-piece units
// merged in the decode: batched GQA 63.8 against 70.9 us, 64-row fp8 134 against 158 us,
// head-dim-256 Sq = 64 B = 8 203 against 231 us, the rest equal).
inline int decode_merge_limit(int split_merge, int path) {
  (void)path;
  if (split_merge == PA_MERGE_IN_DECODE) return 1 << 30;
  return 1;
}

// Query rows per kv head above which a 128-dim head runs on the tcgen05 kernel.
constexpr int kTcMinRows = 33;

// Everything but the grid size, which needs the device (see api.cu).
// Every cache whose tile row is at least one 128-byte slab runs on tensor cores: a 16-bit
// cache with head dim 128 or 256, or an fp8 cache with head dim 128 (any scale mode), and
// more than 32 query rows per kv head on tcgen05 (row tiles of 64 or 128, the MMA always
// 128 rows), otherwise on mma.sync with the rows padded to 16, 32 or 64 (larger groups cut
// into 64-row tiles): even a tile of one real row in sixteen costs less there than
// CUDA-core arithmetic.  A 64-dim fp8 cache (64-byte rows) runs on the CUDA-core kernel, in
// tiles of up to 8 rows.
inline Variant make_variant(const pa_config& c) {
  Variant v{};
  v.rows = (c.num_q_heads / c.num_kv_heads) * c.max_q_len;
  v.bpe = c.kv_dtype == PA_FP8_E4M3 ? 1 : 2;
  v.path = c.head_dim * v.bpe >= 128 ? 1 : 0;
  if (v.path == 1 && c.head_dim >= 128 && v.rows >= kTcMinRows &&
      (c.kv_dtype != PA_FP8_E4M3 || c.head_dim == 128))
    v.path = 2;
  if (v.path == 2)
    v.mp = v.rows <= 64 ? 64 : 128;
  else if (v.path == 1)
    v.mp = v.rows >= kMmaMaxRows ? kMmaMaxRows : (v.rows <= 16 ? 16 : pow2_at_least(v.rows));
  else
    v.mp = v.rows <= kSimtMaxRows ? pow2_at_least(v.rows) : kSimtMaxRows;
  v.rb = ceil_div(v.rows, v.mp);
  v.tt = v.path == 2 ? kTcStepTokens : kTileBytes / (c.head_dim * v.bpe);
  // the item cost is measured in 16 KB tiles of streaming (tcgen05: in steps), rounded up
  // to whole tiles
  v.item_cost = v.path == 2 ? kTcItemCostSteps * kTcStepTokens
                            : round_up(kItemCostTiles * (kTileBytes / (c.head_dim * v.bpe)), v.tt);
  v.units = c.batch * c.num_kv_heads * v.rb;
  const int kvk = c.kv_dtype == PA_FP8_E4M3 ? 2 : (c.kv_dtype == PA_FP16 ? 1 : 0);
  const bool toks = c.kv_scale_mode == PA_SCALE_PER_TOKEN;
  v.ctas_per_sm = v.path == 2   ? 1
                  : v.path == 1 ? mma_ctas_per_sm(c.head_dim, v.mp, kvk, toks)
                                : simt_ctas_per_sm(c.head_dim, v.mp, kvk, toks);
  v.ns_dec = decode_merge_limit(c.split_merge, v.path);
  v.ctas = 0;
  return v;
}

// ---------------------------------------------------------------------------------
// Workspace layout (byte offsets from ws, every section 256-byte aligned).
//   header     int32[64]: [0] flags, [1] chunk, [2] active CTAs, [3] items,
//                         [4] units left to the reduce kernel, [5] how many of them have
//                         at most kReduceWarpPieces pieces
//   item_off   int32[C + 1]      first work item of each CTA
//   first_item int4[C]           each CTA's first work item again ((0, 0, 0, -1) if none), so
//                                that a CTA reads it together with its offsets
//   items      int4[C + units]   (unit, t0, t1, partial slot or -1)
//   unit_info  int2[units]       (slot of the first piece, number of pieces); piece s > 0
//                                of a unit sits in slot 2 * (first / 2 + s)
//   unit_cnt   int32[units]      pieces of each unit finished so far (merge in decode)
//   red_units  int32[units]      units the reduce kernel merges: those of at most
//                                kReduceWarpPieces pieces, then the others, each in unit order
//   seq_start  int32[B + 1]      planner scratch for very large batches
//   seq_len    int32[B]
//   o_part     f32[2C * mp * D]  normalised partial outputs (CTA c: slots 2c, 2c + 1)
//   lse_part   f32[2C * mp]      their log2-sum-exp
struct WsLayout {
  size_t header, item_off, first_item, items, unit_info, unit_cnt, red_units, seq_start, seq_len,
      o_part, lse_part, total;
};

inline WsLayout ws_layout(const pa_config& c, const Variant& v) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = round_up_sz(off + bytes, 256);
    return at;
  };
  const size_t max_items = (size_t)v.ctas + (size_t)v.units;
  L.header = take(64 * sizeof(int32_t));
  L.item_off = take(((size_t)v.ctas + 1) * sizeof(int32_t));
  L.first_item = take((size_t)v.ctas * sizeof(int4));
  L.items = take(max_items * sizeof(int4));
  L.unit_info = take((size_t)v.units * sizeof(int2));
  L.unit_cnt = take((size_t)v.units * sizeof(int32_t));
  L.red_units = take((size_t)v.units * sizeof(int32_t));
  L.seq_start = take(((size_t)c.batch + 1) * sizeof(int32_t));
  L.seq_len = take((size_t)c.batch * sizeof(int32_t));
  const size_t slots = 2 * (size_t)v.ctas;
  L.o_part = take(slots * (size_t)v.mp * c.head_dim * sizeof(float));
  L.lse_part = take(slots * (size_t)v.mp * sizeof(float));
  L.total = off;
  return L;
}

enum HeaderSlot {
  HDR_FLAGS = 0, HDR_CHUNK = 1, HDR_ACTIVE = 2, HDR_ITEMS = 3, HDR_NRED = 4, HDR_NRED_SMALL = 5
};

// Split units of at most this many pieces are merged by the reduce kernel one warp per row
// (all of a row's pieces loaded at once); larger ones with eight warps per row.
constexpr int kReduceWarpPieces = 16;

// Division by a run-time constant d in [1, 2^31) of a dividend n in [0, 2^31) with one
// multiply-high, add and shift (the round-up multiplier method of Granlund and Montgomery,
// "Division by invariant integers using multiplication", 1994): with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1, n / d = (mulhi(n, m) + n) >> s.
struct FastDiv {
  uint32_t d, m, s;
  __host__ __device__ FastDiv() : d(1), m(1), s(0) {}
  __host__ __device__ explicit FastDiv(uint32_t div) : d(div) {
    s = 0;
    while ((1u << s) < d) ++s;
    m = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << s) - d)) / d) + 1;
  }
  __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
#if defined(__CUDA_ARCH__)
    const uint32_t hi = __umulhi(n, m);
#else
    const uint32_t hi = (uint32_t)(((uint64_t)n * m) >> 32);
#endif
    return (hi + n) >> s;
  }
  __host__ __device__ __forceinline__ uint32_t mod(uint32_t n) const { return n - div(n) * d; }
};

// log2 of a power of two.
__host__ __device__ constexpr int ilog2(uint32_t x) { return x <= 1 ? 0 : 1 + ilog2(x >> 1); }

// Partial slot of piece s of a unit whose first piece sits in slot `first`.
__host__ __device__ inline int piece_slot(int first, int s) {
  return s == 0 ? first : 2 * ((first >> 1) + s);
}

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device, once per
// device: the attribute belongs to the device, so a process that launches on several GPUs
// sets it on each.  `done` is the caller's per-kernel bit set of devices already set up
// (devices past the 64th are set up on every launch).
inline cudaError_t set_smem_attr_once(std::atomic<uint64_t>& done, const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launch helpers implemented in plan.cu / decode_*.cu / reduce.cu.
struct ProblemArgs {
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* q_lens;
  int batch, max_q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks, num_blocks;
  int causal;
};

cudaError_t launch_plan(const ProblemArgs& a, const Variant& v, const WsLayout& L, char* ws,
                        cudaStream_t s);

struct DecodeArgs {
  ProblemArgs p;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const float* k_scale;
  const float* v_scale;
  int scale_mode;
  float qk_scale;  // sm_scale * log2(e)
  void* out;
  float* lse;
  char* ws;
  WsLayout L;
  Variant v;
  int q_kind, kv_kind;
};

// Returns cudaErrorNotSupported when no kernel instance matches.
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t s);

cudaError_t launch_reduce(const DecodeArgs& a, cudaStream_t s);

// ---------------------------------------------------------------------------------
// Device helpers.
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Longest a kernel waits for one of its own copies before it gives up.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Bounded wait on phase `parity`.  Returns false when the wait ran out or another warp of
// the CTA has already given up (*abort != 0); the caller then records the failure and
// stops waiting, so the kernel always ends.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*abort) return false;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// Bounded wait that ignores the abort flag: used at exit, to let copies already in
// flight land before the CTA's shared memory is released.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// A box of a 4-D tensor into L2 (no shared-memory destination, no barrier): the same
// coordinates as the load of that box.
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* m, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// 4-D tiled TMA load of one box into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
      : "memory");
}

// Untiled bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// global into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32x2 multiply-add (sm_100 family): d = a * b + c, lane-wise on float2.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}

// Programmatic dependent launch: wait until the preceding kernel in the stream has
// completed and its writes are visible / let the following kernel start launching.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over the first `count` threads of the CTA (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

#endif  // __CUDACC__

}  // namespace pa
