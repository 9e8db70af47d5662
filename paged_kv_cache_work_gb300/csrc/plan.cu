// Planner: turns the device-resident context lengths into the persistent grid's work list.
//
// The split follows "Optimize paged-attention metadata decode" (FlyDSL PR #910, Summary and
// Changes): metadata is generated on the device for a persistent decode grid sized as SMs x
// a grid multiplier (default 1, the safe one-grid-per-CU choice), and ranges that a unit
// does not finish in one piece are merged by a split reducer.  Here every unit (sequence,
// kv head, row tile) contributes its context length, rounded up to whole tiles, plus a fixed
// item cost (the time a CTA spends starting and finishing a unit, in tokens of streaming)
// to one concatenated token space; that space is cut into C equal tile-aligned pieces, one
// per CTA, so every CTA gets the same time's work.  A piece that crosses unit boundaries
// becomes several work items, processed by its CTA in order; the item-cost stretch after a
// unit's tokens holds no work, and a piece (or its part) that falls there gets no item tokens.
//
// Only the first and the last item of a piece can be part of a unit cut into several
// pieces, so CTA c writes at most two partial results, in slots 2c (its first item) and
// 2c + 1 (its last): the slots of a unit follow from the first CTA it appears in, with no
// prefix sum over units.  All units of a sequence have the same length, so the planner works
// on per-sequence prefix sums in shared memory.  One CTA does everything; it checks the
// lengths and, on a bad one, emits an empty work list so the decode kernel touches nothing
// (the flags word records why).  Block ids are checked by the decode kernel as it reads them.
// It also lists the split units whose partials are too large for the decode kernel's own
// merge (more pieces than ns_dec); the reduce kernel merges those.
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kPlanThreads = 512;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kPlanSmemSeqs = 4096;  // sequences whose prefix sums fit in shared memory

struct PlanParams {
  const int32_t* ctx;
  const int32_t* qlens;
  int32_t* hdr;
  int32_t* item_off;
  int4* items;
  int2* unit_info;
  int32_t* unit_cnt;
  int32_t* red_units;    // units whose pieces the reduce kernel merges
  int32_t* seq_start_g;  // B + 1 ints in the workspace, used when B > kPlanSmemSeqs
  int32_t* seq_len_g;    // B ints
  int batch, max_q_len, num_kv_heads, rb, block_size, max_blocks, tt, ctas, units;
  int item_cost;   // tokens of the space a unit costs beyond its own (a tile multiple)
  int ns_dec;      // the decode merges units of at most this many pieces
  int tt_shift;    // log2(tt): tiles are a power of two
  FastDiv ups_div; // units per sequence
};

// Exclusive prefix sum of one value per thread over the block.
__device__ int block_exclusive_scan(int v, int* total, int* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kPlanWarps ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kPlanWarps) sh[lane] = w;
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? sh[warp - 1] : 0);
  *total = sh[kPlanWarps - 1];
  __syncthreads();
  return excl;
}

// Last sequence whose start is <= x (sequences with no tokens share their successor's
// start and are skipped by taking the last such index).
__device__ int find_seq(const int32_t* start, int batch, int x) {
  int lo = 0, hi = batch;  // start[batch] > x for every x inside the token space
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (start[mid] <= x)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo - 1;
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(const PlanParams p) {
  __shared__ int sh[32];
  __shared__ int s_flags;
  __shared__ int32_t s_start[kPlanSmemSeqs + 1];
  __shared__ int32_t s_len[kPlanSmemSeqs];
  __shared__ uint32_t s_chunk_div[3];  // FastDiv of the chunk: d, m, s
  grid_dependency_wait();     // lengths may come from the previous kernel in the stream
  grid_dependents_launch();   // the decode grid can stage its prologue meanwhile
  const int tid = threadIdx.x;
  const bool in_smem = p.batch <= kPlanSmemSeqs;
  int32_t* seq_start = in_smem ? s_start : p.seq_start_g;
  int32_t* seq_len = in_smem ? s_len : p.seq_len_g;
  if (tid == 0) s_flags = 0;
  __syncthreads();

  // 1. lengths
  for (int b = tid; b < p.batch; b += kPlanThreads) {
    const int n = __ldg(p.ctx + b), ql = __ldg(p.qlens + b);
    const long long cap = (long long)p.max_blocks * p.block_size;
    const bool bad = ql < 0 || ql > p.max_q_len || n < ql || (long long)n > cap;
    if (bad) atomicOr(&s_flags, PA_FLAG_BAD_LENGTHS);
    seq_len[b] = n;
  }
  __syncthreads();
  const int flags = s_flags;
  const int ups = p.num_kv_heads * p.rb;  // units per sequence
  auto pad = [&](int len) { return ((len + p.tt - 1) >> p.tt_shift) << p.tt_shift; };
  // a unit's stretch of the space: its tokens rounded up to tiles, then the item cost
  auto stride = [&](int len) { return len > 0 ? pad(len) + p.item_cost : 0; };

  // 2. start of each sequence's units in the concatenated, tile-padded token space
  int carry = 0, tot = 0;
  for (int base = 0; base < p.batch; base += kPlanThreads) {
    const int b = base + tid;
    int len = 0;
    if (b < p.batch && flags == 0) len = stride(seq_len[b]) * ups;
    const int excl = block_exclusive_scan(len, &tot, sh);
    if (b < p.batch) seq_start[b] = carry + excl;
    carry += tot;
  }
  const int T = carry;
  if (tid == 0) seq_start[p.batch] = T;
  __syncthreads();

  // 3. equal tile-aligned pieces, one per CTA
  const int chunk = T > 0 ? pad(ceil_div(T, p.ctas)) : p.tt;
  const int active = T > 0 ? ceil_div(T, chunk) : 0;
  if (tid == 0) {
    const FastDiv f((uint32_t)chunk);
    s_chunk_div[0] = f.d;
    s_chunk_div[1] = f.m;
    s_chunk_div[2] = f.s;
  }
  __syncthreads();
  FastDiv cdiv;
  cdiv.d = s_chunk_div[0];
  cdiv.m = s_chunk_div[1];
  cdiv.s = s_chunk_div[2];

  // 4. per unit: its pieces and the slot of its first partial, and the list of split units
  //    too large for the decode's own merge: units of at most kReduceWarpPieces pieces
  //    first (the reduce kernel merges their rows a warp each), then the others, each part
  //    in unit order
  int nred = 0, nsmall = 0;
  for (int pass = 0; pass < 2; ++pass) {
    for (int base = 0; base < p.units; base += kPlanThreads) {
      const int u = base + tid;
      int ns = 0, first = 0;
      if (u < p.units && flags == 0) {
        const int b = p.ups_div.div(u), k = u - b * ups;
        const int plen = pad(seq_len[b]);
        const int st = seq_start[b] + k * stride(seq_len[b]);
        if (plen > 0) {
          const int c0 = cdiv.div(st);
          ns = cdiv.div(st + plen - 1) - c0 + 1;
          first = 2 * c0 + (c0 * chunk < st ? 1 : 0);  // the last item of CTA c0, or its first
        }
      }
      const bool small = ns <= kReduceWarpPieces;
      const int to_reduce = (ns > p.ns_dec && small == (pass == 0)) ? 1 : 0;
      const int excl = block_exclusive_scan(to_reduce, &tot, sh);
      if (u < p.units) {
        if (pass == 0) {
          p.unit_info[u] = make_int2(first, ns);
          p.unit_cnt[u] = 0;
        }
        if (to_reduce) p.red_units[nred + excl] = u;
      }
      nred += tot;
    }
    if (pass == 0) nsmall = nred;
  }

  // 5. work items, CTA by CTA
  carry = 0;
  for (int base = 0; base < p.ctas; base += kPlanThreads) {
    const int c = base + tid;
    int cnt = 0, uf = 0, lo = 0, hi = 0;
    if (c < active) {
      lo = c * chunk;
      hi = min(lo + chunk, T) - 1;
      const int bf = find_seq(seq_start, p.batch, lo), bl = find_seq(seq_start, p.batch, hi);
      const int pf = stride(seq_len[bf]), pl = stride(seq_len[bl]);
      uf = bf * ups + (lo - seq_start[bf]) / pf;
      const int ul = bl * ups + (hi - seq_start[bl]) / pl;
      cnt = ul - uf + 1;
    }
    const int excl = block_exclusive_scan(cnt, &tot, sh);
    if (c < p.ctas) p.item_off[c] = carry + excl;
    for (int k = 0; k < cnt; ++k) {
      const int u = uf + k;
      const int b = p.ups_div.div(u), ku = u - b * ups;
      const int len = seq_len[b];
      const int plen = pad(len);
      const int st = seq_start[b] + ku * stride(len);
      int t0 = 0, t1 = 0, slot = -1;
      if (plen > 0) {
        t0 = max(lo, st) - st;
        t1 = min(hi + 1 - st, len);
        if (t1 <= t0) {
          t0 = t1 = 0;  // only the item-cost stretch of the unit lies in this piece
        } else if (cdiv.div(st + plen - 1) != cdiv.div(st)) {
          slot = 2 * c + (k > 0 ? 1 : 0);
        }
      }
      p.items[carry + excl + k] = make_int4(u, t0, t1, slot);
    }
    carry += tot;
  }
  if (tid == 0) {
    p.item_off[p.ctas] = carry;
    p.hdr[HDR_FLAGS] = flags;
    p.hdr[HDR_CHUNK] = chunk;
    p.hdr[HDR_ACTIVE] = active;
    p.hdr[HDR_ITEMS] = carry;
    p.hdr[HDR_NRED] = nred;
    p.hdr[HDR_NRED_SMALL] = nsmall;
  }
}

}  // namespace

cudaError_t launch_plan(const ProblemArgs& a, const Variant& v, const WsLayout& L, char* ws,
                        cudaStream_t s) {
  PlanParams p;
  p.ctx = a.context_lens;
  p.qlens = a.q_lens;
  p.hdr = reinterpret_cast<int32_t*>(ws + L.header);
  p.item_off = reinterpret_cast<int32_t*>(ws + L.item_off);
  p.items = reinterpret_cast<int4*>(ws + L.items);
  p.unit_info = reinterpret_cast<int2*>(ws + L.unit_info);
  p.unit_cnt = reinterpret_cast<int32_t*>(ws + L.unit_cnt);
  p.red_units = reinterpret_cast<int32_t*>(ws + L.red_units);
  p.seq_start_g = reinterpret_cast<int32_t*>(ws + L.seq_start);
  p.seq_len_g = reinterpret_cast<int32_t*>(ws + L.seq_len);
  p.batch = a.batch;
  p.max_q_len = a.max_q_len;
  p.num_kv_heads = a.num_kv_heads;
  p.rb = v.rb;
  p.block_size = a.block_size;
  p.max_blocks = a.max_blocks;
  p.tt = v.tt;
  p.item_cost = v.item_cost;
  p.ctas = v.ctas;
  p.units = v.units;
  p.ns_dec = v.ns_dec;
  p.tt_shift = ilog2((uint32_t)v.tt);
  p.ups_div = FastDiv((uint32_t)(a.num_kv_heads * v.rb));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, p);
}

}  // namespace pa
