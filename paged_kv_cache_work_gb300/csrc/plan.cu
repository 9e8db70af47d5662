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
#include <algorithm>
#include <climits>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kPlanMaxThreads = 512;
constexpr int kPlanSmemSeqs = 4096;  // sequences whose prefix sums fit in shared memory

struct PlanParams {
  const int32_t* ctx;
  const int32_t* qlens;
  int32_t* hdr;
  int32_t* item_off;
  int4* first_item;
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
  int spt, upt, cpt;  // sequences, units and CTAs each thread takes (runs of contiguous ones)
  FastDiv ups_div;    // units per sequence
  FastDiv ctas_div;   // CTAs
};

// Exclusive prefix sums of N counters over the block, with one barrier: each warp scans its
// lanes and publishes its totals in `buf` (one row per warp, used by this scan only); after
// the barrier every warp reads all warps' totals, a lane each, and scans them too.  Returns
// the OR of `pred` over the block, taken at the same barrier.
template <int N>
__device__ __forceinline__ int block_scan(const int (&v)[N], int (&excl)[N], int (&tot)[N],
                                          int (*buf)[N], int pred) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x[N];
#pragma unroll
  for (int i = 0; i < N; ++i) x[i] = v[i];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int y = __shfl_up_sync(kFull, x[i], o);
      if (lane >= o) x[i] += y;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int i = 0; i < N; ++i) buf[warp][i] = x[i];
  }
  const int any = __syncthreads_or(pred);
  int t[N];
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = lane < nw ? buf[lane][i] : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int y = __shfl_up_sync(kFull, t[i], o);
      if (lane >= o) t[i] += y;
    }
  }
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const int before = __shfl_sync(kFull, t[i], warp > 0 ? warp - 1 : 0);
    excl[i] = x[i] - v[i] + (warp > 0 ? before : 0);
    tot[i] = __shfl_sync(kFull, t[i], 31);
  }
  return any;
}

// floor(x / d) for 0 <= x < 2^31 and 0 < d < 2^31 whose quotient is below 2^21, with rd a
// float within one ulp of 1/d (recip below).  The float estimate x * rd is within a relative
// 5.0001 * 2^-24 of x / d (x and d rounded to nearest, rd within 2^-23, the product rounded
// to nearest): less than one from it.  Truncated, it is the quotient or one off either way,
// and the remainder says which.  (The products below stay under 2^32.)  A division that the
// compiler expands costs about as much as the planner's other arithmetic put together.
__device__ __forceinline__ int div_small(int x, int d, float rd) {
  uint32_t q = (uint32_t)__float2int_rz(__int2float_rn(x) * rd);
  const uint32_t qd = q * (uint32_t)d;
  if (qd > (uint32_t)x)
    --q;
  else if ((uint32_t)x - qd >= (uint32_t)d)
    ++q;
  return (int)q;
}

// 1/d within one ulp (the approximate reciprocal's documented bound).
__device__ __forceinline__ float recip(int d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__int2float_rn(d)));
  return r;
}

// Last sequences whose start is <= x and <= y (sequences with no tokens share their
// successor's start and are skipped by taking the last such index): two searches by binary
// lifting in one loop, so their shared-memory loads overlap.  start[0] = 0 <= x, y.
__device__ __forceinline__ void find_seq2(const int32_t* start, int batch, int x, int y,
                                          int& bx, int& by) {
  int px = 0, py = 0;
  for (int step = 1 << (31 - __clz(batch)); step > 0; step >>= 1) {
    const int cx = px + step, cy = py + step;
    const int sx = cx < batch ? start[cx] : INT_MAX;
    const int sy = cy < batch ? start[cy] : INT_MAX;
    if (sx <= x) px = cx;
    if (sy <= y) py = cy;
  }
  bx = px;
  by = py;
}

// The block is short: three barriers in all.  Every thread takes a contiguous run of
// sequences, of units and of CTAs (one of each when the block is large enough), so one
// scan per phase serves any batch size.
__global__ void __launch_bounds__(kPlanMaxThreads, 1) plan_kernel(const PlanParams p) {
  __shared__ int scan_len[32][1];
  __shared__ int scan_cnt[32][3];
  __shared__ int32_t s_start[kPlanSmemSeqs + 1];
  __shared__ int32_t s_len[kPlanSmemSeqs];
  grid_dependency_wait();     // lengths may come from the previous kernel in the stream
  grid_dependents_launch();   // the decode grid can stage its prologue meanwhile
  const int tid = threadIdx.x;
  const bool in_smem = p.batch <= kPlanSmemSeqs;
  int32_t* seq_start = in_smem ? s_start : p.seq_start_g;
  int32_t* seq_len = in_smem ? s_len : p.seq_len_g;
  const int ups = p.num_kv_heads * p.rb;  // units per sequence
  auto pad = [&](int len) { return ((len + p.tt - 1) >> p.tt_shift) << p.tt_shift; };
  // a unit's stretch of the space: its tokens rounded up to tiles, then the item cost
  auto stride = [&](int len) { return len > 0 ? pad(len) + p.item_cost : 0; };

  // 1. lengths, checked, and each thread's share of the space
  const int b0 = min(tid * p.spt, p.batch), b1 = min(b0 + p.spt, p.batch);
  const long long cap = (long long)p.max_blocks * p.block_size;
  int bad = 0, span = 0;
  for (int b = b0; b < b1; ++b) {
    const int n = __ldg(p.ctx + b), ql = __ldg(p.qlens + b);
    const bool bad_b = ql < 0 || ql > p.max_q_len || n < ql || (long long)n > cap;
    bad |= bad_b ? 1 : 0;
    seq_len[b] = n;
    if (!bad_b) span += stride(n) * ups;
  }
  int excl1[1], tot1[1];
  const int spans[1] = {span};
  const int flags = block_scan<1>(spans, excl1, tot1, scan_len, bad) ? PA_FLAG_BAD_LENGTHS : 0;

  // 2. start of each sequence's units in the concatenated, tile-padded token space (an
  //    empty space when any length is bad, so the decode touches nothing)
  const int T = flags == 0 ? tot1[0] : 0;
  int run = flags == 0 ? excl1[0] : 0;
  for (int b = b0; b < b1; ++b) {
    seq_start[b] = run;
    if (flags == 0) run += stride(seq_len[b]) * ups;
  }
  if (tid == 0) seq_start[p.batch] = T;

  // 3. equal tile-aligned pieces, one per CTA (the same in every thread)
  const int chunk = T > 0 ? pad((int)p.ctas_div.div((uint32_t)T + p.ctas - 1)) : p.tt;
  const float rchunk = recip(chunk);
  const int active = T > 0 ? div_small(T - 1, chunk, rchunk) + 1 : 0;
  __syncthreads();

  // per unit: its pieces and the slot of its first partial
  auto unit_pieces = [&](int u, int& first) {
    first = 0;
    if (flags != 0) return 0;
    const int b = p.ups_div.div(u), k = u - b * ups;
    const int len = seq_len[b];
    const int plen = pad(len);
    if (plen == 0) return 0;
    const int st = seq_start[b] + k * stride(len);
    const int c0 = div_small(st, chunk, rchunk);
    first = 2 * c0 + (c0 * chunk < st ? 1 : 0);  // the last item of CTA c0, or its first
    return div_small(st + plen - 1, chunk, rchunk) - c0 + 1;
  };
  // per CTA: its first unit and how many units its piece overlaps
  auto cta_units = [&](int c, int& uf, int& lo, int& hi) {
    uf = lo = hi = 0;
    if (c >= active) return 0;
    lo = c * chunk;
    hi = min(lo + chunk, T) - 1;
    int bf, bl;
    find_seq2(seq_start, p.batch, lo, hi, bf, bl);
    const int pf = stride(seq_len[bf]), pl = stride(seq_len[bl]);
    uf = bf * ups + div_small(lo - seq_start[bf], pf, recip(pf));
    const int ul = bl * ups + div_small(hi - seq_start[bl], pl, recip(pl));
    return ul - uf + 1;
  };

  // 4. counts: split units the reduce kernel merges (at most kReduceWarpPieces pieces, and
  //    more), and work items, each thread over its own units and CTAs (the first of each
  //    kept for the writes below); one scan places them
  const int u0 = min(tid * p.upt, p.units), u1 = min(u0 + p.upt, p.units);
  const int cb = min(tid * p.cpt, p.ctas), ce = min(cb + p.cpt, p.ctas);
  int n_small = 0, n_large = 0, n_items = 0;
  int ns0 = 0, first0 = 0, n0 = 0, uf0 = 0, lo0 = 0, hi0 = 0;
  for (int u = u0; u < u1; ++u) {
    int first;
    const int ns = unit_pieces(u, first);
    if (u == u0) {
      ns0 = ns;
      first0 = first;
    }
    if (ns > p.ns_dec) {
      if (ns <= kReduceWarpPieces)
        ++n_small;
      else
        ++n_large;
    }
  }
  for (int c = cb; c < ce; ++c) {
    int uf, lo, hi;
    const int n = cta_units(c, uf, lo, hi);
    if (c == cb) {
      n0 = n;
      uf0 = uf;
      lo0 = lo;
      hi0 = hi;
    }
    n_items += n;
  }
  const int cnt[3] = {n_small, n_large, n_items};
  int ex[3], tot[3];
  block_scan<3>(cnt, ex, tot, scan_cnt, 0);
  const int nsmall = tot[0], nred = tot[0] + tot[1], nitems = tot[2];

  // 5. the unit table and the reduce list (the few-piece units first, then the others, each
  //    part in unit order)
  int at_small = ex[0], at_large = nsmall + ex[1];
  for (int u = u0; u < u1; ++u) {
    int first = first0, ns = ns0;
    if (u != u0) ns = unit_pieces(u, first);
    p.unit_info[u] = make_int2(first, ns);
    p.unit_cnt[u] = 0;
    if (ns > p.ns_dec) {
      if (ns <= kReduceWarpPieces)
        p.red_units[at_small++] = u;
      else
        p.red_units[at_large++] = u;
    }
  }

  // 6. work items, CTA by CTA
  int at = ex[2];
  for (int c = cb; c < ce; ++c) {
    int uf = uf0, lo = lo0, hi = hi0, n = n0;
    if (c != cb) n = cta_units(c, uf, lo, hi);
    p.item_off[c] = at;
    if (n == 0) p.first_item[c] = make_int4(0, 0, 0, -1);
    for (int k = 0; k < n; ++k) {
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
        } else if (st < lo || st + plen - 1 > hi) {
          // the unit's tiles reach out of this piece: it is cut into several
          slot = 2 * c + (k > 0 ? 1 : 0);
        }
      }
      const int4 item = make_int4(u, t0, t1, slot);
      if (k == 0) p.first_item[c] = item;
      p.items[at++] = item;
    }
  }
  if (tid == 0) {
    p.item_off[p.ctas] = nitems;
    p.hdr[HDR_FLAGS] = flags;
    p.hdr[HDR_CHUNK] = chunk;
    p.hdr[HDR_ACTIVE] = active;
    p.hdr[HDR_ITEMS] = nitems;
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
  p.first_item = reinterpret_cast<int4*>(ws + L.first_item);
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
  p.ctas_div = FastDiv((uint32_t)v.ctas);
  cudaLaunchConfig_t cfg = {};
  // a thread per sequence, unit or CTA (whichever is most) up to the block limit; past it
  // each thread takes a contiguous run of each
  const int work = std::max(a.batch, std::max(v.units, v.ctas));
  const int threads = std::min(kPlanMaxThreads, std::max(64, round_up(work, 32)));
  p.spt = ceil_div(a.batch, threads);
  p.upt = ceil_div(v.units, threads);
  p.cpt = ceil_div(v.ctas, threads);
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, p);
}

}  // namespace pa
