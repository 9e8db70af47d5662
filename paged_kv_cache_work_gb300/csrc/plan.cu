// Planner: turns the device-resident context lengths into the persistent grid's work list.
//
// The split follows "Optimize paged-attention metadata decode" (FlyDSL PR #910, Summary and
// Changes): metadata is generated on the device for a persistent decode grid sized as SMs x
// a grid multiplier (default 1, the safe one-grid-per-CU choice), and ranges that a unit
// does not finish in one piece are merged by a separate reducer.  Here every unit
// (sequence, kv head, row tile) contributes its context length, rounded up to whole tiles,
// to one concatenated token space; that space is cut into C equal tile-aligned pieces, one
// per CTA, so every CTA streams the same number of KV bytes.  A piece that crosses unit
// boundaries becomes several work items, processed by its CTA in order.
//
// One CTA of 1024 threads does everything with block-wide scans; it also checks the
// lengths and every block id in use and, on any problem, emits an empty work list so the
// decode kernel touches nothing (the flags word records why).
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kPlanThreads = 1024;

struct PlanParams {
  const int32_t* bt;
  const int32_t* ctx;
  const int32_t* qlens;
  int32_t* hdr;
  int32_t* item_off;
  int4* items;
  int2* unit_info;
  int32_t* unit_start;
  int batch, max_q_len, num_kv_heads, rb, block_size, max_blocks, num_blocks, tt, ctas, units;
};

// Exclusive prefix sum of one value per thread over the 1024-thread block.
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
    int w = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? sh[warp - 1] : 0);
  *total = sh[31];
  __syncthreads();
  return excl;
}

// Last unit whose start is <= x (units of zero length share their successor's start and
// are skipped by taking the last such index).
__device__ int find_unit(const int32_t* start, int units, int x) {
  int lo = 0, hi = units;  // start[units] > x for every x inside the token space
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
  const int tid = threadIdx.x;
  if (tid == 0) s_flags = 0;
  __syncthreads();

  // 1. lengths
  for (int b = tid; b < p.batch; b += kPlanThreads) {
    const int n = p.ctx[b], ql = p.qlens[b];
    const long long cap = (long long)p.max_blocks * p.block_size;
    if (ql < 0 || ql > p.max_q_len || n < ql || (long long)n > cap)
      atomicOr(&s_flags, PA_FLAG_BAD_LENGTHS);
  }
  __syncthreads();
  // 2. block ids of every page in use (only once the lengths are known to be sane)
  if (s_flags == 0) {
    const long long total = (long long)p.batch * p.max_blocks;
    for (long long idx = tid; idx < total; idx += kPlanThreads) {
      const int b = (int)(idx / p.max_blocks), pg = (int)(idx % p.max_blocks);
      const int pages = (p.ctx[b] + p.block_size - 1) / p.block_size;
      if (pg < pages) {
        const int id = p.bt[idx];
        if (id < 0 || id >= p.num_blocks) atomicOr(&s_flags, PA_FLAG_BAD_BLOCK_ID);
      }
    }
  }
  __syncthreads();
  const int flags = s_flags;
  const int per_seq = p.num_kv_heads * p.rb;

  // 3. unit starts in the concatenated, tile-padded token space
  int carry = 0, tot = 0;
  for (int base = 0; base < p.units; base += kPlanThreads) {
    const int u = base + tid;
    int len = 0;
    if (u < p.units && flags == 0) len = round_up(p.ctx[u / per_seq], p.tt);
    const int excl = block_exclusive_scan(len, &tot, sh);
    if (u < p.units) p.unit_start[u] = carry + excl;
    carry += tot;
  }
  const int T = carry;
  if (tid == 0) p.unit_start[p.units] = T;
  __syncthreads();

  // 4. equal tile-aligned pieces, one per CTA
  const int chunk = T > 0 ? round_up(ceil_div(T, p.ctas), p.tt) : p.tt;
  const int active = T > 0 ? ceil_div(T, chunk) : 0;

  // 5. splits per unit and the first partial slot of units done in several pieces
  carry = 0;
  for (int base = 0; base < p.units; base += kPlanThreads) {
    const int u = base + tid;
    int ns = 0;
    if (u < p.units) {
      const int st = p.unit_start[u], en = p.unit_start[u + 1];
      if (en > st) ns = (en - 1) / chunk - st / chunk + 1;
    }
    const int parts = ns >= 2 ? ns : 0;
    const int excl = block_exclusive_scan(parts, &tot, sh);
    if (u < p.units) p.unit_info[u] = make_int2(carry + excl, ns);
    carry += tot;
  }
  __syncthreads();

  // 6. work items, CTA by CTA
  carry = 0;
  for (int base = 0; base < p.ctas; base += kPlanThreads) {
    const int c = base + tid;
    int cnt = 0, uf = 0, lo = 0, hi = 0;
    if (c < active) {
      lo = c * chunk;
      hi = min(lo + chunk, T) - 1;
      uf = find_unit(p.unit_start, p.units, lo);
      cnt = find_unit(p.unit_start, p.units, hi) - uf + 1;
    }
    const int excl = block_exclusive_scan(cnt, &tot, sh);
    if (c < p.ctas) p.item_off[c] = carry + excl;
    for (int k = 0; k < cnt; ++k) {
      const int u = uf + k;
      const int st = p.unit_start[u], en = p.unit_start[u + 1];
      int t0 = 0, t1 = 0;
      if (en > st) {
        const int len = p.ctx[u / per_seq];
        t0 = max(lo, st) - st;
        t1 = min(hi + 1 - st, len);
      }
      const int2 info = p.unit_info[u];
      const int slot = info.y >= 2 ? info.x + (c - st / chunk) : -1;
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
  }
}

}  // namespace

cudaError_t launch_plan(const ProblemArgs& a, const Variant& v, const WsLayout& L, char* ws,
                        cudaStream_t s) {
  PlanParams p;
  p.bt = a.block_tables;
  p.ctx = a.context_lens;
  p.qlens = a.q_lens;
  p.hdr = reinterpret_cast<int32_t*>(ws + L.header);
  p.item_off = reinterpret_cast<int32_t*>(ws + L.item_off);
  p.items = reinterpret_cast<int4*>(ws + L.items);
  p.unit_info = reinterpret_cast<int2*>(ws + L.unit_info);
  p.unit_start = reinterpret_cast<int32_t*>(ws + L.unit_start);
  p.batch = a.batch;
  p.max_q_len = a.max_q_len;
  p.num_kv_heads = a.num_kv_heads;
  p.rb = v.rb;
  p.block_size = a.block_size;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.tt = v.tt;
  p.ctas = v.ctas;
  p.units = v.units;
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
