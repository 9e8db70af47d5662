// Pieces shared by the CUDA-core and tensor-core decode kernels: kernel parameters, element
// conversions, the TMA side of the shared-memory page ring, and the split merge that the last
// CTA to finish a unit runs inside the decode kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pa_internal.cuh"

namespace pa {

__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

struct KernelParams {
  const void* q;
  const float* k_scale;
  const float* v_scale;
  const int32_t* bt;
  const int32_t* ctx;
  const int32_t* qlens;
  void* out;
  float* lse;
  const int32_t* item_off;
  const int4* first_item;  // [C]: item item_off[c] of CTA c, or (0, 0, 0, -1)
  const int4* items;
  float* o_part;
  float* lse_part;
  int32_t* flags;
  const int2* unit_info;
  int32_t* unit_cnt;
  int units;
  int ns_dec;  // split units of at most this many pieces are merged here (see merge_if_last)
  int scale_mode;
  int Sq, Hq, Hkv, G, M, RB, bs, maxb, nblocks, causal;
  int bs_shift;  // log2(bs): pages are a power of two
  float qk_scale;
  // the planner's inputs, for a CTA that derives its own first work item (first_item_of)
  int batch, tt, tt_shift, item_cost;
};

// The first work item of CTA c of C, derived from the lengths with the planner's own rules
// and integer arithmetic (the concatenated token space of plan.cu: each unit its tile-padded
// length plus the item cost, cut into C equal tile-aligned pieces), so that a CTA can start
// on it before the planner has finished.  One whole warp: one pass sums the space (any bad
// length gives no items, as in the planner), a second finds the sequence holding the
// piece's first position with a running warp scan.  Returns (0, 0, 0, -1) when the CTA has
// no items.
static __device__ __forceinline__ int4 first_item_of(const KernelParams& p, int c, int C, int lane) {
  const int4 none = make_int4(0, 0, 0, -1);
  const int ups = p.Hkv * p.RB;
  const long long cap = (long long)p.maxb * p.bs;
  auto pad = [&](int len) { return ((len + p.tt - 1) >> p.tt_shift) << p.tt_shift; };
  auto stride = [&](int len) { return len > 0 ? pad(len) + p.item_cost : 0; };
  int total = 0;
  bool bad = false;
  for (int b0 = 0; b0 < p.batch; b0 += 32) {
    const int b = b0 + lane;
    if (b < p.batch) {
      const int n = __ldg(p.ctx + b), ql = __ldg(p.qlens + b);
      if (ql < 0 || ql > p.Sq || n < ql || (long long)n > cap)
        bad = true;
      else
        total += stride(n) * ups;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(kFull, total, o);
  if (__any_sync(kFull, bad) || total <= 0) return none;
  const int T = total;
  const int chunk = pad((int)(((uint32_t)T + (uint32_t)C - 1u) / (uint32_t)C));
  if (c >= (T - 1) / chunk + 1) return none;  // past the active CTAs
  const int lo = c * chunk, hi = min(lo + chunk, T) - 1;
  // the last sequence whose start is <= lo (a sequence with no tokens shares its
  // successor's start, so the last one is never empty)
  int run = 0, start_f = 0, n_f = 0, b_f = 0;
  for (int b0 = 0; b0 < p.batch && run <= lo; b0 += 32) {
    const int b = b0 + lane;
    const int n = b < p.batch ? __ldg(p.ctx + b) : 0;
    const int span = stride(n) * ups;
    int x = span;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    const int start = run + x - span;
    const unsigned m = __ballot_sync(kFull, b < p.batch && start <= lo);
    if (m) {
      const int l = 31 - __clz(m);
      b_f = b0 + l;
      start_f = __shfl_sync(kFull, start, l);
      n_f = __shfl_sync(kFull, n, l);
    }
    run += __shfl_sync(kFull, x, 31);
  }
  const int pf = stride(n_f);
  const int ku = (lo - start_f) / pf;
  const int st = start_f + ku * pf;
  int t0 = max(lo, st) - st, t1 = min(hi + 1 - st, n_f), slot = -1;
  if (t1 <= t0)
    t0 = t1 = 0;  // only the item-cost stretch of the unit lies in this piece
  else if (st < lo || st + pad(n_f) - 1 > hi)
    slot = 2 * c;  // the unit's tiles reach out of this piece
  return make_int4(b_f * ups + ku, t0, t1, slot);
}

// ---- element conversion -----------------------------------------------------------
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ float2 f16x2_to_f2(uint32_t w) {
  return __half22float2(*reinterpret_cast<__half2*>(&w));
}
__device__ __forceinline__ void e4m3x4_to_f2(uint32_t w, float2* f) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
  f[0] = __half22float2(*reinterpret_cast<__half2*>(&lo));
  f[1] = __half22float2(*reinterpret_cast<__half2*>(&hi));
}

// Raw chunk of cache elements in registers: CB bytes = CB / 4 words.
template <int CB>
struct RawChunk {
  uint32_t w[CB / 4];
};

template <int CB>
__device__ __forceinline__ RawChunk<CB> lds_chunk(const char* src) {
  RawChunk<CB> r;
  if constexpr (CB == 16) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
  } else if constexpr (CB == 8) {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    r.w[0] = v.x; r.w[1] = v.y;
  } else {
    r.w[0] = *reinterpret_cast<const uint32_t*>(src);
  }
  return r;
}

// Convert a raw chunk of EPC elements to EPC / 2 float2 pairs (element order kept).
template <int KVK, int CB>
__device__ __forceinline__ void chunk_to_f2(const RawChunk<CB>& r, float2* f) {
#pragma unroll
  for (int j = 0; j < CB / 4; ++j) {
    if constexpr (KVK == KV_FP8) {
      e4m3x4_to_f2(r.w[j], f + 2 * j);
    } else if constexpr (KVK == KV_BF16) {
      f[j] = bf16x2_to_f2(r.w[j]);
    } else {
      f[j] = f16x2_to_f2(r.w[j]);
    }
  }
}

template <int QK>
__device__ __forceinline__ float2 q_pair(uint32_t w) {
  if constexpr (QK == Q_BF16)
    return bf16x2_to_f2(w);
  else
    return f16x2_to_f2(w);
}

template <int QK>
__device__ __forceinline__ void store_out(void* out, size_t idx, float v) {
  if constexpr (QK == Q_BF16)
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
}

// Four consecutive outputs (idx a multiple of 4: one 8-byte store).
template <int QK>
__device__ __forceinline__ void store_out4(void* out, size_t idx, float4 v) {
  uint2 w;
  if constexpr (QK == Q_BF16) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    w.x = *reinterpret_cast<uint32_t*>(&a);
    w.y = *reinterpret_cast<uint32_t*>(&b);
  } else {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    w.x = *reinterpret_cast<uint32_t*>(&a);
    w.y = *reinterpret_cast<uint32_t*>(&b);
  }
  *reinterpret_cast<uint2*>(static_cast<char*>(out) + idx * 2) = w;
}

// The TMA side of the ring, run by warp 0 (all lanes, same state) between its own tiles.
// R describes the ring: TT tokens per stage of STAGE bytes (K tile of KTILE bytes, then V,
// then per-token scales when TOKS), NSTAGE stages, and how a tile row is laid out: either
// one box across the whole head dimension (NSLAB = 1) or NSLAB column slabs of ROWB = 128
// bytes per row, each written with the 128-byte swizzle.  With WITH_Q the query rows of an
// item are copied into NQ shared-memory slots together with the item's first tile.
template <class R>
struct TileProducer {
  using T = R;
  static constexpr int D = R::D;
  static constexpr int MP = R::MP;
  static constexpr bool TOKS = R::TOKS;
  const KernelParams* p;
  const CUtensorMap* kmap;
  const CUtensorMap* vmap;
  char* smem;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* qfull;
  volatile int* abort_flag;
  int lane, it, it_end;
  int k, ntiles, t0, t1, b, g, rb;
  uint32_t issued, items_started;
  int box_rows, nbox;  // rows per box (one page or one tile), boxes (pages) per tile
  uint32_t box_bytes;  // bytes of one box
  int blk_next;
  bool have;        // current item has tiles left
  bool next_ready;  // blk_next already holds the next item's first-tile block ids
  int4 item_next;

  // lane -> (page of the tile, column slab): lane = page * NSLAB + slab
  __device__ __forceinline__ int box_block_of(int bb, int tt0, int tt1, int kk) const {
    const int tokb = tt0 + kk * T::TT + (lane / T::NSLAB) * box_rows;
    return (lane < nbox * T::NSLAB && tokb < tt1)
               ? __ldg(p->bt + (size_t)bb * p->maxb + (tokb >> p->bs_shift))
               : -1;
  }
  __device__ __forceinline__ int box_block(int kk) const { return box_block_of(b, t0, t1, kk); }

  __device__ __forceinline__ void init(const KernelParams* prm, const CUtensorMap* km,
                                       const CUtensorMap* vm, char* sm, uint64_t* f,
                                       uint64_t* e, uint64_t* qf, volatile int* ab, int ln,
                                       int ib, int ie, int4 first) {
    p = prm; kmap = km; vmap = vm; smem = sm; full = f; empty = e; qfull = qf; abort_flag = ab;
    lane = ln; it = ib - 1; it_end = ie; k = 0; ntiles = 0; issued = 0; items_started = 0;
    box_rows = min(p->bs, T::TT);
    nbox = T::TT / box_rows;
    box_bytes = (uint32_t)box_rows * T::ROWB;
    have = false;
    next_ready = false;
    item_next = first;  // item ib, or (0, 0, 0, -1)
  }

  // Move to the next item with tokens; false when the CTA's list is exhausted.
  __device__ __forceinline__ bool advance() {
    while (!have) {
      if (++it >= it_end) return false;
      const int4 item = item_next;
      if (it + 1 < it_end) item_next = p->items[it + 1];
      t0 = item.y;
      t1 = item.z;
      if (t1 <= t0) continue;
      const int u = item.x;
      b = u / (p->Hkv * p->RB);
      g = (u / p->RB) % p->Hkv;
      rb = u % p->RB;
      k = 0;
      ntiles = ceil_div(t1 - t0, T::TT);
      if (!next_ready) blk_next = box_block(0);
      next_ready = false;
      have = true;
    }
    return true;
  }

  // Issue the next tile of the CTA's sequence into its stage (waiting for the stage to be
  // released by every warp); the query rows of an item go out with its first tile.
  __device__ __forceinline__ bool issue_one() {
    if (!advance()) return false;
    const int s = issued % T::NSTAGE;
    const uint32_t ph = (issued / T::NSTAGE) & 1;
    const int tok0 = t0 + k * T::TT;
    const int page = lane / T::NSLAB, slab = lane % T::NSLAB;
    const int tokb = tok0 + page * box_rows;
    const int blk = blk_next;
    const bool want = lane < nbox * T::NSLAB && tokb < t1;
    const bool ok = want && blk >= 0 && blk < p->nblocks;
    if (want && !ok) atomicOr(p->flags, PA_FLAG_BAD_BLOCK_ID);
    const uint32_t nvalid = __popc(__ballot_sync(kFull, ok));
    // overlap the next lookup: the next tile of this item, or the first of the next item
    if (k + 1 < ntiles) {
      blk_next = box_block(k + 1);
    } else if (it + 1 < it_end && item_next.z > item_next.y) {
      blk_next = box_block_of(item_next.x / (p->Hkv * p->RB), item_next.y, item_next.z, 0);
      next_ready = true;
    }
    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
      atomicOr(p->flags, PA_FLAG_WAIT_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
    if (T::WITH_Q && k == 0) {
      // query rows of this item: MP rows x D, 16-byte cp.async, completing on qfull
      const int qs = items_started % T::NQ;
      ++items_started;
      char* qslot = smem + T::OFF_Q + qs * T::QSLOT;
      constexpr int QCH = D * 2 / 16;
      for (int c = lane; c < MP * QCH; c += 32) {
        const int r = c / QCH, cc = c % QCH, rg = rb * MP + r;
        if (rg < p->M) {
          const int i = rg / p->G, gq = rg % p->G;
          const char* src = reinterpret_cast<const char*>(p->q) +
                            ((((size_t)b * p->Sq + i) * p->Hq + (size_t)g * p->G + gq) * D) * 2 +
                            cc * 16;
          cp_async_16(qslot + r * D * 2 + cc * 16, src);
        }
      }
      cp_async_arrive_noinc(&qfull[qs]);
    }
    char* st = smem + s * T::STAGE;
    // per-token scales of one kv head on a page that holds the whole tile: two contiguous
    // runs of TT floats, copied by two bulk copies that complete on the stage's barrier
    bool scale_bulk = false, ok0 = false;
    if constexpr (TOKS) {
      scale_bulk = p->Hkv == 1 && box_rows == T::TT &&
                   ((reinterpret_cast<uintptr_t>(p->k_scale) |
                     reinterpret_cast<uintptr_t>(p->v_scale)) & 15) == 0;
      ok0 = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;  // lane 0's box is the tile's one page
    }
    if (lane == 0)
      mbar_arrive_expect_tx(&full[s], nvalid * 2u * box_bytes +
                                          (scale_bulk && ok0 ? 2u * T::TT * 4u : 0u));
    __syncwarp();
    if (ok) {
      // slab h of page j lands at h * (TT rows) + j * (box rows), in units of ROWB bytes
      const int row = tokb & (p->bs - 1);
      const uint32_t dst = (uint32_t)(slab * T::TT + page * box_rows) * T::ROWB;
      const int x = slab * (T::ROWB / T::BPE);
      tma_load_4d(st + dst, kmap, &full[s], x, g, row, blk);
      tma_load_4d(st + T::KTILE + dst, vmap, &full[s], x, g, row, blk);
    }
    if constexpr (TOKS) {
      float* sks = reinterpret_cast<float*>(st + 2 * T::KTILE);
      float* svs = sks + T::TT;
      if (scale_bulk) {
        if (lane == 0 && ok0) {
          const size_t idx = (size_t)blk * p->bs + (tokb & (p->bs - 1));
          bulk_load_1d(sks, p->k_scale + idx, T::TT * 4, &full[s]);
          bulk_load_1d(svs, p->v_scale + idx, T::TT * 4, &full[s]);
        }
        mbar_arrive(&full[s]);  // the 32 arrivals the stage expects besides the copy's
        ++issued;
        if (++k >= ntiles) have = false;
        return true;
      }
      for (int t = lane; t < T::TT; t += 32) {
        const int bb = __shfl_sync(kFull, blk, (t / box_rows) * T::NSLAB);
        const int tok = tok0 + t;
        if (tok < t1 && bb >= 0 && bb < p->nblocks) {
          const size_t idx = ((size_t)bb * p->bs + (tok & (p->bs - 1))) * p->Hkv + g;
          cp_async_4(sks + t, p->k_scale + idx);
          cp_async_4(svs + t, p->v_scale + idx);
        }
      }
      cp_async_arrive_noinc(&full[s]);
    }
    ++issued;
    if (++k >= ntiles) have = false;
    return true;
  }

  // Keep the ring filled up to tile `upto` (global tile index of this CTA).
  __device__ __forceinline__ void fill(uint32_t upto) {
    while (issued <= upto && !*abort_flag) {
      if (!issue_one()) break;
    }
  }

  // Let every copy this warp started land before the CTA may exit.
  __device__ __forceinline__ void drain() {
    cp_async_wait_all();
    const uint32_t first = issued > (uint32_t)T::NSTAGE ? issued - T::NSTAGE : 0;
    for (uint32_t j = first; j < issued; ++j)
      mbar_wait_drain(&full[j % T::NSTAGE], (j / T::NSTAGE) & 1);
  }
};

// ---- split units ----------------------------------------------------------------------
// A unit cut into ns pieces is merged inside the decode kernel when ns <= ns_dec (larger
// ones are left to the reduce kernel).  unit_cnt[u] counts the pieces whose partial
// (o_part, lse_part) is published.  When piece 0 ends and finds every other piece published
// (count == ns - 1, read with acquire), it is the last: it combines the others' partials with
// its own state in registers and writes the output, without publishing.  Any other piece
// writes its partial and publishes it with an acquire-release add; the add that returns
// ns - 1 belongs to a piece that turned out last after all, and that CTA merges the unit from
// the partials after its own work list (the add's result is only waited for there).
// Exactly one piece merges each unit, no CTA ever waits for another, and the merging CTA
// sets the count back to zero, so the next decode on the same plan starts clean.
//
// Both ways of merging do the same arithmetic, so the result does not depend on which piece
// ends last: per row m = max_s l_s, w_s = 2^(l_s - m) (0 for l_s = -inf), W = sum of w_s
// added in piece order, O = fma(w_s, o_s, O) in piece order from O = 0, out = O * (1 / W),
// where o_s is a piece's normalised partial exactly as it is stored.
constexpr int kFlagBytes = 32;  // abort flag, pending merges, count seen (after the barriers)

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* ptr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v)
               : "memory");
  return old;
}
// Piece index of `slot` within a unit whose first piece sits in slot `first`.
__device__ __forceinline__ int piece_index(int first, int slot) {
  return slot == first ? 0 : (slot >> 1) - (first >> 1);
}

// Merge every published piece of unit u with the log-sum-exp rule and write its output
// rows, then reset its count.  All NW warps of the CTA take part.
// `tid` numbers the NW warps that take part from 0 (they use named barrier 1).
template <int D, int MP, int QK, int NW>
__device__ __forceinline__ void merge_unit(const KernelParams& p, int u, float* wtab, int wcap,
                                           float* stat, int tid) {
  constexpr int NT = NW * 32;
  constexpr int D4 = D / 4;
  const int2 info = __ldg(&p.unit_info[u]);
  const int first = info.x, ns = info.y;
  const int b = u / (p.Hkv * p.RB), g = (u / p.RB) % p.Hkv, rb = u % p.RB;
  __threadfence();
  const bool tab = MP * ns <= wcap;  // weights fit in shared memory
  const int warp = tid >> 5, lane = tid & 31;
  // per row: max over the pieces (lanes over pieces), then weights and their sum in order
  for (int r = warp; r < MP; r += NW) {
    float m = -INFINITY;
    for (int s = lane; s < ns; s += 32)
      m = fmaxf(m, __ldcg(p.lse_part + (size_t)piece_slot(first, s) * MP + r));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    if (tab)
      for (int s = lane; s < ns; s += 32) {
        const float ls = __ldcg(p.lse_part + (size_t)piece_slot(first, s) * MP + r);
        wtab[r * ns + s] = (ls == -INFINITY) ? 0.f : fast_exp2(ls - m);
      }
    __syncwarp();
    if (lane == 0) {
      float W = 0.f;
      for (int s = 0; s < ns; ++s) {
        float w;
        if (tab) {
          w = wtab[r * ns + s];
        } else {
          const float ls = __ldcg(p.lse_part + (size_t)piece_slot(first, s) * MP + r);
          w = (ls == -INFINITY) ? 0.f : fast_exp2(ls - m);
        }
        W = W + w;
      }
      stat[2 * r] = m;
      stat[2 * r + 1] = W;
    }
  }
  named_barrier_sync(1, NT);
  // weighted sum: each thread owns four consecutive head dims of a row
  for (int e = tid; e < MP * D4; e += NT) {
    const int r = e / D4, d = (e % D4) * 4, rg = rb * MP + r;
    if (rg >= p.M) continue;
    const float m = stat[2 * r], W = stat[2 * r + 1];
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    if (W > 0.f) {
#pragma unroll 4
      for (int s = 0; s < ns; ++s) {
        const size_t part = (size_t)piece_slot(first, s) * MP + r;
        float w;
        if (tab) {
          w = wtab[r * ns + s];
        } else {
          const float ls = __ldcg(p.lse_part + part);
          w = (ls == -INFINITY) ? 0.f : fast_exp2(ls - m);
        }
        if (w == 0.f) continue;  // no key of this row in the piece
        const float4 o = __ldcg(reinterpret_cast<const float4*>(p.o_part + part * D + d));
        O.x = __fmaf_rn(w, o.x, O.x);
        O.y = __fmaf_rn(w, o.y, O.y);
        O.z = __fmaf_rn(w, o.z, O.z);
        O.w = __fmaf_rn(w, o.w, O.w);
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    const size_t row = ((size_t)b * p.Sq + rg / p.G) * p.Hq + g * p.G + rg % p.G;
    const float4 v = W > 0.f ? make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    store_out4<QK>(p.out, row * D + d, v);
    if (d == 0 && p.lse) p.lse[row] = W > 0.f ? (m + fast_log2(W)) * kLn2 : -INFINITY;
  }
  if (tid == 0) p.unit_cnt[u] = 0;
  named_barrier_sync(1, NT);  // the shared buffers are reused next
}

// Publish the partial of the piece in `slot` (every thread's partial writes precede this
// call behind a CTA barrier).  Called by one thread; the add's result is kept, by the slot's
// parity, in *pend_even / *pend_odd as (unit, pieces published before this one), to be looked
// at after the CTA's work list (finish_pending).
__device__ __forceinline__ void publish_piece(const KernelParams& p, int u, int slot,
                                              int2* pend_even, int2* pend_odd) {
  const int before = atom_add_acq_rel_gpu(&p.unit_cnt[u], 1);
  if (slot & 1)
    *pend_odd = make_int2(u, before);
  else
    *pend_even = make_int2(u, before);
}

// After the work list: merge the units whose publishing add this CTA made last.
// `pend` is shared memory holding the two (unit, before) pairs, unit -1 for none.
template <int D, int MP, int QK, int NW>
__device__ __forceinline__ void finish_pending(const KernelParams& p, const volatile int* pend,
                                               float* wtab, int wcap, float* stat,
                                               int tid = threadIdx.x) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int u = pend[2 * j], before = pend[2 * j + 1];
    if (u >= 0 && before == __ldg(&p.unit_info[u].y) - 1)
      merge_unit<D, MP, QK, NW>(p, u, wtab, wcap, stat, tid);
  }
}

// Units with no keys at all: padding rows (zero, lse = -inf), spread over the CTAs.
template <int D, int MP, int QK, int NT>
__device__ __forceinline__ void zero_empty_units(const KernelParams& p, int tid = threadIdx.x) {
  for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
    if (__ldg(&p.unit_info[u].y) != 0) continue;
    const int b = u / (p.Hkv * p.RB), g = (u / p.RB) % p.Hkv, rb = u % p.RB;
    for (int e = tid; e < MP * D; e += NT) {
      const int r = e / D, d = e % D, rg = rb * MP + r;
      if (rg >= p.M) continue;
      const size_t row = ((size_t)b * p.Sq + rg / p.G) * p.Hq + g * p.G + rg % p.G;
      store_out<QK>(p.out, row * D + d, 0.f);
      if (d == 0 && p.lse) p.lse[row] = -INFINITY;
    }
  }
}

KernelParams make_kernel_params(const DecodeArgs& a);

}  // namespace pa
