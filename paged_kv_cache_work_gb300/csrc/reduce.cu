// Split reducer and the decode dispatch.
//
// The reducer merges, for every unit the planner cut into several pieces, the normalised
// partials o_s and their log2-sum-exp l_s:  m* = max_s l_s,  w_s = 2^(l_s - m*),
// out = sum_s w_s o_s / sum_s w_s,  lse = (m* + log2 sum_s w_s) ln 2.  This is the "split
// reducer" that follows the persistent decode in "Optimize paged-attention metadata
// decode" (FlyDSL PR #910, Summary and Performance: metadata decode plus split reducer).
// Units the decode finished in one piece are skipped; units with no keys at all (a
// sequence with no context) get zero rows and lse = -inf.  Sums over splits run in a fixed
// order (lane-strided, then a fixed shuffle tree), so repeated calls are bitwise identical.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_common.cuh"

namespace pa {

cudaError_t launch_simt_d64(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                            int, int, bool, cudaStream_t);
int simt_ctas_per_sm_d64(int, int, bool);

cudaError_t launch_tc_d128(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                           int, int, bool, cudaStream_t);
cudaError_t launch_tc_d256(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                           int, int, bool, cudaStream_t);
cudaError_t launch_tc_fp8_d128(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int,
                               int, int, bool, cudaStream_t);

int mma_ctas_per_sm_d64(int, int, bool);
int mma_ctas_per_sm_d128(int, int, bool);
int mma_ctas_per_sm_d256(int, int, bool);
cudaError_t launch_mma_d64(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                           int, int, bool, cudaStream_t);
cudaError_t launch_mma_d128(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                            int, int, bool, cudaStream_t);
cudaError_t launch_mma_d256(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                            int, int, bool, cudaStream_t);

// The CUDA-core kernel serves 64-dim fp8 caches only (rows shorter than a 128-byte slab).
int simt_ctas_per_sm(int head_dim, int mp, int kvk, bool toks) {
  return head_dim == 64 ? simt_ctas_per_sm_d64(mp, kvk, toks) : 1;
}

int mma_ctas_per_sm(int head_dim, int mp, int kvk, bool toks) {
  switch (head_dim) {
    case 64: return mma_ctas_per_sm_d64(mp, kvk, toks);
    case 128: return mma_ctas_per_sm_d128(mp, kvk, toks);
    default: return mma_ctas_per_sm_d256(mp, kvk, toks);
  }
}

KernelParams make_kernel_params(const DecodeArgs& a) {
  KernelParams p{};
  p.q = a.q;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.bt = a.p.block_tables;
  p.ctx = a.p.context_lens;
  p.qlens = a.p.q_lens;
  p.out = a.out;
  p.lse = a.lse;
  p.item_off = reinterpret_cast<const int32_t*>(a.ws + a.L.item_off);
  p.first_item = reinterpret_cast<const int4*>(a.ws + a.L.first_item);
  p.items = reinterpret_cast<const int4*>(a.ws + a.L.items);
  p.o_part = reinterpret_cast<float*>(a.ws + a.L.o_part);
  p.lse_part = reinterpret_cast<float*>(a.ws + a.L.lse_part);
  p.flags = reinterpret_cast<int32_t*>(a.ws + a.L.header) + HDR_FLAGS;
  p.unit_info = reinterpret_cast<const int2*>(a.ws + a.L.unit_info);
  p.unit_cnt = reinterpret_cast<int32_t*>(a.ws + a.L.unit_cnt);
  p.units = a.v.units;
  p.ns_dec = a.v.ns_dec;
  p.scale_mode = a.scale_mode;
  p.Sq = a.p.max_q_len;
  p.Hq = a.p.num_q_heads;
  p.Hkv = a.p.num_kv_heads;
  p.G = a.p.num_q_heads / a.p.num_kv_heads;
  p.M = a.v.rows;
  p.RB = a.v.rb;
  p.bs = a.p.block_size;
  p.bs_shift = ilog2((uint32_t)a.p.block_size);
  p.maxb = a.p.max_blocks;
  p.nblocks = a.p.num_blocks;
  p.causal = a.p.causal;
  p.qk_scale = a.qk_scale;
  p.batch = a.p.batch;
  p.tt = a.v.tt;
  p.tt_shift = ilog2((uint32_t)a.v.tt);
  p.item_cost = a.v.item_cost;
  return p;
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t s) {
  const KernelParams prm = make_kernel_params(a);
  const bool toks = a.scale_mode == PA_SCALE_PER_TOKEN;
  if (a.v.path == 2) {
    if (a.kv_kind == KV_FP8)
      return a.p.head_dim == 128
                 ? launch_tc_fp8_d128(prm, kmap, vmap, a.v.ctas, a.v.mp, a.q_kind, toks, s)
                 : cudaErrorNotSupported;
    switch (a.p.head_dim) {
      case 128: return launch_tc_d128(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
      case 256: return launch_tc_d256(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
      default: return cudaErrorNotSupported;
    }
  }
  if (a.v.path == 1) {
    switch (a.p.head_dim) {
      case 64: return launch_mma_d64(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
      case 128: return launch_mma_d128(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
      case 256: return launch_mma_d256(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
      default: return cudaErrorNotSupported;
    }
  }
  if (a.p.head_dim == 64)
    return launch_simt_d64(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
  return cudaErrorNotSupported;
}

namespace {

struct ReduceParams {
  void* out;
  float* lse;
  const int32_t* hdr;
  const int32_t* red_units;
  const int2* unit_info;
  const float* o_part;
  const float* lse_part;
  int Sq, Hq, Hkv, G, M, RB, MP;
  int R;  // rows of a unit in the row space: M when a unit is one row block (the tile's
          // padding rows are left out), else MP (only the last block has padding rows)
};

constexpr int kReduceWarps = 8;

// The listed units come in two parts (the planner's order): units of at most
// kReduceWarpPieces pieces, then the rest.
//  * Few pieces: one warp per (unit, row), lanes over the head dimension (four floats a
//    lane); lane s holds piece s's log2-sum-exp, so the row's max and weights are one
//    shuffle reduction.  Each warp takes a contiguous run of rows (consecutive rows share
//    their unit, so the unit's entry is read once), and the next row's log2-sum-exps and
//    partial rows are in flight while the current row is merged: a warp's run costs about
//    one memory round trip plus the arithmetic of its rows.
//  * Many pieces: one CTA per (unit, row): warp w folds pieces w, w + 8, ... into a running
//    (max, weight sum, weighted sum), loading the partials of four pieces at a time (the
//    first four with the log2-sum-exps); the eight warps' results are then combined in
//    shared memory, so a unit cut into many pieces is merged by many SMs at once.
// Every sum runs in piece order.
template <int D>
struct RowBuf {
  static constexpr int D4 = D / 4;
  static constexpr int NV = (D4 + 31) / 32;  // float4 columns per lane
  static constexpr int CH = NV > 1 ? 2 : 4;  // pieces held at once (two rows' worth in flight)
  float ls;                                  // lane s: piece s's log2-sum-exp
  float4 o4[CH][NV];
};

// One row of a few-piece unit: the pieces' log2-sum-exps and the partial rows of the first
// CH pieces, issued together.  Rows past the unit's query rows load nothing.
template <int D>
__device__ __forceinline__ void load_row(const ReduceParams& p, int u, int2 info, int r,
                                         int lane, RowBuf<D>& b, int s0) {
  using B = RowBuf<D>;
  const int rg = (u % p.RB) * p.MP + r;
  const bool live = rg < p.M;
  const int ns = info.y;
  if (s0 == 0)
    b.ls = (live && lane < ns) ? __ldcg(&p.lse_part[(size_t)piece_slot(info.x, lane) * p.MP + r])
                               : -INFINITY;
#pragma unroll
  for (int j = 0; j < B::CH; ++j) {
    const int s = s0 + j;
    const bool ok = live && s < ns;
    const size_t part = ok ? (size_t)piece_slot(info.x, s) * p.MP + r : 0;
#pragma unroll
    for (int v = 0; v < B::NV; ++v) {
      const int c = lane + 32 * v;
      b.o4[j][v] = (ok && c < B::D4)
                       ? __ldcg(reinterpret_cast<const float4*>(p.o_part + part * D) + c)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// Merge the row whose first pieces sit in b and store it.
template <int D, int QK>
__device__ __forceinline__ void merge_row(const ReduceParams& p, int u, int2 info, int r,
                                          int lane, RowBuf<D>& b) {
  using B = RowBuf<D>;
  const int rg = (u % p.RB) * p.MP + r;
  if (rg >= p.M) return;  // uniform over the warp
  const int ns = info.y;  // <= kReduceWarpPieces
  float m = b.ls;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  const float wl = (b.ls == -INFINITY) ? 0.f : fast_exp2(b.ls - m);
  float W = wl;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(kFull, W, o);
  float4 acc[B::NV];
#pragma unroll
  for (int v = 0; v < B::NV; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < ns; s0 += B::CH) {
    if (s0 > 0) load_row<D>(p, u, info, r, lane, b, s0);
#pragma unroll
    for (int j = 0; j < B::CH; ++j) {
      const float x = __shfl_sync(kFull, wl, (s0 + j) & 31);  // 0 for pieces past ns
      const float xw = s0 + j < ns ? x : 0.f;
#pragma unroll
      for (int v = 0; v < B::NV; ++v) {
        acc[v].x += xw * b.o4[j][v].x;
        acc[v].y += xw * b.o4[j][v].y;
        acc[v].z += xw * b.o4[j][v].z;
        acc[v].w += xw * b.o4[j][v].w;
      }
    }
  }
  const int bq = u / (p.Hkv * p.RB), g = (u / p.RB) % p.Hkv;
  const size_t row = ((size_t)bq * p.Sq + rg / p.G) * p.Hq + g * p.G + rg % p.G;
  const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
  for (int v = 0; v < B::NV; ++v) {
    const int c = lane + 32 * v;
    if (c < B::D4)
      store_out4<QK>(p.out, row * D + 4 * c,
                     make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv));
  }
  if (lane == 0 && p.lse) p.lse[row] = W > 0.f ? (m + fast_log2(W)) * kLn2 : -INFINITY;
}

template <int D, int QK>
__global__ void __launch_bounds__(kReduceWarps * 32) reduce_kernel(const ReduceParams p) {
  constexpr int D4 = D / 4;
  constexpr int NV = (D4 + 31) / 32;  // float4 columns per lane
  __shared__ float s_m[kReduceWarps], s_w[kReduceWarps];
  __shared__ float4 s_acc[kReduceWarps][D4];
  // The work list (header, reduce list, unit table) is the planner's, and the planner has
  // finished before this grid starts: this grid starts once every CTA of the decode grid
  // has passed its own wait on the planner.  So the list is read before this grid's wait,
  // through L2 (these lines may sit stale in an SM's L1 from an earlier step), and only the
  // partials, which the decode writes, after it.
  const int nred = __ldcg(&p.hdr[HDR_NRED]), nsmall = __ldcg(&p.hdr[HDR_NRED_SMALL]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // few-piece rows: warp gw takes rows [w0, w1) of the nsmall * MP
  const int rows = nsmall * p.R, nw = gridDim.x * kReduceWarps;
  const int per = (rows + nw - 1) / nw, gw = blockIdx.x * kReduceWarps + warp;
  const int w0 = min(gw * per, rows), w1 = min(w0 + per, rows);
  const int wl0 = blockIdx.x;
  int us0 = 0, ul0 = 0;
  int2 infos0 = make_int2(0, 0), infol0 = make_int2(0, 0);
  if (w0 < w1) {
    us0 = __ldcg(&p.red_units[w0 / p.R]);
    infos0 = __ldcg(&p.unit_info[us0]);
  }
  if (wl0 < (nred - nsmall) * p.R) {
    ul0 = __ldcg(&p.red_units[nsmall + wl0 / p.R]);
    infol0 = __ldcg(&p.unit_info[ul0]);
  }
  grid_dependency_wait();  // partials come from the decode kernel launched just before
  // the next kernel may start launching now: it is held in its own grid_dependency_wait
  // until this grid has completed, and it cannot take the place of a CTA of this grid
  grid_dependents_launch();
  // few-piece units: the next row's loads are issued before the current row is merged
  if (w0 < w1) {
    RowBuf<D> ba, bb;
    int u = us0;
    int2 info = infos0;
    load_row<D>(p, u, info, w0 % p.R, lane, ba, 0);
    // the row after w (its unit's entry read again only where the unit changes)
    auto next_meta = [&](int w, int& un, int2& in) {
      un = u;
      in = info;
      if ((w + 1) % p.R == 0) {
        un = __ldcg(&p.red_units[(w + 1) / p.R]);
        in = __ldcg(&p.unit_info[un]);
      }
    };
    for (int w = w0; w < w1; w += 2) {
      int un = u;
      int2 in = info;
      if (w + 1 < w1) {
        next_meta(w, un, in);
        load_row<D>(p, un, in, (w + 1) % p.R, lane, bb, 0);
      }
      merge_row<D, QK>(p, u, info, w % p.R, lane, ba);
      if (w + 1 >= w1) break;
      u = un;
      info = in;
      if (w + 2 < w1) {
        next_meta(w + 1, un, in);
        load_row<D>(p, un, in, (w + 2) % p.R, lane, ba, 0);
      }
      merge_row<D, QK>(p, u, info, (w + 1) % p.R, lane, bb);
      u = un;
      info = in;
    }
  }
  // many-piece units: a CTA per row
  for (int w = wl0; w < (nred - nsmall) * p.R; w += gridDim.x) {
    const int u = w == wl0 ? ul0 : __ldcg(&p.red_units[nsmall + w / p.R]), r = w % p.R;
    const int rb = u % p.RB, rg = rb * p.MP + r;
    if (rg >= p.M) continue;  // uniform over the CTA
    const int2 info = w == wl0 ? infol0 : __ldcg(&p.unit_info[u]);
    float m = -INFINITY, W = 0.f;
    float4 acc[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    // batches of up to 32 pieces per warp: lane j holds the weight of piece s0 + 8 j; the
    // batch's log2-sum-exps and its first four partial rows are loaded together
    for (int s0 = warp; s0 < info.y; s0 += 32 * kReduceWarps) {
      const int sl = s0 + lane * kReduceWarps;
      const int cnt = min(32, (info.y - s0 + kReduceWarps - 1) / kReduceWarps);
      float4 o[4][NV];
      auto load4 = [&](int j0) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const bool ok = j0 + jj < cnt;
          const size_t part = ok ? (size_t)piece_slot(info.x, s0 + (j0 + jj) * kReduceWarps) * p.MP + r : 0;
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            const int c = lane + 32 * v;
            o[jj][v] = (ok && c < D4) ? reinterpret_cast<const float4*>(p.o_part + part * D)[c]
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      };
      const float ls = sl < info.y ? p.lse_part[(size_t)piece_slot(info.x, sl) * p.MP + r]
                                   : -INFINITY;
      load4(0);
      float mb = ls;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o2));
      if (mb == -INFINITY) continue;  // no key of this row in the batch (uniform)
      const float mn = fmaxf(m, mb);
      const float sc = m == -INFINITY ? 0.f : fast_exp2(m - mn);
      m = mn;
      W *= sc;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        acc[v].x *= sc;
        acc[v].y *= sc;
        acc[v].z *= sc;
        acc[v].w *= sc;
      }
      const float wl = ls == -INFINITY ? 0.f : fast_exp2(ls - m);
      float wsum = wl;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) wsum += __shfl_xor_sync(kFull, wsum, o2);
      W += wsum;
      for (int j0 = 0; j0 < cnt; j0 += 4) {
        if (j0 > 0) load4(j0);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const float x = __shfl_sync(kFull, wl, (j0 + jj) & 31);
          const float xw = j0 + jj < cnt ? x : 0.f;
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            acc[v].x += xw * o[jj][v].x;
            acc[v].y += xw * o[jj][v].y;
            acc[v].z += xw * o[jj][v].z;
            acc[v].w += xw * o[jj][v].w;
          }
        }
      }
    }
    if (lane == 0) {
      s_m[warp] = m;
      s_w[warp] = W;
    }
#pragma unroll
    for (int v = 0; v < NV; ++v)
      if (lane + 32 * v < D4) s_acc[warp][lane + 32 * v] = acc[v];
    __syncthreads();
    float mt = -INFINITY;
#pragma unroll
    for (int k = 0; k < kReduceWarps; ++k) mt = fmaxf(mt, s_m[k]);
    float Wt = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    const int c = threadIdx.x;
#pragma unroll
    for (int k = 0; k < kReduceWarps; ++k) {
      if (s_m[k] == -INFINITY) continue;
      const float sc = fast_exp2(s_m[k] - mt);
      Wt += sc * s_w[k];
      if (c < D4) {
        const float4 a = s_acc[k][c];
        O.x += sc * a.x;
        O.y += sc * a.y;
        O.z += sc * a.z;
        O.w += sc * a.w;
      }
    }
    const int b = u / (p.Hkv * p.RB), g = (u / p.RB) % p.Hkv;
    const size_t row = ((size_t)b * p.Sq + rg / p.G) * p.Hq + g * p.G + rg % p.G;
    if (c < D4) {
      const float inv = Wt > 0.f ? 1.f / Wt : 0.f;
      store_out4<QK>(p.out, row * D + 4 * c, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
    }
    if (c == 0 && p.lse) p.lse[row] = Wt > 0.f ? (mt + fast_log2(Wt)) * kLn2 : -INFINITY;
    __syncthreads();  // shared results are rewritten by the next row
  }
}

// CTAs of a reduce kernel instance that fit on one SM at once, per device (0: not yet asked).
template <int D, int QK>
int reduce_blocks_per_sm() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, reduce_kernel<D, QK>, kReduceWarps * 32, 0) !=
      cudaSuccess)
    return 0;
  if (dev >= 0 && dev < 64 && nb > 0) cached[dev].store(nb, std::memory_order_relaxed);
  return nb;
}

// need: CTAs the rows could use; the grid is capped at what fits on the GPU at once, so every
// CTA is resident when the decode has finished and the warps' runs of rows overlap their loads
template <int D>
cudaError_t launch_reduce_d(const ReduceParams& p, int q_kind, long long need, int sms,
                            cudaStream_t s) {
  const int per_sm = q_kind == Q_BF16 ? reduce_blocks_per_sm<D, Q_BF16>()
                                      : reduce_blocks_per_sm<D, Q_FP16>();
  if (per_sm <= 0) return cudaErrorUnknown;
  const int grid = (int)std::max(1LL, std::min(need, (long long)per_sm * sms));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kReduceWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (q_kind == Q_BF16) return cudaLaunchKernelEx(&cfg, reduce_kernel<D, Q_BF16>, p);
  return cudaLaunchKernelEx(&cfg, reduce_kernel<D, Q_FP16>, p);
}

}  // namespace

cudaError_t launch_reduce(const DecodeArgs& a, cudaStream_t s) {
  ReduceParams p;
  p.out = a.out;
  p.lse = a.lse;
  p.hdr = reinterpret_cast<const int32_t*>(a.ws + a.L.header);
  p.red_units = reinterpret_cast<const int32_t*>(a.ws + a.L.red_units);
  p.unit_info = reinterpret_cast<const int2*>(a.ws + a.L.unit_info);
  p.o_part = reinterpret_cast<const float*>(a.ws + a.L.o_part);
  p.lse_part = reinterpret_cast<const float*>(a.ws + a.L.lse_part);
  p.Sq = a.p.max_q_len;
  p.Hq = a.p.num_q_heads;
  p.Hkv = a.p.num_kv_heads;
  p.G = a.p.num_q_heads / a.p.num_kv_heads;
  p.M = a.v.rows;
  p.RB = a.v.rb;
  p.MP = a.v.mp;
  p.R = a.v.rb == 1 ? std::min(a.v.rows, a.v.mp) : a.v.mp;
  if (a.v.units == 0) return cudaSuccess;
  // Rows to merge (R a unit): few-piece units take a warp per (unit, row), so at most
  // units x R / 8 CTAs; many-piece units a CTA per row, and as a unit of more than
  // kReduceWarpPieces pieces holds that many of the 2C partial slots, at most
  // 2C / (kReduceWarpPieces + 1) units are of that kind.  The grid is capped at the CTAs that
  // fit at once; each warp then takes a run of rows, each CTA every grid-th many-piece row.
  int sms = a.v.sms;
  if (sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorUnknown;
  }
  const long long units = a.v.units, rows = p.R;
  const long long large_units =
      std::min(units, 2LL * a.v.ctas / (kReduceWarpPieces + 1));
  const long long need = std::max((units * rows + kReduceWarps - 1) / kReduceWarps,
                                  large_units * rows);
  switch (a.p.head_dim) {
    case 64: return launch_reduce_d<64>(p, a.q_kind, need, sms, s);
    case 128: return launch_reduce_d<128>(p, a.q_kind, need, sms, s);
    case 256: return launch_reduce_d<256>(p, a.q_kind, need, sms, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace pa
