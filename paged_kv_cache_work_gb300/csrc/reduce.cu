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
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_common.cuh"

namespace pa {

cudaError_t launch_simt_d64(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                            int, int, bool, cudaStream_t);
int simt_ctas_per_sm_d64(int, int, bool);
int simt_ctas_per_sm_d128(int, int, bool);
int simt_ctas_per_sm_d256(int, int, bool);

int mma_ctas_per_sm_d64(int, int, bool);
int mma_ctas_per_sm_d128(int, int, bool);
int mma_ctas_per_sm_d256(int, int, bool);
cudaError_t launch_mma_d64(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                           int, int, bool, cudaStream_t);
cudaError_t launch_mma_d128(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                            int, int, bool, cudaStream_t);
cudaError_t launch_mma_d256(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                            int, int, bool, cudaStream_t);

int simt_ctas_per_sm(int head_dim, int mp, int kvk, bool toks) {
  switch (head_dim) {
    case 64: return simt_ctas_per_sm_d64(mp, kvk, toks);
    case 128: return simt_ctas_per_sm_d128(mp, kvk, toks);
    default: return simt_ctas_per_sm_d256(mp, kvk, toks);
  }
}

int mma_ctas_per_sm(int head_dim, int mp, int kvk, bool toks) {
  switch (head_dim) {
    case 64: return mma_ctas_per_sm_d64(mp, kvk, toks);
    case 128: return mma_ctas_per_sm_d128(mp, kvk, toks);
    default: return mma_ctas_per_sm_d256(mp, kvk, toks);
  }
}
cudaError_t launch_simt_d128(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                             int, int, bool, cudaStream_t);
cudaError_t launch_simt_d256(const KernelParams&, const CUtensorMap&, const CUtensorMap&, int, int,
                             int, int, bool, cudaStream_t);

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
  p.items = reinterpret_cast<const int4*>(a.ws + a.L.items);
  p.o_part = reinterpret_cast<float*>(a.ws + a.L.o_part);
  p.lse_part = reinterpret_cast<float*>(a.ws + a.L.lse_part);
  p.flags = reinterpret_cast<int32_t*>(a.ws + a.L.header) + HDR_FLAGS;
  p.unit_info = reinterpret_cast<const int2*>(a.ws + a.L.unit_info);
  p.unit_cnt = reinterpret_cast<int32_t*>(a.ws + a.L.unit_cnt);
  p.units = a.v.units;
  p.merge_in_decode = a.merge_in_decode;
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
  return p;
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t s) {
  const KernelParams prm = make_kernel_params(a);
  const bool toks = a.scale_mode == PA_SCALE_PER_TOKEN;
  if (a.v.path == 1) {
    switch (a.p.head_dim) {
      case 64: return launch_mma_d64(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
      case 128: return launch_mma_d128(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
      case 256: return launch_mma_d256(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
      default: return cudaErrorNotSupported;
    }
  }
  switch (a.p.head_dim) {
    case 64: return launch_simt_d64(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
    case 128: return launch_simt_d128(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
    case 256: return launch_simt_d256(prm, kmap, vmap, a.v.ctas, a.v.mp, a.kv_kind, a.q_kind, toks, s);
    default: return cudaErrorNotSupported;
  }
}

namespace {

struct ReduceParams {
  void* out;
  float* lse;
  const int2* unit_info;
  const float* o_part;
  const float* lse_part;
  int Sq, Hq, Hkv, G, M, RB, MP, D;
  int q_kind;
};

constexpr int kReduceWarps = 4;

// One CTA per unit; warp w merges rows w, w + 4, ...: the lanes share the splits for the
// max and the weight sum, then the head dimensions for the weighted sum of the partials.
__global__ void __launch_bounds__(kReduceWarps * 32) reduce_kernel(const ReduceParams p) {
  grid_dependency_wait();  // partials come from the decode kernel launched just before
  const int u = blockIdx.x;
  const int2 info = p.unit_info[u];
  if (info.y != 1) {
    const int b = u / (p.Hkv * p.RB), g = (u / p.RB) % p.Hkv, rb = u % p.RB;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = warp; r < p.MP; r += kReduceWarps) {
      const int rg = rb * p.MP + r;
      if (rg >= p.M) continue;
      const int i = rg / p.G, h = g * p.G + rg % p.G;
      const size_t row = ((size_t)b * p.Sq + i) * p.Hq + h;
      float m = -INFINITY;
      for (int s = lane; s < info.y; s += 32)
        m = fmaxf(m, p.lse_part[(size_t)piece_slot(info.x, s) * p.MP + r]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      float W = 0.f;
      if (m != -INFINITY) {
        for (int s = lane; s < info.y; s += 32) {
          const float ls = p.lse_part[(size_t)piece_slot(info.x, s) * p.MP + r];
          W += ls == -INFINITY ? 0.f : fast_exp2(ls - m);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(kFull, W, o);
      }
      const float inv = W > 0.f ? 1.f / W : 0.f;
      for (int d = lane; d < p.D; d += 32) {
        float O = 0.f;
        if (W > 0.f) {
#pragma unroll 4
          for (int s = 0; s < info.y; ++s) {
            const size_t part = (size_t)piece_slot(info.x, s) * p.MP + r;
            const float ls = p.lse_part[part];
            const float w = ls == -INFINITY ? 0.f : fast_exp2(ls - m);
            O += w * p.o_part[part * p.D + d];
          }
        }
        const float val = O * inv;
        if (p.q_kind == Q_BF16)
          reinterpret_cast<__nv_bfloat16*>(p.out)[row * p.D + d] = __float2bfloat16_rn(val);
        else
          reinterpret_cast<__half*>(p.out)[row * p.D + d] = __float2half_rn(val);
      }
      if (lane == 0 && p.lse) p.lse[row] = W > 0.f ? (m + fast_log2(W)) * kLn2 : -INFINITY;
    }
  }
  grid_dependents_launch();
}

}  // namespace

cudaError_t launch_reduce(const DecodeArgs& a, cudaStream_t s) {
  ReduceParams p;
  p.out = a.out;
  p.lse = a.lse;
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
  p.D = a.p.head_dim;
  p.q_kind = a.q_kind;
  if (a.v.units == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.v.units);
  cfg.blockDim = dim3(kReduceWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, reduce_kernel, p);
}

}  // namespace pa
