// pa_append_kv: a decode step's new K/V rows written into the paged cache, with fp8
// quantise-on-write.
//
// New row i < q_lens[b] of sequence b is cache position pos = context_lens[b] - q_lens[b] + i
// (the new tokens are the last q_lens[b] of the context_lens[b] cached tokens, as the decode
// reads them), i.e. slot pos % block_size of physical block block_tables[b][pos / block_size]
// ("HSTU Paged Attention", RecSDK issue 1281, background: K/V live in a paged cache reached
// through per-sequence page lists).  A 16-bit cache receives the row unchanged.  An fp8 cache
// receives OCP E4M3 codes of the row over its scale, in one of the scale modes of "Optimize
// paged-attention metadata decode" (FlyDSL PR #910, Breaking Changes: per_token_kv):
// per-token, the row's scale is amax / 448 (1 for an all-zero row) and is written beside the
// codes; per-tensor, the caller's one scale is read; with no scale the values are encoded as
// they are.  The scale and every quotient are IEEE fp32 operations (correctly rounded
// division), and the code is the E4M3 value nearest to the quotient, ties to even, magnitudes
// past 448 saturating to 448.
//
// One warp per (sequence, new row, kv head): each lane holds D / 32 consecutive elements
// (8 to 16 bytes of input), the row's amax is a shuffle reduction, and the codes go out as
// one 2-, 4- or 8-byte store per lane.  The work is a few bytes per new token, a latency-bound
// kernel on the path before pa_plan / pa_decode.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kAppendWarps = 8;

struct AppendParams {
  const char* k_new;
  const char* v_new;
  const int32_t* bt;
  const int32_t* ctx;
  const int32_t* qlens;
  char* k_cache;
  char* v_cache;
  float* k_scale;
  float* v_scale;
  int32_t* flags;
  long long rows;  // B * Sq * Hkv
  int Sq, Hkv, bs, bs_shift, maxb, nblocks, scale_mode;
};

template <int QK>
__device__ __forceinline__ float to_f32(uint16_t h) {
  if constexpr (QK == Q_BF16)
    return __uint_as_float((uint32_t)h << 16);
  else
    return __half2float(__ushort_as_half(h));
}

// Two fp32 values to two E4M3 codes (lo -> low byte): round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t r;
  asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n mov.b16 %0, t;\n}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}

template <int D, int QK, bool FP8>
__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(const AppendParams p) {
  constexpr int E = D / 32;  // elements per lane: 2, 4 or 8
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * kAppendWarps;
  grid_dependency_wait();
  for (long long row = (long long)blockIdx.x * kAppendWarps + (threadIdx.x >> 5); row < p.rows;
       row += warps) {
    const int g = (int)(row % p.Hkv);
    const int i = (int)((row / p.Hkv) % p.Sq);
    const int b = (int)(row / ((long long)p.Hkv * p.Sq));
    const int n = __ldg(p.ctx + b), ql = __ldg(p.qlens + b);
    const long long cap = (long long)p.maxb * p.bs;
    if (ql < 0 || ql > p.Sq || n < ql || (long long)n > cap) {
      if (lane == 0 && i == 0 && g == 0 && p.flags) atomicOr(p.flags, PA_FLAG_BAD_LENGTHS);
      continue;
    }
    if (i >= ql) continue;
    const int pos = n - ql + i;
    const int blk = __ldg(p.bt + (size_t)b * p.maxb + (pos >> p.bs_shift));
    if (blk < 0 || blk >= p.nblocks) {
      if (lane == 0 && p.flags) atomicOr(p.flags, PA_FLAG_BAD_BLOCK_ID);
      continue;
    }
    const size_t crow = ((size_t)blk * p.bs + (pos & (p.bs - 1))) * p.Hkv + g;  // cache row
    const size_t src = (size_t)row * D + (size_t)lane * E;                       // element
#pragma unroll
    for (int t = 0; t < 2; ++t) {  // K, then V
      const char* nw = t ? p.v_new : p.k_new;
      char* cache = t ? p.v_cache : p.k_cache;
      if constexpr (!FP8) {
        // the row as it is: E 16-bit values per lane
        const char* s = nw + src * 2;
        char* d = cache + (crow * D + (size_t)lane * E) * 2;
        if constexpr (E == 8)
          *reinterpret_cast<uint4*>(d) = __ldg(reinterpret_cast<const uint4*>(s));
        else if constexpr (E == 4)
          *reinterpret_cast<uint2*>(d) = __ldg(reinterpret_cast<const uint2*>(s));
        else
          *reinterpret_cast<uint32_t*>(d) = __ldg(reinterpret_cast<const uint32_t*>(s));
      } else {
        uint16_t h[E];
        if constexpr (E == 8) {
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(nw + src * 2));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            h[2 * k] = (uint16_t)(ws[k] & 0xffffu);
            h[2 * k + 1] = (uint16_t)(ws[k] >> 16);
          }
        } else if constexpr (E == 4) {
          const uint2 w = __ldg(reinterpret_cast<const uint2*>(nw + src * 2));
          h[0] = (uint16_t)(w.x & 0xffffu);
          h[1] = (uint16_t)(w.x >> 16);
          h[2] = (uint16_t)(w.y & 0xffffu);
          h[3] = (uint16_t)(w.y >> 16);
        } else {
          const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(nw + src * 2));
          h[0] = (uint16_t)(w & 0xffffu);
          h[1] = (uint16_t)(w >> 16);
        }
        float x[E];
#pragma unroll
        for (int k = 0; k < E; ++k) x[k] = to_f32<QK>(h[k]);
        float s = 1.f;
        if (p.scale_mode == PA_SCALE_PER_TOKEN) {
          float amax = 0.f;
#pragma unroll
          for (int k = 0; k < E; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
          s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
          if (lane == 0) (t ? p.v_scale : p.k_scale)[crow] = s;
        } else if (p.scale_mode == PA_SCALE_PER_TENSOR) {
          s = __ldg(t ? p.v_scale : p.k_scale);
        }
        uint32_t c[E / 2];
#pragma unroll
        for (int k = 0; k < E / 2; ++k) {
          const float a = p.scale_mode == PA_SCALE_NONE ? x[2 * k] : __fdiv_rn(x[2 * k], s);
          const float bq = p.scale_mode == PA_SCALE_NONE ? x[2 * k + 1] : __fdiv_rn(x[2 * k + 1], s);
          c[k] = e4m3x2_rn_sat(a, bq);
        }
        char* d = cache + crow * D + (size_t)lane * E;
        if constexpr (E == 8)
          *reinterpret_cast<uint2*>(d) = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
        else if constexpr (E == 4)
          *reinterpret_cast<uint32_t*>(d) = c[0] | (c[1] << 16);
        else
          *reinterpret_cast<uint16_t*>(d) = (uint16_t)c[0];
      }
    }
  }
  grid_dependents_launch();
}

template <int D>
cudaError_t launch_append_d(const AppendParams& p, int qk, bool fp8, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kAppendWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (fp8) {
    if (qk == Q_BF16) return cudaLaunchKernelEx(&cfg, append_kernel<D, Q_BF16, true>, p);
    return cudaLaunchKernelEx(&cfg, append_kernel<D, Q_FP16, true>, p);
  }
  if (qk == Q_BF16) return cudaLaunchKernelEx(&cfg, append_kernel<D, Q_BF16, false>, p);
  return cudaLaunchKernelEx(&cfg, append_kernel<D, Q_FP16, false>, p);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_append_kv(const pa_config* cfg, const void* k_new, const void* v_new,
                                  const int32_t* block_tables, const int32_t* context_lens,
                                  const int32_t* q_lens, void* k_cache, void* v_cache,
                                  float* k_scale, float* v_scale, int32_t* flags,
                                  pa_stream stream) {
  if (!cfg || !k_new || !v_new || !block_tables || !context_lens || !q_lens || !k_cache ||
      !v_cache)
    return PA_ERR_INVALID_ARG;
  const pa_config& c = *cfg;
  if (c.batch < 1 || c.max_q_len < 1 || c.num_kv_heads < 1 || c.max_blocks_per_seq < 1 ||
      c.num_blocks < 1 || c.head_dim < 1 || c.block_size < 1)
    return PA_ERR_INVALID_ARG;
  if (c.kv_scale_mode < PA_SCALE_NONE || c.kv_scale_mode > PA_SCALE_PER_TOKEN)
    return PA_ERR_INVALID_ARG;
  if (c.head_dim != 64 && c.head_dim != 128 && c.head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (c.block_size < 16 || c.block_size > 1024 || (c.block_size & (c.block_size - 1)))
    return PA_ERR_UNSUPPORTED;
  if (c.q_dtype != PA_BF16 && c.q_dtype != PA_FP16) return PA_ERR_UNSUPPORTED;
  if (c.kv_dtype != c.q_dtype && c.kv_dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  const bool fp8 = c.kv_dtype == PA_FP8_E4M3;
  if (!fp8 && c.kv_scale_mode != PA_SCALE_NONE) return PA_ERR_UNSUPPORTED;
  if (fp8 && c.kv_scale_mode != PA_SCALE_NONE && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  auto aligned = [](const void* ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) % a) == 0;
  };
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return PA_ERR_INVALID_ARG;
  if ((k_scale && !aligned(k_scale, 4)) || (v_scale && !aligned(v_scale, 4)) ||
      (flags && !aligned(flags, 4)))
    return PA_ERR_INVALID_ARG;
  AppendParams p;
  p.k_new = static_cast<const char*>(k_new);
  p.v_new = static_cast<const char*>(v_new);
  p.bt = block_tables;
  p.ctx = context_lens;
  p.qlens = q_lens;
  p.k_cache = static_cast<char*>(k_cache);
  p.v_cache = static_cast<char*>(v_cache);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.flags = flags;
  p.rows = (long long)c.batch * c.max_q_len * c.num_kv_heads;
  p.Sq = c.max_q_len;
  p.Hkv = c.num_kv_heads;
  p.bs = c.block_size;
  p.bs_shift = ilog2((uint32_t)c.block_size);
  p.maxb = c.max_blocks_per_seq;
  p.nblocks = c.num_blocks;
  p.scale_mode = fp8 ? c.kv_scale_mode : PA_SCALE_NONE;
  const long long ctas = (p.rows + kAppendWarps - 1) / kAppendWarps;
  const int grid = (int)(ctas < 65535 ? ctas : 65535);
  const int qk = c.q_dtype == PA_FP16 ? Q_FP16 : Q_BF16;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (c.head_dim) {
    case 64: e = launch_append_d<64>(p, qk, fp8, grid, s); break;
    case 128: e = launch_append_d<128>(p, qk, fp8, grid, s); break;
    default: e = launch_append_d<256>(p, qk, fp8, grid, s); break;
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
