// Persistent split-KV paged decode on CUDA cores, for query tiles of at most 8 rows.
//
// Page gather.  One producer warp streams the KV pages of its CTA's work items into a
// 4-stage shared-memory ring: for every tile of TT tokens it looks up the physical block of
// each page through the block table and issues one 4-D TMA box (D x 1 head x rows x 1
// block) per page for K and one for V, completing on the stage's mbarrier.  While the
// consumers work on stage s, the next three stages are in flight.  This is the GB300 form
// of the K/V ping-pong of "HSTU Paged Attention" (RecSDK issue 1281, optimisation plan:
// split the buffer into K/V tensors and two ping-pong stages, overlap the next chunk's load
// with the current chunk's use, chunk capacity derived from the buffer budget and D); here
// the buffer is shared memory, the copy engine is TMA, and the stage count is four.
//
// Math.  Eight consumer warps split each tile's tokens between token groups of LPT lanes;
// each lane owns DPL = D / LPT dimensions of every query row.  Per token a group forms the
// MP partial dot products, reduce-scatters them across its lanes with warp shuffles (each
// lane ends with one row's logit), updates that row's running max and sum, and broadcasts
// the MP softmax weights back for the P.V accumulation.  Each group keeps its own online
// softmax state, so groups never wait on one another inside an item; the states are merged
// with the log-sum-exp rule when the item ends (first across the groups of a warp with
// shuffles, then across warps through shared memory).  The running max is only moved when a
// logit exceeds it by more than 2^8 (logits are kept in log2 units), which keeps the
// rescale of the accumulators off the common path; the final normalisation uses the same
// reference max, so the result is exact up to rounding.
//
// fp8 caches are dequantised in registers (E4M3 pairs to half2 to float); a per-tensor K
// scale is folded into the query, a per-tensor V scale into the final normalisation, and
// per-token scales (staged with the tile by cp.async) into each logit and weight.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pa_internal.cuh"

namespace pa {

struct SimtParams {
  const void* q;
  const float* k_scale;
  const float* v_scale;
  const int32_t* bt;
  const int32_t* ctx;
  const int32_t* qlens;
  void* out;
  float* lse;
  const int32_t* item_off;
  const int4* items;
  float* o_part;
  float* lse_part;
  int32_t* flags;
  int scale_mode;
  int Sq, Hq, Hkv, G, M, RB, bs, maxb, nblocks, causal;
  float qk_scale;
};

template <int D, int MP, int KVK, bool TOKS>
struct SimtTraits {
  static constexpr int BPE = KVK == KV_FP8 ? 1 : 2;
  static constexpr int DPL = MP <= 4 ? 16 : 8;  // dims per lane
  static constexpr int LPT = D / DPL;            // lanes per token group
  static constexpr int GPW = 32 / LPT;           // token groups per warp
  static constexpr int NCW = 8;                  // consumer warps
  static constexpr int NG = NCW * GPW;           // token groups per CTA
  static constexpr int NTHREADS = (NCW + 1) * 32;
  static constexpr int TT = kTileBytes / (D * BPE);  // tokens per stage
  static constexpr int NSTAGE = 4;
  static constexpr int CB = DPL * BPE < 16 ? DPL * BPE : 16;  // bytes per chunk
  static constexpr int EPC = CB / BPE;                         // elements per chunk
  static constexpr int CH = DPL / EPC;                         // chunks per lane
  static constexpr int RSTRIDE = LPT / MP;  // lanes holding one row after the reduce-scatter
  static constexpr int KTILE = TT * D * BPE;
  static constexpr int STAGE = round_up(2 * KTILE + (TOKS ? 2 * TT * 4 : 0), 1024);
  static constexpr int QHDR = 128;
  static constexpr int QSLOT = round_up(QHDR + MP * D * 2, 128);
  static constexpr int MERGE = NCW * MP * D * 4 + 2 * NCW * MP * 4;
  static constexpr int OFF_Q = NSTAGE * STAGE;
  static constexpr int OFF_MERGE = OFF_Q + 2 * QSLOT;
  static constexpr int OFF_BAR = round_up(OFF_MERGE + MERGE, 64);
  static constexpr int NBAR = 2 * NSTAGE + 4;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;  // + alignment slack
  static_assert(MP <= LPT && LPT <= 32 && 32 % LPT == 0, "row tile vs lanes");
  static_assert(DPL % EPC == 0 && TT % 32 == 0 && TT <= 256, "tile shape");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// ---- element conversion -----------------------------------------------------------
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float* f) {
  f[0] = __uint_as_float(w << 16);
  f[1] = __uint_as_float(w & 0xffff0000u);
}
__device__ __forceinline__ void f16x2_to_f32(uint32_t w, float* f) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  float2 r = __half22float2(h);
  f[0] = r.x;
  f[1] = r.y;
}
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* f) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
  float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
  float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}

// Load one chunk of EPC cache elements from shared memory as floats.
template <int KVK, int EPC>
__device__ __forceinline__ void load_kv_chunk(const char* src, float* f) {
  if constexpr (KVK == KV_FP8) {
    if constexpr (EPC == 16) {
      const uint4 w = *reinterpret_cast<const uint4*>(src);
      e4m3x4_to_f32(w.x, f);
      e4m3x4_to_f32(w.y, f + 4);
      e4m3x4_to_f32(w.z, f + 8);
      e4m3x4_to_f32(w.w, f + 12);
    } else {
      const uint2 w = *reinterpret_cast<const uint2*>(src);
      e4m3x4_to_f32(w.x, f);
      e4m3x4_to_f32(w.y, f + 4);
    }
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if constexpr (KVK == KV_BF16)
        bf16x2_to_f32(ws[j], f + 2 * j);
      else
        f16x2_to_f32(ws[j], f + 2 * j);
    }
  }
}

// Load n 16-bit query elements (n a multiple of 8) from shared memory as floats.
template <int QK>
__device__ __forceinline__ void load_q_elems(const char* src, int n, float* f) {
  for (int c = 0; c < n / 8; ++c) {
    const uint4 w = *reinterpret_cast<const uint4*>(src + 16 * c);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if constexpr (QK == Q_BF16)
        bf16x2_to_f32(ws[j], f + 8 * c + 2 * j);
      else
        f16x2_to_f32(ws[j], f + 8 * c + 2 * j);
    }
  }
}

template <int QK>
__device__ __forceinline__ void store_out(void* out, size_t idx, float v) {
  if constexpr (QK == Q_BF16)
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
}

// Reduce-scatter of N values over the lanes of a token group, starting at lane offset OFF
// (= LPT / 2): after it, lane l of the group holds in v[0] the group sum of value
// number l / (LPT / N).
template <int N, int OFF>
__device__ __forceinline__ void reduce_scatter(float* v, int lane) {
  if constexpr (OFF > 0) {
    if constexpr (N > 1) {
      const bool upper = (lane & OFF) != 0;
#pragma unroll
      for (int j = 0; j < N / 2; ++j) {
        const float send = upper ? v[j] : v[j + N / 2];
        const float keep = upper ? v[j + N / 2] : v[j];
        v[j] = keep + __shfl_xor_sync(kFull, send, OFF);
      }
      reduce_scatter<N / 2, OFF / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], OFF);
      reduce_scatter<1, OFF / 2>(v, lane);
    }
  }
}

constexpr float kRescaleSlack = 8.0f;  // log2 units: weights stay <= 2^8 between rescales

template <int D, int MP, int KVK, int QK, bool TOKS>
__global__ void __launch_bounds__(SimtTraits<D, MP, KVK, TOKS>::NTHREADS, 1)
    decode_simt_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const SimtParams p) {
  using T = SimtTraits<D, MP, KVK, TOKS>;
  extern __shared__ char smem_raw[];
  char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty = full + T::NSTAGE;
  uint64_t* qfull = empty + T::NSTAGE;
  uint64_t* qempty = qfull + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(qempty + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < T::NSTAGE; ++s) {
      mbar_init(&full[s], TOKS ? 33 : 1);
      mbar_init(&empty[s], T::NCW);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qfull[s], 32);
      mbar_init(&qempty[s], T::NCW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int it_begin = p.item_off[blockIdx.x], it_end = p.item_off[blockIdx.x + 1];

  if (warp == T::NCW) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    const int box_rows = min(p.bs, T::TT);
    const int nbox = T::TT / box_rows;
    const uint32_t box_bytes = (uint32_t)box_rows * D * T::BPE;
    uint32_t tile_ctr = 0, item_ctr = 0;
    bool running = true;
    for (int it = it_begin; it < it_end && running; ++it) {
      const int4 item = p.items[it];
      const int u = item.x, t0 = item.y, t1 = item.z;
      const int b = u / (p.Hkv * p.RB), g = (u / p.RB) % p.Hkv, rb = u % p.RB;
      const int qs = item_ctr & 1;
      const uint32_t qph = (item_ctr >> 1) & 1;
      ++item_ctr;
      if (!mbar_wait(&qempty[qs], qph ^ 1, abort_flag)) {
        atomicOr(p.flags, PA_FLAG_WAIT_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      char* qslot = smem + T::OFF_Q + qs * T::QSLOT;
      if (t1 > t0) {
        if (lane == 0) cp_async_4(qslot + 16, p.ctx + b);
        if (lane == 1) cp_async_4(qslot + 20, p.qlens + b);
        constexpr int QCH = D * 2 / 16;  // 16-byte chunks per query row
        for (int c = lane; c < MP * QCH; c += 32) {
          const int r = c / QCH, cc = c % QCH, rg = rb * MP + r;
          if (rg < p.M) {
            const int i = rg / p.G, gq = rg % p.G;
            const char* src = reinterpret_cast<const char*>(p.q) +
                              ((((size_t)b * p.Sq + i) * p.Hq + (size_t)g * p.G + gq) * D) * 2 +
                              cc * 16;
            cp_async_16(qslot + T::QHDR + r * D * 2 + cc * 16, src);
          }
        }
      }
      cp_async_arrive_noinc(&qfull[qs]);
      if (t1 <= t0) continue;

      const int ntiles = ceil_div(t1 - t0, T::TT);
      const int32_t* btrow = p.bt + (size_t)b * p.maxb;
      auto box_block = [&](int k) {
        const int tokb = t0 + k * T::TT + lane * box_rows;
        return (lane < nbox && tokb < t1) ? __ldg(btrow + tokb / p.bs) : -1;
      };
      int blk_next = box_block(0);
      for (int k = 0; k < ntiles; ++k) {
        const int s = tile_ctr % T::NSTAGE;
        const uint32_t ph = (tile_ctr / T::NSTAGE) & 1;
        const int tok0 = t0 + k * T::TT;
        const int tokb = tok0 + lane * box_rows;
        const int blk = blk_next;
        const bool want = lane < nbox && tokb < t1;
        const bool ok = want && blk >= 0 && blk < p.nblocks;
        if (want && !ok) atomicOr(p.flags, PA_FLAG_BAD_BLOCK_ID);
        const uint32_t nvalid = __popc(__ballot_sync(kFull, ok));
        if (k + 1 < ntiles) blk_next = box_block(k + 1);  // overlap the next lookup
        if (!mbar_wait(&empty[s], ph ^ 1, abort_flag)) {
          atomicOr(p.flags, PA_FLAG_WAIT_TIMEOUT);
          *abort_flag = 1;
          running = false;
          break;
        }
        char* st = smem + s * T::STAGE;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], nvalid * 2u * box_bytes);
        __syncwarp();
        if (ok) {
          const int row = tokb % p.bs;
          tma_load_4d(st + lane * box_bytes, &kmap, &full[s], 0, g, row, blk);
          tma_load_4d(st + T::KTILE + lane * box_bytes, &vmap, &full[s], 0, g, row, blk);
        }
        if constexpr (TOKS) {
          float* sks = reinterpret_cast<float*>(st + 2 * T::KTILE);
          float* svs = sks + T::TT;
          for (int t = lane; t < T::TT; t += 32) {
            const int bb = __shfl_sync(kFull, blk, t / box_rows);
            const int tok = tok0 + t;
            if (tok < t1 && bb >= 0 && bb < p.nblocks) {
              const size_t idx = ((size_t)bb * p.bs + tok % p.bs) * p.Hkv + g;
              cp_async_4(sks + t, p.k_scale + idx);
              cp_async_4(svs + t, p.v_scale + idx);
            }
          }
          cp_async_arrive_noinc(&full[s]);
        }
        ++tile_ctr;
      }
    }
    // Let every copy this warp started land before the CTA may exit.
    cp_async_wait_all();
    const uint32_t first = tile_ctr > (uint32_t)T::NSTAGE ? tile_ctr - T::NSTAGE : 0;
    for (uint32_t j = first; j < tile_ctr; ++j)
      mbar_wait_drain(&full[j % T::NSTAGE], (j / T::NSTAGE) & 1);
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int grp = lane / T::LPT, lg = lane % T::LPT, gbase = lane - lg;
  const int r_own = lg / T::RSTRIDE;
  const bool tensor_scale = p.scale_mode == PA_SCALE_PER_TENSOR;
  const float kts = tensor_scale ? __ldg(p.k_scale) : 1.f;
  const float vts = tensor_scale ? __ldg(p.v_scale) : 1.f;
  const float qmul = p.qk_scale * kts;
  float* mbuf = reinterpret_cast<float*>(smem + T::OFF_MERGE);  // [NCW][MP]
  float* lbuf = mbuf + T::NCW * MP;                               // [NCW][MP]
  float* obuf = lbuf + T::NCW * MP;                               // [NCW][MP][D]
  constexpr int NCT = T::NCW * 32;
  uint32_t tile_ctr = 0, item_ctr = 0;

  int4 item_next = it_begin < it_end ? p.items[it_begin] : make_int4(0, 0, 0, -1);
  for (int it = it_begin; it < it_end; ++it) {
    const int4 item = item_next;
    if (it + 1 < it_end) item_next = p.items[it + 1];
    const int u = item.x, t0 = item.y, t1 = item.z, slot = item.w;
    const int b = u / (p.Hkv * p.RB), g = (u / p.RB) % p.Hkv, rb = u % p.RB;
    const int qs = item_ctr & 1;
    const uint32_t qph = (item_ctr >> 1) & 1;
    ++item_ctr;
    if (!mbar_wait(&qfull[qs], qph, abort_flag)) {
      atomicOr(p.flags, PA_FLAG_WAIT_TIMEOUT);
      *abort_flag = 1;
    }
    const char* qslot = smem + T::OFF_Q + qs * T::QSLOT;
    const int n = *reinterpret_cast<const int*>(qslot + 16);
    const int ql = *reinterpret_cast<const int*>(qslot + 20);
    float q[MP][T::DPL];
#pragma unroll
    for (int r = 0; r < MP; ++r) {
      const bool row_real = rb * MP + r < p.M;
#pragma unroll
      for (int c = 0; c < T::CH; ++c) {
        const int ch = lg + c * T::LPT;
        float f[T::EPC];
        load_q_elems<QK>(qslot + T::QHDR + (r * D + ch * T::EPC) * 2, T::EPC, f);
#pragma unroll
        for (int e = 0; e < T::EPC; ++e) q[r][c * T::EPC + e] = row_real ? f[e] * qmul : 0.f;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&qempty[qs]);
    if (t1 <= t0) continue;

    const int rg_own = rb * MP + r_own;
    const int i_own = rg_own / p.G;
    const bool valid_own = rg_own < p.M && i_own < ql;
    const int limit_own = valid_own ? (p.causal ? n - ql + i_own + 1 : n) : 0;

    float m_own = -INFINITY, l_own = 0.f;
    float o[MP][T::DPL];
#pragma unroll
    for (int r = 0; r < MP; ++r)
#pragma unroll
      for (int d = 0; d < T::DPL; ++d) o[r][d] = 0.f;

    const int ntiles = ceil_div(t1 - t0, T::TT);
    for (int k = 0; k < ntiles; ++k) {
      const int s = tile_ctr % T::NSTAGE;
      const uint32_t ph = (tile_ctr / T::NSTAGE) & 1;
      ++tile_ctr;
      if (!mbar_wait(&full[s], ph, abort_flag)) {
        atomicOr(p.flags, PA_FLAG_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
      const char* ks = smem + s * T::STAGE;
      const char* vs = ks + T::KTILE;
      const float* sks = reinterpret_cast<const float*>(ks + 2 * T::KTILE);
      const float* svs = sks + T::TT;
      const int tok0 = t0 + k * T::TT;
      const int n_in = min(T::TT, t1 - tok0);
      for (int base = warp * T::GPW; base < n_in; base += T::NG) {
        const int t = base + grp;
        const bool tv = t < n_in;
        const int tl = tv ? t : 0;
        float kf[T::DPL];
#pragma unroll
        for (int c = 0; c < T::CH; ++c)
          load_kv_chunk<KVK, T::EPC>(ks + (size_t)tl * D * T::BPE + (lg + c * T::LPT) * T::CB,
                                     kf + c * T::EPC);
        float acc[MP];
#pragma unroll
        for (int r = 0; r < MP; ++r) {
          float a = 0.f;
#pragma unroll
          for (int d = 0; d < T::DPL; ++d) a = fmaf(q[r][d], kf[d], a);
          acc[r] = a;
        }
        reduce_scatter<MP, T::LPT / 2>(acc, lane);
        float sc = acc[0];
        if constexpr (TOKS) sc *= sks[tl];
        const int tok = tok0 + t;
        sc = (tv && tok < limit_own) ? sc : -INFINITY;
        const bool need = sc > m_own + kRescaleSlack;
        if (__any_sync(kFull, need)) {
          const float mn = need ? sc : m_own;
          const float alpha = (mn == m_own) ? 1.f : fast_exp2(m_own - mn);
          l_own *= alpha;
          m_own = mn;
#pragma unroll
          for (int r = 0; r < MP; ++r) {
            const float a = __shfl_sync(kFull, alpha, gbase + r * T::RSTRIDE);
#pragma unroll
            for (int d = 0; d < T::DPL; ++d) o[r][d] *= a;
          }
        }
        const float pr = (sc == -INFINITY) ? 0.f : fast_exp2(sc - m_own);
        l_own += pr;
        float pv = pr;
        if constexpr (TOKS) pv *= svs[tl];
        float pw[MP];
#pragma unroll
        for (int r = 0; r < MP; ++r) pw[r] = __shfl_sync(kFull, pv, gbase + r * T::RSTRIDE);
        if (tv) {
          float vf[T::DPL];
#pragma unroll
          for (int c = 0; c < T::CH; ++c)
            load_kv_chunk<KVK, T::EPC>(vs + (size_t)t * D * T::BPE + (lg + c * T::LPT) * T::CB,
                                       vf + c * T::EPC);
#pragma unroll
          for (int r = 0; r < MP; ++r)
#pragma unroll
            for (int d = 0; d < T::DPL; ++d) o[r][d] = fmaf(pw[r], vf[d], o[r][d]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- merge the token groups' states: within the warp, then across warps
    float mr[MP], lr[MP];
#pragma unroll
    for (int r = 0; r < MP; ++r) {
      mr[r] = __shfl_sync(kFull, m_own, gbase + r * T::RSTRIDE);
      lr[r] = __shfl_sync(kFull, l_own, gbase + r * T::RSTRIDE);
    }
#pragma unroll
    for (int off = T::LPT; off < 32; off <<= 1) {
#pragma unroll
      for (int r = 0; r < MP; ++r) {
        const float mo = __shfl_xor_sync(kFull, mr[r], off);
        const float lo = __shfl_xor_sync(kFull, lr[r], off);
        const float mn = fmaxf(mr[r], mo);
        const float a = (mr[r] == -INFINITY) ? 0.f : fast_exp2(mr[r] - mn);
        const float bw = (mo == -INFINITY) ? 0.f : fast_exp2(mo - mn);
        lr[r] = lr[r] * a + lo * bw;
        mr[r] = mn;
#pragma unroll
        for (int d = 0; d < T::DPL; ++d)
          o[r][d] = o[r][d] * a + __shfl_xor_sync(kFull, o[r][d], off) * bw;
      }
    }
    if (lane < T::LPT) {
#pragma unroll
      for (int r = 0; r < MP; ++r) {
        if (lane == 0) {
          mbuf[warp * MP + r] = mr[r];
          lbuf[warp * MP + r] = lr[r];
        }
#pragma unroll
        for (int c = 0; c < T::CH; ++c) {
          const int d0 = (lg + c * T::LPT) * T::EPC;
#pragma unroll
          for (int e = 0; e < T::EPC; ++e)
            obuf[(warp * MP + r) * D + d0 + e] = o[r][c * T::EPC + e];
        }
      }
    }
    named_barrier_sync(1, NCT);
    for (int e = threadIdx.x; e < MP * D; e += NCT) {
      const int r = e / D, d = e % D, rg = rb * MP + r;
      if (rg >= p.M) continue;
      float mstar = -INFINITY;
#pragma unroll
      for (int w = 0; w < T::NCW; ++w) mstar = fmaxf(mstar, mbuf[w * MP + r]);
      float L = 0.f, O = 0.f;
      if (mstar != -INFINITY) {
#pragma unroll
        for (int w = 0; w < T::NCW; ++w) {
          const float mw = mbuf[w * MP + r];
          const float wt = (mw == -INFINITY) ? 0.f : fast_exp2(mw - mstar);
          L += lbuf[w * MP + r] * wt;
          O += obuf[(w * MP + r) * D + d] * wt;
        }
      }
      const float val = L > 0.f ? (O / L) * vts : 0.f;
      const float lse2 = L > 0.f ? mstar + fast_log2(L) : -INFINITY;
      if (slot < 0) {
        const int i = rg / p.G, h = g * p.G + rg % p.G;
        const size_t row = ((size_t)b * p.Sq + i) * p.Hq + h;
        store_out<QK>(p.out, row * D + d, val);
        if (d == 0 && p.lse) p.lse[row] = lse2 * kLn2;
      } else {
        p.o_part[((size_t)slot * MP + r) * D + d] = val;
        if (d == 0) p.lse_part[(size_t)slot * MP + r] = lse2;
      }
    }
    named_barrier_sync(1, NCT);
  }
}

template <int D, int MP, int KVK, int QK, bool TOKS>
cudaError_t launch_simt_instance(const SimtParams& prm, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, int grid, cudaStream_t s) {
  using T = SimtTraits<D, MP, KVK, TOKS>;
  auto kern = decode_simt_kernel<D, MP, KVK, QK, TOKS>;
  static bool attr_set = false;  // benign race: every caller sets the same value
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<grid, T::NTHREADS, T::SMEM, s>>>(kmap, vmap, prm);
  return cudaGetLastError();
}

// Dispatch over the row tile and the dtype combination for one head dimension.
template <int D>
cudaError_t launch_simt_for_dim(const SimtParams& prm, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, int grid, int mp, int kvk, int qk,
                                bool toks, cudaStream_t s) {
#define PA_SIMT_CASE(MP_, KVK_, QK_, TOKS_)                                      \
  if (mp == MP_ && kvk == KVK_ && qk == QK_ && toks == TOKS_)                   \
    return launch_simt_instance<D, MP_, KVK_, QK_, TOKS_>(prm, kmap, vmap, grid, s);
#define PA_SIMT_ROWS(MP_)                   \
  PA_SIMT_CASE(MP_, KV_BF16, Q_BF16, false) \
  PA_SIMT_CASE(MP_, KV_FP16, Q_FP16, false) \
  PA_SIMT_CASE(MP_, KV_FP8, Q_BF16, false)  \
  PA_SIMT_CASE(MP_, KV_FP8, Q_BF16, true)   \
  PA_SIMT_CASE(MP_, KV_FP8, Q_FP16, false)  \
  PA_SIMT_CASE(MP_, KV_FP8, Q_FP16, true)
  PA_SIMT_ROWS(1)
  PA_SIMT_ROWS(2)
  PA_SIMT_ROWS(4)
  PA_SIMT_ROWS(8)
#undef PA_SIMT_ROWS
#undef PA_SIMT_CASE
  return cudaErrorNotSupported;
}

SimtParams make_simt_params(const DecodeArgs& a);

}  // namespace pa
