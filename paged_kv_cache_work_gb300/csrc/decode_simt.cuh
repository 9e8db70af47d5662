// Persistent split-KV paged decode on CUDA cores, for query tiles of at most 8 rows.
//
// Page gather.  Warp 0 streams the KV pages of its CTA's work items into a 3-stage
// shared-memory ring while it also computes: for every tile of TT tokens it looks up the
// physical block of each page through the block table and issues one 4-D TMA box
// (D x 1 head x rows x 1 block) per page for K and one for V, completing on the stage's
// mbarrier; the next tile's block ids are fetched while the current tile is in flight.
// While the CTA works on stage s the next two stages are loading, and two CTAs share each
// SM, so four tiles per SM are always in flight.  This is the GB300 form of the K/V
// ping-pong of "HSTU Paged Attention" (RecSDK issue 1281, optimisation plan: K/V buffers in
// two ping-pong stages, the next chunk's load overlapping the current chunk's use, the chunk
// capacity derived from the buffer budget and D): the buffer is shared memory, the copy
// engine is TMA and the ring is deeper.
//
// Math.  The CTA's four warps split each tile's tokens between token groups of LPT lanes;
// a lane owns DPL = D / LPT dimensions of every query row.  A group takes two tokens per
// step: the 2 * MP partial dot products (packed fp32x2 FMA) are reduce-scattered across
// the group's lanes with warp shuffles so that each lane ends with one (token, row) logit;
// the two lanes of a row agree on its running max, each exponentiates its own logit, and
// the 2 * MP weights are broadcast back for the P.V accumulation (packed FMA again).  Each
// group keeps its own online-softmax state, merged with the log-sum-exp rule when an item
// ends (across the groups of a warp with shuffles, then across warps through shared
// memory).  Logits are in log2 units and the running max is only moved when a logit beats
// it by more than 2^8, which keeps the accumulator rescale off the common path; the final
// normalisation uses the same reference max, so the result is exact up to rounding.
//
// fp8 caches are dequantised in registers (E4M3 pairs to half2 to float); a per-tensor K
// scale is folded into the query, a per-tensor V scale into the final normalisation, and
// per-token scales (staged with the tile by cp.async) into each logit and weight.
#pragma once

#include "decode_common.cuh"

namespace pa {



template <int D_, int MP_, int KVK, bool TOKS_>
struct SimtTraits {
  static constexpr int D = D_;
  static constexpr int MP = MP_;
  static constexpr bool TOKS = TOKS_;
  static constexpr int BPE = KVK == KV_FP8 ? 1 : 2;
  static constexpr int LPT0 = cmax(D / 16, 2 * MP);
  static constexpr int LPT = (MP * (D / LPT0) > 64) ? 2 * LPT0 : LPT0;  // lanes per token group
  static constexpr int DPL = D / LPT;                                    // dims per lane
  static constexpr int GPW = 32 / LPT;                                   // groups per warp
  static constexpr int NW = 4;                                           // warps per CTA
  static constexpr int NG = NW * GPW;                                    // groups per CTA
  static constexpr int NTHREADS = NW * 32;
  static constexpr int NV = 2 * MP;           // values per group step: 2 tokens x MP rows
  static constexpr int RSTRIDE = LPT / NV;    // lanes holding one value after the scatter
  static constexpr int TT = kTileBytes / (D * BPE);  // tokens per stage
  static constexpr int NSTAGE = 3;
  static constexpr int NQ = NSTAGE;           // query slots (one per item a stage can start)
  static constexpr int CB = cmin(16, DPL * BPE);  // bytes per chunk
  static constexpr int EPC = CB / BPE;            // elements per chunk
  static constexpr int CH = DPL / EPC;            // chunks per lane
  static constexpr int KTILE = TT * D * BPE;
  static constexpr int NSLAB = 1;       // one TMA box spans the head dimension
  static constexpr int ROWB = D * BPE;  // bytes per tile row
  static constexpr bool WITH_Q = true;  // query rows travel through shared memory
  static constexpr int STAGE = round_up(2 * KTILE + (TOKS ? 2 * TT * 4 : 0), 1024);
  static constexpr int QSLOT = round_up(MP * D * 2, 128);
  // The item-end merge needs the warps' accumulators (MERGE_O) and running max and sum
  // (MERGE_ML).  The accumulators get their own buffer when two CTAs still fit on an SM;
  // otherwise they borrow the stage of the item's last tile, released after the merge.
  static constexpr int MERGE_O = NW * MP * D * 4;
  static constexpr int MERGE_ML = 2 * NW * MP * 4;
  static constexpr int OFF_Q = NSTAGE * STAGE;
  static constexpr int BASE_BYTES = OFF_Q + NQ * QSLOT + MERGE_ML + 64 + (2 * NSTAGE + NQ) * 8 + kFlagBytes + 1024;
  static constexpr bool OWN_MERGE = 2 * (BASE_BYTES + MERGE_O + 1024) <= 228 * 1024;
  static constexpr int OFF_MERGE = OFF_Q + NQ * QSLOT;
  static constexpr int OFF_MERGE_O = OFF_MERGE + MERGE_ML;
  static constexpr int OFF_BAR = round_up(OFF_MERGE_O + (OWN_MERGE ? MERGE_O : 0), 64);
  static constexpr int NBAR = 2 * NSTAGE + NQ;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + kFlagBytes + 1024;  // + alignment slack
  static constexpr int CTAS_PER_SM = 2 * (SMEM + 1024) <= 228 * 1024 ? 2 : 1;
  static_assert(NV <= LPT && LPT <= 32 && 32 % LPT == 0, "row tile vs lanes");
  static_assert(DPL % EPC == 0 && EPC % 2 == 0, "chunking");
  static_assert(MERGE_O <= STAGE, "merge buffer must fit in one stage");
  static_assert(TT % 32 == 0 && TT <= 256, "tile shape");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};


// Reduce-scatter of N values over the lanes of a token group, starting at lane offset OFF
// (= LPT / 2).  Each lane keeps its values in a lane-specific order: position p holds value
// p XOR v_own, where v_own = (lane within the group) / (LPT / N).  With that order every lane
// keeps the lower half and sends the upper half at each halving step, and the partner's
// upper-half entry is the same value, so a step is N / 2 shuffles and adds with no selects.
// Afterwards v[0] holds the group sum of value v_own.
template <int N, int OFF>
__device__ __forceinline__ void reduce_scatter(float* v) {
  if constexpr (OFF > 0) {
    if constexpr (N > 1) {
#pragma unroll
      for (int j = 0; j < N / 2; ++j) v[j] += __shfl_xor_sync(kFull, v[j + N / 2], OFF);
      reduce_scatter<N / 2, OFF / 2>(v);
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], OFF);
      reduce_scatter<1, OFF / 2>(v);
    }
  }
}

constexpr float kRescaleSlack = 8.0f;  // log2 units: weights stay <= 2^8 between rescales


// Per-tile context of a consumer lane.
template <int D, int MP, int KVK, bool TOKS>
struct StepCtx {
  const char* ks;     // K tile [TT][D]
  const char* vs;     // V tile [TT][D]
  const float* sks;   // per-token K scales [TT] (per-token mode)
  const float* svs;   // per-token V scales [TT]
  int tok0;           // first token of the tile
  int n_in;           // valid tokens in the tile
  int limit_own;      // keys visible to this lane's row
  int lg, gbase, tk_own;
};

// One step of a token group: tokens ta and ta + 1 of the tile.  The lane accumulates the
// token it owns after the reduce-scatter first (tk_own), so its partials are already in the
// scatter order: position tk * MP + r holds token (tk ^ tk_own), row (r ^ r_own).
template <bool CHECK, int D, int MP, int KVK, bool TOKS>
__device__ __forceinline__ void token_step(const StepCtx<D, MP, KVK, TOKS>& cx, int ta,
                                           const float2 (&q)[MP][SimtTraits<D, MP, KVK, TOKS>::DPL / 2],
                                           float2 (&o)[MP][SimtTraits<D, MP, KVK, TOKS>::DPL / 2],
                                           float& m_run, float& l_own) {
  using T = SimtTraits<D, MP, KVK, TOKS>;
  constexpr int PAIR = MP * T::RSTRIDE;  // lane distance to the same row's other token
  const int tb = ta + 1;
  const bool va = !CHECK || ta < cx.n_in, vb = !CHECK || tb < cx.n_in;
  // this lane's own token first
  const int t_first = cx.tk_own ? tb : ta, t_second = cx.tk_own ? ta : tb;
  const bool v_first = cx.tk_own ? vb : va, v_second = cx.tk_own ? va : vb;
  const int tl_first = (!CHECK || v_first) ? t_first : 0;
  const int tl_second = (!CHECK || v_second) ? t_second : 0;
  float acc[T::NV];
  {
    float2 s1[MP], s2[MP];
#pragma unroll
    for (int r = 0; r < MP; ++r) s1[r] = s2[r] = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < T::CH; ++c) {
      const int off = (cx.lg + c * T::LPT) * T::CB;
      const RawChunk<T::CB> r1 = lds_chunk<T::CB>(cx.ks + (size_t)tl_first * D * T::BPE + off);
      const RawChunk<T::CB> r2 = lds_chunk<T::CB>(cx.ks + (size_t)tl_second * D * T::BPE + off);
      float2 f1[T::EPC / 2], f2[T::EPC / 2];
      chunk_to_f2<KVK, T::CB>(r1, f1);
      chunk_to_f2<KVK, T::CB>(r2, f2);
#pragma unroll
      for (int e = 0; e < T::EPC / 2; ++e) {
#pragma unroll
        for (int r = 0; r < MP; ++r) {
          s1[r] = ffma2(q[r][c * T::EPC / 2 + e], f1[e], s1[r]);
          s2[r] = ffma2(q[r][c * T::EPC / 2 + e], f2[e], s2[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < MP; ++r) {
      acc[r] = s1[r].x + s1[r].y;
      acc[MP + r] = s2[r].x + s2[r].y;
    }
  }
  reduce_scatter<T::NV, T::LPT / 2>(acc);
  // this lane's (token, row) logit, masked
  float sc = acc[0];
  if constexpr (TOKS) sc *= cx.sks[tl_first];
  sc = ((!CHECK || v_first) && cx.tok0 + t_first < cx.limit_own) ? sc : -INFINITY;
  // the two lanes of a row agree on its running max
  const float s_pair = fmaxf(sc, __shfl_xor_sync(kFull, sc, PAIR));
  const bool need = s_pair > m_run + kRescaleSlack;
  if (__any_sync(kFull, need)) {
    const float mn = need ? s_pair : m_run;
    const float alpha = (mn == m_run) ? 1.f : fast_exp2(m_run - mn);
    l_own *= alpha;
    m_run = mn;
#pragma unroll
    for (int r = 0; r < MP; ++r) {
      const float a = __shfl_sync(kFull, alpha, cx.gbase + r * T::RSTRIDE);
#pragma unroll
      for (int d = 0; d < T::DPL / 2; ++d) {
        o[r][d].x *= a;
        o[r][d].y *= a;
      }
    }
  }
  const float pr = (sc == -INFINITY) ? 0.f : fast_exp2(sc - m_run);
  l_own += pr;
  float pv = pr;
  if constexpr (TOKS) pv = pr > 0.f ? pv * cx.svs[tl_first] : 0.f;
  float pw[T::NV];  // weights by value: token a rows, then token b rows
#pragma unroll
  for (int v = 0; v < T::NV; ++v) pw[v] = __shfl_sync(kFull, pv, cx.gbase + v * T::RSTRIDE);
  // P.V for both tokens (an invalid token has weight 0 and is skipped)
#pragma unroll
  for (int c = 0; c < T::CH; ++c) {
    const int off = (cx.lg + c * T::LPT) * T::CB;
    float2 fa[T::EPC / 2], fb[T::EPC / 2];
    if (!CHECK || va) {
      const RawChunk<T::CB> ra = lds_chunk<T::CB>(cx.vs + (size_t)ta * D * T::BPE + off);
      chunk_to_f2<KVK, T::CB>(ra, fa);
    } else {
#pragma unroll
      for (int e = 0; e < T::EPC / 2; ++e) fa[e] = make_float2(0.f, 0.f);
    }
    if (!CHECK || vb) {
      const RawChunk<T::CB> rb2 = lds_chunk<T::CB>(cx.vs + (size_t)tb * D * T::BPE + off);
      chunk_to_f2<KVK, T::CB>(rb2, fb);
    } else {
#pragma unroll
      for (int e = 0; e < T::EPC / 2; ++e) fb[e] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int r = 0; r < MP; ++r) {
      const float2 wa = make_float2(pw[r], pw[r]);
      const float2 wb = make_float2(pw[MP + r], pw[MP + r]);
#pragma unroll
      for (int e = 0; e < T::EPC / 2; ++e) {
        o[r][c * T::EPC / 2 + e] = ffma2(wa, fa[e], o[r][c * T::EPC / 2 + e]);
        o[r][c * T::EPC / 2 + e] = ffma2(wb, fb[e], o[r][c * T::EPC / 2 + e]);
      }
    }
  }
}


template <int D, int MP, int KVK, int QK, bool TOKS>
__global__ void __launch_bounds__(SimtTraits<D, MP, KVK, TOKS>::NTHREADS, 2)
    decode_simt_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const KernelParams p) {
  using T = SimtTraits<D, MP, KVK, TOKS>;
  extern __shared__ char smem_raw[];
  char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty = full + T::NSTAGE;
  uint64_t* qfull = empty + T::NSTAGE;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(qfull + T::NQ);
  volatile int* pend = abort_flag + 2;  // [4]: split pieces published, see finish_pending

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < T::NSTAGE; ++s) {
      mbar_init(&full[s], TOKS ? 33 : 1);
      mbar_init(&empty[s], T::NW);
    }
    for (int s = 0; s < T::NQ; ++s) mbar_init(&qfull[s], 32);
    *abort_flag = 0;
    pend[0] = -1;
    pend[2] = -1;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  __syncthreads();
  grid_dependency_wait();  // the work list comes from the planner launched just before
  // the next kernel may start launching now: it is held in its own grid_dependency_wait
  // until this grid has completed, and it cannot take the place of a CTA of this grid
  grid_dependents_launch();

  // the CTA's item range and its first item, read together (one round trip)
  const int it_begin = p.item_off[blockIdx.x], it_end = p.item_off[blockIdx.x + 1];
  const int4 first = p.first_item[blockIdx.x];
  TileProducer<T> prod;
  if (warp == 0) {
    prod.init(&p, &kmap, &vmap, smem, full, empty, qfull, abort_flag, lane, it_begin, it_end,
              first);
    prod.fill(T::NSTAGE - 1);  // every stage starts free
  }

  const int grp = lane / T::LPT, lg = lane % T::LPT, gbase = lane - lg;
  const int v_own = lg / T::RSTRIDE;      // value this lane holds after the scatter
  const int r_own = v_own % MP;           // its query row
  const int tk_own = v_own / MP;          // its token of the pair (0 or 1)
  constexpr int PAIR = MP * T::RSTRIDE;   // lane distance to the same row's other token
  const bool tensor_scale = p.scale_mode == PA_SCALE_PER_TENSOR;
  const float kts = tensor_scale ? __ldg(p.k_scale) : 1.f;
  const float vts = tensor_scale ? __ldg(p.v_scale) : 1.f;
  const float qmul = p.qk_scale * kts;
  float* mbuf = reinterpret_cast<float*>(smem + T::OFF_MERGE);  // [NW][MP]
  float* lbuf = mbuf + T::NW * MP;                                // [NW][MP]
  uint32_t tile_ctr = 0, items_seen = 0;
  int2 pend_even = make_int2(-1, 0), pend_odd = make_int2(-1, 0);  // held by thread 32

  int4 item_next = first;
  int n_next = 0, ql_next = 0;
  if (it_begin < it_end) {
    const int bn = item_next.x / (p.Hkv * p.RB);
    n_next = __ldg(p.ctx + bn);
    ql_next = __ldg(p.qlens + bn);
  }
  for (int it = it_begin; it < it_end; ++it) {
    const int4 item = item_next;
    const int n = n_next, ql = ql_next;
    if (it + 1 < it_end) {
      item_next = p.items[it + 1];
      const int bn = item_next.x / (p.Hkv * p.RB);
      n_next = __ldg(p.ctx + bn);
      ql_next = __ldg(p.qlens + bn);
    }
    const int u = item.x, t0 = item.y, t1 = item.z, slot = item.w;
    if (t1 <= t0) continue;
    const int b = u / (p.Hkv * p.RB), g = (u / p.RB) % p.Hkv, rb = u % p.RB;
    const int qs = items_seen % T::NQ;
    const uint32_t qph = (items_seen / T::NQ) & 1;
    ++items_seen;
    if (!mbar_wait(&qfull[qs], qph, abort_flag)) {
      atomicOr(p.flags, PA_FLAG_WAIT_TIMEOUT);
      *abort_flag = 1;
    }
    // query rows as float pairs, pre-scaled by sm_scale * log2(e) (and a per-tensor K scale),
    // stored in this lane's reduce-scatter order: slot r holds row r ^ r_own
    const char* qslot = smem + T::OFF_Q + qs * T::QSLOT;
    float2 q[MP][T::DPL / 2];
#pragma unroll
    for (int rp = 0; rp < MP; ++rp) {
      const int r = rp ^ r_own;
      const bool row_real = rb * MP + r < p.M;
#pragma unroll
      for (int c = 0; c < T::CH; ++c) {
        const int ch = lg + c * T::LPT;
#pragma unroll
        for (int e = 0; e < T::EPC / 2; ++e) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(qslot + (r * D + ch * T::EPC + 2 * e) * 2);
          const float2 f = q_pair<QK>(w);
          q[rp][c * T::EPC / 2 + e] = row_real ? make_float2(f.x * qmul, f.y * qmul)
                                               : make_float2(0.f, 0.f);
        }
      }
    }

    const int rg_own = rb * MP + r_own;
    const int i_own = rg_own / p.G;
    const bool valid_own = rg_own < p.M && i_own < ql;
    const int limit_own = valid_own ? (p.causal ? n - ql + i_own + 1 : n) : 0;

    float m_run = -INFINITY, l_own = 0.f;
    float2 o[MP][T::DPL / 2];
#pragma unroll
    for (int r = 0; r < MP; ++r)
#pragma unroll
      for (int d = 0; d < T::DPL / 2; ++d) o[r][d] = make_float2(0.f, 0.f);

    const int ntiles = ceil_div(t1 - t0, T::TT);
    int s_last = 0;
    for (int k = 0; k < ntiles; ++k) {
      if (warp == 0) prod.fill(tile_ctr + T::NSTAGE - 1);
      const int s = tile_ctr % T::NSTAGE;
      s_last = s;
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
      StepCtx<D, MP, KVK, TOKS> cx{ks, vs, sks, svs, tok0, n_in, limit_own, lg, gbase, tk_own};
      int base = warp * T::GPW * 2;
      for (; base + 2 * T::GPW <= n_in; base += T::NG * 2)  // every token of the warp step valid
        token_step<false>(cx, base + 2 * grp, q, o, m_run, l_own);
      for (; base < n_in; base += T::NG * 2)
        token_step<true>(cx, base + 2 * grp, q, o, m_run, l_own);
      __syncwarp();
      // without its own merge buffer, the item's last stage holds the merge until it is done
      if (lane == 0 && (T::OWN_MERGE || k + 1 < ntiles)) mbar_arrive(&empty[s]);
    }

    // ---- merge the token groups' states: within the warp, then across warps
    float* obuf = reinterpret_cast<float*>(
        smem + (T::OWN_MERGE ? T::OFF_MERGE_O : s_last * T::STAGE));  // [NW][MP][D]
    __syncwarp();
    float mr[MP], lr[MP];
#pragma unroll
    for (int r = 0; r < MP; ++r) {
      const int la = gbase + r * T::RSTRIDE, lb = la + PAIR;
      mr[r] = __shfl_sync(kFull, m_run, la);
      lr[r] = __shfl_sync(kFull, l_own, la) + __shfl_sync(kFull, l_own, lb);
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
        for (int d = 0; d < T::DPL / 2; ++d) {
          const float ox = __shfl_xor_sync(kFull, o[r][d].x, off);
          const float oy = __shfl_xor_sync(kFull, o[r][d].y, off);
          o[r][d] = make_float2(o[r][d].x * a + ox * bw, o[r][d].y * a + oy * bw);
        }
      }
    }
    if constexpr (!T::OWN_MERGE) {
      named_barrier_sync(1, T::NTHREADS);  // every warp is done reading the last stage
    } else {
      // every warp has released the item's last tile: refill the whole ring before merging,
      // so the copies keep flowing while the warps combine their states
      if (warp == 0) prod.fill(tile_ctr + T::NSTAGE - 1);
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
          for (int e = 0; e < T::EPC / 2; ++e)
            *reinterpret_cast<float2*>(&obuf[(warp * MP + r) * D + d0 + 2 * e]) =
                o[r][c * T::EPC / 2 + e];
        }
      }
    }
    named_barrier_sync(1, T::NTHREADS);
    for (int e = threadIdx.x; e < MP * D; e += T::NTHREADS) {
      const int r = e / D, d = e % D, rg = rb * MP + r;
      if (rg >= p.M) continue;
      float mstar = -INFINITY;
#pragma unroll
      for (int w = 0; w < T::NW; ++w) mstar = fmaxf(mstar, mbuf[w * MP + r]);
      float L = 0.f, O = 0.f;
      if (mstar != -INFINITY) {
#pragma unroll
        for (int w = 0; w < T::NW; ++w) {
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
    named_barrier_sync(1, T::NTHREADS);  // partials written
    if (slot >= 0 && threadIdx.x == 32 && __ldg(&p.unit_info[u].y) <= p.ns_dec) {
      __threadfence();
      publish_piece(p, u, slot, &pend_even, &pend_odd);
    }
    if (!T::OWN_MERGE && lane == 0) mbar_arrive(&empty[s_last]);
  }
  if (threadIdx.x == 32) {
    pend[0] = pend_even.x;
    pend[1] = pend_even.y;
    pend[2] = pend_odd.x;
    pend[3] = pend_odd.y;
  }
  if (warp == 0) prod.drain();
  named_barrier_sync(1, T::NTHREADS);  // no copy in flight: stage 0 is free for the merge
  finish_pending<D, MP, QK, T::NW>(
      p, pend, reinterpret_cast<float*>(smem + (T::OWN_MERGE ? T::OFF_MERGE_O : 0)),
      T::MERGE_O / 4, mbuf);
  zero_empty_units<D, MP, QK, T::NTHREADS>(p);
}

template <int D, int MP, int KVK, int QK, bool TOKS>
cudaError_t launch_simt_instance(const KernelParams& prm, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, int grid, cudaStream_t s) {
  using T = SimtTraits<D, MP, KVK, TOKS>;
  auto kern = decode_simt_kernel<D, MP, KVK, QK, TOKS>;
  static std::atomic<uint64_t> attr_done{0};  // devices whose limit is raised
  const cudaError_t e = set_smem_attr_once(attr_done, reinterpret_cast<const void*>(kern), T::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(T::NTHREADS);
  cfg.dynamicSmemBytes = T::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, prm);
}

// Dispatch over the row tile and the dtype combination for one head dimension.  Only caches
// whose rows are shorter than one 128-byte slab come here (64-dim fp8: every 16-bit cache
// and every other fp8 cache runs on tensor cores), so only fp8 instances are built.
#define PA_SIMT_ROWS(X, MP_)        \
  X(MP_, KV_FP8, Q_BF16, false)     \
  X(MP_, KV_FP8, Q_BF16, true)      \
  X(MP_, KV_FP8, Q_FP16, false)     \
  X(MP_, KV_FP8, Q_FP16, true)
#define PA_SIMT_ALL(X) PA_SIMT_ROWS(X, 1) PA_SIMT_ROWS(X, 2) PA_SIMT_ROWS(X, 4) PA_SIMT_ROWS(X, 8)

template <int D>
cudaError_t launch_simt_for_dim(const KernelParams& prm, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, int grid, int mp, int kvk, int qk,
                                bool toks, cudaStream_t s) {
#define PA_SIMT_CASE(MP_, KVK_, QK_, TOKS_)                                      \
  if (mp == MP_ && kvk == KVK_ && qk == QK_ && toks == TOKS_)                   \
    return launch_simt_instance<D, MP_, KVK_, QK_, TOKS_>(prm, kmap, vmap, grid, s);
  PA_SIMT_ALL(PA_SIMT_CASE)
#undef PA_SIMT_CASE
  return cudaErrorNotSupported;
}

// CTAs of one instance that fit on an SM (by shared memory).
template <int D>
int simt_ctas_per_sm_for_dim(int mp, int kvk, bool toks) {
#define PA_SIMT_OCC(MP_, KVK_, QK_, TOKS_) \
  if (mp == MP_ && kvk == KVK_ && toks == TOKS_) return SimtTraits<D, MP_, KVK_, TOKS_>::CTAS_PER_SM;
  PA_SIMT_ALL(PA_SIMT_OCC)
#undef PA_SIMT_OCC
  return 1;
}


}  // namespace pa
