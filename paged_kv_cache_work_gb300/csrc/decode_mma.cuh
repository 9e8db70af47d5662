// Persistent split-KV paged decode on tensor cores (mma.sync m16n8k16, fp32 accumulation),
// for query tiles of 16, 32 or 64 rows: the grouped-query tile G * Sq is then a real dense
// contraction of every staged key and value row against many query rows.
//
// Staging.  The page ring and its producer are those of the CUDA-core kernel, but each tile
// row lands in 128-byte column slabs written with the TMA 128-byte swizzle (16-byte chunk c
// of row r stored at chunk c ^ (r & 7)), so the ldmatrix loads below hit eight different
// bank groups for eight rows.
//
// Math.  Warp w owns WR 16-row tiles of the query block and one of TS token streams; the
// 16-token chunks of an item go round-robin to the streams.  Per chunk: S = Q K^T with K
// fragments from ldmatrix (Q fragments stay in registers for the whole item); an online
// softmax in log2 units on the accumulator layout (a row's 16 logits sit in the four lanes of
// a quad, so a row max is two shuffles; the running max only moves when a logit beats it by
// more than 2^8); P packed to 16-bit straight from the accumulators as the A operand of
// O += P V, with V fragments from ldmatrix.trans.  The streams' states are merged with the
// log-sum-exp rule when an item ends (a tree through the stage of the item's last tile).
//
// fp8 caches.  The MMA runs on f16 operands (E4M3 converts to f16 exactly; the query is
// converted from bf16 once per item).  ldmatrix moves the fp8 bytes as 16-bit pairs: for
// Q K^T each lane's four consecutive fp8 dimensions become its two k-pairs (the query
// fragments use the same permuted k order); for P V the transposed pairs hold two tokens
// of two adjacent dimensions, and a byte permute splits them into the fragments of an
// even-dimension and an odd-dimension n-block.
#pragma once

#include "decode_common.cuh"

namespace pa {

template <int D_, int MP_, int KVK_, bool TOKS_>
struct MmaTraits {
  static constexpr int D = D_;
  static constexpr int MP = MP_;
  static constexpr int KVK = KVK_;
  static constexpr bool TOKS = TOKS_;
  static constexpr bool FP8 = KVK == KV_FP8;
  static constexpr int BPE = FP8 ? 1 : 2;
  static constexpr int NW = 4;
  static constexpr int NTHREADS = NW * 32;
  static constexpr int WR = (D <= 128 && MP >= 32) ? 2 : 1;  // 16-row tiles per warp
  static constexpr int RBW = MP / (16 * WR);                 // row blocks
  static constexpr int TS = NW / RBW;                        // token streams
  static constexpr int TT = kTileBytes / (D * BPE);          // tokens per stage
  static constexpr int CPT = TT / 16;                        // 16-token chunks per tile
  static constexpr int NSTAGE = 3;
  static constexpr int NB = D / 8;                          // n-blocks of the output
  static constexpr int MERGE_SLOT_O = WR * NB * 4 * 32 * 4;  // one warp's accumulators
  static constexpr int MERGE_O = (NW / 2) * MERGE_SLOT_O;    // tree-merge buffer (last stage)
  static constexpr int ML_BYTES = round_up(cmax((NW / 2) * WR * 4 * 32 * 4, 2 * MP * 4), 128);
  static constexpr int ROWB = 128;       // swizzled slabs of 128 bytes per row
  static constexpr int NSLAB = D * BPE / 128;
  static constexpr int SLAB = TT * ROWB;  // bytes of one slab of a tile
  static constexpr int KTILE = TT * D * BPE;
  static constexpr int STAGE = round_up(2 * KTILE + (TOKS ? 2 * TT * 4 : 0), 1024);
  // Query fragments are read from global memory at the start of an item (staging them in
  // shared memory with the item's first tile measured slower: the wait at an item's start is
  // the copy pipeline refilling, not the query rows).
  static constexpr bool WITH_Q = false;
  static constexpr int NQ = 1;
  static constexpr int QSLOT = 0;
  static constexpr int OFF_Q = NSTAGE * STAGE;
  static constexpr int OFF_ML = OFF_Q + NQ * QSLOT;  // merge max/sum + merge stats
  static constexpr int OFF_BAR = round_up(OFF_ML + ML_BYTES, 64);
  static constexpr int NBAR = 2 * NSTAGE + NQ;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + kFlagBytes + 1024;
  static constexpr int CTAS_PER_SM = 2 * (SMEM + 1024) <= 228 * 1024 ? 2 : 1;
  static_assert(D * BPE >= 128 && (D * BPE) % 128 == 0, "whole 128-byte slabs");
  static_assert(MP % (16 * WR) == 0 && NW % RBW == 0, "row blocks");
  static_assert(TT % 32 == 0 && TT <= 256, "tile shape");
  static_assert(MERGE_O <= STAGE, "merge buffer must fit in one stage");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// ---- PTX wrappers -------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A * B with A 16x16, B 16x8 (both bf16 or both f16), D fp32.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Two floats to a packed 16-bit pair (low half = x).
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float x, float y) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Two E4M3 codes (low byte first) to an f16 pair.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xffffu), __NV_E4M3);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Byte permute: result byte i = byte sel_i of the 8-byte value {hi:lo}.
__device__ __forceinline__ uint32_t prmt(uint32_t lo, uint32_t hi, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(lo), "r"(hi), "r"(sel));
  return r;
}

// Shared-memory address of 16-byte chunk `chunk` (0..7 within its slab) of tile row `row`.
template <class T>
__device__ __forceinline__ uint32_t tile_chunk_addr(uint32_t tile, int row, int slab, int chunk) {
  return tile + slab * T::SLAB + row * T::ROWB + ((chunk ^ (row & 7)) << 4);
}

template <int D, int MP, int KVK, int QK, bool TOKS>
__global__ void __launch_bounds__(MmaTraits<D, MP, KVK, TOKS>::NTHREADS, 2)
    decode_mma_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const KernelParams p) {
  using T = MmaTraits<D, MP, KVK, TOKS>;
  constexpr bool F16 = KVK != KV_BF16;  // operand type of the MMA: f16 for f16 and fp8 caches
  constexpr int WR = T::WR, NB = T::NB, KSTEPS = D / 16;
  extern __shared__ char smem_raw[];
  char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty = full + T::NSTAGE;
  uint64_t* qfull = empty + T::NSTAGE;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(qfull + T::NQ);
  volatile int* pend = abort_flag + 2;       // [4]: split pieces published, see finish_pending
  volatile int* cnt_seen_s = abort_flag + 6;  // published pieces of the item's unit, seen late
  float* mlbuf = reinterpret_cast<float*>(smem + T::OFF_ML);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = lane >> 2, qi = lane & 3;  // accumulator row within a tile / column pair
  const int rblk = warp % T::RBW, ts = warp / T::RBW;
  if (threadIdx.x == 0) {
    for (int s = 0; s < T::NSTAGE; ++s) {
      mbar_init(&full[s], TOKS ? 33 : 1);
      mbar_init(&empty[s], T::NW);
    }
    mbar_init(&qfull[0], 32);
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
  if (D == 128 && warp == 1) {
    // Before this warp's wait on the planner, the first tile of the CTA's first item (derived
    // from the lengths with the planner's rules) goes into L2, so that its copies (issued by
    // warp 0 once the planner has finished) read L2 rather than HBM.  Only a prefetch: the
    // work list itself is the planner's.  Head dim 128 only: at head dim 256 (32-token
    // tiles) the steps measured 2-3 us longer with it, at 128 up to 1 us shorter.
    const int4 f = first_item_of(p, blockIdx.x, gridDim.x, lane);
    if (f.z > f.y) {
      const int b = f.x / (p.Hkv * p.RB), g = (f.x / p.RB) % p.Hkv;
      const int box_rows = min(p.bs, T::TT), nbox = T::TT / box_rows;
      const int tokb = f.y + (lane / T::NSLAB) * box_rows;
      if (lane < nbox * T::NSLAB && tokb < f.z) {
        const int blk = __ldg(p.bt + (size_t)b * p.maxb + (tokb >> p.bs_shift));
        if (blk >= 0 && blk < p.nblocks) {
          const int x = (lane % T::NSLAB) * (T::ROWB / T::BPE), row = tokb & (p.bs - 1);
          tma_prefetch_l2_4d(&kmap, x, g, row, blk);
          tma_prefetch_l2_4d(&vmap, x, g, row, blk);
        }
      }
    }
  }
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
    prod.fill(T::NSTAGE - 1);
  }
  const bool tensor_scale = p.scale_mode == PA_SCALE_PER_TENSOR;
  const float kts = tensor_scale ? __ldg(p.k_scale) : 1.f;
  const float vts = tensor_scale ? __ldg(p.v_scale) : 1.f;
  const float qk_scale = p.qk_scale * kts;
  uint32_t tile_ctr = 0;
  int2 pend_even = make_int2(-1, 0), pend_odd = make_int2(-1, 0);  // held by thread 32

  // the next item and its sequence's lengths are read one item ahead
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
    // a piece of a split unit the decode merges: who finishes last is decided at the end
    const int2 uinfo = slot >= 0 ? __ldg(&p.unit_info[u]) : make_int2(0, 1);
    const bool in_dec = slot >= 0 && uinfo.y <= p.ns_dec;
    int cnt_seen = -1;

    // query fragments of this warp's rows (A operand, row-major 16 x 16 per k-step)
    uint32_t qa[WR][KSTEPS][4];
    int lim[WR][2];  // keys visible to rows quad and quad + 8 of each tile
#pragma unroll
    for (int w = 0; w < WR; ++w) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rl = (rblk * WR + w) * 16 + quad + 8 * h;  // row within the unit's tile
        const int rg = rb * MP + rl;
        const bool real = rg < p.M;
        const int i = rg / p.G, gq = rg % p.G;
        lim[w][h] = (real && i < ql) ? (p.causal ? n - ql + i + 1 : n) : 0;
        const char* qrow = reinterpret_cast<const char*>(p.q) +
                           ((((size_t)b * p.Sq + (real ? i : 0)) * p.Hq + (size_t)g * p.G + gq) * D) * 2;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
          uint32_t lo = 0, hi = 0;
          if (real) {
            if constexpr (T::FP8) {
              // permuted k order: dims 16kk + 4qi + {0,1} and + {2,3}
              const uint2 v = __ldg(reinterpret_cast<const uint2*>(qrow + (16 * kk + 4 * qi) * 2));
              lo = v.x;
              hi = v.y;
              if constexpr (QK == Q_BF16) {
                const float2 a = bf16x2_to_f2(lo), c = bf16x2_to_f2(hi);
                lo = pack2<true>(a.x, a.y);
                hi = pack2<true>(c.x, c.y);
              }
            } else {
              lo = __ldg(reinterpret_cast<const uint32_t*>(qrow + (16 * kk + 2 * qi) * 2));
              hi = __ldg(reinterpret_cast<const uint32_t*>(qrow + (16 * kk + 8 + 2 * qi) * 2));
            }
          }
          qa[w][kk][h] = lo;      // a0a1 (h = 0) / a2a3 (h = 1)
          qa[w][kk][2 + h] = hi;  // a4a5 / a6a7
        }
      }
    }

    float o[WR][NB][4];
    float m_run[WR][2], l_run[WR][2];
#pragma unroll
    for (int w = 0; w < WR; ++w) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) o[w][nb][0] = o[w][nb][1] = o[w][nb][2] = o[w][nb][3] = 0.f;
      m_run[w][0] = m_run[w][1] = -INFINITY;
      l_run[w][0] = l_run[w][1] = 0.f;
    }

    const int ntiles = ceil_div(t1 - t0, T::TT);
    int s_last = 0;
    for (int k = 0; k < ntiles; ++k) {
      if (warp == 0) prod.fill(tile_ctr + T::NSTAGE - 1);
      const int s = tile_ctr % T::NSTAGE;
      const uint32_t ph = (tile_ctr / T::NSTAGE) & 1;
      ++tile_ctr;
      s_last = s;
      if (!mbar_wait(&full[s], ph, abort_flag)) {
        atomicOr(p.flags, PA_FLAG_WAIT_TIMEOUT);
        *abort_flag = 1;
      }
      // with the item's last tile, look how many other pieces are published already
      if (in_dec && k + 1 == ntiles && threadIdx.x == 32) cnt_seen = ld_acquire_gpu(&p.unit_cnt[u]);
      char* st = smem + s * T::STAGE;
      const uint32_t kt = smem_addr(st), vt = smem_addr(st + T::KTILE);
      const float* sks = reinterpret_cast<const float*>(st + 2 * T::KTILE);
      const float* svs = sks + T::TT;
      const int tok0 = t0 + k * T::TT;
      const int n_in = min(T::TT, t1 - tok0);
      // chunks of this item go round-robin to the token streams
      const int first_q = ((ts - (k * T::CPT) % T::TS) + T::TS) % T::TS;
      for (int q = first_q; q < T::CPT; q += T::TS) {
        const int c0 = q * 16;  // first token of the chunk within the tile
        if (c0 >= n_in) break;
        const bool partial = c0 + 16 > n_in;
        if (partial) {
          // value rows past the last token may hold anything: make them zero so that
          // zero weights stay zero (keys there are masked out below)
          __syncwarp();
          for (int e = lane; e < 16 * (D * T::BPE / 16); e += 32) {
            const int r = c0 + e / (D * T::BPE / 16), cc = e % (D * T::BPE / 16);
            if (r >= n_in)
              *reinterpret_cast<uint4*>(st + T::KTILE + (cc >> 3) * T::SLAB + r * T::ROWB +
                                        (((cc & 7) ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        // ---- S = Q K^T for 16 tokens: two n-blocks of 8 tokens
        float sacc[WR][2][4];
#pragma unroll
        for (int w = 0; w < WR; ++w)
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) sacc[w][nb][0] = sacc[w][nb][1] = sacc[w][nb][2] = sacc[w][nb][3] = 0.f;
        if constexpr (!T::FP8) {
          // 16-bit cache: one ldmatrix.x4 per k-step = (tokens 0-7 | 8-15) x (k lo | hi)
          const int mat = lane >> 3;
          const int row = c0 + (lane & 7) + ((mat >> 1) << 3);
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            const int chunk = 2 * kk + (mat & 1);  // 16-byte chunk of the row
            uint32_t r0, r1, r2, r3;
            ldsm_x4(tile_chunk_addr<T>(kt, row, chunk >> 3, chunk & 7), r0, r1, r2, r3);
#pragma unroll
            for (int w = 0; w < WR; ++w) {
              mma16816<F16>(sacc[w][0], qa[w][kk], r0, r1);
              mma16816<F16>(sacc[w][1], qa[w][kk], r2, r3);
            }
          }
        } else {
          // fp8 cache: one ldmatrix.x4 = (tokens 0-7 | 8-15) x (two 16-dim k-steps)
          const int mat = lane >> 3;
          const int row = c0 + (lane & 7) + ((mat & 1) << 3);
#pragma unroll
          for (int kk2 = 0; kk2 < KSTEPS; kk2 += 2) {
            const int chunk = kk2 + (mat >> 1);
            uint32_t r[4];
            ldsm_x4(tile_chunk_addr<T>(kt, row, chunk >> 3, chunk & 7), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int j = 0; j < 2; ++j) {  // k-step kk2 + j: r[2j] tokens 0-7, r[2j+1] 8-15
#pragma unroll
              for (int nb = 0; nb < 2; ++nb) {
                const uint32_t w4 = r[2 * j + nb];
                const uint32_t b0 = e4m3x2_to_f16x2(w4), b1 = e4m3x2_to_f16x2(w4 >> 16);
#pragma unroll
                for (int w = 0; w < WR; ++w) mma16816<true>(sacc[w][nb], qa[w][kk2 + j], b0, b1);
              }
            }
          }
        }
        // ---- online softmax on the accumulators (rows quad, quad + 8; 4 tokens each)
        uint32_t pa[WR][4];
#pragma unroll
        for (int w = 0; w < WR; ++w) {
          float sv[2][4];  // [row half][token]: tokens 2qi, 2qi + 1, 8 + 2qi, 9 + 2qi
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int tt = (j >> 1) * 8 + 2 * qi + (j & 1);  // token within the chunk
              float x = sacc[w][j >> 1][2 * h + (j & 1)] * qk_scale;
              if constexpr (TOKS) x *= sks[c0 + tt];
              const bool vis = c0 + tt < n_in && tok0 + c0 + tt < lim[w][h];
              sv[h][j] = vis ? x : -INFINITY;
            }
          }
          float rmax[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float mx = fmaxf(fmaxf(sv[h][0], sv[h][1]), fmaxf(sv[h][2], sv[h][3]));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
            rmax[h] = mx;
          }
          const bool need0 = rmax[0] > m_run[w][0] + 8.f, need1 = rmax[1] > m_run[w][1] + 8.f;
          if (__any_sync(kFull, need0 || need1)) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const bool need = h ? need1 : need0;
              const float mn = need ? rmax[h] : m_run[w][h];
              const float alpha = (mn == m_run[w][h]) ? 1.f : fast_exp2(m_run[w][h] - mn);
              m_run[w][h] = mn;
              l_run[w][h] *= alpha;
#pragma unroll
              for (int nb = 0; nb < NB; ++nb) {
                o[w][nb][2 * h] *= alpha;
                o[w][nb][2 * h + 1] *= alpha;
              }
            }
          }
          float pr[2][4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const bool vis = sv[h][j] != -INFINITY;
              pr[h][j] = vis ? fast_exp2(sv[h][j] - m_run[w][h]) : 0.f;
              l_run[w][h] += pr[h][j];
              // a masked token's scale slot may be stale: only visible tokens are scaled
              if constexpr (TOKS) pr[h][j] = vis ? pr[h][j] * svs[c0 + (j >> 1) * 8 + 2 * qi + (j & 1)] : 0.f;
            }
          }
          pa[w][0] = pack2<F16>(pr[0][0], pr[0][1]);  // row quad,     tokens 2qi, 2qi+1
          pa[w][1] = pack2<F16>(pr[1][0], pr[1][1]);  // row quad + 8
          pa[w][2] = pack2<F16>(pr[0][2], pr[0][3]);  // row quad,     tokens 8+2qi, 9+2qi
          pa[w][3] = pack2<F16>(pr[1][2], pr[1][3]);  // row quad + 8
        }
        // ---- O += P V
        if constexpr (!T::FP8) {
          const int mat = lane >> 3;
          const int row = c0 + (lane & 7) + ((mat & 1) << 3);
#pragma unroll
          for (int nd = 0; nd < KSTEPS; ++nd) {
            const int chunk = 2 * nd + (mat >> 1);
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(tile_chunk_addr<T>(vt, row, chunk >> 3, chunk & 7), r0, r1, r2, r3);
#pragma unroll
            for (int w = 0; w < WR; ++w) {
              mma16816<F16>(o[w][2 * nd], pa[w], r0, r1);
              mma16816<F16>(o[w][2 * nd + 1], pa[w], r2, r3);
            }
          }
        } else {
          // fp8: a transposed 16-bit pair holds tokens (2qi, 2qi+1) of dims (2 quad, 2 quad+1)
          // -> n-block 2c carries even dims, 2c + 1 odd dims of the 16-dim chunk c
          const int mat = lane >> 3;
          const int row = c0 + (lane & 7) + ((mat & 1) << 3);
#pragma unroll
          for (int c2 = 0; c2 < KSTEPS; c2 += 2) {
            const int chunk = c2 + (mat >> 1);
            uint32_t r[4];
            ldsm_x4_t(tile_chunk_addr<T>(vt, row, chunk >> 3, chunk & 7), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int j = 0; j < 2; ++j) {  // chunk c2 + j: r[2j] tokens 0-7, r[2j+1] 8-15
              const uint32_t lo = r[2 * j], hi = r[2 * j + 1];
              const uint32_t ev0 = e4m3x2_to_f16x2(prmt(lo, 0, 0x0020)), od0 = e4m3x2_to_f16x2(prmt(lo, 0, 0x0031));
              const uint32_t ev1 = e4m3x2_to_f16x2(prmt(hi, 0, 0x0020)), od1 = e4m3x2_to_f16x2(prmt(hi, 0, 0x0031));
#pragma unroll
              for (int w = 0; w < WR; ++w) {
                mma16816<true>(o[w][2 * (c2 + j)], pa[w], ev0, ev1);
                mma16816<true>(o[w][2 * (c2 + j) + 1], pa[w], od0, od1);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0 && k + 1 < ntiles) mbar_arrive(&empty[s]);  // the last stage holds the merge
    }

    // ---- merge the token streams of each row block (tree through the last stage)
    float* obuf = reinterpret_cast<float*>(smem + s_last * T::STAGE);
    if (threadIdx.x == 32) *cnt_seen_s = cnt_seen;
    named_barrier_sync(1, T::NTHREADS);  // every warp is done reading the last stage
    // piece 0, when it ends last, combines the published pieces instead of publishing its own
    const bool fin = in_dec && slot == uinfo.x && *cnt_seen_s == uinfo.y - 1;
#pragma unroll
    for (int step = 1; step < T::TS; step <<= 1) {
      const bool writer = (ts & (2 * step - 1)) == step;
      const bool reader = (ts & (2 * step - 1)) == 0;
      const int mslot = rblk + T::RBW * (ts / (2 * step));
      float* so = obuf + mslot * (T::MERGE_SLOT_O / 4);
      float* sm = mlbuf + mslot * (WR * 4 * 32);
      if (writer) {
#pragma unroll
        for (int w = 0; w < WR; ++w) {
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int j = 0; j < 4; ++j) so[((w * NB + nb) * 4 + j) * 32 + lane] = o[w][nb][j];
          sm[(w * 4 + 0) * 32 + lane] = m_run[w][0];
          sm[(w * 4 + 1) * 32 + lane] = m_run[w][1];
          sm[(w * 4 + 2) * 32 + lane] = l_run[w][0];
          sm[(w * 4 + 3) * 32 + lane] = l_run[w][1];
        }
      }
      named_barrier_sync(1, T::NTHREADS);
      if (reader) {
        const int rslot = rblk + T::RBW * ((ts + step) / (2 * step));
        const float* ro = obuf + rslot * (T::MERGE_SLOT_O / 4);
        const float* rm = mlbuf + rslot * (WR * 4 * 32);
#pragma unroll
        for (int w = 0; w < WR; ++w) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float mo = rm[(w * 4 + h) * 32 + lane], lo = rm[(w * 4 + 2 + h) * 32 + lane];
            const float mn = fmaxf(m_run[w][h], mo);
            const float a = m_run[w][h] == -INFINITY ? 0.f : fast_exp2(m_run[w][h] - mn);
            const float bw = mo == -INFINITY ? 0.f : fast_exp2(mo - mn);
            m_run[w][h] = mn;
            l_run[w][h] = l_run[w][h] * a + lo * bw;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              o[w][nb][2 * h] = o[w][nb][2 * h] * a + ro[((w * NB + nb) * 4 + 2 * h) * 32 + lane] * bw;
              o[w][nb][2 * h + 1] =
                  o[w][nb][2 * h + 1] * a + ro[((w * NB + nb) * 4 + 2 * h + 1) * 32 + lane] * bw;
            }
          }
        }
      }
      named_barrier_sync(1, T::NTHREADS);
    }
    // ---- normalise and write (stream 0 of each row block holds the merged state)
    if (ts == 0) {
#pragma unroll
      for (int w = 0; w < WR; ++w) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float L = l_run[w][h];
          L += __shfl_xor_sync(kFull, L, 1);
          L += __shfl_xor_sync(kFull, L, 2);
          const float m = m_run[w][h];
          const int r = (rblk * WR + w) * 16 + quad + 8 * h;  // row within the unit's block
          const int rg = rb * MP + r;
          float inv = L > 0.f ? vts / L : 0.f;
          float lse2 = L > 0.f ? m + fast_log2(L) : -INFINITY;
          // output dims of accumulator entries (2h, 2h + 1) of n-block nb: d0(nb), + DSTEP
          constexpr int DSTEP = T::FP8 ? 2 : 1;
          auto d0_of = [&](int nb) {
            return T::FP8 ? (nb >> 1) * 16 + 4 * qi + (nb & 1) : nb * 8 + 2 * qi;
          };
          if (rg < p.M) {
            const int i = rg / p.G, hq = g * p.G + rg % p.G;
            const size_t orow = ((size_t)b * p.Sq + i) * p.Hq + hq;
            if (fin) {
              // this piece (0) merged with pieces 1 .. ns-1, in the arithmetic of merge_unit:
              // its normalised partial as it would be stored, then fma in piece order
              float mx = lse2;
              for (int sp = 1; sp < uinfo.y; ++sp)
                mx = fmaxf(mx, __ldcg(p.lse_part + (size_t)piece_slot(uinfo.x, sp) * MP + r));
              const float wown = lse2 == -INFINITY ? 0.f : fast_exp2(lse2 - mx);
              float W = 0.f + wown;
#pragma unroll
              for (int nb = 0; nb < NB; ++nb) {
                const float a0 = o[w][nb][2 * h] * inv, a1 = o[w][nb][2 * h + 1] * inv;
                o[w][nb][2 * h] = wown == 0.f ? 0.f : __fmaf_rn(wown, a0, 0.f);
                o[w][nb][2 * h + 1] = wown == 0.f ? 0.f : __fmaf_rn(wown, a1, 0.f);
              }
              for (int sp = 1; sp < uinfo.y; ++sp) {
                const size_t part = (size_t)piece_slot(uinfo.x, sp) * MP + r;
                const float ls = __ldcg(p.lse_part + part);
                const float ws = ls == -INFINITY ? 0.f : fast_exp2(ls - mx);
                W = W + ws;
                if (ws == 0.f) continue;
                const float* op = p.o_part + part * D;
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                  o[w][nb][2 * h] = __fmaf_rn(ws, __ldcg(op + d0_of(nb)), o[w][nb][2 * h]);
                  o[w][nb][2 * h + 1] =
                      __fmaf_rn(ws, __ldcg(op + d0_of(nb) + DSTEP), o[w][nb][2 * h + 1]);
                }
              }
              inv = W > 0.f ? 1.f / W : 0.f;
              lse2 = W > 0.f ? mx + fast_log2(W) : -INFINITY;
            }
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              const int d0 = d0_of(nb);
              const float v0 = o[w][nb][2 * h] * inv, v1 = o[w][nb][2 * h + 1] * inv;
              if (slot < 0 || fin) {
                store_out<QK>(p.out, orow * D + d0, v0);
                store_out<QK>(p.out, orow * D + d0 + DSTEP, v1);
              } else {
                p.o_part[((size_t)slot * MP + r) * D + d0] = v0;
                p.o_part[((size_t)slot * MP + r) * D + d0 + DSTEP] = v1;
              }
            }
            if (qi == 0) {
              if (slot < 0 || fin) {
                if (p.lse) p.lse[orow] = lse2 * kLn2;
              } else {
                p.lse_part[(size_t)slot * MP + r] = lse2;
              }
            }
          }
        }
      }
    }
    named_barrier_sync(1, T::NTHREADS);  // partials written (or the unit finished)
    if (in_dec && threadIdx.x == 32) {
      if (fin) {
        p.unit_cnt[u] = 0;  // every other piece is published: nobody counts this unit again
      } else {
        __threadfence();
        publish_piece(p, u, slot, &pend_even, &pend_odd);
      }
    }
    if (lane == 0) mbar_arrive(&empty[s_last]);
  }
  if (threadIdx.x == 32) {
    pend[0] = pend_even.x;
    pend[1] = pend_even.y;
    pend[2] = pend_odd.x;
    pend[3] = pend_odd.y;
  }
  if (warp == 0) prod.drain();
  named_barrier_sync(1, T::NTHREADS);  // no copy in flight: stage 0 is free for the merge
  finish_pending<D, MP, QK, T::NW>(p, pend, reinterpret_cast<float*>(smem), T::STAGE / 4, mlbuf);
  zero_empty_units<D, MP, QK, T::NTHREADS>(p);
}

template <int D, int MP, int KVK, int QK, bool TOKS>
cudaError_t launch_mma_instance(const KernelParams& prm, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, int grid, cudaStream_t s) {
  using T = MmaTraits<D, MP, KVK, TOKS>;
  auto kern = decode_mma_kernel<D, MP, KVK, QK, TOKS>;
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

#define PA_MMA_ROWS(X, MP_)      \
  X(MP_, KV_BF16, Q_BF16, false) \
  X(MP_, KV_FP16, Q_FP16, false) \
  X(MP_, KV_FP8, Q_BF16, false)  \
  X(MP_, KV_FP8, Q_BF16, true)   \
  X(MP_, KV_FP8, Q_FP16, false)  \
  X(MP_, KV_FP8, Q_FP16, true)
#define PA_MMA_ALL(X) PA_MMA_ROWS(X, 16) PA_MMA_ROWS(X, 32) PA_MMA_ROWS(X, 64)

// A cache row must hold whole 128-byte slabs (a 64-dim fp8 cache stays on CUDA cores).
constexpr bool mma_fits(int D, int kvk) { return D * (kvk == KV_FP8 ? 1 : 2) >= 128; }

template <int D>
cudaError_t launch_mma_for_dim(const KernelParams& prm, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, int grid, int mp, int kvk, int qk,
                               bool toks, cudaStream_t s) {
#define PA_MMA_CASE(MP_, KVK_, QK_, TOKS_)                                          \
  if constexpr (mma_fits(D, KVK_)) {                                                \
    if (mp == MP_ && kvk == KVK_ && qk == QK_ && toks == TOKS_)                     \
      return launch_mma_instance<D, MP_, KVK_, QK_, TOKS_>(prm, kmap, vmap, grid, s); \
  }
  PA_MMA_ALL(PA_MMA_CASE)
#undef PA_MMA_CASE
  return cudaErrorNotSupported;
}

template <int D>
int mma_ctas_per_sm_for_dim(int mp, int kvk, bool toks) {
#define PA_MMA_OCC(MP_, KVK_, QK_, TOKS_)                                            \
  if constexpr (mma_fits(D, KVK_)) {                                                 \
    if (mp == MP_ && kvk == KVK_ && toks == TOKS_) return MmaTraits<D, MP_, KVK_, TOKS_>::CTAS_PER_SM; \
  }
  PA_MMA_ALL(PA_MMA_OCC)
#undef PA_MMA_OCC
  return 1;
}

}  // namespace pa
