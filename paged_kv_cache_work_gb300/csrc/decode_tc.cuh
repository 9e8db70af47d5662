// Fifth-generation tensor-core decode (tcgen05, accumulators in tensor memory) for large
// query tiles: 33 to 128 query rows per kv head, head dim 128.
//
// The CTA is split into roles that talk only through mbarriers, so copies, conversions,
// MMAs and the softmax of different 64-token steps overlap:
//   warp 0      streams the items' K/V tiles through the TMA ring (TileProducer);
//   warp 1      one thread issues, per step g, S = Q K^T (M = 128, N = 64, K = 128) into
//               tensor-memory buffer g % 2, and then O += P V for step g - 1 (M = 128,
//               N = 128, K = 64, V read as an MN-major operand), so the next logits are being
//               computed while the softmax works on the current ones;
//   warps 2-5   one query row per thread: load the row's 64 logits with tcgen05.ld, online
//               softmax in registers (a row never leaves its thread), write the row of P into
//               a 128-byte-swizzled shared tile; at the end of an item load O from tensor
//               memory and write the output or the split partial (merge protocol of
//               decode_common.cuh);
//   warps 6-7   (fp8 caches) widen each step's 64 rows of K and V to f16 in shared memory,
//               two steps ahead, and release the ring stage once its rows are widened.
// The unit's query rows (Q, as 16-bit pairs: lane = row), the logits S (two buffers), the
// probabilities P (two buffers) and the output accumulator O all live in tensor memory, so
// shared memory carries only K and V.  The instances built are the 16-bit caches; the fp8
// roles are kept but not dispatched, because widening fp8 in shared memory measured slower
// than the mma.sync kernel's widening in registers.
#pragma once

#include "decode_common.cuh"

namespace pa {

template <int D_, int MP_, int KVK_, bool TOKS_>
struct TcTraits {
  static constexpr int D = D_;  // 128 or 256
  static constexpr int MP = MP_;  // query rows of a unit; the MMA always has M = 128
  static constexpr int KVK = KVK_;
  static constexpr bool TOKS = TOKS_;
  static constexpr bool FP8 = KVK == KV_FP8;
  static constexpr int BPE = FP8 ? 1 : 2;
  static constexpr int W_PROD = 0, W_MMA = 1, W_SOFT = 2, W_CONV = 6;
  static constexpr int NCW = FP8 ? 2 : 0;  // converter warps
  static constexpr int NW = 6 + NCW;
  static constexpr int NTHREADS = NW * 32;
  static constexpr int TT = kTileBytes / (D * BPE);  // tokens per stage: 64, or 128 for fp8
  static constexpr int SUB = FP8 ? 64 : TT;          // tokens per MMA step: 64, or 32 for D 256
  static constexpr int NSUB = TT / SUB;
  static constexpr int NSTAGE = FP8 ? 3 : 6;
  static constexpr int NQ = 1;
  static constexpr int QSLOT = 0;
  static constexpr bool WITH_Q = false;
  static constexpr int ROWB = 128;             // swizzled slabs of 128 bytes per row
  static constexpr int NSLAB = D * BPE / 128;  // slabs of a cache tile row
  static constexpr int KTILE = TT * D * BPE;
  static constexpr int STAGE = round_up(2 * KTILE + (TOKS ? 2 * TT * 4 : 0), 1024);
  static constexpr int OFF_Q = 0;                       // (query rows live in tensor memory)
  static constexpr int OFF_CV = NSTAGE * STAGE;         // fp8: 64 tokens of K, then V, as f16
  static constexpr int CV_SLAB = SUB * 128;             // one 64-dim slab of 64 converted rows
  static constexpr int CV_BUF = 2 * 2 * CV_SLAB;        // K and V of one step
  static constexpr int CV_BYTES = FP8 ? 2 * CV_BUF : 0;  // two steps
  static constexpr int KSLAB = FP8 ? CV_SLAB : TT * 128;  // slab stride of the K and V operands
  static constexpr int OFF_SC = OFF_CV + CV_BYTES;        // per-token scales of two steps
  static constexpr int SC_BYTES = TOKS ? 2 * 2 * SUB * 4 : 0;
  static constexpr int OFF_ML = OFF_SC + SC_BYTES;
  static constexpr int ML_BYTES = round_up(2 * MP * 4, 128);
  static constexpr int OFF_BAR = round_up(OFF_ML + ML_BYTES, 64);
  // full, empty, (unused query slot), s_full x2, s_free x2, p_full x2, pv_done x2, o_free,
  // q_full, cv_full x2, cv_free x2, mma_end, sc_full x2
  static constexpr int NBAR = 2 * NSTAGE + NQ + 18;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + kFlagBytes + 16 + 1024;
  static constexpr int CTAS_PER_SM = 1;
  // Tensor memory (lane = query row, 32-bit columns): two S buffers of SUB fp32 columns, O
  // (D fp32 columns), Q (D / 2 columns of 16-bit pairs) and two P buffers (SUB / 2 columns).
  // Head dim 128: S [0, 128), O [128, 256), Q [256, 320), P [320, 384).  Head dim 256
  // (32-token steps): S [0, 64), Q [64, 192), P [192, 224), O [256, 512).
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = D == 256 ? 256 : 2 * SUB;
  static constexpr uint32_t COL_Q = D == 256 ? 2 * SUB : COL_O + D;
  static constexpr uint32_t COL_P = COL_Q + D / 2;
  static_assert(COL_P + SUB <= TMEM_COLS && (D != 256 || COL_P + SUB <= COL_O), "tensor memory");
  static_assert(MP == 64 || MP == 128, "row tile");
  static_assert(D == 128 || D == 256, "head dim");
  static_assert(SUB == 32 || SUB == 64, "step");
  static_assert(TT % SUB == 0, "tile");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// ---- tcgen05 wrappers ------------------------------------------------------------------
// Shared-memory matrix descriptor: 128-byte swizzle, start address, leading and stride byte
// offsets (all in 16-byte units), descriptor version 1 of the sm_100 family.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::f16 with fp32 accumulation: operand type (0 f16, 1 bf16),
// A K-major, B K-major or MN-major, N / 8 and M / 16.
__host__ __device__ constexpr uint32_t umma_idesc(int m, int n, bool bf16, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}
// The same with the A operand in tensor memory (lane = row, a 32-bit column = two K elements).
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
// A row of P (N packed 16-bit pairs) into tensor memory.
template <int N>
__device__ __forceinline__ void tmem_st_p(uint32_t taddr, const uint32_t (&v)[N]) {
  if constexpr (N == 32)
    tmem_st32u(taddr, v);
  else
    tmem_st16u(taddr, v);
}

// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 32 lanes x 32 bits x 32 columns per warp: thread t of warp w gets columns [col, col + 32)
// of tensor-memory lane 32 w + t.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Byte offset of 16-byte chunk c of row r in a tile of 128-byte swizzled rows.
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c) {
  return (uint32_t)r * 128u + ((uint32_t)((c ^ r) & 7) << 4);
}
// Two 16-bit values of the MMA operand type.
template <bool BF>
__device__ __forceinline__ uint32_t pack16x2(float a, float b) {
  if constexpr (BF) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t w) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// One 64-token step g of an item: first token of its tile, offset in the tile, tokens of the
// item in it, and whether it is the last step of its tile.
struct TcStep {
  int tok0, c0, n;
  bool last;
};
__device__ __forceinline__ TcStep tc_step(int t0, int t1, int j, int tt, int nsub, int sub) {
  TcStep q;
  const int k = j / nsub;
  q.c0 = (j % nsub) * sub;
  q.tok0 = t0 + k * tt;
  const int n_in = min(tt, t1 - q.tok0);
  q.n = min(sub, n_in - q.c0);
  q.last = q.c0 + sub >= n_in;
  return q;
}

// 32 lanes x 32 bits x 64 columns: thread t of warp w gets columns [col, col + 64) of lane
// 32 (w % 4) + t, with one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,"
      "%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,"
      "%59,%60,%61,%62,%63}, [%64];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int j = 0; j < 64; ++j) v[j] = __uint_as_float(r[j]);
}

template <int D_, int MP, int KVK, int QK, bool TOKS>
__global__ void __launch_bounds__(TcTraits<D_, MP, KVK, TOKS>::NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const KernelParams p) {
  using T = TcTraits<D_, MP, KVK, TOKS>;
  constexpr int SUB = T::SUB;
  constexpr int D = T::D;
  constexpr bool BF = !T::FP8 && KVK == KV_BF16;  // MMA operands bf16 (else f16)
  constexpr uint32_t ID_S = umma_idesc(128, T::SUB, BF, false);
  constexpr uint32_t ID_PV = umma_idesc(128, D, BF, true);
  constexpr int SOFT_BAR = 2;  // named barrier of the four softmax warps
  extern __shared__ char smem_raw[];
  char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty = full + T::NSTAGE;
  uint64_t* qfull = empty + T::NSTAGE;
  uint64_t* s_full = qfull + T::NQ;  // [2]
  uint64_t* s_free = s_full + 2;     // [2]
  uint64_t* p_full = s_free + 2;     // [2]: one per P buffer
  uint64_t* pv_done = p_full + 2;    // [2]: the PV that read P buffer b has completed
  uint64_t* o_free = pv_done + 2;
  uint64_t* q_full = o_free + 1;
  uint64_t* cv_full = q_full + 1;  // [2]
  uint64_t* cv_free = cv_full + 2;  // [2]
  uint64_t* mma_end = cv_free + 2;
  uint64_t* sc_full = mma_end + 1;  // [2]: per-token scales of a step staged (fp8)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sc_full + 2);
  volatile int* pend = abort_flag + 2;        // [4]: split pieces published, see finish_pending
  volatile int* cnt_seen_s = abort_flag + 6;  // published pieces of the item's unit, seen late
  uint32_t* tslot = reinterpret_cast<uint32_t*>(const_cast<int*>(abort_flag + 7));
  float* mlbuf = reinterpret_cast<float*>(smem + T::OFF_ML);
  char* scv = smem + T::OFF_CV;
  float* ssc = reinterpret_cast<float*>(smem + T::OFF_SC);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < T::NSTAGE; ++s) {
      mbar_init(&full[s], TOKS ? 33 : 1);
      mbar_init(&empty[s], T::FP8 ? T::NCW : 1);  // converter warps, or the MMA commit
    }
    mbar_init(&qfull[0], 32);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 4);
      mbar_init(&cv_full[b], T::FP8 ? T::NCW : 1);
      mbar_init(&cv_free[b], 1);
      mbar_init(&sc_full[b], T::FP8 ? T::NCW : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&p_full[b], 4);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(o_free, 4);
    mbar_init(q_full, 4);
    mbar_init(mma_end, 1);
    *abort_flag = 0;
    pend[0] = -1;
    pend[2] = -1;
    fence_barrier_init();
  }
  if (warp == T::W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tslot)),
                 "r"(T::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == T::W_PROD && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t t_s = tmem, t_o = tmem + T::COL_O, t_q = tmem + T::COL_Q, t_p = tmem + T::COL_P;
  grid_dependency_wait();  // the work list comes from the planner launched just before
  // the next kernel may start launching now: it is held in its own grid_dependency_wait
  // until this grid has completed, and it cannot take the place of a CTA of this grid
  grid_dependents_launch();

  const int it_begin = p.item_off[blockIdx.x], it_end = p.item_off[blockIdx.x + 1];
  auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
    if (!mbar_wait(bar, parity, abort_flag)) {
      atomicOr(p.flags, PA_FLAG_WAIT_TIMEOUT);
      *abort_flag = 1;
    }
  };

  if (warp == T::W_PROD) {
    // ================================================================ TMA producer
    TileProducer<T> prod;
    prod.init(&p, &kmap, &vmap, smem, full, empty, qfull, abort_flag, lane, it_begin, it_end);
    prod.fill(0xFFFFFFFFu);  // every tile of the work list, as stages come free
    prod.drain();
  } else if (warp == T::W_MMA) {
    // ================================================================ MMA issue
    if (lane == 0) {
      uint32_t g = 0, tile_ctr = 0, items_done = 0;
      uint32_t q_ph = 0, o_ph = 0, pf_ph[2] = {0, 0}, sfree_ph[2] = {0, 0}, cvf_ph[2] = {0, 0};
      // O += P V of step gp (P of that step, in buffer gp % 2, must be written)
      auto issue_pv = [&](uint32_t gp, uint32_t vaddr, bool first, int stage, bool last) {
        wait_bar(&p_full[gp & 1], pf_ph[gp & 1]);
        pf_ph[gp & 1] ^= 1u;
        if (first && items_done > 0) {  // the previous item's epilogue has read O
          wait_bar(o_free, o_ph);
          o_ph ^= 1u;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < T::SUB / 16; ++kk) {
          const uint64_t bd = umma_desc(vaddr + kk * 2048, T::KSLAB, 1024);
          umma_f16_ta(t_o, t_p + (gp & 1) * (T::SUB / 2) + kk * 8, bd, ID_PV, !(first && kk == 0));
        }
        umma_commit(&pv_done[gp & 1]);
        if constexpr (T::FP8) {
          umma_commit(&cv_free[gp & 1]);
        } else {
          if (last) umma_commit(&empty[stage]);  // the stage's K and V are read
        }
      };
      for (int it = it_begin; it < it_end; ++it) {
        const int4 item = p.items[it];
        const int t0 = item.y, t1 = item.z;
        if (t1 <= t0) continue;
        const int nsub = ceil_div(t1 - t0, T::SUB);
        wait_bar(q_full, q_ph);  // the item's query tile is in shared memory
        q_ph ^= 1u;
        uint32_t pv_vaddr = 0, pv_g = 0;
        int pv_stage = 0;
        bool pv_last = false;
        int stage = 0;
        for (int j = 0; j < nsub; ++j, ++g) {
          const TcStep q = tc_step(t0, t1, j, T::TT, T::NSUB, T::SUB);
          if (q.c0 == 0) {
            stage = tile_ctr % T::NSTAGE;
            if constexpr (!T::FP8) wait_bar(&full[stage], (tile_ctr / T::NSTAGE) & 1);
            ++tile_ctr;
          }
          uint32_t kbase, vaddr;
          if constexpr (T::FP8) {
            wait_bar(&cv_full[g & 1], cvf_ph[g & 1]);
            cvf_ph[g & 1] ^= 1u;
            kbase = smem_addr(scv + (g & 1) * T::CV_BUF);
            vaddr = kbase + 2 * T::CV_SLAB;
          } else {
            kbase = smem_addr(smem + stage * T::STAGE) + q.c0 * 128;
            vaddr = smem_addr(smem + stage * T::STAGE + T::KTILE) + q.c0 * 128;
          }
          if (g >= 2) {  // the softmax has loaded the logits of step g - 2 from this buffer
            wait_bar(&s_free[g & 1], sfree_ph[g & 1]);
            sfree_ph[g & 1] ^= 1u;
          }
          tc_fence_after();
          const uint32_t t_sg = t_s + (g & 1) * T::SUB;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t bd = umma_desc(kbase + (kk >> 2) * T::KSLAB + (kk & 3) * 32, 16, 1024);
            umma_f16_ta(t_sg, t_q + kk * 8, bd, ID_S, kk > 0);
          }
          umma_commit(&s_full[g & 1]);
          if (j > 0) issue_pv(pv_g, pv_vaddr, j == 1, pv_stage, pv_last);
          pv_g = g;
          pv_vaddr = vaddr;
          pv_stage = stage;
          pv_last = q.last;
        }
        issue_pv(pv_g, pv_vaddr, nsub == 1, pv_stage, pv_last);
        ++items_done;
      }
      umma_commit(mma_end);
      if (!mbar_wait_drain(mma_end, 0)) atomicOr(p.flags, PA_FLAG_WAIT_TIMEOUT);
    }
  } else if (warp < T::W_CONV) {
    // ================================================================ softmax and epilogue
    const int stid = tid - T::W_SOFT * 32;            // 0 .. 127 over the four warps
    const int r = 32 * (warp & 3) + lane;            // query row = this thread's TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const bool tensor_scale = p.scale_mode == PA_SCALE_PER_TENSOR;
    const float kts = tensor_scale ? __ldg(p.k_scale) : 1.f;
    const float vts = tensor_scale ? __ldg(p.v_scale) : 1.f;
    const float qk_scale = p.qk_scale * kts;
    uint32_t g = 0, sfull_ph[2] = {0, 0}, sc_ph[2] = {0, 0};
    uint32_t pv_seen[2] = {0, 0};  // completions of pv_done[b] consumed so far
    // wait until the PV of step x (which read P buffer x % 2) has completed; each buffer's
    // completions are consumed in order, and none is ever two ahead of its consumer
    auto wait_pv_step = [&](uint32_t x) {
      const uint32_t bx = x & 1, ux = x >> 1;
      while (pv_seen[bx] <= ux) {
        wait_bar(&pv_done[bx], pv_seen[bx] & 1);
        ++pv_seen[bx];
      }
      tc_fence_after();
    };
    uint32_t tile_base = 0;  // tiles of the earlier items (ring position of this item's first)
    int2 pend_even = make_int2(-1, 0), pend_odd = make_int2(-1, 0);  // held by stid 0
    int4 item_next = it_begin < it_end ? p.items[it_begin] : make_int4(0, 0, 0, -1);
    for (int it = it_begin; it < it_end; ++it) {
      const int4 item = item_next;
      if (it + 1 < it_end) item_next = p.items[it + 1];
      const int u = item.x, t0 = item.y, t1 = item.z, slot = item.w;
      if (t1 <= t0) continue;
      const int b = u / (p.Hkv * p.RB), g_kv = (u / p.RB) % p.Hkv, rb = u % p.RB;
      const int n = __ldg(p.ctx + b), ql = __ldg(p.qlens + b);
      const int2 uinfo = slot >= 0 ? __ldg(&p.unit_info[u]) : make_int2(0, 1);
      const bool in_dec = slot >= 0 && uinfo.y <= p.ns_dec;
      const int nsub = ceil_div(t1 - t0, T::SUB);
      int cnt_seen = -1;
      const int rg = rb * MP + r;
      const bool real = r < MP && rg < p.M;
      const int qi = real ? rg / p.G : 0, hq = g_kv * p.G + (real ? rg % p.G : 0);
      const int lim = (real && qi < ql) ? (p.causal ? n - ql + qi + 1 : n) : 0;
      // ---- this thread's query row into tensor memory, 16-bit pairs (every MMA of the
      // previous item has completed); rows of no query are zero
      {
        const uint4* qrow = reinterpret_cast<const uint4*>(
            reinterpret_cast<const char*>(p.q) + ((((size_t)b * p.Sq + qi) * p.Hq + hq) * D) * 2);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 v = real ? __ldg(qrow + 8 * h + c) : make_uint4(0, 0, 0, 0);
            if constexpr (T::FP8 && QK == Q_BF16) {  // f16 operands for an fp8 cache
              uint32_t t4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int jw = 0; jw < 4; ++jw) {
                const float2 f = bf16x2_to_f2(t4[jw]);
                t4[jw] = pack16x2<false>(f.x, f.y);
              }
              v = make_uint4(t4[0], t4[1], t4[2], t4[3]);
            }
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
          }
          tmem_st32u(t_q + lane_off + 32 * h, w);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);

      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nsub; ++j, ++g) {
        const TcStep q = tc_step(t0, t1, j, T::TT, T::NSUB, T::SUB);
        if (in_dec && j + 1 == nsub && stid == 0) cnt_seen = ld_acquire_gpu(&p.unit_cnt[u]);
        if (!T::FP8 && q.n < T::SUB) {
          // the zeroing below writes into the ring stage: the tile must have landed (the
          // MMA warp has waited for it; this wait is for the ordering of the writes)
          const uint32_t tc = tile_base + (uint32_t)(j / T::NSUB);
          wait_bar(&full[tc % T::NSTAGE], (tc / T::NSTAGE) & 1);
        }
        wait_bar(&s_full[g & 1], sfull_ph[g & 1]);
        sfull_ph[g & 1] ^= 1u;
        tc_fence_after();
        float x[SUB];
        if constexpr (SUB == 64)
          tmem_ld64(t_s + (g & 1) * SUB + lane_off, x);
        else
          tmem_ld32(t_s + (g & 1) * SUB + lane_off, x);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[g & 1]);
        const float* ksc = nullptr;
        const float* vsc = nullptr;
        if constexpr (TOKS) {
          wait_bar(&sc_full[g & 1], sc_ph[g & 1]);
          sc_ph[g & 1] ^= 1u;
          ksc = ssc + (g & 1) * 2 * T::SUB;
          vsc = ksc + T::SUB;
        }
        // ---- online softmax of this thread's row (log2 units), two logits per instruction
        const float2 s2 = make_float2(qk_scale, qk_scale), z2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < SUB / 2; ++i) {
          float2 y = ffma2(make_float2(x[2 * i], x[2 * i + 1]), s2, z2);
          if constexpr (TOKS) y = ffma2(y, make_float2(ksc[2 * i], ksc[2 * i + 1]), z2);
          x[2 * i] = y.x;
          x[2 * i + 1] = y.y;
        }
        // masked keys (past the item's tokens or past the row's causal limit) become -inf;
        // most steps have none
        if (q.n < T::SUB || q.tok0 + q.c0 + T::SUB > lim) {
#pragma unroll
          for (int jj = 0; jj < SUB; ++jj)
            if (jj >= q.n || q.tok0 + q.c0 + jj >= lim) x[jj] = -INFINITY;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < SUB; jj += 2) mx = fmaxf(mx, fmaxf(x[jj], x[jj + 1]));
        const bool need = mx > m_run + 8.f;  // lazy rescale: only when the max grows by 2^8
        const bool rescale = __any_sync(kFull, need);
        const float mn = need ? mx : m_run;
        const float alpha = (mn == m_run || m_run == -INFINITY) ? 1.f : fast_exp2(m_run - mn);
        m_run = mn;
        // this thread's row of P, packed: 64 tokens = eight 16-byte chunks; a masked logit
        // (-inf) gives exp2 = 0, and a row with no visible key so far has only zeros
        float lsum = 0.f;
        uint32_t pk[SUB / 2];
        if (m_run == -INFINITY) {
#pragma unroll
          for (int i = 0; i < SUB / 2; ++i) pk[i] = 0u;
        } else {
          const float2 nm = make_float2(-m_run, -m_run), one2 = make_float2(1.f, 1.f);
          float2 ls2 = z2;
#pragma unroll
          for (int i = 0; i < SUB / 2; ++i) {
            const float2 t = ffma2(make_float2(x[2 * i], x[2 * i + 1]), one2, nm);
            float p0 = fast_exp2(t.x), p1 = fast_exp2(t.y);
            ls2 = ffma2(make_float2(p0, p1), one2, ls2);
            if constexpr (TOKS) {  // a masked token's scale slot may be stale
              p0 = p0 > 0.f ? p0 * vsc[2 * i] : 0.f;
              p1 = p1 > 0.f ? p1 * vsc[2 * i + 1] : 0.f;
            }
            pk[i] = pack16x2<BF>(p0, p1);
          }
          lsum = ls2.x + ls2.y;
        }
        l_run = l_run * alpha + lsum;
        if (rescale && j > 0) {
          // O holds earlier tokens of this item: scale this warp's rows once every PV into
          // O has completed
          wait_pv_step(g - 1);
#pragma unroll
          for (int h = 0; h < D / 32; ++h) {
            float o[32];
            tmem_ld32(t_o + lane_off + 32 * h, o);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) o[jj] *= alpha;
            tmem_st32(t_o + lane_off + 32 * h, o);
          }
          tmem_wait_st();
        }
        if (g >= 2) wait_pv_step(g - 2);  // P buffer g % 2 was last read by the PV of step g - 2
        tmem_st_p<SUB / 2>(t_p + (g & 1) * (SUB / 2) + lane_off, pk);
        tmem_wait_st();
        if constexpr (!T::FP8) {
          if (q.n < T::SUB) {
            // value rows past the item's tokens may hold anything: zero them (before this
            // step's PV reads them) so that zero weights stay zero
            const int stage = (int)(tile_base + (uint32_t)(j / T::NSUB)) % T::NSTAGE;
            char* vt = smem + stage * T::STAGE + T::KTILE;
            for (int e = stid; e < (T::SUB - q.n) * T::NSLAB * 8; e += 128) {
              const int rr = q.n + e / (T::NSLAB * 8), sl = (e / 8) % T::NSLAB, c = e & 7;
              *reinterpret_cast<uint4*>(vt + sl * (T::TT * 128) + sw128_chunk(q.c0 + rr, c)) =
                  make_uint4(0, 0, 0, 0);
            }
          }
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[g & 1]);
      }
      tile_base += (uint32_t)ceil_div(t1 - t0, T::TT);

      // ---- epilogue: O of this thread's row from tensor memory, in two halves of 64 dims
      if (g >= 2) wait_pv_step(g - 2);  // the item's last two PVs (in order)
      wait_pv_step(g - 1);
      if (stid == 0) *cnt_seen_s = cnt_seen;
      named_barrier_sync(SOFT_BAR, 128);
      const bool fin = in_dec && slot == uinfo.x && *cnt_seen_s == uinfo.y - 1;
      const size_t orow = ((size_t)b * p.Sq + qi) * p.Hq + hq;
      float inv = l_run > 0.f ? vts / l_run : 0.f;
      float lse2 = l_run > 0.f ? m_run + fast_log2(l_run) : -INFINITY;
      // piece 0 finishing the unit: merged with pieces 1 .. ns-1 in the arithmetic of merge_unit
      float mx = lse2, wown = 0.f, W = 0.f;
      if (fin && real) {
        for (int sp2 = 1; sp2 < uinfo.y; ++sp2)
          mx = fmaxf(mx, __ldcg(p.lse_part + (size_t)piece_slot(uinfo.x, sp2) * MP + r));
        wown = lse2 == -INFINITY ? 0.f : fast_exp2(lse2 - mx);
        W = 0.f + wown;
      }
      const bool to_out = slot < 0 || fin;
#pragma unroll 1
      for (int h = 0; h < D / 64; ++h) {
        float o[64];
        tmem_ld64(t_o + lane_off + 64 * h, o);
        if (h == D / 64 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_free);  // the next item's first PV may overwrite O
        }
        if (!real) continue;
        float oinv = inv;
        if (fin) {
#pragma unroll
          for (int d = 0; d < 64; ++d) o[d] = wown == 0.f ? 0.f : __fmaf_rn(wown, o[d] * inv, 0.f);
          float Wh = 0.f + wown;
          for (int sp2 = 1; sp2 < uinfo.y; ++sp2) {
            const size_t part = (size_t)piece_slot(uinfo.x, sp2) * MP + r;
            const float ls = __ldcg(p.lse_part + part);
            const float ws = ls == -INFINITY ? 0.f : fast_exp2(ls - mx);
            Wh = Wh + ws;
            if (ws == 0.f) continue;
            const float4* op = reinterpret_cast<const float4*>(p.o_part + part * D + 64 * h);
#pragma unroll
            for (int d4 = 0; d4 < 16; ++d4) {
              const float4 w4 = __ldcg(op + d4);
              o[4 * d4] = __fmaf_rn(ws, w4.x, o[4 * d4]);
              o[4 * d4 + 1] = __fmaf_rn(ws, w4.y, o[4 * d4 + 1]);
              o[4 * d4 + 2] = __fmaf_rn(ws, w4.z, o[4 * d4 + 2]);
              o[4 * d4 + 3] = __fmaf_rn(ws, w4.w, o[4 * d4 + 3]);
            }
          }
          W = Wh;
          oinv = W > 0.f ? 1.f / W : 0.f;
        }
        if (to_out) {
#pragma unroll
          for (int d = 0; d < 64; d += 4)
            store_out4<QK>(p.out, orow * D + 64 * h + d,
                           make_float4(o[d] * oinv, o[d + 1] * oinv, o[d + 2] * oinv, o[d + 3] * oinv));
        } else {
          float4* op = reinterpret_cast<float4*>(p.o_part + ((size_t)slot * MP + r) * D + 64 * h);
#pragma unroll
          for (int d = 0; d < 64; d += 4)
            op[d / 4] = make_float4(o[d] * oinv, o[d + 1] * oinv, o[d + 2] * oinv, o[d + 3] * oinv);
        }
      }
      if (real) {
        if (fin) lse2 = W > 0.f ? mx + fast_log2(W) : -INFINITY;
        if (to_out) {
          if (p.lse) p.lse[orow] = lse2 * kLn2;
        } else {
          p.lse_part[(size_t)slot * MP + r] = lse2;
        }
      }
      named_barrier_sync(SOFT_BAR, 128);  // partials written (or the unit finished)
      if (in_dec && stid == 0) {
        if (fin) {
          p.unit_cnt[u] = 0;  // every other piece is published: nobody counts this unit again
        } else {
          __threadfence();
          publish_piece(p, u, slot, &pend_even, &pend_odd);
        }
      }
    }
    if (stid == 0) {
      pend[0] = pend_even.x;
      pend[1] = pend_even.y;
      pend[2] = pend_odd.x;
      pend[3] = pend_odd.y;
    }
  } else {
    // ================================================================ fp8 widening
    if constexpr (T::FP8) {
      const int ctid = tid - T::W_CONV * 32;  // 0 .. 63
      uint32_t g = 0, tile_ctr = 0, cvfree_ph[2] = {0, 0};
      int stage = 0;
      for (int it = it_begin; it < it_end; ++it) {
        const int4 item = p.items[it];
        const int t0 = item.y, t1 = item.z;
        if (t1 <= t0) continue;
        const int nsub = ceil_div(t1 - t0, T::SUB);
        for (int j = 0; j < nsub; ++j, ++g) {
          const TcStep q = tc_step(t0, t1, j, T::TT, T::NSUB, T::SUB);
          if (q.c0 == 0) {
            stage = tile_ctr % T::NSTAGE;
            wait_bar(&full[stage], (tile_ctr / T::NSTAGE) & 1);
            ++tile_ctr;
          }
          if (g >= 2) {  // the PV of step g - 2 has read this buffer
            wait_bar(&cv_free[g & 1], cvfree_ph[g & 1]);
            cvfree_ph[g & 1] ^= 1u;
          }
          const char* st = smem + stage * T::STAGE;
          char* cv = scv + (g & 1) * T::CV_BUF;
          for (int e = ctid; e < 2 * T::SUB * 8; e += 32 * T::NCW) {
            const int kv = e / (T::SUB * 8), rr = (e / 8) % T::SUB, c = e & 7;
            uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
            if (rr < q.n) {  // rows past the item's tokens become zero
              const uint4 w = *reinterpret_cast<const uint4*>(st + kv * T::KTILE + sw128_chunk(q.c0 + rr, c));
              lo = make_uint4(e4m3x2_to_h2(w.x), e4m3x2_to_h2(w.x >> 16), e4m3x2_to_h2(w.y),
                              e4m3x2_to_h2(w.y >> 16));
              hi = make_uint4(e4m3x2_to_h2(w.z), e4m3x2_to_h2(w.z >> 16), e4m3x2_to_h2(w.w),
                              e4m3x2_to_h2(w.w >> 16));
            }
            // dims 16c .. 16c + 15 -> 16-bit slab c / 4, chunks 2 (c % 4) and 2 (c % 4) + 1
            char* dst = cv + kv * (2 * T::CV_SLAB) + (c >> 2) * T::CV_SLAB;
            *reinterpret_cast<uint4*>(dst + sw128_chunk(rr, 2 * (c & 3))) = lo;
            *reinterpret_cast<uint4*>(dst + sw128_chunk(rr, 2 * (c & 3) + 1)) = hi;
          }
          if constexpr (TOKS) {  // the scales leave the stage with the rows
            const float* sks = reinterpret_cast<const float*>(st + 2 * T::KTILE);
            float* sc = ssc + (g & 1) * 2 * T::SUB;
            sc[ctid] = sks[q.c0 + ctid];
            sc[T::SUB + ctid] = sks[T::TT + q.c0 + ctid];
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&cv_full[g & 1]);
            if constexpr (TOKS) mbar_arrive(&sc_full[g & 1]);
            if (q.last) mbar_arrive(&empty[stage]);  // this warp is done with the stage
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();  // every role is done: no copy or MMA in flight
  if (warp >= T::W_SOFT && warp < T::W_CONV) {
    const int stid = tid - T::W_SOFT * 32;
    finish_pending<D, MP, QK, 4>(p, pend, reinterpret_cast<float*>(smem), T::STAGE / 4, mlbuf, stid);
    zero_empty_units<D, MP, QK, 128>(p, stid);
  }
  __syncthreads();
  if (warp == T::W_MMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(T::TMEM_COLS));
  }
}

template <int D, int MP, int KVK, int QK, bool TOKS>
cudaError_t launch_tc_instance(const KernelParams& prm, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, int grid, cudaStream_t s) {
  using T = TcTraits<D, MP, KVK, TOKS>;
  auto kern = decode_tc_kernel<D, MP, KVK, QK, TOKS>;
  static bool attr_set = false;  // benign race: every caller sets the same value
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
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

}  // namespace pa
