// Fifth-generation tensor-core decode (tcgen05, accumulators in tensor memory) for large
// query tiles: 33 to 128 query rows per kv head, 16-bit caches of head dim 128 or 256 and
// fp8 caches of head dim 128 with per-tensor or no scales.
//
// A step is a tile of 64 tokens.  The CTA is split into roles that talk only through
// mbarriers, so copies, MMAs and the softmax of different steps overlap:
//   warp 0      streams the items' K and V tiles through two TMA rings (TcProducer) of
//               96 KB each: a K slot is released by the S that read it and a V slot by its
//               PV, and K is copied one step ahead of V;
//   warp 1      one thread issues, per step g, S = Q K^T (M = 128, N = 64, K = head dim)
//               into tensor-memory buffer g % NSP, and then O += P V for step g - LAG
//               (M = 128, N = head dim, K = 64, V read as an MN-major operand), so the
//               in-order tensor pipe holds the next logits ahead of any PV that waits for
//               the softmax;
//   warps 2-5   one query row per thread: load the row's logits with tcgen05.ld, online
//               softmax in registers (a row never leaves its thread), write the row of P as
//               16-bit pairs over the first half of the same logits buffer; at the end of an
//               item load O from tensor memory and write the output or the split partial
//               (merge protocol of decode_common.cuh);
//   warps 6-9   (fp8 caches) widen each step's e4m3 K rows to f16 in one of three
//               shared-memory buffers, released by the step's S, and its V rows in one of
//               four, released by its PV (one warp per SM sub-partition: with fewer, the
//               conversion rate, not the copy, bounds the kernel).
// Buffer g % NSP holds S(g) and then P(g) until the PV of step g has read it, so the MMA
// thread waits for that PV before it writes S(g + NSP) there: NSP = 4 at head dim 128 and
// 2 at head dim 256, as many as tensor memory holds next to O and the query rows (Q, as
// 16-bit pairs: lane = row).  Shared memory carries only K and V (and, for fp8, their f16
// widening).
//
// A tcgen05.mma of K = 16 occupies the tensor pipe about equally long at every N up to
// 256, so these N = 64 logits use a quarter of its peak: at head dim 256 (16 S MMAs and 4
// PV MMAs per 64 KB of cache) the pipe keeps up with HBM, at head dim 128 it is close to
// being the limit.
#pragma once

#include "decode_common.cuh"

namespace pa {

template <int D_, int MP_, int KVK_, bool TOKS_>
struct TcTraits {
  static constexpr int D = D_;    // 128 or 256
  static constexpr int MP = MP_;  // query rows of a unit; the MMA always has M = 128
  static constexpr int KVK = KVK_;
  static constexpr bool TOKS = TOKS_;
  static constexpr bool FP8 = KVK == KV_FP8;
  static constexpr int BPE = FP8 ? 1 : 2;
  static constexpr int W_PROD = 0, W_MMA = 1, W_SOFT = 2, W_CONV = 6;
  static constexpr int NCW = FP8 ? 4 : 0;  // warps that widen fp8 tiles to f16
  static constexpr int NW = 6 + NCW;
  static constexpr int NTHREADS = NW * 32;
  static constexpr int TT = kTcStepTokens;  // tokens per tile and per MMA step: 64
  static constexpr int SUB = TT;
  static constexpr int KTILE = TT * D * BPE;  // 16 KB, 32 KB at head dim 256, 8 KB for fp8
  static constexpr int SLOT = KTILE;  // a ring slot
  static constexpr int NSTAGE = FP8 ? 5 : 98304 / KTILE;  // slots of each ring: 6, 3 or 5
  static constexpr int ROWB = 128;             // swizzled slabs of 128 bytes per row
  static constexpr int NSLAB = D * BPE / 128;  // slabs of a cache tile row
  // S/P buffers in tensor memory: four at head dim 128 (S(g) waits only for the PV of
  // step g - 4), two at 256
  static constexpr int NSP = D == 128 ? 4 : 2;
  static constexpr int OFF_K = 0;                      // K ring: NSTAGE slots
  static constexpr int OFF_V = OFF_K + NSTAGE * SLOT;  // V ring: NSTAGE slots
  // fp8: the widened (f16) K rows of NCK steps and V rows of NCV steps, each a
  // 128-byte-swizzled operand of two 64-dim slabs (a K buffer is released by its S, a V
  // buffer by its PV)
  static constexpr int NCK = FP8 ? 3 : 0;
  static constexpr int NCV = FP8 ? 4 : 0;
  static constexpr int CV_SLAB = SUB * 128;
  static constexpr int CV_BUF = 2 * CV_SLAB;
  static constexpr int OFF_CV = OFF_V + NSTAGE * SLOT;  // K buffers, then V buffers
  static constexpr int SCRATCH = OFF_CV;  // bytes free for the merges at the end (the rings)
  static constexpr int LAG = NSP - 1;  // steps a PV trails its S
  static constexpr int KSLAB = FP8 ? CV_SLAB : TT * 128;  // slab stride of the MMA operands
  static constexpr int OFF_ML = OFF_CV + (NCK + NCV) * CV_BUF;
  static constexpr int ML_BYTES = round_up(2 * MP * 4, 128);
  static constexpr int OFF_BAR = round_up(OFF_ML + ML_BYTES, 64);
  // full_k, empty_k, full_v, empty_v (NSTAGE each), s_full, p_full, pv_done (NSP each),
  // o_free, q_full, mma_end, full and free of the K buffers and of the V buffers
  static constexpr int NBAR = 4 * NSTAGE + 3 * NSP + 3 + 2 * (NCK + NCV);
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + kFlagBytes + 16 + 1024;
  static constexpr int CTAS_PER_SM = 1;
  // Tensor memory (lane = query row, 32-bit columns): NSP S/P buffers of SUB fp32 columns
  // (P, SUB / 2 columns of 16-bit pairs, overwrites the first half of its own S), O (D fp32
  // columns) and Q (D / 2 columns of 16-bit pairs).  Head dim 128: S/P [0, 256), O
  // [256, 384), Q [384, 448).  Head dim 256: S/P [0, 128), Q [128, 256), O [256, 512).
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = D == 256 ? 256 : NSP * SUB;
  static constexpr uint32_t COL_Q = D == 256 ? NSP * SUB : COL_O + D;
  static_assert(NSP * SUB + D + D / 2 <= (int)TMEM_COLS, "tensor memory");
  static_assert(!TOKS, "per-token scales stay on the mma.sync kernel");
  static_assert(!FP8 || D == 128, "fp8 caches at head dim 128");
  static_assert(!FP8 || (SUB * 8) % (32 * NCW) == 0, "widening: whole passes");
  // the V rows of step g wait for the PV of step g - NCV, issued after the S of step
  // g - NCV + LAG, which waits for the K rows of that step: the widening, K(g) then V(g),
  // must not need K rows past g
  static_assert(LAG < NSP && (!FP8 || LAG <= NCV), "no cycle between the roles");
  static_assert(MP == 64 || MP == 128, "row tile");
  static_assert(D == 128 || D == 256, "head dim");
  static_assert(SUB == 64, "step");
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
// Two E4M3 codes (low byte first) to an f16 pair (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t w) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
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

// The TMA side of the tcgen05 kernel, run by warp 0 (all lanes, same state).  Tile n of the
// CTA's work list goes to slot n % NSTAGE of the K ring and of the V ring; lane
// page * NSLAB + slab copies one 128-byte column slab of one page of the tile.  The order of
// the copies is K(0), K(1), V(0), K(2), V(1), ...: a copy waits until the tile NSTAGE
// earlier has been read from its slot (by its S for K and its PV for V, or, for fp8, by the
// widening warps).
template <class T>
struct TcProducer {
  struct Box {
    int blk, row, g;
    bool ok;
    uint32_t nvalid;
  };
  const KernelParams* p;
  const CUtensorMap* kmap;
  const CUtensorMap* vmap;
  char* smem;
  uint64_t *full_k, *empty_k, *full_v, *empty_v;
  volatile int* abort_flag;
  int lane, it, it_end, k, ntiles, t0, t1, b, g, box_rows, nbox, blk_next;
  uint32_t box_bytes, nk, nv;
  bool have, next_ready;
  int4 item_next;

  __device__ __forceinline__ int block_of(int bb, int tt0, int tt1, int kk) const {
    const int tokb = tt0 + kk * T::TT + (lane / T::NSLAB) * box_rows;
    return (lane < nbox * T::NSLAB && tokb < tt1)
               ? __ldg(p->bt + (size_t)bb * p->maxb + (tokb >> p->bs_shift))
               : -1;
  }

  __device__ __forceinline__ void init(const KernelParams* prm, const CUtensorMap* km,
                                       const CUtensorMap* vm, char* sm, uint64_t* fk,
                                       uint64_t* ek, uint64_t* fv, uint64_t* ev,
                                       volatile int* ab, int ln, int ib, int ie) {
    p = prm; kmap = km; vmap = vm; smem = sm; full_k = fk; empty_k = ek; full_v = fv;
    empty_v = ev; abort_flag = ab; lane = ln; it = ib - 1; it_end = ie; k = 0; ntiles = 0;
    box_rows = min(p->bs, T::TT);
    nbox = T::TT / box_rows;
    box_bytes = (uint32_t)box_rows * T::ROWB;
    nk = nv = 0;
    have = next_ready = false;
    blk_next = -1;
    item_next = ib < ie ? p->items[ib] : make_int4(0, 0, 0, -1);
  }

  // This lane's box of the next tile of the list; false when the list is exhausted.  The
  // block id of the tile after it is loaded here too, to land during the waits.
  __device__ __forceinline__ bool next_tile(Box& bx) {
    while (!have) {
      if (++it >= it_end) return false;
      const int4 item = item_next;
      if (it + 1 < it_end) item_next = p->items[it + 1];
      t0 = item.y;
      t1 = item.z;
      if (t1 <= t0) continue;
      b = item.x / (p->Hkv * p->RB);
      g = (item.x / p->RB) % p->Hkv;
      k = 0;
      ntiles = ceil_div(t1 - t0, T::TT);
      if (!next_ready) blk_next = block_of(b, t0, t1, 0);
      next_ready = false;
      have = true;
    }
    const int tokb = t0 + k * T::TT + (lane / T::NSLAB) * box_rows;
    const bool want = lane < nbox * T::NSLAB && tokb < t1;
    bx.blk = blk_next;
    bx.ok = want && blk_next >= 0 && blk_next < p->nblocks;
    if (want && !bx.ok) atomicOr(p->flags, PA_FLAG_BAD_BLOCK_ID);
    bx.nvalid = __popc(__ballot_sync(kFull, bx.ok));
    bx.row = tokb & (p->bs - 1);
    bx.g = g;
    if (k + 1 < ntiles) {
      blk_next = block_of(b, t0, t1, k + 1);
    } else if (it + 1 < it_end && item_next.z > item_next.y) {
      blk_next = block_of(item_next.x / (p->Hkv * p->RB), item_next.y, item_next.z, 0);
      next_ready = true;
    }
    if (++k >= ntiles) have = false;
    return true;
  }

  // Copy a tile's boxes into slot n % NSTAGE of one ring once the slot is released.
  __device__ __forceinline__ bool issue(const Box& bx, uint32_t n, uint64_t* full,
                                        uint64_t* empty, const CUtensorMap* map, int ring) {
    const int s = (int)(n % T::NSTAGE);
    if (!mbar_wait(&empty[s], ((n / T::NSTAGE) & 1) ^ 1, abort_flag)) {
      atomicOr(p->flags, PA_FLAG_WAIT_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
    if (lane == 0) mbar_arrive_expect_tx(&full[s], bx.nvalid * box_bytes);
    __syncwarp();
    char* slot = smem + ring + s * T::SLOT;
    if (bx.ok) {
      // slab h of page j lands at h * (TT rows) + j * (box rows), in units of ROWB bytes
      const int page = lane / T::NSLAB, slab = lane % T::NSLAB;
      const uint32_t dst = (uint32_t)(slab * T::TT + page * box_rows) * T::ROWB;
      tma_load_4d(slot + dst, map, &full[s], slab * (T::ROWB / T::BPE), bx.g, bx.row, bx.blk);
    }
    return true;
  }

  __device__ __forceinline__ void run() {
    Box cur, nxt;
    if (!next_tile(cur)) return;
    if (!issue(cur, nk, full_k, empty_k, kmap, T::OFF_K)) return;
    ++nk;
    while (true) {
      const bool more = next_tile(nxt);
      if (more) {
        if (!issue(nxt, nk, full_k, empty_k, kmap, T::OFF_K)) return;
        ++nk;
      }
      if (!issue(cur, nv, full_v, empty_v, vmap, T::OFF_V)) return;
      ++nv;
      if (!more) return;
      cur = nxt;
    }
  }

  // Let every copy this warp started land before the CTA may exit.
  __device__ __forceinline__ void drain() {
    for (uint32_t j = nk > (uint32_t)T::NSTAGE ? nk - T::NSTAGE : 0; j < nk; ++j)
      mbar_wait_drain(&full_k[j % T::NSTAGE], (j / T::NSTAGE) & 1);
    for (uint32_t j = nv > (uint32_t)T::NSTAGE ? nv - T::NSTAGE : 0; j < nv; ++j)
      mbar_wait_drain(&full_v[j % T::NSTAGE], (j / T::NSTAGE) & 1);
  }
};

template <int D_, int MP, int KVK, int QK, bool TOKS>
__global__ void __launch_bounds__(TcTraits<D_, MP, KVK, TOKS>::NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const KernelParams p) {
  using T = TcTraits<D_, MP, KVK, TOKS>;
  constexpr int SUB = T::SUB;
  constexpr int D = T::D;
  constexpr bool BF = KVK == KV_BF16;  // MMA operands bf16 (else f16: f16 and fp8 caches)
  constexpr uint32_t ID_S = umma_idesc(128, SUB, BF, false);
  constexpr uint32_t ID_PV = umma_idesc(128, D, BF, true);
  constexpr int SOFT_BAR = 2;  // named barrier of the four softmax warps
  extern __shared__ char smem_raw[];
  char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t* full_k = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty_k = full_k + T::NSTAGE;
  uint64_t* full_v = empty_k + T::NSTAGE;
  uint64_t* empty_v = full_v + T::NSTAGE;
  uint64_t* s_full = empty_v + T::NSTAGE;  // [NSP]
  uint64_t* p_full = s_full + T::NSP;      // [NSP]: P of the step in buffer b is written
  uint64_t* pv_done = p_full + T::NSP;     // [NSP]: the PV that read buffer b has completed
  uint64_t* o_free = pv_done + T::NSP;
  uint64_t* q_full = o_free + 1;
  uint64_t* mma_end = q_full + 1;
  uint64_t* ck_full = mma_end + 1;       // [NCK]: widened K rows of the step in buffer b
  uint64_t* ck_free = ck_full + T::NCK;  // [NCK]: the S that read buffer b has completed
  uint64_t* cv_full = ck_free + T::NCK;  // [NCV]: widened V rows of the step in buffer b
  uint64_t* cv_free = cv_full + T::NCV;  // [NCV]: the PV that read buffer b has completed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(cv_free + T::NCV);
  volatile int* pend = abort_flag + 2;        // [4]: split pieces published, see finish_pending
  volatile int* cnt_seen_s = abort_flag + 6;  // published pieces of the item's unit, seen late
  uint32_t* tslot = reinterpret_cast<uint32_t*>(const_cast<int*>(abort_flag + 7));
  float* mlbuf = reinterpret_cast<float*>(smem + T::OFF_ML);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < T::NSTAGE; ++s) {
      mbar_init(&full_k[s], 1);  // the expect_tx arrival of the copy
      mbar_init(&full_v[s], 1);
      // readers: the commit of the S (K) or PV (V) that read the slot, or the fp8 widening
      mbar_init(&empty_k[s], T::FP8 ? T::NCW : 1);
      mbar_init(&empty_v[s], T::FP8 ? T::NCW : 1);
    }
    for (int b = 0; b < T::NCK; ++b) {
      mbar_init(&ck_full[b], T::NCW);
      mbar_init(&ck_free[b], 1);
    }
    for (int b = 0; b < T::NCV; ++b) {
      mbar_init(&cv_full[b], T::NCW);
      mbar_init(&cv_free[b], 1);
    }
    for (int b = 0; b < T::NSP; ++b) {
      mbar_init(&s_full[b], 1);
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
  const uint32_t t_s = tmem, t_o = tmem + T::COL_O, t_q = tmem + T::COL_Q;
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
    TcProducer<T> prod;
    prod.init(&p, &kmap, &vmap, smem, full_k, empty_k, full_v, empty_v, abort_flag, lane,
              it_begin, it_end);
    prod.run();  // every tile of the work list, as slots come free
    prod.drain();
  } else if (warp == T::W_MMA) {
    // ================================================================ MMA issue
    if (lane == 0) {
      uint32_t g = 0, items_done = 0;
      uint32_t q_ph = 0, o_ph = 0;
      // step x uses buffer x % NSP; every barrier of a buffer completes once per use, in
      // step order, so the phase of step x is (x / NSP) & 1
      // O += P V of step gp (its P, in buffer gp % NSP, must be written); the commit releases
      // the V slot (fp8: the V buffer)
      auto issue_pv = [&](uint32_t gp, bool first) {
        const int slot = (int)(gp % T::NSTAGE);
        uint32_t vaddr;
        if constexpr (T::FP8) {
          wait_bar(&cv_full[gp % T::NCV], (gp / T::NCV) & 1);
          vaddr = smem_addr(smem + T::OFF_CV + (T::NCK + gp % T::NCV) * T::CV_BUF);
        } else {
          vaddr = smem_addr(smem + T::OFF_V + slot * T::SLOT);
          wait_bar(&full_v[slot], (gp / T::NSTAGE) & 1);
        }
        wait_bar(&p_full[gp % T::NSP], (gp / T::NSP) & 1);
        if (first && items_done > 0) {  // the previous item's epilogue has read O
          wait_bar(o_free, o_ph);
          o_ph ^= 1u;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < SUB / 16; ++kk) {
          const uint64_t bd = umma_desc(vaddr + kk * 2048, T::KSLAB, 1024);
          umma_f16_ta(t_o, t_s + (gp % T::NSP) * SUB + kk * 8, bd, ID_PV, !(first && kk == 0));
        }
        umma_commit(&pv_done[gp % T::NSP]);
        if constexpr (T::FP8)
          umma_commit(&cv_free[gp % T::NCV]);
        else
          umma_commit(&empty_v[slot]);
      };
      for (int it = it_begin; it < it_end; ++it) {
        const int4 item = p.items[it];
        const int t0 = item.y, t1 = item.z;
        if (t1 <= t0) continue;
        const int nsub = ceil_div(t1 - t0, SUB);
        wait_bar(q_full, q_ph);  // the item's query rows are in tensor memory
        q_ph ^= 1u;
        // the PVs trail the S MMAs by LAG steps, so the in-order tensor pipe always holds
        // the logits of the next steps ahead of a PV that waits for the softmax (LAG < NSP:
        // S(g) waits for the PV of step g - NSP, issued before it)
        constexpr int LAG = T::LAG;
        const uint32_t g_item = g;  // the item's first step
        for (int j = 0; j < nsub; ++j, ++g) {
          const int slot = (int)(g % T::NSTAGE);
          uint32_t kbase;
          if constexpr (T::FP8) {
            wait_bar(&ck_full[g % T::NCK], (g / T::NCK) & 1);
            kbase = smem_addr(smem + T::OFF_CV + (g % T::NCK) * T::CV_BUF);
          } else {
            wait_bar(&full_k[slot], (g / T::NSTAGE) & 1);
            kbase = smem_addr(smem + T::OFF_K + slot * T::SLOT);
          }
          if (g >= (uint32_t)T::NSP) {  // the buffer holds P(g - NSP) until its PV has read it
            const uint32_t x = g - T::NSP;
            wait_bar(&pv_done[x % T::NSP], (x / T::NSP) & 1);
          }
          tc_fence_after();
          const uint32_t t_sg = t_s + (g % T::NSP) * SUB;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t bd = umma_desc(kbase + (kk >> 2) * T::KSLAB + (kk & 3) * 32, 16, 1024);
            umma_f16_ta(t_sg, t_q + kk * 8, bd, ID_S, kk > 0);
          }
          umma_commit(&s_full[g % T::NSP]);
          if constexpr (T::FP8)
            umma_commit(&ck_free[g % T::NCK]);
          else
            umma_commit(&empty_k[slot]);
          if (j >= LAG) issue_pv(g - LAG, j == LAG);
        }
        for (int j = nsub > LAG ? nsub - LAG : 0; j < nsub; ++j) issue_pv(g_item + j, j == 0);
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
    uint32_t g = 0;
    uint32_t pv_next = 0;  // the first step whose PV completion is not consumed yet
    // wait until the PV of step x (which read buffer x % NSP) has completed; completions
    // are consumed in step order, and none is ever two ahead of its consumer on a buffer
    auto wait_pv_step = [&](uint32_t x) {
      for (; pv_next <= x; ++pv_next)
        wait_bar(&pv_done[pv_next % T::NSP], (pv_next / T::NSP) & 1);
      tc_fence_after();
    };
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
      const int nsub = ceil_div(t1 - t0, SUB);
      int cnt_seen = -1;
      const int rg = rb * MP + r;
      const bool real = r < MP && rg < p.M;
      const int qi = real ? rg / p.G : 0, hq = g_kv * p.G + (real ? rg % p.G : 0);
      const int lim = (real && qi < ql) ? (p.causal ? n - ql + qi + 1 : n) : 0;
      // a warp whose 32 rows hold no query (the upper half of a 64-row tile) skips the
      // softmax; its rows of P and O are never read, and it keeps only the waits and
      // arrivals that keep the barriers' phases in step
      const bool warp_dead = __all_sync(kFull, !real);
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
        const int tok0 = t0 + j * SUB, nv = min(SUB, t1 - tok0);  // tokens of the item here
        if (in_dec && j + 1 == nsub && stid == 0) cnt_seen = ld_acquire_gpu(&p.unit_cnt[u]);
        if (!T::FP8 && nv < SUB) {
          // the zeroing below writes into the V slot: the tile must have landed (this wait
          // orders the writes after the copy)
          wait_bar(&full_v[g % T::NSTAGE], (g / T::NSTAGE) & 1);
        }
        wait_bar(&s_full[g % T::NSP], (g / T::NSP) & 1);
        tc_fence_after();
        if (g >= (uint32_t)T::NSP) wait_pv_step(g - T::NSP);  // (complete: S(g) came after it)
        if (!warp_dead) {
          const uint32_t t_sg = t_s + (g % T::NSP) * SUB + lane_off;
          float x[SUB];
          tmem_ld64(t_sg, x);
          // ---- online softmax of this thread's row (log2 units), two logits per instruction
          const float2 s2 = make_float2(qk_scale, qk_scale), z2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < SUB / 2; ++i) {
            const float2 y = ffma2(make_float2(x[2 * i], x[2 * i + 1]), s2, z2);
            x[2 * i] = y.x;
            x[2 * i + 1] = y.y;
          }
          // masked keys (past the item's tokens or past the row's causal limit) become -inf;
          // most steps have none
          if (nv < SUB || tok0 + SUB > lim) {
#pragma unroll
            for (int jj = 0; jj < SUB; ++jj)
              if (jj >= nv || tok0 + jj >= lim) x[jj] = -INFINITY;
          }
          float mx = -INFINITY;
#pragma unroll
          for (int jj = 0; jj < SUB; jj += 2) mx = fmaxf(mx, fmaxf(x[jj], x[jj + 1]));
          const bool need = mx > m_run + 8.f;  // lazy rescale: only when the max grows by 2^8
          const bool rescale = __any_sync(kFull, need);
          const float mn = need ? mx : m_run;
          const float alpha = (mn == m_run || m_run == -INFINITY) ? 1.f : fast_exp2(m_run - mn);
          m_run = mn;
          // this thread's row of P, 16-bit pairs over the first SUB / 2 columns of its own
          // logits (all of them are in registers); a masked logit (-inf) gives exp2 = 0, and a
          // row with no visible key so far has only zeros
          float lsum = 0.f;
          {
            const float2 nm = make_float2(m_run == -INFINITY ? 0.f : -m_run,
                                          m_run == -INFINITY ? 0.f : -m_run);
            const float2 one2 = make_float2(1.f, 1.f);
            float2 ls2 = z2;
#pragma unroll
            for (int h = 0; h < SUB / 32; ++h) {  // 32 tokens = 16 columns at a time
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float2 t = ffma2(make_float2(x[32 * h + 2 * i], x[32 * h + 2 * i + 1]), one2, nm);
                const float p0 = fast_exp2(t.x), p1 = fast_exp2(t.y);
                ls2 = ffma2(make_float2(p0, p1), one2, ls2);
                pk[i] = pack16x2<BF>(p0, p1);
              }
              tmem_st16u(t_sg + 16 * h, pk);
            }
            lsum = ls2.x + ls2.y;
          }
          l_run = l_run * alpha + lsum;
          if (rescale && j > 0) {
            // O holds earlier tokens of this item: scale this warp's rows once every PV into
            // O has completed (the PV of this step waits for p_full below)
            wait_pv_step(g - 1);
#pragma unroll 1
            for (int h = 0; h < D / 32; ++h) {
              float o[32];
              tmem_ld32(t_o + lane_off + 32 * h, o);
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) o[jj] *= alpha;
              tmem_st32(t_o + lane_off + 32 * h, o);
            }
          }
        }  // !warp_dead
        tmem_wait_st();
        if (!T::FP8 && nv < SUB) {
          // value rows past the item's tokens may hold anything: zero them (before this
          // step's PV reads them) so that zero weights stay zero
          char* vt = smem + T::OFF_V + (g % T::NSTAGE) * T::SLOT;
          for (int e = stid; e < (SUB - nv) * T::NSLAB * 8; e += 128) {
            const int rr = nv + e / (T::NSLAB * 8), sl = (e / 8) % T::NSLAB, c = e & 7;
            *reinterpret_cast<uint4*>(vt + sl * T::KSLAB + sw128_chunk(rr, c)) =
                make_uint4(0, 0, 0, 0);
          }
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[g % T::NSP]);
      }
      // ---- epilogue: O of this thread's row from tensor memory, in two halves of 64 dims
      wait_pv_step(g - 1);  // every PV of the item (in order)
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
      // step g: the e4m3 K rows of ring slot g % NSTAGE become the f16 rows of K buffer
      // g % NCK, then its V rows those of V buffer g % NCV (rows past the item's tokens
      // become zero); the per-tensor scales are applied to the logits and the output
      const int ctid = tid - T::W_CONV * 32;  // 0 .. 32 NCW - 1
      // one operand: 64 rows of 128 e4m3 codes -> two slabs of 64 rows of 64 f16 values
      auto widen = [&](const char* src, char* dst, int nv) {
#pragma unroll
        for (int k = 0; k < SUB * 8 / (32 * T::NCW); ++k) {
          const int e = ctid + k * 32 * T::NCW;
          const int rr = e / 8, c = e & 7;
          uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
          if (rr < nv) {
            const uint4 w = *reinterpret_cast<const uint4*>(src + sw128_chunk(rr, c));
            lo = make_uint4(e4m3x2_to_h2(w.x), e4m3x2_to_h2(w.x >> 16), e4m3x2_to_h2(w.y),
                            e4m3x2_to_h2(w.y >> 16));
            hi = make_uint4(e4m3x2_to_h2(w.z), e4m3x2_to_h2(w.z >> 16), e4m3x2_to_h2(w.w),
                            e4m3x2_to_h2(w.w >> 16));
          }
          // dims 16c .. 16c + 15 -> f16 slab c / 4, chunks 2 (c % 4) and 2 (c % 4) + 1
          char* d = dst + (c >> 2) * T::CV_SLAB;
          *reinterpret_cast<uint4*>(d + sw128_chunk(rr, 2 * (c & 3))) = lo;
          *reinterpret_cast<uint4*>(d + sw128_chunk(rr, 2 * (c & 3) + 1)) = hi;
        }
        fence_async_smem();
        __syncwarp();
      };
      uint32_t g = 0;
      for (int it = it_begin; it < it_end; ++it) {
        const int4 item = p.items[it];
        const int t0 = item.y, t1 = item.z;
        if (t1 <= t0) continue;
        const int nsub = ceil_div(t1 - t0, SUB);
        for (int j = 0; j < nsub; ++j, ++g) {
          const int nv = min(SUB, t1 - (t0 + j * SUB));
          const int slot = (int)(g % T::NSTAGE);
          const uint32_t ph = (g / T::NSTAGE) & 1;
          // ---- K rows
          wait_bar(&full_k[slot], ph);
          if (g >= (uint32_t)T::NCK) {  // the S of step g - NCK has read this buffer
            const uint32_t x = g - T::NCK;
            wait_bar(&ck_free[x % T::NCK], (x / T::NCK) & 1);
          }
          widen(smem + T::OFF_K + slot * T::SLOT,
                smem + T::OFF_CV + (g % T::NCK) * T::CV_BUF, nv);
          if (lane == 0) {
            mbar_arrive(&ck_full[g % T::NCK]);
            mbar_arrive(&empty_k[slot]);  // this warp is done with the K slot
          }
          // ---- V rows
          wait_bar(&full_v[slot], ph);
          if (g >= (uint32_t)T::NCV) {  // the PV of step g - NCV has read this buffer
            const uint32_t x = g - T::NCV;
            wait_bar(&cv_free[x % T::NCV], (x / T::NCV) & 1);
          }
          widen(smem + T::OFF_V + slot * T::SLOT,
                smem + T::OFF_CV + (T::NCK + g % T::NCV) * T::CV_BUF, nv);
          if (lane == 0) {
            mbar_arrive(&cv_full[g % T::NCV]);
            mbar_arrive(&empty_v[slot]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();  // every role is done: no copy or MMA in flight
  if (warp >= T::W_SOFT && warp < T::W_CONV) {
    const int stid = tid - T::W_SOFT * 32;
    finish_pending<D, MP, QK, 4>(p, pend, reinterpret_cast<float*>(smem), T::SCRATCH / 4, mlbuf, stid);
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
