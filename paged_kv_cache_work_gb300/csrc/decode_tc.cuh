// Fifth-generation tensor-core decode (tcgen05, accumulators in tensor memory) for large
// query tiles: 33 to 128 query rows per kv head, 16-bit caches of head dim 128 or 256 and
// fp8 caches of head dim 128 with per-tensor, per-token or no scales.
//
// A step is a tile of 64 tokens.  The CTA is split into roles that talk only through
// mbarriers, so copies, MMAs and the softmax of different steps overlap:
//   warp 0      streams the items' K and V tiles through two TMA rings (TcProducer), K one
//               step ahead of V, and, for per-token fp8 scales, each step's 64 K and 64 V
//               scales into a small shared-memory ring of their own;
//   warp 1      one thread issues, per step g, S = Q K^T (M = 128, N = 64, K = head dim)
//               into tensor-memory buffer g % NSP, and then O += P V for step g - LAG
//               (M = 128, N = head dim, K = 64, V read as an MN-major operand); for an fp8
//               cache S is of kind f8f6f4 on the K codes as they landed, against the query
//               row held as two E4M3 terms (hi + lo, exact for a bf16 query but for elements
//               below about a thousandth of the row's largest);
//   warps 2-5   the softmax: tensor-memory lane L is owned by one thread, which loads its
//               logits with tcgen05.ld, runs the online softmax in registers and writes its
//               row of P as 16-bit pairs over the first half of the same logits buffer; at
//               the end of an item it loads O and writes the output or the split partial
//               (merge protocol of decode_common.cuh);
//   warps 6-9   (fp8 caches) widen each step's e4m3 V rows to f16 operands in shared memory
//               (one warp per SM sub-partition).
//
// Issue cost.  The tensor pipe takes about 48 SM clocks for an N = 64 logits MMA and 64 for
// an N = 128 one when they are issued back to back, but each tcgen05.commit costs it about
// 90 clocks more, and a wait for an MMA's completion right after issuing it drains the pipe
// (measured on GB300 with standalone issue probes).  So every buffer is indexed by the step
// modulo NSP, the number of S/P buffers, wherever shared memory allows: the commit that
// tells the softmax its logits are ready also frees the step's K slot, and the commit that
// ends a PV also frees its V slot (or widened V buffer): two commits per step.  And
// the PV of step g trails its S by LAG = NSP - 2 steps where NSP >= 4, so the S that reuses
// a buffer waits for a PV issued a step earlier, with MMAs still queued behind it.
//
// Query tiles of 64 rows (head dim 128) run as two token streams: rows 64-127 of the MMA
// repeat rows 0-63 (the query rows are loaded twice), the thread of lane r < 64 takes the
// first 32 tokens of every step and the thread of lane r + 64 the last 32, each with its own
// running max and sum (the other half of its row of P is zero), so the softmax runs on all
// four SM sub-partitions with half the exponentials per thread.  At the end of an item the
// two streams of a row are merged with the log-sum-exp rule through shared memory.
#pragma once

#include "decode_common.cuh"

namespace pa {

template <int D_, int MP_, int KVK_, bool TOKS_>
struct TcTraits {
  static constexpr int D = D_;    // 128 or 256
  static constexpr int MP = MP_;  // query rows of a unit; the MMA always has M = 128
  static constexpr int KVK = KVK_;
  static constexpr bool TOKS = TOKS_;  // per-token fp8 scales
  static constexpr bool FP8 = KVK == KV_FP8;
  static constexpr int BPE = FP8 ? 1 : 2;
  static constexpr int W_PROD = 0, W_MMA = 1, W_SOFT = 2, W_CONV = 6;
  static constexpr int NCW = FP8 ? 4 : 0;  // warps that widen fp8 tiles to f16
  static constexpr int NW = 6 + NCW;
  static constexpr int NTHREADS = NW * 32;
  static constexpr int TT = kTcStepTokens;  // tokens per tile and per MMA step: 64
  static constexpr int SUB = TT;
  // two token streams per query row (64-row tiles of head dim 128)
  static constexpr bool DUAL = MP == 64 && D == 128;
  static constexpr int NL = DUAL ? SUB / 2 : SUB;  // logits of a step per softmax thread
  // S/P buffers in tensor memory and how many steps a PV trails its S
  static constexpr int NSP = D == 256 ? 2 : (FP8 ? 4 : 5);
  static constexpr int LAG = NSP >= 4 ? NSP - 2 : NSP - 1;
  static constexpr int KTILE = TT * D * BPE;  // 16 KB, 32 KB at head dim 256, 8 KB for fp8
  static constexpr int SLOT = KTILE;          // a ring slot
  // Slots of each TMA ring.  16-bit caches of head dim 128: NSP, so that slot g % NSP is
  // released by the commit of the S (K) or the PV (V) of step g that the softmax and the MMA
  // thread wait for anyway.  Head dim 256: three slots (two S/P buffers fit in tensor
  // memory, two slots would leave too little in flight), released by commits of their own.
  // fp8: the logits MMA reads the K codes in their ring slot (NSP slots, released by the S's
  // commit); the V codes are widened out of a ring of their own, released by the widening
  // warps.
  static constexpr int NK = D == 256 && !FP8 ? 3 : NSP;    // K ring slots
  static constexpr int NV = FP8 ? 5 : (D == 256 ? 3 : NSP);  // V ring slots
  static constexpr bool K_BY_S = NK == NSP;            // a K slot is released by its S's commit
  // steps the copy warp issues K ahead of V: for fp8 the V slots wait for the widening, which
  // waits for the PV of four steps back, and K copies held behind them left the logits MMA
  // waiting for its codes (per-tensor fp8 Sq = 4: 76.6 -> 76.0 us).  With per-token scales,
  // which go out with K, the longer lead measured slower.
  static constexpr int KLEAD = FP8 && !TOKS ? 2 : 1;
  static constexpr bool V_BY_PV = !FP8 && NV == NSP;  // a V slot is released by its PV's commit
  static constexpr int ROWB = 128;             // swizzled slabs of 128 bytes per row
  static constexpr int NSLAB = D * BPE / 128;  // slabs of a cache tile row
  static constexpr int OFF_K = 0;                      // K ring
  static constexpr int OFF_V = OFF_K + NK * SLOT;      // V ring
  // fp8: the widened (f16) V rows of NCV steps, 128-byte-swizzled operands of two 64-dim
  // slabs, indexed by the step modulo NSP, so that the buffer of step g is released by the
  // PV's commit to pv_done.  The K codes are not widened: the logits MMA is of kind f8f6f4,
  // with the query rows split into two E4M3 terms.
  static constexpr int NCV = FP8 ? NSP : 0;
  static constexpr int CV_SLAB = SUB * 128;
  static constexpr int CV_BUF = 2 * CV_SLAB;
  static constexpr int OFF_CV = OFF_V + NV * SLOT;     // K buffers, then V buffers
  static constexpr int SCRATCH = OFF_CV;  // bytes free for the merges at the end (the rings)
  static constexpr int KSLAB = FP8 ? CV_SLAB : TT * 128;  // slab stride of the MMA operands
  // two-stream merge: the second stream's O rows (fp32, 16-byte chunks swizzled by row)
  static constexpr int OFF_MRG = OFF_CV + NCV * CV_BUF;
  static constexpr int MRG_BYTES = DUAL ? 64 * D * 4 : 0;
  // per-token scales: NSC slots of 64 K then 64 V fp32 scales
  static constexpr int NSC = TOKS ? 8 : 0;
  static constexpr int SC_SLOT = 2 * TT * 4;
  static constexpr int OFF_SC = OFF_MRG + MRG_BYTES;
  static constexpr int OFF_ML = OFF_SC + NSC * SC_SLOT;
  static constexpr int ML_BYTES = round_up(2 * MP * 4 + (DUAL ? 2 * 64 * 4 : 0), 128);
  static constexpr int OFF_BAR = round_up(OFF_ML + ML_BYTES, 64);
  // full_k, empty_k (NK each), full_v, empty_v (NV each), s_full, p_full, pv_done (NSP each),
  // o_free, q_full, mma_end, cv_full (NCV), sc_full and
  // sc_free (NSC each)
  static constexpr int NBAR = 2 * NK + 2 * NV + 3 * NSP + 3 + NCV + 2 * NSC;
  // after the barriers: the flag words, the derived first item and the CTA's flags
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + kFlagBytes + 32 + 1024;
  static constexpr int CTAS_PER_SM = 1;
  // Tensor memory (lane = query row, 32-bit columns): NSP S/P buffers of SUB fp32 columns
  // (P, SUB / 2 columns of 16-bit pairs, overwrites the first half of its own S), O (D fp32
  // columns) and Q (D / 2 columns of 16-bit pairs).  Head dim 128: S/P [0, 64 NSP), O
  // [64 NSP, 64 NSP + 128), Q after O.  Head dim 256: S/P [0, 128), Q [128, 256),
  // O [256, 512).
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = D == 256 ? 256 : NSP * SUB;
  static constexpr uint32_t COL_Q = D == 256 ? NSP * SUB : COL_O + D;
  // query columns: D / 2 16-bit pairs, or for an fp8 cache up to three E4M3 terms of D / 4
  static constexpr int QCOLS = FP8 ? 3 * D / 4 : D / 2;
  static_assert(NSP * SUB + D + QCOLS <= (int)TMEM_COLS, "tensor memory");
  static_assert(!TOKS || FP8, "per-token scales belong to fp8 caches");
  static_assert(!FP8 || D == 128, "fp8 caches at head dim 128");
  static_assert(!FP8 || (SUB * 8) % (32 * (NCW > 0 ? NCW : 1)) == 0, "widening: whole passes");
  // the V rows of step g wait for the PV of step g - NSP, issued after the S of step
  // g - NSP + LAG: the PVs trail the S MMAs by fewer steps than there are buffers
  static_assert(LAG >= 1 && LAG < NSP, "no cycle between the roles");
  static_assert(!FP8 || NCV == NSP, "a widened V buffer is released through pv_done");
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
// kind::f8f6f4 with A in tensor memory (lane = row, a 32-bit column = four E4M3 K elements)
// and B an E4M3 shared operand; the instruction descriptor's operand formats are 0 (E4M3).
__device__ __forceinline__ void umma_f8_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
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
// tmem_ld32 in two halves, so that independent work can run while the load is in flight:
// the issue, and the wait, which takes the destination registers as operands so that no use
// of them can be moved above it.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
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
// Two fp32 values to two E4M3 codes (a -> low byte): round to nearest even, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b) {
  uint16_t r;
  asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n mov.b16 %0, t;\n}"
      : "=h"(r)
      : "f"(b), "f"(a));
  return r;
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
// CTA's work list goes to slot n % NK of the K ring and n % NV of the V ring; lane
// page * NSLAB + slab copies one 128-byte column slab of one page of the tile.  The order of
// the copies is K(0), K(1), V(0), K(2), V(1), ...: a copy waits until the tile one ring
// length earlier has been read from its slot (by its S for K and its PV for V, or, for fp8, by the
// widening warps).  Per-token scales of tile n go to slot n % NSC of the scale ring, which
// the softmax releases.
//
// The warp issues a tile's copies every few hundred clocks, so nothing on its path may wait
// on memory: the parameters it uses live in registers, and each lane's block id is looked
// up two tiles before its copy is issued (and not at all while the tile stays on the page of
// the previous one).
// A CTA's work list as one thread sees it: item 0 is the one the CTA derived from the lengths
// (first_item_of); the rest are the planner's, items [lb + 1, le) of its list, read after
// the first wait on the planner, which also lets the next launch start (so the next launch
// starts only once the planner has finished: the reduce kernel reads the planner's list
// before its own wait on this grid).
struct ItemList {
  const int32_t* item_off;
  const int4* items;
  int4 first;
  int lb, le;  // le < 0 until the planner's list has been read

  __device__ __forceinline__ void init(const KernelParams& p, int4 f) {
    item_off = p.item_off;
    items = p.items;
    first = f;
    lb = 0;
    le = -1;
  }
  // wait for the planner (a no-op once it has finished for this thread)
  __device__ __forceinline__ void wait_planner() {
    grid_dependency_wait();
    grid_dependents_launch();
  }
  // wait for the planner (once) and read the CTA's range of its list
  __device__ __forceinline__ void planned() {
    if (le >= 0) return;
    wait_planner();
    lb = item_off[blockIdx.x];
    le = item_off[blockIdx.x + 1];
  }
  // item k (k >= 1 waits for the planner); false past the list's end
  __device__ __forceinline__ bool get(int k, int4& item) {
    if (k == 0) {
      item = first;
      return true;
    }
    planned();
    if (lb + k >= le) return false;
    item = items[lb + k];
    return true;
  }
};

template <class T>
struct TcProducer {
  struct Box {
    int blk, row, g, tok0, t1;
    bool ok;
    uint32_t nvalid;
  };
  // a tile whose block id (this lane's page) is being fetched
  struct Ahead {
    int b, g, tok0, t1, blk;
    bool want, valid;
  };
  const CUtensorMap* kmap;
  const CUtensorMap* vmap;
  char* smem;
  uint64_t *full_k, *rel_k, *full_v, *rel_v, *sc_full, *sc_free;
  volatile int* abort_flag;
  int* flags;  // the CTA's flags in shared memory, published once the planner has finished
  const int32_t* bt;
  const int4* items;
  const float* kscale;
  const float* vscale;
  int maxb, bs, bs_shift, nblocks, Hkv, RB;
  int lane, box_rows, nbox;
  uint32_t box_bytes, nk, nv, nsc;
  bool scale_bulk;  // a tile's scales are two contiguous 256-byte runs (one kv head, big pages)
  // walk over the work list (the tile after the two being fetched)
  ItemList list;
  int it, k, ntiles, t0, t1, b, g;
  bool have;
  int4 item_next;  // item it + 1 once past item 0
  int last_b, last_page, last_blk;  // this lane's previous lookup
  Ahead q0, q1;

  __device__ __forceinline__ void init(const KernelParams* prm, const CUtensorMap* km,
                                       const CUtensorMap* vm, char* sm, uint64_t* fk,
                                       uint64_t* rk, uint64_t* fv, uint64_t* rv, uint64_t* scf,
                                       uint64_t* scr, volatile int* ab, int* sflags, int ln,
                                       int4 first) {
    kmap = km; vmap = vm; smem = sm; full_k = fk; rel_k = rk; full_v = fv; rel_v = rv;
    sc_full = scf; sc_free = scr; abort_flag = ab; lane = ln;
    flags = sflags; bt = prm->bt; items = prm->items; kscale = prm->k_scale;
    vscale = prm->v_scale; maxb = prm->maxb; bs = prm->bs; bs_shift = prm->bs_shift;
    nblocks = prm->nblocks; Hkv = prm->Hkv; RB = prm->RB;
    box_rows = min(bs, T::TT);
    nbox = T::TT / box_rows;
    box_bytes = (uint32_t)box_rows * T::ROWB;
    scale_bulk = T::TOKS && Hkv == 1 && box_rows == T::TT &&
                 ((reinterpret_cast<uintptr_t>(kscale) | reinterpret_cast<uintptr_t>(vscale)) & 15) == 0;
    nk = nv = nsc = 0;
    list.init(*prm, first);
    it = -1;
    have = false;
    last_b = -1;
    last_page = -1;
    last_blk = -1;
    fetch(q0);
    fetch(q1);
  }

  // The next tile of the work list into a, with this lane's block id lookup started.
  __device__ __forceinline__ void fetch(Ahead& a) {
    while (!have) {
      int4 item;
      if (++it == 0) {
        item = list.first;
      } else {
        // item it, read one ahead from item 1 on (item 0 needs no list: no wait for it)
        if (it == 1 && !list.get(1, item_next)) {
          a.valid = false;
          return;
        }
        if (list.lb + it >= list.le) {
          a.valid = false;
          return;
        }
        item = item_next;
        if (!list.get(it + 1, item_next)) item_next = make_int4(0, 0, 0, -1);
      }
      t0 = item.y;
      t1 = item.z;
      if (t1 <= t0) continue;
      b = item.x / (Hkv * RB);
      g = (item.x / RB) % Hkv;
      k = 0;
      ntiles = ceil_div(t1 - t0, T::TT);
      have = true;
    }
    a.valid = true;
    a.b = b;
    a.g = g;
    a.tok0 = t0 + k * T::TT;
    a.t1 = t1;
    if (++k >= ntiles) have = false;
    const int tokb = a.tok0 + (lane / T::NSLAB) * box_rows;
    a.want = lane < nbox * T::NSLAB && tokb < a.t1;
    a.blk = -1;
    if (a.want) {
      const int page = tokb >> bs_shift;
      if (a.b != last_b || page != last_page) {
        last_blk = __ldg(bt + (size_t)a.b * maxb + page);
        last_b = a.b;
        last_page = page;
      }
      a.blk = last_blk;
    }
  }

  // This lane's box of the next tile of the list; false when the list is exhausted.
  __device__ __forceinline__ bool next_tile(Box& bx) {
    if (!q0.valid) return false;
    bx.tok0 = q0.tok0;
    bx.t1 = q0.t1;
    bx.g = q0.g;
    bx.blk = q0.blk;
    bx.ok = q0.want && q0.blk >= 0 && q0.blk < nblocks;
    if (q0.want && !bx.ok) atomicOr(flags, PA_FLAG_BAD_BLOCK_ID);
    bx.nvalid = __popc(__ballot_sync(kFull, bx.ok));
    bx.row = (q0.tok0 + (lane / T::NSLAB) * box_rows) & (bs - 1);
    q0 = q1;
    fetch(q1);
    return true;
  }

  __device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity) {
    if (mbar_wait(bar, parity, abort_flag)) return true;
    atomicOr(flags, PA_FLAG_WAIT_TIMEOUT);
    *abort_flag = 1;
    return false;
  }

  // Copy a tile's boxes into slot n % NS of one ring once the slot is released (the release
  // barrier completes once per use of the slot, in tile order).
  template <int NS>
  __device__ __forceinline__ bool issue(const Box& bx, uint32_t n, uint64_t* full,
                                        uint64_t* rel, const CUtensorMap* map, int ring) {
    const int s = (int)(n % NS);
    if (!wait_or_abort(&rel[s], ((n / NS) & 1) ^ 1)) return false;
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

  // The K and V scales of tile n's tokens into scale slot n % NSC, completing on sc_full
  // (32 arrivals: one per lane).  One kv head and pages of at least a tile: the tile's scales
  // are two contiguous 256-byte runs, copied by two bulk copies; otherwise 4-byte cp.async,
  // two tokens a lane.  Tokens past the item or on a bad page keep a stale value: the softmax
  // masks them.
  __device__ __forceinline__ bool issue_scales(const Box& bx, uint32_t n) {
    if constexpr (T::TOKS) {
      const int s = (int)(n % T::NSC);
      if (!wait_or_abort(&sc_free[s], ((n / T::NSC) & 1) ^ 1)) return false;
      float* ks = reinterpret_cast<float*>(smem + T::OFF_SC + s * T::SC_SLOT);
      float* vs = ks + T::TT;
      if (scale_bulk) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&sc_full[s], bx.ok ? 2u * T::TT * 4 : 0u);
          if (bx.ok) {  // lane 0's box is the tile's one page
            const size_t idx = (size_t)bx.blk * bs + bx.row;
            bulk_load_1d(ks, kscale + idx, T::TT * 4, &sc_full[s]);
            bulk_load_1d(vs, vscale + idx, T::TT * 4, &sc_full[s]);
          }
        } else {
          mbar_arrive(&sc_full[s]);
        }
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int t = lane + 32 * h;
          const int src = (t / box_rows) * T::NSLAB;  // the lane holding the page's block id
          const int blk = __shfl_sync(kFull, bx.blk, src);
          const bool ok = __shfl_sync(kFull, bx.ok ? 1 : 0, src) != 0;
          const int tok = bx.tok0 + t;
          if (ok && tok < bx.t1) {
            const size_t idx = ((size_t)blk * bs + (tok & (bs - 1))) * Hkv + bx.g;
            cp_async_4(ks + t, kscale + idx);
            cp_async_4(vs + t, vscale + idx);
          }
        }
        cp_async_arrive_noinc(&sc_full[s]);
      }
    }
    return true;
  }

  // K (and the scales) of a tile, counted as soon as each copy is in flight
  __device__ __forceinline__ bool issue_k(const Box& bx) {
    if (!issue<T::NK>(bx, nk, full_k, rel_k, kmap, T::OFF_K)) return false;
    ++nk;
    if (!issue_scales(bx, nsc)) return false;
    ++nsc;
    return true;
  }

  __device__ __forceinline__ void run() {
    // K runs KLEAD steps ahead of V: q[0 .. pending) are the tiles whose K is out and whose
    // V is not yet, oldest first (fixed indices, shifted down after each V, so that they
    // stay in registers)
    constexpr int KLEAD = T::KLEAD;
    Box q[KLEAD + 1];
    int pending = 0;
    bool more = true;
#pragma unroll
    for (int i = 0; i < KLEAD; ++i) {
      if (more) more = next_tile(q[i]);
      if (more) {
        if (!issue_k(q[i])) return;
        pending = i + 1;
      }
    }
    while (pending > 0) {
      bool added = false;
      if (more && pending == KLEAD) {  // steady state: one tile in, one out
        more = next_tile(q[KLEAD]);
        if (more) {
          if (!issue_k(q[KLEAD])) return;
          added = true;
        }
      }
      if (!issue<T::NV>(q[0], nv, full_v, rel_v, vmap, T::OFF_V)) return;
      ++nv;
#pragma unroll
      for (int i = 0; i < KLEAD; ++i) q[i] = q[i + 1];
      if (!added) --pending;
    }
  }

  // Let every copy this warp started land before the CTA may exit.
  __device__ __forceinline__ void drain() {
    if constexpr (T::TOKS) {
      cp_async_wait_all();
      for (uint32_t j = nsc > (uint32_t)T::NSC ? nsc - T::NSC : 0; j < nsc; ++j)
        mbar_wait_drain(&sc_full[j % T::NSC], (j / T::NSC) & 1);
    }
    for (uint32_t j = nk > (uint32_t)T::NK ? nk - T::NK : 0; j < nk; ++j)
      mbar_wait_drain(&full_k[j % T::NK], (j / T::NK) & 1);
    for (uint32_t j = nv > (uint32_t)T::NV ? nv - T::NV : 0; j < nv; ++j)
      mbar_wait_drain(&full_v[j % T::NV], (j / T::NV) & 1);
  }
};

template <int D_, int MP, int KVK, int QK, bool TOKS>
__global__ void __launch_bounds__(TcTraits<D_, MP, KVK, TOKS>::NTHREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const KernelParams p) {
  using T = TcTraits<D_, MP, KVK, TOKS>;
  constexpr int SUB = T::SUB;
  constexpr int D = T::D;
  constexpr int NSP = T::NSP;
  constexpr bool BF = KVK == KV_BF16;  // MMA operands bf16 (else f16: f16 and fp8 caches)
  constexpr uint32_t ID_S = umma_idesc(128, SUB, BF, false);
  constexpr uint32_t ID_S8 = umma_idesc(128, SUB, false, false);  // f8f6f4: E4M3 x E4M3
  // E4M3 terms of a query row for an fp8 cache: a bf16 query's 8 significant bits fit in two
  // of 4, an fp16 query's 11 in three
  constexpr int QTERMS = QK == Q_BF16 ? 2 : 3;
  constexpr uint32_t ID_PV = umma_idesc(128, D, BF, true);
  constexpr int SOFT_BAR = 2;  // named barrier of the four softmax warps
  extern __shared__ char smem_raw[];
  char* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t* full_k = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty_k = full_k + T::NK;
  uint64_t* full_v = empty_k + T::NK;
  uint64_t* empty_v = full_v + T::NV;
  uint64_t* s_full = empty_v + T::NV;  // [NSP]: S of the step in buffer b is complete
  uint64_t* p_full = s_full + NSP;        // [NSP]: P of the step in buffer b is written
  uint64_t* pv_done = p_full + NSP;       // [NSP]: the PV that read buffer b has completed
  uint64_t* o_free = pv_done + NSP;
  uint64_t* q_full = o_free + 1;
  uint64_t* mma_end = q_full + 1;
  uint64_t* cv_full = mma_end + 1;       // [NCV]: widened V rows of the step in buffer b
  uint64_t* sc_full = cv_full + T::NCV;  // [NSC]: per-token scales of the step in slot b
  uint64_t* sc_free = sc_full + T::NSC;  // [NSC]: the softmax is done with slot b
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sc_free + T::NSC);
  volatile int* pend = abort_flag + 2;        // [4]: split pieces published, see finish_pending
  volatile int* cnt_seen_s = abort_flag + 6;  // published pieces of the item's unit, seen late
  uint32_t* tslot = reinterpret_cast<uint32_t*>(const_cast<int*>(abort_flag + 7));
  float* mlbuf = reinterpret_cast<float*>(smem + T::OFF_ML);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    // readers of a ring slot: the widening warps (fp8 V), or the commit of the S (K) or PV
    // (V) that read it when the ring is not released through s_full / pv_done; full: the
    // expect_tx arrival of the copy
    for (int s = 0; s < T::NK; ++s) {
      mbar_init(&full_k[s], 1);
      mbar_init(&empty_k[s], 1);
    }
    for (int s = 0; s < T::NV; ++s) {
      mbar_init(&full_v[s], 1);
      mbar_init(&empty_v[s], T::FP8 ? T::NCW : 1);
    }
    for (int b = 0; b < T::NCV; ++b) mbar_init(&cv_full[b], T::NCW);
    for (int b = 0; b < NSP; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
      mbar_init(&pv_done[b], 1);
    }
    for (int b = 0; b < T::NSC; ++b) {
      mbar_init(&sc_full[b], 32);  // one cp.async arrival per producer lane
      mbar_init(&sc_free[b], 4);   // the four softmax warps
    }
    mbar_init(o_free, 4);
    mbar_init(q_full, 4);
    mbar_init(mma_end, 1);
    *abort_flag = 0;
    pend[0] = -1;
    pend[2] = -1;
    abort_flag[12] = 0;  // the CTA's flags (s_flags)
    abort_flag[13] = 0;  // 1 once the derived first item is checked against the planner's
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
  // The CTA's first work item, derived from the lengths (the planner's rules), so that its
  // copies and MMAs start while the planner may still be running.  The lengths, the tables,
  // the queries and the caches were written before the planner ran (this grid starts only
  // once the planner has passed its own wait), so they may be read now; the planner's list
  // and every write wait for the planner (ItemList::planned).
  volatile int* s_first = abort_flag + 8;  // 4 ints
  if (warp == T::W_SOFT) {
    const int4 f = first_item_of(p, blockIdx.x, gridDim.x, lane);
    if (lane == 0) {
      s_first[0] = f.x;
      s_first[1] = f.y;
      s_first[2] = f.z;
      s_first[3] = f.w;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t t_s = tmem, t_o = tmem + T::COL_O, t_q = tmem + T::COL_Q;
  const int4 first = make_int4(s_first[0], s_first[1], s_first[2], s_first[3]);
  // flags raised before the planner's own header write could be overwritten by it: they are
  // gathered here and published at the end
  int* s_flags = const_cast<int*>(abort_flag + 12);
  volatile int* first_checked = abort_flag + 13;
  // the item this CTA derived must be the planner's (else the lengths changed between the
  // planner's launch and this one)
  auto check_first = [&](int4 pf) {
    if (pf.x != first.x || pf.y != first.y || pf.z != first.z || pf.w != first.w)
      atomicOr(s_flags, PA_FLAG_STALE_PLAN);
  };
  auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
    if (!mbar_wait(bar, parity, abort_flag)) {
      atomicOr(s_flags, PA_FLAG_WAIT_TIMEOUT);
      *abort_flag = 1;
    }
  };

  if (warp == T::W_PROD) {
    // ================================================================ TMA producer
    TcProducer<T> prod;
    prod.init(&p, &kmap, &vmap, smem, full_k, T::K_BY_S ? s_full : empty_k, full_v,
              T::V_BY_PV ? pv_done : empty_v, sc_full, sc_free, abort_flag, s_flags, lane, first);
    prod.run();  // every tile of the work list, as slots come free
    prod.drain();
  } else if (warp == T::W_MMA) {
    // ================================================================ MMA issue
    if (lane == 0) {
      uint32_t g = 0, items_done = 0;
      uint32_t q_ph = 0, o_ph = 0;
      // step x uses buffer x % NSP; every barrier of a buffer completes once per use, in
      // step order, so the phase of step x is (x / NSP) & 1
      // O += P V of step gp (its P, in buffer gp % NSP, must be written); the commit to
      // pv_done also releases the V slot (or the widened V buffer) of the step
      auto issue_pv = [&](uint32_t gp, bool first) {
        uint32_t vaddr;
        if constexpr (T::FP8) {
          wait_bar(&cv_full[gp % NSP], (gp / NSP) & 1);
          vaddr = smem_addr(smem + T::OFF_CV + (gp % NSP) * T::CV_BUF);
        } else {
          const int slot = (int)(gp % T::NV);
          wait_bar(&full_v[slot], (gp / T::NV) & 1);
          vaddr = smem_addr(smem + T::OFF_V + slot * T::SLOT);
        }
        wait_bar(&p_full[gp % NSP], (gp / NSP) & 1);
        if (first && items_done > 0) {  // the previous item's epilogue has read O
          wait_bar(o_free, o_ph);
          o_ph ^= 1u;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < SUB / 16; ++kk) {
          const uint64_t bd = umma_desc(vaddr + kk * 2048, T::KSLAB, 1024);
          umma_f16_ta(t_o, t_s + (gp % NSP) * SUB + kk * 8, bd, ID_PV, !(first && kk == 0));
        }
        umma_commit(&pv_done[gp % NSP]);
        if constexpr (!T::FP8 && !T::V_BY_PV) umma_commit(&empty_v[gp % T::NV]);
      };
      ItemList list;
      list.init(p, first);
      int4 item;
      for (int it = 0; list.get(it, item); ++it) {
        const int t0 = item.y, t1 = item.z;
        if (t1 <= t0) continue;
        const int nsub = ceil_div(t1 - t0, SUB);
        wait_bar(q_full, q_ph);  // the item's query rows are in tensor memory
        q_ph ^= 1u;
        // the PVs trail the S MMAs by LAG steps, so the in-order tensor pipe holds the
        // logits of the next steps ahead of a PV that waits for the softmax, and the S that
        // reuses a buffer (after the PV of step g - NSP) finds MMAs still queued
        constexpr int LAG = T::LAG;
        const uint32_t g_item = g;  // the item's first step
        for (int j = 0; j < nsub; ++j, ++g) {
          const int slot = (int)(g % T::NK);
          wait_bar(&full_k[slot], (g / T::NK) & 1);
          const uint32_t kbase = smem_addr(smem + T::OFF_K + slot * T::SLOT);
          if (g >= (uint32_t)NSP) {  // the buffer holds P(g - NSP) until its PV has read it
            const uint32_t x = g - NSP;
            wait_bar(&pv_done[x % NSP], (x / NSP) & 1);
          }
          tc_fence_after();
          const uint32_t t_sg = t_s + (g % NSP) * SUB;
          if constexpr (T::FP8) {
            // the E4M3 codes against the query's E4M3 terms (columns [t D/4, (t + 1) D/4) of
            // Q for term t), 32 codes a MMA, all into the same logits
#pragma unroll
            for (int tm = 0; tm < QTERMS; ++tm) {
#pragma unroll
              for (int kk = 0; kk < D / 32; ++kk) {
                const uint64_t bd = umma_desc(kbase + kk * 32, 16, 1024);
                umma_f8_ta(t_sg, t_q + tm * (D / 4) + kk * 8, bd, ID_S8, tm > 0 || kk > 0);
              }
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t bd = umma_desc(kbase + (kk >> 2) * T::KSLAB + (kk & 3) * 32, 16, 1024);
              umma_f16_ta(t_sg, t_q + kk * 8, bd, ID_S, kk > 0);
            }
          }
          // the logits are ready; the K slot of the step is free
          umma_commit(&s_full[g % NSP]);
          if constexpr (!T::K_BY_S) umma_commit(&empty_k[g % T::NK]);
          if (j >= LAG) issue_pv(g - LAG, j == LAG);
        }
        for (int j = nsub > LAG ? nsub - LAG : 0; j < nsub; ++j) issue_pv(g_item + j, j == 0);
        ++items_done;
      }
      umma_commit(mma_end);
      if (!mbar_wait_drain(mma_end, 0)) atomicOr(s_flags, PA_FLAG_WAIT_TIMEOUT);
    }
    // 16-bit caches: the idle lanes wait here for lane 0.  The divergent paths of a warp run
    // one after the other, and lanes 1-31 going on to the final wait on the grid before (the
    // previous decode, when launched back to back) held lane 0's MMAs until it had ended
    // (back-to-back decodes of head dim 256, Sq = 64: 174.7 -> 164.5 us at B = 8).  With an
    // fp8 cache the same convergence point measured slower (74.7 -> 77.3 us), so there the
    // lanes go on.
    if constexpr (!T::FP8) __syncwarp();
  } else if (warp < T::W_CONV) {
    // ================================================================ softmax and epilogue
    constexpr bool DUAL = T::DUAL;
    constexpr int NL = T::NL;                       // logits of a step per thread
    const int stid = tid - T::W_SOFT * 32;          // 0 .. 127 over the four warps
    const int r = 32 * (warp & 3) + lane;           // this thread's tensor-memory lane
    const int hs = DUAL ? (r >> 6) : 0;             // token stream: the step's tokens [NL hs, NL hs + NL)
    const int qr = DUAL ? (r & 63) : r;             // query row of the unit's tile
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const bool tensor_scale = p.scale_mode == PA_SCALE_PER_TENSOR;
    const float kts = tensor_scale ? __ldg(p.k_scale) : 1.f;
    const float vts = tensor_scale ? __ldg(p.v_scale) : 1.f;
    const float qk_scale = p.qk_scale * kts;
    float* mrg = reinterpret_cast<float*>(smem + T::OFF_MRG);  // [64][D], chunks swizzled
    float* mrg_ml = mlbuf + 2 * MP;                             // [64][2]: m, l of stream 1
    uint32_t g = 0;
    uint32_t pv_next = 0;  // the first step whose PV completion is not consumed yet
    // wait until the PV of step x (which read buffer x % NSP) has completed; completions
    // are consumed in step order, and none is ever two ahead of its consumer on a buffer
    auto wait_pv_step = [&](uint32_t x) {
      for (; pv_next <= x; ++pv_next)
        wait_bar(&pv_done[pv_next % NSP], (pv_next / NSP) & 1);
      tc_fence_after();
    };
    int2 pend_even = make_int2(-1, 0), pend_odd = make_int2(-1, 0);  // held by stid 0
    ItemList list;
    list.init(p, first);
    int4 item, item_next;
    bool have_next = false;
    for (int it = 0;; ++it) {
      if (it == 0)
        item = first;
      else if (have_next)
        item = item_next;
      else if (!list.get(it, item))
        break;
      // the next item is read ahead from item 1 on (item 0 waits for nothing)
      have_next = it >= 1 && list.get(it + 1, item_next);
      const int u = item.x, t0 = item.y, t1 = item.z, slot = item.w;
      if (t1 <= t0) continue;
      const int b = u / (p.Hkv * p.RB), g_kv = (u / p.RB) % p.Hkv, rb = u % p.RB;
      const int n = __ldg(p.ctx + b), ql = __ldg(p.qlens + b);
      // the unit's pieces (planner data): for item 0 read halfway through it, when the
      // planner has long finished, off the path of its last steps
      int2 uinfo = make_int2(0, 1);
      bool in_dec = false;
      auto read_uinfo = [&]() {
        list.wait_planner();
        int4 pf = first;
        if (it == 0 && stid == 0) pf = p.first_item[blockIdx.x];
        if (slot >= 0) {
          uinfo = __ldg(&p.unit_info[u]);
          in_dec = uinfo.y <= p.ns_dec;
        }
        if (it == 0 && stid == 0) {
          check_first(pf);
          first_checked[0] = 1;
        }
      };
      if (it > 0) read_uinfo();
      const int nsub = ceil_div(t1 - t0, SUB);
      int cnt_seen = -1;
      const int rg = rb * MP + qr;
      const bool real = qr < MP && rg < p.M;
      const int qi = real ? rg / p.G : 0, hq = g_kv * p.G + (real ? rg % p.G : 0);
      const int lim = (real && qi < ql) ? (p.causal ? n - ql + qi + 1 : n) : 0;
      // a warp whose 32 rows hold no query (padding rows of a tile) skips the softmax; its
      // rows of P and O are never read, and it keeps only the waits and arrivals that keep
      // the barriers' phases in step
      const bool warp_dead = __all_sync(kFull, !real);
      // ---- this thread's query row into tensor memory (every MMA of the previous item has
      // completed); rows of no query are zero
      const uint4* qrow = reinterpret_cast<const uint4*>(
          reinterpret_cast<const char*>(p.q) + ((((size_t)b * p.Sq + qi) * p.Hq + hq) * D) * 2);
      float qk_row = qk_scale;  // the logit scale of this row
      if constexpr (T::FP8) {
        // fp8 cache: the row times a power of two sq (the largest with |q| sq <= 448) as
        // QTERMS E4M3 terms, t0 = e4m3(q sq), t1 = e4m3(q sq - t0), t2 = e4m3(q sq - t0 - t1),
        // term t in columns [t D/4, (t + 1) D/4), four codes a column.  Each term carries the
        // next 4 significant bits, so the terms sum to the query exactly (two for bf16's 8
        // bits, three for fp16's 11) but for elements whose low bits fall below the smallest
        // E4M3 subnormal, about a thousandth of the row's largest and smaller; the MMAs of
        // each 32 codes accumulate all terms into the logits, and 1/sq goes into the row's
        // logit scale
        auto q_f2 = [&](uint32_t w) { return QK == Q_BF16 ? bf16x2_to_f2(w) : f16x2_to_f2(w); };
        float amax = 0.f;
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = real ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int jw = 0; jw < 4; ++jw) {
            const float2 f = q_f2(wv[jw]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
        int e = 0;  // floor(log2(448 / amax)), from the exponent field of the quotient
        if (amax > 0.f) {
          e = (int)((__float_as_uint(__fdiv_rn(448.f, amax)) >> 23) & 0xff) - 127;
          e = max(-126, min(126, e));
        }
        const float sq = __uint_as_float((uint32_t)(e + 127) << 23);
        qk_row = qk_scale * __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll 1
        for (int h = 0; h < D / 64; ++h) {  // 64 dims: 16 columns of each term
          uint32_t wt[QTERMS][16];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = real ? __ldg(qrow + 8 * h + c) : make_uint4(0, 0, 0, 0);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q4 = 0; q4 < 2; ++q4) {  // four dims, one column
              const float2 fa = q_f2(wv[2 * q4]), fb = q_f2(wv[2 * q4 + 1]);
              // what is left of the four scaled elements after the terms so far (exact)
              float r0 = fa.x * sq, r1 = fa.y * sq, r2 = fb.x * sq, r3 = fb.y * sq;
#pragma unroll
              for (int tm = 0; tm < QTERMS; ++tm) {
                const uint32_t c01 = f32x2_to_e4m3x2(r0, r1), c23 = f32x2_to_e4m3x2(r2, r3);
                wt[tm][2 * c + q4] = c01 | (c23 << 16);
                if (tm + 1 < QTERMS) {
                  const float2 d01 = f16x2_to_f2(e4m3x2_to_h2(c01));
                  const float2 d23 = f16x2_to_f2(e4m3x2_to_h2(c23));
                  r0 -= d01.x;
                  r1 -= d01.y;
                  r2 -= d23.x;
                  r3 -= d23.y;
                }
              }
            }
          }
#pragma unroll
          for (int tm = 0; tm < QTERMS; ++tm) tmem_st16u(t_q + lane_off + tm * (D / 4) + 16 * h, wt[tm]);
        }
        tmem_wait_st();
      } else {
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = real ? __ldg(qrow + 8 * h + c) : make_uint4(0, 0, 0, 0);
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
        const int c0 = NL * hs;  // this stream's first token of the step
        if (it == 0 && j == (nsub - 1) / 2) read_uinfo();
        if (in_dec && j + 1 == nsub && stid == 0) cnt_seen = ld_acquire_gpu(&p.unit_cnt[u]);
        if (!T::FP8 && nv < SUB) {
          // the zeroing below writes into the V slot: the tile must have landed (this wait
          // orders the writes after the copy)
          wait_bar(&full_v[g % T::NV], (g / T::NV) & 1);
        }
        wait_bar(&s_full[g % NSP], (g / NSP) & 1);
        tc_fence_after();
        if (g >= (uint32_t)NSP) wait_pv_step(g - NSP);  // (complete: S(g) came after it)
        const float* sks = reinterpret_cast<const float*>(smem + T::OFF_SC);  // K, then V scales
        if constexpr (T::TOKS) {
          sks += (g % T::NSC) * (T::SC_SLOT / 4);
          wait_bar(&sc_full[g % T::NSC], (g / T::NSC) & 1);
        }
        if (!warp_dead) {
          const uint32_t t_sg = t_s + (g % NSP) * SUB + lane_off;
          float x[NL];
          // per-token scales of this stream's keys and values (two streams): read from shared
          // memory while the logits are on their way from tensor memory
          float ksc[NL], vsc[NL];
          constexpr bool SC_REG = T::TOKS && NL == 32;
          if constexpr (NL == 64) {
            tmem_ld64(t_sg, x);
          } else if constexpr (SC_REG) {
            uint32_t xr[32];
            tmem_ld32_issue(t_sg + c0, xr);
#pragma unroll
            for (int i = 0; i < NL / 4; ++i) {
              const float4 k4 = *reinterpret_cast<const float4*>(sks + c0 + 4 * i);
              const float4 v4 = *reinterpret_cast<const float4*>(sks + T::TT + c0 + 4 * i);
              ksc[4 * i] = k4.x;
              ksc[4 * i + 1] = k4.y;
              ksc[4 * i + 2] = k4.z;
              ksc[4 * i + 3] = k4.w;
              vsc[4 * i] = v4.x;
              vsc[4 * i + 1] = v4.y;
              vsc[4 * i + 2] = v4.z;
              vsc[4 * i + 3] = v4.w;
            }
            tmem_ld32_wait(xr);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) x[jj] = __uint_as_float(xr[jj]);
          } else {
            tmem_ld32(t_sg + c0, x);
          }
          // ---- online softmax of this thread's logits (log2 units), two per instruction
          const float2 s2 = make_float2(qk_row, qk_row), z2 = make_float2(0.f, 0.f);
          if constexpr (T::TOKS) {
            // logit j of the step times its key's scale
#pragma unroll
            for (int i = 0; i < NL / 4; ++i) {
              const float4 k4 = SC_REG ? make_float4(ksc[4 * i], ksc[4 * i + 1], ksc[4 * i + 2],
                                                     ksc[4 * i + 3])
                                       : *reinterpret_cast<const float4*>(sks + c0 + 4 * i);
              const float2 a = ffma2(make_float2(x[4 * i], x[4 * i + 1]), s2, z2);
              const float2 c = ffma2(make_float2(x[4 * i + 2], x[4 * i + 3]), s2, z2);
              const float2 ya = ffma2(a, make_float2(k4.x, k4.y), z2);
              const float2 yc = ffma2(c, make_float2(k4.z, k4.w), z2);
              x[4 * i] = ya.x;
              x[4 * i + 1] = ya.y;
              x[4 * i + 2] = yc.x;
              x[4 * i + 3] = yc.y;
            }
          } else {
#pragma unroll
            for (int i = 0; i < NL / 2; ++i) {
              const float2 y = ffma2(make_float2(x[2 * i], x[2 * i + 1]), s2, z2);
              x[2 * i] = y.x;
              x[2 * i + 1] = y.y;
            }
          }
          // masked keys (past the item's tokens or past the row's causal limit) become -inf;
          // most steps have none
          if (c0 + NL > nv || tok0 + c0 + NL > lim) {
#pragma unroll
            for (int jj = 0; jj < NL; ++jj)
              if (c0 + jj >= nv || tok0 + c0 + jj >= lim) x[jj] = -INFINITY;
          }
          float mx = -INFINITY;
#pragma unroll
          for (int jj = 0; jj < NL; jj += 2) mx = fmaxf(mx, fmaxf(x[jj], x[jj + 1]));
          const bool need = mx > m_run + 8.f;  // lazy rescale: only when the max grows by 2^8
          const bool rescale = __any_sync(kFull, need);
          const float mn = need ? mx : m_run;
          const float alpha = (mn == m_run || m_run == -INFINITY) ? 1.f : fast_exp2(m_run - mn);
          m_run = mn;
          // this thread's part of its row of P, 16-bit pairs over the first SUB / 2 columns
          // of its own logits (all of them are in registers); a masked logit (-inf) gives
          // exp2 = 0, and a row with no visible key so far has only zeros.  With two streams
          // the other stream's half of the row is written as zeros.
          float lsum = 0.f;
          {
            const float2 nm = make_float2(m_run == -INFINITY ? 0.f : -m_run,
                                          m_run == -INFINITY ? 0.f : -m_run);
            const float2 one2 = make_float2(1.f, 1.f);
            float2 ls2 = z2;
            const float* svs = sks + T::TT;
#pragma unroll
            for (int h = 0; h < NL / 32; ++h) {  // 32 tokens = 16 columns at a time
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float2 t = ffma2(make_float2(x[32 * h + 2 * i], x[32 * h + 2 * i + 1]), one2, nm);
                float p0 = fast_exp2(t.x), p1 = fast_exp2(t.y);
                ls2 = ffma2(make_float2(p0, p1), one2, ls2);
                if constexpr (T::TOKS) {
                  // the value row's scale enters P (a stale scale past the item's tokens meets
                  // a zero weight and is dropped)
                  const float2 v2 =
                      SC_REG ? make_float2(vsc[32 * h + 2 * i], vsc[32 * h + 2 * i + 1])
                             : *reinterpret_cast<const float2*>(svs + c0 + 32 * h + 2 * i);
                  p0 = p0 == 0.f ? 0.f : p0 * v2.x;
                  p1 = p1 == 0.f ? 0.f : p1 * v2.y;
                }
                pk[i] = pack16x2<BF>(p0, p1);
              }
              tmem_st16u(t_sg + (c0 + 32 * h) / 2, pk);
            }
            lsum = ls2.x + ls2.y;
            if constexpr (DUAL) {
              uint32_t zk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) zk[i] = 0u;
              tmem_st16u(t_sg + (NL - c0) / 2, zk);
            }
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
          char* vt = smem + T::OFF_V + (g % T::NV) * T::SLOT;
          for (int e = stid; e < (SUB - nv) * T::NSLAB * 8; e += 128) {
            const int rr = nv + e / (T::NSLAB * 8), sl = (e / 8) % T::NSLAB, c = e & 7;
            *reinterpret_cast<uint4*>(vt + sl * T::KSLAB + sw128_chunk(rr, c)) =
                make_uint4(0, 0, 0, 0);
          }
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&p_full[g % NSP]);
          if constexpr (T::TOKS) mbar_arrive(&sc_free[g % T::NSC]);
        }
      }
      // ---- epilogue: O of this thread's row from tensor memory, in two halves of 64 dims
      list.wait_planner();  // nothing is written before the planner has finished
      wait_pv_step(g - 1);  // every PV of the item (in order)
      if (stid == 0) *cnt_seen_s = cnt_seen;
      named_barrier_sync(SOFT_BAR, 128);
      const bool fin = in_dec && slot == uinfo.x && *cnt_seen_s == uinfo.y - 1;
      const size_t orow = ((size_t)b * p.Sq + qi) * p.Hq + hq;
      // two streams: the second hands its O row, max and sum to the first through shared
      // memory, and the first merges them with its own (log-sum-exp rule)
      float w_own = 1.f, w_oth = 0.f;
      if constexpr (DUAL) {
        if (hs == 1) {
#pragma unroll 1
          for (int h = 0; h < D / 64; ++h) {
            float o[64];
            tmem_ld64(t_o + lane_off + 64 * h, o);
            float* row = mrg + qr * D;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int ch = 16 * h + c;  // 16-byte chunk of the row
              *reinterpret_cast<float4*>(row + 4 * (ch ^ (qr & 7))) =
                  make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            }
          }
          mrg_ml[2 * qr] = m_run;
          mrg_ml[2 * qr + 1] = l_run;
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_free);  // this warp has read its rows of O
        }
        named_barrier_sync(SOFT_BAR, 128);  // the second stream's rows are in shared memory
        if (hs == 0) {
          const float m2 = mrg_ml[2 * qr], l2 = mrg_ml[2 * qr + 1];
          const float mm = fmaxf(m_run, m2);
          w_own = m_run == -INFINITY ? 0.f : fast_exp2(m_run - mm);
          w_oth = m2 == -INFINITY ? 0.f : fast_exp2(m2 - mm);
          l_run = l_run * w_own + l2 * w_oth;
          m_run = mm;
        }
      }
      if (!DUAL || hs == 0) {
        float inv = l_run > 0.f ? vts / l_run : 0.f;
        float lse2 = l_run > 0.f ? m_run + fast_log2(l_run) : -INFINITY;
        // piece 0 finishing the unit: merged with pieces 1 .. ns-1 in the arithmetic of
        // merge_unit
        float mx = lse2, wown = 0.f, W = 0.f;
        if (fin && real) {
          for (int sp2 = 1; sp2 < uinfo.y; ++sp2)
            mx = fmaxf(mx, __ldcg(p.lse_part + (size_t)piece_slot(uinfo.x, sp2) * MP + qr));
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
          if constexpr (DUAL) {
            const float* row = mrg + qr * D;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int ch = 16 * h + c;
              const float4 q4 = *reinterpret_cast<const float4*>(row + 4 * (ch ^ (qr & 7)));
              o[4 * c] = o[4 * c] * w_own + q4.x * w_oth;
              o[4 * c + 1] = o[4 * c + 1] * w_own + q4.y * w_oth;
              o[4 * c + 2] = o[4 * c + 2] * w_own + q4.z * w_oth;
              o[4 * c + 3] = o[4 * c + 3] * w_own + q4.w * w_oth;
            }
          }
          float oinv = inv;
          if (fin) {
#pragma unroll
            for (int d = 0; d < 64; ++d) o[d] = wown == 0.f ? 0.f : __fmaf_rn(wown, o[d] * inv, 0.f);
            float Wh = 0.f + wown;
            for (int sp2 = 1; sp2 < uinfo.y; ++sp2) {
              const size_t part = (size_t)piece_slot(uinfo.x, sp2) * MP + qr;
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
            float4* op = reinterpret_cast<float4*>(p.o_part + ((size_t)slot * MP + qr) * D + 64 * h);
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
            p.lse_part[(size_t)slot * MP + qr] = lse2;
          }
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
  } else if (warp < T::W_CONV + T::NCW) {
    // ================================================================ fp8 widening
    if constexpr (T::FP8) {
      // step g: the e4m3 V rows of ring slot g % NV become the f16 rows of V buffer g % NSP
      // (rows past the item's tokens become zero); the scales are applied to the logits and
      // P, not here, and the K codes go to the MMA as they are
      const int ctid = tid - T::W_CONV * 32;  // 0 .. 32 NCW - 1
      // one operand: 64 rows of 128 e4m3 codes -> two slabs of 64 rows of 64 f16 values.
      // Lane l of a warp takes 16-byte chunk l % 8 of a row, so each group of eight lanes
      // reads one 128-byte row.  Every load is issued before the first conversion: the
      // compiler does not move a shared-memory load above a store to shared memory by
      // itself, and with one load, its conversions and its stores after another the
      // widening set the step's pace (measured: per-tensor fp8 Sq = 4 decode 94.8 us ->
      // 83.5 us; writing the second slab's two chunks in the opposite order, to spread the
      // stores over the banks, measured slower).
      auto widen = [&](const char* src, char* dst, int nv) {
        constexpr int NIT = SUB * 8 / (32 * T::NCW);
        uint4 w[NIT];
#pragma unroll
        for (int k = 0; k < NIT; ++k) {
          const int e = ctid + k * 32 * T::NCW;
          const int rr = e >> 3, c = e & 7;
          w[k] = rr < nv ? *reinterpret_cast<const uint4*>(src + sw128_chunk(rr, c))
                         : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < NIT; ++k) {
          const int e = ctid + k * 32 * T::NCW;
          const int rr = e >> 3, c = e & 7;
          const uint4 lo = make_uint4(e4m3x2_to_h2(w[k].x), e4m3x2_to_h2(w[k].x >> 16),
                                      e4m3x2_to_h2(w[k].y), e4m3x2_to_h2(w[k].y >> 16));
          const uint4 hi = make_uint4(e4m3x2_to_h2(w[k].z), e4m3x2_to_h2(w[k].z >> 16),
                                      e4m3x2_to_h2(w[k].w), e4m3x2_to_h2(w[k].w >> 16));
          // dims 16c .. 16c + 15 -> f16 slab c / 4, chunks 2 (c % 4) and 2 (c % 4) + 1
          char* d = dst + (c >> 2) * T::CV_SLAB;
          *reinterpret_cast<uint4*>(d + sw128_chunk(rr, 2 * (c & 3))) = lo;
          *reinterpret_cast<uint4*>(d + sw128_chunk(rr, 2 * (c & 3) + 1)) = hi;
        }
        fence_async_smem();
        __syncwarp();
      };
      uint32_t g = 0;
      ItemList list;
      list.init(p, first);
      int4 item;
      for (int it = 0; list.get(it, item); ++it) {
        const int t0 = item.y, t1 = item.z;
        if (t1 <= t0) continue;
        const int nsub = ceil_div(t1 - t0, SUB);
        for (int j = 0; j < nsub; ++j, ++g) {
          const int nv = min(SUB, t1 - (t0 + j * SUB));
          const int vslot = (int)(g % T::NV);
          // ---- V rows (buffer g % NSP is free once the PV of step g - NSP has completed)
          wait_bar(&full_v[vslot], (g / T::NV) & 1);
          if (g >= (uint32_t)NSP) {
            const uint32_t x = g - NSP;
            wait_bar(&pv_done[x % NSP], (x / NSP) & 1);
          }
          widen(smem + T::OFF_V + vslot * T::SLOT, smem + T::OFF_CV + (g % NSP) * T::CV_BUF, nv);
          if (lane == 0) {
            mbar_arrive(&cv_full[g % NSP]);
            mbar_arrive(&empty_v[vslot]);
          }
        }
      }
    }
  }

  // every thread past the planner (a role may have needed none of its list) before the
  // writes below
  grid_dependency_wait();
  grid_dependents_launch();
  tc_fence_before();
  __syncthreads();  // every role is done: no copy or MMA in flight
  if (warp >= T::W_SOFT && warp < T::W_CONV) {
    const int stid = tid - T::W_SOFT * 32;
    finish_pending<D, MP, QK, 4>(p, pend, reinterpret_cast<float*>(smem), T::SCRATCH / 4, mlbuf, stid);
    zero_empty_units<D, MP, QK, 128>(p, stid);
  }
  __syncthreads();
  if (tid == 0) {
    // a CTA whose first item was empty or absent checks it here
    if (*first_checked == 0) check_first(p.first_item[blockIdx.x]);
    if (*s_flags != 0) atomicOr(p.flags, *s_flags);
  }
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

}  // namespace pa
