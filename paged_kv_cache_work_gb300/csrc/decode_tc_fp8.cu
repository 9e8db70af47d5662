// tcgen05 decode kernel instances for fp8 (E4M3) caches: head dim 128, query tiles of 64 or
// 128 rows, widened to f16 in shared memory; per-tensor or no scales (false) and per-token
// scales (true).
#include "decode_tc.cuh"

namespace pa {

#define PA_TC_FP8_ALL(X)        \
  X(64, KV_FP8, Q_BF16, false)  \
  X(64, KV_FP8, Q_FP16, false)  \
  X(128, KV_FP8, Q_BF16, false) \
  X(128, KV_FP8, Q_FP16, false) \
  X(64, KV_FP8, Q_BF16, true)   \
  X(64, KV_FP8, Q_FP16, true)   \
  X(128, KV_FP8, Q_BF16, true)  \
  X(128, KV_FP8, Q_FP16, true)

cudaError_t launch_tc_fp8_d128(const KernelParams& prm, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, int grid, int mp, int qk, bool toks,
                               cudaStream_t s) {
#define PA_TC_CASE(MP_, KVK_, QK_, TOKS_)   \
  if (mp == MP_ && qk == QK_ && toks == TOKS_) \
    return launch_tc_instance<128, MP_, KVK_, QK_, TOKS_>(prm, kmap, vmap, grid, s);
  PA_TC_FP8_ALL(PA_TC_CASE)
#undef PA_TC_CASE
  return cudaErrorNotSupported;
}

}  // namespace pa
