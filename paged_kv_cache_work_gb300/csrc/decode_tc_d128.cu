// tcgen05 decode kernel instances (16-bit caches, head dim 128, query tiles of 64 or 128 rows).
#include "decode_tc.cuh"

namespace pa {

#define PA_TC_ALL(X)            \
  X(64, KV_BF16, Q_BF16, false)  \
  X(64, KV_FP16, Q_FP16, false)  \
  X(128, KV_BF16, Q_BF16, false) \
  X(128, KV_FP16, Q_FP16, false)

cudaError_t launch_tc_d128(const KernelParams& prm, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           int grid, int mp, int kvk, int qk, bool toks, cudaStream_t s) {
#define PA_TC_CASE(MP_, KVK_, QK_, TOKS_)                     \
  if (mp == MP_ && kvk == KVK_ && qk == QK_ && toks == TOKS_) \
    return launch_tc_instance<128, MP_, KVK_, QK_, TOKS_>(prm, kmap, vmap, grid, s);
  PA_TC_ALL(PA_TC_CASE)
#undef PA_TC_CASE
  return cudaErrorNotSupported;
}

}  // namespace pa
