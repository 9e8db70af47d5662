// CUDA-core decode kernel instances for head dim 128 (one translation unit per head dim
// so the instances compile in parallel).
#include "decode_simt.cuh"

namespace pa {

cudaError_t launch_simt_d128(const KernelParams& prm, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           int grid, int mp, int kvk, int qk, bool toks, cudaStream_t s) {
  return launch_simt_for_dim<128>(prm, kmap, vmap, grid, mp, kvk, qk, toks, s);
}

int simt_ctas_per_sm_d128(int mp, int kvk, bool toks) {
  return simt_ctas_per_sm_for_dim<128>(mp, kvk, toks);
}

}  // namespace pa
