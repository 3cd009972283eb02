// Instantiation of the tensor-core decode kernel for head size 64.
#include "pd_kernel.cuh"

namespace pd {

cudaError_t launch_mma_d64(bool bf16, int path, const CUtensorMap &tk, const CUtensorMap &tv,
                           const Params &p, const Launch &l, cudaStream_t stream) {
  if (path == 5) return cudaErrorInvalidValue;  // tensor-memory prefill: head size 128
  if (path == 4)
    return bf16 ? launch_mma_t<64, true, false, false, true>(tk, tv, p, l, stream)
                : launch_mma_t<64, false, false, false, true>(tk, tv, p, l, stream);
  if (path == 2)
    return bf16 ? launch_mma_t<64, true, false, true>(tk, tv, p, l, stream)
                : launch_mma_t<64, false, false, true>(tk, tv, p, l, stream);
  const bool tc = path == 3;
  if (tc)
    return bf16 ? launch_mma_t<64, true, true>(tk, tv, p, l, stream)
                : launch_mma_t<64, false, true>(tk, tv, p, l, stream);
  return bf16 ? launch_mma_t<64, true, false>(tk, tv, p, l, stream)
              : launch_mma_t<64, false, false>(tk, tv, p, l, stream);
}

}  // namespace pd
