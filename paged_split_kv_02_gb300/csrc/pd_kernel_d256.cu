// Instantiation of the tensor-core decode kernel for head size 256.
#include "pd_kernel.cuh"

namespace pd {

cudaError_t launch_mma_d256(bool bf16, int path, const CUtensorMap &tk, const CUtensorMap &tv,
                           const Params &p, const Launch &l, cudaStream_t stream) {
  if (path == 5) return cudaErrorInvalidValue;  // tensor-memory prefill: head size 128
  if (path == 4) return cudaErrorInvalidValue;  // rows-on-M: head sizes up to 128
  if (path == 2)
    return bf16 ? launch_mma_t<256, true, false, true>(tk, tv, p, l, stream)
                : launch_mma_t<256, false, false, true>(tk, tv, p, l, stream);
  const bool tc = path == 3;
  if (tc)
    return bf16 ? launch_mma_t<256, true, true>(tk, tv, p, l, stream)
                : launch_mma_t<256, false, true>(tk, tv, p, l, stream);
  return bf16 ? launch_mma_t<256, true, false>(tk, tv, p, l, stream)
              : launch_mma_t<256, false, false>(tk, tv, p, l, stream);
}

}  // namespace pd
