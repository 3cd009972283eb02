// Instantiation of the tensor-core decode kernel for head size 128.
#include "pd_kernel.cuh"

namespace pd {

cudaError_t launch_mma_d128(bool bf16, int path, const CUtensorMap &tk, const CUtensorMap &tv,
                           const Params &p, const Launch &l, cudaStream_t stream) {
  if (path == 5)
    return bf16 ? launch_mma_t<128, true, false, false, false, true>(tk, tv, p, l, stream)
                : launch_mma_t<128, false, false, false, false, true>(tk, tv, p, l, stream);
  if (path == 4)
    return bf16 ? launch_mma_t<128, true, false, false, true>(tk, tv, p, l, stream)
                : launch_mma_t<128, false, false, false, true>(tk, tv, p, l, stream);
  if (path == 2)
    return bf16 ? launch_mma_t<128, true, false, true>(tk, tv, p, l, stream)
                : launch_mma_t<128, false, false, true>(tk, tv, p, l, stream);
  const bool tc = path == 3;
  if (tc)
    return bf16 ? launch_mma_t<128, true, true>(tk, tv, p, l, stream)
                : launch_mma_t<128, false, true>(tk, tv, p, l, stream);
  return bf16 ? launch_mma_t<128, true, false>(tk, tv, p, l, stream)
              : launch_mma_t<128, false, false>(tk, tv, p, l, stream);
}

}  // namespace pd
