// Instantiation of the tensor-core decode kernel for head size 512.
#include "pd_kernel.cuh"

namespace pd {

cudaError_t launch_mma_d512(bool bf16, int path, const CUtensorMap &tk, const CUtensorMap &tv,
                           const Params &p, const Launch &l, cudaStream_t stream) {
  // the tensor-memory path needs 2 x 16 + 512 columns: more than one SM has;
  // the warp dot-product path keeps head sizes up to 256
  if (path != 1) return cudaErrorInvalidValue;
  return bf16 ? launch_mma_t<512, true, false>(tk, tv, p, l, stream)
              : launch_mma_t<512, false, false>(tk, tv, p, l, stream);
}

}  // namespace pd
