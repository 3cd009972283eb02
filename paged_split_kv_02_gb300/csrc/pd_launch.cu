// Dispatch of a launch to the kernel instance of its head size.
#include "pd_internal.h"

namespace pd {

cudaError_t launch_mma_d64(bool, int, const CUtensorMap &, const CUtensorMap &, const Params &,
                           const Launch &, cudaStream_t);
cudaError_t launch_mma_d128(bool, int, const CUtensorMap &, const CUtensorMap &, const Params &,
                            const Launch &, cudaStream_t);
cudaError_t launch_mma_d256(bool, int, const CUtensorMap &, const CUtensorMap &, const Params &,
                            const Launch &, cudaStream_t);
cudaError_t launch_mma_d512(bool, int, const CUtensorMap &, const CUtensorMap &, const Params &,
                            const Launch &, cudaStream_t);

cudaError_t launch_mma(int D, bool bf16, int path, const CUtensorMap &tk, const CUtensorMap &tv,
                       const Params &p, const Launch &l, cudaStream_t stream) {
  switch (D) {
    case 64: return launch_mma_d64(bf16, path, tk, tv, p, l, stream);
    case 128: return launch_mma_d128(bf16, path, tk, tv, p, l, stream);
    case 256: return launch_mma_d256(bf16, path, tk, tv, p, l, stream);
    case 512: return launch_mma_d512(bf16, path, tk, tv, p, l, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pd
