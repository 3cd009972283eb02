// Dispatch of a launch to the kernel instance of its head size.
#include "pd_internal.h"

namespace pd {

cudaError_t launch_mma_d64(bool, bool, const CUtensorMap &, const CUtensorMap &, const Params &,
                           const Launch &, cudaStream_t);
cudaError_t launch_mma_d128(bool, bool, const CUtensorMap &, const CUtensorMap &, const Params &,
                            const Launch &, cudaStream_t);
cudaError_t launch_mma_d256(bool, bool, const CUtensorMap &, const CUtensorMap &, const Params &,
                            const Launch &, cudaStream_t);
cudaError_t launch_mma_d512(bool, bool, const CUtensorMap &, const CUtensorMap &, const Params &,
                            const Launch &, cudaStream_t);

cudaError_t launch_mma(int D, bool bf16, bool tc, const CUtensorMap &tk, const CUtensorMap &tv,
                       const Params &p, const Launch &l, cudaStream_t stream) {
  switch (D) {
    case 64: return launch_mma_d64(bf16, tc, tk, tv, p, l, stream);
    case 128: return launch_mma_d128(bf16, tc, tk, tv, p, l, stream);
    case 256: return launch_mma_d256(bf16, tc, tk, tv, p, l, stream);
    case 512: return launch_mma_d512(bf16, tc, tk, tv, p, l, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pd
