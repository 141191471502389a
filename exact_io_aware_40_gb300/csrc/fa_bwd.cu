// fa_bwd.cu -- backward pass (placeholder until the tcgen05 kernel lands).
#include "kernels.h"

namespace fa {

cudaError_t launch_bwd(int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                       const CUtensorMap&, const BwdArgs&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace fa
