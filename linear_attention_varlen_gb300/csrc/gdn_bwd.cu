// Backward kernels of the chunked Gated DeltaNet.
#include "gdn_bwd.h"

namespace gdn {

int launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  (void)a;
  (void)stream;
  return kErrUnsupported;
}

}  // namespace gdn
