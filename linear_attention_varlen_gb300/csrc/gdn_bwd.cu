// Backward kernels of the chunked Gated DeltaNet.
#include "gdn_bwd.h"

namespace gdn {

int launch_bwd(const BwdArgs& a, cudaStream_t stream, cudaEvent_t* events) {
  (void)a;
  (void)stream;
  (void)events;
  return kErrUnsupported;
}

}  // namespace gdn
