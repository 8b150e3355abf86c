// Tensor-core (tcgen05 / TMEM) tree-verify attention: not built yet.
#include "mt_internal.h"

namespace mt {
cudaError_t launch_verify_tc(const VerifyArgs&, int, cudaStream_t) { return cudaErrorNotSupported; }
int verify_tc_launches(int, int, int, int) { return 0; }
}  // namespace mt
