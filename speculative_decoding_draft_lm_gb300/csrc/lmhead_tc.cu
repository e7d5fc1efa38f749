// Tensor-core LM-head (tcgen05 + TMA); placeholder until the kernel lands.
#include "internal.h"

namespace domino {
bool lmhead_tc_supported(const domino_ctx*) { return false; }
cudaError_t launch_lmhead_tc(domino_ctx*, RunArgs&) { return cudaErrorNotSupported; }
}  // namespace domino
