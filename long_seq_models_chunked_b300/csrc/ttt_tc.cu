// Tensor-core (tcgen05) bf16 path: not built yet.
#include "ttt_internal.h"

namespace ttt {
bool tc_supported(const ttt_cfg&) { return false; }
size_t tc_workspace_bytes(const ttt_cfg&) { return 0; }
int tc_run(const Call&) { return TTT_ERR_UNSUPPORTED; }
}  // namespace ttt
