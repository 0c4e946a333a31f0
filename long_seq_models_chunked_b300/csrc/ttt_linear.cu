// Linear small-chunk path: not built yet.
#include "ttt_internal.h"

namespace ttt {
bool linear_supported(const ttt_cfg&) { return false; }
size_t linear_workspace_bytes(const ttt_cfg&) { return 0; }
int linear_run(const Call&) { return TTT_ERR_UNSUPPORTED; }
}  // namespace ttt
