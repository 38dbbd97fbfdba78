// Tensor-core backward: not yet available; the SIMT backward serves bf16.
#include "common.h"

namespace st {
int launch_bwd_tc(const st_layout&, const BwdArgs&, void*, bool* handled) {
    *handled = false;
    return 0;
}
int bwd_tc_device_error(bool) { return 0; }
}  // namespace st
