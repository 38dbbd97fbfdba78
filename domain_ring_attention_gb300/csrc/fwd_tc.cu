// Tensor-core (tcgen05 + TMA) forward: placeholder until the kernel lands.
#include "common.h"

namespace st {
int launch_fwd_tc(const st_layout&, const AttnArgs&, void*, bool* handled) {
    *handled = false;
    return 0;
}
int launch_bwd_tc(const st_layout&, const BwdArgs&, void*, bool* handled) {
    *handled = false;
    return 0;
}
}  // namespace st
