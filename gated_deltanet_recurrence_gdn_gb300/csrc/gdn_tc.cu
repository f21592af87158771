// gdn_tc.cu -- tcgen05 tensor-core path (bf16 I/O, fp32 state).
#include "gdn_internal.h"

namespace gdn {

bool tc_supported(const FwdArgs &) { return false; }

gdn_status tc_forward(const FwdArgs &) { return GDN_ERR_UNSUPPORTED; }

}  // namespace gdn
