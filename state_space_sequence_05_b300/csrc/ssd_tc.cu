// ssd_tc.cu -- tcgen05 tensor-core SSD forward (bf16 inputs).
#include "ssd_internal.h"

namespace ssd {

bool tc_supported(const FwdArgs&) { return false; }
size_t tc_workspace_bytes(const FwdArgs&) { return 0; }
ssd_status_t tc_forward(const FwdArgs&) { return SSD_ERR_UNSUPPORTED; }

}  // namespace ssd
