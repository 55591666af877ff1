// kernels_tc.cu -- tcgen05 tensor-core paths (3xTF32 and TF32).
#include "../../include/sgemm.h"
#include "internal.h"

namespace sg {

int launch_tc(Plan &plan)
{
    (void)plan;
    return SGEMM_ERR_UNSUPPORTED;
}

}  // namespace sg
