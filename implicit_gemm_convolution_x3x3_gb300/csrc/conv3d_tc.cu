// Tensor-core (tcgen05) conv3d path -- placeholder until the kernel lands.
#include "ig3_internal.h"

namespace ig3 {

const char* conv3d_tc_unsupported_reason(int, int, int, int, int, int, int) {
  return "the tensor-core conv3d kernel is not built in this version";
}

size_t conv3d_tc_workspace(const Conv3dArgs&) { return 0; }

int conv3d_tc_launch(const Conv3dArgs&) {
  return fail(IG3_ERR_UNSUPPORTED, "%s", conv3d_tc_unsupported_reason(0, 0, 0, 0, 0, 0, 0));
}

}  // namespace ig3
