// Placeholder until the tcgen05 LM-head kernel lands.
#include "sv_internal.h"

namespace sv {

size_t lmhead_workspace_bytes(int M, int H) { return 256 + (size_t)M * H * 2 + 256; }

int lmhead_launch(const void*, const void*, float, const void*, void*, sv_dtype, int, int, int,
                  void*, size_t, void*, std::string* err) {
  *err = "sv_lmhead_rmsnorm is not implemented in this build";
  return SV_ERR_UNSUPPORTED;
}

}  // namespace sv
