// Chunked prefill (WY / UT-transform form on tensor cores).
#include "gdn_common.cuh"
#include "gdn_launch.h"

namespace gdn {

size_t prefill_workspace_bytes(int, int, int, int, int, int) { return 0; }

int launch_prefill(const void*, const void*, const void*, bool, const float*, const float*, int,
                   int, int, int, int, int, float*, float*, void*, cudaStream_t) {
  return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn
