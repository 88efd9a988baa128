// bf16 tensor-core path (placeholder: routes to the SIMT kernels until the
// tcgen05 kernels are in place).
#include "gdn_internal.h"

namespace gdn {
size_t tc_workspace_bytes(const Problem& p, int mode) { return simt_workspace_bytes(p, mode); }
int tc_forward(const Problem& p, void* ws, cudaStream_t st) { return simt_forward(p, ws, st); }
}  // namespace gdn
