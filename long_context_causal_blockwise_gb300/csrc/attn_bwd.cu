// Backward kernels (placeholder until the dK/dV and dQ passes land).
#include "lcb_internal.h"

namespace lcb {
int launch_attn_bwd_dkdv(const BwdLaunch&, cudaStream_t) { return -2; }
int launch_attn_bwd_dq(const BwdLaunch&, cudaStream_t) { return -2; }
}  // namespace lcb
