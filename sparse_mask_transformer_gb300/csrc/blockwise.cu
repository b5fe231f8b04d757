// Block-wise masked attention kernel (tcgen05 / TMEM / TMA).  Placeholder
// until the kernel lands: reports the configuration as unsupported.
#include "internal.h"

namespace stof {
stof_status launch_blockwise(const AttnParams&, bool, cudaStream_t) { return STOF_ERR_UNSUPPORTED; }
}  // namespace stof
