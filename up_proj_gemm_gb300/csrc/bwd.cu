// Backward kernels (dgrad, wgrad + bias gradient): placeholder until written.
#include "internal.h"

namespace mlaq {
int launch_dgrad(const BwdArgs&, cudaStream_t) { return MLA_ERR_UNSUPPORTED; }
int launch_wgrad(const BwdArgs&, cudaStream_t) { return MLA_ERR_UNSUPPORTED; }
}  // namespace mlaq
