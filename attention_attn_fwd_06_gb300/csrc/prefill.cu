// prefill.cu -- placeholder until the tcgen05 prefill kernel lands.
#include "kernels.h"

namespace attn {
cudaError_t launch_prefill(const PrefillLaunch&) { return cudaErrorNotSupported; }
}  // namespace attn
