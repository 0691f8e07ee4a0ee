// bf16 backward (placeholder until the tensor-core backward lands).
#include "fa_internal.h"

namespace fa {

cudaError_t launch_bwd_bf16(const BwdBf16Args&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace fa
