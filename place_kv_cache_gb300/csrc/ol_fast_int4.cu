// ol_fast_int4.cu -- tensor-core decode attention over the INT4
// blockwise-affine cache (not yet built: the generic kernel serves INT4).
#include "ol_common.cuh"

namespace ol {

bool fast_int4_supported(const AttnParams&) { return false; }

cudaError_t launch_fast_int4(const AttnParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ol
