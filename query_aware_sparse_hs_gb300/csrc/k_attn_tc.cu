// Tensor-core (tcgen05) gather-attention: not built yet.
#include "hs_internal.h"

namespace hs {

bool attn_tc_supported(const KvView&) { return false; }

cudaError_t launch_attn_tc(const KvView&, const AttnArgs&, unsigned*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace hs
