// Tensor-core (tcgen05) prefill.  Placeholder until the kernel lands: the
// scheduler asks prefill_tc_supported() and routes prefill work to the SIMT
// kernel while it answers false.
#include "common.cuh"
#include "rpa_internal.h"

namespace rpa {

bool prefill_tc_supported(int32_t, int32_t, int32_t) { return false; }

int prefill_ctas_per_sm(int32_t) { return 1; }

int prefill_tokens_per_block(int32_t, int32_t group) { return group >= 128 ? 1 : 128 / group; }

int launch_prefill_tc(const Plan&, const Args&, void*) {
  return static_cast<int>(cudaErrorNotSupported);
}

}  // namespace rpa
