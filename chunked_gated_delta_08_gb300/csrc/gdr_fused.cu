// gdr_fused.cu -- the fused single-pass forward (placeholder until the
// tensor-core kernel lands): reports every request as unsupported so the
// dispatcher takes the chunked form.
#include "gdr_internal.h"

namespace gdr {

int run_fused(const gdr_desc &, const void *, const void *, const void *, const float *, const void *,
              const float *, const int64_t *, int, int, void *, float *, int *, cudaStream_t) {
  return GDR_ERR_UNSUPPORTED;
}

}  // namespace gdr
