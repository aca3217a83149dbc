// Forward attention with the K/V reconstruction fused into the attention
// kernel (each CTA rebuilds its key/value tiles from the latent tile).
#include "internal.h"

namespace laga {

LaunchResult tc_attn_fwd_fused(const Dims&, const bf16*, const bf16*, const bf16*, const bf16*, const bf16*, bf16*,
                               float*, cudaStream_t) {
  LaunchResult r;
  r.err = cudaErrorNotSupported;
  r.what = "fused-reconstruction forward";
  return r;
}

}  // namespace laga
