// decode_hq2b.cu -- split-K decode attention over 2-bit pages (placeholder: generic kernel).
#include "kvq_internal.cuh"
#include "attn_args.cuh"

namespace kvq {
int launch_attn_generic(int fmt, const AttnArgs& a, int decode, cudaStream_t stream);

int launch_decode_hq2b(const AttnArgs& a, cudaStream_t stream) {
  return launch_attn_generic(KVQ_FMT_HQ2B, a, 1, stream);
}
}  // namespace kvq
