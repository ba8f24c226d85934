// Expert FFN for prefill chunks (large T).
#include "internal.cuh"

namespace ds4 {

cudaError_t launch_ffn_prefill(const FfnArgs &a, cudaStream_t s) {
  // Same bucketed per-expert kernels as decode; each expert's token list is
  // processed in passes.
  return launch_ffn_decode(a, s);
}

}  // namespace ds4
