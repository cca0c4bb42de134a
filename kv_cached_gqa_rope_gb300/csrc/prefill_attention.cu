// K4: causal GQA prefill attention (placeholder until the tcgen05 kernel lands).
#include <cuda_runtime.h>

#include "kvgqa_internal.h"

namespace kvgqa {

cudaError_t launch_prefill_attention(const PrefillParams& p, cudaStream_t stream) {
  (void)p;
  (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace kvgqa
