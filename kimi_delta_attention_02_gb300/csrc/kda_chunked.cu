// kda_chunked.cu -- tensor-core chunkwise KDA prefill (bf16, d_k = d_v = 128).
#include "kda_common.cuh"

namespace kda {

bool chunked_supported(int, int, bool, float) { return false; }

kda_status launch_chunked(const void *, const void *, const void *, const float *, const float *, const int32_t *,
                          int, int64_t, int, bool, float, float, const float *, void *, float *, cudaStream_t) {
  return KDA_ERR_UNSUPPORTED;
}

}  // namespace kda
