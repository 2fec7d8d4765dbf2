// kda_chunked_gate.cu -- the chunkwise prefill kernels that write the output through the
// output gate with head-wise RMSNorm (Kimi K3 -- Architecture Notes, section 1.3). A
// translation unit of its own so that it compiles beside kda_chunked.cu.
#include "kda_chunked_kernel.cuh"

namespace kda {
namespace chunked {

KernelFn gate_kernel(bool out_bf16, bool gated) {
  constexpr int C = DECAY_CLAMPED, G = DECAY_GATED;
  return out_bf16 ? (gated ? kda_chunked_kernel<true, G, true> : kda_chunked_kernel<true, C, true>)
                  : (gated ? kda_chunked_kernel<false, G, true> : kda_chunked_kernel<false, C, true>);
}

}  // namespace chunked
}  // namespace kda
