// kda_chunked_unbounded.cu -- the chunkwise prefill kernels of the unbounded decay map
// g = -e^{A_h} Softplus(z) (Kimi K3 -- Architecture Notes, section 1.2, the map of the
// earlier models), with and without the output gate. A translation unit of its own so that
// it compiles beside kda_chunked.cu and kda_chunked_gate.cu.
#include "kda_chunked_kernel.cuh"

namespace kda {
namespace chunked {

KernelFn unbounded_kernel(bool out_bf16, bool norm_gate) {
  constexpr int U = DECAY_UNBOUNDED;
  return out_bf16 ? (norm_gate ? kda_chunked_kernel<true, U, true> : kda_chunked_kernel<true, U, false>)
                  : (norm_gate ? kda_chunked_kernel<false, U, true> : kda_chunked_kernel<false, U, false>);
}

}  // namespace chunked
}  // namespace kda
