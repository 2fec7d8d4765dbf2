// kda_chunked.cu -- host side of the tensor-core chunkwise prefill (the kernel is in
// kda_chunked_kernel.cuh): tensor maps, kernel choice and launch. The instantiations
// of the bounded maps without the output gate live here; those with it in
// kda_chunked_gate.cu and those of the unbounded map in kda_chunked_unbounded.cu, so that
// the three compile in parallel.
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_chunked_kernel.cuh"
#include "kda_tma_host.h"

namespace kda {
namespace chunked {

// kernel with the output gate (kda_chunked_gate.cu)
KernelFn gate_kernel(bool out_bf16, bool gated);
// kernel of the unbounded map (kda_chunked_unbounded.cu)
KernelFn unbounded_kernel(bool out_bf16, bool norm_gate);

KernelFn plain_kernel(bool out_bf16, bool gated) {
  constexpr int C = DECAY_CLAMPED, G = DECAY_GATED;
  return out_bf16 ? (gated ? kda_chunked_kernel<true, G, false> : kda_chunked_kernel<true, C, false>)
                  : (gated ? kda_chunked_kernel<false, G, false> : kda_chunked_kernel<false, C, false>);
}

}  // namespace chunked

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The chunked kernel's maps over [T, H, 128] tensors: boxes of 32 tokens x 64 channels (bf16,
// 128-byte swizzle: the MMA operands q, k, v) or 32 tokens x 128 channels without swizzle (the
// decay input: fp32 log_alpha or bf16 logits z; the output gate's bf16 logits; the output,
// bf16 or fp32, written by TMA stores).
bool make_map(CUtensorMap *map, const void *base, bool bf16, bool swizzled, int64_t T, int H) {
  return tensor_map_3d(map, base, bf16, T, H, chunked::kD, swizzled ? 64u : 128u, uint32_t(chunked::kC), swizzled);
}

}  // namespace

bool tensor_map_3d(CUtensorMap *map, const void *base, bool bf16, int64_t T, int H, int d, uint32_t box_d,
                   uint32_t box_t, bool swizzle128) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const uint64_t es = bf16 ? 2 : 4;
  const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(H), cuuint64_t(T)};
  const cuuint64_t strides[2] = {cuuint64_t(d) * es, cuuint64_t(H) * d * es};
  const cuuint32_t box[3] = {box_d, 1u, box_t};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                        const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Scratch of the parallel schedules (none yet: every chain runs in one CTA).
size_t prefill_workspace_bytes(int64_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v) {
  (void)total_tokens, (void)num_seqs, (void)H, (void)d_k, (void)d_v;
  return 0;
}

// The bounded maps need log-decay >= -5 (the clamp's or the gated map's lower bound); the
// unbounded map takes any decay.
bool chunked_supported(int d_k, int d_v, bool in_bf16, float lb, int decay_form) {
  return in_bf16 && d_k == chunked::kD && d_v == chunked::kD && (decay_form == DECAY_UNBOUNDED || lb >= -5.0f);
}

// decay: log_alpha (fp32) for DECAY_CLAMPED, else the bf16 logits z of the gated or the
// unbounded map, with A_log.
// out_gate: bf16 gate logits [T, H, 128] of the output gate, or null (out = o).
kda_status launch_chunked(const void *q, const void *k, const void *v, const void *decay, int decay_form,
                          const float *A_log, const float *beta, const int32_t *cu_seqlens, int num_seqs,
                          int64_t total_tokens, int H, bool out_bf16, float lb, float scale, const float *init_state,
                          const void *out_gate, const float *norm_weight, float norm_eps, void *out,
                          float *final_state, cudaStream_t stream) {
  const bool gated = decay_form != DECAY_CLAMPED, norm_gate = out_gate != nullptr;
  const bool unbounded = decay_form == DECAY_UNBOUNDED;
  CUtensorMap mq, mk, mv, mg, mr, mo;
  if (!make_map(&mq, q, true, true, total_tokens, H) || !make_map(&mk, k, true, true, total_tokens, H) ||
      !make_map(&mv, v, true, true, total_tokens, H) || !make_map(&mg, decay, gated, false, total_tokens, H))
    return KDA_ERR_CUDA;
  if (!make_map(&mo, out, out_bf16, false, total_tokens, H)) return KDA_ERR_CUDA;
  if (norm_gate) {
    if (!make_map(&mr, out_gate, true, false, total_tokens, H)) return KDA_ERR_CUDA;
  } else {
    mr = mg;  // not read
  }
  const chunked::OutGate og{static_cast<const uint16_t *>(out_gate), norm_weight, norm_eps};
  const chunked::KernelFn kern = unbounded   ? chunked::unbounded_kernel(out_bf16, norm_gate)
                                 : norm_gate ? chunked::gate_kernel(out_bf16, gated)
                                             : chunked::plain_kernel(out_bf16, gated);
  const uint32_t smem = unbounded ? chunked::smem_bytes<DECAY_UNBOUNDED>() : chunked::smem_bytes<DECAY_CLAMPED>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return KDA_ERR_CUDA;
  const dim3 grid(unsigned(int64_t(num_seqs) * H)), block(chunked::kThreads);
  kern<<<grid, block, smem, stream>>>(mq, mk, mv, mg, mr, mo, og, A_log, beta, cu_seqlens, init_state, out,
                                      final_state, H, lb, scale, device_error_word());
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
