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

cudaError_t launch_order_longest_first(const int32_t *cu_seqlens, int num_seqs, int32_t *order, cudaStream_t stream);
cudaError_t launch_segment_scan(const float *runs, float *states, const float *init_state, int H, int m,
                                cudaStream_t stream);

namespace {

// The schedules are planned for a GB300's 152 SMs (a fixed figure, so that the workspace query
// needs no device): one chunked CTA per SM.
constexpr int kPlanSMs = 152;
constexpr int64_t kMinSegTokens = 4096;  // shorter segments do not repay the extra passes
constexpr int kMaxOrderSeqs = 8192;      // the order kernel compares every pair of sequences
constexpr size_t kStateBytes = size_t(chunked::kD) * chunked::kD * 4;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Segmented schedule of ONE sequence of T tokens and H heads: m segments of L tokens (a multiple
// of the chunk length; the last one shorter). Pass 1 runs, per head, segment 0 from the initial
// state and, for segments 1 .. m-2, the segment from 0 (its B) and from I with v = 0 (its M):
// R = 2m - 3 runs (1 when m = 2). Pass 2 scans S_{s+1} = M_s S_s + B_s. Pass 3 runs all m
// segments from their entering states. m is the largest count whose passes each fit one CTA per
// SM with segments of at least kMinSegTokens; m = 0 means one CTA per head is used.
struct SegPlan {
  int m = 0, runs = 0;
  int64_t L = 0;
};
SegPlan seg_plan(int64_t T, int H) {
  SegPlan p;
  if (H < 1 || T <= 0) return p;
  for (int m = 2; 2 * m - 3 <= chunked::kMaxRuns && m <= chunked::kMaxRuns; ++m) {
    const int64_t runs = m == 2 ? 1 : 2 * m - 3;
    if (int64_t(H) * runs > kPlanSMs || int64_t(H) * m > kPlanSMs) break;
    const int64_t L = ((T + m - 1) / m + chunked::kC - 1) / chunked::kC * chunked::kC;
    if (L < kMinSegTokens || (m - 1) * L >= T) break;
    p.m = m;
    p.runs = int(runs);
    p.L = L;
  }
  return p;
}

// Workspace of the segmented schedule: the pass-1 run states (reused for the pass-3 final
// states, hence at least m slots), then the m entering states of pass 3; [slots, H, 128, 128] fp32.
size_t seg_runs_bytes(const SegPlan &p, int H) {
  return align256(size_t(p.runs > p.m ? p.runs : p.m) * size_t(H) * kStateBytes);
}
size_t seg_bytes(const SegPlan &p, int H) { return seg_runs_bytes(p, H) + align256(size_t(p.m) * H * kStateBytes); }

// Longest-first order of the sequences: worth it once there are more chains than SMs.
bool wants_order(int32_t num_seqs, int32_t H) {
  return num_seqs > 1 && num_seqs <= kMaxOrderSeqs && int64_t(num_seqs) * H > kPlanSMs;
}

}  // namespace

// Scratch of the parallel schedules for these sizes (0: none applies).
size_t prefill_workspace_bytes(int64_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v) {
  if (d_k != chunked::kD || d_v != chunked::kD || H < 1 || total_tokens <= 0) return 0;
  if (num_seqs == 1) {
    const SegPlan p = seg_plan(total_tokens, H);
    return p.m >= 2 ? seg_bytes(p, H) : 0;
  }
  return wants_order(num_seqs, H) ? align256(size_t(num_seqs) * 4) : 0;
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
                          float *final_state, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
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
  uint32_t *err_word = device_error_word();
  const dim3 block(chunked::kThreads);
  auto launch = [&](chunked::KernelFn fn, const chunked::Runs &runs, int64_t units, const float *init,
                    float *fin) {
    fn<<<dim3(unsigned(units * H)), block, smem, stream>>>(mq, mk, mv, mg, mr, mo, og, runs, A_log, beta, cu_seqlens,
                                                           init, out, fin, H, lb, scale, err_word);
    return cudaGetLastError() == cudaSuccess;
  };
  chunked::Runs runs{};
  const size_t need = prefill_workspace_bytes(total_tokens, num_seqs, H, chunked::kD, chunked::kD);
  if (workspace == nullptr || need == 0 || workspace_bytes < need)  // one CTA per (sequence, head)
    return launch(kern, runs, num_seqs, init_state, final_state) ? KDA_OK : KDA_ERR_CUDA;

  if (num_seqs > 1) {  // longest sequences first
    runs.order = static_cast<int32_t *>(workspace);
    if (launch_order_longest_first(cu_seqlens, num_seqs, static_cast<int32_t *>(workspace), stream) != cudaSuccess)
      return KDA_ERR_CUDA;
    return launch(kern, runs, num_seqs, init_state, final_state) ? KDA_OK : KDA_ERR_CUDA;
  }

  // One sequence in m segments (see seg_plan).
  const SegPlan p = seg_plan(total_tokens, H);
  float *run_states = static_cast<float *>(workspace);
  float *entry_states = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + seg_runs_bytes(p, H));
  // pass 1: segment 0 from the initial state, then B and M of segments 1 .. m-2; no output
  using namespace chunked;
  runs.count = p.runs;
  for (int r = 0; r < p.runs; ++r) {
    const int seg = r == 0 ? 0 : r <= p.m - 2 ? r : r - (p.m - 2);
    runs.bos[r] = int32_t(seg * p.L);
    runs.eos[r] = int32_t((seg + 1) * p.L);
    runs.flags[r] = RUN_NO_OUT | (r == 0 ? (init_state != nullptr ? 0u : RUN_INIT_ZERO)
                                  : r <= p.m - 2 ? RUN_INIT_ZERO : RUN_INIT_IDENTITY | RUN_ZERO_V);
  }
  const KernelFn state_kern = unbounded ? unbounded_kernel(out_bf16, false) : plain_kernel(out_bf16, gated);
  if (cudaFuncSetAttribute(state_kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (!launch(state_kern, runs, p.runs, init_state, run_states)) return KDA_ERR_CUDA;
  // pass 2: the entering state of every segment
  if (launch_segment_scan(run_states, entry_states, init_state, H, p.m, stream) != cudaSuccess) return KDA_ERR_CUDA;
  // pass 3: every segment from its entering state, with the outputs; final states over the runs
  runs.count = p.m;
  for (int s = 0; s < p.m; ++s) {
    runs.bos[s] = int32_t(s * p.L);
    runs.eos[s] = int32_t(s + 1 < p.m ? (s + 1) * p.L : total_tokens);
    runs.flags[s] = 0u;
  }
  if (!launch(kern, runs, p.m, entry_states, run_states)) return KDA_ERR_CUDA;
  if (final_state != nullptr &&
      cudaMemcpyAsync(final_state, run_states + size_t(p.m - 1) * H * kD * kD, size_t(H) * kStateBytes,
                      cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  return KDA_OK;
}

}  // namespace kda
