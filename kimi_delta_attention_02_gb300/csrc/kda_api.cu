// kda_api.cu -- the C ABI of libkda (declared in include/kda.h): argument
// validation on the host, dispatch to the kernels, the device error word.
#include <cmath>
#include <cstdint>

#include "kda_common.cuh"

#include <atomic>
#include <mutex>

namespace kda {

namespace {
__device__ uint32_t g_device_error = 0;
// what the last kda_check_device_error took out of g_device_error (read back by the host)
__device__ uint32_t g_device_error_taken = 0;
constexpr int kMaxDevices = 64;
std::atomic<uint32_t *> g_error_word[kMaxDevices];
std::mutex g_error_word_mu;
std::mutex g_check_mu;  // one kda_check_device_error at a time: they share g_device_error_taken

// Read and clear the error word in one step, behind the work already on the stream.
__global__ void take_device_error_kernel() { g_device_error_taken = atomicExch(&g_device_error, 0u); }
}  // namespace

uint32_t *device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  uint32_t *p = g_error_word[dev].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  std::lock_guard<std::mutex> lock(g_error_word_mu);
  p = g_error_word[dev].load(std::memory_order_relaxed);
  if (p == nullptr) {
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) return nullptr;
    p = static_cast<uint32_t *>(addr);
    g_error_word[dev].store(p, std::memory_order_release);
  }
  return p;
}

// ---------------------------------------------------------------------------------------------
// Scratch of kda_prefill_noalloc, for callers that cannot hand the library a workspace. It is a
// file-scope device array, so every GPU that loads this library holds these 16 MiB until the
// process exits. Host code may not use its name as a device address (on the host it names a
// stand-in): noalloc_scratch() looks the address up once per device, with that device current.
// ---------------------------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::atomic<void *> g_noalloc_ptr[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of g_noalloc_scratch on the current device (nullptr if the lookup failed). The
// first call on a device does the lookup, which may load the library's device code: it must not
// happen inside a stream capture.
void *noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void *p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  p = g_noalloc_ptr[dev].load(std::memory_order_relaxed);
  if (p == nullptr) {
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) return nullptr;
    p = addr;
    g_noalloc_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}
}  // namespace

// Each launcher takes the decay input as `decay` + `A_log`: log_alpha (fp32) with A_log null
// (the clamped form), or the gated form's logits z (input dtype) with A_log [H]; and the output
// gate as `out_gate` (gate logits, input dtype; null = plain read-out) + `norm_weight` + `norm_eps`.
cudaError_t launch_decode(const void *q, const void *k, const void *v, const void *decay, int decay_form,
                          const float *A_log, const float *beta, float *state, const void *out_gate,
                          const float *norm_weight, float norm_eps, const float *conv_w, void *conv_state,
                          float l2_eps, void *out, int B, int H, int d_k, int d_v, bool in_bf16, bool out_bf16,
                          float lb, float scale, cudaStream_t stream);
cudaError_t launch_prologue(const void *q_raw, const void *k_raw, const void *v_raw, const float *conv_w,
                            const int32_t *cu_seqlens, int num_seqs, int64_t total_tokens, int H, int d_k, int d_v,
                            bool bf16, const void *conv_init, float eps, void *q, void *k, void *v,
                            void *conv_final, cudaStream_t stream);
cudaError_t launch_recurrent(const void *q, const void *k, const void *v, const void *decay, int decay_form,
                             const float *A_log, const float *beta, const int32_t *cu_seqlens, int num_seqs, int H,
                             int d_k, int d_v, bool in_bf16, bool out_bf16, float lb, float scale,
                             const float *init_state, const void *out_gate, const float *norm_weight,
                             float norm_eps, void *out, float *final_state, cudaStream_t stream);
bool chunked_supported(int d_k, int d_v, bool in_bf16, float lb, int decay_form);
size_t prefill_workspace_bytes(int64_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v);
kda_status launch_chunked(const void *q, const void *k, const void *v, const void *decay, int decay_form,
                          const float *A_log, const float *beta, const int32_t *cu_seqlens, int num_seqs,
                          int64_t total_tokens, int H, bool out_bf16, float lb, float scale, const float *init_state,
                          const void *out_gate, const float *norm_weight, float norm_eps, void *out,
                          float *final_state, void *workspace, size_t workspace_bytes, cudaStream_t stream);

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool finite_nonneg(float x) { return x >= 0.f && x < INFINITY; }  // false for NaN

// whether the byte ranges [a, a + na) and [b, b + nb) intersect (null or empty never does)
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || !na || !nb) return false;
  const char *pa = static_cast<const char *>(a), *pb = static_cast<const char *>(b);
  return pa < pb + nb && pb < pa + na;
}

// decay: log_alpha (fp32) when A_log is null, else the gated form's logits z (in_dtype)
kda_status check_prefill_args(const void *q, const void *k, const void *v, const void *decay, const float *A_log,
                              const float *beta, const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                              int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype, kda_dtype out_dtype,
                              const float *init_state, const void *out, const float *final_state,
                              const void *out_gate = nullptr, const float *norm_weight = nullptr) {
  if (in_dtype != KDA_F32 && in_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (out_dtype != KDA_F32 && out_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_tokens < 0 || H < 1 || d_k < 1 || d_v < 1) return KDA_ERR_INVALID_ARG;
  if (d_k > 128 || d_v > 128) return KDA_ERR_UNSUPPORTED;
  if (total_tokens > INT32_MAX) return KDA_ERR_UNSUPPORTED;  // cu_seqlens are int32
  if (int64_t(num_seqs) * H > INT32_MAX / 4) return KDA_ERR_UNSUPPORTED;
  if (cu_seqlens == nullptr || !aligned4(cu_seqlens)) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0) {
    if (!q || !k || !v || !decay || !beta || !out) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(decay) || !aligned16(out) ||
        !aligned4(beta))
      return KDA_ERR_INVALID_ARG;
  }
  if (init_state && !aligned16(init_state)) return KDA_ERR_INVALID_ARG;
  if (final_state && !aligned16(final_state)) return KDA_ERR_INVALID_ARG;
  // outputs must not overlap the inputs (final_state == init_state is allowed)
  const size_t es = in_dtype == KDA_BF16 ? 2 : 4, eo = out_dtype == KDA_BF16 ? 2 : 4;
  const size_t nk = size_t(total_tokens) * H * d_k, nv = size_t(total_tokens) * H * d_v;
  const size_t ns = size_t(num_seqs) * H * d_k * d_v * 4;
  if (total_tokens > 0 && out_gate != nullptr && !aligned16(out_gate)) return KDA_ERR_INVALID_ARG;
  if (norm_weight != nullptr && !aligned4(norm_weight)) return KDA_ERR_INVALID_ARG;
  const void *ins[8] = {q, k, v, decay, beta, A_log, out_gate, norm_weight};
  const size_t in_bytes[8] = {nk * es, nk * es, nv * es, nk * (A_log ? es : 4), size_t(total_tokens) * H * 4,
                              A_log ? size_t(H) * 4 : 0, out_gate ? nv * es : 0,
                              norm_weight ? size_t(d_v) * 4 : 0};
  for (int i = 0; i < 8; ++i) {
    if (overlaps(out, nv * eo, ins[i], in_bytes[i])) return KDA_ERR_INVALID_ARG;
    if (overlaps(final_state, ns, ins[i], in_bytes[i])) return KDA_ERR_INVALID_ARG;
  }
  if (overlaps(out, nv * eo, init_state, ns) || overlaps(out, nv * eo, final_state, ns))
    return KDA_ERR_INVALID_ARG;
  if (final_state != init_state && overlaps(final_state, ns, init_state, ns)) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

// The workspace: NULL with 0 bytes, or a 16-byte-aligned device range that overlaps no tensor argument.
kda_status check_workspace(const void *ws, size_t ws_bytes, const void *q, const void *k, const void *v,
                           const void *decay, const float *A_log, const float *beta, const int32_t *cu_seqlens,
                           int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                           kda_dtype in_dtype, kda_dtype out_dtype, const float *init_state, const void *out,
                           const float *final_state, const void *out_gate, const float *norm_weight) {
  if (ws == nullptr) return ws_bytes == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
  if (ws_bytes == 0 || !aligned16(ws)) return KDA_ERR_INVALID_ARG;
  const size_t es = in_dtype == KDA_BF16 ? 2 : 4, eo = out_dtype == KDA_BF16 ? 2 : 4;
  const size_t nk = size_t(total_tokens) * H * d_k, nv = size_t(total_tokens) * H * d_v;
  const size_t ns = size_t(num_seqs) * H * d_k * d_v * 4;
  const void *args[12] = {q, k, v, decay, beta, A_log, out_gate, norm_weight, cu_seqlens, init_state, out,
                          final_state};
  const size_t bytes[12] = {nk * es, nk * es, nv * es, nk * (A_log ? es : 4), size_t(total_tokens) * H * 4,
                            A_log ? size_t(H) * 4 : 0, out_gate ? nv * es : 0, norm_weight ? size_t(d_v) * 4 : 0,
                            size_t(num_seqs + 1) * 4, init_state ? ns : 0, nv * eo, final_state ? ns : 0};
  for (int i = 0; i < 12; ++i)
    if (overlaps(ws, ws_bytes, args[i], bytes[i])) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

// the gated form's parameters: A_log [H] fp32 on the device, g_min finite and <= 0
kda_status check_gate_args(const float *A_log, float g_min) {
  if (A_log == nullptr || !aligned4(A_log)) return KDA_ERR_INVALID_ARG;
  if (!(g_min <= 0.f) || !(g_min > -INFINITY)) return KDA_ERR_INVALID_ARG;  // rejects NaN and -inf
  return KDA_OK;
}

// the output gate's parameters: the weight only with gate logits, eps finite and >= 0
kda_status check_out_gate_args(const void *out_gate, const float *norm_weight, float norm_eps) {
  if (out_gate == nullptr) return norm_weight == nullptr ? KDA_OK : KDA_ERR_INVALID_ARG;
  if (!(norm_eps >= 0.f) || !(norm_eps < INFINITY)) return KDA_ERR_INVALID_ARG;  // rejects NaN and inf
  return KDA_OK;
}

kda_status prefill_impl(const void *q, const void *k, const void *v, const void *decay, const float *A_log,
                        const float *beta, const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                        int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype, kda_dtype out_dtype, float lb,
                        float scale, const float *init_state, void *out, float *final_state, void *stream,
                        bool force_recurrent, const void *out_gate = nullptr, const float *norm_weight = nullptr,
                        float norm_eps = 0.f, int decay_form = -1, void *workspace = nullptr,
                        size_t workspace_bytes = 0) {
  if (decay_form < 0) decay_form = A_log != nullptr ? DECAY_GATED : DECAY_CLAMPED;
  kda_status st = check_out_gate_args(out_gate, norm_weight, norm_eps);
  if (st != KDA_OK) return st;
  st = check_prefill_args(q, k, v, decay, A_log, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype,
                          out_dtype, init_state, out, final_state, out_gate, norm_weight);
  if (st != KDA_OK) return st;
  st = check_workspace(workspace, workspace_bytes, q, k, v, decay, A_log, beta, cu_seqlens, num_seqs, total_tokens,
                       H, d_k, d_v, in_dtype, out_dtype, init_state, out, final_state, out_gate, norm_weight);
  if (st != KDA_OK) return st;
  if (num_seqs == 0) return KDA_OK;
  if (total_tokens == 0) out_gate = norm_weight = nullptr;  // nothing is read out
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the chunked kernels: bf16 inputs, d = 128; a bounded map with a lower bound >= -5, or the
  // unbounded map
  if (!force_recurrent && total_tokens > 0 && chunked_supported(d_k, d_v, in_dtype == KDA_BF16, lb, decay_form))
    return launch_chunked(q, k, v, decay, decay_form, A_log, beta, cu_seqlens, num_seqs, total_tokens, H,
                          out_dtype == KDA_BF16, lb, scale, init_state, out_gate, norm_weight, norm_eps, out,
                          final_state, workspace, workspace_bytes, s);
  const cudaError_t err = launch_recurrent(q, k, v, decay, decay_form, A_log, beta, cu_seqlens, num_seqs, H, d_k, d_v,
                                           in_dtype == KDA_BF16, out_dtype == KDA_BF16, lb, scale, init_state,
                                           out_gate, norm_weight, norm_eps, out, final_state, s);
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status decode_impl(const void *q, const void *k, const void *v, const void *decay, const float *A_log,
                       const float *beta, float *state, void *out, int32_t B, int32_t H, int32_t d_k, int32_t d_v,
                       kda_dtype in_dtype, kda_dtype out_dtype, float lb, float scale, void *stream,
                       const void *out_gate = nullptr, const float *norm_weight = nullptr, float norm_eps = 0.f,
                       const float *conv_weight = nullptr, void *conv_state = nullptr, float l2_eps = 0.f,
                       int decay_form = -1) {
  if (decay_form < 0) decay_form = A_log != nullptr ? DECAY_GATED : DECAY_CLAMPED;
  if (in_dtype != KDA_F32 && in_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (out_dtype != KDA_F32 && out_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || d_k < 1 || d_v < 1) return KDA_ERR_INVALID_ARG;
  if (d_k > 128 || d_v > 128 || (d_v & 3) != 0) return KDA_ERR_UNSUPPORTED;
  if (int64_t(B) * H > INT32_MAX) return KDA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !decay || !beta || !state || !out) return KDA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(decay) || !aligned16(state) ||
      !aligned16(out) || !aligned4(beta))
    return KDA_ERR_INVALID_ARG;
  const kda_status st = check_out_gate_args(out_gate, norm_weight, norm_eps);
  if (st != KDA_OK) return st;
  if ((out_gate && !aligned16(out_gate)) || (norm_weight && !aligned4(norm_weight))) return KDA_ERR_INVALID_ARG;
  {  // state (read and rewritten) and out (written) must not overlap each other or any input
    const size_t es = in_dtype == KDA_BF16 ? 2 : 4, eo = out_dtype == KDA_BF16 ? 2 : 4;
    const size_t nk = size_t(B) * H * d_k, nv = size_t(B) * H * d_v, ns = size_t(B) * H * d_k * d_v * 4;
    const void *ins[8] = {q, k, v, decay, beta, A_log, out_gate, norm_weight};
    const size_t in_bytes[8] = {nk * es, nk * es, nv * es, nk * (A_log ? es : 4), size_t(B) * H * 4,
                                A_log ? size_t(H) * 4 : 0, out_gate ? nv * es : 0, norm_weight ? size_t(d_v) * 4 : 0};
    for (int i = 0; i < 8; ++i)
      if (overlaps(state, ns, ins[i], in_bytes[i]) || overlaps(out, nv * eo, ins[i], in_bytes[i]))
        return KDA_ERR_INVALID_ARG;
    if (overlaps(out, nv * eo, state, ns)) return KDA_ERR_INVALID_ARG;
  }
  if (conv_state != nullptr) {  // the prologue: weights and state on the device, eps finite
    if (conv_weight == nullptr || !aligned16(conv_weight) || !aligned16(conv_state) || !finite_nonneg(l2_eps))
      return KDA_ERR_INVALID_ARG;
    const size_t es = in_dtype == KDA_BF16 ? 2 : 4, eo = out_dtype == KDA_BF16 ? 2 : 4;
    const size_t ncs = size_t(B) * H * 3 * (2 * d_k + d_v) * es;
    const size_t nk = size_t(B) * H * d_k, nv = size_t(B) * H * d_v;
    if (overlaps(conv_state, ncs, state, size_t(B) * H * d_k * d_v * 4) ||
        overlaps(conv_state, ncs, out, nv * eo) || overlaps(conv_state, ncs, q, nk * es) ||
        overlaps(conv_state, ncs, k, nk * es) || overlaps(conv_state, ncs, v, nv * es) ||
        overlaps(conv_state, ncs, conv_weight, size_t(H) * (2 * d_k + d_v) * 16) ||
        overlaps(state, size_t(B) * H * d_k * d_v * 4, conv_weight, size_t(H) * (2 * d_k + d_v) * 16) ||
        overlaps(out, nv * eo, conv_weight, size_t(H) * (2 * d_k + d_v) * 16))
      return KDA_ERR_INVALID_ARG;
  } else if (conv_weight != nullptr) {
    return KDA_ERR_INVALID_ARG;  // weights without a state
  }
  const cudaError_t err = launch_decode(q, k, v, decay, decay_form, A_log, beta, state, out_gate, norm_weight, norm_eps,
                                        conv_weight, conv_state, l2_eps, out, B, H, d_k, d_v, in_dtype == KDA_BF16,
                                        out_dtype == KDA_BF16, lb, scale, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// the decay form of a parameter block: the clamped form takes no A_log, the gated ones need it
// (the unbounded one has no bound to check)
kda_status check_decay_form(kda_decay_form form, const float *A_log, float bound) {
  if (form == KDA_DECAY_CLAMPED) return A_log == nullptr ? KDA_OK : KDA_ERR_INVALID_ARG;
  if (form == KDA_DECAY_GATED) return check_gate_args(A_log, bound);
  if (form == KDA_DECAY_UNBOUNDED) return (A_log != nullptr && aligned4(A_log)) ? KDA_OK : KDA_ERR_INVALID_ARG;
  return KDA_ERR_INVALID_ARG;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

kda_status kda_prefill_recurrent(const void *q, const void *k, const void *v, const float *log_alpha,
                                 const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                 int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype,
                                 kda_dtype out_dtype, float lower_bound, float scale, const float *init_state,
                                 void *out, float *final_state, void *stream) {
  return prefill_impl(q, k, v, log_alpha, nullptr, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype,
                      out_dtype, lower_bound, scale, init_state, out, final_state, stream, true);
}

kda_status kda_prefill(const void *q, const void *k, const void *v, const float *log_alpha, const float *beta,
                       const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                       int32_t d_v, kda_dtype in_dtype, kda_dtype out_dtype, float lower_bound, float scale,
                       const float *init_state, void *out, float *final_state, void *workspace,
                       size_t workspace_bytes, void *stream) {
  return prefill_impl(q, k, v, log_alpha, nullptr, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype,
                      out_dtype, lower_bound, scale, init_state, out, final_state, stream, false, nullptr, nullptr,
                      0.f, -1, workspace, workspace_bytes);
}

size_t kda_prefill_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v) {
  return prefill_workspace_bytes(total_tokens, num_seqs, H, d_k, d_v);
}

// kda_prefill with its scratch in g_noalloc_scratch instead of a caller's workspace: the same
// validation, schedule and kernels, and no allocation of any kind. Sizes whose schedule needs more
// scratch than the array holds are refused before anything is enqueued.
kda_status kda_prefill_noalloc(const void *q, const void *k, const void *v, const float *log_alpha,
                               const float *beta, const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                               int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype, kda_dtype out_dtype,
                               float lower_bound, float scale, const float *init_state, void *out,
                               float *final_state, void *stream) {
  const kda_status st = check_prefill_args(q, k, v, log_alpha, nullptr, beta, cu_seqlens, num_seqs, total_tokens, H,
                                           d_k, d_v, in_dtype, out_dtype, init_state, out, final_state);
  if (st != KDA_OK) return st;
  if (prefill_workspace_bytes(total_tokens, num_seqs, H, d_k, d_v) > kNoAllocScratchBytes) return KDA_ERR_UNSUPPORTED;
  void *scratch = noalloc_scratch();
  if (scratch == nullptr) return KDA_ERR_CUDA;
  return prefill_impl(q, k, v, log_alpha, nullptr, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype,
                      out_dtype, lower_bound, scale, init_state, out, final_state, stream, false, nullptr, nullptr,
                      0.f, -1, scratch, kNoAllocScratchBytes);
}

kda_status kda_prefill_gated(const void *q, const void *k, const void *v, const void *z, const float *A_log,
                             const float *beta, const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                             int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype, kda_dtype out_dtype,
                             float g_min, float scale, const float *init_state, void *out, float *final_state,
                             void *stream) {
  const kda_status st = check_gate_args(A_log, g_min);
  if (st != KDA_OK) return st;
  return prefill_impl(q, k, v, z, A_log, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype, out_dtype,
                      g_min, scale, init_state, out, final_state, stream, false);
}

kda_status kda_prefill_gated_recurrent(const void *q, const void *k, const void *v, const void *z,
                                       const float *A_log, const float *beta, const int32_t *cu_seqlens,
                                       int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                       kda_dtype in_dtype, kda_dtype out_dtype, float g_min, float scale,
                                       const float *init_state, void *out, float *final_state, void *stream) {
  const kda_status st = check_gate_args(A_log, g_min);
  if (st != KDA_OK) return st;
  return prefill_impl(q, k, v, z, A_log, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype, out_dtype,
                      g_min, scale, init_state, out, final_state, stream, true);
}

kda_status kda_decode(const void *q, const void *k, const void *v, const float *log_alpha, const float *beta,
                      float *state, void *out, int32_t B, int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype,
                      kda_dtype out_dtype, float lower_bound, float scale, void *stream) {
  return decode_impl(q, k, v, log_alpha, nullptr, beta, state, out, B, H, d_k, d_v, in_dtype, out_dtype,
                     lower_bound, scale, stream);
}

kda_status kda_decode_gated(const void *q, const void *k, const void *v, const void *z, const float *A_log,
                            const float *beta, float *state, void *out, int32_t B, int32_t H, int32_t d_k,
                            int32_t d_v, kda_dtype in_dtype, kda_dtype out_dtype, float g_min, float scale,
                            void *stream) {
  const kda_status st = check_gate_args(A_log, g_min);
  if (st != KDA_OK) return st;
  return decode_impl(q, k, v, z, A_log, beta, state, out, B, H, d_k, d_v, in_dtype, out_dtype, g_min, scale, stream);
}

kda_status kda_prefill_ex(const kda_prefill_params *p, void *stream) {
  if (p == nullptr || p->struct_size != sizeof(kda_prefill_params)) return KDA_ERR_INVALID_ARG;
  const kda_status st = check_decay_form(p->decay_form, p->A_log, p->decay_bound);
  if (st != KDA_OK) return st;
  return prefill_impl(p->q, p->k, p->v, p->decay, p->A_log, p->beta, p->cu_seqlens, p->num_seqs, p->total_tokens,
                      p->H, p->d_k, p->d_v, p->in_dtype, p->out_dtype, p->decay_bound, p->scale, p->init_state,
                      p->out, p->final_state, stream, p->force_recurrent != 0, p->out_gate, p->norm_weight,
                      p->norm_eps, int(p->decay_form), p->workspace, p->workspace_bytes);
}

kda_status kda_decode_ex(const kda_decode_params *p, void *stream) {
  if (p == nullptr || p->struct_size != sizeof(kda_decode_params)) return KDA_ERR_INVALID_ARG;
  const kda_status st = check_decay_form(p->decay_form, p->A_log, p->decay_bound);
  if (st != KDA_OK) return st;
  return decode_impl(p->q, p->k, p->v, p->decay, p->A_log, p->beta, p->state, p->out, p->B, p->H, p->d_k, p->d_v,
                     p->in_dtype, p->out_dtype, p->decay_bound, p->scale, stream, p->out_gate, p->norm_weight,
                     p->norm_eps, p->conv_weight, p->conv_state, p->l2_eps, int(p->decay_form));
}

kda_status kda_prologue(const void *q_raw, const void *k_raw, const void *v_raw, const float *conv_weight,
                        const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t d_k,
                        int32_t d_v, kda_dtype dtype, const void *conv_init, float l2_eps, void *q, void *k, void *v,
                        void *conv_final, void *stream) {
  if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_tokens < 0 || H < 1 || d_k < 1 || d_v < 1) return KDA_ERR_INVALID_ARG;
  if (d_k > 128 || d_v > 128) return KDA_ERR_UNSUPPORTED;
  if (total_tokens > INT32_MAX || H > 65535) return KDA_ERR_UNSUPPORTED;
  if (num_seqs == 0 && total_tokens > 0) return KDA_ERR_INVALID_ARG;
  if (!finite_nonneg(l2_eps)) return KDA_ERR_INVALID_ARG;
  if (cu_seqlens == nullptr || !aligned4(cu_seqlens)) return KDA_ERR_INVALID_ARG;
  if (conv_weight == nullptr || !aligned16(conv_weight)) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0) {
    if (!q_raw || !k_raw || !v_raw || !q || !k || !v) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q_raw) || !aligned16(k_raw) || !aligned16(v_raw) || !aligned16(q) || !aligned16(k) ||
        !aligned16(v))
      return KDA_ERR_INVALID_ARG;
  }
  if ((conv_init && !aligned16(conv_init)) || (conv_final && !aligned16(conv_final))) return KDA_ERR_INVALID_ARG;
  const size_t es = dtype == KDA_BF16 ? 2 : 4;
  const size_t nk = size_t(total_tokens) * H * d_k * es, nv = size_t(total_tokens) * H * d_v * es;
  const size_t ns = size_t(num_seqs) * H * 3 * (2 * d_k + d_v) * es;
  const void *ins[6] = {q_raw, k_raw, v_raw, conv_weight, cu_seqlens, conv_init};
  const size_t in_bytes[6] = {nk, nk, nv, size_t(H) * (2 * d_k + d_v) * 16, size_t(num_seqs + 1) * 4, ns};
  const void *outs[4] = {q, k, v, conv_final};
  const size_t out_bytes[4] = {nk, nk, nv, conv_final ? ns : 0};
  for (int o = 0; o < 4; ++o) {
    for (int i = 0; i < 6; ++i)
      if (overlaps(outs[o], out_bytes[o], ins[i], in_bytes[i])) return KDA_ERR_INVALID_ARG;
    for (int o2 = o + 1; o2 < 4; ++o2)
      if (overlaps(outs[o], out_bytes[o], outs[o2], out_bytes[o2])) return KDA_ERR_INVALID_ARG;
  }
  if (num_seqs == 0) return KDA_OK;
  const cudaError_t err = launch_prologue(q_raw, k_raw, v_raw, conv_weight, cu_seqlens, num_seqs, total_tokens, H,
                                          d_k, d_v, dtype == KDA_BF16, conv_init, l2_eps, q, k, v, conv_final,
                                          static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_check_device_error(void *stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_check_mu);
  take_device_error_kernel<<<1, 1, 0, s>>>();
  if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpyFromSymbolAsync(&word, g_device_error_taken, sizeof word, 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (word & (DEVERR_TMA_TIMEOUT | DEVERR_MMA_TIMEOUT)) return KDA_ERR_TIMEOUT;
  if (word & DEVERR_RANGE) return KDA_ERR_RANGE;
  return KDA_OK;
}

const char *kda_status_string(kda_status status) {
  switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    case KDA_ERR_RANGE: return "KDA_ERR_RANGE";
  }
  return "KDA_ERR_UNKNOWN";
}

int32_t kda_version(void) { return 100; }

}  // extern "C"
