// kda_recurrent.cu -- fp32 token-recurrent KDA prefill (reference-accuracy path).
//
// Runs the defining recurrence of Kimi K3 -- Architecture Notes, section 1.1,
// one token at a time, with the d_k x d_v state held in registers across the
// whole sequence:
//     S' = Diag(a_t) S,  y = S'^T k_t,  z = S'^T q_t,  u = b_t (v_t - y),
//     S  = S' + k_t u^T,  o_t = scale (z + u (k_t . q_t)).
// Every value column of S evolves independently, so a sequence-head chain is
// split into 32-column slices, one CTA each. In a CTA, warp w owns key rows
// 32w .. 32w+31 and lane l owns value column 32*slice + l; the reductions over
// key rows go through shared memory. Token t+1's inputs are fetched while
// token t is computed. It handles every supported shape and both dtypes; the
// tensor-core chunked kernels are the fast path for bf16, d = 128. The log-decay
// is either the clamped log_alpha input or, in the gated form (section 1.2),
// g = g_min * Sigmoid(e^{A_h} z) from decay logits z in the input dtype.
#include "kda_common.cuh"

namespace kda {

constexpr int kRecThreads = 128;  // 4 warps x 32 key rows
constexpr int kRecCols = 32;      // value columns per CTA

template <bool kInBF16, bool kOutBF16, bool kGated>
__global__ void __launch_bounds__(kRecThreads)
    kda_recurrent_kernel(const void *__restrict__ q, const void *__restrict__ k, const void *__restrict__ v,
                         const void *__restrict__ decay, const float *__restrict__ A_log,
                         const float *__restrict__ beta,
                         const int32_t *__restrict__ cu_seqlens, const float *__restrict__ init_state,
                         void *__restrict__ out, float *__restrict__ final_state, int H, int d_k, int d_v,
                         int n_slices, float lb, float scale) {
  __shared__ __align__(16) float s_k[2][128], s_q[2][128], s_a[2][128];
  __shared__ float s_v[2][kRecCols], s_b[2], s_kq[2][4];
  __shared__ float s_y[2][4][kRecCols], s_z[2][4][kRecCols];

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int slice = blockIdx.x % n_slices;
  const int64_t nh = blockIdx.x / n_slices;  // (sequence, head)
  const int h = int(nh % H);
  const int64_t n = nh / H;
  const int col = slice * kRecCols + lane;
  const bool col_ok = col < d_v;
  const int64_t bos = cu_seqlens[n], eos = cu_seqlens[n + 1];
  const float a_h = kGated ? __expf(A_log[h]) : 0.f;  // e^{A_h} of the gated form

  // state rows 32w + r of column `col`
  float S[32];
  const int64_t state_base = nh * int64_t(d_k) * d_v;
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const int c = 32 * w + r;
    S[r] = (init_state != nullptr && col_ok && c < d_k) ? init_state[state_base + int64_t(c) * d_v + col] : 0.f;
  }

  // prefetched inputs of the next token: thread tid holds channel tid
  float pk = 0.f, pq = 0.f, pla = 0.f, pv = 0.f, pb = 0.f;
  auto fetch = [&](int64_t t) {
    const int64_t base = (t * H + h);
    if (tid < d_k) {
      pk = load_elem<kInBF16>(k, base * d_k + tid);
      pq = load_elem<kInBF16>(q, base * d_k + tid);
      pla = kGated ? load_elem<kInBF16>(decay, base * d_k + tid)
                   : static_cast<const float *>(decay)[base * d_k + tid];
    }
    if (w == 0) pv = col_ok ? load_elem<kInBF16>(v, base * d_v + col) : 0.f;
    if (tid == 0) pb = beta[base];
  };
  if (bos < eos) fetch(bos);

  for (int64_t t = bos; t < eos; ++t) {
    const int buf = int((t - bos) & 1);
    // publish token t
    {
      const bool ch = tid < d_k;
      s_k[buf][tid] = ch ? pk : 0.f;
      s_q[buf][tid] = ch ? pq : 0.f;
      s_a[buf][tid] = ch ? __expf(kGated ? gated_log_decay(pla, a_h, lb) : clamp_log_decay(pla, lb)) : 0.f;
      float kq = ch ? pk * pq : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
      if (lane == 0) s_kq[buf][w] = kq;
      if (w == 0) s_v[buf][lane] = pv;
      if (tid == 0) s_b[buf] = pb;
    }
    __syncthreads();
    if (t + 1 < eos) fetch(t + 1);

    // decay own rows, partial y and z
    float y = 0.f, z = 0.f;
#pragma unroll
    for (int r4 = 0; r4 < 8; ++r4) {
      const float4 a4 = *reinterpret_cast<const float4 *>(&s_a[buf][32 * w + 4 * r4]);
      const float4 k4 = *reinterpret_cast<const float4 *>(&s_k[buf][32 * w + 4 * r4]);
      const float4 q4 = *reinterpret_cast<const float4 *>(&s_q[buf][32 * w + 4 * r4]);
      const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w},
                  qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float s = S[4 * r4 + e] * av[e];
        S[4 * r4 + e] = s;
        y = fmaf(s, kv[e], y);
        z = fmaf(s, qv[e], z);
      }
    }
    s_y[buf][w][lane] = y;
    s_z[buf][w][lane] = z;
    __syncthreads();

    const float yt = s_y[buf][0][lane] + s_y[buf][1][lane] + s_y[buf][2][lane] + s_y[buf][3][lane];
    const float zt = s_z[buf][0][lane] + s_z[buf][1][lane] + s_z[buf][2][lane] + s_z[buf][3][lane];
    const float kq = s_kq[buf][0] + s_kq[buf][1] + s_kq[buf][2] + s_kq[buf][3];
    const float u = s_b[buf] * (s_v[buf][lane] - yt);
#pragma unroll
    for (int r4 = 0; r4 < 8; ++r4) {
      const float4 k4 = *reinterpret_cast<const float4 *>(&s_k[buf][32 * w + 4 * r4]);
      S[4 * r4 + 0] = fmaf(k4.x, u, S[4 * r4 + 0]);
      S[4 * r4 + 1] = fmaf(k4.y, u, S[4 * r4 + 1]);
      S[4 * r4 + 2] = fmaf(k4.z, u, S[4 * r4 + 2]);
      S[4 * r4 + 3] = fmaf(k4.w, u, S[4 * r4 + 3]);
    }
    if (w == 0 && col_ok) store_elem<kOutBF16>(out, (t * H + h) * d_v + col, scale * fmaf(u, kq, zt));
  }

  if (final_state != nullptr && col_ok) {
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const int c = 32 * w + r;
      if (c < d_k) final_state[state_base + int64_t(c) * d_v + col] = S[r];
    }
  }
}

// decay: log_alpha (fp32) when A_log is null, else the gated form's logits z (input dtype)
cudaError_t launch_recurrent(const void *q, const void *k, const void *v, const void *decay, const float *A_log,
                             const float *beta, const int32_t *cu_seqlens, int num_seqs, int H, int d_k, int d_v,
                             bool in_bf16, bool out_bf16, float lb, float scale, const float *init_state,
                             void *out, float *final_state, cudaStream_t stream) {
  const int n_slices = (d_v + kRecCols - 1) / kRecCols;
  const dim3 grid(unsigned(int64_t(num_seqs) * H * n_slices)), block(kRecThreads);
  using Kern = decltype(&kda_recurrent_kernel<false, false, false>);
  static const Kern table[8] = {
      kda_recurrent_kernel<false, false, false>, kda_recurrent_kernel<false, false, true>,
      kda_recurrent_kernel<false, true, false>,  kda_recurrent_kernel<false, true, true>,
      kda_recurrent_kernel<true, false, false>,  kda_recurrent_kernel<true, false, true>,
      kda_recurrent_kernel<true, true, false>,   kda_recurrent_kernel<true, true, true>};
  const Kern kern = table[4 * int(in_bf16) + 2 * int(out_bf16) + int(A_log != nullptr)];
  kern<<<grid, block, 0, stream>>>(q, k, v, decay, A_log, beta, cu_seqlens, init_state, out, final_state, H, d_k,
                                   d_v, n_slices, lb, scale);
  return cudaGetLastError();
}

}  // namespace kda
