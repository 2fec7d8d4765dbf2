// kda_recurrent.cu -- fp32 token-recurrent KDA prefill (reference-accuracy path).
//
// Runs the defining recurrence of Kimi K3 -- Architecture Notes, section 1.1,
// one token at a time, with the d_k x d_v state held in registers across the
// whole sequence:
//     S' = Diag(a_t) S,  y = S'^T k_t,  z = S'^T q_t,  u = b_t (v_t - y),
//     S  = S' + k_t u^T,  o_t = scale (z + u (k_t . q_t)).
// Every value column of S evolves independently, so a sequence-head chain is
// split into slices of 32 kCG value columns, one CTA each. In a CTA, warp w owns
// key rows 32 (w % 4) .. + 31 of column group w / 4, and lane l owns value column
// 32 (kCG slice + w / 4) + l; the reductions over key rows go through shared
// memory. Token t+1's inputs are fetched while token t is computed. It handles
// every supported shape and both dtypes; the tensor-core chunked kernels are the
// fast path for bf16, d = 128. The log-decay is the clamped log_alpha input, or, in
// the gated form (section 1.2), g = g_min * Sigmoid(e^{A_h} z) from decay logits z in
// the input dtype, or the unbounded g = -e^{A_h} Softplus(z) of the earlier models,
// which only this kernel and decode accept (the chunked kernels need the bound).
//
// With the output gate of section 1.3 a CTA holds all value columns of its chain
// (kCG = 4, 16 warps), so that the RMS of a token's read-out over its d_v channels
// is a sum over the four column groups' warps in shared memory.
#include "kda_common.cuh"

namespace kda {

constexpr int kRecCols = 32;  // value columns per column group

template <bool kInBF16, bool kOutBF16, int kDecay, bool kNormGate>
__global__ void __launch_bounds__(kNormGate ? 512 : 128)
    kda_recurrent_kernel(const void *__restrict__ q, const void *__restrict__ k, const void *__restrict__ v,
                         const void *__restrict__ decay, const float *__restrict__ A_log,
                         const float *__restrict__ beta,
                         const int32_t *__restrict__ cu_seqlens, const float *__restrict__ init_state,
                         const void *__restrict__ out_gate, const float *__restrict__ norm_weight, float norm_eps,
                         void *__restrict__ out, float *__restrict__ final_state, int H, int d_k, int d_v,
                         int n_slices, float lb, float scale) {
  constexpr int kCG = kNormGate ? 4 : 1;  // column groups per CTA
  constexpr int kCols = kCG * kRecCols;
  __shared__ __align__(16) float s_k[2][128], s_q[2][128], s_a[2][128];
  __shared__ float s_v[2][kCols], s_b[2], s_kq[2][4];
  __shared__ float s_y[2][4][kCols], s_z[2][4][kCols];
  __shared__ float s_ss[2][kCG];

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int rg = w & 3, cg = w >> 2;  // key-row group, column group
  const int slice = blockIdx.x % n_slices;
  const int64_t nh = blockIdx.x / n_slices;  // (sequence, head)
  const int h = int(nh % H);
  const int64_t n = nh / H;
  const int lc = cg * kRecCols + lane;  // column within the CTA
  const int col = slice * kCols + lc;
  const bool col_ok = col < d_v;
  const int64_t bos = cu_seqlens[n], eos = cu_seqlens[n + 1];
  constexpr bool kGated = kDecay != DECAY_CLAMPED;   // log-decay from logits z
  const float a_h = kGated ? __expf(A_log[h]) : 0.f;  // e^{A_h} of the gated forms
  const float w_norm = (kNormGate && norm_weight != nullptr && col_ok) ? norm_weight[col] : 1.f;

  // state rows 32 rg + r of column `col`
  float S[32];
  const int64_t state_base = nh * int64_t(d_k) * d_v;
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const int c = 32 * rg + r;
    S[r] = (init_state != nullptr && col_ok && c < d_k) ? init_state[state_base + int64_t(c) * d_v + col] : 0.f;
  }

  // prefetched inputs of the next token: thread tid < 128 holds channel tid
  float pk = 0.f, pq = 0.f, pla = 0.f, pv = 0.f, pb = 0.f, pr = 0.f;
  auto fetch = [&](int64_t t) {
    const int64_t base = (t * H + h);
    if (tid < d_k) {
      pk = load_elem<kInBF16>(k, base * d_k + tid);
      pq = load_elem<kInBF16>(q, base * d_k + tid);
      pla = kGated ? load_elem<kInBF16>(decay, base * d_k + tid)
                   : static_cast<const float *>(decay)[base * d_k + tid];
    }
    if (rg == 0) {
      pv = col_ok ? load_elem<kInBF16>(v, base * d_v + col) : 0.f;
      if (kNormGate) pr = col_ok ? load_elem<kInBF16>(out_gate, base * d_v + col) : 0.f;
    }
    if (tid == 0) pb = beta[base];
  };
  if (bos < eos) fetch(bos);

  for (int64_t t = bos; t < eos; ++t) {
    const int buf = int((t - bos) & 1);
    const float r_gate = pr;
    // publish token t
    if (tid < 128) {
      const bool ch = tid < d_k;
      s_k[buf][tid] = ch ? pk : 0.f;
      s_q[buf][tid] = ch ? pq : 0.f;
      s_a[buf][tid] = ch ? __expf(kDecay == DECAY_UNBOUNDED ? unbounded_log_decay(pla, a_h)
                                  : kDecay == DECAY_GATED   ? gated_log_decay(pla, a_h, lb)
                                                            : clamp_log_decay(pla, lb))
                         : 0.f;
      float kq = ch ? pk * pq : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
      if (lane == 0) s_kq[buf][w] = kq;
    }
    if (rg == 0) s_v[buf][lc] = pv;
    if (tid == 0) s_b[buf] = pb;
    __syncthreads();
    if (t + 1 < eos) fetch(t + 1);

    // decay own rows, partial y and z
    float y = 0.f, z = 0.f;
#pragma unroll
    for (int r4 = 0; r4 < 8; ++r4) {
      const float4 a4 = *reinterpret_cast<const float4 *>(&s_a[buf][32 * rg + 4 * r4]);
      const float4 k4 = *reinterpret_cast<const float4 *>(&s_k[buf][32 * rg + 4 * r4]);
      const float4 q4 = *reinterpret_cast<const float4 *>(&s_q[buf][32 * rg + 4 * r4]);
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
    s_y[buf][rg][lc] = y;
    s_z[buf][rg][lc] = z;
    __syncthreads();

    const float yt = s_y[buf][0][lc] + s_y[buf][1][lc] + s_y[buf][2][lc] + s_y[buf][3][lc];
    const float zt = s_z[buf][0][lc] + s_z[buf][1][lc] + s_z[buf][2][lc] + s_z[buf][3][lc];
    const float kq = s_kq[buf][0] + s_kq[buf][1] + s_kq[buf][2] + s_kq[buf][3];
    const float u = s_b[buf] * (s_v[buf][lc] - yt);
#pragma unroll
    for (int r4 = 0; r4 < 8; ++r4) {
      const float4 k4 = *reinterpret_cast<const float4 *>(&s_k[buf][32 * rg + 4 * r4]);
      S[4 * r4 + 0] = fmaf(k4.x, u, S[4 * r4 + 0]);
      S[4 * r4 + 1] = fmaf(k4.y, u, S[4 * r4 + 1]);
      S[4 * r4 + 2] = fmaf(k4.z, u, S[4 * r4 + 2]);
      S[4 * r4 + 3] = fmaf(k4.w, u, S[4 * r4 + 3]);
    }
    if (rg == 0) {
      const float o = col_ok ? scale * fmaf(u, kq, zt) : 0.f;
      if constexpr (kNormGate) {
        // RMS over the d_v channels: the 4 column-group warps meet on barrier 1
        float ss = o * o;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) s_ss[buf][cg] = ss;
        named_bar_sync(1, 128);
        const float rstd = rsqrtf(((s_ss[buf][0] + s_ss[buf][1]) + (s_ss[buf][2] + s_ss[buf][3])) / float(d_v) +
                                  norm_eps);
        if (col_ok) store_elem<kOutBF16>(out, (t * H + h) * d_v + col, output_gate(o, rstd, w_norm, r_gate));
      } else if (col_ok) {
        store_elem<kOutBF16>(out, (t * H + h) * d_v + col, o);
      }
    }
  }

  if (final_state != nullptr && col_ok) {
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const int c = 32 * rg + r;
      if (c < d_k) final_state[state_base + int64_t(c) * d_v + col] = S[r];
    }
  }
}

// decay: log_alpha (fp32) for DECAY_CLAMPED, else the gated forms' logits z (input dtype) with A_log.
// out_gate: gate logits [T, H, d_v] (input dtype) of the output gate, or null (out = o).
cudaError_t launch_recurrent(const void *q, const void *k, const void *v, const void *decay, int decay_form,
                             const float *A_log, const float *beta, const int32_t *cu_seqlens, int num_seqs, int H,
                             int d_k, int d_v, bool in_bf16, bool out_bf16, float lb, float scale,
                             const float *init_state, const void *out_gate, const float *norm_weight,
                             float norm_eps, void *out, float *final_state, cudaStream_t stream) {
  const bool norm_gate = out_gate != nullptr;
  const int cols = norm_gate ? 4 * kRecCols : kRecCols;
  const int n_slices = (d_v + cols - 1) / cols;
  const dim3 grid(unsigned(int64_t(num_seqs) * H * n_slices)), block(norm_gate ? 512 : 128);
  using Kern = decltype(&kda_recurrent_kernel<false, false, 0, false>);
#define KDA_REC_ROW(ib, ob, ng) \
  kda_recurrent_kernel<ib, ob, 0, ng>, kda_recurrent_kernel<ib, ob, 1, ng>, kda_recurrent_kernel<ib, ob, 2, ng>
#define KDA_REC_BLOCK(ng) \
  KDA_REC_ROW(false, false, ng), KDA_REC_ROW(false, true, ng), KDA_REC_ROW(true, false, ng), KDA_REC_ROW(true, true, ng)
  static const Kern table[24] = {KDA_REC_BLOCK(false), KDA_REC_BLOCK(true)};
#undef KDA_REC_BLOCK
#undef KDA_REC_ROW
  const Kern kern = table[12 * int(norm_gate) + 6 * int(in_bf16) + 3 * int(out_bf16) + decay_form];
  kern<<<grid, block, 0, stream>>>(q, k, v, decay, A_log, beta, cu_seqlens, init_state, out_gate, norm_weight,
                                   norm_eps, out, final_state, H, d_k, d_v, n_slices, lb, scale);
  return cudaGetLastError();
}

}  // namespace kda
