// kda_decode.cu -- one-token KDA decode step, state updated in place.
//
// Kimi K3 -- Architecture Notes, section 1.1: S_t = (I - b k k^T) Diag(a) S_{t-1}
// + b k v^T, o_t = S_t^T q. With D = Diag(a) and S' = D S_{t-1} this is
//     y = S'^T k,   z = S'^T q,   u = b (v - y),
//     S_t = S' + k u^T,           o = scale (z + u (k . q)),
// one read and one write of the d_k x d_v fp32 state per (sequence, head): the
// step is bound by HBM bandwidth (about 0.86 flop per byte).
//
// One CTA of 256 threads per (sequence, head). Thread (ty, tx) owns value
// columns 4tx..4tx+3 of key rows ty, ty+8, ..., ty+120: every state access is a
// 128-bit copy or store and each warp touches whole 512-byte rows, so the state
// streams through HBM fully coalesced. The state comes into shared memory by
// cp.async (16 copies per thread, issued before anything waits on them), so that
// it takes no registers: 80 registers and 72 KB of shared memory per CTA let
// three CTAs share an SM. The log-decay is either the clamped log_alpha
// input or, in the gated form (section 1.2), g = g_min * Sigmoid(e^{A_h} z).
// Optionally the read-out goes through the output gate of section 1.3,
// Sigmoid(r) * w * o / rms(o), before it is written: warp 0 holds the whole d_v
// row, so the RMS is one warp reduction. Optionally the token's raw q, k, v first
// pass the prologue of section 1.1 (4-tap short convolution over the sequence's
// convolution state, which is shifted in place, then Swish, then the L2 norm of q
// and k): the conv state adds 3 x (2 d_k + d_v) values per (sequence, head).
#include <atomic>

#include "kda_common.cuh"

namespace kda {

constexpr int kDecodeThreads = 256;
constexpr int kDecodeRowsPerThread = 16;  // 128 key rows / 8 row groups

// The prologue's parameters: conv weights [H, 2 d_k + d_v, 4] fp32, the conv state
// [B, H, 3, 2 d_k + d_v] (input dtype, read and shifted in place) and the L2 norm's eps.
struct Prologue {
  const float *w;
  void *state;
  float eps;
};

template <bool kInBF16, bool kOutBF16, int kDecay, bool kNormGate, bool kPrologue>
__global__ void __launch_bounds__(kDecodeThreads, 3)
    kda_decode_kernel(const void *__restrict__ q, const void *__restrict__ k, const void *__restrict__ v,
                      const void *__restrict__ decay, const float *__restrict__ A_log,
                      const float *__restrict__ beta, float *__restrict__ state, const void *__restrict__ out_gate,
                      const float *__restrict__ norm_weight, float norm_eps, const Prologue pro,
                      void *__restrict__ out, int H, int d_k, int d_v, float lb, float scale) {
  __shared__ float s_k[128], s_q[128], s_a[128], s_v[128];
  __shared__ float s_red_y[8][128], s_red_z[8][128];
  __shared__ float s_kq[8], s_nrm[2][4];

  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int64_t bh = blockIdx.x;  // (sequence, head) pair, head fastest
  const int64_t vec_base = bh * d_k;
  float *S = state + bh * int64_t(d_k) * d_v;
  const int col = 4 * tx;
  const bool col_ok = col < d_v;

  // The state goes into shared memory (cp.async, L2 only; rows or columns past d_k, d_v read
  // as zeros), so that it holds no registers and three CTAs fit on an SM. Where the copies
  // are issued was measured per form: after the token loads when the prologue feeds a
  // logit-mapped decay (0.51 against 0.56 ms for B=256, H=96), before them otherwise (with
  // the prologue and the clamped decay 0.54 against 0.71 ms; with the output gate 0.47
  // against 0.49 ms).
  constexpr bool kTokensFirst = kPrologue && kDecay != DECAY_CLAMPED;
  extern __shared__ __align__(16) float s_st[];  // [128 key rows][128 value columns]
  auto issue_state_copies = [&]() {
#pragma unroll
    for (int j = 0; j < kDecodeRowsPerThread; ++j) {
      const int c = ty + 8 * j;
      const bool ok = col_ok && c < d_k;
      cp_async_16_zfill(s_st + c * 128 + col, ok ? S + int64_t(c) * d_v + col : S, ok);
    }
  };
  if constexpr (!kTokensFirst) issue_state_copies();

  // 1. token vectors, spread over all 8 warps: warps 0-3 take the query and key channels (and
  // k.q by warp reduction), warps 4-7 the value channels and the decay; through the prologue
  // if asked (the prologue's convolution state and weights are loaded here too).
  const int c2 = tid & 127;  // channel of this thread in step 2
  const bool lo = tid < 128;
  float kq = 0.f, x0 = 0.f, x1 = 0.f;  // lo: query, key; hi: value, decay input
  if (lo) {
    if (c2 < d_k) {
      x0 = load_elem<kInBF16>(q, vec_base + c2);
      x1 = load_elem<kInBF16>(k, vec_base + c2);
    }
  } else {
    if (c2 < d_v) x0 = load_elem<kInBF16>(v, bh * d_v + c2);
    if (c2 < d_k)
      x1 = kDecay == DECAY_CLAMPED ? static_cast<const float *>(decay)[vec_base + c2]
                                   : load_elem<kInBF16>(decay, vec_base + c2);
  }
  // the prologue's loads: convolution state and weights of this thread's channels
  const int C3 = 2 * d_k + d_v;
  const int64_t sb = bh * 3 * C3;
  const int np = lo ? 2 : 1;  // convolutions of this thread: q and k, or v
  const bool on = c2 < (lo ? d_k : d_v);
  const int cc0 = lo ? c2 : 2 * d_k + c2, cc1 = d_k + c2;
  float xs[2][3], wv[2][4];
  if constexpr (kPrologue) {
    const int h = int(bh % H);
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int cc = p == 0 ? cc0 : cc1;
      const bool onp = on && p < np;
#pragma unroll
      for (int j = 0; j < 3; ++j) xs[p][j] = onp ? load_elem<kInBF16>(pro.state, sb + j * C3 + cc) : 0.f;
      const float4 w4 = onp ? *reinterpret_cast<const float4 *>(pro.w + (int64_t(h) * C3 + cc) * 4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      wv[p][0] = w4.x;
      wv[p][1] = w4.y;
      wv[p][2] = w4.z;
      wv[p][3] = w4.w;
    }
  }

  // the output gate's logits of warp 0's columns, read at the very end: copied into shared
  // memory now (the API keeps out_gate 16-byte aligned and d_v a multiple of 4)
  constexpr int kEs = kInBF16 ? 2 : 4;
  __shared__ __align__(16) uint8_t s_gr[128 * kEs];
  if constexpr (kNormGate) {
    if (ty == 0 && col_ok)
      cp_async_small<4 * kEs>(s_gr + col * kEs, static_cast<const uint8_t *>(out_gate) + (bh * d_v + col) * kEs);
  }

  // 2. the state copies of this thread (rows ty + 8 j), issued here or before step 1
  if constexpr (kTokensFirst) issue_state_copies();

  if constexpr (kPrologue) {
    // the 4-tap convolutions and Swish, then the state shifted by one token (its loads all
    // came first: the stores would otherwise order them)
    const float xt[2] = {x0, lo ? x1 : 0.f};
    float u[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      float acc = wv[p][0] * xs[p][0];
      acc = fmaf(wv[p][1], xs[p][1], acc);
      acc = fmaf(wv[p][2], xs[p][2], acc);
      acc = fmaf(wv[p][3], xt[p], acc);
      u[p] = acc * sigmoid_approx(acc);  // Swish
    }
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      if (on && p < np) {
        const int cc = p == 0 ? cc0 : cc1;
        store_elem<kInBF16>(pro.state, sb + cc, xs[p][1]);
        store_elem<kInBF16>(pro.state, sb + C3 + cc, xs[p][2]);
        store_elem<kInBF16>(pro.state, sb + 2 * C3 + cc, xt[p]);
      }
    }
    x0 = on ? u[0] : 0.f;
    if (lo) {
      x1 = on ? u[1] : 0.f;
      float nq = x0 * x0, nk = x1 * x1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        nq += __shfl_xor_sync(0xffffffffu, nq, o);
        nk += __shfl_xor_sync(0xffffffffu, nk, o);
      }
      if (tx == 0) {
        s_nrm[0][ty] = nq;
        s_nrm[1][ty] = nk;
      }
    }
    // q and k stay unnormalised here: their norms are applied after the barrier below, as
    // factors on y, z, k.q and the state update
  }
  if (lo) {
    s_q[c2] = x0;
    s_k[c2] = x1;
    kq = x0 * x1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
    if (tx == 0) s_kq[ty] = kq;
  } else {
    float a = 0.f;
    if (c2 < d_k) {
      if constexpr (kDecay == DECAY_CLAMPED) a = __expf(clamp_log_decay(x1, lb));
      else if constexpr (kDecay == DECAY_GATED) a = __expf(gated_log_decay(x1, __expf(A_log[bh % H]), lb));
      else a = __expf(unbounded_log_decay(x1, __expf(A_log[bh % H])));
    }
    s_a[c2] = a;
    s_v[c2] = x0;
  }
  const float b = beta[bh];
  __syncthreads();

  // 3. decay rows, partial predictions y = S'^T k and readouts z = S'^T q (each thread reads
  // back the rows it copied)
  cp_async_wait_all();
  float y[4] = {0.f, 0.f, 0.f, 0.f}, z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kDecodeRowsPerThread; ++j) {
    const int c = ty + 8 * j;
    const float a = s_a[c & 127], kc = s_k[c & 127], qc = s_q[c & 127];
    float4 sv = *reinterpret_cast<const float4 *>(s_st + c * 128 + col);
    sv.x *= a; sv.y *= a; sv.z *= a; sv.w *= a;
    y[0] += kc * sv.x; y[1] += kc * sv.y; y[2] += kc * sv.z; y[3] += kc * sv.w;
    z[0] += qc * sv.x; z[1] += qc * sv.y; z[2] += qc * sv.z; z[3] += qc * sv.w;
  }
  *reinterpret_cast<float4 *>(&s_red_y[ty][col]) = make_float4(y[0], y[1], y[2], y[3]);
  *reinterpret_cast<float4 *>(&s_red_z[ty][col]) = make_float4(z[0], z[1], z[2], z[3]);
  __syncthreads();

  float yt[4] = {0.f, 0.f, 0.f, 0.f}, zt[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const float4 ya = *reinterpret_cast<const float4 *>(&s_red_y[r][col]);
    const float4 za = *reinterpret_cast<const float4 *>(&s_red_z[r][col]);
    yt[0] += ya.x; yt[1] += ya.y; yt[2] += ya.z; yt[3] += ya.w;
    zt[0] += za.x; zt[1] += za.y; zt[2] += za.z; zt[3] += za.w;
  }
  kq = s_kq[0] + s_kq[1] + s_kq[2] + s_kq[3];
  float rk = 1.f;  // the prologue's L2 norms of q and k: 1 / |q|, 1 / |k|
  if constexpr (kPrologue) {
    const float rq = rsqrtf(((s_nrm[0][0] + s_nrm[0][1]) + (s_nrm[0][2] + s_nrm[0][3])) + pro.eps);
    rk = rsqrtf(((s_nrm[1][0] + s_nrm[1][1]) + (s_nrm[1][2] + s_nrm[1][3])) + pro.eps);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      yt[e] *= rk;
      zt[e] *= rq;
    }
    kq *= rq * rk;
  }

  // 4. delta-rule write u = b (v - y), S_t = S' + k u^T, o = scale (z + u (k.q))
  float u[4], uk[4];  // uk = u / |k| when k is normalised here, so that k_c uk = k^_c u
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    u[e] = b * (s_v[(col + e) & 127] - yt[e]);
    uk[e] = kPrologue ? u[e] * rk : u[e];
  }
#pragma unroll
  for (int j = 0; j < kDecodeRowsPerThread; ++j) {
    const int c = ty + 8 * j;
    if (col_ok && c < d_k) {
      const float kc = s_k[c], a = s_a[c];
      const float4 sv = *reinterpret_cast<const float4 *>(s_st + c * 128 + col);
      const float4 w = make_float4(fmaf(sv.x, a, kc * uk[0]), fmaf(sv.y, a, kc * uk[1]),
                                   fmaf(sv.z, a, kc * uk[2]), fmaf(sv.w, a, kc * uk[3]));
      __stcs(reinterpret_cast<float4 *>(S + int64_t(c) * d_v + col), w);
    }
  }
  if (ty == 0) {
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = col_ok ? scale * (zt[e] + u[e] * kq) : 0.f;
    if constexpr (kNormGate) {
      float ss = (o[0] * o[0] + o[1] * o[1]) + (o[2] * o[2] + o[3] * o[3]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float rstd = rsqrtf(ss / float(d_v) + norm_eps);
      if (col_ok) {
        cp_async_wait_all();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float w = norm_weight != nullptr ? norm_weight[col + e] : 1.f;
          const float r = load_elem<kInBF16>(s_gr, col + e);
          store_elem<kOutBF16>(out, bh * d_v + col + e, output_gate(o[e], rstd, w, r));
        }
      }
    } else if (col_ok) {
#pragma unroll
      for (int e = 0; e < 4; ++e) store_elem<kOutBF16>(out, bh * d_v + col + e, o[e]);
    }
  }
}

// decay: log_alpha (fp32) for DECAY_CLAMPED, else the gated forms' logits z (input dtype) with A_log.
// out_gate: gate logits [B, H, d_v] (input dtype) of the output gate, or null (out = o).
// conv_w / conv_state: the prologue's weights and state, or null (q, k, v used as given).
cudaError_t launch_decode(const void *q, const void *k, const void *v, const void *decay, int decay_form,
                          const float *A_log, const float *beta, float *state, const void *out_gate,
                          const float *norm_weight, float norm_eps, const float *conv_w, void *conv_state,
                          float l2_eps, void *out, int B, int H, int d_k, int d_v, bool in_bf16, bool out_bf16,
                          float lb, float scale, cudaStream_t stream) {
  const dim3 grid(unsigned(int64_t(B) * H)), block(kDecodeThreads);
  using Kern = decltype(&kda_decode_kernel<false, false, 0, false, false>);
#define KDA_DEC_ROW(ib, ob, ng, pr) \
  kda_decode_kernel<ib, ob, 0, ng, pr>, kda_decode_kernel<ib, ob, 1, ng, pr>, kda_decode_kernel<ib, ob, 2, ng, pr>
#define KDA_DEC_BLOCK(ng, pr)                                                                        \
  KDA_DEC_ROW(false, false, ng, pr), KDA_DEC_ROW(false, true, ng, pr), KDA_DEC_ROW(true, false, ng, pr), \
      KDA_DEC_ROW(true, true, ng, pr)
  static const Kern table[48] = {KDA_DEC_BLOCK(false, false), KDA_DEC_BLOCK(true, false),
                                 KDA_DEC_BLOCK(false, true), KDA_DEC_BLOCK(true, true)};
#undef KDA_DEC_BLOCK
#undef KDA_DEC_ROW
  const bool pro = conv_state != nullptr;
  const Kern kern = table[24 * int(pro) + 12 * int(out_gate != nullptr) + 6 * int(in_bf16) + 3 * int(out_bf16) +
                          decay_form];
  const Prologue pr{conv_w, conv_state, l2_eps};
  constexpr int kStateBytes = 128 * 128 * 4;  // the state tile in dynamic shared memory
  // the kernel attributes, set once per kernel and device (bit d of attr_set[idx] for device d;
  // a device past 63 sets them at every launch)
  static std::atomic<uint64_t> attr_set[48];
  const int idx = 24 * int(pro) + 12 * int(out_gate != nullptr) + 6 * int(in_bf16) + 3 * int(out_bf16) + decay_form;
  int dev = 0;
  if (const cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? uint64_t(1) << dev : 0;
  if (bit == 0 || (attr_set[idx].load(std::memory_order_acquire) & bit) == 0) {
    // and the whole of the SM's unified memory as shared memory, so that three CTAs fit
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kStateBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_set[idx].fetch_or(bit, std::memory_order_release);
  }
  kern<<<grid, block, kStateBytes, stream>>>(q, k, v, decay, A_log, beta, state, out_gate, norm_weight, norm_eps, pr, out, H,
                                   d_k, d_v, lb, scale);
  return cudaGetLastError();
}

}  // namespace kda
