// kda_prologue.cu -- the input prologue of a KDA layer over packed sequences.
//
// Kimi K3 -- Architecture Notes, section 1.1: the q, k and v projections pass a short
// convolution and then Swish, and q and k are L2-normalised (kernel size 4: the
// visualiser page "Kimi K3"). Per (token t, head h, channel c) of each projection:
//     conv_t = sum_{j<4} w[h, c, j] x_{t-3+j}   (causal, depthwise; before the sequence
//                                                start x comes from its convolution state)
//     u_t = conv_t Sigmoid(conv_t);   q_t, k_t = u_t / sqrt(sum_c u_tc^2 + eps);   v_t = u_t.
//
// The pass reads each raw input once and writes each result once. In the general kernel one
// CTA of 12 warps takes a tile of 32 tokens of one head (the persistent TMA kernel below walks
// a head's tiles instead). The tile's raw rows (and
// the 3 rows before it) are first copied to shared memory with coalesced loads. Then each
// warp takes one projection and 8 tokens; a lane owns 4 adjacent channels of a token row, so
// the 4 taps are 4 short shared-memory reads, the L2 norm of a token is one warp reduction,
// and every store of a warp is one contiguous row. A tile's tokens may belong to several
// sequences: a token's window stops at its own sequence start, where the sequence's state
// (or zero) takes over. Extra CTAs, one per sequence, write the final convolution states
// (the last three inputs of each sequence, shifted in from its initial state when the
// sequence is shorter than three).
#include <type_traits>

#include "kda_common.cuh"
#include "kda_tma_host.h"

namespace kda {

constexpr int kProThreads = 384;  // 12 warps: 3 projections x 4 warps of 8 tokens
constexpr int kProTile = 32;      // tokens per tile

template <bool kBF16>
__global__ void __launch_bounds__(kProThreads, 2)
    kda_prologue_kernel(const void *__restrict__ q_raw, const void *__restrict__ k_raw,
                        const void *__restrict__ v_raw, const float *__restrict__ conv_w,
                        const int32_t *__restrict__ cu_seqlens, int num_seqs, const void *__restrict__ conv_init,
                        void *__restrict__ q_out, void *__restrict__ k_out, void *__restrict__ v_out,
                        void *__restrict__ conv_final, int64_t T, int H, int d_k, int d_v, int n_tiles, float eps) {
  using Elem = typename std::conditional<kBF16, uint16_t, float>::type;
  extern __shared__ __align__(128) uint8_t pro_smem[];
  Elem *s_x = reinterpret_cast<Elem *>(pro_smem);  // [kProTile + 3][C3]: raw rows t0 - 3 .. t0 + 31
  __shared__ int32_t s_seq[kProTile];
  __shared__ int64_t s_bos[kProTile];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C3 = 2 * d_k + d_v;
  const int h = blockIdx.y;
  auto src_of = [&](int cc, const void *&base, int &d, int &c) {  // packed channel -> projection
    if (cc < d_k) { base = q_raw; d = d_k; c = cc; }
    else if (cc < 2 * d_k) { base = k_raw; d = d_k; c = cc - d_k; }
    else { base = v_raw; d = d_v; c = cc - 2 * d_k; }
  };

  if (int(blockIdx.x) >= n_tiles) {  // final convolution state of one sequence
    const int n = int(blockIdx.x) - n_tiles;
    if (conv_final == nullptr || n >= num_seqs) return;
    const int64_t bos = cu_seqlens[n], eos = cu_seqlens[n + 1];
    for (int cc = tid; cc < C3; cc += kProThreads) {
      const void *base;
      int d, c;
      src_of(cc, base, d, c);
      const int64_t sbase = (int64_t(n) * H + h) * 3 * C3 + cc;
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int64_t pos = eos - 3 + i;
        float val = 0.f;
        if (pos >= bos) val = load_elem<kBF16>(base, (pos * H + h) * d + c);
        else if (conv_init != nullptr) val = load_elem<kBF16>(conv_init, sbase + (i + (eos - bos)) * C3);
        store_elem<kBF16>(conv_final, sbase + int64_t(i) * C3, val);
      }
    }
    return;
  }

  const int64_t t0 = int64_t(blockIdx.x) * kProTile;
  if (tid < kProTile) {  // sequence of each token: the last n with cu_seqlens[n] <= t
    const int64_t t = t0 + tid;
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu_seqlens[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    s_seq[tid] = lo;
    s_bos[tid] = cu_seqlens[lo];
  }
  // raw rows t0 - 3 .. t0 + 31 of the three projections (zero outside [0, T)), all of a
  // thread's loads issued before the first is used: 16-byte vectors (at most 5 per thread for
  // bf16, 9 for fp32) when d_k and d_v are whole vectors, else single elements (at most 35).
  constexpr int V = 16 / int(sizeof(Elem));                                             // elements per vector
  constexpr int kSlots = (kProTile + 3 + kProThreads / (384 / V) - 1) / (kProThreads / (384 / V));  // C3 <= 384
  if (d_k % V == 0 && d_v % V == 0) {
    // thread -> one vector column of the packed row and rows r0, r0 + R, ...
    const int per_row = C3 / V, R = kProThreads / per_row;  // per_row <= 48 here, so R >= 8
    const int r0 = tid / per_row, col = tid - r0 * per_row;
    const void *base;
    int d, c;
    src_of(col * V, base, d, c);
    const bool on = r0 < R;  // threads past R rows' worth of columns stay idle
    const Elem *src = static_cast<const Elem *>(base) + int64_t(h) * d + c;
    const int64_t tok_stride = int64_t(H) * d;
    uint4 val[kSlots];
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      const int r = r0 + i * R;
      const int64_t pos = t0 - 3 + r;
      val[i] = make_uint4(0, 0, 0, 0);
      if (on && r < kProTile + 3 && pos >= 0 && pos < T)
        val[i] = *reinterpret_cast<const uint4 *>(src + pos * tok_stride);
    }
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      const int r = r0 + i * R;
      if (on && r < kProTile + 3) reinterpret_cast<uint4 *>(s_x + r * C3)[col] = val[i];
    }
  } else {
    const int units = (kProTile + 3) * C3;
    Elem val[kProTile + 3];
#pragma unroll
    for (int i = 0; i < kProTile + 3; ++i) {
      const int e = tid + i * kProThreads;
      val[i] = Elem(0);
      if (e < units) {
        const int r = e / C3, cc = e - r * C3;
        const int64_t pos = t0 - 3 + r;
        const void *base;
        int d, c;
        src_of(cc, base, d, c);
        if (pos >= 0 && pos < T) val[i] = static_cast<const Elem *>(base)[(pos * H + h) * d + c];
      }
    }
#pragma unroll
    for (int i = 0; i < kProTile + 3; ++i) {
      const int e = tid + i * kProThreads;
      if (e < units) s_x[e] = val[i];
    }
  }
  __syncthreads();

  // warp -> projection p, tokens 8 (warp % 4) ..; lane -> channels 4 lane .. 4 lane + 3
  const int p = warp >> 2, tw = 8 * (warp & 3);
  const int d = p == 2 ? d_v : d_k;
  const int c0 = 4 * lane;
  const int cc0 = (p == 0 ? 0 : p == 1 ? d_k : 2 * d_k) + c0;
  void *x_out = p == 0 ? q_out : p == 1 ? k_out : v_out;
  float w[4][4];  // [channel][tap]
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) w[i][j] = c0 + i < d ? conv_w[(int64_t(h) * C3 + cc0 + i) * 4 + j] : 0.f;

  const bool vec4 = (d_k % 4 == 0) && (d_v % 4 == 0);  // a lane's 4 channels are one 8/16-byte word
  // Writes the results of one token: Swish, then for q and k the L2 norm (one warp reduction).
  auto finish = [&](int64_t tok, const float (&acc)[4]) {
    float u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = acc[i] * sigmoid_approx(acc[i]);  // Swish
    if (p < 2) {
      float ss = (u[0] * u[0] + u[1] * u[1]) + (u[2] * u[2] + u[3] * u[3]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rn = rsqrtf(ss + eps);
#pragma unroll
      for (int i = 0; i < 4; ++i) u[i] *= rn;
    }
    const int64_t obase = (tok * H + h) * d + c0;
    if (vec4) {  // one 8-byte (bf16) or 16-byte (fp32) store per lane
      if (c0 < d) {
        if constexpr (kBF16)
          *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(x_out) + obase) =
              make_uint2(pack_bf16x2(u[0], u[1]), pack_bf16x2(u[2], u[3]));
        else
          *reinterpret_cast<float4 *>(static_cast<float *>(x_out) + obase) = make_float4(u[0], u[1], u[2], u[3]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (c0 + i < d) store_elem<kBF16>(x_out, obase + i, u[i]);
    }
  };
  auto row4 = [&](int r, float (&x)[4]) {  // this lane's 4 channels of shared-memory row r
    const Elem *src = s_x + r * C3 + cc0;
    if constexpr (kBF16) {
      const uint2 wv = *reinterpret_cast<const uint2 *>(src);
      const float2 a = unpack_bf16x2(wv.x), b = unpack_bf16x2(wv.y);
      x[0] = a.x;
      x[1] = a.y;
      x[2] = b.x;
      x[3] = b.y;
    } else {
      const float4 f = *reinterpret_cast<const float4 *>(src);
      x[0] = f.x;
      x[1] = f.y;
      x[2] = f.z;
      x[3] = f.w;
    }
  };

  // Fast path: every row of the tile and its 3 predecessors in one sequence, all tokens in range:
  // a sliding window of 4 rows in registers, one shared-memory word per token.
  const bool one_seq = vec4 && t0 + kProTile <= T && s_seq[0] == s_seq[kProTile - 1] && t0 - 3 >= s_bos[0];
  if (one_seq) {
    float win[4][4] = {};  // rows tw + tt .. tw + tt + 3 (token tw + tt's window)
    if (c0 < d) {
#pragma unroll
      for (int j = 0; j < 3; ++j) row4(tw + j, win[j + 1]);
    }
#pragma unroll
    for (int tt = 0; tt < 8; ++tt) {
#pragma unroll
      for (int j = 0; j < 3; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) win[j][i] = win[j + 1][i];
      if (c0 < d) row4(tw + tt + 3, win[3]);
      float acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i] = w[i][0] * win[0][i];
        acc[i] = fmaf(w[i][1], win[1][i], acc[i]);
        acc[i] = fmaf(w[i][2], win[2][i], acc[i]);
        acc[i] = fmaf(w[i][3], win[3][i], acc[i]);
      }
      finish(t0 + tw + tt, acc);
    }
    return;
  }

  for (int tt = 0; tt < 8; ++tt) {  // general path: per token, per tap, per channel
    const int t = tw + tt;
    const int64_t tok = t0 + t;
    if (tok >= T) break;  // warp-uniform
    const int64_t bos = s_bos[t];
    float acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t pos = tok - 3 + j;
        float xv = 0.f;
        if (c0 + i < d) {
          if (pos >= bos) xv = bf16_or_f32(s_x[(t + j) * C3 + cc0 + i]);
          else if (conv_init != nullptr)
            xv = load_elem<kBF16>(conv_init, ((int64_t(s_seq[t]) * H + h) * 3 + (3 + pos - bos)) * C3 + cc0 + i);
        }
        acc[i] = fmaf(w[i][j], xv, acc[i]);
      }
    }
    finish(tok, acc);
  }
}

// Persistent variant for d_k, d_v multiples of 8 (whole 16-byte rows): a CTA keeps one head
// (its weights stay in registers) and walks that head's 32-token tiles through a TMA pipeline of
// kProStages tiles. Warp 12 only loads: it issues tile k + S into a stage once the 12 compute
// warps have released it (an mbarrier per stage, one arrival per warp), so that no compute warp
// waits on another: warp w (< 12) waits for the stage to land, finds its own tokens' sequences,
// computes and releases the stage. Warp w takes projection w / 4 and tokens 8 (w % 4) .. + 7, a
// lane 4 adjacent channels of a row, so a token's L2 norm is one warp reduction, the 4 taps come
// from a sliding window of shared-memory rows, and each lane stores 8 or 16 bytes; the arithmetic
// runs on fp32 pairs. Rows before token 0 and past the end read as zero.
constexpr int kProRows = kProTile + 3;
constexpr int kProWarps = kProThreads / 32;         // compute warps
constexpr int kProTmaThreads = kProThreads + 32;    // + the loading warp
template <bool kBF16>
constexpr int kProStages = kBF16 ? 3 : 2;  // 3 x 26,880 (bf16) or 2 x 53,760 (fp32) bytes of tiles per CTA

__host__ __device__ constexpr uint32_t round128(uint32_t x) { return (x + 127u) & ~127u; }

template <bool kBF16>
__global__ void __launch_bounds__(kProTmaThreads, 2)
    kda_prologue_tma_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ conv_w,
                            const int32_t *__restrict__ cu_seqlens, int num_seqs,
                            const void *__restrict__ conv_init, void *__restrict__ q_out, void *__restrict__ k_out,
                            void *__restrict__ v_out, int64_t T, int H, int d_k, int d_v, int n_tiles, float eps,
                            uint32_t *err_word) {
  using Elem = typename std::conditional<kBF16, uint16_t, float>::type;
  constexpr uint32_t es = sizeof(Elem);
  extern __shared__ __align__(128) uint8_t pro_smem[];
  constexpr int S = kProStages<kBF16>;
  __shared__ __align__(8) uint64_t s_full[S], s_empty[S];
  __shared__ uint32_t s_bad;
  constexpr int kCuSmem = 1024;  // sequence offsets kept in shared memory when they fit
  __shared__ int32_t s_cu[kCuSmem];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C3 = 2 * d_k + d_v;
  const uint32_t off_k = round128(kProRows * d_k * es), off_v = 2 * off_k;
  const uint32_t stage_bytes = off_v + round128(kProRows * d_v * es);
  const uint32_t tx_bytes = kProRows * uint32_t(C3) * es;
  // this CTA: head h, tiles tile0, tile0 + m, ... (gridDim.x = m H)
  const int m = int(gridDim.x) / H, h = int(blockIdx.x) % H, tile0 = int(blockIdx.x) / H;
  const bool cu_in_smem = num_seqs + 1 <= kCuSmem;
  if (cu_in_smem)
    for (int i = tid; i <= num_seqs; i += kProTmaThreads) s_cu[i] = cu_seqlens[i];
  const int32_t *cu = cu_in_smem ? s_cu : cu_seqlens;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kProWarps);
    }
    fence_mbarrier_init();
    s_bad = 0u;
  }
  __syncthreads();  // barriers and sequence offsets ready; from here no CTA-wide barrier

  if (warp == kProWarps) {
    // ------------------------------------------------------------ loading warp (lane 0)
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int k = 0;
      for (int tile = tile0; tile < n_tiles; tile += m, ++k) {
        const int s = k % S;
        // the compute warps have released this stage (its previous tile, k - S)
        if (k >= S && !mbar_wait_sleep(&s_empty[s], uint32_t(((k - S) / S) & 1), err_word, DEVERR_TMA_TIMEOUT)) {
          s_bad = 1u;
          break;
        }
        const int32_t y0 = tile * kProTile - 3;
        uint8_t *st = pro_smem + s * stage_bytes;
        mbar_arrive_expect_tx(&s_full[s], tx_bytes);
        tma_load_3d(st, &tm_q, &s_full[s], 0, h, y0);
        tma_load_3d(st + off_k, &tm_k, &s_full[s], 0, h, y0);
        tma_load_3d(st + off_v, &tm_v, &s_full[s], 0, h, y0);
      }
      // wait for the loads issued last (bounded) before this CTA's shared memory goes away
      const int issued = k;
      for (int kk = issued - S > 0 ? issued - S : 0; kk < issued; ++kk)
        mbar_wait_sleep(&s_full[kk % S], uint32_t((kk / S) & 1), err_word, DEVERR_TMA_TIMEOUT);
    }
    return;
  }

  const int p = warp >> 2;
  const int tb = 8 * (warp & 3);  // this warp's first token in the tile
  const int d = p == 2 ? d_v : d_k;
  const int c0 = 4 * lane;
  const bool on = c0 < d;
  const int pbase = p == 0 ? 0 : p == 1 ? d_k : 2 * d_k;  // packed channel of this projection
  const uint32_t roff = p == 0 ? 0u : p == 1 ? off_k : off_v;
  void *x_out = p == 0 ? q_out : p == 1 ? k_out : v_out;

  float2 wp[2][4];  // [channel pair][tap] of head h
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float *wr = conv_w + (int64_t(h) * C3 + pbase + c0 + 2 * i) * 4;
    const float4 a = on ? *reinterpret_cast<const float4 *>(wr) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 b = on ? *reinterpret_cast<const float4 *>(wr + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    wp[i][0] = make_float2(a.x, b.x);
    wp[i][1] = make_float2(a.y, b.y);
    wp[i][2] = make_float2(a.z, b.z);
    wp[i][3] = make_float2(a.w, b.w);
  }
  // the last n with cu[n] <= t
  auto seq_of = [&](int64_t t) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  };
  int k = 0;
  for (int tile = tile0; tile < n_tiles; tile += m, ++k) {
    const int s = k % S;
    const int64_t t0 = int64_t(tile) * kProTile;
    // the sequences of this warp's tokens (lanes 0..7), and whether the whole tile with the 3 rows
    // before it lies in one sequence (lanes 8 and 9 find the first and last token's)
    int my_seq = 0;
    int64_t my_bos = 0;
    if (lane < 8 || lane == 8 || lane == 9) {
      const int64_t t = lane < 8 ? t0 + tb + lane : lane == 8 ? t0 : t0 + kProTile - 1;
      my_seq = seq_of(t < T ? t : T - 1);
      my_bos = cu[my_seq];
    }
    const int seq_first = __shfl_sync(0xffffffffu, my_seq, 8), seq_last = __shfl_sync(0xffffffffu, my_seq, 9);
    const int64_t bos_first = __shfl_sync(0xffffffffu, my_bos, 8);
    const bool one_seq = t0 + kProTile <= T && seq_first == seq_last && t0 - 3 >= bos_first;
    if (!mbar_wait_sleep(&s_full[s], uint32_t((k / S) & 1), err_word, DEVERR_TMA_TIMEOUT) || s_bad != 0u) break;
    const Elem *rows = reinterpret_cast<const Elem *>(pro_smem + s * stage_bytes + roff);  // [35][d]
    auto row4 = [&](int r, float2 (&x)[2]) {  // this lane's 4 channels of row r, as pairs
      if constexpr (kBF16) {
        const uint2 v2 = *reinterpret_cast<const uint2 *>(rows + r * d + c0);
        x[0] = unpack_bf16x2(v2.x);
        x[1] = unpack_bf16x2(v2.y);
      } else {
        const float4 a = *reinterpret_cast<const float4 *>(rows + r * d + c0);
        x[0] = make_float2(a.x, a.y);
        x[1] = make_float2(a.z, a.w);
      }
    };
    auto finish = [&](int64_t tok, float2 (&u)[2]) {  // Swish, L2 norm of q / k, store (channel pairs)
#pragma unroll
      for (int i = 0; i < 2; ++i) {  // Swish(x) = x / (1 + 2^{-x log2 e})
        const float2 e = f2_mul(u[i], make_float2(-1.4426950408889634f, -1.4426950408889634f));
        float2 den;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(den.x) : "f"(e.x));
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(den.y) : "f"(e.y));
        den = f2_add(den, make_float2(1.f, 1.f));
        float2 r;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(den.x));
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(den.y));
        u[i] = f2_mul(u[i], r);
      }
      if (p < 2) {
        const float2 s2 = f2_fma(u[1], u[1], f2_mul(u[0], u[0]));
        float ss = s2.x + s2.y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float rn = rsqrtf(ss + eps);
        u[0] = f2_mul(u[0], make_float2(rn, rn));
        u[1] = f2_mul(u[1], make_float2(rn, rn));
      }
      if (on && tok < T) {
        const int64_t o = (tok * H + h) * d + c0;
        if constexpr (kBF16)
          *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(x_out) + o) =
              make_uint2(pack_bf16x2(u[0].x, u[0].y), pack_bf16x2(u[1].x, u[1].y));
        else
          *reinterpret_cast<float4 *>(static_cast<float *>(x_out) + o) = make_float4(u[0].x, u[0].y, u[1].x, u[1].y);
      }
    };

    // two consecutive tokens tok, tok + 1: Swish, the L2 norms of q / k in one halving reduction
    // (lanes 0..15 end with token tok's sum of squares, lanes 16..31 with token tok + 1's), store
    auto finish2 = [&](Elem *op, float2 (&u)[2][2]) {  // op: this lane's channels of the first token
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int i = 0; i < 2; ++i) {  // Swish(x) = x / (1 + 2^{-x log2 e})
          const float2 e = f2_mul(u[a][i], make_float2(-1.4426950408889634f, -1.4426950408889634f));
          float2 den;
          asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(den.x) : "f"(e.x));
          asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(den.y) : "f"(e.y));
          den = f2_add(den, make_float2(1.f, 1.f));
          float2 r;
          asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(den.x));
          asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(den.y));
          u[a][i] = f2_mul(u[a][i], r);
        }
      if (p < 2) {
        float ss[2];
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          const float2 s2 = f2_fma(u[a][1], u[a][1], f2_mul(u[a][0], u[a][0]));
          ss[a] = s2.x + s2.y;
        }
        const float tot = lane_sums<2>(ss, lane);  // token tok + (lane >> 4)
        const float rn_l = rsqrtf(tot + eps);
        const float rn0 = __shfl_sync(0xffffffffu, rn_l, 0), rn1 = __shfl_sync(0xffffffffu, rn_l, 16);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          u[0][i] = f2_mul(u[0][i], make_float2(rn0, rn0));
          u[1][i] = f2_mul(u[1][i], make_float2(rn1, rn1));
        }
      }
      if (on) {  // both tokens lie inside the tile's one sequence, before T
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          Elem *o = op + int64_t(a) * H * d;
          if constexpr (kBF16)
            *reinterpret_cast<uint2 *>(o) = make_uint2(pack_bf16x2(u[a][0].x, u[a][0].y), pack_bf16x2(u[a][1].x, u[a][1].y));
          else
            *reinterpret_cast<float4 *>(o) = make_float4(u[a][0].x, u[a][0].y, u[a][1].x, u[a][1].y);
        }
      }
    };

    if (one_seq) {  // every row of the tile and the 3 before it in one sequence: a sliding window
      Elem *op = static_cast<Elem *>(x_out) + ((t0 + tb) * H + h) * d + c0;  // token t0 + tb
      const int64_t ostep = int64_t(2) * H * d;                                  // two tokens
      // two tokens per step (rows tb + tt .. tb + tt + 4): two independent chains, and one
      // reduction for both tokens' L2 norms; row and output pointers step instead of indexing
      float2 win[5][2] = {};  // [row][channel pair]
      const Elem *rp = rows + tb * d + c0;  // row tb
      auto rowp = [&](const Elem *r, float2 (&x)[2]) {
        if constexpr (kBF16) {
          const uint2 v2 = *reinterpret_cast<const uint2 *>(r);
          x[0] = unpack_bf16x2(v2.x);
          x[1] = unpack_bf16x2(v2.y);
        } else {
          const float4 a = *reinterpret_cast<const float4 *>(r);
          x[0] = make_float2(a.x, a.y);
          x[1] = make_float2(a.z, a.w);
        }
      };
      if (on) {
        rowp(rp, win[2]);
        rowp(rp + d, win[3]);
        rowp(rp + 2 * d, win[4]);
      }
      rp += 3 * d;  // row tb + 3
#pragma unroll
      for (int tt = 0; tt < 8; tt += 2) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          win[j][0] = win[j + 2][0];
          win[j][1] = win[j + 2][1];
        }
        if (on) {
          rowp(rp, win[3]);
          rowp(rp + d, win[4]);
        }
        rp += 2 * d;
        float2 u[2][2];  // [token][channel pair]
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            u[a][i] = f2_mul(wp[i][0], win[a][i]);
            u[a][i] = f2_fma(wp[i][1], win[a + 1][i], u[a][i]);
            u[a][i] = f2_fma(wp[i][2], win[a + 2][i], u[a][i]);
            u[a][i] = f2_fma(wp[i][3], win[a + 3][i], u[a][i]);
          }
        finish2(op, u);
        op += ostep;
      }
    } else {  // per token and tap: before its sequence start a token reads the state (or zero)
      for (int tt = 0; tt < 8; ++tt) {
        const int t = tb + tt;
        const int64_t tok = t0 + t;
        const int seq = __shfl_sync(0xffffffffu, my_seq, tt);
        const int64_t bos = __shfl_sync(0xffffffffu, my_bos, tt);
        float2 up[2] = {};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t pos = tok - 3 + j;
          float2 x[2] = {};
          if (on) {
            if (pos >= bos) {
              row4(t + j, x);
            } else if (conv_init != nullptr) {
              const int64_t sb = ((int64_t(seq) * H + h) * 3 + (3 + pos - bos)) * C3 + pbase + c0;
              x[0] = make_float2(load_elem<kBF16>(conv_init, sb), load_elem<kBF16>(conv_init, sb + 1));
              x[1] = make_float2(load_elem<kBF16>(conv_init, sb + 2), load_elem<kBF16>(conv_init, sb + 3));
            }
          }
          up[0] = f2_fma(wp[0][j], x[0], up[0]);
          up[1] = f2_fma(wp[1][j], x[1], up[1]);
        }
        finish(tok, up);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s_empty[s]);  // this warp is done with the stage
  }
}

cudaError_t launch_prologue(const void *q_raw, const void *k_raw, const void *v_raw, const float *conv_w,
                            const int32_t *cu_seqlens, int num_seqs, int64_t total_tokens, int H, int d_k, int d_v,
                            bool bf16, const void *conv_init, float eps, void *q, void *k, void *v,
                            void *conv_final, cudaStream_t stream) {
  const int n_tiles = int((total_tokens + kProTile - 1) / kProTile);
  const uint32_t es = bf16 ? 2 : 4;
  // whole 16-byte rows, rows of 8 channels per lane, and a work-item count that fits an int
  const bool tma = d_k % 8 == 0 && d_v % 8 == 0 && int64_t(n_tiles) * H < (int64_t(1) << 30);
  if (tma && n_tiles > 0) {
    CUtensorMap mq, mk, mv;
    if (!tensor_map_3d(&mq, q_raw, bf16, total_tokens, H, d_k, uint32_t(d_k), kProRows, false) ||
        !tensor_map_3d(&mk, k_raw, bf16, total_tokens, H, d_k, uint32_t(d_k), kProRows, false) ||
        !tensor_map_3d(&mv, v_raw, bf16, total_tokens, H, d_v, uint32_t(d_v), kProRows, false))
      return cudaErrorInvalidValue;
    auto kern = bf16 ? kda_prologue_tma_kernel<true> : kda_prologue_tma_kernel<false>;
    const uint32_t stage = 2 * round128(kProRows * d_k * es) + round128(kProRows * d_v * es);
    const size_t smem = size_t(bf16 ? kProStages<true> : kProStages<false>) * stage;  // <= 107,520 bytes (80,640 bf16)
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
      return cudaGetLastError();
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaGetLastError();
    // m CTAs per head, m H about two per SM (at least one per head)
    const int m = (2 * sms) / H > 1 ? (2 * sms) / H : 1;
    const unsigned grid = unsigned(m * H);
    kern<<<grid, kProTmaThreads, smem, stream>>>(mq, mk, mv, conv_w, cu_seqlens, num_seqs, conv_init, q, k, v,
                                                 total_tokens, H, d_k, d_v, n_tiles, eps, device_error_word());
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // the general kernel: the tiles when the TMA path does not apply, and the final states
  const int tiles = tma ? 0 : n_tiles;
  const dim3 grid(unsigned(tiles + (conv_final != nullptr ? num_seqs : 0)), unsigned(H)), block(kProThreads);
  if (grid.x == 0) return cudaSuccess;
  auto kern = bf16 ? kda_prologue_kernel<true> : kda_prologue_kernel<false>;
  const size_t smem = tiles > 0 ? size_t(kProRows) * (2 * d_k + d_v) * es : 0;  // <= 53,760 bytes
  if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
                              cudaSuccess)
    return cudaGetLastError();
  kern<<<grid, block, smem, stream>>>(q_raw, k_raw, v_raw, conv_w, cu_seqlens, num_seqs, conv_init, q, k, v,
                                      conv_final, total_tokens, H, d_k, d_v, tiles, eps);
  return cudaGetLastError();
}

}  // namespace kda
