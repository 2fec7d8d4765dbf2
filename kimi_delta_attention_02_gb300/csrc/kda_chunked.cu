// kda_chunked.cu -- tensor-core chunkwise KDA prefill (bf16 q/k/v, d_k = d_v = 128).
//
// Kimi K3 -- Architecture Notes, section 1.2: the kernel is recurrent across
// chunks and parallel within each chunk; relative decay is kept in range with
// 16-token tiles, and with log-decay >= -5 every rescaling factor inside a tile
// stays below e^80, so all intra-chunk products are dense tensor-core matmuls.
//
// Math for one chunk of L <= 32 tokens entered with state S (d_k x d_v), from
// the section 1.1 recurrence. G_t = cumulative clamped log-decay inside the
// chunk, Gamma_t = exp(G_t):
//   A[t,i] = b_t sum_c k_tc k_ic e^{G_tc - G_ic}   (i < t)      T = (I + A)^{-1}
//   P[t,i] =     sum_c q_tc k_ic e^{G_tc - G_ic}   (i <= t)     T' = T Diag(b)
//   W = T' (K * Gamma),  U~ = T' V,  U = U~ - W S
//   O = (Q * Gamma) S + P U,   S <- Diag(Gamma_last) S + (K * e^{G_last - G})^T U
// e^{G_t - G_i} is split per 16-token subtile s with reference r_s = G at the
// end of subtile s-1: the query/key side q_t e^{G_t - r_s} <= 1 is built once,
// the other side k_i e^{r_s - G_i} once per row subtile (<= 1 below the
// diagonal, < e^80 on it). Every factor is a running product of alpha = exp(g)
// inside a subtile times per-channel subtile totals.
//
// Precision. Outputs and states are heavy-tailed (their largest entries are
// about ten times their rms), so a per-element relative error e shows up as
// about 10e in max|error| / rms. bf16 operands (e = 2^-9) therefore cannot meet
// a 2e-2 bound. The Gram operands carry factors up to e^80 and go through the
// tensor cores as tf32 (fp32 range, rounded to nearest, e = 2^-11); every other
// operand is bounded (|factor| <= 1, T' and U of order one) and goes as fp16
// (e = 2^-11), which needs no more shared memory than bf16. Accumulation is
// fp32 throughout and the state is kept in fp32 registers.
//
// Layout of the work. One CTA (256 threads) per (sequence, head) chain walks
// its 32-token chunks in order; thread (v = 32 (warp % 4) + lane, half =
// warp / 4) owns S[c][v] for c in [64 half, 64 half + 64). Per chunk:
//   1. TMA has landed q, k, v (bf16, 128-byte swizzle) and g (fp32) two chunks
//      ahead. Threads build the decay factors and the operand tiles.
//   2. tcgen05 kind::tf32: Gram tiles per row subtile (M=64, N=32, K=128).
//   3. Threads read P and A out of tensor memory; SIMT fp32 blocked inverse.
//   4. tcgen05 kind::f16: W = T' Kg (M=64) and U~^T = V^T T'^T (M=128).
//   5. The state-dependent chain, all M=128 (rows = value channels):
//      U^T = U~^T - S^T W^T ; O^T = S^T Q~^T + U^T P^T ; dS^T = U^T K^
//      with an fp16 copy of S^T as the A operand; fp32 state update.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kC = 32;      // chunk length (two 16-token subtiles)
constexpr int kD = 128;     // d_k = d_v
constexpr int kThreads = 256;
constexpr int kALd = 36;    // fp32 row stride of the A / T scratch (16-byte rows, spread banks)

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t kStageBytes = 40 * 1024;  // one input stage: q | k | v (bf16) | g (fp32)
constexpr uint32_t SQ = 0, SK = 8 * 1024, SV = 16 * 1024, SG = 24 * 1024;
constexpr uint32_t OFF_STAGE = 0;            // two stages
constexpr uint32_t OFF_GRAM = 80 * 1024;     // 60 KB reused by phase:
//   Gram: QK tf32 [64 rows][128] at +0 (32 KB; rows 32s.. = subtile s: 16 query then 16 key rows),
//         B_0 tf32 [16][128] at +32 KB, B_1 tf32 [32][128] at +40 KB; the M = 64 reads of B_1 end at +60 KB
//   inverse: A fp32 [32][36] at +0, T fp32 at +5 KB, X at +10 KB
//   chain: W fp16 [32][128] at +0, S^T fp16 [128][128] at +8 KB, U^T fp16 [128][64] at +40 KB
constexpr uint32_t OFF_TP = 140 * 1024;      // T' = T Diag(beta) fp16 [64 rows][64] (rows, cols >= 32 unused)
constexpr uint32_t OFF_P = 148 * 1024;       // P fp16 [32 t][64]
constexpr uint32_t OFF_KG = 152 * 1024;      // K * Gamma fp16 [32 i][128 c] (MN-major B of W)
constexpr uint32_t OFF_KH = 160 * 1024;      // K * e^{G_last - G} fp16 [32 i][128 c] (MN-major B of dS)
constexpr uint32_t OFF_QT = 168 * 1024;      // Q * Gamma fp16 [32 t][128 c] (K-major B of O)
constexpr uint32_t OFF_MISC = 176 * 1024;    // beta, Gamma_last, subtile totals, barriers
constexpr uint32_t kSmemBytes = 178 * 1024 + 1024;

constexpr uint32_t G_QK = 0, G_B0 = 32 * 1024, G_B1 = 40 * 1024;
constexpr uint32_t G_A = 0, G_T = 5 * 1024, G_X = 10 * 1024;
constexpr uint32_t G_W = 0, G_ST = 8 * 1024, G_UT = 40 * 1024;

// TMEM columns
constexpr uint32_t TM_GRAM = 0, TM_W = 64, TM_U = 192, TM_O = 224, TM_DS = 256, TM_COLS = 512;

constexpr uint32_t IDESC_GRAM = umma_idesc(UMMA_TF32, 64, 32, false, false, false);
constexpr uint32_t IDESC_W = umma_idesc(UMMA_F16, 64, 128, false, true, false);
constexpr uint32_t IDESC_UT = umma_idesc(UMMA_F16, 128, 32, true, false, false);
constexpr uint32_t IDESC_SW_NEG = umma_idesc(UMMA_F16, 128, 32, false, false, true);
constexpr uint32_t IDESC_O = umma_idesc(UMMA_F16, 128, 32, false, false, false);
constexpr uint32_t IDESC_DS = umma_idesc(UMMA_F16, 128, 128, false, true, false);

constexpr uint32_t kKmajLbo = 16, kSbo = 1024;  // 128-byte swizzle: 8-row atoms of 1 KB
constexpr uint32_t kMnBlock = kC * 128;         // MN-major tiles of 32 rows: next 64-wide block

__device__ __forceinline__ uint64_t kdesc(uint32_t addr) { return umma_desc(addr, kKmajLbo, kSbo, kSwizzle128B); }
__device__ __forceinline__ uint64_t mndesc(uint32_t addr) { return umma_desc(addr, kMnBlock, kSbo, kSwizzle128B); }

template <typename T>
__device__ __forceinline__ void st_at(uint8_t *base, uint32_t off, T v) {
  *reinterpret_cast<T *>(base + off) = v;
}
__device__ __forceinline__ uint4 pack8_f16(const float *x) {
  return make_uint4(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]), pack_f16x2(x[4], x[5]), pack_f16x2(x[6], x[7]));
}

template <bool kOutBF16>
__global__ void __launch_bounds__(kThreads, 1)
    kda_chunked_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                       const float *__restrict__ beta, const int32_t *__restrict__ cu_seqlens,
                       const float *__restrict__ init_state, void *__restrict__ out,
                       float *__restrict__ final_state, int H, float lb, float scale, uint32_t *err_word) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *gram = sm + OFF_GRAM;
  float *s_beta = reinterpret_cast<float *>(sm + OFF_MISC);  // [32]
  float *s_gamma = s_beta + 32;                               // [128] Gamma_last
  float *s_tau = s_gamma + 128;                               // [2][128] subtile totals
  uint64_t *bar_in = reinterpret_cast<uint64_t *>(s_tau + 2 * 128);  // [2]
  uint64_t *bar_mma = bar_in + 2;
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar_in + 3);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int h = int(blockIdx.x % H);
  const int64_t n = blockIdx.x / H;
  const int64_t bos = cu_seqlens[n], eos = cu_seqlens[n + 1];
  const int n_chunks = int((eos - bos + kC - 1) / kC);
  const uint32_t sbase = smem_u32(sm);

  if (tid == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_g);
    mbar_init(&bar_in[0], 1);
    mbar_init(&bar_in[1], 1);
    mbar_init(bar_mma, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, TM_COLS);
    tmem_relinquish();
  }

  // state: S[c][v] for v = 32 quarter + lane, c = 64 half + j
  const int v_own = 32 * quarter + lane;
  float S[64];
  const int64_t st_base = (n * H + h) * int64_t(kD) * kD;
#pragma unroll
  for (int j = 0; j < 64; ++j)
    S[j] = init_state != nullptr ? init_state[st_base + int64_t(64 * half + j) * kD + v_own] : 0.f;

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_base = uint32_t(32 * quarter) << 16;

  auto issue_stage = [&](int chunk) {  // thread 0 only
    const int32_t t0 = int32_t(bos + int64_t(chunk) * kC);
    uint8_t *st = sm + OFF_STAGE + (chunk & 1) * kStageBytes;
    uint64_t *bar = &bar_in[chunk & 1];
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_3d(st + SQ, &tm_q, bar, 0, h, t0);
    tma_load_3d(st + SQ + 4096, &tm_q, bar, 64, h, t0);
    tma_load_3d(st + SK, &tm_k, bar, 0, h, t0);
    tma_load_3d(st + SK + 4096, &tm_k, bar, 64, h, t0);
    tma_load_3d(st + SV, &tm_v, bar, 0, h, t0);
    tma_load_3d(st + SV + 4096, &tm_v, bar, 64, h, t0);
    tma_load_3d(st + SG, &tm_g, bar, 0, h, t0);
  };
  // parity of the outstanding load of each stage (-1: none); every thread tracks it
  int inflight[2] = {-1, -1};
  for (int c = 0; c < 2 && c < n_chunks; ++c) {
    if (tid == 0) issue_stage(c);
    inflight[c] = 0;
  }

  uint32_t mma_phase = 0;
  bool bad = false;

  for (int chunk = 0; chunk < n_chunks; ++chunk) {
    const int64_t t0 = bos + int64_t(chunk) * kC;
    const int L = int(eos - t0 < kC ? eos - t0 : kC);
    const int stg = chunk & 1;
    uint8_t *st = sm + OFF_STAGE + stg * kStageBytes;
    const uint32_t st_addr = sbase + OFF_STAGE + stg * kStageBytes;

    // ---------------- 1. decay factors and operand tiles ----------------
    float b_pref = 0.f;
    if (tid < L) b_pref = beta[(t0 + tid) * H + h];
    bad |= !mbar_wait(&bar_in[stg], uint32_t((chunk >> 1) & 1), err_word, DEVERR_TMA_TIMEOUT);
    inflight[stg] = -1;
    {
      const int c = tid & 127, s = tid >> 7;  // channel c, subtile s
      const float *gin = reinterpret_cast<const float *>(st + SG);
      float e1[16], e2[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = 16 * s + j;
        e1[j] = t < L ? __expf(clamp_log_decay(gin[t * kD + c], lb)) : 1.f;  // alpha for now
      }
      // e2[j] = prod_{i > j} alpha_i ; e1[j] = prod_{i <= j} alpha_i (inside the subtile)
      e2[15] = 1.f;
#pragma unroll
      for (int j = 14; j >= 0; --j) e2[j] = e2[j + 1] * e1[j + 1];
#pragma unroll
      for (int j = 1; j < 16; ++j) e1[j] *= e1[j - 1];
      s_tau[s * kD + c] = e1[15];
      if (tid < kC) s_beta[tid] = b_pref;
      __syncthreads();

      const float tau0 = s_tau[c], tau1 = s_tau[kD + c];
      const float pre = s == 1 ? tau0 : 1.f;   // Gamma at the start of the subtile
      const float post = s == 0 ? tau1 : 1.f;  // decay from the end of the subtile to the chunk end
      const float inv_tau = 1.f / (s == 0 ? tau0 : tau1);
      if (s == 0) s_gamma[c] = tau0 * tau1;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = 16 * s + j;
        float q = 0.f, k = 0.f;
        if (t < L) {
          q = bf16_to_f32(*reinterpret_cast<const uint16_t *>(st + SQ + sw128_offset(t, c, kC)));
          k = bf16_to_f32(*reinterpret_cast<const uint16_t *>(st + SK + sw128_offset(t, c, kC)));
        }
        const float qs = q * e1[j], ks = k * e1[j], kb = k * e2[j];
        // Gram N side: rows 32 s + j (query) and 32 s + 16 + j (key) of a 64-row tf32 tile
        st_at(gram, G_QK + sw128_offset32(32 * s + j, c, 64), round_tf32(qs));
        st_at(gram, G_QK + sw128_offset32(32 * s + 16 + j, c, 64), round_tf32(ks));
        // Gram M side: B_s holds the keys of subtiles 0..s scaled to subtile s's reference
        if (s == 0) {
          st_at(gram, G_B0 + sw128_offset32(t, c, 16), round_tf32(kb * inv_tau));
          st_at(gram, G_B1 + sw128_offset32(t, c, 32), round_tf32(kb));
        } else {
          st_at(gram, G_B1 + sw128_offset32(t, c, 32), round_tf32(kb * inv_tau));
        }
        st_at(sm, OFF_QT + sw128_offset(t, c, kC), f32_to_f16(qs * pre));
        st_at(sm, OFF_KG + sw128_offset(t, c, kC), f32_to_f16(ks * pre));
        st_at(sm, OFF_KH + sw128_offset(t, c, kC), f32_to_f16(kb * post));
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();

    // ---------------- 2. Gram tiles (tf32 tensor cores) ----------------
    if (tid == 0) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const uint32_t rows = 16u * (s + 1);
        const uint32_t a0 = sbase + OFF_GRAM + (s == 0 ? G_B0 : G_B1);
        const uint32_t b0 = sbase + OFF_GRAM + G_QK + 32 * s * 128;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
          umma_tf32(tmem + TM_GRAM + 32 * s, kdesc(a0 + kb * rows * 128 + ko), kdesc(b0 + kb * 64 * 128 + ko),
                    IDESC_GRAM, ks > 0);
        }
      }
      umma_commit(bar_mma);
    }
    bad |= !mbar_wait(bar_mma, mma_phase, err_word, DEVERR_MMA_TIMEOUT);
    mma_phase ^= 1;
    tc_fence_after();

    // ---------------- 3a. P and A out of TMEM ----------------
    // accumulator row i = 16 quarter + lane (M = 64 layout: lanes 0..15 of each quarter);
    // columns 32 s + 0..15 are query rows (P), 32 s + 16..31 key rows (A)
    if (quarter < 2) {
      float *As = reinterpret_cast<float *>(gram + G_A);
      const int i = 16 * quarter + lane;
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        float vals[16];
        tmem_ld16(tmem + lane_base + TM_GRAM + 32 * s + 16 * half, vals);
        tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = 16 * s + j;
            if (half == 0)
              st_at(sm, OFF_P + sw128_offset(t, i, kC), f32_to_f16((i <= t && t < L) ? vals[j] : 0.f));
            else
              As[t * kALd + i] = (i < t && t < L) ? s_beta[t] * vals[j] : 0.f;
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---------------- 3b. T = (I + A)^{-1}, blocked by 16; T' = T Diag(beta) ----------------
    {
      const float *As = reinterpret_cast<const float *>(gram + G_A);
      float *Ts = reinterpret_cast<float *>(gram + G_T);
      float *Xs = reinterpret_cast<float *>(gram + G_X);
      if (warp < 2 && lane < 16) {
        // diagonal block `warp`, column `lane`: forward substitution
        const int s = warp, j = lane;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float acc = (r == j) ? 1.f : 0.f;
#pragma unroll
          for (int m = 0; m < r; ++m) acc = fmaf(-As[(16 * s + r) * kALd + 16 * s + m], x[m], acc);
          x[r] = acc;
          Ts[(16 * s + r) * kALd + 16 * s + j] = acc;
        }
      } else if (warp == 2) {
        for (int e = lane; e < 256; e += 32) Ts[(e >> 4) * kALd + 16 + (e & 15)] = 0.f;  // block above
      }
      __syncthreads();
      const int r = tid >> 4, cc = tid & 15;
      {
        float acc = 0.f;  // X = A_10 T_00
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) acc = fmaf(As[(16 + r) * kALd + kk], Ts[kk * kALd + cc], acc);
        Xs[r * 16 + cc] = acc;
      }
      __syncthreads();
      {
        float acc = 0.f;  // T_10 = -T_11 X
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          if (kk <= r) acc = fmaf(Ts[(16 + r) * kALd + 16 + kk], Xs[kk * 16 + cc], acc);
        Ts[(16 + r) * kALd + cc] = -acc;
      }
      __syncthreads();
      if (tid < 128) {
        const int t = tid >> 2, cj = tid & 3;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = Ts[t * kALd + 8 * cj + e] * s_beta[8 * cj + e];
        st_at(sm, OFF_TP + sw128_chunk(t, cj, 0, 64), pack8_f16(x));
      }
      // v tile: bf16 -> fp16 in place; rows past the sequence end are zeroed
      for (int e = tid; e < kC * 16; e += kThreads) {
        const int t = e >> 4, cj = e & 15;
        uint4 *p = reinterpret_cast<uint4 *>(st + SV + sw128_chunk(t, cj & 7, cj >> 3, kC));
        uint4 w = make_uint4(0, 0, 0, 0);
        if (t < L) {
          const uint4 b = *p;
          float x[8];
          const float2 a0 = unpack_bf16x2(b.x), a1 = unpack_bf16x2(b.y), a2 = unpack_bf16x2(b.z),
                       a3 = unpack_bf16x2(b.w);
          x[0] = a0.x; x[1] = a0.y; x[2] = a1.x; x[3] = a1.y; x[4] = a2.x; x[5] = a2.y; x[6] = a3.x; x[7] = a3.y;
          w = pack8_f16(x);
        }
        *p = w;
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();

    // ---------------- 4. W = T' Kg and U~^T = V^T T'^T (fp16) ----------------
    if (tid == 0) {
      const uint32_t tp = sbase + OFF_TP, kg = sbase + OFF_KG, vin = st_addr + SV;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
        umma_f16(tmem + TM_W, kdesc(tp + ks * 32), mndesc(kg + ks * 2048), IDESC_W, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
        umma_f16(tmem + TM_U, mndesc(vin + ks * 2048), kdesc(tp + ks * 32), IDESC_UT, ks > 0);
      umma_commit(bar_mma);
    }
    bad |= !mbar_wait(bar_mma, mma_phase, err_word, DEVERR_MMA_TIMEOUT);
    mma_phase ^= 1;
    tc_fence_after();
    // the stage is fully consumed: load the chunk after next into it
    if (chunk + 2 < n_chunks) {
      if (tid == 0) issue_stage(chunk + 2);
      inflight[stg] = ((chunk + 2) >> 1) & 1;
    }

    // ---------------- W and S^T to shared memory (fp16) ----------------
    if (quarter < 2) {
      // W rows t = 16 quarter + lane (lane < 16), columns 64 half .. 64 half + 63
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float vals[16];
        tmem_ld16(tmem + lane_base + TM_W + 64 * half + 16 * u, vals);
        tmem_ld_wait();
        if (lane < 16) {
          const int t = 16 * quarter + lane;
          st_at(gram, G_W + sw128_chunk(t, 2 * u, half, kC), pack8_f16(vals));
          st_at(gram, G_W + sw128_chunk(t, 2 * u + 1, half, kC), pack8_f16(vals + 8));
        }
      }
    }
#pragma unroll
    for (int cj = 0; cj < 8; ++cj) st_at(gram, G_ST + sw128_chunk(v_own, cj, half, 128), pack8_f16(S + 8 * cj));
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---------------- 5. state-dependent chain (fp16) ----------------
    if (tid == 0) {
      const uint32_t stt = sbase + OFF_GRAM + G_ST, w = sbase + OFF_GRAM + G_W, qt = sbase + OFF_QT;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {  // U^T = U~^T - S^T W^T
        const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
        umma_f16(tmem + TM_U, kdesc(stt + kb * 16384 + ko), kdesc(w + kb * 4096 + ko), IDESC_SW_NEG, 1);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {  // O^T = S^T Q~^T
        const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
        umma_f16(tmem + TM_O, kdesc(stt + kb * 16384 + ko), kdesc(qt + kb * 4096 + ko), IDESC_O, ks > 0);
      }
      umma_commit(bar_mma);
    }
    bad |= !mbar_wait(bar_mma, mma_phase, err_word, DEVERR_MMA_TIMEOUT);
    mma_phase ^= 1;
    tc_fence_after();
    {
      // U^T row v_own, columns t in [16 half, 16 half + 16) -> fp16 K-major [v][i]
      float vals[16];
      tmem_ld16(tmem + lane_base + TM_U + 16 * half, vals);
      tmem_ld_wait();
      st_at(gram, G_UT + sw128_chunk(v_own, 2 * half, 0, 128), pack8_f16(vals));
      st_at(gram, G_UT + sw128_chunk(v_own, 2 * half + 1, 0, 128), pack8_f16(vals + 8));
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();
    if (tid == 0) {
      const uint32_t ut = sbase + OFF_GRAM + G_UT, pp = sbase + OFF_P, kh = sbase + OFF_KH;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)  // O^T += U^T P^T
        umma_f16(tmem + TM_O, kdesc(ut + ks * 32), kdesc(pp + ks * 32), IDESC_O, 1);
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)  // dS^T = U^T K^
        umma_f16(tmem + TM_DS, kdesc(ut + ks * 32), mndesc(kh + ks * 2048), IDESC_DS, ks > 0);
      umma_commit(bar_mma);
    }
    bad |= !mbar_wait(bar_mma, mma_phase, err_word, DEVERR_MMA_TIMEOUT);
    mma_phase ^= 1;
    tc_fence_after();
    {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float vals[16];
        tmem_ld16(tmem + lane_base + TM_DS + 64 * half + 16 * u, vals);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) S[16 * u + j] = fmaf(s_gamma[64 * half + 16 * u + j], S[16 * u + j], vals[j]);
      }
      float vals[16];
      tmem_ld16(tmem + lane_base + TM_O + 16 * half, vals);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = 16 * half + j;
        if (t < L) store_elem<kOutBF16>(out, ((t0 + t) * H + h) * int64_t(kD) + v_own, scale * vals[j]);
      }
    }
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();
  }

  if (final_state != nullptr) {
#pragma unroll
    for (int j = 0; j < 64; ++j) final_state[st_base + int64_t(64 * half + j) * kD + v_own] = S[j];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
  return;

abort:
  // a bounded wait gave up: let this CTA's own copies in flight land (bounded), release TMEM
  if (tid == 0) {
    for (int s = 0; s < 2; ++s)
      if (inflight[s] >= 0) mbar_wait(&bar_in[s], uint32_t(inflight[s]), err_word, DEVERR_TMA_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
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

// 3-D map over a token-major [T, H, 128] tensor: dims (channel, head, token); boxes of
// 32 tokens x 64 channels (bf16, 128-byte swizzle) or 32 tokens x 128 channels (fp32).
bool make_map(CUtensorMap *map, const void *base, bool bf16, int64_t T, int H) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const uint64_t es = bf16 ? 2 : 4;
  const cuuint64_t dims[3] = {cuuint64_t(kD), cuuint64_t(H), cuuint64_t(T)};
  const cuuint64_t strides[2] = {cuuint64_t(kD * es), cuuint64_t(H) * kD * es};
  const cuuint32_t box[3] = {bf16 ? 64u : 128u, 1u, cuuint32_t(kC)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                        const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        bf16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

bool chunked_supported(int d_k, int d_v, bool in_bf16, float lb) {
  return in_bf16 && d_k == kD && d_v == kD && lb >= -5.0f;
}

kda_status launch_chunked(const void *q, const void *k, const void *v, const float *log_alpha, const float *beta,
                          const int32_t *cu_seqlens, int num_seqs, int64_t total_tokens, int H, bool out_bf16,
                          float lb, float scale, const float *init_state, void *out, float *final_state,
                          cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mg;
  if (!make_map(&mq, q, true, total_tokens, H) || !make_map(&mk, k, true, total_tokens, H) ||
      !make_map(&mv, v, true, total_tokens, H) || !make_map(&mg, log_alpha, false, total_tokens, H))
    return KDA_ERR_CUDA;
  auto kern = out_bf16 ? kda_chunked_kernel<true> : kda_chunked_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes)) != cudaSuccess)
    return KDA_ERR_CUDA;
  const dim3 grid(unsigned(int64_t(num_seqs) * H)), block(kThreads);
  kern<<<grid, block, kSmemBytes, stream>>>(mq, mk, mv, mg, beta, cu_seqlens, init_state, out, final_state, H, lb,
                                            scale, device_error_word());
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
