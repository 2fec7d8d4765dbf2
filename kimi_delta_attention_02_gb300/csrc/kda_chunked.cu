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
// fp32 throughout and the state is kept in fp32 (tensor memory).
//
// Layout of the work. One CTA per (sequence, head) chain: 16 compute warps and one
// issuing warp (one thread of it issues every TMA load and tensor-core MMA, so the
// ~90 cycles each MMA issue takes never holds up the compute warps). The fp32
// state S^T (rows v = value channels, columns c = key channels) stays in tensor
// memory for the whole sequence. Each iteration j runs the state chain of chunk
// j interleaved with the state-independent work of chunk j+1, so that each
// tensor-core group runs while the threads work on the other stream:
//   P1  chain j : fp16 copy of S^T, S^T <- S^T Diag(Gamma_j) in place;
//                 MMA1: [U^T | O^T] += S^T [-W^T | Q~^T]              (N = 64)
//   P2  next j+1: decay scan (shuffles), operand tiles; Gram (kind::tf32,
//                 M = 64 query/key rows x N = 48 keys under the two references)
//   P3  chain j : U^T to fp16; MMA2: O^T += U^T P^T, S^T += U^T K^     (N = 32, 128)
//   P4  next j+1: P and A out of TMEM, fp32 inverse of I + A (one warp), T',
//                 v -> fp16; W^T = Kg^T T'^T and [U~^T | 0] = V^T [T'; 0]^T
//   P5  chain j : O^T out of TMEM to global memory
//   P6  next j+1: -W^T into the [-W^T | Q~^T] tile
// Per-chunk operand tiles are double-buffered by chunk parity. TMA brings q, k
// and log-decay one chunk ahead and v two chunks ahead (128-byte swizzle).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kC = 32;      // chunk length (two 16-token subtiles)
constexpr int kD = 128;     // d_k = d_v
constexpr int kWorkers = 512;               // 16 compute warps
constexpr int kThreads = kWorkers + 32;     // + one warp that issues TMA loads and MMAs
constexpr int kALd = 36;    // fp32 row stride of the A / T scratch

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_QKG = 0;              // q [32][128] bf16 | k | log-decay [32][128] fp32
constexpr uint32_t SQ = 0, SK = 8 * 1024, SG = 16 * 1024;
constexpr uint32_t OFF_V = 32 * 1024;        // two v stages [32][128] bf16, converted to fp16 in place
constexpr uint32_t OFF_QK = 48 * 1024;       // Gram A side: tf32 [64 rows][128] (rows 32 s..: 16 query, 16 key)
constexpr uint32_t OFF_B = 80 * 1024;        // Gram B side: tf32 [48 rows][128] (0..15: r_0, 16..47: r_1)
constexpr uint32_t OFF_ST = 104 * 1024;      // S^T fp16 [128][128]; the inverse's fp32 A, T, X alias it
constexpr uint32_t G_A = 0, G_T = 5 * 1024, G_X = 10 * 1024;
constexpr uint32_t OFF_UT = 136 * 1024;      // U^T fp16 [128][32], 64-byte swizzle
constexpr uint32_t OFF_TP = 144 * 1024;      // T' fp16 [64][32], 64-byte swizzle; rows 32..63 stay zero
constexpr uint32_t OFF_KG = 148 * 1024;      // K * Gamma fp16 [32 i][128 c] (MN-major A of W^T)
constexpr uint32_t OFF_WQ = 156 * 1024;      // 2 x [-W^T | Q~^T] fp16 [128 c][64] (MN-major B of MMA1)
constexpr uint32_t kWQBytes = 16 * 1024;
constexpr uint32_t OFF_PK = 188 * 1024;      // 2 x [P ; K^^T] fp16 [160 rows][32], 64-byte swizzle
constexpr uint32_t kPKBytes = 10 * 1024;
constexpr uint32_t OFF_MISC = 208 * 1024;    // beta, Gamma_last x2, subtile totals, barriers
constexpr uint32_t kSmemBytes = 212 * 1024 + 1024;

// TMEM columns: Gram | W^T | [U^T | O^T] x 2 | S^T
constexpr uint32_t TM_GRAM = 0, TM_W = 64, TM_UO = 128, TM_S = 256, TM_COLS = 512;
__device__ __forceinline__ uint32_t tm_uo(int b) { return TM_UO + 64u * uint32_t(b); }

constexpr uint32_t IDESC_GRAM = umma_idesc(UMMA_TF32, 64, 48, false, false, false);
constexpr uint32_t IDESC_WT = umma_idesc(UMMA_F16, 128, 32, true, false, false);   // W^T = Kg^T T'^T
constexpr uint32_t IDESC_UT = umma_idesc(UMMA_F16, 128, 64, true, false, false);   // [U~^T | 0] = V^T [T'; 0]^T
constexpr uint32_t IDESC_UO = umma_idesc(UMMA_F16, 128, 64, false, true, false);   // += S^T [-W^T | Q~^T]
constexpr uint32_t IDESC_O2 = umma_idesc(UMMA_F16, 128, 32, false, false, false);  // O^T += U^T P^T
constexpr uint32_t IDESC_S2 = umma_idesc(UMMA_F16, 128, 128, false, false, false); // S^T += U^T K^

__device__ __forceinline__ uint64_t kdesc128(uint32_t addr) { return umma_desc(addr, 16, 1024, kSwizzle128B); }
__device__ __forceinline__ uint64_t kdesc64(uint32_t addr) { return umma_desc(addr, 16, 512, kSwizzle64B); }
__device__ __forceinline__ uint64_t mndesc(uint32_t addr, uint32_t lbo) {
  return umma_desc(addr, lbo, 1024, kSwizzle128B);
}
// Advance a descriptor's start address by `bytes` (shared-memory addresses here stay below
// 2^18, so the 14-bit address field never carries into the next field).
__device__ __forceinline__ uint64_t dadv(uint64_t desc, uint32_t bytes) { return desc + uint64_t(bytes >> 4); }

template <typename T>
__device__ __forceinline__ void st_at(uint8_t *base, uint32_t off, T v) {
  *reinterpret_cast<T *>(base + off) = v;
}
__device__ __forceinline__ uint4 pack8_f16(const float *x) {
  return make_uint4(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]), pack_f16x2(x[4], x[5]), pack_f16x2(x[6], x[7]));
}
// byte offset of the 16-byte group holding fp32 elements (row, c0..c0+3) in a 128-byte
// swizzled tf32 tile of `rows` rows (32 elements per 128-byte row)
__device__ __forceinline__ uint32_t tf32_quad(uint32_t row, uint32_t c0, uint32_t rows) {
  return (c0 >> 5) * rows * 128u + row * 128u + (((((c0 & 31u) >> 2) ^ row) & 7u) << 4);
}

struct Bars {
  uint64_t qkg, v[2], mma1, gram, mma2, wu;
};

template <bool kOutBF16>
__global__ void __launch_bounds__(kThreads, 1)
    kda_chunked_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                       const float *__restrict__ beta, const int32_t *__restrict__ cu_seqlens,
                       const float *__restrict__ init_state, void *__restrict__ out,
                       float *__restrict__ final_state, int H, float lb, float scale, uint32_t *err_word) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *s_beta = reinterpret_cast<float *>(sm + OFF_MISC);  // [32] of the chunk being prepared
  float *s_gamma = s_beta + 32;                               // [2][128] Gamma_last by chunk parity
  float *s_tau = s_gamma + 2 * 128;                           // [2][128] subtile totals
  Bars *bars = reinterpret_cast<Bars *>(s_tau + 2 * 128);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, grp = warp >> 2;  // TMEM lane quarter, column group (compute warps)
  const bool issuer = tid == kWorkers;             // lane 0 of warp 16
  const bool worker = tid < kWorkers;
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
    mbar_init(&bars->qkg, 1);
    mbar_init(&bars->v[0], 1);
    mbar_init(&bars->v[1], 1);
    mbar_init(&bars->mma1, 1);
    mbar_init(&bars->gram, 1);
    mbar_init(&bars->mma2, 1);
    mbar_init(&bars->wu, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, TM_COLS);
    tmem_relinquish();
  }
  // rows 32..63 of the T' tile stay zero: the U~ product reads them to clear the O^T columns
  for (int e = tid; e < 32 * 4; e += kThreads)
    st_at(sm, OFF_TP + sw64_chunk(32 + (e >> 2), e & 3), make_uint4(0, 0, 0, 0));

  const int v_own = 32 * quarter + lane;  // state row (TMEM lane) of this thread
  const int64_t st_base = (n * H + h) * int64_t(kD) * kD;

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_base = uint32_t(32 * quarter) << 16;
  const uint32_t s_cols = tmem + lane_base + TM_S + 32 * grp;  // this thread's 32 state columns
  if (worker) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float x[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        x[j] = init_state != nullptr ? init_state[st_base + int64_t(32 * grp + 16 * u + j) * kD + v_own] : 0.f;
      tmem_st16(s_cols + 16 * u, x);
    }
    tmem_st_wait();
  }

  auto chunk_t0 = [&](int c) { return bos + int64_t(c) * kC; };
  auto chunk_len = [&](int c) {
    const int64_t r = eos - chunk_t0(c);
    return int(r < kC ? r : kC);
  };
  auto issue_qkg = [&](int c) {  // issuer
    const int32_t t0 = int32_t(chunk_t0(c));
    mbar_arrive_expect_tx(&bars->qkg, 2 * 8192 + 16384);
    tma_load_3d(sm + OFF_QKG + SQ, &tm_q, &bars->qkg, 0, h, t0);
    tma_load_3d(sm + OFF_QKG + SQ + 4096, &tm_q, &bars->qkg, 64, h, t0);
    tma_load_3d(sm + OFF_QKG + SK, &tm_k, &bars->qkg, 0, h, t0);
    tma_load_3d(sm + OFF_QKG + SK + 4096, &tm_k, &bars->qkg, 64, h, t0);
    tma_load_3d(sm + OFF_QKG + SG, &tm_g, &bars->qkg, 0, h, t0);
  };
  auto issue_v = [&](int c) {  // issuer
    const int32_t t0 = int32_t(chunk_t0(c));
    uint8_t *dst = sm + OFF_V + (c & 1) * 8192;
    mbar_arrive_expect_tx(&bars->v[c & 1], 8192);
    tma_load_3d(dst, &tm_v, &bars->v[c & 1], 0, h, t0);
    tma_load_3d(dst + 4096, &tm_v, &bars->v[c & 1], 64, h, t0);
  };

  bool bad = false;
  // chunk index of a TMA load issued and not yet waited for (-1: none); tracked by every thread
  int qkg_inflight = -1, v_inflight[2] = {-1, -1};
  if (n_chunks > 0) {
    if (issuer) issue_qkg(0);
    qkg_inflight = 0;
  }
  for (int c = 0; c < 2 && c < n_chunks; ++c) {
    if (issuer) issue_v(c);
    v_inflight[c] = c;
  }
  float b_next = (tid < kC && tid < eos - bos) ? beta[(bos + tid) * H + h] : 0.f;  // beta of chunk 0

  // ------------------------------------------------------------------ P2: operand tiles
  auto prep = [&](int c) {
    const int b = c & 1, L = chunk_len(c);
    const int64_t t0 = chunk_t0(c);
    const float b_pref = b_next;
    if (tid < kC) b_next = (tid < eos - t0 - kC) ? beta[(t0 + kC + tid) * H + h] : 0.f;  // next chunk's
    bad |= !mbar_wait_sleep(&bars->qkg, uint32_t(c & 1), err_word, DEVERR_TMA_TIMEOUT);
    qkg_inflight = -1;
    // warp: subtile s = warp / 8, channels 16 (warp % 8) .. +15; lane: token pair tp = lane % 8
    // (tokens 16 s + 2 tp, +1), channel quad cg = lane / 8 (channels c0 .. c0 + 3); compute warps only
    const int s = (warp >> 3) & 1, tp = lane & 7, cg = lane >> 3;
    const int c0 = 16 * (warp & 7) + 4 * cg, tb = 16 * s + 2 * tp;
    const float *gin = reinterpret_cast<const float *>(sm + OFF_QKG + SG);
    float a[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float4 g = worker ? *reinterpret_cast<const float4 *>(gin + (tb + r) * kD + c0)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
      const bool ok = tb + r < L;
      a[r][0] = ok ? __expf(clamp_log_decay(g.x, lb)) : 1.f;
      a[r][1] = ok ? __expf(clamp_log_decay(g.y, lb)) : 1.f;
      a[r][2] = ok ? __expf(clamp_log_decay(g.z, lb)) : 1.f;
      a[r][3] = ok ? __expf(clamp_log_decay(g.w, lb)) : 1.f;
    }
    // e1 = product of alpha over the subtile up to and including the token, e2 = product over
    // the tokens after it; scans over the 8 lanes of a token-pair group
    float e1[2][4], e2[2][4], tau[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float tot = a[0][e] * a[1][e];
      float inc = tot;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        const float up = __shfl_up_sync(0xffffffffu, inc, o, 8);
        if (tp >= o) inc *= up;
      }
      float ex = __shfl_up_sync(0xffffffffu, inc, 1, 8);
      if (tp == 0) ex = 1.f;
      float sinc = tot;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        const float dn = __shfl_down_sync(0xffffffffu, sinc, o, 8);
        if (tp + o < 8) sinc *= dn;
      }
      float sex = __shfl_down_sync(0xffffffffu, sinc, 1, 8);
      if (tp == 7) sex = 1.f;
      tau[e] = __shfl_sync(0xffffffffu, inc, (lane & ~7) | 7, 32);
      e1[0][e] = ex * a[0][e];
      e1[1][e] = ex * tot;
      e2[0][e] = sex * a[1][e];
      e2[1][e] = sex;
    }
    if (worker && tp == 0)
      *reinterpret_cast<float4 *>(s_tau + s * kD + c0) = make_float4(tau[0], tau[1], tau[2], tau[3]);
    if (tid < kC) s_beta[tid] = b_pref;
    __syncthreads();
    if (!worker) return;
    const float4 t0v = *reinterpret_cast<const float4 *>(s_tau + c0);
    const float4 t1v = *reinterpret_cast<const float4 *>(s_tau + kD + c0);
    const float tau0[4] = {t0v.x, t0v.y, t0v.z, t0v.w}, tau1[4] = {t1v.x, t1v.y, t1v.z, t1v.w};
    float pre[4], post[4], inv_tau[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      pre[e] = s == 1 ? tau0[e] : 1.f;   // Gamma at the start of the subtile
      post[e] = s == 0 ? tau1[e] : 1.f;  // decay from the end of the subtile to the chunk end
      inv_tau[e] = __fdividef(1.f, s == 0 ? tau0[e] : tau1[e]);
    }
    if (s == 0 && tp == 0)
      *reinterpret_cast<float4 *>(s_gamma + b * kD + c0) =
          make_float4(tau0[0] * tau1[0], tau0[1] * tau1[1], tau0[2] * tau1[2], tau0[3] * tau1[3]);
    const uint32_t j16 = uint32_t((c0 & 63) >> 3), sub16 = uint32_t(c0 & 4) * 2, blk16 = uint32_t(c0 >> 6);
    float qt_col[4][2], kh_col[4][2];  // [channel][token] for the transposed tiles
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int t = tb + r;
      float q[4] = {0.f, 0.f, 0.f, 0.f}, k[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t off16 = blk16 * (kC * 128) + t * 128 + (((j16 ^ t) & 7u) << 4) + sub16;
      if (t < L) {
        const uint2 qb = *reinterpret_cast<const uint2 *>(sm + OFF_QKG + SQ + off16);
        const uint2 kb2 = *reinterpret_cast<const uint2 *>(sm + OFF_QKG + SK + off16);
        const float2 q01 = unpack_bf16x2(qb.x), q23 = unpack_bf16x2(qb.y);
        const float2 k01 = unpack_bf16x2(kb2.x), k23 = unpack_bf16x2(kb2.y);
        q[0] = q01.x; q[1] = q01.y; q[2] = q23.x; q[3] = q23.y;
        k[0] = k01.x; k[1] = k01.y; k[2] = k23.x; k[3] = k23.y;
      }
      float qs[4], ks[4], kb[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qs[e] = q[e] * e1[r][e];
        ks[e] = k[e] * e1[r][e];
        kb[e] = k[e] * e2[r][e];
        qt_col[e][r] = qs[e] * pre[e];
        kh_col[e][r] = kb[e] * post[e];
      }
      auto f4 = [](float x0, float x1, float x2, float x3) {
        return make_float4(round_tf32(x0), round_tf32(x1), round_tf32(x2), round_tf32(x3));
      };
      st_at(sm, OFF_QK + tf32_quad(32 * s + 2 * tp + r, c0, 64), f4(qs[0], qs[1], qs[2], qs[3]));
      st_at(sm, OFF_QK + tf32_quad(32 * s + 16 + 2 * tp + r, c0, 64), f4(ks[0], ks[1], ks[2], ks[3]));
      if (s == 0) {
        st_at(sm, OFF_B + tf32_quad(t, c0, 48),
              f4(kb[0] * inv_tau[0], kb[1] * inv_tau[1], kb[2] * inv_tau[2], kb[3] * inv_tau[3]));
        st_at(sm, OFF_B + tf32_quad(16 + t, c0, 48), f4(kb[0], kb[1], kb[2], kb[3]));
      } else {
        st_at(sm, OFF_B + tf32_quad(16 + t, c0, 48),
              f4(kb[0] * inv_tau[0], kb[1] * inv_tau[1], kb[2] * inv_tau[2], kb[3] * inv_tau[3]));
      }
      st_at(sm, OFF_KG + off16,
            make_uint2(pack_f16x2(ks[0] * pre[0], ks[1] * pre[1]), pack_f16x2(ks[2] * pre[2], ks[3] * pre[3])));
    }
    // transposed tiles, per channel the 2 tokens of this thread: Q~^T into columns 32 + t of
    // [-W^T | Q~^T], K^^T into row 32 + c of [P ; K^^T]
    uint8_t *wq = sm + OFF_WQ + b * kWQBytes;
    uint8_t *pk = sm + OFF_PK + b * kPKBytes;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t c = uint32_t(c0 + e);
      const uint32_t col = 32u + uint32_t(tb);
      st_at(wq, c * 128 + ((((col >> 3) ^ c) & 7u) << 4) + (col & 7u) * 2, pack_f16x2(qt_col[e][0], qt_col[e][1]));
      st_at(pk, sw64_offset(32 + c, uint32_t(tb)), pack_f16x2(kh_col[e][0], kh_col[e][1]));
    }
  };

  auto issue_gram = [&]() {  // issuer
    const uint64_t qk = kdesc128(sbase + OFF_QK), bb = kdesc128(sbase + OFF_B);
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
      umma_tf32(tmem + TM_GRAM, dadv(qk, kb * 64 * 128 + ko), dadv(bb, kb * 48 * 128 + ko), IDESC_GRAM, ks > 0);
    }
    umma_commit(&bars->gram);
  };

  // ------------------------------------------------------------------ P4: P, A, inverse, T', v
  auto extract_inverse = [&](int c) {
    const int b = c & 1, L = chunk_len(c);
    bad |= !mbar_wait_sleep(&bars->gram, uint32_t(c & 1), err_word, DEVERR_MMA_TIMEOUT);
    tc_fence_after();
    // Gram row t' = 16 quarter + lane (M = 64 layout, lanes 0..15 of each quarter): quarters
    // 0 / 2 hold the query rows of subtile 0 / 1 (P), quarters 1 / 3 the key rows (A)
    uint8_t *pk = sm + OFF_PK + b * kPKBytes;
    float *As = reinterpret_cast<float *>(sm + OFF_ST + G_A);
    if (grp < 2) {
      const int s = quarter >> 1, part = grp, t = 16 * s + (lane & 15);
      const bool is_p = (quarter & 1) == 0, have = part <= s;
      float vals[16];
      if (have) {
        tmem_ld16(tmem + lane_base + TM_GRAM + (s == 0 ? 0 : 16) + 16 * part, vals);
        tmem_ld_wait();
      }
      if (lane < 16) {
        const float bt = s_beta[t];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int i = 16 * part + e;
          const bool keep = have && t < L && (is_p ? i <= t : i < t);
          vals[e] = keep ? (is_p ? vals[e] : bt * vals[e]) : 0.f;
        }
        if (is_p) {
          st_at(pk, sw64_chunk(t, 2 * part), pack8_f16(vals));
          st_at(pk, sw64_chunk(t, 2 * part + 1), pack8_f16(vals + 8));
        } else {
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4)
            *reinterpret_cast<float4 *>(As + t * kALd + 16 * part + 4 * i4) =
                make_float4(vals[4 * i4], vals[4 * i4 + 1], vals[4 * i4 + 2], vals[4 * i4 + 3]);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    float *Ts = reinterpret_cast<float *>(sm + OFF_ST + G_T);
    float *Xs = reinterpret_cast<float *>(sm + OFF_ST + G_X);
    if (warp == 0) {
      // T = (I + A)^{-1}: lanes 0..15 column `lane` of diagonal block 0, lanes 16..31 of block 1
      // (right-looking forward substitution); the block below the diagonal follows
      const int s = lane >> 4, j = lane & 15;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        Ts[(16 * s + m) * kALd + 16 * s + j] = x[m];
#pragma unroll
        for (int r = m + 1; r < 16; ++r) x[r] = fmaf(-As[(16 * s + r) * kALd + 16 * s + m], x[m], x[r]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) Ts[(lane >> 1) * kALd + 16 + 8 * (lane & 1) + e] = 0.f;  // block above
    } else if (worker) {
      // v tile of this chunk: bf16 -> fp16 in place, rows past the sequence end zeroed
      bad |= !mbar_wait_sleep(&bars->v[b], uint32_t((c >> 1) & 1), err_word, DEVERR_TMA_TIMEOUT);
      uint8_t *vt = sm + OFF_V + b * 8192;
      for (int e = tid - 32; e < kC * 16; e += kWorkers - 32) {
        const int t = e >> 4, cj = e & 15;
        uint4 *p = reinterpret_cast<uint4 *>(vt + sw128_chunk(t, cj & 7, cj >> 3, kC));
        uint4 w = make_uint4(0, 0, 0, 0);
        if (t < L) {
          const uint4 bv = *p;
          const float2 a0 = unpack_bf16x2(bv.x), a1 = unpack_bf16x2(bv.y), a2 = unpack_bf16x2(bv.z),
                       a3 = unpack_bf16x2(bv.w);
          const float x[8] = {a0.x, a0.y, a1.x, a1.y, a2.x, a2.y, a3.x, a3.y};
          w = pack8_f16(x);
        }
        *p = w;
      }
    }
    v_inflight[b] = -1;
    __syncthreads();
    {
      // T_10 = -T_11 (A_10 T_00): thread (r, col) of the 16 x 16 block on warps 0..7
      const int r = (tid >> 4) & 15, col = tid & 15;
      float xv = 0.f;
      if (tid < 256) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) xv = fmaf(As[(16 + r) * kALd + kk], Ts[kk * kALd + col], xv);
        Xs[r * 16 + col] = xv;
      }
      __syncthreads();
      if (tid < 256) {
        xv = 0.f;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          if (kk <= r) xv = fmaf(Ts[(16 + r) * kALd + 16 + kk], Xs[kk * 16 + col], xv);
        Ts[(16 + r) * kALd + col] = -xv;
      }
      __syncthreads();
    }
    if (tid < 128) {  // T' = T Diag(beta) -> fp16 [t][i]
      const int t = tid >> 2, cj = tid & 3;
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = Ts[t * kALd + 8 * cj + e] * s_beta[8 * cj + e];
      st_at(sm, OFF_TP + sw64_chunk(t, cj), pack8_f16(x));
    }
  };

  auto issue_wu = [&](int c) {  // issuer: W^T and [U~^T | 0]
    const int b = c & 1;
    const uint64_t tp = kdesc64(sbase + OFF_TP), kg = mndesc(sbase + OFF_KG, kC * 128),
                   vin = mndesc(sbase + OFF_V + b * 8192, kC * 128);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      umma_f16(tmem + TM_W, dadv(kg, ks * 2048), dadv(tp, ks * 32), IDESC_WT, ks > 0);
      umma_f16(tmem + tm_uo(b), dadv(vin, ks * 2048), dadv(tp, ks * 32), IDESC_UT, ks > 0);
    }
    umma_commit(&bars->wu);
  };

  // ------------------------------------------------------------------ P6: -W^T
  auto wt_extract = [&](int c) {
    const int b = c & 1;
    bad |= !mbar_wait_sleep(&bars->wu, uint32_t(c & 1), err_word, DEVERR_MMA_TIMEOUT);
    tc_fence_after();
    if (c + 2 < n_chunks) {  // the v stage of chunk c is consumed: load chunk c + 2 into it
      if (issuer) issue_v(c + 2);
      v_inflight[b] = c + 2;
    }
    if (!worker) return;
    float x[8];
    tmem_ld8(tmem + lane_base + TM_W + 8 * grp, x);  // W^T row c = v_own, columns t = 8 grp ..
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = -x[e];
    const uint32_t cr = uint32_t(v_own);
    st_at(sm + OFF_WQ + b * kWQBytes, cr * 128 + (((uint32_t(grp) ^ cr) & 7u) << 4), pack8_f16(x));
  };

  // ------------------------------------------------------------------ prologue: chunk 0's operands
  if (n_chunks > 0) {
    prep(0);
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();
    if (n_chunks > 1) {
      if (issuer) issue_qkg(1);
      qkg_inflight = 1;
    }
    if (issuer) issue_gram();
    extract_inverse(0);
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();
    if (issuer) issue_wu(0);
    wt_extract(0);
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();
  }

  for (int j = 0; j < n_chunks; ++j) {
    const int b = j & 1;
    const bool more = j + 1 < n_chunks;
    // ---------------- P1: chain j, fp16 copy of S^T and decay in place; MMA1
    if (worker) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float x[16];
        tmem_ld16(s_cols + 16 * u, x);
        tmem_ld_wait();
        const uint32_t col = uint32_t(32 * grp + 16 * u);  // state column c of x[0]
        st_at(sm + OFF_ST, sw128_chunk(v_own, (col & 63u) >> 3, col >> 6, 128), pack8_f16(x));
        st_at(sm + OFF_ST, sw128_chunk(v_own, ((col & 63u) >> 3) + 1, col >> 6, 128), pack8_f16(x + 8));
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] *= s_gamma[b * kD + col + e];
        tmem_st16(s_cols + 16 * u, x);
      }
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();
    if (issuer) {
      const uint64_t st = kdesc128(sbase + OFF_ST), wq = mndesc(sbase + OFF_WQ + b * kWQBytes, 128 * 128);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {  // [U^T | O^T] += S^T [-W^T | Q~^T]
        const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
        umma_f16(tmem + tm_uo(b), dadv(st, kb * 16384 + ko), dadv(wq, ks * 2048), IDESC_UO, 1);
      }
      umma_commit(&bars->mma1);
    }
    // ---------------- P2: operand tiles of chunk j + 1; Gram
    if (more) {
      prep(j + 1);
      fence_proxy_async_smem();
      tc_fence_before();
      if (__syncthreads_or(bad)) goto abort;
      tc_fence_after();
      if (j + 2 < n_chunks) {
        if (issuer) issue_qkg(j + 2);
        qkg_inflight = j + 2;
      }
      if (issuer) issue_gram();
    }
    // ---------------- P3: chain j, U^T to fp16; MMA2
    bad |= !mbar_wait_sleep(&bars->mma1, uint32_t(j & 1), err_word, DEVERR_MMA_TIMEOUT);
    tc_fence_after();
    if (worker) {
      float x[8];
      tmem_ld8(tmem + lane_base + tm_uo(b) + 8 * grp, x);  // U^T row v, columns t = 8 grp ..
      tmem_ld_wait();
      st_at(sm + OFF_UT, sw64_chunk(uint32_t(v_own), uint32_t(grp)), pack8_f16(x));
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();
    if (issuer) {
      const uint64_t ut = kdesc64(sbase + OFF_UT), pk = kdesc64(sbase + OFF_PK + b * kPKBytes);
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {  // O^T += U^T P^T ; S^T += U^T K^
        umma_f16(tmem + tm_uo(b) + 32, dadv(ut, ks * 32), dadv(pk, ks * 32), IDESC_O2, 1);
        umma_f16(tmem + TM_S, dadv(ut, ks * 32), dadv(pk, 32 * 64 + ks * 32), IDESC_S2, 1);
      }
      umma_commit(&bars->mma2);
    }
    // ---------------- P4: P, A, inverse, T', v of chunk j + 1; W^T and U~^T
    if (more) {
      extract_inverse(j + 1);
      fence_proxy_async_smem();
      tc_fence_before();
      if (__syncthreads_or(bad)) goto abort;
      tc_fence_after();
      if (issuer) issue_wu(j + 1);
    }
    // ---------------- P5: chain j, outputs
    bad |= !mbar_wait_sleep(&bars->mma2, uint32_t(j & 1), err_word, DEVERR_MMA_TIMEOUT);
    tc_fence_after();
    if (worker) {
      const int L = chunk_len(j);
      const int64_t t0 = chunk_t0(j);
      float x[8];
      tmem_ld8(tmem + lane_base + tm_uo(b) + 32 + 8 * grp, x);  // O^T row v, tokens 8 grp ..
      tmem_ld_wait();
      int64_t idx = ((t0 + 8 * grp) * H + h) * int64_t(kD) + v_own;
      const int64_t step = int64_t(H) * kD;
#pragma unroll
      for (int e = 0; e < 8; ++e, idx += step)
        if (8 * grp + e < L) store_elem<kOutBF16>(out, idx, scale * x[e]);
    }
    // ---------------- P6: -W^T of chunk j + 1
    if (more) wt_extract(j + 1);
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();
  }

  if (final_state != nullptr && worker) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float x[16];
      tmem_ld16(s_cols + 16 * u, x);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) final_state[st_base + int64_t(32 * grp + 16 * u + e) * kD + v_own] = x[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
  return;

abort:
  // a bounded wait gave up: let this CTA's own copies in flight land (bounded), release TMEM
  if (issuer) {
    if (qkg_inflight >= 0) mbar_wait_sleep(&bars->qkg, uint32_t(qkg_inflight & 1), err_word, DEVERR_TMA_TIMEOUT);
    for (int s = 0; s < 2; ++s)
      if (v_inflight[s] >= 0)
        mbar_wait_sleep(&bars->v[s], uint32_t((v_inflight[s] >> 1) & 1), err_word, DEVERR_TMA_TIMEOUT);
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
