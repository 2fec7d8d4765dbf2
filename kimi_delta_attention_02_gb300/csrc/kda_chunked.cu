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
// Layout of the work. One CTA (256 threads) per (sequence, head) chain walks
// its 32-token chunks in order. The fp32 state S^T (rows v = value channels,
// columns c = key channels) stays in tensor memory for the whole sequence;
// thread (v = 32 (warp % 4) + lane, half = warp / 4) reads and rewrites its row
// v, columns [64 half, 64 half + 64). Per chunk:
//   1. TMA has landed q, k, v (bf16, 128-byte swizzle) and g (fp32) two chunks
//      ahead. Threads build the decay factors and the operand tiles.
//   2. tcgen05 kind::tf32: Gram tiles per subtile (M=64 query/key rows, N=16/32 keys, K=128).
//   3. Threads read P and A out of tensor memory; SIMT fp32 blocked inverse.
//   4. tcgen05 kind::f16: W^T = Kg^T T'^T and U~^T = V^T T'^T (M=128).
//   5. The state-dependent chain, all M=128 (rows = value channels), two MMA
//      chains into adjacent tensor-memory columns [U^T | O^T | S^T]:
//      [U^T | O^T] += S^T [-W^T | Q~^T]       (N = 64; O^T starts at zero)
//      [O^T | S^T] += U^T [P ; K^^T]^T        (N = 160)
//      with an fp16 copy of S^T as the A operand; the same pass over S^T applies
//      Diag(Gamma_last) in place before the second chain accumulates onto it.
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
//         B tf32 [48 rows][128] at +32 KB (rows 0..15: subtile-0 keys for reference r_0,
//         rows 16..47: all keys for reference r_1)
//   inverse: A fp32 [32][36] at +0, T fp32 at +5 KB, X at +10 KB
//   chain: S^T fp16 [128][128] at +8 KB, U^T fp16 [128][64] at +40 KB
constexpr uint32_t OFF_TP = 140 * 1024;      // T' = T Diag(beta) fp16 [64 rows][64] (rows 32.. stay zero)
constexpr uint32_t OFF_KG = 148 * 1024;      // K * Gamma fp16 [32 i][128 c] (MN-major A of W^T)
constexpr uint32_t OFF_WQ = 156 * 1024;      // [-W^T | Q~^T] fp16 [128 c][64]: MN-major B of U and O
constexpr uint32_t OFF_PK = 172 * 1024;      // [P ; K^^T] fp16 [160 rows][64]: K-major B of O and dS
constexpr uint32_t OFF_MISC = 192 * 1024;    // beta, Gamma_last, subtile totals, barriers
constexpr uint32_t kSmemBytes = 194 * 1024 + 1024;

constexpr uint32_t G_QK = 0, G_B = 32 * 1024;
constexpr uint32_t G_A = 0, G_T = 5 * 1024, G_X = 10 * 1024;
constexpr uint32_t G_ST = 8 * 1024, G_UT = 40 * 1024;

// TMEM columns
constexpr uint32_t TM_GRAM = 0, TM_W = 64, TM_U = 192, TM_O = 224, TM_S = 256, TM_COLS = 512;  // U, O, S adjacent

constexpr uint32_t IDESC_GRAM = umma_idesc(UMMA_TF32, 64, 48, false, false, false);
constexpr uint32_t IDESC_WT = umma_idesc(UMMA_F16, 128, 32, true, false, false);   // W^T = Kg^T T'^T
constexpr uint32_t IDESC_UT = umma_idesc(UMMA_F16, 128, 64, true, false, false);   // [U~^T | 0] = V^T [T'; 0]^T
constexpr uint32_t IDESC_UO = umma_idesc(UMMA_F16, 128, 64, false, true, false);   // += S^T [-W^T | Q~^T]
constexpr uint32_t IDESC_OS = umma_idesc(UMMA_F16, 128, 160, false, false, false); // += U^T [P ; K^^T]^T

constexpr uint32_t kKmajLbo = 16, kSbo = 1024;  // 128-byte swizzle: 8-row atoms of 1 KB
constexpr uint32_t kMnBlock = kC * 128;         // MN-major tiles of 32 rows: next 64-wide block
constexpr uint32_t kMnBlockWQ = kD * 128;       // the [-W^T | Q~^T] tile has 128 rows (one 64-wide block)

__device__ __forceinline__ uint64_t kdesc(uint32_t addr) { return umma_desc(addr, kKmajLbo, kSbo, kSwizzle128B); }
__device__ __forceinline__ uint64_t mndesc(uint32_t addr, uint32_t lbo = kMnBlock) {
  return umma_desc(addr, lbo, kSbo, kSwizzle128B);
}

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

  // state: S^T[v][c] for v = 32 quarter + lane, c = 64 half + j, kept in tensor memory
  const int v_own = 32 * quarter + lane;
  const int64_t st_base = (n * H + h) * int64_t(kD) * kD;

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_base = uint32_t(32 * quarter) << 16;
  const uint32_t s_row = tmem + lane_base + TM_S + 64 * half;  // this thread's 64 state columns
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    float x[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      x[j] = init_state != nullptr ? init_state[st_base + int64_t(64 * half + 16 * u + j) * kD + v_own] : 0.f;
    tmem_st16(s_row + 16 * u, x);
  }
  tmem_st_wait();

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
  // rows 32..63 of the T' tile stay zero: the U~ product reads them to clear the O^T columns
  for (int e = tid; e < 32 * 8; e += kThreads)
    st_at(sm, OFF_TP + sw128_chunk(32 + (e >> 3), e & 7, 0, 64), make_uint4(0, 0, 0, 0));
  // parity of the outstanding load of each stage (-1: none); every thread tracks it
  int inflight[2] = {-1, -1};
  for (int c = 0; c < 2 && c < n_chunks; ++c) {
    if (tid == 0) issue_stage(c);
    inflight[c] = 0;
  }

  uint32_t mma_phase = 0;
  bool bad = false;
  float b_next = (tid < kC && tid < eos - bos) ? beta[(bos + tid) * H + h] : 0.f;  // beta of chunk 0

  for (int chunk = 0; chunk < n_chunks; ++chunk) {
    const int64_t t0 = bos + int64_t(chunk) * kC;
    const int L = int(eos - t0 < kC ? eos - t0 : kC);
    const int stg = chunk & 1;
    uint8_t *st = sm + OFF_STAGE + stg * kStageBytes;
    const uint32_t st_addr = sbase + OFF_STAGE + stg * kStageBytes;

    // ---------------- 1. decay factors and operand tiles ----------------
    const float b_pref = b_next;
    if (tid < kC) b_next = (tid < eos - t0 - kC) ? beta[(t0 + kC + tid) * H + h] : 0.f;  // next chunk's
    bad |= !mbar_wait(&bar_in[stg], uint32_t((chunk >> 1) & 1), err_word, DEVERR_TMA_TIMEOUT);
    inflight[stg] = -1;
    {
      // warp w: subtile s = w / 4, channels 32 (w % 4) .. +31; lane: token quad tq = lane % 4
      // (tokens 16 s + 4 tq .. +3), channel quad cg = lane / 4 (channels c0 = 32 (w % 4) + 4 cg .. +3)
      const int s = warp >> 2, cb = warp & 3, tq = lane & 3, cg = lane >> 2;
      const int c0 = 32 * cb + 4 * cg, tb = 16 * s + 4 * tq;
      const float *gin = reinterpret_cast<const float *>(st + SG);
      float a[4][4];  // [token r][channel e]: alpha, then the running products
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float4 g = *reinterpret_cast<const float4 *>(gin + (tb + r) * kD + c0);
        const bool ok = tb + r < L;
        a[r][0] = ok ? __expf(clamp_log_decay(g.x, lb)) : 1.f;
        a[r][1] = ok ? __expf(clamp_log_decay(g.y, lb)) : 1.f;
        a[r][2] = ok ? __expf(clamp_log_decay(g.z, lb)) : 1.f;
        a[r][3] = ok ? __expf(clamp_log_decay(g.w, lb)) : 1.f;
      }
      // e1 = product of alpha over the subtile up to and including the token,
      // e2 = product over the tokens after it (inside the subtile); scans over the 4 lanes of a quad group
      float e1[4][4], e2[4][4], tau[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = a[0][e], p1 = p0 * a[1][e], p2 = p1 * a[2][e], p3 = p2 * a[3][e];  // local prefix
        const float s3 = 1.f, s2 = a[3][e], s1 = s2 * a[2][e], s0 = s1 * a[1][e];          // local suffix
        // inclusive prefix of the quad totals over tq, then exclusive
        float inc = p3;
        float up = __shfl_up_sync(0xffffffffu, inc, 1, 4);
        if (tq >= 1) inc *= up;
        up = __shfl_up_sync(0xffffffffu, inc, 2, 4);
        if (tq >= 2) inc *= up;
        float ex = __shfl_up_sync(0xffffffffu, inc, 1, 4);
        if (tq == 0) ex = 1.f;
        // inclusive suffix of the quad totals over tq, then exclusive
        float sinc = p3;
        float dn = __shfl_down_sync(0xffffffffu, sinc, 1, 4);
        if (tq <= 2) sinc *= dn;
        dn = __shfl_down_sync(0xffffffffu, sinc, 2, 4);
        if (tq <= 1) sinc *= dn;
        float sex = __shfl_down_sync(0xffffffffu, sinc, 1, 4);
        if (tq == 3) sex = 1.f;
        tau[e] = __shfl_sync(0xffffffffu, inc, (lane & ~3) | 3, 32);
        e1[0][e] = ex * p0; e1[1][e] = ex * p1; e1[2][e] = ex * p2; e1[3][e] = ex * p3;
        e2[0][e] = sex * s0; e2[1][e] = sex * s1; e2[2][e] = sex * s2; e2[3][e] = sex * s3;
      }
      if (tq == 0) *reinterpret_cast<float4 *>(s_tau + s * kD + c0) = make_float4(tau[0], tau[1], tau[2], tau[3]);
      if (tid < kC) s_beta[tid] = b_pref;
      __syncthreads();

      const float4 t0v = *reinterpret_cast<const float4 *>(s_tau + c0);
      const float4 t1v = *reinterpret_cast<const float4 *>(s_tau + kD + c0);
      const float tau0[4] = {t0v.x, t0v.y, t0v.z, t0v.w}, tau1[4] = {t1v.x, t1v.y, t1v.z, t1v.w};
      float pre[4], post[4], inv_tau[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pre[e] = s == 1 ? tau0[e] : 1.f;   // Gamma at the start of the subtile
        post[e] = s == 0 ? tau1[e] : 1.f;  // decay from the end of the subtile to the chunk end
        inv_tau[e] = 1.f / (s == 0 ? tau0[e] : tau1[e]);
      }
      if (s == 0 && tq == 0)
        *reinterpret_cast<float4 *>(s_gamma + c0) =
            make_float4(tau0[0] * tau1[0], tau0[1] * tau1[1], tau0[2] * tau1[2], tau0[3] * tau1[3]);
      // byte offsets inside the tiles for channels c0..c0+3: fp32 tiles (32-wide blocks), 16-bit (64-wide)
      const uint32_t j16 = uint32_t((c0 & 63) >> 3), sub16 = uint32_t(c0 & 4) * 2, blk16 = uint32_t(c0 >> 6);
      float qt_col[4][4], kh_col[4][4];  // [channel][token] for the transposed tiles
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int t = tb + r;
        float q[4] = {0.f, 0.f, 0.f, 0.f}, k[4] = {0.f, 0.f, 0.f, 0.f};
        if (t < L) {
          const uint32_t off = blk16 * (kC * 128) + t * 128 + (((j16 ^ t) & 7u) << 4) + sub16;
          const uint2 qb = *reinterpret_cast<const uint2 *>(st + SQ + off);
          const uint2 kb = *reinterpret_cast<const uint2 *>(st + SK + off);
          const float2 q01 = unpack_bf16x2(qb.x), q23 = unpack_bf16x2(qb.y);
          const float2 k01 = unpack_bf16x2(kb.x), k23 = unpack_bf16x2(kb.y);
          q[0] = q01.x; q[1] = q01.y; q[2] = q23.x; q[3] = q23.y;
          k[0] = k01.x; k[1] = k01.y; k[2] = k23.x; k[3] = k23.y;
        }
        float qs[4], ks[4], kb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qs[e] = q[e] * e1[r][e];
          ks[e] = k[e] * e1[r][e];
          kb[e] = k[e] * e2[r][e];
        }
        // Gram A side: rows 32 s + t' of a 64-row tf32 tile (query rows, then key rows)
        auto f32row = [&](uint32_t tile, uint32_t rows, uint32_t row, float x0, float x1, float x2, float x3) {
          const uint32_t off = uint32_t(cb) * rows * 128 + row * 128 + (((uint32_t(cg) ^ row) & 7u) << 4);
          *reinterpret_cast<float4 *>(gram + tile + off) =
              make_float4(round_tf32(x0), round_tf32(x1), round_tf32(x2), round_tf32(x3));
        };
        f32row(G_QK, 64, 32 * s + 4 * tq + r, qs[0], qs[1], qs[2], qs[3]);
        f32row(G_QK, 64, 32 * s + 16 + 4 * tq + r, ks[0], ks[1], ks[2], ks[3]);
        // Gram B side: rows 0..15 hold subtile-0 keys for reference r_0, rows 16..47 all keys for r_1
        if (s == 0) {
          f32row(G_B, 48, t, kb[0] * inv_tau[0], kb[1] * inv_tau[1], kb[2] * inv_tau[2], kb[3] * inv_tau[3]);
          f32row(G_B, 48, 16 + t, kb[0], kb[1], kb[2], kb[3]);
        } else {
          f32row(G_B, 48, 16 + t, kb[0] * inv_tau[0], kb[1] * inv_tau[1], kb[2] * inv_tau[2], kb[3] * inv_tau[3]);
        }
        const uint32_t off16 = blk16 * (kC * 128) + t * 128 + (((j16 ^ t) & 7u) << 4) + sub16;
        *reinterpret_cast<uint2 *>(sm + OFF_KG + off16) =
            make_uint2(pack_f16x2(ks[0] * pre[0], ks[1] * pre[1]), pack_f16x2(ks[2] * pre[2], ks[3] * pre[3]));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qt_col[e][r] = qs[e] * pre[e];
          kh_col[e][r] = kb[e] * post[e];
        }
      }
      // transposed tiles: per channel, the 4 consecutive tokens of this thread (8 bytes)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t c = uint32_t(c0 + e);
        const uint32_t jq = uint32_t(4 + (tb >> 3)), sub = uint32_t(tb & 4) * 2;  // columns 32 + t in [-W^T | Q~^T]
        *reinterpret_cast<uint2 *>(sm + OFF_WQ + c * 128 + (((jq ^ c) & 7u) << 4) + sub) =
            make_uint2(pack_f16x2(qt_col[e][0], qt_col[e][1]), pack_f16x2(qt_col[e][2], qt_col[e][3]));
        const uint32_t row = 32 + c, jk = uint32_t(tb >> 3);                       // row 32 + c of [P ; K^^T]
        *reinterpret_cast<uint2 *>(sm + OFF_PK + row * 128 + (((jk ^ row) & 7u) << 4) + sub) =
            make_uint2(pack_f16x2(kh_col[e][0], kh_col[e][1]), pack_f16x2(kh_col[e][2], kh_col[e][3]));
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(bad)) goto abort;
    tc_fence_after();

    // ---------------- 2. Gram tiles (tf32 tensor cores) ----------------
    if (tid == 0) {
      // D[t'][i'] = sum_c QK[t'][c] B[i'][c]: M = 64 (all query/key rows), N = 48 (keys under the
      // two references); only each subtile's own rows are kept
      const uint32_t qk = sbase + OFF_GRAM + G_QK, bb = sbase + OFF_GRAM + G_B;
#pragma unroll
      for (int ks = 0; ks < 16; ++ks) {
        const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
        umma_tf32(tmem + TM_GRAM, kdesc(qk + kb * 64 * 128 + ko), kdesc(bb + kb * 48 * 128 + ko), IDESC_GRAM, ks > 0);
      }
      umma_commit(bar_mma);
    }
    bad |= !mbar_wait(bar_mma, mma_phase, err_word, DEVERR_MMA_TIMEOUT);
    mma_phase ^= 1;
    tc_fence_after();

    // ---------------- 3a. P and A out of TMEM ----------------
    // accumulator row t' = 16 quarter + lane (M = 64 layout: lanes 0..15 of each quarter):
    // quarter 0 / 2 hold the query rows of subtile 0 / 1 (P), quarter 1 / 3 the key rows (A)
    if (half == 0) {
      const int s = quarter >> 1, t = 16 * s + (lane & 15);
      const bool is_p = (quarter & 1) == 0;
      const float bt = s_beta[t & 31];
      float *Arow = reinterpret_cast<float *>(gram + G_A) + (t & 31) * kALd;
#pragma unroll
      for (int part = 0; part < 2; ++part) {  // columns i = 16 part .. 16 part + 15
        float vals[16];
        const bool have = part <= s;            // subtile 0 has 16 key columns, subtile 1 has 32
        if (have) {
          tmem_ld16(tmem + lane_base + TM_GRAM + (s == 0 ? 0 : 16) + 16 * part, vals);
          tmem_ld_wait();
        }
        if (lane < 16) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = 16 * part + e;
            const bool keep = have && t < L && (is_p ? i <= t : i < t);
            vals[e] = keep ? (is_p ? vals[e] : bt * vals[e]) : 0.f;
          }
          if (is_p) {
            st_at(sm, OFF_PK + sw128_chunk(t, 2 * part, 0, 160), pack8_f16(vals));
            st_at(sm, OFF_PK + sw128_chunk(t, 2 * part + 1, 0, 160), pack8_f16(vals + 8));
          } else {
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4)
              *reinterpret_cast<float4 *>(Arow + 16 * part + 4 * i4) =
                  make_float4(vals[4 * i4], vals[4 * i4 + 1], vals[4 * i4 + 2], vals[4 * i4 + 3]);
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
        // diagonal block `warp`, column `lane`: forward substitution, right-looking so the
        // dependent chain is 16 steps long
        const int s = warp, j = lane;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          Ts[(16 * s + m) * kALd + 16 * s + j] = x[m];
#pragma unroll
          for (int r = m + 1; r < 16; ++r) x[r] = fmaf(-As[(16 * s + r) * kALd + 16 * s + m], x[m], x[r]);
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

    // ---------------- 4. W^T = Kg^T T'^T and [U~^T | 0] = V^T [T' ; 0]^T (fp16) ----------------
    if (tid == 0) {
      const uint32_t tp = sbase + OFF_TP, kg = sbase + OFF_KG, vin = st_addr + SV;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        umma_f16(tmem + TM_W, mndesc(kg + ks * 2048), kdesc(tp + ks * 32), IDESC_WT, ks > 0);
        umma_f16(tmem + TM_U, mndesc(vin + ks * 2048), kdesc(tp + ks * 32), IDESC_UT, ks > 0);
      }
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

    // ---------------- -W^T and S^T to shared memory (fp16) ----------------
    {
      // W^T row c = v_own (the lane), columns t in [16 half, 16 half + 16) -> -W^T into the WQ tile
      float vals[16];
      tmem_ld16(tmem + lane_base + TM_W + 16 * half, vals);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) vals[j] = -vals[j];
      st_at(sm, OFF_WQ + sw128_chunk(v_own, 2 * half, 0, 128), pack8_f16(vals));
      st_at(sm, OFF_WQ + sw128_chunk(v_own, 2 * half + 1, 0, 128), pack8_f16(vals + 8));
    }
    // fp16 copy of S^T for this chunk's products, then S^T <- S^T Diag(Gamma_last) in place
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float x[16];
      tmem_ld16(s_row + 16 * u, x);
      tmem_ld_wait();
      st_at(gram, G_ST + sw128_chunk(v_own, 2 * u, half, 128), pack8_f16(x));
      st_at(gram, G_ST + sw128_chunk(v_own, 2 * u + 1, half, 128), pack8_f16(x + 8));
#pragma unroll
      for (int j = 0; j < 16; ++j) x[j] *= s_gamma[64 * half + 16 * u + j];
      tmem_st16(s_row + 16 * u, x);
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---------------- 5. state-dependent chain (fp16) ----------------
    if (tid == 0) {
      const uint32_t stt = sbase + OFF_GRAM + G_ST, wq = sbase + OFF_WQ;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {  // [U^T | O^T] += S^T [-W^T | Q~^T]
        const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
        umma_f16(tmem + TM_U, kdesc(stt + kb * 16384 + ko), mndesc(wq + ks * 2048, kMnBlockWQ), IDESC_UO, 1);
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
      const uint32_t ut = sbase + OFF_GRAM + G_UT, pk = sbase + OFF_PK;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)  // [O^T | S^T] += U^T [P ; K^^T]^T
        umma_f16(tmem + TM_O, kdesc(ut + ks * 32), kdesc(pk + ks * 32), IDESC_OS, 1);
      umma_commit(bar_mma);
    }
    bad |= !mbar_wait(bar_mma, mma_phase, err_word, DEVERR_MMA_TIMEOUT);
    mma_phase ^= 1;
    tc_fence_after();
    {
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
    for (int u = 0; u < 4; ++u) {
      float x[16];
      tmem_ld16(s_row + 16 * u, x);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) final_state[st_base + int64_t(64 * half + 16 * u + j) * kD + v_own] = x[j];
    }
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
