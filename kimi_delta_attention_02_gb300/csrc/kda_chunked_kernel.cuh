// kda_chunked_kernel.cuh -- tensor-core chunkwise KDA prefill (bf16 q/k/v, d_k = d_v = 128).
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
// e^{G_t - G_i} is split at one reference per chunk, r = G at the end of its first
// 16-token subtile: e^{G_t - G_i} = f_t g_i with f = e^{G - r}, g = 1 / f. Both
// lie in [e^-80, e^80] (at most 16 clamped steps on either side of r), inside the
// fp32 / tf32 range. The Gram products [Q * f ; K * f] (K * g)^T are exact on
// and below the diagonal, where the two factors meet as e^{G_t - G_i} <= 1; the
// entries above it may overflow and are never read. Every other operand is the
// same rescaled by a per-channel constant: Q * Gamma = (Q * f) e^r,
// K * Gamma = (K * f) e^r, K * e^{G_last - G} = (K * g) e^{G_last - r}.
//
// Unbounded decay (the earlier models' map g = -e^{A_h} Softplus(z), the same
// section): one step may fall far below -5, so a 16-token subtile can span more than
// e^80 in some channel. The reference r = G at the subtile boundary still bounds the
// block below the diagonal (rows t >= 16 by f <= 1, columns i < 16 by g <= 1); only
// the two diagonal 16 x 16 blocks depend on the span. A channel whose decay over a
// diagonal block exceeds 2^114 (about e^79) is "wide" there: its Gram operands for that
// block are zero (rows t < 16 of [Q f ; K f] for the first block, columns i >= 16 of
// K g for the second) and its share of the block's entries is formed from position
// pairs, sum over the wide channels of x_tc k_ic e^{G_tc - G_ic} with one exponential
// per pair and channel (the Kimi Linear treatment of the diagonal tiles), on the CUDA
// cores, and added where A and P leave tensor memory. A chunk without a wide channel
// runs exactly the bounded path; its cost is the map itself.
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
// Layout of the work. One CTA per (sequence, head) chain of 20 warps: 16 compute warps, one
// issuing warp (one thread of it issues every TMA load and the chain's tensor-core MMAs, so the
// ~50-120 cycles each MMA issue takes never holds up the compute warps) and, for the bounded
// maps, a Gram warp that issues the Gram MMAs and an inverse pair (warps 18, 19) that inverts
// I + A one chunk ahead of the chain. The fp32 state S^T (rows v = value channels, columns c =
// key channels) stays in tensor memory for the whole sequence, in two copies used alternately.
// Each iteration j runs the state chain of chunk j interleaved with the state-independent work
// of chunks j+1 and j+2, so that each tensor-core group runs while the threads work on the
// other streams:
//   P1  chain j : fp16 copy of S^T; Gamma_j-decayed S^T into the other copy (bounded maps:
//                 O^T of chunk j - 1 comes out of tensor memory in the same round trip)
//   P6  chain j : -W^T of chunk j into the [-W^T | Q~^T] tile (its MMA ran during
//                 P1); MMA1: [U^T | O^T] += S^T [-W^T | Q~^T]           (N = 64); bounded maps:
//                 beside MMA1, O^T of chunk j - 1 leaves for global memory (with the output
//                 gate of section 1.3, through the RMSNorm over the 128 value channels and the
//                 Sigmoid of the gate logits, whose tile the Gram warp loads into the Gram
//                 operand tiles that the Gram of chunk j + 1 freed)
//   P2  next j+2: decay prefix sums and the operand tiles (a thread owns one key
//                 channel and 8 tokens); the Gram of chunk j+2 (kind::tf32, M = 64 rows
//                 [Q f ; K f] x N = 32 keys K g) follows, queued behind MMA2
//   P3  chain j : U^T to fp16 (P of chunk j + 1 leaves tensor memory in the same round
//                 trip); MMA2: [O^T | S^T] += U^T [P ; K^^T]^T  (N = 160)
//   P4  next j+1: the inverse side. The inverse pair takes A of chunk j + 1 out of its TMEM
//                 lanes, forms T' = (I + A)^{-1} Diag(b) by back substitution (one row per
//                 lane) and converts v to fp16 while the compute warps run P1..P3; the pair
//                 hands T' over on an mbarrier, which alone gates W^T / U~^T:
//                 -W^T = -Kg^T T'^T (negated by the MMA) and [U~^T | 0] = V^T [T'; 0]^T.
//                 (The earlier four-warp inverse, with warps 2, 3, 6, 7 inverting I + A in
//                 8 x 8 and 16 x 16 blocks while 12 warps wrote the outputs, is still in this
//                 file behind kDedInv; every instantiation now takes the pair.)
// Per-chunk operand tiles are double-buffered by chunk parity ([P ; K^^T] three
// times, since it lives from P2 of chunk j to MMA2 of chunk j + 2), and so are the
// Gram accumulators. TMA brings q, k and log-decay one chunk ahead of P2 and v two
// chunks ahead of P4 (128-byte swizzle).
#pragma once

#include <cuda.h>

#include <type_traits>

#include "kda_common.cuh"

namespace kda {
namespace chunked {

constexpr int kC = 32;      // chunk length (two 16-token subtiles)
constexpr int kD = 128;     // d_k = d_v
constexpr int kWorkers = 512;               // 16 compute warps (warps 0..15)
constexpr int kHandoff = kWorkers + 32;     // + warp 16, which issues TMA loads and MMAs
// Warps 18 and 19 (TMEM lane quarters 2 and 3, where the key rows of the Gram land) are the
// inverse pair of the bounded maps, and warp 17 issues their Gram MMAs (a second issuer, so that
// the 16 Gram MMAs of a chunk do not queue in front of the chain's). 20 warps at 96 registers
// each fit the register file exactly as 17 would (registers are granted to warps in groups of four).
constexpr int kInvWarp0 = 18, kGramWarp = 17;
constexpr int kThreads = 640;
// Every warp from kInvWarp0 on runs the inverse pair's code, which indexes its lane quarter as 2 or 3:
// the pair must be the launch's last two warps.
static_assert(kThreads / 32 == kInvWarp0 + 2, "the inverse pair is the last two warps");
constexpr int kALd = 36;    // fp32 row stride of the A / T scratch
constexpr float kLog2e = 1.4426950408889634f;

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_QKG = 0;              // q [32][128] bf16 | k | log-decay [32][128] fp32 (or bf16 logits)
constexpr uint32_t SQ = 0, SK = 8 * 1024, SG = 16 * 1024;
constexpr uint32_t OFF_V = 32 * 1024;        // two v stages [32][128] bf16, converted to fp16 in place
constexpr uint32_t OFF_QK = 48 * 1024;       // Gram A side, tf32 [64 rows][128 c]: Q f (rows t), K f (rows 32 + t)
constexpr uint32_t OFF_B = 80 * 1024;        // Gram B side, tf32 [32 rows i][128 c]: K g
constexpr uint32_t OFF_ST = 96 * 1024;       // S^T fp16 [128][128]; the inverse's fp32 A, T, X alias it,
constexpr uint32_t G_A = 0, G_T = 5 * 1024, G_X = 10 * 1024;  // and so does the output gate's logit tile
constexpr uint32_t G_R = 16 * 1024;          // (bf16 [32 tokens][128], loaded once MMA1 has read S^T)
constexpr uint32_t G_O = 16 * 1024;          // and the output rows of a full chunk on their way to the TMA store
constexpr uint32_t OFF_UT = 128 * 1024;      // U^T fp16 [128][32], 64-byte swizzle
constexpr uint32_t OFF_TP = 136 * 1024;      // T' fp16 [64][32], 64-byte swizzle; rows 32..63 stay zero
constexpr uint32_t OFF_KG = 140 * 1024;      // 2 x Kg^T = (K * Gamma)^T fp16 [128 c][32 i], 64-byte swizzle
constexpr uint32_t kKGBytes = 8 * 1024;
constexpr uint32_t OFF_WQ = 156 * 1024;      // 2 x [-W^T | Q~^T] fp16 [128 c][64] (MN-major B of MMA1)
constexpr uint32_t kWQBytes = 16 * 1024;
constexpr uint32_t OFF_PK = 188 * 1024;      // 3 x [P ; K^^T] fp16 [160 rows][32], 64-byte swizzle
constexpr uint32_t kPKBytes = 10 * 1024;
constexpr uint32_t OFF_MISC = 218 * 1024;    // beta x2, Gamma_last x2, group decay totals, barriers
constexpr uint32_t OFF_SS = OFF_MISC + 3520; // output gate: per-token partial sums of squares [32][4] fp32
constexpr uint32_t kSmemBytes = 222 * 1024 + 1024;
static_assert(OFF_SS + 32 * 16 + 1023 <= kSmemBytes, "shared memory map exceeds the allocation");
// The inverse pair's copy of A [32][32] fp32, which takes the allocation to the 227 KB a CTA may have.
constexpr uint32_t OFF_PAIR = 222 * 1024;
constexpr uint32_t kSmemBytesUnbounded = 226 * 1024 + 1024;
static_assert(OFF_SS + 32 * 16 <= OFF_PAIR && kSmemBytesUnbounded <= 232448, "shared memory map exceeds 227 KB");
// Unbounded decay only: the position-pair shares of the diagonal blocks, by chunk parity,
// [2][512] fp32 (A entries first, then P; see pair_row_a), in the 8 KB that the bf16 decay logits
// leave free in the q/k/decay staging area (no TMA load writes there). The cumulative log2 decays
// [32 tokens][128 c] of a chunk that has wide channels pass through the lower half of the S^T
// tile (free between MMA1 of chunk c - 2, which reads it, and P1 of chunk c - 1).
constexpr uint32_t OFF_SHARES = OFF_QKG + SG + 8 * 1024;
static_assert(OFF_SHARES + 2 * 512 * 4 <= OFF_V, "position-pair shares overlap the v stages");
template <int kDecay>
constexpr uint32_t smem_bytes() { return kSmemBytesUnbounded; }
// a channel is wide in a diagonal block when its log2 decay over the block's tokens is below
// -kWideBlock (the bound gives every Gram factor of a narrow channel a magnitude <= 2^114)
constexpr float kWideBlock = 114.f;
// The largest clamped log-decay the clamped form computes exactly: with every log-decay of a
// 32-token chunk in [-5, 1/3] no fp16 operand exceeds 2^(32/3 log2 e) = 2^15.4 (inside fp16's
// 65504) and no tf32 Gram factor exceeds 2^115.4. A larger one is reported (DEVERR_RANGE).
constexpr float kMaxGrowth = 1.f / 3.f;

// A chunk's 512 position-pair shares: entries A[t][i] (i < t) of the two diagonal blocks
// (120 each, row-major inside a block), then P[t][i] (i <= t, 136 each). The first slot of
// row tl (block-local) of diagonal block blk:
__host__ __device__ constexpr uint32_t pair_row_a(uint32_t blk, uint32_t tl) { return blk * 120 + tl * (tl - 1) / 2; }
__host__ __device__ constexpr uint32_t pair_row_p(uint32_t blk, uint32_t tl) { return 240 + blk * 136 + tl * (tl + 1) / 2; }
static_assert(pair_row_a(1, 15) + 14 == 239 && pair_row_p(1, 15) + 15 == 511, "pair share layout");

// TMEM columns: two groups [U^T | O^T | S^T] (32 + 32 + 128) used by chunk parity, then
// Gram (chunk parity 0), -W^T, Gram (parity 1). Chunk j's MMA1 and MMA2 write group j % 2;
// its MMA2 leaves the state for chunk j + 1 there, which P1 of chunk j + 1 reads and
// rewrites, decayed, into the other.
constexpr uint32_t TM_GROUP = 192, TM_O = 32, TM_SS = 64, TM_GRAM = 384, TM_W = 416, TM_COLS = 512;
__device__ __forceinline__ uint32_t tm_grp(int b) { return TM_GROUP * uint32_t(b); }
__device__ __forceinline__ uint32_t tm_gram(int c) { return TM_GRAM + 64u * uint32_t(c & 1); }

constexpr uint32_t IDESC_GRAM = umma_idesc(UMMA_TF32, 64, 32, false, false, false);
constexpr uint32_t IDESC_WT = umma_idesc(UMMA_F16, 128, 32, false, false, true);   // -W^T = -Kg^T T'^T (negate A)
constexpr uint32_t IDESC_UT = umma_idesc(UMMA_F16, 128, 64, true, false, false);   // [U~^T | 0] = V^T [T'; 0]^T
constexpr uint32_t IDESC_UO = umma_idesc(UMMA_F16, 128, 64, false, true, false);   // += S^T [-W^T | Q~^T]
constexpr uint32_t IDESC_OS = umma_idesc(UMMA_F16, 128, 160, false, false, false); // [O^T | S^T] += U^T [P ; K^^T]^T

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
// 2^x on the SFU (ex2.approx, subnormal results flushed to zero)
__device__ __forceinline__ float exp2_sfu(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

struct Bars {
  uint64_t qkg, v[2], mma1, gram[2], mma2, wu, gate[4], drain, invd, aread[2], drain2, prep;
};
static_assert(OFF_MISC + (2 * 32 + 2 * 128 + 4 * 128) * 4 + sizeof(Bars) + 48 <= OFF_SS, "misc overlaps");

// Which token ranges the CTAs walk. count == 0: CTA b takes sequence n = b / H of cu_seqlens, or
// n = order[b / H] when an order is given (the longest sequences first). count > 0: CTA b takes
// run n = b / H, tokens [bos[n], eos[n]) of the packed tensors, with init_state / final_state
// indexed by n and the run's flags: RUN_ZERO_V reads v as zeros (its TMA boxes start before the
// tensor, where the copy fills zeros), RUN_INIT_IDENTITY / RUN_INIT_ZERO start from I or 0
// instead of init_state, RUN_NO_OUT writes no output. The segmented schedule of one long
// sequence runs its passes through this table.
constexpr int kMaxRuns = 64;
enum : uint32_t { RUN_ZERO_V = 1u, RUN_INIT_IDENTITY = 2u, RUN_INIT_ZERO = 4u, RUN_NO_OUT = 8u };
struct Runs {
  int32_t count;
  const int32_t *order;
  int32_t bos[kMaxRuns], eos[kMaxRuns];
  uint32_t flags[kMaxRuns];
};

// The output gate of section 1.3: bf16 gate logits r [T, H, 128], the RMSNorm weight w [128]
// (nullptr = ones) and eps.
struct OutGate {
  const uint16_t *r;
  const float *w;
  float eps;
};

// kDecay: DECAY_GATED, the log-decay is the gated form g = g_min Sigmoid(e^{A_h} z) of
// section 1.2 (tm_g then maps the bf16 logits z; lb holds g_min); DECAY_UNBOUNDED, the
// unbounded map g = -e^{A_h} Softplus(z) of the same logits (lb unused); DECAY_CLAMPED,
// tm_g maps the fp32 log_alpha, clamped below at lb. kNormGate: each output row is written as Sigmoid(r) * w * o / rms(o)
// (section 1.3) instead of o; tm_r maps the gate logits, for L2 prefetches.
template <bool kOutBF16, int kDecay, bool kNormGate>
__global__ void __launch_bounds__(kThreads, 1)
    kda_chunked_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                       const __grid_constant__ CUtensorMap tm_r, const __grid_constant__ CUtensorMap tm_o,
                       const OutGate og, const __grid_constant__ Runs runs,
                       const float *__restrict__ A_log, const float *__restrict__ beta,
                       const int32_t *__restrict__ cu_seqlens,
                       const float *__restrict__ init_state, void *__restrict__ out,
                       float *__restrict__ final_state, int H, float lb, float scale, uint32_t *err_word) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *s_beta = reinterpret_cast<float *>(sm + OFF_MISC);  // [2][32] beta by chunk parity
  float *s_gamma = s_beta + 2 * 32;                           // [2][128] Gamma_last by chunk parity
  float *s_tot = s_gamma + 2 * 128;                           // [4][128] log2 decay of each 8-token group
  Bars *bars = reinterpret_cast<Bars *>(s_tot + 4 * 128);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + 1);
  float4 *s_ss = reinterpret_cast<float4 *>(sm + OFF_SS);    // [32 tokens] x 4 lane quarters: sums of o^2

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, grp = warp >> 2;  // TMEM lane quarter, column group (compute warps)
  const bool worker = tid < kWorkers;              // warps 0..15; warp 16 issues TMA loads and MMAs
  // Every map inverts I + A on a pair of warps of their own (warps 18, 19), one chunk ahead of the
  // state chain. (The four-warp inverse on the compute warps below is the earlier form.)
  constexpr bool kDedInv = true;
  const bool inv_pair = kDedInv && warp >= kInvWarp0;  // warps 18, 19: the last two (see kThreads)
  // (Unused: with the four-warp inverse, full chunks left the output gate through a staged TMA store.)
  constexpr bool kStaged = kNormGate && !kDedInv;
  // Read-out with the inverse pair: the outputs of chunk j - 1 leave with P1 of chunk j (both wait
  // for MMA2 of chunk j - 1 and read tensor memory in the same round trip; the output gate's
  // logits of chunk j - 1 wait in the Gram operand tiles, see the Gram warp), and P of chunk j + 1
  // leaves tensor memory with U^T of chunk j in P3; no separate output phase.
  constexpr bool kMerged = kDedInv;
  const int h = int(blockIdx.x % H);
  const int64_t blk = blockIdx.x / H;
  const int64_t n = runs.count > 0 ? blk : runs.order != nullptr ? int64_t(runs.order[blk]) : blk;
  const int64_t bos = runs.count > 0 ? runs.bos[blk] : cu_seqlens[n];
  const int64_t eos = runs.count > 0 ? runs.eos[blk] : cu_seqlens[n + 1];
  const uint32_t rflags = runs.count > 0 ? runs.flags[blk] : 0u;
  const bool no_out = (rflags & RUN_NO_OUT) != 0;
  const int n_chunks = int((eos - bos + kC - 1) / kC);
  const uint32_t sbase = smem_u32(sm);
  constexpr bool kGated = kDecay != DECAY_CLAMPED;  // tm_g maps bf16 logits
  constexpr bool kUnb = kDecay == DECAY_UNBOUNDED;
  const float a_h = kGated ? __expf(A_log[h]) : 0.f;  // e^{A_h} of the logit maps

  if (tid == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_g);
    if (kNormGate) tma_prefetch_desc(&tm_r);
    tma_prefetch_desc(&tm_o);
    mbar_init(&bars->qkg, 1);
    mbar_init(&bars->v[0], 1);
    mbar_init(&bars->v[1], 1);
    mbar_init(&bars->mma1, 1);
    mbar_init(&bars->gram[0], 1);
    mbar_init(&bars->gram[1], 1);
    mbar_init(&bars->mma2, 1);
    mbar_init(&bars->wu, 1);
    if constexpr (kNormGate) {  // (with the inverse pair, one per logits slot of the output gate)
      for (int i = 0; i < 4; ++i) mbar_init(&bars->gate[i], 1);
    } else {
      mbar_init(&bars->gate[0], 1);
    }
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->invd, 1);
    mbar_init(&bars->aread[0], 1);
    mbar_init(&bars->aread[1], 1);
    mbar_init(&bars->drain2, 1);
    mbar_init(&bars->prep, kWorkers);  // every compute thread: the Gram operands of a chunk are written
    fence_mbarrier_init();
    s_tmem[1] = 0u;            // abort flag
    s_tmem[2] = s_tmem[3] = ~0u;  // unbounded map: the last chunk of each parity with wide channels
    // (s_tmem[4 .. 11]: the wide channels of a chunk's two diagonal blocks, 4 x 32 bits each)
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, TM_COLS);
    tmem_relinquish();
  }
  // rows 32..63 of the T' tile stay zero: the U~ product reads them to clear the O^T columns
  for (int e = tid; e < 32 * 4; e += kThreads)
    st_at(sm, OFF_TP + sw64_chunk(32 + (e >> 2), e & 3), make_uint4(0, 0, 0, 0));

  const int v_own = 32 * quarter + lane;  // state row (TMEM lane) of this thread; key channel in P2
  const float w_own = (kNormGate && og.w != nullptr) ? og.w[v_own] : 1.f;  // RMSNorm weight of channel v_own
  const int64_t st_base = (n * H + h) * int64_t(kD) * kD;

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_base = uint32_t(32 * quarter) << 16;
  // this thread's 32 state columns in group b
  auto s_cols = [&](int b) { return tmem + lane_base + tm_grp(b) + TM_SS + 32 * grp; };
  if (worker) {  // the state entering chunk 0 sits where chunk -1 would have left it: group 1
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float x[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = 32 * grp + 16 * u + j;  // key row of S
        x[j] = (rflags & RUN_INIT_IDENTITY)                                 ? (c == v_own ? 1.f : 0.f)
               : ((rflags & RUN_INIT_ZERO) || init_state == nullptr) ? 0.f
                                                                      : init_state[st_base + int64_t(c) * kD + v_own];
      }
      tmem_st16(s_cols(1) + 16 * u, x);
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
    mbar_arrive_expect_tx(&bars->qkg, 2 * 8192 + (kGated ? 8192 : 16384));
    tma_load_3d(sm + OFF_QKG + SQ, &tm_q, &bars->qkg, 0, h, t0);
    tma_load_3d(sm + OFF_QKG + SQ + 4096, &tm_q, &bars->qkg, 64, h, t0);
    tma_load_3d(sm + OFF_QKG + SK, &tm_k, &bars->qkg, 0, h, t0);
    tma_load_3d(sm + OFF_QKG + SK + 4096, &tm_k, &bars->qkg, 64, h, t0);
    tma_load_3d(sm + OFF_QKG + SG, &tm_g, &bars->qkg, 0, h, t0);
  };
  auto issue_v = [&](int c) {  // issuer
    // a run that reads v as zeros takes boxes 64 tokens before the tensor, which TMA fills with zeros
    const int32_t t0 = (rflags & RUN_ZERO_V) ? -64 : int32_t(chunk_t0(c));
    uint8_t *dst = sm + OFF_V + (c & 1) * 8192;
    mbar_arrive_expect_tx(&bars->v[c & 1], 8192);
    tma_load_3d(dst, &tm_v, &bars->v[c & 1], 0, h, t0);
    tma_load_3d(dst + 4096, &tm_v, &bars->v[c & 1], 64, h, t0);
    if (kNormGate && !no_out) tma_prefetch_l2_3d(&tm_r, 0, h, t0);  // chunk c's gate logits, read when written
  };

  bool bad = false;  // a bounded wait of this thread gave up
  volatile uint32_t *s_abort = s_tmem + 1;
  // chunks whose q/k/g and v loads were issued last (the issuer's abort path waits for them)
  int qkg_last = -1, v_last[2] = {-1, -1}, gate_last = -1;
  bool store_pending = false;  // thread 0: an output tile store whose shared-memory read may be running
  float b_next = (tid < kC && tid < eos - bos) ? beta[(bos + tid) * H + h] : 0.f;  // beta of chunk 0

  // Synchronisation. The 16 compute warps meet on barrier BAR_WORK where they share
  // data. They hand each finished group of operands to the issuing warp through one
  // barrier per event (compute warps arrive, the issuer syncs), so MMA issue never
  // holds them up. An event of chunk j + 1 always comes after a wait on an MMA or a
  // load the issuer starts only past the same event of chunk j, so the compute warps
  // never arrive twice at a barrier the issuer has not yet passed. If a compute
  // thread's wait gave up, the compute warps raise s_abort before the hand-off the
  // issuer waits for next, and both sides leave for the teardown.
  constexpr uint32_t BAR_WORK = 1, H_COPY = 2, H_PREP = 3, H_U = 4, H_INV = 5, BAR_INV = 6;
  auto handoff = [&](uint32_t id) {  // compute warps: operands of this event written
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar_arrive(id, kHandoff);
    // with the inverse pair, the Gram warp learns of the Gram operands on an mbarrier (it issues
    // the Gram; a bounded wait, so that it never waits on a hand-off that an abort skips)
    if (kDedInv && id == H_PREP) mbar_arrive(&bars->prep);
  };
  auto give_up = [&](uint32_t id) {
    if (tid == 0) *s_abort = 1u;
    handoff(id);
  };

  // ------------------------------------------------------------------ P2: operand tiles
  // Thread (channel ch = v_own, tokens 8 grp .. 8 grp + 7): the decay prefix sums run
  // along its own 8 tokens; the 4 group totals of a channel meet in shared memory.
  // Everything is kept in log2 units (x log2 e), so each factor is one ex2.
  // Runs two chunks ahead of the state chain. Returns false when the compute warps give up.
  auto prep = [&](int c) -> bool {
    const int b = c & 1, L = chunk_len(c);
    const int64_t t0 = chunk_t0(c);
    const float b_pref = b_next;
    if (tid < kC) b_next = (tid < eos - t0 - kC) ? beta[(t0 + kC + tid) * H + h] : 0.f;  // next chunk's
    bad |= !mbar_wait_sleep(&bars->qkg, uint32_t(c & 1), err_word, DEVERR_TMA_TIMEOUT);
    if (c >= 1)  // the Gram of chunk c - 1 has read the Gram tiles
      bad |= !mbar_wait_sleep(&bars->gram[(c - 1) & 1], uint32_t(((c - 1) >> 1) & 1), err_word,
                              DEVERR_MMA_TIMEOUT);
    const int ch = v_own, tb = 8 * grp;
    // Every chunk but the last of a sequence is full: it takes code without the masks.
    const bool full = L == kC;
    float lg[8];  // log2 of Gamma within the group: sum of the group's decays up to each token
    bool maybe_wide = false;  // unbounded map: this group's decay passes half the wide bound
    auto decay_sums = [&](auto full_tag) {
      constexpr bool kFull = decltype(full_tag)::value;
      const float *gin = reinterpret_cast<const float *>(sm + OFF_QKG + SG) + tb * kD + ch;
      const uint16_t *zin = reinterpret_cast<const uint16_t *>(sm + OFF_QKG + SG) + tb * kD + ch;
      float run = 0.f;
      float gmax = -INFINITY;  // clamped form: the largest log-decay (NaN is not counted, as in g > bound)
#pragma unroll
      for (int r = 0; r < 8; ++r) {  // alpha = 1 past the end of the sequence
        const float g = !(kFull || tb + r < L) ? 0.f
                        : kUnb                ? unbounded_log_decay(bf16_to_f32(zin[r * kD]), a_h)
                        : kGated              ? gated_log_decay(bf16_to_f32(zin[r * kD]), a_h, lb)
                                              : clamp_log_decay(gin[r * kD], lb);
        if (!kGated) gmax = fmaxf(gmax, g);
        run = fmaf(g, kLog2e, run);
        lg[r] = run;
      }
      if (!kGated && gmax > kMaxGrowth) raise_device_error(err_word, DEVERR_RANGE);  // results unspecified
      s_tot[grp * kD + ch] = run;
      maybe_wide = kUnb && run < -0.5f * kWideBlock;  // a wide channel has such a group in its block
    };
    if (full) decay_sums(std::true_type{});
    else decay_sums(std::false_type{});
    if (tid < kC) s_beta[b * kC + tid] = b_pref;
    if (kStaged && store_pending) {  // the U^T tile is written after this barrier
      bulk_wait_read();
      store_pending = false;
    }
    // unbounded map: `flagged` also says that some group decays past half the wide bound, so
    // that only such chunks pay for the exact test below (which also catches a wait that gave up)
    const bool flagged = named_bar_or(BAR_WORK, kWorkers, bad || maybe_wide);
    if (!kUnb && flagged) {
      give_up(H_PREP);
      return false;
    }
    bool wide_here = false;  // unbounded map: this channel wide in this thread's diagonal block
    const uint32_t row = uint32_t(ch) * 128u, sw = uint32_t(ch) & 7u;
    uint32_t hq[4], hk[4], hg[4];  // fp16 pairs
    auto operands = [&](auto full_tag) {
      constexpr bool kFull = decltype(full_tag)::value;
      const float T0 = s_tot[ch], T1 = s_tot[kD + ch], T2 = s_tot[2 * kD + ch], T3 = s_tot[3 * kD + ch];
      const float r2 = T0 + T1;                                                // log2 e^r
      const float last2 = r2 + (T2 + T3);                                      // log2 Gamma_last
      const float start = grp == 0 ? -r2 : grp == 1 ? -T1 : grp == 2 ? 0.f : T2;  // log2 e^{G_start - r}
      const float tau0 = exp2_sfu(r2), tau1 = exp2_sfu(last2 - r2);
      if (grp == 0) s_gamma[b * kD + ch] = exp2_sfu(last2);
      // unbounded map: this channel wide in this thread's diagonal block (the same test as
      // the position-pair step's)
      [[maybe_unused]] const bool wide = kUnb && (grp < 2 ? T0 + T1 : T2 + T3) < -kWideBlock;
      if constexpr (kUnb) {  // the wide channels of each diagonal block, 32 per warp
        const uint32_t wm = __ballot_sync(0xffffffffu, wide);
        if (lane == 0 && (grp & 1) == 0) s_tmem[4 + 4 * (grp >> 1) + quarter] = wm;
        wide_here = wide;
      }
      // q and k of the 8 tokens: bf16 element (t, ch) of the 128-byte-swizzled TMA tiles
      const uint32_t cc = uint32_t(ch & 63);
      const uint8_t *qk0 = sm + OFF_QKG + (ch >> 6) * 4096 + tb * 128 + (cc & 7u) * 2;
      const uint32_t xj = (cc >> 3) << 4;
      // Gram operands, K-major tf32 (blocks of 32 channels, one 128-byte row per token): the 32
      // lanes of a warp hold one whole row, so each 4-byte store is conflict-free. fp16 operands,
      // one 16-byte chunk each: Q~^T (columns 32 + t of [-W^T | Q~^T]), K^^T (row 32 + ch of
      // [P ; K^^T]) and Kg^T (row ch). Two halves of 4 tokens keep few values live.
      const uint32_t cb = uint32_t(ch >> 5), cq = uint32_t(ch & 31) >> 2;
      float *gq = reinterpret_cast<float *>(sm + OFF_QK + cb * 64 * 128 + tb * 128 + (ch & 3) * 4);
      float *gk = reinterpret_cast<float *>(sm + OFF_QK + cb * 64 * 128 + (32 + tb) * 128 + (ch & 3) * 4);
      float *gb = reinterpret_cast<float *>(sm + OFF_B + cb * 32 * 128 + tb * 128 + (ch & 3) * 4);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float qf[4], kf[4], kg[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = 4 * half + e;
          const uint32_t off = r * 128 + (xj ^ uint32_t(r << 4));
          const bool ok = kFull || tb + r < L;
          const float q = ok ? bf16_to_f32(*reinterpret_cast<const uint16_t *>(qk0 + SQ + off)) : 0.f;
          const float k = ok ? bf16_to_f32(*reinterpret_cast<const uint16_t *>(qk0 + SK + off)) : 0.f;
          const float d = start + lg[r];  // log2 e^{G_t - r}
          const float f = exp2_sfu(d), g = exp2_sfu(-d);
          const float2 qk_f = f2_mul(make_float2(q, k), make_float2(f, f));    // (packed pairs)
          const float2 qk_t = f2_mul(qk_f, make_float2(tau0, tau0));
          float qv = qk_f.x, kv = qk_f.y, gv = k * g;               // tf32 Gram operands
          qf[e] = qk_t.x;                                             // fp16 operands: Q Gamma,
          kf[e] = qk_t.y;                                             // K Gamma,
          kg[e] = gv * tau1;                                          // K e^{G_last - G}
          if constexpr (kUnb) {
            if (wide) {  // f (first block) or g (second) may overflow: out of the Gram, and
              if (grp < 2) {  // the fp16 operands from their own exponentials (<= 1)
                const float gm = exp2_sfu(d + r2);
                qf[e] = q * gm;
                kf[e] = k * gm;
                qv = kv = 0.f;
              } else {
                kg[e] = k * exp2_sfu(last2 - r2 - d);
                gv = 0.f;
              }
            }
          }
          const uint32_t o4 = (r * 128 + ((cq ^ uint32_t(r)) << 4)) >> 2;  // row tb + r, whose t & 7 = r
          gq[o4] = round_tf32(qv);
          gk[o4] = round_tf32(kv);
          gb[o4] = round_tf32(gv);
        }
        hq[2 * half] = pack_f16x2(qf[0], qf[1]);
        hq[2 * half + 1] = pack_f16x2(qf[2], qf[3]);
        hk[2 * half] = pack_f16x2(kf[0], kf[1]);
        hk[2 * half + 1] = pack_f16x2(kf[2], kf[3]);
        hg[2 * half] = pack_f16x2(kg[0], kg[1]);
        hg[2 * half + 1] = pack_f16x2(kg[2], kg[3]);
      }
    };
    // Unbounded map. A thread whose channel is wide in its diagonal block puts its tokens'
    // cumulative log2 decays (from the chunk start) into the S^T tile, once MMA1 of chunk
    // c - 2 has read it: [128 c][36] (a row stride of 36 words keeps both the row writes and
    // the column reads free of bank conflicts); the rows of narrow channels are not read.
    float *Gs = reinterpret_cast<float *>(sm + OFF_ST);
    auto stage_decays = [&](int c) {
      if (c >= 2) bad |= !mbar_wait_sleep(&bars->mma1, uint32_t(c & 1), err_word, DEVERR_MMA_TIMEOUT);
      const float T0 = s_tot[ch], T1 = s_tot[kD + ch], T2 = s_tot[2 * kD + ch];
      const float g0 = grp == 0 ? 0.f : grp == 1 ? T0 : grp == 2 ? T0 + T1 : (T0 + T1) + T2;
      float4 *dst = reinterpret_cast<float4 *>(Gs + ch * 36 + tb);
      dst[0] = make_float4(g0 + lg[0], g0 + lg[1], g0 + lg[2], g0 + lg[3]);
      dst[1] = make_float4(g0 + lg[4], g0 + lg[5], g0 + lg[6], g0 + lg[7]);
    };
    // A chunk with wide channels: their shares of the entries of the two diagonal blocks,
    // A: sum_c k_tc k_ic e^{G_tc - G_ic} (i < t) and P: sum_c q_tc k_ic e^{G_tc - G_ic}
    // (i <= t), from position pairs, one exponential (<= 1) per pair and wide channel,
    // shared by A and P. Thread (block b, row tl, column il) owns entry (16 b + tl, 16 b + il)
    // and walks the block's list of wide channels. Tokens past the end of the
    // sequence only reach entries that the A and P masks clear.
    auto pair_shares = [&](int c) -> bool {
      if (tid == 0) s_tmem[2 + (c & 1)] = uint32_t(c);  // for the A and P extraction of chunk c
      // Work items: threads 0..479 take the 240 entries below the diagonals (120 per block), two
      // adjacent lanes per entry, each over half of the channels (mask words 2 hh, 2 hh + 1);
      // threads 480..511 take the 32 diagonal entries, which need P only and no exponential
      // (e^{G_tc - G_tc} = 1).
      const bool diag = tid >= 480;
      const int hh = tid & 1, r = (tid >> 1) % 120;  // r: entry inside its block's lower triangle
      const int pb = diag ? (tid - 480) >> 4 : (tid >> 1) / 120;
      int tl = int((1.f + sqrtf(8.f * float(r) + 1.f)) * 0.5f);  // r = tl (tl - 1) / 2 + il, il < tl
      if (tl * (tl - 1) / 2 > r) --tl;                             // (against rounding of the root)
      else if ((tl + 1) * tl / 2 <= r) ++tl;
      int il = r - tl * (tl - 1) / 2;
      if (diag) tl = il = (tid - 480) & 15;
      const int t = 16 * pb + tl, i = 16 * pb + il;
      // bf16 element (token, channel w) of the 128-byte-swizzled q / k tiles
      auto elem = [&](uint32_t tile, int tok, int w) {
        const uint32_t cw = uint32_t(w & 63);
        return bf16_to_f32(*reinterpret_cast<const uint16_t *>(
            sm + OFF_QKG + tile + uint32_t(w >> 6) * 4096u + uint32_t(tok) * 128u +
            (((cw >> 3) ^ uint32_t(tok & 7)) << 4) + (cw & 7u) * 2u));
      };
      float a = 0.f, p = 0.f;
      if (diag) {  // a whole warp: P[t][t] = sum over the wide channels of q_tc k_tc
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t m = s_tmem[4 + 4 * pb + q4];
          while (m != 0u) {
            const int w = 32 * q4 + __ffs(int(m)) - 1;
            m &= m - 1u;
            p = fmaf(elem(SQ, t, w), elem(SK, t, w), p);
          }
        }
      } else {  // whole warps too: the two halves of an entry meet by one shuffle
#pragma unroll 1
        for (int q4 = 2 * hh; q4 < 2 * hh + 2; ++q4) {
          uint32_t m = s_tmem[4 + 4 * pb + q4];
          while (m != 0u) {
            const int w = 32 * q4 + __ffs(int(m)) - 1;
            m &= m - 1u;
            const float e = exp2_sfu(Gs[w * 36 + t] - Gs[w * 36 + i]);
            const float ke = elem(SK, i, w) * e;
            a = fmaf(elem(SK, t, w), ke, a);
            p = fmaf(elem(SQ, t, w), ke, p);
          }
        }
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        p += __shfl_xor_sync(0xffffffffu, p, 1);
      }
      float *corr = reinterpret_cast<float *>(sm + OFF_SHARES) + (c & 1) * 512;
      if (diag) {
        corr[pair_row_p(uint32_t(pb), uint32_t(tl)) + il] = p;
      } else if (hh == 0) {
        corr[pair_row_a(uint32_t(pb), uint32_t(tl)) + il] = a;
        corr[pair_row_p(uint32_t(pb), uint32_t(tl)) + il] = p;
      }
      // every thread is past the decays before P1 of the next chain step rewrites the S^T tile
      if (named_bar_or(BAR_WORK, kWorkers, bad)) {
        give_up(H_PREP);
        return false;
      }
      return true;
    };
    if (full) operands(std::true_type{});
    else operands(std::false_type{});
    if constexpr (kUnb) {  // does any channel of this chunk need position pairs?
      if (flagged) {
        if (wide_here) stage_decays(c);
        if (named_bar_or(BAR_WORK, kWorkers, wide_here || bad) && !pair_shares(c)) return false;
      }
    }
    handoff(H_PREP);  // the Gram operands are complete; the fp16 tiles are needed later
    st_at(sm, OFF_PK + (c % 3) * kPKBytes + sw64_chunk(32u + ch, grp), make_uint4(hg[0], hg[1], hg[2], hg[3]));
    st_at(sm, OFF_KG + b * kKGBytes + sw64_chunk(ch, grp), make_uint4(hk[0], hk[1], hk[2], hk[3]));
    if (c >= 2)  // MMA1 of chunk c - 2 has read its [-W^T | Q~^T] buffer, which chunk c reuses
      bad |= !mbar_wait_sleep(&bars->mma1, uint32_t(c & 1), err_word, DEVERR_MMA_TIMEOUT);
    st_at(sm, OFF_WQ + b * kWQBytes + row + (((4u + grp) ^ sw) << 4), make_uint4(hq[0], hq[1], hq[2], hq[3]));
    return true;
  };

  auto issue_gram = [&](int c) {  // issuer: 16 steps of 8 channels (32 bytes; 4 per 32-channel block)
    const uint64_t qk = kdesc128(sbase + OFF_QK), bb = kdesc128(sbase + OFF_B);
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
      umma_tf32(tmem + tm_gram(c), dadv(qk, kb * 64 * 128 + ko), dadv(bb, kb * 32 * 128 + ko), IDESC_GRAM,
                ks > 0);
    }
    umma_commit(&bars->gram[c & 1]);
  };

  // Warps 2, 3, 6, 7 (TMEM lane quarters 2 and 3, column groups 0 and 1) form the inverse
  // group: the key rows of the Gram (A) live in their lanes. The other 12 warps write
  // outputs, convert v and take the query rows (P).
  const bool inv_group = !kDedInv && quarter >= 2 && grp < 2;
  const int iw = (quarter - 2) + 2 * grp;  // inverse group: warp 0..3 of the group
  const int itid = 32 * iw + lane;         // inverse group: thread 0..127 of the group

  // ------------------------------------------------------------------ P5: outputs
  // O^T of chunk j out of TMEM to global memory. With the inverse pair every compute warp writes
  // 8 tokens of its 32 channels, read in P1 of chunk j + 1 and written once MMA1 of chunk j + 1
  // is issued (the last chunk after the loop); with the
  // four-warp inverse, the 12 warps outside the inverse group do it in P4: lane quarters 0 and 1
  // have 4 of them (8 tokens each), quarters 2 and 3 have 2 (16 each).
  //
  // With the output gate, a token's 128 channels are spread over four warps (one per lane
  // quarter): each warp sums o^2 of its 32 channels for each of its tokens, the output warps
  // meet on BAR_OUT, lane l of each warp then adds token l's four partial sums in a fixed order
  // and passes 1 / rms to the other lanes. The per-token partial sums have one buffer: the next
  // read-out writes it only after MMA2 of a later chunk, which needs every output thread's
  // hand-off after its reads of this one.
  // Output rows of chunk j held by this thread (channel v_own, tokens t0 .. t0 + N - 1). They go
  // out as row stores (a warp writes 32 consecutive channels of a token), except with the output
  // gate and the four-warp inverse, where a full chunk's rows go through shared memory and out
  // with one TMA store by thread 0: the 16 scattered row stores per thread there lengthen the
  // output warps' path past the inverse's. A bf16 tile is staged in the U^T tile (free from MMA2
  // of chunk j until P3 of the next step): thread 0 waits for the store to have read it only
  // before the operand barrier of the next step (or at once when the next step has none). An
  // fp32 tile is staged in the upper half of the S^T tile, which the next step rewrites at its
  // start, so thread 0 waits before it joins the barrier that ends this step. A partial chunk
  // (the last of a sequence) is always stored row by row, so that nothing past the sequence is
  // written. Both paths round bf16 alike.
  constexpr uint32_t BAR_OUT = 7;
  constexpr uint32_t kOutThreads = kDedInv ? kWorkers : 384;  // the warps that write outputs
  // With the inverse pair, the four warps of column group grp (one per lane quarter) hold all 128
  // channels of tokens 8 grp .. 8 grp + 7: the sums of squares meet on one barrier per group.
  constexpr uint32_t BAR_NORM0 = 9;  // .. 12
  auto write_rows = [&](const auto &x, int t0, int j, int L) {
    constexpr int N = int(sizeof(x) / sizeof(x[0]));
    if (kStaged && L == kC) {
      uint8_t *stage = kOutBF16 ? sm + OFF_UT : sm + OFF_ST + G_O;
#pragma unroll
      for (int e = 0; e < N; ++e) {
        if constexpr (kOutBF16) reinterpret_cast<uint16_t *>(stage)[(t0 + e) * kD + v_own] = f32_to_bf16(x[e]);
        else reinterpret_cast<float *>(stage)[(t0 + e) * kD + v_own] = x[e];
      }
      fence_proxy_async_smem();
      named_bar_sync(BAR_OUT, kOutThreads);
      if (tid == 0 && !no_out) {
        tma_store_3d(&tm_o, stage, 0, h, int32_t(chunk_t0(j)));
        bulk_commit();
        if (kOutBF16 && j + 3 < n_chunks) store_pending = true;  // read before prep(j + 3)'s barrier
        else bulk_wait_read();
      }
    } else if (!no_out) {
      const int64_t step = int64_t(H) * kD;
      const int64_t base = ((chunk_t0(j) + t0) * H + h) * int64_t(kD) + v_own;
      if (L == kC) {  // a full chunk: no masks
        using E = typename std::conditional<kOutBF16, uint16_t, float>::type;
        E *p = static_cast<E *>(out) + base;
#pragma unroll
        for (int e = 0; e < N; ++e, p += step) {
          if constexpr (kOutBF16) *p = f32_to_bf16(x[e]);
          else *p = x[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < N; ++e)
          if (t0 + e < L) store_elem<kOutBF16>(out, base + e * step, x[e]);
      }
    }
  };
  // The output gate's logits of chunk c. With the four-warp inverse, one tile in the upper half of
  // the S^T tile, loaded by the issuer once MMA1 of chunk c has read S^T (barrier gate[0], one
  // phase per chunk). With the inverse pair, slot c % 4 of the Gram operand tiles, loaded by the
  // Gram warp once the Gram of chunk c + 2 has read them (barrier gate[c % 4]); the read-out of
  // chunk c, in P1 of chunk c + 1, reads it before the operand build of chunk c + 3 rewrites them.
  auto gate_tile = [&](int c) {
    return reinterpret_cast<const uint16_t *>(kDedInv ? sm + OFF_QK + uint32_t(c & 3) * 8192u : sm + OFF_ST + G_R);
  };
  auto wait_gate = [&](int c) {
    if (kDedInv) bad |= !mbar_wait_sleep(&bars->gate[c & 3], uint32_t((c >> 2) & 1), err_word, DEVERR_TMA_TIMEOUT);
    else bad |= !mbar_wait_sleep(&bars->gate[0], uint32_t(c & 1), err_word, DEVERR_TMA_TIMEOUT);
  };
  auto issue_gate = [&](int c) {  // issuer, four-warp inverse
    if constexpr (kStaged) {
      mbar_wait_sleep(&bars->mma1, uint32_t(c & 1), err_word, DEVERR_MMA_TIMEOUT);  // S^T read
      mbar_arrive_expect_tx(&bars->gate[0], 8192);
      tma_load_3d(sm + OFF_ST + G_R, &tm_r, &bars->gate[0], 0, h, int32_t(chunk_t0(c)));
    }
  };
  // Sigmoid(r) w of this thread's rows (channel v_own, tokens t0 ..) of chunk c
  auto gate_weights = [&](auto &gw, int t0, int c) {
    constexpr int N = int(sizeof(gw) / sizeof(gw[0]));
    const uint16_t *rt = gate_tile(c) + t0 * kD + v_own;
#pragma unroll
    for (int e = 0; e < N; e += 2) {  // packed pairs: the same roundings as scalar operations
      const float2 g = f2_mul(make_float2(w_own, w_own),
                              sigmoid2_approx(make_float2(bf16_to_f32(rt[e * kD]), bf16_to_f32(rt[(e + 1) * kD]))));
      gw[e] = g.x;
      gw[e + 1] = g.y;
    }
  };
  // x: this thread's rows of O^T of chunk j, as read from tensor memory. Scaled, divided by the
  // rms over each token's 128 channels, gated and written; x is kept in registers across the
  // barrier (no second tensor-memory read), and every value is formed before the (masked) stores.
  auto norm_rows = [&](auto &x, const auto &gw, int t0, int j, int L) {
    constexpr int N = int(sizeof(x) / sizeof(x[0]));  // tokens of this warp: 8 or 16
    float sq[N];
#pragma unroll
    for (int e = 0; e < N; e += 2) {  // packed pairs: the same roundings as scalar multiplies
      const float2 y = f2_mul(make_float2(scale, scale), make_float2(x[e], x[e + 1]));
      const float2 y2 = f2_mul(y, y);
      x[e] = y.x;
      x[e + 1] = y.y;
      sq[e] = y2.x;
      sq[e + 1] = y2.y;
    }
    const float part = lane_sums<N>(sq, lane);
    constexpr int kShift = N == 8 ? 2 : 1;  // lane l holds the sum of token (l >> kShift) & (N - 1)
    if ((lane & ((1 << kShift) - 1)) == 0)
      reinterpret_cast<float *>(s_ss)[4 * (t0 + ((lane >> kShift) & (N - 1))) + quarter] = part;
    if (kDedInv) named_bar_sync(BAR_NORM0 + uint32_t(grp), 128);
    else named_bar_sync(BAR_OUT, kOutThreads);
    const float4 p = s_ss[t0 + (lane & (N - 1))];
    const float rstd_l = rsqrtf(((p.x + p.y) + (p.z + p.w)) * (1.f / kD) + og.eps);  // token t0 + (lane & (N-1))
#pragma unroll
    for (int e = 0; e < N; e += 2) {  // (x rstd) (Sigmoid(r) w), packed pairs
      const float2 y = f2_mul(f2_mul(make_float2(x[e], x[e + 1]), make_float2(__shfl_sync(0xffffffffu, rstd_l, e),
                                                                              __shfl_sync(0xffffffffu, rstd_l, e + 1))),
                              make_float2(gw[e], gw[e + 1]));
      x[e] = y.x;
      x[e + 1] = y.y;
    }
    write_rows(x, t0, j, L);
  };
  auto out_gated_rows = [&](auto n_tag, int t0, int j, int L, uint32_t ocols) {
    constexpr int N = decltype(n_tag)::value;  // tokens of this warp: 8 or 16
    if (kDedInv && no_out) return;  // (the Gram warp loads no logits then)
    // Sigmoid(r) w first: the gate tile is there well before MMA2 has finished
    wait_gate(j);
    float gw[N];
    gate_weights(gw, t0, j);
    bad |= !mbar_wait_sleep(&bars->mma2, uint32_t(j & 1), err_word, DEVERR_MMA_TIMEOUT);
    tc_fence_after();
    float x[N];
    if constexpr (N == 8) tmem_ld8_wait(ocols + t0, x);
    else tmem_ld16_wait(ocols + t0, x);
    norm_rows(x, gw, t0, j, L);
  };
  // the read-out without the output gate: this thread's rows of O^T of chunk j, scaled and written
  auto plain_read_out = [&](float (&x)[8], int j) {
#pragma unroll
    for (int e = 0; e < 8; e += 2) {  // packed pairs: the same roundings as scalar multiplies
      const float2 y = f2_mul(make_float2(x[e], x[e + 1]), make_float2(scale, scale));
      x[e] = y.x;
      x[e + 1] = y.y;
    }
    write_rows(x, 8 * grp, j, chunk_len(j));
  };
  auto out_chunk = [&](int j) {
    if (!kNormGate) {
      bad |= !mbar_wait_sleep(&bars->mma2, uint32_t(j & 1), err_word, DEVERR_MMA_TIMEOUT);
      tc_fence_after();
    }
    const int L = chunk_len(j);
    const uint32_t ocols = tmem + lane_base + tm_grp(j & 1) + TM_O;
    if constexpr (kNormGate) {
      if (kDedInv || quarter < 2) out_gated_rows(std::integral_constant<int, 8>{}, 8 * grp, j, L, ocols);
      else out_gated_rows(std::integral_constant<int, 16>{}, 16 * (grp - 2), j, L, ocols);
    } else if (kDedInv || quarter < 2) {
      float x[8];
      tmem_ld8_wait(ocols + 8 * grp, x);  // O^T row v, tokens 8 grp ..
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= scale;
      write_rows(x, 8 * grp, j, L);
    } else {
      const int t0 = 16 * (grp - 2);
      float x[16];
      tmem_ld16_wait(ocols + t0, x);  // O^T row v, tokens t0 ..
#pragma unroll
      for (int e = 0; e < 16; ++e) x[e] *= scale;
      write_rows(x, t0, j, L);
    }
  };

  // Diagonal 16 x 16 block iw of T = (I + A)^{-1} (rows and columns 16 iw ..) from A, in 8 x 8
  // pieces, on one warp: the two diagonal pieces by forward substitution (16 lanes, a lane per
  // column), the zero piece above them, then the piece below, -T_11 (A_10 T_00). Xs: 64 floats
  // of scratch per block.
  auto diag_block_inverse = [&](int iw, const float *As, float *Ts, float *Xs) {
    // diagonal block iw (16 x 16) in 8 x 8 pieces, warp-synchronous
    const int base = 16 * iw;
    if (lane < 16) {  // the two 8 x 8 diagonal pieces: lane = column of its piece
      const int o = base + 8 * (lane >> 3), cc = lane & 7;
      float x[8], a[28];  // column cc of the piece's inverse; the piece's strictly lower entries
#pragma unroll
      for (int r = 0; r < 8; ++r) x[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0, n = 0; m < 8; ++m)  // all loads before the first store (which may alias)
#pragma unroll
        for (int r = m + 1; r < 8; ++r, ++n) a[n] = As[(o + r) * kALd + o + m];
#pragma unroll
      for (int m = 0, n = 0; m < 8; ++m)
#pragma unroll
        for (int r = m + 1; r < 8; ++r, ++n) x[r] = fmaf(-a[n], x[m], x[r]);
#pragma unroll
      for (int m = 0; m < 8; ++m) Ts[(o + m) * kALd + o + cc] = x[m];
    } else {  // the zero 8 x 8 piece above the diagonal
      const int l = lane - 16;
      *reinterpret_cast<float4 *>(Ts + (base + (l >> 1)) * kALd + base + 8 + 4 * (l & 1)) =
          make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncwarp();
    // piece below the diagonal: -T_11 (A_10 T_00); lane (row r8, columns 2 c8, 2 c8 + 1)
    float *Xw = Xs + 64 * iw;
    const int r8 = lane >> 2, c8 = lane & 3;
    float a8[8];
    auto load8 = [&](const float *src) {
      const float4 p0 = reinterpret_cast<const float4 *>(src)[0], p1 = reinterpret_cast<const float4 *>(src)[1];
      a8[0] = p0.x;
      a8[1] = p0.y;
      a8[2] = p0.z;
      a8[3] = p0.w;
      a8[4] = p1.x;
      a8[5] = p1.y;
      a8[6] = p1.z;
      a8[7] = p1.w;
      };
      load8(As + (base + 8 + r8) * kALd + base);
      float2 acc8 = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 t2 = *reinterpret_cast<const float2 *>(Ts + (base + k) * kALd + base + 2 * c8);
        acc8.x = fmaf(a8[k], t2.x, acc8.x);
        acc8.y = fmaf(a8[k], t2.y, acc8.y);
      }
      *reinterpret_cast<float2 *>(Xw + r8 * 8 + 2 * c8) = acc8;
      __syncwarp();
      load8(Ts + (base + 8 + r8) * kALd + base + 8);
      acc8 = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 x2 = *reinterpret_cast<const float2 *>(Xw + k * 8 + 2 * c8);
        acc8.x = fmaf(-a8[k], x2.x, acc8.x);
        acc8.y = fmaf(-a8[k], x2.y, acc8.y);
      }
      *reinterpret_cast<float2 *>(Ts + (base + 8 + r8) * kALd + base + 2 * c8) = acc8;
  };

  // P rows t = 16 quarter + lane (lanes 0..15) of chunk c, columns 8 grp .. + 7 (compute warps of
  // TMEM quarters 0 and 1), into the [P ; K^^T] tile of chunk c. Waits for the tensor-memory loads
  // issued before it as well.
  auto extract_p = [&](int c, auto &...also) {  // also: arrays loaded before it, completed by its wait
    const int b = c & 1, L = chunk_len(c);
    bad |= !mbar_wait_sleep(&bars->gram[b], uint32_t((c >> 1) & 1), err_word, DEVERR_MMA_TIMEOUT);
    tc_fence_after();
    const int t = 16 * quarter + (lane & 15);
    const bool have = grp < 2 * (quarter + 1);  // columns up to the row block's end
    float vals[8] = {};
    if (have) tmem_ld8(tmem + lane_base + tm_gram(c) + 8 * grp, vals);
    tmem_ld_wait(vals, also...);
    if (lane < 16) {
      // keep i <= t. In the unbounded map the column group goes in opaque: with it visible,
      // nvcc 13.0 took this limit to be at least 2 there and dropped the mask on the entries
      // above the diagonal. (The bounded maps compile right, and would spill with it.)
      const int lim = (have && t < L) ? t + 1 - 8 * (kUnb ? opaque_int(grp) : grp) : 0;
      if constexpr (kUnb) {  // the position-pair shares of chunk c's diagonal blocks, if it has any
        const bool slow = *reinterpret_cast<volatile uint32_t *>(s_tmem + 2 + b) == uint32_t(c);
        if (slow && have && grp >= 2 * quarter) {  // columns inside the diagonal block
          const float *cr = reinterpret_cast<const float *>(sm + OFF_SHARES) + b * 512 +
                            pair_row_p(uint32_t(quarter), uint32_t(t & 15)) + 8 * (grp - 2 * quarter);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e < lim) vals[e] += cr[e];
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) vals[e] = e < lim ? vals[e] : 0.f;
      st_at(sm + OFF_PK + (c % 3) * kPKBytes, sw64_chunk(t, grp), pack8_f16(vals));
    }
  };

  // ------------------------------------------------------------------ P4: P, A, inverse, T', v
  // The four-warp inverse (unused: every instantiation takes the inverse pair): inverse-side work of
  // chunk c; the 12 warps outside the inverse group also write the outputs of chunk j_out (if >= 0).
  // Returns false when the compute warps give up.
  auto extract_inverse = [&](int c, int j_out) -> bool {
    const int b = c & 1, L = chunk_len(c);
    float *As = reinterpret_cast<float *>(sm + OFF_ST + G_A);
    // unbounded map: the position-pair shares of chunk c's diagonal blocks, if it has any
    const bool slow = kUnb && *reinterpret_cast<volatile uint32_t *>(s_tmem + 2 + b) == uint32_t(c);
    const float *corr = reinterpret_cast<const float *>(sm + OFF_SHARES) + b * 512;
    if (inv_group) {
      bad |= !mbar_wait_sleep(&bars->gram[b], uint32_t((c >> 1) & 1), err_word, DEVERR_MMA_TIMEOUT);
      tc_fence_after();
      {  // A rows t = 16 (quarter - 2) + lane (lanes 0..15; M = 64 layout), columns 16 grp .. + 15
        const int s = quarter - 2, t = 16 * s + (lane & 15);
        if (grp <= s) {  // columns past the row block are all zero and never read
          float vals[16];
          tmem_ld16_wait(tmem + lane_base + tm_gram(c) + 16 * grp, vals);
          if (lane < 16) {
            const float bt = s_beta[b * kC + t];
            const int lim = t < L ? t - 16 * opaque_int(grp) : 0;  // keep i < t (opaque: as for P below)
            if (slow && grp == s) {
              const float *cr = corr + pair_row_a(uint32_t(s), uint32_t(t & 15));
#pragma unroll
              for (int e = 0; e < 16; ++e)
                if (e < lim) vals[e] += cr[e];
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) vals[e] = e < lim ? bt * vals[e] : 0.f;
            float4 *arow = reinterpret_cast<float4 *>(As + t * kALd + 16 * grp);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              arow[q4] = make_float4(vals[4 * q4], vals[4 * q4 + 1], vals[4 * q4 + 2], vals[4 * q4 + 3]);
          }
        }
      }
      named_bar_sync(BAR_INV, 128);
      // T = (I + A)^{-1}, then T' = T Diag(beta)
      float *Ts = reinterpret_cast<float *>(sm + OFF_ST + G_T);
      float *Xs = reinterpret_cast<float *>(sm + OFF_ST + G_X);
      if (iw < 2) {
        diag_block_inverse(iw, As, Ts, Xs);
      } else {  // the zero 16 x 16 block above the diagonal
        const int l = itid - 64;
        *reinterpret_cast<float4 *>(Ts + (l >> 2) * kALd + 16 + 4 * (l & 3)) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      named_bar_sync(BAR_INV, 128);
      // block below the diagonal, T_10 = -T_11 (A_10 T_00): thread (row r, columns 2 c2, 2 c2 + 1)
      const int r = itid >> 3, c2 = itid & 7;
      float rowv[16];
      auto load_row = [&](const float *src) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 v4 = reinterpret_cast<const float4 *>(src)[q4];
          rowv[4 * q4] = v4.x;
          rowv[4 * q4 + 1] = v4.y;
          rowv[4 * q4 + 2] = v4.z;
          rowv[4 * q4 + 3] = v4.w;
        }
      };
      load_row(As + (16 + r) * kALd);  // A_10 row r
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float2 t2 = *reinterpret_cast<const float2 *>(Ts + k * kALd + 2 * c2);  // T_00 row k
        acc.x = fmaf(rowv[k], t2.x, acc.x);
        acc.y = fmaf(rowv[k], t2.y, acc.y);
      }
      *reinterpret_cast<float2 *>(Xs + r * 16 + 2 * c2) = acc;
      named_bar_sync(BAR_INV, 128);
      load_row(Ts + (16 + r) * kALd + 16);  // T_11 row r (zero above its diagonal)
      acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float2 x2 = *reinterpret_cast<const float2 *>(Xs + k * 16 + 2 * c2);
        acc.x = fmaf(-rowv[k], x2.x, acc.x);
        acc.y = fmaf(-rowv[k], x2.y, acc.y);
      }
      *reinterpret_cast<float2 *>(Ts + (16 + r) * kALd + 2 * c2) = acc;
      named_bar_sync(BAR_INV, 128);
      {  // T' = T Diag(beta) -> fp16 [t][i]
        const int t = itid >> 2, cj = itid & 3;
        const float4 *trow = reinterpret_cast<const float4 *>(Ts + t * kALd + 8 * cj);
        const float4 *brow = reinterpret_cast<const float4 *>(s_beta + b * kC + 8 * cj);
        const float4 t0v = trow[0], t1v = trow[1], b0v = brow[0], b1v = brow[1];
        const float x[8] = {t0v.x * b0v.x, t0v.y * b0v.y, t0v.z * b0v.z, t0v.w * b0v.w,
                            t1v.x * b1v.x, t1v.y * b1v.y, t1v.z * b1v.z, t1v.w * b1v.w};
        st_at(sm, OFF_TP + sw64_chunk(t, cj), pack8_f16(x));
      }
    } else {
      // the 12 other warps: v tile of this chunk bf16 -> fp16 in place (rows past the end
      // zeroed), the query rows P of the Gram, then the outputs of chunk j_out
      const int ot = (quarter < 2 ? 64 * grp + 32 * quarter : 256 + 64 * (grp - 2) + 32 * (quarter - 2)) + lane;
      bad |= !mbar_wait_sleep(&bars->v[b], uint32_t((c >> 1) & 1), err_word, DEVERR_TMA_TIMEOUT);
      for (int e = ot; e < kC * 16; e += int(kOutThreads)) {
        const int t = e >> 4, cj = e & 15;
        uint4 *p = reinterpret_cast<uint4 *>(sm + OFF_V + b * 8192 + sw128_chunk(t, cj & 7, cj >> 3, kC));
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
      if (quarter < 2) {  // P rows t = 16 quarter + lane (lanes 0..15), columns 8 grp .. + 7
        bad |= !mbar_wait_sleep(&bars->gram[b], uint32_t((c >> 1) & 1), err_word, DEVERR_MMA_TIMEOUT);
        tc_fence_after();
        const int t = 16 * quarter + (lane & 15);
        const bool have = grp < 2 * (quarter + 1);  // columns up to the row block's end
        float vals[8];
        if (have) {
          tmem_ld8_wait(tmem + lane_base + tm_gram(c) + 8 * grp, vals);
        }
        if (lane < 16) {
          // keep i <= t. In the unbounded map the column group goes in opaque: with it visible,
          // nvcc 13.0 took this limit to be at least 2 there and dropped the mask on the entries
          // above the diagonal. (The bounded maps compile right, and would spill with it.)
          const int lim = (have && t < L) ? t + 1 - 8 * (kUnb ? opaque_int(grp) : grp) : 0;
          if (slow && have && grp >= 2 * quarter) {  // columns inside the diagonal block
            const float *cr = corr + pair_row_p(uint32_t(quarter), uint32_t(t & 15)) + 8 * (grp - 2 * quarter);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (e < lim) vals[e] += cr[e];
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) vals[e] = e < lim ? vals[e] : 0.f;
          st_at(sm + OFF_PK + (c % 3) * kPKBytes, sw64_chunk(t, grp), pack8_f16(vals));
        }
      }
      if (j_out >= 0) out_chunk(j_out);
    }
    // the next chain step rewrites the S^T tile (the inverse's scratch, the output gate's tiles):
    // all compute threads are past this phase before any goes on
    fence_proxy_async_smem();
    tc_fence_before();
    const bool ab = named_bar_or(BAR_WORK, kWorkers, bad);
    if (ab) give_up(H_INV);
    else handoff(H_INV);
    return !ab;
  };

  // ------------------------------------------------------------------ the inverse pair
  // Warps 18 and 19 (bounded maps): T' = (I + A)^{-1} Diag(beta) of chunk c and the fp16 v tile of
  // chunk c, while the compute warps run the chain of chunk c - 1 and build the operands of chunk
  // c + 1. A lives in the lanes of TMEM quarters 2 (rows 0..15) and 3 (rows 16..31); both warps
  // copy their rows into the pair's own 4 KB of shared memory, then warp 18 forms T' a row per
  // lane: row j of T solves x^T (I + A) = e_j^T, i.e. x_m = [m == j] - sum_{i > m} x_i A[i][m]
  // (A is strictly lower triangular), taken from m = 31 down with every finished x_i folded into
  // the rows below it. The T' tile is free once the W^T / U~^T product of chunk c - 1 has read
  // it. The pair reports chunk c done on the invd barrier, after which the issuer reads T' and v.
  // Returns false when a wait gave up.
  constexpr uint32_t BAR_PAIR = 8;
  auto inverse_pair = [&](int c) -> bool {
    const int b = c & 1, L = chunk_len(c);
    const int s = quarter - 2;          // TMEM quarter 2 + s holds A rows 16 s ..
    const int ptid = 32 * s + lane;     // 0 .. 63
    float *As = reinterpret_cast<float *>(sm + OFF_PAIR);  // [32][32]
    bool ok = mbar_wait_sleep(&bars->gram[b], uint32_t((c >> 1) & 1), err_word, DEVERR_MMA_TIMEOUT);
    tc_fence_after();
    // A rows t = 16 s + lane (lanes 0..15; M = 64 layout), columns 16 h2 .. 16 h2 + 15 up to the
    // row block's end (the substitution reads no entry on or past a row's diagonal);
    // A[t][i] = beta_t G[t][i] for i < t (and t inside the sequence), else 0
    for (int h2 = 0; h2 <= s; ++h2) {
      float vals[16];
      tmem_ld16_wait(tmem + lane_base + tm_gram(c) + 16 * h2, vals);
      if (lane < 16) {
        const int t = 16 * s + lane;
        const float bt = s_beta[b * kC + t];
        const int lim = t < L ? t - 16 * (kUnb ? opaque_int(h2) : h2) : 0;  // keep i < t (opaque: as for P)
        if constexpr (kUnb) {  // the diagonal block of a chunk with wide channels: their position-pair shares
          const bool slow = *reinterpret_cast<volatile uint32_t *>(s_tmem + 2 + b) == uint32_t(c);
          if (slow && h2 == s) {
            const float *cr = reinterpret_cast<const float *>(sm + OFF_SHARES) + b * 512 + pair_row_a(uint32_t(s), uint32_t(lane));
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (e < lim) vals[e] += cr[e];
          }
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) vals[e] = e < lim ? bt * vals[e] : 0.f;
        float4 *arow = reinterpret_cast<float4 *>(As + t * 32 + 16 * h2);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          arow[q4] = make_float4(vals[4 * q4], vals[4 * q4 + 1], vals[4 * q4 + 2], vals[4 * q4 + 3]);
      }
    }
    // v of chunk c, bf16 -> fp16 in place (rows past the end zeroed): 8 of the 512 16-byte pieces each
    ok &= mbar_wait_sleep(&bars->v[b], uint32_t((c >> 1) & 1), err_word, DEVERR_TMA_TIMEOUT);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int e = ptid + 64 * k, t = e >> 4, cj = e & 15;
      uint4 *p = reinterpret_cast<uint4 *>(sm + OFF_V + b * 8192 + sw128_chunk(t, cj & 7, cj >> 3, kC));
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
    tc_fence_before();
    named_bar_sync(BAR_PAIR, 64);
    if (ptid == 0) mbar_arrive(&bars->aread[b]);  // A of chunk c is out of its Gram slot
    if (s == 0) {
      float2 x[16];  // row `lane` of T, as pairs of columns (packed fp32 FMAs)
#pragma unroll
      for (int m = 0; m < 16; ++m) x[m] = make_float2(2 * m == lane ? 1.f : 0.f, 2 * m + 1 == lane ? 1.f : 0.f);
#pragma unroll
      for (int i = 31; i >= 1; --i) {
        const float xi = (i & 1) ? x[i >> 1].y : x[i >> 1].x;  // final: every row below i is folded in
        const float2 nxi = make_float2(-xi, -xi);
#pragma unroll
        for (int m4 = 0; m4 < (i + 3) / 4; ++m4) {  // row i of A (the same for every lane)
          const float4 a = *reinterpret_cast<const float4 *>(As + i * 32 + 4 * m4);
          if (4 * m4 + 1 < i) x[2 * m4] = f2_fma(nxi, make_float2(a.x, a.y), x[2 * m4]);
          else if (4 * m4 < i) x[2 * m4].x = fmaf(-xi, a.x, x[2 * m4].x);
          if (4 * m4 + 3 < i) x[2 * m4 + 1] = f2_fma(nxi, make_float2(a.z, a.w), x[2 * m4 + 1]);
          else if (4 * m4 + 2 < i) x[2 * m4 + 1].x = fmaf(-xi, a.z, x[2 * m4 + 1].x);
        }
      }
      // T'[j][m] = T[j][m] beta_m -> fp16, row j = lane
      if (c >= 1) ok &= mbar_wait_sleep(&bars->wu, uint32_t((c - 1) & 1), err_word, DEVERR_MMA_TIMEOUT);
      const float4 *bt = reinterpret_cast<const float4 *>(s_beta + b * kC);
#pragma unroll
      for (int cj = 0; cj < 4; ++cj) {
        const float4 b0 = bt[2 * cj], b1 = bt[2 * cj + 1];
        const float2 x0 = x[4 * cj], x1 = x[4 * cj + 1], x2 = x[4 * cj + 2], x3 = x[4 * cj + 3];
        const float y[8] = {x0.x * b0.x, x0.y * b0.y, x1.x * b0.z, x1.y * b0.w,
                            x2.x * b1.x, x2.y * b1.y, x3.x * b1.z, x3.y * b1.w};
        st_at(sm, OFF_TP + sw64_chunk(uint32_t(lane), uint32_t(cj)), pack8_f16(y));
      }
    }
    fence_proxy_async_smem();  // T' and v are read by the tensor cores
    tc_fence_before();
    // one verdict for the pair, then chunk c is reported done (also when a wait gave up, so that
    // the waiters move on; the abort flag then tells the issuer and the compute warps)
    const bool fail = named_bar_or(BAR_PAIR, 64, !ok);
    if (fail && ptid == 0) *s_abort = 1u;
    if (ptid == 0) mbar_arrive(&bars->invd);
    return !fail;
  };

  auto issue_wu = [&](int c) {  // issuer: W^T and [U~^T | 0]
    const int b = c & 1;
    const uint64_t tp = kdesc64(sbase + OFF_TP), kg = kdesc64(sbase + OFF_KG + b * kKGBytes),
                   vin = mndesc(sbase + OFF_V + b * 8192, kC * 128);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      umma_f16(tmem + TM_W, dadv(kg, ks * 32), dadv(tp, ks * 32), IDESC_WT, ks > 0);
      umma_f16(tmem + tm_grp(b), dadv(vin, ks * 2048), dadv(tp, ks * 32), IDESC_UT, ks > 0);
    }
    umma_commit(&bars->wu);
  };

  // ------------------------------------------------------------------ P6: -W^T
  auto wt_extract = [&](int c) {
    const int b = c & 1;
    bad |= !mbar_wait_sleep(&bars->wu, uint32_t(c & 1), err_word, DEVERR_MMA_TIMEOUT);
    tc_fence_after();
    float x[8];
    tmem_ld8_wait(tmem + lane_base + TM_W + 8 * grp, x);  // -W^T row c = v_own, columns t = 8 grp ..
    const uint32_t cr = uint32_t(v_own);
    st_at(sm + OFF_WQ + b * kWQBytes, cr * 128 + (((uint32_t(grp) ^ cr) & 7u) << 4), pack8_f16(x));
  };

  if (worker) {
    // ---------------------------------------------------------------- compute warps
    if (n_chunks > 0) {  // operands of chunks 0 and 1
      if (!prep(0)) goto teardown;
      if (n_chunks > 1 && !prep(1)) goto teardown;
      if (kMerged) {
        if (quarter < 2) extract_p(0);
      } else if (!extract_inverse(0, -1)) {
        goto teardown;
      }
    }
    for (int j = 0; j < n_chunks; ++j) {
      const int b = j & 1;
      const bool more = j + 1 < n_chunks;
      // ---------------- P1: chain j, fp16 copy of S^T; decayed S^T into group j % 2
      if (j > 0 && (inv_group || kMerged)) {  // the state MMA2 of chunk j - 1 left
        bad |= !mbar_wait_sleep(&bars->mma2, uint32_t((j - 1) & 1), err_word, DEVERR_MMA_TIMEOUT);
        tc_fence_after();
      }
      float ox[8];  // merged read-out: O^T row v of chunk j - 1, tokens 8 grp ..
      if (kMerged && j > 0) tmem_ld8(tmem + lane_base + tm_grp(b ^ 1) + TM_O + 8 * grp, ox);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float x[16];
        if constexpr (kMerged) {
          tmem_ld16(s_cols(b ^ 1) + 16 * u, x);
          tmem_ld_wait(x, ox);  // and the merged read-out's row
        } else {
          tmem_ld16_wait(s_cols(b ^ 1) + 16 * u, x);
        }
        const uint32_t col = uint32_t(32 * grp + 16 * u);  // state column c of x[0]
        st_at(sm + OFF_ST, sw128_chunk(v_own, (col & 63u) >> 3, col >> 6, 128), pack8_f16(x));
        st_at(sm + OFF_ST, sw128_chunk(v_own, ((col & 63u) >> 3) + 1, col >> 6, 128), pack8_f16(x + 8));
        const float4 *gam = reinterpret_cast<const float4 *>(s_gamma + b * kD + col);
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // packed pairs: the same roundings as scalar multiplies
          const float4 gv = gam[e];
          const float2 lo = f2_mul(make_float2(x[4 * e], x[4 * e + 1]), make_float2(gv.x, gv.y));
          const float2 hi = f2_mul(make_float2(x[4 * e + 2], x[4 * e + 3]), make_float2(gv.z, gv.w));
          x[4 * e] = lo.x;
          x[4 * e + 1] = lo.y;
          x[4 * e + 2] = hi.x;
          x[4 * e + 3] = hi.y;
        }
        tmem_st16(s_cols(b) + 16 * u, x);
      }
      tmem_st_wait();
      if constexpr (kMerged && !kNormGate && kGated) {  // (the gated decay's read-out: here, which
        if (j > 0) plain_read_out(ox, j - 1);           // measured faster than beside MMA1)
      }
      // ---------------- P6: -W^T of chunk j (its W^T / U~^T MMA ran during P1) -> MMA1
      wt_extract(j);
      handoff(H_COPY);
      // ---------------- read-out of chunk j - 1 (its O^T came with S^T in P1), beside MMA1
      if constexpr (kMerged && !kNormGate && !kGated) {
        if (j > 0) plain_read_out(ox, j - 1);
      }
      if constexpr (kNormGate && kMerged) {  // through the output gate
        if (j > 0 && !no_out) {
          wait_gate(j - 1);
          float gw[8];
          gate_weights(gw, 8 * grp, j - 1);
          norm_rows(ox, gw, 8 * grp, j - 1, chunk_len(j - 1));
        }
      }
      // ---------------- P2: operand tiles of chunk j + 2 -> Gram
      if (j + 2 < n_chunks && !prep(j + 2)) goto teardown;
      // ---------------- P3: chain j, U^T to fp16 -> MMA2
      bad |= !mbar_wait_sleep(&bars->mma1, uint32_t(j & 1), err_word, DEVERR_MMA_TIMEOUT);
      tc_fence_after();
      {
        float x[8];
        tmem_ld8(tmem + lane_base + tm_grp(b) + 8 * grp, x);  // U^T row v, columns t = 8 grp ..
        if (kMerged && more && quarter < 2) extract_p(j + 1, x);  // waits for U^T's load with its own
        else tmem_ld_wait(x);
        st_at(sm + OFF_UT, sw64_chunk(uint32_t(v_own), uint32_t(grp)), pack8_f16(x));
      }
      handoff(H_U);
      // ---------------- the last chunk's outputs (the inverse side of chunk j + 1 is the pair's)
      if (kMerged) {
        if (!more) out_chunk(j);
      } else if (more) {
        if (!extract_inverse(j + 1, j)) goto teardown;
      } else if (!inv_group) {
        out_chunk(j);
      }
    }
    if (n_chunks > 0) {  // the last chunk's MMA2 (the warps outside the inverse group waited already)
      bad |= !mbar_wait_sleep(&bars->mma2, uint32_t((n_chunks - 1) & 1), err_word, DEVERR_MMA_TIMEOUT);
      tc_fence_after();
    }
    if (final_state != nullptr) {  // the last chunk's MMA2 left the state in its group
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        float x[16];
        tmem_ld16_wait(s_cols((n_chunks + 1) & 1) + 16 * u, x);
#pragma unroll
        for (int e = 0; e < 16; ++e) final_state[st_base + int64_t(32 * grp + 16 * u + e) * kD + v_own] = x[e];
      }
    }
  } else if (kDedInv && warp == kGramWarp) {
    // ---------------------------------------------------------------- Gram warp
    // The Gram of chunk c once its operand tiles are written (H_PREP) and the pair has taken A of
    // chunk c - 2 out of the same tensor-memory slot. Lane 0 issues; on leaving early it waits for
    // its own MMAs (bounded) before the teardown frees tensor memory.
    bool issued = false;
    int gate_hi = -1;  // output gate: the last chunk whose logits tile this warp has loaded
    for (int c = 0; c < n_chunks; ++c) {
      const bool ok = mbar_wait_sleep(&bars->prep, uint32_t(c & 1), err_word, DEVERR_MMA_TIMEOUT);
      tc_fence_after();
      if (__any_sync(0xffffffffu, !ok || *s_abort != 0u)) break;  // one verdict for the warp
      const bool read = c < 2 ||
                        mbar_wait_sleep(&bars->aread[c & 1], uint32_t(((c - 2) >> 1) & 1), err_word, DEVERR_MMA_TIMEOUT);
      if (__any_sync(0xffffffffu, !read)) {
        if (lane == 0) *s_abort = 1u;
        break;
      }
      tc_fence_after();
      if (lane == 0) issue_gram(c);
      issued = true;
      // output gate: the logits of chunk c - 2 into the slot that this Gram frees, once it has read
      // its operands; after the last Gram nothing rewrites the operand tiles, so the logits of the
      // chunks left follow at once (at most three, in slots of their own)
      if constexpr (kNormGate) {
        const bool last = c == n_chunks - 1;
        if (!no_out && (last || c >= 2)) {
          const bool read_ops =
              mbar_wait_sleep(&bars->gram[c & 1], uint32_t((c >> 1) & 1), err_word, DEVERR_MMA_TIMEOUT);
          if (__any_sync(0xffffffffu, !read_ops)) {
            if (lane == 0) *s_abort = 1u;
            break;
          }
          const int k1 = last ? c : c - 2;
          if (lane == 0)
            for (int k = c >= 2 ? c - 2 : 0; k <= k1; ++k) {
              mbar_arrive_expect_tx(&bars->gate[k & 3], 8192);
              tma_load_3d(sm + OFF_QK + uint32_t(k & 3) * 8192u, &tm_r, &bars->gate[k & 3], 0, h,
                          int32_t(chunk_t0(k)));
            }
          gate_hi = k1;
        }
      }
    }
    // the logits tiles in flight land before the teardown (the latest phase of each slot's barrier)
    if constexpr (kNormGate)
      for (int k = gate_hi >= 3 ? gate_hi - 3 : 0; k <= gate_hi; ++k)
        mbar_wait_sleep(&bars->gate[k & 3], uint32_t((k >> 2) & 1), err_word, DEVERR_TMA_TIMEOUT);
    if (issued && *s_abort != 0u) {
      if (lane == 0) umma_commit(&bars->drain2);
      __syncwarp();
      mbar_wait_sleep(&bars->drain2, 0u, err_word, DEVERR_MMA_TIMEOUT);
    }
  } else if (inv_pair) {
    // ---------------------------------------------------------------- inverse pair
    for (int c = 0; c < n_chunks; ++c) {
      if (!inverse_pair(c)) break;
      // the compute warps gave up: leave (one verdict for the pair, so that both warps leave together)
      if (named_bar_or(BAR_PAIR, 64, *s_abort != 0u)) break;
    }
  } else if (warp == kInvWarp0 - 2) {
    // ---------------------------------------------------------------- issuing warp
    // The whole warp follows the hand-offs; lane 0 issues.
    const bool leader = lane == 0;
    auto sync_on = [&](uint32_t id) {
      named_bar_sync(id, kHandoff);
      tc_fence_after();
      return *s_abort == 0u;
    };
    // the inverse pair has written T' of chunk c (bounded; a pair that gave up raised the abort flag)
    auto pair_done = [&](int c) {
      if (!kDedInv) return true;
      const bool ok = mbar_wait_sleep(&bars->invd, uint32_t(c & 1), err_word, DEVERR_MMA_TIMEOUT);
      tc_fence_after();
      return ok && *s_abort == 0u;
    };
    if (n_chunks > 0) {
      if (leader) {
        issue_qkg(0);
        issue_v(0);
        if (n_chunks > 1) issue_v(1);
      }
      qkg_last = 0;
      v_last[0] = 0;
      if (n_chunks > 1) v_last[1] = 1;
      for (int c = 0; c < 2 && c < n_chunks; ++c) {
        if (!sync_on(H_PREP)) goto issuer_abort;
        if (leader) {
          if (c + 1 < n_chunks) issue_qkg(c + 1);
          if (!kDedInv) issue_gram(c);
        }
        if (c + 1 < n_chunks) qkg_last = c + 1;
      }
      if ((!kDedInv && !sync_on(H_INV)) || !pair_done(0)) goto issuer_abort;
      if (leader) issue_wu(0);
      if (n_chunks > 2) {  // v stage 0 is free once W^T / U~^T of chunk 0 are done
        mbar_wait_sleep(&bars->wu, 0u, err_word, DEVERR_MMA_TIMEOUT);
        if (leader) issue_v(2);
        v_last[0] = 2;
      }
    }
    for (int j = 0; j < n_chunks; ++j) {
      const int b = j & 1;
      const bool more = j + 1 < n_chunks;
      if (!sync_on(H_COPY)) goto issuer_abort;
      if (leader) {  // MMA1: [U^T | O^T] += S^T [-W^T | Q~^T]
        const uint64_t st = kdesc128(sbase + OFF_ST), wq = mndesc(sbase + OFF_WQ + b * kWQBytes, 128 * 128);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
          umma_f16(tmem + tm_grp(b), dadv(st, kb * 16384 + ko), dadv(wq, ks * 2048), IDESC_UO, 1);
        }
        umma_commit(&bars->mma1);
      }
      // the operands of chunk j + 2 (H_PREP) come just before U^T of chunk j (H_U): MMA2 first,
      // which the chain and the read-out wait for, then the next chunk's loads and the Gram of
      // chunk j + 2, which queues behind MMA2 and is needed only one iteration later
      if (j + 2 < n_chunks && !sync_on(H_PREP)) goto issuer_abort;
      if (!sync_on(H_U)) goto issuer_abort;
      if (leader) {  // MMA2: [O^T | S^T] += U^T [P ; K^^T]^T
        const uint64_t ut = kdesc64(sbase + OFF_UT), pk = kdesc64(sbase + OFF_PK + (j % 3) * kPKBytes);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          umma_f16(tmem + tm_grp(b) + TM_O, dadv(ut, ks * 32), dadv(pk, ks * 32), IDESC_OS, 1);
        umma_commit(&bars->mma2);
      }
      if (j + 2 < n_chunks) {
        if (leader) {
          if (j + 3 < n_chunks) issue_qkg(j + 3);
          issue_gate(j);
          if (!kDedInv) issue_gram(j + 2);
        }
        if (j + 3 < n_chunks) qkg_last = j + 3;
        if (kStaged) gate_last = j;
      }
      if (kStaged && j + 2 >= n_chunks) {  // no operand hand-off left to piggyback on
        if (leader) issue_gate(j);
        gate_last = j;
      }
      if (more) {
        if ((!kDedInv && !sync_on(H_INV)) || !pair_done(j + 1)) goto issuer_abort;
        if (leader) issue_wu(j + 1);
        if (j + 3 < n_chunks) {  // v stage (j + 1) % 2 is free once W^T / U~^T of chunk j + 1 are done
          mbar_wait_sleep(&bars->wu, uint32_t((j + 1) & 1), err_word, DEVERR_MMA_TIMEOUT);
          if (leader) issue_v(j + 3);
          v_last[(j + 3) & 1] = j + 3;
        }
      }
    }
  }
  goto teardown;

issuer_abort:
  // the compute warps gave up: let this CTA's own MMAs and loads in flight finish (bounded) before
  // teardown frees the tensor memory and the CTA's shared memory. A commit tracks every tcgen05.mma
  // this thread issued before it, so one more commit on a barrier of its own covers them all.
  if (lane == 0) umma_commit(&bars->drain);
  __syncwarp();
  mbar_wait_sleep(&bars->drain, 0u, err_word, DEVERR_MMA_TIMEOUT);
  if (qkg_last >= 0) mbar_wait_sleep(&bars->qkg, uint32_t(qkg_last & 1), err_word, DEVERR_TMA_TIMEOUT);
  for (int s = 0; s < 2; ++s)
    if (v_last[s] >= 0) mbar_wait_sleep(&bars->v[s], uint32_t((v_last[s] >> 1) & 1), err_word, DEVERR_TMA_TIMEOUT);
  if (gate_last >= 0) mbar_wait_sleep(&bars->gate[0], uint32_t(gate_last & 1), err_word, DEVERR_TMA_TIMEOUT);

teardown:
  if (tid == 0) bulk_wait_all();  // the output tiles this thread stored
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

// the kernel's pointer type, spelled out (naming an instantiation here would instantiate it in
// every translation unit that includes this header)
using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, OutGate,
                          Runs, const float *, const float *, const int32_t *, const float *, void *, float *, int,
                          float, float, uint32_t *);

}  // namespace chunked
}  // namespace kda
