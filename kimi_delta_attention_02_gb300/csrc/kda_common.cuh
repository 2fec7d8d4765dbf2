// kda_common.cuh -- device helpers shared by the libkda kernels (sm_103a only).
//
// bf16 conversion, the library's device error word, mbarrier / TMA / tcgen05
// inline-PTX wrappers and the shared-memory operand layout used by the
// tensor-core kernels. Everything here is written for Blackwell (sm_100 family,
// compiled as sm_103a); nothing has a fallback for older architectures.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// ---------------------------------------------------------------------------
// Device error word. Kernels OR a code into it when a bounded wait gives up or
// an input is out of their range; kda_check_device_error() reads and clears it. It lives in kda_api.cu; kernels
// receive its device address (device_error_word()) as an argument.
// ---------------------------------------------------------------------------
enum : uint32_t {
  DEVERR_NONE = 0,
  DEVERR_TMA_TIMEOUT = 1u << 0,
  DEVERR_MMA_TIMEOUT = 1u << 1,
  DEVERR_RANGE = 1u << 2,  // an input outside the range the kernel computes exactly
};

// Device address of the error word on the current device (nullptr if the
// lookup failed). Host only; defined in kda_api.cu.
uint32_t *device_error_word();

__device__ __forceinline__ void raise_device_error(uint32_t *word, uint32_t code) {
  if (word != nullptr) atomicOr(word, code);
}

// A spin of this many polls (each a try_wait that itself suspends for a
// hardware-chosen time) is far beyond any legitimate wait in these kernels.
constexpr uint32_t kSpinLimit = 1u << 24;

// ---------------------------------------------------------------------------
// bf16 <-> fp32 without the cuda_bf16 header: bf16 is the top half of binary32.
// Conversion to bf16 rounds to nearest-even (NaN stays NaN).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t f32_to_bf16(float x) { return uint16_t(pack_bf16x2(x, 0.f) & 0xffffu); }

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t p) {
  return make_float2(__uint_as_float(p << 16), __uint_as_float(p & 0xffff0000u));
}

// fp16 pack (round to nearest-even); used for tensor-core operands whose range fits binary16
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t f32_to_f16(float x) { return uint16_t(pack_f16x2(x, 0.f) & 0xffffu); }

// fp32 -> tf32 (10-bit mantissa), round to nearest with ties away from zero; the
// tensor core would otherwise drop the low mantissa bits
__device__ __forceinline__ float round_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

__device__ __forceinline__ float bf16_or_f32(uint16_t h) { return bf16_to_f32(h); }
__device__ __forceinline__ float bf16_or_f32(float x) { return x; }

// Element load/store for the two I/O dtypes (fp32 or bf16 bits).
template <bool kBF16>
__device__ __forceinline__ float load_elem(const void *base, int64_t idx) {
  if constexpr (kBF16) return bf16_to_f32(static_cast<const uint16_t *>(base)[idx]);
  else return static_cast<const float *>(base)[idx];
}
template <bool kBF16>
__device__ __forceinline__ void store_elem(void *base, int64_t idx, float x) {
  if constexpr (kBF16) static_cast<uint16_t *>(base)[idx] = f32_to_bf16(x);
  else static_cast<float *>(base)[idx] = x;
}

// log-decay clamp: g < lb ? lb : g (a NaN compares false and passes through)
__device__ __forceinline__ float clamp_log_decay(float g, float lb) { return g < lb ? lb : g; }

// The gated log-decay (Kimi K3 -- Architecture Notes, section 1.2, the K3 row of the
// mapping table from decay logits to log-decay): g = g_min * Sigmoid(e^{A_h} z), with
// a_h = e^{A_h} taken once per head. The result lies in (g_min, 0]. Where e^{-a_h z} is
// beyond 2^100 the quotient is below 2^-97 |g_min|, i.e. alpha = 1 in fp32, so the
// denominator is capped there to keep the fast division in its range; a NaN logit
// stays NaN.
__device__ __forceinline__ float gated_log_decay(float z, float a_h, float g_min) {
  float e = __expf(-a_h * z);
  e = e > 0x1p100f ? 0x1p100f : e;
  return __fdividef(g_min, 1.f + e);
}

// Sigmoid(x) = 1 / (1 + 2^{-x log2 e}) on the SFU: ex2.approx and rcp.approx (each about one
// ulp). 2^{-x log2 e} = inf gives 0; a NaN stays NaN.
__device__ __forceinline__ float sigmoid_approx(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return r;
}

// Packed fp32 pairs (Blackwell's two-wide fp32 FMA / multiply / add: one instruction, two
// results, each rounded as its scalar counterpart).
__device__ __forceinline__ unsigned long long f2_pack(float2 a) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(unsigned long long r) {
  float2 a;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
  return a;
}
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)), "l"(f2_pack(c)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(r);
}
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(r);
}

// sigmoid_approx of two values, its multiply and add packed (the same roundings, so the same bits)
__device__ __forceinline__ float2 sigmoid2_approx(float2 x) {
  const float2 s = f2_mul(x, make_float2(-1.4426950408889634f, -1.4426950408889634f));
  float e0, e1, r0, r1;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(s.x));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(s.y));
  const float2 d = f2_add(make_float2(e0, e1), make_float2(1.f, 1.f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(d.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(d.y));
  return make_float2(r0, r1);
}

// The output gate of Kimi K3 -- Architecture Notes, section 1.3 ("Full-rank output gate"):
// out = Sigmoid(r) * w * o * rstd, with rstd = 1 / sqrt(mean of o^2 over the head's d_v
// channels + eps) formed by the caller.
__device__ __forceinline__ float output_gate(float o, float rstd, float w, float r) {
  return o * rstd * w * sigmoid_approx(r);
}

// Sums v[e] over the 32 lanes of a warp for all N entries at once (N a power of two, 2..32):
// each halving round sends one half of the remaining entries to the partner lane and adds the
// other half, so N - 1 shuffles leave one entry per lane, which the remaining rounds sum as a
// plain butterfly. Afterwards lane l holds the total of entry (l >> (5 - log2 N)) & (N - 1).
// v is overwritten.
template <int N>
__device__ __forceinline__ float lane_sums(float (&v)[N], int lane) {
  int off = 16;
#pragma unroll
  for (int n = N; n > 1; n >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float s = v[0];
#pragma unroll
  for (; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

// The unbounded log-decay of the earlier models (Kimi K3 -- Architecture Notes, section 1.2,
// the GDN / Mamba-2 / Kimi Linear row of the mapping table): g = -e^{A_h} Softplus(z), with
// Softplus(z) = max(z, 0) + log(1 + e^{-|z|}) (no overflow for large |z|); a NaN stays NaN.
__device__ __forceinline__ float unbounded_log_decay(float z, float a_h) {
  return -a_h * (fmaxf(z, 0.f) + __logf(1.f + __expf(-fabsf(z))));
}

// Decay forms of the token-recurrent and decode kernels.
enum : int { DECAY_CLAMPED = 0, DECAY_GATED = 1, DECAY_UNBOUNDED = 2 };

// ---------------------------------------------------------------------------
// Shared-memory addresses and fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Make generic-proxy shared-memory writes visible to the async proxy (TMA, tcgen05.mma).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// One arrival on `bar` (release: this thread's earlier writes are visible to a thread whose wait
// sees the phase complete).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait that lets the thread sleep until the phase completes or `ns` nanoseconds pass
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity to complete. Returns false
// (and records `code` in the device error word) when the limit is reached.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *err_word, uint32_t code) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  raise_device_error(err_word, code);
  return false;
}
// The same bound, waiting in sleeps of up to 10 microseconds (about 2 s in total):
// a waiting thread issues a handful of instructions instead of spinning. A phase that
// has already completed is seen by one plain probe, which is much cheaper than a
// probe with a suspend-time hint.
constexpr uint32_t kSleepNs = 10000, kSleepLimit = 200000;
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t *err_word, uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < kSleepLimit; ++i)
    if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
  raise_device_error(err_word, code);
  return false;
}

// The value itself, hidden from the optimizer's range and relation analysis.
__device__ __forceinline__ int opaque_int(int x) {
  asm volatile("" : "+r"(x));
  return x;
}

// ---------------------------------------------------------------------------
// Named CTA barriers (ids 1..15; id 0 is the one __syncthreads uses). `n` counts
// threads, a multiple of 32; each taking part warp executes the call as a whole.
// An arrive does not wait; it releases the arriving threads' earlier writes to
// the threads that sync on the same barrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// barrier among `n` threads that also returns the OR of `pred` over them
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(uint32_t(pred)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------------------
// TMA (tensor map loads into shared memory, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const void *tmap, uint64_t *bar, int32_t x,
                                            int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
      "%5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// Store a shared-memory tile to global memory through a tensor map (bulk-group completion):
// the issuing thread commits the group and waits on it with bulk_wait_read (the tile may be
// overwritten) or bulk_wait_all (the writes are done).
__device__ __forceinline__ void tma_store_3d(const void *tmap, const void *smem_src, int32_t x, int32_t y,
                                             int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(tmap),
               "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
// A small asynchronous copy global -> shared of kBytes (4, 8 or 16; both addresses aligned to
// it), through L1; cp_async_wait_all makes this thread's copies visible to it.
template <int kBytes>
__device__ __forceinline__ void cp_async_small(void *smem, const void *gmem) {
  static_assert(kBytes == 4 || kBytes == 8 || kBytes == 16, "cp.async takes 4, 8 or 16 bytes");
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(smem_u32(smem)), "l"(gmem), "n"(kBytes)
               : "memory");
}
// 16 bytes global -> shared through L2 only; ok == false writes 16 zero bytes and reads nothing
__device__ __forceinline__ void cp_async_16_zfill(void *smem, const void *gmem, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bring a tile of a tensor map into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_3d(const void *tmap, int32_t x, int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(tmap), "r"(x), "r"(y),
               "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory allocation, MMA, commit, loads, fences
// ---------------------------------------------------------------------------
// Allocate `ncols` TMEM columns (power of two >= 32); whole warp; address -> *dst (smem).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] x B[smem desc], kind::f16 (bf16 or fp16 inputs per the
// instruction descriptor, fp32 accumulate).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A x B, kind::tf32 (fp32 operands read as tf32, fp32 accumulate).
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 32-bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {  // v: 16 registers
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 lanes x 32-bit, 8 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float *v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
// The same loads with their wait in one statement: the registers are complete when the
// compiler first sees them (for a load whose wait follows at once).
__device__ __forceinline__ void tmem_ld16_wait(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld8_wait(uint32_t taddr, float *v) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
// tcgen05.ld fills its destination registers asynchronously: nothing may read them before
// tcgen05.wait::ld. The compiler sees them as written by the load itself and may move plain
// arithmetic on them above the wait, so the wait takes the arrays it completes and passes each
// register through an empty volatile statement after it: every later use depends on that
// statement, and volatile statements keep their order.
template <int N>
__device__ __forceinline__ void tmem_regs_ready(float (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+f"(v[i]));
}
template <typename... Arrays>
__device__ __forceinline__ void tmem_ld_wait(Arrays &...loaded) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  (tmem_regs_ready(loaded), ...);
}

// 32 lanes x 32-bit, 16 consecutive columns per thread, registers -> tensor memory.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Operand layouts in shared memory (128-byte swizzle, bf16).
//
// A tile is stored as "blocks" of 64 contiguous elements (128 bytes) along its
// contiguous dimension; within a block, row r occupies 128 bytes at r*128 and
// its 16-byte chunk j sits at chunk (j XOR (r mod 8)). Blocks follow each other
// at `rows * 128` bytes. Block bases are 1024-byte aligned. This is the layout
// TMA writes with CU_TENSOR_MAP_SWIZZLE_128B and a 64-element inner box.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col, uint32_t rows) {
  // byte offset of 16-bit element (row, col) in a tile with `rows` rows
  const uint32_t blk = col >> 6, c = col & 63u;
  return blk * rows * 128u + row * 128u + ((((c >> 3) ^ row) & 7u) << 4) + ((c & 7u) << 1);
}
__device__ __forceinline__ uint32_t sw128_offset32(uint32_t row, uint32_t col, uint32_t rows) {
  // byte offset of 32-bit element (row, col): blocks of 32 elements per 128-byte row
  const uint32_t blk = col >> 5, c = col & 31u;
  return blk * rows * 128u + row * 128u + ((((c >> 2) ^ row) & 7u) << 4) + ((c & 3u) << 2);
}
// byte offset of the 16-byte chunk holding elements (row, 8*j .. 8*j+7) of block `blk`
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t row, uint32_t j, uint32_t blk, uint32_t rows) {
  return blk * rows * 128u + row * 128u + (((j ^ row) & 7u) << 4);
}

// The 64-byte swizzle (K-major tiles whose rows hold 32 16-bit elements): row r
// occupies 64 bytes at r*64 and its 16-byte chunk j sits at chunk (j XOR ((r/2) mod 4));
// atoms of 8 rows (512 bytes) are 512-byte aligned.
__device__ __forceinline__ uint32_t sw64_chunk(uint32_t row, uint32_t j) {
  return row * 64u + (((j ^ (row >> 1)) & 3u) << 4);
}
__device__ __forceinline__ uint32_t sw64_offset(uint32_t row, uint32_t col) {
  return sw64_chunk(row, col >> 3) + ((col & 7u) << 1);
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and stride
// byte offsets (all >> 4), fixed version bits 0b001 at [46,49), swizzle mode at [61,64).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle_mode) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(swizzle_mode & 7u) << 61;
  return d;
}
constexpr uint32_t kSwizzle128B = 2, kSwizzle64B = 4;

// Instruction descriptor with fp32 D. Operand format codes: kind::f16 takes
// 0 = f16 or 1 = bf16 (A and B the same), kind::tf32 takes 2 = tf32.
enum : uint32_t { UMMA_F16 = 0, UMMA_BF16 = 1, UMMA_TF32 = 2 };
__host__ __device__ constexpr uint32_t umma_idesc(uint32_t fmt, uint32_t M, uint32_t N, bool a_mn_major,
                                                  bool b_mn_major, bool negate_a) {
  return (1u << 4)                      // D format: f32
         | (fmt << 7)                   // A format
         | (fmt << 10)                  // B format
         | (uint32_t(negate_a) << 13)   // negate A
         | (uint32_t(a_mn_major) << 15) // A major: 0 = K-major, 1 = MN-major
         | (uint32_t(b_mn_major) << 16) // B major
         | ((N >> 3) << 17)             // N / 8
         | ((M >> 4) << 24);            // M / 16
}
__host__ __device__ constexpr uint32_t umma_idesc_bf16(uint32_t M, uint32_t N, bool a_mn_major, bool b_mn_major,
                                                       bool negate_a) {
  return umma_idesc(UMMA_BF16, M, N, a_mn_major, b_mn_major, negate_a);
}

}  // namespace kda
