// kda_selftest.cu -- a single tcgen05.mma on operands staged in the same
// 128-byte-swizzled shared-memory layouts the chunked prefill kernel uses, with
// the whole 128-lane accumulator copied back. Tests compare it with a host
// matrix product to pin the descriptor encodings (K-major and MN-major
// operands, the M = 64 accumulator lanes, the negate bit) that the chunked
// kernel depends on.
#include "../../include/kda_selftest.h"
#include "kda_common.cuh"

namespace kda {

constexpr int kSelftestTileBytes = 64 * 1024;  // per operand; twice the largest tile

__global__ void __launch_bounds__(128, 1)
    selftest_umma_kernel(const float *__restrict__ A, const float *__restrict__ B, float *__restrict__ D, int M,
                         int N, int K, int fmt, int sw64, int a_mn, int b_mn, int neg_a, uint32_t a_lbo,
                         uint32_t a_sbo,
                         uint32_t b_lbo, uint32_t b_sbo, int *__restrict__ status, uint32_t *err_word) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = smem, *sB = smem + kSelftestTileBytes;
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int i = tid; i < 2 * kSelftestTileBytes / 16; i += 128) reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  // stage A[m][k] and B[n][k] in the operand format. K-major tiles have rows m (or n)
  // and 128-byte K blocks (64 16-bit or 32 tf32 elements); MN-major tiles (16-bit
  // only) have rows k and 64-wide M (or N) blocks.
  // with sw64, K-major 16-bit tiles use 64-byte rows: blocks of 32 K elements, `rows` * 64 bytes apart
  // (MN-major tiles keep the 128-byte swizzle)
  auto put = [&](uint8_t *tile, uint32_t row, uint32_t col, uint32_t rows, float x, bool k_major) {
    if (sw64 && k_major) {
      const uint16_t h = fmt == UMMA_BF16 ? f32_to_bf16(x) : f32_to_f16(x);
      *reinterpret_cast<uint16_t *>(tile + (col >> 5) * rows * 64 + sw64_offset(row, col & 31)) = h;
    } else if (fmt == UMMA_TF32) {
      *reinterpret_cast<float *>(tile + sw128_offset32(row, col, rows)) = round_tf32(x);
    } else {
      const uint16_t h = fmt == UMMA_BF16 ? f32_to_bf16(x) : f32_to_f16(x);
      *reinterpret_cast<uint16_t *>(tile + sw128_offset(row, col, rows)) = h;
    }
  };
  for (int i = tid; i < M * K; i += 128) {
    const int m = i / K, kk = i % K;
    if (a_mn) put(sA, kk, m, K, A[i], false);
    else put(sA, m, kk, M, A[i], true);
  }
  for (int i = tid; i < N * K; i += 128) {
    const int n = i / K, kk = i % K;
    if (b_mn) put(sB, kk, n, K, B[i], false);
    else put(sB, n, kk, N, B[i], true);
  }
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (tid == 0) {
    const uint32_t idesc = umma_idesc(uint32_t(fmt), M, N, a_mn, b_mn, neg_a);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    const int kstep = fmt == UMMA_TF32 ? 8 : 16;  // K per instruction: 32 bytes of either type
    for (int ks = 0; ks < K / kstep; ++ks) {
      // K-major: 4 instruction steps of 32 bytes per 128-byte block, then the next block
      // MN-major: the next 16 rows of K are 16 * 128 bytes further on
      const uint32_t per_blk = sw64 ? 2 : 4, row_bytes = sw64 ? 64 : 128;
      const uint32_t a_addr = a_mn ? a0 + ks * 2048 : a0 + (ks / per_blk) * M * row_bytes + (ks % per_blk) * 32;
      const uint32_t b_addr = b_mn ? b0 + ks * 2048 : b0 + (ks / per_blk) * N * row_bytes + (ks % per_blk) * 32;
      const uint64_t ad = umma_desc(a_addr, a_lbo, a_sbo, (sw64 && !a_mn) ? kSwizzle64B : kSwizzle128B);
      const uint64_t bd = umma_desc(b_addr, b_lbo, b_sbo, (sw64 && !b_mn) ? kSwizzle64B : kSwizzle128B);
      if (fmt == UMMA_TF32) umma_tf32(tmem, ad, bd, idesc, ks > 0);
      else umma_f16(tmem, ad, bd, idesc, ks > 0);
    }
    umma_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0, err_word, DEVERR_MMA_TIMEOUT);
  if (!ok && tid == 0) *status = 1;
  tc_fence_after();
  // copy the accumulator: warp w reads lanes 32w..32w+31, all N columns
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 16) {
      float vals[16];
      tmem_ld16_wait(tmem + (uint32_t(32 * warp) << 16) + c0, vals);
      for (int j = 0; j < 16; ++j) D[(32 * warp + lane) * N + c0 + j] = vals[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace kda

namespace kda {
namespace {
// Whether every shared-memory byte the MMAs of kda_selftest_umma read for one operand stays inside
// its kSelftestTileBytes tile, given the descriptor offsets the caller chose. K-major: the last
// instruction starts in 128-byte (or 64-byte) K block (steps - 1) / per_block, and its `rows` rows
// span (rows / 8 - 1) SBO strides plus one 8-row atom. MN-major: the last instruction starts
// (steps - 1) * 2048 bytes in, its rows of 64 elements span ceil(rows / 64) - 1 LBO strides, and
// its 16 K rows one SBO stride plus one 8-row atom of 128 bytes.
bool selftest_footprint_ok(uint32_t rows, uint32_t K, int fmt, bool sw64, bool mn_major, uint32_t lbo,
                           uint32_t sbo) {
  const uint64_t kstep = fmt == UMMA_TF32 ? 8 : 16, steps = K / kstep;
  uint64_t end;
  if (mn_major) {
    end = (steps - 1) * 2048 + ((rows + 63) / 64 - 1) * uint64_t(lbo) + uint64_t(sbo) + 1024;
  } else {
    const uint64_t per_blk = sw64 ? 2 : 4, row_bytes = sw64 ? 64 : 128;
    end = ((steps - 1) / per_blk) * rows * row_bytes + (rows / 8 - 1) * uint64_t(sbo) + 8 * row_bytes;
  }
  return end <= uint64_t(kSelftestTileBytes);
}
}  // namespace
}  // namespace kda

extern "C" kda_status kda_selftest_umma(const float *A, const float *B, float *D, int32_t M, int32_t N, int32_t K,
                                        int32_t fmt, int32_t sw64, int32_t a_mn_major, int32_t b_mn_major,
                                        int32_t negate_a,
                                        uint32_t a_lbo, uint32_t a_sbo, uint32_t b_lbo, uint32_t b_sbo,
                                        int32_t *status, void *stream) {
  using namespace kda;
  if (!A || !B || !D || !status) return KDA_ERR_INVALID_ARG;
  if (fmt < 0 || fmt > 2) return KDA_ERR_INVALID_ARG;
  if (!(M == 64 || M == 128) || N < 16 || N > 256 || N % 16 || K < 16 || K > 128 || K % 16)
    return KDA_ERR_UNSUPPORTED;
  if (a_mn_major && (M % 64 || fmt == UMMA_TF32)) return KDA_ERR_UNSUPPORTED;
  if (b_mn_major && (N % 64 || fmt == UMMA_TF32)) return KDA_ERR_UNSUPPORTED;
  if (fmt == UMMA_TF32 && negate_a) return KDA_ERR_UNSUPPORTED;
  if (sw64 && fmt == UMMA_TF32) return KDA_ERR_UNSUPPORTED;
  if (a_lbo > 32768 || a_sbo > 32768 || b_lbo > 32768 || b_sbo > 32768) return KDA_ERR_UNSUPPORTED;
  // descriptors whose reads would leave the operand's staged tile
  if (!selftest_footprint_ok(uint32_t(M), uint32_t(K), fmt, sw64 != 0, a_mn_major != 0, a_lbo, a_sbo) ||
      !selftest_footprint_ok(uint32_t(N), uint32_t(K), fmt, sw64 != 0, b_mn_major != 0, b_lbo, b_sbo))
    return KDA_ERR_UNSUPPORTED;
  const int smem = 2 * kSelftestTileBytes + 1024;
  if (cudaFuncSetAttribute(selftest_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return KDA_ERR_CUDA;
  selftest_umma_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
      A, B, D, M, N, K, fmt, sw64 != 0, a_mn_major, b_mn_major, negate_a, a_lbo, a_sbo, b_lbo, b_sbo, status,
      device_error_word());
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

namespace kda {
namespace {

// A bounded wait on a phase that never completes: the failure path of every wait in the library.
__global__ void selftest_wait_kernel(uint32_t *status, uint32_t *err_word) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none comes
    fence_mbarrier_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_sleep(&bar, 0u, err_word, DEVERR_TMA_TIMEOUT);
  if (threadIdx.x == 0) *status = ok ? 0u : 1u;
}

}  // namespace
}  // namespace kda

extern "C" kda_status kda_selftest_wait_timeout(uint32_t *status, void *stream) {
  if (status == nullptr || (reinterpret_cast<uintptr_t>(status) & 3u) != 0) return KDA_ERR_INVALID_ARG;
  kda::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, kda::device_error_word());
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
