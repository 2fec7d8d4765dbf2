// kda_schedule.cu -- the two small kernels of the chunked prefill's schedules:
//
//  * longest-first order of packed sequences: the chunked kernel gives each (sequence, head)
//    chain one CTA and an SM holds one such CTA, so chains are dealt out in block order; putting
//    the longest sequences first keeps a long chain from starting in the last wave;
//  * the scan of the segmented schedule of one long sequence. The recurrence of Kimi K3 --
//    Architecture Notes, section 1.1 is affine in the state: over a segment of tokens,
//    S_end = M S_start + B, with M the product of the segment's (I - beta k k^T) Diag(alpha) and
//    B the state the segment reaches from zero. The chunked kernel computes M (the segment run
//    from S = I with v = 0) and B (run from S = 0); this kernel chains the segments,
//    S_{s+1} = M_s S_s + B_s, in fp32.
#include "kda_common.cuh"

namespace kda {

// order[r] = the sequence of rank r when sequences are sorted by length, longest first (ties by
// index). One thread per sequence counts the sequences that go before it; the lengths pass
// through shared memory in tiles.
__global__ void order_longest_first_kernel(const int32_t *__restrict__ cu_seqlens, int num_seqs,
                                           int32_t *__restrict__ order) {
  __shared__ int32_t len_tile[1024];
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  const int32_t mine = n < num_seqs ? cu_seqlens[n + 1] - cu_seqlens[n] : 0;
  int rank = 0;
  for (int base = 0; base < num_seqs; base += 1024) {
    __syncthreads();
    for (int i = threadIdx.x; i < 1024 && base + i < num_seqs; i += blockDim.x)
      len_tile[i] = cu_seqlens[base + i + 1] - cu_seqlens[base + i];
    __syncthreads();
    const int lim = num_seqs - base < 1024 ? num_seqs - base : 1024;
    for (int i = 0; i < lim; ++i) {
      const int32_t other = len_tile[i];
      rank += (other > mine || (other == mine && base + i < n)) ? 1 : 0;
    }
  }
  if (n < num_seqs) order[rank] = n;
}

// Scan of the segmented schedule, one CTA of 256 threads per head h (d_k = d_v = 128):
//   states[0] = init (or 0);  states[1] = runs[0] (segment 0 run from init);
//   states[s + 1] = M_s states[s] + B_s,  s = 1 .. m - 2,
// with B_s = runs[s] and M_s = runs[m - 2 + s]. Every array is [*, H, 128, 128] fp32, row-major
// (row = key channel c, column = value channel). Thread t forms an 8 x 8 block of the product:
// rows 8 (t / 16) .., columns 8 (t % 16) ..; S and M sit in shared memory.
__global__ void __launch_bounds__(256, 1)
    segment_scan_kernel(const float *__restrict__ runs, float *__restrict__ states,
                        const float *__restrict__ init_state, int H, int m) {
  constexpr int D = 128, DD = D * D;
  extern __shared__ __align__(16) float sh[];
  float *S = sh, *Mx = sh + DD;  // [128][128] each
  const int h = blockIdx.x, t = threadIdx.x;
  auto at = [&](const float *base, int slot) { return base + (int64_t(slot) * H + h) * DD; };
  auto at_w = [&](float *base, int slot) { return base + (int64_t(slot) * H + h) * DD; };
  // states[0]: the initial state; states[1]: segment 0's final state, which S starts from
  for (int i = t; i < DD / 4; i += 256) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4 *>(at_w(states, 0))[i] =
        init_state != nullptr ? reinterpret_cast<const float4 *>(at(init_state, 0))[i] : z;
    const float4 b0 = reinterpret_cast<const float4 *>(at(runs, 0))[i];
    reinterpret_cast<float4 *>(at_w(states, 1))[i] = b0;
    reinterpret_cast<float4 *>(S)[i] = b0;
  }
  const int r0 = 8 * (t >> 4), c0 = 8 * (t & 15);
  for (int s = 1; s + 1 < m; ++s) {
    __syncthreads();
    for (int i = t; i < DD / 4; i += 256) reinterpret_cast<float4 *>(Mx)[i] = reinterpret_cast<const float4 *>(at(runs, m - 2 + s))[i];
    __syncthreads();
    float acc[8][8];
    const float *B = at(runs, s);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 b0 = reinterpret_cast<const float4 *>(B + (r0 + i) * D + c0)[0];
      const float4 b1 = reinterpret_cast<const float4 *>(B + (r0 + i) * D + c0)[1];
      acc[i][0] = b0.x, acc[i][1] = b0.y, acc[i][2] = b0.z, acc[i][3] = b0.w;
      acc[i][4] = b1.x, acc[i][5] = b1.y, acc[i][6] = b1.z, acc[i][7] = b1.w;
    }
#pragma unroll 4
    for (int k = 0; k < D; ++k) {
      float mk[8], sk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mk[i] = Mx[(r0 + i) * D + k];
      const float4 s0 = reinterpret_cast<const float4 *>(S + k * D + c0)[0];
      const float4 s1 = reinterpret_cast<const float4 *>(S + k * D + c0)[1];
      sk[0] = s0.x, sk[1] = s0.y, sk[2] = s0.z, sk[3] = s0.w, sk[4] = s1.x, sk[5] = s1.y, sk[6] = s1.z, sk[7] = s1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(mk[i], sk[j], acc[i][j]);
    }
    __syncthreads();  // every thread is past S before it is overwritten
    float *dst = at_w(states, s + 1);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 a0 = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      const float4 a1 = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
      reinterpret_cast<float4 *>(S + (r0 + i) * D + c0)[0] = a0;
      reinterpret_cast<float4 *>(S + (r0 + i) * D + c0)[1] = a1;
      reinterpret_cast<float4 *>(dst + (r0 + i) * D + c0)[0] = a0;
      reinterpret_cast<float4 *>(dst + (r0 + i) * D + c0)[1] = a1;
    }
  }
}

cudaError_t launch_order_longest_first(const int32_t *cu_seqlens, int num_seqs, int32_t *order, cudaStream_t stream) {
  order_longest_first_kernel<<<(num_seqs + 255) / 256, 256, 0, stream>>>(cu_seqlens, num_seqs, order);
  return cudaGetLastError();
}

cudaError_t launch_segment_scan(const float *runs, float *states, const float *init_state, int H, int m,
                                cudaStream_t stream) {
  const int smem = 2 * 128 * 128 * 4;
  const cudaError_t attr = cudaFuncSetAttribute(segment_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (attr != cudaSuccess) return attr;
  segment_scan_kernel<<<H, 256, smem, stream>>>(runs, states, init_state, H, m);
  return cudaGetLastError();
}

}  // namespace kda
