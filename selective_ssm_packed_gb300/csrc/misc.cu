// misc.cu -- position indices from cu_seqlens, and fixed-order row sums.
#include "common.cuh"
#include "kernels.h"

namespace vssm {

// position_indices[t] = t - cu[s] for the sequence s holding token t: the
// largest s with cu[s] <= t (upper-bound search), which skips zero-length
// sequences.  The same grid also checks cu_seqlens (starts at 0, never
// decreases, ends at T) and ORs kStatusBadCu into *status on failure.
__global__ void __launch_bounds__(256) position_indices_kernel(const int32_t* __restrict__ cu,
                                                               int32_t S, int64_t T,
                                                               int32_t* __restrict__ pos,
                                                               int32_t* status) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t s = i0; s <= S; s += stride) {
    const int32_t c = cu[s];
    bool bad = (s == 0 && c != 0) || (s > 0 && c < cu[s - 1]) || (s == S && (int64_t)c != T);
    if (bad && status) atomicOr(status, kStatusBadCu);
  }
  for (int64_t t = i0; t < T; t += stride) {
    int32_t lo = 0, hi = S;  // answer in [lo, hi]
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    pos[t] = (int32_t)(t - (int64_t)cu[lo]);
  }
}

cudaError_t launch_position_indices(const int32_t* cu, int32_t num_seqs, int64_t T, int32_t* pos,
                                    int32_t* status, cudaStream_t st) {
  const int64_t work = T > (int64_t)num_seqs + 1 ? T : (int64_t)num_seqs + 1;
  int64_t blocks = (work + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  position_indices_kernel<<<(unsigned)blocks, 256, 0, st>>>(cu, num_seqs, T, pos, status);
  return cudaGetLastError();
}

// out[m] = sum over p = 0..P-1 (in order) of in[p*ld + m].  One thread per
// column, so the summation order is fixed and the result bitwise repeatable.
__global__ void __launch_bounds__(256) sum_rows_kernel(const float* __restrict__ in, int64_t P,
                                                       int64_t M, int64_t ld,
                                                       float* __restrict__ out) {
  const int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  float acc = 0.0f;
  const float* p = in + m;
  int64_t r = 0;
  for (; r + 4 <= P; r += 4) {
    const float a0 = __ldcs(p + (r + 0) * ld), a1 = __ldcs(p + (r + 1) * ld);
    const float a2 = __ldcs(p + (r + 2) * ld), a3 = __ldcs(p + (r + 3) * ld);
    acc += a0; acc += a1; acc += a2; acc += a3;
  }
  for (; r < P; ++r) acc += __ldcs(p + r * ld);
  out[m] = acc;
}

cudaError_t launch_sum_rows(const float* in, int64_t P, int64_t M, int64_t ld, float* out,
                            cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  const int64_t blocks = (M + 255) / 256;
  sum_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(in, P, M, ld, out);
  return cudaGetLastError();
}

}  // namespace vssm
