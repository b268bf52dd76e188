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
  int64_t blocks = grid_stride_blocks(work);
  if (blocks < 1) blocks = 1;
  position_indices_kernel<<<(unsigned)blocks, 256, 0, st>>>(cu, num_seqs, T, pos, status);
  return cudaGetLastError();
}

// BD[(t NSP + p) 2 + o] = (b0, b0, b1, b1) for o = 0 and (b1, b1, b0, b0) for
// o = 1, with (b0, b1) = (B[t][2p], B[t][2p+1]) as fp32, zero for t >= T; CD
// likewise from C.  One thread per (token, state pair).
// packed (N = 16, CD unused): per chunk of kBwdChunk tokens, kBwdChunkRow
// bytes: first the float4 rows [token][state pair][order] = (b0, b1, c0, c1)
// for o = 0 and (b1, b0, c1, c0) for o = 1, then the chunk's position
// indices (zero past T, written by the chunk's first state pair).
template <typename T>
__global__ void __launch_bounds__(256) double_bc_kernel(const T* __restrict__ B, const T* __restrict__ C,
                                                        int64_t nT, int64_t n_items, int N, int packed,
                                                        const int32_t* __restrict__ pos,
                                                        float4* __restrict__ BD, float4* __restrict__ CD) {
  const int NSP = N / 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_items; i += stride) {
    const int64_t t = i / NSP;
    const int p = (int)(i - t * NSP);
    float2 b = make_float2(0.0f, 0.0f), c = make_float2(0.0f, 0.0f);
    if (t < nT) {
      b = make_float2(to_f(B[t * N + 2 * p]), to_f(B[t * N + 2 * p + 1]));
      c = make_float2(to_f(C[t * N + 2 * p]), to_f(C[t * N + 2 * p + 1]));
    }
    if (packed) {
      const int64_t ch = t / kBwdChunk, tl = t - ch * kBwdChunk;
      float4* row = BD + ch * (kBwdChunkRow / 16) + (tl * NSP + p) * 2;
      row[0] = make_float4(b.x, b.y, c.x, c.y);
      row[1] = make_float4(b.y, b.x, c.y, c.x);
      if (p == 0)
        reinterpret_cast<int32_t*>(BD + ch * (kBwdChunkRow / 16) + kBwdChunk * NSP * 2)[tl] = t < nT ? pos[t] : 0;
    } else {
      BD[2 * i] = make_float4(b.x, b.x, b.y, b.y);
      BD[2 * i + 1] = make_float4(b.y, b.y, b.x, b.x);
      CD[2 * i] = make_float4(c.x, c.x, c.y, c.y);
      CD[2 * i + 1] = make_float4(c.y, c.y, c.x, c.x);
    }
  }
}

cudaError_t launch_double_bc(const void* B, const void* C, IO io, int64_t T, int64_t T_pad, int N, bool packed,
                             const int32_t* pos, float4* BD, float4* CD, cudaStream_t st) {
  if (packed && (N != 16 || !pos)) return cudaErrorInvalidValue;
  const int64_t n_items = T_pad * (N / 2);
  if (n_items <= 0) return cudaSuccess;
  const int64_t blocks = grid_stride_blocks(n_items);
  if (io == IO::F32)
    double_bc_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(static_cast<const float*>(B),
                                                              static_cast<const float*>(C), T, n_items, N, packed ? 1 : 0, pos, BD,
                                                              CD);
  else
    double_bc_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(B), static_cast<const __nv_bfloat16*>(C), T, n_items, N, packed ? 1 : 0, pos,
        BD, CD);
  return cudaGetLastError();
}

// dst[i] = src[i] widened from bf16 (the upper half of the fp32 word), eight
// values per thread and 16-byte access where the arrays allow it.
__global__ void __launch_bounds__(256) widen_bf16_kernel(const uint16_t* __restrict__ src,
                                                         float* __restrict__ dst, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t n8 = n / 8;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 q = reinterpret_cast<const uint4*>(src)[i];
    float4* d = reinterpret_cast<float4*>(dst) + 2 * i;
    d[0] = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xffff0000u),
                       __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xffff0000u));
    d[1] = make_float4(__uint_as_float(q.z << 16), __uint_as_float(q.z & 0xffff0000u),
                       __uint_as_float(q.w << 16), __uint_as_float(q.w & 0xffff0000u));
  }
  for (int64_t i = 8 * n8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = __uint_as_float((uint32_t)src[i] << 16);
}

cudaError_t launch_widen_bf16(const void* src, float* dst, int64_t n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = grid_stride_blocks((n + 7) / 8);
  widen_bf16_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint16_t*>(src), dst, n);
  return cudaGetLastError();
}

// The N = 16 backward's tile parameters: for each 64-channel tile, A * log2 e
// as [channel][n] (A = -exp(A_log), as -2^(A_log log2 e), when the rows hold
// A_log), then dt_bias and Dskip; zero for absent vectors and channels >= D.
__global__ void __launch_bounds__(256) bwd_tile_params_kernel(const float* __restrict__ A,
                                                              const float* __restrict__ bias,
                                                              const float* __restrict__ dsk, int D, int a_log,
                                                              float* __restrict__ out, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = i / kBwdTileParams;
    const int k = (int)(i - tile * kBwdTileParams);
    float v = 0.0f;
    if (k < 64 * 16) {
      const int64_t d = tile * 64 + k / 16;
      if (d < D) {
        const float r = __ldg(A + d * 16 + k % 16);
        v = a_log ? -ex2(r * kLog2e) * kLog2e : r * kLog2e;
      }
    } else if (k < 64 * 16 + 64) {
      const int64_t d = tile * 64 + (k - 64 * 16);
      if (bias && d < D) v = __ldg(bias + d);
    } else {
      const int64_t d = tile * 64 + (k - 64 * 16 - 64);
      if (dsk && d < D) v = __ldg(dsk + d);
    }
    out[i] = v;
  }
}

cudaError_t launch_bwd_tile_params(const float* A, const float* dt_bias, const float* Dskip, int D, bool a_log,
                                   float* tpar, cudaStream_t st) {
  const int64_t n = (int64_t)(D + 63) / 64 * kBwdTileParams;
  if (n <= 0) return cudaSuccess;
  bwd_tile_params_kernel<<<(unsigned)grid_stride_blocks(n), 256, 0, st>>>(A, dt_bias, Dskip, D, a_log ? 1 : 0, tpar,
                                                                          n);
  return cudaGetLastError();
}

// The forward's A rows: out[(tile * N/4 + b) * 32 + c] = the states 4b .. 4b+3
// of channel d = 32 tile + c, each A * log2 e, where A = -exp(A_log) (as
// -2^(A_log log2 e)) when the rows hold A_log; zero for d >= D.
__global__ void __launch_bounds__(256) prep_a_kernel(const float* __restrict__ A, int D, int N, int a_log,
                                                     float4* __restrict__ out, int64_t n) {
  const int nb = N / 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % kTile);
    const int64_t tb = i / kTile;
    const int b = (int)(tb % nb);
    const int64_t d = (tb / nb) * kTile + c;
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (d < D) {
      const float4 r = __ldg(reinterpret_cast<const float4*>(A + d * N) + b);
      if (a_log)
        v = make_float4(-ex2(r.x * kLog2e) * kLog2e, -ex2(r.y * kLog2e) * kLog2e, -ex2(r.z * kLog2e) * kLog2e,
                        -ex2(r.w * kLog2e) * kLog2e);
      else
        v = make_float4(r.x * kLog2e, r.y * kLog2e, r.z * kLog2e, r.w * kLog2e);
    }
    out[i] = v;
  }
}

cudaError_t launch_prep_a(const float* A, int D, int N, bool a_log, float4* Af, cudaStream_t st) {
  const int64_t n = (int64_t)(D + kTile - 1) / kTile * kTile * (N / 4);
  if (n <= 0) return cudaSuccess;
  prep_a_kernel<<<(unsigned)grid_stride_blocks(n), 256, 0, st>>>(A, D, N, a_log ? 1 : 0, Af, n);
  return cudaGetLastError();
}

// A value is NaN or infinite when its exponent bits are all ones: bits
// 0x7f800000 of an f32, 0x7f80 of a bf16 (two bf16 values per 32-bit word).
__global__ void __launch_bounds__(256) nonfinite_kernel(const uint32_t* __restrict__ p, int64_t words,
                                                        int bf16, int32_t* status) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += stride) {
    const uint32_t v = __ldg(p + i);
    bad |= (v & 0x7f800000u) == 0x7f800000u;
    if (bf16) bad |= (v & 0x7f80u) == 0x7f80u;
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, kStatusNonFinite);
}

// The last value of an odd count of bf16 values, which has no word of its own.
__global__ void nonfinite_bf16_tail_kernel(const uint16_t* __restrict__ p, int32_t* status) {
  if ((p[0] & 0x7f80u) == 0x7f80u) atomicOr(status, kStatusNonFinite);
}

cudaError_t launch_nonfinite_check(const void* p, int64_t n, bool f32, int32_t* status, cudaStream_t st) {
  if (!p || n <= 0) return cudaSuccess;
  const int64_t words = f32 ? n : n / 2;
  const int64_t blocks = grid_stride_blocks(words);
  if (blocks > 0)
    nonfinite_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint32_t*>(p), words, f32 ? 0 : 1, status);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && !f32 && (n & 1)) {
    nonfinite_bf16_tail_kernel<<<1, 1, 0, st>>>(static_cast<const uint16_t*>(p) + (n - 1), status);
    e = cudaGetLastError();
  }
  return e;
}

// pos[t] must be t - cu[s] for the sequence s holding token t.
__global__ void __launch_bounds__(256) position_check_kernel(const int32_t* __restrict__ cu, int32_t S,
                                                             int64_t T, const int32_t* __restrict__ pos,
                                                             int32_t* status) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  bool bad = false;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T; t += stride) {
    int32_t lo = 0, hi = S;
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    bad |= (int64_t)pos[t] != t - (int64_t)cu[lo];
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, kStatusBadCu);
}

cudaError_t launch_position_check(const int32_t* cu, int32_t num_seqs, int64_t T, const int32_t* pos,
                                  int32_t* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int64_t blocks = grid_stride_blocks(T);
  position_check_kernel<<<(unsigned)blocks, 256, 0, st>>>(cu, num_seqs, T, pos, status);
  return cudaGetLastError();
}

// seq[t] = the sequence holding token t: the largest s with cu[s] <= t (the
// same upper-bound search, so zero-length sequences hold no token).  The scan
// calls read it only where a sequence starts or ends, to find its state row.
// A malformed cu_seqlens (reported through the status word) can leave tokens
// past cu[S]; they are given the last sequence, so that every state row the
// kernels touch exists.
__global__ void __launch_bounds__(256) sequence_index_kernel(const int32_t* __restrict__ cu,
                                                             int32_t S, int64_t T,
                                                             int32_t* __restrict__ seq) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T; t += stride) {
    int32_t lo = 0, hi = S;
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    seq[t] = lo < S ? lo : S - 1;
  }
}

cudaError_t launch_sequence_index(const int32_t* cu, int32_t num_seqs, int64_t T, int32_t* seq,
                                  cudaStream_t st) {
  const int64_t blocks = grid_stride_blocks(T);
  if (blocks < 1) return cudaSuccess;
  sequence_index_kernel<<<(unsigned)blocks, 256, 0, st>>>(cu, num_seqs, T, seq);
  return cudaGetLastError();
}

// For every EMPTY sequence s (cu[s] == cu[s+1]), dst[s] = src[s] (rows of DN
// floats; zeros when src is NULL): the state, or its gradient, passes a
// sequence with no token unchanged.  One block per sequence.
__global__ void __launch_bounds__(256) empty_sequence_states_kernel(const int32_t* __restrict__ cu,
                                                                    int64_t DN,
                                                                    const float* __restrict__ src,
                                                                    float* __restrict__ dst) {
  const int64_t s = blockIdx.x;
  if (cu[s] != cu[s + 1]) return;
  for (int64_t i = threadIdx.x; i < DN; i += blockDim.x) dst[s * DN + i] = src ? src[s * DN + i] : 0.0f;
}

cudaError_t launch_empty_sequence_states(const int32_t* cu, int32_t num_seqs, int64_t DN,
                                         const float* src, float* dst, cudaStream_t st) {
  if (num_seqs <= 0 || !dst) return cudaSuccess;
  empty_sequence_states_kernel<<<(unsigned)num_seqs, 256, 0, st>>>(cu, DN, src, dst);
  return cudaGetLastError();
}

// out[m] = sum over p = 0..P-1 of in[p*ld + m], in a fixed order: rows are
// summed in order within groups of R consecutive rows, then the group sums in
// order.  One thread per (column, group), so the result is bitwise repeatable.
//
// Group pass: the sum of rows g*R .. g*R+R-1 replaces row g*R (the partial
// buffer is scratch owned by the caller).
__global__ void __launch_bounds__(256) sum_row_groups_kernel(float* __restrict__ in, int64_t P,
                                                             int64_t M, int64_t ld, int64_t R,
                                                             int64_t col_blocks) {
  const int64_t g = blockIdx.x / col_blocks;
  const int64_t m = (blockIdx.x - g * col_blocks) * blockDim.x + threadIdx.x;
  if (m >= M) return;
  const int64_t r0 = g * R, r1 = (r0 + R < P) ? r0 + R : P;
  float* p = in + m;
  float acc = 0.0f;
  int64_t r = r0;
  for (; r + 8 <= r1; r += 8) {  // 8 loads in flight, added in row order
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = __ldcs(p + (r + q) * ld);
#pragma unroll
    for (int q = 0; q < 8; ++q) acc += v[q];
  }
  for (; r + 4 <= r1; r += 4) {
    const float a0 = __ldcs(p + (r + 0) * ld), a1 = __ldcs(p + (r + 1) * ld);
    const float a2 = __ldcs(p + (r + 2) * ld), a3 = __ldcs(p + (r + 3) * ld);
    acc += a0; acc += a1; acc += a2; acc += a3;
  }
  for (; r < r1; ++r) acc += __ldcs(p + r * ld);
  p[r0 * ld] = acc;
}

// Final pass: out[m] = sum over p = 0..P-1 (in order) of in[p*ld + m]; with
// inner > 0 the columns are an (M / inner, inner) array written out
// transposed: out[(m % inner) * (M / inner) + m / inner].
__global__ void __launch_bounds__(256) sum_rows_kernel(const float* __restrict__ in, int64_t P,
                                                       int64_t M, int64_t ld, int64_t inner,
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
  if (inner > 0) {
    const int64_t q = m / inner;
    out[(m - q * inner) * (M / inner) + q] = acc;
  } else {
    out[m] = acc;
  }
}

cudaError_t launch_sum_rows(float* in, int64_t P, int64_t M, int64_t ld, float* out, cudaStream_t st,
                            int64_t inner) {
  if (M <= 0) return cudaSuccess;
  const int64_t col_blocks = (M + 255) / 256;
  constexpr int64_t kGroup = 32;
  if (P > 2 * kGroup) {
    // enough groups to fill the GPU, at most 2^31 - 1 blocks in all
    int64_t R = kGroup;
    while (((P + R - 1) / R) * col_blocks > 2147483647LL) R *= 2;
    const int64_t G = (P + R - 1) / R;
    sum_row_groups_kernel<<<(unsigned)(G * col_blocks), 256, 0, st>>>(in, P, M, ld, R, col_blocks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    P = G;
    ld *= R;
  }
  sum_rows_kernel<<<(unsigned)col_blocks, 256, 0, st>>>(in, P, M, ld, inner, out);
  return cudaGetLastError();
}

}  // namespace vssm
