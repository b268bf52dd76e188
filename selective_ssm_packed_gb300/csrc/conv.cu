// conv.cu -- packed depthwise causal conv1d (width W <= 4), forward and backward.
//
// Layout: thread block = 32 threads along channels x 8 along tokens; a 1-D grid
// where consecutive blocks cover consecutive channel columns of the same token
// rows, so the blocks running together read and write whole rows.  Each
// thread owns V consecutive channels (one 16-byte vector in the forward, an
// 8/16-byte vector in the backward) and a short run of R consecutive tokens,
// so every warp reads and writes whole contiguous row segments.  The
// sequence-boundary mask comes from position_indices: tap k (k tokens back)
// is used only if pos[t] >= k, and in the backward the tap that token t feeds
// k tokens later is used only if pos[t+k] >= k (the conv1d_pack early stop of
// the article "Shanghai AI Lab: packed variable-length Mamba training").
#include "common.cuh"
#include "kernels.h"

namespace vssm {

namespace {

constexpr int kRowsPerBlock = 8;  // threadIdx.y extent
constexpr int kFwdRun = 8;        // tokens per thread, forward
constexpr int kBwdRun = 8;        // tokens per thread, backward

template <typename T, int V>
__device__ __forceinline__ void stv(T* p, const float (&v)[V]);

// 16-byte loads / stores
template <>
__device__ __forceinline__ void stv<float, 4>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void stv<__nv_bfloat16, 8>(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 q;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
  for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
  *reinterpret_cast<uint4*>(p) = q;
}
// 8-byte bf16 loads / stores (backward, 4 channels per thread)
template <>
__device__ __forceinline__ void stv<__nv_bfloat16, 4>(__nv_bfloat16* p, const float (&v)[4]) {
  uint2 q;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
  h[0] = __floats2bfloat162_rn(v[0], v[1]);
  h[1] = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = q;
}

__device__ __forceinline__ float silu_grad(float x) {
  const float s = sigmoidf_fast(x);
  return s * fmaf(x, 1.0f - s, 1.0f);
}

// Raw (still packed) row segments: loaded in one vector access, widened later.
template <typename T, int V> struct RawRow;
template <> struct RawRow<float, 4> { uint4 r; };
template <> struct RawRow<__nv_bfloat16, 8> { uint4 r; };
template <> struct RawRow<__nv_bfloat16, 4> { uint2 r; };

template <typename T, int V>
__device__ __forceinline__ void ld_raw(const T* p, RawRow<T, V>& out) {
  if constexpr (sizeof(out.r) == 16) out.r = __ldg(reinterpret_cast<const uint4*>(p));
  else out.r = __ldg(reinterpret_cast<const uint2*>(p));
}
template <typename T, int V>
__device__ __forceinline__ void zero_raw(RawRow<T, V>& out) {
  if constexpr (sizeof(out.r) == 16) out.r = make_uint4(0, 0, 0, 0);
  else out.r = make_uint2(0, 0);
}
template <typename T, int V>
__device__ __forceinline__ void widen(const RawRow<T, V>& in, float (&v)[V]) {
  if constexpr (sizeof(T) == 4) {
    v[0] = __uint_as_float(in.r.x); v[1] = __uint_as_float(in.r.y);
    v[2] = __uint_as_float(in.r.z); v[3] = __uint_as_float(in.r.w);
  } else {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&in.r);
#pragma unroll
    for (int j = 0; j < V / 2; ++j) {
      const float2 f = __bfloat1622float2(h[j]);
      v[2 * j] = f.x; v[2 * j + 1] = f.y;
    }
  }
}

// Stages the block's conv weights ([tap][channel], channel-contiguous) and
// biases in shared memory with coalesced loads.
template <int W, int CH>
__device__ __forceinline__ void stage_weights(const ConvArgs& a, int c0, float (*wS)[CH], float* bS,
                                              int tid) {
  for (int i = tid; i < CH * W; i += 256) {
    const int c = i / W, k = i - c * W;
    wS[k][c] = (c0 + c < a.D) ? __ldg(a.w + (int64_t)c0 * W + i) : 0.0f;
  }
  for (int i = tid; i < CH; i += 256) bS[i] = (a.bias && c0 + i < a.D) ? __ldg(a.bias + c0 + i) : 0.0f;
}

// ------------------------------------------------------------------ forward
template <typename T, int W>
__global__ void __launch_bounds__(256, 2) conv_fwd_kernel(ConvArgs a) {
  constexpr int V = 16 / sizeof(T);
  constexpr int R = kFwdRun;
  constexpr int E = R + W - 1;  // rows loaded: t0-(W-1) .. t0+R-1
  constexpr int CH = 32 * V;    // channels per block
  __shared__ __align__(16) float wS[W][CH];
  __shared__ __align__(16) float bS[CH];
  const int ncols = (a.D / V + 31) / 32;
  const int64_t row = blockIdx.x / ncols;
  const int c0 = (int)(blockIdx.x - row * ncols) * CH;
  stage_weights<W, CH>(a, c0, wS, bS, threadIdx.y * 32 + threadIdx.x);
  __syncthreads();
  const int d0 = c0 + threadIdx.x * V;
  const int64_t t0 = (row * kRowsPerBlock + threadIdx.y) * R;
  if (d0 >= a.D || t0 >= a.T) return;
  const T* __restrict__ x = static_cast<const T*>(a.x);
  T* __restrict__ u = static_cast<T*>(a.out);
  const int64_t D = a.D;

  // every load of the thread is issued before any arithmetic
  RawRow<T, V> xr[E];
  int p[R];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int64_t t = t0 - (W - 1) + i;
    if (t >= 0 && t < a.T) ld_raw<T, V>(x + t * D + d0, xr[i]); else zero_raw<T, V>(xr[i]);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) p[r] = (t0 + r < a.T) ? __ldg(a.pos + t0 + r) : 0;

  float w[W][V], b[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
#pragma unroll
    for (int k = 0; k < W; ++k) w[k][v] = wS[k][threadIdx.x * V + v];
    b[v] = bS[threadIdx.x * V + v];
  }

#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t t = t0 + r;
    if (t >= a.T) break;
    float xs[W][V];
#pragma unroll
    for (int k = 0; k < W; ++k) widen<T, V>(xr[r + W - 1 - k], xs[k]);   // xs[k] = x[t - k]
    float o[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      float pre = fmaf(w[W - 1][v], xs[0][v], b[v]);
#pragma unroll
      for (int k = 1; k < W; ++k)
        if (p[r] >= k) pre = fmaf(w[W - 1 - k][v], xs[k][v], pre);
      o[v] = a.apply_silu ? siluf(pre) : pre;
    }
    stv<T, V>(u + t * D + d0, o);
  }
}

// ------------------------------------------------------------------ backward
// Each thread loads all of its rows up front (x for t0-(W-1) .. t0+R+W-2, du
// and pos for t0 .. t0+R+W-2), then streams over t' = t0 .. t0+R+W-2 keeping
// windows of g = du * du/dpre and of pos, and emits dx[t'-(W-1)] once g[t'] is
// known.
template <typename T, int W>
__global__ void __launch_bounds__(256, 2) conv_bwd_kernel(ConvArgs a) {
  constexpr int V = 4;
  constexpr int R = kBwdRun;
  constexpr int CH = 32 * V;
  constexpr int EG = R + W - 1;        // tokens t0 .. t0+R+W-2 (g, du, pos)
  constexpr int EX = EG + W - 1;       // x rows t0-(W-1) .. t0+R+W-2
  __shared__ __align__(16) float wS[W][CH];
  __shared__ __align__(16) float bS[CH];
  __shared__ float red[kRowsPerBlock][32][V * (W + 1)];
  const int ncols = (a.D / V + 31) / 32;
  const int64_t row = blockIdx.x / ncols;
  const int c0 = (int)(blockIdx.x - row * ncols) * CH;
  stage_weights<W, CH>(a, c0, wS, bS, threadIdx.y * 32 + threadIdx.x);
  __syncthreads();
  const int d0 = c0 + threadIdx.x * V;
  const int64_t t0 = (row * kRowsPerBlock + threadIdx.y) * R;
  const bool active = d0 < a.D && t0 < a.T;
  const T* __restrict__ x = static_cast<const T*>(a.x);
  const T* __restrict__ du = static_cast<const T*>(a.du);
  T* __restrict__ dx = static_cast<T*>(a.out);
  const int64_t D = a.D;

  float dw[W][V], db[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    db[v] = 0.0f;
#pragma unroll
    for (int k = 0; k < W; ++k) dw[k][v] = 0.0f;
  }

  if (active) {
    RawRow<T, V> xr[EX], dr[EG];
    int p[EG];
#pragma unroll
    for (int i = 0; i < EX; ++i) {
      const int64_t t = t0 - (W - 1) + i;
      if (t >= 0 && t < a.T) ld_raw<T, V>(x + t * D + d0, xr[i]); else zero_raw<T, V>(xr[i]);
    }
#pragma unroll
    for (int j = 0; j < EG; ++j) {
      const int64_t t = t0 + j;
      if (t < a.T) {
        ld_raw<T, V>(du + t * D + d0, dr[j]);
        p[j] = __ldg(a.pos + t);
      } else {
        zero_raw<T, V>(dr[j]);
        p[j] = 0;
      }
    }
    float w[W][V], b[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
#pragma unroll
      for (int k = 0; k < W; ++k) w[k][v] = wS[k][threadIdx.x * V + v];
      b[v] = bS[threadIdx.x * V + v];
    }
    float gw[W][V];   // after step j: gw[k] = g[t0 + j - (W-1) + k]
#pragma unroll
    for (int k = 0; k < W; ++k)
#pragma unroll
      for (int v = 0; v < V; ++v) gw[k][v] = 0.0f;
#pragma unroll
    for (int j = 0; j < EG; ++j) {
      const int64_t tp = t0 + j;
      float xs[W][V];   // xs[k] = x[t' - k]
#pragma unroll
      for (int k = 0; k < W; ++k) widen<T, V>(xr[j + W - 1 - k], xs[k]);
      float dc[V];
      widen<T, V>(dr[j], dc);
#pragma unroll
      for (int k = 0; k < W - 1; ++k)
#pragma unroll
        for (int v = 0; v < V; ++v) gw[k][v] = gw[k + 1][v];
#pragma unroll
      for (int v = 0; v < V; ++v) {
        float g = 0.0f;
        if (tp < a.T) {
          float pre = fmaf(w[W - 1][v], xs[0][v], b[v]);
#pragma unroll
          for (int k = 1; k < W; ++k)
            if (p[j] >= k) pre = fmaf(w[W - 1 - k][v], xs[k][v], pre);
          g = a.apply_silu ? dc[v] * silu_grad(pre) : dc[v];
        }
        gw[W - 1][v] = g;
        if (j < R && tp < a.T) {
          db[v] += g;
#pragma unroll
          for (int k = 0; k < W; ++k)
            if (p[j] >= k) dw[W - 1 - k][v] = fmaf(g, xs[k][v], dw[W - 1 - k][v]);
        }
      }
      // dx at t = t' - (W-1), complete now that g[t .. t+W-1] is known
      if (j >= W - 1) {
        const int64_t t = tp - (W - 1);
        const int r = j - (W - 1);
        if (t < a.T) {
          float o[V];
#pragma unroll
          for (int v = 0; v < V; ++v) {
            float acc = 0.0f;
#pragma unroll
            for (int k = 0; k < W; ++k)
              if (t + k < a.T && p[r + k] >= k) acc = fmaf(w[W - 1 - k][v], gw[k][v], acc);
            o[v] = acc;
          }
          stv<T, V>(dx + t * D + d0, o);
        }
      }
    }
  }

  // reduce dw / db over the 8 token rows of the block, write one partial row
#pragma unroll
  for (int v = 0; v < V; ++v) {
#pragma unroll
    for (int k = 0; k < W; ++k) red[threadIdx.y][threadIdx.x][v * (W + 1) + k] = dw[k][v];
    red[threadIdx.y][threadIdx.x][v * (W + 1) + W] = db[v];
  }
  __syncthreads();
  if (threadIdx.y == 0 && d0 < a.D) {
    float* part = a.partial + row * (D * (W + 1));
#pragma unroll
    for (int v = 0; v < V; ++v) {
      float s[W + 1];
#pragma unroll
      for (int k = 0; k <= W; ++k) s[k] = 0.0f;
      for (int r = 0; r < kRowsPerBlock; ++r)
#pragma unroll
        for (int k = 0; k <= W; ++k) s[k] += red[r][threadIdx.x][v * (W + 1) + k];
      // partial row layout: dweight (D, W) first, then dbias (D)
#pragma unroll
      for (int k = 0; k < W; ++k) part[(int64_t)(d0 + v) * W + k] = s[k];
      part[D * W + d0 + v] = s[W];
    }
  }
}

template <typename T, int W>
cudaError_t fwd_w(const ConvArgs& a, cudaStream_t st) {
  constexpr int V = 16 / sizeof(T);
  const int64_t cols = (a.D / V + 31) / 32;
  const int64_t rows = (a.T + kRowsPerBlock * kFwdRun - 1) / (kRowsPerBlock * kFwdRun);
  if (rows * cols > 2147483647LL) return cudaErrorInvalidConfiguration;
  conv_fwd_kernel<T, W><<<(unsigned)(rows * cols), dim3(32, kRowsPerBlock), 0, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int W>
cudaError_t bwd_w(const ConvArgs& a, cudaStream_t st) {
  const int64_t cols = (a.D / 4 + 31) / 32;
  const int64_t rows = conv_bwd_partial_rows(a.T);
  if (rows * cols > 2147483647LL) return cudaErrorInvalidConfiguration;
  conv_bwd_kernel<T, W><<<(unsigned)(rows * cols), dim3(32, kRowsPerBlock), 0, st>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t fwd_t(const ConvArgs& a, cudaStream_t st) {
  switch (a.W) {
    case 1: return fwd_w<T, 1>(a, st);
    case 2: return fwd_w<T, 2>(a, st);
    case 3: return fwd_w<T, 3>(a, st);
    case 4: return fwd_w<T, 4>(a, st);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t bwd_t(const ConvArgs& a, cudaStream_t st) {
  switch (a.W) {
    case 1: return bwd_w<T, 1>(a, st);
    case 2: return bwd_w<T, 2>(a, st);
    case 3: return bwd_w<T, 3>(a, st);
    case 4: return bwd_w<T, 4>(a, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int64_t conv_bwd_partial_rows(int64_t T) {
  const int64_t per = kRowsPerBlock * kBwdRun;
  const int64_t r = (T + per - 1) / per;
  return r > 0 ? r : 1;
}

cudaError_t launch_conv1d_fwd(const ConvArgs& a, IO io, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  return io == IO::F32 ? fwd_t<float>(a, st) : fwd_t<__nv_bfloat16>(a, st);
}

cudaError_t launch_conv1d_bwd(const ConvArgs& a, IO io, float* dweight, float* dbias,
                              cudaStream_t st) {
  const int64_t P = conv_bwd_partial_rows(a.T);
  if (a.T > 0) {
    cudaError_t e = io == IO::F32 ? bwd_t<float>(a, st) : bwd_t<__nv_bfloat16>(a, st);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = cudaMemsetAsync(a.partial, 0, sizeof(float) * (size_t)a.D * (a.W + 1), st);
    if (e != cudaSuccess) return e;
  }
  const int64_t ld = (int64_t)a.D * (a.W + 1);
  cudaError_t e = launch_sum_rows(a.partial, a.T > 0 ? P : 1, (int64_t)a.D * a.W, ld, dweight, st);
  if (e != cudaSuccess) return e;
  if (dbias) e = launch_sum_rows(a.partial + (int64_t)a.D * a.W, a.T > 0 ? P : 1, a.D, ld, dbias, st);
  return e;
}

}  // namespace vssm
