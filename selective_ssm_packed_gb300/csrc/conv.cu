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
constexpr int kFwdRun = 4;        // tokens per thread, forward
constexpr int kBwdRun = 8;        // tokens per thread, backward

template <typename T, int V>
__device__ __forceinline__ void ldv(const T* p, float (&v)[V]);
template <typename T, int V>
__device__ __forceinline__ void stv(T* p, const float (&v)[V]);

// 16-byte loads / stores
template <>
__device__ __forceinline__ void ldv<float, 4>(const float* p, float (&v)[4]) {
  const float4 q = __ldg(reinterpret_cast<const float4*>(p));
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
template <>
__device__ __forceinline__ void stv<float, 4>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void ldv<__nv_bfloat16, 8>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = __bfloat1622float2(h[j]);
    v[2 * j] = f.x; v[2 * j + 1] = f.y;
  }
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
__device__ __forceinline__ void ldv<__nv_bfloat16, 4>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
  const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
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

// ------------------------------------------------------------------ forward
template <typename T, int W>
__global__ void __launch_bounds__(256) conv_fwd_kernel(ConvArgs a) {
  constexpr int V = 16 / sizeof(T);
  constexpr int R = kFwdRun;
  constexpr int E = R + W - 1;  // rows loaded: t0-(W-1) .. t0+R-1
  const int ncols = (a.D / V + 31) / 32;
  const int64_t row = blockIdx.x / ncols;
  const int d0 = ((int)(blockIdx.x - row * ncols) * 32 + threadIdx.x) * V;
  const int64_t t0 = (row * kRowsPerBlock + threadIdx.y) * R;
  if (d0 >= a.D || t0 >= a.T) return;
  const T* __restrict__ x = static_cast<const T*>(a.x);
  T* __restrict__ u = static_cast<T*>(a.out);
  const int64_t D = a.D;

  float xr[E][V];
  int p[R];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int64_t t = t0 - (W - 1) + i;
    if (t >= 0 && t < a.T) {
      ldv<T, V>(x + t * D + d0, xr[i]);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) xr[i][v] = 0.0f;
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) p[r] = (t0 + r < a.T) ? __ldg(a.pos + t0 + r) : 0;

  float w[W][V], b[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
#pragma unroll
    for (int k = 0; k < W; ++k) w[k][v] = __ldg(a.w + (int64_t)(d0 + v) * W + k);
    b[v] = a.bias ? __ldg(a.bias + d0 + v) : 0.0f;
  }

#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t t = t0 + r;
    if (t >= a.T) break;
    float o[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
      float pre = fmaf(w[W - 1][v], xr[r + W - 1][v], b[v]);
#pragma unroll
      for (int k = 1; k < W; ++k)
        if (p[r] >= k) pre = fmaf(w[W - 1 - k][v], xr[r + W - 1 - k][v], pre);
      o[v] = a.apply_silu ? siluf(pre) : pre;
    }
    stv<T, V>(u + t * D + d0, o);
  }
}

// ------------------------------------------------------------------ backward
// Each thread streams over tokens t' = t0 .. t0+R+W-2, keeping windows of x,
// of g = du * du/dpre and of pos, and emits dx[t'-(W-1)] once g[t'] is known.
template <typename T, int W>
__global__ void __launch_bounds__(256) conv_bwd_kernel(ConvArgs a) {
  constexpr int V = 4;
  constexpr int R = kBwdRun;
  const int ncols = (a.D / V + 31) / 32;
  const int64_t row = blockIdx.x / ncols;
  const int d0 = ((int)(blockIdx.x - row * ncols) * 32 + threadIdx.x) * V;
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
    float w[W][V], b[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
#pragma unroll
      for (int k = 0; k < W; ++k) w[k][v] = __ldg(a.w + (int64_t)(d0 + v) * W + k);
      b[v] = a.bias ? __ldg(a.bias + d0 + v) : 0.0f;
    }
    float xw[W][V];   // after the shift at step t': xw[k] = x[t' - k]
    float gw[W][V];   // after step t': gw[k] = g[t' - (W-1) + k]
    int pw[W];        // after step t': pw[k] = pos[t' - (W-1) + k]
#pragma unroll
    for (int k = 0; k < W; ++k) {
      pw[k] = 0;
#pragma unroll
      for (int v = 0; v < V; ++v) { xw[k][v] = 0.0f; gw[k][v] = 0.0f; }
    }
    // before the first step xw[k-1] holds x[t0 - k], so the shift lines it up
#pragma unroll
    for (int k = 1; k < W; ++k) {
      const int64_t t = t0 - k;
      if (t >= 0) ldv<T, V>(x + t * D + d0, xw[k - 1]);
    }
#pragma unroll
    for (int j = 0; j < R + W - 1; ++j) {
      const int64_t tp = t0 + j;
      const bool in = tp < a.T;
      float xc[V], dc[V];
      int p = 0;
      if (in) {
        ldv<T, V>(x + tp * D + d0, xc);
        ldv<T, V>(du + tp * D + d0, dc);
        p = __ldg(a.pos + tp);
      } else {
#pragma unroll
        for (int v = 0; v < V; ++v) { xc[v] = 0.0f; dc[v] = 0.0f; }
      }
      // shift the windows by one token
#pragma unroll
      for (int k = W - 1; k > 0; --k) {
#pragma unroll
        for (int v = 0; v < V; ++v) xw[k][v] = xw[k - 1][v];
      }
#pragma unroll
      for (int v = 0; v < V; ++v) xw[0][v] = xc[v];
#pragma unroll
      for (int k = 0; k < W - 1; ++k) {
        pw[k] = pw[k + 1];
#pragma unroll
        for (int v = 0; v < V; ++v) gw[k][v] = gw[k + 1][v];
      }
      pw[W - 1] = p;
      // g at t'
#pragma unroll
      for (int v = 0; v < V; ++v) {
        float g = 0.0f;
        if (in) {
          float pre = fmaf(w[W - 1][v], xw[0][v], b[v]);
#pragma unroll
          for (int k = 1; k < W; ++k)
            if (p >= k) pre = fmaf(w[W - 1 - k][v], xw[k][v], pre);
          g = a.apply_silu ? dc[v] * silu_grad(pre) : dc[v];
        }
        gw[W - 1][v] = g;
        if (j < R && in) {
          db[v] += g;
#pragma unroll
          for (int k = 0; k < W; ++k)
            if (p >= k) dw[W - 1 - k][v] = fmaf(g, xw[k][v], dw[W - 1 - k][v]);
        }
      }
      // dx at t = t' - (W-1), complete now that g[t .. t+W-1] is known
      if (j >= W - 1) {
        const int64_t t = tp - (W - 1);
        if (t < a.T) {
          float o[V];
#pragma unroll
          for (int v = 0; v < V; ++v) {
            float acc = 0.0f;
#pragma unroll
            for (int k = 0; k < W; ++k)
              if (t + k < a.T && pw[k] >= k) acc = fmaf(w[W - 1 - k][v], gw[k][v], acc);
            o[v] = acc;
          }
          stv<T, V>(dx + t * D + d0, o);
        }
      }
    }
  }

  // reduce dw / db over the 8 token rows of the block, write one partial row
  __shared__ float red[kRowsPerBlock][32][V * (W + 1)];
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
