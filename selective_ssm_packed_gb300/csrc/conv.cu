// conv.cu -- packed depthwise causal conv1d (width W <= 4), forward and backward.
//
// One CTA per tile of 192 tokens x 128 channels.  The x rows of the tile (plus
// the W-1 rows before it, and for the backward the W-1 after it) and the du
// rows come into shared memory by 2-D tensor copies, so every row is read from
// HBM about once; rows before the first token or past the last are zero-filled
// by the copy.  Warp w owns 24 consecutive tokens of the tile, lane l owns 4
// consecutive channels, so stores are whole 256- or 512-byte row segments per
// warp.  The sequence-boundary mask comes from position_indices: tap k (k
// tokens back) is used only if pos[t] >= k, and in the backward the tap that
// token t feeds k tokens later is used only if pos[t+k] >= k (the conv1d_pack
// early stop of the article "Shanghai AI Lab: packed variable-length Mamba
// training").
#include "common.cuh"
#include "kernels.h"

namespace vssm {

namespace {


// 8-byte bf16 store of 4 channels
__device__ __forceinline__ void st_bf16x4(__nv_bfloat16* p, const float (&v)[4]) {
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

// ------------------------------------------------------------------ tiled kernels
// One CTA per tile of CT tokens x kCC = 128 channels.  The x rows the tile
// needs (its tokens plus the W-1 before them, and for the backward the W-1
// after them) and the du rows arrive by 2-D tensor copies on one mbarrier;
// rows before the first token or past the last come back as zeros.  Warp w
// owns tokens (CT/8)w .. (CT/8)(w+1)-1 of the tile, lane l owns channels
// 4l .. 4l+3, and every row a thread touches after the copies is read from
// shared memory.  The backward recomputes g for the W-1 tokens after a warp's
// own, so the longer the warp's run of tokens, the smaller that share (3 of
// 27 at 24 tokens).  The forward's tile holds only its x rows (bf16: 17 KB
// at 64 tokens, 50 KB at 192); tiles of 192 tokens measured faster than 128
// and 64 for both directions.
// (a tensor-copy box is at most 256 rows: 192 + 2(W-1) fits)
constexpr int kCTF = 192;  // tokens per forward tile
constexpr int kCTB = 192;  // tokens per backward tile
constexpr int kCC = 128;   // channels per tile

template <typename T>
__device__ __forceinline__ void lds4(const T* p, float (&v)[4]) {
  if constexpr (sizeof(T) == 4) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  } else {
    const uint2 q = *reinterpret_cast<const uint2*>(p);
    const float2 a0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
    const float2 a1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
    v[0] = a0.x; v[1] = a0.y; v[2] = a1.x; v[3] = a1.y;
  }
}

template <typename T>
__device__ __forceinline__ void stg4(T* p, const float (&v)[4]) {
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
    st_bf16x4(p, v);
  }
}

// kBwd: the backward's tile (x rows on both sides, du rows, and room for the
// per-warp dweight / dbias partials); the forward's holds its x rows only.
template <typename T, int W, int CT, bool kBwd>
struct ConvTileSmem {
  static constexpr int XR = CT + (kBwd ? 2 : 1) * (W - 1);  // x rows from t0-(W-1)
  static constexpr int GR = kBwd ? CT + W - 1 : 0;          // du rows t0 .. t0+CT+W-2
  static constexpr size_t kIO = sizeof(T) * (size_t)(XR + GR) * kCC;
  static constexpr size_t kRed = kBwd ? sizeof(float) * 8 * kCC * (W + 1) : 0;
  // x rows, then du rows (both 256-byte multiples: kCC * sizeof(T)); after
  // the backward's arithmetic, the per-warp dweight / dbias partials
  alignas(128) unsigned char io[kIO > kRed ? kIO : kRed];
  __device__ T* x() { return reinterpret_cast<T*>(io); }
  __device__ T* du() { return reinterpret_cast<T*>(io + sizeof(T) * (size_t)XR * kCC); }
  __device__ float* red() { return reinterpret_cast<float*>(io); }
  alignas(16) float w[W][kCC];
  alignas(16) float b[kCC];
  int pos[CT + W - 1];
  alignas(8) uint64_t bar;
};

// Forward: u[t] = SiLU(bias + sum_k w[W-1-k] x[t-k] [pos[t] >= k]) for the tile.
// kTail: the call passes tail values (x_init) for the first W-1 tokens of a
// sequence; without them the kernel carries no code for them.
template <typename T, int W, bool kTail>
__global__ void __launch_bounds__(256, 4) conv_fwd_tile_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                            ConvArgs a) {
  using SM = ConvTileSmem<T, W, kCTF, false>;
  constexpr int kTokPerWarp = kCTF / 8;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  const int ncols = (a.D + kCC - 1) / kCC;
  const int64_t row = blockIdx.x / ncols;
  const int c0 = (int)(blockIdx.x - row * ncols) * kCC;
  const int64_t t0 = row * kCTF;
  const int bx = a.D < kCC ? a.D : kCC;  // row pitch of the staged tile
  constexpr int FR = SM::XR;             // x rows the forward needs
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&sm.bar, (uint32_t)bx * FR * sizeof(T));
    tma_load_2d(sm.x(), &tm_x, c0, (int)(t0 - (W - 1)), &sm.bar);
  }
  for (int i = tid; i < kCC * W; i += 256) {
    const int c = i / W, k = i - c * W;
    sm.w[k][c] = (c0 + c < a.D) ? __ldg(a.w + (int64_t)c0 * W + i) : 0.0f;
  }
  for (int i = tid; i < kCC; i += 256) sm.b[i] = (a.bias && c0 + i < a.D) ? __ldg(a.bias + c0 + i) : 0.0f;
  for (int i = tid; i < kCTF; i += 256) sm.pos[i] = (t0 + i < a.T) ? __ldg(a.pos + t0 + i) : 0;
  __syncthreads();
  const int c = 4 * lane;
  const bool active = c < bx && c0 + c < a.D;
  float w[W][4], bb[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
#pragma unroll
    for (int k = 0; k < W; ++k) w[k][v] = sm.w[k][c + v];
    bb[v] = sm.b[c + v];
  }
  // the tile copy: a wait that runs out (or the test knob's CTA) is reported in
  // the status word; the CTA then gives the copy one more, long limit to land
  // before it leaves, so that nothing it requested still writes into its
  // shared memory afterwards
  if (!__syncthreads_and(mbar_wait(&sm.bar, 0, a.wait_ns) && (long long)blockIdx.x != a.force_timeout_cta)) {
    if (tid == 0 && a.status) atomicOr(a.status, kStatusTmaTimeout);
    mbar_wait(&sm.bar, 0, kCopyDrainNs);
    return;
  }
  if (!active) return;
  T* __restrict__ u = static_cast<T*>(a.out);
  float xw[W][4];  // xw[k] = x[t - (W-1) + k]
#pragma unroll
  for (int k = 0; k < W - 1; ++k) lds4<T>(sm.x() + (kTokPerWarp * wp + k) * bx + c, xw[k]);
#pragma unroll
  for (int j = 0; j < kTokPerWarp; ++j) {
    const int tl = kTokPerWarp * wp + j;
    lds4<T>(sm.x() + (tl + W - 1) * bx + c, xw[W - 1]);
    const int p = sm.pos[tl];
    // a tap reaching before the sequence start reads the sequence's tail value
    const float* trow = nullptr;
    if constexpr (kTail) {
      if (p < W - 1 && t0 + tl < a.T &&
          VSSM_CHECKED((unsigned)a.seq[t0 + tl] < (unsigned)a.num_seqs, a.status))
        trow = a.x_init + ((int64_t)a.seq[t0 + tl] * a.D + c0 + c) * (W - 1);
    }
    float o[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      float pre = fmaf(w[W - 1][v], xw[W - 1][v], bb[v]);
#pragma unroll
      for (int k = 1; k < W; ++k) {
        if (p >= k) pre = fmaf(w[W - 1 - k][v], xw[W - 1 - k][v], pre);
        else if (kTail && trow) pre = fmaf(w[W - 1 - k][v], __ldg(trow + v * (W - 1) + W - 1 + p - k), pre);
      }
      o[v] = a.apply_silu ? siluf(pre) : pre;
    }
    if (t0 + tl < a.T) stg4<T>(u + (t0 + tl) * (int64_t)a.D + c0 + c, o);
#pragma unroll
    for (int k = 0; k < W - 1; ++k)
#pragma unroll
      for (int v = 0; v < 4; ++v) xw[k][v] = xw[k + 1][v];
  }
}

// Backward: g[t] = du[t] SiLU'(pre[t]) for the tile's tokens and the W-1 after
// them; dx[t] = sum_k w[W-1-k] g[t+k] [t+k < T and pos[t+k] >= k]; dweight and
// dbias partials of the tile's own tokens, summed over the 8 warps in a fixed
// order into one partial row per tile row.  A warp's lanes share their token,
// so every mask is warp-uniform; the 4 channels of a lane run as 2 packed pairs.
// kTail: the call passes tail values (x_init) and/or gradients reaching
// sequences' last W-1 inputs (dx_last); without them the kernel carries no
// code for them.
template <typename T, int W, bool kTail>
__global__ void __launch_bounds__(256, 2) conv_bwd_tile_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                               const __grid_constant__ CUtensorMap tm_du,
                                                               ConvArgs a) {
  using SM = ConvTileSmem<T, W, kCTB, true>;
  constexpr int kTokPerWarp = kCTB / 8;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  const int ncols = (a.D + kCC - 1) / kCC;
  const int64_t row = blockIdx.x / ncols;
  const int c0 = (int)(blockIdx.x - row * ncols) * kCC;
  const int64_t t0 = row * kCTB;
  const int bx = a.D < kCC ? a.D : kCC;
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&sm.bar, (uint32_t)bx * (SM::XR + SM::GR) * sizeof(T));
    tma_load_2d(sm.x(), &tm_x, c0, (int)(t0 - (W - 1)), &sm.bar);
    tma_load_2d(sm.du(), &tm_du, c0, (int)t0, &sm.bar);
  }
  for (int i = tid; i < kCC * W; i += 256) {
    const int c = i / W, k = i - c * W;
    sm.w[k][c] = (c0 + c < a.D) ? __ldg(a.w + (int64_t)c0 * W + i) : 0.0f;
  }
  for (int i = tid; i < kCC; i += 256) sm.b[i] = (a.bias && c0 + i < a.D) ? __ldg(a.bias + c0 + i) : 0.0f;
  // pos of tokens past T is 0, so every tap from there is masked off
  for (int i = tid; i < SM::GR; i += 256) sm.pos[i] = (t0 + i < a.T) ? __ldg(a.pos + t0 + i) : 0;
  __syncthreads();
  const int c = 4 * lane;
  const bool active = c < bx && c0 + c < a.D;
  float2 w[W][2], bb[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int k = 0; k < W; ++k) w[k][h] = make_float2(sm.w[k][c + 2 * h], sm.w[k][c + 2 * h + 1]);
    bb[h] = make_float2(sm.b[c + 2 * h], sm.b[c + 2 * h + 1]);
  }
  // the tile copies: a wait that runs out (or the test knob's CTA) is reported
  // in the status word, and the CTA gives the copies one more, long limit to
  // land; it still reaches the barriers below, with zero contributions
  const bool got =
      __syncthreads_and(mbar_wait(&sm.bar, 0, a.wait_ns) && (long long)blockIdx.x != a.force_timeout_cta);
  if (!got) {
    if (tid == 0 && a.status) atomicOr(a.status, kStatusTmaTimeout);
    mbar_wait(&sm.bar, 0, kCopyDrainNs);
  }
  float2 dw[W][2], db[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    db[h] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < W; ++k) dw[k][h] = make_float2(0.0f, 0.0f);
  }
  if (got && active) {
    T* __restrict__ dx = static_cast<T*>(a.out);
    const int tb = kTokPerWarp * wp;
    float2 xw[W][2];  // xw[k] = x[t - (W-1) + k] for the g token t
    float2 gw[W][2];  // gw[k] = g[t - (W-1) + k]
    int pw[W];        // pw[k] = pos[t - (W-1) + k] (tile-relative tokens >= tb only)
#pragma unroll
    for (int k = 0; k < W - 1; ++k) {
      float v[4];
      lds4<T>(sm.x() + (tb + k) * bx + c, v);
      xw[k][0] = make_float2(v[0], v[1]);
      xw[k][1] = make_float2(v[2], v[3]);
      gw[k][0] = gw[k][1] = make_float2(0.0f, 0.0f);
      pw[k] = 0;
    }
#pragma unroll
    for (int j = 0; j < kTokPerWarp + W - 1; ++j) {
      const int tl = tb + j;  // g token (tile-relative); its x row is tl + W - 1
      {
        float v[4];
        lds4<T>(sm.x() + (tl + W - 1) * bx + c, v);
        xw[W - 1][0] = make_float2(v[0], v[1]);
        xw[W - 1][1] = make_float2(v[2], v[3]);
      }
      float dv[4];
      lds4<T>(sm.du() + tl * bx + c, dv);
      const int p = sm.pos[tl];
      pw[W - 1] = p;
      // taps reaching before the sequence start read the sequence's tail values
      const float* trow = nullptr;
      if constexpr (kTail) {
        if (a.x_init && p < W - 1 && t0 + tl < a.T &&
            VSSM_CHECKED((unsigned)a.seq[t0 + tl] < (unsigned)a.num_seqs, a.status))
          trow = a.x_init + ((int64_t)a.seq[t0 + tl] * a.D + c0 + c) * (W - 1);
      }
      auto tail2 = [&](int h, int k) {  // the tail pair for tap k (k > p) of channels c+2h, c+2h+1
        return make_float2(__ldg(trow + (2 * h) * (W - 1) + W - 1 + p - k),
                           __ldg(trow + (2 * h + 1) * (W - 1) + W - 1 + p - k));
      };
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float2 pre = fma2(w[W - 1][h], xw[W - 1][h], bb[h]);
#pragma unroll
        for (int k = 1; k < W; ++k) {
          if (p >= k) pre = fma2(w[W - 1 - k][h], xw[W - 1 - k][h], pre);
          else if (kTail && trow) pre = fma2(w[W - 1 - k][h], tail2(h, k), pre);
        }
        // rows past T are zero-filled, so g = 0 there
        const float2 dv2 = make_float2(dv[2 * h], dv[2 * h + 1]);
        const float2 g = a.apply_silu ? mul2(dv2, make_float2(silu_grad(pre.x), silu_grad(pre.y))) : dv2;
        gw[W - 1][h] = g;
        if (j < kTokPerWarp) {
          db[h] = __fadd2_rn(db[h], g);
#pragma unroll
          for (int k = 0; k < W; ++k) {
            if (p >= k) dw[W - 1 - k][h] = fma2(g, xw[W - 1 - k][h], dw[W - 1 - k][h]);
            else if (kTail && trow) dw[W - 1 - k][h] = fma2(g, tail2(h, k), dw[W - 1 - k][h]);
          }
        }
      }
      if (j >= W - 1) {  // dx of token tl - (W-1), which now has g[t .. t+W-1]
        const int to = tl - (W - 1);
        const int64_t t = t0 + to;
        if (t < a.T) {
          float2 acc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
          for (int k = 0; k < W; ++k)
            if (pw[k] >= k)
#pragma unroll
              for (int h = 0; h < 2; ++h) acc[h] = fma2(w[W - 1 - k][h], gw[k][h], acc[h]);
          if constexpr (kTail) {
            // token t is W-1-ke from its sequence's end when token t+ke is the next
            // start (or past T, where pos is 0): the gradient reaching the
            // sequence's last W-1 inputs from outside adds to its own
            if (a.dx_last) {
              int ke = 0;
#pragma unroll
              for (int k = W - 1; k >= 1; --k)
                if (pw[k] == 0) ke = k;
              if (ke && VSSM_CHECKED((unsigned)a.seq[t] < (unsigned)a.num_seqs, a.status)) {
                const float* drow = a.dx_last + ((int64_t)a.seq[t] * a.D + c0 + c) * (W - 1) + W - 1 - ke;
                acc[0] = __fadd2_rn(acc[0], make_float2(__ldg(drow), __ldg(drow + (W - 1))));
                acc[1] = __fadd2_rn(acc[1], make_float2(__ldg(drow + 2 * (W - 1)), __ldg(drow + 3 * (W - 1))));
              }
            }
          }
          const float o[4] = {acc[0].x, acc[0].y, acc[1].x, acc[1].y};
          stg4<T>(dx + t * (int64_t)a.D + c0 + c, o);
        }
      }
#pragma unroll
      for (int k = 0; k < W - 1; ++k) {
        pw[k] = pw[k + 1];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          xw[k][h] = xw[k + 1][h];
          gw[k][h] = gw[k + 1][h];
        }
      }
    }
  }
  // dweight / dbias: sum the 8 warps in order (the input tiles are free now)
  __syncthreads();
  float* red = sm.red();  // [8][kCC][W + 1]
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const int h = v >> 1;
#pragma unroll
    for (int k = 0; k < W; ++k) red[(wp * kCC + c + v) * (W + 1) + k] = (v & 1) ? dw[k][h].y : dw[k][h].x;
    red[(wp * kCC + c + v) * (W + 1) + W] = (v & 1) ? db[h].y : db[h].x;
  }
  __syncthreads();
  float* part = a.partial + row * ((int64_t)a.D * (W + 1));
  for (int i = tid; i < kCC * (W + 1); i += 256) {
    const int cc = i / (W + 1), k = i - cc * (W + 1);
    if (cc >= bx || c0 + cc >= a.D) continue;
    float acc = 0.0f;
#pragma unroll
    for (int r = 0; r < 8; ++r) acc += red[(r * kCC + cc) * (W + 1) + k];
    // partial row layout: dweight (D, W) first, then dbias (D)
    if (k < W) part[(int64_t)(c0 + cc) * W + k] = acc;
    else part[(int64_t)a.D * W + c0 + cc] = acc;
  }
}

template <typename T, int W, bool kTail>
cudaError_t fwd_tile_k(const ConvArgs& a, const CUtensorMap& tm_x, cudaStream_t st) {
  const size_t smem = sizeof(ConvTileSmem<T, W, kCTF, false>);
  cudaError_t e = cudaFuncSetAttribute(conv_fwd_tile_kernel<T, W, kTail>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t cols = (a.D + kCC - 1) / kCC;
  const int64_t rows = (a.T + kCTF - 1) / kCTF;
  if (rows * cols > 2147483647LL) return cudaErrorInvalidConfiguration;
  conv_fwd_tile_kernel<T, W, kTail><<<(unsigned)(rows * cols), 256, smem, st>>>(tm_x, a);
  return cudaGetLastError();
}

template <typename T, int W>
cudaError_t fwd_tile_w(const ConvArgs& a, const CUtensorMap& tm_x, cudaStream_t st) {
  return a.x_init ? fwd_tile_k<T, W, true>(a, tm_x, st) : fwd_tile_k<T, W, false>(a, tm_x, st);
}

template <typename T, int W, bool kTail>
cudaError_t bwd_tile_k(const ConvArgs& a, const CUtensorMap& tm_x, const CUtensorMap& tm_du,
                       cudaStream_t st) {
  const size_t smem = sizeof(ConvTileSmem<T, W, kCTB, true>);
  cudaError_t e = cudaFuncSetAttribute(conv_bwd_tile_kernel<T, W, kTail>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t cols = (a.D + kCC - 1) / kCC;
  const int64_t rows = (a.T + kCTB - 1) / kCTB;
  if (rows * cols > 2147483647LL) return cudaErrorInvalidConfiguration;
  conv_bwd_tile_kernel<T, W, kTail><<<(unsigned)(rows * cols), 256, smem, st>>>(tm_x, tm_du, a);
  return cudaGetLastError();
}

template <typename T, int W>
cudaError_t bwd_tile_w(const ConvArgs& a, const CUtensorMap& tm_x, const CUtensorMap& tm_du,
                       cudaStream_t st) {
  return (a.x_init || a.dx_last) ? bwd_tile_k<T, W, true>(a, tm_x, tm_du, st)
                                 : bwd_tile_k<T, W, false>(a, tm_x, tm_du, st);
}

template <typename T>
cudaError_t fwd_t(const ConvArgs& a, const CUtensorMap& tm_x, cudaStream_t st) {
  switch (a.W) {
    case 1: return fwd_tile_w<T, 1>(a, tm_x, st);
    case 2: return fwd_tile_w<T, 2>(a, tm_x, st);
    case 3: return fwd_tile_w<T, 3>(a, tm_x, st);
    case 4: return fwd_tile_w<T, 4>(a, tm_x, st);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t bwd_t(const ConvArgs& a, const CUtensorMap& tm_x, const CUtensorMap& tm_du, cudaStream_t st) {
  switch (a.W) {
    case 1: return bwd_tile_w<T, 1>(a, tm_x, tm_du, st);
    case 2: return bwd_tile_w<T, 2>(a, tm_x, tm_du, st);
    case 3: return bwd_tile_w<T, 3>(a, tm_x, tm_du, st);
    case 4: return bwd_tile_w<T, 4>(a, tm_x, tm_du, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

// Conv tails of cut sequences, one block per sequence s (tokens [cu[s],
// cu[s+1]), length L), threads over channels.  With xe the sequence's inputs
// preceded by its tail values (x_init, or zeros):
//   forward:  x_last[s][d][j] = xe[L - (W-1) + j], the tail the sequence's
//             next part starts from;
//   backward: dx_init[s][d][j] = the gradient reaching xe[j - (W-1)]: the
//             taps of the first W-1 tokens that read it (their g recomputed
//             from x, x_init, the weights and du) plus, for a sequence shorter
//             than W-1, the part of dx_last that lands there.
// The tile kernels handle everything that touches the real tokens.
template <typename T>
__global__ void __launch_bounds__(256) conv_tail_kernel(ConvArgs a, int bwd) {
  const int s = blockIdx.x;
  const int W = a.W;
  const int64_t start = a.cu[s], L = (int64_t)a.cu[s + 1] - start;
  const T* x = static_cast<const T*>(a.x);
  auto xe = [&](int64_t q, int d) {  // q = position in the sequence, from -(W-1)
    if (q >= 0) return to_f(x[(start + q) * a.D + d]);
    return a.x_init ? a.x_init[((int64_t)s * a.D + d) * (W - 1) + (W - 1) + q] : 0.0f;
  };
  for (int d = threadIdx.x; d < a.D; d += blockDim.x) {
    const int64_t row = ((int64_t)s * a.D + d) * (W - 1);
    if (!bwd) {
      for (int j = 0; j < W - 1; ++j) a.x_last[row + j] = xe(L - (W - 1) + j, d);
      continue;
    }
    float acc[3] = {0.0f, 0.0f, 0.0f};  // dxe[q] for q = -(W-1) .. -1, W <= 4
    const T* du = static_cast<const T*>(a.du);
    for (int64_t p = 0; p < L && p < W - 1; ++p) {
      float pre = a.bias ? a.bias[d] : 0.0f;
      for (int k = 0; k < W; ++k) pre = fmaf(a.w[(int64_t)d * W + (W - 1 - k)], xe(p - k, d), pre);
      const float gu = to_f(du[(start + p) * a.D + d]);
      const float g = a.apply_silu ? gu * silu_grad(pre) : gu;
      for (int k = p + 1; k < W; ++k)  // taps reaching q = p - k < 0
        acc[W - 1 + p - k] = fmaf(a.w[(int64_t)d * W + (W - 1 - k)], g, acc[W - 1 + p - k]);
    }
    if (a.dx_last)
      for (int j = 0; j < W - 1; ++j) {  // x_last[j] was read from xe[L - (W-1) + j]
        const int64_t q = L - (W - 1) + j;
        if (q < 0) acc[W - 1 + q] += a.dx_last[row + j];
      }
    for (int j = 0; j < W - 1; ++j) a.dx_init[row + j] = acc[j];
  }
}

cudaError_t launch_conv_tails(const ConvArgs& a, IO io, bool bwd, cudaStream_t st) {
  if ((bwd ? (void*)a.dx_init : (void*)a.x_last) == nullptr || a.num_seqs <= 0 || a.W < 2) return cudaSuccess;
  if (io == IO::F32) conv_tail_kernel<float><<<(unsigned)a.num_seqs, 256, 0, st>>>(a, bwd ? 1 : 0);
  else conv_tail_kernel<__nv_bfloat16><<<(unsigned)a.num_seqs, 256, 0, st>>>(a, bwd ? 1 : 0);
  return cudaGetLastError();
}

int64_t conv_bwd_partial_rows(int64_t T) {
  const int64_t per = kCTB;
  const int64_t r = (T + per - 1) / per;
  return r > 0 ? r : 1;
}

int conv_tile_rows(int W, bool bwd, bool x) {
  return x ? (bwd ? kCTB + 2 * (W - 1) : kCTF + W - 1) : kCTB + W - 1;
}
int conv_tile_cols() { return kCC; }

cudaError_t launch_conv1d_fwd(const ConvArgs& a, IO io, const CUtensorMap& tm_x, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  return io == IO::F32 ? fwd_t<float>(a, tm_x, st) : fwd_t<__nv_bfloat16>(a, tm_x, st);
}

cudaError_t launch_conv1d_bwd(const ConvArgs& a, IO io, const CUtensorMap& tm_x, const CUtensorMap& tm_du,
                              float* dweight, float* dbias, cudaStream_t st) {
  const int64_t P = conv_bwd_partial_rows(a.T);
  if (a.T > 0) {
    kernel_timer_mark(kTimeConvBwd, true, st);
    cudaError_t e = io == IO::F32 ? bwd_t<float>(a, tm_x, tm_du, st) : bwd_t<__nv_bfloat16>(a, tm_x, tm_du, st);
    kernel_timer_mark(kTimeConvBwd, false, st);
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
