// scan_bwd.cu -- packed selective scan, backward (sm_103a).
//
// Work item = (chunk of kBwdChunk = 32 tokens, the saved-state granule) x
// (tile of kTile = 32 channels); items are taken in DESCENDING chunk order
// from an atomic ticket because the state gradient flows from the end of a
// sequence to its start.  The kernel is persistent (one CTA per resident slot,
// looping over tickets); each item's inputs are requested by one thread with
// tensor / bulk copies on one mbarrier while the previous item finishes.
// CTA = 8 warps; warp s owns K = 4 tokens, lane l owns channel d0 + l with
// all N states.
//
// With a_t = exp(delta_t A) (0 at a sequence start), g_t = dout_t SiLU(z_t),
// the state gradient obeys dh_t = a_{t+1} dh_{t+1} + C_t g_t and is zero after
// the last token of every sequence (a_{t+1} = 0 when t+1 starts a sequence):
// the reverse scan that resets at sequence ends.
//
//   1. Copies (issued during the previous item): u, delta_raw, dout, z tiles
//      (32 x 32), B and C rows, A rows, dt_bias, Dskip, saved states,
//      position indices; per-token delta, SiLU(z), g kept in registers.
//   2. Forward states: pass over the K tokens from h = 0 -> sub-chunk
//      aggregates; exclusive scan seeded with the chunk's saved state
//      (chunk_states from the forward call) gives each thread its start state.
//   3. Reverse aggregates: pass over the K tokens backwards from dh = 0; the
//      left-going carry of a block is (prod a) * carry_in + G, with G the carry
//      out when nothing comes in; exclusive reverse scan in shared memory.
//   4. Decoupled look-back towards HIGHER chunks for the carry entering the
//      chunk from the right, re-applied in a fixed order (bitwise repeatable),
//      time-bounded waits.
//   5. Recompute the K forward states into shared memory, then walk the K
//      tokens backwards producing du, d(delta_raw), dz and per-token partial
//      dB, dC (reduced over the warp's 32 channels with a butterfly
//      reduce-scatter, no atomics) and per-thread partial dA, dDskip, d_dt_bias.
//   6. Fixed-order CTA reduction of the partials; separate fixed-order kernels
//      sum them over channel tiles (dB, dC) and chunks (dA, dDskip, d_dt_bias).
#include "common.cuh"
#include "kernels.h"

namespace vssm {

namespace {

constexpr int kL = kBwdChunk;   // 32
constexpr int kS = 8;
constexpr int kK = kL / kS;     // 4
constexpr int kThreads = kS * 32;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T, int N>
struct BwdSmem {
  // ---- inputs of one work item, written by tensor / bulk copies and refilled
  //      for the next item while this one is still being processed
  alignas(128) T u[kL * kTile];
  alignas(128) T dr[kL * kTile];
  alignas(128) T z[kL * kTile];
  alignas(128) T dout[kL * kTile];
  alignas(128) T B[kL * N];
  alignas(128) T C[kL * N];
  alignas(16) float Araw[kTile * N];   // A rows d0 .. d0+31
  alignas(16) float Hraw[kTile * N];   // saved states at the chunk start, same rows
  alignas(16) float bias[kTile];
  alignas(16) float dsk[kTile];
  alignas(16) int pos[kL];
  // ---- working set of the item being processed
  // B and C widened to fp32 once per work item (bf16 I/O only; fp32 I/O reads B, C directly)
  alignas(16) float Bf[sizeof(T) == 2 ? kL * N : 4];
  alignas(16) float Cf[sizeof(T) == 2 ? kL * N : 4];
  // states after a thread's first K-1 tokens ([k][n/4][tid]); the state after
  // its last token stays in registers
  alignas(16) float4 hist[(kK - 1) * (N / 4) * kThreads];
  alignas(16) float aggH[kS * N * kTile];  // forward aggregates, then each warp's start state
  alignas(16) float aggG[kS * N * kTile];  // reverse aggregates, then exclusive suffixes, then the dA block
  float tot[N * kTile];
  float rin[N * kTile];
  float aggSD[kS * kTile];
  float redD[kS * kTile];
  float redB[kS * kTile];
  int aggRS[kS];
  int ticket;
  alignas(8) uint64_t bar;
};

// Butterfly reduce-scatter over the 32 lanes of a warp: on entry each lane
// holds C values; on exit v[0] of lane l is the sum over all lanes of value
// l >> (5 - log2 C).  Fixed pairing order, so the sums are reproducible.
template <int C, int M>
struct ReduceScatter {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (C > 1) {
      constexpr int H = C / 2;
      const bool up = (lane & M) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = up ? v[i] : v[i + H];
        const float keep = up ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
      }
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
    }
    if constexpr (M > 1) ReduceScatter<(C > 1 ? C / 2 : 1), M / 2>::run(v, lane);
  }
};

template <typename T, int N>
__global__ void __launch_bounds__(kThreads, 2)
scan_bwd_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dr,
                const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_dout,
                const ScanArgs a) {
  using SM = BwdSmem<T, N>;
  constexpr int P = N / 2;                       // state pairs
  constexpr int V = 2 * N;                       // dB and dC values per token
  constexpr int kRep = 32 / (V < 32 ? V : 32);   // lanes holding the same value
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, s = tid >> 5;

  const int n_items = a.n_chunks * a.n_tiles;

  // Requests every input of work item `tkn` on the barrier: u, delta_raw,
  // dout, z tiles; B and C rows; A rows, dt_bias, Dskip and the saved states
  // of the tile's channels; position indices (whole groups of 4 tokens).
  auto issue = [&](int tkn) {
    const int rv = tkn / a.n_tiles;
    const int tl = tkn - rv * a.n_tiles;
    const int ch = a.n_chunks - 1 - rv;
    const int64_t tt0 = (int64_t)ch * kL;
    const int nrows = (int)((a.T - tt0) < kL ? (a.T - tt0) : kL);
    const int dd0 = tl * kTile;
    const uint32_t nval = (uint32_t)(a.D - dd0 < kTile ? a.D - dd0 : kTile);
    const uint32_t bc = (uint32_t)nrows * N * sizeof(T);
    const uint32_t rows4 = (uint32_t)nrows & ~3u;
    const uint32_t box = (uint32_t)a.box_x * (uint32_t)a.box_y * sizeof(T);
    mbar_arrive_expect_tx(&sm.bar, box * (a.has_z ? 4u : 3u) + 2u * bc + 2u * nval * N * 4u +
                                       rows4 * 4u + (a.dt_bias ? nval * 4u : 0u) +
                                       (a.Dskip ? nval * 4u : 0u));
    tma_load_2d(sm.u, &tm_u, dd0, (int)tt0, &sm.bar);
    tma_load_2d(sm.dr, &tm_dr, dd0, (int)tt0, &sm.bar);
    tma_load_2d(sm.dout, &tm_dout, dd0, (int)tt0, &sm.bar);
    if (a.has_z) tma_load_2d(sm.z, &tm_z, dd0, (int)tt0, &sm.bar);
    bulk_load_1d(sm.B, static_cast<const T*>(a.B) + tt0 * N, bc, &sm.bar);
    bulk_load_1d(sm.C, static_cast<const T*>(a.C) + tt0 * N, bc, &sm.bar);
    bulk_load_1d(sm.Araw, a.A + (int64_t)dd0 * N, nval * N * 4u, &sm.bar);
    bulk_load_1d(sm.Hraw, a.chunk_states + ((int64_t)ch * a.D + dd0) * N, nval * N * 4u, &sm.bar);
    if (a.dt_bias) bulk_load_1d(sm.bias, a.dt_bias + dd0, nval * 4u, &sm.bar);
    if (a.Dskip) bulk_load_1d(sm.dsk, a.Dskip + dd0, nval * 4u, &sm.bar);
    if (rows4) bulk_load_1d(sm.pos, a.pos + tt0, rows4 * 4u, &sm.bar);
  };

  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
    const int first = (int)atomicAdd(a.ticket, 1u);
    sm.ticket = first;
    if (first < n_items) issue(first);
  }
  __syncthreads();

  // Persistent loop: one work item per pass.  The next ticket is drawn once
  // this item has read its inputs for the last time (after step 7) and its
  // copies land while this item finishes its reductions.  An earlier draw
  // would hold tickets back from the look-back chains (an item whose
  // neighbour sits reserved behind a running item waits for both), which
  // measurably slows the whole kernel.  Items only ever wait on items with
  // smaller tickets, all of which are done or in hand of a running CTA, so
  // the loop cannot deadlock.
  for (uint32_t it = 0;; ++it) {
  const int tk = sm.ticket;
  if (tk >= n_items) break;
  const int rev = tk / a.n_tiles;
  const int tile = tk - rev * a.n_tiles;
  const int chunk = a.n_chunks - 1 - rev;
  const int64_t t0 = (int64_t)chunk * kL;
  const int rows = (int)((a.T - t0) < kL ? (a.T - t0) : kL);
  const int rows4 = rows & ~3;
  const int d0 = tile * kTile;
  const int bx = a.box_x;
  const int d = d0 + lane;
  const bool valid = lane < bx && d < a.D;

  if (!__syncthreads_and(mbar_wait(&sm.bar, it & 1u, a.wait_ns))) {
    if (tid == 0) atomicOr(a.status, kStatusTmaTimeout);
    break;
  }
  const float bias = (valid && a.dt_bias) ? sm.bias[lane] : 0.0f;
  const float Dsk = (valid && a.Dskip) ? sm.dsk[lane] : 0.0f;
  const float* Bf = widen_rows<T>(sm.B, sm.Bf, rows * N, tid, kThreads);
  const float* Cf = widen_rows<T>(sm.C, sm.Cf, rows * N, tid, kThreads);
  float2 A2[P];
  if (valid) {
    load_scaled_pairs<N>(A2, sm.Araw + lane * N, kLog2e);
  } else {
#pragma unroll
    for (int i = 0; i < P; ++i) A2[i] = make_float2(0.0f, 0.0f);
  }

  const int tb = s * kK;
  // ---- 1. per-token values (registers); lanes without a channel get u = g = 0
  //         so that every partial they feed into a channel sum is exactly 0
  float dl[kK], sg[kK], uu[kK], g[kK], dzf[kK];
  int rst = 0;  // bit k: token tb+k starts a sequence (warp-uniform)
#pragma unroll
  for (int k = 0; k < kK; ++k) {
    const int t = tb + k;
    dl[k] = sg[k] = uu[k] = g[k] = dzf[k] = 0.0f;
    if (t < rows) {
      const float r = to_f(sm.dr[t * bx + lane]) + bias;
      if (a.delta_softplus) {
        dl[k] = softplusf(r);
        sg[k] = sigmoidf_fast(r);
      } else {
        dl[k] = r;
        sg[k] = 1.0f;
      }
      uu[k] = valid ? to_f(sm.u[t * bx + lane]) : 0.0f;
      const float go = valid ? to_f(sm.dout[t * bx + lane]) : 0.0f;
      if (a.has_z) {
        const float zz = to_f(sm.z[t * bx + lane]);
        const float sz = sigmoidf_fast(zz);
        g[k] = go * (zz * sz);
        dzf[k] = go * sz * fmaf(zz, 1.0f - sz, 1.0f);
      } else {
        g[k] = go;
      }
      const int pt = t < rows4 ? sm.pos[t] : __ldg(a.pos + t0 + t);
      if (pt == 0) rst |= 1 << k;
    }
  }
  __syncthreads();  // Bf, Cf complete

  // ---- 2. both aggregates of my K tokens: forward (state from 0) and reverse
  //         (carry leaving to the left when nothing enters from the right)
  {
    float2 h[P];
#pragma unroll
    for (int i = 0; i < P; ++i) h[i] = make_float2(0.0f, 0.0f);
    float sd = 0.0f;
#pragma unroll
    for (int k = 0; k < kK; ++k) {
      const int t = tb + k;
      if (t >= rows) break;
      if (rst & (1 << k)) {
#pragma unroll
        for (int i = 0; i < P; ++i) h[i] = make_float2(0.0f, 0.0f);
        sd = 0.0f;
      }
      const float2 dl2 = splat2(dl[k]), du2 = splat2(dl[k] * uu[k]);
      float2 Bv[P];
      lds_pairs<N>(Bv, Bf + t * N);
#pragma unroll
      for (int i = 0; i < P; ++i) h[i] = fma2(ex2x2(mul2(dl2, A2[i])), h[i], mul2(du2, Bv[i]));
      sd += dl[k];
    }
    float2 q[P];
#pragma unroll
    for (int i = 0; i < P; ++i) q[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = kK - 1; k >= 0; --k) {
      const int t = tb + k;
      if (t >= rows) continue;
      float2 Cv[P];
      lds_pairs<N>(Cv, Cf + t * N);
      // ex2(-inf) = 0: the transition factor of a sequence's first token, for any A
      const float2 off2 = splat2((rst & (1 << k)) ? -INFINITY : 0.0f);
      const float2 dl2 = splat2(dl[k]), g2 = splat2(g[k]);
#pragma unroll
      for (int i = 0; i < P; ++i) q[i] = mul2(ex2x2(fma2(dl2, A2[i], off2)), fma2(Cv[i], g2, q[i]));
    }
#pragma unroll
    for (int i = 0; i < P; ++i) {
      sm.aggH[(s * N + 2 * i) * kTile + lane] = h[i].x;
      sm.aggH[(s * N + 2 * i + 1) * kTile + lane] = h[i].y;
      sm.aggG[(s * N + 2 * i) * kTile + lane] = q[i].x;
      sm.aggG[(s * N + 2 * i + 1) * kTile + lane] = q[i].y;
    }
    sm.aggSD[s * kTile + lane] = sd;
    if (lane == 0) sm.aggRS[s] = rst != 0;
  }
  __syncthreads();

  // ---- 3. both in-CTA scans over the kS sub-chunks; chain (lane, n), n % kS == s.
  //         Forward: exclusive prefix seeded with the saved state of the chunk.
  //         Reverse: exclusive suffix with nothing entering from the right.
  {
    float sdj[kS];
    int rsj[kS];
#pragma unroll
    for (int j = 0; j < kS; ++j) {
      sdj[j] = sm.aggSD[j * kTile + lane];
      rsj[j] = sm.aggRS[j];
    }
#pragma unroll
    for (int n = 0; n < N; ++n) {
      if (n % kS != s) continue;
      const float a2 = (n & 1) ? A2[n / 2].y : A2[n / 2].x;
      float Pj[kS], Hj[kS], Gj[kS];
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        Pj[j] = rsj[j] ? 0.0f : ex2(a2 * sdj[j]);
        Hj[j] = sm.aggH[(j * N + n) * kTile + lane];
        Gj[j] = sm.aggG[(j * N + n) * kTile + lane];
      }
      float x = valid ? sm.Hraw[lane * N + n] : 0.0f;
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        sm.aggH[(j * N + n) * kTile + lane] = x;
        x = fmaf(Pj[j], x, Hj[j]);
      }
      float y = 0.0f;
#pragma unroll
      for (int j = kS - 1; j >= 0; --j) {
        sm.aggG[(j * N + n) * kTile + lane] = y;
        y = fmaf(Pj[j], y, Gj[j]);
      }
      sm.tot[n * kTile + lane] = y;
    }
  }
  __syncthreads();

  // ---- 4. decoupled look-back towards higher chunks (warp 0); the other warps
  //         go straight on to step 5, which needs no carry from the right
  if (s == 0) {
    int rs_any = 0;
    float sd_tot = 0.0f;
#pragma unroll
    for (int j = 0; j < kS; ++j) {
      rs_any |= sm.aggRS[j];
      sd_tot += sm.aggSD[j * kTile + lane];
    }
    const int64_t base = (int64_t)tile * a.n_chunks;
    const int64_t slot = base + chunk;
    const bool publish = (long long)tk != a.drop_ticket;
    float* my_agg = a.agg + slot * (N * kTile);
    float* my_inc = a.incl + slot * (N * kTile);
    // every lane is its own chain (one channel): it publishes its payload and
    // then its own flag with a release store, and readers acquire that flag
    int* my_flag = a.flags + slot * kTile + lane;
    if (rs_any) {
      // a sequence starts in this chunk: the carry leaving it to the left does
      // not depend on what enters from the right, publish it at once
#pragma unroll
      for (int n = 0; n < N; ++n) my_inc[n * kTile + lane] = sm.tot[n * kTile + lane];
      if (publish) st_release_gpu(my_flag, kFlagInclusive);
    }
    float x[N];
#pragma unroll
    for (int n = 0; n < N; ++n) x[n] = 0.0f;
    if (chunk < a.n_chunks - 1) {
      // the next chunk of the tile started long before this one and has
      // usually published its inclusive carry: look first, and publish this
      // chunk's aggregate only when the walk has to go further
      int j = chunk + 1, found = -1, timed_out = 0;
      if (ld_acquire_gpu(a.flags + (base + j) * kTile + lane) == kFlagInclusive) {
        found = j;
      } else {
        if (!rs_any) {
#pragma unroll
          for (int n = 0; n < N; ++n) my_agg[n * kTile + lane] = sm.tot[n * kTile + lane];
          a.agg_sd[slot * kTile + lane] = sd_tot;
          if (publish) st_release_gpu(my_flag, kFlagAggregate);
        }
        while (j < a.n_chunks) {
          const int f = wait_flag(a.flags + (base + j) * kTile + lane, a.wait_ns);
          if (f == kFlagInclusive) { found = j; break; }
          if (f == kFlagNone) { timed_out = 1; break; }
          ++j;
        }
      }
      if (timed_out) atomicOr(a.status, kStatusLookbackTimeout);
      int last = j - 1;
      if (found >= 0) {
        const float* inc = a.incl + (base + found) * (N * kTile);
#pragma unroll
        for (int n = 0; n < N; ++n) x[n] = __ldcg(inc + n * kTile + lane);
        last = found - 1;
      }
      for (int i = last; i > chunk; --i) {
        const float* ag = a.agg + (base + i) * (N * kTile);
        const float sdi = __ldcg(a.agg_sd + (base + i) * kTile + lane);
#pragma unroll
        for (int n = 0; n < N; ++n) {
          const float a2 = (n & 1) ? A2[n / 2].y : A2[n / 2].x;
          x[n] = fmaf(ex2(a2 * sdi), x[n], __ldcg(ag + n * kTile + lane));
        }
      }
    }
#pragma unroll
    for (int n = 0; n < N; ++n) sm.rin[n * kTile + lane] = x[n];
    if (!rs_any) {
      // released at once: the next chunk of the tile may already be waiting,
      // and every link of that chain adds this item's publication delay
#pragma unroll
      for (int n = 0; n < N; ++n) {
        const float a2 = (n & 1) ? A2[n / 2].y : A2[n / 2].x;
        my_inc[n * kTile + lane] = fmaf(ex2(a2 * sd_tot), x[n], sm.tot[n * kTile + lane]);
      }
      if (publish) st_release_gpu(my_flag, kFlagInclusive);
    }
  }

  // ---- 5. recompute the forward states of my K tokens from my start state;
  //         the first K-1 go to shared memory, the last stays in registers
  float2 h[P];
#pragma unroll
  for (int i = 0; i < P; ++i)
    h[i] = make_float2(sm.aggH[(s * N + 2 * i) * kTile + lane], sm.aggH[(s * N + 2 * i + 1) * kTile + lane]);
  float yk[kK];
#pragma unroll
  for (int k = 0; k < kK; ++k) {
    const int t = tb + k;
    yk[k] = 0.0f;
    if (t >= rows) continue;
    if (rst & (1 << k)) {
#pragma unroll
      for (int i = 0; i < P; ++i) h[i] = make_float2(0.0f, 0.0f);
    }
    const float2 dl2 = splat2(dl[k]), du2 = splat2(dl[k] * uu[k]);
    float2 Bv[P], Cv[P];
    lds_pairs<N>(Bv, Bf + t * N);
    lds_pairs<N>(Cv, Cf + t * N);
    float2 y2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < P; ++i) {
      h[i] = fma2(ex2x2(mul2(dl2, A2[i])), h[i], mul2(du2, Bv[i]));
      y2 = fma2(Cv[i], h[i], y2);
    }
    if (k < kK - 1) {
#pragma unroll
      for (int i = 0; i < P; i += 2)
        sm.hist[(k * (N / 4) + i / 2) * kThreads + tid] = make_float4(h[i].x, h[i].y, h[i + 1].x, h[i + 1].y);
    }
    yk[k] = fmaf(Dsk, uu[k], y2.x + y2.y);
  }
  __syncthreads();

  // the next ticket, drawn now and used once this item's inputs are consumed
  // (the atomic's latency hides behind step 7)
  // ---- 6. carry entering my last token from the right
  float2 dh[P];
  {
    int rs_post = 0;
    float sd_post = 0.0f;
    for (int j = s + 1; j < kS; ++j) {
      rs_post |= sm.aggRS[j];
      sd_post += sm.aggSD[j * kTile + lane];
    }
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const float2 E = make_float2(sm.aggG[(s * N + 2 * i) * kTile + lane],
                                   sm.aggG[(s * N + 2 * i + 1) * kTile + lane]);
      const float2 R = make_float2(sm.rin[(2 * i) * kTile + lane], sm.rin[(2 * i + 1) * kTile + lane]);
      dh[i] = rs_post ? E : fma2(ex2x2(mul2(A2[i], splat2(sd_post))), R, E);
    }
  }

  // ---- 7. reverse walk over my tokens
  float2 dA[P];
#pragma unroll
  for (int i = 0; i < P; ++i) dA[i] = make_float2(0.0f, 0.0f);
  float sDD = 0.0f, sDB = 0.0f;
  T* gdu = static_cast<T*>(a.du);
  T* gddr = static_cast<T*>(a.ddr);
  T* gdz = static_cast<T*>(a.dz);
#pragma unroll
  for (int k = kK - 1; k >= 0; --k) {
    const int t = tb + k;
    if (t >= rows) continue;  // warp-uniform
    float2 Bv[P], Cv[P];
    lds_pairs<N>(Bv, Bf + t * N);
    lds_pairs<N>(Cv, Cf + t * N);
    const float2 off2 = splat2((rst & (1 << k)) ? -INFINITY : 0.0f);
    const float2 dl2 = splat2(dl[k]), g2 = splat2(g[k]), du2 = splat2(dl[k] * uu[k]);
    float v[V];
    float2 s1 = make_float2(0.0f, 0.0f), s2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < P; i += 2) {
      float2 hc[2], hp[2];
      if (k == kK - 1) {
        hc[0] = h[i];
        hc[1] = h[i + 1];
      } else {
        const float4 c4 = sm.hist[(k * (N / 4) + i / 2) * kThreads + tid];
        hc[0] = make_float2(c4.x, c4.y);
        hc[1] = make_float2(c4.z, c4.w);
      }
      if (k > 0) {
        const float4 p4 = sm.hist[((k - 1) * (N / 4) + i / 2) * kThreads + tid];
        hp[0] = make_float2(p4.x, p4.y);
        hp[1] = make_float2(p4.z, p4.w);
      } else {
        hp[0] = make_float2(sm.aggH[(s * N + 2 * i) * kTile + lane], sm.aggH[(s * N + 2 * i + 1) * kTile + lane]);
        hp[1] = make_float2(sm.aggH[(s * N + 2 * i + 2) * kTile + lane], sm.aggH[(s * N + 2 * i + 3) * kTile + lane]);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = i + e;
        dh[j] = fma2(Cv[j], g2, dh[j]);  // total gradient w.r.t. h_t
        const float2 at = ex2x2(fma2(dl2, A2[j], off2));
        const float2 dhq = mul2(dh[j], mul2(at, hp[e]));
        dA[j] = fma2(dl2, dhq, dA[j]);
        s2 = fma2(A2[j], dhq, s2);
        s1 = fma2(dh[j], Bv[j], s1);
        const float2 vb = mul2(dh[j], du2);   // 0 on lanes without a channel (u = 0)
        const float2 vc = mul2(g2, hc[e]);    // 0 on lanes without a channel (g = 0)
        v[2 * j] = vb.x;
        v[2 * j + 1] = vb.y;
        v[N + 2 * j] = vc.x;
        v[N + 2 * j + 1] = vc.y;
        dh[j] = mul2(dh[j], at);               // carry to h_{t-1}
      }
    }
    const float s1t = s1.x + s1.y, s2t = s2.x + s2.y;
    const float gdu_t = fmaf(dl[k], s1t, Dsk * g[k]);
    const float gdl_t = fmaf(uu[k], s1t, s2t * kLn2);
    const float gdr_t = gdl_t * sg[k];
    sDD = fmaf(g[k], uu[k], sDD);
    sDB += gdr_t;
    const int64_t at_td = (t0 + t) * a.D + d;
    if (valid) {
      gdu[at_td] = from_f<T>(gdu_t);
      gddr[at_td] = from_f<T>(gdr_t);
      if (gdz) gdz[at_td] = from_f<T>(dzf[k] * yk[k]);
    }
    ReduceScatter<V, 16>::run(v, lane);
    if ((lane & (kRep - 1)) == 0)
      a.part_dBC[((int64_t)tile * a.T + t0 + t) * V + lane / kRep] = v[0];
  }

  // ---- 8. fixed-order CTA reduction of dA, dDskip, d_dt_bias partials
  __syncthreads();
  // no input buffer is read any more: draw the next item and request its
  // inputs, which land while this item finishes its reductions
  if (tid == 0) {
    const int next = (int)atomicAdd(a.ticket, 1u);
    sm.ticket = next;
    if (next < n_items) issue(next);
  }
#pragma unroll
  for (int i = 0; i < P; ++i) {
    sm.aggH[(s * N + 2 * i) * kTile + lane] = dA[i].x;
    sm.aggH[(s * N + 2 * i + 1) * kTile + lane] = dA[i].y;
  }
  sm.redD[s * kTile + lane] = sDD;
  sm.redB[s * kTile + lane] = sDB;
  __syncthreads();
#pragma unroll
  for (int n = 0; n < N; ++n) {
    if (n % kS != s) continue;
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < kS; ++j) acc += sm.aggH[(j * N + n) * kTile + lane];
    sm.aggG[lane * (N + 4) + n] = acc;
  }
  if (s == 0 && valid) {
    float accD = 0.0f, accB = 0.0f;
#pragma unroll
    for (int j = 0; j < kS; ++j) {
      accD += sm.redD[j * kTile + lane];
      accB += sm.redB[j * kTile + lane];
    }
    a.part_dD[(int64_t)chunk * a.D + d] = accD;
    a.part_dbias[(int64_t)chunk * a.D + d] = accB;
  }
  __syncthreads();
  // the tile's dA partial block is contiguous in part_dA: write it coalesced
  {
    float* dst = a.part_dA + ((int64_t)chunk * a.D + d0) * N;
    const int nvalid = (a.D - d0 < kTile ? a.D - d0 : kTile) * N;
    for (int i = tid; i < nvalid; i += kThreads) dst[i] = sm.aggG[(i / N) * (N + 4) + (i % N)];
  }
  }  // persistent loop
}

// dB[t][n] = sum over tiles of part[tile][t][n]; dC[t][n] likewise from
// part[tile][t][N + n].  One thread per output, tiles summed in order.
__global__ void __launch_bounds__(256) sum_tiles_bc_kernel(const float* __restrict__ part,
                                                           int n_tiles, int64_t T, int N,
                                                           float* __restrict__ dB,
                                                           float* __restrict__ dC) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t M = T * 2 * N;
  if (i >= M) return;
  float acc = 0.0f;
  for (int k = 0; k < n_tiles; ++k) acc += __ldcs(part + (int64_t)k * M + i);
  const int64_t t = i / (2 * N);
  const int j = (int)(i - t * 2 * N);
  if (j < N) dB[t * N + j] = acc; else dC[t * N + (j - N)] = acc;
}

template <typename T, int N>
cudaError_t launch_n(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, const CUtensorMap& tm_dout, cudaStream_t st) {
  const size_t smem = sizeof(BwdSmem<T, N>);
  cudaError_t e = cudaFuncSetAttribute(scan_bwd_kernel<T, N>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.n_chunks * a.n_tiles;
  int grid = 0;
  e = persistent_grid(scan_bwd_kernel<T, N>, kThreads, smem, items, &grid);
  if (e != cudaSuccess) return e;
  scan_bwd_kernel<T, N><<<grid, kThreads, smem, st>>>(tm_u, tm_dr, tm_z, tm_dout, a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, const CUtensorMap& tm_dout, cudaStream_t st) {
  if (a.N == 16) return launch_n<T, 16>(a, tm_u, tm_dr, tm_z, tm_dout, st);
  if (a.N == 8) return launch_n<T, 8>(a, tm_u, tm_dr, tm_z, tm_dout, st);
  if constexpr (sizeof(T) == 4) {
    if (a.N == 4) return launch_n<T, 4>(a, tm_u, tm_dr, tm_z, tm_dout, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_scan_bwd(const ScanArgs& a, IO io, const CUtensorMap& tm_u,
                            const CUtensorMap& tm_dr, const CUtensorMap& tm_z,
                            const CUtensorMap& tm_dout, float* dA, float* dB, float* dC,
                            float* dDskip, float* d_dt_bias, cudaStream_t st) {
  const int64_t DN = (int64_t)a.D * a.N;
  if (a.T <= 0) {
    cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(float) * DN, st);
    if (e == cudaSuccess && dDskip) e = cudaMemsetAsync(dDskip, 0, sizeof(float) * a.D, st);
    if (e == cudaSuccess && d_dt_bias) e = cudaMemsetAsync(d_dt_bias, 0, sizeof(float) * a.D, st);
    return e;
  }
  cudaError_t e = io == IO::F32 ? launch_t<float>(a, tm_u, tm_dr, tm_z, tm_dout, st)
                                : launch_t<__nv_bfloat16>(a, tm_u, tm_dr, tm_z, tm_dout, st);
  if (e != cudaSuccess) return e;
  const int64_t M = a.T * 2 * a.N;
  sum_tiles_bc_kernel<<<(unsigned)((M + 255) / 256), 256, 0, st>>>(a.part_dBC, a.n_tiles, a.T, a.N,
                                                                   dB, dC);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_sum_rows(a.part_dA, a.n_chunks, DN, DN, dA, st);
  if (e == cudaSuccess && dDskip) e = launch_sum_rows(a.part_dD, a.n_chunks, a.D, a.D, dDskip, st);
  if (e == cudaSuccess && d_dt_bias)
    e = launch_sum_rows(a.part_dbias, a.n_chunks, a.D, a.D, d_dt_bias, st);
  return e;
}

}  // namespace vssm
