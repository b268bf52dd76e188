// scan_fwd.cu -- packed selective scan, forward (sm_103a).
//
// Work item = (chunk of kFwdChunk = 128 tokens) x (tile of kTile = 32 channels).
// A CTA of 256 threads = 8 warps; warp s owns sub-chunk s (K = 16 tokens) and
// lane l owns channel d0 + l with all N states in registers.
//
//   1. Copies: u, delta_raw, z tiles (128 x 32) with 2-D tensor maps; B and C
//      rows (128 x N, contiguous), A rows, dt_bias, Dskip and position indices
//      with 1-D bulk copies; one mbarrier.  The kernel is persistent (one CTA
//      per resident slot, looping over tickets), and one thread requests the
//      next item's copies as soon as the current item has read its inputs.
//   2. delta = softplus(delta_raw + dt_bias) once per (token, channel), in
//      pass 1, kept in shared memory for pass 2.
//   3. Pass 1: every thread scans its K tokens from h = 0 and records the
//      sub-chunk aggregate: H (the state reached) and the sum of delta since
//      the last sequence start; the product of the transition factors over the
//      sub-chunk is then exp2(A*log2e * sum) or exactly 0 if a sequence starts
//      inside it (the article's SSM_pack zeroes the factor at a start).
//   4. Exclusive scan of the 8 sub-chunk aggregates per (channel, state) in
//      shared memory; warp s takes the states n = s (mod 8).
//   5. Decoupled look-back across chunks, each warp on its own states' chain:
//      the inclusive state of a chunk is stored word by word, each word its
//      own "stored" flag (the array starts as all-ones NaNs); an aggregate is
//      published, behind a fence and the warp's flag, only when a walk has to
//      go past it.  The walk goes back to the nearest inclusive state and
//      re-applies the aggregates FORWARD from there in chunk order, which gives
//      the same floating-point result whatever the timing (bitwise repeatable).
//      Work items take chunk ids from an atomic ticket, so a CTA only ever waits
//      on items already running; every wait is time-bounded and a timeout is
//      reported through the status word instead of hanging.
//      Once the entering state is known, the owning warp turns each sub-chunk's
//      prefix into its exact start state (prefix + entering state times the
//      product of the factors of the sub-chunks before it).
//   6. Pass 2: each thread starts from its exact state, recomputes its K tokens
//      and writes out = (C.h + Dskip u) * SiLU(z); states at multiples of 32
//      tokens go to chunk_states for the backward pass.
#include "common.cuh"
#include "kernels.h"

namespace vssm {

namespace {

constexpr int kL = kFwdChunk;   // 128
constexpr int kS = 8;           // sub-chunks (warps)
constexpr int kK = kL / kS;     // 16 tokens per thread
constexpr int kThreads = kS * 32;

constexpr int kHalo = 3;        // x rows before the chunk a fused conv of width <= 4 reads
constexpr int kMaxW = 4;        // widest fused conv

// Buffers of the inputs pass 2 reads (u, z, B, C, positions): two for bf16
// I/O without the fused conv, so that the next work item's copies land while
// pass 2 runs; one otherwise (the fp32 tiles and the conv's x tile leave no
// room for a second CTA per SM with two).
template <typename T, bool kConv>
constexpr int fwd_buffers() { return (sizeof(T) == 2 && !kConv) ? 2 : 1; }

template <typename T, int N, bool kConv>
struct FwdSmem {
  static constexpr int NB = fwd_buffers<T, kConv>();
  alignas(128) T u[NB][kL * kTile];
  // fused conv1d: x rows t0 - 3 .. t0 + 127 (by one tensor copy; rows before
  // the first token come back zero), the tile's weights (D, W) and bias
  alignas(128) T x[kConv ? (kL + kHalo) * kTile : 8];
  alignas(16) float cw[kConv ? kTile * kMaxW : 4];
  alignas(16) float cb[kConv ? kTile : 4];
  alignas(128) T dr[kL * kTile];
  alignas(128) T z[NB][kL * kTile];
  // B and C rows as fp32 (for bf16 I/O widened once per call, before the kernel)
  alignas(128) float B[NB][kL * N];
  alignas(128) float C[NB][kL * N];
  alignas(16) float dlt[kL * kTile];
  alignas(16) float aggH[kS * N * kTile];
  float aggSD[kS * kTile];
  alignas(16) float4 Af[N / 4 * kTile];  // the tile's A rows, prepared once per call (ScanArgs::Af)
  alignas(16) float bias[kTile];
  alignas(16) float dsk[kTile];
  alignas(16) int pos[NB][kL];
  int aggRS[kS];
  int ticket;
  alignas(8) uint64_t bar;
};

// kStates: the call passes sequence states (initial and/or final); without
// them the kernel carries no code for them.  kConv: the call passes the conv1d
// input x instead of u (tm_u maps x), and the kernel computes
// u = SiLU(bias + sum_k w[W-1-k] x[t-k] [pos[t] >= k]) itself in pass 1, with
// the conv kernel's arithmetic in the conv kernel's order, rounding u to the
// I/O type as that kernel's store does (so the results equal the two calls'
// bit for bit); u goes to a.u_out when the call asks for it (the backward
// needs it).
template <typename T, int N, bool kStates, bool kKnob, bool kConv>
__global__ void __launch_bounds__(kThreads, 2)
scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dr,
                const __grid_constant__ CUtensorMap tm_z, const ScanArgs a) {
  using SM = FwdSmem<T, N, kConv>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, s = tid >> 5;

  const int n_items = a.n_chunks * a.n_tiles;

  // Requests warp wq's share of the inputs of work item `tkn` on the barrier,
  // which expects one arrival per warp: lane 0 of each warp posts its share's
  // bytes and issues its copies (one thread issuing all of them in turn held
  // its warp, and the CTA behind it, for about a thousand cycles).  Shares:
  // 0 the u tile (the fused conv: the x tile, weights and bias) and the
  // position indices (whole groups of 4 tokens), 1 delta_raw, 2 z, 3 B rows,
  // 4 C rows, 5 A rows, 6 dt_bias, 7 Dskip.  With no item left, every warp
  // arrives without data, so that the barrier still completes and tells
  // every thread to stop.
  auto issue = [&](int tkn, int buf, int wq) {
    if (tkn >= n_items) {
      mbar_arrive(&sm.bar);
      return;
    }
    const int ch = tkn / a.n_tiles;
    const int tl = tkn - ch * a.n_tiles;
    const int64_t tt0 = (int64_t)ch * kL;
    const int nrows = (int)((a.T - tt0) < kL ? (a.T - tt0) : kL);
    const int dd0 = tl * kTile;
    const uint32_t nval = (uint32_t)(a.D - dd0 < kTile ? a.D - dd0 : kTile);
    const uint32_t bc = (uint32_t)nrows * N * 4u;
    const uint32_t box = (uint32_t)a.box_x * (uint32_t)a.box_y * sizeof(T);
    if (wq == 0) {
      const uint32_t rows4 = (uint32_t)nrows & ~3u;
      if constexpr (kConv) {
        // the fused conv's x box has kHalo more rows
        const uint32_t xbox = (uint32_t)a.box_x * (uint32_t)(a.box_y + kHalo) * sizeof(T);
        const uint32_t wbytes = nval * (uint32_t)a.conv_W * 4u;
        mbar_arrive_expect_tx(&sm.bar, xbox + wbytes + (a.conv_b ? nval * 4u : 0u) + rows4 * 4u);
        tma_load_2d(sm.x, &tm_u, dd0, (int)tt0 - kHalo, &sm.bar);
        bulk_load_1d(sm.cw, a.conv_w + (int64_t)dd0 * a.conv_W, wbytes, &sm.bar);
        if (a.conv_b) bulk_load_1d(sm.cb, a.conv_b + dd0, nval * 4u, &sm.bar);
      } else {
        mbar_arrive_expect_tx(&sm.bar, box + rows4 * 4u);
        tma_load_2d(sm.u[buf], &tm_u, dd0, (int)tt0, &sm.bar);
      }
      if (rows4) bulk_load_1d(sm.pos[buf], a.pos + tt0, rows4 * 4u, &sm.bar);
    } else if (wq == 1) {
      mbar_arrive_expect_tx(&sm.bar, box);
      tma_load_2d(sm.dr, &tm_dr, dd0, (int)tt0, &sm.bar);
    } else if (wq == 2) {
      mbar_arrive_expect_tx(&sm.bar, a.has_z ? box : 0u);
      if (a.has_z) tma_load_2d(sm.z[buf], &tm_z, dd0, (int)tt0, &sm.bar);
    } else if (wq == 3) {
      mbar_arrive_expect_tx(&sm.bar, bc);
      bulk_load_1d(sm.B[buf], (sizeof(T) == 4 ? static_cast<const float*>(a.B) : a.Bf32) + tt0 * N, bc, &sm.bar);
    } else if (wq == 4) {
      mbar_arrive_expect_tx(&sm.bar, bc);
      bulk_load_1d(sm.C[buf], (sizeof(T) == 4 ? static_cast<const float*>(a.C) : a.Cf32) + tt0 * N, bc, &sm.bar);
    } else if (wq == 5) {
      mbar_arrive_expect_tx(&sm.bar, (uint32_t)kTile * N * 4u);
      bulk_load_1d(sm.Af, a.Af + (int64_t)tl * (N / 4) * kTile, (uint32_t)kTile * N * 4u, &sm.bar);
    } else if (wq == 6) {
      mbar_arrive_expect_tx(&sm.bar, a.dt_bias ? nval * 4u : 0u);
      if (a.dt_bias) bulk_load_1d(sm.bias, a.dt_bias + dd0, nval * 4u, &sm.bar);
    } else {
      mbar_arrive_expect_tx(&sm.bar, a.Dskip ? nval * 4u : 0u);
      if (a.Dskip) bulk_load_1d(sm.dsk, a.Dskip + dd0, nval * 4u, &sm.bar);
    }
  };
  static_assert(kThreads == 8 * 32, "one share of the copies per warp");

  if (tid == 0) {
    mbar_init(&sm.bar, kThreads / 32);
    fence_mbar_init();
    sm.ticket = (int)atomicAdd(a.ticket, 1u);
  }
  __syncthreads();
  if (lane == 0) issue(sm.ticket, 0, s);

  // Persistent loop: one work item per pass.  The next ticket is drawn when
  // the in-CTA scan starts, so that the atomic's round trip overlaps the scan
  // and look-back, and published to every warp by the barrier before pass 2;
  // each warp requests its share of the next item's copies halfway through
  // its pass 2 into the other buffer set (two buffers), or at the end of
  // pass 2, when the inputs are free (one).  A draw at the start of the item
  // would hold tickets back from the look-back chains (an item whose
  // neighbour sits reserved behind a running item waits for both); pass 2
  // waits on nothing, so a ticket held through it is not held back long.
  // Items only ever wait on items with smaller tickets, all of which are done
  // or in hand of a running CTA, so the loop cannot deadlock.
  for (uint32_t it = 0;; ++it) {
  if (!__syncthreads_and(mbar_wait(&sm.bar, it & 1u, a.wait_ns))) {
    // report, and give the copies one more, long limit to land before the CTA
    // leaves (nothing it requested may still write into its shared memory)
    if (tid == 0) atomicOr(a.status, kStatusTmaTimeout);
    mbar_wait(&sm.bar, it & 1u, kCopyDrainNs);
    break;
  }
  const int tk = sm.ticket;
  if (tk >= n_items) break;
  // test knob (its own instantiation, so the others carry no code for it):
  // this item starts late, so its inclusive state is stored late and the
  // items after it on the chain walk back past their aggregates
  if constexpr (kKnob) {
    if ((long long)tk == a.delay_ticket) sleep_ns(a.delay_ns);
  }
  const int chunk = tk / a.n_tiles;
  const int tile = tk - chunk * a.n_tiles;
  const int64_t t0 = (int64_t)chunk * kL;
  // this item's buffers of the double-buffered inputs
  constexpr int kNB = SM::NB;
  const int buf = kNB == 2 ? (int)(it & 1u) : 0;
  T* const su = sm.u[buf];
  const T* const sz = sm.z[buf];
  const int* const spos = sm.pos[buf];
  const int rows = (int)((a.T - t0) < kL ? (a.T - t0) : kL);
  const int rows4 = rows & ~3;
  const int d0 = tile * kTile;
  const int bx = a.box_x;
  const int d = d0 + lane;
  const bool valid = lane < bx && d < a.D;
  constexpr int P = N / 2;  // state pairs
  const float bias = (valid && a.dt_bias) ? sm.bias[lane] : 0.0f;
  const float Dsk = (valid && a.Dskip) ? sm.dsk[lane] : 0.0f;
  // position index of token t < rows of the chunk (the last chunk's ragged
  // tail, past the last whole group of 4, is read from global memory)
  auto pos_at = [&](int t) { return t < rows4 ? spos[t] : __ldg(a.pos + t0 + t); };
  // fused conv1d: tap k (k tokens back) of this lane's channel; zero past W
  float tapw[kMaxW] = {0.0f, 0.0f, 0.0f, 0.0f}, cbias = 0.0f;
  if constexpr (kConv) {
#pragma unroll
    for (int k = 0; k < kMaxW; ++k) tapw[k] = (valid && k < a.conv_W) ? sm.cw[lane * a.conv_W + a.conv_W - 1 - k] : 0.0f;
    cbias = (valid && a.conv_b) ? sm.cb[lane] : 0.0f;
  }
  // u of chunk token t (< rows) for this lane's channel, computed from the x
  // tile: kept in the u tile for both passes and stored for the caller when asked
  auto conv_u = [&](int t) {
    const T* xr = sm.x + (t + kHalo) * bx + lane;
    const int p = pos_at(t);
    float pre = fmaf(tapw[0], to_f(xr[0]), cbias);
#pragma unroll
    for (int k = 1; k < kMaxW; ++k)
      if (k < a.conv_W && p >= k) pre = fmaf(tapw[k], to_f(xr[-k * bx]), pre);
    const T ot = from_f<T>(a.conv_silu ? siluf(pre) : pre);
    su[t * bx + lane] = ot;
    if (a.u_out && valid) static_cast<T*>(a.u_out)[(t0 + t) * a.D + d] = ot;
  };
  // the state a sequence starting at token t (of the chunk) starts from: its
  // row of the initial states, or zero
  auto start_state = [&](float2 (&hs)[N / 2], int t) {
    if (kStates && a.h_init && valid &&
        VSSM_CHECKED((unsigned)a.seq[t0 + t] < (unsigned)a.num_seqs, a.status)) {
      const float4* row = reinterpret_cast<const float4*>(a.h_init + ((int64_t)a.seq[t0 + t] * a.D + d) * N);
#pragma unroll
      for (int i = 0; i < N / 4; ++i) {
        const float4 q = __ldg(row + i);
        hs[2 * i] = make_float2(q.x, q.y);
        hs[2 * i + 1] = make_float2(q.z, q.w);
      }
    } else {
#pragma unroll
      for (int i = 0; i < N / 2; ++i) hs[i] = make_float2(0.0f, 0.0f);
    }
  };
  // the state after the last token t (of the chunk) of a sequence, into its
  // row of the final states
  auto end_state = [&](const float2 (&hs)[N / 2], int t) {
    if (valid && VSSM_CHECKED((unsigned)a.seq[t0 + t] < (unsigned)a.num_seqs, a.status)) {
      float4* row = reinterpret_cast<float4*>(a.h_final + ((int64_t)a.seq[t0 + t] * a.D + d) * N);
#pragma unroll
      for (int i = 0; i < N / 4; ++i)
        row[i] = make_float4(hs[2 * i].x, hs[2 * i].y, hs[2 * i + 1].x, hs[2 * i + 1].y);
    }
  };
  // token t (< rows) is the last of its sequence: the next token starts one,
  // or there is none
  auto seq_end = [&](int t) {
    const int n = t + 1;
    if (t0 + n >= a.T) return true;
    return (n < rows ? pos_at(n) : __ldg(a.pos + t0 + n)) == 0;
  };

  const int tb = s * kK;  // first token (within the chunk) of this thread
  const float* Bf = sm.B[buf];
  const float* Cf = sm.C[buf];
  // A * log2 e of this lane's channel (zero past D), as state pairs
  float2 A2[P];
#pragma unroll
  for (int b = 0; b < N / 4; ++b) {
    const float4 q = sm.Af[b * kTile + lane];
    A2[2 * b] = make_float2(q.x, q.y);
    A2[2 * b + 1] = make_float2(q.z, q.w);
  }

  // fused conv1d: this thread's 16 u values first, in a loop of independent
  // iterations (kept out of the walk's dependency chain), into the u tile
  if constexpr (kConv) {
#pragma unroll 4
    for (int k = 0; k < kK; ++k)
      if (tb + k < rows) conv_u(tb + k);
  }

  // ---- steps 2-3: delta for my tokens (kept for pass 2) and pass 1, the
  //      sub-chunk aggregate from h = 0
  float2 h[P];
#pragma unroll
  for (int i = 0; i < P; ++i) h[i] = make_float2(0.0f, 0.0f);
  float sd = 0.0f;
  int rs = 0;
  // bit k: token tb + k starts a sequence (tokens past the chunk's end never do)
  const unsigned rm = __ballot_sync(0xffffffffu, lane < kK && tb + lane < rows && pos_at(tb + lane) == 0);
  // the common case, a whole sub-chunk of a full-width tile, is walked with
  // compile-time offsets; the last chunk's ragged tail and narrow tiles take
  // the general loop
  const bool whole = tb + kK <= rows && bx == kTile;
  if (whole) {
    const T* const drp = sm.dr + tb * kTile + lane;
    const T* const up = su + tb * kTile + lane;
    float* const dlp = sm.dlt + tb * kTile + lane;
    const float* const bp = Bf + tb * N;
    // groups of 8 tokens, unrolled; the loop over the groups keeps the body
    // small enough for the instruction cache (the fully unrolled 16 tokens
    // of both passes stalled on instruction fetch)
#pragma unroll 1
    for (int kg = 0; kg < kK; kg += 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = kg + e;
      const float r = to_f(drp[k * kTile]) + bias;
      const float dl = a.delta_softplus ? softplusf(r) : r;
      dlp[k * kTile] = dl;
      if ((rm >> k) & 1u) {
        start_state(h, tb + k);
        sd = 0.0f;
        rs = 1;
      }
      const float2 dl2 = splat2(dl), du2 = splat2(dl * to_f(up[k * kTile]));
      float2 Bv[P];
      lds_pairs<N>(Bv, bp + k * N);
#pragma unroll
      for (int i = 0; i < P; ++i) h[i] = fma2(ex2x2(mul2(dl2, A2[i])), h[i], mul2(du2, Bv[i]));
      sd += dl;
    }
    }
  } else {
#pragma unroll 1  // ragged tails and narrow tiles only: kept small for the instruction cache
  for (int k = 0; k < kK; ++k) {
    const int t = tb + k;
    if (t >= rows) break;
    const float r = to_f(sm.dr[t * bx + lane]) + bias;
    const float dl = a.delta_softplus ? softplusf(r) : r;
    sm.dlt[t * kTile + lane] = dl;
    if (pos_at(t) == 0) {
      start_state(h, t);
      sd = 0.0f;
      rs = 1;
    }
    const float2 dl2 = splat2(dl), du2 = splat2(dl * to_f(su[t * bx + lane]));
    float2 Bv[P];
    lds_pairs<N>(Bv, Bf + t * N);
#pragma unroll
    for (int i = 0; i < P; ++i) h[i] = fma2(ex2x2(mul2(dl2, A2[i])), h[i], mul2(du2, Bv[i]));
    sd += dl;
  }
  }
#pragma unroll
  for (int i = 0; i < P; ++i) {
    sm.aggH[(s * N + 2 * i) * kTile + lane] = h[i].x;
    sm.aggH[(s * N + 2 * i + 1) * kTile + lane] = h[i].y;
  }
  sm.aggSD[s * kTile + lane] = sd;
  if (lane == 0) sm.aggRS[s] = rs;
  __syncthreads();

  // ---- steps 4-5, per warp: warp s owns the state chains n = s (and s + kS
  //      when N = 16); with N = 4 only warps 0-3 own one.  For each of its
  //      states it runs the exclusive scan over the 8 sub-chunk aggregates,
  //      then the decoupled look-back across chunks on its own chain.  Each
  //      (chunk, state, channel) word of the inclusive array holds kCarryUnset
  //      until its value is stored (the call fills the array before the
  //      launch), so a word is its own flag: no fence, and no flag for the
  //      common case.  Only the aggregate of a chunk, published when a walk
  //      must go past it, is announced by the warp's flag after a fence.
  int next = 0;  // thread 0: the next ticket, stored for every warp before pass 2
  if (tid == 0) next = (int)atomicAdd(a.ticket, 1u);
  constexpr bool kTwo = N > kS;     // two states per warp
  const bool own = s < N;           // the warp owns at least one state
  const int n0 = s, n1 = kTwo ? s + kS : s;
  const bool need_in = chunk > 0 && pos_at(0) != 0;  // a state enters from the previous chunk
  const int64_t base = (int64_t)tile * a.n_chunks;
  // the chain word of state n for chunk j, this lane's channel
  auto word = [&](int64_t j, int n) { return (base + j) * (N * kTile) + n * kTile + lane; };
  // early look at the previous chunk's inclusive state: that chunk started
  // long before this one and has nearly always stored it by now; the loads
  // land during the scan below
  float2 early = make_float2(0.0f, 0.0f);
  if (own && need_in) {
    early.x = ld_carry1(a.incl + word(chunk - 1, n0));
    if (kTwo) early.y = ld_carry1(a.incl + word(chunk - 1, n1));
  }
  if (own) {
    float sdj[kS];
    int rsj[kS];
    int rs_any = 0;
    float sd_tot = 0.0f;
#pragma unroll
    for (int j = 0; j < kS; ++j) {
      sdj[j] = sm.aggSD[j * kTile + lane];
      rsj[j] = sm.aggRS[j];
      rs_any |= rsj[j];
      sd_tot += sdj[j];
    }
    // A*log2e of the warp's states, picked with compile-time register indices
    float2 a2w = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < P; ++i) {
      if (2 * i == n0) a2w.x = A2[i].x;
      if (2 * i + 1 == n0) a2w.x = A2[i].y;
      if (2 * i == n1) a2w.y = A2[i].x;
      if (2 * i + 1 == n1) a2w.y = A2[i].y;
    }
    // exclusive scan per state; the chunk's totals, the prefixes and the
    // sub-chunks' factors stay in registers until the entering state is known
    float2 tot = make_float2(0.0f, 0.0f);
    float Pj[2][kS], Ej[2][kS];
#pragma unroll
    for (int q = 0; q < (kTwo ? 2 : 1); ++q) {
      const int n = q ? n1 : n0;
      const float a2 = q ? a2w.y : a2w.x;
      float Hj[kS];
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        Pj[q][j] = rsj[j] ? 0.0f : ex2(a2 * sdj[j]);
        Hj[j] = sm.aggH[(j * N + n) * kTile + lane];
      }
      float x = 0.0f;
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        Ej[q][j] = x;
        x = fmaf(Pj[q][j], x, Hj[j]);
      }
      if (q) tot.y = x;
      else tot.x = x;
    }
    const bool publish = (long long)tk != a.drop_ticket;
    int* const my_flag = a.flags + (base + chunk) * kS + s;
    auto store_incl = [&](float2 v) {
      st_carry1(a.incl + word(chunk, n0), v.x);
      if (kTwo) st_carry1(a.incl + word(chunk, n1), v.y);
    };
    // a sequence starts in this chunk: the state leaving it does not depend
    // on the state entering, store it at once
    if (rs_any && publish) store_incl(tot);
    float2 x = make_float2(0.0f, 0.0f);
    if (need_in) {
      int j = chunk - 1, found = -1, timed_out = 0;
      float2 v = early;
      if (__all_sync(0xffffffffu, carry_set1(v.x) && (!kTwo || carry_set1(v.y)))) {
        found = j;
      } else {
        if (!rs_any) {
          // publish this chunk's aggregate for walks that must go past it;
          // every warp stores the same sum of delta, its flag covers its own
          a.agg[word(chunk, n0)] = tot.x;
          if (kTwo) a.agg[word(chunk, n1)] = tot.y;
          a.agg_sd[(base + chunk) * kTile + lane] = sd_tot;
          fence_acq_rel_gpu();
          __syncwarp();
          if (lane == 0 && publish) st_relaxed_gpu(my_flag, kFlagAggregate);
        }
        const uint64_t t_start = globaltimer_ns();
        while (j >= 0) {
          // wait for chunk j: its inclusive words, or its aggregate flag
          unsigned backoff = 32;
          int f = kFlagNone;
          for (;;) {
            v.x = ld_carry1(a.incl + word(j, n0));
            if (kTwo) v.y = ld_carry1(a.incl + word(j, n1));
            if (__all_sync(0xffffffffu, carry_set1(v.x) && (!kTwo || carry_set1(v.y)))) {
              f = kFlagInclusive;
              break;
            }
            if (__all_sync(0xffffffffu, ld_acquire_gpu(a.flags + (base + j) * kS + s) == kFlagAggregate)) {
              f = kFlagAggregate;
              break;
            }
            if (__shfl_sync(0xffffffffu, globaltimer_ns() - t_start > a.wait_ns, 0)) break;
            __nanosleep(backoff);
            if (backoff < 1024) backoff <<= 1;
          }
          if (f == kFlagInclusive) { found = j; break; }
          if (f == kFlagNone) { timed_out = 1; break; }
          --j;
        }
      }
      if (timed_out) atomicOr(a.status, kStatusLookbackTimeout);
      // forward re-evaluation from the nearest inclusive state, in chunk order
      int first = j + 1;
      if (found >= 0) {
        x = v;
        first = found + 1;
      }
      for (int i = first; i < chunk; ++i) {
        const float sdi = __ldcg(a.agg_sd + (base + i) * kTile + lane);
        x.x = fmaf(ex2(a2w.x * sdi), x.x, __ldcg(a.agg + word(i, n0)));
        if (kTwo) x.y = fmaf(ex2(a2w.y * sdi), x.y, __ldcg(a.agg + word(i, n1)));
      }
    }
    // stored at once: the next chunk of the tile may already be waiting
    if (!rs_any && publish)
      store_incl(make_float2(fmaf(ex2(a2w.x * sd_tot), x.x, tot.x), fmaf(ex2(a2w.y * sd_tot), x.y, tot.y)));
    // the exact state each sub-chunk starts from: its prefix plus the entering
    // state carried over the sub-chunks before it (their factors' product, 0
    // past a sequence start)
#pragma unroll
    for (int q = 0; q < (kTwo ? 2 : 1); ++q) {
      const int n = q ? n1 : n0;
      const float xin = q ? x.y : x.x;
      float pp = 1.0f;
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        sm.aggH[(j * N + n) * kTile + lane] = fmaf(pp, xin, Ej[q][j]);
        pp *= Pj[q][j];
      }
    }
  }
  // every thread has read this item's ticket at the top of the loop
  if (tid == 0) sm.ticket = next;
  __syncthreads();

  // ---- step 6: exact start state, pass 2
  // with two buffers, each warp requests its share of the next item's inputs
  // halfway through its pass 2: the single buffers (delta_raw, A rows,
  // dt_bias, Dskip) were read before pass 2, the other buffer set by the
  // item before this one
  bool issued = false;
  auto issue_next = [&]() {
    if (kNB == 2 && lane == 0 && !issued) {
      issue(sm.ticket, buf ^ 1, s);
      issued = true;
    }
  };
#pragma unroll
  for (int i = 0; i < P; ++i)
    h[i] = make_float2(sm.aggH[(s * N + 2 * i) * kTile + lane], sm.aggH[(s * N + 2 * i + 1) * kTile + lane]);
  const int64_t ts = t0 + tb;
  if (a.chunk_states && valid && ts < a.T && (ts % kStateChunk) == 0) {
    // layout [chunk][n][d]: the 32 lanes store 32 consecutive floats per state
    float* cs = a.chunk_states + (ts / kStateChunk) * N * a.D + d;
#pragma unroll
    for (int i = 0; i < P; ++i) {
      cs[(2 * i) * (int64_t)a.D] = h[i].x;
      cs[(2 * i + 1) * (int64_t)a.D] = h[i].y;
    }
  }

  T* out = static_cast<T*>(a.out);
  T* ypre = static_cast<T*>(a.y);  // the output before the gate (nullable)
  if (whole) {
    const T* const up = su + tb * kTile + lane;
    const T* const zp = sz + tb * kTile + lane;
    const float* const dlp = sm.dlt + tb * kTile + lane;
    const float* const bp = Bf + tb * N;
    const float* const cp = Cf + tb * N;
    T* op = out + (t0 + tb) * a.D + d;
    T* yp = ypre ? ypre + (t0 + tb) * a.D + d : nullptr;
#pragma unroll 1  // groups of 8 tokens, as in pass 1
    for (int kg = 0; kg < kK; kg += 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = kg + e;
      if ((rm >> k) & 1u) {
        // the previous token ended a sequence (a token of this warp's when k > 0;
        // the warp before stores its own last token's state)
        if constexpr (kStates) {
          if (a.h_final && k > 0) end_state(h, tb + k - 1);
        }
        start_state(h, tb + k);
      }
      const float dl = dlp[k * kTile];
      const float uu = to_f(up[k * kTile]);
      const float2 dl2 = splat2(dl), du2 = splat2(dl * uu);
      float2 Bv[P], Cv[P];
      lds_pairs<N>(Bv, bp + k * N);
      lds_pairs<N>(Cv, cp + k * N);
      float2 y2 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int i = 0; i < P; ++i) {
        h[i] = fma2(ex2x2(mul2(dl2, A2[i])), h[i], mul2(du2, Bv[i]));
        y2 = fma2(Cv[i], h[i], y2);
      }
      float y = fmaf(Dsk, uu, y2.x + y2.y);
      if (yp) {
        if (valid) *yp = from_f<T>(y);
        yp += a.D;
      }
      if (a.has_z) y *= siluf(to_f(zp[k * kTile])) + a.gate_floor;
      if (valid) *op = from_f<T>(y);
      op += a.D;
    }
    if (kg == 0) issue_next();
    }
    if constexpr (kStates) {
      if (a.h_final && seq_end(tb + kK - 1)) end_state(h, tb + kK - 1);
    }
  } else {
#pragma unroll 1  // ragged tails and narrow tiles only: kept small for the instruction cache
  for (int k = 0; k < kK; ++k) {
    const int t = tb + k;
    if (t >= rows) break;
    if (pos_at(t) == 0) start_state(h, t);
    const float dl = sm.dlt[t * kTile + lane];
    const float uu = to_f(su[t * bx + lane]);
    const float2 dl2 = splat2(dl), du2 = splat2(dl * uu);
    float2 Bv[P], Cv[P];
    lds_pairs<N>(Bv, Bf + t * N);
    lds_pairs<N>(Cv, Cf + t * N);
    float2 y2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < P; ++i) {
      h[i] = fma2(ex2x2(mul2(dl2, A2[i])), h[i], mul2(du2, Bv[i]));
      y2 = fma2(Cv[i], h[i], y2);
    }
    float y = fmaf(Dsk, uu, y2.x + y2.y);
    if (ypre && valid) ypre[(t0 + t) * a.D + d] = from_f<T>(y);
    if (a.has_z) y *= siluf(to_f(sz[t * bx + lane])) + a.gate_floor;
    if (valid) out[(t0 + t) * a.D + d] = from_f<T>(y);
    if constexpr (kStates) {
      if (a.h_final && seq_end(t)) end_state(h, t);
    }
  }
  }

  if constexpr (kNB == 2) {
    issue_next();  // the ragged paths: at the end of pass 2
  } else {
    // every input of this item has been read: request the next one's
    __syncthreads();
    if (lane == 0) issue(sm.ticket, 0, s);
  }
  }  // persistent loop
}

template <typename T, int N, bool kStates, bool kKnob = false, bool kConv = false>
cudaError_t launch_k(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, cudaStream_t st) {
  auto kern = scan_fwd_kernel<T, N, kStates, kKnob, kConv>;
  const size_t smem = sizeof(FwdSmem<T, N, kConv>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.n_chunks * a.n_tiles;
  int grid = 0;
  e = persistent_grid(kern, kThreads, smem, items, &grid);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(tm_u, tm_dr, tm_z, a);
  return cudaGetLastError();
}

template <typename T, int N>
cudaError_t launch_n(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, cudaStream_t st) {
  if (a.conv_w)  // the fused conv1d + scan forward
    return a.seq ? launch_k<T, N, true, false, true>(a, tm_u, tm_dr, tm_z, st)
                 : launch_k<T, N, false, false, true>(a, tm_u, tm_dr, tm_z, st);
  if constexpr (sizeof(T) == 4 && N == 16) {  // the delay knob's instantiation
    if (a.delay_ticket >= 0 && !a.seq) return launch_k<T, N, false, true>(a, tm_u, tm_dr, tm_z, st);
  }
  return a.seq ? launch_k<T, N, true>(a, tm_u, tm_dr, tm_z, st) : launch_k<T, N, false>(a, tm_u, tm_dr, tm_z, st);
}

template <typename T>
cudaError_t launch_t(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, cudaStream_t st) {
  if (a.N == 16) return launch_n<T, 16>(a, tm_u, tm_dr, tm_z, st);
  if (a.N == 8) return launch_n<T, 8>(a, tm_u, tm_dr, tm_z, st);
  if constexpr (sizeof(T) == 4) {
    if (a.N == 4) return launch_n<T, 4>(a, tm_u, tm_dr, tm_z, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_scan_fwd(const ScanArgs& a, IO io, const CUtensorMap& tm_u,
                            const CUtensorMap& tm_dr, const CUtensorMap& tm_z, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  if (!a.Af) return cudaErrorInvalidValue;
  cudaError_t pe = launch_prep_a(a.A, a.D, a.N, a.a_log != 0, const_cast<float4*>(a.Af), st);
  if (pe != cudaSuccess) return pe;
  if (io == IO::BF16) {  // every work item then copies fp32 B and C rows as they are
    if (!a.Bf32 || !a.Cf32) return cudaErrorInvalidValue;
    cudaError_t e = launch_widen_bf16(a.B, const_cast<float*>(a.Bf32), a.T * a.N, st);
    if (e == cudaSuccess) e = launch_widen_bf16(a.C, const_cast<float*>(a.Cf32), a.T * a.N, st);
    if (e != cudaSuccess) return e;
  }
  kernel_timer_mark(kTimeScanFwd, true, st);
  const cudaError_t e = io == IO::F32 ? launch_t<float>(a, tm_u, tm_dr, tm_z, st)
                                      : launch_t<__nv_bfloat16>(a, tm_u, tm_dr, tm_z, st);
  kernel_timer_mark(kTimeScanFwd, false, st);
  return e;
}

}  // namespace vssm
