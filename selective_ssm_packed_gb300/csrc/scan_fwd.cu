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
//      shared memory.
//   5. Decoupled look-back across chunks (warp 0): publish the chunk aggregate
//      (or, if a sequence starts inside the chunk, the inclusive state at once),
//      walk back over predecessors' flags to the nearest inclusive state, then
//      re-apply the aggregates FORWARD from there in chunk order, which gives
//      the same floating-point result whatever the timing (bitwise repeatable).
//      Work items take chunk ids from an atomic ticket, so a CTA only ever waits
//      on items already running; every wait is time-bounded and a timeout is
//      reported through the status word instead of hanging.
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

template <typename T, int N>
struct FwdSmem {
  alignas(128) T u[kL * kTile];
  alignas(128) T dr[kL * kTile];
  alignas(128) T z[kL * kTile];
  alignas(128) T B[kL * N];
  alignas(128) T C[kL * N];
  // B and C widened to fp32 once per work item (bf16 I/O only)
  alignas(16) float Bf[sizeof(T) == 2 ? kL * N : 4];
  alignas(16) float Cf[sizeof(T) == 2 ? kL * N : 4];
  alignas(16) float dlt[kL * kTile];
  alignas(16) float aggH[kS * N * kTile];
  float totH[N * kTile];
  float hin[N * kTile];
  float aggSD[kS * kTile];
  alignas(16) float Araw[kTile * N];  // A rows d0 .. d0+31
  alignas(16) float bias[kTile];
  alignas(16) float dsk[kTile];
  alignas(16) int pos[kL];
  int aggRS[kS];
  int ticket;
  alignas(8) uint64_t bar;
};

// kStates: the call passes sequence states (initial and/or final); without
// them the kernel carries no code for them.
template <typename T, int N, bool kStates>
__global__ void __launch_bounds__(kThreads, 2)
scan_fwd_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dr,
                const __grid_constant__ CUtensorMap tm_z, const ScanArgs a) {
  using SM = FwdSmem<T, N>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, s = tid >> 5;

  const int n_items = a.n_chunks * a.n_tiles;

  // Requests every input of work item `tkn` on the barrier: u, delta_raw, z
  // tiles; B and C rows; A rows, dt_bias, Dskip; position indices (whole
  // groups of 4 tokens).  With no item left, thread 0 arrives without data so
  // that the barrier still completes and tells every thread to stop.
  auto issue = [&](int tkn) {
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
    const uint32_t bc = (uint32_t)nrows * N * sizeof(T);
    const uint32_t rows4 = (uint32_t)nrows & ~3u;
    const uint32_t box = (uint32_t)a.box_x * (uint32_t)a.box_y * sizeof(T);
    mbar_arrive_expect_tx(&sm.bar, box * (a.has_z ? 3u : 2u) + 2u * bc + nval * N * 4u + rows4 * 4u +
                                       (a.dt_bias ? nval * 4u : 0u) + (a.Dskip ? nval * 4u : 0u));
    tma_load_2d(sm.u, &tm_u, dd0, (int)tt0, &sm.bar);
    tma_load_2d(sm.dr, &tm_dr, dd0, (int)tt0, &sm.bar);
    if (a.has_z) tma_load_2d(sm.z, &tm_z, dd0, (int)tt0, &sm.bar);
    bulk_load_1d(sm.B, static_cast<const T*>(a.B) + tt0 * N, bc, &sm.bar);
    bulk_load_1d(sm.C, static_cast<const T*>(a.C) + tt0 * N, bc, &sm.bar);
    bulk_load_1d(sm.Araw, a.A + (int64_t)dd0 * N, nval * N * 4u, &sm.bar);
    if (a.dt_bias) bulk_load_1d(sm.bias, a.dt_bias + dd0, nval * 4u, &sm.bar);
    if (a.Dskip) bulk_load_1d(sm.dsk, a.Dskip + dd0, nval * 4u, &sm.bar);
    if (rows4) bulk_load_1d(sm.pos, a.pos + tt0, rows4 * 4u, &sm.bar);
  };

  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
    const int first = (int)atomicAdd(a.ticket, 1u);
    sm.ticket = first;
    issue(first);
  }
  __syncthreads();

  // Persistent loop: one work item per pass.  The inputs are read until the
  // end of pass 2, so the next ticket is drawn and its copies requested there;
  // an earlier draw would hold tickets back from the look-back chains (an
  // item whose neighbour sits reserved behind a running item waits for both).
  // Items only ever wait on items with smaller tickets, all of which are done
  // or in hand of a running CTA, so the loop cannot deadlock.
  for (uint32_t it = 0;; ++it) {
  // the barrier's completion also publishes thread 0's write of sm.ticket
  if (!__syncthreads_and(mbar_wait(&sm.bar, it & 1u, a.wait_ns))) {
    if (tid == 0) atomicOr(a.status, kStatusTmaTimeout);
    break;
  }
  const int tk = sm.ticket;
  if (tk >= n_items) break;
  const int chunk = tk / a.n_tiles;
  const int tile = tk - chunk * a.n_tiles;
  const int64_t t0 = (int64_t)chunk * kL;
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
  auto pos_at = [&](int t) { return t < rows4 ? sm.pos[t] : __ldg(a.pos + t0 + t); };
  // the state a sequence starting at token t (of the chunk) starts from: its
  // row of the initial states, or zero
  auto start_state = [&](float2 (&hs)[N / 2], int t) {
    if (kStates && a.h_init && valid) {
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
    if (valid) {
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
  // B and C rows of this warp's own tokens, widened to fp32 by the warp: no
  // other warp reads them, so a warp barrier is enough
  const int wr0 = tb < rows ? tb : rows, wr1 = tb + kK < rows ? tb + kK : rows;
  const float* Bf = widen_rows<T>(sm.B + wr0 * N, sm.Bf + wr0 * N, (wr1 - wr0) * N, lane, 32) - wr0 * N;
  const float* Cf = widen_rows<T>(sm.C + wr0 * N, sm.Cf + wr0 * N, (wr1 - wr0) * N, lane, 32) - wr0 * N;
  __syncwarp();
  float2 A2[P];
  if (valid) {
    load_row_pairs_rotated<N>(A2, sm.Araw + lane * N, lane, a.a_log ? 1.0f : kLog2e);
    if (a.a_log) {
      // the rows hold A_log: A = -exp(A_log), kept scaled by log2 e for ex2
#pragma unroll
      for (int i = 0; i < P; ++i)
        A2[i] = make_float2(-ex2(A2[i].x * kLog2e) * kLog2e, -ex2(A2[i].y * kLog2e) * kLog2e);
    }
  } else {
#pragma unroll
    for (int i = 0; i < P; ++i) A2[i] = make_float2(0.0f, 0.0f);
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
    const T* const up = sm.u + tb * kTile + lane;
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
    const float2 dl2 = splat2(dl), du2 = splat2(dl * to_f(sm.u[t * bx + lane]));
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

  // Warp 0 acquires the previous chunk's flag and reads its inclusive state
  // now; the loads land during the scan below.  (That chunk started long
  // before this one: its state is nearly always published by now.  The reads
  // follow the acquire in program order, so they see what the flag publishes.)
  int early_f = kFlagNone;
  float early_x[N];
  if (s == 0 && chunk > 0 && pos_at(0) != 0) {
    const int64_t jslot = (int64_t)tile * a.n_chunks + chunk - 1;
    early_f = ld_acquire_gpu(a.flags + jslot * kTile + lane);
    const float* inc = a.incl + jslot * (N * kTile);
#pragma unroll
    for (int n = 0; n < N; ++n) early_x[n] = __ldcg(inc + n * kTile + lane);
  }

  // ---- step 4: exclusive scan over sub-chunks; chain (lane, n) with n % kS == s
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
      float Pj[kS], Hj[kS];
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        Pj[j] = rsj[j] ? 0.0f : ex2(a2 * sdj[j]);
        Hj[j] = sm.aggH[(j * N + n) * kTile + lane];
      }
      float x = 0.0f;
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        sm.aggH[(j * N + n) * kTile + lane] = x;
        x = fmaf(Pj[j], x, Hj[j]);
      }
      sm.totH[n * kTile + lane] = x;
    }
  }
  __syncthreads();

  // ---- step 5: decoupled look-back (warp 0)
  bool release_incl = false;  // warp 0: inclusive state stored, flag not yet released
  if (s == 0) {
    int rs_any = 0;
    float sd_tot = 0.0f;
#pragma unroll
    for (int j = 0; j < kS; ++j) {
      rs_any |= sm.aggRS[j];
      sd_tot += sm.aggSD[j * kTile + lane];
    }
    const int64_t slot = (int64_t)tile * a.n_chunks + chunk;
    const bool publish = (long long)tk != a.drop_ticket;
    float* my_agg = a.agg + slot * (N * kTile);
    float* my_inc = a.incl + slot * (N * kTile);
    // every lane is its own chain (one channel): it publishes its payload and
    // then its own flag with a release store, and readers acquire that flag
    int* my_flag = a.flags + slot * kTile + lane;
    if (rs_any) {
      // a sequence starts in this chunk: the state leaving it does not depend
      // on the state entering, publish it at once
#pragma unroll
      for (int n = 0; n < N; ++n) my_inc[n * kTile + lane] = sm.totH[n * kTile + lane];
      if (publish) st_release_gpu(my_flag, kFlagInclusive);
    }
    float x[N];
#pragma unroll
    for (int n = 0; n < N; ++n) x[n] = 0.0f;
    // no entering state is needed when a sequence starts at the first token
    if (chunk > 0 && pos_at(0) != 0) {
      // the previous chunk of the tile started long before this one and has
      // usually published its inclusive state: look first, and publish this
      // chunk's aggregate only when the walk has to go further
      const int64_t base = (int64_t)tile * a.n_chunks;
      int j = chunk - 1, found = -1, timed_out = 0;
      bool have_x = false;
      if (early_f == kFlagInclusive) {
        found = j;
        have_x = true;
#pragma unroll
        for (int n = 0; n < N; ++n) x[n] = early_x[n];
      } else if (ld_acquire_gpu(a.flags + (base + j) * kTile + lane) == kFlagInclusive) {
        found = j;
      } else {
        if (!rs_any) {
#pragma unroll
          for (int n = 0; n < N; ++n) my_agg[n * kTile + lane] = sm.totH[n * kTile + lane];
          a.agg_sd[slot * kTile + lane] = sd_tot;
          if (publish) st_release_gpu(my_flag, kFlagAggregate);
        }
        while (j >= 0) {
          const int f = wait_flag(a.flags + (base + j) * kTile + lane, a.wait_ns);
          if (f == kFlagInclusive) { found = j; break; }
          if (f == kFlagNone) { timed_out = 1; break; }
          --j;
        }
      }
      if (timed_out) atomicOr(a.status, kStatusLookbackTimeout);
      int first = j + 1;
      if (found >= 0) {
        if (!have_x) {
          const float* inc = a.incl + (base + found) * (N * kTile);
#pragma unroll
          for (int n = 0; n < N; ++n) x[n] = __ldcg(inc + n * kTile + lane);
        }
        first = found + 1;
      }
      for (int i = first; i < chunk; ++i) {
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
    for (int n = 0; n < N; ++n) sm.hin[n * kTile + lane] = x[n];
    if (!rs_any) {
      // payload now, flag after the barrier below, when these stores have drained
#pragma unroll
      for (int n = 0; n < N; ++n) {
        const float a2 = (n & 1) ? A2[n / 2].y : A2[n / 2].x;
        my_inc[n * kTile + lane] = fmaf(ex2(a2 * sd_tot), x[n], sm.totH[n * kTile + lane]);
      }
      release_incl = publish;
    }
  }
  __syncthreads();
  if (release_incl)
    st_release_gpu(a.flags + ((int64_t)tile * a.n_chunks + chunk) * kTile + lane, kFlagInclusive);

  // ---- step 6: exact start state, pass 2
  int rs_pre = 0;
  float sd_pre = 0.0f;
  for (int j = 0; j < s; ++j) {
    rs_pre |= sm.aggRS[j];
    sd_pre += sm.aggSD[j * kTile + lane];
  }
#pragma unroll
  for (int i = 0; i < P; ++i) {
    const float2 E = make_float2(sm.aggH[(s * N + 2 * i) * kTile + lane], sm.aggH[(s * N + 2 * i + 1) * kTile + lane]);
    const float2 R = make_float2(sm.hin[(2 * i) * kTile + lane], sm.hin[(2 * i + 1) * kTile + lane]);
    h[i] = rs_pre ? E : fma2(ex2x2(mul2(A2[i], splat2(sd_pre))), R, E);
  }
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
    const T* const up = sm.u + tb * kTile + lane;
    const T* const zp = sm.z + tb * kTile + lane;
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
    const float uu = to_f(sm.u[t * bx + lane]);
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
    if (a.has_z) y *= siluf(to_f(sm.z[t * bx + lane])) + a.gate_floor;
    if (valid) out[(t0 + t) * a.D + d] = from_f<T>(y);
    if constexpr (kStates) {
      if (a.h_final && seq_end(t)) end_state(h, t);
    }
  }
  }

  // every input of this item has been read: draw the next one
  __syncthreads();
  if (tid == 0) {
    const int next = (int)atomicAdd(a.ticket, 1u);
    sm.ticket = next;
    issue(next);
  }
  }  // persistent loop
}

template <typename T, int N, bool kStates>
cudaError_t launch_k(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, cudaStream_t st) {
  const size_t smem = sizeof(FwdSmem<T, N>);
  cudaError_t e = cudaFuncSetAttribute(scan_fwd_kernel<T, N, kStates>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.n_chunks * a.n_tiles;
  int grid = 0;
  e = persistent_grid(scan_fwd_kernel<T, N, kStates>, kThreads, smem, items, &grid);
  if (e != cudaSuccess) return e;
  scan_fwd_kernel<T, N, kStates><<<grid, kThreads, smem, st>>>(tm_u, tm_dr, tm_z, a);
  return cudaGetLastError();
}

template <typename T, int N>
cudaError_t launch_n(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, cudaStream_t st) {
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
  return io == IO::F32 ? launch_t<float>(a, tm_u, tm_dr, tm_z, st)
                       : launch_t<__nv_bfloat16>(a, tm_u, tm_dr, tm_z, st);
}

}  // namespace vssm
