// scan_bwd.cu -- packed selective scan, backward (sm_103a).
//
// Work item = (chunk of kBwdChunk = 32 tokens, the saved-state granule) x
// (tile of kTile = 32 channels); items are taken in DESCENDING chunk order
// from an atomic ticket because the state gradient flows from the end of a
// sequence to its start.  The kernel is persistent (one CTA per resident slot,
// looping over tickets); one thread requests each item's inputs with tensor /
// bulk copies on one mbarrier while the previous item finishes.
//
// CTA = N/2 warps.  Warp w owns the state pair (2w, 2w+1) for ALL 32 tokens
// of the item, lane l owns channel d0 + l.  The forward states therefore need
// no scan inside the CTA: every warp starts from the saved state of the chunk
// (chunk_states, written by the forward call) and walks its 32 tokens.
//
// With a_t = exp(delta_t A) (0 at a sequence start), b_t = delta_t u_t B_t,
// g_t = dout_t (SiLU(z_t) + gate floor):
//   h_t  = a_t h_{t-1} + b_t                       (forward walk)
//   dh_t = C_t g_t + a_{t+1} dh_{t+1}              (reverse walk; a_{t+1} = 0
//                                                   at a sequence start, so the
//                                                   scan resets at sequence ends)
// The carry handed to the previous chunk is a_{t0} dh_{t0} = sum_t E_t C_t g_t
// + E_last * (carry from the next chunk), with E_t = a_{t0} ... a_t: both terms
// are accumulated during the FORWARD walk, so the look-back needs no extra
// pass and no extra exponential.
//
//   1. Per-(token, channel) values once per item, by all threads: delta,
//      delta u, g, d delta / d delta_raw, in [channel][token] arrays; B and C
//      transposed to [state][token] (fp32).
//   2. Forward walk per warp: states h_t kept in registers (32 tokens x 2
//      states); E and the carry aggregate accumulated; dC_t[n] contributions
//      g_t h_t summed over the tile's channels (ColSum16 shuffle butterflies,
//      fed token by token); C_t.h_t partials for y.
//   3. Decoupled look-back per warp towards HIGHER chunks for the carry
//      entering from the right; aggregates re-applied in a fixed order
//      (bitwise repeatable); time-bounded waits.  An inclusive carry is its
//      own flag (the carry array starts filled with a NaN word that no
//      stored value equals), so it is stored and read with no fence; only an
//      aggregate is announced by a flag, behind a fence.
//   4. Reverse walk per warp in blocks of 8 tokens: dA (per thread), dB
//      contributions (ColSum16), partial sums over the warp's states
//      for du and d delta; after each block all threads add the warps'
//      partials in a fixed order and write du, d delta_raw and dz (with
//      y = the forward's pre-gate output when the call passes it, else the
//      warps' C.h partials + Dskip u).
//   5. dA partials per chunk; fixed-order CTA sums for dDskip, d_dt_bias.
// Separate fixed-order kernels sum the partials over channel tiles (dB, dC)
// and chunks (dA, dDskip, d_dt_bias).  No atomics anywhere in the arithmetic.
#include "common.cuh"
#include "kernels.h"

namespace vssm {

namespace {

constexpr int kL = kBwdChunk;   // 32 tokens per work item
constexpr int kP = kL + 4;      // row pitch of the [channel][token] arrays
constexpr int kPP = kL + 2;     // token pitch (in pairs) of the paired B / C arrays
constexpr int kRB = 8;          // tokens per block of the reverse walk
constexpr float kLn2 = 0.6931471805599453f;

template <typename T, int N>
struct BwdSmem {
  static constexpr int W = N / 2;  // warps = state pairs
  // ---- inputs of one work item, written by tensor / bulk copies and refilled
  //      for the next item once this one has read them for the last time
  alignas(128) T u[kL * kTile];
  alignas(128) T dr[kL * kTile];
  alignas(128) T z[kL * kTile];
  alignas(128) T dout[kL * kTile];
  alignas(128) T y[kL * kTile];  // the forward's pre-gate output, when the call has it
  alignas(128) T B[kL * N];
  alignas(128) T C[kL * N];
  alignas(16) float Araw[kTile * N];  // A rows d0 .. d0+31
  alignas(128) float H[N * kTile];    // saved states at the chunk start, [n][channel]
  alignas(16) float bias[kTile];
  alignas(16) float dsk[kTile];
  alignas(16) int pos[kL];
  // ---- per-(token, channel) values, [channel][token] with pitch kP: a lane
  //      reads 4 tokens of its channel with one conflict-free 16-byte access
  alignas(16) float dl[kTile * kP];   // delta
  alignas(16) float dlu[kTile * kP];  // delta * u
  alignas(16) float g[kTile * kP];    // dout * SiLU(z)
  alignas(16) float sg[kTile * kP];   // d delta / d delta_raw
  // ---- B, C paired per warp, fp32 (zero past the last token): entry
  //      [o][w][t] of BP is (B_t[2w], B_t[2w+1]) for o = 0 and the swapped
  //      pair for o = 1, so a lane loads its state pair, in its own order,
  //      for 2 tokens with one 16-byte access and feeds it to the paired FP32
  //      instructions as loaded; the pitch kPP keeps the stores conflict-free
  alignas(16) float BP[2 * W * kPP * 2];
  alignas(16) float CP[2 * W * kPP * 2];
  // ---- exponent offset per token: -inf at a sequence start, else 0
  alignas(16) float off[kL];
  // ---- cross-warp partials: C.h of each warp's state pair [W][kL][kTile]
  //      from the forward walk, and (du, d delta) partials
  //      [2][W][kRB][kTile] float2 from each block of the reverse walk
  alignas(16) float ypart[W * kL * kTile];
  alignas(16) float part[W * kL * kTile];
  float redD[W * kTile];
  float redB[W * kTile];
  int ticket;
  alignas(8) uint64_t bar;
};

// Column sums over the 32 lanes of a warp (lane = channel) for groups of 16
// tokens x 2 states, fed one token at a time by shuffle butterflies.  A lane
// keeps its state pair in its own order, the "first" state being n0 + bit4:
//   level 1 (every token): lanes l, l^16 exchange the state the other keeps,
//   level 2 (every token pair): lanes l, l^8 exchange the token the other
//     keeps (bit 3 picks the odd token),
//   levels 3, 4, 5 likewise over lane bits 2, 1, 0 for pairs of pairs, ...
// After the 16th token, lane l holds the sum over all 32 lanes for token
// 8 b0 + 4 b1 + 2 b2 + b3 of the group (b_i = bit i of l) and its first
// state.  The pairing is fixed, so the sums are bitwise repeatable; tokens may
// come in ascending or descending order.
struct ColSum16 {
  float p1[2], p2[2], p3[2], p4[2];  // pending sums, by the parity of the token group at each level

  static __device__ __forceinline__ int token(int lane) {
    return 8 * (lane & 1) + 4 * ((lane >> 1) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 3) & 1);
  }

  static __device__ __forceinline__ float combine(float lo, float hi, int lane, int mask) {
    const bool up = (lane & mask) != 0;
    return (up ? hi : lo) + __shfl_xor_sync(0xffffffffu, up ? lo : hi, mask);
  }

  // Token c (0..15) of the group with this lane's values in its state order;
  // returns true once the group is complete (*sum then holds the lane's result).
  __device__ __forceinline__ bool feed(int c, bool ascending, float2 v, int lane, float* sum) {
    p1[c & 1] = v.x + __shfl_xor_sync(0xffffffffu, v.y, 16);
    if ((c & 1) != (ascending ? 1 : 0)) return false;
    p2[(c >> 1) & 1] = combine(p1[0], p1[1], lane, 8);
    if ((c & 3) != (ascending ? 3 : 0)) return false;
    p3[(c >> 2) & 1] = combine(p2[0], p2[1], lane, 4);
    if ((c & 7) != (ascending ? 7 : 0)) return false;
    p4[(c >> 3) & 1] = combine(p3[0], p3[1], lane, 2);
    if ((c & 15) != (ascending ? 15 : 0)) return false;
    *sum = combine(p4[0], p4[1], lane, 1);
    return true;
  }
};

// Publishes a warp's look-back payload: every lane has stored its part; the
// fence orders each lane's stores before the barrier, and lane 0 then sets the
// warp's flag.
__device__ __forceinline__ void publish_flag(int* flag, int value, bool publish, int lane) {
  fence_acq_rel_gpu();
  __syncwarp();
  if (lane == 0 && publish) st_relaxed_gpu(flag, value);
}

// kStates: the call passes sequence states (initial states, final-state or
// starting-state gradients); without them the kernel carries no code for them.
template <typename T, int N, bool kStates, bool kKnob>
__global__ void __launch_bounds__(16 * N, 512 / (16 * N))
scan_bwd_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dr,
                const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_dout,
                const __grid_constant__ CUtensorMap tm_cs, const __grid_constant__ CUtensorMap tm_y,
                const ScanArgs a) {
  using SM = BwdSmem<T, N>;
  constexpr int W = SM::W;
  constexpr int kThr = 32 * W;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int n_items = a.n_chunks * a.n_tiles;

  // Requests every input of work item `tkn` on the barrier: u, delta_raw,
  // dout, z (and y) tiles; B and C rows; A rows, dt_bias, Dskip and the saved states
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
    mbar_arrive_expect_tx(&sm.bar, box * (3u + (a.has_z ? 1u : 0u) + (a.has_y ? 1u : 0u)) + 2u * bc + nval * N * 4u +
                                       (uint32_t)a.box_x * N * 4u + rows4 * 4u +
                                       (a.dt_bias ? nval * 4u : 0u) + (a.Dskip ? nval * 4u : 0u));
    tma_load_2d(sm.u, &tm_u, dd0, (int)tt0, &sm.bar);
    tma_load_2d(sm.dr, &tm_dr, dd0, (int)tt0, &sm.bar);
    tma_load_2d(sm.dout, &tm_dout, dd0, (int)tt0, &sm.bar);
    if (a.has_z) tma_load_2d(sm.z, &tm_z, dd0, (int)tt0, &sm.bar);
    if (a.has_y) tma_load_2d(sm.y, &tm_y, dd0, (int)tt0, &sm.bar);
    bulk_load_1d(sm.B, static_cast<const T*>(a.B) + tt0 * N, bc, &sm.bar);
    bulk_load_1d(sm.C, static_cast<const T*>(a.C) + tt0 * N, bc, &sm.bar);
    bulk_load_1d(sm.Araw, a.A + (int64_t)dd0 * N, nval * N * 4u, &sm.bar);
    tma_load_2d(sm.H, &tm_cs, dd0, ch * N, &sm.bar);
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
  // this item has read its inputs for the last time and its copies land while
  // this item writes its last partials.  An earlier draw would hold tickets
  // back from the look-back chains (an item whose neighbour sits reserved
  // behind a running item waits for both).  Items only ever wait on items
  // with smaller tickets, all of which are done or in hand of a running CTA,
  // so the loop cannot deadlock.
  for (uint32_t it = 0;; ++it) {
  const int tk = sm.ticket;
  if (tk >= n_items) break;
  // test knob (its own instantiation, so the others carry no code for it):
  // this item starts late, so its inclusive state is stored late and the
  // items after it on the chain walk back past their aggregates
  if constexpr (kKnob) {
    if ((long long)tk == a.delay_ticket) sleep_ns(a.delay_ns);
  }
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

  // ---- 1. per-(token, channel) values; all zero past the last token and on
  //         channels past D (a = 1, b = 0, g = 0 there), so that those feed
  //         exactly 0 into every sum they enter
  // a warp's 32 lanes take 8 channels x 4 tokens: the [channel][token]
  // stores then hit 32 different banks.  Straight-line code over the thread's
  // kPer elements (no per-element branches), so their exp / log chains overlap;
  // out-of-range elements are computed on whatever the buffers hold and then
  // replaced by zeros with selects.
  {
    constexpr int kPer = kL * kTile / kThr;
    float rv[kPer], uv[kPer], gov[kPer], dlv[kPer], sgv[kPer], gv[kPer];
    int cs[kPer], ts[kPer];
    bool ok[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int i = tid + q * kThr;
      const int b = i >> 5, l = i & 31;
      const int c = 8 * (b & 3) + (l >> 2), t = 4 * (b >> 2) + (l & 3);
      cs[q] = c;
      ts[q] = t;
      ok[q] = t < rows && c < bx && d0 + c < a.D;
      rv[q] = to_f(sm.dr[t * bx + c]) + (a.dt_bias ? sm.bias[c] : 0.0f);
      uv[q] = to_f(sm.u[t * bx + c]);
      gov[q] = to_f(sm.dout[t * bx + c]);
      gv[q] = a.has_z ? to_f(sm.z[t * bx + c]) : 0.0f;
    }
    if (a.delta_softplus) {
#pragma unroll
      for (int q = 0; q < kPer; ++q) dlv[q] = softplus_sig(rv[q], &sgv[q]);
    } else {
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        dlv[q] = rv[q];
        sgv[q] = 1.0f;
      }
    }
    if (a.has_z) {
#pragma unroll
      for (int q = 0; q < kPer; ++q) gv[q] = gov[q] * (siluf(gv[q]) + a.gate_floor);
    } else {
#pragma unroll
      for (int q = 0; q < kPer; ++q) gv[q] = gov[q];
    }
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int at = cs[q] * kP + ts[q];
      const float dl_q = ok[q] ? dlv[q] : 0.0f;
      sm.dl[at] = dl_q;
      sm.dlu[at] = ok[q] ? dl_q * uv[q] : 0.0f;
      sm.g[at] = ok[q] ? gv[q] : 0.0f;
      sm.sg[at] = ok[q] ? sgv[q] : 0.0f;
    }
  }
#pragma unroll
  for (int i = tid; i < N * kL; i += kThr) {
    const int t = i / N, n = i - t * N;  // consecutive lanes: consecutive states
    const int pw = n >> 1, e = n & 1;
    const float bv = t < rows ? to_f(sm.B[t * N + n]) : 0.0f;
    const float cv = t < rows ? to_f(sm.C[t * N + n]) : 0.0f;
    sm.BP[(pw * kPP + t) * 2 + e] = bv;
    sm.BP[((W + pw) * kPP + t) * 2 + 1 - e] = bv;
    sm.CP[(pw * kPP + t) * 2 + e] = cv;
    sm.CP[((W + pw) * kPP + t) * 2 + 1 - e] = cv;
  }
  // bit t: token t starts a sequence
  const unsigned rst =
      __ballot_sync(0xffffffffu, lane < rows && (lane < rows4 ? sm.pos[lane] : __ldg(a.pos + t0 + lane)) == 0);
  // ex2(-inf) = 0: the transition factor of a sequence's first token, for any A
  if (w == 0) sm.off[lane] = ((rst >> lane) & 1u) ? -INFINITY : 0.0f;
  // the warp's state pair, in this lane's order: "first" = n0 + bit4(lane)
  // (the column-sum butterflies keep a lane's first state)
  const int n0 = 2 * w;
  const int nF = n0 + ((lane >> 4) & 1), nS = n0 + 1 - ((lane >> 4) & 1);
  const float* const bp = sm.BP + ((((lane >> 4) & 1) * W + w) * kPP) * 2;  // this lane's pairs
  const float* const cp = sm.CP + ((((lane >> 4) & 1) * W + w) * kPP) * 2;
  float2 A2 = make_float2(0.0f, 0.0f), h = make_float2(0.0f, 0.0f);
  if (valid) {
    A2 = make_float2(sm.Araw[lane * N + nF], sm.Araw[lane * N + nS]);
    // the rows hold A or A_log (A = -exp(A_log)); kept scaled by log2 e for ex2
    if (a.a_log) A2 = make_float2(-ex2(A2.x * kLog2e), -ex2(A2.y * kLog2e));
    A2 = make_float2(A2.x * kLog2e, A2.y * kLog2e);
    h = make_float2(sm.H[nF * bx + lane], sm.H[nS * bx + lane]);
  }
  const float Dsk = (valid && a.Dskip) ? sm.dsk[lane] : 0.0f;
  // Sequence-state events of this item, bit t for token t of the chunk:
  //   evH: a sequence starts from a given initial state,
  //   evG: a sequence starts and the gradient reaching its initial state is asked for,
  //   evF: a sequence ends and a gradient reaches its final state from outside.
  unsigned evH = 0u, evG = 0u, evF = 0u;
  if (kStates && a.seq) {
    const unsigned live = rows >= 32 ? 0xffffffffu : ((1u << rows) - 1u);
    const unsigned starts = rst & live;
    evH = a.h_init ? starts : 0u;
    evG = a.dh_init ? starts : 0u;
    if (a.dh_final) {
      // token t ends a sequence when token t + 1 starts one or does not exist
      unsigned ends = starts >> 1;
      if (t0 + rows >= a.T || (rows == 32 && __ldg(a.pos + t0 + 32) == 0)) ends |= 1u << (rows - 1);
      evF = ends & live;
    }
  }
  // the (nF, nS) entries of a sequence-state row for token t's sequence
  auto state_pair = [&](const float* st, int t) {
    if (!valid) return make_float2(0.0f, 0.0f);
    const float2 v = __ldg(reinterpret_cast<const float2*>(st + ((int64_t)a.seq[t0 + t] * a.D + d) * N + n0));
    return (lane & 16) ? make_float2(v.y, v.x) : v;
  };
  __syncthreads();

  // ---- 2. forward walk over the 32 tokens (state pair n0, n0+1)
  float2 hist[kL];
  float2 E = make_float2(1.0f, 1.0f), tot = make_float2(0.0f, 0.0f);
  ColSum16 colsum;
  // the forward walk's dC sums (one per lane and 16-token group), stored only
  // after the look-back, so that a fence there does not wait for them
  float dcs[kL / 16];
  {
    constexpr bool kEv = kStates;
    const float* rowc = sm.dl + lane * kP;
#pragma unroll
    for (int kb = 0; kb < kL / 4; ++kb) {
      const float4 dl4 = *reinterpret_cast<const float4*>(rowc + 4 * kb);
      const float4 du4 = *reinterpret_cast<const float4*>(sm.dlu + lane * kP + 4 * kb);
      const float4 g4 = *reinterpret_cast<const float4*>(sm.g + lane * kP + 4 * kb);
      const float4 b01 = *reinterpret_cast<const float4*>(bp + 8 * kb);
      const float4 b23 = *reinterpret_cast<const float4*>(bp + 8 * kb + 4);
      const float4 c01 = *reinterpret_cast<const float4*>(cp + 8 * kb);
      const float4 c23 = *reinterpret_cast<const float4*>(cp + 8 * kb + 4);
      const float4 of4 = *reinterpret_cast<const float4*>(sm.off + 4 * kb);
      const float ofa[4] = {of4.x, of4.y, of4.z, of4.w};
      const float dla[4] = {dl4.x, dl4.y, dl4.z, dl4.w};
      const float dua[4] = {du4.x, du4.y, du4.z, du4.w};
      const float ga[4] = {g4.x, g4.y, g4.z, g4.w};
      const float2 Ba[4] = {make_float2(b01.x, b01.y), make_float2(b01.z, b01.w), make_float2(b23.x, b23.y),
                            make_float2(b23.z, b23.w)};
      const float2 Ca[4] = {make_float2(c01.x, c01.y), make_float2(c01.z, c01.w), make_float2(c23.x, c23.y),
                            make_float2(c23.z, c23.w)};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = 4 * kb + e;
        const float2 at = make_float2(ex2(fmaf(dla[e], A2.x, ofa[e])), ex2(fmaf(dla[e], A2.y, ofa[e])));
        const float2 Ct = Ca[e];
        h = fma2(at, h, mul2(splat2(dua[e]), Ba[e]));
        if constexpr (kEv) {
          if ((evH >> t) & 1u)  // a start from a given state: h = a h_init + b, a's own value
            h = fma2(make_float2(ex2(dla[e] * A2.x), ex2(dla[e] * A2.y)), state_pair(a.h_init, t), h);
        }
        hist[t] = h;
        E = mul2(E, at);
        tot = fma2(E, mul2(Ct, splat2(ga[e])), tot);
        if constexpr (kEv) {
          // the gradient reaching a final state joins dh_t, and the left carry through E_t
          if ((evF >> t) & 1u) tot = fma2(E, state_pair(a.dh_final, t), tot);
        }
        if (a.has_z && !a.has_y) sm.ypart[(w * kL + t) * kTile + lane] = fmaf(Ct.x, h.x, Ct.y * h.y);
        // dC contributions g_t h_t, summed over the tile's channels
        colsum.feed(t & 15, true, mul2(splat2(ga[e]), h), lane, &dcs[t >> 4]);
      }
    }
  }

  // ---- 3. decoupled look-back towards higher chunks (every warp for its pair)
  float2 x = make_float2(0.0f, 0.0f);
  {
    const int64_t base = (int64_t)tile * a.n_chunks;
    const int64_t wslot = (base + chunk) * W + w;
    const bool publish = (long long)tk != a.drop_ticket;
    float2* const agg = reinterpret_cast<float2*>(a.agg);
    float2* const aggp = reinterpret_cast<float2*>(a.agg_sd);
    float2* const inc = reinterpret_cast<float2*>(a.incl);
    // the carry words are their own flags (filled with kCarryUnset before the
    // launch); only an aggregate, published when the walk must go further,
    // is announced by the warp's flag
    int* const my_flag = a.flags + wslot;
    // a sequence starts in this chunk: E = 0 exactly, and the carry leaving
    // to the left does not depend on what enters from the right
    const bool rs_any = (rst & (rows >= 32 ? 0xffffffffu : ((1u << rows) - 1u))) != 0u;
    if (rs_any && publish) st_carry(inc + wslot * 32 + lane, tot);
    if (chunk < a.n_chunks - 1) {
      // the next chunk of the tile started long before this one and has
      // usually stored its inclusive carry: look first, and publish this
      // chunk's aggregate only when the walk has to go further
      int j = chunk + 1, found = -1, timed_out = 0;
      float2 v = ld_carry(inc + ((base + j) * W + w) * 32 + lane);
      if (__all_sync(0xffffffffu, carry_set(v))) {
        found = j;
      } else {
        if (!rs_any) {
          agg[wslot * 32 + lane] = tot;
          aggp[wslot * 32 + lane] = E;
          publish_flag(my_flag, kFlagAggregate, publish, lane);
        }
        while (j < a.n_chunks) {
          const int f = wait_carry(inc + ((base + j) * W + w) * 32 + lane, a.flags + (base + j) * W + w,
                                   a.wait_ns, &v);
          if (f == kFlagInclusive) { found = j; break; }
          if (f == kFlagNone) { timed_out = 1; break; }
          ++j;
        }
      }
      if (timed_out) atomicOr(a.status, kStatusLookbackTimeout);
      int last = j - 1;
      if (found >= 0) {
        x = v;
        last = found - 1;
      }
      for (int i = last; i > chunk; --i) {
        const int64_t ws = ((base + i) * W + w) * 32 + lane;
        x = fma2(__ldcg(aggp + ws), x, __ldcg(agg + ws));
      }
    }
    // stored at once: the previous chunk of the tile may already be waiting,
    // and every link of that chain adds this item's delay
    if (!rs_any && publish) st_carry(inc + wslot * 32 + lane, fma2(E, x, tot));
  }
#pragma unroll
  for (int q = 0; q < kL / 16; ++q) {
    const int tt = 16 * q + ColSum16::token(lane);
    if (tt < rows) a.part_dBC[((int64_t)tile * 2 * N + N + nF) * a.T + t0 + tt] = dcs[q];
  }
  // no barrier here: the reverse walk writes only its own partial buffers,
  // and the block barriers below order every cross-warp read

  // ---- 5. reverse walk in blocks of kRB tokens
  float2 dA = make_float2(0.0f, 0.0f);
  int next = 0;  // thread 0: the next ticket, drawn before the last block
  float sDD = 0.0f, sDB = 0.0f;
  {
    float2* const part2 = reinterpret_cast<float2*>(sm.part);  // [2][W][kRB][kTile]
    T* gdu = static_cast<T*>(a.du);
    T* gddr = static_cast<T*>(a.ddr);
    T* gdz = static_cast<T*>(a.dz);
    float2 r = x;  // carry entering the current token from the right
    constexpr bool kEv = kStates;
#pragma unroll
    for (int blk = kL / kRB - 1; blk >= 0; --blk) {
      const int buf = blk & 1;
      if (blk == 0 && tid == 0) next = (int)atomicAdd(a.ticket, 1u);
#pragma unroll
      for (int kb = (blk + 1) * kRB / 4 - 1; kb >= blk * kRB / 4; --kb) {
        const float4 dl4 = *reinterpret_cast<const float4*>(sm.dl + lane * kP + 4 * kb);
        const float4 du4 = *reinterpret_cast<const float4*>(sm.dlu + lane * kP + 4 * kb);
        const float4 g4 = *reinterpret_cast<const float4*>(sm.g + lane * kP + 4 * kb);
        const float4 b01 = *reinterpret_cast<const float4*>(bp + 8 * kb);
        const float4 b23 = *reinterpret_cast<const float4*>(bp + 8 * kb + 4);
        const float4 c01 = *reinterpret_cast<const float4*>(cp + 8 * kb);
        const float4 c23 = *reinterpret_cast<const float4*>(cp + 8 * kb + 4);
        const float4 of4 = *reinterpret_cast<const float4*>(sm.off + 4 * kb);
        const float ofa[4] = {of4.x, of4.y, of4.z, of4.w};
        const float dla[4] = {dl4.x, dl4.y, dl4.z, dl4.w};
        const float dua[4] = {du4.x, du4.y, du4.z, du4.w};
        const float ga[4] = {g4.x, g4.y, g4.z, g4.w};
        const float2 Ba[4] = {make_float2(b01.x, b01.y), make_float2(b01.z, b01.w), make_float2(b23.x, b23.y),
                              make_float2(b23.z, b23.w)};
        const float2 Ca[4] = {make_float2(c01.x, c01.y), make_float2(c01.z, c01.w), make_float2(c23.x, c23.y),
                              make_float2(c23.z, c23.w)};
#pragma unroll
        for (int e = 3; e >= 0; --e) {
          const int t = 4 * kb + e;
          const float2 at = make_float2(ex2(fmaf(dla[e], A2.x, ofa[e])), ex2(fmaf(dla[e], A2.y, ofa[e])));
          const float2 Bt = Ba[e];
          float2 dh = fma2(Ca[e], splat2(ga[e]), r);  // total gradient w.r.t. h_t
          if constexpr (kEv) {
            if ((evF >> t) & 1u) dh = __fadd2_rn(dh, state_pair(a.dh_final, t));
          }
          // a_t h_{t-1} = h_t - delta u B: no need for the previous state
          const float2 dhq = mul2(dh, fma2(splat2(-dua[e]), Bt, hist[t]));
          dA = fma2(splat2(dla[e]), dhq, dA);
          part2[((buf * W + w) * kRB + (t - blk * kRB)) * kTile + lane] =
              make_float2(fmaf(dh.x, Bt.x, dh.y * Bt.y), fmaf(A2.x, dhq.x, A2.y * dhq.y));
          float sum;  // dB contributions dh_t delta u, summed over the tile's channels
          if (colsum.feed(t & 15, false, mul2(dh, splat2(dua[e])), lane, &sum)) {
            const int tt = t + ColSum16::token(lane);
            if (tt < rows) a.part_dBC[((int64_t)tile * 2 * N + nF) * a.T + t0 + tt] = sum;
          }
          if constexpr (kEv) {
            if (((evG >> t) & 1u) && valid) {
              // the gradient reaching the starting state: dh_t times a's own value
              const float2 g0 = mul2(dh, make_float2(ex2(dla[e] * A2.x), ex2(dla[e] * A2.y)));
              float2* row = reinterpret_cast<float2*>(a.dh_init + ((int64_t)a.seq[t0 + t] * a.D + d) * N + n0);
              *row = (lane & 16) ? make_float2(g0.y, g0.x) : g0;
            }
          }
          r = mul2(dh, at);  // carry to h_{t-1}
        }
      }
      __syncthreads();  // the block's partials are complete
      // du, d delta_raw and dz of the block: thread i takes token
      // blk*kRB + i / kTile, channel i % kTile (= lane), and adds the warps'
      // partials in order
      for (int i = tid; i < kRB * kTile; i += kThr) {
        const int e = i / kTile;
        const int t = blk * kRB + e;
        float2 sp = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int v = 0; v < W; ++v) sp = __fadd2_rn(sp, part2[((buf * W + v) * kRB + e) * kTile + lane]);
        float y = 0.0f;  // C.h, for dz, when the call has no y to read
        if (a.has_z && !a.has_y) {
#pragma unroll
          for (int v = 0; v < W; ++v) y += sm.ypart[(v * kL + t) * kTile + lane];
        }
        const float dlt = sm.dl[lane * kP + t], gt = sm.g[lane * kP + t];
        const float uv = to_f(sm.u[t * bx + lane]);
        const float gdu_t = fmaf(dlt, sp.x, Dsk * gt);
        const float gdr_t = fmaf(uv, sp.x, sp.y * kLn2) * sm.sg[lane * kP + t];
        if (t < rows && valid) {
          const int64_t at_td = (t0 + t) * a.D + d;
          gdu[at_td] = from_f<T>(gdu_t);
          gddr[at_td] = from_f<T>(gdr_t);
          if (a.has_z) {
            const float go = to_f(sm.dout[t * bx + lane]);
            const float zz = to_f(sm.z[t * bx + lane]);
            const float sz = sigmoidf_fast(zz);
            const float yf = a.has_y ? to_f(sm.y[t * bx + lane]) : fmaf(Dsk, uv, y);
            gdz[at_td] = from_f<T>(go * sz * fmaf(zz, 1.0f - sz, 1.0f) * yf);
          }
          sDD = fmaf(gt, uv, sDD);
          sDB += gdr_t;
        }
      }
    }
  }

  // ---- 6. dA partials of the chunk ([chunk][n][d]); fixed-order CTA sums of
  //         the dDskip and d_dt_bias partials
  if (valid) {
    // for A_log the chain rule gives dA_log = dA * A (A = A2 ln 2), applied to
    // every chunk's partial before the fixed-order sum
    const float2 s = a.a_log ? make_float2(A2.x * kLn2, A2.y * kLn2) : make_float2(1.0f, 1.0f);
    a.part_dA[((int64_t)chunk * N + nF) * a.D + d] = dA.x * s.x;
    a.part_dA[((int64_t)chunk * N + nS) * a.D + d] = dA.y * s.y;
  }
  sm.redD[w * kTile + lane] = sDD;
  sm.redB[w * kTile + lane] = sDB;
  __syncthreads();
  // no input buffer is read any more: draw the next item and request its
  // inputs, which land while this item writes its last partials
  if (tid == 0) {
    sm.ticket = next;
    if (next < n_items) issue(next);
  }
  if (w == 0 && valid) {
    float accD = 0.0f, accB = 0.0f;
#pragma unroll
    for (int v = 0; v < W; ++v) {
      accD += sm.redD[v * kTile + lane];
      accB += sm.redB[v * kTile + lane];
    }
    a.part_dD[(int64_t)chunk * a.D + d] = accD;
    a.part_dbias[(int64_t)chunk * a.D + d] = accB;
  }
  __syncthreads();  // redD / redB and the ticket are consumed before the next pass
  }  // persistent loop
}

// dB[t][n] = sum over tiles of part[tile][n][t]; dC[t][n] likewise from
// part[tile][N + n][t].  One thread per output, tiles summed in order.
__global__ void __launch_bounds__(256) sum_tiles_bc_kernel(const float* __restrict__ part,
                                                           int n_tiles, int64_t T, int N,
                                                           float* __restrict__ dB,
                                                           float* __restrict__ dC) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t M = T * 2 * N;
  if (i >= M) return;
  float acc = 0.0f;
  int k = 0;
  for (; k + 8 <= n_tiles; k += 8) {  // 8 loads in flight, added in tile order
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = __ldcs(part + (int64_t)(k + q) * M + i);
#pragma unroll
    for (int q = 0; q < 8; ++q) acc += v[q];
  }
  for (; k < n_tiles; ++k) acc += __ldcs(part + (int64_t)k * M + i);
  const int64_t v = i / T;
  const int64_t t = i - v * T;
  if (v < N) dB[t * N + v] = acc; else dC[t * N + (v - N)] = acc;
}

template <typename T, int N, bool kStates, bool kKnob = false>
cudaError_t launch_k(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, const CUtensorMap& tm_dout, const CUtensorMap& tm_cs,
                     const CUtensorMap& tm_y, cudaStream_t st) {
  const size_t smem = sizeof(BwdSmem<T, N>);
  cudaError_t e = cudaFuncSetAttribute(scan_bwd_kernel<T, N, kStates, kKnob>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.n_chunks * a.n_tiles;
  int grid = 0;
  e = persistent_grid(scan_bwd_kernel<T, N, kStates, kKnob>, 16 * N, smem, items, &grid);
  if (e != cudaSuccess) return e;
  scan_bwd_kernel<T, N, kStates, kKnob><<<grid, 16 * N, smem, st>>>(tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, a);
  return cudaGetLastError();
}

template <typename T, int N>
cudaError_t launch_n(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, const CUtensorMap& tm_dout, const CUtensorMap& tm_cs,
                     const CUtensorMap& tm_y, cudaStream_t st) {
  if constexpr (sizeof(T) == 4 && N == 16) {  // the delay knob's instantiation
    if (a.delay_ticket >= 0 && !a.seq) return launch_k<T, N, false, true>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
  }
  return a.seq ? launch_k<T, N, true>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st)
               : launch_k<T, N, false>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
}

template <typename T>
cudaError_t launch_t(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, const CUtensorMap& tm_dout, const CUtensorMap& tm_cs,
                     const CUtensorMap& tm_y, cudaStream_t st) {
  if (a.N == 16) return launch_n<T, 16>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
  if (a.N == 8) return launch_n<T, 8>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
  if (a.N == 4) return launch_n<T, 4>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_scan_bwd(const ScanArgs& a, IO io, const CUtensorMap& tm_u,
                            const CUtensorMap& tm_dr, const CUtensorMap& tm_z,
                            const CUtensorMap& tm_dout, const CUtensorMap& tm_cs,
                            const CUtensorMap& tm_y, float* dA, float* dB, float* dC, float* dDskip,
                            float* d_dt_bias, cudaStream_t st) {
  const int64_t DN = (int64_t)a.D * a.N;
  if (a.T <= 0) {
    cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(float) * DN, st);
    if (e == cudaSuccess && dDskip) e = cudaMemsetAsync(dDskip, 0, sizeof(float) * a.D, st);
    if (e == cudaSuccess && d_dt_bias) e = cudaMemsetAsync(d_dt_bias, 0, sizeof(float) * a.D, st);
    return e;
  }
  cudaError_t e = io == IO::F32 ? launch_t<float>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st)
                                : launch_t<__nv_bfloat16>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
  if (e != cudaSuccess) return e;
  const int64_t M = a.T * 2 * a.N;
  sum_tiles_bc_kernel<<<(unsigned)((M + 255) / 256), 256, 0, st>>>(a.part_dBC, a.n_tiles, a.T, a.N,
                                                                   dB, dC);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // part_dA is [chunk][n][d]: sum over chunks, written out as dA[d][n]
  e = launch_sum_rows(a.part_dA, a.n_chunks, DN, DN, dA, st, a.D);
  if (e == cudaSuccess && dDskip) e = launch_sum_rows(a.part_dD, a.n_chunks, a.D, a.D, dDskip, st);
  if (e == cudaSuccess && d_dt_bias)
    e = launch_sum_rows(a.part_dbias, a.n_chunks, a.D, a.D, d_dt_bias, st);
  return e;
}

}  // namespace vssm
