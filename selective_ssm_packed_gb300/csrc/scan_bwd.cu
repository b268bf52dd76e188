// scan_bwd.cu -- packed selective scan, backward (sm_103a).
//
// Work item = (chunk of kBwdChunk = 32 tokens, the saved-state granule) x
// (tile of kTile = 32 channels); items are taken in DESCENDING chunk order
// from an atomic ticket because the state gradient flows from the end of a
// sequence to its start.  The kernel is persistent (one CTA per resident slot,
// looping over tickets); one thread requests each item's inputs with tensor /
// bulk copies on one mbarrier while the previous item finishes.
//
// CTA = N/4 warps.  A thread owns one channel PAIR (lane % 16: channels 2c,
// 2c+1 of the tile) and one state pair (warp w, lane / 16: states 2p, 2p+1,
// p = 2w + lane / 16): four (channel, state) chains.  The paired FP32
// instructions run over the channel pair, so the per-(token, channel) values
// (delta, delta u, g) are used as loaded and the per-(token, state) values (B,
// C) come from shared memory already doubled (x, x).
//
// With a_t = exp(delta_t A) (0 at a sequence start), b_t = delta_t u_t B_t,
// g_t = dout_t (SiLU(z_t) + gate floor):
//   h_t  = a_t h_{t-1} + b_t                       (forward walk)
//   dh_t = C_t g_t + a_{t+1} dh_{t+1}              (reverse walk; a_{t+1} = 0
//                                                   at a sequence start, so the
//                                                   scan resets at sequence ends)
//   du_t     = delta_t sum_n dh_t B_t + Dskip g_t
//   d delta_t = u_t sum_n dh_t B_t + sum_n A dh_t p_t,   p_t = a_t h_{t-1}
//   dA       = sum_t delta_t dh_t p_t,  dB_t = sum_d dh_t delta_t u_t,  dC_t = sum_d g_t h_t
//
//   1. Per-(token, channel) values once per item: delta (softplus), delta u,
//      g, d delta / d delta_raw into [channel pair][token] arrays, and dz from
//      the forward's pre-gate output y (so the gate is evaluated once); a
//      per-token exponent offset (-inf at a start).  B and C arrive doubled
//      per state pair, built once per call for every item (launch_double_bc).
//   2. Forward walk per thread from the saved state of the chunk: p_t goes to
//      TENSOR MEMORY (4 words per token, 128 columns per warp) for the reverse
//      walk, so the history costs no registers; the left-going carry aggregate
//      sum_t E_t C_t g_t (E_t = a_t0 ... a_t) is accumulated on the way; dC
//      sums over the tile's channels by shuffle butterflies.
//   3. Decoupled look-back per thread towards HIGHER chunks for the carry
//      entering from the right; aggregates re-applied in a fixed order
//      (bitwise repeatable); time-bounded waits.  An inclusive carry is its
//      own flag (the carry array starts filled with a NaN word that no stored
//      value equals); only an aggregate is announced by a flag, behind a fence.
//   4. Reverse walk in blocks of 4 tokens, reading p_t back from tensor
//      memory: dA per thread, dB by shuffle butterflies, and per-thread
//      partial sums over its 2 states of sum_n dh B and sum_n A dh p, added
//      over the state pairs after each block (fixed order) into du and
//      d delta_raw.
//   5. dA partials per chunk; fixed-order CTA sums for dDskip and d_dt_bias.
// Separate fixed-order kernels sum the partials over channel tiles (dB, dC)
// and chunks (dA, dDskip, d_dt_bias).  No atomics anywhere in the arithmetic.
#include <cstddef>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace vssm {

namespace {

constexpr int kL = kBwdChunk;   // 32 tokens per work item
constexpr int kCP = kTile / 2;  // 16 channel pairs per item
constexpr int kPT = kL + 2;     // token pitch (in pairs) of the [channel pair][token] arrays
constexpr int kRB = 4;          // tokens per block of the reverse walk
constexpr float kLn2 = 0.6931471805599453f;

template <typename T, int N, bool kRecY>
struct BwdSmem {
  static constexpr int NW = N / 4;   // warps
  static constexpr int NSP = N / 2;  // state pairs
  // ---- inputs of one work item, written by tensor / bulk copies and refilled
  //      for the next item once this one has read them for the last time
  alignas(128) T u[kL * kTile];
  alignas(128) T dr[kL * kTile];
  alignas(128) T z[kL * kTile];
  alignas(128) T dout[kL * kTile];
  alignas(128) T y[kL * kTile];  // the forward's pre-gate output, when the call has it
  alignas(16) float Araw[kTile * N];  // A rows d0 .. d0+31
  alignas(128) float H[N * kTile];    // saved states at the chunk start, [n][channel]
  alignas(16) float bias[kTile];
  alignas(16) float dsk[kTile];
  alignas(16) int pos[kL];
  // ---- per-(token, channel pair) values, [channel pair][token] float2 with
  //      token pitch kPT: a lane reads 2 tokens of its pair with one 16-byte
  //      access, the 8 lanes of an access phase in distinct banks
  alignas(16) float2 dl[kCP * kPT];   // delta
  alignas(16) float2 dlu[kCP * kPT];  // delta * u
  alignas(16) float2 g[kCP * kPT];    // dout * (SiLU(z) + gate floor)
  alignas(16) float2 sg[kCP * kPT];   // d delta / d delta_raw
  alignas(16) float2 dzf[kRecY ? kCP * kPT : 2];  // d out / d y, when y is recomputed
  // ---- B and C doubled, [token][state pair][order] float4: order 0 holds
  //      (B[2p], B[2p], B[2p+1], B[2p+1]), order 1 the two states swapped, the
  //      order the lanes with bit 3 set keep (see ColSum8); zero past the last
  //      token.  Token-major, so that the four entries a warp reads for a
  //      token are adjacent (one bank-conflict-free access)
  alignas(16) float4 BD[kL * NSP * 2];
  alignas(16) float4 CD[kL * NSP * 2];
  // ---- exponent offset per token pair (off_t, off_t, off_t+1, off_t+1): -inf
  //      at a sequence start, else 0
  alignas(16) float4 off[kL / 2];
  // ---- partial sums over each thread's state pair from the reverse walk,
  //      [buffer][token of the block][state pair][channel pair] float4 =
  //      (sum dh B for the pair's two channels, sum A dh p for them)
  alignas(16) float4 nred[2 * kRB * NSP * kCP];
  alignas(16) float2 nY[kRecY ? 2 * kRB * NSP * kCP : 2];  // C.h partials, when y is recomputed
  alignas(16) float2 redD[32 * NW];
  alignas(16) float2 redB[32 * NW];
  uint32_t taddr;
  int ticket;
  alignas(8) uint64_t bar;
};

// Column sums over the 16 lanes of a half warp (lane % 16 = channel pair) for
// groups of 8 tokens x 2 states, fed one token at a time by shuffle
// butterflies.  A lane keeps its state pair in its own order, the "first"
// state being 2p + bit3(lane):
//   level 1 (every token): lanes l, l^8 exchange the state the other keeps,
//   level 2 (every token pair): lanes l, l^4 exchange the token the other
//     keeps (bit 2 picks the odd token),
//   levels 3, 4 likewise over lane bits 1, 0 for pairs of pairs, ...
// After the 8th token, lane l holds the sum over the half warp for token
// 4 b0 + 2 b1 + b2 of the group (b_i = bit i of l) and its first state.  The
// pairing is fixed, so the sums are bitwise repeatable; tokens may come in
// ascending or descending order.
struct ColSum8 {
  float p1[2], p2[2], p3[2];  // pending sums, by the parity of the token group at each level

  static __device__ __forceinline__ int token(int lane) {
    return 4 * (lane & 1) + 2 * ((lane >> 1) & 1) + ((lane >> 2) & 1);
  }

  static __device__ __forceinline__ float combine(float lo, float hi, int lane, int mask) {
    const bool up = (lane & mask) != 0;
    return (up ? hi : lo) + __shfl_xor_sync(0xffffffffu, up ? lo : hi, mask);
  }

  // Token c (0..7) of the group with this lane's two values in its state
  // order; returns true once the group is complete (*sum then holds the result).
  __device__ __forceinline__ bool feed(int c, bool ascending, float vF, float vS, int lane, float* sum) {
    p1[c & 1] = vF + __shfl_xor_sync(0xffffffffu, vS, 8);
    if ((c & 1) != (ascending ? 1 : 0)) return false;
    p2[(c >> 1) & 1] = combine(p1[0], p1[1], lane, 4);
    if ((c & 3) != (ascending ? 3 : 0)) return false;
    p3[(c >> 2) & 1] = combine(p2[0], p2[1], lane, 2);
    if ((c & 7) != (ascending ? 7 : 0)) return false;
    *sum = combine(p3[0], p3[1], lane, 1);
    return true;
  }
};

__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  const float2 l = __fadd2_rn(lo2(a), lo2(b)), h = __fadd2_rn(hi2(a), hi2(b));
  return make_float4(l.x, l.y, h.x, h.y);
}
__device__ __forceinline__ float hsum(float2 v) { return v.x + v.y; }
__device__ __forceinline__ uint32_t fbits(float v) { return __float_as_uint(v); }
__device__ __forceinline__ float bitsf(uint32_t v) { return __uint_as_float(v); }

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
// kRecY: the call has z but no y, so dz needs y = C.h + Dskip u recomputed
// (the reverse walk adds C.h partials).
template <typename T, int N, bool kStates, bool kRecY, bool kKnob>
__global__ void __launch_bounds__(8 * N, N == 16 ? 3 : 4)
scan_bwd_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dr,
                const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_dout,
                const __grid_constant__ CUtensorMap tm_cs, const __grid_constant__ CUtensorMap tm_y,
                const ScanArgs a) {
  using SM = BwdSmem<T, N, kRecY>;
  constexpr int NW = SM::NW, NSP = SM::NSP;
  constexpr int kThr = 32 * NW;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int n_items = a.n_chunks * a.n_tiles;
  const int cp = lane & 15;                        // channel pair of the tile
  const int sp = 2 * w + (lane >> 4);              // state pair
  const int o = (lane >> 3) & 1;                   // this lane's state order
  const int nF = 2 * sp + o, nS = 2 * sp + 1 - o;  // its "first" and "second" state
  const int c0 = 2 * cp;                           // first channel of the pair (in the tile)

  // Requests every input of work item `tkn` on the barrier: u, delta_raw,
  // dout, z (and y) tiles; B and C rows; A rows, dt_bias, Dskip and the saved
  // states of the tile's channels; position indices (whole groups of 4 tokens).
  auto issue = [&](int tkn) {
    const int rv = tkn / a.n_tiles;
    const int tl = tkn - rv * a.n_tiles;
    const int ch = a.n_chunks - 1 - rv;
    const int64_t tt0 = (int64_t)ch * kL;
    const int nrows = (int)((a.T - tt0) < kL ? (a.T - tt0) : kL);
    const int dd0 = tl * kTile;
    const uint32_t nval = (uint32_t)(a.D - dd0 < kTile ? a.D - dd0 : kTile);
    const uint32_t bcd = (uint32_t)kL * N * 16u;  // the chunk's doubled B (or C) rows
    const uint32_t rows4 = (uint32_t)nrows & ~3u;
    const uint32_t box = (uint32_t)a.box_x * (uint32_t)a.box_y * sizeof(T);
    mbar_arrive_expect_tx(&sm.bar, box * (3u + (a.has_z ? 1u : 0u) + (a.has_y ? 1u : 0u)) + 2u * bcd + nval * N * 4u +
                                       (uint32_t)a.box_x * N * 4u + rows4 * 4u +
                                       (a.dt_bias ? nval * 4u : 0u) + (a.Dskip ? nval * 4u : 0u));
    tma_load_2d(sm.u, &tm_u, dd0, (int)tt0, &sm.bar);
    tma_load_2d(sm.dr, &tm_dr, dd0, (int)tt0, &sm.bar);
    tma_load_2d(sm.dout, &tm_dout, dd0, (int)tt0, &sm.bar);
    if (a.has_z) tma_load_2d(sm.z, &tm_z, dd0, (int)tt0, &sm.bar);
    if (a.has_y) tma_load_2d(sm.y, &tm_y, dd0, (int)tt0, &sm.bar);
    bulk_load_1d(sm.BD, a.BD + tt0 * N, bcd, &sm.bar);
    bulk_load_1d(sm.CD, a.CD + tt0 * N, bcd, &sm.bar);
    bulk_load_1d(sm.Araw, a.A + (int64_t)dd0 * N, nval * N * 4u, &sm.bar);
    tma_load_2d(sm.H, &tm_cs, dd0, ch * N, &sm.bar);
    if (a.dt_bias) bulk_load_1d(sm.bias, a.dt_bias + dd0, nval * 4u, &sm.bar);
    if (a.Dskip) bulk_load_1d(sm.dsk, a.Dskip + dd0, nval * 4u, &sm.bar);
    if (rows4) bulk_load_1d(sm.pos, a.pos + tt0, rows4 * 4u, &sm.bar);
  };

  // tensor memory for the forward walk's history: 128 columns, warp w on the
  // lanes 32 (w % 4) .. +31 (the CTA has at most 4 warps)
  if (w == 0) tmem_alloc128(&sm.taddr);
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
    const int first = (int)atomicAdd(a.ticket, 1u);
    sm.ticket = first;
    if (first < n_items) issue(first);
  }
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t thist = sm.taddr + ((uint32_t)(32 * (w & 3)) << 16);

  // Persistent loop: one work item per pass.  The next ticket is drawn in
  // the last block of the reverse walk and its inputs are requested once this
  // item has read its own for the last time.  An earlier draw would hold
  // tickets back from the look-back chains (an item whose neighbour sits
  // reserved behind a running item waits for both).  Items only ever wait on
  // items with smaller tickets, all of which are done or in hand of a running
  // CTA, so the loop cannot deadlock.
  for (uint32_t it = 0;; ++it) {
  const int tk = sm.ticket;
  if (tk >= n_items) break;
  // test knob (its own instantiation, so the others carry no code for it):
  // this item starts late, so its inclusive carry is stored late and the
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
  const int d = d0 + c0;                       // first channel of this thread's pair
  const bool valid = c0 < bx && d < a.D;       // D is even, so the pair is whole

  if (!__syncthreads_and(mbar_wait(&sm.bar, it & 1u, a.wait_ns))) {
    // the copies did not land within the limit: report it, give them a
    // second limit to complete (so that no copy is left writing into this
    // CTA's shared memory once it has exited), and stop
    if (tid == 0) atomicOr(a.status, kStatusTmaTimeout);
    mbar_wait(&sm.bar, it & 1u, kCopyDrainNs);
    break;
  }

  // ---- 1. per-(token, channel pair) values; all zero past the last token and
  //         on channels past D (a = 1, b = 0, g = 0 there), so that those feed
  //         exactly 0 into every sum they enter.  Lanes take 16 pairs x 2
  //         tokens; a thread keeps the same pair (tid % 16) throughout.
  float2 accD = make_float2(0.0f, 0.0f);  // dDskip partial: sum g u of this thread's pair
  {
    T* gdz = static_cast<T*>(a.dz);
    const float2 bias2 = a.dt_bias ? make_float2(sm.bias[c0 & 31], sm.bias[(c0 + 1) & 31]) : make_float2(0.0f, 0.0f);
#pragma unroll 2
    for (int i = tid; i < kL * kCP; i += kThr) {
      const int t = i >> 4;
      const int at = t * bx + c0;  // raw tiles are [token][bx]
      const bool ok = t < rows && valid;
      const float2 rr = __fadd2_rn(ld_io2(sm.dr + at), bias2);
      const float2 uu = ld_io2(sm.u + at);
      const float2 go = ld_io2(sm.dout + at);
      float2 dl2, sg2;
      if (a.delta_softplus) {
        dl2.x = softplus_sig(rr.x, &sg2.x);
        dl2.y = softplus_sig(rr.y, &sg2.y);
      } else {
        dl2 = rr;
        sg2 = make_float2(1.0f, 1.0f);
      }
      float2 gv = go;
      if (a.has_z) {
        const float2 zz = ld_io2(sm.z + at);
        const float2 s = make_float2(sigmoidf_fast(zz.x), sigmoidf_fast(zz.y));
        gv = mul2(go, fma2(zz, s, splat2(a.gate_floor)));
        // d out / d y, and dz = dout SiLU'(z) y (SiLU'(z) = s (1 + z (1 - s)))
        const float2 f = mul2(mul2(go, s), fma2(zz, make_float2(1.0f - s.x, 1.0f - s.y), splat2(1.0f)));
        if (a.has_y) {
          if (ok) st_io2(gdz + (t0 + t) * a.D + d, mul2(f, ld_io2(sm.y + at)));
        } else if constexpr (kRecY) {
          sm.dzf[cp * kPT + t] = ok ? f : make_float2(0.0f, 0.0f);
        }
      }
      const float2 z0 = make_float2(0.0f, 0.0f);
      sm.dl[cp * kPT + t] = ok ? dl2 : z0;
      sm.dlu[cp * kPT + t] = ok ? mul2(dl2, uu) : z0;
      sm.g[cp * kPT + t] = ok ? gv : z0;
      sm.sg[cp * kPT + t] = ok ? sg2 : z0;
      if (ok) accD = fma2(gv, uu, accD);
    }
  }
  // bit t: token t starts a sequence
  const unsigned rst =
      __ballot_sync(0xffffffffu, lane < rows && (lane < rows4 ? sm.pos[lane] : __ldg(a.pos + t0 + lane)) == 0);
  if (w == 0 && lane < kL / 2) {
    // ex2(-inf) = 0: the transition factor of a sequence's first token, for any A
    const float o0 = ((rst >> (2 * lane)) & 1u) ? -INFINITY : 0.0f;
    const float o1 = ((rst >> (2 * lane + 1)) & 1u) ? -INFINITY : 0.0f;
    sm.off[lane] = make_float4(o0, o0, o1, o1);
  }
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
  // a sequence-state row entry pair (channels d, d+1) of state n for token t's sequence
  auto state_pair = [&](const float* st, int t, int n) {
    if (!valid || !VSSM_CHECKED((unsigned)a.seq[t0 + t] < (unsigned)a.num_seqs, a.status))
      return make_float2(0.0f, 0.0f);
    const float* row = st + ((int64_t)a.seq[t0 + t] * a.D + d) * N + n;
    return make_float2(__ldg(row), __ldg(row + N));
  };
  __syncthreads();

  // the thread's A pairs (A * log2 e for ex2; the rows hold A or A_log) and
  // the saved states at the chunk start
  float2 AF = make_float2(0.0f, 0.0f), AS = make_float2(0.0f, 0.0f);
  float2 hF = make_float2(0.0f, 0.0f), hS = make_float2(0.0f, 0.0f);
  if (valid) {
    AF = make_float2(sm.Araw[c0 * N + nF], sm.Araw[(c0 + 1) * N + nF]);
    AS = make_float2(sm.Araw[c0 * N + nS], sm.Araw[(c0 + 1) * N + nS]);
    if (a.a_log) {
      AF = make_float2(-ex2(AF.x * kLog2e), -ex2(AF.y * kLog2e));
      AS = make_float2(-ex2(AS.x * kLog2e), -ex2(AS.y * kLog2e));
    }
    AF = mul2(AF, splat2(kLog2e));
    AS = mul2(AS, splat2(kLog2e));
    hF = *reinterpret_cast<const float2*>(sm.H + nF * bx + c0);
    hS = *reinterpret_cast<const float2*>(sm.H + nS * bx + c0);
  }
  const float2* const dlr = sm.dl + cp * kPT;
  const float2* const dur = sm.dlu + cp * kPT;
  const float2* const gr = sm.g + cp * kPT;
  const float4* const bdr = sm.BD + sp * 2 + o;  // entry of token t at [t * 2 NSP]
  const float4* const cdr = sm.CD + sp * 2 + o;
  float* const pdB = a.part_dBC + ((int64_t)tile * 2 * N + nF) * a.T + t0;
  float* const pdC = a.part_dBC + ((int64_t)tile * 2 * N + N + nF) * a.T + t0;

  // ---- 2. forward walk over the 32 tokens; p_t = a_t h_{t-1} to tensor memory
  float2 EF = make_float2(1.0f, 1.0f), ES = make_float2(1.0f, 1.0f);
  float2 totF = make_float2(0.0f, 0.0f), totS = make_float2(0.0f, 0.0f);
  {
    ColSum8 colsum;
#pragma unroll 1
    for (int g8 = 0; g8 < kL / 8; ++g8) {
      uint32_t hist[16];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const int t = 8 * g8 + e;
        const float4 dl4 = *reinterpret_cast<const float4*>(dlr + t);
        const float4 du4 = *reinterpret_cast<const float4*>(dur + t);
        const float4 g4 = *reinterpret_cast<const float4*>(gr + t);
        const float4 of4 = sm.off[t >> 1];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int tt = t + j, e2 = e + j;
          const float2 dlp = j ? hi2(dl4) : lo2(dl4);
          const float2 dup = j ? hi2(du4) : lo2(du4);
          const float2 gp = j ? hi2(g4) : lo2(g4);
          const float2 ofp = j ? hi2(of4) : lo2(of4);
          const float4 bd = bdr[tt * 2 * NSP], cd = cdr[tt * 2 * NSP];
          const float2 aF = ex2x2(fma2(dlp, AF, ofp)), aS = ex2x2(fma2(dlp, AS, ofp));
          float2 pF = mul2(aF, hF), pS = mul2(aS, hS);
          if constexpr (kStates) {
            if ((evH >> tt) & 1u) {  // a start from a given state: p = a h_init, a's own value
              pF = mul2(ex2x2(mul2(dlp, AF)), state_pair(a.h_init, tt, nF));
              pS = mul2(ex2x2(mul2(dlp, AS)), state_pair(a.h_init, tt, nS));
            }
          }
          hF = fma2(dup, lo2(bd), pF);
          hS = fma2(dup, hi2(bd), pS);
          EF = mul2(EF, aF);
          ES = mul2(ES, aS);
          totF = fma2(EF, mul2(lo2(cd), gp), totF);
          totS = fma2(ES, mul2(hi2(cd), gp), totS);
          if constexpr (kStates) {
            // the gradient reaching a final state joins dh_t, and the left carry through E_t
            if ((evF >> tt) & 1u) {
              totF = fma2(EF, state_pair(a.dh_final, tt, nF), totF);
              totS = fma2(ES, state_pair(a.dh_final, tt, nS), totS);
            }
          }
          const int hw = 4 * (e2 & 3);
          hist[hw + 0] = fbits(pF.x);
          hist[hw + 1] = fbits(pF.y);
          hist[hw + 2] = fbits(pS.x);
          hist[hw + 3] = fbits(pS.y);
          // dC contributions g_t h_t over the pair's channels, then over the tile's
          float sum;
          if (colsum.feed(e2, true, hsum(mul2(gp, hF)), hsum(mul2(gp, hS)), lane, &sum)) {
            const int ts = 8 * g8 + ColSum8::token(lane);
            if (ts < rows) pdC[ts] = sum;
          }
          if ((e2 & 3) == 3) {
            __syncwarp();  // the tensor-memory instructions are warp-collective
            tmem_st16(thist + (uint32_t)(4 * (tt & ~3)), hist);
            tmem_wait_st16(hist);
          }
        }
      }
    }
  }

  // ---- 3. decoupled look-back towards higher chunks (one chain per thread)
  float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  {
    const int64_t base = (int64_t)tile * a.n_chunks;
    const int64_t wslot = (base + chunk) * kThr + tid;
    const bool publish = (long long)tk != a.drop_ticket;
    float4* const agg = reinterpret_cast<float4*>(a.agg);
    float4* const aggp = reinterpret_cast<float4*>(a.agg_sd);
    float4* const inc = reinterpret_cast<float4*>(a.incl);
    // the carry words are their own flags (filled with kCarryUnset before the
    // launch); only an aggregate, published when the walk must go further,
    // is announced by the warp's flag
    int* const my_flag = a.flags + (base + chunk) * NW + w;
    const float4 tot = make_float4(totF.x, totF.y, totS.x, totS.y);
    const float4 E = make_float4(EF.x, EF.y, ES.x, ES.y);
    // a sequence starts in this chunk: E = 0 exactly, and the carry leaving
    // to the left does not depend on what enters from the right
    const bool rs_any = (rst & (rows >= 32 ? 0xffffffffu : ((1u << rows) - 1u))) != 0u;
    if (rs_any && publish) st_carry4(inc + wslot, tot);
    if (chunk < a.n_chunks - 1) {
      // the next chunk of the tile started long before this one and has
      // usually stored its inclusive carry: look first, and publish this
      // chunk's aggregate only when the walk has to go further
      int j = chunk + 1, found = -1, timed_out = 0;
      float4 v = ld_carry4(inc + (base + j) * kThr + tid);
      if (__all_sync(0xffffffffu, carry_set4(v))) {
        found = j;
      } else {
        if (!rs_any) {
          agg[wslot] = tot;
          aggp[wslot] = E;
          publish_flag(my_flag, kFlagAggregate, publish, lane);
        }
        while (j < a.n_chunks) {
          const int f = wait_carry4(inc + (base + j) * kThr + tid, a.flags + (base + j) * NW + w, a.wait_ns, &v);
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
        const int64_t ws = (base + i) * kThr + tid;
        const float4 p = __ldcg(aggp + ws), q = __ldcg(agg + ws);
        const float2 lo = fma2(lo2(p), lo2(x), lo2(q)), hi = fma2(hi2(p), hi2(x), hi2(q));
        x = make_float4(lo.x, lo.y, hi.x, hi.y);
      }
    }
    // stored at once: the previous chunk of the tile may already be waiting,
    // and every link of that chain adds this item's delay
    if (!rs_any && publish) {
      const float2 lo = fma2(lo2(E), lo2(x), lo2(tot)), hi = fma2(hi2(E), hi2(x), hi2(tot));
      st_carry4(inc + wslot, make_float4(lo.x, lo.y, hi.x, hi.y));
    }
  }

  // ---- 4. reverse walk in blocks of kRB tokens, p_t read back from tensor memory
  float2 dAF = make_float2(0.0f, 0.0f), dAS = make_float2(0.0f, 0.0f);
  float2 accB = make_float2(0.0f, 0.0f);  // d_dt_bias partial of this thread's finalize pair
  int next = 0;  // thread 0: the next ticket, drawn in the last block
  {
    T* gdu = static_cast<T*>(a.du);
    T* gddr = static_cast<T*>(a.ddr);
    T* gdz = static_cast<T*>(a.dz);
    float2 rF = lo2(x), rS = hi2(x);  // carry entering the current token from the right
    ColSum8 colsum;
    // One block of 4 tokens (descending) with its history in hb, then the
    // block's du and d delta_raw once every state pair has added its partials.
    auto block = [&](auto parity, int bp, uint32_t (&hb)[16]) {
      constexpr int buf = decltype(parity)::value;  // blocks 2 bp + 1 and 2 bp form one 8-token group
      const int blk = 2 * bp + buf;
      if (blk == 0 && tid == 0) next = (int)atomicAdd(a.ticket, 1u);
#pragma unroll
      for (int e = kRB - 2; e >= 0; e -= 2) {
        const int t = blk * kRB + e;
        const float4 dl4 = *reinterpret_cast<const float4*>(dlr + t);
        const float4 du4 = *reinterpret_cast<const float4*>(dur + t);
        const float4 g4 = *reinterpret_cast<const float4*>(gr + t);
        const float4 of4 = sm.off[t >> 1];
#pragma unroll
        for (int j = 1; j >= 0; --j) {
          const int tt = t + j, e2 = e + j;
          const float2 dlp = j ? hi2(dl4) : lo2(dl4);
          const float2 dup = j ? hi2(du4) : lo2(du4);
          const float2 gp = j ? hi2(g4) : lo2(g4);
          const float2 ofp = j ? hi2(of4) : lo2(of4);
          const float4 bd = bdr[tt * 2 * NSP], cd = cdr[tt * 2 * NSP];
          const float2 pF = make_float2(bitsf(hb[4 * e2]), bitsf(hb[4 * e2 + 1]));
          const float2 pS = make_float2(bitsf(hb[4 * e2 + 2]), bitsf(hb[4 * e2 + 3]));
          const float2 aF = ex2x2(fma2(dlp, AF, ofp)), aS = ex2x2(fma2(dlp, AS, ofp));
          float2 dhF = fma2(lo2(cd), gp, rF);  // total gradient w.r.t. h_t
          float2 dhS = fma2(hi2(cd), gp, rS);
          if constexpr (kStates) {
            if ((evF >> tt) & 1u) {
              dhF = __fadd2_rn(dhF, state_pair(a.dh_final, tt, nF));
              dhS = __fadd2_rn(dhS, state_pair(a.dh_final, tt, nS));
            }
          }
          const float2 qF = mul2(dhF, pF), qS = mul2(dhS, pS);
          dAF = fma2(dlp, qF, dAF);
          dAS = fma2(dlp, qS, dAS);
          const float2 s1 = fma2(dhS, hi2(bd), mul2(dhF, lo2(bd)));
          const float2 s2 = fma2(AS, qS, mul2(AF, qF));
          sm.nred[((buf * kRB + e2) * NSP + sp) * kCP + cp] = make_float4(s1.x, s1.y, s2.x, s2.y);
          if constexpr (kRecY) {  // C.h_t partials for y, h_t = p_t + delta u B
            const float2 yv = fma2(hi2(cd), fma2(dup, hi2(bd), pS), mul2(lo2(cd), fma2(dup, lo2(bd), pF)));
            sm.nY[((buf * kRB + e2) * NSP + sp) * kCP + cp] = yv;
          }
          // dB contributions dh_t delta u over the pair's channels, then over the tile's
          float sum;
          if (colsum.feed(4 * buf + e2, false, hsum(mul2(dup, dhF)), hsum(mul2(dup, dhS)), lane, &sum)) {
            const int ts = tt + ColSum8::token(lane);
            if (ts < rows) pdB[ts] = sum;
          }
          if constexpr (kStates) {
            if (((evG >> tt) & 1u) && valid &&
                VSSM_CHECKED((unsigned)a.seq[t0 + tt] < (unsigned)a.num_seqs, a.status)) {
              // the gradient reaching the starting state: dh_t times a's own value
              const float2 gF = mul2(dhF, ex2x2(mul2(dlp, AF))), gS = mul2(dhS, ex2x2(mul2(dlp, AS)));
              float* row = a.dh_init + ((int64_t)a.seq[t0 + tt] * a.D + d) * N;
              row[nF] = gF.x;
              row[N + nF] = gF.y;
              row[nS] = gS.x;
              row[N + nS] = gS.y;
            }
          }
          rF = mul2(dhF, aF);  // carry to h_{t-1}
          rS = mul2(dhS, aS);
        }
      }
    };
    // du and d delta_raw (and dz when y is recomputed) of block blk: 64
    // (token, channel pair) items, taken by warps 0-1 for even blocks and
    // 2-3 for odd ones when the CTA has 4 warps; the state pairs' partials are
    // added in order
    auto finalize = [&](int blk) {
      const int buf = blk & 1;
      constexpr int kFin = kThr >= 128 ? 64 : kThr;
      const bool mine = kThr >= 128 ? ((tid >> 6) == (blk & 1)) : true;
      if (!mine) return;
      for (int i = tid & (kFin - 1); i < kRB * kCP; i += kFin) {
        const int e = i >> 4, q = i & 15;
        const int t = blk * kRB + e;
        const float4* np = sm.nred + (buf * kRB + e) * NSP * kCP + q;
        float4 s = np[0];
#pragma unroll
        for (int v = 1; v < NSP; ++v) s = add4(s, np[v * kCP]);
        const float2 dlv = sm.dl[q * kPT + t], gv = sm.g[q * kPT + t], sgv = sm.sg[q * kPT + t];
        const int at = t * bx + 2 * q;
        const float2 uv = ld_io2(sm.u + at);
        const float2 dsk = a.Dskip ? make_float2(sm.dsk[(2 * q) & 31], sm.dsk[(2 * q + 1) & 31]) : make_float2(0.0f, 0.0f);
        const float2 du = fma2(dlv, lo2(s), mul2(dsk, gv));
        const float2 ddr = mul2(fma2(uv, lo2(s), mul2(hi2(s), splat2(kLn2))), sgv);
        const bool ok = t < rows && 2 * q < bx && d0 + 2 * q < a.D;
        if (ok) {
          const int64_t o2 = (t0 + t) * a.D + d0 + 2 * q;
          st_io2(gdu + o2, du);
          st_io2(gddr + o2, ddr);
          if constexpr (kRecY) {
            const float2* yp = sm.nY + (buf * kRB + e) * NSP * kCP + q;
            float2 ys = yp[0];
#pragma unroll
            for (int v = 1; v < NSP; ++v) ys = __fadd2_rn(ys, yp[v * kCP]);
            st_io2(gdz + o2, mul2(sm.dzf[q * kPT + t], fma2(dsk, uv, ys)));
          }
        }
        accB = __fadd2_rn(accB, ddr);  // zero past the last token and on missing channels
      }
    };
    // (the tensor-memory instructions are warp-collective: each follows a
    // __syncwarp so that the warp is converged)
    uint32_t hb0[16], hb1[16];
    __syncwarp();
    tmem_ld16(thist + 4 * kRB * (kL / kRB - 1), hb1);
    tmem_wait_ld16(hb1);
#pragma unroll 1
    for (int bp = kL / (2 * kRB) - 1; bp >= 0; --bp) {
      // block 2 bp + 1 from hb1, while block 2 bp's history loads into hb0
      __syncwarp();
      tmem_ld16(thist + 4 * kRB * (2 * bp), hb0);
      block(std::integral_constant<int, 1>{}, bp, hb1);
      __syncwarp();
      tmem_wait_ld16(hb0);
      __syncthreads();  // the block's partials are complete
      finalize(2 * bp + 1);
      __syncwarp();
      if (bp > 0) tmem_ld16(thist + 4 * kRB * (2 * bp - 1), hb1);
      block(std::integral_constant<int, 0>{}, bp, hb0);
      __syncwarp();
      if (bp > 0) tmem_wait_ld16(hb1);
      __syncthreads();
      finalize(2 * bp);
    }
  }

  // ---- 5. dA partials of the chunk ([chunk][n][d]); fixed-order CTA sums of
  //         the dDskip and d_dt_bias partials
  if (valid) {
    // for A_log the chain rule gives dA_log = dA * A (A = A2 ln 2), applied to
    // every chunk's partial before the fixed-order sum
    const float2 sF = a.a_log ? mul2(AF, splat2(kLn2)) : make_float2(1.0f, 1.0f);
    const float2 sS = a.a_log ? mul2(AS, splat2(kLn2)) : make_float2(1.0f, 1.0f);
    *reinterpret_cast<float2*>(a.part_dA + ((int64_t)chunk * N + nF) * a.D + d) = mul2(dAF, sF);
    *reinterpret_cast<float2*>(a.part_dA + ((int64_t)chunk * N + nS) * a.D + d) = mul2(dAS, sS);
  }
  sm.redD[tid] = accD;
  sm.redB[tid] = accB;
  __syncthreads();
  // no input buffer is read any more: request the next item's inputs, which
  // land while this item writes its last partials
  if (tid == 0) {
    sm.ticket = next;
    if (next < n_items) issue(next);
  }
  if (tid < kCP && d0 + 2 * tid < a.D && 2 * tid < bx) {
    float2 sD = make_float2(0.0f, 0.0f), sB = make_float2(0.0f, 0.0f);
    for (int v = tid; v < kThr; v += kCP) {
      sD = __fadd2_rn(sD, sm.redD[v]);
      sB = __fadd2_rn(sB, sm.redB[v]);
    }
    *reinterpret_cast<float2*>(a.part_dD + (int64_t)chunk * a.D + d0 + 2 * tid) = sD;
    *reinterpret_cast<float2*>(a.part_dbias + (int64_t)chunk * a.D + d0 + 2 * tid) = sB;
  }
  __syncthreads();  // redD / redB and the ticket are consumed before the next pass
  }  // persistent loop

  // every warp's tensor-memory accesses are complete (waited) before the free
  tmem_fence_before_sync();
  __syncthreads();
  if (w == 0) {
    tmem_fence_after_sync();
    tmem_dealloc128(sm.taddr);
  }
}

// ============================================================================
// N = 16: a thread owns two channel pairs and one state pair
// ============================================================================
// Work item = 32 tokens x kTW = 64 channels; CTA = 4 warps in two channel
// groups (warps 2g, 2g+1 take the channels 32g .. 32g+31).  A thread owns a
// channel quad q of its group (channels 4q .. 4q+3: two pairs for the paired
// FP32 instructions) and a state pair p of its warp's four (p = 4 (w % 2) ..
// +3): eight (channel, state) chains; the lane map is given in the kernel.
// Against the pair-by-pair layout above, every per-token value a thread
// loads serves twice the chains, the channel sums for dB / dC start over 4
// channels in registers, and the history takes 8 words per token (256
// tensor-memory columns per warp, 2 CTAs per SM).  The partial
// sums over state pairs for du / d delta_raw come from the two warps of a
// channel group only, so a block's epilogue waits on a 64-thread named
// barrier, not on the whole CTA; each block is finalized after the walk over
// the next one.  The next item's copies are split over the four warps, two
// each (the barrier takes four arrivals).  Fewer shared-memory loads pay here even at
// the cost of register moves: B and C arrive packed, (B_n, B_m, C_n, C_m) in
// one 16-byte row per token and state pair, each value splatted for the paired
// instructions, and the exponent offsets are selects on the start ballot.
// For bf16 I/O step 1 keeps d delta / d delta_raw (a by-product of softplus)
// for the finalize, which otherwise recomputes it from delta_raw.
constexpr int kTW = 2 * kTile;  // 64 channels per work item
constexpr int kCQ = kTW / 4;    // 16 channel quads
constexpr int kQT = kL + 1;     // token pitch (float4) of the [channel quad][token] arrays
constexpr int kSP = 8;          // state pairs

template <typename T, bool kRecY>
struct Bwd16Smem {
  alignas(128) T u[kL * kTW];
  alignas(128) T dr[kL * kTW];
  alignas(128) T z[kL * kTW];
  alignas(128) T dout[kL * kTW];
  alignas(128) T y[kL * kTW];
  alignas(128) float H[16 * kTW];  // saved states at the chunk start, [n][channel]
  // the tile's parameters as one copy brings them (ScanArgs::tpar): A * log2 e
  // [channel][n], dt_bias, Dskip
  alignas(16) float Araw[kTW * 16];
  alignas(16) float bias[kTW];
  alignas(16) float dsk[kTW];
  // ---- per-(token, channel quad) values, [quad][token] float4 with token
  //      pitch kQT: the 8 quads a warp reads for a token are in distinct banks
  alignas(16) float4 dl[kCQ * kQT];   // delta
  alignas(16) float4 dlu[kCQ * kQT];  // delta * u
  alignas(16) float4 g[kCQ * kQT];    // dout * (SiLU(z) + gate floor)
  // d delta / d delta_raw = sigmoid(delta_raw + dt_bias), for bf16 I/O (the
  // fp32 tiles leave no room: the finalize recomputes it there)
  alignas(16) float4 sg[sizeof(T) == 2 ? kCQ * kQT : 1];
  // ---- B and C packed, [token][state pair][order] float4 = (B_n, B_m, C_n,
  //      C_m), (n, m) the pair in the thread's order
  alignas(16) float4 BC[kL * kSP * 2];
  alignas(16) int pos[kL];  // the chunk's position indices (zero past T), copied with BC
  // ---- partial sums over each thread's state pair from the reverse walk,
  //      [buffer][token of the block][state pair][channel pair parity][quad]
  //      float4 = (sum dh B for the pair's two channels, sum A dh p for them)
  alignas(16) float4 nred[2 * kRB * kSP * 2 * kCQ];
  // C.h partials, when y is recomputed: [buffer][token of the block][warp of
  // the group][group][channel of the group], each summed over the warp's
  // four state pairs
  alignas(16) float ysum[kRecY ? 2 * kRB * 2 * 2 * kTile : 2];
  alignas(16) float4 redD[128];
  alignas(16) float2 redB[128];
  uint32_t taddr;
  int ticket;
  alignas(8) uint64_t bar;
};

// Column sums over the 8 lanes of a warp that share a state pair for groups
// of 4 tokens x 2 states, by shuffle butterflies.  The 8 lanes differ in lane
// bits 0 and 1 (channel quads) and in bits 3 and 4 together (the quarter-warps
// k and k ^ 3).  Level 1 exchanges states over lane bit 0 (a lane keeps its
// first state, 2p + bit 0: lanes l and l ^ 1 hold the pair in opposite
// orders), level 2 pairs tokens over bit 1, level 3 over the quarter pair
// (xor 24, the upper quarter of the two keeping the odd pair).  After the 4th
// token, lane l holds the sum over the 8 lanes for token bit1(l) + 2 bit4(l)
// of the group.
struct ColSum4 {
  float p2[2], p3[2];

  static __device__ __forceinline__ int token(int lane) { return ((lane >> 1) & 1) + 2 * ((lane >> 4) & 1); }

  // lo + hi over the lane pair (l, l ^ xor_mask): the lane with up_bit set
  // keeps the hi sum, its partner the lo sum
  static __device__ __forceinline__ float combine(float lo, float hi, int lane, int xor_mask, int up_bit) {
    const bool up = (lane & up_bit) != 0;
    return (up ? hi : lo) + __shfl_xor_sync(0xffffffffu, up ? lo : hi, xor_mask);
  }

  __device__ __forceinline__ bool feed(int c, bool ascending, float vF, float vS, int lane, float* sum) {
    p2[c & 1] = vF + __shfl_xor_sync(0xffffffffu, vS, 1);
    if ((c & 1) != (ascending ? 1 : 0)) return false;
    p3[(c >> 1) & 1] = combine(p2[0], p2[1], lane, 2, 2);
    if ((c & 3) != (ascending ? 3 : 0)) return false;
    *sum = combine(p3[0], p3[1], lane, 24, 16);
    return true;
  }
};

// Index (float4 or float2 units) of the n-sum partial of state pair sp,
// channel pair j of quad cq, token e of buffer buf.  The quad is swizzled by
// the parity of j and sp so that the walk's stores (a quarter-warp: 4 quads x
// 2 state pairs, fixed j) and the finalize's loads (a quarter-warp: 4 quads x
// 2 pairs j, fixed sp) each hit 8 distinct 16-byte bank groups.
__device__ __forceinline__ int nred_at(int buf, int e, int sp, int j, int cq) {
  return ((buf * kRB + e) * kSP + sp) * 2 * kCQ + j * kCQ + (cq ^ (4 * (j ^ (sp & 1))));
}

__device__ __forceinline__ void st_io4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st_io4(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 a = __float22bfloat162_rn(make_float2(v.x, v.y));
  const __nv_bfloat162 b = __float22bfloat162_rn(make_float2(v.z, v.w));
  uint2 q;
  q.x = *reinterpret_cast<const uint32_t*>(&a);
  q.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = q;
}
__device__ __forceinline__ float4 mk4(float2 lo, float2 hi) { return make_float4(lo.x, lo.y, hi.x, hi.y); }

template <typename T, bool kStates, bool kRecY, bool kKnob>
__global__ void __launch_bounds__(128, 2)
scan_bwd16_kernel(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dr,
                  const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_dout,
                  const __grid_constant__ CUtensorMap tm_cs, const __grid_constant__ CUtensorMap tm_y,
                  const ScanArgs a) {
  constexpr int N = 16;
  constexpr int kThr = 128;
  using SM = Bwd16Smem<T, kRecY>;
  // one bulk copy fills each of these runs of shared memory
  static_assert(offsetof(SM, pos) == offsetof(SM, BC) + sizeof(SM::BC) &&
                    sizeof(SM::BC) + sizeof(SM::pos) == kBwdChunkRow,
                "B / C rows and positions must be contiguous");
  static_assert(offsetof(SM, bias) == offsetof(SM, Araw) + sizeof(SM::Araw) &&
                    offsetof(SM, dsk) == offsetof(SM, bias) + sizeof(SM::bias) &&
                    sizeof(SM::Araw) + sizeof(SM::bias) + sizeof(SM::dsk) == kBwdTileParams * 4,
                "the tile's parameters must be contiguous");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SM& sm = *reinterpret_cast<SM*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int n_items = a.n_chunks * a.n_tiles;
  // Lane map: quarter-warp k = lane / 8 holds 4 channel quads x 2 state pairs,
  // the quads 4 (k % 2) .. +3 of the group and the state pairs
  // 2 ((k % 2) ^ (k / 2)) .. +1 of the warp's four.  The two quarters of a
  // half-warp then read disjoint quads (per-(token, channel) values) and
  // disjoint state pairs (B, C), so a 16-byte load of either kind is two
  // shared-memory wavefronts per warp, not four.
  const int grp = w >> 1;                          // channel group
  const int qk = lane >> 3, qr = lane & 7;
  const int cq = 8 * grp + 4 * (qk & 1) + (qr & 3);                 // channel quad of the tile
  const int sp = 4 * (w & 1) + 2 * ((qk & 1) ^ (qk >> 1)) + (qr >> 2);  // state pair
  const int o = lane & 1;                          // this lane's state order
  const int nF = 2 * sp + o, nS = 2 * sp + 1 - o;  // its "first" and "second" state
  const int c0 = 4 * cq;                           // first channel of the quad (in the tile)

  // The item's eight copies, two per warp: lane 0 of warp wq posts its
  // share's bytes on the barrier (which expects four arrivals) and issues its
  // copies.  One thread issuing twelve copies in turn spent about 1.4k cycles
  // on them while the rest of the CTA waited, and a warp's copies still issue
  // one after another: the chunk's B / C rows come with its positions, and the
  // tile's A rows with dt_bias and Dskip, each in one copy (built per call).
  auto issue = [&](int tkn, int wq) {
    const int rv = tkn / a.n_tiles;
    const int tl = tkn - rv * a.n_tiles;
    const int ch = a.n_chunks - 1 - rv;
    const int64_t tt0 = (int64_t)ch * kL;
    const int dd0 = tl * kTW;
    const uint32_t box = (uint32_t)a.box_x * (uint32_t)a.box_y * sizeof(T);
    if (wq == 0) {
      mbar_arrive_expect_tx(&sm.bar, 2u * box);
      tma_load_2d(sm.u, &tm_u, dd0, (int)tt0, &sm.bar);
      tma_load_2d(sm.dr, &tm_dr, dd0, (int)tt0, &sm.bar);
    } else if (wq == 1) {
      mbar_arrive_expect_tx(&sm.bar, box * (1u + (a.has_z ? 1u : 0u)));
      tma_load_2d(sm.dout, &tm_dout, dd0, (int)tt0, &sm.bar);
      if (a.has_z) tma_load_2d(sm.z, &tm_z, dd0, (int)tt0, &sm.bar);
    } else if (wq == 2) {
      mbar_arrive_expect_tx(&sm.bar, box * (a.has_y ? 1u : 0u) + (uint32_t)a.box_x * N * 4u);
      if (a.has_y) tma_load_2d(sm.y, &tm_y, dd0, (int)tt0, &sm.bar);
      tma_load_2d(sm.H, &tm_cs, dd0, ch * N, &sm.bar);
    } else {
      // the chunk's B / C rows with its positions, and the tile's parameters
      mbar_arrive_expect_tx(&sm.bar, (uint32_t)kBwdChunkRow + kBwdTileParams * 4u);
      bulk_load_1d(sm.BC, a.BD + (int64_t)ch * (kBwdChunkRow / 16), kBwdChunkRow, &sm.bar);
      bulk_load_1d(sm.Araw, a.tpar + (int64_t)tl * kBwdTileParams, kBwdTileParams * 4u, &sm.bar);
    }
  };

  // tensor memory for the forward walk's history: 256 columns, warp w on the
  // lanes 32 w .. 32 w + 31
  if (w == 0) tmem_alloc256(&sm.taddr);
  if (tid == 0) {
    mbar_init(&sm.bar, 4);
    fence_mbar_init();
    sm.ticket = (int)atomicAdd(a.ticket, 1u);
  }
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (lane == 0 && sm.ticket < n_items) issue(sm.ticket, w);
  const uint32_t thist = sm.taddr + ((uint32_t)(32 * w) << 16);

  for (uint32_t it = 0;; ++it) {
  const int tk = sm.ticket;
  if (tk >= n_items) break;
  if constexpr (kKnob) {
    if ((long long)tk == a.delay_ticket) sleep_ns(a.delay_ns);
  }
  const int rev = tk / a.n_tiles;
  const int tile = tk - rev * a.n_tiles;
  const int chunk = a.n_chunks - 1 - rev;
  const int64_t t0 = (int64_t)chunk * kL;
  const int rows = (int)((a.T - t0) < kL ? (a.T - t0) : kL);
  const int d0 = tile * kTW;
  const int bx = a.box_x;
  const int d = d0 + c0;                   // first channel of this thread's quad
  const bool valid = c0 < bx && d < a.D;   // D is a multiple of 4: the quad is whole

  if (!__syncthreads_and(mbar_wait(&sm.bar, it & 1u, a.wait_ns))) {
    // see scan_bwd_kernel: report, give the copies a second limit, stop
    if (tid == 0) atomicOr(a.status, kStatusTmaTimeout);
    mbar_wait(&sm.bar, it & 1u, kCopyDrainNs);
    break;
  }

  // ---- 1. per-(token, channel quad) values (zero past the last token and on
  //         channels past D), and dz from the pre-gate output y
  float4 accD = make_float4(0.0f, 0.0f, 0.0f, 0.0f);  // dDskip partial of quad tid % 16
  {
    T* gdz = static_cast<T*>(a.dz);
    const int q = tid & 15;
    const float4 bias4 = a.dt_bias ? *reinterpret_cast<const float4*>(sm.bias + 4 * q) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
    for (int i = tid; i < kL * kCQ; i += kThr) {
      const int t = i >> 4;
      const int at = t * bx + 4 * q;
      const bool ok = t < rows && 4 * q < bx && d0 + 4 * q < a.D;
      const float4 r4 = ld_io4(sm.dr + at);
      const float4 u4 = ld_io4(sm.u + at);
      const float4 go = ld_io4(sm.dout + at);
      const float2 rlo = __fadd2_rn(lo2(r4), lo2(bias4)), rhi = __fadd2_rn(hi2(r4), hi2(bias4));
      float4 dl4, sg4 = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
      if (a.delta_softplus) {
        dl4 = make_float4(softplus_sig(rlo.x, &sg4.x), softplus_sig(rlo.y, &sg4.y),
                          softplus_sig(rhi.x, &sg4.z), softplus_sig(rhi.y, &sg4.w));
      } else {
        dl4 = mk4(rlo, rhi);
      }
      if constexpr (sizeof(T) == 2) sm.sg[q * kQT + t] = sg4;
      float4 gv = go;
      if (a.has_z) {
        const float4 z4 = ld_io4(sm.z + at);
        const float4 s4 = make_float4(sigmoidf_fast(z4.x), sigmoidf_fast(z4.y), sigmoidf_fast(z4.z),
                                      sigmoidf_fast(z4.w));
        const float2 glo = mul2(lo2(go), fma2(lo2(z4), lo2(s4), splat2(a.gate_floor)));
        const float2 ghi = mul2(hi2(go), fma2(hi2(z4), hi2(s4), splat2(a.gate_floor)));
        gv = mk4(glo, ghi);
        // d out / d y = dout SiLU'(z), SiLU'(z) = s (1 + z (1 - s))
        const float2 flo = mul2(mul2(lo2(go), lo2(s4)),
                                fma2(lo2(z4), make_float2(1.0f - s4.x, 1.0f - s4.y), splat2(1.0f)));
        const float2 fhi = mul2(mul2(hi2(go), hi2(s4)),
                                fma2(hi2(z4), make_float2(1.0f - s4.z, 1.0f - s4.w), splat2(1.0f)));
        if (a.has_y) {
          if (ok) {
            const float4 y4 = ld_io4(sm.y + at);
            st_io4(gdz + (t0 + t) * a.D + d0 + 4 * q, mk4(mul2(flo, lo2(y4)), mul2(fhi, hi2(y4))));
          }
        }
      }
      const float4 z0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      sm.dl[q * kQT + t] = ok ? dl4 : z0;
      sm.dlu[q * kQT + t] = ok ? mk4(mul2(lo2(dl4), lo2(u4)), mul2(hi2(dl4), hi2(u4))) : z0;
      sm.g[q * kQT + t] = ok ? gv : z0;
      if (ok) accD = mk4(fma2(lo2(gv), lo2(u4), lo2(accD)), fma2(hi2(gv), hi2(u4), hi2(accD)));
    }
  }
  const unsigned rst = __ballot_sync(0xffffffffu, lane < rows && sm.pos[lane] == 0);
  unsigned evH = 0u, evG = 0u, evF = 0u;
  if (kStates && a.seq) {
    const unsigned live = rows >= 32 ? 0xffffffffu : ((1u << rows) - 1u);
    const unsigned starts = rst & live;
    evH = a.h_init ? starts : 0u;
    evG = a.dh_init ? starts : 0u;
    if (a.dh_final) {
      unsigned ends = starts >> 1;
      if (t0 + rows >= a.T || (rows == 32 && __ldg(a.pos + t0 + 32) == 0)) ends |= 1u << (rows - 1);
      evF = ends & live;
    }
  }
  // sequence-state entries (channels d + 2j, d + 2j + 1) of state n for token t's sequence
  auto state_pair = [&](const float* st, int t, int n, int j) {
    if (!valid || !VSSM_CHECKED((unsigned)a.seq[t0 + t] < (unsigned)a.num_seqs, a.status))
      return make_float2(0.0f, 0.0f);
    const float* row = st + ((int64_t)a.seq[t0 + t] * a.D + d + 2 * j) * N + n;
    return make_float2(__ldg(row), __ldg(row + N));
  };
  __syncthreads();

  // A * log2 e pairs [state F / S][channel pair] and the saved states
  float2 A[2][2], h[2][2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int n = q ? nS : nF;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      A[q][j] = make_float2(0.0f, 0.0f);
      h[q][j] = make_float2(0.0f, 0.0f);
      if (valid) {
        A[q][j] = make_float2(sm.Araw[(c0 + 2 * j) * N + n], sm.Araw[(c0 + 2 * j + 1) * N + n]);
        h[q][j] = *reinterpret_cast<const float2*>(sm.H + n * bx + c0 + 2 * j);
      }
    }
  }
  const float4* const dlr = sm.dl + cq * kQT;
  const float4* const dur = sm.dlu + cq * kQT;
  const float4* const gr = sm.g + cq * kQT;
  const float4* const bcr = sm.BC + sp * 2 + o;  // entry of token t at [t * 2 kSP]
  const int part = 2 * tile + grp;               // 32-channel partial row group
  float* const pdB = a.part_dBC + ((int64_t)part * 2 * N + nF) * a.T + t0;
  float* const pdC = a.part_dBC + ((int64_t)part * 2 * N + N + nF) * a.T + t0;

  // the right neighbour's inclusive carry words, first read two groups before
  // the walk ends (that chunk started about a fifth of an item earlier and
  // has nearly always stored them by then), so the read's round trip is over
  // when the look-back checks them
  const bool has_right = chunk < a.n_chunks - 1;
  const float4* const right_carry =
      reinterpret_cast<const float4*>(a.incl) + (((int64_t)tile * a.n_chunks + chunk + 1) * kThr + tid) * 2;
  float4 early_lo = make_float4(0.0f, 0.0f, 0.0f, 0.0f), early_hi = early_lo;

  // ---- 2. forward walk; p_t = a_t h_{t-1} (8 words per token) to tensor memory
  float2 E[2][2], tot[2][2];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      E[q][j] = make_float2(1.0f, 1.0f);
      tot[q][j] = make_float2(0.0f, 0.0f);
    }
  {
    ColSum4 colsum;
    // the group's dC sum is stored during the next group, once its shuffles
    // have long completed (no stall on them)
    float pend = 0.0f;
    int pend_t = kL;
#pragma unroll 1
    for (int g4 = 0; g4 < kL / 4; ++g4) {
      if (g4 == kL / 4 - 2 && has_right) {
        early_lo = ld_carry4(right_carry);
        early_hi = ld_carry4(right_carry + 1);
      }
      uint32_t hist[32];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tt = 4 * g4 + e;
        if (e == 2 && pend_t < rows) pdC[pend_t] = pend;
        const float4 dl4 = dlr[tt], du4 = dur[tt], gq = gr[tt];
        // exponent offset: -inf at a sequence start (the factor is zeroed)
        const float2 ofp = splat2(((rst >> tt) & 1u) ? -INFINITY : 0.0f);
        const float4 bc = bcr[tt * 2 * kSP];
        const float2 dlp[2] = {lo2(dl4), hi2(dl4)}, dup[2] = {lo2(du4), hi2(du4)}, gp[2] = {lo2(gq), hi2(gq)};
        float v[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float2 Bq = splat2(q ? bc.y : bc.x), Cq = splat2(q ? bc.w : bc.z);
          const int n = q ? nS : nF;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float2 at = ex2x2(fma2(dlp[j], A[q][j], ofp));
            float2 p = mul2(at, h[q][j]);
            if constexpr (kStates) {
              if ((evH >> tt) & 1u) p = mul2(ex2x2(mul2(dlp[j], A[q][j])), state_pair(a.h_init, tt, n, j));
            }
            h[q][j] = fma2(dup[j], Bq, p);
            E[q][j] = mul2(E[q][j], at);
            tot[q][j] = fma2(E[q][j], mul2(Cq, gp[j]), tot[q][j]);
            if constexpr (kStates) {
              if ((evF >> tt) & 1u) tot[q][j] = fma2(E[q][j], state_pair(a.dh_final, tt, n, j), tot[q][j]);
            }
            hist[8 * e + 4 * q + 2 * j] = fbits(p.x);
            hist[8 * e + 4 * q + 2 * j + 1] = fbits(p.y);
          }
          v[q] = hsum(fma2(gp[1], h[q][1], mul2(gp[0], h[q][0])));
        }
        // dC contributions g_t h_t over the quad's channels, then over the group's
        if (colsum.feed(e, true, v[0], v[1], lane, &pend)) pend_t = 4 * g4 + ColSum4::token(lane);
      }
      // the store reads its registers when it issues; the reverse walk waits
      // for the stores to land before its first load
      __syncwarp();
      tmem_st32(thist + (uint32_t)(32 * g4), hist);
    }
    if (pend_t < rows) pdC[pend_t] = pend;
    tmem_wait_st();
  }

  // ---- 3. decoupled look-back towards higher chunks (one chain per thread, 8 words)
  float4 xlo = make_float4(0.0f, 0.0f, 0.0f, 0.0f), xhi = xlo;
  {
    const int64_t base = (int64_t)tile * a.n_chunks;
    const int64_t wslot = ((base + chunk) * kThr + tid) * 2;
    const bool publish = (long long)tk != a.drop_ticket;
    float4* const agg = reinterpret_cast<float4*>(a.agg);
    float4* const aggp = reinterpret_cast<float4*>(a.agg_sd);
    float4* const inc = reinterpret_cast<float4*>(a.incl);
    int* const my_flag = a.flags + (base + chunk) * 4 + w;
    const float4 tlo = mk4(tot[0][0], tot[0][1]), thi = mk4(tot[1][0], tot[1][1]);
    const float4 elo = mk4(E[0][0], E[0][1]), ehi = mk4(E[1][0], E[1][1]);
    const bool rs_any = (rst & (rows >= 32 ? 0xffffffffu : ((1u << rows) - 1u))) != 0u;
    if (rs_any && publish) {
      st_carry4(inc + wslot, tlo);
      st_carry4(inc + wslot + 1, thi);
    }
    auto combine8 = [&](float4 p_lo, float4 p_hi, float4 q_lo, float4 q_hi) {
      xlo = mk4(fma2(lo2(p_lo), lo2(xlo), lo2(q_lo)), fma2(hi2(p_lo), hi2(xlo), hi2(q_lo)));
      xhi = mk4(fma2(lo2(p_hi), lo2(xhi), lo2(q_hi)), fma2(hi2(p_hi), hi2(xhi), hi2(q_hi)));
    };
    if (chunk < a.n_chunks - 1) {
      int j = chunk + 1, found = -1, timed_out = 0;
      float4 vlo = early_lo, vhi = early_hi;  // read during the forward walk
      if (__all_sync(0xffffffffu, carry_set4(vlo) && carry_set4(vhi))) {
        found = j;
      } else {
        if (!rs_any) {
          agg[wslot] = tlo;
          agg[wslot + 1] = thi;
          aggp[wslot] = elo;
          aggp[wslot + 1] = ehi;
          publish_flag(my_flag, kFlagAggregate, publish, lane);
        }
        const uint64_t t_start = globaltimer_ns();
        while (j < a.n_chunks) {
          const int64_t ks = ((base + j) * kThr + tid) * 2;
          unsigned backoff = 32;
          int f = kFlagNone;
          for (;;) {
            vlo = ld_carry4(inc + ks);
            vhi = ld_carry4(inc + ks + 1);
            if (__all_sync(0xffffffffu, carry_set4(vlo) && carry_set4(vhi))) { f = kFlagInclusive; break; }
            if (__all_sync(0xffffffffu, ld_acquire_gpu(a.flags + (base + j) * 4 + w) == kFlagAggregate)) {
              f = kFlagAggregate;
              break;
            }
            if (__shfl_sync(0xffffffffu, globaltimer_ns() - t_start > a.wait_ns, 0)) break;
            __nanosleep(backoff);
            if (backoff < 1024) backoff <<= 1;
          }
          if (f == kFlagInclusive) { found = j; break; }
          if (f == kFlagNone) { timed_out = 1; break; }
          ++j;
        }
      }
      if (timed_out) atomicOr(a.status, kStatusLookbackTimeout);
      int last = j - 1;
      if (found >= 0) {
        xlo = vlo;
        xhi = vhi;
        last = found - 1;
      }
      for (int i = last; i > chunk; --i) {
        const int64_t ws = ((base + i) * kThr + tid) * 2;
        combine8(__ldcg(aggp + ws), __ldcg(aggp + ws + 1), __ldcg(agg + ws), __ldcg(agg + ws + 1));
      }
    }
    if (!rs_any && publish) {
      st_carry4(inc + wslot, mk4(fma2(lo2(elo), lo2(xlo), lo2(tlo)), fma2(hi2(elo), hi2(xlo), hi2(tlo))));
      st_carry4(inc + wslot + 1, mk4(fma2(lo2(ehi), lo2(xhi), lo2(thi)), fma2(hi2(ehi), hi2(xhi), hi2(thi))));
    }
  }

  // ---- 4. reverse walk in blocks of kRB tokens
  float2 dA[2][2];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int j = 0; j < 2; ++j) dA[q][j] = make_float2(0.0f, 0.0f);
  float2 accB = make_float2(0.0f, 0.0f);  // d_dt_bias partial of this thread's epilogue pair
  int next = 0;
  {
    T* gdu = static_cast<T*>(a.du);
    T* gddr = static_cast<T*>(a.ddr);
    T* gdz = static_cast<T*>(a.dz);
    float2 r[2][2] = {{lo2(xlo), hi2(xlo)}, {lo2(xhi), hi2(xhi)}};
    float pendB = 0.0f;
    int pendB_t = kL;
    auto block = [&](auto parity, int bp, uint32_t (&hb)[32]) {
      constexpr int buf = decltype(parity)::value;
      const int blk = 2 * bp + buf;
      // the next ticket, drawn a block ahead of the tail so that its round
      // trip is over when the tail hands it to the copies
      if (blk == 1 && tid == 0) next = (int)atomicAdd(a.ticket, 1u);
      ColSum4 colsum;
#pragma unroll
      for (int e = kRB - 1; e >= 0; --e) {
        const int tt = blk * kRB + e;
        // the previous block's dB sum, long since complete
        if (e == kRB - 2 && pendB_t < rows) pdB[pendB_t] = pendB;
        const float4 dl4 = dlr[tt], du4 = dur[tt], gq = gr[tt];
        // exponent offset: -inf at a sequence start (the factor is zeroed)
        const float2 ofp = splat2(((rst >> tt) & 1u) ? -INFINITY : 0.0f);
        const float4 bc = bcr[tt * 2 * kSP];
        const float2 dlp[2] = {lo2(dl4), hi2(dl4)}, dup[2] = {lo2(du4), hi2(du4)}, gp[2] = {lo2(gq), hi2(gq)};
        float2 dh[2][2], qq[2][2], at[2][2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float2 Cq = splat2(q ? bc.w : bc.z);
          [[maybe_unused]] const int n = q ? nS : nF;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float2 p = make_float2(bitsf(hb[8 * e + 4 * q + 2 * j]), bitsf(hb[8 * e + 4 * q + 2 * j + 1]));
            at[q][j] = ex2x2(fma2(dlp[j], A[q][j], ofp));
            dh[q][j] = fma2(Cq, gp[j], r[q][j]);
            if constexpr (kStates) {
              if ((evF >> tt) & 1u) dh[q][j] = __fadd2_rn(dh[q][j], state_pair(a.dh_final, tt, n, j));
            }
            qq[q][j] = mul2(dh[q][j], p);
            dA[q][j] = fma2(dlp[j], qq[q][j], dA[q][j]);
          }
        }
        const float2 BF = splat2(bc.x), BS = splat2(bc.y);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 s1 = fma2(dh[1][j], BS, mul2(dh[0][j], BF));
          const float2 s2 = fma2(A[1][j], qq[1][j], mul2(A[0][j], qq[0][j]));
          sm.nred[nred_at(buf, e, sp, j, cq)] = mk4(s1, s2);
        }
        if constexpr (kRecY) {
          // C.h_t over this thread's two states (h_t = p_t + delta u B), for
          // the quad's channel pairs; summed over the warp's four state pairs
          // of the quad (lanes l ^ 4, l ^ 16) so that lane l keeps channel
          // 2 bit2(l) + bit4(l) of its quad
          float2 yv[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float2 pF = make_float2(bitsf(hb[8 * e + 2 * j]), bitsf(hb[8 * e + 2 * j + 1]));
            const float2 pS = make_float2(bitsf(hb[8 * e + 4 + 2 * j]), bitsf(hb[8 * e + 4 + 2 * j + 1]));
            yv[j] = fma2(splat2(bc.w), fma2(dup[j], BS, pS), mul2(splat2(bc.z), fma2(dup[j], BF, pF)));
          }
          const bool b2 = (lane & 4) != 0, b4 = (lane & 16) != 0;
          float2 keep = b2 ? yv[1] : yv[0];
          const float2 send = b2 ? yv[0] : yv[1];
          keep.x += __shfl_xor_sync(0xffffffffu, send.x, 4);
          keep.y += __shfl_xor_sync(0xffffffffu, send.y, 4);
          float k1 = b4 ? keep.y : keep.x;
          k1 += __shfl_xor_sync(0xffffffffu, b4 ? keep.x : keep.y, 16);
          sm.ysum[((buf * kRB + e) * 2 + (w & 1)) * (2 * kTile) + grp * kTile + 4 * (cq - 8 * grp) + 2 * (b2 ? 1 : 0) +
                  (b4 ? 1 : 0)] = k1;
        }
        float wv[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) wv[q] = hsum(fma2(dup[1], dh[q][1], mul2(dup[0], dh[q][0])));
        // dB contributions dh_t delta u over the quad's channels, then over the
        // group's; stored during the next block (no stall on the shuffles)
        if (colsum.feed(e, false, wv[0], wv[1], lane, &pendB)) pendB_t = blk * kRB + ColSum4::token(lane);
        if constexpr (kStates) {
          if (((evG >> tt) & 1u) && valid &&
              VSSM_CHECKED((unsigned)a.seq[t0 + tt] < (unsigned)a.num_seqs, a.status)) {
            float* row = a.dh_init + ((int64_t)a.seq[t0 + tt] * a.D + d) * N;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int n = q ? nS : nF;
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const float2 gq2 = mul2(dh[q][j], ex2x2(mul2(dlp[j], A[q][j])));
                row[(2 * j) * N + n] = gq2.x;
                row[(2 * j + 1) * N + n] = gq2.y;
              }
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int j = 0; j < 2; ++j) r[q][j] = mul2(dh[q][j], at[q][j]);
      }
    };
    // du and d delta_raw (and dz when y is recomputed) of block blk for this
    // thread's channel group: item (token e, channel pair) per thread of the
    // group; the state pairs' partials are added in order
    // this thread's channel pair in every finalize, and its dt_bias / Dskip
    const int fin_cpl = tid & 15;
    const int fin_cp = 16 * grp + fin_cpl;
    const float2 fin_bias = a.dt_bias ? *reinterpret_cast<const float2*>(sm.bias + 2 * fin_cp) : make_float2(0.0f, 0.0f);
    const float2 fin_dsk = a.Dskip ? *reinterpret_cast<const float2*>(sm.dsk + 2 * fin_cp) : make_float2(0.0f, 0.0f);
    auto finalize = [&](int blk) {
      const int buf = blk & 1;
      const int e = (tid & 63) >> 4, cpl = fin_cpl;
      const int cp = fin_cp, hh = cp & 1, qd = cp >> 1;
      const int t = blk * kRB + e;
      float4 pv[kSP];
#pragma unroll
      for (int v = 0; v < kSP; ++v) pv[v] = sm.nred[nred_at(buf, e, v, hh, qd)];
      // fixed pairwise tree over the 8 state pairs
      const float4 s = add4(add4(add4(pv[0], pv[1]), add4(pv[2], pv[3])), add4(add4(pv[4], pv[5]), add4(pv[6], pv[7])));
      const float2 dlv = reinterpret_cast<const float2*>(sm.dl + qd * kQT + t)[hh];
      const float2 gv = reinterpret_cast<const float2*>(sm.g + qd * kQT + t)[hh];
      const int at = t * bx + 2 * cp;
      const float2 uv = ld_io2(sm.u + at);
      float2 sgv = make_float2(1.0f, 1.0f);
      if constexpr (sizeof(T) == 2) {
        sgv = reinterpret_cast<const float2*>(sm.sg + qd * kQT + t)[hh];
      } else if (a.delta_softplus) {  // d softplus / dx = sigmoid(delta_raw + dt_bias)
        const float2 rr = __fadd2_rn(ld_io2(sm.dr + at), fin_bias);
        sgv = make_float2(sigmoidf_fast(rr.x), sigmoidf_fast(rr.y));
      }
      const float2 dsk = fin_dsk;
      const float2 du = fma2(dlv, lo2(s), mul2(dsk, gv));
      const bool ok = t < rows && 2 * cp < bx && d0 + 2 * cp < a.D;
      const float2 ddr = ok ? mul2(fma2(uv, lo2(s), mul2(hi2(s), splat2(kLn2))), sgv) : make_float2(0.0f, 0.0f);
      if (ok) {
        const int64_t o2 = (t0 + t) * a.D + d0 + 2 * cp;
        st_io2(gdu + o2, du);
        st_io2(gddr + o2, ddr);
        if constexpr (kRecY) {
          // y = C.h (the two warps' sums, in warp order) + Dskip u, and
          // d out / d y = dout SiLU'(z), SiLU'(z) = s (1 + z (1 - s))
          const float* yr = sm.ysum + (buf * kRB + e) * 2 * (2 * kTile) + grp * kTile + 2 * cpl;
          const float2 ys = __fadd2_rn(*reinterpret_cast<const float2*>(yr),
                                       *reinterpret_cast<const float2*>(yr + 2 * kTile));
          const float2 zz = ld_io2(sm.z + at), go = ld_io2(sm.dout + at);
          const float2 sz = make_float2(sigmoidf_fast(zz.x), sigmoidf_fast(zz.y));
          const float2 f = mul2(mul2(go, sz), fma2(zz, make_float2(1.0f - sz.x, 1.0f - sz.y), splat2(1.0f)));
          st_io2(gdz + o2, mul2(f, fma2(dsk, uv, ys)));
        }
      }
      accB = __fadd2_rn(accB, ddr);
    };
    // one block of history in registers: the next block's load is issued once
    // the walk has used the current one.  Block k + 1 is finalized after the
    // walk over block k (its n-sums are complete since the barrier that ended
    // that walk's predecessor); the barrier after the finalize also frees
    // block k + 1's n-sum buffer for block k - 1.
    uint32_t hb[32];
    __syncwarp();
    tmem_ld32(thist + 32 * (kL / kRB - 1), hb);
    tmem_wait_ld32(hb);
    block(std::integral_constant<int, 1>{}, kL / (2 * kRB) - 1, hb);
    __syncwarp();
    tmem_ld32(thist + 32 * (kL / kRB - 2), hb);
    named_barrier(1 + grp, 64);
#pragma unroll 1
    for (int bp = kL / (2 * kRB) - 1; bp >= 0; --bp) {
      tmem_wait_ld32(hb);
      block(std::integral_constant<int, 0>{}, bp, hb);
      __syncwarp();
      if (bp > 0) tmem_ld32(thist + 32 * (2 * bp - 1), hb);
      finalize(2 * bp + 1);
      named_barrier(1 + grp, 64);
      if (bp == 0) break;
      tmem_wait_ld32(hb);
      block(std::integral_constant<int, 1>{}, bp - 1, hb);
      __syncwarp();
      tmem_ld32(thist + 32 * (2 * bp - 2), hb);
      finalize(2 * bp);
      named_barrier(1 + grp, 64);
    }
    finalize(0);
    if (pendB_t < rows) pdB[pendB_t] = pendB;
  }

  // ---- 5. dA partials ([chunk][n][d]); fixed-order CTA sums of dDskip, d_dt_bias
  if (valid) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int n = q ? nS : nF;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float2 sc = a.a_log ? mul2(A[q][j], splat2(kLn2)) : make_float2(1.0f, 1.0f);
        *reinterpret_cast<float2*>(a.part_dA + ((int64_t)chunk * N + n) * a.D + d + 2 * j) = mul2(dA[q][j], sc);
      }
    }
  }
  sm.redD[tid] = accD;
  sm.redB[tid] = accB;
  if (tid == 0) sm.ticket = next;
  __syncthreads();
  if (lane == 0 && sm.ticket < n_items) issue(sm.ticket, w);
  if (tid < kCQ && 4 * tid < bx && d0 + 4 * tid < a.D) {
    // dDskip: phase-1 quad q = tid % 16 of every thread, in thread order
    float4 sD = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int v = tid; v < kThr; v += kCQ) sD = add4(sD, sm.redD[v]);
    *reinterpret_cast<float4*>(a.part_dD + (int64_t)chunk * a.D + d0 + 4 * tid) = sD;
  }
  if (tid < 2 * kCQ && 2 * tid < bx && d0 + 2 * tid < a.D) {
    // d_dt_bias: channel pair cp = 16 g + cpl was finalized by the threads
    // 64 g + 16 e + cpl, e = 0..3
    const int g = tid >> 4, cpl = tid & 15;
    float2 sB = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int e = 0; e < kRB; ++e) sB = __fadd2_rn(sB, sm.redB[64 * g + 16 * e + cpl]);
    *reinterpret_cast<float2*>(a.part_dbias + (int64_t)chunk * a.D + d0 + 2 * tid) = sB;
  }
  __syncthreads();
  }  // persistent loop

  tmem_fence_before_sync();
  __syncthreads();
  if (w == 0) {
    tmem_fence_after_sync();
    tmem_dealloc256(sm.taddr);
  }
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

template <typename T, bool kStates, bool kRecY, bool kKnob = false>
cudaError_t launch_k16(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                       const CUtensorMap& tm_z, const CUtensorMap& tm_dout, const CUtensorMap& tm_cs,
                       const CUtensorMap& tm_y, cudaStream_t st) {
  auto kern = scan_bwd16_kernel<T, kStates, kRecY, kKnob>;
  const size_t smem = sizeof(Bwd16Smem<T, kRecY>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.n_chunks * a.n_tiles;
  int grid = 0;
  // every CTA holds 256 of the SM's 512 tensor-memory columns: at most 2 per SM
  e = persistent_grid(kern, 128, smem, items, &grid, 2);
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, smem, st>>>(tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, a);
  return cudaGetLastError();
}

template <typename T, int N, bool kStates, bool kRecY, bool kKnob = false>
cudaError_t launch_k(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, const CUtensorMap& tm_dout, const CUtensorMap& tm_cs,
                     const CUtensorMap& tm_y, cudaStream_t st) {
  auto kern = scan_bwd_kernel<T, N, kStates, kRecY, kKnob>;
  const size_t smem = sizeof(BwdSmem<T, N, kRecY>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.n_chunks * a.n_tiles;
  int grid = 0;
  // every CTA holds 128 of the SM's 512 tensor-memory columns: at most 4 per SM
  e = persistent_grid(kern, 8 * N, smem, items, &grid, 4);
  if (e != cudaSuccess) return e;
  kern<<<grid, 8 * N, smem, st>>>(tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, a);
  return cudaGetLastError();
}

template <typename T, int N, bool kRecY>
cudaError_t launch_y(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, const CUtensorMap& tm_dout, const CUtensorMap& tm_cs,
                     const CUtensorMap& tm_y, cudaStream_t st) {
  if constexpr (N == 16) {
    if constexpr (sizeof(T) == 4 && kRecY) {  // the delay knob's instantiation
      if (a.delay_ticket >= 0 && !a.seq)
        return launch_k16<T, false, kRecY, true>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
    }
    return a.seq ? launch_k16<T, true, kRecY>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st)
                 : launch_k16<T, false, kRecY>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
  } else {
    return a.seq ? launch_k<T, N, true, kRecY>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st)
                 : launch_k<T, N, false, kRecY>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
  }
}

template <typename T, int N>
cudaError_t launch_n(const ScanArgs& a, const CUtensorMap& tm_u, const CUtensorMap& tm_dr,
                     const CUtensorMap& tm_z, const CUtensorMap& tm_dout, const CUtensorMap& tm_cs,
                     const CUtensorMap& tm_y, cudaStream_t st) {
  return (a.has_z && !a.has_y) ? launch_y<T, N, true>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st)
                               : launch_y<T, N, false>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
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
  // B and C doubled once per call; every work item copies its chunk's rows
  cudaError_t e = launch_double_bc(a.B, a.C, io, a.T, (int64_t)a.n_chunks * kBwdChunk, a.N, a.N == 16, a.pos,
                                   const_cast<float4*>(a.BD), const_cast<float4*>(a.CD), st);
  if (e == cudaSuccess && a.N == 16)
    e = launch_bwd_tile_params(a.A, a.dt_bias, a.Dskip, a.D, a.a_log != 0, const_cast<float*>(a.tpar), st);
  if (e != cudaSuccess) return e;
  kernel_timer_mark(kTimeScanBwd, true, st);
  e = io == IO::F32 ? launch_t<float>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st)
                    : launch_t<__nv_bfloat16>(a, tm_u, tm_dr, tm_z, tm_dout, tm_cs, tm_y, st);
  kernel_timer_mark(kTimeScanBwd, false, st);
  if (e != cudaSuccess) return e;
  const int64_t M = a.T * 2 * a.N;
  // partial rows come in groups of 32 channels: two per tile when N = 16
  const int parts = a.n_tiles * (a.N == 16 ? 2 : 1);
  sum_tiles_bc_kernel<<<(unsigned)((M + 255) / 256), 256, 0, st>>>(a.part_dBC, parts, a.T, a.N, dB, dC);
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
