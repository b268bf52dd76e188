// kernels.h -- internal launcher interface between the C ABI (api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

// 1 in the checked build (-DVSSM_CHECKS=1): kernels check the sequence-state
// rows they index and the calls check caller-supplied position indices.
#ifndef VSSM_CHECKS
#define VSSM_CHECKS 0
#endif

namespace vssm {

enum class IO { F32 = 0, BF16 = 1 };

inline int io_bytes(IO t) { return t == IO::F32 ? 4 : 2; }

constexpr int kStateChunk = 32;  // tokens per saved scan-state chunk

// status-word bits written by kernels (the host maps them to VSSM_ERR_* codes)
enum : int { kStatusBadCu = 1, kStatusLookbackTimeout = 2, kStatusTmaTimeout = 4, kStatusNonFinite = 8,
             kStatusDeviceCheck = 16 };

// ---------------------------------------------------------------- position indices
// seq[t] = the sequence holding token t (read where sequences start or end).
cudaError_t launch_sequence_index(const int32_t* cu, int32_t num_seqs, int64_t T, int32_t* seq,
                                  cudaStream_t st);
// dst[s] = src[s] (or zeros) for every empty sequence s; rows of DN floats.
cudaError_t launch_empty_sequence_states(const int32_t* cu, int32_t num_seqs, int64_t DN,
                                         const float* src, float* dst, cudaStream_t st);
cudaError_t launch_position_indices(const int32_t* cu, int32_t num_seqs, int64_t T, int32_t* pos,
                                    int32_t* status, cudaStream_t st);
// The backward's doubled B and C (see ScanArgs::BD) for tokens 0 .. T_pad-1;
// packed (N = 16): per 32-token chunk, B and C in one array (see ScanArgs::BD)
// followed by the chunk's 32 position indices (zero past T), kBwdChunkRow
// bytes a chunk; CD unused.
cudaError_t launch_double_bc(const void* B, const void* C, IO io, int64_t T, int64_t T_pad, int N, bool packed,
                             const int32_t* pos, float4* BD, float4* CD, cudaStream_t st);
// The N = 16 backward's tile parameters (see ScanArgs::tpar).
cudaError_t launch_bwd_tile_params(const float* A, const float* dt_bias, const float* Dskip, int D, bool a_log,
                                   float* tpar, cudaStream_t st);
// dst[i] = the bf16 value src[i] as fp32, i < n.
cudaError_t launch_widen_bf16(const void* src, float* dst, int64_t n, cudaStream_t st);
// The forward's A rows (see ScanArgs::Af) for the ceil(D / 32) channel tiles.
cudaError_t launch_prep_a(const float* A, int D, int N, bool a_log, float4* Af, cudaStream_t st);
// ORs kStatusNonFinite into *status when any of the n values at p (io type,
// or f32 when f32 is true) is a NaN or an infinity.
cudaError_t launch_nonfinite_check(const void* p, int64_t n, bool f32, int32_t* status, cudaStream_t st);
// ORs kStatusBadCu into *status when a caller's position indices disagree
// with cu_seqlens (pos[t] != t - cu[s] for the sequence s holding t).
cudaError_t launch_position_check(const int32_t* cu, int32_t num_seqs, int64_t T, const int32_t* pos,
                                  int32_t* status, cudaStream_t st);

// ---------------------------------------------------------------- conv1d
struct ConvArgs {
  const void* x;
  const float* w;      // (D, W)
  const float* bias;   // (D) or null
  const int32_t* pos;  // (T)
  const void* du;      // bwd only
  void* out;           // fwd: u; bwd: dx
  float* partial;      // bwd: [rows_of_ctas][D*W + D]
  // conv tails of cut sequences, (num_seqs, D, W-1) f32, all nullable: the
  // W-1 inputs before each sequence (x_init), its last W-1 inputs (x_last,
  // fwd), and their gradients (dx_last in, dx_init out, bwd); seq[t] is the
  // sequence of token t (set whenever one of them is given)
  const int32_t* seq;
  const float* x_init;
  float* x_last;
  const float* dx_last;
  float* dx_init;
  int64_t T;
  int D;
  int W;
  int apply_silu;
  int num_seqs;
  const int32_t* cu;
  int* status;                      // device status word (workspace header)
  unsigned long long wait_ns;       // limit of the tile-copy wait
  long long force_timeout_cta;      // test knob: this CTA reports its copy wait as timed out
};
// Number of token-rows of CTAs the backward kernel uses (partial buffer rows).
int64_t conv_bwd_partial_rows(int64_t T);
// Tensor-map boxes of the conv tiles: rows of x (fwd or bwd) or of du, and channels.
int conv_tile_rows(int W, bool bwd, bool x);
int conv_tile_cols();
cudaError_t launch_conv1d_fwd(const ConvArgs& a, IO io, const CUtensorMap& tm_x, cudaStream_t st);
cudaError_t launch_conv1d_bwd(const ConvArgs& a, IO io, const CUtensorMap& tm_x, const CUtensorMap& tm_du,
                              float* dweight, float* dbias, cudaStream_t st);
// x_last (fwd) or dx_init (bwd) of every sequence, one block per sequence.
cudaError_t launch_conv_tails(const ConvArgs& a, IO io, bool bwd, cudaStream_t st);

// ---------------------------------------------------------------- selective scan
constexpr int kFwdChunk = 128;   // tokens per forward work item (look-back granule)
constexpr int kBwdChunk = 32;    // tokens per backward work item (= saved-state chunk)
// N = 16 backward: bytes of a chunk's packed B / C rows and position indices,
// and floats of a 64-channel tile's parameters (A rows, dt_bias, Dskip)
constexpr int kBwdChunkRow = kBwdChunk * 16 * 16 + kBwdChunk * 4;
constexpr int kBwdTileParams = 64 * 16 + 64 + 64;
constexpr int kTile = 32;        // channels per work item

struct ScanArgs {
  const void* u;
  const void* dr;
  const float* A;
  const void* B;
  const void* C;
  // fwd with bf16 I/O: B and C widened to fp32 once per call, (T, N) each
  // (null for fp32 I/O, where the kernel reads B and C themselves)
  const float* Bf32;
  const float* Cf32;
  // fwd: A * log2 e (A = -exp(A_log) when a_log), per 32-channel tile
  // [tile][n / 4][channel of the tile] float4 (zero past D), built once per
  // call, so that lane c of a warp reads channel c's four states n .. n + 3
  const float4* Af;
  // bwd: B and C doubled, [token][state pair][order] float4 (order 0 holds
  // (B[2p], B[2p], B[2p+1], B[2p+1]), order 1 the two states swapped), built
  // once per call for whole 32-token chunks (zero past the last token).  For
  // N = 16, B and C packed in BD alone: (B[2p], B[2p+1], C[2p], C[2p+1]) for
  // order 0, order 1 the two states swapped.
  const float4* BD;
  const float4* CD;
  // N = 16 bwd: per 64-channel tile, A * log2 e (A = -exp(A_log) when
  // a_log) as [channel][n], then dt_bias and Dskip (zero when absent or past
  // D): kBwdTileParams floats per tile, built once per call
  const float* tpar;
  const float* Dskip;
  const void* z;
  const float* dt_bias;
  const void* dout;           // bwd
  const int32_t* pos;
  float* chunk_states;        // fwd: written (nullable); bwd: read
  void* out;                  // fwd
  void* y;                    // fwd: pre-gate output (nullable); bwd: the same, read (nullable)
  // sequence states, (num_seqs, D, N) f32, all nullable: fwd reads h_init and
  // writes h_final; bwd reads h_init and dh_final and writes dh_init.  seq[t]
  // is the sequence of token t (set whenever one of them is given).
  const int32_t* seq;
  int num_seqs;
  const float* h_init;
  float* h_final;
  const float* dh_final;
  float* dh_init;
  void* du;                   // bwd
  void* ddr;                  // bwd
  void* dz;                   // bwd (nullable)
  float* part_dBC;            // bwd [32-channel group][2N][T]
  float* part_dA;             // bwd [n_chunks][N][D]
  float* part_dD;             // bwd [n_chunks][D]
  float* part_dbias;          // bwd [n_chunks][D]
  int* status;
  unsigned* ticket;
  // look-back state.  fwd: one chain per channel, flags [n_tiles][n_chunks][kTile],
  // agg / incl [n_tiles][n_chunks][N][kTile], agg_sd [n_tiles][n_chunks][kTile]
  // (sum of delta).  bwd: one chain per thread (its 4 or 8 (channel, state)
  // words), flags [n_tiles][n_chunks][warp], agg / incl / agg_sd
  // [n_tiles][n_chunks][thread][words], agg_sd holding the products of the
  // transition factors; the flags announce aggregates only, and incl starts
  // filled with kCarryUnset words.
  int* flags;
  float* agg;
  float* agg_sd;
  float* incl;
  int64_t T;
  int D;
  int N;
  int n_tiles;
  int n_chunks;
  int delta_softplus;
  float gate_floor;           // GateFloor: the gate is SiLU(z) + gate_floor
  int a_log;                  // A holds A_log (A = -exp(A_log)); bwd returns dA_log = dA * A
  int has_z;
  int has_y;                  // bwd: dz from the given y instead of recomputed C.h + Dskip u
  int has_skip;
  int box_x;                  // tile row pitch in elements: min(tile width, D)
  int box_y;                  // tile rows: min(chunk, T)
  long long drop_ticket;
  unsigned long long wait_ns;
  long long delay_ticket;       // test knob: this item sleeps delay_ns before storing its inclusive state
  unsigned long long delay_ns;
  // fused conv1d + scan forward (conv_w non-null): u = conv(x) computed in the
  // kernel from the x the u map then covers; u_out (nullable) receives it
  const float* conv_w;        // (D, conv_W)
  const float* conv_b;        // (D) or null
  int conv_W;
  int conv_silu;
  void* u_out;
};

cudaError_t launch_scan_fwd(const ScanArgs& a, IO io, const CUtensorMap& tm_u,
                            const CUtensorMap& tm_dr, const CUtensorMap& tm_z, cudaStream_t st);
cudaError_t launch_scan_bwd(const ScanArgs& a, IO io, const CUtensorMap& tm_u,
                            const CUtensorMap& tm_dr, const CUtensorMap& tm_z,
                            const CUtensorMap& tm_dout, const CUtensorMap& tm_cs,
                            const CUtensorMap& tm_y, float* dA,
                            float* dB, float* dC, float* dDskip, float* d_dt_bias, cudaStream_t st);

// Kernel timing (VSSM_DBG_KERNEL_EVENTS): when it is on, the calls record a
// CUDA event pair on their stream around their main kernel, kind 0 conv1d
// fwd, 1 scan fwd, 2 scan bwd, 3 conv1d bwd.  No-ops when off.
enum : int { kTimeConvFwd = 0, kTimeScanFwd = 1, kTimeScanBwd = 2, kTimeConvBwd = 3, kTimeKinds = 4 };
void kernel_timer_mark(int kind, bool begin, cudaStream_t st);

// Sets the message vssm_last_error() returns on this thread; returns `code`.
int record_error(int code, const char* message);

// ---------------------------------------------------------------- shared host helpers (api.cu)
// Byte offsets of a scan call's workspace: [header 256 B: status int @0,
// ticket uint @4][look-back flags][position indices][sequence index]
// [fwd: B and C as fp32, A rows][aggregates][aggregate factors][inclusive states]
// [backward partials].
// The header and flags (clear_bytes) start at zero; the inclusive states
// (incl, incl_bytes) start as all-ones words.
struct ScanLayout {
  size_t flags = 0, pos = 0, seq = 0, bcf = 0, af = 0, agg = 0, agg_sd = 0, incl = 0;
  size_t part_bc = 0, part_a = 0, part_d = 0, part_b = 0, bcd = 0, tpar = 0;
  size_t clear_bytes = 0, incl_bytes = 0, total = 0;
};
// chunk = tokens per work item (kFwdChunk / kBwdChunk).
ScanLayout scan_workspace_layout(int64_t T, int D, int N, int chunk, bool bwd);
// Channels per work item of a scan call (64 for the backward with N = 16, else 32).
int scan_tile_width(int N, bool bwd);
// 2-D tensor map over a (T, D) row-major tensor, box = box_x channels x
// box_y tokens; returns VSSM_OK or a VSSM_ERR_* code (message recorded).
int encode_tile_map(CUtensorMap* m, const void* base, IO io, int64_t T, int D, int box_x, int box_y);
// The test knobs set by vssm_debug_set, as the kernels take them.
struct DebugKnobs {
  long long drop_ticket;
  unsigned long long wait_ns;
  long long delay_ticket;
  unsigned long long delay_ns;
  bool check_finite;
};
DebugKnobs debug_knobs();
// With the VSSM_DBG_CHECK_FINITE knob on, checks the n outputs (pointer,
// value count, f32 or io bf16) for NaNs and infinities into *status.
int check_outputs_finite(int32_t* status, cudaStream_t st, const void* const* ptrs, const int64_t* counts,
                         const bool* f32, int n);

// ---------------------------------------------------------------- reductions
// out[m] = sum_{p < P} in[p * ld + m] for m < M, in a fixed order (rows in
// order within groups of 32, then the group sums in order); `in` is scratch
// and is overwritten.  With inner > 0 the M columns form an (M / inner, inner)
// array that is written out transposed.
cudaError_t launch_sum_rows(float* in, int64_t P, int64_t M, int64_t ld, float* out, cudaStream_t st,
                            int64_t inner = 0);

}  // namespace vssm
