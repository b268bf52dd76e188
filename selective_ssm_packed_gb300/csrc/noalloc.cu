// noalloc.cu -- the forward selective scan for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run the scan: code that runs inside a host allocator's own callbacks, a
// runtime that has handed every byte of the device to its own pool up front,
// or an embedding that forbids allocation on its hot path so that a step never
// stalls on the allocator.  varlen_selective_scan_fwd needs a caller-supplied
// workspace for its cross-chunk look-back state; this variant keeps that
// scratch in a fixed-size array compiled into the library instead, so the
// caller passes only inputs and outputs.
//
// The scratch is one file-scope __device__ array of VSSM_NOALLOC_SCRATCH_BYTES
// (64 MiB).  Every GPU that loads this part of the library keeps it until the
// process exits, and every call on a device uses the same array, which keeps
// whatever the previous call left: before launching, the call clears the part
// that must start at zero (status, work ticket, look-back flags) and fills the
// look-back states with the all-ones word that reads as "not stored yet".
// Calls that overlap on the GPU (two streams, or two host threads on one
// device) race on it.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "varlen_ssm.h"

namespace vssm {
namespace {

constexpr size_t kScratchBytes = VSSM_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

}  // namespace

// The scratch itself.  In host code this name is only a host-side stand-in for
// the device array; kernels must be given the device address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

int err(int code, const char* fmt, long long a = 0, long long b = 0) {
  char buf[256];
  snprintf(buf, sizeof(buf), fmt, a, b);
  return record_error(code, buf);
}

// Device address of the scratch on the current device, looked up on the first
// call made with that device current and cached per device afterwards.  The
// cache outlives nothing but the device's context: after cudaDeviceReset (or
// anything else that destroys the primary context) the cached address is
// stale, and the process must not call the entry point on that device again.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_error(VSSM_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return err(VSSM_ERR_CUDA, "device ordinal %lld out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      char buf[256];
      snprintf(buf, sizeof(buf), "cudaGetSymbolAddress of the built-in scratch failed: %s",
               cudaGetErrorString(e));
      return record_error(VSSM_ERR_CUDA, buf);
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return VSSM_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace
}  // namespace vssm

using namespace vssm;

extern "C" int varlen_selective_scan_fwd_noalloc(
    const void* u, const void* delta_raw, const float* A, const void* B, const void* C,
    const float* Dskip, const void* z, const float* dt_bias, int32_t delta_softplus, float gate_floor,
    int32_t a_log,
    const int32_t* cu_seqlens, const int32_t* position_indices, int32_t num_seqs,
    int64_t total_tokens, int32_t D, int32_t N, vssm_dtype dtype, void* out, void* y, float* chunk_states,
    const float* initial_states, float* final_states, int32_t* status, void* stream) {
  // ---- argument checks (same rules as varlen_selective_scan_fwd)
  if (dtype != VSSM_F32 && dtype != VSSM_BF16) return err(VSSM_ERR_DTYPE, "dtype %lld not supported", dtype);
  const IO io = dtype == VSSM_F32 ? IO::F32 : IO::BF16;
  const int64_t T = total_tokens;
  if (T < 0 || T > 2147483647LL) return err(VSSM_ERR_ARG, "total_tokens %lld out of range", T);
  if (D <= 0) return err(VSSM_ERR_ARG, "D must be positive (got %lld)", D);
  if (num_seqs < 0 || !cu_seqlens) return record_error(VSSM_ERR_ARG, "bad num_seqs or NULL cu_seqlens");
  if ((initial_states || final_states) && T > 0 && num_seqs < 1)
    return record_error(VSSM_ERR_ARG, "sequence states given for tokens but num_seqs = 0");
  if (N != 4 && N != 8 && N != 16) return err(VSSM_ERR_UNSUPPORTED, "N = %lld not in {4, 8, 16}", N);
  const int e = io_bytes(io);
  if (((int64_t)D * e) % 16 != 0 || (N * e) % 16 != 0)
    return record_error(VSSM_ERR_ALIGN, "D * sizeof(io) and N * sizeof(io) must be multiples of 16");
  if (!A) return record_error(VSSM_ERR_ARG, "A is NULL");
  if (T > 0) {
    const void* need[] = {u, delta_raw, B, C, out};
    for (const void* p : need) {
      if (!p) return record_error(VSSM_ERR_ARG, "u, delta_raw, B, C and out must be non-NULL");
      if (!al16(p)) return record_error(VSSM_ERR_ALIGN, "u, delta_raw, B, C, out must be 16-byte aligned");
    }
  }
  if ((z && !al16(z)) || (y && !al16(y)) || (chunk_states && !al16(chunk_states)) || !al16(A) ||
      (Dskip && !al16(Dskip)) || (dt_bias && !al16(dt_bias)) || (position_indices && !al16(position_indices)) ||
      (initial_states && !al16(initial_states)) || (final_states && !al16(final_states)))
    return record_error(VSSM_ERR_ALIGN,
                        "z, y, chunk_states, A, Dskip, dt_bias, position_indices, initial_states and "
                        "final_states must be 16-byte aligned");

  // ---- the forward call's own workspace layout, placed in the built-in scratch
  const ScanLayout l = scan_workspace_layout(T, D, N, kFwdChunk, false);
  if (l.total > kScratchBytes)
    return err(VSSM_ERR_WORKSPACE,
               "this problem needs %lld bytes of scratch but the built-in scratch holds %lld bytes; "
               "use varlen_selective_scan_fwd with a caller-allocated workspace",
               (long long)l.total, (long long)kScratchBytes);

  void* base = nullptr;
  const int rc = scratch_address(&base);
  if (rc != VSSM_OK) return rc;
  char* s = static_cast<char*>(base);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t ce = cudaMemsetAsync(s, 0, l.clear_bytes, st);  // status, ticket, look-back flags
  // look-back states: all-ones NaN words, read by the kernel as "not stored yet"
  if (ce == cudaSuccess && T > 0) ce = cudaMemsetAsync(s + l.incl, 0xff, l.incl_bytes, st);
  if (ce == cudaSuccess && status) ce = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
  // an empty sequence ends in the state it starts from
  if (ce == cudaSuccess)
    ce = launch_empty_sequence_states(cu_seqlens, num_seqs, (int64_t)D * N, initial_states, final_states, st);
  if (ce != cudaSuccess) return record_error(VSSM_ERR_CUDA, cudaGetErrorString(ce));
  if (T == 0) return VSSM_OK;
  int32_t* status_word = status ? status : reinterpret_cast<int32_t*>(s);
  const int32_t* seq = nullptr;
  if (initial_states || final_states) {
    ce = launch_sequence_index(cu_seqlens, num_seqs, T, reinterpret_cast<int32_t*>(s + l.seq), st);
    if (ce != cudaSuccess) return record_error(VSSM_ERR_CUDA, cudaGetErrorString(ce));
    seq = reinterpret_cast<int32_t*>(s + l.seq);
  }

  const int32_t* pos = position_indices;
  if (VSSM_CHECKS && pos) {  // the checked build verifies the caller's indices
    ce = launch_position_check(cu_seqlens, num_seqs, T, pos, status_word, st);
    if (ce != cudaSuccess) return record_error(VSSM_ERR_CUDA, cudaGetErrorString(ce));
  }
  if (!pos) {
    int32_t* p = reinterpret_cast<int32_t*>(s + l.pos);
    ce = launch_position_indices(cu_seqlens, num_seqs, T, p, status_word, st);
    if (ce != cudaSuccess) return record_error(VSSM_ERR_CUDA, cudaGetErrorString(ce));
    pos = p;
  }

  const int tw = scan_tile_width(N, false);
  const DebugKnobs kn = debug_knobs();
  ScanArgs a{};
  a.u = u; a.dr = delta_raw; a.A = A; a.B = B; a.C = C; a.Dskip = Dskip; a.z = z;
  a.dt_bias = dt_bias; a.pos = pos; a.chunk_states = chunk_states; a.out = out; a.y = y;
  a.seq = seq; a.h_init = initial_states; a.h_final = final_states;
  if (io == IO::BF16) {
    a.Bf32 = reinterpret_cast<float*>(s + l.bcf);
    a.Cf32 = a.Bf32 + T * N;
  }
  a.Af = reinterpret_cast<float4*>(s + l.af);
  a.status = status_word;
  a.ticket = reinterpret_cast<unsigned*>(s + 4);
  a.flags = reinterpret_cast<int*>(s + l.flags);
  a.agg = reinterpret_cast<float*>(s + l.agg);
  a.agg_sd = reinterpret_cast<float*>(s + l.agg_sd);
  a.incl = reinterpret_cast<float*>(s + l.incl);
  a.T = T; a.D = D; a.N = N; a.num_seqs = num_seqs;
  a.n_tiles = (int)cdiv(D, tw);
  a.n_chunks = (int)cdiv(T, kFwdChunk);
  a.delta_softplus = delta_softplus ? 1 : 0;
  a.gate_floor = gate_floor;
  a.a_log = a_log ? 1 : 0;
  a.has_z = z ? 1 : 0;
  a.has_skip = Dskip ? 1 : 0;
  a.box_x = D < tw ? D : tw;
  a.box_y = T < kFwdChunk ? (int)T : kFwdChunk;
  // the test knobs of vssm_debug_set apply here as in the workspace entry point
  a.drop_ticket = kn.drop_ticket;
  a.wait_ns = kn.wait_ns;
  a.delay_ticket = kn.delay_ticket;
  a.delay_ns = kn.delay_ns;
  CUtensorMap mu, mdr, mz;
  int r = encode_tile_map(&mu, u, io, T, D, a.box_x, a.box_y);
  if (r == VSSM_OK) r = encode_tile_map(&mdr, delta_raw, io, T, D, a.box_x, a.box_y);
  if (r == VSSM_OK) r = encode_tile_map(&mz, z, io, T, D, a.box_x, a.box_y);
  if (r != VSSM_OK) return r;
  ce = launch_scan_fwd(a, io, mu, mdr, mz, st);
  if (ce != cudaSuccess) return record_error(VSSM_ERR_CUDA, cudaGetErrorString(ce));
  // with the VSSM_DBG_CHECK_FINITE knob on: NaNs or infinities in the outputs
  const void* outs[] = {out, y};
  const int64_t counts[] = {T * D, y ? T * D : 0};
  const bool f32[] = {io == IO::F32, io == IO::F32};
  return check_outputs_finite(status_word, st, outs, counts, f32, 2);
}
