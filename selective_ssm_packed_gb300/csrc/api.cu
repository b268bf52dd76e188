// api.cu -- the C ABI of libvarlen_ssm.so (declared in include/varlen_ssm.h):
// argument validation, workspace layout, TMA descriptors, kernel launches,
// device status words and error reporting.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <initializer_list>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "kernels.h"
#include "varlen_ssm.h"

using namespace vssm;

namespace {

thread_local std::string g_last_error;
std::atomic<long long> g_drop_ticket{-1};
std::atomic<unsigned long long> g_wait_ns{1000000000ull};
std::atomic<long long> g_delay_ticket{-1};
std::atomic<unsigned long long> g_delay_ns{200000ull};
std::atomic<long long> g_force_copy_timeout{-1};
std::atomic<int> g_check_finite{0};
std::atomic<int> g_kernel_events{0};

// The recorded event pairs of each kind of main kernel, and a pool of events
// to reuse (created on first use).
struct KernelTimer {
  std::mutex mu;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pairs[vssm::kTimeKinds];
  cudaEvent_t open[vssm::kTimeKinds] = {};
  std::vector<cudaEvent_t> pool;
  cudaEvent_t take() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    return cudaEventCreate(&e) == cudaSuccess ? e : nullptr;
  }
  void give(cudaEvent_t e) {
    if (e) pool.push_back(e);
  }
};
KernelTimer& kernel_timer() {
  static KernelTimer t;
  return t;
}

// An NVTX range over a C-ABI call (host side: the call's enqueue), named
// after the call, for timelines taken with a profiler.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(VSSM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- workspace layout
// [header 256 B: status int @0, ticket uint @4][flags, one per (slot, lane)][pos][...call specific]
// header + flags are cleared by one memset at the start of every call.
struct Layout {
  size_t flags = 0, pos = 0, seq = 0, bcf = 0, af = 0, agg = 0, agg_sd = 0, incl = 0;
  size_t part_bc = 0, part_a = 0, part_d = 0, part_b = 0, bcd = 0, tpar = 0, conv_part = 0;
  size_t clear_bytes = 0, incl_bytes = 0, total = 0;
};

// Channels per work item of a scan call: the backward with N = 16 takes 64
// (two 32-channel groups per CTA), every other call 32.
int scan_tile(int N, bool bwd) { return (bwd && N == 16) ? 2 * kTile : kTile; }

Layout scan_layout(int64_t T, int D, int N, int chunk, bool bwd) {
  Layout l;
  const int tw = scan_tile(N, bwd);
  const int64_t n_tiles = cdiv(D, tw);
  const int64_t n_chunks = cdiv(T, chunk);
  const int64_t slots = n_tiles * n_chunks;
  size_t off = kAlign;
  l.flags = off;
  off += up(sizeof(int) * (size_t)slots * tw);
  l.clear_bytes = off;
  l.pos = off;
  off += up(sizeof(int32_t) * (size_t)T);
  l.seq = off;
  off += up(sizeof(int32_t) * (size_t)T);
  if (!bwd) {  // B and C as fp32 for bf16 I/O, widened once per call; the A rows
    l.bcf = off;
    off += up(sizeof(float) * (size_t)T * N * 2);
    l.af = off;
    off += up(sizeof(float) * (size_t)n_tiles * tw * N);
  }
  l.agg = off;
  off += up(sizeof(float) * (size_t)slots * N * tw);
  l.agg_sd = off;
  off += up(sizeof(float) * (size_t)slots * (bwd ? N : 1) * tw);
  l.incl = off;
  l.incl_bytes = sizeof(float) * (size_t)slots * N * tw;
  off += up(l.incl_bytes);
  if (bwd) {
    // dB / dC partials: one row group per 32 channels
    l.part_bc = off;
    off += up(sizeof(float) * (size_t)n_tiles * (tw / kTile) * T * 2 * N);
    l.part_a = off;
    off += up(sizeof(float) * (size_t)n_chunks * D * N);
    l.part_d = off;
    off += up(sizeof(float) * (size_t)n_chunks * D);
    l.part_b = off;
    off += up(sizeof(float) * (size_t)n_chunks * D);
    // B and C doubled for whole chunks: [token][state pair][order] float4
    // (N = 16: packed, with the chunk's position indices, in less room)
    l.bcd = off;
    off += up(sizeof(float) * 4 * (size_t)n_chunks * chunk * N * 2);
    if (N == 16) {  // the tiles' A rows, dt_bias and Dskip
      l.tpar = off;
      off += up(sizeof(float) * (size_t)n_tiles * kBwdTileParams);
    }
  }
  l.total = off;
  return l;
}

Layout conv_layout(int64_t T, int D, int W, bool bwd) {
  Layout l;
  size_t off = kAlign;
  l.clear_bytes = off;
  l.pos = off;
  off += up(sizeof(int32_t) * (size_t)T);
  l.seq = off;
  off += up(sizeof(int32_t) * (size_t)T);
  if (bwd) {
    l.conv_part = off;
    off += up(sizeof(float) * (size_t)conv_bwd_partial_rows(T) * D * (W + 1));
  }
  l.total = off;
  return l;
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

// ---------------------------------------------------------------- TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D map over a (T, D) row-major tensor, box = box_x channels x box_y tokens.
int make_map(CUtensorMap* m, const void* base, IO io, int64_t T, int D, int box_x, int box_y) {
  std::memset(m, 0, sizeof(*m));
  if (!base) return VSSM_OK;
  auto enc = encoder();
  if (!enc) return fail(VSSM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)T};
  const cuuint64_t strides[1] = {(cuuint64_t)D * (cuuint64_t)io_bytes(io)};
  const cuuint32_t box[2] = {(cuuint32_t)box_x, (cuuint32_t)box_y};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, io == IO::F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(VSSM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return VSSM_OK;
}

// ---------------------------------------------------------------- validation
int check_dtype(vssm_dtype dt, IO* io) {
  if (dt == VSSM_F32) { *io = IO::F32; return VSSM_OK; }
  if (dt == VSSM_BF16) { *io = IO::BF16; return VSSM_OK; }
  return fail(VSSM_ERR_DTYPE, "dtype %d is neither VSSM_F32 nor VSSM_BF16", (int)dt);
}

int check_shape(int64_t T, int D, int32_t num_seqs, const int32_t* cu) {
  if (T < 0 || T > 2147483647LL) return fail(VSSM_ERR_ARG, "total_tokens %lld out of range", (long long)T);
  if (D <= 0) return fail(VSSM_ERR_ARG, "D must be positive (got %d)", D);
  if (num_seqs < 0) return fail(VSSM_ERR_ARG, "num_seqs must be >= 0 (got %d)", num_seqs);
  if (!cu) return fail(VSSM_ERR_ARG, "cu_seqlens is NULL");
  return VSSM_OK;
}

int check_io(const void* p, const char* name, int64_t T) {
  if (T == 0) return VSSM_OK;
  if (!p) return fail(VSSM_ERR_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(VSSM_ERR_ALIGN, "%s is not 16-byte aligned", name);
  return VSSM_OK;
}

int check_ws(const void* ws, size_t have, size_t need) {
  if (have < need) return fail(VSSM_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", have, need);
  if (!ws) return fail(VSSM_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned16(ws)) return fail(VSSM_ERR_ALIGN, "workspace is not 16-byte aligned");
  return VSSM_OK;
}

// Resolves the position indices a call uses: the caller's array, or one built
// in the workspace from cu_seqlens (status bits land in the workspace header).
int check_caller_pos(const int32_t* cu, int32_t S, int64_t T, const int32_t* pos, int32_t* status,
                     cudaStream_t st);
int resolve_pos(const int32_t* cu, const int32_t* pos_in, int32_t S, int64_t T, void* ws,
                const Layout& l, cudaStream_t st, const int32_t** pos_out) {
  if (pos_in) {
    *pos_out = pos_in;
    return check_caller_pos(cu, S, T, pos_in, at<int32_t>(ws, 0), st);
  }
  int32_t* p = at<int32_t>(ws, l.pos);
  cudaError_t e = launch_position_indices(cu, S, T, p, at<int32_t>(ws, 0), st);
  if (e != cudaSuccess) return cuda_fail(e, "position_indices launch");
  *pos_out = p;
  return VSSM_OK;
}

// With the VSSM_DBG_CHECK_FINITE knob on, ORs kStatusNonFinite into the
// call's status word when any output holds a NaN or an infinity.
struct OutSpan {
  const void* p;
  int64_t n;
  bool f32;
};
int check_outputs(int32_t* status, cudaStream_t st, std::initializer_list<OutSpan> outs) {
  if (!g_check_finite.load()) return VSSM_OK;
  for (const OutSpan& o : outs) {
    const cudaError_t e = launch_nonfinite_check(o.p, o.n, o.f32, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "non-finite check launch");
  }
  return VSSM_OK;
}

// In the checks build, a caller's position indices are verified against
// cu_seqlens (kStatusBadCu in the status word when they disagree).
int check_caller_pos(const int32_t* cu, int32_t S, int64_t T, const int32_t* pos, int32_t* status,
                     cudaStream_t st) {
  if (!VSSM_CHECKS || !pos || T <= 0) return VSSM_OK;
  const cudaError_t e = launch_position_check(cu, S, T, pos, status, st);
  return e == cudaSuccess ? VSSM_OK : cuda_fail(e, "position check launch");
}

// A (num_seqs, D, N) f32 sequence-state array: nullable, 16-byte aligned.
int check_states(const float* p, const char* name) {
  if (p && !aligned16(p)) return fail(VSSM_ERR_ALIGN, "%s is not 16-byte aligned", name);
  return VSSM_OK;
}

// Sequence states (or conv tails) of a call with tokens need at least one
// sequence to hold them.
int check_states_rows(bool any_states, int32_t num_seqs, int64_t T) {
  if (any_states && T > 0 && num_seqs < 1)
    return fail(VSSM_ERR_ARG, "sequence states or tails given for %lld tokens but num_seqs = %d", (long long)T,
                num_seqs);
  return VSSM_OK;
}

#define VSSM_TRY(expr)              \
  do {                              \
    const int rc_ = (expr);         \
    if (rc_ != VSSM_OK) return rc_; \
  } while (0)

}  // namespace

void vssm::kernel_timer_mark(int kind, bool begin, cudaStream_t st) {
  if (!g_kernel_events.load() || kind < 0 || kind >= kTimeKinds) return;
  KernelTimer& kt = kernel_timer();
  std::lock_guard<std::mutex> lock(kt.mu);
  cudaEvent_t e = kt.take();
  if (!e) return;
  if (cudaEventRecord(e, st) != cudaSuccess) {
    kt.give(e);
    return;
  }
  if (begin) {
    kt.give(kt.open[kind]);  // an unmatched begin is dropped
    kt.open[kind] = e;
  } else if (kt.open[kind]) {
    kt.pairs[kind].emplace_back(kt.open[kind], e);
    kt.open[kind] = nullptr;
  } else {
    kt.give(e);
  }
}

// Lets other translation units of the library report a host-side error
// through vssm_last_error().
int vssm::record_error(int code, const char* message) {
  g_last_error = message ? message : "";
  return code;
}

int vssm::check_outputs_finite(int32_t* status, cudaStream_t st, const void* const* ptrs, const int64_t* counts,
                               const bool* f32, int n) {
  if (!g_check_finite.load()) return VSSM_OK;
  for (int i = 0; i < n; ++i) {
    const cudaError_t e = launch_nonfinite_check(ptrs[i], counts[i], f32[i], status, st);
    if (e != cudaSuccess) return cuda_fail(e, "non-finite check launch");
  }
  return VSSM_OK;
}

vssm::ScanLayout vssm::scan_workspace_layout(int64_t T, int D, int N, int chunk, bool bwd) {
  const Layout l = scan_layout(T, D, N, chunk, bwd);
  ScanLayout o;
  o.flags = l.flags; o.pos = l.pos; o.seq = l.seq; o.bcf = l.bcf; o.af = l.af; o.agg = l.agg; o.agg_sd = l.agg_sd;
  o.incl = l.incl;
  o.part_bc = l.part_bc; o.part_a = l.part_a; o.part_d = l.part_d; o.part_b = l.part_b; o.bcd = l.bcd; o.tpar = l.tpar;
  o.clear_bytes = l.clear_bytes; o.incl_bytes = l.incl_bytes; o.total = l.total;
  return o;
}

int vssm::scan_tile_width(int N, bool bwd) { return scan_tile(N, bwd); }

int vssm::encode_tile_map(CUtensorMap* m, const void* base, IO io, int64_t T, int D, int box_x, int box_y) {
  return make_map(m, base, io, T, D, box_x, box_y);
}

vssm::DebugKnobs vssm::debug_knobs() {
  return DebugKnobs{g_drop_ticket.load(), g_wait_ns.load(), g_delay_ticket.load(), g_delay_ns.load(),
                    g_check_finite.load() != 0};
}

// ============================================================================ C ABI
extern "C" {

int vssm_status_code(int32_t w) {
  if (w & kStatusBadCu) return VSSM_ERR_BAD_CU_SEQLENS;
  if (w & (kStatusLookbackTimeout | kStatusTmaTimeout)) return VSSM_ERR_LOOKBACK_TIMEOUT;
  if (w & kStatusDeviceCheck) return VSSM_ERR_DEVICE_CHECK;
  if (w & kStatusNonFinite) return VSSM_ERR_NONFINITE;
  return VSSM_OK;
}

const char* vssm_strerror(int code) {
  switch (code) {
    case VSSM_OK: return "success";
    case VSSM_ERR_ARG: return "invalid argument";
    case VSSM_ERR_DTYPE: return "unsupported dtype";
    case VSSM_ERR_ALIGN: return "pointer or row pitch not 16-byte aligned";
    case VSSM_ERR_WORKSPACE: return "workspace missing or too small";
    case VSSM_ERR_CUDA: return "CUDA runtime or driver error";
    case VSSM_ERR_UNSUPPORTED: return "unsupported N or conv width";
    case VSSM_ERR_BAD_CU_SEQLENS: return "malformed cu_seqlens, or position indices that disagree with it (device check)";
    case VSSM_ERR_LOOKBACK_TIMEOUT: return "a device-side wait timed out: look-back or tile copy (device check)";
    case VSSM_ERR_NONFINITE: return "an output holds a NaN or an infinity (VSSM_DBG_CHECK_FINITE)";
    case VSSM_ERR_DEVICE_CHECK: return "a device-side index check failed (VSSM_CHECKS build)";
  }
  return "unknown status code";
}

const char* vssm_last_error(void) { return g_last_error.c_str(); }

int vssm_checks_build(void) { return VSSM_CHECKS ? 1 : 0; }

int vssm_kernel_time(int kind, double* total_ms, int64_t* launches) {
  if (kind < 0 || kind >= kTimeKinds || !total_ms || !launches) return fail(VSSM_ERR_ARG, "bad kind or NULL output");
  KernelTimer& kt = kernel_timer();
  std::lock_guard<std::mutex> lock(kt.mu);
  double ms = 0.0;
  int64_t n = 0;
  cudaError_t err = cudaSuccess;
  for (auto& pr : kt.pairs[kind]) {
    float t = 0.0f;
    cudaError_t e = cudaEventSynchronize(pr.second);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, pr.first, pr.second);
    if (e == cudaSuccess) {
      ms += t;
      ++n;
    } else if (err == cudaSuccess) {
      err = e;
    }
    kt.give(pr.first);
    kt.give(pr.second);
  }
  kt.pairs[kind].clear();
  *total_ms = ms;
  *launches = n;
  return err == cudaSuccess ? VSSM_OK : cuda_fail(err, "kernel event timing");
}

int vssm_debug_set(int knob, int64_t value) {
  if (knob == VSSM_DBG_DROP_FLAG) { g_drop_ticket.store(value); return VSSM_OK; }
  if (knob == VSSM_DBG_WAIT_NS) {
    if (value <= 0) return fail(VSSM_ERR_ARG, "wait limit must be positive");
    g_wait_ns.store((unsigned long long)value);
    return VSSM_OK;
  }
  if (knob == VSSM_DBG_DELAY_ITEM) { g_delay_ticket.store(value); return VSSM_OK; }
  if (knob == VSSM_DBG_DELAY_NS) {
    if (value <= 0 || value > 10000000) return fail(VSSM_ERR_ARG, "delay must be in (0, 1e7] ns");
    g_delay_ns.store((unsigned long long)value);
    return VSSM_OK;
  }
  if (knob == VSSM_DBG_FORCE_COPY_TIMEOUT) { g_force_copy_timeout.store(value); return VSSM_OK; }
  if (knob == VSSM_DBG_KERNEL_EVENTS) {
    if (value != 0 && value != 1) return fail(VSSM_ERR_ARG, "VSSM_DBG_KERNEL_EVENTS takes 0 or 1");
    g_kernel_events.store((int)value);
    if (!value) {  // drop what was recorded (completed or not: events are reusable once recorded over)
      KernelTimer& kt = kernel_timer();
      std::lock_guard<std::mutex> lock(kt.mu);
      for (int k = 0; k < kTimeKinds; ++k) {
        for (auto& pr : kt.pairs[k]) {
          kt.give(pr.first);
          kt.give(pr.second);
        }
        kt.pairs[k].clear();
        kt.give(kt.open[k]);
        kt.open[k] = nullptr;
      }
    }
    return VSSM_OK;
  }
  if (knob == VSSM_DBG_CHECK_FINITE) {
    if (value != 0 && value != 1) return fail(VSSM_ERR_ARG, "VSSM_DBG_CHECK_FINITE takes 0 or 1");
    g_check_finite.store((int)value);
    return VSSM_OK;
  }
  return fail(VSSM_ERR_ARG, "unknown debug knob %d", knob);
}

int vssm_read_status(const void* workspace, void* stream, int* status) {
  if (!workspace || !status) return fail(VSSM_ERR_ARG, "workspace and status must be non-NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t w = 0;
  cudaError_t e = cudaMemcpyAsync(&w, workspace, sizeof(w), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  *status = vssm_status_code(w);
  return VSSM_OK;
}

// ---------------------------------------------------------------- position indices
int varlen_position_indices(const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                            int32_t* position_indices, int32_t* status, void* stream) {
  NvtxRange nvtx_("varlen_position_indices");
  VSSM_TRY(check_shape(total_tokens, 1, num_seqs, cu_seqlens));
  if (total_tokens > 0 && !position_indices) return fail(VSSM_ERR_ARG, "position_indices is NULL");
  cudaError_t e = launch_position_indices(cu_seqlens, num_seqs, total_tokens, position_indices,
                                          status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VSSM_OK : cuda_fail(e, "position_indices launch");
}

// ---------------------------------------------------------------- conv1d
size_t varlen_conv1d_fwd_workspace_size(int64_t total_tokens, int32_t D, int32_t W) {
  if (total_tokens < 0 || D <= 0 || W < 1 || W > 4) return 0;
  return conv_layout(total_tokens, D, W, false).total;
}

size_t varlen_conv1d_bwd_workspace_size(int64_t total_tokens, int32_t D, int32_t W) {
  if (total_tokens < 0 || D <= 0 || W < 1 || W > 4) return 0;
  return conv_layout(total_tokens, D, W, true).total;
}

static int conv_common(const void* x, const float* weight, const int32_t* cu, int32_t num_seqs,
                       int64_t T, int32_t D, int32_t W, vssm_dtype dtype, IO* io) {
  VSSM_TRY(check_dtype(dtype, io));
  VSSM_TRY(check_shape(T, D, num_seqs, cu));
  if (W < 1 || W > 4) return fail(VSSM_ERR_UNSUPPORTED, "conv width %d not in 1..4", W);
  if (((int64_t)D * io_bytes(*io)) % 16 != 0)
    return fail(VSSM_ERR_ALIGN, "D * sizeof(io) = %lld is not a multiple of 16",
                (long long)D * io_bytes(*io));
  if (!weight) return fail(VSSM_ERR_ARG, "weight is NULL");
  VSSM_TRY(check_io(x, "x", T));
  return VSSM_OK;
}

int varlen_conv1d_fwd(const void* x, const float* weight, const float* bias,
                      const int32_t* cu_seqlens, const int32_t* position_indices, int32_t num_seqs,
                      int64_t total_tokens, int32_t D, int32_t W, int32_t apply_silu,
                      vssm_dtype dtype, void* u, const float* x_init, float* x_last,
                      void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_("varlen_conv1d_fwd");
  IO io;
  VSSM_TRY(conv_common(x, weight, cu_seqlens, num_seqs, total_tokens, D, W, dtype, &io));
  VSSM_TRY(check_io(u, "u", total_tokens));
  VSSM_TRY(check_states(x_init, "x_init"));
  VSSM_TRY(check_states(x_last, "x_last"));
  VSSM_TRY(check_states_rows(x_init || x_last, num_seqs, total_tokens));
  const Layout l = conv_layout(total_tokens, D, W, false);
  VSSM_TRY(check_ws(workspace, workspace_bytes, l.total));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(workspace, 0, l.clear_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace header");
  ConvArgs a{};
  a.x = x; a.w = weight; a.bias = bias; a.out = u;
  a.T = total_tokens; a.D = D; a.W = W; a.apply_silu = apply_silu ? 1 : 0;
  a.cu = cu_seqlens; a.num_seqs = num_seqs; a.x_init = W > 1 ? x_init : nullptr; a.x_last = x_last;
  a.status = at<int>(workspace, 0);
  a.wait_ns = g_wait_ns.load();
  a.force_timeout_cta = g_force_copy_timeout.load();
  // every sequence's last W-1 inputs (its tail values when it is shorter)
  e = launch_conv_tails(a, io, false, st);
  if (e != cudaSuccess) return cuda_fail(e, "conv tails launch");
  if (total_tokens == 0) return VSSM_OK;
  const int32_t* pos = nullptr;
  VSSM_TRY(resolve_pos(cu_seqlens, position_indices, num_seqs, total_tokens, workspace, l, st, &pos));
  a.pos = pos;
  if (a.x_init) {
    e = launch_sequence_index(cu_seqlens, num_seqs, total_tokens, at<int32_t>(workspace, l.seq), st);
    if (e != cudaSuccess) return cuda_fail(e, "sequence index launch");
    a.seq = at<int32_t>(workspace, l.seq);
  }
  const int bx = D < conv_tile_cols() ? D : conv_tile_cols();
  CUtensorMap mx;
  VSSM_TRY(make_map(&mx, x, io, total_tokens, D, bx, conv_tile_rows(W, false, true)));
  kernel_timer_mark(kTimeConvFwd, true, st);
  e = launch_conv1d_fwd(a, io, mx, st);
  kernel_timer_mark(kTimeConvFwd, false, st);
  if (e != cudaSuccess) return cuda_fail(e, "conv1d_fwd launch");
  const bool f = io == IO::F32;
  return check_outputs(a.status, st, {{u, total_tokens * D, f}});
}

int varlen_conv1d_bwd(const void* x, const float* weight, const float* bias, const void* du,
                      const int32_t* cu_seqlens, const int32_t* position_indices, int32_t num_seqs,
                      int64_t total_tokens, int32_t D, int32_t W, int32_t apply_silu,
                      vssm_dtype dtype, void* dx, float* dweight, float* dbias,
                      const float* x_init, const float* dx_last, float* dx_init,
                      void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_("varlen_conv1d_bwd");
  IO io;
  VSSM_TRY(conv_common(x, weight, cu_seqlens, num_seqs, total_tokens, D, W, dtype, &io));
  VSSM_TRY(check_io(du, "du", total_tokens));
  VSSM_TRY(check_io(dx, "dx", total_tokens));
  if (!dweight) return fail(VSSM_ERR_ARG, "dweight is NULL");
  VSSM_TRY(check_states(x_init, "x_init"));
  VSSM_TRY(check_states(dx_last, "dx_last"));
  VSSM_TRY(check_states(dx_init, "dx_init"));
  VSSM_TRY(check_states_rows(x_init || dx_last || dx_init, num_seqs, total_tokens));
  const Layout l = conv_layout(total_tokens, D, W, true);
  VSSM_TRY(check_ws(workspace, workspace_bytes, l.total));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(workspace, 0, l.clear_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace header");
  const int32_t* pos = nullptr;
  if (total_tokens > 0)
    VSSM_TRY(resolve_pos(cu_seqlens, position_indices, num_seqs, total_tokens, workspace, l, st, &pos));
  ConvArgs a{};
  a.x = x; a.w = weight; a.bias = bias; a.pos = pos; a.du = du; a.out = dx;
  a.partial = at<float>(workspace, l.conv_part);
  a.T = total_tokens; a.D = D; a.W = W; a.apply_silu = apply_silu ? 1 : 0;
  a.cu = cu_seqlens; a.num_seqs = num_seqs;
  a.status = at<int>(workspace, 0);
  a.wait_ns = g_wait_ns.load();
  a.force_timeout_cta = g_force_copy_timeout.load();
  if (W > 1) { a.x_init = x_init; a.dx_last = dx_last; a.dx_init = dx_init; }
  if (total_tokens > 0 && (a.x_init || a.dx_last)) {
    e = launch_sequence_index(cu_seqlens, num_seqs, total_tokens, at<int32_t>(workspace, l.seq), st);
    if (e != cudaSuccess) return cuda_fail(e, "sequence index launch");
    a.seq = at<int32_t>(workspace, l.seq);
  }
  // the gradient reaching every sequence's tail values
  e = launch_conv_tails(a, io, true, st);
  if (e != cudaSuccess) return cuda_fail(e, "conv tails launch");
  CUtensorMap mx, mdu;
  std::memset(&mx, 0, sizeof(mx));
  std::memset(&mdu, 0, sizeof(mdu));
  if (total_tokens > 0) {
    const int bx = D < conv_tile_cols() ? D : conv_tile_cols();
    VSSM_TRY(make_map(&mx, x, io, total_tokens, D, bx, conv_tile_rows(W, true, true)));
    VSSM_TRY(make_map(&mdu, du, io, total_tokens, D, bx, conv_tile_rows(W, true, false)));
  }
  e = launch_conv1d_bwd(a, io, mx, mdu, dweight, dbias, st);
  if (e != cudaSuccess) return cuda_fail(e, "conv1d_bwd launch");
  return check_outputs(a.status, st, {{dx, total_tokens * D, io == IO::F32}, {dweight, (int64_t)D * W, true},
                                      {dbias, dbias ? (int64_t)D : 0, true}});
}

// ---------------------------------------------------------------- selective scan
size_t varlen_selective_scan_fwd_workspace_size(int64_t total_tokens, int32_t D, int32_t N) {
  if (total_tokens < 0 || D <= 0 || N <= 0) return 0;
  return scan_layout(total_tokens, D, N, kFwdChunk, false).total;
}

size_t varlen_selective_scan_bwd_workspace_size(int64_t total_tokens, int32_t D, int32_t N) {
  if (total_tokens < 0 || D <= 0 || N <= 0) return 0;
  return scan_layout(total_tokens, D, N, kBwdChunk, true).total;
}

size_t varlen_selective_scan_chunk_states_size(int64_t total_tokens, int32_t D, int32_t N) {
  if (total_tokens < 0 || D <= 0 || N <= 0) return 0;
  return sizeof(float) * (size_t)cdiv(total_tokens, kStateChunk) * (size_t)D * (size_t)N;
}

static int scan_common(const void* u, const void* delta_raw, const float* A, const void* B,
                       const void* C, const void* z, const float* Dskip, const float* dt_bias,
                       const int32_t* pos, const int32_t* cu, int32_t num_seqs,
                       int64_t T, int32_t D, int32_t N, vssm_dtype dtype, IO* io) {
  // the kernels copy these with 16-byte bulk copies
  if (Dskip && !aligned16(Dskip)) return fail(VSSM_ERR_ALIGN, "Dskip is not 16-byte aligned");
  if (dt_bias && !aligned16(dt_bias)) return fail(VSSM_ERR_ALIGN, "dt_bias is not 16-byte aligned");
  if (pos && !aligned16(pos)) return fail(VSSM_ERR_ALIGN, "position_indices is not 16-byte aligned");
  VSSM_TRY(check_dtype(dtype, io));
  VSSM_TRY(check_shape(T, D, num_seqs, cu));
  if (N != 4 && N != 8 && N != 16) return fail(VSSM_ERR_UNSUPPORTED, "N = %d not in {4, 8, 16}", N);
  const int e = io_bytes(*io);
  if (((int64_t)D * e) % 16 != 0)
    return fail(VSSM_ERR_ALIGN, "D * sizeof(io) = %lld is not a multiple of 16", (long long)D * e);
  if ((N * e) % 16 != 0)
    return fail(VSSM_ERR_ALIGN, "N * sizeof(io) = %d is not a multiple of 16", N * e);
  if (!A) return fail(VSSM_ERR_ARG, "A is NULL");
  if (!aligned16(A)) return fail(VSSM_ERR_ALIGN, "A is not 16-byte aligned");
  VSSM_TRY(check_io(u, "u", T));
  VSSM_TRY(check_io(delta_raw, "delta_raw", T));
  VSSM_TRY(check_io(B, "B", T));
  VSSM_TRY(check_io(C, "C", T));
  if (z && !aligned16(z)) return fail(VSSM_ERR_ALIGN, "z is not 16-byte aligned");
  return VSSM_OK;
}

int varlen_selective_scan_fwd(const void* u, const void* delta_raw, const float* A,
                              const void* B, const void* C, const float* Dskip, const void* z,
                              const float* dt_bias, int32_t delta_softplus, float gate_floor,
                              int32_t a_log, const int32_t* cu_seqlens,
                              const int32_t* position_indices,
                              int32_t num_seqs, int64_t total_tokens, int32_t D, int32_t N,
                              vssm_dtype dtype, void* out, void* y, float* chunk_states,
                              const float* initial_states, float* final_states,
                              void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_("varlen_selective_scan_fwd");
  IO io;
  VSSM_TRY(scan_common(u, delta_raw, A, B, C, z, Dskip, dt_bias, position_indices, cu_seqlens,
                        num_seqs, total_tokens, D, N, dtype, &io));
  VSSM_TRY(check_io(out, "out", total_tokens));
  if (y) VSSM_TRY(check_io(y, "y", total_tokens));
  if (chunk_states && !aligned16(chunk_states))
    return fail(VSSM_ERR_ALIGN, "chunk_states is not 16-byte aligned");
  VSSM_TRY(check_states(initial_states, "initial_states"));
  VSSM_TRY(check_states(final_states, "final_states"));
  VSSM_TRY(check_states_rows(initial_states || final_states, num_seqs, total_tokens));
  const int64_t T = total_tokens;
  const Layout l = scan_layout(T, D, N, kFwdChunk, false);
  VSSM_TRY(check_ws(workspace, workspace_bytes, l.total));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(workspace, 0, l.clear_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace header");
  // every inclusive-state word starts as the all-ones NaN (bytes 0xff) that
  // the kernel reads as "not stored yet": a word is its own flag
  if (T > 0) e = cudaMemsetAsync(at<char>(workspace, l.incl), 0xff, l.incl_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "filling the look-back states");
  // an empty sequence ends in the state it starts from
  e = launch_empty_sequence_states(cu_seqlens, num_seqs, (int64_t)D * N, initial_states, final_states, st);
  if (e != cudaSuccess) return cuda_fail(e, "empty-sequence states launch");
  if (T == 0) return VSSM_OK;
  const int32_t* pos = nullptr;
  VSSM_TRY(resolve_pos(cu_seqlens, position_indices, num_seqs, T, workspace, l, st, &pos));
  const int32_t* seq = nullptr;
  if (initial_states || final_states) {
    e = launch_sequence_index(cu_seqlens, num_seqs, T, at<int32_t>(workspace, l.seq), st);
    if (e != cudaSuccess) return cuda_fail(e, "sequence index launch");
    seq = at<int32_t>(workspace, l.seq);
  }

  ScanArgs a{};
  a.u = u; a.dr = delta_raw; a.A = A; a.B = B; a.C = C; a.Dskip = Dskip; a.z = z;
  a.dt_bias = dt_bias; a.pos = pos; a.chunk_states = chunk_states; a.out = out; a.y = y;
  a.seq = seq; a.h_init = initial_states; a.h_final = final_states;
  if (io == IO::BF16) {
    a.Bf32 = at<float>(workspace, l.bcf);
    a.Cf32 = a.Bf32 + T * N;
  }
  a.Af = at<float4>(workspace, l.af);
  a.status = at<int>(workspace, 0);
  a.ticket = at<unsigned>(workspace, 4);
  a.flags = at<int>(workspace, l.flags);
  a.agg = at<float>(workspace, l.agg);
  a.agg_sd = at<float>(workspace, l.agg_sd);
  a.incl = at<float>(workspace, l.incl);
  a.T = T; a.D = D; a.N = N; a.num_seqs = num_seqs;
  a.n_tiles = (int)cdiv(D, kTile);
  a.n_chunks = (int)cdiv(T, kFwdChunk);
  a.delta_softplus = delta_softplus ? 1 : 0;
  a.gate_floor = gate_floor;
  a.a_log = a_log ? 1 : 0;
  a.has_z = z ? 1 : 0;
  a.has_skip = Dskip ? 1 : 0;
  a.box_x = D < kTile ? D : kTile;
  a.box_y = T < kFwdChunk ? (int)T : kFwdChunk;
  a.drop_ticket = g_drop_ticket.load();
  a.wait_ns = g_wait_ns.load();
  a.delay_ticket = g_delay_ticket.load();
  a.delay_ns = g_delay_ns.load();
  CUtensorMap mu, mdr, mz;
  VSSM_TRY(make_map(&mu, u, io, T, D, a.box_x, a.box_y));
  VSSM_TRY(make_map(&mdr, delta_raw, io, T, D, a.box_x, a.box_y));
  VSSM_TRY(make_map(&mz, z, io, T, D, a.box_x, a.box_y));
  e = launch_scan_fwd(a, io, mu, mdr, mz, st);
  if (e != cudaSuccess) return cuda_fail(e, "selective_scan_fwd launch");
  return check_outputs(a.status, st, {{out, T * D, io == IO::F32}, {y, y ? T * D : 0, io == IO::F32},
                                      {final_states, final_states ? (int64_t)num_seqs * D * N : 0, true}});
}

int varlen_conv1d_scan_fwd(const void* x, const float* conv_weight, const float* conv_bias, int32_t W,
                           int32_t apply_silu, const void* delta_raw, const float* A, const void* B,
                           const void* C, const float* Dskip, const void* z, const float* dt_bias,
                           int32_t delta_softplus, float gate_floor, int32_t a_log,
                           const int32_t* cu_seqlens, const int32_t* position_indices, int32_t num_seqs,
                           int64_t total_tokens, int32_t D, int32_t N, vssm_dtype dtype, void* u, void* out,
                           void* y, float* chunk_states, const float* initial_states, float* final_states,
                           void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_("varlen_conv1d_scan_fwd");
  IO io;
  // x takes u's place in the scan's checks (same shape, dtype and alignment)
  VSSM_TRY(scan_common(x, delta_raw, A, B, C, z, Dskip, dt_bias, position_indices, cu_seqlens,
                        num_seqs, total_tokens, D, N, dtype, &io));
  if (W < 1 || W > 4) return fail(VSSM_ERR_UNSUPPORTED, "conv width %d not in 1..4", W);
  if (!conv_weight) return fail(VSSM_ERR_ARG, "conv_weight is NULL");
  if (!aligned16(conv_weight)) return fail(VSSM_ERR_ALIGN, "conv_weight is not 16-byte aligned");
  if (conv_bias && !aligned16(conv_bias)) return fail(VSSM_ERR_ALIGN, "conv_bias is not 16-byte aligned");
  VSSM_TRY(check_io(out, "out", total_tokens));
  if (u) VSSM_TRY(check_io(u, "u", total_tokens));
  if (y) VSSM_TRY(check_io(y, "y", total_tokens));
  if (chunk_states && !aligned16(chunk_states))
    return fail(VSSM_ERR_ALIGN, "chunk_states is not 16-byte aligned");
  VSSM_TRY(check_states(initial_states, "initial_states"));
  VSSM_TRY(check_states(final_states, "final_states"));
  VSSM_TRY(check_states_rows(initial_states || final_states, num_seqs, total_tokens));
  const int64_t T = total_tokens;
  const Layout l = scan_layout(T, D, N, kFwdChunk, false);
  VSSM_TRY(check_ws(workspace, workspace_bytes, l.total));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(workspace, 0, l.clear_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace header");
  if (T > 0) e = cudaMemsetAsync(at<char>(workspace, l.incl), 0xff, l.incl_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "filling the look-back states");
  e = launch_empty_sequence_states(cu_seqlens, num_seqs, (int64_t)D * N, initial_states, final_states, st);
  if (e != cudaSuccess) return cuda_fail(e, "empty-sequence states launch");
  if (T == 0) return VSSM_OK;
  const int32_t* pos = nullptr;
  VSSM_TRY(resolve_pos(cu_seqlens, position_indices, num_seqs, T, workspace, l, st, &pos));
  const int32_t* seq = nullptr;
  if (initial_states || final_states) {
    e = launch_sequence_index(cu_seqlens, num_seqs, T, at<int32_t>(workspace, l.seq), st);
    if (e != cudaSuccess) return cuda_fail(e, "sequence index launch");
    seq = at<int32_t>(workspace, l.seq);
  }
  ScanArgs a{};
  a.u = x; a.dr = delta_raw; a.A = A; a.B = B; a.C = C; a.Dskip = Dskip; a.z = z;
  a.dt_bias = dt_bias; a.pos = pos; a.chunk_states = chunk_states; a.out = out; a.y = y;
  a.seq = seq; a.h_init = initial_states; a.h_final = final_states;
  if (io == IO::BF16) {
    a.Bf32 = at<float>(workspace, l.bcf);
    a.Cf32 = a.Bf32 + T * N;
  }
  a.Af = at<float4>(workspace, l.af);
  a.conv_w = conv_weight; a.conv_b = conv_bias; a.conv_W = W; a.conv_silu = apply_silu ? 1 : 0; a.u_out = u;
  a.status = at<int>(workspace, 0);
  a.ticket = at<unsigned>(workspace, 4);
  a.flags = at<int>(workspace, l.flags);
  a.agg = at<float>(workspace, l.agg);
  a.agg_sd = at<float>(workspace, l.agg_sd);
  a.incl = at<float>(workspace, l.incl);
  a.T = T; a.D = D; a.N = N; a.num_seqs = num_seqs;
  a.n_tiles = (int)cdiv(D, kTile);
  a.n_chunks = (int)cdiv(T, kFwdChunk);
  a.delta_softplus = delta_softplus ? 1 : 0;
  a.gate_floor = gate_floor;
  a.a_log = a_log ? 1 : 0;
  a.has_z = z ? 1 : 0;
  a.has_skip = Dskip ? 1 : 0;
  a.box_x = D < kTile ? D : kTile;
  a.box_y = T < kFwdChunk ? (int)T : kFwdChunk;
  a.drop_ticket = g_drop_ticket.load();
  a.wait_ns = g_wait_ns.load();
  a.delay_ticket = -1;  // the delay knob's build does not carry the fused conv
  a.delay_ns = g_delay_ns.load();
  CUtensorMap mx, mdr, mz;
  // x rows t0 - 3 .. t0 + 127 of every chunk: three rows above the u box
  VSSM_TRY(make_map(&mx, x, io, T, D, a.box_x, a.box_y + 3));
  VSSM_TRY(make_map(&mdr, delta_raw, io, T, D, a.box_x, a.box_y));
  VSSM_TRY(make_map(&mz, z, io, T, D, a.box_x, a.box_y));
  e = launch_scan_fwd(a, io, mx, mdr, mz, st);
  if (e != cudaSuccess) return cuda_fail(e, "conv1d_scan_fwd launch");
  return check_outputs(a.status, st, {{u, u ? T * D : 0, io == IO::F32}, {out, T * D, io == IO::F32},
                                      {y, y ? T * D : 0, io == IO::F32},
                                      {final_states, final_states ? (int64_t)num_seqs * D * N : 0, true}});
}

int varlen_selective_scan_bwd(const void* u, const void* delta_raw, const float* A,
                              const void* B, const void* C, const float* Dskip, const void* z,
                              const float* dt_bias, int32_t delta_softplus, float gate_floor,
                              int32_t a_log, const void* dout,
                              const int32_t* cu_seqlens, const int32_t* position_indices,
                              int32_t num_seqs, int64_t total_tokens, int32_t D, int32_t N,
                              vssm_dtype dtype, const float* chunk_states, const void* y,
                              const float* initial_states, const float* d_final_states,
                              float* d_initial_states,
                              void* du, void* ddelta_raw, float* dA, float* dB, float* dC,
                              float* dDskip, void* dz, float* d_dt_bias,
                              void* workspace, size_t workspace_bytes, void* stream) {
  NvtxRange nvtx_("varlen_selective_scan_bwd");
  IO io;
  VSSM_TRY(scan_common(u, delta_raw, A, B, C, z, Dskip, dt_bias, position_indices, cu_seqlens,
                        num_seqs, total_tokens, D, N, dtype, &io));
  const int64_t T = total_tokens;
  VSSM_TRY(check_io(dout, "dout", T));
  VSSM_TRY(check_io(du, "du", T));
  VSSM_TRY(check_io(ddelta_raw, "ddelta_raw", T));
  VSSM_TRY(check_io(dB, "dB", T));
  VSSM_TRY(check_io(dC, "dC", T));
  if (!dA) return fail(VSSM_ERR_ARG, "dA is NULL");
  if (T > 0 && !chunk_states) return fail(VSSM_ERR_ARG, "chunk_states is NULL");
  if (z && T > 0 && !dz) return fail(VSSM_ERR_ARG, "dz is NULL although z is given");
  if (dz && !aligned16(dz)) return fail(VSSM_ERR_ALIGN, "dz is not 16-byte aligned");
  if (y) VSSM_TRY(check_io(y, "y", T));
  VSSM_TRY(check_states(initial_states, "initial_states"));
  VSSM_TRY(check_states(d_final_states, "d_final_states"));
  VSSM_TRY(check_states(d_initial_states, "d_initial_states"));
  VSSM_TRY(check_states_rows(initial_states || d_final_states || d_initial_states, num_seqs, total_tokens));
  const Layout l = scan_layout(T, D, N, kBwdChunk, true);
  VSSM_TRY(check_ws(workspace, workspace_bytes, l.total));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(workspace, 0, l.clear_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace header");
  // every carry word starts as the all-ones NaN (bytes 0xff) that the kernel
  // reads as "not stored yet": a carry is its own flag
  if (T > 0) e = cudaMemsetAsync(at<char>(workspace, l.incl), 0xff, l.incl_bytes, st);
  if (e != cudaSuccess) return cuda_fail(e, "filling the look-back carries");
  // the gradient reaching an empty sequence's final state reaches its start unchanged
  e = launch_empty_sequence_states(cu_seqlens, num_seqs, (int64_t)D * N, d_final_states, d_initial_states, st);
  if (e != cudaSuccess) return cuda_fail(e, "empty-sequence states launch");
  const bool states = initial_states || d_final_states || d_initial_states;
  if (T > 0 && states) {
    e = launch_sequence_index(cu_seqlens, num_seqs, T, at<int32_t>(workspace, l.seq), st);
    if (e != cudaSuccess) return cuda_fail(e, "sequence index launch");
  }

  ScanArgs a{};
  a.u = u; a.dr = delta_raw; a.A = A; a.B = B; a.C = C; a.Dskip = Dskip; a.z = z;
  a.dt_bias = dt_bias; a.dout = dout; a.chunk_states = const_cast<float*>(chunk_states);
  a.du = du; a.ddr = ddelta_raw; a.dz = z ? dz : nullptr;
  a.y = const_cast<void*>(y);
  a.seq = states ? at<int32_t>(workspace, l.seq) : nullptr;
  a.h_init = initial_states; a.dh_final = d_final_states; a.dh_init = d_initial_states;
  a.status = at<int>(workspace, 0);
  a.ticket = at<unsigned>(workspace, 4);
  a.flags = at<int>(workspace, l.flags);
  a.agg = at<float>(workspace, l.agg);
  a.agg_sd = at<float>(workspace, l.agg_sd);
  a.incl = at<float>(workspace, l.incl);
  a.part_dBC = at<float>(workspace, l.part_bc);
  a.part_dA = at<float>(workspace, l.part_a);
  a.part_dD = at<float>(workspace, l.part_d);
  a.part_dbias = at<float>(workspace, l.part_b);
  a.BD = at<float4>(workspace, l.bcd);
  a.CD = a.BD + cdiv(T, kBwdChunk) * kBwdChunk * N;
  a.tpar = N == 16 ? at<float>(workspace, l.tpar) : nullptr;
  a.T = T; a.D = D; a.N = N; a.num_seqs = num_seqs;
  const int tw = scan_tile(N, true);
  a.n_tiles = (int)cdiv(D, tw);
  a.n_chunks = (int)cdiv(T, kBwdChunk);
  a.delta_softplus = delta_softplus ? 1 : 0;
  a.gate_floor = gate_floor;
  a.a_log = a_log ? 1 : 0;
  a.has_z = z ? 1 : 0;
  a.has_y = (z && y) ? 1 : 0;
  a.has_skip = Dskip ? 1 : 0;
  a.box_x = D < tw ? D : tw;
  a.box_y = T < kBwdChunk ? (int)T : kBwdChunk;
  a.drop_ticket = g_drop_ticket.load();
  a.wait_ns = g_wait_ns.load();
  a.delay_ticket = g_delay_ticket.load();
  a.delay_ns = g_delay_ns.load();
  CUtensorMap mu, mdr, mz, mdo, mcs, my;
  std::memset(&my, 0, sizeof(my));
  std::memset(&mu, 0, sizeof(mu));
  std::memset(&mdr, 0, sizeof(mdr));
  std::memset(&mz, 0, sizeof(mz));
  std::memset(&mdo, 0, sizeof(mdo));
  std::memset(&mcs, 0, sizeof(mcs));
  if (T > 0) {
    const int32_t* pos = nullptr;
    VSSM_TRY(resolve_pos(cu_seqlens, position_indices, num_seqs, T, workspace, l, st, &pos));
    a.pos = pos;
    VSSM_TRY(make_map(&mu, u, io, T, D, a.box_x, a.box_y));
    VSSM_TRY(make_map(&mdr, delta_raw, io, T, D, a.box_x, a.box_y));
    VSSM_TRY(make_map(&mz, z, io, T, D, a.box_x, a.box_y));
    VSSM_TRY(make_map(&mdo, dout, io, T, D, a.box_x, a.box_y));
    if (a.has_y) VSSM_TRY(make_map(&my, y, io, T, D, a.box_x, a.box_y));
    // saved states [chunk][n][d] seen as (chunks * N) rows of D floats; one
    // copy fetches an item's N rows of its tile's channels
    VSSM_TRY(make_map(&mcs, chunk_states, IO::F32, cdiv(T, kStateChunk) * N, D, a.box_x, N));
  }
  e = launch_scan_bwd(a, io, mu, mdr, mz, mdo, mcs, my, dA, dB, dC, dDskip, d_dt_bias, st);
  if (e != cudaSuccess) return cuda_fail(e, "selective_scan_bwd launch");
  const bool f = io == IO::F32;
  return check_outputs(a.status, st, {{du, T * D, f}, {ddelta_raw, T * D, f}, {a.dz, a.dz ? T * D : 0, f},
                                      {dA, (int64_t)D * N, true}, {dB, T * N, true}, {dC, T * N, true},
                                      {dDskip, dDskip ? (int64_t)D : 0, true},
                                      {d_dt_bias, d_dt_bias ? (int64_t)D : 0, true},
                                      {d_initial_states, d_initial_states ? (int64_t)num_seqs * D * N : 0, true}});
}

}  // extern "C"
