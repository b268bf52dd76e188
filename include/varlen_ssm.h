/*
 * varlen_ssm.h -- C ABI of libvarlen_ssm.so: Mamba-1's two sequence-wise
 * operators (depthwise causal conv1d and the selective scan), forward and
 * backward, on PACKED variable-length batches, for NVIDIA GB300 (sm_103a).
 *
 * The operators follow the article "Shanghai AI Lab: packed variable-length
 * Mamba training" (gitcode.csdn).  Its section "Mamba block 中的步骤" sorts
 * the block's steps into element-wise, token-wise and sequence-wise ones and
 * names conv1d and the SSM as the only sequence-wise steps; the sections
 * "conv1d_pack 算子" and "SSM_pack算子" ask that these two steps keep the
 * sequences of one pack from interfering.  The packed input is the
 * FlashAttention-style pair (total_tokens, D) tensor + int32 cu_seqlens that
 * the same article's section "基本原理" describes for its cu_seqlens version.
 *
 * ---------------------------------------------------------------- conventions
 * Layouts   (T, D) tensors are row-major, channel index fastest (token t,
 *           channel d at t*D + d).  B and C are (T, N); A is (D, N); the conv
 *           weight is (D, W) with weight[d][W-1] multiplying the current
 *           token (PyTorch's depthwise Conv1d layout).
 * Dtypes    "I/O" tensors (x, u, delta_raw, z, B, C, out, dout and their
 *           gradients du, ddelta_raw, dz, dx) are VSSM_F32 or VSSM_BF16 as the
 *           call's `dtype` says.  Parameters (A, Dskip, dt_bias, conv weight
 *           and bias) and their gradients are always float32.  All arithmetic,
 *           the scan state and every accumulation are float32; bf16 results are
 *           rounded to nearest-even once, at the store.
 * Pointers  Every data pointer is a DEVICE pointer.  (T, D) tensors, B, C,
 *           the workspace and, for the scan calls, A, Dskip, dt_bias,
 *           chunk_states and position_indices must be 16-byte aligned (the
 *           kernels fetch them with bulk copies), and D * sizeof(io) and
 *           N * sizeof(io) must be multiples of 16; otherwise the call returns
 *           VSSM_ERR_ALIGN without launching (there is no slow fallback).
 * Ownership The caller allocates and frees everything: inputs, outputs,
 *           gradients and the workspace, sized by the matching
 *           *_workspace_size query.  The library never allocates, frees or
 *           synchronises, except vssm_read_status, which synchronises `stream`.
 * Streams   `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *           stream).  Calls are enqueued on it and return before the GPU work
 *           finishes.  Calls sharing a workspace must not overlap on the GPU.
 * Outputs   Outputs and gradients are overwritten, never accumulated into.
 * Edge cases T == 0 is a no-op that still zeroes parameter gradients.
 *           Zero-length sequences are allowed (repeated cu_seqlens values).
 * Supported N in {4, 8, 16} (N * sizeof(io) must be a multiple of 16), conv
 *           width W in 1..4, T < 2^31, D >= 1.
 * Errors    Every call validates its arguments on the host and returns a
 *           negative VSSM_ERR_* code without launching anything.  Conditions
 *           only the GPU can see (malformed cu_seqlens, a look-back wait that
 *           ran out of time) are recorded in a status word inside the
 *           workspace; read it with vssm_read_status.  A per-thread message
 *           describing the last host-side error is kept (vssm_last_error).
 * position_indices
 *           Each call takes cu_seqlens AND an optional position_indices array
 *           (int32, T): the per-token position inside its own sequence, built
 *           once per pack by varlen_position_indices and reusable by every
 *           call on that pack.  Pass NULL to have the call build it in its
 *           workspace first.  A non-NULL array must be the one built from the
 *           same cu_seqlens.
 */
#ifndef VARLEN_SSM_H
#define VARLEN_SSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { VSSM_F32 = 0, VSSM_BF16 = 1 } vssm_dtype;

/* Status codes.  0 is success; host-detected errors are -1..-15; errors the
 * GPU detected (reported by vssm_read_status) are -16 and below. */
#define VSSM_OK 0
#define VSSM_ERR_ARG (-1)              /* bad size, NULL where required, bad flag */
#define VSSM_ERR_DTYPE (-2)            /* dtype not VSSM_F32 / VSSM_BF16 */
#define VSSM_ERR_ALIGN (-3)            /* pointer or row pitch not 16-byte aligned */
#define VSSM_ERR_WORKSPACE (-4)        /* workspace NULL or smaller than the query */
#define VSSM_ERR_CUDA (-5)             /* a CUDA runtime / driver call failed */
#define VSSM_ERR_UNSUPPORTED (-6)      /* N or W outside the supported set */
#define VSSM_ERR_BAD_CU_SEQLENS (-16)  /* cu_seqlens[0] != 0, decreasing, or cu[S] != T */
#define VSSM_ERR_LOOKBACK_TIMEOUT (-17)/* a cross-chunk or tile-copy wait gave up; results invalid */
#define VSSM_ERR_NONFINITE (-18)        /* an output holds a NaN / inf (VSSM_DBG_CHECK_FINITE on) */
#define VSSM_ERR_DEVICE_CHECK (-19)     /* a device index check failed (VSSM_CHECKS=1 build only) */

/* Tokens per saved scan-state chunk: the forward scan can save the state at
 * every multiple of this many tokens for the backward scan. */
#define VSSM_STATE_CHUNK 32

/* ------------------------------------------------------------ position indices
 * position_indices[t] = t - cu_seqlens[s] for cu_seqlens[s] <= t < cu_seqlens[s+1]:
 * the token's position inside its own sequence, the auxiliary structure the
 * article's pack() builds ("conv1d_pack 算子", figure (a): lengths [4,2,3,7]
 * give 0 1 2 3 0 1 0 1 2 0 1 2 3 4 5 6).
 *   cu_seqlens        device int32[num_seqs + 1]
 *   position_indices  device int32[total_tokens], written
 *   status            device int32, nullable; the kernel ORs a nonzero value
 *                     into it when cu_seqlens is malformed (see
 *                     vssm_status_code to turn it into a VSSM_ERR_* code).
 */
int varlen_position_indices(const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                            int32_t* position_indices, int32_t* status, void* stream);

/* Maps a raw status word written by the GPU to VSSM_OK or a VSSM_ERR_* code. */
int vssm_status_code(int32_t status_word);

/* ------------------------------------------------------------ conv1d_pack
 * Forward ("conv1d_pack 算子", Algorithm 1): depthwise causal conv of width W
 * whose taps stop early at each sequence's first token; tap k reaches back k
 * tokens and is used only if position_indices[t] >= k:
 *   pre[t,d] = bias[d] + sum_{k=0}^{W-1} [pos[t] >= k] weight[d][W-1-k] x[t-k,d]
 *   u[t,d]   = apply_silu ? pre * sigmoid(pre) : pre
 * x, u: (T, D) io; weight: (D, W) f32; bias: (D) f32, nullable (zero).
 * Conv tails of cut sequences (the conv half of the article's future work:
 * a sequence cut across packs keeps passing data), both nullable f32
 * (num_seqs, D, W-1), entry [s][d][j]:
 *   x_init: the W-1 inputs before each sequence's first token (the previous
 *     part's x_last); a tap that reaches before the start reads them instead
 *     of stopping (zero when NULL: the plain early stop);
 *   x_last: receives each sequence's last W-1 inputs, reaching back into its
 *     x_init when the sequence is shorter than W-1.
 */
size_t varlen_conv1d_fwd_workspace_size(int64_t total_tokens, int32_t D, int32_t W);
int varlen_conv1d_fwd(const void* x, const float* weight, const float* bias,
                      const int32_t* cu_seqlens, const int32_t* position_indices, int32_t num_seqs,
                      int64_t total_tokens, int32_t D, int32_t W, int32_t apply_silu,
                      vssm_dtype dtype, void* u, const float* x_init, float* x_last,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Backward (same section: the backward pass stops dx and dweight at sequence
 * edges too, reading the position W-1 tokens LATER to know where a sequence
 * ends).  With g[t] = du[t] * d(u)/d(pre) at t:
 *   dx[t,d]        = sum_k [t+k < T and pos[t+k] >= k] weight[d][W-1-k] g[t+k,d]
 *   dweight[d][W-1-k] = sum_t [pos[t] >= k] g[t,d] x[t-k,d]
 *   dbias[d]       = sum_t g[t,d]
 * x, du, dx: (T, D) io; dweight (D, W) f32; dbias (D) f32, nullable.  The
 * reductions over tokens run in a fixed order (bitwise repeatable).
 * x_init: the forward call's (nullable).  dx_last: nullable (num_seqs, D,
 * W-1), the gradient reaching each sequence's x_last from outside.  dx_init:
 * nullable (num_seqs, D, W-1), receives the gradient reaching each sequence's
 * x_init.
 */
size_t varlen_conv1d_bwd_workspace_size(int64_t total_tokens, int32_t D, int32_t W);
int varlen_conv1d_bwd(const void* x, const float* weight, const float* bias, const void* du,
                      const int32_t* cu_seqlens, const int32_t* position_indices, int32_t num_seqs,
                      int64_t total_tokens, int32_t D, int32_t W, int32_t apply_silu,
                      vssm_dtype dtype, void* dx, float* dweight, float* dbias,
                      const float* x_init, const float* dx_last, float* dx_init,
                      void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------ SSM_pack
 * Forward ("SSM_pack算子": the state must not pass from one packed sequence to
 * the next; the transition factor is zeroed at every sequence start, which is
 * the same as starting each sequence from h = 0):
 *   r      = delta_raw[t,d] + dt_bias[d]
 *   delta  = delta_softplus ? log(1 + exp(r)) : r
 *   h_t[n] = exp(delta A[d,n]) h_{t-1}[n] + delta B[t,n] u[t,d],  h = 0 before a start
 *   y      = sum_n C[t,n] h_t[n] + Dskip[d] u[t,d]
 *   out    = z ? y * SiLU(z[t,d]) : y
 * u, delta_raw, z, out: (T, D) io; B, C: (T, N) io; A: (D, N) f32;
 * Dskip, dt_bias: (D) f32.  Dskip, z, dt_bias are nullable (zero / no gate).
 * chunk_states: nullable f32 (ceil(T / VSSM_STATE_CHUNK), N, D); when given,
 * entry [c][n][d] receives state n of channel d just before token
 * c*VSSM_STATE_CHUNK, which the backward call needs.
 * y: nullable (T, D) io; when given it receives the output before the gate,
 * y above (equal to out when z is NULL), which the backward call can take
 * instead of recomputing it for dz.  16-byte aligned like out.
 * Two variants from the article's pages, both off at 0:
 *   gate_floor: the GateFloor gate, out = y * (SiLU(z) + gate_floor) (a
 *     positive bias that keeps the gate above zero; no effect without z);
 *   a_log: nonzero when A holds A_log, the stored parameterisation with
 *     A = -exp(A_log); the backward then returns dA_log = dA * A in dA.
 * Sequence states (the article's future work: a long sequence cut at the end
 * of a pack into two parts that still pass data between them), both
 * nullable f32 (num_seqs, D, N), entry [s][d][n] for state n of channel d:
 *   initial_states: the state each sequence starts from (h before its first
 *     token; zero when NULL), e.g. the previous part's final state;
 *   final_states: receives the state after each sequence's last token (the
 *     initial state for an empty sequence).
 */
size_t varlen_selective_scan_fwd_workspace_size(int64_t total_tokens, int32_t D, int32_t N);
size_t varlen_selective_scan_chunk_states_size(int64_t total_tokens, int32_t D, int32_t N);
int varlen_selective_scan_fwd(const void* u, const void* delta_raw, const float* A,
                              const void* B, const void* C, const float* Dskip, const void* z,
                              const float* dt_bias, int32_t delta_softplus, float gate_floor,
                              int32_t a_log, const int32_t* cu_seqlens,
                              const int32_t* position_indices,
                              int32_t num_seqs, int64_t total_tokens, int32_t D, int32_t N,
                              vssm_dtype dtype, void* out, void* y, float* chunk_states,
                              const float* initial_states, float* final_states,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Backward: the reverse scan of the state gradient, which resets at every
 * sequence END (the article's "SSM_pack" backward), recomputing the forward
 * states from chunk_states.  Gradients (all overwritten):
 *   du, ddelta_raw (w.r.t. delta_raw, i.e. before softplus), dz: (T, D) io
 *   dA (D, N), dB (T, N), dC (T, N), dDskip (D), d_dt_bias (D): f32
 * dz, dDskip, d_dt_bias may be NULL.  dz is written only when z is given.
 * chunk_states is the array the forward call filled.  y is nullable: the
 * forward call's pre-gate output (its `y` argument); with z given, dz then
 * uses it (dz = dout * y * SiLU'(z)) instead of recomputing C.h + Dskip u,
 * which saves the backward that work; with y NULL it is recomputed (in fp32,
 * so for bf16 io the two ways differ by y's rounding to bf16).
 * initial_states: the forward call's (nullable; the states are recomputed
 * from it at every sequence start).  d_final_states: nullable (num_seqs, D,
 * N), the gradient reaching each sequence's final state from outside (from
 * the next part of a cut sequence).  d_initial_states: nullable (num_seqs, D,
 * N), receives the gradient reaching each sequence's starting state (for an
 * empty sequence, its d_final_states entry).  Every
 * reduction (over channels for dB/dC, over tokens for dA/dDskip/d_dt_bias) is
 * atomic-free and runs in a fixed order, so results are bitwise repeatable.
 */
size_t varlen_selective_scan_bwd_workspace_size(int64_t total_tokens, int32_t D, int32_t N);
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
                              void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------ allocation-free forward scan
 * The article has no counterpart to this call; it exists for callers of this
 * library that cannot allocate device memory where they run the scan: code
 * running inside an allocator's own callbacks, runtimes that reserved the whole
 * device for their own pool up front, or hot paths where allocation is not
 * allowed because it could stall or fail mid-step.
 *
 * It computes exactly what varlen_selective_scan_fwd computes, with the same
 * arguments minus the workspace: the look-back scratch lives in one static
 * device array of VSSM_NOALLOC_SCRATCH_BYTES built into the library, held by
 * every GPU that loads it until the process exits.  The call allocates nothing
 * (no cudaMalloc, no library allocator); the caller still provides every input
 * and output.
 *   - The first call made with a given device current looks up the array's
 *     device address (cudaGetSymbolAddress) and caches it; make that first call
 *     before any stream capture on that device.  The cached address belongs to
 *     the device's primary context: after cudaDeviceReset (or anything else
 *     that destroys that context) it is stale, and the process must not call
 *     this entry point on that device again.
 *   - A problem whose scratch would not fit (about T*D*(N+1)/16 + 8*T
 *     bytes: T = 8192 tokens at D = 4096, N = 16 needs 36 MB and fits;
 *     T = 16384 needs 69 MB and does not) is rejected with
 *     VSSM_ERR_WORKSPACE and a message naming both sizes, before anything is
 *     launched.
 *   - Every call on a device shares the array and finds the previous call's
 *     contents; on `stream`, before its kernels, the call clears what must
 *     start at zero (status, ticket, look-back flags) and fills the look-back
 *     states with all-ones words.  Calls that overlap on the GPU (other
 *     streams, other host threads) race on the array.
 *   - status: nullable device int32 the call zeroes and into which device-side
 *     errors are OR-ed (decode with vssm_status_code); NULL keeps them in the
 *     scratch, where they cannot be read back.
 *   - The test knobs of vssm_debug_set apply as they do to
 *     varlen_selective_scan_fwd.
 */
#define VSSM_NOALLOC_SCRATCH_BYTES (64u << 20)
int varlen_selective_scan_fwd_noalloc(const void* u, const void* delta_raw, const float* A,
                                      const void* B, const void* C, const float* Dskip,
                                      const void* z, const float* dt_bias, int32_t delta_softplus,
                                      float gate_floor, int32_t a_log,
                                      const int32_t* cu_seqlens, const int32_t* position_indices,
                                      int32_t num_seqs, int64_t total_tokens, int32_t D, int32_t N,
                                      vssm_dtype dtype, void* out, void* y, float* chunk_states,
                                      const float* initial_states, float* final_states,
                                      int32_t* status, void* stream);

/* ------------------------------------------------------------ packing (host)
 * The article's section 结论与讨论: its pack method takes sequences in
 * arrival order and seals a pack when the next sequence does not fit (19.1 %
 * padding on its pretraining data); sorting a portion of the pending
 * sequences first and then packing greedily brings that down to 0.46 %.
 *   VSSM_PACK_SEQUENTIAL: arrival order, sealed when the next does not fit;
 *   VSSM_PACK_LOCAL_GREEDY: the sequences are taken `window` at a time, each
 *     window sorted longest first (equal lengths in arrival order) and every
 *     sequence placed in the first of the window's packs with room for it
 *     (first fit, decreasing); a window's packs are sealed before the next.
 * Host arrays, caller-allocated: lengths[num_seqs] (0 .. pack_size);
 * order[num_seqs] receives the sequence indices pack after pack;
 * pack_offsets[num_seqs + 1]: pack p holds order[pack_offsets[p] ..
 * pack_offsets[p+1]); *num_packs; *padding_rate = padded tokens / (num_packs
 * * pack_size).  Returns VSSM_ERR_ARG for a negative length, a length above
 * pack_size, a non-positive pack_size or (local greedy) window, an unknown
 * method, or a NULL array.  Runs on the calling thread; no GPU work.
 */
enum { VSSM_PACK_SEQUENTIAL = 0, VSSM_PACK_LOCAL_GREEDY = 1 };
int varlen_pack_sequences(const int32_t* lengths, int32_t num_seqs, int32_t pack_size, int32_t method,
                          int32_t window, int32_t* order, int32_t* pack_offsets, int32_t* num_packs,
                          double* padding_rate);

/*
 * varlen_conv1d_scan_fwd: varlen_conv1d_fwd followed by
 * varlen_selective_scan_fwd in one call, with u computed on chip.  It is the
 * fusion idea of the memory-efficient path in "从 1 卡到 N 卡 Mamba 分布式训练"
 * (gsyq.cn), section 显存开关, applied to the two sequence-wise operators of
 * the article's section "Mamba block 中的步骤": the scan kernel reads the conv
 * input x (with the W-1 rows before each chunk) instead of u, evaluates
 * u = SiLU(bias + sum_k weight[d][W-1-k] x[t-k] [pos[t] >= k]) (no SiLU when
 * apply_silu is 0) in the conv call's arithmetic and order, rounds it to the
 * I/O type as that call's store does, and scans it.  The results equal the
 * two calls', bit for bit.
 *   x, conv_weight (D, W), conv_bias (nullable), W (1..4), apply_silu: as
 *       varlen_conv1d_fwd (conv_weight and conv_bias 16-byte aligned); the
 *       calls with conv tails (x_init / x_last) have no fused form.
 *   u:  nullable (T, D) output receiving the conv output, which the backward
 *       call needs; NULL when only the forward is wanted.
 *   every other argument, the workspace (varlen_selective_scan_fwd_workspace_size)
 *   and the status word are those of varlen_selective_scan_fwd.
 */
int varlen_conv1d_scan_fwd(const void* x, const float* conv_weight, const float* conv_bias, int32_t W,
                           int32_t apply_silu, const void* delta_raw, const float* A, const void* B,
                           const void* C, const float* Dskip, const void* z, const float* dt_bias,
                           int32_t delta_softplus, float gate_floor, int32_t a_log,
                           const int32_t* cu_seqlens, const int32_t* position_indices, int32_t num_seqs,
                           int64_t total_tokens, int32_t D, int32_t N, vssm_dtype dtype, void* u, void* out,
                           void* y, float* chunk_states, const float* initial_states, float* final_states,
                           void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------ status, errors, knobs
 * vssm_read_status: synchronises `stream`, reads the status word the last call
 * using `workspace` left there, and stores VSSM_OK or a VSSM_ERR_* code in
 * *status.  Returns VSSM_OK or VSSM_ERR_CUDA / VSSM_ERR_ARG.
 */
int vssm_read_status(const void* workspace, void* stream, int* status);
const char* vssm_strerror(int code);
const char* vssm_last_error(void);      /* thread-local; "" if none */
/* 1 when this library is the checked build (compiled with VSSM_CHECKS=1):
 * its kernels check the sequence-state rows they index by a token's sequence
 * (rows a malformed cu_seqlens could push past num_seqs) and skip a failing
 * access, ORing a bit into the status word instead (vssm_read_status then
 * returns VSSM_ERR_DEVICE_CHECK; nothing traps), and calls given position
 * indices check them against cu_seqlens (VSSM_ERR_BAD_CU_SEQLENS).  0 in the
 * ordinary build, where neither check runs. */
int vssm_checks_build(void);

/* Test knobs (process-wide).  VSSM_DBG_DROP_FLAG: the scan work item with this
 * ticket never publishes its look-back flag (-1 = off), so the waits behind it
 * run out of time and report VSSM_ERR_LOOKBACK_TIMEOUT instead of hanging.
 * VSSM_DBG_WAIT_NS: the time limit of each look-back wait in nanoseconds
 * (default 1e9).  VSSM_DBG_DELAY_ITEM: the scan work item with this ticket
 * sleeps VSSM_DBG_DELAY_NS nanoseconds (default 2e5, at most 1e7) before it
 * stores its inclusive state (-1 = off), so the items after it must walk back
 * past published aggregates; the results do not change, bit for bit.  The
 * delay applies to fp32 scan calls with N = 16 and no sequence states, which
 * then run a build of the kernels of their own (the other builds carry no
 * code for it); other calls ignore it.  VSSM_DBG_FORCE_COPY_TIMEOUT: in the
 * conv calls, the CTA with this index reports its tile-copy wait as timed out
 * once the copy has landed (-1 = off), so a test sees VSSM_ERR_LOOKBACK_TIMEOUT
 * in the call's status word without any copy failing; the conv calls' copy
 * waits also take their limit from VSSM_DBG_WAIT_NS.
 * Returns VSSM_OK or VSSM_ERR_ARG. */
#define VSSM_DBG_DROP_FLAG 1
#define VSSM_DBG_WAIT_NS 2
#define VSSM_DBG_DELAY_ITEM 3
#define VSSM_DBG_DELAY_NS 4
#define VSSM_DBG_FORCE_COPY_TIMEOUT 5
/* VSSM_DBG_CHECK_FINITE: 1 makes every conv / scan call check its outputs
 * after its kernels and OR a bit into its status word when any output holds a
 * NaN or an infinity (vssm_read_status then returns VSSM_ERR_NONFINITE); 0
 * (the default) skips the check.  It makes a run whose values have gone bad
 * fail loudly: the aimodeling.com page on near-zero embedding rows stalling
 * the training of gated models describes how such a failure otherwise stays
 * silent until the loss shows it. */
#define VSSM_DBG_CHECK_FINITE 6
/* VSSM_DBG_KERNEL_EVENTS: 1 makes the conv and scan calls record a CUDA event
 * pair on their stream around their main kernel (the conv1d tile kernel, the
 * scan kernel; not the calls' memsets, operand staging or fixed-order sums),
 * so that a benchmark can time the kernels alone while it times the calls; 0
 * (the default) records nothing and drops what was recorded.  Read the
 * totals with vssm_kernel_time. */
#define VSSM_DBG_KERNEL_EVENTS 7
int vssm_debug_set(int knob, int64_t value);

/* Total device time (ms) and number of launches of the main kernel of one
 * kind of call since the last read, from the events VSSM_DBG_KERNEL_EVENTS
 * records: kind 0 varlen_conv1d_fwd, 1 varlen_selective_scan_fwd (and the
 * fused call), 2 varlen_selective_scan_bwd, 3 varlen_conv1d_bwd.  Waits for
 * the recorded events to complete, then forgets them.  Returns VSSM_OK,
 * VSSM_ERR_ARG (bad kind or NULL pointers) or VSSM_ERR_CUDA. */
int vssm_kernel_time(int kind, double* total_ms, int64_t* launches);

#ifdef __cplusplus
}
#endif
#endif /* VARLEN_SSM_H */
