/*
 * gdp_prefill.h -- C ABI of the GB300 (sm_103a) chunked Gated DeltaProduct
 * varlen prefill library (libgdp_gb300.so).
 *
 * What it computes (FlashInfer API page
 * "flashinfer.gdp_prefill.chunk_gated_delta_product", opening paragraph and
 * display equation): per real token t of each packed sequence,
 *
 *     S *= alpha_t                                   (alpha_t = exp(g_t))
 *     for j = 0 .. n-1:  v_new = beta_{t,j} (v_{t,j} - S k_{t,j});  S += v_new (x) k_{t,j}
 *     o_t = scale * S q_t
 *
 * with n = num_householder updates per token on the expanded sub-token stream
 * (rows t*n .. t*n+n-1 of k, v, beta) and a V-major fp32 state S[v][k] per
 * (sequence, head).  The work is chunked in 64-row chunks (Megatron-Core API
 * page "core.ssm.ops.gdp.chunk", stage list): descriptors, within-chunk base-2
 * decay cumsum (+ optional q/k L2 norm), WY factors, inter-chunk state scan,
 * output combine and final-state scatter.
 *
 * Conventions for every entry point:
 *   - Every pointer is a DEVICE pointer owned by the caller, except the
 *     gdp_prefill_args struct itself (host memory, read during the call only).
 *   - The library allocates nothing, never synchronises the device and never
 *     reads device memory from the host, so a call can be captured in a CUDA
 *     graph (Megatron page, closing paragraph: data-dependent descriptor
 *     lengths on the host are what break capture; here they are built on the
 *     device into buffers whose sizes depend on shapes only).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream); all work is
 *     enqueued on it, in order.
 *   - A host-side argument error returns a non-zero gdp_status before any
 *     launch and leaves every buffer untouched; gdp_last_error() then returns
 *     a one-line reason (per calling thread).  Data-dependent errors that
 *     only the device can see (a bad cu_seqlens entry, an out-of-range slot)
 *     are reported by OR-ing GDP_DEV_ERR_* bits into *device_status (when
 *     given); the affected sequence is skipped, nothing traps.
 *   - The caller serialises calls that share a workspace (same stream).
 */
#ifndef GDP_PREFILL_H
#define GDP_PREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDP_ABI_VERSION 2 /* 2: the input-variant fields at the end of gdp_prefill_args */
#define GDP_CHUNK 64 /* chunk size of both streams (Megatron page, stage list) */

typedef enum gdp_status {
  GDP_OK = 0,
  GDP_ERR_INVALID_ARG = 1, /* NULL required pointer, bad shape, bad stride, bad mode mix */
  GDP_ERR_UNSUPPORTED = 2, /* a shape/dtype this build does not serve (reason in gdp_last_error) */
  GDP_ERR_ALIAS = 3,       /* output_state overlaps initial_state (FlashInfer page, output_state) */
  GDP_ERR_WORKSPACE = 4,   /* workspace NULL, misaligned or smaller than gdp_prefill_workspace_bytes */
  GDP_ERR_CUDA = 5         /* a CUDA launch/attribute call failed (reason in gdp_last_error) */
} gdp_status;

/* Element types of the input-variant fields (gdp_prefill_args, ABI version 2). */
typedef enum gdp_dtype {
  GDP_DTYPE_DEFAULT = 0, /* the field's version-1 type */
  GDP_DTYPE_F32 = 1,
  GDP_DTYPE_BF16 = 2,
  GDP_DTYPE_F16 = 3
} gdp_dtype;

/* Bits OR-ed into *device_status by the kernels. */
#define GDP_DEV_ERR_CU_SEQLENS 0x1u /* cu_seqlens not non-decreasing from 0 to T: bad sequences skipped */
#define GDP_DEV_ERR_SLOT 0x2u       /* state_indices entry outside [-1, num_slots): treated as padding */
#define GDP_DEV_ERR_DESC 0x4u       /* chunk counts exceed the padded descriptor lengths: tail skipped */
#define GDP_DEV_ERR_TIMEOUT 0x8u    /* a kernel gave up a bounded wait on its own tensor-core or copy
                                       completion (about a second); its outputs are undefined */
#define GDP_DEV_ERR_BOUNDS 0x10u    /* (GDP_DEBUG_BOUNDS builds only) a global index failed its range
                                       check; the access was skipped: see gdp_debug_bounds_record */

/*
 * Arguments of one prefill call.  Shapes use T real tokens, N sequences,
 * H state heads (the heads of g, beta, the states and the output; q, k and v
 * have H heads unless the head-count fields at the end say otherwise),
 * K = V = head size, M = num_householder.  Element strides are in ELEMENTS;
 * the innermost dimension is always contiguous (FlashInfer page, parameter q).
 * The types named below are those of a zero-filled variant tail (the fields
 * after device_status); those fields widen them.
 */
typedef struct gdp_prefill_args {
  /* q [T, Hq, K] bf16 at real-token rows (FlashInfer page, parameter q). */
  const void *q;
  int64_t q_stride_t, q_stride_h;
  /* k [T*M, Hk, K] bf16 on the expanded stream: token t's M updates are rows
     t*M .. t*M+M-1 (FlashInfer page, parameter k; Megatron page, parameter k). */
  const void *k;
  int64_t k_stride_t, k_stride_h;
  /* v [T*M, Hv, V] bf16, same rows as k (FlashInfer page, parameter v). */
  const void *v;
  int64_t v_stride_t, v_stride_h;
  /* g [T, H] fp32, contiguous: natural-log decay, alpha_t = exp(g_t)
     (Megatron page, parameter g).  NULL = no decay. */
  const float *g;
  /* beta [T*M, H] fp32, contiguous, post-sigmoid (FlashInfer page, parameter
     beta).  NULL = all ones. */
  const float *beta;
  /* cu_seqlens [N+1] over real tokens, int32 (cu_seqlens_int64 = 0) or int64
     (FlashInfer page, parameter cu_seqlens). */
  const void *cu_seqlens;
  int cu_seqlens_int64;
  int64_t T, N;
  int H, K, V, num_householder;
  /* Readout scale; <= 0 (or NaN) selects 1/sqrt(K) (FlashInfer page, scale:
     None or 0.0; Megatron page, scale: K ** -0.5). */
  float scale;
  /* Non-zero: L2-normalise q and k rows in fp32 inside the kernels,
     x / sqrt(sum x^2 + 1e-6) (FlashInfer page, use_qk_l2norm_in_kernel). */
  int use_qk_l2norm;

  /* Incoming state, one of two modes (or neither = zero state):
     dense: initial_state [N, H, V, K] fp32 V-major (FlashInfer page,
     initial_state); cache: state [num_slots, H, V, K] fp32 read and written IN
     PLACE at slot state_indices[i] (int32 [N]); -1 marks a padding sequence,
     which starts from zero, still produces output and writes no slot
     (Megatron page, parameters state and state_indices).  In cache mode
     output_state must be NULL: the final state goes to the cache only.
     Every state buffer (initial_state, state, output_state, chunk_states) is
     contiguous and 16-byte aligned; a misaligned one is GDP_ERR_INVALID_ARG. */
  const float *initial_state;
  float *state;
  const int32_t *state_indices;
  int64_t num_slots;

  /* o [T, H, V] bf16, contiguous, written (FlashInfer page, output). */
  void *output;
  /* Final state [N, H, V, K] fp32 or NULL.  Must not overlap initial_state:
     several CTAs share one sequence, so a CTA writing the final state would
     race one still reading the incoming state (FlashInfer page,
     output_state). */
  float *output_state;
  /* Chunk states [nt_pad, H, V, K] fp32 or NULL (= return_chunk_states off).
     Row chunk_offsets[i] + c holds sequence i's state ENTERING token chunk c,
     i.e. after its first 64*c tokens (Megatron page, return_chunk_states).
     Rows past the real count are not written. */
  float *chunk_states;

  /* Optional prebuilt descriptors from gdp_build_descriptors (all three or
     none; Megatron page, parameters chunk_indices, chunk_indices_dp,
     chunk_offsets): chunk_indices [nt_pad, 2], chunk_indices_dp [ntdp_pad, 2]
     int32 rows (sequence, local chunk), (-1, -1) past the real count;
     chunk_offsets [N+1] int32 exclusive prefix sum of ceil(L_i / 64).
     They must come from the same cu_seqlens and M.  When NULL the call builds
     them itself on the device.  nt_pad / ntdp_pad must be at least the
     shape-only bounds gdp_nt_pad(T, N) / gdp_ntdp_pad(T, N, M) (0 = use those
     bounds); chunk_states, when given, has nt_pad rows. */
  const int32_t *chunk_indices;
  const int32_t *chunk_indices_dp;
  const int32_t *chunk_offsets;
  int64_t nt_pad, ntdp_pad;

  /* Scratch: at least gdp_prefill_workspace_bytes(...) bytes, 256-byte
     aligned, owned by the caller, contents undefined on entry and exit. */
  void *workspace;
  size_t workspace_bytes;
  /* Optional uint32 status word; GDP_DEV_ERR_* bits are OR-ed in. */
  uint32_t *device_status;

  /* ---- Input variants (ABI version 2; zero keeps every type and head count
     above).  FlashInfer page, parameters q, k, v, g, beta, initial_state. ---- */
  /* Type of q, k, v and output: GDP_DTYPE_BF16 (DEFAULT) or GDP_DTYPE_F16
     (parameters q, k, v: float16 or bfloat16).  The output takes this type. */
  int qkv_dtype;
  /* Type of g: GDP_DTYPE_F32 (DEFAULT), GDP_DTYPE_BF16 or GDP_DTYPE_F16
     (parameter g).  Contiguous [T, H] in every type. */
  int g_dtype;
  /* 0: g holds natural-log decays, alpha_t = exp(g_t) (Megatron page,
     parameter g).  1: g holds alpha_t itself, the forget gate in linear space,
     in (0, 1] (FlashInfer page, parameter g).  An alpha outside that range is
     read as max(alpha, exp(-80)): zero or a negative value decays the state to
     about 1e-35 of itself instead of producing NaN. */
  int g_is_alpha;
  /* Type of beta: GDP_DTYPE_F32 (DEFAULT) or the q/k/v type (parameter beta:
     float32 or q.dtype).  Contiguous [T*M, H]. */
  int beta_dtype;
  /* Type of initial_state: GDP_DTYPE_F32 (DEFAULT) or GDP_DTYPE_BF16
     (parameter initial_state).  The cache `state`, output_state and
     chunk_states are always fp32. */
  int initial_state_dtype;
  /* Head counts of q, k and v; 0 means H.  Every count divides H,
     H = max(num_q_heads, num_v_heads), and num_k_heads equals num_q_heads or
     num_v_heads (parameters k, v).  State head h reads q head
     h / (H / num_q_heads), k head h / (H / num_k_heads) and v head
     h / (H / num_v_heads): a head of a smaller count serves a run of
     consecutive state heads (the page names the counts but not the map; this
     is the reading taken).  The head strides above are per head of each
     tensor.  Any other combination is GDP_ERR_INVALID_ARG. */
  int num_q_heads, num_k_heads, num_v_heads;
} gdp_prefill_args;

/* Shape-only descriptor bounds: floor((T + 63 N) / 64) and floor((M T + 63 N) / 64). */
int64_t gdp_nt_pad(int64_t T, int64_t N);
int64_t gdp_ntdp_pad(int64_t T, int64_t N, int num_householder);

/* Workspace bytes for a call of this shape (shape-only; the same value for
   every cu_seqlens with the same T and N).  Returns 0 for an invalid shape. */
size_t gdp_prefill_workspace_bytes(int64_t T, int64_t N, int H, int K, int V, int num_householder);

/*
 * How a call of this shape runs (shape-only, like the workspace size; no
 * device access).  The scan of each (sequence, head) is a serial chain over
 * its 64-row expanded chunks (Megatron-Core API page "core.ssm.ops.gdp.chunk",
 * stage 3), so a call runs in one of three ways:
 *   - plain: descriptors, WY, scan (3 launches);
 *   - segmented (few long chains): the chunks in *segments of about 128, the
 *     WY of segment k + 1 beside the scan of segment k (1 + 2 segments launches);
 *   - split chains (few sequences, N <= 32, over few heads): every sequence
 *     cut into pieces of *piece_chunks expanded chunks that run side by side.
 *     The recurrence is affine in the state, S' = S Phi + B, so a first scan
 *     pass finds each piece's B (from a zero state) and Phi (from the identity
 *     with V = 0), a combine kernel chains the pieces' entering states, and a
 *     second scan pass runs every piece from its own (5 launches).
 *     *piece_rows bounds the number of pieces.  The results agree with the
 *     plain form to rounding (fp32 state arithmetic in a different order).
 * Outputs (any may be NULL): segments (1 unless segmented), piece_chunks (0
 * unless split), piece_rows, launches (kernels one call enqueues; 0 for
 * N = 0).  GDP_ERR_INVALID_ARG for an invalid shape.
 */
gdp_status gdp_prefill_plan(int64_t T, int64_t N, int H, int K, int V, int num_householder, int64_t *segments,
                            int64_t *piece_chunks, int64_t *piece_rows, int64_t *launches);

/*
 * gdp_prefill_varlen_fused: the same prefill as one fused kernel per (sequence, head) -- the
 * WY work, the state scan, the outputs and the state scatter of every expanded chunk in one
 * CTA, so no operand image or U^T reaches the workspace or HBM (Megatron page, stages 1-4 as
 * one pipeline) -- after the descriptor kernel.  Over few sequences (N <= 32) the chains are
 * split into pieces as in gdp_prefill_plan (a pass from zero and from the identity, the
 * combine, a pass from the entering states).  Arguments, results and tolerances are those of
 * gdp_prefill_varlen; the workspace is the same size.  Served: bf16 q/k/v (heads may be
 * grouped), fp32 natural-log g (or NULL), fp32 beta (or NULL), an fp32 dense initial state or
 * the cache, K = V = 128, num_householder >= 2; anything else is GDP_ERR_UNSUPPORTED before any
 * launch.  Measured on one GB300 it is slower than gdp_prefill_varlen on every benchmark
 * workload (its chunks' WY work lies on the serial state chain), which is why
 * gdp_prefill_varlen does not route calls here.  The _profiled form records 4 events like
 * gdp_prefill_varlen_profiled (the third equal to the second: no WY stage).
 */
gdp_status gdp_prefill_varlen_fused(const gdp_prefill_args *args, void *stream);
gdp_status gdp_prefill_varlen_fused_profiled(const gdp_prefill_args *args, void *stream, void *const *events,
                                             int num_events);

/*
 * 1 when gdp_prefill_varlen_fused serves a common-contract call of this shape (K = V = 128,
 * num_householder >= 2), with its plan: piece_chunks (0 unless the chains are split),
 * piece_rows and launches (any may be NULL); 0 otherwise (nothing written).  Shape-only.
 */
int gdp_prefill_fused(int64_t T, int64_t N, int H, int K, int V, int num_householder, int64_t *piece_chunks,
                      int64_t *piece_rows, int64_t *launches);

/*
 * The prefill forward pass: enqueue descriptors (unless prebuilt), the prep
 * + WY kernel and the state-scan / output kernel on `stream`.
 * Returns GDP_OK once enqueued.
 */
gdp_status gdp_prefill_varlen(const gdp_prefill_args *args, void *stream);

/*
 * Same as gdp_prefill_varlen, and records `events` (cudaEvent_t handles
 * created by the caller with timing enabled) on `stream` around the stages:
 * events[0] before the descriptor kernel, [1] after it, [2] after the WY
 * kernel, [3] after the scan/output kernel (in a split-chains call, after
 * its two scan passes and the combine kernel).  num_events must be 4.  Used by
 * the bench to time each kernel on its own stream; the results are identical
 * to gdp_prefill_varlen.
 */
gdp_status gdp_prefill_varlen_profiled(const gdp_prefill_args *args, void *stream, void *const *events,
                                       int num_events);

/*
 * Sequence-sharded prefill by state passing (blog post "Attention Cache and
 * Sequence Parallelism", section on passing state instead of KV): when the
 * tokens of a sequence are split over ranks, the state the previous ranks
 * leave is the next rank's initial state.  Over a shard the state map is
 * affine, S_end = S_0 Phi + B (the decay and the delta-rule updates of the
 * FlashInfer page's display equation, right-multiplying the V-major state),
 * so every rank finds its (B, Phi) at once, the pairs are exchanged, and each
 * rank chains those of the ranks before it into its initial state.
 *
 * gdp_prefill_transfer: for every sequence i and head h of args (the shard,
 * packed as for gdp_prefill_varlen), pairs[0][i][h] = B (the state after the
 * sequence from a zero state) and pairs[1][i][h] = Phi (the state after it
 * from the identity with v = 0), each [V][K] fp32: the final state from any
 * S_0 is S_0 Phi + B.  pairs: [2][N][H][V][K] fp32 device memory, 16-byte
 * aligned, written whole (B = 0, Phi = I for an empty sequence).  Needs
 * q, k, v, g, beta, cu_seqlens, the workspace and the scalars of args;
 * output, output_state, chunk_states, initial_state and the state cache are
 * not used (they are checked as for gdp_prefill_varlen when given).  Runs
 * whole sequences in one segment (no split chains).  N = 0 returns GDP_OK
 * without a launch.  Errors as gdp_prefill_varlen.
 *
 * gdp_chain_states: S_{j+1} = S_j Phi_j + B_j for j < steps, per (sequence,
 * head), from S_0 = s0 (NULL: zero).  phi, b: [steps][N][H][d][d] fp32 (the
 * pairs of consecutive shards in order), s_out: [steps + 1][N][H][d][d] fp32,
 * s_out[0] = S_0; d is 64 or 128; all device pointers, 16-byte aligned;
 * s_out must not overlap the inputs (GDP_ERR_ALIAS).  The products run in
 * fp32 FMA.  A bounded wait that runs out sets GDP_DEV_ERR_TIMEOUT in
 * *device_status (may be NULL).
 */
gdp_status gdp_prefill_transfer(const gdp_prefill_args *args, float *pairs, void *stream);
gdp_status gdp_chain_states(const float *s0, const float *phi, const float *b, int64_t steps, int64_t N, int H,
                            int d, float *s_out, uint32_t *device_status, void *stream);

/*
 * gdp_arm_wait_expiry_test: a test of the failure path (no counterpart on the
 * pages).  Every spin-wait of the kernels is bounded: a wait that does not
 * complete within its limit (about a second) sets GDP_DEV_ERR_TIMEOUT in
 * *device_status, drains the CTA's own tensor-core work and copies, frees its
 * tensor memory and returns, so the CUDA context stays usable and the host
 * reads the status after the stream completes.  This call arms the calling
 * host thread's NEXT gdp_prefill_varlen* call to exercise that path: the waits
 * of its scan (or fused) kernel give up after limit_ns (1e5 .. 1e9 ns), and that
 * kernel's CTA of sequence 0, head 0 withholds its first copy, so one of its
 * waits runs out.
 * That call's outputs are undefined (those of sequence 0, head 0 at least) and
 * its status word gets GDP_DEV_ERR_TIMEOUT; later calls are unaffected.  No
 * fault, trap or endless loop is involved.  GDP_ERR_INVALID_ARG for a limit
 * outside the range.
 */
gdp_status gdp_arm_wait_expiry_test(uint64_t limit_ns);

/*
 * Debug-bounds builds (libgdp_gb300_debug.so, compiled with -DGDP_DEBUG_BOUNDS=1;
 * no counterpart on the pages).  Every global index that the kernels derive
 * from the descriptors, the sequence table or the state-cache indices is
 * range-checked before its access: a failing check skips the access, ORs
 * GDP_DEV_ERR_BOUNDS into *device_status and records the first violation in a
 * device record of the library (one per CUDA context).  Nothing traps.  The
 * other builds carry no checks and return GDP_ERR_UNSUPPORTED from these calls.
 *
 * gdp_debug_bounds_record: after the calls of interest have completed, copies
 * the record into out[4] = {violations since the last read, site of the first
 * (a GDP_BOUNDS_SITE_* value), its index, its bound} and clears it.
 * Synchronous (waits for the device).
 */
#define GDP_BOUNDS_SITE_DESC 1        /* descriptor kernel: descriptor rows, offsets, order */
#define GDP_BOUNDS_SITE_WY_TILE 2     /* WY kernel: its tile's descriptor entry and workspace row */
#define GDP_BOUNDS_SITE_WY_SCALARS 3  /* WY kernel: the beta / g entries of its rows */
#define GDP_BOUNDS_SITE_SCAN_ORDER 4  /* scan kernel: the longest-first order entry */
#define GDP_BOUNDS_SITE_SCAN_TILE 5   /* scan kernel: workspace row of an image / U^T copy */
#define GDP_BOUNDS_SITE_SCAN_STATE 6  /* scan kernel: entering, chunk-state and final-state rows */
#define GDP_BOUNDS_SITE_SCAN_OUT 7    /* scan kernel: output token rows */
#define GDP_BOUNDS_SITE_DECODE 8      /* decode kernel: sequence row and cache slot */
gdp_status gdp_debug_bounds_record(int64_t out[4]);
/*
 * gdp_arm_bounds_test: a test of the debug-bounds path.  Arms the calling host
 * thread's NEXT gdp_prefill_varlen* call to check its output token rows against
 * T - 1 instead of T, so that the (valid) stores of the last token's output fail
 * their check: they are skipped and recorded (GDP_BOUNDS_SITE_SCAN_OUT), nothing
 * outside the caller's buffers is touched.  Debug-bounds builds only.
 */
gdp_status gdp_arm_bounds_test(void);

/*
 * gdp_prefill_varlen_static_scratch: the same prefill for callers that cannot
 * allocate device memory.  No counterpart on the pages: it exists because the
 * main entry point needs a caller-owned workspace, and some callers cannot
 * provide one -- a plugin inside another runtime that owns all device memory
 * through its own pool, or a host program without a caching allocator that may
 * not call cudaMalloc in its serving loop (cudaMalloc can synchronise the device).
 *
 * Arguments are those of gdp_prefill_varlen, except that args->workspace and
 * args->workspace_bytes are ignored: the scratch is a GDP_STATIC_SCRATCH_BYTES
 * (64 MiB) array inside the library, held by every GPU that loads the library
 * until the process exits.  A shape whose gdp_prefill_workspace_bytes exceeds
 * it is rejected with GDP_ERR_WORKSPACE before any launch.  Nothing is
 * allocated.  Each CUDA context holds its own copy of the array: the first call
 * made in a context (with it current) looks the array's device address up
 * (cudaGetSymbolAddress) and caches it under the context's unique ID, so a
 * context created later -- another runtime's own context, or the primary
 * context that replaces one destroyed by cudaDeviceReset -- gets its own lookup.
 * Make the first call in each context outside any stream capture.  All calls
 * share the array, so calls whose kernels overlap on the GPU (other streams,
 * other threads) race: serialise them.  Nothing in the array needs to start at
 * zero.  gdp_static_scratch_bytes() returns the array's size.
 */
#define GDP_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
gdp_status gdp_prefill_varlen_static_scratch(const gdp_prefill_args *args, void *stream);
size_t gdp_static_scratch_bytes(void);

/*
 * Build the varlen descriptors on the device (Megatron page, parameters
 * chunk_indices, chunk_indices_dp, chunk_offsets; capture note in the closing
 * paragraph).  cu_seqlens [N+1] int32/int64 device; outputs as described in
 * gdp_prefill_args; chunk_offsets_dp (optional, [N+1]) receives the prefix
 * sum of ceil(L_i M / 64).  Grid sizes depend on N, nt_pad, ntdp_pad only.
 */
gdp_status gdp_build_descriptors(const void *cu_seqlens, int cu_seqlens_int64, int64_t T, int64_t N,
                                 int num_householder, int32_t *chunk_indices, int64_t nt_pad,
                                 int32_t *chunk_indices_dp, int64_t ntdp_pad, int32_t *chunk_offsets,
                                 int32_t *chunk_offsets_dp, uint32_t *device_status, void *stream);

/*
 * gdp_decode_step: one token per sequence -- the serving step after prefill
 * (Attention-Cache-and-Sequence-Parallelism page, section "Prefill and decode"
 * and the GDN section: decode keeps only the state and advances it token by token
 * with the recurrent form; Megatron page, parameters state / state_indices).
 * For token i of sequence i (i < N) and every head: S *= exp(g_i); for j < M:
 * v_new = beta (v - S k_j), S += v_new (x) k_j; o_i = scale S q_i.
 *
 * Arguments: a gdp_prefill_args with T == N (token i belongs to sequence i; k, v
 * and beta have N*M rows).  cu_seqlens, the descriptor fields, nt_pad/ntdp_pad and
 * the workspace are ignored; chunk_states must be NULL.  State modes as for the
 * prefill: the cache `state` is read and written in place at state_indices[i] (-1:
 * start from zero, write nothing); otherwise initial_state[i] (or zero) is read and
 * output_state[i] written, and output_state may equal initial_state exactly (an
 * in-place update, fp32 initial state only) but not partly overlap it
 * (GDP_ERR_ALIAS).  The input-variant fields (types, alpha gate, head counts)
 * apply as for the prefill; with g_is_alpha the state is multiplied by
 * max(alpha, exp(-80)) directly.  K = V in {64, 128}, 1 <= M <= 16
 * (GDP_ERR_UNSUPPORTED otherwise).  No workspace; graph-capturable.
 */
gdp_status gdp_decode_step(const gdp_prefill_args *args, void *stream);

/*
 * gdp_prefill_varlen_backward: the backward pass of the prefill, for training.
 *
 * The pages print the forward recurrence only (FlashInfer page, display equation);
 * the blog post "Attention Cache and Sequence Parallelism" (section on passing state
 * instead of KV) notes that training runs it in chunks and that the backward
 * dependence runs the other way round.  This entry point returns the exact derivative
 * of that recurrence: for a loss L with dL/do = d_output and dL/dS_final =
 * d_final_state, the gradients of L with respect to q, k, v, g, beta and the initial
 * state.  It recomputes the forward pass from the inputs (nothing from a forward call
 * is kept), then runs the state scan backwards over 64-row chunks.
 *
 *   fwd            the forward call's arguments: q, k, v, g, beta, cu_seqlens, the
 *                  shapes, scale, use_qk_l2norm, initial_state (as for
 *                  gdp_prefill_varlen).  Its output, output_state, chunk_states,
 *                  descriptor, workspace and device_status fields are ignored.
 *                  Served: bf16 q/k/v with one-to-one heads, fp32 natural-log g (or
 *                  NULL), fp32 beta (or NULL), dense state mode (initial_state or
 *                  NULL; no state cache), K = V in {64, 128}; anything else is
 *                  GDP_ERR_UNSUPPORTED.
 *   d_output       [T, H, V] bf16, contiguous: dL/do.
 *   d_final_state  [N, H, V, K] fp32 or NULL (= 0): dL/dS_final.
 *   dq             [T, H, K] fp32, contiguous, written (with use_qk_l2norm: the
 *                  gradient with respect to the unnormalised rows).
 *   dk             [T*M, H, K] fp32, likewise.
 *   dv             [T*M, H, V] fp32, written.
 *   dg             [T, H] fp32 or NULL; all zeros when fwd->g is NULL.
 *   dbeta          [T*M, H] fp32 or NULL (the gradient at beta = 1 when fwd->beta is NULL).
 *   d_initial_state [N, H, V, K] fp32 or NULL: dL/dS_initial.
 *   workspace      at least gdp_backward_workspace_bytes(...) bytes, 256-byte aligned,
 *                  contents undefined on entry and exit.
 *   device_status  optional, as for the prefill.
 * Every buffer is a device pointer, 16-byte aligned.  Nothing is allocated and
 * nothing synchronises; a call can be captured in a CUDA graph.  Results do not
 * depend on scheduling: every sum runs in a fixed order.
 */
typedef struct gdp_backward_args {
  const gdp_prefill_args *fwd; /* host pointer, read during the call only */
  const void *d_output;
  const float *d_final_state;
  float *dq, *dk, *dv, *dg, *dbeta, *d_initial_state;
  void *workspace;
  size_t workspace_bytes;
  uint32_t *device_status;
} gdp_backward_args;

/* Workspace bytes of gdp_prefill_varlen_backward for this shape (0 for an invalid shape). */
size_t gdp_backward_workspace_bytes(int64_t T, int64_t N, int H, int K, int V, int num_householder);

gdp_status gdp_prefill_varlen_backward(const gdp_backward_args *args, void *stream);

/* One-line reason for the last non-OK status returned on this thread ("" if none). */
const char *gdp_last_error(void);

/* GDP_ABI_VERSION of the loaded library. */
int gdp_abi_version(void);

/* sizeof(gdp_prefill_args) as compiled into the library (lets a binding check its struct layout). */
size_t gdp_prefill_args_size(void);

#ifdef __cplusplus
}
#endif
#endif /* GDP_PREFILL_H */
