// gdp_internal.cuh -- shared definitions of the CUDA library (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdp_prefill.h"

namespace gdp {

constexpr int kChunk = GDP_CHUNK;       // rows per chunk on both streams
constexpr float kL2Eps = 1e-6f;         // L2-norm epsilon: x / sqrt(sum x^2 + eps)
constexpr float kLog2e = 1.4426950408889634f;

// Number of readout rows (rows t*M + M-1) a 64-row expanded chunk can hold,
// rounded up to the MMA N granularity of 16.
__host__ __device__ inline int qpad_for(int M) {
  int q = (kChunk + M - 1) / M;
  return (q + 15) / 16 * 16;
}

// Per-chunk decay rescaling of the scan.  The scan keeps S_hat = S / Gamma in
// tensor memory, where Gamma is a running product of chunk decays, so that the
// per-chunk factor gamma_last never has to be applied to the state on the
// serial chain.  A chunk whose decay is at least 2^kFastMinLog2Gamma has its -W
// and Qh operands written pre-divided by gamma_last ("fast" image); a chunk with
// a smaller decay (including 0) keeps them unscaled and the scan applies its
// decay to S explicitly.  The scan renormalises S_hat (Gamma -> 1) before Gamma
// would drop below kRenormMinGamma.
constexpr float kFastMinLog2Gamma = -20.f;
constexpr float kRenormMinGamma = 0x1p-40f;

// Per-(expanded chunk, head) operand image written by the WY kernel and copied
// into shared memory by the scan kernel in two bulk copies (part 1: b1 + meta,
// part 2: b2).  Every sub-tile is fp32, K-major with the 128-byte swizzle
// (gdp_sm100.cuh), 1024-byte aligned.  The B operands that share an A operand
// are stacked so that one MMA serves both (c = 2^-G2_last for a fast image, else 1):
//   b1: d/32 K-blocks of [qpad + 64 rows][32]: rows 0..qpad-1  c Qh, Qh = scale 2^(G2_p) qhat
//                                              rows qpad..+63  -c W          (A = S)
//   meta: gamma_last, nq, p0, len, fast
//   b2: 2 K-blocks of [d + qpad rows][32]:      rows 0..d-1     Ktil^T = (2^(G2_last-G2_s) khat_s)^T
//                                              rows d..+qpad-1 P = masked decayed scores (A = V_new^T)
struct ImageLayout {
  uint32_t b1, b1_block, meta, part1, b2, b2_block, part2, bytes;
  __host__ __device__ ImageLayout(int d, int qpad) {
    b1 = 0;
    b1_block = (uint32_t)(qpad + 64) * 128u;
    meta = b1 + (uint32_t)(d / 32) * b1_block;
    part1 = meta + 64u;
    b2 = meta + 1024u;
    b2_block = (uint32_t)(d + qpad) * 128u;
    part2 = 2u * b2_block;
    bytes = b2 + part2;
  }
  // byte offsets of element (row, k) inside a region: K-block k/32, swizzled row
  __host__ __device__ uint32_t qh(int qi, int f) const { return b1 + (f >> 5) * b1_block + swz_off(qi, f); }
  __host__ __device__ uint32_t wn(int qpad, int s, int f) const {
    return b1 + (f >> 5) * b1_block + swz_off(qpad + s, f);
  }
  __host__ __device__ uint32_t kt(int f, int s) const { return b2 + (s >> 5) * b2_block + swz_off(f, s); }
  __host__ __device__ uint32_t pm(int d, int qi, int s) const { return b2 + (s >> 5) * b2_block + swz_off(d + qi, s); }
  __host__ __device__ static uint32_t swz_off(int r, int k) {  // fp32 element k (mod 32) of row r
    const uint32_t b = (uint32_t)(k & 31) * 4u;
    return ((uint32_t)r >> 3) * 1024u + ((uint32_t)r & 7u) * 128u + ((((b >> 4) ^ (uint32_t)r) & 7u) << 4) + (b & 15u);
  }
};
// The same operands laid out for the backward's reverse state scan, whose products read
// every block transposed (so that each B operand is K-major again): batch 1 (N = 64 chunk rows
// s) reads Ktil as [s][c] and P^T as [s][q]; batch 2 (N = d features c) reads (-W)^T as [c][s]
// and Qh^T as [c][q], with -W and Qh divided by gamma_last in a fast image as above.  fp32,
// 128-byte swizzle, 32-column K blocks; the chunk's ImageMeta follows batch 1's blocks.
struct BwdImageLayout {
  // tinv: T = (I + A)^-1 of the chunk, dense [64][64] fp32, after the two parts (read by the
  // per-chunk gradient kernel; the scan's copies stop before it)
  uint32_t kt, pt, meta, part1, b2, wt, wt_block, qt, part2, tinv, bytes;
  __host__ __device__ BwdImageLayout(int d, int qpad) {
    const uint32_t nqb = ((uint32_t)qpad + 31u) / 32u;  // K blocks of the readout dimension
    kt = 0;                                             // [d/32][64 rows][128 B]
    pt = kt + (uint32_t)(d / 32) * 8192u;               // [nqb][64 rows][128 B]
    meta = pt + nqb * 8192u;
    part1 = meta + 64u;
    b2 = (part1 + 1023u) & ~1023u;
    wt = b2;                                            // [2][d rows][128 B]
    wt_block = (uint32_t)d * 128u;
    qt = wt + 2u * wt_block;                            // [nqb][d rows][128 B]
    part2 = qt + nqb * wt_block - b2;
    tinv = b2 + part2;
    bytes = tinv + 64u * 64u * 4u;
  }
  __host__ __device__ uint32_t k_at(int s, int c) const { return kt + (c >> 5) * 8192u + ImageLayout::swz_off(s, c); }
  __host__ __device__ uint32_t p_at(int s, int q) const { return pt + (q >> 5) * 8192u + ImageLayout::swz_off(s, q); }
  __host__ __device__ uint32_t w_at(int c, int s) const { return wt + (s >> 5) * wt_block + ImageLayout::swz_off(c, s); }
  __host__ __device__ uint32_t q_at(int c, int q) const { return qt + (q >> 5) * wt_block + ImageLayout::swz_off(c, q); }
};
struct ImageMeta {
  float gamma_last;  // 2^(G2_last): decay of the whole chunk
  int nq;            // readout rows in the chunk
  int p0;            // local row of the first readout row
  int len;           // rows in the chunk (<= 64)
  int fast;          // -W and Qh are divided by gamma_last
};

// Everything a kernel needs about one call (passed by value).
// Element types of g, beta and the initial state (q, k, v and the output: bf16 or f16).
constexpr int kTypeF32 = 0, kTypeBF16 = 1, kTypeF16 = 2;
// An alpha gate is read as max(log(alpha), kMinLogAlpha): alpha <= 0 stays finite.
constexpr float kMinLogAlpha = -80.f;

struct Problem {
  const void *q, *k, *v;  // bf16, or f16 when f16 != 0
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh;
  const void *g, *beta;   // element types g_type, beta_type
  const void *cu;
  int cu64;
  int64_t T, N;
  int H, K, V, M;
  float scale;
  int l2norm;
  const void *init;  // fp32, or bf16 when init_bf16 != 0
  float *cache;
  const int32_t *slots;
  int64_t num_slots;
  void *out;  // same type as q, k, v
  float *out_state;
  float *chunk_states;
  const int32_t *ci, *cid, *co, *cod;
  int64_t nt_pad, ntdp_pad;
  int64_t ws_rows;   // expanded-chunk rows the workspace tiles cover (shape bound)
  // workspace tiles, indexed by (expanded chunk row r, head h): tile (r * H + h)
  unsigned char *img;  // operand images, img_stride bytes per tile (ImageLayout)
  size_t img_stride;
  // U^T = (T diag(beta) V)^T, V x 64 fp32 per tile, in 32-row groups: element (v, s) at
  // ((v / 32) * 16 + s / 4) * 128 + (v % 32) * 4 + s % 4, so that 32 threads reading rows
  // 32g .. 32g + 31 four columns at a time read 512 contiguous bytes
  float *U;
  uint32_t *status;
  int qpad;
  // Chunk segment of this launch: expanded chunks [seg_lo, seg_hi) of every sequence (the
  // whole sequence is [0, INT64_MAX)).  seg_rows > 0: the WY grid is N x seg_rows tiles
  // of the segment.  seg_state: [N][H][V][K] fp32 state carried from one segment to the next.
  int64_t seg_lo, seg_hi;
  int seg_rows;
  float *seg_state;
  // input variants: head counts of q, k, v (each divides H; state head h reads head
  // h / (H / Hx), computed as input_head(h, hmul_x)), element types, linear-space gate
  int Hq, Hk, Hv;
  uint64_t hmul_q, hmul_k, hmul_v;  // ceil(2^32 / (H / Hx))
  int f16;               // q, k, v and the output are float16 (else bfloat16)
  int g_type, beta_type;  // kType*
  int g_alpha;           // g holds alpha itself (else its natural log)
  int init_bf16;         // the dense initial state is bfloat16 (else fp32)
  // launch the WY and scan kernels with programmatic stream serialization: each may start while
  // its predecessor finishes and waits (griddepcontrol.wait) before reading that one's outputs
  int pdl;
  // scan: the two output tensor maps (boxes of 64 / M and ceil(64 / M) token rows) are encoded:
  // a chunk with that many readout rows leaves through one TMA store
  int out_tma;
  // chunk_states row spacing: the scan emits the state entering expanded chunk e when
  // e % cs_div == 0, at row co[seq] + e / cs_div (M: token-chunk starts; 1: every expanded
  // chunk, with co = the expanded-chunk offsets, for the backward pass).  A NULL `out` skips
  // the output stores.
  int cs_div;
  // Split chains (few long chains; 0: off): a sequence of n chunks runs as
  // max(1, ceil(n / piece_len)) pieces of piece_len expanded chunks, numbered sequence by
  // sequence (piece rows).  The state recurrence is affine in the state, S' = S Phi + B, so
  // a piece's entering state follows from its predecessors' (Phi, B) alone.  piece_pass1 = 1:
  // for every piece but a sequence's last, grid row r < piece_rows runs the piece from a zero
  // state (its B) and row piece_rows + r from the identity with V = 0 (its Phi), each leaving
  // its end state in piece_buf row (grid row); no outputs.  piece_pass1 = 0: piece r of a
  // split sequence enters with piece_buf row 2 piece_rows + r (the combine kernel's S_in)
  // and writes outputs, chunk states and, as its sequence's last piece, the final state.
  // piece_buf: [3 piece_rows][H][V][K] fp32.
  int piece_len, piece_rows, piece_pass1;
  float *piece_buf;
  // Transfer pair of every sequence (xfer = 1; no pieces, one segment): grid row i < N runs
  // sequence i from a zero state, row N + i from the identity with V = 0, each writing its end
  // state (B_i, Phi_i: S_end = S_0 Phi_i + B_i for any S_0) to xfer_out row (grid row); no
  // outputs.  xfer_out: [2][N][H][V][K] fp32.
  int xfer;
  float *xfer_out;
  // Limit of every bounded wait of the scan (kWaitLimitNs, about a second, unless a test of the
  // failure path shortened it) and that test's switch: CTA (0, 0) withholds the first image copy,
  // so that one of its waits runs out (gdp_arm_wait_expiry_test).
  uint64_t wait_limit_ns;
  int test_withhold_copy;
  // The fused kernel's CTA order (NULL: sequence by sequence): linear CTA index l runs sequence
  // order[l / H], head l % H, so the longest sequences start first (the descriptor kernel's order)
  const int32_t *order;
  // Debug-bounds builds: the library's violation record (see in_range) and the output-row bound
  // reduction of the bounds test (gdp_arm_bounds_test; 0 otherwise)
  unsigned long long *bounds;
  int64_t bounds_shrink;
  // The backward's forward recompute: the WY kernel also writes each tile's BwdImageLayout image
  // here, bimg_stride bytes apart (NULL otherwise)
  unsigned char *bimg;
  size_t bimg_stride;
};

// Everything the backward kernels need about one call (gdp_backward.cu).  Heads are
// one-to-one, q / k / v / d_output bf16, g natural-log fp32, beta fp32, K = V = D.
struct BwdProblem {
  const __nv_bfloat16 *q, *k, *v;
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh;
  const float *g, *beta;  // NULL: no decay / all ones
  const void *cu;
  int cu64;
  int64_t T, N;
  int H, D, M, qpad;
  float scale;
  int l2norm;
  const int32_t *cid, *cod;  // expanded-chunk descriptors and offsets (forward recompute)
  int64_t ntdp_pad, ws_rows;
  const unsigned char *img;  // the forward's operand images (ImageLayout), img_stride apart
  size_t img_stride;
  const unsigned char *bimg;  // the same operands for the reverse scan (BwdImageLayout), bimg_stride apart
  size_t bimg_stride;
  const float *Sx;           // [ntdp][H][V][K] state entering each expanded chunk
  float *Dx;                 // [ntdp][H][V][K] dL/dS at each expanded chunk's exit
  const __nv_bfloat16 *dout; // [T][H][V] dL/do
  const float *dfin;         // [N][H][V][K] dL/dS_final or NULL
  const float *fin;          // [N][H][V][K] recomputed final state (when dfin)
  float *dinit;              // [N][H][V][K] dL/dS_initial or NULL
  float *tot;                // [N][H] <dS_final, S_final>
  float *sig, *rho;          // [T*M][H] sum_v dv v, [T][H] do . o
  float *dq, *dk, *dv, *dg, *dbeta;
  uint32_t *status;
};
cudaError_t launch_backward(const BwdProblem &p, cudaStream_t stream);
// The reverse state scan on the tensor cores (gdp_bwd_scan_tc.cu) and the byte stride of the
// per-tile backward images (BwdImageLayout, with the inverse, rounded to 1 KB).
cudaError_t launch_bwd_tc_scan(const BwdProblem &p, cudaStream_t stream);
size_t bwd_image_stride(int d, int qpad);

// Launch `kern` on `stream`, with programmatic stream serialization when `pdl`.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                          Args &&...args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Input head h / r of state head h, with m = ceil(2^32 / r): (h m) >> 32 equals h / r for
// every h < 2^16 and r <= 2^16 (the rounding excess of m stays below 2^-16 <= 1 / r), and it
// takes one wide multiply instead of a division.
__device__ __forceinline__ int input_head(int h, uint64_t m) { return (int)(((uint64_t)h * m) >> 32); }
__host__ inline uint64_t head_mul(int ratio) { return ((1ull << 32) + (uint64_t)ratio - 1) / (uint64_t)ratio; }

// One element of a g / beta array of element type `type`, as fp32.
__device__ __forceinline__ float load_typed(const void *base, int64_t i, int type) {
  if (type == kTypeF32) return reinterpret_cast<const float *>(base)[i];
  const uint32_t u = reinterpret_cast<const uint16_t *>(base)[i];
  return type == kTypeBF16 ? __uint_as_float(u << 16) : __half2float(__ushort_as_half((unsigned short)u));
}
// The natural-log decay of token row i of g (alpha = exp of it).
__device__ __forceinline__ float load_log_gate(const Problem &p, int64_t i) {
  const float x = load_typed(p.g, i, p.g_type);
  return p.g_alpha ? fmaxf(logf(x), kMinLogAlpha) : x;  // fmaxf also maps NaN (alpha < 0) to the floor
}

// Long sequences over few (sequence, head) chains are processed in segments of
// kSegChunks expanded chunks, so that the WY tiles of segment k + 1 are built on the
// SMs the scan of segment k leaves free (stream-level overlap, no cross-kernel waits).
constexpr int64_t kSegChunks = 128;
constexpr int64_t kSegMaxChains = 64;
constexpr int kSegMax = 64;

__device__ __forceinline__ int64_t load_cu(const void *cu, int cu64, int64_t i) {
  return cu64 ? reinterpret_cast<const int64_t *>(cu)[i] : (int64_t) reinterpret_cast<const int32_t *>(cu)[i];
}

// Bounds of sequence i; false (and L = 0) unless 0 <= cu[i] <= cu[i+1] <= T.
__device__ __forceinline__ bool seq_bounds(const void *cu, int cu64, int64_t T, int64_t i, int64_t *bos, int64_t *L) {
  const int64_t b = load_cu(cu, cu64, i), e = load_cu(cu, cu64, i + 1);
  const bool ok = (b >= 0) && (b <= e) && (e <= T);
  *bos = ok ? b : 0;
  *L = ok ? e - b : 0;
  return ok;
}

// Split chains: the number of pieces of sequence i, from its chunks whose workspace tile
// exists; at least one, so that an empty sequence still passes its state through.
constexpr int kPieceMaxSeqs = 32;    // sequences a split call may hold (one warp finds a piece)
constexpr int kPieceCtas = 128;      // piece rows x heads of a split call
constexpr int kPieceMinChunks = 6;   // shortest piece (measured: 4 to 7 within 2 %, 6 best)
__device__ __forceinline__ int seq_pieces(const Problem &p, int64_t i) {
  int64_t bos, L;
  seq_bounds(p.cu, p.cu64, p.T, i, &bos, &L);
  const int64_t nch = (L * p.M + kChunk - 1) / kChunk, cod = p.cod[i];
  const int64_t nall = (cod < 0) ? 0 : max((int64_t)0, min(nch, p.ws_rows - cod));
  return (int)max((int64_t)1, (nall + p.piece_len - 1) / p.piece_len);
}
// Warp-wide (all 32 lanes, N <= kPieceMaxSeqs): lane i < N holds its sequence's piece count
// n and the inclusive prefix sum of the counts.
__device__ __forceinline__ void piece_prefix(const Problem &p, int lane, int *n, int *incl) {
  const int c = (lane < p.N) ? seq_pieces(p, lane) : 0;
  int x = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  *n = c;
  *incl = x;
}
// Warp-wide: the sequence holding piece row r, the piece's index in it and the sequence's
// piece count; seq = -1 past the last piece.
__device__ __forceinline__ void piece_of_row(const Problem &p, int r, int lane, int *seq, int *pi, int *np) {
  int n, incl;
  piece_prefix(p, lane, &n, &incl);
  // the counts are positive, so the sequences ending at or before r are a prefix
  const int s = __popc(__ballot_sync(0xffffffffu, lane < p.N && incl <= r));
  const int first = __shfl_sync(0xffffffffu, incl - n, s & 31), cnt = __shfl_sync(0xffffffffu, n, s & 31);
  *seq = (s < p.N) ? s : -1;
  *pi = r - first;
  *np = cnt;
}
// Warp-wide: sequence i's first piece row and piece count.
__device__ __forceinline__ void pieces_of_seq(const Problem &p, int i, int lane, int *first, int *np) {
  int n, incl;
  piece_prefix(p, lane, &n, &incl);
  *first = __shfl_sync(0xffffffffu, incl - n, i & 31);
  *np = __shfl_sync(0xffffffffu, n, i & 31);
}

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// Range check of a global index before its access (debug-bounds builds, -DGDP_DEBUG_BOUNDS=1):
// false when idx is outside [0, bound), after counting the violation in rec[0], recording the
// first one's site, index and bound in rec[1..3] and setting GDP_DEV_ERR_BOUNDS; the caller then
// skips the access.  Other builds: always true, no code.
#ifndef GDP_DEBUG_BOUNDS
#define GDP_DEBUG_BOUNDS 0
#endif
__device__ __forceinline__ bool in_range([[maybe_unused]] unsigned long long *rec, [[maybe_unused]] uint32_t *status,
                                         [[maybe_unused]] int site, [[maybe_unused]] int64_t idx,
                                         [[maybe_unused]] int64_t bound) {
#if GDP_DEBUG_BOUNDS
  if (idx >= 0 && idx < bound) return true;
  if (rec && atomicAdd(&rec[0], 1ull) == 0ull) {
    rec[1] = (unsigned long long)site;
    rec[2] = (unsigned long long)idx;
    rec[3] = (unsigned long long)bound;
  }
  set_status(status, GDP_DEV_ERR_BOUNDS);
  return false;
#else
  return true;
#endif
}

// Kernel launchers (defined in their .cu files).  Each returns a CUDA error.
// order (optional, [N]): the sequences longest first (by expanded chunks; ties in their own
// order) for batches of up to 1024 sequences, the identity beyond.
cudaError_t launch_descriptors(const void *cu, int cu64, int64_t T, int64_t N, int M, int32_t *ci, int64_t nt_pad,
                               int32_t *cid, int64_t ntdp_pad, int32_t *co, int32_t *cod, uint32_t *status,
                               cudaStream_t stream, int32_t *order = nullptr, unsigned long long *bounds = nullptr);
cudaError_t launch_wy(const Problem &p, cudaStream_t stream);
// The WY kernel for float16 inputs (f16) and / or 16-bit or linear-space gates (typed).
cudaError_t launch_wy_variant(const Problem &p, cudaStream_t stream, bool f16, bool typed);
cudaError_t launch_scan(const Problem &p, cudaStream_t stream);
// The scan for float16 inputs (f16) and / or a bfloat16 dense initial state (init16).
cudaError_t launch_scan_variant(const Problem &p, cudaStream_t stream, bool f16, bool init16);
// The fused prefill (gdp_fused.cu): WY work, scan, outputs and state scatter in one kernel, one
// CTA per (sequence, head), for the common contract (bf16 q / k / v, fp32 natural-log g and
// beta, fp32 states, K = V = 128, qpad <= 32); fused_serves says whether a call is served.
bool fused_serves(const Problem &p);
bool fused_shape(int K, int V, int M);
cudaError_t launch_fused(const Problem &p, cudaStream_t stream);
// Split chains: the entering state of every piece of a split sequence (gdp_pieces.cu).
cudaError_t launch_piece_combine(const Problem &p, cudaStream_t stream);
// S_{j+1} = S_j Phi_j + B_j for j < steps from S_0 (NULL: zero), Phi / B [steps][N][H][d][d],
// S_out [steps + 1][N][H][d][d] (S_out[0] = S_0) (gdp_pieces.cu).
cudaError_t launch_chain_states(const float *s0, const float *phi, const float *b, int64_t steps, int64_t N, int H,
                                int d, float *s_out, uint32_t *status, cudaStream_t stream);

// TMA tensor maps (gdp_tmap.cu; `map` points at a 64-byte aligned CUtensorMap; a NULL base
// leaves it zeroed).  All use the 128-byte swizzle.
//   tmap_state:     [rows][d] fp32, 32 x 32 boxes
//   tmap_rows_16:   [rows][H][K] bf16 (f16 = 0) or float16 (f16 = 1) with element strides
//                   (stride_t, stride_h), boxes of 64 features x 1 head x box_rows rows
cudaError_t tmap_state(void *map, float *base, int64_t rows, int d);
cudaError_t tmap_rows_16(void *map, const void *base, int64_t rows, int H, int K, int64_t stride_t, int64_t stride_h,
                         int box_rows, int f16);
//   tmap_out_rows:  the output [T][H][V] (bf16 or float16), unswizzled boxes of V features x
//                   1 head x box_rows tokens
cudaError_t tmap_out_rows(void *map, void *base, int64_t T, int H, int V, int box_rows, int f16);

// Sets the calling thread's gdp_last_error() text (defined in gdp_api.cu).
void set_last_error(const char *fmt, ...);
// Checks the input-variant fields of the arguments and fills p's Hq/Hk/Hv and type fields.
gdp_status resolve_variants(const gdp_prefill_args *a, Problem *p);
// The debug-bounds record of the current CUDA context (gdp_api.cu; NULL outside debug-bounds builds).
unsigned long long *bounds_record();

}  // namespace gdp
