// gdp_api.cu -- host side of the C ABI: argument checks, workspace carving,
// kernel launches on the caller's stream.  Nothing here allocates, syncs or
// reads device memory, so a call can be captured in a CUDA graph (Megatron-Core
// API page "core.ssm.ops.gdp.chunk", closing paragraph).
#include <math.h>
#include <stdint.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "gdp_internal.cuh"

#define GDP_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

thread_local char g_last_error[512] = "";
// gdp_arm_wait_expiry_test: the wait limit (ns) of the calling thread's next prefill, 0 = not armed
thread_local uint64_t g_expiry_test_ns = 0;
// gdp_arm_bounds_test: the calling thread's next prefill checks its output rows against T - 1
thread_local bool g_bounds_test = false;

gdp_status fail(gdp_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int64_t nt_bound(int64_t T, int64_t N) { return (T + (int64_t)(gdp::kChunk - 1) * N) / gdp::kChunk; }
int64_t ntdp_bound(int64_t T, int64_t N, int M) {
  return ((int64_t)M * T + (int64_t)(gdp::kChunk - 1) * N) / gdp::kChunk;
}

// Number of chunk segments the call runs in (shape-only, see gdp::kSegChunks): more than
// one only for few (sequence, head) chains and long sequences.
int seg_count(int64_t T, int64_t N, int H, int M) {
  if (N * (int64_t)H > gdp::kSegMaxChains) return 1;
  const int64_t maxc = ((int64_t)M * T + gdp::kChunk - 1) / gdp::kChunk;  // chunks of the longest sequence
  if (maxc < 3 * gdp::kSegChunks) return 1;
  return (int)min((maxc + gdp::kSegChunks - 1) / gdp::kSegChunks, (int64_t)gdp::kSegMax);
}

// Split chains (shape-only, see gdp::Problem::piece_len): in a one-segment call over few
// sequences, the shortest piece length (at least kPieceMinChunks expanded chunks) whose
// piece-row bound N + ceil(C / len) (C: the expanded-chunk bound; a sequence of n chunks has
// max(1, ceil(n / len)) pieces) times H stays within kPieceCtas; off (len 0) when no piece
// would be shorter than the longest possible sequence.
struct PiecePlan {
  int64_t len, rows;
};
PiecePlan piece_plan(int64_t T, int64_t N, int H, int M) {
  PiecePlan pl{0, 0};
  if (N < 1 || N > gdp::kPieceMaxSeqs || seg_count(T, N, H, M) != 1) return pl;
  const int64_t C = ntdp_bound(T, N, M), maxc = ((int64_t)M * T + gdp::kChunk - 1) / gdp::kChunk;
  for (int64_t len = gdp::kPieceMinChunks; len < maxc; ++len) {
    const int64_t rows = N + (C + len - 1) / len;
    if (rows * H <= gdp::kPieceCtas) {
      pl.len = len;
      pl.rows = rows;
      break;
    }
  }
  return pl;
}

// The split-chains plan of the fused kernel (gdp_fused.cu): as piece_plan, but a fused call runs
// whole sequences in one launch whatever their length, so long chains split as well.
PiecePlan fused_piece_plan(int64_t T, int64_t N, int H, int M) {
  PiecePlan pl{0, 0};
  if (N < 1 || N > gdp::kPieceMaxSeqs) return pl;
  const int64_t C = ntdp_bound(T, N, M), maxc = ((int64_t)M * T + gdp::kChunk - 1) / gdp::kChunk;
  for (int64_t len = gdp::kPieceMinChunks; len < maxc; ++len) {
    const int64_t rows = N + (C + len - 1) / len;
    if (rows * H <= gdp::kPieceCtas) {
      pl.len = len;
      pl.rows = rows;
      break;
    }
  }
  return pl;
}

// Workspace layout; identical for the size query and the carving.
struct Layout {
  size_t cod, ci, cid, co, ord, img, img_stride, U, seg, piece, total;
};

Layout layout_for(int64_t T, int64_t N, int H, int K, int V, int M) {
  Layout l{};
  const int64_t ntp = nt_bound(T, N), ntdp = ntdp_bound(T, N, M);
  const int qp = gdp::qpad_for(M);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  l.cod = take(sizeof(int32_t) * (size_t)(N + 1));
  l.ci = take(sizeof(int32_t) * 2 * (size_t)ntp);
  l.cid = take(sizeof(int32_t) * 2 * (size_t)ntdp);
  l.co = take(sizeof(int32_t) * (size_t)(N + 1));
  l.ord = take(sizeof(int32_t) * (size_t)(N + 1));
  const size_t tiles = (size_t)ntdp * (size_t)H;
  l.img_stride = align_up(gdp::ImageLayout(K, qp).bytes);
  l.img = take(l.img_stride * tiles);
  l.U = take(sizeof(float) * tiles * gdp::kChunk * (size_t)V);
  l.seg = seg_count(T, N, H, M) > 1 ? take(sizeof(float) * (size_t)N * H * (size_t)V * K) : 0;
  // the pieces of either plan (a call over another input type on a fused shape runs the staged one)
  const PiecePlan pp = piece_plan(T, N, H, M);
  const PiecePlan pf = gdp::fused_shape(K, V, M) ? fused_piece_plan(T, N, H, M) : PiecePlan{0, 0};
  const int64_t prow = pp.rows > pf.rows ? pp.rows : pf.rows;
  l.piece = prow > 0 ? take(sizeof(float) * 3 * (size_t)prow * H * (size_t)V * K) : 0;
  l.total = off;
  return l;
}

bool shape_ok(int64_t T, int64_t N, int H, int K, int V, int M) {
  return T >= 0 && N >= 0 && H >= 1 && K >= 1 && V >= 1 && M >= 1 && M <= 64 &&
         T <= (int64_t)INT32_MAX / (M > 0 ? M : 1) && N < (int64_t)INT32_MAX;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

// Internal streams of the segmented mode, per host thread and device: WY tiles on a
// low-priority stream, scan segments on a high-priority one, joined to the caller's stream
// with events (so a call still captures into one CUDA graph).
struct SideStreams {
  bool ok = false;
  cudaStream_t wy = nullptr, scan = nullptr;
  cudaEvent_t ev[gdp::kSegMax + 2] = {};
};
SideStreams *side_streams() {
  constexpr int kMaxDev = 16;
  thread_local SideStreams cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  SideStreams &s = cache[dev];
  if (s.ok) return &s;
  int least = 0, greatest = 0;
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
  if (cudaStreamCreateWithPriority(&s.wy, cudaStreamNonBlocking, least) != cudaSuccess) return nullptr;
  if (cudaStreamCreateWithPriority(&s.scan, cudaStreamNonBlocking, greatest) != cudaSuccess) return nullptr;
  for (auto &e : s.ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
  s.ok = true;
  return &s;
}

gdp_status record(cudaEvent_t ev, cudaStream_t stream) {
  if (!ev) return GDP_OK;
  cudaError_t e = cudaEventRecord(ev, stream);
  return e == cudaSuccess ? GDP_OK : fail(GDP_ERR_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e));
}

}  // namespace

#if GDP_DEBUG_BOUNDS
// The debug-bounds record of the kernels' range checks (count, first site, index, bound); the
// runtime keeps one copy per CUDA context
__device__ unsigned long long g_bounds_rec[4];
#endif
// The record's device address in the current context (NULL in other builds or on failure)
unsigned long long *gdp::bounds_record() {
#if GDP_DEBUG_BOUNDS
  void *ptr = nullptr;
  return cudaGetSymbolAddress(&ptr, g_bounds_rec) == cudaSuccess ? static_cast<unsigned long long *>(ptr) : nullptr;
#else
  return nullptr;
#endif
}

// The input-variant tail of gdp_prefill_args (FlashInfer page, parameters q, k, v, g,
// beta, initial_state): checks it and fills the matching Problem fields.
gdp_status gdp::resolve_variants(const gdp_prefill_args *a, Problem *p) {
  const int H = a->H;
  const int hq = a->num_q_heads ? a->num_q_heads : H, hk = a->num_k_heads ? a->num_k_heads : H,
            hv = a->num_v_heads ? a->num_v_heads : H;
  if (hq < 1 || hk < 1 || hv < 1 || H % hq || H % hk || H % hv || H != (hq > hv ? hq : hv) || (hk != hq && hk != hv))
    return fail(GDP_ERR_INVALID_ARG,
                "head counts q=%d k=%d v=%d: each must divide H=%d, H must equal max(q, v), k must equal q or v",
                hq, hk, hv, H);
  if (H > 65535) return fail(GDP_ERR_UNSUPPORTED, "H=%d above the 65535 heads one launch grid holds", H);
  p->Hq = hq;
  p->Hk = hk;
  p->Hv = hv;
  p->hmul_q = head_mul(H / hq);
  p->hmul_k = head_mul(H / hk);
  p->hmul_v = head_mul(H / hv);
  const int qt = a->qkv_dtype ? a->qkv_dtype : GDP_DTYPE_BF16;
  if (qt != GDP_DTYPE_BF16 && qt != GDP_DTYPE_F16)
    return fail(GDP_ERR_UNSUPPORTED, "qkv_dtype %d: q, k, v are bfloat16 or float16", a->qkv_dtype);
  p->f16 = qt == GDP_DTYPE_F16;
  auto type_of = [](int dt) { return dt == GDP_DTYPE_BF16 ? kTypeBF16 : dt == GDP_DTYPE_F16 ? kTypeF16 : kTypeF32; };
  const int gt = a->g_dtype ? a->g_dtype : GDP_DTYPE_F32;
  if (gt != GDP_DTYPE_F32 && gt != GDP_DTYPE_BF16 && gt != GDP_DTYPE_F16)
    return fail(GDP_ERR_UNSUPPORTED, "g_dtype %d: g is float32, bfloat16 or float16", a->g_dtype);
  p->g_type = type_of(gt);
  const int bt = a->beta_dtype ? a->beta_dtype : GDP_DTYPE_F32;
  if (bt != GDP_DTYPE_F32 && bt != qt)
    return fail(GDP_ERR_UNSUPPORTED, "beta_dtype %d: beta is float32 or the q/k/v type", a->beta_dtype);
  p->beta_type = type_of(bt);
  if (a->g_is_alpha != 0 && a->g_is_alpha != 1) return fail(GDP_ERR_INVALID_ARG, "g_is_alpha must be 0 or 1");
  p->g_alpha = a->g_is_alpha;
  const int st = a->initial_state_dtype ? a->initial_state_dtype : GDP_DTYPE_F32;
  if (st != GDP_DTYPE_F32 && st != GDP_DTYPE_BF16)
    return fail(GDP_ERR_UNSUPPORTED, "initial_state_dtype %d: the initial state is float32 or bfloat16",
                a->initial_state_dtype);
  p->init_bf16 = st == GDP_DTYPE_BF16;
  return GDP_OK;
}

namespace {

// The forward recompute of the backward pass: the scan writes the state entering EVERY
// expanded chunk to `states` (row chunk_offsets_dp[i] + e), the final state to `final_state`
// (or nothing when NULL) and no output; args->output, output_state and chunk_states are ignored.
struct Recompute {
  float *states;
  float *final_state;
  unsigned char *bimg;  // the WY tiles' operands in the reverse scan's layout (BwdImageLayout)
  size_t bimg_stride;
};

// Checks + launches shared by gdp_prefill_varlen, its profiled form, the backward pass and the
// transfer pairs (xfer_out != NULL: B and Phi of every sequence into xfer_out, [2][N][H][V][K];
// output, output_state, chunk_states, initial_state and the state cache are ignored).
gdp_status prefill(const gdp_prefill_args *a, cudaStream_t stream, cudaEvent_t const *ev,
                   const Recompute *rc = nullptr, float *xfer_out = nullptr, bool want_fused = false) {
  g_last_error[0] = 0;
  if (!a) return fail(GDP_ERR_INVALID_ARG, "args is NULL");
  const int64_t T = a->T, N = a->N;
  const int H = a->H, K = a->K, V = a->V, M = a->num_householder;
  if (!shape_ok(T, N, H, K, V, M))
    return fail(GDP_ERR_INVALID_ARG, "bad shape T=%lld N=%lld H=%d K=%d V=%d M=%d", (long long)T, (long long)N, H, K,
                V, M);
  if (K != V || (K != 64 && K != 128))
    return fail(GDP_ERR_UNSUPPORTED, "head sizes K=%d V=%d: this build serves K == V in {64, 128}", K, V);
  if (!a->cu_seqlens && N > 0) return fail(GDP_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if (T > 0 && (!a->q || !a->k || !a->v || (!a->output && !rc && !xfer_out)))
    return fail(GDP_ERR_INVALID_ARG, "q, k, v and output are required");
  gdp::Problem p{};
  gdp_status vst = gdp::resolve_variants(a, &p);
  if (vst != GDP_OK) return vst;
  const int64_t strides[6] = {a->q_stride_t, a->q_stride_h, a->k_stride_t, a->k_stride_h, a->v_stride_t, a->v_stride_h};
  for (int i = 0; i < 6; ++i)
    if (T > 0 && (strides[i] <= 0 || strides[i] % 8 != 0))
      return fail(GDP_ERR_INVALID_ARG, "strides must be positive multiples of 8 elements (16 bytes)");
  if (T > 0 && (a->q_stride_h < K || a->k_stride_h < K || a->v_stride_h < V || a->q_stride_t < (int64_t)p.Hq * K ||
                a->k_stride_t < (int64_t)p.Hk * K || a->v_stride_t < (int64_t)p.Hv * V))
    return fail(GDP_ERR_INVALID_ARG, "strides describe overlapping rows");
  const uintptr_t align16 = ((uintptr_t)a->q | (uintptr_t)a->k | (uintptr_t)a->v | (uintptr_t)a->output) & 15u;
  if (align16) return fail(GDP_ERR_INVALID_ARG, "q, k, v and output must be 16-byte aligned");
  const uintptr_t salign = ((uintptr_t)a->initial_state | (uintptr_t)a->state | (uintptr_t)a->output_state |
                            (uintptr_t)a->chunk_states) & 15u;
  if (salign) return fail(GDP_ERR_INVALID_ARG, "state buffers must be 16-byte aligned");
  if (a->state && a->initial_state)
    return fail(GDP_ERR_INVALID_ARG, "state (cache mode) and initial_state are mutually exclusive");
  if (a->state && (!a->state_indices || a->num_slots < 1))
    return fail(GDP_ERR_INVALID_ARG, "state cache needs state_indices and num_slots >= 1");
  if (a->state && a->output_state)
    return fail(GDP_ERR_INVALID_ARG, "in cache mode the final state is written to the cache; output_state must be NULL");
  const size_t state_bytes = sizeof(float) * (size_t)N * H * (size_t)V * K;
  if (overlaps(a->output_state, state_bytes, a->initial_state, p.init_bf16 ? state_bytes / 2 : state_bytes))
    return fail(GDP_ERR_ALIAS, "output_state must not alias initial_state");
  const int nprebuilt = (a->chunk_indices != nullptr) + (a->chunk_indices_dp != nullptr) + (a->chunk_offsets != nullptr);
  if (nprebuilt != 0 && nprebuilt != 3)
    return fail(GDP_ERR_INVALID_ARG, "pass all three prebuilt descriptors or none");
  const int64_t ntb = nt_bound(T, N), ntdpb = ntdp_bound(T, N, M);
  const int64_t nt_pad = a->nt_pad ? a->nt_pad : ntb, ntdp_pad = a->ntdp_pad ? a->ntdp_pad : ntdpb;
  if (nt_pad < ntb || ntdp_pad < ntdpb)
    return fail(GDP_ERR_INVALID_ARG, "nt_pad/ntdp_pad (%lld/%lld) below the shape bounds (%lld/%lld)",
                (long long)nt_pad, (long long)ntdp_pad, (long long)ntb, (long long)ntdpb);
  if (nprebuilt == 0 && (nt_pad != ntb || ntdp_pad != ntdpb))
    return fail(GDP_ERR_INVALID_ARG, "nt_pad/ntdp_pad other than the bounds need prebuilt descriptors");
  const int64_t hv = (int64_t)H * V;
  if (nt_pad * hv > INT32_MAX || N * hv > INT32_MAX || (a->state && a->num_slots * hv > INT32_MAX))
    return fail(GDP_ERR_UNSUPPORTED, "state arrays above 2^31 rows of K floats");
  const Layout lay = layout_for(T, N, H, K, V, M);
  if (!a->workspace || ((uintptr_t)a->workspace % kAlign) != 0)
    return fail(GDP_ERR_WORKSPACE, "workspace must be non-NULL and %zu-byte aligned", kAlign);
  if (a->workspace_bytes < lay.total)
    return fail(GDP_ERR_WORKSPACE, "workspace of %zu bytes < required %zu", a->workspace_bytes, lay.total);

  gdp_status st;
  if (ev && (st = record(ev[0], stream)) != GDP_OK) return st;
  if (N == 0) {
    for (int i = 1; ev && i < 4; ++i)
      if ((st = record(ev[i], stream)) != GDP_OK) return st;
    return GDP_OK;
  }

  char *ws = (char *)a->workspace;
  p.q = a->q;
  p.k = a->k;
  p.v = a->v;
  p.q_st = a->q_stride_t; p.q_sh = a->q_stride_h;
  p.k_st = a->k_stride_t; p.k_sh = a->k_stride_h;
  p.v_st = a->v_stride_t; p.v_sh = a->v_stride_h;
  p.g = a->g;
  p.beta = a->beta;
  p.cu = a->cu_seqlens;
  p.cu64 = a->cu_seqlens_int64 ? 1 : 0;
  p.T = T; p.N = N; p.H = H; p.K = K; p.V = V; p.M = M;
  p.scale = (a->scale > 0.f && !isnan(a->scale)) ? a->scale : 1.0f / sqrtf((float)K);
  p.l2norm = a->use_qk_l2norm ? 1 : 0;
  p.init = a->initial_state;
  p.cache = a->state;
  p.slots = a->state_indices;
  p.num_slots = a->num_slots;
  p.out = a->output;
  p.out_state = a->output_state;
  p.chunk_states = a->chunk_states;
  p.nt_pad = nt_pad;
  p.ntdp_pad = ntdp_pad;
  p.ws_rows = ntdpb;
  p.cod = (int32_t *)(ws + lay.cod);
  if (nprebuilt == 3) {
    p.ci = a->chunk_indices;
    p.cid = a->chunk_indices_dp;
    p.co = a->chunk_offsets;
  } else {
    p.ci = (int32_t *)(ws + lay.ci);
    p.cid = (int32_t *)(ws + lay.cid);
    p.co = (int32_t *)(ws + lay.co);
  }
  p.img = (unsigned char *)(ws + lay.img);
  p.img_stride = lay.img_stride;
  p.U = (float *)(ws + lay.U);
  p.status = a->device_status;
  p.qpad = gdp::qpad_for(M);
  p.cs_div = M;
  int32_t *const co_desc = (int32_t *)p.co;  // where the descriptor kernel writes chunk_offsets
  if (rc) {  // backward recompute: a state row per expanded chunk, no outputs
    p.out = nullptr;
    p.out_state = rc->final_state;
    p.chunk_states = rc->states;
    p.co = p.cod;
    p.nt_pad = ntdp_pad;
    p.cs_div = 1;
    p.bimg = rc->bimg;
    p.bimg_stride = rc->bimg_stride;
  }
  p.seg_lo = 0;
  p.seg_hi = INT64_MAX;
  p.seg_rows = 0;
  p.seg_state = nullptr;
  // the fused kernel (WY work, scan and outputs in one launch; gdp_prefill_varlen_fused) serves
  // the common contract of a plain forward call
  if (want_fused && (rc || xfer_out || !gdp::fused_serves(p)))
    return fail(GDP_ERR_UNSUPPORTED,
                "the fused kernel serves bf16 q/k/v, fp32 natural-log g and beta, fp32 states, K = V = 128, M >= 2");
  const bool fused = want_fused;
  // a transfer-pair call runs whole sequences in one segment
  const int nseg = xfer_out ? 1 : seg_count(T, N, H, M);
  const PiecePlan pp = xfer_out ? PiecePlan{0, 0} : (fused ? fused_piece_plan(T, N, H, M) : piece_plan(T, N, H, M));
  p.piece_len = (int)pp.len;
  p.piece_rows = (int)pp.rows;
  p.piece_pass1 = 0;
  p.piece_buf = pp.len > 0 ? (float *)(ws + lay.piece) : nullptr;
  p.xfer = 0;
  p.xfer_out = nullptr;
  p.order = nullptr;
  p.wait_limit_ns = 1000000000ull;
  p.test_withhold_copy = 0;
  if (g_expiry_test_ns) {  // armed by gdp_arm_wait_expiry_test: this call only
    p.wait_limit_ns = g_expiry_test_ns;
    p.test_withhold_copy = 1;
    g_expiry_test_ns = 0;
  }
  p.bounds = gdp::bounds_record();
  p.bounds_shrink = g_bounds_test ? 1 : 0;  // armed by gdp_arm_bounds_test: this call only
  g_bounds_test = false;
  if (xfer_out) {  // B (rows 0 .. N-1) and Phi (rows N .. 2N-1) of every sequence, no outputs
    p.xfer = 1;
    p.xfer_out = xfer_out;
    p.out = nullptr;
    p.out_state = nullptr;
    p.chunk_states = nullptr;
    p.init = nullptr;
    p.cache = nullptr;
    p.slots = nullptr;
    p.num_slots = 0;
  }
  // desc -> WY -> scan on one stream overlap their launches (programmatic dependent launch);
  // the profiled form records events between them, so there each kernel runs alone
  p.pdl = ((nseg == 1 || fused) && !ev) ? 1 : 0;
  SideStreams *ss = (nseg > 1 && !fused) ? side_streams() : nullptr;
  if (nseg > 1 && !fused && !ss) return fail(GDP_ERR_CUDA, "could not create the internal streams of the segmented mode");

  // a call over whole sequences in one launch runs them longest first (the descriptor kernel's
  // order); split chains and segments keep the grid order
  int32_t *ord = (pp.len == 0 && N > 1 && !xfer_out && (fused || nseg == 1)) ? (int32_t *)(ws + lay.ord) : nullptr;
  p.order = ord;
  cudaError_t e;
  if (nprebuilt == 3)  // only the internal expanded-stream offsets
    e = gdp::launch_descriptors(p.cu, p.cu64, T, N, M, nullptr, 0, nullptr, 0, nullptr, (int32_t *)p.cod, p.status,
                                stream, ord, p.bounds);
  else
    e = gdp::launch_descriptors(p.cu, p.cu64, T, N, M, (int32_t *)p.ci, nt_pad, (int32_t *)p.cid, ntdp_pad,
                                co_desc, (int32_t *)p.cod, p.status, stream, ord, p.bounds);
  if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "descriptor kernel: %s", cudaGetErrorString(e));
  if (ev && (st = record(ev[1], stream)) != GDP_OK) return st;
  if (fused) {  // no WY stage of its own: events 1 and 2 mark the same point
    if (ev && (st = record(ev[2], stream)) != GDP_OK) return st;
    if (pp.len > 0) {  // split chains: B and Phi of the pieces, their entering states, the pieces
      gdp::Problem q = p;
      q.piece_pass1 = 1;
      q.out = nullptr;
      q.out_state = nullptr;
      q.chunk_states = nullptr;
      e = gdp::launch_fused(q, stream);
      if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "fused kernel (pieces): %s", cudaGetErrorString(e));
      e = gdp::launch_piece_combine(p, stream);
      if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "piece combine kernel: %s", cudaGetErrorString(e));
    }
    e = gdp::launch_fused(p, stream);
    if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "fused kernel: %s", cudaGetErrorString(e));
    if (ev && (st = record(ev[3], stream)) != GDP_OK) return st;
    return GDP_OK;
  }
  if (nseg == 1) {
    e = gdp::launch_wy(p, stream);
    if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "WY kernel: %s", cudaGetErrorString(e));
    if (ev && (st = record(ev[2], stream)) != GDP_OK) return st;
    if (pp.len > 0) {  // split chains: B and Phi of the pieces, their entering states, the pieces
      gdp::Problem q = p;
      q.piece_pass1 = 1;
      q.out = nullptr;
      q.out_state = nullptr;
      q.chunk_states = nullptr;
      e = gdp::launch_scan(q, stream);
      if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "scan kernel (pieces): %s", cudaGetErrorString(e));
      e = gdp::launch_piece_combine(p, stream);
      if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "piece combine kernel: %s", cudaGetErrorString(e));
    }
    e = gdp::launch_scan(p, stream);
    if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "scan kernel: %s", cudaGetErrorString(e));
    if (ev && (st = record(ev[3], stream)) != GDP_OK) return st;
    return GDP_OK;
  }
  // Segmented: WY(k + 1) on the low-priority stream runs beside scan(k) on the high-priority
  // one; scan(k) waits for WY(k) by event, and the state crosses segments through seg_state.
  const int64_t maxc = ((int64_t)M * T + gdp::kChunk - 1) / gdp::kChunk;
  const int64_t S = (maxc + nseg - 1) / nseg;
  p.seg_state = (float *)(ws + lay.seg);
  p.seg_rows = (int)S;
  auto cuda_fail = [](const char *what, cudaError_t err) {
    return fail(GDP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
  };
  if ((e = cudaEventRecord(ss->ev[0], stream)) != cudaSuccess) return cuda_fail("fork", e);
  if ((e = cudaStreamWaitEvent(ss->wy, ss->ev[0], 0)) != cudaSuccess) return cuda_fail("fork", e);
  if ((e = cudaStreamWaitEvent(ss->scan, ss->ev[0], 0)) != cudaSuccess) return cuda_fail("fork", e);
  for (int k = 0; k <= nseg; ++k) {
    if (k < nseg) {  // WY tiles of segment k
      gdp::Problem q = p;
      q.seg_lo = k * S;
      q.seg_hi = (k + 1) * S;
      if ((e = gdp::launch_wy(q, ss->wy)) != cudaSuccess) return cuda_fail("WY kernel", e);
      if ((e = cudaEventRecord(ss->ev[1 + k], ss->wy)) != cudaSuccess) return cuda_fail("event", e);
    }
    if (k > 0) {  // scan of segment k - 1, once its tiles exist
      gdp::Problem q = p;
      q.seg_lo = (k - 1) * S;
      q.seg_hi = (k == nseg) ? INT64_MAX : k * S;
      if ((e = cudaStreamWaitEvent(ss->scan, ss->ev[k], 0)) != cudaSuccess) return cuda_fail("event", e);
      if (k == 1 && ev && (st = record(ev[2], ss->scan)) != GDP_OK) return st;
      if ((e = gdp::launch_scan(q, ss->scan)) != cudaSuccess) return cuda_fail("scan kernel", e);
    }
  }
  if ((e = cudaEventRecord(ss->ev[nseg + 1], ss->scan)) != cudaSuccess) return cuda_fail("join", e);
  if ((e = cudaStreamWaitEvent(stream, ss->ev[nseg + 1], 0)) != cudaSuccess) return cuda_fail("join", e);
  if (ev && (st = record(ev[3], stream)) != GDP_OK) return st;
  return GDP_OK;
}

}  // namespace

void gdp::set_last_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
}

GDP_EXPORT int64_t gdp_nt_pad(int64_t T, int64_t N) { return nt_bound(T, N); }

GDP_EXPORT int64_t gdp_ntdp_pad(int64_t T, int64_t N, int M) { return ntdp_bound(T, N, M); }

GDP_EXPORT size_t gdp_prefill_workspace_bytes(int64_t T, int64_t N, int H, int K, int V, int M) {
  if (!shape_ok(T, N, H, K, V, M)) return 0;
  return layout_for(T, N, H, K, V, M).total;
}

GDP_EXPORT gdp_status gdp_prefill_plan(int64_t T, int64_t N, int H, int K, int V, int M, int64_t *segments,
                                       int64_t *piece_chunks, int64_t *piece_rows, int64_t *launches) {
  g_last_error[0] = 0;
  if (!shape_ok(T, N, H, K, V, M))
    return fail(GDP_ERR_INVALID_ARG, "bad shape T=%lld N=%lld H=%d K=%d V=%d M=%d", (long long)T, (long long)N, H, K,
                V, M);
  const int nseg = seg_count(T, N, H, M);
  const PiecePlan pp = piece_plan(T, N, H, M);
  if (segments) *segments = nseg;
  if (piece_chunks) *piece_chunks = pp.len;
  if (piece_rows) *piece_rows = pp.rows;
  if (launches) *launches = N == 0 ? 0 : 1 + (nseg > 1 ? 2 * nseg : (pp.len > 0 ? 4 : 2));
  return GDP_OK;
}

GDP_EXPORT int gdp_prefill_fused(int64_t T, int64_t N, int H, int K, int V, int M, int64_t *piece_chunks,
                                 int64_t *piece_rows, int64_t *launches) {
  if (!shape_ok(T, N, H, K, V, M) || !gdp::fused_shape(K, V, M)) return 0;
  const PiecePlan pp = fused_piece_plan(T, N, H, M);
  if (piece_chunks) *piece_chunks = pp.len;
  if (piece_rows) *piece_rows = pp.rows;
  if (launches) *launches = N == 0 ? 0 : 1 + (pp.len > 0 ? 3 : 1);
  return 1;
}

GDP_EXPORT const char *gdp_last_error(void) { return g_last_error; }

GDP_EXPORT gdp_status gdp_debug_bounds_record(int64_t out[4]) {
  g_last_error[0] = 0;
#if GDP_DEBUG_BOUNDS
  if (!out) return fail(GDP_ERR_INVALID_ARG, "out is NULL");
  unsigned long long rec[4] = {0, 0, 0, 0};
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(rec, g_bounds_rec, sizeof rec);
  const unsigned long long zero[4] = {0, 0, 0, 0};
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_bounds_rec, zero, sizeof zero);
  if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "debug-bounds record: %s", cudaGetErrorString(e));
  for (int i = 0; i < 4; ++i) out[i] = (int64_t)rec[i];
  return GDP_OK;
#else
  (void)out;
  return fail(GDP_ERR_UNSUPPORTED, "not a debug-bounds build (GDP_DEBUG_BOUNDS)");
#endif
}

GDP_EXPORT gdp_status gdp_arm_bounds_test(void) {
  g_last_error[0] = 0;
#if GDP_DEBUG_BOUNDS
  g_bounds_test = true;
  return GDP_OK;
#else
  return fail(GDP_ERR_UNSUPPORTED, "not a debug-bounds build (GDP_DEBUG_BOUNDS)");
#endif
}

GDP_EXPORT gdp_status gdp_arm_wait_expiry_test(uint64_t limit_ns) {
  g_last_error[0] = 0;
  if (limit_ns < 100000ull || limit_ns > 1000000000ull)
    return fail(GDP_ERR_INVALID_ARG, "limit_ns %llu outside [1e5, 1e9]", (unsigned long long)limit_ns);
  g_expiry_test_ns = limit_ns;
  return GDP_OK;
}

GDP_EXPORT int gdp_abi_version(void) { return GDP_ABI_VERSION; }

GDP_EXPORT size_t gdp_prefill_args_size(void) { return sizeof(gdp_prefill_args); }

GDP_EXPORT gdp_status gdp_build_descriptors(const void *cu_seqlens, int cu_seqlens_int64, int64_t T, int64_t N,
                                            int M, int32_t *chunk_indices, int64_t nt_pad,
                                            int32_t *chunk_indices_dp, int64_t ntdp_pad, int32_t *chunk_offsets,
                                            int32_t *chunk_offsets_dp, uint32_t *device_status, void *stream) {
  g_last_error[0] = 0;
  if (!cu_seqlens) return fail(GDP_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if (T < 0 || N < 0 || M < 1 || M > 64)
    return fail(GDP_ERR_INVALID_ARG, "bad shape T=%lld N=%lld M=%d", (long long)T, (long long)N, M);
  if (chunk_indices && !chunk_offsets) return fail(GDP_ERR_INVALID_ARG, "chunk_indices needs chunk_offsets");
  if (chunk_indices_dp && !chunk_offsets_dp)
    return fail(GDP_ERR_INVALID_ARG, "chunk_indices_dp needs chunk_offsets_dp");
  if (chunk_indices && nt_pad < nt_bound(T, N))
    return fail(GDP_ERR_INVALID_ARG, "nt_pad %lld < bound %lld", (long long)nt_pad, (long long)nt_bound(T, N));
  if (chunk_indices_dp && ntdp_pad < ntdp_bound(T, N, M))
    return fail(GDP_ERR_INVALID_ARG, "ntdp_pad %lld < bound %lld", (long long)ntdp_pad,
                (long long)ntdp_bound(T, N, M));
  cudaError_t e = gdp::launch_descriptors(cu_seqlens, cu_seqlens_int64, T, N, M, chunk_indices, nt_pad,
                                          chunk_indices_dp, ntdp_pad, chunk_offsets, chunk_offsets_dp,
                                          device_status, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "descriptor kernel: %s", cudaGetErrorString(e));
  return GDP_OK;
}

GDP_EXPORT gdp_status gdp_prefill_varlen(const gdp_prefill_args *a, void *stream) {
  return prefill(a, (cudaStream_t)stream, nullptr);
}

GDP_EXPORT gdp_status gdp_prefill_varlen_fused(const gdp_prefill_args *a, void *stream) {
  return prefill(a, (cudaStream_t)stream, nullptr, nullptr, nullptr, true);
}

GDP_EXPORT gdp_status gdp_prefill_varlen_fused_profiled(const gdp_prefill_args *a, void *stream, void *const *events,
                                                        int num_events) {
  if (!events || num_events != 4) {
    g_last_error[0] = 0;
    return fail(GDP_ERR_INVALID_ARG, "gdp_prefill_varlen_fused_profiled needs exactly 4 events");
  }
  cudaEvent_t ev[4];
  for (int i = 0; i < 4; ++i) ev[i] = (cudaEvent_t)events[i];
  return prefill(a, (cudaStream_t)stream, ev, nullptr, nullptr, true);
}

GDP_EXPORT gdp_status gdp_prefill_transfer(const gdp_prefill_args *a, float *pairs, void *stream) {
  g_last_error[0] = 0;
  if (!a) return fail(GDP_ERR_INVALID_ARG, "args is NULL");
  if (a->N > 0 && !pairs) return fail(GDP_ERR_INVALID_ARG, "pairs is NULL");
  if (((uintptr_t)pairs & 15u) != 0) return fail(GDP_ERR_INVALID_ARG, "pairs must be 16-byte aligned");
  if (a->N > 0 && a->H > 0 && 2 * a->N * (int64_t)a->H * a->V > INT32_MAX)
    return fail(GDP_ERR_UNSUPPORTED, "transfer pairs above 2^31 rows of K floats");
  return prefill(a, (cudaStream_t)stream, nullptr, nullptr, pairs);
}

GDP_EXPORT gdp_status gdp_chain_states(const float *s0, const float *phi, const float *b, int64_t steps, int64_t N,
                                       int H, int d, float *s_out, uint32_t *device_status, void *stream) {
  g_last_error[0] = 0;
  if (steps < 0 || N < 0 || H < 1 || (d != 64 && d != 128))
    return fail(GDP_ERR_INVALID_ARG, "bad shape steps=%lld N=%lld H=%d d=%d (d is 64 or 128)", (long long)steps,
                (long long)N, H, d);
  if (N == 0) return GDP_OK;
  if (!s_out || (steps > 0 && (!phi || !b))) return fail(GDP_ERR_INVALID_ARG, "s_out, phi and b are required");
  if ((((uintptr_t)s0 | (uintptr_t)phi | (uintptr_t)b | (uintptr_t)s_out) & 15u) != 0)
    return fail(GDP_ERR_INVALID_ARG, "state buffers must be 16-byte aligned");
  const size_t one = sizeof(float) * (size_t)N * H * (size_t)d * d;
  if (steps * N * (int64_t)H * d > INT32_MAX) return fail(GDP_ERR_UNSUPPORTED, "Phi above 2^31 rows of d floats");
  if (overlaps(s_out, one * (size_t)(steps + 1), s0, one) || overlaps(s_out, one * (size_t)(steps + 1), phi, one * steps) ||
      overlaps(s_out, one * (size_t)(steps + 1), b, one * steps))
    return fail(GDP_ERR_ALIAS, "s_out must not overlap s0, phi or b");
  cudaError_t e = gdp::launch_chain_states(s0, phi, b, steps, N, H, d, s_out, device_status, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(GDP_ERR_CUDA, "chain kernel: %s", cudaGetErrorString(e));
  return GDP_OK;
}

namespace {

// Backward workspace: the forward's layout (recompute) followed by the backward's buffers.
struct BwdLayout {
  size_t Sx, Dx, fin, tot, sig, rho, bimg, bimg_stride, total;
};

BwdLayout bwd_layout_for(int64_t T, int64_t N, int H, int K, int V, int M) {
  BwdLayout l{};
  size_t off = layout_for(T, N, H, K, V, M).total;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  const size_t kv = (size_t)K * V * sizeof(float);
  const int64_t ntdp = ntdp_bound(T, N, M);
  l.Sx = take((size_t)ntdp * H * kv);
  l.Dx = take((size_t)ntdp * H * kv);
  l.fin = take((size_t)N * H * kv);
  l.tot = take((size_t)N * H * sizeof(float));
  l.sig = take((size_t)T * M * H * sizeof(float));
  l.rho = take((size_t)T * H * sizeof(float));
  l.bimg_stride = gdp::bwd_image_stride(K, gdp::qpad_for(M));
  l.bimg = take((size_t)ntdp * H * l.bimg_stride);
  l.total = off;
  return l;
}

gdp_status backward(const gdp_backward_args *b, cudaStream_t stream) {
  g_last_error[0] = 0;
  if (!b || !b->fwd) return fail(GDP_ERR_INVALID_ARG, "args and args->fwd are required");
  const gdp_prefill_args *a = b->fwd;
  const int64_t T = a->T, N = a->N;
  const int H = a->H, K = a->K, V = a->V, M = a->num_householder;
  if (!shape_ok(T, N, H, K, V, M))
    return fail(GDP_ERR_INVALID_ARG, "bad shape T=%lld N=%lld H=%d K=%d V=%d M=%d", (long long)T, (long long)N, H, K,
                V, M);
  if (K != V || (K != 64 && K != 128))
    return fail(GDP_ERR_UNSUPPORTED, "head sizes K=%d V=%d: the backward serves K == V in {64, 128}", K, V);
  if ((a->qkv_dtype && a->qkv_dtype != GDP_DTYPE_BF16) || (a->g_dtype && a->g_dtype != GDP_DTYPE_F32) ||
      a->g_is_alpha || (a->beta_dtype && a->beta_dtype != GDP_DTYPE_F32) ||
      (a->initial_state_dtype && a->initial_state_dtype != GDP_DTYPE_F32))
    return fail(GDP_ERR_UNSUPPORTED,
                "the backward serves bf16 q/k/v, fp32 natural-log g, fp32 beta and an fp32 initial state");
  if ((a->num_q_heads && a->num_q_heads != H) || (a->num_k_heads && a->num_k_heads != H) ||
      (a->num_v_heads && a->num_v_heads != H))
    return fail(GDP_ERR_UNSUPPORTED, "the backward serves one-to-one heads (num_q/k/v_heads 0 or H)");
  if (a->state || a->state_indices)
    return fail(GDP_ERR_UNSUPPORTED, "the backward serves the dense state mode (initial_state), not the cache");
  if (T > 0 && (!b->d_output || !b->dq || !b->dk || !b->dv))
    return fail(GDP_ERR_INVALID_ARG, "d_output, dq, dk and dv are required");
  const uintptr_t al = ((uintptr_t)b->d_output | (uintptr_t)b->dq | (uintptr_t)b->dk | (uintptr_t)b->dv |
                        (uintptr_t)b->d_final_state | (uintptr_t)b->d_initial_state | (uintptr_t)b->dg |
                        (uintptr_t)b->dbeta) & 15u;
  if (al) return fail(GDP_ERR_INVALID_ARG, "d_output and every gradient buffer must be 16-byte aligned");
  const int64_t ntdpb = ntdp_bound(T, N, M);
  if (ntdpb * (int64_t)H * V > INT32_MAX)
    return fail(GDP_ERR_UNSUPPORTED, "per-chunk state arrays above 2^31 rows of K floats");
  const BwdLayout bl = bwd_layout_for(T, N, H, K, V, M);
  if (!b->workspace || ((uintptr_t)b->workspace % kAlign) != 0)
    return fail(GDP_ERR_WORKSPACE, "workspace must be non-NULL and %zu-byte aligned", kAlign);
  if (b->workspace_bytes < bl.total)
    return fail(GDP_ERR_WORKSPACE, "workspace of %zu bytes < required %zu", b->workspace_bytes, bl.total);
  char *ws = (char *)b->workspace;

  // 1. forward recompute: descriptors, WY images, and the state entering every expanded chunk
  gdp_prefill_args f = *a;
  f.output = nullptr;
  f.output_state = nullptr;
  f.chunk_states = nullptr;
  f.chunk_indices = f.chunk_indices_dp = f.chunk_offsets = nullptr;
  f.nt_pad = f.ntdp_pad = 0;
  f.workspace = ws;
  f.workspace_bytes = layout_for(T, N, H, K, V, M).total;
  f.device_status = b->device_status;
  Recompute rc{(float *)(ws + bl.Sx), b->d_final_state ? (float *)(ws + bl.fin) : nullptr,
               (unsigned char *)(ws + bl.bimg), bl.bimg_stride};
  gdp_status st = prefill(&f, stream, nullptr, &rc);
  if (st != GDP_OK) return st;
  if (N == 0) return GDP_OK;

  // 2. reverse state scan, per-chunk gradients, decay gradient
  cudaError_t e;
  const Layout fl = layout_for(T, N, H, K, V, M);
  gdp::BwdProblem p{};
  p.q = (const __nv_bfloat16 *)a->q;
  p.k = (const __nv_bfloat16 *)a->k;
  p.v = (const __nv_bfloat16 *)a->v;
  p.q_st = a->q_stride_t; p.q_sh = a->q_stride_h;
  p.k_st = a->k_stride_t; p.k_sh = a->k_stride_h;
  p.v_st = a->v_stride_t; p.v_sh = a->v_stride_h;
  p.g = a->g;
  p.beta = a->beta;
  p.cu = a->cu_seqlens;
  p.cu64 = a->cu_seqlens_int64 ? 1 : 0;
  p.T = T; p.N = N; p.H = H; p.D = K; p.M = M;
  p.qpad = gdp::qpad_for(M);
  p.scale = (a->scale > 0.f && !isnan(a->scale)) ? a->scale : 1.0f / sqrtf((float)K);
  p.l2norm = a->use_qk_l2norm ? 1 : 0;
  p.cid = (const int32_t *)(ws + fl.cid);
  p.cod = (const int32_t *)(ws + fl.cod);
  p.ntdp_pad = ntdpb;
  p.ws_rows = ntdpb;
  p.img = (const unsigned char *)(ws + fl.img);
  p.img_stride = fl.img_stride;
  p.bimg = (const unsigned char *)(ws + bl.bimg);
  p.bimg_stride = bl.bimg_stride;
  p.Sx = (const float *)(ws + bl.Sx);
  p.Dx = (float *)(ws + bl.Dx);
  p.dout = (const __nv_bfloat16 *)b->d_output;
  p.dfin = b->d_final_state;
  p.fin = b->d_final_state ? (const float *)(ws + bl.fin) : nullptr;
  p.dinit = b->d_initial_state;
  p.tot = (float *)(ws + bl.tot);
  p.sig = (float *)(ws + bl.sig);
  p.rho = (float *)(ws + bl.rho);
  p.dq = b->dq;
  p.dk = b->dk;
  p.dv = b->dv;
  p.dg = b->dg;
  p.dbeta = b->dbeta;
  p.status = b->device_status;
  if ((e = gdp::launch_backward(p, stream)) != cudaSuccess)
    return fail(GDP_ERR_CUDA, "backward kernels: %s", cudaGetErrorString(e));
  return GDP_OK;
}

}  // namespace

GDP_EXPORT size_t gdp_backward_workspace_bytes(int64_t T, int64_t N, int H, int K, int V, int M) {
  if (!shape_ok(T, N, H, K, V, M)) return 0;
  return bwd_layout_for(T, N, H, K, V, M).total;
}

GDP_EXPORT gdp_status gdp_prefill_varlen_backward(const gdp_backward_args *args, void *stream) {
  return backward(args, (cudaStream_t)stream);
}

GDP_EXPORT gdp_status gdp_prefill_varlen_profiled(const gdp_prefill_args *a, void *stream, void *const *events,
                                                  int num_events) {
  if (!events || num_events != 4) {
    g_last_error[0] = 0;
    return fail(GDP_ERR_INVALID_ARG, "gdp_prefill_varlen_profiled needs exactly 4 events");
  }
  cudaEvent_t ev[4];
  for (int i = 0; i < 4; ++i) ev[i] = (cudaEvent_t)events[i];
  return prefill(a, (cudaStream_t)stream, ev);
}
