// gdp_fused.cu -- the fused prefill kernel: per (sequence, head) one CTA runs the WY work of
// every expanded chunk, the inter-chunk state scan, the output combine and the state scatter,
// with nothing of a chunk leaving the SM but its outputs and requested states.
//
// Megatron-Core API page "core.ssm.ops.gdp.chunk", stages 1-4 (decay interleave and base-2
// cumsum, WY build, inter-chunk sweep, output combine) as one pipeline, for the common
// contract of the FlashInfer page "flashinfer.gdp_prefill.chunk_gated_delta_product": bfloat16
// q / k / v (heads may be grouped), natural-log fp32 g, fp32 beta, fp32 states (dense initial
// state or the in-place cache), head size 128, num_householder >= 2.
//
// The algebra is the staged path's (gdp_wy_body.cuh, gdp_scan_body.cuh): for expanded chunk c
// with entering state S (V-major), gamma_r = 2^G2_r the within-chunk decay,
//   A = strictly lower beta_i gamma_i / gamma_j khat_i . khat_j,   T = (I + A)^-1,
//   W = T diag(beta gamma rk) K,   U = T diag(beta) V,
//   V_new^T = U^T - S W^T,   o^T = S Qh^T + V_new^T P^T,   S' = gamma_last S + V_new^T Ktil.
// The state stays in tensor memory as S_hat = S / Gamma (Gamma a running product of chunk
// decays).  Unlike the staged scan, the decay bookkeeping is carried by the operands that the
// CTA builds itself, so V_new and o come out of the tensor cores unscaled:
//   [o | Y] = [0 | U^T] + S_hat [Gamma Qh ; -Gamma W]^T      (Y = V_new^T; U^T written by an MMA)
//   S_hat  += Y (Ktil / Gamma')^T,   o += Y P^T              (Gamma' = Gamma gamma_last)
// A chunk whose decay is below 2^kFastMinLog2Gamma ("slow") runs with Gamma = 1 and its decay
// applied to S_hat between the two products; Gamma is renormalised to 1 before it would drop
// below kRenormMinGamma.
//
// Warp roles (416 threads):
//   warps 0-7   math   : per chunk, a chunk ahead of the scan: row scalars (beta, decay cumsum,
//                        L2 norms), the Gram epilogue (A and P), T = (I + A)^-1, the bf16 hi + lo
//                        splits of T diag(beta gamma rk) and T diag(beta), then the chunk's fp32
//                        operands of the scan (Gamma Qh, -Gamma W, Ktil^T / Gamma', P) in shared
//                        memory; renormalisation, state snapshots and slow-chunk decay in TMEM;
//                        thread 0 issues the TMA loads of the next chunk's k, q, v tiles.
//                        Two warps per TMEM lane quadrant, splitting the columns.
//   warps 8-11  store  : outputs (bf16, one TMA store per full chunk), chunk states, final state.
//   warp 12     control: one thread issues every tcgen05.mma: the Gram [K; Q] K^T, W^T and U^T
//                        (bf16, T split hi + lo), and the two tf32 batches of the scan.
// The tensor pipe runs in issue order, so the control thread places the next chunk's Gram
// between the current chunk's two scan batches: the math warps' CUDA-core work (epilogue,
// inverse, splits) overlaps the scan's products.
//
// Every wait is bounded (Problem::wait_limit_ns); on expiry the CTA sets GDP_DEV_ERR_TIMEOUT,
// drains its own MMAs and copies, frees its tensor memory and returns.
#include <cuda.h>

#include "gdp_scan_body.cuh"  // ChunkInfo, kStTile
#include "gdp_wy_body.cuh"    // In16, in_at / in8_at, tf32 helpers, kLd / kLdT / kLdY

namespace gdp {
namespace {

using namespace sm100;

constexpr int kFusedThreads = 416;
constexpr int kFusedD = 128;
constexpr int kMathThreads = 256;
constexpr uint32_t kBarMath = 1, kBarStore = 2;  // named barriers (0 is __syncthreads)

// Dynamic shared memory (head size 128, qpad <= 32), every region 1024-byte aligned:
//   kq   [2][128 rows][128 B] bf16  rows 0..63 k, 64..64+qpad-1 q (TMA boxes, 128-byte swizzle)
//   vt   [2][64 rows][128 B]  bf16  v
//   b1   [4][qpad + 64][128 B] fp32 rows 0..qpad-1 Gamma Qh, qpad.. -Gamma W (B of batch 1)
//   b2   [2][128 + qpad][128 B] fp32 rows 0..127 Ktil^T / Gamma', 128.. P (B of batch 2)
//   R    32 KB: A [64][65] fp32 + block scratch [32][36] during the inverse, then the splits
//        Tw_hi, Tw_lo, Tu_hi, Tu_lo, bf16 [64][64] K-major swizzled (B of the W / U MMAs)
//   T    [64][68] fp32
//   P    [2][qpad][128 B] fp32, P rows in the swizzle of b2's P rows (copied there later)
//   scal 8 x 64 floats: G2, beta, rk, rq, wc, uc, ks, qs
//   obuf [qpad][128] bf16 output staging
//   st   [4 store warps][4 KB] 32 x 32 fp32 boxes of the state stores
struct FusedLayout {
  uint32_t kq, vt, b1, b1_block, b2, b2_block, R, T, P, scal, obuf, st, total;
  __host__ __device__ explicit FusedLayout(int qpad) {
    kq = 0;
    vt = 32768u;
    b1 = 49152u;
    b1_block = (uint32_t)(qpad + 64) * 128u;
    b2 = b1 + 4u * b1_block;
    b2_block = (uint32_t)(kFusedD + qpad) * 128u;
    R = b2 + 2u * b2_block;
    T = R + 32768u;
    P = T + 17408u;
    scal = P + 2u * (uint32_t)qpad * 128u;
    obuf = scal + 2048u;
    st = obuf + (uint32_t)qpad * kFusedD * 2u;
    total = st + 4u * kStTile;
  }
};

__host__ __device__ inline bool fused_tmem_fits(int qpad) { return 2 * kFusedD + 2 * (qpad + 64) + 64 <= 512; }

// Geometry of expanded chunk c of a sequence starting at token bos with L tokens.
struct ChunkGeo {
  int64_t R0, tok0, tq0;
  int len, r0m, p0, nq;
};
__device__ __forceinline__ ChunkGeo chunk_geo(int64_t bos, int64_t L, int M, int64_t c) {
  ChunkGeo g;
  g.R0 = bos * M + c * kChunk;
  g.len = (int)min((int64_t)kChunk, L * M - c * kChunk);
  g.r0m = (int)(g.R0 % M);
  g.tok0 = (g.R0 - g.r0m) / M;
  g.p0 = (M - 1 - g.r0m) % M;
  g.nq = (g.p0 < g.len) ? (g.len - 1 - g.p0) / M + 1 : 0;
  g.tq0 = (g.R0 + g.p0) / M;
  return g;
}

// 3xTF32 off-diagonal blocks of T (the staged WY kernel's recursive doubling) with the math
// warps' named barrier in place of __syncthreads.
__device__ __forceinline__ void inverse_offdiag_math(const float *A, float *Tm, float *Y, int warp, int lane) {
  const int g = lane >> 2, t = lane & 3;
  if (warp < 4) {
    const int pr = warp >> 1, nh = warp & 1, i = 2 * pr + 1, j = 2 * pr;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ks = 0; ks < 2; ++ks)
      mma3_16x8x8(c, A + (16 * i) * kLd + 16 * j + 8 * ks, kLd, Tm + (16 * j + 8 * ks) * kLdT + 16 * j + 8 * nh, kLdT,
                  lane);
    float *y = Y + (pr * 16) * kLdY + 8 * nh;
    y[g * kLdY + 2 * t] = c[0];
    y[g * kLdY + 2 * t + 1] = c[1];
    y[(g + 8) * kLdY + 2 * t] = c[2];
    y[(g + 8) * kLdY + 2 * t + 1] = c[3];
  }
  named_sync(kBarMath, kMathThreads);
  if (warp < 4) {
    const int pr = warp >> 1, nh = warp & 1, i = 2 * pr + 1, j = 2 * pr;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ks = 0; ks < 2; ++ks)
      mma3_16x8x8(c, Tm + (16 * i) * kLdT + 16 * i + 8 * ks, kLdT, Y + (pr * 16 + 8 * ks) * kLdY + 8 * nh, kLdY, lane);
    float *o = Tm + (16 * i) * kLdT + 16 * j + 8 * nh;
    o[g * kLdT + 2 * t] = -c[0];
    o[g * kLdT + 2 * t + 1] = -c[1];
    o[(g + 8) * kLdT + 2 * t] = -c[2];
    o[(g + 8) * kLdT + 2 * t + 1] = -c[3];
  }
  named_sync(kBarMath, kMathThreads);
  const int mt = warp >> 2, nt = warp & 3;
  {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ks = 0; ks < 4; ++ks)
      mma3_16x8x8(c, A + (32 + 16 * mt) * kLd + 8 * ks, kLd, Tm + (8 * ks) * kLdT + 8 * nt, kLdT, lane);
    float *y = Y + (16 * mt) * kLdY + 8 * nt;
    y[g * kLdY + 2 * t] = c[0];
    y[g * kLdY + 2 * t + 1] = c[1];
    y[(g + 8) * kLdY + 2 * t] = c[2];
    y[(g + 8) * kLdY + 2 * t + 1] = c[3];
  }
  named_sync(kBarMath, kMathThreads);
  {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ks = 0; ks < 4; ++ks)
      mma3_16x8x8(c, Tm + (32 + 16 * mt) * kLdT + 32 + 8 * ks, kLdT, Y + (8 * ks) * kLdY + 8 * nt, kLdY, lane);
    float *o = Tm + (32 + 16 * mt) * kLdT + 8 * nt;
    o[g * kLdT + 2 * t] = -c[0];
    o[g * kLdT + 2 * t + 1] = -c[1];
    o[(g + 8) * kLdT + 2 * t] = -c[2];
    o[(g + 8) * kLdT + 2 * t + 1] = -c[3];
  }
  named_sync(kBarMath, kMathThreads);
}

// Store warp: the 32 state rows of this warp's TMEM lanes (columns from t_lane), times mul, to
// map rows [row, row + 32) as 32 x 32 boxes through this warp's one staging tile.  `read`
// (when given) is arrived on once the columns are in registers.
__device__ __forceinline__ void store_state_one_tile(uint32_t t_lane, unsigned char *tile, int lane, float mul,
                                                     const CUtensorMap *tm, int row, bool &pending, uint64_t *read) {
#pragma unroll 1
  for (int c0 = 0; c0 < kFusedD; c0 += 64) {
    uint32_t x[64];
    tmem_ld32x_nw(t_lane + c0, x);
    tmem_ld32x_nw(t_lane + c0 + 32, x + 32);
    tmem_ld_wait();
    if (read && c0 + 64 >= kFusedD) {
      tc_fence_before();
      mbar_arrive(read);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if (pending) {  // the previous box's store has read the tile
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t *y = x + 32 * c + 4 * j;
        *reinterpret_cast<float4 *>(tile + lane * 128 + ((j ^ (lane & 7)) << 4)) =
            make_float4(mul * __uint_as_float(y[0]), mul * __uint_as_float(y[1]), mul * __uint_as_float(y[2]),
                        mul * __uint_as_float(y[3]));
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tm, tile, c0 + 32 * c, row);
        bulk_commit();
      }
      pending = true;
    }
  }
}

__device__ __forceinline__ void fused_body(const Problem &p, const CUtensorMap &tm_k, const CUtensorMap &tm_q,
                                           const CUtensorMap &tm_v, const CUtensorMap &tm_cs,
                                           const CUtensorMap &tm_fin, const CUtensorMap &tm_seg,
                                           const CUtensorMap &tm_out_a, const CUtensorMap &tm_out_b) {
  using In = In16<false>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int M = p.M, QP = p.qpad, H = p.H;
  constexpr int d = kFusedD;
  // Split chains (Problem::piece_len > 0): this CTA runs one piece.  Pass 1 (piece_pass1): grid
  // row r < piece_rows runs piece r from a zero state (its B), row piece_rows + r from the
  // identity with U = 0 (its Phi), no outputs, the end state to piece_buf row (grid row); a
  // sequence's last piece has no pass 1.  Pass 2: piece r of a split sequence enters with
  // piece_buf row 2 piece_rows + r (the combine kernel's S_in) and writes its outputs, chunk
  // states and, as its sequence's last piece, the final state.
  const bool pieces = p.piece_len > 0, pass1 = pieces && p.piece_pass1;
  const bool transfer = pass1 && (int)blockIdx.x >= p.piece_rows;  // the Phi row of a piece
  const bool outs = !pass1;
  int seq = (int)blockIdx.x, pc_i = 0, pc_n = 1;
  int h = (int)blockIdx.y;
  if (!pieces && p.order) {
    // longest first: linear CTA index l (the order CTAs start in) runs sequence order[l / H],
    // head l % H; the order comes from the descriptor kernel
    pdl_wait();
    const int64_t l = (int64_t)blockIdx.x + (int64_t)blockIdx.y * gridDim.x;
    seq = p.order[l / H];
    h = (int)(l % H);
  }
  if (pieces) {
    // the piece table comes from the descriptors (chunk_offsets_dp); every CTA waits for its
    // predecessor grid before it may exit, so that this grid's completion implies theirs
    pdl_wait();
    __shared__ int pc_sh[3];
    if (warp == 0) {
      int sq, pi, np;
      piece_of_row(p, (int)blockIdx.x - (transfer ? p.piece_rows : 0), lane, &sq, &pi, &np);
      if (lane == 0) {
        pc_sh[0] = sq;
        pc_sh[1] = pi;
        pc_sh[2] = np;
      }
    }
    __syncthreads();
    seq = pc_sh[0];
    pc_i = pc_sh[1];
    pc_n = pc_sh[2];
    if (seq < 0 || (pass1 && pc_i == pc_n - 1)) return;  // past the last piece; a last piece has no pass 1
  }
  int64_t bos, L;
  const bool seq_ok = seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L);  // flagged by the descriptor kernel
  const int64_t nseq = seq_ok ? (L * M + kChunk - 1) / kChunk : 0;  // the sequence's expanded chunks
  // this launch's chunks: global chunk e0 + c for local c in [0, n)
  const int64_t e0 = pieces ? min((int64_t)pc_i * p.piece_len, nseq) : 0;
  const int64_t n = pieces ? max((int64_t)0, min(e0 + p.piece_len, nseq) - e0) : nseq;
  const bool last_piece = pc_i == pc_n - 1;
  const int hq = input_head(h, p.hmul_q), hk = input_head(h, p.hmul_k), hv = input_head(h, p.hmul_v);
  const uint64_t wl = p.wait_limit_ns;

  extern __shared__ __align__(1024) unsigned char fused_smem_raw[];
  // the 1024-aligned base as an offset into the shared array (accesses stay in the shared address space)
  unsigned char *sm = fused_smem_raw + ((1024u - (sm100::smem_u32(fused_smem_raw) & 1023u)) & 1023u);
  const FusedLayout lay(QP);
  unsigned char *kq = sm + lay.kq, *vt = sm + lay.vt;
  float *A = reinterpret_cast<float *>(sm + lay.R);
  float *Yw = A + kChunk * kLdT;
  float *Tm = reinterpret_cast<float *>(sm + lay.T);
  float *G2 = reinterpret_cast<float *>(sm + lay.scal);
  float *bt = G2 + 64, *rk = bt + 64, *rq = rk + 64, *wc = rq + 64, *uc = wc + 64, *ks = uc + 64, *qs = ks + 64;

  __shared__ __align__(8) uint64_t tl_full, gram_go, gram_done, wu_go, wu_done, ops_ready, mid_go, b1_done[2],
      b2_done[2], yo_free[2], bk_free, fin_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int st_ok[4];
  __shared__ int math_ok[2];
  __shared__ int slow_sh[2];
  __shared__ float warp_tot, gam_fin_sh;
  __shared__ volatile int abort_flag;

  if (warp == 12) tmem_alloc(&tmem_slot, 512);
  if (tid == 0) {
    mbar_init(&tl_full, 1);
    mbar_init(&gram_go, 1);
    mbar_init(&gram_done, 1);
    mbar_init(&wu_go, 1);
    mbar_init(&wu_done, 1);
    mbar_init(&ops_ready, 1);
    mbar_init(&mid_go, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b1_done[i], 1);
      mbar_init(&b2_done[i], 1);
      mbar_init(&yo_free[i], 128);
    }
    mbar_init(&bk_free, 128);
    mbar_init(&fin_bar, 1);
    mbar_init_fence();
    abort_flag = 0;
    gam_fin_sh = 1.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // TMEM columns: [0, 128) S_hat | buffer b at 128 + b (qpad + 64): [o: qpad][Y: 64] |
  // Gram, then W^T: 64 | snapshot: 128
  const uint32_t tb = tmem_slot;
  const uint32_t tS = tb;
  auto tO = [&](int b) { return tb + 128u + (uint32_t)b * (uint32_t)(QP + 64); };
  const uint32_t tW = tb + 128u + 2u * (uint32_t)(QP + 64);
  const uint32_t tBk = tW + 64u;

  // incoming state source (cache slot, dense initial state, or zero)
  int slot = -1;
  const float *src = nullptr;
  if (p.cache) {
    slot = p.slots[seq];
    if (slot < -1 || slot >= p.num_slots) {
      if (tid == 0 && !pass1 && pc_i == 0) set_status(p.status, GDP_DEV_ERR_SLOT);
      slot = -1;
    }
    if (slot >= 0) src = p.cache + ((int64_t)slot * H + h) * (int64_t)p.V * d;
  } else if (p.init) {
    src = static_cast<const float *>(p.init) + ((int64_t)seq * H + h) * (int64_t)p.V * d;
  }
  if (pass1 || pc_n > 1)  // zero (or the identity) for B / Phi; a split piece from its S_in
    src = pass1 ? nullptr : p.piece_buf + ((int64_t)(2 * p.piece_rows + (int)blockIdx.x) * H + h) * (int64_t)p.V * d;

  const int q4 = warp & 3;                 // TMEM lane quadrant of math and store warps
  const int v = q4 * 32 + lane;            // state row / feature of this thread's TMEM lane
  const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
  const int hf = (warp < 8) ? (warp >> 2) : 0;  // math warps: column half
  bool load_pending = false;               // (thread 0) a tile load is in flight on tl_full
  int n_loads = 0;

  auto issue_tiles = [&](int64_t c) {  // thread 0: the k, q, v tiles of local chunk c
    const ChunkGeo g = chunk_geo(bos, L, M, e0 + c);
    mbar_arrive_expect_tx(&tl_full, 2u * (uint32_t)(64 + QP + 64) * 128u);
    for (int kb = 0; kb < 2; ++kb) {
      tma_load_3d(kq + kb * 16384u, &tm_k, kb * 64, hk, (int)g.R0, &tl_full);
      tma_load_3d(kq + kb * 16384u + 8192u, &tm_q, kb * 64, hq, (int)g.tq0, &tl_full);
      tma_load_3d(vt + kb * 8192u, &tm_v, kb * 64, hv, (int)g.R0, &tl_full);
    }
    load_pending = true;
    ++n_loads;
    if (c + 2 < n) {  // the tiles two chunks ahead into L2
      const ChunkGeo g2 = chunk_geo(bos, L, M, e0 + c + 2);
      for (int kb = 0; kb < 2; ++kb) {
        tma_prefetch_3d(&tm_k, kb * 64, hk, (int)g2.R0);
        tma_prefetch_3d(&tm_q, kb * 64, hq, (int)g2.tq0);
        tma_prefetch_3d(&tm_v, kb * 64, hv, (int)g2.R0);
      }
    }
  };

  if (warp < 8) {
    // S_0 into TMEM (warps of a quadrant split the columns) and both output buffers zeroed
    for (int c0 = hf * 64; c0 < hf * 64 + 64; c0 += 16) {
      float x[16];
#pragma unroll
      for (int u4 = 0; u4 < 16; u4 += 4) {
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
        if (src) y = *reinterpret_cast<const float4 *>(src + (int64_t)v * d + c0 + u4);
        x[u4] = y.x; x[u4 + 1] = y.y; x[u4 + 2] = y.z; x[u4 + 3] = y.w;
      }
      if (transfer)  // the identity
#pragma unroll
        for (int u = 0; u < 16; ++u) x[u] = (c0 + u == v) ? 1.f : 0.f;
      tmem_st16(tS + lrow + c0, x);
    }
    float z[16];
#pragma unroll
    for (int w = 0; w < 16; ++w) z[w] = 0.f;
    for (int c0 = 0; c0 < QP; c0 += 16) tmem_st16(tO(hf) + lrow + c0, z);
    tmem_st_wait();
    // (a test of the bounded waits withholds the first load of CTA (0, 0): its wait runs out)
    if (tid == 0 && n > 0 && !(p.test_withhold_copy && blockIdx.x == 0 && blockIdx.y == 0)) issue_tiles(0);
  }
  // chunk_offsets (chunk-state rows) come from the descriptor kernel
  if (!pieces && !p.order) pdl_wait();
  const int64_t co_i = p.chunk_states ? (int64_t)p.co[seq] : 0;
  auto emits = [&](int64_t c) {  // local chunk c
    const int64_t eg = e0 + c;
    return p.chunk_states && (eg % M == 0) && co_i >= 0 && co_i + eg / M < p.nt_pad;
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < 8) {
    // ================================ math warps ================================
    float gam = 1.f;  // Gamma of S_hat once the chunks so far are applied
    int n_emit = 0, n_slow = 0;
    // one waiter per mbarrier, the verdict shared through math_ok after the math barrier, so
    // that all math threads leave together (their named barriers are not bounded).  Two slots
    // used in turn: thread 0 rewrites a slot only after a later barrier, which every thread
    // reaches after reading it.
    int wk = 0;
    auto wait1 = [&](uint64_t *bar, uint32_t parity) {
      const int k = wk;
      wk ^= 1;
      if (tid == 0) math_ok[k] = mbar_wait_or_abort(bar, parity, &abort_flag, wl) ? 1 : 0;
      named_sync(kBarMath, kMathThreads);
      return math_ok[k] != 0;
    };
    for (int64_t c = 0; c < n; ++c) {
      const int b = (int)(c & 1);
      const ChunkGeo g = chunk_geo(bos, L, M, e0 + c);
      // per-row beta and decay gate (the decay of token t sits on its first expanded row t*M)
      float b_r = 0.f, gate_r = 0.f;
      if (tid < kChunk && tid < g.len) {
        const int pos = g.r0m + tid;
        b_r = p.beta ? static_cast<const float *>(p.beta)[(g.R0 + tid) * H + h] : 1.f;
        if (p.g && pos % M == 0) gate_r = static_cast<const float *>(p.g)[(g.tok0 + pos / M) * H + h];
      }
      if (!wait1(&tl_full, (uint32_t)(c & 1))) break;
      if (tid == 0) load_pending = false;
      {  // rows past the chunk (another sequence's data, or zero past the tensor) are cleared
        const uint4 zz = make_uint4(0u, 0u, 0u, 0u);
        const int nk = kChunk - g.len, nqz = QP - g.nq;
        for (int idx = tid; idx < 2 * (2 * nk + nqz) * 8; idx += kMathThreads) {
          const int ch = idx & 7, rr = idx >> 3, kb = rr & 1, r = rr >> 1;
          unsigned char *row = (r < nk) ? kq + kb * 16384u + (uint32_t)(g.len + r) * 128u
                               : (r < 2 * nk) ? vt + kb * 8192u + (uint32_t)(g.len + r - nk) * 128u
                                              : kq + kb * 16384u + (uint32_t)(64 + g.nq + r - 2 * nk) * 128u;
          *reinterpret_cast<uint4 *>(row + ch * 16) = zz;
        }
      }
      fence_async_smem();
      named_sync(kBarMath, kMathThreads);
      if (tid == 0) mbar_arrive(&gram_go);  // the control thread issues [K; Q] K^T

      // ---- row scalars: beta, inverse norms, base-2 cumsum of the gates ----
      {
        const int r = tid & 127, chalf = tid >> 7;
        float ss = 0.f;
        if (p.l2norm) {
#pragma unroll 1
          for (int f0 = chalf * (d / 2); f0 < (chalf + 1) * (d / 2); f0 += 8) {
            float x[8];
            in8_at<false>(kq, 128, r, f0, x);
#pragma unroll
            for (int i = 0; i < 8; ++i) ss += x[i] * x[i];
          }
          if (chalf) Yw[r] = ss;
          named_sync(kBarMath, kMathThreads);
          if (!chalf) ss += Yw[r];
        }
        if (!chalf) {
          if (r < kChunk) {
            bt[r] = b_r;
            rk[r] = p.l2norm ? rsqrtf(ss + kL2Eps) : 1.f;
            float x = gate_r;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const float y = __shfl_up_sync(0xffffffffu, x, o);
              if (lane >= o) x += y;
            }
            if (r == 31) warp_tot = x;
            G2[r] = x;
          } else {
            rq[r - kChunk] = p.l2norm ? rsqrtf(ss + kL2Eps) : 1.f;
          }
        }
      }
      named_sync(kBarMath, kMathThreads);
      if (tid < kChunk) G2[tid] = (tid >= 32 ? G2[tid] + warp_tot : G2[tid]) * kLog2e;
      named_sync(kBarMath, kMathThreads);
      const float G2last = G2[g.len - 1];
      const bool fast = G2last >= kFastMinLog2Gamma;
      const float gamma_last = exp2f(G2last);
      const bool renorm = fast ? (gam * gamma_last < kRenormMinGamma) : (gam != 1.f);
      const float gam_pass = renorm ? 1.f : gam;
      const float gam_next = fast ? gam_pass * gamma_last : 1.f;
      if (tid < kChunk) {
        wc[tid] = bt[tid] * exp2f(G2[tid]) * rk[tid];
        uc[tid] = transfer ? 0.f : bt[tid];
        ks[tid] = (tid < g.len) ? exp2f(G2last - G2[tid]) * rk[tid] : 0.f;
        const int pr = g.p0 + tid * M;
        qs[tid] = (tid < g.nq) ? p.scale * exp2f(G2[pr]) * rq[tid] : 0.f;
      }
#pragma unroll 1
      for (int idx = tid; idx < kChunk * kLdT / 4; idx += kMathThreads)
        reinterpret_cast<float4 *>(Tm)[idx] = make_float4(0.f, 0.f, 0.f, 0.f);

      // ---- Gram epilogue: A rows (lanes 0..63) and the scores P (lanes 64..64+qpad) ----
      if (!wait1(&gram_done, (uint32_t)(c & 1))) break;
      tc_fence_after();
      {
        const int r = v, cbeg = hf * 32;
        if (r < kChunk) {
          const bool rowlive = r < g.len;
          const float gi = G2[r], si = bt[r] * rk[r];
#pragma unroll 1
          for (int c0 = cbeg; c0 < cbeg + 32; c0 += 16) {
            float dv[16];
            tmem_ld16(tW + lrow + c0, dv);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const int j = c0 + u;
              A[r * kLd + j] = (j < r && rowlive) ? si * exp2f(gi - G2[j]) * rk[j] * dv[u] : 0.f;
            }
          }
        } else if (outs) {
          // lanes 64..127: the TMEM load is warp-wide (.sync.aligned), so every lane of these
          // quadrants issues it; only the qpad readout rows store
          const int qi = r - kChunk, pr = g.p0 + qi * M;
          const bool inq = qi < QP, live = qi < g.nq;
          const float gp = live ? G2[pr] : 0.f;
          const float sc = live ? p.scale * rq[qi] : 0.f;
          unsigned char *pb = sm + lay.P + (uint32_t)hf * (uint32_t)QP * 128u;  // K-block s / 32 = hf
#pragma unroll 1
          for (int c0 = cbeg; c0 < cbeg + 32; c0 += 16) {
            float dv[16];
            tmem_ld16(tW + lrow + c0, dv);
            if (inq) {
#pragma unroll
              for (int u4 = 0; u4 < 16; u4 += 4) {
                float4 o4;
                float *o = &o4.x;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int s_ = c0 + u4 + u;
                  o[u] = (live && s_ <= pr) ? sc * exp2f(gp - G2[s_]) * rk[s_] * dv[u4 + u] : 0.f;
                }
                *reinterpret_cast<float4 *>(pb + ImageLayout::swz_off(qi, c0 + u4)) = o4;
              }
            }
          }
        }
      }
      tc_fence_before();
      named_sync(kBarMath, kMathThreads);

      // ---- T = (I + A)^-1: 8x8 diagonal blocks by forward substitution, the 8x8 blocks below
      // them inside each 16x16 block, then the off-diagonal blocks by recursive doubling ----
      if (tid < kChunk) {
        const int b0 = (tid >> 3) * 8, cc = tid & 7;
        float t[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < i; ++j) acc += A[(b0 + i) * kLd + b0 + j] * t[j];
          t[i] = (i == cc) ? 1.f : (i < cc ? 0.f : -acc);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) Tm[(b0 + i) * kLdT + b0 + cc] = t[i];
      }
      named_sync(kBarMath, kMathThreads);
      {
        const int bb = tid >> 6, r = (tid >> 3) & 7, cc = tid & 7, r0 = 16 * bb + 8, c0 = 16 * bb;
        float acc = 0.f;
#pragma unroll
        for (int x = 0; x < 8; ++x) acc += A[(r0 + r) * kLd + c0 + x] * Tm[(c0 + x) * kLdT + c0 + cc];
        Yw[tid] = acc;
        named_sync(kBarMath, kMathThreads);
        float o = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) o += (m <= r ? Tm[(r0 + r) * kLdT + r0 + m] : 0.f) * Yw[(tid & ~63) + m * 8 + cc];
        Tm[(r0 + r) * kLdT + c0 + cc] = -o;
      }
      named_sync(kBarMath, kMathThreads);
      inverse_offdiag_math(A, Tm, Yw, warp, lane);

      // ---- T diag(beta gamma rk) and T diag(beta) as bf16 hi + lo over the dead A area ----
      {
        unsigned char *twh = sm + lay.R, *twl = twh + 8192u, *tuh = twh + 16384u, *tul = twh + 24576u;
        for (int it = tid; it < kChunk * 8; it += kMathThreads) {
          const int srow = it >> 3, j0 = (it & 7) * 8;
          const float4 t0 = *reinterpret_cast<const float4 *>(Tm + srow * kLdT + j0);
          const float4 t1 = *reinterpret_cast<const float4 *>(Tm + srow * kLdT + j0 + 4);
          const float t[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
          typename In::T2 wh[4], wlo[4], uh[4], ul[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float w0 = t[2 * i] * wc[j0 + 2 * i], w1 = t[2 * i + 1] * wc[j0 + 2 * i + 1];
            const float u0 = t[2 * i] * uc[j0 + 2 * i], u1 = t[2 * i + 1] * uc[j0 + 2 * i + 1];
            wh[i] = In::from_f2(w0, w1);
            uh[i] = In::from_f2(u0, u1);
            const float2 fw = In::to_f2(wh[i]), fu = In::to_f2(uh[i]);
            wlo[i] = In::from_f2(w0 - fw.x, w1 - fw.y);
            ul[i] = In::from_f2(u0 - fu.x, u1 - fu.y);
          }
          const uint32_t off = swz(srow, j0 * 2u);
          *reinterpret_cast<uint4 *>(twh + off) = *reinterpret_cast<const uint4 *>(wh);
          *reinterpret_cast<uint4 *>(twl + off) = *reinterpret_cast<const uint4 *>(wlo);
          *reinterpret_cast<uint4 *>(tuh + off) = *reinterpret_cast<const uint4 *>(uh);
          *reinterpret_cast<uint4 *>(tul + off) = *reinterpret_cast<const uint4 *>(ul);
        }
      }
      fence_async_smem();
      named_sync(kBarMath, kMathThreads);
      if (tid == 0) mbar_arrive(&wu_go);  // W^T and U^T (into Y of buffer b)

      // ---- the scan operands of chunk c: once W^T is in TMEM and the previous chunk's batch 2
      // has read b1 / b2 and left S_hat final ----
      if (!wait1(&wu_done, (uint32_t)(c & 1))) break;
      if (c >= 1 && !wait1(&b2_done[(c - 1) & 1], (uint32_t)(((c - 1) >> 1) & 1))) break;
      const bool emit = emits(c);
      if (emit && n_emit >= 1 && !wait1(&bk_free, (uint32_t)((n_emit - 1) & 1))) break;
      tc_fence_after();
      if (renorm || emit) {  // y = Gamma S_hat = S: the renormalised state and / or the snapshot
#pragma unroll 1
        for (int c0 = hf * 64; c0 < hf * 64 + 64; c0 += 32) {
          float x[32];
          tmem_ld32x(tS + lrow + c0, x);
#pragma unroll
          for (int w = 0; w < 32; ++w) x[w] *= gam;
          if (renorm) tmem_st32x(tS + lrow + c0, x);
          if (emit) tmem_st32x(tBk + lrow + c0, x);
        }
        tmem_st_wait();
      }
      {
        // b2: Ktil^T / Gamma' rows (row f = this thread's feature, columns s of this half)
        const float c2 = fast ? 1.f / gam_next : 1.f;
        const int f = v;
        unsigned char *row = sm + lay.b2 + (uint32_t)hf * lay.b2_block + (uint32_t)(f >> 3) * 1024u +
                             (uint32_t)(f & 7) * 128u;
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
          const int s0 = hf * 32 + 4 * j;
          float4 o4;
          o4.x = in_at<false>(kq, 128, s0, f) * ks[s0] * c2;
          o4.y = in_at<false>(kq, 128, s0 + 1, f) * ks[s0 + 1] * c2;
          o4.z = in_at<false>(kq, 128, s0 + 2, f) * ks[s0 + 2] * c2;
          o4.w = in_at<false>(kq, 128, s0 + 3, f) * ks[s0 + 3] * c2;
          *reinterpret_cast<float4 *>(row + ((j ^ (f & 7)) << 4)) = o4;
        }
        // b2: P rows (same in-row swizzle: 128 + qi and qi agree mod 8)
        const uint32_t pchunks = outs ? (uint32_t)QP * 8u : 0u;
        for (uint32_t idx = tid; idx < 2u * pchunks; idx += kMathThreads) {
          const uint32_t kb = idx / pchunks, rem = idx % pchunks;
          *reinterpret_cast<uint4 *>(sm + lay.b2 + kb * lay.b2_block + (uint32_t)d * 128u + rem * 16u) =
              *reinterpret_cast<const uint4 *>(sm + lay.P + kb * (uint32_t)QP * 128u + rem * 16u);
        }
        // b1: -Gamma W rows (W^T in TMEM: lane f, columns s) and Gamma Qh rows
        unsigned char *b1 = sm + lay.b1 + (uint32_t)q4 * lay.b1_block;  // K-block f / 32 = q4
        {
          float w[32];
          tmem_ld32x(tW + lrow + hf * 32, w);
#pragma unroll 8
          for (int u = 0; u < 32; ++u)
            *reinterpret_cast<float *>(b1 + ImageLayout::swz_off(QP + hf * 32 + u, f)) = -gam_pass * w[u];
        }
        const int qh = outs ? QP / 2 : 0;
#pragma unroll 4
        for (int qi = hf * qh; qi < hf * qh + qh; ++qi)
          *reinterpret_cast<float *>(b1 + ImageLayout::swz_off(qi, f)) =
              gam_pass * qs[qi] * in_at<false>(kq, 128, 64 + qi, f);
      }
      fence_async_smem();
      tc_fence_before();
      named_sync(kBarMath, kMathThreads);
      if (tid == 0) {
        slow_sh[b] = fast ? 0 : 1;
        if (c == n - 1) gam_fin_sh = gam_next;
        mbar_arrive(&ops_ready);
        if (c + 1 < n) issue_tiles(c + 1);  // every read of this chunk's tiles is done
      }
      if (emit) ++n_emit;
      if (!fast) {  // a slow chunk: S_hat <- gamma_last S_hat between its two batches
        if (!wait1(&b1_done[b], (uint32_t)((c >> 1) & 1))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = hf * 64; c0 < hf * 64 + 64; c0 += 32) {
          float x[32];
          tmem_ld32x(tS + lrow + c0, x);
#pragma unroll
          for (int w = 0; w < 32; ++w) x[w] *= gamma_last;
          tmem_st32x(tS + lrow + c0, x);
        }
        tmem_st_wait();
        tc_fence_before();
        named_sync(kBarMath, kMathThreads);
        if (tid == 0) mbar_arrive(&mid_go);
        ++n_slow;
      }
      gam = gam_next;
    }
    tmem_st_wait();
  } else if (warp < 12) {
    // ================================ store warps ================================
    bool pending = false;  // this warp's staging tile has a TMA store that may still read it
    unsigned char *tile = sm + lay.st + (uint32_t)q4 * kStTile;
    unsigned char *obuf = sm + lay.obuf;
    const int cpr = d / 8;  // 16-byte chunks per output row
    for (int64_t c = 0; c < n; ++c) {
      const int b = (int)(c & 1);
      const bool ok = mbar_wait_or_abort(&b2_done[b], (uint32_t)((c >> 1) & 1), &abort_flag, wl);
      if (lane == 0) st_ok[q4] = ok ? 1 : 0;
      if (tid == 256) bulk_wait_read<0>();  // the previous output TMA store has read the staging
      named_sync(kBarStore, 128);
      if (!(st_ok[0] & st_ok[1] & st_ok[2] & st_ok[3])) break;
      tc_fence_after();
      const ChunkGeo g = chunk_geo(bos, L, M, e0 + c);
      const int nqo = outs ? g.nq : 0;
#pragma unroll 1
      for (int q0 = 0; q0 < nqo; q0 += 32) {
        uint32_t xo[32];
        tmem_ld16_nw(tO(b) + lrow + q0, xo);
        if (q0 + 16 < nqo) tmem_ld16_nw(tO(b) + lrow + q0 + 16, xo + 16);
        tmem_ld_wait();
#pragma unroll
        for (int w = 0; w < 32; ++w)
          if (q0 + w < nqo)
            *reinterpret_cast<__nv_bfloat16 *>(obuf + ((uint32_t)(q0 + w) * d + v) * 2u) =
                __float2bfloat16_rn(__uint_as_float(xo[w]));
      }
      if (outs) {  // the buffer's o columns start the chunk after next at zero
        float z[16];
#pragma unroll
        for (int w = 0; w < 16; ++w) z[w] = 0.f;
        for (int c0 = 0; c0 < QP; c0 += 16) tmem_st16(tO(b) + lrow + c0, z);
        tmem_st_wait();
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&yo_free[b]);
      named_sync(kBarStore, 128);
      if (!outs) {
      } else if (p.out_tma && (g.nq == kChunk / M || g.nq == (kChunk + M - 1) / M)) {
        if (tid == 256) {
          tma_store_3d(g.nq == kChunk / M ? &tm_out_a : &tm_out_b, obuf, 0, h, (int)g.tq0);
          bulk_commit();
        }
      } else {
        for (int cidx = tid - 256; cidx < g.nq * cpr; cidx += 128) {
          const int qi = cidx / cpr, ch = cidx % cpr;
          *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + ((g.tq0 + qi) * H + h) * (int64_t)d + ch * 8) =
              *reinterpret_cast<const uint4 *>(obuf + ((uint32_t)qi * d + ch * 8) * 2u);
        }
      }
      if (emits(c))  // the math warps copied S_c before batch 2 of this chunk was issued
        store_state_one_tile(tBk + lrow, tile, lane, 1.f, &tm_cs,
                             (int)(((co_i + (e0 + c) / M) * H + h) * d + q4 * 32), pending, &bk_free);
    }
    if (seq_ok && !abort_flag) {  // the last chunk's b2_done was waited for above
      int64_t r = -1;
      const CUtensorMap *tm = &tm_fin;
      if (pass1) {  // B or Phi of the piece
        r = ((int64_t)blockIdx.x * H + h) * d;
        tm = &tm_seg;
      } else if (!last_piece) {  // a split piece leaves no state
      } else if (p.cache) {
        if (slot >= 0) r = ((int64_t)slot * H + h) * d;
      } else if (p.out_state) {
        r = ((int64_t)seq * H + h) * d;
      }
      if (r >= 0) store_state_one_tile(tS + lrow, tile, lane, gam_fin_sh, tm, (int)(r + q4 * 32), pending, nullptr);
    }
    if (lane == 0) bulk_wait_all();
  } else if (lane == 0) {
    // ================================ control thread ================================
    const uint32_t gram_id = idesc(kFmtBF16, 0, 0, 64, 128);
    const uint32_t wu_id = idesc(kFmtBF16, 1, 0, 64, d);
    const uint32_t id1 = idesc(kFmtTF32, 0, 0, QP + 64, 128);
    const uint32_t id1y = idesc(kFmtTF32, 0, 0, 64, 128);  // Y only (no outputs)
    const uint32_t id2s = idesc(kFmtTF32, 0, 0, d, 128);
    const uint32_t id2o = idesc(kFmtTF32, 0, 0, QP, 128);
    const uint32_t skq = smem_u32(kq), svt = smem_u32(vt);
    const uint32_t sb1 = smem_u32(sm + lay.b1), sb2 = smem_u32(sm + lay.b2);
    const uint32_t stw = smem_u32(sm + lay.R);
    auto gram = [&]() {
      for (int kk = 0; kk < d / 16; ++kk) {
        const uint32_t a = skq + (kk >> 2) * 16384u + (kk & 3) * 32u;
        mma_bf16_ss(tW, desc_sw128(a, 16, 1024), desc_sw128(a, 16, 1024), gram_id, kk > 0);
      }
      mma_commit(&gram_done);
    };
    int n_mid = 0;
    for (int64_t c = 0; c < n; ++c) {
      const int b = (int)(c & 1);
      if (c == 0) {
        if (!mbar_wait_or_abort(&gram_go, 0, &abort_flag, wl)) break;
        tc_fence_after();
        gram();
      }
      // W^T = K^T (T diag(beta gamma rk))^T -> tW; U^T = V^T (T diag(beta))^T -> Y of buffer b
      if (!mbar_wait_or_abort(&wu_go, (uint32_t)(c & 1), &abort_flag, wl)) break;
      tc_fence_after();
      const uint32_t ty = tO(b) + (uint32_t)QP;
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t dak = desc_sw128(skq + kk * 2048u, 16384, 1024), dav = desc_sw128(svt + kk * 2048u, 8192, 1024);
        mma_bf16_ss(tW, dak, desc_sw128(stw + kk * 32u, 16, 1024), wu_id, kk > 0);
        mma_bf16_ss(tW, dak, desc_sw128(stw + 8192u + kk * 32u, 16, 1024), wu_id, 1);
        mma_bf16_ss(ty, dav, desc_sw128(stw + 16384u + kk * 32u, 16, 1024), wu_id, kk > 0);
        mma_bf16_ss(ty, dav, desc_sw128(stw + 24576u + kk * 32u, 16, 1024), wu_id, 1);
      }
      mma_commit(&wu_done);
      // batch 1: [o | Y] += S_hat [Gamma Qh ; -Gamma W]^T
      if (!mbar_wait_or_abort(&ops_ready, (uint32_t)(c & 1), &abort_flag, wl)) break;
      if (c >= 2 && !mbar_wait_or_abort(&yo_free[b], (uint32_t)(((c >> 1) - 1) & 1), &abort_flag, wl)) break;
      tc_fence_after();
      const bool slow = slow_sh[b] != 0;
      if (outs) {
        for (int kk = 0; kk < d / 8; ++kk)
          mma_tf32_ts(tO(b), tS + kk * 8, desc_sw128(sb1 + (kk >> 2) * lay.b1_block + (kk & 3) * 32u, 16, 1024), id1,
                      1);
      } else {  // the -W rows only: they start qpad rows (whole 1024-byte atoms) into each K-block
        for (int kk = 0; kk < d / 8; ++kk)
          mma_tf32_ts(ty, tS + kk * 8,
                      desc_sw128(sb1 + (kk >> 2) * lay.b1_block + (uint32_t)QP * 128u + (kk & 3) * 32u, 16, 1024),
                      id1y, 1);
      }
      mma_commit(&b1_done[b]);
      // the next chunk's Gram runs between the batches (the math warps need it first)
      if (c + 1 < n) {
        if (!mbar_wait_or_abort(&gram_go, (uint32_t)((c + 1) & 1), &abort_flag, wl)) break;
        tc_fence_after();
        gram();
      }
      if (slow) {
        if (!mbar_wait_or_abort(&mid_go, (uint32_t)(n_mid & 1), &abort_flag, wl)) break;
        ++n_mid;
        tc_fence_after();
      }
      // batch 2: S_hat += Y (Ktil / Gamma')^T, o += Y P^T
      for (int kk = 0; kk < kChunk / 8; ++kk) {
        const uint32_t bk = sb2 + (kk >> 2) * lay.b2_block + (kk & 3) * 32u;
        mma_tf32_ts(tS, ty + kk * 8, desc_sw128(bk, 16, 1024), id2s, 1);
        if (outs) mma_tf32_ts(tO(b), ty + kk * 8, desc_sw128(bk + (uint32_t)d * 128u, 16, 1024), id2o, 1);
      }
      mma_commit(&b2_done[b]);
    }
    if (abort_flag) {
      // drain every MMA issued so far before the columns are freed
      mma_commit(&fin_bar);
      mbar_wait(&fin_bar, 0);
      set_status(p.status, GDP_DEV_ERR_TIMEOUT);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && load_pending) mbar_wait(&tl_full, (uint32_t)((n_loads - 1) & 1));  // (abort) the last load landed
  __syncthreads();
  if (warp == 12) tmem_free(tb, 512);
}

__global__ void __launch_bounds__(kFusedThreads, 1)
    gdp_fused_kernel(Problem p, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_cs,
                     const __grid_constant__ CUtensorMap tm_fin, const __grid_constant__ CUtensorMap tm_seg,
                     const __grid_constant__ CUtensorMap tm_out_a, const __grid_constant__ CUtensorMap tm_out_b) {
  fused_body(p, tm_k, tm_q, tm_v, tm_cs, tm_fin, tm_seg, tm_out_a, tm_out_b);
}

}  // namespace

bool fused_shape(int K, int V, int M) { return K == kFusedD && V == kFusedD && fused_tmem_fits(qpad_for(M)); }

bool fused_serves(const Problem &p) {
  return fused_shape(p.K, p.V, p.M) && !p.f16 && p.g_type == kTypeF32 && !p.g_alpha && p.beta_type == kTypeF32 &&
         !(p.init && p.init_bf16 && !p.cache);
}

size_t fused_smem_bytes(int qpad) { return (size_t)FusedLayout(qpad).total + 1024u; }

cudaError_t launch_fused(const Problem &p, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  const size_t smem = fused_smem_bytes(p.qpad);
  cudaError_t e = cudaFuncSetAttribute(gdp_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap tm_k, tm_q, tm_v, tm_cs, tm_fin, tm_seg, tm_out_a, tm_out_b;
  const int64_t rows = p.T * p.M;
  if ((e = tmap_rows_16(&tm_k, p.k, rows, p.Hk, p.K, p.k_st, p.k_sh, kChunk, 0)) != cudaSuccess) return e;
  if ((e = tmap_rows_16(&tm_q, p.q, p.T, p.Hq, p.K, p.q_st, p.q_sh, p.qpad, 0)) != cudaSuccess) return e;
  if ((e = tmap_rows_16(&tm_v, p.v, rows, p.Hv, p.V, p.v_st, p.v_sh, kChunk, 0)) != cudaSuccess) return e;
  const int64_t hv = (int64_t)p.H * p.V;
  if ((e = tmap_state(&tm_cs, p.chunk_states, p.nt_pad * hv, p.K)) != cudaSuccess) return e;
  if (p.cache)
    e = tmap_state(&tm_fin, p.cache, p.num_slots * hv, p.K);
  else
    e = tmap_state(&tm_fin, p.out_state, p.N * hv, p.K);
  if (e != cudaSuccess) return e;
  // the pieces' states (pass 1 writes B and Phi through it)
  if ((e = tmap_state(&tm_seg, p.piece_len > 0 ? p.piece_buf : nullptr, 3 * (int64_t)p.piece_rows * hv, p.K)) !=
      cudaSuccess)
    return e;
  Problem q = p;
  const int na = kChunk / p.M, nb = (kChunk + p.M - 1) / p.M;
  q.out_tma = (p.out && p.T >= nb) ? 1 : 0;
  if ((e = tmap_out_rows(&tm_out_a, q.out_tma ? p.out : nullptr, p.T, p.H, p.V, na, 0)) != cudaSuccess) return e;
  if ((e = tmap_out_rows(&tm_out_b, q.out_tma ? p.out : nullptr, p.T, p.H, p.V, nb, 0)) != cudaSuccess) return e;
  // one CTA per (sequence, head), or per (piece row, head) -- pass 1 runs two per piece
  const int64_t grid_rows = p.piece_len > 0 ? (p.piece_pass1 ? 2 : 1) * (int64_t)p.piece_rows : p.N;
  dim3 grid((unsigned)grid_rows, (unsigned)p.H);
  if ((e = launch_kernel(gdp_fused_kernel, grid, dim3(kFusedThreads), smem, stream, p.pdl != 0, q, tm_k, tm_q, tm_v,
                         tm_cs, tm_fin, tm_seg, tm_out_a, tm_out_b)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace gdp
