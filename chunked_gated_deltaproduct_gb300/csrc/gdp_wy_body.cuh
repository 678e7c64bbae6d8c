// gdp_wy_body.cuh -- per-(expanded chunk, head) prep + WY kernel on the tcgen05 tensor cores.
//
// Megatron-Core API page "core.ssm.ops.gdp.chunk", stages 1 and 2:
//   stage 1: the log decay of token t is placed on its first expanded row
//            t*M (interleave), the within-chunk cumulative sum is taken on the
//            expanded stream and converted to base 2 (exp2 everywhere); q and k
//            are optionally L2-normalised (FlashInfer page,
//            use_qk_l2norm_in_kernel) -- applied as per-row scale factors;
//   stage 2: A = beta K K^T (strictly lower, decay-weighted), T = (I + A)^-1,
//            then the w and u factors.
// With gamma_r = 2^G2_r, khat = rk k (rk = 1 / |k| or 1):
//   A[i][j] = beta_i 2^(G2_i - G2_j) (khat_i . khat_j)        (i > j)
//   W = T diag(beta gamma) Khat,   U = T diag(beta) V
// so that inside the chunk the new values are V_new = U - W S0^T for the
// entering state S0 (derived from the recurrence on the FlashInfer page,
// display equation).  The kernel also forms what the output stage needs:
//   P[q][s] = scale 2^(G2_p - G2_s) (qhat_t . khat_s)   for s <= p  (p = t*M + M - 1)
//   Qh[q]   = scale 2^(G2_p) qhat_t,    Kt[s] = 2^(G2_last - G2_s) khat_s.
// When 2^G2_last >= 2^kFastMinLog2Gamma, W and Qh are written divided by
// 2^G2_last (the scan keeps its state divided by a running decay product).
// Every exponent is of a difference G2_i - G2_j with i >= j (or of a partial
// sum <= 0), so no factor exceeds 1.
//
// Tensor-core work (cta_group::1, fp32 accumulators in TMEM):
//   [K; Q] K^T  : kind::f16, M = 128 (64 key rows + up to 64 query rows), N = 64, K = d
//   W^T = K^T (T diag(beta gamma rk))^T, U^T = V^T (T diag(beta))^T : kind::f16,
//                 M = d, N = 64, K = 64, with T split as hi + lo of the input type (two
//                 MMAs each) so that T keeps ~16 (bf16) or ~22 (f16) significant bits.
// The inputs q, k, v are bfloat16 or float16 (FlashInfer page, parameters q, k, v); the
// kernel is instantiated per type, since both operands of one MMA share it.  float16 has
// a narrow exponent range, so for it the two T factors are scaled by a power of two that
// brings their largest entry to about 2^14 before the split, and the products are scaled
// back in fp32 (exact).
// Grouped heads: state head h reads head h / (H / Hx) of q, k and v (x = q, k, v).
// The inverse of the unit lower-triangular I + A runs in 16 x 16 blocks: the four
// diagonal blocks by forward substitution on the CUDA cores (one warp each), then
// the blocks below the diagonal by recursive doubling (T_21 = -T_22 A_21 T_11 on 16- then
// 32-row blocks), with warp-level tf32 MMAs in the 3xTF32 split (fp32-level accuracy; these
// 16 x 16 and 32 x 32 products are far below the tcgen05 tile size).
#pragma once
#include <cuda.h>  // CUtensorMap

#include "gdp_internal.cuh"
#include "gdp_sm100.cuh"

namespace gdp {
namespace {

using namespace sm100;

constexpr int kWyThreads = 256;  // 8 warps: two per TMEM lane quadrant, splitting the columns
constexpr int kWyCtasPerSm = 3;   // shared memory (~68 KB), TMEM (128 columns) and 80 registers each
constexpr int kLd = kChunk + 1;   // row stride of an fp32 [64][65] scratch (conflict-free row reads)
constexpr int kLdT = kChunk + 4;  // row stride of A / T (16-byte aligned rows for float4 access)
constexpr int kLdY = 36;          // row stride of the [32][32] block-product scratch

// Shared memory of one tile, small enough for three CTAs per SM.  Lifetimes: the query rows of
// kq die with the [K;Q]K^T epilogue and then hold the inverse's block products (Y) and, after
// the inverse, the hi and lo tiles of one T split at a time (W's, then U's once W's MMAs have
// read them); T is computed in place over A (A strictly lower, T unit lower: the zeros above
// the diagonal serve both).
struct WyLayout {
  uint32_t kq, vt, th, tl, Y, A, scal, total;
  __host__ __device__ WyLayout(int d) {
    const uint32_t nb = (uint32_t)d / 64;  // 64-element (128-byte) K blocks of a 16-bit row
    kq = 0;                                // [nb][128 rows][128 B]: rows 0..63 k, 64..127 q
    vt = kq + nb * 16384u;                 // [nb][64 rows][128 B]
    th = kq + 8192u;                       // the query rows of K block 0
    Y = th;                                // fp32 [32][36] block products (during the inverse)
    if (d == 128) {
      tl = kq + 16384u + 8192u;            // the query rows of K block 1
      A = vt + nb * 8192u;
    } else {
      tl = vt + nb * 8192u;
      A = tl + 8192u;
    }
    scal = A + 4u * kChunk * kLdT;         // A / T: fp32 [64][68]
    total = scal + 4u * 9 * kChunk;        // G2, beta, rk, rq, wc, uc, kscale [7][64]; [128] norms
  }
};

// 3xTF32 warp-level products for the 16 x 16 blocks of the inverse: x = hi + lo with hi, lo
// tf32 (round to nearest), and hi*hi + hi*lo + lo*hi keeps ~fp32 accuracy (lo*lo dropped).
__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void tf32_split(float x, uint32_t &hi, uint32_t &lo) {
  hi = tf32_rna(x);
  lo = tf32_rna(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_m16n8k8_tf32(float *c, const uint32_t *a, const uint32_t *b) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// c += X (16 x 8, row stride lx) * Z (8 x 8, row stride lz) with the fragment layout of
// m16n8k8 (lane = 4 g + t): X rows g, g+8 and columns t, t+4; Z rows t, t+4 and column g.
__device__ __forceinline__ void mma3_16x8x8(float *c, const float *X, int lx, const float *Z, int lz, int lane) {
  const int g = lane >> 2, t = lane & 3;
  uint32_t ah[4], al[4], bh[2], bl[2];
  tf32_split(X[g * lx + t], ah[0], al[0]);
  tf32_split(X[(g + 8) * lx + t], ah[1], al[1]);
  tf32_split(X[g * lx + t + 4], ah[2], al[2]);
  tf32_split(X[(g + 8) * lx + t + 4], ah[3], al[3]);
  tf32_split(Z[t * lz + g], bh[0], bl[0]);
  tf32_split(Z[(t + 4) * lz + g], bh[1], bl[1]);
  mma_m16n8k8_tf32(c, al, bh);
  mma_m16n8k8_tf32(c, ah, bl);
  mma_m16n8k8_tf32(c, ah, bh);
}

// Off-diagonal blocks of T = (I + A)^-1 by recursive doubling, given the inverted 16x16
// diagonal blocks: first T_10 and T_32 of the two 32x32 diagonal blocks,
// T_i,i-1 = -T_ii (A_i,i-1 T_i-1,i-1); then the 32x32 block below the diagonal,
// T_[23][01] = -T_[23][23] (A_[23][01] T_[01][01]).  Each product is split into 16x8 units,
// one per warp, computed with warp-level tf32 MMAs (3xTF32); Y holds the inner products.
// A and Tm may be the same array (row stride kLdT): a block of A is read only before the
// barrier after which its T block is written, and no later step reads it.
__device__ __forceinline__ void inverse_offdiag(const float *A, float *Tm, float *Y, int warp, int lane) {
  const int g = lane >> 2, t = lane & 3;
  // level 1: units (pair p, 8-column half nh): rows 16 i, columns 16 j, i = 2 p + 1, j = 2 p
  if (warp < 4) {
    const int pr = warp >> 1, nh = warp & 1, i = 2 * pr + 1, j = 2 * pr;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ks = 0; ks < 2; ++ks)
      mma3_16x8x8(c, A + (16 * i) * kLdT + 16 * j + 8 * ks, kLdT, Tm + (16 * j + 8 * ks) * kLdT + 16 * j + 8 * nh,
                  kLdT, lane);
    float *y = Y + (pr * 16) * kLdY + 8 * nh;
    y[g * kLdY + 2 * t] = c[0];
    y[g * kLdY + 2 * t + 1] = c[1];
    y[(g + 8) * kLdY + 2 * t] = c[2];
    y[(g + 8) * kLdY + 2 * t + 1] = c[3];
  }
  __syncthreads();
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
  __syncthreads();
  // level 2: 8 units (16-row tile mt, 8-column tile nt) of the 32x32 block, K = 32
  const int mt = warp >> 2, nt = warp & 3;
  {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ks = 0; ks < 4; ++ks)
      mma3_16x8x8(c, A + (32 + 16 * mt) * kLdT + 8 * ks, kLdT, Tm + (8 * ks) * kLdT + 8 * nt, kLdT, lane);
    float *y = Y + (16 * mt) * kLdY + 8 * nt;
    y[g * kLdY + 2 * t] = c[0];
    y[g * kLdY + 2 * t + 1] = c[1];
    y[(g + 8) * kLdY + 2 * t] = c[2];
    y[(g + 8) * kLdY + 2 * t + 1] = c[3];
  }
  __syncthreads();
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
  __syncthreads();
}

// The 16-bit input type: bfloat16, or float16 when F16.
template <bool F16> struct In16;
template <> struct In16<false> {
  using T = __nv_bfloat16;
  using T2 = __nv_bfloat162;
  static constexpr int kFmt = kFmtBF16;
  static __device__ __forceinline__ float to_f(T x) { return __bfloat162float(x); }
  static __device__ __forceinline__ float2 to_f2(T2 x) { return __bfloat1622float2(x); }
  static __device__ __forceinline__ T2 from_f2(float a, float b) { return __floats2bfloat162_rn(a, b); }
};
template <> struct In16<true> {
  using T = __half;
  using T2 = __half2;
  static constexpr int kFmt = kFmtF16;
  static __device__ __forceinline__ float to_f(T x) { return __half2float(x); }
  static __device__ __forceinline__ float2 to_f2(T2 x) { return __half22float2(x); }
  static __device__ __forceinline__ T2 from_f2(float a, float b) { return __floats2half2_rn(a, b); }
};

template <bool F16>
__device__ __forceinline__ float in_at(const unsigned char *tile, int rows_per_block, int r, int f) {
  const uint32_t off = (uint32_t)(f >> 6) * rows_per_block * 128u + swz(r, (uint32_t)(f & 63) * 2u);
  return In16<F16>::to_f(*reinterpret_cast<const typename In16<F16>::T *>(tile + off));
}
// Eight consecutive elements f0 .. f0+7 (f0 % 8 == 0) of row r as floats, one 16-byte load.
template <bool F16>
__device__ __forceinline__ void in8_at(const unsigned char *tile, int rows_per_block, int r, int f0, float *o) {
  const uint32_t off = (uint32_t)(f0 >> 6) * rows_per_block * 128u + swz(r, (uint32_t)(f0 & 63) * 2u);
  const uint4 x = *reinterpret_cast<const uint4 *>(tile + off);
  const typename In16<F16>::T2 *b = reinterpret_cast<const typename In16<F16>::T2 *>(&x);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f2 = In16<F16>::to_f2(b[i]);
    o[2 * i] = f2.x;
    o[2 * i + 1] = f2.y;
  }
}

// Power of two s with (largest |entry|) * s below 2^14, from the largest |entry| m (1 when
// m is 0); the exponent is clamped so that s and 1 / s stay finite.
__device__ __forceinline__ float f16_split_scale(float m, float *inv) {
  int ex = 0;
  if (m > 0.f) frexpf(m, &ex);  // m < 2^ex
  ex = max(-100, min(ex, 100));
  *inv = ldexpf(1.f, ex - 14);
  return ldexpf(1.f, 14 - ex);
}

// The kernel body.  F16: q, k, v are float16 (else bfloat16).  TYPED: g and beta may be
// 16-bit and g may hold alpha itself (else fp32 beta and natural-log g).  Compile-time, so that
// the common kernel carries no code for the other types.
template <bool F16, bool TYPED>
__device__ __forceinline__ void wy_body(const Problem &p, const CUtensorMap &tm_k, const CUtensorMap &tm_q,
                                        const CUtensorMap &tm_v) {
  using In = In16<F16>;
  pdl_wait();     // the descriptors (and, in a segmented call, nothing else) come from the kernel before
  pdl_trigger();  // the scan may start launching: it waits for this grid before reading its tiles
  const int h = blockIdx.y;
  const int hq = input_head(h, p.hmul_q), hk = input_head(h, p.hmul_k), hv = input_head(h, p.hmul_v);
  int row, seq, c;
  if (p.seg_rows > 0) {  // a segment: tile (sequence, chunk seg_lo + x % seg_rows)
    seq = blockIdx.x / p.seg_rows;
    c = (int)(p.seg_lo + blockIdx.x % p.seg_rows);
    if (seq >= p.N) return;
    row = p.cod[seq] + c;
  } else {
    row = blockIdx.x;
    if (!in_range(p.bounds, p.status, GDP_BOUNDS_SITE_WY_TILE, 2 * (int64_t)row + 1, 2 * p.ntdp_pad)) return;
    seq = p.cid[2 * row];
    c = p.cid[2 * row + 1];
  }
  if (seq < 0 || seq >= p.N || row < 0 || row >= p.ws_rows) return;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;
  if (c < 0 || L <= 0 || (int64_t)c * kChunk >= L * p.M) return;
  const int M = p.M, d = p.K, QP = p.qpad;
  const int64_t R0 = bos * M + (int64_t)c * kChunk;  // first global expanded row
  const int len = (int)min((int64_t)kChunk, L * M - (int64_t)c * kChunk);
  const int r0m = (int)(R0 % M);                 // expanded-row phase of the chunk start
  const int64_t tok0 = (R0 - r0m) / M;           // token of row 0
  const int p0 = (M - 1 - r0m) % M;              // first readout row (t*M + M - 1)
  const int nq = (p0 < len) ? (len - 1 - p0) / M + 1 : 0;
  const int64_t tq0 = (R0 + p0) / M;             // token of the first readout row; readout qi is tq0 + qi
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, chalf = warp >> 2;  // TMEM lane quadrant, column half of this warp

  extern __shared__ __align__(1024) unsigned char wy_smem_raw[];
  // the 1024-aligned base as an offset into the shared array, so that accesses stay in the shared
  // address space
  unsigned char *sm = wy_smem_raw + ((1024u - (sm100::smem_u32(wy_smem_raw) & 1023u)) & 1023u);
  const WyLayout lay(d);
  unsigned char *kq = sm + lay.kq, *vt = sm + lay.vt;
  float *A = reinterpret_cast<float *>(sm + lay.A);
  float *Tm = A;  // T = (I + A)^-1 replaces A in place
  float *Y = reinterpret_cast<float *>(sm + lay.Y);
  float *G2 = reinterpret_cast<float *>(sm + lay.scal);
  float *bt = G2 + kChunk, *rk = bt + kChunk, *rq = rk + kChunk, *wc = rq + kChunk, *uc = wc + kChunk;
  float *ks = uc + kChunk;  // 2^(G2_last - G2_s) rk_s (0 past the chunk end)
  float *l2s = ks + kChunk;  // [128] partial squared norms of the key and query rows
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t mma_bar, ld_bar;
  __shared__ float warp_tot;
  __shared__ int abort_flag;

  if (warp == 0) tmem_alloc(&tmem_slot, 128);
  if (tid == 0) {
    mbar_init(&mma_bar, 1);
    mbar_init(&ld_bar, 1);
    mbar_init_fence();
    abort_flag = 0;
  }
  __syncthreads();

  // ---- loads: TMA boxes of 64 features x rows into the swizzled 16-bit tiles: k rows R0.., the
  // readout q rows tq0.. (rows 64.. of kq), v rows R0..; rows past the chunk (another sequence's
  // data, or zero past the tensor) are cleared below so that sequences stay independent ----
  const int nb = d / 64;
  if (tid == 0) {
    mbar_arrive_expect_tx(&ld_bar, (uint32_t)nb * (uint32_t)(64 + QP + 64) * 128u);
    for (int kb = 0; kb < nb; ++kb) {
      tma_load_3d(kq + kb * 16384u, &tm_k, kb * 64, hk, (int)R0, &ld_bar);
      tma_load_3d(kq + kb * 16384u + 8192u, &tm_q, kb * 64, hq, (int)tq0, &ld_bar);
      tma_load_3d(vt + kb * 8192u, &tm_v, kb * 64, hv, (int)R0, &ld_bar);
    }
  }
  // per-row beta and decay gate (the decay of token t sits on its first expanded row t*M),
  // fetched while the tiles land
  float b_r = 0.f, gate_r = 0.f;
  if (tid < kChunk && tid < len &&
      in_range(p.bounds, p.status, GDP_BOUNDS_SITE_WY_SCALARS, (R0 + tid) * p.H + h, p.T * M * p.H) &&
      in_range(p.bounds, p.status, GDP_BOUNDS_SITE_WY_SCALARS, (tok0 + (r0m + tid) / M) * p.H + h, p.T * p.H)) {
    const int pos = r0m + tid;
    if constexpr (TYPED) {
      b_r = p.beta ? load_typed(p.beta, (R0 + tid) * p.H + h, p.beta_type) : 1.f;
      if (p.g && pos % M == 0) gate_r = load_log_gate(p, (tok0 + pos / M) * p.H + h);
    } else {
      b_r = p.beta ? static_cast<const float *>(p.beta)[(R0 + tid) * p.H + h] : 1.f;
      if (p.g && pos % M == 0) gate_r = static_cast<const float *>(p.g)[(tok0 + pos / M) * p.H + h];
    }
  }
  if (!mbar_wait(&ld_bar, 0)) abort_flag = 1;
  {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const int nk = kChunk - len, nqz = QP - nq;  // rows to clear
    for (int idx = tid; idx < nb * (2 * nk + nqz) * 8; idx += kWyThreads) {
      const int ch = idx & 7, rr = idx >> 3, kb = rr % nb, r = rr / nb;
      unsigned char *row = (r < nk) ? kq + kb * 16384u + (uint32_t)(len + r) * 128u
                           : (r < 2 * nk) ? vt + kb * 8192u + (uint32_t)(len + r - nk) * 128u
                                          : kq + kb * 16384u + (uint32_t)(64 + nq + r - 2 * nk) * 128u;
      *reinterpret_cast<uint4 *>(row + ch * 16) = z;
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  // [K;Q]K^T in columns 0..63 until its epilogue; then W^T there and U^T in 64..127
  const uint32_t tD1 = tbase, tW = tbase, tU = tbase + 64;

  // ---- [K; Q] K^T on the tensor cores (issued first, overlaps the scalar prologue) ----
  if (tid == 0) {
    const uint32_t id = idesc(In::kFmt, 0, 0, 64, 128);
    for (int kk = 0; kk < d / 16; ++kk) {
      const uint32_t a = smem_u32(kq) + (kk >> 2) * 16384u + (kk & 3) * 32u;
      mma_bf16_ss(tD1, desc_sw128(a, 16, 1024), desc_sw128(a, 16, 1024), id, kk > 0);
    }
    mma_commit(&mma_bar);
  }

  // ---- per-row scalars: beta, decay gate, inverse norms; base-2 cumsum ----
  {
    const int r = tid & 127;  // rows 0..63 keys, 64..127 query rows; threads 128.. take the upper features
    float ss = 0.f;
    if (p.l2norm) {
#pragma unroll 1
      for (int f0 = chalf * (d / 2); f0 < (chalf + 1) * (d / 2); f0 += 8) {
        float x[8];
        in8_at<F16>(kq, 128, r, f0, x);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += x[i] * x[i];
      }
      if (chalf) l2s[r] = ss;
      __syncthreads();
      if (!chalf) ss += l2s[r];
    }
    if (chalf) {
    } else if (r < kChunk) {
      const float gate = gate_r;
      bt[r] = b_r;
      rk[r] = p.l2norm ? rsqrtf(ss + kL2Eps) : 1.f;
      // inclusive scan of the gates over the 64 rows (two warps)
      float x = gate;
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
  __syncthreads();
  if (tid < kChunk) {
    const float x = (tid >= 32 ? G2[tid] + warp_tot : G2[tid]) * kLog2e;
    G2[tid] = x;
  }
  __syncthreads();
  // a fast image carries -W and Qh divided by the chunk decay 2^G2_last
  const float G2last = G2[len - 1];
  const bool fast = G2last >= kFastMinLog2Gamma;
  const float shift = fast ? G2last : 0.f;
  if (tid < kChunk) {
    wc[tid] = bt[tid] * exp2f(G2[tid] - shift) * rk[tid];
    uc[tid] = bt[tid];
    ks[tid] = (tid < len) ? exp2f(G2[len - 1] - G2[tid]) * rk[tid] : 0.f;
  }

  // ---- epilogue of [K;Q]K^T: A rows (lanes 0..63), score rows and query images (lanes 64..127) ----
  const bool ok1 = mbar_wait(&mma_bar, 0);
  if (!ok1) abort_flag = 1;
  tc_fence_after();
  __syncthreads();
  const ImageLayout il(d, QP);
  unsigned char *img = p.img + (size_t)((int64_t)row * p.H + h) * p.img_stride;
  // the backward's layout of the same operands (its forward recompute only)
  const BwdImageLayout bl(d, QP);
  unsigned char *bimg = p.bimg ? p.bimg + (size_t)((int64_t)row * p.H + h) * p.bimg_stride : nullptr;
  {
    // the TMEM row of this thread, this warp's half of the columns, in 16-column pieces
    const uint32_t taddr = tD1 + ((uint32_t)(quad * 32) << 16);
    const int r = quad * 32 + lane;
    const int cbeg = chalf * 32;
    if (r < kChunk) {
      const int i = r;
      const bool rowlive = i < len;
      const float gi = G2[i], si = bt[i] * rk[i];
#pragma unroll 1
      for (int c0 = cbeg; c0 < cbeg + 32; c0 += 16) {
        float dv[16];
        tmem_ld16(taddr + c0, dv);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int j = c0 + u;
          A[i * kLdT + j] = (j < i && rowlive) ? si * exp2f(gi - G2[j]) * rk[j] * dv[u] : 0.f;
        }
      }
    } else {
      const int qi = r - kChunk;
      const int pr = p0 + qi * M;
      const bool live = qi < nq;
      const float gp = live ? G2[pr] : 0.f;
      const float qscale = live ? p.scale * exp2f(gp - shift) * rq[qi] : 0.f;
      const float sc = live ? p.scale * rq[qi] : 0.f;
#pragma unroll 1
      for (int c0 = cbeg; c0 < cbeg + 32; c0 += 16) {
        float dv[16];
        tmem_ld16(taddr + c0, dv);
        if (qi < QP) {
#pragma unroll
          for (int u4 = 0; u4 < 16; u4 += 4) {
            float4 o4;
            float *o = &o4.x;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int s_ = c0 + u4 + u;
              o[u] = (live && s_ <= pr) ? sc * exp2f(gp - G2[s_]) * rk[s_] * dv[u4 + u] : 0.f;
            }
            *reinterpret_cast<float4 *>(img + il.pm(d, qi, c0 + u4)) = o4;
            if (bimg)  // P^T: row s, column qi (a row segment per warp instruction)
#pragma unroll
              for (int u = 0; u < 4; ++u) *reinterpret_cast<float *>(bimg + bl.p_at(c0 + u4 + u, qi)) = o[u];
          }
        }
      }
      if (qi < QP) {
#pragma unroll 1
        for (int f0 = chalf * (d / 2); f0 < (chalf + 1) * (d / 2); f0 += 8) {
          float x[8];
          in8_at<F16>(kq, 128, r, f0, x);
          *reinterpret_cast<float4 *>(img + il.qh(qi, f0)) =
              make_float4(qscale * x[0], qscale * x[1], qscale * x[2], qscale * x[3]);
          *reinterpret_cast<float4 *>(img + il.qh(qi, f0 + 4)) =
              make_float4(qscale * x[4], qscale * x[5], qscale * x[6], qscale * x[7]);
          if (bimg)  // Qh^T: row f, column qi
#pragma unroll
            for (int j = 0; j < 8; ++j) *reinterpret_cast<float *>(bimg + bl.q_at(f0 + j, qi)) = qscale * x[j];
        }
      }
    }
  }
  __syncthreads();

  // ---- T = (I + A)^-1 in place.  Diagonal 16x16 blocks from 8x8 halves: forward substitution
  // on the eight 8x8 diagonal blocks (a thread per column), then T_21 = -T_22 A_21 T_11 inside
  // each 16x16 block; every block above its block diagonal is zero in A and in T ----
  if (tid < kChunk) {
    const int b0 = (tid >> 3) * 8, cc = tid & 7;
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < i; ++j) acc += A[(b0 + i) * kLdT + b0 + j] * t[j];
      t[i] = (i == cc) ? 1.f : (i < cc ? 0.f : -acc);
    }
    __syncwarp();  // the block's eight threads (one warp) have read A's block before T replaces it
#pragma unroll
    for (int i = 0; i < 8; ++i) Tm[(b0 + i) * kLdT + b0 + cc] = t[i];
  }
  __syncthreads();
  {
    // thread: block b = tid / 64 (rows 16b+8.., columns 16b..), element (r, c) of the 8x8 block
    const int b = tid >> 6, r = (tid >> 3) & 7, cc = tid & 7, r0 = 16 * b + 8, c0 = 16 * b;
    float acc = 0.f;  // (A_21 T_11)[r][cc]
#pragma unroll
    for (int x = 0; x < 8; ++x) acc += A[(r0 + r) * kLdT + c0 + x] * Tm[(c0 + x) * kLdT + c0 + cc];
    Y[tid] = acc;
    __syncthreads();
    float o = 0.f;  // (T_22 Y)[r][cc], T_22 lower triangular
#pragma unroll
    for (int m = 0; m < 8; ++m) o += (m <= r ? Tm[(r0 + r) * kLdT + r0 + m] : 0.f) * Y[(tid & ~63) + m * 8 + cc];
    Tm[(r0 + r) * kLdT + c0 + cc] = -o;
  }
  __syncthreads();
  inverse_offdiag(A, Tm, Y, warp, lane);
  if (bimg)  // T itself for the backward's per-chunk gradients, dense [64][64]
    for (int idx = tid; idx < kChunk * kChunk / 4; idx += kWyThreads) {
      const int r = idx >> 4, c4 = (idx & 15) * 4;
      *reinterpret_cast<float4 *>(bimg + bl.tinv + (uint32_t)(r * kChunk + c4) * 4u) =
          *reinterpret_cast<const float4 *>(Tm + r * kLdT + c4);
    }

  // ---- T diag(beta gamma rk) and T diag(beta) as hi + lo of the input type, K-major swizzled
  // [64 s][64 j]; for float16 first scaled by sw, su (powers of two, see f16_split_scale) ----
  float sw = 1.f, su = 1.f, isw = 1.f, isu = 1.f;
  if constexpr (F16) {
    __shared__ float red[2][kWyThreads / 32];
    float mw = 0.f, mu = 0.f;
    for (int it = tid; it < kChunk * kChunk; it += kWyThreads) {
      const int srow = it >> 6, j = it & 63;
      const float t = fabsf(Tm[srow * kLdT + j]);
      mw = fmaxf(mw, t * fabsf(wc[j]));
      mu = fmaxf(mu, t * fabsf(uc[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
      mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
    }
    if (lane == 0) {
      red[0][warp] = mw;
      red[1][warp] = mu;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kWyThreads / 32; ++w) {
      mw = fmaxf(mw, red[0][w]);
      mu = fmaxf(mu, red[1][w]);
    }
    sw = f16_split_scale(mw, &isw);
    su = f16_split_scale(mu, &isu);
  }
  // T diag(c) sc as hi + lo of the input type into the split tiles (row s, 8 consecutive j
  // per item)
  unsigned char *th = sm + lay.th, *tl = sm + lay.tl;
  auto split = [&](const float *cv, float sc) {
    for (int it = tid; it < kChunk * 8; it += kWyThreads) {
      const int srow = it >> 3, j0 = (it & 7) * 8;
      const float4 t0 = *reinterpret_cast<const float4 *>(Tm + srow * kLdT + j0);
      const float4 t1 = *reinterpret_cast<const float4 *>(Tm + srow * kLdT + j0 + 4);
      const float t[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
      typename In::T2 hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a0 = t[2 * i] * cv[j0 + 2 * i] * sc, a1 = t[2 * i + 1] * cv[j0 + 2 * i + 1] * sc;
        hi[i] = In::from_f2(a0, a1);
        const float2 f = In::to_f2(hi[i]);
        lo[i] = In::from_f2(a0 - f.x, a1 - f.y);
      }
      const uint32_t off = swz(srow, j0 * 2u);
      *reinterpret_cast<uint4 *>(th + off) = *reinterpret_cast<const uint4 *>(hi);
      *reinterpret_cast<uint4 *>(tl + off) = *reinterpret_cast<const uint4 *>(lo);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  // ---- W^T = K^T Tw^T, then U^T = V^T Tu^T through the same split tiles (A operands MN-major
  // from the k / v tiles); each split waits for the MMAs that read the tiles before it ----
  const uint32_t idwu = idesc(In::kFmt, 1, 0, 64, d);
  auto issue_wu = [&](uint32_t tD, const unsigned char *src, uint32_t lbo) {
    if (tid == 0) {
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t da = desc_sw128(smem_u32(src) + kk * 2048u, lbo, 1024);
        mma_bf16_ss(tD, da, desc_sw128(smem_u32(th) + kk * 32u, 16, 1024), idwu, kk > 0);
        mma_bf16_ss(tD, da, desc_sw128(smem_u32(tl) + kk * 32u, 16, 1024), idwu, 1);
      }
      mma_commit(&mma_bar);
    }
  };
  split(wc, sw);
  issue_wu(tW, kq, 16384u);
  if (!mbar_wait(&mma_bar, 1)) abort_flag = 1;
  split(uc, su);
  issue_wu(tU, vt, 8192u);
  if (!mbar_wait(&mma_bar, 0)) abort_flag = 1;
  tc_fence_after();
  __syncthreads();

  // ---- epilogue: -W image, U^T, Ktil^T image; the two warps of a lane quadrant take 32
  // columns s each.  Stores are arranged so that each warp instruction writes whole
  // 128-byte (-W, Ktil^T) or 512-byte (U^T) contiguous segments. ----
  const bool aborted = abort_flag;  // read after the barrier above: the same for every thread
  if (!aborted) {
    // D row f sits in lane f (M = 128) or in lane 32*(f/16) + f%16 (M = 64).
    const int rpw = (d == 128) ? 32 : 16;  // feature rows held by this lane quadrant
    const int f = quad * rpw + lane;
    const bool mine = lane < rpw;
    const uint32_t lrow = (uint32_t)(quad * 32) << 16;
    const int sbeg = chalf * 32;
    float4 *Ut = reinterpret_cast<float4 *>(p.U + ((int64_t)row * p.H + h) * p.V * kChunk) + (f >> 5) * 512 + (f & 31);
    unsigned char *wimg = img + il.b1 + (f >> 5) * il.b1_block;
#pragma unroll 1
    for (int c0 = sbeg; c0 < sbeg + 32; c0 += 16) {
      float wv[16], uv[16];
      tmem_ld16(tW + lrow + c0, wv);
      tmem_ld16(tU + lrow + c0, uv);
      if (mine) {
        // U^T rows in the 32-row-group layout: consecutive lanes at consecutive 16 bytes
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          Ut[((c0 + j) >> 2) * 32] = make_float4(uv[j] * isu, uv[j + 1] * isu, uv[j + 2] * isu, uv[j + 3] * isu);
        // -W image: element (s, f) at row qpad + s of K-block f/32 (a row of 32 lanes = 128
        // bytes).  Rows qpad + c0 + u share (row / 8) for u < 8 and u >= 8, and their in-atom
        // offset depends on u % 8 only: eight offsets per thread, computed once
        uint32_t xo[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) xo[k] = ImageLayout::swz_off(k, f);
        unsigned char *w0 = wimg + (uint32_t)((QP + c0) >> 3) * 1024u;
#pragma unroll
        for (int u = 0; u < 16; ++u)
          *reinterpret_cast<float *>(w0 + (uint32_t)(u >> 3) * 1024u + xo[u & 7]) = -wv[u] * isw;
        if (bimg)  // (-W)^T: row f, columns c0 .. c0 + 15, four 16-byte chunks
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4 *>(bimg + bl.w_at(f, c0 + j)) =
                make_float4(-wv[j] * isw, -wv[j + 1] * isw, -wv[j + 2] * isw, -wv[j + 3] * isw);
      }
    }
    // Ktil^T image: row f = 2^(G2_last - G2_s) rk_s k[s][f], K-block s/32; lane = s, so each
    // store instruction writes one 128-byte row segment.  This warp takes the rows f of its
    // quadrant eight at a time: one 16-byte load of k row s gives features f0 .. f0 + 7, each
    // stored to its own row at the swizzled column s (eight offsets per thread, computed once)
    const int s_ = sbeg + lane;
    const float kss = ks[s_];
    unsigned char *kimg = img + il.b2 + chalf * il.b2_block;
    uint32_t yo[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) yo[j] = ImageLayout::swz_off(j, s_);
#pragma unroll 1
    for (int f0 = quad * (d / 4); f0 < (quad + 1) * (d / 4); f0 += 8) {
      float x[8];
      in8_at<F16>(kq, 128, s_, f0, x);
      unsigned char *r0 = kimg + (uint32_t)(f0 >> 3) * 1024u;
#pragma unroll
      for (int j = 0; j < 8; ++j) *reinterpret_cast<float *>(r0 + yo[j]) = kss * x[j];
      if (bimg) {  // Ktil: row s, features f0 .. f0 + 7, two 16-byte chunks
        *reinterpret_cast<float4 *>(bimg + bl.k_at(s_, f0)) =
            make_float4(kss * x[0], kss * x[1], kss * x[2], kss * x[3]);
        *reinterpret_cast<float4 *>(bimg + bl.k_at(s_, f0 + 4)) =
            make_float4(kss * x[4], kss * x[5], kss * x[6], kss * x[7]);
      }
    }
  }
  if (tid == 0) {
    ImageMeta *mt = reinterpret_cast<ImageMeta *>(img + il.meta);
    mt->gamma_last = exp2f(G2last);
    mt->nq = nq;
    mt->p0 = p0;
    mt->len = len;
    mt->fast = fast ? 1 : 0;
    if (bimg) *reinterpret_cast<ImageMeta *>(bimg + bl.meta) = *mt;
    if (abort_flag) set_status(p.status, GDP_DEV_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_free(tbase, 128);
}

// Shared by the WY kernels of every type combination (one translation unit for the common
// kernel, one for the rest): tensor maps of k, q, v and the grid (expanded chunk, head).
template <typename Kern>
cudaError_t launch_wy_kernel(Kern kern, const Problem &p, cudaStream_t stream) {
  // Beside the scan (a segmented call) the tiles run two per SM, asked for by the shared memory
  // size: with three, the scan beside them ran 2.5 % slower on the 65536-token sequence than the
  // WY tiles gained (A/B on one GB300)
  const size_t smem = p.seg_rows > 0 ? (size_t)100 * 1024 : WyLayout(p.K).total + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap tm_k, tm_q, tm_v;
  const int64_t rows = p.T * p.M;
  if ((e = tmap_rows_16(&tm_k, p.k, rows, p.Hk, p.K, p.k_st, p.k_sh, kChunk, p.f16)) != cudaSuccess) return e;
  if ((e = tmap_rows_16(&tm_q, p.q, p.T, p.Hq, p.K, p.q_st, p.q_sh, p.qpad, p.f16)) != cudaSuccess) return e;
  if ((e = tmap_rows_16(&tm_v, p.v, rows, p.Hv, p.V, p.v_st, p.v_sh, kChunk, p.f16)) != cudaSuccess) return e;
  dim3 grid(p.seg_rows > 0 ? (unsigned)(p.N * p.seg_rows) : (unsigned)p.ntdp_pad, (unsigned)p.H);
  if ((e = launch_kernel(kern, grid, dim3(kWyThreads), smem, stream, p.pdl != 0, p, tm_k, tm_q, tm_v)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

#define GDP_WY_KERNEL(name, f16, typed)                                                                          \
  __global__ void __launch_bounds__(kWyThreads, kWyCtasPerSm)                                                   \
      name(Problem p, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,        \
           const __grid_constant__ CUtensorMap tm_v) {                                                            \
    wy_body<f16, typed>(p, tm_k, tm_q, tm_v);                                                                   \
  }

}  // namespace
}  // namespace gdp
