// gdp_backward.cu -- backward pass of the chunked GDP prefill (training).
//
// The pages give the forward recurrence only (FlashInfer API page
// "flashinfer.gdp_prefill.chunk_gated_delta_product", display equation) and note that
// training runs it in chunks with the backward dependence running the other way round
// (blog post "Attention Cache and Sequence Parallelism", section on passing state instead
// of KV).  The kernels here evaluate the derivative of that recurrence in chunk form.
// For one expanded chunk (rows r < C <= 64, entering state S, gamma_r = exp(G_r) with G
// the within-chunk cumulative log decay, khat / qhat the (optionally L2-normalised) rows,
// L_rj = gamma_r / gamma_j (khat_r . khat_j) for j < r, A = diag(beta) L, readout rows
// p = t*M + M-1 with P_pj = scale gamma_p / gamma_j (qhat_p . khat_j) for j <= p):
//   forward values   e = V - diag(gamma) Khat S^T - L Vt,  Vt = diag(beta) e   (row by row)
//                    o_p = scale gamma_p S qhat_p + sum_j P_pj vt_j
//   exit gradient    D_C = dL/dS at the chunk end, from the reverse state scan:
//                    D_in = D_C (gamma_C I - Ktil^T W) + dO^T (Qh - P W)
//                    (Ktil = diag(gamma_C / gamma) Khat; W, Qh: the forward's WY factors)
//   per row          Delta = (I + A^T)^-1 (Ktil D_C^T + P^T dO)      (back substitution)
//                    dv = diag(beta) Delta,  dbeta_r = e_r . Delta_r
//                    dkhat = diag(beta)[diag(gamma_C/gamma)(e D_C) + M1 Qhat - M2 Khat]
//                            - diag(gamma)(dv S) - M3 Khat
//                    dqhat = scale [diag(gamma_p)(dO S) + M4 Khat]
//   with M1_rp = scale gamma_p/gamma_r (e_r . do_p) [r <= p], M2_rj = gamma_j/gamma_r
//   (e_r . dv_j) [j > r], M3_rj = gamma_r/gamma_j (dv_r . vt_j) [j < r], M4_pj =
//   gamma_p/gamma_j (do_p . vt_j) [j <= p].  The decay gradient needs no state:
//   dg_t = <dS_T, S_T> + sum_{t' >= t} (do_t' . o_t' - sum_j dv_{t'M+j} . v_{t'M+j}).
// Everything above follows from the row recurrence by algebra alone; the float64 oracle
// takes the derivative step by step instead and the parity tests compare the two.
//
// Kernels: the reverse state scan (D_C of every chunk) runs on the tcgen05 tensor cores with D
// resident in TMEM (gdp_bwd_scan_tc.cu), and so do the per-chunk gradients for head size 128 with
// two or more updates per token (gdp_bwd_chunk_tc.cu).  The per-chunk kernel here serves the other
// shapes (head size 64, one update per token) with warp-level tf32 MMAs and fp32 accumulation (the
// triangular solves in the 3xTF32 split):
//   gdp_bwd_chunk_kernel  one CTA per (expanded chunk, head), V in 16- (or 8-) column
//                         slices: the per-row gradients above, the L2-norm chain rule
//                         dx = dxhat / n - x (x . dxhat) / n^3, dq / dk / dv / dbeta stores
//   gdp_bwd_dg_kernel     reverse cumulative sum of the decay gradient per (sequence, head)
#include "gdp_internal.cuh"
#include "gdp_sm100.cuh"

namespace gdp {

// The per-chunk gradients on the tensor cores (gdp_bwd_chunk_tc.cu) for the shapes it serves.
bool bwd_chunk_tc_serves(int d, int qpad);
cudaError_t launch_bwd_chunk_tc(const BwdProblem &p, cudaStream_t stream);

namespace {

using namespace sm100;

__device__ __forceinline__ uint32_t tf32r(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// c[16 x 8] += A[16 x 8] B[8 x 8] (m16n8k8, tf32 in, fp32 out).  Fragments (lane = 4 g + t):
// A (g, t), (g+8, t), (g, t+4), (g+8, t+4); B (t, g), (t+4, g); C (g, 2t), (g, 2t+1),
// (g+8, 2t), (g+8, 2t+1).
__device__ __forceinline__ void mma8(float *c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                     uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------------------
// Per-chunk gradients.
// ---------------------------------------------------------------------------------------
// acc[16 x 8] += A[16 x 8 ks] B[8 ks x 8] for one output tile (m16n8k8 tf32, fp32 accumulate).
// A is read as At[k][m] when AT (else row-major [m][k]); B as Bt[n][k] when BT (else
// row-major [k][n]); pointers are at the tile origin.  arow (per tile row) and bk (per k)
// scale the operands when given.  Within every 8-wide k step the logical k order is
// permuted (logical k = t <-> physical 2t, k = t + 4 <-> 2t + 1) for A and B alike, so
// that row-major A and Bt fragments load as float2.  SPLIT: 3xTF32 (x = hi + lo, the
// lo*lo product dropped), about fp32 accuracy.
template <bool AT, bool BT, bool SPLIT>
__device__ __forceinline__ void tile_mma(float *c, const float *A, int lda, const float *B, int ldb, int ks,
                                         const float *arow, const float *bk, int g, int t) {
  const float sa0 = arow ? arow[g] : 1.f, sa1 = arow ? arow[g + 8] : 1.f;
#pragma unroll 2
  for (int kk = 0; kk < ks; ++kk) {
    const int k0 = 8 * kk + 2 * t;
    float a0, a1, a2, a3, b0, b1;
    if (!AT) {
      const float2 x = *reinterpret_cast<const float2 *>(A + g * lda + k0);
      const float2 y = *reinterpret_cast<const float2 *>(A + (g + 8) * lda + k0);
      a0 = x.x; a2 = x.y; a1 = y.x; a3 = y.y;
    } else {
      a0 = A[k0 * lda + g]; a2 = A[(k0 + 1) * lda + g]; a1 = A[k0 * lda + g + 8]; a3 = A[(k0 + 1) * lda + g + 8];
    }
    if (BT) {
      const float2 x = *reinterpret_cast<const float2 *>(B + g * ldb + k0);
      b0 = x.x; b1 = x.y;
    } else {
      b0 = B[k0 * ldb + g]; b1 = B[(k0 + 1) * ldb + g];
    }
    a0 *= sa0; a2 *= sa0; a1 *= sa1; a3 *= sa1;
    if (bk) {
      b0 *= bk[k0];
      b1 *= bk[k0 + 1];
    }
    if (SPLIT) {
      const uint32_t ah0 = tf32r(a0), ah1 = tf32r(a1), ah2 = tf32r(a2), ah3 = tf32r(a3), bh0 = tf32r(b0),
                     bh1 = tf32r(b1);
      const uint32_t al0 = tf32r(a0 - __uint_as_float(ah0)), al1 = tf32r(a1 - __uint_as_float(ah1)),
                     al2 = tf32r(a2 - __uint_as_float(ah2)), al3 = tf32r(a3 - __uint_as_float(ah3)),
                     bl0 = tf32r(b0 - __uint_as_float(bh0)), bl1 = tf32r(b1 - __uint_as_float(bh1));
      mma8(c, al0, al1, al2, al3, bh0, bh1);
      mma8(c, ah0, ah1, ah2, ah3, bl0, bl1);
      mma8(c, ah0, ah1, ah2, ah3, bh0, bh1);
    } else {
      mma8(c, tf32r(a0), tf32r(a1), tf32r(a2), tf32r(a3), tf32r(b0), tf32r(b1));
    }
  }
}
// As tile_mma for NT adjacent output tiles (columns 8 n .. 8 n + 7 of B for n < NT) that
// share the A fragments: A is loaded, scaled and rounded once per k step.
template <int NT, bool AT, bool BT, bool SPLIT>
__device__ __forceinline__ void tiles_mma(float (*c)[4], const float *A, int lda, const float *B, int ldb, int ks,
                                          const float *arow, const float *bk, int g, int t) {
  const float sa0 = arow ? arow[g] : 1.f, sa1 = arow ? arow[g + 8] : 1.f;
#pragma unroll 1
  for (int kk = 0; kk < ks; ++kk) {
    const int k0 = 8 * kk + 2 * t;
    float a0, a1, a2, a3;
    if (!AT) {
      const float2 x = *reinterpret_cast<const float2 *>(A + g * lda + k0);
      const float2 y = *reinterpret_cast<const float2 *>(A + (g + 8) * lda + k0);
      a0 = x.x; a2 = x.y; a1 = y.x; a3 = y.y;
    } else {
      a0 = A[k0 * lda + g]; a2 = A[(k0 + 1) * lda + g]; a1 = A[k0 * lda + g + 8]; a3 = A[(k0 + 1) * lda + g + 8];
    }
    a0 *= sa0; a2 *= sa0; a1 *= sa1; a3 *= sa1;
    const float s0 = bk ? bk[k0] : 1.f, s1 = bk ? bk[k0 + 1] : 1.f;
    uint32_t ah[4] = {tf32r(a0), tf32r(a1), tf32r(a2), tf32r(a3)};
    uint32_t al[4] = {0u, 0u, 0u, 0u};
    if (SPLIT) {
      al[0] = tf32r(a0 - __uint_as_float(ah[0]));
      al[1] = tf32r(a1 - __uint_as_float(ah[1]));
      al[2] = tf32r(a2 - __uint_as_float(ah[2]));
      al[3] = tf32r(a3 - __uint_as_float(ah[3]));
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      float b0, b1;
      if (BT) {
        const float2 x = *reinterpret_cast<const float2 *>(B + (8 * n + g) * ldb + k0);
        b0 = x.x; b1 = x.y;
      } else {
        b0 = B[k0 * ldb + 8 * n + g]; b1 = B[(k0 + 1) * ldb + 8 * n + g];
      }
      b0 *= s0;
      b1 *= s1;
      const uint32_t bh0 = tf32r(b0), bh1 = tf32r(b1);
      if (SPLIT) {
        const uint32_t bl0 = tf32r(b0 - __uint_as_float(bh0)), bl1 = tf32r(b1 - __uint_as_float(bh1));
        mma8(c[n], al[0], al[1], al[2], al[3], bh0, bh1);
        mma8(c[n], ah[0], ah[1], ah[2], ah[3], bl0, bl1);
      }
      mma8(c[n], ah[0], ah[1], ah[2], ah[3], bh0, bh1);
    }
  }
}
// Row / column of element x of an m16n8 accumulator tile.
__device__ __forceinline__ int trow(int x, int g) { return g + 8 * (x >> 1); }
__device__ __forceinline__ int tcol(int x, int t) { return 2 * t + (x & 1); }

constexpr int kChunkThreads = 512;  // 16 warps
constexpr int kLC = kChunk + 8;     // row stride of [rows][64] tiles (8 mod 32: conflict-free float2)

struct ChunkSmem {
  int ldd, ldv, ldq;
  uint32_t kh, qh, lm, tm, pm, g1, g23, g4, ss, dcs, vs, dos, rhs, qs, zt, dl, vt, scal, total;
  __host__ __device__ ChunkSmem(int d, int qp, int vsl) {
    ldd = d + 8;
    ldv = vsl + 8;
    ldq = qp + 8;
    uint32_t o = 0;
    auto take = [&](uint32_t floats) {
      const uint32_t at = o;
      o += (floats * 4u + 15u) & ~15u;
      return at;
    };
    kh = take(kChunk * ldd);    // khat [64][d]
    qh = take(qp * ldd);        // qhat readout rows [qp][d]
    lm = take(kChunk * kLC);    // L [64][64] (decayed Gram, strictly lower)
    tm = take(kChunk * kLC);    // T = (I + diag(beta) L)^-1 (adjacent to L: together the dkhat staging)
    pm = take(qp * kLC);        // P [qp][64]
    g1 = take(kChunk * ldq);    // sum over V of e dO^T [64][qp]
    g23 = take(kChunk * kLC);   // upper: sum e dv^T, lower: sum dv vt^T [64][64]
    g4 = take(qp * kLC);        // sum dO vt^T [qp][64]
    ss = take(vsl * ldd);       // S slice [vsl][d]
    dcs = take(vsl * ldd);      // D_C slice [vsl][d]
    vs = take(kChunk * ldv);    // v slice [64][vsl]
    dos = take(qp * ldv);       // d_output slice [qp][vsl]
    rhs = take(kChunk * ldv);   // rhs, then e [64][vsl]
    qs = take(qp * ldv);        // qhat S^T [qp][vsl]
    zt = take(kChunk * ldv);    // Ktil D_C^T + P^T dO [64][vsl]
    dl = take(kChunk * ldv);    // Delta [64][vsl]
    vt = take(kChunk * ldv);    // vt [64][vsl]
    scal = take(14 * kChunk);   // per-row factors and sums
    total = o;
  }
};

// One CTA per (expanded chunk, head); V in slices of VSL columns.  T = (I + A)^-1 is formed
// once, so the two triangular solves of every slice are small matrix products (3xTF32).
// dkhat and dqhat sum over the slices in registers and leave through the L2-norm chain
// rule; dbeta, sum_v dv v and do . o are complete per chunk and stored as they are.
template <int D, int VSL>
__global__ void __launch_bounds__(kChunkThreads, 1) gdp_bwd_chunk_kernel(BwdProblem p) {
  const int row = blockIdx.x, h = blockIdx.y;
  const int seq = p.cid[2 * row], c = p.cid[2 * row + 1];
  if (seq < 0 || seq >= p.N || row >= p.ws_rows) return;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;
  if (c < 0 || L <= 0 || (int64_t)c * kChunk >= L * p.M) return;
  const int M = p.M, QP = p.qpad, H = p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int64_t R0 = bos * M + (int64_t)c * kChunk;
  const int len = (int)min((int64_t)kChunk, L * M - (int64_t)c * kChunk);
  const int r0m = (int)(R0 % M);
  const int64_t tok0 = (R0 - r0m) / M;
  const int p0 = (M - 1 - r0m) % M;
  const int nq = (p0 < len) ? (len - 1 - p0) / M + 1 : 0;
  const int64_t tq0 = (R0 + p0) / M;
  const int64_t srow = (int64_t)p.cod[seq] + c;

  extern __shared__ __align__(16) unsigned char bwd_chunk_raw[];
  const ChunkSmem lay(D, QP, VSL);
  const int LDD = lay.ldd, LDV = lay.ldv, LDQ = lay.ldq;
  unsigned char *sm = bwd_chunk_raw;
  auto F = [&](uint32_t off) { return reinterpret_cast<float *>(sm + off); };
  float *kh = F(lay.kh), *qh = F(lay.qh), *lm = F(lay.lm), *tm = F(lay.tm), *pm = F(lay.pm);
  float *g1 = F(lay.g1), *g23 = F(lay.g23), *g4 = F(lay.g4), *ss = F(lay.ss), *dcs = F(lay.dcs);
  float *vs = F(lay.vs), *dos = F(lay.dos), *rhs = F(lay.rhs), *qs = F(lay.qs), *zt = F(lay.zt), *dl = F(lay.dl),
        *vt = F(lay.vt);
  float *G = F(lay.scal), *bt = G + kChunk, *gm = bt + kChunk, *fc = gm + kChunk, *bfc = fc + kChunk,
        *gb = bfc + kChunk, *rk = gb + kChunk, *rq = rk + kChunk, *gq = rq + kChunk, *sdb = gq + kChunk,
        *ssg = sdb + kChunk, *srho = ssg + kChunk, *scq = srho + kChunk, *mgb = scq + kChunk;
  __shared__ float carry;

  // ---- scalars: beta, gates, within-chunk cumulative log decay ----
  if (tid < kChunk) {
    const int r = tid, pos = r0m + r;
    float b = 0.f, gate = 0.f;
    if (r < len) {
      b = p.beta ? p.beta[(R0 + r) * H + h] : 1.f;
      if (p.g && pos % M == 0) gate = p.g[(tok0 + pos / M) * H + h];
    }
    bt[r] = b;
    float x = gate;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (r == 31) carry = x;
    G[r] = x;
    sdb[r] = ssg[r] = srho[r] = 0.f;
  }
  // ---- khat and qhat rows (8 threads per row) ----
  for (int r = tid >> 3; r < kChunk + QP; r += kChunkThreads / 8) {
    const int part = tid & 7;
    const bool isk = r < kChunk;
    const int rr = isk ? r : r - kChunk;
    const bool live = isk ? rr < len : rr < nq;
    const __nv_bfloat16 *src = isk ? p.k + (R0 + rr) * p.k_st + (int64_t)h * p.k_sh
                                   : p.q + (tq0 + rr) * p.q_st + (int64_t)h * p.q_sh;
    float x[D / 8];
    float s2 = 0.f;
#pragma unroll
    for (int i = 0; i < D / 8; i += 8) {
      uint4 u = make_uint4(0u, 0u, 0u, 0u);
      if (live) u = *reinterpret_cast<const uint4 *>(src + part * (D / 8) + i);
      const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const float2 f = __bfloat1622float2(b2[q2]);
        x[i + 2 * q2] = f.x;
        x[i + 2 * q2 + 1] = f.y;
        s2 += f.x * f.x + f.y * f.y;
      }
    }
    s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 4);
    const float inv = p.l2norm ? rsqrtf(s2 + kL2Eps) : 1.f;
    if (part == 0) (isk ? rk : rq)[rr] = inv;
    float *dst = (isk ? kh : qh) + rr * LDD + part * (D / 8);
#pragma unroll
    for (int i = 0; i < D / 8; i += 4)
      *reinterpret_cast<float4 *>(dst + i) = make_float4(x[i] * inv, x[i + 1] * inv, x[i + 2] * inv, x[i + 3] * inv);
  }
  __syncthreads();
  if (tid < kChunk) {
    const float x = (tid >= 32 ? G[tid] + carry : G[tid]);
    G[tid] = x;
  }
  __syncthreads();
  const float GC = G[len - 1], scale = p.scale;
  auto pr = [&](int qi) { return p0 + qi * M; };  // local row of readout qi
  if (tid < kChunk) {
    const int r = tid;
    const float gr = expf(G[r]), f = expf(GC - G[r]), b = bt[r];
    gm[r] = gr;           // gamma_r
    fc[r] = f;            // gamma_C / gamma_r
    bfc[r] = b * f;       // beta_r gamma_C / gamma_r
    gb[r] = gr * b;       // gamma_r beta_r
    mgb[r] = -gr * b;     // -gamma_r beta_r
    gq[r] = (r < nq) ? scale * expf(G[pr(r)]) : 0.f;  // scale gamma_p of readout r
    scq[r] = scale;
  }
  __syncthreads();

  // ---- the V slices' rows: S and D_C rows v0 .. v0 + VSL - 1 (float4 items) and the v / d_output
  // columns v0 .. (4 bf16 per item), at most one item of each per thread; each slice's items are
  // loaded into registers one slice ahead (the first during the Gram and the inverse) and put
  // into shared memory when the slice starts ----
  const int64_t KV = (int64_t)D * D;
  const float *Sg = p.Sx + (srow * H + h) * KV;
  const float *Dg = p.Dx + (srow * H + h) * KV;
  constexpr int NS = VSL * (D / 4), NV = (kChunk + 64) * (VSL / 4);
  static_assert(NS <= kChunkThreads && NV <= kChunkThreads, "one slice item per thread");
  float4 pre_s = make_float4(0.f, 0.f, 0.f, 0.f), pre_d = pre_s;
  uint2 pre_v = make_uint2(0u, 0u);
  auto fetch = [&](int v0) {
    if (tid < NS) {
      const int r = tid / (D / 4), c4 = (tid % (D / 4)) * 4;
      pre_s = *reinterpret_cast<const float4 *>(Sg + (int64_t)(v0 + r) * D + c4);
      pre_d = *reinterpret_cast<const float4 *>(Dg + (int64_t)(v0 + r) * D + c4);
    }
    if (tid < (kChunk + QP) * (VSL / 4)) {
      const int r = tid / (VSL / 4), c4 = (tid % (VSL / 4)) * 4;
      const bool isv = r < kChunk;
      const int rr = isv ? r : r - kChunk;
      pre_v = make_uint2(0u, 0u);
      if (isv ? rr < len : rr < nq)
        pre_v = *reinterpret_cast<const uint2 *>(isv ? p.v + (R0 + rr) * p.v_st + (int64_t)h * p.v_sh + v0 + c4
                                                     : p.dout + ((tq0 + rr) * H + h) * (int64_t)D + v0 + c4);
    }
  };
  auto put = [&](float *ss_, float *dcs_, float *vs_, float *dos_) {
    if (tid < NS) {
      const int r = tid / (D / 4), c4 = (tid % (D / 4)) * 4;
      *reinterpret_cast<float4 *>(ss_ + r * lay.ldd + c4) = pre_s;
      *reinterpret_cast<float4 *>(dcs_ + r * lay.ldd + c4) = pre_d;
    }
    if (tid < (kChunk + QP) * (VSL / 4)) {
      const int r = tid / (VSL / 4), c4 = (tid % (VSL / 4)) * 4;
      const bool isv = r < kChunk;
      const int rr = isv ? r : r - kChunk;
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pre_v.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pre_v.y));
      *reinterpret_cast<float4 *>((isv ? vs_ : dos_) + rr * lay.ldv + c4) = make_float4(a.x, a.y, b.x, b.y);
    }
  };
  fetch(0);

  // ---- L [64 x 64] and P [qp x 64] ----
  for (int u = warp; u < 2 * (4 + QP / 16); u += kChunkThreads / 32) {  // (m-tile, 4 n-tiles) units
    float acc[4][4] = {};
    const bool isL = u < 8;
    const int uu = isL ? u : u - 8, m0 = 16 * (uu >> 1), n0 = 32 * (uu & 1);
    tiles_mma<4, false, true, false>(acc, (isL ? kh : qh) + m0 * LDD, LDD, kh + n0 * LDD, LDD, D / 8, nullptr,
                                     nullptr, g, t);
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int r = m0 + trow(x, g), j = n0 + 8 * n + tcol(x, t);
        if (isL) {
          lm[r * kLC + j] = (j < r) ? expf(G[r] - G[j]) * acc[n][x] : 0.f;
        } else {
          const bool ok = r < nq && j <= pr(r);
          pm[r * kLC + j] = ok ? scale * expf(G[pr(r)] - G[j]) * acc[n][x] : 0.f;
        }
      }
  }
  // zero the slice sums of the Gram matrices
  for (int i = tid; i < kChunk * LDQ; i += kChunkThreads) g1[i] = 0.f;
  for (int i = tid; i < kChunk * kLC; i += kChunkThreads) g23[i] = 0.f;
  for (int i = tid; i < QP * kLC; i += kChunkThreads) g4[i] = 0.f;
  __syncthreads();
  // ---- T = (I + A)^-1, A = diag(beta) L: the forward recompute's WY kernel inverted it (its A is
  // the same matrix: beta_r gamma_r / gamma_j (khat_r . khat_j), j < r) and left it beside the
  // chunk's reverse-scan image ----
  {
    const float *Tg = reinterpret_cast<const float *>(p.bimg + (size_t)(srow * H + h) * p.bimg_stride +
                                                      BwdImageLayout(D, QP).tinv);
    for (int idx = tid; idx < kChunk * kChunk / 4; idx += kChunkThreads) {
      const int r = idx >> 4, c4 = (idx & 15) * 4;
      *reinterpret_cast<float4 *>(tm + r * kLC + c4) = *reinterpret_cast<const float4 *>(Tg + r * kChunk + c4);
    }
  }
  __syncthreads();

  // dkhat / dqhat accumulators: warp w owns output tiles of a fixed m-tile and a run of n-tiles
  constexpr int NTK = (kChunk / 16) * (D / 8) / (kChunkThreads / 32);  // dkhat tiles per warp
  const int mk = warp % 4, nk0 = (warp / 4) * NTK;
  float dk_acc[NTK][4];
#pragma unroll
  for (int i = 0; i < NTK; ++i) dk_acc[i][0] = dk_acc[i][1] = dk_acc[i][2] = dk_acc[i][3] = 0.f;
  const int nqt = (QP / 16) * (D / 8);  // dqhat tiles, dealt round robin: tile warp + 16 i
  constexpr int NTQ = (4 * (D / 8) + kChunkThreads / 32 - 1) / (kChunkThreads / 32);  // qp <= 64
  float dq_acc[NTQ][4];
#pragma unroll
  for (int i = 0; i < NTQ; ++i) dq_acc[i][0] = dq_acc[i][1] = dq_acc[i][2] = dq_acc[i][3] = 0.f;
  auto dq_tile = [&](int i, int &m0, int &n0) {
    const int u = warp + (kChunkThreads / 32) * i;
    m0 = 16 * (u / (D / 8));
    n0 = 8 * (u % (D / 8));
    return u < nqt;
  };

  constexpr int NVS = VSL / 8;  // n-tiles per slice
#pragma unroll 1
  for (int v0 = 0; v0 < D; v0 += VSL) {
    // ---- slice rows: S and D_C rows v0 .., v and d_output columns v0 .. (fetched a slice
    // ahead); the next slice's go out now ----
    put(ss, dcs, vs, dos);
    if (v0 + VSL < D) fetch(v0 + VSL);
    __syncthreads();
    // ---- rhs = v - gamma (Khat S^T);  QS = qhat S^T;  Zt = Ktil D_C^T + P^T dO ----
    for (int u = warp; u < 8 + QP / 16; u += kChunkThreads / 32) {  // (m-tile, all NVS n-tiles) units
      float acc[NVS][4] = {};
      if (u < 4) {
        const int m0 = 16 * u;
        tiles_mma<NVS, false, true, false>(acc, kh + m0 * LDD, LDD, ss, LDD, D / 8, nullptr, nullptr, g, t);
#pragma unroll
        for (int n = 0; n < NVS; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int r = m0 + trow(x, g), j = 8 * n + tcol(x, t);
            rhs[r * LDV + j] = vs[r * LDV + j] - gm[r] * acc[n][x];
          }
      } else if (u < 8) {
        const int m0 = 16 * (u - 4);
        tiles_mma<NVS, false, true, false>(acc, kh + m0 * LDD, LDD, dcs, LDD, D / 8, fc + m0, nullptr, g, t);
        tiles_mma<NVS, true, false, false>(acc, pm + m0, kLC, dos, LDV, QP / 8, nullptr, nullptr, g, t);
#pragma unroll
        for (int n = 0; n < NVS; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) zt[(m0 + trow(x, g)) * LDV + 8 * n + tcol(x, t)] = acc[n][x];
      } else {
        const int m0 = 16 * (u - 8);
        tiles_mma<NVS, false, true, false>(acc, qh + m0 * LDD, LDD, ss, LDD, D / 8, nullptr, nullptr, g, t);
#pragma unroll
        for (int n = 0; n < NVS; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) qs[(m0 + trow(x, g)) * LDV + 8 * n + tcol(x, t)] = acc[n][x];
      }
    }
    __syncthreads();
    // ---- vt = T diag(beta) rhs;  Delta = T^T Zt  (3xTF32) ----
    for (int u = warp; u < 8; u += kChunkThreads / 32) {
      float acc[NVS][4] = {};
      const bool isv = u < 4;
      const int m0 = 16 * (isv ? u : u - 4);
      if (isv)
        tiles_mma<NVS, false, false, true>(acc, tm + m0 * kLC, kLC, rhs, LDV, kChunk / 8, nullptr, bt, g, t);
      else
        tiles_mma<NVS, true, false, true>(acc, tm + m0, kLC, zt, LDV, kChunk / 8, nullptr, nullptr, g, t);
#pragma unroll
      for (int n = 0; n < NVS; ++n)
#pragma unroll
        for (int x = 0; x < 4; ++x) (isv ? vt : dl)[(m0 + trow(x, g)) * LDV + 8 * n + tcol(x, t)] = acc[n][x];
    }
    __syncthreads();
    // ---- e = rhs - L vt (in place);  o = scale gamma_p QS + P vt -> do . o;  dv out ----
    for (int u = warp; u < 4 + QP / 16; u += kChunkThreads / 32) {
      float acc[NVS][4] = {};
      if (u < 4) {
        const int m0 = 16 * u;
        tiles_mma<NVS, false, false, false>(acc, lm + m0 * kLC, kLC, vt, LDV, kChunk / 8, nullptr, nullptr, g, t);
#pragma unroll
        for (int n = 0; n < NVS; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) rhs[(m0 + trow(x, g)) * LDV + 8 * n + tcol(x, t)] -= acc[n][x];
      } else {
        const int m0 = 16 * (u - 4);
        tiles_mma<NVS, false, false, false>(acc, pm + m0 * kLC, kLC, vt, LDV, kChunk / 8, nullptr, nullptr, g, t);
        float part[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < NVS; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int r = m0 + trow(x, g), j = 8 * n + tcol(x, t);
            part[x >> 1] += (gq[r] * qs[r * LDV + j] + acc[n][x]) * dos[r * LDV + j];
          }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {  // the unit covers the slice: one plain add per row
          float s = part[hf];
          s += __shfl_xor_sync(0xffffffffu, s, 1);
          s += __shfl_xor_sync(0xffffffffu, s, 2);
          if (t == 0) srho[m0 + g + 8 * hf] += s;
        }
      }
    }
    for (int idx = tid; idx < len * VSL; idx += kChunkThreads) {
      const int r = idx / VSL, j = idx % VSL;
      p.dv[((R0 + r) * H + h) * (int64_t)D + v0 + j] = bt[r] * dl[r * LDV + j];
    }
    __syncthreads();
    // ---- row sums: dbeta += e . Delta, sum dv v;  Gram sums over V;  dkhat, dqhat shares ----
    if (tid < 2 * kChunk) {
      const int r = tid >> 1, hf = tid & 1;
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int j = hf * (VSL / 2); j < (hf + 1) * (VSL / 2); ++j) {
        a += rhs[r * LDV + j] * dl[r * LDV + j];
        b += dl[r * LDV + j] * vs[r * LDV + j];
      }
      a += __shfl_xor_sync(0xffffffffu, a, 1);
      b += __shfl_xor_sync(0xffffffffu, b, 1);
      if (hf == 0) {
        sdb[r] += a;
        ssg[r] += bt[r] * b;
      }
    }
    {
      // G1 += e dO^T [64 x qp]; G23 += (upper) e dv^T, (lower) dv vt^T; G4 += dO vt^T [qp x 64]
      // units: G1 (m-tile, qp/8 n-tiles), G23 (m-tile, 4 n-tiles, upper and lower products), G4
      // (m-tile, 4 n-tiles); the A rows of G23's lower product are dv = beta Delta
      const int n1 = 4, n4 = 2 * (QP / 16);
      for (int u = warp; u < n1 + 8 + n4; u += kChunkThreads / 32) {
        if (u < n1) {
          const int m0 = 16 * u;
          float acc[8][4] = {};
          if (QP == 16)
            tiles_mma<2, false, true, false>(acc, rhs + m0 * LDV, LDV, dos, LDV, VSL / 8, nullptr, nullptr, g, t);
          else if (QP == 32)
            tiles_mma<4, false, true, false>(acc, rhs + m0 * LDV, LDV, dos, LDV, VSL / 8, nullptr, nullptr, g, t);
          else
            tiles_mma<8, false, true, false>(acc, rhs + m0 * LDV, LDV, dos, LDV, VSL / 8, nullptr, nullptr, g, t);
#pragma unroll
          for (int n = 0; n < 8; ++n)
            if (n < QP / 8)
#pragma unroll
              for (int x = 0; x < 4; ++x) g1[(m0 + trow(x, g)) * LDQ + 8 * n + tcol(x, t)] += acc[n][x];
        } else if (u < n1 + 8) {
          const int uu = u - n1, m0 = 16 * (uu >> 1), n0 = 32 * (uu & 1);
          float up[4][4] = {}, lo[4][4] = {};
          tiles_mma<4, false, true, false>(up, rhs + m0 * LDV, LDV, dl + n0 * LDV, LDV, VSL / 8, nullptr, nullptr, g, t);
          tiles_mma<4, false, true, false>(lo, dl + m0 * LDV, LDV, vt + n0 * LDV, LDV, VSL / 8, bt + m0, nullptr, g, t);
#pragma unroll
          for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const int r = m0 + trow(x, g), j = n0 + 8 * n + tcol(x, t);
              g23[r * kLC + j] += (j > r) ? bt[j] * up[n][x] : (j < r) ? lo[n][x] : 0.f;
            }
        } else {
          const int uu = u - n1 - 8, m0 = 16 * (uu >> 1), n0 = 32 * (uu & 1);
          float acc[4][4] = {};
          tiles_mma<4, false, true, false>(acc, dos + m0 * LDV, LDV, vt + n0 * LDV, LDV, VSL / 8, nullptr, nullptr, g, t);
#pragma unroll
          for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int x = 0; x < 4; ++x) g4[(m0 + trow(x, g)) * kLC + n0 + 8 * n + tcol(x, t)] += acc[n][x];
        }
      }
    }
    // dkhat += (beta gamma_C / gamma) e D_C - (gamma beta Delta) S
    tiles_mma<NTK, false, false, false>(dk_acc, rhs + 16 * mk * LDV, LDV, dcs + 8 * nk0, LDD, VSL / 8, bfc + 16 * mk,
                                        nullptr, g, t);
    tiles_mma<NTK, false, false, false>(dk_acc, dl + 16 * mk * LDV, LDV, ss + 8 * nk0, LDD, VSL / 8, mgb + 16 * mk,
                                        nullptr, g, t);
    // dqhat += (scale gamma_p dO) S
#pragma unroll
    for (int i = 0; i < NTQ; ++i)
      if (int m0, n0; dq_tile(i, m0, n0)) {
        tile_mma<false, false, false>(dq_acc[i], dos + m0 * LDV, LDV, ss + n0, LDD, VSL / 8, gq + m0, nullptr, g, t);
      }
    __syncthreads();
  }

  // ---- masks and decays of the Gram sums: M1 (times beta_r), beta M2 (upper) + M3 (lower), M4 ----
  for (int i = tid; i < kChunk * QP; i += kChunkThreads) {
    const int r = i / QP, qi = i % QP;
    const bool ok = qi < nq && r <= pr(qi);
    g1[r * LDQ + qi] = ok ? bt[r] * scale * expf(G[pr(qi)] - G[r]) * g1[r * LDQ + qi] : 0.f;
  }
  for (int i = tid; i < kChunk * kChunk; i += kChunkThreads) {
    const int r = i >> 6, j = i & 63;
    const float x = g23[r * kLC + j];
    g23[r * kLC + j] = (j > r) ? bt[r] * expf(G[j] - G[r]) * x : (j < r) ? expf(G[r] - G[j]) * x : 0.f;
  }
  for (int i = tid; i < QP * kChunk; i += kChunkThreads) {
    const int qi = i >> 6, j = i & 63;
    const bool ok = qi < nq && j <= pr(qi);
    g4[qi * kLC + j] = ok ? scale * expf(G[pr(qi)] - G[j]) * g4[qi * kLC + j] : 0.f;
  }
  __syncthreads();
  // dkhat += (beta M1) qhat - (beta M2 + M3) khat;  dqhat += scale M4 khat
  tiles_mma<NTK, false, false, false>(dk_acc, g1 + 16 * mk * LDQ, LDQ, qh + 8 * nk0, LDD, QP / 8, nullptr, nullptr, g,
                                      t);
  {
    float neg[NTK][4] = {};
    tiles_mma<NTK, false, false, false>(neg, g23 + 16 * mk * kLC, kLC, kh + 8 * nk0, LDD, kChunk / 8, nullptr, nullptr,
                                        g, t);
#pragma unroll
    for (int i = 0; i < NTK; ++i)
#pragma unroll
      for (int x = 0; x < 4; ++x) dk_acc[i][x] -= neg[i][x];
  }
#pragma unroll
  for (int i = 0; i < NTQ; ++i)
    if (int m0, n0; dq_tile(i, m0, n0)) {
      tile_mma<false, false, false>(dq_acc[i], g4 + m0 * kLC, kLC, kh + n0, LDD, kChunk / 8, nullptr, nullptr, g, t);
    }
  __syncthreads();  // L and T are free: they stage dkhat; the Gram sums stage dqhat
  float *stk = lm;   // [64][LDD] over L and T (2 x 64 x 72 >= 64 x (D + 8) floats)
  float *stq = g23;  // [qp][LDD] over G23 and G4 when they suffice, else over P .. G4
#pragma unroll
  for (int i = 0; i < NTK; ++i)
#pragma unroll
    for (int x = 0; x < 4; ++x) stk[(16 * mk + trow(x, g)) * LDD + 8 * (nk0 + i) + tcol(x, t)] = dk_acc[i][x];
  const bool q_in_g = (uint32_t)QP * LDD * 4u <= lay.ss - lay.g23;
  if (!q_in_g) stq = pm;
#pragma unroll
  for (int i = 0; i < NTQ; ++i)
    if (int m0, n0; dq_tile(i, m0, n0)) {
#pragma unroll
      for (int x = 0; x < 4; ++x) stq[(m0 + trow(x, g)) * LDD + n0 + tcol(x, t)] = dq_acc[i][x];
    }
  __syncthreads();
  // ---- L2-norm chain rule (dx = rx (dxhat - (xhat . dxhat) xhat)), stores, row sums ----
  for (int r = warp; r < len + nq; r += kChunkThreads / 32) {
    const bool isk = r < len;
    const int rr = isk ? r : r - len;
    const float *dh = (isk ? stk : stq) + rr * LDD, *xh = (isk ? kh : qh) + rr * LDD;
    constexpr int PER = D / 32;
    float a[PER], xv[PER], dot = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      a[i] = dh[lane + 32 * i];
      xv[i] = xh[lane + 32 * i];
      dot += a[i] * xv[i];
    }
    float *out = isk ? p.dk + ((R0 + rr) * H + h) * (int64_t)D : p.dq + ((tq0 + rr) * H + h) * (int64_t)D;
    if (p.l2norm) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      const float rx = (isk ? rk : rq)[rr];
#pragma unroll
      for (int i = 0; i < PER; ++i) out[lane + 32 * i] = rx * (a[i] - dot * xv[i]);
    } else {
#pragma unroll
      for (int i = 0; i < PER; ++i) out[lane + 32 * i] = a[i];
    }
  }
  if (tid < len) {
    if (p.dbeta) p.dbeta[(R0 + tid) * H + h] = sdb[tid];
    p.sig[(R0 + tid) * H + h] = ssg[tid];
  }
  if (tid < nq) p.rho[(tq0 + tid) * H + h] = srho[tid];
}

// ---------------------------------------------------------------------------------------
// Finishing passes.
// ---------------------------------------------------------------------------------------
// One CTA per (sequence, head): dg_t = <dS_T, S_T> + sum_{t' >= t} (rho_t' - sum_j sig_{t'M+j}).
__global__ void __launch_bounds__(256) gdp_bwd_dg_kernel(BwdProblem p) {
  const int seq = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;
  const int H = p.H, M = p.M;
  if (!p.g) {
    for (int64_t t = tid; t < L; t += 256) p.dg[(bos + t) * H + h] = 0.f;
    return;
  }
  __shared__ float sums[256];
  const int64_t per = (L + 255) / 256;
  const int64_t t0 = min(L, tid * per), t1 = min(L, t0 + per);
  auto term = [&](int64_t t) {
    float x = p.rho[(bos + t) * H + h];
    for (int j = 0; j < M; ++j) x -= p.sig[((bos + t) * M + j) * H + h];
    return x;
  };
  float s = 0.f;
  for (int64_t t = t0; t < t1; ++t) s += term(t);
  sums[tid] = s;
  __syncthreads();
  if (tid == 0) {  // exclusive suffix sums over the 256 pieces
    float run = p.tot ? p.tot[(int64_t)seq * H + h] : 0.f;
    for (int i = 255; i >= 0; --i) {
      const float x = sums[i];
      sums[i] = run;
      run += x;
    }
  }
  __syncthreads();
  float run = sums[tid];
  for (int64_t t = t1 - 1; t >= t0; --t) {
    run += term(t);
    p.dg[(bos + t) * H + h] = run;
  }
}

// Slice width of the per-chunk kernel: 16 V columns when the shared memory allows, else 8.
int chunk_slice(int d, int qpad) { return ChunkSmem(d, qpad, 16).total <= 227u * 1024u ? 16 : 8; }

template <int D, int VSL>
cudaError_t launch_chunk(const BwdProblem &p, cudaStream_t stream) {
  const size_t smem = ChunkSmem(D, p.qpad, VSL).total;
  cudaError_t e = cudaFuncSetAttribute(gdp_bwd_chunk_kernel<D, VSL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  gdp_bwd_chunk_kernel<D, VSL><<<dim3((unsigned)p.ntdp_pad, (unsigned)p.H), kChunkThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BwdProblem &p, cudaStream_t stream) {
  cudaError_t e;
  const int D = p.D, QP = p.qpad;
  if (p.N > 0 && (e = launch_bwd_tc_scan(p, stream)) != cudaSuccess) return e;
  // the tensor-core kernel addresses the state rows through TMA with 32-bit coordinates
  const bool tc = bwd_chunk_tc_serves(D, QP) && p.ntdp_pad * (int64_t)p.H * D < ((int64_t)1 << 31);
  if (p.ntdp_pad > 0 && tc) {
    if ((e = launch_bwd_chunk_tc(p, stream)) != cudaSuccess) return e;
  } else if (p.ntdp_pad > 0) {
    const int vsl = chunk_slice(D, QP);
    if (D == 128)
      e = vsl == 16 ? launch_chunk<128, 16>(p, stream) : launch_chunk<128, 8>(p, stream);
    else
      e = vsl == 16 ? launch_chunk<64, 16>(p, stream) : launch_chunk<64, 8>(p, stream);
    if (e != cudaSuccess) return e;
  }
  if (p.T > 0 && p.dg) {
    gdp_bwd_dg_kernel<<<dim3((unsigned)p.N, (unsigned)p.H), 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace gdp
