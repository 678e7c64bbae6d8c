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
// Kernels (warp-level tf32 MMAs, fp32 accumulation; the dense chunk products are small
// and varied, the serial part is the state scan):
//   gdp_bwd_scan_kernel   one CTA per (sequence, head): D = dL/dS in registers, chunks in
//                         reverse, operands from the forward's per-chunk images (TMA bulk
//                         copies, double-buffered), writes D_C of every chunk
//   gdp_bwd_chunk_kernel  one CTA per (expanded chunk, head, 32-column slice of V): the
//                         per-row gradients above; the slice's shares of dkhat, dqhat,
//                         dbeta and the dg terms are summed with atomics
//   gdp_bwd_rows_kernel   L2-norm chain rule: dx = dxhat / n - x (x . dxhat) / n^3
//   gdp_bwd_dg_kernel     reverse cumulative sum of the decay gradient per (sequence, head)
#include "gdp_internal.cuh"
#include "gdp_sm100.cuh"

namespace gdp {
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
// c += A B over ks k-steps of 8, with a(row, k) and b(k, col) relative to the tile origin.
template <class FA, class FB>
__device__ __forceinline__ void mma_tile(float *c, int ks, int g, int t, FA a, FB b) {
#pragma unroll 2
  for (int k = 0; k < ks; ++k) {
    const int k0 = 8 * k;
    mma8(c, tf32r(a(g, k0 + t)), tf32r(a(g + 8, k0 + t)), tf32r(a(g, k0 + t + 4)), tf32r(a(g + 8, k0 + t + 4)),
         tf32r(b(k0 + t, g)), tf32r(b(k0 + t + 4, g)));
  }
}

__device__ __forceinline__ float bf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// ---------------------------------------------------------------------------------------
// Reverse state scan.
// ---------------------------------------------------------------------------------------
constexpr uint32_t kBwdScanBudget = 190u * 1024u;

__host__ __device__ inline uint32_t bwd_stage_bytes(int d, int qpad) {
  return (ImageLayout(d, qpad).bytes + 1023u) & ~1023u;
}
__host__ __device__ inline int bwd_scan_stages(int d, int qpad) {
  return 2u * bwd_stage_bytes(d, qpad) + (uint32_t)qpad * (d + 8) * 4u <= kBwdScanBudget ? 2 : 1;
}
__host__ inline size_t bwd_scan_smem(int d, int qpad) {
  return (size_t)bwd_scan_stages(d, qpad) * bwd_stage_bytes(d, qpad) + (size_t)qpad * (d + 8) * 4u + 1024u;
}

template <int D>
__global__ void __launch_bounds__(2 * D, 1) gdp_bwd_scan_kernel(BwdProblem p) {
  constexpr int NW = D / 16;  // warps; warp w holds state rows 16 w .. 16 w + 15
  constexpr int LDO = D + 8;  // row stride of the staged d_output rows (conflict-free A loads)
  const int seq = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;
  const int M = p.M, QP = p.qpad, H = p.H;
  const ImageLayout il(D, QP);
  const uint32_t sbytes = bwd_stage_bytes(D, QP);
  const int nst = bwd_scan_stages(D, QP);
  extern __shared__ __align__(1024) unsigned char bwd_scan_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)bwd_scan_raw + 1023) & ~(uintptr_t)1023);
  float *dos = reinterpret_cast<float *>(sm + nst * sbytes);
  __shared__ __align__(8) uint64_t full[2];
  __shared__ float red[NW];
  const int64_t KV = (int64_t)D * D, sh = (int64_t)seq * H + h;
  const int64_t nchunks = (L * M + kChunk - 1) / kChunk;
  const int64_t cod_i = p.cod[seq];
  const int64_t nall = (cod_i < 0) ? 0 : max((int64_t)0, min(nchunks, p.ws_rows - cod_i));
  const int r0 = 16 * warp + g;  // this thread's rows r0 and r0 + 8

  // D = dL/dS_final; <dS_final, S_final> for the decay gradient
  float dacc[D / 8][4];
  {
    const float *src = p.dfin ? p.dfin + sh * KV : nullptr;
    const float *fin = (p.dfin && p.fin) ? p.fin + sh * KV : nullptr;
    float part = 0.f;
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int64_t off = (int64_t)(r0 + 8 * hf) * D + 8 * j + 2 * t;
        const float2 x = src ? *reinterpret_cast<const float2 *>(src + off) : make_float2(0.f, 0.f);
        dacc[j][2 * hf] = x.x;
        dacc[j][2 * hf + 1] = x.y;
        if (fin) {
          const float2 s = *reinterpret_cast<const float2 *>(fin + off);
          part += x.x * s.x + x.y * s.y;
        }
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) red[warp] = part;
  }
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0 && p.tot) {
    float s = 0.f;
    for (int w = 0; w < NW; ++w) s += red[w];
    p.tot[sh] = s;
  }
  auto image = [&](int64_t e) { return p.img + (size_t)((cod_i + e) * H + h) * p.img_stride; };
  int issued[2] = {0, 0};
  auto issue = [&](int64_t i) {  // chunk nall - 1 - i into stage i % nst (thread 0)
    const int st = (int)(i % nst);
    mbar_arrive_expect_tx(&full[st], il.bytes);
    bulk_g2s(sm + st * sbytes, image(nall - 1 - i), il.bytes, &full[st]);
    ++issued[st];
  };
  if (tid == 0)
    for (int64_t i = 0; i < nst && i < nall; ++i) issue(i);

  bool aborted = false;
  for (int64_t i = 0; i < nall; ++i) {
    const int64_t e = nall - 1 - i;
    const int st = (int)(i % nst);
    const unsigned char *im = sm + st * sbytes;
    // the gradient at chunk e's exit
    float *dst = p.Dx + ((cod_i + e) * H + h) * KV;
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        *reinterpret_cast<float2 *>(dst + (int64_t)(r0 + 8 * hf) * D + 8 * j + 2 * t) =
            make_float2(dacc[j][2 * hf], dacc[j][2 * hf + 1]);
    // d_output rows of the chunk's readouts (fp32, zero past the readout count)
    const ImageMeta mt = *reinterpret_cast<const ImageMeta *>(image(e) + il.meta);
    const int64_t tq0 = (bos * M + e * kChunk + mt.p0) / M;
    for (int idx = tid; idx < QP * (D / 4); idx += 32 * NW) {
      const int qi = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (qi < mt.nq) {
        const __nv_bfloat16 *src = p.dout + ((tq0 + qi) * H + h) * (int64_t)D + c4;
        const uint2 u = *reinterpret_cast<const uint2 *>(src);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
        x = make_float4(a.x, a.y, b.x, b.y);
      }
      *reinterpret_cast<float4 *>(dos + qi * LDO + c4) = x;
    }
    const bool ok = mbar_wait(&full[st], (uint32_t)((i / nst) & 1));
    if (!__syncthreads_and(ok)) {
      aborted = true;
      break;
    }
    auto ld = [&](uint32_t off) { return *reinterpret_cast<const float *>(im + off); };
    // Z = D Ktil^T + dO^T P  (rows v of this warp x 64 chunk rows s).  The D fragments serve
    // as A with the k order permuted within each 8-column step (logical k = t <-> column
    // 2t, k = t + 4 <-> column 2t + 1); B is read in the same order.
    float z[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) z[n][0] = z[n][1] = z[n][2] = z[n][3] = 0.f;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      const uint32_t a0 = tf32r(dacc[j][0]), a1 = tf32r(dacc[j][2]), a2 = tf32r(dacc[j][1]), a3 = tf32r(dacc[j][3]);
      const int f0 = 8 * j + 2 * t;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int s = 8 * n + g;
        mma8(z[n], a0, a1, a2, a3, tf32r(ld(il.kt(f0, s))), tf32r(ld(il.kt(f0 + 1, s))));
      }
    }
    for (int k0 = 0; k0 < QP; k0 += 8) {
      const uint32_t a0 = tf32r(dos[(k0 + t) * LDO + r0]), a1 = tf32r(dos[(k0 + t) * LDO + r0 + 8]),
                     a2 = tf32r(dos[(k0 + t + 4) * LDO + r0]), a3 = tf32r(dos[(k0 + t + 4) * LDO + r0 + 8]);
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int s = 8 * n + g;
        mma8(z[n], a0, a1, a2, a3, tf32r(ld(il.pm(D, k0 + t, s))), tf32r(ld(il.pm(D, k0 + t + 4, s))));
      }
    }
    // D_in = gamma_C D + Z (-W) + dO^T Qh; a fast image holds -W and Qh divided by gamma_C
    const float gam = mt.gamma_last;
    if (!mt.fast)
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x) dacc[j][x] *= gam;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t a0 = tf32r(z[ks][0]), a1 = tf32r(z[ks][2]), a2 = tf32r(z[ks][1]), a3 = tf32r(z[ks][3]);
      const int s0 = 8 * ks + 2 * t;
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        const int f = 8 * j + g;
        mma8(dacc[j], a0, a1, a2, a3, tf32r(ld(il.wn(QP, s0, f))), tf32r(ld(il.wn(QP, s0 + 1, f))));
      }
    }
    for (int k0 = 0; k0 < QP; k0 += 8) {
      const uint32_t a0 = tf32r(dos[(k0 + t) * LDO + r0]), a1 = tf32r(dos[(k0 + t) * LDO + r0 + 8]),
                     a2 = tf32r(dos[(k0 + t + 4) * LDO + r0]), a3 = tf32r(dos[(k0 + t + 4) * LDO + r0 + 8]);
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        const int f = 8 * j + g;
        mma8(dacc[j], a0, a1, a2, a3, tf32r(ld(il.qh(k0 + t, f))), tf32r(ld(il.qh(k0 + t + 4, f))));
      }
    }
    if (mt.fast)
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
#pragma unroll
        for (int x = 0; x < 4; ++x) dacc[j][x] *= gam;
    __syncthreads();  // every warp is done with this stage and with dos
    if (tid == 0 && i + nst < nall) issue(i + nst);
  }
  if (aborted) {
    if (tid == 0) {
      set_status(p.status, GDP_DEV_ERR_TIMEOUT);
      for (int st = 0; st < nst; ++st)  // bounded: the copies issued on each stage have landed
        if (issued[st] > 0) mbar_wait(&full[st], (uint32_t)((issued[st] - 1) & 1));
    }
    __syncthreads();
    return;
  }
  if (p.dinit) {
    float *dst = p.dinit + sh * KV;
#pragma unroll
    for (int j = 0; j < D / 8; ++j)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        *reinterpret_cast<float2 *>(dst + (int64_t)(r0 + 8 * hf) * D + 8 * j + 2 * t) =
            make_float2(dacc[j][2 * hf], dacc[j][2 * hf + 1]);
  }
}

// ---------------------------------------------------------------------------------------
// Per-chunk gradients.
// ---------------------------------------------------------------------------------------
constexpr int kVS = 32;        // V columns per CTA
constexpr int kLS = kVS + 4;   // row stride of [rows][kVS] tiles
constexpr int kLC = kChunk + 4;  // row stride of [rows][64] tiles

struct ChunkSmem {
  uint32_t kh, qh, vs, dos, ss, dcs, lm, pm, et, vt, dl, qs, m1, m3, scal, total;
  __host__ __device__ ChunkSmem(int d, int qp) {
    const uint32_t ld = (uint32_t)(d + 4) * 4u;
    uint32_t o = 0;
    kh = o; o += kChunk * ld;           // khat [64][d]
    qh = o; o += qp * ld;               // qhat readout rows [qp][d]
    vs = o; o += kChunk * kLS * 4u;     // v slice [64][32]
    dos = o; o += qp * kLS * 4u;        // d_output slice [qp][32]
    ss = o; o += kVS * ld;              // S slice [32][d]
    dcs = o; o += kVS * ld;             // D_C slice [32][d]
    lm = o; o += kChunk * kLC * 4u;     // L, then M2 [64][64]
    pm = o; o += qp * kLC * 4u;         // P, then M4 [qp][64]
    et = o; o += kChunk * kLS * 4u;     // rhs, then e [64][32]
    vt = o; o += kChunk * kLS * 4u;     // vt [64][32]
    dl = o; o += kChunk * kLS * 4u;     // Zt, then Delta [64][32]
    qs = o; o += qp * kLS * 4u;         // qhat S^T [qp][32]
    m1 = o; o += kChunk * (qp + 4) * 4u;  // M1 [64][qp]
    m3 = o; o += kChunk * kLC * 4u;     // M3 [64][64]
    scal = o; o += 5u * kChunk * 4u;    // G, beta, rk, rq, gamma
    total = o;
  }
};

template <int D>
__global__ void __launch_bounds__(256, 1) gdp_bwd_chunk_kernel(BwdProblem p) {
  constexpr int LD = D + 4;
  const int row = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * kVS;
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
  const int64_t srow = (int64_t)p.cod[seq] + c;  // state rows of this chunk in Sx / Dx

  extern __shared__ __align__(16) unsigned char bwd_chunk_raw[];
  const ChunkSmem lay(D, QP);
  unsigned char *sm = bwd_chunk_raw;
  float *kh = reinterpret_cast<float *>(sm + lay.kh), *qh = reinterpret_cast<float *>(sm + lay.qh);
  float *vs = reinterpret_cast<float *>(sm + lay.vs), *dos = reinterpret_cast<float *>(sm + lay.dos);
  float *ss = reinterpret_cast<float *>(sm + lay.ss), *dcs = reinterpret_cast<float *>(sm + lay.dcs);
  float *lm = reinterpret_cast<float *>(sm + lay.lm), *pm = reinterpret_cast<float *>(sm + lay.pm);
  float *et = reinterpret_cast<float *>(sm + lay.et), *vt = reinterpret_cast<float *>(sm + lay.vt);
  float *dl = reinterpret_cast<float *>(sm + lay.dl), *qs = reinterpret_cast<float *>(sm + lay.qs);
  float *m1 = reinterpret_cast<float *>(sm + lay.m1), *m3 = reinterpret_cast<float *>(sm + lay.m3);
  float *G = reinterpret_cast<float *>(sm + lay.scal), *bt = G + kChunk, *rk = bt + kChunk, *rq = rk + kChunk,
        *gm = rq + kChunk;
  const int LM1 = QP + 4;
  __shared__ float carry;

  // ---- scalars: beta, gates, within-chunk cumulative log decay ----
  if (tid < kChunk) {
    const int r = tid;
    const int pos = r0m + r;
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
  }
  // ---- khat rows (4 threads per row), qhat readout rows, slices of v, d_output, S, D_C ----
  {
    const int r = tid >> 2, part = tid & 3;  // 64 rows x 4 parts of D / 4 features
    float x[D / 4];
    float ss2 = 0.f;
    const bool live = r < len;
    const __nv_bfloat16 *src = p.k + (R0 + r) * p.k_st + (int64_t)h * p.k_sh + part * (D / 4);
#pragma unroll
    for (int i = 0; i < D / 4; i += 8) {
      uint4 u = make_uint4(0u, 0u, 0u, 0u);
      if (live) u = *reinterpret_cast<const uint4 *>(src + i);
      const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const float2 f = __bfloat1622float2(b2[q2]);
        x[i + 2 * q2] = f.x;
        x[i + 2 * q2 + 1] = f.y;
        ss2 += f.x * f.x + f.y * f.y;
      }
    }
    ss2 += __shfl_xor_sync(0xffffffffu, ss2, 1);
    ss2 += __shfl_xor_sync(0xffffffffu, ss2, 2);
    const float inv = p.l2norm ? rsqrtf(ss2 + kL2Eps) : 1.f;
    if (part == 0) rk[r] = inv;
#pragma unroll
    for (int i = 0; i < D / 4; i += 4)
      *reinterpret_cast<float4 *>(kh + r * LD + part * (D / 4) + i) =
          make_float4(x[i] * inv, x[i + 1] * inv, x[i + 2] * inv, x[i + 3] * inv);
  }
  for (int r = tid >> 2; r < QP; r += 64) {
    const int part = tid & 3;
    float x[D / 4];
    float ss2 = 0.f;
    const bool live = r < nq;
    const __nv_bfloat16 *src = p.q + (tq0 + r) * p.q_st + (int64_t)h * p.q_sh + part * (D / 4);
#pragma unroll
    for (int i = 0; i < D / 4; i += 8) {
      uint4 u = make_uint4(0u, 0u, 0u, 0u);
      if (live) u = *reinterpret_cast<const uint4 *>(src + i);
      const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const float2 f = __bfloat1622float2(b2[q2]);
        x[i + 2 * q2] = f.x;
        x[i + 2 * q2 + 1] = f.y;
        ss2 += f.x * f.x + f.y * f.y;
      }
    }
    ss2 += __shfl_xor_sync(0xffffffffu, ss2, 1);
    ss2 += __shfl_xor_sync(0xffffffffu, ss2, 2);
    const float inv = p.l2norm ? rsqrtf(ss2 + kL2Eps) : 1.f;
    if (part == 0) rq[r] = inv;
#pragma unroll
    for (int i = 0; i < D / 4; i += 4)
      *reinterpret_cast<float4 *>(qh + r * LD + part * (D / 4) + i) =
          make_float4(x[i] * inv, x[i + 1] * inv, x[i + 2] * inv, x[i + 3] * inv);
  }
  for (int idx = tid; idx < kChunk * (kVS / 4); idx += 256) {  // v slice
    const int r = idx / (kVS / 4), c4 = (idx % (kVS / 4)) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < len) {
      const uint2 u = *reinterpret_cast<const uint2 *>(p.v + (R0 + r) * p.v_st + (int64_t)h * p.v_sh + v0 + c4);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
      x = make_float4(a.x, a.y, b.x, b.y);
    }
    *reinterpret_cast<float4 *>(vs + r * kLS + c4) = x;
  }
  for (int idx = tid; idx < QP * (kVS / 4); idx += 256) {  // d_output slice
    const int r = idx / (kVS / 4), c4 = (idx % (kVS / 4)) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nq) {
      const uint2 u = *reinterpret_cast<const uint2 *>(p.dout + ((tq0 + r) * H + h) * (int64_t)D + v0 + c4);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
      x = make_float4(a.x, a.y, b.x, b.y);
    }
    *reinterpret_cast<float4 *>(dos + r * kLS + c4) = x;
  }
  {
    const int64_t KV = (int64_t)D * D;
    const float *S = p.Sx + (srow * H + h) * KV + (int64_t)v0 * D;
    const float *Dc = p.Dx + (srow * H + h) * KV + (int64_t)v0 * D;
    for (int idx = tid; idx < kVS * (D / 4); idx += 256) {
      const int r = idx / (D / 4), c4 = (idx % (D / 4)) * 4;
      *reinterpret_cast<float4 *>(ss + r * LD + c4) = *reinterpret_cast<const float4 *>(S + (int64_t)r * D + c4);
      *reinterpret_cast<float4 *>(dcs + r * LD + c4) = *reinterpret_cast<const float4 *>(Dc + (int64_t)r * D + c4);
    }
  }
  __syncthreads();
  if (tid < kChunk) {
    const float x = (tid >= 32 ? G[tid] + carry : G[tid]);
    G[tid] = x;
    gm[tid] = expf(x);
  }
  __syncthreads();
  const float GC = G[len - 1], scale = p.scale;
  auto pr = [&](int qi) { return p0 + qi * M; };  // local row of readout qi

  // ---- Gram products: L (64 x 64) and P (qp x 64) ----
  for (int u = warp; u < 4 * 8 + (QP / 16) * 8; u += 8) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const bool isL = u < 32;
    const int uu = isL ? u : u - 32;
    const int m0 = 16 * (uu >> 3), n0 = 8 * (uu & 7);
    const float *A = isL ? kh : qh;
    mma_tile(acc, D / 8, g, t, [&](int r, int k) { return A[(m0 + r) * LD + k]; },
             [&](int k, int n) { return kh[(n0 + n) * LD + k]; });
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int r = m0 + g + 8 * (x >> 1), j = n0 + 2 * t + (x & 1);
      if (isL) {
        lm[r * kLC + j] = (j < r) ? expf(G[r] - G[j]) * acc[x] : 0.f;
      } else {
        const int pp = pr(r);
        pm[r * kLC + j] = (r < nq && j <= pp) ? scale * expf(G[pp] - G[j]) * acc[x] : 0.f;
      }
    }
  }
  __syncthreads();
  // ---- rhs = v - gamma (Khat S^T);  qhat S^T;  Zt = Ktil D_C^T + P^T dO ----
  for (int u = warp; u < 16 + (QP / 16) * 4 + 16; u += 8) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (u < 16) {
      const int m0 = 16 * (u >> 2), n0 = 8 * (u & 3);
      mma_tile(acc, D / 8, g, t, [&](int r, int k) { return kh[(m0 + r) * LD + k]; },
               [&](int k, int n) { return ss[(n0 + n) * LD + k]; });
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int r = m0 + g + 8 * (x >> 1), j = n0 + 2 * t + (x & 1);
        et[r * kLS + j] = vs[r * kLS + j] - gm[r] * acc[x];
      }
    } else if (u < 16 + (QP / 16) * 4) {
      const int uu = u - 16, m0 = 16 * (uu >> 2), n0 = 8 * (uu & 3);
      mma_tile(acc, D / 8, g, t, [&](int r, int k) { return qh[(m0 + r) * LD + k]; },
               [&](int k, int n) { return ss[(n0 + n) * LD + k]; });
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int r = m0 + g + 8 * (x >> 1), j = n0 + 2 * t + (x & 1);
        qs[r * kLS + j] = acc[x];
      }
    } else {
      const int uu = u - 16 - (QP / 16) * 4, m0 = 16 * (uu >> 2), n0 = 8 * (uu & 3);
      mma_tile(acc, D / 8, g, t, [&](int r, int k) { return expf(GC - G[m0 + r]) * kh[(m0 + r) * LD + k]; },
               [&](int k, int n) { return dcs[(n0 + n) * LD + k]; });
      mma_tile(acc, QP / 8, g, t, [&](int r, int k) { return pm[k * kLC + m0 + r]; },
               [&](int k, int n) { return dos[k * kLS + n0 + n]; });
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int r = m0 + g + 8 * (x >> 1), j = n0 + 2 * t + (x & 1);
        dl[r * kLS + j] = acc[x];
      }
    }
  }
  __syncthreads();
  // ---- substitutions, per column (8 threads per column, row terms split by j mod 8) ----
  {
    const int col = tid >> 3, i = tid & 7;
    float hist[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // e_r = rhs_r - sum_{j<r} L_rj vt_j;  vt_r = beta_r e_r
#pragma unroll
    for (int r = 0; r < kChunk; ++r) {
      float part = 0.f;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (8 * jj < r) {  // rows j = 8 jj + i < r (the entries of L at j >= r are zero)
          part += lm[r * kLC + 8 * jj + i] * hist[jj];
        }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      part += __shfl_xor_sync(0xffffffffu, part, 4);
      const float e = et[r * kLS + col] - part;
      const float vv = bt[r] * e;
      if ((r & 7) == i) {
        hist[r >> 3] = vv;
        et[r * kLS + col] = e;
        vt[r * kLS + col] = vv;
      }
    }
    // Delta_r = Zt_r - sum_{j>r} beta_j L_jr Delta_j
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) hist[jj] = 0.f;
#pragma unroll
    for (int r = kChunk - 1; r >= 0; --r) {
      float part = 0.f;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj)
        if (8 * jj + 7 > r) {
          const int j = 8 * jj + i;
          part += (j > r) ? bt[j] * lm[j * kLC + r] * hist[jj] : 0.f;
        }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      part += __shfl_xor_sync(0xffffffffu, part, 4);
      const float dd = dl[r * kLS + col] - part;
      if ((r & 7) == i) {
        hist[r >> 3] = dd;
        dl[r * kLS + col] = dd;
      }
    }
  }
  __syncthreads();
  // ---- dv (this slice), and the slice's shares of dbeta and of sum_v dv v ----
  for (int r = warp; r < len; r += 8) {
    const float d = dl[r * kLS + lane], b = bt[r];
    p.dv[((R0 + r) * H + h) * (int64_t)D + v0 + lane] = b * d;
    float sdb = et[r * kLS + lane] * d, ssg = b * d * vs[r * kLS + lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sdb += __shfl_xor_sync(0xffffffffu, sdb, o);
      ssg += __shfl_xor_sync(0xffffffffu, ssg, o);
    }
    if (lane == 0) {
      if (p.dbeta) atomicAdd(p.dbeta + (R0 + r) * H + h, sdb);
      atomicAdd(p.sig + (R0 + r) * H + h, ssg);
    }
  }
  // ---- o (this slice) = scale gamma_p (qhat S^T) + P vt, and the slice's share of do . o ----
  for (int u = warp; u < (QP / 16) * 4; u += 8) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int m0 = 16 * (u >> 2), n0 = 8 * (u & 3);
    mma_tile(acc, kChunk / 8, g, t, [&](int r, int k) { return pm[(m0 + r) * kLC + k]; },
             [&](int k, int n) { return vt[k * kLS + n0 + n]; });
    float part[2] = {0.f, 0.f};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int r = m0 + g + 8 * (x >> 1), j = n0 + 2 * t + (x & 1);
      const float o = (r < nq) ? scale * gm[pr(r)] * qs[r * kLS + j] + acc[x] : 0.f;
      part[x >> 1] += o * dos[r * kLS + j];
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      float s = part[hf];
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      const int r = m0 + g + 8 * hf;
      if (t == 0 && r < nq) atomicAdd(p.rho + (tq0 + r) * H + h, s);
    }
  }
  __syncthreads();
  // ---- M1 [64 x qp], M2 [64 x 64] (into L), M3 [64 x 64], M4 [qp x 64] (into P) ----
  {
    const int n1 = 4 * (QP / 8), n2 = 32, n3 = 32, n4 = (QP / 16) * 8;
    for (int u = warp; u < n1 + n2 + n3 + n4; u += 8) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (u < n1) {  // e dO^T
        const int m0 = 16 * (u / (QP / 8)), c0 = 8 * (u % (QP / 8));
        mma_tile(acc, kVS / 8, g, t, [&](int r, int k) { return et[(m0 + r) * kLS + k]; },
                 [&](int k, int n) { return dos[(c0 + n) * kLS + k]; });
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int r = m0 + g + 8 * (x >> 1), qi = c0 + 2 * t + (x & 1);
          const int pp = pr(qi);
          m1[r * LM1 + qi] = (qi < nq && r <= pp) ? scale * expf(G[pp] - G[r]) * acc[x] : 0.f;
        }
      } else if (u < n1 + n2) {  // e dv^T
        const int uu = u - n1, m0 = 16 * (uu >> 3), c0 = 8 * (uu & 7);
        mma_tile(acc, kVS / 8, g, t, [&](int r, int k) { return et[(m0 + r) * kLS + k]; },
                 [&](int k, int n) { return bt[c0 + n] * dl[(c0 + n) * kLS + k]; });
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int r = m0 + g + 8 * (x >> 1), j = c0 + 2 * t + (x & 1);
          lm[r * kLC + j] = (j > r) ? expf(G[j] - G[r]) * acc[x] : 0.f;
        }
      } else if (u < n1 + n2 + n3) {  // dv vt^T
        const int uu = u - n1 - n2, m0 = 16 * (uu >> 3), c0 = 8 * (uu & 7);
        mma_tile(acc, kVS / 8, g, t, [&](int r, int k) { return bt[m0 + r] * dl[(m0 + r) * kLS + k]; },
                 [&](int k, int n) { return vt[(c0 + n) * kLS + k]; });
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int r = m0 + g + 8 * (x >> 1), j = c0 + 2 * t + (x & 1);
          m3[r * kLC + j] = (j < r) ? expf(G[r] - G[j]) * acc[x] : 0.f;
        }
      } else {  // dO vt^T
        const int uu = u - n1 - n2 - n3, m0 = 16 * (uu >> 3), c0 = 8 * (uu & 7);
        mma_tile(acc, kVS / 8, g, t, [&](int r, int k) { return dos[(m0 + r) * kLS + k]; },
                 [&](int k, int n) { return vt[(c0 + n) * kLS + k]; });
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int qi = m0 + g + 8 * (x >> 1), j = c0 + 2 * t + (x & 1);
          const int pp = pr(qi);
          pm[qi * kLC + j] = (qi < nq && j <= pp) ? expf(G[pp] - G[j]) * acc[x] : 0.f;
        }
      }
    }
  }
  __syncthreads();
  // ---- the slice's shares of dkhat [64 x D] and dqhat [qp x D] ----
  for (int u = warp; u < 4 * (D / 8) + (QP / 16) * (D / 8); u += 8) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (u < 4 * (D / 8)) {
      const int m0 = 16 * (u / (D / 8)), f0 = 8 * (u % (D / 8));
      // (beta gamma_C / gamma) e D_C
      mma_tile(acc, kVS / 8, g, t,
               [&](int r, int k) { return bt[m0 + r] * expf(GC - G[m0 + r]) * et[(m0 + r) * kLS + k]; },
               [&](int k, int n) { return dcs[k * LD + f0 + n]; });
      // - gamma dv S
      mma_tile(acc, kVS / 8, g, t,
               [&](int r, int k) { return -gm[m0 + r] * bt[m0 + r] * dl[(m0 + r) * kLS + k]; },
               [&](int k, int n) { return ss[k * LD + f0 + n]; });
      // beta M1 qhat
      mma_tile(acc, QP / 8, g, t, [&](int r, int k) { return bt[m0 + r] * m1[(m0 + r) * LM1 + k]; },
               [&](int k, int n) { return qh[k * LD + f0 + n]; });
      // - (beta M2 + M3) khat
      mma_tile(acc, kChunk / 8, g, t,
               [&](int r, int k) { return -(bt[m0 + r] * lm[(m0 + r) * kLC + k] + m3[(m0 + r) * kLC + k]); },
               [&](int k, int n) { return kh[k * LD + f0 + n]; });
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = m0 + g + 8 * hf;
        if (r < len)
          atomicAdd(reinterpret_cast<float2 *>(p.dkh + ((R0 + r) * H + h) * (int64_t)D + f0 + 2 * t),
                    make_float2(acc[2 * hf], acc[2 * hf + 1]));
      }
    } else {
      const int uu = u - 4 * (D / 8), m0 = 16 * (uu / (D / 8)), f0 = 8 * (uu % (D / 8));
      // scale gamma_p dO S
      mma_tile(acc, kVS / 8, g, t,
               [&](int r, int k) {
                 const int qi = m0 + r;
                 return qi < nq ? scale * gm[pr(qi)] * dos[qi * kLS + k] : 0.f;
               },
               [&](int k, int n) { return ss[k * LD + f0 + n]; });
      // scale M4 khat
      mma_tile(acc, kChunk / 8, g, t, [&](int r, int k) { return scale * pm[(m0 + r) * kLC + k]; },
               [&](int k, int n) { return kh[k * LD + f0 + n]; });
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int qi = m0 + g + 8 * hf;
        if (qi < nq)
          atomicAdd(reinterpret_cast<float2 *>(p.dqh + ((tq0 + qi) * H + h) * (int64_t)D + f0 + 2 * t),
                    make_float2(acc[2 * hf], acc[2 * hf + 1]));
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Finishing passes.
// ---------------------------------------------------------------------------------------
// One warp per (row, head): dx = dxhat / n - x (x . dxhat) / n^3 with n = sqrt(|x|^2 + eps)
// (or dx = dxhat without the L2 norm).  blockIdx.y: 0 = k rows (T*M), 1 = q rows (T).
template <int D>
__global__ void __launch_bounds__(256) gdp_bwd_rows_kernel(BwdProblem p) {
  const int which = blockIdx.y;
  const int64_t rows = (which == 0 ? p.T * p.M : p.T) * p.H;
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= rows) return;
  const int64_t r = w / p.H;
  const int h = (int)(w % p.H);
  const float *acc = (which == 0 ? p.dkh : p.dqh) + w * D;
  float *out = (which == 0 ? p.dk : p.dq) + w * D;
  const __nv_bfloat16 *x = which == 0 ? p.k + r * p.k_st + (int64_t)h * p.k_sh : p.q + r * p.q_st + (int64_t)h * p.q_sh;
  constexpr int PER = D / 32;
  float a[PER], xv[PER], ss = 0.f, dot = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    a[i] = acc[lane * PER + i];
    xv[i] = bf(x + lane * PER + i);
    ss += xv[i] * xv[i];
    dot += xv[i] * a[i];
  }
  if (p.l2norm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ss += __shfl_xor_sync(0xffffffffu, ss, o);
      dot += __shfl_xor_sync(0xffffffffu, dot, o);
    }
    const float inv = rsqrtf(ss + kL2Eps), inv3 = inv * inv * inv;
#pragma unroll
    for (int i = 0; i < PER; ++i) out[lane * PER + i] = a[i] * inv - xv[i] * dot * inv3;
  } else {
#pragma unroll
    for (int i = 0; i < PER; ++i) out[lane * PER + i] = a[i];
  }
}

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

}  // namespace

cudaError_t launch_backward(const BwdProblem &p, cudaStream_t stream) {
  cudaError_t e;
  const int D = p.D, QP = p.qpad;
  if (p.N > 0) {
    const size_t smem = bwd_scan_smem(D, QP);
    dim3 grid((unsigned)p.N, (unsigned)p.H);
    if (D == 128) {
      if ((e = cudaFuncSetAttribute(gdp_bwd_scan_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem)) != cudaSuccess)
        return e;
      gdp_bwd_scan_kernel<128><<<grid, 256, smem, stream>>>(p);
    } else {
      if ((e = cudaFuncSetAttribute(gdp_bwd_scan_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem)) != cudaSuccess)
        return e;
      gdp_bwd_scan_kernel<64><<<grid, 128, smem, stream>>>(p);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (p.ntdp_pad > 0) {
    const size_t smem = ChunkSmem(D, QP).total;
    dim3 grid((unsigned)p.ntdp_pad, (unsigned)p.H, (unsigned)(D / kVS));
    if (D == 128) {
      if ((e = cudaFuncSetAttribute(gdp_bwd_chunk_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem)) != cudaSuccess)
        return e;
      gdp_bwd_chunk_kernel<128><<<grid, 256, smem, stream>>>(p);
    } else {
      if ((e = cudaFuncSetAttribute(gdp_bwd_chunk_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem)) != cudaSuccess)
        return e;
      gdp_bwd_chunk_kernel<64><<<grid, 256, smem, stream>>>(p);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (p.T > 0) {
    const int64_t rows = p.T * p.M * p.H;
    dim3 grid((unsigned)((rows + 7) / 8), 2);
    if (D == 128)
      gdp_bwd_rows_kernel<128><<<grid, 256, 0, stream>>>(p);
    else
      gdp_bwd_rows_kernel<64><<<grid, 256, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (p.dg) {
      gdp_bwd_dg_kernel<<<dim3((unsigned)p.N, (unsigned)p.H), 256, 0, stream>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

size_t backward_chunk_smem(int d, int qpad) { return ChunkSmem(d, qpad).total; }

}  // namespace gdp
