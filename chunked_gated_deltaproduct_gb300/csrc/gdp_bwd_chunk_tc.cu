// gdp_bwd_chunk_tc.cu -- the backward pass's per-chunk gradients on the tcgen05 tensor cores
// (head size 128 and at most 32 readout rows per expanded chunk, i.e. two or more Householder
// updates per token; gdp_bwd_chunk_kernel in gdp_backward.cu serves the other shapes).
//
// The algebra is the one gdp_backward.cu derives from the recurrence (FlashInfer API page
// "flashinfer.gdp_prefill.chunk_gated_delta_product", display equation); for one expanded chunk
// (rows r, j < 64, readout rows p < qpad, entering state S and exit gradient D_C, both [V][K]):
//   rhs = V - diag(gamma) Khat S^T,  QS = Qhat S^T,  Zt = diag(gamma_C/gamma) Khat D_C^T + P^T dO
//   vt  = T diag(beta) rhs,          Delta = T^T Zt
//   e   = rhs - L vt,                o = diag(scale gamma_p) QS + P vt
//   dv  = diag(beta) Delta,  dbeta_r = e_r . Delta_r,  sig_r = beta_r Delta_r . v_r,  rho_p = dO_p . o_p
//   G1 = e dO^T, G2 = e dv^T, G3 = dv vt^T, G4 = dO vt^T     (sums over V)
//   dkhat = diag(beta gamma_C/gamma) e D_C - diag(gamma beta) Delta S + (beta M1) Qhat - M23 Khat
//   dqhat = diag(scale gamma_p) dO S + M4 Khat
// with M1, M23 = beta M2 (upper) + M3 (lower), M4 the masked, decayed G1 .. G4.
//
// Every product is a kind::tf32 MMA (M = 128, fp32 accumulators in TMEM) whose operands are
// K-major 128-byte-swizzled fp32 tiles in shared memory, except the products that contract over
// V and leave dkhat / dqhat: their A operands -- the slice's D_C^T and S^T, then Qhat^T and
// Khat^T -- are written into TMEM (lanes = the K index), so that no state slice is transposed in
// shared memory.  64-row operands are stacked in pairs to fill M = 128: [Khat; Qhat] against the
// state slice gives rhs and QS in one accumulator, [T; T^T] against [beta rhs^T; Zt^T] gives vt and
// Delta, [L T; P T] (formed once per chunk) against beta rhs^T gives L vt and P vt in the same
// batch, [e; vt] against [dv; dO] gives the four Gram sums at once.  V runs in four slices of 32
// columns, the slice's S and D_C rows brought by TMA (double-buffered, a slice ahead); per slice
// two MMA round trips alternate with the threads' epilogues (the accumulator rows on the TMEM lanes
// are written back as the next batch's operand tiles), the slice's last products (Gram sums,
// dkhat^T, dqhat^T, which stay in TMEM across the slices) going out with the next slice's first.
// The masked, decayed Gram sums feed one last batch.  The threads round every operand they write
// to the nearest tf32 value (the tensor cores would otherwise drop the low mantissa bits, which
// doubled the gradients' error against the float64 oracle); the state slices that TMA brings are
// taken as they are.  The triangular products with T run in plain tf32 as well: against the
// oracle, the 3xTF32 split changed the gradients' relative error by less than 1e-4.
//
// One CTA of 256 threads per (expanded chunk, head): warp w reads TMEM lane quadrant w % 4 and the
// half w / 4 of the columns; thread 0 issues the MMAs and the TMA loads.  Every wait is bounded
// (GDP_DEV_ERR_TIMEOUT on expiry).
#include <cuda.h>

#include "gdp_internal.cuh"
#include "gdp_sm100.cuh"

namespace gdp {
namespace {

using namespace sm100;

constexpr int kCtThreads = 256;
constexpr int kCtVs = 32;  // V columns per slice
constexpr int kCtD = 128;  // head size served
constexpr int kCtSlices = kCtD / kCtVs;

// Byte offset of element (row r, column c) of a K-major 128B-swizzled fp32 tile whose K blocks
// (32 columns each) hold `rows` rows.
__device__ __forceinline__ uint32_t toff(uint32_t rows, int r, int c) {
  return (uint32_t)(c >> 5) * rows * 128u + swz((uint32_t)r, (uint32_t)(c & 31) * 4u);
}

// Shared-memory plan (bytes from a 1024-aligned base).  The M = 128 products over 64 + qpad valid
// rows read the rows past the valid ones from the region that follows (their accumulator lanes are
// never read).
struct CtLayout {
  uint32_t rkq, kq, tt, lp, pt, b1, dot, b2, dl, fb, fq, raw5, gb, dqb, stk, stq, total;
  static constexpr uint32_t kB1 = 4u * 64u * 128u;  // one slice buffer
  __host__ __device__ uint32_t b1s(int s) const { return b1 + (uint32_t)(s & 1) * kB1; }
  __host__ __device__ CtLayout(int qp) {
    rkq = 64u + (uint32_t)qp;
    uint32_t o = 0;
    auto take = [&](uint32_t bytes) {
      const uint32_t at = o;
      o += (bytes + 1023u) & ~1023u;
      return at;
    };
    kq = take(4u * rkq * 128u);  // [Khat; Qhat], K = d
    tt = take(2u * 128u * 128u); // [T; T^T], K = 64
    lp = take(2u * rkq * 128u);  // [L; P], K = 64; then [L T; P T]
    pt = take(64u * 128u);       // P^T rows r, K = qpad
    b1 = take(2u * kB1);         // two slice buffers: [S_s; D_s] rows v, K = d (TMA), then [e_s; vt_s]
                                 // (K = VS, 128 rows) and [bfc e_s | -gamma beta Delta_s] (rows r, K = 2 VS)
    fb = b1;                  // at the end [beta M1 | -M23] rows r, K = qpad + 64
    dot = take(32u * 128u);      // dO_s^T rows v, K = qpad
    b2 = take(2u * 64u * 128u);  // [beta rhs^T; Zt^T] rows n, K = 64
    dl = b2 + 2u * 32u * 128u;   //   then Delta_s [64][32] (16-byte chunks swizzled by row)
    fq = b2 + 2u * 32u * 128u;   //   at the end scale M4 rows p, K = 64 (after the Gram staging)
    gb = take(rkq * 128u);       // [dv_s; dO_s], K = VS
    dqb = take((uint32_t)qp * 128u);  // scale gamma_p dO_s rows p, K = VS
    raw5 = b1 + 3u * 64u * 128u; // the Gram sums as they leave TMEM, [128][kRawLd] (after fb)
    stk = b1;                    // the last staging: dkhat [64][132], dqhat [qpad][132]
    stq = b1 + 64u * 132u * 4u;
    total = o;
  }
};
constexpr int kStLd = 132;  // row stride of the staging rows (floats)
constexpr int kRawLd = 100; // row stride of the raw Gram-sum staging (floats)
constexpr int kRaw0Ld = 68; // row stride of the raw [L; P] staging (floats)

// 32 lanes x 32 bit, 4 consecutive columns per thread (thread i of the warp <-> lane 32*(warp%4)+i).
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float *v) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// Round to the nearest tf32 value (the tensor cores would otherwise drop the low mantissa bits).
__device__ __forceinline__ float tf32r(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}
__device__ __forceinline__ float4 tf32r4(float4 x) { return make_float4(tf32r(x.x), tf32r(x.y), tf32r(x.z), tf32r(x.w)); }

__device__ __forceinline__ void unpack8(const uint4 &u, float *x) {
  const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(b2[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ float4 unpack4(const uint2 &u) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__global__ void __launch_bounds__(kCtThreads, 1)
    gdp_bwd_chunk_tc_kernel(BwdProblem p, const __grid_constant__ CUtensorMap tm_s,
                            const __grid_constant__ CUtensorMap tm_d) {
  const int row = blockIdx.x, h = blockIdx.y;
  const int seq = p.cid[2 * row], c = p.cid[2 * row + 1];
  if (seq < 0 || seq >= p.N || row >= p.ws_rows) return;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;
  if (c < 0 || L <= 0 || (int64_t)c * kChunk >= L * p.M) return;
  const int M = p.M, QP = p.qpad, H = p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, hh = warp >> 2;
  const int m = 32 * q4 + lane;  // this thread's TMEM lane
  const int64_t R0 = bos * M + (int64_t)c * kChunk;
  const int len = (int)min((int64_t)kChunk, L * M - (int64_t)c * kChunk);
  const int r0m = (int)(R0 % M);
  const int64_t tok0 = (R0 - r0m) / M;
  const int p0 = (M - 1 - r0m) % M;
  const int nq = (p0 < len) ? (len - 1 - p0) / M + 1 : 0;
  const int64_t tq0 = (R0 + p0) / M;
  const int64_t srow = (int64_t)p.cod[seq] + c;
  const CtLayout lay(QP);
  const uint32_t RKQ = lay.rkq;

  extern __shared__ __align__(1024) unsigned char ct_raw[];
  // the 1024-aligned base as an offset into the shared array (a pointer rebuilt from an integer
  // would lose its address space and turn every access below into a generic one)
  unsigned char *sm = ct_raw + ((1024u - (smem_u32(ct_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  auto at = [&](uint32_t off) { return reinterpret_cast<float *>(sm + off); };
  __shared__ float sG[64], sbt[64], sgm[64], sfc[64], sbfc[64], smgb[64], srk[64], sgq[32], srq[32];
  __shared__ float sdb2[2][64], ssg2[2][64], srho2[2][32];
  __shared__ float carry;
  __shared__ __align__(8) uint64_t bar, sbar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  // the slice's S rows v0 .. v0 + 31 (rows 0-31 of each K block) and D_C rows (rows 32-63), TMA
  const int srow_v = (int)((srow * H + h) * kCtD);
  auto issue_slice = [&](int s) {
    const int b = s & 1;
    mbar_arrive_expect_tx(&sbar[b], 2u * kCtVs * kCtD * 4u);
#pragma unroll
    for (int kb = 0; kb < kCtD / 32; ++kb) {
      tma_load_2d(sm + lay.b1s(b) + kb * 8192u, &tm_s, kb * 32, srow_v + s * kCtVs, &sbar[b]);
      tma_load_2d(sm + lay.b1s(b) + kb * 8192u + 4096u, &tm_d, kb * 32, srow_v + s * kCtVs, &sbar[b]);
    }
  };
  if (warp == 0) tmem_alloc(&tmem_slot, 512);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&sbar[0], 1);
    mbar_init(&sbar[1], 1);
    mbar_init_fence();
    abort_flag = 0;
    issue_slice(0);
    issue_slice(1);
  }
  tc_fence_before();

  // ---- the prologue's global loads, all in flight before any is used: T (the forward recompute's
  // WY kernel left T = (I + A)^-1 beside the chunk's reverse-scan image), khat / qhat rows (8
  // threads per row, 16 columns each), beta and the gates, slice 0's d_output and v ----
  float4 tr[4];
  {
    const float *Tg = reinterpret_cast<const float *>(p.bimg + (size_t)(srow * H + h) * p.bimg_stride +
                                                      BwdImageLayout(kCtD, QP).tinv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + kCtThreads * i, r = idx >> 4, c4 = (idx & 15) * 4;
      tr[i] = *reinterpret_cast<const float4 *>(Tg + r * kChunk + c4);
    }
  }
  const int part = tid & 7;
  uint4 kr[3][2];
#pragma unroll
  for (int ps = 0; ps < 3; ++ps) {
    const int r = (tid >> 3) + 32 * ps;
    const bool isk = r < 64;
    const int rr = isk ? r : r - 64;
    const bool live = (r < 64 + QP) && (isk ? rr < len : rr < nq);
    kr[ps][0] = kr[ps][1] = make_uint4(0u, 0u, 0u, 0u);
    if (live) {
      const __nv_bfloat16 *src = isk ? p.k + (R0 + rr) * p.k_st + (int64_t)h * p.k_sh
                                     : p.q + (tq0 + rr) * p.q_st + (int64_t)h * p.q_sh;
      kr[ps][0] = *reinterpret_cast<const uint4 *>(src + part * 16);
      kr[ps][1] = *reinterpret_cast<const uint4 *>(src + part * 16 + 8);
    }
  }
  float bv = 0.f, gate = 0.f;
  if (tid < kChunk && tid < len) {
    const int pos = r0m + tid;
    bv = p.beta ? p.beta[(R0 + tid) * H + h] : 1.f;
    if (p.g && pos % M == 0) gate = p.g[(tok0 + pos / M) * H + h];
  }
  const int dp = tid >> 3, dv4 = (tid & 7) * 4;  // d_output item of this thread (rows dp < qpad)
  auto load_do = [&](int s) {
    uint2 u = make_uint2(0u, 0u);
    if (dp < nq) u = *reinterpret_cast<const uint2 *>(p.dout + ((tq0 + dp) * H + h) * (int64_t)kCtD + s * kCtVs + dv4);
    return u;
  };
  auto load_v = [&](int s, uint4 *u) {
    u[0] = u[1] = make_uint4(0u, 0u, 0u, 0u);
    if (q4 < 2 && m < len) {
      const __nv_bfloat16 *src = p.v + (R0 + m) * p.v_st + (int64_t)h * p.v_sh + s * kCtVs + 16 * hh;
      u[0] = *reinterpret_cast<const uint4 *>(src);
      u[1] = *reinterpret_cast<const uint4 *>(src + 8);
    }
  };
  uint2 do_cur = load_do(0), do_nx = make_uint2(0u, 0u);
  uint4 v_cur[2], v_nx[2];
  load_v(0, v_cur);

  // ---- scalars: beta, within-chunk cumulative log decay ----
  if (tid < kChunk) {
    sbt[tid] = bv;
    float x = gate;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (tid == 31) carry = x;
    sG[tid] = x;
  }
  // ---- [Khat; Qhat] ----
#pragma unroll
  for (int ps = 0; ps < 3; ++ps) {
    const int r = (tid >> 3) + 32 * ps;
    float x[16];
    unpack8(kr[ps][0], x);
    unpack8(kr[ps][1], x + 8);
    float s2 = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s2 += x[i] * x[i];
    s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
    s2 += __shfl_xor_sync(0xffffffffu, s2, 4);
    if (r < 64 + QP) {
      const float inv = p.l2norm ? rsqrtf(s2 + kL2Eps) : 1.f;
      if (part == 0) (r < 64 ? srk : srq)[r < 64 ? r : r - 64] = inv;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4 *>(sm + lay.kq + toff(RKQ, r, part * 16 + 4 * i)) =
            tf32r4(make_float4(x[4 * i] * inv, x[4 * i + 1] * inv, x[4 * i + 2] * inv, x[4 * i + 3] * inv));
    }
  }
  // ---- [T; T^T] ----
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = tid + kCtThreads * i, r = idx >> 4, c4 = (idx & 15) * 4;
    const float4 x = tf32r4(tr[i]);
    *reinterpret_cast<float4 *>(sm + lay.tt + toff(128, r, c4)) = x;
    *at(lay.tt + toff(128, 64 + c4, r)) = x.x;
    *at(lay.tt + toff(128, 64 + c4 + 1, r)) = x.y;
    *at(lay.tt + toff(128, 64 + c4 + 2, r)) = x.z;
    *at(lay.tt + toff(128, 64 + c4 + 3, r)) = x.w;
  }
  // ---- slice 0's dO_s^T ----
  auto put_dot = [&](const uint2 &u) {
    if (dp < QP) {
      const float4 x = unpack4(u);
      *at(lay.dot + toff(32, dv4, dp)) = x.x;
      *at(lay.dot + toff(32, dv4 + 1, dp)) = x.y;
      *at(lay.dot + toff(32, dv4 + 2, dp)) = x.z;
      *at(lay.dot + toff(32, dv4 + 3, dp)) = x.w;
    }
  };
  put_dot(do_cur);
  __syncthreads();
  tc_fence_after();
  if (tid < kChunk && tid >= 32) sG[tid] += carry;
  __syncthreads();
  const float scale = p.scale;
  auto pr = [&](int qi) { return p0 + qi * M; };  // local row of readout qi (qi < nq)
  if (tid < kChunk) {
    const int r = tid;
    const float GC = sG[len - 1];
    const float gr = expf(sG[r]), f = expf(GC - sG[r]), b = sbt[r];
    sgm[r] = gr;        // gamma_r
    sfc[r] = f;         // gamma_C / gamma_r
    sbfc[r] = b * f;    // beta_r gamma_C / gamma_r
    smgb[r] = -gr * b;  // -gamma_r beta_r
    if (r < 32) sgq[r] = (r < nq) ? scale * expf(sG[pr(r)]) : 0.f;  // scale gamma_p of readout r
  }

  const uint32_t tb = tmem_slot;
  const uint32_t lanes = tb + ((uint32_t)(32 * q4) << 16);
  // TMEM columns
  constexpr uint32_t tA1 = 0, tZp = 64, tA2 = 96, tA3 = 160, tGr = 192, tDK = 288, tDQ = 352, tAT = 384;
  const uint32_t id64 = idesc(kFmtTF32, 0, 0, 64, 128), id32 = idesc(kFmtTF32, 0, 0, 32, 128);
  const uint32_t idq = idesc(kFmtTF32, 0, 0, QP, 128), idg = idesc(kFmtTF32, 0, 0, 64 + QP, 128);
  // D (+)= A B^T over ks K steps of 8, both operands K-major swizzled tiles (K blocks of arows /
  // brows rows), or A from TMEM columns
  auto mma_ss = [&](uint32_t tD, uint32_t a, uint32_t arows, uint32_t b, uint32_t brows, int ks, uint32_t id,
                    bool acc) {
    // (the descriptors' start-address field is the byte address / 16: a K step adds its offset / 16)
    const uint64_t da0 = desc_sw128(sb + a, 16, 1024), db0 = desc_sw128(sb + b, 16, 1024);
    for (int kk = 0; kk < ks; ++kk) {
      const uint64_t da = da0 + (((uint32_t)(kk >> 2) * arows * 128u + (uint32_t)(kk & 3) * 32u) >> 4);
      const uint64_t db = db0 + (((uint32_t)(kk >> 2) * brows * 128u + (uint32_t)(kk & 3) * 32u) >> 4);
      mma_tf32_ss(tb + tD, da, db, id, (acc || kk > 0) ? 1u : 0u);
    }
  };
  auto mma_ts = [&](uint32_t tD, uint32_t ta, uint32_t b, uint32_t brows, int ks, uint32_t id, bool acc) {
    const uint64_t db0 = desc_sw128(sb + b, 16, 1024);
    for (int kk = 0; kk < ks; ++kk) {
      const uint64_t db = db0 + (((uint32_t)(kk >> 2) * brows * 128u + (uint32_t)(kk & 3) * 32u) >> 4);
      mma_tf32_ts(tb + tD, tb + ta + (uint32_t)kk * 8u, db, id, (acc || kk > 0) ? 1u : 0u);
    }
  };
  uint32_t ph = 0;
  bool ok = true;
  // operands written -> visible to the tensor cores, all threads past this point
  auto to_mma = [&]() {
    fence_async_smem();
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
  };
  auto wait_mma = [&]() {
    ok = mbar_wait_or_abort(&bar, ph, &abort_flag, kWaitLimitNs) && ok;
    ph ^= 1u;
    tc_fence_after();
  };
  auto wait_slice = [&](int s) {
    ok = mbar_wait_or_abort(&sbar[s & 1], (uint32_t)((s >> 1) & 1), &abort_flag, kWaitLimitNs) && ok;
  };
  // batch 1 of slice s: [rhs-part | Zk] = [Khat; Qhat] [S_s; D_s]^T, Zp = P^T dO_s
  auto batch1 = [&](int s) {
    wait_slice(s);
    mma_ss(tA1, lay.kq, RKQ, lay.b1s(s), 64, kCtD / 8, id64, false);
    mma_ss(tZp, lay.pt, 64, lay.dot, 32, QP / 8, id32, false);
  };

  // ---- batch 0: [L; P] = [Khat; Qhat] Khat^T ----
  to_mma();
  if (tid == 0) {
    tc_fence_after();
    mma_ss(tA1, lay.kq, RKQ, lay.kq, RKQ, kCtD / 8, id64, false);
    mma_commit(&bar);
  }
  wait_mma();
  // the raw products go through shared memory (b2 .. dqb, free until the first slice); the masks and
  // decays then run with each thread on a fixed row
  {
    float *raw = at(lay.b2);  // [64 + qpad][kRaw0Ld]
    if (q4 < 3) {
      float a[32];
      tmem_ld32x(lanes + tA1 + 32 * hh, a);
      if (m < 64 + QP) {
#pragma unroll
        for (int j4 = 0; j4 < 32; j4 += 4)
          *reinterpret_cast<float4 *>(raw + m * kRaw0Ld + 32 * hh + j4) = make_float4(a[j4], a[j4 + 1], a[j4 + 2], a[j4 + 3]);
      }
    }
    __syncthreads();
    {  // L: row tid / 4, columns 16 (tid % 4) .. + 15
      const int r = tid >> 2, c0 = 16 * (tid & 3);
      const float gr = sG[r];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int j0 = c0 + 4 * g;
        const float4 x = *reinterpret_cast<const float4 *>(raw + r * kRaw0Ld + j0);
        const float xv[4] = {x.x, x.y, x.z, x.w};
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = (j0 + i < r) ? tf32r(expf(gr - sG[j0 + i]) * xv[i]) : 0.f;
        *reinterpret_cast<float4 *>(sm + lay.lp + toff(RKQ, r, j0)) = make_float4(o[0], o[1], o[2], o[3]);
      }
    }
    if ((tid >> 3) < QP) {  // P (and P^T): row tid / 8, columns 8 (tid % 8) .. + 7
      const int qi = tid >> 3;
      const bool live = qi < nq;
      const int pq = live ? pr(qi) : 0;
      const float gq = sG[pq];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int j0 = 8 * (tid & 7) + 4 * g;
        const float4 x = *reinterpret_cast<const float4 *>(raw + (64 + qi) * kRaw0Ld + j0);
        const float xv[4] = {x.x, x.y, x.z, x.w};
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[i] = (live && j0 + i <= pq) ? tf32r(scale * expf(gq - sG[j0 + i]) * xv[i]) : 0.f;
          *at(lay.pt + toff(64, j0 + i, qi)) = o[i];
        }
        *reinterpret_cast<float4 *>(sm + lay.lp + toff(RKQ, 64 + qi, j0)) = make_float4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  // ---- batch 0b: [L T; P T] = [L; P] T (T^T are rows 64-127 of [T; T^T]), written over [L; P]:
  // the slices then take L vt and P vt from beta rhs with vt itself, one batch ----
  to_mma();
  if (tid == 0) {
    tc_fence_after();
    mma_ss(tA2, lay.lp, RKQ, lay.tt + 64u * 128u, 128, kChunk / 8, id64, false);
    mma_commit(&bar);
  }
  wait_mma();
  if (q4 < 3) {
    float a[32];
    tmem_ld32x(lanes + tA2 + 32 * hh, a);
    if (m < 64 + QP) {
#pragma unroll
      for (int j4 = 0; j4 < 32; j4 += 4)
        *reinterpret_cast<float4 *>(sm + lay.lp + toff(RKQ, m, 32 * hh + j4)) =
            tf32r4(make_float4(a[j4], a[j4 + 1], a[j4 + 2], a[j4 + 3]));
    }
  }
  to_mma();
  if (tid == 0) {
    tc_fence_after();
    batch1(0);
    mma_commit(&bar);
  }

  float rhs[16], vin[16];
  float sdb_acc = 0.f, ssg_acc = 0.f, rho_acc = 0.f;
#pragma unroll 1
  for (int s = 0; s < kCtSlices; ++s) {
    const int v0 = s * kCtVs;
    const uint32_t b1 = lay.b1s(s), ga = b1, dkb = b1 + 128u * 128u;
    wait_mma();  // batch 1 of this slice (and the previous slice's last products)
    wait_slice(s);
    if (tid == 0 && s >= 1 && s + 1 < kCtSlices) issue_slice(s + 1);  // into the buffer slice s - 1 freed
    if (s + 1 < kCtSlices) {
      do_nx = load_do(s + 1);
      load_v(s + 1, v_nx);
    }
    // ---- D_C^T | S^T of the slice into TMEM (lanes k) for the V contractions; the slice's dO rows
    // into the Gram and dqhat operands ----
    {
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = tf32r(*at(b1 + toff(64, (hh ? 0 : 32) + i, m)));
      tmem_st32x(lanes + tAT + 32 * hh, x);
    }
    if (dp < QP) {
      const float4 x = unpack4(do_cur);
      *reinterpret_cast<float4 *>(sm + lay.gb + toff(RKQ, 64 + dp, dv4)) = x;
      const float gq = sgq[dp];
      *reinterpret_cast<float4 *>(sm + lay.dqb + toff(QP, dp, dv4)) =
          tf32r4(make_float4(gq * x.x, gq * x.y, gq * x.z, gq * x.w));
    }
    // ---- rhs = v - gamma Khat S^T, Zt = fc Khat D_C^T + P^T dO into [beta rhs^T; Zt^T] ----
    if (q4 < 2) {
      const int r = m;
      unpack8(v_cur[0], vin);
      unpack8(v_cur[1], vin + 8);
      uint32_t sa[16], za[16], zp[16];
      tmem_ld16_nw(lanes + tA1 + 16 * hh, sa);
      tmem_ld16_nw(lanes + tA1 + 32 + 16 * hh, za);
      tmem_ld16_nw(lanes + tZp + 16 * hh, zp);
      tmem_ld_wait();
      const float gm = sgm[r], b = sbt[r], f = sfc[r];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        rhs[i] = vin[i] - gm * __uint_as_float(sa[i]);
        const int n = 16 * hh + i;
        *at(lay.b2 + toff(64, n, r)) = tf32r(b * rhs[i]);
        *at(lay.b2 + toff(64, 32 + n, r)) = tf32r(f * __uint_as_float(za[i]) + __uint_as_float(zp[i]));
      }
    }
    // ---- batch 2: [vt | Delta] = [T; T^T] [beta rhs^T; Zt^T]^T and [L vt; P vt] = [L T; P T] beta rhs ----
    to_mma();
    if (tid == 0) {
      tc_fence_after();
      mma_ss(tA2, lay.tt, 128, lay.b2, 64, kChunk / 8, id64, false);
      mma_ss(tA3, lay.lp, RKQ, lay.b2, 64, kChunk / 8, id32, false);
      mma_commit(&bar);
    }
    wait_mma();
    if (q4 < 2) {  // rows r: vt, e = rhs - L vt
      const int r = m;
      uint32_t vr[16], lr[16];
      tmem_ld16_nw(lanes + tA2 + 16 * hh, vr);
      tmem_ld16_nw(lanes + tA3 + 16 * hh, lr);
      tmem_ld_wait();
      const float bf = sbfc[r];
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 vt = tf32r4(make_float4(__uint_as_float(vr[i]), __uint_as_float(vr[i + 1]),
                                             __uint_as_float(vr[i + 2]), __uint_as_float(vr[i + 3])));
        *reinterpret_cast<float4 *>(sm + ga + toff(128, 64 + r, 16 * hh + i)) = vt;
        rhs[i] -= __uint_as_float(lr[i]);  // e
        rhs[i + 1] -= __uint_as_float(lr[i + 1]);
        rhs[i + 2] -= __uint_as_float(lr[i + 2]);
        rhs[i + 3] -= __uint_as_float(lr[i + 3]);
        const float4 e = make_float4(rhs[i], rhs[i + 1], rhs[i + 2], rhs[i + 3]);
        *reinterpret_cast<float4 *>(sm + ga + toff(128, r, 16 * hh + i)) = tf32r4(e);
        *reinterpret_cast<float4 *>(sm + dkb + toff(64, r, 16 * hh + i)) =
            tf32r4(make_float4(bf * e.x, bf * e.y, bf * e.z, bf * e.w));
      }
    } else {  // rows r: Delta, dv; readout rows p (quadrant 2): rho_p += dO_p . o_p
      const int r = m - 64;
      float dl[16];
      tmem_ld16(lanes + tA2 + 32 + 16 * hh, dl);
      const float b = sbt[r], mg = smgb[r];
      float *dvo = p.dv + ((R0 + r) * H + h) * (int64_t)kCtD + v0 + 16 * hh;
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 x = make_float4(dl[i], dl[i + 1], dl[i + 2], dl[i + 3]);
        const float4 bx = make_float4(b * x.x, b * x.y, b * x.z, b * x.w);
        if (r < len) *reinterpret_cast<float4 *>(dvo + i) = bx;
        *reinterpret_cast<float4 *>(sm + lay.gb + toff(RKQ, r, 16 * hh + i)) = tf32r4(bx);
        *reinterpret_cast<float4 *>(sm + dkb + toff(64, r, 32 + 16 * hh + i)) =
            tf32r4(make_float4(mg * x.x, mg * x.y, mg * x.z, mg * x.w));
        const int ch = ((4 * hh + (i >> 2)) ^ (r & 7));
        *reinterpret_cast<float4 *>(sm + lay.dl + (uint32_t)r * 128u + (uint32_t)ch * 16u) = x;
      }
      if (q4 == 2) {
        const int qi = lane;
        uint32_t qa[16], ea[16];
        tmem_ld16_nw(lanes + tA1 + 16 * hh, qa);
        tmem_ld16_nw(lanes + tA3 + 16 * hh, ea);
        tmem_ld_wait();
        if (qi < QP) {
          const float gq = sgq[qi];
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 d = *reinterpret_cast<const float4 *>(sm + lay.gb + toff(RKQ, 64 + qi, 16 * hh + i));
            rho_acc += d.x * (gq * __uint_as_float(qa[i]) + __uint_as_float(ea[i])) +
                       d.y * (gq * __uint_as_float(qa[i + 1]) + __uint_as_float(ea[i + 1])) +
                       d.z * (gq * __uint_as_float(qa[i + 2]) + __uint_as_float(ea[i + 2])) +
                       d.w * (gq * __uint_as_float(qa[i + 3]) + __uint_as_float(ea[i + 3]));
          }
        }
      }
    }
    __syncthreads();  // Delta rows -> the row sums
    if (q4 < 2) {  // dbeta_r += e_r . Delta_r, sig_r += Delta_r . v_r
      const int r = m;
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const int ch = ((4 * hh + (i >> 2)) ^ (r & 7));
        const float4 x = *reinterpret_cast<const float4 *>(sm + lay.dl + (uint32_t)r * 128u + (uint32_t)ch * 16u);
        sdb_acc += rhs[i] * x.x + rhs[i + 1] * x.y + rhs[i + 2] * x.z + rhs[i + 3] * x.w;
        ssg_acc += x.x * vin[i] + x.y * vin[i + 1] + x.z * vin[i + 2] + x.w * vin[i + 3];
      }
    }
    if (s + 1 < kCtSlices) put_dot(do_nx);  // the next slice's batch 1 reads it
    // ---- batch 3: Gram sums [e; vt] [dv; dO]^T, dkhat^T += [D_s^T | S_s^T] [bfc e | -gb Delta]^T,
    // dqhat^T += S_s^T (scale gamma_p dO_s)^T; with the next slice's batch 1 ----
    to_mma();
    if (tid == 0) {
      tc_fence_after();
      mma_ss(tGr, ga, 128, lay.gb, RKQ, kCtVs / 8, idg, s > 0);
      mma_ts(tDK, tAT, dkb, 64, 2 * kCtVs / 8, id64, s > 0);
      mma_ts(tDQ, tAT + 32, lay.dqb, QP, kCtVs / 8, idq, s > 0);
      if (s + 1 < kCtSlices) batch1(s + 1);
      mma_commit(&bar);
    }
    do_cur = do_nx;
    v_cur[0] = v_nx[0];
    v_cur[1] = v_nx[1];
  }
  wait_mma();

  // ---- masks and decays of the Gram sums into the last batch's B tiles; [Qhat^T | Khat^T] into
  // TMEM as its A operand ----
  {
    float *raw = at(lay.raw5);  // [128][kRawLd]: rows e (0-63) and vt (64-127) of the Gram sums
    {
      float a[32];
      tmem_ld32x(lanes + tGr + 32 * hh, a);
#pragma unroll
      for (int j4 = 0; j4 < 32; j4 += 4)
        *reinterpret_cast<float4 *>(raw + m * kRawLd + 32 * hh + j4) = make_float4(a[j4], a[j4 + 1], a[j4 + 2], a[j4 + 3]);
      if (hh == 0) {
        tmem_ld32x(lanes + tGr + 64, a);  // columns past 64 + qpad are not used
#pragma unroll
        for (int j4 = 0; j4 < 32; j4 += 4)
          *reinterpret_cast<float4 *>(raw + m * kRawLd + 64 + j4) = make_float4(a[j4], a[j4 + 1], a[j4 + 2], a[j4 + 3]);
      }
    }
    __syncthreads();
    // [beta M1 | -M23] rows r: beta_r M1 (readouts), -beta_r M2 (j > r, from e . dv), -M3 (j < r,
    // from vt_j . dv_r); groups of 4 columns (qpad is a multiple of 16: a group lies in one part)
    {  // row tid / 4; 16-column blocks of [M1 | M23], 4 columns each (qpad is a multiple of 16)
      const int r = tid >> 2, sub = tid & 3;
      const float b = sbt[r], gr = sG[r];
#pragma unroll
      for (int k = 0; k < 6; ++k) {
        if (16 * k >= QP + 64) break;
        const int pos0 = 16 * k + 4 * sub;
        float o[4];
        if (16 * k < QP) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int qi = pos0 + i;
            const bool live = qi < nq && r <= pr(qi);
            o[i] = live ? tf32r(b * scale * expf(sG[live ? pr(qi) : 0] - gr) * raw[r * kRawLd + 64 + qi]) : 0.f;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = pos0 - QP + i;
            const float gj = sG[j];
            o[i] = (j > r)   ? tf32r(-(b * expf(gj - gr) * raw[r * kRawLd + j]))
                   : (j < r) ? tf32r(-(expf(gr - gj) * raw[(64 + j) * kRawLd + r]))
                             : 0.f;
          }
        }
        *reinterpret_cast<float4 *>(sm + lay.fb + toff(64, r, pos0)) = make_float4(o[0], o[1], o[2], o[3]);
      }
    }
    if ((tid >> 3) < QP) {  // scale M4 (from vt_j . dO_p): row tid / 8, columns 8 (tid % 8) .. + 7
      const int qi = tid >> 3;
      const bool qlive = qi < nq;
      const int pq = qlive ? pr(qi) : 0;
      const float gq = sG[pq];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int j0 = 8 * (tid & 7) + 4 * g;
        float o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = j0 + i;
          o[i] = (qlive && j <= pq) ? tf32r(scale * expf(gq - sG[j]) * raw[(64 + j) * kRawLd + 64 + qi]) : 0.f;
        }
        *reinterpret_cast<float4 *>(sm + lay.fq + toff(QP, qi, j0)) = make_float4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  // [Qhat^T | Khat^T]: 16 columns at a time (hh = 0: Qhat^T then Khat rows 0-31; hh = 1: rows 32-63)
  {
    const int ng = (hh == 0 ? QP : 0) / 16 + 2;
#pragma unroll 1
    for (int gi = 0; gi < ng; ++gi) {
      const int col = (hh == 0) ? 16 * gi : QP + 32 + 16 * gi;   // TMEM column
      const int src = (hh == 0) ? (gi < QP / 16 ? 64 + 16 * gi : 16 * gi - QP) : 32 + 16 * gi;  // KQ row
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = *at(lay.kq + toff(RKQ, src + i, m));
      tmem_st16(lanes + tAT + col, x);
    }
  }
  // ---- last batch: dkhat^T += [Qhat^T | Khat^T] [beta M1 | -M23]^T, dqhat^T += Khat^T (M4)^T ----
  to_mma();
  if (tid == 0) {
    tc_fence_after();
    mma_ts(tDK, tAT, lay.fb, 64, (QP + 64) / 8, id64, true);
    mma_ts(tDQ, tAT + QP, lay.fq, QP, kChunk / 8, idq, true);
    mma_commit(&bar);
  }
  wait_mma();
#pragma unroll 1
  for (int r4 = 0; r4 < 32; r4 += 4) {
    float a[4];
    tmem_ld4(lanes + tDK + 32 * hh + r4, a);
#pragma unroll
    for (int i = 0; i < 4; ++i) at(lay.stk)[(32 * hh + r4 + i) * kStLd + m] = a[i];
  }
  if (hh == 0) {
#pragma unroll 1
    for (int q0 = 0; q0 < QP; q0 += 4) {
      float a[4];
      tmem_ld4(lanes + tDQ + q0, a);
#pragma unroll
      for (int i = 0; i < 4; ++i) at(lay.stq)[(q0 + i) * kStLd + m] = a[i];
    }
  }
  if (q4 < 2) {
    sdb2[hh][m] = sdb_acc;
    ssg2[hh][m] = ssg_acc;
  } else if (q4 == 2) {
    srho2[hh][lane] = rho_acc;
  }
  tc_fence_before();
  __syncthreads();
  // ---- L2-norm chain rule (dx = rx (dxhat - (xhat . dxhat) xhat), xhat from the input row in full
  // precision), stores, row sums ----
  for (int r = warp; r < len + nq; r += kCtThreads / 32) {
    const bool isk = r < len;
    const int rr = isk ? r : r - len;
    const float *dh = at(isk ? lay.stk : lay.stq) + rr * kStLd;
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = dh[lane + 32 * i];
    float *out = isk ? p.dk + ((R0 + rr) * H + h) * (int64_t)kCtD : p.dq + ((tq0 + rr) * H + h) * (int64_t)kCtD;
    if (p.l2norm) {
      const __nv_bfloat16 *src = isk ? p.k + (R0 + rr) * p.k_st + (int64_t)h * p.k_sh
                                     : p.q + (tq0 + rr) * p.q_st + (int64_t)h * p.q_sh;
      const float rx = (isk ? srk : srq)[rr];
      float xv[4], dot = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xv[i] = __bfloat162float(src[lane + 32 * i]) * rx;
        dot += a[i] * xv[i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
#pragma unroll
      for (int i = 0; i < 4; ++i) out[lane + 32 * i] = rx * (a[i] - dot * xv[i]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) out[lane + 32 * i] = a[i];
    }
  }
  if (tid < len) {
    if (p.dbeta) p.dbeta[(R0 + tid) * H + h] = sdb2[0][tid] + sdb2[1][tid];
    p.sig[(R0 + tid) * H + h] = sbt[tid] * (ssg2[0][tid] + ssg2[1][tid]);
  }
  if (tid < nq) p.rho[(tq0 + tid) * H + h] = srho2[0][tid] + srho2[1][tid];
  if (!ok && tid == 0 && p.status) set_status(p.status, GDP_DEV_ERR_TIMEOUT);
  __syncthreads();
  if (warp == 0) tmem_free(tb, 512);
}

}  // namespace

bool bwd_chunk_tc_serves(int d, int qpad) { return d == kCtD && qpad <= 32; }

cudaError_t launch_bwd_chunk_tc(const BwdProblem &p, cudaStream_t stream) {
  const size_t smem = CtLayout(p.qpad).total + 1024u;
  cudaError_t e =
      cudaFuncSetAttribute(gdp_bwd_chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // the states entering and the gradients leaving every expanded chunk, [ntdp][H][V][K] fp32, as
  // rows of K in 32 x 32 boxes
  alignas(64) CUtensorMap tm_s, tm_d;
  const int64_t rows = p.ntdp_pad * (int64_t)p.H * p.D;
  if ((e = tmap_state(&tm_s, const_cast<float *>(p.Sx), rows, p.D)) != cudaSuccess) return e;
  if ((e = tmap_state(&tm_d, p.Dx, rows, p.D)) != cudaSuccess) return e;
  gdp_bwd_chunk_tc_kernel<<<dim3((unsigned)p.ntdp_pad, (unsigned)p.H), kCtThreads, smem, stream>>>(p, tm_s, tm_d);
  return cudaGetLastError();
}

}  // namespace gdp
