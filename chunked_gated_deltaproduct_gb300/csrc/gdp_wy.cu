// gdp_wy.cu -- per-(expanded chunk, head) prep + WY kernel.
//
// Megatron-Core API page "core.ssm.ops.gdp.chunk", stages 1 and 2:
//   stage 1: the log decay of token t is placed on its first expanded row
//            t*M (interleave), the within-chunk cumulative sum is taken on the
//            expanded stream and converted to base 2 (exp2 everywhere);
//   stage 2: A = beta K K^T (strictly lower, decay-weighted), T = (I + A)^-1,
//            then the w and u factors.
// With gamma_r = 2^G2_r and khat = k / |k| (or k):
//   A[i][j] = beta_i 2^(G2_i - G2_j) (khat_i . khat_j)        (i > j)
//   W = T diag(beta gamma) Khat,   U = T diag(beta) V
// so that inside the chunk the new values are V_new = U - W S0^T for the
// entering state S0 (derived from the recurrence on the FlashInfer page,
// display equation).  The kernel also forms the masked, decay-weighted
// intra-chunk scores of the readout rows used by the output stage:
//   P[q][s] = scale 2^(G2_p - G2_s) (qhat_t . khat_s)   for s <= p,
// where p = t*M + M - 1 is the readout row of token t.  Every exponent is of
// a difference G2_i - G2_j with i >= j, so every factor is <= 1.
#include "gdp_internal.cuh"

namespace gdp {
namespace {

constexpr int kWyThreads = 256;

struct WySmem {
  float *ks, *vs, *qs, *A, *Tm;
  float *G2, *bt, *rk, *rq, *wc, *uc;
  __device__ WySmem(float *base, int K, int V, int QP) {
    ks = base;
    vs = ks + kChunk * (K + 1);
    qs = vs + kChunk * (V + 1);
    A = qs + QP * (K + 1);
    Tm = A + kChunk * (kChunk + 1);
    G2 = Tm + kChunk * (kChunk + 1);
    bt = G2 + kChunk;
    rk = bt + kChunk;
    rq = rk + kChunk;
    wc = rq + kChunk;
    uc = wc + kChunk;
  }
  __host__ __device__ static size_t bytes(int K, int V, int QP) {
    return sizeof(float) * ((size_t)kChunk * (K + 1) + (size_t)kChunk * (V + 1) + (size_t)QP * (K + 1) +
                            2 * (size_t)kChunk * (kChunk + 1) + 6 * kChunk);
  }
};

__global__ void __launch_bounds__(kWyThreads) gdp_wy_kernel(Problem p) {
  const int row = blockIdx.x, h = blockIdx.y;
  const int seq = p.cid[2 * row], c = p.cid[2 * row + 1];
  if (seq < 0 || seq >= p.N || row >= p.ws_rows) return;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;
  if (c < 0 || L <= 0 || (int64_t)c * kChunk >= L * p.M) return;
  const int M = p.M, K = p.K, V = p.V, QP = p.qpad;
  const int64_t R0 = bos * M + (int64_t)c * kChunk;  // first global expanded row
  const int len = (int)min((int64_t)kChunk, L * M - (int64_t)c * kChunk);
  const int p0 = (int)((M - 1 - (R0 % M)) % M);
  const int nq = (p0 < len) ? (len - 1 - p0) / M + 1 : 0;

  extern __shared__ float4 smem_f4[];
  WySmem sm(reinterpret_cast<float *>(smem_f4), K, V, QP);
  const int tid = threadIdx.x;

  // ---- loads (zero past the chunk end) ----
  for (int idx = tid; idx < kChunk * K; idx += blockDim.x) {
    int r = idx / K, f = idx % K;
    float x = 0.f;
    if (r < len) x = __bfloat162float(p.k[(R0 + r) * p.k_st + (int64_t)h * p.k_sh + f]);
    sm.ks[r * (K + 1) + f] = x;
  }
  for (int idx = tid; idx < kChunk * V; idx += blockDim.x) {
    int r = idx / V, f = idx % V;
    float x = 0.f;
    if (r < len) x = __bfloat162float(p.v[(R0 + r) * p.v_st + (int64_t)h * p.v_sh + f]);
    sm.vs[r * (V + 1) + f] = x;
  }
  for (int idx = tid; idx < QP * K; idx += blockDim.x) {
    int qi = idx / K, f = idx % K;
    float x = 0.f;
    if (qi < nq) {
      int64_t t = (R0 + p0 + (int64_t)qi * M) / M;
      x = __bfloat162float(p.q[t * p.q_st + (int64_t)h * p.q_sh + f]);
    }
    sm.qs[qi * (K + 1) + f] = x;
  }
  __syncthreads();

  // ---- per-row scalars: beta, decay gate, inverse norms ----
  if (tid < kChunk) {
    const int r = tid;
    const int64_t gr = R0 + r;
    float b = 0.f, gate = 0.f;
    if (r < len) {
      b = p.beta ? p.beta[gr * p.H + h] : 1.f;
      if (p.g && gr % M == 0) gate = p.g[(gr / M) * p.H + h];
    }
    sm.bt[r] = b;
    sm.G2[r] = gate;  // raw gate; the scan below turns it into the cumsum
    float ss = 0.f;
    for (int f = 0; f < K; ++f) ss += sm.ks[r * (K + 1) + f] * sm.ks[r * (K + 1) + f];
    sm.rk[r] = p.l2norm ? rsqrtf(ss + kL2Eps) : 1.f;
    float sq = 0.f;
    if (r < QP)
      for (int f = 0; f < K; ++f) sq += sm.qs[r * (K + 1) + f] * sm.qs[r * (K + 1) + f];
    sm.rq[r] = p.l2norm ? rsqrtf(sq + kL2Eps) : 1.f;
  }
  __syncthreads();
  if (tid == 0) {  // within-chunk cumsum, base 2
    float acc = 0.f;
    for (int r = 0; r < kChunk; ++r) {
      acc += sm.G2[r];
      sm.G2[r] = acc * kLog2e;
    }
  }
  __syncthreads();
  if (tid < kChunk) {
    const int j = tid;
    sm.wc[j] = sm.bt[j] * exp2f(sm.G2[j]) * sm.rk[j];
    sm.uc[j] = sm.bt[j];
  }

  // ---- A = beta K K^T, strictly lower, decay weighted ----
  for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x) {
    int i = idx / kChunk, j = idx % kChunk;
    float a = 0.f;
    if (j < i && i < len) {
      float d = 0.f;
      for (int f = 0; f < K; ++f) d += sm.ks[i * (K + 1) + f] * sm.ks[j * (K + 1) + f];
      a = sm.bt[i] * exp2f(sm.G2[i] - sm.G2[j]) * sm.rk[i] * sm.rk[j] * d;
    }
    sm.A[i * (kChunk + 1) + j] = a;
  }
  __syncthreads();

  // ---- T = (I + A)^-1, unit lower triangular; one column per thread ----
  if (tid < kChunk) {
    const int cc = tid;
    for (int i = 0; i < kChunk; ++i) {
      float t;
      if (i < cc) t = 0.f;
      else if (i == cc) t = 1.f;
      else {
        float acc = 0.f;
        for (int j = cc; j < i; ++j) acc += sm.A[i * (kChunk + 1) + j] * sm.Tm[j * (kChunk + 1) + cc];
        t = -acc;
      }
      sm.Tm[i * (kChunk + 1) + cc] = t;
    }
  }
  __syncthreads();

  const int64_t tile = (int64_t)row * p.H + h;
  // ---- W (stored negated) and U ----
  float *Wt = p.W + tile * (int64_t)kChunk * K;
  for (int idx = tid; idx < kChunk * K; idx += blockDim.x) {
    int s = idx / K, f = idx % K;
    float acc = 0.f;
    for (int j = 0; j <= s; ++j) acc += sm.Tm[s * (kChunk + 1) + j] * sm.wc[j] * sm.ks[j * (K + 1) + f];
    Wt[idx] = -acc;
  }
  float *Ut = p.U + tile * (int64_t)kChunk * V;
  for (int idx = tid; idx < kChunk * V; idx += blockDim.x) {
    int s = idx / V, f = idx % V;
    float acc = 0.f;
    for (int j = 0; j <= s; ++j) acc += sm.Tm[s * (kChunk + 1) + j] * sm.uc[j] * sm.vs[j * (V + 1) + f];
    Ut[idx] = acc;
  }
  // ---- masked decayed scores of the readout rows ----
  float *Pt = p.P + tile * (int64_t)QP * kChunk;
  for (int idx = tid; idx < QP * kChunk; idx += blockDim.x) {
    int qi = idx / kChunk, s = idx % kChunk;
    float val = 0.f;
    if (qi < nq) {
      int pr = p0 + qi * M;
      if (s <= pr) {
        float d = 0.f;
        for (int f = 0; f < K; ++f) d += sm.qs[qi * (K + 1) + f] * sm.ks[s * (K + 1) + f];
        val = p.scale * exp2f(sm.G2[pr] - sm.G2[s]) * sm.rq[qi] * sm.rk[s] * d;
      }
    }
    Pt[idx] = val;
  }
  // ---- metadata for the scan ----
  ChunkMeta *mt = p.meta + tile;
  const float G2last = sm.G2[len - 1];
  if (tid < kChunk) {
    const int s = tid;
    mt->kscale[s] = (s < len) ? exp2f(G2last - sm.G2[s]) * sm.rk[s] : 0.f;
    float qsc = 0.f;
    if (s < nq) qsc = p.scale * exp2f(sm.G2[p0 + s * M]) * sm.rq[s];
    mt->qscale[s] = qsc;
  }
  if (tid == 0) {
    mt->gamma_last = exp2f(G2last);
    mt->nq = nq;
    mt->p0 = p0;
    mt->len = len;
  }
}

}  // namespace

cudaError_t launch_wy(const Problem &p, cudaStream_t stream) {
  if (p.ntdp_pad == 0) return cudaSuccess;
  size_t smem = WySmem::bytes(p.K, p.V, p.qpad);
  cudaError_t e = cudaFuncSetAttribute(gdp_wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.ntdp_pad, (unsigned)p.H);
  gdp_wy_kernel<<<grid, kWyThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdp
