// gdp_scan.cu -- inter-chunk state scan, output combine and state scatter.
//
// Megatron-Core API page "core.ssm.ops.gdp.chunk", stages 3 and 4, with the
// chunk-state rows of parameter return_chunk_states and the in-place state
// cache of parameters state / state_indices.  For expanded chunk e of a
// sequence with entering state S_e (V-major, [V][K]):
//   V_new   = U - W S_e^T                                         [64 x V]
//   o_t     = Qhat_t S_e^T + sum_{s <= p} P[t][s] V_new[s]        (readout rows)
//   S_{e+1} = gamma_last S_e + V_new^T Ktil,  Ktil_s = 2^(G2_last - G2_s) khat_s
// where Qhat_t = scale 2^(G2_p) qhat_t.  Every M-th expanded chunk starts a
// token chunk (64 c tokens = 64 c M rows): its entering state is chunk-state
// row chunk_offsets[i] + e / M.
//
// Rows of S evolve independently (row v of V_new reads row v of S only), so
// the V dimension is split across CTAs (FlashInfer page, output_state: one
// sequence is split across CTAs).
#include "gdp_internal.cuh"

namespace gdp {
namespace {

constexpr int kScanThreads = 256;
constexpr int kVS = 16;  // state rows per CTA

__global__ void __launch_bounds__(kScanThreads) gdp_scan_kernel(Problem p) {
  const int seq = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * kVS;
  const int K = p.K, V = p.V, M = p.M, QP = p.qpad, H = p.H;
  const int tid = threadIdx.x;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;  // flagged by the descriptor kernel
  const int nv = min(kVS, V - v0);

  extern __shared__ float4 smem_f4[];
  float *S = reinterpret_cast<float *>(smem_f4);  // [kVS][K+1]
  float *Wn = S + kVS * (K + 1);                  // [64][K+1]  (-W)
  float *Kt = Wn + kChunk * (K + 1);              // [64][K+1]
  float *Qh = Kt + kChunk * (K + 1);              // [QP][K+1]
  float *Pm = Qh + QP * (K + 1);                  // [QP][65]
  float *Us = Pm + QP * (kChunk + 1);             // [64][kVS+1]
  float *Vn = Us + kChunk * (kVS + 1);            // [64][kVS+1]
  __shared__ ChunkMeta mt;

  // incoming state
  int slot = -1;
  const float *src = nullptr;
  if (p.cache) {
    slot = p.slots[seq];
    if (slot < -1 || slot >= p.num_slots) {
      if (tid == 0 && blockIdx.z == 0) set_status(p.status, GDP_DEV_ERR_SLOT);
      slot = -1;
    }
    if (slot >= 0) src = p.cache + ((int64_t)slot * H + h) * (int64_t)V * K;
  } else if (p.init) {
    src = p.init + ((int64_t)seq * H + h) * (int64_t)V * K;
  }
  for (int idx = tid; idx < kVS * K; idx += blockDim.x) {
    int r = idx / K, f = idx % K;
    S[r * (K + 1) + f] = (src && r < nv) ? src[(int64_t)(v0 + r) * K + f] : 0.f;
  }
  __syncthreads();

  const int64_t nchunks = (L * M + kChunk - 1) / kChunk;
  const int cod_i = p.cod[seq];
  const int co_i = p.chunk_states ? p.co[seq] : 0;
  for (int64_t e = 0; e < nchunks; ++e) {
    const int64_t row = cod_i + e;
    if (row < 0 || row >= p.ws_rows) break;  // flagged by the descriptor kernel
    const int64_t tile = row * H + h;
    const int64_t R0 = bos * M + e * kChunk;
    if (p.chunk_states && e % M == 0 && co_i >= 0 && co_i + e / M < p.nt_pad) {
      float *dst = p.chunk_states + ((co_i + e / M) * H + h) * (int64_t)V * K;
      for (int idx = tid; idx < nv * K; idx += blockDim.x) {
        int r = idx / K, f = idx % K;
        dst[(int64_t)(v0 + r) * K + f] = S[r * (K + 1) + f];
      }
    }
    if (tid == 0) mt = p.meta[tile];
    __syncthreads();
    const int len = mt.len, nq = mt.nq, p0 = mt.p0;
    const float *Wt = p.W + tile * (int64_t)kChunk * K;
    for (int idx = tid; idx < kChunk * K; idx += blockDim.x) {
      int s = idx / K, f = idx % K;
      Wn[s * (K + 1) + f] = Wt[idx];
      float x = 0.f;
      if (s < len) x = mt.kscale[s] * __bfloat162float(p.k[(R0 + s) * p.k_st + (int64_t)h * p.k_sh + f]);
      Kt[s * (K + 1) + f] = x;
    }
    for (int idx = tid; idx < QP * K; idx += blockDim.x) {
      int qi = idx / K, f = idx % K;
      float x = 0.f;
      if (qi < nq) {
        int64_t t = (R0 + p0 + (int64_t)qi * M) / M;
        x = mt.qscale[qi] * __bfloat162float(p.q[t * p.q_st + (int64_t)h * p.q_sh + f]);
      }
      Qh[qi * (K + 1) + f] = x;
    }
    const float *Pt = p.P + tile * (int64_t)QP * kChunk;
    for (int idx = tid; idx < QP * kChunk; idx += blockDim.x)
      Pm[(idx / kChunk) * (kChunk + 1) + idx % kChunk] = Pt[idx];
    const float *Ut = p.U + tile * (int64_t)kChunk * V;
    for (int idx = tid; idx < kChunk * kVS; idx += blockDim.x) {
      int s = idx / kVS, r = idx % kVS;
      Us[s * (kVS + 1) + r] = (r < nv) ? Ut[(int64_t)s * V + v0 + r] : 0.f;
    }
    __syncthreads();
    // V_new = U - W S^T
    for (int idx = tid; idx < kChunk * kVS; idx += blockDim.x) {
      int s = idx / kVS, r = idx % kVS;
      float acc = Us[s * (kVS + 1) + r];
      for (int f = 0; f < K; ++f) acc += Wn[s * (K + 1) + f] * S[r * (K + 1) + f];
      Vn[s * (kVS + 1) + r] = acc;
    }
    __syncthreads();
    // outputs of the readout rows
    for (int idx = tid; idx < nq * kVS; idx += blockDim.x) {
      int qi = idx / kVS, r = idx % kVS;
      if (r >= nv) continue;
      float acc = 0.f;
      for (int f = 0; f < K; ++f) acc += Qh[qi * (K + 1) + f] * S[r * (K + 1) + f];
      for (int s = 0; s < kChunk; ++s) acc += Pm[qi * (kChunk + 1) + s] * Vn[s * (kVS + 1) + r];
      int64_t t = (R0 + p0 + (int64_t)qi * M) / M;
      p.out[(t * H + h) * (int64_t)V + v0 + r] = __float2bfloat16_rn(acc);
    }
    __syncthreads();
    // S <- gamma_last S + V_new^T Ktil
    const float gl = mt.gamma_last;
    for (int idx = tid; idx < kVS * K; idx += blockDim.x) {
      int r = idx / K, f = idx % K;
      float acc = gl * S[r * (K + 1) + f];
      for (int s = 0; s < kChunk; ++s) acc += Vn[s * (kVS + 1) + r] * Kt[s * (K + 1) + f];
      S[r * (K + 1) + f] = acc;
    }
    __syncthreads();
  }

  // final state: dense output and/or cache slot
  float *dst = nullptr;
  if (p.cache) {
    if (slot >= 0) dst = p.cache + ((int64_t)slot * H + h) * (int64_t)V * K;
  } else if (p.out_state) {
    dst = p.out_state + ((int64_t)seq * H + h) * (int64_t)V * K;
  }
  if (dst)
    for (int idx = tid; idx < nv * K; idx += blockDim.x) {
      int r = idx / K, f = idx % K;
      dst[(int64_t)(v0 + r) * K + f] = S[r * (K + 1) + f];
    }
}

}  // namespace

cudaError_t launch_scan(const Problem &p, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  size_t smem = sizeof(float) * ((size_t)kVS * (p.K + 1) + 2 * (size_t)kChunk * (p.K + 1) +
                                 (size_t)p.qpad * (p.K + 1) + (size_t)p.qpad * (kChunk + 1) +
                                 2 * (size_t)kChunk * (kVS + 1));
  cudaError_t e = cudaFuncSetAttribute(gdp_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.N, (unsigned)p.H, (unsigned)((p.V + kVS - 1) / kVS));
  gdp_scan_kernel<<<grid, kScanThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdp
