// gdp_scan.cu -- inter-chunk state scan, output combine and state scatter on the
// tcgen05 tensor cores, with the state resident in tensor memory.
//
// Megatron-Core API page "core.ssm.ops.gdp.chunk", stages 3 and 4, with the
// chunk-state rows of parameter return_chunk_states and the in-place state
// cache of parameters state / state_indices.  For expanded chunk e of a
// sequence with entering state S_e (V-major, [V][K]):
//   V_new^T = U^T + S_e (-W)^T                                 [V x 64]
//   o^T     = S_e Qh^T + V_new^T P^T                           [V x qpad] (readout rows)
//   S_{e+1} = gamma_last S_e + V_new^T Ktil                    [V x K]
// Every M-th expanded chunk starts a token chunk (64 c tokens = 64 c M rows):
// its entering state is chunk-state row chunk_offsets[i] + e / M.
//
// One CTA per (sequence, head); 4 warps; TMEM lane v = state row v.  S lives
// in TMEM columns [0, d) for the whole sequence and is read by the MMAs
// directly as the tf32 A operand, so the recurrence never leaves the SM.  All
// products are kind::tf32 (fp32 operands truncated to tf32, fp32 accumulate):
// the state feeds back into every later chunk, and bf16 operands would add a
// ~2^-9 relative error per chunk.  The B operands come from one operand image
// per chunk (written by the WY kernel), fetched by a single bulk copy into a
// double-buffered shared-memory stage while the previous chunk computes.
#include "gdp_internal.cuh"
#include "gdp_sm100.cuh"

namespace gdp {
namespace {

using namespace sm100;

constexpr int kScanThreads = 128;
constexpr uint32_t kScanSmemBudget = 220u * 1024u;

__host__ __device__ inline uint32_t stage_bytes(int d, int qpad) {
  return (ImageLayout(d, qpad).bytes + 1023u) & ~1023u;
}
__host__ __device__ inline int num_stages(int d, int qpad) {
  return 2u * stage_bytes(d, qpad) <= kScanSmemBudget ? 2 : 1;
}

__global__ void __launch_bounds__(kScanThreads) gdp_scan_kernel(Problem p) {
  const int seq = blockIdx.x, h = blockIdx.y;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;  // flagged by the descriptor kernel
  const int d = p.K, V = p.V, M = p.M, QP = p.qpad, H = p.H;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int v = tid;  // state row = TMEM lane
  const ImageLayout il(d, QP);
  const uint32_t sbytes = stage_bytes(d, QP);
  const int nst = num_stages(d, QP);

  extern __shared__ __align__(1024) unsigned char scan_smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)scan_smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full_bar[2];
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ uint32_t tmem_slot;

  // incoming state source
  int slot = -1;
  const float *src = nullptr;
  if (p.cache) {
    slot = p.slots[seq];
    if (slot < -1 || slot >= p.num_slots) {
      if (tid == 0) set_status(p.status, GDP_DEV_ERR_SLOT);
      slot = -1;
    }
    if (slot >= 0) src = p.cache + ((int64_t)slot * H + h) * (int64_t)V * d;
  } else if (p.init) {
    src = p.init + ((int64_t)seq * H + h) * (int64_t)V * d;
  }

  const int64_t nchunks = (L * M + kChunk - 1) / kChunk;
  const int64_t cod_i = p.cod[seq];
  const int64_t co_i = p.chunk_states ? (int64_t)p.co[seq] : 0;
  // chunks whose workspace tile exists (a flagged descriptor overflow truncates the sequence)
  const int64_t nrun = (cod_i < 0) ? 0 : max((int64_t)0, min(nchunks, p.ws_rows - cod_i));

  if (warp == 0) tmem_alloc(&tmem_slot, 256);
  if (tid == 0) {
    mbar_init(&full_bar[0], 1);
    mbar_init(&full_bar[1], 1);
    mbar_init(&mma_bar, 1);
    mbar_init_fence();
    for (int s = 0; s < nst && s < nrun; ++s) {
      const unsigned char *g = p.img + (size_t)((cod_i + s) * H + h) * p.img_stride;
      mbar_arrive_expect_tx(&full_bar[s], il.bytes);
      bulk_g2s(sm + s * sbytes, g, il.bytes, &full_bar[s]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_slot;
  const uint32_t tS = tb, tVn = tb + 128, tO = tb + 192;  // S: d cols, V_new^T: 64, o^T: qpad (<= 64)
  const uint32_t lrow = (uint32_t)(warp * 32) << 16;

  // S_0 into TMEM (rows >= V stay zero)
  for (int c0 = 0; c0 < d; c0 += 16) {
    float x[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) x[u] = (src && v < V) ? src[(int64_t)v * d + c0 + u] : 0.f;
    tmem_st16(tS + lrow + c0, x);
  }
  // U of the first chunk into registers: u[s] = U[s][v]
  float u[64];
  if (nrun > 0) {
    const float *Ut = p.U + (cod_i * H + h) * (int64_t)kChunk * V;
#pragma unroll
    for (int s = 0; s < kChunk; ++s) u[s] = (v < V) ? Ut[(int64_t)s * V + v] : 0.f;
  }
  tmem_st_wait();

  uint32_t full_phase[2] = {0, 0}, mma_phase = 0;
  bool aborted = false;
  const uint32_t id_vn = idesc(kFmtTF32, 0, 0, 64, 128);
  const uint32_t id_o = idesc(kFmtTF32, 0, 0, QP, 128);
  const uint32_t id_s = idesc(kFmtTF32, 0, 0, d, 128);
  for (int64_t e = 0; e < nrun; ++e) {
    const int st = (int)(e % nst);
    unsigned char *stage = sm + st * sbytes;
    const int64_t R0 = bos * M + e * kChunk;
    // V_new^T <- U^T (accumulated onto by the first product)
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) tmem_st16(tVn + lrow + c0, u + c0);
    tmem_st_wait();
    if (e + 1 < nrun) {  // prefetch the next chunk's U while this one computes
      const float *Ut = p.U + ((cod_i + e + 1) * H + h) * (int64_t)kChunk * V;
#pragma unroll
      for (int s = 0; s < kChunk; ++s) u[s] = (v < V) ? Ut[(int64_t)s * V + v] : 0.f;
    }
    const bool okf = mbar_wait(&full_bar[st], full_phase[st]);
    full_phase[st] ^= 1u;
    tc_fence_before();
    if (__syncthreads_or(!okf)) { aborted = true; break; }
    tc_fence_after();
    const ImageMeta mt = *reinterpret_cast<const ImageMeta *>(stage + il.meta);

    // batch 1: V_new^T += S (-W)^T ; o^T = S Qh^T
    if (tid == 0) {
      const uint32_t sb = smem_u32(stage);
      for (int kk = 0; kk < d / 8; ++kk) {
        const uint32_t koff = (kk & 3) * 32u;
        mma_tf32_ts(tVn, tS + kk * 8, desc_sw128(sb + il.wn + (kk >> 2) * (64u * 128u) + koff, 16, 1024), id_vn, 1);
        mma_tf32_ts(tO, tS + kk * 8, desc_sw128(sb + il.qh + (kk >> 2) * ((uint32_t)QP * 128u) + koff, 16, 1024),
                    id_o, kk > 0);
      }
      mma_commit(&mma_bar);
    }
    const bool ok1 = mbar_wait(&mma_bar, mma_phase);
    mma_phase ^= 1u;
    tc_fence_after();

    // state pass: emit the entering state at token-chunk starts, then S <- gamma_last S
    const bool emit = p.chunk_states && (e % M == 0) && co_i >= 0 && co_i + e / M < p.nt_pad && v < V;
    float *cs = emit ? p.chunk_states + ((co_i + e / M) * H + h) * (int64_t)V * d + (int64_t)v * d : nullptr;
    for (int c0 = 0; c0 < d; c0 += 16) {
      float x[16];
      tmem_ld16(tS + lrow + c0, x);
      if (cs) {
#pragma unroll
        for (int u4 = 0; u4 < 16; u4 += 4)
          *reinterpret_cast<float4 *>(cs + c0 + u4) = make_float4(x[u4], x[u4 + 1], x[u4 + 2], x[u4 + 3]);
      }
#pragma unroll
      for (int w = 0; w < 16; ++w) x[w] *= mt.gamma_last;
      tmem_st16(tS + lrow + c0, x);
    }
    tmem_st_wait();
    tc_fence_before();
    if (__syncthreads_or(!ok1)) { aborted = true; break; }
    tc_fence_after();

    // batch 2: o^T += V_new^T P^T ; S += V_new^T Ktil
    if (tid == 0) {
      const uint32_t sb = smem_u32(stage);
      for (int kk = 0; kk < kChunk / 8; ++kk) {
        const uint32_t koff = (kk & 3) * 32u;
        mma_tf32_ts(tO, tVn + kk * 8, desc_sw128(sb + il.pm + (kk >> 2) * ((uint32_t)QP * 128u) + koff, 16, 1024),
                    id_o, 1);
        mma_tf32_ts(tS, tVn + kk * 8, desc_sw128(sb + il.kt + (kk >> 2) * ((uint32_t)d * 128u) + koff, 16, 1024),
                    id_s, 1);
      }
      mma_commit(&mma_bar);
    }
    const bool ok2 = mbar_wait(&mma_bar, mma_phase);
    mma_phase ^= 1u;
    tc_fence_after();
    // the stage is free: fetch chunk e + nst into it
    if (tid == 0 && ok2 && e + nst < nrun) {
      fence_async_smem();
      const unsigned char *g = p.img + (size_t)((cod_i + e + nst) * H + h) * p.img_stride;
      mbar_arrive_expect_tx(&full_bar[st], il.bytes);
      bulk_g2s(stage, g, il.bytes, &full_bar[st]);
    }
    // outputs of the readout rows: o[t][h][v]
    for (int c0 = 0; c0 < QP; c0 += 16) {
      float ov[16];
      tmem_ld16(tO + lrow + c0, ov);
#pragma unroll
      for (int w = 0; w < 16; ++w) {
        const int qi = c0 + w;
        if (qi < mt.nq && v < V) {
          const int64_t t = (R0 + mt.p0 + (int64_t)qi * M) / M;
          p.out[(t * H + h) * (int64_t)V + v] = __float2bfloat16_rn(ov[w]);
        }
      }
    }
    tc_fence_before();
    if (__syncthreads_or(!ok2)) { aborted = true; break; }
    tc_fence_after();
  }

  if (aborted) {
    if (tid == 0) {
      set_status(p.status, GDP_DEV_ERR_TIMEOUT);
      mma_commit(&mma_bar);  // tracks every MMA issued so far
    }
    mbar_wait(&mma_bar, mma_phase);
    for (int s = 0; s < nst; ++s) mbar_wait(&full_bar[s], full_phase[s]);
  } else {
    // final state: dense output and/or cache slot
    float *dst = nullptr;
    if (p.cache) {
      if (slot >= 0) dst = p.cache + ((int64_t)slot * H + h) * (int64_t)V * d;
    } else if (p.out_state) {
      dst = p.out_state + ((int64_t)seq * H + h) * (int64_t)V * d;
    }
    for (int c0 = 0; c0 < d; c0 += 16) {
      float x[16];
      tmem_ld16(tS + lrow + c0, x);
      if (dst && v < V) {
#pragma unroll
        for (int u4 = 0; u4 < 16; u4 += 4)
          *reinterpret_cast<float4 *>(dst + (int64_t)v * d + c0 + u4) = make_float4(x[u4], x[u4 + 1], x[u4 + 2], x[u4 + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_free(tb, 256);
}

}  // namespace

cudaError_t launch_scan(const Problem &p, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  const size_t smem = (size_t)num_stages(p.K, p.qpad) * stage_bytes(p.K, p.qpad) + 1024;
  cudaError_t e = cudaFuncSetAttribute(gdp_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.N, (unsigned)p.H);
  gdp_scan_kernel<<<grid, kScanThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdp
