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
constexpr uint32_t kScanSmemBudget = 200u * 1024u;   // operand stages
constexpr uint32_t kXposeBytes = 4u * 32u * 33u * 4u;  // per-warp 32 x 33 fp32 transpose buffers

__host__ __device__ inline uint32_t stage_bytes(int d, int qpad) {
  return (ImageLayout(d, qpad).bytes + 1023u) & ~1023u;
}
__host__ __device__ inline int num_stages(int d, int qpad) {
  return 2u * stage_bytes(d, qpad) <= kScanSmemBudget ? 2 : 1;
}

// Rows 32w..32w+31 of a [V][d] fp32 state block <-> TMEM lanes of warp w, with
// every global access a full 128-byte row segment (transposed through a
// 32 x 33 shared buffer).  scale multiplies what is written back to TMEM.
__device__ __forceinline__ void state_to_global(uint32_t t_lane, float *xb, int lane, int row0, int V, int d,
                                                float *dst, float scale_back, bool write_back) {
  for (int c0 = 0; c0 < d; c0 += 32) {
    float x[32];
    tmem_ld16(t_lane + c0, x);
    tmem_ld16(t_lane + c0 + 16, x + 16);
    if (dst) {
#pragma unroll
      for (int j = 0; j < 32; ++j) xb[lane * 33 + j] = x[j];
      __syncwarp();
      for (int r = 0; r < 32; ++r)
        if (row0 + r < V) dst[(int64_t)(row0 + r) * d + c0 + lane] = xb[r * 33 + lane];
      __syncwarp();
    }
    if (write_back) {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] *= scale_back;
      tmem_st16(t_lane + c0, x);
      tmem_st16(t_lane + c0 + 16, x + 16);
    }
  }
}

__global__ void __launch_bounds__(kScanThreads, 1) gdp_scan_kernel(Problem p) {
  const int seq = blockIdx.x, h = blockIdx.y;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;  // flagged by the descriptor kernel
  const int d = p.K, V = p.V, M = p.M, QP = p.qpad, H = p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int v = tid;  // state row = TMEM lane
  const ImageLayout il(d, QP);
  const uint32_t sbytes = stage_bytes(d, QP);
  const int nst = num_stages(d, QP);

  extern __shared__ __align__(1024) unsigned char scan_smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)scan_smem_raw + 1023) & ~(uintptr_t)1023);
  float *xb = reinterpret_cast<float *>(sm + nst * sbytes) + warp * 32 * 33;
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
  // TMEM columns: [S: d][o^T: qpad][V_new^T: 64] -- [o | V_new] and [S | o] are each contiguous,
  // so one MMA per K step serves both products that share an A operand.
  const uint32_t tb = tmem_slot;
  const uint32_t lrow = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tb, tO = tb + d, tVn = tb + d + QP;
  const int row0 = warp * 32;

  // S_0 into TMEM (coalesced reads through the transpose buffer; rows >= V stay zero)
  for (int c0 = 0; c0 < d; c0 += 32) {
    for (int r = 0; r < 32; ++r)
      xb[r * 33 + lane] = (src && row0 + r < V) ? src[(int64_t)(row0 + r) * d + c0 + lane] : 0.f;
    __syncwarp();
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = xb[lane * 33 + j];
    __syncwarp();
    tmem_st16(tS + lrow + c0, x);
    tmem_st16(tS + lrow + c0 + 16, x + 16);
  }
  // U^T row v of the first chunk into registers
  float u[64];
  auto load_u = [&](int64_t e) {
    const float4 *Ut = reinterpret_cast<const float4 *>(p.U + (((cod_i + e) * H + h) * V + (v < V ? v : 0)) * kChunk);
#pragma unroll
    for (int s4 = 0; s4 < 16; ++s4) {
      const float4 x = (v < V) ? Ut[s4] : make_float4(0.f, 0.f, 0.f, 0.f);
      u[4 * s4] = x.x; u[4 * s4 + 1] = x.y; u[4 * s4 + 2] = x.z; u[4 * s4 + 3] = x.w;
    }
  };
  if (nrun > 0) load_u(0);
  tmem_st_wait();

  uint32_t full_phase[2] = {0, 0}, mma_phase = 0;
  bool aborted = false;
  const uint32_t id1 = idesc(kFmtTF32, 0, 0, QP + 64, 128);  // [o | V_new] += S [Qh ; -W]^T
  const uint32_t id2 = idesc(kFmtTF32, 0, 0, d + QP, 128);   // [S | o] += V_new^T [Ktil^T ; P]^T
  const float zeros[16] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int64_t e = 0; e < nrun; ++e) {
    const int st = (int)(e % nst);
    unsigned char *stage = sm + st * sbytes;
    // V_new^T <- U^T and o^T <- 0 (both accumulated onto by the first batch)
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) tmem_st16(tVn + lrow + c0, u + c0);
    for (int c0 = 0; c0 < QP; c0 += 16) tmem_st16(tO + lrow + c0, zeros);
    tmem_st_wait();
    if (e + 1 < nrun) load_u(e + 1);  // next chunk's U^T, in flight while this chunk computes
    const bool okf = mbar_wait(&full_bar[st], full_phase[st]);
    full_phase[st] ^= 1u;
    tc_fence_before();
    if (__syncthreads_or(!okf)) { aborted = true; break; }
    tc_fence_after();
    const ImageMeta mt = *reinterpret_cast<const ImageMeta *>(stage + il.meta);

    // batch 1: [o^T | V_new^T] += S [Qh ; -W]^T
    if (tid == 0) {
      const uint32_t sb = smem_u32(stage) + il.b1;
      for (int kk = 0; kk < d / 8; ++kk)
        mma_tf32_ts(tO, tS + kk * 8, desc_sw128(sb + (kk >> 2) * il.b1_block + (kk & 3) * 32u, 16, 1024), id1, 1);
      mma_commit(&mma_bar);
    }
    const bool ok1 = mbar_wait(&mma_bar, mma_phase);
    mma_phase ^= 1u;
    tc_fence_after();

    // state pass: emit the entering state at token-chunk starts, then S <- gamma_last S
    const bool emit = p.chunk_states && (e % M == 0) && co_i >= 0 && co_i + e / M < p.nt_pad;
    float *cs = emit ? p.chunk_states + ((co_i + e / M) * H + h) * (int64_t)V * d : nullptr;
    state_to_global(tS + lrow, xb, lane, row0, V, d, cs, mt.gamma_last, true);
    tmem_st_wait();
    tc_fence_before();
    if (__syncthreads_or(!ok1)) { aborted = true; break; }
    tc_fence_after();

    // batch 2: [S | o^T] += V_new^T [Ktil^T ; P]^T
    if (tid == 0) {
      const uint32_t sb = smem_u32(stage) + il.b2;
      for (int kk = 0; kk < kChunk / 8; ++kk)
        mma_tf32_ts(tS, tVn + kk * 8, desc_sw128(sb + (kk >> 2) * il.b2_block + (kk & 3) * 32u, 16, 1024), id2, 1);
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
    // outputs of the readout rows: consecutive readout rows are consecutive tokens
    const int64_t tq0 = (bos * M + e * kChunk + mt.p0) / M;
    for (int c0 = 0; c0 < QP; c0 += 16) {
      float ov[16];
      tmem_ld16(tO + lrow + c0, ov);
#pragma unroll
      for (int w = 0; w < 16; ++w) {
        const int qi = c0 + w;
        if (qi < mt.nq && v < V) p.out[((tq0 + qi) * H + h) * (int64_t)V + v] = __float2bfloat16_rn(ov[w]);
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
    state_to_global(tS + lrow, xb, lane, row0, V, d, dst, 1.f, false);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_free(tb, 256);
}

}  // namespace

cudaError_t launch_scan(const Problem &p, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  const size_t smem = (size_t)num_stages(p.K, p.qpad) * stage_bytes(p.K, p.qpad) + kXposeBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(gdp_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.N, (unsigned)p.H);
  gdp_scan_kernel<<<grid, kScanThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdp
