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
// One CTA per (sequence, head); TMEM lane v = state row v.  S lives in TMEM
// columns [0, d) for the whole sequence and is read by the MMAs directly as
// the tf32 A operand, so the recurrence never leaves the SM.  All
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

// Warp roles (warp specialisation keeps loads and stores off the serial chain):
//   warp 8     control : image copies (bulk TMA) and MMA issue
//   warps 0-3  state   : S <- gamma_last S (+ unscaled copy at token-chunk starts),
//                        V_new += U^T, then the chunk's o columns -> a 2-slot TMEM ring
//   warps 4-7  store   : ring -> bf16 outputs, state copy -> chunk_states, final state
// Per chunk the chain is: batch 1 -> state pass -> batch 2 -> ring copy -> next batch 1.
// An SM stores only ~30 B/cycle, so outputs and 64 KB state snapshots drain behind it.
// TMEM lanes: state and store warps w access lanes 32 (w % 4) .. +31.
constexpr int kScanThreads = 288;
constexpr uint32_t kScanSmemBudget = 200u * 1024u;  // operand stages
constexpr uint32_t kXpose = 32u * 36u * 4u;         // per store warp: 32 x 36 fp32 transpose tile

__host__ __device__ inline uint32_t stage_bytes(int d, int qpad) {
  return (ImageLayout(d, qpad).bytes + 1023u) & ~1023u;
}
__host__ __device__ inline int num_stages(int d, int qpad) {
  return 2u * stage_bytes(d, qpad) <= kScanSmemBudget ? 2 : 1;
}
__host__ __device__ inline uint32_t obuf_bytes(int qpad, int V) { return (uint32_t)qpad * V * 2u; }
__host__ inline size_t scan_smem_bytes(int d, int qpad, int V) {
  return (size_t)num_stages(d, qpad) * stage_bytes(d, qpad) + obuf_bytes(qpad, V) + 4u * kXpose + 1024u;
}

// Store warp: rows [row0, row0 + 32) of a [V][d] fp32 block from this warp's TMEM
// lanes (columns from t_lane).  Each 32 x 32 block goes through a shared tile
// (rows padded to 36 floats: 16-byte aligned, conflict-free) so that every global
// store instruction writes four full 128-byte row segments with 16-byte stores.
__device__ __forceinline__ void store_state_rows(uint32_t t_lane, float *xb, int lane, int row0, int V, int d,
                                                 float *dst) {
  const int rq = lane >> 3, cq = (lane & 7) * 4;  // this lane's row (of 4) and column in a store
  for (int c0 = 0; c0 < d; c0 += 32) {
    float x[32];
    tmem_ld32(t_lane + c0, x);
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      *reinterpret_cast<float4 *>(xb + lane * 36 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
    __syncwarp();
#pragma unroll
    for (int r0 = 0; r0 < 32; r0 += 4) {
      const int r = r0 + rq;
      if (row0 + r < V)
        *reinterpret_cast<float4 *>(dst + (int64_t)(row0 + r) * d + c0 + cq) =
            *reinterpret_cast<const float4 *>(xb + r * 36 + cq);
    }
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kScanThreads, 1) gdp_scan_kernel(Problem p) {
  const int seq = blockIdx.x, h = blockIdx.y;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;  // flagged by the descriptor kernel
  const int d = p.K, V = p.V, M = p.M, QP = p.qpad, H = p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3;
  const int v = q4 * 32 + lane;  // state row (TMEM lane) of state and store threads
  const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
  const ImageLayout il(d, QP);
  const uint32_t sbytes = stage_bytes(d, QP);
  const int nst = num_stages(d, QP);

  extern __shared__ __align__(1024) unsigned char scan_smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)scan_smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char *obuf = sm + nst * sbytes;  // [qpad][V] bf16 output staging
  float *xb = reinterpret_cast<float *>(obuf + obuf_bytes(QP, V)) + q4 * 32 * 36;
  __shared__ __align__(8) uint64_t full_bar[2], b1_done, b2_done, spass_done, o_free, ring_full[2], ring_free[2],
      bk_free, fin_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int ring_nq[2], ring_p0[2];
  __shared__ volatile int abort_flag;

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
  auto emits = [&](int64_t e) { return p.chunk_states && (e % M == 0) && co_i >= 0 && co_i + e / M < p.nt_pad; };

  if (warp == 8) tmem_alloc(&tmem_slot, 512);
  if (tid == 0) {
    mbar_init(&full_bar[0], 1);
    mbar_init(&full_bar[1], 1);
    mbar_init(&b1_done, 1);
    mbar_init(&b2_done, 1);
    mbar_init(&spass_done, 128);
    mbar_init(&o_free, 128);
    mbar_init(&ring_full[0], 128);
    mbar_init(&ring_full[1], 128);
    mbar_init(&ring_free[0], 128);
    mbar_init(&ring_free[1], 128);
    mbar_init(&bk_free, 128);
    mbar_init(&fin_bar, 1);
    mbar_init_fence();
    abort_flag = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // TMEM columns: [S: d][o^T: qpad][V_new^T: 64] | 256: o ring 2 x 64 | 384: state copy 128.
  // [o | V_new] and [S | o] are each contiguous, so one MMA per K step serves both
  // products that share an A operand.
  const uint32_t tb = tmem_slot;
  const uint32_t tS = tb, tO = tb + d, tVn = tb + d + QP, tRing = tb + 256, tBk = tb + 384;
  const uint32_t id1 = idesc(kFmtTF32, 0, 0, QP + 64, 128);  // [o | V_new] = S [Qh ; -W]^T
  const uint32_t id2s = idesc(kFmtTF32, 0, 0, d, 128);       // S += V_new^T Ktil
  const uint32_t id2o = idesc(kFmtTF32, 0, 0, QP, 128);      // o += V_new^T P^T

  if (warp < 4) {
    // S_0 into TMEM (rows >= V stay zero)
    for (int c0 = 0; c0 < d; c0 += 16) {
      float x[16];
#pragma unroll
      for (int u4 = 0; u4 < 16; u4 += 4) {
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
        if (src && v < V) y = *reinterpret_cast<const float4 *>(src + (int64_t)v * d + c0 + u4);
        x[u4] = y.x; x[u4 + 1] = y.y; x[u4 + 2] = y.z; x[u4 + 3] = y.w;
      }
      tmem_st16(tS + lrow + c0, x);
    }
    tmem_st_wait();
  }
  if (warp == 8 && lane == 0) {
    for (int s = 0; s < nst && s < nrun; ++s) {
      mbar_arrive_expect_tx(&full_bar[s], il.bytes);
      bulk_g2s(sm + s * sbytes, p.img + (size_t)((cod_i + s) * H + h) * p.img_stride, il.bytes, &full_bar[s]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < 4) {
    // ---------------- state warps ----------------
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
    for (int64_t e = 0; e < nrun; ++e) {
      if (!mbar_wait_or_abort(&b1_done, (uint32_t)(e & 1), &abort_flag)) break;
      tc_fence_after();
      const ImageMeta mt = *reinterpret_cast<const ImageMeta *>(sm + (e % nst) * sbytes + il.meta);
      const bool emit = emits(e);
      if (emit && e / M >= 1) {  // the store warps have drained the previous state copy
        if (!mbar_wait_or_abort(&bk_free, (uint32_t)((e / M - 1) & 1), &abort_flag)) break;
        tc_fence_after();
      }
      for (int c0 = 0; c0 < d; c0 += 32) {
        float x[32];
        tmem_ld32(tS + lrow + c0, x);
        if (emit) {
          tmem_st16(tBk + lrow + c0, x);
          tmem_st16(tBk + lrow + c0 + 16, x + 16);
        }
#pragma unroll
        for (int w = 0; w < 32; ++w) x[w] *= mt.gamma_last;
        tmem_st16(tS + lrow + c0, x);
        tmem_st16(tS + lrow + c0 + 16, x + 16);
      }
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        float x[32];
        tmem_ld32(tVn + lrow + c0, x);
#pragma unroll
        for (int w = 0; w < 32; ++w) x[w] += u[c0 + w];
        tmem_st16(tVn + lrow + c0, x);
        tmem_st16(tVn + lrow + c0 + 16, x + 16);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&spass_done);
      if (e + 1 < nrun) load_u(e + 1);  // next chunk's U^T, in flight while batch 2 runs

      if (!mbar_wait_or_abort(&b2_done, (uint32_t)(e & 1), &abort_flag)) break;
      tc_fence_after();
      if (e >= 2 && !mbar_wait_or_abort(&ring_free[e & 1], (uint32_t)(((e >> 1) - 1) & 1), &abort_flag)) break;
      tc_fence_after();
      const uint32_t slot_col = tRing + (uint32_t)(e & 1) * 64u;
      for (int c0 = 0; c0 < QP; c0 += 16) {
        float x[16];
        tmem_ld16(tO + lrow + c0, x);
        tmem_st16(slot_col + lrow + c0, x);
      }
      if (tid == 0) {
        ring_nq[e & 1] = mt.nq;
        ring_p0[e & 1] = mt.p0;
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&o_free);
      mbar_arrive(&ring_full[e & 1]);
    }
  } else if (warp < 8) {
    // ---------------- store warps ----------------
    for (int64_t e = 0; e < nrun; ++e) {
      if (!mbar_wait_or_abort(&ring_full[e & 1], (uint32_t)((e >> 1) & 1), &abort_flag)) break;
      tc_fence_after();
      const int nq = ring_nq[e & 1], p0 = ring_p0[e & 1];
      float ov[64];
      const uint32_t slot_col = tRing + (uint32_t)(e & 1) * 64u;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16)
        if (c0 < QP) tmem_ld16(slot_col + lrow + c0, ov + c0);
      tc_fence_before();
      mbar_arrive(&ring_free[e & 1]);
      // outputs: bf16 staging [q][v], then full-row 16-byte stores
      named_sync(1, 128);  // every thread has finished reading the previous chunk's staging
      if (v < V) {
#pragma unroll
        for (int w = 0; w < 64; ++w)
          if (w < nq) *reinterpret_cast<__nv_bfloat16 *>(obuf + ((uint32_t)w * V + v) * 2u) = __float2bfloat16_rn(ov[w]);
      }
      named_sync(1, 128);
      const int64_t tq0 = (bos * M + e * kChunk + p0) / M;  // readout rows are consecutive tokens
      const int cpr = V / 8;                                  // 16-byte chunks per output row
      for (int c = tid - 128; c < nq * cpr; c += 128) {
        const int qi = c / cpr, ch = c % cpr;
        *reinterpret_cast<uint4 *>(p.out + ((tq0 + qi) * H + h) * (int64_t)V + ch * 8) =
            *reinterpret_cast<const uint4 *>(obuf + ((uint32_t)qi * V + ch * 8) * 2u);
      }
      if (emits(e)) {  // the state warps copied S_e before filling this ring slot
        float *dst = p.chunk_states + ((co_i + e / M) * H + h) * (int64_t)V * d;
        store_state_rows(tBk + lrow, xb, lane, q4 * 32, V, d, dst);
        tc_fence_before();
        mbar_arrive(&bk_free);
      }
    }
    if (!abort_flag && (nrun == 0 || mbar_wait_or_abort(&b2_done, (uint32_t)((nrun - 1) & 1), &abort_flag))) {
      tc_fence_after();
      float *dst = nullptr;
      if (p.cache) {
        if (slot >= 0) dst = p.cache + ((int64_t)slot * H + h) * (int64_t)V * d;
      } else if (p.out_state) {
        dst = p.out_state + ((int64_t)seq * H + h) * (int64_t)V * d;
      }
      if (dst) store_state_rows(tS + lrow, xb, lane, q4 * 32, V, d, dst);
    }
  } else if (lane == 0) {
    // ---------------- control thread: image loads and MMA issue ----------------
    for (int64_t e = 0; e < nrun; ++e) {
      const int st = (int)(e % nst);
      unsigned char *stage = sm + st * sbytes;
      if (!mbar_wait_or_abort(&full_bar[st], (uint32_t)((e / nst) & 1), &abort_flag)) break;
      if (e >= 1 && !mbar_wait_or_abort(&o_free, (uint32_t)((e - 1) & 1), &abort_flag)) break;
      tc_fence_after();
      const uint32_t sb1 = smem_u32(stage) + il.b1, sb2 = smem_u32(stage) + il.b2;
      for (int kk = 0; kk < d / 8; ++kk)
        mma_tf32_ts(tO, tS + kk * 8, desc_sw128(sb1 + (kk >> 2) * il.b1_block + (kk & 3) * 32u, 16, 1024), id1,
                    kk > 0);
      mma_commit(&b1_done);
      if (!mbar_wait_or_abort(&spass_done, (uint32_t)(e & 1), &abort_flag)) break;
      tc_fence_after();
      // two MMAs per K step (N = d and N = qpad): past N = 128 an MMA costs far more than
      // two narrower ones (measured)
      for (int kk = 0; kk < kChunk / 8; ++kk) {
        const uint32_t bk = sb2 + (kk >> 2) * il.b2_block + (kk & 3) * 32u;
        mma_tf32_ts(tS, tVn + kk * 8, desc_sw128(bk, 16, 1024), id2s, 1);
        mma_tf32_ts(tO, tVn + kk * 8, desc_sw128(bk + (uint32_t)d * 128u, 16, 1024), id2o, 1);
      }
      mma_commit(&b2_done);
      if (e + nst < nrun) {  // the stage is free once this chunk's products are done
        if (!mbar_wait_or_abort(&b2_done, (uint32_t)(e & 1), &abort_flag)) break;
        fence_async_smem();
        mbar_arrive_expect_tx(&full_bar[st], il.bytes);
        bulk_g2s(stage, p.img + (size_t)((cod_i + e + nst) * H + h) * p.img_stride, il.bytes, &full_bar[st]);
      }
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
  if (abort_flag && warp == 8 && lane == 0)
    for (int s = 0; s < nst; ++s) mbar_wait(&full_bar[s], 0);  // bounded; covers a copy still landing
  __syncthreads();
  if (warp == 8) tmem_free(tb, 512);
}

}  // namespace

cudaError_t launch_scan(const Problem &p, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  const size_t smem = scan_smem_bytes(p.K, p.qpad, p.V);
  cudaError_t e = cudaFuncSetAttribute(gdp_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.N, (unsigned)p.H);
  gdp_scan_kernel<<<grid, kScanThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdp
