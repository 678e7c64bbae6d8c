// gdp_bwd_scan_tc.cu -- the backward pass's reverse state scan on the tcgen05 tensor cores.
//
// The derivative of the chunked recurrence (FlashInfer API page
// "flashinfer.gdp_prefill.chunk_gated_delta_product", display equation; the chunk form and its
// reverse dependence as in gdp_backward.cu): with D = dL/dS at an expanded chunk's exit, the
// gradient at its entry is
//   Z    = D Ktil^T + dO^T P                                      [V x 64]
//   D_in = gamma_last D - Z W + dO^T Qh                            [V x K]
// for the chunk's forward operands (Ktil, P, W, Qh; dO^T its readout rows' output gradients,
// [V x qpad]).  It is the forward scan's algebra with the transition transposed, so the kernel
// mirrors gdp_scan_kernel: one CTA per (sequence, head), D resident in TMEM as D_hat = D / Gamma
// (Gamma a running product of chunk decays) and updated in place by kind::tf32 MMAs whose A
// operand is read from TMEM; chunks run last to first.  With the fast image's -W and Qh divided
// by gamma_last and Gamma' = Gamma gamma_last:
//   batch 1:  Z_hat  = D_hat Ktil^T + O_hat P^T          (O_hat = dO^T / Gamma, preloaded)
//   batch 2:  D_hat += Z_hat (-W / gamma_last) + O_hat (Qh / gamma_last)    ( = D_in / Gamma')
// A slow image (gamma_last < 2^kFastMinLog2Gamma) is unscaled: D is renormalised to Gamma = 1
// before it and multiplied by gamma_last between its batches; Gamma is renormalised to 1 before
// it would drop below kRenormMinGamma.  The B operands come from the chunk's BwdImageLayout image
// (the forward's operands transposed, written by the WY kernel of the backward's forward
// recompute), two bulk copies into a double-buffered stage.  Every chunk's exit gradient
// D = Gamma D_hat (before its batch 2) is copied to one of two TMEM snapshots between the
// batches and stored to Dx by the store warps (TMA tensor stores of 32 x 32 boxes) while the
// chain goes on; the entry gradient of the first chunk is d_initial_state.  O_hat and Z_hat have
// one set of columns, refilled once the previous step's batch 2 is complete.
//
// Warp roles (320 threads): warp 8 lane 0 issues the MMAs, warp 9 lane 0 the image copies and
// the TMA loads of each step's output-gradient rows (a [qpad][V] box, a step ahead),
// warps 0-3 (prep, TMEM lane quadrants) preload O_hat, renormalise, copy the snapshots and apply
// slow-chunk decays, warps 4-7 (store) drain the snapshots and store d_initial_state.  Every
// wait is bounded (GDP_DEV_ERR_TIMEOUT on expiry).
#include <cuda.h>

#include "gdp_internal.cuh"
#include "gdp_scan_body.cuh"  // store_state_tma, kStTile
#include "gdp_sm100.cuh"

namespace gdp {
namespace {

using namespace sm100;

constexpr int kBtThreads = 320;
constexpr uint32_t kBtStageBudget = 200u * 1024u;

// a stage holds the image's two parts (the inverse after them stays in global memory)
__host__ __device__ inline uint32_t bt_stage_bytes(int d, int qpad) {
  return (BwdImageLayout(d, qpad).tinv + 1023u) & ~1023u;
}
__host__ __device__ inline int bt_stages(int d, int qpad) {
  return 2u * bt_stage_bytes(d, qpad) <= kBtStageBudget ? 2 : 1;
}
// the readout rows' output gradients of one step, [qpad][V] bf16 (one TMA box)
__host__ __device__ inline uint32_t bt_do_bytes(int qpad, int V) { return ((uint32_t)qpad * V * 2u + 1023u) & ~1023u; }
__host__ inline size_t bt_smem_bytes(int d, int qpad) {
  return (size_t)bt_stages(d, qpad) * bt_stage_bytes(d, qpad) + bt_do_bytes(qpad, d) + 4u * 2u * kStTile + 1024u;
}

// Per-chunk facts the prep warps hand to the store warps (one slot per TMEM buffer).
struct BtInfo {
  float gam_next;  // Gamma' after the chunk: the entry gradient is gam_next D_hat
};

__global__ void __launch_bounds__(kBtThreads, 1)
    gdp_bwd_tc_scan_kernel(BwdProblem p, const __grid_constant__ CUtensorMap tm_dx,
                           const __grid_constant__ CUtensorMap tm_dinit, const __grid_constant__ CUtensorMap tm_do) {
  const int seq = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;
  const int d = p.D, V = p.D, M = p.M, QP = p.qpad, H = p.H;
  const int q4 = warp & 3;
  const int v = q4 * 32 + lane;  // state row (TMEM lane) of prep and store threads
  const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
  const BwdImageLayout bl(d, QP);
  const uint32_t sbytes = bt_stage_bytes(d, QP);
  const int nst = bt_stages(d, QP);
  const int64_t sh = (int64_t)seq * H + h;
  const int64_t KV = (int64_t)d * V;
  const int64_t nchunks = (L * M + kChunk - 1) / kChunk;
  const int64_t cod_i = p.cod[seq];
  const int64_t nall = (cod_i < 0) ? 0 : max((int64_t)0, min(nchunks, p.ws_rows - cod_i));

  extern __shared__ __align__(1024) unsigned char bt_smem_raw[];
  // the 1024-aligned base as an offset into the shared array, so that accesses stay in the shared
  // address space
  unsigned char *sm = bt_smem_raw + ((1024u - (sm100::smem_u32(bt_smem_raw) & 1023u)) & 1023u);
  const uint16_t *dos = reinterpret_cast<const uint16_t *>(sm + nst * sbytes);  // [qpad][V] bf16
  unsigned char *sttiles = sm + nst * sbytes + bt_do_bytes(QP, V) + (uint32_t)q4 * 2u * kStTile;  // this store warp's
  __shared__ __align__(8) uint64_t full1[2], full2[2], o_ready[2], b1_done[2], b2_done[2], bk_free[2], mid_done,
      do_full, do_free, fin_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ BtInfo info[2];
  __shared__ float red[4];
  __shared__ volatile int abort_flag;
  const uint64_t wl = kWaitLimitNs;

  if (warp == 8) tmem_alloc(&tmem_slot, 512);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full1[i], 1);
      mbar_init(&full2[i], 1);
      mbar_init(&o_ready[i], 128);
      mbar_init(&b1_done[i], 1);
      mbar_init(&b2_done[i], 1);
      mbar_init(&bk_free[i], 128);
    }
    mbar_init(&mid_done, 128);
    mbar_init(&do_full, 1);
    mbar_init(&do_free, 128);
    mbar_init(&fin_bar, 1);
    mbar_init_fence();
    abort_flag = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // TMEM columns: [0, d) D_hat | from 128: O_hat (two buffers of qpad when qpad <= 32, used by
  // the steps in turn, so that the next step's O_hat is written while this step runs; one of 64
  // otherwise), then 64 of Z_hat | two exit-gradient snapshots at 256 and 384, used by the steps
  // in turn (every step emits one: with two, the store warps drain one while the next is copied)
  const uint32_t tb = tmem_slot;
  const bool dbl = QP <= 32;
  const uint32_t tD = tb, tZ = tb + 128u + (uint32_t)(dbl ? 2 * QP : QP);
  auto tO = [&](int b) { return tb + 128u + (dbl ? (uint32_t)b * (uint32_t)QP : 0u); };
  auto tBk = [&](int b) { return tb + 256u + (uint32_t)b * 128u; };
  const uint32_t id1 = idesc(kFmtTF32, 0, 0, 64, 128);  // Z_hat (+)= D_hat Ktil^T, O_hat P^T
  const uint32_t id2 = idesc(kFmtTF32, 0, 0, d, 128);   // D_hat += Z_hat (-W)', O_hat Qh'

  // processing step i runs expanded chunk nall - 1 - i
  auto image = [&](int64_t i) { return p.bimg + (size_t)((cod_i + nall - 1 - i) * H + h) * p.bimg_stride; };
  int n1[2] = {0, 0}, n2[2] = {0, 0}, n_do = 0;
  // the readout rows of step i's chunk follow from the sequence's geometry
  auto readouts = [&](int64_t i, int *nq, int64_t *tq0) {
    const int64_t e = nall - 1 - i;
    const int64_t R0 = bos * M + e * kChunk;  // first expanded row of the chunk
    const int len = (int)min((int64_t)kChunk, L * M - e * kChunk);
    const int p0 = (M - 1 - (int)(R0 % M)) % M;  // first readout row (t M + M - 1)
    *nq = (p0 < len) ? (len - 1 - p0) / M + 1 : 0;
    *tq0 = (R0 + p0) / M;
  };
  // producer: the output-gradient rows of step i (one box of qpad token rows; rows past the
  // chunk's readouts are ignored by the reader)
  auto load_do = [&](int64_t i) {
    int nq;
    int64_t tq0;
    readouts(i, &nq, &tq0);
    mbar_arrive_expect_tx(&do_full, (uint32_t)QP * V * 2u);
    tma_load_3d(const_cast<uint16_t *>(dos), &tm_do, 0, h, (int)tq0, &do_full);
    ++n_do;
  };
  auto load_part1 = [&](int64_t i) {
    const int st = (int)(i % nst);
    mbar_arrive_expect_tx(&full1[st], bl.part1);
    bulk_g2s(sm + st * sbytes, image(i), bl.part1, &full1[st]);
    ++n1[st];
  };
  auto load_part2 = [&](int64_t i) {
    const int st = (int)(i % nst);
    mbar_arrive_expect_tx(&full2[st], bl.part2);
    bulk_g2s(sm + st * sbytes + bl.b2, image(i) + bl.b2, bl.part2, &full2[st]);
    ++n2[st];
  };

  if (warp < 4) {
    // D_hat = dL/dS_final (zero without one); <dS_final, S_final> for the decay gradient
    const float *src = p.dfin ? p.dfin + sh * KV + (int64_t)v * d : nullptr;
    const float *fin = (p.dfin && p.fin) ? p.fin + sh * KV + (int64_t)v * d : nullptr;
    float part = 0.f;
    for (int c0 = 0; c0 < d; c0 += 16) {
      float x[16];
#pragma unroll
      for (int u4 = 0; u4 < 16; u4 += 4) {
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
        if (src && v < V) y = *reinterpret_cast<const float4 *>(src + c0 + u4);
        x[u4] = y.x; x[u4 + 1] = y.y; x[u4 + 2] = y.z; x[u4 + 3] = y.w;
        if (fin && v < V) {
          const float4 s4 = *reinterpret_cast<const float4 *>(fin + c0 + u4);
          part += y.x * s4.x + y.y * s4.y + y.z * s4.z + y.w * s4.w;
        }
      }
      tmem_st16(tD + lrow + c0, x);
    }
    tmem_st_wait();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) red[q4] = part;
    named_sync(2, 128);
    if (tid == 0 && p.tot) p.tot[sh] = red[0] + red[1] + red[2] + red[3];
  }
  if (warp == 9 && lane == 0) {
    for (int64_t i = 0; i < nst && i < nall; ++i) {
      load_part1(i);
      load_part2(i);
    }
    if (nall > 0) load_do(0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < 4) {
    // ---------------- prep warps ----------------
    // step j's meta from its stage (part 1 holds it; waits for the copy)
    auto stage_meta = [&](int64_t j, ImageMeta *m) {
      const int st = (int)(j % nst);
      if (!mbar_wait_or_abort(&full1[st], (uint32_t)((j / nst) & 1), &abort_flag, wl)) return false;
      *m = *reinterpret_cast<const ImageMeta *>(sm + st * sbytes + bl.meta);
      return true;
    };
    // the decay bookkeeping of a step entered with Gamma g: renormalise first?, Gamma during the
    // step's products, Gamma' after it
    struct Plan {
      bool renorm;
      float pass, next;
    };
    auto plan = [&](float g, const ImageMeta &m) {
      Plan r;
      const bool fast = m.fast != 0;
      r.renorm = fast ? (g * m.gamma_last < kRenormMinGamma) : (g != 1.f);
      r.pass = r.renorm ? 1.f : g;
      r.next = fast ? r.pass * m.gamma_last : 1.f;
      return r;
    };
    // O_hat of step j = dO^T / Gamma into buffer buf: column v of the step's output-gradient rows
    // (staged by the producer), zero past the readouts
    auto preload = [&](int64_t j, int buf, float gpass) {
      int nq;
      int64_t tq0;
      readouts(j, &nq, &tq0);
      if (!mbar_wait_or_abort(&do_full, (uint32_t)(j & 1), &abort_flag, wl)) return false;
      const float inv = 1.f / gpass;
      for (int c0 = 0; c0 < QP; c0 += 16) {
        float x[16];
#pragma unroll
        for (int w = 0; w < 16; ++w)
          x[w] = (c0 + w < nq && v < V) ? __uint_as_float((uint32_t)dos[(c0 + w) * V + v] << 16) * inv : 0.f;
        tmem_st16(tO(buf) + lrow + c0, x);
      }
      mbar_arrive(&do_free);  // the rows have been read
      return true;
    };
    float gam = 1.f;  // Gamma of D_hat
    ImageMeta mt{};
    bool ok = nall == 0 || stage_meta(0, &mt);
    if (ok && dbl && nall > 0) ok = preload(0, 0, plan(1.f, mt).pass);
    for (int64_t i = 0; ok && i < nall; ++i) {
      const int b = (int)(i & 1);
      const bool fast = mt.fast != 0;
      const Plan pl = plan(gam, mt);
      // Z_hat's columns and (one buffer) O_hat's are free once step i - 1's batch 2 is complete,
      // which also makes D_hat final for this step's renormalisation and snapshot
      if (i >= 1) {
        if (!mbar_wait_or_abort(&b2_done[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1), &abort_flag, wl)) break;
        tc_fence_after();
      }
      if (pl.renorm) {
        for (int c0 = 0; c0 < d; c0 += 32) {
          float x[32];
          tmem_ld32(tD + lrow + c0, x);
#pragma unroll
          for (int w = 0; w < 32; ++w) x[w] *= gam;
          tmem_st16(tD + lrow + c0, x);
          tmem_st16(tD + lrow + c0 + 16, x + 16);
        }
      }
      if (!dbl && !preload(i, 0, pl.pass)) break;
      if (tid == 0) info[b] = BtInfo{pl.next};
      tmem_st_wait();  // (also the O_hat written at the end of the last step)
      tc_fence_before();
      mbar_arrive(&o_ready[b]);
      // between the two batches: the snapshot D = Gamma D_hat (every step) into snapshot b, which
      // the store warps drained for step i - 2, and, for a slow image, D_hat <- gamma_last D_hat
      // once batch 1 has read it
      if (i >= 2 && !mbar_wait_or_abort(&bk_free[b], (uint32_t)(((i - 2) >> 1) & 1), &abort_flag, wl)) break;
      if (!fast && !mbar_wait_or_abort(&b1_done[b], (uint32_t)((i >> 1) & 1), &abort_flag, wl)) break;
      tc_fence_after();
      for (int c0 = 0; c0 < d; c0 += 32) {
        float x[32];
        tmem_ld32x(tD + lrow + c0, x);
#pragma unroll
        for (int w = 0; w < 32; ++w) x[w] *= pl.pass;
        tmem_st32x(tBk(b) + lrow + c0, x);
        if (!fast) {
#pragma unroll
          for (int w = 0; w < 32; ++w) x[w] *= mt.gamma_last;  // (the pass Gamma is 1 on a slow step)
          tmem_st32x(tD + lrow + c0, x);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&mid_done);
      gam = pl.next;
      if (i + 1 < nall) {
        // the next step's meta and, with two O_hat buffers, its O_hat (its buffer was last read
        // by step i - 1's batch 2, complete above), while this step's products run
        if (!stage_meta(i + 1, &mt)) break;
        if (dbl && !preload(i + 1, (int)((i + 1) & 1), plan(gam, mt).pass)) break;
      }
    }
    tmem_st_wait();  // (an aborted step may leave stores in flight; the columns are freed below)
  } else if (warp < 8) {
    // ---------------- store warps: exit gradients, then d_initial_state ----------------
    int nblk = 0;
    const bool has_rows = q4 * 32 < V;
    float gam_fin = 1.f;
    bool ok = true;
    for (int64_t i = 0; i < nall; ++i) {
      const int b = (int)(i & 1);
      // the snapshot of step i was copied before its batch 2 was issued; the decision is the
      // warp's (its TMEM loads are warp-wide)
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&b2_done[b], (uint32_t)((i >> 1) & 1), &abort_flag, wl));
      if (!ok) break;
      tc_fence_after();
      gam_fin = info[b].gam_next;
      const int64_t e = nall - 1 - i;
      if (has_rows) {  // bk_free: the snapshot columns have been read
        store_state_tma(tBk(b) + lrow, sttiles, lane, d, 1.f, &tm_dx, (int)(((cod_i + e) * H + h) * V + q4 * 32),
                        nblk, &bk_free[b]);
      } else {
        tc_fence_before();
        mbar_arrive(&bk_free[b]);
      }
    }
    if (ok && p.dinit && has_rows && __shfl_sync(0xffffffffu, abort_flag == 0 ? 1 : 0, 0))
      store_state_tma(tD + lrow, sttiles, lane, d, gam_fin, &tm_dinit, (int)(sh * V + q4 * 32), nblk, nullptr);
    if (lane == 0) bulk_wait_all();  // this warp's tensor stores are complete
  } else if (warp == 8) {
    if (lane == 0) {
      // ---------------- control thread: MMA issue ----------------
      for (int64_t i = 0; i < nall; ++i) {
        const int st = (int)(i % nst), b = (int)(i & 1);
        unsigned char *stage = sm + st * sbytes;
        if (!mbar_wait_or_abort(&full1[st], (uint32_t)((i / nst) & 1), &abort_flag, wl)) break;
        if (!mbar_wait_or_abort(&o_ready[b], (uint32_t)((i >> 1) & 1), &abort_flag, wl)) break;
        tc_fence_after();
        const uint32_t s1 = smem_u32(stage), s2 = smem_u32(stage) + bl.b2;
        for (int kk = 0; kk < d / 8; ++kk)
          mma_tf32_ts(tZ, tD + kk * 8, desc_sw128(s1 + bl.kt + (kk >> 2) * 8192u + (kk & 3) * 32u, 16, 1024), id1,
                      kk > 0);
        for (int kk = 0; kk < QP / 8; ++kk)
          mma_tf32_ts(tZ, tO(b) + kk * 8, desc_sw128(s1 + bl.pt + (kk >> 2) * 8192u + (kk & 3) * 32u, 16, 1024), id1,
                      1);
        mma_commit(&b1_done[b]);
        if (!mbar_wait_or_abort(&full2[st], (uint32_t)((i / nst) & 1), &abort_flag, wl)) break;
        if (!mbar_wait_or_abort(&mid_done, (uint32_t)(i & 1), &abort_flag, wl)) break;
        tc_fence_after();
        for (int kk = 0; kk < kChunk / 8; ++kk)
          mma_tf32_ts(tD, tZ + kk * 8,
                      desc_sw128(s2 + (bl.wt - bl.b2) + (kk >> 2) * bl.wt_block + (kk & 3) * 32u, 16, 1024), id2, 1);
        for (int kk = 0; kk < QP / 8; ++kk)
          mma_tf32_ts(tD, tO(b) + kk * 8,
                      desc_sw128(s2 + (bl.qt - bl.b2) + (kk >> 2) * bl.wt_block + (kk & 3) * 32u, 16, 1024), id2, 1);
        mma_commit(&b2_done[b]);
      }
      if (abort_flag) {
        // drain every MMA issued so far before the columns are freed
        mma_commit(&fin_bar);
        mbar_wait(&fin_bar, 0);
        set_status(p.status, GDP_DEV_ERR_TIMEOUT);
      }
    }
  } else if (lane == 0) {
    // ---------------- producer thread: image copies and output-gradient rows ----------------
    for (int64_t i = 0; i < nall; ++i) {
      const int b = (int)(i & 1);
      // step i's rows have been read: the next step's go into the same buffer
      if (!mbar_wait_or_abort(&do_free, (uint32_t)(i & 1), &abort_flag, wl)) break;
      if (i + 1 < nall) load_do(i + 1);
      if (i + nst >= nall) continue;
      if (!mbar_wait_or_abort(&b1_done[b], (uint32_t)((i >> 1) & 1), &abort_flag, wl)) break;
      load_part1(i + nst);
      if (!mbar_wait_or_abort(&b2_done[b], (uint32_t)((i >> 1) & 1), &abort_flag, wl)) break;
      load_part2(i + nst);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (abort_flag && warp == 9 && lane == 0)
    for (int st = 0; st < nst; ++st) {  // bounded; the last copy issued on each barrier has landed
      if (n1[st] > 0) mbar_wait(&full1[st], (uint32_t)((n1[st] - 1) & 1));
      if (n2[st] > 0) mbar_wait(&full2[st], (uint32_t)((n2[st] - 1) & 1));
      if (st == 0 && n_do > 0) mbar_wait(&do_full, (uint32_t)((n_do - 1) & 1));
    }
  __syncthreads();
  if (warp == 8) tmem_free(tb, 512);
}

}  // namespace

size_t bwd_tc_scan_smem(int d, int qpad) { return bt_smem_bytes(d, qpad); }
size_t bwd_image_stride(int d, int qpad) { return (BwdImageLayout(d, qpad).bytes + 1023u) & ~1023u; }

cudaError_t launch_bwd_tc_scan(const BwdProblem &p, cudaStream_t stream) {
  const size_t smem = bt_smem_bytes(p.D, p.qpad);
  cudaError_t e =
      cudaFuncSetAttribute(gdp_bwd_tc_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap tm_dx, tm_dinit, tm_do;
  // the output gradients [T][H][V] bf16 in boxes of qpad token rows (rows past T read as zero)
  if ((e = tmap_out_rows(&tm_do, const_cast<__nv_bfloat16 *>(p.dout), p.T, p.H, p.D, p.qpad, 0)) != cudaSuccess)
    return e;
  const int64_t hv = (int64_t)p.H * p.D;
  if ((e = tmap_state(&tm_dx, p.Dx, p.ntdp_pad * hv, p.D)) != cudaSuccess) return e;
  if ((e = tmap_state(&tm_dinit, p.dinit ? p.dinit : p.Dx, p.dinit ? p.N * hv : p.ntdp_pad * hv, p.D)) !=
      cudaSuccess)
    return e;
  gdp_bwd_tc_scan_kernel<<<dim3((unsigned)p.N, (unsigned)p.H), kBtThreads, smem, stream>>>(p, tm_dx, tm_dinit,
                                                                                           tm_do);
  return cudaGetLastError();
}

}  // namespace gdp
