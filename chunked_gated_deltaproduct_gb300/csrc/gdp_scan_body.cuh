// gdp_scan_body.cuh -- inter-chunk state scan, output combine and state scatter on the
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
// One CTA per (sequence, head); TMEM lane v = state row v.  The state lives in
// TMEM columns [0, d) for the whole sequence as S_hat = S / Gamma (Gamma: a
// running product of chunk decays), read by the MMAs directly as the tf32 A
// operand and updated in place by them, so the recurrence never leaves the
// SM and no thread touches it on the serial chain.  With the operands of a
// "fast" image pre-divided by gamma_last (gdp_internal.cuh) and Gamma' = Gamma
// gamma_last, the chunk's update is the same algebra in scaled form:
//   Y       = U^T / Gamma' + S_hat (-W / gamma_last)^T    ( = V_new^T / Gamma')
//   o_hat   = S_hat (Qh / gamma_last)^T + Y P^T           ( = o^T / Gamma')
//   S_hat  += Y Ktil                                      ( = S_{e+1} / Gamma')
// Y starts as U^T / Gamma' (written into TMEM by threads ahead of time), so a
// chunk is two MMA batches back to back on the tensor pipe.  A "slow" image
// (gamma_last < 2^kFastMinLog2Gamma, e.g. 0) is unscaled: the state is
// renormalised to Gamma = 1 before it and scaled by gamma_last between its
// two batches.  Gamma is renormalised to 1 whenever it would fall below
// kRenormMinGamma.  All products are kind::tf32 (fp32 operands truncated to
// tf32, fp32 accumulate): the state feeds back into every later chunk, and
// bf16 operands would add a ~2^-9 relative error per chunk.  The B operands
// come from one operand image per chunk (written by the WY kernel), fetched by
// two bulk copies into a double-buffered shared-memory stage while the
// previous chunk computes.
//
// The same kernel runs three other grids (Problem fields piece_len, piece_pass1, xfer):
// the two passes of split chains (one CTA per piece of a sequence: pass 1 from a zero
// state and from the identity with U^T read as zero, storing the piece's B and Phi;
// pass 2 from the piece's entering state), and the transfer pairs of whole sequences
// (one CTA per sequence from zero, one from the identity).  A launch without outputs
// skips the o_hat products and stores.
#pragma once
#include <cuda.h>  // CUtensorMap

#include "gdp_internal.cuh"
#include "gdp_sm100.cuh"

namespace gdp {
namespace {

using namespace sm100;

// Warp roles:
//   warp 8     control : MMA issue
//   warp 9     producer: image copies (bulk TMA); part 1 of a stage is refilled once batch 1
//                        has read it, part 2 once batch 2 has
//   warps 0-3  prep    : per chunk, Y <- U^T / Gamma' and o_hat <- 0 in the chunk's TMEM
//                        buffer (two buffers), renormalisation, the state snapshot at
//                        token-chunk starts (-> TMEM copy) and the slow-image decay
//   warps 4-7  store   : o_hat * Gamma' -> bf16 outputs, snapshot -> chunk_states,
//                        final state (states leave by TMA tensor stores of 32 x 32 blocks,
//                        so the load/store unit that the control warp shares stays free)
// TMEM lanes: prep and store warps w access lanes 32 (w % 4) .. +31.
constexpr int kScanThreads = 320;
constexpr uint32_t kScanSmemBudget = 200u * 1024u;  // operand stages
constexpr uint32_t kStTile = 4096u;                 // one 32 x 32 fp32 box, 128-byte swizzle

__host__ __device__ inline uint32_t stage_bytes(int d, int qpad) {
  return (ImageLayout(d, qpad).bytes + 1023u) & ~1023u;
}
__host__ __device__ inline int num_stages(int d, int qpad) {
  return 2u * stage_bytes(d, qpad) <= kScanSmemBudget ? 2 : 1;
}
__host__ __device__ inline uint32_t obuf_bytes(int qpad, int V) { return (uint32_t)qpad * V * 2u; }
__host__ inline size_t scan_smem_bytes(int d, int qpad, int V) {
  return (size_t)num_stages(d, qpad) * stage_bytes(d, qpad) + obuf_bytes(qpad, V) + 4u * 2u * kStTile + 1024u;
}

// Store warp: the state rows held in this warp's TMEM lanes (columns from t_lane), times
// mul, to map rows [row, row + 32).  The columns are read from TMEM 64 at a time under one
// wait; `read` (when given) is arrived on once the last of them is in registers, since the
// columns may be overwritten from there on.  Per 32 columns the rows leave as one 32 x 32 box
// staged in shared memory (row r at r * 128 bytes, 16-byte chunk j at position j ^ (r & 7):
// the map's 128-byte swizzle, conflict-free for a thread per row) and written by one TMA
// tensor store.  The warp's two tiles alternate; nblk counts the boxes this warp has issued.
__device__ __forceinline__ void store_state_tma(uint32_t t_lane, unsigned char *tiles, int lane, int d, float mul,
                                                const CUtensorMap *tm, int row, int &nblk, uint64_t *read) {
#pragma unroll 1
  for (int c0 = 0; c0 < d; c0 += 64) {
    uint32_t x[64];
    tmem_ld32x_nw(t_lane + c0, x);
    tmem_ld32x_nw(t_lane + c0 + 32, x + 32);
    tmem_ld_wait();
    if (read && c0 + 64 >= d) {
      tc_fence_before();
      mbar_arrive(read);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      unsigned char *tile = tiles + (uint32_t)(nblk & 1) * kStTile;
      if (nblk >= 2) {  // the store issued from this tile two boxes ago has read it
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t *y = x + 32 * c + 4 * j;
        *reinterpret_cast<float4 *>(tile + lane * 128 + ((j ^ (lane & 7)) << 4)) =
            make_float4(mul * __uint_as_float(y[0]), mul * __uint_as_float(y[1]), mul * __uint_as_float(y[2]),
                        mul * __uint_as_float(y[3]));
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tm, tile, c0 + 32 * c, row);
        bulk_commit();
      }
      ++nblk;
    }
  }
}

// Per-chunk facts the prep warps hand to the store warps (one slot per TMEM buffer).
struct ChunkInfo {
  float out_scale;  // Gamma' of the chunk: o = Gamma' o_hat
  int nq, p0;
};

// The kernel body.  F16: the output is float16 (else bfloat16).  INIT16: the dense initial
// state is bfloat16 (else fp32).  Compile-time, so that the common kernel carries no code for
// the other types; each type pair has a plain __global__ kernel below (a template kernel
// came out larger than the same body in a plain one).
template <bool F16, bool INIT16>
__device__ __forceinline__ void scan_body(const Problem &p, const CUtensorMap &tm_cs, const CUtensorMap &tm_fin,
                                          const CUtensorMap &tm_seg, const CUtensorMap &tm_out_a,
                                          const CUtensorMap &tm_out_b) {
  int h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // split chains: this CTA's piece (pass 1: grid row r and piece_rows + r run the same piece)
  const bool pieces = p.piece_len > 0, pass1 = pieces && p.piece_pass1, xfer = p.xfer != 0;
  // from the identity with V = 0: the second half of the rows of a pass 1 or a transfer-pair launch
  const bool transfer = (pass1 && (int)blockIdx.x >= p.piece_rows) || (xfer && (int64_t)blockIdx.x >= p.N);
  int seq = (xfer && transfer) ? (int)(blockIdx.x - p.N) : (int)blockIdx.x, pc_i = 0, pc_n = 1;
  if (p.order && !pieces && !xfer) {
    // longest first: linear CTA index l (the order CTAs start in) runs sequence order[l / H],
    // head l % H, so that the longest chains do not start in the last wave; the order comes
    // from the descriptor kernel
    pdl_wait();
    const int64_t l = (int64_t)blockIdx.x + (int64_t)blockIdx.y * gridDim.x;
    if (!in_range(p.bounds, p.status, GDP_BOUNDS_SITE_SCAN_ORDER, l / p.H, p.N)) return;
    seq = p.order[l / p.H];
    h = (int)(l % p.H);
    if (!in_range(p.bounds, p.status, GDP_BOUNDS_SITE_SCAN_ORDER, seq, p.N)) return;
  }
  if (pieces) {
    // the piece table comes from the descriptors; every CTA waits for its predecessor grid
    // before it may exit, so that this grid's completion implies the predecessors'
    pdl_wait();
    pdl_trigger();
    __shared__ int pc_sh[3];
    if (warp == 0) {
      int sq, pi, np;
      piece_of_row(p, (int)blockIdx.x - (transfer ? p.piece_rows : 0), lane, &sq, &pi, &np);
      if (lane == 0) {
        pc_sh[0] = sq;
        pc_sh[1] = pi;
        pc_sh[2] = np;
      }
    }
    __syncthreads();
    seq = pc_sh[0];
    pc_i = pc_sh[1];
    pc_n = pc_sh[2];
    if (seq < 0 || (pass1 && pc_i == pc_n - 1)) return;  // past the last piece; a last piece has no pass 1
  }
  int64_t bos, L;
  if (!seq_bounds(p.cu, p.cu64, p.T, seq, &bos, &L)) return;  // flagged by the descriptor kernel
  const int d = p.K, V = p.V, M = p.M, QP = p.qpad, H = p.H;
  const int q4 = warp & 3;
  const int v = q4 * 32 + lane;  // state row (TMEM lane) of prep and store threads
  const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
  const ImageLayout il(d, QP);
  const uint32_t sbytes = stage_bytes(d, QP);
  const int nst = num_stages(d, QP);

  extern __shared__ __align__(1024) unsigned char scan_smem_raw[];
  // the 1024-aligned base as an offset into the shared array, so that accesses stay in the shared
  // address space
  unsigned char *sm = scan_smem_raw + ((1024u - (sm100::smem_u32(scan_smem_raw) & 1023u)) & 1023u);
  unsigned char *obuf = sm + nst * sbytes;  // [qpad][V] 16-bit output staging
  unsigned char *sttiles = obuf + obuf_bytes(QP, V) + (uint32_t)q4 * 2u * kStTile;  // this store warp's boxes
  __shared__ __align__(8) uint64_t full1[2], full2[2], yo_ready[2], yo_free[2], b1_done[2], b2_done[2], mid_done,
      bk_free, fin_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ ChunkInfo info[2];
  __shared__ int st_ok[4];
  __shared__ volatile int abort_flag;
  // every wait of this launch gives up after wl (about a second unless a test shortened it)
  const uint64_t wl = p.wait_limit_ns;

  // incoming state source
  int slot = -1;
  const float *src = nullptr;
  [[maybe_unused]] const __nv_bfloat16 *src16 = nullptr;  // a bf16 dense initial state (INIT16)
  if (!in_range(p.bounds, p.status, GDP_BOUNDS_SITE_SCAN_STATE, seq, p.N)) return;
  if (p.cache) {
    slot = p.slots[seq];
    if (slot < -1 || slot >= p.num_slots) {
      if (tid == 0 && p.seg_lo == 0 && !pass1 && !xfer && pc_i == 0) set_status(p.status, GDP_DEV_ERR_SLOT);
      slot = -1;
    }
    if (slot >= 0) src = p.cache + ((int64_t)slot * H + h) * (int64_t)V * d;
  } else if (p.init) {
    if constexpr (INIT16)
      src16 = static_cast<const __nv_bfloat16 *>(p.init) + ((int64_t)seq * H + h) * (int64_t)V * d;
    else
      src = static_cast<const float *>(p.init) + ((int64_t)seq * H + h) * (int64_t)V * d;
  }
  if (pass1 || xfer || pc_n > 1) {  // zero (or the identity) for B / Phi; a split piece from its S_in
    src = (pass1 || xfer) ? nullptr
                          : p.piece_buf + ((int64_t)(2 * p.piece_rows + (int)blockIdx.x) * H + h) * (int64_t)V * d;
    if constexpr (INIT16) src16 = nullptr;
  }

  // Descriptors, workspace tiles and a carried state come from earlier kernels of the stream:
  // read only after pdl_wait().  The first segment (the whole sequence when unsegmented) loads
  // its incoming state, which is the caller's, before waiting.
  const int64_t nchunks = (L * M + kChunk - 1) / kChunk;
  int64_t cod_i = 0, co_i = 0, nall = 0, e0 = 0, nrun = 0;
  bool last_seg = true;
  auto resolve = [&]() {
    cod_i = p.cod[seq];
    co_i = p.chunk_states ? (int64_t)p.co[seq] : 0;
    // chunks whose workspace tile exists (a flagged descriptor overflow truncates the sequence)
    nall = (cod_i < 0) ? 0 : max((int64_t)0, min(nchunks, p.ws_rows - cod_i));
    // this launch's chunks: global chunk e0 + e for local e in [0, nrun)
    if (pieces) {
      e0 = min((int64_t)pc_i * p.piece_len, nall);
      nrun = max((int64_t)0, min(e0 + p.piece_len, nall) - e0);
      last_seg = pc_i == pc_n - 1;
      return;
    }
    e0 = min(p.seg_lo, nall);
    nrun = max((int64_t)0, min(p.seg_hi, nall) - e0);
    last_seg = e0 + nrun == nall;
    if (e0 > 0) {  // carried from the last segment (fp32)
      src = p.seg_state + ((int64_t)seq * H + h) * (int64_t)V * d;
      if constexpr (INIT16) src16 = nullptr;
    }
  };
  if (p.seg_lo > 0) {
    pdl_wait();
    resolve();
    if (nrun == 0) return;  // the sequence has no chunk in this segment
  }
  // token-chunk starts whose state is requested (a prefix of the chunks e % M == 0; every
  // chunk when cs_div is 1, the backward pass's recompute)
  const int csd = p.cs_div;
  auto emits = [&](int64_t e) {  // chunk indices fit 32 bits (the host checks T * M)
    const int eg = (int)(e0 + e);
    return p.chunk_states && (eg % csd == 0) && co_i >= 0 && co_i + eg / csd < p.nt_pad;
  };

  if (warp == 8) tmem_alloc(&tmem_slot, 512);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full1[i], 1);
      mbar_init(&full2[i], 1);
      mbar_init(&yo_ready[i], 128);
      mbar_init(&yo_free[i], 128);
      mbar_init(&b1_done[i], 1);
      mbar_init(&b2_done[i], 1);
    }
    mbar_init(&mid_done, 128);
    mbar_init(&bk_free, 128);
    mbar_init(&fin_bar, 1);
    mbar_init_fence();
    abort_flag = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // TMEM columns: [0, d) S_hat | buffer b at 128 + b (qpad + 64): [o_hat: qpad][Y: 64] |
  // [384, 384 + d) state snapshot.  [o_hat | Y] is contiguous so that one MMA per K step
  // serves both products of batch 1.
  const uint32_t tb = tmem_slot;
  const uint32_t tS = tb, tBk = tb + 384;
  auto tO = [&](int b) { return tb + 128u + (uint32_t)b * (uint32_t)(QP + 64); };
  const uint32_t id1 = idesc(kFmtTF32, 0, 0, QP + 64, 128);  // [o_hat | Y] += S_hat [Qh ; -W]^T
  const uint32_t id1y = idesc(kFmtTF32, 0, 0, 64, 128);      // Y += S_hat (-W)^T (no outputs)
  const uint32_t id2s = idesc(kFmtTF32, 0, 0, d, 128);       // S_hat += Y Ktil
  const uint32_t id2o = idesc(kFmtTF32, 0, 0, QP, 128);      // o_hat += Y P^T

  auto image = [&](int64_t e) { return p.img + (size_t)((cod_i + e0 + e) * H + h) * p.img_stride; };
  // producer thread: part 1 / part 2 of chunk e's image into stage e % nst (n1, n2: copies issued)
  int n1[2] = {0, 0}, n2[2] = {0, 0};
  // (a workspace row that fails its debug range check is not copied: the stage completes empty)
  auto load_part1 = [&](int64_t e) {
    const int st = (int)(e % nst);
    if (in_range(p.bounds, p.status, GDP_BOUNDS_SITE_SCAN_TILE, cod_i + e0 + e, p.ws_rows)) {
      mbar_arrive_expect_tx(&full1[st], il.part1);
      bulk_g2s(sm + st * sbytes, image(e), il.part1, &full1[st]);
    } else {
      mbar_arrive(&full1[st]);
    }
    ++n1[st];
  };
  auto load_part2 = [&](int64_t e) {
    const int st = (int)(e % nst);
    if (in_range(p.bounds, p.status, GDP_BOUNDS_SITE_SCAN_TILE, cod_i + e0 + e, p.ws_rows)) {
      mbar_arrive_expect_tx(&full2[st], il.part2);
      bulk_g2s(sm + st * sbytes + il.b2, image(e) + il.b2, il.part2, &full2[st]);
    } else {
      mbar_arrive(&full2[st]);
    }
    ++n2[st];
  };

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
      if (transfer)  // the identity (V == K)
#pragma unroll
        for (int u = 0; u < 16; ++u) x[u] = (c0 + u == v) ? 1.f : 0.f;
      if constexpr (INIT16) {
        if (src16 && v < V) {  // eight bf16 per 16-byte load
#pragma unroll
          for (int u8 = 0; u8 < 16; u8 += 8) {
            const uint4 y = *reinterpret_cast<const uint4 *>(src16 + (int64_t)v * d + c0 + u8);
            const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&y);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f2 = __bfloat1622float2(b[i]);
              x[u8 + 2 * i] = f2.x;
              x[u8 + 2 * i + 1] = f2.y;
            }
          }
        }
      }
      tmem_st16(tS + lrow + c0, x);
    }
    tmem_st_wait();
  }
  if (p.seg_lo == 0) {
    pdl_wait();
    resolve();
  }
  if (warp == 9 && lane == 0)
    for (int64_t e = 0; e < nst && e < nrun; ++e) {
      // (a test of the bounded waits withholds the first copy of CTA (0, 0): its wait runs out)
      if (!(p.test_withhold_copy && e == 0 && blockIdx.x == 0 && blockIdx.y == 0)) load_part1(e);
      load_part2(e);
    }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < 4) {
    // ---------------- prep warps ----------------
    float u[64];
    auto load_u = [&](int64_t e) {  // row v of U^T: one 512-byte segment per load instruction of the warp
      const float4 *Ut = reinterpret_cast<const float4 *>(p.U + ((cod_i + e0 + e) * H + h) * (int64_t)V * kChunk) +
                         (v < V ? q4 * 512 + lane : 0);
      const bool urow = v < V && !transfer &&
                        in_range(p.bounds, p.status, GDP_BOUNDS_SITE_SCAN_TILE, cod_i + e0 + e, p.ws_rows);
#pragma unroll
      for (int s4 = 0; s4 < 16; ++s4) {
        const float4 x = urow ? Ut[s4 * 32] : make_float4(0.f, 0.f, 0.f, 0.f);
        u[4 * s4] = x.x; u[4 * s4 + 1] = x.y; u[4 * s4 + 2] = x.z; u[4 * s4 + 3] = x.w;
      }
    };
    float gam = 1.f;  // Gamma of the state in TMEM
    int n_emit = 0;
    auto meta_at = [&](int64_t e) { return *reinterpret_cast<const ImageMeta *>(image(e) + il.meta); };
    ImageMeta mt_next{};
    if (nrun > 0) {
      load_u(0);
      mt_next = meta_at(0);
    }
    for (int64_t e = 0; e < nrun; ++e) {
      const int b = (int)(e & 1);
      const ImageMeta mt = mt_next;  // read from the image in global memory a chunk ahead
      const bool fast = mt.fast != 0, emit = emits(e);
      const bool renorm = fast ? (gam * mt.gamma_last < kRenormMinGamma) : (gam != 1.f);
      const float gam_pass = renorm ? 1.f : gam;                  // Gamma during the chunk's products
      const float gam_next = fast ? gam_pass * mt.gamma_last : 1.f;  // Gamma' after it
      if (e >= 2 && !mbar_wait_or_abort(&yo_free[b], (uint32_t)(((e >> 1) - 1) & 1), &abort_flag, wl)) break;
      tc_fence_after();
      const uint32_t to = tO(b), ty = to + (uint32_t)QP;
      const float inv = 1.f / gam_next;
#pragma unroll
      for (int w = 0; w < 64; ++w) u[w] *= inv;  // u is reloaded for the next chunk below
      tmem_st32x(ty + lrow, u);
      tmem_st32x(ty + lrow + 32, u + 32);
      if (p.out) {  // without outputs the MMAs leave o_hat alone
        float z[16];
#pragma unroll
        for (int w = 0; w < 16; ++w) z[w] = 0.f;
        for (int c0 = 0; c0 < QP; c0 += 16) tmem_st16(to + lrow + c0, z);
      }
      if (tid == 0) info[b] = ChunkInfo{gam_next, mt.nq, mt.p0};
      if (renorm && e >= 1) {  // the renormalisation rewrites the final S_hat of chunk e
        if (!mbar_wait_or_abort(&b2_done[(e - 1) & 1], (uint32_t)(((e - 1) >> 1) & 1), &abort_flag, wl)) break;
        tc_fence_after();
      }
      if (renorm) {
        for (int c0 = 0; c0 < d; c0 += 32) {
          float x[32];
          tmem_ld32(tS + lrow + c0, x);
#pragma unroll
          for (int w = 0; w < 32; ++w) x[w] *= gam;
          tmem_st16(tS + lrow + c0, x);
          tmem_st16(tS + lrow + c0 + 16, x + 16);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&yo_ready[b]);
      if (e + 1 < nrun) {  // next chunk's U^T and meta, in flight while this chunk runs
        load_u(e + 1);
        mt_next = meta_at(e + 1);
      }
      if (emit || !fast) {
        // between the two batches: snapshot S_e = gam_pass S_hat (read alongside batch 1) and,
        // for a slow image, S_hat <- gamma_last S_hat once batch 1 has read it
        if (emit && n_emit >= 1 && !mbar_wait_or_abort(&bk_free, (uint32_t)((n_emit - 1) & 1), &abort_flag, wl)) break;
        if (!fast) {  // batch 1 has read S_hat (so chunk e - 1's batch 2 is complete too)
          if (!mbar_wait_or_abort(&b1_done[b], (uint32_t)((e >> 1) & 1), &abort_flag, wl)) break;
        } else if (!renorm && e >= 1) {  // S_hat of chunk e is final; waited for only now, so that
          // batch 1 (issued on yo_ready above) is not held back by this round trip
          if (!mbar_wait_or_abort(&b2_done[(e - 1) & 1], (uint32_t)(((e - 1) >> 1) & 1), &abort_flag, wl)) break;
        }
        tc_fence_after();
        // (a slow chunk was renormalised, so gam_pass is 1 there and one array serves both)
        for (int c0 = 0; c0 < d; c0 += 32) {
          float x[32];
          tmem_ld32x(tS + lrow + c0, x);
          if (emit) {
#pragma unroll
            for (int w = 0; w < 32; ++w) x[w] *= gam_pass;
            tmem_st32x(tBk + lrow + c0, x);
          }
          if (!fast) {
#pragma unroll
            for (int w = 0; w < 32; ++w) x[w] *= mt.gamma_last;
            tmem_st32x(tS + lrow + c0, x);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&mid_done);
        if (emit) ++n_emit;
      }
      gam = gam_next;
    }
    tmem_st_wait();  // (an aborted chunk may leave stores in flight; the columns are freed below)
  } else if (warp < 8) {
    // ---------------- store warps ----------------
    float gam_fin = 1.f;
    int nblk = 0;
    const bool has_rows = q4 * 32 < V;
    for (int64_t e = 0; e < nrun; ++e) {
      const int b = (int)(e & 1);
      // the four store warps take the same exit decision (they meet at named barriers)
      const bool ok = mbar_wait_or_abort(&b2_done[b], (uint32_t)((e >> 1) & 1), &abort_flag, wl);
      if (lane == 0) st_ok[q4] = ok ? 1 : 0;
      if (tid == 128) bulk_wait_read<0>();  // the output staging's TMA store (if any) has read it
      named_sync(1, 128);  // also: every thread has finished reading the previous chunk's staging
      if (!(st_ok[0] & st_ok[1] & st_ok[2] & st_ok[3])) break;
      tc_fence_after();
      const ChunkInfo ci = info[b];
      gam_fin = ci.out_scale;
      // outputs: the chunk's o_hat columns (read under one wait), 16-bit staging [q][v]
#pragma unroll 1
      for (int q0 = 0; p.out && q0 < ci.nq; q0 += 32) {  // 32 readout rows per wait
        uint32_t xo[32];
        tmem_ld16_nw(tO(b) + lrow + q0, xo);
        if (q0 + 16 < ci.nq) tmem_ld16_nw(tO(b) + lrow + q0 + 16, xo + 16);
        tmem_ld_wait();
        if (v < V) {
#pragma unroll
          for (int w = 0; w < 32; ++w)
            if (q0 + w < ci.nq) {
              const float o = __uint_as_float(xo[w]) * ci.out_scale;
              if constexpr (F16)
                *reinterpret_cast<__half *>(obuf + ((uint32_t)(q0 + w) * V + v) * 2u) = __float2half_rn(o);
              else
                *reinterpret_cast<__nv_bfloat16 *>(obuf + ((uint32_t)(q0 + w) * V + v) * 2u) =
                    __float2bfloat16_rn(o);
            }
        }
      }
      fence_async_smem();  // the staging may leave by a TMA store
      tc_fence_before();
      mbar_arrive(&yo_free[b]);  // the chunk's o_hat columns have been read
      named_sync(1, 128);
      const int64_t tq0 = (bos * M + (e0 + e) * kChunk + ci.p0) / M;  // readout rows are consecutive tokens
      if (p.out && p.out_tma && (ci.nq == kChunk / M || ci.nq == (kChunk + M - 1) / M)) {
        // one box of exactly nq token rows (x = 0, head h, token tq0)
        if (tid == 128 && in_range(p.bounds, p.status, GDP_BOUNDS_SITE_SCAN_OUT, tq0 + ci.nq - 1, p.T - p.bounds_shrink)) {
          tma_store_3d(ci.nq == kChunk / M ? &tm_out_a : &tm_out_b, obuf, 0, h, (int)tq0);
          bulk_commit();
        }
      } else {
        const int cpr = V / 8;  // 16-byte chunks per output row
        for (int c = tid - 128; p.out && c < ci.nq * cpr; c += 128) {
          const int qi = c / cpr, ch = c % cpr;
          if (in_range(p.bounds, p.status, GDP_BOUNDS_SITE_SCAN_OUT, tq0 + qi, p.T - p.bounds_shrink))
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + ((tq0 + qi) * H + h) * (int64_t)V + ch * 8) =
                *reinterpret_cast<const uint4 *>(obuf + ((uint32_t)qi * V + ch * 8) * 2u);
        }
      }
      if (emits(e)) {  // the prep warps copied S_e before batch 2 of this chunk was issued
        if (has_rows) {  // bk_free: the snapshot columns have been read
          store_state_tma(tBk + lrow, sttiles, lane, d, 1.f, &tm_cs,
                          (int)(((co_i + (e0 + e) / csd) * H + h) * V + q4 * 32), nblk, &bk_free);
        } else {
          tc_fence_before();
          mbar_arrive(&bk_free);
        }
      }
    }
    if (!abort_flag && has_rows) {  // the last chunk's b2_done was waited for above
      int64_t r = -1;
      const CUtensorMap *tm = &tm_fin;
      if (pass1 || xfer) {  // B or Phi of the piece / sequence (piece_buf or xfer_out: the segment map)
        r = ((int64_t)blockIdx.x * H + h) * V;
        tm = &tm_seg;
      } else if (!last_seg) {  // carried to the next segment (a split piece leaves nothing)
        if (!pieces) r = ((int64_t)seq * H + h) * V;
        tm = &tm_seg;
      } else if (p.cache) {
        if (slot >= 0) r = ((int64_t)slot * H + h) * V;
      } else if (p.out_state) {
        r = ((int64_t)seq * H + h) * V;
      }
      if (r >= 0) store_state_tma(tS + lrow, sttiles, lane, d, gam_fin, tm, (int)(r + q4 * 32), nblk, nullptr);
    }
    if (lane == 0) bulk_wait_all();  // this warp's tensor stores are complete
  } else if (warp == 8) {
    if (lane == 0) {
      // ---------------- control thread: MMA issue ----------------
      int n_mid = 0;
      for (int64_t e = 0; e < nrun; ++e) {
        const int st = (int)(e % nst), b = (int)(e & 1);
        unsigned char *stage = sm + st * sbytes;
        if (!mbar_wait_or_abort(&full1[st], (uint32_t)((e / nst) & 1), &abort_flag, wl)) break;
        if (!mbar_wait_or_abort(&yo_ready[b], (uint32_t)((e >> 1) & 1), &abort_flag, wl)) break;
        tc_fence_after();
        const ImageMeta mt = *reinterpret_cast<const ImageMeta *>(stage + il.meta);
        const bool mid = emits(e) || mt.fast == 0;
        const uint32_t to = tO(b), ty = to + (uint32_t)QP;
        const uint32_t sb1 = smem_u32(stage) + il.b1, sb2 = smem_u32(stage) + il.b2;
        if (p.out) {
          for (int kk = 0; kk < d / 8; ++kk)
            mma_tf32_ts(to, tS + kk * 8, desc_sw128(sb1 + (kk >> 2) * il.b1_block + (kk & 3) * 32u, 16, 1024), id1,
                        1);
        } else {  // the -W rows only: they start qpad rows (whole 1024-byte atoms) into each K-block
          for (int kk = 0; kk < d / 8; ++kk)
            mma_tf32_ts(ty, tS + kk * 8,
                        desc_sw128(sb1 + (kk >> 2) * il.b1_block + (uint32_t)QP * 128u + (kk & 3) * 32u, 16, 1024),
                        id1y, 1);
        }
        mma_commit(&b1_done[b]);
        if (!mbar_wait_or_abort(&full2[st], (uint32_t)((e / nst) & 1), &abort_flag, wl)) break;
        if (mid) {
          if (!mbar_wait_or_abort(&mid_done, (uint32_t)(n_mid & 1), &abort_flag, wl)) break;
          ++n_mid;
          tc_fence_after();
        }
        // two MMAs per K step (N = d and N = qpad): past N = 128 an MMA costs far more than
        // two narrower ones (measured)
        for (int kk = 0; kk < kChunk / 8; ++kk) {
          const uint32_t bk = sb2 + (kk >> 2) * il.b2_block + (kk & 3) * 32u;
          mma_tf32_ts(tS, ty + kk * 8, desc_sw128(bk, 16, 1024), id2s, 1);
          if (p.out) mma_tf32_ts(to, ty + kk * 8, desc_sw128(bk + (uint32_t)d * 128u, 16, 1024), id2o, 1);
        }
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
    // ---------------- producer thread: image copies ----------------
    // (no L2 prefetch ahead of the copies: with the WY kernel writing the next segment's images
    // beside the scan, prefetching 2 / 4 / 8 / 16 chunks ahead measured 0 / 3 / 5 / 8 % slower on
    // the 65536-token sequence than none: the prefetched lines are evicted before their copy)
    for (int64_t e = 0; e + nst < nrun; ++e) {
      const int b = (int)(e & 1);
      if (!mbar_wait_or_abort(&b1_done[b], (uint32_t)((e >> 1) & 1), &abort_flag, wl)) break;
      load_part1(e + nst);
      if (!mbar_wait_or_abort(&b2_done[b], (uint32_t)((e >> 1) & 1), &abort_flag, wl)) break;
      load_part2(e + nst);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (abort_flag && warp == 9 && lane == 0)
    for (int st = 0; st < nst; ++st) {  // bounded; the last copy issued on each barrier has landed
      if (n1[st] > 0) mbar_wait(&full1[st], (uint32_t)((n1[st] - 1) & 1));
      if (n2[st] > 0) mbar_wait(&full2[st], (uint32_t)((n2[st] - 1) & 1));
    }
  __syncthreads();
  if (warp == 8) tmem_free(tb, 512);
}

// Shared by the scan kernels of every type pair (one translation unit each, so that the
// common kernel's code is laid out exactly as when it is alone): tensor maps, dynamic shared
// memory, grid (sequence, head), one CTA per SM.
template <typename Kern>
cudaError_t launch_scan_kernel(Kern kern, const Problem &p, cudaStream_t stream) {
  const size_t smem = scan_smem_bytes(p.K, p.qpad, p.V);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap tm_cs, tm_fin, tm_seg;
  const int64_t hv = (int64_t)p.H * p.V;
  if ((e = tmap_state(&tm_cs, p.chunk_states, p.nt_pad * hv, p.K)) != cudaSuccess) return e;
  if (p.cache)
    e = tmap_state(&tm_fin, p.cache, p.num_slots * hv, p.K);
  else
    e = tmap_state(&tm_fin, p.out_state, p.N * hv, p.K);
  if (e != cudaSuccess) return e;
  if (p.piece_len > 0)  // the piece states (pass 1 writes B and Phi through it)
    e = tmap_state(&tm_seg, p.piece_buf, 3 * (int64_t)p.piece_rows * hv, p.K);
  else if (p.xfer)  // the transfer pairs
    e = tmap_state(&tm_seg, p.xfer_out, 2 * p.N * hv, p.K);
  else
    e = tmap_state(&tm_seg, p.seg_state, p.N * hv, p.K);
  if (e != cudaSuccess) return e;
  // output boxes of 64 / M and ceil(64 / M) token rows: the readout counts of a full chunk
  alignas(64) CUtensorMap tm_out_a, tm_out_b;
  Problem q = p;
  const int na = kChunk / p.M, nb = (kChunk + p.M - 1) / p.M;
  q.out_tma = (p.out && p.T >= nb) ? 1 : 0;
  if ((e = tmap_out_rows(&tm_out_a, q.out_tma ? p.out : nullptr, p.T, p.H, p.V, na, p.f16)) != cudaSuccess) return e;
  if ((e = tmap_out_rows(&tm_out_b, q.out_tma ? p.out : nullptr, p.T, p.H, p.V, nb, p.f16)) != cudaSuccess) return e;
  // one CTA per (sequence, head), or per (piece row, head) -- pass 1 runs two per piece
  const int64_t rows = p.piece_len > 0 ? (p.piece_pass1 ? 2 : 1) * (int64_t)p.piece_rows : (p.xfer ? 2 : 1) * p.N;
  dim3 grid((unsigned)rows, (unsigned)p.H);
  if ((e = launch_kernel(kern, grid, dim3(kScanThreads), smem, stream, p.pdl != 0, q, tm_cs, tm_fin, tm_seg, tm_out_a,
                         tm_out_b)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

#define GDP_SCAN_KERNEL(name, f16, init16)                                                                       \
  __global__ void __launch_bounds__(kScanThreads, 1)                                                            \
      name(Problem p, const __grid_constant__ CUtensorMap tm_cs, const __grid_constant__ CUtensorMap tm_fin,     \
           const __grid_constant__ CUtensorMap tm_seg, const __grid_constant__ CUtensorMap tm_out_a,              \
           const __grid_constant__ CUtensorMap tm_out_b) {                                                        \
    scan_body<f16, init16>(p, tm_cs, tm_fin, tm_seg, tm_out_a, tm_out_b);                                       \
  }

}  // namespace
}  // namespace gdp
