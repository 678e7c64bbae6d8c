// gdp_pieces.cu -- split chains: the entering state of every piece of a split sequence.
//
// Over its expanded chunks a sequence's state follows the affine recurrence
// S_{e+1} = S_e A_e + B_e (V-major state, right multiplication by K x K maps; the
// decay, the delta-rule updates and the readouts of Megatron-Core API page
// "core.ssm.ops.gdp.chunk", stages 3 and 4).  Cut into pieces of piece_len chunks, piece j
// maps its entering state to S_in(j) Phi_j + B_j, where B_j is the piece run from a zero
// state and Phi_j the piece run from the identity with V = 0 -- the scan kernel's first
// pass computes both for every piece but a sequence's last, all pieces at once.  This
// kernel chains them,
//   S_in(0) = the sequence's initial state,   S_in(j + 1) = S_in(j) Phi_j + B_j,
// in fp32 FMA, and stores every S_in for the scan's second
// pass, which then runs all pieces at once from their own entering states.  Rows of the state
// are independent: one CTA per (sequence, head, 16 state rows), one CTA per SM, so a
// (sequence, head) spreads over V / 16 SMs.  Phi_{j+2} and B_{j+2} arrive by TMA while step j
// computes.
#include <cuda.h>  // CUtensorMap

#include "gdp_internal.cuh"
#include "gdp_sm100.cuh"

namespace gdp {
namespace {

constexpr int kCmbThreads = 512;    // 16 warps: k splits x 4 row groups x D / 4 column groups
constexpr int kCmbRows = 16;        // state rows per CTA
constexpr int kCmbStStride = 20;    // floats per k row of the transposed rows (16 + 4 pad)
constexpr size_t kCmbMinSmem = 116u * 1024u;  // at most one CTA per SM: the steps are serial, an SM each

__host__ __device__ constexpr int cmb_splits(int d) { return kCmbThreads / d; }  // k splits
// Shared memory: Phi_j in two stages as 32 x 32 boxes of the state map (128-byte swizzle: row r
// of a box at r * 128 bytes, its 16-byte chunk q at position q ^ (r % 8)); B_j (this CTA's 16
// rows) in two stages; S_j transposed, [D][kCmbStStride], in two buffers; the partial products
// of the k splits after the first, [KS - 1][16][D].
__host__ __device__ constexpr uint32_t cmb_phi_bytes(int d) { return (uint32_t)d * d * 4u; }
__host__ __device__ constexpr uint32_t cmb_b_bytes(int d) { return (uint32_t)kCmbRows * d * 4u; }
__host__ __device__ constexpr uint32_t cmb_st_floats(int d) { return (uint32_t)d * kCmbStStride; }
__host__ inline size_t cmb_smem(int d) {
  const size_t need = 2 * (size_t)cmb_phi_bytes(d) + 2 * (size_t)cmb_b_bytes(d) + 2 * 4 * (size_t)cmb_st_floats(d) +
                      4 * (size_t)(cmb_splits(d) - 1) * kCmbRows * d + 1024;
  return need > kCmbMinSmem ? need : kCmbMinSmem;
}

// One chain of steps for a CTA's 16 state rows: S_{j+1} = S_j Phi_j + B_j for j < steps.
// Pointers are already offset to the CTA's rows.
struct ChainRows {
  int steps;
  int64_t phi_row0, phi_row_step;  // first row of Phi_j in the tensor map: phi_row0 + j phi_row_step
  const float *b0;                 // B_j's rows: b0 + j b_step
  int64_t b_step;
  float *s0;                       // S_j's rows (j = 0 .. steps): s0 + j s_step
  int64_t s_step;
  const float *src;                // S_0's rows, fp32, or
  const __nv_bfloat16 *src16;      // bf16; both NULL: zero
};

// The steps in fp32 FMA.  Thread (ks, rg, cg) sums k split ks (D / KS values of k) for rows
// 4 rg .. 4 rg + 3 and columns 4 cg .. 4 cg + 3; split 0 adds the other splits' partial products
// and B_j and owns S_{j+1}.  Thread 0 brings Phi_j (tensor boxes) and B_j (one bulk copy) in two
// steps ahead.  Measured on this part: warp-level tf32 MMAs in the 3xTF32 split took ~1.7 us per
// step (the legacy MMA path runs at about the FFMA rate, and the split needs three products);
// sharing Phi_j among a (sequence, head)'s row blocks by cluster multicast was slower (clusters
// of 8 whole-SM CTAs start late).  Called by all threads once the mbarriers are initialised.
template <int D, bool INIT16>
__device__ __forceinline__ void run_chain(const ChainRows &c, const CUtensorMap *tm_phi, unsigned char *sm,
                                          uint64_t *full, uint32_t *status) {
  constexpr int NB = D / 32, CG = D / 4, KS = cmb_splits(D), KL = D / KS;
  constexpr uint32_t PB = cmb_phi_bytes(D), BB = cmb_b_bytes(D), STF = cmb_st_floats(D);
  static_assert(KS * D == kCmbThreads && KL * KS == D, "thread layout");
  float *bst = reinterpret_cast<float *>(sm + 2 * PB);  // B_j stages, [2][16][D]
  float *sts = bst + 2 * BB / 4;                         // S_j^T buffers, [2][D][kCmbStStride]
  float *part = sts + 2 * STF;                           // [KS - 1][16][D]
  const int tid = threadIdx.x;
  const int ks = tid / D, tt = tid % D, rg = tt / CG, cg = tt % CG;
  int issued[2] = {0, 0};
  auto issue = [&](int j) {  // Phi_j and B_j into stage j % 2 (thread 0)
    const int sg = j & 1;
    unsigned char *dst = sm + sg * PB;
    sm100::mbar_arrive_expect_tx(&full[sg], PB + BB);
    const int y0 = (int)(c.phi_row0 + (int64_t)j * c.phi_row_step);
#pragma unroll
    for (int kb = 0; kb < NB; ++kb)
#pragma unroll
      for (int cb = 0; cb < NB; ++cb)
        sm100::tma_load_2d(dst + (kb * NB + cb) * 4096, tm_phi, 32 * cb, y0 + 32 * kb, &full[sg]);
    sm100::bulk_g2s(bst + sg * (BB / 4), c.b0 + (int64_t)j * c.b_step, BB, &full[sg]);
    ++issued[sg];
  };
  if (tid == 0)
    for (int j = 0; j < 2 && j < c.steps; ++j) issue(j);

  for (int idx = tid; idx < kCmbRows * D / 2; idx += kCmbThreads) {  // S_0 -> global, S^T buffer 0
    const int row = idx / (D / 2), col = 2 * (idx % (D / 2));
    const int64_t off = (int64_t)row * D + col;
    float2 x = make_float2(0.f, 0.f);
    if (c.src) x = *reinterpret_cast<const float2 *>(c.src + off);
    if constexpr (INIT16) {
      if (c.src16) x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(c.src16 + off));
    }
    *reinterpret_cast<float2 *>(c.s0 + off) = x;
    sts[col * kCmbStStride + row] = x.x;
    sts[(col + 1) * kCmbStStride + row] = x.y;
  }
  // Phi element (k, 4 cg .. 4 cg + 3), one 16-byte chunk: box (k / 32, col / 32), row k % 32,
  // chunk position ((col % 32) / 4) ^ (k % 8); the part that depends on the thread only
  const uint32_t cbase = (uint32_t)(cg >> 3) * 1024u;  // floats
  const uint32_t cq = (uint32_t)(cg & 7);
  bool ok = true;
#pragma unroll 1
  for (int j = 0; j < c.steps; ++j) {
    const int sg = j & 1;
    // also publishes S_j^T and frees the partial products of the step before
    ok = __syncthreads_and(sm100::mbar_wait(&full[sg], (uint32_t)((j >> 1) & 1)));
    if (!ok) break;
    const float *phi = reinterpret_cast<const float *>(sm + sg * PB);
    const float *st = sts + (j & 1) * STF;
    float acc[4][4];
    if (ks == 0) {  // B_j now: the stage is refilled once everyone has passed the barrier below
      const float *bj = bst + sg * (BB / 4);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 bv = *reinterpret_cast<const float4 *>(bj + (4 * rg + i) * D + 4 * cg);
        acc[i][0] = bv.x; acc[i][1] = bv.y; acc[i][2] = bv.z; acc[i][3] = bv.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    }
#pragma unroll 8
    for (int k = ks * KL; k < ks * KL + KL; ++k) {
      const float4 sv = *reinterpret_cast<const float4 *>(st + k * kCmbStStride + 4 * rg);
      const float4 pv = *reinterpret_cast<const float4 *>(
          phi + (uint32_t)(k >> 5) * (uint32_t)NB * 1024u + cbase + (uint32_t)(k & 31) * 32u + ((cq ^ (uint32_t)(k & 7)) << 2));
      const float sa[4] = {sv.x, sv.y, sv.z, sv.w}, pa[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(sa[i], pa[q], acc[i][q]);
    }
    if (ks > 0)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4 *>(part + ((ks - 1) * kCmbRows + 4 * rg + i) * D + 4 * cg) =
            make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    __syncthreads();  // stage sg (Phi_j, B_j) and S_j^T are read; the partial products are in place
    if (tid == 0 && j + 2 < c.steps) issue(j + 2);
    if (ks == 0) {
      float *nst = sts + ((j + 1) & 1) * STF;
      float *dst = c.s0 + (int64_t)(j + 1) * c.s_step;
#pragma unroll
      for (int x = 0; x < KS - 1; ++x)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 y = *reinterpret_cast<const float4 *>(part + (x * kCmbRows + 4 * rg + i) * D + 4 * cg);
          acc[i][0] += y.x; acc[i][1] += y.y; acc[i][2] += y.z; acc[i][3] += y.w;
        }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4 *>(dst + (int64_t)(4 * rg + i) * D + 4 * cg) =
            make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<float4 *>(nst + (4 * cg + q) * kCmbStStride + 4 * rg) =
            make_float4(acc[0][q], acc[1][q], acc[2][q], acc[3][q]);
    }
  }
  if (!ok && tid == 0) {
    set_status(status, GDP_DEV_ERR_TIMEOUT);
    for (int sg = 0; sg < 2; ++sg)  // bounded: the last copies issued on each stage have landed
      if (issued[sg] > 0) sm100::mbar_wait(&full[sg], (uint32_t)((issued[sg] - 1) & 1));
  }
}

__device__ __forceinline__ unsigned char *cmb_smem_base() {
  extern __shared__ __align__(1024) unsigned char cmb_smem_raw[];
  // the 1024-aligned base as an offset into the shared array (accesses stay in the shared address space)
  return cmb_smem_raw + ((1024u - (sm100::smem_u32(cmb_smem_raw) & 1023u)) & 1023u);
}

// Split chains: the pieces of sequence blockIdx.x, head blockIdx.y, state rows 16 blockIdx.z ..:
// S_in(0) is the caller's state (cache slot, dense fp32 / bf16, or zero), S_in(j) goes to
// piece_buf row 2 piece_rows + first + j, Phi_j / B_j come from rows piece_rows + first + j / first + j.
template <int D, bool INIT16>
__global__ void __launch_bounds__(kCmbThreads, 1) gdp_piece_combine_kernel(Problem p,
                                                                        const __grid_constant__ CUtensorMap tm_phi) {
  __shared__ __align__(8) uint64_t full[2];
  __shared__ int sh[2];
  const int seq = blockIdx.x, h = blockIdx.y, r0 = kCmbRows * (int)blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // B and Phi come from the grid before; wait before any exit so that this grid's
  // completion implies its predecessors'
  sm100::pdl_wait();
  sm100::pdl_trigger();
  if (warp == 0) {
    int first, np;
    pieces_of_seq(p, seq, lane, &first, &np);
    if (lane == 0) {
      sh[0] = first;
      sh[1] = np;
    }
  }
  if (tid == 0) {
    sm100::mbar_init(&full[0], 1);
    sm100::mbar_init(&full[1], 1);
    sm100::mbar_init_fence();
  }
  __syncthreads();
  const int first = sh[0], np = sh[1];
  if (np <= 1) return;  // one piece: the scan reads the caller's state itself
  const int64_t KV = (int64_t)D * D, R = p.piece_rows, step = (int64_t)p.H * KV;
  auto rows_of = [&](int64_t prow) { return p.piece_buf + (prow * p.H + h) * KV + (int64_t)r0 * D; };
  ChainRows c{};
  c.steps = np - 1;
  c.phi_row0 = ((R + first) * p.H + h) * D;
  c.phi_row_step = (int64_t)p.H * D;
  c.b0 = rows_of(first);
  c.b_step = step;
  c.s0 = rows_of(2 * R + first);
  c.s_step = step;
  if (p.cache) {  // an out-of-range slot reads as no state (the scan reports it)
    const int slot = p.slots[seq];
    if (slot >= 0 && slot < p.num_slots) c.src = p.cache + ((int64_t)slot * p.H + h) * KV + (int64_t)r0 * D;
  } else if (p.init) {
    if constexpr (INIT16)
      c.src16 = static_cast<const __nv_bfloat16 *>(p.init) + ((int64_t)seq * p.H + h) * KV + (int64_t)r0 * D;
    else
      c.src = static_cast<const float *>(p.init) + ((int64_t)seq * p.H + h) * KV + (int64_t)r0 * D;
  }
  run_chain<D, INIT16>(c, &tm_phi, cmb_smem_base(), full, p.status);
}

// The general chain (gdp_chain_states): sequence blockIdx.x, head blockIdx.y, rows 16 blockIdx.z ..;
// Phi / B / S_out indexed [step][N][H][D][D].
struct ChainArgs {
  const float *s0, *b;
  float *s_out;
  int64_t steps, N;
  int H;
  uint32_t *status;
};
template <int D>
__global__ void __launch_bounds__(kCmbThreads, 1) gdp_chain_states_kernel(ChainArgs a,
                                                                       const __grid_constant__ CUtensorMap tm_phi) {
  __shared__ __align__(8) uint64_t full[2];
  const int seq = blockIdx.x, h = blockIdx.y, r0 = kCmbRows * (int)blockIdx.z;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&full[0], 1);
    sm100::mbar_init(&full[1], 1);
    sm100::mbar_init_fence();
  }
  __syncthreads();
  const int64_t KV = (int64_t)D * D, step = a.N * a.H * KV, base = ((int64_t)seq * a.H + h) * KV + (int64_t)r0 * D;
  ChainRows c{};
  c.steps = (int)a.steps;
  c.phi_row0 = ((int64_t)seq * a.H + h) * D;
  c.phi_row_step = a.N * a.H * D;
  c.b0 = a.b + base;
  c.b_step = step;
  c.s0 = a.s_out + base;
  c.s_step = step;
  c.src = a.s0 ? a.s0 + base : nullptr;
  run_chain<D, false>(c, &tm_phi, cmb_smem_base(), full, a.status);
}

template <int D, bool INIT16>
cudaError_t launch_combine_d(const Problem &p, cudaStream_t stream) {
  const size_t smem = cmb_smem(D);
  cudaError_t e = cudaFuncSetAttribute(gdp_piece_combine_kernel<D, INIT16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap tm_phi;  // the piece states, [3 piece_rows][H][V][K] fp32, 32 x 32 boxes
  if ((e = tmap_state(&tm_phi, p.piece_buf, 3 * (int64_t)p.piece_rows * p.H * p.V, p.K)) != cudaSuccess) return e;
  e = launch_kernel(gdp_piece_combine_kernel<D, INIT16>, dim3((unsigned)p.N, (unsigned)p.H, (unsigned)(D / kCmbRows)),
                    dim3(kCmbThreads), smem, stream, p.pdl != 0, p, tm_phi);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_chain_d(const ChainArgs &a, const float *phi, cudaStream_t stream) {
  const size_t smem = cmb_smem(D);
  cudaError_t e = cudaFuncSetAttribute(gdp_chain_states_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap tm_phi;  // Phi, [steps][N][H][D][D] fp32, 32 x 32 boxes
  if ((e = tmap_state(&tm_phi, const_cast<float *>(phi), a.steps * a.N * a.H * D, D)) != cudaSuccess) return e;
  gdp_chain_states_kernel<D><<<dim3((unsigned)a.N, (unsigned)a.H, (unsigned)(D / kCmbRows)), kCmbThreads, smem,
                               stream>>>(a, tm_phi);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chain_states(const float *s0, const float *phi, const float *b, int64_t steps, int64_t N, int H,
                                int d, float *s_out, uint32_t *status, cudaStream_t stream) {
  if (N == 0) return cudaSuccess;
  const ChainArgs a{s0, b, s_out, steps, N, H, status};
  if (d == 64) return launch_chain_d<64>(a, phi, stream);
  if (d == 128) return launch_chain_d<128>(a, phi, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_piece_combine(const Problem &p, cudaStream_t stream) {
  if (p.N == 0 || p.piece_len <= 0) return cudaSuccess;
  const bool init16 = p.init && p.init_bf16 && !p.cache;
  if (p.K == 64) return init16 ? launch_combine_d<64, true>(p, stream) : launch_combine_d<64, false>(p, stream);
  if (p.K == 128) return init16 ? launch_combine_d<128, true>(p, stream) : launch_combine_d<128, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdp
