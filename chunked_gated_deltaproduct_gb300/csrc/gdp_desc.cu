// gdp_desc.cu -- varlen descriptor builder (K1).
//
// Megatron-Core API page "core.ssm.ops.gdp.chunk": parameters chunk_indices,
// chunk_indices_dp (the expanded stream, M times longer; not a rescaling of
// chunk_indices since ceil(L*M/64) != M*ceil(L/64) in general), chunk_offsets
// (prefix sum of the unexpanded chunk counts), and the closing paragraph
// (descriptors padded to a fixed length keep the launch grids constant, which
// makes the call capturable).
//
// One CTA: a block-wide exclusive scan over the sequences (tiles of 1024),
// then every padded row finds its sequence by binary search over the offsets
// (kept in shared memory up to kDescSmemSeqs sequences, else read back from
// global memory).  Grid and block sizes depend on nothing but the padded lengths.
#include "gdp_internal.cuh"
#include "gdp_sm100.cuh"

namespace gdp {
namespace {

constexpr int kDescThreads = 1024;
constexpr int kDescSmemSeqs = 2048;  // offsets of up to this many sequences stay in shared memory

__device__ __forceinline__ int block_exclusive_scan(int x, int *warp_sums, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_sums[lane] = wi - w;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  int r = warp_sums[warp] + incl - x;
  __syncthreads();
  return r;
}

// Rows of one descriptor table: row r -> (sequence, local chunk), (-1,-1) past the end.
__device__ void fill_rows(int32_t *rows, int64_t pad, const int32_t *offs, int64_t N) {
  const int64_t total = offs[N];
  for (int64_t r = threadIdx.x; r < pad; r += blockDim.x) {
    int32_t seq = -1, c = -1;
    if (r < total) {
      int64_t lo = 0, hi = N - 1;  // last i with offs[i] <= r
      while (lo < hi) {
        int64_t mid = (lo + hi + 1) >> 1;
        if (offs[mid] <= r) lo = mid; else hi = mid - 1;
      }
      seq = (int32_t)lo;
      c = (int32_t)(r - offs[lo]);
    }
    rows[2 * r] = seq;
    rows[2 * r + 1] = c;
  }
}

// Sequences the longest-first order is computed for (one thread per sequence, a count over all
// of them); larger batches keep their own order.
constexpr int64_t kOrderMaxSeqs = kDescThreads;

__global__ void __launch_bounds__(kDescThreads) gdp_desc_kernel(const void *cu, int cu64, int64_t T, int64_t N,
                                                                int M, int32_t *ci, int64_t nt_pad, int32_t *cid,
                                                                int64_t ntdp_pad, int32_t *co, int32_t *cod,
                                                                int32_t *order, uint32_t *status,
                                                                unsigned long long *bounds) {
  __shared__ int warp_sums[32];
  __shared__ int tot_a, tot_b;
  __shared__ int carry_a, carry_b;
  __shared__ int32_t s_co[kDescSmemSeqs + 1], s_cod[kDescSmemSeqs + 1];
  const bool in_smem = N <= kDescSmemSeqs;
  sm100::pdl_trigger();  // the WY kernel may start launching; it waits for these descriptors
  if (threadIdx.x == 0) {
    carry_a = carry_b = 0;
    if (N > 0 && (load_cu(cu, cu64, 0) != 0 || load_cu(cu, cu64, N) != T)) set_status(status, GDP_DEV_ERR_CU_SEQLENS);
  }
  __syncthreads();
  for (int64_t base = 0; base < N; base += blockDim.x) {
    const int64_t i = base + threadIdx.x;
    int a = 0, b = 0;
    if (i < N) {
      int64_t bos, L;
      if (!seq_bounds(cu, cu64, T, i, &bos, &L)) set_status(status, GDP_DEV_ERR_CU_SEQLENS);  // owns no chunks
      a = (int)((L + kChunk - 1) / kChunk);
      b = (int)((L * M + kChunk - 1) / kChunk);
    }
    int ea = block_exclusive_scan(a, warp_sums, &tot_a);
    int eb = block_exclusive_scan(b, warp_sums, &tot_b);
    if (i < N) {
      if (co) co[i] = carry_a + ea;
      if (cod) cod[i] = carry_b + eb;
      if (in_smem) {
        s_co[i] = carry_a + ea;
        s_cod[i] = carry_b + eb;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry_a += tot_a;
      carry_b += tot_b;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int a = carry_a, b = carry_b;
    if ((ci && a > nt_pad) || (cid && b > ntdp_pad)) set_status(status, GDP_DEV_ERR_DESC);
    if (co) co[N] = a;
    if (cod) cod[N] = b;
    if (in_smem) {
      s_co[N] = a;
      s_cod[N] = b;
    }
  }
  __syncthreads();  // makes the offsets written above visible to the whole block
  if (ci) fill_rows(ci, nt_pad, in_smem ? s_co : co, N);
  if (cid) fill_rows(cid, ntdp_pad, in_smem ? s_cod : cod, N);
  if (order) {
    // longest first: sequence i goes to position #{j : n_j > n_i} + #{j < i : n_j == n_i}, n the
    // expanded-chunk counts (a permutation: ties keep the sequences' own order)
    if (N <= kOrderMaxSeqs && in_smem) {
      const int64_t i = threadIdx.x;
      if (i < N) {
        const int ni = s_cod[i + 1] - s_cod[i];
        int rank = 0;
        for (int64_t j = 0; j < N; ++j) {
          const int nj = s_cod[j + 1] - s_cod[j];
          rank += (nj > ni) || (nj == ni && j < i);
        }
        if (in_range(bounds, status, GDP_BOUNDS_SITE_DESC, rank, N)) order[rank] = (int32_t)i;
      }
    } else {
      for (int64_t i = threadIdx.x; i < N; i += blockDim.x) order[i] = (int32_t)i;
    }
  }
}

}  // namespace

cudaError_t launch_descriptors(const void *cu, int cu64, int64_t T, int64_t N, int M, int32_t *ci, int64_t nt_pad,
                               int32_t *cid, int64_t ntdp_pad, int32_t *co, int32_t *cod, uint32_t *status,
                               cudaStream_t stream, int32_t *order, unsigned long long *bounds) {
  gdp_desc_kernel<<<1, kDescThreads, 0, stream>>>(cu, cu64, T, N, M, ci, nt_pad, cid, ntdp_pad, co, cod, order,
                                                  status, bounds);
  return cudaGetLastError();
}

}  // namespace gdp
