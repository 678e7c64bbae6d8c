// gdp_decode.cu -- one-token decode step of Gated DeltaProduct (the serving step after prefill).
//
// Attention-Cache-and-Sequence-Parallelism page, section "Prefill and decode" and the GDN
// section (decode keeps only the state S_t and advances it one token at a time with the
// recurrent form); Megatron-Core API page "core.ssm.ops.gdp.chunk", parameters state /
// state_indices (the per-request state cache, written in place; -1 marks padding);
// FlashInfer API page, display equation (the recurrence).  For the one token t = i of
// sequence i and every head:
//   S *= exp(g_t);  for j < M:  v_new = beta_j (v_j - S k_j),  S += v_new (x) k_j;
//   o_t = scale S q_t
// (k_j, q optionally L2-normalised: x / sqrt(sum x^2 + 1e-6)).  The input variants of the
// prefill apply (FlashInfer page, parameters q, k, v, g, beta, initial_state): float16
// q / k / v / output, a linear-space alpha gate (multiplied in directly), bf16 / f16 g and
// beta, a bf16 initial state, and q / k / v heads grouped over the state heads.
//
// The step is bandwidth-bound: per (sequence, head) it reads and writes the 64 KB fp32
// state and touches only M + 1 vectors of inputs.  One CTA per (sequence, head, 32 state
// rows); row v of S lives in the registers of four threads, which hold interleaved
// 16-byte column groups so that every load and store instruction of a warp moves whole
// 64-byte runs of eight rows.
#include "gdp_internal.cuh"

namespace gdp {
namespace {

constexpr int kDecRows = 32;             // state rows per CTA
constexpr int kDecThreads = kDecRows * 4;  // four threads per row
constexpr int kDecMaxM = 16;             // sub-token updates per token served by this kernel

struct DecodeProblem {
  const void *q, *k, *v;  // bf16, or f16 when f16 != 0
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh;
  const void *g, *beta;   // element types g_type, beta_type
  int64_t N;
  int H, K, V, M;
  uint64_t hmul_q, hmul_k, hmul_v;  // state head h reads head input_head(h, hmul_x) of q, k, v
  int f16, g_type, beta_type, g_alpha, init_bf16;
  float scale;
  int l2norm;
  const void *init;       // fp32, or bf16 when init_bf16 != 0
  float *cache;
  const int32_t *slots;
  int64_t num_slots;
  void *out;              // the q / k / v type
  float *out_state;
  uint32_t *status;
  unsigned long long *bounds;  // debug-bounds record (see in_range)
  int vec_in;  // q, k, v rows start on 16-byte boundaries (bases and strides): 16-byte input loads
};

__device__ __forceinline__ float load16(const void *base, int64_t i, int f16) {
  return f16 ? __half2float(static_cast<const __half *>(base)[i])
             : __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[i]);
}

template <int D>
__global__ void __launch_bounds__(kDecThreads) gdp_decode_kernel(DecodeProblem p) {
  constexpr int G = D / 16;  // float4 column groups per thread
  const int i = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, r = tid >> 2, qd = tid & 3;
  const int vrow = blockIdx.z * kDecRows + r;
  const int M = p.M;
  const int hq = input_head(h, p.hmul_q), hk = input_head(h, p.hmul_k), hv = input_head(h, p.hmul_v);
  __shared__ float kf[kDecMaxM][D];
  __shared__ float qf[D];
  __shared__ float vv[kDecMaxM][kDecRows];
  __shared__ float bt[kDecMaxM];
  __shared__ float red[kDecMaxM + 1];

  // the state row: slot / initial state / zero
  int slot = -1;
  const float *src = nullptr;
  const __nv_bfloat16 *src16 = nullptr;  // a bf16 initial state
  float *dst = nullptr;
  if (!in_range(p.bounds, p.status, GDP_BOUNDS_SITE_DECODE, i, p.N)) return;
  if (p.cache) {
    slot = p.slots[i];
    if (slot < -1 || slot >= p.num_slots) {
      if (tid == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_status(p.status, GDP_DEV_ERR_SLOT);
      slot = -1;
    }
    if (slot >= 0 && !in_range(p.bounds, p.status, GDP_BOUNDS_SITE_DECODE, slot, p.num_slots)) slot = -1;
    if (slot >= 0) src = dst = p.cache + ((int64_t)slot * p.H + h) * (int64_t)p.V * D;
  } else {
    if (p.init && p.init_bf16)
      src16 = static_cast<const __nv_bfloat16 *>(p.init) + ((int64_t)i * p.H + h) * (int64_t)p.V * D;
    else if (p.init)
      src = static_cast<const float *>(p.init) + ((int64_t)i * p.H + h) * (int64_t)p.V * D;
    if (p.out_state) dst = p.out_state + ((int64_t)i * p.H + h) * (int64_t)p.V * D;
  }
  // thread (row, qd) holds columns 16 g' + 4 qd .. + 3 for g' < G: a warp's 4-thread groups
  // read 64 contiguous bytes of each of its 8 rows per instruction
  float s[4 * G];
  // issued first, so that the state's HBM latency overlaps the input loads below
#pragma unroll
  for (int gi = 0; gi < G; ++gi) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (src) {
      x = *reinterpret_cast<const float4 *>(src + (int64_t)vrow * D + gi * 16 + qd * 4);
    } else if (src16) {
      const uint2 y = *reinterpret_cast<const uint2 *>(src16 + (int64_t)vrow * D + gi * 16 + qd * 4);
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&y.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&y.y));
      x = make_float4(a.x, a.y, b.x, b.y);
    }
    s[4 * gi] = x.x; s[4 * gi + 1] = x.y; s[4 * gi + 2] = x.z; s[4 * gi + 3] = x.w;
  }
  // inputs of the token: k rows i*M + j, q row i, this block's v entries, beta, gate -- every load
  // issued before any is used (16-byte groups of 8 elements when the layout allows)
  const float graw = p.g ? load_typed(p.g, (int64_t)i * p.H + h, p.g_type) : 0.f;
  const float braw = (tid < M && p.beta) ? load_typed(p.beta, ((int64_t)i * M + tid) * p.H + h, p.beta_type) : 1.f;
  if (p.vec_in) {
    constexpr int GPR = D / 8;  // 8-element groups per row
    const int ng = (M + 1) * GPR;
    auto kq_src = [&](int gi) {
      const int j = gi / GPR, c8 = (gi % GPR) * 8;
      return j < M ? static_cast<const uint16_t *>(p.k) + ((int64_t)i * M + j) * p.k_st + (int64_t)hk * p.k_sh + c8
                   : static_cast<const uint16_t *>(p.q) + (int64_t)i * p.q_st + (int64_t)hq * p.q_sh + c8;
    };
    uint4 raw[3], rv = make_uint4(0u, 0u, 0u, 0u);  // (M + 1) * GPR <= 17 * 16 = 272 groups
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      const int gi = tid + u * kDecThreads;
      raw[u] = gi < ng ? *reinterpret_cast<const uint4 *>(kq_src(gi)) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid < M * (kDecRows / 8))
      rv = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p.v) +
                                            ((int64_t)i * M + tid / (kDecRows / 8)) * p.v_st + (int64_t)hv * p.v_sh +
                                            blockIdx.z * kDecRows + (tid % (kDecRows / 8)) * 8);
    auto widen8 = [&](const uint4 &x, float *o) {
      const uint16_t *e = reinterpret_cast<const uint16_t *>(&x);
#pragma unroll
      for (int w = 0; w < 8; ++w)
        o[w] = p.f16 ? __half2float(__ushort_as_half(e[w])) : __uint_as_float((uint32_t)e[w] << 16);
    };
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      const int gi = tid + u * kDecThreads;
      if (gi < ng) {
        const int j = gi / GPR, c8 = (gi % GPR) * 8;
        widen8(raw[u], j < M ? &kf[j][c8] : &qf[c8]);
      }
    }
    if (tid < M * (kDecRows / 8)) widen8(rv, &vv[tid / (kDecRows / 8)][(tid % (kDecRows / 8)) * 8]);
  } else {
    for (int idx = tid; idx < (M + 1) * D; idx += kDecThreads) {
      const int j = idx / D, c = idx % D;
      float x;
      if (j < M)
        x = load16(p.k, ((int64_t)i * M + j) * p.k_st + (int64_t)hk * p.k_sh + c, p.f16);
      else
        x = load16(p.q, (int64_t)i * p.q_st + (int64_t)hq * p.q_sh + c, p.f16);
      if (j < M) kf[j][c] = x; else qf[c] = x;
    }
    for (int idx = tid; idx < M * kDecRows; idx += kDecThreads) {
      const int j = idx / kDecRows, rr = idx % kDecRows;
      vv[j][rr] = load16(p.v, ((int64_t)i * M + j) * p.v_st + (int64_t)hv * p.v_sh + blockIdx.z * kDecRows + rr, p.f16);
    }
  }
  if (tid < M) bt[tid] = braw;
  __syncthreads();
  if (p.l2norm) {  // one warp per vector: 1 / sqrt(sum x^2 + eps)
    const int warp = tid >> 5, lane = tid & 31;
    for (int j = warp; j <= M; j += kDecThreads / 32) {
      const float *x = (j < M) ? kf[j] : qf;
      float ss = 0.f;
      for (int c = lane; c < D; c += 32) ss += x[c] * x[c];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) red[j] = rsqrtf(ss + kL2Eps);
    }
    __syncthreads();
    for (int idx = tid; idx < (M + 1) * D; idx += kDecThreads) {
      const int j = idx / D, c = idx % D;
      if (j < M) kf[j][c] *= red[j]; else qf[c] *= red[M];
    }
    __syncthreads();
  }

  // alpha_t = exp(g_t), or g_t itself for a linear-space gate (floored like the prefill's)
  float decay = 1.f;
  if (p.g) decay = p.g_alpha ? fmaxf(graw, __expf(kMinLogAlpha)) : __expf(graw);
#pragma unroll
  for (int c = 0; c < 4 * G; ++c) s[c] *= decay;
  for (int j = 0; j < M; ++j) {
    float dot = 0.f;
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
#pragma unroll
      for (int u = 0; u < 4; ++u) dot += s[4 * gi + u] * kf[j][gi * 16 + qd * 4 + u];
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
    const float vn = bt[j] * (vv[j][r] - dot);
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
#pragma unroll
      for (int u = 0; u < 4; ++u) s[4 * gi + u] += vn * kf[j][gi * 16 + qd * 4 + u];
  }
  float o = 0.f;
#pragma unroll
  for (int gi = 0; gi < G; ++gi)
#pragma unroll
    for (int u = 0; u < 4; ++u) o += s[4 * gi + u] * qf[gi * 16 + qd * 4 + u];
  o += __shfl_xor_sync(0xffffffffu, o, 1);
  o += __shfl_xor_sync(0xffffffffu, o, 2);
  if (qd == 0) {
    uint16_t *out = static_cast<uint16_t *>(p.out) + ((int64_t)i * p.H + h) * p.V + vrow;
    *out = p.f16 ? __half_as_ushort(__float2half_rn(p.scale * o)) : __bfloat16_as_ushort(__float2bfloat16_rn(p.scale * o));
  }
  if (dst) {
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
      *reinterpret_cast<float4 *>(dst + (int64_t)vrow * D + gi * 16 + qd * 4) =
          make_float4(s[4 * gi], s[4 * gi + 1], s[4 * gi + 2], s[4 * gi + 3]);
  }
}

}  // namespace
}  // namespace gdp

#define GDP_EXPORT extern "C" __attribute__((visibility("default")))

GDP_EXPORT gdp_status gdp_decode_step(const gdp_prefill_args *a, void *stream) {
  gdp::set_last_error("");
  auto fail = [](gdp_status st, const char *why) {
    gdp::set_last_error("%s", why);
    return st;
  };
  if (!a) return fail(GDP_ERR_INVALID_ARG, "args is NULL");
  const int64_t T = a->T, N = a->N;
  const int H = a->H, K = a->K, V = a->V, M = a->num_householder;
  if (T != N || N < 0 || H < 1 || M < 1) return fail(GDP_ERR_INVALID_ARG, "decode takes one token per sequence: T == N >= 0, H >= 1, M >= 1");
  if (K != V || (K != 64 && K != 128)) return fail(GDP_ERR_UNSUPPORTED, "head size K = V must be 64 or 128");
  if (M > gdp::kDecMaxM) return fail(GDP_ERR_UNSUPPORTED, "num_householder above 16 is not served by the decode step");
  if (N > INT32_MAX || H > 65535) return fail(GDP_ERR_UNSUPPORTED, "grid limits: N < 2^31, H <= 65535");
  if (N > 0 && (!a->q || !a->k || !a->v || !a->output)) return fail(GDP_ERR_INVALID_ARG, "q, k, v and output are required");
  const int64_t strides[6] = {a->q_stride_t, a->q_stride_h, a->k_stride_t, a->k_stride_h, a->v_stride_t, a->v_stride_h};
  for (int s = 0; s < 6; ++s)
    if (N > 0 && strides[s] <= 0) return fail(GDP_ERR_INVALID_ARG, "strides must be positive");
  const uintptr_t salign = ((uintptr_t)a->initial_state | (uintptr_t)a->state | (uintptr_t)a->output_state) & 15u;
  if (salign) return fail(GDP_ERR_INVALID_ARG, "state buffers must be 16-byte aligned");
  if (a->state && a->initial_state) return fail(GDP_ERR_INVALID_ARG, "state (cache mode) and initial_state are mutually exclusive");
  if (a->state && (!a->state_indices || a->num_slots < 1))
    return fail(GDP_ERR_INVALID_ARG, "state cache needs state_indices and num_slots >= 1");
  if (a->state && a->output_state)
    return fail(GDP_ERR_INVALID_ARG, "in cache mode the final state is written to the cache; output_state must be NULL");
  if (a->chunk_states) return fail(GDP_ERR_INVALID_ARG, "chunk_states has no meaning for a decode step");
  gdp::Problem vp{};
  const gdp_status vst = gdp::resolve_variants(a, &vp);
  if (vst != GDP_OK) return vst;
  if (a->initial_state && a->output_state) {
    const size_t bytes = sizeof(float) * (size_t)N * H * (size_t)V * K;
    const size_t ibytes = vp.init_bf16 ? bytes / 2 : bytes;
    const uintptr_t x = (uintptr_t)a->initial_state, y = (uintptr_t)a->output_state;
    if ((x != y || vp.init_bf16) && x < y + bytes && y < x + ibytes)
      return fail(GDP_ERR_ALIAS, "output_state overlaps initial_state (only an exact in-place fp32 update is allowed)");
  }
  if (N == 0) return GDP_OK;
  gdp::DecodeProblem p{};
  p.q = a->q; p.k = a->k; p.v = a->v;
  p.hmul_q = vp.hmul_q; p.hmul_k = vp.hmul_k; p.hmul_v = vp.hmul_v;
  p.f16 = vp.f16; p.g_type = vp.g_type; p.beta_type = vp.beta_type; p.g_alpha = vp.g_alpha; p.init_bf16 = vp.init_bf16;
  p.q_st = a->q_stride_t; p.q_sh = a->q_stride_h;
  p.k_st = a->k_stride_t; p.k_sh = a->k_stride_h;
  p.v_st = a->v_stride_t; p.v_sh = a->v_stride_h;
  p.g = a->g; p.beta = a->beta;
  p.N = N; p.H = H; p.K = K; p.V = V; p.M = M;
  p.scale = (a->scale > 0.f && a->scale == a->scale) ? a->scale : 1.0f / sqrtf((float)K);
  p.l2norm = a->use_qk_l2norm ? 1 : 0;
  p.init = a->initial_state; p.cache = a->state; p.slots = a->state_indices; p.num_slots = a->num_slots;
  p.out = a->output; p.out_state = a->output_state; p.status = a->device_status;
  p.bounds = gdp::bounds_record();
  p.vec_in = (((uintptr_t)a->q | (uintptr_t)a->k | (uintptr_t)a->v) & 15u) == 0 && p.q_st % 8 == 0 &&
             p.q_sh % 8 == 0 && p.k_st % 8 == 0 && p.k_sh % 8 == 0 && p.v_st % 8 == 0 && p.v_sh % 8 == 0;
  dim3 grid((unsigned)N, (unsigned)H, (unsigned)(V / gdp::kDecRows));
  cudaStream_t s = (cudaStream_t)stream;
  if (K == 128)
    gdp::gdp_decode_kernel<128><<<grid, gdp::kDecThreads, 0, s>>>(p);
  else
    gdp::gdp_decode_kernel<64><<<grid, gdp::kDecThreads, 0, s>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    gdp::set_last_error("decode kernel: %s", cudaGetErrorString(e));
    return GDP_ERR_CUDA;
  }
  return GDP_OK;
}
