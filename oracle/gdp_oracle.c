/*
 * gdp_oracle.c -- float64 CPU oracle for the chunked, variable-length Gated
 * DeltaProduct (GDP) prefill forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py may load this library.  It shares no code,
 * header, table or helper with the CUDA library; it is written from the
 * method's definition alone:
 *
 *   FlashInfer API page "flashinfer.gdp_prefill.chunk_gated_delta_product",
 *   opening paragraph and its display equation: per real token t,
 *       S *= alpha_t
 *       for j = 0 .. n-1:  v_new = beta_{t,j} (v_{t,j} - S k_{t,j});  S += v_new (x) k_{t,j}
 *       o_t = scale * S q_t
 *   with the n sub-token rows of k / v / beta at t*n .. t*n+n-1 (parameters k, v, beta),
 *   the state V-major [.., V, K] (parameter initial_state), packed THD input over
 *   cu_seqlens (parameter cu_seqlens).
 *
 *   Megatron-Core API page "core.ssm.ops.gdp.chunk": g holds natural-log decays
 *   (parameter g), so alpha_t = exp(g_t); chunk size 64 and the two chunkings
 *   (stage list, last paragraph; parameter chunk_indices_dp); the chunk-state row
 *   chunk_offsets[i] + c is the state ENTERING chunk c, i.e. after 64*c tokens
 *   (parameter return_chunk_states); the state cache is written in place at
 *   state_indices, -1 marking padding (parameters state, state_indices).
 *
 * Everything is computed in float64 from the exact values of the bf16 / f16 /
 * fp32 inputs (every such bit pattern widens to float64 exactly).  The only liberty
 * taken: the V rows of S are handed to different threads.  Each row of S
 * evolves on its own (row v of v_new only reads row v of S), so every row
 * sees exactly the arithmetic of the unsplit loop, in the same order.
 *
 * Input variants (FlashInfer page, parameters q, k, v, g, beta,
 * initial_state): q / k / v may be float16 instead of bfloat16 (widened
 * exactly by widen_f16 below, from the IEEE 754 binary16 definition); g may
 * hold the gate alpha itself in linear space instead of its natural log, in
 * which case S is multiplied by alpha as given; the head counts of q, k and v
 * may be smaller than the state head count H.  Reading of the head relation
 * (the page names the counts but not the map): H is the larger of the q and v
 * head counts, every count divides H, and state head h reads q head
 * h / (H / Hq), k head h / (H / Hk) and v head h / (H / Hv), so each head of a
 * smaller count serves a run of consecutive state heads.  g, beta, the states
 * and the output have H heads.
 *
 * Readings where the pages are silent (the same list is kept in the design
 * notes): q/k L2 normalisation is x / sqrt(sum x^2 + 1e-6), applied in float64
 * and not rounded; a padding sequence (slot -1) starts from a zero state, its
 * output is still produced, and nothing is written to the cache for it; an
 * empty sequence copies its initial state through and owns no chunk rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_CHUNK 64
#define ORACLE_L2_EPS 1e-6
#define ORACLE_VROWS 16

static double widen_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE 754 binary16: sign bit, 5-bit exponent with bias 15, 10-bit fraction;
 * exponent 0 holds zero and the subnormals (fraction * 2^-24), exponent 31
 * infinity and NaN. */
static double widen_f16(uint16_t bits) {
  const int sign = (bits >> 15) & 1, ex = (bits >> 10) & 31, fr = bits & 1023;
  double mag;
  if (ex == 0)
    mag = ldexp((double)fr, -24);
  else if (ex == 31)
    mag = fr ? NAN : INFINITY;
  else
    mag = ldexp((double)(1024 + fr), ex - 25);
  return sign ? -mag : mag;
}

static double widen_half(uint16_t bits, int f16) { return f16 ? widen_f16(bits) : widen_bf16(bits); }

/* Exported for the tests: the binary16 widening above, one bit pattern. */
double gdp_oracle_widen_f16(uint16_t bits) { return widen_f16(bits); }

static int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Varlen descriptors (Megatron page, parameters chunk_indices, chunk_indices_dp,
 * chunk_offsets; capture note in the closing paragraph).  Rows are
 * (sequence, local chunk); rows past the real count are (-1, -1).
 * Returns 0, or -1 if cu_seqlens is not non-decreasing from 0, or -2 if a
 * padded bound is too small. */
int gdp_oracle_descriptors(const int64_t *cu_seqlens, int64_t N, int M,
                           int32_t *chunk_indices, int64_t nt_pad,
                           int32_t *chunk_indices_dp, int64_t ntdp_pad,
                           int32_t *chunk_offsets, int32_t *chunk_offsets_dp) {
  int64_t nt = 0, ntdp = 0;
  if (N > 0 && cu_seqlens[0] != 0) return -1;
  for (int64_t i = 0; i < N; ++i) {
    int64_t L = cu_seqlens[i + 1] - cu_seqlens[i];
    if (L < 0) return -1;
    if (chunk_offsets) chunk_offsets[i] = (int32_t)nt;
    if (chunk_offsets_dp) chunk_offsets_dp[i] = (int32_t)ntdp;
    nt += ceil_div64(L, ORACLE_CHUNK);
    ntdp += ceil_div64(L * M, ORACLE_CHUNK);
  }
  if (chunk_offsets) chunk_offsets[N] = (int32_t)nt;
  if (chunk_offsets_dp) chunk_offsets_dp[N] = (int32_t)ntdp;
  if ((chunk_indices && nt > nt_pad) || (chunk_indices_dp && ntdp > ntdp_pad)) return -2;
  if (chunk_indices) {
    int64_t r = 0;
    for (int64_t i = 0; i < N; ++i) {
      int64_t n = ceil_div64(cu_seqlens[i + 1] - cu_seqlens[i], ORACLE_CHUNK);
      for (int64_t c = 0; c < n; ++c, ++r) {
        chunk_indices[2 * r] = (int32_t)i;
        chunk_indices[2 * r + 1] = (int32_t)c;
      }
    }
    for (; r < nt_pad; ++r) chunk_indices[2 * r] = chunk_indices[2 * r + 1] = -1;
  }
  if (chunk_indices_dp) {
    int64_t r = 0;
    for (int64_t i = 0; i < N; ++i) {
      int64_t n = ceil_div64((cu_seqlens[i + 1] - cu_seqlens[i]) * M, ORACLE_CHUNK);
      for (int64_t c = 0; c < n; ++c, ++r) {
        chunk_indices_dp[2 * r] = (int32_t)i;
        chunk_indices_dp[2 * r + 1] = (int32_t)c;
      }
    }
    for (; r < ntdp_pad; ++r) chunk_indices_dp[2 * r] = chunk_indices_dp[2 * r + 1] = -1;
  }
  return 0;
}

/* Load a head-row of a bf16 (f16 = 0) or float16 (f16 = 1) [rows][H][D]
 * tensor as float64, optionally L2-normalised (FlashInfer page, parameter
 * use_qk_l2norm_in_kernel). */
static void load_row(const uint16_t *base, int64_t row, int H, int h, int D,
                     int f16, int normalise, double *out) {
  const uint16_t *p = base + (row * H + h) * (int64_t)D;
  double ss = 0.0;
  for (int d = 0; d < D; ++d) {
    out[d] = widen_half(p[d], f16);
    ss += out[d] * out[d];
  }
  if (normalise) {
    double inv = 1.0 / sqrt(ss + ORACLE_L2_EPS);
    for (int d = 0; d < D; ++d) out[d] *= inv;
  }
}

/*
 * The forward pass, token by token.
 *
 *   q [T][Hq][K], k [T*M][Hk][K], v [T*M][Hv][V]: bf16 (qkv_f16 = 0) or
 *   float16 (qkv_f16 = 1) bit patterns; state head h reads q head h / (H / Hq),
 *   k head h / (H / Hk), v head h / (H / Hv) (each count divides H).
 *   g [T][H]: natural-log decay (g_is_alpha = 0) or alpha itself (g_is_alpha = 1);
 *   NULL: no decay.  beta [T*M][H] (NULL: ones).
 *   Incoming state: state-cache mode when state_in != NULL (slot = state_indices[i],
 *   slot >= 0 reads state_in[slot], slot -1 starts from zero); otherwise
 *   initial_state[i] when non-NULL; otherwise zero.  States are [..][H][V][K] fp32.
 *   head_mask [H] (NULL: all heads) selects the heads computed; other heads'
 *   outputs are left as they are.
 * Outputs (float64, any may be NULL):
 *   o [T][H][V]; final_state [N][H][V][K] (every sequence, padding included);
 *   state_out [num_slots][H][V][K]: in cache mode, the final state of each
 *   sequence with slot >= 0 is stored at its slot (the caller fills the rest);
 *   chunk_states [NT][H][V][K] with NT = chunk_offsets[N]: row
 *   chunk_offsets[i] + c holds the state entering token chunk c.
 * Returns 0, or a negative code for an argument the definition cannot serve.
 */
int gdp_oracle_forward(int64_t T, int64_t N, int H, int K, int V, int M,
                       int Hq, int Hk, int Hv, int qkv_f16, int g_is_alpha,
                       const int64_t *cu_seqlens,
                       const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const float *g, const float *beta, double scale,
                       int use_qk_l2norm,
                       const float *initial_state,
                       const float *state_in, const int32_t *state_indices,
                       int64_t num_slots,
                       const int32_t *chunk_offsets,
                       const uint8_t *head_mask,
                       double *o, double *final_state, double *state_out,
                       double *chunk_states, int num_threads) {
  if (T < 0 || N < 0 || H <= 0 || K <= 0 || V <= 0 || M <= 0) return -1;
  if (Hq <= 0 || Hk <= 0 || Hv <= 0 || H % Hq || H % Hk || H % Hv) return -6;
  if (chunk_states && !chunk_offsets) return -2;
  if (state_in && !state_indices) return -3;
  if (N > 0 && (cu_seqlens[0] != 0 || cu_seqlens[N] != T)) return -4;
  for (int64_t i = 0; i < N; ++i)
    if (cu_seqlens[i + 1] < cu_seqlens[i]) return -4;
  if (state_in)
    for (int64_t i = 0; i < N; ++i)
      if (state_indices[i] >= num_slots || state_indices[i] < -1) return -5;

  const int vblocks = (V + ORACLE_VROWS - 1) / ORACLE_VROWS;
  const int64_t ntasks = N * (int64_t)H * vblocks;
  const int64_t KV = (int64_t)K * V;
  int rc = 0;

#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel
#endif
  {
    double *S = (double *)malloc(sizeof(double) * ORACLE_VROWS * K);
    double *kr = (double *)malloc(sizeof(double) * K);
    double *qt = (double *)malloc(sizeof(double) * K);
    if (!S || !kr || !qt) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      rc = -10;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int64_t task = 0; task < ntasks; ++task) {
        const int64_t i = task / ((int64_t)H * vblocks);
        const int h = (int)((task / vblocks) % H);
        const int vb = (int)(task % vblocks);
        if (head_mask && !head_mask[h]) continue;
        const int v0 = vb * ORACLE_VROWS;
        const int nv = (V - v0) < ORACLE_VROWS ? (V - v0) : ORACLE_VROWS;
        const int64_t bos = cu_seqlens[i], eos = cu_seqlens[i + 1];

        /* incoming state rows v0 .. v0+nv-1 */
        const float *src = NULL;
        if (state_in) {
          int32_t slot = state_indices[i];
          if (slot >= 0) src = state_in + ((int64_t)slot * H + h) * KV;
        } else if (initial_state) {
          src = initial_state + (i * H + h) * KV;
        }
        for (int r = 0; r < nv; ++r)
          for (int d = 0; d < K; ++d)
            S[r * K + d] = src ? (double)src[(int64_t)(v0 + r) * K + d] : 0.0;

        for (int64_t t = bos; t < eos; ++t) {
          const int64_t lt = t - bos;
          if (chunk_states && lt % ORACLE_CHUNK == 0) {
            double *dst = chunk_states +
                          (((int64_t)chunk_offsets[i] + lt / ORACLE_CHUNK) * H + h) * KV;
            for (int r = 0; r < nv; ++r)
              for (int d = 0; d < K; ++d) dst[(int64_t)(v0 + r) * K + d] = S[r * K + d];
          }
          /* decay once per real token, before its updates */
          const double alpha = !g ? 1.0 : g_is_alpha ? (double)g[t * H + h] : exp((double)g[t * H + h]);
          for (int x = 0; x < nv * K; ++x) S[x] *= alpha;
          /* n beta-gated Householder updates on the expanded rows t*M + j */
          for (int j = 0; j < M; ++j) {
            const int64_t row = t * M + j;
            load_row(k, row, Hk, h / (H / Hk), K, qkv_f16, use_qk_l2norm, kr);
            const double b = beta ? (double)beta[row * H + h] : 1.0;
            for (int r = 0; r < nv; ++r) {
              double *Sr = S + r * K;
              double pred = 0.0;
              for (int d = 0; d < K; ++d) pred += Sr[d] * kr[d];
              const double vv = widen_half(v[(row * Hv + h / (H / Hv)) * (int64_t)V + v0 + r], qkv_f16);
              const double vnew = b * (vv - pred);
              for (int d = 0; d < K; ++d) Sr[d] += vnew * kr[d];
            }
          }
          /* readout after the last update */
          if (o) {
            load_row(q, t, Hq, h / (H / Hq), K, qkv_f16, use_qk_l2norm, qt);
            for (int r = 0; r < nv; ++r) {
              const double *Sr = S + r * K;
              double acc = 0.0;
              for (int d = 0; d < K; ++d) acc += Sr[d] * qt[d];
              o[(t * H + h) * (int64_t)V + v0 + r] = scale * acc;
            }
          }
        }

        if (final_state) {
          double *dst = final_state + (i * H + h) * KV;
          for (int r = 0; r < nv; ++r)
            for (int d = 0; d < K; ++d) dst[(int64_t)(v0 + r) * K + d] = S[r * K + d];
        }
        if (state_in && state_out && state_indices[i] >= 0) {
          double *dst = state_out + ((int64_t)state_indices[i] * H + h) * KV;
          for (int r = 0; r < nv; ++r)
            for (int d = 0; d < K; ++d) dst[(int64_t)(v0 + r) * K + d] = S[r * K + d];
        }
      }
    }
    free(S);
    free(kr);
    free(qt);
  }
  return rc;
}

/* Within-chunk cumulative decay of the expanded stream in base 2 (Megatron
 * page, stage 1): row r = t*M + j carries g_t when j == 0 and 0 otherwise;
 * the sum restarts at every 64-row chunk of the expanded sequence and is
 * multiplied by log2(e).  Output G2 [T*M][H] (float64). */
int gdp_oracle_decay_cumsum(int64_t T, int64_t N, int H, int M,
                            const int64_t *cu_seqlens, const float *g, double *G2) {
  const double log2e = 1.0 / log(2.0);
  for (int64_t i = 0; i < N; ++i) {
    const int64_t r0 = cu_seqlens[i] * M, r1 = cu_seqlens[i + 1] * M;
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int64_t r = r0; r < r1; ++r) {
        if ((r - r0) % ORACLE_CHUNK == 0) acc = 0.0;
        if (g && r % M == 0) acc += (double)g[(r / M) * H + h];
        G2[r * H + h] = acc * log2e;
      }
    }
  }
  return 0;
}

/*
 * The backward pass (reverse mode of the recurrence above), for training.
 *
 * The blog post "Attention Cache and Sequence Parallelism" (GDN section and the
 * section on passing state instead of KV) notes that training runs the same
 * recurrence in chunks and that its backward dependence runs the other way
 * round; the pages print no backward formula, so this function is the
 * derivative of the forward definition taken step by step, nothing else.
 * For a loss L with dL/do = d_output and dL/dS_final = d_final_state, walking
 * the expanded rows of each sequence backwards with D = dL/dS:
 *
 *   readout row r = t*M + M-1:  D += scale do_t qhat_t^T;  dqhat_t = scale S_r^T do_t
 *   update row r (P_r = the state before the update, e_r = v_r - P_r khat_r):
 *       delta = D khat_r;  dv_r = beta_r delta;  dbeta_r = e_r . delta
 *       dkhat_r = beta_r D^T e_r - P_r^T dv_r;   D <- D - dv_r khat_r^T
 *   first row of token t (the decay S <- alpha_t S, alpha_t = exp(g_t)):
 *       dg_t = <D, P_r> (Frobenius);  D <- alpha_t D
 *   start of the sequence: d_initial_state = D.
 * With use_qk_l2norm, xhat = x / n, n = sqrt(|x|^2 + eps), and
 *   dx = dxhat / n - x (x . dxhat) / n^3.
 *
 * Inputs are float64 (the caller widens bf16 / fp32 values exactly); heads are
 * one-to-one (Hq = Hk = Hv = H) and g is a natural-log decay.  The states P_r
 * of one 64-token block are recomputed from a checkpoint taken in a forward
 * sweep (the same arithmetic, in the same order, as that sweep).  One task per
 * (sequence, head).  Optional o and final_state receive the forward values.
 * Returns 0, or a negative code for an argument it cannot serve.
 */
int gdp_oracle_backward(int64_t T, int64_t N, int H, int K, int V, int M,
                        const int64_t *cu_seqlens,
                        const double *q, const double *k, const double *v,
                        const double *g, const double *beta, double scale,
                        int use_qk_l2norm, const double *initial_state,
                        const double *d_output, const double *d_final_state,
                        double *dq, double *dk, double *dv, double *dg,
                        double *dbeta, double *d_initial_state,
                        double *o, double *final_state, int num_threads) {
  if (T < 0 || N < 0 || H <= 0 || K <= 0 || V <= 0 || M <= 0) return -1;
  if (N > 0 && (cu_seqlens[0] != 0 || cu_seqlens[N] != T)) return -4;
  for (int64_t i = 0; i < N; ++i)
    if (cu_seqlens[i + 1] < cu_seqlens[i]) return -4;
  if (!d_output) return -2;
  const int64_t KV = (int64_t)K * V;
  const int B = ORACLE_CHUNK;  /* tokens per checkpoint block */
  const int64_t ntasks = N * (int64_t)H;
  int rc = 0;

#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel
#endif
  {
    double *S = (double *)malloc(sizeof(double) * KV);
    double *D = (double *)malloc(sizeof(double) * KV);
    double *Pst = (double *)malloc(sizeof(double) * KV * (size_t)B * M);  /* P_r of one block */
    double *kh = (double *)malloc(sizeof(double) * K);
    double *qh = (double *)malloc(sizeof(double) * K);
    double *dkh = (double *)malloc(sizeof(double) * K);
    double *e = (double *)malloc(sizeof(double) * V);
    double *dl = (double *)malloc(sizeof(double) * V);
    double *dvv = (double *)malloc(sizeof(double) * V);
    if (!S || !D || !Pst || !kh || !qh || !dkh || !e || !dl || !dvv) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      rc = -10;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int64_t task = 0; task < ntasks; ++task) {
        const int64_t i = task / H;
        const int h = (int)(task % H);
        const int64_t bos = cu_seqlens[i], eos = cu_seqlens[i + 1], L = eos - bos;
        const int64_t nblk = (L + B - 1) / B;
        double *ck = (double *)malloc(sizeof(double) * KV * (size_t)(nblk + 1));
        if (!ck) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
          rc = -10;
          continue;
        }
        /* row loaders: khat_r and qhat_t of head h (optionally L2-normalised) */
#define ORACLE_HAT(src, row, out)                                             \
  do {                                                                        \
    const double *p_ = (src) + ((int64_t)(row) * H + h) * (int64_t)K;         \
    double ss_ = 0.0;                                                         \
    for (int d_ = 0; d_ < K; ++d_) ss_ += p_[d_] * p_[d_];                    \
    const double inv_ = use_qk_l2norm ? 1.0 / sqrt(ss_ + ORACLE_L2_EPS) : 1.0; \
    for (int d_ = 0; d_ < K; ++d_) (out)[d_] = p_[d_] * inv_;                 \
  } while (0)

        /* one token of the forward recurrence on S; with Pout, stores P_r of every row */
#define ORACLE_TOKEN(t, Pout)                                                                   \
  do {                                                                                          \
    const double a_ = g ? exp(g[(t) * H + h]) : 1.0;                                            \
    for (int64_t x_ = 0; x_ < KV; ++x_) S[x_] *= a_;                                            \
    for (int j_ = 0; j_ < M; ++j_) {                                                            \
      const int64_t r_ = (t) * M + j_;                                                          \
      ORACLE_HAT(k, r_, kh);                                                                    \
      if (Pout) memcpy((Pout) + (size_t)j_ * KV, S, sizeof(double) * KV);                       \
      const double b_ = beta ? beta[r_ * H + h] : 1.0;                                          \
      for (int vv_ = 0; vv_ < V; ++vv_) {                                                       \
        double *Sr_ = S + (int64_t)vv_ * K, pred_ = 0.0;                                        \
        for (int d_ = 0; d_ < K; ++d_) pred_ += Sr_[d_] * kh[d_];                               \
        const double vn_ = b_ * (v[(r_ * H + h) * (int64_t)V + vv_] - pred_);                   \
        for (int d_ = 0; d_ < K; ++d_) Sr_[d_] += vn_ * kh[d_];                                 \
      }                                                                                         \
    }                                                                                           \
  } while (0)

        /* forward sweep: checkpoints at the start of every block, outputs, final state */
        for (int64_t x = 0; x < KV; ++x) S[x] = initial_state ? initial_state[(i * H + h) * KV + x] : 0.0;
        for (int64_t t = bos; t < eos; ++t) {
          if ((t - bos) % B == 0) memcpy(ck + (size_t)((t - bos) / B) * KV, S, sizeof(double) * KV);
          ORACLE_TOKEN(t, (double *)NULL);
          if (o) {
            ORACLE_HAT(q, t, qh);
            for (int vv = 0; vv < V; ++vv) {
              double acc = 0.0;
              for (int d = 0; d < K; ++d) acc += S[(int64_t)vv * K + d] * qh[d];
              o[(t * H + h) * (int64_t)V + vv] = scale * acc;
            }
          }
        }
        if (final_state) memcpy(final_state + (i * H + h) * KV, S, sizeof(double) * KV);

        /* backward sweep */
        for (int64_t x = 0; x < KV; ++x) D[x] = d_final_state ? d_final_state[(i * H + h) * KV + x] : 0.0;
        for (int64_t blk = nblk - 1; blk >= 0; --blk) {
          const int64_t t0 = bos + blk * B, t1 = (t0 + B < eos) ? t0 + B : eos;
          memcpy(S, ck + (size_t)blk * KV, sizeof(double) * KV);
          for (int64_t t = t0; t < t1; ++t) ORACLE_TOKEN(t, Pst + (size_t)(t - t0) * M * KV);
          for (int64_t t = t1 - 1; t >= t0; --t) {
            for (int j = M - 1; j >= 0; --j) {
              const int64_t r = t * M + j;
              const double *P = Pst + ((size_t)(t - t0) * M + j) * KV;
              const double b = beta ? beta[r * H + h] : 1.0;
              ORACLE_HAT(k, r, kh);
              for (int vv = 0; vv < V; ++vv) {  /* e_r = v_r - P_r khat_r */
                double pred = 0.0;
                for (int d = 0; d < K; ++d) pred += P[(int64_t)vv * K + d] * kh[d];
                e[vv] = v[(r * H + h) * (int64_t)V + vv] - pred;
              }
              if (j == M - 1) {  /* readout after row r: S_r = P_r + beta e khat^T */
                ORACLE_HAT(q, t, qh);
                const double *dOt = d_output + (t * H + h) * (int64_t)V;
                for (int d = 0; d < K; ++d) {
                  double acc = 0.0;
                  for (int vv = 0; vv < V; ++vv) acc += (P[(int64_t)vv * K + d] + b * e[vv] * kh[d]) * dOt[vv];
                  dkh[d] = scale * acc;  /* dqhat_t, staged in dkh */
                }
                if (dq) {
                  const double *qr = q + (t * H + h) * (int64_t)K;
                  double ss = 0.0, dot = 0.0;
                  for (int d = 0; d < K; ++d) ss += qr[d] * qr[d];
                  const double n = use_qk_l2norm ? sqrt(ss + ORACLE_L2_EPS) : 1.0;
                  for (int d = 0; d < K; ++d) dot += qr[d] * dkh[d];
                  for (int d = 0; d < K; ++d)
                    dq[(t * H + h) * (int64_t)K + d] = use_qk_l2norm ? dkh[d] / n - qr[d] * dot / (n * n * n) : dkh[d];
                }
                for (int vv = 0; vv < V; ++vv)
                  for (int d = 0; d < K; ++d) D[(int64_t)vv * K + d] += scale * dOt[vv] * qh[d];
              }
              /* the update S_r = P_r + beta e khat^T, reversed */
              double db = 0.0;
              for (int vv = 0; vv < V; ++vv) {
                double acc = 0.0;
                for (int d = 0; d < K; ++d) acc += D[(int64_t)vv * K + d] * kh[d];
                dl[vv] = acc;
                dvv[vv] = b * acc;
                db += e[vv] * acc;
              }
              for (int d = 0; d < K; ++d) {
                double acc = 0.0;
                for (int vv = 0; vv < V; ++vv)
                  acc += b * D[(int64_t)vv * K + d] * e[vv] - P[(int64_t)vv * K + d] * dvv[vv];
                dkh[d] = acc;
              }
              if (dbeta) dbeta[r * H + h] = db;
              if (dv)
                for (int vv = 0; vv < V; ++vv) dv[(r * H + h) * (int64_t)V + vv] = dvv[vv];
              if (dk) {
                const double *kr = k + (r * H + h) * (int64_t)K;
                double ss = 0.0, dot = 0.0;
                for (int d = 0; d < K; ++d) ss += kr[d] * kr[d];
                const double n = use_qk_l2norm ? sqrt(ss + ORACLE_L2_EPS) : 1.0;
                for (int d = 0; d < K; ++d) dot += kr[d] * dkh[d];
                for (int d = 0; d < K; ++d)
                  dk[(r * H + h) * (int64_t)K + d] = use_qk_l2norm ? dkh[d] / n - kr[d] * dot / (n * n * n) : dkh[d];
              }
              for (int vv = 0; vv < V; ++vv)
                for (int d = 0; d < K; ++d) D[(int64_t)vv * K + d] -= dvv[vv] * kh[d];
              if (j == 0) {  /* the decay S <- alpha_t S before row t*M */
                double acc = 0.0;
                for (int64_t x = 0; x < KV; ++x) acc += D[x] * P[x];
                if (dg) dg[t * H + h] = g ? acc : 0.0;
                const double a = g ? exp(g[t * H + h]) : 1.0;
                for (int64_t x = 0; x < KV; ++x) D[x] *= a;
              }
            }
          }
        }
        if (d_initial_state) memcpy(d_initial_state + (i * H + h) * KV, D, sizeof(double) * KV);
        free(ck);
#undef ORACLE_TOKEN
#undef ORACLE_HAT
      }
    }
    free(S);
    free(D);
    free(Pst);
    free(kh);
    free(qh);
    free(dkh);
    free(e);
    free(dl);
    free(dvv);
  }
  return rc;
}
