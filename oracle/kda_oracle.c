/*
 * kda_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU oracle of the Kimi Delta Attention (KDA) recurrent
 * state path served under speculative decoding and hybrid prefix caching.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this file's library; the product path never does.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * The recurrence (a gated delta rule with per-channel decay).  The pages name
 * KDA but print no equation ("Kimi K3 stresses the whole stack" and "Confirmed"
 * on the vLLM Kimi K3 pages), so the reading used everywhere is
 *
 *     S_t = (I - beta_t k_t k_t^T) . Diag(alpha_t) . S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * with S a d_k x d_v matrix, alpha_t in R^{d_k} acting on the key (row) index,
 * beta_t a scalar, and o_t read from the post-update state.  No 1/sqrt(d_k)
 * scaling of q and no normalisation of k happen inside the path.
 *
 * Layout used by this file only: S is row-major, S[c * d_v + j], c the key
 * channel and j the value channel.  Packed token tensors are [N][H][d] with
 * beta [N][H]; cu_seqlens[B + 1] delimits sequence i as [cu[i], cu[i+1]).
 * States for sequence i, head h are at S + (i * H + h) * d_k * d_v.
 *
 * Every function below evaluates the formula as written, in fp64, token by
 * token; the only regrouping is (I - b k k^T) M = M - b k (k^T M), which is
 * associativity of the matrix product.  Build without fast-math and with
 * floating-point contraction off so x86 and Arm give identical bits.
 *
 * Each routine loops over (sequence, head) units with OpenMP when it is
 * available; units are independent, so the thread count does not change any
 * result.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One token of the recurrence on one (sequence, head) state.
 * S (d_k x d_v) is updated in place; o (d_v) receives S_t^T q when non-NULL.
 * work must hold d_k * d_v + d_v doubles. */
static void kdao_token(int dk, int dv, double *S, const double *q,
                       const double *k, const double *v, const double *alpha,
                       double beta, double *o, double *work) {
  double *M = work;            /* M = Diag(alpha) S          */
  double *kM = work + dk * dv; /* kM = k^T M  (a row vector) */
  for (int c = 0; c < dk; ++c)
    for (int j = 0; j < dv; ++j) M[c * dv + j] = alpha[c] * S[c * dv + j];
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int c = 0; c < dk; ++c) acc += k[c] * M[c * dv + j];
    kM[j] = acc;
  }
  /* S_t = M - beta k (k^T M) + beta k v^T */
  for (int c = 0; c < dk; ++c)
    for (int j = 0; j < dv; ++j)
      S[c * dv + j] = M[c * dv + j] - beta * k[c] * kM[j] + beta * k[c] * v[j];
  if (o) {
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int c = 0; c < dk; ++c) acc += S[c * dv + j] * q[c];
      o[j] = acc;
    }
  }
}

int kdao_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void kdao_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Single token, single state: the bare recurrence, for the closed-form pins. */
void kdao_step(int dk, int dv, double *S, const double *q, const double *k,
               const double *v, const double *alpha, double beta, double *o) {
  double *work = (double *)malloc(sizeof(double) * (size_t)(dk * dv + dv));
  kdao_token(dk, dv, S, q, k, v, alpha, beta, o, work);
  free(work);
}

/*
 * Prefill with in-pass checkpoints ("KDA checkpoints stay inside the prefill":
 * the recurrent-state checkpoint is exported during the original prefill pass).
 *
 * For sequence i, head h: start from S_in, run every token of the segment in
 * order, write o_t, and after the token at absolute position p (1-based count
 * of tokens in the sequence, p = start_pos[i] + local index + 1) with
 * p % ckpt_every == 0, copy the state into the next checkpoint entry of that
 * sequence: ckpt[(i * max_ckpt + m) * H + h], m = 0, 1, ...  Checkpoints past
 * max_ckpt are dropped and counted in n_ckpt[i] anyway.  ckpt_every <= 0
 * disables checkpoints.  The final state goes to S_out (may alias S_in).
 * start_pos may be NULL (all zero).
 */
void kdao_prefill(int B, int H, int dk, int dv, const int32_t *cu_seqlens,
                  const double *q, const double *k, const double *v,
                  const double *alpha, const double *beta, const double *S_in,
                  double *S_out, double *o, const int32_t *start_pos,
                  int ckpt_every, int max_ckpt, double *ckpt, int32_t *n_ckpt) {
  const size_t sd = (size_t)dk * dv;
  if (n_ckpt)
    for (int i = 0; i < B; ++i) n_ckpt[i] = 0;
#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
#endif
  for (int i = 0; i < B; ++i) {
    for (int h = 0; h < H; ++h) {
      double *S = (double *)malloc(sizeof(double) * sd);
      double *work = (double *)malloc(sizeof(double) * (sd + dv));
      memcpy(S, S_in + ((size_t)i * H + h) * sd, sizeof(double) * sd);
      const int p0 = start_pos ? start_pos[i] : 0;
      int m = 0;
      for (int t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
        const size_t r = (size_t)t * H + h;
        kdao_token(dk, dv, S, q + r * dk, k + r * dk, v + r * dv,
                   alpha + r * dk, beta[r], o ? o + r * dv : NULL, work);
        const int p = p0 + (t - cu_seqlens[i]) + 1;
        if (ckpt_every > 0 && p % ckpt_every == 0) {
          if (ckpt && m < max_ckpt)
            memcpy(ckpt + (((size_t)i * max_ckpt + m) * H + h) * sd, S,
                   sizeof(double) * sd);
          ++m;
        }
      }
      if (n_ckpt && h == 0) n_ckpt[i] = m;
      memcpy(S_out + ((size_t)i * H + h) * sd, S, sizeof(double) * sd);
      free(work);
      free(S);
    }
  }
}

/*
 * Draft verification ("ReplaySSM shrinks rollback state"): the target runs the
 * recurrence over the drafted positions to produce their outputs, but the
 * committed state is not changed.  For every sequence the segment's tokens are
 * run on a copy of S; o receives every position's output.
 */
void kdao_verify(int B, int H, int dk, int dv, const int32_t *cu_seqlens,
                 const double *q, const double *k, const double *v,
                 const double *alpha, const double *beta, const double *S,
                 double *o) {
  const size_t sd = (size_t)dk * dv;
#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
#endif
  for (int i = 0; i < B; ++i) {
    for (int h = 0; h < H; ++h) {
      double *W = (double *)malloc(sizeof(double) * sd);
      double *work = (double *)malloc(sizeof(double) * (sd + dv));
      memcpy(W, S + ((size_t)i * H + h) * sd, sizeof(double) * sd);
      for (int t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
        const size_t r = (size_t)t * H + h;
        kdao_token(dk, dv, W, q + r * dk, k + r * dk, v + r * dv,
                   alpha + r * dk, beta[r], o + r * dv, work);
      }
      free(work);
      free(W);
    }
  }
}

/*
 * Commit ("Rejecting a draft only moves the buffer pointer"; the accepted state
 * is reconstructed at commit time): the committed state becomes the state after
 * the first accepted_len[i] tokens of sequence i's segment.  accepted_len[i] = 0
 * leaves S untouched.  Values outside [0, segment length] are clamped into it.
 */
void kdao_commit(int B, int H, int dk, int dv, const int32_t *cu_seqlens,
                 const double *q, const double *k, const double *v,
                 const double *alpha, const double *beta,
                 const int32_t *accepted_len, double *S) {
  const size_t sd = (size_t)dk * dv;
#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
#endif
  for (int i = 0; i < B; ++i) {
    for (int h = 0; h < H; ++h) {
      double *work = (double *)malloc(sizeof(double) * (sd + dv));
      double *Si = S + ((size_t)i * H + h) * sd;
      int a = accepted_len[i];
      const int len = cu_seqlens[i + 1] - cu_seqlens[i];
      if (a < 0) a = 0;
      if (a > len) a = len;
      for (int t = cu_seqlens[i]; t < cu_seqlens[i] + a; ++t) {
        const size_t r = (size_t)t * H + h;
        kdao_token(dk, dv, Si, q + r * dk, k + r * dk, v + r * dv,
                   alpha + r * dk, beta[r], NULL, work);
      }
      free(work);
    }
  }
}
