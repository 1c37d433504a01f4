/*
 * fp64 CPU oracle for causal linear attention with a per-head scalar decay.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What is computed (the definition, evaluated exactly as written):
 *
 *     S_t = lambda * S_{t-1} + k_t v_t^T          (S_{-1} = init, or 0)
 *     o_t = S_t^T q_t
 *
 * i.e. o_t = sum_{s<=t} lambda^{t-s} (q_t . k_s) v_s  +  lambda^{t+1} init^T q_t.
 * S is d_k x d_v ("memory state whose size does not depend on the sequence
 * length": LASP-2 page, abstract).  lambda = 1 is plain linear attention.
 *
 * Sources on the pages:
 *   - right-product-first evaluation, length-independent memory state:
 *     "LASP-2: Rethinking Sequence Parallelism for Linear Attention and Its
 *     Hybrid", abstract;
 *   - ordinary (masked) attention inside a block, linear-attention kernel
 *     trick between blocks: same page, related-paper entry "Lightning
 *     Attention-2";
 *   - the state that precedes a segment is what each rank needs to start:
 *     "ZeCO: Zero Communication Overhead Sequence Parallelism for Linear
 *     Attention", abstract (All-Scan).
 * The pages never print the formula itself; the recurrence above is the
 * plainest reading of "right-product-first" linear attention with a scalar
 * per-head decay.
 *
 * Layout of every sequence tensor: [BH][T][d] row-major, double.
 * States: [BH][d_k][d_v] row-major (row index = key dimension).
 * lam: [BH] decay per (batch, head) sequence, or NULL for lambda = 1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef int64_t i64;

static double lam_of(const double *lam, i64 bh) { return lam ? lam[bh] : 1.0; }

static double powi(double x, i64 n) {
  double r = 1.0;
  for (i64 i = 0; i < n; ++i) r *= x;
  return r;
}

/* ---------------------------------------------------------------------- */
/* Forward, recurrent form (the definition).                               */
/* chunk > 0 and chunk_states != NULL: emits the state entering every chunk */
/* (exclusive: chunk 0 gets init).  final_state: the state after token T-1. */
/* ---------------------------------------------------------------------- */
void oracle_fwd_recurrent(i64 BH, i64 T, i64 dk, i64 dv, const double *lam,
                          const double *q, const double *k, const double *v,
                          const double *init, i64 chunk, double *o,
                          double *chunk_states, double *final_state) {
  const i64 nchunk = chunk > 0 ? (T + chunk - 1) / chunk : 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 bh = 0; bh < BH; ++bh) {
    double *S = calloc((size_t)(dk * dv), sizeof(double));
    if (init) memcpy(S, init + bh * dk * dv, sizeof(double) * dk * dv);
    const double l = lam_of(lam, bh);
    for (i64 t = 0; t < T; ++t) {
      if (chunk_states && chunk > 0 && t % chunk == 0)
        memcpy(chunk_states + (bh * nchunk + t / chunk) * dk * dv, S,
               sizeof(double) * dk * dv);
      const double *qt = q + (bh * T + t) * dk;
      const double *kt = k + (bh * T + t) * dk;
      const double *vt = v + (bh * T + t) * dv;
      double *ot = o + (bh * T + t) * dv;
      for (i64 a = 0; a < dk; ++a)
        for (i64 b = 0; b < dv; ++b)
          S[a * dv + b] = l * S[a * dv + b] + kt[a] * vt[b];
      for (i64 b = 0; b < dv; ++b) {
        double acc = 0.0;
        for (i64 a = 0; a < dk; ++a) acc += S[a * dv + b] * qt[a];
        ot[b] = acc;
      }
    }
    if (final_state) memcpy(final_state + bh * dk * dv, S, sizeof(double) * dk * dv);
    free(S);
  }
}

/* ---------------------------------------------------------------------- */
/* Backward, recurrent form.  With S_t the inclusive forward state and      */
/* R_t = sum_{u>=t} lambda^{u-t} q_u dO_u^T the inclusive reverse state:    */
/*   dq_t = S_t dO_t,   dk_t = R_t v_t,   dv_t = R_t^T k_t,                  */
/*   d_init = lambda * R_0  (= sum_t lambda^{t+1} q_t dO_t^T).              */
/* These follow from o_t being linear in every one of q_t, k_s, v_s.        */
/* ---------------------------------------------------------------------- */
void oracle_bwd_recurrent(i64 BH, i64 T, i64 dk, i64 dv, const double *lam,
                          const double *q, const double *k, const double *v,
                          const double *dO, const double *init, const double *d_final,
                          double *dq, double *dkk, double *dvv, double *d_init) {
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 bh = 0; bh < BH; ++bh) {
    double *S = calloc((size_t)(dk * dv), sizeof(double));
    const double l = lam_of(lam, bh);
    if (init) memcpy(S, init + bh * dk * dv, sizeof(double) * dk * dv);
    for (i64 t = 0; t < T; ++t) {
      const double *kt = k + (bh * T + t) * dk;
      const double *vt = v + (bh * T + t) * dv;
      const double *gt = dO + (bh * T + t) * dv;
      double *dqt = dq + (bh * T + t) * dk;
      for (i64 a = 0; a < dk; ++a) {
        double acc = 0.0;
        for (i64 b = 0; b < dv; ++b) {
          S[a * dv + b] = l * S[a * dv + b] + kt[a] * vt[b];
          acc += S[a * dv + b] * gt[b];
        }
        dqt[a] = acc;
      }
    }
    /* R_t = dL/dS_t = q_t dO_t^T + lambda R_{t+1}, where the term after the
     * last token is the gradient arriving at the final state (d_final, the
     * state the next segment starts from), or 0. */
    double *R = S; /* reuse the buffer */
    if (d_final) memcpy(R, d_final + bh * dk * dv, sizeof(double) * dk * dv);
    else memset(R, 0, sizeof(double) * dk * dv);
    for (i64 t = T - 1; t >= 0; --t) {
      const double *qt = q + (bh * T + t) * dk;
      const double *kt = k + (bh * T + t) * dk;
      const double *vt = v + (bh * T + t) * dv;
      const double *gt = dO + (bh * T + t) * dv;
      double *dkt = dkk + (bh * T + t) * dk;
      double *dvt = dvv + (bh * T + t) * dv;
      const double carry = (t == T - 1) ? 1.0 : l; /* d_final enters undecayed at t = T-1 */
      for (i64 a = 0; a < dk; ++a)
        for (i64 b = 0; b < dv; ++b)
          R[a * dv + b] = carry * R[a * dv + b] + qt[a] * gt[b];
      for (i64 a = 0; a < dk; ++a) {
        double acc = 0.0;
        for (i64 b = 0; b < dv; ++b) acc += R[a * dv + b] * vt[b];
        dkt[a] = acc;
      }
      for (i64 b = 0; b < dv; ++b) {
        double acc = 0.0;
        for (i64 a = 0; a < dk; ++a) acc += R[a * dv + b] * kt[a];
        dvt[b] = acc;
      }
    }
    /* dL/d(init) = lambda R_0; with no tokens the initial state is the final one */
    if (d_init)
      for (i64 i = 0; i < dk * dv; ++i) d_init[bh * dk * dv + i] = (T > 0 ? l : 1.0) * R[i];
    free(S);
  }
}

/* ---------------------------------------------------------------------- */
/* Forward, chunked form (any chunk length C >= 1, ragged last chunk).      */
/* Per chunk, in the pages' order: ordinary masked attention inside the     */
/* chunk, the kernel trick (query times the state) across chunks, then the  */
/* state update with the chunk's keys and values.                           */
/*   o_i = sum_{j<=i} lambda^{i-j} (q_i.k_j) v_j + lambda^{i+1} S^T q_i     */
/*   S  <- lambda^n S + sum_j lambda^{n-1-j} k_j v_j^T      (n = chunk len) */
/* ---------------------------------------------------------------------- */
void oracle_fwd_chunked(i64 BH, i64 T, i64 dk, i64 dv, const double *lam, i64 C,
                        const double *q, const double *k, const double *v,
                        const double *init, double *o, double *chunk_states,
                        double *final_state) {
  const i64 nchunk = (T + C - 1) / C;
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 bh = 0; bh < BH; ++bh) {
    double *S = calloc((size_t)(dk * dv), sizeof(double));
    if (init) memcpy(S, init + bh * dk * dv, sizeof(double) * dk * dv);
    const double l = lam_of(lam, bh);
    for (i64 c = 0; c < nchunk; ++c) {
      const i64 c0 = c * C;
      const i64 n = (T - c0) < C ? (T - c0) : C;
      if (chunk_states)
        memcpy(chunk_states + (bh * nchunk + c) * dk * dv, S, sizeof(double) * dk * dv);
      for (i64 i = 0; i < n; ++i) {
        const double *qi = q + (bh * T + c0 + i) * dk;
        double *oi = o + (bh * T + c0 + i) * dv;
        /* inter-chunk: lambda^{i+1} S^T q_i */
        const double li = powi(l, i + 1);
        for (i64 b = 0; b < dv; ++b) {
          double acc = 0.0;
          for (i64 a = 0; a < dk; ++a) acc += S[a * dv + b] * qi[a];
          oi[b] = li * acc;
        }
        /* intra-chunk: masked scores times values */
        for (i64 j = 0; j <= i; ++j) {
          const double *kj = k + (bh * T + c0 + j) * dk;
          const double *vj = v + (bh * T + c0 + j) * dv;
          double s = 0.0;
          for (i64 a = 0; a < dk; ++a) s += qi[a] * kj[a];
          s *= powi(l, i - j);
          for (i64 b = 0; b < dv; ++b) oi[b] += s * vj[b];
        }
      }
      /* state update */
      const double ln = powi(l, n);
      for (i64 a = 0; a < dk * dv; ++a) S[a] *= ln;
      for (i64 j = 0; j < n; ++j) {
        const double *kj = k + (bh * T + c0 + j) * dk;
        const double *vj = v + (bh * T + c0 + j) * dv;
        const double w = powi(l, n - 1 - j);
        for (i64 a = 0; a < dk; ++a)
          for (i64 b = 0; b < dv; ++b) S[a * dv + b] += w * kj[a] * vj[b];
      }
    }
    if (final_state) memcpy(final_state + bh * dk * dv, S, sizeof(double) * dk * dv);
    free(S);
  }
}

/* ---------------------------------------------------------------------- */
/* Backward, chunked form (any C).  S_prev = state entering the chunk,      */
/* Rbar = sum_{u > chunk end} lambda^{u - end} q_u dO_u^T (zero after the   */
/* last chunk).  For a chunk of n tokens, local indices i, j:               */
/*   dq_i = sum_{j<=i} lambda^{i-j} (dO_i.v_j) k_j + lambda^{i+1} S_prev dO_i */
/*   dk_j = sum_{i>=j} lambda^{i-j} (dO_i.v_j) q_i + lambda^{n-1-j} Rbar v_j   */
/*   dv_j = sum_{i>=j} lambda^{i-j} (q_i.k_j) dO_i + lambda^{n-1-j} Rbar^T k_j */
/*   Rbar <- lambda^n Rbar + sum_i lambda^{i+1} q_i dO_i^T                   */
/* d_init is Rbar after the first chunk has been processed.                 */
/* ---------------------------------------------------------------------- */
void oracle_bwd_chunked(i64 BH, i64 T, i64 dk, i64 dv, const double *lam, i64 C,
                        const double *q, const double *k, const double *v,
                        const double *dO, const double *init, double *dq,
                        double *dkk, double *dvv, double *d_init) {
  const i64 nchunk = (T + C - 1) / C;
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 bh = 0; bh < BH; ++bh) {
    const double l = lam_of(lam, bh);
    /* forward pass: states entering each chunk */
    double *Sprev = calloc((size_t)(nchunk * dk * dv), sizeof(double));
    double *S = calloc((size_t)(dk * dv), sizeof(double));
    if (init) memcpy(S, init + bh * dk * dv, sizeof(double) * dk * dv);
    for (i64 c = 0; c < nchunk; ++c) {
      const i64 c0 = c * C;
      const i64 n = (T - c0) < C ? (T - c0) : C;
      memcpy(Sprev + c * dk * dv, S, sizeof(double) * dk * dv);
      const double ln = powi(l, n);
      for (i64 a = 0; a < dk * dv; ++a) S[a] *= ln;
      for (i64 j = 0; j < n; ++j) {
        const double *kj = k + (bh * T + c0 + j) * dk;
        const double *vj = v + (bh * T + c0 + j) * dv;
        const double w = powi(l, n - 1 - j);
        for (i64 a = 0; a < dk; ++a)
          for (i64 b = 0; b < dv; ++b) S[a * dv + b] += w * kj[a] * vj[b];
      }
    }
    double *R = S;
    memset(R, 0, sizeof(double) * dk * dv);
    for (i64 c = nchunk - 1; c >= 0; --c) {
      const i64 c0 = c * C;
      const i64 n = (T - c0) < C ? (T - c0) : C;
      const double *Sp = Sprev + c * dk * dv;
      for (i64 i = 0; i < n; ++i) {
        const double *gi = dO + (bh * T + c0 + i) * dv;
        double *dqi = dq + (bh * T + c0 + i) * dk;
        const double li = powi(l, i + 1);
        for (i64 a = 0; a < dk; ++a) {
          double acc = 0.0;
          for (i64 b = 0; b < dv; ++b) acc += Sp[a * dv + b] * gi[b];
          dqi[a] = li * acc;
        }
        for (i64 j = 0; j <= i; ++j) {
          const double *kj = k + (bh * T + c0 + j) * dk;
          const double *vj = v + (bh * T + c0 + j) * dv;
          double s = 0.0;
          for (i64 b = 0; b < dv; ++b) s += gi[b] * vj[b];
          s *= powi(l, i - j);
          for (i64 a = 0; a < dk; ++a) dqi[a] += s * kj[a];
        }
      }
      for (i64 j = 0; j < n; ++j) {
        const double *kj = k + (bh * T + c0 + j) * dk;
        const double *vj = v + (bh * T + c0 + j) * dv;
        double *dkj = dkk + (bh * T + c0 + j) * dk;
        double *dvj = dvv + (bh * T + c0 + j) * dv;
        const double w = powi(l, n - 1 - j);
        for (i64 a = 0; a < dk; ++a) {
          double acc = 0.0;
          for (i64 b = 0; b < dv; ++b) acc += R[a * dv + b] * vj[b];
          dkj[a] = w * acc;
        }
        for (i64 b = 0; b < dv; ++b) {
          double acc = 0.0;
          for (i64 a = 0; a < dk; ++a) acc += R[a * dv + b] * kj[a];
          dvj[b] = w * acc;
        }
        for (i64 i = j; i < n; ++i) {
          const double *qi = q + (bh * T + c0 + i) * dk;
          const double *gi = dO + (bh * T + c0 + i) * dv;
          const double dec = powi(l, i - j);
          double sg = 0.0, sq = 0.0;
          for (i64 b = 0; b < dv; ++b) sg += gi[b] * vj[b];
          for (i64 a = 0; a < dk; ++a) sq += qi[a] * kj[a];
          for (i64 a = 0; a < dk; ++a) dkj[a] += dec * sg * qi[a];
          for (i64 b = 0; b < dv; ++b) dvj[b] += dec * sq * gi[b];
        }
      }
      const double ln = powi(l, n);
      for (i64 a = 0; a < dk * dv; ++a) R[a] *= ln;
      for (i64 i = 0; i < n; ++i) {
        const double *qi = q + (bh * T + c0 + i) * dk;
        const double *gi = dO + (bh * T + c0 + i) * dv;
        const double w = powi(l, i + 1);
        for (i64 a = 0; a < dk; ++a)
          for (i64 b = 0; b < dv; ++b) R[a * dv + b] += w * qi[a] * gi[b];
      }
    }
    if (d_init) memcpy(d_init + bh * dk * dv, R, sizeof(double) * dk * dv);
    free(S);
    free(Sprev);
  }
}

/* ---------------------------------------------------------------------- */
/* Segment-local states: U_g = sum_{s in segment g} lambda^{end_g - s} k_s v_s^T */
/* for contiguous segments of L tokens (last one may be shorter).           */
/* Output layout [G][BH][dk][dv].  This is the length-independent memory    */
/* state each sequence-parallel rank computes from its own segment.         */
/* ---------------------------------------------------------------------- */
void oracle_segment_states(i64 BH, i64 T, i64 dk, i64 dv, const double *lam, i64 L,
                           const double *k, const double *v, double *out) {
  const i64 G = (T + L - 1) / L;
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 bh = 0; bh < BH; ++bh) {
    const double l = lam_of(lam, bh);
    for (i64 g = 0; g < G; ++g) {
      double *U = out + (g * BH + bh) * dk * dv;
      memset(U, 0, sizeof(double) * dk * dv);
      const i64 s0 = g * L;
      const i64 n = (T - s0) < L ? (T - s0) : L;
      /* Horner order over the segment: U <- lambda U + k v^T */
      for (i64 s = 0; s < n; ++s) {
        const double *ks = k + (bh * T + s0 + s) * dk;
        const double *vs = v + (bh * T + s0 + s) * dv;
        for (i64 a = 0; a < dk; ++a)
          for (i64 b = 0; b < dv; ++b) U[a * dv + b] = l * U[a * dv + b] + ks[a] * vs[b];
      }
    }
  }
}

/* ---------------------------------------------------------------------- */
/* Segment-local gradient states for the backward of a split sequence:     */
/*   W_g = sum_{s in segment g} lambda^{s - start_g + 1} q_s dO_s^T,         */
/* what segment g adds to the gradient arriving at the final state of the   */
/* segment before it (the reverse counterpart of the All-Scan input).       */
/* Horner order from the segment end: W <- lambda (W + q_s dO_s^T).         */
/* ---------------------------------------------------------------------- */
void oracle_segment_grad_states(i64 BH, i64 T, i64 dk, i64 dv, const double *lam, i64 L,
                                const double *q, const double *dO, double *out) {
  const i64 G = (T + L - 1) / L;
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 bh = 0; bh < BH; ++bh) {
    const double l = lam_of(lam, bh);
    for (i64 g = 0; g < G; ++g) {
      double *W = out + (g * BH + bh) * dk * dv;
      memset(W, 0, sizeof(double) * dk * dv);
      const i64 s0 = g * L;
      const i64 n = (T - s0) < L ? (T - s0) : L;
      for (i64 s = n - 1; s >= 0; --s) {
        const double *qs = q + (bh * T + s0 + s) * dk;
        const double *gs = dO + (bh * T + s0 + s) * dv;
        for (i64 a = 0; a < dk; ++a)
          for (i64 b = 0; b < dv; ++b) W[a * dv + b] = l * (W[a * dv + b] + qs[a] * gs[b]);
      }
    }
  }
}

/* ---------------------------------------------------------------------- */
/* Exclusive prefix scan of segment states (the single-device reading of   */
/* All-Scan / the gather-then-combine of length-independent states):        */
/*   S_0 = init (or 0),  S_g = a * S_{g-1} + U_{g-1},  total = a S_{G-1} + U_{G-1} */
/* with a = seg_decay[bh] (lambda^L; NULL means 1).  Sequential in g.       */
/* ---------------------------------------------------------------------- */
void oracle_state_scan(i64 G, i64 BH, i64 dk, i64 dv, const double *seg_decay,
                       const double *local, const double *init, double *out,
                       double *total) {
  const i64 D = dk * dv;
#pragma omp parallel for schedule(static)
  for (i64 bh = 0; bh < BH; ++bh) {
    const double a = seg_decay ? seg_decay[bh] : 1.0;
    double *S = calloc((size_t)D, sizeof(double));
    if (init) memcpy(S, init + bh * D, sizeof(double) * D);
    for (i64 g = 0; g < G; ++g) {
      memcpy(out + (g * BH + bh) * D, S, sizeof(double) * D);
      const double *U = local + (g * BH + bh) * D;
      for (i64 i = 0; i < D; ++i) S[i] = a * S[i] + U[i];
    }
    if (total) memcpy(total + bh * D, S, sizeof(double) * D);
    free(S);
  }
}

/* ====================================================================== */
/* Data-dependent gates: a decay per token per head (the gated variant the  */
/* LASP-2 page names beside the plain one).  With g_t = log(alpha_t) <= 0:  */
/*     S_t = alpha_t S_{t-1} + k_t v_t^T,     o_t = S_t^T q_t,                */
/* the plain definition with lambda replaced by the token's own gate.        */
/* log_gate: [BH][T].                                                       */
/* ====================================================================== */
void oracle_fwd_gated(i64 BH, i64 T, i64 dk, i64 dv, const double *log_gate, const double *q,
                      const double *k, const double *v, const double *init, double *o,
                      double *final_state) {
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 bh = 0; bh < BH; ++bh) {
    double *S = calloc((size_t)(dk * dv), sizeof(double));
    if (init) memcpy(S, init + bh * dk * dv, sizeof(double) * dk * dv);
    for (i64 t = 0; t < T; ++t) {
      const double a = exp(log_gate[bh * T + t]);
      const double *qt = q + (bh * T + t) * dk;
      const double *kt = k + (bh * T + t) * dk;
      const double *vt = v + (bh * T + t) * dv;
      double *ot = o + (bh * T + t) * dv;
      for (i64 i = 0; i < dk; ++i)
        for (i64 j = 0; j < dv; ++j) S[i * dv + j] = a * S[i * dv + j] + kt[i] * vt[j];
      for (i64 j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (i64 i = 0; i < dk; ++i) acc += S[i * dv + j] * qt[i];
        ot[j] = acc;
      }
    }
    if (final_state) memcpy(final_state + bh * dk * dv, S, sizeof(double) * dk * dv);
    free(S);
  }
}

/* Backward of oracle_fwd_gated, by the chain rule on the recurrence:       */
/*   R_t = dL/dS_t = q_t dO_t^T + alpha_{t+1} R_{t+1}   (R_T-ish = d_final)   */
/*   dq_t = S_t dO_t,  dk_t = R_t v_t,  dv_t = R_t^T k_t,                    */
/*   dL/dg_t = alpha_t <R_t, S_{t-1}>   (S_t depends on g_t only through      */
/*             alpha_t S_{t-1}),        d_init = alpha_0 R_0.                  */
/* S_{t-1} for the reverse sweep is recomputed per 64-token block from the   */
/* states kept at block starts.                                              */
void oracle_bwd_gated(i64 BH, i64 T, i64 dk, i64 dv, const double *log_gate, const double *q,
                      const double *k, const double *v, const double *dO, const double *init,
                      const double *d_final, double *dq, double *dkk, double *dvv, double *d_log_gate,
                      double *d_init) {
  const i64 D = dk * dv, NB = 64, nblk = (T + NB - 1) / NB;
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 bh = 0; bh < BH; ++bh) {
    const double *lg = log_gate + bh * T;
    double *S = calloc((size_t)D, sizeof(double));
    double *keep = calloc((size_t)((nblk + 1) * D), sizeof(double)); /* state entering each block */
    double *blk = calloc((size_t)((NB + 1) * D), sizeof(double));    /* S_{t-1} for the block's t */
    double *R = calloc((size_t)D, sizeof(double));
    if (init) memcpy(S, init + bh * D, sizeof(double) * D);
    for (i64 t = 0; t < T; ++t) {
      if (t % NB == 0) memcpy(keep + (t / NB) * D, S, sizeof(double) * D);
      const double a = exp(lg[t]);
      const double *kt = k + (bh * T + t) * dk, *vt = v + (bh * T + t) * dv, *gt = dO + (bh * T + t) * dv;
      double *dqt = dq + (bh * T + t) * dk;
      for (i64 i = 0; i < dk; ++i) {
        double acc = 0.0;
        for (i64 j = 0; j < dv; ++j) {
          S[i * dv + j] = a * S[i * dv + j] + kt[i] * vt[j];
          acc += S[i * dv + j] * gt[j];
        }
        dqt[i] = acc;
      }
    }
    if (d_final) memcpy(R, d_final + bh * D, sizeof(double) * D);
    for (i64 b = nblk - 1; b >= 0; --b) {
      const i64 t0 = b * NB, t1 = (t0 + NB < T) ? t0 + NB : T;
      /* blk[m] = S_{t0+m-1}: the state before token t0+m */
      memcpy(blk, keep + b * D, sizeof(double) * D);
      for (i64 t = t0; t < t1 - 1; ++t) {
        const double a = exp(lg[t]);
        const double *kt = k + (bh * T + t) * dk, *vt = v + (bh * T + t) * dv;
        double *prev = blk + (t - t0) * D, *next = blk + (t - t0 + 1) * D;
        for (i64 i = 0; i < dk; ++i)
          for (i64 j = 0; j < dv; ++j) next[i * dv + j] = a * prev[i * dv + j] + kt[i] * vt[j];
      }
      for (i64 t = t1 - 1; t >= t0; --t) {
        const double *qt = q + (bh * T + t) * dk, *kt = k + (bh * T + t) * dk;
        const double *vt = v + (bh * T + t) * dv, *gt = dO + (bh * T + t) * dv;
        const double carry = (t == T - 1) ? 1.0 : exp(lg[t + 1]);
        for (i64 i = 0; i < dk; ++i)
          for (i64 j = 0; j < dv; ++j) R[i * dv + j] = carry * R[i * dv + j] + qt[i] * gt[j];
        double *dkt = dkk + (bh * T + t) * dk, *dvt = dvv + (bh * T + t) * dv;
        for (i64 i = 0; i < dk; ++i) {
          double acc = 0.0;
          for (i64 j = 0; j < dv; ++j) acc += R[i * dv + j] * vt[j];
          dkt[i] = acc;
        }
        for (i64 j = 0; j < dv; ++j) {
          double acc = 0.0;
          for (i64 i = 0; i < dk; ++i) acc += R[i * dv + j] * kt[i];
          dvt[j] = acc;
        }
        if (d_log_gate) {
          const double *sp = blk + (t - t0) * D;
          double acc = 0.0;
          for (i64 x = 0; x < D; ++x) acc += R[x] * sp[x];
          d_log_gate[bh * T + t] = exp(lg[t]) * acc;
        }
      }
    }
    if (d_init)
      for (i64 x = 0; x < D; ++x) d_init[bh * D + x] = (T > 0 ? exp(lg[0]) : 1.0) * R[x];
    free(S);
    free(keep);
    free(blk);
    free(R);
  }
}

/* ====================================================================== */
/* Per-dimension gates (the vector form of the data-dependent gate, as in   */
/* "Gated Linear Attention ..." on the LASP-2 page's related list): one      */
/* decay per token, head and key dimension, g_t[i] = log(alpha_t[i]) <= 0:  */
/*     S_t = diag(alpha_t) S_{t-1} + k_t v_t^T,     o_t = S_t^T q_t.        */
/* log_gate: [BH][T][dk].                                                   */
/* ====================================================================== */
void oracle_fwd_gated_vec(i64 BH, i64 T, i64 dk, i64 dv, const double *log_gate, const double *q,
                          const double *k, const double *v, const double *init, double *o,
                          double *final_state) {
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 bh = 0; bh < BH; ++bh) {
    double *S = calloc((size_t)(dk * dv), sizeof(double));
    if (init) memcpy(S, init + bh * dk * dv, sizeof(double) * dk * dv);
    for (i64 t = 0; t < T; ++t) {
      const double *g = log_gate + (bh * T + t) * dk;
      const double *qt = q + (bh * T + t) * dk;
      const double *kt = k + (bh * T + t) * dk;
      const double *vt = v + (bh * T + t) * dv;
      double *ot = o + (bh * T + t) * dv;
      for (i64 i = 0; i < dk; ++i) {
        const double a = exp(g[i]);
        for (i64 j = 0; j < dv; ++j) S[i * dv + j] = a * S[i * dv + j] + kt[i] * vt[j];
      }
      for (i64 j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (i64 i = 0; i < dk; ++i) acc += S[i * dv + j] * qt[i];
        ot[j] = acc;
      }
    }
    if (final_state) memcpy(final_state + bh * dk * dv, S, sizeof(double) * dk * dv);
    free(S);
  }
}

/* Backward of oracle_fwd_gated_vec, the chain rule on the recurrence row by */
/* row:  R_t = q_t dO_t^T + diag(alpha_{t+1}) R_{t+1}   (starting at d_final) */
/*   dq_t = S_t dO_t,  dk_t = R_t v_t,  dv_t = R_t^T k_t,                    */
/*   dL/dg_t[i] = alpha_t[i] sum_j R_t[i][j] S_{t-1}[i][j],                   */
/*   d_init = diag(alpha_0) R_0.   S_{t-1} recomputed per 64-token block.      */
void oracle_bwd_gated_vec(i64 BH, i64 T, i64 dk, i64 dv, const double *log_gate, const double *q,
                          const double *k, const double *v, const double *dO, const double *init,
                          const double *d_final, double *dq, double *dkk, double *dvv, double *d_log_gate,
                          double *d_init) {
  const i64 D = dk * dv, NB = 64, nblk = (T + NB - 1) / NB;
#pragma omp parallel for schedule(dynamic, 1)
  for (i64 bh = 0; bh < BH; ++bh) {
    const double *lg = log_gate + bh * T * dk;
    double *S = calloc((size_t)D, sizeof(double));
    double *keep = calloc((size_t)((nblk + 1) * D), sizeof(double));
    double *blk = calloc((size_t)((NB + 1) * D), sizeof(double));
    double *R = calloc((size_t)D, sizeof(double));
    if (init) memcpy(S, init + bh * D, sizeof(double) * D);
    for (i64 t = 0; t < T; ++t) {
      if (t % NB == 0) memcpy(keep + (t / NB) * D, S, sizeof(double) * D);
      const double *kt = k + (bh * T + t) * dk, *vt = v + (bh * T + t) * dv, *gt = dO + (bh * T + t) * dv;
      double *dqt = dq + (bh * T + t) * dk;
      for (i64 i = 0; i < dk; ++i) {
        const double a = exp(lg[t * dk + i]);
        double acc = 0.0;
        for (i64 j = 0; j < dv; ++j) {
          S[i * dv + j] = a * S[i * dv + j] + kt[i] * vt[j];
          acc += S[i * dv + j] * gt[j];
        }
        dqt[i] = acc;
      }
    }
    if (d_final) memcpy(R, d_final + bh * D, sizeof(double) * D);
    for (i64 b = nblk - 1; b >= 0; --b) {
      const i64 t0 = b * NB, t1 = (t0 + NB < T) ? t0 + NB : T;
      memcpy(blk, keep + b * D, sizeof(double) * D);
      for (i64 t = t0; t < t1 - 1; ++t) {
        const double *kt = k + (bh * T + t) * dk, *vt = v + (bh * T + t) * dv;
        double *prev = blk + (t - t0) * D, *next = blk + (t - t0 + 1) * D;
        for (i64 i = 0; i < dk; ++i) {
          const double a = exp(lg[t * dk + i]);
          for (i64 j = 0; j < dv; ++j) next[i * dv + j] = a * prev[i * dv + j] + kt[i] * vt[j];
        }
      }
      for (i64 t = t1 - 1; t >= t0; --t) {
        const double *qt = q + (bh * T + t) * dk, *kt = k + (bh * T + t) * dk;
        const double *vt = v + (bh * T + t) * dv, *gt = dO + (bh * T + t) * dv;
        for (i64 i = 0; i < dk; ++i) {
          const double carry = (t == T - 1) ? 1.0 : exp(lg[(t + 1) * dk + i]);
          for (i64 j = 0; j < dv; ++j) R[i * dv + j] = carry * R[i * dv + j] + qt[i] * gt[j];
        }
        double *dkt = dkk + (bh * T + t) * dk, *dvt = dvv + (bh * T + t) * dv;
        for (i64 i = 0; i < dk; ++i) {
          double acc = 0.0;
          for (i64 j = 0; j < dv; ++j) acc += R[i * dv + j] * vt[j];
          dkt[i] = acc;
        }
        for (i64 j = 0; j < dv; ++j) {
          double acc = 0.0;
          for (i64 i = 0; i < dk; ++i) acc += R[i * dv + j] * kt[i];
          dvt[j] = acc;
        }
        if (d_log_gate) {
          const double *sp = blk + (t - t0) * D;
          for (i64 i = 0; i < dk; ++i) {
            double acc = 0.0;
            for (i64 j = 0; j < dv; ++j) acc += R[i * dv + j] * sp[i * dv + j];
            d_log_gate[(bh * T + t) * dk + i] = exp(lg[t * dk + i]) * acc;
          }
        }
      }
    }
    if (d_init)
      for (i64 i = 0; i < dk; ++i) {
        const double a0 = T > 0 ? exp(lg[i]) : 1.0;
        for (i64 j = 0; j < dv; ++j) d_init[bh * D + i * dv + j] = a0 * R[i * dv + j];
      }
    free(S);
    free(keep);
    free(blk);
    free(R);
  }
}
