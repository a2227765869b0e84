/*
 * sdm_oracle.h -- plain, slow, single-threaded CPU oracle for the Sparse Delta
 * Memory (SDM) forward step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA path and must never be linked into it.
 *
 * Sources (web pages, cited by title and section):
 *   [SDM notes]   "Sparse Delta Memory：中文精读笔记" (reading notes on
 *                 arXiv 2607.07386v1), sections 2.2-2.5, Eq. (3)-(5), Fig. 2.
 *   [SDM blog]    Korean blog post on SDM, section "핵심 세 가지 / 하나"
 *                 (restates Eq. (3)-(4): only selected write slots decay).
 *   [FwPKM notes] "Fast-weight Product Key Memory" reading notes, section 2.2
 *                 (product keys with inverse-distance sub-scores).
 *
 * Precision: sub-scores are computed in double and rounded once to float;
 * every selection decision (per-half order, candidate sums, final order) is
 * taken in float, the precision the device path decides in.  Softmax weights,
 * the write recurrence and the read are carried in double.
 *
 * All arrays are dense, row-major, host memory.  Functions return 0 on
 * success and a negative value on an argument error (nothing is written).
 */
#ifndef SDM_ORACLE_H
#define SDM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int B, H, T;      /* batch, heads, tokens                                   */
  int n_sub;        /* s = sqrt(N): entries per sub-key table; N = s*s         */
  int d_h;          /* half-query / sub-key dimension                          */
  int d_v;          /* value (row) width                                       */
  int W, R;         /* write / read slots per token and head                   */
  int k_w, k_r;     /* per-half top-k; 0 means min(W, s) / min(R, s)           */
  int score_kind;   /* 0: dot product; 1: inverse distance -log(eps+|q-K|^2)   */
  double idw_eps;   /* eps of the inverse-distance score (1e-3 on the page)    */
  int update_form;  /* 0: per-slot Eq. (4); 1: shared residual read off Fig. 2 */
} sdm_ref_shape;

/* Sub-scores of one selection (write or read).
 * q: [B,H,T,2,d_h] half-queries; K: [H,2,s,d_h] sub-key tables (one pair per
 * head, shared by the write and the read selection).
 * S: [B,H,T,2,s] out, S[..,p,j] = <q_p, K_p[j]>  or  -ln(eps + |q_p - K_p[j]|^2). */
int sdm_ref_subscores(const sdm_ref_shape* sh, const float* q, const float* K,
                      float* S);

/* Product-key selection of one branch (which = 0: write, W and k_w;
 * which = 1: read, R and k_r) from float sub-scores S [B,H,T,2,s].
 * idx: [B,H,T,n_sel] slot = a*s + b in rank order (score desc, slot asc);
 * score: [B,H,T,n_sel] the float candidate sums fl(S1[a] + S2[b]);
 * wt: [B,H,T,n_sel] softmax of the selected sums (double). */
int sdm_ref_select(const sdm_ref_shape* sh, int which, const float* S,
                   int32_t* idx, float* score, double* wt);

/* Softmax weights of a given slot list: idx [B,H,T,n_sel] (n_sel = W for
 * which = 0, R for which = 1; slots in any order) against float sub-scores
 * S [B,H,T,2,s]; wt [B,H,T,n_sel] (double) is the softmax of the listed
 * slots' float sums fl(S1[a] + S2[b]).  Returns -2 for a slot outside [0, N). */
int sdm_ref_slot_weights(const sdm_ref_shape* sh, int which, const float* S,
                         const int32_t* idx, double* wt);

/* The write-then-read recurrence, sequential in t, for every (b,h) chain.
 * idx_w/wt_w: [B,H,T,W]; idx_r/wt_r: [B,H,T,R]; alpha, beta: [B,H,T];
 * v: [B,H,T,d_v]; M: [B,H,N,d_v] in/out (double); y: [B,H,T,d_v] out. */
int sdm_ref_scan(const sdm_ref_shape* sh,
                 const int32_t* idx_w, const double* wt_w,
                 const int32_t* idx_r, const double* wt_r,
                 const float* alpha, const float* beta, const float* v,
                 double* M, double* y);

/* sdm_ref_scan that also logs, before each step's write, the value of every
 * row it writes: undo [B,H,T,W,d_v] out (double), undo[b,h,t,j,:] =
 * M_{t-1}[idx_w[b,h,t,j], :]. */
int sdm_ref_scan_logged(const sdm_ref_shape* sh,
                        const int32_t* idx_w, const double* wt_w,
                        const int32_t* idx_r, const double* wt_r,
                        const float* alpha, const float* beta, const float* v,
                        double* M, double* y, double* undo);

/* Restore M [B,H,N,d_v] (in/out, double) to its value before a logged
 * segment: steps T-1 down to 0 put their logged rows back. */
int sdm_ref_undo(const sdm_ref_shape* sh, const int32_t* idx_w,
                 const double* undo, double* M);

/* Per-head RMS-Norm and element-wise output gate on the read result:
 * out = y / sqrt(mean_c y^2 + eps) * gamma[h,:] * g.  y, out: [B,H,T,d_v]
 * (double); g: [B,H,T,d_v] float; gamma: [H,d_v] float or NULL (ones). */
int sdm_ref_rmsnorm_gate(const sdm_ref_shape* sh, const double* y, const float* g,
                         const float* gamma, double eps, double* out);

/* Sub-scores, both selections and the scan, in that order.  The selected
 * indices and weights are returned too (none of the idx and wt outputs may be NULL). */
int sdm_ref_forward(const sdm_ref_shape* sh,
                    const float* q_w, const float* q_r, const float* K,
                    const float* alpha, const float* beta, const float* v,
                    double* M, double* y,
                    int32_t* idx_w, double* wt_w, int32_t* idx_r, double* wt_r);

#ifdef __cplusplus
}
#endif
#endif /* SDM_ORACLE_H */
