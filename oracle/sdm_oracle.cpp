// sdm_oracle.cpp -- the plain CPU oracle of the SDM forward step.
//
// TEST INFRASTRUCTURE ONLY (see sdm_oracle.h).  Deliberately naive:
// single-threaded, no blocking, no fusion, library sorts, every step in the
// order the pages give it.  Build: g++ -std=c++17 -O2 -ffp-contract=off.
//
// Page citations (title + section):
//   [SDM notes]   "Sparse Delta Memory：中文精读笔记", 2.3 (PKM addressing),
//                 2.4 (Eq. (3)-(5): decay, per-slot delta, untouched slots,
//                 read after write), 2.5 (Fig. 2 shared-residual reading).
//   [FwPKM notes] Fast-weight Product Key Memory reading notes, 2.2 (IDW).
#include "sdm_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstddef>
#include <vector>

namespace {

int resolve_k(int k_given, int n_sel, int s) {
  if (k_given > 0) return k_given;
  return n_sel < s ? n_sel : s;
}

bool shape_ok(const sdm_ref_shape* sh) {
  if (!sh) return false;
  if (sh->B < 0 || sh->H < 0 || sh->T < 0) return false;
  if (sh->n_sub < 1 || sh->d_h < 1 || sh->d_v < 1) return false;
  if (sh->W < 1 || sh->R < 1) return false;
  if (sh->score_kind != 0 && sh->score_kind != 1) return false;
  if (sh->update_form != 0 && sh->update_form != 1) return false;
  const int s = sh->n_sub;
  const int kw = resolve_k(sh->k_w, sh->W, s), kr = resolve_k(sh->k_r, sh->R, s);
  if (kw < 1 || kw > s || kr < 1 || kr > s) return false;
  // The W (R) best pairs must exist among the k x k candidates.
  if ((long long)kw * kw < sh->W || (long long)kr * kr < sh->R) return false;
  return true;
}

}  // namespace

// [SDM notes] 2.3: each branch projects two half-score vectors of length
// sqrt(N).  [FwPKM notes] 2.2: the same two vectors obtained as half-query
// against sub-key tables, with the inverse-distance score
// s_j = -log(1e-3 + |q - K_j|^2).  Computed in double, rounded once to float.
extern "C" int sdm_ref_subscores(const sdm_ref_shape* sh, const float* q,
                                 const float* K, float* S) {
  if (!shape_ok(sh) || !q || !K || !S) return -1;
  const int B = sh->B, H = sh->H, T = sh->T, s = sh->n_sub, dh = sh->d_h;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h)
      for (int t = 0; t < T; ++t)
        for (int p = 0; p < 2; ++p) {
          const size_t qrow = ((((size_t)b * H + h) * T + t) * 2 + p) * dh;
          const size_t srow = ((((size_t)b * H + h) * T + t) * 2 + p) * s;
          for (int j = 0; j < s; ++j) {
            const size_t krow = (((size_t)h * 2 + p) * s + j) * dh;
            double acc = 0.0;
            if (sh->score_kind == 0) {
              for (int c = 0; c < dh; ++c) acc += (double)q[qrow + c] * (double)K[krow + c];
              S[srow + j] = (float)acc;
            } else {
              for (int c = 0; c < dh; ++c) {
                const double d = (double)q[qrow + c] - (double)K[krow + c];
                acc += d * d;
              }
              S[srow + j] = (float)(-std::log(sh->idw_eps + acc));
            }
          }
        }
  return 0;
}

// [SDM notes] 2.3: slot (a,b) scores s_{a,b} = k'_{1,a} + k'_{2,b}; the best
// W slots are found among the k*k sums of each half's top-k, then a softmax is
// taken over the selected scores (2.2, weights k_t^(i), q_t^(i)).
// Readings: slot = a*s + b; order (score desc, index asc) at both levels;
// the candidate sum is rounded to float before ranking; no temperature.
extern "C" int sdm_ref_select(const sdm_ref_shape* sh, int which, const float* S,
                              int32_t* idx, float* score, double* wt) {
  if (!shape_ok(sh) || !S || !idx || !score || !wt) return -1;
  if (which != 0 && which != 1) return -1;
  const int B = sh->B, H = sh->H, T = sh->T, s = sh->n_sub;
  const int n_sel = which == 0 ? sh->W : sh->R;
  const int k = resolve_k(which == 0 ? sh->k_w : sh->k_r, n_sel, s);

  struct Cand {
    float c;
    int32_t slot;
  };
  std::vector<int> order(s);
  std::vector<int> top1(k), top2(k);
  std::vector<Cand> cand((size_t)k * k);

  for (size_t row = 0; row < (size_t)B * H * T; ++row) {
    const float* s1 = S + (row * 2 + 0) * s;
    const float* s2 = S + (row * 2 + 1) * s;
    // Per-half top-k by (score desc, index asc).
    for (int p = 0; p < 2; ++p) {
      const float* sp = p == 0 ? s1 : s2;
      for (int j = 0; j < s; ++j) order[j] = j;
      std::sort(order.begin(), order.end(), [sp](int x, int y) {
        if (sp[x] != sp[y]) return sp[x] > sp[y];
        return x < y;
      });
      std::vector<int>& top = p == 0 ? top1 : top2;
      for (int a = 0; a < k; ++a) top[a] = order[a];
    }
    // All k*k candidate pairs, ranked by (float sum desc, slot asc).
    size_t n = 0;
    for (int a = 0; a < k; ++a)
      for (int bb = 0; bb < k; ++bb) {
        const float c = (float)(s1[top1[a]] + s2[top2[bb]]);
        cand[n++] = Cand{c, (int32_t)(top1[a] * s + top2[bb])};
      }
    std::sort(cand.begin(), cand.begin() + n, [](const Cand& x, const Cand& y) {
      if (x.c != y.c) return x.c > y.c;
      return x.slot < y.slot;
    });
    // Softmax over the selected float sums, max subtracted, sum in rank order.
    const double mx = (double)cand[0].c;
    double tot = 0.0;
    std::vector<double> e(n_sel);
    for (int j = 0; j < n_sel; ++j) {
      e[j] = std::exp((double)cand[j].c - mx);
      tot += e[j];
    }
    for (int j = 0; j < n_sel; ++j) {
      idx[row * n_sel + j] = cand[j].slot;
      score[row * n_sel + j] = cand[j].c;
      wt[row * n_sel + j] = e[j] / tot;
    }
  }
  return 0;
}

// [SDM notes] 2.3 / 2.2 again, for a slot list chosen elsewhere: the weight
// of each listed slot is the softmax over the listed slots' float sums
// fl(S1[a] + S2[b]) (slot = a*s + b), max subtracted, sum in list order.
// Parity tests use it to give the oracle's own weights to a selection the
// device made, when that selection legitimately differs from the oracle's
// inside the score-gap tolerance.
extern "C" int sdm_ref_slot_weights(const sdm_ref_shape* sh, int which, const float* S,
                                    const int32_t* idx, double* wt) {
  if (!shape_ok(sh) || !S || !idx || !wt) return -1;
  if (which != 0 && which != 1) return -1;
  const int s = sh->n_sub;
  const int n_sel = which == 0 ? sh->W : sh->R;
  const long long N = (long long)s * s;
  std::vector<double> c(n_sel);
  for (size_t row = 0; row < (size_t)sh->B * sh->H * sh->T; ++row) {
    const float* s1 = S + (row * 2 + 0) * s;
    const float* s2 = S + (row * 2 + 1) * s;
    double mx = -INFINITY;
    for (int j = 0; j < n_sel; ++j) {
      const int32_t slot = idx[row * n_sel + j];
      if (slot < 0 || slot >= N) return -2;
      c[j] = (double)(float)(s1[slot / s] + s2[slot % s]);
      if (c[j] > mx) mx = c[j];
    }
    double tot = 0.0;
    for (int j = 0; j < n_sel; ++j) {
      c[j] = std::exp(c[j] - mx);
      tot += c[j];
    }
    for (int j = 0; j < n_sel; ++j) wt[row * n_sel + j] = c[j] / tot;
  }
  return 0;
}

// [SDM notes] 2.4, Eq. (3)-(4): for i in the write set,
//   M~[i] = alpha_t M[i];  M[i] = M~[i] + beta_t k^(i) (v_t - M~[i]);
// rows outside the write set are left exactly as they were (no global decay).
// Eq. (5): y_t = sum_{i in read set} q^(i) M_t[i], read after the write.
// update_form 1 ([SDM notes] 2.5, reading of Fig. 2): the residual is shared,
//   vhat = sum_j k^(j) M~[j];  M[i] = M~[i] + beta_t k^(i) (v_t - vhat).
// When `undo` is given, the value every written row had just before the
// write of step t is copied to undo[b,h,t,j,:] ([SDM notes] 2.9, appendix
// A.3 "backward memory": the forward pass writes in place and the backward
// pass restores earlier states by undoing the sparse writes, for O(T W d_v)
// extra memory -- i.e. a log of the W overwritten rows of every step).
static int scan_impl(const sdm_ref_shape* sh, const int32_t* idx_w, const double* wt_w,
                     const int32_t* idx_r, const double* wt_r, const float* alpha,
                     const float* beta, const float* v, double* M, double* y,
                     double* undo) {
  if (!shape_ok(sh) || !idx_w || !wt_w || !idx_r || !wt_r || !alpha || !beta ||
      !v || !M || !y)
    return -1;
  const int B = sh->B, H = sh->H, T = sh->T, W = sh->W, R = sh->R, dv = sh->d_v;
  const long long N = (long long)sh->n_sub * sh->n_sub;
  // Indices must address the table and a step's write slots must be distinct.
  for (size_t i = 0; i < (size_t)B * H * T * W; ++i)
    if (idx_w[i] < 0 || idx_w[i] >= N) return -2;
  for (size_t i = 0; i < (size_t)B * H * T * R; ++i)
    if (idx_r[i] < 0 || idx_r[i] >= N) return -2;
  for (size_t row = 0; row < (size_t)B * H * T; ++row) {
    std::vector<int32_t> ws(idx_w + row * W, idx_w + row * W + W);
    std::sort(ws.begin(), ws.end());
    if (std::adjacent_find(ws.begin(), ws.end()) != ws.end()) return -3;
  }

  std::vector<double> vhat(dv);
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) {
      double* Mc = M + ((size_t)b * H + h) * (size_t)N * dv;
      for (int t = 0; t < T; ++t) {
        const size_t row = ((size_t)b * H + h) * T + t;
        const double a = alpha[row], be = beta[row];
        const float* vt = v + row * dv;
        if (undo) {
          for (int j = 0; j < W; ++j) {
            const double* m = Mc + (size_t)idx_w[row * W + j] * dv;
            double* u = undo + (row * W + j) * (size_t)dv;
            for (int col = 0; col < dv; ++col) u[col] = m[col];
          }
        }
        if (sh->update_form == 0) {
          for (int j = 0; j < W; ++j) {
            double* m = Mc + (size_t)idx_w[row * W + j] * dv;
            const double c = be * wt_w[row * W + j];
            for (int col = 0; col < dv; ++col) {
              const double mt = a * m[col];
              m[col] = mt + c * ((double)vt[col] - mt);
            }
          }
        } else {
          for (int col = 0; col < dv; ++col) vhat[col] = 0.0;
          for (int j = 0; j < W; ++j) {
            const double* m = Mc + (size_t)idx_w[row * W + j] * dv;
            for (int col = 0; col < dv; ++col) vhat[col] += wt_w[row * W + j] * (a * m[col]);
          }
          for (int j = 0; j < W; ++j) {
            double* m = Mc + (size_t)idx_w[row * W + j] * dv;
            const double c = be * wt_w[row * W + j];
            for (int col = 0; col < dv; ++col) {
              const double mt = a * m[col];
              m[col] = mt + c * ((double)vt[col] - vhat[col]);
            }
          }
        }
        double* yt = y + row * dv;
        for (int col = 0; col < dv; ++col) yt[col] = 0.0;
        for (int j = 0; j < R; ++j) {
          const double* m = Mc + (size_t)idx_r[row * R + j] * dv;
          const double q = wt_r[row * R + j];
          for (int col = 0; col < dv; ++col) yt[col] += q * m[col];
        }
      }
    }
  return 0;
}

extern "C" int sdm_ref_scan(const sdm_ref_shape* sh, const int32_t* idx_w,
                            const double* wt_w, const int32_t* idx_r,
                            const double* wt_r, const float* alpha,
                            const float* beta, const float* v, double* M,
                            double* y) {
  return scan_impl(sh, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y, nullptr);
}

extern "C" int sdm_ref_scan_logged(const sdm_ref_shape* sh, const int32_t* idx_w,
                                   const double* wt_w, const int32_t* idx_r,
                                   const double* wt_r, const float* alpha,
                                   const float* beta, const float* v, double* M,
                                   double* y, double* undo) {
  if (!undo) return -1;
  return scan_impl(sh, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y, undo);
}

// Undo a segment ([SDM notes] 2.9, A.3): walk the steps backwards and put
// every logged row back; a row written at several steps ends with the copy
// of its earliest write, i.e. the value it had before the segment.
extern "C" int sdm_ref_undo(const sdm_ref_shape* sh, const int32_t* idx_w,
                            const double* undo, double* M) {
  if (!shape_ok(sh) || !idx_w || !undo || !M) return -1;
  const int B = sh->B, H = sh->H, T = sh->T, W = sh->W, dv = sh->d_v;
  const long long N = (long long)sh->n_sub * sh->n_sub;
  for (size_t i = 0; i < (size_t)B * H * T * W; ++i)
    if (idx_w[i] < 0 || idx_w[i] >= N) return -2;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) {
      double* Mc = M + ((size_t)b * H + h) * (size_t)N * dv;
      for (int t = T - 1; t >= 0; --t) {
        const size_t row = ((size_t)b * H + h) * T + t;
        for (int j = 0; j < W; ++j) {
          double* m = Mc + (size_t)idx_w[row * W + j] * dv;
          const double* u = undo + (row * W + j) * (size_t)dv;
          for (int col = 0; col < dv; ++col) m[col] = u[col];
        }
      }
    }
  return 0;
}

// [SDM notes] 2.4, after Eq. (5): each head's read result goes through an
// RMS-Norm and an element-wise output gate (the head-mixing projection W_o
// that follows is not part of this step).  RMSNorm(y) = y / sqrt(mean(y^2)
// + eps) times a per-head learned scale gamma[h,:]; the gate g is applied as
// given.
extern "C" int sdm_ref_rmsnorm_gate(const sdm_ref_shape* sh, const double* y,
                                    const float* g, const float* gamma, double eps,
                                    double* out) {
  if (!shape_ok(sh) || !y || !g || !out || !(eps > 0.0)) return -1;
  const int H = sh->H, T = sh->T, dv = sh->d_v;
  for (size_t row = 0; row < (size_t)sh->B * H * T; ++row) {
    const int h = (int)((row / T) % H);
    const double* yr = y + row * dv;
    double ss = 0.0;
    for (int c = 0; c < dv; ++c) ss += yr[c] * yr[c];
    const double inv = 1.0 / std::sqrt(ss / dv + eps);
    for (int c = 0; c < dv; ++c) {
      const double sc = gamma ? (double)gamma[(size_t)h * dv + c] : 1.0;
      out[row * dv + c] = yr[c] * inv * sc * (double)g[row * dv + c];
    }
  }
  return 0;
}

extern "C" int sdm_ref_forward(const sdm_ref_shape* sh, const float* q_w,
                               const float* q_r, const float* K,
                               const float* alpha, const float* beta,
                               const float* v, double* M, double* y,
                               int32_t* idx_w, double* wt_w, int32_t* idx_r,
                               double* wt_r) {
  if (!shape_ok(sh) || !q_w || !q_r || !K || !idx_w || !wt_w || !idx_r || !wt_r)
    return -1;
  const size_t rows = (size_t)sh->B * sh->H * sh->T;
  std::vector<float> S(rows * 2 * sh->n_sub);
  std::vector<float> sc_w(rows * sh->W), sc_r(rows * sh->R);
  int rc = sdm_ref_subscores(sh, q_w, K, S.data());
  if (rc) return rc;
  rc = sdm_ref_select(sh, 0, S.data(), idx_w, sc_w.data(), wt_w);
  if (rc) return rc;
  rc = sdm_ref_subscores(sh, q_r, K, S.data());
  if (rc) return rc;
  rc = sdm_ref_select(sh, 1, S.data(), idx_r, sc_r.data(), wt_r);
  if (rc) return rc;
  return sdm_ref_scan(sh, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y);
}
