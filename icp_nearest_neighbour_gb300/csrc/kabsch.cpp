// Host rigid-motion solve ("Implementing ICP with CUDA-KDTree", section 2.1):
// from the accepted pairs' centroids and cross-covariance H, the rotation that
// best maps the de-meaned source onto the de-meaned target, then the
// translation from the centroid difference.
//
// H = sum (s - mu_s)(q - mu_q)^T is factored as U S V^T with a one-sided
// (Hestenes) Jacobi SVD in double precision: plane rotations applied to the
// columns of A = H V until they are mutually orthogonal; then the column
// norms are the singular values and the normalised columns are U.  The
// rotation is R = V diag(1, 1, d) U^T with d = sign det(V U^T), which keeps R
// a proper rotation when the best orthogonal fit is a reflection (the
// Kabsch / Umeyama guard; the page itself writes R = U V^T for the transposed
// H), and t = mu_q - R mu_s.
#include <algorithm>
#include <cmath>

#include "icpnn_internal.h"

namespace icpnn {
namespace {

double det3(const double M[3][3]) {
  return M[0][0] * (M[1][1] * M[2][2] - M[1][2] * M[2][1]) -
         M[0][1] * (M[1][0] * M[2][2] - M[1][2] * M[2][0]) +
         M[0][2] * (M[1][0] * M[2][1] - M[1][1] * M[2][0]);
}

}  // namespace

int kabsch_solve(const icpnn_moments& m, double T[16]) {
  if (m.n_accepted < 3) return ICPNN_ERR_DEGENERATE;
  double A[3][3], V[3][3];
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 3; ++j) {
      A[i][j] = m.H[3 * i + j];
      V[i][j] = (i == j) ? 1.0 : 0.0;
    }
  for (int i = 0; i < 9; ++i)
    if (!std::isfinite(m.H[i])) return ICPNN_ERR_DEGENERATE;

  static const int pairs[3][2] = {{0, 1}, {0, 2}, {1, 2}};
  for (int sweep = 0; sweep < 64; ++sweep) {
    bool rotated = false;
    for (const auto& pq : pairs) {
      const int p = pq[0], q = pq[1];
      double alpha = 0, beta = 0, gamma = 0;
      for (int i = 0; i < 3; ++i) {
        alpha += A[i][p] * A[i][p];
        beta += A[i][q] * A[i][q];
        gamma += A[i][p] * A[i][q];
      }
      if (gamma == 0.0 || std::fabs(gamma) <= 1e-15 * std::sqrt(alpha * beta)) continue;
      rotated = true;
      const double zeta = (beta - alpha) / (2.0 * gamma);
      const double tn = std::copysign(1.0, zeta) / (std::fabs(zeta) + std::sqrt(1.0 + zeta * zeta));
      const double c = 1.0 / std::sqrt(1.0 + tn * tn);
      const double s = c * tn;
      for (int i = 0; i < 3; ++i) {
        const double ap = A[i][p], aq = A[i][q];
        A[i][p] = c * ap - s * aq;
        A[i][q] = s * ap + c * aq;
        const double vp = V[i][p], vq = V[i][q];
        V[i][p] = c * vp - s * vq;
        V[i][q] = s * vp + c * vq;
      }
    }
    if (!rotated) break;
  }

  // singular values = column norms; order them descending
  double sig[3];
  int ord[3] = {0, 1, 2};
  for (int j = 0; j < 3; ++j)
    sig[j] = std::sqrt(A[0][j] * A[0][j] + A[1][j] * A[1][j] + A[2][j] * A[2][j]);
  std::sort(ord, ord + 3, [&](int a, int b) { return sig[a] > sig[b]; });
  double U[3][3], Vs[3][3], s_sorted[3];
  for (int k = 0; k < 3; ++k) {
    const int j = ord[k];
    s_sorted[k] = sig[j];
    for (int i = 0; i < 3; ++i) {
      Vs[i][k] = V[i][j];
      U[i][k] = A[i][j];
    }
  }
  if (!(s_sorted[0] > 0.0) || s_sorted[1] <= 1e-12 * s_sorted[0]) return ICPNN_ERR_DEGENERATE;
  for (int k = 0; k < 2; ++k)
    for (int i = 0; i < 3; ++i) U[i][k] /= s_sorted[k];
  // third left vector from the first two (exactly orthonormal even when
  // sigma_3 is zero); flip the third right vector with it so H = U S V^T holds
  const double u3[3] = {U[1][0] * U[2][1] - U[2][0] * U[1][1],
                        U[2][0] * U[0][1] - U[0][0] * U[2][1],
                        U[0][0] * U[1][1] - U[1][0] * U[0][1]};
  const double along = U[0][2] * u3[0] + U[1][2] * u3[1] + U[2][2] * u3[2];
  for (int i = 0; i < 3; ++i) {
    U[i][2] = u3[i];
    if (along < 0.0) Vs[i][2] = -Vs[i][2];
  }
  // R = V diag(1, 1, d) U^T, d = sign det(V U^T) = sign det(V) since det U = +1
  const double d = det3(Vs) >= 0.0 ? 1.0 : -1.0;
  double R[3][3];
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 3; ++j)
      R[i][j] = Vs[i][0] * U[j][0] + Vs[i][1] * U[j][1] + d * Vs[i][2] * U[j][2];
  for (int i = 0; i < 3; ++i) {
    const double t = m.mu_tgt[i] -
                     (R[i][0] * m.mu_src[0] + R[i][1] * m.mu_src[1] + R[i][2] * m.mu_src[2]);
    for (int j = 0; j < 3; ++j) T[4 * i + j] = R[i][j];
    T[4 * i + 3] = t;
  }
  T[12] = T[13] = T[14] = 0.0;
  T[15] = 1.0;
  return ICPNN_OK;
}

}  // namespace icpnn
