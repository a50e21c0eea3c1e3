// Muon optimizer step: plain fp64 CPU oracle.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
// restatement of the Muon step that the CUDA path is checked against.  It is
// never linked into, loaded by or called from the product library; only the
// tests, the smoke check and the benchmark's CPU-baseline leg use it.  It
// shares no code, header, table or constant with the CUDA path.
//
// What it follows (HyperParallel FSDP Muon optimizer RFC, mindspore
// hyper-parallel issue "HyperParallel FSDP Muon优化器性能优化 RFC"):
//   * section 1(1): Newton-Schulz is applied to the whole gradient-momentum
//     matrix M_t;
//   * section 2: the iteration depends only on the last two dims, so the E
//     slices of an [E, M, N] expert tensor are independent;
//   * section 3: parameters whose trailing dims agree are regrouped into one
//     contiguous [B, M, N] batch;
//   * section 6: an AdamW-style (decoupled) weight-decay term is added to the
//     Muon update.
// The RFC fixes neither the iteration nor its constants.  The readings taken
// here, each a stated parameter of this library:
//   * momentum  M' = beta*M + G;  V = G + beta*M' (Nesterov) or V = M';
//   * normalise X0 = V / (||V||_F + eps), eps = 1e-7;
//   * work on X0^T when M > N so that the iterate has min(M,N) rows;
//   * quintic Newton-Schulz, T steps:  A = X X^T;  B = b*A + c*A*A;
//     X <- a*X + B*X, default (a,b,c) = (3.4445, -4.7750, 2.0315), T = 5;
//   * update  W' = W*(1 - lr*wd) - lr*s*O,  s = sqrt(max(1, M/N)).
// Everything is computed in IEEE double with plain loops; build it without
// -ffast-math and with -ffp-contract=off so x86 and Arm builds agree.
//
// Parity pins of every function here live in tests/test_oracle_pins.py.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

// Split rows [0, rows) across `threads` workers and run fn(r0, r1).
template <class F>
void parallel_rows(int64_t rows, int threads, F fn) {
  if (threads <= 1 || rows < 2) { fn(0, rows); return; }
  int t = (int)std::min<int64_t>(threads, rows);
  std::vector<std::thread> pool;
  int64_t per = (rows + t - 1) / t;
  for (int i = 0; i < t; ++i) {
    int64_t r0 = i * per, r1 = std::min(rows, r0 + per);
    if (r0 >= r1) break;
    pool.emplace_back([=] { fn(r0, r1); });
  }
  for (auto& th : pool) th.join();
}

// Run fn(i) for every row i of [0, rows), rows dealt to `threads` workers
// in turn (row i to worker i mod threads), for rows of unequal cost.
template <class F>
void parallel_rows_dealt(int64_t rows, int threads, F fn) {
  int t = (int)std::max<int64_t>(1, std::min<int64_t>(threads, rows));
  if (t == 1) { for (int64_t i = 0; i < rows; ++i) fn(i); return; }
  std::vector<std::thread> pool;
  for (int w = 0; w < t; ++w)
    pool.emplace_back([=] { for (int64_t i = w; i < rows; i += t) fn(i); });
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Plan: RFC section 3 (regroup same trailing dims into [B, M, N]) and
// section 2 (an [E, M, N] tensor contributes E independent slices).
//
// Parameters are walked in call order, slices e = 0..E-1 inside each.  The
// key is (M, N, dtype); groups are numbered by the first appearance of their
// key; a slice's index inside its group is its order of encounter.  A 2D
// parameter is a one-slice stack.  tr = (M > N).  The update scale s (the
// RFC leaves it open) is, rounded once to float,
//   scale_mode 0: s = sqrt(max(1, M/N));
//   scale_mode 1: s = 0.2 * sqrt(max(M, N)) (an update of RMS 0.2 when O has
//                 unit singular values).
//
// dims: 3 entries per parameter (unused ones ignored); ndim in {2, 3}.
// Outputs per slice (in walk order): slice_group, slice_index.
// Outputs per group (capacity max_groups): M, N, dtype, count, tr, scale.
// Returns the number of groups, or -1 on an invalid shape, -2 when more
// than max_groups groups would be needed.
int oracle_plan(int nparams, const int* ndim, const int64_t* dims,
                const int* dtype, int* slice_group, int* slice_index,
                int max_groups, int64_t* group_M, int64_t* group_N,
                int* group_dtype, int* group_count, int* group_tr,
                float* group_scale, int scale_mode) {
  int ngroups = 0;
  int64_t s = 0;
  for (int p = 0; p < nparams; ++p) {
    int64_t E, M, N;
    if (ndim[p] == 2) { E = 1; M = dims[3 * p + 0]; N = dims[3 * p + 1]; }
    else if (ndim[p] == 3) { E = dims[3 * p + 0]; M = dims[3 * p + 1]; N = dims[3 * p + 2]; }
    else return -1;
    if (E < 1 || M < 1 || N < 1) return -1;
    int g = -1;
    for (int k = 0; k < ngroups; ++k)
      if (group_M[k] == M && group_N[k] == N && group_dtype[k] == dtype[p]) { g = k; break; }
    if (g < 0) {
      if (ngroups == max_groups) return -2;
      g = ngroups++;
      group_M[g] = M; group_N[g] = N; group_dtype[g] = dtype[p];
      group_count[g] = 0;
      group_tr[g] = M > N ? 1 : 0;
      if (scale_mode == 1) {
        group_scale[g] = (float)(0.2 * std::sqrt((double)(M > N ? M : N)));
      } else {
        double ratio = (double)M / (double)N;
        group_scale[g] = (float)std::sqrt(ratio > 1.0 ? ratio : 1.0);
      }
    }
    for (int64_t e = 0; e < E; ++e, ++s) {
      slice_group[s] = g;
      slice_index[s] = group_count[g]++;
    }
  }
  return ngroups;
}

// ---------------------------------------------------------------------------
// Momentum (RFC section 1(1): the iteration's input is the gradient
// momentum M_t).  Elementwise over `count` values:
//   M' = beta*M + G;   V = G + beta*M' if nesterov else M'.
void oracle_momentum(int64_t count, const double* G, const double* Mom,
                     double beta, int nesterov, double* Mom_out, double* V_out) {
  for (int64_t i = 0; i < count; ++i) {
    double m = beta * Mom[i] + G[i];
    Mom_out[i] = m;
    V_out[i] = nesterov ? G[i] + beta * m : m;
  }
}

// Frobenius normalisation: X = V / (||V||_F + eps).
void oracle_normalize(int64_t count, const double* V, double eps, double* X_out) {
  double ss = 0.0;
  for (int64_t i = 0; i < count; ++i) ss += V[i] * V[i];
  double d = std::sqrt(ss) + eps;
  for (int64_t i = 0; i < count; ++i) X_out[i] = V[i] / d;
}

// Quintic Newton-Schulz on one [M, N] matrix X (row-major), T steps.
// When M > N the iteration runs on X^T (min(M,N) rows) and the result is
// transposed back, so O always has X's shape.  Each step:
//   A = X X^T;  B = b*A + c*(A A);  X <- a*X + B X.
// `threads` splits the rows of each product across workers; every output
// entry is still one plain sum in index order.  X X^T and A A are symmetric
// by definition: entry (j, i) of either is the sum of the same products as
// entry (i, j), in the same order (A itself is exactly symmetric), so it is
// the same number; each is computed for j >= i and copied to (j, i).
void oracle_newton_schulz(int64_t M, int64_t N, const double* X_in, int T,
                          double a, double b, double c, int threads,
                          double* O_out) {
  const bool tr = M > N;
  const int64_t m = tr ? N : M, n = tr ? M : N;
  std::vector<double> X((size_t)(m * n)), Xn((size_t)(m * n));
  for (int64_t i = 0; i < m; ++i)
    for (int64_t k = 0; k < n; ++k)
      X[i * n + k] = tr ? X_in[k * N + i] : X_in[i * n + k];
  std::vector<double> A((size_t)(m * m)), At((size_t)(m * m)), B((size_t)(m * m));
  for (int t = 0; t < T; ++t) {
    // A = X X^T (upper triangle, then mirrored)
    parallel_rows_dealt(m, threads, [&](int64_t i) {
      for (int64_t j = i; j < m; ++j) {
        double acc = 0.0;
        for (int64_t k = 0; k < n; ++k) acc += X[i * n + k] * X[j * n + k];
        A[i * m + j] = acc;
      }
    });
    for (int64_t i = 0; i < m; ++i)
      for (int64_t j = 0; j < i; ++j) A[i * m + j] = A[j * m + i];
    // B = b*A + c*(A A); the second factor is read from a transposed copy
    // At[j][k] = A[k][j] so that both operands stream along rows
    for (int64_t i = 0; i < m; ++i)
      for (int64_t j = 0; j < m; ++j) At[j * m + i] = A[i * m + j];
    parallel_rows_dealt(m, threads, [&](int64_t i) {
      for (int64_t j = i; j < m; ++j) {
        double acc = 0.0;
        for (int64_t k = 0; k < m; ++k) acc += A[i * m + k] * At[j * m + k];
        B[i * m + j] = b * A[i * m + j] + c * acc;
      }
    });
    for (int64_t i = 0; i < m; ++i)
      for (int64_t j = 0; j < i; ++j) B[i * m + j] = B[j * m + i];
    // X <- a*X + B X
    parallel_rows(m, threads, [&](int64_t r0, int64_t r1) {
      std::vector<double> row((size_t)n);
      for (int64_t i = r0; i < r1; ++i) {
        std::fill(row.begin(), row.end(), 0.0);
        for (int64_t j = 0; j < m; ++j) {
          const double bij = B[i * m + j];
          const double* xj = &X[j * n];
          for (int64_t k = 0; k < n; ++k) row[k] += bij * xj[k];
        }
        for (int64_t k = 0; k < n; ++k) Xn[i * n + k] = a * X[i * n + k] + row[k];
      }
    });
    X.swap(Xn);
  }
  for (int64_t i = 0; i < m; ++i)
    for (int64_t k = 0; k < n; ++k) {
      if (tr) O_out[k * N + i] = X[i * n + k];
      else O_out[i * n + k] = X[i * n + k];
    }
}

// Decoupled weight decay and the scaled orthogonal update (RFC section 6):
//   W' = W*(1 - lr*wd) - lr*scale*O.
void oracle_update(int64_t count, const double* W, const double* O, double lr,
                   double wd, double scale, double* W_out) {
  const double decay = 1.0 - lr * wd;
  for (int64_t i = 0; i < count; ++i) W_out[i] = W[i] * decay - lr * scale * O[i];
}

// One whole Muon step for one [M, N] slice: momentum, normalisation,
// Newton-Schulz, update.  O_out (may be null) receives the orthogonalised
// momentum.  scale is the update scale s of the slice's group.
void oracle_muon_slice(int64_t M, int64_t N, const double* W, const double* G,
                       const double* Mom, double lr, double beta, double wd,
                       int nesterov, int T, const double* coeffs, double eps,
                       double scale, int threads, double* W_out,
                       double* Mom_out, double* O_out) {
  const int64_t cnt = M * N;
  std::vector<double> V((size_t)cnt), X((size_t)cnt), O((size_t)cnt);
  oracle_momentum(cnt, G, Mom, beta, nesterov, Mom_out, V.data());
  oracle_normalize(cnt, V.data(), eps, X.data());
  oracle_newton_schulz(M, N, X.data(), T, coeffs[0], coeffs[1], coeffs[2],
                       threads, O.data());
  oracle_update(cnt, W, O.data(), lr, wd, scale, W_out);
  if (O_out) std::memcpy(O_out, O.data(), sizeof(double) * (size_t)cnt);
}

// Many independent slices (RFC section 2: slices are independent), spread
// over `threads` workers, one slice per worker at a time.  Arrays hold one
// entry per slice.  Returns the number of worker threads used.
int oracle_muon_slices(int nslices, const int64_t* Ms, const int64_t* Ns,
                       const double* const* W, const double* const* G,
                       const double* const* Mom, double lr, double beta,
                       double wd, int nesterov, int T, const double* coeffs,
                       double eps, const double* scales, int threads,
                       double* const* W_out, double* const* Mom_out,
                       double* const* O_out) {
  int nt = std::max(1, std::min(threads, nslices));
  std::vector<std::thread> pool;
  for (int w = 0; w < nt; ++w) {
    pool.emplace_back([=] {
      for (int s = w; s < nslices; s += nt)
        oracle_muon_slice(Ms[s], Ns[s], W[s], G[s], Mom[s], lr, beta, wd,
                          nesterov, T, coeffs, eps, scales[s], 1, W_out[s],
                          Mom_out[s], O_out ? O_out[s] : nullptr);
    });
  }
  for (auto& th : pool) th.join();
  return nt;
}

// Loss scaling (Paddle PR "Support Muon sharding optimizer comm overlap",
// review of the AMP GradScaler path: the Muon step runs on gradients that a
// loss scaler has multiplied by S and must unscale and check first).
// 1 when every one of `count` values is finite, else 0.
int oracle_all_finite(int64_t count, const double* G) {
  for (int64_t i = 0; i < count; ++i)
    if (!std::isfinite(G[i])) return 0;
  return 1;
}

// Unscaled gradient: out = G * inv_scale.
void oracle_unscale(int64_t count, const double* G, double inv_scale, double* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = G[i] * inv_scale;
}

// AdamW for the parameters Muon does not orthogonalise (1-D and other
// non-matrix tensors; the Paddle Muon sharding PR keeps separate 2-D and 1-D
// communication buffers because the two kinds take different update rules).
// Standard AdamW with bias correction and decoupled weight decay, step t >= 1:
//   m' = b1*m + (1-b1)*g;  v' = b2*v + (1-b2)*g^2
//   W' = W*(1 - lr*wd) - lr * (m'/(1-b1^t)) / (sqrt(v'/(1-b2^t)) + eps)
void oracle_adamw(int64_t count, const double* W, const double* G, const double* Mm,
                  const double* Vv, double lr, double b1, double b2, double eps, double wd,
                  int t, double* W_out, double* M_out, double* V_out) {
  const double c1 = 1.0 - std::pow(b1, t), c2 = 1.0 - std::pow(b2, t);
  for (int64_t i = 0; i < count; ++i) {
    const double m = b1 * Mm[i] + (1.0 - b1) * G[i];
    const double v = b2 * Vv[i] + (1.0 - b2) * G[i] * G[i];
    M_out[i] = m;
    V_out[i] = v;
    W_out[i] = W[i] * (1.0 - lr * wd) - lr * (m / c1) / (std::sqrt(v / c2) + eps);
  }
}

}  // extern "C"
