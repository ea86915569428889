// aq_decompose.cu -- the decomposition that produces a theta bundle, on the GPU
// ("How attnquant works", "How the decomposition produces s, U, and V"):
//   W0     = the element-wise mean of the band's layer weights            (aq_band_mean)
//   s[o]   = (w[o] . W0[o]) / (W0[o] . W0[o]), stored in bf16              (aq_ls_residual)
//   resid  = w - diag(s) W0, with the stored s
//   U, V   = rank-r factors of resid, U = U_svd S, by the randomized SVD   (aq_randomized_svd)
//            of Halko, Martinsson and Tropp (2009) the pages name: the range finder Y = A Omega,
//            Q = orth(Y) (q power iterations optional), B = Q^T A, the SVD of the small B.
// The decomposition is a load-time step, so it runs in double precision on the CUDA cores: a
// tiled fp64 GEMM, CholeskyQR2 for orth(), and one-CTA cyclic Jacobi (round-robin pairs, all
// rotations of a step at once) for the eigenvalues of B B^T, from which B's SVD follows.
// Every kernel is a plain launch on the caller's stream; aq_randomized_svd synchronises it at the
// end to report a numerical breakdown (a non-positive Cholesky pivot).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>

#include <algorithm>

#include "aq.h"
#include "aq_internal.h"

namespace aq {
namespace {

constexpr int kMaxBandLayers = 256;   // weights one aq_band_mean call averages
constexpr int kMaxSvdK = 256;          // columns of the test matrix Omega

aq_status err(aq_status st, const char* msg) { return static_cast<aq_status>(set_last_error(st, msg)); }

aq_status cuda_err(cudaError_t e, const char* what) {
  char buf[256];
  snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
  return static_cast<aq_status>(set_last_error(AQ_ERR_CUDA, buf));
}

__device__ __forceinline__ double bf16_bits_to_f64(uint16_t b) {
  return static_cast<double>(__uint_as_float(static_cast<uint32_t>(b) << 16));
}

__device__ __forceinline__ uint16_t f64_to_bf16_rn(double v) {
  return __bfloat16_as_ushort(__double2bfloat16(v));
}

// ------------------------------------------------------------------------------------
// band mean: W0 = RN_bf16( (sum over the layers, in layer order) / L ), in fp64
// ------------------------------------------------------------------------------------
struct BandMeanParams {
  const uint16_t* w[kMaxBandLayers];
  int32_t L;
  int32_t out, in;
  int64_t ld;
  uint16_t* W0;
  int64_t ld_w0;
};

__global__ void __launch_bounds__(256) band_mean_kernel(const __grid_constant__ BandMeanParams p) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(p.out) * p.in) return;
  const int o = static_cast<int>(idx / p.in), i = static_cast<int>(idx % p.in);
  double acc = 0.0;
  for (int l = 0; l < p.L; ++l) acc += bf16_bits_to_f64(p.w[l][static_cast<int64_t>(o) * p.ld + i]);
  p.W0[static_cast<int64_t>(o) * p.ld_w0 + i] = f64_to_bf16_rn(acc / p.L);
}

// ------------------------------------------------------------------------------------
// least-squares scale and residual: one CTA per output row, fixed-order fp64 reduction
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) ls_residual_kernel(const uint16_t* __restrict__ w, int64_t ldw,
                                                          const uint16_t* __restrict__ W0, int64_t ld_w0, int in,
                                                          uint16_t* s, double* resid, int64_t ld_r) {
  __shared__ double red_n[256], red_d[256];
  __shared__ double s_used;
  const int o = blockIdx.x;
  const uint16_t* wr = w + static_cast<int64_t>(o) * ldw;
  const uint16_t* br = W0 + static_cast<int64_t>(o) * ld_w0;
  double num = 0.0, den = 0.0;
  for (int i = threadIdx.x; i < in; i += 256) {
    const double a = bf16_bits_to_f64(wr[i]), b = bf16_bits_to_f64(br[i]);
    num = fma(a, b, num);
    den = fma(b, b, den);
  }
  red_n[threadIdx.x] = num;
  red_d[threadIdx.x] = den;
  __syncthreads();
  for (int h = 128; h > 0; h >>= 1) {
    if (static_cast<int>(threadIdx.x) < h) {
      red_n[threadIdx.x] += red_n[threadIdx.x + h];
      red_d[threadIdx.x] += red_d[threadIdx.x + h];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    // a W0 row of zeros has no least-squares scale; it keeps 1 (its residual is the weight)
    const double sc = red_d[0] == 0.0 ? 1.0 : red_n[0] / red_d[0];
    const uint16_t sb = f64_to_bf16_rn(sc);
    s[o] = sb;
    s_used = bf16_bits_to_f64(sb);   // the residual is taken against the stored scale
  }
  __syncthreads();
  const double sc = s_used;
  double* rr = resid + static_cast<int64_t>(o) * ld_r;
  for (int i = threadIdx.x; i < in; i += 256) rr[i] = bf16_bits_to_f64(wr[i]) - sc * bf16_bits_to_f64(br[i]);
}

// ------------------------------------------------------------------------------------
// fp64 GEMM: C[i][j] = sum_p A(i, p) B(p, j), with A(i, p) = A[i * a_rs + p * a_cs] and
// B(p, j) = B[p * b_rs + j * b_cs] (the strides express transposes). C is fp64 [M][ldc] or,
// when c16 is set, bf16 (one rounding). 64 x 64 tiles, 256 threads of 4 x 4 outputs.
// ------------------------------------------------------------------------------------
struct GemmF64 {
  const double* A;
  int64_t a_rs, a_cs;
  const double* B;
  int64_t b_rs, b_cs;
  double* C;
  uint16_t* c16;
  int64_t ldc;
  int M, N, K;
};

__global__ void __launch_bounds__(256) gemm_f64_kernel(const __grid_constant__ GemmF64 g) {
  __shared__ double As[16][65];
  __shared__ double Bs[16][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
  double acc[4][4] = {};
  for (int p0 = 0; p0 < g.K; p0 += 16) {
    for (int e = threadIdx.x; e < 64 * 16; e += 256) {
      const int ii = e >> 4, pp = e & 15;   // A tile element (row ii, depth pp)
      const int i = i0 + ii, p = p0 + pp;
      As[pp][ii] = (i < g.M && p < g.K) ? g.A[static_cast<int64_t>(i) * g.a_rs + static_cast<int64_t>(p) * g.a_cs] : 0.0;
      const int jj = e & 63, qq = e >> 6;   // B tile element (depth qq, column jj)
      const int j = j0 + jj, q = p0 + qq;
      Bs[qq][jj] = (j < g.N && q < g.K) ? g.B[static_cast<int64_t>(q) * g.b_rs + static_cast<int64_t>(j) * g.b_cs] : 0.0;
    }
    __syncthreads();
#pragma unroll
    for (int pp = 0; pp < 16; ++pp) {
      double a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        a[u] = As[pp][ty * 4 + u];
        b[u] = Bs[pp][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fma(a[u], b[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int i = i0 + ty * 4 + u, j = j0 + tx * 4 + v;
      if (i < g.M && j < g.N) {
        if (g.c16) {
          g.c16[static_cast<int64_t>(i) * g.ldc + j] = f64_to_bf16_rn(acc[u][v]);
        } else {
          g.C[static_cast<int64_t>(i) * g.ldc + j] = acc[u][v];
        }
      }
    }
}

cudaError_t gemm_f64(const GemmF64& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  const dim3 grid((g.N + 63) / 64, (g.M + 63) / 64);
  gemm_f64_kernel<<<grid, 256, 0, st>>>(g);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------
// Cholesky of a k x k symmetric positive definite G (row-major, in place, one CTA): the lower
// triangle becomes L with G = L L^T. A pivot that is not positive and finite sets *fail.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cholesky_kernel(double* G, int k, int* fail) {
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int j = 0; j < k; ++j) {
    if (threadIdx.x == 0) {
      const double d = G[j * k + j];
      if (!(d > 0.0) || !isfinite(d)) {
        bad = 1;
        G[j * k + j] = 1.0;
      } else {
        G[j * k + j] = sqrt(d);
      }
    }
    __syncthreads();
    if (bad) break;
    const double djj = G[j * k + j];
    for (int i = j + 1 + threadIdx.x; i < k; i += 256) G[i * k + j] /= djj;
    __syncthreads();
    // trailing lower triangle: G[i][l] -= L[i][j] L[l][j] for j < l <= i
    const int t = k - j - 1;
    for (int e = threadIdx.x; e < t * t; e += 256) {
      const int i = j + 1 + e / t, l = j + 1 + e % t;
      if (l <= i) G[i * k + l] -= G[i * k + j] * G[l * k + j];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0 && bad) atomicExch(fail, 1);
}

// Rows of Y [m][ldy] (first k columns) times L^-T, in place: q L^T = y, forward substitution
// per row (one thread per row).
__global__ void __launch_bounds__(128) rows_solve_lt_kernel(double* Y, int64_t ldy, int m, const double* L, int k) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= m) return;
  double* y = Y + static_cast<int64_t>(row) * ldy;
  for (int j = 0; j < k; ++j) {
    double acc = y[j];
    const double* Lj = L + static_cast<int64_t>(j) * k;
    for (int p = 0; p < j; ++p) acc = fma(-y[p], Lj[p], acc);
    y[j] = acc / Lj[j];
  }
}

// ------------------------------------------------------------------------------------
// Symmetric eigen-decomposition of a k x k S (row-major, in place) by cyclic Jacobi with
// round-robin pairs: in every step k/2 disjoint rotations are formed from the current S and
// applied together (rows, then columns), the eigenvector matrix W accumulates the columns.
// Then the eigenvalues are sorted in descending order: lam[i], and Ws[:, i] the matching column.
// One CTA; sweeps until the off-diagonal mass is below 1e-30 of the diagonal's, at most 60.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) jacobi_eig_kernel(double* S, double* W, double* Ws, double* lam, int k) {
  __shared__ double cs[kMaxSvdK / 2], sn[kMaxSvdK / 2];
  __shared__ int pa[kMaxSvdK / 2], pb[kMaxSvdK / 2];
  __shared__ double red[256];
  __shared__ int done;
  __shared__ int order[kMaxSvdK];
  const int tid = threadIdx.x;
  for (int e = tid; e < k * k; e += 256) W[e] = (e / k == e % k) ? 1.0 : 0.0;
  const int n2 = (k + 1) & ~1;   // players, a dummy one when k is odd
  const int npair = n2 / 2;
  __syncthreads();
  for (int sweep = 0; sweep < 60; ++sweep) {
    for (int step = 0; step < n2 - 1; ++step) {
      // round-robin: position 0 stays, positions 1..n2-1 rotate by `step`
      for (int i = tid; i < npair; i += 256) {
        auto pos = [&](int j) { return j == 0 ? 0 : 1 + (j - 1 + step) % (n2 - 1); };
        int a = pos(i), b = pos(n2 - 1 - i);
        if (a > b) {
          const int tmp = a;
          a = b;
          b = tmp;
        }
        double c = 1.0, s = 0.0;
        if (b < k) {
          const double app = S[a * k + a], aqq = S[b * k + b], apq = S[a * k + b];
          if (apq != 0.0) {
            const double tau = (aqq - app) / (2.0 * apq);
            const double t = (tau >= 0.0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
            c = 1.0 / sqrt(1.0 + t * t);
            s = t * c;
          }
        }
        pa[i] = a;
        pb[i] = b;
        cs[i] = c;
        sn[i] = s;
      }
      __syncthreads();
      // rows: row_a' = c row_a - s row_b, row_b' = s row_a + c row_b
      for (int e = tid; e < npair * k; e += 256) {
        const int i = e / k, col = e % k;
        const int a = pa[i], b = pb[i];
        if (b >= k || sn[i] == 0.0) continue;
        const double x = S[a * k + col], y = S[b * k + col];
        S[a * k + col] = cs[i] * x - sn[i] * y;
        S[b * k + col] = sn[i] * x + cs[i] * y;
      }
      __syncthreads();
      // columns of S and of W
      for (int e = tid; e < npair * k; e += 256) {
        const int i = e / k, row = e % k;
        const int a = pa[i], b = pb[i];
        if (b >= k || sn[i] == 0.0) continue;
        const double x = S[row * k + a], y = S[row * k + b];
        S[row * k + a] = cs[i] * x - sn[i] * y;
        S[row * k + b] = sn[i] * x + cs[i] * y;
        const double u = W[row * k + a], v = W[row * k + b];
        W[row * k + a] = cs[i] * u - sn[i] * v;
        W[row * k + b] = sn[i] * u + cs[i] * v;
      }
      __syncthreads();
    }
    // convergence: off-diagonal mass against the diagonal's
    double off = 0.0, dia = 0.0;
    for (int e = tid; e < k * k; e += 256) {
      const double v = S[e];
      if (e / k == e % k) dia += v * v; else off += v * v;
    }
    red[tid] = off;
    __syncthreads();
    for (int h = 128; h > 0; h >>= 1) {
      if (tid < h) red[tid] += red[tid + h];
      __syncthreads();
    }
    const double off_t = red[0];
    __syncthreads();
    red[tid] = dia;
    __syncthreads();
    for (int h = 128; h > 0; h >>= 1) {
      if (tid < h) red[tid] += red[tid + h];
      __syncthreads();
    }
    if (tid == 0) done = !(off_t > 1e-30 * red[0]);
    __syncthreads();
    if (done) break;
  }
  // eigenvalues in descending order (a selection sort of k <= 256 values by one thread)
  if (tid == 0) {
    for (int i = 0; i < k; ++i) order[i] = i;
    for (int i = 0; i < k; ++i) {
      int best = i;
      for (int j = i + 1; j < k; ++j)
        if (S[order[j] * k + order[j]] > S[order[best] * k + order[best]]) best = j;
      const int t = order[i];
      order[i] = order[best];
      order[best] = t;
    }
  }
  __syncthreads();
  for (int i = tid; i < k; i += 256) lam[i] = S[order[i] * k + order[i]];
  for (int e = tid; e < k * k; e += 256) {
    const int row = e / k, i = e % k;
    Ws[row * k + i] = W[row * k + order[i]];
  }
}

// Columns of the factors' small right-hand matrices: Wsc[p][i] = Ws[p][i] * sigma_i and
// Wsi[p][i] = Ws[p][i] / sigma_i (0 where sigma_i is 0), sigma_i = sqrt(max(lam_i, 0)), i < r.
__global__ void scale_cols_kernel(const double* Ws, const double* lam, int k, int r, double* Wsc, double* Wsi) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= k * r) return;
  const int p = e / r, i = e % r;
  const double sg = sqrt(fmax(lam[i], 0.0));
  const double w = Ws[p * k + i];
  Wsc[e] = w * sg;
  Wsi[e] = sg > 0.0 ? w / sg : 0.0;
}

// ------------------------------------------------------------------------------------
// workspace of aq_randomized_svd (doubles unless noted)
// ------------------------------------------------------------------------------------
struct SvdWs {
  size_t y, z, g, b, s, w, ws, lam, wsc, wsi, flag, total;
};

SvdWs svd_ws(int64_t m, int64_t n, int64_t k, int64_t r) {
  SvdWs o = {};
  size_t at = 0;
  auto take = [&](size_t bytes) {
    const size_t here = at;
    at += (bytes + 255) / 256 * 256;
    return here;
  };
  o.y = take(static_cast<size_t>(m * k) * 8);
  o.z = take(static_cast<size_t>(n * k) * 8);
  o.g = take(static_cast<size_t>(k * k) * 8);
  o.b = take(static_cast<size_t>(k * n) * 8);
  o.s = take(static_cast<size_t>(k * k) * 8);
  o.w = take(static_cast<size_t>(k * k) * 8);
  o.ws = take(static_cast<size_t>(k * k) * 8);
  o.lam = take(static_cast<size_t>(k) * 8);
  o.wsc = take(static_cast<size_t>(k * std::max<int64_t>(r, 1)) * 8);
  o.wsi = take(static_cast<size_t>(k * std::max<int64_t>(r, 1)) * 8);
  o.flag = take(16);
  o.total = at;
  return o;
}

// orth(Y) by CholeskyQR2: twice G = Y^T Y, G = L L^T, Y <- Y L^-T (in place)
cudaError_t cholqr2(double* Y, int64_t ldy, int m, int k, double* G, int* fail, cudaStream_t st) {
  for (int pass = 0; pass < 2; ++pass) {
    GemmF64 g = {};
    g.A = Y;
    g.a_rs = 1;
    g.a_cs = ldy;
    g.B = Y;
    g.b_rs = ldy;
    g.b_cs = 1;
    g.C = G;
    g.ldc = k;
    g.M = k;
    g.N = k;
    g.K = m;
    cudaError_t e = gemm_f64(g, st);
    if (e != cudaSuccess) return e;
    cholesky_kernel<<<1, 256, 0, st>>>(G, k, fail);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    rows_solve_lt_kernel<<<(m + 127) / 128, 128, 0, st>>>(Y, ldy, m, G, k);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

bool aligned16p(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace aq

using namespace aq;

extern "C" aq_status aq_band_mean(const void* const* weights, int32_t L, int32_t out, int32_t in, int64_t ld, void* W0,
                                  int64_t ld_w0, void* stream) {
  if (!weights || !W0) return err(AQ_ERR_INVALID_ARG, "aq_band_mean: NULL argument");
  if (L < 1 || L > kMaxBandLayers) return err(AQ_ERR_INVALID_ARG, "aq_band_mean: L must be in [1, 256]");
  if (out < 1 || in < 1 || ld < in || ld_w0 < in) return err(AQ_ERR_SHAPE, "aq_band_mean: bad shape or leading dimension");
  BandMeanParams p = {};
  for (int l = 0; l < L; ++l) {
    if (!weights[l]) return err(AQ_ERR_INVALID_ARG, "aq_band_mean: a weight pointer is NULL");
    p.w[l] = static_cast<const uint16_t*>(weights[l]);
  }
  p.L = L;
  p.out = out;
  p.in = in;
  p.ld = ld;
  p.W0 = static_cast<uint16_t*>(W0);
  p.ld_w0 = ld_w0;
  const int64_t n = static_cast<int64_t>(out) * in;
  band_mean_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? AQ_OK : cuda_err(e, "aq_band_mean: launch");
}

extern "C" aq_status aq_ls_residual(const void* weight, int64_t ldw, const void* W0, int64_t ld_w0, int32_t out,
                                    int32_t in, void* s, double* resid, int64_t ld_r, void* stream) {
  if (!weight || !W0 || !s || !resid) return err(AQ_ERR_INVALID_ARG, "aq_ls_residual: NULL argument");
  if (out < 1 || in < 1 || ldw < in || ld_w0 < in || ld_r < in)
    return err(AQ_ERR_SHAPE, "aq_ls_residual: bad shape or leading dimension");
  ls_residual_kernel<<<out, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(weight), ldw, static_cast<const uint16_t*>(W0), ld_w0, in,
      static_cast<uint16_t*>(s), resid, ld_r);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? AQ_OK : cuda_err(e, "aq_ls_residual: launch");
}

extern "C" size_t aq_randomized_svd_workspace_bytes(int32_t m, int32_t n, int32_t k, int32_t r) {
  if (m < 1 || n < 1 || k < 1 || k > kMaxSvdK || r < 0 || r > k) return static_cast<size_t>(-1);
  return svd_ws(m, n, k, r).total;
}

extern "C" aq_status aq_randomized_svd(const double* A, int64_t lda, int32_t m, int32_t n, int32_t r,
                                       const double* omega, int64_t ld_omega, int32_t k, int32_t power_iters, void* U,
                                       int64_t ld_u, void* V, int64_t ld_v, void* workspace, size_t ws_bytes,
                                       void* stream) {
  if (!A || !omega) return err(AQ_ERR_INVALID_ARG, "aq_randomized_svd: NULL argument");
  if (m < 1 || n < 1 || lda < n || ld_omega < k) return err(AQ_ERR_SHAPE, "aq_randomized_svd: bad shape");
  if (k < 1 || k > kMaxSvdK || r < 0 || r > k || k > std::min(m, n))
    return err(AQ_ERR_SHAPE, "aq_randomized_svd: need 0 <= r <= k <= min(m, n) and k <= 256");
  if (power_iters < 0 || power_iters > 16) return err(AQ_ERR_INVALID_ARG, "aq_randomized_svd: power_iters in [0, 16]");
  if (r > 0 && (!U || !V || ld_u < r || ld_v < r)) return err(AQ_ERR_SHAPE, "aq_randomized_svd: U / V missing or too narrow");
  if (r == 0) return AQ_OK;
  const SvdWs w = svd_ws(m, n, k, r);
  if (!workspace || ws_bytes < w.total || !aligned16p(workspace)) {
    char buf[160];
    snprintf(buf, sizeof buf, "aq_randomized_svd: workspace of %zu bytes (16-byte aligned) required, got %zu", w.total,
             ws_bytes);
    return err(AQ_ERR_WORKSPACE, buf);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  double* Y = reinterpret_cast<double*>(base + w.y);
  double* Z = reinterpret_cast<double*>(base + w.z);
  double* G = reinterpret_cast<double*>(base + w.g);
  double* B = reinterpret_cast<double*>(base + w.b);
  double* S = reinterpret_cast<double*>(base + w.s);
  double* W = reinterpret_cast<double*>(base + w.w);
  double* Ws = reinterpret_cast<double*>(base + w.ws);
  double* lam = reinterpret_cast<double*>(base + w.lam);
  double* Wsc = reinterpret_cast<double*>(base + w.wsc);
  double* Wsi = reinterpret_cast<double*>(base + w.wsi);
  int* fail = reinterpret_cast<int*>(base + w.flag);
  cudaError_t e;
  if ((e = cudaMemsetAsync(fail, 0, sizeof(int), st)) != cudaSuccess) return cuda_err(e, "aq_randomized_svd: memset");
  auto gemm = [&](const double* a, int64_t ars, int64_t acs, const double* b, int64_t brs, int64_t bcs, double* c,
                  uint16_t* c16, int64_t ldc, int M, int N, int K) {
    GemmF64 g = {};
    g.A = a;
    g.a_rs = ars;
    g.a_cs = acs;
    g.B = b;
    g.b_rs = brs;
    g.b_cs = bcs;
    g.C = c;
    g.c16 = c16;
    g.ldc = ldc;
    g.M = M;
    g.N = N;
    g.K = K;
    return gemm_f64(g, st);
  };
  // range finder: Y = A Omega, Q = orth(Y) (Q overwrites Y)
  if ((e = gemm(A, lda, 1, omega, ld_omega, 1, Y, nullptr, k, m, k, n)) != cudaSuccess) return cuda_err(e, "gemm A Omega");
  if ((e = cholqr2(Y, k, m, k, G, fail, st)) != cudaSuccess) return cuda_err(e, "orth(Y)");
  for (int it = 0; it < power_iters; ++it) {
    // Z = orth(A^T Q), Q = orth(A Z)
    if ((e = gemm(A, 1, lda, Y, k, 1, Z, nullptr, k, n, k, m)) != cudaSuccess) return cuda_err(e, "gemm A^T Q");
    if ((e = cholqr2(Z, k, n, k, G, fail, st)) != cudaSuccess) return cuda_err(e, "orth(Z)");
    if ((e = gemm(A, lda, 1, Z, k, 1, Y, nullptr, k, m, k, n)) != cudaSuccess) return cuda_err(e, "gemm A Z");
    if ((e = cholqr2(Y, k, m, k, G, fail, st)) != cudaSuccess) return cuda_err(e, "orth(Y)");
  }
  // B = Q^T A [k x n]; B B^T = Ws diag(lam) Ws^T
  if ((e = gemm(Y, 1, k, A, lda, 1, B, nullptr, n, k, n, m)) != cudaSuccess) return cuda_err(e, "gemm Q^T A");
  if ((e = gemm(B, n, 1, B, 1, n, S, nullptr, k, k, k, n)) != cudaSuccess) return cuda_err(e, "gemm B B^T");
  jacobi_eig_kernel<<<1, 256, 0, st>>>(S, W, Ws, lam, k);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_err(e, "jacobi");
  scale_cols_kernel<<<(k * r + 255) / 256, 256, 0, st>>>(Ws, lam, k, r, Wsc, Wsi);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_err(e, "scale");
  // U = Q Ws[:, :r] diag(sigma), V = B^T Ws[:, :r] diag(1 / sigma), each rounded once to bf16
  if ((e = gemm(Y, k, 1, Wsc, r, 1, nullptr, static_cast<uint16_t*>(U), ld_u, m, r, k)) != cudaSuccess)
    return cuda_err(e, "gemm U");
  if ((e = gemm(B, 1, n, Wsi, r, 1, nullptr, static_cast<uint16_t*>(V), ld_v, n, r, k)) != cudaSuccess)
    return cuda_err(e, "gemm V");
  int h_fail = 0;
  if ((e = cudaMemcpyAsync(&h_fail, fail, sizeof(int), cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return cuda_err(e, "aq_randomized_svd: synchronise");
  if (h_fail)
    return err(AQ_ERR_NUMERIC, "aq_randomized_svd: a Cholesky pivot was not positive: A Omega is rank deficient");
  return AQ_OK;
}
