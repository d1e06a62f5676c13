// Blocked right-looking Cholesky (lower factor) and blocked inverse of a lower triangular
// matrix.  LASER Methodology 1 names S_x and S_g Cholesky factors of X and G; S_x is the
// transpose of the lower factor of X, S_g the lower factor of G.
//
// Each 64-wide panel: the diagonal block is factored in shared memory by one CTA, which
// also inverts it; the panel below is L21 = A21 L11^-T (a GEMM with the inverse); the
// trailing matrix gets A22 -= L21 L21^T on its lower triangle.  A pivot <= 0 or not finite
// raises KF_ERR_NOT_SPD (detail: global pivot index) and the factorisation continues with
// a unit pivot so that no NaN or infinity spreads.
#include "kf_internal.cuh"

namespace kf {
namespace {

constexpr int NB = CHOL_NB;

__global__ void __launch_bounds__(256) chol_diag_kernel(float* __restrict__ A, int64_t lda, int nb,
                                                        float* __restrict__ dinv, int* status,
                                                        int64_t k0) {
  __shared__ float a[NB][NB + 1];
  __shared__ float inv[NB][NB + 1];
  const int t = threadIdx.x;
  for (int idx = t; idx < nb * nb; idx += blockDim.x) {
    const int i = idx / nb, j = idx % nb;
    a[i][j] = (j <= i) ? A[int64_t(i) * lda + j] : 0.f;
  }
  __syncthreads();
  for (int j = 0; j < nb; ++j) {
    if (t == 0) {
      const float p = a[j][j];
      float r;
      if (!(p > 0.f) || !isfinite(p)) {
        raise_status(status, KF_ERR_NOT_SPD, int(k0 + j));
        r = 1.f;
      } else {
        r = sqrtf(p);
      }
      a[j][j] = r;
    }
    __syncthreads();
    const float ljj = a[j][j];
    for (int i = j + 1 + t; i < nb; i += blockDim.x) a[i][j] = __fdiv_rn(a[i][j], ljj);
    __syncthreads();
    const int rem = nb - j - 1;
    for (int idx = t; idx < rem * rem; idx += blockDim.x) {
      const int i = j + 1 + idx / rem, k = j + 1 + idx % rem;
      if (k <= i) a[i][k] = fmaf(-a[i][j], a[k][j], a[i][k]);
    }
    __syncthreads();
  }
  // Inverse of the lower factor: column c solves L x = e_c by forward substitution.
  if (t < nb) {
    const int c = t;
    for (int i = 0; i < nb; ++i) inv[i][c] = 0.f;
    inv[c][c] = 1.0f / a[c][c];
    for (int i = c + 1; i < nb; ++i) {
      float s = 0.f;
      for (int k = c; k < i; ++k) s = fmaf(a[i][k], inv[k][c], s);
      inv[i][c] = __fdiv_rn(-s, a[i][i]);
    }
  }
  __syncthreads();
  for (int idx = t; idx < nb * nb; idx += blockDim.x) {
    const int i = idx / nb, j = idx % nb;
    A[int64_t(i) * lda + j] = (j <= i) ? a[i][j] : 0.f;
  }
  for (int idx = t; idx < nb * NB; idx += blockDim.x) {
    const int i = idx / NB, j = idx % NB;
    dinv[int64_t(i) * NB + j] = (j < nb && j <= i) ? inv[i][j] : 0.f;
  }
}

__global__ void zero_upper_kernel(float* __restrict__ A, int64_t lda, int64_t n) {
  const int64_t i = int64_t(blockIdx.y) * 16 + threadIdx.y;
  const int64_t j = int64_t(blockIdx.x) * 16 + threadIdx.x;
  if (i < n && j < n && j > i) A[i * lda + j] = 0.f;
}

}  // namespace

kf_status cholesky_lower(kf_ctx* ctx, float* A, int64_t lda, int64_t n, float* dinv,
                         cudaStream_t st) {
  for (int64_t k0 = 0; k0 < n; k0 += NB) {
    const int nb = int(n - k0 < NB ? n - k0 : NB);
    chol_diag_kernel<<<1, 256, 0, st>>>(A + k0 * lda + k0, lda, nb, dinv + k0 * NB, ctx->d_status, k0); note_launch();
    KF_CUDA(cudaGetLastError());
    const int64_t r = n - k0 - nb;
    if (r <= 0) break;
    float* P = A + (k0 + nb) * lda + k0;
    GemmDesc g{};
    g.M = r; g.N = nb; g.K = nb;
    g.A = P; g.lda = lda; g.trans_a = false;
    g.B = dinv + k0 * NB; g.ldb = NB; g.trans_b = true;   // (L11^-1)^T
    g.C = P; g.ldc = lda;
    g.alpha = 1.f; g.beta = 0.f; g.batch = 1;
    KF_TRY(simt_gemm(g, st));
    GemmDesc h{};
    h.M = r; h.N = r; h.K = nb;
    h.A = P; h.lda = lda; h.trans_a = false;
    h.B = P; h.ldb = lda; h.trans_b = true;
    h.C = A + (k0 + nb) * lda + (k0 + nb); h.ldc = lda;
    h.alpha = -1.f; h.beta = 1.f; h.out_mask = OUT_LOWER; h.batch = 1;
    KF_TRY(simt_gemm(h, st));
  }
  dim3 grid(unsigned((n + 15) / 16), unsigned((n + 15) / 16));
  zero_upper_kernel<<<grid, dim3(16, 16), 0, st>>>(A, lda, n); note_launch();
  return check_cuda(cudaGetLastError(), "zero_upper launch");
}

size_t trtri_tmp_floats(int64_t n) { return size_t(NB) * size_t(n > 0 ? n : 1); }

kf_status trtri_lower(kf_ctx* ctx, const float* L, int64_t ldl, int64_t n, const float* dinv,
                      float* M, int64_t ldm, float* tmp, cudaStream_t st) {
  (void)ctx;
  KF_CUDA(cudaMemset2DAsync(M, size_t(ldm) * sizeof(float), 0, size_t(n) * sizeof(float), size_t(n), st));
  for (int64_t i0 = 0; i0 < n; i0 += NB) {
    const int nb = int(n - i0 < NB ? n - i0 : NB);
    // Diagonal block: the inverse of L_ii from the factorisation.
    KF_TRY(launch_copy(dinv + i0 * NB, NB, M + i0 * ldm + i0, ldm, nb, nb, false, st));
    if (i0 == 0) continue;
    // T = L[i, 0:i] * M[0:i, 0:i]   (M lower triangular: k >= column)
    GemmDesc g{};
    g.M = nb; g.N = i0; g.K = i0;
    g.A = L + i0 * ldl; g.lda = ldl;
    g.B = M; g.ldb = ldm;
    g.C = tmp; g.ldc = i0;
    g.alpha = 1.f; g.beta = 0.f; g.krange = KR_GE_COL; g.batch = 1;
    KF_TRY(simt_gemm(g, st));
    // M[i, 0:i] = -L_ii^-1 * T
    GemmDesc h{};
    h.M = nb; h.N = i0; h.K = nb;
    h.A = dinv + i0 * NB; h.lda = NB;
    h.B = tmp; h.ldb = i0;
    h.C = M + i0 * ldm; h.ldc = ldm;
    h.alpha = -1.f; h.beta = 0.f; h.batch = 1;
    KF_TRY(simt_gemm(h, st));
  }
  return KF_OK;
}

}  // namespace kf
