// Blocked right-looking Cholesky (lower factor) and blocked inverse of a lower triangular
// matrix.  LASER Methodology 1 names S_x and S_g Cholesky factors of X and G; S_x is the
// transpose of the lower factor of X, S_g the lower factor of G.
//
// Cholesky, in column strips of CHOL_STRIP = 256:
//   * the strip (its 256 x 256 diagonal block and every row below) is factored by 64-wide
//     panels: one CTA factors and inverts each 64 x 64 diagonal block in shared memory
//     (chol_diag_kernel); the panel below becomes A21 L11^-T and the rest of the strip gets
//     its rank-64 update, both float32 SIMT GEMMs on tall, narrow operands;
//   * the trailing matrix gets A22 -= L21 L21^T (L21: the strip below its diagonal block,
//     K = 256) on the tensor cores: L21 split into three bfloat16 planes, the six cross terms
//     down to the last plane's weight summed in one launch, lower tiles only.
// A pivot <= 0 or not finite raises KF_ERR_NOT_SPD (detail: global pivot index) and the
// factorisation continues with a unit pivot so that no NaN or infinity spreads.
//
// Inverse M = L^-1: the 256 x 256 diagonal blocks by 64-row steps from the diagonal inverses
// of the factorisation (SIMT), then doubling levels h = 256, 512, ...: for adjacent blocks
// B1 = [i, i + h), B2 = [i + h, i + 2h), M[B2][B1] = -M[B2][B2] (L[B2][B1] M[B1][B1]), two
// triangular-aware tensor-core products with three-plane operands.
#include "kf_internal.cuh"

namespace kf {
namespace {

constexpr int NB = CHOL_NB;

// Factors the nb x nb (nb <= 64) lower block at A in shared memory and writes its lower
// factor back (zeros above) and the inverse of that factor to dinv (NB columns, row-major).
// Column j: every thread takes the pivot from a[j][j], the threads of rows below scale
// column j into L (one IEEE division per entry), then after a barrier the trailing lower
// triangle gets its rank-1 update from L's column (thread (ty, tx): rows j + 1 + ty + 4 i,
// column j + 1 + tx).  The inverse solves L X = I for all columns at once: step k scales row
// k of X, then updates the rows below with it.
__global__ void __launch_bounds__(256) chol_diag_kernel(float* __restrict__ A, int64_t lda, int nb,
                                                        float* __restrict__ dinv, int* status, int64_t k0) {
  __shared__ float a[NB][NB + 1];
  __shared__ float L[NB][NB + 1];
  const int t = threadIdx.x, tx = t & 63, ty = t >> 6;
  for (int idx = t; idx < NB * NB; idx += blockDim.x) {
    const int i = idx / NB, j = idx % NB;
    const bool in = i < nb && j < nb && j <= i;
    a[i][j] = in ? A[int64_t(i) * lda + j] : 0.f;
    L[i][j] = 0.f;
  }
  __syncthreads();
  for (int j = 0; j < nb; ++j) {
    const float p = a[j][j];
    const bool bad = !(p > 0.f) || !isfinite(p);
    const float ljj = bad ? 1.f : sqrtf(p);
    if (t == 0) {
      if (bad) raise_status(status, KF_ERR_NOT_SPD, int(k0 + j));
      L[j][j] = ljj;
    }
    if (t > j && t < nb) L[t][j] = __fdiv_rn(a[t][j], ljj);
    __syncthreads();
    const int k = j + 1 + tx;
    if (k < nb) {
      const float lk = L[k][j];
      for (int i = k + ty; i < nb; i += 4) a[i][k] = fmaf(-L[i][j], lk, a[i][k]);
    }
    __syncthreads();
  }
  // X = L^-1 in `a` (its old contents are no longer needed): start from I; step k:
  // X[k][c] /= L[k][k] for c <= k, then X[i][c] -= L[i][k] X[k][c] for i > k, c <= k.
  for (int idx = t; idx < NB * NB; idx += blockDim.x) {
    const int i = idx / NB, c = idx % NB;
    a[i][c] = (i == c && i < nb) ? 1.f : 0.f;
  }
  __syncthreads();
  for (int k = 0; k < nb; ++k) {
    if (t <= k) a[k][t] = __fdiv_rn(a[k][t], L[k][k]);
    __syncthreads();
    if (tx <= k) {
      const float xk = a[k][tx];
      for (int i = k + 1 + ty; i < nb; i += 4) a[i][tx] = fmaf(-L[i][k], xk, a[i][tx]);
    }
    __syncthreads();
  }
  for (int idx = t; idx < nb * nb; idx += blockDim.x) {
    const int i = idx / nb, j = idx % nb;
    A[int64_t(i) * lda + j] = (j <= i) ? L[i][j] : 0.f;
  }
  for (int idx = t; idx < nb * NB; idx += blockDim.x) {
    const int i = idx / NB, c = idx % NB;
    dinv[int64_t(i) * NB + c] = (c < nb && c <= i) ? a[i][c] : 0.f;
  }
}

__global__ void zero_upper_kernel(float* __restrict__ A, int64_t lda, int64_t n) {
  const int64_t i = int64_t(blockIdx.y) * 16 + threadIdx.y;
  const int64_t j = int64_t(blockIdx.x) * 16 + threadIdx.x;
  if (i < n && j < n && j > i) A[i * lda + j] = 0.f;
}

// Factors the column strip of width w at A (its w x w diagonal block and the rows - w rows
// below) by 64-wide panels; dinv receives the 64 x 64 diagonal inverses (NB columns each).
kf_status chol_strip(kf_ctx* ctx, float* A, int64_t lda, int64_t rows, int64_t w, float* dinv, int64_t kbase,
                     cudaStream_t st) {
  for (int64_t j0 = 0; j0 < w; j0 += NB) {
    const int nb = int(w - j0 < NB ? w - j0 : NB);
    chol_diag_kernel<<<1, 256, 0, st>>>(A + j0 * lda + j0, lda, nb, dinv + j0 * NB, ctx->d_status, kbase + j0);
    note_launch();
    KF_CUDA(cudaGetLastError());
    const int64_t rb = rows - j0 - nb;
    if (rb <= 0) break;
    float* P = A + (j0 + nb) * lda + j0;
    GemmDesc g{};
    g.M = rb; g.N = nb; g.K = nb;
    g.A = P; g.lda = lda; g.trans_a = false;
    g.B = dinv + j0 * NB; g.ldb = NB; g.trans_b = true;   // (L11^-1)^T
    g.C = P; g.ldc = lda;
    g.alpha = 1.f; g.beta = 0.f; g.batch = 1;
    KF_TRY(simt_gemm(g, st));
    const int64_t wrem = w - j0 - nb;
    if (wrem <= 0) continue;
    GemmDesc h{};
    h.M = rb; h.N = wrem; h.K = nb;
    h.A = P; h.lda = lda; h.trans_a = false;
    h.B = P; h.ldb = lda; h.trans_b = true;
    h.C = A + (j0 + nb) * lda + (j0 + nb); h.ldc = lda;
    h.alpha = -1.f; h.beta = 1.f; h.out_mask = OUT_LOWER; h.batch = 1;
    KF_TRY(simt_gemm(h, st));
  }
  return KF_OK;
}

// M (n x n lower, zeros above already) = inverse of the lower triangular L by 64-row steps:
// M[i, 0:i] = -L_ii^-1 (L[i, 0:i] M[0:i, 0:i]) with the diagonal inverses from dinv.
kf_status trtri_simt(const float* L, int64_t ldl, int64_t n, const float* dinv, float* M, int64_t ldm, float* tmp,
                     cudaStream_t st) {
  for (int64_t i0 = 0; i0 < n; i0 += NB) {
    const int nb = int(n - i0 < NB ? n - i0 : NB);
    KF_TRY(launch_copy(dinv + i0 * NB, NB, M + i0 * ldm + i0, ldm, nb, nb, false, st));
    if (i0 == 0) continue;
    GemmDesc g{};
    g.M = nb; g.N = i0; g.K = i0;
    g.A = L + i0 * ldl; g.lda = ldl;
    g.B = M; g.ldb = ldm;
    g.C = tmp; g.ldc = i0;
    g.alpha = 1.f; g.beta = 0.f; g.krange = KR_GE_COL; g.batch = 1;
    KF_TRY(simt_gemm(g, st));
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

int64_t trtri_top_level(int64_t n) {  // largest doubling block h (0: none)
  int64_t h = 0;
  for (int64_t x = CHOL_STRIP; x < n; x *= 2) h = x;
  return h;
}

struct TrtriBufs {
  float* T;
  int64_t ldT;
  PlaneBuf l21, m11, t, m22;
};
size_t trtri_carve(Carve& cv, int64_t n, TrtriBufs& b) {
  const int64_t h = trtri_top_level(n);
  const int64_t hh = h > 0 ? h : 1;
  b.ldT = (hh + 7) / 8 * 8;
  b.T = cv.take<float>(size_t(hh) * b.ldT);
  b.l21 = take_planes(cv, hh, hh, 3);
  b.m11 = take_planes(cv, hh, hh, 3);
  b.t = take_planes(cv, hh, hh, 3);
  b.m22 = take_planes(cv, hh, hh, 3);
  return cv.off;
}

}  // namespace

size_t chol_workspace_bytes(int64_t n) {
  Carve cv(nullptr, 0, true);
  const int64_t r = n > CHOL_STRIP ? n - CHOL_STRIP : 1;
  take_planes(cv, r, CHOL_STRIP, 3);
  return cv.off + 256;
}

kf_status cholesky_lower(kf_ctx* ctx, float* A, int64_t lda, int64_t n, float* dinv, void* ws, size_t ws_bytes,
                         cudaStream_t st) {
  for (int64_t k0 = 0; k0 < n; k0 += CHOL_STRIP) {
    const int64_t w = n - k0 < CHOL_STRIP ? n - k0 : CHOL_STRIP;
    KF_TRY(chol_strip(ctx, A + k0 * lda + k0, lda, n - k0, w, dinv + k0 * NB, k0, st));
    const int64_t r = n - k0 - w;
    if (r <= 0) break;
    Carve cv(ws, ws_bytes, false);
    PlaneBuf pb = take_planes(cv, r, w, 3);
    if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "cholesky: workspace too small");
    Planes pl;
    KF_TRY(split_f32(A + (k0 + w) * lda + k0, lda, r, w, pb, &pl, st));
    ProductOpts o;
    o.accumulate = true;
    o.negate = true;
    o.lower = true;
    o.kchunk = 0;
    KF_TRY(tc_product(ctx, r, r, w, pl, false, pl, false, KR_FULL, A + (k0 + w) * lda + (k0 + w), lda, st, o));
  }
  dim3 grid(unsigned((n + 15) / 16), unsigned((n + 15) / 16));
  zero_upper_kernel<<<grid, dim3(16, 16), 0, st>>>(A, lda, n); note_launch();
  return check_cuda(cudaGetLastError(), "zero_upper launch");
}

size_t trtri_tmp_floats(int64_t n) { return size_t(NB) * size_t(n > 0 ? n : 1); }

size_t trtri_workspace_bytes(int64_t n) {
  Carve cv(nullptr, 0, true);
  TrtriBufs b;
  trtri_carve(cv, n, b);
  return cv.off + 256;
}

kf_status trtri_lower(kf_ctx* ctx, const float* L, int64_t ldl, int64_t n, const float* dinv, float* M, int64_t ldm,
                      float* tmp, void* ws, size_t ws_bytes, cudaStream_t st) {
  KF_CUDA(cudaMemset2DAsync(M, size_t(ldm) * sizeof(float), 0, size_t(n) * sizeof(float), size_t(n), st));
  // diagonal blocks of CHOL_STRIP (the 64-block inverses come from the factorisation)
  for (int64_t b0 = 0; b0 < n; b0 += CHOL_STRIP) {
    const int64_t bw = n - b0 < CHOL_STRIP ? n - b0 : CHOL_STRIP;
    KF_TRY(trtri_simt(L + b0 * ldl + b0, ldl, bw, dinv + b0 * NB, M + b0 * ldm + b0, ldm, tmp, st));
  }
  if (n <= CHOL_STRIP) return KF_OK;
  Carve cv(ws, ws_bytes, false);
  TrtriBufs b;
  trtri_carve(cv, n, b);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "trtri: workspace too small");
  for (int64_t h = CHOL_STRIP; h < n; h *= 2) {
    for (int64_t i = 0; i + h < n; i += 2 * h) {
      const int64_t h2 = n - i - h < h ? n - i - h : h;
      // T = L[B2][B1] M[B1][B1]   (M11 lower: column j needs k >= j)
      Planes pl, pm, pt, pm2;
      KF_TRY(split_f32(L + (i + h) * ldl + i, ldl, h2, h, b.l21, &pl, st));
      KF_TRY(split_f32(M + i * ldm + i, ldm, h, h, b.m11, &pm, st));
      KF_TRY(tc_product(ctx, h2, h, h, pl, false, pm, true, KR_GE_COL, b.T, b.ldT, st));
      // M[B2][B1] = -M[B2][B2] T   (M22 lower: row i needs k <= i)
      KF_TRY(split_f32(b.T, b.ldT, h2, h, b.t, &pt, st));
      KF_TRY(split_f32(M + (i + h) * ldm + (i + h), ldm, h2, h2, b.m22, &pm2, st));
      ProductOpts o;
      o.negate = true;
      KF_TRY(tc_product(ctx, h2, h, h2, pm2, false, pt, true, KR_LE_ROW, M + (i + h) * ldm + i, ldm, st, o));
    }
  }
  return KF_OK;
}

}  // namespace kf
