// Spectrum of the whitened weight through its Gram matrix (Swift-SVD 2A: one
// eigendecomposition of the aggregated covariance instead of repeated SVDs), by a blocked
// parallel cyclic Jacobi eigensolver:
//   * C (s x s, float32, padded to a multiple of 64) is cut into 32-wide blocks; a
//     round-robin tournament pairs the blocks so that every step visits nblk/2 disjoint
//     pairs and a sweep (nblk - 1 steps) visits every pair once;
//   * jac_solve: one CTA per pair loads the 64 x 64 problem [[C_II C_IJ][C_JI C_JJ]] into
//     shared memory and diagonalises it by threshold cyclic Jacobi (32 disjoint rotations per
//     round), accumulating the 64 x 64 orthogonal V_p;
//   * jac_apply: C <- P^T C P and Q <- Q P for the block-diagonal P = diag(V_p), as 64 x 64
//     tile products (only tiles with p <= q of C, mirrored);
//   * a sweep in which no pair had |c_pq| > tol * sqrt(c_pp c_qq) (entries below a float32
//     rounding floor count as zero) ends the iteration for that problem.
// The singular values are then the Rayleigh quotients sigma_i = ||W~ q_i|| / ||q_i||,
// evaluated on W~ rather than on C so that the Gram's rounding errors enter only at second
// order, sorted descending with their vectors.
#include "kf_internal.cuh"

#include <cfloat>
#include <vector>

namespace kf {
namespace {

constexpr int JB = 32, JP = 64, TS = 68;  // block, pair problem, smem row stride (floats)

__device__ __forceinline__ int rr_pos(int pos, int round, int n) {  // circle method
  return pos == 0 ? 0 : 1 + (pos - 1 + round) % (n - 1);
}

__device__ __forceinline__ int64_t gidx(int r, int b0, int b1) {  // pair-local -> global index
  return r < JB ? int64_t(b0) * JB + r : int64_t(b1) * JB + (r - JB);
}

// ----------------------------------------------------------------------- prepare
// Mirror the Gram's lower triangle, zero the padding, set Q = I.
__global__ void jac_prepare_kernel(float* __restrict__ Call, float* __restrict__ Qall, int64_t s,
                                   int64_t sp) {
  const int64_t u = blockIdx.y;
  float* C = Call + u * sp * sp;
  float* Q = Qall + u * sp * sp;
  const int64_t n = sp * sp;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t i = e / sp, j = e - i * sp;
    if (i < s && j < s) {
      if (j > i) C[e] = C[j * sp + i];
    } else {
      C[e] = 0.f;
    }
    Q[e] = (i == j) ? 1.f : 0.f;
  }
}

__global__ void jac_floor_kernel(const float* __restrict__ Call, int64_t sp, float* __restrict__ floorv,
                                 float floor_factor, int* __restrict__ conv, unsigned* __restrict__ off,
                                 int* __restrict__ sweeps) {
  __shared__ float red[256];
  const int64_t u = blockIdx.x;
  const float* C = Call + u * sp * sp;
  float m = 0.f;
  for (int64_t i = threadIdx.x; i < sp; i += blockDim.x) m = fmaxf(m, C[i * sp + i]);
  red[threadIdx.x] = m;
  __syncthreads();
  for (int s = 128; s; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + s]);
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    floorv[u] = floor_factor * FLT_EPSILON * red[0];
    conv[u] = red[0] > 0.f ? 0 : 1;  // an all-zero Gram is already diagonal
    off[u] = 0u;
    if (sweeps) sweeps[u] = 0;
  }
}

// ------------------------------------------------------------------------- solve
__global__ void __launch_bounds__(256) jac_solve_kernel(float* __restrict__ Call, int64_t sp, int nblk,
                                                        int step, float* __restrict__ Vall,
                                                        int* __restrict__ skipall,
                                                        const int* __restrict__ conv,
                                                        unsigned* __restrict__ offmax,
                                                        const float* __restrict__ floorv, float tol,
                                                        int max_inner) {
  __shared__ float A[JP][JP + 1];
  __shared__ float V[JP][JP + 1];
  __shared__ float rc[32], rs[32], rap[32], raq[32];
  __shared__ int rp[32], rq[32], ract[32];
  __shared__ float red[8];

  const int k = blockIdx.x, u = blockIdx.y, t = threadIdx.x;
  if (conv[u]) return;
  const int npairs = nblk / 2;
  const float* C = Call + int64_t(u) * sp * sp;
  const int b0 = rr_pos(k, step, nblk), b1 = rr_pos(nblk - 1 - k, step, nblk);
  for (int e = t; e < JP * JP; e += 256) {
    const int r = e >> 6, c = e & 63;
    A[r][c] = C[gidx(r, b0, b1) * sp + gidx(c, b0, b1)];
  }
  __syncthreads();
  const float flo = floorv[u];

  // Largest relative coupling between the two blocks.
  float m = 0.f;
  for (int e = t; e < JB * JB; e += 256) {
    const int r = e >> 5, c = JB + (e & 31);
    const float v = fabsf(A[r][c]);
    if (v > flo) {
      const float den = fmaxf(sqrtf(A[r][r] * A[c][c]), flo);
      m = fmaxf(m, v / den);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((t & 31) == 0) red[t >> 5] = m;
  __syncthreads();
  if (t == 0) {
    float mm = red[0];
    for (int w = 1; w < 8; ++w) mm = fmaxf(mm, red[w]);
    red[0] = mm;
    if (mm > 0.f) atomicMax(offmax + u, __float_as_uint(mm));
  }
  __syncthreads();
  int* skip = skipall + int64_t(u) * npairs;
  if (red[0] <= tol) {
    if (t == 0) skip[k] = 1;
    return;
  }

  for (int e = t; e < JP * JP; e += 256) V[e >> 6][e & 63] = ((e >> 6) == (e & 63)) ? 1.f : 0.f;
  __syncthreads();

  for (int sweep = 0; sweep < max_inner; ++sweep) {
    int rotated = 0;
    for (int r = 0; r < JP - 1; ++r) {
      int act = 0;
      if (t < 32) {
        const int p = rr_pos(t, r, JP), q = rr_pos(JP - 1 - t, r, JP);
        const float a = A[p][p], b = A[q][q], d = A[p][q];
        float c = 1.f, s = 0.f, td = 0.f;
        if (fabsf(d) > flo && fabsf(d) > tol * sqrtf(fmaxf(a * b, 0.f))) {
          const float tau = __fdiv_rn(b - a, 2.f * d);
          const float tt = copysignf(1.f, tau) / (fabsf(tau) + sqrtf(fmaf(tau, tau, 1.f)));
          c = 1.0f / sqrtf(fmaf(tt, tt, 1.f));
          s = tt * c;
          td = tt * d;
          act = 1;
        }
        rc[t] = c; rs[t] = s; rp[t] = p; rq[t] = q; ract[t] = act;
        rap[t] = a - td; raq[t] = b + td;
      }
      if (!__syncthreads_or(act)) continue;
      rotated = 1;
      // Columns: A <- A J, V <- V J.
      for (int e = t; e < 2 * 32 * JP; e += 256) {
        const int mat = e >> 11, rem = e & 2047, j = rem >> 6, i = rem & 63;
        if (!ract[j]) continue;
        const int p = rp[j], q = rq[j];
        const float c = rc[j], s = rs[j];
        float (*M)[JP + 1] = mat ? V : A;
        const float x = M[i][p], y = M[i][q];
        M[i][p] = c * x - s * y;
        M[i][q] = s * x + c * y;
      }
      __syncthreads();
      // Rows: A <- J^T A, with the rotated 2 x 2 block set exactly.
      for (int e = t; e < 32 * JP; e += 256) {
        const int j = e >> 6, i = e & 63;
        if (!ract[j]) continue;
        const int p = rp[j], q = rq[j];
        if (i == p) {
          A[p][p] = rap[j];
          A[q][p] = 0.f;
        } else if (i == q) {
          A[p][q] = 0.f;
          A[q][q] = raq[j];
        } else {
          const float c = rc[j], s = rs[j];
          const float x = A[p][i], y = A[q][i];
          A[p][i] = c * x - s * y;
          A[q][i] = s * x + c * y;
        }
      }
      __syncthreads();
    }
    if (!rotated) break;
  }
  // One Newton-Schulz step V <- V (3I - V^T V) / 2 removes the orthogonality drift that the
  // rounding of many plane rotations leaves in V (A is free now: the apply step rebuilds C).
  for (int e = t; e < JP * JP; e += 256) {
    const int i = e >> 6, j = e & 63;
    float acc = 0.f;
#pragma unroll 8
    for (int k = 0; k < JP; ++k) acc = fmaf(V[k][i], V[k][j], acc);
    A[i][j] = (i == j ? 1.5f : 0.f) - 0.5f * acc;
  }
  __syncthreads();
  float vout[JP * JP / 256];
#pragma unroll
  for (int x = 0; x < JP * JP / 256; ++x) {
    const int e = t + x * 256, i = e >> 6, j = e & 63;
    float acc = 0.f;
#pragma unroll 8
    for (int k = 0; k < JP; ++k) acc = fmaf(V[i][k], A[k][j], acc);
    vout[x] = acc;
  }
  __syncthreads();
#pragma unroll
  for (int x = 0; x < JP * JP / 256; ++x) {
    const int e = t + x * 256;
    V[e >> 6][e & 63] = vout[x];
  }
  __syncthreads();
  float* Vo = Vall + (int64_t(u) * npairs + k) * (JP * JP);
  for (int e = t; e < JP * JP; e += 256) Vo[e] = V[e >> 6][e & 63];
  if (t == 0) skip[k] = 0;
}

// ------------------------------------------------------------------------- apply
// 64 x 64 x 64 product out = X^T-stored-as-rows * Y: out[i][j] = sum_k Xt[k][i] * Y[k][j].
__device__ __forceinline__ void mm64(const float (*Xt)[TS], const float (*Y)[TS], float acc[4][4], int tx,
                                     int ty) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
  for (int k = 0; k < JP; ++k) {
    const float4 x = *reinterpret_cast<const float4*>(&Xt[k][ty * 4]);
    const float4 y = *reinterpret_cast<const float4*>(&Y[k][tx * 4]);
    const float xa[4] = {x.x, x.y, x.z, x.w}, yb[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(xa[a], yb[b], acc[a][b]);
  }
}

__global__ void __launch_bounds__(256) jac_apply_kernel(float* __restrict__ Call, float* __restrict__ Qall,
                                                        int64_t sp, int nblk, int step,
                                                        const float* __restrict__ Vall,
                                                        const int* __restrict__ skipall,
                                                        const int* __restrict__ conv, int ntile_c,
                                                        unsigned long long* __restrict__ flops) {
  extern __shared__ __align__(16) float sm[];
  float (*Xt)[TS] = reinterpret_cast<float (*)[TS]>(sm);
  float (*Va)[TS] = reinterpret_cast<float (*)[TS]>(sm + JP * TS);
  float (*Vb)[TS] = reinterpret_cast<float (*)[TS]>(sm + 2 * JP * TS);
  float (*Ub)[TS] = reinterpret_cast<float (*)[TS]>(sm + 3 * JP * TS);

  const int u = blockIdx.y, t = threadIdx.x, tx = t & 15, ty = t >> 4;
  if (conv[u]) return;
  const int npairs = nblk / 2;
  const int* skip = skipall + int64_t(u) * npairs;
  const float* Vu = Vall + int64_t(u) * npairs * (JP * JP);
  float* C = Call + int64_t(u) * sp * sp;
  float* Q = Qall + int64_t(u) * sp * sp;
  int task = blockIdx.x;

  if (task < ntile_c) {
    int p = 0;
    while (task >= npairs - p) { task -= npairs - p; ++p; }
    const int q = p + task;
    const int sp_ = skip[p], sq = skip[q];
    if (sp_ && sq) return;
    if (flops && t == 0) atomicAdd(flops, (unsigned long long)((sp_ ? 0 : 1) + (sq ? 0 : 1)) * 2ull * JP * JP * JP);
    const int p0 = rr_pos(p, step, nblk), p1 = rr_pos(nblk - 1 - p, step, nblk);
    const int q0 = rr_pos(q, step, nblk), q1 = rr_pos(nblk - 1 - q, step, nblk);
    // Xt = T^T where T = C[rows of pair p, cols of pair q].
    for (int e = t; e < JP * JP; e += 256) {
      const int i = e >> 6, c = e & 63;
      Xt[c][i] = C[gidx(i, p0, p1) * sp + gidx(c, q0, q1)];
      if (!sq) Vb[i][c] = Vu[int64_t(q) * JP * JP + e];
      if (!sp_) Va[i][c] = Vu[int64_t(p) * JP * JP + e];
    }
    __syncthreads();
    float acc[4][4];
    if (!sq) {
      mm64(Xt, Vb, acc, tx, ty);  // U = T Vq
    } else {
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = Xt[tx * 4 + b][ty * 4 + a];
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
      *reinterpret_cast<float4*>(&Ub[ty * 4 + a][tx * 4]) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    __syncthreads();
    if (!sp_) {
      mm64(Va, Ub, acc, tx, ty);  // T' = Vp^T U
    }
    // acc holds T' (rows ty*4+a, cols tx*4+b); stage it for the mirrored write.
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = ty * 4 + a;
      const int64_t gr = gidx(i, p0, p1);
      const int64_t gc = gidx(tx * 4, q0, q1);
      *reinterpret_cast<float4*>(&C[gr * sp + gc]) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
      *reinterpret_cast<float4*>(&Xt[i][tx * 4]) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    }
    if (p != q) {
      __syncthreads();
      for (int e = t; e < JP * JP; e += 256) {
        const int a = e >> 6, b = e & 63;  // mirrored tile row a (pair q), col b (pair p)
        C[gidx(a, q0, q1) * sp + gidx(b, p0, p1)] = Xt[b][a];
      }
    }
    return;
  }

  // Q panel: rows rp*64..+63, columns of pair q.
  task -= ntile_c;
  const int rp = task / npairs, q = task - (task / npairs) * npairs;
  if (skip[q]) return;
  if (flops && t == 0) atomicAdd(flops, 2ull * JP * JP * JP);
  const int q0 = rr_pos(q, step, nblk), q1 = rr_pos(nblk - 1 - q, step, nblk);
  for (int e = t; e < JP * JP; e += 256) {
    const int i = e >> 6, c = e & 63;
    Xt[c][i] = Q[(int64_t(rp) * JP + i) * sp + gidx(c, q0, q1)];
    Vb[i][c] = Vu[int64_t(q) * JP * JP + e];
  }
  __syncthreads();
  float acc[4][4];
  mm64(Xt, Vb, acc, tx, ty);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int64_t gr = int64_t(rp) * JP + ty * 4 + a;
    const int64_t gc = gidx(tx * 4, q0, q1);
    *reinterpret_cast<float4*>(&Q[gr * sp + gc]) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
  }
}

__global__ void jac_check_kernel(int n_units, int* __restrict__ conv, unsigned* __restrict__ off, float tol,
                                 int sweep, int max_sweeps, int* __restrict__ sweeps, int* status) {
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) {
    if (conv[u]) continue;
    const float o = __uint_as_float(off[u]);
    off[u] = 0u;
    if (sweeps) sweeps[u] = sweep + 1;
    if (o <= tol) {
      conv[u] = 1;
    } else if (sweep + 1 == max_sweeps) {
      raise_status(status, KF_ERR_NO_CONVERGENCE, u);
    }
  }
}

// ------------------------------------------------------------- Rayleigh + sort
// sig2[j] = sum_i Y[i][j]^2 / sum_i Q[i][j]^2 (float64 sums), per column.
__global__ void col_norms_kernel(const float* __restrict__ Y, int64_t ldy, int64_t rows_y,
                                 const float* __restrict__ Q, int64_t ldq, int64_t rows_q, int64_t s,
                                 float* __restrict__ sigma, float* __restrict__ qinv) {
  const int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= s) return;
  double a = 0.0, b = 0.0;
  for (int64_t i = 0; i < rows_y; ++i) {
    const double v = Y[i * ldy + j];
    a += v * v;
  }
  for (int64_t i = 0; i < rows_q; ++i) {
    const double v = Q[i * ldq + j];
    b += v * v;
  }
  sigma[j] = b > 0.0 ? float(sqrt(a / b)) : 0.f;
  qinv[j] = b > 0.0 ? float(1.0 / sqrt(b)) : 0.f;
}

// One CTA per problem: bitonic sort of (sigma, index) by sigma descending, index ascending.
__global__ void __launch_bounds__(1024) sort_desc_kernel(const float* __restrict__ sig_in, int64_t s, int P,
                                                          int* __restrict__ perm_out, int64_t perm_stride) {
  extern __shared__ __align__(16) unsigned char sbuf[];
  float* key = reinterpret_cast<float*>(sbuf);
  int* idx = reinterpret_cast<int*>(sbuf + sizeof(float) * P);
  const int64_t u = blockIdx.x;
  const float* sig = sig_in + u * s;
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    key[i] = i < s ? sig[i] : -INFINITY;
    idx[i] = i;
  }
  __syncthreads();
  for (int kk = 2; kk <= P; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const int l = i ^ j;
        if (l > i) {
          const float ki = key[i], kl = key[l];
          const int ii = idx[i], il = idx[l];
          const bool l_before_i = kl > ki || (kl == ki && il < ii);
          const bool i_before_l = ki > kl || (ki == kl && ii < il);
          const bool up = (i & kk) == 0;
          if (up ? l_before_i : i_before_l) {
            key[i] = kl; key[l] = ki;
            idx[i] = il; idx[l] = ii;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < s; i += blockDim.x) perm_out[u * perm_stride + i] = idx[i];
}

__global__ void gather_kernel(const float* __restrict__ Q, int64_t ldq, int64_t s, const int* __restrict__ perm,
                              const float* __restrict__ sig, const float* __restrict__ qinv,
                              float* __restrict__ vecs, int64_t ldv, float* __restrict__ sigma_out) {
  const int64_t n = s * s;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = e / s, i = e - r * s;
    const int j = perm[i];
    vecs[r * ldv + i] = Q[r * ldq + j] * qinv[j];
    if (r == 0) sigma_out[i] = sig[j];
  }
}

}  // namespace

struct JacPlan {
  int64_t s, sp;
  int nblk, npairs;
};

static JacPlan jac_plan(int64_t s) {
  JacPlan p;
  p.s = s;
  p.sp = (s + JP - 1) / JP * JP;
  p.nblk = int(p.sp / JB);
  p.npairs = p.nblk / 2;
  return p;
}

static size_t svd_carve(Carve& cv, int nu, int64_t m_max, int64_t n_max, int64_t s, float** C, float** Q,
                        float** V, int** skip, int** conv, unsigned** off, float** flo, float** Y,
                        float** sig, float** qinv, int** perm) {
  const JacPlan pl = jac_plan(s);
  *C = cv.take<float>(size_t(nu) * pl.sp * pl.sp);
  *Q = cv.take<float>(size_t(nu) * pl.sp * pl.sp);
  *V = cv.take<float>(size_t(nu) * pl.npairs * JP * JP);
  *skip = cv.take<int>(size_t(nu) * pl.npairs);
  *conv = cv.take<int>(nu);
  *off = cv.take<unsigned>(nu);
  *flo = cv.take<float>(nu);
  *Y = cv.take<float>(size_t(m_max > n_max ? m_max : n_max) * s);
  *sig = cv.take<float>(size_t(nu) * s);
  *qinv = cv.take<float>(size_t(nu) * s);
  *perm = cv.take<int>(size_t(nu) * s);
  return cv.off;
}

size_t svd_workspace(int32_t nu, int64_t m_max, int64_t n_max, int64_t s) {
  Carve cv(nullptr, 0, true);
  float *C, *Q, *V, *flo, *Y, *sig, *qinv;
  int *skip, *conv, *perm;
  unsigned* off;
  return svd_carve(cv, nu, m_max, n_max, s, &C, &Q, &V, &skip, &conv, &off, &flo, &Y, &sig, &qinv, &perm) + 256;
}

kf_status svd_run(kf_ctx* ctx, int32_t nu, const kf_svd_problem* pr, float tol, int32_t max_sweeps, void* ws,
                  size_t ws_bytes, cudaStream_t st) {
  int64_t s = pr[0].m < pr[0].n ? pr[0].m : pr[0].n, m_max = 0, n_max = 0;
  for (int i = 0; i < nu; ++i) {
    m_max = pr[i].m > m_max ? pr[i].m : m_max;
    n_max = pr[i].n > n_max ? pr[i].n : n_max;
  }
  const JacPlan pl = jac_plan(s);
  Carve cv(ws, ws_bytes, false);
  float *C, *Q, *V, *flo, *Y, *sig, *qinv;
  int *skip, *conv, *perm;
  unsigned* off;
  svd_carve(cv, nu, m_max, n_max, s, &C, &Q, &V, &skip, &conv, &off, &flo, &Y, &sig, &qinv, &perm);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "whitened_svd: workspace too small");

  const bool prof = ctx->prof_enabled;
  unsigned long long* flops = prof ? ctx->prof_flops() : nullptr;
  if (prof) {
    for (int e = 0; e < 5; ++e)
      if (!ctx->prof_ev[e]) KF_CUDA(cudaEventCreate(&ctx->prof_ev[e]));
    KF_CUDA(cudaMemsetAsync(flops, 0, sizeof(unsigned long long), st));
    KF_CUDA(cudaEventRecord(ctx->prof_ev[0], st));
    ctx->prof_steps = int64_t(max_sweeps) * (pl.nblk - 1);
    ctx->prof_valid = true;
  }
  // Gram of the smaller side, lower triangle, float32 SIMT (accuracy matters here).
  for (int i = 0; i < nu; ++i) {
    const kf_svd_problem& p = pr[i];
    GemmDesc g{};
    g.M = s; g.N = s; g.batch = 1;
    g.C = C + int64_t(i) * pl.sp * pl.sp; g.ldc = pl.sp;
    g.alpha = 1.f; g.beta = 0.f; g.out_mask = OUT_LOWER;
    if (kf_gram_side(p.m, p.n) == KF_SIDE_RIGHT) {  // W~^T W~
      g.K = p.m;
      g.A = p.Wt; g.lda = p.ldw; g.trans_a = true;
      g.B = p.Wt; g.ldb = p.ldw; g.trans_b = false;
    } else {  // W~ W~^T
      g.K = p.n;
      g.A = p.Wt; g.lda = p.ldw; g.trans_a = false;
      g.B = p.Wt; g.ldb = p.ldw; g.trans_b = true;
    }
    KF_TRY(simt_gemm(g, st));
  }
  {
    dim3 grid(unsigned((pl.sp * pl.sp + 255) / 256 > 4096 ? 4096 : (pl.sp * pl.sp + 255) / 256), unsigned(nu));
    jac_prepare_kernel<<<grid, 256, 0, st>>>(C, Q, s, pl.sp); note_launch();
    KF_CUDA(cudaGetLastError());
    int* sweeps_tmp = nullptr;
    jac_floor_kernel<<<nu, 256, 0, st>>>(C, pl.sp, flo, 8.0f, conv, off, sweeps_tmp); note_launch();
    KF_CUDA(cudaGetLastError());
  }
  // Per-problem sweep counters (copied to the callers' pointers after the sweeps).
  int* sweeps_dev = perm;  // reuse: perm is rewritten by the sort afterwards
  KF_CUDA(cudaMemsetAsync(sweeps_dev, 0, sizeof(int) * nu, st));

  const int ntile_c = pl.npairs * (pl.npairs + 1) / 2;
  const int ntile_q = int(pl.sp / JP) * pl.npairs;
  const size_t apply_smem = size_t(4) * JP * TS * sizeof(float);
  static bool attr = false;
  if (!attr) {
    KF_CUDA(cudaFuncSetAttribute(jac_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(apply_smem)));
    attr = true;
  }
  const int max_inner = 12;
  if (prof) KF_CUDA(cudaEventRecord(ctx->prof_ev[1], st));
  for (int sw = 0; sw < max_sweeps; ++sw) {
    for (int step = 0; step < pl.nblk - 1; ++step) {
      jac_solve_kernel<<<dim3(pl.npairs, nu), 256, 0, st>>>(C, pl.sp, pl.nblk, step, V, skip, conv, off, flo, tol,
                                                           max_inner); note_launch();
      KF_CUDA(cudaGetLastError());
      jac_apply_kernel<<<dim3(ntile_c + ntile_q, nu), 256, apply_smem, st>>>(C, Q, pl.sp, pl.nblk, step, V, skip,
                                                                             conv, ntile_c, flops); note_launch();
      KF_CUDA(cudaGetLastError());
    }
    jac_check_kernel<<<1, 256, 0, st>>>(nu, conv, off, tol, sw, max_sweeps, sweeps_dev, ctx->d_status); note_launch();
    KF_CUDA(cudaGetLastError());
  }
  if (prof) KF_CUDA(cudaEventRecord(ctx->prof_ev[2], st));
  for (int i = 0; i < nu; ++i)
    if (pr[i].sweeps) KF_CUDA(cudaMemcpyAsync(pr[i].sweeps, sweeps_dev + i, sizeof(int), cudaMemcpyDeviceToDevice, st));

  // Rayleigh quotients on W~ itself, then sort and gather.
  int P = 1;
  while (P < s) P <<= 1;
  const size_t sort_smem = size_t(P) * 8;
  if (sort_smem > 227 * 1024) return fail(KF_ERR_UNSUPPORTED, "whitened_svd: s too large for the in-CTA sort");
  static bool sattr = false;
  if (!sattr) {
    KF_CUDA(cudaFuncSetAttribute(sort_desc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024));
    sattr = true;
  }
  for (int i = 0; i < nu; ++i) {
    const kf_svd_problem& p = pr[i];
    const float* Qi = Q + int64_t(i) * pl.sp * pl.sp;
    const bool right = kf_gram_side(p.m, p.n) == KF_SIDE_RIGHT;
    const int64_t rows_y = right ? p.m : p.n;
    GemmDesc g{};
    g.M = rows_y; g.N = s; g.K = s; g.batch = 1;
    g.A = p.Wt; g.lda = p.ldw; g.trans_a = !right;   // W~ (m x n) or W~^T
    g.B = Qi; g.ldb = pl.sp;
    g.C = Y; g.ldc = s;
    g.alpha = 1.f; g.beta = 0.f;
    KF_TRY(simt_gemm(g, st));
    col_norms_kernel<<<unsigned((s + 127) / 128), 128, 0, st>>>(Y, s, rows_y, Qi, pl.sp, s, s, sig + int64_t(i) * s,
                                                                qinv + int64_t(i) * s); note_launch();
    KF_CUDA(cudaGetLastError());
  }
  if (prof) KF_CUDA(cudaEventRecord(ctx->prof_ev[3], st));
  sort_desc_kernel<<<unsigned(nu), 1024, sort_smem, st>>>(sig, s, P, perm, s); note_launch();
  KF_CUDA(cudaGetLastError());
  for (int i = 0; i < nu; ++i) {
    const kf_svd_problem& p = pr[i];
    int64_t n = s * s, blocks = (n + 255) / 256;
    if (blocks > 148 * 16) blocks = 148 * 16;
    gather_kernel<<<unsigned(blocks), 256, 0, st>>>(Q + int64_t(i) * pl.sp * pl.sp, pl.sp, s, perm + int64_t(i) * s,
                                                    sig + int64_t(i) * s, qinv + int64_t(i) * s, p.vecs, p.ldv,
                                                    p.sigma); note_launch();
    KF_CUDA(cudaGetLastError());
  }
  if (prof) KF_CUDA(cudaEventRecord(ctx->prof_ev[4], st));
  return KF_OK;
}

kf_status svd_profile_read(kf_ctx* ctx, kf_svd_profile* out) {
  if (!ctx->prof_valid) return fail(KF_ERR_INVALID, "kf_svd_profile_read: no profiled whitened_svd call");
  KF_CUDA(cudaEventSynchronize(ctx->prof_ev[4]));
  float t[4];
  for (int i = 0; i < 4; ++i) KF_CUDA(cudaEventElapsedTime(&t[i], ctx->prof_ev[i], ctx->prof_ev[i + 1]));
  unsigned long long f = 0;
  KF_CUDA(cudaMemcpy(&f, ctx->prof_flops(), sizeof(f), cudaMemcpyDeviceToHost));
  out->gram_ms = t[0];
  out->jacobi_ms = t[1];
  out->rayleigh_ms = t[2];
  out->sort_ms = t[3];
  out->jacobi_steps = ctx->prof_steps;
  out->jacobi_apply_flops = double(f);
  return KF_OK;
}

}  // namespace kf
