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
//     tile products (only tiles with p <= q of C, mirrored; since C stays symmetric the
//     transposed operand is read from the mirrored tile).  Q is stored transposed (one
//     eigenvector per row), so Q P becomes P^T Qt, again without any transposition;
//   * a sweep in which no pair had |c_pq| > tol * sqrt(c_pp c_qq) (entries below a float32
//     rounding floor count as zero) ends the iteration for that problem.
// The singular values are then the Rayleigh quotients sigma_i = ||W~ q_i|| / ||q_i||,
// evaluated on W~ rather than on C so that the Gram's rounding errors enter only at second
// order, sorted descending with their vectors.
// The same solver serves a symmetric matrix given directly (Swift-SVD 2A's covariance of
// the layer output): the values are then the Rayleigh quotients q.Cq / q.q.
#include "kf_internal.cuh"

#include <cfloat>
#include <vector>

namespace kf {
namespace {

constexpr int JB = 32, JP = 64;  // block width, pair problem size
#ifndef KF_JAC_MAX_INNER
#define KF_JAC_MAX_INNER 12  // inner sweeps of a pair problem
#endif

// Alignment self-check for vector accesses: a misaligned address is recorded in the status
// word (KF_ERR_INVALID, info = site) and the access is skipped instead of faulting.
__device__ __forceinline__ bool aligned16(const void* p, int* st, int site) {
  if ((reinterpret_cast<uintptr_t>(p) & 15) == 0) return true;
  raise_status(st, KF_ERR_INVALID, site);
  return false;
}

// Circle method: the element at position pos in round `round` of a round-robin over n.
// Every caller has 0 <= pos < n and 0 <= round < n - 1, so pos - 1 + round < 2 (n - 1) and
// the reduction modulo n - 1 is one conditional subtraction.
__device__ __forceinline__ int rr_pos(int pos, int round, int n) {
  if (pos == 0) return 0;
  int v = pos - 1 + round;
  if (v >= n - 1) v -= n - 1;
  return 1 + v;
}

__device__ __forceinline__ int64_t gidx(int r, int b0, int b1) {  // pair-local -> global index
  return r < JB ? int64_t(b0) * JB + r : int64_t(b1) * JB + (r - JB);
}

// ----------------------------------------------------------------------- prepare
// Mirror the Gram's lower triangle, zero the padding, set Q = I (Q is kept transposed).
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
  // Row stride JP + 2: the 32 couplings A[p][q] that one rotation round reads lie on an
  // anti-diagonal (p + q constant), which a stride of JP + 1 would put in a single bank.
  __shared__ float A[JP][JP + 2];
  __shared__ float V[JP][JP + 1];
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
      const float den = fmaxf(sqrtf(fmaxf(A[r][r] * A[c][c], 0.f)), flo);
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

  // Threshold cyclic Jacobi on the 64 x 64 pair problem, 32 disjoint rotations per round.
  // Every warp computes all 32 rotations of a round (lane l: pair l) from the same entries,
  // so the parameters reach the threads that need them by warp shuffles rather than
  // through shared memory; thread (warp w, lane k) then updates the 2 x 2 blocks (j, k),
  // j = w, w + 8, w + 16, w + 24, and rows w, w + 8, ... of the columns p_k, q_k of V.
  const int lane = t & 31, warp = t >> 5;
  for (int sweep = 0; sweep < max_inner; ++sweep) {
    int rotated = 0;
    for (int r = 0; r < JP - 1; ++r) {
      const int p = rr_pos(lane, r, JP), q = rr_pos(JP - 1 - lane, r, JP);
      const float a = A[p][p], b = A[q][q], d = A[p][q];
      float c = 1.f, sn = 0.f, td = 0.f;
      int act = 0;
      if (fabsf(d) > flo && fabsf(d) > tol * sqrtf(fmaxf(a * b, 0.f))) {
        const float tau = __fdiv_rn(b - a, 2.f * d);
        const float tt = copysignf(1.f, tau) / (fabsf(tau) + sqrtf(fmaf(tau, tau, 1.f)));
        c = 1.0f / sqrtf(fmaf(tt, tt, 1.f));
        sn = tt * c;
        td = tt * d;
        act = 1;
      }
      // identical in every warp (same inputs), so the branch is uniform over the CTA
      if (!__any_sync(0xffffffffu, act)) continue;
      rotated = 1;
      __syncthreads();  // every warp has read the entries this round rewrites
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int j = warp + 8 * x;
        const int pj = __shfl_sync(0xffffffffu, p, j), qj = __shfl_sync(0xffffffffu, q, j);
        const float cj = __shfl_sync(0xffffffffu, c, j), sj = __shfl_sync(0xffffffffu, sn, j);
        const int actj = __shfl_sync(0xffffffffu, act, j);
        if (j == lane) {
          if (act) {
            A[p][p] = a - td;
            A[q][q] = b + td;
            A[p][q] = 0.f;
            A[q][p] = 0.f;
          }
          continue;
        }
        if (!actj && !act) continue;
        const float e00 = A[pj][p], e01 = A[pj][q], e10 = A[qj][p], e11 = A[qj][q];
        const float a1 = e00 * c - e01 * sn, b1 = e00 * sn + e01 * c;
        const float c1 = e10 * c - e11 * sn, d1 = e10 * sn + e11 * c;
        A[pj][p] = cj * a1 - sj * c1;
        A[pj][q] = cj * b1 - sj * d1;
        A[qj][p] = sj * a1 + cj * c1;
        A[qj][q] = sj * b1 + cj * d1;
      }
      if (act) {
#pragma unroll
        for (int y = 0; y < JP / 8; ++y) {
          const int i = warp + 8 * y;
          const float x0 = V[i][p], y0 = V[i][q];
          V[i][p] = c * x0 - sn * y0;
          V[i][q] = sn * x0 + c * y0;
        }
      }
      __syncthreads();
    }
    if (!rotated) break;
  }
  // Rounds without an active rotation have no barrier: every warp must have finished reading
  // A before it is reused as scratch below.
  __syncthreads();
#ifdef KF_JAC_SORT_PAIRS
  // Order the pair's eigenvectors by eigenvalue, largest first, so that the first block of
  // the pair receives the larger half of the pair's spectrum.
  __shared__ int pord[JP];
  if (t < JP) {
    const float di = A[t][t];
    int rank = 0;
    for (int j = 0; j < JP; ++j) {
      const float dj = A[j][j];
      rank += (dj > di) || (dj == di && j < t);
    }
    pord[rank] = t;
  }
  __syncthreads();
#endif
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
#ifdef KF_JAC_SORT_PAIRS
  for (int e = t; e < JP * JP; e += 256) {
    const int oc = pord[e & 63];
    Vo[e] = V[e >> 6][oc >= 0 && oc < JP ? oc : (e & 63)];
  }
#else
  for (int e = t; e < JP * JP; e += 256) Vo[e] = V[e >> 6][e & 63];
#endif
  if (t == 0) skip[k] = 0;
}

// ------------------------------------------------------------------------- apply
// 64 x 64 x 64 product out[i][j] = sum_k X[k][i] * Y[k][j] with X, Y dense row-major
// 64 x 64 in shared memory; thread (tx, ty) owns rows ty*4..+3, columns tx*4..+3.
__device__ __forceinline__ void mm64(const float* __restrict__ X, const float* __restrict__ Y, float acc[4][4],
                                     int tx, int ty) {
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 8
  for (int k = 0; k < JP; ++k) {
    const float4 x = *reinterpret_cast<const float4*>(X + k * JP + ty * 4);
    const float4 y = *reinterpret_cast<const float4*>(Y + k * JP + tx * 4);
    const float xa[4] = {x.x, x.y, x.z, x.w}, yb[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(xa[a], yb[b], acc[a][b]);
  }
}

__device__ __forceinline__ void cp_async16(float* smem_dst, const float* gsrc) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// One task of a Jacobi step: a tile of C (pair p rows x pair q columns, p <= q) or a
// 64-column panel cb of the transposed eigenvector matrix for pair q.
struct ApplyTask {
  int u, kind, p, q, cb, wp, wq;  // kind 0: C tile, 1: Qt panel; wp/wq: V_p, V_q are applied
};

__device__ __forceinline__ bool decode_apply(int g, int per_u, int ntile_c, int npairs, const int* __restrict__ skipall,
                                             const int* __restrict__ conv, ApplyTask& t) {
  t.u = g / per_u;
  int task = g - t.u * per_u;
  if (conv[t.u]) return false;
  const int* skip = skipall + int64_t(t.u) * npairs;
  if (task < ntile_c) {
    // Row p of the upper triangle (p <= q) holds npairs - p tiles; S(p) = p (2 npairs - p + 1) / 2
    // tiles precede it.  p = the largest row with S(p) <= task: the root of the quadratic,
    // then an exact integer correction (at most a step or two for npairs <= 256).
    const int n2 = 2 * npairs + 1;
    int p = int((float(n2) - sqrtf(float(n2) * float(n2) - 8.f * float(task))) * 0.5f);
    p = p < 0 ? 0 : (p > npairs - 1 ? npairs - 1 : p);
    while (p > 0 && p * (n2 - p) / 2 > task) --p;
    while (p + 1 < npairs && (p + 1) * (n2 - p - 1) / 2 <= task) ++p;
    task -= p * (n2 - p) / 2;
    t.kind = 0; t.p = p; t.q = p + task; t.cb = 0;
    t.wp = !skip[t.p]; t.wq = !skip[t.q];
    return t.wp || t.wq;
  }
  task -= ntile_c;
  t.kind = 1; t.cb = task / npairs; t.q = task - t.cb * npairs; t.p = t.q;
  t.wp = 0; t.wq = !skip[t.q];
  return t.wq != 0;
}

// Stage layout (floats): X (64 x 64) | Vp (64 x 64) | Vq (64 x 64).
constexpr int STAGE_F = 3 * JP * JP;

__device__ __forceinline__ void issue_apply_loads(const ApplyTask& t, float* stage, const float* __restrict__ Call,
                                                  const float* __restrict__ Qtall, const float* __restrict__ Vall,
                                                  int64_t sp, int nblk, int step, int npairs, int tid, int* st) {
  const float* C = Call + int64_t(t.u) * sp * sp;
  const float* Qt = Qtall + int64_t(t.u) * sp * sp;
  const float* Vu = Vall + int64_t(t.u) * npairs * (JP * JP);
  const int q0 = rr_pos(t.q, step, nblk), q1 = rr_pos(nblk - 1 - t.q, step, nblk);
  if (t.kind == 0) {
    const int p0 = rr_pos(t.p, step, nblk), p1 = rr_pos(nblk - 1 - t.p, step, nblk);
    // C stays symmetric, so X[k][i] = C[q_k][p_i] is the transpose of T = C[rows p][cols q].
    for (int e = tid; e < JP * JP / 4; e += 256) {
      const int k = e >> 4, c = (e & 15) * 4;
      const float* a = C + gidx(k, q0, q1) * sp + gidx(c, p0, p1);
      if (aligned16(a, st, 101)) cp_async16(stage + k * JP + c, a);
      const float* vp = Vu + int64_t(t.p) * JP * JP + 4 * e;
      const float* vq = Vu + int64_t(t.q) * JP * JP + 4 * e;
      if (t.wp && aligned16(vp, st, 102)) cp_async16(stage + JP * JP + 4 * e, vp);
      if (t.wq && aligned16(vq, st, 103)) cp_async16(stage + 2 * JP * JP + 4 * e, vq);
    }
  } else {
    for (int e = tid; e < JP * JP / 4; e += 256) {
      const int k = e >> 4, c = (e & 15) * 4;
      const float* a = Qt + gidx(k, q0, q1) * sp + int64_t(t.cb) * JP + c;
      const float* vq = Vu + int64_t(t.q) * JP * JP + 4 * e;
      if (aligned16(a, st, 104)) cp_async16(stage + k * JP + c, a);
      if (aligned16(vq, st, 105)) cp_async16(stage + 2 * JP * JP + 4 * e, vq);
    }
  }
}

// Persistent: each CTA walks the tasks of every problem (stride gridDim.x), prefetching the
// next task's three 16 KB operands with cp.async while it computes the current one.
__global__ void __launch_bounds__(256, 2) jac_apply_kernel(float* __restrict__ Call, float* __restrict__ Qtall,
                                                           int64_t sp, int nblk, int step,
                                                           const float* __restrict__ Vall,
                                                           const int* __restrict__ skipall,
                                                           const int* __restrict__ conv, int ntile_c, int per_u,
                                                           int total, unsigned long long* __restrict__ flops,
                                                           int* status) {
  extern __shared__ __align__(16) float sm[];
  float* stages[2] = {sm, sm + STAGE_F};
  float* Ub = sm + 2 * STAGE_F;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int npairs = nblk / 2;

  ApplyTask cur, nxt;
  int g = blockIdx.x;
  while (g < total && !decode_apply(g, per_u, ntile_c, npairs, skipall, conv, cur)) g += gridDim.x;
  if (g >= total) return;
  issue_apply_loads(cur, stages[0], Call, Qtall, Vall, sp, nblk, step, npairs, tid, status);
  cp_async_commit();
  int s = 0;
  unsigned long long done_flops = 0;
  while (true) {
    int gn = g + gridDim.x;
    while (gn < total && !decode_apply(gn, per_u, ntile_c, npairs, skipall, conv, nxt)) gn += gridDim.x;
    const bool more = gn < total;
    if (more) {
      issue_apply_loads(nxt, stages[s ^ 1], Call, Qtall, Vall, sp, nblk, step, npairs, tid, status);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* X = stages[s];
    const float* Vp = stages[s] + JP * JP;
    const float* Vq = stages[s] + 2 * JP * JP;
    float acc[4][4];
    const int q0 = rr_pos(cur.q, step, nblk), q1 = rr_pos(nblk - 1 - cur.q, step, nblk);
    if (cur.kind == 0) {
      float* C = Call + int64_t(cur.u) * sp * sp;
      const int p0 = rr_pos(cur.p, step, nblk), p1 = rr_pos(nblk - 1 - cur.p, step, nblk);
      if (cur.wq) {
        mm64(X, Vq, acc, tx, ty);  // U = T Vq
      } else {
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) acc[a][b] = X[(tx * 4 + b) * JP + ty * 4 + a];
      }
      if (cur.wp) {
#pragma unroll
        for (int a = 0; a < 4; ++a)
          *reinterpret_cast<float4*>(Ub + (ty * 4 + a) * JP + tx * 4) =
              make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        __syncthreads();
        mm64(Vp, Ub, acc, tx, ty);  // T' = Vp^T U
      }
      done_flops += (unsigned long long)(cur.wp + cur.wq) * 2ull * JP * JP * JP;
      // T' (rows ty*4+a, cols tx*4+b) -> C[rows p][cols q]; the mirrored tile gets T'^T,
      // which this thread holds as four contiguous runs of 4 (rows tx*4+b, cols ty*4..+3).
      if (cur.p != cur.q) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          float* d = C + gidx(ty * 4 + a, p0, p1) * sp + gidx(tx * 4, q0, q1);
          if (aligned16(d, status, 106)) *reinterpret_cast<float4*>(d) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          float* d = C + gidx(tx * 4 + b, q0, q1) * sp + gidx(ty * 4, p0, p1);
          if (aligned16(d, status, 107)) *reinterpret_cast<float4*>(d) = make_float4(acc[0][b], acc[1][b], acc[2][b], acc[3][b]);
        }
      } else {
        // Diagonal tile: keep it exactly symmetric by writing entries i <= j to (i, j) and (j, i).
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int i = ty * 4 + a, j = tx * 4 + b;
            if (i <= j) {
              C[gidx(i, p0, p1) * sp + gidx(j, p0, p1)] = acc[a][b];
              C[gidx(j, p0, p1) * sp + gidx(i, p0, p1)] = acc[a][b];
            }
          }
      }
    } else {
      float* Qt = Qtall + int64_t(cur.u) * sp * sp;
      mm64(Vq, X, acc, tx, ty);  // Qt[rows q][panel] <- Vq^T Qt[rows q][panel]
      done_flops += 2ull * JP * JP * JP;
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        float* d = Qt + gidx(ty * 4 + a, q0, q1) * sp + int64_t(cur.cb) * JP + tx * 4;
        if (aligned16(d, status, 108)) *reinterpret_cast<float4*>(d) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
      }
    }
    __syncthreads();  // the stage and Ub are rewritten by the next iteration's loads
    if (!more) break;
    cur = nxt;
    g = gn;
    s ^= 1;
  }
  if (flops && tid == 0 && done_flops) atomicAdd(flops, done_flops);
}

__global__ void jac_check_kernel(int n_units, int* __restrict__ conv, unsigned* __restrict__ off, float tol,
                                 int sweep, int max_sweeps, int* __restrict__ sweeps, int* status,
                                 int* __restrict__ all_conv) {
  int mine = 1;
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) {
    if (conv[u]) continue;
    const float o = __uint_as_float(off[u]);
    off[u] = 0u;
    if (sweeps) sweeps[u] = sweep + 1;
    if (o <= tol) {
      conv[u] = 1;
    } else {
      mine = 0;
      if (sweep + 1 == max_sweeps) raise_status(status, KF_ERR_NO_CONVERGENCE, u);
    }
  }
  const int all = __syncthreads_and(mine);
  if (threadIdx.x == 0) *all_conv = all;
}

// ------------------------------------------------------------- Rayleigh + sort
// sigma_j^2 = ||y_j||^2 / ||q_j||^2 with y_j = W~ q_j (right side) or W~^T q_j (left side):
// one CTA per vector j, float64 sums over row j of Yt and of Qt (both contiguous).
// dot != 0 (a symmetric matrix C given directly, y_j = C q_j): the Rayleigh quotient
// lambda_j = (q_j . y_j) / ||q_j||^2 instead (the first len_q entries of both rows).
__global__ void __launch_bounds__(256) rayleigh_norms_kernel(const float* __restrict__ Yt, int64_t ldy,
                                                             int64_t len_y, const float* __restrict__ Qt,
                                                             int64_t ldq, int64_t len_q,
                                                             float* __restrict__ sigma, float* __restrict__ qinv,
                                                             int* status, int dot) {
  __shared__ double ra[8], rb[8];
  const int64_t j = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  double a = 0.0, b = 0.0;
  if (dot) {
    for (int64_t i = threadIdx.x; i < len_q; i += blockDim.x) a += double(Yt[j * ldy + i]) * double(Qt[j * ldq + i]);
  } else {
    for (int64_t i = threadIdx.x; i < len_y; i += blockDim.x) {
      const double v = Yt[j * ldy + i];
      a += v * v;
    }
  }
  for (int64_t i = threadIdx.x; i < len_q; i += blockDim.x) {
    const double v = Qt[j * ldq + i];
    b += v * v;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if (lane == 0) { ra[w] = a; rb[w] = b; }
  __syncthreads();
  if (threadIdx.x == 0) {
    double aa = 0.0, bb = 0.0;
    for (int x = 0; x < 8; ++x) { aa += ra[x]; bb += rb[x]; }
    sigma[j] = bb > 0.0 ? float(dot ? aa / bb : sqrt(aa / bb)) : 0.f;
    qinv[j] = bb > 0.0 ? float(1.0 / sqrt(bb)) : 0.f;
    if (!isfinite(aa) || !isfinite(bb)) raise_status(status, KF_ERR_INVALID, 141);
  }
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
    const float v = i < s ? sig[i] : -INFINITY;
    key[i] = isnan(v) ? -INFINITY : v;  // padding and non-numbers sort last
    idx[i] = i < s ? i : P + i;         // padding after every real index on ties
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
  for (int i = threadIdx.x; i < s; i += blockDim.x) perm_out[u * perm_stride + i] = idx[i] < s ? idx[i] : 0;
}

// vecs[r][i] = Qt[perm[i]][r] * qinv[perm[i]] (column i of vecs = i-th sorted vector), as
// 32 x 32 tiles transposed through shared memory so that reads and writes are coalesced.
// sqrt_out: the sorted values are eigenvalues of a symmetric C; sigma_out gets sqrt(max(., 0)).
__global__ void gather_kernel(const float* __restrict__ Qt, int64_t ldq, int64_t s, const int* __restrict__ perm,
                              const float* __restrict__ sig, const float* __restrict__ qinv,
                              float* __restrict__ vecs, int64_t ldv, float* __restrict__ sigma_out, int sqrt_out) {
  __shared__ float tile[32][33];
  const int64_t i0 = int64_t(blockIdx.x) * 32, r0 = int64_t(blockIdx.y) * 32;
  for (int k = threadIdx.y; k < 32; k += 8) {
    const int64_t i = i0 + k, r = r0 + threadIdx.x;
    if (i < s && r < s) {
      const int j = perm[i];
      tile[k][threadIdx.x] = Qt[int64_t(j) * ldq + r] * qinv[j];
    }
  }
  __syncthreads();
  for (int k = threadIdx.y; k < 32; k += 8) {
    const int64_t r = r0 + k, i = i0 + threadIdx.x;
    if (r < s && i < s) vecs[r * ldv + i] = tile[threadIdx.x][k];
  }
  if (blockIdx.y == 0 && threadIdx.y == 0) {
    const int64_t i = i0 + threadIdx.x;
    if (i < s) {
      const float v = sig[perm[i]];
      sigma_out[i] = sqrt_out ? sqrtf(fmaxf(v, 0.f)) : v;
    }
  }
}

// ------------------------------------------------------ windowed Rayleigh-Ritz refinement
// The rounding of thousands of block rotations applied as 64-term products leaves the
// accumulated eigenvectors with couplings of order 1e-5 ||C|| to their neighbours in the
// spectrum, which the Rayleigh quotient turns into relative errors of order 1e-4 on the
// smaller kept singular values.  The refinement removes them: with the vectors sorted by
// Rayleigh value, every window of RW consecutive vectors gets the exact Gram of its images,
// B = Y_w Y_w^T (y_i = W~ q_i, float32 products summed in float64), which is diagonalised in
// shared memory; the window's q and y rows are rotated by the eigenvectors.  Two passes with
// windows offset by RW/2 leave every vector in the interior of one window; couplings to
// vectors outside the window only enter at second order, divided by large gaps.
constexpr int RW = 128;

// Dst[r][c] = Src[perm[r]][c] for r < s, zero rows for s <= r < rows; one CTA per row.
__global__ void gather_rows_kernel(const float* __restrict__ Src, int64_t lds, int64_t prob_src,
                                   const int* __restrict__ perm, int64_t s, float* __restrict__ Dst, int64_t ldd,
                                   int64_t prob_dst, int64_t cols) {
  const int64_t r = blockIdx.x, u = blockIdx.y;
  float* d = Dst + u * prob_dst + r * ldd;
  if (r >= s) {
    for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) d[c] = 0.f;
    return;
  }
  const float* src = Src + u * prob_src + int64_t(perm[u * s + r]) * lds;
  for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) d[c] = src[c];
}

// Loads rows [0, RW) x columns [k0, k0 + 32) of Y (ldy) transposed into T[k][i].
__device__ __forceinline__ void win_load_t(float (*T)[RW + 4], const float* __restrict__ Y, int64_t ldy,
                                           int64_t k0, int64_t cols, int t, int* status) {
  // 128 rows x 32 columns: lane-consecutive rows, so the transposed shared stores do not conflict
  for (int e = t; e < RW * 8; e += 256) {
    const int i = e & (RW - 1), kc = e >> 7;  // kc: 4-column chunk 0..7
    const int64_t k = k0 + kc * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (k + 3 < cols) {
      const float* a = Y + int64_t(i) * ldy + k;
      if (aligned16(a, status, 111)) v = *reinterpret_cast<const float4*>(a);
    } else {
      float tmp[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < 4; ++q)
        if (k + q < cols) tmp[q] = Y[int64_t(i) * ldy + k + q];
      v = make_float4(tmp[0], tmp[1], tmp[2], tmp[3]);
    }
    T[kc * 4 + 0][i] = v.x;
    T[kc * 4 + 1][i] = v.y;
    T[kc * 4 + 2][i] = v.z;
    T[kc * 4 + 3][i] = v.w;
  }
}

// B_w = Y_w Y_w^T for the RW rows of window w of problem u (rows start at off + w * RW):
// float32 products over k-blocks of 32 columns, block partial sums added in float64.
// With Xs != nullptr the cross product B_w = X_w Y_w^T instead (X_w the same rows of Xs):
// for a symmetric C given directly, X = the vectors and Y = their images C q, so B_w is the
// window's Rayleigh-Ritz matrix (symmetrised by the window eigensolver).
__global__ void __launch_bounds__(256) win_gram_kernel(const float* __restrict__ Ys, int64_t ldy, int64_t prob_y,
                                                       int64_t cols, int64_t off, float* __restrict__ B,
                                                       int nwin, int* status, const float* __restrict__ Xs,
                                                       int64_t ldx, int64_t prob_x) {
  __shared__ __align__(16) float T[32][RW + 4];   // T[k][i] = Y[row i][k0 + k]
  __shared__ __align__(16) float T2[32][RW + 4];  // the same for X (cross product only)
  const int w = blockIdx.x, u = blockIdx.y, t = threadIdx.x;
  const int tx = t & 15, ty = t >> 4;             // output rows ty*8.., columns tx*8..
  const float* Y = Ys + int64_t(u) * prob_y + (off + int64_t(w) * RW) * ldy;
  const float* X = Xs ? Xs + int64_t(u) * prob_x + (off + int64_t(w) * RW) * ldx : nullptr;
  float (*TX)[RW + 4] = X ? T2 : T;
  float part[8][8];
  double tot[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) tot[a][b] = 0.0;
  for (int64_t k0 = 0; k0 < cols; k0 += 32) {
    win_load_t(T, Y, ldy, k0, cols, t, status);
    if (X) win_load_t(T2, X, ldx, k0, cols, t, status);
    __syncthreads();
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b) part[a][b] = 0.f;
#pragma unroll 4
    for (int k = 0; k < 32; ++k) {
      const float4 x0 = *reinterpret_cast<const float4*>(&TX[k][ty * 8]);
      const float4 x1 = *reinterpret_cast<const float4*>(&TX[k][ty * 8 + 4]);
      const float4 y0 = *reinterpret_cast<const float4*>(&T[k][tx * 8]);
      const float4 y1 = *reinterpret_cast<const float4*>(&T[k][tx * 8 + 4]);
      const float xa[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const float yb[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) part[a][b] = fmaf(xa[a], yb[b], part[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b) tot[a][b] += double(part[a][b]);
    __syncthreads();
  }
  float* Bw = B + (int64_t(u) * nwin + w) * RW * RW;
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) Bw[(ty * 8 + a) * RW + tx * 8 + b] = float(tot[a][b]);
}

// Diagonalises B_w (RW x RW, symmetric) in shared memory by threshold cyclic Jacobi (RW/2
// disjoint rotations per round, one pass over the 2 x 2 blocks of the round's pairing) and
// writes its eigenvectors as columns of V_w, ordered by eigenvalue, largest first.
__global__ void __launch_bounds__(256) win_eig_kernel(const float* __restrict__ B, float* __restrict__ Vout,
                                                      float tol, int max_sweeps, int* status) {
  extern __shared__ __align__(16) float smw[];
  float (*A)[RW + 1] = reinterpret_cast<float (*)[RW + 1]>(smw);
  float (*V)[RW + 1] = reinterpret_cast<float (*)[RW + 1]>(smw + RW * (RW + 1));
  __shared__ float rc[RW / 2], rs[RW / 2], rap[RW / 2], raq[RW / 2];
  __shared__ int rp[RW / 2], rq[RW / 2], ract[RW / 2];
  __shared__ int order[RW];
  __shared__ float dmax;
  const int t = threadIdx.x;
  const int64_t wid = blockIdx.x;
  const float* Bw = B + wid * RW * RW;
  for (int e = t; e < RW * RW; e += 256) {
    const int i = e / RW, j = e % RW;
    A[i][j] = 0.5f * (Bw[i * RW + j] + Bw[j * RW + i]);
    V[i][j] = i == j ? 1.f : 0.f;
  }
  __syncthreads();
  if (t == 0) {
    float m = 0.f;
    for (int i = 0; i < RW; ++i) m = fmaxf(m, A[i][i]);
    dmax = m;
  }
  __syncthreads();
  const float flo = 2.f * FLT_EPSILON * dmax;  // couplings below the window's float32 noise count as zero
  for (int sweep = 0; sweep < max_sweeps; ++sweep) {
    int rotated = 0;
    for (int r = 0; r < RW - 1; ++r) {
      int act = 0;
      if (t < RW / 2) {
        const int p = rr_pos(t, r, RW), q = rr_pos(RW - 1 - t, r, RW);
        const float a = A[p][p], b = A[q][q], d = A[p][q];
        float c = 1.f, sn = 0.f, td = 0.f;
        if (fabsf(d) > flo && fabsf(d) > tol * sqrtf(fmaxf(a * b, 0.f))) {
          const float tau = __fdiv_rn(b - a, 2.f * d);
          const float tt = copysignf(1.f, tau) / (fabsf(tau) + sqrtf(fmaf(tau, tau, 1.f)));
          c = 1.0f / sqrtf(fmaf(tt, tt, 1.f));
          sn = tt * c;
          td = tt * d;
          act = 1;
        }
        rc[t] = c; rs[t] = sn; rp[t] = p; rq[t] = q; ract[t] = act;
        rap[t] = a - td; raq[t] = b + td;
      }
      if (!__syncthreads_or(act)) continue;
      rotated = 1;
      for (int e = t; e < (RW / 2) * (RW / 2); e += 256) {
        const int j = e / (RW / 2), k = e % (RW / 2);
        const int pj = rp[j], qj = rq[j], pk = rp[k], qk = rq[k];
        if (j == k) {
          if (ract[j]) {
            A[pj][pj] = rap[j];
            A[qj][qj] = raq[j];
            A[pj][qj] = 0.f;
            A[qj][pj] = 0.f;
          }
          continue;
        }
        if (!ract[j] && !ract[k]) continue;
        const float cj = rc[j], sj = rs[j], ck = rc[k], sk = rs[k];
        const float a = A[pj][pk], b = A[pj][qk], c = A[qj][pk], d = A[qj][qk];
        const float a1 = a * ck - b * sk, b1 = a * sk + b * ck;
        const float c1 = c * ck - d * sk, d1 = c * sk + d * ck;
        A[pj][pk] = cj * a1 - sj * c1;
        A[pj][qk] = cj * b1 - sj * d1;
        A[qj][pk] = sj * a1 + cj * c1;
        A[qj][qk] = sj * b1 + cj * d1;
      }
      for (int e = t; e < (RW / 2) * RW; e += 256) {
        const int j = e / RW, i = e % RW;
        if (!ract[j]) continue;
        const int p = rp[j], q = rq[j];
        const float c = rc[j], sn = rs[j];
        const float x = V[i][p], y = V[i][q];
        V[i][p] = c * x - sn * y;
        V[i][q] = sn * x + c * y;
      }
      __syncthreads();
    }
    if (!rotated) break;
  }
  // Order by eigenvalue, descending (ties: lower index first; a value that is not a number
  // sorts last), so that `order` is always a permutation of 0..RW-1.
  if (t < RW) {
    const float di = isnan(A[t][t]) ? -INFINITY : A[t][t];
    if (isnan(A[t][t])) raise_status(status, KF_ERR_INVALID, 123);
    int rank = 0;
    for (int j = 0; j < RW; ++j) {
      const float dj = isnan(A[j][j]) ? -INFINITY : A[j][j];
      rank += (dj > di) || (dj == di && j < t);
    }
    order[rank] = t;
  }
  __syncthreads();
  float* Vw = Vout + wid * RW * RW;
  for (int e = t; e < RW * RW; e += 256) {
    const int i = e / RW, c = e % RW;
    int oc = order[c];
    if (oc < 0 || oc >= RW) {  // bounds self-check
      raise_status(status, KF_ERR_INVALID, 124);
      oc = c;
    }
    Vw[i * RW + c] = V[i][oc];
  }
}

// X_w <- V_w^T X_w in place for the RW rows of every window (rows start at off + w * RW)
// and one 64-column block per CTA: out[i][j] = sum_k V[k][i] X[k][j].
__global__ void __launch_bounds__(256) win_rotate_kernel(float* __restrict__ Xs, int64_t ldx, int64_t prob_x,
                                                         int64_t cols, int64_t off, const float* __restrict__ Vw_all,
                                                         int nwin, int* status) {
  extern __shared__ __align__(16) float smr[];
  float* Vs = smr;              // RW x RW
  float* Xb = smr + RW * RW;    // RW x 64
  const int cb = blockIdx.x, w = blockIdx.y % nwin, u = blockIdx.y / nwin, t = threadIdx.x;
  const float* Vw = Vw_all + (int64_t(u) * nwin + w) * RW * RW;
  float* X = Xs + int64_t(u) * prob_x + (off + int64_t(w) * RW) * ldx + int64_t(cb) * 64;
  const int64_t c0 = int64_t(cb) * 64;
  for (int e = t; e < RW * RW / 4; e += 256)
    if (aligned16(Vw + 4 * e, status, 121)) reinterpret_cast<float4*>(Vs)[e] = reinterpret_cast<const float4*>(Vw)[e];
  for (int e = t; e < RW * 16; e += 256) {
    const int i = e >> 4, c = (e & 15) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c0 + c + 3 < cols) {
      const float* a = X + int64_t(i) * ldx + c;
      if (aligned16(a, status, 122)) v = *reinterpret_cast<const float4*>(a);
    } else {
      float tmp[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < 4; ++q)
        if (c0 + c + q < cols) tmp[q] = X[int64_t(i) * ldx + c + q];
      v = make_float4(tmp[0], tmp[1], tmp[2], tmp[3]);
    }
    *reinterpret_cast<float4*>(Xb + i * 64 + c) = v;
  }
  __syncthreads();
  const int tx = t & 15, ty = t >> 4;  // rows ty*8..+7, columns tx*4..+3
  float acc[8][4];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 4
  for (int k = 0; k < RW; ++k) {
    const float4 v0 = *reinterpret_cast<const float4*>(Vs + k * RW + ty * 8);
    const float4 v1 = *reinterpret_cast<const float4*>(Vs + k * RW + ty * 8 + 4);
    const float4 x = *reinterpret_cast<const float4*>(Xb + k * 64 + tx * 4);
    const float va[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    const float xb[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(va[a], xb[b], acc[a][b]);
  }
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const int i = ty * 8 + a;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t c = c0 + tx * 4 + b;
      if (c < cols) X[int64_t(i) * ldx + tx * 4 + b] = acc[a][b];
    }
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

struct SvdBufs {
  float *C, *Q, *V, *flo, *Y, *sig, *qinv, *Qs, *Ys, *Bw, *Vw;
  int *skip, *conv, *perm;
  unsigned* off;
  int64_t R, lyM;
  int nwin;
};

static size_t svd_carve(Carve& cv, int nu, int64_t m_max, int64_t n_max, int64_t s, SvdBufs& b) {
  const JacPlan pl = jac_plan(s);
  // image rows of every problem padded to one length that keeps float4 rows aligned
  b.lyM = ((m_max > n_max ? m_max : n_max) + 3) / 4 * 4;
  b.nwin = int((s + RW - 1) / RW);
  b.R = int64_t(b.nwin) * RW + RW / 2;
  b.C = cv.take<float>(size_t(nu) * pl.sp * pl.sp);
  b.Q = cv.take<float>(size_t(nu) * pl.sp * pl.sp);
  b.V = cv.take<float>(size_t(nu) * pl.npairs * JP * JP);
  b.skip = cv.take<int>(size_t(nu) * pl.npairs);
  b.conv = cv.take<int>(nu);
  b.off = cv.take<unsigned>(nu);
  b.flo = cv.take<float>(nu);
  b.Y = cv.take<float>(size_t(nu) * s * b.lyM);
  b.sig = cv.take<float>(size_t(nu) * s);
  b.qinv = cv.take<float>(size_t(nu) * s);
  b.perm = cv.take<int>(size_t(nu) * s);
  b.Qs = cv.take<float>(size_t(nu) * b.R * pl.sp);
  b.Ys = cv.take<float>(size_t(nu) * b.R * b.lyM);
  b.Bw = cv.take<float>(size_t(nu) * b.nwin * RW * RW);
  b.Vw = cv.take<float>(size_t(nu) * b.nwin * RW * RW);
  return cv.off;
}

size_t svd_workspace(int32_t nu, int64_t m_max, int64_t n_max, int64_t s) {
  Carve cv(nullptr, 0, true);
  SvdBufs b;
  return svd_carve(cv, nu, m_max, n_max, s, b) + 256;
}

// sym: every problem's Wt is a symmetric s x s matrix C whose eigenpairs are wanted (its lower
// triangle is read); the images are y = C q, the values Rayleigh quotients q.Cq / q.q, the
// refinement uses the windows' Rayleigh-Ritz matrices, and sigma = sqrt(max(lambda, 0)).
kf_status svd_run(kf_ctx* ctx, int32_t nu, const kf_svd_problem* pr, float tol, int32_t max_sweeps, void* ws,
                  size_t ws_bytes, cudaStream_t st, bool sym) {
  int64_t s = pr[0].m < pr[0].n ? pr[0].m : pr[0].n, m_max = 0, n_max = 0;
  for (int i = 0; i < nu; ++i) {
    m_max = pr[i].m > m_max ? pr[i].m : m_max;
    n_max = pr[i].n > n_max ? pr[i].n : n_max;
  }
  const JacPlan pl = jac_plan(s);
  Carve cv(ws, ws_bytes, false);
  SvdBufs bf;
  svd_carve(cv, nu, m_max, n_max, s, bf);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "whitened_svd: workspace too small");
  float *C = bf.C, *Q = bf.Q, *V = bf.V, *flo = bf.flo, *sig = bf.sig, *qinv = bf.qinv;
  int *skip = bf.skip, *conv = bf.conv, *perm = bf.perm;
  unsigned* off = bf.off;

  const bool prof = ctx->prof_enabled;
  unsigned long long* flops = prof ? ctx->prof_flops() : nullptr;
  if (prof) {
    for (int e = 0; e < 5; ++e)
      if (!ctx->prof_ev[e]) KF_CUDA(cudaEventCreate(&ctx->prof_ev[e]));
    KF_CUDA(cudaMemsetAsync(flops, 0, sizeof(unsigned long long), st));
    KF_CUDA(cudaEventRecord(ctx->prof_ev[0], st));
    ctx->prof_kev_used = 0;
    ctx->prof_steps = int64_t(max_sweeps) * (pl.nblk - 1);
    ctx->prof_valid = true;
  }
  // Gram of the smaller side, lower triangle, float32 SIMT (accuracy matters here).
  for (int i = 0; i < nu; ++i) {
    const kf_svd_problem& p = pr[i];
    if (sym) {  // the matrix itself
      KF_TRY(launch_copy(p.Wt, p.ldw, C + int64_t(i) * pl.sp * pl.sp, pl.sp, s, s, false, st));
      continue;
    }
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
    KF_TRY(check_cuda(cudaGetLastError(), "jac_prepare_kernel"));
    int* sweeps_tmp = nullptr;
    jac_floor_kernel<<<nu, 256, 0, st>>>(C, pl.sp, flo, 8.0f, conv, off, sweeps_tmp); note_launch();
    KF_TRY(check_cuda(cudaGetLastError(), "jac_floor_kernel"));
  }
  // Per-problem sweep counters (copied to the callers' pointers after the sweeps).
  int* sweeps_dev = perm;  // reuse: perm is rewritten by the sort afterwards
  KF_CUDA(cudaMemsetAsync(sweeps_dev, 0, sizeof(int) * nu, st));

  const int ntile_c = pl.npairs * (pl.npairs + 1) / 2;
  const int ntile_q = int(pl.sp / JP) * pl.npairs;
  const size_t apply_smem = size_t(2 * STAGE_F + JP * JP) * sizeof(float);
  const int per_u = ntile_c + ntile_q;
  const int64_t total_tasks = int64_t(per_u) * nu;
  if (total_tasks > 0x7fffffff) return fail(KF_ERR_UNSUPPORTED, "whitened_svd: too many Jacobi tasks");
  const int apply_grid = int(total_tasks < int64_t(ctx->sm_count) * 2 ? total_tasks : int64_t(ctx->sm_count) * 2);
  static std::atomic<unsigned long long> attr_done{0};
  KF_TRY(set_attr_once(attr_done, [&] {
    return check_cuda(cudaFuncSetAttribute(jac_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           int(apply_smem)), "jac_apply smem attribute");
  }));
  const int max_inner = KF_JAC_MAX_INNER;
  int sweeps_run = 0;
  if (prof) KF_CUDA(cudaEventRecord(ctx->prof_ev[1], st));
  for (int sw = 0; sw < max_sweeps; ++sw) {
    for (int step = 0; step < pl.nblk - 1; ++step) {
      cudaEvent_t* kev = nullptr;
      if (prof) {
        while (int64_t(ctx->prof_kev.size()) < ctx->prof_kev_used + 3) {
          cudaEvent_t e;
          KF_CUDA(cudaEventCreate(&e));
          ctx->prof_kev.push_back(e);
        }
        kev = ctx->prof_kev.data() + ctx->prof_kev_used;
        ctx->prof_kev_used += 3;
        KF_CUDA(cudaEventRecord(kev[0], st));
      }
      jac_solve_kernel<<<dim3(pl.npairs, nu), 256, 0, st>>>(C, pl.sp, pl.nblk, step, V, skip, conv, off, flo, tol,
                                                           max_inner); note_launch();
      KF_TRY(check_cuda(cudaGetLastError(), "jac_solve_kernel"));
      if (prof) KF_CUDA(cudaEventRecord(kev[1], st));
      jac_apply_kernel<<<apply_grid, 256, apply_smem, st>>>(C, Q, pl.sp, pl.nblk, step, V, skip, conv, ntile_c,
                                                            per_u, int(total_tasks), flops, ctx->d_status); note_launch();
      KF_TRY(check_cuda(cudaGetLastError(), "jac_apply_kernel"));
      if (prof) KF_CUDA(cudaEventRecord(kev[2], st));
    }
    jac_check_kernel<<<1, 256, 0, st>>>(nu, conv, off, tol, sw, max_sweeps, sweeps_dev, ctx->d_status,
                                        ctx->d_status + 2); note_launch();
    KF_TRY(check_cuda(cudaGetLastError(), "jac_check_kernel"));
    ++sweeps_run;
    // Convergence poll: once every problem has converged no further sweep is launched.
    if (sw >= 2 && sw + 1 < max_sweeps) {
      KF_CUDA(cudaMemcpyAsync(ctx->h_flag, ctx->d_status + 2, sizeof(int), cudaMemcpyDeviceToHost, st));
      KF_CUDA(cudaStreamSynchronize(st));
      if (*ctx->h_flag) break;
    }
  }
  if (prof) ctx->prof_steps = int64_t(sweeps_run) * (pl.nblk - 1);
  if (prof) KF_CUDA(cudaEventRecord(ctx->prof_ev[2], st));
  for (int i = 0; i < nu; ++i)
    if (pr[i].sweeps) KF_CUDA(cudaMemcpyAsync(pr[i].sweeps, sweeps_dev + i, sizeof(int), cudaMemcpyDeviceToDevice, st));

  // Rayleigh quotients on W~ itself, sort, windowed Rayleigh-Ritz refinement, final sort.
  int P = 1;
  while (P < s) P <<= 1;
  const size_t sort_smem = size_t(P) * 8;
  if (sort_smem > 227 * 1024) return fail(KF_ERR_UNSUPPORTED, "whitened_svd: s too large for the in-CTA sort");
  const size_t eig_smem = size_t(2) * RW * (RW + 1) * sizeof(float);
  const size_t rot_smem = size_t(RW * RW + RW * 64) * sizeof(float);
  static std::atomic<unsigned long long> sattr_done{0};
  KF_TRY(set_attr_once(sattr_done, [&]() -> kf_status {
    KF_CUDA(cudaFuncSetAttribute(sort_desc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024));
    KF_CUDA(cudaFuncSetAttribute(win_eig_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(eig_smem)));
    KF_CUDA(cudaFuncSetAttribute(win_rotate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(rot_smem)));
    return KF_OK;
  }));
  const int64_t lyM = bf.lyM, R = bf.R;
  const int nwin = bf.nwin;
  KF_CUDA(cudaMemsetAsync(bf.Y, 0, sizeof(float) * size_t(nu) * s * lyM, st));
  for (int i = 0; i < nu; ++i) {
    const kf_svd_problem& p = pr[i];
    const float* Qti = Q + int64_t(i) * pl.sp * pl.sp;  // eigenvectors as rows
    const bool right = kf_gram_side(p.m, p.n) == KF_SIDE_RIGHT;
    const int64_t len_y = right ? p.m : p.n;
    float* Yi = bf.Y + int64_t(i) * s * lyM;
    // Yt = Qt W~^T (right side, y_j = W~ q_j) or Qt W~ (left side, y_j = W~^T q_j)
    GemmDesc g{};
    g.M = s; g.N = len_y; g.K = s; g.batch = 1;
    g.A = Qti; g.lda = pl.sp;
    g.B = p.Wt; g.ldb = p.ldw; g.trans_b = right;
    g.C = Yi; g.ldc = lyM;
    g.alpha = 1.f; g.beta = 0.f;
    KF_TRY(simt_gemm(g, st));
    rayleigh_norms_kernel<<<unsigned(s), 256, 0, st>>>(Yi, lyM, len_y, Qti, pl.sp, s, sig + int64_t(i) * s,
                                                      qinv + int64_t(i) * s, ctx->d_status, int(sym)); note_launch();
    KF_TRY(check_cuda(cudaGetLastError(), "rayleigh_norms_kernel"));
  }
  if (prof) KF_CUDA(cudaEventRecord(ctx->prof_ev[3], st));
  sort_desc_kernel<<<unsigned(nu), 1024, sort_smem, st>>>(sig, s, P, perm, s); note_launch();
  KF_TRY(check_cuda(cudaGetLastError(), "sort_desc_kernel"));
  // vectors and their images in sorted order, zero rows up to R
  gather_rows_kernel<<<dim3(unsigned(R), unsigned(nu)), 256, 0, st>>>(Q, pl.sp, pl.sp * pl.sp, perm, s, bf.Qs, pl.sp,
                                                                      R * pl.sp, pl.sp); note_launch();
  KF_TRY(check_cuda(cudaGetLastError(), "gather_rows_kernel"));
  gather_rows_kernel<<<dim3(unsigned(R), unsigned(nu)), 256, 0, st>>>(bf.Y, lyM, s * lyM, perm, s, bf.Ys, lyM,
                                                                      R * lyM, lyM); note_launch();
  KF_TRY(check_cuda(cudaGetLastError(), "gather_rows_kernel"));
  if (int64_t(nu) * nwin > 65535) return fail(KF_ERR_UNSUPPORTED, "whitened_svd: too many refinement windows");
  for (int pass = 0; pass < 2; ++pass) {
    const int64_t offr = pass * (RW / 2);
    win_gram_kernel<<<dim3(unsigned(nwin), unsigned(nu)), 256, 0, st>>>(bf.Ys, lyM, R * lyM, lyM, offr, bf.Bw, nwin,
                                                                        ctx->d_status, sym ? bf.Qs : nullptr, pl.sp,
                                                                        R * pl.sp);
    note_launch();
    KF_TRY(check_cuda(cudaGetLastError(), "win_gram_kernel"));
    win_eig_kernel<<<unsigned(nu * nwin), 256, eig_smem, st>>>(bf.Bw, bf.Vw, 1e-6f, 12, ctx->d_status); note_launch();
    KF_TRY(check_cuda(cudaGetLastError(), "win_eig_kernel"));
    win_rotate_kernel<<<dim3(unsigned(pl.sp / 64), unsigned(nu * nwin)), 256, rot_smem, st>>>(
        bf.Qs, pl.sp, R * pl.sp, pl.sp, offr, bf.Vw, nwin, ctx->d_status); note_launch();
    KF_TRY(check_cuda(cudaGetLastError(), "win_rotate_kernel"));
    win_rotate_kernel<<<dim3(unsigned((lyM + 63) / 64), unsigned(nu * nwin)), 256, rot_smem, st>>>(
        bf.Ys, lyM, R * lyM, lyM, offr, bf.Vw, nwin, ctx->d_status); note_launch();
    KF_TRY(check_cuda(cudaGetLastError(), "win_rotate_kernel"));
  }
  for (int i = 0; i < nu; ++i) {
    rayleigh_norms_kernel<<<unsigned(s), 256, 0, st>>>(bf.Ys + int64_t(i) * R * lyM, lyM, lyM,
                                                      bf.Qs + int64_t(i) * R * pl.sp, pl.sp, s, sig + int64_t(i) * s,
                                                      qinv + int64_t(i) * s, ctx->d_status, int(sym)); note_launch();
    KF_TRY(check_cuda(cudaGetLastError(), "rayleigh_norms_kernel"));
  }
  sort_desc_kernel<<<unsigned(nu), 1024, sort_smem, st>>>(sig, s, P, perm, s); note_launch();
  KF_TRY(check_cuda(cudaGetLastError(), "sort_desc_kernel"));
  for (int i = 0; i < nu; ++i) {
    const kf_svd_problem& p = pr[i];
    dim3 grid(unsigned((s + 31) / 32), unsigned((s + 31) / 32));
    gather_kernel<<<grid, dim3(32, 8), 0, st>>>(bf.Qs + int64_t(i) * R * pl.sp, pl.sp, s, perm + int64_t(i) * s,
                                                sig + int64_t(i) * s, qinv + int64_t(i) * s, p.vecs, p.ldv, p.sigma,
                                                int(sym));
    note_launch();
    KF_TRY(check_cuda(cudaGetLastError(), "gather_kernel"));
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
  out->refine_ms = t[3];
  out->jacobi_steps = ctx->prof_steps;
  double ts = 0.0, ta = 0.0;
  for (int64_t i = 0; i + 3 <= ctx->prof_kev_used; i += 3) {
    float a = 0.f, b = 0.f;
    KF_CUDA(cudaEventElapsedTime(&a, ctx->prof_kev[i], ctx->prof_kev[i + 1]));
    KF_CUDA(cudaEventElapsedTime(&b, ctx->prof_kev[i + 1], ctx->prof_kev[i + 2]));
    ts += a;
    ta += b;
  }
  out->jacobi_solve_ms = float(ts);
  out->jacobi_apply_ms = float(ta);
  out->jacobi_apply_launches = ctx->prof_kev_used / 3;
  out->jacobi_apply_flops = double(f);
  return KF_OK;
}

}  // namespace kf
