// Spectrum of the whitened weight through its Gram matrix (Swift-SVD 2A: one
// eigendecomposition of the aggregated covariance instead of repeated SVDs), by a blocked
// parallel cyclic Jacobi eigensolver:
//   * C (s x s, float32, padded to a multiple of 64) is cut into 32-wide blocks; a
//     round-robin tournament pairs the blocks so that every step visits nblk/2 disjoint
//     pairs and a sweep (nblk - 1 steps) visits every pair once;
//   * jac_solve: one CTA per pair loads the 64 x 64 problem [[C_II C_IJ][C_JI C_JJ]] into
//     shared memory and runs threshold cyclic Jacobi on it (32 disjoint rotations per round,
//     KF_JAC_MAX_INNER sweeps), accumulating the 64 x 64 orthogonal V_p, which it writes as
//     three bfloat16 planes in the tensor-core apply's operand layout;
//   * jac_apply_tc: C <- P^T C P and Q <- Q P for the block-diagonal P = diag(V_p) on the
//     tensor cores (tcgen05, float32 accumulation in tensor memory): every operand enters as
//     three bfloat16 planes (the full float32 significand) and the six cross terms down to
//     the last plane's weight are summed, so the products are float32-accurate.  C is taken
//     in 128 x 128 super-tiles (two pairs of rows by two pairs of columns, only super-tiles
//     on or above the diagonal, the result mirrored), each as two chained products with
//     M = 128: U = S diag(V_q1, V_q2), then the transposed second product
//     (V_p^T U_p)^T = U_p^T V_p, whose result lands in tensor memory one column of S per lane
//     for coalesced stores.  Q is stored transposed (one eigenvector per row), so Q P becomes
//     P^T Qt, computed per 64 x 128 panel as (panel^T V_q) for the same reason;
//   * a sweep in which no pair had |c_pq| > tol * sqrt(c_pp c_qq) (entries below a float32
//     rounding floor count as zero) ends the iteration for that problem.
// The singular values are then the Rayleigh quotients sigma_i = ||W~ q_i|| / ||q_i||,
// evaluated on W~ rather than on C so that the Gram's rounding errors enter only at second
// order, sorted descending with their vectors.
// The same solver serves a symmetric matrix given directly (Swift-SVD 2A's covariance of
// the layer output): the values are then the Rayleigh quotients q.Cq / q.q.
#include "kf_internal.cuh"
#include "kf_tc_ptx.cuh"

#include <cfloat>
#include <vector>

namespace kf {
namespace {

constexpr int JB = 32, JP = 64;  // block width, pair problem size
constexpr int JS = JP + 4;  // row stride of V and of the Newton-Schulz factor in the pair solve
constexpr size_t JAC_SOLVE_SMEM = size_t(2 * JP * JS) * sizeof(float);
// Inner sweeps of a pair problem.  Measured on the 7B block (7 Gram matrices of 4096): one
// sweep of rotations per pair problem instead of up to 12 costs at most one more outer sweep,
// the final singular values come out as accurate (about 6e-5 relative on the kept components
// either way), and the pair solves take 40% less time.
#ifndef KF_JAC_MAX_INNER
#define KF_JAC_MAX_INNER 1
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

// Shared-memory operand images of the tensor-core apply (bfloat16, 128-byte swizzle: the
// 16-byte chunk index inside a 128-byte row is XORed with the row index mod 8; buffers
// 1024-byte aligned).  The same layouts TMA produces for the GEMM engine's operands.
//   V image (B operand, K = 64 old indices x N = 64 new indices, MN-major): 3 planes of 8 KB.
//   A image, K-major (M = 128 rows x K = 64): 3 planes of 16 KB, row m at m * 128 bytes.
//   A image, MN-major (M = 128 x K = 64): 3 planes of 16 KB, two 64-wide M chunks 8 KB apart,
//   row k at k * 128 bytes inside a chunk.
constexpr int VPLANE_BYTES = 8192, VIMG_BYTES = 3 * VPLANE_BYTES;
constexpr int APLANE_BYTES = 16384, AIMG_BYTES = 3 * APLANE_BYTES;
__host__ __device__ __forceinline__ uint32_t vimg_off(int k, int n) {
  return uint32_t(k) * 128u + ((uint32_t((n >> 3) ^ (k & 7))) << 4) + uint32_t(n & 7) * 2u;
}
__device__ __forceinline__ uint32_t akm_off(int m, int k) {
  return uint32_t(m) * 128u + ((uint32_t((k >> 3) ^ (m & 7))) << 4) + uint32_t(k & 7) * 2u;
}
__device__ __forceinline__ uint32_t amn_off(int m, int k) {
  return uint32_t(m >> 6) * 8192u + uint32_t(k) * 128u + ((uint32_t(((m & 63) >> 3) ^ (k & 7))) << 4) +
         uint32_t(m & 7) * 2u;
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
// The pair problem's 64 indices sit in 64 slots of a circle-method tournament: slot k < 32 is
// the first index of rotation pair k, slot 32 + k its second.  After every round each slot's
// contents move one place round the circle (slot 0 stays; 1 -> 32; k -> k - 1 for 2 <= k < 32;
// 32 + k -> 33 + k for k < 31; 63 -> 31), so that the 63 rounds of a sweep meet every pair of
// indices once and bring every index back to its starting slot.  The index that starts in
// slot k < 32 is the pair-local column k (first block), the one in slot 32 + k is 63 - k
// (second block), which makes round r pair exactly the indices rr_pos(k, r, 64) and
// rr_pos(63 - k, r, 64).  In shared memory slot k < 32 is row/column k and slot 32 + k is
// 32 + ((k + 31) & 31): with this placement every load and store of a round, including the
// moved stores, touches 32 different banks.
__device__ __forceinline__ int slot_phys(int s) { return s < JB ? s : JB + ((s - JB + JB - 1) & (JB - 1)); }
__device__ __forceinline__ int slot_next(int s) {
  if (s == 0) return 0;
  if (s == 1) return JB;
  if (s < JB) return s - 1;
  if (s == JP - 1) return JB - 1;
  return s + 1;
}
__device__ __forceinline__ int index_phys(int x) { return slot_phys(x < JB ? x : JP + JB - 1 - x); }

// One rotation round of the pair solve (see jac_solve_kernel): reads the slot-ordered matrix
// A, writes the rotated matrix at the moved slots of An, and rotates and moves this thread's
// rows of V.  Every warp computes all 32 rotations of the round (lane l: pair l) from the
// same entries.  The rotation parameters use the hardware's approximate reciprocal and
// square root: a rotation only has to be (nearly) orthogonal and to shrink its coupling,
// and the Newton-Schulz step after the sweep re-orthogonalises the accumulated V.  Returns
// whether any rotation of the round was active (the same in every warp).
struct RoundMap {
  int ct, cb, dct, dcb;
  int rt[4], rb[4], drt[4], drb[4];
};
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ bool solve_round(const float* __restrict__ A, float* __restrict__ An, float (&vt)[8],
                                            float (&vb)[8], const RoundMap& q, int lane, int warp, float flo,
                                            float tol2) {
  const float a = A[q.ct * JP + q.ct], b = A[q.cb * JP + q.cb], d = A[q.ct * JP + q.cb];
  float c = 1.f, sn = 0.f, td = 0.f;
  const bool act = fabsf(d) > flo && d * d > tol2 * fmaxf(a * b, 0.f);
  if (act) {
    const float tau = (b - a) * rcp_approx(2.f * d);
    const float tt = copysignf(rcp_approx(fabsf(tau) + sqrt_approx(fmaf(tau, tau, 1.f))), tau);
    c = rsqrtf(fmaf(tt, tt, 1.f));
    sn = tt * c;
    td = tt * d;
  }
  const bool any = __any_sync(0xffffffffu, act);
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int j = warp + 8 * x;
    const float cj = __shfl_sync(0xffffffffu, c, j), sj = __shfl_sync(0xffffffffu, sn, j);
    // an inactive rotation has c = 1, s = 0 and reproduces its entries exactly; the diagonal
    // block of pair l (j == l) takes its closed form instead (selected, not branched)
    const float e00 = A[q.rt[x] + q.ct], e01 = A[q.rt[x] + q.cb], e10 = A[q.rb[x] + q.ct], e11 = A[q.rb[x] + q.cb];
    const float a1 = e00 * c - e01 * sn, b1 = e00 * sn + e01 * c;
    const float c1 = e10 * c - e11 * sn, d1 = e10 * sn + e11 * c;
    const bool dg = j == lane;
    An[q.drt[x] + q.dct] = dg ? a - td : cj * a1 - sj * c1;
    An[q.drt[x] + q.dcb] = dg ? (act ? 0.f : e01) : cj * b1 - sj * d1;
    An[q.drb[x] + q.dct] = dg ? (act ? 0.f : e10) : sj * a1 + cj * c1;
    An[q.drb[x] + q.dcb] = dg ? b + td : sj * b1 + cj * d1;
  }
#pragma unroll
  for (int y = 0; y < 8; ++y) {
    const float x0 = vt[y], y0 = vb[y];
    const float nt = c * x0 - sn * y0, nb = sn * x0 + c * y0;
    // slot l + 1 -> l, slot 32 + l - 1 -> 32 + l; slot 1 -> 32, slot 63 -> 31, slot 0 stays
    const float dn = __shfl_down_sync(0xffffffffu, nt, 1);
    const float up = __shfl_up_sync(0xffffffffu, nb, 1);
    vt[y] = lane == 0 ? nt : (lane == JB - 1 ? nb : dn);
    vb[y] = lane == 0 ? dn : up;
  }
  __syncthreads();
  return any;
}
// One sweep (63 rounds, an odd number: the result ends in B).
__device__ __forceinline__ bool solve_sweep(float* __restrict__ A, float* __restrict__ B, float (&vt)[8],
                                            float (&vb)[8], const RoundMap& q, int lane, int warp, float flo,
                                            float tol2) {
  bool rotated = false;
  for (int r = 0; r < (JP - 2) / 2; ++r) {
    rotated |= solve_round(A, B, vt, vb, q, lane, warp, flo, tol2);
    rotated |= solve_round(B, A, vt, vb, q, lane, warp, flo, tol2);
  }
  rotated |= solve_round(A, B, vt, vb, q, lane, warp, flo, tol2);
  return rotated;
}

__global__ void __launch_bounds__(256, 4) jac_solve_kernel(float* __restrict__ Call, int64_t sp, int nblk,
                                                        int step, uint8_t* __restrict__ Vimg,
                                                        int* __restrict__ skipall,
                                                        const int* __restrict__ conv,
                                                        unsigned* __restrict__ offmax,
                                                        const float* __restrict__ floorv, float tol,
                                                        int max_inner) {
  // Two slot-ordered copies of the 64 x 64 problem (row stride JP): a round reads one and
  // writes every entry of the other at its moved position, so a round needs one barrier.
  // The same JAC_SOLVE_SMEM bytes later hold V and the Newton-Schulz factor (stride JS).
  extern __shared__ float jsm[];
  float* const A = jsm;
  float* const An = jsm + JP * JS;
  __shared__ float red[8];

  const int k = blockIdx.x, u = blockIdx.y, t = threadIdx.x;
  if (conv[u]) return;
  const int npairs = nblk / 2;
  const float* C = Call + int64_t(u) * sp * sp;
  const int b0 = rr_pos(k, step, nblk), b1 = rr_pos(nblk - 1 - k, step, nblk);
  for (int e = t; e < JP * JP; e += 256) {
    const int r = e >> 6, c = e & 63;
    A[index_phys(r) * JP + index_phys(c)] = C[gidx(r, b0, b1) * sp + gidx(c, b0, b1)];
  }
  __syncthreads();
  const float flo = floorv[u];

  // Largest relative coupling between the two blocks.
  float m = 0.f;
  for (int e = t; e < JB * JB; e += 256) {
    const int r = index_phys(e >> 5), c = index_phys(JB + (e & 31));
    const float v = fabsf(A[r * JP + c]);
    if (v > flo) {
      const float den = fmaxf(sqrtf(fmaxf(A[r * JP + r] * A[c * JP + c], 0.f)), flo);
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

  // Threshold cyclic Jacobi, 32 disjoint rotations per round (solve_round).  Thread (warp w,
  // lane l) updates the 2 x 2 blocks (pair j, pair l), j = w, w + 8, w + 16, w + 24, and holds
  // rows w, w + 8, ..., w + 56 of the two columns of V in slots l and 32 + l in registers; V's
  // columns follow the circle by warp shuffles.  Every address of a round is fixed per thread.
  const int lane = t & 31, warp = t >> 5;
  RoundMap q;
  q.ct = lane;
  q.cb = slot_phys(JB + lane);
  q.dct = slot_phys(slot_next(lane));
  q.dcb = slot_phys(slot_next(JB + lane));
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int j = warp + 8 * x;
    q.rt[x] = j * JP;
    q.rb[x] = slot_phys(JB + j) * JP;
    q.drt[x] = slot_phys(slot_next(j)) * JP;
    q.drb[x] = slot_phys(slot_next(JB + j)) * JP;
  }
  float vt[8], vb[8];
#pragma unroll
  for (int y = 0; y < 8; ++y) {
    const int i = warp + 8 * y;
    vt[y] = (i == lane) ? 1.f : 0.f;
    vb[y] = (i == JP - 1 - lane) ? 1.f : 0.f;
  }
  const float tol2 = tol * tol;
  for (int sweep = 0; sweep < max_inner; ++sweep) {
    // the two buffers' roles are fixed inside each call (constant shared-memory offsets)
    const bool rotated = (sweep & 1) ? solve_sweep(An, A, vt, vb, q, lane, warp, flo, tol2)
                                     : solve_sweep(A, An, vt, vb, q, lane, warp, flo, tol2);
    if (!rotated) break;
  }
  // After whole sweeps every index is back in its starting slot: the vector in slot l is the
  // new direction l, the one in slot 32 + l the new direction 63 - l.
  float* V = jsm;               // V[i][n], stride JS (A is no longer needed)
  float* M = jsm + JP * JS;
#pragma unroll
  for (int y = 0; y < 8; ++y) {
    const int i = warp + 8 * y;
    V[i * JS + lane] = vt[y];
    V[i * JS + JP - 1 - lane] = vb[y];
  }
  __syncthreads();
  // One Newton-Schulz step V <- V (3I - V^T V) / 2 removes the orthogonality drift that the
  // rounding of many plane rotations leaves in V; each thread computes a 4 x 4 tile of each
  // product (rows 4 ti .. 4 ti + 3, columns 4 tj .. 4 tj + 3).
  const int ti = t >> 4, tj = t & 15;
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 4
  for (int kk = 0; kk < JP; ++kk) {
    const float4 p = *reinterpret_cast<const float4*>(V + kk * JS + 4 * ti);
    const float4 q = *reinterpret_cast<const float4*>(V + kk * JS + 4 * tj);
    const float pa[4] = {p.x, p.y, p.z, p.w}, qb[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(pa[a], qb[b], acc[a][b]);
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    float4 w;
    w.x = (4 * ti + a == 4 * tj + 0 ? 1.5f : 0.f) - 0.5f * acc[a][0];
    w.y = (4 * ti + a == 4 * tj + 1 ? 1.5f : 0.f) - 0.5f * acc[a][1];
    w.z = (4 * ti + a == 4 * tj + 2 ? 1.5f : 0.f) - 0.5f * acc[a][2];
    w.w = (4 * ti + a == 4 * tj + 3 ? 1.5f : 0.f) - 0.5f * acc[a][3];
    *reinterpret_cast<float4*>(M + (4 * ti + a) * JS + 4 * tj) = w;
  }
  __syncthreads();
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 2
  for (int kk = 0; kk < JP; kk += 4) {
    float pv[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const float4 p = *reinterpret_cast<const float4*>(V + (4 * ti + a) * JS + kk);
      pv[a][0] = p.x; pv[a][1] = p.y; pv[a][2] = p.z; pv[a][3] = p.w;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 mq = *reinterpret_cast<const float4*>(M + (kk + q) * JS + 4 * tj);
      const float mb[4] = {mq.x, mq.y, mq.z, mq.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(pv[a][q], mb[b], acc[a][b]);
    }
  }
  // V (row = old index, column = new index) as three bfloat16 planes in the shared-memory
  // image the tensor-core apply copies verbatim (B operand, MN-major, 128-byte swizzle): four
  // consecutive new indices of one old index are 8 bytes of one 16-byte chunk of each plane.
  uint8_t* img = Vimg + (int64_t(u) * npairs + k) * VIMG_BYTES;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    __nv_bfloat16 h[4][3];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float v = acc[a][b];
      h[b][0] = __float2bfloat16_rn(v);
      const float r1 = v - __bfloat162float(h[b][0]);
      h[b][1] = __float2bfloat16_rn(r1);
      h[b][2] = __float2bfloat16_rn(r1 - __bfloat162float(h[b][1]));
    }
    const uint32_t o = vimg_off(4 * ti + a, 4 * tj);
#pragma unroll
    for (int pl = 0; pl < 3; ++pl) {
      const uint32_t lo = uint32_t(__bfloat16_as_ushort(h[0][pl])) | (uint32_t(__bfloat16_as_ushort(h[1][pl])) << 16);
      const uint32_t hi = uint32_t(__bfloat16_as_ushort(h[2][pl])) | (uint32_t(__bfloat16_as_ushort(h[3][pl])) << 16);
      *reinterpret_cast<uint2*>(img + pl * VPLANE_BYTES + o) = make_uint2(lo, hi);
    }
  }
  if (t == 0) skip[k] = 0;
}

// ------------------------------------------------------------------------- apply
// Three-plane split of a float32 value (bfloat16 terms holding its full significand).
__device__ __forceinline__ void split3(float v, __nv_bfloat16& h1, __nv_bfloat16& h2, __nv_bfloat16& h3) {
  h1 = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(h1);
  h2 = __float2bfloat16_rn(r1);
  h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
}
__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return uint32_t(__bfloat16_as_ushort(a)) | (uint32_t(__bfloat16_as_ushort(b)) << 16);
}
// Four consecutive elements (along the contiguous dimension of one 16-byte chunk) into the
// three planes of an A image at byte offset `off` (8-byte aligned).
__device__ __forceinline__ void put4(uint8_t* img, uint32_t off, float4 v) {
  __nv_bfloat16 a1, a2, a3, b1, b2, b3, c1, c2, c3, d1, d2, d3;
  split3(v.x, a1, a2, a3);
  split3(v.y, b1, b2, b3);
  split3(v.z, c1, c2, c3);
  split3(v.w, d1, d2, d3);
  *reinterpret_cast<uint2*>(img + off) = make_uint2(pack2(a1, b1), pack2(c1, d1));
  *reinterpret_cast<uint2*>(img + APLANE_BYTES + off) = make_uint2(pack2(a2, b2), pack2(c2, d2));
  *reinterpret_cast<uint2*>(img + 2 * APLANE_BYTES + off) = make_uint2(pack2(a3, b3), pack2(c3, d3));
}
// Eight consecutive elements into one 16-byte chunk of each plane.
__device__ __forceinline__ void put8(uint8_t* img, uint32_t off, const uint32_t* w) {
  uint32_t p[3][4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat16 x1, x2, x3, y1, y2, y3;
    split3(__uint_as_float(w[2 * q]), x1, x2, x3);
    split3(__uint_as_float(w[2 * q + 1]), y1, y2, y3);
    p[0][q] = pack2(x1, y1);
    p[1][q] = pack2(x2, y2);
    p[2][q] = pack2(x3, y3);
  }
#pragma unroll
  for (int pl = 0; pl < 3; ++pl)
    *reinterpret_cast<uint4*>(img + pl * APLANE_BYTES + off) = make_uint4(p[pl][0], p[pl][1], p[pl][2], p[pl][3]);
}

// Starts the copy of one 24 KB V image (global, 16-byte aligned) into shared memory with
// cp.async (16 bytes per thread and step) and commits it as one group: the caller waits for
// the group (cp.async.wait_group) before the MMA phase that reads the image.
__device__ __forceinline__ void copy_vimg_async(uint8_t* dst, const uint8_t* __restrict__ src, int tid) {
#pragma unroll
  for (int i = 0; i < VIMG_BYTES / (16 * 256); ++i) {
    const int e = tid + i * 256;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + 16 * e)), "l"(src + 16 * e)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Instruction descriptors, kind::f16: D float32, A and B bfloat16, M = 128, N = 64; B is
// always the MN-major V image; A is K-major (S blocks) or MN-major (transposed operands).
constexpr uint32_t IDESC_N64 = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((64u >> 3) << 17) |
                               ((128u >> 4) << 24);
constexpr uint32_t IDESC_A_MN = 1u << 15;

struct TcApplyCtl {
  uint32_t bar;          // mbarrier address (shared)
  uint32_t tmem;         // tensor-memory base of this CTA (256 columns)
  uint32_t ph;           // phase parity of the next wait
  unsigned long long wait_ns;
  int* status;
  int ok;                // 0 after a wait that gave up (uniform over the CTA)
};

// One product phase: the A image (three planes, K-major or MN-major) times the V image into
// tensor-memory columns [dcol, dcol + 64), all six cross terms over K = 64 (24 MMAs issued by
// one thread), then every thread waits for their completion.  Returns false (for every
// thread) if the wait gave up; the CTA then drains and stops.
__device__ __forceinline__ bool mma_phase(TcApplyCtl& c, uint32_t a_img, bool a_mn, uint32_t v_img, uint32_t dcol,
                                          int tid) {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idesc = IDESC_N64 | (a_mn ? IDESC_A_MN : 0u);
    constexpr int TI[6] = {0, 0, 1, 0, 1, 2}, TJ[6] = {0, 1, 0, 2, 1, 0};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int t = 0; t < 6; ++t) {
        const uint32_t ab = a_img + uint32_t(TI[t]) * APLANE_BYTES;
        const uint64_t ad = a_mn ? smem_desc(ab + kk * 2048, 8192, 1024) : smem_desc(ab + kk * 32, 16, 1024);
        const uint64_t bd = smem_desc(v_img + uint32_t(TJ[t]) * VPLANE_BYTES + kk * 2048, 8192, 1024);
        tc_mma(c.tmem + dcol, ad, bd, idesc, (kk | t) ? 1u : 0u);
      }
    }
    tc_commit(c.bar);
  }
  const uint32_t want = c.ph;
  c.ph ^= 1u;
  const bool ok = mbar_wait(c.bar, want, c.wait_ns);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) raise_status(c.status, KF_ERR_TIMEOUT, WAIT_MMA_DONE);
    mbar_wait(c.bar, want);  // the issued MMAs still read shared memory: drain (long limit)
    c.ok = 0;
    return false;
  }
  tc_fence_after();
  return true;
}

// A task of the tensor-core apply: a super-tile (super-pairs P <= Q; super-pair P = pairs 2P
// and 2P + 1) of C, or a 64 x 256 panel (pair q, columns 256 cb ..) of Qt.
struct TcTask {
  int kind;  // 0: C super-tile, 1: Qt panel
  int u, P, Q, q, cb;
};

// Advances g (in steps of the grid) to the next task that runs and decodes it; false if none
// is left.  A task runs unless its problem has converged or all its pairs skipped rotation.
__device__ __forceinline__ bool next_tc_task(int& g, int total, int per_u, int nsup, int nsp, int npairs,
                                             const int* __restrict__ skipall, const int* __restrict__ conv,
                                             TcTask& t) {
  for (; g < total; g += gridDim.x) {
    const int u = g / per_u;
    int task = g - u * per_u;
    if (conv[u]) continue;
    const int* skip = skipall + int64_t(u) * npairs;
    if (task < nsup) {
      // row P of the upper triangle of super-tiles holds nsp - P of them
      const int n2 = 2 * nsp + 1;
      int P = int((float(n2) - sqrtf(float(n2) * float(n2) - 8.f * float(task))) * 0.5f);
      P = P < 0 ? 0 : (P > nsp - 1 ? nsp - 1 : P);
      while (P > 0 && P * (n2 - P) / 2 > task) --P;
      while (P + 1 < nsp && (P + 1) * (n2 - P - 1) / 2 <= task) ++P;
      const int Q = P + (task - P * (n2 - P) / 2);
      if (skip[2 * P] && skip[2 * P + 1] && skip[2 * Q] && skip[2 * Q + 1]) continue;
      t.kind = 0; t.u = u; t.P = P; t.Q = Q; t.q = 0; t.cb = 0;
      return true;
    }
    task -= nsup;
    const int cb = task / npairs, q = task - cb * npairs;
    if (skip[q]) continue;
    t.kind = 1; t.u = u; t.P = 0; t.Q = 0; t.q = q; t.cb = cb;
    return true;
  }
  return false;
}

// Issues the global loads of a task's float32 operand into R (16 float4 per thread): a
// super-tile's S = C[rows of P][cols of Q] (warp w rows w + 8 i, lane l columns 4 l ..), or a
// panel's two 128-column halves (rows w + 8 i of the pair, columns 4 l .. of each half).
// The rows of task t into R[lo .. hi) only (the registers freed so far).
__device__ __forceinline__ void load_tc_task_part(const TcTask& t, float4* R, const float* __restrict__ Call,
                                                  const float* __restrict__ Qtall, int64_t sp, int nblk, int step,
                                                  int warp, int lane, int lo, int hi) {
  if (t.kind == 0) {
    const float* C = Call + int64_t(t.u) * sp * sp;
    const int cl = 4 * lane, qp = 2 * t.Q + (cl >> 6);
    const int64_t gcol = int64_t(((cl >> 5) & 1) ? rr_pos(nblk - 1 - qp, step, nblk) : rr_pos(qp, step, nblk)) * JB +
                         (cl & 31);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < lo || i >= hi) continue;
      const int r = warp + 8 * i, pp = 2 * t.P + (r >> 6);
      const int64_t grow = int64_t(((r >> 5) & 1) ? rr_pos(nblk - 1 - pp, step, nblk) : rr_pos(pp, step, nblk)) * JB +
                           (r & 31);
      R[i] = *reinterpret_cast<const float4*>(C + grow * sp + gcol);
    }
  } else {
    const float* Qt = Qtall + int64_t(t.u) * sp * sp;
    const int b0 = rr_pos(t.q, step, nblk), b1 = rr_pos(nblk - 1 - t.q, step, nblk);
    const int64_t col0 = int64_t(t.cb) * 256;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (col0 + 128 * h < sp) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (8 * h + i < lo || 8 * h + i >= hi) continue;
          const int r = warp + 8 * i;
          R[8 * h + i] = *reinterpret_cast<const float4*>(Qt + gidx(r, b0, b1) * sp + col0 + 128 * h + 4 * lane);
        }
      }
    }
  }
}
__device__ __forceinline__ void load_tc_task(const TcTask& t, float4* R, const float* __restrict__ Call,
                                             const float* __restrict__ Qtall, int64_t sp, int nblk, int step,
                                             int warp, int lane) {
  if (t.kind == 0) {
    const float* C = Call + int64_t(t.u) * sp * sp;
    const int cl = 4 * lane, qp = 2 * t.Q + (cl >> 6);
    const int64_t gcol = int64_t(((cl >> 5) & 1) ? rr_pos(nblk - 1 - qp, step, nblk) : rr_pos(qp, step, nblk)) * JB +
                         (cl & 31);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int r = warp + 8 * i, pp = 2 * t.P + (r >> 6);
      const int64_t grow = int64_t(((r >> 5) & 1) ? rr_pos(nblk - 1 - pp, step, nblk) : rr_pos(pp, step, nblk)) * JB +
                           (r & 31);
      R[i] = *reinterpret_cast<const float4*>(C + grow * sp + gcol);
    }
  } else {
    const float* Qt = Qtall + int64_t(t.u) * sp * sp;
    const int b0 = rr_pos(t.q, step, nblk), b1 = rr_pos(nblk - 1 - t.q, step, nblk);
    const int64_t col0 = int64_t(t.cb) * 256;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (col0 + 128 * h < sp) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = warp + 8 * i;
          R[8 * h + i] = *reinterpret_cast<const float4*>(Qt + gidx(r, b0, b1) * sp + col0 + 128 * h + 4 * lane);
        }
      }
    }
  }
}

__device__ __forceinline__ const uint8_t* vimg_src(const uint8_t* Vimg, const uint8_t* Iimg, const int* skipall,
                                                   int u, int npairs, int pair) {
  return skipall[int64_t(u) * npairs + pair] ? Iimg : Vimg + (int64_t(u) * npairs + pair) * VIMG_BYTES;
}

// Persistent apply of one Jacobi step on the tensor cores over the tasks above.  Tasks whose
// pairs all skipped their rotation are not run; a skipped pair inside a run task enters with
// the identity image (exact in three planes).  Latency hiding inside a CTA: the next task's
// rows are loaded into registers as soon as the current task has staged its own, and its V
// images are copied (cp.async) as soon as the current task's last product has completed, so
// both overlap the current task's remaining products and its stores.
__global__ void __launch_bounds__(256, 2) jac_apply_tc_kernel(
    float* __restrict__ Call, float* __restrict__ Qtall, int64_t sp, int nblk, int step,
    const uint8_t* __restrict__ Vimg, const uint8_t* __restrict__ Iimg, const int* __restrict__ skipall,
    const int* __restrict__ conv, int nsup, int nsp, int per_u, int total, unsigned long long* __restrict__ ctr,
    int* status, unsigned long long wait_ns) {
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Abuf = sm;
  uint8_t* Vb0 = sm + AIMG_BYTES;
  uint8_t* Vb1 = Vb0 + VIMG_BYTES;
  uint64_t* bar = reinterpret_cast<uint64_t*>(Vb1 + VIMG_BYTES);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npairs = nblk / 2;

  if (tid == 0) {
    mbar_init(smem_u32(bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(tslot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  TcApplyCtl c;
  c.bar = smem_u32(bar);
  c.tmem = *tslot;
  c.ph = 0;
  c.wait_ns = wait_ns;
  c.status = status;
  c.ok = 1;
  const uint32_t a_img = smem_u32(Abuf), v0 = smem_u32(Vb0), v1 = smem_u32(Vb1);
  const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
  unsigned long long bytes = 0, flops = 0;

  TcTask cur, nxt;
  float4 R[16];
  int g = blockIdx.x;
  bool have = next_tc_task(g, total, per_u, nsup, nsp, npairs, skipall, conv, cur);
  if (have) {
    load_tc_task(cur, R, Call, Qtall, sp, nblk, step, warp, lane);
    if (cur.kind == 0) {
      copy_vimg_async(Vb0, vimg_src(Vimg, Iimg, skipall, cur.u, npairs, 2 * cur.Q), tid);
      copy_vimg_async(Vb1, vimg_src(Vimg, Iimg, skipall, cur.u, npairs, 2 * cur.Q + 1), tid);
    } else {
      copy_vimg_async(Vb0, vimg_src(Vimg, Iimg, skipall, cur.u, npairs, cur.q), tid);
    }
  }
  while (have && c.ok) {
    int g2 = g + gridDim.x;
    bool have2 = false;
    if (cur.kind == 0) {
      // ---------------- C super-tile (P, Q)
      const int u = cur.u, P = cur.P, Q = cur.Q;
      const int pr[2] = {2 * P, 2 * P + 1}, qr[2] = {2 * Q, 2 * Q + 1};
      const bool diag = P == Q;
      float* C = Call + int64_t(u) * sp * sp;
      int pb[2][2], qb[2][2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        pb[i][0] = rr_pos(pr[i], step, nblk); pb[i][1] = rr_pos(nblk - 1 - pr[i], step, nblk);
        qb[i][0] = rr_pos(qr[i], step, nblk); qb[i][1] = rr_pos(nblk - 1 - qr[i], step, nblk);
      }
      const int cl = 4 * lane;
      have2 = next_tc_task(g2, total, per_u, nsup, nsp, npairs, skipall, conv, nxt);
      // step 1a: U[:, 0:64] = S[:, q pair 0] V_q0   (lanes 0..15 hold those columns); their
      // registers are then free and start fetching the next task's rows at once
      if (lane < 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) put4(Abuf, akm_off(warp + 8 * i, cl), R[i]);
        if (have2) load_tc_task(nxt, R, Call, Qtall, sp, nblk, step, warp, lane);
      }
      cp_async_wait<0>();
      if (!mma_phase(c, a_img, false, v0, 0, tid)) break;
      copy_vimg_async(Vb0, vimg_src(Vimg, Iimg, skipall, u, npairs, pr[0]), tid);  // during step 1b
      // step 1b: U[:, 64:128] = S[:, q pair 1] V_q1 (lanes 16..31), then their next rows
      if (lane >= 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) put4(Abuf, akm_off(warp + 8 * i, cl - 64), R[i]);
        if (have2) load_tc_task(nxt, R, Call, Qtall, sp, nblk, step, warp, lane);
      }
      if (!mma_phase(c, a_img, false, v1, 64, tid)) break;
      copy_vimg_async(Vb1, vimg_src(Vimg, Iimg, skipall, u, npairs, pr[1]), tid);  // during step 2a
      // step 2: D_p = U_p^T V_p for p pair 0 (U rows 0..63) and 1 (rows 64..127): the threads of
      // TMEM lanes of rows of p write U_p^T (M = U column, K = row within p) as MN-major planes
      for (int pp = 0; pp < 2; ++pp) {
        if (((warp & 3) >> 1) == pp) {
          const int k = (warp & 1) * 32 + lane;      // row within pair pp
          const int m0 = (warp >> 2) * 64;           // U columns m0 .. m0 + 63
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
            tmem_ld32(c.tmem + lane_base + uint32_t(m0 + 32 * h), v);
#pragma unroll
            for (int q = 0; q < 4; ++q) put8(Abuf, amn_off(m0 + 32 * h + 8 * q, k), v + 8 * q);
          }
        }
        if (pp == 0) cp_async_wait<1>(); else cp_async_wait<0>();
        if (!mma_phase(c, a_img, true, pp ? v1 : v0, 128 + 64 * pp, tid)) break;
      }
      if (!c.ok) break;
      if (have2) {  // both V buffers are free: the next task's first images
        if (nxt.kind == 0) {
          copy_vimg_async(Vb0, vimg_src(Vimg, Iimg, skipall, nxt.u, npairs, 2 * nxt.Q), tid);
          copy_vimg_async(Vb1, vimg_src(Vimg, Iimg, skipall, nxt.u, npairs, 2 * nxt.Q + 1), tid);
        } else {
          copy_vimg_async(Vb0, vimg_src(Vimg, Iimg, skipall, nxt.u, npairs, nxt.q), tid);
        }
      }
      // epilogue: D_p (lane = column c of Q, TMEM column n = row of pair p) -> C[p rows][Q cols]
      // and, mirrored, C[Q cols][p rows]; a diagonal super-tile writes the pair-0 x pair-1 tile
      // and the upper halves of its two diagonal tiles, each with its mirror (C stays exactly
      // symmetric).
      const int cc = (warp & 3) * 32 + lane;
      const int64_t gc = int64_t(qb[cc >> 6][(cc >> 5) & 1]) * JB + (cc & 31);
      const int nh = warp >> 2;                      // rows 32 nh .. 32 nh + 31 of the pair
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        const int qq = cc >> 6;
        if (diag && pp > qq) continue;               // uniform per warp (cc >> 6 fixed per warp)
        uint32_t v[32];
        tmem_ld32(c.tmem + lane_base + uint32_t(128 + 64 * pp + 32 * nh), v);
        const int64_t rb = int64_t(pb[pp][nh]) * JB;  // the 32 rows lie in one block
        if (diag && pp == qq) {
          const int cl2 = cc & 63;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int n = 32 * nh + j;
            if (n <= cl2) {
              C[(rb + j) * sp + gc] = __uint_as_float(v[j]);
              C[gc * sp + rb + j] = __uint_as_float(v[j]);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) C[(rb + j) * sp + gc] = __uint_as_float(v[j]);
          float* mr = C + gc * sp + rb;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4*>(mr)[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                          __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        }
      }
      bytes += 65536ull + (diag ? 65536ull : 131072ull);
      flops += 96ull * 262144ull;
    } else {
      // ---------------- Qt panel: rows of pair q, columns 256 cb .. 256 cb + 255 (the second
      // 128-column half only where the rows are that long), each half one product
      const int u = cur.u, q = cur.q;
      float* Qt = Qtall + int64_t(u) * sp * sp;
      const int b0 = rr_pos(q, step, nblk), b1 = rr_pos(nblk - 1 - q, step, nblk);
      const int64_t col0 = int64_t(cur.cb) * 256;
      const int halves = col0 + 128 < sp ? 2 : 1;     // uniform over the CTA
      bool fine = true;
      have2 = next_tc_task(g2, total, per_u, nsup, nsp, npairs, skipall, conv, nxt);
      for (int h = 0; h < halves && fine; ++h) {
        // A = half^T (M = column of the half, K = row of the pair), MN-major
#pragma unroll
        for (int i = 0; i < 8; ++i) put4(Abuf, amn_off(4 * lane, warp + 8 * i), R[8 * h + i]);
        // the registers of this half (of both halves after the last one) fetch the next task
        if (have2) load_tc_task_part(nxt, R, Call, Qtall, sp, nblk, step, warp, lane, 8 * h,
                                     h + 1 == halves ? 16 : 8 * h + 8);
        cp_async_wait<0>();
        fine = mma_phase(c, a_img, true, v0, 64 * h, tid);
      }
      if (!fine) break;
      if (have2) {
        if (nxt.kind == 0) {
          copy_vimg_async(Vb0, vimg_src(Vimg, Iimg, skipall, nxt.u, npairs, 2 * nxt.Q), tid);
          copy_vimg_async(Vb1, vimg_src(Vimg, Iimg, skipall, nxt.u, npairs, 2 * nxt.Q + 1), tid);
        } else {
          copy_vimg_async(Vb0, vimg_src(Vimg, Iimg, skipall, nxt.u, npairs, nxt.q), tid);
        }
      }
      const int cc = (warp & 3) * 32 + lane;
      const int nh = warp >> 2;
      const int64_t rb = int64_t(nh ? b1 : b0) * JB;
      for (int h = 0; h < halves; ++h) {
        uint32_t v[32];
        tmem_ld32(c.tmem + lane_base + uint32_t(64 * h + 32 * nh), v);
#pragma unroll
        for (int j = 0; j < 32; ++j) Qt[(rb + j) * sp + col0 + 128 * h + cc] = __uint_as_float(v[j]);
      }
      bytes += 65536ull * uint64_t(halves);
      flops += 24ull * 262144ull * uint64_t(halves);
    }
    cur = nxt;
    have = have2;
    g = g2;
  }
  cp_async_wait<0>();  // no copy into this CTA's shared memory may still be in flight at exit
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(c.tmem) : "memory");
  }
  if (ctr && tid == 0) {
    if (flops) atomicAdd(ctr, flops);
    if (bytes) atomicAdd(ctr + 1, bytes);
  }
}

// The identity in the V image layout: plane 1 = I, planes 2 and 3 zero.
__global__ void ident_img_kernel(uint8_t* __restrict__ img) {
  for (int e = threadIdx.x; e < VIMG_BYTES / 16; e += blockDim.x) reinterpret_cast<uint4*>(img)[e] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (threadIdx.x < JP)
    *reinterpret_cast<__nv_bfloat16*>(img + vimg_off(threadIdx.x, threadIdx.x)) = __float2bfloat16_rn(1.f);
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
  p.sp = (s + 127) / 128 * 128;  // an even number of pairs: whole 128 x 128 super-tiles
  p.nblk = int(p.sp / JB);
  p.npairs = p.nblk / 2;
  return p;
}

struct SvdBufs {
  float *C, *Q, *flo, *Y, *sig, *qinv, *Qs, *Ys, *Bw, *Vw;
  uint8_t *Vimg, *Iimg;
  PlaneBuf wpl, qpl;  // three-plane copies of one problem's W~ (or C) and of its eigenvector rows
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
  b.Vimg = cv.take<uint8_t>(size_t(nu) * pl.npairs * VIMG_BYTES);
  b.Iimg = cv.take<uint8_t>(VIMG_BYTES);
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
  b.wpl = take_planes(cv, m_max, n_max, 3);
  b.qpl = take_planes(cv, s, s, 3);
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
  float *C = bf.C, *Q = bf.Q, *flo = bf.flo, *sig = bf.sig, *qinv = bf.qinv;
  int *skip = bf.skip, *conv = bf.conv, *perm = bf.perm;
  unsigned* off = bf.off;

  const bool prof = ctx->prof_enabled;
  unsigned long long* flops = prof ? ctx->prof_flops() : nullptr;
  if (prof) {
    for (int e = 0; e < 5; ++e)
      if (!ctx->prof_ev[e]) KF_CUDA(cudaEventCreate(&ctx->prof_ev[e]));
    KF_CUDA(cudaMemsetAsync(flops, 0, 2 * sizeof(unsigned long long), st));
    KF_CUDA(cudaEventRecord(ctx->prof_ev[0], st));
    ctx->prof_kev_used = 0;
    ctx->prof_steps = int64_t(max_sweeps) * (pl.nblk - 1);
    ctx->prof_valid = true;
  }
  // Gram of the smaller side, lower triangle, on the tensor cores with W~ as three bfloat16
  // planes (all six cross terms, float32 accumulation over K chunks of 1024): float32-level
  // products, as the eigenvalues need.
  for (int i = 0; i < nu; ++i) {
    const kf_svd_problem& p = pr[i];
    float* Ci = C + int64_t(i) * pl.sp * pl.sp;
    if (sym) {  // the matrix itself
      KF_TRY(launch_copy(p.Wt, p.ldw, Ci, pl.sp, s, s, false, st));
      continue;
    }
    Planes pw;
    KF_TRY(split_f32(p.Wt, p.ldw, p.m, p.n, bf.wpl, &pw, st));
    ProductOpts o;
    o.lower = true;
    if (kf_gram_side(p.m, p.n) == KF_SIDE_RIGHT) {  // W~^T W~: A = W~^T (MN-major), B = W~ (MN-major)
      KF_TRY(tc_product(ctx, s, s, p.m, pw, true, pw, true, KR_FULL, Ci, pl.sp, st, o));
    } else {                                        // W~ W~^T: A = W~ (K-major), B = W~^T (K-major)
      KF_TRY(tc_product(ctx, s, s, p.n, pw, false, pw, false, KR_FULL, Ci, pl.sp, st, o));
    }
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

  // tensor-core apply: super-tiles of two pairs by two pairs (on or above the diagonal) and
  // 128-column panels of Qt per pair
  const int nsp = pl.npairs / 2;
  const int nsup = nsp * (nsp + 1) / 2;
  const int ntile_q = int((pl.sp + 255) / 256) * pl.npairs;
  const size_t apply_smem = 1024 + size_t(AIMG_BYTES) + 2 * size_t(VIMG_BYTES) + 64;
  const int per_u = nsup + ntile_q;
  const int64_t total_tasks = int64_t(per_u) * nu;
  if (total_tasks > 0x7fffffff) return fail(KF_ERR_UNSUPPORTED, "whitened_svd: too many Jacobi tasks");
  const int apply_grid = int(total_tasks < int64_t(ctx->sm_count) * 2 ? total_tasks : int64_t(ctx->sm_count) * 2);
  static std::atomic<unsigned long long> attr_done{0};
  KF_TRY(set_attr_once(attr_done, [&] {
    KF_TRY(check_cuda(cudaFuncSetAttribute(jac_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           int(JAC_SOLVE_SMEM)), "jac_solve smem attribute"));
    return check_cuda(cudaFuncSetAttribute(jac_apply_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           int(apply_smem)), "jac_apply_tc smem attribute");
  }));
  if ((reinterpret_cast<uintptr_t>(C) & 15) || (reinterpret_cast<uintptr_t>(Q) & 15) ||
      (reinterpret_cast<uintptr_t>(bf.Vimg) & 15) || (reinterpret_cast<uintptr_t>(bf.Iimg) & 15))
    return fail(KF_ERR_INVALID, "whitened_svd: workspace not 16-byte aligned");
  ident_img_kernel<<<1, 256, 0, st>>>(bf.Iimg); note_launch();
  KF_TRY(check_cuda(cudaGetLastError(), "ident_img_kernel"));
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
      jac_solve_kernel<<<dim3(pl.npairs, nu), 256, JAC_SOLVE_SMEM, st>>>(C, pl.sp, pl.nblk, step, bf.Vimg, skip, conv, off, flo,
                                                           tol, max_inner); note_launch();
      KF_TRY(check_cuda(cudaGetLastError(), "jac_solve_kernel"));
      if (prof) KF_CUDA(cudaEventRecord(kev[1], st));
      jac_apply_tc_kernel<<<apply_grid, 256, apply_smem, st>>>(C, Q, pl.sp, pl.nblk, step, bf.Vimg, bf.Iimg, skip,
                                                               conv, nsup, nsp, per_u, int(total_tasks), flops,
                                                               ctx->d_status, ctx->wait_ns); note_launch();
      KF_TRY(check_cuda(cudaGetLastError(), "jac_apply_tc_kernel"));
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
    // Yt = Qt W~^T (right side, y_j = W~ q_j) or Qt W~ (left side, y_j = W~^T q_j), on the
    // tensor cores with both operands as three bfloat16 planes (the images enter sigma at
    // first order, so they need float32-level products)
    Planes pq, pw;
    KF_TRY(split_f32(Qti, pl.sp, s, s, bf.qpl, &pq, st));
    KF_TRY(split_f32(p.Wt, p.ldw, p.m, p.n, bf.wpl, &pw, st));
    KF_TRY(tc_product(ctx, s, len_y, s, pq, false, pw, !right, KR_FULL, Yi, lyM, st));
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
  unsigned long long f[2] = {0, 0};
  KF_CUDA(cudaMemcpy(f, ctx->prof_flops(), sizeof(f), cudaMemcpyDeviceToHost));
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
  out->jacobi_apply_flops = double(f[0]);
  out->jacobi_apply_bytes = double(f[1]);
  return KF_OK;
}

}  // namespace kf
