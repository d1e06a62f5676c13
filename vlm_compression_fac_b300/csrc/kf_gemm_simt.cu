// float32 SIMT GEMM for the steps that need float32-accurate products (Gram matrix,
// Cholesky trailing updates, triangular inverses, Rayleigh products, re-orthogonalisation).
// 128 x 128 output tile per 256-thread CTA, 8 x 8 register micro-tile per thread,
// k-slices of 8 staged in double-buffered shared memory.  Triangular operands skip the
// k-range that is structurally zero (KRange); OUT_LOWER computes and writes only i >= j.
#include "kf_internal.cuh"

namespace kf {
namespace {

constexpr int BM = 128, BN = 128, BK = 8, PAD = 4;

template <bool BF>
__device__ __forceinline__ float ld_elem(const void* p, int64_t idx) {
  if (BF) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[idx]);
  return reinterpret_cast<const float*>(p)[idx];
}

template <bool A_BF, bool TA, bool B_BF, bool TB>
__global__ void __launch_bounds__(256) sgemm_kernel(GemmDesc g) {
  __shared__ __align__(16) float As[2][BK][BM + PAD];
  __shared__ __align__(16) float Bs[2][BK][BN + PAD];

  const int t = threadIdx.x;
  const int64_t m0 = int64_t(blockIdx.y) * BM, n0 = int64_t(blockIdx.x) * BN;
  if (g.out_mask == OUT_LOWER && n0 > m0 + BM - 1) return;
  const int64_t z = blockIdx.z;
  const void* A = g.a_bf16 ? (const void*)((const __nv_bfloat16*)g.A + z * g.sA)
                           : (const void*)((const float*)g.A + z * g.sA);
  const void* B = g.b_bf16 ? (const void*)((const __nv_bfloat16*)g.B + z * g.sB)
                           : (const void*)((const float*)g.B + z * g.sB);
  float* C = g.C + z * g.sC;

  int64_t klo = 0, khi = g.K;
  if (g.krange == KR_GE_ROW) klo = m0;
  else if (g.krange == KR_LE_ROW) khi = min(g.K, m0 + BM);
  else if (g.krange == KR_GE_COL) klo = n0;
  else if (g.krange == KR_LE_COL) khi = min(g.K, n0 + BN);

  // Load mapping.
  int am, ak, bk, bn;
  if (!TA) { am = t >> 1; ak = (t & 1) * 4; } else { ak = t >> 5; am = (t & 31) * 4; }
  if (!TB) { bk = t >> 5; bn = (t & 31) * 4; } else { bn = t >> 1; bk = (t & 1) * 4; }

  float ra[4], rb[4];
  auto load = [&](int64_t k0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int64_t m, k;
      if (!TA) { m = m0 + am; k = k0 + ak + i; } else { m = m0 + am + i; k = k0 + ak; }
      bool ok = m < g.M && k < khi;
      ra[i] = ok ? (TA ? ld_elem<A_BF>(A, k * g.lda + m) : ld_elem<A_BF>(A, m * g.lda + k)) : 0.f;
      int64_t kk, n;
      if (!TB) { kk = k0 + bk; n = n0 + bn + i; } else { kk = k0 + bk + i; n = n0 + bn; }
      ok = n < g.N && kk < khi;
      rb[i] = ok ? (TB ? ld_elem<B_BF>(B, n * g.ldb + kk) : ld_elem<B_BF>(B, kk * g.ldb + n)) : 0.f;
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (!TA) As[buf][ak + i][am] = ra[i]; else As[buf][ak][am + i] = ra[i];
      if (!TB) Bs[buf][bk][bn + i] = rb[i]; else Bs[buf][bk + i][bn] = rb[i];
    }
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  const int tx = t & 15, ty = t >> 4;
  int buf = 0;
  if (klo < khi) {
    load(klo);
    store(0);
    __syncthreads();
    for (int64_t k0 = klo; k0 < khi; k0 += BK) {
      const bool more = k0 + BK < khi;
      if (more) load(k0 + BK);
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        float a[8], b[8];
        *reinterpret_cast<float4*>(a) = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4]);
        *reinterpret_cast<float4*>(a + 4) = *reinterpret_cast<const float4*>(&As[buf][k][64 + ty * 4]);
        *reinterpret_cast<float4*>(b) = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
        *reinterpret_cast<float4*>(b + 4) = *reinterpret_cast<const float4*>(&Bs[buf][k][64 + tx * 4]);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      if (more) {
        store(buf ^ 1);
        __syncthreads();
        buf ^= 1;
      }
    }
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t row = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (row >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t col = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (col >= g.N) continue;
      if (g.out_mask == OUT_LOWER && col > row) continue;
      float v = g.alpha * acc[i][j];
      if (g.beta != 0.f) v = fmaf(g.beta, C[row * g.ldc + col], v);
      C[row * g.ldc + col] = v;
    }
  }
}

template <bool A_BF, bool TA>
kf_status dispatch_b(const GemmDesc& g, dim3 grid, cudaStream_t st) {
  if (g.b_bf16) {
    if (g.trans_b) sgemm_kernel<A_BF, TA, true, true><<<grid, 256, 0, st>>>(g);
    else sgemm_kernel<A_BF, TA, true, false><<<grid, 256, 0, st>>>(g);
  } else {
    if (g.trans_b) sgemm_kernel<A_BF, TA, false, true><<<grid, 256, 0, st>>>(g);
    else sgemm_kernel<A_BF, TA, false, false><<<grid, 256, 0, st>>>(g);
  }
  note_launch();
  return check_cuda(cudaGetLastError(), "sgemm launch");
}

}  // namespace

kf_status simt_gemm(const GemmDesc& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0 || g.batch <= 0) return KF_OK;
  const int64_t gy = (g.M + BM - 1) / BM, gx = (g.N + BN - 1) / BN;
  if (gy > 65535 || g.batch > 65535) return fail(KF_ERR_UNSUPPORTED, "sgemm: grid too large");
  dim3 grid(unsigned(gx), unsigned(gy), unsigned(g.batch));
  if (g.a_bf16) {
    if (g.trans_a) return dispatch_b<true, true>(g, grid, st);
    return dispatch_b<true, false>(g, grid, st);
  }
  if (g.trans_a) return dispatch_b<false, true>(g, grid, st);
  return dispatch_b<false, false>(g, grid, st);
}

}  // namespace kf
