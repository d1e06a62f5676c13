// Float32 operands of the tensor-core engine as bfloat16 planes, and products of such
// operands with every cross term down to the last plane's weight.
#include "kf_internal.cuh"

namespace kf {

PlaneBuf take_planes(Carve& cv, int64_t rows, int64_t cols, int nplanes) {
  PlaneBuf b;
  b.ld = (cols + 7) / 8 * 8;
  b.n = nplanes;
  for (int i = 0; i < nplanes; ++i) b.p[i] = cv.take<__nv_bfloat16>(size_t(rows) * b.ld);
  return b;
}

kf_status split_f32(const float* in, int64_t ld, int64_t rows, int64_t cols, const PlaneBuf& b, Planes* out,
                    cudaStream_t st) {
  if (b.n == 3) {
    KF_TRY(launch_split3_bf16(in, rows, cols, ld, b.p[0], b.p[1], b.p[2], b.ld, st));
  } else {
    KF_TRY(launch_split_bf16(in, rows, cols, ld, b.p[0], b.p[1], b.ld, st));
  }
  *out = Planes{{b.p[0], b.p[1], b.n == 3 ? b.p[2] : nullptr}, b.ld, b.n};
  return KF_OK;
}

kf_status as_planes(const void* in, kf_dtype dt, int64_t ld, int64_t rows, int64_t cols, const PlaneBuf& b,
                    Planes* out, cudaStream_t st) {
  if (dt == KF_F32) return split_f32(static_cast<const float*>(in), ld, rows, cols, b, out, st);
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(in);
  if ((reinterpret_cast<uintptr_t>(x) & 15) == 0 && (ld % 8) == 0) {
    *out = Planes{{x, nullptr, nullptr}, ld, 1};
    return KF_OK;
  }
  KF_TRY(launch_copy_bf16(x, rows, cols, ld, b.p[0], b.ld, st));
  *out = Planes{{b.p[0], nullptr, nullptr}, b.ld, 1};
  return KF_OK;
}

kf_status tc_product(kf_ctx* ctx, int64_t M, int64_t N, int64_t K, const Planes& A, bool a_mn, const Planes& B,
                     bool b_mn, int krange, float* D, int64_t ldd, cudaStream_t st, const ProductOpts& o) {
  const int L = A.n > B.n ? A.n : B.n;
  TcGemm g{};
  g.M = M; g.N = N; g.K = K;
  g.D = D; g.ldd = ldd; g.accumulate = o.accumulate; g.negate = o.negate;
  g.sched = o.lower ? TC_LOWER : TC_FULL; g.krange = krange;
  g.kchunk = o.kchunk;
  g.npass = 0;
  for (int i = 0; i < A.n; ++i)
    for (int j = 0; j < B.n; ++j)
      if (i + j < L) {
        g.a[g.npass] = TcOperand{A.p[i], A.ld, a_mn};
        g.b[g.npass] = TcOperand{B.p[j], B.ld, b_mn};
        ++g.npass;
      }
  return tc_gemm(ctx, g, st);
}

}  // namespace kf
