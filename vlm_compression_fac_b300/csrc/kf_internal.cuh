// Internal declarations shared by the libkfsvd translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include <atomic>
#include <string>
#include <vector>

#include "../../include/kfsvd.h"

namespace kf {

// Device status word layout (int32[4]): [0] error code (first one wins), [1] detail.
enum : int { ST_CODE = 0, ST_INFO = 1 };

// Wait-site codes reported with KF_ERR_TIMEOUT.
enum : int { WAIT_TMA_EMPTY = 1, WAIT_TMA_FULL = 2, WAIT_MMA_DONE = 3, WAIT_DRAIN = 4, WAIT_LOOKBACK = 5 };

__device__ __forceinline__ void raise_status(int* st, int code, int info) {
  if (atomicCAS(st + ST_CODE, 0, code) == 0) st[ST_INFO] = info;
}

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace kf

struct kf_ctx {
  int device = 0;
  int sm_count = 148;
  int cc_major = 0, cc_minor = 0;
  int* d_status = nullptr;          // int32[4] on the device: code, info, Jacobi flag, spare
  int* h_flag = nullptr;            // pinned host int: the Jacobi convergence poll
  kf::PFN_encodeTiled encode = nullptr;
  unsigned long long wait_ns = 4000000000ull;  // limit of the tensor-core pipeline waits
  // internal streams for independent chains of work inside one call (factor_covariances),
  // created on first use, joined back into the caller's stream before the call returns
  static constexpr int NSTREAMS = 8;
  cudaStream_t streams[NSTREAMS] = {};
  cudaEvent_t stream_ev[NSTREAMS + 1] = {};
  // whitened_svd profile (events on the caller's stream; flop counter at d_status + 4)
  bool prof_enabled = false;
  bool prof_valid = false;
  cudaEvent_t prof_ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  int64_t prof_steps = 0;
  // per-step events of the profiled Jacobi (solve start, apply start, apply end per step)
  std::vector<cudaEvent_t> prof_kev;
  int64_t prof_kev_used = 0;
  unsigned long long* prof_flops() { return reinterpret_cast<unsigned long long*>(d_status + 4); }
};

namespace kf {

// Counts kernel launches made by the library (reported by kf_launch_count).
void note_launch();

// Host-side error reporting (thread-local message).
kf_status fail(kf_status st, const std::string& msg);
kf_status check_cuda(cudaError_t e, const char* what);
#define KF_TRY(expr)                        \
  do {                                      \
    kf_status _s = (expr);                  \
    if (_s != KF_OK) return _s;             \
  } while (0)
#define KF_CUDA(expr) KF_TRY(::kf::check_cuda((expr), #expr))

// A kernel's large shared-memory opt-in is an attribute per device: `done` records, for each
// device below 64, that `set()` has succeeded there; it is called on the current device until
// then (devices from 64 up: on every call).  Concurrent first calls both set it (idempotent).
template <typename F>
kf_status set_attr_once(std::atomic<unsigned long long>& done, F&& set) {
  int dev = 0;
  KF_CUDA(cudaGetDevice(&dev));
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return KF_OK;
  KF_TRY(set());
  if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return KF_OK;
}

// Bump allocator over a caller workspace (256-byte aligned slices).
struct Carve {
  char* base;
  size_t cap, off = 0;
  bool dry;  // sizing pass: base may be null
  Carve(void* b, size_t c, bool dry_run) : base((char*)b), cap(c), dry(dry_run) {}
  template <typename T>
  T* take(size_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = dry ? nullptr : (T*)(base + off);
    off += count * sizeof(T);
    return p;
  }
  bool fits() const { return off <= cap; }
};

// ---------------------------------------------------------------- SIMT GEMM
// C[M x N] = alpha * op(A) * op(B) + beta * C, float32 accumulation.
// op(A) is M x K: stored row-major M x K (trans_a = false) or K x M (trans_a = true).
// op(B) is K x N: stored row-major K x N (trans_b = false) or N x K (trans_b = true).
enum KRange { KR_FULL = 0, KR_GE_ROW, KR_LE_ROW, KR_GE_COL, KR_LE_COL };
enum OutMask { OUT_ALL = 0, OUT_LOWER = 1 };
struct GemmDesc {
  int64_t M, N, K;
  const void* A; int64_t lda; int64_t sA; bool a_bf16; bool trans_a;
  const void* B; int64_t ldb; int64_t sB; bool b_bf16; bool trans_b;
  float* C; int64_t ldc; int64_t sC;
  float alpha, beta;
  int krange, out_mask, batch;
};
kf_status simt_gemm(const GemmDesc& g, cudaStream_t st);

// --------------------------------------------------------- tcgen05 GEMM / SYRK
// D[M x N] (float32, ldd) (+)= sum over passes p of A_p * B_p with bfloat16 operands in
// global memory.  A_p: M x K, K-major (row-major M x K) or MN-major (row-major K x M).
// B_p: K x N, K-major (row-major N x K) or MN-major (row-major K x N).
struct TcOperand {
  const __nv_bfloat16* ptr;
  int64_t ld;      // elements
  bool mn_major;
};
enum TcSched { TC_FULL = 0, TC_LOWER = 1 };
struct TcGemm {
  int64_t M, N, K;
  int npass;         // 1..6
  TcOperand a[6], b[6];
  float* D; int64_t ldd;
  bool accumulate;   // D += result (else D = result)
  bool negate;       // the result enters with a minus sign (D -= ..., or D = -...)
  int sched;         // TC_LOWER: only tiles touching i >= j, only i >= j written
  int krange;        // KR_FULL / KR_GE_ROW / KR_LE_ROW / KR_GE_COL / KR_LE_COL
  int64_t kchunk;    // longest K range accumulated inside the tensor cores (0: unbounded);
                     // each chunk's partial result is added to D in float32
};
kf_status tc_gemm(kf_ctx* ctx, const TcGemm& g, cudaStream_t st);

// A matrix operand for the tensor-core engine: bfloat16 planes whose sum is the value
// (one plane for bfloat16 data; two (hi + lo, 16 significant bits) or three (the full 24-bit
// float32 significand) for float32 data), 16-byte aligned rows.
struct Planes {
  const __nv_bfloat16* p[3];
  int64_t ld;
  int n;  // 1, 2 or 3
};
// Room for the planes of a rows x cols operand (rows padded to 8 elements).
struct PlaneBuf {
  __nv_bfloat16* p[3] = {nullptr, nullptr, nullptr};
  int64_t ld = 0;
  int n = 0;
};
PlaneBuf take_planes(Carve& cv, int64_t rows, int64_t cols, int nplanes);
// float32 rows x cols (ld) -> the buffer's planes (two or three).
kf_status split_f32(const float* in, int64_t ld, int64_t rows, int64_t cols, const PlaneBuf& b, Planes* out,
                    cudaStream_t st);
// A caller matrix (bfloat16 or float32) as planes: bfloat16 rows that are already aligned
// are used in place; other bfloat16 rows are copied to an aligned plane; float32 is split.
kf_status as_planes(const void* in, kf_dtype dt, int64_t ld, int64_t rows, int64_t cols, const PlaneBuf& b,
                    Planes* out, cudaStream_t st);
// Tokens (K) summed inside the tensor cores before a partial is added in float32: long
// mixed-sign sums of products (whitening, unwhitening; up to 28672 terms, several planes).
#ifndef KF_PRODUCT_KCHUNK
#define KF_PRODUCT_KCHUNK 1024
#endif
constexpr int64_t PRODUCT_KCHUNK = KF_PRODUCT_KCHUNK;
struct ProductOpts {
  bool accumulate = false;   // D += result
  bool negate = false;       // the result enters negated
  bool lower = false;        // only tiles touching i >= j, only i >= j written
  int64_t kchunk = PRODUCT_KCHUNK;
};
// D (M x N float32, ldd) = A B on the tensor cores, A and B given as planes: every cross
// term A_i B_j with i + j < max(A.n, B.n) (0-based), i.e. all terms down to the last plane's
// weight (at most six, one launch); the omitted terms are below the rounding of the planes
// themselves.  a_mn / b_mn: the operand is stored MN-major (A as K x M rows, B as K x N rows).
kf_status tc_product(kf_ctx* ctx, int64_t M, int64_t N, int64_t K, const Planes& A, bool a_mn, const Planes& B,
                     bool b_mn, int krange, float* D, int64_t ldd, cudaStream_t st,
                     const ProductOpts& o = ProductOpts());

// ------------------------------------------------------------ small kernels
kf_status launch_ffma_probe(int sm_count, int64_t iters, float* sink, double* flops, cudaStream_t st);
kf_status launch_fake_quant(const void* in, kf_dtype dt, int64_t rows, int64_t d, int64_t ld,
                            __nv_bfloat16* out, cudaStream_t st);
kf_status launch_split_bf16(const float* in, int64_t rows, int64_t d, int64_t ld,
                            __nv_bfloat16* hi, __nv_bfloat16* lo, int64_t ldo, cudaStream_t st);
kf_status launch_split3_bf16(const float* in, int64_t rows, int64_t d, int64_t ld, __nv_bfloat16* p1,
                             __nv_bfloat16* p2, __nv_bfloat16* p3, int64_t ldo, cudaStream_t st);
kf_status launch_copy_bf16(const __nv_bfloat16* in, int64_t rows, int64_t d, int64_t ld,
                           __nv_bfloat16* out, int64_t ldo, cudaStream_t st);
kf_status launch_fisher_reduce(const float* P, int64_t ldp, const float* Q, int64_t ldq, int64_t rows, int64_t cols,
                               double* acc, cudaStream_t st);
kf_status launch_coldot(const float* D, int64_t ldd, const float* E, int64_t lde, int64_t rows, int64_t cols,
                        double* acc, float* keys, cudaStream_t st);
kf_status launch_sub_from(const void* W, kf_dtype dt, int64_t ldw, float* D, int64_t ldd, int64_t rows, int64_t cols,
                          cudaStream_t st);
kf_status launch_gather2d(const void* src, kf_dtype dt, int64_t lds, int64_t src_rows, int64_t src_cols,
                          const int64_t* ri, int64_t rows, const int64_t* ci, int64_t cols, void* dst, int64_t ldd,
                          int* status, cudaStream_t st);
kf_status launch_compact_mask(const unsigned char* mask, int64_t n, int want, int64_t* idx, int64_t* count,
                              cudaStream_t st);
kf_status launch_fisher_finalize(const double* sum, int64_t n, int64_t n_tokens, float* keys, cudaStream_t st);
kf_status launch_finalize(float* C, int64_t ldc, int64_t d, int64_t n_tokens, float lambda,
                          float* scratch, cudaStream_t st);
kf_status launch_copy(const float* src, int64_t lds, float* dst, int64_t ldd, int64_t rows,
                      int64_t cols, bool transpose, cudaStream_t st);
kf_status launch_transpose_inplace(float* A, int64_t lda, int64_t n, cudaStream_t st);
kf_status launch_scale_cols(float* A, int64_t lda, int64_t rows, int64_t cols,
                            const float* s, bool invert, cudaStream_t st);
kf_status launch_scale_rows(float* A, int64_t lda, int64_t rows, int64_t cols,
                            const float* s, bool invert, cudaStream_t st);

// Cholesky: A (n x n, lda) lower triangle in, L out in place (zeros above), and the
// inverses of the 64 x 64 diagonal blocks into dinv (n x 64 scratch, row-major).  Column
// strips of CHOL_STRIP; trailing updates on the tensor cores (workspace: chol_workspace_bytes).
constexpr int CHOL_NB = 64;
constexpr int64_t CHOL_STRIP = 256;
size_t chol_workspace_bytes(int64_t n);
kf_status cholesky_lower(kf_ctx* ctx, float* A, int64_t lda, int64_t n, float* dinv, void* ws, size_t ws_bytes,
                         cudaStream_t st);
// Inverse of a lower triangular L (n x n) into M (lower, zeros above), using the diagonal
// block inverses produced by cholesky_lower; tmp: trtri_tmp_floats(n) floats; ws:
// trtri_workspace_bytes(n) (tensor-core doubling levels).
kf_status trtri_lower(kf_ctx* ctx, const float* L, int64_t ldl, int64_t n, const float* dinv,
                      float* M, int64_t ldm, float* tmp, void* ws, size_t ws_bytes, cudaStream_t st);
size_t trtri_tmp_floats(int64_t n);
size_t trtri_workspace_bytes(int64_t n);

}  // namespace kf
