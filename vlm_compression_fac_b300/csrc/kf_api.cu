// C ABI entry points of libkfsvd.so (declared in include/kfsvd.h): argument validation on
// the host, workspace carving, and the launch sequence of each step of the path.
#include "kf_internal.cuh"

#include <cstring>
#include <string>
#include <vector>

namespace kf {
const char* last_error_cstr();
unsigned long long launch_count();
size_t svd_workspace(int32_t nu, int64_t m_max, int64_t n_max, int64_t s);
kf_status svd_run(kf_ctx* ctx, int32_t nu, const kf_svd_problem* pr, float tol, int32_t max_sweeps, void* ws,
                  size_t ws_bytes, cudaStream_t st, bool sym);
kf_status svd_profile_read(kf_ctx* ctx, kf_svd_profile* out);
size_t alloc_workspace(int64_t n, int64_t n_energy);
kf_status alloc_run(kf_ctx* ctx, const float* sigma, const int64_t* off, const int64_t* cost, int32_t n_units,
                    int64_t n, int64_t budget, kf_alloc_mode mode, const int32_t* fixed, const float* weight,
                    int32_t* ranks, float* cut, int64_t* used, void* ws, size_t ws_bytes, cudaStream_t st,
                    unsigned char* keep, double alpha);
int alloc_mode_given_keys();
int alloc_mode_swift_hybrid();
}  // namespace kf

using namespace kf;

namespace {

constexpr int64_t ACC_CHUNK = 8192;   // tokens per preprocessing chunk of float32 input (two planes)
// Tokens per fake-quantised chunk: each chunk is one SYRK launch, which reads and writes the
// whole d x d float32 accumulator once, so chunks are long (at d = 18944 one pass over the
// accumulator moves 2.9 GB; over 32768 tokens the chunk's own rows are 1.2 GB).
constexpr int64_t QAW_CHUNK = 32768;
// Tokens accumulated inside the tensor cores before the partial sum is added to the float32
// covariance in global memory.  The tensor cores' float32 accumulation loses accuracy on
// long sums of positive terms: the error of a diagonal entry grows about linearly with the
// number of tokens summed in one pass (about 6e-4 relative after 131072 tokens, 1e-5 after
// 4096); 2048-token partials keep it near 5e-6.
#ifndef KF_SYRK_KCHUNK
#define KF_SYRK_KCHUNK 2048
#endif
constexpr int64_t SYRK_KCHUNK = KF_SYRK_KCHUNK;
constexpr int FINAL_SLOTS = 1024;

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

kf_status need(bool cond, const char* msg) { return cond ? KF_OK : fail(KF_ERR_INVALID, msg); }

size_t elem_size(kf_dtype d) { return d == KF_BF16 ? 2 : 4; }

}  // namespace

extern "C" {

const char* kf_last_error(void) { return last_error_cstr(); }

uint64_t kf_launch_count(void) { return launch_count(); }

kf_side kf_gram_side(int64_t m, int64_t n) { return n <= m ? KF_SIDE_RIGHT : KF_SIDE_LEFT; }

kf_status kf_create(int device, kf_ctx** out) {
  if (!out) return fail(KF_ERR_INVALID, "kf_create: out is null");
  *out = nullptr;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) return fail(KF_ERR_CUDA, "kf_create: no CUDA device");
  if (device < 0 || device >= count) return fail(KF_ERR_INVALID, "kf_create: bad device index");
  KF_CUDA(cudaSetDevice(device));
  kf_ctx* c = new kf_ctx();
  c->device = device;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
    delete c;
    return fail(KF_ERR_CUDA, "kf_create: cudaGetDeviceProperties failed");
  }
  c->sm_count = prop.multiProcessorCount;
  c->cc_major = prop.major;
  c->cc_minor = prop.minor;
  if (!(prop.major == 10 && prop.minor == 3)) {
    delete c;
    return fail(KF_ERR_UNSUPPORTED, "kf_create: libkfsvd is built for sm_103a (compute capability 10.3)");
  }
  // status int32[4] followed by the finalisation scratch ring
  const size_t bytes = 64 + sizeof(float) * FINAL_SLOTS;
  if (cudaMalloc(&c->d_status, bytes) != cudaSuccess) {
    delete c;
    return fail(KF_ERR_CUDA, "kf_create: cudaMalloc of the status word failed");
  }
  cudaMemset(c->d_status, 0, bytes);
  if (cudaHostAlloc(reinterpret_cast<void**>(&c->h_flag), sizeof(int), cudaHostAllocDefault) != cudaSuccess) {
    cudaFree(c->d_status);
    delete c;
    return fail(KF_ERR_CUDA, "kf_create: cudaHostAlloc of the poll flag failed");
  }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    cudaFree(c->d_status);
    delete c;
    return fail(KF_ERR_CUDA, "kf_create: cuTensorMapEncodeTiled entry point not found");
  }
  c->encode = reinterpret_cast<PFN_encodeTiled>(fn);
  *out = c;
  return KF_OK;
}

void kf_destroy(kf_ctx* ctx) {
  if (!ctx) return;
  for (int i = 0; i < kf_ctx::NSTREAMS; ++i)
    if (ctx->streams[i]) cudaStreamDestroy(ctx->streams[i]);
  for (int i = 0; i <= kf_ctx::NSTREAMS; ++i)
    if (ctx->stream_ev[i]) cudaEventDestroy(ctx->stream_ev[i]);
  for (int e = 0; e < 5; ++e)
    if (ctx->prof_ev[e]) cudaEventDestroy(ctx->prof_ev[e]);
  for (cudaEvent_t e : ctx->prof_kev) cudaEventDestroy(e);
  if (ctx->d_status) cudaFree(ctx->d_status);
  if (ctx->h_flag) cudaFreeHost(ctx->h_flag);
  delete ctx;
}

kf_status kf_fp32_fma_probe(kf_ctx* ctx, int64_t iters, float* sink, double* flops, kf_stream_t stream) {
  if (!ctx) return fail(KF_ERR_INVALID, "kf_fp32_fma_probe: null context");
  if (iters <= 0 || !sink || !flops) return fail(KF_ERR_INVALID, "kf_fp32_fma_probe: arguments");
  return launch_ffma_probe(ctx->sm_count, iters, sink, flops, reinterpret_cast<cudaStream_t>(stream));
}

kf_status kf_set_wait_limit(kf_ctx* ctx, uint64_t limit_ns) {
  if (!ctx) return fail(KF_ERR_INVALID, "kf_set_wait_limit: null context");
  ctx->wait_ns = limit_ns ? static_cast<unsigned long long>(limit_ns) : 4000000000ull;
  return KF_OK;
}

kf_status kf_sync_status(kf_ctx* ctx, kf_stream_t stream, int32_t* info) {
  if (!ctx) return fail(KF_ERR_INVALID, "kf_sync_status: null context");
  KF_CUDA(cudaStreamSynchronize(stream));
  int h[2] = {0, 0};
  KF_CUDA(cudaMemcpy(h, ctx->d_status, sizeof(h), cudaMemcpyDeviceToHost));
  KF_CUDA(cudaMemset(ctx->d_status, 0, sizeof(h)));
  if (info) *info = h[1];
  if (h[0] == 0) return KF_OK;
  const char* what = h[0] == KF_ERR_NOT_SPD ? "Cholesky pivot <= 0 (factor not positive definite)"
                     : h[0] == KF_ERR_NO_CONVERGENCE ? "Jacobi did not converge within max_sweeps"
                     : h[0] == KF_ERR_TIMEOUT ? "a device-side wait timed out"
                                              : "device error";
  return fail(kf_status(h[0]), std::string("device status: ") + what + " (info " + std::to_string(h[1]) + ")");
}

// ----------------------------------------------------------------------- (1)
size_t kfac_accumulate_workspace_size(kf_dtype dtype, kf_quant quant, int64_t d) {
  const int64_t dp = round_up(d > 0 ? d : 1, 8);
  if (dtype == KF_BF16 && quant == KF_QUANT_NONE) return 0;
  if (quant == KF_QUANT_INT8_TOKEN) return size_t(QAW_CHUNK) * dp * 2 + 256;
  return size_t(2) * ACC_CHUNK * dp * 2 + 512;  // float32: hi and lo planes
}

kf_status kfac_accumulate(kf_ctx* ctx, const void* act, kf_dtype dtype, int64_t n_tokens, int64_t d, int64_t ld,
                          kf_quant quant, float* cov_sum, int64_t ldc, void* workspace, size_t workspace_bytes,
                          kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "kfac_accumulate: null context"));
  KF_TRY(need(dtype == KF_BF16 || dtype == KF_F32, "kfac_accumulate: dtype"));
  KF_TRY(need(quant == KF_QUANT_NONE || quant == KF_QUANT_INT8_TOKEN, "kfac_accumulate: quant"));
  KF_TRY(need(n_tokens >= 0 && d > 0 && ld >= d && ldc >= d, "kfac_accumulate: sizes"));
  if (n_tokens == 0) return KF_OK;
  KF_TRY(need(act && cov_sum, "kfac_accumulate: null pointer"));
  if (workspace_bytes < kfac_accumulate_workspace_size(dtype, quant, d))
    return fail(KF_ERR_WORKSPACE, "kfac_accumulate: workspace too small");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  TcGemm g{};
  g.M = d; g.N = d; g.D = cov_sum; g.ldd = ldc; g.accumulate = true; g.sched = TC_LOWER; g.krange = KR_FULL;
  g.kchunk = SYRK_KCHUNK;
  if (dtype == KF_BF16 && quant == KF_QUANT_NONE) {
    KF_TRY(need((reinterpret_cast<uintptr_t>(act) & 15) == 0 && (ld * 2) % 16 == 0,
                "kfac_accumulate: bf16 rows need a 16-byte aligned base and ld a multiple of 8"));
    g.K = n_tokens; g.npass = 1;
    g.a[0] = TcOperand{(const __nv_bfloat16*)act, ld, true};
    g.b[0] = g.a[0];
    return tc_gemm(ctx, g, st);
  }
  const int64_t dp = round_up(d, 8);
  const int64_t chunk = quant == KF_QUANT_INT8_TOKEN ? QAW_CHUNK : ACC_CHUNK;
  Carve cv(workspace, workspace_bytes, false);
  __nv_bfloat16* p0 = cv.take<__nv_bfloat16>(size_t(chunk) * dp);
  __nv_bfloat16* p1 = quant == KF_QUANT_NONE ? cv.take<__nv_bfloat16>(size_t(chunk) * dp) : nullptr;
  for (int64_t t0 = 0; t0 < n_tokens; t0 += chunk) {
    const int64_t rows = n_tokens - t0 < chunk ? n_tokens - t0 : chunk;
    const char* src = static_cast<const char*>(act) + size_t(t0) * ld * elem_size(dtype);
    g.K = rows;
    if (quant == KF_QUANT_INT8_TOKEN) {
      KF_TRY(launch_fake_quant(src, dtype, rows, d, ld, p0, st));
      // fake-quant writes rows with leading dimension d; re-pad when d is not a multiple of 8
      if (dp != d) return fail(KF_ERR_INVALID, "kfac_accumulate: quantised rows need d a multiple of 8");
      g.npass = 1;
      g.a[0] = TcOperand{p0, dp, true};
      g.b[0] = g.a[0];
    } else {
      KF_TRY(launch_split_bf16(reinterpret_cast<const float*>(src), rows, d, ld, p0, p1, dp, st));
      g.npass = 3;  // hi*hi + hi*lo + lo*hi
      g.a[0] = TcOperand{p0, dp, true}; g.b[0] = TcOperand{p0, dp, true};
      g.a[1] = TcOperand{p0, dp, true}; g.b[1] = TcOperand{p1, dp, true};
      g.a[2] = TcOperand{p1, dp, true}; g.b[2] = TcOperand{p0, dp, true};
    }
    KF_TRY(tc_gemm(ctx, g, st));
  }
  return KF_OK;
}

kf_status fake_quant_rows(kf_ctx* ctx, const void* in, kf_dtype dtype, int64_t n_tokens, int64_t d, int64_t ld,
                          void* out, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "fake_quant_rows: null context"));
  KF_TRY(need(dtype == KF_BF16 || dtype == KF_F32, "fake_quant_rows: dtype"));
  KF_TRY(need(n_tokens >= 0 && d > 0 && ld >= d, "fake_quant_rows: sizes"));
  KF_TRY(need(n_tokens <= 0x7fffffff, "fake_quant_rows: at most 2^31 - 1 rows per call"));
  if (n_tokens == 0) return KF_OK;
  KF_TRY(need(in && out, "fake_quant_rows: null pointer"));
  return launch_fake_quant(in, dtype, n_tokens, d, ld, static_cast<__nv_bfloat16*>(out),
                           reinterpret_cast<cudaStream_t>(stream));
}

kf_status kf_finalize_covariance(kf_ctx* ctx, float* cov, int64_t ldc, int64_t d, int64_t n_tokens, float lambda,
                                 kf_stream_t stream) {
  KF_TRY(need(ctx && cov, "kf_finalize_covariance: null pointer"));
  KF_TRY(need(d > 0 && ldc >= d && n_tokens > 0 && lambda >= 0.f, "kf_finalize_covariance: sizes"));
  static std::atomic<unsigned> slot{0};
  float* scratch =
      reinterpret_cast<float*>(reinterpret_cast<char*>(ctx->d_status) + 64) + (slot.fetch_add(1) % FINAL_SLOTS);
  return launch_finalize(cov, ldc, d, n_tokens, lambda, scratch, reinterpret_cast<cudaStream_t>(stream));
}

// --------------------------------------------------------------------- (2)+(3)
namespace {

struct WhitenBufs {
  float *dinv, *T, *tt;
  PlaneBuf w, sg, t, sx;
  int64_t ldT;
  char *cws, *tws;          // Cholesky trailing-update planes; triangular-inverse doubling levels
  size_t cws_bytes, tws_bytes;
};

size_t whiten_carve(Carve& cv, int64_t m, int64_t n, bool w_f32, WhitenBufs& b) {
  const int64_t mx = m > n ? m : n;
  b.dinv = cv.take<float>(size_t(round_up(mx, CHOL_NB)) * CHOL_NB);
  b.ldT = round_up(n, 8);
  b.T = cv.take<float>(size_t(m) * b.ldT);
  b.tt = cv.take<float>(trtri_tmp_floats(mx));
  b.cws_bytes = chol_workspace_bytes(mx);
  b.cws = cv.take<char>(b.cws_bytes);
  b.tws_bytes = trtri_workspace_bytes(m < n ? m : n);
  b.tws = cv.take<char>(b.tws_bytes);
  b.w = take_planes(cv, m, n, w_f32 ? 3 : 1);
  b.sg = take_planes(cv, n, n, 3);
  b.t = take_planes(cv, m, n, 3);
  b.sx = take_planes(cv, m, m, 3);
  return cv.off;
}
}  // namespace

size_t whiten_workspace_size(int64_t m, int64_t n) {
  if (m <= 0 || n <= 0) return 0;
  Carve cv(nullptr, 0, true);
  WhitenBufs b;
  return whiten_carve(cv, m, n, true, b) + 256;
}

kf_status whiten(kf_ctx* ctx, const float* X, int64_t ldx, int64_t m, const float* G, int64_t ldg, int64_t n,
                 const void* W, kf_dtype w_dtype, int64_t ldw, uint32_t flags, float* Sx, int64_t ldsx, float* Sg,
                 int64_t ldsg, float* Sinv, int64_t ldsi, float* Wt, int64_t ldwt, void* workspace,
                 size_t workspace_bytes, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "whiten: null context"));
  KF_TRY(need(m > 0 && n > 0, "whiten: sizes"));
  KF_TRY(need(X && G && W && Sx && Sg && Sinv && Wt, "whiten: null pointer"));
  KF_TRY(need(ldx >= m && ldg >= n && ldw >= n && ldsx >= m && ldsg >= n && ldwt >= n, "whiten: leading dimension"));
  KF_TRY(need(w_dtype == KF_BF16 || w_dtype == KF_F32, "whiten: dtype"));
  const kf_side side = kf_gram_side(m, n);
  const int64_t s = side == KF_SIDE_RIGHT ? n : m;
  KF_TRY(need(ldsi >= s, "whiten: ldsi"));
  Carve cv(workspace, workspace_bytes, false);
  WhitenBufs b;
  whiten_carve(cv, m, n, true, b);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "whiten: workspace too small");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  // S_x = chol_lower(X)^T  (and S_x^-1 for the left Gram side)
  if (!(flags & KF_REUSE_SX)) {
    KF_TRY(launch_copy(X, ldx, Sx, ldsx, m, m, false, st));
    KF_TRY(cholesky_lower(ctx, Sx, ldsx, m, b.dinv, b.cws, b.cws_bytes, st));
    if (side == KF_SIDE_LEFT && !(flags & KF_REUSE_SINV)) {
      KF_TRY(trtri_lower(ctx, Sx, ldsx, m, b.dinv, Sinv, ldsi, b.tt, b.tws, b.tws_bytes, st));   // L_x^-1
      KF_TRY(launch_transpose_inplace(Sinv, ldsi, m, st));                   // S_x^-1 = L_x^-T
    }
    KF_TRY(launch_transpose_inplace(Sx, ldsx, m, st));                       // S_x = L_x^T
  }
  // S_g = chol_lower(G)  (and S_g^-1 for the right Gram side)
  if (!(flags & KF_REUSE_SG)) {
    KF_TRY(launch_copy(G, ldg, Sg, ldsg, n, n, false, st));
    KF_TRY(cholesky_lower(ctx, Sg, ldsg, n, b.dinv, b.cws, b.cws_bytes, st));
    if (side == KF_SIDE_RIGHT && !(flags & KF_REUSE_SINV)) {
      KF_TRY(trtri_lower(ctx, Sg, ldsg, n, b.dinv, Sinv, ldsi, b.tt, b.tws, b.tws_bytes, st));
    }
  }
  // Tensor cores, float32 operands as three bfloat16 planes (float32-accurate products):
  // T = W S_g (S_g lower, so output column j needs k >= j), then W~ = S_x T (S_x upper,
  // output row i needs k >= i).
  Planes pw, psg, pt, psx;
  KF_TRY(as_planes(W, w_dtype, ldw, m, n, b.w, &pw, st));
  if (flags & KF_REUSE_SG_PLANES) {
    psg = Planes{{b.sg.p[0], b.sg.p[1], b.sg.p[2]}, b.sg.ld, 3};
  } else {
    KF_TRY(split_f32(Sg, ldsg, n, n, b.sg, &psg, st));
  }
  KF_TRY(tc_product(ctx, m, n, n, pw, false, psg, true, KR_GE_COL, b.T, b.ldT, st));
  KF_TRY(split_f32(b.T, b.ldT, m, n, b.t, &pt, st));
  if (flags & KF_REUSE_SX_PLANES) {
    psx = Planes{{b.sx.p[0], b.sx.p[1], b.sx.p[2]}, b.sx.ld, 3};
  } else {
    KF_TRY(split_f32(Sx, ldsx, m, m, b.sx, &psx, st));
  }
  return tc_product(ctx, m, n, m, psx, false, pt, true, KR_GE_ROW, Wt, ldwt, st);
}

// --------------------------------------------------------- batched factorisation
namespace {
struct FactorBufs {
  float *dinv, *tt;
  char *cws, *tws;
  size_t cws_bytes, tws_bytes;
};
size_t factor_carve(Carve& cv, int32_t n_jobs, const kf_factor_job* jobs, std::vector<FactorBufs>* out) {
  for (int32_t j = 0; j < n_jobs; ++j) {
    const int64_t n = jobs[j].n > 0 ? jobs[j].n : 1;
    FactorBufs b;
    b.dinv = cv.take<float>(size_t(round_up(n, CHOL_NB)) * CHOL_NB);
    b.cws_bytes = chol_workspace_bytes(n);
    b.cws = cv.take<char>(b.cws_bytes);
    const bool inv = jobs[j].Sinv != nullptr;
    b.tt = inv ? cv.take<float>(trtri_tmp_floats(n)) : nullptr;
    b.tws_bytes = inv ? trtri_workspace_bytes(n) : 0;
    b.tws = inv ? cv.take<char>(b.tws_bytes) : nullptr;
    if (out) out->push_back(b);
  }
  return cv.off;
}

kf_status ensure_streams(kf_ctx* ctx) {
  for (int i = 0; i < kf_ctx::NSTREAMS; ++i)
    if (!ctx->streams[i]) KF_CUDA(cudaStreamCreateWithFlags(&ctx->streams[i], cudaStreamNonBlocking));
  for (int i = 0; i <= kf_ctx::NSTREAMS; ++i)
    if (!ctx->stream_ev[i]) KF_CUDA(cudaEventCreateWithFlags(&ctx->stream_ev[i], cudaEventDisableTiming));
  return KF_OK;
}
}  // namespace

size_t factor_covariances_workspace_size(int32_t n_jobs, const kf_factor_job* jobs) {
  if (n_jobs <= 0 || !jobs) return 0;
  Carve cv(nullptr, 0, true);
  return factor_carve(cv, n_jobs, jobs, nullptr) + 256;
}

kf_status factor_covariances(kf_ctx* ctx, int32_t n_jobs, const kf_factor_job* jobs, void* workspace,
                             size_t workspace_bytes, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "factor_covariances: null context"));
  if (n_jobs == 0) return KF_OK;
  KF_TRY(need(n_jobs > 0 && jobs, "factor_covariances: jobs"));
  for (int32_t j = 0; j < n_jobs; ++j) {
    const kf_factor_job& f = jobs[j];
    KF_TRY(need(f.A && f.S && f.n > 0 && f.lda >= f.n && f.lds >= f.n && (!f.Sinv || f.ldsi >= f.n),
                "factor_covariances: job fields"));
  }
  Carve cv(workspace, workspace_bytes, false);
  std::vector<FactorBufs> bufs;
  factor_carve(cv, n_jobs, jobs, &bufs);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "factor_covariances: workspace too small");
  KF_TRY(ensure_streams(ctx));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int used = n_jobs < kf_ctx::NSTREAMS ? n_jobs : kf_ctx::NSTREAMS;
  // fork: every internal stream starts after the work already queued on the caller's stream
  KF_CUDA(cudaEventRecord(ctx->stream_ev[kf_ctx::NSTREAMS], st));
  for (int i = 0; i < used; ++i) KF_CUDA(cudaStreamWaitEvent(ctx->streams[i], ctx->stream_ev[kf_ctx::NSTREAMS], 0));
  kf_status rc = KF_OK;
  for (int32_t j = 0; j < n_jobs && rc == KF_OK; ++j) {
    const kf_factor_job& f = jobs[j];
    const FactorBufs& b = bufs[size_t(j)];
    cudaStream_t sj = ctx->streams[j % kf_ctx::NSTREAMS];
    rc = launch_copy(f.A, f.lda, f.S, f.lds, f.n, f.n, false, sj);
    if (rc == KF_OK) rc = cholesky_lower(ctx, f.S, f.lds, f.n, b.dinv, b.cws, b.cws_bytes, sj);
    if (rc == KF_OK && f.Sinv) rc = trtri_lower(ctx, f.S, f.lds, f.n, b.dinv, f.Sinv, f.ldsi, b.tt, b.tws, b.tws_bytes, sj);
    if (rc == KF_OK && f.upper) {
      rc = launch_transpose_inplace(f.S, f.lds, f.n, sj);
      if (rc == KF_OK && f.Sinv) rc = launch_transpose_inplace(f.Sinv, f.ldsi, f.n, sj);
    }
  }
  // join (also after a failed launch, so that the caller's stream never runs ahead of them)
  for (int i = 0; i < used; ++i) {
    KF_CUDA(cudaEventRecord(ctx->stream_ev[i], ctx->streams[i]));
    KF_CUDA(cudaStreamWaitEvent(st, ctx->stream_ev[i], 0));
  }
  return rc;
}

// ------------------------------------------------------------------------ (4)
size_t whitened_svd_workspace_size(int32_t n_problems, int64_t m_max, int64_t n_max, int64_t s) {
  if (n_problems <= 0 || s <= 0) return 0;
  return svd_workspace(n_problems, m_max, n_max, s);
}

kf_status whitened_svd(kf_ctx* ctx, int32_t n_problems, const kf_svd_problem* problems, float tol,
                       int32_t max_sweeps, void* workspace, size_t workspace_bytes, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "whitened_svd: null context"));
  if (n_problems == 0) return KF_OK;
  KF_TRY(need(n_problems > 0 && problems, "whitened_svd: problems"));
  KF_TRY(need(n_problems <= 65535, "whitened_svd: at most 65535 problems per call"));
  KF_TRY(need(tol > 0.f && max_sweeps > 0, "whitened_svd: tol and max_sweeps must be positive"));
  int64_t s0 = -1, m_max = 0, n_max = 0;
  for (int i = 0; i < n_problems; ++i) {
    const kf_svd_problem& p = problems[i];
    KF_TRY(need(p.Wt && p.sigma && p.vecs && p.m > 0 && p.n > 0 && p.ldw >= p.n, "whitened_svd: problem fields"));
    const int64_t s = p.m < p.n ? p.m : p.n;
    KF_TRY(need(p.ldv >= s, "whitened_svd: ldv"));
    if (s0 < 0) s0 = s;
    KF_TRY(need(s == s0, "whitened_svd: all problems of a call need the same min(m, n)"));
    m_max = p.m > m_max ? p.m : m_max;
    n_max = p.n > n_max ? p.n : n_max;
  }
  if (s0 > 16384) return fail(KF_ERR_UNSUPPORTED, "whitened_svd: min(m, n) > 16384");
  if (workspace_bytes < svd_workspace(n_problems, m_max, n_max, s0))
    return fail(KF_ERR_WORKSPACE, "whitened_svd: workspace too small");
  return svd_run(ctx, n_problems, problems, tol, max_sweeps, workspace, workspace_bytes,
                 reinterpret_cast<cudaStream_t>(stream), false);
}

kf_status empirical_fisher_finalize(kf_ctx* ctx, const double* score_sum, int64_t n, int64_t n_tokens, float* keys,
                                    kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "empirical_fisher_finalize: null context"));
  KF_TRY(need(n >= 0 && n_tokens > 0, "empirical_fisher_finalize: sizes"));
  if (n == 0) return KF_OK;
  KF_TRY(need(score_sum && keys, "empirical_fisher_finalize: null pointer"));
  return launch_fisher_finalize(score_sum, n, n_tokens, keys, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------- index plumbing
kf_status gather_rows_cols(kf_ctx* ctx, const void* src, kf_dtype dtype, int64_t lds, int64_t src_rows,
                           int64_t src_cols, const int64_t* row_idx, int64_t rows, const int64_t* col_idx, int64_t cols,
                           void* dst, int64_t ldd, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "gather_rows_cols: null context"));
  KF_TRY(need(dtype == KF_BF16 || dtype == KF_F32, "gather_rows_cols: dtype"));
  KF_TRY(need(rows >= 0 && cols >= 0 && src_rows >= 0 && src_cols >= 0, "gather_rows_cols: sizes"));
  if (rows == 0 || cols == 0) return KF_OK;
  KF_TRY(need(src && dst, "gather_rows_cols: null pointer"));
  KF_TRY(need(lds >= src_cols && ldd >= cols, "gather_rows_cols: leading dimension"));
  KF_TRY(need(row_idx || rows <= src_rows, "gather_rows_cols: rows"));
  KF_TRY(need(col_idx || cols <= src_cols, "gather_rows_cols: cols"));
  return launch_gather2d(src, dtype, lds, src_rows, src_cols, row_idx, rows, col_idx, cols, dst, ldd, ctx->d_status,
                         reinterpret_cast<cudaStream_t>(stream));
}

kf_status compact_mask(kf_ctx* ctx, const uint8_t* mask, int64_t n, int32_t want, int64_t* idx, int64_t* count,
                       kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "compact_mask: null context"));
  KF_TRY(need(n >= 0 && count, "compact_mask: sizes"));
  KF_TRY(need(n == 0 || (mask && idx), "compact_mask: null pointer"));
  return launch_compact_mask(mask, n, want, idx, count, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------- LASER hybrid FFN channel errors
namespace {
struct ChanBufs {
  float *D, *E;
  int64_t ld;
  PlaneBuf u, v, x, d;
};
size_t chan_carve(Carve& cv, int64_t m, int64_t n, int32_t r, ChanBufs& b) {
  b.ld = round_up(n, 8);
  b.D = cv.take<float>(size_t(m) * b.ld);
  b.E = cv.take<float>(size_t(m) * b.ld);
  b.u = take_planes(cv, m, r > 0 ? r : 1, 3);
  b.v = take_planes(cv, r > 0 ? r : 1, n, 3);
  b.x = take_planes(cv, m, m, 3);
  b.d = take_planes(cv, m, n, 3);
  return cv.off;
}
}  // namespace

size_t channel_errors_workspace_size(int64_t m, int64_t n, int32_t r) {
  if (m <= 0 || n <= 0 || r < 0) return 0;
  Carve cv(nullptr, 0, true);
  ChanBufs b;
  return chan_carve(cv, m, n, r, b) + 256;
}

kf_status channel_errors(kf_ctx* ctx, const void* W, kf_dtype w_dtype, int64_t ldw, int64_t m, int64_t n,
                         const float* U, int64_t ldu, const float* V, int64_t ldv, int32_t r, const float* X,
                         int64_t ldx, double* err_sum, float* keys, void* workspace, size_t workspace_bytes,
                         kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "channel_errors: null context"));
  KF_TRY(need(m > 0 && n > 0 && r >= 0, "channel_errors: sizes"));
  KF_TRY(need(W && X && err_sum, "channel_errors: null pointer"));
  KF_TRY(need(r == 0 || (U && V), "channel_errors: null factor"));
  KF_TRY(need(ldw >= n && ldx >= m && (r == 0 || (ldu >= r && ldv >= n)), "channel_errors: leading dimension"));
  KF_TRY(need(w_dtype == KF_BF16 || w_dtype == KF_F32, "channel_errors: dtype"));
  Carve cv(workspace, workspace_bytes, false);
  ChanBufs b;
  chan_carve(cv, m, n, r, b);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "channel_errors: workspace too small");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // D = W - U V (U, V as three bfloat16 planes: float32-level products), E = X D, and the
  // column dots e_j = d_j . (X d_j) in float64.
  if (r > 0) {
    Planes pu, pv;
    KF_TRY(split_f32(U, ldu, m, r, b.u, &pu, st));
    KF_TRY(split_f32(V, ldv, r, n, b.v, &pv, st));
    KF_TRY(tc_product(ctx, m, n, r, pu, false, pv, true, KR_FULL, b.D, b.ld, st));
  } else {
    KF_CUDA(cudaMemsetAsync(b.D, 0, sizeof(float) * size_t(m) * b.ld, st));
  }
  KF_TRY(launch_sub_from(W, w_dtype, ldw, b.D, b.ld, m, n, st));
  Planes px, pd;
  KF_TRY(split_f32(X, ldx, m, m, b.x, &px, st));
  KF_TRY(split_f32(b.D, b.ld, m, n, b.d, &pd, st));
  KF_TRY(tc_product(ctx, m, n, m, px, false, pd, true, KR_FULL, b.E, b.ld, st));
  return launch_coldot(b.D, b.ld, b.E, b.ld, m, n, err_sum, keys, st);
}

// ------------------------------------------------- Swift-SVD activation-only route
namespace {
struct ActCovBufs {
  float* T;
  int64_t ldT;
  PlaneBuf x, w, t;
};
size_t actcov_carve(Carve& cv, int64_t m, int64_t n, ActCovBufs& b) {
  b.ldT = round_up(n, 8);
  b.T = cv.take<float>(size_t(m) * b.ldT);
  b.x = take_planes(cv, m, m, 3);
  b.w = take_planes(cv, m, n, 3);
  b.t = take_planes(cv, m, n, 3);
  return cv.off;
}
}  // namespace

size_t activation_covariance_workspace_size(int64_t m, int64_t n) {
  if (m <= 0 || n <= 0) return 0;
  Carve cv(nullptr, 0, true);
  ActCovBufs b;
  return actcov_carve(cv, m, n, b) + 256;
}

kf_status activation_covariance(kf_ctx* ctx, const float* X, int64_t ldx, int64_t m, const void* W, kf_dtype w_dtype,
                                int64_t ldw, int64_t n, float* C, int64_t ldc, void* workspace,
                                size_t workspace_bytes, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "activation_covariance: null context"));
  KF_TRY(need(m > 0 && n > 0, "activation_covariance: sizes"));
  KF_TRY(need(X && W && C, "activation_covariance: null pointer"));
  KF_TRY(need(ldx >= m && ldw >= n && ldc >= n, "activation_covariance: leading dimension"));
  KF_TRY(need(w_dtype == KF_BF16 || w_dtype == KF_F32, "activation_covariance: dtype"));
  Carve cv(workspace, workspace_bytes, false);
  ActCovBufs b;
  actcov_carve(cv, m, n, b);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "activation_covariance: workspace too small");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // T = X W, then C = W^T T; float32 operands as three bfloat16 planes, W^T read MN-major
  Planes px, pw, pt;
  KF_TRY(split_f32(X, ldx, m, m, b.x, &px, st));
  KF_TRY(as_planes(W, w_dtype, ldw, m, n, b.w, &pw, st));
  KF_TRY(tc_product(ctx, m, n, m, px, false, pw, true, KR_FULL, b.T, b.ldT, st));
  KF_TRY(split_f32(b.T, b.ldT, m, n, b.t, &pt, st));
  return tc_product(ctx, n, n, m, pw, true, pt, true, KR_FULL, C, ldc, st);
}

size_t activation_eig_workspace_size(int32_t n_problems, int64_t n) {
  if (n_problems <= 0 || n <= 0) return 0;
  return svd_workspace(n_problems, n, n, n);
}

kf_status activation_eig(kf_ctx* ctx, int32_t n_problems, const kf_sym_problem* problems, float tol,
                         int32_t max_sweeps, void* workspace, size_t workspace_bytes, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "activation_eig: null context"));
  if (n_problems == 0) return KF_OK;
  KF_TRY(need(n_problems > 0 && problems, "activation_eig: problems"));
  KF_TRY(need(n_problems <= 65535, "activation_eig: at most 65535 problems per call"));
  KF_TRY(need(tol > 0.f && max_sweeps > 0, "activation_eig: tol and max_sweeps must be positive"));
  std::vector<kf_svd_problem> pr(static_cast<size_t>(n_problems));
  const int64_t n0 = problems[0].n;
  for (int i = 0; i < n_problems; ++i) {
    const kf_sym_problem& p = problems[i];
    KF_TRY(need(p.C && p.sigma && p.vecs && p.n > 0 && p.ldc >= p.n && p.ldv >= p.n,
                "activation_eig: problem fields"));
    KF_TRY(need(p.n == n0, "activation_eig: all problems of a call need the same n"));
    pr[size_t(i)] = kf_svd_problem{p.C, p.n, p.n, p.ldc, p.sigma, p.vecs, p.ldv, p.sweeps};
  }
  if (n0 > 16384) return fail(KF_ERR_UNSUPPORTED, "activation_eig: n > 16384");
  if (workspace_bytes < svd_workspace(n_problems, n0, n0, n0))
    return fail(KF_ERR_WORKSPACE, "activation_eig: workspace too small");
  return svd_run(ctx, n_problems, pr.data(), tol, max_sweeps, workspace, workspace_bytes,
                 reinterpret_cast<cudaStream_t>(stream), true);
}

namespace {
struct ActFacBufs {
  PlaneBuf w, v;
};
size_t actfac_carve(Carve& cv, int64_t m, int64_t n, int32_t r, ActFacBufs& b) {
  b.w = take_planes(cv, m, n, 2);
  b.v = take_planes(cv, n, r, 2);
  return cv.off;
}
}  // namespace

size_t activation_factors_workspace_size(int64_t m, int64_t n, int32_t r) {
  if (m <= 0 || n <= 0 || r <= 0) return 0;
  Carve cv(nullptr, 0, true);
  ActFacBufs b;
  return actfac_carve(cv, m, n, r, b) + 256;
}

kf_status activation_factors(kf_ctx* ctx, const void* W, kf_dtype w_dtype, int64_t ldw, int64_t m, int64_t n,
                             const float* vecs, int64_t ldv, int32_t r, float* U, int64_t ldu, float* V,
                             int64_t ldvo, void* workspace, size_t workspace_bytes, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "activation_factors: null context"));
  KF_TRY(need(m > 0 && n > 0 && r >= 0 && r <= n, "activation_factors: sizes"));
  if (r == 0) return KF_OK;
  KF_TRY(need(W && vecs && U && V, "activation_factors: null pointer"));
  KF_TRY(need(ldw >= n && ldv >= n && ldu >= r && ldvo >= n, "activation_factors: leading dimension"));
  KF_TRY(need(w_dtype == KF_BF16 || w_dtype == KF_F32, "activation_factors: dtype"));
  Carve cv(workspace, workspace_bytes, false);
  ActFacBufs b;
  actfac_carve(cv, m, n, r, b);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "activation_factors: workspace too small");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // U = W V_r (V_r: the first r columns of vecs, n x r, read MN-major), V = V_r^T
  Planes pw, pv;
  KF_TRY(as_planes(W, w_dtype, ldw, m, n, b.w, &pw, st));
  KF_TRY(split_f32(vecs, ldv, n, r, b.v, &pv, st));
  KF_TRY(tc_product(ctx, m, r, n, pw, false, pv, true, KR_FULL, U, ldu, st));
  return launch_copy(vecs, ldv, V, ldvo, r, n, true, st);
}

kf_status kf_svd_profile_enable(kf_ctx* ctx, int enable) {
  KF_TRY(need(ctx != nullptr, "kf_svd_profile_enable: null context"));
  ctx->prof_enabled = enable != 0;
  return KF_OK;
}

kf_status kf_svd_profile_read(kf_ctx* ctx, kf_svd_profile* out) {
  KF_TRY(need(ctx && out, "kf_svd_profile_read: null pointer"));
  return svd_profile_read(ctx, out);
}

// ----------------------------------------------------------------------- (5a)
size_t score_and_allocate_workspace_size(int64_t n_components, int32_t n_units) {
  // room for the per-unit energies too, so one size serves every mode
  return alloc_workspace(n_components > 0 ? n_components : 1, n_units > 0 ? n_units : 0);
}

namespace {
kf_status allocate_common(kf_ctx* ctx, const char* who, const float* sigma, const int64_t* seg_offset,
                          const int64_t* cost, int32_t n_units, int64_t n_components, int64_t budget,
                          kf_alloc_mode mode, const int32_t* fixed_rank, const float* weight, int32_t* ranks,
                          float* cut, int64_t* used, void* workspace, size_t workspace_bytes, kf_stream_t stream) {
  const std::string w(who);
  KF_TRY(need(ctx != nullptr, (w + ": null context").c_str()));
  KF_TRY(need(n_units > 0 && n_components >= 0, (w + ": sizes").c_str()));
  KF_TRY(need(n_components < (int64_t(1) << 32), (w + ": at most 2^32 - 1 components").c_str()));
  KF_TRY(need(seg_offset && cost && ranks, (w + ": null pointer").c_str()));
  KF_TRY(need(mode == KF_KEY_HALF_SIGMA2 || mode == KF_KEY_PER_PARAM || mode == KF_FIXED_RANK ||
                  mode == KF_KEY_ENERGY_RATIO,
              (w + ": mode").c_str()));
  if (mode == KF_FIXED_RANK) KF_TRY(need(fixed_rank != nullptr, (w + ": fixed_rank is null").c_str()));
  else KF_TRY(need(sigma != nullptr || n_components == 0, (w + ": sigma is null").c_str()));
  const int64_t n_energy = mode == KF_KEY_ENERGY_RATIO ? n_units : 0;
  if (mode != KF_FIXED_RANK && workspace_bytes < alloc_workspace(n_components > 0 ? n_components : 1, n_energy))
    return fail(KF_ERR_WORKSPACE, w + ": workspace too small");
  if (mode != KF_FIXED_RANK && n_components == 0) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    KF_CUDA(cudaMemsetAsync(ranks, 0, sizeof(int32_t) * size_t(n_units), st));
    if (used) KF_CUDA(cudaMemsetAsync(used, 0, sizeof(int64_t), st));
    if (cut) KF_CUDA(cudaMemsetAsync(cut, 0xFF, 2 * sizeof(float), st));  // NaN
    return KF_OK;
  }
  return alloc_run(ctx, sigma, seg_offset, cost, n_units, n_components, budget, mode, fixed_rank, weight, ranks, cut,
                   used, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr, 0.0);
}
}  // namespace

kf_status score_and_allocate(kf_ctx* ctx, const float* sigma, const int64_t* seg_offset, const int64_t* cost,
                             int32_t n_units, int64_t n_components, int64_t budget, kf_alloc_mode mode,
                             const int32_t* fixed_rank, int32_t* ranks, float* cut, int64_t* used, void* workspace,
                             size_t workspace_bytes, kf_stream_t stream) {
  return allocate_common(ctx, "score_and_allocate", sigma, seg_offset, cost, n_units, n_components, budget, mode,
                         fixed_rank, nullptr, ranks, cut, used, workspace, workspace_bytes, stream);
}

kf_status score_and_allocate_weighted(kf_ctx* ctx, const float* sigma, const int64_t* seg_offset,
                                      const int64_t* cost, int32_t n_units, int64_t n_components, int64_t budget,
                                      kf_alloc_mode mode, const float* unit_weight, int32_t* ranks, float* cut,
                                      int64_t* used, void* workspace, size_t workspace_bytes, kf_stream_t stream) {
  if (mode == KF_FIXED_RANK) return fail(KF_ERR_INVALID, "score_and_allocate_weighted: KF_FIXED_RANK has no scores");
  return allocate_common(ctx, "score_and_allocate_weighted", sigma, seg_offset, cost, n_units, n_components, budget,
                         mode, nullptr, unit_weight, ranks, cut, used, workspace, workspace_bytes, stream);
}

kf_status score_and_allocate_keys(kf_ctx* ctx, const float* keys, const int64_t* seg_offset, const int64_t* cost,
                                  int32_t n_units, int64_t n_components, int64_t budget, int32_t* ranks,
                                  uint8_t* keep, float* cut, int64_t* used, void* workspace, size_t workspace_bytes,
                                  kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "score_and_allocate_keys: null context"));
  KF_TRY(need(n_units > 0 && n_components >= 0, "score_and_allocate_keys: sizes"));
  KF_TRY(need(n_components < (int64_t(1) << 32), "score_and_allocate_keys: at most 2^32 - 1 components"));
  KF_TRY(need(seg_offset && cost && ranks && (keys != nullptr || n_components == 0),
              "score_and_allocate_keys: null pointer"));
  if (workspace_bytes < alloc_workspace(n_components > 0 ? n_components : 1, 0))
    return fail(KF_ERR_WORKSPACE, "score_and_allocate_keys: workspace too small");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n_components == 0) {
    KF_CUDA(cudaMemsetAsync(ranks, 0, sizeof(int32_t) * size_t(n_units), st));
    if (used) KF_CUDA(cudaMemsetAsync(used, 0, sizeof(int64_t), st));
    if (cut) KF_CUDA(cudaMemsetAsync(cut, 0xFF, 2 * sizeof(float), st));
    return KF_OK;
  }
  return alloc_run(ctx, keys, seg_offset, cost, n_units, n_components, budget,
                   static_cast<kf_alloc_mode>(alloc_mode_given_keys()), nullptr, nullptr, ranks, cut, used, workspace,
                   workspace_bytes, st, keep, 0.0);
}

kf_status score_and_allocate_hybrid(kf_ctx* ctx, const float* sigma, const int64_t* seg_offset, const int64_t* cost,
                                    int32_t n_units, int64_t n_components, int64_t budget, const float* importance,
                                    double alpha, int32_t* ranks, float* cut, int64_t* used, void* workspace,
                                    size_t workspace_bytes, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "score_and_allocate_hybrid: null context"));
  KF_TRY(need(n_units > 0 && n_components >= 0, "score_and_allocate_hybrid: sizes"));
  KF_TRY(need(n_components < (int64_t(1) << 32), "score_and_allocate_hybrid: at most 2^32 - 1 components"));
  KF_TRY(need(alpha >= 0.0 && alpha <= 1.0, "score_and_allocate_hybrid: alpha must lie in [0, 1]"));
  KF_TRY(need(seg_offset && cost && ranks && (sigma != nullptr || n_components == 0),
              "score_and_allocate_hybrid: null pointer"));
  if (workspace_bytes < alloc_workspace(n_components > 0 ? n_components : 1, 0))
    return fail(KF_ERR_WORKSPACE, "score_and_allocate_hybrid: workspace too small");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n_components == 0) {
    KF_CUDA(cudaMemsetAsync(ranks, 0, sizeof(int32_t) * size_t(n_units), st));
    if (used) KF_CUDA(cudaMemsetAsync(used, 0, sizeof(int64_t), st));
    if (cut) KF_CUDA(cudaMemsetAsync(cut, 0xFF, 2 * sizeof(float), st));
    return KF_OK;
  }
  return alloc_run(ctx, sigma, seg_offset, cost, n_units, n_components, budget,
                   static_cast<kf_alloc_mode>(alloc_mode_swift_hybrid()), nullptr, importance, ranks, cut, used,
                   workspace, workspace_bytes, st, nullptr, alpha);
}

int64_t kf_hybrid_ffn_budget(int64_t budget, int32_t n, const int64_t* d_model, const int64_t* n_dense,
                             int64_t* dense_cost) {
  if (n < 0 || (n > 0 && (!d_model || !n_dense))) {
    fail(KF_ERR_INVALID, "kf_hybrid_ffn_budget: sizes or null pointer");
    return -1;
  }
  int64_t cost = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (d_model[i] < 0 || n_dense[i] < 0) {
      fail(KF_ERR_INVALID, "kf_hybrid_ffn_budget: negative entry");
      return -1;
    }
    cost += d_model[i] * n_dense[i];
  }
  if (dense_cost) *dense_cost = cost;
  const int64_t left = budget - cost;
  return left > 0 ? left : 0;
}

// ----------------------------------------------------------------------- (5b)
namespace {
struct UnwhitenBufs {
  float *q0, *q1, *gm, *li, *dinv, *tt, *P;
  int64_t ldP;
  PlaneBuf c, w, sg, si, p;
  PlaneBuf q3, l3;  // CholeskyQR2 operands as three planes
  char *cws, *tws;
  size_t cws_bytes, tws_bytes;
};

size_t unwhiten_carve(Carve& cv, int64_t m, int64_t n, int64_t r, UnwhitenBufs& b) {
  const int64_t s = m < n ? m : n, mx = m > n ? m : n;
  b.q0 = cv.take<float>(size_t(s) * r);
  b.q1 = cv.take<float>(size_t(s) * r);
  b.gm = cv.take<float>(size_t(r) * r);
  b.li = cv.take<float>(size_t(r) * r);
  b.dinv = cv.take<float>(size_t(round_up(r, CHOL_NB)) * CHOL_NB);
  b.tt = cv.take<float>(trtri_tmp_floats(r));
  b.cws_bytes = chol_workspace_bytes(r);
  b.cws = cv.take<char>(b.cws_bytes);
  b.tws_bytes = trtri_workspace_bytes(r);
  b.tws = cv.take<char>(b.tws_bytes);
  b.ldP = round_up(mx, 8);
  b.P = cv.take<float>(size_t(mx) * b.ldP);   // n x r (right side) or r x m (left side)
  b.c = take_planes(cv, s, r, 2);
  b.w = take_planes(cv, m, n, 2);
  b.sg = take_planes(cv, mx, mx, 2);          // S_g (right) or S_x (left)
  b.si = take_planes(cv, s, s, 2);            // the Gram-side inverse
  b.p = take_planes(cv, mx, mx, 2);           // P as an operand (n x r or r x m)
  b.q3 = take_planes(cv, s, r, 3);
  b.l3 = take_planes(cv, r, r, 3);
  return cv.off;
}
}  // namespace

size_t unwhiten_workspace_size(int64_t m, int64_t n, int32_t r) {
  if (m <= 0 || n <= 0 || r <= 0) return 0;
  Carve cv(nullptr, 0, true);
  UnwhitenBufs b;
  return unwhiten_carve(cv, m, n, r, b) + 256;
}

kf_status unwhiten(kf_ctx* ctx, const void* W, kf_dtype w_dtype, int64_t ldw, int64_t m, int64_t n, const float* Sx,
                   int64_t ldsx, const float* Sg, int64_t ldsg, const float* Sinv, int64_t ldsi, const float* sigma,
                   const float* vecs, int64_t ldv, int32_t r, float* U, int64_t ldu, float* V, int64_t ldvo,
                   void* workspace, size_t workspace_bytes, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "unwhiten: null context"));
  KF_TRY(need(m > 0 && n > 0, "unwhiten: sizes"));
  const int64_t s = m < n ? m : n;
  KF_TRY(need(r >= 0 && r <= s, "unwhiten: r must be in [0, min(m, n)]"));
  if (r == 0) return KF_OK;
  // Only the Gram-side factor is read (S_g for KF_SIDE_RIGHT, S_x for KF_SIDE_LEFT).
  const bool right_side = kf_gram_side(m, n) == KF_SIDE_RIGHT;
  KF_TRY(need(W && Sinv && sigma && vecs && U && V && (right_side ? Sg != nullptr : Sx != nullptr),
              "unwhiten: null pointer"));
  KF_TRY(need(ldw >= n && (right_side ? ldsg >= n : ldsx >= m) && ldsi >= s && ldv >= s && ldu >= r && ldvo >= n,
              "unwhiten: leading dimension"));
  KF_TRY(need(w_dtype == KF_BF16 || w_dtype == KF_F32, "unwhiten: dtype"));
  Carve cv(workspace, workspace_bytes, false);
  UnwhitenBufs b;
  unwhiten_carve(cv, m, n, r, b);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "unwhiten: workspace too small");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  // CholeskyQR2 of the r leading Gram-side vectors: twice Q <- Q L^-T with L L^T = Q^T Q.
  // The Gram of nearly orthonormal columns needs float32 accuracy: both products run on the
  // tensor cores with three-plane operands (all six cross terms).
  KF_TRY(launch_copy(vecs, ldv, b.q0, r, s, r, false, st));
  float* cur = b.q0;
  float* nxt = b.q1;
  for (int it = 0; it < 2; ++it) {
    Planes pq, pl;
    KF_TRY(split_f32(cur, r, s, r, b.q3, &pq, st));
    ProductOpts lo;
    lo.lower = true;
    KF_TRY(tc_product(ctx, r, r, s, pq, true, pq, true, KR_FULL, b.gm, r, st, lo));  // Q^T Q, lower
    KF_TRY(cholesky_lower(ctx, b.gm, r, r, b.dinv, b.cws, b.cws_bytes, st));
    KF_TRY(trtri_lower(ctx, b.gm, r, r, b.dinv, b.li, r, b.tt, b.tws, b.tws_bytes, st));
    KF_TRY(split_f32(b.li, r, r, r, b.l3, &pl, st));
    KF_TRY(tc_product(ctx, s, r, r, pq, false, pl, false, KR_LE_COL, nxt, r, st));   // (L^-1)^T is upper
    float* tmp = cur; cur = nxt; nxt = tmp;
  }
  // The remaining products run on the tensor cores with float32 operands split hi + lo.
  Planes pc, pw, pf, pi, pp;
  KF_TRY(split_f32(cur, r, s, r, b.c, &pc, st));
  KF_TRY(as_planes(W, w_dtype, ldw, m, n, b.w, &pw, st));
  if (kf_gram_side(m, n) == KF_SIDE_RIGHT) {
    // P = S_g V~_r (S_g lower: row i needs k <= i);  U = W P;  V = V~_r^T S_g^-1.
    KF_TRY(split_f32(Sg, ldsg, n, n, b.sg, &pf, st));
    KF_TRY(tc_product(ctx, n, r, n, pf, false, pc, true, KR_LE_ROW, b.P, b.ldP, st));
    KF_TRY(split_f32(b.P, b.ldP, n, r, b.p, &pp, st));
    KF_TRY(tc_product(ctx, m, r, n, pw, false, pp, true, KR_FULL, U, ldu, st));
    KF_TRY(split_f32(Sinv, ldsi, n, n, b.si, &pi, st));
    return tc_product(ctx, r, n, n, pc, true, pi, true, KR_GE_COL, V, ldvo, st);  // S_g^-1 lower
  }
  // Left side: U = S_x^-1 U~_r Sigma_r;  V = Sigma_r^-1 (U~_r^T S_x) W.
  KF_TRY(split_f32(Sinv, ldsi, m, m, b.si, &pi, st));
  KF_TRY(tc_product(ctx, m, r, m, pi, false, pc, true, KR_GE_ROW, U, ldu, st));  // S_x^-1 upper
  KF_TRY(launch_scale_cols(U, ldu, m, r, sigma, false, st));
  KF_TRY(split_f32(Sx, ldsx, m, m, b.sg, &pf, st));
  KF_TRY(tc_product(ctx, r, m, m, pc, true, pf, true, KR_LE_COL, b.P, b.ldP, st));  // S_x upper: k <= j
  KF_TRY(split_f32(b.P, b.ldP, r, m, b.p, &pp, st));
  KF_TRY(tc_product(ctx, r, n, m, pp, false, pw, true, KR_FULL, V, ldvo, st));
  return launch_scale_rows(V, ldvo, r, n, sigma, true, st);
}

// ------------------------------------------------------- empirical-Fisher scores
namespace {
constexpr int64_t FISHER_CHUNK = 4096;  // tokens per projection chunk

struct FisherBufs {
  PlaneBuf a, g, u, v;
  float *P, *Q;
  int64_t ldPQ;
};

size_t fisher_carve(Carve& cv, int64_t m, int64_t n, int64_t r, FisherBufs& b) {
  b.a = take_planes(cv, FISHER_CHUNK, m, 2);
  b.g = take_planes(cv, FISHER_CHUNK, n, 2);
  b.u = take_planes(cv, m, r, 2);
  b.v = take_planes(cv, r, n, 2);
  b.ldPQ = round_up(r, 4);
  b.P = cv.take<float>(size_t(FISHER_CHUNK) * b.ldPQ);
  b.Q = cv.take<float>(size_t(FISHER_CHUNK) * b.ldPQ);
  return cv.off;
}
}  // namespace

size_t empirical_fisher_workspace_size(int64_t m, int64_t n, int32_t r) {
  if (m <= 0 || n <= 0 || r <= 0) return 0;
  Carve cv(nullptr, 0, true);
  FisherBufs b;
  return fisher_carve(cv, m, n, r, b) + 256;
}

kf_status empirical_fisher_accumulate(kf_ctx* ctx, const void* act, kf_dtype act_dtype, int64_t lda,
                                      const void* grad, kf_dtype grad_dtype, int64_t ldg, int64_t n_tokens,
                                      int64_t m, int64_t n, const float* U, int64_t ldu, const float* V,
                                      int64_t ldv, int32_t r, double* score_sum, void* workspace,
                                      size_t workspace_bytes, kf_stream_t stream) {
  KF_TRY(need(ctx != nullptr, "empirical_fisher_accumulate: null context"));
  KF_TRY(need(n_tokens >= 0 && m > 0 && n > 0 && r >= 0, "empirical_fisher_accumulate: sizes"));
  if (n_tokens == 0 || r == 0) return KF_OK;
  KF_TRY(need(act && grad && U && V && score_sum, "empirical_fisher_accumulate: null pointer"));
  KF_TRY(need(lda >= m && ldg >= n && ldu >= r && ldv >= n, "empirical_fisher_accumulate: leading dimension"));
  KF_TRY(need((act_dtype == KF_BF16 || act_dtype == KF_F32) && (grad_dtype == KF_BF16 || grad_dtype == KF_F32),
              "empirical_fisher_accumulate: dtype"));
  Carve cv(workspace, workspace_bytes, false);
  FisherBufs b;
  fisher_carve(cv, m, n, r, b);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "empirical_fisher_accumulate: workspace too small");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Planes pu, pv, pa, pg;
  KF_TRY(split_f32(U, ldu, m, r, b.u, &pu, st));
  KF_TRY(split_f32(V, ldv, r, n, b.v, &pv, st));
  const size_t ea = act_dtype == KF_BF16 ? 2 : 4, eg = grad_dtype == KF_BF16 ? 2 : 4;
  for (int64_t t0 = 0; t0 < n_tokens; t0 += FISHER_CHUNK) {
    const int64_t rows = n_tokens - t0 < FISHER_CHUNK ? n_tokens - t0 : FISHER_CHUNK;
    const void* ac = static_cast<const char*>(act) + size_t(t0) * lda * ea;
    const void* gc = static_cast<const char*>(grad) + size_t(t0) * ldg * eg;
    KF_TRY(as_planes(ac, act_dtype, lda, rows, m, b.a, &pa, st));
    KF_TRY(as_planes(gc, grad_dtype, ldg, rows, n, b.g, &pg, st));
    // P = A_c U (a_t . u_i), Q = Gr_c V^T (g_t . v_i); V is r x n, i.e. V^T stored K-major
    KF_TRY(tc_product(ctx, rows, r, m, pa, false, pu, true, KR_FULL, b.P, b.ldPQ, st));
    KF_TRY(tc_product(ctx, rows, r, n, pg, false, pv, false, KR_FULL, b.Q, b.ldPQ, st));
    KF_TRY(launch_fisher_reduce(b.P, b.ldPQ, b.Q, b.ldPQ, rows, r, score_sum, st));
  }
  return KF_OK;
}

}  // extern "C"
