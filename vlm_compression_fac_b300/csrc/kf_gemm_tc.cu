// Tensor-core GEMM / SYRK engine for sm_103a: tcgen05.mma (kind::f16, bfloat16 operands,
// float32 accumulation in tensor memory), operands staged by TMA (cp.async.bulk.tensor,
// 128-byte swizzle) through a 4-stage mbarrier pipeline, accumulators read back with
// tcgen05.ld.  One 128 x 256 output tile per CTA of 10 warps:
//   warp 0 lane 0  TMA producer           warp 1 lane 0  MMA issuer (single thread)
//   warp 0         TMEM alloc / dealloc    warps 2-9      epilogue (TMEM lanes 32(w%4)..+31,
//                                                         128 of the 256 columns each)
// The K range is cut into chunks (at most `kcb` k-blocks of 64 each): a chunk accumulates
// in one of two TMEM accumulators while the epilogue warps add the previous chunk into a
// float32 running sum held in registers (IEEE adds).  Bounding the length of each in-tensor-
// core accumulation keeps long sums (a covariance over 10^5 tokens) float32-accurate.
// Several "passes" (A_p, B_p) accumulate into the same tile, which is how float32 operands
// enter as bfloat16 hi/lo splits.  TC_LOWER visits only the tiles that touch the lower
// triangle (the covariance SYRK X += A^T A) and writes only i >= j.
//
// Every mbarrier wait is bounded (wall-clock limit read from %globaltimer; the pipeline
// waits use the context's limit, 4 s unless set otherwise); on expiry the thread records
// KF_ERR_TIMEOUT in the device status word and the CTA stops issuing work.  Before it frees
// its tensor memory and returns, the CTA always waits, on the long 4 s limit, for the last
// TMA loads it issued and for every MMA it issued, so nothing it started is still writing
// shared or tensor memory when it exits.
#include "kf_internal.cuh"
#include "kf_tc_ptx.cuh"

#include <cstring>

namespace kf {
namespace {

constexpr int TBM = 128, TBN = 256, TBK = 64, STAGES = 4;
constexpr uint32_t A_BYTES = TBM * TBK * 2;  // 16 KB
constexpr uint32_t B_BYTES = TBN * TBK * 2;  // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;  // stages + alignment + barriers
constexpr uint32_t TMEM_COLS = 256;
constexpr int SUPER_M = 8, SUPER_N = 4;

constexpr int MAX_PASS = 6;
struct TcMaps {
  CUtensorMap a[MAX_PASS];
  CUtensorMap b[MAX_PASS];
};

struct TcArgs {
  int64_t M, N, K;
  int npass;
  float* D;
  int64_t ldd;
  int accumulate, sched, krange;
  int negate;    // D (+)= -result
  int vec_ok;    // D base 16-byte aligned and ldd a multiple of 4 (host-checked)
  int64_t kcb;   // k-blocks per accumulation chunk (0: the whole K range)
  int64_t ntm, ntn;
  int* status;
  unsigned long long wait_ns;  // limit of the pipeline waits
};

// Instruction descriptor, kind::f16: D float32, A and B bfloat16, M = 128, N = 256.
__host__ __device__ constexpr uint32_t make_idesc(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16) |
         (uint32_t(TBN >> 3) << 17) | (uint32_t(TBM >> 4) << 24);
}

__device__ __forceinline__ int64_t lower_limit(int64_t tm) {  // last valid n-tile of row tm
  return (tm * TBM + TBM - 1) / TBN;
}

// Maps a linear tile index to (tm, tn): super-tiles of SUPER_M x SUPER_N tiles in
// row-major order, tiles row-major inside a super-tile; TC_LOWER skips the tiles that lie
// entirely above the diagonal.
__device__ bool decode_tile(int64_t idx, const TcArgs& g, int64_t& tm, int64_t& tn) {
  const int64_t sm_rows = (g.ntm + SUPER_M - 1) / SUPER_M, sm_cols = (g.ntn + SUPER_N - 1) / SUPER_N;
  for (int64_t sr = 0; sr < sm_rows; ++sr) {
    for (int64_t sc = 0; sc < sm_cols; ++sc) {
      const int64_t m_lo = sr * SUPER_M, m_hi = min(g.ntm, m_lo + SUPER_M);
      const int64_t n_lo = sc * SUPER_N, n_hi = min(g.ntn, n_lo + SUPER_N);
      if (g.sched == TC_LOWER && n_lo > lower_limit(m_hi - 1)) break;  // rest of row is above
      for (int64_t r = m_lo; r < m_hi; ++r) {
        const int64_t lim = g.sched == TC_LOWER ? min(n_hi, lower_limit(r) + 1) : n_hi;
        const int64_t cnt = lim > n_lo ? lim - n_lo : 0;
        if (idx < cnt) {
          tm = r;
          tn = n_lo + idx;
          return true;
        }
        idx -= cnt;
      }
    }
  }
  return false;
}

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(320, 1) tc_gemm_kernel(const __grid_constant__ TcMaps maps,
                                                         const TcArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars: full[STAGES] | empty[STAGES] | acc_full[2] | acc_empty[2] | done ; then the TMEM slot
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t accf0 = smem_u32(bars + 2 * STAGES), acce0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t done = smem_u32(bars + 2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int64_t tm, tn;
  if (!decode_tile(blockIdx.x, g, tm, tn)) return;  // uniform over the CTA
  const int64_t m0 = tm * TBM, n0 = tn * TBN;

  int64_t klo = 0, khi = g.K;
  if (g.krange == KR_GE_ROW) klo = m0;
  else if (g.krange == KR_LE_ROW) khi = min(g.K, m0 + TBM);
  else if (g.krange == KR_GE_COL) klo = n0;
  else if (g.krange == KR_LE_COL) khi = min(g.K, n0 + TBN);
  const int64_t nkb = khi > klo ? (khi - klo + TBK - 1) / TBK : 0;
  const int64_t kcb = (g.kcb > 0 && g.kcb < nkb) ? g.kcb : (nkb > 0 ? nkb : 1);
  const int64_t nchunks = nkb > 0 ? (nkb + kcb - 1) / kcb : 1;
  const uint32_t tmem_cols = nchunks > 1 ? 2 * TMEM_COLS : TMEM_COLS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accf0, 1);
    mbar_init(accf0 + 8, 1);
    mbar_init(acce0, 8);
    mbar_init(acce0 + 8, 8);
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: k-blocks of every chunk, every pass
      int64_t issued = 0, it = 0;
      for (int64_t c = 0; c < nchunks && nkb > 0; ++c) {
        const int64_t kb0 = c * kcb, kb1 = min(nkb, kb0 + kcb);
        for (int p = 0; p < g.npass; ++p) {
          for (int64_t kb = kb0; kb < kb1; ++kb, ++it) {
            const int s = int(it % STAGES);
            const uint32_t ph = uint32_t((it / STAGES) & 1);
            if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, g.wait_ns)) {
              raise_status(g.status, KF_ERR_TIMEOUT, WAIT_TMA_EMPTY);
              atomicExch(&abort_flag, 1);
            }
            if (*(volatile int*)&abort_flag) goto producer_done;
            const int32_t k0 = int32_t(klo + kb * TBK);
            const uint32_t sa = smem_u32(smem + s * STAGE_BYTES), sb = sa + A_BYTES;
            const uint32_t fb = full0 + 8 * s;
            mbar_expect_tx(fb, STAGE_BYTES);
            if (A_MN) {
              tma_load_2d(sa, &maps.a[p], int32_t(m0), k0, fb);
              tma_load_2d(sa + 8192, &maps.a[p], int32_t(m0 + 64), k0, fb);
            } else {
              tma_load_2d(sa, &maps.a[p], k0, int32_t(m0), fb);
            }
            if (B_MN) {
#pragma unroll
              for (int h = 0; h < 4; ++h) tma_load_2d(sb + 8192 * h, &maps.b[p], int32_t(n0 + 64 * h), k0, fb);
            } else {
              tma_load_2d(sb, &maps.b[p], k0, int32_t(n0), fb);
            }
            issued = it + 1;
          }
        }
      }
    producer_done:
      // Every issued load must land before the CTA may exit, also when another thread gives
      // up after this one has finished issuing: wait for the last STAGES loads (one per
      // stage; earlier ones were consumed).  Without an abort they have landed already.
      for (int64_t j = (issued > STAGES ? issued - STAGES : 0); j < issued; ++j) {
        if (!mbar_wait(full0 + 8 * int(j % STAGES), uint32_t((j / STAGES) & 1)))
          raise_status(g.status, KF_ERR_TIMEOUT, WAIT_DRAIN);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer (one thread)
      constexpr uint32_t idesc = make_idesc(A_MN, B_MN);
      int64_t it = 0;
      for (int64_t c = 0; c < nchunks; ++c) {
        const int b = int(c & 1);
        if (c >= 2 && !*(volatile int*)&abort_flag) {
          if (!mbar_wait(acce0 + 8 * b, uint32_t(((c >> 1) - 1) & 1), g.wait_ns)) {
            raise_status(g.status, KF_ERR_TIMEOUT, WAIT_MMA_DONE);
            atomicExch(&abort_flag, 1);
          }
        }
        tc_fence_after();
        const uint32_t acc = tmem + uint32_t(b * TMEM_COLS);
        const int64_t kb0 = c * kcb, kb1 = nkb > 0 ? min(nkb, kb0 + kcb) : 0;
        int64_t first = 1;
        for (int p = 0; p < g.npass && !*(volatile int*)&abort_flag; ++p) {
          for (int64_t kb = kb0; kb < kb1; ++kb, ++it) {
            const int s = int(it % STAGES);
            const uint32_t ph = uint32_t((it / STAGES) & 1);
            if (!mbar_wait(full0 + 8 * s, ph, g.wait_ns)) {
              raise_status(g.status, KF_ERR_TIMEOUT, WAIT_TMA_FULL);
              atomicExch(&abort_flag, 1);
            }
            if (*(volatile int*)&abort_flag) break;
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * STAGE_BYTES), sb = sa + A_BYTES;
#pragma unroll
            for (int kk = 0; kk < TBK / 16; ++kk) {
              // A: K-major SW128 (rows of 128 B, 8-row groups 1024 B apart, k-step 32 B) or
              //    MN-major SW128 (64-wide MN chunks 8 KB apart, 8-row k groups 1024 B apart).
              const uint64_t ad = A_MN ? smem_desc(sa + kk * 2048, 8192, 1024) : smem_desc(sa + kk * 32, 16, 1024);
              const uint64_t bd = B_MN ? smem_desc(sb + kk * 2048, 8192, 1024) : smem_desc(sb + kk * 32, 16, 1024);
              tc_mma(acc, ad, bd, idesc, (first && kk == 0) ? 0u : 1u);
            }
            first = 0;
            tc_commit(empty0 + 8 * s);
          }
        }
        tc_commit(accf0 + 8 * b);
      }
      tc_commit(done);
    }
  } else {
    // ---------------- epilogue warps 2..9: warp w reads TMEM lanes 32 (w % 4) .. + 31 (one
    // output row per thread) and 128 of the 256 columns ((w - 2) / 4 selects the half).  The
    // chunk partials are summed in registers with IEEE float32 adds; global memory is touched
    // once per tile, after the last chunk.
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int64_t row = m0 + quarter * 32 + lane;
    const int64_t col0 = n0 + half * 128;
    float acc[128];
#pragma unroll
    for (int j = 0; j < 128; ++j) acc[j] = 0.f;
    bool all_ok = true;
    for (int64_t c = 0; c < nchunks; ++c) {
      const int b = int(c & 1);
      bool ok = mbar_wait(accf0 + 8 * b, uint32_t((c >> 1) & 1), g.wait_ns);
      if (!ok) {
        raise_status(g.status, KF_ERR_TIMEOUT, WAIT_MMA_DONE);
        atomicExch(&abort_flag, 1);
      }
      if (*(volatile int*)&abort_flag) ok = false;
      all_ok = all_ok && ok;
      tc_fence_after();
      if (ok && nkb > 0) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          const uint32_t taddr =
              tmem + (uint32_t(quarter * 32) << 16) + uint32_t(b * TMEM_COLS + half * 128 + cc * 32);
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
              "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
              : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
                "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
              : "r"(taddr));
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[cc * 32 + j] += __uint_as_float(v[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(acce0 + 8 * b) : "memory");
    }
    // Write the tile: D = acc (or D += acc), rows < M, columns < N, lower triangle for TC_LOWER.
    if (all_ok && row < g.M) {
      const bool vec_ok = g.vec_ok != 0;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int64_t c0 = col0 + cc * 32;
        if (c0 >= g.N || (g.sched == TC_LOWER && c0 > row)) continue;
        float* dst = g.D + row * g.ldd + c0;
        bool full = vec_ok && c0 + 32 <= g.N && (g.sched != TC_LOWER || c0 + 31 <= row);
        if (full && (reinterpret_cast<uintptr_t>(dst) & 15) != 0) {  // alignment self-check
          raise_status(g.status, KF_ERR_INVALID, 131);
          full = false;
        }
        if (full) {
          float4 old[8];
          if (g.accumulate) {
#pragma unroll
            for (int j = 0; j < 8; ++j) old[j] = reinterpret_cast<const float4*>(dst)[j];
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float4 o = make_float4(acc[cc * 32 + 4 * j], acc[cc * 32 + 4 * j + 1], acc[cc * 32 + 4 * j + 2],
                                   acc[cc * 32 + 4 * j + 3]);
            if (g.negate) {
              o.x = -o.x; o.y = -o.y; o.z = -o.z; o.w = -o.w;
            }
            if (g.accumulate) {
              o.x += old[j].x; o.y += old[j].y; o.z += old[j].z; o.w += old[j].w;
            }
            reinterpret_cast<float4*>(dst)[j] = o;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t col = c0 + j;
            if (col >= g.N || (g.sched == TC_LOWER && col > row)) continue;
            const float v = g.negate ? -acc[cc * 32 + j] : acc[cc * 32 + j];
            dst[j] = g.accumulate ? dst[j] + v : v;
          }
        }
      }
    }
  }
  __syncwarp();
  // Every MMA must have completed before the tensor memory is released.
  if (!mbar_wait(done, 0)) raise_status(g.status, KF_ERR_TIMEOUT, WAIT_MMA_DONE);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
  }
}

kf_status encode_operand(kf_ctx* ctx, CUtensorMap* map, const TcOperand& op, int64_t rows_mn,
                         int64_t k, bool is_b) {
  // Global tensor: MN-major -> {MN (inner), K}; K-major -> {K (inner), MN}.
  cuuint64_t dims[2], strides[1];
  cuuint32_t box[2], estr[2] = {1, 1};
  if (op.mn_major) {
    dims[0] = cuuint64_t(rows_mn); dims[1] = cuuint64_t(k);
    box[0] = 64; box[1] = TBK;
  } else {
    dims[0] = cuuint64_t(k); dims[1] = cuuint64_t(rows_mn);
    box[0] = TBK; box[1] = is_b ? TBN : TBM;
  }
  strides[0] = cuuint64_t(op.ld) * 2;
  if ((reinterpret_cast<uintptr_t>(op.ptr) & 15) != 0 || (strides[0] & 15) != 0)
    return fail(KF_ERR_INVALID, "tensor-core operand: base must be 16-byte aligned and ld*2 a multiple of 16");
  if (dims[0] == 0 || dims[1] == 0) return fail(KF_ERR_INVALID, "tensor-core operand: empty");
  CUresult r = ctx->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(op.ptr), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KF_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string(int(r)) + ")");
  return KF_OK;
}

int64_t count_tiles(const TcGemm& g, int64_t ntm, int64_t ntn) {
  if (g.sched != TC_LOWER) return ntm * ntn;
  int64_t c = 0;
  for (int64_t tm = 0; tm < ntm; ++tm) {
    const int64_t lim = (tm * TBM + TBM - 1) / TBN + 1;
    c += lim < ntn ? lim : ntn;
  }
  return c;
}

template <bool AM, bool BM_>
kf_status launch_tc(const TcMaps& maps, const TcArgs& a, int64_t ntiles, cudaStream_t st) {
  static std::atomic<unsigned long long> attr_done{0};  // per instantiation and device
  KF_TRY(set_attr_once(attr_done, [] {
    return check_cuda(cudaFuncSetAttribute(tc_gemm_kernel<AM, BM_>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           int(SMEM_BYTES)), "tc_gemm smem attribute");
  }));
  tc_gemm_kernel<AM, BM_><<<unsigned(ntiles), 320, SMEM_BYTES, st>>>(maps, a); note_launch();
  return check_cuda(cudaGetLastError(), "tc_gemm launch");
}

}  // namespace

kf_status tc_gemm(kf_ctx* ctx, const TcGemm& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return KF_OK;
  if (g.npass < 1 || g.npass > MAX_PASS) return fail(KF_ERR_INVALID, "tc_gemm: 1..6 passes");
  if (!ctx->encode) return fail(KF_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  TcMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  for (int p = 0; p < g.npass; ++p) {
    if (g.a[p].mn_major != g.a[0].mn_major || g.b[p].mn_major != g.b[0].mn_major)
      return fail(KF_ERR_INVALID, "tc_gemm: all passes need the same operand majors");
    KF_TRY(encode_operand(ctx, &maps.a[p], g.a[p], g.M, g.K, false));
    KF_TRY(encode_operand(ctx, &maps.b[p], g.b[p], g.N, g.K, true));
  }
  TcArgs a{};
  a.M = g.M; a.N = g.N; a.K = g.K; a.npass = g.npass;
  a.D = g.D; a.ldd = g.ldd;
  a.accumulate = g.accumulate ? 1 : 0; a.sched = g.sched; a.krange = g.krange;
  a.negate = g.negate ? 1 : 0;
  a.vec_ok = ((g.ldd % 4) == 0 && (reinterpret_cast<uintptr_t>(g.D) & 15) == 0) ? 1 : 0;
  a.kcb = g.kchunk > 0 ? (g.kchunk + TBK - 1) / TBK : 0;
  a.ntm = (g.M + TBM - 1) / TBM; a.ntn = (g.N + TBN - 1) / TBN;
  a.status = ctx->d_status;
  a.wait_ns = ctx->wait_ns;
  const int64_t ntiles = count_tiles(g, a.ntm, a.ntn);
  if (ntiles > 0x7fffffff) return fail(KF_ERR_UNSUPPORTED, "tc_gemm: too many tiles");
  const bool am = g.a[0].mn_major, bm = g.b[0].mn_major;
  if (am && bm) return launch_tc<true, true>(maps, a, ntiles, st);
  if (am) return launch_tc<true, false>(maps, a, ntiles, st);
  if (bm) return launch_tc<false, true>(maps, a, ntiles, st);
  return launch_tc<false, false>(maps, a, ntiles, st);
}

}  // namespace kf
