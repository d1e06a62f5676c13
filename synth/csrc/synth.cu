// Device twin of synth/philox.py: Philox4x32-10 (Salmon et al., SC'11) and the
// twelve-term integer Irwin-Hall normal.  Fills row ranges of a synthetic calibration
// stream or weight matrix directly in device memory, so that large workloads never
// pass through the host.  Bit-identical to the numpy definition (tests/test_synth.py).
//
// This library holds no arithmetic of the compression method itself.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

struct u32x4 { uint32_t x, y, z, w; };

__device__ __forceinline__ u32x4 philox4x32_10(u32x4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = u32x4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ int halves(uint32_t w) { return int(w & 0xFFFFu) + int(w >> 16); }

__device__ __forceinline__ float irwin_hall_normal(uint64_t e, uint32_t k0, uint32_t k1) {
  const uint32_t lo = uint32_t(e), hi = uint32_t(e >> 32);
  const u32x4 a = philox4x32_10(u32x4{lo, hi, 0u, 0u}, k0, k1);
  const u32x4 b = philox4x32_10(u32x4{lo, hi, 0u, 1u}, k0, k1);
  const int s = halves(a.x) + halves(a.y) + halves(a.z) + halves(a.w) + halves(b.x) + halves(b.y);
  return __fmul_rn(float(s - 393210), 1.0f / 65536.0f);
}

template <bool BF16>
__global__ void fill_kernel(void* __restrict__ out, int64_t rows, int64_t cols, int64_t ld,
                            int64_t row0, int64_t total_cols, int64_t col0, uint32_t k0,
                            uint32_t k1, const float* __restrict__ stdv, float scale) {
  const int64_t n = rows * cols;
  for (int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
       idx += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = idx / cols, c = idx - r * cols;
    const uint64_t e = uint64_t(row0 + r) * uint64_t(total_cols) + uint64_t(col0 + c);
    const float sd = stdv ? stdv[col0 + c] : scale;
    const float v = __fmul_rn(irwin_hall_normal(e, k0, k1), sd);
    if (BF16)
      reinterpret_cast<__nv_bfloat16*>(out)[r * ld + c] = __float2bfloat16_rn(v);
    else
      reinterpret_cast<float*>(out)[r * ld + c] = v;
  }
}

}  // namespace

extern "C" {

// out: device buffer, rows x cols with leading dimension ld (elements); dtype 0 = bf16,
// 1 = float32.  Element (r, c) takes the generator value of element index
// (row0 + r) * total_cols + (col0 + c) under `seed`, times stdv[col0 + c] (device array,
// may be NULL, then `scale`).  Returns a cudaError_t value.
int kfsynth_fill(void* out, int dtype, int64_t rows, int64_t cols, int64_t ld, int64_t row0,
                 int64_t total_cols, int64_t col0, uint64_t seed, const float* stdv, float scale,
                 cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return 0;
  if (!out || ld < cols) return int(cudaErrorInvalidValue);
  const uint32_t k0 = uint32_t(seed), k1 = uint32_t(seed >> 32);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n = rows * cols;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = int64_t(sms) * 16;
  if (blocks > cap) blocks = cap;
  if (dtype == 0)
    fill_kernel<true><<<unsigned(blocks), 256, 0, stream>>>(out, rows, cols, ld, row0, total_cols,
                                                             col0, k0, k1, stdv, scale);
  else
    fill_kernel<false><<<unsigned(blocks), 256, 0, stream>>>(out, rows, cols, ld, row0, total_cols,
                                                              col0, k0, k1, stdv, scale);
  return int(cudaGetLastError());
}

}  // extern "C"
