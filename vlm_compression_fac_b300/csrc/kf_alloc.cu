// Global sort-and-truncate rank allocation (UniRank 2.1; LASER Methodology 2).
//   keys:  k = (~bits(score) << 32) | component id, score = 0.5f * (sigma * sigma) [/ cost],
//          or UniRank's energy ratio sigma^2 / sum_unit sigma^2, optionally times a per-unit
//          weight (UniRank's layer importance I_l);
//          ascending k is score descending, then lower unit, then lower component index
//          (ids are assigned in unit order), which makes the order total and deterministic;
//   sort:  LSD radix sort of the score word, 4 passes of 8 bits (equal scores keep their id
//          order, since the keys start in id order and every pass is stable); each pass = per-tile digit histogram,
//          one exclusive scan over (digit, tile), stable scatter (warp match + per-warp
//          digit counters keep the original order inside a tile);
//   cut:   inclusive prefix sum of the kept pairs' cost m+n in sorted order; the kept
//          prefix is every position whose prefix sum is <= budget (costs are positive, so
//          the walk stops at the first overflow); ranks = kept count per unit.
#include "kf_internal.cuh"

#include <mutex>

namespace kf {
namespace {

constexpr int RT = 256;            // threads per tile
constexpr int RI = 16;             // keys per thread
constexpr int TILE = RT * RI;      // 4096 keys per tile
constexpr int SCAN_T = 1024;

__device__ __forceinline__ int unit_of(const int64_t* __restrict__ off, int n_units, int64_t g) {
  int lo = 0, hi = n_units;  // off[lo] <= g < off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= g) lo = mid; else hi = mid;
  }
  return lo;
}

// Key of every component: base score per mode (KF_KEY_HALF_SIGMA2: 0.5 sigma^2;
// KF_KEY_PER_PARAM: that divided by the unit's m + n; KF_KEY_ENERGY_RATIO: sigma^2 divided
// by the unit's energy sum sigma^2), times the unit's weight when weights are given (a
// weight that is negative or not a number counts as 0).  float32, one rounding per operation.
constexpr int MODE_GIVEN_KEYS = 100;  // internal: the caller's keys, as given
constexpr int MODE_SWIFT_HYBRID = 101;  // internal: Swift-SVD B hybrid keys built from sigma

// The low word of a key is the component id, or, when no caller needs ids (no keep mask), the
// unit index: the sort orders by the score word only and is stable, so equal scores stay in
// id order either way, and every later pass needs only the unit (its cost, its rank count).
__global__ void build_keys_kernel(const float* __restrict__ sigma, const int64_t* __restrict__ off,
                                  const int64_t* __restrict__ cost, int n_units, int64_t n, int mode,
                                  const float* __restrict__ weight, const float* __restrict__ energy,
                                  unsigned long long* __restrict__ keys, int low_is_unit) {
  for (int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; g < n; g += int64_t(gridDim.x) * blockDim.x) {
    const int u = unit_of(off, n_units, g);
    const float s = sigma[g];
    const float q = __fmul_rn(s, s);
    float sc;
    if (mode == MODE_GIVEN_KEYS) {
      sc = s > 0.f ? s : 0.f;  // a negative or not-a-number key counts as 0
    } else if (mode == KF_KEY_ENERGY_RATIO) {
      const float e = energy[u];
      sc = e > 0.f ? __fdiv_rn(q, e) : 0.f;
    } else {
      sc = 0.5f * q;
      if (mode == KF_KEY_PER_PARAM) sc = __fdiv_rn(sc, float(cost[u]));
    }
    if (weight) {
      const float w = weight[u];
      sc = (w > 0.f) ? __fmul_rn(w, sc) : 0.f;  // also maps a NaN weight to 0
    }
    const unsigned bits = ~__float_as_uint(sc);
    const uint32_t low = low_is_unit ? uint32_t(u) : uint32_t(g);
    keys[g] = (static_cast<unsigned long long>(bits) << 32) | static_cast<unsigned long long>(low);
  }
}

// Swift-SVD B: the closed-form loss of unit u truncated to rank k is the energy it drops,
// eps[g] = sum of sigma^2 from component g to the end of the unit (float64, one term at a
// time from the unit's last component upward: the square of a float32 value is exact in
// float64, so the sum order alone fixes the result).  One thread per unit.
__global__ void swift_eps_kernel(const float* __restrict__ sigma, const int64_t* __restrict__ off, int n_units,
                                 double* __restrict__ eps) {
  for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += gridDim.x * blockDim.x) {
    double acc = 0.0;
    for (int64_t g = off[u + 1] - 1; g >= off[u]; --g) {
      const double v = sigma[g];
      acc = acc + v * v;
      eps[g] = acc;
    }
  }
}

// Swift-SVD B hybrid score as a key per component: component k of unit u gets the unit's
// score at rank k, beta_u^alpha * (log(e + eps_k))^(1 - alpha), in float64 rounded once to
// float32 (beta not positive or not a number: key 0).
__global__ void swift_keys_kernel(const double* __restrict__ eps, const int64_t* __restrict__ off, int n_units,
                                  int64_t n, const float* __restrict__ beta, double alpha, float* __restrict__ keys) {
  for (int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; g < n; g += int64_t(gridDim.x) * blockDim.x) {
    const int u = unit_of(off, n_units, g);
    const float b = beta ? beta[u] : 1.f;
    float k = 0.f;
    if (b > 0.f) k = float(pow(double(b), alpha) * pow(log(2.718281828459045 + eps[g]), 1.0 - alpha));
    keys[g] = k;
  }
}

// energy[u] = sum of sigma^2 over unit u's segment (float64 sum of exact squares, rounded).
__global__ void __launch_bounds__(256) unit_energy_kernel(const float* __restrict__ sigma,
                                                          const int64_t* __restrict__ off,
                                                          float* __restrict__ energy) {
  __shared__ double red[8];
  const int u = blockIdx.x;
  double acc = 0.0;
  for (int64_t g = off[u] + threadIdx.x; g < off[u + 1]; g += blockDim.x) {
    const double v = sigma[g];
    acc += v * v;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < 8; ++w) t += red[w];
    energy[u] = float(t);
  }
}

__global__ void __launch_bounds__(RT) hist_kernel(const unsigned long long* __restrict__ keys, int64_t n, int shift,
                                                  int ntiles, unsigned* __restrict__ hist) {
  __shared__ unsigned h[256];
  h[threadIdx.x] = 0;
  const int64_t base = int64_t(blockIdx.x) * TILE;
  const unsigned lane = threadIdx.x & 31u;
  // all of this thread's keys are requested before the first is used
  unsigned long long k[RI];
#pragma unroll
  for (int i = 0; i < RI; ++i) {
    const int64_t g = base + int64_t(i) * RT + threadIdx.x;
    k[i] = g < n ? keys[g] : 0ull;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < RI; ++i) {
    const int64_t g = base + int64_t(i) * RT + threadIdx.x;
    const unsigned d = g < n ? unsigned((k[i] >> shift) & 255u) : 256u;
    // one shared atomic per distinct digit of the warp (the leading bytes of the keys are
    // often nearly constant, which would serialise per-key atomics on one bin)
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    if (d < 256u && (peers & ((1u << lane) - 1u)) == 0u) atomicAdd(&h[d], unsigned(__popc(peers)));
  }
  __syncthreads();
  hist[int64_t(threadIdx.x) * ntiles + blockIdx.x] = h[threadIdx.x];
}

// Multi-CTA exclusive scan of a long uint array in chunks of SCAN_CHUNK: block sums, a scan of
// the sums, then every chunk rescanned from its base (same result as one sequential scan).
constexpr int64_t SCAN_CHUNK = 8 * 1024;

__global__ void __launch_bounds__(1024) chunk_sum_u32_kernel(const unsigned* __restrict__ a, int64_t len,
                                                             unsigned* __restrict__ bsum) {
  __shared__ unsigned red[32];
  const int64_t c0 = int64_t(blockIdx.x) * SCAN_CHUNK;
  unsigned s = 0;
  for (int64_t i = c0 + threadIdx.x; i < len && i < c0 + SCAN_CHUNK; i += 1024) s += a[i];
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned t = 0;
    for (int w = 0; w < 32; ++w) t += red[w];
    bsum[blockIdx.x] = t;
  }
}

// Exclusive scan of a uint array: CTA b scans [b * chunk, min(len, (b + 1) * chunk)) in steps
// of SCAN_T, starting from base[b] (or 0 without base).  One CTA with chunk >= len scans the
// whole array.
__global__ void __launch_bounds__(SCAN_T) scan_u32_kernel(unsigned* __restrict__ a, int64_t len, int64_t chunk,
                                                          const unsigned* __restrict__ cbase) {
  __shared__ unsigned ws[32];
  __shared__ unsigned carry;
  if (threadIdx.x == 0) carry = cbase ? cbase[blockIdx.x] : 0u;
  __syncthreads();
  const int64_t lo = int64_t(blockIdx.x) * chunk;
  const int64_t hi = lo + chunk < len ? lo + chunk : len;
  for (int64_t c0 = lo; c0 < hi; c0 += SCAN_T) {
    const int64_t i = c0 + threadIdx.x;
    const unsigned v = i < hi ? a[i] : 0u;
    unsigned x = v;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) ws[w] = x;
    __syncthreads();
    if (w == 0) {
      unsigned z = ws[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, z, o);
        if (lane >= o) z += y;
      }
      ws[lane] = z;
    }
    __syncthreads();
    const unsigned incl = x + (w > 0 ? ws[w - 1] : 0u) + carry;
    if (i < hi) a[i] = incl - v;
    __syncthreads();
    if (threadIdx.x == SCAN_T - 1) carry = incl;
    __syncthreads();
  }
}

// Stable scatter of one 4096-key tile.  Warp w owns the tile's keys w * WK .. w * WK + WK - 1
// (WK = TILE / 8; the warp's round r holds keys w * WK + 32 r + lane), so the tile's index
// order is (warp, round, lane) order.  All keys are loaded first; phase 1 counts each warp's
// keys per digit (one counter update per distinct digit of a round, by warp match); one pass
// over the warps per digit turns the counts into each (digit, warp)'s first position in the
// tile's digit-ordered copy in shared memory; phase 2 puts every key at its warp's running
// position for its digit plus its rank among the round's equal digits; the copy is then
// written out so that consecutive threads write consecutive addresses of one digit's run
// (coalesced).  The tile's digit counts come from the scanned (digit, tile) histogram:
// count[d] = base of the next tile (or digit) minus this base.
constexpr int WK = TILE / (RT / 32);
__global__ void __launch_bounds__(RT, 3) scatter_kernel(const unsigned long long* __restrict__ in,
                                                     unsigned long long* __restrict__ out, int64_t n, int shift,
                                                     int ntiles, const unsigned* __restrict__ hist) {
  __shared__ unsigned base[256];
  __shared__ unsigned start[256];   // the digit's first position in the tile's ordered copy
  __shared__ unsigned wpos[RT / 32][256];   // per-warp digit counts, then running positions
  __shared__ unsigned long long tk[TILE];
  __shared__ unsigned wsum[RT / 32];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int64_t tile0 = int64_t(blockIdx.x) * TILE;
  const int tile_n = int(n - tile0 < TILE ? n - tile0 : TILE);
  unsigned long long key[RI];
#pragma unroll
  for (int r = 0; r < RI; ++r) {
    const int li = w * WK + r * 32 + lane;
    key[r] = li < tile_n ? in[tile0 + li] : 0ull;
  }
  for (int x = lane; x < 256; x += 32) wpos[w][x] = 0;
  {
    const int64_t hi = int64_t(t) * ntiles + blockIdx.x;
    base[t] = hist[hi];
    const unsigned nxt = (blockIdx.x + 1 < ntiles) ? hist[hi + 1] : (t + 1 < 256 ? hist[int64_t(t + 1) * ntiles] : unsigned(n));
    const unsigned cnt = nxt - base[t];
    // exclusive scan of the 256 counts (one per thread) -> start
    unsigned x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    unsigned pre = 0;
    for (int ww = 0; ww < w; ++ww) pre += wsum[ww];
    start[t] = pre + x - cnt;
  }
  unsigned peers[RI];
#pragma unroll
  for (int r = 0; r < RI; ++r) {
    const bool valid = w * WK + r * 32 + lane < tile_n;
    const unsigned d = valid ? unsigned((key[r] >> shift) & 255u) : 256u;
    peers[r] = __match_any_sync(0xffffffffu, d);
    if (valid && (peers[r] & lt_mask) == 0u) wpos[w][d] += __popc(peers[r]);
    __syncwarp();
  }
  __syncthreads();
  {  // per digit: each warp's first position, in warp order
    unsigned acc = start[t];
#pragma unroll
    for (int ww = 0; ww < RT / 32; ++ww) {
      const unsigned c = wpos[ww][t];
      wpos[ww][t] = acc;
      acc += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < RI; ++r) {
    const bool valid = w * WK + r * 32 + lane < tile_n;
    const unsigned d = valid ? unsigned((key[r] >> shift) & 255u) : 0u;
    const unsigned pos = valid ? wpos[w][d] : 0u;
    if (valid) tk[pos + __popc(peers[r] & lt_mask)] = key[r];
    __syncwarp();
    if (valid && (peers[r] & lt_mask) == 0u) wpos[w][d] = pos + __popc(peers[r]);
    __syncwarp();
  }
  __syncthreads();
  for (int i = t; i < tile_n; i += RT) {
    const unsigned long long k = tk[i];
    const unsigned d = unsigned((k >> shift) & 255u);
    out[base[d] + (unsigned(i) - start[d])] = k;
  }
}

__device__ __forceinline__ int key_unit(unsigned long long k, const int64_t* __restrict__ off, int n_units,
                                        int low_is_unit) {
  return low_is_unit ? int(uint32_t(k)) : unit_of(off, n_units, int64_t(uint32_t(k)));
}

// Inclusive prefix sums of the sorted components' costs, per 1024-item block.
__global__ void __launch_bounds__(SCAN_T) cost_block_sum_kernel(const unsigned long long* __restrict__ keys,
                                                                const int64_t* __restrict__ off,
                                                                const int64_t* __restrict__ cost, int n_units,
                                                                int64_t n, long long* __restrict__ bsum,
                                                                int low_is_unit) {
  __shared__ long long red[SCAN_T / 32];
  const int64_t i = int64_t(blockIdx.x) * SCAN_T + threadIdx.x;
  long long c = 0;
  if (i < n) c = cost[key_unit(keys[i], off, n_units, low_is_unit)];
#pragma unroll
  for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long s = 0;
    for (int w = 0; w < SCAN_T / 32; ++w) s += red[w];
    bsum[blockIdx.x] = s;
  }
}

__global__ void __launch_bounds__(SCAN_T) scan_i64_kernel(long long* __restrict__ a, int64_t len) {
  __shared__ long long ws[32];
  __shared__ long long carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int64_t c0 = 0; c0 < len; c0 += SCAN_T) {
    const int64_t i = c0 + threadIdx.x;
    const long long v = i < len ? a[i] : 0;
    long long x = v;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) ws[w] = x;
    __syncthreads();
    if (w == 0) {
      long long z = ws[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, z, o);
        if (lane >= o) z += y;
      }
      ws[lane] = z;
    }
    __syncthreads();
    const long long incl = x + (w > 0 ? ws[w - 1] : 0) + carry;
    if (i < len) a[i] = incl - v;
    __syncthreads();
    if (threadIdx.x == SCAN_T - 1) carry = incl;
    __syncthreads();
  }
}

// Per item: the inclusive prefix sum of the costs in sorted order.
__global__ void __launch_bounds__(SCAN_T) cut_kernel(const unsigned long long* __restrict__ keys,
                                                     const int64_t* __restrict__ off, const int64_t* __restrict__ cost,
                                                     int n_units, int64_t n, const long long* __restrict__ bexcl,
                                                     long long* __restrict__ prefix, int low_is_unit) {
  __shared__ long long ws[32];
  const int64_t i = int64_t(blockIdx.x) * SCAN_T + threadIdx.x;
  long long c = 0;
  if (i < n) c = cost[key_unit(keys[i], off, n_units, low_is_unit)];
  long long x = c;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[w] = x;
  __syncthreads();
  if (w == 0) {
    long long z = ws[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    ws[lane] = z;
  }
  __syncthreads();
  const long long incl = x + (w > 0 ? ws[w - 1] : 0) + bexcl[blockIdx.x];
  if (i < n) prefix[i] = incl;
}

// kcount = the length of the kept prefix: the largest k with prefix[k - 1] <= budget.  The
// costs are non-negative, so the prefix sums never decrease and a binary search finds it
// (one thread, about log2(n) reads).
__global__ void kcount_kernel(const long long* __restrict__ prefix, int64_t n, long long budget,
                              unsigned long long* __restrict__ kcount) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    const int64_t mid = lo + (hi - lo + 1) / 2;
    if (prefix[mid - 1] <= budget) lo = mid; else hi = mid - 1;
  }
  *kcount = static_cast<unsigned long long>(lo);
}

// ranks[u] += the kept components of unit u.  With at most RANKS_SMEM_UNITS units each
// block counts in shared memory and adds its nonzero counts once; beyond that, one global
// atomic per component.
constexpr int RANKS_SMEM_UNITS = 8192;
__global__ void ranks_kernel(const unsigned long long* __restrict__ keys, const int64_t* __restrict__ off,
                             int n_units, const unsigned long long* __restrict__ kcount, int* __restrict__ ranks,
                             int low_is_unit) {
  extern __shared__ int rcount[];
  const bool local = n_units <= RANKS_SMEM_UNITS;  // uniform over the grid
  if (local) {
    for (int u = threadIdx.x; u < n_units; u += blockDim.x) rcount[u] = 0;
    __syncthreads();
  }
  const int64_t k = int64_t(*kcount);
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < k; i += int64_t(gridDim.x) * blockDim.x) {
    const int u = key_unit(keys[i], off, n_units, low_is_unit);
    if (local) atomicAdd(&rcount[u], 1); else atomicAdd(&ranks[u], 1);
  }
  if (local) {
    __syncthreads();
    for (int u = threadIdx.x; u < n_units; u += blockDim.x)
      if (rcount[u]) atomicAdd(&ranks[u], rcount[u]);
  }
}

// keep[id] = 1 for the components of the kept prefix (the mask was cleared before).
__global__ void keep_mask_kernel(const unsigned long long* __restrict__ keys,
                                 const unsigned long long* __restrict__ kcount, unsigned char* __restrict__ keep) {
  const int64_t k = int64_t(*kcount);
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < k; i += int64_t(gridDim.x) * blockDim.x)
    keep[uint32_t(keys[i])] = 1;
}

__device__ __forceinline__ float key_score(unsigned long long k) { return __uint_as_float(~unsigned(k >> 32)); }

__global__ void finish_kernel(const unsigned long long* __restrict__ keys, const long long* __restrict__ prefix,
                              int64_t n, const unsigned long long* __restrict__ kcount, float* __restrict__ cut,
                              long long* __restrict__ used) {
  const int64_t k = int64_t(*kcount);
  if (cut) {
    cut[0] = k > 0 ? key_score(keys[k - 1]) : __int_as_float(0x7fc00000);
    cut[1] = k < n ? key_score(keys[k]) : __int_as_float(0x7fc00000);
  }
  if (used) *used = k > 0 ? prefix[k - 1] : 0;
}

__global__ void fixed_rank_kernel(const int64_t* __restrict__ off, const int64_t* __restrict__ cost, int n_units,
                                  const int* __restrict__ fixed, int* __restrict__ ranks, float* __restrict__ cut,
                                  long long* __restrict__ used) {
  __shared__ long long red[256];
  long long acc = 0;
  for (int u = threadIdx.x; u < n_units; u += blockDim.x) {
    const long long len = off[u + 1] - off[u];
    long long r = fixed[u] < 0 ? 0 : fixed[u];
    if (r > len) r = len;
    ranks[u] = int(r);
    acc += r * cost[u];
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (used) *used = red[0];
    if (cut) cut[0] = cut[1] = __int_as_float(0x7fc00000);
  }
}

unsigned grid_cap(int64_t n, int per) {
  int64_t b = (n + per - 1) / per;
  if (b > 148 * 16) b = 148 * 16;
  return unsigned(b < 1 ? 1 : b);
}

struct AllocBufs {
  unsigned long long *ka, *kb, *kcount;
  unsigned *hist, *hsum;
  long long *bsum, *prefix;
  float* energy;
};

// n_energy: units whose energy is needed (KF_KEY_ENERGY_RATIO), else 0.
size_t alloc_carve(Carve& cv, int64_t n, int64_t n_energy, AllocBufs& b) {
  const int64_t ntiles = (n + TILE - 1) / TILE;
  const int64_t nb = (n + SCAN_T - 1) / SCAN_T;
  b.ka = cv.take<unsigned long long>(n > 0 ? n : 1);
  b.kb = cv.take<unsigned long long>(n > 0 ? n : 1);
  b.hist = cv.take<unsigned>(size_t(256) * (ntiles > 0 ? ntiles : 1));
  b.hsum = cv.take<unsigned>(size_t((256 * (ntiles > 0 ? ntiles : 1) + SCAN_CHUNK - 1) / SCAN_CHUNK));
  b.bsum = cv.take<long long>(nb > 0 ? nb : 1);
  b.prefix = cv.take<long long>(n > 0 ? n : 1);
  b.kcount = cv.take<unsigned long long>(1);
  b.energy = n_energy > 0 ? cv.take<float>(n_energy) : nullptr;
  return cv.off;
}

}  // namespace

int alloc_mode_given_keys() { return MODE_GIVEN_KEYS; }
int alloc_mode_swift_hybrid() { return MODE_SWIFT_HYBRID; }

size_t alloc_workspace(int64_t n, int64_t n_energy) {
  Carve cv(nullptr, 0, true);
  AllocBufs b;
  return alloc_carve(cv, n, n_energy, b) + 256;
}

kf_status alloc_run(kf_ctx* ctx, const float* sigma, const int64_t* off, const int64_t* cost, int32_t n_units,
                    int64_t n, int64_t budget, kf_alloc_mode mode, const int32_t* fixed, const float* weight,
                    int32_t* ranks, float* cut, int64_t* used, void* ws, size_t ws_bytes, cudaStream_t st,
                    unsigned char* keep, double alpha) {
  (void)ctx;
  KF_CUDA(cudaMemsetAsync(ranks, 0, sizeof(int32_t) * size_t(n_units), st));
  if (mode == KF_FIXED_RANK) {
    fixed_rank_kernel<<<1, 256, 0, st>>>(off, cost, n_units, fixed, ranks, cut, (long long*)used); note_launch();
    return check_cuda(cudaGetLastError(), "fixed_rank launch");
  }
  Carve cv(ws, ws_bytes, false);
  AllocBufs b;
  alloc_carve(cv, n, mode == KF_KEY_ENERGY_RATIO ? n_units : 0, b);
  if (!cv.fits()) return fail(KF_ERR_WORKSPACE, "score_and_allocate: workspace too small");
  const int ntiles = int((n + TILE - 1) / TILE);
  const int low_is_unit = keep ? 0 : 1;
  if (mode == KF_KEY_ENERGY_RATIO) {
    unit_energy_kernel<<<unsigned(n_units), 256, 0, st>>>(sigma, off, b.energy); note_launch();
    KF_CUDA(cudaGetLastError());
  }
  if (int(mode) == MODE_SWIFT_HYBRID) {
    // eps (float64) in the second key buffer and the float keys in the prefix buffer: both
    // are free until the first radix scatter and the cost prefix respectively.
    double* eps = reinterpret_cast<double*>(b.kb);
    float* hk = reinterpret_cast<float*>(b.prefix);
    swift_eps_kernel<<<unsigned((n_units + 127) / 128), 128, 0, st>>>(sigma, off, n_units, eps); note_launch();
    KF_CUDA(cudaGetLastError());
    swift_keys_kernel<<<grid_cap(n, 256), 256, 0, st>>>(eps, off, n_units, n, weight, alpha, hk); note_launch();
    KF_CUDA(cudaGetLastError());
    build_keys_kernel<<<grid_cap(n, 256), 256, 0, st>>>(hk, off, cost, n_units, n, MODE_GIVEN_KEYS, nullptr,
                                                        nullptr, b.ka, low_is_unit); note_launch();
  } else {
    build_keys_kernel<<<grid_cap(n, 256), 256, 0, st>>>(sigma, off, cost, n_units, n, int(mode), weight, b.energy,
                                                        b.ka, low_is_unit); note_launch();
  }
  KF_CUDA(cudaGetLastError());
  // The keys are built in id order and every pass is stable, so sorting by the score word
  // alone (the upper 32 bits, four 8-bit passes) leaves equal scores in id order: the same
  // total order as sorting all 64 bits, at half the passes.
  unsigned long long* src = b.ka;
  unsigned long long* dst = b.kb;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 32 + pass * 8;
    hist_kernel<<<ntiles, RT, 0, st>>>(src, n, shift, ntiles, b.hist); note_launch();
    KF_CUDA(cudaGetLastError());
    const int64_t hlen = int64_t(256) * ntiles;
    if (hlen <= SCAN_CHUNK) {
      scan_u32_kernel<<<1, SCAN_T, 0, st>>>(b.hist, hlen, hlen, nullptr); note_launch();
      KF_CUDA(cudaGetLastError());
    } else {
      const int64_t nch = (hlen + SCAN_CHUNK - 1) / SCAN_CHUNK;
      chunk_sum_u32_kernel<<<unsigned(nch), 1024, 0, st>>>(b.hist, hlen, b.hsum); note_launch();
      KF_CUDA(cudaGetLastError());
      scan_u32_kernel<<<1, SCAN_T, 0, st>>>(b.hsum, nch, nch, nullptr); note_launch();
      KF_CUDA(cudaGetLastError());
      scan_u32_kernel<<<unsigned(nch), SCAN_T, 0, st>>>(b.hist, hlen, SCAN_CHUNK, b.hsum); note_launch();
      KF_CUDA(cudaGetLastError());
    }
    scatter_kernel<<<ntiles, RT, 0, st>>>(src, dst, n, shift, ntiles, b.hist); note_launch();
    KF_CUDA(cudaGetLastError());
    unsigned long long* tmp = src;
    src = dst;
    dst = tmp;
  }
  // src now holds the sorted keys.
  const int64_t nb = (n + SCAN_T - 1) / SCAN_T;
  cost_block_sum_kernel<<<unsigned(nb), SCAN_T, 0, st>>>(src, off, cost, n_units, n, b.bsum, low_is_unit);
  note_launch();
  KF_CUDA(cudaGetLastError());
  scan_i64_kernel<<<1, SCAN_T, 0, st>>>(b.bsum, nb); note_launch();
  KF_CUDA(cudaGetLastError());
  cut_kernel<<<unsigned(nb), SCAN_T, 0, st>>>(src, off, cost, n_units, n, b.bsum, b.prefix, low_is_unit);
  note_launch();
  KF_CUDA(cudaGetLastError());
  kcount_kernel<<<1, 1, 0, st>>>(b.prefix, n, budget, b.kcount); note_launch();
  KF_CUDA(cudaGetLastError());
  const size_t rsmem = n_units <= RANKS_SMEM_UNITS ? sizeof(int) * size_t(n_units > 0 ? n_units : 1) : 0;
  ranks_kernel<<<grid_cap(n, 256), 256, rsmem, st>>>(src, off, n_units, b.kcount, ranks, low_is_unit);
  note_launch();
  KF_CUDA(cudaGetLastError());
  if (keep) {
    KF_CUDA(cudaMemsetAsync(keep, 0, size_t(n), st));
    keep_mask_kernel<<<grid_cap(n, 256), 256, 0, st>>>(src, b.kcount, keep); note_launch();
    KF_CUDA(cudaGetLastError());
  }
  finish_kernel<<<1, 1, 0, st>>>(src, b.prefix, n, b.kcount, cut, (long long*)used); note_launch();
  return check_cuda(cudaGetLastError(), "allocation launch");
}

// ------------------------------------------------------------------------------------
// Allocation-free variant of score_and_allocate.  Its scratch (sort keys, digit
// histograms, prefix sums) lives in one file-scope device array instead of a caller
// workspace, so neither the library nor the caller allocates device memory for the call.
// The array is sized for NOALLOC_MAX_COMPONENTS components and stays resident on every
// GPU that loads the library until the process exits.
namespace {
constexpr int64_t NOALLOC_MAX_COMPONENTS = int64_t(1) << 20;
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(25) << 20;  // >= alloc_workspace(1 << 20, 0)
constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};
}  // namespace

}  // namespace kf

// Scratch of score_and_allocate_noalloc (file scope, internal linkage).
static __device__ __align__(256) unsigned char g_alloc_scratch[kf::NOALLOC_SCRATCH_BYTES];

namespace kf {

// Device address of g_alloc_scratch on `device`, looked up once per device with that device
// current (host code only sees a host-side stand-in for the symbol).
static kf_status noalloc_scratch(int device, void** out) {
  if (device < 0 || device >= NOALLOC_MAX_DEVICES) return fail(KF_ERR_UNSUPPORTED, "score_and_allocate_noalloc: device index");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[device]) {
    if (alloc_workspace(NOALLOC_MAX_COMPONENTS, 0) > NOALLOC_SCRATCH_BYTES)
      return fail(KF_ERR_UNSUPPORTED, "score_and_allocate_noalloc: static scratch smaller than its stated maximum");
    int prev = 0;
    KF_CUDA(cudaGetDevice(&prev));
    if (prev != device) KF_CUDA(cudaSetDevice(device));
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_alloc_scratch);
    if (prev != device) cudaSetDevice(prev);
    if (e != cudaSuccess || !p) return check_cuda(e != cudaSuccess ? e : cudaErrorInvalidSymbol, "cudaGetSymbolAddress(scratch)");
    g_noalloc_ptr[device] = p;
  }
  *out = g_noalloc_ptr[device];
  return KF_OK;
}

}  // namespace kf

extern "C" kf_status score_and_allocate_noalloc(kf_ctx* ctx, const float* sigma, const int64_t* seg_offset,
                                                const int64_t* cost, int32_t n_units, int64_t n_components,
                                                int64_t budget, kf_alloc_mode mode, const int32_t* fixed_rank,
                                                int32_t* ranks, float* cut, int64_t* used, kf_stream_t stream) {
  using namespace kf;
  if (!ctx) return fail(KF_ERR_INVALID, "score_and_allocate_noalloc: null context");
  if (n_units <= 0 || n_components < 0) return fail(KF_ERR_INVALID, "score_and_allocate_noalloc: sizes");
  if (n_components > NOALLOC_MAX_COMPONENTS)
    return fail(KF_ERR_UNSUPPORTED, "score_and_allocate_noalloc: at most 1048576 components (static scratch limit); "
                                    "use score_and_allocate with a workspace for more");
  if (!seg_offset || !cost || !ranks) return fail(KF_ERR_INVALID, "score_and_allocate_noalloc: null pointer");
  if (mode != KF_KEY_HALF_SIGMA2 && mode != KF_KEY_PER_PARAM && mode != KF_FIXED_RANK)
    return fail(KF_ERR_INVALID, "score_and_allocate_noalloc: mode");
  if (mode == KF_FIXED_RANK && !fixed_rank) return fail(KF_ERR_INVALID, "score_and_allocate_noalloc: fixed_rank is null");
  if (mode != KF_FIXED_RANK && !sigma && n_components > 0)
    return fail(KF_ERR_INVALID, "score_and_allocate_noalloc: sigma is null");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (mode != KF_FIXED_RANK && n_components == 0) {
    KF_CUDA(cudaMemsetAsync(ranks, 0, sizeof(int32_t) * size_t(n_units), st));
    if (used) KF_CUDA(cudaMemsetAsync(used, 0, sizeof(int64_t), st));
    if (cut) KF_CUDA(cudaMemsetAsync(cut, 0xFF, 2 * sizeof(float), st));
    return KF_OK;
  }
  void* scratch = nullptr;
  KF_TRY(noalloc_scratch(ctx->device, &scratch));
  return alloc_run(ctx, sigma, seg_offset, cost, n_units, n_components, budget, mode, fixed_rank, nullptr, ranks, cut,
                   used, scratch, NOALLOC_SCRATCH_BYTES, st, nullptr, 0.0);
}
