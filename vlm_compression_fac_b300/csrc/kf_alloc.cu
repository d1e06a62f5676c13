// Global sort-and-truncate rank allocation (UniRank 2.1; LASER Methodology 2).
//   keys:  k = (~bits(score) << 32) | component id, score = 0.5f * (sigma * sigma) [/ cost],
//          or UniRank's energy ratio sigma^2 / sum_unit sigma^2, optionally times a per-unit
//          weight (UniRank's layer importance I_l);
//          ascending k is score descending, then lower unit, then lower component index
//          (ids are assigned in unit order), which makes the order total and deterministic;
//   sort:  LSD radix sort of the score word, 4 passes of 8 bits (equal scores keep their id
//          order, since the keys start in id order and every pass is stable).  The digit
//          counts of all four passes are taken while the keys are built; each pass is then a
//          single kernel over 4096-key tiles taken in launch order: a tile counts its digits,
//          publishes the counts, adds up the counts of the tiles before it (decoupled
//          look-back) and scatters its keys stably (warp match and per-warp digit counters keep
//          the original order inside the tile) through a digit-ordered copy in shared memory;
//   cut:   inclusive prefix sum of the kept pairs' cost m+n in sorted order, by one look-back
//          scan; the kept prefix is every position whose prefix sum is <= budget (costs are
//          non-negative, so it is a prefix), found by the tile that holds its end; ranks =
//          kept count per unit.
// Every wait of a look-back is bounded: a tile that has not published within the context's
// wait limit records KF_ERR_TIMEOUT and is counted as empty, so no launch can hang.
#include "kf_internal.cuh"
#include "kf_tc_ptx.cuh"

#include <mutex>

namespace kf {
namespace {

constexpr int RT = 256;            // threads per tile
constexpr int RI = 16;             // keys per thread
constexpr int TILE = RT * RI;      // 4096 keys per tile
constexpr int WK = TILE / (RT / 32);  // keys of one warp's contiguous run in a tile

__device__ __forceinline__ int unit_of(const int64_t* __restrict__ off, int n_units, int64_t g) {
  int lo = 0, hi = n_units;  // off[lo] <= g < off[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= g) lo = mid; else hi = mid;
  }
  return lo;
}
// Every CTA of the key builders takes one contiguous range of components (a multiple of 256
// long) and walks it in steps of its 256 threads; a thread's unit only moves forward, so
// after one binary search for its first component each step costs at most a few compares.
__device__ __forceinline__ void chunk_range(int64_t n, int64_t& beg, int64_t& end) {
  int64_t chunk = (n + gridDim.x - 1) / gridDim.x;
  chunk = (chunk + 255) & ~int64_t(255);
  beg = int64_t(blockIdx.x) * chunk;
  end = beg + chunk < n ? beg + chunk : n;
}
__device__ __forceinline__ int advance_unit(const int64_t* __restrict__ off, int n_units, int u, int64_t g) {
  while (u + 1 < n_units && off[u + 1] <= g) ++u;
  return u;
}

// Key of every component: base score per mode (KF_KEY_HALF_SIGMA2: 0.5 sigma^2;
// KF_KEY_PER_PARAM: that divided by the unit's m + n; KF_KEY_ENERGY_RATIO: sigma^2 divided
// by the unit's energy sum sigma^2), times the unit's weight when weights are given (a
// weight that is negative or not a number counts as 0).  float32, one rounding per operation.
constexpr int MODE_GIVEN_KEYS = 100;  // internal: the caller's keys, as given
constexpr int MODE_SWIFT_HYBRID = 101;  // internal: Swift-SVD B hybrid keys built from sigma

// Score word of one component (~bits of its float32 score): the same function builds the
// sort keys and, for the modes whose keys never increase along a unit, counts each unit's
// kept prefix after the cut.
__device__ __forceinline__ unsigned score_word(float s, int u, int mode, const int64_t* __restrict__ cost,
                                               const float* __restrict__ weight,
                                               const float* __restrict__ energy) {
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
  return ~__float_as_uint(sc);
}

// The low word of a key is the component id, or, when no caller needs ids (no keep mask), the
// unit index: the sort orders by the score word only and is stable, so equal scores stay in
// id order either way, and every later pass needs only the unit (its cost, its rank count).
// The kernel also counts the four 8-bit digits of the score words (ghist[pass][digit]) for
// the radix passes: consecutive lanes hold consecutive components, whose digits come in runs
// (a unit's scores are sorted), so each run of equal digits in a warp is added once.
__global__ void __launch_bounds__(256) build_keys_kernel(const float* __restrict__ sigma,
                                                         const int64_t* __restrict__ off,
                                                         const int64_t* __restrict__ cost, int n_units, int64_t n,
                                                         int mode, const float* __restrict__ weight,
                                                         const float* __restrict__ energy,
                                                         unsigned long long* __restrict__ keys, int low_is_unit,
                                                         unsigned* __restrict__ ghist) {
  __shared__ unsigned h[4 * 256];
  for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  int64_t beg, end;
  chunk_range(n, beg, end);
  int u = beg + threadIdx.x < n ? unit_of(off, n_units, beg + threadIdx.x) : 0;
  constexpr int BK_UNROLL = 4;   // components per thread and step, their loads issued together
  for (int64_t g0 = beg; g0 < end; g0 += BK_UNROLL * 256) {   // the same trip count for the whole CTA
    float sv[BK_UNROLL];
#pragma unroll
    for (int i = 0; i < BK_UNROLL; ++i) {
      const int64_t g = g0 + i * 256 + threadIdx.x;
      sv[i] = g < end ? sigma[g] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < BK_UNROLL; ++i) {
      const int64_t g = g0 + i * 256 + threadIdx.x;
      const bool valid = g < end;
      unsigned bits = 0;
      if (valid) {
        u = advance_unit(off, n_units, u, g);
        bits = score_word(sv[i], u, mode, cost, weight, energy);
        const uint32_t low = low_is_unit ? uint32_t(u) : uint32_t(g);
        keys[g] = (static_cast<unsigned long long>(bits) << 32) | static_cast<unsigned long long>(low);
      }
      const unsigned vmask = __ballot_sync(0xffffffffu, valid);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const unsigned d = (bits >> (8 * b)) & 255u;
        const unsigned prev = __shfl_up_sync(0xffffffffu, d, 1);
        const bool head = valid && (lane == 0 || d != prev);
        const unsigned ends = __ballot_sync(0xffffffffu, head) | ~vmask;  // a run ends at the next head
        if (head) {
          const unsigned above = ends & ~((2u << lane) - 1u);
          const int nxt = above ? __ffs(int(above)) - 1 : 32;
          atomicAdd(&h[b * 256 + int(d)], unsigned(nxt - lane));
        }
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x)
    if (h[i]) atomicAdd(&ghist[i], h[i]);
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
  int64_t beg, end;
  chunk_range(n, beg, end);
  int u = beg + threadIdx.x < n ? unit_of(off, n_units, beg + threadIdx.x) : 0;
  for (int64_t g = beg + threadIdx.x; g < end; g += blockDim.x) {
    u = advance_unit(off, n_units, u, g);
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

// Exclusive scan of each pass's 256 digit counts: gbase[pass][d] = the first sorted position
// of digit d in that pass.  One CTA of 256 threads per pass.
__global__ void __launch_bounds__(256) digit_base_kernel(const unsigned* __restrict__ ghist,
                                                         unsigned* __restrict__ gbase) {
  __shared__ unsigned wsum[8];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const unsigned v = ghist[blockIdx.x * 256 + t];
  unsigned x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  unsigned pre = 0;
  for (int ww = 0; ww < w; ++ww) pre += wsum[ww];
  gbase[blockIdx.x * 256 + t] = pre + x - v;
}

// Look-back status words, one per (tile, slot): bits 63..62 flag (1: the tile's own count,
// 2: the inclusive sum through the tile), bits 61..56 the tag of the pass that wrote it (the
// words are cleared once per call and reused by the passes), bits 55..0 the value.
constexpr unsigned long long LB_OWN = 1ull << 62, LB_INCL = 2ull << 62;
constexpr unsigned long long LB_VAL = (1ull << 56) - 1;
__device__ __forceinline__ void lb_store(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long lb_load(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Sum of one slot's values over the tiles before `tile` (status word of tile k at
// st[k * stride]): walks back adding own counts until a tile's inclusive sum is found,
// reading the words of LB_WIN predecessors at a time.  Tiles take their numbers in launch
// order, so every tile waited on is held by a CTA that is already running; each wait is
// still bounded by wait_ns (then KF_ERR_TIMEOUT is recorded and the tile counted as empty).
constexpr int LB_WIN = 8;
__device__ unsigned long long lookback(const unsigned long long* st, int64_t stride, int tile,
                                       unsigned long long tag, unsigned long long wait_ns, int* status) {
  unsigned long long acc = 0;
  int k = tile - 1;
  unsigned long long t0 = 0;
  while (k >= 0) {
    unsigned long long w[LB_WIN];
#pragma unroll
    for (int i = 0; i < LB_WIN; ++i) w[i] = k - i >= 0 ? lb_load(st + int64_t(k - i) * stride) : 0ull;
    int used = 0;
    bool found = false;
#pragma unroll
    for (int i = 0; i < LB_WIN; ++i) {
      if (found || used < i || k - i < 0) continue;       // stop at the first gap
      const bool ready = (w[i] >> 62) != 0 && (w[i] & (63ull << 56)) == tag;
      if (!ready) continue;
      acc += w[i] & LB_VAL;
      used = i + 1;
      found = (w[i] >> 62) == 2;
    }
    if (found) break;
    if (used > 0) {
      k -= used;
      t0 = 0;
      continue;
    }
    const unsigned long long now = now_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > wait_ns) {
      raise_status(status, KF_ERR_TIMEOUT, WAIT_LOOKBACK);
      --k;
      t0 = 0;
      continue;
    }
    __nanosleep(64);
  }
  return acc;
}

// lookback() for one slot per tile, by a whole warp: lane i reads the word of tile k - i, so
// 32 predecessors are examined per round trip; the nearest inclusive sum ends the walk when
// every nearer tile has published.  Every lane returns the same sum.
__device__ unsigned long long warp_lookback(const unsigned long long* st, int tile, unsigned long long tag,
                                            unsigned long long wait_ns, int* status, int lane) {
  unsigned long long acc = 0;
  int k = tile - 1;
  unsigned long long t0 = 0;
  while (k >= 0) {
    const int kk = k - lane;
    const unsigned long long w = kk >= 0 ? lb_load(st + kk) : (LB_INCL | tag);  // before tile 0: sum 0
    const bool ready = (w >> 62) != 0 && (w & (63ull << 56)) == tag;
    const bool incl = ready && (w >> 62) == 2;
    const unsigned notready = __ballot_sync(0xffffffffu, !ready);
    const unsigned inclm = __ballot_sync(0xffffffffu, incl);
    const int first_gap = notready ? __ffs(int(notready)) - 1 : 32;
    const int first_incl = inclm ? __ffs(int(inclm)) - 1 : 32;
    if (first_incl < first_gap) {          // lanes 0 .. first_incl all published: done
      unsigned long long v = (lane <= first_incl && kk >= 0) ? (w & LB_VAL) : 0ull;
#pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      return acc + v;
    }
    if (first_gap > 0) {                   // own counts of lanes 0 .. first_gap - 1, go on
      unsigned long long v = lane < first_gap ? (w & LB_VAL) : 0ull;
#pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc += v;
      k -= first_gap;
      t0 = 0;
      continue;
    }
    const unsigned long long now = now_ns();   // the nearest predecessor has not published
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > wait_ns) {
      if (lane == 0) raise_status(status, KF_ERR_TIMEOUT, WAIT_LOOKBACK);
      --k;
      t0 = 0;
      continue;
    }
    __nanosleep(64);
  }
  return acc;
}

// The lanes of the warp holding the same 8-bit digit as this lane (itself included; invalid
// lanes never count): eight ballots, one per bit of the digit.
__device__ __forceinline__ unsigned digit_peers(unsigned d, bool valid) {
  unsigned peers = __ballot_sync(0xffffffffu, valid);
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const bool bit = (d >> b) & 1u;
    const unsigned m = __ballot_sync(0xffffffffu, bit);
    peers &= bit ? m : ~m;
  }
  return peers;
}

// One radix pass over the score word's byte `pass`, one 4096-key tile per CTA (tile number
// from a counter, in launch order).  Warp w owns the tile's keys w * WK .. w * WK + WK - 1
// (the warp's round r holds keys w * WK + 32 r + lane), so the tile's index order is (warp,
// round, lane) order.  All keys are loaded first; phase 1 counts each warp's keys per digit
// (one counter update per distinct digit of a round, the lanes of equal digits found by
// ballots over the digit's bits); the tile's counts are
// published and the counts of the tiles before it summed by look-back (thread d for digit d);
// phase 2 puts every key at its warp's running position for its digit in the tile's
// digit-ordered copy in shared memory, plus its rank among the round's equal digits; the copy
// is then written out at gbase[d] + (keys of digit d in earlier tiles) + (rank in the tile),
// consecutive threads on consecutive addresses of one digit's run (coalesced).
__global__ void __launch_bounds__(RT, 3) onesweep_kernel(const unsigned long long* __restrict__ in,
                                                         unsigned long long* __restrict__ out, int64_t n, int pass,
                                                         const unsigned* __restrict__ gbase,
                                                         unsigned long long* __restrict__ lbst,
                                                         unsigned* __restrict__ tile_ctr, int* status,
                                                         unsigned long long wait_ns) {
  __shared__ unsigned start[256];   // the digit's first position in the tile's ordered copy
  __shared__ unsigned gpos[256];    // the digit's first position in the output
  __shared__ unsigned wpos[RT / 32][256];   // per-warp digit counts, then running positions
  __shared__ unsigned long long tk[TILE];
  __shared__ unsigned wsum[RT / 32];
  __shared__ int tile_s;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  if (t == 0) tile_s = int(atomicAdd(tile_ctr, 1u));
  for (int x = lane; x < 256; x += 32) wpos[w][x] = 0;
  __syncthreads();
  const int tile = tile_s;
  const int shift = 32 + 8 * pass;
  const int64_t tile0 = int64_t(tile) * TILE;
  const int tile_n = int(n - tile0 < TILE ? n - tile0 : TILE);
  unsigned long long key[RI];
#pragma unroll
  for (int r = 0; r < RI; ++r) {
    const int li = w * WK + r * 32 + lane;
    key[r] = li < tile_n ? in[tile0 + li] : 0ull;
  }
  unsigned peers[RI];
#pragma unroll
  for (int r = 0; r < RI; ++r) {
    const bool valid = w * WK + r * 32 + lane < tile_n;
    const unsigned d = unsigned((key[r] >> shift) & 255u);
    peers[r] = digit_peers(d, valid);
    if (valid && (peers[r] & lt_mask) == 0u) wpos[w][d] += __popc(peers[r]);
    __syncwarp();
  }
  __syncthreads();
  // thread t = digit t: the tile's count, published at once; then its place in the tile
  unsigned cnt = 0;
#pragma unroll
  for (int ww = 0; ww < RT / 32; ++ww) cnt += wpos[ww][t];
  const unsigned long long tag = (unsigned long long)(pass + 1) << 56;
  unsigned long long* mine = lbst + int64_t(tile) * 256 + t;
  lb_store(mine, (tile == 0 ? LB_INCL : LB_OWN) | tag | cnt);
  {
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
    unsigned acc = start[t];
#pragma unroll
    for (int ww = 0; ww < RT / 32; ++ww) {
      const unsigned c = wpos[ww][t];
      wpos[ww][t] = acc;
      acc += c;
    }
  }
  unsigned long long before = 0;
  if (tile > 0) {
    before = lookback(lbst + t, 256, tile, tag, wait_ns, status);
    lb_store(mine, LB_INCL | tag | (before + cnt));
  }
  gpos[t] = gbase[pass * 256 + t] + unsigned(before);
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
    out[gpos[d] + (unsigned(i) - start[d])] = k;
  }
}

__device__ __forceinline__ int key_unit(unsigned long long k, const int64_t* __restrict__ off, int n_units,
                                        int low_is_unit) {
  return low_is_unit ? int(uint32_t(k)) : unit_of(off, n_units, int64_t(uint32_t(k)));
}
__device__ __forceinline__ float key_score(unsigned long long k) { return __uint_as_float(~unsigned(k >> 32)); }

// The cost prefix and the cut in one pass over the sorted keys: tile = 4096 keys (16
// consecutive per thread), the tile's cost total published and the totals of the tiles
// before it summed by look-back.  The kept prefix is every position whose inclusive cost
// prefix is <= budget; the one tile whose range of prefixes contains the budget (or the last
// tile when everything fits, or the first when the budget is negative) writes its length
// (kcount), the cost it uses and the scores on both sides of the cut.
__global__ void __launch_bounds__(RT) cost_scan_kernel(const unsigned long long* __restrict__ keys,
                                                       const int64_t* __restrict__ off,
                                                       const int64_t* __restrict__ cost, int n_units, int64_t n,
                                                       long long budget, int low_is_unit,
                                                       unsigned long long* __restrict__ lbst,
                                                       unsigned* __restrict__ tile_ctr,
                                                       unsigned long long* __restrict__ kcount, float* __restrict__ cut,
                                                       long long* __restrict__ used, int* status,
                                                       unsigned long long wait_ns) {
  __shared__ long long wsum[RT / 32];
  __shared__ long long excl_s;
  __shared__ int tile_s;
  __shared__ int kept_w[RT / 32];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  if (t == 0) tile_s = int(atomicAdd(tile_ctr, 1u));
  __syncthreads();
  const int tile = tile_s;
  const int64_t tile0 = int64_t(tile) * TILE;
  const int64_t g0 = tile0 + int64_t(t) * RI;
  long long c[RI];
  long long sum = 0;
  if (g0 + RI <= n) {  // 16 consecutive keys: eight 16-byte loads
    const ulonglong2* kv = reinterpret_cast<const ulonglong2*>(keys + g0);
    ulonglong2 kk[RI / 2];
#pragma unroll
    for (int i = 0; i < RI / 2; ++i) kk[i] = kv[i];
#pragma unroll
    for (int i = 0; i < RI / 2; ++i) {
      c[2 * i] = cost[key_unit(kk[i].x, off, n_units, low_is_unit)];
      c[2 * i + 1] = cost[key_unit(kk[i].y, off, n_units, low_is_unit)];
    }
  } else {
#pragma unroll
    for (int i = 0; i < RI; ++i) {
      const int64_t g = g0 + i;
      c[i] = g < n ? cost[key_unit(keys[g], off, n_units, low_is_unit)] : 0;
    }
  }
#pragma unroll
  for (int i = 0; i < RI; ++i) sum += c[i];
  // exclusive scan of the thread sums over the tile
  long long x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  long long pre = 0, total = 0;
  for (int ww = 0; ww < RT / 32; ++ww) {
    if (ww < w) pre += wsum[ww];
    total += wsum[ww];
  }
  const long long texcl = pre + x - sum;
  if (w == 0) {   // warp 0: publish, then look back 32 predecessors per round trip
    unsigned long long* mine = lbst + tile;
    const unsigned long long tag = 1ull << 56;
    if (lane == 0) lb_store(mine, (tile == 0 ? LB_INCL : LB_OWN) | tag | (unsigned long long)total);
    const long long e = tile > 0 ? (long long)warp_lookback(lbst, tile, tag, wait_ns, status, lane) : 0;
    if (lane == 0) {
      if (tile > 0) lb_store(mine, LB_INCL | tag | (unsigned long long)(e + total));
      excl_s = e;
    }
  }
  __syncthreads();
  const long long E = excl_s;
  const int64_t tile_end = tile0 + TILE < n ? tile0 + TILE : n;
  const bool writer = (E <= budget && budget < E + total) || (tile == 0 && budget < 0) ||
                      (tile_end == n && E + total <= budget);   // uniform over the CTA
  if (!writer) return;
  // kept items of this tile (a prefix of it: the prefix sums do not decrease)
  int k_t = 0;
  long long run = E + texcl, last_incl = E + texcl;
#pragma unroll
  for (int i = 0; i < RI; ++i) {
    run += c[i];
    if (g0 + i < n && run <= budget) {
      ++k_t;
      last_incl = run;
    }
  }
  int kw = k_t;
#pragma unroll
  for (int o = 16; o; o >>= 1) kw += __shfl_xor_sync(0xffffffffu, kw, o);
  if (lane == 0) kept_w[w] = kw;
  __syncthreads();
  int K = 0;
  for (int ww = 0; ww < RT / 32; ++ww) K += kept_w[ww];
  const int64_t kc = tile0 + K;
  // the thread holding the last kept item reports the cost used
  if (K > 0 && t == (K - 1) / RI && used) *used = last_incl;
  if (t == 0) {
    if (K == 0 && used) *used = E;
    *kcount = static_cast<unsigned long long>(kc);
    if (cut) {
      cut[0] = kc > 0 ? key_score(keys[kc - 1]) : __int_as_float(0x7fc00000);
      cut[1] = kc < n ? key_score(keys[kc]) : __int_as_float(0x7fc00000);
    }
  }
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

// ranks[u] for keys that never increase along a unit (the sigma-based keys, sigma being in
// descending order, and the hybrid keys) without reading the kept keys: the kept components
// of unit u are its leading ones whose key sorts before the last kept key K* =
// sorted[kcount - 1] (key order: score word, then unit), plus, in K*'s own unit, the kept
// ones among the components equal to K* (equal keys of one unit keep their id order, and the
// first kcount - first(K*) of them are kept).  One thread per unit, a binary search over the
// unit's score words recomputed by the same function that built the keys.
__global__ void ranks_search_kernel(const float* __restrict__ x, const int64_t* __restrict__ off,
                                    const int64_t* __restrict__ cost, int n_units, int mode,
                                    const float* __restrict__ weight, const float* __restrict__ energy,
                                    const unsigned long long* __restrict__ sorted, int64_t n,
                                    const unsigned long long* __restrict__ kcount, int* __restrict__ ranks) {
  __shared__ unsigned long long kstar_s;
  __shared__ long long eq_s;
  if (threadIdx.x == 0) {
    const int64_t kc = int64_t(*kcount);
    if (kc == 0) {
      eq_s = -1;
    } else {
      const unsigned long long ks = sorted[kc - 1];
      int64_t lo = 0, hi = kc - 1;  // first position holding ks
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (sorted[mid] < ks) lo = mid + 1; else hi = mid;
      }
      kstar_s = ks;
      eq_s = kc - lo;
    }
  }
  __syncthreads();
  const long long eq = eq_s;
  if (eq < 0) return;  // nothing kept: the ranks were cleared before
  const unsigned hw = unsigned(kstar_s >> 32);
  const int us = int(uint32_t(kstar_s));
  for (int u = blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += gridDim.x * blockDim.x) {
    int64_t a = off[u], b = off[u + 1];
    const int64_t base = a;
    while (a < b) {   // first component that is not kept by its score word
      const int64_t mid = (a + b) >> 1;
      const unsigned wd = score_word(x[mid], u, mode, cost, weight, energy);
      const bool kept = u < us ? wd <= hw : wd < hw;
      if (kept) a = mid + 1; else b = mid;
    }
    ranks[u] = int(a - base + (u == us ? eq : 0));
  }
}

// keep[id] = 1 for the components of the kept prefix (the mask was cleared before).
__global__ void keep_mask_kernel(const unsigned long long* __restrict__ keys,
                                 const unsigned long long* __restrict__ kcount, unsigned char* __restrict__ keep) {
  const int64_t k = int64_t(*kcount);
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < k; i += int64_t(gridDim.x) * blockDim.x)
    keep[uint32_t(keys[i])] = 1;
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
  unsigned long long *lbst, *lbst2;       // look-back words of the radix passes and of the cost scan
  unsigned *ghist, *gbase, *ctr;          // digit counts, digit bases, tile counters (4 passes + scan)
  float* aux;                             // Swift hybrid keys before they become sort keys
  float* energy;
  unsigned char *clear0, *clear1;         // [clear0, clear1) is zeroed once per call
};

// n_energy: units whose energy is needed (KF_KEY_ENERGY_RATIO), else 0.
size_t alloc_carve(Carve& cv, int64_t n, int64_t n_energy, AllocBufs& b) {
  const int64_t ntiles = (n + TILE - 1) / TILE;
  const int64_t nt = ntiles > 0 ? ntiles : 1;
  b.ka = cv.take<unsigned long long>(n > 0 ? n : 1);
  b.kb = cv.take<unsigned long long>(n > 0 ? n : 1);
  b.lbst = cv.take<unsigned long long>(size_t(256) * nt);
  b.clear0 = reinterpret_cast<unsigned char*>(b.lbst);
  b.lbst2 = cv.take<unsigned long long>(size_t(nt));
  b.ghist = cv.take<unsigned>(4 * 256);
  b.ctr = cv.take<unsigned>(8);
  b.kcount = cv.take<unsigned long long>(1);   // cleared too: 0 unless the cost scan sets it
  b.clear1 = reinterpret_cast<unsigned char*>(b.kcount + 1);
  b.gbase = cv.take<unsigned>(4 * 256);
  b.aux = cv.take<float>(n > 0 ? n : 1);
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
  KF_CUDA(cudaMemsetAsync(b.clear0, 0, size_t(b.clear1 - b.clear0), st));
  if (mode == KF_KEY_ENERGY_RATIO) {
    unit_energy_kernel<<<unsigned(n_units), 256, 0, st>>>(sigma, off, b.energy); note_launch();
    KF_CUDA(cudaGetLastError());
  }
  if (int(mode) == MODE_SWIFT_HYBRID) {
    // eps (float64) in the second key buffer, free until the first radix pass
    double* eps = reinterpret_cast<double*>(b.kb);
    swift_eps_kernel<<<unsigned((n_units + 127) / 128), 128, 0, st>>>(sigma, off, n_units, eps); note_launch();
    KF_CUDA(cudaGetLastError());
    swift_keys_kernel<<<grid_cap(n, 256), 256, 0, st>>>(eps, off, n_units, n, weight, alpha, b.aux); note_launch();
    KF_CUDA(cudaGetLastError());
    build_keys_kernel<<<grid_cap(n, 256), 256, 0, st>>>(b.aux, off, cost, n_units, n, MODE_GIVEN_KEYS, nullptr,
                                                        nullptr, b.ka, low_is_unit, b.ghist); note_launch();
  } else {
    build_keys_kernel<<<grid_cap(n, 256), 256, 0, st>>>(sigma, off, cost, n_units, n, int(mode), weight, b.energy,
                                                        b.ka, low_is_unit, b.ghist); note_launch();
  }
  KF_CUDA(cudaGetLastError());
  digit_base_kernel<<<4, 256, 0, st>>>(b.ghist, b.gbase); note_launch();
  KF_CUDA(cudaGetLastError());
  // The keys are built in id order and every pass is stable, so sorting by the score word
  // alone (the upper 32 bits, four 8-bit passes) leaves equal scores in id order: the same
  // total order as sorting all 64 bits, at half the passes.
  unsigned long long* src = b.ka;
  unsigned long long* dst = b.kb;
  for (int pass = 0; pass < 4; ++pass) {
    onesweep_kernel<<<ntiles, RT, 0, st>>>(src, dst, n, pass, b.gbase, b.lbst, b.ctr + pass, ctx->d_status,
                                           WAIT_LIMIT_NS); note_launch();
    KF_CUDA(cudaGetLastError());
    unsigned long long* tmp = src;
    src = dst;
    dst = tmp;
  }
  // src now holds the sorted keys.
  cost_scan_kernel<<<ntiles, RT, 0, st>>>(src, off, cost, n_units, n, budget, low_is_unit, b.lbst2, b.ctr + 4,
                                          b.kcount, cut, (long long*)used, ctx->d_status, WAIT_LIMIT_NS);
  note_launch();
  KF_CUDA(cudaGetLastError());
  // ranks: by a search per unit where its keys never increase along the unit (the ids are
  // not needed and the keys come from sigma or from the hybrid score), else by counting
  // the kept keys
  const bool monotone = low_is_unit && (mode == KF_KEY_HALF_SIGMA2 || mode == KF_KEY_PER_PARAM ||
                                        mode == KF_KEY_ENERGY_RATIO || int(mode) == MODE_SWIFT_HYBRID);
  if (monotone) {
    const bool hyb = int(mode) == MODE_SWIFT_HYBRID;
    ranks_search_kernel<<<unsigned((n_units + 255) / 256), 256, 0, st>>>(
        hyb ? b.aux : sigma, off, cost, n_units, hyb ? MODE_GIVEN_KEYS : int(mode), hyb ? nullptr : weight,
        hyb ? nullptr : b.energy, src, n, b.kcount, ranks); note_launch();
  } else {
    const size_t rsmem = n_units <= RANKS_SMEM_UNITS ? sizeof(int) * size_t(n_units > 0 ? n_units : 1) : 0;
    ranks_kernel<<<grid_cap(n, 256), 256, rsmem, st>>>(src, off, n_units, b.kcount, ranks, low_is_unit);
    note_launch();
  }
  KF_CUDA(cudaGetLastError());
  if (keep) {
    KF_CUDA(cudaMemsetAsync(keep, 0, size_t(n), st));
    keep_mask_kernel<<<grid_cap(n, 256), 256, 0, st>>>(src, b.kcount, keep); note_launch();
    KF_CUDA(cudaGetLastError());
  }
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
