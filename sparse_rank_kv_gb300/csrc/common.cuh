// Device helpers shared by the ShadowKV kernels: element conversion, 16-byte
// vector access, RoPE angles, block-wide scans and the radix top-k select.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace skv {

typedef __nv_bfloat16 bf16;

// status-word codes written by kernels that find an out-of-range index
enum : int {
  DEV_OK = 0,
  DEV_BAD_CHUNK = 1,
  DEV_BAD_SLOT = 2,
  DEV_BAD_OUTLIER = 3,
  DEV_BAD_COUNT = 4,
  DEV_TIMEOUT = 5,      // a bounded mbarrier wait gave up
  DEV_NUMERIC = 6,      // the SVD's orthonormalisation met a non-positive pivot
};

// Nanoseconds a bounded mbarrier wait lasts before a kernel gives up and
// reports DEV_TIMEOUT (every legitimate wait is microseconds).
constexpr unsigned long long kWaitLimit = 2000000000ull;

__device__ __forceinline__ void flag_error(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------ elements
template <typename T> struct Ty;
template <> struct Ty<float> {
  static constexpr int kVec = 4;  // elements per 16 bytes
  __device__ __forceinline__ static float to_f(float x) { return x; }
  __device__ __forceinline__ static float from_f(float x) { return x; }
  // 16 bytes at p -> 4 floats
  __device__ __forceinline__ static void load16(const float* p, float* o) {
    float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  __device__ __forceinline__ static void load16_cg(const float* p, float* o) {
    float4 v = __ldcg(reinterpret_cast<const float4*>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
};
template <> struct Ty<bf16> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float to_f(bf16 x) { return __bfloat162float(x); }
  __device__ __forceinline__ static bf16 from_f(float x) { return __float2bfloat16_rn(x); }
  __device__ __forceinline__ static void unpack(uint4 v, float* o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static void load16(const bf16* p, float* o) {
    unpack(*reinterpret_cast<const uint4*>(p), o);
  }
  __device__ __forceinline__ static void load16_cg(const bf16* p, float* o) {
    unpack(__ldcg(reinterpret_cast<const uint4*>(p)), o);
  }
};

// ------------------------------------------------------------ RoPE angles
// Rotate-half RoPE turns dimension pair (i, i + d/2) by pos * inv_freq_i
// radians.  tab[i] = (hi, lo) with hi + lo = inv_freq_i / (2 pi) to about
// 48 bits (computed on the host in double).  The product pos * hi is split
// exactly into (prod, err) by an FMA, the integer part of prod is dropped
// exactly, and the remaining fraction of a turn goes to sincospif, so the
// angle stays accurate to ~1e-7 rad at positions up to 2^24.
__device__ __forceinline__ void rope_sincos(int pos, float2 f, float* sn, float* cs) {
  const float p = static_cast<float>(pos);
  const float prod = p * f.x;
  const float err = fmaf(p, f.x, -prod);
  const float frac = prod - rintf(prod);
  const float turns = frac + (err + p * f.y);
  sincospif(2.0f * turns, sn, cs);
}

// Same angle, evaluated with the hardware sine/cosine on the reduced angle in
// [-pi, pi] (absolute error about 4e-7): the form used by hot epilogues.
__device__ __forceinline__ void rope_sincos_fast(int pos, float2 f, float* sn, float* cs) {
  const float p = static_cast<float>(pos);
  const float prod = p * f.x;
  const float err = fmaf(p, f.x, -prod);
  const float frac = prod - rintf(prod);
  const float turns = frac + (err + p * f.y);
  __sincosf(turns * 6.283185307179586f, sn, cs);
}

// ------------------------------------------------------ tiled value rows
// Values of bf16 contexts with d = 128 are stored in 8-token groups laid out
// as the tensor core's no-swizzle K-major tiles of V^T: element (token t,
// dimension j) of a group at (j/8)*64 + (j%8)*8 + t.  transpose8x8 turns the
// row-major group held by a half-warp -- lane q holds the 16-byte piece q
// (dimensions 8q..8q+7) of rows 0..7 in in[t] -- into the tiled group: out[r]
// = the 8 tokens of dimension 8q + r, stored at 16-byte unit 8q + r.
__device__ __forceinline__ void transpose8x8(const uint4 (&in)[8], uint4 (&out)[8]) {
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    uint32_t e[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t w = (r >> 1) == 0 ? in[t].x : (r >> 1) == 1 ? in[t].y : (r >> 1) == 2 ? in[t].z : in[t].w;
      e[t] = (r & 1) ? (w >> 16) : (w & 0xffffu);
    }
    out[r] = make_uint4(e[0] | (e[1] << 16), e[2] | (e[3] << 16), e[4] | (e[5] << 16), e[6] | (e[7] << 16));
  }
}
// Offset of element (row t, dimension j) of a tiled [rows][128] block whose
// 8-row groups start at multiples of 8 rows.
__host__ __device__ __forceinline__ size_t vt_off(size_t t, int j) {
  return (t >> 3) * 1024 + static_cast<size_t>(j >> 3) * 64 + (j & 7) * 8 + (t & 7);
}

// ------------------------------------------------------------ reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide exclusive scan of one int per thread.  `tmp` holds >= 32 ints of
// shared memory.  Returns the exclusive prefix; *total gets the block sum.
// Every thread of the block must call it.  One barrier: every warp scans the
// per-warp totals itself.
// With last_use, tmp is not written again before the block's next barrier,
// and the scan skips its closing barrier.
__device__ __forceinline__ int block_exclusive_scan(int v, int* tmp, int* total, bool last_use = false) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  int w = lane < nwarps ? tmp[lane] : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, w, o);
    if (lane >= o) w += y;
  }
  // w: inclusive totals of warps 0..lane
  const int before = __shfl_sync(0xffffffffu, w, warp > 0 ? warp - 1 : 0);
  const int excl = (warp ? before : 0) + x - v;
  *total = __shfl_sync(0xffffffffu, w, nwarps - 1);
  if (!last_use) __syncthreads();
  return excl;
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
// Never returns 0 for a non-NaN input, so 0 can mark "excluded".
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ------------------------------------------------------------ top-k select
constexpr int kTopkCand = 4096;   // boundary-bin candidates kept after the first pass

// Shared memory (ints) block_topk needs besides the keys.
__host__ __device__ constexpr int topk_scratch_ints(int nthreads) {
  // max of the radix path's needs and (values + their indices + block_kth
  // scratch + scans)
  return (nthreads / 32) * 256 + 256 + 64 + kTopkCand > 8 * nthreads + (nthreads / 32) * 256 + 256 + 48
             ? (nthreads / 32) * 256 + 256 + 64 + kTopkCand
             : 8 * nthreads + (nthreads / 32) * 256 + 256 + 48;
}

// Radix version of block_topk below (same contract, no bitmap): radix select
// on r = key - kmin (kmin: smallest non-zero key), 8-bit digits
// taken from the highest bit in which keys can differ downward, so no pass is
// spent on bits every key shares.  Each warp counts into a private 256-bin
// histogram (no cross-warp contention on popular bins).  After the first
// digit is fixed, the keys in its bin are compacted into a candidate list
// (if there are at most kTopkCand of them) and the remaining digits are
// resolved on that list only.  A final order-preserving compaction writes the
// chosen indices.  All threads of the block must call it; blockDim.x must be
// a multiple of 32.
__device__ __forceinline__ void block_topk_radix(const uint32_t* keys, int n, int k, int* out, int* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  const int nwarps = nthr >> 5;
  int* whist = scratch;                       // [nwarps][256]
  int* hist = scratch + nwarps * 256;         // [256]
  int* tmp = hist + 256;                      // 33 ints for the scans
  int* bc = tmp + 40;                         // broadcast slots
  int* cand = tmp + 64;                       // [kTopkCand] indices
  // smallest and largest non-zero key
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int j = tid; j < n; j += nthr) {
    const uint32_t key = keys[j];
    if (key) { kmin = min(kmin, key); kmax = max(kmax, key); }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) { whist[warp] = static_cast<int>(kmin); whist[32 + warp] = static_cast<int>(kmax); }
  __syncthreads();
  if (tid < 32) {
    uint32_t m = tid < nwarps ? static_cast<uint32_t>(whist[tid]) : 0xffffffffu;
    uint32_t M = tid < nwarps ? static_cast<uint32_t>(whist[32 + tid]) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
      M = max(M, __shfl_xor_sync(0xffffffffu, M, o));
    }
    if (tid == 0) { bc[2] = static_cast<int>(m); bc[3] = static_cast<int>(M); }
  }
  __syncthreads();
  kmin = static_cast<uint32_t>(bc[2]);
  kmax = static_cast<uint32_t>(bc[3]);
  const uint32_t span = kmax - kmin;          // every r = key - kmin is <= span
  int hb = span ? 32 - __clz(span) : 1;       // r < 2^hb
  uint32_t prefix = 0, pmask = 0;
  int need = k;
  int ncand = -1;                             // -1: scan all keys
  while (hb > 0) {
    const int width = hb < 8 ? hb : 8;
    const int shift = hb - width;
    const uint32_t dmask = (1u << width) - 1u;
    int* wh = whist + warp * 256;
    for (int i = lane; i < 256; i += 32) wh[i] = 0;
    __syncwarp();
    if (ncand < 0) {
      for (int j = tid; j < n; j += nthr) {
        const uint32_t key = keys[j];
        const uint32_t r = key - kmin;
        if (key && (r & pmask) == prefix) atomicAdd(&wh[(r >> shift) & dmask], 1);
      }
    } else {
      for (int c = tid; c < ncand; c += nthr) {
        const uint32_t r = keys[cand[c]] - kmin;
        if ((r & pmask) == prefix) atomicAdd(&wh[(r >> shift) & dmask], 1);
      }
    }
    __syncthreads();
    for (int i = tid; i < 256; i += nthr) {
      int acc = 0;
      for (int w = 0; w < nwarps; ++w) acc += whist[w * 256 + i];
      hist[i] = acc;
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns bins 255-8l .. 248-8l, visited from the top
      int cnt[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { cnt[i] = hist[255 - 8 * lane - i]; sum += cnt[i]; }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - sum;
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
      const int first = __ffs(hit) - 1;   // need <= number of candidates by construction
      if (lane == first) {
        int acc = excl, digit = 255 - 8 * lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc + cnt[i] >= need) { digit = 255 - 8 * lane - i; break; }
          acc += cnt[i];
        }
        bc[0] = digit;
        bc[1] = need - acc;
        bc[4] = cnt[digit == 255 - 8 * lane ? 0 : (255 - 8 * lane - digit)];   // keys in the bin
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(bc[0]) << shift;
    pmask |= dmask << shift;
    need = bc[1];
    const int inbin = bc[4];
    hb = shift;
    __syncthreads();
    if (ncand < 0 && hb > 0 && inbin <= kTopkCand) {
      // compact the bin's keys into the candidate list (order not needed)
      const int per = (n + nthr - 1) / nthr;
      const int j0 = tid * per, j1 = min(n, j0 + per);
      int mine = 0;
      for (int j = j0; j < j1; ++j) {
        const uint32_t key = keys[j];
        mine += key && ((key - kmin) & pmask) == prefix;
      }
      int tot;
      int pos = block_exclusive_scan(mine, tmp, &tot);
      for (int j = j0; j < j1; ++j) {
        const uint32_t key = keys[j];
        if (key && ((key - kmin) & pmask) == prefix) cand[pos++] = j;
      }
      ncand = tot;
      __syncthreads();
    }
  }
  // kmin + prefix is the k-th largest key; take every key above it and the
  // first `need` keys equal to it (lowest indices first).
  const uint32_t T = kmin + prefix;
  const int per = (n + nthr - 1) / nthr;
  const int j0 = tid * per, j1 = min(n, j0 + per);
  int gt = 0, eq = 0;
  for (int j = j0; j < j1; ++j) {
    const uint32_t key = keys[j];
    gt += key > T;
    eq += key == T;
  }
  int tot;
  const int eq_before = block_exclusive_scan(eq, tmp, &tot);
  const int eq_take = max(0, min(eq, need - eq_before));
  const int pos0 = block_exclusive_scan(gt + eq_take, tmp, &tot);
  int pos = pos0, taken = 0;
  for (int j = j0; j < j1; ++j) {
    const uint32_t key = keys[j];
    bool take = key > T;
    if (key == T && taken < eq_take) { take = true; ++taken; }
    if (take) out[pos++] = j;
  }
  __syncthreads();
}

// Rounds a shared-memory int pointer up to a 16-byte boundary (the top-k
// scratch holds 64-bit entries).
__device__ __forceinline__ int* align16(int* p) {
  return reinterpret_cast<int*>((reinterpret_cast<uintptr_t>(p) + 15) & ~static_cast<uintptr_t>(15));
}

// The k-th largest (1-based) of the values v[0..cnt) (shared memory, all
// non-zero, cnt <= 4 * blockDim.x, 1 <= kth <= cnt).  Returns it in *T and in
// *need how many of the values equal to it are within the top kth.  Radix
// select from the highest bit in which the values differ, 8 bits per pass,
// each thread holding up to 4 values in registers and each warp counting into
// its own 256-bin histogram.  All threads of the block must call it.
__device__ __forceinline__ void block_kth(const uint32_t* v, int cnt, int kth, int* scratch, uint32_t* T,
                                          int* need_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  const int nwarps = nthr >> 5;
  int* whist = scratch;                     // [nwarps][256]
  int* hist = scratch + nwarps * 256;       // [256]
  int* bc = hist + 256;                     // broadcast slots
  uint32_t x[4];
  uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = tid + q * nthr;
    x[q] = i < cnt ? v[i] : 0u;
    if (x[q]) { lo = min(lo, x[q]); hi = max(hi, x[q]); }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) { whist[warp] = static_cast<int>(lo); whist[32 + warp] = static_cast<int>(hi); }
  __syncthreads();
  if (tid < 32) {
    uint32_t m = tid < nwarps ? static_cast<uint32_t>(whist[tid]) : 0xffffffffu;
    uint32_t M = tid < nwarps ? static_cast<uint32_t>(whist[32 + tid]) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
      M = max(M, __shfl_xor_sync(0xffffffffu, M, o));
    }
    if (tid == 0) { bc[2] = static_cast<int>(m); bc[3] = static_cast<int>(M); }
  }
  __syncthreads();
  const uint32_t vmin = static_cast<uint32_t>(bc[2]);
  const uint32_t span = static_cast<uint32_t>(bc[3]) - vmin;
  int hb = span ? 32 - __clz(span) : 1;
  uint32_t prefix = 0, pmask = 0;
  int need = kth;
  while (hb > 0) {
    const int width = hb < 8 ? hb : 8;
    const int shift = hb - width;
    const uint32_t dmask = (1u << width) - 1u;
    int* wh = whist + warp * 256;
    for (int i = lane; i < 256; i += 32) wh[i] = 0;
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t r = x[q] - vmin;
      if (x[q] && (r & pmask) == prefix) atomicAdd(&wh[(r >> shift) & dmask], 1);
    }
    __syncthreads();
    for (int i = tid; i < 256; i += nthr) {
      int acc = 0;
      for (int w = 0; w < nwarps; ++w) acc += whist[w * 256 + i];
      hist[i] = acc;
    }
    __syncthreads();
    if (tid < 32) {
      int cnt8[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { cnt8[i] = hist[255 - 8 * lane - i]; sum += cnt8[i]; }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
      const int first = __ffs(hit) - 1;
      if (lane == first) {
        int acc = incl - sum, digit = 255 - 8 * lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc + cnt8[i] >= need) { digit = 255 - 8 * lane - i; break; }
          acc += cnt8[i];
        }
        bc[0] = digit;
        bc[1] = need - acc;
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(bc[0]) << shift;
    pmask |= dmask << shift;
    need = bc[1];
    hb = shift;
    __syncthreads();
  }
  *T = vmin + prefix;
  *need_out = need;
}

// block_kth for at most 256 V values, computed by the block's first 256
// threads alone (eight warps meeting at named barrier 1, V values per
// thread): far fewer threads wait at each of the passes' barriers.  The
// k-th largest lands in scratch[kKth8T] and the count of its equals within
// the top kth in scratch[kKth8Need]; the caller synchronises the block before
// reading them.  scratch holds kKth8Ints ints.  With max_passes < 4 the
// select may stop before the last digit: scratch[kKth8T] is then the lower
// edge of the digit range that holds the k-th largest (a lower bound of it)
// and scratch[kKth8Need] is not meaningful.  After a complete select
// scratch[kKth8Eq] is the number of values equal to the k-th largest.  A
// caller that knows a range [rlo, rhi] (rhi != 0) holding every non-zero
// value passes it, and the select skips its min/max reduction.  With
// whole_bucket, the select stops as soon as every value of the digit range
// holding the k-th largest is among the kth largest: scratch[kKth8T] is then
// that range's lower edge, and the values at or above it are exactly the kth
// largest (scratch[kKth8Eq] == scratch[kKth8Need]).
constexpr int kKth8T = 8 * 256 + 256 + 4, kKth8Need = kKth8T + 1, kKth8Eq = kKth8T + 2,
              kKth8Ints = 8 * 256 + 256 + 8;
template <int V = 4>
__device__ __forceinline__ void block_kth_256(const uint32_t* v, int cnt, int kth, int* scratch,
                                              int max_passes = 4, uint32_t rlo = 0u, uint32_t rhi = 0u,
                                              bool whole_bucket = false) {
  const int tid = threadIdx.x;
  if (tid >= 256) return;
  const int lane = tid & 31, warp = tid >> 5;
  int* whist = scratch;             // [8][256]
  int* hist = scratch + 8 * 256;    // [256]
  int* bc = hist + 256;             // broadcast slots
  auto bar = []() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
  uint32_t x[V];
  uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
  for (int q = 0; q < V; ++q) {
    const int i = tid + q * 256;
    x[q] = i < cnt ? v[i] : 0u;
    if (x[q]) { lo = min(lo, x[q]); hi = max(hi, x[q]); }
  }
  if (rhi == 0u) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) { whist[warp] = static_cast<int>(lo); whist[32 + warp] = static_cast<int>(hi); }
  bar();
  if (tid < 32) {
    uint32_t m = tid < 8 ? static_cast<uint32_t>(whist[tid]) : 0xffffffffu;
    uint32_t M = tid < 8 ? static_cast<uint32_t>(whist[32 + tid]) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
      M = max(M, __shfl_xor_sync(0xffffffffu, M, o));
    }
    if (tid == 0) { bc[2] = static_cast<int>(m); bc[3] = static_cast<int>(M); }
  }
  bar();
  }
  const uint32_t vmin = rhi != 0u ? rlo : static_cast<uint32_t>(bc[2]);
  const uint32_t span = (rhi != 0u ? rhi : static_cast<uint32_t>(bc[3])) - vmin;
  int hb = span ? 32 - __clz(span) : 1;
  uint32_t prefix = 0, pmask = 0;
  int need = kth;
  for (int pass = 0; hb > 0 && pass < max_passes; ++pass) {
    const int width = hb < 8 ? hb : 8;
    const int shift = hb - width;
    const uint32_t dmask = (1u << width) - 1u;
    int* wh = whist + warp * 256;
#pragma unroll
    for (int i = 0; i < 8; ++i) wh[i * 32 + lane] = 0;
    __syncwarp();
#pragma unroll
    for (int q = 0; q < V; ++q) {
      const uint32_t r = x[q] - vmin;
      if (x[q] && (r & pmask) == prefix) atomicAdd(&wh[(r >> shift) & dmask], 1);
    }
    bar();
    {
      int acc = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) acc += whist[w * 256 + tid];
      hist[tid] = acc;
    }
    bar();
    if (tid < 32) {
      int cnt8[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { cnt8[i] = hist[255 - 8 * lane - i]; sum += cnt8[i]; }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
      const int first = __ffs(hit) - 1;
      if (lane == first) {
        int acc = incl - sum, digit = 255 - 8 * lane, in_digit = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc + cnt8[i] >= need) {
            digit = 255 - 8 * lane - i;
            in_digit = cnt8[i];
            break;
          }
          acc += cnt8[i];
        }
        bc[0] = digit;
        bc[1] = need - acc;
        bc[6] = in_digit;   // after the last digit: the values equal to the result
      }
    }
    bar();
    // bc[0..1] are rewritten only after two more barriers of the next pass
    prefix |= static_cast<uint32_t>(bc[0]) << shift;
    pmask |= dmask << shift;
    need = bc[1];
    hb = shift;
    if (whole_bucket && bc[6] == need) break;   // the whole range is taken
  }
  if (tid == 0) {
    bc[4] = static_cast<int>(vmin + prefix);
    bc[5] = need;
  }
}

// Block-wide selection of the k largest keys among keys[0..n) (shared
// memory), ties broken toward the lower index; key 0 marks an excluded entry
// and is never chosen when at least k keys are non-zero.  On return out[0..k)
// holds the chosen indices in ascending order, bits[0..ceil(n/32)) is their
// bitmap and wpref[w] the number of chosen indices below 32 w (all three in
// shared memory).  `scratch` holds topk_scratch_ints(blockDim.x) ints and is
// 16-byte aligned.
//
// The k-th largest key T is found on small sets only: 1024 evenly spaced
// keys give a threshold T0 a little below the k-th largest (its rank in the
// sample leaves about 1.5k + margin keys above it in expectation); the keys
// >= T0 (normally a few hundred) are gathered and T is their k-th largest.
// A final pass marks every key above T and, in index order, the first keys
// equal to T that the top k needs.  If the sample misjudges (fewer than k or
// more than 4 blockDim.x survivors) the radix select over all keys decides
// instead.  All threads of the block must call it.
constexpr int kTopkSample = 1024;

// The indices set in bits[0..nw) in ascending order into out[], and wpref[w]
// = the number of them below 32 w (all in shared memory; tmp holds >= 33
// ints).  All threads of the block must call it.
__device__ __forceinline__ void bitmap_list(const uint32_t* bits, int nw, int* out, int* wpref, int* tmp) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int per = (nw + nthr - 1) / nthr;
  const int w0 = tid * per, w1 = min(nw, w0 + per);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
  int tot;
  int ex = block_exclusive_scan(cnt, tmp, &tot, true);   // tmp is not written again here
  for (int w = w0; w < w1; ++w) {
    wpref[w] = ex;
    uint32_t b = bits[w];
    while (b) {
      const int bit = __ffs(b) - 1;
      out[ex++] = w * 32 + bit;
      b &= b - 1;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void block_topk(const uint32_t* keys, int n, int k, int* out, int* scratch,
                                           uint32_t* bits, int* wpref) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  const int nwarps = nthr >> 5;
  const int nw = (n + 31) >> 5;
  const int cap = 4 * nthr;
  uint32_t* vals = reinterpret_cast<uint32_t*>(scratch);   // cap values
  int* vidx = scratch + cap;                                // their indices
  int* ks = vidx + cap;                                     // block_kth scratch
  int* tmp = ks + (nthr / 32) * 256 + 256 + 8;              // 40 ints for the scans
  int* cnt_slot = tmp + 36;                                 // survivor counter
  int* eq_slot = tmp + 37;                                  // survivors equal to T
  // each warp owns a contiguous range of 32-key rows; lanes read consecutive
  // keys, so shared-memory reads are conflict-free
  const int rows = (n + 31) >> 5;
  const int rpw = (rows + nwarps - 1) / nwarps;
  const int r0 = warp * rpw, r1 = min(rows, r0 + rpw);
  uint32_t T = 0;
  int need = 0;
  bool ok = true;
  if (tid == 0) {
    *cnt_slot = 0;
    *eq_slot = 0;
  }
  __syncthreads();
  uint32_t T0 = 1u;                  // keys >= T0 are gathered (all non-zero keys when n <= cap)
  if (n > cap) {
    const int S = kTopkSample;
    // non-zero samples of evenly spaced keys (order irrelevant)
    for (int s2 = tid; s2 < ((S + 31) & ~31); s2 += nthr) {
      const uint32_t x = s2 < S ? keys[static_cast<int>((static_cast<long long>(s2) * n) / S)] : 0u;
      const unsigned m = __ballot_sync(0xffffffffu, x != 0u);
      int base = 0;
      if (lane == 0 && m) base = atomicAdd(cnt_slot, __popc(m));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (x) vals[base + __popc(m & ((1u << lane) - 1u))] = x;
    }
    __syncthreads();
    const int tot = *cnt_slot;
    // rank r (0-based) among the samples: expected survivors ~ (r + 1) n / S
    int r = static_cast<int>((3LL * k * S + 2LL * n - 1) / (2LL * n)) + 12;
    if (r > tot - 1) r = tot - 1;
    T0 = 0xffffffffu;                // no non-zero sample: no survivor, radix decides
    if (tot > 0) block_kth_256(vals, tot, r + 1, ks);
    __syncthreads();
    if (tot > 0) T0 = static_cast<uint32_t>(ks[kKth8T]);
    if (tid == 0) *cnt_slot = 0;
    __syncthreads();
  }
  // gather the survivors (keys >= T0, non-zero) while they fit in `vals`:
  // each warp counts its rows' survivors, reserves one range, then stores
  {
    int wcnt = 0;
    for (int row = r0; row < r1; ++row) {
      const int j = row * 32 + lane;
      const uint32_t key = j < n ? keys[j] : 0u;
      wcnt += __popc(__ballot_sync(0xffffffffu, key != 0u && key >= T0));
    }
    int base = 0;
    if (lane == 0 && wcnt) base = atomicAdd(cnt_slot, wcnt);
    base = __shfl_sync(0xffffffffu, base, 0);
    for (int row = r0; row < r1; ++row) {
      const int j = row * 32 + lane;
      const uint32_t key = j < n ? keys[j] : 0u;
      const bool keep = key != 0u && key >= T0;
      const unsigned m = __ballot_sync(0xffffffffu, keep);
      const int pos = base + __popc(m & ((1u << lane) - 1u));
      if (keep && pos < cap) {
        vals[pos] = key;
        vidx[pos] = j;
      }
      base += __popc(m);
    }
  }
  __syncthreads();
  const int nsurv = *cnt_slot;
  ok = nsurv >= k && nsurv <= cap;
  for (int w = tid; w < nw; w += nthr) bits[w] = 0u;
  if (ok && nsurv <= 1024) {
    block_kth_256(vals, nsurv, k, ks);
    __syncthreads();
    T = static_cast<uint32_t>(ks[kKth8T]);
    need = ks[kKth8Need];
  } else if (ok) {
    block_kth(vals, nsurv, k, ks, &T, &need);
  }
  // survivors equal to T: when the top k takes all of them (the usual case)
  // the bitmap follows from the survivors alone
  int eq_total = 0;
  if (ok) {
    int eq = 0;
    for (int i = tid; i < nsurv; i += nthr) eq += vals[i] == T;
    eq = __reduce_add_sync(0xffffffffu, eq);
    if (lane == 0 && eq) atomicAdd(eq_slot, eq);
  }
  __syncthreads();
  if (ok) eq_total = *eq_slot;
  if (ok && eq_total == need) {
    for (int i = tid; i < nsurv; i += nthr)
      if (vals[i] >= T) atomicOr(&bits[vidx[i] >> 5], 1u << (vidx[i] & 31));
  } else if (ok) {
    // every key above T; the keys equal to T in index order until `need`
    int eq = 0;
    for (int row = r0; row < r1; ++row) {
      const int j = row * 32 + lane;
      const uint32_t key = j < n ? keys[j] : 0u;
      const unsigned gt = __ballot_sync(0xffffffffu, key > T);
      if (lane == 0) bits[row] = gt;
      eq += __popc(__ballot_sync(0xffffffffu, key == T));
    }
    // warp totals of equal keys -> exclusive prefix over warps
    if (lane == 0) tmp[warp] = eq;
    __syncthreads();
    if (warp == 0) {
      int v = lane < nwarps ? tmp[lane] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      __syncwarp();
      if (lane < nwarps) tmp[lane] = incl - v;
    }
    __syncthreads();
    int before = tmp[warp];
    for (int row = r0; row < r1 && before < need; ++row) {
      const int j = row * 32 + lane;
      const uint32_t key = j < n ? keys[j] : 0u;
      const unsigned e = __ballot_sync(0xffffffffu, key == T);
      const int rank = before + __popc(e & ((1u << lane) - 1u));
      const unsigned take = __ballot_sync(0xffffffffu, key == T && rank < need);
      if (lane == 0) bits[row] |= take;
      before += __popc(e);
    }
  } else {
    block_topk_radix(keys, n, k, out, scratch);
    for (int i = tid; i < k; i += nthr) atomicOr(&bits[out[i] >> 5], 1u << (out[i] & 31));
  }
  __syncthreads();
  bitmap_list(bits, nw, out, wpref, tmp);
}

// The step's value misses, for bf16 records with d = 128: thread h of nh
// (a half-warp per 8-token group of a missed chunk) reads the group's values
// from the mapped pinned host copy of V and writes the V^T half of the
// chunk's cache-slot record (one 128-byte run per lane).  The miss list
// holds (pair * n + chunk, pair * k + slot) per missed chunk.
__device__ __forceinline__ void fetch_value_groups(const __nv_bfloat16* __restrict__ vcpu,
                                                   __nv_bfloat16* __restrict__ KV_slot,
                                                   const int32_t* __restrict__ miss_chunk,
                                                   const int32_t* __restrict__ miss_slot, int total,
                                                   int s, int n, int c, int k, int npairs, long long h,
                                                   long long nh, int* __restrict__ status) {
  const int q = threadIdx.x & 15;
  if (total > npairs * k) {
    if (h == 0) flag_error(status, DEV_BAD_COUNT);
    total = npairs * k;
  }
  const int gpc = c >> 3;   // groups per chunk
  const long long groups = static_cast<long long>(total) * gpc, step = nh >> 4;
  // two groups per round, both read before either is written, so that a
  // half-warp with two groups waits for the host link once
  for (long long g0 = h >> 4; g0 < groups; g0 += 2 * step) {
    uint4 in[2][8];
    uint4* dst[2] = {nullptr, nullptr};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const long long gi = g0 + u * step;
      if (gi >= groups) break;
      const int m = static_cast<int>(gi / gpc), gs = static_cast<int>(gi - static_cast<long long>(m) * gpc);
      const int pc = miss_chunk[m], ps = miss_slot[m];
      const int pair = pc / n, chunk = pc - pair * n;
      const int slot = ps - pair * k;
      if (pair < 0 || pair >= npairs || chunk < 0 || slot < 0 || slot >= k) {
        if (q == 0) flag_error(status, DEV_BAD_SLOT);
        continue;
      }
      const uint4* src = reinterpret_cast<const uint4*>(
          vcpu + (static_cast<size_t>(pair) * s + static_cast<size_t>(chunk) * c + gs * 8) * 128);
      dst[u] = reinterpret_cast<uint4*>(KV_slot + ((static_cast<size_t>(pair) * k + slot) * c + gs * 8) * 256 + 1024);
#pragma unroll
      for (int t = 0; t < 8; ++t) in[u][t] = src[t * 16 + q];
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (dst[u] == nullptr) continue;
      uint4 outv[8];
      transpose8x8(in[u], outv);
#pragma unroll
      for (int r = 0; r < 8; ++r) dst[u][q * 8 + r] = outv[r];
    }
  }
}

}  // namespace skv
