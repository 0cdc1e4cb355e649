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

// Block-wide exclusive scan of one int per thread.  `tmp` holds >= 33 ints of
// shared memory.  Returns the exclusive prefix; *total gets the block sum.
// Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_scan(int v, int* tmp, int* total) {
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
  if (warp == 0) {
    int w = lane < nwarps ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nwarps) tmp[lane] = w;  // inclusive warp totals
    if (lane == nwarps - 1) tmp[32] = w;
  }
  __syncthreads();
  const int excl = (warp ? tmp[warp - 1] : 0) + x - v;
  *total = tmp[32];
  __syncthreads();
  return excl;
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
// Never returns 0 for a non-NaN input, so 0 can mark "excluded".
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------------ top-k select
// Block-wide selection of the k largest keys among keys[0..n) (shared
// memory), ties broken toward the lower index; key 0 marks an excluded entry
// and is never chosen when at least k keys are non-zero.  The chosen indices
// are written to out[0..k) in ascending order (shared or global memory).
// `scratch` holds >= 256 + 40 ints of shared memory.  Radix select on the
// 32-bit key, 8 bits per pass from the top, then an order-preserving
// compaction.  All threads of the block must call it.
__device__ __forceinline__ void block_topk(const uint32_t* keys, int n, int k, int* out, int* scratch) {
  int* hist = scratch;          // 256
  int* tmp = scratch + 256;     // 33 for the scans
  int* bcast = scratch + 256 + 34;  // 2: digit, remaining need
  const int tid = threadIdx.x, lane = tid & 31, nthr = blockDim.x;
  uint32_t prefix = 0, pmask = 0;
  int need = k;
  const int n_pad = ((n + nthr - 1) / nthr) * nthr;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += nthr) hist[i] = 0;
    __syncthreads();
    for (int j = tid; j < n_pad; j += nthr) {
      int bin = 256;
      if (j < n) {
        const uint32_t key = keys[j];
        if ((key & pmask) == prefix) bin = (key >> shift) & 255;
      }
      const unsigned grp = __match_any_sync(0xffffffffu, bin);
      if (bin < 256 && lane == __ffs(grp) - 1) atomicAdd(&hist[bin], __popc(grp));
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
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - sum;
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
      const int first = __ffs(hit) - 1;  // need <= total count by construction
      if (lane == first) {
        int acc = excl, digit = 255 - 8 * lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc + cnt[i] >= need) { digit = 255 - 8 * lane - i; break; }
          acc += cnt[i];
        }
        bcast[0] = digit;
        bcast[1] = need - acc;
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(bcast[0]) << shift;
    pmask |= 255u << shift;
    need = bcast[1];
    __syncthreads();
  }
  // prefix is the k-th largest key; take every key above it and the first
  // `need` keys equal to it (lowest indices first).
  const uint32_t T = prefix;
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

}  // namespace skv
