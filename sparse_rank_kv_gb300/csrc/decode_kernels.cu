// Decode-step kernels of ShadowKV (Algorithm 2 of the ShadowKV review page):
//   k_score   P = MatMul(Q, L^T) / sqrt(d), with per-tile softmax statistics
//   k_select  S2 and I = ArgTopK(S2, k) per KV head, the set difference
//             against the previous step's GPU-resident chunks, and the
//             local-window append of the new token
//   k_fetch   Gather(V_CPU, I) for the chunks that missed the cache, read
//             zero-copy from pinned host memory on the side stream
//   k_attn    split-KV attention over [outliers; RoPE(K_sparse); local]
//             with the split combine done by the last block of each head
#include "common.cuh"
#include "internal.h"

namespace skv {

constexpr int kScoreTile = 128;      // landmarks per score tile (one per thread)
constexpr int kSelectThreads = 1024;
constexpr int kAttnThreads = 128;
constexpr int kFetchWarps = 8;

// ------------------------------------------------------------------ score
// One thread per landmark row; q for the KV head's G query heads sits in
// shared memory (pre-scaled by 1/sqrt(d)).  Tiles of 128 consecutive
// landmarks of one (batch, KV head) are visited by a grid-stride loop.
template <typename T, int D, int G>
__global__ void __launch_bounds__(kScoreTile)
k_score(const T* __restrict__ L, const T* __restrict__ q, const uint32_t* __restrict__ mask,
        float* __restrict__ P, float2* __restrict__ part, int n, int ntile, int total_tiles,
        float scale) {
  __shared__ __align__(16) float qs[G * D];
  __shared__ float red[kScoreTile / 32][G];
  __shared__ float bmax[G];
  constexpr int V = Ty<T>::kVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int cur = -1;
  for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
    const int pair = tile / ntile, ti = tile - pair * ntile;
    if (pair != cur) {
      __syncthreads();
      for (int i = tid; i < G * D; i += kScoreTile)
        qs[i] = Ty<T>::to_f(q[static_cast<size_t>(pair) * G * D + i]) * scale;
      __syncthreads();
      cur = pair;
    }
    const int j = ti * kScoreTile + tid;
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.f;
    if (j < n) {
      const T* row = L + (static_cast<size_t>(pair) * n + j) * D;
#pragma unroll 4
      for (int d0 = 0; d0 < D; d0 += V) {
        float x[V];
        Ty<T>::load16(row + d0, x);
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
          for (int e = 0; e < V; ++e) acc[g] = fmaf(x[e], qs[g * D + d0 + e], acc[g]);
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) P[(static_cast<size_t>(pair) * G + g) * n + j] = acc[g];
    }
    const bool valid = j < n && !((mask[static_cast<size_t>(pair) * ((n + 31) >> 5) + (j >> 5)] >> (j & 31)) & 1u);
    // tile max and sum of exp over valid rows, per head
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float m = warp_max(valid ? acc[g] : -INFINITY);
      if (lane == 0) red[warp][g] = m;
    }
    __syncthreads();
    if (tid < G) {
      float m = -INFINITY;
      for (int w = 0; w < kScoreTile / 32; ++w) m = fmaxf(m, red[w][tid]);
      bmax[tid] = m;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float m = bmax[g];
      const float e = warp_sum(valid ? __expf(acc[g] - m) : 0.f);
      if (lane == 0) red[warp][g] = e;
    }
    __syncthreads();
    if (tid < G) {
      float z = 0.f;
      for (int w = 0; w < kScoreTile / 32; ++w) z += red[w][tid];
      part[(static_cast<size_t>(pair) * G + tid) * ntile + ti] = make_float2(bmax[tid], z);
    }
    __syncthreads();
  }
}

// ----------------------------------------------------------------- select
// One block per (batch, KV head).  Shared memory: keys[n], then the cache
// bookkeeping arrays.
template <typename T, int D>
__global__ void __launch_bounds__(kSelectThreads)
k_select(const float* __restrict__ P, const float2* __restrict__ part,
         const uint32_t* __restrict__ mask, int G, int n, int ntile, int k, int group_reduce,
         int cache_on, int32_t* __restrict__ sel, int32_t* __restrict__ sel_slot,
         int32_t* __restrict__ slot_chunk, int32_t* __restrict__ miss_chunk,
         int32_t* __restrict__ miss_slot, int32_t* __restrict__ miss_count,
         int32_t* __restrict__ hits, unsigned long long* __restrict__ counters,
         const T* __restrict__ k_new, const T* __restrict__ v_new, T* __restrict__ K_loc,
         T* __restrict__ V_loc, int loc_row, int loc_cap, int* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int nw = (n + 31) >> 5;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  uint32_t* words = keys + n;
  int* wpref = reinterpret_cast<int*>(words + nw);
  int* s_sel = wpref + nw;
  int* s_slot = s_sel + k;
  int* s_hit = s_slot + k;
  int* s_keep = s_hit + k;
  int* s_free = s_keep + k;
  int* scratch = s_free + k;   // 300 ints
  float* lse = reinterpret_cast<float*>(scratch + 300);  // G floats
  int* tmp = scratch + 256;

  const int pair = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;

  // append the new token's key/value to the local window
  if (k_new != nullptr) {
    for (int i = tid; i < D; i += nthr) {
      const size_t dst = (static_cast<size_t>(pair) * loc_cap + loc_row) * D + i;
      K_loc[dst] = k_new[static_cast<size_t>(pair) * D + i];
      V_loc[dst] = v_new[static_cast<size_t>(pair) * D + i];
    }
  }
  // log-sum-exp of each query head over the candidate chunks
  for (int g = warp; g < G; g += nthr / 32) {
    const float2* pp = part + (static_cast<size_t>(pair) * G + g) * ntile;
    float m = -INFINITY;
    for (int t = lane; t < ntile; t += 32) m = fmaxf(m, pp[t].x);
    m = warp_max(m);
    float z = 0.f;
    for (int t = lane; t < ntile; t += 32) {
      const float2 v = pp[t];
      if (v.y > 0.f) z += v.y * __expf(v.x - m);
    }
    z = warp_sum(z);
    if (lane == 0) lse[g] = m + __logf(z);
  }
  __syncthreads();
  // selection keys: S2 per chunk, 0 for outliers
  const uint32_t* mk = mask + static_cast<size_t>(pair) * nw;
  for (int j = tid; j < n; j += nthr) {
    uint32_t key = 0;
    if (!((mk[j >> 5] >> (j & 31)) & 1u)) {
      if (group_reduce == 0) {
        float sc = -INFINITY;
        for (int g = 0; g < G; ++g)
          sc = fmaxf(sc, P[(static_cast<size_t>(pair) * G + g) * n + j] - lse[g]);
        key = order_key(sc);
      } else {
        float sc = 0.f;
        for (int g = 0; g < G; ++g)
          sc += __expf(P[(static_cast<size_t>(pair) * G + g) * n + j] - lse[g]);
        key = __float_as_uint(sc) + 1u;
      }
    }
    keys[j] = key;
  }
  __syncthreads();
  block_topk(keys, n, k, s_sel, scratch);

  // bitmap of the selection and prefix popcounts per 32-chunk word
  for (int i = tid; i < nw; i += nthr) words[i] = 0u;
  __syncthreads();
  for (int i = tid; i < k; i += nthr) atomicOr(&words[s_sel[i] >> 5], 1u << (s_sel[i] & 31));
  __syncthreads();
  {
    const int per = (nw + nthr - 1) / nthr;
    const int w0 = tid * per, w1 = min(nw, w0 + per);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(words[w]);
    int tot;
    int ex = block_exclusive_scan(cnt, tmp, &tot);
    for (int w = w0; w < w1; ++w) { wpref[w] = ex; ex += __popc(words[w]); }
  }
  for (int i = tid; i < k; i += nthr) s_hit[i] = 0;
  __syncthreads();
  // slots whose chunk is selected again keep it (hits)
  int32_t* sc_row = slot_chunk + static_cast<size_t>(pair) * k;
  for (int i = tid; i < k; i += nthr) {
    int ch = cache_on ? sc_row[i] : -1;
    if (ch >= n) { flag_error(status, DEV_BAD_CHUNK); ch = -1; }
    int keep = 0;
    if (ch >= 0 && ((words[ch >> 5] >> (ch & 31)) & 1u)) {
      const int pos = wpref[ch >> 5] + __popc(words[ch >> 5] & ((1u << (ch & 31)) - 1u));
      s_slot[pos] = i;
      s_hit[pos] = 1;
      keep = 1;
    }
    s_keep[i] = keep;
  }
  __syncthreads();
  // the m-th missing chunk (ascending) takes the m-th freed slot (ascending)
  const int is_miss = tid < k ? !s_hit[tid] : 0;
  const int is_free = tid < k ? !s_keep[tid] : 0;
  int nmiss, nfree;
  const int mrank = block_exclusive_scan(is_miss, tmp, &nmiss);
  const int frank = block_exclusive_scan(is_free, tmp, &nfree);
  if (is_free) s_free[frank] = tid;
  __syncthreads();
  if (nmiss != nfree) flag_error(status, DEV_BAD_COUNT);
  if (is_miss && mrank < nfree) {
    const int slot = s_free[mrank];
    s_slot[tid] = slot;
    sc_row[slot] = s_sel[tid];
    miss_chunk[static_cast<size_t>(pair) * k + mrank] = s_sel[tid];
    miss_slot[static_cast<size_t>(pair) * k + mrank] = slot;
  }
  __syncthreads();
  for (int i = tid; i < k; i += nthr) {
    sel[static_cast<size_t>(pair) * k + i] = s_sel[i];
    sel_slot[static_cast<size_t>(pair) * k + i] = s_slot[i];
  }
  if (tid == 0) {
    miss_count[pair] = min(nmiss, nfree);
    hits[pair] = k - nmiss;
    atomicAdd(&counters[0], static_cast<unsigned long long>(k - nmiss));
    atomicAdd(&counters[1], static_cast<unsigned long long>(nmiss));
  }
}

// ------------------------------------------------------------------ fetch
// Warp per missed chunk: c*d elements copied from pinned host memory (read
// through its mapped device address) into the chunk's cache slot.
template <typename T>
__global__ void __launch_bounds__(kFetchWarps * 32)
k_fetch(const T* __restrict__ vcpu, T* __restrict__ slot_V, const int32_t* __restrict__ miss_chunk,
        const int32_t* __restrict__ miss_slot, const int32_t* __restrict__ miss_count, int s,
        int n, int c, int d, int k, int* __restrict__ status) {
  const int pair = blockIdx.x;
  const int m = blockIdx.y * kFetchWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (m >= miss_count[pair]) return;
  const int chunk = miss_chunk[static_cast<size_t>(pair) * k + m];
  const int slot = miss_slot[static_cast<size_t>(pair) * k + m];
  if (chunk < 0 || chunk >= n || slot < 0 || slot >= k) {
    if (lane == 0) flag_error(status, DEV_BAD_SLOT);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(vcpu + (static_cast<size_t>(pair) * s + static_cast<size_t>(chunk) * c) * d);
  uint4* dst = reinterpret_cast<uint4*>(slot_V + ((static_cast<size_t>(pair) * k + slot) * c) * d);
  const int nvec = c * d * static_cast<int>(sizeof(T)) / 16;
  constexpr int U = 4;
  for (int base = 0; base < nvec; base += 32 * U) {
    uint4 buf[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nvec) buf[u] = src[i];
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * 32 + lane;
      if (i < nvec) dst[i] = buf[u];
    }
  }
}

// -------------------------------------------------------------- attention
// Block (pair, split) covers tokens [split*S, min(T, split*S + S)) of the
// concatenation [outliers (n_out); rebuilt chunks (n_sp); local (n_loc)].
// Logits and probabilities stay in shared memory; the block writes its
// partial (max, sum, sum p v) per query head; the last block of the pair
// (atomic ticket) combines all splits in split order.
template <typename T, int D, int G>
__global__ void __launch_bounds__(kAttnThreads)
k_attn(const T* __restrict__ K_out, const T* __restrict__ V_out, const T* __restrict__ K_sp,
       const T* __restrict__ slot_V, const int32_t* __restrict__ sel_slot,
       const T* __restrict__ K_loc, const T* __restrict__ V_loc, const T* __restrict__ q,
       T* __restrict__ out, float* __restrict__ part, int32_t* __restrict__ ticket, int n_out,
       int n_sp, int n_loc, int loc_cap, int c, int k, int S, int nsplit, int max_splits,
       float scale_log2) {
  extern __shared__ __align__(16) float sm[];
  float* qs = sm;               // G*D
  float* ps = qs + G * D;       // G*S
  __shared__ float red[kAttnThreads / 32][G];
  __shared__ float hm[G], hl[G];
  __shared__ int last;
  constexpr int V = Ty<T>::kVec;
  const int pair = blockIdx.x, split = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T_all = n_out + n_sp + n_loc;
  const int t0 = split * S, t1 = min(T_all, t0 + S), cnt = t1 - t0;

  for (int i = tid; i < G * D; i += kAttnThreads)
    qs[i] = Ty<T>::to_f(q[static_cast<size_t>(pair) * G * D + i]) * scale_log2;
  __syncthreads();

  auto key_row = [&](int t) -> const T* {
    if (t < n_out) return K_out + (static_cast<size_t>(pair) * n_out + t) * D;
    t -= n_out;
    if (t < n_sp) return K_sp + (static_cast<size_t>(pair) * n_sp + t) * D;
    t -= n_sp;
    return K_loc + (static_cast<size_t>(pair) * loc_cap + t) * D;
  };
  auto val_row = [&](int t) -> const T* {
    if (t < n_out) return V_out + (static_cast<size_t>(pair) * n_out + t) * D;
    t -= n_out;
    if (t < n_sp) {
      const int slot = sel_slot[static_cast<size_t>(pair) * k + t / c];
      return slot_V + ((static_cast<size_t>(pair) * k + slot) * c + (t % c)) * D;
    }
    t -= n_sp;
    return V_loc + (static_cast<size_t>(pair) * loc_cap + t) * D;
  };

  // logits (log2 domain)
  float lmax[G];
#pragma unroll
  for (int g = 0; g < G; ++g) lmax[g] = -INFINITY;
  for (int i = tid; i < cnt; i += kAttnThreads) {
    const T* row = key_row(t0 + i);
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.f;
#pragma unroll 4
    for (int d0 = 0; d0 < D; d0 += V) {
      float x[V];
      Ty<T>::load16(row + d0, x);
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int e = 0; e < V; ++e) acc[g] = fmaf(x[e], qs[g * D + d0 + e], acc[g]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      ps[g * S + i] = acc[g];
      lmax[g] = fmaxf(lmax[g], acc[g]);
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float m = warp_max(lmax[g]);
    if (lane == 0) red[warp][g] = m;
  }
  __syncthreads();
  if (tid < G) {
    float m = -INFINITY;
    for (int w = 0; w < kAttnThreads / 32; ++w) m = fmaxf(m, red[w][tid]);
    hm[tid] = m;
  }
  __syncthreads();
  float lsum[G];
#pragma unroll
  for (int g = 0; g < G; ++g) lsum[g] = 0.f;
  for (int i = tid; i < cnt; i += kAttnThreads) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float p = exp2f(ps[g * S + i] - hm[g]);
      ps[g * S + i] = p;
      lsum[g] += p;
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float z = warp_sum(lsum[g]);
    if (lane == 0) red[warp][g] = z;
  }
  __syncthreads();
  if (tid < G) {
    float z = 0.f;
    for (int w = 0; w < kAttnThreads / 32; ++w) z += red[w][tid];
    hl[tid] = z;
  }
  __syncthreads();

  // P V: thread owns output dimension tid
  const size_t pbase = static_cast<size_t>(pair) * G * max_splits;
  if (tid < D) {
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.f;
    for (int i = 0; i < cnt; ++i) {
      const float v = Ty<T>::to_f(val_row(t0 + i)[tid]);
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = fmaf(ps[g * S + i], v, acc[g]);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* pp = part + ((pbase + static_cast<size_t>(g) * max_splits + split) * (D + 2));
      pp[tid] = acc[g];
      if (tid == 0) { pp[D] = hm[g]; pp[D + 1] = hl[g]; }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last = (atomicAdd(&ticket[pair], 1) == nsplit - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (tid < D) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float* pp = part + (pbase + static_cast<size_t>(g) * max_splits) * (D + 2);
      float M = -INFINITY;
      for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, __ldcg(pp + sp * (D + 2) + D));
      float num = 0.f, den = 0.f;
      for (int sp = 0; sp < nsplit; ++sp) {
        const float* q2 = pp + sp * (D + 2);
        const float wgt = exp2f(__ldcg(q2 + D) - M);
        num = fmaf(wgt, __ldcg(q2 + tid), num);
        den = fmaf(wgt, __ldcg(q2 + D + 1), den);
      }
      out[(static_cast<size_t>(pair) * G + g) * D + tid] = Ty<T>::from_f(num / den);
    }
  }
  if (tid == 0) ticket[pair] = 0;
}

// --------------------------------------------------------- outlier mask
// Rebuilds the per-(batch, KV head) outlier bitmap from outlier_ids and
// checks that the ids are ascending, distinct and < n.
__global__ void k_build_mask(const int32_t* __restrict__ ids, uint32_t* __restrict__ mask, int n,
                             int o, int* __restrict__ status) {
  const int pair = blockIdx.x;
  const int nw = (n + 31) >> 5;
  uint32_t* mk = mask + static_cast<size_t>(pair) * nw;
  for (int i = threadIdx.x; i < nw; i += blockDim.x) mk[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < o; i += blockDim.x) {
    const int id = ids[static_cast<size_t>(pair) * o + i];
    const int prev = i ? ids[static_cast<size_t>(pair) * o + i - 1] : -1;
    if (id < 0 || id >= n || id <= prev) {
      flag_error(status, DEV_BAD_OUTLIER);
      continue;
    }
    atomicOr(&mk[id >> 5], 1u << (id & 31));
  }
}

// =============================================================== launchers
template <typename T, int D, int G>
static void score_t(Ctx& c, const void* q, cudaStream_t st) {
  const int pairs = c.p.b * c.p.h_kv;
  const int total = pairs * c.ntile;
  const int grid = min(total, num_sms(c) * 8);
  k_score<T, D, G><<<grid, kScoreTile, 0, st>>>(
      static_cast<const T*>(c.L), static_cast<const T*>(q), c.out_mask, c.logits, c.score_part,
      c.n, c.ntile, total, 1.0f / sqrtf(static_cast<float>(D)));
}

template <typename T, int D>
static void score_d(Ctx& c, const void* q, cudaStream_t st) {
  switch (c.G) {
    case 1: score_t<T, D, 1>(c, q, st); break;
    case 2: score_t<T, D, 2>(c, q, st); break;
    case 4: score_t<T, D, 4>(c, q, st); break;
    default: score_t<T, D, 8>(c, q, st); break;
  }
}

cudaError_t launch_score(Ctx& c, const void* q, cudaStream_t st) {
  kbegin(c, K_SCORE, st);
  if (c.p.dtype == SKV_DTYPE_BF16) {
    if (c.p.d == 128) score_d<bf16, 128>(c, q, st); else score_d<bf16, 64>(c, q, st);
  } else {
    if (c.p.d == 128) score_d<float, 128>(c, q, st); else score_d<float, 64>(c, q, st);
  }
  kend(c, K_SCORE, st);
  return cudaGetLastError();
}

size_t select_smem_bytes(int n, int k, int G) {
  const int nw = (n + 31) / 32;
  return sizeof(uint32_t) * (static_cast<size_t>(n) + 2 * nw) + sizeof(int) * (5 * static_cast<size_t>(k) + 300) +
         sizeof(float) * G + 16;
}

template <typename T, int D>
static cudaError_t select_t(Ctx& c, const void* k_new, const void* v_new, int loc_row,
                            cudaStream_t st) {
  const size_t smem = select_smem_bytes(c.n, c.p.k, c.G);
  auto kern = k_select<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<c.p.b * c.p.h_kv, kSelectThreads, smem, st>>>(
      c.logits, c.score_part, c.out_mask, c.G, c.n, c.ntile, c.p.k, c.p.group_reduce,
      c.cache_on ? 1 : 0, c.sel, c.sel_slot, c.slot_chunk, c.miss_chunk, c.miss_slot,
      c.miss_count, c.hits, c.counters, static_cast<const T*>(k_new), static_cast<const T*>(v_new),
      static_cast<T*>(c.K_loc), static_cast<T*>(c.V_loc), loc_row, c.loc_cap, c.status);
  return cudaGetLastError();
}

cudaError_t launch_select(Ctx& c, const void* k_new, const void* v_new, int loc_row,
                          cudaStream_t st) {
  kbegin(c, K_SELECT, st);
  cudaError_t e;
  if (c.p.dtype == SKV_DTYPE_BF16)
    e = c.p.d == 128 ? select_t<bf16, 128>(c, k_new, v_new, loc_row, st)
                     : select_t<bf16, 64>(c, k_new, v_new, loc_row, st);
  else
    e = c.p.d == 128 ? select_t<float, 128>(c, k_new, v_new, loc_row, st)
                     : select_t<float, 64>(c, k_new, v_new, loc_row, st);
  kend(c, K_SELECT, st);
  return e;
}

cudaError_t launch_fetch(Ctx& c, cudaStream_t st) {
  kbegin(c, K_FETCH, st);
  dim3 grid(c.p.b * c.p.h_kv, (c.p.k + kFetchWarps - 1) / kFetchWarps);
  if (c.p.dtype == SKV_DTYPE_BF16)
    k_fetch<bf16><<<grid, kFetchWarps * 32, 0, st>>>(
        static_cast<const bf16*>(c.v_cpu_dev), static_cast<bf16*>(c.slot_V), c.miss_chunk,
        c.miss_slot, c.miss_count, c.p.s, c.n, c.p.c, c.p.d, c.p.k, c.status);
  else
    k_fetch<float><<<grid, kFetchWarps * 32, 0, st>>>(
        static_cast<const float*>(c.v_cpu_dev), static_cast<float*>(c.slot_V), c.miss_chunk,
        c.miss_slot, c.miss_count, c.p.s, c.n, c.p.c, c.p.d, c.p.k, c.status);
  kend(c, K_FETCH, st);
  return cudaGetLastError();
}

size_t attn_smem_bytes(int G, int D, int S) {
  return sizeof(float) * (static_cast<size_t>(G) * D + static_cast<size_t>(G) * S);
}

template <typename T, int D, int G>
static cudaError_t attn_t(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st) {
  const int S = c.split_tokens;
  const int n_out = c.p.o * c.p.c, n_sp = c.p.k * c.p.c;
  const int T_all = n_out + n_sp + n_loc;
  const int nsplit = (T_all + S - 1) / S;
  if (nsplit > c.max_splits) return cudaErrorInvalidValue;
  const size_t smem = attn_smem_bytes(G, D, S);
  auto kern = k_attn<T, D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  kern<<<dim3(c.p.b * c.p.h_kv, nsplit), kAttnThreads, smem, st>>>(
      static_cast<const T*>(c.K_out), static_cast<const T*>(c.V_out),
      static_cast<const T*>(c.K_sparse), static_cast<const T*>(c.slot_V), c.sel_slot,
      static_cast<const T*>(c.K_loc), static_cast<const T*>(c.V_loc), static_cast<const T*>(q),
      static_cast<T*>(out), c.attn_part, c.attn_count, n_out, n_sp, n_loc, c.loc_cap, c.p.c,
      c.p.k, S, nsplit, c.max_splits, scale_log2);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t attn_d(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st) {
  switch (c.G) {
    case 1: return attn_t<T, D, 1>(c, q, out, n_loc, st);
    case 2: return attn_t<T, D, 2>(c, q, out, n_loc, st);
    case 4: return attn_t<T, D, 4>(c, q, out, n_loc, st);
    default: return attn_t<T, D, 8>(c, q, out, n_loc, st);
  }
}

cudaError_t launch_attn(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st) {
  kbegin(c, K_ATTN, st);
  cudaError_t e;
  if (c.p.dtype == SKV_DTYPE_BF16)
    e = c.p.d == 128 ? attn_d<bf16, 128>(c, q, out, n_loc, st) : attn_d<bf16, 64>(c, q, out, n_loc, st);
  else
    e = c.p.d == 128 ? attn_d<float, 128>(c, q, out, n_loc, st) : attn_d<float, 64>(c, q, out, n_loc, st);
  kend(c, K_ATTN, st);
  return e;
}

cudaError_t launch_build_mask(Ctx& c, cudaStream_t st) {
  kbegin(c, K_OUTLIERS, st);
  k_build_mask<<<c.p.b * c.p.h_kv, 256, 0, st>>>(c.out_ids, c.out_mask, c.n, c.p.o, c.status);
  kend(c, K_OUTLIERS, st);
  return cudaGetLastError();
}

}  // namespace skv
