// Decode-step kernels of ShadowKV (Algorithm 2 of the ShadowKV review page):
//   k_score   P = MatMul(Q, L^T) / sqrt(d), with per-tile softmax statistics
//   k_select  S2 and I = ArgTopK(S2, k) per KV head, the set difference
//             against the previous step's GPU-resident chunks, and the
//             local-window append of the new token
//   k_fetch   Gather(V_CPU, I) for the chunks that missed the cache, read
//             zero-copy from pinned host memory on the side stream (row-major
//             contexts; with K/V records the rebuild's launch does the fetch)
// (the attention kernels are in attn*.cu, the key rebuild in rebuild.cu)
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace skv {

constexpr int kScoreTile = 128;      // landmarks per score tile (one per thread)
constexpr int kSelectThreads = 1024;
// How far below the previous step's k-th largest S2 (a log softmax weight)
// the selection's first threshold try sits: the k-th S2 moved by at most
// 0.05 per step on the synthetic queries of the headline workload and by
// 0.24 at a hit rate of about 0.6
constexpr float kWarmMargin = 0.25f;
constexpr int kFetchWarps = 32;

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
    // per-warp (32-row) max and sum of exp over the valid rows, per head
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float m = warp_max(valid ? acc[g] : -INFINITY);
      const float e = warp_sum(valid ? __expf(acc[g] - m) : 0.f);
      if (lane == 0) part[((static_cast<size_t>(pair) * G + g) * ntile + ti) * 4 + warp] = make_float2(m, e);
    }
  }
}

// ----------------------------------------------------------------- select
// One block per (batch, KV head).  Shared memory: keys[n], then the cache
// bookkeeping arrays.
template <typename T, int D, int G, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT)
k_select(const float* __restrict__ P, const float2* __restrict__ part, const float* __restrict__ m8,
         const uint32_t* __restrict__ mask, int n, int ntile, int k, int group_reduce,
         int cache_on, int32_t* __restrict__ sel, int32_t* __restrict__ sel_slot,
         int32_t* __restrict__ slot_chunk, int32_t* __restrict__ miss_chunk,
         int32_t* __restrict__ miss_slot, int32_t* __restrict__ miss_total,
         int32_t* __restrict__ miss_base, int32_t* __restrict__ att_slot, int par,
         int32_t* __restrict__ hits, unsigned long long* __restrict__ counters,
         const T* __restrict__ k_new, const T* __restrict__ v_new, T* __restrict__ K_loc,
         T* __restrict__ V_loc, T* __restrict__ KV_loc, int loc_row, int loc_cap,
         uint32_t* __restrict__ warm_b, int* __restrict__ status) {
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
  int* scratch = align16(s_free + k);   // topk_scratch_ints(NT) ints, 16-byte aligned
  float* lse = reinterpret_cast<float*>(scratch + topk_scratch_ints(NT));  // G floats
  int* tmp = scratch;          // block scans after the top-k

  const int pair = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
  tc::grid_dep_launch();

  // append the new token's key/value to the local window (the score kernel,
  // which may still be finishing, does not touch it)
  if (k_new != nullptr) {
    for (int i = tid; i < D; i += nthr) {
      const size_t dst = (static_cast<size_t>(pair) * loc_cap + loc_row) * D + i;
      const T kv = k_new[static_cast<size_t>(pair) * D + i], vv = v_new[static_cast<size_t>(pair) * D + i];
      K_loc[dst] = kv;
      V_loc[dst] = vv;
      if (KV_loc != nullptr) {
        // the token's place in its group record: K tile, then V^T tile
        T* rec = KV_loc + (static_cast<size_t>(pair) * loc_cap + (loc_row & ~7)) * 2 * D;
        rec[(i >> 3) * 64 + (loc_row & 7) * 8 + (i & 7)] = kv;
        rec[1024 + (i >> 3) * 64 + (i & 7) * 8 + (loc_row & 7)] = vv;
      }
    }
  }
  for (int i = tid; i < k; i += nthr) s_hit[i] = 0;
  // this head's cache slots (written by the previous step's selection)
  int32_t* sc_row = slot_chunk + static_cast<size_t>(pair) * k;
  const int my_slot_chunk = cache_on && tid < k ? sc_row[tid] : -1;
  // the previous step's k-th largest S2 minus a margin, as a key (0: none)
  const uint32_t b_warm = warm_b != nullptr ? warm_b[pair] : 0u;
  uint32_t b_next = 0u;
  const int n8 = (n + 7) >> 3;
  const bool bounded = m8 != nullptr && group_reduce == 0 && 2 * n8 <= n && n8 <= 4 * nthr;
  // the bounded path's shared state (below); its counters and the bitmap of
  // the selection are set before the wait
  const int cap = 4 * nthr;
  uint32_t* bkey = keys;                                   // [n8] group bounds (0: no valid chunk)
  int* cand = reinterpret_cast<int*>(keys + n8);           // [n8] candidate groups
  uint32_t* vals = reinterpret_cast<uint32_t*>(scratch);  // survivors' keys
  int* vidx = scratch + cap;                               // their chunks
  int* ks = vidx + cap;                                    // block_kth scratch
  int* stmp = ks + (nthr / 32) * 256 + 256 + 8;            // scans; then +33..+39 below
  unsigned* bmax_slot = reinterpret_cast<unsigned*>(stmp + 33);   // largest non-zero bound
  unsigned* bmin_slot = reinterpret_cast<unsigned*>(stmp + 34);   // smallest non-zero bound
  unsigned* smax_slot = reinterpret_cast<unsigned*>(stmp + 35);   // largest survivor key
  int* cnt_slot = stmp + 36;
  int* nnz_slot = stmp + 38;
  int* ncand_slot = stmp + 39;
  if (bounded) {
    if (tid == 0) {
      *cnt_slot = *nnz_slot = *ncand_slot = 0;
      *bmax_slot = *smax_slot = 0u;
      *bmin_slot = 0xffffffffu;
    }
    for (int w = tid; w < nw; w += nthr) words[w] = 0u;
  }
  tc::grid_dep_wait();   // the logits and partials of the score kernel
  // with at most 2 groups per thread, their maxima are loaded before the
  // log-sum-exp, so that the two round trips overlap
  const bool pre = bounded && n8 <= 2 * nthr;
  float gm[2][G];
  if (pre) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int w = tid + u * nthr;
#pragma unroll
      for (int g = 0; g < G; ++g)
        gm[u][g] = w < n8 ? __ldcg(m8 + (static_cast<size_t>(pair) * G + g) * n8 + w) : -INFINITY;
    }
  }
  // log-sum-exp of each query head over the candidate chunks (4 partials
  // of 32 landmarks per 128-landmark score tile): a warp per head, one pass
  // (each lane's partials two per 16-byte load, in rounds of 8 loads: one
  // round up to 128K tokens at 8 per chunk; merged as (max, sum))
  for (int g = warp; g < G; g += nthr / 32) {
    const float4* pp = reinterpret_cast<const float4*>(part + (static_cast<size_t>(pair) * G + g) * ntile * 4);
    const int lim = 2 * ntile;
    float m = -INFINITY, z = 0.f;
    for (int t0 = 0; t0 < lim; t0 += 32 * 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int t = t0 + u * 32 + lane;
        v[u] = t < lim ? __ldcg(pp + t) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      }
      float mc = m;
#pragma unroll
      for (int u = 0; u < 8; ++u) mc = fmaxf(mc, fmaxf(v[u].x, v[u].z));
      float zc = z > 0.f ? z * __expf(m - mc) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (v[u].y > 0.f) zc += v[u].y * __expf(v[u].x - mc);
        if (v[u].w > 0.f) zc += v[u].w * __expf(v[u].z - mc);
      }
      m = mc;
      z = zc;
    }
    const float M = warp_max(m);
    z = warp_sum(z > 0.f ? z * __expf(m - M) : 0.f);
    if (lane == 0) lse[g] = M + __logf(z);
  }
  __syncthreads();
  const uint32_t* mk = mask + static_cast<size_t>(pair) * nw;
  // With the max reading of S2 and the score kernel's maxima of each 8
  // consecutive chunks, the top k is taken among few chunks: the bound of a
  // group, max over heads of (its max logit - lse), is the largest S2 of the
  // group; the k-th largest bound B is at most the k-th largest S2, so every
  // chunk of the top k lies in a group with bound >= B and has S2 >= B.  Only
  // those groups' chunks get keys; the top k of the ones with key >= B
  // (survivors), ties toward the lower index, is the answer.  Too many
  // candidates (massive ties) take the general path below.
  bool topk_done = false;
  if (bounded) {
    int nz = 0;
    uint32_t kmax = 0u, kmin = 0xffffffffu;
    // with a carried threshold (below) the groups that reach it are
    // compacted as candidates while the bounds are formed
    const bool warm = b_warm != 0u;
    auto put_bound = [&](int w, float bnd) {
      const uint32_t kb = w < n8 && bnd != -INFINITY ? order_key(bnd) : 0u;
      if (w < n8) bkey[w] = kb;
      if (kb != 0u) {
        ++nz;
        kmax = max(kmax, kb);
        kmin = min(kmin, kb);
      }
      if (warm) {
        const bool isc = kb != 0u && kb >= b_warm;
        const unsigned m = __ballot_sync(0xffffffffu, isc);
        int base = 0;
        if (lane == 0 && m) base = atomicAdd(ncand_slot, __popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (isc) cand[base + __popc(m & ((1u << lane) - 1u))] = w;
      }
    };
    if (pre) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int w = tid + u * nthr;
        float bnd = -INFINITY;
#pragma unroll
        for (int g = 0; g < G; ++g) bnd = fmaxf(bnd, gm[u][g] - lse[g]);
        put_bound(w, bnd);
      }
    } else {
      for (int w0 = 0; w0 < n8; w0 += nthr) {
        const int w = w0 + tid;
        float bnd = -INFINITY;
        if (w < n8) {
#pragma unroll
          for (int g = 0; g < G; ++g)
            bnd = fmaxf(bnd, __ldcg(m8 + (static_cast<size_t>(pair) * G + g) * n8 + w) - lse[g]);
        }
        put_bound(w, bnd);
      }
    }
    nz = __reduce_add_sync(0xffffffffu, nz);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    if (lane == 0 && nz) {
      atomicAdd(nnz_slot, nz);
      atomicMax(bmax_slot, kmax);
      atomicMin(bmin_slot, kmin);
    }
    __syncthreads();
    // The threshold B: first, when the previous step left one, its k-th
    // largest S2 minus a margin (that value moves little from step to step).
    // The chunks with S2 >= B are exactly the survivors below, so with at
    // least k of them the top k is among them; else (the first step, a
    // larger move) B is taken from the bounds as follows.
    for (int attempt = warm ? 0 : 1; attempt < 2 && !topk_done; ++attempt) {
    uint32_t B = 1u;    // fewer than k groups with a valid chunk: all of them are candidates
    if (attempt == 0) {
      B = b_warm;
    } else {
      if (warm) {
        // start over: every thread has read the first try's counts
        __syncthreads();
        if (tid == 0) {
          *cnt_slot = *ncand_slot = 0;
          *smax_slot = 0u;
        }
        __syncthreads();
      }
      if (*nnz_slot >= k) {
        // two 8-bit digits: B is the lower edge of the range that holds the
        // k-th largest bound, still a lower bound of the k-th largest S2
        // (the bounds' range is known)
        if (n8 <= 2048) block_kth_256<8>(bkey, n8, k, ks, 2, *bmin_slot, *bmax_slot);
        else block_kth_256<16>(bkey, n8, k, ks, 2, *bmin_slot, *bmax_slot);
        __syncthreads();
        B = static_cast<uint32_t>(ks[kKth8T]);
      }
    }
    // candidate groups, compacted by warps of 32 groups (the first try's
    // were compacted with the bounds)
    if (attempt == 1) {
    for (int w0 = warp * 32; w0 < n8; w0 += nthr) {
      const int w = w0 + lane;
      const bool isc = w < n8 && bkey[w] != 0u && bkey[w] >= B;
      const unsigned m = __ballot_sync(0xffffffffu, isc);
      int base = 0;
      if (lane == 0 && m) base = atomicAdd(ncand_slot, __popc(m));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (isc) cand[base + __popc(m & ((1u << lane) - 1u))] = w;
    }
    __syncthreads();
    }
    const int ne = *ncand_slot * 8;
    if (ne <= 2 * cap) {
      // the candidates' chunks, in rounds of 4 per thread: all loads of a
      // round issued before any key is formed; survivors appended by warp
      // ballots (at most cap of them are kept)
      uint32_t kept_max = 0u;
      for (int h0 = 0; h0 < ne; h0 += 4 * nthr) {
      float pv[4][G];
      int jj[4];
      uint32_t mw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = h0 + u * nthr + tid;
        jj[u] = -1;
        mw[u] = 0u;
        if (e < ne) {
          const int j = cand[e >> 3] * 8 + (e & 7);
          if (j < n) {
            jj[u] = j;
            mw[u] = mk[j >> 5];
#pragma unroll
            for (int g = 0; g < G; ++g) pv[u][g] = __ldcg(P + (static_cast<size_t>(pair) * G + g) * n + j);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (h0 + u * nthr >= ne) break;
        uint32_t key = 0u;
        if (jj[u] >= 0 && !((mw[u] >> (jj[u] & 31)) & 1u)) {
          float sm = -INFINITY;
#pragma unroll
          for (int g = 0; g < G; ++g) sm = fmaxf(sm, pv[u][g] - lse[g]);
          key = order_key(sm);
        }
        const bool keep = key != 0u && key >= B;
        if (keep) kept_max = max(kept_max, key);
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        int base = 0;
        if (lane == 0 && m) base = atomicAdd(cnt_slot, __popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        const int pos = base + __popc(m & ((1u << lane) - 1u));
        if (keep && pos < cap) {
          vals[pos] = key;
          vidx[pos] = jj[u];
        }
      }
      }
      kept_max = __reduce_max_sync(0xffffffffu, kept_max);
      if (lane == 0 && kept_max) atomicMax(smax_slot, kept_max);
      __syncthreads();
      const int nsurv = *cnt_slot;
      if (nsurv >= k && nsurv <= cap) {
        // Tk = the k-th largest survivor (all survivors lie in [B, their
        // largest key]); `need` of the survivors equal to Tk are taken
        // (every chunk equal to Tk is a survivor)
        const uint32_t shi = *smax_slot;
        if (nsurv <= 1024) block_kth_256<4>(vals, nsurv, k, ks, 4, B, shi, true);
        else if (nsurv <= 2048) block_kth_256<8>(vals, nsurv, k, ks, 4, B, shi, true);
        else block_kth_256<16>(vals, nsurv, k, ks, 4, B, shi, true);
        __syncthreads();
        const uint32_t Tk = static_cast<uint32_t>(ks[kKth8T]);
        const int need = ks[kKth8Need];
        b_next = max(order_key(from_order_key(Tk) - kWarmMargin), 1u);
        if (ks[kKth8Eq] == need) {
          for (int i = tid; i < nsurv; i += nthr)
            if (vals[i] >= Tk) atomicOr(&words[vidx[i] >> 5], 1u << (vidx[i] & 31));
        } else {
          // the survivors above Tk, then the `need` lowest chunks equal to Tk:
          // the need-th largest of n - chunk among those
          for (int i = tid; i < nsurv; i += nthr)
            if (vals[i] > Tk) atomicOr(&words[vidx[i] >> 5], 1u << (vidx[i] & 31));
          __syncthreads();
          for (int i = tid; i < nsurv; i += nthr) vals[i] = vals[i] == Tk ? static_cast<uint32_t>(n - vidx[i]) : 0u;
          __syncthreads();
          uint32_t R;
          int unused;
          block_kth(vals, nsurv, need, ks, &R, &unused);
          for (int i = tid; i < nsurv; i += nthr)
            if (vals[i] != 0u && vals[i] >= R) atomicOr(&words[vidx[i] >> 5], 1u << (vidx[i] & 31));
        }
        __syncthreads();
        bitmap_list(words, nw, s_sel, wpref, stmp);
        topk_done = true;
      }
    }
    }   // attempts
  }
  // selection keys: S2 per chunk, 0 for outliers
  auto key_of = [&](float sc_max, float sc_sum, bool excluded) -> uint32_t {
    if (excluded) return 0u;
    return group_reduce == 0 ? order_key(sc_max) : __float_as_uint(sc_sum) + 1u;
  };
  if (topk_done) {
  } else if ((n & 3) == 0) {
    // 16-byte loads of 4 consecutive chunks per head; a batch of IT x G loads
    // is issued before any key of the batch is computed
    constexpr int IT = G >= 8 ? 1 : 8 / G;
    const float4* P4 = reinterpret_cast<const float4*>(P + static_cast<size_t>(pair) * G * n);
    const int n4 = n >> 2;
    for (int jb = 0; jb < n4; jb += IT * nthr) {
      float4 v[IT][G];
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int j4 = jb + it * nthr + tid;
#pragma unroll
        for (int g = 0; g < G; ++g)
          v[it][g] = j4 < n4 ? __ldcg(P4 + static_cast<size_t>(g) * n4 + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int j4 = jb + it * nthr + tid;
        if (j4 >= n4) continue;
        const uint32_t mbits = mk[j4 >> 3] >> ((j4 & 7) * 4);
        uint32_t kq[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float smax = -INFINITY, ssum = 0.f;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float pv = e == 0 ? v[it][g].x : e == 1 ? v[it][g].y : e == 2 ? v[it][g].z : v[it][g].w;
            const float x = pv - lse[g];
            smax = fmaxf(smax, x);
            if (group_reduce) ssum += __expf(x);
          }
          kq[e] = key_of(smax, ssum, (mbits >> e) & 1u);
        }
        // one 16-byte store: four consecutive keys of a thread
        reinterpret_cast<uint4*>(keys)[j4] = make_uint4(kq[0], kq[1], kq[2], kq[3]);
      }
    }
  } else
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
  // the selection (ascending), its bitmap and per-word prefix popcounts
  if (!topk_done) {
    __syncthreads();
    block_topk(keys, n, k, s_sel, scratch, words, wpref);
  }
  // slots whose chunk is selected again keep it (hits); k <= blockDim.x
  int my_keep = 0;
  for (int i = tid; i < k; i += nthr) {
    int ch = my_slot_chunk;
    if (ch >= n) { flag_error(status, DEV_BAD_CHUNK); ch = -1; }
    int keep = 0;
    if (ch >= 0 && ((words[ch >> 5] >> (ch & 31)) & 1u)) {
      const int pos = wpref[ch >> 5] + __popc(words[ch >> 5] & ((1u << (ch & 31)) - 1u));
      s_slot[pos] = i;
      s_hit[pos] = 1;
      keep = 1;
    }
    s_keep[i] = keep;
    my_keep = keep;
  }
  // the head's misses (each kept slot is one hit): its range of the step's
  // compact miss list is reserved now, the atomic's round trip overlapping
  // the scan below; the block of head 0 also clears the other step
  // parity's counter for the next step
  const int nres = k - __syncthreads_count(my_keep);
  int base_r = 0;
  if (tid == 0) {
    base_r = atomicAdd(&miss_total[par], nres);
    if (pair == 0) miss_total[par ^ 1] = 0;
  }
  // the m-th missing chunk (ascending) takes the m-th freed slot (ascending)
  const int is_miss = tid < k ? !s_hit[tid] : 0;
  const int is_free = tid < k ? !s_keep[tid] : 0;
  // both ranks from one scan (counts < 2^16)
  int both;
  const int ranks = block_exclusive_scan(is_miss | (is_free << 16), tmp, &both, true);
  const int mrank = ranks & 0xffff, frank = ranks >> 16;
  const int nmiss = both & 0xffff, nfree = both >> 16;
  if (is_free) s_free[frank] = tid;
  // the attention's list of the selected chunks' slots: the kept slots in
  // ascending order (slot tid after the kept slots below it), then the
  // misses' slots (ascending too); consecutive slots hold adjacent records
  if (att_slot != nullptr && tid < k && !is_free)
    att_slot[static_cast<size_t>(pair) * k + tid - frank] = tid;
  // the reserved range's start (the atomic issued before the scan)
  __shared__ int s_base;
  if (tid == 0) {
    s_base = base_r;
    miss_base[pair] = base_r;
  }
  __syncthreads();
  if (nmiss != nfree || nmiss != nres) flag_error(status, DEV_BAD_COUNT);
  // (k <= blockDim.x: thread i writes selection entry i, its slot included)
  if (tid < k) {
    int slot = s_slot[tid];
    if (is_miss && mrank < nfree && mrank < nres) {
      slot = s_free[mrank];
      sc_row[slot] = s_sel[tid];
      miss_chunk[s_base + mrank] = pair * n + s_sel[tid];
      miss_slot[s_base + mrank] = pair * k + slot;
      if (att_slot != nullptr) att_slot[static_cast<size_t>(pair) * k + (k - nmiss) + mrank] = slot;
    }
    sel[static_cast<size_t>(pair) * k + tid] = s_sel[tid];
    sel_slot[static_cast<size_t>(pair) * k + tid] = slot;
  }
  if (tid == 0) {
    if (warm_b != nullptr) warm_b[pair] = b_next;
    hits[pair] = k - nmiss;
    atomicAdd(&counters[0], static_cast<unsigned long long>(k - nmiss));
    atomicAdd(&counters[1], static_cast<unsigned long long>(nmiss));
  }
}

// ------------------------------------------------------------------ fetch
// The step's misses form one compact list (entries pair * n + chunk and
// pair * k + slot, count miss_total[par]).  A small fixed grid (fetch_sms
// blocks of 32 warps, enough loads in flight to fill the host link) walks it,
// a warp per chunk: c*d elements read from pinned host memory through its
// mapped device address into the chunk's cache slot.  The key rebuild,
// running alongside, leaves those SMs free.
template <typename T>
__global__ void __launch_bounds__(kFetchWarps * 32)
k_fetch(const T* __restrict__ vcpu, T* __restrict__ slot_V, const int32_t* __restrict__ miss_chunk,
        const int32_t* __restrict__ miss_slot, const int32_t* __restrict__ miss_total, int par, int s,
        int n, int c, int d, int k, int npairs, int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int w0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  int total = miss_total[par];
  if (total > npairs * k) {
    if (w0 == 0 && lane == 0) flag_error(status, DEV_BAD_COUNT);
    total = npairs * k;
  }
  const int nvec = c * d * static_cast<int>(sizeof(T)) / 16;
  for (int m = w0; m < total; m += nwarps) {
    const int pc = miss_chunk[m], ps = miss_slot[m];
    const int pair = pc / n, chunk = pc - pair * n;
    const int slot = ps - pair * k;
    if (pair < 0 || pair >= npairs || chunk < 0 || slot < 0 || slot >= k) {
      if (lane == 0) flag_error(status, DEV_BAD_SLOT);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(vcpu + (static_cast<size_t>(pair) * s + static_cast<size_t>(chunk) * c) * d);
    uint4* dst = reinterpret_cast<uint4*>(slot_V + ((static_cast<size_t>(pair) * k + slot) * c) * d);
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
}

// Fetch into slot records (bf16, d = 128): a half-warp per 8-token group,
// lane q reading the 16-byte piece q of the group's 8 rows from pinned host
// memory and writing the V^T half of the group's record (one 128-byte run per
// lane).
__global__ void __launch_bounds__(kFetchWarps * 32)
k_fetch_rec(const bf16* __restrict__ vcpu, bf16* __restrict__ KV_slot, const int32_t* __restrict__ miss_chunk,
              const int32_t* __restrict__ miss_slot, const int32_t* __restrict__ miss_total, int par, int s,
              int n, int c, int k, int npairs, int* __restrict__ status) {
  fetch_value_groups(vcpu, KV_slot, miss_chunk, miss_slot, miss_total[par], s, n, c, k, npairs,
                     static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x,
                     static_cast<long long>(gridDim.x) * blockDim.x, status);
}

// Records of row-major [rows][128] bf16 keys and values (rows a multiple of
// 8): a half-warp per 8-token group, lane q moving the 16-byte piece q of the
// group's key rows into the K tile (pieces ordered [q][row]) and the
// transposed values into the V^T tile.
__global__ void __launch_bounds__(256)
k_pack_kv(const bf16* __restrict__ K, const bf16* __restrict__ V, bf16* __restrict__ KV, long long groups) {
  const int lane = threadIdx.x & 31, q = lane & 15;
  const long long h0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const long long nh = (static_cast<long long>(gridDim.x) * blockDim.x) >> 4;
  for (long long g = h0; g < groups; g += nh) {
    const uint4* ks = reinterpret_cast<const uint4*>(K + g * 1024);
    const uint4* vs = reinterpret_cast<const uint4*>(V + g * 1024);
    uint4* rec = reinterpret_cast<uint4*>(KV + g * 2048);
    uint4 in[8], outv[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) rec[q * 8 + t] = ks[t * 16 + q];
#pragma unroll
    for (int t = 0; t < 8; ++t) in[t] = vs[t * 16 + q];
    transpose8x8(in, outv);
#pragma unroll
    for (int r = 0; r < 8; ++r) rec[128 + q * 8 + r] = outv[r];
  }
}

cudaError_t launch_pack_kv(Ctx& c, cudaStream_t st) {
  if (!c.kv_rec) return cudaSuccess;
  const long long pairs = static_cast<long long>(c.p.b) * c.p.h_kv;
  const long long g_out = pairs * c.p.o * c.p.c / 8, g_loc = pairs * c.loc_cap / 8;
  kbegin(c, K_MISC, st);
  if (g_out > 0)
    k_pack_kv<<<static_cast<int>(std::min<long long>((g_out + 15) / 16, 8LL * c.nsm)), 256, 0, st>>>(
        static_cast<const bf16*>(c.K_out), static_cast<const bf16*>(c.V_out), static_cast<bf16*>(c.KV_out), g_out);
  k_pack_kv<<<static_cast<int>(std::min<long long>((g_loc + 15) / 16, 8LL * c.nsm)), 256, 0, st>>>(
      static_cast<const bf16*>(c.K_loc), static_cast<const bf16*>(c.V_loc), static_cast<bf16*>(c.KV_loc), g_loc);
  kend(c, K_MISC, st);
  return cudaGetLastError();
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
  const cudaError_t et = launch_score_tc(c, q, st);
  if (et != cudaErrorNotSupported) {
    kend(c, K_SCORE, st);
    return et;
  }
  if (c.p.dtype == SKV_DTYPE_BF16) {
    if (c.p.d == 128) score_d<bf16, 128>(c, q, st); else score_d<bf16, 64>(c, q, st);
  } else {
    if (c.p.d == 128) score_d<float, 128>(c, q, st); else score_d<float, 64>(c, q, st);
  }
  kend(c, K_SCORE, st);
  return cudaGetLastError();
}

size_t select_smem_bytes(int n, int k, int G, int nthreads) {
  const int nw = (n + 31) / 32;
  return sizeof(uint32_t) * (static_cast<size_t>(n) + 2 * nw) +
         sizeof(int) * (5 * static_cast<size_t>(k) + topk_scratch_ints(nthreads)) + sizeof(float) * G + 16;
}

template <typename T, int D, int G>
static cudaError_t select_t(Ctx& c, const void* k_new, const void* v_new, int loc_row,
                            cudaStream_t st) {
  // more heads than SMs: 512-thread CTAs, two per SM (each thread keeps one
  // cache slot, so k <= 512); else one 1024-thread CTA per head
  constexpr bool kHalf = std::is_same<T, bf16>::value && D == 128;
  const bool half = kHalf && c.p.b * c.p.h_kv > c.nsm && c.p.k <= kSelectThreads / 2;
  const int nt = half ? kSelectThreads / 2 : kSelectThreads;
  const size_t smem = select_smem_bytes(c.n, c.p.k, c.G, nt);
  auto kern = half ? k_select<T, D, G, (kHalf ? kSelectThreads / 2 : kSelectThreads)> : k_select<T, D, G, kSelectThreads>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(c.p.b * c.p.h_kv), dim3(nt), smem, st,
      c.logits, c.score_part, static_cast<const float*>(c.m8_step == c.t ? c.score_m8 : nullptr), c.out_mask,
      c.n, c.ntile, c.p.k, c.p.group_reduce,
      c.cache_on ? 1 : 0, c.sel, c.sel_slot, c.slot_chunk, c.miss_chunk, c.miss_slot,
      c.miss_count, c.miss_base, c.att_slot, static_cast<int>(c.t & 1), c.hits, c.counters, static_cast<const T*>(k_new),
      static_cast<const T*>(v_new),
      static_cast<T*>(c.K_loc), static_cast<T*>(c.V_loc), static_cast<T*>(c.KV_loc), loc_row, c.loc_cap,
      c.warm_b, c.status);
}

template <typename T, int D>
static cudaError_t select_g(Ctx& c, const void* k_new, const void* v_new, int loc_row, cudaStream_t st) {
  switch (c.G) {
    case 1: return select_t<T, D, 1>(c, k_new, v_new, loc_row, st);
    case 2: return select_t<T, D, 2>(c, k_new, v_new, loc_row, st);
    case 4: return select_t<T, D, 4>(c, k_new, v_new, loc_row, st);
    default: return select_t<T, D, 8>(c, k_new, v_new, loc_row, st);
  }
}

cudaError_t launch_select(Ctx& c, const void* k_new, const void* v_new, int loc_row,
                          cudaStream_t st) {
  kbegin(c, K_SELECT, st);
  cudaError_t e;
  if (c.p.dtype == SKV_DTYPE_BF16)
    e = c.p.d == 128 ? select_g<bf16, 128>(c, k_new, v_new, loc_row, st)
                     : select_g<bf16, 64>(c, k_new, v_new, loc_row, st);
  else
    e = c.p.d == 128 ? select_g<float, 128>(c, k_new, v_new, loc_row, st)
                     : select_g<float, 64>(c, k_new, v_new, loc_row, st);
  kend(c, K_SELECT, st);
  return e;
}

cudaError_t launch_fetch(Ctx& c, cudaStream_t st) {
  kbegin(c, K_FETCH, st);
  const int par = static_cast<int>(c.t & 1);
  const int npairs = c.p.b * c.p.h_kv;
  if (c.kv_rec)
    k_fetch_rec<<<std::min(c.nsm, c.fetch_sms), kFetchWarps * 32, 0, st>>>(
        static_cast<const bf16*>(c.v_cpu_dev), static_cast<bf16*>(c.KV_slot), c.miss_chunk,
        c.miss_slot, c.miss_count, par, c.p.s, c.n, c.p.c, c.p.k, npairs, c.status);
  else if (c.p.dtype == SKV_DTYPE_BF16)
    k_fetch<bf16><<<std::min(c.nsm, c.fetch_sms), kFetchWarps * 32, 0, st>>>(
        static_cast<const bf16*>(c.v_cpu_dev), static_cast<bf16*>(c.slot_V), c.miss_chunk,
        c.miss_slot, c.miss_count, par, c.p.s, c.n, c.p.c, c.p.d, c.p.k, npairs, c.status);
  else
    k_fetch<float><<<std::min(c.nsm, c.fetch_sms), kFetchWarps * 32, 0, st>>>(
        static_cast<const float*>(c.v_cpu_dev), static_cast<float*>(c.slot_V), c.miss_chunk,
        c.miss_slot, c.miss_count, par, c.p.s, c.n, c.p.c, c.p.d, c.p.k, npairs, c.status);
  kend(c, K_FETCH, st);
  return cudaGetLastError();
}

cudaError_t launch_build_mask(Ctx& c, cudaStream_t st) {
  kbegin(c, K_OUTLIERS, st);
  k_build_mask<<<c.p.b * c.p.h_kv, 256, 0, st>>>(c.out_ids, c.out_mask, c.n, c.p.o, c.status);
  kend(c, K_OUTLIERS, st);
  return cudaGetLastError();
}

}  // namespace skv
