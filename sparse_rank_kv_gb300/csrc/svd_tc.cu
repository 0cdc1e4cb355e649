// Rank-r SVD of each sequence's pre-RoPE key matrix for bf16 contexts
// (Algorithm 1 step 1 of the ShadowKV review: A, B <- SVD(K)), through the
// Gram matrix on the tensor cores.
//
// M_b[t][h d + e] = K[b][h][t][e] is s x D (D = h_kv d).  The keys are bf16,
// so every product M[t][i] M[t][j] is exact in fp32; the Gram matrix
// G_b = M_b^T M_b is accumulated by tcgen05.mma in fp32 over splits of
// s_z tokens (the accumulator sees one split only) and the splits are summed
// in fp64, which keeps G's error far below the smallest eigenvalues that
// matter.  The right singular subspace of M_b is then the top-r invariant
// subspace of G_b (D x D, small): subspace iteration X <- orth(X G) from a
// seeded Gaussian start, each orthonormalisation a shifted CholeskyQR3
// (Fukaya, Kannan, Nakatsukasa, Zhang and Yamamoto, "Shifted Cholesky QR for
// computing the QR factorization of ill-conditioned matrices", SIAM J. Sci.
// Comput. 42 (2020)): a first pass whose Gram matrix and Cholesky factor are
// fp64, with a small diagonal shift, then two plain passes in fp32.  A = M X^T and B = X (split per KV head) follow;
// only the product A B is unique.
//
//   k_transpose_m  K (b h_kv) x s x d -> MT b x D x s (tokens contiguous), so
//                  both Gram operands are K-major
//   k_gram_tc      persistent; warp 0 TMA (two 128 x 64 token tiles of MT per
//                  stage, 128-byte swizzle), warp 1 tcgen05.mma (M = N = 128,
//                  K = 16) into two TMEM accumulators, warps 2-5 write each
//                  unit's 128 x 128 fp32 partial.  Units: (sequence, split,
//                  tile pair i <= j) with the pair fastest, so the CTAs
//                  working at once share tiles in L2.
//   k_gram_reduce  G[i][j] = sum over splits in fp64 (the (min, max) entry for
//                  both triangles, so G is exactly symmetric)
//   k_gemm_xg      Y = X G (fp32, 64 x 64 tiles)
//   k_syrk         W = Y Y^T in the pass's precision
//   k_chol         W = L L^T in place, one CTA per sequence (shift on pass 1)
//   k_trsm         Q = L^-1 Y in fp32, eight lanes per column of Y
#include <cudaTypedefs.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace skv {

constexpr int kGmTile = 128;
constexpr int kGmStages = 6;
constexpr int kGmThreads = 192;                         // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kGmStageBytes = 2 * kGmTile * 128;        // two 128 x 64 bf16 tiles
constexpr int kGmSmem = 1024 + 1024 + kGmStages * kGmStageBytes;
constexpr int kGmSplitTokens = 16384;                   // tokens per fp32 accumulation, at most

// ---------------------------------------------------------------- transpose
// One CTA moves a 64-token x 64-dimension block of one (sequence, KV head):
// rows of 128 bytes in, rows of 128 bytes out, through shared memory.
__global__ void __launch_bounds__(256)
k_transpose_m(const bf16* __restrict__ K, bf16* __restrict__ MT, int h, int s, int d) {
  __shared__ __align__(16) bf16 tile[64][64 + 8];
  const int t0 = blockIdx.x * 64, e0 = blockIdx.y * 64, pair = blockIdx.z;
  const int seq = pair / h, hh = pair - seq * h;
  const int tid = threadIdx.x;
  const bf16* src = K + (static_cast<size_t>(pair) * s + t0) * d + e0;
  for (int i = tid; i < 64 * 8; i += 256) {
    const int tr = i >> 3, ch = i & 7;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (t0 + tr < s) v = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(tr) * d + ch * 8);
    *reinterpret_cast<uint4*>(&tile[tr][ch * 8]) = v;
  }
  __syncthreads();
  const int D = h * d;
  bf16* dst = MT + (static_cast<size_t>(seq) * D + hh * d + e0) * s + t0;
  for (int i = tid; i < 64 * 8; i += 256) {
    const int er = i >> 3, ch = i & 7;      // dimension row, 8-token piece
    if (t0 + ch * 8 >= s) continue;          // s is a multiple of 8
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t lo = __bfloat16_as_ushort(tile[ch * 8 + 2 * q][er]);
      const uint32_t hi = __bfloat16_as_ushort(tile[ch * 8 + 2 * q + 1][er]);
      w[q] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(er) * s + ch * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ------------------------------------------------------------- Gram (tcgen05)
__device__ __forceinline__ void gram_pair(int p, int ntile, int* ti, int* tj) {
  int i = 0;
  while (p >= ntile - i) {
    p -= ntile - i;
    ++i;
  }
  *ti = i;
  *tj = i + p;
}

__global__ void __launch_bounds__(kGmThreads, 1)
k_gram_tc(const __grid_constant__ CUtensorMap mapMT, float* __restrict__ part, int D, int ntile,
          int npairs, int nz, int kb_per_z, int nkb, int nunits, int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kGmStages;
  uint64_t* tfull = empty + kGmStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* s_consumed = reinterpret_cast<int*>(tmem_slot + 1);
  unsigned char* stages = smem + 1024;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tc::prefetch_tensormap(&mapMT);
    for (int s = 0; s < kGmStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&tfull[a], 1);
      tc::mbar_init(&tempty[a], 128);
    }
    tc::mbar_init(drain, 1);
    *s_consumed = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 2 * kGmTile);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  int issued = 0;

  auto unit_of = [&](int u, int* seq, int* z, int* ti, int* tj) {
    const int pr = u % npairs;
    const int sz = u / npairs;
    *z = sz % nz;
    *seq = sz / nz;
    gram_pair(pr, ntile, ti, tj);
  };

  if (warp == 0) {
    if (lane == 0) {
      for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
        int seq, z, ti, tj;
        unit_of(u, &seq, &z, &ti, &tj);
        const int kb0 = z * kb_per_z, kb1 = min(nkb, kb0 + kb_per_z);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb, ++issued) {
          const int s = issued % kGmStages;
          if (!tc::mbar_wait(&empty[s], ((issued / kGmStages) & 1) ^ 1, kWaitLimit)) {
            flag_error(status, DEV_TIMEOUT);
            ok = false;
            break;
          }
          tc::mbar_expect_tx(&full[s], kGmStageBytes);
          unsigned char* st = stages + s * kGmStageBytes;
          tc::tma_load_2d(st, &mapMT, &full[s], kb * 64, seq * D + ti * kGmTile);
          tc::tma_load_2d(st + kGmTile * 128, &mapMT, &full[s], kb * 64, seq * D + tj * kGmTile);
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kGmTile, kGmTile);
      int it = 0, ul = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++ul) {
        int seq, z, ti, tj;
        unit_of(u, &seq, &z, &ti, &tj);
        const int kb0 = z * kb_per_z, kb1 = min(nkb, kb0 + kb_per_z);
        const int acc = ul & 1;
        if (!tc::mbar_wait(&tempty[acc], ((ul >> 1) & 1) ^ 1, kWaitLimit)) {
          flag_error(status, DEV_TIMEOUT);
          break;
        }
        tc::fence_after();
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % kGmStages;
          if (!tc::mbar_wait(&full[s], (it / kGmStages) & 1, kWaitLimit)) {
            flag_error(status, DEV_TIMEOUT);
            ok = false;
            break;
          }
          tc::fence_after();
          const uint32_t a0 = tc::smem_u32(stages + s * kGmStageBytes);
          const uint32_t b0 = a0 + kGmTile * 128;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16(tmem + acc * kGmTile, tc::desc_k_sw128(a0 + kk * 32, 1024),
                         tc::desc_k_sw128(b0 + kk * 32, 1024), idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
          tc::mma_commit(&empty[s]);
        }
        if (ok) tc::mma_commit(&tfull[acc]);
      }
      *s_consumed = it;
      // every MMA this thread issued has completed before TMEM is released
      tc::mma_commit(drain);
      if (!tc::mbar_wait(drain, 0, kWaitLimit)) flag_error(status, DEV_TIMEOUT);
    }
  } else {
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    int ul = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++ul) {
      const int acc = ul & 1;
      const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&tfull[acc], (ul >> 1) & 1, kWaitLimit));
      if (!ok) {
        if (lane == 0) flag_error(status, DEV_TIMEOUT);
        break;
      }
      tc::fence_after();
      float* dst = part + (static_cast<size_t>(u) * kGmTile + row) * kGmTile;
#pragma unroll 1
      for (int c = 0; c < kGmTile / 32; ++c) {
        float v[32];
        tc::tmem_ld32(tmem + (static_cast<uint32_t>(q4 * 32) << 16) + acc * kGmTile + c * 32, v);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(dst + c * 32 + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
      tc::fence_before();
      tc::mbar_arrive(&tempty[acc]);
    }
  }
  tc::fence_before();
  __syncthreads();
  // copies the MMA warp did not consume (a timeout) land before the CTA exits
  if (warp == 0 && lane == 0) {
    for (int it = *s_consumed; it < issued; ++it)
      if (!tc::mbar_wait(&full[it % kGmStages], (it / kGmStages) & 1, kWaitLimit)) {
        flag_error(status, DEV_TIMEOUT);
        break;
      }
  }
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * kGmTile);
}

// G[seq][i][j] = sum_z part[(seq, z, pair(ti, tj))][i % 128][j % 128] in fp64,
// with (i, j) taken as (min, max) so that G is exactly symmetric.
__global__ void k_gram_reduce(const float* __restrict__ part, float* __restrict__ G, int b, int D,
                              int ntile, int npairs, int nz) {
  const size_t total = static_cast<size_t>(b) * D * D;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int seq = static_cast<int>(idx / (static_cast<size_t>(D) * D));
    const int rem = static_cast<int>(idx - static_cast<size_t>(seq) * D * D);
    int i = rem / D, j = rem - (rem / D) * D;
    if (i > j) { const int t = i; i = j; j = t; }
    const int ti = i / kGmTile, tj = j / kGmTile;
    const int p = ti * ntile - ti * (ti - 1) / 2 + (tj - ti);
    double acc = 0.0;
    for (int z = 0; z < nz; ++z) {
      const size_t u = (static_cast<size_t>(seq) * nz + z) * npairs + p;
      acc += static_cast<double>(__ldcs(part + (u * kGmTile + (i - ti * kGmTile)) * kGmTile + (j - tj * kGmTile)));
    }
    G[idx] = static_cast<float>(acc);
  }
}

// ------------------------------------------------------------- small GEMM
// Y[seq] = X[seq] G[seq]: X r x D, G D x D (symmetric); 64 x 64 tiles,
// 4 x 4 outputs per thread, fp32.
__global__ void __launch_bounds__(256)
k_gemm_xg(const float* __restrict__ X, const float* __restrict__ G, float* __restrict__ Y, int r, int D) {
  __shared__ __align__(16) float Xs[16][68];
  __shared__ __align__(16) float Gs[16][68];
  const int seq = blockIdx.z;
  const float* Xb = X + static_cast<size_t>(seq) * r * D;
  const float* Gb = G + static_cast<size_t>(seq) * D * D;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < D; k0 += 16) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = tid + 256 * q;
      const int rr = e >> 4, kk = e & 15;          // X rows i0 + rr, columns k0 + kk
      Xs[kk][rr] = (i0 + rr < r) ? Xb[static_cast<size_t>(i0 + rr) * D + k0 + kk] : 0.f;
      const int kr = e >> 6, cc = e & 63;          // G rows k0 + kr, columns j0 + cc
      Gs[kr][cc] = Gb[static_cast<size_t>(k0 + kr) * D + j0 + cc];
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&Xs[kk][ty * 4]);
      const float4 g = *reinterpret_cast<const float4*>(&Gs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], gv[v], acc[u][v]);
    }
    __syncthreads();
  }
  float* Yb = Y + static_cast<size_t>(seq) * r * D;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + ty * 4 + u;
    if (i >= r) continue;
    *reinterpret_cast<float4*>(Yb + static_cast<size_t>(i) * D + j0 + tx * 4) =
        make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
  }
}

// ------------------------------------------------------ shifted CholeskyQR
constexpr int kSyrkSplit = 4;   // slices of D: W = sum of kSyrkSplit partial Gram matrices

// Wp[slice][seq] = Y_slice Y_slice^T (r x r) accumulated in S over the
// slice's D / kSyrkSplit columns; tiles of 32 x 32 above the diagonal,
// mirrored.  The Cholesky kernel sums the slices in a fixed order.
template <typename S>
__global__ void __launch_bounds__(256)
k_syrk(const float* __restrict__ Y, S* __restrict__ Wp, int r, int D, int b) {
  const int bi = blockIdx.y, bj = blockIdx.x;
  if (bi > bj) return;
  __shared__ S Ys[2][32][33];
  const int seq = blockIdx.z % b, slice = blockIdx.z / b;
  const int dper = D / kSyrkSplit, d0 = slice * dper;
  const float* Yb = Y + static_cast<size_t>(seq) * r * D;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  S acc[2][2] = {};
  for (int k0 = d0; k0 < d0 + dper; k0 += 32) {
    for (int e = tid; e < 2 * 32 * 32; e += 256) {
      const int w = e >> 10, rr = (e >> 5) & 31, kk = e & 31;
      const int row = (w ? bj : bi) * 32 + rr;
      Ys[w][rr][kk] = (row < r) ? static_cast<S>(Yb[static_cast<size_t>(row) * D + k0 + kk]) : S(0);
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk)
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int v = 0; v < 2; ++v) acc[u][v] += Ys[0][ty * 2 + u][kk] * Ys[1][tx * 2 + v][kk];
    __syncthreads();
  }
  S* Wb = Wp + (static_cast<size_t>(slice) * b + seq) * r * r;
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const int i = bi * 32 + ty * 2 + u, j = bj * 32 + tx * 2 + v;
      if (i < r && j < r) {
        Wb[static_cast<size_t>(i) * r + j] = acc[u][v];
        Wb[static_cast<size_t>(j) * r + i] = acc[u][v];
      }
    }
}

// Cholesky W = L L^T of W = sum of the kSyrkSplit partials Wp[slice][seq],
// one CTA (1024 threads) per sequence, on a shared-memory copy of the packed
// lower triangle when it fits (else in place in the first partial); L is left
// in the lower triangle of the first partial.  With `shift`, the diagonal
// first gets 11 (D r + r (r + 1)) u tr(W) added (u the unit roundoff of S),
// the shift of shifted CholeskyQR.  Per column: the scaled column into a
// vector, then the trailing update, during which the thread that finishes
// the next pivot also takes its square root (two barriers per column).  A
// zero W (zero keys) becomes the identity; any other non-positive pivot is
// reported.
__host__ __device__ constexpr size_t chol_tri(int r) { return static_cast<size_t>(r) * (r + 1) / 2; }
constexpr int kCholThreads = 1024;

template <typename S>
__global__ void __launch_bounds__(kCholThreads)
k_chol(S* __restrict__ Wp, int r, int D, int b, int shift, int in_smem, int* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char csm[];
  const int seq = blockIdx.x;
  const size_t rr = static_cast<size_t>(r) * r;
  S* Wg = Wp + static_cast<size_t>(seq) * rr;                 // slice 0: holds W, then L
  S* T = reinterpret_cast<S*>(csm);                           // packed lower triangle, row i at i (i + 1) / 2
  S* col = T + (in_smem ? chol_tri(r) : 0);                   // scaled column j
  __shared__ S red[kCholThreads / 32];
  __shared__ S s_inv;
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kCholThreads / 32;
  auto at = [&](int i, int k) -> S& {
    return in_smem ? T[static_cast<size_t>(i) * (i + 1) / 2 + k] : Wg[static_cast<size_t>(i) * r + k];
  };
  // W = sum of the slices (fixed order), lower triangle
  for (int i = warp; i < r; i += NW)
    for (int k = lane; k <= i; k += 32) {
      S w = Wg[static_cast<size_t>(i) * r + k];
      for (int sl = 1; sl < kSyrkSplit; ++sl) w += Wp[(static_cast<size_t>(sl) * b + seq) * rr + static_cast<size_t>(i) * r + k];
      if (in_smem) T[static_cast<size_t>(i) * (i + 1) / 2 + k] = w;
      else Wg[static_cast<size_t>(i) * r + k] = w;
    }
  __syncthreads();
  S tr = 0;
  for (int i = tid; i < r; i += kCholThreads) tr += at(i, i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tr += __shfl_xor_sync(0xffffffffu, tr, o);
  if (lane == 0) red[warp] = tr;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  S trace = 0;
  for (int w = 0; w < NW; ++w) trace += red[w];
  if (trace == S(0)) {
    for (int e = tid; e < r * r; e += kCholThreads) Wg[e] = (e / r == e % r) ? S(1) : S(0);
    return;
  }
  if (shift) {
    const S u = sizeof(S) == 8 ? S(1.1102230246251565e-16) : S(5.9604645e-08);
    const S sh = S(11) * (static_cast<S>(D) * r + static_cast<S>(r) * (r + 1)) * u * trace;
    for (int i = tid; i < r; i += kCholThreads) at(i, i) += sh;
  }
  __syncthreads();
  auto pivot = [&](int j) {
    S dj = at(j, j);
    if (!(dj > S(0))) {
      s_bad = 1;
      dj = S(1);
    }
    const S lj = sqrt(dj);
    at(j, j) = lj;
    s_inv = S(1) / lj;
  };
  if (tid == 0) pivot(0);
  __syncthreads();
  for (int j = 0; j < r; ++j) {
    const S inv = s_inv;
    S* cj = in_smem ? col : nullptr;
    for (int i = j + 1 + tid; i < r; i += kCholThreads) {
      const S l = at(i, j) * inv;
      at(i, j) = l;
      if (cj) cj[i] = l;
    }
    __syncthreads();
    // trailing update of the lower triangle, row i handled by a warp; the
    // lane that finishes (j + 1, j + 1) takes the next pivot
    for (int i = j + 1 + warp; i < r; i += NW) {
      const S lij = cj ? cj[i] : at(i, j);
      for (int k = j + 1 + lane; k <= i; k += 32) {
        at(i, k) -= lij * (cj ? cj[k] : at(k, j));
        if (i == j + 1 && k == j + 1) pivot(j + 1);
      }
    }
    __syncthreads();
  }
  if (in_smem) {
    for (int i = warp; i < r; i += NW)
      for (int k = lane; k <= i; k += 32) Wg[static_cast<size_t>(i) * r + k] = T[static_cast<size_t>(i) * (i + 1) / 2 + k];
  }
  if (tid == 0 && s_bad) flag_error(status, DEV_NUMERIC);
}

// Q = L^-1 Y by forward substitution in fp32: eight lanes per column of Y
// (32 columns per 256-thread CTA), each summing every eighth term of a row's
// inner product, combined by shuffles; L's packed lower triangle (rounded to
// fp32) and the columns' results in shared memory.  After the shifted first
// pass cond(L) is a few thousand at most, so fp32 substitution leaves Q
// orthogonal to ~1e-3 or better, which the two plain passes that follow
// remove.
constexpr int kTrCols = 32;
template <typename S>
__global__ void __launch_bounds__(256) k_trsm(const S* __restrict__ L, const float* __restrict__ Y,
                                               float* __restrict__ Q, int r, int D) {
  extern __shared__ __align__(16) unsigned char tsm[];
  float* Lp = reinterpret_cast<float*>(tsm);             // packed lower triangle, row i at i (i + 1) / 2
  float* q = Lp + (chol_tri(r) + 3) / 4 * 4;             // [r][kTrCols]
  const int seq = blockIdx.y, tid = threadIdx.x;
  const int lc = tid >> 3, part = tid & 7;               // column within the CTA, lane within the column
  const int c = blockIdx.x * kTrCols + lc;
  const S* Lb = L + static_cast<size_t>(seq) * r * r;
  for (int e = tid; e < r * r; e += 256) {
    const int i = e / r, k = e - (e / r) * r;
    if (k <= i) Lp[static_cast<size_t>(i) * (i + 1) / 2 + k] = static_cast<float>(Lb[e]);
  }
  __syncthreads();
  const bool live = c < D;
  const float* Yb = Y + static_cast<size_t>(seq) * r * D;
  float* Qb = Q + static_cast<size_t>(seq) * r * D;
  // the CTA's columns of Y, loaded once; row i's entry is replaced by the
  // solution once it is known (it is read only for the rows after it)
  const int c0 = blockIdx.x * kTrCols;
  for (int e = tid; e < r * kTrCols; e += 256) {
    const int i = e / kTrCols, cc = e - (e / kTrCols) * kTrCols;
    q[e] = c0 + cc < D ? Yb[static_cast<size_t>(i) * D + c0 + cc] : 0.f;
  }
  __syncthreads();
  for (int i = 0; i < r; ++i) {
    const float* Li = Lp + static_cast<size_t>(i) * (i + 1) / 2;
    float a = 0.f;
    for (int k = part; k < i; k += 8) a = fmaf(Li[k], q[k * kTrCols + lc], a);
    a += __shfl_xor_sync(0xffffffffu, a, 1);
    a += __shfl_xor_sync(0xffffffffu, a, 2);
    a += __shfl_xor_sync(0xffffffffu, a, 4);
    const float x = (q[i * kTrCols + lc] - a) / Li[i];
    __syncwarp();
    if (part == 0) {
      q[i * kTrCols + lc] = x;
      if (live) Qb[static_cast<size_t>(i) * D + c] = x;
    }
    __syncwarp();
  }
}

static size_t trsm_smem(int r) { return ((chol_tri(r) + 3) / 4 * 4 + static_cast<size_t>(r) * kTrCols) * sizeof(float); }

// ------------------------------------------------------- A = M X^T (tcgen05)
// Unit = 128 tokens of one sequence.  Per 64-dimension block of M (one KV
// head's 64 dimensions): the 128 x 64 key tile by a 3D TMA box of K, and the
// r x 64 blocks of the basis' bf16 hi and lo parts; tcgen05.mma M = 128,
// N = r, K = 16 adds M Xh^T and M Xl^T into one fp32 accumulator (the
// products are exact, the basis keeps ~16 significant bits).  Two TMEM
// accumulators; warps 2-5 turn each row into bf16 A.
constexpr int kFaThreads = 192;

__host__ __device__ constexpr int fa_stage_bytes(int r) { return kGmTile * 128 + 2 * r * 128; }
__host__ __device__ constexpr int fa_stages(int r) {
  return (225 * 1024 - 2048) / fa_stage_bytes(r) < 4 ? (225 * 1024 - 2048) / fa_stage_bytes(r) : 4;
}
__host__ __device__ constexpr int fa_acc_cols(int r) { return r <= 128 ? 128 : 256; }

__global__ void __launch_bounds__(kFaThreads, 1)
k_factor_a_tc(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapXh,
              const __grid_constant__ CUtensorMap mapXl, bf16* __restrict__ A, int h, int s, int d, int r,
              int nunits, int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = fa_stages(r), SB = fa_stage_bytes(r), AC = fa_acc_cols(r);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + 4;
  uint64_t* tfull = empty + 4;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* s_consumed = reinterpret_cast<int*>(tmem_slot + 1);
  unsigned char* stages = smem + 1024;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = (s + kGmTile - 1) / kGmTile;
  const int dblk = d / 64, nkb = h * dblk;

  if (threadIdx.x == 0) {
    tc::prefetch_tensormap(&mapK);
    tc::prefetch_tensormap(&mapXh);
    tc::prefetch_tensormap(&mapXl);
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&tfull[a], 1);
      tc::mbar_init(&tempty[a], 128);
    }
    tc::mbar_init(drain, 1);
    *s_consumed = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 2 * AC);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  int issued = 0;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
        const int seq = u / tiles, t0 = (u - seq * tiles) * kGmTile;
        for (int kb = 0; kb < nkb; ++kb, ++issued) {
          const int st = issued % S;
          if (!tc::mbar_wait(&empty[st], ((issued / S) & 1) ^ 1, kWaitLimit)) {
            flag_error(status, DEV_TIMEOUT);
            ok = false;
            break;
          }
          tc::mbar_expect_tx(&full[st], SB);
          unsigned char* sp = stages + st * SB;
          const int hh = kb / dblk, e0 = (kb - hh * dblk) * 64;
          tc::tma_load_3d(sp, &mapK, &full[st], e0, t0, seq * h + hh);
          tc::tma_load_2d(sp + kGmTile * 128, &mapXh, &full[st], kb * 64, seq * r);
          tc::tma_load_2d(sp + kGmTile * 128 + r * 128, &mapXl, &full[st], kb * 64, seq * r);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(kGmTile, r);
      int it = 0, ul = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++ul) {
        const int acc = ul & 1;
        if (!tc::mbar_wait(&tempty[acc], ((ul >> 1) & 1) ^ 1, kWaitLimit)) {
          flag_error(status, DEV_TIMEOUT);
          break;
        }
        tc::fence_after();
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int st = it % S;
          if (!tc::mbar_wait(&full[st], (it / S) & 1, kWaitLimit)) {
            flag_error(status, DEV_TIMEOUT);
            ok = false;
            break;
          }
          tc::fence_after();
          const uint32_t a0 = tc::smem_u32(stages + st * SB);
          const uint32_t bh0 = a0 + kGmTile * 128, bl0 = bh0 + r * 128;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t da = tc::desc_k_sw128(a0 + kk * 32, 1024);
            tc::mma_bf16(tmem + acc * AC, da, tc::desc_k_sw128(bh0 + kk * 32, 1024), idesc,
                         (kb != 0 || kk != 0) ? 1u : 0u);
            tc::mma_bf16(tmem + acc * AC, da, tc::desc_k_sw128(bl0 + kk * 32, 1024), idesc, 1u);
          }
          tc::mma_commit(&empty[st]);
        }
        if (ok) tc::mma_commit(&tfull[acc]);
      }
      *s_consumed = it;
      tc::mma_commit(drain);
      if (!tc::mbar_wait(drain, 0, kWaitLimit)) flag_error(status, DEV_TIMEOUT);
    }
  } else {
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    int ul = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++ul) {
      const int acc = ul & 1;
      const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&tfull[acc], (ul >> 1) & 1, kWaitLimit));
      if (!ok) {
        if (lane == 0) flag_error(status, DEV_TIMEOUT);
        break;
      }
      tc::fence_after();
      const int seq = u / tiles, t = (u - seq * tiles) * kGmTile + row;
      bf16* dst = A + (static_cast<size_t>(seq) * s + t) * r;
#pragma unroll 1
      for (int c0 = 0; c0 < r; c0 += 16) {
        float v[16];
        tc::tmem_ld16(tmem + (static_cast<uint32_t>(q4 * 32) << 16) + acc * AC + c0, v);
        if (t < s) {
          uint32_t w[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            w[q] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * q]))) |
                   (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * q + 1]))) << 16);
          *reinterpret_cast<uint4*>(dst + c0) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(dst + c0 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
      tc::fence_before();
      tc::mbar_arrive(&tempty[acc]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    for (int it = *s_consumed; it < issued; ++it)
      if (!tc::mbar_wait(&full[it % S], (it / S) & 1, kWaitLimit)) {
        flag_error(status, DEV_TIMEOUT);
        break;
      }
  }
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * AC);
}

// bf16 hi / lo parts of the basis: X = Xh + Xl + O(2^-17 |X|).
__global__ void k_split_hilo(const float* __restrict__ X, bf16* __restrict__ Xh, bf16* __restrict__ Xl, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float x = X[i];
    const bf16 h = __float2bfloat16_rn(x);
    Xh[i] = h;
    Xl[i] = __float2bfloat16_rn(x - __bfloat162float(h));
  }
}

// =============================================================== host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool svd_tc_supported(const shadowkv_params& p) {
  const int D = p.h_kv * p.d;
  return p.dtype == SKV_DTYPE_BF16 && D % kGmTile == 0 && p.s % 8 == 0 && p.r % 16 == 0 && p.r <= 256;
}

// Splits of the token range: at most kGmSplitTokens per split, and enough
// units to give every SM several.
static void gram_splits(const shadowkv_params& p, int nsm, int* nz, int* kb_per_z, int* nkb) {
  const int D = p.h_kv * p.d;
  const int ntile = D / kGmTile, npairs = ntile * (ntile + 1) / 2;
  *nkb = (p.s + 63) / 64;
  int z = (p.s + kGmSplitTokens - 1) / kGmSplitTokens;
  const int want = (8 * nsm + p.b * npairs - 1) / (p.b * npairs);
  z = std::max(z, std::min(want, std::max(1, *nkb / 16)));
  z = std::max(1, std::min(z, *nkb));
  *kb_per_z = (*nkb + z - 1) / z;
  *nz = (*nkb + *kb_per_z - 1) / *kb_per_z;   // no empty split
}

size_t svd_tc_workspace_bytes(const shadowkv_params& p, int nsm) {
  const size_t D = static_cast<size_t>(p.h_kv) * p.d, b = p.b, r = p.r, s = p.s;
  int nz, kbz, nkb;
  gram_splits(p, nsm, &nz, &kbz, &nkb);
  const size_t ntile = D / kGmTile, npairs = ntile * (ntile + 1) / 2;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(b * D * s * 2) + up(b * nz * npairs * kGmTile * kGmTile * 4) + up(b * D * D * 4) +
         up(b * r * D * 4) + up(kSyrkSplit * b * r * r * 8) + 2 * up(b * r * D * 2);
}

#define SVD_TRY(...)                    \
  do {                                  \
    cudaError_t e_ = (__VA_ARGS__);     \
    if (e_ != cudaSuccess) return e_;   \
  } while (0)

// One orthonormalisation of the rows of Y (b x r x D): shifted CholeskyQR
// in fp64, then two CholeskyQR passes in fp32; the result goes to X.
static cudaError_t orth_rows(Ctx& c, float* Y, float* X, void* W, cudaStream_t st) {
  const int b = c.p.b, r = c.p.r, D = c.p.h_kv * c.p.d;
  const int nt = (r + 31) / 32;
  const dim3 gs(nt, nt, b * kSyrkSplit);
  const dim3 gt((D + kTrCols - 1) / kTrCols, b);
  SVD_TRY(set_smem_once(reinterpret_cast<const void*>(k_trsm<double>), static_cast<int>(trsm_smem(r))));
  SVD_TRY(set_smem_once(reinterpret_cast<const void*>(k_trsm<float>), static_cast<int>(trsm_smem(r))));
  for (int pass = 0; pass < 3; ++pass) {
    const float* in = pass == 1 ? X : Y;
    float* out = pass == 1 ? Y : X;   // Y -> X -> Y -> X
    kbegin(c, K_ORTH, st);
    if (pass == 0) {
      const size_t cs = (chol_tri(r) + r) * 8;
      const int sm = cs <= 200 * 1024;
      if (sm) SVD_TRY(set_smem_once(reinterpret_cast<const void*>(k_chol<double>), static_cast<int>(cs)));
      k_syrk<double><<<gs, 256, 0, st>>>(in, static_cast<double*>(W), r, D, b);
      k_chol<double><<<b, kCholThreads, sm ? cs : 0, st>>>(static_cast<double*>(W), r, D, b, 1, sm, c.status);
      k_trsm<double><<<gt, 256, trsm_smem(r), st>>>(static_cast<const double*>(W), in, out, r, D);
    } else {
      const size_t cs = (chol_tri(r) + r) * 4;
      SVD_TRY(set_smem_once(reinterpret_cast<const void*>(k_chol<float>), static_cast<int>(cs)));
      k_syrk<float><<<gs, 256, 0, st>>>(in, static_cast<float*>(W), r, D, b);
      k_chol<float><<<b, kCholThreads, cs, st>>>(static_cast<float*>(W), r, D, b, 0, 1, c.status);
      k_trsm<float><<<gt, 256, trsm_smem(r), st>>>(static_cast<const float*>(W), in, out, r, D);
    }
    kend(c, K_ORTH, st);
    SVD_TRY(cudaGetLastError());
  }
  return cudaSuccess;
}

// The basis X (b x r x D, fp32) of each sequence's rank-r right singular
// subspace, into c.basis; also bf16 hi/lo copies for the product A = M X^T.
// ws: svd_tc_workspace_bytes of device memory.
cudaError_t svd_tc_basis(Ctx& c, const void* Kv, void* ws, cudaStream_t st) {
  const bf16* K = static_cast<const bf16*>(Kv);
  const int b = c.p.b, h = c.p.h_kv, d = c.p.d, s = c.p.s, r = c.p.r, D = h * d;
  int nz, kb_per_z, nkb;
  gram_splits(c.p, c.nsm, &nz, &kb_per_z, &nkb);
  const int ntile = D / kGmTile, npairs = ntile * (ntile + 1) / 2;
  const int nunits = b * nz * npairs;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  char* cur = static_cast<char*>(ws);
  bf16* MT = reinterpret_cast<bf16*>(cur);
  cur += up(static_cast<size_t>(b) * D * s * 2);
  float* part = reinterpret_cast<float*>(cur);
  cur += up(static_cast<size_t>(nunits) * kGmTile * kGmTile * 4);
  float* G = reinterpret_cast<float*>(cur);
  cur += up(static_cast<size_t>(b) * D * D * 4);
  float* Y = reinterpret_cast<float*>(cur);
  cur += up(static_cast<size_t>(b) * r * D * 4);
  void* W = cur;
  float* X = c.basis;

  // MT and the Gram matrices
  kbegin(c, K_MISC, st);
  k_transpose_m<<<dim3((s + 63) / 64, d / 64, b * h), 256, 0, st>>>(K, MT, h, s, d);
  kend(c, K_MISC, st);
  SVD_TRY(cudaGetLastError());
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(s), static_cast<cuuint64_t>(b) * D};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(s) * 2};
  const cuuint32_t box[2] = {64, kGmTile};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, MT, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  SVD_TRY(set_smem_once(reinterpret_cast<const void*>(k_gram_tc), kGmSmem));
  kbegin(c, K_GRAM, st);
  k_gram_tc<<<std::min(nunits, c.nsm), kGmThreads, kGmSmem, st>>>(map, part, D, ntile, npairs, nz, kb_per_z, nkb,
                                                             nunits, c.status);
  kend(c, K_GRAM, st);
  SVD_TRY(cudaGetLastError());
  kbegin(c, K_MISC, st);
  const size_t gtot = static_cast<size_t>(b) * D * D;
  k_gram_reduce<<<static_cast<int>(std::min<size_t>((gtot + 255) / 256, 8192)), 256, 0, st>>>(part, G, b, D, ntile,
                                                                                       npairs, nz);
  kend(c, K_MISC, st);
  SVD_TRY(cudaGetLastError());

  bf16* Xh = reinterpret_cast<bf16*>(cur + (static_cast<size_t>(kSyrkSplit) * b * r * r * 8 + 255) / 256 * 256);
  bf16* Xl = Xh + (static_cast<size_t>(b) * r * D * 2 + 255) / 256 * 128;

  // subspace iteration on G from a seeded Gaussian start
  const int iters = c.p.svd_iters > 0 ? c.p.svd_iters : 3;
  // (the Gaussian start needs no orthonormalisation: only its span matters,
  // and the first product X G is orthonormalised)
  SVD_TRY(launch_random_basis(c, X, st));
  const dim3 gg(D / 64, (r + 63) / 64, b);
  for (int it = 0; it < iters; ++it) {
    kbegin(c, K_GEMM, st);
    k_gemm_xg<<<gg, 256, 0, st>>>(X, G, Y, r, D);
    kend(c, K_GEMM, st);
    SVD_TRY(cudaGetLastError());
    SVD_TRY(orth_rows(c, Y, X, W, st));
  }

  // A = M X^T on the tensor cores
  const size_t nx = static_cast<size_t>(b) * r * D;
  kbegin(c, K_MISC, st);
  k_split_hilo<<<static_cast<int>(std::min<size_t>((nx + 255) / 256, 4096)), 256, 0, st>>>(X, Xh, Xl, nx);
  kend(c, K_MISC, st);
  SVD_TRY(cudaGetLastError());
  CUtensorMap mk, mxh, mxl;
  {
    const cuuint64_t kd[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(s),
                              static_cast<cuuint64_t>(b) * h};
    const cuuint64_t ks[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(s) * d * 2};
    const cuuint32_t kbox[3] = {64, kGmTile, 1};
    const cuuint32_t kes[3] = {1, 1, 1};
    if (fn(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<bf16*>(K), kd, ks, kbox, kes,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    const cuuint64_t xd[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(b) * r};
    const cuuint64_t xs[1] = {static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t xbox[2] = {64, static_cast<cuuint32_t>(r)};
    for (int w = 0; w < 2; ++w)
      if (fn(w ? &mxl : &mxh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w ? Xl : Xh, xd, xs, xbox, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
  }
  const int fa_smem = 2048 + fa_stages(r) * fa_stage_bytes(r);
  SVD_TRY(set_smem_once(reinterpret_cast<const void*>(k_factor_a_tc), fa_smem));
  const int funits = b * ((s + kGmTile - 1) / kGmTile);
  kbegin(c, K_SVD_A, st);
  k_factor_a_tc<<<std::min(funits, c.nsm), kFaThreads, fa_smem, st>>>(mk, mxh, mxl, static_cast<bf16*>(c.A), h, s,
                                                                     d, r, funits, c.status);
  kend(c, K_SVD_A, st);
  return cudaGetLastError();
}

}  // namespace skv
