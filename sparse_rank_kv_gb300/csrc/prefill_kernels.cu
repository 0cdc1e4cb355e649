// Prefill kernels of ShadowKV (Algorithm 1 of the ShadowKV review page):
//   k_chunkstats     K_RoPE = RoPE(K) on the fly; landmarks L = chunk means
//                    (Reduce, step 2); min over the chunk of the cosine of
//                    each token to its mean (steps 3-4)
//   k_outlier_select I = ArgTopK(-Min(S), o) per (batch, KV head)
//   k_gather_rows    post-RoPE keys and values of the outlier chunks and of
//                    the local window, kept exactly on the GPU (step 5)
//   SVD (step 1)     rank-r right singular subspace of each sequence's
//                    s x (h_kv d) pre-RoPE key matrix M by randomized
//                    subspace iteration: a seeded Gaussian basis X, then
//                    X <- orth((M X^T)^T M) a few times (M^T M applied one
//                    factor at a time, so fp32 never sees its squared
//                    condition number), then A = M X^T and B = X split per
//                    KV head.  Only the product A B is unique, so X is any
//                    orthonormal basis of that subspace.
#include "common.cuh"
#include "internal.h"

namespace skv {

// ---------------------------------------------------------- chunk stats
// Warp per chunk.  Lane l handles the RoPE pairs (i, i + D/2) for
// i = l + 32 p.  Two passes over the chunk's c tokens: the mean, then the
// cosine of each token to it (keys are re-rotated rather than kept).
template <typename T, int D>
__global__ void __launch_bounds__(256)
k_chunkstats(const T* __restrict__ K, const float2* __restrict__ rope_tab, T* __restrict__ L,
             float* __restrict__ mcos, int s, int c, int n) {
  constexpr int NP = D / 64;
  const int pair = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * 8 + warp;
  if (j >= n) return;
  const T* base = K + (static_cast<size_t>(pair) * s + static_cast<size_t>(j) * c) * D;
  float2 f[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) f[p] = rope_tab[lane + 32 * p];
  float mean[2 * NP];
#pragma unroll
  for (int p = 0; p < 2 * NP; ++p) mean[p] = 0.f;
  for (int u = 0; u < c; ++u) {
    const T* row = base + static_cast<size_t>(u) * D;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const int i = lane + 32 * p;
      float sn, cs;
      rope_sincos(j * c + u, f[p], &sn, &cs);
      const float x1 = Ty<T>::to_f(row[i]), x2 = Ty<T>::to_f(row[i + D / 2]);
      mean[p] += x1 * cs - x2 * sn;
      mean[NP + p] += x2 * cs + x1 * sn;
    }
  }
  float nm2 = 0.f;
#pragma unroll
  for (int p = 0; p < 2 * NP; ++p) {
    mean[p] = mean[p] / static_cast<float>(c);
    nm2 += mean[p] * mean[p];
  }
  nm2 = warp_sum(nm2);
  const float nm = sqrtf(nm2);
  float mn = INFINITY;
  for (int u = 0; u < c; ++u) {
    const T* row = base + static_cast<size_t>(u) * D;
    float dot = 0.f, nx2 = 0.f;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const int i = lane + 32 * p;
      float sn, cs;
      rope_sincos(j * c + u, f[p], &sn, &cs);
      const float x1 = Ty<T>::to_f(row[i]), x2 = Ty<T>::to_f(row[i + D / 2]);
      const float y1 = x1 * cs - x2 * sn, y2 = x2 * cs + x1 * sn;
      dot += y1 * mean[p] + y2 * mean[NP + p];
      nx2 += y1 * y1 + y2 * y2;
    }
    dot = warp_sum(dot);
    nx2 = warp_sum(nx2);
    mn = fminf(mn, dot / fmaxf(sqrtf(nx2) * nm, 1e-8f));
  }
  T* lrow = L + (static_cast<size_t>(pair) * n + j) * D;
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    lrow[lane + 32 * p] = Ty<T>::from_f(mean[p]);
    lrow[lane + 32 * p + D / 2] = Ty<T>::from_f(mean[NP + p]);
  }
  if (lane == 0) mcos[static_cast<size_t>(pair) * n + j] = mn;
}

// ------------------------------------------------------ outlier select
__global__ void __launch_bounds__(1024)
k_outlier_select(const float* __restrict__ mcos, int32_t* __restrict__ out_ids, int n, int o) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int nw = (n + 31) >> 5;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  uint32_t* bits = keys + n;
  int* wpref = reinterpret_cast<int*>(bits + nw);
  int* s_out = wpref + nw;
  int* scratch = align16(s_out + o);
  const int pair = blockIdx.x;
  for (int j = threadIdx.x; j < n; j += blockDim.x)
    keys[j] = order_key(-mcos[static_cast<size_t>(pair) * n + j]);
  __syncthreads();
  block_topk(keys, n, o, s_out, scratch, bits, wpref);
  for (int i = threadIdx.x; i < o; i += blockDim.x) out_ids[static_cast<size_t>(pair) * o + i] = s_out[i];
}

// ---------------------------------------------------------- row gathers
// mode 0: the o*c rows of the outlier chunks; mode 1: the w local rows.
// Keys are rotated to their positions, values copied.  V may be the mapped
// address of pinned host memory.
template <typename T, int D>
__global__ void __launch_bounds__(256)
k_gather_rows(const T* __restrict__ K, const T* __restrict__ V, const int32_t* __restrict__ out_ids,
              const float2* __restrict__ rope_tab, T* __restrict__ Kd, T* __restrict__ Vd, int s,
              int c, int o, int n, int nrows, int dst_stride, int mode, int* __restrict__ status) {
  const int pair = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.y * 8 + warp;
  if (row >= nrows) return;
  int pos;
  if (mode == 0) {
    const int id = out_ids[static_cast<size_t>(pair) * o + row / c];
    if (id < 0 || id >= n) {
      if (lane == 0) flag_error(status, DEV_BAD_OUTLIER);
      return;
    }
    pos = id * c + row % c;
  } else {
    pos = n * c + row;
  }
  const T* ks = K + (static_cast<size_t>(pair) * s + pos) * D;
  const T* vs = V + (static_cast<size_t>(pair) * s + pos) * D;
  T* kd = Kd + (static_cast<size_t>(pair) * dst_stride + row) * D;
  T* vd = Vd + (static_cast<size_t>(pair) * dst_stride + row) * D;
  for (int i = lane; i < D / 2; i += 32) {
    float sn, cs;
    rope_sincos(pos, rope_tab[i], &sn, &cs);
    const float x1 = Ty<T>::to_f(ks[i]), x2 = Ty<T>::to_f(ks[i + D / 2]);
    kd[i] = Ty<T>::from_f(x1 * cs - x2 * sn);
    kd[i + D / 2] = Ty<T>::from_f(x2 * cs + x1 * sn);
  }
  for (int i = lane; i < D; i += 32) vd[i] = vs[i];
}

// ---------------------------------------------------------------- GEMMs
// Accessors: the pre-RoPE key matrix of one sequence, M[t][h*d + e] =
// K[h][t][e], and a plain row-major fp32 matrix.
template <typename T>
struct HeadSplit {
  const T* K;
  int s, dshift;
  __device__ __forceinline__ float operator()(int t, int col) const {
    const int h = col >> dshift, e = col & ((1 << dshift) - 1);
    return Ty<T>::to_f(K[((static_cast<size_t>(h) * s + t) << dshift) + e]);
  }
};
struct RowF {
  const float* p;
  int ld;
  __device__ __forceinline__ float operator()(int r, int c) const {
    return p[static_cast<size_t>(r) * ld + c];
  }
};

template <typename TO> __device__ __forceinline__ TO cvt_out(float x);
template <> __device__ __forceinline__ float cvt_out<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 cvt_out<bf16>(float x) { return __float2bfloat16_rn(x); }

// C[z][i][j] = sum_{t in split z} X(t, i) Y(t, j); 64x64 tiles, 4x4 per
// thread.  symmetric: only tiles with i-block <= j-block are computed.
template <class AX, class AY>
__global__ void __launch_bounds__(256)
k_gemm_tn(AX X, AY Y, float* __restrict__ C, int Mi, int Nj, int t_len, int t_per, int ldc,
          size_t zstride, int symmetric) {
  if (symmetric && blockIdx.y > blockIdx.x) return;
  __shared__ __align__(16) float Xs[16][68];
  __shared__ __align__(16) float Ys[16][68];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
  const int tb = blockIdx.z * t_per, te = min(t_len, tb + t_per);
  float acc[4][4] = {};
  for (int t = tb; t < te; t += 16) {
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      const int e = tid + 256 * qd, rr = e >> 6, cc = e & 63, tt = t + rr;
      Xs[rr][cc] = (tt < te && i0 + cc < Mi) ? X(tt, i0 + cc) : 0.f;
      Ys[rr][cc] = (tt < te && j0 + cc < Nj) ? Y(tt, j0 + cc) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&Xs[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Ys[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
    __syncthreads();
  }
  float* Cz = C + zstride * blockIdx.z;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + ty * 4 + u;
    if (i >= Mi) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int j = j0 + tx * 4 + v;
      if (j < Nj) Cz[static_cast<size_t>(i) * ldc + j] = acc[u][v];
    }
  }
}

// C[m][n] = sum_k A(m, k) B(n, k); 64x64 tiles, 4x4 per thread.
template <class AA, class AB, typename TO>
__global__ void __launch_bounds__(256)
k_gemm_nt(AA Aop, AB Bop, TO* __restrict__ C, int M, int N, int K, int ldc) {
  __shared__ __align__(16) float As[16][68];
  __shared__ __align__(16) float Bs[16][68];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      const int e = tid + 256 * qd, rr = e >> 4, kk = e & 15, kq = k0 + kk;
      As[kk][rr] = (m0 + rr < M && kq < K) ? Aop(m0 + rr, kq) : 0.f;
      Bs[kk][rr] = (n0 + rr < N && kq < K) ? Bop(n0 + rr, kq) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int m = m0 + ty * 4 + u;
    if (m >= M) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int nn = n0 + tx * 4 + v;
      if (nn < N) C[static_cast<size_t>(m) * ldc + nn] = cvt_out<TO>(acc[u][v]);
    }
  }
}

// out[i][j] = sum_z part[z][i][j]; symmetric: (i, j) below the diagonal
// blocks reads the mirrored upper entry.
__global__ void k_reduce_splits(const float* __restrict__ part, float* __restrict__ out, int nz,
                                int M, int N, size_t zstride, int symmetric) {
  const size_t total = static_cast<size_t>(M) * N;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    int i = static_cast<int>(idx / N), j = static_cast<int>(idx % N);
    if (symmetric && (i >> 6) > (j >> 6)) { const int t = i; i = j; j = t; }
    float acc = 0.f;
    for (int z = 0; z < nz; ++z) acc += part[zstride * z + static_cast<size_t>(i) * N + j];
    out[idx] = acc;
  }
}

// --------------------------------------------------- orthonormalisation
// Modified Gram-Schmidt on the r rows (length D) of X, repeated `passes`
// times.  One block; warp w updates rows j+1+w, j+33+w, ... at step j.
__global__ void __launch_bounds__(1024) k_mgs(float* __restrict__ X, int r, int D, int passes) {
  __shared__ float red[32];
  __shared__ float s_norm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int pass = 0; pass < passes; ++pass) {
    for (int j = 0; j < r; ++j) {
      float* xj = X + static_cast<size_t>(j) * D;
      float ss = 0.f;
      for (int e = tid; e < D; e += blockDim.x) ss += xj[e] * xj[e];
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += red[w];
        s_norm = sqrtf(t);
      }
      __syncthreads();
      const float nrm = s_norm;
      if (nrm > 1e-30f) {
        const float inv = 1.f / nrm;
        for (int e = tid; e < D; e += blockDim.x) xj[e] *= inv;
      } else {
        // a direction the basis lost: restart it from a coordinate vector
        const int hot = (j * 7 + 3) % D;
        for (int e = tid; e < D; e += blockDim.x) xj[e] = e == hot ? 1.f : 0.f;
      }
      __syncthreads();
      for (int i = j + 1 + warp; i < r; i += 32) {
        float* xi = X + static_cast<size_t>(i) * D;
        float dp = 0.f;
        for (int e = lane; e < D; e += 32) dp += xi[e] * xj[e];
        dp = warp_sum(dp);
        for (int e = lane; e < D; e += 32) xi[e] -= dp * xj[e];
      }
      __syncthreads();
    }
  }
}

// Seeded standard-normal starting basis: splitmix64 counter hash and the
// Box-Muller transform.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}
__global__ void k_random_basis(float* __restrict__ X, int r, int D, unsigned long long seed, int seq) {
  const int total = r * D;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
    const uint64_t h = splitmix64(seed ^ splitmix64((static_cast<uint64_t>(seq) << 40) + idx));
    const float u1 = (static_cast<float>(h >> 40) + 1.0f) * (1.0f / 16777217.0f);
    const float u2 = static_cast<float>((h >> 16) & 0xFFFFFF) * (1.0f / 16777216.0f);
    X[idx] = sqrtf(-2.0f * logf(u1)) * cospif(2.0f * u2);
  }
}

// Bt[h][e][i] = X[i][h*d + e] for one sequence.
template <typename T>
__global__ void k_basis_to_bt(const float* __restrict__ X, T* __restrict__ Bt, int r, int D) {
  const int total = r * D;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
    const int col = idx / r, i = idx - col * r;   // col = h*d + e
    Bt[idx] = cvt_out<T>(X[static_cast<size_t>(i) * D + col]);
  }
}

// Bt[pair][e][i] = B[pair][i][e] (caller-supplied B in the page's layout).
template <typename T>
__global__ void k_b_to_bt(const T* __restrict__ B, T* __restrict__ Bt, int pairs, int r, int d) {
  const size_t total = static_cast<size_t>(pairs) * r * d;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t pair = idx / (static_cast<size_t>(r) * d);
    const int rem = static_cast<int>(idx - pair * r * d);
    const int e = rem / r, i = rem - e * r;
    Bt[idx] = B[(pair * r + i) * d + e];
  }
}

__global__ void k_fill_i32(int32_t* __restrict__ p, int32_t v, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    p[i] = v;
}

// =============================================================== host side
#define SKV_TRY(...)                    \
  do {                                  \
    cudaError_t e_ = (__VA_ARGS__);     \
    if (e_ != cudaSuccess) return e_;   \
  } while (0)

static int grid_for(size_t total, int threads, int cap) {
  size_t g = (total + threads - 1) / threads;
  if (g > static_cast<size_t>(cap)) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

// Reads 16 bytes of every 4 KB page of the pinned host copy of V through its
// device mapping: the first GPU access to a host page is slow, and this moves
// that cost out of the decode steps' value fetches.  The result only feeds a
// store under `keep`, which the host passes as 0; it keeps the loads from
// being optimised away.
__global__ void k_read_host(const unsigned char* __restrict__ p, size_t pages, int keep,
                            unsigned int* __restrict__ sink) {
  unsigned int acc = 0;
  const size_t nt = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < pages; i += nt) {
    const uint4 v = *reinterpret_cast<const uint4*>(p + (i << 12));
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (keep) atomicXor(sink, acc);
}

cudaError_t launch_read_host_v(Ctx& c, cudaStream_t st) {
  const size_t pages = (c.v_bytes + 4095) >> 12;
  kbegin(c, K_MISC, st);
  k_read_host<<<grid_for(pages, 256, 4 * c.nsm), 256, 0, st>>>(static_cast<const unsigned char*>(c.v_cpu_dev), pages,
                                                              0, reinterpret_cast<unsigned int*>(c.status));
  kend(c, K_MISC, st);
  return cudaGetLastError();
}

cudaError_t launch_fill_i32(Ctx& c, int32_t* p, int32_t v, size_t n, cudaStream_t st) {
  kbegin(c, K_MISC, st);
  k_fill_i32<<<grid_for(n, 256, 4096), 256, 0, st>>>(p, v, n);
  kend(c, K_MISC, st);
  return cudaGetLastError();
}

cudaError_t launch_transpose_b(Ctx& c, const void* B, cudaStream_t st) {
  const int pairs = c.p.b * c.p.h_kv;
  const size_t total = static_cast<size_t>(pairs) * c.p.r * c.p.d;
  kbegin(c, K_MISC, st);
  if (c.p.dtype == SKV_DTYPE_BF16)
    k_b_to_bt<bf16><<<grid_for(total, 256, 8192), 256, 0, st>>>(static_cast<const bf16*>(B),
                                                                static_cast<bf16*>(c.Bt), pairs, c.p.r, c.p.d);
  else
    k_b_to_bt<float><<<grid_for(total, 256, 8192), 256, 0, st>>>(static_cast<const float*>(B),
                                                                 static_cast<float*>(c.Bt), pairs, c.p.r, c.p.d);
  kend(c, K_MISC, st);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t prefill_stats(Ctx& c, const T* K, const T* V, cudaStream_t st) {
  const int pairs = c.p.b * c.p.h_kv;
  const int n = c.n, cc = c.p.c, o = c.p.o, s = c.p.s;
  kbegin(c, K_CHUNKSTATS, st);
  k_chunkstats<T, D><<<dim3((n + 7) / 8, pairs), 256, 0, st>>>(K, c.rope_tab, static_cast<T*>(c.L),
                                                                c.min_cos, s, cc, n);
  kend(c, K_CHUNKSTATS, st);
  SKV_TRY(cudaGetLastError());
  if (o > 0) {
    const size_t smem = sizeof(uint32_t) * (n + 2 * ((n + 31) / 32)) + sizeof(int) * (o + topk_scratch_ints(1024)) + 16;
    SKV_TRY(set_smem_once(reinterpret_cast<const void*>(k_outlier_select), static_cast<int>(smem)));
    kbegin(c, K_OUTLIERS, st);
    k_outlier_select<<<pairs, 1024, smem, st>>>(c.min_cos, c.out_ids, n, o);
    kend(c, K_OUTLIERS, st);
    SKV_TRY(cudaGetLastError());
  }
  SKV_TRY(launch_build_mask(c, st));
  if (o > 0) {
    kbegin(c, K_GATHER, st);
    k_gather_rows<T, D><<<dim3(pairs, (o * cc + 7) / 8), 256, 0, st>>>(
        K, V, c.out_ids, c.rope_tab, static_cast<T*>(c.K_out), static_cast<T*>(c.V_out), s, cc, o,
        n, o * cc, o * cc, 0, c.status);
    kend(c, K_GATHER, st);
  }
  if (c.p.w > 0) {
    kbegin(c, K_GATHER, st);
    k_gather_rows<T, D><<<dim3(pairs, (c.p.w + 7) / 8), 256, 0, st>>>(
        K, V, c.out_ids, c.rope_tab, static_cast<T*>(c.K_loc), static_cast<T*>(c.V_loc), s, cc, o,
        n, c.p.w, c.loc_cap, 1, c.status);
    kend(c, K_GATHER, st);
  }
  return cudaGetLastError();
}

cudaError_t launch_random_basis(Ctx& c, float* X, cudaStream_t st) {
  const size_t n_x = static_cast<size_t>(c.p.r) * c.p.h_kv * c.p.d;
  for (int bb = 0; bb < c.p.b; ++bb) {
    kbegin(c, K_MISC, st);
    k_random_basis<<<grid_for(n_x, 256, 1024), 256, 0, st>>>(X + bb * n_x, c.p.r, c.p.h_kv * c.p.d, c.p.seed, bb);
    kend(c, K_MISC, st);
  }
  return cudaGetLastError();
}

// bf16 contexts whose shapes the tensor-core SVD takes: the basis and
// A = M X^T (svd_tc.cu), then B^T per head.  One workspace allocation for
// the whole batch.
static cudaError_t prefill_svd_tc(Ctx& c, const bf16* K, cudaStream_t st) {
  const int d = c.p.d, h = c.p.h_kv, r = c.p.r, D = h * d;
  void* ws = nullptr;
  SKV_TRY(cudaMalloc(&ws, svd_tc_workspace_bytes(c.p, c.nsm)));
  cudaError_t err = svd_tc_basis(c, K, ws, st);
  const size_t n_x = static_cast<size_t>(r) * D;
  for (int bb = 0; bb < c.p.b && err == cudaSuccess; ++bb) {
    const float* X = c.basis + bb * n_x;
    kbegin(c, K_MISC, st);
    k_basis_to_bt<bf16><<<grid_for(n_x, 256, 1024), 256, 0, st>>>(X, static_cast<bf16*>(c.Bt) + bb * n_x, r, D);
    kend(c, K_MISC, st);
    err = cudaGetLastError();
  }
  cudaError_t e2 = cudaStreamSynchronize(st);
  cudaFree(ws);
  return err != cudaSuccess ? err : e2;
}

template <typename T>
static cudaError_t prefill_svd(Ctx& c, const T* K, cudaStream_t st) {
  if constexpr (sizeof(T) == 2) {
    if (svd_tc_supported(c.p) && !c.force_simt) return prefill_svd_tc(c, K, st);
  }
  const int s = c.p.s, d = c.p.d, h = c.p.h_kv, r = c.p.r, D = h * d;
  const int dshift = d == 128 ? 7 : 6;
  const int nsm = num_sms(c);
  const int tiles_y = ((r + 63) / 64) * (D / 64);
  int nz_y = (4 * nsm + tiles_y - 1) / tiles_y;
  nz_y = max(1, min(nz_y, s / 256));
  const int iters = c.p.svd_iters > 0 ? c.p.svd_iters : 3;

  // one sequence's workspace: basis X, next basis Y (r x D), Z = M X^T
  // (s x r), and the split-K partials of Z^T M
  const size_t n_x = static_cast<size_t>(r) * D, n_z = static_cast<size_t>(s) * r;
  const size_t n_ypart = static_cast<size_t>(nz_y) * r * D;
  float* ws = nullptr;
  SKV_TRY(cudaMalloc(&ws, sizeof(float) * (2 * n_x + n_z + n_ypart)));
  float* X = ws;
  float* Y = X + n_x;
  float* Z = Y + n_x;
  float* Yp = Z + n_z;
  const int tper_y = ((s + nz_y - 1) / nz_y + 15) / 16 * 16;
  cudaError_t err = cudaSuccess;
  for (int bb = 0; bb < c.p.b && err == cudaSuccess; ++bb) {
    const HeadSplit<T> M{K + static_cast<size_t>(bb) * h * s * d, s, dshift};
    kbegin(c, K_MISC, st);
    k_random_basis<<<grid_for(n_x, 256, 1024), 256, 0, st>>>(X, r, D, c.p.seed, bb);
    kend(c, K_MISC, st);
    kbegin(c, K_ORTH, st);
    k_mgs<<<1, 1024, 0, st>>>(X, r, D, 2);
    kend(c, K_ORTH, st);
    // subspace iteration on M^T M, one factor at a time: Y = (M X^T)^T M
    for (int it = 0; it < iters; ++it) {
      kbegin(c, K_GRAM, st);
      k_gemm_nt<<<dim3((r + 63) / 64, (s + 63) / 64), 256, 0, st>>>(M, RowF{X, D}, Z, s, r, D, r);
      kend(c, K_GRAM, st);
      kbegin(c, K_GEMM, st);
      k_gemm_tn<<<dim3(D / 64, (r + 63) / 64, nz_y), 256, 0, st>>>(RowF{Z, r}, M, Yp, r, D, s,
                                                                   tper_y, D, n_x, 0);
      kend(c, K_GEMM, st);
      kbegin(c, K_MISC, st);
      k_reduce_splits<<<grid_for(n_x, 256, 4096), 256, 0, st>>>(Yp, Y, nz_y, r, D, n_x, 0);
      kend(c, K_MISC, st);
      kbegin(c, K_ORTH, st);
      k_mgs<<<1, 1024, 0, st>>>(Y, r, D, 2);
      kend(c, K_ORTH, st);
      float* t = X; X = Y; Y = t;
    }
    // A = M X^T, B^T per head, and the basis for export
    kbegin(c, K_GRAM, st);
    k_gemm_nt<<<dim3((r + 63) / 64, (s + 63) / 64), 256, 0, st>>>(
        M, RowF{X, D}, static_cast<T*>(c.A) + static_cast<size_t>(bb) * s * r, s, r, D, r);
    kend(c, K_GRAM, st);
    kbegin(c, K_MISC, st);
    k_basis_to_bt<T><<<grid_for(n_x, 256, 1024), 256, 0, st>>>(
        X, static_cast<T*>(c.Bt) + static_cast<size_t>(bb) * n_x, r, D);
    kend(c, K_MISC, st);
    err = cudaGetLastError();
    if (err == cudaSuccess)
      err = cudaMemcpyAsync(c.basis + static_cast<size_t>(bb) * n_x, X, sizeof(float) * n_x,
                            cudaMemcpyDeviceToDevice, st);
  }
  cudaError_t e2 = cudaStreamSynchronize(st);
  cudaFree(ws);
  return err != cudaSuccess ? err : e2;
}

cudaError_t prefill_device(Ctx& c, const void* k_pre, const void* v, cudaStream_t st) {
  if (c.p.dtype == SKV_DTYPE_BF16) {
    const bf16* K = static_cast<const bf16*>(k_pre);
    const bf16* V = static_cast<const bf16*>(v);
    SKV_TRY(c.p.d == 128 ? prefill_stats<bf16, 128>(c, K, V, st) : prefill_stats<bf16, 64>(c, K, V, st));
    return prefill_svd<bf16>(c, K, st);
  }
  const float* K = static_cast<const float*>(k_pre);
  const float* V = static_cast<const float*>(v);
  SKV_TRY(c.p.d == 128 ? prefill_stats<float, 128>(c, K, V, st) : prefill_stats<float, 64>(c, K, V, st));
  return prefill_svd<float>(c, K, st);
}

}  // namespace skv
