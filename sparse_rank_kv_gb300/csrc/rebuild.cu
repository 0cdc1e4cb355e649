// Key rebuild of ShadowKV's decode step (Algorithm 2 step 3, key branch, and
// the RoPE of step 4): K_sparse = RoPE(MatMul(Gather(A, I), B)) for the k
// selected chunks of every (batch, KV head), at each token's position.
//
// Output layout: K_sparse[b][h][pos*c + u][:] for the pos-th selected chunk
// (ascending chunk order) and in-chunk token u.
#include "common.cuh"
#include "internal.h"

namespace skv {

constexpr int kRbRows = 64;       // output rows per block
constexpr int kRbThreads = 256;

// SIMT reference kernel: fp32 products and sums.  Shared memory holds the
// block's 64 gathered A rows and the head's B (both as fp32).  Thread
// (ty, tx) owns rows ty + 8 i and columns tx + 32 j, so the RoPE partners
// (col, col + D/2) are in the same thread.
template <typename T, int D>
__global__ void __launch_bounds__(kRbThreads)
k_rebuild_simt(const T* __restrict__ A, const T* __restrict__ Bt, const int32_t* __restrict__ sel,
               const float2* __restrict__ rope_tab, T* __restrict__ K_sp, int h_kv, int s, int r,
               int c, int k) {
  extern __shared__ __align__(16) float sm[];
  float* As = sm;                 // [kRbRows][r]
  float* Bs = sm + kRbRows * r;   // [r][D]
  const int pair = blockIdx.y, bb = pair / h_kv;
  const int row0 = blockIdx.x * kRbRows;
  const int rows = k * c;
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;

  // gathered A rows
  for (int i = tid; i < kRbRows * r; i += kRbThreads) {
    const int rr = i / r, kk = i - rr * r;
    const int R = row0 + rr;
    float v = 0.f;
    if (R < rows) {
      const int chunk = sel[static_cast<size_t>(pair) * k + R / c];
      const int tok = chunk * c + (R % c);
      v = Ty<T>::to_f(A[(static_cast<size_t>(bb) * s + tok) * r + kk]);
    }
    As[i] = v;
  }
  // B[kk][col] = Bt[col][kk]
  const T* Bp = Bt + static_cast<size_t>(pair) * D * r;
  for (int i = tid; i < D * r; i += kRbThreads) {
    const int col = i / r, kk = i - col * r;
    Bs[kk * D + col] = Ty<T>::to_f(Bp[i]);
  }
  __syncthreads();

  constexpr int RI = kRbRows / 8, CJ = D / 32;
  float acc[RI][CJ];
#pragma unroll
  for (int i = 0; i < RI; ++i)
#pragma unroll
    for (int j = 0; j < CJ; ++j) acc[i][j] = 0.f;
  for (int kk = 0; kk < r; ++kk) {
    float a[RI], b[CJ];
#pragma unroll
    for (int i = 0; i < RI; ++i) a[i] = As[(ty + 8 * i) * r + kk];
#pragma unroll
    for (int j = 0; j < CJ; ++j) b[j] = Bs[kk * D + tx + 32 * j];
#pragma unroll
    for (int i = 0; i < RI; ++i)
#pragma unroll
      for (int j = 0; j < CJ; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
  // RoPE epilogue and store
#pragma unroll
  for (int i = 0; i < RI; ++i) {
    const int R = row0 + ty + 8 * i;
    if (R >= rows) continue;
    const int chunk = sel[static_cast<size_t>(pair) * k + R / c];
    const int pos = chunk * c + (R % c);
    T* dst = K_sp + (static_cast<size_t>(pair) * rows + R) * D;
#pragma unroll
    for (int j = 0; j < CJ / 2; ++j) {
      const int col = tx + 32 * j;
      float sn, cs;
      rope_sincos(pos, rope_tab[col], &sn, &cs);
      const float x1 = acc[i][j], x2 = acc[i][j + CJ / 2];
      dst[col] = Ty<T>::from_f(x1 * cs - x2 * sn);
      dst[col + D / 2] = Ty<T>::from_f(x2 * cs + x1 * sn);
    }
  }
}

template <typename T, int D>
static cudaError_t rebuild_simt(Ctx& c, cudaStream_t st) {
  const size_t smem = sizeof(float) * (static_cast<size_t>(kRbRows) * c.p.r + static_cast<size_t>(c.p.r) * D);
  auto kern = k_rebuild_simt<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((c.p.k * c.p.c + kRbRows - 1) / kRbRows, c.p.b * c.p.h_kv);
  kern<<<grid, kRbThreads, smem, st>>>(static_cast<const T*>(c.A), static_cast<const T*>(c.Bt),
                                        c.sel, c.rope_tab, static_cast<T*>(c.K_sparse), c.p.h_kv,
                                        c.p.s, c.p.r, c.p.c, c.p.k);
  return cudaGetLastError();
}

cudaError_t launch_rebuild(Ctx& c, cudaStream_t st) {
  kbegin(c, K_REBUILD, st);
  cudaError_t e;
  if (c.p.dtype == SKV_DTYPE_BF16)
    e = c.p.d == 128 ? rebuild_simt<bf16, 128>(c, st) : rebuild_simt<bf16, 64>(c, st);
  else
    e = c.p.d == 128 ? rebuild_simt<float, 128>(c, st) : rebuild_simt<float, 64>(c, st);
  kend(c, K_REBUILD, st);
  return e;
}

}  // namespace skv
