// Key rebuild of ShadowKV's decode step (Algorithm 2 step 3, key branch, and
// the RoPE of step 4): K_sparse = RoPE(MatMul(Gather(A, I), B)) for the k
// selected chunks of every (batch, KV head), at each token's position.
//
// Output layout: K_sparse[b][h][pos*c + u][:] for the pos-th selected chunk
// (ascending chunk order) and in-chunk token u.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

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


// ------------------------------------------------------------ tcgen05 path
// One CTA per (batch, KV head, 128-row tile of the k*c selected rows).
//   warp 0   : TMA loads -- the tile's selected chunks of A (one c x 32 box
//              per chunk and 32-column K block) and the head's B^T, all into
//              K-major 64-byte-swizzled shared memory: [K block][row][64 B]
//   thread 0 : ceil(r/32) x 2 tcgen05.mma (M=128, N=d, K=16) into a TMEM
//              accumulator of d fp32 columns x 128 lanes
//   4 warps  : TMEM -> registers (lane = row), RoPE at the row's position,
//              bf16 pack into a swizzled staging tile, coalesced stores.
constexpr int kTcRows = 128;

// Shared memory: a 1 KB header (barriers, TMEM address, RoPE frequencies),
// then, 1 KB aligned, the operand tiles A [KB][128][64 B] and B [KB][D][64 B];
// after the MMAs the bf16 output staging tile (128 x D) reuses that region.
__host__ __device__ constexpr int tc_tiles_bytes(int KB, int D) {
  return KB * (kTcRows + D) * 64 > kTcRows * D * 2 ? KB * (kTcRows + D) * 64 : kTcRows * D * 2;
}
__host__ __device__ constexpr int tc_smem_bytes(int KB, int D) {
  return 1024 /* alignment slack */ + 1024 /* header */ + tc_tiles_bytes(KB, D);
}

template <int D>
__global__ void __launch_bounds__(kTcRows, 2)
k_rebuild_tc(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapBt,
             const int32_t* __restrict__ sel, const float2* __restrict__ rope_tab,
             bf16* __restrict__ K_sp, int h_kv, int s, int r, int c, int k, int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int KB = (r + 31) / 32;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);            // [0] loads, [1] MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  int* s_flag = reinterpret_cast<int*>(bars + 3);
  float2* ftab = reinterpret_cast<float2*>(bars + 8);            // D/2 <= 64 entries
  unsigned char* sA = smem + 1024;                   // KB x [128 rows][64 B]
  unsigned char* sB = sA + KB * kTcRows * 64;        // KB x [D rows][64 B]

  const int pair = blockIdx.y, bb = pair / h_kv;
  const int rows = k * c;
  const int row0 = blockIdx.x * kTcRows;
  const int nrow = min(kTcRows, rows - row0);        // a multiple of c
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tc::prefetch_tensormap(&mapA);
    tc::prefetch_tensormap(&mapBt);
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    tc::fence_mbar_init();
    *s_flag = 1;
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, D);
    tc::tmem_relinquish();
  }
  for (int i = tid; i < D / 2; i += kTcRows) ftab[i] = rope_tab[i];
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- TMA producer (warp 0)
  if (warp == 0) {
    const int nch = nrow / c;
    if (lane == 0) tc::mbar_expect_tx(&bars[0], static_cast<uint32_t>(KB * (nrow + D) * 64));
    __syncwarp();
    const int nA = nch * KB;
    const int32_t* srow = sel + static_cast<size_t>(pair) * k + row0 / c;
    for (int i = lane; i < nA + KB; i += 32) {
      if (i < nA) {
        const int ch = i / KB, kb = i - ch * KB;
        const int chunk = srow[ch];
        tc::tma_load_2d(sA + kb * (kTcRows * 64) + ch * c * 64, &mapA, &bars[0], kb * 32,
                        bb * s + chunk * c);
      } else {
        const int kb = i - nA;
        tc::tma_load_2d(sB + kb * (D * 64), &mapBt, &bars[0], kb * 32, pair * D);
      }
    }
  }
  // ---- MMA issue (thread 0)
  if (tid == 0) {
    if (tc::mbar_wait(&bars[0], 0, kWaitLimit)) {
      tc::fence_after();
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTcRows, D);
      const uint32_t a0 = tc::smem_u32(sA), b0 = tc::smem_u32(sB);
      for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const uint64_t ad = tc::desc_k_sw64(a0 + kb * (kTcRows * 64) + ks * 32, 512);
          const uint64_t bd = tc::desc_k_sw64(b0 + kb * (D * 64) + ks * 32, 512);
          tc::mma_bf16(tmem, ad, bd, idesc, (kb | ks) != 0);
        }
      }
      tc::mma_commit(&bars[1]);
    } else {
      *s_flag = 0;
      flag_error(status, DEV_TIMEOUT);
      tc::mbar_wait(&bars[0], 0, kWaitLimit);   // let copies in flight land
    }
  }
  __syncthreads();
  bool ok = *s_flag != 0;
  if (ok) ok = tc::mbar_wait(&bars[1], 0, kWaitLimit);
  ok = __syncthreads_and(ok);
  if (ok) {
    tc::fence_after();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    // ---- epilogue: lane = row of the tile
    const int row = warp * 32 + lane;
    const int R = row0 + row;
    int pos = 0;
    if (row < nrow) pos = sel[static_cast<size_t>(pair) * k + R / c] * c + (R % c);
    uint4* stage = reinterpret_cast<uint4*>(sA);      // [128][D/8] x 16 B, chunk-swizzled;
                                                       // tc_tiles_bytes() >= 128 * D * 2
    constexpr int Q = D / 8;                           // 16-byte chunks per row
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
    for (int half = 0; half < D / 64; ++half) {
      float lo[32], hi[32];
      tc::tmem_ld32(trow + half * 32, lo);
      tc::tmem_ld32(trow + D / 2 + half * 32, hi);
      uint32_t plo[16], phi[16];
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        float y1[2], y2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float sn, cs;
          rope_sincos_fast(pos, ftab[half * 32 + i + e], &sn, &cs);
          y1[e] = lo[i + e] * cs - hi[i + e] * sn;
          y2[e] = hi[i + e] * cs + lo[i + e] * sn;
        }
        const __nv_bfloat162 a = __floats2bfloat162_rn(y1[0], y1[1]);
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(y2[0], y2[1]);
        plo[i / 2] = *reinterpret_cast<const uint32_t*>(&a);
        phi[i / 2] = *reinterpret_cast<const uint32_t*>(&b2);
      }
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int qlo = half * 4 + q4, qhi = Q / 2 + half * 4 + q4;
        stage[row * Q + (qlo ^ (row & (Q - 1)))] =
            make_uint4(plo[4 * q4], plo[4 * q4 + 1], plo[4 * q4 + 2], plo[4 * q4 + 3]);
        stage[row * Q + (qhi ^ (row & (Q - 1)))] =
            make_uint4(phi[4 * q4], phi[4 * q4 + 1], phi[4 * q4 + 2], phi[4 * q4 + 3]);
      }
    }
    tc::fence_before();
    __syncthreads();
    uint4* dst = reinterpret_cast<uint4*>(K_sp + (static_cast<size_t>(pair) * rows + row0) * D);
    for (int idx = tid; idx < nrow * Q; idx += kTcRows) {
      const int rr = idx / Q, q = idx - rr * Q;
      dst[idx] = stage[rr * Q + (q ^ (rr & (Q - 1)))];
    }
  } else {
    tc::fence_before();
    __syncthreads();
  }
  if (warp == 0) tc::tmem_dealloc(tmem, D);
}

bool tc_rebuild_supported(const shadowkv_params& p) {
  return p.dtype == SKV_DTYPE_BF16 && (p.d == 64 || p.d == 128) && p.c % 8 == 0 &&
         kTcRows % p.c == 0 && p.r % 8 == 0 && p.r <= 256;
}

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

// 2D bf16 map over a row-major [rows][r] matrix with a 32-column x box_rows
// box and the 64-byte swizzle.
static cudaError_t encode_rows(CUtensorMap* map, void* base, uint64_t nrows, int r, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(r), nrows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(r) * 2};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_rebuild_maps(Ctx& c) {
  c.tc_rebuild = false;
  if (!tc_rebuild_supported(c.p)) return cudaSuccess;
  const uint64_t pairs = static_cast<uint64_t>(c.p.b) * c.p.h_kv;
  cudaError_t e = encode_rows(&c.mapA, c.A, static_cast<uint64_t>(c.p.b) * c.p.s, c.p.r, c.p.c);
  if (e == cudaSuccess) e = encode_rows(&c.mapBt, c.Bt, pairs * c.p.d, c.p.r, c.p.d);
  if (e == cudaSuccess) c.tc_rebuild = true;
  return e;
}

template <int D>
static cudaError_t rebuild_tc(Ctx& c, cudaStream_t st) {
  const int KB = (c.p.r + 31) / 32;
  const int smem = tc_smem_bytes(KB, D);
  auto kern = k_rebuild_tc<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((c.p.k * c.p.c + kTcRows - 1) / kTcRows, c.p.b * c.p.h_kv);
  kern<<<grid, kTcRows, smem, st>>>(c.mapA, c.mapBt, c.sel, c.rope_tab, static_cast<bf16*>(c.K_sparse),
                                     c.p.h_kv, c.p.s, c.p.r, c.p.c, c.p.k, c.status);
  return cudaGetLastError();
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
  if (c.tc_rebuild && !c.force_simt)
    e = c.p.d == 128 ? rebuild_tc<128>(c, st) : rebuild_tc<64>(c, st);
  else if (c.p.dtype == SKV_DTYPE_BF16)
    e = c.p.d == 128 ? rebuild_simt<bf16, 128>(c, st) : rebuild_simt<bf16, 64>(c, st);
  else
    e = c.p.d == 128 ? rebuild_simt<float, 128>(c, st) : rebuild_simt<float, 64>(c, st);
  kend(c, K_REBUILD, st);
  return e;
}

}  // namespace skv
