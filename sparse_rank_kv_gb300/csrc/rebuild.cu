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
// Persistent kernel, one CTA per SM.  The (batch, KV head, 128-row tile)
// work items of the k*c selected rows are split into contiguous ranges, one
// per CTA, so that consecutive tiles of a CTA mostly share the head's B.
//   warp 0     : TMA producer -- for each tile the selected chunks of A (one
//                c x 32 box per chunk and 32-column K block) into an S-stage
//                ring, and the head's B^T into an NB-slot ring when the head
//                changes; K-major, 64-byte swizzle: [K block][row][64 B]
//   warp 1     : TMEM allocation; lane 0 issues ceil(r/32) x 2 tcgen05.mma
//                (M=128, N=d, K=16) per tile into one of two TMEM
//                accumulators (d fp32 columns each)
//   warps 2..9 : epilogue, two groups of four warps; warp w reads TMEM lane
//                quarter w % 4 (row = quarter*32 + lane), group g the RoPE
//                column pairs [g*d/4, (g+1)*d/4) and their partners at +d/2;
//                RoPE at the row's position, bf16 pack into a swizzled
//                staging tile, then coalesced stores of the whole tile.
// Barriers: fullA/emptyA per A stage, fullB/emptyB per B slot, tfull/tempty
// per accumulator.  Every wait is bounded; a timeout sets the status word and
// a shared abort flag that every role checks before its next wait.
constexpr int kTcRows = 128;
constexpr int kPipeThreads = 320;
constexpr int kEpiThreads = 256;

struct PipeShape {
  int KB, S, NB, smem;
};
__host__ __device__ constexpr int pipe_a_bytes(int KB) { return KB * kTcRows * 64; }
__host__ __device__ constexpr int pipe_b_bytes(int KB, int D) { return KB * D * 64; }
__host__ __device__ constexpr int pipe_smem(int KB, int D, int S, int NB) {
  return 1024 /* alignment slack */ + 1024 /* header */ + S * pipe_a_bytes(KB) +
         NB * pipe_b_bytes(KB, D) + kTcRows * D * 2 /* staging */;
}
static PipeShape pipe_shape(int r, int D) {
  const int KB = (r + 31) / 32;
  const int cand[4][2] = {{2, 2}, {2, 1}, {1, 2}, {1, 1}};
  for (auto& sn : cand) {
    const int sm = pipe_smem(KB, D, sn[0], sn[1]);
    if (sm <= 227 * 1024) return {KB, sn[0], sn[1], sm};
  }
  return {KB, 0, 0, 0};
}

template <int D>
__global__ void __launch_bounds__(kPipeThreads, 1)
k_rebuild_pipe(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapBt,
               const int32_t* __restrict__ sel, const float2* __restrict__ rope_tab,
               bf16* __restrict__ K_sp, int npairs, int h_kv, int s, int r, int c, int k, int S,
               int NB, int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int KB = (r + 31) / 32;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);   // <= 12 barriers
  uint64_t* fullA = bars;                                // [S]
  uint64_t* emptyA = bars + 2;                           // [S]
  uint64_t* fullB = bars + 4;                            // [NB]
  uint64_t* emptyB = bars + 6;                           // [NB]
  uint64_t* tfull = bars + 8;                            // [2]
  uint64_t* tempty = bars + 10;                          // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 256);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + 260);
  float2* ftab = reinterpret_cast<float2*>(smem + 512);  // D/2 <= 64 entries
  unsigned char* sA = smem + 1024;
  unsigned char* sB = sA + S * pipe_a_bytes(KB);
  uint4* stage = reinterpret_cast<uint4*>(sB + NB * pipe_b_bytes(KB, D));

  const int rows = k * c;
  const int tpp = (rows + kTcRows - 1) / kTcRows;        // tiles per (batch, KV head)
  const int total = npairs * tpp;
  const int lo = static_cast<int>(static_cast<long long>(blockIdx.x) * total / gridDim.x);
  const int hi = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * total / gridDim.x);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tc::prefetch_tensormap(&mapA);
    tc::prefetch_tensormap(&mapBt);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&fullA[i], 1);
      tc::mbar_init(&emptyA[i], 1);
      tc::mbar_init(&fullB[i], 1);
      tc::mbar_init(&emptyB[i], 1);
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], kEpiThreads / 32);
    }
    tc::fence_mbar_init();
    *s_abort = 0;
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 2 * D);
    tc::tmem_relinquish();
  }
  for (int i = tid; i < D / 2; i += kPipeThreads) ftab[i] = rope_tab[i];
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  auto abort_now = [&]() {
    *s_abort = 1;
    flag_error(status, DEV_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    int prev = -1, nb = -1, lastA[2] = {-1, -1}, lastB[2] = {-1, -1};
    for (int i = 0; i < hi - lo; ++i) {
      const int tile = lo + i, pair = tile / tpp, ti = tile - pair * tpp;
      const int bb = pair / h_kv;
      if (pair != prev) {
        ++nb;
        const int bs = nb % NB, use = nb / NB;
        bool ok = true;
        if (lane == 0) ok = *s_abort == 0 && tc::mbar_wait(&emptyB[bs], (use & 1) ^ 1, kWaitLimit);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0 && *s_abort == 0) abort_now();
          break;
        }
        if (lane == 0) tc::mbar_expect_tx(&fullB[bs], static_cast<uint32_t>(pipe_b_bytes(KB, D)));
        __syncwarp();
        for (int kb = lane; kb < KB; kb += 32)
          tc::tma_load_2d(sB + bs * pipe_b_bytes(KB, D) + kb * (D * 64), &mapBt, &fullB[bs], kb * 32,
                          pair * D);
        lastB[bs] = use;
        prev = pair;
      }
      const int st = i % S, use = i / S;
      const int row0 = ti * kTcRows, nrow = min(kTcRows, rows - row0), nch = nrow / c;
      bool ok = true;
      if (lane == 0) ok = *s_abort == 0 && tc::mbar_wait(&emptyA[st], (use & 1) ^ 1, kWaitLimit);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0 && *s_abort == 0) abort_now();
        break;
      }
      if (lane == 0) tc::mbar_expect_tx(&fullA[st], static_cast<uint32_t>(KB * nrow * 64));
      __syncwarp();
      const int32_t* srow = sel + static_cast<size_t>(pair) * k + row0 / c;
      unsigned char* dstA = sA + st * pipe_a_bytes(KB);
      for (int j = lane; j < nch * KB; j += 32) {
        const int ch = j / KB, kb = j - ch * KB;
        tc::tma_load_2d(dstA + kb * (kTcRows * 64) + ch * c * 64, &mapA, &fullA[st], kb * 32,
                        bb * s + srow[ch] * c);
      }
      lastA[st] = use;
    }
    // every copy issued has landed before the CTA may exit
    if (lane == 0) {
      for (int j = 0; j < 2; ++j) {
        if (lastA[j] >= 0) tc::mbar_wait(&fullA[j], lastA[j] & 1, kWaitLimit);
        if (lastB[j] >= 0) tc::mbar_wait(&fullB[j], lastB[j] & 1, kWaitLimit);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTcRows, D);
      int prev = -1, nb = -1, bs = 0;
      int issued = 0;
      for (int i = 0; i < hi - lo; ++i) {
        const int tile = lo + i, pair = tile / tpp;
        if (pair != prev) {
          ++nb;
          bs = nb % NB;
          if (*s_abort || !tc::mbar_wait(&fullB[bs], (nb / NB) & 1, kWaitLimit)) {
            if (!*s_abort) abort_now();
            break;
          }
          prev = pair;
        }
        const int st = i % S, acc = i & 1;
        if (*s_abort || !tc::mbar_wait(&fullA[st], (i / S) & 1, kWaitLimit) ||
            !tc::mbar_wait(&tempty[acc], ((i >> 1) & 1) ^ 1, kWaitLimit)) {
          if (!*s_abort) abort_now();
          break;
        }
        tc::fence_after();
        const uint32_t a0 = tc::smem_u32(sA + st * pipe_a_bytes(KB));
        const uint32_t b0 = tc::smem_u32(sB + bs * pipe_b_bytes(KB, D));
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * D);
        for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            const uint64_t ad = tc::desc_k_sw64(a0 + kb * (kTcRows * 64) + ks * 32, 512);
            const uint64_t bd = tc::desc_k_sw64(b0 + kb * (D * 64) + ks * 32, 512);
            tc::mma_bf16(d_tmem, ad, bd, idesc, (kb | ks) != 0);
          }
        }
        tc::mma_commit(&emptyA[st]);
        tc::mma_commit(&tfull[acc]);
        const bool last_of_pair = i == hi - lo - 1 || (tile + 1) / tpp != pair;
        if (last_of_pair) tc::mma_commit(&emptyB[bs]);
        ++issued;
      }
      // the MMAs issued have completed before TMEM is released
      if (issued > 0) tc::mbar_wait(&tfull[(issued - 1) & 1], ((issued - 1) >> 1) & 1, kWaitLimit);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int ew = warp - 2, quarter = warp & 3, grp = ew >> 2;
    const int row = quarter * 32 + lane;
    constexpr int Q = D / 8;                 // 16-byte chunks per output row
    constexpr int W = D / 4;                 // RoPE pairs per group
    for (int i = 0; i < hi - lo; ++i) {
      const int tile = lo + i, pair = tile / tpp, ti = tile - pair * tpp;
      const int row0 = ti * kTcRows, nrow = min(kTcRows, rows - row0);
      const int acc = i & 1;
      const int R = row0 + row;
      int pos = 0;
      if (row < nrow) pos = sel[static_cast<size_t>(pair) * k + R / c] * c + (R % c);
      bool ok = *s_abort == 0 && tc::mbar_wait(&tfull[acc], (i >> 1) & 1, kWaitLimit);
      ok = tc::named_sync_and(1, kEpiThreads, ok);
      if (!ok) {
        if (tid == 64 && !*s_abort) abort_now();
        break;
      }
      tc::fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * D + grp * W);
      float lo_v[W], hi_v[W];
      if constexpr (W == 32) {
        tc::tmem_ld32(taddr, lo_v);
        tc::tmem_ld32(taddr + D / 2, hi_v);
      } else {
        tc::tmem_ld16(taddr, lo_v);
        tc::tmem_ld16(taddr + D / 2, hi_v);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[acc]);
      uint32_t plo[W / 2], phi[W / 2];
#pragma unroll
      for (int j = 0; j < W; j += 2) {
        float y1[2], y2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float sn, cs;
          rope_sincos_fast(pos, ftab[grp * W + j + e], &sn, &cs);
          y1[e] = lo_v[j + e] * cs - hi_v[j + e] * sn;
          y2[e] = hi_v[j + e] * cs + lo_v[j + e] * sn;
        }
        const __nv_bfloat162 a = __floats2bfloat162_rn(y1[0], y1[1]);
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(y2[0], y2[1]);
        plo[j / 2] = *reinterpret_cast<const uint32_t*>(&a);
        phi[j / 2] = *reinterpret_cast<const uint32_t*>(&b2);
      }
#pragma unroll
      for (int q4 = 0; q4 < W / 8; ++q4) {
        const int qlo = grp * (W / 8) + q4, qhi = Q / 2 + qlo;
        stage[row * Q + (qlo ^ (row & (Q - 1)))] =
            make_uint4(plo[4 * q4], plo[4 * q4 + 1], plo[4 * q4 + 2], plo[4 * q4 + 3]);
        stage[row * Q + (qhi ^ (row & (Q - 1)))] =
            make_uint4(phi[4 * q4], phi[4 * q4 + 1], phi[4 * q4 + 2], phi[4 * q4 + 3]);
      }
      tc::named_sync(1, kEpiThreads);
      uint4* dst = reinterpret_cast<uint4*>(K_sp + (static_cast<size_t>(pair) * rows + row0) * D);
      for (int idx = tid - 64; idx < nrow * Q; idx += kEpiThreads) {
        const int rr = idx / Q, q = idx - rr * Q;
        dst[idx] = stage[rr * Q + (q ^ (rr & (Q - 1)))];
      }
      tc::named_sync(1, kEpiThreads);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 2 * D);
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
  const PipeShape ps = pipe_shape(c.p.r, D);
  if (ps.S == 0) return cudaErrorNotSupported;
  auto kern = k_rebuild_pipe<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ps.smem);
  if (e != cudaSuccess) return e;
  const int tiles = (c.p.k * c.p.c + kTcRows - 1) / kTcRows * c.p.h_kv * c.p.b;
  const int grid = std::min(c.nsm, tiles);
  kern<<<grid, kPipeThreads, ps.smem, st>>>(c.mapA, c.mapBt, c.sel, c.rope_tab,
                                            static_cast<bf16*>(c.K_sparse), c.p.b * c.p.h_kv,
                                            c.p.h_kv, c.p.s,
                                            c.p.r, c.p.c, c.p.k, ps.S, ps.NB, c.status);
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
