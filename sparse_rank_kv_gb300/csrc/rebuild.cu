// Key rebuild of ShadowKV's decode step (Algorithm 2 step 3, key branch, and
// the RoPE of step 4): K_sparse = RoPE(MatMul(Gather(A, I), B)) for the k
// selected chunks of every (batch, KV head), at each token's position.
//
// Output layout: K_sparse[b][h][pos*c + u][:] for the pos-th selected chunk
// (ascending chunk order) and in-chunk token u.
//
// Layout of A in HBM.  Where the tensor-core path applies, the rows of the
// chunked region [0, n*c) are stored in 8-token groups, each group as r/8
// core matrices of 8 tokens x 8 ranks (128 contiguous bytes):
//   element (t, j) at  (t/8) * 8r + (j/8) * 64 + (t%8) * 8 + j%8
// within its batch's s*r block (tokens >= n*c stay row-major).  A chunk of c
// tokens (c a multiple of 8) is then one contiguous block of c*r elements in
// exactly the order the tensor core reads a K-major operand without swizzle,
// so a single bulk copy moves it to shared memory.  The layout is internal:
// export returns A row-major.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "rebuild_pipe.cuh"

namespace skv {

constexpr int kRbRows = 64;       // output rows per block

// Offset of A element (token t, rank j) within its batch's block in the
// tiled layout.
__host__ __device__ __forceinline__ size_t a_tiled_index(int t, int j, int r) {
  return static_cast<size_t>(t >> 3) * (8 * r) + static_cast<size_t>(j >> 3) * 64 + (t & 7) * 8 + (j & 7);
}

// In-place conversion of the chunked region of A between row-major and the
// tiled layout, one warp per 8-token group: the group's 8*r elements
// (r/8 16-byte pieces per row, <= 256 pieces) are read into registers before
// any lane writes.  to_tiled = 1: row-major -> tiled, 0: back.
__global__ void __launch_bounds__(256)
k_tile_a(uint4* __restrict__ A, int s, int r, int groups_per_batch, long long total_groups, int to_tiled) {
  const int lane = threadIdx.x & 31;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int QR = r / 8, npc = 8 * QR;          // pieces per row, per group
  for (long long g = w0; g < total_groups; g += nw) {
    const long long bb = g / groups_per_batch, gi = g - bb * groups_per_batch;
    uint4* base = A + (bb * s * r + gi * 8 * r) / 8;   // 8 bf16 per piece
    uint4 v[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int i = lane + 32 * m;
      if (i < npc) v[m] = base[i];
    }
    __syncwarp();
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int i = lane + 32 * m;   // source piece index
      if (i < npc) {
        int dst;
        if (to_tiled) {            // row-major piece (u, q) -> core matrix q, row u
          const int u = i / QR, q = i - u * QR;
          dst = q * 8 + u;
        } else {                   // tiled piece (q, u) -> row-major (u, q)
          const int q = i >> 3, u = i & 7;
          dst = u * QR + q;
        }
        base[dst] = v[m];
      }
    }
  }
}

cudaError_t launch_tile_a(Ctx& c, int to_tiled, cudaStream_t st) {
  if (!c.a_tiled) return cudaSuccess;
  const int gpb = c.n * c.p.c / 8;
  const long long total = static_cast<long long>(gpb) * c.p.b;
  const int blocks = static_cast<int>(std::min<long long>((total + 7) / 8, 4LL * c.nsm));
  kbegin(c, K_MISC, st);
  k_tile_a<<<blocks, 256, 0, st>>>(static_cast<uint4*>(c.A), c.p.s, c.p.r, gpb, total, to_tiled);
  kend(c, K_MISC, st);
  return cudaGetLastError();
}
constexpr int kRbThreads = 256;

// SIMT reference kernel: fp32 products and sums.  Shared memory holds the
// block's 64 gathered A rows and the head's B (both as fp32).  Thread
// (ty, tx) owns rows ty + 8 i and columns tx + 32 j, so the RoPE partners
// (col, col + D/2) are in the same thread.
template <typename T, int D>
__global__ void __launch_bounds__(kRbThreads)
k_rebuild_simt(const T* __restrict__ A, const T* __restrict__ Bt, const int32_t* __restrict__ sel,
               const float2* __restrict__ rope_tab, T* __restrict__ K_sp, int h_kv, int s, int r,
               int c, int k, int a_tiled, const int32_t* __restrict__ sel_slot, T* __restrict__ KV_slot) {
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
      const size_t in_batch = a_tiled ? a_tiled_index(tok, kk, r) : static_cast<size_t>(tok) * r + kk;
      v = Ty<T>::to_f(A[static_cast<size_t>(bb) * s * r + in_batch]);
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
    // row-major K_sparse, or (records) the K tile of the chunk's slot record:
    // element (row u, column j) at (j / 8) * 64 + (u % 8) * 8 + j % 8
    T* dst;
    int u8 = 0;
    if (KV_slot != nullptr) {
      const int u = R % c, slot = sel_slot[static_cast<size_t>(pair) * k + R / c];
      dst = KV_slot + ((static_cast<size_t>(pair) * k + slot) * (c / 8) + (u >> 3)) * 2048;
      u8 = u & 7;
    } else {
      dst = K_sp + (static_cast<size_t>(pair) * rows + R) * D;
    }
    auto at = [&](int j) -> T& { return KV_slot != nullptr ? dst[(j >> 3) * 64 + u8 * 8 + (j & 7)] : dst[j]; };
#pragma unroll
    for (int j = 0; j < CJ / 2; ++j) {
      const int col = tx + 32 * j;
      float sn, cs;
      rope_sincos(pos, rope_tab[col], &sn, &cs);
      const float x1 = acc[i][j], x2 = acc[i][j + CJ / 2];
      at(col) = Ty<T>::from_f(x1 * cs - x2 * sn);
      at(col + D / 2) = Ty<T>::from_f(x2 * cs + x1 * sn);
    }
  }
}


template <int D, bool REC>
__global__ void __launch_bounds__(kPipeThreads, 1)
k_rebuild_pipe(const bf16* __restrict__ A, const __grid_constant__ CUtensorMap mapBt,
               const __grid_constant__ CUtensorMap mapK,
               const int32_t* __restrict__ sel, const float2* __restrict__ rope_tab,
               const int32_t* __restrict__ miss_chunk, const int32_t* __restrict__ miss_slot,
               const int32_t* __restrict__ miss_base, const int32_t* __restrict__ hits,
               bf16* __restrict__ KV_slot, int n, int npairs, int h_kv, int s, int r, int c, int k,
               int S, int NB, int NS, const bf16* __restrict__ vcpu, const int32_t* __restrict__ miss_total,
               int par, int nfetch, int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  if constexpr (REC) {
    // the first nfetch CTAs move the step's value misses over the host link
    // while the others rebuild the missed chunks' keys
    if (static_cast<int>(blockIdx.x) < nfetch) {
      // the attention launched behind may start once the selection is
      // complete (it reads the selection, not this launch's results, until
      // its own wait)
      tc::grid_dep_wait();
      tc::grid_dep_launch();
      fetch_value_groups(vcpu, KV_slot, miss_chunk, miss_slot, miss_total[par], s, n, c, k, npairs,
                         static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x,
                         static_cast<long long>(nfetch) * blockDim.x, status);
      return;
    }
  }
  rebuild_pipe_body<D, REC, kEpiThreads / 32>(
      smem_raw, static_cast<int>(blockIdx.x) - nfetch, static_cast<int>(gridDim.x) - nfetch, false, nullptr, A,
      mapBt, mapK, sel, rope_tab, miss_chunk, miss_slot, miss_base, hits, KV_slot, n, npairs, h_kv, s, r, c,
      k, S, NB, NS, status);
}

bool tc_rebuild_supported(const shadowkv_params& p) {
  return p.dtype == SKV_DTYPE_BF16 && (p.d == 64 || p.d == 128) && p.c % 8 == 0 &&
         kTcRows % p.c == 0 && p.r % 16 == 0 && p.r <= 256 && pipe_shape(p.r, p.d).S > 0;
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

// 3D bf16 map over K_sparse [pairs][k*c][d]: box 64 columns x 128 rows x 1
// with the 128-byte swizzle (rows past k*c of a head are clipped on store).
static cudaError_t encode_ksparse(CUtensorMap* map, void* base, int D, int rows, uint64_t pairs) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), pairs};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kTcRows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_rebuild_maps(Ctx& c) {
  c.tc_rebuild = false;
  c.a_tiled = false;
  if (!tc_rebuild_supported(c.p)) return cudaSuccess;
  const uint64_t pairs = static_cast<uint64_t>(c.p.b) * c.p.h_kv;
  cudaError_t e = encode_rows(&c.mapBt, c.Bt, pairs * c.p.d, c.p.r, c.p.d);
  if (e == cudaSuccess && !c.kv_rec) e = encode_ksparse(&c.mapK, c.K_sparse, c.p.d, c.p.k * c.p.c, pairs);
  if (e == cudaSuccess) c.tc_rebuild = c.a_tiled = true;
  return e;
}

template <int D, bool REC>
static cudaError_t rebuild_tc(Ctx& c, cudaStream_t st) {
  const int npairs = c.p.b * c.p.h_kv;
  PipeShape ps = pipe_shape(c.p.r, D);
  if (REC) {
    // no staging tiles; the head tile tables instead
    ps = {0, 0, 0, 0};
    const int tables = (3 * npairs + 1) * 4;
    const int cand[4][2] = {{2, 2}, {2, 1}, {1, 2}, {1, 1}};
    for (auto& x : cand) {
      const int sm = pipe_smem(c.p.r, D, x[0], x[1], 0) + tables;
      if (sm <= 227 * 1024) { ps = {x[0], x[1], 0, sm}; break; }
    }
  }
  if (ps.S == 0 || !c.a_tiled) return cudaErrorNotSupported;
  auto kern = k_rebuild_pipe<D, REC>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), ps.smem);
  if (e != cudaSuccess) return e;
  const int tiles = (c.p.k * c.p.c + kTcRows - 1) / kTcRows * npairs;
  // records: the value fetch runs in the attention's launch, or in this one
  // on its own CTAs; otherwise it runs on a side stream and the rebuild
  // leaves it its SMs
  const int nfetch = REC && rebuild_fetches(c) ? std::min(c.fetch_sms, c.nsm / 2) : 0;
  const int sms = REC ? std::min(kRebuildSMsRec, c.nsm - nfetch)
                      : c.nsm > 2 * c.fetch_sms ? c.nsm - c.fetch_sms : c.nsm;
  const int grid = nfetch + std::min(sms, tiles);
  return launch_pdl(kern, dim3(grid), dim3(kPipeThreads), ps.smem, st, static_cast<const bf16*>(c.A),
                    c.mapBt, c.mapK, static_cast<const int32_t*>(c.sel),
                    static_cast<const float2*>(c.rope_tab), static_cast<const int32_t*>(c.miss_chunk),
                    static_cast<const int32_t*>(c.miss_slot), static_cast<const int32_t*>(c.miss_base),
                    static_cast<const int32_t*>(c.hits), static_cast<bf16*>(c.KV_slot), c.n, npairs, c.p.h_kv,
                    c.p.s, c.p.r, c.p.c, c.p.k, ps.S, ps.NB, ps.NS,
                    static_cast<const bf16*>(REC ? c.v_cpu_dev : nullptr),
                    static_cast<const int32_t*>(c.miss_count), static_cast<int>(c.t & 1), nfetch, c.status);
}

bool rebuild_fetches(const Ctx& c) {
  return c.tc_rebuild && !c.force_simt && c.kv_rec && c.a_tiled && !attn_fetches(c);
}

template <typename T, int D>
static cudaError_t rebuild_simt(Ctx& c, cudaStream_t st) {
  const size_t smem = sizeof(float) * (static_cast<size_t>(kRbRows) * c.p.r + static_cast<size_t>(c.p.r) * D);
  auto kern = k_rebuild_simt<T, D>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((c.p.k * c.p.c + kRbRows - 1) / kRbRows, c.p.b * c.p.h_kv);
  kern<<<grid, kRbThreads, smem, st>>>(static_cast<const T*>(c.A), static_cast<const T*>(c.Bt),
                                        c.sel, c.rope_tab, static_cast<T*>(c.K_sparse), c.p.h_kv,
                                        c.p.s, c.p.r, c.p.c, c.p.k, c.a_tiled ? 1 : 0, c.sel_slot,
                                        static_cast<T*>(c.KV_slot));
  return cudaGetLastError();
}

cudaError_t launch_rebuild(Ctx& c, cudaStream_t st) {
  kbegin(c, K_REBUILD, st);
  cudaError_t e;
  if (c.tc_rebuild && !c.force_simt && c.kv_rec)
    e = rebuild_tc<128, true>(c, st);
  else if (c.tc_rebuild && !c.force_simt)
    e = c.p.d == 128 ? rebuild_tc<128, false>(c, st) : rebuild_tc<64, false>(c, st);
  else if (c.p.dtype == SKV_DTYPE_BF16)
    e = c.p.d == 128 ? rebuild_simt<bf16, 128>(c, st) : rebuild_simt<bf16, 64>(c, st);
  else
    e = c.p.d == 128 ? rebuild_simt<float, 128>(c, st) : rebuild_simt<float, 64>(c, st);
  kend(c, K_REBUILD, st);
  return e;
}

}  // namespace skv
