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


// ------------------------------------------------------------ tcgen05 path
// Persistent kernel, one CTA per SM.  The (batch, KV head, 128-row tile)
// work items of the k*c selected rows are split into contiguous ranges, one
// per CTA, so that consecutive tiles of a CTA mostly share the head's B.
//   warp 0     : producer -- for each tile the selected chunks of A into an
//                S-stage ring, one bulk copy per run of consecutive chunk ids
//                (tiled A: a chunk is c*r contiguous elements already in the
//                no-swizzle K-major order; gathering with TMA boxes of c rows
//                x 32 ranks costs one TMA instruction per 512 bytes, and
//                16-byte cp.async copies run out of requests in flight, both
//                far below HBM speed); the head's B^T into an NB-slot ring by
//                TMA (64-byte swizzle, [K block][row][64 B]) when the head
//                changes
//   warp 1     : TMEM allocation; lane 0 issues ceil(r/32) x 2 tcgen05.mma
//                (M=128, N=d, K=16) per tile into one of four TMEM
//                accumulators (d fp32 columns each)
//   warps 2..17: epilogue, four groups of four warps; warp w reads TMEM lane
//                quarter w % 4 (row = quarter*32 + lane), group g the RoPE
//                column pairs [g*d/8, (g+1)*d/8) and their partners at +d/2;
//                RoPE at the row's position, bf16 pack into a staging tile
//                laid out as TMA's 128-byte swizzle ([d/64][128 rows][128 B]),
//                then one thread stores it with d/64 TMA tensor stores that
//                complete while the next tile is computed.
// Barriers: fullA/emptyA per A stage, fullB/emptyB per B slot, tfull/tempty
// per accumulator.  Every wait is bounded; a timeout sets the status word and
// a shared abort flag that every role checks before its next wait.
constexpr int kTcRows = 128;
constexpr int kEpiThreads = 512;
constexpr int kPipeThreads = 64 + kEpiThreads;
constexpr int kNAcc = 4;          // TMEM accumulators (4 x d <= 512 columns)

struct PipeShape {
  int S, NB, NS, smem;   // A stages, B slots, output staging buffers
};
__host__ __device__ constexpr int pipe_a_bytes(int r) { return kTcRows * r * 2; }
__host__ __device__ constexpr int pipe_b_bytes(int KB, int D) { return KB * D * 64; }
__host__ __device__ constexpr int pipe_smem(int r, int D, int S, int NB, int NS) {
  return 1024 /* alignment slack */ + 1024 /* header */ + S * pipe_a_bytes(r) +
         NB * pipe_b_bytes((r + 31) / 32, D) + NS * kTcRows * D * 2 /* staging */;
}
static PipeShape pipe_shape(int r, int D) {
  const int cand[6][3] = {{2, 2, 2}, {2, 1, 2}, {2, 2, 1}, {2, 1, 1}, {1, 2, 1}, {1, 1, 1}};
  for (auto& x : cand) {
    const int sm = pipe_smem(r, D, x[0], x[1], x[2]);
    if (sm <= 227 * 1024) return {x[0], x[1], x[2], sm};
  }
  return {0, 0, 0, 0};
}

// REC = false: every selected row, in selection order, to K_sparse (TMA
// store).  REC = true (d = 128): only the chunks that missed the cache, from
// the step's miss list, into the K tiles of their slot records; the other
// slots keep the keys rebuilt at earlier steps (the rebuilt keys of a chunk
// depend only on A, B and its positions).
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
  const int cta = static_cast<int>(blockIdx.x) - nfetch, ncta = static_cast<int>(gridDim.x) - nfetch;
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int KB = (r + 31) / 32;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);   // <= 12 barriers
  uint64_t* fullA = bars;                                // [S]
  uint64_t* emptyA = bars + 2;                           // [S]
  uint64_t* fullB = bars + 4;                            // [NB]
  uint64_t* emptyB = bars + 6;                           // [NB]
  uint64_t* tfull = bars + 8;                            // [kNAcc]
  uint64_t* tempty = bars + 12;                          // [kNAcc]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 256);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + 260);
  float2* ftab = reinterpret_cast<float2*>(smem + 512);  // D/2 <= 64 entries
  unsigned char* sA = smem + 1024;
  const int a_bytes = pipe_a_bytes(r);
  unsigned char* sB = sA + S * a_bytes;
  unsigned char* stage0 = sB + NB * pipe_b_bytes(KB, D);   // NS x [D/64][128][128 B], 1024-aligned
  int* s_tp = reinterpret_cast<int*>(stage0 + NS * (kTcRows * D * 2));   // REC: tile prefix [npairs + 1]
  int* s_rows = s_tp + npairs + 1;                                      // REC: missed rows per head
  int* s_mb = s_rows + npairs;                                          // REC: miss-list start per head

  const int rows = k * c;
  const int tpp = (rows + kTcRows - 1) / kTcRows;        // tiles per (batch, KV head)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = (warp & 3) * 32 + lane;   // epilogue: TMEM lane = tile row
  int total = npairs * tpp, lo = 0, hi = 0;

  // a tile: its head, first row, rows, and the index of its first chunk in
  // the selection (REC: in the step's miss list)
  struct Tile {
    int pair, row0, nrow, e0;
  };
  auto tinfo = [&](int tile) -> Tile {
    if constexpr (REC) {
      int a = 0, b = npairs;   // the last head whose tiles start at or before `tile`
      while (b - a > 1) {
        const int m = (a + b) >> 1;
        if (s_tp[m] <= tile) a = m;
        else b = m;
      }
      const int r0 = (tile - s_tp[a]) * kTcRows;
      return {a, r0, min(kTcRows, s_rows[a] - r0), s_mb[a] + r0 / c};
    } else {
      const int pr = tile / tpp, r0 = (tile - pr * tpp) * kTcRows;
      return {pr, r0, min(kTcRows, rows - r0), pr * k + r0 / c};
    }
  };
  auto chunk_at = [&](int e, int pr) -> int {
    if constexpr (REC) return miss_chunk[e] - pr * n;
    else return sel[e];
  };
  // producer lane l: chunk id of the tile's l-th chunk (<= 128 / 8 chunks)
  auto chunk_ids = [&](int tile) {
    const Tile t = tinfo(tile);
    return lane < t.nrow / c ? chunk_at(t.e0 + lane, t.pair) : 0;
  };
  // epilogue thread: position of its row, and (REC) the slot its chunk fills
  struct RowInfo {
    int pos, slot;
  };
  auto row_info = [&](int tile) -> RowInfo {
    const Tile t = tinfo(tile);
    if (row >= t.nrow) return {0, 0};
    const int e = t.e0 + row / c;
    const int slot = REC ? miss_slot[e] - t.pair * k : 0;
    return {chunk_at(e, t.pair) * c + (row % c), slot};
  };
  if (!REC) tc::grid_dep_launch();
  if (tid == 0) {
    tc::prefetch_tensormap(&mapBt);
    if (!REC) tc::prefetch_tensormap(&mapK);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&fullA[i], 1);
      tc::mbar_init(&emptyA[i], 1);
      tc::mbar_init(&fullB[i], 1);
      tc::mbar_init(&emptyB[i], 1);
    }
    for (int i = 0; i < kNAcc; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], kEpiThreads / 32);
    }
    tc::fence_mbar_init();
    *s_abort = 0;
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kNAcc * D);
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
  // the selection may still be finishing: its chunk ids are read after this
  tc::grid_dep_wait();
  if (REC) tc::grid_dep_launch();
  if constexpr (REC) {
    if (warp == 0) {
      // exclusive prefix of the heads' tile counts, 32 heads per round
      int base = 0;
      for (int p0 = 0; p0 < npairs; p0 += 32) {
        const int p = p0 + lane;
        const int mrows = p < npairs ? max(0, k - hits[p]) * c : 0;
        const int nt = (mrows + kTcRows - 1) / kTcRows;
        int incl = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (p < npairs) {
          s_tp[p] = base + incl - nt;
          s_rows[p] = mrows;
          s_mb[p] = miss_base[p];
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) s_tp[npairs] = base;
    }
    __syncthreads();
    total = s_tp[npairs];
  }
  lo = static_cast<int>(static_cast<long long>(cta) * total / ncta);
  hi = static_cast<int>(static_cast<long long>(cta + 1) * total / ncta);
  // both are loaded one tile ahead
  int first = 0;
  RowInfo first_row{0, 0};
  if (hi > lo) {
    if (warp == 0) first = chunk_ids(lo);
    else if (warp >= 2) first_row = row_info(lo);
  }

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    const uint32_t cbytes = static_cast<uint32_t>(c) * r * 2;   // one chunk of tiled A
    int prev = -1, nb = -1, lastA0 = -1, lastA1 = -1, lastB0 = -1, lastB1 = -1;
    int cid_next = first;
    for (int i = 0; i < hi - lo; ++i) {
      const int tile = lo + i;
      const Tile tl = tinfo(tile);
      const int pair = tl.pair, bb = pair / h_kv;
      const int cid = cid_next;
      if (i + 1 < hi - lo) cid_next = chunk_ids(tile + 1);
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
        if (lane == 0)
          for (int kb = 0; kb < KB; ++kb)
            tc::tma_load_2d(sB + bs * pipe_b_bytes(KB, D) + kb * (D * 64), &mapBt, &fullB[bs],
                            kb * 32, pair * D);
        (bs ? lastB1 : lastB0) = use;
        prev = pair;
      }
      const int st = i % S, use = i / S;
      const int nch = tl.nrow / c;
      bool ok = true;
      if (lane == 0) ok = *s_abort == 0 && tc::mbar_wait(&emptyA[st], (use & 1) ^ 1, kWaitLimit);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0 && *s_abort == 0) abort_now();
        break;
      }
      if (lane == 0) tc::mbar_expect_tx(&fullA[st], static_cast<uint32_t>(nch) * cbytes);
      // lane l copies the run of consecutive chunk ids that starts at the
      // tile's l-th chunk (chunk ids ascend; consecutive ids are contiguous)
      const int cprev = __shfl_up_sync(0xffffffffu, cid, 1);
      const bool cont = lane > 0 && lane < nch && cid == cprev + 1;
      const unsigned long long cmask = __ballot_sync(0xffffffffu, cont);
      if (lane < nch && !cont) {
        const int len = __ffsll(~(cmask >> (lane + 1)));
        tc::bulk_load(sA + st * a_bytes + lane * cbytes,
                      A + (static_cast<size_t>(bb) * s + static_cast<size_t>(cid) * c) * r,
                      static_cast<uint32_t>(len) * cbytes, &fullA[st]);
      }
      (st ? lastA1 : lastA0) = use;
    }
    // every copy issued has landed before the CTA may exit
    if (lane == 0) {
      if (lastA0 >= 0) tc::mbar_wait(&fullA[0], lastA0 & 1, kWaitLimit);
      if (lastA1 >= 0) tc::mbar_wait(&fullA[1], lastA1 & 1, kWaitLimit);
      if (lastB0 >= 0) tc::mbar_wait(&fullB[0], lastB0 & 1, kWaitLimit);
      if (lastB1 >= 0) tc::mbar_wait(&fullB[1], lastB1 & 1, kWaitLimit);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTcRows, D);
      int prev = -1, nb = -1, bs = 0;
      int issued = 0;
      for (int i = 0; i < hi - lo; ++i) {
        const int tile = lo + i, pair = tinfo(tile).pair;
        if (pair != prev) {
          ++nb;
          bs = nb % NB;
          if (*s_abort || !tc::mbar_wait(&fullB[bs], (nb / NB) & 1, kWaitLimit)) {
            if (!*s_abort) abort_now();
            break;
          }
          prev = pair;
        }
        const int st = i % S, acc = i % kNAcc;
        if (*s_abort || !tc::mbar_wait(&fullA[st], (i / S) & 1, kWaitLimit) ||
            !tc::mbar_wait(&tempty[acc], ((i / kNAcc) & 1) ^ 1, kWaitLimit)) {
          if (!*s_abort) abort_now();
          break;
        }
        tc::fence_after();
        const uint32_t a0 = tc::smem_u32(sA + st * a_bytes);
        const uint32_t b0 = tc::smem_u32(sB + bs * pipe_b_bytes(KB, D));
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * D);
        // K steps of 16: A = two core matrices (128 B apart, 8-row groups
        // 16r bytes apart); B = half of a 64-byte swizzled K block
        for (int ks = 0; ks < r / 16; ++ks) {
          const uint64_t ad = tc::desc_k_none(a0 + ks * 256, 128, static_cast<uint32_t>(r) * 16);
          const uint64_t bd = tc::desc_k_sw64(b0 + (ks >> 1) * (D * 64) + (ks & 1) * 32, 512);
          tc::mma_bf16(d_tmem, ad, bd, idesc, ks != 0);
        }
        tc::mma_commit(&emptyA[st]);
        tc::mma_commit(&tfull[acc]);
        const bool last_of_pair = i == hi - lo - 1 || tinfo(tile + 1).pair != pair;
        if (last_of_pair) tc::mma_commit(&emptyB[bs]);
        ++issued;
      }
      // the MMAs issued have completed before TMEM is released
      if (issued > 0)
        tc::mbar_wait(&tfull[(issued - 1) % kNAcc], ((issued - 1) / kNAcc) & 1, kWaitLimit);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int ew = warp - 2, quarter = warp & 3, grp = ew >> 2;
    constexpr int Q = D / 8;                 // 16-byte chunks per output row
    constexpr int W = D / 8;                 // RoPE pairs per group
    RowInfo ri_next = first_row;
    for (int i = 0; i < hi - lo; ++i) {
      const int tile = lo + i;
      const Tile tl = tinfo(tile);
      const int pair = tl.pair, row0 = tl.row0, nrow = tl.nrow;
      const int acc = i % kNAcc;
      const RowInfo ri = ri_next;
      const int pos = ri.pos;
      if (i + 1 < hi - lo) ri_next = row_info(tile + 1);
      // the stores that last read this tile's staging buffer are done reading
      if (!REC && tid == 64) {
        if (NS == 1) tc::bulk_wait_read_all();
        else tc::bulk_wait_read_1();
      }
      unsigned char* stage = stage0 + (REC ? 0 : (i % NS) * (kTcRows * D * 2));
      bool ok = *s_abort == 0 && tc::mbar_wait(&tfull[acc], (i / kNAcc) & 1, kWaitLimit);
      ok = tc::named_sync_and(1, kEpiThreads, ok);
      if (!ok) {
        if (tid == 64 && !*s_abort) abort_now();
        break;
      }
      tc::fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * D + grp * W);
      float lo_v[W], hi_v[W];
      if constexpr (W == 16) {
        tc::tmem_ld16(taddr, lo_v);
        tc::tmem_ld16(taddr + D / 2, hi_v);
      } else {
        tc::tmem_ld8(taddr, lo_v);
        tc::tmem_ld8(taddr + D / 2, hi_v);
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
      if constexpr (REC) {
        // the row's 16-byte pieces go straight to the K tile of its slot's
        // group record: piece qq of row u at qq * 128 + u * 16 bytes
        if (row < nrow) {
          const int u = row % c;
          uint4* recp = reinterpret_cast<uint4*>(
              KV_slot + ((static_cast<size_t>(pair) * k + ri.slot) * (c / 8) + (u >> 3)) * 2048);
#pragma unroll
          for (int q4 = 0; q4 < W / 8; ++q4) {
            const int qlo = grp * (W / 8) + q4;
            recp[qlo * 8 + (u & 7)] = make_uint4(plo[4 * q4], plo[4 * q4 + 1], plo[4 * q4 + 2], plo[4 * q4 + 3]);
            recp[(Q / 2 + qlo) * 8 + (u & 7)] =
                make_uint4(phi[4 * q4], phi[4 * q4 + 1], phi[4 * q4 + 2], phi[4 * q4 + 3]);
          }
        }
      } else {
        // 16-byte unit qq of the row: column block qq/8, unit qq%8 XOR row%8
        auto st16 = [&](int qq, uint4 v) {
          const int off = (qq >> 3) * (kTcRows * 128) + row * 128 + (((qq & 7) ^ (row & 7)) << 4);
          *reinterpret_cast<uint4*>(stage + off) = v;
        };
#pragma unroll
        for (int q4 = 0; q4 < W / 8; ++q4) {
          const int qlo = grp * (W / 8) + q4;
          st16(qlo, make_uint4(plo[4 * q4], plo[4 * q4 + 1], plo[4 * q4 + 2], plo[4 * q4 + 3]));
          st16(Q / 2 + qlo, make_uint4(phi[4 * q4], phi[4 * q4 + 1], phi[4 * q4 + 2], phi[4 * q4 + 3]));
        }
        tc::fence_proxy_async_smem();
        tc::named_sync(1, kEpiThreads);
        if (tid == 64) {
          for (int cb = 0; cb < D / 64; ++cb)
            tc::tma_store_3d(&mapK, stage + cb * (kTcRows * 128), cb * 64, row0, pair);
          tc::bulk_commit();
        }
      }
    }
  }
  if (!REC && tid == 64) tc::bulk_wait_all();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kNAcc * D);
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
