// The tensor-core key rebuild of ShadowKV's decode step (Algorithm 2 step 3,
// key branch, and the RoPE of step 4) as a device function, shared by its
// own launch and by the tensor-core attention's launch (whose first CTAs
// run it).
#pragma once
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace skv {

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
//   warps 2..17: epilogue, four groups of four warps (inside the attention's
//                launch warps 2..9, two groups); warp w reads TMEM lane
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
inline PipeShape pipe_shape(int r, int D) {
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
// The pipeline of one CTA of the tensor-core rebuild (the CTA's index cta of
// ncta; NEPI epilogue warps, 16 or, with records, 8; interleave: every
// ncta-th tile instead of a contiguous range).  With tile_done (the CTA is
// one of the attention launch's first CTAs), each tile's count is raised
// once its keys are in place, and the CTA keeps its TMEM allocation permit
// and ends with its barriers invalidated, so that it can go on as an
// attention CTA over the same shared memory.  Warps past 2 + NEPI only take
// part in the block-wide barriers.
template <int D, bool REC, int NEPI>
__device__ __forceinline__ void rebuild_pipe_body(
    unsigned char* smem_raw, int cta, int ncta, bool interleave, int32_t* __restrict__ tile_done,
    const bf16* __restrict__ A, const CUtensorMap& mapBt, const CUtensorMap& mapK,
    const int32_t* __restrict__ sel, const float2* __restrict__ rope_tab,
    const int32_t* __restrict__ miss_chunk, const int32_t* __restrict__ miss_slot,
    const int32_t* __restrict__ miss_base, const int32_t* __restrict__ hits,
    bf16* __restrict__ KV_slot, int n, int npairs, int h_kv, int s, int r, int c, int k,
    int S, int NB, int NS, int* __restrict__ status) {
  static_assert(NEPI == 16 || (REC && NEPI == 8), "epilogue warps");
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
      tc::mbar_init(&tempty[i], NEPI);
    }
    tc::fence_mbar_init();
    *s_abort = 0;
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kNAcc * D);
    // inside the attention's launch (tile_done given) the CTA allocates
    // again for its attention role, which a relinquished permit forbids
    if (tile_done == nullptr) tc::tmem_relinquish();
  }
  for (int i = tid; i < D / 2; i += static_cast<int>(blockDim.x)) ftab[i] = rope_tab[i];
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
      // exclusive prefix of the heads' tile counts, 32 heads per round (the
      // hit counts of up to 512 heads loaded before any is used)
      int base = 0;
      int hv[16];
      for (int p0 = 0; p0 < npairs; p0 += 32) {
        const int u = (p0 >> 5) & 15;
        if (u == 0) {
#pragma unroll
          for (int v = 0; v < 16; ++v) {
            const int pv = p0 + v * 32 + lane;
            hv[v] = pv < npairs ? hits[pv] : k;
          }
        }
        int hp = k;
#pragma unroll
        for (int v = 0; v < 16; ++v)
          if (v == u) hp = hv[v];
        const int p = p0 + lane;
        const int mrows = p < npairs ? max(0, k - hp) * c : 0;
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
  // this CTA's tiles: a contiguous range, or (interleave) every ncta-th tile
  // from tile cta, so that tiles complete roughly in order across CTAs
  const int ntl = interleave ? (cta < total ? (total - cta + ncta - 1) / ncta : 0) : hi - lo;
  auto tile_at = [&](int i) { return interleave ? cta + i * ncta : lo + i; };
  // both are loaded one tile ahead
  int first = 0;
  RowInfo first_row{0, 0};
  if (ntl > 0) {
    if (warp == 0) first = chunk_ids(tile_at(0));
    else if (warp >= 2 && warp < 2 + NEPI) first_row = row_info(tile_at(0));
  }

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    const uint32_t cbytes = static_cast<uint32_t>(c) * r * 2;   // one chunk of tiled A
    int prev = -1, nb = -1, lastA0 = -1, lastA1 = -1, lastB0 = -1, lastB1 = -1;
    int cid_next = first;
    for (int i = 0; i < ntl; ++i) {
      const int tile = tile_at(i);
      const Tile tl = tinfo(tile);
      const int pair = tl.pair, bb = pair / h_kv;
      const int cid = cid_next;
      if (i + 1 < ntl) cid_next = chunk_ids(tile_at(i + 1));
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
      for (int i = 0; i < ntl; ++i) {
        const int tile = tile_at(i), pair = tinfo(tile).pair;
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
        const bool last_of_pair = i == ntl - 1 || tinfo(tile_at(i + 1)).pair != pair;
        if (last_of_pair) tc::mma_commit(&emptyB[bs]);
        ++issued;
      }
      // the MMAs issued have completed, and the barriers their commits
      // signal have had their last arrivals, before TMEM (and, inside the
      // attention's launch, the shared memory) is released
      if (issued > 0) {
        const int il = issued - 1;
        if (tc::mbar_wait(&tfull[il % kNAcc], (il / kNAcc) & 1, kWaitLimit) && !*s_abort) {
          tc::mbar_wait(&emptyA[il % S], (il / S) & 1, kWaitLimit);
          tc::mbar_wait(&emptyB[bs], (nb / NB) & 1, kWaitLimit);
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + NEPI) {
    // ---------------------------------------------------------- epilogue
    const int ew = warp - 2, quarter = warp & 3, grp = ew >> 2;
    constexpr int Q = D / 8;                 // 16-byte chunks per output row
    constexpr int W = D / 8;                 // RoPE pairs per group
    RowInfo ri_next = first_row;
    for (int i = 0; i < ntl; ++i) {
      const int tile = tile_at(i);
      const Tile tl = tinfo(tile);
      const int pair = tl.pair, row0 = tl.row0, nrow = tl.nrow;
      const int acc = i % kNAcc;
      const RowInfo ri = ri_next;
      const int pos = ri.pos;
      if (i + 1 < ntl) ri_next = row_info(tile_at(i + 1));
      // the stores that last read this tile's staging buffer are done reading
      if (!REC && tid == 64) {
        if (NS == 1) tc::bulk_wait_read_all();
        else tc::bulk_wait_read_1();
      }
      unsigned char* stage = stage0 + (REC ? 0 : (i % NS) * (kTcRows * D * 2));
      bool ok = *s_abort == 0 && tc::mbar_wait(&tfull[acc], (i / kNAcc) & 1, kWaitLimit);
      ok = tc::named_sync_and(1, NEPI * 32, ok);
      if (!ok) {
        if (tid == 64 && !*s_abort) abort_now();
        break;
      }
      tc::fence_after();
      // column blocks of this warp group (NEPI / 4 groups share the d / 2
      // RoPE pairs); the accumulator is released after the last TMEM read
      for (int cg = grp; cg < 4; cg += NEPI / 4) {
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * D + cg * W);
      float lo_v[W], hi_v[W];
      if constexpr (W == 16) {
        tc::tmem_ld16(taddr, lo_v);
        tc::tmem_ld16(taddr + D / 2, hi_v);
      } else {
        tc::tmem_ld8(taddr, lo_v);
        tc::tmem_ld8(taddr + D / 2, hi_v);
      }
      if (cg + NEPI / 4 >= 4) {
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&tempty[acc]);
      }
      uint32_t plo[W / 2], phi[W / 2];
#pragma unroll
      for (int j = 0; j < W; j += 2) {
        float y1[2], y2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float sn, cs;
          rope_sincos_fast(pos, ftab[cg * W + j + e], &sn, &cs);
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
            const int qlo = cg * (W / 8) + q4;
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
          const int qlo = cg * (W / 8) + q4;
          st16(qlo, make_uint4(plo[4 * q4], plo[4 * q4 + 1], plo[4 * q4 + 2], plo[4 * q4 + 3]));
          st16(Q / 2 + qlo, make_uint4(phi[4 * q4], phi[4 * q4 + 1], phi[4 * q4 + 2], phi[4 * q4 + 3]));
        }
      }
      }   // column blocks
      if constexpr (!REC) {
        tc::fence_proxy_async_smem();
        tc::named_sync(1, NEPI * 32);
        if (tid == 64) {
          for (int cb = 0; cb < D / 64; ++cb)
            tc::tma_store_3d(&mapK, stage + cb * (kTcRows * 128), cb * 64, row0, pair);
          tc::bulk_commit();
        }
      } else if (tile_done != nullptr) {
        // the tile's keys are in their slot records (visible to the
        // consumers' bulk copies) before its count moves
        tc::fence_proxy_async_global();
        tc::named_sync(1, NEPI * 32);
        if (tid == 64) {
          tc::fence_acq_rel_gpu();
          atomicAdd(tile_done + tile, 1);
        }
      }
    }
  }
  if (!REC && tid == 64) tc::bulk_wait_all();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kNAcc * D);
  if constexpr (REC) {
    // inside the attention's launch the CTA reuses this shared memory next,
    // partly as the destination of its bulk copies (async proxy)
    tc::fence_proxy_async_smem();
    if (tid == 0) {
      for (int i = 0; i < 2; ++i) {
        tc::mbar_inval(&fullA[i]);
        tc::mbar_inval(&emptyA[i]);
        tc::mbar_inval(&fullB[i]);
        tc::mbar_inval(&emptyB[i]);
      }
      for (int i = 0; i < kNAcc; ++i) {
        tc::mbar_inval(&tfull[i]);
        tc::mbar_inval(&tempty[i]);
      }
    }
    __syncthreads();
  }
}


}  // namespace skv
