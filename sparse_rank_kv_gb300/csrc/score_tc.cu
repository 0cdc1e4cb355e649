// Landmark scores of ShadowKV's decode step on the tensor cores (Algorithm 2
// step 1): P = MatMul(Q, L^T) / sqrt(d) for every landmark of every
// (batch, KV head), with the G query heads of the KV head as the N side of
// the MMA (padded to 16 with zeros).  The landmark stream is the largest HBM
// read of a decode step, so this kernel is built to keep HBM busy:
//
//   persistent: one CTA per SM, each owning a contiguous range of 128-row
//               landmark tiles (a tile never spans two KV heads) for about
//               85% of the work; the remaining tiles go one at a time, from a
//               step-wide counter, to whichever CTAs finish first (SMs do not
//               all read HBM at the same rate)
//   warp 0    : TMA producer -- per tile (its number goes to a ring in shared
//               memory that the MMA warp passes on to the epilogue through a
//               per-accumulator barrier), d/64 boxes of 128 landmark rows x
//               64 columns and d/64 boxes of the head's q (16 rows; rows past
//               G are zero-filled by TMA) into a 5-stage shared-memory ring,
//               K-major with the 128-byte swizzle; lanes 0..2d/64-1 issue one
//               box each
//   warp 1    : tcgen05.mma (M=128, N=16, K=16) x (d/16) per tile into one of
//               eight TMEM accumulators; commits free the ring slot and publish
//               the accumulator
//   warps 2-17: epilogue, four warpgroups taking every fourth tile (eight
//               TMEM accumulators let the MMAs run ahead) -- one landmark row
//               per thread (TMEM lane), scale, store the G logits, and per
//               32-row warp the max (one integer warp reduction of
//               order-preserving keys) and sum of exp over the non-outlier
//               rows (softmax partials), and per 8 rows the max logit (the
//               selection bounds each 8-chunk group's S2 by it); the tile's
//               outlier-mask word is loaded while its MMAs run
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace skv {

constexpr int kScTile = 128;
constexpr int kScStages = 5;
constexpr int kScGroups = 4;     // epilogue warpgroups
constexpr int kScThreads = 64 + kScGroups * 128;
constexpr int kScAcc = 8;        // TMEM accumulators of 16 columns
constexpr int kScRing = 32;      // tile numbers in flight (producer <= 13 ahead of the epilogue, plus 4 end marks)
constexpr int kScStaticPct = 85; // share of the tiles assigned as contiguous ranges

__host__ __device__ constexpr int sc_stage_bytes(int D) { return (D / 32) * (kScTile + 16) * 64; }
__host__ __device__ constexpr int sc_smem_bytes(int D) {
  return 1024 /* alignment slack */ + 1024 /* header */ + kScStages * sc_stage_bytes(D);
}

template <int D, int G>
__global__ void __launch_bounds__(kScThreads, 1)
k_score_tc(const __grid_constant__ CUtensorMap mapL, const __grid_constant__ CUtensorMap mapQ,
           const uint32_t* __restrict__ mask, float* __restrict__ P, float2* __restrict__ part, int n,
           int ntile, int total_tiles, int per_cta, int* __restrict__ tail, int* __restrict__ tail_next,
           float* __restrict__ m8, int n8, float scale, int* __restrict__ status) {
  constexpr int KA = D / 64;                  // landmark and q boxes of 64 dims (128-byte swizzle)
  constexpr int A_BYTES = KA * kScTile * 128;
  constexpr int STAGE = sc_stage_bytes(D);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kScStages;
  uint64_t* tfull = empty + kScStages;
  uint64_t* tempty = tfull + kScAcc;
  uint64_t* tinfo = tempty + kScAcc;                        // [kScAcc]: the accumulator's tile number is set
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tinfo + kScAcc);
  int* ring = reinterpret_cast<int*>(smem + 512);          // [kScRing] tile numbers (-1: no more)
  unsigned char* stages = smem + 1024;

  // this CTA's contiguous range, then the shared tail [tail0, total_tiles)
  const int t_begin = per_cta * static_cast<int>(blockIdx.x);
  const int tail0 = per_cta * static_cast<int>(gridDim.x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  tc::grid_dep_launch();

  if (threadIdx.x == 0) {
    tc::prefetch_tensormap(&mapL);
    tc::prefetch_tensormap(&mapQ);
    for (int s = 0; s < kScStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kScAcc; ++a) {
      tc::mbar_init(&tfull[a], 1);
      tc::mbar_init(&tempty[a], 128);
      tc::mbar_init(&tinfo[a], 1);
    }
    tc::fence_mbar_init();
    // the next step's tail counter starts at zero
    if (blockIdx.x == 0) *tail_next = 0;
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 16 * kScAcc);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  // the queries may come from the stream's previous kernel, and the previous
  // step may still be reading the logits
  tc::grid_dep_wait();

  if (warp == 0) {
    // lane 0 waits for the stage and arms its barrier; lanes 0..2KB-1 then
    // issue one box each (landmark boxes, then q boxes), so the copies of a
    // stage are not serialised behind one thread's issue.  Tail tiles are
    // requested one ahead, so the atomic's round trip overlaps a stage.
    int next = -1;
    if (lane == 0 && per_cta == 0) next = tail0 + atomicAdd(tail, 1);
    // the landmarks are read once per step: evicted from L2 first, so that
    // the logits, partials and maxima this kernel writes stay there for the
    // selection
    const uint64_t evict_first = tc::l2_evict_first_policy();
    for (int i = 0;; ++i) {
      const int s = i % kScStages;
      const uint32_t ph = (i / kScStages) & 1;
      int tile = -1;
      if (lane == 0) {
        if (i < per_cta) {
          tile = t_begin + i;
          if (i + 1 == per_cta) next = tail0 + atomicAdd(tail, 1);
        } else {
          tile = next;
          if (tile < total_tiles) next = tail0 + atomicAdd(tail, 1);
        }
        if (tile >= total_tiles) tile = -1;
      }
      tile = __shfl_sync(0xffffffffu, tile, 0);
      bool ok = true;
      if (lane == 0) {
        ok = tc::mbar_wait(&empty[s], ph ^ 1, kWaitLimit);
        if (!ok) {
          flag_error(status, DEV_TIMEOUT);
        } else if (tile < 0) {
          // no more tiles: an end mark for the MMA warp and for each of the
          // four epilogue warpgroups' next tile
          for (int u = 0; u < kScGroups; ++u) ring[(i + u) % kScRing] = -1;
          tc::mbar_arrive(&full[s]);
        } else {
          ring[i % kScRing] = tile;
          tc::mbar_expect_tx(&full[s], STAGE);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0) || tile < 0) break;
      const int pair = tile / ntile, ti = tile - pair * ntile;
      unsigned char* st = stages + s * STAGE;
      if (lane < KA)
        tc::tma_load_2d_hint(st + lane * (kScTile * 128), &mapL, &full[s], lane * 64, pair * n + ti * kScTile,
                             evict_first);
      else if (lane < 2 * KA)
        tc::tma_load_3d(st + A_BYTES + (lane - KA) * (16 * 128), &mapQ, &full[s], (lane - KA) * 64, 0, pair);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kScTile, 16);
      for (int i = 0;; ++i) {
        const int s = i % kScStages;
        const uint32_t ph = (i / kScStages) & 1;
        const int a = i % kScAcc;
        const uint32_t tph = (i / kScAcc) & 1;
        if (!tc::mbar_wait(&full[s], ph, kWaitLimit) || !tc::mbar_wait(&tempty[a], tph ^ 1, kWaitLimit)) {
          flag_error(status, DEV_TIMEOUT);
          break;
        }
        if (ring[i % kScRing] < 0) {
          // the end: pass the mark to the epilogue warpgroups' next tiles,
          // each once its accumulator is free (keeps the barriers' phases)
          for (int u = 0; u < kScGroups; ++u) {
            const int au = (i + u) % kScAcc;
            if (u > 0 && !tc::mbar_wait(&tempty[au], (((i + u) / kScAcc) & 1) ^ 1, kWaitLimit)) {
              flag_error(status, DEV_TIMEOUT);
              break;
            }
            tc::mbar_arrive(&tinfo[au]);
          }
          break;
        }
        tc::fence_after();
        const uint32_t a0 = tc::smem_u32(stages + s * STAGE);
        const uint32_t b0 = a0 + A_BYTES;
        // K steps of 16 dims: landmarks and q in 128-byte swizzled boxes of
        // 64 dims (+32 B per step inside a box)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_bf16(tmem + a * 16, tc::desc_k_sw128(a0 + (kk >> 2) * (kScTile * 128) + (kk & 3) * 32, 1024),
                       tc::desc_k_sw128(b0 + (kk >> 2) * (16 * 128) + (kk & 3) * 32, 1024), idesc, kk != 0);
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&tfull[a]);
        tc::mbar_arrive(&tinfo[a]);
      }
    }
  } else {
    const int q4 = warp & 3;               // TMEM lane quarter of this warp
    const int eg = (warp - 2) >> 2;        // epilogue warpgroup: tiles eg, eg + kScGroups, ...
    const int row = q4 * 32 + lane;
    const int nw = (n + 31) >> 5;
    for (int i = eg;; i += kScGroups) {
      const int a = i % kScAcc;
      const uint32_t tph = (i / kScAcc) & 1;
      // the tile number (published by the MMA warp after the producer's),
      // then the outlier-mask word, loaded while the MMA runs
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&tinfo[a], tph, kWaitLimit))) {
        if (lane == 0) flag_error(status, DEV_TIMEOUT);
        break;
      }
      const int tile = ring[i % kScRing];
      if (tile < 0) break;
      const int pair = tile / ntile, ti = tile - pair * ntile;
      const int w = ti * (kScTile / 32) + q4;
      const uint32_t mword = w < nw ? __ldg(&mask[static_cast<size_t>(pair) * nw + w]) : 0u;
      const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&tfull[a], tph, kWaitLimit));
      if (!ok) {
        if (lane == 0) flag_error(status, DEV_TIMEOUT);
        break;
      }
      tc::fence_after();
      float acc[8];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + a * 16;
      if constexpr (G <= 4) tc::tmem_ld4(taddr, acc);
      else tc::tmem_ld8(taddr, acc);
      tc::fence_before();
      tc::mbar_arrive(&tempty[a]);
      const int j = ti * kScTile + row;
      const bool valid = j < n && !((mword >> lane) & 1u);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float x = acc[g] * scale;
        if (j < n) P[(static_cast<size_t>(pair) * G + g) * n + j] = x;
        const float m = from_order_key(__reduce_max_sync(0xffffffffu, order_key(valid ? x : -INFINITY)));
        const float e = warp_sum(valid ? __expf(x - m) : 0.f);
        if (lane == 0) part[((static_cast<size_t>(pair) * G + g) * ntile + ti) * 4 + q4] = make_float2(m, e);
        // the max over each 8 consecutive rows (-inf: none valid)
        float y = valid ? x : -INFINITY;
        y = fmaxf(y, __shfl_xor_sync(0xffffffffu, y, 1));
        y = fmaxf(y, __shfl_xor_sync(0xffffffffu, y, 2));
        y = fmaxf(y, __shfl_xor_sync(0xffffffffu, y, 4));
        if ((lane & 7) == 0 && j < n) m8[(static_cast<size_t>(pair) * G + g) * n8 + (j >> 3)] = y;
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 16 * kScAcc);
}

bool tc_score_supported(const shadowkv_params& p) {
  return p.dtype == SKV_DTYPE_BF16 && (p.d == 64 || p.d == 128);
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

cudaError_t make_score_map(Ctx& c) {
  c.tc_score = false;
  if (!tc_score_supported(c.p)) return cudaSuccess;
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t rows = static_cast<cuuint64_t>(c.p.b) * c.p.h_kv * c.n;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(c.p.d), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(c.p.d) * 2};
  const cuuint32_t box[2] = {64, kScTile};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(&c.mapL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.L, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  c.tc_score = true;
  return cudaSuccess;
}

// The queries live in the caller's buffer: a 3D view {d, G, b*h_kv} read in
// 128-byte swizzled boxes of 64 x 16 x 1, the rows past G being zero-filled.
cudaError_t encode_q_map(const Ctx& c, const void* q, CUtensorMap* map) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if (reinterpret_cast<uintptr_t>(q) % 16) return cudaErrorMisalignedAddress;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(c.p.d), static_cast<cuuint64_t>(c.G),
                              static_cast<cuuint64_t>(c.p.b) * c.p.h_kv};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(c.p.d) * 2,
                                 static_cast<cuuint64_t>(c.p.d) * 2 * c.G};
  const cuuint32_t box[3] = {64, 16, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t q_map_for(Ctx& c, const void* q, CUtensorMap* map) {
  if (!c.q_map || q != c.q_enc) {
    c.q_map = false;
    const cudaError_t e = encode_q_map(c, q, &c.mapQ);
    if (e != cudaSuccess) return e;
    c.q_enc = q;
    c.q_map = true;
  }
  *map = c.mapQ;
  return cudaSuccess;
}

template <int D, int G>
static cudaError_t score_tc_t(Ctx& c, const CUtensorMap& mq, cudaStream_t st) {
  const int smem = sc_smem_bytes(D);
  auto kern = k_score_tc<D, G>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int total = c.p.b * c.p.h_kv * c.ntile;
  const int grid = total < c.nsm ? total : c.nsm;
  const int per_cta = static_cast<int>(static_cast<long long>(total) * kScStaticPct / 100 / grid);
  const int par = static_cast<int>(c.t & 1);
  // each launch clears the other parity's tail counter for the next step;
  // after a step on the CUDA-core kernel this parity's is cleared here
  if (c.sc_last != c.t - 1) {
    e = cudaMemsetAsync(c.sc_ctr + par, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
  }
  c.sc_last = c.t;
  c.m8_step = c.t;
  // the prologue overlaps the tail of the stream's previous kernel
  return launch_pdl(kern, dim3(grid), dim3(kScThreads), static_cast<size_t>(smem), st, c.mapL, mq,
                    static_cast<const uint32_t*>(c.out_mask), c.logits, c.score_part, c.n, c.ntile, total,
                    per_cta, c.sc_ctr + par, c.sc_ctr + (par ^ 1), c.score_m8, (c.n + 7) / 8,
                    1.0f / sqrtf(static_cast<float>(D)), c.status);
}

template <int D>
static cudaError_t score_tc_d(Ctx& c, const CUtensorMap& mq, cudaStream_t st) {
  switch (c.G) {
    case 1: return score_tc_t<D, 1>(c, mq, st);
    case 2: return score_tc_t<D, 2>(c, mq, st);
    case 4: return score_tc_t<D, 4>(c, mq, st);
    default: return score_tc_t<D, 8>(c, mq, st);
  }
}

// Returns cudaErrorNotSupported when the tensor-core kernel does not apply
// (the caller then uses the CUDA-core kernel).
cudaError_t launch_score_tc(Ctx& c, const void* q, cudaStream_t st) {
  if (!c.tc_score || c.force_simt) return cudaErrorNotSupported;
  CUtensorMap mq;
  if (q_map_for(c, q, &mq) != cudaSuccess) return cudaErrorNotSupported;
  return c.p.d == 128 ? score_tc_d<128>(c, mq, st) : score_tc_d<64>(c, mq, st);
}

}  // namespace skv
