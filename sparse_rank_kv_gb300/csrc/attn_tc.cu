// Sparse attention of ShadowKV's decode step (Algorithm 2 step 4) on the
// tensor cores, for bf16 state with d = 128: out = softmax(q K^T / sqrt(d)) V
// over [outliers; RoPE(K_sparse); local window], the G query heads of a KV
// head sharing every K/V row.
//
// Work items are 128-token pieces of one segment (outliers, rebuilt chunks,
// local window) of one (batch, KV head); one persistent CTA per SM owns a
// contiguous range of items.
//   warp 0     : producer -- the head's q (TMA, 16 rows of which the rows
//                past G read as zeros) into a 2-slot ring when the head
//                changes; per item the keys and values by bulk copies into a
//                3-stage ring.  Keys and values are stored by 8-token group
//                in 4 KB records laid out as the tensor core's no-swizzle
//                K-major tiles: K ([d/8][token%8][d%8], 2 KB), then V^T
//                ([d/8][d%8][token%8], 2 KB); a selected chunk is one copy
//                from its cache slot, the outliers or the local window one
//                copy per item.
//   warp 1     : tcgen05.mma.  S = K q^T (M = 128 tokens, N = 16, K = d) into
//                one of two TMEM S buffers; after the softmax warps publish
//                P, O = V^T P^T (M = d, N = 16, K = 128 tokens) into one of
//                two TMEM O buffers.  The warp polls both queues and issues
//                whichever product is ready, so P V never waits for the next
//                item's loads.
//   warps 2..5 : softmax and accumulation, thread = TMEM lane: for S the
//                token row (scale, mask, head maxima by integer warp
//                reductions, p = 2^(s - m), bf16 P^T into shared memory, head
//                sums), for O the dimension d (running rescale and add).
//                When the head changes (or the range ends) the CTA writes one
//                partial (max, sum, sum p v) per query head in the slot of
//                its first item of that head; the CTA that completes a head's
//                last items (atomic count) combines the partials in slot
//                order (the slots follow from the fixed item ranges).
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace skv {

constexpr int kAtT = 128;                    // tokens per item
constexpr int kAtD = 128;                    // head dimension handled here
constexpr int kAtStages = 3;
constexpr int kAtThreads = 192;
constexpr int kAtSoft = 128;                 // softmax / accumulation threads
constexpr int kAtStage = kAtT / 8 * 4096;   // 16 group records (K tile | V^T tile)
constexpr int kAtQBytes = 16 * kAtD * 2;     // q: 4 x [16 rows][64 B]
constexpr int kAtPBytes = 16 * kAtT * 2;     // P^T: 16 x 128 bf16
__host__ __device__ constexpr int at_smem_bytes() {
  return 1024 /* alignment slack */ + kAtStages * kAtStage + 2 * kAtQBytes + 2 * kAtPBytes +
         1024 /* barriers, reductions */;
}

struct AtSeg {
  int seg, t0, cnt;
};
__device__ __forceinline__ AtSeg at_item(int j, int i_out, int i_sp, int n_out, int n_sp, int n_loc) {
  if (j < i_out) return {0, j * kAtT, min(kAtT, n_out - j * kAtT)};
  j -= i_out;
  if (j < i_sp) return {1, j * kAtT, min(kAtT, n_sp - j * kAtT)};
  j -= i_sp;
  return {2, j * kAtT, min(kAtT, n_loc - j * kAtT)};
}

template <int G>
__global__ void __launch_bounds__(kAtThreads, 1)
k_attn_tc(const __grid_constant__ CUtensorMap mapQ, const bf16* __restrict__ KV_out,
          const bf16* __restrict__ KV_slot, const int32_t* __restrict__ sel_slot,
          const bf16* __restrict__ KV_loc,
          bf16* __restrict__ out, float* __restrict__ part, int32_t* __restrict__ ticket, int n_out,
          int n_sp, int n_loc, int loc_cap, int c, int k, int npairs, int max_splits, float scale_log2,
          int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* stages = smem;
  unsigned char* qbuf = stages + kAtStages * kAtStage;    // [2][kAtQBytes]
  unsigned char* pbuf = qbuf + 2 * kAtQBytes;             // [2][kAtPBytes]
  unsigned char* misc = pbuf + 2 * kAtPBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);     // [kAtStages]
  uint64_t* empty = full + kAtStages;                     // [kAtStages]
  uint64_t* qfull = empty + kAtStages;                    // [2]
  uint64_t* qempty = qfull + 2;                           // [2]
  uint64_t* sfull = qempty + 2;                           // [2]
  uint64_t* sempty = sfull + 2;                           // [2]
  uint64_t* pfull = sempty + 2;                           // [2]
  uint64_t* ofull = pfull + 2;                            // [2]
  uint64_t* oempty = ofull + 2;                           // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 256);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + 260);
  int* s_last = reinterpret_cast<int*>(misc + 264);
  float* red = reinterpret_cast<float*>(misc + 512);      // [2][4][8]

  const int i_out = (n_out + kAtT - 1) / kAtT, i_sp = (n_sp + kAtT - 1) / kAtT,
            i_loc = (n_loc + kAtT - 1) / kAtT;
  const int nsplit = i_out + i_sp + i_loc;
  const int total = npairs * nsplit;
  const int lo = static_cast<int>(static_cast<long long>(blockIdx.x) * total / gridDim.x);
  const int hi = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * total / gridDim.x);
  const int nit = hi - lo;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  tc::grid_dep_launch();

  if (tid == 0) {
    tc::prefetch_tensormap(&mapQ);
    for (int i = 0; i < kAtStages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&qfull[i], 1);
      tc::mbar_init(&qempty[i], 1);
      tc::mbar_init(&sfull[i], 1);
      tc::mbar_init(&sempty[i], kAtSoft / 32);
      tc::mbar_init(&pfull[i], 1);
      tc::mbar_init(&ofull[i], 1);
      tc::mbar_init(&oempty[i], kAtSoft / 32);
    }
    tc::fence_mbar_init();
    *s_abort = 0;
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, 64);
    tc::tmem_relinquish();
  }
  // the P rows past G are multiplied by zero values of V: start them at
  // zero so that they are finite (the producer does the same for the value
  // record that pads a partial item to 16 tokens)
  for (int i = tid; i < 2 * kAtPBytes / 16; i += kAtThreads)
    reinterpret_cast<uint4*>(pbuf)[i] = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async_smem();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  auto abort_now = [&]() {
    if (!*s_abort) {
      *s_abort = 1;
      flag_error(status, DEV_TIMEOUT);
    }
  };
  // the rebuild may still be finishing: its keys are read after this
  tc::grid_dep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int prev = -1, nq = -1, lastA[kAtStages], lastQ[2] = {-1, -1};
#pragma unroll
    for (int i = 0; i < kAtStages; ++i) lastA[i] = -1;
    for (int it = 0; it < nit; ++it) {
      const int item = lo + it, pair = item / nsplit, j = item - pair * nsplit;
      const AtSeg sg = at_item(j, i_out, i_sp, n_out, n_sp, n_loc);
      bool ok = true;
      if (pair != prev) {
        ++nq;
        const int qs = nq & 1, use = nq >> 1;
        if (lane == 0) ok = !*s_abort && tc::mbar_wait(&qempty[qs], (use & 1) ^ 1, kWaitLimit);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          if (lane == 0) abort_now();
          break;
        }
        if (lane == 0) {
          tc::mbar_expect_tx(&qfull[qs], kAtQBytes);
#pragma unroll
          for (int kb = 0; kb < kAtD / 32; ++kb)
            tc::tma_load_3d(qbuf + qs * kAtQBytes + kb * (16 * 64), &mapQ, &qfull[qs], kb * 32, 0, pair);
        }
        lastQ[qs] = use;
        prev = pair;
      }
      const int st = it % kAtStages, use = it / kAtStages;
      // cache slots of the item's chunks (lane = chunk), loaded before the wait
      const int ch0 = sg.t0 / c, nch = sg.seg == 1 ? sg.cnt / c : 0;
      const int slot = lane < nch ? sel_slot[static_cast<size_t>(pair) * k + ch0 + lane] : 0;
      if (lane == 0) ok = !*s_abort && tc::mbar_wait(&empty[st], (use & 1) ^ 1, kWaitLimit);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) abort_now();
        break;
      }
      unsigned char* sR = stages + st * kAtStage;
      const int groups = (sg.cnt + 7) >> 3;
      if ((groups & 1) && groups < kAtT / 8) {
        // P V runs over whole 16-token steps: the V^T half of the record
        // after an odd count of groups meets zero weights and must be finite
        uint4* pad = reinterpret_cast<uint4*>(sR + groups * 4096 + 2048);
#pragma unroll
        for (int i = 0; i < 2048 / 16 / 32; ++i) pad[i * 32 + lane] = make_uint4(0, 0, 0, 0);
        tc::fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc::mbar_expect_tx(&full[st], static_cast<uint32_t>(groups * 4096));
        if (sg.seg == 0)
          tc::bulk_load(sR, KV_out + (static_cast<size_t>(pair) * n_out + sg.t0) * 2 * kAtD,
                        static_cast<uint32_t>(groups * 4096), &full[st]);
        else if (sg.seg == 2)
          tc::bulk_load(sR, KV_loc + (static_cast<size_t>(pair) * loc_cap + sg.t0) * 2 * kAtD,
                        static_cast<uint32_t>(groups * 4096), &full[st]);
      }
      __syncwarp();
      if (lane < nch)
        tc::bulk_load(sR + lane * c * 512, KV_slot + (static_cast<size_t>(pair) * k + slot) * c * 2 * kAtD,
                      static_cast<uint32_t>(c * 512), &full[st]);
      lastA[st] = use;
    }
    if (lane == 0) {
      for (int i = 0; i < kAtStages; ++i)
        if (lastA[i] >= 0) tc::mbar_wait(&full[i], lastA[i] & 1, kWaitLimit);
      for (int i = 0; i < 2; ++i)
        if (lastQ[i] >= 0) tc::mbar_wait(&qfull[i], lastQ[i] & 1, kWaitLimit);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 16);
      // S of item i needs its K tile, the head's q and a free S buffer; O of
      // item i needs its P and a free O buffer.  Whichever is ready is issued
      // (polling), so P V never waits for the next item's loads.
      int prev = -1, nq = -1, ns = 0, no = 0;
      bool q_ready = false;
      auto s_ready = [&](int it) -> bool {
        const int item = lo + it, pair = item / nsplit;
        if (pair != prev && !q_ready) {
          if (!tc::mbar_test(&qfull[(nq + 1) & 1], ((nq + 1) >> 1) & 1)) return false;
          q_ready = true;
        }
        return tc::mbar_test(&full[it % kAtStages], (it / kAtStages) & 1) &&
               tc::mbar_test(&sempty[it & 1], ((it >> 1) & 1) ^ 1);
      };
      auto issue_s = [&](int it) {
        const int item = lo + it, pair = item / nsplit;
        if (pair != prev) {
          ++nq;
          prev = pair;
          q_ready = false;
        }
        const int st = it % kAtStages, sb = it & 1;
        tc::fence_after();
        const uint32_t a0 = tc::smem_u32(stages + st * kAtStage);
        const uint32_t b0 = tc::smem_u32(qbuf + (nq & 1) * kAtQBytes);
        // K tiles: core matrices of 8 tokens x 8 dims; dim groups 128 B
        // apart, token groups (records) 4 KB apart.  q: 64-byte swizzle.
#pragma unroll
        for (int kb = 0; kb < kAtD / 32; ++kb)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            tc::mma_bf16(tmem + sb * 16, tc::desc_k_none(a0 + (kb * 2 + ks) * 256, 128, 4096),
                         tc::desc_k_sw64(b0 + kb * (16 * 64) + ks * 32, 512), idesc, (kb | ks) != 0);
        tc::mma_commit(&sfull[sb]);
        const bool last_of_pair = it == nit - 1 || (item + 1) / nsplit != pair;
        if (last_of_pair) tc::mma_commit(&qempty[nq & 1]);
      };
      auto o_ready = [&](int it) -> bool {
        return tc::mbar_test(&pfull[it & 1], (it >> 1) & 1) &&
               tc::mbar_test(&oempty[it & 1], ((it >> 1) & 1) ^ 1);
      };
      auto issue_o = [&](int it) {
        const int st = it % kAtStages, b = it & 1;
        const int item = lo + it, pair = item / nsplit;
        const int nks = (at_item(item - pair * nsplit, i_out, i_sp, n_out, n_sp, n_loc).cnt + 15) >> 4;
        tc::fence_after();
        const uint32_t a0 = tc::smem_u32(stages + st * kAtStage + 2048);
        const uint32_t b0 = tc::smem_u32(pbuf + b * kAtPBytes);
        // V^T: core matrices of 8 dims x 8 tokens; dim groups 128 B apart,
        // token groups (records) 4 KB apart.  P^T: 8 heads x 8 tokens; head
        // groups 128 B apart, token groups 256 B apart.  16 tokens per MMA.
#pragma unroll
        for (int ks = 0; ks < kAtT / 16; ++ks)
          if (ks < nks)
            tc::mma_bf16(tmem + 32 + b * 16, tc::desc_k_none(a0 + ks * 8192, 4096, 128),
                         tc::desc_k_none(b0 + ks * 512, 256, 128), idesc, ks != 0);
        tc::mma_commit(&ofull[b]);
        tc::mma_commit(&empty[st]);
      };
      uint64_t t_last = tc::globaltimer_ns();
      while (no < nit) {
        bool progressed = false;
        if (ns < nit && ns < no + 2 && s_ready(ns)) {
          issue_s(ns++);
          progressed = true;
        }
        if (no < ns && o_ready(no)) {
          issue_o(no++);
          progressed = true;
        }
        if (progressed) {
          t_last = tc::globaltimer_ns();
        } else if (*s_abort || tc::globaltimer_ns() - t_last > kWaitLimit) {
          abort_now();
          break;
        }
      }
      // every MMA issued has completed before TMEM is released
      if (nit > 0) tc::mbar_wait(&ofull[(nit - 1) & 1], ((nit - 1) >> 1) & 1, kWaitLimit);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax, accumulation
    const int ct = tid - 64, quarter = warp & 3;
    const int row = quarter * 32 + lane;          // TMEM lane: token row for S, dimension for O
    const uint32_t tlane = static_cast<uint32_t>(quarter * 32) << 16;
    float m_run[G], l_run[G], acc[G], m_hist[2][G], m_acc[G];
    int cur = -1, seg_first = 0, items_in_pair = 0, pending = -1;
    bool dead = false;
    auto load_cols = [&](uint32_t taddr, float* v) {
      if constexpr (G <= 4) {
        float t4[4];
        tc::tmem_ld4(taddr, t4);
#pragma unroll
        for (int g = 0; g < G; ++g) v[g] = t4[g];
      } else {
        tc::tmem_ld8(taddr, v);
      }
    };
    // fold item j's P V (in TMEM O buffer j & 1) into the running sums
    auto accumulate = [&](int j) {
      if (!dead) {
        bool ok = !*s_abort && tc::mbar_wait(&ofull[j & 1], (j >> 1) & 1, kWaitLimit);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) abort_now();
          dead = true;
        }
      }
      if (dead) return;
      tc::fence_after();
      float o[G];
      load_cols(tmem + tlane + 32 + (j & 1) * 16, o);
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&oempty[j & 1]);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mj = m_hist[j & 1][g];
        const float sc = m_acc[g] == -INFINITY ? 0.f : exp2f(m_acc[g] - mj);
        acc[g] = acc[g] * sc + o[g];
        m_acc[g] = mj;
      }
    };
    auto lo_of = [&](int b) { return static_cast<int>(static_cast<long long>(b) * total / gridDim.x); };
    auto finish_pair = [&](int pair) {
      // this CTA's partial of the head, in the slot of its first item
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float* pp = part + ((static_cast<size_t>(pair) * G + g) * max_splits + seg_first) * (kAtD + 2);
        pp[row] = acc[g];
        if (ct == 0) {
          pp[kAtD] = m_run[g];
          pp[kAtD + 1] = l_run[g];
        }
      }
      __threadfence();
      tc::named_sync(1, kAtSoft);
      if (ct == 0) *s_last = atomicAdd(&ticket[pair], items_in_pair) + items_in_pair == nsplit;
      tc::named_sync(1, kAtSoft);
      if (!*s_last) return;
      __threadfence();
      // CTAs cta_of(x0) .. cta_of(x1 - 1) hold the head's items [x0, x1),
      // each its partial in the slot of its first item of the head.  Every
      // thread loads the (max, sum, value) of all heads for up to U CTAs at
      // once (one round trip) and merges them online.
      const int x0 = pair * nsplit, x1 = x0 + nsplit;
      const int nb = static_cast<int>(gridDim.x);
      auto cta_of = [&](int x) {
        return static_cast<int>((static_cast<long long>(x + 1) * nb - 1) / total);
      };
      const int b0 = cta_of(x0), b1 = cta_of(x1 - 1);
      constexpr int U = G <= 4 ? 4 : 2;
      const size_t pb = static_cast<size_t>(pair) * G * max_splits;
      float M[G], den[G], num[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        M[g] = -INFINITY;
        den[g] = 0.f;
        num[g] = 0.f;
      }
      for (int bb = b0; bb <= b1; bb += U) {
        float mv[U][G], lv[U][G], pv[U][G];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int slot = bb + u <= b1 ? max(lo_of(bb + u), x0) - x0 : -1;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            if (slot >= 0) {
              const float* pp = part + (pb + static_cast<size_t>(g) * max_splits + slot) * (kAtD + 2);
              mv[u][g] = __ldcg(pp + kAtD);
              lv[u][g] = __ldcg(pp + kAtD + 1);
              pv[u][g] = __ldcg(pp + row);
            } else {
              mv[u][g] = -INFINITY;
              lv[u][g] = 0.f;
              pv[u][g] = 0.f;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int g = 0; g < G; ++g) {
            if (mv[u][g] == -INFINITY) continue;
            const float mn = fmaxf(M[g], mv[u][g]);
            const float so = M[g] == -INFINITY ? 0.f : exp2f(M[g] - mn), ss = exp2f(mv[u][g] - mn);
            den[g] = den[g] * so + lv[u][g] * ss;
            num[g] = num[g] * so + pv[u][g] * ss;
            M[g] = mn;
          }
      }
#pragma unroll
      for (int g = 0; g < G; ++g)
        out[(static_cast<size_t>(pair) * G + g) * kAtD + row] = __float2bfloat16_rn(num[g] / den[g]);
      if (ct == 0) ticket[pair] = 0;
      tc::named_sync(1, kAtSoft);
    };
    for (int it = 0; it < nit; ++it) {
      const int item = lo + it, pair = item / nsplit, j = item - pair * nsplit;
      const AtSeg sg = at_item(j, i_out, i_sp, n_out, n_sp, n_loc);
      if (pair != cur) {
        if (cur >= 0) {
          if (pending >= 0) accumulate(pending);
          pending = -1;
          finish_pair(cur);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          m_run[g] = -INFINITY;
          l_run[g] = 0.f;
          acc[g] = 0.f;
          m_acc[g] = -INFINITY;
        }
        cur = pair;
        seg_first = j;
        items_in_pair = 0;
      }
      ++items_in_pair;
      const int sb = it & 1;
      if (!dead) {
        bool ok = !*s_abort && tc::mbar_wait(&sfull[sb], (it >> 1) & 1, kWaitLimit);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) abort_now();
          dead = true;
        }
      }
      float s[8];
      if (!dead) {
        tc::fence_after();
        load_cols(tmem + tlane + sb * 16, s);
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sempty[sb]);
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) s[g] = 0.f;
      }
      const bool valid = row < sg.cnt;
      float* rmax = red + (it & 1) * 64;            // [4][8] maxima, then [4][8] sums at +32
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s[g] = valid ? s[g] * scale_log2 : -INFINITY;
        const uint32_t m = __reduce_max_sync(0xffffffffu, order_key(s[g]));
        if (lane == 0) rmax[quarter * 8 + g] = from_order_key(m);
      }
      tc::named_sync(1, kAtSoft);
      unsigned char* P = pbuf + sb * kAtPBytes;
      float alpha[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mi = rmax[g];
#pragma unroll
        for (int w = 1; w < 4; ++w) mi = fmaxf(mi, rmax[w * 8 + g]);
        const float m_new = fmaxf(m_run[g], mi);
        alpha[g] = m_run[g] == -INFINITY ? 0.f : exp2f(m_run[g] - m_new);
        m_run[g] = m_new;
        m_hist[sb][g] = m_new;
        const float p = valid ? exp2f(s[g] - m_new) : 0.f;
        // P^T[g][row]: token group row/8 (256 B), head group g/8 (128 B), head row g%8 (16 B)
        *reinterpret_cast<bf16*>(P + (row >> 3) * 256 + (g >> 3) * 128 + (g & 7) * 16 + (row & 7) * 2) =
            __float2bfloat16_rn(p);
        const float z = warp_sum(p);
        if (lane == 0) rmax[32 + quarter * 8 + g] = z;
      }
      tc::fence_proxy_async_smem();
      tc::named_sync(1, kAtSoft);
      if (ct == 0 && !dead) tc::mbar_arrive(&pfull[sb]);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float z = rmax[32 + g] + rmax[40 + g] + rmax[48 + g] + rmax[56 + g];
        l_run[g] = l_run[g] * alpha[g] + z;
      }
      if (pending >= 0) accumulate(pending);
      pending = it;
    }
    if (cur >= 0) {
      if (pending >= 0) accumulate(pending);
      finish_pair(cur);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, 64);
}

// ---------------------------------------------------------------- host side
bool attn_tc_supported(const shadowkv_params& p) {
  return p.dtype == SKV_DTYPE_BF16 && p.d == kAtD && p.c % 8 == 0 && kAtT % p.c == 0 &&
         static_cast<long long>(p.b) * p.h_kv <= 1024 && at_smem_bytes() <= 227 * 1024;
}

int attn_tc_splits(const Ctx& c, int n_loc) {
  const int n_out = c.p.o * c.p.c, n_sp = c.p.k * c.p.c;
  return (n_out + kAtT - 1) / kAtT + (n_sp + kAtT - 1) / kAtT + (n_loc + kAtT - 1) / kAtT;
}

template <int G>
static cudaError_t attn_tc_t(Ctx& c, const CUtensorMap& mq, void* out, int n_loc, cudaStream_t st) {
  const int smem = at_smem_bytes();
  auto kern = k_attn_tc<G>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int npairs = c.p.b * c.p.h_kv;
  const int items = npairs * attn_tc_splits(c, n_loc);
  const int grid = std::min(c.nsm, items);
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kAtD));
  // after a launch that also fetches values over the host link the
  // attention's CTAs are not made resident early: they slow the fetch
  return launch_ex(!rebuild_fetches(c), kern, dim3(grid), dim3(kAtThreads), smem, st, mq, static_cast<const bf16*>(c.KV_out),
                    static_cast<const bf16*>(c.KV_slot), static_cast<const int32_t*>(c.sel_slot),
                    static_cast<const bf16*>(c.KV_loc),
                    static_cast<bf16*>(out), c.attn_part, c.attn_count, c.p.o * c.p.c, c.p.k * c.p.c,
                    n_loc, c.loc_cap, c.p.c, c.p.k, npairs, c.max_splits, scale_log2, c.status);
}

cudaError_t launch_attn_tc(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st) {
  if (attn_tc_splits(c, n_loc) > c.max_splits) return cudaErrorInvalidValue;
  CUtensorMap mq;
  {
    const cudaError_t e = q_map_for(c, q, &mq);
    if (e != cudaSuccess) return e;
  }
  switch (c.G) {
    case 1: return attn_tc_t<1>(c, mq, out, n_loc, st);
    case 2: return attn_tc_t<2>(c, mq, out, n_loc, st);
    case 4: return attn_tc_t<4>(c, mq, out, n_loc, st);
    default: return attn_tc_t<8>(c, mq, out, n_loc, st);
  }
}

}  // namespace skv
