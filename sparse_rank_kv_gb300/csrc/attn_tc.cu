// Sparse attention of ShadowKV's decode step (Algorithm 2 step 4) on the
// tensor cores, for bf16 state with d = 128: out = softmax(q K^T / sqrt(d)) V
// over [outliers; RoPE(K_sparse); local window], the G query heads of a KV
// head sharing every K/V row.
//
// Work items are 128-token pieces of one (batch, KV head): its outliers, its
// local window, its cache hits (16 chunks of 8 tokens per item), then its
// missed chunks.  Items are taken from two step-wide counters: phase 0
// (outliers, local window, hits) needs nothing the step's key rebuild or
// value fetch produce, so it runs while they do (this kernel is launched with
// programmatic dependent launch right behind the rebuild); phase 1 (the
// misses) starts after griddepcontrol.wait, each item once its own values
// have arrived.  Keys and values are stored by 8-token
// group in 4 KB records laid out as the tensor core's no-swizzle K-major
// tiles: K ([d/8][token%8][d%8], 2 KB), then V^T ([d/8][d%8][token%8], 2 KB).
//   warp 0     : producer -- per item the keys and values by bulk copies
//                (one per run of adjacent cache-slot records among the item's
//                selected chunks, one for a piece of the outliers or local
//                window) and the head's q (TMA, 16 rows of which the rows past
//                G read as zeros) into a 3-stage ring, with the item's
//                description in the stage; phase-0 item numbers come two at
//                a time.
//   warp 1     : tcgen05.mma.  S = K q^T (M = 128 tokens, N = 16, K = d) into
//                one of two TMEM S buffers; after the softmax warps publish
//                P, O = V^T P^T (M = d, N = 16, K = 16-token steps) into one
//                of four TMEM O buffers (two per softmax group), polling both
//                queues.
//   warps 2..9 : softmax, two groups of four taking alternate items (each
//                with its own S, O and P^T buffers); thread = TMEM lane: for S
//                the token row (scale, mask, head maxima by integer warp
//                reductions, p = 2^(s - m),
//                bf16 P^T into shared memory, head sums), for O the dimension:
//                the item's partial (max, sum, sum p v) per query head goes to
//                the item's slot, and a ticket per head counts finished items
//                (phase-1 items in its upper 16 bits).  Once the producer
//                takes missed chunks, a group publishes each phase-0 item as
//                soon as it is done rather than with later items.
//   warps 10..13: the step's value fetch (Algorithm 2 step 3, V from the host):
//                8-token groups of the missed chunks, taken from a fourth
//                counter in phase-1 item order, read from pinned host memory
//                through its device mapping and written as the V^T half of the
//                chunk's cache-slot record; a count per phase-1 item tells
//                the producer when all of the item's groups are in place.
// When both counters are exhausted a CTA takes heads from a third counter and
// merges each head's item partials: the phase-0 ones as soon as its ticket
// shows all of them, then the phase-1 ones, so that after the last missed
// chunk only its few partials remain to be read.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "rebuild_pipe.cuh"

namespace skv {

constexpr int kAtT = 128;                    // tokens per item
constexpr int kAtD = 128;                    // head dimension handled here
constexpr int kAtStages = 3;
constexpr int kAtFetchWarps = 4;
constexpr int kAtSoftGroups = 2;            // softmax warpgroups, taking alternate items
constexpr int kAtThreads = 64 + 128 * kAtSoftGroups + 32 * kAtFetchWarps;
constexpr int kAtSoft = 128;                 // softmax threads
// O accumulators: two per softmax group, so that an item's P V never waits
// for the group's previous item's partial to be read out of TMEM
constexpr int kAtOBufs = 4;
constexpr int kAtTmemCols = 128;             // S: 2 x 16 columns, O: kAtOBufs x 16 (allocated as a power of 2)
static_assert(32 + 16 * kAtOBufs <= kAtTmemCols, "TMEM columns");
constexpr int kAtRec = kAtT / 8 * 4096;      // 16 group records (K tile | V^T tile)
constexpr int kAtQBytes = 16 * kAtD * 2;     // q: 4 x [16 rows][64 B]
constexpr int kAtStage = kAtRec + kAtQBytes;
constexpr int kAtPBytes = 16 * kAtT * 2;     // P^T: 16 x 128 bf16
constexpr int kAtMisc = 1280;                // barriers, item descriptions, reductions, the second group's lists
constexpr int kAtDone = 44;                  // finished items whose tickets are not yet counted
__host__ __device__ constexpr int at_smem_bytes(int npairs) {
  return 1024 /* alignment slack */ + kAtStages * kAtStage + 2 * kAtPBytes + kAtMisc + (3 * npairs + 2) * 4;
}

// An item: its head, kind (0 outliers, 1 local window, 2 hit chunks, 3 missed
// chunks), first token (0, 1) or first position in the head's slot list (2,
// 3), tokens, and the slot of its partial among the head's items.
struct AtItem {
  int pair, seg, t0, cnt, li;
};

template <int G>
__global__ void __launch_bounds__(kAtThreads, 1)
k_attn_tc(const __grid_constant__ CUtensorMap mapQ, const bf16* __restrict__ KV_out,
          bf16* KV_slot, const int32_t* __restrict__ att_slot,
          const int32_t* __restrict__ hits_in, const bf16* __restrict__ KV_loc,
          bf16* __restrict__ out, float* __restrict__ part, int32_t* __restrict__ ticket,
          int32_t* __restrict__ ctr, int32_t* __restrict__ ctr_next, int n_out, int n_loc,
          int loc_cap, int c, int k, int npairs, int max_splits, float scale_log2,
          const bf16* __restrict__ vcpu, const int32_t* __restrict__ miss_chunk,
          const int32_t* __restrict__ miss_slot, const int32_t* __restrict__ miss_base,
          int32_t* __restrict__ item_done, int s, int n_chunks, const bf16* __restrict__ A,
          const __grid_constant__ CUtensorMap mapBt, const float2* __restrict__ rope_tab, int r, int h_kv,
          int nreb, int rbS, int rbNB, int* __restrict__ status) {
  extern __shared__ unsigned char smem_raw[];
  if (static_cast<int>(blockIdx.x) < nreb) {
    // the first nreb CTAs first rebuild the missed chunks' keys, every
    // nreb-th tile from their own, each tile counted on its phase-1 item (a
    // tile is that item's 128 rows); then they take attention items like
    // the others, so every CTA a phase-1 item waits for is resident (one
    // CTA per SM)
    rebuild_pipe_body<kAtD, true, 8>(smem_raw, static_cast<int>(blockIdx.x), nreb, true, item_done, A, mapBt,
                                     mapBt, nullptr, rope_tab, miss_chunk, miss_slot, miss_base, hits_in,
                                     KV_slot, n_chunks, npairs, h_kv, s, r, c, k, rbS, rbNB, 0, status);
  }
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* stages = smem;                           // [kAtStages][records | q]
  unsigned char* pbuf = stages + kAtStages * kAtStage;    // [2][kAtPBytes]
  unsigned char* misc = pbuf + 2 * kAtPBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(misc);     // [kAtStages]
  uint64_t* empty = full + kAtStages;                     // [kAtStages]
  uint64_t* sfull = empty + kAtStages;                    // [2]
  uint64_t* sempty = sfull + 2;                           // [2]
  uint64_t* pfull = sempty + 2;                           // [2]
  uint64_t* ofull = pfull + 2;                            // [kAtOBufs]
  uint64_t* oempty = ofull + kAtOBufs;                    // [kAtOBufs]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 192);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + 196);
  volatile int* s_end = reinterpret_cast<volatile int*>(misc + 200);    // items of this CTA, once known
  volatile int* s_phase1 = reinterpret_cast<volatile int*>(misc + 212); // the producer takes missed chunks
  int* s_dec_g[2] = {reinterpret_cast<int*>(misc + 216), reinterpret_cast<int*>(misc + 220)};
  // per softmax group: its current merge head, its count and list of
  // finished items whose tickets are not yet counted
  int* s_task_g[2] = {reinterpret_cast<int*>(misc + 204), reinterpret_cast<int*>(misc + 1216)};
  int* s_ndone_g[2] = {reinterpret_cast<int*>(misc + 208), reinterpret_cast<int*>(misc + 1220)};
  int* s_done_g[2] = {reinterpret_cast<int*>(misc + 328), reinterpret_cast<int*>(misc + 1024)};   // [kAtDone]
  int* info = reinterpret_cast<int*>(misc + 256);         // [kAtStages][6]: head (-1: no more), tokens, partial slot, kind
  float* red = reinterpret_cast<float*>(misc + 512);      // [2][4][8] maxima, then sums at +32
  int* s_p0 = reinterpret_cast<int*>(misc + kAtMisc);     // [npairs + 1] phase-0 item prefix
  int* s_p1 = s_p0 + npairs + 1;                          // [npairs + 1] phase-1 item prefix
  int* s_hits = s_p1 + npairs + 1;                        // [npairs]

  const int i_out = (n_out + kAtT - 1) / kAtT, i_loc = (n_loc + kAtT - 1) / kAtT;
  const int cpi = kAtT / c;                               // chunks per item
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  tc::grid_dep_launch();

  if (tid == 0) {
    tc::prefetch_tensormap(&mapQ);
    for (int i = 0; i < kAtStages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sfull[i], 1);
      tc::mbar_init(&sempty[i], kAtSoft / 32);
      tc::mbar_init(&pfull[i], 1);
    }
    for (int i = 0; i < kAtOBufs; ++i) {
      tc::mbar_init(&ofull[i], 1);
      tc::mbar_init(&oempty[i], kAtSoft / 32);
    }
    tc::fence_mbar_init();
    *s_abort = 0;
    *s_end = -1;
    *s_phase1 = 0;
    *s_ndone_g[0] = *s_ndone_g[1] = 0;
    // the next step's counters start at zero
    if (blockIdx.x == 0) ctr_next[0] = ctr_next[1] = ctr_next[2] = ctr_next[3] = 0;
  }
  // with the rebuild in this launch (launched right behind the selection),
  // the selection's results are read only after its grid has completed
  if (nreb > 0) tc::grid_dep_wait();
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kAtTmemCols);
    tc::tmem_relinquish();
  } else if (warp == 0) {
    // item counts per head from its cache hits, as exclusive prefixes (the
    // hit counts of up to 512 heads loaded before any is used)
    int b0 = 0, b1 = 0;
    int hv[16];
    for (int p0 = 0; p0 < npairs; p0 += 32) {
      const int u = (p0 >> 5) & 15;
      if (u == 0) {
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          const int pv = p0 + v * 32 + lane;
          hv[v] = pv < npairs ? hits_in[pv] : 0;
        }
      }
      const int p = p0 + lane;
      int h = 0;
#pragma unroll
      for (int v = 0; v < 16; ++v)
        if (v == u) h = hv[v];
      if (h < 0 || h > k) {
        flag_error(status, DEV_BAD_COUNT);
        h = min(max(h, 0), k);
      }
      const int n0 = p < npairs ? i_out + i_loc + (h + cpi - 1) / cpi : 0;
      const int n1 = p < npairs ? (k - h + cpi - 1) / cpi : 0;
      int x0 = n0, x1 = n1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
        if (lane >= o) {
          x0 += y0;
          x1 += y1;
        }
      }
      if (p < npairs) {
        s_p0[p] = b0 + x0 - n0;
        s_p1[p] = b1 + x1 - n1;
        s_hits[p] = h;
      }
      b0 += __shfl_sync(0xffffffffu, x0, 31);
      b1 += __shfl_sync(0xffffffffu, x1, 31);
    }
    if (lane == 0) {
      s_p0[npairs] = b0;
      s_p1[npairs] = b1;
    }
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
  const int T0 = s_p0[npairs], T1 = s_p1[npairs];
  auto abort_now = [&]() {
    if (!*s_abort) {
      *s_abort = 1;
      flag_error(status, DEV_TIMEOUT);
    }
  };
  // the head whose items [base[p], base[p + 1]) contain x
  auto head_of = [&](const int* base, int x) {
    int a = 0, b = npairs;
    while (b - a > 1) {
      const int m = (a + b) >> 1;
      if (base[m] <= x) a = m;
      else b = m;
    }
    return a;
  };
  auto item_of = [&](int phase, int x) -> AtItem {
    AtItem t;
    if (phase == 0) {
      const int p = head_of(s_p0, x), j = x - s_p0[p];
      t.pair = p;
      t.li = j;
      if (j < i_out) {
        t.seg = 0;
        t.t0 = j * kAtT;
        t.cnt = min(kAtT, n_out - t.t0);
      } else if (j < i_out + i_loc) {
        t.seg = 1;
        t.t0 = (j - i_out) * kAtT;
        t.cnt = min(kAtT, n_loc - t.t0);
      } else {
        t.seg = 2;
        t.t0 = (j - i_out - i_loc) * cpi;
        t.cnt = min(cpi, s_hits[p] - t.t0) * c;
      }
    } else {
      const int p = head_of(s_p1, x), j = x - s_p1[p];
      t.pair = p;
      t.seg = 3;
      t.t0 = s_hits[p] + j * cpi;
      t.cnt = min(cpi, k - t.t0) * c;
      t.li = s_p0[p + 1] - s_p0[p] + j;
    }
    return t;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int lastA[kAtStages];
#pragma unroll
    for (int i = 0; i < kAtStages; ++i) lastA[i] = -1;
    // phase-0 item numbers come two at a time, the next pair requested as
    // the current pair starts, so that no atomic's round trip stalls the
    // loop; in phase 1 (about one item per CTA) the next number is requested
    // only once the current item's copies are issued, so that every CTA has
    // taken its first item before any takes a second
    int phase = 0, x = 0, pcur = 0, pnext = 0, pidx = 0;
    if (lane == 0) {
      pcur = atomicAdd(&ctr[0], 2);
      pnext = atomicAdd(&ctr[0], 2);
      x = pcur;
    }
    for (int it = 0;; ++it) {
      x = __shfl_sync(0xffffffffu, x, 0);
      if (phase == 0 && x >= T0) {
        // the misses' keys and values come from the launch before this one
        // (the number requested ahead is past T0 as well)
        phase = 1;
        tc::grid_dep_wait();
        if (lane == 0) {
          *s_phase1 = 1;
          x = atomicAdd(&ctr[1], 1);
        }
        x = __shfl_sync(0xffffffffu, x, 0);
      }
      const int st = it % kAtStages, use = it / kAtStages;
      const bool done = phase == 1 && x >= T1;
      const AtItem t = done ? AtItem{-1, 0, 0, 0, 0} : item_of(phase, x);
      // cache slots of the item's chunks (lane = chunk), loaded before the wait
      const int nch = t.seg >= 2 ? t.cnt / c : 0;
      const int slot = lane < nch ? att_slot[static_cast<size_t>(t.pair) * k + t.t0 + lane] : 0;
      int xn = 0;
      bool ok = true;
      if (lane == 0) ok = !*s_abort && tc::mbar_wait(&empty[st], (use & 1) ^ 1, kWaitLimit);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) abort_now();
        break;
      }
      int* inf = info + st * 6;
      if (done) {
        // no more items: an empty stage tells the MMA warp (its previous
        // item's copies have landed: the stage was released after them)
        if (lane == 0) {
          inf[0] = -1;
          tc::mbar_arrive(&full[st]);
        }
        lastA[st] = -1;
        break;
      }
      unsigned char* sR = stages + st * kAtStage;
      const int groups = (t.cnt + 7) >> 3;
      if ((groups & 1) && groups < kAtT / 8) {
        // P V runs over whole 16-token steps: the V^T half of the record
        // after an odd count of groups meets zero weights and must be finite
        uint4* pad = reinterpret_cast<uint4*>(sR + groups * 4096 + 2048);
#pragma unroll
        for (int i = 0; i < 2048 / 16 / 32; ++i) pad[i * 32 + lane] = make_uint4(0, 0, 0, 0);
        tc::fence_proxy_async_smem();
        __syncwarp();
      }
      if (t.seg == 3 && vcpu != nullptr) {
        // the item's values come from this launch's fetch warps (and, with
        // the rebuild in this launch, its keys from a rebuild CTA): wait for
        // all of its groups (and its tile), then zero the count for the next
        // step
        bool got = true;
        if (lane == 0) {
          got = tc::wait_count(item_done + x, groups + (nreb > 0 ? 1 : 0), kWaitLimit, s_abort);
          if (got) {
            item_done[x] = 0;
            tc::fence_proxy_async_global();
          }
        }
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          if (lane == 0) abort_now();
          break;
        }
      }
      if (lane == 0) {
        inf[0] = t.pair;
        inf[1] = t.cnt;
        inf[2] = t.li;
        inf[3] = t.seg;
        tc::mbar_expect_tx(&full[st], static_cast<uint32_t>(groups * 4096 + kAtQBytes));
        tc::tma_load_4d(sR + kAtRec, &mapQ, &full[st], 0, 0, 0, t.pair);
        if (t.seg == 0)
          tc::bulk_load(sR, KV_out + (static_cast<size_t>(t.pair) * n_out + t.t0) * 2 * kAtD,
                        static_cast<uint32_t>(groups * 4096), &full[st]);
        else if (t.seg == 1)
          tc::bulk_load(sR, KV_loc + (static_cast<size_t>(t.pair) * loc_cap + t.t0) * 2 * kAtD,
                        static_cast<uint32_t>(groups * 4096), &full[st]);
      }
      __syncwarp();
      {
        // one bulk copy per run of consecutive slots (adjacent records):
        // lane l starts a run unless its slot follows lane l - 1's
        const bool good = lane < nch && slot >= 0 && slot < k;
        const int sprev = __shfl_up_sync(0xffffffffu, slot, 1);
        const bool gprev = __shfl_up_sync(0xffffffffu, good ? 1 : 0, 1) != 0;
        const bool cont = lane > 0 && good && gprev && slot == sprev + 1;
        const unsigned long long cm = __ballot_sync(0xffffffffu, cont);
        if (lane < nch && !good) flag_error(status, DEV_BAD_SLOT);
        if (good && !cont) {
          const int len = __ffsll(~(cm >> (lane + 1)));
          tc::bulk_load(sR + lane * c * 512, KV_slot + (static_cast<size_t>(t.pair) * k + slot) * c * 2 * kAtD,
                        static_cast<uint32_t>(len * c * 512), &full[st]);
        }
      }
      lastA[st] = use;
      if (phase == 1) {
        if (lane == 0) xn = atomicAdd(&ctr[1], 1);
        x = xn;
      } else if (pidx == 0) {
        pidx = 1;
        x = pcur + 1;
      } else {
        pidx = 0;
        pcur = pnext;
        if (lane == 0) pnext = atomicAdd(&ctr[0], 2);
        x = pcur;
      }
    }
    // no copy may still be landing in this CTA's shared memory at exit
    if (lane == 0)
      for (int i = 0; i < kAtStages; ++i)
        if (lastA[i] >= 0 && !tc::mbar_wait(&full[i], lastA[i] & 1, kWaitLimit)) abort_now();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 16);
      int ns = 0, no = 0, nit = 0x7fffffff;
      uint64_t t_last = tc::globaltimer_ns();
      while (no < nit) {
        bool progressed = false;
        if (ns < nit && ns < no + 2) {
          const int st = ns % kAtStages, sb = ns & 1;
          if (tc::mbar_test(&full[st], (ns / kAtStages) & 1) &&
              tc::mbar_test(&sempty[sb], ((ns >> 1) & 1) ^ 1)) {
            tc::fence_after();
            if (info[st * 6] < 0) {
              // the producer has no more items: tell the softmax group of
              // index ns, then the group of index ns + 1, once it has read
              // the other buffer's S of index ns - 1 (the same condition as
              // for issuing S of index ns + 1; an earlier arrival would end
              // that phase twice)
              nit = ns;
              *s_end = ns;
              tc::mbar_arrive(&sfull[sb]);
              if (tc::mbar_wait(&sempty[sb ^ 1], (((ns + 1) >> 1) & 1) ^ 1, kWaitLimit)) tc::mbar_arrive(&sfull[sb ^ 1]);
              else abort_now();
            } else {
              const uint32_t a0 = tc::smem_u32(stages + st * kAtStage);
              const uint32_t b0 = a0 + kAtRec;
              // K tiles: core matrices of 8 tokens x 8 dims; dim groups 128 B
              // apart, token groups (records) 4 KB apart.  q: core matrices of
              // 8 rows x 8 dims; dim groups 256 B apart, row groups 128 B apart.
#pragma unroll
              for (int kk = 0; kk < kAtD / 16; ++kk)
                tc::mma_bf16(tmem + sb * 16, tc::desc_k_none(a0 + kk * 256, 128, 4096),
                             tc::desc_k_none(b0 + kk * 512, 256, 128), idesc, kk != 0);
              tc::mma_commit(&sfull[sb]);
              ++ns;
            }
            progressed = true;
          }
        }
        if (no < ns && tc::mbar_test(&pfull[no & 1], (no >> 1) & 1) &&
            tc::mbar_test(&oempty[no % kAtOBufs], ((no / kAtOBufs) & 1) ^ 1)) {
          const int st = no % kAtStages, b = no % kAtOBufs;
          const int nks = (info[st * 6 + 1] + 15) >> 4;
          tc::fence_after();
          const uint32_t a0 = tc::smem_u32(stages + st * kAtStage + 2048);
          const uint32_t b0 = tc::smem_u32(pbuf + (no & 1) * kAtPBytes);   // the item's P^T buffer
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
          ++no;
          progressed = true;
        }
        if (progressed) {
          t_last = tc::globaltimer_ns();
        } else if (*s_abort || tc::globaltimer_ns() - t_last > kWaitLimit) {
          abort_now();
          *s_end = ns;
          tc::mbar_arrive(&sfull[0]);
          tc::mbar_arrive(&sfull[1]);
          break;
        }
      }
      // every MMA issued has completed before TMEM is released
      if (no > 0) tc::mbar_wait(&ofull[(no - 1) % kAtOBufs], ((no - 1) / kAtOBufs) & 1, kWaitLimit);
    }
    __syncwarp();
  } else if (warp < 2 + 4 * kAtSoftGroups) {
    // ------------------------------------------------------------ softmax
    // group gs takes the items of its parity: their S and O buffers, P^T
    // buffer and reduction scratch are its own; it meets at named barrier bar
    const int gs = (warp - 2) >> 2, bar = gs ? 3 : 1;
    int* s_done = s_done_g[gs];
    int* s_ndone = s_ndone_g[gs];
    int* s_task = s_task_g[gs];
    int* s_dec = s_dec_g[gs];
    const int ct = tid - 64 - 128 * gs, quarter = warp & 3;
    const int row = quarter * 32 + lane;          // TMEM lane: token row for S, dimension for O
    const uint32_t tlane = static_cast<uint32_t>(quarter * 32) << 16;
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
    bool dead = false;
    // the pending item: its O buffer holds sum p v once ofull completes
    int pj = -1, ppair = 0, pli = 0, pseg = 0;
    float pm[G], pl[G];
    auto finish = [&]() {
      if (!dead) {
        bool ok = !*s_abort && tc::mbar_wait(&ofull[pj % kAtOBufs], (pj / kAtOBufs) & 1, kWaitLimit);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) abort_now();
          dead = true;
        }
      }
      if (dead) return;
      tc::fence_after();
      float o[8];
      load_cols(tmem + tlane + 32 + (pj % kAtOBufs) * 16, o);
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&oempty[pj % kAtOBufs]);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float* pp = part + ((static_cast<size_t>(ppair) * G + g) * max_splits + pli) * (kAtD + 2);
        pp[row] = o[g];
        if (ct == 0) {
          pp[kAtD] = pm[g];
          pp[kAtD + 1] = pl[g];
        }
      }
      // the head's ticket counts the item once its partial is visible (a
      // phase-1 item in the upper 16 bits); the counts are published
      // together, after one fence
      if (ct == 0) s_done[(*s_ndone)++] = ppair | (pseg == 3 ? (1 << 30) : 0);
    };
    auto publish = [&]() {
      tc::named_sync(bar, kAtSoft);
      if (ct == 0 && *s_ndone > 0) {
        tc::fence_acq_rel_gpu();
        for (int i = 0; i < *s_ndone; ++i)
          atomicAdd(&ticket[s_done[i] & 0x3fffffff], (s_done[i] >> 30) ? (1 << 16) : 1);
        *s_ndone = 0;
      }
      tc::named_sync(bar, kAtSoft);
    };
    for (int it = gs;; it += kAtSoftGroups) {
      const int sb = it & 1, st = it % kAtStages;
      // once the producer takes missed chunks (whose items wait for the
      // host link), the phase-0 item this group holds is finished and
      // published while the group waits for its next item, so that the
      // heads' merges can fold their phase-0 partials in early (one
      // decision for the group)
      if (pj >= 0 && !dead) {
        if (ct == 0) {
          // the next item's S or the producer's move to the missed chunks,
          // whichever comes first (a missed wait is reported below)
          int d = 0;
          const uint64_t t0 = tc::globaltimer_ns();
          while (!tc::mbar_test(&sfull[sb], (it >> 1) & 1)) {
            if (*s_phase1) {
              d = 1;
              break;
            }
            if (*s_abort || tc::globaltimer_ns() - t0 > kWaitLimit) break;
            __nanosleep(64);   // leaves the SM's issue slots to the copy, MMA and fetch warps
          }
          *s_dec = d;
        }
        tc::named_sync(bar, kAtSoft);
        if (*s_dec) {
          finish();
          pj = -1;
          publish();
        }
      }
      if (!dead) {
        bool ok = !*s_abort && tc::mbar_wait(&sfull[sb], (it >> 1) & 1, kWaitLimit);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) abort_now();
          dead = true;
        }
      }
      if (dead || (*s_end >= 0 && it >= *s_end)) break;
      // the item's description (its stage is complete and not yet reused)
      if (!tc::mbar_wait(&full[st], (it / kAtStages) & 1, kWaitLimit) && lane == 0) abort_now();
      const int pair = info[st * 6], cnt = info[st * 6 + 1], li = info[st * 6 + 2], seg = info[st * 6 + 3];
      float s[8];
      tc::fence_after();
      load_cols(tmem + tlane + sb * 16, s);
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sempty[sb]);
      const bool valid = row < cnt;
      float* rmax = red + (it & 1) * 64;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s[g] = valid ? s[g] * scale_log2 : -INFINITY;
        const uint32_t m = __reduce_max_sync(0xffffffffu, order_key(s[g]));
        if (lane == 0) rmax[quarter * 8 + g] = from_order_key(m);
      }
      tc::named_sync(bar, kAtSoft);
      unsigned char* P = pbuf + sb * kAtPBytes;
      float mi[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        mi[g] = rmax[g];
#pragma unroll
        for (int w = 1; w < 4; ++w) mi[g] = fmaxf(mi[g], rmax[w * 8 + g]);
        const float p = valid ? exp2f(s[g] - mi[g]) : 0.f;
        // P^T[g][row]: token group row/8 (256 B), head group g/8 (128 B), head row g%8 (16 B)
        *reinterpret_cast<bf16*>(P + (row >> 3) * 256 + (g >> 3) * 128 + (g & 7) * 16 + (row & 7) * 2) =
            __float2bfloat16_rn(p);
        const float z = warp_sum(p);
        if (lane == 0) rmax[32 + quarter * 8 + g] = z;
      }
      tc::fence_proxy_async_smem();
      tc::named_sync(bar, kAtSoft);
      if (ct == 0) tc::mbar_arrive(&pfull[sb]);
      float li_sum[G];
#pragma unroll
      for (int g = 0; g < G; ++g) li_sum[g] = rmax[32 + g] + rmax[40 + g] + rmax[48 + g] + rmax[56 + g];
      if (pj >= 0) {
        if (*s_ndone == kAtDone) publish();
        finish();
      }
      pj = it;
      ppair = pair;
      pli = li;
      pseg = seg;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        pm[g] = mi[g];
        pl[g] = li_sum[g];
      }
      if (seg == 3) {
        // a missed-chunk item (the step's tail): its partial and its head's
        // ticket at once, without waiting for the next item
        finish();
        pj = -1;
        publish();
      }
    }
    if (pj >= 0 && !dead) {
      if (*s_ndone == kAtDone) publish();
      finish();
    }
    if (!dead) publish();

    // ------------------------------------------------------------ combine
    // heads from the third counter.  A head's ticket counts its published
    // phase-0 items (outliers, local window, cache hits) in the low 16 bits
    // and its phase-1 items (missed chunks) above them.  The phase-0
    // partials are folded in once all of them are published, the phase-1
    // partials once those are (all in one stage when the whole count is
    // there at the first look): per query head a running max M, sum of
    // 2^(m - M) l and, per output row, sum of 2^(m - M) pv, divided at the
    // end.  Scratch: [G][wcap] maxima, turned into 2^(m - M), then [G][wcap]
    // sums (P^T is no longer used); the group's reduction scratch holds M,
    // the sum and the factor that rescales the earlier terms, per head.
    float* w = reinterpret_cast<float*>(pbuf + gs * kAtPBytes);
    const int wcap = kAtPBytes / 8 / G;
    float* lsum = w + G * wcap;
    float* mst = red + gs * 64;
    while (!dead) {
      if (ct == 0) *s_task = atomicAdd(&ctr[2], 1);
      tc::named_sync(bar, kAtSoft);
      const int pair = *s_task;
      tc::named_sync(bar, kAtSoft);
      if (pair >= npairs) break;
      const int n0 = s_p0[pair + 1] - s_p0[pair], n1 = s_p1[pair + 1] - s_p1[pair];
      const size_t pb = static_cast<size_t>(pair) * G * max_splits;
      const float* pr = part + pb * (kAtD + 2) + row;
      if (ct < G) {
        mst[ct] = -INFINITY;
        mst[G + ct] = 0.f;
      }
      // R items' partial rows per round; a stage's first round is loaded
      // together with its items' (max, sum), before the weights are known
      constexpr int R = 64 / G;
      float v[R][G], num[G];
#pragma unroll
      for (int g = 0; g < G; ++g) num[g] = 0.f;
      bool ok = n0 + n1 <= wcap;
      const int full = n0 + (n1 << 16);
      int split = n0;   // items folded in the first stage
      for (int stage = 0; stage < 2; ++stage) {
        if (stage == 1 && split == n0 + n1) break;
        if (ct == 0) {
          int seen = 0;
          ok = ok && tc::wait_count(ticket + pair, stage ? full : n0, kWaitLimit, s_abort, stage ? -1 : 0xffff,
                                    &seen);
          if (!ok) abort_now();
          if (stage == 0) *s_dec = seen == full ? n0 + n1 : n0;
        }
        tc::named_sync(bar, kAtSoft);
        if (*s_abort) break;
        if (stage == 0) split = *s_dec;
        const int i0 = stage ? split : 0, ni = stage ? n0 + n1 - split : split;
        if (ni == 0) continue;
        auto load_round = [&](int j0) {
#pragma unroll
          for (int u = 0; u < R; ++u)
#pragma unroll
            for (int g = 0; g < G; ++g)
              v[u][g] = j0 + u < ni
                            ? __ldcg(pr + (static_cast<size_t>(g) * max_splits + i0 + j0 + u) * (kAtD + 2))
                            : 0.f;
        };
        load_round(0);
        for (int e = ct; e < G * ni; e += kAtSoft) {
          const int g = e / ni, i = e - g * ni;
          const float* pp = part + (pb + static_cast<size_t>(g) * max_splits + i0 + i) * (kAtD + 2) + kAtD;
          w[g * wcap + i] = __ldcg(pp);
          lsum[g * wcap + i] = __ldcg(pp + 1);
        }
        tc::named_sync(bar, kAtSoft);
        if (((warp - 2) & 3) < G) {
          // warp g: the new M, the factor for the earlier terms, the sum,
          // and the stage's weights 2^(m - M)
          for (int gg = (warp - 2) & 3; gg < G; gg += 4) {
            float M = -INFINITY;
            for (int i = lane; i < ni; i += 32) M = fmaxf(M, w[gg * wcap + i]);
            const float Mo = mst[gg];
            M = fmaxf(warp_max(M), Mo);
            float den = 0.f;
            for (int i = lane; i < ni; i += 32) {
              const float e = exp2f(w[gg * wcap + i] - M);
              den += e * lsum[gg * wcap + i];
              w[gg * wcap + i] = e;
            }
            den = warp_sum(den);
            __syncwarp();
            if (lane == 0) {
              const float sc = Mo == -INFINITY ? 0.f : exp2f(Mo - M);
              mst[2 * G + gg] = sc;
              mst[G + gg] = mst[G + gg] * sc + den;
              mst[gg] = M;
            }
          }
        }
        tc::named_sync(bar, kAtSoft);
#pragma unroll
        for (int g = 0; g < G; ++g) num[g] *= mst[2 * G + g];
        for (int j0 = 0; j0 < ni; j0 += R) {
          if (j0 > 0) load_round(j0);
#pragma unroll
          for (int u = 0; u < R; ++u)
#pragma unroll
            for (int g = 0; g < G; ++g)
              if (j0 + u < ni) num[g] = fmaf(w[g * wcap + j0 + u], v[u][g], num[g]);
        }
        // the scratch is rewritten by the next stage
        tc::named_sync(bar, kAtSoft);
      }
      if (*s_abort) break;
#pragma unroll
      for (int g = 0; g < G; ++g)
        out[(static_cast<size_t>(pair) * G + g) * kAtD + row] = __float2bfloat16_rn(num[g] / mst[G + g]);
      if (ct == 0) ticket[pair] = 0;
      tc::named_sync(bar, kAtSoft);
    }
  } else if (vcpu != nullptr) {
    // ------------------------------------------------------------ value fetch
    // units: 16 groups of 8 tokens per phase-1 item (a full item holds 128
    // tokens), numbered item-major so that items complete in the order the
    // producers take them; a half-warp moves one group (2 KB), two per round
    // with both read before either is written; a warp takes 4 units at a time
    const int half = lane >> 4, q = lane & 15;
    const int gpc = c >> 3;   // groups per chunk
    const int units = T1 * (kAtT / 8);
    for (;;) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&ctr[3], 4);
      base = __shfl_sync(0xffffffffu, base, 0);
      if (base >= units) break;
      uint4 in[2][8];
      uint4* dst[2] = {nullptr, nullptr};
      int xs[2] = {-1, -1};
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int U = base + 2 * half + u;
        if (U >= units) continue;
        const int x = U / (kAtT / 8), gi = U - x * (kAtT / 8);
        const int p = head_of(s_p1, x), j = x - s_p1[p];
        const int nch = min(cpi, k - s_hits[p] - j * cpi);
        if (gi >= nch * gpc) continue;
        // counted even when its entry is bad, so that no producer waits for it
        xs[u] = x;
        const int l = gi / gpc, gs = gi - l * gpc;
        const int m = miss_base[p] + j * cpi + l;
        int chunk = -1, slot = -1;
        if (m >= 0 && m < npairs * k) {
          chunk = miss_chunk[m] - p * n_chunks;
          slot = miss_slot[m] - p * k;
        }
        if (chunk < 0 || chunk >= n_chunks || slot < 0 || slot >= k) {
          if (q == 0) flag_error(status, DEV_BAD_SLOT);
          continue;
        }
        const uint4* src = reinterpret_cast<const uint4*>(
            vcpu + (static_cast<size_t>(p) * s + static_cast<size_t>(chunk) * c + gs * 8) * kAtD);
        dst[u] = reinterpret_cast<uint4*>(KV_slot + ((static_cast<size_t>(p) * k + slot) * c + gs * 8) * 2 * kAtD +
                                          kAtD * 8);
#pragma unroll
        for (int t = 0; t < 8; ++t) in[u][t] = src[t * 16 + q];
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (dst[u] == nullptr) continue;
        uint4 outv[8];
        transpose8x8(in[u], outv);
#pragma unroll
        for (int r = 0; r < 8; ++r) dst[u][q * 8 + r] = outv[r];
      }
      // the groups' values are visible at device scope (and ordered before
      // the consuming CTA's bulk copies) before their items' counts move
      tc::fence_proxy_async_global();
      tc::fence_acq_rel_gpu();
      __syncwarp();
      if (q == 0)
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if (xs[u] >= 0) atomicAdd(&item_done[xs[u]], 1);
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kAtTmemCols);
}

// ---------------------------------------------------------------- host side
// The queries as a 4D view {8 dims, G rows, d/8 dim groups, b*h_kv} (strides
// 2 B, d*2 B, 16 B, G*d*2 B), read in boxes of 8 x 16 x 16 x 1: a head's q
// lands as [d/8][16 rows][8 dims], the rows past G zero-filled.
cudaError_t qa_map_for(Ctx& c, const void* q, CUtensorMap* map) {
  if (!c.qa_map || q != c.qa_enc) {
    c.qa_map = false;
    if (reinterpret_cast<uintptr_t>(q) % 16) return cudaErrorMisalignedAddress;
    void* fnp = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault, &qr) !=
            cudaSuccess || fnp == nullptr)
      return cudaErrorNotSupported;
    using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    const cuuint64_t dims[4] = {8, static_cast<cuuint64_t>(c.G), static_cast<cuuint64_t>(kAtD / 8),
                                static_cast<cuuint64_t>(c.p.b) * c.p.h_kv};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kAtD) * 2, 16,
                                   static_cast<cuuint64_t>(kAtD) * 2 * c.G};
    const cuuint32_t box[4] = {8, 16, kAtD / 8, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = reinterpret_cast<EncodeFn>(fnp)(
        &c.mapQa, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    c.qa_enc = q;
    c.qa_map = true;
  }
  *map = c.mapQa;
  return cudaSuccess;
}

// Items per head at most: outliers, local window, the hit chunks and the
// missed chunks (whose split may add one item).
static int at_items_max(const shadowkv_params& p, int n_loc) {
  const int cpi = kAtT / p.c;
  return (p.o * p.c + kAtT - 1) / kAtT + (n_loc + kAtT - 1) / kAtT + (p.k + cpi - 1) / cpi + 1;
}

bool attn_tc_supported(const shadowkv_params& p) {
  const int npairs_max = 1024;
  const int G = p.h_q / p.h_kv;
  const int items = at_items_max(p, p.w + p.max_new);
  return p.dtype == SKV_DTYPE_BF16 && p.d == kAtD && p.c % 8 == 0 && kAtT % p.c == 0 &&
         static_cast<long long>(p.b) * p.h_kv <= npairs_max && at_smem_bytes(npairs_max) <= 227 * 1024 &&
         G >= 1 && items * G <= kAtPBytes / 8;
}

template <int G>
static cudaError_t attn_tc_t(Ctx& c, const CUtensorMap& mq, void* out, int n_loc, cudaStream_t st) {
  const int npairs = c.p.b * c.p.h_kv;
  const int smem = at_smem_bytes(npairs);
  auto kern = k_attn_tc<G>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kAtD));
  const int par = static_cast<int>(c.t & 1);
  // each launch clears the other parity's counters for the next step; after
  // a step on another attention path this parity's are cleared here
  if (c.at_last != c.t - 1) {
    e = cudaMemsetAsync(c.at_ctr + 4 * par, 0, 4 * sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
  }
  c.at_last = c.t;
  // launched behind the key rebuild: phase 0 overlaps it and this launch's
  // own value fetch
  const bool fetch = attn_fetches(c);
  int rbS = 0, rbNB = 0;
  const int nreb = attn_rebuilds(c, &rbS, &rbNB) ? std::min(kRebuildSMsRec, c.nsm / 4) : 0;
  return launch_pdl(kern, dim3(c.nsm), dim3(kAtThreads), static_cast<size_t>(smem), st, mq,
                    static_cast<const bf16*>(c.KV_out), static_cast<bf16*>(c.KV_slot),
                    static_cast<const int32_t*>(c.att_slot), static_cast<const int32_t*>(c.hits),
                    static_cast<const bf16*>(c.KV_loc), static_cast<bf16*>(out), c.attn_part, c.attn_count,
                    c.at_ctr + 4 * par, c.at_ctr + 4 * (par ^ 1), c.p.o * c.p.c, n_loc, c.loc_cap, c.p.c,
                    c.p.k, npairs, c.max_splits, scale_log2,
                    static_cast<const bf16*>(fetch ? c.v_cpu_dev : nullptr),
                    static_cast<const int32_t*>(c.miss_chunk), static_cast<const int32_t*>(c.miss_slot),
                    static_cast<const int32_t*>(c.miss_base), c.item_done, c.p.s, c.n,
                    static_cast<const bf16*>(c.A), c.mapBt, static_cast<const float2*>(c.rope_tab), c.p.r,
                    c.p.h_kv, nreb, rbS, rbNB, c.status);
}

bool attn_fetches(const Ctx& c) {
  return c.kv_rec && !c.force_simt && !c.split_set && c.v_cpu_dev != nullptr && c.item_done != nullptr;
}

bool attn_rebuilds(const Ctx& c, int* S, int* NB) {
  if (!c.rebuild_in_attn || !attn_fetches(c) || !c.tc_rebuild || !c.a_tiled || c.p.d != kAtD) return false;
  // the rebuild's pipeline (A stages, B slots, the head tables) in the
  // attention's shared memory
  const int npairs = c.p.b * c.p.h_kv;
  const int room = at_smem_bytes(npairs) - (3 * npairs + 1) * 4;
  const int cand[4][2] = {{2, 2}, {2, 1}, {1, 2}, {1, 1}};
  for (auto& x : cand)
    if (pipe_smem(c.p.r, kAtD, x[0], x[1], 0) <= room) {
      if (S) *S = x[0];
      if (NB) *NB = x[1];
      return true;
    }
  return false;
}

cudaError_t launch_attn_tc(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st) {
  if (at_items_max(c.p, n_loc) > c.max_splits) return cudaErrorInvalidValue;
  CUtensorMap mq;
  {
    const cudaError_t e = qa_map_for(c, q, &mq);
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
