// Pipelined sparse attention of ShadowKV's decode step (Algorithm 2 step 4)
// for bf16 state: out = softmax(q K^T / sqrt(d)) V over the token list
// [outliers; RoPE(K_sparse); local window], the G query heads of a KV head
// sharing every K/V row.
//
// Work items are 64-token pieces of one segment (outliers, rebuilt chunks or
// local window) of one (batch, KV head); each of the persistent CTAs (two per
// SM) owns a contiguous range of items.
//   warp 0     : producer -- per item, the K rows by TMA (box 64 columns x 64
//                rows, 128-byte swizzle) and the V rows by bulk copies (one
//                per selected chunk from its cache slot, or one contiguous
//                copy for the outliers and the local window) into a
//                2- or 3-stage ring
//   warps 1..8 : warp w owns rows 8w .. 8w+7 of every item: logits with four
//                lanes per row (a quarter of d each; the swizzle keeps the
//                reads free of bank conflicts), its own running max and sum
//                over the CTA's consecutive items of the same head, and P V
//                over its rows with d/32 dimensions per lane, accumulators
//                in registers -- no block-wide barrier per item.  When the
//                head changes (or the range ends) a shared-memory tree
//                merges the eight warp states and the CTA writes one partial
//                (max, sum, sum p v) per query head, in the slot of its first
//                item of that head.  The CTA that
//                completes a head's last items (atomic count) combines the
//                partials in slot order (the slots follow from the fixed item
//                ranges), so the result does not depend on which CTA
//                finishes last.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace skv {

constexpr int kApS = 64;            // tokens per work item
constexpr int kApCompute = 256;     // compute threads (warps 1..8)
constexpr int kApThreads = 32 + kApCompute;
constexpr int kApMaxSlots = 64;     // partials of one head (CTA ranges meeting it)

__host__ __device__ constexpr int ap_stage_bytes(int D) { return 2 * kApS * D * 2; }   // K + V
__host__ __device__ constexpr int ap_fixed_bytes(int G, int D) {
  return 1024 /* barriers, slot list */ + G * D * 4 /* q */ + (kApCompute / 32) * G * 8 * 4 /* p per warp */ +
         (kApCompute / 64) * G * (D + 2) * 4 /* warp-state tree, combine scratch */;
}
__host__ __device__ constexpr int ap_smem_bytes(int G, int D, int NST) {
  return 1024 /* alignment slack */ + NST * ap_stage_bytes(D) + ap_fixed_bytes(G, D);
}
// stages that keep two CTAs per SM (<= 113 KB each)
__host__ __device__ constexpr int ap_stages(int G, int D) {
  return ap_smem_bytes(G, D, 3) <= 113 * 1024 ? 3 : 2;
}

struct ApSeg {
  int seg, t0, cnt;   // segment 0 outliers / 1 rebuilt chunks / 2 local; start within it; tokens
};
__device__ __forceinline__ ApSeg ap_item(int j, int i_out, int i_sp, int n_out, int n_sp, int n_loc) {
  if (j < i_out) return {0, j * kApS, min(kApS, n_out - j * kApS)};
  j -= i_out;
  if (j < i_sp) return {1, j * kApS, min(kApS, n_sp - j * kApS)};
  j -= i_sp;
  return {2, j * kApS, min(kApS, n_loc - j * kApS)};
}

template <int D, int G, int NST>
__global__ void __launch_bounds__(kApThreads, 2)
k_attn_pipe(const __grid_constant__ CUtensorMap mapKo, const __grid_constant__ CUtensorMap mapKs,
            const __grid_constant__ CUtensorMap mapKl, const bf16* __restrict__ V_out,
            const bf16* __restrict__ slot_V, const int32_t* __restrict__ sel_slot,
            const bf16* __restrict__ V_loc, const bf16* __restrict__ q, bf16* __restrict__ out,
            float* __restrict__ part, int32_t* __restrict__ ticket, int n_out, int n_sp, int n_loc,
            int loc_cap, int c, int k, int npairs, int max_splits, float scale_log2,
            int* __restrict__ status) {
  constexpr int NCH = D / 8;           // 16-byte chunks per row
  constexpr int NCW = kApCompute / 32; // compute warps
  constexpr int DPL = D / 32;          // P V dimensions per lane
  constexpr int SB = ap_stage_bytes(D);
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* stages = smem;                            // [stage][K (D/64 x 64 x 128 B) | V (64 x D)]
  unsigned char* fixed = smem + NST * SB;
  uint64_t* full = reinterpret_cast<uint64_t*>(fixed);     // [NST]
  uint64_t* empty = full + NST;                      // [NST]
  volatile int* s_abort = reinterpret_cast<volatile int*>(fixed + 128);
  int* s_last = reinterpret_cast<int*>(fixed + 132);
  int* s_nslot = reinterpret_cast<int*>(fixed + 136);
  int* s_slots = reinterpret_cast<int*>(fixed + 256);      // [kApMaxSlots]
  float* qs = reinterpret_cast<float*>(fixed + 1024);      // [G][D], scaled to log2 units
  float* ps = qs + G * D;                                  // [NCW][G][8]
  float* tb = ps + NCW * G * 8;                            // [NCW/2][G][D+2]

  const int i_out = (n_out + kApS - 1) / kApS, i_sp = (n_sp + kApS - 1) / kApS,
            i_loc = (n_loc + kApS - 1) / kApS;
  const int nsplit = i_out + i_sp + i_loc;
  const int total = npairs * nsplit;
  const int lo = static_cast<int>(static_cast<long long>(blockIdx.x) * total / gridDim.x);
  const int hi = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * total / gridDim.x);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    tc::prefetch_tensormap(&mapKs);
    if (n_out > 0) tc::prefetch_tensormap(&mapKo);
    if (n_loc > 0) tc::prefetch_tensormap(&mapKl);
    for (int i = 0; i < NST; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], kApCompute / 32);
    }
    tc::fence_mbar_init();
    *s_abort = 0;
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int last_use[NST];
#pragma unroll
    for (int i = 0; i < NST; ++i) last_use[i] = -1;
    for (int it = 0; it < hi - lo; ++it) {
      const int item = lo + it, pair = item / nsplit, j = item - pair * nsplit;
      const ApSeg sg = ap_item(j, i_out, i_sp, n_out, n_sp, n_loc);
      const int st = it % NST, use = it / NST;
      // cache slots of the item's chunks (lane = chunk), loaded before the wait
      const int ch0 = sg.t0 / c, nch = sg.seg == 1 ? sg.cnt / c : 0;
      const int slot = lane < nch ? sel_slot[static_cast<size_t>(pair) * k + ch0 + lane] : 0;
      bool ok = true;
      if (lane == 0) ok = *s_abort == 0 && tc::mbar_wait(&empty[st], (use & 1) ^ 1, kWaitLimit);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0 && *s_abort == 0) {
          *s_abort = 1;
          flag_error(status, DEV_TIMEOUT);
        }
        break;
      }
      unsigned char* sK = stages + st * SB;
      unsigned char* sV = sK + kApS * D * 2;
      if (lane == 0) {
        tc::mbar_expect_tx(&full[st], static_cast<uint32_t>(kApS * D * 2 + sg.cnt * D * 2));
        const CUtensorMap* m = sg.seg == 0 ? &mapKo : sg.seg == 1 ? &mapKs : &mapKl;
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tc::tma_load_3d(sK + cb * (kApS * 128), m, &full[st], cb * 64, sg.t0, pair);
        if (sg.seg == 0)
          tc::bulk_load(sV, V_out + (static_cast<size_t>(pair) * n_out + sg.t0) * D,
                        static_cast<uint32_t>(sg.cnt * D * 2), &full[st]);
        else if (sg.seg == 2)
          tc::bulk_load(sV, V_loc + (static_cast<size_t>(pair) * loc_cap + sg.t0) * D,
                        static_cast<uint32_t>(sg.cnt * D * 2), &full[st]);
      }
      __syncwarp();
      // one bulk copy per selected chunk, from its cache slot (<= 64 / 8 chunks)
      if (lane < nch)
        tc::bulk_load(sV + lane * c * D * 2, slot_V + (static_cast<size_t>(pair) * k + slot) * c * D,
                      static_cast<uint32_t>(c * D * 2), &full[st]);
      last_use[st] = use;
    }
    // every copy issued has landed before the CTA may exit
    if (lane == 0)
      for (int i = 0; i < NST; ++i)
        if (last_use[i] >= 0) tc::mbar_wait(&full[i], last_use[i] & 1, kWaitLimit);
  } else {
    // ------------------------------------------------------------ compute
    const int ct = tid - 32, cw = ct >> 5;      // compute thread, warp 0..NCW-1
    const int rsub = lane & 7, qsel = lane >> 3, row = cw * 8 + rsub;
    float* pw = ps + cw * (G * 8);              // this warp's p [G][8 rows]
    float m_run[G], l_run[G], acc[G][DPL];
    int cur = -1, seg_first = 0, items_in_pair = 0;
    bool dead = false;                          // a wait gave up: skip the work, keep the barriers
    auto flush = [&](int pair) {
      // tree over the warp states: warps [h, 2h) publish, warps [0, h) merge
      for (int h = NCW / 2; h >= 1; h >>= 1) {
        if (cw >= h && cw < 2 * h) {
          float* bsrc = tb + (cw - h) * (G * (D + 2));
#pragma unroll
          for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int e = 0; e < DPL; ++e) bsrc[g * (D + 2) + lane * DPL + e] = acc[g][e];
            if (lane == 0) {
              bsrc[g * (D + 2) + D] = m_run[g];
              bsrc[g * (D + 2) + D + 1] = l_run[g];
            }
          }
        }
        tc::named_sync(1, kApCompute);
        if (cw < h) {
          const float* bsrc = tb + cw * (G * (D + 2));
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float mo = bsrc[g * (D + 2) + D], lo_ = bsrc[g * (D + 2) + D + 1];
            const float M = fmaxf(m_run[g], mo);
            const float sa = M == -INFINITY ? 0.f : exp2f(m_run[g] - M);
            const float sb = M == -INFINITY ? 0.f : exp2f(mo - M);
            l_run[g] = l_run[g] * sa + lo_ * sb;
#pragma unroll
            for (int e = 0; e < DPL; ++e)
              acc[g][e] = acc[g][e] * sa + bsrc[g * (D + 2) + lane * DPL + e] * sb;
            m_run[g] = M;
          }
        }
        tc::named_sync(1, kApCompute);
      }
      if (cw == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float* pp = part + ((static_cast<size_t>(pair) * G + g) * max_splits + seg_first) * (D + 2);
#pragma unroll
          for (int e = 0; e < DPL; ++e) pp[lane * DPL + e] = acc[g][e];
          if (lane == 0) {
            pp[D] = m_run[g];
            pp[D + 1] = l_run[g];
          }
        }
        __threadfence();
      }
      tc::named_sync(1, kApCompute);
    };
    // first item of CTA b's range
    auto lo_of = [&](int b) { return static_cast<int>(static_cast<long long>(b) * total / gridDim.x); };
    auto combine = [&](int pair) {
      // the head's partials sit in the slots of the first items of the CTA
      // ranges that meet it; combined in slot order
      const int x0 = pair * nsplit, x1 = x0 + nsplit;
      if (ct == 0) {
        const int nb = static_cast<int>(gridDim.x);
        int b = static_cast<int>(static_cast<long long>(x0) * nb / total);
        while (b + 1 < nb && lo_of(b + 1) <= x0) ++b;
        while (b > 0 && lo_of(b) > x0) --b;
        int n = 0;
        for (; b < nb && n < kApMaxSlots; ++b) {
          const int l0 = lo_of(b);
          if (l0 >= x1) break;
          s_slots[n++] = max(l0, x0) - x0;
        }
        *s_nslot = n;
      }
      tc::named_sync(1, kApCompute);
      const int ns = *s_nslot;
      const size_t pb = static_cast<size_t>(pair) * G * max_splits;
      float* mw = tb;                          // [G][kApMaxSlots] maxima, then weights
      float* lw = tb + G * kApMaxSlots;        // [G][kApMaxSlots] sums
      for (int idx = ct; idx < G * ns; idx += kApCompute) {
        const int g = idx / ns, si = idx - g * ns;
        const float* pp = part + (pb + static_cast<size_t>(g) * max_splits + s_slots[si]) * (D + 2);
        mw[g * kApMaxSlots + si] = __ldcg(pp + D);
        lw[g * kApMaxSlots + si] = __ldcg(pp + D + 1);
      }
      tc::named_sync(1, kApCompute);
      if (ct < G) {
        float M = -INFINITY, den = 0.f;
        for (int si = 0; si < ns; ++si) M = fmaxf(M, mw[ct * kApMaxSlots + si]);
        for (int si = 0; si < ns; ++si) den = fmaf(exp2f(mw[ct * kApMaxSlots + si] - M), lw[ct * kApMaxSlots + si], den);
        const float inv = 1.f / den;
        for (int si = 0; si < ns; ++si) mw[ct * kApMaxSlots + si] = exp2f(mw[ct * kApMaxSlots + si] - M) * inv;
      }
      tc::named_sync(1, kApCompute);
      for (int idx = ct; idx < G * D; idx += kApCompute) {
        const int g = idx / D, dd = idx - g * D;
        const float* pg = part + (pb + static_cast<size_t>(g) * max_splits) * (D + 2) + dd;
        float num = 0.f;
#pragma unroll 4
        for (int si = 0; si < ns; ++si) num = fmaf(mw[g * kApMaxSlots + si], __ldcg(pg + s_slots[si] * (D + 2)), num);
        out[(static_cast<size_t>(pair) * G + g) * D + dd] = __float2bfloat16_rn(num);
      }
      if (ct == 0) ticket[pair] = 0;
      tc::named_sync(1, kApCompute);
    };
    auto finish_pair = [&](int pair, int items) {
      flush(pair);
      if (ct == 0) *s_last = atomicAdd(&ticket[pair], items) + items == nsplit;
      tc::named_sync(1, kApCompute);
      if (*s_last) {
        __threadfence();
        combine(pair);
      }
    };
    for (int it = 0; it < hi - lo; ++it) {
      const int item = lo + it, pair = item / nsplit, j = item - pair * nsplit;
      const ApSeg sg = ap_item(j, i_out, i_sp, n_out, n_sp, n_loc);
      if (pair != cur) {
        if (cur >= 0) finish_pair(cur, items_in_pair);
        // new head: q (scaled to log2 units) and fresh running state
        for (int i = ct; i < G * D; i += kApCompute)
          qs[i] = __bfloat162float(q[static_cast<size_t>(pair) * G * D + i]) * scale_log2;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          m_run[g] = -INFINITY;
          l_run[g] = 0.f;
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[g][e] = 0.f;
        }
        cur = pair;
        seg_first = j;
        items_in_pair = 0;
        tc::named_sync(1, kApCompute);
      }
      ++items_in_pair;
      const int st = it % NST;
      if (!dead) {
        bool ok = *s_abort == 0 && tc::mbar_wait(&full[st], (it / NST) & 1, kWaitLimit);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0 && !*s_abort) {
            *s_abort = 1;
            flag_error(status, DEV_TIMEOUT);
          }
          dead = true;
        }
      }
      if (dead) continue;
      const unsigned char* sK = stages + st * SB;
      const unsigned char* sV = sK + kApS * D * 2;
      // ---- logits of row `row`, quarter `qsel` of d
      float2 a2[G];
#pragma unroll
      for (int g = 0; g < G; ++g) a2[g] = make_float2(0.f, 0.f);
#pragma unroll
      for (int jj = 0; jj < NCH / 4; ++jj) {
        const int cc = qsel * (NCH / 4) + jj, cb = cc >> 3, u = cc & 7;
        const uint4 raw = *reinterpret_cast<const uint4*>(sK + cb * (kApS * 128) + row * 128 +
                                                           ((u ^ (row & 7)) << 4));
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4* qv = reinterpret_cast<const float4*>(qs + g * D + cc * 8);
          const float4 q0 = qv[0], q1 = qv[1];
          const float qq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 x = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
            a2[g] = __ffma2_rn(x, make_float2(qq[2 * e], qq[2 * e + 1]), a2[g]);
          }
        }
      }
      // ---- this warp's 8 rows: max, p, sum (lanes of one quarter hold all 8)
      const bool valid = row < sg.cnt;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float v = a2[g].x + a2[g].y;
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        float m = valid ? v : -INFINITY;
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        const float m_new = fmaxf(m_run[g], m);
        const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run[g] - m_new);
        const float p = valid ? exp2f(v - m_new) : 0.f;
        float z = p;
        z += __shfl_xor_sync(0xffffffffu, z, 1);
        z += __shfl_xor_sync(0xffffffffu, z, 2);
        z += __shfl_xor_sync(0xffffffffu, z, 4);
        l_run[g] = l_run[g] * alpha + z;
        m_run[g] = m_new;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[g][e] *= alpha;
        if (qsel == 0) pw[g * 8 + rsub] = p;
      }
      __syncwarp();
      // ---- P V over this warp's rows that hold tokens (V past cnt may be stale)
      const int nv = min(8, sg.cnt - cw * 8);
      for (int t = 0; t < nv; ++t) {
        const unsigned char* vr = sV + (cw * 8 + t) * (D * 2) + lane * (DPL * 2);
        float v[DPL];
        if constexpr (DPL == 4) {
          const uint2 raw = *reinterpret_cast<const uint2*>(vr);
          v[0] = __uint_as_float(raw.x << 16); v[1] = __uint_as_float(raw.x & 0xffff0000u);
          v[2] = __uint_as_float(raw.y << 16); v[3] = __uint_as_float(raw.y & 0xffff0000u);
        } else {
          const uint32_t raw = *reinterpret_cast<const uint32_t*>(vr);
          v[0] = __uint_as_float(raw << 16); v[1] = __uint_as_float(raw & 0xffff0000u);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = pw[g * 8 + t];
#pragma unroll
          for (int e = 0; e < DPL; e += 2) {
            const float2 r2 = __ffma2_rn(make_float2(p, p), make_float2(v[e], v[e + 1]),
                                         make_float2(acc[g][e], acc[g][e + 1]));
            acc[g][e] = r2.x;
            acc[g][e + 1] = r2.y;
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[st]);
    }
    if (cur >= 0) finish_pair(cur, items_in_pair);
  }
  __syncthreads();
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 ap_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 3D bf16 map over [pairs][rows][D]: box 64 columns x 64 rows x 1, 128-byte
// swizzle; rows past `rows` of a head read as zeros.
static cudaError_t ap_encode(CUtensorMap* map, void* base, int D, int rows, uint64_t pairs) {
  auto fn = ap_encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), pairs};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kApS), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool attn_pipe_supported(const shadowkv_params& p) {
  const int G = p.h_q / p.h_kv;
  return p.dtype == SKV_DTYPE_BF16 && (p.d == 64 || p.d == 128) && p.c <= kApS && kApS % p.c == 0 &&
         ap_smem_bytes(G, p.d, ap_stages(G, p.d)) <= 113 * 1024;
}

cudaError_t make_attn_maps(Ctx& c) {
  c.attn_pipe = false;
  if (!attn_pipe_supported(c.p)) return cudaSuccess;
  const uint64_t pairs = static_cast<uint64_t>(c.p.b) * c.p.h_kv;
  const int n_out = c.p.o * c.p.c;
  cudaError_t e = ap_encode(&c.mapKs, c.K_sparse, c.p.d, c.p.k * c.p.c, pairs);
  if (e == cudaSuccess && n_out > 0) e = ap_encode(&c.mapKo, c.K_out, c.p.d, n_out, pairs);
  if (e == cudaSuccess) e = ap_encode(&c.mapKl, c.K_loc, c.p.d, c.loc_cap, pairs);
  if (e == cudaSuccess) c.attn_pipe = true;
  return e;
}

int attn_pipe_splits(const Ctx& c, int n_loc) {
  const int n_out = c.p.o * c.p.c, n_sp = c.p.k * c.p.c;
  return (n_out + kApS - 1) / kApS + (n_sp + kApS - 1) / kApS + (n_loc + kApS - 1) / kApS;
}

template <int D, int G>
static cudaError_t attn_pipe_t(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st) {
  constexpr int NST = ap_stages(G, D);
  const int smem = ap_smem_bytes(G, D, NST);
  auto kern = k_attn_pipe<D, G, NST>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int npairs = c.p.b * c.p.h_kv;
  const int items = npairs * attn_pipe_splits(c, n_loc);
  // each CTA owns >= 1 item, so a head meets at most nsplit ranges; bounding
  // the grid by npairs * (kApMaxSlots - 2) keeps that within kApMaxSlots
  const int grid = std::min(std::min(2 * c.nsm, items), npairs * (kApMaxSlots - 2));
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  kern<<<grid, kApThreads, smem, st>>>(
      c.mapKo, c.mapKs, c.mapKl, static_cast<const bf16*>(c.V_out), static_cast<const bf16*>(c.slot_V),
      c.sel_slot, static_cast<const bf16*>(c.V_loc), static_cast<const bf16*>(q), static_cast<bf16*>(out),
      c.attn_part, c.attn_count, c.p.o * c.p.c, c.p.k * c.p.c, n_loc, c.loc_cap, c.p.c, c.p.k, npairs,
      c.max_splits, scale_log2, c.status);
  return cudaGetLastError();
}

cudaError_t launch_attn_pipe(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st) {
  if (attn_pipe_splits(c, n_loc) > c.max_splits) return cudaErrorInvalidValue;
  if (c.p.d == 128) {
    switch (c.G) {
      case 1: return attn_pipe_t<128, 1>(c, q, out, n_loc, st);
      case 2: return attn_pipe_t<128, 2>(c, q, out, n_loc, st);
      case 4: return attn_pipe_t<128, 4>(c, q, out, n_loc, st);
      default: return attn_pipe_t<128, 8>(c, q, out, n_loc, st);
    }
  }
  switch (c.G) {
    case 1: return attn_pipe_t<64, 1>(c, q, out, n_loc, st);
    case 2: return attn_pipe_t<64, 2>(c, q, out, n_loc, st);
    case 4: return attn_pipe_t<64, 4>(c, q, out, n_loc, st);
    default: return attn_pipe_t<64, 8>(c, q, out, n_loc, st);
  }
}

}  // namespace skv
