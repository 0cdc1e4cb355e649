// Sparse attention of ShadowKV's decode step (Algorithm 2 step 4):
// out = softmax(q K^T / sqrt(d)) V over [outliers; RoPE(K_sparse); local],
// split-KV over the token list with the G query heads of a KV head sharing
// every K/V row.
//
// Block (pair, split) owns tokens [split*S, min(T, split*S + S)).  All its
// K and V rows are copied to shared memory with cp.async at once (the copies
// of one block are all in flight together); K rows are stored with their
// 16-byte chunks XOR-swizzled by the row index so that the one-row-per-thread
// dot products read shared memory without bank conflicts.  Logits and
// probabilities stay in shared memory.  Each block writes a partial
// (max, sum, sum p v) per head; the last block of the pair (atomic ticket)
// combines the splits in split order, so the result does not depend on which
// block finishes last.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace skv {

constexpr int kAt = 256;        // threads per attention block
constexpr int kMaxSplit = 256;  // largest split (tokens)

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

template <typename T, int D>
struct AttnLayout {
  static constexpr int RB = D * static_cast<int>(sizeof(T));  // bytes per K/V row
  static constexpr int NCH = RB / 16;                          // 16-byte chunks per row
  static constexpr int V = 16 / static_cast<int>(sizeof(T));   // elements per chunk
};

// Shared memory: K and V rows [S][D] each, q [G][D] and p [G][S] in fp32, and
// the split weights of the combine [G][max_splits]; the P V partial sums
// [kAt/(D/2)][G][D] reuse the K/V space (extended if they are larger).
size_t attn_smem_bytes(int E, int G, int D, int S, int max_splits) {
  const size_t rb = static_cast<size_t>(D) * E;
  const size_t pv = static_cast<size_t>(kAt / (D / 2)) * G * D * sizeof(float);
  const size_t kv = 2 * static_cast<size_t>(S) * rb;
  return (kv > pv ? kv : pv) +
         sizeof(float) * (static_cast<size_t>(G) * D + static_cast<size_t>(G) * S +
                          static_cast<size_t>(G) * max_splits);
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kAt)
k_attn(const T* __restrict__ K_out, const T* __restrict__ V_out, const T* __restrict__ K_sp,
       const T* __restrict__ slot_V, const int32_t* __restrict__ sel_slot,
       const T* __restrict__ K_loc, const T* __restrict__ V_loc, const T* __restrict__ q,
       T* __restrict__ out, float* __restrict__ part, int32_t* __restrict__ ticket, int n_out,
       int n_sp, int n_loc, int loc_cap, int c, int c_shift, int k, int S, int nsplit, int max_splits,
       float scale_log2, const T* __restrict__ KVo, const T* __restrict__ KVs, const T* __restrict__ KVl) {
  using Lay = AttnLayout<T, D>;
  constexpr int RB = Lay::RB, NCH = Lay::NCH, V = Lay::V;
  constexpr int NDP = D / 2;          // dimension pairs
  constexpr int TG = kAt / NDP;       // token groups in P V
  extern __shared__ __align__(16) unsigned char sm[];
  unsigned char* Ks = sm;
  unsigned char* Vs = sm + static_cast<size_t>(S) * RB;
  constexpr int PVB = (kAt / (D / 2)) * G * D * 4;   // bytes of the P V partial sums
  const int kvb = 2 * S * RB;
  float* qs = reinterpret_cast<float*>(sm + (kvb > PVB ? kvb : PVB));
  float* ps = qs + G * D;
  float* wts = ps + G * S;                       // [G][max_splits], combine only
  float* pvred = reinterpret_cast<float*>(sm);   // reuses K/V after the logits
  __shared__ float red[kAt / 32][G];
  __shared__ float hm[G], hl[G];
  __shared__ int last;
  __shared__ int s_slot[kMaxSplit + 1];   // cache slots of the split's rebuilt chunks

  const int pair = blockIdx.x, split = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T_all = n_out + n_sp + n_loc;
  const int t0 = split * S, cnt = min(T_all, t0 + S) - t0;
  // chunk range of the split's part of the rebuilt segment
  const int sp0 = max(t0, n_out) - n_out, sp1 = min(t0 + cnt, n_out + n_sp) - n_out;
  const int ch0 = sp0 / c;
  if (sp1 > sp0)
    for (int i = tid; i <= (sp1 - 1) / c - ch0; i += kAt) s_slot[i] = sel_slot[static_cast<size_t>(pair) * k + ch0 + i];
  __syncthreads();

  // ---- copy the split's K and V rows to shared memory: LPR lanes per row,
  // one 16-byte chunk each, so every warp instruction covers whole rows
  constexpr int LPR = NCH < 32 ? NCH : 32;
  constexpr int RPI = kAt / LPR;
  const int lc = tid % LPR;
  for (int i = tid / LPR; i < cnt; i += RPI) {
    int t = t0 + i;
    const T *kr = nullptr, *vr = nullptr, *rec = nullptr;
    int u = 0;   // row within its 8-row group record
    if (t < n_out) {
      if (KVo) rec = KVo + (static_cast<size_t>(pair) * n_out + (t & ~7)) * 2 * D;
      kr = K_out + (static_cast<size_t>(pair) * n_out + t) * D;
      vr = V_out + (static_cast<size_t>(pair) * n_out + t) * D;
      u = t & 7;
    } else if ((t -= n_out) < n_sp) {
      const int cq = c_shift >= 0 ? (t >> c_shift) : t / c;
      const int slot = s_slot[cq - ch0];
      const int rr = t - cq * c;
      if (KVs) {
        rec = KVs + ((static_cast<size_t>(pair) * k + slot) * c + (rr & ~7)) * 2 * D;
      } else {
        kr = K_sp + (static_cast<size_t>(pair) * n_sp + t) * D;
        vr = slot_V + ((static_cast<size_t>(pair) * k + slot) * c + rr) * D;
      }
      u = rr & 7;
    } else {
      t -= n_sp;
      if (KVl) rec = KVl + (static_cast<size_t>(pair) * loc_cap + (t & ~7)) * 2 * D;
      kr = K_loc + (static_cast<size_t>(pair) * loc_cap + t) * D;
      vr = V_loc + (static_cast<size_t>(pair) * loc_cap + t) * D;
      u = t & 7;
    }
    unsigned char* krow = Ks + static_cast<size_t>(i) * RB;
    unsigned char* vrow = Vs + static_cast<size_t>(i) * RB;
#pragma unroll
    for (int ch = lc; ch < NCH; ch += LPR) {
      if (rec == nullptr) {
        cp_async16(krow + ((ch ^ (i & (NCH - 1))) << 4), kr + ch * V);
        cp_async16(vrow + (ch << 4), vr + ch * V);
      } else if constexpr (sizeof(T) == 2 && D == 128) {
        // group record: key piece ch of row u contiguous in the K tile;
        // value dimensions 8ch + r of row u 8 elements apart in the V^T tile
        cp_async16(krow + ((ch ^ (i & (NCH - 1))) << 4), rec + ch * 64 + u * 8);
        const uint16_t* gb = reinterpret_cast<const uint16_t*>(rec + 1024) + ch * 64 + u;
        uint32_t w[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) w[r] = static_cast<uint32_t>(gb[16 * r]) | (static_cast<uint32_t>(gb[16 * r + 8]) << 16);
        *reinterpret_cast<uint4*>(vrow + (ch << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  for (int i = tid; i < G * D; i += kAt)
    qs[i] = Ty<T>::to_f(q[static_cast<size_t>(pair) * G * D + i]) * scale_log2;
  cp_async_wait_all();
  __syncthreads();

  // ---- logits (log2 domain): two threads per token, one half of d each
  float lmax[G];
#pragma unroll
  for (int g = 0; g < G; ++g) lmax[g] = -INFINITY;
  const int hsel = tid & 1;
  for (int i0 = 0; i0 < cnt; i0 += kAt / 2) {
    const int i = i0 + (tid >> 1);
    float2 acc2[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc2[g] = make_float2(0.f, 0.f);
    if (i < cnt) {
      const unsigned char* row = Ks + static_cast<size_t>(i) * RB;
#pragma unroll
      for (int j = 0; j < NCH / 2; ++j) {
        const int ch = hsel * (NCH / 2) + j;
        float x[V];
        Ty<T>::load16(reinterpret_cast<const T*>(row + ((ch ^ (i & (NCH - 1))) << 4)), x);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2* qg = reinterpret_cast<const float2*>(qs + g * D + ch * V);
#pragma unroll
          for (int e = 0; e < V / 2; ++e)
            acc2[g] = __ffma2_rn(make_float2(x[2 * e], x[2 * e + 1]), qg[e], acc2[g]);
        }
      }
    }
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      acc[g] = acc2[g].x + acc2[g].y;
      acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 1);
      if (i < cnt) {
        if (hsel == 0) ps[g * S + i] = acc[g];
        lmax[g] = fmaxf(lmax[g], acc[g]);
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float m = warp_max(lmax[g]);
    if (lane == 0) red[warp][g] = m;
  }
  __syncthreads();
  if (tid < G) {
    float m = -INFINITY;
    for (int w = 0; w < kAt / 32; ++w) m = fmaxf(m, red[w][tid]);
    hm[tid] = m;
  }
  __syncthreads();
  float lsum[G];
#pragma unroll
  for (int g = 0; g < G; ++g) lsum[g] = 0.f;
  for (int i = tid; i < cnt; i += kAt) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float p = exp2f(ps[g * S + i] - hm[g]);
      ps[g * S + i] = p;
      lsum[g] += p;
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float z = warp_sum(lsum[g]);
    if (lane == 0) red[warp][g] = z;
  }
  __syncthreads();
  if (tid < G) {
    float z = 0.f;
    for (int w = 0; w < kAt / 32; ++w) z += red[w][tid];
    hl[tid] = z;
  }

  // ---- P V: thread owns dimensions (2 dp, 2 dp + 1) for tokens tg, tg + TG, ...
  const int dp = tid % NDP, tg = tid / NDP;
  float2 acc[G];
#pragma unroll
  for (int g = 0; g < G; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll 4
  for (int i = tg; i < cnt; i += TG) {
    float2 v;
    if constexpr (sizeof(T) == 2) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(Vs + static_cast<size_t>(i) * RB + dp * 4);
      v = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
      v = *reinterpret_cast<const float2*>(Vs + static_cast<size_t>(i) * RB + dp * 8);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float p = ps[g * S + i];
      acc[g] = __ffma2_rn(make_float2(p, p), v, acc[g]);
    }
  }
  __syncthreads();   // K/V no longer read: reuse for the token-group sums
#pragma unroll
  for (int g = 0; g < G; ++g)
    *reinterpret_cast<float2*>(&pvred[(tg * G + g) * D + 2 * dp]) = acc[g];
  __syncthreads();
  const size_t pbase = static_cast<size_t>(pair) * G * max_splits;
  for (int idx = tid; idx < G * D; idx += kAt) {
    const int g = idx / D, dd = idx - g * D;
    float sacc = 0.f;
#pragma unroll
    for (int z = 0; z < TG; ++z) sacc += pvred[(z * G + g) * D + dd];
    float* pp = part + ((pbase + static_cast<size_t>(g) * max_splits + split) * (D + 2));
    pp[dd] = sacc;
    if (dd == 0) { pp[D] = hm[g]; pp[D + 1] = hl[g]; }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last = (atomicAdd(&ticket[pair], 1) == nsplit - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  // combine: weight of split sp for head g = 2^(m_sp - M) / sum_sp' 2^(m_sp' - M) l_sp'
  for (int idx = tid; idx < G * nsplit; idx += kAt) {
    const int g = idx / nsplit, sp = idx - g * nsplit;
    wts[idx] = __ldcg(part + (pbase + static_cast<size_t>(g) * max_splits + sp) * (D + 2) + D);
  }
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY, den = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, wts[tid * nsplit + sp]);
    for (int sp = 0; sp < nsplit; ++sp) {
      const float l = __ldcg(part + (pbase + static_cast<size_t>(tid) * max_splits + sp) * (D + 2) + D + 1);
      den = fmaf(exp2f(wts[tid * nsplit + sp] - M), l, den);
    }
    hm[tid] = M;
    hl[tid] = 1.f / den;
  }
  __syncthreads();
  for (int idx = tid; idx < G * nsplit; idx += kAt) {
    const int g = idx / nsplit;
    wts[idx] = exp2f(wts[idx] - hm[g]) * hl[g];
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kAt) {
    const int g = idx / D, dd = idx - g * D;
    const float* pp = part + (pbase + static_cast<size_t>(g) * max_splits) * (D + 2) + dd;
    float num = 0.f;
#pragma unroll 8
    for (int sp = 0; sp < nsplit; ++sp) num = fmaf(wts[g * nsplit + sp], __ldcg(pp + sp * (D + 2)), num);
    out[(static_cast<size_t>(pair) * G + g) * D + dd] = Ty<T>::from_f(num);
  }
  if (tid == 0) ticket[pair] = 0;
}

template <typename T, int D, int G>
static cudaError_t attn_t(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st) {
  const int S = c.split_tokens;
  const int n_out = c.p.o * c.p.c, n_sp = c.p.k * c.p.c;
  const int T_all = n_out + n_sp + n_loc;
  const int nsplit = (T_all + S - 1) / S;
  if (nsplit > c.max_splits) return cudaErrorInvalidValue;
  const size_t smem = attn_smem_bytes(sizeof(T), G, D, S, c.max_splits);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto kern = k_attn<T, D, G>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  kern<<<dim3(c.p.b * c.p.h_kv, nsplit), kAt, smem, st>>>(
      static_cast<const T*>(c.K_out), static_cast<const T*>(c.V_out),
      static_cast<const T*>(c.K_sparse), static_cast<const T*>(c.slot_V), c.sel_slot,
      static_cast<const T*>(c.K_loc), static_cast<const T*>(c.V_loc), static_cast<const T*>(q),
      static_cast<T*>(out), c.attn_part, c.attn_count, n_out, n_sp, n_loc, c.loc_cap, c.p.c,
      (c.p.c & (c.p.c - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(c.p.c)) : -1, c.p.k, S, nsplit,
      c.max_splits, scale_log2, static_cast<const T*>(c.KV_out), static_cast<const T*>(c.KV_slot),
      static_cast<const T*>(c.KV_loc));
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t attn_d(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st) {
  switch (c.G) {
    case 1: return attn_t<T, D, 1>(c, q, out, n_loc, st);
    case 2: return attn_t<T, D, 2>(c, q, out, n_loc, st);
    case 4: return attn_t<T, D, 4>(c, q, out, n_loc, st);
    default: return attn_t<T, D, 8>(c, q, out, n_loc, st);
  }
}

cudaError_t launch_attn(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st) {
  kbegin(c, K_ATTN, st);
  cudaError_t e;
  if (c.kv_rec && !c.force_simt && !c.split_set)
    e = launch_attn_tc(c, q, out, n_loc, st);
  else if (c.attn_pipe && !c.kv_rec && !c.force_simt && !c.split_set)
    e = launch_attn_pipe(c, q, out, n_loc, st);
  else if (c.p.dtype == SKV_DTYPE_BF16)
    e = c.p.d == 128 ? attn_d<bf16, 128>(c, q, out, n_loc, st) : attn_d<bf16, 64>(c, q, out, n_loc, st);
  else
    e = c.p.d == 128 ? attn_d<float, 128>(c, q, out, n_loc, st) : attn_d<float, 64>(c, q, out, n_loc, st);
  kend(c, K_ATTN, st);
  return e;
}

}  // namespace skv

// ============================================= attention without allocation
// Scratch of shadowkv_attention_noalloc: the split partials, then (from the
// next 256-byte boundary) one completion ticket per (batch, KV head).  One
// copy per device, alive until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SKV_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the symbol's host-side name is not a device address).
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

template <typename T, int D, int G>
cudaError_t noalloc_launch(const shadowkv_params& p, const void* q, const void* K, const void* V,
                           int n_tokens, void* out, float* part, int32_t* ticket, int nsplit,
                           cudaStream_t st) {
  constexpr int S = 128;
  const size_t smem = skv::attn_smem_bytes(sizeof(T), G, D, S, nsplit);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto kern = skv::k_attn<T, D, G>;
  cudaError_t e = skv::set_smem_once(reinterpret_cast<const void*>(kern), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  // every token is one plain segment: no rebuilt chunks, no local window
  kern<<<dim3(p.b * p.h_kv, nsplit), skv::kAt, smem, st>>>(
      static_cast<const T*>(K), static_cast<const T*>(V), static_cast<const T*>(K),
      static_cast<const T*>(V), nullptr, static_cast<const T*>(K), static_cast<const T*>(V),
      static_cast<const T*>(q), static_cast<T*>(out), part, ticket, n_tokens, 0, 0, 0, 1, 0, 1, S,
      nsplit, nsplit, scale_log2, nullptr, nullptr, nullptr);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t noalloc_g(const shadowkv_params& p, const void* q, const void* K, const void* V,
                      int n_tokens, void* out, float* part, int32_t* ticket, int nsplit,
                      cudaStream_t st) {
  switch (p.h_q / p.h_kv) {
    case 1: return noalloc_launch<T, D, 1>(p, q, K, V, n_tokens, out, part, ticket, nsplit, st);
    case 2: return noalloc_launch<T, D, 2>(p, q, K, V, n_tokens, out, part, ticket, nsplit, st);
    case 4: return noalloc_launch<T, D, 4>(p, q, K, V, n_tokens, out, part, ticket, nsplit, st);
    default: return noalloc_launch<T, D, 8>(p, q, K, V, n_tokens, out, part, ticket, nsplit, st);
  }
}
}  // namespace

extern "C" skv_status shadowkv_attention_noalloc(const shadowkv_params* p, const void* q,
                                                 const void* K, const void* V, int n_tokens,
                                                 void* out, void* stream) {
  using skv::set_error;
  if (!p || !q || !K || !V || !out) return set_error(SKV_ERR_INVALID_ARG, "NULL argument");
  if (p->b < 1 || p->h_kv < 1 || p->h_q < 1 || p->h_q % p->h_kv)
    return set_error(SKV_ERR_INVALID_ARG, "need b, h_kv >= 1 and h_q a multiple of h_kv");
  const int G = p->h_q / p->h_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return set_error(SKV_ERR_UNSUPPORTED, "h_q / h_kv must be 1, 2, 4 or 8");
  if (p->d != 64 && p->d != 128) return set_error(SKV_ERR_UNSUPPORTED, "d must be 64 or 128");
  if (p->dtype != SKV_DTYPE_F32 && p->dtype != SKV_DTYPE_BF16)
    return set_error(SKV_ERR_INVALID_ARG, "bad dtype");
  // K and V rows are copied to shared memory 16 bytes at a time; q and out
  // are read and written element by element
  const size_t E = p->dtype == SKV_DTYPE_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(K) % 16 || reinterpret_cast<uintptr_t>(V) % 16)
    return set_error(SKV_ERR_INVALID_ARG, "K and V must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(q) % E || reinterpret_cast<uintptr_t>(out) % E)
    return set_error(SKV_ERR_INVALID_ARG, "q and out must be aligned to their element size");
  if (n_tokens < 1) return set_error(SKV_ERR_INVALID_ARG, "n_tokens must be >= 1");
  const int nsplit = (n_tokens + 127) / 128;
  const size_t part_bytes = static_cast<size_t>(p->b) * p->h_q * nsplit * (p->d + 2) * sizeof(float);
  const size_t ticket_bytes = static_cast<size_t>(p->b) * p->h_kv * sizeof(int32_t);
  const size_t part_room = (part_bytes + 255) & ~static_cast<size_t>(255);
  const size_t ticket_room = (ticket_bytes + 255) & ~static_cast<size_t>(255);
  if (part_room + ticket_room > static_cast<size_t>(SKV_NOALLOC_SCRATCH_BYTES)) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "attention_noalloc needs %zu bytes of partials and %zu of tickets; the static scratch "
             "holds %zu in all",
             part_room, ticket_room, static_cast<size_t>(SKV_NOALLOC_SCRATCH_BYTES));
    return set_error(SKV_ERR_UNSUPPORTED, msg);
  }
  void* base = nullptr;
  cudaError_t e = noalloc_scratch(&base);
  if (e != cudaSuccess) return set_error(SKV_ERR_CUDA, cudaGetErrorString(e));
  float* part = static_cast<float*>(base);
  int32_t* ticket = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(base) + part_room);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(ticket, 0, ticket_bytes, st);   // the kernel's tickets start at zero
  if (e == cudaSuccess) {
    if (p->dtype == SKV_DTYPE_BF16)
      e = p->d == 128 ? noalloc_g<skv::bf16, 128>(*p, q, K, V, n_tokens, out, part, ticket, nsplit, st)
                      : noalloc_g<skv::bf16, 64>(*p, q, K, V, n_tokens, out, part, ticket, nsplit, st);
    else
      e = p->d == 128 ? noalloc_g<float, 128>(*p, q, K, V, n_tokens, out, part, ticket, nsplit, st)
                      : noalloc_g<float, 64>(*p, q, K, V, n_tokens, out, part, ticket, nsplit, st);
  }
  if (e != cudaSuccess) return set_error(SKV_ERR_CUDA, cudaGetErrorString(e));
  return SKV_OK;
}
