// C ABI of the ShadowKV library (include/shadowkv.h): parameter checks, the
// per-context device arena and pinned host copy of V, the decode step's
// stream/event choreography, per-kernel timing, and state export.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "internal.h"

namespace skv {
cudaError_t set_smem_once(const void* func, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  int& have = done[{dev, func}];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}
}  // namespace skv

struct shadowkv_ctx {
  skv::Ctx c;
};

namespace {

thread_local std::string g_err;

skv_status fail(skv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

skv_status cuda_fail(cudaError_t e, const char* what) {
  if (e == cudaErrorMemoryAllocation)
    return fail(SKV_ERR_OOM, "%s: %s", what, cudaGetErrorString(e));
  return fail(SKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CK(expr)                                      \
  do {                                                \
    cudaError_t e_ = (expr);                          \
    if (e_ != cudaSuccess) return cuda_fail(e_, #expr); \
  } while (0)

const char* kKernelNames[skv::K_NUM] = {
    "score", "select", "fetch", "rebuild", "attention", "chunkstats",
    "outliers", "gather", "svd_gram", "svd_iter", "orth", "misc", "svd_a"};

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Byte sizes of every device buffer of a context, in allocation order.
struct Sizes {
  size_t A, Bt, L, K_out, V_out, K_loc, V_loc, slot_V, K_sparse, KV_out, KV_loc, KV_slot;
  size_t min_cos, logits, score_part, score_m8, attn_part, basis, rope_tab;
  size_t out_ids, out_mask, sel, sel_slot, slot_chunk, miss_chunk, miss_slot;
  size_t miss_count, miss_base, att_slot, at_ctr, item_done, sc_ctr, hits, warm_b, attn_count, counters, status;
  size_t q_stage, kv_stage, out_stage;
  size_t total() const {
    const size_t v[] = {A, Bt, L, K_out, V_out, K_loc, V_loc, slot_V, K_sparse, KV_out, KV_loc, KV_slot,
                        min_cos, logits, score_part, score_m8, attn_part, basis, rope_tab, out_ids, out_mask, sel,
                        sel_slot, slot_chunk, miss_chunk, miss_slot, miss_count, miss_base, att_slot,
                        at_ctr, item_done, sc_ctr, hits, warm_b, attn_count, counters, status, q_stage, kv_stage,
                        out_stage};
    size_t t = 0;
    for (size_t x : v) t += up(x);
    return t;
  }
};

int n_of(const shadowkv_params& p) { return (p.s - p.w) / p.c; }
// Local-window rows per (batch, KV head): w + max_new rounded up to whole
// 8-token groups (tiled values are stored by group).
int loc_cap_of(const shadowkv_params& p) { return (p.w + p.max_new + 7) / 8 * 8; }
int max_splits_of(const shadowkv_params& p) {
  const long long T = static_cast<long long>(p.o + p.k) * p.c + p.w + p.max_new;
  // the smallest classic split is 32 tokens; the pipelined kernel's 64-token
  // items are aligned to the three segments (at most 3 more)
  return static_cast<int>((T + 31) / 32) + 3;
}

Sizes sizes_of(const shadowkv_params& p) {
  const size_t E = p.dtype == SKV_DTYPE_BF16 ? 2 : 4;
  const size_t b = p.b, h = p.h_kv, hq = p.h_q, d = p.d, s = p.s, r = p.r, c = p.c, k = p.k,
               o = p.o, n = n_of(p);
  const size_t cap = loc_cap_of(p);
  const size_t ntile = (n + 127) / 128, nw = (n + 31) / 32;
  Sizes z{};
  z.A = b * s * r * E;
  z.Bt = b * h * d * r * E;
  z.L = b * h * n * d * E;
  z.K_out = z.V_out = b * h * o * c * d * E;
  z.K_loc = z.V_loc = b * h * cap * d * E;
  const bool rec = skv::attn_tc_supported(p);   // records replace slot_V and K_sparse
  z.slot_V = z.K_sparse = rec ? 0 : b * h * k * c * d * E;
  z.KV_out = rec ? 2 * z.K_out : 0;
  z.KV_loc = rec ? 2 * z.K_loc : 0;
  z.KV_slot = rec ? 2 * b * h * k * c * d * E : 0;
  z.min_cos = b * h * n * 4;
  z.logits = b * hq * n * 4;
  z.score_part = b * hq * ntile * 4 * 8;   // 4 softmax partials per 128-landmark tile
  z.score_m8 = b * hq * ((n + 7) / 8) * 4;
  z.attn_part = b * hq * static_cast<size_t>(max_splits_of(p)) * (d + 2) * 4;
  z.basis = b * r * h * d * 4;
  z.rope_tab = d / 2 * 8;
  z.out_ids = b * h * o * 4;
  z.out_mask = b * h * nw * 4;
  z.sel = z.sel_slot = z.slot_chunk = z.miss_chunk = z.miss_slot = b * h * k * 4;
  z.hits = z.attn_count = z.miss_base = z.warm_b = b * h * 4;
  z.att_slot = rec ? b * h * k * 4 : 0;
  z.at_ctr = rec ? 8 * 4 : 0;
  z.item_done = rec ? b * h * k * 4 : 0;   // at most k phase-1 attention items per head
  z.sc_ctr = 2 * 4;
  z.miss_count = 2 * 4;   // compact miss-list length per step parity
  z.counters = 2 * 8;
  z.status = 4;
  // staging buffers of shadowkv_decode_step_host: q, (k_new, v_new), out
  z.q_stage = z.out_stage = b * hq * d * E;
  z.kv_stage = 2 * b * h * d * E;
  return z;
}

skv_status validate(const shadowkv_params* p) {
  if (!p) return fail(SKV_ERR_INVALID_ARG, "params is NULL");
  const shadowkv_params& q = *p;
  if (q.b < 1 || q.h_kv < 1 || q.h_q < 1) return fail(SKV_ERR_INVALID_ARG, "b, h_q, h_kv must be >= 1");
  if (q.h_q % q.h_kv) return fail(SKV_ERR_INVALID_ARG, "h_q (%d) must be a multiple of h_kv (%d)", q.h_q, q.h_kv);
  const int G = q.h_q / q.h_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(SKV_ERR_UNSUPPORTED, "h_q / h_kv = %d: supported group sizes are 1, 2, 4, 8", G);
  if (q.d != 64 && q.d != 128) return fail(SKV_ERR_UNSUPPORTED, "d = %d: supported head dims are 64, 128", q.d);
  if (q.c < 1) return fail(SKV_ERR_INVALID_ARG, "chunk size c must be >= 1");
  if (q.w < 0 || q.s <= q.w) return fail(SKV_ERR_INVALID_ARG, "need 0 <= w < s (w=%d, s=%d)", q.w, q.s);
  if ((q.s - q.w) % q.c)
    return fail(SKV_ERR_INVALID_ARG, "s - w = %d is not a multiple of c = %d", q.s - q.w, q.c);
  const int n = n_of(q);
  if (q.o < 0 || q.o >= n) return fail(SKV_ERR_INVALID_ARG, "need 0 <= o < n (o=%d, n=%d)", q.o, n);
  if (q.k < 1 || q.k > n - q.o) return fail(SKV_ERR_INVALID_ARG, "need 1 <= k <= n - o (k=%d, n-o=%d)", q.k, n - q.o);
  if (q.k > 1024) return fail(SKV_ERR_UNSUPPORTED, "k = %d > 1024 chunks per head", q.k);
  if (q.r < 1 || q.r > std::min(q.s, q.h_kv * q.d))
    return fail(SKV_ERR_INVALID_ARG, "need 1 <= r <= min(s, h_kv*d) (r=%d)", q.r);
  if (q.r > 256) return fail(SKV_ERR_UNSUPPORTED, "r = %d > 256", q.r);
  if (q.max_new < 0) return fail(SKV_ERR_INVALID_ARG, "max_new must be >= 0");
  if (static_cast<long long>(q.b) * q.h_kv * n >= (1LL << 31))
    return fail(SKV_ERR_UNSUPPORTED, "b * h_kv * n must be < 2^31 (32-bit chunk ids)");
  if (static_cast<long long>(q.s) + q.max_new >= (1LL << 24))
    return fail(SKV_ERR_UNSUPPORTED, "s + max_new must be < 2^24 (fp32-exact positions)");
  if (q.dtype != SKV_DTYPE_F32 && q.dtype != SKV_DTYPE_BF16) return fail(SKV_ERR_INVALID_ARG, "bad dtype %d", q.dtype);
  if (q.group_reduce != SKV_GROUP_MAX && q.group_reduce != SKV_GROUP_SUM)
    return fail(SKV_ERR_INVALID_ARG, "bad group_reduce %d", q.group_reduce);
  if (q.svd_iters < 0 || q.svd_iters > 64) return fail(SKV_ERR_INVALID_ARG, "svd_iters must be in [0, 64]");
  if (q.reserved != 0) return fail(SKV_ERR_INVALID_ARG, "reserved must be 0");
  if (!(q.rope_theta > 0.f) || !std::isfinite(q.rope_theta)) return fail(SKV_ERR_INVALID_ARG, "rope_theta must be > 0");
  if (skv::select_smem_bytes(n, q.k, G) > 220 * 1024)
    return fail(SKV_ERR_UNSUPPORTED, "n = %d chunks per head exceeds the selection's shared memory", n);
  return SKV_OK;
}

// Copies host memory with several threads (pageable -> pinned).
void parallel_memcpy(void* dst, const void* src, size_t bytes) {
  const size_t chunk = size_t(64) << 20;
  if (bytes <= chunk) { std::memcpy(dst, src, bytes); return; }
  unsigned nt = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
  std::vector<std::thread> th;
  for (unsigned t = 0; t < nt; ++t) {
    th.emplace_back([=] {
      const size_t per = (bytes + nt - 1) / nt;
      const size_t a = per * t, b = std::min(bytes, a + per);
      if (a < b) std::memcpy(static_cast<char*>(dst) + a, static_cast<const char*>(src) + a, b - a);
    });
  }
  for (auto& x : th) x.join();
}

// Pinned, device-mapped host memory for V: an aligned allocation whose pages
// several threads touch first, then registered with the driver (mapped,
// portable).  Registering touched pages is far cheaper than cudaHostAlloc
// of the same size, which faults and pins every page on one thread.
cudaError_t pinned_alloc(void** out, size_t bytes) {
  *out = nullptr;
  const size_t align = size_t(2) << 20;
  const size_t n = (bytes + align - 1) / align * align;
  void* p = std::aligned_alloc(align, n);
  if (!p) return cudaErrorMemoryAllocation;
  const unsigned nt = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
  std::vector<std::thread> th;
  for (unsigned t = 0; t < nt; ++t)
    th.emplace_back([=] {
      const size_t per = (n / nt + 4095) / 4096 * 4096;
      const size_t a = std::min(n, per * t), b = std::min(n, a + per);
      if (a < b) std::memset(static_cast<char*>(p) + a, 0, b - a);
    });
  for (auto& x : th) x.join();
  cudaError_t e = cudaHostRegister(p, n, cudaHostRegisterMapped | cudaHostRegisterPortable);
  if (e != cudaSuccess) {
    std::free(p);
    return e;
  }
  *out = p;
  return cudaSuccess;
}

void pinned_free(void* p) {
  if (!p) return;
  cudaHostUnregister(p);
  std::free(p);
}

void destroy(shadowkv_ctx* h) {
  if (!h) return;
  skv::Ctx& c = h->c;
  cudaSetDevice(c.device);
  cudaDeviceSynchronize();
  for (auto& t : c.pending) { cudaEventDestroy(t.a); cudaEventDestroy(t.b); }
  if (c.open.a) cudaEventDestroy(c.open.a);
  for (auto e : c.ev_free) cudaEventDestroy(e);
  if (c.ev_fork) cudaEventDestroy(c.ev_fork);
  if (c.ev_join) cudaEventDestroy(c.ev_join);
  if (c.side) cudaStreamDestroy(c.side);
  if (c.arena) cudaFree(c.arena);
  pinned_free(c.v_cpu);
  delete h;
}

// Allocates and initialises a context for params p (already validated).
skv_status create(const shadowkv_params* p, cudaStream_t st, shadowkv_ctx** out) {
  shadowkv_ctx* h = new (std::nothrow) shadowkv_ctx();
  if (!h) return fail(SKV_ERR_OOM, "host allocation of the context failed");
  skv::Ctx& c = h->c;
  c.p = *p;
  c.E = p->dtype == SKV_DTYPE_BF16 ? 2 : 4;
  c.n = n_of(*p);
  c.G = p->h_q / p->h_kv;
  c.ntile = (c.n + 127) / 128;
  c.loc_cap = loc_cap_of(*p);
  c.kv_rec = skv::attn_tc_supported(*p);
  c.fetch_sms = c.kv_rec ? skv::kFetchSMsRec : skv::kFetchSMs;
  c.max_splits = max_splits_of(*p);
  c.split_tokens = 128;
  auto bail = [&](skv_status s) { destroy(h); return s; };
  cudaError_t e = cudaGetDevice(&c.device);
  if (e != cudaSuccess) return bail(cuda_fail(e, "cudaGetDevice"));
  e = cudaDeviceGetAttribute(&c.nsm, cudaDevAttrMultiProcessorCount, c.device);
  if (e != cudaSuccess) return bail(cuda_fail(e, "cudaDeviceGetAttribute"));

  const Sizes z = sizes_of(*p);
  c.arena_bytes = z.total();
  e = cudaMalloc(reinterpret_cast<void**>(&c.arena), c.arena_bytes);
  if (e != cudaSuccess) return bail(cuda_fail(e, "cudaMalloc(context arena)"));
  char* cur = c.arena;
  auto take = [&](size_t bytes) { char* q = cur; cur += up(bytes); return static_cast<void*>(q); };
  c.A = take(z.A); c.Bt = take(z.Bt); c.L = take(z.L);
  c.K_out = take(z.K_out); c.V_out = take(z.V_out);
  c.K_loc = take(z.K_loc); c.V_loc = take(z.V_loc);
  c.slot_V = take(z.slot_V); c.K_sparse = take(z.K_sparse);
  c.KV_out = take(z.KV_out); c.KV_loc = take(z.KV_loc); c.KV_slot = take(z.KV_slot);
  if (c.kv_rec) c.slot_V = c.K_sparse = nullptr;
  else c.KV_out = c.KV_loc = c.KV_slot = nullptr;
  c.min_cos = static_cast<float*>(take(z.min_cos));
  c.logits = static_cast<float*>(take(z.logits));
  c.score_part = static_cast<float2*>(take(z.score_part));
  c.score_m8 = static_cast<float*>(take(z.score_m8));
  c.attn_part = static_cast<float*>(take(z.attn_part));
  c.basis = static_cast<float*>(take(z.basis));
  c.rope_tab = static_cast<float2*>(take(z.rope_tab));
  c.out_ids = static_cast<int32_t*>(take(z.out_ids));
  c.out_mask = static_cast<uint32_t*>(take(z.out_mask));
  c.sel = static_cast<int32_t*>(take(z.sel));
  c.sel_slot = static_cast<int32_t*>(take(z.sel_slot));
  c.slot_chunk = static_cast<int32_t*>(take(z.slot_chunk));
  c.miss_chunk = static_cast<int32_t*>(take(z.miss_chunk));
  c.miss_slot = static_cast<int32_t*>(take(z.miss_slot));
  c.miss_count = static_cast<int32_t*>(take(z.miss_count));
  c.miss_base = static_cast<int32_t*>(take(z.miss_base));
  c.att_slot = c.kv_rec ? static_cast<int32_t*>(take(z.att_slot)) : nullptr;
  c.at_ctr = c.kv_rec ? static_cast<int32_t*>(take(z.at_ctr)) : nullptr;
  c.item_done = c.kv_rec ? static_cast<int32_t*>(take(z.item_done)) : nullptr;
  c.sc_ctr = static_cast<int32_t*>(take(z.sc_ctr));
  c.hits = static_cast<int32_t*>(take(z.hits));
  c.warm_b = static_cast<uint32_t*>(take(z.warm_b));
  c.attn_count = static_cast<int32_t*>(take(z.attn_count));
  c.counters = static_cast<unsigned long long*>(take(z.counters));
  c.status = static_cast<int*>(take(z.status));
  c.q_stage = take(z.q_stage);
  c.kv_stage = take(z.kv_stage);
  c.out_stage = take(z.out_stage);

  // small state: zeroed; the cache starts empty
  const size_t small0 = static_cast<size_t>(reinterpret_cast<char*>(c.out_ids) - c.arena);
  e = cudaMemsetAsync(c.arena + small0, 0, c.arena_bytes - small0, st);
  if (e != cudaSuccess) return bail(cuda_fail(e, "cudaMemsetAsync"));
  e = skv::launch_fill_i32(c, c.slot_chunk, -1, z.slot_chunk / 4, st);
  // local window rows not yet written read as zeros (finite under zero weights)
  if (e == cudaSuccess) e = cudaMemsetAsync(c.K_loc, 0, z.K_loc, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(c.V_loc, 0, z.V_loc, st);
  if (e == cudaSuccess && c.kv_rec) e = cudaMemsetAsync(c.KV_loc, 0, z.KV_loc, st);
  if (e == cudaSuccess && c.kv_rec) e = cudaMemsetAsync(c.at_ctr, 0, z.at_ctr, st);
  if (e != cudaSuccess) return bail(cuda_fail(e, "fill slot table"));

  // RoPE frequency table: inv_freq_i / (2 pi) as an fp32 (hi, lo) pair
  std::vector<float2> tab(p->d / 2);
  for (int i = 0; i < p->d / 2; ++i) {
    const double f = std::pow(static_cast<double>(p->rope_theta), -2.0 * i / p->d) / (2.0 * M_PI);
    const float hi = static_cast<float>(f);
    tab[i] = make_float2(hi, static_cast<float>(f - static_cast<double>(hi)));
  }
  e = cudaMemcpyAsync(c.rope_tab, tab.data(), z.rope_tab, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return bail(cuda_fail(e, "upload RoPE table"));

  // pinned, mapped host copy of V
  c.v_bytes = static_cast<size_t>(p->b) * p->h_kv * p->s * p->d * c.E;
  e = pinned_alloc(&c.v_cpu, c.v_bytes);
  if (e != cudaSuccess) return bail(cuda_fail(e, "pinned host memory for V"));
  e = cudaHostGetDevicePointer(&c.v_cpu_dev, c.v_cpu, 0);
  if (e != cudaSuccess) return bail(cuda_fail(e, "cudaHostGetDevicePointer(V)"));

  e = skv::make_rebuild_maps(c);
  if (e == cudaSuccess) e = skv::make_score_map(c);
  if (e == cudaSuccess) e = skv::make_attn_maps(c);
  if (e != cudaSuccess) return bail(cuda_fail(e, "encode TMA descriptors"));

  e = cudaStreamCreateWithFlags(&c.side, cudaStreamNonBlocking);
  if (e != cudaSuccess) return bail(cuda_fail(e, "create side stream"));
  e = cudaEventCreateWithFlags(&c.ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c.ev_join, cudaEventDisableTiming);
  if (e != cudaSuccess) return bail(cuda_fail(e, "create events"));
  *out = h;
  return SKV_OK;
}

skv_status read_status(skv::Ctx& c) {
  int st = 0;
  CK(cudaMemcpy(&st, c.status, sizeof(int), cudaMemcpyDeviceToHost));
  if (st != 0) return fail(SKV_ERR_DEVICE_CHECK, "a kernel reported an out-of-range index (code %d)", st);
  return SKV_OK;
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int now = -1;
    if (prev >= 0 && cudaGetDevice(&now) == cudaSuccess && now != prev) cudaSetDevice(prev);
  }
};

// The decode step's launches (arguments already checked).
skv_status enqueue_step(skv::Ctx& c, const void* q, const void* k_new, const void* v_new, void* out,
                        cudaStream_t st) {
  const int loc_row = c.p.w + c.n_app;
  const int n_loc = loc_row + (k_new ? 1 : 0);
  CK(skv::launch_score(c, q, st));
  CK(skv::launch_select(c, k_new, v_new, loc_row, st));
  // the value fetch overlaps the key rebuild: warps of the attention's
  // launch, CTAs of the rebuild's own launch, or a kernel on the side stream
  const bool fused = skv::attn_fetches(c) || skv::rebuild_fetches(c);
  if (!fused) {
    CK(cudaEventRecord(c.ev_fork, st));
    CK(cudaStreamWaitEvent(c.side, c.ev_fork, 0));
    CK(skv::launch_fetch(c, c.side));
    CK(cudaEventRecord(c.ev_join, c.side));
  }
  if (!skv::attn_rebuilds(c)) CK(skv::launch_rebuild(c, st));
  if (!fused) CK(cudaStreamWaitEvent(st, c.ev_join, 0));
  CK(skv::launch_attn(c, q, out, n_loc, st));
  if (k_new) ++c.n_app;
  ++c.t;
  return SKV_OK;
}

// *dev = the device address of host pointer p when p is pinned host memory
// mapped into the device's address space (else nullptr).  The last few
// answers are cached by address.
cudaError_t mapped_view(skv::Ctx& c, const void* p, const void** dev) {
  *dev = nullptr;
  if (!p) return cudaSuccess;
  for (size_t i = 0; i < c.map_cache.size(); ++i)
    if (c.map_cache[i].first == p) {
      *dev = c.map_cache[i].second;
      // most recently used last, so a buffer used every step stays cached
      std::rotate(c.map_cache.begin() + i, c.map_cache.begin() + i + 1, c.map_cache.end());
      return cudaSuccess;
    }
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();   // pageable memory on older drivers: not mapped
    a.type = cudaMemoryTypeUnregistered;
  }
  const void* d = (a.type == cudaMemoryTypeHost && a.devicePointer) ? a.devicePointer : nullptr;
  if (c.map_cache.size() >= 8) c.map_cache.erase(c.map_cache.begin());
  c.map_cache.emplace_back(p, d);
  *dev = d;
  return cudaSuccess;
}

}  // namespace

// ------------------------------------------------------------- hooks
namespace skv {
int num_sms(const Ctx& c) { return c.nsm; }

static cudaEvent_t pop_event(Ctx& c) {
  if (!c.ev_free.empty()) {
    cudaEvent_t e = c.ev_free.back();
    c.ev_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

void kbegin(Ctx& c, int kid, cudaStream_t st) {
  ++c.launches;
  if (!c.timing_on) return;
  c.open.kid = kid;
  c.open.a = pop_event(c);
  if (c.open.a) cudaEventRecord(c.open.a, st);
}

void kend(Ctx& c, int kid, cudaStream_t st) {
  if (!c.timing_on || !c.open.a || c.open.kid != kid) return;
  c.open.b = pop_event(c);
  if (c.open.b) {
    cudaEventRecord(c.open.b, st);
    c.pending.push_back(c.open);
  } else {
    c.ev_free.push_back(c.open.a);
  }
  c.open = Timed{-1, nullptr, nullptr};
}
}  // namespace skv

static void drain_timers(skv::Ctx& c) {
  for (auto& t : c.pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(t.b) == cudaSuccess && cudaEventElapsedTime(&ms, t.a, t.b) == cudaSuccess) {
      c.kms[t.kid] += ms;
      c.kcount[t.kid] += 1;
    }
    c.ev_free.push_back(t.a);
    c.ev_free.push_back(t.b);
  }
  c.pending.clear();
}

namespace skv {
skv_status set_error(skv_status st, const char* msg) {
  g_err = msg;
  return st;
}
}  // namespace skv

// ============================================================== C ABI
extern "C" {

const char* shadowkv_last_error(void) { return g_err.c_str(); }

skv_status shadowkv_validate_params(const shadowkv_params* p) { return validate(p); }

skv_status shadowkv_footprint(const shadowkv_params* p, size_t* device_bytes, size_t* host_bytes) {
  skv_status s = validate(p);
  if (s != SKV_OK) return s;
  if (!device_bytes || !host_bytes) return fail(SKV_ERR_INVALID_ARG, "NULL output pointer");
  *device_bytes = sizes_of(*p).total();
  *host_bytes = static_cast<size_t>(p->b) * p->h_kv * p->s * p->d * (p->dtype == SKV_DTYPE_BF16 ? 2 : 4);
  return SKV_OK;
}

skv_status shadowkv_prefill(const shadowkv_params* p, const void* k_pre, const void* v,
                            int v_on_host, void* stream, shadowkv_ctx** out) {
  if (!out) return fail(SKV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  skv_status s = validate(p);
  if (s != SKV_OK) return s;
  if (!k_pre || !v) return fail(SKV_ERR_INVALID_ARG, "k_pre and v must be non-NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  shadowkv_ctx* h = nullptr;
  s = create(p, st, &h);
  if (s != SKV_OK) return s;
  skv::Ctx& c = h->c;
  // the prefill's kernels are always timed (CUDA events on their streams);
  // shadowkv_kernel_times reports them until the next reset
  c.timing_on = true;
  const void* v_src = v;
  cudaError_t e = cudaSuccess;
  if (v_on_host) {
    parallel_memcpy(c.v_cpu, v, c.v_bytes);
    v_src = c.v_cpu_dev;
  } else {
    // the offload to pinned host memory (and its read pass) runs on the side
    // stream beside the prefill kernels, which read the device copy of V
    e = cudaEventRecord(c.ev_fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c.side, c.ev_fork, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c.v_cpu, v, c.v_bytes, cudaMemcpyDeviceToHost, c.side);
    if (e == cudaSuccess) e = skv::launch_read_host_v(c, c.side);
    if (e == cudaSuccess) e = cudaEventRecord(c.ev_join, c.side);
  }
  if (e == cudaSuccess) e = skv::prefill_device(c, k_pre, v_src, st);
  if (e == cudaSuccess) e = skv::launch_tile_a(c, 1, st);
  if (e == cudaSuccess) e = skv::launch_pack_kv(c, st);
  if (e == cudaSuccess && v_on_host) e = skv::launch_read_host_v(c, st);
  if (e == cudaSuccess && !v_on_host) e = cudaStreamWaitEvent(st, c.ev_join, 0);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  c.timing_on = false;
  if (e != cudaSuccess) { s = cuda_fail(e, "prefill"); destroy(h); return s; }
  s = read_status(c);
  if (s != SKV_OK) { destroy(h); return s; }
  c.has_min_cos = c.has_basis = true;
  *out = h;
  return SKV_OK;
}

skv_status shadowkv_load_state(const shadowkv_params* p, const shadowkv_state_in* in, void* stream,
                               shadowkv_ctx** out) {
  if (!out) return fail(SKV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  skv_status s = validate(p);
  if (s != SKV_OK) return s;
  if (!in || !in->A || !in->B || !in->L || !in->V || (p->o > 0 && (!in->outlier_ids || !in->K_out || !in->V_out)) ||
      (p->w > 0 && (!in->K_loc || !in->V_loc)))
    return fail(SKV_ERR_INVALID_ARG, "a required state pointer is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  shadowkv_ctx* h = nullptr;
  s = create(p, st, &h);
  if (s != SKV_OK) return s;
  skv::Ctx& c = h->c;
  const Sizes z = sizes_of(*p);
  const size_t E = c.E;
  const size_t pairs = static_cast<size_t>(p->b) * p->h_kv;
  cudaError_t e = cudaMemcpyAsync(c.A, in->A, z.A, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = skv::launch_tile_a(c, 1, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c.L, in->L, z.L, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && p->o > 0) e = cudaMemcpyAsync(c.out_ids, in->outlier_ids, z.out_ids, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && p->o > 0) e = cudaMemcpyAsync(c.K_out, in->K_out, z.K_out, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && p->o > 0) e = cudaMemcpyAsync(c.V_out, in->V_out, z.V_out, cudaMemcpyDeviceToDevice, st);
  const size_t row = static_cast<size_t>(p->d) * E;
  if (e == cudaSuccess && p->w > 0)
    e = cudaMemcpy2DAsync(c.K_loc, row * c.loc_cap, in->K_loc, row * p->w, row * p->w, pairs,
                          cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && p->w > 0)
    e = cudaMemcpy2DAsync(c.V_loc, row * c.loc_cap, in->V_loc, row * p->w, row * p->w, pairs,
                          cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = skv::launch_transpose_b(c, in->B, st);
  if (e == cudaSuccess) e = skv::launch_pack_kv(c, st);
  if (e == cudaSuccess) e = skv::launch_build_mask(c, st);
  if (e == cudaSuccess) {
    if (in->v_on_host) parallel_memcpy(c.v_cpu, in->V, c.v_bytes);
    else e = cudaMemcpyAsync(c.v_cpu, in->V, c.v_bytes, cudaMemcpyDeviceToHost, st);
  }
  if (e == cudaSuccess) e = skv::launch_read_host_v(c, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) { s = cuda_fail(e, "load_state"); destroy(h); return s; }
  s = read_status(c);
  if (s != SKV_OK) { destroy(h); return s; }
  *out = h;
  return SKV_OK;
}

skv_status shadowkv_decode_step(shadowkv_ctx* h, const void* q, const void* k_new, const void* v_new,
                                void* out, void* stream) {
  if (!h) return fail(SKV_ERR_INVALID_ARG, "ctx is NULL");
  if (!q || !out) return fail(SKV_ERR_INVALID_ARG, "q and out must be non-NULL");
  if ((k_new == nullptr) != (v_new == nullptr)) return fail(SKV_ERR_INVALID_ARG, "k_new and v_new must both be given or both NULL");
  if (reinterpret_cast<uintptr_t>(q) % 16)
    return fail(SKV_ERR_INVALID_ARG, "q must be 16-byte aligned (it is read through tensor maps)");
  skv::Ctx& c = h->c;
  if (k_new && c.n_app >= c.p.max_new)
    return fail(SKV_ERR_STATE, "local window full: %d tokens appended (max_new)", c.n_app);
  DeviceGuard g(c.device);
  return enqueue_step(c, q, k_new, v_new, out, static_cast<cudaStream_t>(stream));
}

skv_status shadowkv_decode_step_host(shadowkv_ctx* h, const void* q, const void* k_new, const void* v_new,
                                     void* out, void* stream) {
  if (!h) return fail(SKV_ERR_INVALID_ARG, "ctx is NULL");
  if (!q || !out) return fail(SKV_ERR_INVALID_ARG, "q and out must be non-NULL");
  if ((k_new == nullptr) != (v_new == nullptr)) return fail(SKV_ERR_INVALID_ARG, "k_new and v_new must both be given or both NULL");
  skv::Ctx& c = h->c;
  if (k_new && c.n_app >= c.p.max_new)
    return fail(SKV_ERR_STATE, "local window full: %d tokens appended (max_new)", c.n_app);
  DeviceGuard g(c.device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t qb = static_cast<size_t>(c.p.b) * c.p.h_q * c.p.d * c.E;
  const size_t kb = static_cast<size_t>(c.p.b) * c.p.h_kv * c.p.d * c.E;
  // q goes to the staging buffer (the tensor maps stay cached on its address),
  // copied first so that the copy's start overlaps the lookups below; k_new,
  // v_new and out are used through their device mapping when they are
  // pinned host memory, else staged
  CK(cudaMemcpyAsync(c.q_stage, q, qb, cudaMemcpyHostToDevice, st));
  const void* kd = nullptr;
  const void* vd = nullptr;
  const void* oview = nullptr;
  CK(mapped_view(c, k_new, &kd));
  CK(mapped_view(c, v_new, &vd));
  CK(mapped_view(c, out, &oview));
  void* od = const_cast<void*>(oview);
  if (k_new && !kd) {
    CK(cudaMemcpyAsync(c.kv_stage, k_new, kb, cudaMemcpyHostToDevice, st));
    kd = c.kv_stage;
  }
  if (v_new && !vd) {
    CK(cudaMemcpyAsync(static_cast<char*>(c.kv_stage) + kb, v_new, kb, cudaMemcpyHostToDevice, st));
    vd = static_cast<char*>(c.kv_stage) + kb;
  }
  skv_status s = enqueue_step(c, c.q_stage, kd, vd, od ? od : c.out_stage, st);
  if (s != SKV_OK) return s;
  if (!od) CK(cudaMemcpyAsync(out, c.out_stage, qb, cudaMemcpyDeviceToHost, st));
  return SKV_OK;
}

skv_status shadowkv_rewind(shadowkv_ctx* h, void* stream) {
  if (!h) return fail(SKV_ERR_INVALID_ARG, "ctx is NULL");
  skv::Ctx& c = h->c;
  DeviceGuard g(c.device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CK(cudaStreamWaitEvent(st, c.ev_join, 0));   // the last fetch on the side stream
  CK(skv::launch_fill_i32(c, c.slot_chunk, -1, static_cast<size_t>(c.p.b) * c.p.h_kv * c.p.k, st));
  if (c.at_ctr) CK(cudaMemsetAsync(c.at_ctr, 0, 8 * sizeof(int32_t), st));
  if (c.item_done)
    CK(cudaMemsetAsync(c.item_done, 0, static_cast<size_t>(c.p.b) * c.p.h_kv * c.p.k * sizeof(int32_t), st));
  CK(cudaMemsetAsync(c.sc_ctr, 0, 2 * sizeof(int32_t), st));
  CK(cudaMemsetAsync(c.warm_b, 0, static_cast<size_t>(c.p.b) * c.p.h_kv * sizeof(uint32_t), st));
  c.n_app = 0;
  return SKV_OK;
}

void shadowkv_free(shadowkv_ctx* h) { destroy(h); }

skv_status shadowkv_set_option(shadowkv_ctx* h, int option, long long value) {
  if (!h) return fail(SKV_ERR_INVALID_ARG, "ctx is NULL");
  skv::Ctx& c = h->c;
  switch (option) {
    case SKV_OPT_CACHE:
      if (value != 0 && value != 1) return fail(SKV_ERR_INVALID_ARG, "cache option must be 0 or 1");
      c.cache_on = value == 1;
      return SKV_OK;
    case SKV_OPT_TIMING:
      if (value != 0 && value != 1) return fail(SKV_ERR_INVALID_ARG, "timing option must be 0 or 1");
      c.timing_on = value == 1;
      return SKV_OK;
    case SKV_OPT_SPLIT_TOKENS: {
      if (value < 32 || value > 256 || value % 32)
        return fail(SKV_ERR_INVALID_ARG, "split tokens must be a multiple of 32 in [32, 256]");
      if (skv::attn_smem_bytes(c.E, c.G, c.p.d, static_cast<int>(value), c.max_splits) > 227 * 1024)
        return fail(SKV_ERR_UNSUPPORTED, "split of %lld tokens does not fit in shared memory", value);
      c.split_tokens = static_cast<int>(value);
      c.split_set = true;
      return SKV_OK;
    }
    case SKV_OPT_CUDA_CORES:
      if (value != 0 && value != 1) return fail(SKV_ERR_INVALID_ARG, "option must be 0 or 1");
      c.force_simt = value == 1;
      return SKV_OK;
    case SKV_OPT_REBUILD_IN_ATTENTION:
      if (value != 0 && value != 1) return fail(SKV_ERR_INVALID_ARG, "option must be 0 or 1");
      c.rebuild_in_attn = value == 1;
      return SKV_OK;
    default:
      return fail(SKV_ERR_INVALID_ARG, "unknown option %d", option);
  }
}

skv_status shadowkv_get_stats(shadowkv_ctx* h, shadowkv_stats* out) {
  if (!h || !out) return fail(SKV_ERR_INVALID_ARG, "NULL argument");
  skv::Ctx& c = h->c;
  DeviceGuard g(c.device);
  CK(cudaDeviceSynchronize());
  unsigned long long cnt[2] = {0, 0};
  CK(cudaMemcpy(cnt, c.counters, sizeof(cnt), cudaMemcpyDeviceToHost));
  out->steps = c.t;
  out->hits = static_cast<long long>(cnt[0]);
  out->misses = static_cast<long long>(cnt[1]);
  out->link_bytes = out->misses * static_cast<long long>(c.p.c) * c.p.d * c.E;
  out->launches = c.launches;
  return SKV_OK;
}

skv_status shadowkv_get_layout(const shadowkv_ctx* h, shadowkv_layout* out) {
  if (!h || !out) return fail(SKV_ERR_INVALID_ARG, "NULL argument");
  const skv::Ctx& c = h->c;
  out->kv_records = c.kv_rec ? 1 : 0;
  out->a_tiled = c.a_tiled ? 1 : 0;
  out->tc_score = c.tc_score && !c.force_simt ? 1 : 0;
  out->tc_rebuild = c.tc_rebuild && !c.force_simt ? 1 : 0;
  out->tc_attention = c.kv_rec && !c.force_simt && !c.split_set ? 1 : 0;
  out->fetch_in_rebuild = skv::rebuild_fetches(c) ? 1 : 0;
  out->fetch_in_attention = skv::attn_fetches(c) ? 1 : 0;
  out->rebuild_in_attention = skv::attn_rebuilds(c) ? 1 : 0;
  return SKV_OK;
}

skv_status shadowkv_check(shadowkv_ctx* h) {
  if (!h) return fail(SKV_ERR_INVALID_ARG, "ctx is NULL");
  DeviceGuard g(h->c.device);
  CK(cudaDeviceSynchronize());
  return read_status(h->c);
}

int shadowkv_num_kernels(void) { return skv::K_NUM; }

const char* shadowkv_kernel_name(int id) {
  return (id >= 0 && id < skv::K_NUM) ? kKernelNames[id] : "";
}

skv_status shadowkv_kernel_times(shadowkv_ctx* h, double* ms, long long* launches, int n) {
  if (!h || n < 0 || (n > 0 && (!ms || !launches))) return fail(SKV_ERR_INVALID_ARG, "bad arguments");
  skv::Ctx& c = h->c;
  DeviceGuard g(c.device);
  drain_timers(c);
  for (int i = 0; i < n; ++i) {
    ms[i] = i < skv::K_NUM ? c.kms[i] : 0.0;
    launches[i] = i < skv::K_NUM ? c.kcount[i] : 0;
  }
  return SKV_OK;
}

skv_status shadowkv_reset_timers(shadowkv_ctx* h) {
  if (!h) return fail(SKV_ERR_INVALID_ARG, "ctx is NULL");
  skv::Ctx& c = h->c;
  DeviceGuard g(c.device);
  drain_timers(c);
  for (int i = 0; i < skv::K_NUM; ++i) { c.kms[i] = 0.0; c.kcount[i] = 0; }
  return SKV_OK;
}

static void* field_ptr(skv::Ctx& c, int field, size_t* bytes, bool* on_host) {
  const Sizes z = sizes_of(c.p);
  *on_host = false;
  switch (field) {
    case SKV_FIELD_A: *bytes = z.A; return c.A;
    case SKV_FIELD_BT: *bytes = z.Bt; return c.Bt;
    case SKV_FIELD_L: *bytes = z.L; return c.L;
    case SKV_FIELD_MIN_COS: *bytes = z.min_cos; return c.has_min_cos ? c.min_cos : nullptr;
    case SKV_FIELD_OUTLIER_IDS: *bytes = z.out_ids; return c.out_ids;
    case SKV_FIELD_K_OUT: *bytes = z.K_out; return c.K_out;
    case SKV_FIELD_V_OUT: *bytes = z.V_out; return c.V_out;
    // the local window is exported as w + max_new rows per (batch, KV head)
    case SKV_FIELD_K_LOC: *bytes = z.K_loc / c.loc_cap * (c.p.w + c.p.max_new); return c.K_loc;
    case SKV_FIELD_V_LOC: *bytes = z.V_loc / c.loc_cap * (c.p.w + c.p.max_new); return c.V_loc;
    case SKV_FIELD_SEL: *bytes = z.sel; return c.sel;
    case SKV_FIELD_SEL_SLOT: *bytes = z.sel_slot; return c.sel_slot;
    case SKV_FIELD_HITS: *bytes = z.hits; return c.hits;
    case SKV_FIELD_LOGITS: *bytes = z.logits; return c.logits;
    case SKV_FIELD_K_SPARSE:
      *bytes = c.kv_rec ? z.KV_slot / 2 : z.K_sparse;
      return c.kv_rec ? c.KV_slot : c.K_sparse;
    case SKV_FIELD_SLOT_CHUNK: *bytes = z.slot_chunk; return c.slot_chunk;
    case SKV_FIELD_SLOT_V:
      *bytes = c.kv_rec ? z.KV_slot / 2 : z.slot_V;
      return c.kv_rec ? c.KV_slot : c.slot_V;
    case SKV_FIELD_V_CPU: *bytes = c.v_bytes; *on_host = true; return c.v_cpu;
    case SKV_FIELD_SVD_BASIS: *bytes = z.basis; return c.has_basis ? c.basis : nullptr;
    default: *bytes = 0; return nullptr;
  }
}

skv_status shadowkv_field_bytes(const shadowkv_ctx* h, int field, size_t* bytes) {
  if (!h || !bytes) return fail(SKV_ERR_INVALID_ARG, "NULL argument");
  if (field < 0 || field >= SKV_FIELD_COUNT) return fail(SKV_ERR_INVALID_ARG, "unknown field %d", field);
  bool on_host;
  field_ptr(const_cast<skv::Ctx&>(h->c), field, bytes, &on_host);
  return SKV_OK;
}

// Host copy of the tiled A back to row-major: per 8-token group of the
// chunked region, core matrix q row u (16 bytes) -> row u, piece q.
static void untile_a_host(const skv::Ctx& c, unsigned char* A) {
  const int r = c.p.r, QR = r / 8;
  const size_t gbytes = static_cast<size_t>(8) * r * c.E;
  const int gpb = c.n * c.p.c / 8;
  std::vector<unsigned char> tmp(gbytes);
  for (int bb = 0; bb < c.p.b; ++bb) {
    unsigned char* base = A + static_cast<size_t>(bb) * c.p.s * r * c.E;
    for (int g = 0; g < gpb; ++g) {
      unsigned char* grp = base + g * gbytes;
      std::memcpy(tmp.data(), grp, gbytes);
      for (int q = 0; q < QR; ++q)
        for (int u = 0; u < 8; ++u) std::memcpy(grp + (u * QR + q) * 16, tmp.data() + (q * 8 + u) * 16, 16);
    }
  }
}

skv_status shadowkv_export(shadowkv_ctx* h, int field, void* dst, size_t bytes) {
  if (!h || !dst) return fail(SKV_ERR_INVALID_ARG, "NULL argument");
  if (field < 0 || field >= SKV_FIELD_COUNT) return fail(SKV_ERR_INVALID_ARG, "unknown field %d", field);
  skv::Ctx& c = h->c;
  size_t want = 0;
  bool on_host = false;
  void* src = field_ptr(c, field, &want, &on_host);
  if (!src) return fail(SKV_ERR_STATE, "field %d is not available for this context", field);
  if (bytes != want) return fail(SKV_ERR_INVALID_ARG, "field %d has %zu bytes, got %zu", field, want, bytes);
  DeviceGuard g(c.device);
  CK(cudaDeviceSynchronize());
  const size_t pairs = static_cast<size_t>(c.p.b) * c.p.h_kv;
  if (field == SKV_FIELD_K_LOC || field == SKV_FIELD_V_LOC) {
    // whole buffer, values untiled, then w + max_new of the loc_cap rows per head
    const size_t row = static_cast<size_t>(c.p.d) * c.E, keep = static_cast<size_t>(c.p.w) + c.p.max_new;
    std::vector<unsigned char> full(pairs * c.loc_cap * row);
    CK(cudaMemcpy(full.data(), src, full.size(), cudaMemcpyDeviceToHost));
    for (size_t pr = 0; pr < pairs; ++pr)
      std::memcpy(static_cast<unsigned char*>(dst) + pr * keep * row, full.data() + pr * c.loc_cap * row, keep * row);
    return SKV_OK;
  }
  if (c.kv_rec && (field == SKV_FIELD_SLOT_V || field == SKV_FIELD_K_SPARSE)) {
    // from the slot records: values per slot, or the rebuilt keys of the
    // selected chunks in selection order
    std::vector<uint16_t> rec(pairs * c.p.k * c.p.c * 256);
    CK(cudaMemcpy(rec.data(), c.KV_slot, rec.size() * 2, cudaMemcpyDeviceToHost));
    std::vector<int32_t> sel_slot(pairs * c.p.k);
    CK(cudaMemcpy(sel_slot.data(), c.sel_slot, sel_slot.size() * 4, cudaMemcpyDeviceToHost));
    uint16_t* o = static_cast<uint16_t*>(dst);
    const int gpc = c.p.c / 8;
    for (size_t pr = 0; pr < pairs; ++pr)
      for (int i = 0; i < c.p.k; ++i) {
        const int slot = field == SKV_FIELD_SLOT_V ? i : sel_slot[pr * c.p.k + i];
        if (slot < 0 || slot >= c.p.k) return fail(SKV_ERR_STATE, "slot %d out of range", slot);
        for (int u = 0; u < c.p.c; ++u) {
          const uint16_t* r = rec.data() + ((pr * c.p.k + slot) * gpc + u / 8) * 2048;
          uint16_t* row = o + ((pr * c.p.k + i) * c.p.c + u) * 128;
          for (int j = 0; j < 128; ++j)
            row[j] = field == SKV_FIELD_K_SPARSE ? r[(j >> 3) * 64 + (u & 7) * 8 + (j & 7)]
                                                 : r[1024 + (j >> 3) * 64 + (j & 7) * 8 + (u & 7)];
        }
      }
    return SKV_OK;
  }
  if (on_host) std::memcpy(dst, src, bytes);
  else CK(cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost));
  if (field == SKV_FIELD_A && c.a_tiled) untile_a_host(c, static_cast<unsigned char*>(dst));
  return SKV_OK;
}

}  // extern "C"
