// Host-side internals of the ShadowKV library: the context and the kernel
// launchers each .cu file provides to the C ABI in api.cu.
#pragma once
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>
#include <string>
#include <vector>

#include "../../include/shadowkv.h"

namespace skv {

// Kernel ids for timing and launch counting (names in api.cu).
enum KernelId {
  K_SCORE = 0,      // landmark scores P = q L^T / sqrt(d) and per-tile softmax stats
  K_SELECT,         // S2, top-k, cache set difference, local-window append
  K_FETCH,          // value misses from pinned host memory into cache slots (side stream)
  K_REBUILD,        // RoPE(Gather(A, I) B); with K/V records and the classic attention also the value fetch
  K_ATTN,           // attention over [outliers; rebuilt chunks; local window] and its merge; tensor-core path also the value fetch
  K_CHUNKSTATS,     // prefill: RoPE, chunk means, min cosine
  K_OUTLIERS,       // prefill: ArgTopK(-min cos, o) + mask
  K_GATHER,         // prefill: outlier / local-window rows
  K_GRAM,           // prefill: Gram matrix M^T M (tensor cores); CUDA-core path: M X^T
  K_GEMM,           // prefill: X G of the subspace iteration; CUDA-core path: (M X^T)^T M
  K_ORTH,           // prefill: orthonormalisation (CholeskyQR; CUDA-core path: Gram-Schmidt)
  K_MISC,           // prefill: reductions, transposes, fills
  K_SVD_A,          // prefill: the factor A = M X^T
  K_NUM
};

struct Timed {
  int kid;
  cudaEvent_t a, b;
};

// SMs reserved for the host-memory value fetch, which runs next to the key
// rebuild: on a side stream, the rebuild's grid leaving it these SMs, or
// (records with the classic attention) as the first CTAs of the rebuild's own
// launch; the tensor-core attention moves the values with its own warps.  When only the
// missed chunks are rebuilt (records) the rebuild is small and the fetch gets
// more SMs.
constexpr int kFetchSMs = 16;
constexpr int kFetchSMsRec = 64;
// CTAs of the record rebuild (missed chunks only): the attention's first
// phase runs beside it on the remaining SMs
constexpr int kRebuildSMsRec = 32;

struct Ctx {
  shadowkv_params p{};
  int device = 0;
  int nsm = 148;      // SMs of the device
  int E = 2;          // element bytes
  int n = 0, G = 1;
  int ntile = 0;      // score tiles per (b, h_kv)
  int loc_cap = 0;    // w + max_new
  int split_tokens = 128;
  bool split_set = false;       // split size chosen by the caller: classic split-KV kernel
  int max_splits = 0;
  bool cache_on = true, timing_on = false;
  long long t = 0;    // decode steps enqueued
  int n_app = 0;      // tokens appended to the local window
  long long launches = 0;
  bool has_min_cos = false, has_basis = false;

  // device arena
  char* arena = nullptr;
  size_t arena_bytes = 0;
  void *A = nullptr, *Bt = nullptr, *L = nullptr, *K_out = nullptr, *V_out = nullptr;
  void *K_loc = nullptr, *V_loc = nullptr, *slot_V = nullptr, *K_sparse = nullptr;
  float *min_cos = nullptr, *logits = nullptr, *attn_part = nullptr, *basis = nullptr;
  float2 *score_part = nullptr, *rope_tab = nullptr;
  int32_t *out_ids = nullptr, *sel = nullptr, *sel_slot = nullptr, *slot_chunk = nullptr;
  // step's compact miss list (pair*n + chunk, pair*k + slot) and its length
  // per step parity in miss_count[0..1]
  int32_t *miss_chunk = nullptr, *miss_slot = nullptr, *miss_count = nullptr, *hits = nullptr;
  int32_t *attn_count = nullptr;
  uint32_t* out_mask = nullptr;
  unsigned long long* counters = nullptr;  // [0] hits, [1] misses
  int* status = nullptr;
  // staging of shadowkv_decode_step_host, and the host pointers it has seen
  // (address -> device address when pinned and mapped, else nullptr)
  void *q_stage = nullptr, *kv_stage = nullptr, *out_stage = nullptr;
  std::vector<std::pair<const void*, const void*>> map_cache;

  // pinned host copy of V (mapped)
  void* v_cpu = nullptr;
  void* v_cpu_dev = nullptr;
  size_t v_bytes = 0;

  // tensor-core rebuild: TMA descriptors of A (b*s x r) and B^T (b*h_kv*d x r)
  CUtensorMap mapBt{}, mapK{};
  bool a_tiled = false;   // chunked region of A stored in 8-token core-matrix groups
  // Tensor-core attention (bf16, d = 128): keys and values of every 8-token
  // group in one 4 KB record, K tiles then V^T tiles in the MMA operand order;
  // the cache slots keep their rebuilt keys, so only missed chunks are rebuilt
  bool kv_rec = false;
  int fetch_sms = kFetchSMs;
  void *KV_out = nullptr, *KV_loc = nullptr, *KV_slot = nullptr;
  int32_t* miss_base = nullptr;   // per (batch, KV head): start of its misses in the step's list
  int32_t* att_slot = nullptr;    // per head: slots of its hits, then of its misses (attention order)
  int32_t* at_ctr = nullptr;      // attention work counters, 4 per step parity
  int32_t* item_done = nullptr;   // per phase-1 attention item: its value groups fetched this step
  long long at_last = -2;         // step of the last tensor-core attention launch
  uint32_t* warm_b = nullptr;     // per head: the next selection's first threshold try (0: none)
  int32_t* sc_ctr = nullptr;      // landmark-score tail tile counters, one per step parity
  long long sc_last = -2;         // step of the last tensor-core score launch
  float* score_m8 = nullptr;      // per (batch, query head, 8 chunks): max logit (tensor-core score)
  long long m8_step = -2;         // step whose score launch wrote score_m8
  // tensor map of the caller's query buffer (16-row boxes), encoded again
  // only when the buffer's address changes
  const void* q_enc = nullptr;
  CUtensorMap mapQ{};
  bool q_map = false;
  // the same queries for the attention: one 4D box per head lands in the
  // no-swizzle K-major core-matrix order ([d/8][16 rows][8])
  const void* qa_enc = nullptr;
  CUtensorMap mapQa{};
  bool qa_map = false;
  CUtensorMap mapL{};           // landmarks (b*h_kv*n x d) for the tensor-core score kernel
  bool tc_rebuild = false;      // shapes and dtype allow the tcgen05 rebuild
  bool tc_score = false;        // ... and the tcgen05 landmark scores
  bool rebuild_in_attn = false; // the attention's launch also rebuilds the missed keys
  bool force_simt = false;      // test hook: use the CUDA-core kernels anyway
  bool attn_pipe = false;       // bf16 shapes the pipelined attention handles
  CUtensorMap mapKo{}, mapKs{}, mapKl{};   // K_out, K_sparse, K_loc (64-row boxes)

  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;

  // timing
  Timed open{-1, nullptr, nullptr};
  std::vector<Timed> pending;
  std::vector<cudaEvent_t> ev_free;
  double kms[K_NUM] = {};
  long long kcount[K_NUM] = {};
};

size_t select_smem_bytes(int n, int k, int G, int nthreads = 1024);
size_t attn_smem_bytes(int E, int G, int D, int S, int max_splits);

// Records the text of a failure for shadowkv_last_error (api.cu).
skv_status set_error(skv_status st, const char* msg);

// ------------------------------------------------------------ launch hooks
// Every launcher brackets its kernel with kbegin/kend (api.cu): they count
// the launch and, with timing on, record CUDA events on the launch stream.
void kbegin(Ctx& c, int kid, cudaStream_t st);
void kend(Ctx& c, int kid, cudaStream_t st);
int num_sms(const Ctx& c);

// ------------------------------------------------------------ launchers
// decode_kernels.cu
cudaError_t launch_score(Ctx& c, const void* q, cudaStream_t st);
cudaError_t launch_select(Ctx& c, const void* k_new, const void* v_new, int loc_row,
                          cudaStream_t st);
cudaError_t launch_fetch(Ctx& c, cudaStream_t st);
// score_tc.cu (cudaErrorNotSupported: use the CUDA-core score kernel)
cudaError_t launch_score_tc(Ctx& c, const void* q, cudaStream_t st);
bool tc_score_supported(const shadowkv_params& p);
cudaError_t make_score_map(Ctx& c);
// attn.cu
cudaError_t launch_attn(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st);
// Launches kern with programmatic stream serialization: it may begin while
// the previous kernel of the stream finishes (it calls grid_dep_wait before
// reading that kernel's results).
// With pdl false it is a plain launch (the kernel's grid_dep_wait returns
// at once).
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  return launch_ex(true, kern, grid, block, smem, st, std::forward<Args>(args)...);
}
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per device, kernel and size
cudaError_t set_smem_once(const void* func, int bytes);
bool attn_pipe_supported(const shadowkv_params& p);
cudaError_t make_attn_maps(Ctx& c);
cudaError_t launch_attn_pipe(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st);
cudaError_t launch_build_mask(Ctx& c, cudaStream_t st);
// rebuild.cu
cudaError_t launch_rebuild(Ctx& c, cudaStream_t st);
// true when launch_rebuild also moves the step's value misses (records with
// the tensor-core rebuild and the classic attention): no separate fetch
// launch then
bool rebuild_fetches(const Ctx& c);
bool tc_rebuild_supported(const shadowkv_params& p);
cudaError_t make_rebuild_maps(Ctx& c);   // encodes mapBt
cudaError_t launch_tile_a(Ctx& c, int to_tiled, cudaStream_t st);   // no-op unless a_tiled
cudaError_t launch_pack_kv(Ctx& c, cudaStream_t st);                // records of outliers and local window (kv_rec)
bool attn_tc_supported(const shadowkv_params& p);
cudaError_t launch_attn_tc(Ctx& c, const void* q, void* out, int n_loc, cudaStream_t st);
// true when the tensor-core attention moves the step's value misses itself
// (warps of its own launch): no separate fetch launch then
bool attn_fetches(const Ctx& c);
// true when the tensor-core attention's launch also rebuilds the missed
// chunks' keys (its first CTAs): no separate rebuild launch then; *S, *NB
// get the rebuild pipeline's A stages and B slots
bool attn_rebuilds(const Ctx& c, int* S = nullptr, int* NB = nullptr);
cudaError_t encode_q_map(const Ctx& c, const void* q, CUtensorMap* map);
// the query map for buffer q: the context's cached one, encoded when q differs
cudaError_t q_map_for(Ctx& c, const void* q, CUtensorMap* map);
// attn_tc.cu: the attention's query map (one box per head), cached the same way
cudaError_t qa_map_for(Ctx& c, const void* q, CUtensorMap* map);
// prefill_kernels.cu
// Runs Algorithm 1 on the device.  v is a device pointer, or (v_mapped) the
// mapped device address of pinned host memory.
cudaError_t prefill_device(Ctx& c, const void* k_pre, const void* v, cudaStream_t st);
cudaError_t launch_transpose_b(Ctx& c, const void* B, cudaStream_t st);
cudaError_t launch_fill_i32(Ctx& c, int32_t* p, int32_t v, size_t n, cudaStream_t st);
// One read of the whole pinned host copy of V through its device mapping:
// the decode steps' value fetches then do not pay the first GPU access to
// each host page (measured on GB300: the first 32 steps after an offload ran
// 40% slower without it).
cudaError_t launch_read_host_v(Ctx& c, cudaStream_t st);
// b x r x D seeded standard-normal starting bases (the SVD's random start)
cudaError_t launch_random_basis(Ctx& c, float* X, cudaStream_t st);
// svd_tc.cu: the tensor-core SVD of bf16 contexts (Gram matrix + subspace
// iteration); svd_tc_basis writes the orthonormal basis to c.basis
bool svd_tc_supported(const shadowkv_params& p);
size_t svd_tc_workspace_bytes(const shadowkv_params& p, int nsm);
cudaError_t svd_tc_basis(Ctx& c, const void* K, void* ws, cudaStream_t st);   // K: bf16 keys

}  // namespace skv
