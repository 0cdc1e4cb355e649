/*
 * shadowkv.h -- C ABI of the ShadowKV decode path for GB300 (sm_103a).
 *
 * The method is the one of "ShadowKV: KV Cache in Shadows for High-Throughput
 * Long-Context LLM Inference" as the xllm-io paper review page states it:
 *   - Algorithm 1 (Pre-filling): A, B <- SVD(K) over the pre-RoPE keys;
 *     landmarks L <- Reduce(K_RoPE) per chunk of c tokens; S <- cosine of
 *     each token to its chunk mean; outliers I <- ArgTopK(-Min(S), o);
 *     V offloaded to the CPU.
 *   - Algorithm 2 (Decoding): P <- MatMul(Q, L^T); I <- ArgTopK(S2, k);
 *     in parallel V_sparse <- Gather(V_CPU, I) and
 *     K_sparse <- MatMul(Gather(A, I), B); attention over
 *     [K_outlier; RoPE(K_sparse); K_local].
 *   - The temporal-locality cache (section 核心创新, and the Telegram explainer
 *     of ShadowKV): chunks selected at the previous step stay on the GPU and
 *     only the set difference is fetched from host memory.
 *
 * Conventions shared by every entry point
 *   - Tensors are dense, row-major, in the element type given by
 *     shadowkv_params.dtype (SKV_DTYPE_F32: float, SKV_DTYPE_BF16: bfloat16).
 *     Index tensors are int32.
 *   - "device" pointers are CUDA global-memory addresses on the context's
 *     device; "host" pointers are ordinary CPU addresses.  The caller owns
 *     every pointer it passes; the library never frees or keeps them past the
 *     call (prefill copies what it needs).
 *   - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued on it in order; calls return before the GPU
 *     finishes unless stated otherwise.  With bf16, d = 128 contexts the
 *     decode step's kernels all run on `stream`, chained with programmatic
 *     dependent launch; other contexts also use one library-owned side
 *     stream, joined back to `stream` before the call returns.
 *   - Every entry point returns an skv_status; on failure
 *     shadowkv_last_error() (thread-local) describes the cause.  No entry point
 *     aborts the process, traps the GPU, or falls back to the CPU.
 *   - Shapes: n = (s - w) / c chunks form the compressed region [0, s - w);
 *     the last w prompt tokens and every appended token form the exact local
 *     window.  G = h_q / h_kv query heads share a KV head; query head g uses
 *     KV head g / G.
 */
#ifndef SHADOWKV_H
#define SHADOWKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum skv_status {
  SKV_OK = 0,
  SKV_ERR_INVALID_ARG = 1,   /* bad shape, pointer, option or size */
  SKV_ERR_OOM = 2,           /* device or pinned-host allocation failed */
  SKV_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  SKV_ERR_DEVICE_CHECK = 4,  /* a kernel found an out-of-range index (status word) */
  SKV_ERR_TIMEOUT = 5,       /* a bounded device wait gave up */
  SKV_ERR_STATE = 6,         /* call not valid in the context's state (e.g. max_new reached) */
  SKV_ERR_UNSUPPORTED = 7    /* a combination the kernels do not implement */
} skv_status;

enum { SKV_DTYPE_F32 = 0, SKV_DTYPE_BF16 = 1 };
/* How S2 combines the softmax scores of a KV head's query group (S2 is not
 * defined on the page): maximum over the group (default) or their sum. */
enum { SKV_GROUP_MAX = 0, SKV_GROUP_SUM = 1 };

/* Shapes and parameters of one attention layer.  Algorithm 1's r, c, o and
 * Algorithm 2's k follow the page's notation. */
typedef struct shadowkv_params {
  int b;            /* sequences in the batch */
  int h_q;          /* query heads (multiple of h_kv) */
  int h_kv;         /* key/value heads */
  int d;            /* head dimension: 64 or 128 */
  int s;            /* prompt tokens */
  int c;            /* chunk size (tokens per landmark) */
  int r;            /* SVD rank of the pre-RoPE key cache, <= min(s, h_kv*d), <= 256 */
  int k;            /* chunks selected per KV head per step, 1..min(n - o, 1024) */
  int o;            /* outlier chunks per KV head, 0..n - 1 */
  int w;            /* local-window prompt tokens; (s - w) must be a positive multiple of c */
  int max_new;      /* decode steps the context can append */
  float rope_theta; /* RoPE base; rotate-half pairing (i, i + d/2) */
  int dtype;        /* SKV_DTYPE_F32 or SKV_DTYPE_BF16 */
  int group_reduce; /* SKV_GROUP_MAX or SKV_GROUP_SUM */
  int svd_iters;    /* subspace iterations of the prefill SVD; 0 = default (3) */
  int reserved;     /* must be 0 */
  unsigned long long seed; /* seed of the SVD's random starting basis */
} shadowkv_params;

typedef struct shadowkv_ctx shadowkv_ctx;   /* opaque, library-owned */

/* Cumulative counters of a context. */
typedef struct shadowkv_stats {
  long long steps;       /* decode steps enqueued */
  long long hits;        /* selected chunks already resident in the cache */
  long long misses;      /* selected chunks fetched from host memory */
  long long link_bytes;  /* value bytes read over the host link by the fetch */
  long long launches;    /* kernels launched by this context */
} shadowkv_stats;

/* Checks the parameters without touching the GPU. */
skv_status shadowkv_validate_params(const shadowkv_params* p);

/* Bytes the context will hold on the device and in pinned host memory
 * (excluding the transient prefill workspace).  Host-only. */
skv_status shadowkv_footprint(const shadowkv_params* p, size_t* device_bytes,
                              size_t* host_bytes);

/*
 * Algorithm 1 (Pre-filling).
 *   k_pre : device, b x h_kv x s x d, pre-RoPE keys.
 *   v     : b x h_kv x s x d values; a host pointer if v_on_host != 0, else device.
 * Computes K_RoPE (position = token index), landmarks L (chunk means of
 * K_RoPE over [0, s - w)), the per-chunk minimum cosine, the o outlier chunks
 * per (sequence, KV head) by ArgTopK(-min cos) (ties to the lower index),
 * the rank-r factors A (b x s x r) and B (b x h_kv x r x d) of the pre-RoPE
 * keys of each sequence viewed as an s x (h_kv d) matrix, the post-RoPE keys
 * and values of the outlier chunks and of the local window, and copies V to
 * library-owned pinned host memory.  On success *out owns everything; k_pre
 * and v may be freed once the call returns (it synchronizes `stream`).  The
 * prefill's kernels are timed with CUDA events whatever SKV_OPT_TIMING says;
 * shadowkv_kernel_times reports them until shadowkv_reset_timers.
 */
skv_status shadowkv_prefill(const shadowkv_params* p, const void* k_pre, const void* v,
                            int v_on_host, void* stream, shadowkv_ctx** out);

/* A compressed layer state supplied by the caller instead of computed by
 * shadowkv_prefill (checkpoint restore, or a prefill done elsewhere).  All
 * device pointers, element type p->dtype, except V (see v_on_host). */
typedef struct shadowkv_state_in {
  const void* A;               /* b x s x r */
  const void* B;               /* b x h_kv x r x d */
  const void* L;               /* b x h_kv x n x d landmarks */
  const int32_t* outlier_ids;  /* b x h_kv x o, ascending, distinct, < n */
  const void* K_out;           /* b x h_kv x (o c) x d post-RoPE outlier keys, chunk order of outlier_ids */
  const void* V_out;           /* b x h_kv x (o c) x d outlier values */
  const void* K_loc;           /* b x h_kv x w x d post-RoPE local-window keys */
  const void* V_loc;           /* b x h_kv x w x d */
  const void* V;               /* b x h_kv x s x d values (host if v_on_host) */
  int v_on_host;
} shadowkv_state_in;

/* Builds a context from a given compressed state (no prefill).  Outlier ids
 * are checked on the device; a bad id makes the call return
 * SKV_ERR_DEVICE_CHECK.  Synchronizes `stream`. */
skv_status shadowkv_load_state(const shadowkv_params* p, const shadowkv_state_in* st,
                               void* stream, shadowkv_ctx** out);

/*
 * Algorithm 2 (Decoding), one token for every sequence.
 *   q     : device, b x h_q x d, post-RoPE queries of the new token.
 *   k_new : device, b x h_kv x d, post-RoPE key of the new token, or NULL.
 *   v_new : device, b x h_kv x d, its value (NULL iff k_new is NULL).
 *   out   : device, b x h_q x d, attention output; it may also be the device
 *           address of mapped pinned host memory (the result is then written
 *           over the host link, with no separate copy).
 * With k_new given, the token is appended to the local window first (at most
 * max_new times; then SKV_ERR_STATE).  Step t (0-based) scores
 * P = q L^T / sqrt(d) over the non-outlier chunks, forms S2 (group_reduce),
 * selects the top-k chunks per KV head (ties to the lower index), rebuilds
 * their keys as RoPE(Gather(A, I) B) at their token positions, takes their
 * values from the GPU chunk cache (hits of the previous step) or from pinned
 * host memory (misses, fetched while the rest is attended), and writes
 * softmax(q K^T / sqrt(d)) V over [outliers; rebuilt chunks; local window].
 * The kernels read q in place through tensor maps: q must be 16-byte aligned
 * (else SKV_ERR_INVALID_ARG before any work is enqueued) and must not change
 * before the step has completed on `stream`.  Asynchronous on `stream`.
 */
skv_status shadowkv_decode_step(shadowkv_ctx* ctx, const void* q, const void* k_new,
                                const void* v_new, void* out, void* stream);

/* The same step with the token's inputs and output in host memory (the call
 * a caller makes whose decode loop lives on the CPU side):
 *   q     : host, b x h_q x d (copied into a library-owned device buffer)
 *   k_new, v_new : host, b x h_kv x d, or NULL; read in place through their
 *           device mapping when they are pinned host memory, else copied
 *   out   : host, b x h_q x d; written in place by the attention when it is
 *           pinned host memory, else copied back after the step
 * Pinned (page-locked) buffers make every copy asynchronous on `stream`;
 * the result is in `out` once `stream` has passed the call.  Pageable
 * buffers work too, with the copies the CUDA runtime makes for them.  The
 * pinned-or-not answer is cached per address (the last 8 addresses). */
skv_status shadowkv_decode_step_host(shadowkv_ctx* ctx, const void* q, const void* k_new,
                                     const void* v_new, void* out, void* stream);

/* Returns the context to its state right after prefill / load_state: the
 * appended tokens are dropped (the local window holds the w prompt tokens
 * again) and the chunk cache is emptied.  Stream-ordered on `stream` after
 * every earlier decode step of this context. */
skv_status shadowkv_rewind(shadowkv_ctx* ctx, void* stream);

/* Releases everything the context owns (NULL-safe).  Synchronizes the device. */
void shadowkv_free(shadowkv_ctx* ctx);

/* Text of the last failure of this thread ("" if none). */
const char* shadowkv_last_error(void);

/* ---------------------------------------------------------------- options */
enum {
  SKV_OPT_CACHE = 0,        /* 1 (default): reuse the previous step's chunks; 0: fetch all k */
  SKV_OPT_TIMING = 1,       /* 1: time each kernel with CUDA events on its stream */
  SKV_OPT_SPLIT_TOKENS = 2, /* tokens per attention split (multiple of 32 in 32..256 whose K/V
                               rows fit in shared memory; default 128).  Setting it selects the
                               classic split-KV attention kernel.  By default bf16 contexts
                               with d = 128 and c a multiple of 8 dividing 128 use the
                               tensor-core attention over K/V records; other bf16 contexts
                               use the pipelined (TMA-fed, 64-token items) kernel */
  SKV_OPT_CUDA_CORES = 3,   /* 1: compute the landmark scores and rebuild the keys with the
                               CUDA-core kernels even where the tensor-core (tcgen05) kernels
                               apply (bf16; for the rebuild also c a multiple of 8 dividing 128
                               and r a multiple of 16), and run the classic split-KV attention
                               instead of the pipelined one; for cross-checking the paths */
  SKV_OPT_REBUILD_IN_ATTENTION = 4 /* 1: where the tensor-core attention moves the values itself
                               (shadowkv_layout.fetch_in_attention) and the rebuild runs on the
                               tensor cores over tiled A, the missed chunks' keys are rebuilt
                               inside the attention's launch: its first CTAs rebuild them
                               (Algorithm 2 step 3, key branch) into the cache slots before
                               they take attention items, and each missed chunk's item waits
                               for its own keys and values.  Three launches per step instead
                               of four.  0 (default): a rebuild launch of its own */
};
skv_status shadowkv_set_option(shadowkv_ctx* ctx, int option, long long value);

/* Synchronizes the context's streams and reads the cumulative counters. */
skv_status shadowkv_get_stats(shadowkv_ctx* ctx, shadowkv_stats* out);

/* Which storage layout and kernels the context uses; they follow from the
 * parameters (and SKV_OPT_CUDA_CORES / SKV_OPT_SPLIT_TOKENS).  Host-only. */
typedef struct shadowkv_layout {
  int kv_records;       /* keys and values of every 8-token group in one 4 KB record;
                           cache slots keep their rebuilt keys, so a step rebuilds
                           only the chunks it fetches */
  int a_tiled;          /* A's chunked region in 8-token core-matrix groups */
  int tc_score;         /* landmark scores on the tensor cores (tcgen05) */
  int tc_rebuild;       /* key rebuild on the tensor cores */
  int tc_attention;     /* attention on the tensor cores over K/V records */
  int fetch_in_rebuild; /* value fetch runs as CTAs of the rebuild launch (one stream) */
  int fetch_in_attention; /* value fetch runs as warps of the tensor-core attention's
                           launch; each missed chunk is attended as soon as its
                           values are in its cache slot */
  int rebuild_in_attention; /* SKV_OPT_REBUILD_IN_ATTENTION is on and applies: the missed
                           chunks' keys are rebuilt by the first CTAs of the attention's
                           launch (three launches per step) */
} shadowkv_layout;
skv_status shadowkv_get_layout(const shadowkv_ctx* ctx, shadowkv_layout* out);

/* Synchronizes and reads the device status word (kernel bounds checks);
 * SKV_ERR_DEVICE_CHECK if any kernel recorded a violation. */
skv_status shadowkv_check(shadowkv_ctx* ctx);

/* ----------------------------------------------- attention without allocation
 * (no counterpart in the paper: a service for callers that cannot allocate)
 *
 * Some callers cannot call cudaMalloc: an inference engine that hands every
 * byte of device memory to its own pool at start-up, or code that records a
 * decode loop into a CUDA graph and must not allocate inside it.  This entry
 * point runs the library's split-KV GQA attention kernel on keys and values
 * the caller already holds and allocates nothing: its scratch (the per-split
 * partial results and the per-head completion tickets) lives in one static
 * device array of SKV_NOALLOC_SCRATCH_BYTES that the library image carries,
 * so every GPU that loads the library holds that array until the process
 * exits.
 *   p        : b, h_q, h_kv, d and dtype are used (h_q / h_kv in {1,2,4,8},
 *              d in {64, 128}); the other fields are ignored.
 *   q        : device, b x h_q x d, post-RoPE queries.
 *   K, V     : device, b x h_kv x n_tokens x d, post-RoPE keys and values.
 *   out      : device, b x h_q x d; out = softmax(q K^T / sqrt(d)) V, query
 *              head g reading KV head g / G.
 * K and V must be 16-byte aligned (their rows are copied 16 bytes at a time)
 * and q and out aligned to their element size; otherwise SKV_ERR_INVALID_ARG
 * is returned before anything is enqueued.
 * Needs P = b * h_q * ceil(n_tokens / 128) * (d + 2) * 4 bytes of partials
 * and T = b * h_kv * 4 bytes of tickets, each rounded up to 256 bytes; when
 * P + T exceeds SKV_NOALLOC_SCRATCH_BYTES the call returns
 * SKV_ERR_UNSUPPORTED.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call shares the one array and clears the
 * tickets it needs, so calls whose GPU work overlaps (different streams, or
 * different host threads on the same device without ordering) race; order
 * them on one stream.  Asynchronous on `stream`. */
#define SKV_NOALLOC_SCRATCH_BYTES (8u << 20)
skv_status shadowkv_attention_noalloc(const shadowkv_params* p, const void* q, const void* K,
                                      const void* V, int n_tokens, void* out, void* stream);

/* ------------------------------------------------------ timing / counting */
/* Kernels are numbered 0..shadowkv_num_kernels()-1 with stable names. */
int shadowkv_num_kernels(void);
const char* shadowkv_kernel_name(int id);
/* With SKV_OPT_TIMING on: total milliseconds and launch count per kernel id
 * since the last reset (arrays of n entries).  Synchronizes.  With K/V
 * records (bf16, d = 128) the value fetch runs inside the "attention" launch
 * (or, with SKV_OPT_SPLIT_TOKENS set, inside the "rebuild" launch), and
 * "fetch" counts no launches.  The events recorded between launches
 * remove the overlap between consecutive kernels, so the per-kernel times sum
 * to more than a step takes with timing off. */
skv_status shadowkv_kernel_times(shadowkv_ctx* ctx, double* ms, long long* launches, int n);
skv_status shadowkv_reset_timers(shadowkv_ctx* ctx);

/* ---------------------------------------------------------- introspection */
enum {
  SKV_FIELD_A = 0,            /* dtype b x s x r */
  SKV_FIELD_BT = 1,           /* dtype b x h_kv x d x r  (B transposed per head) */
  SKV_FIELD_L = 2,            /* dtype b x h_kv x n x d */
  SKV_FIELD_MIN_COS = 3,      /* f32 b x h_kv x n  (prefill only) */
  SKV_FIELD_OUTLIER_IDS = 4,  /* i32 b x h_kv x o */
  SKV_FIELD_K_OUT = 5,        /* dtype b x h_kv x (o c) x d */
  SKV_FIELD_V_OUT = 6,        /* dtype b x h_kv x (o c) x d */
  SKV_FIELD_K_LOC = 7,        /* dtype b x h_kv x (w + max_new) x d */
  SKV_FIELD_V_LOC = 8,        /* dtype b x h_kv x (w + max_new) x d */
  SKV_FIELD_SEL = 9,          /* i32 b x h_kv x k: last step's chunks, ascending */
  SKV_FIELD_SEL_SLOT = 10,    /* i32 b x h_kv x k: cache slot holding each selected chunk */
  SKV_FIELD_HITS = 11,        /* i32 b x h_kv: last step's cache hits */
  SKV_FIELD_LOGITS = 12,      /* f32 b x h_q x n: last step's q.L/sqrt(d) (outliers included) */
  SKV_FIELD_K_SPARSE = 13,    /* dtype b x h_kv x (k c) x d: last step's RoPE(Gather(A,I) B) */
  SKV_FIELD_SLOT_CHUNK = 14,  /* i32 b x h_kv x k: chunk in each cache slot (-1 empty) */
  SKV_FIELD_SLOT_V = 15,      /* dtype b x h_kv x k x c x d: cached values */
  SKV_FIELD_V_CPU = 16,       /* dtype b x h_kv x s x d: the pinned host copy of V */
  SKV_FIELD_SVD_BASIS = 17,   /* f32 b x r x (h_kv d): orthonormal rows spanning the rank-r
                                 right singular subspace (prefill only) */
  SKV_FIELD_COUNT = 18
};
/* Size in bytes of a field. Host-only. */
skv_status shadowkv_field_bytes(const shadowkv_ctx* ctx, int field, size_t* bytes);
/* Copies a field to host memory dst (bytes must equal the field size).
 * Synchronizes the context's streams. */
skv_status shadowkv_export(shadowkv_ctx* ctx, int field, void* dst, size_t bytes);

#ifdef __cplusplus
}
#endif
#endif /* SHADOWKV_H */
