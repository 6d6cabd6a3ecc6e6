/*
 * injectscale.h -- C ABI of libinjectscale.so: GPU-resident fact store,
 * cosine top-k retrieval, Chunked RoPE and paged KV injection on one GB300.
 *
 * The operations follow InferScale ("InferScale: GPU-Native KV Injection for
 * Personalized LLM Serving", arXiv 2607.27090): memory facts are encoded
 * offline, their keys captured before the rotary embedding and stored with
 * the raw values and a semantic embedding on the GPU; at serving time the
 * relevant facts are retrieved, composed into one contiguous segment, their
 * keys rotated to the serving positions (Chunked RoPE) and the K/V
 * scatter-copied into a vLLM-style paged KV cache.  The pages give no API;
 * the calls below follow their statement of the problem (store, retrieve,
 * compose, rotate, inject).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every call returns is_status_t and throws nothing.  Host-detectable
 *   errors return before anything is enqueued; is_last_error_message() then
 *   describes the error of the calling thread's last failed call.
 * - Calls taking a cudaStream_t are asynchronous on that stream unless
 *   stated.  Pointers documented "device" must be device (or managed)
 *   memory owned by the caller and stay valid until the stream reaches the
 *   call.  Pointers documented "host" are read before the call returns.
 * - Device-detected errors (bad ids, block tables that do not cover a
 *   position, ...) never trap: the offending write is skipped and a bit of
 *   IS_ST_* is OR-ed into the store's device status word, read (and
 *   cleared) by is_get_status().
 * - A store is used by one stream at a time; calls on one store are not
 *   thread-safe.
 * - Dtypes: K/V in the store and in the cache share one dtype (f32, bf16 or
 *   f16), or the cache is FP8 E4M3 for a bf16 / f16 store (is_cache_desc_t);
 *   embeddings and query embeddings share one dtype (f16 or f32).  Rotation
 *   arithmetic is fp32; rotated keys are rounded to the cache dtype to
 *   nearest even; values are copied bit for bit (FP8: converted like keys).
 */
#ifndef INJECTSCALE_H
#define INJECTSCALE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define IS_ABI_VERSION 1

/* Hard limits (per call). */
#define IS_MAX_K          1024   /* retrieval budget / facts per injected request */
#define IS_MAX_QUERIES    1024   /* queries per retrieval call */
#define IS_MAX_REQUESTS   4096   /* requests per injection call */
#define IS_MAX_HEAD_DIM   512
#define IS_MAX_POSITION   (1 << 24)  /* positions must stay below 2^24 */
#define IS_EMB_TILE       128    /* embedding rows per store tile (one user per tile) */
#define IS_MAX_FACTS_PER_USER (1 << 20)  /* facts of one user (retrieval row index width) */
#define IS_MAX_LAYERS_PER_CALL 128  /* per-layer cache tensors one is_inject_layers call writes */

typedef enum {
  IS_OK = 0,
  IS_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad enum, dtype mismatch */
  IS_ERR_OOM = 2,           /* device allocation failed at store creation */
  IS_ERR_CAPACITY = 3,      /* store arena (facts, tokens, tiles) is full */
  IS_ERR_OUT_OF_RANGE = 4,  /* host-visible index out of range (user, k > max_k, ...) */
  IS_ERR_CUDA = 5,          /* a CUDA runtime call failed */
  IS_ERR_TIMEOUT = 6,       /* a bounded device wait gave up (IS_ST_TIMEOUT latched) */
  IS_ERR_DEVICE = 7,        /* is_get_status found device status bits set */
  IS_ERR_UNSUPPORTED = 8    /* shape outside what the kernels handle */
} is_status_t;

/* Bits of the device status word (see is_get_status). */
#define IS_ST_FACT_RANGE   0x01u  /* fact id < 0 or >= number of stored facts */
#define IS_ST_FACT_USER    0x02u  /* fact id belongs to another user than requested */
#define IS_ST_BLOCK_TABLE  0x04u  /* position / block_size >= max_blocks_per_seq */
#define IS_ST_BLOCK_ID     0x08u  /* block table entry < 0 or >= num_blocks */
#define IS_ST_USER_RANGE   0x10u  /* user id < 0 or >= max_users */
#define IS_ST_POSITION     0x20u  /* seg_start < 0 or seg_start + length > IS_MAX_POSITION */
#define IS_ST_COUNT        0x40u  /* n_ids[r] < 0 or > ids_stride */
#define IS_ST_TIMEOUT      0x80u  /* a bounded device wait gave up */

/* IS_FP8_E4M3 is a paged-cache type only (never a store type): 8-bit floats
 * in the OCP E4M3 format (no infinities, largest finite 448), the 8-bit KV
 * cache of vLLM, the engine InferScale injects into. */
typedef enum { IS_F32 = 0, IS_BF16 = 1, IS_F16 = 2, IS_FP8_E4M3 = 3 } is_dtype_t;

/* Where the store's K/V arena lives (is_store_config_t.kv_placement).
 * InferScale ("Résultats", Scalabilité) offloads the KV store to host DRAM to go past the
 * GPU's memory capacity, at a small cost in time to first token; the retrieval
 * index stays on the GPU.  IS_KV_HOST: the arena is page-locked host memory
 * mapped into the device's address space; the injection kernel reads the
 * selected rows over the CPU-GPU link itself, so no call synchronises with the
 * host and the control flow is unchanged. */
typedef enum { IS_KV_DEVICE = 0, IS_KV_HOST = 1 } is_kv_placement_t;

typedef struct is_store is_store_t;   /* opaque */

/* Store capacity and model KV shape.  Fields set to 0 take the default noted. */
typedef struct {
  int32_t num_layers;        /* L */
  int32_t num_kv_heads;      /* H (KV heads after grouping) */
  int32_t head_dim;          /* D: power of two, 16 <= D <= IS_MAX_HEAD_DIM */
  int32_t emb_dim;           /* E: multiple of 8 */
  int32_t kv_dtype;          /* is_dtype_t of K/V */
  int32_t emb_dtype;         /* is_dtype_t of embeddings: IS_F16 or IS_F32 */
  int64_t max_facts;         /* arena capacity in facts */
  int64_t max_tokens;        /* arena capacity in tokens (sum of fact lengths) */
  int32_t max_users;         /* user ids are 0 .. max_users-1 */
  int32_t max_queries;       /* per retrieval call, <= IS_MAX_QUERIES (0: 64) */
  int32_t max_k;             /* retrieval budget / facts per request, <= IS_MAX_K (0: 256) */
  int32_t max_requests;      /* per injection call, <= IS_MAX_REQUESTS (0: max_queries) */
  int64_t max_facts_per_user;/* sizes the score scratch (0: max_facts), <= IS_MAX_FACTS_PER_USER */
  int32_t kv_placement;      /* is_kv_placement_t (0: IS_KV_DEVICE) */
  int32_t reserved;          /* must be 0 */
} is_store_config_t;

/* Rotary embedding of the model the facts were encoded with. */
typedef struct {
  double theta;              /* base, w_i = theta^(-2i/D) */
  int32_t style;             /* 0 = NeoX half split (i, i+D/2); 1 = interleaved (2i, 2i+1).
                                The kernels take at most 32 16-byte vectors per half head
                                (NeoX) or per head (interleaved): D <= 512 for 16-bit NeoX,
                                D <= 256 for 16-bit interleaved and fp32 NeoX, D <= 128 for
                                fp32 interleaved; larger D returns IS_ERR_UNSUPPORTED */
  int32_t scaling;           /* 0 = none; 1 = Llama-3.1 frequency scaling */
  double factor;             /* Llama-3.1: scale factor (e.g. 8) */
  double low_freq_factor;    /* Llama-3.1: e.g. 1 */
  double high_freq_factor;   /* Llama-3.1: e.g. 4 */
  int32_t original_max_pos;  /* Llama-3.1: original context length (e.g. 8192) */
} is_rope_params_t;

/* vLLM-style paged cache [L][2][num_blocks][block_size][H][D]: for layer l,
 * K at [l][0] and V at [l][1]; logical position p of a sequence lives in
 * physical block block_table[p / block_size], row p % block_size. */
typedef struct {
  int32_t block_size;
  int32_t num_blocks;
  int32_t dtype;             /* is_dtype_t: the store's kv_dtype, or IS_FP8_E4M3 for an
                                IS_BF16 / IS_F16 store (see below) */
  float k_scale;             /* IS_FP8_E4M3 only: the cache holds K / k_scale and */
  float v_scale;             /* V / v_scale; finite and > 0 (vLLM's default is 1.0) */
} is_cache_desc_t;
/* FP8 cache: each rotated key element k (fp32) and value element v is stored
 * as E4M3(x * r) with r = fp32(1 / scale) (the reciprocal rounded once from
 * double; equal to x / scale for power-of-two scales), rounded to nearest
 * even and saturated to +-448.  Element order and layout are those of the
 * other caches with 1-byte elements.  The store keeps its 16-bit K/V; only the
 * cache is 8-bit. */

typedef struct {
  int64_t n_facts, n_tokens;
  int32_t n_tiles, max_user_tiles;
  int64_t max_user_facts;
  int64_t kv_bytes, emb_bytes, scratch_bytes;
  int32_t num_sms;
  int32_t kv_placement;      /* is_kv_placement_t of the arena */
} is_store_info_t;

/* ---- store ------------------------------------------------------------------
 * is_store_create: allocate a store for one model's KV shape on `device`:
 * the token-major K/V arena [max_tokens][L][2][H][D], the embedding tiles,
 * per-fact metadata and all per-call scratch, so that no later call
 * allocates device memory.  InferScale keeps precomputed per-fact KV and a
 * semantic embedding GPU-resident (abstract; "Conception de Système Native
 * au GPU").  With kv_placement = IS_KV_HOST the arena alone is page-locked
 * host memory instead (is_kv_placement_t); everything else stays on the
 * device.  Synchronous.  Errors: IS_ERR_INVALID_ARG (bad config),
 * IS_ERR_UNSUPPORTED (head_dim / row size the kernels do not handle, or a
 * device that cannot map host memory), IS_ERR_OOM, IS_ERR_CUDA.  *out is owned
 * by the caller; free with is_store_destroy. */
is_status_t is_store_create(const is_store_config_t* config, int device, cudaStream_t stream,
                            is_store_t** out);

/* Free every allocation of the store.  Synchronises the device first. */
is_status_t is_store_destroy(is_store_t* store);

/* ---- is_store_add_facts -----------------------------------------------------
 * Add n facts of one user.  Keys are captured before RoPE and values raw
 * (Chunked RoPE, "Stockage Pré-RoPE"); the store deep-copies them.
 *   user            0 <= user < max_users
 *   lengths_host    host int32[n], tokens per fact, each >= 1
 *   k_pre_rope, v   device or host (any UVA pointer), [sum(lengths)][L][H][D]
 *                   in kv_dtype, facts back to back in order
 *   emb             device or host, [n][E] in emb_dtype
 *   fact_ids_out    host int64[n] (may be NULL): ids assigned, consecutive in
 *                   insertion order across the store
 * Facts of one user keep insertion order, which is also ascending id order.
 * Synchronous with respect to the host (returns after the copies finished).
 * Errors: IS_ERR_INVALID_ARG, IS_ERR_OUT_OF_RANGE (user), IS_ERR_CAPACITY
 * (nothing is added), IS_ERR_CUDA. */
is_status_t is_store_add_facts(is_store_t* store, int32_t user, int32_t n,
                               const int32_t* lengths_host, const void* k_pre_rope,
                               const void* v, const void* emb, int64_t* fact_ids_out_host,
                               cudaStream_t stream);

/* Counters and sizes of a store (host struct, filled on return): facts and
 * tokens stored, embedding tiles in use, the largest user's tiles and facts,
 * the arena, embedding and scratch bytes, the SM count and where the arena
 * lives.  Reads host-side state only; never synchronises. */
is_status_t is_store_info(const is_store_t* store, is_store_info_t* out);

/* ---- Context-Window Encoding capture ----------------------------------------
 * InferScale ("Méthodologie", phase 1, "Encodage de la Fenêtre de Contexte")
 * encodes each memory fact together with a window of w preceding conversation
 * turns, so that the stored K/V carry the context that disambiguates the fact,
 * and keeps only the fact's tokens: the window's are dropped.  The encoder is
 * the serving engine's own prefill; these calls take its output one layer at a
 * time, as a layer-wise KV connector hands it over, and store the facts.
 *
 * is_store_capture_begin: opens a capture of n facts of `user`.
 *   window_host, lengths_host  host int32[n]: tokens of each fact's window (>= 0)
 *                              and of the fact (>= 1).  Encoded sequence i is
 *                              [window_i tokens || lengths_i tokens]; the layer
 *                              buffers hold the sequences back to back.
 *   emb                        device or host, [n][E] in emb_dtype
 * The facts' embeddings and metadata are written now but the facts stay
 * invisible to retrieval until is_store_capture_end.  n <= IS_MAX_CAPTURE_FACTS.
 * While a capture is open, is_store_add_facts and a second begin fail with
 * IS_ERR_INVALID_ARG.  Errors otherwise as is_store_add_facts.  Synchronous.
 *
 * is_store_capture_layer: one layer of the encoder's output.
 *   k_pre_rope, v   device (or mapped host) [sum(window_i + lengths_i)][H][D] in
 *                   kv_dtype, 16-byte aligned: keys intercepted before RoPE
 * Each layer is captured exactly once per capture (IS_ERR_INVALID_ARG
 * otherwise).  Asynchronous on stream; the buffers must stay valid until the
 * work on stream has run.
 *
 * is_store_capture_end: publishes the facts (retrievable by the next call) and
 * writes their ids to ids_out (host int64[n], may be NULL).  If a layer was not
 * captured it returns IS_ERR_INVALID_ARG and drops the capture: the store is as
 * before begin.  Synchronous.
 *
 * is_store_capture_abort: drops an open capture (no-op if none). */
#define IS_MAX_CAPTURE_FACTS 65536
is_status_t is_store_capture_begin(is_store_t* store, int32_t user, int32_t n,
                                   const int32_t* window_host, const int32_t* lengths_host,
                                   const void* emb, cudaStream_t stream);
is_status_t is_store_capture_layer(is_store_t* store, int32_t layer, const void* k_pre_rope,
                                   const void* v, cudaStream_t stream);
is_status_t is_store_capture_end(is_store_t* store, int64_t* ids_out, cudaStream_t stream);
is_status_t is_store_capture_abort(is_store_t* store);

/* ---- is_retrieve_topk -------------------------------------------------------
 * For each query q, the cosine similarity of q_emb[q] with every stored
 * embedding of user users[q], then the k best (InferScale retrieves the
 * relevant facts under a budget k: "Problématique", "Conception de Système
 * Native au GPU"; the index it names is not described, so retrieval is exact).
 *   Q               1 <= Q <= max_queries
 *   users           device int32[Q]
 *   q_emb           device [Q][E] in emb_dtype (need not be normalised)
 *   k               1 <= k <= max_k
 *   ids_out         device int64[Q][k]: descending score, ties to the lower
 *                   fact id; rows of a user with fewer than k facts end in -1
 *   scores_out      device float[Q][k]: cosine (fp32), -inf where id is -1
 * A zero-norm embedding or query scores 0.  A bad user id latches
 * IS_ST_USER_RANGE and yields an all -1 row. */
is_status_t is_retrieve_topk(is_store_t* store, int32_t Q, const int32_t* users,
                             const void* q_emb, int32_t k, int64_t* ids_out, float* scores_out,
                             cudaStream_t stream);

/* ---- is_inject --------------------------------------------------------------
 * Compose each request's facts, in the order given, into one contiguous
 * segment starting at seg_start[r]; rotate every stored pre-RoPE key to its
 * serving position p = seg_start[r] + t (token t of the segment) and
 * scatter-copy rotated K and raw V for all layers and KV heads into the
 * paged cache ("Rotation Dynamique", "Injection"; exact by Theorem 6).
 *   R                    1 <= R <= max_requests
 *   fact_ids             device int64[R][ids_stride]; first n_ids[r] used
 *   n_ids                device int32[R], 0 <= n_ids[r] <= ids_stride
 *   ids_stride           1 <= ids_stride <= max_k
 *   users                device int32[R] or NULL: if given, every fact of
 *                        request r must belong to users[r]
 *   seg_start            device int32[R], >= 0
 *   rope                 host, read before return
 *   block_table          device int32[R][max_blocks_per_seq]
 *   cache, kv_cache      host descriptor / device cache [L][2][NB][bs][H][D]
 *   seg_len_out          device int32[R] or NULL: tokens injected per request
 *   slot_mapping_out     device int64[sum seg_len] or NULL: slot of every
 *                        injected token, requests back to back
 * An invalid fact (IS_ST_FACT_RANGE / IS_ST_FACT_USER) contributes no
 * tokens; a position the block table does not map (IS_ST_BLOCK_TABLE,
 * IS_ST_BLOCK_ID) is not written.  Cache elements of other slots are never
 * touched.  Slots of one call must be distinct (two tokens on one slot race). */
is_status_t is_inject(is_store_t* store, int32_t R, const int64_t* fact_ids,
                      const int32_t* n_ids, int32_t ids_stride, const int32_t* users,
                      const int32_t* seg_start, const is_rope_params_t* rope,
                      const int32_t* block_table, int32_t max_blocks_per_seq,
                      const is_cache_desc_t* cache, void* kv_cache, int32_t* seg_len_out,
                      int64_t* slot_mapping_out, cudaStream_t stream);

/* ---- is_inject_layer --------------------------------------------------------
 * is_inject for one layer, into that layer's own cache tensor
 * layer_cache [2][num_blocks][block_size][H][D] (K at [0], V at [1]), so an
 * engine can inject layer l while it works on another layer: InferScale
 * ("Méthodologie") integrates through vLLM's KV-connector interface, which
 * saves and loads KV layer by layer.
 *   fact_ids != NULL   plan the segments (as is_inject) and inject `layer`;
 *   fact_ids == NULL   reuse the segment plan of the store's previous
 *                      is_inject, is_inject_layer(s) or
 *                      is_retrieve_and_inject(_host) call, which must have
 *                      had the same R (n_ids, users and
 *                      ids_stride are then ignored); the plan stays valid
 *                      until the next planning call on the store.
 * seg_start and block_table must be the ones the plan was made with.  A plan
 * made by is_inject or is_inject_layer(s) with seg_len_out != NULL keeps its
 * segment lengths in that array: it must stay allocated and unchanged while
 * the plan is reused.
 * slot_mapping_out (if given) is written again for this call.  Errors as
 * is_inject, plus IS_ERR_OUT_OF_RANGE for a bad layer and
 * IS_ERR_INVALID_ARG when there is no plan of R requests to reuse. */
is_status_t is_inject_layer(is_store_t* store, int32_t layer, int32_t R, const int64_t* fact_ids,
                            const int32_t* n_ids, int32_t ids_stride, const int32_t* users,
                            const int32_t* seg_start, const is_rope_params_t* rope,
                            const int32_t* block_table, int32_t max_blocks_per_seq,
                            const is_cache_desc_t* cache, void* layer_cache, int32_t* seg_len_out,
                            int64_t* slot_mapping_out, cudaStream_t stream);

/* ---- is_inject_layers -------------------------------------------------------
 * is_inject_layer for the layers layer0 .. layer0 + n_layers - 1 in one launch,
 * each into its own cache tensor: layer_caches is a host array of n_layers
 * device pointers, entry i being layer (layer0 + i)'s
 * [2][num_blocks][block_size][H][D] tensor, at any addresses (16-byte
 * aligned).  This is how an engine that keeps one KV tensor per layer (vLLM,
 * whose KV-connector interface InferScale integrates through, "Méthodologie")
 * injects a group of layers, or the whole model (layer0 = 0, n_layers = L),
 * at the cost of one launch.  1 <= n_layers <= IS_MAX_LAYERS_PER_CALL and
 * layer0 + n_layers <= the store's layers (IS_ERR_OUT_OF_RANGE otherwise).
 * Planning (fact_ids != NULL) and plan reuse (fact_ids == NULL), the other
 * arguments and the errors are as is_inject_layer. */
is_status_t is_inject_layers(is_store_t* store, int32_t layer0, int32_t n_layers, int32_t R,
                             const int64_t* fact_ids, const int32_t* n_ids, int32_t ids_stride,
                             const int32_t* users, const int32_t* seg_start, const is_rope_params_t* rope,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const is_cache_desc_t* cache, void* const* layer_caches, int32_t* seg_len_out,
                             int64_t* slot_mapping_out, cudaStream_t stream);

/* ---- is_retrieve_and_inject -------------------------------------------------
 * is_retrieve_topk followed by is_inject of each query's k facts in
 * descending-score order, with no host synchronisation between the stages
 * (the ids never leave the device).  Arguments as in those calls; ids_out,
 * scores_out (device [Q][k]), seg_len_out (device int32[Q]) and
 * slot_mapping_out may each be NULL.  The store keeps its own copy of the
 * segment plan, so a later layer call may reuse it whatever becomes of these
 * arrays. */
is_status_t is_retrieve_and_inject(is_store_t* store, int32_t Q, const int32_t* users,
                                   const void* q_emb, int32_t k, const int32_t* seg_start,
                                   const is_rope_params_t* rope, const int32_t* block_table,
                                   int32_t max_blocks_per_seq, const is_cache_desc_t* cache,
                                   void* kv_cache, int64_t* ids_out, float* scores_out,
                                   int32_t* seg_len_out, int64_t* slot_mapping_out,
                                   cudaStream_t stream);

/* ---- is_retrieve_and_inject_host --------------------------------------------
 * is_retrieve_and_inject for a caller whose per-call inputs and outputs are in
 * host memory (any host memory: the library stages them through its own
 * page-locked buffer, mapped into the device's address space).  users
 * (int32[Q]), q_emb ([Q][E] in emb_dtype), seg_start (int32[Q]) and
 * block_table (int32[Q][max_blocks_per_seq]) are copied into that buffer,
 * where the kernels read them over the host link; the path runs on `stream`;
 * the kernels write ids_out (int64[Q][k]), scores_out (float[Q][k]) and
 * seg_len_out (int32[Q]) into the buffer, and the call copies them to the
 * caller's host arrays, which may each be NULL.  The store and the paged
 * cache stay on the device (kv_cache is a device pointer).  Synchronous:
 * returns once the outputs are in host memory and every cache write of the
 * call is complete; the calling thread spins meanwhile.  With the inputs in
 * the mapped buffer it polls a word of mapped host memory that the inject
 * kernel's last CTA sets when the work is done, so the kernel may still be
 * retiring when the call returns: work on `stream` is ordered after it as
 * usual, and work on another stream that must follow it should be ordered
 * after `stream` (an event), not after the return alone.  With the inputs
 * copied, it polls the stream.  The staging buffer belongs to the
 * store; a call that needs more than the last one had grows it (a
 * synchronisation and an allocation; IS_ERR_OOM if that fails,
 * IS_ERR_UNSUPPORTED if the device cannot address it at its host address).
 * Errors as is_retrieve_and_inject, detected before anything is enqueued
 * except device-side ones (read them with is_get_status). */
is_status_t is_retrieve_and_inject_host(is_store_t* store, int32_t Q, const int32_t* users_host,
                                        const void* q_emb_host, int32_t k, const int32_t* seg_start_host,
                                        const is_rope_params_t* rope, const int32_t* block_table_host,
                                        int32_t max_blocks_per_seq, const is_cache_desc_t* cache,
                                        void* kv_cache, int64_t* ids_out_host, float* scores_out_host,
                                        int32_t* seg_len_out_host, cudaStream_t stream);

/* ---- prepared host calls ------------------------------------------------------
 * A serving loop that calls is_retrieve_and_inject_host on the same host
 * buffers every time (their contents change, their addresses do not) can bind
 * them once.  is_host_call_prepare checks and keeps every argument of the call,
 * with copies of *rope and *cache.  is_host_call_run(call) then performs the
 * call exactly as is_retrieve_and_inject_host would with those arguments,
 * reading the buffers' current contents.  A run takes one argument, so a
 * caller going through a foreign-function layer no longer pays to convert
 * fifteen arguments on every request.  The bound buffers, the store, kv_cache
 * and the stream must outlive the call object, and is_host_call_destroy frees
 * it (the store is not touched).  Errors: prepare returns IS_ERR_INVALID_ARG
 * or IS_ERR_OUT_OF_RANGE for the argument checks of is_retrieve_and_inject_host
 * that need no device, and IS_ERR_OOM; run returns what that call returns. */
typedef struct is_host_call is_host_call_t;
is_status_t is_host_call_prepare(is_store_t* store, int32_t Q, const int32_t* users_host,
                                 const void* q_emb_host, int32_t k, const int32_t* seg_start_host,
                                 const is_rope_params_t* rope, const int32_t* block_table_host,
                                 int32_t max_blocks_per_seq, const is_cache_desc_t* cache, void* kv_cache,
                                 int64_t* ids_out_host, float* scores_out_host, int32_t* seg_len_out_host,
                                 cudaStream_t stream, is_host_call_t** call_out);
is_status_t is_host_call_run(is_host_call_t* call);
is_status_t is_host_call_destroy(is_host_call_t* call);

/* ---- is_inject_noalloc ------------------------------------------------------
 * The paper has no counterpart to this call; it exists for callers that
 * cannot allocate device memory: code whose device memory is all owned by
 * another allocator (a serving engine that reserves HBM for its own pools at
 * start-up) or that runs where cudaMalloc is not allowed.  Such a caller
 * keeps facts in its own buffers and still wants the gather + Chunked RoPE +
 * paged scatter.  This call creates no store and allocates nothing: the
 * per-request segment plan lives in a static device array of the library
 * (about 269 KB, held on every device that loads the library until exit).
 *   kv_arena             device, token-major [arena_tokens][L][2][H][D] in kv_dtype
 *                        (per token and layer: K row then V row, K before RoPE)
 *   arena_tokens         tokens in kv_arena, >= 1
 *   fact_tok, fact_len   device int64[n_facts] first arena token, int32[n_facts]
 *                        length.  They are checked on the device: a fact whose
 *                        length is outside [1, max_fact_len] or whose tokens leave
 *                        [0, arena_tokens) latches IS_ST_FACT_RANGE and is left
 *                        out of its segment (length 0), like an id outside
 *                        [0, n_facts); nothing is read for it
 *   R                    1 <= R <= IS_NOALLOC_MAX_REQUESTS
 *   ids_stride           1 <= ids_stride <= IS_NOALLOC_MAX_FACTS
 *   status_out           device uint32, caller-owned: IS_ST_* bits are OR-ed in
 *                        (the caller clears it)
 *   cache                cache->dtype must equal kv_dtype (no FP8 cache here:
 *                        IS_ERR_INVALID_ARG)
 * Other arguments as in is_inject (no user check).  Sizes beyond the limits
 * return IS_ERR_UNSUPPORTED before anything is enqueued.  The first call on a
 * device looks up the static array's device address (once per device, under
 * a lock).  Every call uses
 * the same static array: its planning kernel writes the plan entries and
 * zeroes the work counters its injection kernel then uses, so a call depends
 * on nothing an earlier call left there, but two calls whose kernels overlap
 * on the GPU (different streams, no ordering between them) race on it. */
#define IS_NOALLOC_MAX_REQUESTS 256
#define IS_NOALLOC_MAX_FACTS    256
is_status_t is_inject_noalloc(const void* kv_arena, int64_t arena_tokens,
                              const int64_t* fact_tok, const int32_t* fact_len, int64_t n_facts,
                              int32_t max_fact_len, int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                              int32_t kv_dtype, int32_t R, const int64_t* fact_ids,
                              const int32_t* n_ids, int32_t ids_stride, const int32_t* seg_start,
                              const is_rope_params_t* rope, const int32_t* block_table,
                              int32_t max_blocks_per_seq, const is_cache_desc_t* cache,
                              void* kv_cache, int32_t* seg_len_out, int64_t* slot_mapping_out,
                              uint32_t* status_out, cudaStream_t stream);

/* ---- is_set_retrieval_mode -----------------------------------------------------
 * How the similarity is computed.  IS_RETRIEVAL_PER_QUERY: one launch in
 * which each query's CTAs stream its user's embedding tiles and the last CTA
 * of the query selects its top-k (best when each user has one query in the
 * call).  IS_RETRIEVAL_BATCHED: queries are grouped by user (up to 64 per
 * group) and each (group, 128-row tile) is one tensor-core contraction
 * (tcgen05, fp16 operands, fp32 accumulation), then one top-k CTA per query
 * (best when a user has many queries in the call: the tile is read once for
 * all of them).  IS_RETRIEVAL_AUTO (default): batched when Q >= 32 and the
 * largest user holds >= 1024 facts.  Results are the same up to the order of
 * fp32 accumulation.  Errors: IS_ERR_UNSUPPORTED for the batched mode with
 * fp32 embeddings. */
#define IS_RETRIEVAL_AUTO      0
#define IS_RETRIEVAL_PER_QUERY 1
#define IS_RETRIEVAL_BATCHED   2
is_status_t is_set_retrieval_mode(is_store_t* store, int32_t mode);

/* ---- is_set_wait_budget ---------------------------------------------------------
 * Every wait inside the store's kernels is bounded: a wait for data that does
 * not arrive gives up, latches IS_ST_TIMEOUT, lets the copies it already
 * started land and ends its kernel, so a stalled GPU memory system cannot
 * hang the caller, and is_get_status then returns IS_ERR_TIMEOUT.  This sets
 * the budget, in nanoseconds, of each wait in the injection pipeline and in
 * the batched (tensor-core) similarity: 0 <= budget_ns <= 2 s, default 2 s.
 * With 0 a wait looks once and gives up at once if its data has not landed,
 * which is how the tests exercise the time-out path.  The waits that let
 * copies in flight land before a kernel ends always keep 2 s.  After a time-out
 * the call's outputs are undefined, except that every cache row is either
 * left as it was or holds what the call would have written there.
 * Errors: IS_ERR_INVALID_ARG for a budget outside that range. */
is_status_t is_set_wait_budget(is_store_t* store, int64_t budget_ns);

/* ---- status / diagnostics ---------------------------------------------------
 * is_get_status: synchronise `stream`, read the device status word into
 * *bits_out and clear it.  Returns IS_ERR_DEVICE if any bit was set,
 * IS_ERR_TIMEOUT if IS_ST_TIMEOUT was, IS_ERR_CUDA if the stream reported an
 * error. */
is_status_t is_get_status(is_store_t* store, cudaStream_t stream, uint32_t* bits_out);

/* Message of the calling thread's last failed call ("" if none). */
const char* is_last_error_message(void);
const char* is_status_string(is_status_t status);

/* The rotation frequencies w_i (i < head_dim/2) the kernels use, in fp64,
 * into host double[head_dim/2].  Plain: theta^(-2i/D); Llama-3.1 scaling:
 * the published Llama 3.1 rule (wavelength bands original_max_pos /
 * high_freq_factor and original_max_pos / low_freq_factor). */
is_status_t is_rope_frequencies(const is_rope_params_t* rope, int32_t head_dim,
                                double* inv_freq_out_host);

/* ---- stage timing -------------------------------------------------------------
 * When enabled, every kernel launch of the store is bracketed by CUDA events
 * on its stream.  is_get_timing synchronises the device and returns, for a
 * stage, the summed device time (ms) and the number of launches since the
 * last reset.  Stages: IS_STAGE_SIMILARITY, IS_STAGE_TOPK, IS_STAGE_PLAN,
 * IS_STAGE_INJECT. */
#define IS_STAGE_SIMILARITY 0
#define IS_STAGE_TOPK       1
#define IS_STAGE_PLAN       2
#define IS_STAGE_INJECT     3
#define IS_NUM_STAGES       4
is_status_t is_set_timing(is_store_t* store, int32_t enable);
is_status_t is_get_timing(is_store_t* store, int32_t stage, double* total_ms, int64_t* launches);
is_status_t is_reset_timing(is_store_t* store);

#ifdef __cplusplus
}
#endif

#endif /* INJECTSCALE_H */
