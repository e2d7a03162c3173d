/*
 * cacheblend.h -- C ABI of the GB300 CacheBlend blend-step library (libcacheblend.so).
 *
 * The library computes the per-request blend step of CacheBlend for non-prefix KV
 * reuse, as described on the CacheBlend deep-dive page ("CacheBlend 完全拆解:RAG 多段
 * KV 缓存拼接,为什么还要重算一小部分 token"):
 *   - precomputed chunk caches are placed at new offsets and their K re-rotated
 *     (section "位置恢复、KV 存储与加载流水线", re-RoPE identity k' = R_{n-p} k_p = R_n k);
 *   - the check layer is computed for every token and each token's KV deviation
 *     ||KV_new[j] - KV_pre[j]||^2 ranks the tokens (section "核心思想", Δkv formula);
 *   - the top-r fraction (HKVD tokens) plus the query are recomputed in every later
 *     layer against the blended K/V (section "选 token", Figure 5 and Figure 9).
 *
 * Conventions for every entry point:
 *   - Pointers documented as "device" must be CUDA device (or managed) memory on the
 *     current device; "host" pointers are ordinary host memory read during the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  All
 *     GPU work is enqueued on it; calls return without synchronising the host.
 *   - Arguments are validated on the host before anything is enqueued; on any error
 *     nothing is enqueued, the return code is negative and cb_last_error() describes it.
 *   - No entry point aborts or throws; CUDA launch failures map to CB_ERR_CUDA.
 *   - Calls on one model handle must not run concurrently (they share its workspace).
 */
#ifndef CACHEBLEND_H
#define CACHEBLEND_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CB_OK = 0,
    CB_ERR_INVALID_ARG = -1,   /* a pointer, size, layout or ratio is out of range */
    CB_ERR_UNSUPPORTED = -2,   /* valid but not supported by this library (e.g. head_dim) */
    CB_ERR_OOM = -3,           /* workspace allocation failed at model creation */
    CB_ERR_CUDA = -4,          /* a CUDA call or kernel launch failed */
    CB_ERR_INTERNAL = -5
} cb_status;

typedef enum { CB_F32 = 0, CB_BF16 = 1 } cb_dtype;

/* Llama-style pre-norm decoder shape.  Supported: head_dim in {64, 128},
 * n_heads % n_kv_heads == 0, n_layers >= 2, d_model and ffn_hidden multiples of 64, d_model <= 8192. */
typedef struct {
    int32_t n_layers;
    int32_t d_model;
    int32_t n_heads;         /* query heads */
    int32_t n_kv_heads;      /* K/V heads (GQA: q-head h reads KV head h / (n_heads/n_kv_heads)) */
    int32_t head_dim;
    int32_t ffn_hidden;      /* SwiGLU hidden width */
    int32_t vocab;
    double rope_theta;       /* RoPE base: dims (2i, 2i+1) rotate by angle pos * theta^(-2i/head_dim) */
    float rms_eps;           /* RMSNorm epsilon */
    int32_t dtype;           /* cb_dtype of weights, K/V caches and tensor-core operands */
    int32_t max_tokens;      /* largest n_tokens (context + query) a blend may use; sizes the workspace */
    int32_t max_chunks;      /* largest n_chunks a call may pass (<= CB_MAX_CHUNKS) */
    int32_t precision;       /* cb_precision: how bf16 models feed activations to the tensor cores */
} cb_config;

/* Activation precision of bf16 models (fp32 models compute in fp32 throughout).
 *   CB_PREC_SPLIT: every activation operand of a projection is carried as two bf16 numbers
 *                  (hi + lo, about 16 significant bits) and multiplied with both; the weights are
 *                  exact bf16 values, so the products carry fp32-like activation precision.  Two
 *                  MMAs per k-step.  Default.
 *   CB_PREC_BF16:  activations rounded once to bf16 (one MMA per k-step; faster, and over a deep
 *                  stack the K/V and logits drift by a few bf16 ulps from an exact computation). */
typedef enum { CB_PREC_SPLIT = 0, CB_PREC_BF16 = 1 } cb_precision;

#define CB_MAX_CHUNKS 1024

/* Weights, borrowed (not copied): they must stay valid until cb_model_destroy.
 * Every matrix is row-major [out_features][in_features] in cfg.dtype ("nn.Linear" layout):
 *   embed, lm_head [vocab][d_model]; wq [n_heads*head_dim][d_model];
 *   wk, wv [n_kv_heads*head_dim][d_model]; wo [d_model][n_heads*head_dim];
 *   w_gate, w_up [ffn_hidden][d_model]; w_down [d_model][ffn_hidden];
 *   attn_norm, mlp_norm, final_norm [d_model] (RMSNorm gains).
 * The per-layer members are HOST arrays of n_layers DEVICE pointers; the arrays are
 * copied at creation.  Device pointers must be 16-byte aligned. */
typedef struct {
    const void* embed;
    const void* final_norm;
    const void* lm_head;
    const void* const* attn_norm;
    const void* const* wq;
    const void* const* wk;
    const void* const* wv;
    const void* const* wo;
    const void* const* mlp_norm;
    const void* const* w_gate;
    const void* const* w_up;
    const void* const* w_down;
} cb_weights;

/* One placed chunk: its cache rows were computed at positions src_pos .. src_pos+len-1
 * (the chunk's old start) and now sit at dst_pos .. dst_pos+len-1 (its current start).
 * A negative src_pos means "position unknown" and is rejected: rotating from a wrong
 * source position would silently produce wrong keys. */
typedef struct {
    int32_t src_pos;
    int32_t dst_pos;
    int32_t len;
} cb_chunk;

/* Host-side accounting of one blend (filled when `stats` is non-NULL). */
typedef struct {
    int32_t n_tokens;        /* N = n_ctx + n_query */
    int32_t n_ctx;           /* context rows (sum of chunk lengths) */
    int32_t n_selected;      /* k = HKVD rows chosen at the check layer */
    int32_t n_recompute;     /* M = k + n_query rows recomputed in layers >= 1 */
    int32_t kernel_launches; /* kernels enqueued by this call */
    int32_t reserved;
    double gemm_flops;       /* algorithmic FLOPs of all projections */
    double attn_flops;       /* algorithmic FLOPs of attention (causal key counts) */
    double kv_bytes_moved;   /* algorithmic bytes of re-RoPE/placement, deviation and K/V scatter */
} cb_stats;

typedef struct cb_model cb_model;

/* Create a model handle: copies the config and the weight pointer tables, allocates the
 * device workspace for cfg.max_tokens rows and the RoPE tables (computed in float64 on
 * the host, stored as float32) on the current device.  Synchronous.
 * Errors: CB_ERR_INVALID_ARG (bad shape / null pointer), CB_ERR_UNSUPPORTED,
 * CB_ERR_OOM (workspace), CB_ERR_CUDA. */
cb_status cb_model_create(const cb_config* cfg, const cb_weights* weights, cb_model** out);

/* Free the workspace (synchronises the device).  NULL is accepted. */
cb_status cb_model_destroy(cb_model* model);

/* In-place re-RoPE of a chunk-cache buffer (re-RoPE identity, section
 * "位置恢复、KV 存储与加载流水线"): for every chunk c and every layer, the K rows
 * dst_pos_c .. dst_pos_c+len_c-1 are rotated by R_{dst_pos_c - src_pos_c}; V is untouched.
 *   kv      device, [n_layers][2][n_rows][n_kv_heads][head_dim] in cfg.dtype (2 = K, V)
 *   chunks  host, n_chunks entries; they must tile [0, sum len) in dst order and
 *           sum len <= n_rows.
 * Async on `stream`. */
cb_status cb_rerope(cb_model* model, void* kv, int64_t n_rows, const cb_chunk* chunks, int32_t n_chunks,
                    void* stream);

/* One blend (sections "核心思想" and "选 token"; Figures 5 and 9):
 *   tokens       device int32 [n_tokens]: the context tokens in placed order, then the query.
 *   cached_kv    device [n_layers][2][n_ctx][n_kv_heads][head_dim] (cfg.dtype): the chunk
 *                caches concatenated in placed order, K still rotated at each chunk's src_pos.
 *                May be NULL when n_chunks == 0.
 *   chunks       host, n_chunks entries tiling [0, n_ctx) in dst order (n_ctx = sum len).
 *                n_chunks == 0 makes the call a plain causal prefill of `tokens`.
 *   ratio        fraction r in [0, 1]; k = ceil(r * n_ctx) context rows are recomputed.
 *   out_kv       device [n_layers][2][n_tokens][n_kv_heads][head_dim] (cfg.dtype): the blended
 *                K/V.  out_kv == cached_kv is allowed (in-place blend): cached_kv is then read with
 *                out_kv's layout, the chunk caches sitting in rows 0..n_ctx-1 of every (layer, K/V)
 *                block.  Any other overlap between the two buffers is rejected.
 *   out_logits   device float32 [vocab]: logits of the last token.
 *   out_selected device int32 [k] or NULL: the chosen context rows, ascending.
 *   out_dev      device float32 [n_ctx] or NULL: every context row's deviation at the check layer.
 *   stats        host or NULL: accounting of the call.
 * Requires 0 < n_tokens <= max_tokens and n_tokens > n_ctx (at least one query token).
 * Async on `stream`; no device memory is allocated. */
cb_status cb_blend(cb_model* model, const int32_t* tokens, int32_t n_tokens, const void* cached_kv,
                   const cb_chunk* chunks, int32_t n_chunks, double ratio, void* out_kv, float* out_logits,
                   int32_t* out_selected, float* out_dev, cb_stats* stats, void* stream);

/* One blend whose recomputed set is given by the caller (the page's interface passes the HKVD indices
 * between layers and switches the comparison off with check_flag; section "读源码时的几个观察点"): the
 * check layer compares nothing and every later layer recomputes exactly the k given context rows and the
 * query.  Everything else is cb_blend's.
 *   hkvd  device int32 [k]: context rows, strictly ascending, in [0, n_ctx).  A row out of range or out of
 *         order is replaced by a valid one and recorded as CB_STATUS_BAD_ROW (read with cb_model_status).
 * With the set cb_blend chose for the same inputs the result is bit-identical to cb_blend's.
 * Errors: those of cb_blend, plus CB_ERR_INVALID_ARG for k outside [0, n_ctx] or a NULL hkvd with k > 0. */
cb_status cb_blend_hkvd(cb_model* model, const int32_t* tokens, int32_t n_tokens, const void* cached_kv,
                        const cb_chunk* chunks, int32_t n_chunks, const int32_t* hkvd, int32_t k, void* out_kv,
                        float* out_logits, cb_stats* stats, void* stream);

/* One blend with gradual filtering (section "核心思想", the layer-by-layer funnel of Figure 9): the set
 * of context rows recomputed shrinks from layer to layer, each set nested in the previous one.
 *   ratios      host, n_ratios = n_layers - 1 entries: ratios[l - 1] is r_l of layer l, and
 *               k_l = ceil(r_l * n_ctx - 1e-9) context rows carry an updated hidden state out of layer l.
 *               The counts must not grow (k_l <= k_{l-1}); equal counts keep the set unchanged.
 *   Layer 1 is the check layer of cb_blend (every row compared, the top k_1 kept).  A later layer l with
 *   k_l < k_{l-1} computes fresh K/V for the k_{l-1} candidates (and the query), ranks the candidates by
 *   their deviation against this layer's re-RoPE'd cache, keeps the top k_l (ties to the lower
 *   position), stores the kept rows' and the query's fresh K/V, and runs attention, O and MLP for them
 *   only.  A candidate that drops out keeps its cached K/V from that layer on.
 *   out_selected device int32 or NULL: the check layer's set (k_1 rows, ascending), followed by the set
 *                of every shrinking layer in layer order (k_l rows each, ascending).
 *   out_dev      device float32 or NULL: the check layer's n_ctx deviations, followed by every
 *                shrinking layer's k_{l-1} candidate deviations (candidates in ascending position).
 *   All other arguments, the validation and the asynchrony are those of cb_blend; a constant schedule
 *   gives exactly cb_blend's result.  A growing schedule or n_ratios != n_layers - 1 -> CB_ERR_INVALID_ARG. */
cb_status cb_blend_gradual(cb_model* model, const int32_t* tokens, int32_t n_tokens, const void* cached_kv,
                           const cb_chunk* chunks, int32_t n_chunks, const double* ratios, int32_t n_ratios,
                           void* out_kv, float* out_logits, int32_t* out_selected, float* out_dev, cb_stats* stats,
                           void* stream);

/* Host side of the layer-wise load pipeline (section "位置恢复、KV 存储与加载流水线", Figure 11: while
 * layer i is recomputed, layer i+1's KV is fetched; before each layer a synchronisation makes sure its
 * data has arrived). */
typedef struct {
    const void* cached_kv_host;  /* host [n_layers][2][n_ctx][n_kv_heads][head_dim] (cfg.dtype): the chunk caches
                                    in placed order, K still rotated at each chunk's src_pos.  Page-locked
                                    (pinned) memory, or the copies do not overlap the compute. */
    void* out_kv_host;           /* host [n_layers][2][n_tokens][n_kv_heads][head_dim] or NULL: each layer's
                                    blended K/V, copied back as soon as that layer's recomputed rows are stored
                                    (pinned, as above) */
    void* copy_stream;           /* cudaStream_t of the host-to-device copies; not the compute stream */
    void* copy_back_stream;      /* cudaStream_t of the device-to-host copies, or NULL to use copy_stream */
} cb_layer_io;

/* A blend whose chunk caches stream in from host memory layer by layer (the loading pipeline of
 * section "位置恢复、KV 存储与加载流水线").  Every layer's cache rows are copied into out_kv (rows
 * 0..n_ctx-1 of its K and V blocks) on io->copy_stream, in layer order, each followed by an event; the
 * compute stream waits for layer l's event, re-RoPEs layer l in place and only then computes it, so the
 * copy of layer l+1 overlaps the recompute of layer l.  With io->out_kv_host set, layer l's blended
 * K/V (all n_tokens rows) is copied back on io->copy_back_stream once its recomputed rows are stored.
 *   ratios, n_ratios, out_selected, out_dev: as for cb_blend_gradual (a constant schedule is cb_blend).
 *   tokens, chunks, out_kv, out_logits, stats: as for cb_blend; out_kv is a device buffer of n_tokens rows.
 * The call forks the copy streams off `stream` and joins them back: when `stream` has completed, every
 * copy has too.  Errors: those of cb_blend_gradual, plus CB_ERR_INVALID_ARG for a missing copy stream,
 * a copy stream equal to `stream`, or chunks without a host cache. */
cb_status cb_blend_streamed(cb_model* model, const int32_t* tokens, int32_t n_tokens, const cb_layer_io* io,
                            const cb_chunk* chunks, int32_t n_chunks, const double* ratios, int32_t n_ratios,
                            void* out_kv, float* out_logits, int32_t* out_selected, float* out_dev, cb_stats* stats,
                            void* stream);

/* Paged K/V (section "和前缀缓存、PagedAttention 的分工": find each chunk's physical blocks, assemble the
 * request's block table, write the recomputed K/V back to the right physical place, copy-on-write for
 * shared blocks, writes split at page boundaries).
 * Pool layout: device [n_layers][2][n_pages * page_size][n_kv_heads][head_dim] (cfg.dtype): page p holds
 * rows p*page_size .. p*page_size+page_size-1 of every (layer, K|V) block.  Logical row j of a block table
 * t is pool row t[j / page_size] * page_size + j % page_size.  Tables are DEVICE int32 arrays; a page id
 * outside [0, n_pages) is recorded as CB_STATUS_BAD_ROW and its rows are skipped. */
typedef struct {
    void* pool;                  /* device pool, 16-byte aligned */
    int64_t n_pages;
    int32_t page_size;           /* rows per page: a power of two >= 16 */
    const int32_t* src_table;    /* device, ceil(rows / page_size) entries: where the rows are read from */
    const int32_t* dst_table;    /* device, ceil(rows / page_size) entries: where the rows are written to */
} cb_paged_kv;

/* A blend whose chunk caches and blended K/V live in a paged pool.  src_table maps the n_ctx context rows
 * (the chunk caches in placed order, K still rotated at each chunk's src_pos) to their pages; dst_table
 * maps all n_tokens rows of the blended K/V to the pages that receive it.  A block whose page is shared
 * with other requests gets a fresh page in dst_table (copy-on-write: the shared page is only read); a
 * private block may use the same page in both tables (in place).  The chunk caches are read from their
 * pages, re-rotated and placed into work_kv in one pass, the blend runs there, and every row is then
 * written to its destination page.
 *   work_kv      device [n_layers][2][n_tokens][n_kv_heads][head_dim]: the contiguous working copy (the
 *                caller's memory; holds the blended K/V on return as well).
 *   ratios, n_ratios, out_selected, out_dev: as for cb_blend_gradual (a constant schedule is cb_blend).
 *   tokens, chunks, out_logits, stats: as for cb_blend.  Async on `stream`; no allocation.
 * Errors: those of cb_blend_gradual, plus CB_ERR_INVALID_ARG for a bad pool, page size or missing table. */
cb_status cb_blend_paged(cb_model* model, const int32_t* tokens, int32_t n_tokens, const cb_paged_kv* paged,
                         const cb_chunk* chunks, int32_t n_chunks, const double* ratios, int32_t n_ratios,
                         void* work_kv, float* out_logits, int32_t* out_selected, float* out_dev, cb_stats* stats,
                         void* stream);

/* Paged <-> contiguous conversion of n_rows rows of every (layer, K|V) block, in the model's layout:
 * gather reads the pool through src_table into out_kv [n_layers][2][n_rows][n_kv_heads][head_dim];
 * scatter writes kv (same layout) into the pool through dst_table.  Async on `stream`. */
cb_status cb_kv_gather_pages(cb_model* model, const cb_paged_kv* paged, int32_t n_rows, void* out_kv, void* stream);
cb_status cb_kv_scatter_pages(cb_model* model, const void* kv, int32_t n_rows, const cb_paged_kv* paged, void* stream);

/* Host-side page bookkeeping for a pool (reference counts, allocation, copy-on-write planning); host memory
 * only, no CUDA calls.  A page is free at count 0.
 *   cb_pages_create   n_pages pages, all free.
 *   cb_pages_alloc    n free pages (lowest ids first), each with count 1, into ids; CB_ERR_OOM (nothing
 *                     taken) when fewer are free.
 *   cb_pages_retain   count += 1 for each id (another request shares the page).
 *   cb_pages_release  count -= 1 for each id (a page reaching 0 is free again).
 *   cb_pages_plan_write  for a request about to write its blocks table[0..n): a block whose page is shared
 *                     (count > 1) gets a fresh page in dst (its count 1) and drops its reference to the
 *                     shared one; a private block keeps its page.  Returns the number of copy-on-write
 *                     pages, or CB_ERR_OOM with nothing changed.
 *   cb_pages_count    the reference count of a page (-1 for a bad id). */
typedef struct cb_pages cb_pages;
cb_status cb_pages_create(int64_t n_pages, cb_pages** out);
cb_status cb_pages_destroy(cb_pages* pages);
cb_status cb_pages_alloc(cb_pages* pages, int32_t n, int32_t* ids);
cb_status cb_pages_retain(cb_pages* pages, const int32_t* ids, int32_t n);
cb_status cb_pages_release(cb_pages* pages, const int32_t* ids, int32_t n);
int32_t cb_pages_plan_write(cb_pages* pages, const int32_t* table, int32_t n, int32_t* dst);
int32_t cb_pages_count(const cb_pages* pages, int32_t id);
int64_t cb_pages_free(const cb_pages* pages);

/* Fragment lookup on the GPU (LMCache coordinator blend-index page, sections "四、数据结构与召回" and
 * "六、HTTP 接口"): which indexed chunks a request's tokens contain and where, i.e. the (src_pos, dst_pos)
 * chunk layout of a blend.
 * cb_index_create builds an immutable index on the host and copies it to the current device (it allocates;
 * rebuild it to change the indexed set).  Chunk i has chunk_size tokens tokens[i*chunk_size ..], an
 * occupant id occ_ids[i] (the caller's name for the stored chunk), the position old_st[i] it was stored
 * at, and a namespace ns[i].  A chunk with old_st < 0 (stored position unknown) is not indexed.  A
 * chunk's fingerprint is Horner's rule over its tokens (as unsigned 32-bit values) modulo 2^64 with base
 * 0x9E3779B97F4A7C15; a fingerprint names the first content indexed under it, and a different content
 * with the same fingerprint is not indexed.  Chunks with identical content are occupants of one content,
 * kept in the order given.  max_tokens bounds the requests that cb_index_match accepts.
 * cb_index_match probes the request's windows at positions 0, s, 2s, ... (s = probe_stride); a window
 * whose fingerprint, content and tokens match a content with an occupant in namespace `ns` is verified.
 * The t-th verified window of a content (in position order) takes that content's t-th occupant in `ns`:
 * each occupant matches at most once, at its first place.  Matches are written ascending by position as
 * int32 triples (occupant id, old_st, cur_st) into out (device, max_out triples); with leftmost_greedy a
 * match overlapping an earlier kept one is dropped.  *out_count (device int32) receives the number of
 * matches (which may exceed max_out: only the first max_out are written).  Async on `stream`; no
 * allocation.  Calls on one index must not overlap (they share its scratch buffers).
 * cb_index_size: what = 0 contents, 1 occupants, 2 indexed chunks, 3 chunk_size. */
typedef struct cb_index cb_index;
cb_status cb_index_create(int32_t chunk_size, const uint32_t* tokens, const int32_t* occ_ids, const int32_t* old_st,
                          const int32_t* ns, int32_t n_chunks, int32_t max_tokens, cb_index** out);
cb_status cb_index_destroy(cb_index* index);
int32_t cb_index_size(const cb_index* index, int32_t what);
cb_status cb_index_match(cb_index* index, const int32_t* tokens, int32_t n_tokens, int32_t ns, int32_t probe_stride,
                         int32_t leftmost_greedy, int32_t* out, int32_t max_out, int32_t* out_count, void* stream);

/* Device status bits recorded by the kernels instead of trapping (cumulative since creation). */
#define CB_STATUS_BAD_TOKEN    1u  /* a token id outside [0, vocab) was read; its embedding was zeroed */
#define CB_STATUS_WAIT_TIMEOUT 2u  /* a bounded barrier wait in a tensor-core kernel gave up (~2 s); the
                                      kernel unwound and its outputs are invalid */
#define CB_STATUS_BAD_ROW      4u  /* a row index outside its buffer was seen and skipped */

/* Synchronises the device and returns the status bits in *bits; clear != 0 resets them.
 * Errors: CB_ERR_INVALID_ARG, CB_ERR_CUDA. */
cb_status cb_model_status(cb_model* model, uint32_t* bits, int32_t clear);

/* Synchronises and copies 16 diagnostic words: words[0] = the status bits; when a bounded wait gave
 * up, words[1] = 0xA77E and words[2..7] = {barrier code, parity, counter, block, warp, work unit} of
 * the first one (cleared with the status by cb_model_status(..., clear = 1)). */
cb_status cb_model_diag(cb_model* model, uint32_t* words);

/* Per-kernel-class timing of later cb_blend / cb_rerope calls on this model.  While enabled, each
 * launch is bracketed by CUDA events recorded on the call's stream (this serialises nothing that was
 * not already serial on that stream, but adds event records between kernels).  Classes: "rerope",
 * "embed", "rmsnorm", "gemm_q", "gemm_kv", "gemm_qkv", "gemm_o", "gemm_gateup", "gemm_down",
 * "attention", "deviation", "topk", "gather", "logits", "delta_table", "refilter", "pages". */
typedef struct {
    char name[24];
    int32_t launches;        /* launches recorded since the last read */
    double ms;               /* summed device time of those launches (CUDA events) */
    double flops;            /* summed algorithmic FLOPs (matrix and attention classes) */
    double bytes;            /* summed algorithmic HBM bytes (memory-bound classes; weights for GEMMs) */
} cb_kernel_profile;

/* enable != 0 starts recording (allocating an event pool of `max_launches` pairs on first use);
 * enable == 0 stops.  Synchronous.  Errors: CB_ERR_INVALID_ARG, CB_ERR_CUDA. */
cb_status cb_profile_enable(cb_model* model, int32_t enable, int32_t max_launches);

/* Synchronises the device, writes up to max_entries classes (those with launches) to `out`, resets
 * the accumulators and returns the number written (negative cb_status on error).  Launches beyond
 * the event pool are counted but not timed (their ms is then a lower bound). */
int32_t cb_profile_read(cb_model* model, cb_kernel_profile* out, int32_t max_entries);

/* Re-RoPE with no device allocation.  The pages have no counterpart for this entry point: it serves
 * deployment, not the method.
 * Some callers cannot call cudaMalloc.  A KV-cache manager that has reserved nearly all device memory
 * for its own block pool is one: creating a model (which allocates a workspace sized for whole blends,
 * and needs the weights) would fail or fragment that pool, yet moving cached chunks to new positions
 * needs neither.  This call rotates the K rows of a chunk-cache buffer in place exactly as cb_rerope
 * does, without a model handle.  Its small per-call table (each chunk's start and the cos/sin of its
 * position delta) lives in a file-scope device array with room for CB_STATIC_MAX_CHUNKS chunks: about
 * 129 KiB on every device that loads the library, held until the process exits.
 *   kv, n_rows, chunks, n_chunks, stream: as for cb_rerope.  n_layers, n_kv_heads, head_dim (64 or
 *   128), rope_theta and dtype (cb_dtype) describe the buffer [n_layers][2][n_rows][n_kv_heads][head_dim].
 *   More than CB_STATIC_MAX_CHUNKS chunks -> CB_ERR_INVALID_ARG, with nothing enqueued.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress, with that
 * device current) and keeps it for the life of the process; make that first call before any stream
 * capture, and do not call this entry point on a device after cudaDeviceReset there (the new context
 * may place the array elsewhere).  n_kv_heads * head_dim above 2^24, or chunks covering more than
 * 2^31 - 1 rows -> CB_ERR_INVALID_ARG.  No call allocates or frees device
 * memory.  All calls share the one array; each call writes every entry it reads before reading it, so
 * nothing needs clearing, but calls whose GPU work may overlap (other streams, other threads) race on
 * it and must be serialised by the caller.  Errors are reported through cb_last_error(). */
#define CB_STATIC_MAX_CHUNKS 256
cb_status cb_rerope_static(void* kv, int64_t n_rows, int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
                           double rope_theta, int32_t dtype, const cb_chunk* chunks, int32_t n_chunks, void* stream);

/* HKVD selection on its own (section "选 token:HKVD、逐层过滤与 15% 这个经验值": keep the tokens of largest
 * KV deviation): the k rows of largest dev[0..n-1], ties to the lower row, written ascending to out_rows.
 * This is the select step cb_blend runs after its check layer, for callers that compute deviations
 * themselves.  A value that is not positive (including -0 and NaN) ranks as 0.
 *   dev       device float32 [n]
 *   out_rows  device int32 [k]
 * Requires 0 <= k <= n (else CB_ERR_INVALID_ARG); k = 0 enqueues nothing.  Async on `stream`; no allocation;
 * concurrent calls are independent. */
cb_status cb_select_hkvd(const float* dev, int32_t n, int32_t k, int32_t* out_rows, void* stream);

/* Loading controller (section "位置恢复、KV 存储与加载流水线", Figure 11).  Host arithmetic only.
 * cb_load_time: T_load = per_token_kv_bytes * n_tokens / throughput (seconds); -1 for a non-positive
 *   throughput or negative sizes.
 * cb_controller_ratio: the recompute ratio r whose recompute time r * T_prefill matches T_load, raised
 *   to the quality floor r_min (the page's r* = 15%) and capped at 1; -1 for negative times or r_min
 *   outside [0, 1].
 * cb_pick_storage: among n_devices storage tiers (throughput in bytes/s, cost per GB), the cheapest whose
 *   T_load does not exceed the recompute time at the floor, r_min * T_prefill (ties to the lower index);
 *   when none qualifies, the fastest.  Returns the device index, or CB_ERR_INVALID_ARG. */
double cb_load_time(double per_token_kv_bytes, int64_t n_tokens, double throughput_bytes_per_s);
double cb_controller_ratio(double t_prefill_s, double t_load_s, double r_min);
int32_t cb_pick_storage(const double* throughput_bytes_per_s, const double* cost_per_gb, int32_t n_devices,
                        double per_token_kv_bytes, int64_t n_tokens, double t_prefill_s, double r_min);

/* k = ceil(ratio * n_ctx - 1e-9) clamped to [0, n_ctx]; -1 if ratio is outside [0, 1] or NaN. */
int32_t cb_selected_count(int32_t n_ctx, double ratio);

/* The layout of cb_blend_gradual's (and cb_blend_streamed's) out_selected and out_dev for a schedule
 * (section "核心思想", Figure 9's funnel).  The comparing layers are the check layer 1 and every layer
 * l >= 2 whose count shrinks (k_l < k_{l-1}); for the i-th of them, in layer order:
 *   out_layers[i]   = l
 *   out_kept[i]     = k_l       rows that layer adds to out_selected
 *   out_compared[i] = n_ctx for the check layer, k_{l-1} for a shrinking layer: entries it adds to out_dev
 * Host arrays of max_entries; any of them may be NULL.  Returns the number of comparing layers, or
 * CB_ERR_INVALID_ARG (negative) for n_ctx < 0, n_ratios < 1, a ratio outside [0, 1], a growing schedule,
 * or more comparing layers than max_entries.  Host only. */
int32_t cb_gradual_layout(int32_t n_ctx, const double* ratios, int32_t n_ratios, int32_t* out_layers,
                          int32_t* out_kept, int32_t* out_compared, int32_t max_entries);

/* Description of the last error on the calling thread ("" if none). */
const char* cb_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* CACHEBLEND_H */
