// Internal declarations shared by the CUDA translation units of libcacheblend.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <string>
#include <vector>

#include "../../include/cacheblend.h"

namespace cb {

// ------------------------------------------------------------------------------------------------
// element types
// ------------------------------------------------------------------------------------------------
typedef __nv_bfloat16 bf16;

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// the pair (x0, x1) rotated by the angle whose (cos, sin) is r, with its roundings fixed (one rounded
// product, then one fused multiply-add) so that every re-RoPE kernel produces the same bits
__device__ __forceinline__ float2 rotate_pair(float x0, float x1, float2 r) {
    return make_float2(__fmaf_rn(x0, r.x, -__fmul_rn(x1, r.y)), __fmaf_rn(x0, r.y, __fmul_rn(x1, r.x)));
}

// split of an fp32 value into two bf16 numbers: hi = rn(v), lo = rn(v - hi)
__device__ __forceinline__ void split_bf16(float v, bf16& hi, bf16& lo) {
    hi = __float2bfloat16_rn(v);
    lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// Programmatic dependent launch.  grid_dep_wait: until the grids this one depends on have completed and
// their memory is visible (a no-op for a launch without the attribute); every thread calls it before its
// first global access.  grid_dep_launch: lets the next kernel on the stream start its prologue now.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// device status word bits (model->status); never trap, only record
enum : unsigned {
    ST_BAD_TOKEN = 1u,        // a token id outside [0, vocab) was read (embedding left zero)
    ST_WAIT_TIMEOUT = 2u,     // a bounded mbarrier wait gave up (tensor-core kernels)
    ST_BAD_ROW = 4u,          // a row index outside the buffer was seen and skipped
};

// ------------------------------------------------------------------------------------------------
// GEMM operand description:  Y[r][c] = sum_k X[r][k] * W[c][k]
//   X   token rows (activations), row-major [rows][K]
//   W   weight rows, row-major [out][K]; the output columns may be split over up to three
//       weight matrices ("segments"), e.g. wq | wk | wv.
// ------------------------------------------------------------------------------------------------
struct GemmW {
    const void* w[3];   // segment weight pointers
    int rows[3];        // rows (output columns) of each segment
    int nseg;
    const void* w_up;   // SwiGLU only: the up matrix (w[0] is the gate matrix)
    int layer;          // layer index (selects tensor maps on the tensor-core path)
    int which;          // WSEL_* below
};
enum { WSEL_QKV = 0, WSEL_Q = 1, WSEL_KV = 2, WSEL_O = 3, WSEL_GATEUP = 4, WSEL_DOWN = 5 };

// epilogue kinds
enum { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2 };

struct EpiParams {
    int kind;
    int M;                 // token rows of this GEMM
    const int* pos;        // global position of token row r (NULL: pos_offset + r)
    int pos_offset;
    // EPI_QKV: output column c is column (c + qkv_base) of the concatenated [q | k | v] space
    int qkv_base;
    int nq, nkv, head_dim;
    void* q_out;           // [M][nq] activation type
    void* act_lo;          // EPI_SWIGLU, split precision: low bf16 part of act (NULL otherwise)
    void* q_out_lo;        // EPI_QKV, split precision: low bf16 part of q (NULL otherwise)
    void* k_dst;           // K rows: storage type at row pos(r) (kv_fresh 0), fp32 at row r (1), storage type at row r (2)
    void* v_dst;
    int kv_fresh;          // 0: store K/V into the cache; 1: fp32 rows; 2 (tensor cores): compare, see below
    // kv_fresh == 2: the fresh K/V go to k_dst / v_dst at row r (storage type), and each epilogue warp also
    // compares its 32 features of every token row r < dev_rows with the stored cache row pos(r) of cmp_k /
    // cmp_v and writes the sum of squared differences to dev_part[r][slot], slot = (K: 0, V: nkv / 32) +
    // first feature / 32 (KV deviation, CacheBlend page "核心思想"); dev_parts = 2 * nkv / 32 per row.
    const void* cmp_k;
    const void* cmp_v;
    float* dev_part;
    int dev_parts;
    int dev_rows;
    const float2* rope;    // (cos, sin) [position][head_dim/2]
    // EPI_RESID: h[r][c] += y (fp32).  With the K range split over S > 1 units, unit s stores its sum to
    // part + s * M * ldh instead, and the next RMSNorm adds the S slots to h in slot order.
    float* h;
    int ldh;
    int atomic;
    float* part;           // partial-sum slots (tensor-core path)
    int part_rows;         // capacity of `part` in rows of ldh floats: S * M must not exceed it
    // EPI_SWIGLU: act[r][f] = silu(gate) * up
    void* act;
    int ld_act;
};

// ------------------------------------------------------------------------------------------------
// model
// ------------------------------------------------------------------------------------------------
struct TcMaps;   // tensor maps of the tensor-core path (defined in gemm_tc.cu)

// kernel classes for the opt-in per-class timing
enum KClass { K_REROPE, K_EMBED, K_RMSNORM, K_GEMM_Q, K_GEMM_KV, K_GEMM_QKV, K_GEMM_O, K_GEMM_GATEUP, K_GEMM_DOWN,
              K_ATTENTION, K_DEVIATION, K_TOPK, K_GATHER, K_LOGITS, K_DELTA, K_REFILTER, K_PAGES, K_NCLASS };

struct Profile {
    bool on = false;
    int cap = 0;                       // event pairs in the pool
    std::vector<cudaEvent_t> ev;       // 2 * cap
    std::vector<int> rec_class;        // class of each recorded pair
    int launches[K_NCLASS] = {};
    double flops[K_NCLASS] = {};
    double bytes[K_NCLASS] = {};
};

struct Model {
    cb_config cfg;
    int device;
    int num_sms;
    bool bf16;            // cfg.dtype == CB_BF16
    // borrowed weights
    const void* embed;
    const void* final_norm;
    const void* lm_head;
    std::vector<const void*> attn_norm, wq, wk, wv, wo, mlp_norm, w_gate, w_up, w_down;
    // workspace (device)
    float* h;             // [max_tokens][d] residual stream, all rows
    float* hA;            // [max_tokens][d] residual stream, recomputed rows
    void* x;              // [max_tokens][d] normalised activations (activation type)
    void* xA;             // [max_tokens][d]
    void* q;              // [max_tokens][nq]
    void* attn;           // [max_tokens][nq] attention output
    void* act;            // [max_tokens][ffn] SwiGLU output
    bool split;           // split-bf16 activations (hi + lo)
    void* x_lo;           // low parts of x, xA, attn, act (split precision only)
    void* xA_lo;
    void* attn_lo;
    void* act_lo;
    void* q_lo;           // low part of q (split precision only)
    float* part_o;        // attention key-range partials: [part_items][128][head_dim]
    float* part_ml;       // [part_items][128][2]
    unsigned* attn_sched; // attention work-item counter and finished-CTA count (zero between launches)
    int part_items;
    float* kf;            // [max_tokens][nkv] fresh K at the check layer (fp32)
    float* vf;            // [max_tokens][nkv] fresh V at the check layer (fp32)
    float* dev;           // [max_tokens] deviations
    float* tail_part;     // SwiGLU last-wave split: [tail_units][2][128][256] first-half accumulators
    unsigned* tail_flag;  // [tail_units][2] (zero between launches)
    int tail_units;
    float* part_h;        // [part_rows][d] split-K partial sums of the residual GEMMs (tensor-core path)
    int part_rows;
    float* dev_part;      // [max_tokens][2 * nkv / 32] per-warp deviation partials of the GEMM epilogue (bf16)
    int dev_parts;        // 2 * nkv / 32
    int* rows;            // [max_tokens] recomputed-row positions (selected ascending, then query)
    int* rows2;           // [max_tokens] the other rows buffer of gradual filtering (sets alternate)
    int* sel_local;       // [max_tokens] kept rows of a shrinking layer, as indices into the previous set
    int* iota;            // [max_tokens] 0, 1, 2, ...
    float2* rope;         // [max_tokens][hd/2]
    double* inv_freq;     // [hd/2] theta^(-2i/hd)
    float2* delta_cs;     // [max_chunks][hd/2] rotation of each chunk's position delta
    int* chunk_dst;       // [max_chunks]
    int* chunk_delta;     // [max_chunks]
    float* xfinal;        // [d] final-normed last row
    unsigned* status;     // device status word (ST_* bits)
    TcMaps* tc;           // tensor-core path state (NULL if unavailable)
    bool attn_tc;         // tensor-core attention usable
    alignas(64) unsigned char qmap[128];   // tensor map of the q workspace (attention)
    alignas(64) unsigned char qmap_lo[128];
    size_t ws_bytes;
    bool pdl;             // launch the tensor-core kernels with programmatic dependent launch
    Profile prof;
    std::vector<cudaEvent_t> io_ev;   // layer-wise load pipeline: [n_layers] loaded, [n_layers] final, fork, 2 joins
};

// ------------------------------------------------------------------------------------------------
// kernel launchers (return cudaGetLastError())
// ------------------------------------------------------------------------------------------------
struct ChunkTable {
    int n;
    int dst[CB_MAX_CHUNKS];
    int len[CB_MAX_CHUNKS];
    int delta[CB_MAX_CHUNKS];
};

cudaError_t launch_delta_table(const Model& m, const ChunkTable& t, cudaStream_t s);
cudaError_t launch_rerope(const Model& m, const void* src, void* dst, int64_t src_rows, int64_t dst_rows,
                          int n_ctx, int n_chunks, bool copy_v, cudaStream_t s, int layers = 0,
                          const int* src_pages = nullptr, int page_shift = 0);
// paged pool <-> contiguous rows (k_paged.cu); a NULL table is the identity
cudaError_t launch_page_copy(const Model& m, const void* src, int64_t src_rows, const int* src_pages, void* dst,
                             int64_t dst_rows, const int* dst_pages, int page_shift, int n_rows, cudaStream_t s);
cudaError_t launch_embed(const Model& m, const int* tokens, int n, float* h, cudaStream_t s);
// out = RMSNorm(h) for n rows; when parts > 0, h is first completed as h + part[0] + ... + part[parts-1]
// (slots of n rows each, added in slot order) and written back
cudaError_t launch_rmsnorm(const Model& m, float* h, const float* part, int parts, const void* g, void* out,
                           void* out_lo, int n, cudaStream_t s);
cudaError_t launch_deviation(const Model& m, const float* kf, const float* vf, const void* kv_layer, int64_t kv_rows,
                             const int* crow, int n_ctx, float* dev, cudaStream_t s);
cudaError_t launch_refilter(const Model& m, const int* local, const int* rows_old, int* rows_new, int M_new, int k_new,
                            int* out_sel, const float* h_old, float* h_new, const void* x_old, void* x_new,
                            const void* xlo_old, void* xlo_new, const void* kf, const void* vf, bool kv_f32,
                            void* kv_layer, int64_t kv_rows, cudaStream_t s);
// top-k of the deviations dev_in[n_ctx], or (dev_in NULL) of the sums of dev_part[n_ctx][parts], which are
// then written to dev; rows receives the selected rows ascending, then the query rows n_ctx .. n_ctx+n_query-1
cudaError_t launch_topk(bool pdl, const float* dev_in, const float* dev_part, int parts, float* dev, int n_ctx, int k,
                        int n_query, int* rows, int* out_sel, cudaStream_t s);
// rows = sel[0..k) (validated: ascending, in [0, n)) then the query rows n .. n+n_query-1
cudaError_t launch_given_rows(bool pdl, const int* sel, int k, int n, int n_query, int* rows, int* out_sel,
                              unsigned* status, cudaStream_t s);
// hA/xA <- rows of h/x; with kf (fresh K/V rows, fp32 when kv_f32 else the storage type) also the K/V of those
// rows into the blended cache block kv_layer at their positions
cudaError_t launch_gather(const Model& m, const int* rows, int M, const float* h, float* hA, const void* x, void* xA,
                          const void* x_lo, void* xA_lo, const void* kf, const void* vf, bool kv_f32, void* kv_layer,
                          int64_t kv_rows, cudaStream_t s);
cudaError_t launch_attention(const Model& m, const void* q, const void* q_lo, const int* qpos, int M,
                             const void* kv_layer, int64_t kv_rows, int n_keys, void* out, void* out_lo, cudaStream_t s);
// logits of h_last (+ the pending partial sums part[0 .. parts-1] of that row, slot stride part_stride floats)
cudaError_t launch_logits(const Model& m, const float* h_last, const float* part, int parts, size_t part_stride,
                          float* logits, cudaStream_t s);
cudaError_t launch_gemm_simt(const Model& m, const void* X, const void* X_lo, int M, int K, const GemmW& w, int N,
                             const EpiParams& e, cudaStream_t s);

// tensor-core path (gemm_tc.cu)
bool tc_init(Model& m, std::string& err);
void tc_destroy(Model& m);
// *splits (optional) receives the number of K ranges of a residual GEMM (1: h holds the final sum; S > 1:
// S partial-sum slots are pending)
cudaError_t launch_gemm_tc(const Model& m, int xbuf, int x_row0, int M, int K, const GemmW& w, int N,
                           const EpiParams& e, cudaStream_t s, int* launches, int* splits = nullptr);
enum { XBUF_X = 0, XBUF_XA = 1, XBUF_ATTN = 2, XBUF_ACT = 3 };

// Raise kernel `k`'s dynamic shared-memory limit to `bytes` on the current device, once per device (CUDA
// keeps the attribute per device; `done` holds one bit per device ordinal below 64).
template <typename... KArgs>
cudaError_t smem_limit_once(void (*k)(KArgs...), int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Launch `k` on `s`, with programmatic dependent launch when `pdl` (the kernel calls grid_dep_wait
// before its first global access, so it may start while the previous kernel on the stream drains).
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(bool pdl, void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                      Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &at;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

// records a message for cb_last_error() on the calling thread
void set_last_error(const char* msg);

// tensor-core attention (attn_tc.cu); maps are CUtensorMap (128 bytes, 64-byte aligned)
bool attn_tc_supported(const Model& m);
bool attn_make_qmap(const Model& m, const void* q, void* map_out);
bool attn_make_kvmap(const Model& m, const void* kv, int64_t rows, void* map_out);
cudaError_t launch_attention_tc(const Model& m, const void* qmap, const void* qmap_lo, const void* kvmap, int layer,
                                const int* qpos, int M, int n_keys, void* out, void* out_lo, cudaStream_t s,
                                int* launches);

}  // namespace cb
