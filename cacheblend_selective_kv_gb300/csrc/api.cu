// C ABI of libcacheblend: validation, workspace, and the per-request blend schedule.
//
// The schedule follows the CacheBlend deep-dive page (sections "核心思想" and "选 token",
// Figures 5 and 9): re-RoPE placement, layer 0 over every row with reused context K/V, the
// check layer (fresh K/V of every row, KV deviation, top-k), then selective recompute of the
// chosen rows plus the query in every later layer, and the last row's logits.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "cb_common.cuh"

using namespace cb;

struct cb_model : public cb::Model {};

namespace {

thread_local char g_err[512] = "";

cb_status fail(cb_status code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

#define CB_CUDA(call)                                                                                 \
    do {                                                                                              \
        cudaError_t e_ = (call);                                                                      \
        if (e_ != cudaSuccess) return fail(CB_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_));     \
    } while (0)

size_t act_size(const Model& m) { return m.bf16 ? 2 : 4; }

void free_ws(Model& m) {
    void* ptrs[] = {m.h, m.hA, m.x, m.xA, m.q, m.attn, m.act, m.kf, m.vf, m.dev, m.dev_part, m.part_h, m.tail_part,
                    m.tail_flag, m.rows, m.rows2,
                    m.sel_local, m.iota,
                    m.rope, m.inv_freq, m.delta_cs, m.chunk_dst, m.chunk_delta, m.xfinal, m.status,
                    m.x_lo, m.xA_lo, m.attn_lo, m.act_lo, m.q_lo, m.part_o, m.part_ml, m.attn_sched};
    for (void* p : ptrs)
        if (p) cudaFree(p);
}

bool fault_injected(const char* what) {
    const char* v = getenv("CB_FAULT_INJECT");
    return v && strcmp(v, what) == 0;
}

}  // namespace

void cb::set_last_error(const char* msg) { snprintf(g_err, sizeof g_err, "%s", msg); }

extern "C" {

const char* cb_last_error(void) { return g_err; }

int32_t cb_selected_count(int32_t n_ctx, double ratio) {
    if (!(ratio >= 0.0 && ratio <= 1.0) || n_ctx < 0) return -1;
    double k = std::ceil(ratio * (double)n_ctx - 1e-9);
    if (k < 0) k = 0;
    if (k > n_ctx) k = n_ctx;
    return (int32_t)k;
}

int32_t cb_gradual_layout(int32_t n_ctx, const double* ratios, int32_t n_ratios, int32_t* out_layers,
                          int32_t* out_kept, int32_t* out_compared, int32_t max_entries) {
    if (n_ctx < 0 || n_ratios < 1 || !ratios || max_entries < 0) return CB_ERR_INVALID_ARG;
    int n = 0, prev = 0;
    for (int l = 1; l <= n_ratios; ++l) {
        const int k = cb_selected_count(n_ctx, ratios[l - 1]);
        if (k < 0 || (l >= 2 && k > prev)) return CB_ERR_INVALID_ARG;
        // the rule blend_impl applies: layer 1 always compares, a later layer when its count shrinks
        if (l == 1 || k < prev) {
            if (n >= max_entries) return CB_ERR_INVALID_ARG;
            if (out_layers) out_layers[n] = l;
            if (out_kept) out_kept[n] = k;
            if (out_compared) out_compared[n] = l == 1 ? n_ctx : prev;
            ++n;
        }
        prev = k;
    }
    return n;
}

cb_status cb_model_create(const cb_config* cfg, const cb_weights* w, cb_model** out) {
    g_err[0] = 0;
    if (!cfg || !w || !out) return fail(CB_ERR_INVALID_ARG, "cb_model_create: null argument");
    *out = nullptr;
    const cb_config& c = *cfg;
    if (c.n_layers < 2 || c.d_model <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 || c.head_dim <= 0 ||
        c.ffn_hidden <= 0 || c.vocab <= 0 || c.max_tokens <= 0 || c.max_chunks < 0)
        return fail(CB_ERR_INVALID_ARG, "cb_model_create: non-positive dimension (n_layers must be >= 2)");
    if (c.n_heads % c.n_kv_heads != 0) return fail(CB_ERR_INVALID_ARG, "n_heads must be a multiple of n_kv_heads");
    if (c.head_dim != 64 && c.head_dim != 128) return fail(CB_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (c.d_model % 64 || c.ffn_hidden % 64) return fail(CB_ERR_UNSUPPORTED, "d_model and ffn_hidden must be multiples of 64");
    if (c.d_model > 8192) return fail(CB_ERR_UNSUPPORTED, "d_model above 8192");
    if (c.n_heads / c.n_kv_heads > 8) return fail(CB_ERR_UNSUPPORTED, "at most 8 query heads per KV head");
    if (c.dtype != CB_F32 && c.dtype != CB_BF16) return fail(CB_ERR_INVALID_ARG, "dtype must be CB_F32 or CB_BF16");
    if (c.precision != CB_PREC_SPLIT && c.precision != CB_PREC_BF16)
        return fail(CB_ERR_INVALID_ARG, "precision must be CB_PREC_SPLIT or CB_PREC_BF16");
    if (c.max_chunks > CB_MAX_CHUNKS) return fail(CB_ERR_INVALID_ARG, "max_chunks exceeds CB_MAX_CHUNKS");
    if (!(c.rope_theta > 0) || !(c.rms_eps >= 0)) return fail(CB_ERR_INVALID_ARG, "rope_theta must be > 0, rms_eps >= 0");
    if (!w->embed || !w->final_norm || !w->lm_head || !w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo ||
        !w->mlp_norm || !w->w_gate || !w->w_up || !w->w_down)
        return fail(CB_ERR_INVALID_ARG, "cb_model_create: null weight pointer");
    for (int l = 0; l < c.n_layers; ++l) {
        const void* ps[] = {w->attn_norm[l], w->wq[l], w->wk[l], w->wv[l], w->wo[l], w->mlp_norm[l],
                            w->w_gate[l], w->w_up[l], w->w_down[l]};
        for (const void* p : ps) {
            if (!p) return fail(CB_ERR_INVALID_ARG, "null weight pointer in layer %d", l);
            if ((uintptr_t)p % 16) return fail(CB_ERR_INVALID_ARG, "weight pointer of layer %d not 16-byte aligned", l);
        }
    }

    cb_model* m = new (std::nothrow) cb_model();
    if (!m) return fail(CB_ERR_OOM, "host allocation failed");
    m->cfg = c;
    m->bf16 = c.dtype == CB_BF16;
    m->split = m->bf16 && c.precision == CB_PREC_SPLIT;
    m->x_lo = m->xA_lo = m->attn_lo = m->act_lo = m->q_lo = nullptr;
    m->part_o = m->part_ml = nullptr;
    m->attn_sched = nullptr;
    if (cudaGetDevice(&m->device) != cudaSuccess) { delete m; return fail(CB_ERR_CUDA, "no CUDA device"); }
    cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device);
    m->part_items = m->bf16 ? 8 * m->num_sms : 0;
    m->embed = w->embed;
    m->final_norm = w->final_norm;
    m->lm_head = w->lm_head;
    m->attn_norm.assign(w->attn_norm, w->attn_norm + c.n_layers);
    m->wq.assign(w->wq, w->wq + c.n_layers);
    m->wk.assign(w->wk, w->wk + c.n_layers);
    m->wv.assign(w->wv, w->wv + c.n_layers);
    m->wo.assign(w->wo, w->wo + c.n_layers);
    m->mlp_norm.assign(w->mlp_norm, w->mlp_norm + c.n_layers);
    m->w_gate.assign(w->w_gate, w->w_gate + c.n_layers);
    m->w_up.assign(w->w_up, w->w_up + c.n_layers);
    m->w_down.assign(w->w_down, w->w_down + c.n_layers);
    m->h = m->hA = nullptr; m->x = m->xA = m->q = m->attn = m->act = nullptr;
    m->kf = m->vf = m->dev = m->dev_part = m->part_h = m->tail_part = nullptr;
    m->tail_flag = nullptr;
    m->tail_units = m->bf16 ? (m->num_sms + 1) / 2 : 0;    // at most one unit per CTA pair
    m->rows = m->rows2 = m->sel_local = m->iota = nullptr; m->rope = nullptr;
    // split-K partial-sum slots of the residual GEMMs: splits x rows must fit in part_rows rows of d
    m->part_rows = m->bf16 ? 12288 : 0;
    m->dev_parts = 2 * c.n_kv_heads * c.head_dim / 32;
    m->inv_freq = nullptr;
    m->delta_cs = nullptr; m->chunk_dst = m->chunk_delta = nullptr; m->xfinal = nullptr; m->status = nullptr;
    m->tc = nullptr;

    const size_t T = (size_t)c.max_tokens, d = c.d_model, nq = (size_t)c.n_heads * c.head_dim;
    const size_t nkv = (size_t)c.n_kv_heads * c.head_dim, F = c.ffn_hidden, half = c.head_dim / 2;
    const size_t as = act_size(*m);
    const size_t mc = c.max_chunks > 0 ? c.max_chunks : 1;
    struct { void** p; size_t bytes; } allocs[] = {
        {(void**)&m->h, T * d * 4}, {(void**)&m->hA, T * d * 4}, {&m->x, T * d * as}, {&m->xA, T * d * as},
        {&m->q, T * nq * as}, {&m->attn, T * nq * as}, {&m->act, T * F * as}, {(void**)&m->kf, T * nkv * 4},
        {(void**)&m->vf, T * nkv * 4}, {(void**)&m->dev, T * 4},
        {(void**)&m->dev_part, m->bf16 ? T * (size_t)m->dev_parts * 4 : 0},
        {(void**)&m->part_h, (size_t)m->part_rows * d * 4},
        {(void**)&m->tail_part, (size_t)m->tail_units * 2 * 128 * 256 * 4},
        {(void**)&m->tail_flag, (size_t)m->tail_units * 2 * 4}, {(void**)&m->rows, T * 4},
        {(void**)&m->rows2, T * 4}, {(void**)&m->sel_local, T * 4},
        {(void**)&m->iota, T * 4}, {(void**)&m->rope, T * half * sizeof(float2)},
        {(void**)&m->inv_freq, half * sizeof(double)}, {(void**)&m->delta_cs, mc * half * sizeof(float2)},
        {(void**)&m->chunk_dst, mc * 4}, {(void**)&m->chunk_delta, mc * 4}, {(void**)&m->xfinal, d * 4},
        {(void**)&m->status, 64},
        {&m->x_lo, m->split ? T * d * as : 0}, {&m->xA_lo, m->split ? T * d * as : 0},
        {&m->attn_lo, m->split ? T * nq * as : 0}, {&m->act_lo, m->split ? T * F * as : 0},
        {&m->q_lo, m->split ? T * nq * as : 0},
        {(void**)&m->part_o, (size_t)m->part_items * 128 * c.head_dim * 4},
        {(void**)&m->part_ml, (size_t)m->part_items * 128 * 2 * 4},
        {(void**)&m->attn_sched, 64}};
    size_t total = 0;
    for (auto& a : allocs) {
        if (a.bytes == 0) continue;
        if (fault_injected("alloc") || cudaMalloc(a.p, a.bytes) != cudaSuccess) {
            cudaGetLastError();
            free_ws(*m);
            delete m;
            return fail(CB_ERR_OOM, "workspace allocation of %zu bytes failed", a.bytes);
        }
        total += a.bytes;
        cudaMemset(*a.p, 0, a.bytes);
    }
    m->ws_bytes = total;

    // RoPE tables: angle = pos * theta^(-2i/hd), computed in float64, stored as float32 (cos, sin)
    std::vector<double> inv(half);
    for (size_t i = 0; i < half; ++i) inv[i] = std::pow(c.rope_theta, -2.0 * (double)i / (double)c.head_dim);
    std::vector<float2> tab(T * half);
    for (size_t p = 0; p < T; ++p)
        for (size_t i = 0; i < half; ++i) {
            const double a = (double)p * inv[i];
            tab[p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
        }
    std::vector<int> iota(T);
    for (size_t i = 0; i < T; ++i) iota[i] = (int)i;
    if (cudaMemcpy(m->inv_freq, inv.data(), half * sizeof(double), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(m->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(m->iota, iota.data(), T * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
        free_ws(*m);
        delete m;
        return fail(CB_ERR_CUDA, "table upload failed");
    }
    m->attn_tc = false;
    {
        const char* v = getenv("CB_PDL");
        m->pdl = !(v && v[0] == '0');
    }
    if (m->bf16) {
        std::string err;
        if (!tc_init(*m, err)) m->tc = nullptr;   // CUDA-core path only
        const char* off = getenv("CB_DISABLE_TC_ATTN");
        if (m->tc && !(off && off[0] == '1') && attn_tc_supported(*m) && attn_make_qmap(*m, m->q, m->qmap) &&
            (!m->split || attn_make_qmap(*m, m->q_lo, m->qmap_lo)))
            m->attn_tc = true;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaError_t e = cudaGetLastError();
        tc_destroy(*m);
        free_ws(*m);
        delete m;
        return fail(CB_ERR_CUDA, "model setup: %s", cudaGetErrorString(e));
    }
    *out = m;
    return CB_OK;
}

cb_status cb_model_destroy(cb_model* m) {
    g_err[0] = 0;
    if (!m) return CB_OK;
    cudaDeviceSynchronize();
    for (auto e : m->prof.ev) cudaEventDestroy(e);
    for (auto e : m->io_ev) cudaEventDestroy(e);
    tc_destroy(*m);
    free_ws(*m);
    delete m;
    return CB_OK;
}

}  // extern "C"

namespace {

cb_status check_chunks(const cb_chunk* chunks, int32_t n_chunks, int max_chunks, int& n_ctx, ChunkTable& t) {
    if (n_chunks < 0) return fail(CB_ERR_INVALID_ARG, "n_chunks < 0");
    if (n_chunks > 0 && !chunks) return fail(CB_ERR_INVALID_ARG, "chunks is NULL");
    if (n_chunks > max_chunks) return fail(CB_ERR_INVALID_ARG, "n_chunks %d exceeds the model's max_chunks %d", n_chunks, max_chunks);
    int64_t at = 0;
    t.n = n_chunks;
    for (int i = 0; i < n_chunks; ++i) {
        const cb_chunk& c = chunks[i];
        if (c.src_pos < 0) return fail(CB_ERR_INVALID_ARG, "chunk %d: unknown source position (src_pos < 0)", i);
        if (c.len <= 0) return fail(CB_ERR_INVALID_ARG, "chunk %d: len must be > 0", i);
        if (c.dst_pos != at) return fail(CB_ERR_INVALID_ARG, "chunk %d: chunks must tile [0, n_ctx) in order (dst_pos %d, expected %lld)", i, c.dst_pos, (long long)at);
        at += c.len;
        if (at > (1 << 30)) return fail(CB_ERR_INVALID_ARG, "chunk lengths overflow");
        t.dst[i] = c.dst_pos;
        t.len[i] = c.len;
        t.delta[i] = c.dst_pos - c.src_pos;
    }
    n_ctx = (int)at;
    return CB_OK;
}

const char* const kClassName[K_NCLASS] = {"rerope", "embed", "rmsnorm", "gemm_q", "gemm_kv", "gemm_qkv", "gemm_o",
                                         "gemm_gateup", "gemm_down", "attention", "deviation", "topk",
                                         "gather", "logits", "delta_table", "refilter", "pages"};

// Enqueues launches on one stream; counts them and, when profiling is on, brackets each with events.
struct Sched {
    Model& m;
    cudaStream_t s;
    int launches = 0;
    double gemm_flops = 0;
    int last_splits = 1;     // K ranges of the last residual GEMM (S > 1: S partial-sum slots pending)
    cudaError_t err = cudaSuccess;

    template <typename F>
    void k(int cls, double flops, double bytes, F&& launch, int n_launch = 1) {
        Profile& p = m.prof;
        const bool timed = p.on && (int)p.rec_class.size() < p.cap;
        if (timed) cudaEventRecord(p.ev[2 * p.rec_class.size()], s);
        cudaError_t e = launch();
        if (timed) {
            cudaEventRecord(p.ev[2 * p.rec_class.size() + 1], s);
            p.rec_class.push_back(cls);
        }
        if (p.on) {
            p.launches[cls] += n_launch;
            p.flops[cls] += flops;
            p.bytes[cls] += bytes;
        }
        launches += n_launch;
        if (e != cudaSuccess && err == cudaSuccess) err = e;
    }
    void* xbuf(int id) const {
        switch (id) {
            case XBUF_X: return m.x;
            case XBUF_XA: return m.xA;
            case XBUF_ATTN: return m.attn;
            default: return m.act;
        }
    }
    void* xbuf_lo(int id) const {
        switch (id) {
            case XBUF_X: return m.x_lo;
            case XBUF_XA: return m.xA_lo;
            case XBUF_ATTN: return m.attn_lo;
            default: return m.act_lo;
        }
    }
    void gemm(int cls, int xb, int row0, int M, int K, const GemmW& w, int N, const EpiParams& e) {
        if (M <= 0 || N <= 0) return;
        const double es = act_size(m);
        // algorithmic FLOPs of the projection (the split's second MMA is not counted as work)
        const double f = 2.0 * M * (double)N * K * (e.kind == EPI_SWIGLU ? 2 : 1);
        const double wbytes = (double)N * K * es * (e.kind == EPI_SWIGLU ? 2 : 1);
        gemm_flops += f;
        last_splits = 1;
        if (m.tc) {
            int n = 1;
            k(cls, f, wbytes, [&] { return launch_gemm_tc(m, xb, row0, M, K, w, N, e, s, &n, &last_splits); });
        } else {
            const char* base = (const char*)xbuf(xb) + (size_t)row0 * K * act_size(m);
            const char* lo = m.split ? (const char*)xbuf_lo(xb) + (size_t)row0 * K * act_size(m) : nullptr;
            k(cls, f, wbytes, [&] { return launch_gemm_simt(m, base, lo, M, K, w, N, e, s); });
        }
    }
};

GemmW wsel(const Model& m, int layer, int which) {
    const cb_config& c = m.cfg;
    GemmW g;
    memset(&g, 0, sizeof g);
    g.layer = layer;
    g.which = which;
    const int nq = c.n_heads * c.head_dim, nkv = c.n_kv_heads * c.head_dim;
    switch (which) {
        case WSEL_QKV: g.nseg = 3; g.w[0] = m.wq[layer]; g.w[1] = m.wk[layer]; g.w[2] = m.wv[layer];
                       g.rows[0] = nq; g.rows[1] = nkv; g.rows[2] = nkv; break;
        case WSEL_Q: g.nseg = 1; g.w[0] = m.wq[layer]; g.rows[0] = nq; break;
        case WSEL_KV: g.nseg = 2; g.w[0] = m.wk[layer]; g.w[1] = m.wv[layer]; g.rows[0] = nkv; g.rows[1] = nkv; break;
        case WSEL_O: g.nseg = 1; g.w[0] = m.wo[layer]; g.rows[0] = c.d_model; break;
        case WSEL_GATEUP: g.nseg = 1; g.w[0] = m.w_gate[layer]; g.w_up = m.w_up[layer]; g.rows[0] = c.ffn_hidden; break;
        default: g.nseg = 1; g.w[0] = m.w_down[layer]; g.rows[0] = c.d_model; break;
    }
    return g;
}

EpiParams epi_base(const Model& m, int kind, int M) {
    EpiParams e;
    memset(&e, 0, sizeof e);
    e.part = m.part_h;
    e.part_rows = m.part_rows;
    e.q_out_lo = m.q_lo;
    e.kind = kind;
    e.M = M;
    e.nq = m.cfg.n_heads * m.cfg.head_dim;
    e.nkv = m.cfg.n_kv_heads * m.cfg.head_dim;
    e.head_dim = m.cfg.head_dim;
    e.rope = m.rope;
    return e;
}

}  // namespace

extern "C" {

cb_status cb_rerope(cb_model* m, void* kv, int64_t n_rows, const cb_chunk* chunks, int32_t n_chunks, void* stream) {
    g_err[0] = 0;
    if (!m || !kv) return fail(CB_ERR_INVALID_ARG, "cb_rerope: null model or kv");
    ChunkTable t;
    int n_ctx = 0;
    cb_status st = check_chunks(chunks, n_chunks, m->cfg.max_chunks, n_ctx, t);
    if (st != CB_OK) return st;
    if (n_ctx > n_rows) return fail(CB_ERR_INVALID_ARG, "chunks cover %d rows but the buffer has %lld", n_ctx, (long long)n_rows);
    if (n_chunks == 0) return CB_OK;
    cudaStream_t s = (cudaStream_t)stream;
    Sched S{*m, s};
    const double row = (double)m->cfg.n_kv_heads * m->cfg.head_dim * act_size(*m);
    S.k(K_DELTA, 0, 0, [&] { return launch_delta_table(*m, t, s); });
    S.k(K_REROPE, 0, 2.0 * m->cfg.n_layers * n_ctx * row,
        [&] { return launch_rerope(*m, kv, kv, n_rows, n_rows, n_ctx, n_chunks, false, s); });
    if (S.err != cudaSuccess) return fail(CB_ERR_CUDA, "cb_rerope: %s", cudaGetErrorString(S.err));
    return CB_OK;
}

}  // extern "C"

namespace {

// One blend.  ks[l] (l = 1..L-1) is the number of context rows whose hidden state leaves layer l:
// constant for the blend with one selection at the check layer, non-increasing for gradual filtering
// (a layer with ks[l] < ks[l-1] compares its candidates again and keeps the top ks[l]).
// `io` (optional): the layer-wise load pipeline.  The chunk caches then come from pinned host memory,
// one layer per copy on io->copy_stream, and each layer is re-RoPE'd in place once its copy has landed,
// just before that layer is computed; each layer's finished K/V can be copied back the same way.
cb_status blend_impl(Model& m, const int32_t* tokens, int32_t n_tokens, const void* cached_kv, const ChunkTable& t,
                     int n_chunks, int n_ctx, const std::vector<int>& ks, void* out_kv, float* out_logits,
                     int32_t* out_selected, float* out_dev, cb_stats* stats, cudaStream_t s,
                     const cb_layer_io* io = nullptr, const cb_paged_kv* pg = nullptr, int page_shift = 0,
                     const int32_t* given = nullptr) {
    const cb_config& c = m.cfg;
    const size_t es = act_size(m);
    const int L = c.n_layers, d = c.d_model, nq = c.n_heads * c.head_dim, nkv = c.n_kv_heads * c.head_dim;
    const int F = c.ffn_hidden, N = n_tokens, Q = N - n_ctx;
    const bool inplace = n_chunks > 0 && cached_kv == out_kv;
    const int k = ks[1];
    const int M = k + Q;

    Sched S{m, s};
    char* kvb = (char*)out_kv;
    auto layer_kv = [&](int l) { return (void*)(kvb + (size_t)l * 2 * N * nkv * es); };
    auto layer_v = [&](int l) { return (void*)(kvb + ((size_t)l * 2 + 1) * N * nkv * es); };
    const double row = (double)nkv * es;             // bytes of one token's K (or V) in one layer
    const double hd = c.head_dim, Hq = c.n_heads;
    auto attn_flops = [&](double keys) { return 4.0 * hd * Hq * keys; };
    // causal key counts of the recomputed rows (selected rows at the mean context position)
    const double keys0 = (double)N * (N + 1) / 2.0;
    auto keys_of = [&](int kl) {
        return (double)Q * (n_ctx + 1) + (double)Q * (Q - 1) / 2.0 + (double)kl * (n_ctx + 1) / 2.0;
    };

    // re-RoPE placement of the chunk caches (section "位置恢复、KV 存储与加载流水线")
    cudaStream_t cs = io ? (cudaStream_t)io->copy_stream : nullptr;
    cudaStream_t bs = io ? (io->copy_back_stream ? (cudaStream_t)io->copy_back_stream : cs) : nullptr;
    cudaError_t io_err = cudaSuccess;
    auto io_check = [&](cudaError_t e) { if (e != cudaSuccess && io_err == cudaSuccess) io_err = e; };
    if (io) {
        // fork the copy stream off the compute stream, then queue every layer's load in layer order:
        // layer l's chunk caches land in rows 0..n_ctx-1 of its K and V blocks of out_kv
        io_check(cudaEventRecord(m.io_ev[2 * L], s));
        io_check(cudaStreamWaitEvent(cs, m.io_ev[2 * L], 0));
        if (bs != cs) io_check(cudaStreamWaitEvent(bs, m.io_ev[2 * L], 0));
        if (n_chunks > 0) {
            const size_t w = (size_t)n_ctx * nkv * es;
            for (int l = 0; l < L; ++l) {
                io_check(cudaMemcpy2DAsync(layer_kv(l), (size_t)N * nkv * es,
                                           (const char*)io->cached_kv_host + (size_t)l * 2 * w, w, w, 2,
                                           cudaMemcpyHostToDevice, cs));
                io_check(cudaEventRecord(m.io_ev[l], cs));
            }
            S.k(K_DELTA, 0, 0, [&] { return launch_delta_table(m, t, s); });
        }
    } else if (pg && n_chunks > 0) {
        // paged: the chunk caches are read from their pool pages, re-rotated and placed in the contiguous
        // working copy (out_kv) in one pass; the pool is written back at the end
        S.k(K_DELTA, 0, 0, [&] { return launch_delta_table(m, t, s); });
        S.k(K_REROPE, 0, 4.0 * L * n_ctx * row,
            [&] { return launch_rerope(m, pg->pool, out_kv, pg->n_pages * (int64_t)pg->page_size, N, n_ctx, n_chunks,
                                       true, s, 0, pg->src_table, page_shift); });
    } else if (n_chunks > 0) {
        S.k(K_DELTA, 0, 0, [&] { return launch_delta_table(m, t, s); });
        S.k(K_REROPE, 0, (inplace ? 2.0 : 4.0) * L * n_ctx * row,
            [&] { return launch_rerope(m, cached_kv, out_kv, inplace ? N : n_ctx, N, n_ctx, n_chunks, !inplace, s); });
    }
    // pipeline: layer l's cache must have landed (and be re-rotated) before layer l reads it ...
    auto layer_in = [&](int l) {
        if (!io || n_chunks == 0) return;
        io_check(cudaStreamWaitEvent(s, m.io_ev[l], 0));
        S.k(K_REROPE, 0, 2.0 * n_ctx * row,
            [&] { return launch_rerope(m, layer_kv(l), layer_kv(l), N, N, n_ctx, n_chunks, false, s, 1); });
    };
    // ... and once layer l's K/V are final (its recomputed rows stored), they can go back to the host
    auto layer_out = [&](int l) {
        if (!io || !io->out_kv_host) return;
        io_check(cudaEventRecord(m.io_ev[L + l], s));
        io_check(cudaStreamWaitEvent(bs, m.io_ev[L + l], 0));
        io_check(cudaMemcpyAsync((char*)io->out_kv_host + (size_t)l * 2 * N * nkv * es, layer_kv(l),
                                 (size_t)2 * N * nkv * es, cudaMemcpyDeviceToHost, bs));
    };
    S.k(K_EMBED, 0, (double)N * d * (es + 4), [&] { return launch_embed(m, tokens, N, m.h, s); });
    alignas(64) unsigned char kvmap[128];
    const bool attn_tc = m.attn_tc && attn_make_kvmap(m, out_kv, N, kvmap);
    auto attend = [&](int l, const int* qpos, int rowsq, double keys) {
        int n = 1;
        S.k(K_ATTENTION, attn_flops(keys), 2.0 * N * row, [&] {
            return attn_tc ? launch_attention_tc(m, m.qmap, m.qmap_lo, kvmap, l, qpos, rowsq, N, m.attn, m.attn_lo, s, &n)
                           : launch_attention(m, m.q, m.q_lo, qpos, rowsq, layer_kv(l), N, N, m.attn, m.attn_lo, s);
        });
        S.launches += n - 1;
        if (m.prof.on) m.prof.launches[K_ATTENTION] += n - 1;
    };
    // partial-sum slots the last residual GEMM left for the next norm (or the logits) to add
    int pend = 0;
    auto resid_done = [&] { pend = S.last_splits > 1 ? S.last_splits : 0; };
    auto norm = [&](float* h, const void* g, void* out, int n) {
        void* lo = !m.split ? nullptr : (out == m.x ? m.x_lo : m.xA_lo);
        const int parts = pend;
        pend = 0;
        const double bytes = (double)n * d * (4.0 + (parts ? 4.0 * parts + 4.0 : 0.0) + es * (lo ? 2 : 1));
        S.k(K_RMSNORM, 0, bytes, [&] { return launch_rmsnorm(m, h, m.part_h, parts, g, out, lo, n, s); });
    };

    // ---- layer 0: every row's hidden state; context K/V reused, query K/V fresh --------------
    {
        norm(m.h, m.attn_norm[0], m.x, N);
        EpiParams e = epi_base(m, EPI_QKV, N);
        e.qkv_base = 0;
        e.q_out = m.q;
        S.gemm(K_GEMM_Q, XBUF_X, 0, N, d, wsel(m, 0, WSEL_Q), nq, e);
        EpiParams ekv = epi_base(m, EPI_QKV, Q);
        ekv.qkv_base = nq;
        ekv.pos_offset = n_ctx;
        ekv.k_dst = layer_kv(0);
        ekv.v_dst = layer_v(0);
        S.gemm(K_GEMM_KV, XBUF_X, n_ctx, Q, d, wsel(m, 0, WSEL_KV), 2 * nkv, ekv);
        layer_in(0);
        attend(0, m.iota, N, keys0);
        layer_out(0);
        EpiParams er = epi_base(m, EPI_RESID, N);
        er.h = m.h;
        er.ldh = d;
        S.gemm(K_GEMM_O, XBUF_ATTN, 0, N, nq, wsel(m, 0, WSEL_O), d, er);
        resid_done();
        norm(m.h, m.mlp_norm[0], m.x, N);
        EpiParams eg = epi_base(m, EPI_SWIGLU, N);
        eg.act = m.act;
        eg.act_lo = m.act_lo;
        eg.ld_act = F;
        S.gemm(K_GEMM_GATEUP, XBUF_X, 0, N, d, wsel(m, 0, WSEL_GATEUP), F, eg);
        S.gemm(K_GEMM_DOWN, XBUF_ACT, 0, N, F, wsel(m, 0, WSEL_DOWN), d, er);
        resid_done();
    }

    // ---- check layer 1: fresh K/V of every row, deviation, top-k, then the chosen rows --------
    // With the tensor cores the comparing GEMM's epilogue keeps the fresh K/V as rows of the storage type and
    // compares them with the cache itself (per-warp partial sums, added by the top-k kernel in a fixed
    // order); on the CUDA-core path the GEMM keeps fp32 rows and a separate kernel compares them.
    const bool fused_dev = m.tc != nullptr;
    float* devp = out_dev ? out_dev : m.dev;
    // fresh K/V of `rows` GEMM rows of input buffer `xb` (positions `pos`, NULL: 0..), the first `ncmp` of them
    // compared with the re-RoPE'd cache of layer l: deviations into devd, then the top `kk` of them
    auto compare = [&](int l, int xb, int rows, int ncmp, const int* pos, float* devd, int kk, int* sel_rows,
                       int* sel_out) {
        if (rows > 0) {
            EpiParams ekv = epi_base(m, EPI_QKV, rows);
            ekv.qkv_base = nq;
            ekv.pos = pos;
            ekv.k_dst = m.kf;
            ekv.v_dst = m.vf;
            if (fused_dev) {
                ekv.kv_fresh = 2;
                ekv.cmp_k = layer_kv(l);
                ekv.cmp_v = layer_v(l);
                ekv.dev_part = m.dev_part;
                ekv.dev_parts = m.dev_parts;
                ekv.dev_rows = ncmp;
            } else {
                ekv.kv_fresh = 1;
            }
            S.gemm(K_GEMM_KV, xb, 0, rows, d, wsel(m, l, WSEL_KV), 2 * nkv, ekv);
            if (!fused_dev && ncmp > 0)
                S.k(K_DEVIATION, 0, (double)ncmp * 2 * nkv * (4 + es),
                    [&] { return launch_deviation(m, m.kf, m.vf, layer_kv(l), N, pos, ncmp, devd, s); });
        }
        const double tk_bytes = (double)ncmp * 4 * (fused_dev ? m.dev_parts + 1 : 1);
        S.k(K_TOPK, 0, tk_bytes, [&] {
            return launch_topk(m.pdl, fused_dev ? nullptr : devd, m.dev_part, m.dev_parts, devd, ncmp, kk, Q, sel_rows,
                               sel_out, s);
        });
    };
    const double kvrow_bytes = 2.0 * nkv * ((fused_dev ? es : 4.0) + es);   // one row's fresh K/V read, stored
    {
        norm(m.h, m.attn_norm[1], m.x, N);
        layer_in(1);                                 // the comparison reads the re-RoPE'd cache of layer 1
        if (given) {                                 // the caller's set: no comparison at the check layer
            EpiParams ekv = epi_base(m, EPI_QKV, N);
            ekv.qkv_base = nq;
            ekv.k_dst = m.kf;
            ekv.v_dst = m.vf;
            ekv.kv_fresh = fused_dev ? 2 : 1;        // fresh K/V rows only (nothing to compare: dev_rows 0)
            ekv.dev_part = m.dev_part;
            ekv.dev_parts = m.dev_parts;
            S.gemm(K_GEMM_KV, XBUF_X, 0, N, d, wsel(m, 1, WSEL_KV), 2 * nkv, ekv);
            S.k(K_TOPK, 0, (double)k * 4,
                [&] { return launch_given_rows(m.pdl, given, k, n_ctx, Q, m.rows, out_selected, m.status, s); });
        } else {
            compare(1, XBUF_X, N, n_ctx, nullptr, devp, k, m.rows, out_selected);
        }
        S.k(K_GATHER, 0, (double)M * (8.0 * d + 2.0 * d * es * (m.split ? 2 : 1) + kvrow_bytes),
            [&] { return launch_gather(m, m.rows, M, m.h, m.hA, m.x, m.xA, m.x_lo, m.xA_lo, m.kf, m.vf, !fused_dev,
                                       layer_kv(1), N, s); });
        EpiParams e = epi_base(m, EPI_QKV, M);
        e.qkv_base = 0;
        e.pos = m.rows;
        e.q_out = m.q;
        S.gemm(K_GEMM_Q, XBUF_XA, 0, M, d, wsel(m, 1, WSEL_Q), nq, e);
    }

    // ---- layers >= 1: attention of the recomputed rows over the blended K/V, O, MLP ------------
    // The recomputed rows' state lives in one of two buffer sets; a shrinking layer (gradual
    // filtering) compacts the kept rows into the other set.
    float* hc = m.hA;
    int xc = XBUF_XA;
    int* rows_c = m.rows;
    int k_prev = k;
    size_t dev_at = out_dev ? (size_t)n_ctx : 0;     // out_dev: later shrinking layers follow the check layer
    size_t sel_at = (size_t)k;                       // out_selected: likewise
    double attn_total = attn_flops(keys0);
    for (int l = 1; l < L; ++l) {
        const int kl = ks[l];
        const int Mp = k_prev + Q, Ml = kl + Q;
        void* xcp = xc == XBUF_X ? m.x : m.xA;
        if (l >= 2) layer_in(l);
        if (l >= 2 && kl < k_prev) {
            // shrinking layer (Figure 9): fresh K/V of the candidates (and the query), the candidates compared
            // with the re-RoPE'd cache of this layer, the top kl of them, compaction with the kept rows' K/V
            // stored, then Q of the kept rows
            norm(hc, m.attn_norm[l], xcp, Mp);
            float* devl = (out_dev ? out_dev : m.dev) + dev_at;
            compare(l, xc, Mp, k_prev, rows_c, devl, kl, m.sel_local, nullptr);
            float* hn = hc == m.hA ? m.h : m.hA;
            const int xn = xc == XBUF_XA ? XBUF_X : XBUF_XA;
            void* xnp = xn == XBUF_X ? m.x : m.xA;
            int* rows_n = rows_c == m.rows ? m.rows2 : m.rows;
            int* sel_out = out_selected ? out_selected + sel_at : nullptr;
            S.k(K_REFILTER, 0, (double)Ml * (8.0 * d + 2.0 * d * es * (m.split ? 2 : 1) + kvrow_bytes),
                [&] { return launch_refilter(m, m.sel_local, rows_c, rows_n, Ml, kl, sel_out, hc, hn, xcp, xnp,
                                             m.split ? (xc == XBUF_X ? m.x_lo : m.xA_lo) : nullptr,
                                             m.split ? (xn == XBUF_X ? m.x_lo : m.xA_lo) : nullptr, m.kf, m.vf,
                                             !fused_dev, layer_kv(l), N, s); });
            EpiParams e = epi_base(m, EPI_QKV, Ml);
            e.qkv_base = 0;
            e.pos = rows_n;
            e.q_out = m.q;
            S.gemm(K_GEMM_Q, xn, 0, Ml, d, wsel(m, l, WSEL_Q), nq, e);
            if (out_dev) dev_at += (size_t)k_prev;
            sel_at += (size_t)kl;
            hc = hn;
            xc = xn;
            xcp = xnp;
            rows_c = rows_n;
        } else if (l >= 2) {
            norm(hc, m.attn_norm[l], xcp, Ml);
            EpiParams e = epi_base(m, EPI_QKV, Ml);
            e.qkv_base = 0;
            e.pos = rows_c;
            e.q_out = m.q;
            e.k_dst = layer_kv(l);
            e.v_dst = layer_v(l);
            S.gemm(K_GEMM_QKV, xc, 0, Ml, d, wsel(m, l, WSEL_QKV), nq + 2 * nkv, e);
        }
        attend(l, rows_c, Ml, keys_of(kl));
        layer_out(l);
        attn_total += attn_flops(keys_of(kl));
        EpiParams er = epi_base(m, EPI_RESID, Ml);
        er.h = hc;
        er.ldh = d;
        S.gemm(K_GEMM_O, XBUF_ATTN, 0, Ml, nq, wsel(m, l, WSEL_O), d, er);
        resid_done();
        norm(hc, m.mlp_norm[l], xcp, Ml);
        EpiParams eg = epi_base(m, EPI_SWIGLU, Ml);
        eg.act = m.act;
        eg.act_lo = m.act_lo;
        eg.ld_act = F;
        S.gemm(K_GEMM_GATEUP, xc, 0, Ml, d, wsel(m, l, WSEL_GATEUP), F, eg);
        S.gemm(K_GEMM_DOWN, XBUF_ACT, 0, Ml, F, wsel(m, l, WSEL_DOWN), d, er);
        resid_done();
        k_prev = kl;
    }

    // ---- logits of the last row --------------------------------------------------------------
    const int M_last = k_prev + Q;
    const float* h_last = hc + (size_t)(M_last - 1) * d;
    const float* p_last = m.part_h + (size_t)(M_last - 1) * d;
    S.k(K_LOGITS, 2.0 * d * c.vocab, (double)c.vocab * d * es,
        [&] { return launch_logits(m, h_last, p_last, pend, (size_t)M_last * d, out_logits, s); });

    if (pg) {   // every row of the blended K/V into its destination page (a copy-on-write page when shared)
        S.k(K_PAGES, 0, 4.0 * L * N * row,
            [&] { return launch_page_copy(m, out_kv, N, nullptr, pg->pool, pg->n_pages * (int64_t)pg->page_size,
                                          pg->dst_table, page_shift, N, s); });
    }
    if (io) {   // join: the compute stream completes only after every copy
        io_check(cudaEventRecord(m.io_ev[2 * L + 1], cs));
        io_check(cudaStreamWaitEvent(s, m.io_ev[2 * L + 1], 0));
        if (bs != cs) {
            io_check(cudaEventRecord(m.io_ev[2 * L + 2], bs));
            io_check(cudaStreamWaitEvent(s, m.io_ev[2 * L + 2], 0));
        }
    }
    if (io_err != cudaSuccess) return fail(CB_ERR_CUDA, "layer-wise copies: %s", cudaGetErrorString(io_err));
    if (S.err != cudaSuccess) return fail(CB_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(S.err));
    if (stats) {
        stats->n_tokens = N;
        stats->n_ctx = n_ctx;
        stats->n_selected = k;
        stats->n_recompute = M;
        stats->kernel_launches = S.launches;
        stats->reserved = 0;
        stats->gemm_flops = S.gemm_flops + 2.0 * d * (double)c.vocab;
        stats->attn_flops = attn_total;
        double scat = 0;
        for (int l = 1; l < L; ++l) scat += (double)(ks[l] + Q) * 2 * row;
        stats->kv_bytes_moved = (n_chunks ? (inplace ? 2.0 * L * n_ctx * row : 4.0 * L * n_ctx * row) : 0) +
                                (double)n_ctx * 2 * nkv * (fused_dev ? es : 4 + es) + scat;
    }
    return CB_OK;
}

// validation shared by cb_blend and cb_blend_gradual; fills the chunk table and n_ctx
cb_status check_blend(const Model& m, const int32_t* tokens, int32_t n_tokens, const void* cached_kv,
                      const cb_chunk* chunks, int32_t n_chunks, void* out_kv, float* out_logits, ChunkTable& t,
                      int& n_ctx) {
    const cb_config& c = m.cfg;
    if (!tokens || !out_kv || !out_logits) return fail(CB_ERR_INVALID_ARG, "cb_blend: null tokens, out_kv or out_logits");
    if (n_tokens <= 0 || n_tokens > c.max_tokens)
        return fail(CB_ERR_INVALID_ARG, "n_tokens %d outside (0, max_tokens=%d]", n_tokens, c.max_tokens);
    cb_status st = check_chunks(chunks, n_chunks, c.max_chunks, n_ctx, t);
    if (st != CB_OK) return st;
    if (n_ctx >= n_tokens) return fail(CB_ERR_INVALID_ARG, "need at least one query token after the %d context rows", n_ctx);
    if (n_chunks > 0 && !cached_kv) return fail(CB_ERR_INVALID_ARG, "cached_kv is NULL but chunks were given");
    if (n_chunks > 0 && cached_kv != out_kv) {
        // the two buffers may not overlap unless identical
        const size_t es = act_size(m), nkv = (size_t)c.n_kv_heads * c.head_dim;
        const char* a = (const char*)cached_kv;
        const char* b = (const char*)out_kv;
        const size_t abytes = (size_t)c.n_layers * 2 * n_ctx * nkv * es, bbytes = (size_t)c.n_layers * 2 * n_tokens * nkv * es;
        if (a < b + bbytes && b < a + abytes) return fail(CB_ERR_INVALID_ARG, "cached_kv and out_kv overlap");
    }
    return CB_OK;
}

}  // namespace

extern "C" {

cb_status cb_blend(cb_model* mp, const int32_t* tokens, int32_t n_tokens, const void* cached_kv,
                   const cb_chunk* chunks, int32_t n_chunks, double ratio, void* out_kv, float* out_logits,
                   int32_t* out_selected, float* out_dev, cb_stats* stats, void* stream) {
    g_err[0] = 0;
    if (!mp) return fail(CB_ERR_INVALID_ARG, "cb_blend: null model");
    Model& m = *mp;
    if (!(ratio >= 0.0 && ratio <= 1.0)) return fail(CB_ERR_INVALID_ARG, "ratio must be in [0, 1]");
    ChunkTable t;
    int n_ctx = 0;
    cb_status st = check_blend(m, tokens, n_tokens, cached_kv, chunks, n_chunks, out_kv, out_logits, t, n_ctx);
    if (st != CB_OK) return st;
    std::vector<int> ks(m.cfg.n_layers, cb_selected_count(n_ctx, ratio));
    return blend_impl(m, tokens, n_tokens, cached_kv, t, n_chunks, n_ctx, ks, out_kv, out_logits, out_selected,
                      out_dev, stats, (cudaStream_t)stream);
}

cb_status cb_blend_hkvd(cb_model* mp, const int32_t* tokens, int32_t n_tokens, const void* cached_kv,
                        const cb_chunk* chunks, int32_t n_chunks, const int32_t* hkvd, int32_t k, void* out_kv,
                        float* out_logits, cb_stats* stats, void* stream) {
    g_err[0] = 0;
    if (!mp) return fail(CB_ERR_INVALID_ARG, "cb_blend_hkvd: null model");
    Model& m = *mp;
    ChunkTable t;
    int n_ctx = 0;
    cb_status st = check_blend(m, tokens, n_tokens, cached_kv, chunks, n_chunks, out_kv, out_logits, t, n_ctx);
    if (st != CB_OK) return st;
    if (k < 0 || k > n_ctx) return fail(CB_ERR_INVALID_ARG, "cb_blend_hkvd: k %d outside [0, n_ctx = %d]", k, n_ctx);
    if (k > 0 && !hkvd) return fail(CB_ERR_INVALID_ARG, "cb_blend_hkvd: null hkvd with k > 0");
    std::vector<int> ks(m.cfg.n_layers, k);
    // with k = 0 the set is empty and never read; any device pointer marks the given-set path
    return blend_impl(m, tokens, n_tokens, cached_kv, t, n_chunks, n_ctx, ks, out_kv, out_logits, nullptr, nullptr,
                      stats, (cudaStream_t)stream, nullptr, nullptr, 0, k > 0 ? hkvd : m.rows);
}

cb_status cb_blend_streamed(cb_model* mp, const int32_t* tokens, int32_t n_tokens, const cb_layer_io* io,
                            const cb_chunk* chunks, int32_t n_chunks, const double* ratios, int32_t n_ratios,
                            void* out_kv, float* out_logits, int32_t* out_selected, float* out_dev, cb_stats* stats,
                            void* stream) {
    g_err[0] = 0;
    if (!mp) return fail(CB_ERR_INVALID_ARG, "cb_blend_streamed: null model");
    Model& m = *mp;
    const int L = m.cfg.n_layers;
    if (!io) return fail(CB_ERR_INVALID_ARG, "cb_blend_streamed: null io");
    if (!io->copy_stream || io->copy_stream == stream || (io->copy_back_stream && io->copy_back_stream == stream))
        return fail(CB_ERR_INVALID_ARG, "cb_blend_streamed: the copy streams must be streams of their own");
    if (n_chunks > 0 && !io->cached_kv_host) return fail(CB_ERR_INVALID_ARG, "cb_blend_streamed: chunks given but no host cache");
    if (!ratios || n_ratios != L - 1)
        return fail(CB_ERR_INVALID_ARG, "cb_blend_streamed: need n_layers - 1 = %d ratios (got %d)", L - 1, n_ratios);
    for (int i = 0; i < n_ratios; ++i)
        if (!(ratios[i] >= 0.0 && ratios[i] <= 1.0)) return fail(CB_ERR_INVALID_ARG, "ratio of layer %d outside [0, 1]", i + 1);
    ChunkTable t;
    int n_ctx = 0;
    // validated as an in-place blend: the host cache is copied into out_kv's rows
    cb_status st = check_blend(m, tokens, n_tokens, out_kv, chunks, n_chunks, out_kv, out_logits, t, n_ctx);
    if (st != CB_OK) return st;
    std::vector<int> ks(L, 0);
    for (int l = 1; l < L; ++l) {
        ks[l] = cb_selected_count(n_ctx, ratios[l - 1]);
        if (l >= 2 && ks[l] > ks[l - 1])
            return fail(CB_ERR_INVALID_ARG, "layer %d keeps %d rows, more than layer %d's %d: the sets must be nested",
                        l, ks[l], l - 1, ks[l - 1]);
    }
    ks[0] = ks[1];
    if ((int)m.io_ev.size() < 2 * L + 3) {
        for (int i = (int)m.io_ev.size(); i < 2 * L + 3; ++i) {
            cudaEvent_t e;
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
                return fail(CB_ERR_CUDA, "cb_blend_streamed: cudaEventCreate failed");
            m.io_ev.push_back(e);
        }
    }
    return blend_impl(m, tokens, n_tokens, out_kv, t, n_chunks, n_ctx, ks, out_kv, out_logits, out_selected, out_dev,
                      stats, (cudaStream_t)stream, io);
}

static cb_status check_pages(const Model& m, const cb_paged_kv* pg, int& shift) {
    if (!pg || !pg->pool) return fail(CB_ERR_INVALID_ARG, "paged K/V: null pool");
    if (pg->page_size < 16 || (pg->page_size & (pg->page_size - 1)))
        return fail(CB_ERR_INVALID_ARG, "paged K/V: page_size %d is not a power of two >= 16", pg->page_size);
    if (pg->n_pages <= 0 || pg->n_pages * (int64_t)pg->page_size > ((int64_t)1 << 40))
        return fail(CB_ERR_INVALID_ARG, "paged K/V: bad n_pages");
    if ((uintptr_t)pg->pool % 16) return fail(CB_ERR_INVALID_ARG, "paged K/V: pool not 16-byte aligned");
    shift = 0;
    while ((1 << shift) < pg->page_size) ++shift;
    (void)m;
    return CB_OK;
}

cb_status cb_blend_paged(cb_model* mp, const int32_t* tokens, int32_t n_tokens, const cb_paged_kv* pg,
                         const cb_chunk* chunks, int32_t n_chunks, const double* ratios, int32_t n_ratios,
                         void* work_kv, float* out_logits, int32_t* out_selected, float* out_dev, cb_stats* stats,
                         void* stream) {
    g_err[0] = 0;
    if (!mp) return fail(CB_ERR_INVALID_ARG, "cb_blend_paged: null model");
    Model& m = *mp;
    const int L = m.cfg.n_layers;
    int shift = 0;
    cb_status st = check_pages(m, pg, shift);
    if (st != CB_OK) return st;
    if (!pg->dst_table || (n_chunks > 0 && !pg->src_table))
        return fail(CB_ERR_INVALID_ARG, "cb_blend_paged: missing block table");
    if (!ratios || n_ratios != L - 1)
        return fail(CB_ERR_INVALID_ARG, "cb_blend_paged: need n_layers - 1 = %d ratios (got %d)", L - 1, n_ratios);
    for (int i = 0; i < n_ratios; ++i)
        if (!(ratios[i] >= 0.0 && ratios[i] <= 1.0)) return fail(CB_ERR_INVALID_ARG, "ratio of layer %d outside [0, 1]", i + 1);
    ChunkTable t;
    int n_ctx = 0;
    st = check_blend(m, tokens, n_tokens, work_kv, chunks, n_chunks, work_kv, out_logits, t, n_ctx);
    if (st != CB_OK) return st;
    std::vector<int> ks(L, 0);
    for (int l = 1; l < L; ++l) {
        ks[l] = cb_selected_count(n_ctx, ratios[l - 1]);
        if (l >= 2 && ks[l] > ks[l - 1])
            return fail(CB_ERR_INVALID_ARG, "layer %d keeps %d rows, more than layer %d's %d: the sets must be nested",
                        l, ks[l], l - 1, ks[l - 1]);
    }
    ks[0] = ks[1];
    return blend_impl(m, tokens, n_tokens, nullptr, t, n_chunks, n_ctx, ks, work_kv, out_logits, out_selected, out_dev,
                      stats, (cudaStream_t)stream, nullptr, pg, shift);
}

cb_status cb_kv_gather_pages(cb_model* mp, const cb_paged_kv* pg, int32_t n_rows, void* out_kv, void* stream) {
    g_err[0] = 0;
    if (!mp) return fail(CB_ERR_INVALID_ARG, "cb_kv_gather_pages: null model");
    int shift = 0;
    cb_status st = check_pages(*mp, pg, shift);
    if (st != CB_OK) return st;
    if (!pg->src_table || !out_kv || n_rows < 0) return fail(CB_ERR_INVALID_ARG, "cb_kv_gather_pages: bad arguments");
    cudaError_t e = launch_page_copy(*mp, pg->pool, pg->n_pages * (int64_t)pg->page_size, pg->src_table, out_kv, n_rows,
                                     nullptr, shift, n_rows, (cudaStream_t)stream);
    return e == cudaSuccess ? CB_OK : fail(CB_ERR_CUDA, "cb_kv_gather_pages: %s", cudaGetErrorString(e));
}

cb_status cb_kv_scatter_pages(cb_model* mp, const void* kv, int32_t n_rows, const cb_paged_kv* pg, void* stream) {
    g_err[0] = 0;
    if (!mp) return fail(CB_ERR_INVALID_ARG, "cb_kv_scatter_pages: null model");
    int shift = 0;
    cb_status st = check_pages(*mp, pg, shift);
    if (st != CB_OK) return st;
    if (!pg->dst_table || !kv || n_rows < 0) return fail(CB_ERR_INVALID_ARG, "cb_kv_scatter_pages: bad arguments");
    cudaError_t e = launch_page_copy(*mp, kv, n_rows, nullptr, pg->pool, pg->n_pages * (int64_t)pg->page_size,
                                     pg->dst_table, shift, n_rows, (cudaStream_t)stream);
    return e == cudaSuccess ? CB_OK : fail(CB_ERR_CUDA, "cb_kv_scatter_pages: %s", cudaGetErrorString(e));
}

cb_status cb_blend_gradual(cb_model* mp, const int32_t* tokens, int32_t n_tokens, const void* cached_kv,
                           const cb_chunk* chunks, int32_t n_chunks, const double* ratios, int32_t n_ratios,
                           void* out_kv, float* out_logits, int32_t* out_selected, float* out_dev, cb_stats* stats,
                           void* stream) {
    g_err[0] = 0;
    if (!mp) return fail(CB_ERR_INVALID_ARG, "cb_blend_gradual: null model");
    Model& m = *mp;
    const int L = m.cfg.n_layers;
    if (!ratios || n_ratios != L - 1)
        return fail(CB_ERR_INVALID_ARG, "cb_blend_gradual: need n_layers - 1 = %d ratios (got %d)", L - 1, n_ratios);
    for (int i = 0; i < n_ratios; ++i)
        if (!(ratios[i] >= 0.0 && ratios[i] <= 1.0)) return fail(CB_ERR_INVALID_ARG, "ratio of layer %d outside [0, 1]", i + 1);
    ChunkTable t;
    int n_ctx = 0;
    cb_status st = check_blend(m, tokens, n_tokens, cached_kv, chunks, n_chunks, out_kv, out_logits, t, n_ctx);
    if (st != CB_OK) return st;
    std::vector<int> ks(L, 0);
    for (int l = 1; l < L; ++l) {
        ks[l] = cb_selected_count(n_ctx, ratios[l - 1]);
        if (l >= 2 && ks[l] > ks[l - 1])
            return fail(CB_ERR_INVALID_ARG, "layer %d keeps %d rows, more than layer %d's %d: the sets must be nested",
                        l, ks[l], l - 1, ks[l - 1]);
    }
    ks[0] = ks[1];
    return blend_impl(m, tokens, n_tokens, cached_kv, t, n_chunks, n_ctx, ks, out_kv, out_logits, out_selected,
                      out_dev, stats, (cudaStream_t)stream);
}

cb_status cb_select_hkvd(const float* dev, int32_t n, int32_t k, int32_t* out_rows, void* stream) {
    g_err[0] = 0;
    if (n < 0 || k < 0 || k > n) return fail(CB_ERR_INVALID_ARG, "cb_select_hkvd: need 0 <= k <= n (n %d, k %d)", n, k);
    if (k == 0) return CB_OK;
    if (!dev || !out_rows) return fail(CB_ERR_INVALID_ARG, "cb_select_hkvd: null dev or out_rows");
    const cudaError_t e = launch_topk(false, dev, nullptr, 0, nullptr, n, k, 0, out_rows, nullptr, (cudaStream_t)stream);
    return e == cudaSuccess ? CB_OK : fail(CB_ERR_CUDA, "cb_select_hkvd: %s", cudaGetErrorString(e));
}

double cb_load_time(double per_token_kv_bytes, int64_t n_tokens, double throughput_bytes_per_s) {
    if (!(throughput_bytes_per_s > 0) || !(per_token_kv_bytes >= 0) || n_tokens < 0) return -1.0;
    return per_token_kv_bytes * (double)n_tokens / throughput_bytes_per_s;
}

double cb_controller_ratio(double t_prefill_s, double t_load_s, double r_min) {
    if (!(t_prefill_s >= 0) || !(t_load_s >= 0) || !(r_min >= 0 && r_min <= 1)) return -1.0;
    const double r_match = t_prefill_s > 0 ? t_load_s / t_prefill_s : 1.0;
    const double r = r_match > r_min ? r_match : r_min;
    return r < 1.0 ? r : 1.0;
}

int32_t cb_pick_storage(const double* throughput_bytes_per_s, const double* cost_per_gb, int32_t n_devices,
                        double per_token_kv_bytes, int64_t n_tokens, double t_prefill_s, double r_min) {
    g_err[0] = 0;
    if (!throughput_bytes_per_s || !cost_per_gb || n_devices <= 0)
        return (int32_t)fail(CB_ERR_INVALID_ARG, "cb_pick_storage: no devices");
    const double budget = r_min * t_prefill_s;      // the recompute time at the quality floor
    int best = -1, fastest = 0;
    for (int i = 0; i < n_devices; ++i) {
        const double tl = cb_load_time(per_token_kv_bytes, n_tokens, throughput_bytes_per_s[i]);
        if (tl < 0) return (int32_t)fail(CB_ERR_INVALID_ARG, "cb_pick_storage: device %d has no throughput", i);
        if (throughput_bytes_per_s[i] > throughput_bytes_per_s[fastest]) fastest = i;
        if (tl <= budget && (best < 0 || cost_per_gb[i] < cost_per_gb[best])) best = i;
    }
    return best >= 0 ? best : fastest;
}

cb_status cb_model_status(cb_model* m, uint32_t* bits, int32_t clear) {
    g_err[0] = 0;
    if (!m || !bits) return fail(CB_ERR_INVALID_ARG, "cb_model_status: null argument");
    if (cudaDeviceSynchronize() != cudaSuccess) return fail(CB_ERR_CUDA, "cb_model_status: device error");
    unsigned v = 0;
    CB_CUDA(cudaMemcpy(&v, m->status, sizeof v, cudaMemcpyDeviceToHost));
    *bits = v;
    if (clear) CB_CUDA(cudaMemset(m->status, 0, 64));
    return CB_OK;
}

cb_status cb_model_diag(cb_model* m, uint32_t* words) {
    g_err[0] = 0;
    if (!m || !words) return fail(CB_ERR_INVALID_ARG, "cb_model_diag: null argument");
    if (cudaDeviceSynchronize() != cudaSuccess) return fail(CB_ERR_CUDA, "cb_model_diag: device error");
    CB_CUDA(cudaMemcpy(words, m->status, 16 * sizeof(uint32_t), cudaMemcpyDeviceToHost));
    return CB_OK;
}

cb_status cb_profile_enable(cb_model* m, int32_t enable, int32_t max_launches) {
    g_err[0] = 0;
    if (!m) return fail(CB_ERR_INVALID_ARG, "cb_profile_enable: null model");
    Profile& p = m->prof;
    if (enable && p.cap == 0) {
        if (max_launches <= 0) return fail(CB_ERR_INVALID_ARG, "max_launches must be > 0");
        p.ev.resize(2 * (size_t)max_launches);
        for (auto& e : p.ev)
            if (cudaEventCreate(&e) != cudaSuccess) return fail(CB_ERR_CUDA, "cudaEventCreate failed");
        p.cap = max_launches;
    }
    p.on = enable != 0;
    return CB_OK;
}

int32_t cb_profile_read(cb_model* m, cb_kernel_profile* out, int32_t max_entries) {
    g_err[0] = 0;
    if (!m || (!out && max_entries > 0)) return fail(CB_ERR_INVALID_ARG, "cb_profile_read: null argument");
    Profile& p = m->prof;
    if (cudaDeviceSynchronize() != cudaSuccess) return fail(CB_ERR_CUDA, "cb_profile_read: device error");
    double ms[K_NCLASS] = {};
    for (size_t i = 0; i < p.rec_class.size(); ++i) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, p.ev[2 * i], p.ev[2 * i + 1]) == cudaSuccess) ms[p.rec_class[i]] += t;
    }
    int n = 0;
    for (int c = 0; c < K_NCLASS && n < max_entries; ++c) {
        if (!p.launches[c]) continue;
        memset(&out[n], 0, sizeof out[n]);
        snprintf(out[n].name, sizeof out[n].name, "%s", kClassName[c]);
        out[n].launches = p.launches[c];
        out[n].ms = ms[c];
        out[n].flops = p.flops[c];
        out[n].bytes = p.bytes[c];
        ++n;
    }
    p.rec_class.clear();
    for (int c = 0; c < K_NCLASS; ++c) { p.launches[c] = 0; p.flops[c] = 0; p.bytes[c] = 0; }
    return n;
}

}  // extern "C"
