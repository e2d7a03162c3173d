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
    void* ptrs[] = {m.h, m.hA, m.x, m.xA, m.q, m.attn, m.act, m.kf, m.vf, m.dev, m.rows, m.iota,
                    m.rope, m.inv_freq, m.delta_cs, m.chunk_dst, m.chunk_delta, m.xfinal, m.status};
    for (void* p : ptrs)
        if (p) cudaFree(p);
}

bool fault_injected(const char* what) {
    const char* v = getenv("CB_FAULT_INJECT");
    return v && strcmp(v, what) == 0;
}

}  // namespace

extern "C" {

const char* cb_last_error(void) { return g_err; }

int32_t cb_selected_count(int32_t n_ctx, double ratio) {
    if (!(ratio >= 0.0 && ratio <= 1.0) || n_ctx < 0) return -1;
    double k = std::ceil(ratio * (double)n_ctx - 1e-9);
    if (k < 0) k = 0;
    if (k > n_ctx) k = n_ctx;
    return (int32_t)k;
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
    if (c.n_heads / c.n_kv_heads > 8) return fail(CB_ERR_UNSUPPORTED, "at most 8 query heads per KV head");
    if (c.dtype != CB_F32 && c.dtype != CB_BF16) return fail(CB_ERR_INVALID_ARG, "dtype must be CB_F32 or CB_BF16");
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
    if (cudaGetDevice(&m->device) != cudaSuccess) { delete m; return fail(CB_ERR_CUDA, "no CUDA device"); }
    cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device);
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
    m->kf = m->vf = m->dev = nullptr; m->rows = m->iota = nullptr; m->rope = nullptr; m->inv_freq = nullptr;
    m->delta_cs = nullptr; m->chunk_dst = m->chunk_delta = nullptr; m->xfinal = nullptr; m->status = nullptr;
    m->tc = nullptr;

    const size_t T = (size_t)c.max_tokens, d = c.d_model, nq = (size_t)c.n_heads * c.head_dim;
    const size_t nkv = (size_t)c.n_kv_heads * c.head_dim, F = c.ffn_hidden, half = c.head_dim / 2;
    const size_t as = act_size(*m);
    const size_t mc = c.max_chunks > 0 ? c.max_chunks : 1;
    struct { void** p; size_t bytes; } allocs[] = {
        {(void**)&m->h, T * d * 4}, {(void**)&m->hA, T * d * 4}, {&m->x, T * d * as}, {&m->xA, T * d * as},
        {&m->q, T * nq * as}, {&m->attn, T * nq * as}, {&m->act, T * F * as}, {(void**)&m->kf, T * nkv * 4},
        {(void**)&m->vf, T * nkv * 4}, {(void**)&m->dev, T * 4}, {(void**)&m->rows, T * 4},
        {(void**)&m->iota, T * 4}, {(void**)&m->rope, T * half * sizeof(float2)},
        {(void**)&m->inv_freq, half * sizeof(double)}, {(void**)&m->delta_cs, mc * half * sizeof(float2)},
        {(void**)&m->chunk_dst, mc * 4}, {(void**)&m->chunk_delta, mc * 4}, {(void**)&m->xfinal, d * 4},
        {(void**)&m->status, 16}};
    size_t total = 0;
    for (auto& a : allocs) {
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
    if (m->bf16) {
        std::string err;
        if (!tc_init(*m, err)) m->tc = nullptr;   // CUDA-core path only
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

struct Sched {
    Model& m;
    cudaStream_t s;
    int launches = 0;
    double gemm_flops = 0;
    cudaError_t err = cudaSuccess;
    void ok(cudaError_t e, int n = 1) {
        launches += n;
        if (e != cudaSuccess && err == cudaSuccess) err = e;
    }
    // activation buffer id -> device pointer
    void* xbuf(int id) const {
        switch (id) {
            case XBUF_X: return m.x;
            case XBUF_XA: return m.xA;
            case XBUF_ATTN: return m.attn;
            default: return m.act;
        }
    }
    void gemm(int xb, int row0, int M, int K, const GemmW& w, int N, const EpiParams& e) {
        if (M <= 0 || N <= 0) return;
        gemm_flops += 2.0 * M * (double)N * K * (e.kind == EPI_SWIGLU ? 2 : 1);
        if (m.tc) {
            int n = 0;
            ok(launch_gemm_tc(m, xb, row0, M, K, w, N, e, s, &n), 0);
            launches += n;
        } else {
            const char* base = (const char*)xbuf(xb) + (size_t)row0 * K * act_size(m);
            ok(launch_gemm_simt(m, base, M, K, w, N, e, s));
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
    CB_CUDA(launch_delta_table(*m, t, s));
    CB_CUDA(launch_rerope(*m, kv, kv, n_rows, n_rows, n_ctx, n_chunks, false, s));
    return CB_OK;
}

cb_status cb_blend(cb_model* mp, const int32_t* tokens, int32_t n_tokens, const void* cached_kv,
                   const cb_chunk* chunks, int32_t n_chunks, double ratio, void* out_kv, float* out_logits,
                   int32_t* out_selected, float* out_dev, cb_stats* stats, void* stream) {
    g_err[0] = 0;
    if (!mp) return fail(CB_ERR_INVALID_ARG, "cb_blend: null model");
    Model& m = *mp;
    const cb_config& c = m.cfg;
    if (!tokens || !out_kv || !out_logits) return fail(CB_ERR_INVALID_ARG, "cb_blend: null tokens, out_kv or out_logits");
    if (n_tokens <= 0 || n_tokens > c.max_tokens)
        return fail(CB_ERR_INVALID_ARG, "n_tokens %d outside (0, max_tokens=%d]", n_tokens, c.max_tokens);
    if (!(ratio >= 0.0 && ratio <= 1.0)) return fail(CB_ERR_INVALID_ARG, "ratio must be in [0, 1]");
    ChunkTable t;
    int n_ctx = 0;
    cb_status st = check_chunks(chunks, n_chunks, c.max_chunks, n_ctx, t);
    if (st != CB_OK) return st;
    if (n_ctx >= n_tokens) return fail(CB_ERR_INVALID_ARG, "need at least one query token after the %d context rows", n_ctx);
    if (n_chunks > 0 && !cached_kv) return fail(CB_ERR_INVALID_ARG, "cached_kv is NULL but chunks were given");
    const size_t es = act_size(m);
    const int L = c.n_layers, d = c.d_model, nq = c.n_heads * c.head_dim, nkv = c.n_kv_heads * c.head_dim;
    const int F = c.ffn_hidden, N = n_tokens, Q = N - n_ctx;
    const bool inplace = n_chunks > 0 && cached_kv == out_kv;
    if (n_chunks > 0 && !inplace) {
        // the two buffers may not overlap unless identical
        const char* a = (const char*)cached_kv;
        const char* b = (const char*)out_kv;
        const size_t abytes = (size_t)L * 2 * n_ctx * nkv * es, bbytes = (size_t)L * 2 * N * nkv * es;
        if (a < b + bbytes && b < a + abytes) return fail(CB_ERR_INVALID_ARG, "cached_kv and out_kv overlap");
    }
    const int k = cb_selected_count(n_ctx, ratio);
    const int M = k + Q;

    cudaStream_t s = (cudaStream_t)stream;
    Sched S{m, s};
    char* kvb = (char*)out_kv;
    auto layer_kv = [&](int l) { return (void*)(kvb + (size_t)l * 2 * N * nkv * es); };
    auto layer_v = [&](int l) { return (void*)(kvb + ((size_t)l * 2 + 1) * N * nkv * es); };

    // re-RoPE placement of the chunk caches (section "位置恢复、KV 存储与加载流水线")
    if (n_chunks > 0) {
        S.ok(launch_delta_table(m, t, s));
        S.ok(launch_rerope(m, cached_kv, out_kv, inplace ? N : n_ctx, N, n_ctx, n_chunks, !inplace, s));
    }
    S.ok(launch_embed(m, tokens, N, m.h, s));

    // ---- layer 0: every row's hidden state; context K/V reused, query K/V fresh --------------
    {
        S.ok(launch_rmsnorm(m, m.h, m.attn_norm[0], m.x, N, s));
        EpiParams e = epi_base(m, EPI_QKV, N);
        e.qkv_base = 0;
        e.q_out = m.q;
        S.gemm(XBUF_X, 0, N, d, wsel(m, 0, WSEL_Q), nq, e);
        EpiParams ekv = epi_base(m, EPI_QKV, Q);
        ekv.qkv_base = nq;
        ekv.pos_offset = n_ctx;
        ekv.k_dst = layer_kv(0);
        ekv.v_dst = layer_v(0);
        S.gemm(XBUF_X, n_ctx, Q, d, wsel(m, 0, WSEL_KV), 2 * nkv, ekv);
        S.ok(launch_attention(m, m.q, nullptr, N, layer_kv(0), N, N, m.attn, s));
        EpiParams er = epi_base(m, EPI_RESID, N);
        er.h = m.h;
        er.ldh = d;
        S.gemm(XBUF_ATTN, 0, N, nq, wsel(m, 0, WSEL_O), d, er);
        S.ok(launch_rmsnorm(m, m.h, m.mlp_norm[0], m.x, N, s));
        EpiParams eg = epi_base(m, EPI_SWIGLU, N);
        eg.act = m.act;
        eg.ld_act = F;
        S.gemm(XBUF_X, 0, N, d, wsel(m, 0, WSEL_GATEUP), F, eg);
        S.gemm(XBUF_ACT, 0, N, F, wsel(m, 0, WSEL_DOWN), d, er);
    }

    // ---- check layer 1: fresh K/V of every row, deviation, top-k, then the chosen rows --------
    float* devp = out_dev ? out_dev : m.dev;
    {
        S.ok(launch_rmsnorm(m, m.h, m.attn_norm[1], m.x, N, s));
        EpiParams ekv = epi_base(m, EPI_QKV, N);
        ekv.qkv_base = nq;
        ekv.kv_fresh = 1;
        ekv.k_dst = m.kf;
        ekv.v_dst = m.vf;
        S.gemm(XBUF_X, 0, N, d, wsel(m, 1, WSEL_KV), 2 * nkv, ekv);
        if (n_ctx > 0) S.ok(launch_deviation(m, m.kf, m.vf, layer_kv(1), N, n_ctx, devp, s));
        S.ok(launch_topk(m, devp, n_ctx, k, Q, m.rows, out_selected, s));
        S.ok(launch_gather_scatter(m, m.rows, M, m.h, m.hA, m.x, m.xA, m.kf, m.vf, layer_kv(1), N, s));
        EpiParams e = epi_base(m, EPI_QKV, M);
        e.qkv_base = 0;
        e.pos = m.rows;
        e.q_out = m.q;
        S.gemm(XBUF_XA, 0, M, d, wsel(m, 1, WSEL_Q), nq, e);
    }

    // ---- layers >= 1: attention of the recomputed rows over the blended K/V, O, MLP ------------
    for (int l = 1; l < L; ++l) {
        if (l >= 2) {
            S.ok(launch_rmsnorm(m, m.hA, m.attn_norm[l], m.xA, M, s));
            EpiParams e = epi_base(m, EPI_QKV, M);
            e.qkv_base = 0;
            e.pos = m.rows;
            e.q_out = m.q;
            e.k_dst = layer_kv(l);
            e.v_dst = layer_v(l);
            S.gemm(XBUF_XA, 0, M, d, wsel(m, l, WSEL_QKV), nq + 2 * nkv, e);
        }
        S.ok(launch_attention(m, m.q, m.rows, M, layer_kv(l), N, N, m.attn, s));
        EpiParams er = epi_base(m, EPI_RESID, M);
        er.h = m.hA;
        er.ldh = d;
        S.gemm(XBUF_ATTN, 0, M, nq, wsel(m, l, WSEL_O), d, er);
        S.ok(launch_rmsnorm(m, m.hA, m.mlp_norm[l], m.xA, M, s));
        EpiParams eg = epi_base(m, EPI_SWIGLU, M);
        eg.act = m.act;
        eg.ld_act = F;
        S.gemm(XBUF_XA, 0, M, d, wsel(m, l, WSEL_GATEUP), F, eg);
        S.gemm(XBUF_ACT, 0, M, F, wsel(m, l, WSEL_DOWN), d, er);
    }

    // ---- logits of the last row --------------------------------------------------------------
    S.ok(launch_logits(m, m.hA + (size_t)(M - 1) * d, out_logits, s));

    if (S.err != cudaSuccess) return fail(CB_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(S.err));
    if (stats) {
        stats->n_tokens = N;
        stats->n_ctx = n_ctx;
        stats->n_selected = k;
        stats->n_recompute = M;
        stats->kernel_launches = S.launches;
        stats->reserved = 0;
        stats->gemm_flops = S.gemm_flops + 2.0 * d * (double)c.vocab;
        // causal key counts: layer 0 sees sum_{r<N}(r+1); later layers the query rows exactly and
        // the selected rows at the mean context position (their exact positions stay on the device)
        const double l0 = (double)N * (N + 1) / 2.0;
        const double qk = (double)Q * (n_ctx + 1) + (double)Q * (Q - 1) / 2.0 + (double)k * (n_ctx + 1) / 2.0;
        stats->attn_flops = 4.0 * c.head_dim * c.n_heads * (l0 + (L - 1) * qk);
        const double row = (double)nkv * es;
        stats->kv_bytes_moved = (n_chunks ? (inplace ? 2.0 * L * n_ctx * row : 4.0 * L * n_ctx * row) : 0) +
                                (double)n_ctx * 2 * nkv * (4 + es) + (double)(L - 1) * M * 2 * row;
    }
    return CB_OK;
}

}  // extern "C"
