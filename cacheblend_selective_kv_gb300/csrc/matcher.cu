// GPU fragment matcher (LMCache coordinator blend-index page: sections "四、数据结构与召回" and "六、HTTP 接口"):
// which indexed chunks a request's tokens contain, and where.  The index is built once on the host and
// mirrored on the device; a match is two launches on the caller's stream:
//   window_kernel   one thread per probed position: the window's 64-bit polynomial fingerprint (Horner's
//                   rule modulo 2^64, base 0x9E3779B97F4A7C15, the page's fleet constant), the occupancy
//                   filter, a binary search of the sorted fingerprints, a check that some occupant belongs
//                   to the requester's namespace, then the token-by-token verification
//   assign_kernel   one CTA: the verified windows in position order; the t-th verified window of a content
//                   takes that content's t-th occupant in the requester's namespace (each occupant matches
//                   at most once, at its first place), ranks counted per block of 1024 windows with a
//                   running count per content; then leftmost-greedy non-overlap as a successor chain
//                   (binary search per match, one walk over the kept matches)
#include <algorithm>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "cb_common.cuh"

struct cb_index {
    int chunk_size = 0, n_contents = 0, n_occupants = 0, max_tokens = 0;
    int filter_bits = 0;
    unsigned long long* fps = nullptr;     // [n_contents] ascending
    uint32_t* tokens = nullptr;            // [n_contents][chunk_size]
    int* occ_begin = nullptr;              // [n_contents + 1]
    int* occ_id = nullptr;                 // [n_occupants], first-indexing order within a content
    int* occ_old = nullptr;
    int* occ_ns = nullptr;
    unsigned char* slots = nullptr;        // [2^filter_bits] occupancy filter
    int* hits = nullptr;                   // scratch [max_tokens]: verified content per probe, or -1
    int* list = nullptr;                   // scratch [2 * max_tokens]: (probe, content) of verified probes
    int* matches = nullptr;                // scratch [3 * max_tokens]
    int* seen = nullptr;                   // scratch [n_contents]: verified probes of each content so far
    int* vidx = nullptr;                   // scratch [max_tokens]: matches that took an occupant
    int* nxt = nullptr;                    // scratch [max_tokens]: leftmost-greedy successor of each
    int n_indexed = 0;
};

namespace cb {
namespace {

constexpr unsigned long long kPolyBase = 0x9E3779B97F4A7C15ull;
constexpr int kAssignThreads = 1024;

__global__ void window_kernel(const int32_t* __restrict__ tok, int n_probe, int stride, int C,
                              const unsigned long long* __restrict__ fps, int n_contents,
                              const uint32_t* __restrict__ ctoks, const int* __restrict__ occ_begin,
                              const int* __restrict__ occ_ns, const unsigned char* __restrict__ slots,
                              unsigned long long slot_mask, int ns, int* __restrict__ hits) {
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= n_probe) return;
    const int32_t* w = tok + (size_t)p * stride;
    unsigned long long h = 0;
    for (int j = 0; j < C; ++j) h = h * kPolyBase + (unsigned long long)(uint32_t)w[j];
    int hit = -1;
    if (slots[h & slot_mask]) {
        int lo = 0, hi = n_contents - 1;                        // lower bound of h
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (fps[mid] < h) lo = mid + 1; else hi = mid;
        }
        if (n_contents > 0 && fps[lo] == h) {
            bool mine = false;                                  // an occupant the requester may use
            for (int o = occ_begin[lo]; o < occ_begin[lo + 1] && !mine; ++o) mine = occ_ns[o] == ns;
            if (mine) {
                const uint32_t* c = ctoks + (size_t)lo * C;
                bool eq = true;
                for (int j = 0; j < C && eq; ++j) eq = (uint32_t)w[j] == c[j];
                if (eq) hit = lo;
            }
        }
    }
    hits[p] = hit;
}

// exclusive block-wide prefix count of `flag`, and the block total
__device__ __forceinline__ int block_count(bool flag, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned b = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(b & ((1u << lane) - 1u));
    __syncthreads();
    if (lane == 0) warp_tot[warp] = __popc(b);
    __syncthreads();
    if (warp == 0) {
        const int v = warp_tot[lane];
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        warp_tot[lane] = incl - v;
        if (lane == 31) warp_tot[32] = incl;
    }
    __syncthreads();
    total = warp_tot[32];
    return warp_tot[warp] + in_warp;
}

__global__ void __launch_bounds__(kAssignThreads)
    assign_kernel(const int* __restrict__ hits, int n_probe, int stride, int C, const int* __restrict__ occ_begin,
                  const int* __restrict__ occ_id, const int* __restrict__ occ_old, const int* __restrict__ occ_ns,
                  int n_contents, int ns, int greedy, int* __restrict__ list, int* __restrict__ matches,
                  int* __restrict__ seen, int* __restrict__ vidx, int* __restrict__ nxt, int32_t* __restrict__ out,
                  int max_out, int32_t* __restrict__ out_count) {
    __shared__ int warp_tot[33];
    __shared__ int blk_c[kAssignThreads];
    const int tid = threadIdx.x;
    for (int c = tid; c < n_contents; c += kAssignThreads) seen[c] = 0;
    // verified probes in position order: list[2i] = probe, list[2i+1] = content
    int n = 0;
    for (int t0 = 0; t0 < n_probe; t0 += kAssignThreads) {
        const int p = t0 + tid;
        const int c = p < n_probe ? hits[p] : -1;
        int tot;
        const int at = block_count(c >= 0, warp_tot, tot);
        if (c >= 0) {
            list[2 * (n + at)] = p;
            list[2 * (n + at) + 1] = c;
        }
        n += tot;
    }
    __syncthreads();
    // the rank of each verified probe among the earlier ones of its content -> that occupant.  Blocks of
    // probes in position order: within a block the rank counts the earlier probes of the block with the
    // same content; seen[c] carries the count of content c over the earlier blocks
    for (int b0 = 0; b0 < n; b0 += kAssignThreads) {
        const int i = b0 + tid, nb = min(kAssignThreads, n - b0);
        const int c = i < n ? list[2 * i + 1] : -1;
        blk_c[tid] = c;
        __syncthreads();
        int rank = 0, pick = -1;
        bool last = true;
        if (i < n) {
            for (int j = 0; j < tid; ++j) rank += blk_c[j] == c;
            for (int j = tid + 1; j < nb && last; ++j) last = blk_c[j] != c;
            rank += seen[c];
            int r = rank;
            for (int o = occ_begin[c]; o < occ_begin[c + 1]; ++o)
                if (occ_ns[o] == ns && r-- == 0) { pick = o; break; }
            matches[3 * i] = pick >= 0 ? occ_id[pick] : -1;
            matches[3 * i + 1] = pick >= 0 ? occ_old[pick] : 0;
            matches[3 * i + 2] = list[2 * i] * stride;
        }
        __syncthreads();                               // every rank of this block read seen[] first
        if (i < n && last) seen[c] = rank + 1;         // the block's last probe of c carries its count on
        __syncthreads();
    }
    // matches that took an occupant, in position order
    int m = 0;
    for (int t0 = 0; t0 < n; t0 += kAssignThreads) {
        const int i = t0 + tid;
        const bool ok = i < n && matches[3 * i] >= 0;
        int tot;
        const int at = block_count(ok, warp_tot, tot);
        if (ok) vidx[m + at] = i;
        m += tot;
    }
    __syncthreads();
    if (!greedy) {
        for (int v = tid; v < m && v < max_out; v += kAssignThreads) {
            const int i = vidx[v];
            out[3 * v] = matches[3 * i];
            out[3 * v + 1] = matches[3 * i + 1];
            out[3 * v + 2] = matches[3 * i + 2];
        }
        if (tid == 0) *out_count = m;
        return;
    }
    // leftmost-greedy: after a kept match at cur, the next kept one is the first that starts at or after
    // cur + C.  nxt[v] (binary search over the ascending starts) links each match to that successor; the
    // kept matches are the chain from the first one (at most n_tokens / C links)
    for (int v = tid; v < m; v += kAssignThreads) {
        const int want = matches[3 * vidx[v] + 2] + C;
        int lo = v + 1, hi = m;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (matches[3 * vidx[mid] + 2] < want) lo = mid + 1; else hi = mid;
        }
        nxt[v] = lo;
    }
    __syncthreads();
    if (tid == 0) {
        int k = 0;
        for (int v = 0; v < m; v = nxt[v]) {
            const int i = vidx[v];
            if (k < max_out) {
                out[3 * k] = matches[3 * i];
                out[3 * k + 1] = matches[3 * i + 1];
                out[3 * k + 2] = matches[3 * i + 2];
            }
            ++k;
        }
        *out_count = k;
    }
}

unsigned long long host_fingerprint(const uint32_t* t, int C) {
    unsigned long long h = 0;
    for (int j = 0; j < C; ++j) h = h * kPolyBase + t[j];
    return h;
}

void free_index(cb_index* x) {
    void* ptrs[] = {x->fps, x->tokens, x->occ_begin, x->occ_id, x->occ_old, x->occ_ns, x->slots, x->hits,
                    x->list, x->matches, x->seen, x->vidx, x->nxt};
    for (void* p : ptrs)
        if (p) cudaFree(p);
    delete x;
}

}  // namespace
}  // namespace cb

extern "C" {

cb_status cb_index_create(int32_t chunk_size, const uint32_t* tokens, const int32_t* occ_ids, const int32_t* old_st,
                          const int32_t* ns, int32_t n_chunks, int32_t max_tokens, cb_index** out) {
    using namespace cb;
    if (!out || chunk_size <= 0 || n_chunks < 0 || max_tokens <= 0 || (n_chunks > 0 && (!tokens || !occ_ids ||
                                                                                         !old_st || !ns))) {
        set_last_error("cb_index_create: bad arguments");
        return CB_ERR_INVALID_ARG;
    }
    *out = nullptr;
    // contents in first-indexing order; a fingerprint names the first content stored under it
    struct Content { unsigned long long fp; int first; std::vector<int> occ; };
    std::vector<Content> cont;
    std::unordered_map<unsigned long long, int> by_fp;
    int indexed = 0;
    for (int i = 0; i < n_chunks; ++i) {
        if (old_st[i] < 0) continue;                       // no stored position: not indexed
        const uint32_t* t = tokens + (size_t)i * chunk_size;
        const unsigned long long fp = host_fingerprint(t, chunk_size);
        auto it = by_fp.find(fp);
        if (it == by_fp.end()) {
            by_fp.emplace(fp, (int)cont.size());
            cont.push_back({fp, i, {i}});
            ++indexed;
        } else {
            Content& c = cont[it->second];
            if (memcmp(tokens + (size_t)c.first * chunk_size, t, (size_t)chunk_size * 4) != 0) continue;
            c.occ.push_back(i);
            ++indexed;
        }
    }
    std::sort(cont.begin(), cont.end(), [](const Content& a, const Content& b) { return a.fp < b.fp; });
    const int nc = (int)cont.size();
    std::vector<unsigned long long> fps(nc);
    std::vector<uint32_t> ctok((size_t)nc * chunk_size);
    std::vector<int> begin(nc + 1, 0), oid, oold, ons;
    for (int c = 0; c < nc; ++c) {
        fps[c] = cont[c].fp;
        memcpy(&ctok[(size_t)c * chunk_size], tokens + (size_t)cont[c].first * chunk_size, (size_t)chunk_size * 4);
        for (int i : cont[c].occ) {
            oid.push_back(occ_ids[i]);
            oold.push_back(old_st[i]);
            ons.push_back(ns[i]);
        }
        begin[c + 1] = (int)oid.size();
    }
    int bits = 4;                                          // at least 16 slots per content
    while ((1ll << bits) < 16ll * std::max(nc, 1)) ++bits;
    std::vector<unsigned char> slots((size_t)1 << bits, 0);
    for (int c = 0; c < nc; ++c) slots[fps[c] & ((1ull << bits) - 1)] = 1;

    cb_index* x = new (std::nothrow) cb_index();
    if (!x) return CB_ERR_OOM;
    x->chunk_size = chunk_size;
    x->n_contents = nc;
    x->n_occupants = (int)oid.size();
    x->max_tokens = max_tokens;
    x->filter_bits = bits;
    x->n_indexed = indexed;
    const size_t no = std::max<size_t>(oid.size(), 1), ncs = std::max(nc, 1);
    struct { void** p; size_t bytes; const void* src; size_t n; } a[] = {
        {(void**)&x->fps, ncs * 8, fps.data(), fps.size() * 8},
        {(void**)&x->tokens, ncs * chunk_size * 4, ctok.data(), ctok.size() * 4},
        {(void**)&x->occ_begin, (size_t)(nc + 1) * 4, begin.data(), begin.size() * 4},
        {(void**)&x->occ_id, no * 4, oid.data(), oid.size() * 4},
        {(void**)&x->occ_old, no * 4, oold.data(), oold.size() * 4},
        {(void**)&x->occ_ns, no * 4, ons.data(), ons.size() * 4},
        {(void**)&x->slots, slots.size(), slots.data(), slots.size()},
        {(void**)&x->hits, (size_t)max_tokens * 4, nullptr, 0},
        {(void**)&x->list, (size_t)2 * max_tokens * 4, nullptr, 0},
        {(void**)&x->matches, (size_t)3 * max_tokens * 4, nullptr, 0},
        {(void**)&x->seen, ncs * 4, nullptr, 0},
        {(void**)&x->vidx, (size_t)max_tokens * 4, nullptr, 0},
        {(void**)&x->nxt, (size_t)max_tokens * 4, nullptr, 0}};
    for (auto& e : a) {
        if (cudaMalloc(e.p, e.bytes) != cudaSuccess ||
            (e.n && cudaMemcpy(*e.p, e.src, e.n, cudaMemcpyHostToDevice) != cudaSuccess)) {
            cudaGetLastError();
            free_index(x);
            set_last_error("cb_index_create: device allocation or upload failed");
            return CB_ERR_OOM;
        }
    }
    *out = x;
    return CB_OK;
}

cb_status cb_index_destroy(cb_index* x) {
    if (x) {
        cudaDeviceSynchronize();
        cb::free_index(x);
    }
    return CB_OK;
}

int32_t cb_index_size(const cb_index* x, int32_t what) {
    if (!x) return -1;
    switch (what) {
        case 0: return x->n_contents;
        case 1: return x->n_occupants;
        case 2: return x->n_indexed;
        default: return x->chunk_size;
    }
}

cb_status cb_index_match(cb_index* x, const int32_t* tokens, int32_t n_tokens, int32_t ns, int32_t probe_stride,
                         int32_t leftmost_greedy, int32_t* out, int32_t max_out, int32_t* out_count, void* stream) {
    using namespace cb;
    if (!x || !out_count || n_tokens < 0 || probe_stride <= 0 || max_out < 0 || (max_out > 0 && !out) ||
        (n_tokens > 0 && !tokens)) {
        set_last_error("cb_index_match: bad arguments");
        return CB_ERR_INVALID_ARG;
    }
    if (n_tokens > x->max_tokens) {
        set_last_error("cb_index_match: n_tokens exceeds the index's max_tokens");
        return CB_ERR_INVALID_ARG;
    }
    cudaStream_t s = (cudaStream_t)stream;
    const int C = x->chunk_size;
    const int n_probe = n_tokens >= C ? (n_tokens - C) / probe_stride + 1 : 0;
    if (n_probe > 0)
        window_kernel<<<(n_probe + 255) / 256, 256, 0, s>>>(tokens, n_probe, probe_stride, C, x->fps, x->n_contents,
                                                            x->tokens, x->occ_begin, x->occ_ns, x->slots,
                                                            (1ull << x->filter_bits) - 1, ns, x->hits);
    assign_kernel<<<1, kAssignThreads, 0, s>>>(x->hits, n_probe, probe_stride, C, x->occ_begin, x->occ_id, x->occ_old,
                                               x->occ_ns, x->n_contents, ns, leftmost_greedy ? 1 : 0, x->list,
                                               x->matches, x->seen, x->vidx, x->nxt, out, max_out, out_count);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        return CB_ERR_CUDA;
    }
    return CB_OK;
}

}  // extern "C"
