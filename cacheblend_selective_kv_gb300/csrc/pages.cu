// Host-side page bookkeeping of a paged K/V pool: reference counts, allocation and copy-on-write planning
// (CacheBlend deep-dive page, section "和前缀缓存、PagedAttention 的分工": a block shared by several
// requests is copied before the blend writes into it, never modified in place).  Host memory only.
#include <cstdint>
#include <new>
#include <vector>

#include "cb_common.cuh"

struct cb_pages {
    std::vector<int32_t> count;     // reference count per page; 0 = free
    std::vector<int32_t> free_ids;  // free pages, highest id at the front so pops give the lowest first
};

namespace {

bool valid(const cb_pages* p, int32_t id) { return p && id >= 0 && (size_t)id < p->count.size(); }

void push_free(cb_pages* p, int32_t id) { p->free_ids.push_back(id); }

int32_t pop_free(cb_pages* p) {
    // lowest free id (the free list is kept unsorted; pick the minimum)
    size_t best = 0;
    for (size_t i = 1; i < p->free_ids.size(); ++i)
        if (p->free_ids[i] < p->free_ids[best]) best = i;
    const int32_t id = p->free_ids[best];
    p->free_ids[best] = p->free_ids.back();
    p->free_ids.pop_back();
    return id;
}

}  // namespace

extern "C" {

cb_status cb_pages_create(int64_t n_pages, cb_pages** out) {
    if (!out || n_pages <= 0 || n_pages > INT32_MAX) {
        cb::set_last_error("cb_pages_create: bad arguments");
        return CB_ERR_INVALID_ARG;
    }
    cb_pages* p = new (std::nothrow) cb_pages();
    if (!p) return CB_ERR_OOM;
    p->count.assign((size_t)n_pages, 0);
    p->free_ids.reserve((size_t)n_pages);
    for (int64_t i = n_pages - 1; i >= 0; --i) p->free_ids.push_back((int32_t)i);
    *out = p;
    return CB_OK;
}

cb_status cb_pages_destroy(cb_pages* p) {
    delete p;
    return CB_OK;
}

cb_status cb_pages_alloc(cb_pages* p, int32_t n, int32_t* ids) {
    if (!p || n < 0 || (n > 0 && !ids)) {
        cb::set_last_error("cb_pages_alloc: bad arguments");
        return CB_ERR_INVALID_ARG;
    }
    if ((size_t)n > p->free_ids.size()) {
        cb::set_last_error("cb_pages_alloc: not enough free pages");
        return CB_ERR_OOM;
    }
    for (int32_t i = 0; i < n; ++i) {
        ids[i] = pop_free(p);
        p->count[ids[i]] = 1;
    }
    return CB_OK;
}

cb_status cb_pages_retain(cb_pages* p, const int32_t* ids, int32_t n) {
    for (int32_t i = 0; i < n; ++i)
        if (!valid(p, ids[i]) || p->count[ids[i]] <= 0) {
            cb::set_last_error("cb_pages_retain: free or bad page id");
            return CB_ERR_INVALID_ARG;
        }
    for (int32_t i = 0; i < n; ++i) ++p->count[ids[i]];
    return CB_OK;
}

cb_status cb_pages_release(cb_pages* p, const int32_t* ids, int32_t n) {
    for (int32_t i = 0; i < n; ++i)
        if (!valid(p, ids[i]) || p->count[ids[i]] <= 0) {
            cb::set_last_error("cb_pages_release: free or bad page id");
            return CB_ERR_INVALID_ARG;
        }
    // a page listed several times is released that many times; check the totals first
    std::vector<std::pair<int32_t, int32_t>> seen;
    for (int32_t i = 0; i < n; ++i) {
        bool found = false;
        for (auto& s : seen)
            if (s.first == ids[i]) { ++s.second; found = true; break; }
        if (!found) seen.push_back({ids[i], 1});
    }
    for (auto& s : seen)
        if (s.second > p->count[s.first]) {
            cb::set_last_error("cb_pages_release: a page released more often than it is held");
            return CB_ERR_INVALID_ARG;
        }
    for (int32_t i = 0; i < n; ++i)
        if (--p->count[ids[i]] == 0) push_free(p, ids[i]);
    return CB_OK;
}

int32_t cb_pages_plan_write(cb_pages* p, const int32_t* table, int32_t n, int32_t* dst) {
    if (!p || n < 0 || (n > 0 && (!table || !dst))) {
        cb::set_last_error("cb_pages_plan_write: bad arguments");
        return CB_ERR_INVALID_ARG;
    }
    int32_t need = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (!valid(p, table[i]) || p->count[table[i]] <= 0) {
            cb::set_last_error("cb_pages_plan_write: free or bad page id in the table");
            return CB_ERR_INVALID_ARG;
        }
        if (p->count[table[i]] > 1) ++need;
    }
    if ((size_t)need > p->free_ids.size()) {
        cb::set_last_error("cb_pages_plan_write: not enough free pages for copy-on-write");
        return CB_ERR_OOM;
    }
    for (int32_t i = 0; i < n; ++i) {
        if (p->count[table[i]] > 1) {
            dst[i] = pop_free(p);
            p->count[dst[i]] = 1;
            --p->count[table[i]];
        } else {
            dst[i] = table[i];
        }
    }
    return need;
}

int32_t cb_pages_count(const cb_pages* p, int32_t id) { return valid(p, id) ? p->count[id] : -1; }

int64_t cb_pages_free(const cb_pages* p) { return p ? (int64_t)p->free_ids.size() : -1; }

}  // extern "C"
