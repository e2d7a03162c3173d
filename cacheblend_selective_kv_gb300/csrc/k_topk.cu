// HKVD selection: the k context rows of largest deviation (ties to the lower row), written in
// ascending row order, followed by the query rows -- the recomputed set of every later layer
// (CacheBlend deep-dive page, section "选 token:HKVD、逐层过滤与 15% 这个经验值").
//
// One cluster of TK_CTAS CTAs of 1024 threads; CTA r owns a contiguous range of rows.
//   1. Each row's deviation: the per-warp partial sums the check-layer GEMM epilogue wrote
//      (KV deviation, section "核心思想"), added in a fixed order -- or a given deviation array.  The
//      sums are written to `dev` (the caller's out_dev or the workspace).
//   2. A non-negative float's bit pattern orders like the float, so the k-th largest key is found by
//      an MSB-first radix select: 4 passes of 8-bit digits; each CTA counts its rows into a shared
//      histogram, and every CTA adds the TK_CTAS histograms (distributed shared memory, in rank order)
//      and takes the same digit.
//   3. Every CTA counts its rows above the threshold key and equal to it; from the counts of the lower
//      ranks it knows how many tied rows precede it and where its rows go, and compacts them in index
//      order with ballot/popc block scans.
// The result is identical to a stable sort by decreasing deviation, whatever the number of CTAs.
#include "cb_ptx.cuh"

namespace cb {

static constexpr int TK_THREADS = 1024;
static constexpr int TK_CTAS = 8;

__device__ __forceinline__ unsigned dev_key(float v) {
    // +0 and positive floats order as their bits; anything else (NaN, -0) ranks as 0
    return v > 0.f ? __float_as_uint(v) : 0u;
}

// exclusive block-wide count of `flag` among lower threads, and the block total
__device__ __forceinline__ int block_excl_count(bool flag, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned b = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(b & ((1u << lane) - 1u));
    __syncthreads();                                   // warp_tot reuse guard
    if (lane == 0) warp_tot[warp] = __popc(b);
    __syncthreads();
    if (warp == 0) {
        int v = warp_tot[lane];
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        warp_tot[lane] = incl - v;                     // exclusive per-warp offsets
        if (lane == 31) warp_tot[32] = incl;
    }
    __syncthreads();
    total = warp_tot[32];
    return warp_tot[warp] + in_warp;
}

// a load from another CTA's shared memory (distributed shared memory); callers order it after a cluster
// barrier, itself a compiler barrier
__device__ __forceinline__ unsigned ld_cluster_u32(uint32_t caddr) {
    unsigned v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(caddr));
    return v;
}

struct TopkArgs {
    const float* dev_in;    // deviations [n] (NULL: sum dev_part)
    const float* dev_part;  // [n][parts] partial sums (when dev_in is NULL)
    int parts;
    float* dev;             // [n] the deviations used (written when summed from partials)
    int n, k, n_query;
    int* rows;              // [k + n_query]: selected rows ascending, then n .. n + n_query - 1
    int* out_sel;           // [k] or NULL
};

__global__ void __cluster_dims__(TK_CTAS, 1, 1) __launch_bounds__(TK_THREADS) topk_kernel(const TopkArgs a) {
    grid_dep_launch();
    grid_dep_wait();
    __shared__ unsigned hist[2][256];
    __shared__ unsigned tot[256];                      // cluster-wide count of each digit
    __shared__ int warp_tot[33];
    __shared__ unsigned cnt[2];                        // this CTA's rows above / equal to the threshold
    __shared__ unsigned s_digit;
    __shared__ int s_remaining;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = ptx::cluster_rank();
    const int per = (a.n + TK_CTAS - 1) / TK_CTAS;
    const int lo = min(a.n, (int)rank * per), hi = min(a.n, lo + per);

    if (rank == 0)   // the query rows always follow the k selected rows
        for (int i = tid; i < a.n_query; i += TK_THREADS) a.rows[a.k + i] = a.n + i;

    // 1. deviations of this CTA's rows: a warp adds a row's partials (lane i takes slots i, i + 32, ...)
    //    and reduces them by a fixed butterfly, so the order is the same on every run; eight rows per warp
    //    at a time keep their loads in flight together
    const float* dev = a.dev_in;
    if (!dev) {
        constexpr int RW = 8;
        constexpr int NW = TK_THREADS / 32;
        for (int r0 = lo + warp * RW; r0 < hi; r0 += NW * RW) {
            float v[RW];
#pragma unroll
            for (int j = 0; j < RW; ++j) {
                v[j] = 0.f;
                if (r0 + j < hi) {
                    const float* p = a.dev_part + (size_t)(r0 + j) * a.parts;
                    for (int i = lane; i < a.parts; i += 32) v[j] += p[i];
                }
            }
#pragma unroll
            for (int j = 0; j < RW; ++j) {
                const float t = warp_sum(v[j]);
                if (lane == 0 && r0 + j < hi) a.dev[r0 + j] = t;
            }
        }
        __syncthreads();                               // this CTA's own writes, read back below
        dev = a.dev;
    }
    if (a.k <= 0) return;

    // 2. radix select of the k-th largest key over the whole cluster
    unsigned prefix = 0, mask = 0;
    int remaining = a.k;                               // how many still to take at the current prefix
    for (int pass = 0, shift = 24; shift >= 0; ++pass, shift -= 8) {
        unsigned* h = hist[pass & 1];
        for (int b = tid; b < 256; b += TK_THREADS) h[b] = 0;
        __syncthreads();
        // warp-aggregated counting: the lanes of a warp that fall into the same digit add once (the leading
        // digits of nearby deviations coincide, so plain per-lane atomics would serialise on a few bins)
        for (int j0 = lo + (tid & ~31); j0 < hi; j0 += TK_THREADS) {
            const int j = j0 + lane;
            const unsigned key = j < hi ? dev_key(dev[j]) : 0u;
            const bool in = j < hi && (key & mask) == prefix;
            const unsigned bin = in ? (key >> shift) & 255u : 256u + lane;   // lanes out of the pass stay alone
            const unsigned same = __match_any_sync(0xffffffffu, bin);
            if (in && lane == __ffs(same) - 1) atomicAdd(&h[bin], (unsigned)__popc(same));
        }
        ptx::cluster_sync();                           // every CTA's histogram of this pass is complete
        if (tid < 256) {                               // digit tid over the cluster, added in rank order
            uint32_t src[TK_CTAS];
            unsigned v[TK_CTAS];
#pragma unroll
            for (int q = 0; q < TK_CTAS; ++q) src[q] = ptx::map_to_rank(ptx::smem_u32(h + tid), (uint32_t)q);
#pragma unroll
            for (int q = 0; q < TK_CTAS; ++q) v[q] = ld_cluster_u32(src[q]);
            unsigned c = 0;
#pragma unroll
            for (int q = 0; q < TK_CTAS; ++q) c += v[q];
            tot[tid] = c;
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns digits 8l .. 8l+7
            unsigned c[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = tot[8 * lane + i];
            unsigned own = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) own += c[i];
            // rows in digits above this lane's range: the sum over higher lanes
            unsigned above = own;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned t = __shfl_down_sync(0xffffffffu, above, o);
                if (lane + o < 32) above += t;
            }
            above -= own;
            // the digit holding the remaining-th largest key lies in the lane whose range crosses it
            const bool hit = above < (unsigned)remaining && above + own >= (unsigned)remaining;
            if (hit) {
                unsigned acc = above, dsel = 8 * lane;
                for (int i = 7; i >= 0; --i) {
                    if (acc + c[i] >= (unsigned)remaining) { dsel = 8 * lane + i; break; }
                    acc += c[i];
                }
                s_digit = dsel;
                s_remaining = remaining - (int)acc;
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        mask |= 255u << shift;
        remaining = s_remaining;
        __syncthreads();
    }

    // 3. the threshold key T: every key > T, and the first `remaining` keys == T in row order
    const unsigned T = prefix;
    {
        __shared__ unsigned red[2][32];
        unsigned gt = 0, eq = 0;
        for (int j = lo + tid; j < hi; j += TK_THREADS) {
            const unsigned key = dev_key(dev[j]);
            gt += key > T;
            eq += key == T;
        }
        gt = __reduce_add_sync(0xffffffffu, gt);
        eq = __reduce_add_sync(0xffffffffu, eq);
        if (lane == 0) { red[0][warp] = gt; red[1][warp] = eq; }
        __syncthreads();
        if (warp == 0) {
            const unsigned tg = __reduce_add_sync(0xffffffffu, red[0][lane]);
            const unsigned te = __reduce_add_sync(0xffffffffu, red[1][lane]);
            if (lane == 0) { cnt[0] = tg; cnt[1] = te; }
        }
    }
    ptx::cluster_sync();                               // every CTA's counts are published
    int out_base = 0, eq_base = 0;
    for (int q = 0; q < (int)rank; ++q) {
        const uint32_t base = ptx::map_to_rank(ptx::smem_u32(cnt), (uint32_t)q);
        const int g = (int)ld_cluster_u32(base), e = (int)ld_cluster_u32(base + 4u);
        out_base += g + max(0, min(e, remaining - eq_base));
        eq_base += e;
    }
    for (int t0 = lo; t0 < hi; t0 += TK_THREADS) {
        const int j = t0 + tid;
        const unsigned key = j < hi ? dev_key(dev[j]) : 0u;
        const bool eq = j < hi && key == T;
        int eq_total;
        const int eq_rank = block_excl_count(eq, warp_tot, eq_total);
        const bool take = (j < hi && key > T) || (eq && eq_base + eq_rank < remaining);
        int take_total;
        const int at = block_excl_count(take, warp_tot, take_total);
        if (take) {
            a.rows[out_base + at] = j;
            if (a.out_sel) a.out_sel[out_base + at] = j;
        }
        out_base += take_total;
        eq_base += eq_total;
    }
    ptx::cluster_sync();                               // no CTA exits while another reads its shared memory
}

// A given recomputed set (ascending positions in [0, n)) followed by the query rows.  A position out of
// range or out of order is recorded (ST_BAD_ROW) and replaced by a valid one so nothing reads out of bounds.
__global__ void __launch_bounds__(256) given_rows_kernel(const int* __restrict__ sel, int k, int n, int n_query,
                                                         int* __restrict__ rows, int* __restrict__ out_sel,
                                                         unsigned* status) {
    grid_dep_launch();
    grid_dep_wait();
    for (int i = threadIdx.x; i < k + n_query; i += blockDim.x) {
        int r;
        if (i < k) {
            r = sel[i];
            const bool ok = r >= 0 && r < n && (i == 0 || sel[i - 1] < r);
            if (!ok) {
                atomicOr(status, ST_BAD_ROW);
                r = min(max(r, 0), n - 1);
            }
            if (out_sel) out_sel[i] = r;
        } else {
            r = n + (i - k);
        }
        rows[i] = r;
    }
}

cudaError_t launch_given_rows(bool pdl, const int* sel, int k, int n, int n_query, int* rows, int* out_sel,
                              unsigned* status, cudaStream_t s) {
    return launch_ex(pdl, given_rows_kernel, dim3(1), dim3(256), 0, s, sel, k, n, n_query, rows, out_sel, status);
}

cudaError_t launch_topk(bool pdl, const float* dev_in, const float* dev_part, int parts, float* dev, int n_ctx, int k,
                        int n_query, int* rows, int* out_sel, cudaStream_t s) {
    TopkArgs a;
    a.dev_in = dev_in;
    a.dev_part = dev_part;
    a.parts = parts;
    a.dev = dev;
    a.n = n_ctx;
    a.k = k;
    a.n_query = n_query;
    a.rows = rows;
    a.out_sel = out_sel;
    return launch_ex(pdl, topk_kernel, dim3(TK_CTAS), dim3(TK_THREADS), 0, s, a);
}

}  // namespace cb
