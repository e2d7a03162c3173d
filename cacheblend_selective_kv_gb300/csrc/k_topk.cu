// HKVD selection: the k context rows of largest deviation (ties to the lower row), written in
// ascending row order, followed by the query rows -- the recomputed set of every later layer
// (CacheBlend deep-dive page, section "选 token:HKVD、逐层过滤与 15% 这个经验值").
//
// One CTA of 1024 threads.  A non-negative float's bit pattern orders like the float, so the
// k-th largest key is found by an MSB-first radix select (4 passes of 8-bit digits over shared
// histograms); rows above the threshold key, plus the lowest-index rows equal to it, are then
// compacted in index order with ballot/popc block scans.
#include "cb_common.cuh"

namespace cb {

static constexpr int TK_THREADS = 1024;

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

__global__ void __launch_bounds__(TK_THREADS) topk_kernel(const float* __restrict__ dev, int n, int k, int n_query,
                                                          int* __restrict__ rows, int* __restrict__ out_sel) {
    grid_dep_launch();
    grid_dep_wait();
    __shared__ unsigned hist[256];
    __shared__ int warp_tot[33];
    __shared__ unsigned s_digit;
    __shared__ int s_remaining;
    const int tid = threadIdx.x;

    // query rows always follow the k selected rows
    for (int i = tid; i < n_query; i += TK_THREADS) rows[k + i] = n + i;
    if (k <= 0) return;

    unsigned prefix = 0, mask = 0;
    int remaining = k;                                 // how many still to take at the current prefix
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += TK_THREADS) hist[b] = 0;
        __syncthreads();
        for (int j = tid; j < n; j += TK_THREADS) {
            const unsigned key = dev_key(dev[j]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid == 0) {
            int above = 0;
            unsigned dsel = 0;
            for (int dgt = 255; dgt >= 0; --dgt) {
                const int c = (int)hist[dgt];
                if (above + c >= remaining) { dsel = (unsigned)dgt; break; }
                above += c;
            }
            s_digit = dsel;
            s_remaining = remaining - above;
        }
        __syncthreads();
        prefix |= s_digit << shift;
        mask |= 255u << shift;
        remaining = s_remaining;
        __syncthreads();
    }
    // prefix = threshold key T; take every key > T and the first `remaining` keys == T
    const unsigned T = prefix;
    int out_base = 0, eq_base = 0;
    for (int t0 = 0; t0 < n; t0 += TK_THREADS) {
        const int j = t0 + tid;
        const unsigned key = j < n ? dev_key(dev[j]) : 0u;
        const bool eq = j < n && key == T;
        int eq_total;
        const int eq_rank = block_excl_count(eq, warp_tot, eq_total);
        const bool take = (j < n && key > T) || (eq && eq_base + eq_rank < remaining);
        int take_total;
        const int at = block_excl_count(take, warp_tot, take_total);
        if (take) {
            rows[out_base + at] = j;
            if (out_sel) out_sel[out_base + at] = j;
        }
        out_base += take_total;
        eq_base += eq_total;
    }
}

cudaError_t launch_topk(const Model& m, const float* dev, int n_ctx, int k, int n_query, int* rows, int* out_sel,
                        cudaStream_t s) {
    (void)m;
    topk_kernel<<<1, TK_THREADS, 0, s>>>(dev, n_ctx, k, n_query, rows, out_sel);
    return cudaGetLastError();
}

}  // namespace cb
