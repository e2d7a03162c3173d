// Paged blended K/V (CacheBlend deep-dive page, section "和前缀缓存、PagedAttention 的分工"): the
// blended cache of a request lives in pages of a pool addressed through a block table, and a gather /
// scatter converts between that paged layout and contiguous rows.
//
// Pool layout: [L][2][n_pages * P][W] in the storage type, P = 2^page_shift rows per page: page p holds
// rows p*P .. p*P+P-1 of every (layer, K|V) block, so logical row j of a request whose block table is t
// sits at pool row t[j / P] * P + j % P.  A row crosses no page; a run of rows is split at page
// boundaries by construction.  All accesses are 16-byte vectors, consecutive threads on consecutive
// addresses of one row.
#include "cb_common.cuh"

namespace cb {

template <typename V>
__global__ void page_copy_kernel(const V* __restrict__ src, int64_t src_rows, const int* __restrict__ src_pages,
                                 V* __restrict__ dst, int64_t dst_rows, const int* __restrict__ dst_pages,
                                 int page_shift, int n_rows, int W16, int L2, unsigned* status) {
    grid_dep_launch();
    grid_dep_wait();
    const int64_t per_block = (int64_t)n_rows * W16;             // vectors per (layer, K|V) block
    const int64_t total = (int64_t)L2 * per_block;
    const int mask = (1 << page_shift) - 1;
    const int64_t src_pages_n = src_rows >> page_shift, dst_pages_n = dst_rows >> page_shift;
    for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < total;
         it += (int64_t)gridDim.x * blockDim.x) {
        const int lk = (int)(it / per_block);
        const int64_t rem = it - (int64_t)lk * per_block;
        const int j = (int)(rem / W16), e = (int)(rem - (int64_t)j * W16);
        int64_t sj = j, dj = j;
        if (src_pages) {
            const int pg = src_pages[j >> page_shift];
            if (pg < 0 || pg >= src_pages_n) { atomicOr(status, ST_BAD_ROW); continue; }
            sj = ((int64_t)pg << page_shift) + (j & mask);
        }
        if (dst_pages) {
            const int pg = dst_pages[j >> page_shift];
            if (pg < 0 || pg >= dst_pages_n) { atomicOr(status, ST_BAD_ROW); continue; }
            dj = ((int64_t)pg << page_shift) + (j & mask);
        }
        dst[((int64_t)lk * dst_rows + dj) * W16 + e] = src[((int64_t)lk * src_rows + sj) * W16 + e];
    }
}

cudaError_t launch_page_copy(const Model& m, const void* src, int64_t src_rows, const int* src_pages, void* dst,
                             int64_t dst_rows, const int* dst_pages, int page_shift, int n_rows, cudaStream_t s) {
    const cb_config& c = m.cfg;
    const int row_bytes = c.n_kv_heads * c.head_dim * (m.bf16 ? 2 : 4);
    const int W16 = row_bytes / 16;
    const int64_t items = (int64_t)2 * c.n_layers * n_rows * W16;
    if (items == 0) return cudaSuccess;
    int64_t blocks = (items + 255) / 256;
    const int64_t cap = (int64_t)m.num_sms * 16;
    page_copy_kernel<uint4><<<(int)(blocks < cap ? blocks : cap), 256, 0, s>>>(
        (const uint4*)src, src_rows, src_pages, (uint4*)dst, dst_rows, dst_pages, page_shift, n_rows, W16,
        2 * c.n_layers, m.status);
    return cudaGetLastError();
}

}  // namespace cb
