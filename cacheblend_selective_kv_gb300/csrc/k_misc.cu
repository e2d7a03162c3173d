// Memory-bound kernels of the blend step: re-RoPE placement of chunk caches, embedding,
// RMSNorm, the check-layer KV deviation, gather/scatter of the recomputed rows, and the
// last-token logits.  All vector accesses are 16 bytes wide and consecutive threads touch
// consecutive addresses.
#include "cb_common.cuh"

namespace cb {

// 16-byte vector of 8 storage elements, widened to fp32
template <typename T> struct Vec8;
template <> struct Vec8<bf16> {
    static __device__ __forceinline__ void load(const bf16* p, float* f) {
        uint4 u = *reinterpret_cast<const uint4*>(p);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    static __device__ __forceinline__ void store(bf16* p, const float* f) {
        uint4 u;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        *reinterpret_cast<uint4*>(p) = u;
    }
};
template <> struct Vec8<float> {
    static __device__ __forceinline__ void load(const float* p, float* f) {
        float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
    static __device__ __forceinline__ void store(float* p, const float* f) {
        reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
};

// each value rounded to T and back to float (identity for float)
template <typename T> __device__ __forceinline__ void round_to(const float* v, float* out);
template <> __device__ __forceinline__ void round_to<bf16>(const float* v, float* out) {
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
}
template <> __device__ __forceinline__ void round_to<float>(const float* v, float* out) {
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = v[i];
}

// ------------------------------------------------------------------------------------------------
// (cos, sin) of each chunk's position delta, in float64, and the chunk tables.
// ------------------------------------------------------------------------------------------------
__global__ void delta_table_kernel(ChunkTable t, const double* inv_freq, int half, float2* cs, int* dst,
                                   int* delta) {
    grid_dep_launch();
    grid_dep_wait();
    const int c = blockIdx.x;
    if (c >= t.n) return;
    if (threadIdx.x == 0) {
        dst[c] = t.dst[c];
        delta[c] = t.delta[c];
    }
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        double s, co;
        sincos((double)t.delta[c] * inv_freq[i], &s, &co);
        cs[(size_t)c * half + i] = make_float2((float)co, (float)s);
    }
}

cudaError_t launch_delta_table(const Model& m, const ChunkTable& t, cudaStream_t s) {
    const int half = m.cfg.head_dim / 2;
    delta_table_kernel<<<t.n, 64, 0, s>>>(t, m.inv_freq, half, m.delta_cs, m.chunk_dst, m.chunk_delta);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// Re-RoPE placement: dst K row j = R_{delta(chunk of j)} src K row j; dst V row j = src V row j.
// src and dst are [L][2][rows][W]; they may be the same buffer with the same row count.  With a page
// table, src row j is row (src_pages[j / P] * P + j % P) of a paged pool (P = 2^page_shift); a page id
// outside [0, n_pages) is recorded in the status word and its rows are skipped.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ int chunk_of(const int* dst, int n, int j) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {                       // last chunk with dst <= j
        int mid = (lo + hi + 1) >> 1;
        if (dst[mid] <= j) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <typename T>
__global__ void rerope_kernel(const T* __restrict__ src, T* __restrict__ dst, int64_t src_rows, int64_t dst_rows,
                              int n_ctx, int W, int hd, int kv_count, const int* __restrict__ cdst,
                              const float2* __restrict__ cs, int n_chunks, const int* __restrict__ src_pages,
                              int page_shift, int64_t n_pages, unsigned* status) {
    grid_dep_launch();
    grid_dep_wait();
    // blockIdx.y = (layer, K|V) block; 32-bit indices within it (n_ctx * W / 8 < 2^31)
    const int lk = blockIdx.y;
    const int layer = lk / kv_count, kv = lk - layer * kv_count;
    const int W8 = W / 8, half = hd / 2;
    const int per_lk = n_ctx * W8;
    const T* sblk = src + ((int64_t)layer * 2 + kv) * src_rows * W;
    T* dblk = dst + ((int64_t)layer * 2 + kv) * dst_rows * W;
    for (int it = blockIdx.x * blockDim.x + threadIdx.x; it < per_lk; it += gridDim.x * blockDim.x) {
        const int j = it / W8, e = (it - j * W8) * 8;
        int64_t sj = j;
        if (src_pages) {
            const int pg = src_pages[j >> page_shift];
            if (pg < 0 || pg >= n_pages) {
                atomicOr(status, ST_BAD_ROW);
                continue;
            }
            sj = ((int64_t)pg << page_shift) + (j & ((1 << page_shift) - 1));
        }
        float f[8];
        Vec8<T>::load(sblk + sj * W + e, f);
        if (kv == 0) {
            const int c = chunk_of(cdst, n_chunks, j);
            const float2* t = cs + (size_t)c * half + (e % hd) / 2;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float2 y = rotate_pair(f[2 * p], f[2 * p + 1], t[p]);
                f[2 * p] = y.x;
                f[2 * p + 1] = y.y;
            }
        }
        Vec8<T>::store(dblk + (int64_t)j * W + e, f);
    }
}

cudaError_t launch_rerope(const Model& m, const void* src, void* dst, int64_t src_rows, int64_t dst_rows, int n_ctx,
                          int n_chunks, bool copy_v, cudaStream_t s, int layers, const int* src_pages, int page_shift) {
    const cb_config& c = m.cfg;
    const int W = c.n_kv_heads * c.head_dim, kvc = copy_v ? 2 : 1;
    const int L = layers > 0 ? layers : c.n_layers;
    const int64_t per_lk = (int64_t)n_ctx * (W / 8);
    if (per_lk == 0) return cudaSuccess;
    // about 16 resident blocks per SM over all (layer, K|V) blocks
    int64_t bx = ((int64_t)m.num_sms * 16 + (int64_t)L * kvc - 1) / ((int64_t)L * kvc);
    const int64_t need = (per_lk + 255) / 256;
    if (bx > need) bx = need;
    if (bx < 1) bx = 1;
    const dim3 grid((unsigned)bx, (unsigned)(L * kvc));
    if (m.bf16)
        rerope_kernel<bf16><<<grid, 256, 0, s>>>((const bf16*)src, (bf16*)dst, src_rows, dst_rows, n_ctx, W,
                                                 c.head_dim, kvc, m.chunk_dst, m.delta_cs, n_chunks, src_pages,
                                                 page_shift, src_rows >> page_shift, m.status);
    else
        rerope_kernel<float><<<grid, 256, 0, s>>>((const float*)src, (float*)dst, src_rows, dst_rows, n_ctx, W,
                                                  c.head_dim, kvc, m.chunk_dst, m.delta_cs, n_chunks, src_pages,
                                                  page_shift, src_rows >> page_shift, m.status);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// embedding: h[r] = E[token r] (fp32)
// ------------------------------------------------------------------------------------------------
template <typename T>
__global__ void embed_kernel(const int* __restrict__ tokens, const T* __restrict__ E, int vocab, int d, float* h,
                             unsigned* status) {
    grid_dep_launch();
    grid_dep_wait();
    const int r = blockIdx.x;
    const int t = tokens[r];
    float* out = h + (size_t)r * d;
    if (t < 0 || t >= vocab) {
        if (threadIdx.x == 0) atomicOr(status, ST_BAD_TOKEN);
        for (int e = threadIdx.x; e < d; e += blockDim.x) out[e] = 0.f;
        return;
    }
    const T* row = E + (size_t)t * d;
    for (int e = threadIdx.x * 8; e < d; e += blockDim.x * 8) {
        float f[8];
        Vec8<T>::load(row + e, f);
        reinterpret_cast<float4*>(out + e)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(out + e)[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
}

cudaError_t launch_embed(const Model& m, const int* tokens, int n, float* h, cudaStream_t s) {
    if (m.bf16)
        embed_kernel<bf16><<<n, 128, 0, s>>>(tokens, (const bf16*)m.embed, m.cfg.vocab, m.cfg.d_model, h, m.status);
    else
        embed_kernel<float><<<n, 128, 0, s>>>(tokens, (const float*)m.embed, m.cfg.vocab, m.cfg.d_model, h, m.status);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// RMSNorm: out[r] = g * h[r] / sqrt(mean(h[r]^2) + eps), stored in the activation type (in split
// precision also lo = rn(v - rn(v))).  One CTA per row; a thread keeps its RC chunks of 8 values in
// registers between the sum of squares and the scaled write, so the row is read once.  When the residual
// GEMM before it split its K range, h[r] is first completed with that GEMM's partial sums, added in slot
// order (all slots' loads in flight together) and written back, which makes the residual stream
// independent of which CTA finished first.
// ------------------------------------------------------------------------------------------------
constexpr int NORM_THREADS = 256;
constexpr int NORM_MAX_PARTS = 8;

// P > 0: the number of partial-sum slots, known at compile time for the common counts so that every
// slot's loads are issued before the first addition (P = NORM_MAX_PARTS: any count up to it, predicated)
template <typename T, int RC, int P>
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_kernel(float* __restrict__ h, const float* __restrict__ part,
                                                               int parts, const T* __restrict__ g, T* __restrict__ out,
                                                               T* __restrict__ out_lo, int n, int d, float eps) {
    grid_dep_launch();
    grid_dep_wait();
    __shared__ float red[NORM_THREADS / 32];
    const int r = blockIdx.x, tid = threadIdx.x;
    float* row = h + (size_t)r * d;
    const size_t pstride = (size_t)n * d;
    float f[RC][8];
#pragma unroll
    for (int c = 0; c < RC; ++c) {
        const int e = (tid + c * NORM_THREADS) * 8;
        if (e < d) Vec8<float>::load(row + e, f[c]);
    }
    if (P > 0 && parts > 0) {
#pragma unroll
        for (int c = 0; c < RC; ++c) {
            const int e = (tid + c * NORM_THREADS) * 8;
            if (e < d) {
                float t[P > 0 ? P : 1][8];
#pragma unroll
                for (int p = 0; p < P; ++p)
                    if (p < parts) Vec8<float>::load(part + p * pstride + (size_t)r * d + e, t[p]);
#pragma unroll
                for (int p = 0; p < P; ++p)
                    if (p < parts) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[c][i] += t[p][i];
                    }
            }
        }
#pragma unroll
        for (int c = 0; c < RC; ++c) {
            const int e = (tid + c * NORM_THREADS) * 8;
            if (e < d) Vec8<float>::store(row + e, f[c]);
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < RC; ++c) {
        const int e = (tid + c * NORM_THREADS) * 8;
        if (e < d) {
#pragma unroll
            for (int i = 0; i < 8; ++i) ss += f[c][i] * f[c][i];
        }
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NORM_THREADS / 32; ++w) tot += red[w];
    const float scale = 1.0f / sqrtf(tot / (float)d + eps);
    T* o = out + (size_t)r * d;
    T* ol = out_lo ? out_lo + (size_t)r * d : nullptr;
#pragma unroll
    for (int c = 0; c < RC; ++c) {
        const int e = (tid + c * NORM_THREADS) * 8;
        if (e < d) {
            float gg[8], v[8];
            Vec8<T>::load(g + e, gg);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = f[c][i] * scale * gg[i];
            Vec8<T>::store(o + e, v);
            if (ol) {            // remainder after rounding to T (split precision)
                float hi[8];
                round_to<T>(v, hi);
#pragma unroll
                for (int i = 0; i < 8; ++i) hi[i] = v[i] - hi[i];
                Vec8<T>::store(ol + e, hi);
            }
        }
    }
}

template <typename T, int RC, int P>
cudaError_t launch_norm_p(const Model& m, float* h, const float* part, int parts, const void* g, void* out,
                          void* out_lo, int n, cudaStream_t s) {
    return launch_ex(m.pdl, rmsnorm_kernel<T, RC, P>, dim3(n), dim3(NORM_THREADS), 0, s, h, part, parts, (const T*)g,
                     (T*)out, (T*)out_lo, n, m.cfg.d_model, m.cfg.rms_eps);
}

template <typename T, int RC>
cudaError_t launch_norm_t(const Model& m, float* h, const float* part, int parts, const void* g, void* out,
                          void* out_lo, int n, cudaStream_t s) {
    switch (parts) {
        case 0: return launch_norm_p<T, RC, 0>(m, h, part, parts, g, out, out_lo, n, s);
        case 2: return launch_norm_p<T, RC, 2>(m, h, part, parts, g, out, out_lo, n, s);
        case 3: return launch_norm_p<T, RC, 3>(m, h, part, parts, g, out, out_lo, n, s);
        case 4: return launch_norm_p<T, RC, 4>(m, h, part, parts, g, out, out_lo, n, s);
        default: return launch_norm_p<T, RC, NORM_MAX_PARTS>(m, h, part, parts, g, out, out_lo, n, s);
    }
}

template <typename T>
cudaError_t launch_norm_d(const Model& m, float* h, const float* part, int parts, const void* g, void* out,
                          void* out_lo, int n, cudaStream_t s) {
    const int d = m.cfg.d_model;
    if (parts > NORM_MAX_PARTS) return cudaErrorInvalidValue;
    if (d <= 8 * NORM_THREADS) return launch_norm_t<T, 1>(m, h, part, parts, g, out, out_lo, n, s);
    if (d <= 16 * NORM_THREADS) return launch_norm_t<T, 2>(m, h, part, parts, g, out, out_lo, n, s);
    if (d <= 32 * NORM_THREADS) return launch_norm_t<T, 4>(m, h, part, parts, g, out, out_lo, n, s);
    if (d <= 64 * NORM_THREADS) return launch_norm_t<T, 8>(m, h, part, parts, g, out, out_lo, n, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_rmsnorm(const Model& m, float* h, const float* part, int parts, const void* g, void* out,
                           void* out_lo, int n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    if (m.bf16) return launch_norm_d<bf16>(m, h, part, parts, g, out, out_lo, n, s);
    return launch_norm_d<float>(m, h, part, parts, g, out, nullptr, n, s);
}

// ------------------------------------------------------------------------------------------------
// KV deviation (CacheBlend deep-dive page, section "核心思想", Δkv formula):
// dev[r] = sum over KV heads and dims of (k_new - k_pre)^2 + (v_new - v_pre)^2,
// with fresh fp32 K/V (row r) and the re-RoPE'd stored cache (row crow[r], or r when crow is
// NULL: the check layer compares every context row in place; a later shrinking layer compares
// its candidates, whose cache rows are their positions).  One warp per row.
// ------------------------------------------------------------------------------------------------
template <typename T>
__global__ void deviation_kernel(const float* __restrict__ kf, const float* __restrict__ vf,
                                 const T* __restrict__ kv_layer, int64_t kv_rows, const int* __restrict__ crow,
                                 int n_ctx, int W, float* dev) {
    grid_dep_launch();
    grid_dep_wait();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= n_ctx) return;
    const int64_t j = crow ? crow[warp] : warp;
    const T* kc = kv_layer + j * W;
    const T* vc = kv_layer + (kv_rows + j) * (int64_t)W;
    const float* kn = kf + (int64_t)warp * W;
    const float* vn = vf + (int64_t)warp * W;
    float acc = 0.f;
    for (int e = lane * 8; e < W; e += 256) {
        float a[8], b[8];
        Vec8<T>::load(kc + e, a);
        Vec8<float>::load(kn + e, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) { float t = b[i] - a[i]; acc += t * t; }
        Vec8<T>::load(vc + e, a);
        Vec8<float>::load(vn + e, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) { float t = b[i] - a[i]; acc += t * t; }
    }
    acc = warp_sum(acc);
    if (lane == 0) dev[warp] = acc;
}

cudaError_t launch_deviation(const Model& m, const float* kf, const float* vf, const void* kv_layer, int64_t kv_rows,
                             const int* crow, int n_ctx, float* dev, cudaStream_t s) {
    if (n_ctx <= 0) return cudaSuccess;
    const int W = m.cfg.n_kv_heads * m.cfg.head_dim;
    const int grid = (n_ctx + 7) / 8;
    if (m.bf16)
        deviation_kernel<bf16><<<grid, 256, 0, s>>>(kf, vf, (const bf16*)kv_layer, kv_rows, crow, n_ctx, W, dev);
    else
        deviation_kernel<float><<<grid, 256, 0, s>>>(kf, vf, (const float*)kv_layer, kv_rows, crow, n_ctx, W, dev);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// Rows of the next recomputed set: their hidden state and normalised input are compacted, and their
// fresh K/V (kept by the comparing GEMM as rows of the storage type, or fp32 rows on the CUDA-core path)
// are stored into the blended cache at their positions before attention (Figure 5: assemble the complete
// K/V, then attend).  src[i] is the row of h/x/K/V that becomes compact row i; dst_pos[i] its position.
// ------------------------------------------------------------------------------------------------
template <typename T, typename S>
__device__ __forceinline__ void copy_kv_row(const S* kf, const S* vf, int src, T* kv_layer, int64_t kv_rows, int pos,
                                            int W) {
    for (int e = threadIdx.x * 8; e < W; e += blockDim.x * 8) {
        float f[8];
        Vec8<S>::load(kf + (size_t)src * W + e, f);
        Vec8<T>::store(kv_layer + (int64_t)pos * W + e, f);
        Vec8<S>::load(vf + (size_t)src * W + e, f);
        Vec8<T>::store(kv_layer + (kv_rows + pos) * (int64_t)W + e, f);
    }
}

template <typename T>
__device__ __forceinline__ void copy_state_row(const float* h, float* hn, const T* x, T* xn, const T* xl, T* xln,
                                               int src, int i, int d) {
    for (int e = threadIdx.x * 4; e < d; e += blockDim.x * 4)
        *reinterpret_cast<float4*>(hn + (size_t)i * d + e) = *reinterpret_cast<const float4*>(h + (size_t)src * d + e);
    for (int e = threadIdx.x * 8; e < d; e += blockDim.x * 8) {
        float f[8];
        Vec8<T>::load(x + (size_t)src * d + e, f);
        Vec8<T>::store(xn + (size_t)i * d + e, f);
        if (xl) {
            Vec8<T>::load(xl + (size_t)src * d + e, f);
            Vec8<T>::store(xln + (size_t)i * d + e, f);
        }
    }
}

template <typename T, typename S>
__global__ void gather_kernel(const int* __restrict__ rows, const float* __restrict__ h, float* __restrict__ hA,
                              const T* __restrict__ x, T* __restrict__ xA, const T* __restrict__ x_lo,
                              T* __restrict__ xA_lo, const S* __restrict__ kf, const S* __restrict__ vf, T* kv_layer,
                              int64_t kv_rows, int d, int W) {
    grid_dep_launch();
    grid_dep_wait();
    const int i = blockIdx.x;
    const int r = rows[i];
    copy_state_row<T>(h, hA, x, xA, x_lo, xA_lo, r, i, d);
    if (kf) copy_kv_row<T, S>(kf, vf, r, kv_layer, kv_rows, r, W);
}

template <typename T, typename S>
__global__ void refilter_kernel(const int* __restrict__ local, const int* __restrict__ rows_old, int* __restrict__ rows_new,
                                int k_new, int* __restrict__ out_sel, const float* __restrict__ h_old,
                                float* __restrict__ h_new, const T* __restrict__ x_old, T* __restrict__ x_new,
                                const T* __restrict__ xlo_old, T* __restrict__ xlo_new, const S* __restrict__ kf,
                                const S* __restrict__ vf, T* kv_layer, int64_t kv_rows, int d, int W) {
    grid_dep_launch();
    grid_dep_wait();
    const int i = blockIdx.x;
    const int src = local[i];
    const int r = rows_old[src];
    if (threadIdx.x == 0) {
        rows_new[i] = r;
        if (out_sel && i < k_new) out_sel[i] = r;
    }
    copy_state_row<T>(h_old, h_new, x_old, x_new, xlo_old, xlo_new, src, i, d);
    copy_kv_row<T, S>(kf, vf, src, kv_layer, kv_rows, r, W);
}

cudaError_t launch_gather(const Model& m, const int* rows, int M, const float* h, float* hA, const void* x, void* xA,
                          const void* x_lo, void* xA_lo, const void* kf, const void* vf, bool kv_f32, void* kv_layer,
                          int64_t kv_rows, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    const int d = m.cfg.d_model, W = m.cfg.n_kv_heads * m.cfg.head_dim;
    if (!m.bf16)
        gather_kernel<float, float><<<M, 256, 0, s>>>(rows, h, hA, (const float*)x, (float*)xA, nullptr, nullptr,
                                                      (const float*)kf, (const float*)vf, (float*)kv_layer, kv_rows, d, W);
    else if (kv_f32)
        gather_kernel<bf16, float><<<M, 256, 0, s>>>(rows, h, hA, (const bf16*)x, (bf16*)xA, (const bf16*)x_lo,
                                                     (bf16*)xA_lo, (const float*)kf, (const float*)vf, (bf16*)kv_layer,
                                                     kv_rows, d, W);
    else
        gather_kernel<bf16, bf16><<<M, 256, 0, s>>>(rows, h, hA, (const bf16*)x, (bf16*)xA, (const bf16*)x_lo,
                                                    (bf16*)xA_lo, (const bf16*)kf, (const bf16*)vf, (bf16*)kv_layer,
                                                    kv_rows, d, W);
    return cudaGetLastError();
}

cudaError_t launch_refilter(const Model& m, const int* local, const int* rows_old, int* rows_new, int M_new, int k_new,
                            int* out_sel, const float* h_old, float* h_new, const void* x_old, void* x_new,
                            const void* xlo_old, void* xlo_new, const void* kf, const void* vf, bool kv_f32,
                            void* kv_layer, int64_t kv_rows, cudaStream_t s) {
    if (M_new <= 0) return cudaSuccess;
    const int d = m.cfg.d_model, W = m.cfg.n_kv_heads * m.cfg.head_dim;
    if (!m.bf16)
        refilter_kernel<float, float><<<M_new, 256, 0, s>>>(local, rows_old, rows_new, k_new, out_sel, h_old, h_new,
                                                            (const float*)x_old, (float*)x_new, nullptr, nullptr,
                                                            (const float*)kf, (const float*)vf, (float*)kv_layer,
                                                            kv_rows, d, W);
    else if (kv_f32)
        refilter_kernel<bf16, float><<<M_new, 256, 0, s>>>(local, rows_old, rows_new, k_new, out_sel, h_old, h_new,
                                                           (const bf16*)x_old, (bf16*)x_new, (const bf16*)xlo_old,
                                                           (bf16*)xlo_new, (const float*)kf, (const float*)vf,
                                                           (bf16*)kv_layer, kv_rows, d, W);
    else
        refilter_kernel<bf16, bf16><<<M_new, 256, 0, s>>>(local, rows_old, rows_new, k_new, out_sel, h_old, h_new,
                                                          (const bf16*)x_old, (bf16*)x_new, (const bf16*)xlo_old,
                                                          (bf16*)xlo_new, (const bf16*)kf, (const bf16*)vf,
                                                          (bf16*)kv_layer, kv_rows, d, W);
    return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// Logits of the last row: final RMSNorm (recomputed per block, d floats) then a GEMV over the
// vocabulary; one warp per vocabulary row, 16-byte loads.  HBM-bound on the LM-head read.
// ------------------------------------------------------------------------------------------------
template <typename T>
__global__ void logits_kernel(const float* __restrict__ hl, const float* __restrict__ part, int parts, size_t pstride,
                              const T* __restrict__ g, const T* __restrict__ Wh, int d, int vocab, float eps,
                              float* __restrict__ out) {
    grid_dep_launch();
    grid_dep_wait();
    extern __shared__ float xs[];
    __shared__ float red[32];
    // the last row, completed with the partial sums its residual GEMM left (slot order), kept in shared memory
    for (int e = threadIdx.x; e < d; e += blockDim.x) {
        float v = hl[e];
        for (int p = 0; p < parts; ++p) v += part[p * pstride + e];
        xs[e] = v;
    }
    __syncthreads();
    float ss = 0.f;
    for (int e = threadIdx.x; e < d; e += blockDim.x) { float v = xs[e]; ss += v * v; }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        v = warp_sum(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float scale = 1.0f / sqrtf(red[0] / (float)d + eps);
    for (int e = threadIdx.x; e < d; e += blockDim.x) xs[e] = xs[e] * scale * to_f(g[e]);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int v = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < vocab; v += warps) {
        const T* row = Wh + (size_t)v * d;
        float acc = 0.f;
        for (int e = lane * 8; e < d; e += 256) {
            float f[8];
            Vec8<T>::load(row + e, f);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc += f[i] * xs[e + i];
        }
        acc = warp_sum(acc);
        if (lane == 0) out[v] = acc;
    }
}

cudaError_t launch_logits(const Model& m, const float* h_last, const float* part, int parts, size_t part_stride,
                          float* logits, cudaStream_t s) {
    const int d = m.cfg.d_model;
    const int grid = m.num_sms * 4;
    if (m.bf16)
        logits_kernel<bf16><<<grid, 256, d * sizeof(float), s>>>(h_last, part, parts, part_stride,
                                                                 (const bf16*)m.final_norm, (const bf16*)m.lm_head, d,
                                                                 m.cfg.vocab, m.cfg.rms_eps, logits);
    else
        logits_kernel<float><<<grid, 256, d * sizeof(float), s>>>(h_last, part, parts, part_stride,
                                                                  (const float*)m.final_norm, (const float*)m.lm_head,
                                                                  d, m.cfg.vocab, m.cfg.rms_eps, logits);
    return cudaGetLastError();
}

}  // namespace cb
