// Selective attention over the blended K/V (CacheBlend deep-dive page, Figure 5: the recomputed
// queries attend over every token).  Query row i sits at global position qpos[i] and sees keys
// 0..qpos[i]; q-head h reads KV head h / (Hq/Hkv); scores scaled by 1/sqrt(head_dim); softmax in
// fp32 with a running max (online rescaling), so any number of keys streams through one pass.
//
// CUDA-core version: one CTA per (query row, KV head) handles the whole GQA group, 128 keys
// per step.
#include "cb_common.cuh"

namespace cb {

namespace {
constexpr int KB = 128;   // keys per step (= threads)

template <typename T>
__global__ void __launch_bounds__(KB) attn_simt_kernel(const T* __restrict__ q, const T* __restrict__ q_lo,
                                                       const int* __restrict__ qpos,
                                                       const T* __restrict__ kv, int64_t kv_rows, int n_keys,
                                                       T* __restrict__ out, T* __restrict__ out_lo, int Hq, int Hkv,
                                                       int hd, float scale) {
    grid_dep_launch();
    grid_dep_wait();
    extern __shared__ float sm[];
    const int i = blockIdx.x, g = blockIdx.y, G = Hq / Hkv, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int W = Hkv * hd;
    float* qs = sm;                 // [G][hd]
    float* ps = qs + G * hd;        // [G][KB]
    float* vs = ps + G * KB;        // [KB][hd]
    float* mrun = vs + KB * hd;     // [G]
    float* lrun = mrun + G;         // [G]
    float* alpha = lrun + G;        // [G]
    const int p = qpos ? qpos[i] : i;
    const int nk = min(p + 1, n_keys);
    const T* qrow = q + (size_t)i * Hq * hd + (size_t)g * G * hd;
    const T* qlrow = q_lo ? q_lo + (size_t)i * Hq * hd + (size_t)g * G * hd : nullptr;
    for (int t = tid; t < G * hd; t += KB) qs[t] = (to_f(qrow[t]) + (qlrow ? to_f(qlrow[t]) : 0.f)) * scale;
    if (tid < G) { mrun[tid] = -INFINITY; lrun[tid] = 0.f; }
    const int nslot = (G * hd + KB - 1) / KB;   // <= 8
    float acc[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) acc[s] = 0.f;
    const T* K = kv + (size_t)g * hd;
    const T* V = kv + kv_rows * (int64_t)W + (size_t)g * hd;
    __syncthreads();

    for (int j0 = 0; j0 < nk; j0 += KB) {
        const int j = j0 + tid;
        if (j < nk) {
            const T* kr = K + (int64_t)j * W;
            for (int gg = 0; gg < G; ++gg) {
                float s = 0.f;
                for (int d = 0; d < hd; ++d) s = fmaf(qs[gg * hd + d], to_f(kr[d]), s);
                ps[gg * KB + tid] = s;
            }
        } else {
            for (int gg = 0; gg < G; ++gg) ps[gg * KB + tid] = -INFINITY;
        }
        for (int t = tid; t < KB * hd; t += KB) {
            const int jj = j0 + t / hd, d = t % hd;
            vs[t] = jj < nk ? to_f(V[(int64_t)jj * W + d]) : 0.f;
        }
        __syncthreads();
        for (int gg = warp; gg < G; gg += KB / 32) {
            float mx = -INFINITY;
            for (int t = lane; t < KB; t += 32) mx = fmaxf(mx, ps[gg * KB + t]);
            mx = warp_max(mx);
            const float m_old = mrun[gg], m_new = fmaxf(m_old, mx);
            float sum = 0.f;
            for (int t = lane; t < KB; t += 32) {
                const float e = __expf(ps[gg * KB + t] - m_new);
                ps[gg * KB + t] = e;
                sum += e;
            }
            sum = warp_sum(sum);
            if (lane == 0) {
                const float a = m_old == -INFINITY ? 0.f : __expf(m_old - m_new);
                alpha[gg] = a;
                lrun[gg] = lrun[gg] * a + sum;
                mrun[gg] = m_new;
            }
        }
        __syncthreads();
        for (int s = 0; s < nslot; ++s) {
            const int idx = tid + s * KB;
            if (idx >= G * hd) break;
            const int gg = idx / hd, d = idx % hd;
            float a = acc[s] * alpha[gg];
            for (int t = 0; t < KB; ++t) a = fmaf(ps[gg * KB + t], vs[t * hd + d], a);
            acc[s] = a;
        }
        __syncthreads();
    }
    T* orow = out + (size_t)i * Hq * hd + (size_t)g * G * hd;
    for (int s = 0; s < nslot; ++s) {
        const int idx = tid + s * KB;
        if (idx >= G * hd) break;
        const float o = acc[s] / lrun[idx / hd];
        const T oh = from_f<T>(o);
        orow[idx] = oh;
        if (out_lo) out_lo[(size_t)i * Hq * hd + (size_t)g * G * hd + idx] = from_f<T>(o - to_f(oh));
    }
}
}  // namespace

cudaError_t launch_attention(const Model& m, const void* q, const void* q_lo, const int* qpos, int M,
                             const void* kv_layer, int64_t kv_rows, int n_keys, void* out, void* out_lo, cudaStream_t s) {
    const cb_config& c = m.cfg;
    const int G = c.n_heads / c.n_kv_heads, hd = c.head_dim;
    const size_t smem = sizeof(float) * ((size_t)G * hd + (size_t)G * KB + (size_t)KB * hd + 3 * G);
    const float scale = 1.0f / sqrtf((float)hd);
    dim3 grid(M, c.n_kv_heads);
    if (m.bf16) {
        cudaFuncSetAttribute(attn_simt_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        attn_simt_kernel<bf16><<<grid, KB, smem, s>>>((const bf16*)q, (const bf16*)q_lo, qpos, (const bf16*)kv_layer, kv_rows, n_keys,
                                                      (bf16*)out, (bf16*)out_lo, c.n_heads, c.n_kv_heads, hd, scale);
    } else {
        cudaFuncSetAttribute(attn_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        attn_simt_kernel<float><<<grid, KB, smem, s>>>((const float*)q, nullptr, qpos, (const float*)kv_layer, kv_rows, n_keys,
                                                       (float*)out, nullptr, c.n_heads, c.n_kv_heads, hd, scale);
    }
    return cudaGetLastError();
}

}  // namespace cb
