// Epilogue element operations shared by the GEMM kernels.
#pragma once
#include "cb_common.cuh"

namespace cb {

__device__ __forceinline__ int epi_pos(const EpiParams& e, int r) { return e.pos ? e.pos[r] : e.pos_offset + r; }

// Region of a column of the concatenated [q | k | v] space: 0 = q, 1 = k, 2 = v; `off` = column within it.
__device__ __forceinline__ int qkv_region(const EpiParams& e, int qc, int& off) {
    if (qc < e.nq) { off = qc; return 0; }
    if (qc < e.nq + e.nkv) { off = qc - e.nq; return 1; }
    off = qc - e.nq - e.nkv;
    return 2;
}

// RoPE of one adjacent pair (2i, 2i+1) at position p: block i of R_p (section "位置恢复、KV 存储与加载流水线").
__device__ __forceinline__ void rope_pair(const EpiParams& e, int p, int off, float& x0, float& x1) {
    const int half = e.head_dim >> 1;
    const float2 cs = e.rope[(size_t)p * half + ((off % e.head_dim) >> 1)];
    const float a = x0, b = x1;
    x0 = a * cs.x - b * cs.y;
    x1 = a * cs.y + b * cs.x;
}

// Store one (already rotated) element of region `reg` at column `off` for token row r.
template <typename T>
__device__ __forceinline__ void qkv_store(const EpiParams& e, int reg, int r, int p, int off, float v) {
    if (reg == 0) {
        const T h = from_f<T>(v);
        reinterpret_cast<T*>(e.q_out)[(size_t)r * e.nq + off] = h;
        if (e.q_out_lo) reinterpret_cast<T*>(e.q_out_lo)[(size_t)r * e.nq + off] = from_f<T>(v - to_f(h));
    } else {
        void* dst = reg == 1 ? e.k_dst : e.v_dst;
        if (e.kv_fresh)
            reinterpret_cast<float*>(dst)[(size_t)r * e.nkv + off] = v;
        else
            reinterpret_cast<T*>(dst)[(size_t)p * e.nkv + off] = from_f<T>(v);
    }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

}  // namespace cb
