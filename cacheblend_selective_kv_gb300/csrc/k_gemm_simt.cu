// CUDA-core GEMM with the blend's fused epilogues.  It carries the fp32 configuration (whose
// operands the tensor cores would round) and any shape the tensor-core kernel does not take.
//   Y[r][c] = sum_k X[r][k] W[c][k]    (X token rows, W weight rows; fp32 accumulation)
// Tile 64 token rows x 64 output columns, k-step 16, 256 threads, 4x4 outputs per thread.
#include "cb_epilogue.cuh"

namespace cb {

namespace {
constexpr int BM = 64, BN = 64, BK = 16;

template <typename T>
__device__ __forceinline__ const T* weight_row(const GemmW& w, int c, int K) {
    int base = 0;
    for (int s = 0; s < w.nseg; ++s) {
        if (c < base + w.rows[s]) return reinterpret_cast<const T*>(w.w[s]) + (size_t)(c - base) * K;
        base += w.rows[s];
    }
    return nullptr;
}

template <typename T, int EPI>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T* __restrict__ X, const T* __restrict__ X_lo, int M,
                                                        int K, GemmW w, int N, EpiParams e) {
    grid_dep_launch();
    grid_dep_wait();
    __shared__ float Xs[BK][BM + 4];
    __shared__ float Ws[BK][BN + 4];
    __shared__ float Us[EPI == EPI_SWIGLU ? BK : 1][BN + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int r0 = blockIdx.y * BM, c0 = blockIdx.x * BN;
    const int lr = tid >> 2, lk = (tid & 3) * 4;
    const int xr = r0 + lr;
    const T* xrow = xr < M ? X + (size_t)xr * K : nullptr;
    const T* xlow = (xr < M && X_lo) ? X_lo + (size_t)xr * K : nullptr;
    const T* wrow = (c0 + lr < N) ? weight_row<T>(w, c0 + lr, K) : nullptr;
    const T* urow = nullptr;
    if (EPI == EPI_SWIGLU && c0 + lr < N) urow = reinterpret_cast<const T*>(w.w_up) + (size_t)(c0 + lr) * K;

    float acc[4][4], accu[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = accu[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            Xs[lk + t][lr] = xrow ? to_f(xrow[k0 + lk + t]) + (xlow ? to_f(xlow[k0 + lk + t]) : 0.f) : 0.f;
            Ws[lk + t][lr] = wrow ? to_f(wrow[k0 + lk + t]) : 0.f;
            if (EPI == EPI_SWIGLU) Us[lk + t][lr] = urow ? to_f(urow[k0 + lk + t]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], b[4], u[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = Xs[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                b[j] = Ws[kk][tx * 4 + j];
                if (EPI == EPI_SWIGLU) u[j] = Us[kk][tx * 4 + j];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                    if (EPI == EPI_SWIGLU) accu[i][j] = fmaf(a[i], u[j], accu[i][j]);
                }
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + ty * 4 + i;
        if (r >= M) continue;
        const int c = c0 + tx * 4;
        if (EPI == EPI_QKV) {
            const int p = epi_pos(e, r);
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                if (c + j >= N) continue;
                int off;
                const int reg = qkv_region(e, c + j + e.qkv_base, off);
                float x0 = acc[i][j], x1 = acc[i][j + 1];
                if (reg < 2) rope_pair(e, p, off, x0, x1);
                qkv_store<T>(e, reg, r, p, off, x0);
                qkv_store<T>(e, reg, r, p, off + 1, x1);
            }
        } else if (EPI == EPI_RESID) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (c + j >= N) continue;
                float* hp = e.h + (size_t)r * e.ldh + c + j;
                if (e.atomic) atomicAdd(hp, acc[i][j]); else *hp += acc[i][j];
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (c + j >= N) continue;
                const float a = silu_mul(acc[i][j], accu[i][j]);
                const T ah = from_f<T>(a);
                reinterpret_cast<T*>(e.act)[(size_t)r * e.ld_act + c + j] = ah;
                if (e.act_lo) reinterpret_cast<T*>(e.act_lo)[(size_t)r * e.ld_act + c + j] = from_f<T>(a - to_f(ah));
            }
        }
    }
}

template <typename T>
cudaError_t launch_t(const void* X, const void* X_lo, int M, int K, const GemmW& w, int N, const EpiParams& e,
                     cudaStream_t s) {
    dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
    const T* x = reinterpret_cast<const T*>(X);
    const T* xl = reinterpret_cast<const T*>(X_lo);
    switch (e.kind) {
        case EPI_QKV: gemm_simt_kernel<T, EPI_QKV><<<grid, 256, 0, s>>>(x, xl, M, K, w, N, e); break;
        case EPI_RESID: gemm_simt_kernel<T, EPI_RESID><<<grid, 256, 0, s>>>(x, xl, M, K, w, N, e); break;
        default: gemm_simt_kernel<T, EPI_SWIGLU><<<grid, 256, 0, s>>>(x, xl, M, K, w, N, e); break;
    }
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_gemm_simt(const Model& m, const void* X, const void* X_lo, int M, int K, const GemmW& w, int N,
                             const EpiParams& e, cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    return m.bf16 ? launch_t<bf16>(X, X_lo, M, K, w, N, e, s) : launch_t<float>(X, nullptr, M, K, w, N, e, s);
}

}  // namespace cb
