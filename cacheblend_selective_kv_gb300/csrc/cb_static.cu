// Re-RoPE of a chunk-cache buffer that allocates no device memory.
//
// cb_rerope needs a model handle, whose creation allocates a workspace sized for whole blends.
// Some callers cannot do that: a KV-cache manager that has already reserved nearly all device
// memory for its own block pool (where a late cudaMalloc fails or fragments the pool), or code
// that must not call the allocator at all.  They only need to move cached chunks to new positions,
// which takes no weights and only a small per-call table: each chunk's start and the (cos, sin) of
// its position delta.  Here that table lives in a file-scope device array of fixed size, so a call
// only launches two kernels.
//
// The array is shared by every call in the process (one copy per device that loads the library,
// held until exit).  Each call writes every table entry it reads before reading it, so nothing
// needs to start at zero; calls whose GPU work overlaps (different streams, or threads that do
// not serialise their streams) race on it and must be serialised by the caller.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "cb_common.cuh"

namespace {

constexpr int kMaxChunks = CB_STATIC_MAX_CHUNKS;
constexpr int kMaxHalf = 64;                           // head_dim <= 128
constexpr size_t kCsBytes = sizeof(float2) * kMaxChunks * kMaxHalf;
constexpr size_t kScratchBytes = kCsBytes + sizeof(int) * kMaxChunks;
constexpr int kMaxDevices = 64;

// the scratch: [kMaxChunks][kMaxHalf] float2 (cos, sin), then [kMaxChunks] int chunk starts
static __device__ __align__(256) unsigned char g_rerope_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

cb_status fail(cb_status code, const char* msg) {
    cb::set_last_error(msg);
    return code;
}

struct StaticChunks {
    int n;
    int dst[kMaxChunks];
    int delta[kMaxChunks];
};

struct InvFreq {
    double v[kMaxHalf];
};

__global__ void static_delta_kernel(StaticChunks t, InvFreq f, int half, unsigned char* scratch) {
    float2* cs = reinterpret_cast<float2*>(scratch);
    int* dst = reinterpret_cast<int*>(scratch + kCsBytes);
    const int c = blockIdx.x;
    if (c >= t.n) return;
    if (threadIdx.x == 0) dst[c] = t.dst[c];
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        double s, co;
        sincos((double)t.delta[c] * f.v[i], &s, &co);
        cs[(size_t)c * kMaxHalf + i] = make_float2((float)co, (float)s);
    }
}

template <typename T>
__device__ __forceinline__ void load8(const T* p, float* f);
template <>
__device__ __forceinline__ void load8<float>(const float* p, float* f) {
    float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<cb::bf16>(const cb::bf16* p, float* f) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
template <typename T>
__device__ __forceinline__ void store8(T* p, const float* f);
template <>
__device__ __forceinline__ void store8<float>(float* p, const float* f) {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}
template <>
__device__ __forceinline__ void store8<cb::bf16>(cb::bf16* p, const float* f) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
}

// K rows of every layer rotated by their chunk's delta; V untouched (in place)
template <typename T>
__global__ void static_rerope_kernel(T* kv, int64_t rows, int n_ctx, int W, int hd, int L, int n_chunks,
                                     const unsigned char* scratch) {
    const float2* cs = reinterpret_cast<const float2*>(scratch);
    const int* cdst = reinterpret_cast<const int*>(scratch + kCsBytes);
    const int W8 = W / 8;
    const int64_t per_layer = (int64_t)n_ctx * W8;
    const int64_t total = (int64_t)L * per_layer;
    for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < total;
         it += (int64_t)gridDim.x * blockDim.x) {
        // 64-bit throughout: one layer of a large buffer can hold more than 2^31 vectors
        const int64_t layer = it / per_layer;
        const int64_t rem = it - layer * per_layer;
        const int64_t j = rem / W8;
        const int e = (int)(rem - j * W8) * 8;
        int lo = 0, hi = n_chunks - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)cdst[mid] <= j) lo = mid; else hi = mid - 1;
        }
        T* p = kv + (layer * 2 * rows + j) * W + e;
        float f[8];
        load8<T>(p, f);
        const float2* t = cs + (size_t)lo * kMaxHalf + (e % hd) / 2;
        for (int q = 0; q < 4; ++q) {
            const float2 y = cb::rotate_pair(f[2 * q], f[2 * q + 1], t[q]);
            f[2 * q] = y.x;
            f[2 * q + 1] = y.y;
        }
        store8<T>(p, f);
    }
}

// Device address of the scratch on the current device, queried once per device and kept for the life
// of the process: the library must not be used on a device after cudaDeviceReset there (the array's
// address may change with the new context).
cb_status scratch_on_current_device(unsigned char** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(CB_ERR_CUDA, "cb_rerope_static: no usable current CUDA device");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_rerope_scratch);
        if (e != cudaSuccess || !p) {
            char msg[200];
            snprintf(msg, sizeof msg, "cb_rerope_static: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            return fail(CB_ERR_CUDA, msg);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
    return CB_OK;
}

}  // namespace

extern "C" {

cb_status cb_rerope_static(void* kv, int64_t n_rows, int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
                           double rope_theta, int32_t dtype, const cb_chunk* chunks, int32_t n_chunks, void* stream) {
    cb::set_last_error("");
    if (!kv) return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: kv is NULL");
    if (n_layers < 1 || n_kv_heads < 1 || n_rows < 0) return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: bad shape");
    if (head_dim != 64 && head_dim != 128) return fail(CB_ERR_UNSUPPORTED, "cb_rerope_static: head_dim must be 64 or 128");
    if ((int64_t)n_kv_heads * head_dim > (int64_t)1 << 24)
        return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: n_kv_heads * head_dim exceeds 2^24");
    if (dtype != CB_F32 && dtype != CB_BF16) return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: dtype must be CB_F32 or CB_BF16");
    if (!(rope_theta > 0)) return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: rope_theta must be > 0");
    if (n_chunks < 0 || (n_chunks > 0 && !chunks)) return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: bad chunk list");
    if (n_chunks > kMaxChunks) {
        char msg[160];
        snprintf(msg, sizeof msg, "cb_rerope_static: %d chunks exceed the no-allocation limit of %d chunks", n_chunks,
                 kMaxChunks);
        return fail(CB_ERR_INVALID_ARG, msg);
    }
    if ((uintptr_t)kv % 16) return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: kv must be 16-byte aligned");
    StaticChunks t;
    t.n = n_chunks;
    int64_t at = 0;
    for (int i = 0; i < n_chunks; ++i) {
        const cb_chunk& c = chunks[i];
        if (c.src_pos < 0) return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: unknown source position (src_pos < 0)");
        if (c.len <= 0 || c.dst_pos != at)
            return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: chunks must tile [0, n_ctx) in order");
        at += c.len;
        t.dst[i] = c.dst_pos;
        t.delta[i] = c.dst_pos - c.src_pos;
    }
    if (at > n_rows) return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: chunks cover more rows than the buffer has");
    if (at > INT32_MAX) return fail(CB_ERR_INVALID_ARG, "cb_rerope_static: chunks cover more than 2^31 - 1 rows");
    if (n_chunks == 0) return CB_OK;
    unsigned char* scratch = nullptr;
    cb_status st = scratch_on_current_device(&scratch);
    if (st != CB_OK) return st;
    const int half = head_dim / 2;
    InvFreq f;
    for (int i = 0; i < half; ++i) f.v[i] = std::pow(rope_theta, -2.0 * (double)i / (double)head_dim);
    cudaStream_t s = (cudaStream_t)stream;
    static_delta_kernel<<<n_chunks, 64, 0, s>>>(t, f, half, scratch);
    const int W = n_kv_heads * head_dim;
    const int64_t items = (int64_t)n_layers * at * (W / 8);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t grid = (items + 255) / 256;
    if (grid > (int64_t)sms * 16) grid = (int64_t)sms * 16;
    if (grid < 1) grid = 1;
    if (dtype == CB_BF16)
        static_rerope_kernel<cb::bf16><<<(int)grid, 256, 0, s>>>((cb::bf16*)kv, n_rows, (int)at, W, head_dim, n_layers,
                                                                n_chunks, scratch);
    else
        static_rerope_kernel<float><<<(int)grid, 256, 0, s>>>((float*)kv, n_rows, (int)at, W, head_dim, n_layers,
                                                             n_chunks, scratch);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof msg, "cb_rerope_static: launch failed: %s", cudaGetErrorString(e));
        return fail(CB_ERR_CUDA, msg);
    }
    return CB_OK;
}

}  // extern "C"
