// Tensor-core attention of the recomputed queries over the blended K/V on sm_103a (CacheBlend
// deep-dive page, Figure 5: the selected queries attend over every token).
//
// Work unit = (tile of 128/G consecutive recomputed queries, KV head g): its 128 TMEM lanes hold the
// G query heads that share KV head g for each of those queries (row r = query * G + head), so each
// K/V block is read once for the whole GQA group.  Queries are sorted by position; a unit streams
// key blocks 0 .. pos(last query) and masks keys past each row's own position (causal by global
// position).
//   warp 0      TMA producer: the Q tile (4-D box), then 64-key K and V blocks of KV head g
//   warp 1      MMA issuer: S = Q K^T (TMEM), then O_b = P_b V_b (TMEM)
//   warps 2..5  softmax: one thread per row; online max/sum in fp32 (exp2), P written as bf16 into
//               128-byte-swizzled shared memory (the A operand of the second MMA), and the per-block
//               O_b accumulated in registers with the running rescale; final O / l stored as bf16.
// S and O_b are double buffered in TMEM (4 x 128 columns) so the tensor cores run one block ahead
// of the softmax.  V is consumed as an MN-major operand straight from its [key][dim] layout.
#include <cudaTypedefs.h>

#include "cb_ptx.cuh"

namespace cb {

namespace {

constexpr int BKV = 64;                  // keys per block
constexpr int ROWS = 128;                // TMEM lanes per unit
constexpr int NUM_THREADS = 192;

struct AttnArgs {
    int M;              // recomputed query rows
    int G;              // query heads per KV head
    int QT;             // queries per unit = 128 / G
    int n_qt;           // query tiles
    int Hkv, Hq;
    int n_keys;         // rows of the blended K/V
    int kv_z;           // z coordinate of this layer's K block in the K/V map (V is kv_z + 1)
    int units;
    const int* pos;     // [M] positions (NULL: identity)
    bf16* out;          // [M][Hq * hd]
    bf16* out_lo;       // low parts (split precision) or NULL
    float scale_log2;   // log2(e) / sqrt(hd)
    uint32_t idesc_qk, idesc_pv;
    unsigned* status;
};

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// MN-major operand descriptor, 128-byte swizzle: rows of 64 elements (128 B) along the MN
// dimension, 8-row groups along K 1024 B apart (SBO), the next 64 MN elements `lbo` bytes away.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t lbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, unsigned* status) {
    const uint64_t t0 = ptx::global_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::global_ns() - t0 > ptx::kWaitLimitNs) {
            atomicOr(status, ST_WAIT_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void unit_of(const AttnArgs& a, int u, int& qt, int& g) {
    qt = a.n_qt - 1 - u / a.Hkv;     // latest (longest) query tiles first
    g = u % a.Hkv;
}
__device__ __forceinline__ int tile_blocks(const AttnArgs& a, int qt) {
    const int last = min((qt + 1) * a.QT, a.M) - 1;
    const int pmax = a.pos ? a.pos[last] : last;
    return pmax / BKV + 1;
}

template <int HD, bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mql,
                   const __grid_constant__ CUtensorMap mkv, const AttnArgs a) {
    // split precision carries q and P as hi + lo bf16 pairs: two MMAs into the same accumulator
    constexpr int NP = SPLIT ? 2 : 1;
    constexpr int KV_STAGES = SPLIT ? 2 : 3;
    constexpr int HALVES = HD / 64;
    constexpr int Q_BYTES = ROWS * HD * 2;            // one Q tile (hi or lo)
    constexpr int KB_BYTES = BKV * HD * 2;            // one K (or V) block
    constexpr int P_BYTES = ROWS * BKV * 2;           // one P tile (hi or lo)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                               // [NP] Q tiles
    uint8_t* sK = sQ + NP * Q_BYTES;                  // [KV_STAGES] K blocks
    uint8_t* sV = sK + KV_STAGES * KB_BYTES;          // [KV_STAGES] V blocks
    uint8_t* sP = sV + KV_STAGES * KB_BYTES;          // [2 buffers][NP] P tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * NP * P_BYTES);
    uint64_t* q_full = bars;
    uint64_t* q_empty = bars + 1;
    uint64_t* kv_full = bars + 2;
    uint64_t* kv_empty = kv_full + KV_STAGES;
    uint64_t* s_full = kv_empty + KV_STAGES;
    uint64_t* s_empty = s_full + 2;
    uint64_t* p_full = s_empty + 2;
    uint64_t* p_empty = p_full + 2;
    uint64_t* o_full = p_empty + 2;
    uint64_t* o_empty = o_full + 2;
    uint64_t* drain = o_empty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(q_full), 1);
        ptx::mbar_init(ptx::smem_u32(q_empty), 1);
        for (int i = 0; i < KV_STAGES; ++i) {
            ptx::mbar_init(ptx::smem_u32(kv_full + i), 1);
            ptx::mbar_init(ptx::smem_u32(kv_empty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(s_full + i), 1);
            ptx::mbar_init(ptx::smem_u32(s_empty + i), 4);
            ptx::mbar_init(ptx::smem_u32(p_full + i), 4);
            ptx::mbar_init(ptx::smem_u32(p_empty + i), 1);
            ptx::mbar_init(ptx::smem_u32(o_full + i), 1);
            ptx::mbar_init(ptx::smem_u32(o_empty + i), 4);
        }
        ptx::mbar_init(ptx::smem_u32(drain), 1);
        *abort = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tmap(&mq);
        if (SPLIT) ptx::prefetch_tmap(&mql);
        ptx::prefetch_tmap(&mkv);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;       // S buffers at columns 0, 128; O buffers at 256, 384

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t q_cnt = 0, kv_cnt = 0;
            uint32_t issued = 0, issued_par = 0;
            bool q_issued = false;
            uint32_t q_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
                int qt, g;
                unit_of(a, u, qt, g);
                const int nb = tile_blocks(a, qt);
                if (!ptx::mbar_wait(ptx::smem_u32(q_empty), (q_cnt & 1u) ^ 1u, abort, a.status)) break;
                const uint32_t qb = ptx::smem_u32(q_full);
                ptx::mbar_arrive_expect_tx(qb, NP * Q_BYTES);
                for (int h = 0; h < HALVES; ++h) {
                    tma_load_4d(ptx::smem_u32(sQ + h * (ROWS * 128)), &mq, h * 64, 0, g, qt * a.QT, qb);
                    if (SPLIT)
                        tma_load_4d(ptx::smem_u32(sQ + Q_BYTES + h * (ROWS * 128)), &mql, h * 64, 0, g, qt * a.QT, qb);
                }
                q_issued = true;
                q_par = q_cnt & 1u;
                ++q_cnt;
                for (int b = 0; b < nb; ++b) {
                    const int st = kv_cnt % KV_STAGES;
                    const uint32_t par = (kv_cnt / KV_STAGES) & 1u;
                    if (!ptx::mbar_wait(ptx::smem_u32(kv_empty + st), par ^ 1u, abort, a.status)) { ok = false; break; }
                    const uint32_t fb = ptx::smem_u32(kv_full + st);
                    ptx::mbar_arrive_expect_tx(fb, 2 * KB_BYTES);
                    for (int h = 0; h < HALVES; ++h) {
                        tma_load_3d(ptx::smem_u32(sK + st * KB_BYTES + h * (BKV * 128)), &mkv, g * HD + h * 64,
                                    b * BKV, a.kv_z, fb);
                        tma_load_3d(ptx::smem_u32(sV + st * KB_BYTES + h * (BKV * 128)), &mkv, g * HD + h * 64,
                                    b * BKV, a.kv_z + 1, fb);
                    }
                    issued |= 1u << st;
                    issued_par = (issued_par & ~(1u << st)) | (par << st);
                    ++kv_cnt;
                }
            }
            if (q_issued) drain_wait(ptx::smem_u32(q_full), q_par, a.status);
            for (int i = 0; i < KV_STAGES; ++i)
                if (issued & (1u << i)) drain_wait(ptx::smem_u32(kv_full + i), (issued_par >> i) & 1u, a.status);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t q_cnt = 0, kv_cnt = 0, s_cnt = 0, o_cnt = 0;
            bool ok = true;
            auto pv = [&](uint32_t blk_cnt, uint32_t st) -> bool {
                // O_b = P_b V_b for the block whose S was buffer (blk_cnt & 1)
                const int buf = blk_cnt & 1;
                const uint32_t par = (blk_cnt >> 1) & 1u;
                if (!ptx::mbar_wait(ptx::smem_u32(p_full + buf), par, abort, a.status)) return false;
                if (!ptx::mbar_wait(ptx::smem_u32(o_empty + buf), par ^ 1u, abort, a.status)) return false;
                ptx::tc_fence_after();
                const uint32_t pa = ptx::smem_u32(sP + buf * NP * P_BYTES);
                const uint32_t va = ptx::smem_u32(sV + st * KB_BYTES);
#pragma unroll
                for (int kk = 0; kk < BKV / 16; ++kk) {
                    const uint64_t vd = sdesc_mn_sw128(va + kk * 16 * 128, BKV * 128);
                    ptx::mma_bf16(tmem + 256 + buf * 128, ptx::sdesc_sw128(pa + kk * 32), vd, a.idesc_pv,
                                  kk > 0 ? 1u : 0u);
                    if (SPLIT)
                        ptx::mma_bf16(tmem + 256 + buf * 128, ptx::sdesc_sw128(pa + P_BYTES + kk * 32), vd, a.idesc_pv,
                                      1u);
                }
                ptx::mma_commit(ptx::smem_u32(p_empty + buf));
                ptx::mma_commit(ptx::smem_u32(o_full + buf));
                ptx::mma_commit(ptx::smem_u32(kv_empty + st));
                ++o_cnt;
                return true;
            };
            for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
                int qt, g;
                unit_of(a, u, qt, g);
                const int nb = tile_blocks(a, qt);
                if (!ptx::mbar_wait(ptx::smem_u32(q_full), q_cnt & 1u, abort, a.status)) break;
                ++q_cnt;
                uint32_t prev_st = 0;
                for (int b = 0; b < nb; ++b) {
                    const uint32_t st = kv_cnt % KV_STAGES;
                    const uint32_t kpar = (kv_cnt / KV_STAGES) & 1u;
                    ++kv_cnt;
                    const int buf = s_cnt & 1;
                    const uint32_t spar = (s_cnt >> 1) & 1u;
                    if (!ptx::mbar_wait(ptx::smem_u32(kv_full + st), kpar, abort, a.status) ||
                        !ptx::mbar_wait(ptx::smem_u32(s_empty + buf), spar ^ 1u, abort, a.status)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t qa = ptx::smem_u32(sQ), ka = ptx::smem_u32(sK + st * KB_BYTES);
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t off = (kk & 3) * 32;
                        const uint64_t kd = ptx::sdesc_sw128(ka + (kk >> 2) * (BKV * 128) + off);
                        ptx::mma_bf16(tmem + buf * 128, ptx::sdesc_sw128(qa + (kk >> 2) * (ROWS * 128) + off), kd,
                                      a.idesc_qk, kk > 0 ? 1u : 0u);
                        if (SPLIT)
                            ptx::mma_bf16(tmem + buf * 128,
                                          ptx::sdesc_sw128(qa + Q_BYTES + (kk >> 2) * (ROWS * 128) + off), kd,
                                          a.idesc_qk, 1u);
                    }
                    ptx::mma_commit(ptx::smem_u32(s_full + buf));
                    ++s_cnt;
                    if (b > 0 && !pv(s_cnt - 2, prev_st)) { ok = false; break; }
                    prev_st = st;
                }
                if (!ok) break;
                if (!pv(s_cnt - 1, prev_st)) break;
                ptx::mma_commit(ptx::smem_u32(q_empty));
            }
            ptx::mma_commit(ptx::smem_u32(drain));
            drain_wait(ptx::smem_u32(drain), 0, a.status);
            (void)o_cnt;
        }
    } else {
        // ---------------------------------------------------------------- softmax (4 warps)
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        uint32_t s_cnt = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
            int qt, g;
            unit_of(a, u, qt, g);
            const int nb = tile_blocks(a, qt);
            const int qi = qt * a.QT + row / a.G;
            const bool valid = qi < a.M;
            const int prow = valid ? (a.pos ? a.pos[qi] : qi) : 0;
            float m = -INFINITY, l = 0.f, alpha_pend = 0.f;
            float o[HD];
#pragma unroll
            for (int d = 0; d < HD; ++d) o[d] = 0.f;
            for (int b = 0; b <= nb && ok; ++b) {
                if (b < nb) {
                    const int buf = s_cnt & 1;
                    const uint32_t par = (s_cnt >> 1) & 1u;
                    if (!ptx::mbar_wait(ptx::smem_u32(s_full + buf), par, abort, a.status)) { ok = false; break; }
                    ptx::tc_fence_after();
                    float s[BKV];
#pragma unroll
                    for (int c = 0; c < BKV / 16; ++c) ptx::tmem_ld16(tmem + lane_base + buf * 128 + c * 16, s + c * 16);
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(s_empty + buf));
                    const int j0 = b * BKV;
                    float mx = m;
#pragma unroll
                    for (int i = 0; i < BKV; ++i) {
                        s[i] = (j0 + i <= prow) ? s[i] * a.scale_log2 : -INFINITY;
                        mx = fmaxf(mx, s[i]);
                    }
                    const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - mx);
                    float sum = 0.f;
#pragma unroll
                    for (int i = 0; i < BKV; ++i) {
                        s[i] = exp2f(s[i] - mx);
                        sum += s[i];
                    }
                    l = l * alpha + sum;
                    m = mx;
                    // P row (bf16) into the swizzled A-operand buffer
                    if (!ptx::mbar_wait(ptx::smem_u32(p_empty + buf), par ^ 1u, abort, a.status)) { ok = false; break; }
                    uint8_t* prow_ptr = sP + buf * NP * P_BYTES + row * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 w, wl;
                        bf16* hi = reinterpret_cast<bf16*>(&w);
                        bf16* lo = reinterpret_cast<bf16*>(&wl);
#pragma unroll
                        for (int t = 0; t < 8; ++t) split_bf16(s[c * 8 + t], hi[t], lo[t]);
                        *reinterpret_cast<uint4*>(prow_ptr + ((c ^ (row & 7)) << 4)) = w;
                        if (SPLIT) *reinterpret_cast<uint4*>(prow_ptr + P_BYTES + ((c ^ (row & 7)) << 4)) = wl;
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(p_full + buf));
                    // accumulate the previous block's O_b with its own rescale
                    if (b > 0) {
                        const uint32_t ocnt = s_cnt - 1;
                        const int ob = ocnt & 1;
                        const uint32_t opar = (ocnt >> 1) & 1u;
                        if (!ptx::mbar_wait(ptx::smem_u32(o_full + ob), opar, abort, a.status)) { ok = false; break; }
                        ptx::tc_fence_after();
#pragma unroll
                        for (int c = 0; c < HD / 16; ++c) {
                            float t[16];
                            ptx::tmem_ld16(tmem + lane_base + 256 + ob * 128 + c * 16, t);
#pragma unroll
                            for (int i = 0; i < 16; ++i) o[c * 16 + i] = o[c * 16 + i] * alpha_pend + t[i];
                        }
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(o_empty + ob));
                    }
                    alpha_pend = alpha;
                    ++s_cnt;
                } else {
                    // last block's O_b
                    const uint32_t ocnt = s_cnt - 1;
                    const int ob = ocnt & 1;
                    const uint32_t opar = (ocnt >> 1) & 1u;
                    if (!ptx::mbar_wait(ptx::smem_u32(o_full + ob), opar, abort, a.status)) { ok = false; break; }
                    ptx::tc_fence_after();
#pragma unroll
                    for (int c = 0; c < HD / 16; ++c) {
                        float t[16];
                        ptx::tmem_ld16(tmem + lane_base + 256 + ob * 128 + c * 16, t);
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[c * 16 + i] = o[c * 16 + i] * alpha_pend + t[i];
                    }
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(o_empty + ob));
                }
            }
            if (!ok) break;
            if (valid) {
                const float inv = 1.0f / l;
                const int head = g * a.G + row % a.G;
                const size_t at = (size_t)qi * a.Hq * HD + (size_t)head * HD;
#pragma unroll
                for (int c = 0; c < HD / 8; ++c) {
                    uint4 w, wl;
                    bf16* h = reinterpret_cast<bf16*>(&w);
                    bf16* lo = reinterpret_cast<bf16*>(&wl);
#pragma unroll
                    for (int t = 0; t < 8; ++t) split_bf16(o[c * 8 + t] * inv, h[t], lo[t]);
                    *reinterpret_cast<uint4*>(a.out + at + c * 8) = w;
                    if (a.out_lo) *reinterpret_cast<uint4*>(a.out_lo + at + c * 8) = wl;
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encode() {
    if (g_encode) return true;
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return true;
}

template <int HD, bool SPLIT>
size_t attn_smem() {
    const size_t np = SPLIT ? 2 : 1, stages = SPLIT ? 2 : 3;
    return 1024 + np * ROWS * HD * 2 + 2 * stages * (size_t)BKV * HD * 2 + 2 * np * (size_t)ROWS * BKV * 2 + 256;
}

template <int HD, bool SPLIT>
cudaError_t launch_hd(const CUtensorMap& mq, const CUtensorMap& mql, const CUtensorMap& mkv, const AttnArgs& a,
                      int grid, cudaStream_t s) {
    static bool set = false;
    const size_t sm = attn_smem<HD, SPLIT>();
    if (!set) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
        set = true;
    }
    attn_tc_kernel<HD, SPLIT><<<grid, NUM_THREADS, sm, s>>>(mq, mql, mkv, a);
    return cudaGetLastError();
}

}  // namespace

bool attn_tc_supported(const Model& m) {
    const cb_config& c = m.cfg;
    const int G = c.n_heads / c.n_kv_heads;
    return m.bf16 && m.tc && (c.head_dim == 64 || c.head_dim == 128) && (128 % G == 0) && get_encode();
}

// Q map over the q workspace viewed as [rows][Hkv][G][hd]; box {64, G, 1, 128/G}.
bool attn_make_qmap(const Model& m, const void* q, void* map_out) {
    if (!get_encode()) return false;
    const cb_config& c = m.cfg;
    const int G = c.n_heads / c.n_kv_heads;
    cuuint64_t dims[4] = {(cuuint64_t)c.head_dim, (cuuint64_t)G, (cuuint64_t)c.n_kv_heads, (cuuint64_t)c.max_tokens};
    cuuint64_t strides[3] = {(cuuint64_t)c.head_dim * 2, (cuuint64_t)G * c.head_dim * 2,
                             (cuuint64_t)c.n_heads * c.head_dim * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)G, 1, (cuuint32_t)(128 / G)};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode(reinterpret_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q),
                    dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K/V map over a whole blended cache [2L][rows][Hkv * hd]; box {64, 64 keys, 1}.
bool attn_make_kvmap(const Model& m, const void* kv, int64_t rows, void* map_out) {
    if (!get_encode()) return false;
    const cb_config& c = m.cfg;
    const cuuint64_t W = (cuuint64_t)c.n_kv_heads * c.head_dim;
    cuuint64_t dims[3] = {W, (cuuint64_t)rows, (cuuint64_t)(2 * c.n_layers)};
    cuuint64_t strides[2] = {W * 2, W * 2 * (cuuint64_t)rows};
    cuuint32_t box[3] = {64, BKV, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(reinterpret_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kv),
                    dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_attention_tc(const Model& m, const void* qmap, const void* qmap_lo, const void* kvmap, int layer,
                                const int* qpos, int M, int n_keys, void* out, void* out_lo, cudaStream_t s) {
    const cb_config& c = m.cfg;
    AttnArgs a;
    memset(&a, 0, sizeof a);
    a.M = M;
    a.G = c.n_heads / c.n_kv_heads;
    a.QT = 128 / a.G;
    a.n_qt = (M + a.QT - 1) / a.QT;
    a.Hkv = c.n_kv_heads;
    a.Hq = c.n_heads;
    a.n_keys = n_keys;
    a.kv_z = 2 * layer;
    a.units = a.n_qt * a.Hkv;
    a.pos = qpos;
    a.out = reinterpret_cast<bf16*>(out);
    a.out_lo = reinterpret_cast<bf16*>(out_lo);
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)c.head_dim);
    a.idesc_qk = ptx::idesc_bf16(ROWS, BKV);
    a.idesc_pv = ptx::idesc_bf16(ROWS, c.head_dim) | (1u << 16);    // B (V) is MN-major
    a.status = m.status;
    const int grid = a.units < m.num_sms ? a.units : m.num_sms;
    const CUtensorMap& mq = *reinterpret_cast<const CUtensorMap*>(qmap);
    const CUtensorMap& mql = *reinterpret_cast<const CUtensorMap*>(m.split ? qmap_lo : qmap);
    const CUtensorMap& mkv = *reinterpret_cast<const CUtensorMap*>(kvmap);
    if (c.head_dim == 128)
        return m.split ? launch_hd<128, true>(mq, mql, mkv, a, grid, s) : launch_hd<128, false>(mq, mql, mkv, a, grid, s);
    return m.split ? launch_hd<64, true>(mq, mql, mkv, a, grid, s) : launch_hd<64, false>(mq, mql, mkv, a, grid, s);
}

}  // namespace cb
