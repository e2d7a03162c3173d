// Tensor-core GEMM of the blend's projections on sm_103a: tcgen05.mma (bf16 operands, fp32
// accumulators in TMEM), operands staged by TMA in 128-byte-swizzled shared memory, persistent CTAs
// with warp specialisation:
//   warp 0      TMA producer (one thread): weight tile + token-row tile per 64-wide k-block
//   warp 1      MMA issuer (one thread) and TMEM owner
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, fused epilogue, global stores
//
// Orientation ("swap AB"): the weight rows (output features) are the MMA's M dimension (128 per
// tile) and the token rows its N dimension (16..256 per tile), so the few hundred recomputed rows
// of a selective layer fill an N tile with little padding:
//   D[feature][token] = sum_k W[feature][k] * X[token][k]
// Accumulators are double buffered in TMEM (2 x 256 columns) so the epilogue of one tile overlaps
// the main loop of the next.  The SwiGLU GEMM computes a gate tile and an up tile of the same 128
// features into two accumulators, so each epilogue thread holds gate and up of its feature.
// The residual GEMMs may split K across CTAs; their epilogue adds into the fp32 residual stream
// with atomic adds.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <map>

#include "cb_epilogue.cuh"
#include "cb_ptx.cuh"

namespace cb {

struct TcMaps {
    std::vector<CUtensorMap> wq, wk, wv, wo, wg, wu, wd;   // per layer, box {64, 128}
    const void* xptr[4];                                    // activation buffers (hi) and their row widths
    const void* xptr_lo[4];                                 // low parts (split precision) or NULL
    int xcols[4];
    int rows;
    // token-tile maps, one box of {64, BN} rows per (buffer, BN), made on first use
    mutable std::map<int, CUtensorMap> xb[4], xb_lo[4];
};

namespace {

constexpr int BM = 128, BK = 64, TMEM_COLS = 512, NUM_THREADS = 192;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB per weight tile
constexpr int MAX_STAGES = 8;
constexpr int EPI_SMEM = 4 * 32 * 17 * 4;   // per-epilogue-warp staging (token positions / transposes)

struct TcArgs {
    int M, K, x_row0, kb_total, splits, ttiles, BN, stages, units, prefetch;
    int nseg;
    int seg_tiles[3], seg_rows[3], seg_base[3];
    uint32_t idesc;
    EpiParams e;
    unsigned* status;
};

struct Unit {
    int seg, lt, t, kb0, kb1;
};

__device__ __forceinline__ Unit decode_unit(const TcArgs& a, int u) {
    Unit r;
    r.t = u % a.ttiles;
    const int rest = u / a.ttiles;
    const int s = rest % a.splits;
    int mt = rest / a.splits;
    r.seg = 0;
    while (r.seg < a.nseg - 1 && mt >= a.seg_tiles[r.seg]) {
        mt -= a.seg_tiles[r.seg];
        ++r.seg;
    }
    r.lt = mt;
    r.kb0 = (int)((long long)a.kb_total * s / a.splits);
    r.kb1 = (int)((long long)a.kb_total * (s + 1) / a.splits);
    return r;
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

// ---- epilogues: one thread = one feature (TMEM lane), 16 consecutive token rows -------------------
template <typename T>
__device__ __forceinline__ void store_pair(T* p, float a, float b);
template <>
__device__ __forceinline__ void store_pair<bf16>(bf16* p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}

// QKV epilogue of one tile: RoPE of q/k pairs (partner feature = lane ^ 1), q as bf16 (hi and, in split
// precision, lo), k/v either into the blended cache at each token's position or as fp32 rows.
// Positions come from a per-warp shared-memory copy; the (cos, sin) loads of the next 16 tokens are
// issued before the current 16 are processed.
__device__ __forceinline__ void qkv_tile(const TcArgs& a, const Unit& w, int row, int lane, int tok0, int ntok,
                                         uint32_t tbase, const int* wpos) {
    const EpiParams& e = a.e;
    const int feat = w.lt * BM + row;
    const bool fv = feat < a.seg_rows[w.seg];
    const int col = a.seg_base[w.seg] + feat + e.qkv_base;
    int off;
    const int reg = qkv_region(e, col, off);
    const bool even = (lane & 1) == 0;
    const int half = e.head_dim >> 1, pair = (off % e.head_dim) >> 1;
    const bool rot = reg < 2;
    const int nch = (ntok + 15) / 16;
    float2 cs[16], csn[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        cs[j] = (rot && j < ntok) ? e.rope[(size_t)wpos[j] * half + pair] : make_float2(1.f, 0.f);
    for (int c = 0; c < nch; ++c) {
        float v[16];
        ptx::tmem_ld16(tbase + c * 16, v);
        const int base = c * 16;
        if (c + 1 < nch) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int t = base + 16 + j;
                csn[j] = (rot && t < ntok) ? e.rope[(size_t)wpos[t] * half + pair] : make_float2(1.f, 0.f);
            }
        }
        const int nt = min(16, ntok - base);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j >= nt) break;                     // uniform across the warp
            const int tok = tok0 + base + j;
            const float x = v[j];
            const float y = __shfl_xor_sync(0xffffffffu, x, 1);
            if (even && fv) {
                float x0 = x, x1 = y;
                if (rot) {
                    x0 = x * cs[j].x - y * cs[j].y;
                    x1 = x * cs[j].y + y * cs[j].x;
                }
                if (reg == 0) {
                    bf16 h0, l0, h1, l1;
                    split_bf16(x0, h0, l0);
                    split_bf16(x1, h1, l1);
                    *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<bf16*>(e.q_out) + (size_t)tok * e.nq + off) =
                        __halves2bfloat162(h0, h1);
                    if (e.q_out_lo)
                        *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<bf16*>(e.q_out_lo) + (size_t)tok * e.nq +
                                                           off) = __halves2bfloat162(l0, l1);
                } else {
                    void* dst = reg == 1 ? e.k_dst : e.v_dst;
                    if (e.kv_fresh)
                        *reinterpret_cast<float2*>(reinterpret_cast<float*>(dst) + (size_t)tok * e.nkv + off) =
                            make_float2(x0, x1);
                    else
                        store_pair<bf16>(reinterpret_cast<bf16*>(dst) + (size_t)wpos[base + j] * e.nkv + off, x0, x1);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) cs[j] = csn[j];
    }
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Residual epilogue: h[token][feature] += y.  The warp's 32 features x 16 tokens are transposed
// through shared memory so each lane adds four consecutive features of a token with one 16-byte
// vector reduction (the K range may be split across CTAs, hence the atomic adds).
__device__ __forceinline__ void epi_resid(const TcArgs& a, const Unit& w, int row, int lane, int tok0, const float* v,
                                          float* wst) {
    const EpiParams& e = a.e;
    const int feat0 = w.lt * BM + (row - lane);               // first feature of this warp
    const int col0 = a.seg_base[w.seg] + feat0;
#pragma unroll
    for (int j = 0; j < 16; ++j) wst[lane * 17 + j] = v[j];   // [feature][token]
    __syncwarp();
    const int nf = a.seg_rows[w.seg] - feat0;                 // valid features in this warp (may be < 32)
    const int fq = (lane & 7) * 4;                            // 4 features
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = (lane >> 3) + 4 * i;                    // token within the chunk
        const int tok = tok0 + j;
        if (tok < a.M && fq < nf) {
            float* hp = e.h + (size_t)tok * e.ldh + col0 + fq;
            if (fq + 3 < nf)
                red_add_v4(hp, wst[fq * 17 + j], wst[(fq + 1) * 17 + j], wst[(fq + 2) * 17 + j], wst[(fq + 3) * 17 + j]);
            else
                for (int t = 0; fq + t < nf; ++t) atomicAdd(hp + t, wst[(fq + t) * 17 + j]);
        }
    }
    __syncwarp();
}

__device__ __forceinline__ void epi_swiglu(const TcArgs& a, const Unit& w, int row, int tok0, const float* g,
                                           const float* u) {
    const EpiParams& e = a.e;
    const int feat = w.lt * BM + row;
    if (feat >= a.seg_rows[0]) return;
    bf16* act = reinterpret_cast<bf16*>(e.act);
    bf16* act_lo = reinterpret_cast<bf16*>(e.act_lo);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int tok = tok0 + j;
        if (tok >= a.M) break;
        bf16 hi, lo;
        split_bf16(silu_mul(g[j], u[j]), hi, lo);
        act[(size_t)tok * e.ld_act + feat] = hi;
        if (act_lo) act_lo[(size_t)tok * e.ld_act + feat] = lo;
    }
}

template <int EPI, bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mxl,
                   const __grid_constant__ CUtensorMap mw0, const __grid_constant__ CUtensorMap mw1,
                   const __grid_constant__ CUtensorMap mw2, const TcArgs a) {
    constexpr bool SWIGLU = EPI == EPI_SWIGLU;
    constexpr int A_STAGE = SWIGLU ? 2 * A_BYTES : A_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int b_bytes = a.BN * 128;                      // one token-row tile (hi or lo)
    const int stage_bytes = A_STAGE + (SPLIT ? 2 : 1) * b_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.stages * stage_bytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + MAX_STAGES;
    uint64_t* tfull = bars + 2 * MAX_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_holder + 1);
    float* sepi = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 256);  // [4 warps][32 x 17]
    int* spos = reinterpret_cast<int*>(sepi);                                        // [4 warps][256] (QKV)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            ptx::mbar_init(ptx::smem_u32(full + i), 1);
            ptx::mbar_init(ptx::smem_u32(empty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(tfull + i), 1);
            ptx::mbar_init(ptx::smem_u32(tempty + i), 4);
        }
        ptx::mbar_init(ptx::smem_u32(drain), 1);
        *abort = 0;
        ptx::fence_barrier_init();
        ptx::prefetch_tmap(&mx);
        if (SPLIT) ptx::prefetch_tmap(&mxl);
        ptx::prefetch_tmap(&mw0);
        if (a.nseg > 1 || SWIGLU) ptx::prefetch_tmap(&mw1);
        if (a.nseg > 2) ptx::prefetch_tmap(&mw2);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;                   // bit i: stage i has a load in flight or landed
            uint32_t issued_parity = 0;            // bit i: parity of that load's phase
            bool ok = true;
            // L2 prefetch cursor: walks the same (unit, k-block) sequence PREFETCH_KB steps ahead
            int pu = blockIdx.x, pkb = 0;
            Unit pw;
            bool pvalid = pu < a.units;
            if (pvalid) { pw = decode_unit(a, pu); pkb = pw.kb0; }
            auto prefetch_step = [&]() {
                if (!pvalid) return;
                const int kc = pkb * BK;
                if (SWIGLU) {
                    ptx::tma_prefetch_2d(&mw0, kc, pw.lt * BM);
                    ptx::tma_prefetch_2d(&mw1, kc, pw.lt * BM);
                } else {
                    ptx::tma_prefetch_2d(pw.seg == 0 ? &mw0 : (pw.seg == 1 ? &mw1 : &mw2), kc, pw.lt * BM);
                }
                if (++pkb >= pw.kb1) {
                    pu += gridDim.x;
                    pvalid = pu < a.units;
                    if (pvalid) { pw = decode_unit(a, pu); pkb = pw.kb0; }
                }
            };
            if (a.prefetch == 0) pvalid = false;
            for (int i = 0; i < a.prefetch; ++i) prefetch_step();
            for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
                const Unit w = decode_unit(a, u);
                const CUtensorMap* wm = w.seg == 0 ? &mw0 : (w.seg == 1 ? &mw1 : &mw2);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(empty + stage), phase ^ 1u, abort, a.status)) { ok = false; break; }
                    const uint32_t sa = ptx::smem_u32(smem + stage * stage_bytes);
                    const uint32_t fb = ptx::smem_u32(full + stage);
                    ptx::mbar_arrive_expect_tx(fb, stage_bytes);
                    const int kc = kb * BK;
                    if (SWIGLU) {
                        ptx::tma_load_2d(sa, &mw0, kc, w.lt * BM, fb);
                        ptx::tma_load_2d(sa + A_BYTES, &mw1, kc, w.lt * BM, fb);
                    } else {
                        ptx::tma_load_2d(sa, wm, kc, w.lt * BM, fb);
                    }
                    const uint32_t sb = sa + A_STAGE;
                    const int r0 = a.x_row0 + w.t * a.BN;
                    ptx::tma_load_2d(sb, &mx, kc, r0, fb);                 // the whole token tile, one box
                    if (SPLIT) ptx::tma_load_2d(sb + b_bytes, &mxl, kc, r0, fb);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    prefetch_step();
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
            }
            // every load this thread issued has landed before the CTA may exit
            for (int i = 0; i < a.stages; ++i)
                if (issued & (1u << i)) drain_wait(ptx::smem_u32(full + i), (issued_parity >> i) & 1u, a.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
                const Unit w = decode_unit(a, u);
                if (!ptx::mbar_wait(ptx::smem_u32(tempty + acc), acc_phase ^ 1u, abort, a.status)) break;
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + acc * 256;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(full + stage), phase, abort, a.status)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * stage_bytes);
                    const uint64_t ad = ptx::sdesc_sw128(sa);
                    const uint64_t au = ptx::sdesc_sw128(sa + A_BYTES);
                    const uint64_t bd = ptx::sdesc_sw128(sa + A_STAGE);
                    const uint64_t bl = ptx::sdesc_sw128(sa + A_STAGE + b_bytes);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint32_t accum = (kb > w.kb0 || kk > 0) ? 1u : 0u;
                        ptx::mma_bf16(d, ad + 2 * kk, bd + 2 * kk, a.idesc, accum);
                        if (SPLIT) ptx::mma_bf16(d, ad + 2 * kk, bl + 2 * kk, a.idesc, 1u);
                        if (SWIGLU) {
                            ptx::mma_bf16(d + 128, au + 2 * kk, bd + 2 * kk, a.idesc, accum);
                            if (SPLIT) ptx::mma_bf16(d + 128, au + 2 * kk, bl + 2 * kk, a.idesc, 1u);
                        }
                    }
                    ptx::mma_commit(ptx::smem_u32(empty + stage));
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit(ptx::smem_u32(tfull + acc));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // all MMAs issued by this thread have completed before TMEM is released
            ptx::mma_commit(ptx::smem_u32(drain));
            drain_wait(ptx::smem_u32(drain), 0, a.status);
        }
    } else {
        // ------------------------------------------------------------------ epilogue (4 warps)
        const int q = warp & 3;                    // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;             // feature within the tile
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
            const Unit w = decode_unit(a, u);
            if (!ptx::mbar_wait(ptx::smem_u32(tfull + acc), acc_phase, abort, a.status)) break;
            ptx::tc_fence_after();
            const int tok0 = w.t * a.BN;
            const int ntok = min(a.BN, a.M - tok0);
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256;
            if (EPI == EPI_QKV) {
                int* wpos = spos + (warp - 2) * (32 * 17);
                for (int i = lane; i < ntok; i += 32) wpos[i] = epi_pos(a.e, tok0 + i);
                __syncwarp();
                qkv_tile(a, w, row, lane, tok0, ntok, tbase, wpos);
                __syncwarp();
            }
            for (int c = 0; EPI != EPI_QKV && c * 16 < ntok; ++c) {
                float v[16];
                ptx::tmem_ld16(tbase + c * 16, v);
                if (EPI == EPI_RESID) {
                    epi_resid(a, w, row, lane, tok0 + c * 16, v, sepi + (warp - 2) * (32 * 17));
                } else {
                    float up[16];
                    ptx::tmem_ld16(tbase + 128 + c * 16, up);
                    epi_swiglu(a, w, row, tok0 + c * 16, v, up);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(tempty + acc));
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows, std::string& err) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")";
        return false;
    }
    return true;
}

template <int EPI, bool SPLIT>
cudaError_t launch_kernel(const CUtensorMap& mx, const CUtensorMap& mxl, const CUtensorMap* w0, const CUtensorMap* w1,
                          const CUtensorMap* w2, const TcArgs& a, int grid, size_t smem, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(gemm_tc_kernel<EPI, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    gemm_tc_kernel<EPI, SPLIT><<<grid, NUM_THREADS, smem, s>>>(mx, mxl, *w0, w1 ? *w1 : *w0, w2 ? *w2 : *w0, a);
    return cudaGetLastError();
}

}  // namespace

bool tc_init(Model& m, std::string& err) {
    const char* off = getenv("CB_DISABLE_TC");
    if (off && off[0] == '1') {
        err = "disabled by CB_DISABLE_TC";
        return false;
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, m.device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, m.device);
    if (major != 10 || minor != 3) {
        err = "tensor-core kernels are built for sm_103a";
        return false;
    }
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
            err = "cuTensorMapEncodeTiled unavailable";
            return false;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cb_config& c = m.cfg;
    const uint64_t d = c.d_model, nq = (uint64_t)c.n_heads * c.head_dim, nkv = (uint64_t)c.n_kv_heads * c.head_dim;
    const uint64_t F = c.ffn_hidden, T = c.max_tokens;
    TcMaps* t = new TcMaps();
    const int L = c.n_layers;
    t->wq.resize(L); t->wk.resize(L); t->wv.resize(L); t->wo.resize(L); t->wg.resize(L); t->wu.resize(L);
    t->wd.resize(L);
    bool ok = true;
    for (int l = 0; l < L && ok; ++l) {
        ok = make_map(&t->wq[l], m.wq[l], nq, d, BM, err) && make_map(&t->wk[l], m.wk[l], nkv, d, BM, err) &&
             make_map(&t->wv[l], m.wv[l], nkv, d, BM, err) && make_map(&t->wo[l], m.wo[l], d, nq, BM, err) &&
             make_map(&t->wg[l], m.w_gate[l], F, d, BM, err) && make_map(&t->wu[l], m.w_up[l], F, d, BM, err) &&
             make_map(&t->wd[l], m.w_down[l], d, F, BM, err);
    }
    t->xptr[XBUF_X] = m.x; t->xptr[XBUF_XA] = m.xA; t->xptr[XBUF_ATTN] = m.attn; t->xptr[XBUF_ACT] = m.act;
    t->xptr_lo[XBUF_X] = m.x_lo; t->xptr_lo[XBUF_XA] = m.xA_lo; t->xptr_lo[XBUF_ATTN] = m.attn_lo;
    t->xptr_lo[XBUF_ACT] = m.act_lo;
    t->xcols[XBUF_X] = (int)d; t->xcols[XBUF_XA] = (int)d; t->xcols[XBUF_ATTN] = (int)nq; t->xcols[XBUF_ACT] = (int)F;
    t->rows = (int)T;
    if (!ok) {
        delete t;
        return false;
    }
    m.tc = t;
    return true;
}

void tc_destroy(Model& m) {
    delete m.tc;
    m.tc = nullptr;
}

cudaError_t launch_gemm_tc(const Model& m, int xbuf, int x_row0, int M, int K, const GemmW& w, int N,
                           const EpiParams& e, cudaStream_t s, int* launches) {
    (void)N;
    const TcMaps& t = *m.tc;
    const int l = w.layer;
    const bool swiglu = e.kind == EPI_SWIGLU;
    TcArgs a;
    memset(&a, 0, sizeof a);
    a.M = M;
    a.K = K;
    a.x_row0 = x_row0;
    a.kb_total = K / BK;
    a.e = e;
    a.status = m.status;
    const CUtensorMap* wm[3] = {nullptr, nullptr, nullptr};
    switch (w.which) {
        case WSEL_QKV: wm[0] = &t.wq[l]; wm[1] = &t.wk[l]; wm[2] = &t.wv[l]; break;
        case WSEL_Q: wm[0] = &t.wq[l]; break;
        case WSEL_KV: wm[0] = &t.wk[l]; wm[1] = &t.wv[l]; break;
        case WSEL_O: wm[0] = &t.wo[l]; break;
        case WSEL_GATEUP: wm[0] = &t.wg[l]; wm[1] = &t.wu[l]; break;
        default: wm[0] = &t.wd[l]; break;
    }
    a.nseg = swiglu ? 1 : w.nseg;
    int mtiles = 0, base = 0;
    for (int i = 0; i < a.nseg; ++i) {
        a.seg_rows[i] = w.rows[i];
        a.seg_tiles[i] = (w.rows[i] + BM - 1) / BM;
        a.seg_base[i] = base;
        base += w.rows[i];
        mtiles += a.seg_tiles[i];
    }
    // token tiles: the fewest-padding split into tiles of at most 256 (128 for SwiGLU) rows
    int bn_max = swiglu ? 128 : 256;
    if (const char* t = getenv("CB_TUNE_BN")) bn_max = std::min(bn_max, std::max(16, atoi(t)));
    int best_T = 0, best_BN = 0;
    for (int T0 = (M + bn_max - 1) / bn_max, T = T0; T <= T0 + 2; ++T) {
        int bn = ((M + T - 1) / T + 15) / 16 * 16;
        if (bn < 16) bn = 16;
        if (bn > bn_max) continue;
        if (!best_T || (long long)T * bn < (long long)best_T * best_BN) { best_T = T; best_BN = bn; }
    }
    a.ttiles = best_T;
    a.BN = best_BN;
    // split K only where the epilogue accumulates (residual adds): pick the split that minimises
    // waves x (k-blocks per unit + 2 blocks of per-unit latency)
    a.splits = 1;
    if (e.kind == EPI_RESID) {
        double best = 1e30;
        int smax = 8;
        if (const char* t = getenv("CB_TUNE_SPLITK")) smax = std::max(1, atoi(t));
        for (int S = 1; S <= smax; ++S) {
            if (a.kb_total / S < 4) break;
            const long long units = (long long)mtiles * a.ttiles * S;
            const long long waves = (units + m.num_sms - 1) / m.num_sms;
            const double cost = waves * ((double)a.kb_total / S + 2.0);
            if (cost < best - 1e-9) { best = cost; a.splits = S; }
        }
    }
    a.units = mtiles * a.ttiles * a.splits;
    const bool split = m.split;
    const int stage_bytes = (swiglu ? 2 * A_BYTES : A_BYTES) + (split ? 2 : 1) * a.BN * 128;
    const int budget = 227 * 1024 - 1024 - 256 - EPI_SMEM;
    a.stages = budget / stage_bytes;
    if (a.stages > MAX_STAGES) a.stages = MAX_STAGES;
    if (const char* t = getenv("CB_TUNE_STAGES")) a.stages = std::min(a.stages, std::max(2, atoi(t)));
    a.prefetch = 0;
    if (const char* t = getenv("CB_TUNE_PF")) a.prefetch = std::max(0, atoi(t));
    if (a.stages < 2) return cudaErrorInvalidConfiguration;
    a.idesc = ptx::idesc_bf16(BM, a.BN);
    const size_t smem = 1024 + (size_t)a.stages * stage_bytes + 256 + EPI_SMEM;
    const int grid = a.units < m.num_sms ? a.units : m.num_sms;
    if (launches) *launches = 1;
    auto tile_map = [&](std::map<int, CUtensorMap>& cache, const void* base, CUtensorMap** out) -> bool {
        auto it = cache.find(a.BN);
        if (it == cache.end()) {
            CUtensorMap mp;
            std::string err;
            if (!make_map(&mp, base, (uint64_t)t.rows, (uint64_t)t.xcols[xbuf], (uint32_t)a.BN, err)) return false;
            it = cache.emplace(a.BN, mp).first;
        }
        *out = &it->second;
        return true;
    };
    CUtensorMap *pmx = nullptr, *pmxl = nullptr;
    if (!tile_map(t.xb[xbuf], t.xptr[xbuf], &pmx)) return cudaErrorInvalidValue;
    if (split && !tile_map(t.xb_lo[xbuf], t.xptr_lo[xbuf], &pmxl)) return cudaErrorInvalidValue;
    const CUtensorMap& mx = *pmx;
    const CUtensorMap& mxl = split ? *pmxl : *pmx;
    if (split) {
        switch (e.kind) {
            case EPI_QKV: return launch_kernel<EPI_QKV, true>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s);
            case EPI_RESID: return launch_kernel<EPI_RESID, true>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s);
            default: return launch_kernel<EPI_SWIGLU, true>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s);
        }
    }
    switch (e.kind) {
        case EPI_QKV: return launch_kernel<EPI_QKV, false>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s);
        case EPI_RESID: return launch_kernel<EPI_RESID, false>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s);
        default: return launch_kernel<EPI_SWIGLU, false>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s);
    }
}

}  // namespace cb
