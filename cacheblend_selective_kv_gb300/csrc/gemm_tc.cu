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
#include <cstdio>
#include <cstdlib>
#include <map>

#include "cb_epilogue.cuh"
#include "cb_ptx.cuh"

namespace cb {

struct TcMaps {
    std::vector<CUtensorMap> wq, wk, wv, wo, wg, wu, wd;   // per layer, box {64, 128}
    std::vector<CUtensorMap> wg64, wu64;                    // per layer, box {64, 64} (paired SwiGLU)
    bool pair = true;                                       // CTA-pair kernel usable
    int pair_clusters[2][4] = {};                           // co-resident clusters per (SPLIT, EPI), 0 = unknown
    const void* xptr[4];                                    // activation buffers (hi) and their row widths
    const void* xptr_lo[4];                                 // low parts (split precision) or NULL
    int xcols[4];
    int rows;
    // token-tile maps, one box of {64, rows} per (buffer, box rows), made on first use
    mutable std::map<int, CUtensorMap> xb[4], xb_lo[4];
};

namespace {

constexpr int BM = 128, BK = 64, TMEM_COLS = 512, NUM_THREADS = 192;
// kernel instance of a QKV-epilogue GEMM in comparing mode (EpiParams::kv_fresh == 2), kept apart so the plain
// QKV instance carries none of its code
constexpr int EPI_KVCMP = 3;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB per weight tile
constexpr int MAX_STAGES = 8;
constexpr int EPI_POS_INTS = 32 * 17;           // per epilogue warp: token positions (QKV) / transposes
constexpr int EPI_STG_WORDS = 512;               // per epilogue warp: QKV store staging (2 KB)
constexpr int EPI_SMEM = 4 * (EPI_POS_INTS * 4 + EPI_STG_WORDS * 4);

struct TcArgs {
    int M, K, x_row0, kb_total, splits, ttiles, BN, stages, units, prefetch;
    int nseg;
    int seg_tiles[3], seg_rows[3], seg_base[3];
    uint32_t idesc;
    EpiParams e;
    unsigned* status;
    // SwiGLU last-wave split: the last `tail` whole units (those of a partial last wave) run as two K halves
    // each, work items full_units + j (first half) and full_units + tail + j (second half)
    int full_units, tail;
    float* tail_part;        // [tail][2 CTAs][128 rows][BN] first-half accumulators
    unsigned* tail_flag;     // [tail][2 CTAs]: 1 once the first half's accumulators are stored; reset to 0 after use
};

struct Unit {
    int seg, lt, t, kb0, kb1, s;   // s: index of the unit's K range (split-K, or the half of a tail unit)
    int tail, j;                    // a K half of tail unit j
};

__device__ __forceinline__ Unit decode_whole(const TcArgs& a, int u);

__device__ __forceinline__ Unit decode_unit(const TcArgs& a, int u) {
    if (u >= a.full_units) {
        const int p = u - a.full_units, h = p >= a.tail ? 1 : 0, j = p - h * a.tail;
        Unit r = decode_whole(a, a.full_units + j);
        const int mid = a.kb_total / 2;
        r.kb0 = h ? mid : 0;
        r.kb1 = h ? a.kb_total : mid;
        r.s = h;
        r.tail = 1;
        r.j = j;
        return r;
    }
    return decode_whole(a, u);
}

__device__ __forceinline__ Unit decode_whole(const TcArgs& a, int u) {
    Unit r;
    r.tail = 0;
    r.j = 0;
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
    r.s = s;
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

// QKV epilogue of one tile: RoPE of q/k pairs (partner feature = lane ^ 1), q as bf16 (hi and, in split
// precision, lo), k/v into the blended cache at each token's position -- or, comparing (CMP), as bf16 rows at
// the GEMM row, each warp also writing the squared difference of its features from the cached row.  A warp's 32
// features are consecutive and lie in one region (regions and segments are multiples of 64 wide), so each
// 16-token chunk is transposed through the warp's shared-memory staging area and written as 16-byte
// vectors along the features of each token row.  Positions come from a per-warp shared-memory copy; the
// (cos, sin) loads run DEEP ? two : one chunk of 16 tokens ahead (the shallow form saves 32 registers
// for kernels with twice the epilogue warps, whose extra warps hide the latency instead).
template <bool DEEP, bool CMP>
__device__ __forceinline__ void qkv_tile(const TcArgs& a, const Unit& w, int row, int lane, int tok0, int ntok,
                                         uint32_t tbase, const int* wpos, uint32_t* stg) {
    const EpiParams& e = a.e;
    const int feat = w.lt * BM + row;
    const bool fv = feat < a.seg_rows[w.seg];               // uniform across the warp
    const int col = a.seg_base[w.seg] + feat + e.qkv_base;
    int off;
    const int reg = qkv_region(e, col, off);
    const int off0 = off - lane;                            // the warp's first feature in its region
    const bool even = (lane & 1) == 0;
    const int half = e.head_dim >> 1, pair = (off % e.head_dim) >> 1;
    const bool rot = reg < 2;
    const int nch = (ntok + 15) / 16;
    // software pipeline: the accumulator columns of chunk c+1 are loaded from TMEM, and the (cos, sin)
    // of chunk c+2 from global memory, while chunk c is processed
    auto rope_at = [&](int t) {
        return (rot && t < ntok) ? e.rope[(size_t)wpos[t] * half + pair] : make_float2(1.f, 0.f);
    };
    float2 cs[16], csn[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        cs[j] = rope_at(j);
        if constexpr (DEEP) csn[j] = rope_at(16 + j);
    }
    uint32_t vn[16];
    ptx::tmem_ld16_issue(tbase, vn);
    for (int c = 0; c < nch; ++c) {
        float v[16];
        ptx::tmem_ld_wait16(vn);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(vn[j]);
        if (c + 1 < nch) ptx::tmem_ld16_issue(tbase + (c + 1) * 16, vn);
        const int base = c * 16;
        float2 csn2[16];
        if constexpr (DEEP) {
            if (c + 2 < nch) {
#pragma unroll
                for (int j = 0; j < 16; ++j) csn2[j] = rope_at(base + 32 + j);
            }
        } else if (c + 1 < nch) {
#pragma unroll
            for (int j = 0; j < 16; ++j) csn[j] = rope_at(base + 16 + j);
        }
        const int nt = min(16, ntok - base);
        float r0[16], r1[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float x = v[j];
            const float y = __shfl_xor_sync(0xffffffffu, x, 1);
            r0[j] = rot ? x * cs[j].x - y * cs[j].y : x;
            r1[j] = rot ? x * cs[j].y + y * cs[j].x : y;
        }
        if (fv) {
            if (CMP && reg > 0) {
                // compare with the stored cache: stage [16 tokens][32 features] fp32, feature f of token j at
                // column f ^ j (reads below are then free of bank conflicts); lane = (token lane & 15, half
                // lane >> 4) sums its 16 squared differences in feature order, the two halves are added and
                // the warp's partial for the token is written once
                float* st = reinterpret_cast<float*>(stg);
                if (even) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        *reinterpret_cast<float2*>(st + j * 32 + ((lane ^ j) & ~1)) =
                            (j & 1) ? make_float2(r1[j], r0[j]) : make_float2(r0[j], r1[j]);
                }
                __syncwarp();
                const int t = lane & 15, hs = lane >> 4;
                const int r = tok0 + base + t;
                float acc = 0.f;
                if (t < nt && r < e.dev_rows) {
                    const bf16* cp = reinterpret_cast<const bf16*>(reg == 1 ? e.cmp_k : e.cmp_v) +
                                     (size_t)wpos[base + t] * e.nkv + off0 + hs * 16;
                    const uint4 u0 = *reinterpret_cast<const uint4*>(cp);
                    const uint4 u1 = *reinterpret_cast<const uint4*>(cp + 8);
                    const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&u0);
                    const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&u1);
                    float c[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 a0 = __bfloat1622float2(h0[i]), a1 = __bfloat1622float2(h1[i]);
                        c[2 * i] = a0.x; c[2 * i + 1] = a0.y; c[8 + 2 * i] = a1.x; c[8 + 2 * i + 1] = a1.y;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float dd = st[t * 32 + ((hs * 16 + i) ^ t)] - c[i];
                        acc = fmaf(dd, dd, acc);
                    }
                }
                acc += __shfl_xor_sync(0xffffffffu, acc, 16);
                if (hs == 0 && t < nt && r < e.dev_rows)
                    e.dev_part[(size_t)r * e.dev_parts + (reg - 1) * (e.nkv >> 5) + (off0 >> 5)] = acc;
                __syncwarp();
            }
            {
                // bf16 rows: stage [16 tokens][16 pairs] (hi, then lo for split q), write 4 x 16 bytes per token
                const bool lo = reg == 0 && e.q_out_lo != nullptr;
                if (even) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        bf16 h0, l0, h1, l1;
                        split_bf16(r0[j], h0, l0);
                        split_bf16(r1[j], h1, l1);
                        __nv_bfloat162 hp = __halves2bfloat162(h0, h1), lp = __halves2bfloat162(l0, l1);
                        stg[j * 16 + (lane >> 1)] = *reinterpret_cast<uint32_t*>(&hp);
                        if (lo) stg[256 + j * 16 + (lane >> 1)] = *reinterpret_cast<uint32_t*>(&lp);
                    }
                }
                __syncwarp();
                bf16* hi_base = reinterpret_cast<bf16*>(reg == 0 ? e.q_out : (reg == 1 ? e.k_dst : e.v_dst)) + off0;
                bf16* lo_base = lo ? reinterpret_cast<bf16*>(e.q_out_lo) + off0 : nullptr;
                const int ld = reg == 0 ? e.nq : e.nkv;
                const bool by_pos = reg > 0 && !CMP;                 // K/V into the cache at the position
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int t = (lane >> 2) + 8 * k, sg = lane & 3;
                    if (t < nt) {
                        const size_t r = by_pos ? (size_t)wpos[base + t] : (size_t)(tok0 + base + t);
                        *reinterpret_cast<uint4*>(hi_base + r * ld + sg * 8) =
                            *reinterpret_cast<const uint4*>(stg + t * 16 + sg * 4);
                        if (lo)
                            *reinterpret_cast<uint4*>(lo_base + r * ld + sg * 8) =
                                *reinterpret_cast<const uint4*>(stg + 256 + t * 16 + sg * 4);
                    }
                }
                __syncwarp();
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            cs[j] = csn[j];
            if constexpr (DEEP) csn[j] = csn2[j];
        }
    }
}

// warm L2 with the (cos, sin) rows of a tile's tokens for this warp's 16 pairs (one 128-byte line per
// token), issued while the tile's MMAs run
__device__ __forceinline__ void qkv_prefetch(const TcArgs& a, const Unit& w, int row, int lane, int tok0, int ntok,
                                             int* wpos) {
    const EpiParams& e = a.e;
    for (int i = lane; i < ntok; i += 32) wpos[i] = epi_pos(e, tok0 + i);
    __syncwarp();
    const int feat = w.lt * BM + row;
    int off;
    const int reg = qkv_region(e, a.seg_base[w.seg] + feat + e.qkv_base, off);
    if (reg == 2 || feat >= a.seg_rows[w.seg]) return;
    const int half = e.head_dim >> 1, pair0 = ((off - lane) % e.head_dim) >> 1;
    for (int i = lane; i < ntok; i += 32) {
        const float2* p = e.rope + (size_t)wpos[i] * half + pair0;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Residual epilogue.  The warp's 32 features x 16 tokens are transposed through shared memory so each
// lane handles four consecutive features of a token with 16-byte accesses.  With one K range the unit
// adds its sum into the residual stream with a vector reduction (h[token][feature] += y; the only writer
// of those elements, so the result is fixed).  With the K range split over S units, unit s stores its sum
// to partial slot s ([M][ldh] each) and the next RMSNorm adds the slots to h in slot order, so the result
// does not depend on which CTA finished first.
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
    const bool slots = a.splits > 1;
    float* dst = slots ? e.part + (size_t)w.s * a.M * e.ldh : e.h;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = (lane >> 3) + 4 * i;                    // token within the chunk
        const int tok = tok0 + j;
        if (tok < a.M && fq < nf) {
            float* hp = dst + (size_t)tok * e.ldh + col0 + fq;
            const float y0 = wst[fq * 17 + j], y1 = wst[(fq + 1) * 17 + j], y2 = wst[(fq + 2) * 17 + j],
                        y3 = wst[(fq + 3) * 17 + j];
            if (fq + 3 < nf) {
                if (slots)
                    *reinterpret_cast<float4*>(hp) = make_float4(y0, y1, y2, y3);
                else
                    red_add_v4(hp, y0, y1, y2, y3);
            } else {
#pragma unroll
                for (int t = 0; t < 3; ++t) {               // at most three features left in this warp
                    if (fq + t >= nf) break;
                    const float yt = t == 0 ? y0 : (t == 1 ? y1 : y2);
                    if (slots) hp[t] = yt; else atomicAdd(hp + t, yt);
                }
            }
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
        bf16 hi, lo;
        split_bf16(silu_mul(g[j], u[j]), hi, lo);
        if (tok < a.M) {                               // predicated: the 16 tokens stay interleaved
            act[(size_t)tok * e.ld_act + feat] = hi;
            if (act_lo) act_lo[(size_t)tok * e.ld_act + feat] = lo;
        }
    }
}

template <int EPI, bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mxl,
                   const __grid_constant__ CUtensorMap mw0, const __grid_constant__ CUtensorMap mw1,
                   const __grid_constant__ CUtensorMap mw2, const TcArgs a) {
    constexpr bool SWIGLU = EPI == EPI_SWIGLU;
    constexpr bool IS_QKV = EPI == EPI_QKV || EPI == EPI_KVCMP;
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
    grid_dep_launch();
    grid_dep_wait();                                     // inputs of the previous kernel are visible

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
            const int tok0 = w.t * a.BN;
            const int ntok = min(a.BN, a.M - tok0);
            int* wpos = spos + (warp - 2) * EPI_POS_INTS;
            if (IS_QKV) qkv_prefetch(a, w, row, lane, tok0, ntok, wpos);
            if (!ptx::mbar_wait(ptx::smem_u32(tfull + acc), acc_phase, abort, a.status)) break;
            ptx::tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256;
            if (IS_QKV) {
                qkv_tile<true, EPI == EPI_KVCMP>(a, w, row, lane, tok0, ntok, tbase, wpos,
                               reinterpret_cast<uint32_t*>(spos + 4 * EPI_POS_INTS) + (warp - 2) * EPI_STG_WORDS);
                __syncwarp();
            }
            for (int c = 0; !IS_QKV && c * 16 < ntok; ++c) {
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


// =================================================================================================
// CTA-pair kernel (cluster of 2, tcgen05 cta_group::2).
//
// One MMA covers M = 256 weight rows: each CTA of the pair stages 128 of them and half of the
// token tile, and its TMEM receives the accumulator of its own 128 rows for all BN tokens.  Per
// MMA cycle a CTA thus writes and reads about two thirds of the shared-memory bytes of the
// single-CTA kernel above, whose split-precision main loop is bound by shared-memory bandwidth.
//   rank 0, warp 0 / rank 1, warp 0   TMA of the own A rows and B half; completion on rank 0's
//                                      full barrier (rank 0 expects both CTAs' bytes)
//   rank 0, warp 1                     MMA issuer; commits release both CTAs' stages and signal
//                                      both CTAs' accumulators
//   both, warps 2..5                   epilogue of the own 128 rows; rank 0's tempty barrier
//                                      counts all 8 epilogue warps
// SwiGLU pairs gate and up rows of the same features in one CTA: rows 0-63 gate and 64-127 up of
// 64 features (the pair covers 128), so each feature's gate and up meet in one CTA's TMEM and the
// epilogue exchanges them between lane quarters q and q ^ 2 through shared memory.
// =================================================================================================
// Pair kernel epilogue warps: two per TMEM lane quarter (each takes half of a tile's 16-token chunks) for
// the QKV and residual epilogues, whose last tile is exposed after the main loop; one per quarter for
// SwiGLU, whose exchange buffers ([quarter][slot][32 x 17] floats) would otherwise cost a pipeline stage.
constexpr int pair_epi_warps(int epi) { return epi == EPI_SWIGLU ? 4 : 8; }
constexpr int pair_threads(int epi) { return 64 + 32 * pair_epi_warps(epi); }
constexpr int pair_epi_smem(int epi) {
    return epi == EPI_SWIGLU ? 4 * 2 * 32 * 17 * 4 : pair_epi_warps(epi) * (EPI_POS_INTS + EPI_STG_WORDS) * 4;
}

__device__ __forceinline__ void epi_swiglu_pair(const TcArgs& a, int feat, bool fv, int q, int lane, int tok0,
                                                int ntok_c, int slot, const float* v, float* xs) {
    const EpiParams& e = a.e;
    float* mine = xs + ((q * 2 + slot) * 32) * 17;
#pragma unroll
    for (int j = 0; j < 16; ++j) mine[lane * 17 + j] = v[j];
    ptx::named_bar_sync(1 + (q & 1), 64);
    const float* gs = xs + (((q & 1) * 2 + slot) * 32) * 17;         // gate quarter (q & 1)
    const float* us = xs + ((((q & 1) + 2) * 2 + slot) * 32) * 17;   // up quarter (q & 1) + 2
    const int j0 = q < 2 ? 0 : 8;                                     // gate warp: tokens 0-7, up warp: 8-15
    if (fv) {
        bf16* act = reinterpret_cast<bf16*>(e.act);
        bf16* act_lo = reinterpret_cast<bf16*>(e.act_lo);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int j = j0 + i;
            bf16 hi, lo;
            split_bf16(silu_mul(gs[lane * 17 + j], us[lane * 17 + j]), hi, lo);
            if (j < ntok_c) {                          // predicated: the 8 tokens stay interleaved
                act[(size_t)(tok0 + j) * e.ld_act + feat] = hi;
                if (act_lo) act_lo[(size_t)(tok0 + j) * e.ld_act + feat] = lo;
            }
        }
    }
    __syncwarp();
}

template <int EPI, bool SPLIT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads(EPI), 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mxl,
                     const __grid_constant__ CUtensorMap mw0, const __grid_constant__ CUtensorMap mw1,
                     const __grid_constant__ CUtensorMap mw2, const TcArgs a) {
    constexpr bool SWIGLU = EPI == EPI_SWIGLU;
    constexpr bool IS_QKV = EPI == EPI_QKV || EPI == EPI_KVCMP;
    constexpr int EW = pair_epi_warps(EPI);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int bh_bytes = (a.BN / 2) * 128;               // this CTA's half of a token tile (hi or lo)
    const int stage_bytes = A_BYTES + (SPLIT ? 2 : 1) * bh_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.stages * stage_bytes);
    uint64_t* full = bars;                               // used in rank 0 only
    uint64_t* empty = bars + MAX_STAGES;
    uint64_t* tfull = bars + 2 * MAX_STAGES;
    uint64_t* tempty = tfull + 2;                        // used in rank 0 only
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_holder + 1);
    float* sepi = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 256);
    int* spos = reinterpret_cast<int*>(sepi);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_rank();
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            ptx::mbar_init(ptx::smem_u32(full + i), 1);
            ptx::mbar_init(ptx::smem_u32(empty + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(tfull + i), 1);
            ptx::mbar_init(ptx::smem_u32(tempty + i), 2 * EW);     // every epilogue warp of both CTAs
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
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_holder), TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();                                 // barriers of both CTAs initialised
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    grid_dep_launch();
    grid_dep_wait();                                     // inputs of the previous kernel are visible

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            const uint32_t full0 = ptx::map_to_rank(ptx::smem_u32(full), 0);
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            bool ok = true;
            for (int u = cluster; u < a.units && ok; u += nclusters) {
                const Unit w = decode_unit(a, u);
                const CUtensorMap* wm = w.seg == 0 ? &mw0 : (w.seg == 1 ? &mw1 : &mw2);
                const int arow = SWIGLU ? w.lt * 128 + (int)rank * 64 : (2 * w.lt + (int)rank) * BM;
                const int r0 = a.x_row0 + w.t * a.BN + (int)rank * (a.BN / 2);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(empty + stage), phase ^ 1u, abort, a.status)) { ok = false; break; }
                    const uint32_t sa = ptx::smem_u32(smem + stage * stage_bytes);
                    const uint32_t fb = full0 + stage * 8;
                    if (rank == 0) ptx::mbar_arrive_expect_tx(ptx::smem_u32(full + stage), 2 * stage_bytes);
                    const int kc = kb * BK;
                    if (SWIGLU) {
                        ptx::tma_load_2d_pair(sa, &mw0, kc, arow, fb);
                        ptx::tma_load_2d_pair(sa + A_BYTES / 2, &mw1, kc, arow, fb);
                    } else {
                        ptx::tma_load_2d_pair(sa, wm, kc, arow, fb);
                    }
                    ptx::tma_load_2d_pair(sa + A_BYTES, &mx, kc, r0, fb);
                    if (SPLIT) ptx::tma_load_2d_pair(sa + A_BYTES + bh_bytes, &mxl, kc, r0, fb);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
            }
            // Before the CTA may exit, every load it issued has landed and every release the MMA
            // issuer multicast to this CTA has arrived: wait for the last release of each stage.
            if (!*abort) {
                for (int i = 0; i < a.stages; ++i)
                    if (issued & (1u << i)) drain_wait(ptx::smem_u32(empty + i), (issued_parity >> i) & 1u, a.status);
            } else {
                const uint64_t t0 = ptx::global_ns();   // error path: give loads in flight time to land
                while (ptx::global_ns() - t0 < 200000ull) {}
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer (rank 0)
        if (lane == 0 && rank == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int u = cluster; u < a.units && ok; u += nclusters) {
                const Unit w = decode_unit(a, u);
                if (!ptx::mbar_wait(ptx::smem_u32(tempty + acc), acc_phase ^ 1u, abort, a.status)) break;
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + acc * 256;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait(ptx::smem_u32(full + stage), phase, abort, a.status)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * stage_bytes);
                    const uint64_t ad = ptx::sdesc_sw128(sa);
                    const uint64_t bd = ptx::sdesc_sw128(sa + A_BYTES);
                    const uint64_t bl = ptx::sdesc_sw128(sa + A_BYTES + bh_bytes);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint32_t accum = (kb > w.kb0 || kk > 0) ? 1u : 0u;
                        ptx::mma_bf16_pair(d, ad + 2 * kk, bd + 2 * kk, a.idesc, accum);
                        if (SPLIT) ptx::mma_bf16_pair(d, ad + 2 * kk, bl + 2 * kk, a.idesc, 1u);
                    }
                    ptx::mma_commit_pair(ptx::smem_u32(empty + stage), 0x3);
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit_pair(ptx::smem_u32(tfull + acc), 0x3);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            ptx::mma_commit_pair(ptx::smem_u32(drain), 0x1);
            drain_wait(ptx::smem_u32(drain), 0, a.status);
        }
    } else {
        // ------------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;                          // TMEM lane quarter this warp may access
        const int ew = warp - 2;                         // epilogue warp index
        const int hs = ew >> 2;                          // which half of a tile's chunks (EW == 8)
        const int row = q * 32 + lane;
        const uint32_t tempty0 = ptx::map_to_rank(ptx::smem_u32(tempty), 0);
        int acc = 0, gc = 0;
        uint32_t acc_phase = 0;
        for (int u = cluster; u < a.units; u += nclusters) {
            Unit w = decode_unit(a, u);
            if (!SWIGLU) w.lt = 2 * w.lt + (int)rank;
            const int tok0 = w.t * a.BN;
            const int ntok = min(a.BN, a.M - tok0);
            // this warp's tokens [ta, tb) of the tile: with two warps per quarter the first takes the
            // first ceil(chunks / 2) chunks of 16, the second the rest (possibly none)
            int ta = 0, tb = ntok;
            if (EW == 8) {
                const int mid = min(ntok, ((ntok + 31) / 32) * 16);
                ta = hs ? mid : 0;
                tb = hs ? ntok : mid;
            }
            int* wpos = spos + ew * EPI_POS_INTS;
            if (IS_QKV && tb > ta) qkv_prefetch(a, w, row, lane, tok0 + ta, tb - ta, wpos);
            if (!ptx::mbar_wait(ptx::smem_u32(tfull + acc), acc_phase, abort, a.status)) break;
            ptx::tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * 256;
            if (IS_QKV) {
                if (tb > ta)
                    qkv_tile<EW == 4, EPI == EPI_KVCMP>(a, w, row, lane, tok0 + ta, tb - ta, tbase + ta, wpos,
                                      reinterpret_cast<uint32_t*>(spos + EW * EPI_POS_INTS) + ew * EPI_STG_WORDS);
                __syncwarp();
            } else if (EPI == EPI_RESID) {
                for (int c = ta / 16; c * 16 < tb; ++c) {
                    float v[16];
                    ptx::tmem_ld16(tbase + c * 16, v);
                    epi_resid(a, w, row, lane, tok0 + c * 16, v, sepi + ew * (32 * 17));
                }
            } else {
                const int feat = w.lt * 128 + (int)rank * 64 + (q & 1) * 32 + lane;
                const bool fv = feat < a.seg_rows[0];
                // a K half of a tail unit: the first half stores its accumulator rows ([lane][token] per CTA) and
                // raises the unit's flag; the second half waits for the flag (bounded), adds the stored rows to
                // its own in a fixed order, and only then forms silu(g) * u
                float* tp = w.tail ? a.tail_part + (((size_t)w.j * 2 + rank) * 128 + q * 32 + lane) * a.BN : nullptr;
                unsigned* tf = w.tail ? a.tail_flag + w.j * 2 + rank : nullptr;
                if (w.tail && w.s == 0) {
                    for (int c = 0; c * 16 < ntok; ++c) {
                        float v[16];
                        ptx::tmem_ld16(tbase + c * 16, v);
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(tp + c * 16 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    }
                    ptx::named_bar_sync(3, 128);                      // every epilogue warp's rows are stored
                    if (ew == 0 && lane == 0) {
                        __threadfence();
                        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(tf), "r"(1u) : "memory");
                    }
                } else {
                    if (w.tail) {
                        if (ew == 0 && lane == 0) {
                            const uint64_t t0 = ptx::global_ns();
                            unsigned f = 0;
                            for (;;) {
                                asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(f) : "l"(tf) : "memory");
                                if (f) break;
                                if (ptx::global_ns() - t0 > ptx::kWaitLimitNs) {
                                    atomicOr(a.status, ST_WAIT_TIMEOUT);
                                    break;
                                }
                            }
                            *tf = 0u;                                    // ready for the next launch
                        }
                        ptx::named_bar_sync(3, 128);
                    }
                    for (int c = 0; c * 16 < ntok; ++c, ++gc) {
                        float v[16];
                        __syncwarp();
                        ptx::tmem_ld16(tbase + c * 16, v);
                        if (w.tail) {
#pragma unroll
                            for (int i = 0; i < 16; i += 4) {
                                const float4 f = *reinterpret_cast<const float4*>(tp + c * 16 + i);
                                v[i] += f.x; v[i + 1] += f.y; v[i + 2] += f.z; v[i + 3] += f.w;
                            }
                        }
                        epi_swiglu_pair(a, feat, fv, q, lane, tok0 + c * 16, min(16, ntok - c * 16), gc & 1, v, sepi);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(tempty0 + acc * 8);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }
    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_sync();                                 // no operation of either CTA still targets the other
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
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
                          const CUtensorMap* w2, const TcArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl) {
    static std::atomic<uint64_t> done{0};
    const cudaError_t e = smem_limit_once(gemm_tc_kernel<EPI, SPLIT>, 232448, done);
    if (e != cudaSuccess) return e;
    return launch_ex(pdl, gemm_tc_kernel<EPI, SPLIT>, dim3(grid), dim3(NUM_THREADS), smem, s, mx, mxl, *w0,
                     w1 ? *w1 : *w0, w2 ? *w2 : *w0, a);
}

template <int EPI, bool SPLIT>
cudaError_t launch_pair(const CUtensorMap& mx, const CUtensorMap& mxl, const CUtensorMap* w0, const CUtensorMap* w1,
                        const CUtensorMap* w2, const TcArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl) {
    static std::atomic<uint64_t> done{0};
    const cudaError_t e = smem_limit_once(gemm_pair_kernel<EPI, SPLIT>, 232448, done);
    if (e != cudaSuccess) return e;
    return launch_ex(pdl, gemm_pair_kernel<EPI, SPLIT>, dim3(grid), dim3(pair_threads(EPI)), smem, s, mx, mxl, *w0,
                     w1 ? *w1 : *w0, w2 ? *w2 : *w0, a);
}

// clusters of the pair kernel that fit on the device at once (one CTA per SM)
template <int EPI, bool SPLIT>
int pair_capacity(size_t smem) {
    cudaFuncSetAttribute(gemm_pair_kernel<EPI, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(pair_threads(EPI), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<EPI, SPLIT>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
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
    t->wg64.resize(L); t->wu64.resize(L);
    bool ok = true;
    for (int l = 0; l < L && ok; ++l) {
        ok = make_map(&t->wq[l], m.wq[l], nq, d, BM, err) && make_map(&t->wk[l], m.wk[l], nkv, d, BM, err) &&
             make_map(&t->wv[l], m.wv[l], nkv, d, BM, err) && make_map(&t->wo[l], m.wo[l], d, nq, BM, err) &&
             make_map(&t->wg[l], m.w_gate[l], F, d, BM, err) && make_map(&t->wu[l], m.w_up[l], F, d, BM, err) &&
             make_map(&t->wd[l], m.w_down[l], d, F, BM, err) && make_map(&t->wg64[l], m.w_gate[l], F, d, 64, err) &&
             make_map(&t->wu64[l], m.w_up[l], F, d, 64, err);
    }
    // CTA pairs need at least one co-resident cluster; CB_GEMM_PAIR=0 keeps the single-CTA kernel
    const char* pe = getenv("CB_GEMM_PAIR");
    t->pair = m.num_sms >= 2 && !(pe && pe[0] == '0');
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
                           const EpiParams& e, cudaStream_t s, int* launches, int* splits) {
    (void)N;
    TcMaps& t = *m.tc;
    const int l = w.layer;
    const bool swiglu = e.kind == EPI_SWIGLU;
    const int kind = (e.kind == EPI_QKV && e.kv_fresh == 2) ? EPI_KVCMP : e.kind;   // kernel instance
    if (e.kind == EPI_QKV && e.kv_fresh == 1) return cudaErrorInvalidValue;          // fp32 rows: CUDA-core path only
    const bool split = m.split;
    const bool pair = t.pair;
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
        case WSEL_GATEUP:
            wm[0] = pair ? &t.wg64[l] : &t.wg[l];
            wm[1] = pair ? &t.wu64[l] : &t.wu[l];
            break;
        default: wm[0] = &t.wd[l]; break;
    }
    // weight tiles: 128 rows per CTA; a pair covers 256 rows (SwiGLU: 128 features, gate + up)
    const int rows_per_tile = pair ? (swiglu ? 128 : 256) : BM;
    a.nseg = swiglu ? 1 : w.nseg;
    int mtiles = 0, base = 0;
    for (int i = 0; i < a.nseg; ++i) {
        a.seg_rows[i] = w.rows[i];
        a.seg_tiles[i] = (w.rows[i] + rows_per_tile - 1) / rows_per_tile;
        a.seg_base[i] = base;
        base += w.rows[i];
        mtiles += a.seg_tiles[i];
    }
    // token tiles: the fewest-padding split into tiles of at most 256 rows (single-CTA SwiGLU,
    // whose gate and up accumulators share one TMEM buffer: 128), multiples of 16
    int bn_max = (swiglu && !pair) ? 128 : 256;
    if (const char* v = getenv("CB_TUNE_BN")) bn_max = std::min(bn_max, std::max(16, atoi(v)));
    // The QKV and comparing GEMMs on CTA pairs run few waves, so there the split is the one with the fewest
    // waves x MMA cycles at its tile width (about 99 cycles up to N = 128, 161 at N = 256, linear between),
    // the fewest padded rows breaking ties.
    int best_T = 0, best_BN = 0;
    const char* twv = getenv("CB_TILE_WAVES");
    const bool by_waves = pair && (e.kind == EPI_QKV || e.kind == EPI_KVCMP) && !(twv && twv[0] == '0');
    double best_c = 1e30;
    for (int T0 = (M + bn_max - 1) / bn_max, T = T0; T <= T0 + (by_waves ? 8 : 2); ++T) {
        int bn = ((M + T - 1) / T + 15) / 16 * 16;
        if (bn < 16) bn = 16;
        if (bn > bn_max) continue;
        const long long pad = (long long)T * bn;
        double c = 0.0;
        if (by_waves) {
            const long long w_est = std::max(1, m.num_sms / 2);
            const long long waves = ((long long)mtiles * T + w_est - 1) / w_est;
            c = waves * (bn <= 128 ? 99.0 : 99.0 + (bn - 128) * (62.0 / 128.0));
        }
        if (!best_T || c < best_c - 1e-9 || (c < best_c + 1e-9 && pad < (long long)best_T * best_BN)) {
            best_T = T;
            best_BN = bn;
            best_c = c;
        }
    }
    a.ttiles = best_T;
    a.BN = best_BN;
    const int epi_smem = pair ? pair_epi_smem(e.kind) : EPI_SMEM;
    const int b_rows = pair ? a.BN / 2 : a.BN;                 // token rows one CTA stages
    const int stage_bytes = (swiglu && !pair ? 2 * A_BYTES : A_BYTES) + (split ? 2 : 1) * b_rows * 128;
    const int budget = 227 * 1024 - 1024 - 256 - epi_smem;
    a.stages = budget / stage_bytes;
    if (a.stages > MAX_STAGES) a.stages = MAX_STAGES;
    if (const char* v = getenv("CB_TUNE_STAGES")) a.stages = std::min(a.stages, std::max(2, atoi(v)));
    if (a.stages < 2) return cudaErrorInvalidConfiguration;
    // one CTA per SM (each holds all 512 TMEM columns)
    const size_t smem = std::max<size_t>(1024 + (size_t)a.stages * stage_bytes + 256 + epi_smem, 120 * 1024);
    // co-resident workers: SMs, or clusters of two
    int workers = m.num_sms;
    if (pair) {
        int& cap = t.pair_clusters[split ? 1 : 0][kind];
        if (cap == 0) {
            switch (kind) {
                case EPI_QKV: cap = split ? pair_capacity<EPI_QKV, true>(smem) : pair_capacity<EPI_QKV, false>(smem); break;
                case EPI_KVCMP:
                    cap = split ? pair_capacity<EPI_KVCMP, true>(smem) : pair_capacity<EPI_KVCMP, false>(smem);
                    break;
                case EPI_RESID:
                    cap = split ? pair_capacity<EPI_RESID, true>(smem) : pair_capacity<EPI_RESID, false>(smem);
                    break;
                default: cap = split ? pair_capacity<EPI_SWIGLU, true>(smem) : pair_capacity<EPI_SWIGLU, false>(smem);
            }
            if (cap <= 0) cap = -1;
        }
        if (cap < 0) return cudaErrorInvalidConfiguration;
        workers = cap;
    }
    // split K only where the epilogue accumulates (residual adds): pick the split that minimises the
    // GEMM's waves x (k-blocks per unit + 2 blocks of per-unit latency), in microseconds, plus the time to
    // write the S partial-sum slots and read them back in the next RMSNorm.  A k-block is 4 k-steps (8 MMAs
    // split) of about 99 cycles up to N = 128 and 161 at N = 256 (linear between), at ~2 GHz; the slots move
    // at ~20 TB/s while they fit in L2 next to the rest (48 MB) and at ~5 TB/s from HBM beyond.
    a.splits = 1;
    if (e.kind == EPI_RESID) {
        double best = 1e30;
        int smax = 8;
        if (const char* v = getenv("CB_TUNE_SPLITK")) smax = std::min(8, std::max(1, atoi(v)));   // 8 slots at most
        const char* sm = getenv("CB_SPLIT_TRAFFIC");
        const bool traffic = !(sm && sm[0] == '0');
        const double mma = a.BN <= 128 ? 99.0 : 99.0 + (a.BN - 128) * (62.0 / 128.0);
        const double t_kb = (split ? 8.0 : 4.0) * mma / 2000.0;                          // us per k-block
        const double slot_mb = (double)M * N * 4.0 / 1e6;
        for (int S = 1; S <= smax; ++S) {
            if (a.kb_total / S < 4) break;
            if (S > 1 && (!e.part || (long long)S * M > e.part_rows)) break;   // the partial slots must fit
            const long long units = (long long)mtiles * a.ttiles * S;
            const long long waves = (units + workers - 1) / workers;
            double cost = waves * ((double)a.kb_total / S + 2.0) * t_kb;
            if (traffic && S > 1) cost += 2.0 * S * slot_mb / (S * slot_mb <= 48.0 ? 20.0 : 5.0);   // MB / (TB/s) = us
            if (cost < best - 1e-9) { best = cost; a.splits = S; }
        }
    }
    a.units = mtiles * a.ttiles * a.splits;
    if (splits) *splits = a.splits;
    // SwiGLU on CTA pairs: a partial last wave of T whole units runs as 2T K halves when they fit in one wave
    // (the idle clusters take the second halves); the tail pieces keep weight-tile order, so the token tiles of
    // a weight tile still stream the same weight k-blocks together
    a.full_units = a.units;
    a.tail = 0;
    if (swiglu && pair && m.tail_part && a.kb_total >= 8) {
        const char* tv = getenv("CB_SWIGLU_TAIL");
        const int T = a.units % workers;
        if (!(tv && tv[0] == '0') && T > 0 && 2 * T <= workers && T <= m.tail_units && a.BN <= 256) {
            a.tail = T;
            a.full_units = a.units - T;
            a.units = a.full_units + 2 * T;
            a.tail_part = m.tail_part;
            a.tail_flag = m.tail_flag;
        }
    }
    a.prefetch = 0;
    if (!pair)
        if (const char* v = getenv("CB_TUNE_PF")) a.prefetch = std::max(0, atoi(v));
    a.idesc = ptx::idesc_bf16(pair ? 256 : BM, a.BN);
    const int grid = pair ? 2 * std::min(a.units, workers) : std::min(a.units, workers);
    if (getenv("CB_DEBUG_LAUNCH"))
        fprintf(stderr, "cb gemm: epi %d rows %d K %d N %d | BN %d token tiles %d weight tiles %d splits %d units %d "
                        "(tail %d) workers %d grid %d stages %d\n", e.kind, M, K, N, a.BN, a.ttiles, mtiles, a.splits,
                a.units, a.tail, workers, grid, a.stages);
    if (launches) *launches = 1;
    auto tile_map = [&](std::map<int, CUtensorMap>& cache, const void* ptr, CUtensorMap** out) -> bool {
        auto it = cache.find(b_rows);
        if (it == cache.end()) {
            CUtensorMap mp;
            std::string err;
            if (!make_map(&mp, ptr, (uint64_t)t.rows, (uint64_t)t.xcols[xbuf], (uint32_t)b_rows, err)) return false;
            it = cache.emplace(b_rows, mp).first;
        }
        *out = &it->second;
        return true;
    };
    CUtensorMap *pmx = nullptr, *pmxl = nullptr;
    if (!tile_map(t.xb[xbuf], t.xptr[xbuf], &pmx)) return cudaErrorInvalidValue;
    if (split && !tile_map(t.xb_lo[xbuf], t.xptr_lo[xbuf], &pmxl)) return cudaErrorInvalidValue;
    const CUtensorMap& mx = *pmx;
    const CUtensorMap& mxl = split ? *pmxl : *pmx;
#define CB_GEMM_DISPATCH(LAUNCH)                                                                     \
    do {                                                                                             \
        if (split) {                                                                                 \
            switch (kind) {                                                                          \
                case EPI_QKV: return LAUNCH<EPI_QKV, true>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s, m.pdl);     \
                case EPI_KVCMP: return LAUNCH<EPI_KVCMP, true>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s, m.pdl); \
                case EPI_RESID: return LAUNCH<EPI_RESID, true>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s, m.pdl); \
                default: return LAUNCH<EPI_SWIGLU, true>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s, m.pdl);       \
            }                                                                                        \
        }                                                                                            \
        switch (kind) {                                                                              \
            case EPI_QKV: return LAUNCH<EPI_QKV, false>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s, m.pdl);        \
            case EPI_KVCMP: return LAUNCH<EPI_KVCMP, false>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s, m.pdl);    \
            case EPI_RESID: return LAUNCH<EPI_RESID, false>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s, m.pdl);    \
            default: return LAUNCH<EPI_SWIGLU, false>(mx, mxl, wm[0], wm[1], wm[2], a, grid, smem, s, m.pdl);          \
        }                                                                                            \
    } while (0)
    if (pair) CB_GEMM_DISPATCH(launch_pair);
    CB_GEMM_DISPATCH(launch_kernel);
#undef CB_GEMM_DISPATCH
}

}  // namespace cb
