// Tensor-core attention of the recomputed queries over the blended K/V on sm_103a (CacheBlend
// deep-dive page, Figure 5: the selected queries attend over every token).
//
// Work unit = (tile of 128/G consecutive recomputed queries, KV head g): its 128 TMEM lanes hold the
// G query heads that share KV head g for each of those queries (row r = query * G + head), so each
// K/V block is read once for the whole GQA group.  Queries are sorted by position; a unit streams
// 128-key blocks 0 .. pos(last query) and masks keys past each row's own position (causal by global
// position).
//   warp 0      TMA producer of the Q tile (4-D box) and the K blocks (3-stage ring)
//   warp 10     TMA producer of the V blocks (2-stage ring)
//   warp 1      S issuer: S = Q K^T into a TMEM buffer
//   warp 11     PV issuer: O_h += P_h V_h with P read from TMEM
//   warps 2..9  softmax, two warps per TMEM lane quarter: the warps of half h own keys 64h..64h+63
//               of every block, keep their own running max and sum, and overwrite their S columns
//               with P_h (bf16; in split precision a hi and a lo part), which the PV MMA reads as its
//               A operand straight from tensor memory.  O_h lives in TMEM and is rescaled only when
//               that half's running max grows by more than 2^8 (exp2 domain), so P stays below 256.
// At the end of a unit the half-1 warps combine both halves: O = (O_0 2^(m_0-M) + O_1 2^(m_1-M)) / l.
// S/P is double buffered in TMEM; a buffer is reused for S once the PV MMAs that read its P are done.
// K blocks are released as soon as their S MMAs complete and V blocks once their PV MMAs do, so the
// K loads run up to three blocks ahead.
// At N = 128 one tcgen05.mma executes in about as many cycles as one thread needs to issue it, so the
// S and PV MMAs come from two threads (each one's waits and commits overlap the other's issue) and both
// keep their per-block bookkeeping small: one wait for P (both halves' warps arrive on one barrier), no
// barrier of their own for V stages or for O (the V producer and the softmax warps wait on the S/P
// buffer's free barrier, which completes at the same point), and descriptors formed once per block.
// V is consumed as an MN-major operand from its [key][dim] layout.  The persistent CTAs claim units at
// run time (longest query tiles first) from a counter in global memory; long key ranges are cut into
// parts merged by attn_combine_kernel.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>

#include "cb_ptx.cuh"

namespace cb {

namespace {

constexpr int BKV = 128;                 // keys per block
constexpr int HK = 64;                   // keys per softmax half
constexpr int ROWS = 128;                // TMEM lanes per unit
constexpr int NUM_THREADS = 384;         // K producer, S issuer, 8 softmax warps, V producer, PV issuer
constexpr int V_WARP = 10, PV_WARP = 11;
constexpr int K_STAGES = 3, V_STAGES = 2;
constexpr float RESCALE_LOG2 = 8.0f;     // lazy-rescale threshold (P <= 2^8)
constexpr int SCHED_SLOTS = 4;           // work items published ahead to the consumer roles
constexpr int SCHED_READERS = 11;        // V producer, the two MMA issuers, 8 softmax warps

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
    int parts;          // key-range parts per (query tile, KV head); 1 = write the normalised output
    int part_blocks;    // key blocks per part
    float* part_o;      // parts > 1: [unit * parts + part][128][hd] unnormalised O
    float* part_ml;     // parts > 1: [unit * parts + part][128][2] (max in exp2 domain, sum)
    float scale_log2;   // log2(e) / sqrt(hd)
    uint32_t idesc_qk, idesc_pv;
    unsigned* status;
    unsigned* sched;    // [0] next work item to claim, [1] CTAs finished claiming; both zero between launches
};

// 2^x on the special-function unit (about 2 ulp; the result feeds a bf16 hi+lo pair)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M = 128 rows in the lanes, K = 16 bf16 packed two per 32-bit
// column, 8 columns) read from tensor memory; one thread issues it
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x 32-bit, 16 consecutive columns per thread (raw words)
__device__ __forceinline__ void tmem_st16_u(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
          "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo_k, float hi_k) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo_k, hi_k);      // .x (lower key) in the low 16 bits
    return *reinterpret_cast<uint32_t*>(&t);
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

// A wait that, when it gives up, records where (once per launch) in the diagnostic words after the
// status bits: {magic, barrier code, parity, counter, block, warp, unit}.
__device__ __forceinline__ bool await(uint32_t bar, uint32_t parity, volatile int* abort, unsigned* status, int code,
                                      uint32_t cnt, int unit) {
    if (ptx::mbar_wait(bar, parity, abort, status)) return true;
    if (atomicCAS(status + 1, 0u, 0xA77Eu) == 0u) {
        status[2] = (unsigned)code;
        status[3] = parity;
        status[4] = cnt;
        status[5] = blockIdx.x;
        status[6] = threadIdx.x >> 5;
        status[7] = (unsigned)unit;
    }
    return false;
}

// work item u -> query tile (latest, i.e. longest, first), KV head and key-range part
__device__ __forceinline__ void unit_of(const AttnArgs& a, int u, int& qt, int& g, int& part) {
    part = u % a.parts;
    const int rest = u / a.parts;
    qt = a.n_qt - 1 - rest / a.Hkv;
    g = rest % a.Hkv;
}
__device__ __forceinline__ int tile_blocks(const AttnArgs& a, int qt) {
    const int last = min((qt + 1) * a.QT, a.M) - 1;
    int pmax = a.pos ? a.pos[last] : last;
    if (pmax < 0 || pmax >= a.n_keys) {             // a position outside the cache: record, clamp
        atomicOr(a.status, ST_BAD_ROW);
        pmax = pmax < 0 ? 0 : a.n_keys - 1;
    }
    return pmax / BKV + 1;
}

// key blocks [b0, b1) of an item (empty when the part starts past the tile's last position)
__device__ __forceinline__ void item_blocks(const AttnArgs& a, int qt, int part, int& b0, int& b1) {
    const int nb = tile_blocks(a, qt);
    b0 = part * a.part_blocks;
    b1 = min(b0 + a.part_blocks, nb);
}

template <int HD, bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mql,
                   const __grid_constant__ CUtensorMap mkv, const AttnArgs a) {
    // split precision carries q and P as hi + lo bf16 pairs: two MMAs into the same accumulator
    constexpr int NP = SPLIT ? 2 : 1;
    constexpr int HALVES = HD / 64;
    constexpr int Q_BYTES = ROWS * HD * 2;            // one Q tile (hi or lo)
    constexpr int KB_BYTES = BKV * HD * 2;            // one K (or V) block
    constexpr uint32_t S_COL = 0, O_COL = 256;        // TMEM: S/P buffers at 0 / 128, O_h at 256 + HD h
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                               // [NP] Q tiles
    uint8_t* sK = sQ + NP * Q_BYTES;                  // [K_STAGES] K blocks
    uint8_t* sV = sK + K_STAGES * KB_BYTES;           // [V_STAGES] V blocks
    float* cmb = reinterpret_cast<float*>(sV + V_STAGES * KB_BYTES);   // [128][2] half-0 (max, sum)
    uint64_t* bars = reinterpret_cast<uint64_t*>(cmb + 2 * ROWS);
    uint64_t* q_full = bars;
    uint64_t* q_empty = bars + 1;
    uint64_t* k_full = bars + 2;
    uint64_t* k_empty = k_full + K_STAGES;
    uint64_t* v_full = k_empty + K_STAGES;
    uint64_t* s_full = v_full + V_STAGES;             // [buffer]: S written
    uint64_t* s_free = s_full + 2;                    // [buffer]: the PV MMAs reading its P are done
    uint64_t* p_full = s_free + 2;                    // [buffer]: P written by the 8 softmax warps
    uint64_t* o_free = p_full + 2;
    uint64_t* cmb_bar = o_free + 1;
    uint64_t* drain = cmb_bar + 1;                    // [issuer]: its last MMAs are done
    uint64_t* sched_full = drain + 2;                 // [slot]: a work item (or -1: none left) published
    uint64_t* sched_empty = sched_full + SCHED_SLOTS; // [slot]: every consumer role has read it
    int* sched_u = reinterpret_cast<int*>(sched_empty + SCHED_SLOTS);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sched_u + SCHED_SLOTS);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(q_full), 1);
        ptx::mbar_init(ptx::smem_u32(q_empty), 1);
        for (int i = 0; i < K_STAGES; ++i) {
            ptx::mbar_init(ptx::smem_u32(k_full + i), 1);
            ptx::mbar_init(ptx::smem_u32(k_empty + i), 1);
        }
        for (int i = 0; i < V_STAGES; ++i) {
            ptx::mbar_init(ptx::smem_u32(v_full + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(s_full + i), 1);
            ptx::mbar_init(ptx::smem_u32(s_free + i), 1);
        }
        for (int i = 0; i < 2; ++i) ptx::mbar_init(ptx::smem_u32(p_full + i), 8);
        ptx::mbar_init(ptx::smem_u32(o_free), 4);
        ptx::mbar_init(ptx::smem_u32(cmb_bar), 4);
        ptx::mbar_init(ptx::smem_u32(drain), 1);
        ptx::mbar_init(ptx::smem_u32(drain + 1), 1);
        for (int i = 0; i < SCHED_SLOTS; ++i) {
            ptx::mbar_init(ptx::smem_u32(sched_full + i), 1);
            ptx::mbar_init(ptx::smem_u32(sched_empty + i), SCHED_READERS);
        }
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
    const uint32_t tmem = *tmem_holder;
    grid_dep_launch();
    grid_dep_wait();                                     // q and the blended K/V of the previous kernels

    // Work items are claimed at run time from a global counter, in unit order (longest query tiles
    // first), by the Q/K producer, which skips empty items and publishes each claim through a ring of
    // SCHED_SLOTS shared-memory slots; every other role reads the same sequence from the ring.  Returns
    // the item, -1 when none is left, -2 when a wait gave up.  Called by a whole softmax warp or by the
    // single thread of the V producer and of each MMA issuer.
    uint32_t sched_cnt = 0;
    auto next_unit = [&](bool warp_wide) -> int {
        const uint32_t slot = sched_cnt % SCHED_SLOTS, par = (sched_cnt / SCHED_SLOTS) & 1u;
        if (!await(ptx::smem_u32(sched_full + slot), par, abort, a.status, 61, sched_cnt, -1)) return -2;
        const int v = *reinterpret_cast<volatile int*>(sched_u + slot);
        if (warp_wide) __syncwarp();
        if (!warp_wide || lane == 0) ptx::mbar_arrive(ptx::smem_u32(sched_empty + slot));
        ++sched_cnt;
        return v;
    };

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer: Q and K
        if (lane == 0) {
            uint32_t q_cnt = 0, k_cnt = 0;
            uint32_t issued = 0, issued_par = 0;
            bool q_issued = false;
            uint32_t q_par = 0;
            bool ok = true;
            while (ok) {
                int u, qt = 0, g = 0, part = 0, b0 = 0, b1 = 0;
                do {                                     // claim the next non-empty item
                    u = (int)atomicAdd(a.sched, 1u);
                    if (u >= a.units) break;
                    unit_of(a, u, qt, g, part);
                    item_blocks(a, qt, part, b0, b1);
                } while (b0 >= b1);
                const bool none = u >= a.units;
                {
                    const uint32_t slot = sched_cnt % SCHED_SLOTS, par = (sched_cnt / SCHED_SLOTS) & 1u;
                    if (!await(ptx::smem_u32(sched_empty + slot), par ^ 1u, abort, a.status, 60, sched_cnt, u)) break;
                    sched_u[slot] = none ? -1 : u;
                    ptx::mbar_arrive(ptx::smem_u32(sched_full + slot));
                    ++sched_cnt;
                }
                if (none) break;
                if (!await(ptx::smem_u32(q_empty), (q_cnt & 1u) ^ 1u, abort, a.status, 1, q_cnt, u)) break;
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
                for (int b = b0; b < b1; ++b) {
                    const int st = k_cnt % K_STAGES;
                    const uint32_t par = (k_cnt / K_STAGES) & 1u;
                    if (!await(ptx::smem_u32(k_empty + st), par ^ 1u, abort, a.status, 2, k_cnt, u)) { ok = false; break; }
                    const uint32_t fb = ptx::smem_u32(k_full + st);
                    ptx::mbar_arrive_expect_tx(fb, KB_BYTES);
                    for (int h = 0; h < HALVES; ++h)
                        tma_load_3d(ptx::smem_u32(sK + st * KB_BYTES + h * (BKV * 128)), &mkv, g * HD + h * 64,
                                    b * BKV, a.kv_z, fb);
                    issued |= 1u << st;
                    issued_par = (issued_par & ~(1u << st)) | (par << st);
                    ++k_cnt;
                }
            }
            // claiming is over for this CTA; the last CTA to get here re-arms the counter for the next launch
            __threadfence();
            if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
                atomicExch(a.sched, 0u);
                atomicExch(a.sched + 1, 0u);
            }
            // every load this thread issued has landed before the CTA may exit
            if (q_issued) drain_wait(ptx::smem_u32(q_full), q_par, a.status);
            for (int i = 0; i < K_STAGES; ++i)
                if (issued & (1u << i)) drain_wait(ptx::smem_u32(k_full + i), (issued_par >> i) & 1u, a.status);
        }
    } else if (warp == V_WARP) {
        // ---------------------------------------------------------------- TMA producer: V
        if (lane == 0) {
            uint32_t v_cnt = 0, issued = 0, issued_par = 0;
            bool ok = true;
            while (ok) {
                const int u = next_unit(false);
                if (u < 0) break;
                int qt, g, part, b0, b1;
                unit_of(a, u, qt, g, part);
                item_blocks(a, qt, part, b0, b1);
                for (int b = b0; b < b1; ++b) {
                    const int st = v_cnt % V_STAGES;
                    const uint32_t par = (v_cnt / V_STAGES) & 1u;
                    // V block v_cnt uses stage v_cnt % 2, as its S uses buffer v_cnt % 2: the stage is free
                    // once that buffer's PV MMAs (two blocks back) are done
                    if (!await(ptx::smem_u32(s_free + st), par ^ 1u, abort, a.status, 7, v_cnt, u)) { ok = false; break; }
                    const uint32_t fb = ptx::smem_u32(v_full + st);
                    ptx::mbar_arrive_expect_tx(fb, KB_BYTES);
                    for (int h = 0; h < HALVES; ++h)
                        tma_load_3d(ptx::smem_u32(sV + st * KB_BYTES + h * (BKV * 128)), &mkv, g * HD + h * 64,
                                    b * BKV, a.kv_z + 1, fb);
                    issued |= 1u << st;
                    issued_par = (issued_par & ~(1u << st)) | (par << st);
                    ++v_cnt;
                }
            }
            for (int i = 0; i < V_STAGES; ++i)
                if (issued & (1u << i)) drain_wait(ptx::smem_u32(v_full + i), (issued_par >> i) & 1u, a.status);
        }
    } else if (warp == PV_WARP) {
        // ---------------------------------------------------------------- PV issuer
        if (lane == 0) {
            uint32_t v_cnt = 0, sc = 0, unit_cnt = 0;
            bool ok = true;
            while (ok) {
                const int u = next_unit(false);
                if (u < 0) break;
                int qt, g, part, b0, b1;
                unit_of(a, u, qt, g, part);
                item_blocks(a, qt, part, b0, b1);
                const int nb = b1 - b0;
                // O_h += P_h V_h for each block (P in the block's S buffer)
                for (int b = 0; b < nb; ++b, ++sc) {
                    const bool first = b == 0;
                    const int buf = sc & 1;
                    const uint32_t par = (sc >> 1) & 1u;
                    const uint32_t st = v_cnt % V_STAGES, vpar = (v_cnt / V_STAGES) & 1u;
                    if (first && !await(ptx::smem_u32(o_free), (unit_cnt & 1u) ^ 1u, abort, a.status, 3, unit_cnt, u)) {
                        ok = false;
                        break;
                    }
                    if (!await(ptx::smem_u32(v_full + st), vpar, abort, a.status, 8, v_cnt, u) ||
                        !await(ptx::smem_u32(p_full + buf), par, abort, a.status, 10, sc, u)) {
                        ok = false;
                        break;
                    }
                    ++v_cnt;
                    ptx::tc_fence_after();
                    const uint64_t vd0 = sdesc_mn_sw128(ptx::smem_u32(sV + st * KB_BYTES), BKV * 128);
                    const uint32_t pt = tmem + S_COL + buf * 128;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int kk = 0; kk < HK / 16; ++kk) {
                            const int key = h * HK + kk * 16;
                            const uint64_t vd = vd0 + (uint64_t)((key * 128) >> 4);
                            const uint32_t acc0 = (first && kk == 0) ? 0u : 1u;
                            mma_bf16_tmem_a(tmem + O_COL + h * HD, pt + h * 64 + kk * 8, vd, a.idesc_pv, acc0);
                            if (SPLIT)
                                mma_bf16_tmem_a(tmem + O_COL + h * HD, pt + h * 64 + 32 + kk * 8, vd, a.idesc_pv, 1u);
                        }
                    }
                    ptx::mma_commit(ptx::smem_u32(s_free + buf));
                }
                ++unit_cnt;
            }
            ptx::mma_commit(ptx::smem_u32(drain + 1));
            drain_wait(ptx::smem_u32(drain + 1), 0, a.status);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- S issuer
        if (lane == 0) {
            uint32_t q_cnt = 0, k_cnt = 0, s_cnt = 0;
            bool ok = true;
            while (ok) {
                const int u = next_unit(false);
                if (u < 0) break;
                int qt, g, part, b0, b1;
                unit_of(a, u, qt, g, part);
                item_blocks(a, qt, part, b0, b1);
                const int nb = b1 - b0;
                if (!await(ptx::smem_u32(q_full), q_cnt & 1u, abort, a.status, 4, q_cnt, u)) break;
                ++q_cnt;
                for (int b = 0; b < nb; ++b) {
                    const uint32_t st = k_cnt % K_STAGES;
                    const uint32_t kpar = (k_cnt / K_STAGES) & 1u;
                    ++k_cnt;
                    const int buf = s_cnt & 1;
                    const uint32_t spar = (s_cnt >> 1) & 1u;
                    if (!await(ptx::smem_u32(k_full + st), kpar, abort, a.status, 5, k_cnt, u) ||
                        !await(ptx::smem_u32(s_free + buf), spar ^ 1u, abort, a.status, 6, s_cnt, u)) { ok = false; break; }
                    ptx::tc_fence_after();
                    // descriptors of the tiles' first k-step; a k-step's start address is a constant offset (the
                    // address field holds address / 16, and every address stays below 256 KB)
                    const uint64_t qd0 = ptx::sdesc_sw128(ptx::smem_u32(sQ));
                    const uint64_t kd0 = ptx::sdesc_sw128(ptx::smem_u32(sK + st * KB_BYTES));
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t off = (kk & 3) * 32;
                        const uint64_t kd = kd0 + (uint64_t)(((kk >> 2) * (BKV * 128) + off) >> 4);
                        const uint64_t qd = qd0 + (uint64_t)(((kk >> 2) * (ROWS * 128) + off) >> 4);
                        ptx::mma_bf16(tmem + S_COL + buf * 128, qd, kd, a.idesc_qk, kk > 0 ? 1u : 0u);
                        if (SPLIT)
                            ptx::mma_bf16(tmem + S_COL + buf * 128, qd + (uint64_t)(Q_BYTES >> 4), kd, a.idesc_qk, 1u);
                    }
                    ptx::mma_commit(ptx::smem_u32(s_full + buf));
                    ptx::mma_commit(ptx::smem_u32(k_empty + st));
                    if (b == nb - 1) ptx::mma_commit(ptx::smem_u32(q_empty));
                    ++s_cnt;
                }
            }
            ptx::mma_commit(ptx::smem_u32(drain));
            drain_wait(ptx::smem_u32(drain), 0, a.status);
        }
    } else {
        // ---------------------------------------------------------------- softmax (8 warps)
        const int q4 = warp & 3;                      // TMEM lane quarter
        const int hf = (warp - 2) >> 2;               // key half of every block
        const int row = q4 * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const uint32_t o_tm = tmem + lane_base + O_COL + hf * HD;
        uint32_t sc = 0, unit_cnt = 0;
        bool ok = true;
        while (ok) {
            const int u = next_unit(true);
            if (u < 0) break;
            int qt, g, part, b0, b1;
            unit_of(a, u, qt, g, part);
            item_blocks(a, qt, part, b0, b1);
            const int nb = b1 - b0;
            const int qi = qt * a.QT + row / a.G;
            const bool valid = qi < a.M;
            const int prow = valid ? (a.pos ? a.pos[qi] : qi) : 0;
            const int prow_min = __reduce_min_sync(0xffffffffu, prow);
            float m_run = -INFINITY, m_used = -INFINITY, l = 0.f;
            for (int b = 0; b < nb; ++b) {
                const int buf = sc & 1;
                const uint32_t par = (sc >> 1) & 1u;
                if (!await(ptx::smem_u32(s_full + buf), par, abort, a.status, 20 + hf, sc, u)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t s_tm = tmem + lane_base + S_COL + buf * 128 + hf * HK;
                float s[HK];
#pragma unroll
                for (int c = 0; c < HK / 16; ++c) ptx::tmem_ld16(s_tm + c * 16, s + c * 16);
                const int j0 = (b0 + b) * BKV + hf * HK;
                // causal mask only where this block crosses some row's position (warp-uniform test)
                if (j0 + HK - 1 > prow_min) {
#pragma unroll
                    for (int i = 0; i < HK; ++i) s[i] = (j0 + i <= prow) ? s[i] : -INFINITY;
                }
                float mx = s[0];
#pragma unroll
                for (int i = 1; i < HK; ++i) mx = fmaxf(mx, s[i]);
                m_run = fmaxf(m_run, mx * a.scale_log2);      // exp2 domain
                // rescale O_h when the running max outgrew the scale in use by more than 2^8.  The TMEM
                // accesses are warp-collective (.sync.aligned), so when any lane needs it the whole warp
                // rescales, each row by its own factor (rescaling to the current max is always valid).
                // O_h must first hold block sc-1's update: s_free[x] completes once the PV MMAs of the
                // last block on buffer x (and every MMA before them) are done, and block sc's cannot start
                // before this warp writes its P.
                const bool need = m_used != -INFINITY && m_run > m_used + RESCALE_LOG2;
                if (__any_sync(0xffffffffu, need)) {
                    if (b > 0) {
                        const uint32_t pb = sc - 1;
                        if (!await(ptx::smem_u32(s_free + (pb & 1)), (pb >> 1) & 1u, abort, a.status, 35 + hf, pb,
                                   u)) {
                            ok = false;
                            break;
                        }
                    }
                    ptx::tc_fence_after();
                    const float f = (m_used == -INFINITY) ? 1.f : exp2f(m_used - m_run);
#pragma unroll
                    for (int c = 0; c < HD / 16; ++c) {
                        float t[16];
                        ptx::tmem_ld16(o_tm + c * 16, t);
#pragma unroll
                        for (int i = 0; i < 16; ++i) t[i] *= f;
                        ptx::tmem_st16(o_tm + c * 16, t);
                    }
                    ptx::tmem_wait_st();
                    l *= f;
                    m_used = m_run;
                }
                if (m_used == -INFINITY) m_used = m_run;    // nothing accumulated yet (O_h holds zeros)
                // P = 2^(s * scale - m_used) (zero when nothing is visible yet), summed, and written over
                // this half's S columns as bf16: hi in columns 0..31, lo (split precision) in 32..63,
                // two keys per 32-bit column, the lower key in the low half
                const float neg_m = (m_used == -INFINITY) ? -INFINITY : -m_used;
                float sum = 0.f;
#pragma unroll
                for (int i = 0; i < HK; ++i) {
                    s[i] = ex2_approx(fmaf(s[i], a.scale_log2, neg_m));
                    sum += s[i];
                }
                l += sum;
#pragma unroll
                for (int c = 0; c < HK / 32; ++c) {
                    uint32_t w[16], wl[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const float p0 = s[c * 32 + 2 * t], p1 = s[c * 32 + 2 * t + 1];
                        w[t] = pack_bf16x2(p0, p1);
                        if (SPLIT) {
                            const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&w[t]);
                            const float2 back = __bfloat1622float2(hb);
                            wl[t] = pack_bf16x2(p0 - back.x, p1 - back.y);
                        }
                    }
                    tmem_st16_u(s_tm + c * 16, w);
                    if (SPLIT) tmem_st16_u(s_tm + 32 + c * 16, wl);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(p_full + buf));
                ++sc;
            }
            if (!ok) break;
            // the last block's O_h update
            {
                const uint32_t pb = sc - 1;
                if (!await(ptx::smem_u32(s_free + (pb & 1)), (pb >> 1) & 1u, abort, a.status, 40 + hf, pb, u))
                    break;
            }
            ptx::tc_fence_after();
            if (hf == 0) {
                cmb[row * 2] = m_used;
                cmb[row * 2 + 1] = l;
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(cmb_bar));
            } else {
                if (!await(ptx::smem_u32(cmb_bar), unit_cnt & 1u, abort, a.status, 50, unit_cnt, u)) break;
                ptx::tc_fence_after();
                const float m0 = cmb[row * 2], l0 = cmb[row * 2 + 1];
                const float M = fmaxf(m0, m_used);
                const float f0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - M);
                const float f1 = (m_used == -INFINITY) ? 0.f : exp2f(m_used - M);
                const float L = l0 * f0 + l * f1;
                const uint32_t o0 = tmem + lane_base + O_COL, o1 = o0 + HD;
                if (a.parts == 1) {
                    const float inv = 1.0f / L;
                    const int head = g * a.G + row % a.G;
                    const size_t at = (size_t)qi * a.Hq * HD + (size_t)head * HD;
#pragma unroll
                    for (int c = 0; c < HD / 16; ++c) {
                        float x0[16], x1[16];
                        ptx::tmem_ld16(o0 + c * 16, x0);
                        ptx::tmem_ld16(o1 + c * 16, x1);
                        if (valid) {
                            uint4 w[2], wl[2];
                            bf16* h = reinterpret_cast<bf16*>(w);
                            bf16* lo = reinterpret_cast<bf16*>(wl);
#pragma unroll
                            for (int t = 0; t < 16; ++t) split_bf16((x0[t] * f0 + x1[t] * f1) * inv, h[t], lo[t]);
                            *reinterpret_cast<uint4*>(a.out + at + c * 16) = w[0];
                            *reinterpret_cast<uint4*>(a.out + at + c * 16 + 8) = w[1];
                            if (a.out_lo) {
                                *reinterpret_cast<uint4*>(a.out_lo + at + c * 16) = wl[0];
                                *reinterpret_cast<uint4*>(a.out_lo + at + c * 16 + 8) = wl[1];
                            }
                        }
                    }
                } else {
                    // partial result of this key range: O (scaled to max M), M and the sum L
                    float* po = a.part_o + ((size_t)u * ROWS + row) * HD;
#pragma unroll
                    for (int c = 0; c < HD / 16; ++c) {
                        float x0[16], x1[16];
                        ptx::tmem_ld16(o0 + c * 16, x0);
                        ptx::tmem_ld16(o1 + c * 16, x1);
#pragma unroll
                        for (int t = 0; t < 16; t += 4)
                            *reinterpret_cast<float4*>(po + c * 16 + t) =
                                make_float4(x0[t] * f0 + x1[t] * f1, x0[t + 1] * f0 + x1[t + 1] * f1,
                                            x0[t + 2] * f0 + x1[t + 2] * f1, x0[t + 3] * f0 + x1[t + 3] * f1);
                    }
                    *reinterpret_cast<float2*>(a.part_ml + ((size_t)u * ROWS + row) * 2) = make_float2(M, L);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(o_free));
            }
            ++unit_cnt;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// Merge the key-range parts of each (query, head): O = sum_p O_p 2^(M_p - M) / sum_p L_p 2^(M_p - M).
// One warp per (query, head); each lane owns hd/32 consecutive dims.
template <int HD>
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnArgs a) {
    grid_dep_launch();
    grid_dep_wait();
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (wid >= a.M * a.Hq) return;
    const int qi = wid / a.Hq, head = wid % a.Hq;
    const int qt = qi / a.QT, g = head / a.G;
    const int r = (qi % a.QT) * a.G + head % a.G;
    const int nb = tile_blocks(a, qt);
    const int base = ((a.n_qt - 1 - qt) * a.Hkv + g) * a.parts;
    float M = -INFINITY;
    for (int p = 0; p < a.parts && p * a.part_blocks < nb; ++p)
        M = fmaxf(M, a.part_ml[((size_t)(base + p) * ROWS + r) * 2]);
    constexpr int PER = HD / 32;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    float L = 0.f;
    for (int p = 0; p < a.parts && p * a.part_blocks < nb; ++p) {
        const size_t it = (size_t)(base + p) * ROWS + r;
        const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + it * 2);
        const float f = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
        L += ml.y * f;
        const float* po = a.part_o + it * HD + lane * PER;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] += po[i] * f;
    }
    const float inv = 1.0f / L;
    const size_t at = (size_t)qi * a.Hq * HD + (size_t)head * HD + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        bf16 h, lo;
        split_bf16(acc[i] * inv, h, lo);
        a.out[at + i] = h;
        if (a.out_lo) a.out_lo[at + i] = lo;
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
    const size_t np = SPLIT ? 2 : 1;
    return 1024 + np * ROWS * HD * 2 + (size_t)(K_STAGES + V_STAGES) * BKV * HD * 2 + 2 * ROWS * sizeof(float) + 512;
}

template <int HD, bool SPLIT>
cudaError_t launch_hd(const CUtensorMap& mq, const CUtensorMap& mql, const CUtensorMap& mkv, const AttnArgs& a,
                      int grid, cudaStream_t s, bool pdl) {
    static std::atomic<uint64_t> done{0};
    const size_t sm = attn_smem<HD, SPLIT>();
    const cudaError_t e = smem_limit_once(attn_tc_kernel<HD, SPLIT>, (int)sm, done);
    if (e != cudaSuccess) return e;
    return launch_ex(pdl, attn_tc_kernel<HD, SPLIT>, dim3(grid), dim3(NUM_THREADS), sm, s, mq, mql, mkv, a);
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
                                const int* qpos, int M, int n_keys, void* out, void* out_lo, cudaStream_t s,
                                int* launches) {
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
    // too few (query tile, KV head) units to fill the GPU: cut each key range into parts, merged by
    // attn_combine_kernel, so the longest chain of key blocks shrinks
    a.parts = 1;
    const int nb_max = (n_keys + BKV - 1) / BKV;
    a.part_blocks = nb_max;
    int per_sm = 2;                              // work items aimed at per SM (measured best with run-time claiming)
    if (const char* v = getenv("CB_TUNE_ATTN_ITEMS")) per_sm = std::max(1, atoi(v));
    if (m.part_o && a.units < 2 * m.num_sms && nb_max > 4) {
        int parts = (per_sm * m.num_sms + a.units - 1) / a.units;
        while (parts > 1 && (size_t)a.units * parts > (size_t)m.part_items) --parts;
        if (parts > nb_max) parts = nb_max;
        if (parts > 1) {
            a.part_blocks = (nb_max + parts - 1) / parts;
            a.parts = (nb_max + a.part_blocks - 1) / a.part_blocks;
            a.part_o = m.part_o;
            a.part_ml = m.part_ml;
        }
    }
    a.units *= a.parts;
    a.pos = qpos;
    a.out = reinterpret_cast<bf16*>(out);
    a.out_lo = reinterpret_cast<bf16*>(out_lo);
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)c.head_dim);
    a.idesc_qk = ptx::idesc_bf16(ROWS, BKV);
    a.idesc_pv = ptx::idesc_bf16(ROWS, c.head_dim) | (1u << 16);    // B (V) is MN-major
    a.status = m.status;
    a.sched = m.attn_sched;
    const int grid = a.units < m.num_sms ? a.units : m.num_sms;
    const CUtensorMap& mq = *reinterpret_cast<const CUtensorMap*>(qmap);
    const CUtensorMap& mql = *reinterpret_cast<const CUtensorMap*>(m.split ? qmap_lo : qmap);
    const CUtensorMap& mkv = *reinterpret_cast<const CUtensorMap*>(kvmap);
    cudaError_t e;
    if (c.head_dim == 128)
        e = m.split ? launch_hd<128, true>(mq, mql, mkv, a, grid, s, m.pdl) : launch_hd<128, false>(mq, mql, mkv, a, grid, s, m.pdl);
    else
        e = m.split ? launch_hd<64, true>(mq, mql, mkv, a, grid, s, m.pdl) : launch_hd<64, false>(mq, mql, mkv, a, grid, s, m.pdl);
    if (launches) *launches = 1;
    if (e != cudaSuccess || a.parts == 1) return e;
    const int warps = M * c.n_heads;
    const int blocks = (warps + 7) / 8;
    // programmatic dependent launch: the merge's CTAs take the SMs the attention's tail leaves idle and wait
    // (griddepcontrol.wait) for its partial results
    e = c.head_dim == 128 ? launch_ex(m.pdl, attn_combine_kernel<128>, dim3(blocks), dim3(256), 0, s, a)
                          : launch_ex(m.pdl, attn_combine_kernel<64>, dim3(blocks), dim3(256), 0, s, a);
    if (launches) *launches = 2;
    return e;
}

}  // namespace cb
