// prefill.cu -- paged prefill and chunked-prefill attention on the tcgen05 tensor cores.
//
// What is computed (the pages' definitions):
//   * "理解 KV Cache" (steinslab.io) §1.2: Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k) + M) V
//     with the causal mask M: position i aggregates positions <= i only.  §2.1: prefill
//     processes every prompt position at once, a matrix-matrix product bound by compute,
//     the work tensor cores are made for.
//   * "KV Cache 与推理优化" (note.yj-dis.top): prefill fills every position of the cache;
//     sequences packed into one batch need a per-sequence (block-diagonal) causal mask
//     (pitfalls table); GQA query heads hq = h*g .. h*g+g-1 share KV head h.
//   A batch packs, per sequence b, a chunk of P_b query rows (rows cu_q[b] .. cu_q[b+1]-1 of
//   q) whose K/V are already in the paged cache (kv_append) behind C_b = L_b - P_b earlier
//   positions.  Row cu_q[b] + i is position C_b + i and attends over positions 0 .. C_b + i
//   of its own sequence, gathered through its block table.  C_b = 0 is a whole-prompt
//   prefill; C_b > 0 a chunk of a longer prompt (chunked prefill).
//
// GB300 design:
//   * Work unit = (sequence, KV head, 256 query rows): TP = 256 / g query positions times the
//     g query heads of the KV head, so every K/V tile read serves the whole GQA group and two
//     128-row q-tiles.  Rows r = position * g + head; for g that does not divide 256 the last
//     rows are padding.  Two q-tiles per K/V tile halve the K/V bytes per FLOP: with one,
//     the kernel waited on K/V loads.
//   * A host plan (pkv_prefill_plan) lists the units and assigns them, heaviest first, to
//     the CTAs of a persistent one-wave grid (longest-processing-time first).  The same plan
//     serves every layer of a batch.
//   * One CTA per SM, 15 warps: warps 0, 10 and 11 issue the tiled bulk-tensor (TMA) loads of
//     K, V and Q; warps 1 and 12 issue the tcgen05.mma instructions of S for q-tiles 0 and 1,
//     warps 13 and 14 those of P.V for q-tiles 0 and 1; warps 2-5 run the softmax and
//     epilogue of q-tile 0, warps 6-9 of q-tile 1, one query row per thread.
//   * Per K/V tile of 64 keys (4 paged blocks): S = Q.K^T (M 128, N 64, K D) per q-tile into
//     tensor memory (double-buffered, so the next S is computed while the softmax reads
//     this one); the softmax masks (causal, by select), updates the running max and sum
//     (exp2 domain, rescaling the output accumulator only when the max rises by more than
//     2^8) and writes P as bf16 back into the tensor-memory columns its S came from; O +=
//     P.V (M 128, N D, K 64) reads P from tensor memory and V from shared memory and
//     accumulates in tensor memory.  The S that next overwrites a P waits until that P's
//     P.V is complete.
//   * Feeding the tensor pipe sets the pace: it accepts only a few instructions ahead, a
//     128 x 64 x 16 MMA takes about 36 ns and a 128 x 128 x 16 one about 56 ns, and each
//     satisfied mbarrier wait of the issuing thread costs about 70 ns.  One thread that
//     waited for its inputs between batches left the pipe idle about 40 % of each tile; four
//     issuing threads (S and P.V for each q-tile) overlap one's waits with the others'
//     products.
//   * Keeping P out of shared memory leaves the room for deeper rings and takes P's stores
//     and the tensor core's reads of it off the shared-memory port, and the softmax no
//     longer waits for the previous P.V before writing P (only a rescale of O does).
//   * K and V stream through two separate rings (5 stages each at D = 128).  A K tile is free again once S is
//     computed, a V tile only after P.V: sharing one stage would hold K for a whole tile's
//     pipeline, and with loads of scattered 4 KiB blocks taking microseconds under load, the
//     ring, not the tensor core, would set the pace.  Each 16-token block of one KV head is
//     a contiguous [16, D] tile of the cache, loaded by TMA with a 128-byte swizzle as rows
//     of the [64 keys, D] operand.  V rows past the last key any query of the unit may see
//     are zeroed in shared memory before P.V, so whatever the cache holds there (unused
//     tail slots, NaN included) never meets the tensor core: P is 0 there, but 0 x NaN is
//     not.
//   * All waits are bounded (about 1 s, then PKV_DEVERR_TIMEOUT and a bounded drain).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include "pkv_internal.h"
#include "tc_device.cuh"

namespace pkv {
namespace prefill {

constexpr int BM = 128;            // query rows per q-tile (two q-tiles per unit)
constexpr int BN = 64;             // keys per KV tile (4 blocks)
constexpr int BS = 16;             // tokens per block
constexpr int NTHREADS = 480;      // warp 0 K loads, 1 and 12 S MMAs, 2-9 softmax + epilogue, 10 V, 11 Q loads, 13-14 P.V MMAs
constexpr float FP8_Q_SCALE = 1.0f / 256.0f;   // E4M3 pools: q is taken to f16 as q * 2^-8
constexpr float LOG2E = 1.4426950408889634f;
constexpr float TAU = 8.0f;        // raise the running max only beyond 2^8
constexpr uint32_t PLAN_MAGIC = 0x504b5650u;   // "PVKP"
constexpr uint32_t TMEM_COLS = 512;            // S (and P over it): 2 buffers x 2 q-tiles x 64, O: 2 x D

// A plan: header, per-CTA unit ranges, units.
struct PlanHeader { uint32_t magic; int32_t num_units, grid, group, tp, hq, hkv, pad; };
struct Unit { int32_t b, h, row0, pos0, npos, nkv, kmax, pad; };

__host__ __device__ inline size_t plan_units_offset(int grid)
{
    return (sizeof(PlanHeader) + sizeof(int32_t) * (size_t)(grid + 1) + 31) / 32 * 32;
}

struct Params {
    const int32_t *tables;
    const uint8_t *plan;
    uint16_t *out;
    uint32_t *err;
    int MB, Hq, Hkv, group, TP, num_blocks, grid;
    float score_scale;           // scale * k_scale * log2(e)
    float out_scale;             // v_scale (1 for bf16 pools)
    int test_stall;              // failure-path test: the Q loader waits on a barrier nothing completes
};

template <int D, bool FP8>
struct Smem {
    static constexpr int H = D / 64;                  // 64-column atom columns per row
    // K/V ring depth (what the room allows).  An E4M3 pool streams its tiles through a deeper
    // ring of staging tiles as stored (NSG) and keeps a shallower ring of converted ones.
    static constexpr int NS = FP8 ? (D == 128 ? 3 : 4) : (D == 128 ? 5 : 8);
    static constexpr int NSG = FP8 ? (D == 128 ? 4 : 8) : 0;
    static constexpr int Q = 0;                       // H x [256 rows][64]
    static constexpr int QHALF = BM * 2 * 128;        // bytes of one atom column of Q (256 rows)
    static constexpr int KHALF = BN * 128;            // bytes of one atom column of a K or V tile
    static constexpr int KSTAGE = H * KHALF;          // one K (or V) tile (bf16)
    static constexpr int K = Q + H * QHALF;           // NS K tiles
    static constexpr int V = K + NS * KSTAGE;         // NS V tiles
    // E4M3 pools: NSG staging tiles each for K and V, [64 keys][D bytes] as loaded
    static constexpr int STG = BN * D;
    static constexpr int SK = V + NS * KSTAGE;
    static constexpr int SV = SK + NSG * STG;
    static constexpr int BAR = SV + NSG * STG;        // 14 + 4 NS + 2 NSG mbarriers, then the TMEM slot
    static constexpr int TOTAL = BAR + 512;
    static constexpr int ALLOC = TOTAL + 1024;        // alignment slack
    static_assert(8 * (14 + 4 * NS + 2 * NSG) + 4 <= 512, "barrier area");
    static_assert(ALLOC <= 227 * 1024, "shared memory");
};

template <int D, bool FP8>
__global__ void __launch_bounds__(NTHREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, const Params p)
{
    using L = Smem<D, FP8>;
    constexpr int H = L::H;
    constexpr int NSTAGE = L::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = dev::smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // mbarriers: q_full, q_free (a unit's last S is done with Q); k_full, v_full, k_free
    // [NSTAGE]; s_full [2 q-tiles][2 tile parities]; p_full [2 q-tiles][2 tile parities]
    // (the q-tile's four softmax warps wrote P); o_done [NSTAGE] (both q-tiles' P.V of the
    // stage's tile are complete); o_free [2 q-tiles] (the epilogue has read O).
    // p_full alternates by tile: the softmax does not wait for the previous P.V, so it can
    // finish tile J+1 before the P.V issuer has seen tile J's P, and a single barrier would
    // then run two phases ahead of its waiter.  S(J) waits for o_done of tile J-2, which
    // also covers the softmax's reads of S(J-2): each softmax warp reads its S before it
    // writes P, and P.V(J-2) waits for that P.
    const uint32_t bars = base + L::BAR;
    const uint32_t q_full = bars, q_free = bars + 8;
    auto k_full = [&](int s) { return bars + 8 * (2 + s); };
    auto v_full = [&](int s) { return bars + 8 * (2 + NSTAGE + s); };
    auto k_free = [&](int s) { return bars + 8 * (2 + 2 * NSTAGE + s); };
    auto s_full = [&](int w, int J) { return bars + 8 * (2 + 3 * NSTAGE + 2 * w + (J & 1)); };
    auto p_full = [&](int w, int J) { return bars + 8 * (6 + 3 * NSTAGE + 2 * w + (J & 1)); };
    auto o_done = [&](int s) { return bars + 8 * (10 + 3 * NSTAGE + s); };
    auto o_free = [&](int w) { return bars + 8 * (10 + 4 * NSTAGE + w); };
    const uint32_t never = bars + 8 * (12 + 4 * NSTAGE);     // no thread ever arrives here
    // E4M3 pools: staging tile x of K (or V) landed; a unit's Q rows converted to f16
    constexpr int NSG = L::NSG;
    auto stg_full = [&](bool isk, int x) { return bars + 8 * (13 + 4 * NSTAGE + (isk ? 0 : NSG) + x); };
    const uint32_t q_ready = bars + 8 * (13 + 4 * NSTAGE + 2 * NSG);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::BAR + 8 * (14 + 4 * NSTAGE + 2 * NSG));

    const PlanHeader *hdr = reinterpret_cast<const PlanHeader *>(p.plan);
    const int32_t *cta_off = reinterpret_cast<const int32_t *>(p.plan + sizeof(PlanHeader));
    const Unit *units = reinterpret_cast<const Unit *>(p.plan + plan_units_offset(p.grid));
    if (hdr->magic != PLAN_MAGIC || hdr->grid != p.grid || hdr->group != p.group || hdr->hq != p.Hq ||
        hdr->hkv != p.Hkv || hdr->tp != p.TP) {
        if (tid == 0 && blockIdx.x == 0) dev::flag_error(p.err, PKV_DEVERR_PLAN);
        return;
    }
    const int u0 = cta_off[blockIdx.x], u1 = cta_off[blockIdx.x + 1];

    if (tid == 0) {
        dev::mbar_init(q_full, 1);
        dev::mbar_init(q_free, 2);                    // both S issuers' last S of a unit
        for (int s = 0; s < NSTAGE; ++s) {
            dev::mbar_init(k_full(s), 1);
            dev::mbar_init(v_full(s), 1);
            dev::mbar_init(k_free(s), 2);             // both q-tiles' S of the stage's tile
            dev::mbar_init(o_done(s), 2);             // both q-tiles' P.V of the stage's tile
        }
        for (int b = 0; b < 2; ++b) {
            dev::mbar_init(s_full(b, 0), 1);
            dev::mbar_init(s_full(b, 1), 1);
            dev::mbar_init(p_full(b, 0), 4);          // the q-tile's four softmax warps wrote P
            dev::mbar_init(p_full(b, 1), 4);
            dev::mbar_init(o_free(b), 4);             // the q-tile's four warps read O
        }
        dev::mbar_init(never, 1);
        if constexpr (FP8) {
            for (int x = 0; x < NSG; ++x) {
                dev::mbar_init(stg_full(true, x), 1);
                dev::mbar_init(stg_full(false, x), 1);
            }
            dev::mbar_init(q_ready, 1);
        }
        dev::fence_barrier_init();
    }
    if (warp == 1) tc::tmem_alloc(dev::smem_u32(tmem_slot), TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // tensor memory: S[buffer][q-tile] at columns (2*buffer + q-tile)*64, O[q-tile] at 256 + q-tile*D
    auto tS = [&](int b, int w) { return tmem + (uint32_t)((2 * b + w) * BN); };
    auto tO = [&](int w) { return tmem + 256u + (uint32_t)(w * D); };

    // Block-table entries of K/V tile j of a unit, fetched a tile ahead of their use so that
    // the table's load latency stays off the producers' path (INT_MIN: past the unit's last
    // needed block).  resolve() checks them: -1 for a block not loaded, which an entry
    // outside the pool also flags.
    auto fetch_ids = [&](const Unit &un, int j, int (&raw)[BN / BS]) {
        const int nblk = un.kmax / BS + 1;                   // blocks holding keys 0..kmax
#pragma unroll
        for (int i = 0; i < BN / BS; ++i) {
            const int blk = j * (BN / BS) + i;
            raw[i] = (blk < nblk && blk < p.MB) ? __ldg(p.tables + (size_t)un.b * p.MB + blk) : INT_MIN;
        }
    };
    auto resolve = [&](int id) {
        if (id == INT_MIN) return -1;
        if (id < 0 || id >= p.num_blocks) {
            dev::flag_error(p.err, PKV_DEVERR_BLOCK_ID);
            return -1;
        }
        return id;
    };

    // E4M3 pools: the loader warp of K (warp 0) or V (warp 10), every lane.  Lane 0 walks the
    // CTA's tiles as the bf16 loaders do and copies each tile's blocks, as stored ([16 keys][D
    // bytes] each), into staging tile t % NSG, up to NSG tiles ahead.  Every lane converts
    // tile J into ring stage J % NS as f16, in the 128-byte-swizzled layout that a bulk-tensor
    // copy would have written (16-byte chunk c of row r at chunk c ^ (r % 8)); E4M3 -> f16 is
    // exact.  The products then run in f16 (q is taken to f16 as q * 2^-8 and P is written as
    // f16), and the pool's scales are applied outside: k_scale (and 2^8) in the score scale,
    // v_scale in the epilogue.
    auto load_fp8 = [&](bool isk) {
        const CUtensorMap *map = isk ? &kmap : &vmap;
        const uint32_t stg_base = base + (isk ? L::SK : L::SV);
        const uint8_t *stg = sm + (isk ? L::SK : L::SV);
        uint8_t *ring = sm + (isk ? L::K : L::V);
        int nt = 0;                                  // the CTA's tiles
        for (int u = u0; u < u1; ++u) nt += units[u].nkv;
        // lane 0: the issue cursor (tile ti of unit un, tile jc within it) and the entries of
        // tile ti, fetched one issue ahead; the loaded-block masks of the tiles in flight, 4
        // bits each (tile t at bits 4 (t % 8))
        int ti = 0, uc = u0, jc = 0;
        Unit un = units[u0];
        int raw[BN / BS];
        unsigned masks = 0;
        if (lane == 0) fetch_ids(un, 0, raw);
        auto issue_next = [&]() {
            int ids[BN / BS], n = 0;
            unsigned m = 0;
#pragma unroll
            for (int i = 0; i < BN / BS; ++i) {
                ids[i] = resolve(raw[i]);
                if (ids[i] >= 0) {
                    m |= 1u << i;
                    ++n;
                }
            }
            const int x = ti % NSG;
            const uint32_t bar = stg_full(isk, x);
            dev::mbar_arrive_expect_tx(bar, (uint32_t)(n * BS * D));
#pragma unroll
            for (int i = 0; i < BN / BS; ++i)
                if (ids[i] >= 0)
                    tc::tma_load_3d(stg_base + x * L::STG + i * BS * D, map, 0, 0, ids[i] * p.Hkv + un.h, bar);
            masks = (masks & ~(0xFu << (4 * (ti % 8)))) | (m << (4 * (ti % 8)));
            ++ti;
            if (++jc == un.nkv) {
                jc = 0;
                if (++uc < u1) un = units[uc];
            }
            if (ti < nt) fetch_ids(un, jc, raw);
        };
        if (lane == 0)
            while (ti < nt && ti < NSG) issue_next();
        // lane: 8-byte piece cc of the tile row (bytes 8cc .. 8cc + 7, the output's atom column
        // cc / 8 and 16-byte chunk cc % 8), rows rr, rr + RP, ...: each pass reads RP whole
        // contiguous rows
        constexpr int LPR = D / 8, RP = 32 / LPR;    // lanes per row, rows per pass
        const int cc = lane % LPR, rr = lane / LPR, hf = cc / 8, c = cc % 8;
        bool ok = true;
        int J = 0;                                   // tiles converted
        for (; J < nt; ++J) {
            // tile J: its staging copy, then its ring stage free (S of the stage's previous
            // tile done for K, its P.V for V)
            const int st = J % NSTAGE;
            bool okw = dev::mbar_wait_bounded(stg_full(isk, J % NSG), (uint32_t)((J / NSG) & 1));
            if (okw && J >= NSTAGE) {
                const uint32_t par = ((J - NSTAGE) / NSTAGE) & 1;
                okw = isk ? dev::mbar_wait_bounded(k_free(st), par) : dev::mbar_wait_bounded(o_done(st), par);
            }
            if (!__all_sync(dev::FULL, okw)) {
                ok = false;
                break;
            }
            const unsigned mask = (__shfl_sync(dev::FULL, masks, 0) >> (4 * (J % 8))) & 0xFu;
            const uint8_t *src = stg + (J % NSG) * L::STG;
            uint8_t *dst = ring + st * L::KSTAGE + hf * L::KHALF;
            for (int i = 0; i < BN / BS; ++i) {
                if (!((mask >> i) & 1u)) continue;           // not loaded (uniform over the warp)
#pragma unroll
                for (int p0 = 0; p0 < BS / RP; p0 += 4) {
                    uint2 e[4];                              // four passes' loads in flight
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        e[k] = *reinterpret_cast<const uint2 *>(src + (i * BS + (p0 + k) * RP + rr) * D + cc * 8);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int r = i * BS + (p0 + k) * RP + rr;
                        *reinterpret_cast<uint4 *>(dst + r * 128 + ((c ^ (r & 7)) << 4)) =
                            make_uint4(dev::e4m3x2_to_f16x2((uint16_t)e[k].x),
                                       dev::e4m3x2_to_f16x2((uint16_t)(e[k].x >> 16)),
                                       dev::e4m3x2_to_f16x2((uint16_t)e[k].y),
                                       dev::e4m3x2_to_f16x2((uint16_t)(e[k].y >> 16)));
                    }
                }
            }
            dev::fence_proxy_async_smem();           // converted rows -> tensor core (and the
            __syncwarp();                            // staging tile's reads before its refill)
            if (lane == 0) {
                dev::mbar_arrive(isk ? k_full(st) : v_full(st));
                if (ti < nt) issue_next();           // into the staging tile just converted
            }
        }
        if (lane == 0) {
            if (!ok) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
            // no copy may land after the CTA has left: wait (bounded) for the staging copies
            // issued but not converted
            for (int t = J; t < ti; ++t)
                (void)dev::mbar_wait_bounded(stg_full(isk, t % NSG), (uint32_t)((t / NSG) & 1));
        }
    };

    if (FP8 && warp == 11) {
        // ============ Q for E4M3 pools: every lane.  Lane 0 loads a unit's rows as below; every
        // lane then takes them to f16 in place, as q * 2^-8 (so that queries up to 2^24 in
        // magnitude fit, saturating beyond), and lane 0 marks them ready for the S issuers.
        int uq = 0;
        bool pending = false;                        // lane 0: a Q copy not yet waited for
        int okl = !p.test_stall || lane != 0 || dev::mbar_wait_bounded_ns(never, 0, dev::TEST_EXPIRE_NS);
        bool ok = __shfl_sync(dev::FULL, okl, 0);
        for (int u = u0; u < u1 && ok; ++u, ++uq) {
            const Unit un = units[u];
            okl = 1;
            if (lane == 0) {
                if (uq > 0 && !dev::mbar_wait_bounded(q_free, (uq - 1) & 1)) {
                    okl = 0;
                } else {
                    dev::mbar_arrive_expect_tx(q_full, (uint32_t)(H * 64 * p.group * p.TP * 2));
                    for (int hf = 0; hf < H; ++hf)
                        tc::tma_load_3d(base + L::Q + hf * L::QHALF, &qmap, hf * 64, un.h * p.group, un.row0, q_full);
                    pending = true;
                }
            }
            if (!__shfl_sync(dev::FULL, okl, 0) ||
                !__all_sync(dev::FULL, dev::mbar_wait_bounded(q_full, (uint32_t)(uq & 1)))) {
                ok = false;
                break;
            }
            pending = false;
            uint4 *qs = reinterpret_cast<uint4 *>(sm + L::Q);
            for (int e = lane; e < H * L::QHALF / 16; e += 32) {
                uint4 v = qs[e];
                uint32_t *w4 = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    w4[t] = dev::pack_f16x2_satfinite(dev::bf16_lo(w4[t]) * FP8_Q_SCALE, dev::bf16_hi(w4[t]) * FP8_Q_SCALE);
                qs[e] = v;
            }
            dev::fence_proxy_async_smem();           // converted rows -> tensor core
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(q_ready);
        }
        if (lane == 0) {
            if (!ok) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
            // no copy may land after the CTA has left
            if (pending) (void)dev::mbar_wait_bounded(q_full, (uint32_t)((uq) & 1));
        }
    } else if (warp == 11) {
        // ============ TMA producer of Q: a unit's rows once the previous unit's last S is done
        if (lane == 0) {
            int uq = 0;
            // the failure-path test: a wait that runs out before the first load (nothing in flight)
            bool ok = !p.test_stall || dev::mbar_wait_bounded_ns(never, 0, dev::TEST_EXPIRE_NS);
            for (int u = u0; u < u1 && ok; ++u, ++uq) {
                const Unit un = units[u];
                if (uq > 0 && !dev::mbar_wait_bounded(q_free, (uq - 1) & 1)) {
                    ok = false;
                    break;
                }
                dev::mbar_arrive_expect_tx(q_full, (uint32_t)(H * 64 * p.group * p.TP * 2));
                for (int hf = 0; hf < H; ++hf)
                    tc::tma_load_3d(base + L::Q + hf * L::QHALF, &qmap, hf * 64, un.h * p.group, un.row0, q_full);
            }
            if (!ok) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
            // no copy may land after the CTA has left: wait (bounded) for the last one
            if (uq > 0) (void)dev::mbar_wait_bounded(q_full, (uq - 1) & 1);
        }
    } else if (warp == 0 || warp == 10) {
        // ============ TMA producers: warp 0 loads K, warp 10 loads V ============
        // The two rings are separate because K is free again once S is computed, while V
        // is needed until P.V: a K stage is held for about a load plus S, not for a whole
        // tile's pipeline.  Q has a producer of its own so that the K ring runs ahead into
        // the next unit while the current one finishes.
        if (FP8 && u0 < u1) {
            load_fp8(warp == 0);
        } else if (!FP8 && lane == 0 && u0 < u1) {
            const bool isk = warp == 0;
            const CUtensorMap *map = isk ? &kmap : &vmap;
            int J = 0, arms[NSTAGE] = {};
            bool ok = true;
            // cursor (u, j) over this CTA's tiles; the next tile's entries are in flight while
            // the current one waits for its stage
            int u = u0, j = 0;
            Unit un = units[u];
            int raw[BN / BS];
            fetch_ids(un, 0, raw);
            while (ok) {
                int un_idx = u, jn = j + 1;
                Unit nx = un;
                if (jn == un.nkv) {
                    ++un_idx;
                    jn = 0;
                    if (un_idx < u1) nx = units[un_idx];
                }
                int rawn[BN / BS];
                if (un_idx < u1) fetch_ids(nx, jn, rawn);
                const int s = J % NSTAGE;
                if (J >= NSTAGE) {            // the stage's previous tile: S done (K), P.V done (V)
                    const uint32_t par = ((J - NSTAGE) / NSTAGE) & 1;
                    ok = isk ? dev::mbar_wait_bounded(k_free(s), par) : dev::mbar_wait_bounded(o_done(s), par);
                    if (!ok) break;
                }
                int ids[BN / BS], n = 0;
#pragma unroll
                for (int i = 0; i < BN / BS; ++i) {
                    ids[i] = resolve(raw[i]);
                    n += ids[i] >= 0;
                }
                const uint32_t full = isk ? k_full(s) : v_full(s);
                const uint32_t dst = base + (isk ? L::K : L::V) + s * L::KSTAGE;
                dev::mbar_arrive_expect_tx(full, (uint32_t)(n * H * BS * 128));
                ++arms[s];
#pragma unroll
                for (int i = 0; i < BN / BS; ++i) {
                    if (ids[i] < 0) continue;
                    const int z = ids[i] * p.Hkv + un.h;
                    for (int hf = 0; hf < H; ++hf)
                        tc::tma_load_3d(dst + hf * L::KHALF + i * BS * 128, map, hf * 64, 0, z, full);
                }
                ++J;
                if (un_idx >= u1) break;
                u = un_idx;
                j = jn;
                un = nx;
#pragma unroll
                for (int i = 0; i < BN / BS; ++i) raw[i] = rawn[i];
            }
            if (!ok) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
            // no copy may land after the CTA has left: wait (bounded) for the last of each
            for (int s = 0; s < NSTAGE; ++s)
                if (arms[s]) (void)dev::mbar_wait_bounded(isk ? k_full(s) : v_full(s), (arms[s] - 1) & 1);
        }
    } else if (warp == 1 || warp >= 12) {
        // ============ MMA issuers: per q-tile w, one thread issues S and one P.V ============
        // Warps 1 and 12 issue S of q-tiles 0 and 1, warps 13 and 14 their P.V.  One thread
        // issues a tcgen05.mma only about every 36 ns whatever its shape, longer than the pipe
        // needs for a 128 x 64 x 16 product, so four threads share the issue.  The S of tile J
        // overwrites the tensor memory that P(J-2) was read from, so it waits for the P.V of
        // tile J-2 to be complete.  Every wait is on work issued before it (no cycle); about
        // 1 s without progress ends the launch.
        if (lane == 0) {
            const bool is_s = warp == 1 || warp == 12;
            const int w = (warp == 1 || warp == 13) ? 0 : 1;
            int J = 0, uq = 0;
            bool ok = true;
            auto wait = [&](uint32_t bar, uint32_t par) {
                if (ok && !dev::mbar_wait_bounded(bar, par)) ok = false;
                return ok;
            };
            if (is_s) {
                // S = Q K^T: M 128, N 64 keys (f16 operands for E4M3 pools)
                constexpr uint32_t IDS = FP8 ? tc::idesc_f16(BM, BN, 0) : tc::idesc_bf16(BM, BN, 0);
                // The operand descriptors are built once; each MMA adds its offset.
                const uint64_t dQ = tc::desc_add(tc::smem_desc_sw128(base + L::Q, 16, 1024), (uint32_t)w * 16384);
                const uint64_t dK = tc::smem_desc_sw128(base + L::K, 16, 1024);
                for (int u = u0; u < u1 && ok; ++u, ++uq) {
                    const Unit un = units[u];
                    if (!wait(FP8 ? q_ready : q_full, uq & 1)) break;
                    for (int j = 0; j < un.nkv; ++j, ++J) {
                        const int st = J % NSTAGE;
                        if (!wait(k_full(st), (J / NSTAGE) & 1)) break;
                        // P.V(J-2) has read P(J-2), so the softmax is done with S(J-2) as well
                        if (J >= 2 && !wait(o_done((J - 2) % NSTAGE), ((J - 2) / NSTAGE) & 1)) break;
                        tc::fence_after_sync();
                        const uint64_t dk = tc::desc_add(dK, (uint32_t)st * L::KSTAGE);
                        const uint32_t ts = tS(J & 1, w);
#pragma unroll
                        for (int k = 0; k < 4 * H; ++k) {
                            const uint32_t hf = k >> 2, kk = (k & 3) * 32;
                            tc::mma_bf16(ts, tc::desc_add(dQ, hf * L::QHALF + kk), tc::desc_add(dk, hf * L::KHALF + kk),
                                         IDS, k > 0);
                        }
                        tc::commit(s_full(w, J));
                        tc::commit(k_free(st));                      // (both q-tiles) the K tile may be reloaded
                        if (j == un.nkv - 1) tc::commit(q_free);     // (both q-tiles) the unit is done with Q
                    }
                }
            } else {
                // O += P V: M 128, N D, V MN-major
                constexpr uint32_t IDO = FP8 ? tc::idesc_f16(BM, D, 1) : tc::idesc_bf16(BM, D, 1);
                const uint64_t dV = tc::smem_desc_sw128(base + L::V, L::KHALF, 1024);
                const uint32_t to = tO(w);
                for (int u = u0; u < u1 && ok; ++u, ++uq) {
                    const Unit un = units[u];
                    for (int j = 0; j < un.nkv; ++j, ++J) {
                        const int st = J % NSTAGE;
                        if (!wait(v_full(st), (J / NSTAGE) & 1) || !wait(p_full(w, J), (J >> 1) & 1)) break;
                        // first in a unit: the q-tile's previous output has been read
                        if (j == 0 && uq > 0 && !wait(o_free(w), (uq - 1) & 1)) break;
                        tc::fence_after_sync();
                        const uint64_t dv = tc::desc_add(dV, (uint32_t)st * L::KSTAGE);
                        const uint32_t tp = tS(J & 1, w);
#pragma unroll
                        for (int k = 0; k < BN / 16; ++k)
                            tc::mma_bf16_ts(to, tp + (uint32_t)(k * 8), tc::desc_add(dv, k * 16 * 128), IDO, j > 0 || k > 0);
                        tc::commit(o_done(st));                      // (both q-tiles)
                    }
                }
            }
            if (!ok) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
        }
    } else {
        // ============================ softmax + epilogue ============================
        // Warps 2-5 handle q-tile 0 (rows 0-127 of the unit), warps 6-9 q-tile 1 (rows
        // 128-255).  Warp w % 4 owns tensor-memory lane quarter w % 4: one row per thread,
        // all 64 keys of every tile, all D output columns.
        const int w = (warp - 2) >> 2;
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;                      // row within the q-tile
        const int rg = w * BM + r;                         // row within the unit
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const int st = (tid - 64) & 127;                   // 0..127 within the group
        int J = 0;
        bool ok = true;
        for (int u = u0; u < u1 && ok; ++u) {
            const Unit un = units[u];
            const int pl = rg / p.group, hh = rg - pl * p.group;
            const bool valid = rg < p.TP * p.group && pl < un.npos;
            const int qpos = un.pos0 + pl;                 // keys 0..qpos are visible
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < un.nkv; ++j, ++J) {
                ok = __all_sync(dev::FULL, dev::mbar_wait_bounded(s_full(w, J), (J >> 1) & 1));
                if (!ok) break;
                tc::fence_after_sync();
                float x[BN];
                {
                    uint32_t v0[32], v1[32];
                    tc::tmem_ld32(tS(J & 1, w) + lane_off, v0);
                    tc::tmem_ld32(tS(J & 1, w) + lane_off + 32, v1);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        x[i] = __uint_as_float(v0[i]);
                        x[32 + i] = __uint_as_float(v1[i]);
                    }
                }
                const int kb = j * BN;
                if (kb + BN - 1 > un.pos0) {                  // the causal diagonal crosses the tile
#pragma unroll
                    for (int c = 0; c < BN; ++c) x[c] = (valid && kb + c <= qpos) ? x[c] : -INFINITY;
                }
                float mx4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
                for (int c = 4; c < BN; c += 8)
#pragma unroll
                    for (int t = 0; t < 4; ++t) mx4[t] = tc::fmax3(mx4[t], x[c + t], x[c + 4 + t]);
                const float mx = tc::fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3])) * p.score_scale;   // scale > 0: max commutes
                const bool raise = mx > m + TAU;
                const bool rescale = raise && m != -INFINITY;
                const float f = rescale ? dev::fast_exp2(m - mx) : 1.f;
                if (raise) m = mx;
                // P = exp2(x * scale - m) as packed bf16 (the lower key in the low half)
                const float nm = m == -INFINITY ? 0.f : -m;
                // (packed pairs: one fma and one add per two keys)
                uint32_t pw[BN / 2];
                const float2 sc2 = make_float2(p.score_scale, p.score_scale), nm2 = make_float2(nm, nm);
                float2 ps[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int e = 0; e < BN / 2; ++e) {
                    const float2 t = tc::ffma2(make_float2(x[2 * e], x[2 * e + 1]), sc2, nm2);
                    const float2 pe = make_float2(dev::fast_exp2(t.x), dev::fast_exp2(t.y));
                    ps[e & 1] = tc::fadd2(ps[e & 1], pe);
                    pw[e] = FP8 ? dev::pack_f16x2(pe.x, pe.y) : dev::pack_bf16x2(pe.x, pe.y);
                }
                const float2 ps2 = tc::fadd2(ps[0], ps[1]);
                l = l * f + (ps2.x + ps2.y);
                // P over this tile's S columns (already read): the A operand of this tile's
                // P.V.  No wait: the previous P.V reads the other S buffer.
                tc::tmem_st32(tS(J & 1, w) + lane_off, pw);
                if (__any_sync(dev::FULL, rescale)) {
                    // O may be rescaled only once the previous P.V has accumulated into it
                    ok = __all_sync(dev::FULL, dev::mbar_wait_bounded(o_done((J - 1) % NSTAGE), ((J - 1) / NSTAGE) & 1));
                    if (!ok) break;
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        tc::tmem_ld32(tO(w) + lane_off + 32 * c, v);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * f);
                        tc::tmem_st32(tO(w) + lane_off + 32 * c, v);
                    }
                }
                tc::tmem_wait_st();
                // last tile: zero the V rows past the unit's last visible key (both groups do,
                // each before its own P.V; the stores write the same zeros)
                if (j == un.nkv - 1) {
                    const int first = un.kmax + 1 - kb;
                    if (first < BN) {
                        ok = __all_sync(dev::FULL, dev::mbar_wait_bounded(v_full(J % NSTAGE), (J / NSTAGE) & 1));
                        if (!ok) break;
                        uint8_t *vst = sm + L::V + (J % NSTAGE) * L::KSTAGE;
                        const int chunks = (BN - first) * 8;      // 16-byte chunks per atom column
                        for (int hf = 0; hf < H; ++hf)
                            for (int c = st; c < chunks; c += 128)
                                *reinterpret_cast<uint4 *>(vst + hf * L::KHALF + first * 128 + c * 16) =
                                    make_uint4(0, 0, 0, 0);
                        dev::fence_proxy_async_smem();           // zeroed rows -> tensor core
                    }
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(p_full(w, J));
            }
            if (!ok) break;
            // epilogue: O / l of this row, bf16, to out[row0 + pl][h*g + hh]
            ok = __all_sync(dev::FULL, dev::mbar_wait_bounded(o_done((J - 1) % NSTAGE), ((J - 1) / NSTAGE) & 1));
            if (!ok) break;
            tc::fence_after_sync();
            const float inv = l > 0.f ? p.out_scale / l : 0.f;
            uint16_t *dst = p.out + ((size_t)(un.row0 + pl) * p.Hq + (size_t)un.h * p.group + hh) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tc::tmem_ld32(tO(w) + lane_off + 32 * c, v);
                tc::tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint32_t o4[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            o4[t] = dev::pack_bf16x2(__uint_as_float(v[8 * e + 2 * t]) * inv,
                                                     __uint_as_float(v[8 * e + 2 * t + 1]) * inv);
                        *reinterpret_cast<uint4 *>(dst + 32 * c + 8 * e) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(o_free(w));
        }
        if (!ok && lane == 0) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------------------------
// Host side.
// ------------------------------------------------------------------------------------
bool encode_3d(CUtensorMap *map, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
               uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2)
{
    return encode_tiled_3d(map, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, {d0, d1, d2}, {s1, s2}, {b0, b1, b2},
                           CU_TENSOR_MAP_SWIZZLE_128B);
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

template <int D, bool FP8>
cudaError_t launch(const CUtensorMap &qm, const CUtensorMap &km, const CUtensorMap &vm, const Params &p,
                   cudaStream_t s)
{
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(prefill_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Smem<D, FP8>::ALLOC);
    });
    if (attr != cudaSuccess) return attr;
    prefill_kernel<D, FP8><<<p.grid, NTHREADS, Smem<D, FP8>::ALLOC, s>>>(qm, km, vm, p);
    return cudaGetLastError();
}

int tile_positions(int group) { return 2 * BM / group; }

}  // namespace prefill
}  // namespace pkv

extern "C" size_t pkv_prefill_plan_bytes(const pkv_pool *pool, int32_t batch, int32_t num_q_heads,
                                         int32_t total_q)
{
    using namespace pkv::prefill;
    if (!pool || batch < 1 || num_q_heads < 1 || total_q < 0 || num_q_heads % pool->desc.num_kv_heads) return 0;
    const int g = num_q_heads / pool->desc.num_kv_heads;
    if (g > 16) return 0;
    const int tp = tile_positions(g);
    const size_t units = (size_t)pool->desc.num_kv_heads * ((size_t)total_q / tp + batch);
    const int grid = std::max(1, sm_count());
    return plan_units_offset(grid) + units * sizeof(Unit);
}

extern "C" int pkv_prefill_plan(const pkv_pool *pool, const int32_t *cu_q, const int32_t *seq_lens,
                                int32_t batch, int32_t num_q_heads, int32_t max_blocks, void *plan_out,
                                size_t plan_bytes, int32_t *grid_out)
{
    using namespace pkv::prefill;
    if (!pool || !cu_q || !seq_lens || !plan_out || !grid_out || batch < 1 || num_q_heads < 1 || max_blocks < 1)
        return PKV_ERR_INVALID;
    const int Hkv = pool->desc.num_kv_heads;
    if (num_q_heads % Hkv) return PKV_ERR_INVALID;
    const int g = num_q_heads / Hkv;
    if (g > 16) return PKV_ERR_INVALID;
    const int tp = tile_positions(g);
    if (cu_q[0] != 0) return PKV_ERR_INVALID;
    std::vector<Unit> units;
    for (int b = 0; b < batch; ++b) {
        const int64_t P = (int64_t)cu_q[b + 1] - cu_q[b], L = seq_lens[b];
        if (P < 0 || L < P || L < 1 || (L + BS - 1) / BS > max_blocks) return PKV_ERR_INVALID;
        const int64_t C = L - P;
        for (int64_t qt = 0; qt * tp < P; ++qt) {
            Unit u;
            u.b = b;
            u.row0 = (int32_t)(cu_q[b] + qt * tp);
            u.pos0 = (int32_t)(C + qt * tp);
            u.npos = (int32_t)std::min<int64_t>(tp, P - qt * tp);
            u.kmax = u.pos0 + u.npos - 1;
            u.nkv = u.kmax / BN + 1;
            u.pad = 0;
            for (int h = 0; h < Hkv; ++h) {
                u.h = h;
                units.push_back(u);
            }
        }
    }
    const int sms = sm_count();
    if (sms < 1) return PKV_ERR_CUDA;
    const int grid = std::max(1, std::min<int>(sms, (int)units.size()));
    const size_t need = plan_units_offset(grid) + units.size() * sizeof(Unit);
    if (need > plan_bytes) return PKV_ERR_INVALID;
    // A unit costs its K/V tiles plus about three tile-times of its own: waiting for its Q
    // rows, the S -> softmax -> P.V chain filling and draining, and writing its output
    // (per-CTA end times fit 2.5 to 4 tiles per unit).
    auto cost = [&](int i) { return (int64_t)units[(size_t)i].nkv + 3; };
    // Longest processing time first: heaviest unit to the least-loaded CTA.  The units of one
    // (sequence, KV head) read the same K/V; when the K/V of the batch is larger than about
    // half the L2, they are handed out together (groups heaviest first, heaviest unit first
    // within a group), so that they run side by side on different CTAs and all but the first
    // read of each tile hit L2.  Otherwise every unit is ranked on its own.
    int l2 = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
        return PKV_ERR_CUDA;
    std::vector<int64_t> group_kv((size_t)batch * Hkv, 0);      // largest key count of a group's units
    for (const Unit &u : units) {
        int64_t &gk = group_kv[(size_t)u.b * Hkv + u.h];
        gk = std::max<int64_t>(gk, (int64_t)u.kmax + 1);
    }
    int64_t kv_bytes = 0;
    for (int64_t k : group_kv) kv_bytes += k * pool->desc.head_dim * 2 * 2;
    const bool grouped = kv_bytes > (int64_t)l2 / 2;
    std::vector<int> order(units.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = (int)i;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        const Unit &x = units[(size_t)a], &y = units[(size_t)b];
        if (grouped) {
            const size_t gx = (size_t)x.b * Hkv + x.h, gy = (size_t)y.b * Hkv + y.h;
            if (group_kv[gx] != group_kv[gy]) return group_kv[gx] > group_kv[gy];
            if (gx != gy) return gx < gy;
        }
        return x.nkv > y.nkv;
    });
    std::vector<int> rank(units.size());                      // position in the hand-out order
    for (size_t i = 0; i < order.size(); ++i) rank[(size_t)order[i]] = (int)i;
    using Load = std::pair<int64_t, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int c = 0; c < grid; ++c) heap.push({0, c});
    std::vector<std::vector<int>> per(grid);
    std::vector<int64_t> load(grid, 0);
    for (int i : order) {
        Load top = heap.top();
        heap.pop();
        per[(size_t)top.second].push_back(i);
        top.first += cost(i);
        load[(size_t)top.second] = top.first;
        heap.push(top);
    }
    // Then move a unit, or swap two, between the most and the least loaded CTA while that
    // lowers the larger of their two loads (each step lowers the multiset of loads, so it
    // ends).  With many units per CTA the greedy pass is already fine-grained: swaps are
    // searched only up to 64 units per CTA, which bounds the host time.
    const bool swaps = units.size() <= (size_t)64 * grid;
    for (int it = 0; it < (grouped ? 0 : 16 * grid); ++it) {
        const int ca = (int)(std::max_element(load.begin(), load.end()) - load.begin());
        const int cb = (int)(std::min_element(load.begin(), load.end()) - load.begin());
        const int64_t la = load[(size_t)ca], lb = load[(size_t)cb];
        int64_t best = la;
        int bi = -1, bj = -1;                                   // unit of ca, unit of cb (-1: none)
        for (size_t x = 0; x < per[(size_t)ca].size(); ++x) {
            const int i = per[(size_t)ca][x];
            const int64_t d = cost(i);
            if (std::max(la - d, lb + d) < best) { best = std::max(la - d, lb + d); bi = (int)x; bj = -1; }
            for (size_t y = 0; swaps && y < per[(size_t)cb].size(); ++y) {
                const int64_t e2 = d - cost(per[(size_t)cb][y]);
                if (e2 > 0 && std::max(la - e2, lb + e2) < best) { best = std::max(la - e2, lb + e2); bi = (int)x; bj = (int)y; }
            }
        }
        if (bi < 0) break;
        const int i = per[(size_t)ca][(size_t)bi];
        per[(size_t)ca].erase(per[(size_t)ca].begin() + bi);
        load[(size_t)ca] -= cost(i);
        load[(size_t)cb] += cost(i);
        if (bj >= 0) {
            const int j = per[(size_t)cb][(size_t)bj];
            per[(size_t)cb].erase(per[(size_t)cb].begin() + bj);
            per[(size_t)ca].push_back(j);
            load[(size_t)cb] -= cost(j);
            load[(size_t)ca] += cost(j);
        }
        per[(size_t)cb].push_back(i);
    }
    // within a CTA, the hand-out order: the units of one round run at about the same time on
    // every CTA (a unit the refinement moved keeps its place in that order)
    for (auto &v : per)
        std::sort(v.begin(), v.end(), [&](int a, int b) { return rank[(size_t)a] < rank[(size_t)b]; });
    uint8_t *out = static_cast<uint8_t *>(plan_out);
    PlanHeader hdr{PLAN_MAGIC, (int32_t)units.size(), grid, g, tp, num_q_heads, Hkv, 0};
    std::memcpy(out, &hdr, sizeof(hdr));
    int32_t *off = reinterpret_cast<int32_t *>(out + sizeof(PlanHeader));
    Unit *dst = reinterpret_cast<Unit *>(out + plan_units_offset(grid));
    int32_t n = 0;
    for (int c = 0; c < grid; ++c) {
        off[c] = n;
        for (int i : per[(size_t)c]) dst[n++] = units[(size_t)i];
    }
    off[grid] = n;
    *grid_out = grid;
    return PKV_OK;
}

extern "C" int pkv_paged_prefill(pkv_pool *pool, const void *q, const void *key_cache, const void *value_cache,
                                 const int32_t *block_tables, int32_t batch, int32_t num_q_heads,
                                 int32_t max_blocks, int32_t total_q, float scale, const void *plan,
                                 int32_t grid, void *out, void *stream)
{
    using namespace pkv::prefill;
    int st = pkv::check_attached(pool);
    if (st != PKV_OK) return st;
    const pkv_pool_desc &d = pool->desc;
    if (batch < 1 || num_q_heads < 1 || max_blocks < 1 || total_q < 0 || grid < 1 || !std::isfinite(scale))
        return PKV_ERR_INVALID;
    if (total_q == 0) return PKV_OK;
    if (!q || !key_cache || !value_cache || !block_tables || !plan || !out) return PKV_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(key_cache) & 15u) ||
        (reinterpret_cast<uintptr_t>(value_cache) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u) ||
        (reinterpret_cast<uintptr_t>(plan) & 31u))
        return PKV_ERR_INVALID;
    if (num_q_heads % d.num_kv_heads) return PKV_ERR_INVALID;
    const int g = num_q_heads / d.num_kv_heads;
    if (g > 16) return PKV_ERR_INVALID;
    const int tp = tile_positions(g);
    const int D = d.head_dim;
    const bool fp8 = d.kv_dtype == PKV_KV_FP8E4M3;
    CUtensorMap qm, km, vm;
    const uint64_t rows = (uint64_t)d.num_blocks * d.num_kv_heads;
    if (!encode_3d(&qm, q, D, num_q_heads, total_q, (uint64_t)D * 2, (uint64_t)num_q_heads * D * 2, 64, g, tp))
        return PKV_ERR_CUDA;
    if (fp8) {
        // E4M3 blocks as stored: [16 keys][D bytes] each, copied whole into the staging tiles
        const uint64_t dims[3] = {(uint64_t)D, BS, rows}, strides[2] = {(uint64_t)D, (uint64_t)BS * D};
        const uint32_t box[3] = {(uint32_t)D, BS, 1};
        if (!pkv::encode_tiled_3d(&km, key_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !pkv::encode_tiled_3d(&vm, value_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_NONE))
            return PKV_ERR_CUDA;
    } else if (!encode_3d(&km, key_cache, D, BS, rows, (uint64_t)D * 2, (uint64_t)BS * D * 2, 64, BS, 1) ||
               !encode_3d(&vm, value_cache, D, BS, rows, (uint64_t)D * 2, (uint64_t)BS * D * 2, 64, BS, 1)) {
        return PKV_ERR_CUDA;
    }
    Params p;
    p.tables = block_tables;
    p.plan = static_cast<const uint8_t *>(plan);
    p.out = static_cast<uint16_t *>(out);
    p.err = pool->d_err;
    p.MB = max_blocks;
    p.Hq = num_q_heads;
    p.Hkv = d.num_kv_heads;
    p.group = g;
    p.TP = tp;
    p.num_blocks = d.num_blocks;
    p.grid = grid;
    // (E4M3 pools: q enters the products as q * 2^-8)
    p.score_scale = scale * d.k_scale * LOG2E * (fp8 ? 1.0f / FP8_Q_SCALE : 1.0f);
    p.out_scale = d.v_scale;
    p.test_stall = pkv::test_expire() == PKV_TEST_EXPIRE_PREFILL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = D == 128 ? (fp8 ? launch<128, true>(qm, km, vm, p, s) : launch<128, false>(qm, km, vm, p, s))
                                   : (fp8 ? launch<64, true>(qm, km, vm, p, s) : launch<64, false>(qm, km, vm, p, s));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
