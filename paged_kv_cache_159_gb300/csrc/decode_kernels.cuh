// decode_kernels.cuh -- single-query (decode) GQA attention over the paged KV pool.
//
// What is computed (the pages' definitions):
//   * "传统 Attention 的 KV Cache 问题" (pyllm.pages.dev) §1.1: out = sum_j softmax_j(q.K_j /
//     sqrt(d_k)) V_j.
//   * "理解 KV Cache：Attention、P/D 分离与 vLLM 的页式显存管理" (steinslab.io) §1.2-§1.3: the
//     new token's query attends causally over every cached position of its sequence (j <=
//     its own position, i.e. j < seq_len); §2.2: decode is two GEMVs (q.K^T, then p.V),
//     usually fused into one kernel, bound by reading K and V from HBM; §3.2-§3.3: K/V of
//     a block live at [physical block][kv head][offset][head_dim], physical block =
//     block_table[j / 16].
//   * "KV Cache 与推理优化" (note.yj-dis.top), PagedAttention section: the attention kernel
//     gathers K/V from the physical blocks named by the block table; GQA section: query
//     heads hq = h*g .. h*g+g-1 share KV head h.
//
// GB300 design:
//   * Work unit = (sequence b, KV head h); its work is ceil(L_b/16) blocks.  All g query heads
//     of the group are computed from one read of each K/V tile, so every K/V byte crosses
//     HBM once per step.
//   * Persistent, balanced schedule ("stream-K"): the units' blocks are laid end to end
//     (b-major, then h, then logical block) into W block-tasks and CTA c of a one-wave grid
//     of G CTAs takes tasks [W*c/G, W*(c+1)/G).  Every CTA streams the same number of bytes
//     whatever the batch shape.  W is computed by every CTA from seq_lens (a block-wide scan
//     in shared memory), so the host needs no lengths.
//   * A CTA's range splits into segments at unit boundaries.  A unit that lies wholly in
//     one CTA is finished there.  A unit cut by CTA boundaries leaves a partial softmax
//     state (max, sum, unnormalised output) per CTA in the workspace; each such CTA then
//     bumps the unit's counter, and the one that completes the count merges the partials in
//     CTA order and writes the output (no CTA ever waits for another), then resets the
//     counter to zero.
//   * Each (block, head) tile of K or V is contiguous (16 x head_dim elements: 4 KiB bf16 at
//     head_dim 128), so it is staged by one 1-D bulk (TMA) copy into shared memory.  Every
//     warp owns a ring of `NS` stages (K and V tile each) with one mbarrier per stage and
//     streams the tasks first + warp, first + warp + NW, ...; the copy for a task is issued
//     NS tasks ahead of its use, across segment boundaries.  Physical block ids are fetched
//     32 tasks ahead into registers.  The g query rows of each segment's unit are staged
//     by a bulk copy one segment ahead.  Waits are bounded (about 1 s) and report
//     PKV_DEVERR_TIMEOUT.
//   * Two ways to do the small g x D x 16 contractions, selectable for measurement:
//       - variant 1 (CUDA cores): each lane owns D/32 columns, dot products are finished with
//         warp-shuffle butterflies;
//       - variant 2 (tensor cores, mma.sync m16n8k16): S = Q.K^T with the group padded to 16
//         rows, then O += P.V with P re-used from the S accumulators in registers.  The
//         column order inside the contraction is permuted so that every lane reads whole
//         16-byte pieces of the linear (unswizzled) tiles; Q uses the same permutation.
//   * Online softmax in fp32 in the exp2 domain; the running max is only raised when a new
//     score exceeds it by more than 2^8, which leaves the result unchanged (numerator and
//     denominator share the same reference) and skips almost every accumulator rescale.
//   * Positions past seq_len in the last block are masked by select (scores -> -inf, V rows
//     -> 0), so whatever the tail slots hold (NaN included) never reaches the output.
//   * Every split point and every merge order depends only on seq_lens, the grid size and
//     logical positions, so any physical placement of the blocks gives bit-identical output.
#pragma once

#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "tc_device.cuh"

namespace pkv {
namespace decode {

constexpr int BS = 16;                    // tokens per block
constexpr int MAX_BATCH = 4096;           // sequences per call (prefix scan in shared memory)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_TAU = 8.0f;       // raise the running max only beyond 2^8
constexpr int ACC_PAD = 8;                // floats of padding per merge-area row

struct DecodeParams {
    const uint16_t *q;            // bf16 [layers, B, Hq, D]
    const uint8_t *key_cache;     // [layers, NB, Hkv, 16, D] of bf16 or e4m3
    const uint8_t *value_cache;
    const int32_t *block_tables;  // [B, MB], shared by all layers
    const int32_t *seq_lens;      // [B]
    uint16_t *out;                // bf16 [layers, B, Hq, D]
    int32_t *counters;            // [layers * B * Hkv] arrival counts of split units (kept at zero)
    float *part_o;                // [G][2][group][D]   unnormalised partial outputs
    float *part_ml;               // [G][2][group][2]   (running max in log2 units, sum)
    uint32_t *err;
    const uint16_t *k_new;        // bf16 [layers, B, Hkv, D]: appended at position L-1 (or null)
    const uint16_t *v_new;
    int layers;                   // layers decoded by this launch (stacked layer-major)
    int test_stall;               // failure-path test: streaming warps wait on a barrier nothing completes
    int B, Hq, Hkv, group, MB, num_blocks;
    float score_scale;            // scale * k_scale * log2(e)
    float out_scale;              // v_scale (1 for bf16 pools)
    float inv_k_scale, inv_v_scale;   // fl32(1/scale) for FP8 appends
    // shared-prefix pass (0: none): the leading table entries of sequence b that the prefix
    // pass covered, and its partial state per query row (layer, KV head, sequence, row)
    int shared_prefix;            // blocks the prefix pass may cover
    int unit_cost;                // tasks the split charges each unit besides its blocks
    int32_t *prefix_n;            // [B] covered entries (written by the prefix pass)
    float *pref_o;                // [layers, Hkv, B, group, D]   num * out_scale
    float *pref_ml;               // [layers, Hkv, B, group, 2]   (max in log2 units, sum)
};

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Shared-memory plan of one CTA (host and device agree on it).
struct Layout {
    int stage, q, ml, acc, prefix, lens, pre, nzp, phys, bar, flag, total;
    int ml_slot, acc_slot;                                       // bytes of one merge slot
    __host__ __device__ Layout(int NW, int NS, int tile, int D, int group, int B, int hp)
    {
        int o = 0;
        stage = o;  o += NW * NS * 2 * tile;                      // K and V tiles of every stage
        q = o;      o += 2 * align_up(hp * group * D * 2, 128);  // two segments' q rows
        ml_slot = NW * 16 * 2 * 4;                               // per-warp (max, sum) rows
        ml = o;     o += 2 * ml_slot;
        acc_slot = align_up(NW * group * (D + ACC_PAD) * 4, 128);
        acc = o;    o += 2 * acc_slot;                           // per-warp accumulators
        prefix = o; o += align_up((B + 1) * 4, 16);              // task prefix over sequences
        lens = o;   o += align_up(B * 4, 16);                    // seq_lens
        pre = o;    o += align_up(B * 4, 16);                    // blocks covered by the prefix pass
        nzp = o;    o += align_up((B + 1) * 4, 16);              // sequences with tasks, prefix over b
        phys = o;   o += align_up(NW * NS * 4, 16);              // tile index per stage
        bar = o;    o += (2 * NW * NS + 9) * 8;                  // stage full/empty, q full/free, segment done/free, never
        flag = o;   o += 256;                                    // scan scratch, merge flag
        total = o;
    }
};

__device__ __forceinline__ float warp_allreduce_sum(float x)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(dev::FULL, x, o);
    return x;
}

// a / b for a >= 0, b > 0: the 64-bit division is a long instruction sequence, so operands
// that fit in 32 bits (every practical launch) take the 32-bit one.
__device__ __forceinline__ long long div_nonneg(long long a, long long b)
{
    if ((((unsigned long long)a | (unsigned long long)b) >> 32) == 0)
        return (long long)((uint32_t)a / (uint32_t)b);
    return a / b;
}

// Largest b in [0, B) with prefix[b] <= r (prefix[B] > r assumed).
__device__ __forceinline__ int find_seq(const int32_t *prefix, int B, int r)
{
    int lo = 0, hi = B;                       // invariant: prefix[lo] <= r < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= r) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Unit geometry of task r: layer, sequence, (layer, sequence) row lb = l * B + b, head group h
// (KV heads h*HP .. h*HP + HP - 1), first task of the unit, blocks in it, the sequence's
// length and its blocks covered by the shared-prefix pass.  Layers are laid end to end, each
// with the same task layout (prefix: tasks before sequence b within a layer, W1 per layer).
struct Unit { int l, b, lb, h, L, nb, pre; long long U0; };

// Not inlined: the paths that call it run once per unit or per 32 tasks, mostly at a launch's
// start and end while the instruction cache is cold, so they share one copy of the code.
static __device__ __noinline__ Unit unit_at(long long r, const int32_t *prefix, const int32_t *lens, const int32_t *pre,
                                     int B, int layers, int W1, int HG)
{
    Unit u;
    u.l = 0;
    if (layers > 1) u.l = (int)div_nonneg(r, W1);
    const int rl = (int)(r - (long long)u.l * W1);
    u.b = find_seq(prefix, B, rl);
    u.lb = u.l * B + u.b;
    const int tasks = prefix[u.b + 1] - prefix[u.b];
    u.nb = tasks / HG;
    u.h = (rl - prefix[u.b]) / u.nb;
    u.U0 = (long long)u.l * W1 + prefix[u.b] + (long long)u.h * u.nb;
    u.L = lens[u.b];
    u.pre = pre[u.b];
    return u;
}

// The split of the tasks over G CTAs.  Every unit (layer, sequence, head group with at least
// one task) is charged OV tasks' worth of cost besides its blocks -- the fixed work of a unit
// in a CTA: its q rows, its softmax state's hand-off and merge -- so that a CTA given many
// short units gets fewer blocks.  Cost position of task r: P(r) = r + OV * (ordinal of r's
// unit); the C cost units are cut evenly: task r goes to CTA floor(P(r) G / C).  Within a
// unit P grows by 1 per task and G <= W <= C, so no CTA inside a unit's run is skipped; a CTA
// whose whole share falls between two units gets no task.  With OV = 0 this is the even split
// of the tasks.
struct Split {
    const int32_t *prefix;        // [B + 1] tasks before sequence b, within a layer
    const int32_t *nzp;           // [B + 1] sequences with tasks before b
    int B, HG, OV, G;
    long long W1, W, C1, C;       // tasks, cost of a layer; tasks, cost of the launch

    // CTA of task r of unit (l, b, h)
    __device__ __forceinline__ int owner(long long r, int l, int b, int h) const
    {
        const long long P = r + (long long)OV * ((long long)l * nzp[B] * HG + (long long)nzp[b] * HG + h);
        return (int)div_nonneg(P * G, C);
    }
    // first task whose cost position is at least T (W past the last)
    __device__ __forceinline__ long long first_at(long long T) const
    {
        if (T >= C) return W;
        const int l = (int)div_nonneg(T, C1);
        const long long Tl = T - (long long)l * C1;
        if (Tl >= C1 - OV) return (long long)(l + 1) * W1;        // the gap after the layer's last unit
        // the first sequence whose last task lies at Tl or later
        const long long ovh = (long long)OV * HG;
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid + 1] + ovh * nzp[mid + 1] - OV > Tl) hi = mid;
            else lo = mid + 1;
        }
        const int b = lo;
        const long long local = Tl - (prefix[b] + ovh * nzp[b]);
        long long r = prefix[b];
        if (local > 0) {
            const int nb = (prefix[b + 1] - prefix[b]) / HG;
            const long long hh = div_nonneg(local, nb + OV), k = local - hh * (nb + OV);
            r += hh * nb + (k < nb ? k : nb);
        }
        return (long long)l * W1 + r;
    }
    __device__ __forceinline__ long long start(int c) const { return first_at(div_nonneg(c * C + G - 1, G)); }
};

// ------------------------------------------------------------------------------------
// Tensor-core compute (variant 2).  Lane l: gid = l/4 (mma row group), tid = l%4.
// ------------------------------------------------------------------------------------
template <int D, bool FP8, bool G16>
struct MmaCompute {
    static constexpr bool SWIZZLED = false;    // linear tiles (1-D bulk copies)
    static constexpr bool IDENTITY_SLOTS = false;   // merge-area columns in fragment order
    static constexpr int ELEM = FP8 ? 1 : 2;
    static constexpr int ROW = D * ELEM;
    static constexpr int KS = D / 16;                   // k-steps of S = Q.K^T
    static constexpr int EK = 16 / ELEM;                // elements in a 16-byte piece
    static constexpr int SUBS = EK / 4;                 // k-steps per piece
    static constexpr int NI = D / (4 * EK);             // pieces per lane per K row
    static constexpr int NT = D / 8;                    // n-tiles of O = P.V
    static constexpr int EV = FP8 ? (D == 64 ? 8 : 16) : 8;   // V elements per lane load
    static constexpr int VB = EV * ELEM;                // bytes per V load (16 or 8)
    static constexpr int VCH = D / (8 * EV);            // V loads per lane per row

    uint32_t qa[KS][4];
    float acc[NT][4];
    float m[2], l[2];

    // Column d of O held by n-tile nt, mma column n.
    __device__ static int dmap(int nt, int n) { return (n + 8 * (nt / EV)) * EV + nt % EV; }
    // Where column d sits in a merge-area row (fragment order: nt*8 + n).
    __device__ static int slot_of_d(int d) { return ((d / (8 * EV)) * EV + d % EV) * 8 + (d / EV) % 8; }

    // Load the q fragments of rows 0..group-1 (bf16 [group][D] in shared memory) and reset
    // the softmax state.
    __device__ void start(const uint16_t *qs, int group, int lane)
    {
        const int gid = lane >> 2, tid = lane & 3;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int d0 = (4 * (ks / SUBS) + tid) * EK + (ks % SUBS) * 4;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int row = gid + 8 * r;
                uint32_t lo = 0, hi = 0;
                if (row < group && (r == 0 || G16)) {
                    const uint32_t *src = reinterpret_cast<const uint32_t *>(qs + row * D + d0);
                    lo = src[0];
                    hi = src[1];
                    if constexpr (FP8) {
                        lo = dev::pack_f16x2(dev::bf16_lo(lo), dev::bf16_hi(lo));
                        hi = dev::pack_f16x2(dev::bf16_lo(hi), dev::bf16_hi(hi));
                    }
                }
                qa[ks][r] = lo;          // a0 (row gid) / a1 (row gid+8): k = 2tid, 2tid+1
                qa[ks][2 + r] = hi;      // a2 / a3: k = 2tid+8, 2tid+9
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[nt][c] = 0.f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
    }

    __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
    {
        if constexpr (FP8) dev::mma_f16_16816(d, a, b0, b1);
        else dev::mma_bf16_16816(d, a, b0, b1);
    }

    // One 16-token block from a staged K/V tile; ntok valid tokens (1..16).
    __device__ void block(const uint8_t *kt, const uint8_t *vt, int ntok, float score_scale, int lane)
    {
        const int gid = lane >> 2, tid = lane & 3;
        // ---- S = Q K^T : rows = query heads, columns = tokens (n-tile 0: 0-7, 1: 8-15)
        float s[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
            const uint8_t *row = kt + (gid + 8 * nt) * ROW;
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const uint4 c = *reinterpret_cast<const uint4 *>(row + (4 * i + tid) * 16);
                const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                for (int sub = 0; sub < SUBS; ++sub) {
                    uint32_t b0, b1;
                    if constexpr (FP8) {
                        b0 = dev::e4m3x2_to_f16x2((uint16_t)(w[sub] & 0xffffu));
                        b1 = dev::e4m3x2_to_f16x2((uint16_t)(w[sub] >> 16));
                    } else {
                        b0 = w[2 * sub];
                        b1 = w[2 * sub + 1];
                    }
                    mma(s[nt], qa[i * SUBS + sub], b0, b1);
                }
            }
        }
        // ---- mask, scale, running max (rows gid and gid+8)
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int tok = nt * 8 + 2 * tid + (c & 1);
                const float x = s[nt][c] * score_scale;
                s[nt][c] = tok < ntok ? x : -INFINITY;
                mx[c >> 1] = fmaxf(mx[c >> 1], s[nt][c]);
            }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(dev::FULL, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(dev::FULL, mx[r], 2));
        }
        const bool need = (mx[0] > m[0] + RESCALE_TAU) || (mx[1] > m[1] + RESCALE_TAU);
        if (__any_sync(dev::FULL, need)) {
            float alpha[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float mn = fmaxf(m[r], mx[r]);
                alpha[r] = dev::fast_exp2(m[r] - mn);
                m[r] = mn;
                l[r] *= alpha[r];
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                acc[nt][0] *= alpha[0];
                acc[nt][1] *= alpha[0];
                acc[nt][2] *= alpha[1];
                acc[nt][3] *= alpha[1];
            }
        }
        // ---- P = exp2(S - m), row sums, P as the A operand of P.V
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                s[nt][c] = dev::fast_exp2(s[nt][c] - m[c >> 1]);
                l[c >> 1] += s[nt][c];
            }
        uint32_t pa[4];
        if (FP8) {
            pa[0] = dev::pack_f16x2(s[0][0], s[0][1]);
            pa[1] = dev::pack_f16x2(s[0][2], s[0][3]);
            pa[2] = dev::pack_f16x2(s[1][0], s[1][1]);
            pa[3] = dev::pack_f16x2(s[1][2], s[1][3]);
        } else {
            pa[0] = dev::pack_bf16x2(s[0][0], s[0][1]);
            pa[1] = dev::pack_bf16x2(s[0][2], s[0][3]);
            pa[2] = dev::pack_bf16x2(s[1][0], s[1][1]);
            pa[3] = dev::pack_bf16x2(s[1][2], s[1][3]);
        }
        // ---- O += P V.  Lane gid reads pieces gid + 8c of the V rows 2tid, 2tid+1, 2tid+8,
        //      2tid+9 (the tokens its B fragments need); n-tile nt = c*EV + e covers the
        //      columns dmap(nt, 0..7).  One piece at a time keeps register use low.
#pragma unroll
        for (int c = 0; c < VCH; ++c) {
            uint32_t vw[4][VB / 4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int tok = 2 * tid + (r & 1) + 8 * (r >> 1);
                const uint8_t *row = vt + tok * ROW;
                if constexpr (VB == 16) {
                    const uint4 x = *reinterpret_cast<const uint4 *>(row + (gid + 8 * c) * 16);
                    vw[r][0] = x.x; vw[r][1] = x.y; vw[r][2] = x.z; vw[r][3] = x.w;
                } else {
                    const uint2 x = *reinterpret_cast<const uint2 *>(row + (gid + 8 * c) * 8);
                    vw[r][0] = x.x; vw[r][1] = x.y;
                }
                if (tok >= ntok) {              // masked row: zero, whatever the slot holds
#pragma unroll
                    for (int w = 0; w < VB / 4; ++w) vw[r][w] = 0u;
                }
            }
#pragma unroll
            for (int e = 0; e < EV; ++e) {
                const int nt = c * EV + e;
                uint32_t b0, b1;
                if constexpr (FP8) {
                    const uint32_t sel = (uint32_t)((e & 3) | ((4 + (e & 3)) << 4));
                    b0 = dev::e4m3x2_to_f16x2((uint16_t)__byte_perm(vw[0][e >> 2], vw[1][e >> 2], sel));
                    b1 = dev::e4m3x2_to_f16x2((uint16_t)__byte_perm(vw[2][e >> 2], vw[3][e >> 2], sel));
                } else {
                    const uint32_t sel = (e & 1) ? 0x7632u : 0x5410u;
                    b0 = __byte_perm(vw[0][e >> 1], vw[1][e >> 1], sel);
                    b1 = __byte_perm(vw[2][e >> 1], vw[3][e >> 1], sel);
                }
                mma(acc[nt], pa, b0, b1);
            }
        }
    }

    // Write this warp's (max, sum) rows and accumulators into the merge area.
    __device__ void dump(float *ml, float *accs, int group, int lane)
    {
        const int gid = lane >> 2, tid = lane & 3;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l[r] += __shfl_xor_sync(dev::FULL, l[r], 1);
            l[r] += __shfl_xor_sync(dev::FULL, l[r], 2);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = gid + 8 * r;
            if (row < group) {
                if (tid == 0) {
                    ml[row * 2] = m[r];
                    ml[row * 2 + 1] = l[r];
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    *reinterpret_cast<float2 *>(accs + row * (D + ACC_PAD) + nt * 8 + 2 * tid) =
                        make_float2(acc[nt][2 * r], acc[nt][2 * r + 1]);
            }
        }
    }
};

// ------------------------------------------------------------------------------------
// CUDA-core compute (variant 1).  Lane l owns columns [l*EPL, l*EPL + EPL).
// ------------------------------------------------------------------------------------
template <int D, bool FP8, int GP>
struct SimtCompute {
    static constexpr bool SWIZZLED = false;    // linear tiles (1-D bulk copies)
    static constexpr bool IDENTITY_SLOTS = true;    // merge-area column d at d
    static constexpr int ELEM = FP8 ? 1 : 2;
    static constexpr int ROW = D * ELEM;
    static constexpr int EPL = D / 32;
    static constexpr int HALF = 8;                       // tokens per softmax step

    float qf[GP][EPL];
    float acc[GP][EPL];
    float m[GP], l[GP];
    float sscale;

    __device__ static int slot_of_d(int d) { return d; }

    __device__ void start(const uint16_t *qs, int group, int lane)
    {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                float x = 0.f;
                if (g < group) x = __uint_as_float((uint32_t)qs[g * D + lane * EPL + e] << 16);
                if (FP8) x = __half2float(__float2half_rn(x));   // same q rounding as variant 2
                qf[g][e] = x * sscale;
                acc[g][e] = 0.f;
            }
            m[g] = -INFINITY;
            l[g] = 0.f;
        }
    }

    __device__ __forceinline__ void load_row(const uint8_t *row, int lane, float (&x)[EPL])
    {
        if constexpr (FP8) {
            const uint8_t *src = row + lane * EPL;
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
                const uint32_t h2 = dev::e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t *>(src + e));
                const __half2 hv = *reinterpret_cast<const __half2 *>(&h2);
                x[e] = __low2float(hv);
                x[e + 1] = __high2float(hv);
            }
        } else {
            const uint32_t *src = reinterpret_cast<const uint32_t *>(row + lane * EPL * 2);
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
                const uint32_t w = src[e / 2];
                x[e] = dev::bf16_lo(w);
                x[e + 1] = dev::bf16_hi(w);
            }
        }
    }

    __device__ void block(const uint8_t *kt, const uint8_t *vt, int ntok, float /*score_scale*/, int lane)
    {
#pragma unroll
        for (int t0 = 0; t0 < BS; t0 += HALF) {
            if (t0 >= ntok) break;
            float s[HALF][GP];
#pragma unroll
            for (int t = 0; t < HALF; ++t) {
                float k[EPL];
                load_row(kt + (t0 + t) * ROW, lane, k);
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    float part = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) part = fmaf(qf[g][e], k[e], part);
                    s[t][g] = warp_allreduce_sum(part);
                }
            }
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                float mx = -INFINITY;
#pragma unroll
                for (int t = 0; t < HALF; ++t) {
                    if (t0 + t >= ntok) s[t][g] = -INFINITY;
                    mx = fmaxf(mx, s[t][g]);
                }
                if (mx > m[g] + RESCALE_TAU) {
                    const float mn = fmaxf(m[g], mx);
                    const float alpha = dev::fast_exp2(m[g] - mn);
                    m[g] = mn;
                    l[g] *= alpha;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[g][e] *= alpha;
                }
#pragma unroll
                for (int t = 0; t < HALF; ++t) {
                    s[t][g] = dev::fast_exp2(s[t][g] - m[g]);
                    l[g] += s[t][g];
                }
            }
#pragma unroll
            for (int t = 0; t < HALF; ++t) {
                if (t0 + t >= ntok) break;
                float v[EPL];
                load_row(vt + (t0 + t) * ROW, lane, v);
#pragma unroll
                for (int g = 0; g < GP; ++g)
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(s[t][g], v[e], acc[g][e]);
            }
        }
    }

    __device__ void dump(float *ml, float *accs, int group, int lane)
    {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            if (g < group) {
                if (lane == 0) {
                    ml[g * 2] = m[g];
                    ml[g * 2 + 1] = l[g];
                }
#pragma unroll
                for (int e = 0; e < EPL; ++e) accs[g * (D + ACC_PAD) + lane * EPL + e] = acc[g][e];
            }
        }
    }
};

// ------------------------------------------------------------------------------------
// Tensor-core compute with the block's 16 tokens as the mma rows (variant 3).
//
//   S^T = K . Q^T      (M 16 tokens, N 8 query heads per n-tile, K head_dim)
//   O^T += V^T . P^T   (M 16 output columns per m-tile, N 8 heads, K 16 tokens)
//
// The g <= 8 heads of a group fill one n-tile of 8 (two for g <= 16), so at most half of each
// product is padding, against 3/4 with the heads as the 16 rows.  K and V tiles arrive in
// shared memory through tensor (TMA) copies with a 128-byte swizzle (64-byte for 64-byte
// rows), so the 8 token rows that one ldmatrix reads lie in 8 different bank groups: the
// reads are conflict-free.  The same per-lane ldmatrix addresses serve K (plain) and V
// (transposed).  P^T, the B operand of the second product, comes from the S^T accumulators by
// one movmatrix per 8 tokens.
//
// FP8 pools: S^T runs on the E4M3 tensor-core product (k 32), K straight from shared memory.
// The queries, scaled by a power of two per unit (exact) so that their largest magnitude lies
// in [128, 256), are split into two E4M3 terms q = q_hi + q_lo; for every bf16 query value
// whose scaled magnitude is at least 2^-2 the split is exact (the rounding residual of a
// 4-significant-bit code on an 8-significant-bit value has at most 4 significant bits), and
// below that its error is at most 2^-10 of the scaled value's unit, 2^-18 of the largest
// query.  V codes are converted to fp16 (exact) after a transposed ldmatrix and multiplied
// with P in fp16.
// ------------------------------------------------------------------------------------
template <int D, bool FP8, int NH>
struct TokCompute {
    static constexpr bool SWIZZLED = true;
    static constexpr bool IDENTITY_SLOTS = true;    // merge-area column d at d
    static constexpr int ELEM = FP8 ? 1 : 2;
    static constexpr int ROWB = D * ELEM;                 // bytes of one token row
    static constexpr int SEG = ROWB < 128 ? ROWB : 128;   // bytes of one swizzled row segment
    static constexpr int SEGBYTES = BS * SEG;             // one [16 tokens][SEG] segment of a tile
    static constexpr int STEPS = ROWB / 32;               // ldmatrix.x4 steps (two 16-byte chunks each)
    static constexpr int MT = D / 16;                     // m-tiles of O^T
    static constexpr int NOFF = STEPS < 4 ? STEPS : 4;
    static constexpr int QW = FP8 ? 4 : 2;                // B-fragment words of Q^T per step

    uint32_t qb[STEPS][NH][QW];
    float acc[MT][NH][4];
    float m[NH][2], l[NH][2];
    uint32_t loff[NOFF];          // this lane's ldmatrix row address within a tile, per step % 4
    float base_sc = 0.f;          // scale * k_scale * log2(e)
    float sc = 0.f;               // the unit's score scale (FP8: with the queries' power of two)
    int lim[NH][2];               // column mode: positions < lim of this lane's columns are valid

    // Output column of O^T row r (0..15) of m-tile mt.
    __device__ static int dcol(int mt, int r) { return FP8 ? 16 * mt + 2 * (r & 7) + (r >> 3) : 16 * mt + r; }
    __device__ static int slot_of_d(int d) { return d; }

    // Lane l gives the row address of ldmatrix matrix l/8: token (l%8) + 8((l/8)%2), 16-byte
    // chunk 2 step + l/16.  With the swizzle the chunk lands at (chunk % 8) xor (row % 8)
    // (128-byte segments) or chunk xor ((row/2) % 4) (64-byte rows).
    __device__ void setup(int lane)
    {
        const int tok = (lane & 7) + 8 * ((lane >> 3) & 1), hi = lane >> 4;
#pragma unroll
        for (int k = 0; k < NOFF; ++k) {
            if constexpr (SEG == 128) loff[k] = tok * 128 + (((2 * k) ^ (hi ^ (tok & 7))) << 4);
            else loff[k] = tok * 64 + (((2 * k) ^ (hi ^ ((tok >> 1) & 3))) << 4);
        }
    }

    __device__ __forceinline__ uint32_t step_addr(uint32_t tile, int i) const
    {
        return tile + loff[i & 3] + (uint32_t)((i >> 2) * SEGBYTES);
    }

    // Four E4M3 codes (round to nearest even, saturating) of four floats.
    __device__ static uint32_t e4m3x4(float a, float b, float c, float d)
    {
        return dev::e4m3x2_satfinite(a, b) | (dev::e4m3x2_satfinite(c, d) << 16);
    }
    __device__ static float2 e4m3x2_value(uint32_t codes)
    {
        const uint32_t h = dev::e4m3x2_to_f16x2((uint16_t)codes);
        return __half22float2(*reinterpret_cast<const __half2 *>(&h));
    }

    // Load the Q^T fragments of the unit's g query rows (bf16 [group][D] in shared memory)
    // and reset the softmax state.  Heads past the group are zero.
    __device__ void start(const uint16_t *qs, int group, int lane)
    {
        const int gid = lane >> 2, tid = lane & 3;
        sc = base_sc;
        if constexpr (!FP8) {
#pragma unroll
            for (int i = 0; i < STEPS; ++i)
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    const int head = 8 * j + gid;
                    const uint32_t *row = reinterpret_cast<const uint32_t *>(qs + head * D + 16 * i + 2 * tid);
                    qb[i][j][0] = head < group ? row[0] : 0u;     // d 16i + 2tid, +1
                    qb[i][j][1] = head < group ? row[4] : 0u;     // d 16i + 8 + 2tid, +1
                }
        } else {
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < STEPS; ++i)
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    const int head = 8 * j + gid;
                    uint2 lo = make_uint2(0u, 0u), hi = make_uint2(0u, 0u);
                    if (head < group) {
                        lo = *reinterpret_cast<const uint2 *>(qs + head * D + 32 * i + 4 * tid);        // d 32i+4tid..+3
                        hi = *reinterpret_cast<const uint2 *>(qs + head * D + 32 * i + 16 + 4 * tid);   // d 32i+16+4tid..
                    }
                    qb[i][j][0] = lo.x; qb[i][j][1] = lo.y; qb[i][j][2] = hi.x; qb[i][j][3] = hi.y;
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        amax = fmaxf(amax, fmaxf(fabsf(dev::bf16_lo(qb[i][j][w])), fabsf(dev::bf16_hi(qb[i][j][w]))));
                }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(dev::FULL, amax, o));
            // 2^e: amax * 2^e in [128, 256); e within the normal exponent range
            int e = 0;
            if (amax > 0.f) e = 7 - (((__float_as_uint(amax) >> 23) & 0xff) - 127);
            e = max(-126, min(126, e));
            const float up = __uint_as_float((uint32_t)(127 + e) << 23);
            sc = base_sc * __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
            for (int i = 0; i < STEPS; ++i)
#pragma unroll
                for (int j = 0; j < NH; ++j) {
                    float x[8];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        x[2 * w] = dev::bf16_lo(qb[i][j][w]) * up;
                        x[2 * w + 1] = dev::bf16_hi(qb[i][j][w]) * up;
                    }
                    const uint32_t h0 = e4m3x4(x[0], x[1], x[2], x[3]), h1 = e4m3x4(x[4], x[5], x[6], x[7]);
                    const float2 a = e4m3x2_value(h0), b = e4m3x2_value(h0 >> 16);
                    const float2 c = e4m3x2_value(h1), d = e4m3x2_value(h1 >> 16);
                    qb[i][j][0] = h0;                                   // b0 of the high term
                    qb[i][j][1] = h1;                                   // b1 of the high term
                    qb[i][j][2] = e4m3x4(x[0] - a.x, x[1] - a.y, x[2] - b.x, x[3] - b.y);   // low term
                    qb[i][j][3] = e4m3x4(x[4] - c.x, x[5] - c.y, x[6] - d.x, x[7] - d.y);
                }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int j = 0; j < NH; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[mt][j][c] = 0.f;
#pragma unroll
        for (int j = 0; j < NH; ++j) {
            m[j][0] = m[j][1] = -INFINITY;
            l[j][0] = l[j][1] = 0.f;
        }
    }

    __device__ __forceinline__ void pv_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
    {
        if constexpr (FP8) dev::mma_f16_16816(d, a, b0, b1);
        else dev::mma_bf16_16816(d, a, b0, b1);
    }

    // One 16-token block; PARTIAL: only tokens < ntok are valid (the rest masked by select).
    // COLS: besides, position pos0 + token is valid for column (query row) c only below
    // lim[][] -- the rows of several sequences over a shared block.
    template <bool PARTIAL, bool COLS = false>
    __device__ __forceinline__ void block_impl(uint32_t kt, uint32_t vt, int ntok, int lane, int pos0 = 0)
    {
        const int gid = lane >> 2, tid = lane & 3;
        // ---- S^T = K Q^T: rows = tokens gid, gid + 8; columns = heads 8j + 2tid, +1.  Two
        //      independent accumulator chains (FP8: the high and low query terms; bf16: even
        //      and odd k-steps) halve the dependent mma latency, then add.
        float s[NH][4], s2[NH][4];
#pragma unroll
        for (int j = 0; j < NH; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[j][c] = s2[j][c] = 0.f;
#pragma unroll
        for (int i = 0; i < STEPS; ++i) {
            uint32_t a[4];
            dev::ldsm_x4(step_addr(kt, i), a);
#pragma unroll
            for (int j = 0; j < NH; ++j) {
                if constexpr (FP8) {
                    dev::mma_e4m3_16832(s[j], a, qb[i][j][0], qb[i][j][1]);
                    dev::mma_e4m3_16832(s2[j], a, qb[i][j][2], qb[i][j][3]);
                } else {
                    dev::mma_bf16_16816((i & 1) ? s2[j] : s[j], a, qb[i][j][0], qb[i][j][1]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < NH; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[j][c] += s2[j][c];
        // ---- scale, mask, lazy running max (heads 8j + 2tid + r: values c = r and r + 2)
        bool need = false;
#pragma unroll
        for (int j = 0; j < NH; ++j) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float x = s[j][c] * sc;
                const int tok = gid + 8 * (c >> 1);
                bool valid = !PARTIAL || tok < ntok;
                if constexpr (COLS) valid = valid && pos0 + tok < lim[j][c & 1];
                s[j][c] = valid ? x : -INFINITY;
            }
            need |= fmaxf(s[j][0], s[j][2]) > m[j][0] + RESCALE_TAU;
            need |= fmaxf(s[j][1], s[j][3]) > m[j][1] + RESCALE_TAU;
        }
        if (__any_sync(dev::FULL, need)) {
#pragma unroll
            for (int j = 0; j < NH; ++j)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    float mx = fmaxf(s[j][r], s[j][r + 2]);
                    mx = fmaxf(mx, __shfl_xor_sync(dev::FULL, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(dev::FULL, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(dev::FULL, mx, 16));
                    const float mn = fmaxf(m[j][r], mx);
                    const float alpha = dev::fast_exp2(m[j][r] - mn);
                    m[j][r] = mn;
                    l[j][r] *= alpha;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        acc[mt][j][r] *= alpha;
                        acc[mt][j][r + 2] *= alpha;
                    }
                }
        }
        // ---- P = exp2(S - m); P^T as the B operand of the second product (one movmatrix per
        //      8 tokens: tokens 2tid, 2tid+1 of head gid in b0, tokens 8 + those in b1)
        uint32_t pb[NH][2];
#pragma unroll
        for (int j = 0; j < NH; ++j) {
            const float p0 = dev::fast_exp2(s[j][0] - m[j][0]), p1 = dev::fast_exp2(s[j][1] - m[j][1]);
            const float p2 = dev::fast_exp2(s[j][2] - m[j][0]), p3 = dev::fast_exp2(s[j][3] - m[j][1]);
            l[j][0] += p0 + p2;
            l[j][1] += p1 + p3;
            const uint32_t r0 = FP8 ? dev::pack_f16x2(p0, p1) : dev::pack_bf16x2(p0, p1);
            const uint32_t r1 = FP8 ? dev::pack_f16x2(p2, p3) : dev::pack_bf16x2(p2, p3);
            pb[j][0] = dev::movmatrix_trans(r0);
            pb[j][1] = dev::movmatrix_trans(r1);
        }
        // ---- O^T += V^T P^T.  Transposed ldmatrix of step i: registers 0 and 2 hold tokens
        //      2tid, 2tid+1 (low and high halves), 1 and 3 tokens 8 + those; rows past ntok are
        //      zeroed in the registers (a NaN there would survive P = 0).
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if constexpr (PARTIAL) {
            mlo = (2 * tid < ntok ? 0x0000ffffu : 0u) | (2 * tid + 1 < ntok ? 0xffff0000u : 0u);
            mhi = (2 * tid + 8 < ntok ? 0x0000ffffu : 0u) | (2 * tid + 9 < ntok ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int i = 0; i < STEPS; ++i) {
            uint32_t v[4];
            dev::ldsm_x4_trans(step_addr(vt, i), v);
            if constexpr (PARTIAL) {
                v[0] &= mlo; v[2] &= mlo;
                v[1] &= mhi; v[3] &= mhi;
            }
            if constexpr (!FP8) {
                // m-tile i: rows d 16i + gid (chunk 2i) and 16i + 8 + gid (chunk 2i + 1)
                const uint32_t a[4] = {v[0], v[2], v[1], v[3]};
#pragma unroll
                for (int j = 0; j < NH; ++j) pv_mma(acc[i][j], a, pb[j][0], pb[j][1]);
            } else {
                // m-tiles 2i (chunk 2i: v0, v1) and 2i + 1 (chunk 2i + 1: v2, v3); a register's
                // bytes are (token 2tid: d, d + 1), (token 2tid + 1: d, d + 1) with d = 2gid in
                // the chunk: bytes 0 and 2 make row d, bytes 1 and 3 row d + 1
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t x = v[2 * h], y = v[2 * h + 1];
                    const uint32_t a[4] = {dev::e4m3x2_to_f16x2((uint16_t)__byte_perm(x, 0u, 0x20u)),
                                           dev::e4m3x2_to_f16x2((uint16_t)__byte_perm(x, 0u, 0x31u)),
                                           dev::e4m3x2_to_f16x2((uint16_t)__byte_perm(y, 0u, 0x20u)),
                                           dev::e4m3x2_to_f16x2((uint16_t)__byte_perm(y, 0u, 0x31u))};
#pragma unroll
                    for (int j = 0; j < NH; ++j) pv_mma(acc[2 * i + h][j], a, pb[j][0], pb[j][1]);
                }
            }
        }
    }

    __device__ void block(const uint8_t *kt, const uint8_t *vt, int ntok, float /*score_scale*/, int lane)
    {
        if (ntok == BS) block_impl<false>(dev::smem_u32(kt), dev::smem_u32(vt), BS, lane);
        else block_impl<true>(dev::smem_u32(kt), dev::smem_u32(vt), ntok, lane);
    }

    // Write this warp's (max, sum) rows and accumulators into the merge area ([head][d]).
    __device__ void dump(float *ml, float *accs, int group, int lane)
    {
        const int gid = lane >> 2, tid = lane & 3;
#pragma unroll
        for (int j = 0; j < NH; ++j)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float x = l[j][r];
                x += __shfl_xor_sync(dev::FULL, x, 4);
                x += __shfl_xor_sync(dev::FULL, x, 8);
                x += __shfl_xor_sync(dev::FULL, x, 16);
                l[j][r] = x;
            }
#pragma unroll
        for (int j = 0; j < NH; ++j)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int head = 8 * j + 2 * tid + r;
                if (head < group) {
                    if (gid == 0) {
                        ml[head * 2] = m[j][r];
                        ml[head * 2 + 1] = l[j][r];
                    }
                    float *row = accs + head * (D + ACC_PAD);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        row[dcol(mt, gid)] = acc[mt][j][r];
                        row[dcol(mt, gid + 8)] = acc[mt][j][r + 2];
                    }
                }
            }
    }
};

// ------------------------------------------------------------------------------------
// The decode kernel body: NW streaming warps and one epilogue warp.
// ------------------------------------------------------------------------------------
template <int D, bool FP8, int NW, int NS, int HP, class Compute>
__device__ __forceinline__ void decode_body(const DecodeParams &p, Compute &cmp, const CUtensorMap *kmap,
                                            const CUtensorMap *vmap)
{
    constexpr int ELEM = FP8 ? 1 : 2;
    constexpr int TILE = BS * D * ELEM;           // one (block, KV head) tile of K or V
    constexpr int NWARP = NW + 2;                 // NW consumers, the epilogue warp, the producer
    constexpr int NTHR = NWARP * 32;
    // A task is one block of HP consecutive KV heads, loaded by one copy of HP tiles for K and
    // one for V.  Consumer warp w takes head w % HP of the tasks of stream w / HP.
    constexpr int NSTREAM = NW / HP;
    constexpr int NSTAGE = NSTREAM * NS;          // CTA-wide ring; task i: stage i % NSTAGE, stream i % NSTREAM
    constexpr int STAGE = 2 * HP * TILE;          // K tiles, then V tiles
    static_assert(NW % HP == 0 && NSTAGE <= 32 && 32 % NSTREAM == 0, "ring and step shapes");
    // swizzled tiles: SEG-byte row segments, [segment][16 tokens][SEG] per tile
    constexpr int SEG = D * ELEM < 128 ? D * ELEM : 128;
    constexpr int NSEG = D * ELEM / SEG;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the stage ring starts 1024-byte aligned (the swizzle pattern repeats every 1024 bytes)
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);
    const Layout lay(NW, NS, TILE, D, p.group, p.B, HP);
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + lay.prefix);
    int32_t *stage_tile = reinterpret_cast<int32_t *>(smem + lay.phys);
    int *flag = reinterpret_cast<int *>(smem + lay.flag);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int Hkv = p.Hkv, group = p.group;
    const int HG = Hkv / HP;                      // head groups: units are (layer, sequence, head group)

    // ---- 0. warm L2 with this CTA's share of the block tables and queries (hints), and
    //         set up the barriers; both overlap the scan below.
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bar);
    const uint32_t full0 = dev::smem_u32(bars);                   // stage j loaded: +8*j
    const uint32_t empty0 = dev::smem_u32(bars + NSTAGE);         // stage j consumed: +8*j
    const uint32_t qbar0 = dev::smem_u32(bars + 2 * NSTAGE);      // q slot j full: +8*j
    const uint32_t done0 = dev::smem_u32(bars + 2 * NSTAGE + 2);  // merge slot j dumped
    const uint32_t free0 = dev::smem_u32(bars + 2 * NSTAGE + 4);  // merge slot j merged
    const uint32_t never = dev::smem_u32(bars + 2 * NSTAGE + 6);  // no thread ever arrives here
    const uint32_t qfree0 = dev::smem_u32(bars + 2 * NSTAGE + 7); // q slot j read into registers
    if (tid == 0) {
        auto slice = [&](const void *base, size_t bytes) {
            const uintptr_t a0 = (reinterpret_cast<uintptr_t>(base) + bytes * c / gridDim.x + 15) & ~uintptr_t(15);
            const uintptr_t a1 = (reinterpret_cast<uintptr_t>(base) + bytes * (c + 1) / gridDim.x) & ~uintptr_t(15);
            if (a1 > a0) dev::prefetch_l2(reinterpret_cast<const void *>(a0), (uint32_t)(a1 - a0));
        };
        slice(p.block_tables, (size_t)p.B * p.MB * 4);
        slice(p.q, (size_t)p.layers * p.B * p.Hq * D * 2);
        for (int j = 0; j < 2; ++j) {
            dev::mbar_init(qbar0 + 8 * j, 1);
            dev::mbar_init(done0 + 8 * j, NW * 32);
            dev::mbar_init(free0 + 8 * j, 1);
            dev::mbar_init(qfree0 + 8 * j, NW);
        }
        dev::mbar_init(never, 1);
    }
    if (warp == NW + 1 && lane == 31 && kmap) {               // descriptors, ahead of the first copy
        tc::prefetch_tensormap(kmap);
        tc::prefetch_tensormap(vmap);
    }
    if (warp == NW + 1 && lane < NSTAGE) {
        dev::mbar_init(full0 + 8 * lane, 1);          // the producer's arrive (+ the copies' bytes)
        dev::mbar_init(empty0 + 8 * lane, HP);        // the stream's HP consumer warps
    }
    dev::fence_barrier_init();

    // ---- 1. tasks per sequence (Hkv * ceil(L/16); 0 for an invalid length) and their
    //         exclusive prefix, by a block-wide scan; CTA 0 zeroes invalid sequences' rows.
    int32_t *lens = reinterpret_cast<int32_t *>(smem + lay.lens);
    int32_t *pre = reinterpret_cast<int32_t *>(smem + lay.pre);
    int32_t *nzp = reinterpret_cast<int32_t *>(smem + lay.nzp);
    {
        const int per = (p.B + NTHR - 1) / NTHR;
        const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
        int run = 0, nz = 0, lo = INT_MAX, hi = -1;       // lo/hi: blocks per sequence
        for (int b = b0; b < b1; ++b) {
            const int L = __ldg(p.seq_lens + b);
            lens[b] = L;
            pre[b] = p.shared_prefix ? p.prefix_n[b] : 0;
            const bool ok = L >= 1 && L <= p.MB * BS;
            if (!ok && c == 0) {
                dev::flag_error(p.err, PKV_DEVERR_SEQ_LEN);
                for (int l = 0; l < p.layers; ++l)
                    for (int e = 0; e < p.Hq * D; ++e) p.out[((size_t)l * p.B + b) * p.Hq * D + e] = 0;
            }
            // blocks past those the prefix pass covered; an invalid length breaks uniformity
            const int nb = ok ? (L + BS - 1) / BS - pre[b] : 0;
            run += HG * nb;
            nz += nb > 0;
            lo = min(lo, nb);
            hi = max(hi, nb);
        }
        int incl = run, incz = nz;                        // inclusive scans over the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(dev::FULL, incl, o), vz = __shfl_up_sync(dev::FULL, incz, o);
            if (lane >= o) {
                incl += v;
                incz += vz;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            lo = min(lo, __shfl_xor_sync(dev::FULL, lo, o));
            hi = max(hi, __shfl_xor_sync(dev::FULL, hi, o));
        }
        int *wsum = flag, *wlo = flag + 10, *whi = flag + 20, *wnz = flag + 32;  // NWARP <= 10 warps
        if (lane == 31) {
            wsum[warp] = incl;
            wnz[warp] = incz;
        }
        if (lane == 0) {
            wlo[warp] = lo;
            whi[warp] = hi;
        }
        __syncthreads();
        if (warp == 0) {
            // All units the same length (and at least as many units as CTAs): if the unit
            // count has a divisor within 80% of the grid, work with that many CTAs, so that
            // every CTA gets whole units and nothing is merged.  Lanes test 32 candidates at
            // a time; the result goes to flag[30] (0: keep the grid).
            int glo = INT_MAX, ghi = -1;
            for (int w = 0; w < NWARP; ++w) {
                glo = min(glo, wlo[w]);
                ghi = max(ghi, whi[w]);
            }
            const int units = p.layers * p.B * HG, grid = (int)gridDim.x;
            int pick = 0;
            if (glo == ghi && glo > 0 && units >= grid) {
                for (int g0 = grid; pick == 0 && 5 * g0 >= 4 * grid; g0 -= 32) {
                    const int g2 = g0 - lane;
                    const bool okd = g2 > 0 && 5 * g2 >= 4 * grid && units % g2 == 0;
                    const unsigned m = __ballot_sync(dev::FULL, okd);
                    if (m) pick = g0 - (__ffs(m) - 1);       // the largest divisor found
                }
            }
            if (lane == 0) flag[30] = pick;
        }
        int base = 0, zbase = 0;
        for (int w = 0; w < warp; ++w) {
            base += wsum[w];
            zbase += wnz[w];
        }
        int acc = base + incl - run;                       // exclusive prefixes of b0
        int zacc = zbase + incz - nz;
        for (int b = b0; b < b1; ++b) {
            prefix[b] = acc;
            nzp[b] = zacc;
            const int L = lens[b];
            const bool ok = L >= 1 && L <= p.MB * BS;
            const int nb = ok ? (L + BS - 1) / BS - pre[b] : 0;
            acc += HG * nb;
            zacc += nb > 0;
        }
        if (tid == NTHR - 1) {
            prefix[p.B] = base + incl;
            nzp[p.B] = zbase + incz;
        }
        __syncthreads();
    }
    const int W1 = prefix[p.B];                            // tasks of one layer
    const long long W = (long long)W1 * p.layers;
    // With fewer tasks than CTAs only the first W CTAs take part.  A CTA whose share holds no
    // task leaves; the CTAs that cut a unit are exactly c0..c1 (no CTA inside a unit's run is
    // skipped).
    int G = (int)(W < (long long)gridDim.x ? W : (long long)gridDim.x);
    if (flag[30] > 0) G = flag[30];                        // whole units per CTA (see above)
    if (c >= G) return;                                    // uniform over the CTA
    Split sp;
    sp.prefix = prefix;
    sp.nzp = nzp;
    sp.B = p.B;
    sp.HG = HG;
    sp.OV = p.unit_cost;
    sp.G = G;
    sp.W1 = W1;
    sp.W = W;
    sp.C1 = W1 + (long long)p.unit_cost * nzp[p.B] * HG;
    sp.C = sp.C1 * p.layers;
    const long long s = sp.start(c), e = sp.start(c + 1);
    if (s >= e) return;                                    // uniform over the CTA

    auto unit_of = [&](long long r) { return unit_at(r, prefix, lens, pre, p.B, p.layers, W1, HG); };
    const int R = HP * group;                              // query rows of a unit
    const int qbytes = R * D * 2;
    const int qslot_bytes = align_up(qbytes, 128);
    float *ml_base = reinterpret_cast<float *>(smem + lay.ml);
    float *acc_base = reinterpret_cast<float *>(smem + lay.acc);
    const int rowstride = D + ACC_PAD;

    // The shared-prefix pass's state of query row `row` of unit u: returns (max, sum) and this
    // lane's DPL columns of num * out_scale.
    auto load_pref = [&](const Unit &u, int row, float (&pn)[D / 32]) {
        const int kvh = u.h * HP + row / group, r = row - (row / group) * group;
        const size_t pr = (((size_t)u.l * Hkv + kvh) * p.B + u.b) * group + r;
        if constexpr (D == 128) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.pref_o + pr * D) + lane);
            pn[0] = v.x; pn[1] = v.y; pn[2] = v.z; pn[3] = v.w;
        } else {
            const float2 v = __ldcg(reinterpret_cast<const float2 *>(p.pref_o + pr * D) + lane);
            pn[0] = v.x; pn[1] = v.y;
        }
        return __ldcg(reinterpret_cast<const float2 *>(p.pref_ml + pr * 2));
    };

    // The epilogue of segment k: merge the NW streaming warps' states (merge slot k&1), then
    // write the output of a whole unit, or this CTA's partial followed by the hand-off (the
    // last CTA of the unit to arrive merges every partial, in CTA order, and resets the
    // counter).  Run by the epilogue warp alone for all but the CTA's last segment, which the
    // team -- the streaming warps and the producer -- handles once streaming is over, while
    // the epilogue warp may still be finishing the segment before it (another merge slot).
    constexpr int TEAM = (NW + 1) * 32;                    // team threads (named barrier 1)
    auto seg_epilogue = [&](const Unit &u, long long seg_lo, long long seg_hi, int k, bool team_cta) {
        const long long U1 = u.U0 + u.nb;
        const int tw = warp < NW ? warp : NW;              // team warp index (the producer is NW)
        const int tt = team_cta ? tw * 32 + lane : lane;
        const int twarp = team_cta ? tw : 0, tnw = team_cta ? NW + 1 : 1;
        const float *ml_all = ml_base + (k & 1) * (lay.ml_slot / 4);
        const float *acc_all = acc_base + (k & 1) * (lay.acc_slot / 4);
        const bool whole = seg_lo == u.U0 && seg_hi == U1;
        const int slot = k == 0 ? 0 : 1;
        const size_t prow = ((size_t)c * 2 + slot) * R;            // partial rows of this CTA
        // a warp per output row (head j = row / group of the unit, query row r): the weights
        // 2^(m_w - M) of the stream warps that held head j, and the sum, once per row; then lane
        // l combines columns l*DPL .. l*DPL + DPL - 1 (vector accesses where the merge area
        // keeps columns in order)
        constexpr int DPL = D / 32;
        // one output row: pm, pn are the shared-prefix pass's state of the row (whole units)
        auto merge_row = [&](int row, const float2 pm, const float (&pn)[DPL]) {
            const int hj = row / group, r = row - hj * group;
            float mw[NSTREAM], M = -INFINITY;
#pragma unroll
            for (int q = 0; q < NSTREAM; ++q) {
                mw[q] = ml_all[(q * HP + hj) * 32 + r * 2];
                M = fmaxf(M, mw[q]);
            }
            float wt[NSTREAM], den = 0.f;
#pragma unroll
            for (int q = 0; q < NSTREAM; ++q) {
                wt[q] = (M == -INFINITY || mw[q] == -INFINITY) ? 0.f : dev::fast_exp2(mw[q] - M);
                den += wt[q] * ml_all[(q * HP + hj) * 32 + r * 2 + 1];
            }
            float num[DPL];
#pragma unroll
            for (int x = 0; x < DPL; ++x) num[x] = 0.f;
#pragma unroll
            for (int q = 0; q < NSTREAM; ++q) {
                const float *src = acc_all + ((q * HP + hj) * group + r) * rowstride;
                float a[DPL];
                if constexpr (Compute::IDENTITY_SLOTS && DPL == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(src + lane * 4);
                    a[0] = v.x; a[1] = v.y; a[2] = v.z; a[3] = v.w;
                } else if constexpr (Compute::IDENTITY_SLOTS && DPL == 2) {
                    const float2 v = *reinterpret_cast<const float2 *>(src + lane * 2);
                    a[0] = v.x; a[1] = v.y;
                } else {
#pragma unroll
                    for (int x = 0; x < DPL; ++x) a[x] = src[Compute::slot_of_d(lane * DPL + x)];
                }
#pragma unroll
                for (int x = 0; x < DPL; ++x) num[x] += wt[q] * a[x];
            }
            if (whole) {
                float o[DPL];
                if (u.pre > 0) {
                    // and the shared-prefix pass's state of this row
                    const float Mn = fmaxf(M, pm.x);
                    const float a = M == -INFINITY ? 0.f : dev::fast_exp2(M - Mn), bw = dev::fast_exp2(pm.x - Mn);
                    const float dd = den * a + pm.y * bw;
                    const float inv = dd > 0.f ? 1.f / dd : 0.f;
#pragma unroll
                    for (int x = 0; x < DPL; ++x) o[x] = (num[x] * p.out_scale * a + pn[x] * bw) * inv;
                } else {
                    const float inv = den > 0.f ? p.out_scale / den : 0.f;
#pragma unroll
                    for (int x = 0; x < DPL; ++x) o[x] = num[x] * inv;
                }
                uint16_t ob[DPL];
#pragma unroll
                for (int x = 0; x < DPL; ++x) {
                    const __nv_bfloat16 b = __float2bfloat16_rn(o[x]);
                    ob[x] = *reinterpret_cast<const uint16_t *>(&b);
                }
                uint16_t *dst = p.out + ((size_t)u.lb * p.Hq + (size_t)u.h * R + row) * D + lane * DPL;
                if constexpr (DPL == 4)
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(ob[0] | ((uint32_t)ob[1] << 16), ob[2] | ((uint32_t)ob[3] << 16));
                else
                    *reinterpret_cast<uint32_t *>(dst) = ob[0] | ((uint32_t)ob[1] << 16);
            } else {
                float *dst = p.part_o + (prow + row) * D + lane * DPL;
                if constexpr (DPL == 4)
                    *reinterpret_cast<float4 *>(dst) = make_float4(num[0] * p.out_scale, num[1] * p.out_scale,
                                                                   num[2] * p.out_scale, num[3] * p.out_scale);
                else
                    *reinterpret_cast<float2 *>(dst) = make_float2(num[0] * p.out_scale, num[1] * p.out_scale);
                if (lane == 0) {
                    p.part_ml[(prow + row) * 2] = M;
                    p.part_ml[(prow + row) * 2 + 1] = den;
                }
            }
        };
        constexpr int RB = 4;               // rows whose prefix-pass states are loaded together
        for (int row0 = twarp; row0 < R; row0 += RB * tnw) {
            float2 pmb[RB];
            float pnb[RB][DPL];
#pragma unroll
            for (int j = 0; j < RB; ++j) {
                pmb[j] = make_float2(-INFINITY, 0.f);
                const int row = row0 + j * tnw;
                if (whole && u.pre > 0 && row < R) pmb[j] = load_pref(u, row, pnb[j]);
            }
#pragma unroll
            for (int j = 0; j < RB; ++j)
                if (row0 + j * tnw < R) merge_row(row0 + j * tnw, pmb[j], pnb[j]);
        }
        if (whole) return;
        // hand-off.  The team barrier orders every partial store before the release-acquire
        // add of the team's first thread; the merge's loads follow that add through the next
        // team barrier.
        const int c0 = sp.owner(u.U0, u.l, u.b, u.h), c1 = sp.owner(U1 - 1, u.l, u.b, u.h);
        int *counter = p.counters + (size_t)u.lb * HG + u.h;
        int last;
        if (team_cta) {
            dev::named_bar_sync(1, TEAM);
            if (tt == 0) flag[31] = dev::atomic_add_acq_rel_gpu(counter, 1) == c1 - c0;
            dev::named_bar_sync(1, TEAM);
            last = flag[31];
        } else {
            __syncwarp();
            last = 0;
            if (lane == 0) last = dev::atomic_add_acq_rel_gpu(counter, 1) == c1 - c0;
            last = __shfl_sync(dev::FULL, last, 0);
            __syncwarp();
        }
        if (!last) return;
        // merge: a warp per RM output rows, lanes own D/32 columns; an online merge over the
        // partials in CTA order, four CTAs' partials of the RM rows in flight at a time.
        // The unit is c0's second or later segment when c0 also owns the task before it.
        bool c0_shared = false;
        if (u.U0 > 0) {
            const Unit v = unit_of(u.U0 - 1);
            c0_shared = sp.owner(u.U0 - 1, v.l, v.b, v.h) == c0;
        }
        constexpr int RM = 2;                     // rows merged together, their loads in flight at once
        for (int row0 = twarp; row0 < R; row0 += RM * tnw) {
            float pn[RM][DPL];                    // the shared-prefix pass's states, loaded first
            float2 pm[RM];
            float Mr[RM], den[RM], num[RM][DPL];
#pragma unroll
            for (int j = 0; j < RM; ++j) {
                const int row = row0 + j * tnw;
                pm[j] = make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int x = 0; x < DPL; ++x) pn[j][x] = num[j][x] = 0.f;
                if (u.pre > 0 && row < R) pm[j] = load_pref(u, row, pn[j]);
                Mr[j] = -INFINITY;
                den[j] = 0.f;
            }
            for (int cb = c0; cb <= c1; cb += 4) {
                float2 ml[RM][4];
                float oc[RM][4][DPL];
#pragma unroll
                for (int j = 0; j < RM; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int cc = cb + q, row = row0 + j * tnw;
                        ml[j][q] = make_float2(-INFINITY, 0.f);
#pragma unroll
                        for (int x = 0; x < DPL; ++x) oc[j][q][x] = 0.f;
                        if (cc <= c1 && row < R) {
                            const int sl = (cc == c0 && c0_shared) ? 1 : 0;
                            const size_t pr = ((size_t)cc * 2 + sl) * R + row;
                            ml[j][q] = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + pr * 2));
                            if constexpr (DPL == 4) {
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.part_o + pr * D) + lane);
                                oc[j][q][0] = v.x; oc[j][q][1] = v.y; oc[j][q][2] = v.z; oc[j][q][3] = v.w;
                            } else {
                                const float2 v = __ldcg(reinterpret_cast<const float2 *>(p.part_o + pr * D) + lane);
                                oc[j][q][0] = v.x; oc[j][q][1] = v.y;
                            }
                        }
                    }
#pragma unroll
                for (int j = 0; j < RM; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (ml[j][q].x == -INFINITY) continue;
                        const float Mn = fmaxf(Mr[j], ml[j][q].x);
                        const float a = Mr[j] == -INFINITY ? 0.f : dev::fast_exp2(Mr[j] - Mn);
                        const float bw = dev::fast_exp2(ml[j][q].x - Mn);
                        den[j] = den[j] * a + ml[j][q].y * bw;
#pragma unroll
                        for (int x = 0; x < DPL; ++x) num[j][x] = num[j][x] * a + oc[j][q][x] * bw;
                        Mr[j] = Mn;
                    }
            }
#pragma unroll
            for (int j = 0; j < RM; ++j) {
                const int row = row0 + j * tnw;
                if (row >= R) break;
                if (u.pre > 0) {                  // and the shared-prefix pass's state of this row
                    const float Mn = fmaxf(Mr[j], pm[j].x);
                    const float a = Mr[j] == -INFINITY ? 0.f : dev::fast_exp2(Mr[j] - Mn);
                    const float bw = dev::fast_exp2(pm[j].x - Mn);
                    den[j] = den[j] * a + pm[j].y * bw;
#pragma unroll
                    for (int x = 0; x < DPL; ++x) num[j][x] = num[j][x] * a + pn[j][x] * bw;
                }
                const float inv = den[j] > 0.f ? 1.f / den[j] : 0.f;
                uint16_t ob[DPL];
#pragma unroll
                for (int x = 0; x < DPL; ++x) {
                    const __nv_bfloat16 bv = __float2bfloat16_rn(num[j][x] * inv);
                    ob[x] = *reinterpret_cast<const uint16_t *>(&bv);
                }
                uint16_t *dst = p.out + ((size_t)u.lb * p.Hq + (size_t)u.h * R + row) * D + lane * DPL;
                if constexpr (DPL == 4)
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(ob[0] | ((uint32_t)ob[1] << 16), ob[2] | ((uint32_t)ob[3] << 16));
                else
                    *reinterpret_cast<uint32_t *>(dst) = ob[0] | ((uint32_t)ob[1] << 16);
            }
        }
        if (tt == 0) atomicExch(counter, 0);
    };

    if (warp == NW) {
        // ================= epilogue warp: q staging and every segment but the last ========
        auto issue_q = [&](long long seg_start, int k) {        // lane 0 only
            const Unit u = unit_of(seg_start);
            const uint32_t bar = qbar0 + 8 * (k & 1);
            dev::fence_proxy_async_smem();
            dev::mbar_arrive_expect_tx(bar, qbytes);
            dev::bulk_g2s(dev::smem_u32(smem + lay.q + (k & 1) * qslot_bytes),
                          p.q + ((size_t)u.lb * p.Hq + (size_t)u.h * R) * D, qbytes, bar);
        };
        long long nxt = s;                                        // first two segments' q rows
        for (int k = 0; k < 2 && nxt < e; ++k) {
            const Unit u = unit_of(nxt);
            if (lane == 0) issue_q(nxt, k);
            nxt = min(e, u.U0 + (long long)u.nb);
        }
        long long seg_lo = s;
        for (int k = 0; seg_lo < e; ++k) {
            const Unit u = unit_of(seg_lo);
            const long long seg_hi = min(e, u.U0 + (long long)u.nb);
            if (seg_hi == e) break;                               // the last segment: below
            // every streaming warp holds segment k's q rows in registers, so q slot k&1 takes
            // segment k+2's rows at once (two segments ahead of their use)
            if (!__all_sync(dev::FULL, dev::mbar_wait_bounded(qfree0 + 8 * (k & 1), (uint32_t)((k >> 1) & 1)))) {
                if (lane == 0) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
                break;
            }
            {
                const Unit u1 = unit_of(seg_hi);
                const long long h1 = min(e, u1.U0 + (long long)u1.nb);
                if (h1 < e && lane == 0) issue_q(h1, k + 2);
            }
            if (!__all_sync(dev::FULL, dev::mbar_wait_bounded(done0 + 8 * (k & 1), (uint32_t)((k >> 1) & 1)))) {
                if (lane == 0) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
                break;
            }
            seg_epilogue(u, seg_lo, seg_hi, k, false);
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(free0 + 8 * (k & 1)); // merge slot k&1 reusable
            seg_lo = seg_hi;
        }
    } else if (warp == NW + 1) {
        // ================= producer warp: every copy of the CTA's tasks ===================
        // Task i of the CTA (global task s + i) is loaded into stage i % NSTAGE and consumed
        // by the HP warps of stream i % NSTREAM.  The tasks go NSTREAM at a time: lane j issues
        // task i0 + j, so one warp-instruction issues the copies of a whole step, once each of
        // those stages has been released by its consumers.
        const int n_all = (int)(e - s);
        // index of the first tile ((layer * NB + phys) * Hkv + h*HP, or -1 if the table entry
        // is invalid) of task i, for a chunk of 32 tasks: lane x holds task chunk*32 + x; and,
        // when appending, (layer * B + b) * 16 + the new token's offset if task i is its
        // unit's last block
        // The lookup is split in two so that the table load is in flight for a whole chunk of
        // 32 tasks before its value is needed: fetch() issues it, finish() checks the entry.
        struct Pending { int id, tbase, app, valid; };
        auto fetch = [&](int chunk) {
            const int i = chunk * 32 + lane;
            Pending q{-1, 0, -1, 0};
            if (i < n_all) {
                const long long r = s + i;
                const Unit u = unit_of(r);
                const int blk = (int)(r - u.U0);
                q.id = __ldg(p.block_tables + (size_t)u.b * p.MB + u.pre + blk);
                q.tbase = u.l * p.num_blocks * Hkv + u.h * HP;
                if (p.k_new && blk == u.nb - 1) q.app = u.lb * BS + (u.L - 1) % BS;
                q.valid = 1;
            }
            return q;
        };
        auto finish = [&](const Pending &q, int &app) {
            int t = -1;
            app = -1;
            if (q.valid) {
                if (q.id >= 0 && q.id < p.num_blocks) {
                    t = q.tbase + q.id * Hkv;
                    app = q.app;
                } else {
                    dev::flag_error(p.err, PKV_DEVERR_BLOCK_ID);
                }
            }
            return t;
        };
        // the whole warp writes the new token's K/V row (a = (layer * B + b) * 16 + offset)
        // into tile t's slot
        auto write_row = [&](int a, int t) {
            const int lb = a / BS, off = a % BS, h = t % Hkv;
            const size_t src = ((size_t)lb * Hkv + h) * D;
            const size_t dst = ((size_t)t * BS + off) * D;               // element index
            constexpr int EPL = D / 32;
            if constexpr (FP8) {
                const uint16_t *ks = p.k_new + src + lane * EPL;
                const uint16_t *vs = p.v_new + src + lane * EPL;
                uint32_t kc = 0, vc = 0;
#pragma unroll
                for (int x = 0; x < EPL; x += 2) {
                    const uint32_t kw = *reinterpret_cast<const uint32_t *>(ks + x);
                    const uint32_t vw = *reinterpret_cast<const uint32_t *>(vs + x);
                    kc |= dev::e4m3x2_satfinite(dev::bf16_lo(kw) * p.inv_k_scale, dev::bf16_hi(kw) * p.inv_k_scale) << (8 * x);
                    vc |= dev::e4m3x2_satfinite(dev::bf16_lo(vw) * p.inv_v_scale, dev::bf16_hi(vw) * p.inv_v_scale) << (8 * x);
                }
                uint8_t *kd = const_cast<uint8_t *>(p.key_cache) + dst + lane * EPL;
                uint8_t *vd = const_cast<uint8_t *>(p.value_cache) + dst + lane * EPL;
                if constexpr (EPL == 4) {
                    *reinterpret_cast<uint32_t *>(kd) = kc;
                    *reinterpret_cast<uint32_t *>(vd) = vc;
                } else {
                    *reinterpret_cast<uint16_t *>(kd) = (uint16_t)kc;
                    *reinterpret_cast<uint16_t *>(vd) = (uint16_t)vc;
                }
            } else {
                uint16_t *kd = reinterpret_cast<uint16_t *>(const_cast<uint8_t *>(p.key_cache)) + dst + lane * EPL;
                uint16_t *vd = reinterpret_cast<uint16_t *>(const_cast<uint8_t *>(p.value_cache)) + dst + lane * EPL;
                if constexpr (EPL == 4) {
                    *reinterpret_cast<uint2 *>(kd) = *reinterpret_cast<const uint2 *>(p.k_new + src + lane * EPL);
                    *reinterpret_cast<uint2 *>(vd) = *reinterpret_cast<const uint2 *>(p.v_new + src + lane * EPL);
                } else {
                    *reinterpret_cast<uint32_t *>(kd) = *reinterpret_cast<const uint32_t *>(p.k_new + src + lane * EPL);
                    *reinterpret_cast<uint32_t *>(vd) = *reinterpret_cast<const uint32_t *>(p.v_new + src + lane * EPL);
                }
            }
        };
        const Pending first = fetch(0);
        Pending pend = fetch(1);                          // both chunks' loads in flight
        int acur;
        int tcur = finish(first, acur);
        bool ok = true;
        int issued = 0;                                   // tasks whose copies are issued
        for (int i0 = 0; i0 < n_all; i0 += NSTREAM) {
            if ((i0 & 31) == 0 && i0 > 0) {
                tcur = finish(pend, acur);                // loaded a chunk ago
                pend = fetch((i0 >> 5) + 1);
            }
            const int i = i0 + lane % NSTREAM;
            const int t = __shfl_sync(dev::FULL, tcur, i & 31);
            const int a = __shfl_sync(dev::FULL, acur, i & 31);
            const bool mine = lane < NSTREAM && i < n_all;
            const int st = i % NSTAGE;
            // the stage's previous task has been consumed
            const bool freed = !mine || i < NSTAGE ||
                               dev::mbar_wait_bounded(empty0 + 8 * st, (uint32_t)(((i / NSTAGE) - 1) & 1));
            if (!__all_sync(dev::FULL, freed)) {
                ok = false;
                break;
            }
            // blocks holding a new token: write each K/V row into its slot first, then order
            // those generic writes before the copies that read the block
            unsigned am = __ballot_sync(dev::FULL, mine && a >= 0);
            if (am) {
                while (am) {
                    const int from = __ffs(am) - 1;
                    am &= am - 1;
                    const int aa = __shfl_sync(dev::FULL, a, from), tt0 = __shfl_sync(dev::FULL, t, from);
#pragma unroll
                    for (int j = 0; j < HP; ++j) write_row(aa, tt0 + j);
                }
                dev::fence_proxy_async_global();
                __syncwarp();
            }
            if (mine) {
                const uint32_t bar = full0 + 8 * st;
                stage_tile[st] = t;
                if (t >= 0) {
                    dev::mbar_arrive_expect_tx(bar, STAGE);
                    const uint32_t dk = dev::smem_u32(smem + lay.stage + st * STAGE);
                    if constexpr (Compute::SWIZZLED) {
                        // one tensor copy of HP tiles each, [head][segment][16 tokens][SEG
                        // bytes], swizzled (two row segments: a 4-D map whose third
                        // dimension is the segment)
                        if constexpr (NSEG == 2) {
                            tc::tma_load_4d(dk, kmap, 0, 0, 0, t, bar);
                            tc::tma_load_4d(dk + HP * TILE, vmap, 0, 0, 0, t, bar);
                        } else {
                            static_assert(NSEG == 1, "row segments");
                            tc::tma_load_3d(dk, kmap, 0, 0, t, bar);
                            tc::tma_load_3d(dk + HP * TILE, vmap, 0, 0, t, bar);
                        }
                    } else {
                        const size_t off = (size_t)t * TILE;
                        dev::bulk_g2s(dk, p.key_cache + off, HP * TILE, bar);
                        dev::bulk_g2s(dk + HP * TILE, p.value_cache + off, HP * TILE, bar);
                    }
                } else {
                    dev::mbar_arrive(bar);                // nothing to copy; the block is masked
                }
            }
            issued = min(n_all, i0 + NSTREAM);
        }
        if (!ok && lane == 0) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
        // no copy may land after the CTA has left: wait (bounded) for the last task issued
        // into each stage (at once if its consumer already has)
        if (lane < NSTAGE && lane < issued) {
            const int last = lane + (issued - 1 - lane) / NSTAGE * NSTAGE;
            (void)dev::mbar_wait_bounded(full0 + 8 * lane, (uint32_t)((last / NSTAGE) & 1));
        }
    } else {
        // ================= consumer warps: head hj of tasks sw, sw + NSTREAM, ... ========
        const int sw = warp / HP, hj = warp - sw * HP;
        const int n_all = (int)(e - s);
        const int n_mine = max(0, (n_all - sw + NSTREAM - 1) / NSTREAM);
        bool aborted = false;
        if (p.test_stall)          // the failure-path test: a wait that runs out (copies in flight)
            aborted = !__all_sync(dev::FULL, dev::mbar_wait_bounded_ns(never, 0, dev::TEST_EXPIRE_NS));
        int ic = 0;
        int k = 0;
        for (long long seg_lo = s; seg_lo < e; ++k) {
            const Unit u = unit_of(seg_lo);
            const long long seg_hi = min(e, u.U0 + (long long)u.nb);
            const bool qok = __all_sync(dev::FULL, dev::mbar_wait_bounded(qbar0 + 8 * (k & 1), (uint32_t)((k >> 1) & 1)));
            aborted |= !qok;
            cmp.start(reinterpret_cast<const uint16_t *>(smem + lay.q + (k & 1) * qslot_bytes) + hj * group * D,
                      group, lane);
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(qfree0 + 8 * (k & 1));   // q slot k&1 read
            while (!aborted && ic < n_mine && s + sw + (long long)NSTREAM * ic < seg_hi) {
                const int i = sw + NSTREAM * ic;
                const int st = i % NSTAGE;
                if (!__all_sync(dev::FULL, dev::mbar_wait_bounded(full0 + 8 * st, (uint32_t)((i / NSTAGE) & 1)))) {
                    aborted = true;
                    break;
                }
                const int blk = (int)(s + i - u.U0) + u.pre;
                const int ntok = stage_tile[st] >= 0 ? min(BS, u.L - blk * BS) : 0;
                if (ntok > 0) {
                    const uint8_t *stage = smem + lay.stage + st * STAGE + hj * TILE;
                    cmp.block(stage, stage + HP * TILE, ntok, p.score_scale, lane);
                }
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(empty0 + 8 * st);   // this head of the stage is done
                ++ic;
            }
            // hand this segment's state to the epilogue (merge slot k&1, free once the
            // epilogue warp has merged segment k-2 out of it)
            if (k >= 2 && !__all_sync(dev::FULL, dev::mbar_wait_bounded(free0 + 8 * (k & 1), (uint32_t)(((k >> 1) - 1) & 1))))
                aborted = true;
            cmp.dump(ml_base + (k & 1) * (lay.ml_slot / 4) + warp * 32,
                     acc_base + (k & 1) * (lay.acc_slot / 4) + warp * group * rowstride, group, lane);
            if (seg_hi < e) dev::mbar_arrive(done0 + 8 * (k & 1));
            seg_lo = seg_hi;
        }
        // a wait gave up: report it (the producer waits for every copy it issued)
        if (aborted && lane == 0) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
    }

    // ---- 5. the CTA's last segment, by the team (every warp but the epilogue warp, which
    //         leaves once it has handled its segments)
    if (warp == NW) return;
    dev::named_bar_sync(1, TEAM);
    {
        long long seg_lo = s;
        int k = 0;
        Unit u = unit_of(seg_lo);
        while (min(e, u.U0 + (long long)u.nb) < e) {
            seg_lo = u.U0 + u.nb;
            u = unit_of(seg_lo);
            ++k;
        }
        seg_epilogue(u, seg_lo, e, k, true);
    }
}

// Register budget for two CTAs of NW + 2 warps per SM (the shared-memory ring allows no
// more with NW = 4).
template <int D, bool FP8, int NW, int NS, bool G16>
__global__ void __launch_bounds__((NW + 2) * 32, 8 / NW) decode_mma_kernel(const DecodeParams p)
{
    MmaCompute<D, FP8, G16> cmp;
    decode_body<D, FP8, NW, NS, 1>(p, cmp, nullptr, nullptr);
}

template <int D, bool FP8, int NW, int NS, int HP, int NH>
__global__ void __launch_bounds__((NW + 2) * 32, 8 / NW)
decode_tok_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p)
{
    TokCompute<D, FP8, NH> cmp;
    cmp.setup(threadIdx.x & 31);
    cmp.base_sc = p.score_scale;
    decode_body<D, FP8, NW, NS, HP>(p, cmp, &kmap, &vmap);
}

// ------------------------------------------------------------------------------------
// Shared-prefix pass.  Blocks that many sequences' tables share (a common prompt prefix stored
// once and referenced by every table, "KV Cache 与推理优化", PagedAttention section) are read
// once per KV head and up to 64 query rows -- all g query heads of up to 64 / g sequences --
// instead of once per sequence.  The reference table is the longest sequence's (the smallest
// index among equals).  Sequence b's covered blocks are the leading entries of its table,
// at most shared_prefix of them and never the block that receives an appended token, that
// equal the reference's, so any tables give the same result.  Each covered query row's
// partial softmax state (max, sum, unnormalised output) over its covered positions goes to
// the workspace -- or, for a sequence covered entirely, its output -- and the decode kernel
// streams the remaining blocks and merges the two.
// ------------------------------------------------------------------------------------
constexpr int PRE_ROWS = 64;        // query rows per CTA: 4 consumer warps of 16
constexpr int PRE_NST = 4;          // K/V ring stages
constexpr int PRE_THREADS = 160;    // 4 consumer warps and the producer warp

template <int D, bool FP8>
struct PrefixSmem {
    static constexpr int TILE = BS * D * (FP8 ? 1 : 2);
    static constexpr int RING = 0;                          // PRE_NST x (K, V), 1024-aligned
    static constexpr int Q = RING + PRE_NST * 2 * TILE;     // [64 rows][D] bf16
    static constexpr int SEQ = Q + PRE_ROWS * D * 2;        // [64 sequences] (length, covered blocks)
    static constexpr int TOK = SEQ + PRE_ROWS * 2 * 4;      // [PRE_NST] the stage holds a loaded tile
    static constexpr int RED = TOK + PRE_NST * 4;           // reduction scratch
    static constexpr int BAR = align_up(RED + 16 * 8, 8);   // full and empty mbarriers
    static constexpr int TOTAL = BAR + 2 * PRE_NST * 8;
    static constexpr int ALLOC = TOTAL + 1024;              // + alignment slack
};

template <int D, bool FP8>
__global__ void __launch_bounds__(PRE_THREADS)
decode_prefix_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const DecodeParams p)
{
    using SM = PrefixSmem<D, FP8>;
    constexpr int ELEM = FP8 ? 1 : 2;
    constexpr int TILE = SM::TILE;
    constexpr int SEG = D * ELEM < 128 ? D * ELEM : 128;
    constexpr int NSEG = D * ELEM / SEG;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = p.group, spc = PRE_ROWS / g;              // sequences per CTA
    const int b0 = blockIdx.x * spc, h = blockIdx.y, l = blockIdx.z;
    int32_t *seq = reinterpret_cast<int32_t *>(smem + SM::SEQ);
    int32_t *tok_ok = reinterpret_cast<int32_t *>(smem + SM::TOK);
    unsigned long long *red = reinterpret_cast<unsigned long long *>(smem + SM::RED);
    const uint32_t full0 = dev::smem_u32(smem + SM::BAR), empty0 = full0 + 8 * PRE_NST;
    if (tid == 0)
        for (int st = 0; st < PRE_NST; ++st) {
            dev::mbar_init(full0 + 8 * st, 1);
            dev::mbar_init(empty0 + 8 * st, 4);         // the four consumer warps
        }
    dev::fence_barrier_init();

    // ---- 1. the reference: the longest valid sequence, the smallest index among equals
    unsigned long long key = 0;                           // length << 32 | (~index)
    for (int b = tid; b < p.B; b += PRE_THREADS) {
        const int L = __ldg(p.seq_lens + b);
        if (L >= 1 && L <= p.MB * BS) {
            const unsigned long long k = ((unsigned long long)L << 32) | (0xffffffffu - (unsigned)b);
            key = k > key ? k : key;
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long k = __shfl_xor_sync(dev::FULL, key, o);
        key = k > key ? k : key;
    }
    if (lane == 0) red[warp] = key;
    __syncthreads();
    if (tid == 0) {
        unsigned long long k = 0;
        for (int w = 0; w < PRE_THREADS / 32; ++w) k = red[w] > k ? red[w] : k;
        red[8] = k;
    }
    __syncthreads();
    const unsigned long long best = red[8];
    const int Lref = (int)(best >> 32);
    const int bref = best ? (int)(0xffffffffu - (unsigned)(best & 0xffffffffu)) : -1;
    const int spe = bref >= 0 ? min(p.shared_prefix, (Lref + BS - 1) / BS) : 0;

    // ---- 2. blocks covered for each of this CTA's sequences (written once, by the CTAs of
    //         KV head 0 of layer 0, for the decode kernel)
    for (int sq = warp; sq < spc; sq += PRE_THREADS / 32) {
        const int b = b0 + sq;
        int L = 0, cov = 0;
        if (b < p.B) {
            L = __ldg(p.seq_lens + b);
            if (L >= 1 && L <= p.MB * BS && spe > 0) {
                const int nb = (L + BS - 1) / BS;
                int lim = min(spe, nb);
                if (p.k_new) lim = min(lim, nb - 1);    // the block that receives the new token
                cov = lim;
                for (int j0 = 0; j0 < lim; j0 += 32) {
                    const int j = j0 + lane;
                    const bool diff = j < lim && __ldg(p.block_tables + (size_t)b * p.MB + j) !=
                                                     __ldg(p.block_tables + (size_t)bref * p.MB + j);
                    const unsigned m = __ballot_sync(dev::FULL, diff);
                    if (m) {
                        cov = j0 + __ffs(m) - 1;
                        break;
                    }
                }
            }
            if (lane == 0 && h == 0 && l == 0) p.prefix_n[b] = cov;
        }
        if (lane == 0) {
            seq[2 * sq] = L;
            seq[2 * sq + 1] = cov;
        }
    }
    __syncthreads();
    int spc_blocks = 0;                                   // blocks this CTA streams
    for (int sq = 0; sq < spc; ++sq) spc_blocks = max(spc_blocks, seq[2 * sq + 1]);
    if (spc_blocks == 0) return;                          // uniform over the CTA

    if (warp == 4) {
        // ================= producer: the reference's first spc_blocks blocks of head h
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            for (int j = 0; j < spc_blocks; ++j) {
                const int st = j % PRE_NST;
                if (j >= PRE_NST && !dev::mbar_wait_bounded(empty0 + 8 * st, (uint32_t)(((j / PRE_NST) - 1) & 1))) {
                    ok = false;
                    break;
                }
                const int id = __ldg(p.block_tables + (size_t)bref * p.MB + j);
                const uint32_t bar = full0 + 8 * st;
                if (id >= 0 && id < p.num_blocks) {
                    tok_ok[st] = 1;
                    const int t = (l * p.num_blocks + id) * p.Hkv + h;
                    const uint32_t dk = dev::smem_u32(smem + SM::RING + st * 2 * TILE);
                    dev::mbar_arrive_expect_tx(bar, 2 * TILE);
                    if constexpr (NSEG == 2) {
                        tc::tma_load_4d(dk, &kmap, 0, 0, 0, t, bar);
                        tc::tma_load_4d(dk + TILE, &vmap, 0, 0, 0, t, bar);
                    } else {
                        tc::tma_load_3d(dk, &kmap, 0, 0, t, bar);
                        tc::tma_load_3d(dk + TILE, &vmap, 0, 0, t, bar);
                    }
                } else {
                    dev::flag_error(p.err, PKV_DEVERR_BLOCK_ID);
                    tok_ok[st] = 0;
                    dev::mbar_arrive(bar);
                }
                issued = j + 1;
            }
            if (!ok) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
            // no copy may land after the CTA has left
            for (int st = 0; st < PRE_NST && st < issued; ++st) {
                const int last = st + (issued - 1 - st) / PRE_NST * PRE_NST;
                (void)dev::mbar_wait_bounded(full0 + 8 * st, (uint32_t)((last / PRE_NST) & 1));
            }
        }
        return;
    }

    // ================= consumers: warp w holds query rows 16w .. 16w + 15 of the CTA
    // (row x: sequence b0 + x / g, query head h*g + x % g); rows of sequences with nothing
    // covered, and padding rows, are zero and written nowhere.
    uint16_t *qs = reinterpret_cast<uint16_t *>(smem + SM::Q) + warp * 16 * D;
    for (int e = lane; e < 16 * D / 8; e += 32) {
        const int i = e / (D / 8), c8 = e % (D / 8);
        const int x = 16 * warp + i, sq = x / g;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (sq < spc && seq[2 * sq + 1] > 0)
            v = *reinterpret_cast<const uint4 *>(p.q + (((size_t)l * p.B + b0 + sq) * p.Hq + (size_t)h * g + x % g) * D + c8 * 8);
        *reinterpret_cast<uint4 *>(qs + i * D + c8 * 8) = v;
    }
    __syncwarp();
    TokCompute<D, FP8, 2> cmp;
    cmp.setup(lane);
    cmp.base_sc = p.score_scale;
    cmp.start(qs, 16, lane);
    const int gid = lane >> 2, tid4 = lane & 3;
#pragma unroll
    for (int jn = 0; jn < 2; ++jn)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int x = 16 * warp + 8 * jn + 2 * tid4 + c, sq = x / g;
            const bool row = sq < spc && seq[2 * sq + 1] > 0;
            cmp.lim[jn][c] = row ? min(seq[2 * sq], BS * seq[2 * sq + 1]) : BS * spc_blocks;
        }
    bool ok = true;
    for (int j = 0; j < spc_blocks; ++j) {
        const int st = j % PRE_NST;
        if (!__all_sync(dev::FULL, dev::mbar_wait_bounded(full0 + 8 * st, (uint32_t)((j / PRE_NST) & 1)))) {
            ok = false;
            break;
        }
        const int ntok = min(BS, Lref - BS * j);          // positions the reference holds
        if (tok_ok[st]) {
            const uint32_t kt = dev::smem_u32(smem + SM::RING + st * 2 * TILE);
            if (ntok == BS) cmp.template block_impl<false, true>(kt, kt + TILE, BS, lane, BS * j);
            else cmp.template block_impl<true, true>(kt, kt + TILE, ntok, lane, BS * j);
        }
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(empty0 + 8 * st);
    }
    if (!ok) {
        if (lane == 0) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
        return;
    }
    // ---- each covered row: its partial state, or the output of a sequence covered entirely
#pragma unroll
    for (int jn = 0; jn < 2; ++jn)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float x = cmp.l[jn][r];
            x += __shfl_xor_sync(dev::FULL, x, 4);
            x += __shfl_xor_sync(dev::FULL, x, 8);
            x += __shfl_xor_sync(dev::FULL, x, 16);
            cmp.l[jn][r] = x;
        }
#pragma unroll
    for (int jn = 0; jn < 2; ++jn)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int x = 16 * warp + 8 * jn + 2 * tid4 + c, sq = x / g;
            if (sq >= spc || seq[2 * sq + 1] == 0) continue;
            const int b = b0 + sq, r = x % g, L = seq[2 * sq];
            const bool entire = !p.k_new && seq[2 * sq + 1] == (L + BS - 1) / BS;
            const size_t pr = (((size_t)l * p.Hkv + h) * p.B + b) * g + r;
            const float lsum = cmp.l[jn][c];
            if (entire) {
                uint16_t *dst = p.out + (((size_t)l * p.B + b) * p.Hq + (size_t)h * g + r) * D;
                const float inv = lsum > 0.f ? p.out_scale / lsum : 0.f;
#pragma unroll
                for (int mt = 0; mt < TokCompute<D, FP8, 2>::MT; ++mt) {
                    const __nv_bfloat16 v0 = __float2bfloat16_rn(cmp.acc[mt][jn][c] * inv);
                    const __nv_bfloat16 v1 = __float2bfloat16_rn(cmp.acc[mt][jn][c + 2] * inv);
                    dst[TokCompute<D, FP8, 2>::dcol(mt, gid)] = *reinterpret_cast<const uint16_t *>(&v0);
                    dst[TokCompute<D, FP8, 2>::dcol(mt, gid + 8)] = *reinterpret_cast<const uint16_t *>(&v1);
                }
            } else {
                float *dst = p.pref_o + pr * D;
#pragma unroll
                for (int mt = 0; mt < TokCompute<D, FP8, 2>::MT; ++mt) {
                    dst[TokCompute<D, FP8, 2>::dcol(mt, gid)] = cmp.acc[mt][jn][c] * p.out_scale;
                    dst[TokCompute<D, FP8, 2>::dcol(mt, gid + 8)] = cmp.acc[mt][jn][c + 2] * p.out_scale;
                }
                if (gid == 0) *reinterpret_cast<float2 *>(p.pref_ml + pr * 2) = make_float2(cmp.m[jn][c], lsum);
            }
        }
}

template <int D, bool FP8, int NW, int NS, int GP>
__global__ void __launch_bounds__((NW + 2) * 32) decode_simt_kernel(const DecodeParams p)
{
    SimtCompute<D, FP8, GP> cmp;
    cmp.sscale = p.score_scale;
    decode_body<D, FP8, NW, NS, 1>(p, cmp, nullptr, nullptr);
}

// ------------------------------------------------------------------------------------
// Launch plan and per-instantiation launchers.
// ------------------------------------------------------------------------------------
// Everything a launch needs: the parameters and, for variant 3, the K and V tensor maps.
struct LaunchArgs {
    DecodeParams p;
    CUtensorMap kmap, vmap;
};

struct Plan {
    int variant, nw, ns;
    int hp;                   // KV heads per task (one copy of hp tiles); variant 3 only
    int sp;                   // blocks the shared-prefix pass may cover (0: no pass)
    int uc;                   // tasks the split charges each unit besides its blocks
    size_t ws_pre_n, ws_pre_o, ws_pre_ml;   // its areas of the workspace
    int grid;                 // CTAs (one wave)
    size_t smem;              // dynamic shared memory per CTA
    size_t ws_counters, ws_o, ws_ml, ws_bytes;
};

template <class K>
cudaError_t prepare(K kernel, size_t smem, int threads, int *per_sm)
{
    // Once per (kernel, device): allow the device's full opt-in shared memory, so that no
    // later call can lower the limit below a size that an earlier call relies on.  Once per
    // (kernel, device, size): the occupancy, cached for the plan.
    struct Entry { const void *fn; int dev; size_t smem; int per_sm; };
    static std::mutex mu;
    static Entry seen[1024];
    static int nseen = 0;
    static const void *opted_fn[256];
    static int opted_dev[256];
    static int nopted = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> g(mu);
    bool opted = false;
    for (int i = 0; i < nopted; ++i)
        if (opted_fn[i] == (const void *)kernel && opted_dev[i] == dev) opted = true;
    if (!opted) {
        int limit = 0;
        cudaError_t e = cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
        if (e != cudaSuccess) return e;
        if (nopted < 256) {
            opted_fn[nopted] = (const void *)kernel;
            opted_dev[nopted] = dev;
            ++nopted;
        }
    }
    if (!per_sm) return cudaSuccess;
    for (int i = 0; i < nseen; ++i)
        if (seen[i].fn == (const void *)kernel && seen[i].dev == dev && seen[i].smem == smem) {
            *per_sm = seen[i].per_sm;
            return cudaSuccess;
        }
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
    if (e != cudaSuccess) return e;
    if (nseen < 1024) seen[nseen++] = Entry{(const void *)kernel, dev, smem, n};
    *per_sm = n;
    return cudaSuccess;
}

// Either report CTAs per SM (launch == false) or launch.
template <int D, bool FP8, int NW, int NS>
cudaError_t run_decode(const Plan &pl, int group, bool launch, int *per_sm, cudaStream_t s,
                       const LaunchArgs *a)
{
    const int threads = (NW + 2) * 32;                   // + the epilogue and producer warps
    auto go = [&](auto kernel) -> cudaError_t {
        cudaError_t e = prepare(kernel, pl.smem, threads, launch ? nullptr : per_sm);
        if (e != cudaSuccess || !launch) return e;
        kernel<<<pl.grid, threads, pl.smem, s>>>(a->p);
        return cudaGetLastError();
    };
    if (pl.variant == 3) {
        auto go_tok = [&](auto kernel) -> cudaError_t {
            cudaError_t e = prepare(kernel, pl.smem, threads, launch ? nullptr : per_sm);
            if (e != cudaSuccess || !launch) return e;
            kernel<<<pl.grid, threads, pl.smem, s>>>(a->kmap, a->vmap, a->p);
            return cudaGetLastError();
        };
        auto by_nh = [&](auto hpc) -> cudaError_t {
            constexpr int H = decltype(hpc)::value;
            if (group > 8) return go_tok(decode_tok_kernel<D, FP8, NW, NS, H, 2>);
            return go_tok(decode_tok_kernel<D, FP8, NW, NS, H, 1>);
        };
        if (pl.hp == 1) return by_nh(std::integral_constant<int, 1>{});
        if (pl.hp == 2) return by_nh(std::integral_constant<int, 2>{});
        if (pl.hp == 4) return by_nh(std::integral_constant<int, 4>{});
        return cudaErrorInvalidConfiguration;
    }
    if (pl.variant == 2) {
        if (group > 8) return go(decode_mma_kernel<D, FP8, NW, NS, true>);
        return go(decode_mma_kernel<D, FP8, NW, NS, false>);
    }
    if constexpr (NW == 4 && NS == 2) {
        if (group <= 1) return go(decode_simt_kernel<D, FP8, NW, NS, 1>);
        if (group <= 2) return go(decode_simt_kernel<D, FP8, NW, NS, 2>);
        if (group <= 4) return go(decode_simt_kernel<D, FP8, NW, NS, 4>);
        return go(decode_simt_kernel<D, FP8, NW, NS, 8>);
    }
    return cudaErrorInvalidConfiguration;
}

// The shared-prefix pass: grid (sequence groups, KV heads, layers); launched before the decode
// on the same stream.
template <int D, bool FP8>
cudaError_t run_prefix(const LaunchArgs *a, cudaStream_t s)
{
    auto kernel = decode_prefix_kernel<D, FP8>;
    const size_t smem = PrefixSmem<D, FP8>::ALLOC;
    cudaError_t e = prepare(kernel, smem, PRE_THREADS, nullptr);
    if (e != cudaSuccess) return e;
    const int spc = PRE_ROWS / a->p.group;
    const dim3 grid((unsigned)((a->p.B + spc - 1) / spc), (unsigned)a->p.Hkv, (unsigned)a->p.layers);
    kernel<<<grid, PRE_THREADS, smem, s>>>(a->kmap, a->vmap, a->p);
    return cudaGetLastError();
}

// (warps per CTA, stages per warp) pairs that are compiled.  The CUDA-core variant exists
// for comparison only and is compiled for one pair.
template <int D, bool FP8>
cudaError_t dispatch_nw_ns(const Plan &pl, int group, bool launch, int *per_sm, cudaStream_t s,
                           const LaunchArgs *a)
{
    if (pl.variant == 1 && !(pl.nw == 4 && pl.ns == 2)) return cudaErrorInvalidConfiguration;
    if (pl.nw == 4 && pl.ns == 2) return run_decode<D, FP8, 4, 2>(pl, group, launch, per_sm, s, a);
    if (pl.nw == 4 && pl.ns == 3) return run_decode<D, FP8, 4, 3>(pl, group, launch, per_sm, s, a);
    if (pl.nw == 4 && pl.ns == 4) return run_decode<D, FP8, 4, 4>(pl, group, launch, per_sm, s, a);
    if (pl.nw == 8 && pl.ns == 2) return run_decode<D, FP8, 8, 2>(pl, group, launch, per_sm, s, a);
    if (pl.nw == 8 && pl.ns == 3) return run_decode<D, FP8, 8, 3>(pl, group, launch, per_sm, s, a);
    return cudaErrorInvalidConfiguration;
}

}  // namespace decode
}  // namespace pkv
