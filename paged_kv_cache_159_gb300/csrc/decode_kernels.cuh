// paged_decode.cu -- single-query (decode) GQA attention over the paged KV pool, plus the
// split-KV combine kernel.
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
//   * One CTA per (sequence, KV head, partition of logical blocks).  All g query heads of
//     the group are computed from one read of each K/V tile, so every K/V byte crosses HBM
//     once per step.
//   * Each (block, head) tile of K or V is contiguous (16 x head_dim elements: 4 KiB bf16 at
//     head_dim 128), so it is staged by one 1-D bulk (TMA) copy into shared memory.  Every
//     warp owns a ring of `NS` stages (K and V tile each) with one mbarrier per stage and
//     streams the blocks j = first + warp, first + warp + NW, ...; no CTA-wide barrier sits in
//     the loop.  Waits are bounded (about 1 s) and report PKV_DEVERR_TIMEOUT.
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
//   * Partitions: a sequence longer than one partition writes (max, sum, unnormalised
//     output) per partition to the workspace and `combine_kernel` merges them; the merge
//     order and every partition boundary depend only on logical positions, so any physical
//     placement of the blocks gives bit-identical results.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace decode {

constexpr int BS = 16;                    // tokens per block
constexpr int PB_MAX = 1024;              // table entries one CTA may stage
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_TAU = 8.0f;       // raise the running max only beyond 2^8

struct DecodeParams {
    const uint16_t *q;            // bf16 [B, Hq, D]
    const uint8_t *key_cache;     // [NB, Hkv, 16, D] of bf16 or e4m3
    const uint8_t *value_cache;
    const int32_t *block_tables;  // [B, MB]
    const int32_t *seq_lens;      // [B]
    uint16_t *out;                // bf16 [B, Hq, D]
    float *part_o;                // [B, Hq, P, D]   unnormalised partial outputs
    float *part_ml;               // [B, Hq, P, 2]   (running max in log2 units, sum)
    uint32_t *err;
    int B, Hq, Hkv, group, MB, P, PB, num_blocks;
    float score_scale;            // scale * k_scale * log2(e)
    float out_scale;              // v_scale (1 for bf16 pools)
};

__device__ __forceinline__ float warp_allreduce_sum(float x)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(dev::FULL, x, o);
    return x;
}

// ------------------------------------------------------------------------------------
// Shared-memory plan of one CTA:
//   [stage area: NW * NS * 2 * TILE bytes, reused as the merge area after the loop]
//   [table: PB_MAX int32] [barriers: NW * NS * 8 bytes]
// ------------------------------------------------------------------------------------
template <int D, bool FP8, int NW, int NS>
struct Smem {
    static constexpr int ELEM = FP8 ? 1 : 2;
    static constexpr int ROW = D * ELEM;                  // bytes of one token row
    static constexpr int TILE = BS * ROW;                 // one (block, head) tile of K or V
    static constexpr int STAGE = 2 * TILE;
    static constexpr int STAGE_AREA = NW * NS * STAGE;
    static constexpr int MERGE_AREA = NW * (16 * D * 4 + 2 * 16 * 4);
    static constexpr int AREA = STAGE_AREA > MERGE_AREA ? STAGE_AREA : MERGE_AREA;
    static constexpr int TABLE_OFF = AREA;
    static constexpr int BAR_OFF = TABLE_OFF + PB_MAX * 4;
    static constexpr int BYTES = BAR_OFF + NW * NS * 8;
};

// Issue the copies of this warp's i-th block into stage s (lane 0 only).
template <int D, bool FP8, int NW, int NS>
__device__ __forceinline__ void issue_block(const DecodeParams &p, int h, uint8_t *smem,
                                            const int32_t *tbl, int warp, int i)
{
    using S = Smem<D, FP8, NW, NS>;
    const int s = i % NS;
    const int local = warp + NW * i;                    // index within the partition
    const int phys = tbl[local];
    uint8_t *stage = smem + (warp * NS + s) * S::STAGE;
    const uint32_t bar = dev::smem_u32(smem + S::BAR_OFF + (warp * NS + s) * 8);
    if (phys >= 0) {
        const size_t off = ((size_t)phys * p.Hkv + h) * S::TILE;
        dev::mbar_arrive_expect_tx(bar, 2 * S::TILE);
        dev::bulk_g2s(dev::smem_u32(stage), p.key_cache + off, S::TILE, bar);
        dev::bulk_g2s(dev::smem_u32(stage + S::TILE), p.value_cache + off, S::TILE, bar);
    } else {
        dev::mbar_arrive(bar);                          // nothing to copy; block is masked
    }
}

// ------------------------------------------------------------------------------------
// Tensor-core compute (variant 2).  Lane l: gid = l/4 (mma row group), tid = l%4.
// ------------------------------------------------------------------------------------
template <int D, bool FP8, bool G16>
struct MmaCompute {
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

    __device__ void init(const DecodeParams &p, int b, int h, int lane)
    {
        const int gid = lane >> 2, tid = lane & 3;
        const uint16_t *qb = p.q + ((size_t)b * p.Hq + (size_t)h * p.group) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int d0 = (4 * (ks / SUBS) + tid) * EK + (ks % SUBS) * 4;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int row = gid + 8 * r;
                uint32_t lo = 0, hi = 0;
                if (row < p.group && (r == 0 || G16)) {
                    const uint32_t *src = reinterpret_cast<const uint32_t *>(qb + (size_t)row * D + d0);
                    lo = __ldg(src);
                    hi = __ldg(src + 1);
                    if (FP8) {
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

    // Write this warp's (m, l, acc) for rows < group into the merge area.
    __device__ void dump(float *ms, float *ls, float *accs, int group, int lane)
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
                    ms[row] = m[r];
                    ls[row] = l[r];
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    accs[row * D + dmap(nt, 2 * tid)] = acc[nt][2 * r];
                    accs[row * D + dmap(nt, 2 * tid + 1)] = acc[nt][2 * r + 1];
                }
            }
        }
    }
};

// ------------------------------------------------------------------------------------
// CUDA-core compute (variant 1).  Lane l owns columns [l*EPL, l*EPL + EPL).
// ------------------------------------------------------------------------------------
template <int D, bool FP8, int GP>
struct SimtCompute {
    static constexpr int ELEM = FP8 ? 1 : 2;
    static constexpr int ROW = D * ELEM;
    static constexpr int EPL = D / 32;
    static constexpr int HALF = 8;                       // tokens per softmax step

    float qf[GP][EPL];
    float acc[GP][EPL];
    float m[GP], l[GP];
    int group;

    __device__ void init(const DecodeParams &p, int b, int h, int lane, float score_scale)
    {
        group = p.group;
        const uint16_t *qb = p.q + ((size_t)b * p.Hq + (size_t)h * p.group) * D;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                float x = 0.f;
                if (g < p.group) x = __uint_as_float((uint32_t)__ldg(qb + (size_t)g * D + lane * EPL + e) << 16);
                if (FP8) x = __half2float(__float2half_rn(x));   // same q rounding as variant 2
                qf[g][e] = x * score_scale;
                acc[g][e] = 0.f;
            }
            m[g] = -INFINITY;
            l[g] = 0.f;
        }
    }

    __device__ __forceinline__ void load_row(const uint8_t *row, int lane, float (&x)[EPL])
    {
        if (FP8) {
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

    __device__ void dump(float *ms, float *ls, float *accs, int grp, int lane)
    {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            if (g < grp) {
                if (lane == 0) {
                    ms[g] = m[g];
                    ls[g] = l[g];
                }
#pragma unroll
                for (int e = 0; e < EPL; ++e) accs[g * D + lane * EPL + e] = acc[g][e];
            }
        }
    }
};

// ------------------------------------------------------------------------------------
// The decode kernel: pipeline + compute + in-CTA merge + output / partial write.
// ------------------------------------------------------------------------------------
template <int D, bool FP8, int NW, int NS, class Compute>
__device__ __forceinline__ void decode_body(const DecodeParams &p, Compute &cmp)
{
    using S = Smem<D, FP8, NW, NS>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int item = blockIdx.x;
    const int h = item % p.Hkv;
    item /= p.Hkv;
    const int b = item % p.B;
    const int part = item / p.B;

    const int L = __ldg(p.seq_lens + b);
    if (L < 1 || L > p.MB * BS) {                    // uniform over the CTA
        if (threadIdx.x == 0) dev::flag_error(p.err, PKV_DEVERR_SEQ_LEN);
        if (part == 0) {
            for (int e = threadIdx.x; e < p.group * D; e += NW * 32)
                p.out[((size_t)b * p.Hq + (size_t)h * p.group) * D + e] = 0;
        }
        return;
    }
    const int nblk = (L + BS - 1) / BS;
    const int nparts = (nblk + p.PB - 1) / p.PB;
    const int blk0 = part * p.PB;
    if (blk0 >= nblk) return;                        // uniform: nothing in this partition
    const int blk1 = min(nblk, blk0 + p.PB);
    const int nloc = blk1 - blk0;

    // Stage this partition's table entries (validated) in shared memory.
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + S::TABLE_OFF);
    const int32_t *row = p.block_tables + (size_t)b * p.MB + blk0;
    for (int i = threadIdx.x; i < nloc; i += NW * 32) {
        int32_t id = __ldg(row + i);
        if (id < 0 || id >= p.num_blocks) {
            dev::flag_error(p.err, PKV_DEVERR_BLOCK_ID);
            id = -1;
        }
        tbl[i] = id;
    }
    if (lane == 0) {
        for (int s = 0; s < NS; ++s)
            dev::mbar_init(dev::smem_u32(smem + S::BAR_OFF + (warp * NS + s) * 8), 1);
        dev::fence_barrier_init();
    }
    __syncthreads();

    const int n_mine = (nloc - warp + NW - 1) / NW;  // blocks warp, warp+NW, ... (may be 0)
    cmp.init(p, b, h, lane, p.score_scale);

    if (lane == 0)
        for (int i = 0; i < NS && i < n_mine; ++i) issue_block<D, FP8, NW, NS>(p, h, smem, tbl, warp, i);
    __syncwarp();

    int i = 0;
    for (; i < n_mine; ++i) {
        const int s = i % NS;
        const uint32_t bar = dev::smem_u32(smem + S::BAR_OFF + (warp * NS + s) * 8);
        const bool ok = __all_sync(dev::FULL, dev::mbar_wait_bounded(bar, (uint32_t)((i / NS) & 1)));
        if (!ok) break;
        const int local = warp + NW * i;
        const int j = blk0 + local;
        const int ntok = tbl[local] >= 0 ? min(BS, L - j * BS) : 0;
        if (ntok > 0) {
            const uint8_t *stage = smem + (warp * NS + s) * S::STAGE;
            cmp.block(stage, stage + S::TILE, ntok, p.score_scale, lane);
        }
        __syncwarp();
        if (lane == 0 && i + NS < n_mine) {
            dev::fence_proxy_async_smem();
            issue_block<D, FP8, NW, NS>(p, h, smem, tbl, warp, i + NS);
        }
    }
    if (i < n_mine) {
        // A wait gave up: report it, then give the copies still in flight one more bounded
        // wait so that none lands after this CTA has left.
        if (lane == 0) dev::flag_error(p.err, PKV_DEVERR_TIMEOUT);
        const int last = min(n_mine, i + NS);
        for (int k = i; k < last; ++k) {
            const uint32_t bar = dev::smem_u32(smem + S::BAR_OFF + (warp * NS + (k % NS)) * 8);
            (void)dev::mbar_wait_bounded(bar, (uint32_t)((k / NS) & 1));
        }
    }
    __syncthreads();                                 // every warp done with its stages

    // ---- merge the warps' partial softmax states (fixed warp order)
    float *ms = reinterpret_cast<float *>(smem);     // [NW][16]
    float *ls = ms + NW * 16;                        // [NW][16]
    float *accs = ls + NW * 16;                      // [NW][16][D]
    cmp.dump(ms + warp * 16, ls + warp * 16, accs + (size_t)warp * 16 * D, p.group, lane);
    __syncthreads();

    const int hq0 = h * p.group;
    for (int e = threadIdx.x; e < p.group * D; e += NW * 32) {
        const int r = e / D, d = e - r * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, ms[w * 16 + r]);
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float mw = ms[w * 16 + r];
                const float wt = mw == -INFINITY ? 0.f : dev::fast_exp2(mw - M);
                num += wt * accs[((size_t)w * 16 + r) * D + d];
                den += wt * ls[w * 16 + r];
            }
        }
        const size_t bh = (size_t)b * p.Hq + hq0 + r;
        if (nparts == 1) {
            const float o = den > 0.f ? num / den * p.out_scale : 0.f;
            const __nv_bfloat16 ob = __float2bfloat16_rn(o);
            p.out[bh * D + d] = *reinterpret_cast<const uint16_t *>(&ob);
        } else {
            p.part_o[(bh * p.P + part) * D + d] = num * p.out_scale;
            if (d == 0) {
                p.part_ml[(bh * p.P + part) * 2 + 0] = M;
                p.part_ml[(bh * p.P + part) * 2 + 1] = den;
            }
        }
    }
}

// MmaCompute::init takes no score_scale (it is applied to S); adapt decode_body's call.
template <int D, bool FP8, bool G16>
struct MmaAdapter : MmaCompute<D, FP8, G16> {
    __device__ void init(const DecodeParams &p, int b, int h, int lane, float)
    {
        MmaCompute<D, FP8, G16>::init(p, b, h, lane);
    }
};

// At most 128 registers per thread: 16 warps (512 threads) can be resident per SM.
template <int D, bool FP8, int NW, int NS, bool G16>
__global__ void __launch_bounds__(NW * 32, 16 / NW) decode_mma_kernel(const DecodeParams p)
{
    MmaAdapter<D, FP8, G16> cmp;
    decode_body<D, FP8, NW, NS>(p, cmp);
}

template <int D, bool FP8, int NW, int NS, int GP>
__global__ void __launch_bounds__(NW * 32) decode_simt_kernel(const DecodeParams p)
{
    SimtCompute<D, FP8, GP> cmp;
    decode_body<D, FP8, NW, NS>(p, cmp);
}

// ------------------------------------------------------------------------------------
// Launch plan and per-instantiation launchers.
// ------------------------------------------------------------------------------------
struct Plan {
    int variant, nw, ns, pb, parts;
    size_t ws_o, ws_ml;                              // workspace byte offsets
    size_t ws_bytes;
};

template <class K>
cudaError_t launch_with_smem(K kernel, int grid, int threads, size_t smem, cudaStream_t s,
                             const DecodeParams &p)
{
    // cudaFuncSetAttribute is cheap but not free; remember per (kernel, device).
    static std::mutex mu;
    static const void *seen_fn[256];
    static int seen_dev[256];
    static int nseen = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    bool known = false;
    {
        std::lock_guard<std::mutex> g(mu);
        for (int i = 0; i < nseen; ++i)
            if (seen_fn[i] == (const void *)kernel && seen_dev[i] == dev) known = true;
        if (!known) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            if (nseen < 256) {
                seen_fn[nseen] = (const void *)kernel;
                seen_dev[nseen] = dev;
                ++nseen;
            }
        }
    }
    kernel<<<grid, threads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int D, bool FP8, int NW, int NS>
cudaError_t launch_decode(const Plan &pl, int group, int grid, cudaStream_t s, const DecodeParams &p)
{
    using S = Smem<D, FP8, NW, NS>;
    const int threads = NW * 32;
    if (pl.variant == 2) {
        if (group > 8)
            return launch_with_smem(decode_mma_kernel<D, FP8, NW, NS, true>, grid, threads, S::BYTES, s, p);
        return launch_with_smem(decode_mma_kernel<D, FP8, NW, NS, false>, grid, threads, S::BYTES, s, p);
    }
    if constexpr (NW == 4 && NS == 2) {
        if (group <= 1) return launch_with_smem(decode_simt_kernel<D, FP8, NW, NS, 1>, grid, threads, S::BYTES, s, p);
        if (group <= 2) return launch_with_smem(decode_simt_kernel<D, FP8, NW, NS, 2>, grid, threads, S::BYTES, s, p);
        if (group <= 4) return launch_with_smem(decode_simt_kernel<D, FP8, NW, NS, 4>, grid, threads, S::BYTES, s, p);
        return launch_with_smem(decode_simt_kernel<D, FP8, NW, NS, 8>, grid, threads, S::BYTES, s, p);
    }
    return cudaErrorInvalidConfiguration;
}

// (warps per CTA, stages per warp) pairs that are compiled.  The CUDA-core variant exists
// for comparison only and is compiled for the default pair.
template <int D, bool FP8>
cudaError_t dispatch_nw_ns(const Plan &pl, int group, int grid, cudaStream_t s, const DecodeParams &p)
{
    if (pl.variant == 1 && !(pl.nw == 4 && pl.ns == 2)) return cudaErrorInvalidConfiguration;
    if (pl.nw == 4 && pl.ns == 2) return launch_decode<D, FP8, 4, 2>(pl, group, grid, s, p);
    if (pl.nw == 4 && pl.ns == 3) return launch_decode<D, FP8, 4, 3>(pl, group, grid, s, p);
    if (pl.nw == 8 && pl.ns == 2) return launch_decode<D, FP8, 8, 2>(pl, group, grid, s, p);
    if (pl.nw == 2 && pl.ns == 4) return launch_decode<D, FP8, 2, 4>(pl, group, grid, s, p);
    return cudaErrorInvalidConfiguration;
}

}  // namespace decode
}  // namespace pkv
