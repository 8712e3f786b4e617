// ne_fwd.cu -- forward kernel: causal grouped-query attention with RoPE fused
// into the Q/K tile load, tcgen05 tensor-core MMAs accumulating in TMEM and an
// online softmax (the tiled FlashAttention of the NanoEuler walkthrough,
// section 3.4, and of the NanoEuler README's "CUDA engine" section, rebuilt
// for sm_103a).
//
// Persistent: one CTA per SM walks a snake-ordered list of work units
// (b, kv head j, query tile m, chunk of GC query heads that share j),
// heaviest (largest m) first.  Per unit the loop runs over the causal key
// tiles jk <= m, each split into two halves of 64 keys, and the GC heads:
// an "item" is one 128 x 64 score block (jk, head, half).  Each K/V tile is
// loaded once by TMA, rotated once and used by all GC heads.
// Warp roles (512 threads):
//   warps 0-3, 4-7  two softmax warpgroups.  The unit's 2*GC (head, key
//               half) pairs are split between them: group w owns pairs
//               w*GC .. w*GC+GC-1 (pair 2h + x = head h, keys [64x, 64x+64)
//               of every key tile), so each group runs its own items with
//               its running max and sum in registers; thread r owns query
//               row r (TMEM lane r) of the item's 128 x 64 score block.  For
//               odd GC one head is split between the groups: each keeps a
//               partial O, max and sum, merged once at the end of the unit
//               (by group 0 in even units, group 1 in odd ones).
//               The running max moves lazily (only when it grows by more
//               than 2^8; the final division by l makes the result exact
//               either way).  Each group has one S buffer, released as soon
//               as the group has loaded it (so S(n+1) is computed while the
//               group works on item n), and two P buffers.
//   warps 8-11  RoPE: rotate the unit's Q tiles and each K tile in place
//               (bf16 in, fp16 out), in the order the MMAs first need them,
//               and record rows of large norm (see "exact scores of large
//               rows" below).
//   warp 12     TMA producer.
//   warps 13, 14  MMA issuers of softmax groups 0 and 1 (warp 13 also
//               allocates TMEM): S(n) into the group's S buffer, then
//               PV(n - 1) reading P from the group's P buffer (n - 1) % 2.
//   warp 15     training path only: stores each rotated Q' tile and each K'
//               tile once into the backward's workspace, and tells the
//               producer when a buffer it stored from may be reloaded.
// After the loop the softmax warps repair the rows of the CTA's units that
// see a recorded large row (rare; nothing happens on ordinary inputs).
// TMEM: one 64-column S buffer per group (columns 0-127), two 32-column P
// buffers per group (bf16 pairs, columns 128-255), then the groups' O
// accumulators (COL_O + (w*NSL + slot)*D).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ne_common.cuh"
#include "ne_kernels.h"

namespace ne {

// Shared-memory plan: QB Q-tile sets of GC heads (two for D <= 64, so the
// next unit's Q' is loaded and rotated while the current unit runs), ST K/V
// stages (as many as fit, at most four), two O staging blocks (D <= 64) and
// the running max / sum of a split head.
template <int D, int GC>
struct FwdPlan {
    using TL = Tile<D>;
    static constexpr bool STAGE = (D <= 64);
    static constexpr int QB = (D <= 64) ? 2 : 1;
    static constexpr int fixed_bytes()
    {
        return QB * GC * TL::BYTES + (STAGE ? 2 * TL::BLOCK : 0) + 2 * kRows * 4 + 1024;
    }
    static constexpr int stages()
    {
        int st = 4;
        while (st > 1 && fixed_bytes() + st * 2 * TL::BYTES > 232448 - 1024)
            --st;
        return st;
    }
    static constexpr int ST = stages();
};

template <int D, int GC, int ST>
struct FwdCfg {
    using TL = Tile<D>;
    using PL = FwdPlan<D, GC>;
    static constexpr bool STAGE = PL::STAGE;                 // O leaves by TMA store
    static constexpr int QB = PL::QB;
    static constexpr int OFF_Q = 0;                          // [QB][GC] tiles
    static constexpr int OFF_K = OFF_Q + QB * GC * TL::BYTES;
    static constexpr int OFF_V = OFF_K + ST * TL::BYTES;
    static constexpr int OFF_O = OFF_V + ST * TL::BYTES;      // [2] staging blocks
    // group 1's running max and sum of the split head: float [2][128]
    static constexpr int OFF_SPL = OFF_O + (STAGE ? 2 * TL::BLOCK : 0);
    static constexpr int SMEM_BYTES = smem_one_cta(OFF_SPL + 2 * kRows * 4 + 1024);
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int NSL = (GC + 1) / 2;          // O accumulators per softmax group
    static constexpr bool SPLIT = (GC & 1) != 0;      // one head's key halves in both groups
    static constexpr uint32_t COL_S = 0;              // S buffer of group w: 64 w
    static constexpr uint32_t COL_P = 128;            // P buffer b of group w: COL_P + 64 w + 32 b
    static constexpr uint32_t COL_O = 256;            // O slot s of group w: COL_O + (w NSL + s) D
    static_assert(COL_O + 2 * NSL * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448 - 1024, "shared memory budget");
    static_assert(ST >= 2, "K/V double buffering");
    static_assert(!STAGE || TL::NB == 1, "staged epilogue stores one column block per head");
};

struct FwdUnit {
    int m, b, j, h0, lo;   // lo: first key tile (sliding window; 0 otherwise)
    SeqLoc sq;             // where sequence b's rows live
};

// VAR: u indexes the launch's table of live units (padded variable-length
// batches), which holds indices into the full enumeration below.
template <bool VAR>
__device__ __forceinline__ FwdUnit fwd_unit(int u, int GC, const AttnParams &p)
{
    if constexpr (VAR)
        u = __ldg(p.units + u);
    FwdUnit w;
    const int per_m = p.B * p.Hkv * p.nchunks;
    w.m = p.M - 1 - u / per_m;
    int rem = u % per_m;
    const int chunk = rem % p.nchunks;
    rem /= p.nchunks;
    w.j = rem % p.Hkv;
    w.b = rem / p.Hkv;
    w.h0 = w.j * p.G + chunk * GC;
    w.lo = key_tile_lo(w.m, p.window);
    w.sq = seq_loc<VAR>(p, w.b);
    return w;
}

// The order in which the producer loads, the RoPE warps rotate and the store
// warp saves a unit's tiles: [Q' of head 0], K lo, [Q' of heads 1..GC-1],
// K lo+1..m, [Q' of the next unit].  The unit's own Q' tiles are listed only
// when they were not loaded with the previous unit (nq0 = GC or 0); the next
// unit's only when they are prefetched (nq1 = GC or 0).  K lo right after the
// first Q' tile lets the first S start after two rotations; the next unit's
// Q' tiles come last so that they never hold up this unit's K tiles.
struct UnitTile {
    bool isq;
    int qunit;   // unit whose Q' tile it is (k or k + 1)
    int g;       // head of the unit's chunk (Q' tiles)
    int jk;      // key tile (K tiles)
};

__device__ __forceinline__ int unit_tiles(int nq0, int nq1, const FwdUnit &w)
{
    return nq0 + 1 + (w.m - w.lo) + nq1;
}

__device__ __forceinline__ UnitTile unit_tile(int t, int k, int nq0, const FwdUnit &w)
{
    const int a = nq0 > 0 ? 1 : 0, nk = w.m - w.lo;
    if (t < a)
        return UnitTile{true, k, 0, 0};
    if (t == a)
        return UnitTile{false, k, 0, w.lo};
    if (t <= nq0)
        return UnitTile{true, k, t - 1, 0};
    if (t <= nq0 + nk)
        return UnitTile{false, k, 0, w.lo + t - nq0};
    return UnitTile{true, k + 1, t - nq0 - nk - 1, 0};
}

// ------------------------------------------------ exact scores of large rows ---
//
// A row of a Q or K tile is "large" when its rotated vector has mean square
// above 4 (sum of squares > 4 D): the fp16 rounding error of its scores,
// proportional to |q'||k'|, would exceed what the 1e-3 lse tolerance allows.
// A unit-variance row passes that bound with probability below 1e-12 at
// d = 32 (chi-squared tail), so ordinary inputs never take this path.
//
// The RoPE thread that rotates such a row records it in the CTA's flag list:
// a query row under its unit, a key row once per (sequence, kv head).  After
// the persistent loop, when the list is not empty, the CTA's softmax warps
// repair the rows of their own units from global memory (every O tile of the
// CTA is stored by then; no other CTA writes these rows):
//   - a large query row is recomputed exactly: fp32 scores from the bf16
//     inputs over all its visible keys, then its O row and lse;
//   - every other row t of the unit that sees large keys s_i is corrected.
//     With p(S) = exp(S / sqrt(d) - lse_t), S_i the exact fp32 score and
//     F_i the product of the fp16 operands the tensor cores saw:
//         delta_i = p(S_i) - p(F_i),   Delta = sum_i delta_i
//         lse_t' = lse_t + log1p(Delta)
//         O_t'   = (O_t + sum_i delta_i v_i) / (1 + Delta)
//     which is the softmax with those pairs' scores made exact.
// A CTA records up to kFlagCap rows; more set NE_WARN_PRECISION (the rows
// left out keep the fp16 error on their pairs).
constexpr int kFlagCap = 48;
constexpr uint32_t kFlagKey = 15u;   // entry kind of a key row (a query row: its head g < 4)

// Entry: bits 0-23 the row's position in its sequence, 24-27 the kind,
// 32-63 the unit index (query rows) or b * Hkv + j (key rows).
__device__ __forceinline__ uint64_t flag_entry(uint32_t hi, uint32_t kind, uint32_t pos)
{
    return (static_cast<uint64_t>(hi) << 32) | (kind << 24) | pos;
}
__device__ __forceinline__ uint32_t flag_hi(uint64_t e) { return static_cast<uint32_t>(e >> 32); }
__device__ __forceinline__ uint32_t flag_kind(uint64_t e)
{
    return (static_cast<uint32_t>(e) >> 24) & 15u;
}
__device__ __forceinline__ int flag_pos(uint64_t e)
{
    return static_cast<int>(static_cast<uint32_t>(e) & 0xFFFFFFu);
}

// Records entry e; a key row only once (every unit that reads its tile
// rotates it again, always in the same thread, which sees its own entry).
// Free slots hold ~0, which no entry equals.
__device__ __forceinline__ void flag_row(uint64_t *list, uint32_t *cnt, uint64_t e, bool once,
                                         uint32_t *status)
{
    volatile uint64_t *vl = list;
    if (once) {
        const uint32_t n = *reinterpret_cast<volatile uint32_t *>(cnt);
        for (uint32_t i = 0; i < n && i < static_cast<uint32_t>(kFlagCap); ++i)
            if (vl[i] == e)
                return;
    }
    const uint32_t i = atomicAdd(cnt, 1u);
    if (i < static_cast<uint32_t>(kFlagCap))
        vl[i] = e;
    else
        atomicOr(status, kDevPrecision);
}

// Pair i (elements i and i + D/2) of the bf16 row at `row`, rotated exactly
// as the RoPE warps rotate it, in fp32.
__device__ __forceinline__ void exact_pair(const __nv_bfloat16 *row, int half_d, uint32_t pos,
                                           const RopeFreqs &fr, int i, float &u, float &w)
{
    float sn, cs;
    rope_sincos(pos, fr, i, sn, cs);
    rope_rotate(__bfloat162float(row[i]), __bfloat162float(row[i + half_d]), cs, sn, u, w);
}

// The value the tensor cores see for x (the fp16 operand of a score).
__device__ __forceinline__ float as_f16(float x) { return __half2float(__float2half_rn(x)); }

// Scratch (floats, in the CTA's idle tile buffers) of the repair below.
template <int D>
struct FixScratch {
    static constexpr int NT = 256;                    // the softmax threads
    static constexpr int QV = 0;                      // exact q' of the row recomputed [D]
    static constexpr int PART = QV + D;               // per warp: max, sum, O [8][D + 2]
    static constexpr int KPOS = PART + 8 * (D + 2);   // int: the unit's large keys, ascending
    static constexpr int NK = KPOS + kFlagCap;        // int: how many
    static constexpr int KDAT = NK + 4;               // per key: exact k', fp16 k', v [3][D]
    static constexpr int DPS = KDAT + kFlagCap * 3 * D;   // delta_i per thread [kFlagCap][NT]
    static constexpr int BYTES = (DPS + kFlagCap * NT) * 4;
};

// The repair of the rows of this CTA's units (the comment block above).  Run
// by the 256 softmax threads, which meet at named barrier 1; every branch
// around a barrier depends only on the list and the unit, so it is uniform.
template <int D, int GC, bool WIN, bool VAR>
__device__ __noinline__ void fix_large_rows(float *scr, const uint64_t *list, int nflag, int cta,
                                            int P, int NU, const AttnParams &p)
{
    using FS = FixScratch<D>;
    constexpr int NT = FS::NT, D2 = D / 2, PPL = (D2 + 31) / 32;   // pairs per lane
    const int tid = static_cast<int>(threadIdx.x), warp = tid / 32, lane = tid % 32;
    const __nv_bfloat16 *qin = static_cast<const __nv_bfloat16 *>(p.q_in);
    const __nv_bfloat16 *kin = static_cast<const __nv_bfloat16 *>(p.k_in);
    const __nv_bfloat16 *vin = static_cast<const __nv_bfloat16 *>(p.v_in);
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out0);
    const float sl2 = p.scale_log2;
    float *qv = scr + FS::QV, *part = scr + FS::PART, *kdat = scr + FS::KDAT, *dps = scr + FS::DPS;
    int *kpos = reinterpret_cast<int *>(scr + FS::KPOS);
    int *nkp = reinterpret_cast<int *>(scr + FS::NK);
    for (int k = 0;; ++k) {
        const int u = snake_unit(k, cta, P);
        if (u >= NU)
            break;
        const FwdUnit w = fwd_unit<VAR>(u, GC, p);
        const uint32_t kvid = static_cast<uint32_t>(w.b * p.Hkv + w.j);
        const int s_lo = w.lo * kRows, s_hi = w.m * kRows + kRows - 1;
        bool anyq = false, anyk = false;
        for (int i = 0; i < nflag; ++i) {
            const uint64_t e = list[i];
            const uint32_t kind = flag_kind(e);
            anyq = anyq || (kind < static_cast<uint32_t>(GC) && flag_hi(e) == static_cast<uint32_t>(k));
            anyk = anyk || (kind == kFlagKey && flag_hi(e) == kvid && flag_pos(e) >= s_lo &&
                            flag_pos(e) <= s_hi);
        }
        if (!anyq && !anyk)
            continue;

        // ---- large query rows of the unit: recomputed exactly.  Keys are
        // dealt to the 8 warps in turn, rotate-half pairs to the lanes; each
        // warp keeps an online max / sum / O, merged in warp order.
        for (int i = 0; i < nflag && anyq; ++i) {
            const uint64_t e = list[i];
            const int g = static_cast<int>(flag_kind(e));
            if (g >= GC || flag_hi(e) != static_cast<uint32_t>(k))
                continue;
            const int t = flag_pos(e), h = w.h0 + g;
            const size_t orow = static_cast<size_t>(seq_row(p, w.sq, t)) * p.Hq + h;
            for (int pi = tid; pi < D2; pi += NT)
                exact_pair(qin + orow * D, D2, static_cast<uint32_t>(t), p.rope, pi, qv[pi],
                           qv[pi + D2]);
            named_bar_sync(1, NT);
            float qa[PPL], qb[PPL], acc[2 * PPL];
#pragma unroll
            for (int c = 0; c < PPL; ++c) {
                const int pi = lane + 32 * c;
                qa[c] = pi < D2 ? qv[pi] : 0.f;
                qb[c] = pi < D2 ? qv[pi + D2] : 0.f;
                acc[2 * c] = acc[2 * c + 1] = 0.f;
            }
            float m = -INFINITY, l = 0.f;
            const int s0 = WIN ? max(0, t - p.window + 1) : 0;
            for (int s = s0 + warp; s <= t; s += 8) {
                const size_t krow = (static_cast<size_t>(seq_row(p, w.sq, s)) * p.Hkv + w.j) * D;
                float dot = 0.f;
#pragma unroll
                for (int c = 0; c < PPL; ++c) {
                    const int pi = lane + 32 * c;
                    if (pi < D2) {
                        float a, b;
                        exact_pair(kin + krow, D2, static_cast<uint32_t>(s), p.rope, pi, a, b);
                        dot = fmaf(qa[c], a, fmaf(qb[c], b, dot));
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    dot += __shfl_down_sync(0xffffffffu, dot, o);
                const float sc = __shfl_sync(0xffffffffu, dot, 0) * sl2;   // log2 units
                const float mn = fmaxf(m, sc);
                const float a = exp2f(m - mn), pp = exp2f(sc - mn);
                l = fmaf(l, a, pp);
#pragma unroll
                for (int c = 0; c < PPL; ++c) {
                    const int pi = lane + 32 * c;
                    if (pi < D2) {
                        acc[2 * c] = fmaf(acc[2 * c], a, pp * __bfloat162float(vin[krow + pi]));
                        acc[2 * c + 1] =
                            fmaf(acc[2 * c + 1], a, pp * __bfloat162float(vin[krow + pi + D2]));
                    }
                }
                m = mn;
            }
            float *pw = part + warp * (D + 2);
            if (lane == 0) {
                pw[0] = m;
                pw[1] = l;
            }
#pragma unroll
            for (int c = 0; c < PPL; ++c) {
                const int pi = lane + 32 * c;
                if (pi < D2) {
                    pw[2 + pi] = acc[2 * c];
                    pw[2 + pi + D2] = acc[2 * c + 1];
                }
            }
            named_bar_sync(1, NT);
            if (tid < D) {
                float mt = -INFINITY;
                for (int v = 0; v < 8; ++v)
                    mt = fmaxf(mt, part[v * (D + 2)]);
                float lt = 0.f, ot = 0.f;
                for (int v = 0; v < 8; ++v) {
                    const float mv = part[v * (D + 2)];
                    if (mv == -INFINITY)
                        continue;   // a warp that saw no key
                    const float f = exp2f(mv - mt);
                    lt = fmaf(part[v * (D + 2) + 1], f, lt);
                    ot = fmaf(part[v * (D + 2) + 2 + tid], f, ot);
                }
                out[orow * D + tid] = __float2bfloat16_rn(ot / lt);
                if (tid == 0)
                    p.lse[(static_cast<size_t>(w.sq.bc) * p.Hq + h) * p.T + w.sq.base + t] =
                        (mt + __log2f(lt)) * kLn2;
            }
            named_bar_sync(1, NT);   // qv and part are reused
        }

        // ---- rows that see the unit's large keys
        if (!anyk)
            continue;
        if (tid == 0) {   // the keys in ascending order: a fixed summation order
            int nk = 0;
            for (int i = 0; i < nflag; ++i) {
                const uint64_t e = list[i];
                const int s = flag_pos(e);
                if (flag_kind(e) != kFlagKey || flag_hi(e) != kvid || s < s_lo || s > s_hi)
                    continue;
                int j = nk++;
                for (; j > 0 && kpos[j - 1] > s; --j)
                    kpos[j] = kpos[j - 1];
                kpos[j] = s;
            }
            *nkp = nk;
        }
        named_bar_sync(1, NT);
        const int nk = *nkp;
        for (int it = tid; it < nk * D2; it += NT) {
            const int i = it / D2, pi = it % D2, s = kpos[i];
            const size_t krow = (static_cast<size_t>(seq_row(p, w.sq, s)) * p.Hkv + w.j) * D;
            float *kd = kdat + i * 3 * D;
            float a, b;
            exact_pair(kin + krow, D2, static_cast<uint32_t>(s), p.rope, pi, a, b);
            kd[pi] = a;
            kd[pi + D2] = b;
            kd[D + pi] = as_f16(a);
            kd[D + pi + D2] = as_f16(b);
            kd[2 * D + pi] = __bfloat162float(vin[krow + pi]);
            kd[2 * D + pi + D2] = __bfloat162float(vin[krow + pi + D2]);
        }
        named_bar_sync(1, NT);
        for (int rr = tid; rr < GC * kRows; rr += NT) {
            const int g = rr / kRows, t = w.m * kRows + rr % kRows, h = w.h0 + g;
            if (t >= w.sq.len)
                continue;
            bool exact = false;   // a large query row, already recomputed
            for (int i = 0; i < nflag; ++i)
                exact = exact || list[i] == flag_entry(static_cast<uint32_t>(k),
                                                        static_cast<uint32_t>(g),
                                                        static_cast<uint32_t>(t));
            if (exact)
                continue;
            const size_t orow = static_cast<size_t>(seq_row(p, w.sq, t)) * p.Hq + h;
            float *lp = p.lse + (static_cast<size_t>(w.sq.bc) * p.Hq + h) * p.T + w.sq.base + t;
            const float lse = __ldcg(lp), lse2 = lse * kLog2e;
            float delta = 0.f;
            bool any = false;
            for (int i = 0; i < nk; ++i) {
                const int s = kpos[i];
                float dp = 0.f;
                if (s <= t && (!WIN || t - s < p.window)) {
                    const float *kd = kdat + i * 3 * D;
                    float se = 0.f, sh = 0.f;
                    for (int pi = 0; pi < D2; ++pi) {
                        float a, b;
                        exact_pair(qin + orow * D, D2, static_cast<uint32_t>(t), p.rope, pi, a, b);
                        se = fmaf(a, kd[pi], fmaf(b, kd[pi + D2], se));
                        sh = fmaf(as_f16(a), kd[D + pi], fmaf(as_f16(b), kd[D + pi + D2], sh));
                    }
                    dp = exp2f(se * sl2 - lse2) - exp2f(sh * sl2 - lse2);
                    any = true;
                }
                dps[i * NT + tid] = dp;
                delta += dp;
            }
            if (!any)
                continue;
            const float inv = 1.f / (1.f + delta);
            uint4 *o4 = reinterpret_cast<uint4 *>(out + orow * D);
            for (int c = 0; c < D / 8; ++c) {
                const uint4 v4 = __ldcg(o4 + c);
                const uint32_t wv[4] = {v4.x, v4.y, v4.z, v4.w};
                float x[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    x[2 * e] = bf16_lo(wv[e]);
                    x[2 * e + 1] = bf16_hi(wv[e]);
                }
                for (int i = 0; i < nk; ++i) {
                    const float dp = dps[i * NT + tid];
                    const float *vv = kdat + i * 3 * D + 2 * D + 8 * c;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        x[e] = fmaf(dp, vv[e], x[e]);
                }
                o4[c] = make_uint4(pack_bf16x2(x[0] * inv, x[1] * inv),
                                   pack_bf16x2(x[2] * inv, x[3] * inv),
                                   pack_bf16x2(x[4] * inv, x[5] * inv),
                                   pack_bf16x2(x[6] * inv, x[7] * inv));
            }
            *lp = lse + log1pf(delta);
        }
        named_bar_sync(1, NT);   // kpos and kdat are reused
    }
}

// WIN: a sliding window may mask keys off the diagonal tile (compiled out of
// the causal instantiations).  VAR: padded variable-length batch, the units
// come from a table that leaves out every query tile past its sequence's
// length; rows of a live tile past that length are computed like any other
// (over the padding keys) and overwritten afterwards by the padding fill.
template <int D, int GC, int ST, bool WIN, bool VAR>
__global__ void __launch_bounds__(512, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
               const __grid_constant__ CUtensorMap tmQs, const __grid_constant__ CUtensorMap tmKs,
               const AttnParams p)
{
    using C = FwdCfg<D, GC, ST>;
    using TL = Tile<D>;
    static_assert(FixScratch<D>::BYTES <= C::OFF_SPL, "repair scratch fits the tile buffers");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    constexpr int QB = C::QB;
    __shared__ uint64_t bar_q_full[QB][GC], bar_q_ready[QB][GC], bar_q_empty[QB][GC];
    __shared__ uint64_t bar_k_full[ST], bar_k_ready[ST], bar_v_full[ST], bar_kv_empty[ST];
    // per softmax group w: S written (MMA commit), S loaded by the group (its
    // four warps); per P buffer b: P written (four warps), P read by the PV
    // MMA (commit)
    __shared__ uint64_t bar_s_full[2], bar_s_empty[2], bar_p_full[2][2], bar_p_free[2][2];
    __shared__ uint64_t bar_o_free[2][C::NSL], bar_split, bar_drain;
    // O staging block of group w written (its four warps) / read by its store
    // training path: the RoPE warps finished the n-th tile to be stored
    // (ring of 16: they are never 16 such tiles ahead of warp 15, which must
    // release a Q slot or a stored K stage before it is reloaded), and warp
    // 15's store has read a Q slot / K stage
    __shared__ uint64_t bar_sv[16], bar_q_rd[QB][GC], bar_k_rd[ST];
    // rows of large norm recorded by the RoPE warps
    __shared__ uint64_t flag_list[kFlagCap];
    __shared__ uint32_t flag_cnt;
    __shared__ uint32_t tmem_base_s;
    __shared__ uint32_t abort_s;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cta = static_cast<int>(blockIdx.x), P = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        abort_s = 0;
        for (int g = 0; g < GC; ++g) {
            for (int qb = 0; qb < QB; ++qb) {
                mbar_init(smem_u32(&bar_q_full[qb][g]), 1);
                mbar_init(smem_u32(&bar_q_ready[qb][g]), 4);
                mbar_init(smem_u32(&bar_q_empty[qb][g]), 2);
                mbar_init(smem_u32(&bar_q_rd[qb][g]), 1);
            }
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&bar_k_full[s]), 1);
            mbar_init(smem_u32(&bar_k_ready[s]), 4);
            mbar_init(smem_u32(&bar_v_full[s]), 1);
            mbar_init(smem_u32(&bar_kv_empty[s]), 2);
            mbar_init(smem_u32(&bar_k_rd[s]), 1);
        }
        flag_cnt = 0;
        for (int i = 0; i < kFlagCap; ++i)
            flag_list[i] = ~0ull;
        for (int w = 0; w < 2; ++w) {
            mbar_init(smem_u32(&bar_s_full[w]), 1);
            mbar_init(smem_u32(&bar_s_empty[w]), 4);
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_u32(&bar_p_full[w][b]), 4);
                mbar_init(smem_u32(&bar_p_free[w][b]), 1);
            }
            for (int sl = 0; sl < C::NSL; ++sl)
                mbar_init(smem_u32(&bar_o_free[w][sl]), 4);
        }
        mbar_init(smem_u32(&bar_split), 4);
        mbar_init(smem_u32(&bar_drain), 2);
        for (int i = 0; i < 16; ++i)
            mbar_init(smem_u32(&bar_sv[i]), 4);
        fence_mbar_init();
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(&tmem_base_s), C::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_s;
    // Only shared memory and TMEM were touched so far: from here on global
    // memory is read and written, so wait for the previous grid in the stream
    // (programmatic dependent launch).
    griddep_wait();
    const int NU = unit_total<VAR>(p);   // work units of the launch
    const WaitCtl wc{&abort_s, p.status, p.wait_limit_ns};
    // Each role ends with its own teardown: after setmaxnreg the warps run
    // under different register budgets, so their code paths never re-join.
    auto teardown = [&]() {
        tc_fence_before();
        __syncthreads();
        griddep_launch_dependents();   // this CTA's work is done
        if (warp == 13) {
            tc_fence_after();
            tmem_dealloc(tbase, C::TMEM_COLS);
        }
    };

    // Register budgets after the split (launched with 128 per thread x 512):
    // softmax 184 x 256 + RoPE 80 x 128 + TMA/MMA 64 x 128 = 65536.
    if (warp >= 12) {
        regs_release<64>();
        if (warp == 12) {
            // ------------------------------------------------ TMA producer ---
            // The whole warp waits (a suspended warp leaves the issue slots to
            // the softmax warps); lane 0 issues the copies.
            if (lane == 0) {
                tma_prefetch_desc(&tmQ);
                tma_prefetch_desc(&tmK);
                tma_prefetch_desc(&tmV);
            }
            bool ok = true;
            int kt = 0;
            int qloads[QB][GC] = {};   // loads issued per Q slot (for the abort drain)
            // Q' tiles of unit kk into set kk % QB, once the set's previous
            // unit has issued its last S
            auto load_q = [&](int kk, int g0, int g1) {
                const FwdUnit w = fwd_unit<VAR>(snake_unit(kk, cta, P), GC, p);
                const int qb = kk % QB, use = kk / QB;
                for (int g = g0; g < g1; ++g) {
                    if (use >= 1 && !mbar_wait_warp(smem_u32(&bar_q_empty[qb][g]), (use - 1) & 1, wc))
                        return false;
                    // training path: the previous tile of this slot was stored
                    if (p.save_rot && use >= 1 &&
                        !mbar_wait_warp(smem_u32(&bar_q_rd[qb][g]), (use - 1) & 1, wc))
                        return false;
                    const uint32_t bar = smem_u32(&bar_q_full[qb][g]);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar, TL::BYTES);
                        for (int cb = 0; cb < TL::NB; ++cb)
                            tma_load_4d(smem_u32(smem + C::OFF_Q + (qb * GC + g) * TL::BYTES +
                                                 cb * TL::BLOCK),
                                        &tmQ, bar, cb * TL::BOX_COLS, w.h0 + g,
                                        w.sq.base + w.m * kRows, w.sq.bc);
                    }
                    __syncwarp();
                    ++qloads[qb][g];
                }
                return true;
            };
            // training path: K' tiles stored from each stage (count, and
            // whether the stage's last tile was one)
            int ksaved[ST] = {};
            uint32_t last_saved = 0;
            auto load_kv = [&](const FwdUnit &w, int jk) {
                const int st = kt % ST, u2 = kt / ST;
                if (u2 >= 1 && !mbar_wait_warp(smem_u32(&bar_kv_empty[st]), (u2 - 1) & 1, wc))
                    return false;
                if (((last_saved >> st) & 1u) &&
                    !mbar_wait_warp(smem_u32(&bar_k_rd[st]), (ksaved[st] - 1) & 1, wc))
                    return false;
                const bool saved = p.save_rot && jk == w.m && w.h0 == w.j * p.G;
                last_saved = (last_saved & ~(1u << st)) | (saved ? 1u << st : 0u);
                ksaved[st] += saved ? 1 : 0;
                const uint32_t kb = smem_u32(&bar_k_full[st]), vb = smem_u32(&bar_v_full[st]);
                if (lane == 0) {
                    mbar_arrive_expect_tx(kb, TL::BYTES);
                    for (int cb = 0; cb < TL::NB; ++cb)
                        tma_load_4d(smem_u32(smem + C::OFF_K + st * TL::BYTES + cb * TL::BLOCK),
                                    &tmK, kb, cb * TL::BOX_COLS, w.j, w.sq.base + jk * kRows,
                                    w.sq.bc);
                    mbar_arrive_expect_tx(vb, TL::BYTES);
                    for (int cb = 0; cb < TL::NB; ++cb)
                        tma_load_4d(smem_u32(smem + C::OFF_V + st * TL::BYTES + cb * TL::BLOCK),
                                    &tmV, vb, cb * TL::BOX_COLS, w.j, w.sq.base + jk * kRows,
                                    w.sq.bc);
                }
                __syncwarp();
                ++kt;
                return true;
            };
            for (int k = 0; ok; ++k) {
                const int u = snake_unit(k, cta, P);
                if (u >= NU)
                    break;
                const FwdUnit w = fwd_unit<VAR>(u, GC, p);
                // tile order of unit_tile()
                const bool own_q = QB == 1 || k == 0;
                if (own_q)
                    ok = load_q(k, 0, 1);
                ok = ok && load_kv(w, w.lo);
                if (own_q && ok)
                    ok = load_q(k, 1, GC);
                for (int jk = w.lo + 1; jk <= w.m && ok; ++jk)
                    ok = load_kv(w, jk);
                if (QB == 2 && ok && snake_unit(k + 1, cta, P) < NU)
                    ok = load_q(k + 1, 0, GC);
            }
            if (*wc.abort && lane == 0) {
                for (int qb = 0; qb < QB; ++qb)
                    for (int g = 0; g < GC; ++g)
                        if (qloads[qb][g] > 0)
                            mbar_wait_drain(smem_u32(&bar_q_full[qb][g]), (qloads[qb][g] - 1) & 1,
                                            wc.limit_ns);
                for (int t = (kt > ST ? kt - ST : 0); t < kt; ++t) {
                    mbar_wait_drain(smem_u32(&bar_k_full[t % ST]), (t / ST) & 1, wc.limit_ns);
                    mbar_wait_drain(smem_u32(&bar_v_full[t % ST]), (t / ST) & 1, wc.limit_ns);
                }
            }
        } else if (warp == 15 && p.save_rot) {
            // ------------------------------- stores of rotated tiles ---
            // Same tile order as the RoPE warpgroup.  A tile handed over on
            // bar_sv is rotated (and fenced for the async proxy); its store
            // reads the buffer while the MMAs read it too; the producer
            // reloads the buffer only after bar_q_rd / bar_k_rd.
            if (lane == 0) {
                tma_prefetch_desc(&tmQs);
                tma_prefetch_desc(&tmKs);
            }
            bool ok = true;
            int kt = 0;
            uint32_t nsv = 0;
            for (int k = 0; ok; ++k) {
                const int u = snake_unit(k, cta, P);
                if (u >= NU)
                    break;
                const FwdUnit w = fwd_unit<VAR>(u, GC, p);
                const int nq0 = (QB == 1 || k == 0) ? GC : 0;
                const bool has_next = QB == 2 && snake_unit(k + 1, cta, P) < NU;
                const int nq1 = has_next ? GC : 0;
                for (int t = 0; t < unit_tiles(nq0, nq1, w) && ok; ++t) {
                    const UnitTile ut = unit_tile(t, k, nq0, w);
                    const bool isq = ut.isq;
                    const int qunit = ut.qunit, g = ut.g, jk = ut.jk;
                    const int qb = qunit % QB, st = kt % ST;
                    if (!isq)
                        ++kt;
                    if (!isq && !(jk == w.m && w.h0 == w.j * p.G))
                        continue;   // this K' tile is stored by its diagonal unit
                    if (!mbar_wait_warp_idle(smem_u32(&bar_sv[nsv % 16]), (nsv / 16) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    ++nsv;
                    const uint8_t *tile = smem + (isq ? C::OFF_Q + (qb * GC + g) * TL::BYTES
                                                      : C::OFF_K + st * TL::BYTES);
                    if (lane == 0) {
                        const FwdUnit wq =
                            isq && qunit != k ? fwd_unit<VAR>(snake_unit(qunit, cta, P), GC, p) : w;
                        for (int cb = 0; cb < TL::NB; ++cb) {
                            const uint32_t src = smem_u32(tile + cb * TL::BLOCK);
                            if (isq)
                                tma_store_4d(&tmQs, src, cb * TL::BOX_COLS, wq.h0 + g,
                                             wq.sq.base + wq.m * kRows, wq.sq.bc);
                            else
                                tma_store_4d(&tmKs, src, cb * TL::BOX_COLS, w.j,
                                             w.sq.base + jk * kRows, w.sq.bc);
                        }
                        bulk_commit();
                        bulk_wait_read0();
                        mbar_arrive(isq ? smem_u32(&bar_q_rd[qb][g]) : smem_u32(&bar_k_rd[st]));
                    }
                    __syncwarp();
                }
            }
            if (lane == 0)
                bulk_wait0();
        } else if (warp == 13 || warp == 14) {
            // -------------------------------------------------- MMA issuers ---
            // Warp 13 + w issues the MMAs of softmax group w, in the group's
            // item order: S(n) into the group's S buffer once the group has
            // loaded S(n - 1), then PV(n - 1) once P(n - 1) is written; at a
            // unit boundary the previous unit's last PV goes first (its
            // epilogue waits for it; S(n) waits for the new unit's tiles).
            const int wg = warp - 13;
            constexpr uint32_t ID_S = idesc_f16(128, 64, false, false, false);
            constexpr uint32_t ID_PV = idesc_f16(128, TL::NPV, true, false, true);
            constexpr uint32_t TSTEP = TL::BYTES >> 4;
            constexpr uint32_t KHALF = (64 * TL::SWB) >> 4;   // rows 64.. of a K' tile
            const uint32_t sbase = __shfl_sync(0xffffffffu, smem_u32(smem), 0);
            const uint32_t tb = __shfl_sync(0xffffffffu, tbase, 0);
            const uint64_t dQ0 = desc_kmajor_base<D>(sbase + C::OFF_Q);
            const uint64_t dK0 = desc_kmajor_base<D>(sbase + C::OFF_K);
            const uint64_t dV0 = desc_mnmajor_base<D>(sbase + C::OFF_V);
            bool ok = true;
            uint32_t n = 0;
            int kt = 0;
            // the previous item, whose PV is issued after the next S
            struct Pend {
                int k, st, kt, p;
                bool first, last_in_tile;
            } prev{};
            bool have_prev = false;
            auto issue_pv = [&](const Pend &x, uint32_t nx) {
                const int pair = wg * GC + x.p, half = pair & 1;
                const int slot = (pair >> 1) - ((wg * GC) >> 1);
                const uint32_t b = nx & 1u;
                if (!mbar_wait_warp(smem_u32(&bar_p_full[wg][b]), (nx >> 1) & 1, wc) ||
                    !mbar_wait_warp(smem_u32(&bar_v_full[x.st]), (x.kt / ST) & 1, wc) ||
                    (x.first && x.k >= 1 &&
                     !mbar_wait_warp(smem_u32(&bar_o_free[wg][slot]), (x.k - 1) & 1, wc)))
                    return false;
                tc_fence_after();
                const uint64_t vm = dV0 + x.st * TSTEP;
                const uint32_t ocol = tb + C::COL_O + (wg * C::NSL + slot) * D;
                const uint32_t pcol = tb + C::COL_P + 64u * wg + 32u * b;
                if (elect_one()) {
#pragma unroll
                    for (int nc = 0; nc < D / TL::NPV; ++nc)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f16_ts(ocol + nc * TL::NPV, pcol + 8 * kk,
                                       vm + mnmajor_off<D>(nc, 4 * half + kk), ID_PV,
                                       (kk > 0 || !x.first) ? 1u : 0u);
                    mma_commit(smem_u32(&bar_p_free[wg][b]));
                    if (x.last_in_tile)
                        mma_commit(smem_u32(&bar_kv_empty[x.st]));
                }
                __syncwarp();
                return true;
            };
            for (int k = 0; ok; ++k) {
                const int u = snake_unit(k, cta, P);
                if (u >= NU)
                    break;
                const FwdUnit w = fwd_unit<VAR>(u, GC, p);
                const int qb = k % QB;
                for (int jk = w.lo; jk <= w.m && ok; ++jk, ++kt) {
                    const int st = kt % ST;
                    for (int pi = 0; pi < GC; ++pi, ++n) {
                        const int pair = wg * GC + pi, hrel = pair >> 1, half = pair & 1;
                        const bool first = jk == w.lo && (pi == 0 || ((pair - 1) >> 1) != hrel);
                        if (jk == w.lo && pi == 0 && have_prev) {
                            if (!issue_pv(prev, n - 1)) {
                                ok = false;
                                break;
                            }
                            have_prev = false;
                        }
                        // S(n) = Q'_hrel K'[64 half, +64)^T
                        if ((pi == 0 &&
                             !mbar_wait_warp(smem_u32(&bar_k_ready[st]), (kt / ST) & 1, wc)) ||
                            (jk == w.lo && !mbar_wait_warp(smem_u32(&bar_q_ready[qb][hrel]),
                                                           (k / QB) & 1, wc)) ||
                            (n >= 1 &&
                             !mbar_wait_warp(smem_u32(&bar_s_empty[wg]), (n - 1) & 1, wc))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t qd = dQ0 + (qb * GC + hrel) * TSTEP;
                        const uint64_t kd = dK0 + st * TSTEP + half * KHALF;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_f16_ss(tb + C::COL_S + 64u * wg,
                                           qd + kmajor_off<D>(kk), kd + kmajor_off<D>(kk), ID_S,
                                           kk > 0 ? 1u : 0u);
                            mma_commit(smem_u32(&bar_s_full[wg]));
                            if (jk == w.m && pi == GC - 1)   // last S of the unit
                                for (int g = 0; g < GC; ++g)
                                    mma_commit(smem_u32(&bar_q_empty[qb][g]));
                        }
                        __syncwarp();
                        if (have_prev && !issue_pv(prev, n - 1)) {
                            ok = false;
                            break;
                        }
                        prev = Pend{k, st, kt, pi, first, pi == GC - 1};
                        have_prev = true;
                    }
                }
            }
            if (ok && have_prev)
                issue_pv(prev, n - 1);
            if (elect_one())
                mma_commit(smem_u32(&bar_drain));
            __syncwarp();
            mbar_wait_warp(smem_u32(&bar_drain), 0, wc);
        }
        teardown();
        return;
    }
    if (warp >= 8) {
        // ------------------------------------------------------ RoPE ---
        regs_release<80>();
        const int r = threadIdx.x - 256;
        float mx = 0.f;
        bool ok = true;
        int kt = 0;
        uint32_t nsv = 0;     // tiles handed to warp 15 (training path)
        for (int k = 0; ok; ++k) {
            const int u = snake_unit(k, cta, P);
            if (u >= NU)
                break;
            const FwdUnit w = fwd_unit<VAR>(u, GC, p);
            // Tiles in the order the producer loads them (unit_tile()).  One
            // call site keeps the unrolled rotation in the instruction cache
            // once.
            const int nq0 = (QB == 1 || k == 0) ? GC : 0;
            const bool has_next = QB == 2 && snake_unit(k + 1, cta, P) < NU;
            const int nq1 = has_next ? GC : 0;
            const FwdUnit wn = has_next ? fwd_unit<VAR>(snake_unit(k + 1, cta, P), GC, p) : w;
            for (int t = 0; t < unit_tiles(nq0, nq1, w) && ok; ++t) {
                const UnitTile ut = unit_tile(t, k, nq0, w);
                const bool isq = ut.isq;
                const int qunit = ut.qunit, g = ut.g, jk = ut.jk;
                const int qb = qunit % QB, st = kt % ST;
                const uint32_t full = isq ? smem_u32(&bar_q_full[qb][g]) : smem_u32(&bar_k_full[st]);
                const uint32_t par = isq ? ((qunit / QB) & 1) : ((kt / ST) & 1);
                if (!mbar_wait_warp(full, par, wc)) {
                    ok = false;
                    break;
                }
                uint8_t *tile = smem + (isq ? C::OFF_Q + (qb * GC + g) * TL::BYTES
                                            : C::OFF_K + st * TL::BYTES);
                const FwdUnit &tu = (isq && qunit != k) ? wn : w;   // the tile's unit
                const int row0 = isq ? tu.m : jk;
                const uint32_t pos = static_cast<uint32_t>(row0 * kRows + r);
                float ss;
                mx = fmaxf(mx, rope_row_ilp<D>(tile, r, pos, p.rope, ss));
                fence_proxy_async_smem();
                // rows of large norm (rare): recorded for the repair
                if (static_cast<int>(pos) < tu.sq.len && ss > 4.f * D)
                    flag_row(flag_list, &flag_cnt,
                             isq ? flag_entry(static_cast<uint32_t>(qunit), static_cast<uint32_t>(g),
                                              pos)
                                 : flag_entry(static_cast<uint32_t>(w.b * p.Hkv + w.j), kFlagKey,
                                              pos),
                             !isq, p.status);
                const uint32_t ready =
                    isq ? smem_u32(&bar_q_ready[qb][g]) : smem_u32(&bar_k_ready[st]);
                if (lane == 0)
                    mbar_arrive(ready);
                if (p.save_rot && (isq || (jk == w.m && w.h0 == w.j * p.G))) {
                    if (lane == 0)
                        mbar_arrive(smem_u32(&bar_sv[nsv % 16]));
                    ++nsv;
                }
                if (!isq)
                    ++kt;
            }
        }
        if (mx > kFp16Max)
            atomicOr(p.status, kDevRange);
        teardown();
        return;
    }

    // ----------------------------------------------------- softmax rows ---
    // Group wg owns the (head, key half) pairs wg*GC .. wg*GC + GC - 1 of the
    // unit (pair 2h + x = head h, keys [64x, 64x + 64) of every key tile), so
    // the running max and sum of each of its heads stay in registers.  With
    // GC odd one head's two halves belong to different groups; the groups
    // merge it at the end of the unit.
    regs_claim<184>();
    const int wg = warp >> 2;               // softmax group
    const int q4 = warp & 3;                // TMEM lane quarter
    static_assert(kFwdOStoreRows == 32, "a warp stores the rows of its TMEM lane quarter");
    const int r = threadIdx.x & 127;        // query row == TMEM lane
    const uint32_t lane_base = tmem_addr(tbase, q4 * 32, 0);
    const float sl2 = p.scale_log2;
    float *split_ml = reinterpret_cast<float *>(smem + C::OFF_SPL);   // [m | l][row]
    bool ok = true;
    uint32_t n = 0;          // this group's items so far
    uint8_t *stage = smem + C::OFF_O + wg * TL::BLOCK;
    uint32_t nepi = 0;       // O stores this group has issued
    float mr0 = 0.f, mr1 = 0.f, lr0 = 0.f, lr1 = 0.f;   // running max (log2 units) / sum per slot
    // lse of head h for this thread's row (ln units), rows past the sequence
    // skipped
    auto store_lse = [&](const FwdUnit &un, int h, float lse2) {
        const int t = un.m * kRows + r;
        if (t < un.sq.len)
            p.lse[(static_cast<size_t>(un.sq.bc) * p.Hq + h) * p.T + un.sq.base + t] = lse2 * kLn2;
    };
    // Writes O_slot / l of head h (rows of this thread).  The caller folds
    // 1 / l into the scales: O = O_a * fa (+ O_b * fb with a second
    // accumulator, merge), on packed fp32 pairs.
    auto store_head = [&](const FwdUnit &un, int h, uint32_t oa, bool merge, uint32_t ob, float fa,
                          float fb) -> bool {
        const int t = un.m * kRows + r;
        // columns c .. c + 31 of this thread's row, scaled, as bf16 pairs
        auto chunk = [&](int c, uint32_t (&pk)[16]) {
            uint32_t o[32];
            tmem_ld32(oa + c, o);
            tmem_ld_wait(o);
            uint64_t x2[16];
            const uint64_t fa2 = f32x2(fa, fa);
#pragma unroll
            for (int e = 0; e < 16; ++e)
                x2[e] = mul_f32x2(f32x2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])),
                                  fa2);
            if (merge) {
                tmem_ld32(ob + c, o);
                tmem_ld_wait(o);
                const uint64_t fb2 = f32x2(fb, fb);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    x2[e] = fma_f32x2(
                        f32x2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), fb2,
                        x2[e]);
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                float x0, x1;
                f32x2_split(x2[e], x0, x1);
                pk[e] = pack_bf16x2(x0, x1);
            }
        };
        // O row by row from registers (rows past the sequence skipped)
        auto store_direct = [&]() {
            __nv_bfloat16 *dst =
                static_cast<__nv_bfloat16 *>(p.out0) + (seq_row(p, un.sq, t) * p.Hq + h) * D;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t pk[16];
                chunk(c, pk);
                if (t < un.sq.len) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
        };
        if constexpr (C::STAGE) {
            // The last tile of a packed sequence goes out row by row: a tile
            // store would overwrite the next sequence's first rows.
            if (VAR && p.cu != nullptr && (un.m + 1) * kRows > un.sq.len) {
                store_direct();
            } else {
                // Each warp sends its own 32 rows out with its own TMA store
                // (the output map's box is kFwdOStoreRows rows), so no warp
                // waits for another; its rows of the staging block are free
                // once the warp's previous store has read them.
                if (nepi >= 1) {
                    if (lane == 0)
                        bulk_wait_read0();
                    __syncwarp();
                }
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t pk[16];
                    chunk(c, pk);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4 *>(stage + tile_chunk<D>(r, c / 8 + q)) =
                            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_4d(&tmO, smem_u32(stage + q4 * kFwdOStoreRows * TL::SWB), 0, h,
                                 un.sq.base + un.m * kRows + q4 * kFwdOStoreRows, un.sq.bc);
                    bulk_commit();
                }
                __syncwarp();
                ++nepi;
            }
        } else {
            store_direct();
        }
        return true;
    };
    for (int k = 0; ok; ++k) {
        const int u = snake_unit(k, cta, P);
        if (u >= NU)
            break;
        const FwdUnit un = fwd_unit<VAR>(u, GC, p);
        for (int jk = un.lo; jk <= un.m && ok; ++jk) {
            for (int pi = 0; pi < GC; ++pi, ++n) {
                const int pair = wg * GC + pi, hrel = pair >> 1, half = pair & 1;
                const int slot = hrel - ((wg * GC) >> 1);
                const bool first = jk == un.lo && (pi == 0 || ((pair - 1) >> 1) != hrel);
                const uint32_t b = n & 1u;
                const uint32_t s_addr = lane_base + C::COL_S + 64u * wg;
                const uint32_t p_addr = lane_base + C::COL_P + 64u * wg + 32u * b;
                if (!mbar_wait_warp(smem_u32(&bar_s_full[wg]), n & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t s[2][32];
                tmem_ld32(s_addr, s[0]);
                tmem_ld32(s_addr + 32, s[1]);
                tmem_ld_wait_only();
                tmem_tie(s[0]);
                tmem_tie(s[1]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_s_empty[wg]));

                // causal mask on the diagonal tile (key > query row); with a
                // sliding window also keys at or below row - W (local index
                // <= wlim) on the tiles the window edge crosses
                int wlim = -1;
                if constexpr (WIN)
                    wlim = un.m * kRows + r - p.window - (jk * kRows + 64 * half);
                if (jk == un.m || (WIN && __any_sync(0xffffffffu, wlim >= 0))) {
                    const int clim = (!WIN || jk == un.m) ? r - 64 * half : 1 << 30;
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (32 * c + e > clim || (WIN && 32 * c + e <= wlim))
                                s[c][e] = __float_as_uint(-INFINITY);
                }
                float mx;
                {
                    float m2[2];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        m2[c] = fmaxf(__uint_as_float(s[c][0]), __uint_as_float(s[c][1]));
#pragma unroll
                        for (int e = 2; e < 32; e += 2)
                            m2[c] = fmax3(m2[c], __uint_as_float(s[c][e]),
                                          __uint_as_float(s[c][e + 1]));
                    }
                    mx = fmaxf(m2[0], m2[1]);
                }
                const float m_tile = mx * sl2;
                // running max: moves lazily, only when it grows by more than
                // 2^8 (the final division by l makes the result exact either
                // way); a row with no visible key in its items so far keeps -inf
                float m_use = m_tile, alpha = 1.f;
                bool resc = false;
                if (!first) {
                    const float m_prev = slot ? mr1 : mr0;
                    m_use = m_prev;
                    if (m_tile > m_prev + 8.f) {
                        alpha = ex2_approx(m_prev - m_tile);
                        m_use = m_tile;
                        resc = true;
                    }
                }
                if (slot)
                    mr1 = m_use;
                else
                    mr0 = m_use;
                const float m_exp = m_use == -INFINITY ? 0.f : m_use;

                // P = 2^(S*scale*log2e - m) as bf16 pairs into P buffer b; the
                // exponent arguments and the row sum run on packed fp32 pairs
                uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
                {
                    uint32_t pk[32];
                    const uint64_t sl2x2 = f32x2(sl2, sl2), nm2 = f32x2(-m_exp, -m_exp);
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const uint64_t x2 = fma_f32x2(
                                f32x2(__uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1])),
                                sl2x2, nm2);
                            float x0, x1;
                            f32x2_split(x2, x0, x1);
                            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                            sum2[(e >> 1) & 3] = add_f32x2(sum2[(e >> 1) & 3], f32x2(p0, p1));
                            pk[16 * c + e / 2] = pack_bf16x2(p0, p1);
                        }
                    // buffer b is free once PV(n - 2) has read it
                    if (n >= 2 &&
                        !mbar_wait_warp(smem_u32(&bar_p_free[wg][b]), ((n - 2) >> 1) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tmem_st32(p_addr, pk);
                }
                float sum;
                {
                    const uint64_t s01 = add_f32x2(sum2[0], sum2[1]);
                    const uint64_t s23 = add_f32x2(sum2[2], sum2[3]);
                    float a0, a1;
                    f32x2_split(add_f32x2(s01, s23), a0, a1);
                    sum = a0 + a1;
                }
                if (__any_sync(0xffffffffu, resc)) {
                    // O_slot must hold every earlier PV of this group before it
                    // is rescaled: wait for PV(n - 1) (its commit covers all of
                    // this issuer's earlier MMAs)
                    if (!mbar_wait_warp(smem_u32(&bar_p_free[wg][(n - 1) & 1u]), ((n - 1) >> 1) & 1,
                                        wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t oa = lane_base + C::COL_O + (wg * C::NSL + slot) * D;
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(oa + c, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(oa + c, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_p_full[wg][b]));
                if (first) {
                    if (slot)
                        lr1 = sum;
                    else
                        lr0 = sum;
                } else if (slot) {
                    lr1 = fmaf(lr1, alpha, sum);
                } else {
                    lr0 = fmaf(lr0, alpha, sum);
                }
            }
        }
        if (!ok)
            break;

        // ---- end of the unit: O / l and lse of this group's heads ----
        // The split head (odd GC) is merged and stored by group k % 2, so the
        // two groups' epilogues carry the same work over consecutive units.
        // What needs only this group's running max and sum comes first, while
        // the unit's last PV may still run: the other group's half of the
        // split head is handed over, and the lse of each whole head is written.
        const int ss = wg == 0 ? C::NSL - 1 : 0;            // this group's split slot
        const int og = 1 - wg, oss = og == 0 ? C::NSL - 1 : 0;
        const bool merging = !C::SPLIT || (k & 1) == wg;
        float inv_l[C::NSL];
#pragma unroll
        for (int slot = 0; slot < C::NSL; ++slot) {
            const float m_s = slot ? mr1 : mr0, l_s = slot ? lr1 : lr0;
            inv_l[slot] = 1.f;
            if (C::SPLIT && slot == ss) {
                if (!merging) {
                    split_ml[r] = m_s;
                    split_ml[kRows + r] = l_s;
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_u32(&bar_split));
                }
            } else {
                inv_l[slot] = 1.f / l_s;
                store_lse(un, un.h0 + ((wg * GC) >> 1) + slot, m_s + __log2f(l_s));
            }
        }
        // every PV of the unit has completed once PV(n - 1) has
        if (!mbar_wait_warp(smem_u32(&bar_p_free[wg][(n - 1) & 1u]), ((n - 1) >> 1) & 1, wc)) {
            ok = false;
            break;
        }
        tc_fence_after();
        // the merging group stores its own head first
        for (int i = 0; i < C::NSL && ok; ++i) {
            int slot = i;
            if constexpr (C::SPLIT && C::NSL == 2)
                slot = (merging == (i == 1)) ? ss : 1 - ss;
            const bool split = C::SPLIT && slot == ss;
            if (split && !merging)
                continue;
            const int h = un.h0 + ((wg * GC) >> 1) + slot;
            const uint32_t oa = lane_base + C::COL_O + (wg * C::NSL + slot) * D;
            float fa = slot ? inv_l[1 % C::NSL] : inv_l[0], fb = 0.f;
            uint32_t ob = 0u;
            if (split) {
                if (!mbar_wait_warp(smem_u32(&bar_split), k & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float m_s = slot ? mr1 : mr0, l_s = slot ? lr1 : lr0;
                const float m1 = split_ml[r], l1 = split_ml[kRows + r];
                const float m_tot = fmaxf(m_s, m1);
                const float sa = ex2_approx(m_s - m_tot);
                const float sb = ex2_approx(m1 - m_tot);   // 0 when that half saw no key
                const float l_tot = fmaf(l_s, sa, l1 * sb);
                const float il = 1.f / l_tot;
                fa = sa * il;
                fb = sb * il;
                ob = lane_base + C::COL_O + (og * C::NSL + oss) * D;
                store_lse(un, h, m_tot + __log2f(l_tot));
            }
            if (!store_head(un, h, oa, split, ob, fa, fb)) {
                ok = false;
                break;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&bar_o_free[wg][slot]));
                if (split)
                    mbar_arrive(smem_u32(&bar_o_free[og][oss]));
            }
        }
    }
    if constexpr (C::STAGE) {
        if (lane == 0) {
            bulk_wait0();               // this warp's O rows are in global memory
            fence_proxy_async_global();  // and visible to the generic loads below
        }
    }
    teardown();
    const int nflag = static_cast<int>(flag_cnt < kFlagCap ? flag_cnt : kFlagCap);
    if (nflag > 0 && abort_s == 0u)
        fix_large_rows<D, GC, WIN, VAR>(reinterpret_cast<float *>(smem), flag_list, nflag, cta, P,
                                        NU, p);
}
// ------------------------------------------------------------- launch ---

template <int D, int GC, int ST, bool WIN, bool VAR>
static cudaError_t launch_fwd_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const CUtensorMap &o, const CUtensorMap &qs, const CUtensorMap &ks,
                                const AttnParams &p0, cudaStream_t stream)
{
    using C = FwdCfg<D, GC, ST>;
    auto kern = fwd_kernel<D, GC, ST, WIN, VAR>;
    static bool attr_done[64] = {};   // one flag set per template instantiation
    cudaError_t e = ensure_smem_attr(kern, C::SMEM_BYTES, attr_done);
    if (e != cudaSuccess)
        return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    AttnParams p = p0;
    if (!VAR)
        p.num_units = p.M * p.B * p.Hkv * p.nchunks;   // varlen: the table's length
    // a count in device memory is unknown here: one CTA per SM
    const int nu = (VAR && p.unit_count != nullptr) ? sms : p.num_units;
    const unsigned grid = static_cast<unsigned>(nu < sms ? nu : sms);
    return launch_pdl(kern, grid, 512, C::SMEM_BYTES, stream, q, k, v, o, qs, ks, p);
}

template <int D, int GC>
static cudaError_t launch_fwd_p(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const CUtensorMap &o, const CUtensorMap &qs, const CUtensorMap &ks,
                                const AttnParams &p, cudaStream_t stream)
{
    if (p.window > 0)
        return launch_fwd_t<D, GC, FwdPlan<D, GC>::ST, true, false>(q, k, v, o, qs, ks, p, stream);
    if (p.units)
        return launch_fwd_t<D, GC, FwdPlan<D, GC>::ST, false, true>(q, k, v, o, qs, ks, p, stream);
    return launch_fwd_t<D, GC, FwdPlan<D, GC>::ST, false, false>(q, k, v, o, qs, ks, p, stream);
}

cudaError_t launch_fwd(int d, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                       const CUtensorMap &o, const CUtensorMap &qs, const CUtensorMap &ks,
                       const AttnParams &p, cudaStream_t stream)
{
    switch (d) {
    case 32:
        switch (p.GC) {
        case 1: return launch_fwd_p<32, 1>(q, k, v, o, qs, ks, p, stream);
        case 2: return launch_fwd_p<32, 2>(q, k, v, o, qs, ks, p, stream);
        case 3: return launch_fwd_p<32, 3>(q, k, v, o, qs, ks, p, stream);
        case 4: return launch_fwd_p<32, 4>(q, k, v, o, qs, ks, p, stream);
        default: break;
        }
        break;
    case 64:
        switch (p.GC) {
        case 1: return launch_fwd_p<64, 1>(q, k, v, o, qs, ks, p, stream);
        case 2: return launch_fwd_p<64, 2>(q, k, v, o, qs, ks, p, stream);
        case 3: return launch_fwd_p<64, 3>(q, k, v, o, qs, ks, p, stream);
        default: break;
        }
        break;
    case 128:
        switch (p.GC) {
        case 1: return launch_fwd_p<128, 1>(q, k, v, o, qs, ks, p, stream);
        case 2: return launch_fwd_p<128, 2>(q, k, v, o, qs, ks, p, stream);
        default: break;
        }
        break;
    default: break;
    }
    return cudaErrorInvalidValue;
}

} // namespace ne
