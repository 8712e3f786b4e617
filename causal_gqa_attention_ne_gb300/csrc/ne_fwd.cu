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
//               (bf16 in, fp16 out), in the order the MMAs first need them.
//   warp 12     TMA producer.
//   warps 13, 14  MMA issuers of softmax groups 0 and 1 (warp 13 also
//               allocates TMEM): S(n) into the group's S buffer, then
//               PV(n - 1) reading P from the group's P buffer (n - 1) % 2.
//   warp 15     training path only: stores each rotated Q' tile and each K'
//               tile once into the backward's workspace, and tells the
//               producer when a buffer it stored from may be reloaded.
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
// stages (as many as fit, at most four), two O staging blocks (D <= 64), the
// running max / sum of a split head, and the exact-score bookkeeping of
// large-norm rows: per Q slot the ballot of its large rows and their exact
// rotated vectors, the exact vectors of one K tile's large rows, and per K
// stage a patch record (see below).
template <int D, int GC>
struct FwdPlan {
    using TL = Tile<D>;
    static constexpr bool STAGE = (D <= 64);
    static constexpr int QB = (D <= 64) ? 2 : 1;
    // large-norm rows scored exactly per Q tile and per K tile
    static constexpr int NOUT = (D == 64) ? 2 : 4;
    static constexpr int BALLOT_BYTES = 256;                    // [2][GC][4] + [ST][4] words
    static constexpr int QOV_BYTES = 2 * GC * NOUT * D * 4;     // exact q' of large rows
    static constexpr int KOV_BYTES = NOUT * D * 4;              // exact k' of large rows
    static constexpr int PHDR_BYTES = 256;                      // counts and row indices
    // per stage: header, then dS_k [NOUT][GC][128] and dS_q [GC][NOUT][128] (fp16)
    static constexpr int PREC_BYTES = PHDR_BYTES + 2 * NOUT * GC * kRows * 2;
    static constexpr int fixed_bytes()
    {
        return QB * GC * TL::BYTES + (STAGE ? 2 * TL::BLOCK : 0) + 2 * kRows * 4 + BALLOT_BYTES +
               QOV_BYTES + KOV_BYTES + 1024;
    }
    static constexpr int stages()
    {
        int st = 4;
        while (st > 1 && fixed_bytes() + st * (2 * TL::BYTES + PREC_BYTES) > 232448 - 1024)
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
    static constexpr int NOUT = PL::NOUT;
    static constexpr int OFF_Q = 0;                          // [QB][GC] tiles
    static constexpr int OFF_K = OFF_Q + QB * GC * TL::BYTES;
    static constexpr int OFF_V = OFF_K + ST * TL::BYTES;
    static constexpr int OFF_O = OFF_V + ST * TL::BYTES;      // [2] staging blocks
    // group 1's running max and sum of the split head: float [2][128]
    static constexpr int OFF_SPL = OFF_O + (STAGE ? 2 * TL::BLOCK : 0);
    // uint32 ballots of large rows (one word per RoPE warp): the Q tiles of
    // units of each parity [2][GC][4], then the K stages [ST][4]
    static constexpr int OFF_BAL = OFF_SPL + 2 * kRows * 4;
    static constexpr int OFF_QOV = OFF_BAL + PL::BALLOT_BYTES;   // float [2][GC][NOUT][D]
    static constexpr int OFF_KOV = OFF_QOV + PL::QOV_BYTES;      // float [NOUT][D]
    static constexpr int OFF_PREC = OFF_KOV + PL::KOV_BYTES;     // [ST] patch records
    static constexpr int SMEM_BYTES = smem_one_cta(OFF_PREC + ST * PL::PREC_BYTES + 1024);
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
    static_assert(2 * GC * 4 * 4 + ST * 4 * 4 <= PL::BALLOT_BYTES, "ballot words");
    static_assert(4 * (1 + NOUT + GC + GC * NOUT) <= PL::PHDR_BYTES, "patch record header");
};

// Patch record of one K stage, written by the RoPE warpgroup once it has
// rotated the stage's K tile, read by the softmax groups for every item of
// that tile.  A row whose rotated vector has mean square above 2 (sum of
// squares > 2 D) is "large": its scores' fp16 rounding error, proportional to
// |q'||k'|, would exceed what the 1e-3 lse tolerance allows.  For the pairs
// with a large key row (column kcol[i] of the tile) or a large query row
// (row qrow[g][i] of head g's Q tile) the record holds
//   delta = <q', k'> exact (fp32 from the bf16 inputs) - <fp16 q', fp16 k'>
// which the softmax thread adds to the score the tensor cores computed from
// the fp16 operands.
struct PatchHdr {
    int kcnt;        // large key rows in the tile (<= NOUT)
    int qcnt[4];     // per head of the unit: large query rows (<= NOUT)
    int kcol[4];     // their key indices in the tile
    int qrow[4][4];  // [head][i]: their row indices in the Q tile
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


// ---------------------------------------------- exact scores of large rows ---

// The rotated row of the bf16 vector at `row` (global memory) in fp32:
// f(i, x'_i, x'_{i + D/2}) for every rotate-half pair i, position pos.  One
// pair per iteration, so the few registers of the RoPE warps suffice (this
// runs only for tiles with large rows).
template <int D, typename F>
__device__ __forceinline__ void exact_pairs(const __nv_bfloat16 *row, uint32_t pos,
                                            const RopeFreqs &fr, F &&f)
{
#pragma unroll 1
    for (int i = 0; i < D / 2; ++i) {
        float sn, cs;
        rope_sincos(pos, fr, i, sn, cs);
        const float x = __bfloat162float(row[i]);
        const float y = __bfloat162float(row[i + D / 2]);
        float u, w;
        rope_rotate(x, y, cs, sn, u, w);
        f(i, u, w);
    }
}

// Element (r, col) of a rotated fp16 tile in shared memory.
template <int D>
__device__ __forceinline__ float tile_f16(const uint8_t *tile, int r, int col)
{
    return __half2float(
        *reinterpret_cast<const __half *>(tile + tile_chunk<D>(r, col >> 3) + (col & 7) * 2));
}

// Row index (32 w + lane) of the o-th set bit of four ballot words, in
// increasing row order; -1 if there are not that many.
__device__ __forceinline__ int nth_row(const uint32_t *bal, int o)
{
    for (int w = 0; w < 4; ++w) {
        uint32_t m = bal[w];
        const int c = __popc(m);
        if (o < c) {
            for (int i = 0; i < o; ++i)
                m &= m - 1u;
            return 32 * w + __ffs(m) - 1;
        }
        o -= c;
    }
    return -1;
}

// Rank of row r among the set bits of four ballot words (rows below it), or
// -1 if its bit is clear.
__device__ __forceinline__ int row_rank(const uint32_t *bal, int r)
{
    const int wr = r >> 5;
    if (!((bal[wr] >> (r & 31)) & 1u))
        return -1;
    int rank = __popc(bal[wr] & ((1u << (r & 31)) - 1u));
    for (int i = 0; i < wr; ++i)
        rank += __popc(bal[i]);
    return rank;
}

// Builds the patch record of K stage st (key tile jk of unit w, whose Q
// tiles sit in slot qslot and whose ballots are those of unit parity up).
// Runs in all 128 threads of the RoPE warpgroup after the ballots of the K
// tile are visible; thread r stands for query row r of the Q tiles and key
// row r of the K tile.  Without large rows it only clears the counts.
template <int D, int GC, int ST, bool VAR, typename Sync>
__device__ __forceinline__ bool patch_tile(uint8_t *smem, int r, int st, int jk, const FwdUnit &w,
                                        int qslot, int up, const uint32_t *qbal,
                                        const uint32_t *kbal, const AttnParams &p, Sync &rsync)
{
    using C = FwdCfg<D, GC, ST>;
    using TL = Tile<D>;
    constexpr int NOUT = C::NOUT;
    uint8_t *rec = smem + C::OFF_PREC + st * C::PL::PREC_BYTES;
    PatchHdr *hdr = reinterpret_cast<PatchHdr *>(rec);
    __half *dk = reinterpret_cast<__half *>(rec + C::PL::PHDR_BYTES);   // [NOUT][GC][128]
    __half *dq = dk + NOUT * GC * kRows;                               // [GC][NOUT][128]
    const uint32_t *kb = kbal + st * 4;
    const uint32_t *qb0 = qbal + up * GC * 4;
    const int nk = __popc(kb[0]) + __popc(kb[1]) + __popc(kb[2]) + __popc(kb[3]);
    int anyq = 0, overq = 0;
#pragma unroll
    for (int g = 0; g < GC; ++g) {
        const uint32_t *qg = qb0 + g * 4;
        const int n = __popc(qg[0]) + __popc(qg[1]) + __popc(qg[2]) + __popc(qg[3]);
        anyq |= n;
        overq |= n > NOUT ? 1 : 0;
    }
    if (nk == 0 && anyq == 0) {
        if (r == 0) {
            hdr->kcnt = 0;
#pragma unroll
            for (int g = 0; g < GC; ++g)
                hdr->qcnt[g] = 0;
        }
        return true;
    }
    // ---- a tile with large rows: exact scores for their pairs ----
    const int kc = nk < NOUT ? nk : NOUT;
    if (r == 0 && (nk > NOUT || overq))
        atomicOr(p.status, kDevPrecision);
    const uint8_t *ktile = smem + C::OFF_K + st * TL::BYTES;
    float *kov = reinterpret_cast<float *>(smem + C::OFF_KOV);                        // [NOUT][D]
    float *qov = reinterpret_cast<float *>(smem + C::OFF_QOV) + up * GC * NOUT * D;   // [GC][NOUT][D]
    const __nv_bfloat16 *qin = static_cast<const __nv_bfloat16 *>(p.q_in);
    const __nv_bfloat16 *kin = static_cast<const __nv_bfloat16 *>(p.k_in);
    const int t = w.m * kRows + r;   // this thread's query row
    const int s = jk * kRows + r;    // this thread's key row
    const __nv_bfloat16 *krow = kin + (seq_row(p, w.sq, s) * p.Hkv + w.j) * D;
    auto qrow_ptr = [&](int g) { return qin + (seq_row(p, w.sq, t) * p.Hq + w.h0 + g) * D; };
    // 1. the owners of large rows write their exact rotated vectors
    const int krank = row_rank(kb, r);
    if (krank >= 0 && krank < NOUT)
        exact_pairs<D>(krow, static_cast<uint32_t>(s), p.rope, [&](int i, float x, float y) {
            kov[krank * D + i] = x;
            kov[krank * D + i + D / 2] = y;
        });
#pragma unroll 1
    for (int g = 0; g < GC; ++g) {
        const int qrank = row_rank(qb0 + g * 4, r);
        if (qrank >= 0 && qrank < NOUT) {
            float *dst = qov + (g * NOUT + qrank) * D;
            exact_pairs<D>(qrow_ptr(g), static_cast<uint32_t>(t), p.rope,
                           [&](int i, float x, float y) {
                               dst[i] = x;
                               dst[i + D / 2] = y;
                           });
        }
    }
    if (!rsync())
        return false;
    if (r == 0) {
        hdr->kcnt = kc;
        for (int o = 0; o < kc; ++o)
            hdr->kcol[o] = nth_row(kb, o);
        for (int g = 0; g < GC; ++g) {
            const uint32_t *qg = qb0 + g * 4;
            const int n = __popc(qg[0]) + __popc(qg[1]) + __popc(qg[2]) + __popc(qg[3]);
            hdr->qcnt[g] = n < NOUT ? n : NOUT;
            for (int o = 0; o < NOUT && o < n; ++o)
                hdr->qrow[g][o] = nth_row(qg, o);
        }
    }
    float dmax = 0.f;
    // 2. pairs (query row r, large key o), every head: the exact score minus
    //    the product of the fp16 operands the tensor cores see.  One pair
    //    list entry at a time, so few registers stay live.
#pragma unroll 1
    for (int g = 0; g < GC; ++g) {
        const uint8_t *qtile = smem + C::OFF_Q + (qslot * GC + g) * TL::BYTES;
#pragma unroll 1
        for (int o = 0; o < kc; ++o) {
            const int kr = nth_row(kb, o);
            const float *kv = kov + o * D;
            float ae = 0.f, ah = 0.f;
            if (t < w.sq.len)
                exact_pairs<D>(qrow_ptr(g), static_cast<uint32_t>(t), p.rope,
                               [&](int i, float x, float y) {
                                   ae = fmaf(x, kv[i], fmaf(y, kv[i + D / 2], ae));
                                   ah = fmaf(tile_f16<D>(qtile, r, i), tile_f16<D>(ktile, kr, i),
                                             fmaf(tile_f16<D>(qtile, r, i + D / 2),
                                                  tile_f16<D>(ktile, kr, i + D / 2), ah));
                               });
            dmax = fmaxf(dmax, fabsf(ae - ah));
            dk[(o * GC + g) * kRows + r] = __float2half_rn(ae - ah);
        }
    }
    // 3. pairs (large query row o of head g, key row r); a key that is itself
    //    corrected in step 2 gets 0 here, so no pair is corrected twice
    const bool key_patched = krank >= 0 && krank < NOUT;
#pragma unroll 1
    for (int g = 0; g < GC; ++g) {
        const uint32_t *qg = qb0 + g * 4;
        const int n = __popc(qg[0]) + __popc(qg[1]) + __popc(qg[2]) + __popc(qg[3]);
        const int qc = n < NOUT ? n : NOUT;
        const uint8_t *qtile = smem + C::OFF_Q + (qslot * GC + g) * TL::BYTES;
#pragma unroll 1
        for (int o = 0; o < qc; ++o) {
            const int qr = nth_row(qg, o);
            const float *qv = qov + (g * NOUT + o) * D;
            float ae = 0.f, ah = 0.f;
            if (s < w.sq.len && !key_patched)
                exact_pairs<D>(krow, static_cast<uint32_t>(s), p.rope,
                               [&](int i, float x, float y) {
                                   ae = fmaf(x, qv[i], fmaf(y, qv[i + D / 2], ae));
                                   ah = fmaf(tile_f16<D>(ktile, r, i), tile_f16<D>(qtile, qr, i),
                                             fmaf(tile_f16<D>(ktile, r, i + D / 2),
                                                  tile_f16<D>(qtile, qr, i + D / 2), ah));
                               });
            dmax = fmaxf(dmax, fabsf(ae - ah));
            dq[(g * NOUT + o) * kRows + r] = __float2half_rn(ae - ah);
        }
    }
    if (dmax > kFp16Max)
        atomicOr(p.status, kDevRange);
    return true;
}

// Adds a K stage's exact-score corrections to the 64 raw scores a softmax
// thread holds for query row r and key half `half` of head hrel: the column
// of every large key row in this half, and every column if r is a large
// query row of that head.
template <int NOUT, int GC>
__device__ __forceinline__ void apply_patches(uint32_t (&s)[2][32], const uint8_t *deltas,
                                              const PatchHdr *hdr, int kc, int qc, int hrel,
                                              int half, int r)
{
    const __half *dk = reinterpret_cast<const __half *>(deltas);   // [NOUT][GC][128]
    const __half *dq = dk + NOUT * GC * kRows;                     // [GC][NOUT][128]
    for (int o = 0; o < kc; ++o) {
        const int col = hdr->kcol[o] - 64 * half;
        if (col < 0 || col >= 64)
            continue;
        const float d = __half2float(dk[(o * GC + hrel) * kRows + r]);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (32 * c + e == col)
                    s[c][e] = __float_as_uint(__uint_as_float(s[c][e]) + d);
    }
    for (int o = 0; o < qc; ++o) {
        if (hdr->qrow[hrel][o] != r)
            continue;
        const __half *row = dq + (hrel * NOUT + o) * kRows + 64 * half;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
                s[c][e] = __float_as_uint(__uint_as_float(s[c][e]) + __half2float(row[32 * c + e]));
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
    __shared__ uint64_t bar_stg_full[2], bar_stg_free[2];
    // training path: the RoPE warps finished the n-th tile to be stored
    // (ring of 16: they are never 16 such tiles ahead of warp 15, which must
    // release a Q slot or a stored K stage before it is reloaded), and warp
    // 15's store has read a Q slot / K stage
    __shared__ uint64_t bar_sv[16], bar_q_rd[QB][GC], bar_k_rd[ST];
    // patch record of stage st written (four RoPE warps); barrier of the RoPE
    // warpgroup for the exact-score path
    __shared__ uint64_t bar_patch[ST], bar_rsync;
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
            mbar_init(smem_u32(&bar_patch[s]), 4);
        }
        mbar_init(smem_u32(&bar_rsync), 4);
        for (int w = 0; w < 2; ++w) {
            mbar_init(smem_u32(&bar_s_full[w]), 1);
            mbar_init(smem_u32(&bar_s_empty[w]), 4);
            for (int b = 0; b < 2; ++b) {
                mbar_init(smem_u32(&bar_p_full[w][b]), 4);
                mbar_init(smem_u32(&bar_p_free[w][b]), 1);
            }
            for (int sl = 0; sl < C::NSL; ++sl)
                mbar_init(smem_u32(&bar_o_free[w][sl]), 4);
            mbar_init(smem_u32(&bar_stg_full[w]), 4);
            mbar_init(smem_u32(&bar_stg_free[w]), 1);
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
            auto load_q = [&](int kk) {
                const FwdUnit w = fwd_unit<VAR>(snake_unit(kk, cta, P), GC, p);
                const int qb = kk % QB, use = kk / QB;
                for (int g = 0; g < GC; ++g) {
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
                if (u >= p.num_units)
                    break;
                const FwdUnit w = fwd_unit<VAR>(u, GC, p);
                // order: [Q of this unit if not prefetched], K/V lo, [Q of the
                // next unit], K/V lo+1..m
                if (QB == 1 || k == 0)
                    ok = load_q(k);
                ok = ok && load_kv(w, w.lo);
                if (QB == 2 && ok && snake_unit(k + 1, cta, P) < p.num_units)
                    ok = load_q(k + 1);
                for (int jk = w.lo + 1; jk <= w.m && ok; ++jk)
                    ok = load_kv(w, jk);
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
                if (u >= p.num_units)
                    break;
                const FwdUnit w = fwd_unit<VAR>(u, GC, p);
                const int nq0 = (QB == 1 || k == 0) ? GC : 0;
                const bool has_next = QB == 2 && snake_unit(k + 1, cta, P) < p.num_units;
                const int nq1 = has_next ? GC : 0;
                for (int t = 0; t < nq0 + 1 + nq1 + w.m - w.lo && ok; ++t) {
                    const bool isq = t < nq0 || (t > nq0 && t <= nq0 + nq1);
                    const int qunit = t < nq0 ? k : k + 1;
                    const int g = t < nq0 ? t : t - nq0 - 1;
                    const int jk = w.lo + (t == nq0 ? 0 : t - nq0 - nq1);
                    const int qb = qunit % QB, st = kt % ST;
                    if (!isq)
                        ++kt;
                    if (!isq && !(jk == w.m && w.h0 == w.j * p.G))
                        continue;   // this K' tile is stored by its diagonal unit
                    if (!mbar_wait_warp(smem_u32(&bar_sv[nsv % 16]), (nsv / 16) & 1, wc)) {
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
                if (u >= p.num_units)
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
        const int rw = warp - 8;              // warp within the RoPE warpgroup
        uint32_t *qbal = reinterpret_cast<uint32_t *>(smem + C::OFF_BAL);   // [2][GC][4]
        uint32_t *kbal = qbal + 2 * GC * 4;                                  // [ST][4]
        float mx = 0.f;
        bool ok = true;
        int kt = 0;
        uint32_t nsv = 0;     // tiles handed to warp 15 (training path)
        uint32_t nsync = 0;   // uses of bar_rsync
        // bounded barrier of the four RoPE warps (all take the same path)
        auto rsync = [&]() {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_rsync));
            const bool r_ok = mbar_wait_warp(smem_u32(&bar_rsync), nsync & 1, wc);
            ++nsync;
            return r_ok;
        };
        for (int k = 0; ok; ++k) {
            const int u = snake_unit(k, cta, P);
            if (u >= p.num_units)
                break;
            const FwdUnit w = fwd_unit<VAR>(u, GC, p);
            // Tiles in the order the producer loads them: [Q of this unit
            // unless prefetched], K 0, [Q of the next unit], K 1..m.  One call
            // site keeps the unrolled rotation in the instruction cache once.
            const int nq0 = (QB == 1 || k == 0) ? GC : 0;
            const bool has_next = QB == 2 && snake_unit(k + 1, cta, P) < p.num_units;
            const int nq1 = has_next ? GC : 0;
            const FwdUnit wn = has_next ? fwd_unit<VAR>(snake_unit(k + 1, cta, P), GC, p) : w;
            for (int t = 0; t < nq0 + 1 + nq1 + w.m - w.lo && ok; ++t) {
                const bool isq = t < nq0 || (t > nq0 && t <= nq0 + nq1);
                const int qunit = t < nq0 ? k : k + 1;
                const int g = t < nq0 ? t : t - nq0 - 1;
                const int jk = w.lo + (t == nq0 ? 0 : t - nq0 - nq1);
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
                // rows whose rotated vector is large get exact scores
                const int limit = tu.sq.len;
                const uint32_t bal =
                    __ballot_sync(0xffffffffu, static_cast<int>(pos) < limit && ss > 2.f * D);
                if (lane == 0) {
                    if (isq)
                        qbal[((qunit & 1) * GC + g) * 4 + rw] = bal;
                    else
                        kbal[st * 4 + rw] = bal;
                }
                __syncwarp();
                const uint32_t ready =
                    isq ? smem_u32(&bar_q_ready[qb][g]) : smem_u32(&bar_k_ready[st]);
                if (lane == 0)
                    mbar_arrive(ready);
                if (p.save_rot && (isq || (jk == w.m && w.h0 == w.j * p.G))) {
                    if (lane == 0)
                        mbar_arrive(smem_u32(&bar_sv[nsv % 16]));
                    ++nsv;
                }
                if (!isq) {
                    // k_ready completes once all four warps have rotated the
                    // tile and posted their ballots
                    if (!mbar_wait_warp(smem_u32(&bar_k_ready[st]), (kt / ST) & 1, wc) ||
                        !patch_tile<D, GC, ST, VAR>(smem, r, st, jk, w, k % QB, k & 1, qbal, kbal,
                                                    p, rsync)) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_u32(&bar_patch[st]));
                    ++kt;
                }
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
    const int r = threadIdx.x & 127;        // query row == TMEM lane
    const uint32_t lane_base = tmem_addr(tbase, q4 * 32, 0);
    const float sl2 = p.scale_log2;
    uint8_t *stage = smem + C::OFF_O + wg * TL::BLOCK;
    float *split_ml = reinterpret_cast<float *>(smem + C::OFF_SPL);   // [m | l][row]
    bool ok = true;
    uint32_t n = 0;          // this group's items so far
    uint32_t kts = 0;        // key tiles this group has started (K stage kts % ST)
    uint32_t nepi = 0;       // O stores this group has issued
    float mr0 = 0.f, mr1 = 0.f, lr0 = 0.f, lr1 = 0.f;   // running max (log2 units) / sum per slot
    // Writes O_slot / l of head h (rows of this thread) and its lse.  With a
    // second accumulator (merge), O = (O_a * sa + O_b * sb) * inv_l.
    auto store_head = [&](const FwdUnit &un, int h, uint32_t oa, bool merge, uint32_t ob, float sa,
                          float sb, float inv_l, float lse2) -> bool {
        const int t = un.m * kRows + r;
        // O row by row from registers (rows past the sequence skipped)
        auto store_direct = [&]() {
            __nv_bfloat16 *dst =
                static_cast<__nv_bfloat16 *>(p.out0) + (seq_row(p, un.sq, t) * p.Hq + h) * D;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tmem_ld32(oa + c, o);
                tmem_ld_wait(o);
                float x[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    x[e] = __uint_as_float(o[e]) * sa;
                if (merge) {
                    tmem_ld32(ob + c, o);
                    tmem_ld_wait(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        x[e] = fmaf(__uint_as_float(o[e]), sb, x[e]);
                }
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    x[e] *= inv_l;
                if (t < un.sq.len)
                    store_row32_bf16(dst + c, x);
            }
        };
        if constexpr (C::STAGE) {
            // The last tile of a packed sequence goes out row by row: a tile
            // store would overwrite the next sequence's first rows.
            if (VAR && p.cu != nullptr && (un.m + 1) * kRows > un.sq.len) {
                store_direct();
            } else {
                // the staging block is free once this group's previous store
                // has read it
                if (nepi >= 1) {
                    if (warp == 4 * wg && lane == 0) {
                        bulk_wait_read0();
                        mbar_arrive(smem_u32(&bar_stg_free[wg]));
                    }
                    if (!mbar_wait_warp(smem_u32(&bar_stg_free[wg]), (nepi - 1) & 1, wc))
                        return false;
                }
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(oa + c, o);
                    tmem_ld_wait(o);
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        x[e] = __uint_as_float(o[e]) * sa;
                    if (merge) {
                        tmem_ld32(ob + c, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            x[e] = fmaf(__uint_as_float(o[e]), sb, x[e]);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4 *>(stage + tile_chunk<D>(r, c / 8 + q)) =
                            make_uint4(pack_bf16x2(x[8 * q + 0] * inv_l, x[8 * q + 1] * inv_l),
                                       pack_bf16x2(x[8 * q + 2] * inv_l, x[8 * q + 3] * inv_l),
                                       pack_bf16x2(x[8 * q + 4] * inv_l, x[8 * q + 5] * inv_l),
                                       pack_bf16x2(x[8 * q + 6] * inv_l, x[8 * q + 7] * inv_l));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_stg_full[wg]));
                if (warp == 4 * wg) {
                    if (!mbar_wait_warp(smem_u32(&bar_stg_full[wg]), nepi & 1, wc))
                        return false;
                    if (lane == 0) {
                        tma_store_4d(&tmO, smem_u32(stage), 0, h, un.sq.base + un.m * kRows,
                                     un.sq.bc);
                        bulk_commit();
                    }
                    __syncwarp();
                }
                ++nepi;
            }
        } else {
            store_direct();
        }
        if (t < un.sq.len)
            p.lse[(static_cast<size_t>(un.sq.bc) * p.Hq + h) * p.T + un.sq.base + t] = lse2 * kLn2;
        return true;
    };
    for (int k = 0; ok; ++k) {
        const int u = snake_unit(k, cta, P);
        if (u >= p.num_units)
            break;
        const FwdUnit un = fwd_unit<VAR>(u, GC, p);
        for (int jk = un.lo; jk <= un.m && ok; ++jk, ++kts) {
            // the K stage's patch record (exact scores of large rows): its
            // counts are read once per key tile
            const int pst = kts % ST;
            if (!mbar_wait_warp(smem_u32(&bar_patch[pst]), (kts / ST) & 1, wc)) {
                ok = false;
                break;
            }
            const uint8_t *prec = smem + C::OFF_PREC + pst * C::PL::PREC_BYTES;
            const PatchHdr *phdr = reinterpret_cast<const PatchHdr *>(prec);
            const int pkc = phdr->kcnt;
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
                const int pqc = phdr->qcnt[hrel];
                if (pkc > 0 || pqc > 0)
                    apply_patches<C::NOUT, GC>(s, prec + C::PL::PHDR_BYTES, phdr, pkc, pqc, hrel,
                                               half, r);

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
        // every PV of the unit has completed once PV(n - 1) has
        if (!mbar_wait_warp(smem_u32(&bar_p_free[wg][(n - 1) & 1u]), ((n - 1) >> 1) & 1, wc)) {
            ok = false;
            break;
        }
        tc_fence_after();
        // The split head (odd GC) is merged and stored by group k % 2, so the
        // two groups' epilogues carry the same work over consecutive units;
        // the merging group stores its own head first, the other group
        // publishes its half first.
        const int ss = wg == 0 ? C::NSL - 1 : 0;            // this group's split slot
        const int og = 1 - wg, oss = og == 0 ? C::NSL - 1 : 0;
        const bool merging = !C::SPLIT || (k & 1) == wg;
        for (int i = 0; i < C::NSL && ok; ++i) {
            int slot = i;
            if constexpr (C::SPLIT && C::NSL == 2)
                slot = (merging == (i == 1)) ? ss : 1 - ss;
            const int h = un.h0 + ((wg * GC) >> 1) + slot;
            const float m_s = slot ? mr1 : mr0, l_s = slot ? lr1 : lr0;
            const uint32_t oa = lane_base + C::COL_O + (wg * C::NSL + slot) * D;
            const bool split = C::SPLIT && slot == ss;
            if (split && !merging) {
                // hand this half's max and sum to the merging group
                split_ml[r] = m_s;
                split_ml[kRows + r] = l_s;
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_split));
                continue;
            }
            float sa = 1.f, sb = 0.f, l_tot = l_s, m_tot = m_s;
            uint32_t ob = 0u;
            if (split) {
                if (!mbar_wait_warp(smem_u32(&bar_split), k & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float m1 = split_ml[r], l1 = split_ml[kRows + r];
                m_tot = fmaxf(m_s, m1);
                sa = ex2_approx(m_s - m_tot);
                sb = ex2_approx(m1 - m_tot);   // 0 when that half saw no key
                l_tot = fmaf(l_s, sa, l1 * sb);
                ob = lane_base + C::COL_O + (og * C::NSL + oss) * D;
            }
            const float inv_l = 1.f / l_tot;
            if (!store_head(un, h, oa, split, ob, sa, sb, inv_l, m_tot + __log2f(l_tot))) {
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
        if (warp == 4 * wg && lane == 0)
            bulk_wait0();
    }
    teardown();
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
    const unsigned grid = static_cast<unsigned>(p.num_units < sms ? p.num_units : sms);
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
