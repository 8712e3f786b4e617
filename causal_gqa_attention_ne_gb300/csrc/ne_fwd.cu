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
// an "item" is (jk, half, g), numbered gi across the CTA's lifetime.  Each
// K/V tile is loaded once by TMA, rotated once and used by all GC heads.
// Warp roles (512 threads):
//   warps 0-3, 4-7  two softmax warpgroups in ping-pong: warpgroup w takes
//               the items with gi % 2 == w, thread r owns query row r (TMEM
//               lane r) of the item's 128 x 64 score block.  S buffers are
//               released as soon as the group has loaded them, so the S
//               issuer runs up to NSB items ahead, and each group writes P
//               into a P buffer of its own, so one group's exponentials
//               overlap the other's TMEM traffic and the MMAs.  The running max and sum
//               of (head g, row r) live in shared memory; when GC is odd a
//               head's consecutive items belong to different groups and the
//               two values pass between them through mbarriers.  The running
//               max moves lazily (only when it grows by more than 2^8; the
//               final division by l makes the result exact either way), and
//               the group that raises it rescales that head's O row in TMEM.
//               The group that finishes the last item of a head writes O / l
//               (through shared memory and a TMA store) and lse.
//   warps 8-11  RoPE: rotate the unit's Q tiles and each K tile in place
//               (bf16 in, fp16 out), in the order the MMAs first need them.
//   warp 12     TMA producer.   warp 13  TMEM allocator + S issuer.
//   warp 14     PV issuer.
//   warp 15     training path only: stores each rotated Q' tile and each K'
//               tile once into the backward's workspace, and tells the
//               producer when a buffer it stored from may be reloaded.
// TMEM: NSB S buffers of 64 columns (item gi uses gi % NSB), two P buffers
// of 32 columns (bf16 pairs; group w uses P_w), then O of head g at
// COL_O + g*D.
#include <cuda_bf16.h>

#include "ne_common.cuh"
#include "ne_kernels.h"

namespace ne {

// Shared-memory plan: QB Q-tile sets of GC heads (two for D <= 64, so the
// next unit's Q' is loaded and rotated while the current unit runs), ST K/V
// stages (as many as fit, at most four), two O staging blocks (D <= 64), the
// running max / sum.
template <int D, int GC>
struct FwdPlan {
    using TL = Tile<D>;
    static constexpr bool STAGE = (D <= 64);
    static constexpr int QB = (D <= 64) ? 2 : 1;
    static constexpr int fixed_bytes()
    {
        return QB * GC * TL::BYTES + (STAGE ? 2 * TL::BLOCK : 0) + 2 * GC * kRows * 4 + 1024;
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
    static constexpr bool STAGE = FwdPlan<D, GC>::STAGE;     // O leaves by TMA store
    static constexpr int QB = FwdPlan<D, GC>::QB;
    static constexpr int OFF_Q = 0;                          // [QB][GC] tiles
    static constexpr int OFF_K = OFF_Q + QB * GC * TL::BYTES;
    static constexpr int OFF_V = OFF_K + ST * TL::BYTES;
    static constexpr int OFF_O = OFF_V + ST * TL::BYTES;      // [2] staging blocks
    static constexpr int OFF_M = OFF_O + (STAGE ? 2 * TL::BLOCK : 0);   // float [GC][128]
    static constexpr int OFF_L = OFF_M + GC * kRows * 4;                // float [GC][128]
    static constexpr int SMEM_BYTES = smem_one_cta(OFF_L + GC * kRows * 4 + 1024);
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int NSB = (512 - 64 - GC * D) / 64 < 4 ? (512 - 64 - GC * D) / 64 : 4;
    static constexpr uint32_t COL_P = 64 * NSB;
    static constexpr uint32_t COL_O = COL_P + 64;
    static_assert(NSB >= 2, "at least two S buffers");
    static_assert(COL_O + GC * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448 - 1024, "shared memory budget");
    static_assert(ST >= 2, "K/V double buffering");
    static_assert(!STAGE || TL::NB == 1, "staged epilogue stores one column block per head");
};

struct FwdUnit {
    int m, b, j, h0;
};

__device__ __forceinline__ FwdUnit fwd_unit(int u, int GC, const AttnParams &p)
{
    FwdUnit w;
    const int per_m = p.B * p.Hkv * p.nchunks;
    w.m = p.M - 1 - u / per_m;
    int rem = u % per_m;
    const int chunk = rem % p.nchunks;
    rem /= p.nchunks;
    w.j = rem % p.Hkv;
    w.b = rem / p.Hkv;
    w.h0 = w.j * p.G + chunk * GC;
    return w;
}

template <int D, int GC, int ST>
__global__ void __launch_bounds__(512, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
               const __grid_constant__ CUtensorMap tmQs, const __grid_constant__ CUtensorMap tmKs,
               const AttnParams p)
{
    using C = FwdCfg<D, GC, ST>;
    using TL = Tile<D>;
    constexpr bool ODD = (GC & 1) != 0;   // a head's items alternate between the groups
    constexpr int IPT = 2 * GC;           // items per key tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    constexpr int QB = C::QB;
    __shared__ uint64_t bar_q_full[QB][GC], bar_q_ready[QB][GC], bar_q_empty[QB][GC];
    __shared__ uint64_t bar_k_full[ST], bar_k_ready[ST], bar_v_full[ST], bar_kv_empty[ST];
    constexpr int NSB = C::NSB;
    __shared__ uint64_t bar_s_full[NSB], bar_s_empty[NSB], bar_p_full[2], bar_p_empty[2];
    __shared__ uint64_t bar_o_free[GC], bar_drain;
    // hand-off of the running max / sum: group w's n-th item arrives on
    // [w][n % 3] (a group is never more than two items past the one its
    // partner waits for, so the parity of n / 3 is unambiguous)
    __shared__ uint64_t bar_hm[2][3], bar_hl[2][3];
    __shared__ uint64_t bar_stg_full[2], bar_stg_free[2];
    // training path: the RoPE warps finished the n-th tile to be stored
    // (ring of 16: they are never 16 such tiles ahead of warp 15, which must
    // release a Q slot or a stored K stage before it is reloaded), and warp
    // 15's store has read a Q slot / K stage
    __shared__ uint64_t bar_sv[16], bar_q_rd[QB][GC], bar_k_rd[ST];
    __shared__ uint32_t tmem_base_s;
    __shared__ uint32_t abort_s;
    float *mrun = reinterpret_cast<float *>(smem + C::OFF_M);   // [g][row], log2 units
    float *lrun = reinterpret_cast<float *>(smem + C::OFF_L);   // [g][row]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cta = static_cast<int>(blockIdx.x), P = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        abort_s = 0;
        for (int g = 0; g < GC; ++g) {
            for (int qb = 0; qb < QB; ++qb) {
                mbar_init(smem_u32(&bar_q_full[qb][g]), 1);
                mbar_init(smem_u32(&bar_q_ready[qb][g]), 4);
                mbar_init(smem_u32(&bar_q_empty[qb][g]), 1);
                mbar_init(smem_u32(&bar_q_rd[qb][g]), 1);
            }
            mbar_init(smem_u32(&bar_o_free[g]), 4);
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&bar_k_full[s]), 1);
            mbar_init(smem_u32(&bar_k_ready[s]), 4);
            mbar_init(smem_u32(&bar_v_full[s]), 1);
            mbar_init(smem_u32(&bar_kv_empty[s]), 1);
            mbar_init(smem_u32(&bar_k_rd[s]), 1);
        }
        for (int b = 0; b < NSB; ++b) {
            mbar_init(smem_u32(&bar_s_full[b]), 1);
            mbar_init(smem_u32(&bar_s_empty[b]), 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_p_full[b]), 4);
            mbar_init(smem_u32(&bar_p_empty[b]), 1);
        }
        for (int w = 0; w < 2; ++w) {
            for (int i = 0; i < 3; ++i) {
                mbar_init(smem_u32(&bar_hm[w][i]), 4);
                mbar_init(smem_u32(&bar_hl[w][i]), 4);
            }
            mbar_init(smem_u32(&bar_stg_full[w]), 4);
            mbar_init(smem_u32(&bar_stg_free[w]), 1);
        }
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
        if (warp == 12 && lane == 0) {
            // ------------------------------------------------ TMA producer ---
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            bool ok = true;
            int kt = 0;
            int qloads[QB][GC] = {};   // loads issued per Q slot (for the abort drain)
            // Q' tiles of unit kk into set kk % QB, once the set's previous
            // unit has issued its last S
            auto load_q = [&](int kk) {
                const FwdUnit w = fwd_unit(snake_unit(kk, cta, P), GC, p);
                const int qb = kk % QB, use = kk / QB;
                for (int g = 0; g < GC; ++g) {
                    if (use >= 1 && !mbar_wait(smem_u32(&bar_q_empty[qb][g]), (use - 1) & 1, wc))
                        return false;
                    // training path: the previous tile of this slot was stored
                    if (p.save_rot && use >= 1 &&
                        !mbar_wait(smem_u32(&bar_q_rd[qb][g]), (use - 1) & 1, wc))
                        return false;
                    const uint32_t bar = smem_u32(&bar_q_full[qb][g]);
                    mbar_arrive_expect_tx(bar, TL::BYTES);
                    for (int cb = 0; cb < TL::NB; ++cb)
                        tma_load_4d(smem_u32(smem + C::OFF_Q + (qb * GC + g) * TL::BYTES +
                                             cb * TL::BLOCK),
                                    &tmQ, bar, cb * TL::BOX_COLS, w.h0 + g, w.m * kRows, w.b);
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
                if (u2 >= 1 && !mbar_wait(smem_u32(&bar_kv_empty[st]), (u2 - 1) & 1, wc))
                    return false;
                if (((last_saved >> st) & 1u) &&
                    !mbar_wait(smem_u32(&bar_k_rd[st]), (ksaved[st] - 1) & 1, wc))
                    return false;
                const bool saved = p.save_rot && jk == w.m && w.h0 == w.j * p.G;
                last_saved = (last_saved & ~(1u << st)) | (saved ? 1u << st : 0u);
                ksaved[st] += saved ? 1 : 0;
                const uint32_t kb = smem_u32(&bar_k_full[st]), vb = smem_u32(&bar_v_full[st]);
                mbar_arrive_expect_tx(kb, TL::BYTES);
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_K + st * TL::BYTES + cb * TL::BLOCK), &tmK,
                                kb, cb * TL::BOX_COLS, w.j, jk * kRows, w.b);
                mbar_arrive_expect_tx(vb, TL::BYTES);
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_V + st * TL::BYTES + cb * TL::BLOCK), &tmV,
                                vb, cb * TL::BOX_COLS, w.j, jk * kRows, w.b);
                ++kt;
                return true;
            };
            for (int k = 0; ok; ++k) {
                const int u = snake_unit(k, cta, P);
                if (u >= p.num_units)
                    break;
                const FwdUnit w = fwd_unit(u, GC, p);
                // order: [Q of this unit if not prefetched], K/V 0, [Q of the
                // next unit], K/V 1..m
                if (QB == 1 || k == 0)
                    ok = load_q(k);
                ok = ok && load_kv(w, 0);
                if (QB == 2 && ok && snake_unit(k + 1, cta, P) < p.num_units)
                    ok = load_q(k + 1);
                for (int jk = 1; jk <= w.m && ok; ++jk)
                    ok = load_kv(w, jk);
            }
            if (*wc.abort) {
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
                const FwdUnit w = fwd_unit(u, GC, p);
                const int nq0 = (QB == 1 || k == 0) ? GC : 0;
                const bool has_next = QB == 2 && snake_unit(k + 1, cta, P) < p.num_units;
                const int nq1 = has_next ? GC : 0;
                for (int t = 0; t < nq0 + 1 + nq1 + w.m && ok; ++t) {
                    const bool isq = t < nq0 || (t > nq0 && t <= nq0 + nq1);
                    const int qunit = t < nq0 ? k : k + 1;
                    const int g = t < nq0 ? t : t - nq0 - 1;
                    const int jk = t == nq0 ? 0 : t - nq0 - nq1;
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
                            isq && qunit != k ? fwd_unit(snake_unit(qunit, cta, P), GC, p) : w;
                        for (int cb = 0; cb < TL::NB; ++cb) {
                            const uint32_t src = smem_u32(tile + cb * TL::BLOCK);
                            if (isq)
                                tma_store_4d(&tmQs, src, cb * TL::BOX_COLS, wq.h0 + g,
                                             wq.m * kRows, wq.b);
                            else
                                tma_store_4d(&tmKs, src, cb * TL::BOX_COLS, w.j, jk * kRows, w.b);
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
            int gi = 0, kt = 0;
            for (int k = 0; ok; ++k) {
                const int u = snake_unit(k, cta, P);
                if (u >= p.num_units)
                    break;
                const FwdUnit w = fwd_unit(u, GC, p);
                const int nitems = (w.m + 1) * IPT;
                for (int it = 0; it < nitems; ++it, ++gi) {
                    const int jk = it / IPT, half = (it / GC) & 1, g = it % GC, st = kt % ST;
                    const int sb = gi % NSB, pw = gi & 1;
                    if (warp == 13) {
                        // S_sb = Q'_g K'[64 half, +64)^T once the operands are
                        // rotated and buffer sb has been read by its last item
                        if ((half == 0 && g == 0 &&
                             !mbar_wait_warp(smem_u32(&bar_k_ready[st]), (kt / ST) & 1, wc)) ||
                            (it < GC && !mbar_wait_warp(smem_u32(&bar_q_ready[k % QB][g]),
                                                        (k / QB) & 1, wc)) ||
                            (gi >= NSB && !mbar_wait_warp(smem_u32(&bar_s_empty[sb]),
                                                          ((gi - NSB) / NSB) & 1, wc))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t qd = dQ0 + ((k % QB) * GC + g) * TSTEP;
                        const uint64_t kd = dK0 + st * TSTEP + half * KHALF;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_f16_ss(tb + 64u * sb, qd + kmajor_off<D>(kk),
                                           kd + kmajor_off<D>(kk), ID_S, kk > 0 ? 1u : 0u);
                            mma_commit(smem_u32(&bar_s_full[sb]));
                            if (jk == w.m && half == 1)   // last use of head g's Q'
                                mma_commit(smem_u32(&bar_q_empty[k % QB][g]));
                        }
                        __syncwarp();
                    } else {
                        // O_g += P_pw V[64 half, +64) once the softmax has written P_pw
                        if (!mbar_wait_warp(smem_u32(&bar_p_full[pw]), (gi >> 1) & 1, wc) ||
                            (half == 0 && g == 0 &&
                             !mbar_wait_warp(smem_u32(&bar_v_full[st]), (kt / ST) & 1, wc)) ||
                            (it < GC && k >= 1 &&
                             !mbar_wait_warp(smem_u32(&bar_o_free[g]), (k - 1) & 1, wc))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t vm = dV0 + st * TSTEP;
                        const uint32_t first = (it >= GC) ? 1u : 0u;
                        if (elect_one()) {
#pragma unroll
                            for (int nc = 0; nc < D / TL::NPV; ++nc)
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk)
                                    mma_f16_ts(tb + C::COL_O + g * D + nc * TL::NPV,
                                               tb + C::COL_P + 32u * pw + 8 * kk,
                                               vm + mnmajor_off<D>(nc, 4 * half + kk), ID_PV,
                                               kk > 0 ? 1u : first);
                            mma_commit(smem_u32(&bar_p_empty[pw]));
                            if (half == 1 && g == GC - 1)
                                mma_commit(smem_u32(&bar_kv_empty[st]));
                        }
                        __syncwarp();
                    }
                    if (half == 1 && g == GC - 1)
                        ++kt;
                }
            }
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
        uint32_t nsv = 0;   // tiles handed to warp 15 (training path)
        for (int k = 0; ok; ++k) {
            const int u = snake_unit(k, cta, P);
            if (u >= p.num_units)
                break;
            const FwdUnit w = fwd_unit(u, GC, p);
            // Tiles in the order the producer loads them: [Q of this unit
            // unless prefetched], K 0, [Q of the next unit], K 1..m.  One call
            // site keeps the unrolled rotation in the instruction cache once.
            const int nq0 = (QB == 1 || k == 0) ? GC : 0;
            const bool has_next = QB == 2 && snake_unit(k + 1, cta, P) < p.num_units;
            const int nq1 = has_next ? GC : 0;
            const int mnext = has_next ? fwd_unit(snake_unit(k + 1, cta, P), GC, p).m : 0;
            for (int t = 0; t < nq0 + 1 + nq1 + w.m && ok; ++t) {
                const bool isq = t < nq0 || (t > nq0 && t <= nq0 + nq1);
                const int qunit = t < nq0 ? k : k + 1;
                const int g = t < nq0 ? t : t - nq0 - 1;
                const int jk = t == nq0 ? 0 : t - nq0 - nq1;
                const int qb = qunit % QB, st = kt % ST;
                const uint32_t full = isq ? smem_u32(&bar_q_full[qb][g]) : smem_u32(&bar_k_full[st]);
                const uint32_t par = isq ? ((qunit / QB) & 1) : ((kt / ST) & 1);
                if (!mbar_wait_warp(full, par, wc)) {
                    ok = false;
                    break;
                }
                uint8_t *tile = smem + (isq ? C::OFF_Q + (qb * GC + g) * TL::BYTES
                                            : C::OFF_K + st * TL::BYTES);
                const int row0 = isq ? (qunit == k ? w.m : mnext) : jk;
                mx = fmaxf(mx, rope_row_ilp<D>(tile, r, static_cast<uint32_t>(row0 * kRows + r),
                                               p.rope));
                fence_proxy_async_smem();
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
    regs_claim<184>();
    const int wg = warp >> 2;               // this group's item parity
    const int q4 = warp & 3;                // TMEM lane quarter
    const int r = threadIdx.x & 127;        // query row == TMEM lane
    const uint32_t lane_base = tmem_addr(tbase, q4 * 32, 0);
    const float sl2 = p.scale_log2;
    uint8_t *stage = smem + C::OFF_O + wg * TL::BLOCK;
    bool ok = true;
    int gi = 0;
    uint32_t nepi = 0;       // epilogues this group has run
    for (int k = 0; ok; ++k) {
        const int u = snake_unit(k, cta, P);
        if (u >= p.num_units)
            break;
        const FwdUnit un = fwd_unit(u, GC, p);
        const int nitems = (un.m + 1) * IPT;
        for (int it = 0; it < nitems; ++it, ++gi) {
            if ((gi & 1) != wg)
                continue;
            const uint32_t n = static_cast<uint32_t>(gi) >> 1;   // this group's item count
            const int jk = it / IPT, half = (it / GC) & 1, g = it % GC;
            const int pos = 2 * jk + half;                        // head g's item in the unit
            const int sb = gi % NSB;
            const uint32_t s_addr = lane_base + 64u * sb;
            const uint32_t p_addr = lane_base + C::COL_P + 32u * wg;
            // the previous item of head g ran on the other group (odd GC)
            const int xprev = gi - GC;
            const bool handoff = ODD && xprev >= 0;
            const uint32_t xa = static_cast<uint32_t>(xprev) >> 1;   // its index there
            if (!mbar_wait_warp(smem_u32(&bar_s_full[sb]), (gi / NSB) & 1, wc)) {
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
                mbar_arrive(smem_u32(&bar_s_empty[sb]));

            // causal mask on the diagonal tile (key > query row)
            if (jk == un.m) {
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (64 * half + 32 * c + e > r)
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
                        m2[c] = fmax3(m2[c], __uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1]));
                }
                mx = fmaxf(m2[0], m2[1]);
            }
            const float m_tile = mx * sl2;

            // running max of (head g, row r): read, move lazily, publish
            if (handoff &&
                !mbar_wait_warp(smem_u32(&bar_hm[xprev & 1][xa % 3]), (xa / 3) & 1, wc)) {
                ok = false;
                break;
            }
            float m_use = m_tile, alpha = 1.f;
            bool resc = false;
            if (pos > 0) {
                const float m_prev = mrun[g * kRows + r];
                m_use = m_prev;
                if (m_tile > m_prev + 8.f) {
                    alpha = ex2_approx(m_prev - m_tile);
                    m_use = m_tile;
                    resc = true;
                }
            }
            mrun[g * kRows + r] = m_use;
            if (ODD) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_hm[wg][n % 3]));
            }

            // P = 2^(S*scale*log2e - m) as bf16 pairs into P_wg
            float sum4[4] = {0.f, 0.f, 0.f, 0.f};
            {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float p0 = ex2_approx(fmaf(__uint_as_float(s[c][e]), sl2, -m_use));
                        const float p1 =
                            ex2_approx(fmaf(__uint_as_float(s[c][e + 1]), sl2, -m_use));
                        sum4[(e >> 1) & 3] += p0 + p1;
                        pk[16 * c + e / 2] = pack_bf16x2(p0, p1);
                    }
                // P_wg is free once PV(gi - 2) has completed (this group's
                // previous item; the one before was waited for then, so the
                // parity is exact)
                if (gi >= 2 &&
                    !mbar_wait_warp(smem_u32(&bar_p_empty[wg]), ((gi - 2) >> 1) & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_st32(p_addr, pk);
            }
            const float sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
            if (__any_sync(0xffffffffu, resc)) {
                // O_g must hold the previous item of head g (gi - GC) before it
                // is rescaled.  PVs complete in order, so for GC >= 2 the wait
                // for PV(gi - 2) above covers it; for GC == 1 it is the other
                // group's PV(gi - 1) (PV(gi - 3) is complete, parity exact).
                if (GC == 1 &&
                    !mbar_wait_warp(smem_u32(&bar_p_empty[wg ^ 1]), ((gi - 1) >> 1) & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t oa = lane_base + C::COL_O + g * D;
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
                mbar_arrive(smem_u32(&bar_p_full[wg]));

            // running sum of (head g, row r)
            if (handoff &&
                !mbar_wait_warp(smem_u32(&bar_hl[xprev & 1][xa % 3]), (xa / 3) & 1, wc)) {
                ok = false;
                break;
            }
            const float l_now = (pos > 0 ? lrun[g * kRows + r] * alpha : 0.f) + sum;
            lrun[g * kRows + r] = l_now;
            if (ODD) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_hl[wg][n % 3]));
            }
            if (jk != un.m || half != 1)
                continue;

            // ---- last item of head g in this unit: O_g / l and lse ----
            if (!mbar_wait_warp(smem_u32(&bar_p_empty[wg]), (gi >> 1) & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv_l = 1.f / l_now;
            const int h = un.h0 + g;
            const int t = un.m * kRows + r;
            const uint32_t oa = lane_base + C::COL_O + g * D;
            if constexpr (C::STAGE) {
                // the staging block is free once this group's previous
                // store has read it
                if (nepi >= 1) {
                    if (warp == 4 * wg && lane == 0) {
                        bulk_wait_read0();
                        mbar_arrive(smem_u32(&bar_stg_free[wg]));
                    }
                    if (!mbar_wait_warp(smem_u32(&bar_stg_free[wg]), (nepi - 1) & 1, wc)) {
                        ok = false;
                        break;
                    }
                }
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(oa + c, o);
                    tmem_ld_wait(o);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4 *>(stage + tile_chunk<D>(r, c / 8 + q)) =
                            make_uint4(pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv_l,
                                                   __uint_as_float(o[8 * q + 1]) * inv_l),
                                       pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l,
                                                   __uint_as_float(o[8 * q + 3]) * inv_l),
                                       pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l,
                                                   __uint_as_float(o[8 * q + 5]) * inv_l),
                                       pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l,
                                                   __uint_as_float(o[8 * q + 7]) * inv_l));
                }
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&bar_o_free[g]));
                    mbar_arrive(smem_u32(&bar_stg_full[wg]));
                }
                if (warp == 4 * wg) {
                    if (!mbar_wait_warp(smem_u32(&bar_stg_full[wg]), nepi & 1, wc)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        tma_store_4d(&tmO, smem_u32(stage), 0, h, un.m * kRows, un.b);
                        bulk_commit();
                    }
                    __syncwarp();
                }
            } else {
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out0) +
                                     ((static_cast<size_t>(un.b) * p.T + t) * p.Hq + h) * D;
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(oa + c, o);
                    tmem_ld_wait(o);
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        x[e] = __uint_as_float(o[e]) * inv_l;
                    if (t < p.T)
                        store_row32_bf16(dst + c, x);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_o_free[g]));
            }
            if (t < p.T)
                p.lse[(static_cast<size_t>(un.b) * p.Hq + h) * p.T + t] =
                    (m_use + __log2f(l_now)) * kLn2;
            ++nepi;
        }
    }
    if constexpr (C::STAGE) {
        if (warp == 4 * wg && lane == 0)
            bulk_wait0();
    }
    teardown();
}

// ------------------------------------------------------------- launch ---

template <int D, int GC, int ST>
static cudaError_t launch_fwd_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const CUtensorMap &o, const CUtensorMap &qs, const CUtensorMap &ks,
                                const AttnParams &p0, cudaStream_t stream)
{
    using C = FwdCfg<D, GC, ST>;
    auto kern = fwd_kernel<D, GC, ST>;
    static bool attr_done[64] = {};   // one flag set per template instantiation
    cudaError_t e = ensure_smem_attr(kern, C::SMEM_BYTES, attr_done);
    if (e != cudaSuccess)
        return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    AttnParams p = p0;
    p.num_units = p.M * p.B * p.Hkv * p.nchunks;
    const unsigned grid = static_cast<unsigned>(p.num_units < sms ? p.num_units : sms);
    return launch_pdl(kern, grid, 512, C::SMEM_BYTES, stream, q, k, v, o, qs, ks, p);
}

template <int D, int GC>
static cudaError_t launch_fwd_p(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const CUtensorMap &o, const CUtensorMap &qs, const CUtensorMap &ks,
                                const AttnParams &p, cudaStream_t stream)
{
    return launch_fwd_t<D, GC, FwdPlan<D, GC>::ST>(q, k, v, o, qs, ks, p, stream);
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
