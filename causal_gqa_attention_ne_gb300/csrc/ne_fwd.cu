// ne_fwd.cu -- forward kernel: causal grouped-query attention with RoPE fused
// into the Q/K tile load, tcgen05 tensor-core MMAs accumulating in TMEM and an
// online softmax (the tiled FlashAttention of the NanoEuler walkthrough,
// section 3.4, and of the NanoEuler README's "CUDA engine" section, rebuilt
// for sm_103a).
//
// Persistent: one CTA per SM walks a snake-ordered list of work units
// (b, kv head j, query tile m, chunk of GC query heads that share j),
// heaviest (largest m) first.  Per unit the loop runs over the causal key
// tiles jk <= m and the GC heads ("items"); each K/V tile is loaded once by
// TMA, rotated once and used by all GC heads.  Warp roles (512 threads):
//   warps 0-7   two softmax warpgroups; warpgroup w handles key columns
//               [64w, 64w+64) of each 128x128 score tile, thread r query row
//               r (TMEM lane r).  The two halves of a row exchange their
//               maxima through shared memory; both then keep the same running
//               max, write P (bf16) back to TMEM as the A operand of O += P V,
//               rescale their half of O when the max grows by more than 2^8,
//               and at the end of a unit store their half of O / l (and lse).
//   warps 8-11  RoPE: rotate the unit's Q tiles and each K tile in place
//               (bf16 in, fp16 out), in the order the MMAs first need them.
//   warp 12     TMA producer.   warp 13  TMEM allocator + S issuer.
//   warp 14     PV issuer.      warp 15  idle.
// TMEM: S [0,128), P [128,192), O of head g at 192 + g*D.
#include <cuda_bf16.h>

#include "ne_common.cuh"
#include "ne_kernels.h"

namespace ne {

template <int D, int GC, int ST>
struct FwdCfg {
    using TL = Tile<D>;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + GC * TL::BYTES;
    static constexpr int OFF_V = OFF_K + ST * TL::BYTES;
    static constexpr int OFF_X = OFF_V + ST * TL::BYTES;          // float [2][2][128] maxima
    static constexpr int OFF_L = OFF_X + 2 * 2 * kRows * 4;        // float [GC][2][128] sums
    static constexpr int SMEM_BYTES = smem_one_cta(OFF_L + GC * 2 * kRows * 4 + 1024);
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0, COL_P = 128, COL_O = 192;
    static_assert(COL_O + GC * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
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

// Scale 16 or 32 TMEM columns of this thread's lane by `alpha` (O rescale).
template <int N>
__device__ __forceinline__ void tmem_scale_cols(uint32_t taddr, float alpha)
{
    if constexpr (N == 32) {
        uint32_t o[32];
        tmem_ld32(taddr, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int e = 0; e < 32; ++e)
            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32(taddr, o);
    } else {
        uint32_t o[16];
        tmem_ld16(taddr, o);
        tmem_ld_wait_only();
        tmem_tie16(o);
#pragma unroll
        for (int e = 0; e < 16; ++e)
            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st16(taddr, o);
    }
}

template <int D, int GC, int ST>
__global__ void __launch_bounds__(512, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const AttnParams p)
{
    using C = FwdCfg<D, GC, ST>;
    using TL = Tile<D>;
    constexpr int HALF = D / 2;                     // O columns per softmax warpgroup
    constexpr int OSTEP = (HALF >= 32) ? 32 : 16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_q_full[GC], bar_q_ready[GC], bar_q_empty[GC];
    __shared__ uint64_t bar_k_full[ST], bar_k_ready[ST], bar_v_full[ST], bar_kv_empty[ST];
    __shared__ uint64_t bar_s_full, bar_s_empty, bar_p_full, bar_p_empty;
    __shared__ uint64_t bar_o_done, bar_o_free, bar_drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ uint32_t abort_s;
    float *xmax = reinterpret_cast<float *>(smem + C::OFF_X);   // [parity][w][row]
    float *xsum = reinterpret_cast<float *>(smem + C::OFF_L);   // [g][w][row]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cta = static_cast<int>(blockIdx.x), P = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        abort_s = 0;
        for (int g = 0; g < GC; ++g) {
            mbar_init(smem_u32(&bar_q_full[g]), 1);
            mbar_init(smem_u32(&bar_q_ready[g]), 4);
            mbar_init(smem_u32(&bar_q_empty[g]), 1);
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&bar_k_full[s]), 1);
            mbar_init(smem_u32(&bar_k_ready[s]), 4);
            mbar_init(smem_u32(&bar_v_full[s]), 1);
            mbar_init(smem_u32(&bar_kv_empty[s]), 1);
        }
        mbar_init(smem_u32(&bar_s_full), 1);
        mbar_init(smem_u32(&bar_s_empty), 8);
        mbar_init(smem_u32(&bar_p_full), 8);
        mbar_init(smem_u32(&bar_p_empty), 1);
        mbar_init(smem_u32(&bar_o_done), 1);
        mbar_init(smem_u32(&bar_o_free), 8);
        mbar_init(smem_u32(&bar_drain), 2);
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
    const WaitCtl wc{&abort_s, p.status, p.wait_limit_ns};
    // Each role ends with its own teardown: after setmaxnreg the warps run
    // under different register budgets, so their code paths never re-join.
    auto teardown = [&]() {
        tc_fence_before();
        __syncthreads();
        if (warp == 13) {
            tc_fence_after();
            tmem_dealloc(tbase, C::TMEM_COLS);
        }
    };

    // Register budgets after the split (launched with 128 per thread x 512):
    // softmax 184 x 256 + RoPE 72 x 128 + TMA/MMA 72 x 128 = 65536.
    if (warp >= 12) {
        regs_release<72>();
        if (warp == 12 && lane == 0) {
            // ------------------------------------------------ TMA producer ---
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            bool ok = true;
            int kt = 0, k = 0;
            for (; ok; ++k) {
                const int u = snake_unit(k, cta, P);
                if (u >= p.num_units)
                    break;
                const FwdUnit w = fwd_unit(u, GC, p);
                for (int g = 0; g < GC && ok; ++g) {
                    if (k >= 1 && !mbar_wait(smem_u32(&bar_q_empty[g]), (k - 1) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    const uint32_t qb = smem_u32(&bar_q_full[g]);
                    mbar_arrive_expect_tx(qb, TL::BYTES);
                    for (int cb = 0; cb < TL::NB; ++cb)
                        tma_load_4d(smem_u32(smem + C::OFF_Q + g * TL::BYTES + cb * TL::BLOCK),
                                    &tmQ, qb, cb * TL::BOX_COLS, w.h0 + g, w.m * kRows, w.b);
                }
                for (int jk = 0; jk <= w.m && ok; ++jk, ++kt) {
                    const int st = kt % ST, u2 = kt / ST;
                    if (u2 >= 1 && !mbar_wait(smem_u32(&bar_kv_empty[st]), (u2 - 1) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    const uint32_t kb = smem_u32(&bar_k_full[st]), vb = smem_u32(&bar_v_full[st]);
                    mbar_arrive_expect_tx(kb, TL::BYTES);
                    for (int cb = 0; cb < TL::NB; ++cb)
                        tma_load_4d(smem_u32(smem + C::OFF_K + st * TL::BYTES + cb * TL::BLOCK),
                                    &tmK, kb, cb * TL::BOX_COLS, w.j, jk * kRows, w.b);
                    mbar_arrive_expect_tx(vb, TL::BYTES);
                    for (int cb = 0; cb < TL::NB; ++cb)
                        tma_load_4d(smem_u32(smem + C::OFF_V + st * TL::BYTES + cb * TL::BLOCK),
                                    &tmV, vb, cb * TL::BOX_COLS, w.j, jk * kRows, w.b);
                }
            }
            if (*wc.abort) {
                for (int g = 0; g < GC; ++g)
                    mbar_wait_drain(smem_u32(&bar_q_full[g]), (k > 0 ? k - 1 : 0) & 1, wc.limit_ns);
                for (int t = (kt > ST ? kt - ST : 0); t < kt; ++t) {
                    mbar_wait_drain(smem_u32(&bar_k_full[t % ST]), (t / ST) & 1, wc.limit_ns);
                    mbar_wait_drain(smem_u32(&bar_v_full[t % ST]), (t / ST) & 1, wc.limit_ns);
                }
            }
        } else if (warp == 13 || warp == 14) {
            // -------------------------------------------------- MMA issuers ---
            constexpr uint32_t ID_S = idesc_f16(128, 128, false, false, false);
            constexpr uint32_t ID_PV = idesc_f16(128, TL::NPV, true, false, true);
            constexpr uint32_t TSTEP = TL::BYTES >> 4;
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
                const int nitems = (w.m + 1) * GC;
                for (int it = 0; it < nitems; ++it, ++gi) {
                    const int jk = it / GC, g = it % GC, st = kt % ST;
                    if (warp == 13) {
                        // S = Q'_g K'^T as soon as the operands and the S buffer are ready
                        if ((g == 0 &&
                             !mbar_wait_warp(smem_u32(&bar_k_ready[st]), (kt / ST) & 1, wc)) ||
                            (jk == 0 && !mbar_wait_warp(smem_u32(&bar_q_ready[g]), k & 1, wc)) ||
                            (gi >= 1 &&
                             !mbar_wait_warp(smem_u32(&bar_s_empty), (gi - 1) & 1, wc))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t qd = dQ0 + g * TSTEP, kd = dK0 + st * TSTEP;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_f16_ss(tb + C::COL_S, qd + kmajor_off<D>(kk),
                                           kd + kmajor_off<D>(kk), ID_S, kk > 0 ? 1u : 0u);
                            mma_commit(smem_u32(&bar_s_full));
                            if (jk == w.m)   // last use of head g's Q' in this unit
                                mma_commit(smem_u32(&bar_q_empty[g]));
                        }
                        __syncwarp();
                    } else {
                        // O_g += P V once the softmax has written P
                        if (!mbar_wait_warp(smem_u32(&bar_p_full), gi & 1, wc) ||
                            (g == 0 &&
                             !mbar_wait_warp(smem_u32(&bar_v_full[st]), (kt / ST) & 1, wc)) ||
                            (it == 0 && k >= 1 &&
                             !mbar_wait_warp(smem_u32(&bar_o_free), (k - 1) & 1, wc))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t vm = dV0 + st * TSTEP;
                        const uint32_t first = (jk > 0) ? 1u : 0u;
                        if (elect_one()) {
#pragma unroll
                            for (int nc = 0; nc < D / TL::NPV; ++nc)
#pragma unroll
                                for (int kk = 0; kk < 8; ++kk)
                                    mma_f16_ts(tb + C::COL_O + g * D + nc * TL::NPV,
                                               tb + C::COL_P + 8 * kk, vm + mnmajor_off<D>(nc, kk),
                                               ID_PV, kk > 0 ? 1u : first);
                            mma_commit(smem_u32(&bar_p_empty));
                            if (g == GC - 1)
                                mma_commit(smem_u32(&bar_kv_empty[st]));
                            if (it == nitems - 1)
                                mma_commit(smem_u32(&bar_o_done));
                        }
                        __syncwarp();
                    }
                    if (g == GC - 1)
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
        regs_release<72>();
        const int r = threadIdx.x - 256;
        float mx = 0.f;
        bool ok = true;
        int kt = 0;
        auto rot_q = [&](int g, int k, int m) {
            if (!mbar_wait_warp(smem_u32(&bar_q_full[g]), k & 1, wc)) {
                ok = false;
                return;
            }
            mx = fmaxf(mx, rope_row_ilp<D>(smem + C::OFF_Q + g * TL::BYTES, r,
                                           static_cast<uint32_t>(m * kRows + r), p.rope));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_q_ready[g]));
        };
        auto rot_k = [&](int jk) {
            const int st = kt % ST;
            if (!mbar_wait_warp(smem_u32(&bar_k_full[st]), (kt / ST) & 1, wc)) {
                ok = false;
                return;
            }
            mx = fmaxf(mx, rope_row_ilp<D>(smem + C::OFF_K + st * TL::BYTES, r,
                                           static_cast<uint32_t>(jk * kRows + r), p.rope));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_k_ready[st]));
            ++kt;
        };
        for (int k = 0; ok; ++k) {
            const int u = snake_unit(k, cta, P);
            if (u >= p.num_units)
                break;
            const FwdUnit w = fwd_unit(u, GC, p);
            // in the order the S issuer first needs them: Q0, K0, Q1.., K1..
            rot_q(0, k, w.m);
            if (ok)
                rot_k(0);
            for (int g = 1; g < GC && ok; ++g)
                rot_q(g, k, w.m);
            for (int jk = 1; jk <= w.m && ok; ++jk)
                rot_k(jk);
        }
        if (mx > kFp16Max)
            atomicOr(p.status, kDevRange);
        teardown();
        return;
    }

    // ----------------------------------------------------- softmax rows ---
    regs_claim<184>();
    const int w = warp >> 2;                // key-column half of the score tile
    const int r = threadIdx.x & 127;        // query row == TMEM lane
    const uint32_t lane_base = tmem_addr(tbase, (warp & 3) * 32, 0);
    const float sl2 = p.scale_log2;
    bool ok = true;
    int gi = 0;
    for (int k = 0; ok; ++k) {
        const int u = snake_unit(k, cta, P);
        if (u >= p.num_units)
            break;
        const FwdUnit un = fwd_unit(u, GC, p);
        const int nitems = (un.m + 1) * GC;
        float m_run[GC], l_run[GC];
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            m_run[g] = -INFINITY;
            l_run[g] = 0.f;
        }
        for (int it = 0; it < nitems; ++it, ++gi) {
            const int jk = it / GC, g = it % GC;
            if (!mbar_wait_warp(smem_u32(&bar_s_full), gi & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[2][32];
            tmem_ld32(lane_base + C::COL_S + 64 * w, sv[0]);
            tmem_ld32(lane_base + C::COL_S + 64 * w + 32, sv[1]);
            tmem_ld_wait_only();
            tmem_tie(sv[0]);
            tmem_tie(sv[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_s_empty));

            // causal mask on the diagonal tile (key column c > query row r)
            if (jk == un.m) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (64 * w + 32 * h + e > r)
                            sv[h][e] = __float_as_uint(-INFINITY);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    mx = fmaxf(mx, __uint_as_float(sv[h][e]));
            // the two halves of the row agree on one maximum; the buffer
            // alternates with the item parity so a fast half never overwrites
            // a value its partner has not read yet
            float *xm = xmax + (gi & 1) * 2 * kRows;
            xm[w * kRows + r] = mx;
            named_bar_sync(1, 256);
            mx = fmaxf(mx, xm[(1 - w) * kRows + r]);
            const float m_tile = mx * sl2;

            float mref = m_run[0], lcur = l_run[0];
#pragma unroll
            for (int q = 1; q < GC; ++q)
                if (g == q) {
                    mref = m_run[q];
                    lcur = l_run[q];
                }
            float alpha = 1.f;
            bool resc = false;
            if (mref == -INFINITY) {
                mref = m_tile;
            } else if (m_tile > mref + 8.f) {
                // Lazy rescale: only when the max grew by more than 2^8; the
                // final division by l makes the result exact either way.
                alpha = ex2_approx(mref - m_tile);
                mref = m_tile;
                resc = true;
            }
            float sum = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(sv[h][e]), sl2, -mref));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(sv[h][e + 1]), sl2, -mref));
                    sum += p0 + p1;
                    pk[16 * h + e / 2] = pack_bf16x2(p0, p1);
                }
            lcur = lcur * alpha + sum;
#pragma unroll
            for (int q = 0; q < GC; ++q)
                if (g == q) {
                    m_run[q] = mref;
                    l_run[q] = lcur;
                }
            // O_g must be stable and the P buffer free: PV of the previous item done.
            if (gi >= 1 && !mbar_wait_warp(smem_u32(&bar_p_empty), (gi - 1) & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (__any_sync(0xffffffffu, resc)) {
                const uint32_t oa = lane_base + C::COL_O + g * D + w * HALF;
#pragma unroll
                for (int c = 0; c < HALF; c += OSTEP)
                    tmem_scale_cols<OSTEP>(oa + c, alpha);
            }
            tmem_st32(lane_base + C::COL_P + 32 * w, pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_p_full));
        }
        if (!ok)
            break;
        // ---- unit epilogue: O / l, lse ----
        if (!mbar_wait_warp(smem_u32(&bar_o_done), k & 1, wc)) {
            ok = false;
            break;
        }
        tc_fence_after();
#pragma unroll
        for (int g = 0; g < GC; ++g)
            xsum[(g * 2 + w) * kRows + r] = l_run[g];
        named_bar_sync(1, 256);
        const int t = un.m * kRows + r;
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out0);
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            const float l = l_run[g] + xsum[(g * 2 + (1 - w)) * kRows + r];
            const float inv_l = 1.f / l;
            const int h = un.h0 + g;
            const uint32_t oa = lane_base + C::COL_O + g * D + w * HALF;
            __nv_bfloat16 *dst =
                o + ((static_cast<size_t>(un.b) * p.T + t) * p.Hq + h) * D + w * HALF;
#pragma unroll
            for (int c = 0; c < HALF; c += OSTEP) {
                if constexpr (OSTEP == 32) {
                    uint32_t ov[32];
                    tmem_ld32(oa + c, ov);
                    tmem_ld_wait(ov);
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        x[e] = __uint_as_float(ov[e]) * inv_l;
                    if (t < p.T)
                        store_row32_bf16(dst + c, x);
                } else {
                    uint32_t ov[16];
                    tmem_ld16(oa + c, ov);
                    tmem_ld_wait_only();
                    tmem_tie16(ov);
                    float x[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        x[e] = __uint_as_float(ov[e]) * inv_l;
                    if (t < p.T) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            d4[q] = make_uint4(pack_bf16x2(x[q * 8 + 0], x[q * 8 + 1]),
                                               pack_bf16x2(x[q * 8 + 2], x[q * 8 + 3]),
                                               pack_bf16x2(x[q * 8 + 4], x[q * 8 + 5]),
                                               pack_bf16x2(x[q * 8 + 6], x[q * 8 + 7]));
                    }
                }
            }
            if (w == 0 && t < p.T)
                p.lse[(static_cast<size_t>(un.b) * p.Hq + h) * p.T + t] =
                    (m_run[g] + __log2f(l)) * kLn2;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&bar_o_free));
    }
    teardown();
}

// ------------------------------------------------------------- launch ---

template <int D, int GC, int ST>
static cudaError_t launch_fwd_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
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
    kern<<<grid, 512, C::SMEM_BYTES, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int d, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                       const AttnParams &p, cudaStream_t stream)
{
    switch (d) {
    case 32:
        switch (p.GC) {
        case 1: return launch_fwd_t<32, 1, 4>(q, k, v, p, stream);
        case 2: return launch_fwd_t<32, 2, 4>(q, k, v, p, stream);
        case 3: return launch_fwd_t<32, 3, 4>(q, k, v, p, stream);
        case 4: return launch_fwd_t<32, 4, 4>(q, k, v, p, stream);
        default: break;
        }
        break;
    case 64:
        switch (p.GC) {
        case 1: return launch_fwd_t<64, 1, 4>(q, k, v, p, stream);
        case 2: return launch_fwd_t<64, 2, 4>(q, k, v, p, stream);
        case 3: return launch_fwd_t<64, 3, 4>(q, k, v, p, stream);
        case 4: return launch_fwd_t<64, 4, 4>(q, k, v, p, stream);
        default: break;
        }
        break;
    case 128:
        switch (p.GC) {
        case 1: return launch_fwd_t<128, 1, 2>(q, k, v, p, stream);
        case 2: return launch_fwd_t<128, 2, 2>(q, k, v, p, stream);
        default: break;
        }
        break;
    default: break;
    }
    return cudaErrorInvalidValue;
}

} // namespace ne
