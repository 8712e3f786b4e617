// ne_fwd.cu -- forward kernel: causal grouped-query attention with RoPE fused
// into the Q/K tile load, tcgen05 tensor-core MMAs accumulating in TMEM and an
// online softmax (the tiled FlashAttention of the NanoEuler walkthrough,
// section 3.4, and of the NanoEuler README's "CUDA engine" section, rebuilt
// for sm_103a).
//
// One CTA owns one 128-row query tile of GC query heads that share a KV head
// (b, kv head j, tile m).  Each K/V tile is loaded once by TMA, rotated once
// and used by all GC heads.  Warp roles (320 threads):
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r); reads S,
//              keeps the running max / sum, writes P (bf16) to shared memory,
//              rescales O when the max grows, runs the epilogue.
//   warps 4-7  RoPE: rotate the Q tiles once and every K tile in place
//              (bf16 in, fp16 out).
//   warp 8     TMA producer.
//   warp 9     TMEM allocator and MMA issuer (one thread).
// TMEM columns: S double buffer [0,256), O of head g at 256 + g*D.
#include <cuda_bf16.h>

#include "ne_common.cuh"
#include "ne_kernels.h"

namespace ne {

template <int D, int GC, int ST, int NP>
struct FwdCfg {
    using TL = Tile<D>;
    static constexpr int PTILE = kRows * 128 * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + GC * TL::BYTES;
    static constexpr int OFF_V = OFF_K + ST * TL::BYTES;
    static constexpr int OFF_P = OFF_V + ST * TL::BYTES;
    static constexpr int SMEM_BYTES = smem_one_cta(OFF_P + NP * PTILE + 1024);   // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(256 + GC * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <int D, int GC, int ST, int NP>
__global__ void __launch_bounds__(320, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const AttnParams p)
{
    using C = FwdCfg<D, GC, ST, NP>;
    using TL = Tile<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_q_full, bar_q_ready, bar_drain;
    __shared__ uint64_t bar_k_full[ST], bar_k_ready[ST], bar_v_full[ST], bar_kv_empty[ST];
    __shared__ uint64_t bar_s_full[2], bar_s_empty[2], bar_p_full[NP], bar_pv_done[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ uint32_t abort_s;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // Work decode: heaviest (last) query tiles first.
    const int per_m = p.B * p.Hkv * p.nchunks;
    const int m = p.M - 1 - static_cast<int>(blockIdx.x) / per_m;
    int rem = static_cast<int>(blockIdx.x) % per_m;
    const int chunk = rem % p.nchunks;
    rem /= p.nchunks;
    const int j = rem % p.Hkv;
    const int b = rem / p.Hkv;
    const int h0 = j * p.G + chunk * GC;
    const int t0 = m * kRows;
    const int nkv = m + 1;
    const int nitems = nkv * GC;

    if (threadIdx.x == 0) {
        abort_s = 0;
        mbar_init(smem_u32(&bar_q_full), 1);
        mbar_init(smem_u32(&bar_q_ready), 4);
        mbar_init(smem_u32(&bar_drain), 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&bar_k_full[s]), 1);
            mbar_init(smem_u32(&bar_k_ready[s]), 4);
            mbar_init(smem_u32(&bar_v_full[s]), 1);
            mbar_init(smem_u32(&bar_kv_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bar_s_full[s]), 1);
            mbar_init(smem_u32(&bar_s_empty[s]), 4);
            mbar_init(smem_u32(&bar_pv_done[s]), 1);
        }
        for (int s = 0; s < NP; ++s)
            mbar_init(smem_u32(&bar_p_full[s]), 4);
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(&tmem_base_s), C::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_s;
    const WaitCtl wc{&abort_s, p.status, p.wait_limit_ns};

    if (warp == 8) {
        // ------------------------------------------------ TMA producer ---
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            const uint32_t qb = smem_u32(&bar_q_full);
            mbar_arrive_expect_tx(qb, GC * TL::BYTES);
            for (int g = 0; g < GC; ++g)
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_Q + g * TL::BYTES + cb * TL::BLOCK), &tmQ,
                                qb, cb * TL::BOX_COLS, h0 + g, t0, b);
            int issued = 0;
            for (int jk = 0; jk < nkv; ++jk) {
                const int st = jk % ST, u = jk / ST;
                if (u >= 1 && !mbar_wait(smem_u32(&bar_kv_empty[st]), (u - 1) & 1, wc))
                    break;
                const uint32_t kb = smem_u32(&bar_k_full[st]), vb = smem_u32(&bar_v_full[st]);
                mbar_arrive_expect_tx(kb, TL::BYTES);
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_K + st * TL::BYTES + cb * TL::BLOCK), &tmK,
                                kb, cb * TL::BOX_COLS, j, jk * kRows, b);
                mbar_arrive_expect_tx(vb, TL::BYTES);
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_V + st * TL::BYTES + cb * TL::BLOCK), &tmV,
                                vb, cb * TL::BOX_COLS, j, jk * kRows, b);
                issued = jk + 1;
            }
            if (*wc.abort) {
                // Drain this CTA's own copies still in flight before exiting.
                for (int jk = (issued > ST ? issued - ST : 0); jk < issued; ++jk) {
                    const int st = jk % ST, u = jk / ST;
                    mbar_wait_drain(smem_u32(&bar_k_full[st]), u & 1, wc.limit_ns);
                    mbar_wait_drain(smem_u32(&bar_v_full[st]), u & 1, wc.limit_ns);
                }
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------- MMA issuer ---
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_f16(128, 128, false, false, false);
            constexpr uint32_t ID_PV = idesc_f16(128, TL::NPV, true, false, true);
            const uint32_t q_addr = smem_u32(smem + C::OFF_Q);
            const uint32_t k_addr = smem_u32(smem + C::OFF_K);
            const uint32_t v_addr = smem_u32(smem + C::OFF_V);
            const uint32_t p_addr = smem_u32(smem + C::OFF_P);
            bool ok = mbar_wait(smem_u32(&bar_q_ready), 0, wc);
            auto do_pv = [&](int x) -> bool {
                const int jx = x / GC, gx = x % GC, stx = jx % ST;
                if (gx == 0 && !mbar_wait(smem_u32(&bar_v_full[stx]), (jx / ST) & 1, wc))
                    return false;
                if (!mbar_wait(smem_u32(&bar_p_full[x % NP]), (x / NP) & 1, wc))
                    return false;
                tc_fence_after();
                const uint32_t pa = p_addr + (x % NP) * C::PTILE;
                const uint32_t va = v_addr + stx * TL::BYTES;
                const uint32_t od = tbase + 256 + gx * D;
#pragma unroll
                for (int nc = 0; nc < D / TL::NPV; ++nc)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_f16_ss(od + nc * TL::NPV, desc_ptile(pa, kk),
                                   desc_mnmajor<D>(va, nc, kk), ID_PV,
                                   (jx > 0 || kk > 0) ? 1u : 0u);
                mma_commit(smem_u32(&bar_pv_done[x % 2]));
                if (gx == GC - 1)
                    mma_commit(smem_u32(&bar_kv_empty[stx]));
                return true;
            };
            for (int i = 0; ok && i < nitems; ++i) {
                const int jk = i / GC, g = i % GC, st = jk % ST;
                if (g == 0 && !mbar_wait(smem_u32(&bar_k_ready[st]), (jk / ST) & 1, wc)) {
                    ok = false;
                    break;
                }
                if (i >= 2 && !mbar_wait(smem_u32(&bar_s_empty[i % 2]), ((i - 2) / 2) & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t qa = q_addr + g * TL::BYTES;
                const uint32_t ka = k_addr + st * TL::BYTES;
                const uint32_t sd = tbase + (i % 2) * 128;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_f16_ss(sd, desc_kmajor<D>(qa, kk), desc_kmajor<D>(ka, kk), ID_S,
                               kk > 0 ? 1u : 0u);
                mma_commit(smem_u32(&bar_s_full[i % 2]));
                if (i >= 1 && !do_pv(i - 1)) {
                    ok = false;
                    break;
                }
            }
            if (ok)
                do_pv(nitems - 1);
            mma_commit(smem_u32(&bar_drain));
            mbar_wait(smem_u32(&bar_drain), 0, wc);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------ RoPE ---
        const int r = threadIdx.x - 128;
        float mx = 0.f;
        bool ok = mbar_wait_warp(smem_u32(&bar_q_full), 0, wc);
        if (ok) {
            for (int g = 0; g < GC; ++g)
                mx = fmaxf(mx, rope_row_to_f16<D>(smem + C::OFF_Q + g * TL::BYTES, r,
                                                  static_cast<uint32_t>(t0 + r), p.rope));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_q_ready));
            for (int jk = 0; jk < nkv; ++jk) {
                const int st = jk % ST;
                if (!mbar_wait_warp(smem_u32(&bar_k_full[st]), (jk / ST) & 1, wc))
                    break;
                mx = fmaxf(mx, rope_row_to_f16<D>(smem + C::OFF_K + st * TL::BYTES, r,
                                                  static_cast<uint32_t>(jk * kRows + r), p.rope));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_k_ready[st]));
            }
        }
        if (mx > kFp16Max)
            atomicOr(p.status, kDevRange);
    } else {
        // --------------------------------------------------- softmax ---
        const int r = threadIdx.x;              // query row within the tile == TMEM lane
        const int t = t0 + r;
        const uint32_t lane_base = tmem_addr(tbase, warp * 32, 0);
        float m_run[GC], l_run[GC];
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            m_run[g] = -INFINITY;
            l_run[g] = 0.f;
        }
        constexpr int LAG = (GC < NP) ? GC : NP;
        bool ok = true;
        for (int i = 0; i < nitems; ++i) {
            const int jk = i / GC, g = i % GC;
            if (!mbar_wait_warp(smem_u32(&bar_s_full[i % 2]), (i / 2) & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[4][32];
            const uint32_t sa = lane_base + (i % 2) * 128;
            tmem_ld32(sa, s[0]);
            tmem_ld32(sa + 32, s[1]);
            tmem_ld32(sa + 64, s[2]);
            tmem_ld32(sa + 96, s[3]);
            tmem_ld_wait_only();
            tmem_tie(s[0]);
            tmem_tie(s[1]);
            tmem_tie(s[2]);
            tmem_tie(s[3]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_s_empty[i % 2]));

            // causal mask on the diagonal tile, then the row max
            const bool diag = (jk == m);
            float mx = -INFINITY;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float x = __uint_as_float(s[q4][c]);
                    if (diag && (q4 * 32 + c) > r)
                        x = -INFINITY;
                    s[q4][c] = __float_as_uint(x);
                    mx = fmaxf(mx, x);
                }
            const float m_tile = mx * p.scale_log2;
            float mref = m_run[g];
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
            m_run[g] = mref;
            float sum = 0.f;
            uint32_t pk[4][16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const float p0 =
                        ex2_approx(fmaf(__uint_as_float(s[q4][c]), p.scale_log2, -mref));
                    const float p1 =
                        ex2_approx(fmaf(__uint_as_float(s[q4][c + 1]), p.scale_log2, -mref));
                    sum += p0 + p1;
                    pk[q4][c / 2] = pack_bf16x2(p0, p1);
                }
            l_run[g] = l_run[g] * alpha + sum;

            // O_g must be stable and the P buffer free: wait for PV(i - LAG).
            if (i >= LAG) {
                const int x = i - LAG;
                if (!mbar_wait_warp(smem_u32(&bar_pv_done[x % 2]), (x / 2) & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, resc)) {
                const uint32_t oa = lane_base + 256 + g * D;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(oa + cc * 32, o);
                    tmem_ld_wait(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(oa + cc * 32, o);
                }
                tmem_st_wait();
            }
            uint8_t *pt = smem + C::OFF_P + (i % NP) * C::PTILE;
#pragma unroll
            for (int c8 = 0; c8 < 16; ++c8) {
                const int q4 = c8 / 4, w = (c8 % 4) * 4;
                *reinterpret_cast<uint4 *>(pt + ptile_chunk(r, c8)) =
                    make_uint4(pk[q4][w], pk[q4][w + 1], pk[q4][w + 2], pk[q4][w + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_p_full[i % NP]));
        }
        // ----------------------------------------------------- epilogue ---
        if (ok) {
            const int x = nitems - 1;
            ok = mbar_wait_warp(smem_u32(&bar_pv_done[x % 2]), (x / 2) & 1, wc);
        }
        if (ok) {
            tc_fence_after();
            __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.out0);
#pragma unroll
            for (int g = 0; g < GC; ++g) {
                const int h = h0 + g;
                const float inv_l = 1.f / l_run[g];
                const uint32_t oa = lane_base + 256 + g * D;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    tmem_ld32(oa + cc * 32, ov);
                    tmem_ld_wait(ov);
                    if (t < p.T) {
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            o + ((static_cast<size_t>(b) * p.T + t) * p.Hq + h) * D + cc * 32);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                w[e] = pack_bf16x2(__uint_as_float(ov[q * 8 + 2 * e]) * inv_l,
                                                   __uint_as_float(ov[q * 8 + 2 * e + 1]) * inv_l);
                            dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                if (t < p.T)
                    p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.T + t] =
                        (m_run[g] + __log2f(l_run[g])) * kLn2;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------- launch ---

template <int D, int GC, int ST, int NP>
static cudaError_t launch_fwd_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                const AttnParams &p, cudaStream_t stream)
{
    using C = FwdCfg<D, GC, ST, NP>;
    auto kern = fwd_kernel<D, GC, ST, NP>;
    static bool attr_done[64] = {};   // one flag set per template instantiation
    cudaError_t e = ensure_smem_attr(kern, C::SMEM_BYTES, attr_done);
    if (e != cudaSuccess)
        return e;
    const unsigned grid = static_cast<unsigned>(p.M) * p.B * p.Hkv * p.nchunks;
    kern<<<grid, 320, C::SMEM_BYTES, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int d, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                       const AttnParams &p, cudaStream_t stream)
{
    switch (d) {
    case 32:
        switch (p.GC) {
        case 1: return launch_fwd_t<32, 1, 2, 2>(q, k, v, p, stream);
        case 2: return launch_fwd_t<32, 2, 2, 2>(q, k, v, p, stream);
        case 3: return launch_fwd_t<32, 3, 2, 2>(q, k, v, p, stream);
        case 4: return launch_fwd_t<32, 4, 2, 2>(q, k, v, p, stream);
        default: break;
        }
        break;
    case 64:
        switch (p.GC) {
        case 1: return launch_fwd_t<64, 1, 2, 2>(q, k, v, p, stream);
        case 2: return launch_fwd_t<64, 2, 2, 2>(q, k, v, p, stream);
        case 3: return launch_fwd_t<64, 3, 2, 2>(q, k, v, p, stream);
        case 4: return launch_fwd_t<64, 4, 2, 2>(q, k, v, p, stream);
        default: break;
        }
        break;
    case 128:
        switch (p.GC) {
        case 1: return launch_fwd_t<128, 1, 2, 1>(q, k, v, p, stream);
        case 2: return launch_fwd_t<128, 2, 2, 1>(q, k, v, p, stream);
        default: break;
        }
        break;
    default: break;
    }
    return cudaErrorInvalidValue;
}

} // namespace ne
