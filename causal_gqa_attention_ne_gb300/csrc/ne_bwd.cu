// ne_bwd.cu -- backward kernels of causal grouped-query attention with RoPE.
//
// The pages describe a hand-written backward validated by central finite
// differences (NanoEuler walkthrough, section 2.1; README "validation").  For
// L = sum(O * dO), with P = exp(S - lse):
//   D[t]  = <dO[t], O[t]>                       (bwd_pre_kernel)
//   dP    = dO V^T,  dS = P * (dP - D)
//   dV    = P^T dO      summed over the query heads of a KV head
//   dK'   = dS^T Q' / sqrt(d)                    (dkdv_kernel, key-tile major)
//   dQ'   = dS K'  / sqrt(d)                     (dq_kernel, query-tile major)
//   dq = R(t)^T dQ',  dk = R(s)^T dK'            (inverse RoPE in the epilogues)
// Every output element is produced by exactly one CTA with a fixed reduction
// order, so the backward is deterministic and uses no floating-point atomics.
#include <cuda_bf16.h>

#include "ne_common.cuh"
#include "ne_kernels.h"

namespace ne {

// ---------------------------------------------------------- preprocess ---

// One thread per 16-byte chunk (8 elements) of a (b, t, h) row; the D/8
// threads of a row reduce with shuffles.  Pure streaming over O and dO.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const AttnParams p)
{
    constexpr int TPR = D / 8;   // threads per row
    const size_t nrows = static_cast<size_t>(p.B) * p.T * p.Hq;
    const size_t nchunks = nrows * TPR;
    const uint4 *o = static_cast<const uint4 *>(p.o_in);
    const uint4 *g = static_cast<const uint4 *>(p.do_in);
    for (size_t c = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         c - (threadIdx.x % 32) < nchunks;   // keep whole warps in the loop for the shuffles
         c += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float acc = 0.f;
        if (c < nchunks) {
            const uint4 a = o[c], b = g[c];
            const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                acc += bf16_lo(av[e]) * bf16_lo(bv[e]) + bf16_hi(av[e]) * bf16_hi(bv[e]);
        }
#pragma unroll
        for (int off = TPR / 2; off >= 1; off /= 2)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (c < nchunks && (c % TPR) == 0) {
            const size_t row = c / TPR;                  // ((b*T + t)*Hq + h)
            const int h = static_cast<int>(row % p.Hq);
            const size_t bt = row / p.Hq;
            const int t = static_cast<int>(bt % p.T);
            const int b = static_cast<int>(bt / p.T);
            p.Dws[(static_cast<size_t>(b) * p.Hq + h) * p.T + t] = acc;
        }
    }
}

cudaError_t launch_bwd_pre(int d, const AttnParams &p, cudaStream_t stream)
{
    const size_t nchunks = static_cast<size_t>(p.B) * p.T * p.Hq * (d / 8);
    size_t blocks = (nchunks + 255) / 256;
    const size_t cap = 152 * 16;
    if (blocks > cap)
        blocks = cap;
    switch (d) {
    case 32: bwd_pre_kernel<32><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p); break;
    case 64: bwd_pre_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p); break;
    case 128: bwd_pre_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// Stores 32 consecutive fp32 values as bf16 (64 bytes).
__device__ __forceinline__ void store_row32_bf16(__nv_bfloat16 *dst, const float *v)
{
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        d4[q] = make_uint4(pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]),
                           pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]),
                           pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]),
                           pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]));
}

// Epilogue for a gradient of a rotated operand: reads the D fp32 columns of
// this thread's TMEM row at `col`, multiplies by `scale`, rotates back by
// -angle(pos) and stores bf16 to dst (when `store`).
template <int D>
__device__ __forceinline__ void epilogue_inverse_rope(uint32_t taddr, float scale, uint32_t pos,
                                                      const RopeFreqs &fr, __nv_bfloat16 *dst,
                                                      bool store)
{
    if constexpr (D >= 64) {
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
            uint32_t a[32], b[32];
            tmem_ld32(taddr + c0, a);
            tmem_ld32(taddr + c0 + D / 2, b);
            tmem_ld_wait(a);
            tmem_tie(b);
            float x[32], y[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                x[e] = __uint_as_float(a[e]) * scale;
                y[e] = __uint_as_float(b[e]) * scale;
                rope_inverse_pair(x[e], y[e], pos, fr.turn[c0 + e]);
            }
            if (store) {
                store_row32_bf16(dst + c0, x);
                store_row32_bf16(dst + c0 + D / 2, y);
            }
        }
    } else {
        uint32_t a[32];
        tmem_ld32(taddr, a);
        tmem_ld_wait(a);
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e)
            x[e] = __uint_as_float(a[e]) * scale;
#pragma unroll
        for (int e = 0; e < 16; ++e)
            rope_inverse_pair(x[e], x[e + 16], pos, fr.turn[e]);
        if (store)
            store_row32_bf16(dst, x);
    }
}

// ------------------------------------------------------------------ dQ ---
//
// CTA = (b, kv head j, query tile m, GC query heads).  Roles as in the
// forward kernel.  TMEM: S [0,128), dP [128,256), dQ of head g at 256 + g*D.

template <int D, int GC, int ST>
struct DqCfg {
    using TL = Tile<D>;
    static constexpr int PTILE = kRows * 128 * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = OFF_Q + GC * TL::BYTES;
    static constexpr int OFF_K = OFF_DO + GC * TL::BYTES;
    static constexpr int OFF_V = OFF_K + ST * TL::BYTES;
    static constexpr int OFF_DS = OFF_V + ST * TL::BYTES;
    static constexpr int SMEM_BYTES = smem_one_cta(OFF_DS + PTILE + 1024);
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(256 + GC * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <int D, int GC, int ST>
__global__ void __launch_bounds__(320, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const AttnParams p)
{
    using C = DqCfg<D, GC, ST>;
    using TL = Tile<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_q_full, bar_do_full, bar_q_ready, bar_drain;
    __shared__ uint64_t bar_k_full[ST], bar_k_ready[ST], bar_v_full[ST], bar_kv_empty[ST];
    __shared__ uint64_t bar_s_full, bar_s_empty, bar_ds_full, bar_dq_done[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ uint32_t abort_s;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
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
        mbar_init(smem_u32(&bar_do_full), 1);
        mbar_init(smem_u32(&bar_q_ready), 4);
        mbar_init(smem_u32(&bar_drain), 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&bar_k_full[s]), 1);
            mbar_init(smem_u32(&bar_k_ready[s]), 4);
            mbar_init(smem_u32(&bar_v_full[s]), 1);
            mbar_init(smem_u32(&bar_kv_empty[s]), 1);
        }
        mbar_init(smem_u32(&bar_s_full), 1);
        mbar_init(smem_u32(&bar_s_empty), 4);
        mbar_init(smem_u32(&bar_ds_full), 4);
        mbar_init(smem_u32(&bar_dq_done[0]), 1);
        mbar_init(smem_u32(&bar_dq_done[1]), 1);
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
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmDO);
            const uint32_t qb = smem_u32(&bar_q_full), db = smem_u32(&bar_do_full);
            mbar_arrive_expect_tx(qb, GC * TL::BYTES);
            for (int g = 0; g < GC; ++g)
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_Q + g * TL::BYTES + cb * TL::BLOCK), &tmQ,
                                qb, cb * TL::BOX_COLS, h0 + g, t0, b);
            mbar_arrive_expect_tx(db, GC * TL::BYTES);
            for (int g = 0; g < GC; ++g)
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_DO + g * TL::BYTES + cb * TL::BLOCK),
                                &tmDO, db, cb * TL::BOX_COLS, h0 + g, t0, b);
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
                mbar_wait_drain(smem_u32(&bar_do_full), 0, wc.limit_ns);
                for (int jk = (issued > ST ? issued - ST : 0); jk < issued; ++jk) {
                    const int st = jk % ST, u = jk / ST;
                    mbar_wait_drain(smem_u32(&bar_k_full[st]), u & 1, wc.limit_ns);
                    mbar_wait_drain(smem_u32(&bar_v_full[st]), u & 1, wc.limit_ns);
                }
            }
        }
    } else if (warp == 9) {
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_f16(128, 128, false, false, false);
            constexpr uint32_t ID_DP = idesc_f16(128, 128, true, false, false);
            constexpr uint32_t ID_DQ = idesc_f16(128, TL::NPV, false, false, true);
            const uint32_t q_addr = smem_u32(smem + C::OFF_Q);
            const uint32_t do_addr = smem_u32(smem + C::OFF_DO);
            const uint32_t k_addr = smem_u32(smem + C::OFF_K);
            const uint32_t v_addr = smem_u32(smem + C::OFF_V);
            const uint32_t ds_addr = smem_u32(smem + C::OFF_DS);
            bool ok = mbar_wait(smem_u32(&bar_q_ready), 0, wc) &&
                      mbar_wait(smem_u32(&bar_do_full), 0, wc);
            auto do_dq = [&](int x) -> bool {
                const int jx = x / GC, gx = x % GC, stx = jx % ST;
                if (!mbar_wait(smem_u32(&bar_ds_full), x & 1, wc))
                    return false;
                tc_fence_after();
                const uint32_t ka = k_addr + stx * TL::BYTES;
                const uint32_t dd = tbase + 256 + gx * D;
#pragma unroll
                for (int nc = 0; nc < D / TL::NPV; ++nc)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_f16_ss(dd + nc * TL::NPV, desc_ptile(ds_addr, kk),
                                   desc_mnmajor<D>(ka, nc, kk), ID_DQ,
                                   (jx > 0 || kk > 0) ? 1u : 0u);
                mma_commit(smem_u32(&bar_dq_done[x % 2]));
                if (gx == GC - 1)
                    mma_commit(smem_u32(&bar_kv_empty[stx]));
                return true;
            };
            for (int i = 0; ok && i < nitems; ++i) {
                const int jk = i / GC, g = i % GC, st = jk % ST;
                if (g == 0 && !(mbar_wait(smem_u32(&bar_k_ready[st]), (jk / ST) & 1, wc) &&
                                mbar_wait(smem_u32(&bar_v_full[st]), (jk / ST) & 1, wc))) {
                    ok = false;
                    break;
                }
                if (i >= 1 && !mbar_wait(smem_u32(&bar_s_empty), (i - 1) & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t qa = q_addr + g * TL::BYTES, oa = do_addr + g * TL::BYTES;
                const uint32_t ka = k_addr + st * TL::BYTES, va = v_addr + st * TL::BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_f16_ss(tbase, desc_kmajor<D>(qa, kk), desc_kmajor<D>(ka, kk), ID_S,
                               kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_f16_ss(tbase + 128, desc_kmajor<D>(oa, kk), desc_kmajor<D>(va, kk), ID_DP,
                               kk > 0 ? 1u : 0u);
                mma_commit(smem_u32(&bar_s_full));
                if (i >= 1 && !do_dq(i - 1)) {
                    ok = false;
                    break;
                }
            }
            if (ok)
                do_dq(nitems - 1);
            mma_commit(smem_u32(&bar_drain));
            mbar_wait(smem_u32(&bar_drain), 0, wc);
        }
    } else if (warp >= 4) {
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
        const int r = threadIdx.x;
        const int t = t0 + r;
        const uint32_t lane_base = tmem_addr(tbase, warp * 32, 0);
        float lse2[GC], Dv[GC];
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            const size_t idx = (static_cast<size_t>(b) * p.Hq + h0 + g) * p.T + t;
            lse2[g] = (t < p.T) ? p.lse[idx] * kLog2e : 0.f;
            Dv[g] = (t < p.T) ? p.Dws[idx] : 0.f;
        }
        float maxds = 0.f;
        bool ok = true;
        uint8_t *dst = smem + C::OFF_DS;
        for (int i = 0; i < nitems; ++i) {
            const int jk = i / GC, g = i % GC;
            if (!mbar_wait_warp(smem_u32(&bar_s_full), i & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (i >= 1 &&
                !mbar_wait_warp(smem_u32(&bar_dq_done[(i - 1) % 2]), ((i - 1) / 2) & 1, wc)) {
                ok = false;
                break;
            }
            const bool diag = (jk == m);
            const float lg = lse2[g], dg = Dv[g];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t sv[32], pv[32];
                tmem_ld32(lane_base + cc * 32, sv);
                tmem_ld32(lane_base + 128 + cc * 32, pv);
                tmem_ld_wait(sv);
                tmem_tie(pv);
                if (cc == 3) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_u32(&bar_s_empty));
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int c = cc * 32 + e;
                    float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), p.scale_log2, -lg));
                    float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), p.scale_log2, -lg));
                    if (diag && c > r)
                        p0 = 0.f;
                    if (diag && c + 1 > r)
                        p1 = 0.f;
                    const float d0 = p0 * (__uint_as_float(pv[e]) - dg);
                    const float d1 = p1 * (__uint_as_float(pv[e + 1]) - dg);
                    maxds = fmaxf(maxds, fmaxf(fabsf(d0), fabsf(d1)));
                    pk[e / 2] = pack_f16x2(d0, d1);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4 *>(dst + ptile_chunk(r, cc * 4 + q)) =
                        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_ds_full));
        }
        if (maxds > kFp16Max)
            atomicOr(p.status, kDevRange);
        if (ok) {
            const int x = nitems - 1;
            ok = mbar_wait_warp(smem_u32(&bar_dq_done[x % 2]), (x / 2) & 1, wc);
        }
        if (ok) {
            tc_fence_after();
            __nv_bfloat16 *dq = static_cast<__nv_bfloat16 *>(p.out0);
#pragma unroll
            for (int g = 0; g < GC; ++g) {
                __nv_bfloat16 *row =
                    dq + ((static_cast<size_t>(b) * p.T + t) * p.Hq + h0 + g) * D;
                epilogue_inverse_rope<D>(lane_base + 256 + g * D, p.scale,
                                         static_cast<uint32_t>(t), p.rope, row, t < p.T);
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

// ---------------------------------------------------------------- dK dV ---
//
// CTA = (b, kv head j, key tile n).  K' and V stay in shared memory; the loop
// runs over the G query heads of the group and the causal query tiles m >= n.
// Transposed scores: thread r owns key row r.  TMEM: S^T [0,128),
// dP^T [128,256), dV [256, 256+D), dK [256+D, 256+2D).

template <int D, int ST>
struct DkvCfg {
    using TL = Tile<D>;
    static constexpr int PTILE = kRows * 128 * 2;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = TL::BYTES;
    static constexpr int OFF_Q = 2 * TL::BYTES;
    static constexpr int OFF_DO = OFF_Q + ST * TL::BYTES;
    static constexpr int OFF_PT = OFF_DO + ST * TL::BYTES;
    static constexpr int OFF_DST = OFF_PT + PTILE;
    static constexpr int SMEM_BYTES = smem_one_cta(OFF_DST + PTILE + 1024);
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(256 + 2 * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <int D, int ST>
__global__ void __launch_bounds__(320, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                const AttnParams p)
{
    using C = DkvCfg<D, ST>;
    using TL = Tile<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_k_full, bar_v_full, bar_k_ready, bar_drain, bar_acc_done;
    __shared__ uint64_t bar_q_full[ST], bar_do_full[ST], bar_q_ready[ST], bar_st_empty[ST];
    __shared__ uint64_t bar_s_full, bar_s_empty, bar_pds_full, bar_pds_empty;
    __shared__ float2 lsed[2][kRows];
    __shared__ uint32_t tmem_base_s;
    __shared__ uint32_t abort_s;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int per_n = p.B * p.Hkv;
    const int n = static_cast<int>(blockIdx.x) / per_n;   // heaviest (n = 0) first
    const int rem = static_cast<int>(blockIdx.x) % per_n;
    const int j = rem % p.Hkv;
    const int b = rem / p.Hkv;
    const int s0 = n * kRows;
    const int nitems = (p.M - n) * p.G;

    if (threadIdx.x == 0) {
        abort_s = 0;
        mbar_init(smem_u32(&bar_k_full), 1);
        mbar_init(smem_u32(&bar_v_full), 1);
        mbar_init(smem_u32(&bar_k_ready), 4);
        mbar_init(smem_u32(&bar_drain), 1);
        mbar_init(smem_u32(&bar_acc_done), 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&bar_q_full[s]), 1);
            mbar_init(smem_u32(&bar_do_full[s]), 1);
            mbar_init(smem_u32(&bar_q_ready[s]), 4);
            mbar_init(smem_u32(&bar_st_empty[s]), 1);
        }
        mbar_init(smem_u32(&bar_s_full), 1);
        mbar_init(smem_u32(&bar_s_empty), 4);
        mbar_init(smem_u32(&bar_pds_full), 4);
        mbar_init(smem_u32(&bar_pds_empty), 1);
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
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmDO);
            const uint32_t kb = smem_u32(&bar_k_full), vb = smem_u32(&bar_v_full);
            mbar_arrive_expect_tx(kb, TL::BYTES);
            for (int cb = 0; cb < TL::NB; ++cb)
                tma_load_4d(smem_u32(smem + C::OFF_K + cb * TL::BLOCK), &tmK, kb,
                            cb * TL::BOX_COLS, j, s0, b);
            mbar_arrive_expect_tx(vb, TL::BYTES);
            for (int cb = 0; cb < TL::NB; ++cb)
                tma_load_4d(smem_u32(smem + C::OFF_V + cb * TL::BLOCK), &tmV, vb,
                            cb * TL::BOX_COLS, j, s0, b);
            int issued = 0;
            for (int i = 0; i < nitems; ++i) {
                const int st = i % ST, u = i / ST;
                if (u >= 1 && !mbar_wait(smem_u32(&bar_st_empty[st]), (u - 1) & 1, wc))
                    break;
                const int mt = n + i / p.G, h = j * p.G + i % p.G;
                const uint32_t qb = smem_u32(&bar_q_full[st]), db = smem_u32(&bar_do_full[st]);
                mbar_arrive_expect_tx(qb, TL::BYTES);
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_Q + st * TL::BYTES + cb * TL::BLOCK), &tmQ,
                                qb, cb * TL::BOX_COLS, h, mt * kRows, b);
                mbar_arrive_expect_tx(db, TL::BYTES);
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_DO + st * TL::BYTES + cb * TL::BLOCK),
                                &tmDO, db, cb * TL::BOX_COLS, h, mt * kRows, b);
                issued = i + 1;
            }
            if (*wc.abort) {
                mbar_wait_drain(smem_u32(&bar_k_full), 0, wc.limit_ns);
                mbar_wait_drain(smem_u32(&bar_v_full), 0, wc.limit_ns);
                for (int i = (issued > ST ? issued - ST : 0); i < issued; ++i) {
                    const int st = i % ST, u = i / ST;
                    mbar_wait_drain(smem_u32(&bar_q_full[st]), u & 1, wc.limit_ns);
                    mbar_wait_drain(smem_u32(&bar_do_full[st]), u & 1, wc.limit_ns);
                }
            }
        }
    } else if (warp == 9) {
        if (lane == 0) {
            constexpr uint32_t ID_S = idesc_f16(128, 128, false, false, false);
            constexpr uint32_t ID_DP = idesc_f16(128, 128, true, false, false);
            constexpr uint32_t ID_DV = idesc_f16(128, TL::NPV, true, false, true);
            constexpr uint32_t ID_DK = idesc_f16(128, TL::NPV, false, false, true);
            const uint32_t k_addr = smem_u32(smem + C::OFF_K);
            const uint32_t v_addr = smem_u32(smem + C::OFF_V);
            const uint32_t q_addr = smem_u32(smem + C::OFF_Q);
            const uint32_t do_addr = smem_u32(smem + C::OFF_DO);
            const uint32_t pt_addr = smem_u32(smem + C::OFF_PT);
            const uint32_t dst_addr = smem_u32(smem + C::OFF_DST);
            bool ok = mbar_wait(smem_u32(&bar_k_ready), 0, wc) &&
                      mbar_wait(smem_u32(&bar_v_full), 0, wc);
            auto do_acc = [&](int x) -> bool {
                const int stx = x % ST;
                if (!mbar_wait(smem_u32(&bar_pds_full), x & 1, wc))
                    return false;
                tc_fence_after();
                const uint32_t oa = do_addr + stx * TL::BYTES, qa = q_addr + stx * TL::BYTES;
#pragma unroll
                for (int nc = 0; nc < D / TL::NPV; ++nc)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_f16_ss(tbase + 256 + nc * TL::NPV, desc_ptile(pt_addr, kk),
                                   desc_mnmajor<D>(oa, nc, kk), ID_DV,
                                   (x > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int nc = 0; nc < D / TL::NPV; ++nc)
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_f16_ss(tbase + 256 + D + nc * TL::NPV, desc_ptile(dst_addr, kk),
                                   desc_mnmajor<D>(qa, nc, kk), ID_DK,
                                   (x > 0 || kk > 0) ? 1u : 0u);
                mma_commit(smem_u32(&bar_pds_empty));
                mma_commit(smem_u32(&bar_st_empty[stx]));
                return true;
            };
            for (int i = 0; ok && i < nitems; ++i) {
                const int st = i % ST, u = i / ST;
                if (!(mbar_wait(smem_u32(&bar_q_ready[st]), u & 1, wc) &&
                      mbar_wait(smem_u32(&bar_do_full[st]), u & 1, wc))) {
                    ok = false;
                    break;
                }
                if (i >= 1 && !mbar_wait(smem_u32(&bar_s_empty), (i - 1) & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t qa = q_addr + st * TL::BYTES, oa = do_addr + st * TL::BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_f16_ss(tbase, desc_kmajor<D>(k_addr, kk), desc_kmajor<D>(qa, kk), ID_S,
                               kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    mma_f16_ss(tbase + 128, desc_kmajor<D>(v_addr, kk), desc_kmajor<D>(oa, kk),
                               ID_DP, kk > 0 ? 1u : 0u);
                mma_commit(smem_u32(&bar_s_full));
                // With two or more Q/dO stages, item i's S^T and dP^T are issued
                // before item i-1's dV/dK so the tensor core overlaps the softmax
                // work; with a single stage, item i's tile can only land after
                // item i-1's dV/dK have released the stage, so they go in order.
                const int acc_item = (ST >= 2) ? i - 1 : i;
                if (acc_item >= 0 && !do_acc(acc_item)) {
                    ok = false;
                    break;
                }
            }
            if (ok && (ST == 1 || do_acc(nitems - 1)))
                mma_commit(smem_u32(&bar_acc_done));
            mma_commit(smem_u32(&bar_drain));
            mbar_wait(smem_u32(&bar_drain), 0, wc);
        }
    } else if (warp >= 4) {
        const int r = threadIdx.x - 128;
        float mx = 0.f;
        bool ok = mbar_wait_warp(smem_u32(&bar_k_full), 0, wc);
        if (ok) {
            mx = rope_row_to_f16<D>(smem + C::OFF_K, r, static_cast<uint32_t>(s0 + r), p.rope);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_k_ready));
            for (int i = 0; i < nitems; ++i) {
                const int st = i % ST, u = i / ST;
                const int mt = n + i / p.G;
                if (!mbar_wait_warp(smem_u32(&bar_q_full[st]), u & 1, wc))
                    break;
                mx = fmaxf(mx, rope_row_to_f16<D>(smem + C::OFF_Q + st * TL::BYTES, r,
                                                  static_cast<uint32_t>(mt * kRows + r), p.rope));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_q_ready[st]));
            }
        }
        if (mx > kFp16Max)
            atomicOr(p.status, kDevRange);
    } else {
        const int r = threadIdx.x;            // key row == TMEM lane
        const int s = s0 + r;
        const uint32_t lane_base = tmem_addr(tbase, warp * 32, 0);
        auto fetch = [&](int i, float &l2, float &dd) {
            const int mt = n + i / p.G, h = j * p.G + i % p.G;
            const int t = mt * kRows + r;
            const size_t idx = (static_cast<size_t>(b) * p.Hq + h) * p.T + t;
            l2 = (t < p.T) ? p.lse[idx] * kLog2e : INFINITY;
            dd = (t < p.T) ? p.Dws[idx] : 0.f;
        };
        float nl2, ndd;
        fetch(0, nl2, ndd);
        float maxds = 0.f;
        bool ok = true;
        uint8_t *pt = smem + C::OFF_PT;
        uint8_t *dst = smem + C::OFF_DST;
        for (int i = 0; i < nitems; ++i) {
            const int mt = n + i / p.G;
            lsed[i % 2][r] = make_float2(nl2, ndd);
            if (i + 1 < nitems)
                fetch(i + 1, nl2, ndd);
            // Every warp passes this barrier once per item, also after an
            // abort (a failed warp keeps looping without work), so no warp is
            // ever left waiting here.
            named_bar_sync(1, 128);
            if (!ok)
                continue;
            if (!mbar_wait_warp(smem_u32(&bar_s_full), i & 1, wc)) {
                ok = false;
                continue;
            }
            tc_fence_after();
            if (i >= 1 && !mbar_wait_warp(smem_u32(&bar_pds_empty), (i - 1) & 1, wc)) {
                ok = false;
                continue;
            }
            const bool diag = (mt == n);
            const float2 *ld = lsed[i % 2];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t sv[32], pv[32];
                tmem_ld32(lane_base + cc * 32, sv);
                tmem_ld32(lane_base + 128 + cc * 32, pv);
                tmem_ld_wait(sv);
                tmem_tie(pv);
                if (cc == 3) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_u32(&bar_s_empty));
                }
                uint32_t pp[16], dk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int c = cc * 32 + e;
                    const float2 a0 = ld[c], a1 = ld[c + 1];
                    float p0 = ex2_approx(fmaf(__uint_as_float(sv[e]), p.scale_log2, -a0.x));
                    float p1 = ex2_approx(fmaf(__uint_as_float(sv[e + 1]), p.scale_log2, -a1.x));
                    if (diag && c < r)
                        p0 = 0.f;
                    if (diag && c + 1 < r)
                        p1 = 0.f;
                    const float d0 = p0 * (__uint_as_float(pv[e]) - a0.y);
                    const float d1 = p1 * (__uint_as_float(pv[e + 1]) - a1.y);
                    maxds = fmaxf(maxds, fmaxf(fabsf(d0), fabsf(d1)));
                    pp[e / 2] = pack_bf16x2(p0, p1);
                    dk[e / 2] = pack_f16x2(d0, d1);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t off = ptile_chunk(r, cc * 4 + q);
                    *reinterpret_cast<uint4 *>(pt + off) =
                        make_uint4(pp[4 * q], pp[4 * q + 1], pp[4 * q + 2], pp[4 * q + 3]);
                    *reinterpret_cast<uint4 *>(dst + off) =
                        make_uint4(dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_pds_full));
        }
        if (maxds > kFp16Max)
            atomicOr(p.status, kDevRange);
        if (ok)
            ok = mbar_wait_warp(smem_u32(&bar_acc_done), 0, wc);
        if (ok) {
            tc_fence_after();
            const size_t rowoff = ((static_cast<size_t>(b) * p.T + s) * p.Hkv + j) * D;
            __nv_bfloat16 *dv = static_cast<__nv_bfloat16 *>(p.out1) + rowoff;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t a[32];
                tmem_ld32(lane_base + 256 + cc * 32, a);
                tmem_ld_wait(a);
                float x[32];
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    x[e] = __uint_as_float(a[e]);
                if (s < p.T)
                    store_row32_bf16(dv + cc * 32, x);
            }
            __nv_bfloat16 *dk = static_cast<__nv_bfloat16 *>(p.out0) + rowoff;
            epilogue_inverse_rope<D>(lane_base + 256 + D, p.scale, static_cast<uint32_t>(s),
                                     p.rope, dk, s < p.T);
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

template <int D, int GC, int ST>
static cudaError_t launch_dq_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                               const CUtensorMap &dO, const AttnParams &p, cudaStream_t stream)
{
    using C = DqCfg<D, GC, ST>;
    auto kern = dq_kernel<D, GC, ST>;
    static bool attr_done[64] = {};   // one flag set per template instantiation
    cudaError_t e = ensure_smem_attr(kern, C::SMEM_BYTES, attr_done);
    if (e != cudaSuccess)
        return e;
    const unsigned grid = static_cast<unsigned>(p.M) * p.B * p.Hkv * p.nchunks;
    kern<<<grid, 320, C::SMEM_BYTES, stream>>>(q, k, v, dO, p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(int d, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                          const CUtensorMap &dO, const AttnParams &p, cudaStream_t stream)
{
    switch (d) {
    case 32:
        switch (p.GC) {
        case 1: return launch_dq_t<32, 1, 2>(q, k, v, dO, p, stream);
        case 2: return launch_dq_t<32, 2, 2>(q, k, v, dO, p, stream);
        case 3: return launch_dq_t<32, 3, 2>(q, k, v, dO, p, stream);
        case 4: return launch_dq_t<32, 4, 2>(q, k, v, dO, p, stream);
        default: break;
        }
        break;
    case 64:
        switch (p.GC) {
        case 1: return launch_dq_t<64, 1, 2>(q, k, v, dO, p, stream);
        case 2: return launch_dq_t<64, 2, 2>(q, k, v, dO, p, stream);
        case 3: return launch_dq_t<64, 3, 2>(q, k, v, dO, p, stream);
        case 4: return launch_dq_t<64, 4, 2>(q, k, v, dO, p, stream);
        default: break;
        }
        break;
    case 128:
        if (p.GC == 1)
            return launch_dq_t<128, 1, 2>(q, k, v, dO, p, stream);
        break;
    default: break;
    }
    return cudaErrorInvalidValue;
}

template <int D, int ST>
static cudaError_t launch_dkdv_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                 const CUtensorMap &dO, const AttnParams &p, cudaStream_t stream)
{
    using C = DkvCfg<D, ST>;
    auto kern = dkdv_kernel<D, ST>;
    static bool attr_done[64] = {};   // one flag set per template instantiation
    cudaError_t e = ensure_smem_attr(kern, C::SMEM_BYTES, attr_done);
    if (e != cudaSuccess)
        return e;
    const unsigned grid = static_cast<unsigned>(p.M) * p.B * p.Hkv;
    kern<<<grid, 320, C::SMEM_BYTES, stream>>>(q, k, v, dO, p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(int d, const CUtensorMap &q, const CUtensorMap &k,
                            const CUtensorMap &v, const CUtensorMap &dO, const AttnParams &p,
                            cudaStream_t stream)
{
    switch (d) {
    case 32: return launch_dkdv_t<32, 2>(q, k, v, dO, p, stream);
    case 64: return launch_dkdv_t<64, 2>(q, k, v, dO, p, stream);
    case 128: return launch_dkdv_t<128, 1>(q, k, v, dO, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace ne
