// ne_decode.cu -- decode attention against a key/value cache: one new token
// per sequence attends over the Tk cached positions (its own key and value
// are the cache's last rows, so it sits at position Tk - 1 and sees every
// key).  By definition this is the last row of the causal GQA + RoPE
// attention of the training kernels, for the chat loop the NanoEuler README
// describes (its KV-cache inference engine).
//
// It reads every cached key and value once and does 4*d flops per key and
// query head, so it is bound by HBM bandwidth: CUDA cores, no tensor cores.
// Split over the keys into work items (b, kv head j, chunk c of CH = 128
// keys).  Persistent: two CTAs per SM (one at d = 128) each walk their share
// of the items with the chunk's K and V tiles streamed by TMA through a ring
// of shared-memory stages, so the next items' loads are in flight while one
// is computed.  Per item, one thread per key reads its key row from the
// swizzled tile, rotates it at its position pair by pair straight into its
// scores against the G query heads of the group (rotated once per item at
// Tk - 1); then one partial (max, sum, O) per head.  A second kernel merges
// the partials of each (b, h) in chunk order: deterministic, no atomics.
#include <cuda_bf16.h>

#include "ne_common.cuh"
#include "ne_kernels.h"

namespace ne {

constexpr int kDecCh = 128;        // keys per work item (one per thread)
constexpr int kDecThreads = 256;   // two per key

template <int D>
struct DecCfg {
    using TL = Tile<D>;
    static constexpr int ST = (D == 128) ? 2 : 3;              // K/V stages
    static constexpr int CTAS = (D == 128) ? 1 : 2;            // per SM
    static constexpr int STAGE = 2 * TL::BYTES;                // K tile, V tile
    static constexpr int OFF_Q = ST * STAGE;                   // float [G][D]
    static constexpr int OFF_P = OFF_Q + kMaxDecodeGroup * D * 4;          // float [G][CH]
    static constexpr int OFF_ML = OFF_P + kMaxDecodeGroup * kDecCh * 4;    // float [G][2]
    static constexpr int BYTES = OFF_ML + kMaxDecodeGroup * 2 * 4 + 1024;  // + alignment
    static_assert(CTAS * BYTES <= 232448, "shared memory budget");
};

// The P V step's split: key groups of threads, each over a column pair per
// thread, as many as 128 threads hold and the K tile holds their sums
// ([KG][G][D] floats).
template <int D, int GB>
struct PvCfg {
    static constexpr int byfit = Tile<D>::BYTES / (GB * D * 4);
    static constexpr int bythreads = kDecThreads / (D / 2);
    static constexpr int KG = byfit < bythreads ? byfit : bythreads;
    static_assert(KG >= 1 && kDecCh % KG == 0, "P V key groups");
};

// GB = the group size G rounded up to a power of two (the kernel keeps GB
// score accumulators per thread; heads g >= G are skipped).
template <int D, int GB>
__global__ void __launch_bounds__(kDecThreads, (D == 128) ? 1 : 2)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const DecodeParams p)
{
    using C = DecCfg<D>;
    using TL = Tile<D>;
    constexpr int ST = C::ST;
    constexpr int HC = D / 16;     // chunks in the first half of a row
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_full[ST];
    __shared__ uint32_t abort_s;
    float *qs = reinterpret_cast<float *>(smem + C::OFF_Q);
    float *ps = reinterpret_cast<float *>(smem + C::OFF_P);
    float *ml = reinterpret_cast<float *>(smem + C::OFF_ML);

    const int t = threadIdx.x, lane = t % 32, warp = t / 32;
    const int G = p.G;
    const int nitems = p.B * p.Hkv * p.nchunks;
    if (t == 0) {
        abort_s = 0;
        for (int s = 0; s < ST; ++s)
            mbar_init(smem_u32(&bar_full[s]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    griddep_wait();
    const WaitCtl wc{&abort_s, p.status, p.wait_limit_ns};
    // the k-th item of this CTA: its K and V tiles into stage k % ST (thread 0)
    int issued = 0;
    auto issue = [&](int k) {
        const int it = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
        if (it >= nitems)
            return;
        const int c = it % p.nchunks, j = (it / p.nchunks) % p.Hkv, b = it / (p.nchunks * p.Hkv);
        const uint32_t bar = smem_u32(&bar_full[k % ST]);
        uint8_t *stg = smem + (k % ST) * C::STAGE;
        mbar_arrive_expect_tx(bar, 2 * TL::BYTES);
        for (int cb = 0; cb < TL::NB; ++cb) {
            tma_load_4d(smem_u32(stg + cb * TL::BLOCK), &tmK, bar, cb * TL::BOX_COLS, j,
                        c * kDecCh, b);
            tma_load_4d(smem_u32(stg + TL::BYTES + cb * TL::BLOCK), &tmV, bar, cb * TL::BOX_COLS,
                        j, c * kDecCh, b);
        }
        issued = k + 1;
    };
    if (t == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        for (int k = 0; k < ST; ++k)
            issue(k);
    }
    const uint32_t qpos = static_cast<uint32_t>(p.Tk - 1);
    const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
    bool ok = true;
    int k = 0;
    for (;; ++k) {
        const int it = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
        if (it >= nitems)
            break;
        const int c = it % p.nchunks, j = (it / p.nchunks) % p.Hkv, b = it / (p.nchunks * p.Hkv);
        const int s0 = c * kDecCh;
        // the group's G query rows, rotated at position Tk - 1, in fp32 (while
        // the tiles land)
        for (int idx = t; idx < G * (D / 2); idx += kDecThreads) {
            const int g = idx / (D / 2), i = idx % (D / 2);
            const __nv_bfloat16 *qrow = qg + (static_cast<size_t>(b) * p.Hq + j * G + g) * D;
            float sn, cs;
            rope_sincos(qpos, p.rope, i, sn, cs);
            const float x = __bfloat162float(qrow[i]), y = __bfloat162float(qrow[i + D / 2]);
            qs[g * D + i] = x * cs - y * sn;
            qs[g * D + i + D / 2] = y * cs + x * sn;
        }
        ok = mbar_wait_warp(smem_u32(&bar_full[k % ST]), (k / ST) & 1, wc);
        if (!__syncthreads_and(ok))
            break;
        const uint8_t *kt = smem + (k % ST) * C::STAGE, *vt = kt + TL::BYTES;

        // two threads per key (its row from the tile, zero past Tk): each
        // rotates half of the rotate-half pairs straight into partial scores
        // against the G query heads; the pair of threads adds its halves
        {
            const int key = t >> 1, half = t & 1;
            const int s = s0 + key;
            float acc[GB];
#pragma unroll
            for (int g = 0; g < GB; ++g)
                acc[g] = 0.f;
            if (s < p.Tk) {
#pragma unroll
                for (int c2 = 0; c2 < HC / 2; ++c2) {
                    const int cc = half * (HC / 2) + c2;
                    const uint4 a4 = *reinterpret_cast<const uint4 *>(kt + tile_chunk<D>(key, cc));
                    const uint4 b4 =
                        *reinterpret_cast<const uint4 *>(kt + tile_chunk<D>(key, cc + HC));
                    const uint32_t av[4] = {a4.x, a4.y, a4.z, a4.w},
                                   bv[4] = {b4.x, b4.y, b4.z, b4.w};
                    float xr[8], yr[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float sn, cs;
                        rope_sincos(static_cast<uint32_t>(s), p.rope, 8 * cc + e, sn, cs);
                        const float x = (e & 1) ? bf16_hi(av[e >> 1]) : bf16_lo(av[e >> 1]);
                        const float y = (e & 1) ? bf16_hi(bv[e >> 1]) : bf16_lo(bv[e >> 1]);
                        xr[e] = x * cs - y * sn;
                        yr[e] = y * cs + x * sn;
                    }
                    // the heads' query values for these 8 pairs: 16-byte
                    // loads, two addresses per warp (broadcast)
#pragma unroll
                    for (int g = 0; g < GB; ++g)
                        if (g < G) {
                            const float4 *qa = reinterpret_cast<const float4 *>(qs + g * D + 8 * cc);
                            const float4 *qb =
                                reinterpret_cast<const float4 *>(qs + g * D + D / 2 + 8 * cc);
                            const float4 q0 = qa[0], q1 = qa[1], r0 = qb[0], r1 = qb[1];
                            const float qx[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                            const float qy[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                acc[g] = fmaf(qy[e], yr[e], fmaf(qx[e], xr[e], acc[g]));
                        }
                }
            }
#pragma unroll
            for (int g = 0; g < GB; ++g) {
                acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 1);
                if (g < G && half == 0)
                    ps[g * kDecCh + key] = s < p.Tk ? acc[g] * p.scale_log2 : -INFINITY;
            }
        }
        __syncthreads();

        // per head: the chunk's max m, P = 2^(S - m) and its sum l (warp w
        // takes heads w, w + 4, ...; every chunk has at least one key, so m is
        // finite)
        for (int g = warp; g < G; g += kDecThreads / 32) {
            float *row = ps + g * kDecCh;
            float m = -INFINITY;
            for (int r = lane; r < kDecCh; r += 32)
                m = fmaxf(m, row[r]);
#pragma unroll
            for (int off = 16; off >= 1; off /= 2)
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            float l = 0.f;
            for (int r = lane; r < kDecCh; r += 32) {
                const float pr = ex2_approx(row[r] - m);
                row[r] = pr;
                l += pr;
            }
#pragma unroll
            for (int off = 16; off >= 1; off /= 2)
                l += __shfl_xor_sync(0xffffffffu, l, off);
            if (lane == 0) {
                ml[2 * g] = m;
                ml[2 * g + 1] = l;
            }
        }
        __syncthreads();

        // O_g[e..e+1] = sum_r P_g[r] v[r][e..e+1]: thread (key group kg,
        // column pair cp) sums its KG-th of the keys for every head (one V
        // load per key, P read as a broadcast), then the key groups' sums
        // meet in the K tile (no longer needed) and go out as the partials
        const size_t part0 = (static_cast<size_t>(b) * p.Hq + j * G) * p.nchunks + c;
        {
            constexpr int CP = D / 2;                       // column pairs
            constexpr int KG = PvCfg<D, GB>::KG;            // key groups
            constexpr int KPG = kDecCh / KG;                // keys per group
            const int kg = t / CP, cp = t % CP, e = 2 * cp;
            float *red = reinterpret_cast<float *>(const_cast<uint8_t *>(kt));   // [KG][G][D]
            if (kg < KG) {
                float a0[GB], a1[GB];
#pragma unroll
                for (int g = 0; g < GB; ++g)
                    a0[g] = a1[g] = 0.f;
#pragma unroll 8
                for (int r = kg * KPG; r < (kg + 1) * KPG; ++r) {
                    const uint32_t off = tile_chunk<D>(r, e >> 3) + (e & 7) * 2;
                    const uint32_t v2 = *reinterpret_cast<const uint32_t *>(vt + off);
                    const float v0 = bf16_lo(v2), v1 = bf16_hi(v2);
#pragma unroll
                    for (int g = 0; g < GB; ++g)
                        if (g < G) {
                            const float pr = ps[g * kDecCh + r];
                            a0[g] = fmaf(pr, v0, a0[g]);
                            a1[g] = fmaf(pr, v1, a1[g]);
                        }
                }
#pragma unroll
                for (int g = 0; g < GB; ++g)
                    if (g < G)
                        *reinterpret_cast<float2 *>(red + (kg * G + g) * D + e) =
                            make_float2(a0[g], a1[g]);
            }
            __syncthreads();
            for (int o = t; o < G * CP; o += kDecThreads) {
                const int g = o / CP, e2 = 2 * (o % CP);
                float s0v = 0.f, s1v = 0.f;
#pragma unroll
                for (int q = 0; q < KG; ++q) {
                    const float2 v = *reinterpret_cast<const float2 *>(red + (q * G + g) * D + e2);
                    s0v += v.x;
                    s1v += v.y;
                }
                float *dst = p.part_o + (part0 + static_cast<size_t>(g) * p.nchunks) * D + e2;
                *reinterpret_cast<float2 *>(dst) = make_float2(s0v, s1v);
            }
        }
        if (t < G) {
            const size_t pi = part0 + static_cast<size_t>(t) * p.nchunks;
            p.part_ml[2 * pi] = ml[2 * t];
            p.part_ml[2 * pi + 1] = ml[2 * t + 1];
        }
        __syncthreads();   // the stage, qs and ps are free
        if (t == 0)
            issue(k + ST);
    }
    // after a timeout, the loads still in flight land before the CTA exits
    if (t == 0 && *wc.abort)
        for (int kk = k; kk < issued; ++kk)
            mbar_wait_drain(smem_u32(&bar_full[kk % ST]), (kk / ST) & 1, wc.limit_ns);
    griddep_launch_dependents();
}

// One CTA per (b, h), thread e owns column e: merge the chunk partials in
// chunk order, O = sum_c O_c 2^(m_c - M) / sum_c l_c 2^(m_c - M).
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeParams p)
{
    const int e = threadIdx.x;
    const size_t bh = blockIdx.x;      // b * Hq + h
    griddep_wait();
    const float *ml = p.part_ml + 2 * bh * p.nchunks;
    const float *po = p.part_o + bh * p.nchunks * D;
    float M = -INFINITY;
    for (int c = 0; c < p.nchunks; ++c)
        M = fmaxf(M, ml[2 * c]);
    float l = 0.f, acc = 0.f;
    for (int c = 0; c < p.nchunks; ++c) {
        const float w = ex2_approx(ml[2 * c] - M);
        l = fmaf(ml[2 * c + 1], w, l);
        acc = fmaf(po[static_cast<size_t>(c) * D + e], w, acc);
    }
    static_cast<__nv_bfloat16 *>(p.o)[bh * D + e] = __float2bfloat16_rn(acc / l);
    if (e == 0)
        p.lse[bh] = (M + __log2f(l)) * kLn2;
    griddep_launch_dependents();
}

int decode_chunk_keys() { return kDecCh; }

template <int D, int GB>
static cudaError_t launch_decode_t(const CUtensorMap &k, const CUtensorMap &v,
                                   const DecodeParams &p, cudaStream_t stream)
{
    using C = DecCfg<D>;
    auto kern = decode_partial_kernel<D, GB>;
    static bool attr_done[64] = {};   // one flag set per template instantiation
    cudaError_t e = ensure_smem_attr(kern, C::BYTES, attr_done);
    if (e != cudaSuccess)
        return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int nitems = p.B * p.Hkv * p.nchunks;
    const int grid = nitems < C::CTAS * sms ? nitems : C::CTAS * sms;
    if ((e = launch_pdl(kern, static_cast<unsigned>(grid), kDecThreads, C::BYTES, stream, k, v,
                        p)) != cudaSuccess)
        return e;
    return launch_pdl(decode_combine_kernel<D>, static_cast<unsigned>(p.B * p.Hq), D, 0, stream,
                      p);
}

template <int D>
static cudaError_t launch_decode_d(const CUtensorMap &k, const CUtensorMap &v,
                                   const DecodeParams &p, cudaStream_t stream)
{
    if (p.G <= 1)
        return launch_decode_t<D, 1>(k, v, p, stream);
    if (p.G <= 2)
        return launch_decode_t<D, 2>(k, v, p, stream);
    if (p.G <= 4)
        return launch_decode_t<D, 4>(k, v, p, stream);
    if (p.G <= 8)
        return launch_decode_t<D, 8>(k, v, p, stream);
    return launch_decode_t<D, 16>(k, v, p, stream);
}

cudaError_t launch_decode(int d, const CUtensorMap &k, const CUtensorMap &v,
                          const DecodeParams &p, cudaStream_t stream)
{
    switch (d) {
    case 32: return launch_decode_d<32>(k, v, p, stream);
    case 64: return launch_decode_d<64>(k, v, p, stream);
    case 128: return launch_decode_d<128>(k, v, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace ne
