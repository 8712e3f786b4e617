// ne_decode.cu -- decode attention against a key/value cache: one new token
// per sequence attends over the Tk cached positions (its own key and value
// are the cache's last rows, so it sits at position Tk - 1 and sees every
// key).  By definition this is the last row of the causal GQA + RoPE
// attention of the training kernels, for the chat loop the NanoEuler README
// describes (its KV-cache inference engine).
//
// It reads every cached key and value once and does 4*d flops per key and
// query head, so it is bound by HBM bandwidth: CUDA cores, no tensor cores.
// Split over the keys: CTA (b, kv head j, chunk c) takes CH = 128 keys, stages
// the chunk's V in shared memory with coalesced read-only loads, and one
// thread per key reads the key row, rotates it at its position pair by pair
// straight into its scores against the G query heads of the group (rotated
// once per CTA at Tk - 1); then one partial (max, sum, O) per head.  Small
// enough (64 registers, 19 KB at d = 64) for eight CTAs per SM, so a layer's
// chunks run in one wave.  A second kernel merges the partials of
// each (b, h) in chunk order: deterministic, no atomics.
#include <cuda_bf16.h>

#include "ne_common.cuh"
#include "ne_kernels.h"

namespace ne {

constexpr int kDecCh = 128;        // keys per CTA (one per thread)
constexpr int kDecThreads = 128;

template <int D>
struct DecCfg {
    static constexpr int OFF_V = 0;                                   // bf16 [CH][D]
    static constexpr int OFF_Q = OFF_V + kDecCh * D * 2;              // float [G][D]
    static __host__ __device__ constexpr int off_p(int G) { return OFF_Q + G * D * 4; }  // float [G][CH]
    static __host__ __device__ constexpr int off_ml(int G) { return off_p(G) + G * kDecCh * 4; }
    static __host__ __device__ constexpr int bytes(int G) { return off_ml(G) + 2 * G * 4; }
};

// GB = the group size G rounded up to a power of two (the kernel keeps GB
// score accumulators per thread; heads g >= G are skipped).
template <int D, int GB>
__global__ void __launch_bounds__(kDecThreads, 8)
    decode_partial_kernel(const DecodeParams p)
{
    using C = DecCfg<D>;
    constexpr int CPR = D / 8;     // 16-byte chunks per row
    constexpr int HC = D / 16;     // chunks in the first half of a row
    extern __shared__ __align__(16) uint8_t smem[];
    __nv_bfloat16 *vs = reinterpret_cast<__nv_bfloat16 *>(smem + C::OFF_V);
    float *qs = reinterpret_cast<float *>(smem + C::OFF_Q);
    float *ps = reinterpret_cast<float *>(smem + C::off_p(p.G));
    float *ml = reinterpret_cast<float *>(smem + C::off_ml(p.G));

    const int t = threadIdx.x, lane = t % 32, warp = t / 32;
    const int c = blockIdx.x % p.nchunks;
    const int j = (blockIdx.x / p.nchunks) % p.Hkv;
    const int b = blockIdx.x / (p.nchunks * p.Hkv);
    const int s0 = c * kDecCh;
    const int G = p.G;
    griddep_wait();

    // V rows s0 .. s0+127 of (b, j) into shared memory (coalesced 16-byte
    // loads, zero past Tk)
    const uint4 *kg = static_cast<const uint4 *>(p.k);
    const uint4 *vg = static_cast<const uint4 *>(p.v);
    for (int idx = t; idx < kDecCh * CPR; idx += kDecThreads) {
        const int r = idx / CPR, cc = idx % CPR, s = s0 + r;
        uint4 vv = make_uint4(0u, 0u, 0u, 0u);
        if (s < p.Tk)
            vv = ld_stream(vg + ((static_cast<size_t>(b) * p.Tk + s) * p.Hkv + j) * CPR + cc);
        *reinterpret_cast<uint4 *>(vs + r * D + cc * 8) = vv;
    }
    // the group's G query rows, rotated at position Tk - 1, in fp32
    const uint32_t qpos = static_cast<uint32_t>(p.Tk - 1);
    const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
    for (int idx = t; idx < G * (D / 2); idx += kDecThreads) {
        const int g = idx / (D / 2), i = idx % (D / 2);
        const __nv_bfloat16 *qrow = qg + (static_cast<size_t>(b) * p.Hq + j * G + g) * D;
        float sn, cs;
        rope_sincos(qpos, p.rope, i, sn, cs);
        const float x = __bfloat162float(qrow[i]), y = __bfloat162float(qrow[i + D / 2]);
        qs[g * D + i] = x * cs - y * sn;
        qs[g * D + i + D / 2] = y * cs + x * sn;
    }
    __syncthreads();

    // one key per thread, read from global memory in rotate-half chunk pairs
    // (c, c + D/16) and rotated pair by pair straight into the G scores
    {
        const int s = s0 + t;
        float acc[GB];
#pragma unroll
        for (int g = 0; g < GB; ++g)
            acc[g] = 0.f;
        if (s < p.Tk) {
            const uint4 *krow = kg + ((static_cast<size_t>(b) * p.Tk + s) * p.Hkv + j) * CPR;
#pragma unroll
            for (int cc = 0; cc < HC; ++cc) {
                const uint4 a4 = krow[cc], b4 = krow[cc + HC];
                const uint32_t av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = 8 * cc + e;
                    float sn, cs;
                    rope_sincos(static_cast<uint32_t>(s), p.rope, i, sn, cs);
                    const float x = (e & 1) ? bf16_hi(av[e >> 1]) : bf16_lo(av[e >> 1]);
                    const float y = (e & 1) ? bf16_hi(bv[e >> 1]) : bf16_lo(bv[e >> 1]);
                    const float xr = x * cs - y * sn, yr = y * cs + x * sn;
#pragma unroll
                    for (int g = 0; g < GB; ++g)
                        if (g < G)
                            acc[g] = fmaf(qs[g * D + i + D / 2], yr, fmaf(qs[g * D + i], xr, acc[g]));
                }
            }
        }
#pragma unroll
        for (int g = 0; g < GB; ++g)
            if (g < G)
                ps[g * kDecCh + t] = s < p.Tk ? acc[g] * p.scale_log2 : -INFINITY;
    }
    __syncthreads();

    // per head: the chunk's max m, P = 2^(S - m) and its sum l (warp w takes
    // heads w, w + 4, ...; every chunk has at least one key, so m is finite)
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

    // O_g[e..e+1] = sum_r P_g[r] v[r][e..e+1] (column pairs); partials to the
    // workspace
    const size_t part0 = (static_cast<size_t>(b) * p.Hq + j * G) * p.nchunks + c;
    for (int o = t; o < G * (D / 2); o += kDecThreads) {
        const int g = o / (D / 2), e = 2 * (o % (D / 2));
        const float *prow = ps + g * kDecCh;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
        for (int r = 0; r < kDecCh; ++r) {
            const uint32_t v2 = *reinterpret_cast<const uint32_t *>(vs + r * D + e);
            const float pr = prow[r];
            a0 = fmaf(pr, bf16_lo(v2), a0);
            a1 = fmaf(pr, bf16_hi(v2), a1);
        }
        float *dst = p.part_o + (part0 + static_cast<size_t>(g) * p.nchunks) * D + e;
        *reinterpret_cast<float2 *>(dst) = make_float2(a0, a1);
    }
    if (t < G) {
        const size_t pi = part0 + static_cast<size_t>(t) * p.nchunks;
        p.part_ml[2 * pi] = ml[2 * t];
        p.part_ml[2 * pi + 1] = ml[2 * t + 1];
    }
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
static cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t stream)
{
    const int smem = DecCfg<D>::bytes(p.G);
    auto kern = decode_partial_kernel<D, GB>;
    static bool attr_done[64] = {};   // one flag set per template instantiation
    cudaError_t e = ensure_smem_attr(kern, DecCfg<D>::bytes(kMaxDecodeGroup), attr_done);
    if (e != cudaSuccess)
        return e;
    const unsigned nb = static_cast<unsigned>(p.B * p.Hkv * p.nchunks);
    if ((e = launch_pdl(kern, nb, kDecThreads, smem, stream, p)) != cudaSuccess)
        return e;
    return launch_pdl(decode_combine_kernel<D>, static_cast<unsigned>(p.B * p.Hq), D, 0, stream,
                      p);
}

template <int D>
static cudaError_t launch_decode_d(const DecodeParams &p, cudaStream_t stream)
{
    if (p.G <= 1)
        return launch_decode_t<D, 1>(p, stream);
    if (p.G <= 2)
        return launch_decode_t<D, 2>(p, stream);
    if (p.G <= 4)
        return launch_decode_t<D, 4>(p, stream);
    if (p.G <= 8)
        return launch_decode_t<D, 8>(p, stream);
    return launch_decode_t<D, 16>(p, stream);
}

cudaError_t launch_decode(int d, const DecodeParams &p, cudaStream_t stream)
{
    switch (d) {
    case 32: return launch_decode_d<32>(p, stream);
    case 64: return launch_decode_d<64>(p, stream);
    case 128: return launch_decode_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace ne
