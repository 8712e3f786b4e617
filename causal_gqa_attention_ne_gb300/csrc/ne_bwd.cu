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

// Partial sum of dO * O over one 16-byte chunk (8 elements) in a fixed
// order.  D of a row is then the chunks' partials added pairwise by a
// butterfly: chunk c with chunk c + D/16 first (one thread of bwd_pre_kernel,
// or two lanes of bwd_d_kernel), then the shuffle levels; both kernels use
// this order, so the standalone backward and the training pair get the same
// D bit for bit.
__device__ __forceinline__ float d_chunk(const uint4 &o4, const uint4 &g4)
{
    const uint32_t oa[4] = {o4.x, o4.y, o4.z, o4.w};
    const uint32_t ga[4] = {g4.x, g4.y, g4.z, g4.w};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e)
        acc = __fmaf_rn(bf16_hi(oa[e]), bf16_hi(ga[e]), __fmaf_rn(bf16_lo(oa[e]), bf16_lo(ga[e]), acc));
    return acc;
}

// Position of row bt = b*T + t of the [B][T] row space, and whether it is a
// valid row: plain batches, t; padded variable-length batches, t, valid if
// t < seqlen[b]; packed batches (B = 1, cu set), the row's offset in its
// sequence (cu[i] <= bt < cu[i+1], found by binary search; every row is in
// one).
struct RowPos {
    uint32_t pos;
    bool valid;
};
__device__ __forceinline__ RowPos row_pos(const AttnParams &p, size_t bt)
{
    if (p.cu != nullptr) {
        int lo = 0, hi = p.nseq;   // cu[lo] <= bt < cu[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (static_cast<size_t>(__ldg(p.cu + mid)) <= bt)
                lo = mid;
            else
                hi = mid;
        }
        return RowPos{static_cast<uint32_t>(bt - static_cast<size_t>(__ldg(p.cu + lo))), true};
    }
    const int t = static_cast<int>(bt % p.T);
    if (p.seqlen != nullptr)
        return RowPos{static_cast<uint32_t>(t), t < __ldg(p.seqlen + bt / p.T)};
    return RowPos{static_cast<uint32_t>(t), true};
}

// One pass over the query-side rows (b, t, h), one thread per pair of
// 16-byte chunks (c, c + D/16) of a row, so the thread holds rotate-half
// partners:
//   D[b][h][t] = sum_c dO[b,t,h,c] * O[b,t,h,c]       (fp32; the D/16
//                threads of a row reduce with shuffles)
//   Q'[b,t,h,:] = R(t) q[b,t,h,:] as fp16              (the score-side operands
//   K'[b,s,j,:] = R(s) k[b,s,j,:] as fp16               of the backward, rotated
//                once here instead of once per tile inside the loops)
// Pure streaming over O, dO, q and k.  With qrot == nullptr (Q' and K' already
// in the workspace, stored by the forward's training path) only D is computed.
// Rows past a padded sequence's length are not read: their D is never used
// (the kernels give such rows lse = +inf and D = 0) and their Q', K' rows are
// written as zeros, so the tiles that straddle a sequence's end stay finite.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const AttnParams p, const uint4 *q,
                                                      uint4 *qrot, const uint4 *k, uint4 *krot)
{
    constexpr int TPR = D / 16;          // threads per row
    constexpr int CPR = D / 8;           // 16-byte chunks per row
    const size_t nrows = static_cast<size_t>(p.B) * p.T * p.Hq;
    const size_t nthreads = nrows * TPR;
    const uint4 *o = static_cast<const uint4 *>(p.o_in);
    const uint4 *g = static_cast<const uint4 *>(p.do_in);
    // programmatic dependent launch: O comes from the previous grid
    griddep_wait();
    float mx = 0.f;
    for (size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         idx - (threadIdx.x % 32) < nthreads;   // whole warps stay in the loop for the shuffles
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float acc = 0.f;
        const size_t row = idx / TPR;                // ((b*T + t)*Hq + h)
        const int c = static_cast<int>(idx % TPR);
        const RowPos rp = idx < nthreads ? row_pos(p, row / p.Hq) : RowPos{0u, false};
        if (rp.valid) {
            const size_t c0 = row * CPR + c, c1 = c0 + TPR;
            // chunks c and c + D/16: each chunk's partial sum, then the pair
            // (the same order as bwd_d_kernel, so both give the same bits)
            acc = d_chunk(o[c0], g[c0]) + d_chunk(o[c1], g[c1]);
        }
        if (idx < nthreads && qrot != nullptr) {
            const size_t c0 = row * CPR + c, c1 = c0 + TPR;
            const uint4 qa = rp.valid ? q[c0] : make_uint4(0u, 0u, 0u, 0u);
            const uint4 qb = rp.valid ? q[c1] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t qav[4] = {qa.x, qa.y, qa.z, qa.w}, qbv[4] = {qb.x, qb.y, qb.z, qb.w};
            const uint32_t t = rp.pos;
            uint32_t ra[4], rb[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float u[2], w[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float sn, cs;
                    rope_sincos(t, p.rope, 8 * c + 2 * e + hh, sn, cs);
                    const float x = hh ? bf16_hi(qav[e]) : bf16_lo(qav[e]);
                    const float y = hh ? bf16_hi(qbv[e]) : bf16_lo(qbv[e]);
                    rope_rotate(x, y, cs, sn, u[hh], w[hh]);
                    mx = fmaxf(mx, fmaxf(fabsf(u[hh]), fabsf(w[hh])));
                }
                ra[e] = pack_f16x2(u[0], u[1]);
                rb[e] = pack_f16x2(w[0], w[1]);
            }
            qrot[c0] = make_uint4(ra[0], ra[1], ra[2], ra[3]);
            qrot[c1] = make_uint4(rb[0], rb[1], rb[2], rb[3]);
        }
#pragma unroll
        for (int off = TPR / 2; off >= 1; off /= 2)
            acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (rp.valid && c == 0) {
            const int h = static_cast<int>(row % p.Hq);
            const size_t bt = row / p.Hq;
            const int t = static_cast<int>(bt % p.T);
            const int b = static_cast<int>(bt / p.T);
            p.Dws[(static_cast<size_t>(b) * p.Hq + h) * p.T + t] = acc;
        }
    }
    // K' = R(s) k as fp16, same layout as k.
    const size_t krows = qrot != nullptr ? static_cast<size_t>(p.B) * p.T * p.Hkv : 0;
    for (size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         idx < krows * TPR; idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t row = idx / TPR;                // ((b*T + s)*Hkv + j)
        const int c = static_cast<int>(idx % TPR);
        const size_t c0 = row * CPR + c, c1 = c0 + TPR;
        const RowPos rp = row_pos(p, row / p.Hkv);
        const uint4 ka = rp.valid ? k[c0] : make_uint4(0u, 0u, 0u, 0u);
        const uint4 kb = rp.valid ? k[c1] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t kav[4] = {ka.x, ka.y, ka.z, ka.w}, kbv[4] = {kb.x, kb.y, kb.z, kb.w};
        const uint32_t pos = rp.pos;
        uint32_t ra[4], rb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float u[2], w[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float sn, cs;
                rope_sincos(pos, p.rope, 8 * c + 2 * e + hh, sn, cs);
                const float x = hh ? bf16_hi(kav[e]) : bf16_lo(kav[e]);
                const float y = hh ? bf16_hi(kbv[e]) : bf16_lo(kbv[e]);
                rope_rotate(x, y, cs, sn, u[hh], w[hh]);
                mx = fmaxf(mx, fmaxf(fabsf(u[hh]), fabsf(w[hh])));
            }
            ra[e] = pack_f16x2(u[0], u[1]);
            rb[e] = pack_f16x2(w[0], w[1]);
        }
        krot[c0] = make_uint4(ra[0], ra[1], ra[2], ra[3]);
        krot[c1] = make_uint4(rb[0], rb[1], rb[2], rb[3]);
    }
    if (mx > kFp16Max)
        atomicOr(p.status, kDevRange);
    griddep_launch_dependents();
}

// D alone (Q' and K' already in the workspace): a pure streaming pass over O
// and dO.  A row of D/8 16-byte chunks is read by D/8 consecutive lanes, so
// one warp-wide load covers 32 / (D/8) whole rows; RU such loads of O and of
// dO are in flight per lane before the row sums are reduced with shuffles.
// Persistent: four CTAs per SM (the register budget of RU loads in flight),
// all resident at once, striding over the rows.  (Two rounds in flight per
// warp, or bulk asynchronous copies into shared memory, measured slower.)
constexpr int kDCtasPerSm = 4;
template <int D>
__global__ void __launch_bounds__(256, kDCtasPerSm) bwd_d_kernel(const AttnParams p)
{
    constexpr int LPR = D / 8;                 // lanes per row (one 16-byte chunk each)
    constexpr int RPW = 32 / LPR;              // rows per warp-wide load
    constexpr int RU = 4;                      // loads of each tensor in flight per lane
    const size_t nrows = static_cast<size_t>(p.B) * p.T * p.Hq;
    const uint4 *o = static_cast<const uint4 *>(p.o_in);
    const uint4 *g = static_cast<const uint4 *>(p.do_in);
    const int lane = threadIdx.x % 32;
    const size_t warp = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const size_t nwarps = static_cast<size_t>(gridDim.x) * blockDim.x / 32;
    const bool small = nrows <= 0xFFFFFFFFull;
    const uint32_t hq32 = static_cast<uint32_t>(p.Hq), t32 = static_cast<uint32_t>(p.T);
    griddep_wait();   // O comes from the previous grid
    for (size_t r0 = warp * RPW * RU; r0 < nrows; r0 += nwarps * RPW * RU) {
        uint4 ov[RU], gv[RU];
#pragma unroll
        for (int i = 0; i < RU; ++i) {
            const size_t row = r0 + i * RPW + lane / LPR;
            if (row < nrows) {
                const size_t c = row * LPR + lane % LPR;
                ov[i] = ld_stream(o + c);
                gv[i] = ld_stream(g + c);
            } else {
                ov[i] = make_uint4(0u, 0u, 0u, 0u);
                gv[i] = ov[i];
            }
        }
#pragma unroll
        for (int i = 0; i < RU; ++i) {
            float acc = d_chunk(ov[i], gv[i]);
#pragma unroll
            for (int off = LPR / 2; off >= 1; off /= 2)
                acc += __shfl_xor_sync(0xffffffffu, acc, off);
            const size_t row = r0 + i * RPW + lane / LPR;   // ((b*T + t)*Hq + h)
            if (lane % LPR == 0 && row < nrows) {
                size_t h, t, b;
                if (small) {   // 32-bit division where the row count allows it
                    const uint32_t r32 = static_cast<uint32_t>(row);
                    const uint32_t bt32 = r32 / hq32;
                    const uint32_t b32 = bt32 / t32;
                    h = r32 - bt32 * hq32;
                    t = bt32 - b32 * t32;
                    b = b32;
                } else {
                    h = row % p.Hq;
                    const size_t bt = row / p.Hq;
                    t = bt % p.T;
                    b = bt / p.T;
                }
                p.Dws[(b * p.Hq + h) * p.T + t] = acc;
            }
        }
    }
    griddep_launch_dependents();
}

cudaError_t launch_bwd_pre(int d, const AttnParams &p, const void *q, void *qrot, const void *k,
                           void *krot, cudaStream_t stream)
{
    if (qrot == nullptr) {
        int dev = 0, sms = 0;
        cudaError_t e;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return e;
        const unsigned nb = static_cast<unsigned>(sms * kDCtasPerSm);
        switch (d) {
        case 32: return launch_pdl(bwd_d_kernel<32>, nb, 256, 0, stream, p);
        case 64: return launch_pdl(bwd_d_kernel<64>, nb, 256, 0, stream, p);
        case 128: return launch_pdl(bwd_d_kernel<128>, nb, 256, 0, stream, p);
        default: return cudaErrorInvalidValue;
        }
    }
    const size_t nthreads = static_cast<size_t>(p.B) * p.T * p.Hq * (d / 16);
    size_t blocks = (nthreads + 255) / 256;
    // With the rotations, a grid-stride loop over a capped grid (the K'
    // rows are covered by the same threads); D alone is one row chunk per
    // thread, so the whole grid streams without a loop.
    const size_t cap = qrot != nullptr ? 152 * 16 : 152 * 256;
    if (blocks > cap)
        blocks = cap;
    const uint4 *qi = static_cast<const uint4 *>(q), *ki = static_cast<const uint4 *>(k);
    uint4 *qo = static_cast<uint4 *>(qrot), *ko = static_cast<uint4 *>(krot);
    const unsigned nb = static_cast<unsigned>(blocks);
    switch (d) {
    case 32: return launch_pdl(bwd_pre_kernel<32>, nb, 256, 0, stream, p, qi, qo, ki, ko);
    case 64: return launch_pdl(bwd_pre_kernel<64>, nb, 256, 0, stream, p, qi, qo, ki, ko);
    case 128: return launch_pdl(bwd_pre_kernel<128>, nb, 256, 0, stream, p, qi, qo, ki, ko);
    default: return cudaErrorInvalidValue;
    }
}

// The same for a D <= 64 tile leaving through shared memory: the row is
// written as bf16 into this thread's row r of a 128-byte or 64-byte swizzled
// staging block (the layout the TMA store of the output tensor reads).
template <int D>
__device__ __forceinline__ void epilogue_inverse_rope_stage(uint32_t taddr, float scale,
                                                            const float (&sn)[D / 2],
                                                            const float (&cs)[D / 2],
                                                            uint8_t *stage, int r)
{
    static_assert(D <= 64, "one column block");
    uint32_t a[32];
    float x[D];
    tmem_ld32(taddr, a);
    if constexpr (D == 64) {
        uint32_t b[32];
        tmem_ld32(taddr + 32, b);
        tmem_ld_wait(a);
        tmem_tie(b);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(a[e]) * scale;
            x[e + 32] = __uint_as_float(b[e]) * scale;
        }
    } else {
        tmem_ld_wait(a);
#pragma unroll
        for (int e = 0; e < 32; ++e)
            x[e] = __uint_as_float(a[e]) * scale;
    }
    // rotation by -angle: (x, y) -> (x cos + y sin, y cos - x sin)
#pragma unroll
    for (int e = 0; e < D / 2; ++e) {
        const float u = x[e] * cs[e] + x[e + D / 2] * sn[e];
        const float w = x[e + D / 2] * cs[e] - x[e] * sn[e];
        x[e] = u;
        x[e + D / 2] = w;
    }
#pragma unroll
    for (int c = 0; c < D / 8; ++c)
        *reinterpret_cast<uint4 *>(stage + tile_chunk<D>(r, c)) =
            make_uint4(pack_bf16x2(x[8 * c + 0], x[8 * c + 1]), pack_bf16x2(x[8 * c + 2], x[8 * c + 3]),
                       pack_bf16x2(x[8 * c + 4], x[8 * c + 5]), pack_bf16x2(x[8 * c + 6], x[8 * c + 7]));
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
                rope_inverse_pair(x[e], y[e], pos, fr, c0 + e);
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
            rope_inverse_pair(x[e], x[e + 16], pos, fr, e);
        if (store)
            store_row32_bf16(dst, x);
    }
}

// ------------------------------------------------------------------ dQ ---
//
// Persistent: one CTA per SM walks a snake-ordered list of work units
// (b, kv head j, query tile m, chunk of GC query heads), heaviest (largest m)
// first.  Per unit the loop runs over the causal key tiles jk <= m and the GC
// heads ("items"); each K'/V tile is loaded once and used by the GC heads.
// Warp roles (384 threads):
//   warps 0-7   two row warpgroups; warpgroup w handles key columns
//               [64w, 64w+64) of every 128x128 tile: P = exp(S - lse),
//               dS = P (dP - D), dS (fp16) to TMEM as the A operand of
//               dQ += dS K'; at the end of a unit, dQ * scale with the inverse
//               RoPE to bf16 (warpgroup w takes heads g = w, w+2, ...).
//   warp 8      TMA producer.
//   warps 9, 11 S/dP issuers of row warpgroups 0 and 1 (each group's 64 key
//               columns are their own N = 64 MMAs with their own barriers, so
//               the groups never wait for each other); warp 9 also allocates
//               TMEM.
//   warp 10     dQ issuer (per item group 0's key K steps, then group 1's).
// TMEM: S [0,128) dP [128,256) dS [256,320) dQ of head g at 320 + g*D.

template <int D, int GC, int ST>
struct DqCfg {
    using TL = Tile<D>;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = OFF_Q + GC * TL::BYTES;
    static constexpr int OFF_K = OFF_DO + GC * TL::BYTES;
    static constexpr int OFF_V = OFF_K + ST * TL::BYTES;
    // d <= 64: dq leaves through one shared-memory staging block per row
    // warpgroup and a TMA store (a thread's own row would be 16-byte stores
    // Hq*d*2 bytes apart, 32 transactions per warp store)
    static constexpr bool STAGE = (D <= 64);
    static constexpr int OFF_STG = OFF_V + ST * TL::BYTES;
    static constexpr int SMEM_BYTES = smem_one_cta(OFF_STG + (STAGE ? 2 * TL::BLOCK : 0) + 1024);
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DS = 256, COL_DQ = 320;
    static_assert(!STAGE || TL::NB == 1, "staged epilogue stores one column block per head");
    static_assert(COL_DQ + GC * D <= 512, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct DqUnit {
    int m, b, j, h0, lo;   // lo: first key tile (sliding window; 0 otherwise)
    int tl;                // valid rows of sequence b (varlen; T otherwise)
    SeqLoc sq;             // where sequence b's rows live
};

// VAR: u indexes the launch's table of live units (padded variable-length
// batches), which holds indices into the full enumeration below.
template <bool VAR>
__device__ __forceinline__ DqUnit dq_unit(int u, int GC, const AttnParams &p)
{
    if constexpr (VAR)
        u = __ldg(p.units + u);
    DqUnit w;
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
    w.tl = w.sq.len;
    return w;
}

// WIN: a sliding window may mask keys off the diagonal tile.  VAR: padded
// variable-length batch; rows past their sequence's length get lse = +inf
// (P = 0, dS = 0), and their dq is overwritten afterwards by the padding fill.
template <int D, int GC, int ST, bool WIN, bool VAR>
__global__ void __launch_bounds__(384, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmDQ, const AttnParams p)
{
    using C = DqCfg<D, GC, ST>;
    using TL = Tile<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_q_full[GC], bar_q_empty[GC];
    __shared__ uint64_t bar_kv_full[ST], bar_kv_empty[ST];
    // per row warpgroup w: its key columns of S/dP computed (s_full), loaded
    // (s_empty), its dS written (ds_full) and read by the dQ MMAs (ds_empty)
    __shared__ uint64_t bar_s_full[2], bar_s_empty[2], bar_ds_full[2], bar_ds_empty[2];
    __shared__ uint64_t bar_dq_done, bar_dq_free, bar_drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ uint32_t abort_s;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cta = static_cast<int>(blockIdx.x), P = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        abort_s = 0;
        for (int g = 0; g < GC; ++g) {
            mbar_init(smem_u32(&bar_q_full[g]), 1);
            mbar_init(smem_u32(&bar_q_empty[g]), 2);   // both S/dP issuers
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&bar_kv_full[s]), 1);
            mbar_init(smem_u32(&bar_kv_empty[s]), 1);
        }
        for (int w2 = 0; w2 < 2; ++w2) {
            mbar_init(smem_u32(&bar_s_full[w2]), 1);
            mbar_init(smem_u32(&bar_s_empty[w2]), 4);
            mbar_init(smem_u32(&bar_ds_full[w2]), 4);
            mbar_init(smem_u32(&bar_ds_empty[w2]), 1);
        }
        mbar_init(smem_u32(&bar_dq_done), 1);
        mbar_init(smem_u32(&bar_dq_free), 8);
        mbar_init(smem_u32(&bar_drain), 3);
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
    // Only shared memory and TMEM were touched so far: from here on global
    // memory is read and written, so wait for the previous grid in the stream
    // (programmatic dependent launch).
    griddep_wait();
    const int NU = unit_total<VAR>(p);   // work units of the launch
    const WaitCtl wc{&abort_s, p.status, p.wait_limit_ns};
    auto teardown = [&]() {
        tc_fence_before();
        __syncthreads();
        griddep_launch_dependents();   // this CTA's work is done
        if (warp == 9) {
            tc_fence_after();
            tmem_dealloc(tbase, C::TMEM_COLS);
        }
    };

    // Register budgets after the split (launched with 168 per thread x 384):
    // rows 216 x 256 + the rest 64 x 128 <= 64512.
    if (warp >= 8) {
        regs_release<64>();
        if (warp == 8 && lane == 0) {
            // ------------------------------------------------ TMA producer ---
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmDO);
            bool ok = true;
            int kt = 0, k = 0;
            for (; ok; ++k) {
                const int u = snake_unit(k, cta, P);
                if (u >= NU)
                    break;
                const DqUnit w = dq_unit<VAR>(u, GC, p);
                auto load_kv = [&](int jk) {
                    const int st = kt % ST, u2 = kt / ST;
                    if (u2 >= 1 && !mbar_wait(smem_u32(&bar_kv_empty[st]), (u2 - 1) & 1, wc))
                        return false;
                    const uint32_t kb = smem_u32(&bar_kv_full[st]);
                    mbar_arrive_expect_tx(kb, 2 * TL::BYTES);
                    for (int cb = 0; cb < TL::NB; ++cb) {
                        tma_load_4d(smem_u32(smem + C::OFF_K + st * TL::BYTES + cb * TL::BLOCK),
                                    &tmK, kb, cb * TL::BOX_COLS, w.j, w.sq.base + jk * kRows,
                                    w.sq.bc);
                        tma_load_4d(smem_u32(smem + C::OFF_V + st * TL::BYTES + cb * TL::BLOCK),
                                    &tmV, kb, cb * TL::BOX_COLS, w.j, w.sq.base + jk * kRows,
                                    w.sq.bc);
                    }
                    ++kt;
                    return true;
                };
                // The unit's first K/V tile goes first: a stage is free while
                // the previous unit's last items run, but the Q'/dO slots only
                // free at those items, so the tile lands during them.
                ok = load_kv(w.lo);
                for (int g = 0; g < GC && ok; ++g) {
                    if (k >= 1 && !mbar_wait(smem_u32(&bar_q_empty[g]), (k - 1) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    const uint32_t qb = smem_u32(&bar_q_full[g]);
                    mbar_arrive_expect_tx(qb, 2 * TL::BYTES);
                    for (int cb = 0; cb < TL::NB; ++cb) {
                        tma_load_4d(smem_u32(smem + C::OFF_Q + g * TL::BYTES + cb * TL::BLOCK),
                                    &tmQ, qb, cb * TL::BOX_COLS, w.h0 + g,
                                    w.sq.base + w.m * kRows, w.sq.bc);
                        tma_load_4d(smem_u32(smem + C::OFF_DO + g * TL::BYTES + cb * TL::BLOCK),
                                    &tmDO, qb, cb * TL::BOX_COLS, w.h0 + g,
                                    w.sq.base + w.m * kRows, w.sq.bc);
                    }
                }
                for (int jk = w.lo + 1; jk <= w.m && ok; ++jk)
                    ok = load_kv(jk);
            }
            if (*wc.abort) {
                for (int g = 0; g < GC; ++g)
                    mbar_wait_drain(smem_u32(&bar_q_full[g]), (k > 0 ? k - 1 : 0) & 1, wc.limit_ns);
                for (int t = (kt > ST ? kt - ST : 0); t < kt; ++t)
                    mbar_wait_drain(smem_u32(&bar_kv_full[t % ST]), (t / ST) & 1, wc.limit_ns);
            }
        } else if (warp >= 9) {
            // -------------------------------------------------- MMA issuers ---
            // Row warpgroup w owns key columns [64w, 64w+64) of every item; its
            // S/dP columns are issued by their own warp (9 for w = 0, 11 for
            // w = 1) as soon as that group has loaded its previous ones.  Warp
            // 10 issues dQ += dS K': per item the K steps of group 0's keys,
            // then group 1's, always in that order (a fixed accumulation
            // order).
            constexpr uint32_t ID_S = idesc_f16(128, 64, false, false, false);
            constexpr uint32_t ID_DP = idesc_f16(128, 64, true, false, false);
            constexpr uint32_t ID_DQ = idesc_f16(128, TL::NPV, false, false, true);
            constexpr uint32_t TSTEP = TL::BYTES >> 4;
            constexpr uint32_t RHALF = (64 * TL::SWB) >> 4;   // rows 64.. of a K'/V tile
            const uint32_t sbase = __shfl_sync(0xffffffffu, smem_u32(smem), 0);
            const uint32_t tb = __shfl_sync(0xffffffffu, tbase, 0);
            bool ok = true;
            int gi = 0, kt = 0;
            if (warp != 10) {
                const int wg = warp == 9 ? 0 : 1;
                const uint64_t dQ0 = desc_kmajor_base<D>(sbase + C::OFF_Q);
                const uint64_t dO0 = desc_kmajor_base<D>(sbase + C::OFF_DO);
                const uint64_t dK0 = desc_kmajor_base<D>(sbase + C::OFF_K) + wg * RHALF;
                const uint64_t dV0 = desc_kmajor_base<D>(sbase + C::OFF_V) + wg * RHALF;
                const uint32_t col_s = tb + C::COL_S + 64 * wg, col_dp = tb + C::COL_DP + 64 * wg;
                for (int k = 0; ok; ++k) {
                    const int u = snake_unit(k, cta, P);
                    if (u >= NU)
                        break;
                    const DqUnit w = dq_unit<VAR>(u, GC, p);
                    const int nitems = (w.m - w.lo + 1) * GC;
                    for (int it = 0; it < nitems; ++it, ++gi) {
                        const int jk = w.lo + it / GC, g = it % GC;
                        const int st = kt % ST;
                        if ((g == 0 && !mbar_wait_warp(smem_u32(&bar_kv_full[st]), (kt / ST) & 1, wc)) ||
                            (jk == w.lo && !mbar_wait_warp(smem_u32(&bar_q_full[g]), k & 1, wc)) ||
                            (gi >= 1 &&
                             !mbar_wait_warp(smem_u32(&bar_s_empty[wg]), (gi - 1) & 1, wc))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t qd = dQ0 + g * TSTEP, od = dO0 + g * TSTEP;
                        const uint64_t kd = dK0 + st * TSTEP, vd = dV0 + st * TSTEP;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_f16_ss(col_s, qd + kmajor_off<D>(kk), kd + kmajor_off<D>(kk),
                                           ID_S, kk > 0 ? 1u : 0u);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_f16_ss(col_dp, od + kmajor_off<D>(kk), vd + kmajor_off<D>(kk),
                                           ID_DP, kk > 0 ? 1u : 0u);
                            mma_commit(smem_u32(&bar_s_full[wg]));
                            if (jk == w.m)   // last use of head g's Q'/dO in this unit
                                mma_commit(smem_u32(&bar_q_empty[g]));
                        }
                        __syncwarp();
                        if (g == GC - 1)
                            ++kt;
                    }
                }
            } else {
                const uint64_t dKm0 = desc_mnmajor_base<D>(sbase + C::OFF_K);
                for (int k = 0; ok; ++k) {
                    const int u = snake_unit(k, cta, P);
                    if (u >= NU)
                        break;
                    const DqUnit w = dq_unit<VAR>(u, GC, p);
                    const int nitems = (w.m - w.lo + 1) * GC;
                    for (int it = 0; it < nitems && ok; ++it, ++gi) {
                        const int jk = w.lo + it / GC, g = it % GC;
                        const int st = kt % ST;
                        const uint64_t km = dKm0 + st * TSTEP;
                        for (int wg = 0; wg < 2; ++wg) {
                            if (!mbar_wait_warp(smem_u32(&bar_ds_full[wg]), gi & 1, wc) ||
                                (it == 0 && wg == 0 && k >= 1 &&
                                 !mbar_wait_warp(smem_u32(&bar_dq_free), (k - 1) & 1, wc))) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t first = (jk > w.lo || wg > 0) ? 1u : 0u;
                            if (elect_one()) {
#pragma unroll
                                for (int nc = 0; nc < D / TL::NPV; ++nc)
#pragma unroll
                                    for (int kq = 0; kq < 4; ++kq)
                                        mma_f16_ts(tb + C::COL_DQ + g * D + nc * TL::NPV,
                                                   tb + C::COL_DS + 32 * wg + 8 * kq,
                                                   km + mnmajor_off<D>(nc, 4 * wg + kq), ID_DQ,
                                                   kq > 0 ? 1u : first);
                                mma_commit(smem_u32(&bar_ds_empty[wg]));
                                if (wg == 1) {
                                    if (g == GC - 1)
                                        mma_commit(smem_u32(&bar_kv_empty[st]));
                                    if (it == nitems - 1)
                                        mma_commit(smem_u32(&bar_dq_done));
                                }
                            }
                            __syncwarp();
                        }
                        if (g == GC - 1)
                            ++kt;
                    }
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

    // ---------------------------------------------------- row warpgroups ---
    regs_claim<216>();
    const int w = warp >> 2;                // key-column half of the score tile
    static_assert(kDqStoreRows == 32, "a warp stores the rows of its TMEM lane quarter");
    const int r = threadIdx.x & 127;        // query row == TMEM lane
    const uint32_t lane_base = tmem_addr(tbase, (warp & 3) * 32, 0);
    float maxds = 0.f;
    bool ok = true;
    int gi = 0;
    float nl2[GC], nD[GC];
    auto fetch = [&](int k, float (&l2)[GC], float (&dd)[GC]) {
        const int u = snake_unit(k, cta, P);
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            l2[g] = 0.f;
            dd[g] = 0.f;
        }
        if (u >= NU)
            return;
        const DqUnit un = dq_unit<VAR>(u, GC, p);
        const int t = un.m * kRows + r;
        if (t < un.tl) {
#pragma unroll
            for (int g = 0; g < GC; ++g) {
                const size_t idx =
                    (static_cast<size_t>(un.sq.bc) * p.Hq + un.h0 + g) * p.T + un.sq.base + t;
                l2[g] = p.lse[idx] * kLog2e;
                dd[g] = p.Dws[idx];
            }
        } else if constexpr (VAR) {
#pragma unroll
            for (int g = 0; g < GC; ++g)
                l2[g] = INFINITY;
        }
    };
    // A unit's epilogue (dq out of TMEM) runs after the next unit's first
    // item has been handed to the dQ issuer: the wait for the unit's last dQ
    // MMA then overlaps that item's softmax work, and the next unit's first
    // dQ MMA waits for dq_free anyway.
    int pend_k = -1;
    DqUnit pend{};
    uint8_t *stage = smem + C::OFF_STG + w * TL::BLOCK;   // this warpgroup's staging block
    uint32_t nepi = 0;                                   // dq tiles this warpgroup has stored
    auto epilogue = [&]() {
        if (!mbar_wait_warp(smem_u32(&bar_dq_done), pend_k & 1, wc))
            return false;
        tc_fence_after();
        const int t = pend.m * kRows + r;
        __nv_bfloat16 *dq = static_cast<__nv_bfloat16 *>(p.out0);
        // the row's sines and cosines, shared by the warpgroup's heads
        float sn[D <= 64 ? D / 2 : 1], cs[D <= 64 ? D / 2 : 1];
        if constexpr (C::STAGE) {
#pragma unroll
            for (int e = 0; e < D / 2; ++e)
                rope_sincos(static_cast<uint32_t>(t), p.rope, e, sn[e], cs[e]);
        }
        // the last tile of a packed sequence goes out row by row: a tile
        // store would overwrite the next sequence's first rows
        const bool direct = VAR && p.cu != nullptr && (pend.m + 1) * kRows > pend.tl;
        auto store_direct = [&](int g) {
            __nv_bfloat16 *row = dq + (seq_row(p, pend.sq, t) * p.Hq + pend.h0 + g) * D;
            epilogue_inverse_rope<D>(lane_base + C::COL_DQ + g * D, p.scale,
                                     static_cast<uint32_t>(t), p.rope, row, t < pend.tl);
        };
#pragma unroll
        for (int g = 0; g < GC; ++g)
            if ((g & 1) == w) {
                if constexpr (C::STAGE) {
                    if (direct) {
                        store_direct(g);
                        continue;
                    }
                    // Each warp sends its own 32 rows out with its own TMA
                    // store (the dq map's box is kDqStoreRows rows); its rows
                    // of the staging block are free once the warp's previous
                    // store has read them.
                    if (nepi >= 1) {
                        if (lane == 0)
                            bulk_wait_read0();
                        __syncwarp();
                    }
                    epilogue_inverse_rope_stage<D>(lane_base + C::COL_DQ + g * D, p.scale, sn, cs,
                                                   stage, r);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_4d(&tmDQ, smem_u32(stage + (warp & 3) * kDqStoreRows * TL::SWB),
                                     0, pend.h0 + g,
                                     pend.sq.base + pend.m * kRows + (warp & 3) * kDqStoreRows,
                                     pend.sq.bc);
                        bulk_commit();
                    }
                    __syncwarp();
                    ++nepi;
                } else {
                    store_direct(g);
                }
            }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&bar_dq_free));
        pend_k = -1;
        return true;
    };
    fetch(0, nl2, nD);
    for (int k = 0; ok; ++k) {
        const int u = snake_unit(k, cta, P);
        if (u >= NU)
            break;
        const DqUnit un = dq_unit<VAR>(u, GC, p);
        float l2[GC], dd[GC];
#pragma unroll
        for (int g = 0; g < GC; ++g) {
            l2[g] = nl2[g];
            dd[g] = nD[g];
        }
        fetch(k + 1, nl2, nD);              // next unit's row scalars, in flight meanwhile
        const int nitems = (un.m - un.lo + 1) * GC;
        for (int it = 0; it < nitems; ++it, ++gi) {
            const int jk = un.lo + it / GC, g = it % GC;
            if (!mbar_wait_warp(smem_u32(&bar_s_full[w]), gi & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[2][32], pv[2][32];
            tmem_ld32(lane_base + C::COL_S + 64 * w, sv[0]);
            tmem_ld32(lane_base + C::COL_S + 64 * w + 32, sv[1]);
            tmem_ld32(lane_base + C::COL_DP + 64 * w, pv[0]);
            tmem_ld32(lane_base + C::COL_DP + 64 * w + 32, pv[1]);
            tmem_ld_wait_only();
            tmem_tie(sv[0]);
            tmem_tie(sv[1]);
            tmem_tie(pv[0]);
            tmem_tie(pv[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_s_empty[w]));

            // the per-head row scalars, selected without dynamic indexing
            float lg = l2[0], dg = dd[0];
#pragma unroll
            for (int q = 1; q < GC; ++q)
                if (g == q) {
                    lg = l2[q];
                    dg = dd[q];
                }
            const float sl2 = p.scale_log2;
            uint32_t dk[32];
            // sliding window: key columns c <= wlim (key <= row - W) are masked
            int wlim = -1;
            if constexpr (WIN)
                wlim = un.m * kRows + r - p.window - jk * kRows;
            if (jk != un.m && !(WIN && __any_sync(0xffffffffu, wlim >= 0))) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float p0 = ex2_approx(fmaf(__uint_as_float(sv[h][e]), sl2, -lg));
                        const float p1 = ex2_approx(fmaf(__uint_as_float(sv[h][e + 1]), sl2, -lg));
                        const float d0 = p0 * (__uint_as_float(pv[h][e]) - dg);
                        const float d1 = p1 * (__uint_as_float(pv[h][e + 1]) - dg);
                        maxds = fmaxf(maxds, fmaxf(fabsf(d0), fabsf(d1)));
                        dk[16 * h + e / 2] = pack_f16x2(d0, d1);
                    }
            } else {
                // diagonal tile: key column c > query row r is masked; window:
                // columns c <= wlim
                const int clim = (!WIN || jk == un.m) ? r : 1 << 30;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const int c = 64 * w + 32 * h + e;
                        float p0 = ex2_approx(fmaf(__uint_as_float(sv[h][e]), sl2, -lg));
                        float p1 = ex2_approx(fmaf(__uint_as_float(sv[h][e + 1]), sl2, -lg));
                        p0 = (c > clim || (WIN && c <= wlim)) ? 0.f : p0;
                        p1 = (c + 1 > clim || (WIN && c + 1 <= wlim)) ? 0.f : p1;
                        const float d0 = p0 * (__uint_as_float(pv[h][e]) - dg);
                        const float d1 = p1 * (__uint_as_float(pv[h][e + 1]) - dg);
                        maxds = fmaxf(maxds, fmaxf(fabsf(d0), fabsf(d1)));
                        dk[16 * h + e / 2] = pack_f16x2(d0, d1);
                    }
            }
            if (gi >= 1 && !mbar_wait_warp(smem_u32(&bar_ds_empty[w]), (gi - 1) & 1, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_st32(lane_base + C::COL_DS + 32 * w, dk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_ds_full[w]));
            if (it == 0 && pend_k >= 0 && !epilogue()) {
                ok = false;
                break;
            }
        }
        if (!ok)
            break;
        pend_k = k;          // dq = R(t)^T dQ' * scale of this unit: out at the next unit's first item
        pend = un;
    }
    if (ok && pend_k >= 0)
        ok = epilogue();
    if constexpr (C::STAGE) {
        if (lane == 0)
            bulk_wait0();   // this warp's dq rows have left shared memory
    }
    if (maxds > kFp16Max)
        atomicOr(p.status, kDevRange);
    teardown();
}

// ---------------------------------------------------------------- dK dV ---
//
// Persistent: one CTA per SM walks a snake-ordered list of work units
// (b, kv head j, key tile n), heaviest (n = 0) first.  Within a unit K' and
// V stay in shared memory and the loop runs over the G query heads of the
// group and the causal query tiles m >= n ("items").  Transposed scores: key
// row r lives in TMEM lane r.  K/V are double-buffered across units (D <= 64)
// so the next unit's tiles land and are rotated while the current one runs.
// Warp roles (512 threads):
//   warps 0-7   two "row" warpgroups; warpgroup w handles query columns
//               [64w, 64w+64) of every 128x128 tile of S^T and dP^T: reads them
//               from TMEM, computes P^T = exp(S^T - lse) and
//               dS^T = P^T (dP^T - D), writes both back to TMEM (bf16 / fp16)
//               where they are the A operands of dV += P^T dO and dK += dS^T Q';
//               at the end of a unit they store dV (warpgroup 0) and dK
//               (warpgroup 1, inverse RoPE).
//   warps 8-11  lse/D of each item's 128 queries into shared memory.  Q' and
//               K' arrive already rotated (fp16) from the preprocess pass,
//               through the workspace.
//   warp 12     TMA producer.      warp 13  TMEM allocator + S^T/dP^T issuer.
//   warp 14     dV/dK issuer.
// TMEM (D <= 64): S^T [0,128) dP^T [128,256) P^T [256,320) dS^T [320,384)
// dV [384, 384+D) dK [384+D, 384+2D).  D = 128: P^T / dS^T overwrite the
// half of S^T / dP^T each warpgroup has already read, dV [256,384),
// dK [384,512), and the items run in order (no overlap of item i's dV/dK
// with item i+1's scores).

template <int D, int ST>
struct DkvCfg {
    using TL = Tile<D>;
    static constexpr bool ALIAS = (D == 128);
    static constexpr int KB = (D == 128) ? 1 : 2;                    // K/V buffers
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = KB * TL::BYTES;
    static constexpr int OFF_Q = 2 * KB * TL::BYTES;
    static constexpr int OFF_DO = OFF_Q + ST * TL::BYTES;
    // float [ST][64 column pairs][-l2_c, -l2_c+1, -D_c, -D_c+1]
    static constexpr int OFF_LSED = OFF_DO + ST * TL::BYTES;
    static constexpr int SMEM_BYTES = smem_one_cta(OFF_LSED + ST * kRows * 8 + 1024);
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0, COL_DP = 128;
    static constexpr uint32_t COL_DV = ALIAS ? 256 : 384;
    static constexpr uint32_t COL_DK = COL_DV + D;
    static __host__ __device__ constexpr uint32_t col_p(int w) { return ALIAS ? 64 * w : 256 + 32 * w; }
    static __host__ __device__ constexpr uint32_t col_ds(int w) { return ALIAS ? 128 + 64 * w : 320 + 32 * w; }
    static_assert(COL_DK + D <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct DkvUnit {
    int n, b, j, nitems;
    int tl;                // valid rows of sequence b (varlen; T otherwise)
    SeqLoc sq;             // where sequence b's rows live
};

// VAR: u indexes the launch's table of live units (padded variable-length
// batches); a unit's query tiles then end at its sequence's last tile.
template <bool VAR>
__device__ __forceinline__ DkvUnit dkv_unit(int u, const AttnParams &p)
{
    if constexpr (VAR)
        u = __ldg(p.units + u);
    DkvUnit w;
    const int per_n = p.B * p.Hkv;
    w.n = u / per_n;
    const int rem = u % per_n;
    w.j = rem % p.Hkv;
    w.b = rem / p.Hkv;
    w.sq = seq_loc<VAR>(p, w.b);
    w.tl = w.sq.len;
    const int mtiles = VAR ? (w.tl + kRows - 1) / kRows : p.M;
    w.nitems = (query_tile_hi(w.n, p.window, mtiles) - w.n + 1) * p.G;
    return w;
}

// WIN: a sliding window may mask queries off the diagonal tile.  VAR: padded
// variable-length batch; query rows past their sequence's length get
// lse = +inf and D = 0 (P = 0, dS = 0), like rows past T, and the dk/dv rows
// of padding keys are overwritten afterwards by the padding fill.
template <int D, int ST, bool WIN, bool VAR>
__global__ void __launch_bounds__(512, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                const AttnParams p)
{
    using C = DkvCfg<D, ST>;
    using TL = Tile<D>;
    constexpr int KB = C::KB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_k_full[KB], bar_v_full[KB], bar_kv_empty[KB];
    __shared__ uint64_t bar_q_full[ST], bar_do_full[ST], bar_q_ready[ST], bar_st_empty[ST];
    __shared__ uint64_t bar_s_full, bar_s_empty, bar_pds_full, bar_pds_empty;
    __shared__ uint64_t bar_acc_done, bar_acc_free, bar_drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ uint32_t abort_s;
    float *lsed = reinterpret_cast<float *>(smem + C::OFF_LSED);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cta = static_cast<int>(blockIdx.x), P = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        abort_s = 0;
        for (int s = 0; s < KB; ++s) {
            mbar_init(smem_u32(&bar_k_full[s]), 1);
            mbar_init(smem_u32(&bar_v_full[s]), 1);
            mbar_init(smem_u32(&bar_kv_empty[s]), 1);
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&bar_q_full[s]), 1);
            mbar_init(smem_u32(&bar_do_full[s]), 1);
            mbar_init(smem_u32(&bar_q_ready[s]), 4);
            mbar_init(smem_u32(&bar_st_empty[s]), 1);
        }
        mbar_init(smem_u32(&bar_s_full), 1);
        mbar_init(smem_u32(&bar_s_empty), 8);
        mbar_init(smem_u32(&bar_pds_full), 8);
        mbar_init(smem_u32(&bar_pds_empty), 1);
        mbar_init(smem_u32(&bar_acc_done), 1);
        mbar_init(smem_u32(&bar_acc_free), 8);
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
    // Only shared memory and TMEM were touched so far: from here on global
    // memory is read and written, so wait for the previous grid in the stream
    // (programmatic dependent launch).
    griddep_wait();
    const int NU = unit_total<VAR>(p);   // work units of the launch
    const WaitCtl wc{&abort_s, p.status, p.wait_limit_ns};
    // Each role ends with its own copy of the teardown: warps run under
    // different register budgets after setmaxnreg, so their code paths never
    // re-join.
    auto teardown = [&]() {
        tc_fence_before();
        __syncthreads();
        griddep_launch_dependents();   // this CTA's work is done
        if (warp == 13) {
            tc_fence_after();
            tmem_dealloc(tbase, C::TMEM_COLS);
        }
    };

    // Register budgets after the split (launched with 128 per thread x 512,
    // four warps per sub-partition: 2 rows + lse/D + TMA/MMA <= 4 x 128):
    // d <= 64: rows 192 + 56 + 72 = 512 / 2; d = 128 (wider issue loops):
    // rows 184 + 56 + 80 = 504 / 2.
    constexpr int kRowRegs = D == 128 ? 184 : 192;
    if (warp >= 12) {
        if constexpr (D == 128)
            regs_release<80>();
        else
            regs_release<72>();
        if (warp == 12 && lane == 0) {
            // ------------------------------------------------ TMA producer ---
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmDO);
            bool ok = true;
            int gi = 0, k = 0;
            for (; ok; ++k) {
                const int u = snake_unit(k, cta, P);
                if (u >= NU)
                    break;
                const DkvUnit w = dkv_unit<VAR>(u, p);
                const int kb = k % KB, ku = k / KB;
                if (ku >= 1 && !mbar_wait(smem_u32(&bar_kv_empty[kb]), (ku - 1) & 1, wc)) {
                    ok = false;
                    break;
                }
                const uint32_t kbar = smem_u32(&bar_k_full[kb]), vbar = smem_u32(&bar_v_full[kb]);
                mbar_arrive_expect_tx(kbar, TL::BYTES);
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_K + kb * TL::BYTES + cb * TL::BLOCK), &tmK,
                                kbar, cb * TL::BOX_COLS, w.j, w.sq.base + w.n * kRows, w.sq.bc);
                mbar_arrive_expect_tx(vbar, TL::BYTES);
                for (int cb = 0; cb < TL::NB; ++cb)
                    tma_load_4d(smem_u32(smem + C::OFF_V + kb * TL::BYTES + cb * TL::BLOCK), &tmV,
                                vbar, cb * TL::BOX_COLS, w.j, w.sq.base + w.n * kRows, w.sq.bc);
                for (int it = 0; it < w.nitems; ++it, ++gi) {
                    const int st = gi % ST, su = gi / ST;
                    if (su >= 1 && !mbar_wait(smem_u32(&bar_st_empty[st]), (su - 1) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    const int mt = w.n + it / p.G, h = w.j * p.G + it % p.G;
                    const uint32_t qb = smem_u32(&bar_q_full[st]), db = smem_u32(&bar_do_full[st]);
                    mbar_arrive_expect_tx(qb, TL::BYTES);
                    for (int cb = 0; cb < TL::NB; ++cb)
                        tma_load_4d(smem_u32(smem + C::OFF_Q + st * TL::BYTES + cb * TL::BLOCK),
                                    &tmQ, qb, cb * TL::BOX_COLS, h, w.sq.base + mt * kRows,
                                    w.sq.bc);
                    mbar_arrive_expect_tx(db, TL::BYTES);
                    for (int cb = 0; cb < TL::NB; ++cb)
                        tma_load_4d(smem_u32(smem + C::OFF_DO + st * TL::BYTES + cb * TL::BLOCK),
                                    &tmDO, db, cb * TL::BOX_COLS, h, w.sq.base + mt * kRows,
                                    w.sq.bc);
                }
            }
            if (*wc.abort) {
                // Drain this CTA's own copies still in flight (each buffer's
                // latest load), bounded, before the CTA exits.
                for (int kk = (k > KB ? k - KB : 0); kk <= k && kk >= 0; ++kk) {
                    const int kb = kk % KB, ku = kk / KB;
                    mbar_wait_drain(smem_u32(&bar_k_full[kb]), ku & 1, wc.limit_ns);
                    mbar_wait_drain(smem_u32(&bar_v_full[kb]), ku & 1, wc.limit_ns);
                }
                for (int g = (gi > ST ? gi - ST : 0); g < gi; ++g) {
                    const int st = g % ST, su = g / ST;
                    mbar_wait_drain(smem_u32(&bar_q_full[st]), su & 1, wc.limit_ns);
                    mbar_wait_drain(smem_u32(&bar_do_full[st]), su & 1, wc.limit_ns);
                }
            }
        } else if (warp == 13 || warp == 14) {
            // -------------------------------------------------- MMA issuers ---
            // Two warps issue independently so neither stream blocks the other:
            // warp 13 issues S^T and dP^T as soon as an item's operands are in,
            // warp 14 issues dV/dK as soon as the rows have written P^T / dS^T.
            // Each warp runs its loop whole (warp-uniform descriptor math) and
            // one elected lane issues.  The releases of K/V and Q/dO buffers are
            // committed by warp 14 only: warp 13's MMAs on an item complete
            // before s_full, which precedes the rows' pds_full for that item.
            constexpr uint32_t ID_S = idesc_f16(128, 128, false, false, false);
            constexpr uint32_t ID_DP = idesc_f16(128, 128, true, false, false);
            constexpr uint32_t ID_DV = idesc_f16(128, TL::NPV, true, false, true);
            constexpr uint32_t ID_DK = idesc_f16(128, TL::NPV, false, false, true);
            constexpr uint32_t TSTEP = TL::BYTES >> 4;
            const uint32_t sbase = __shfl_sync(0xffffffffu, smem_u32(smem), 0);
            const uint32_t tb = __shfl_sync(0xffffffffu, tbase, 0);
            bool ok = true;
            int gi = 0;
            if (warp == 13) {
                const uint64_t dK0 = desc_kmajor_base<D>(sbase + C::OFF_K);
                const uint64_t dV0 = desc_kmajor_base<D>(sbase + C::OFF_V);
                const uint64_t dQk0 = desc_kmajor_base<D>(sbase + C::OFF_Q);
                const uint64_t dOk0 = desc_kmajor_base<D>(sbase + C::OFF_DO);
                const uint32_t b_s_full = smem_u32(&bar_s_full);
                const uint32_t b_s_empty = smem_u32(&bar_s_empty);
                const uint32_t b_pds_empty = smem_u32(&bar_pds_empty);
                for (int k = 0; ok; ++k) {
                    const int u = snake_unit(k, cta, P);
                    if (u >= NU)
                        break;
                    const DkvUnit w = dkv_unit<VAR>(u, p);
                    const int kb = k % KB, ku = k / KB;
                    if (!(mbar_wait_warp(smem_u32(&bar_k_full[kb]), ku & 1, wc) &&
                          mbar_wait_warp(smem_u32(&bar_v_full[kb]), ku & 1, wc))) {
                        ok = false;
                        break;
                    }
                    const uint64_t kd = dK0 + kb * TSTEP, vd = dV0 + kb * TSTEP;
                    for (int it = 0; it < w.nitems; ++it, ++gi) {
                        const int st = gi % ST, su = gi / ST;
                        if (!(mbar_wait_warp(smem_u32(&bar_q_ready[st]), su & 1, wc) &&
                              mbar_wait_warp(smem_u32(&bar_do_full[st]), su & 1, wc))) {
                            ok = false;
                            break;
                        }
                        if (gi >= 1 && !mbar_wait_warp(b_s_empty, (gi - 1) & 1, wc)) {
                            ok = false;
                            break;
                        }
                        // D = 128: P^T / dS^T live in S^T / dP^T's columns, so the
                        // previous item's dV/dK must be done before S^T is rewritten.
                        if (C::ALIAS && gi >= 1 &&
                            !mbar_wait_warp(b_pds_empty, (gi - 1) & 1, wc)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t qd = dQk0 + st * TSTEP, od = dOk0 + st * TSTEP;
                        if (elect_one()) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_f16_ss(tb + C::COL_S, kd + kmajor_off<D>(kk),
                                           qd + kmajor_off<D>(kk), ID_S, kk > 0 ? 1u : 0u);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_f16_ss(tb + C::COL_DP, vd + kmajor_off<D>(kk),
                                           od + kmajor_off<D>(kk), ID_DP, kk > 0 ? 1u : 0u);
                            mma_commit(b_s_full);
                        }
                        __syncwarp();
                    }
                }
            } else {
                const uint64_t dQm0 = desc_mnmajor_base<D>(sbase + C::OFF_Q);
                const uint64_t dOm0 = desc_mnmajor_base<D>(sbase + C::OFF_DO);
                const uint32_t b_pds_full = smem_u32(&bar_pds_full);
                const uint32_t b_pds_empty = smem_u32(&bar_pds_empty);
                for (int k = 0; ok; ++k) {
                    const int u = snake_unit(k, cta, P);
                    if (u >= NU)
                        break;
                    const DkvUnit w = dkv_unit<VAR>(u, p);
                    const int kb = k % KB;
                    for (int it = 0; it < w.nitems; ++it, ++gi) {
                        const int st = gi % ST;
                        if (!mbar_wait_warp(b_pds_full, gi & 1, wc) ||
                            (it == 0 && k >= 1 &&
                             !mbar_wait_warp(smem_u32(&bar_acc_free), (k - 1) & 1, wc))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t om = dOm0 + st * TSTEP, qm = dQm0 + st * TSTEP;
                        const uint32_t first = (it > 0) ? 1u : 0u;
                        if (elect_one()) {
#pragma unroll
                            for (int nc = 0; nc < D / TL::NPV; ++nc)
#pragma unroll
                                for (int kk = 0; kk < 8; ++kk)
                                    mma_f16_ts(tb + C::COL_DV + nc * TL::NPV,
                                               tb + C::col_p(kk >> 2) + 8 * (kk & 3),
                                               om + mnmajor_off<D>(nc, kk), ID_DV,
                                               kk > 0 ? 1u : first);
#pragma unroll
                            for (int nc = 0; nc < D / TL::NPV; ++nc)
#pragma unroll
                                for (int kk = 0; kk < 8; ++kk)
                                    mma_f16_ts(tb + C::COL_DK + nc * TL::NPV,
                                               tb + C::col_ds(kk >> 2) + 8 * (kk & 3),
                                               qm + mnmajor_off<D>(nc, kk), ID_DK,
                                               kk > 0 ? 1u : first);
                            mma_commit(b_pds_empty);
                            mma_commit(smem_u32(&bar_st_empty[st]));
                            if (it == w.nitems - 1) {
                                mma_commit(smem_u32(&bar_acc_done));
                                mma_commit(smem_u32(&bar_kv_empty[kb]));
                            }
                        }
                        __syncwarp();
                    }
                }
            }
            // Drain: each issuing warp's MMAs complete before TMEM is freed.
            if (elect_one())
                mma_commit(smem_u32(&bar_drain));
            __syncwarp();
            mbar_wait_warp(smem_u32(&bar_drain), 0, wc);
        }
        teardown();
        return;
    } else if (warp >= 8) {
        // ---------------------------------------- lse / D staging ---
        regs_release<56>();
        const int r = threadIdx.x - 256;
        bool ok = true;
        int gi = 0;
        float mx = 0.f;
        for (int k = 0; ok; ++k) {
            const int u = snake_unit(k, cta, P);
            if (u >= NU)
                break;
            const DkvUnit w = dkv_unit<VAR>(u, p);
            // lse and D of the item's queries are fetched one item ahead so the
            // global-load latency overlaps the wait for the previous item.
            auto fetch = [&](int it, float &l, float &dd) {
                const int mt = w.n + it / p.G, h = w.j * p.G + it % p.G;
                const int t = mt * kRows + r;
                l = INFINITY;
                dd = 0.f;
                if (t < w.tl) {
                    const size_t idx =
                        (static_cast<size_t>(w.sq.bc) * p.Hq + h) * p.T + w.sq.base + t;
                    l = p.lse[idx];
                    dd = p.Dws[idx];
                }
            };
            float nl, nd;
            fetch(0, nl, nd);
            for (int it = 0; it < w.nitems; ++it, ++gi) {
                const int st = gi % ST, su = gi / ST;
                const float l2 = nl * kLog2e, dd = nd;
                if (it + 1 < w.nitems)
                    fetch(it + 1, nl, nd);
                // The stage's previous item is finished once the TMA has refilled
                // it, so its lse/D slots can be overwritten.
                if (!mbar_wait_warp_idle(smem_u32(&bar_q_full[st]), su & 1, wc)) {
                    ok = false;
                    break;
                }
                // negated, paired by columns: one 16-byte load gives the row
                // warps two columns' (-lse, -D) as packed fp32 pairs
                lsed[st * 2 * kRows + (r >> 1) * 4 + (r & 1)] = -l2;
                lsed[st * 2 * kRows + (r >> 1) * 4 + 2 + (r & 1)] = -dd;
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_q_ready[st]));
            }
        }
        if (mx > kFp16Max)
            atomicOr(p.status, kDevRange);
        teardown();
        return;
    } else {
        // ---------------------------------------------- row warpgroups ---
        regs_claim<kRowRegs>();
        const int w = warp >> 2;                // column half of the score tile
        const int r = threadIdx.x & 127;        // key row == TMEM lane
        const uint32_t lane_base = tmem_addr(tbase, (warp & 3) * 32, 0);
        float maxds = 0.f;
        bool ok = true;
        int gi = 0;
        // The epilogue of a unit (dV, dK out of TMEM) runs after the next
        // unit's first item has been handed to the dV/dK issuer, so the wait
        // for the unit's last MMAs overlaps that item's softmax work; the
        // first dV/dK of the next unit waits for acc_free anyway.
        int pend_k = -1;
        DkvUnit pend{};
        auto epilogue = [&]() {
            if (!mbar_wait_warp(smem_u32(&bar_acc_done), pend_k & 1, wc))
                return false;
            tc_fence_after();
            const int s = pend.n * kRows + r;
            const size_t rowoff = (seq_row(p, pend.sq, s) * p.Hkv + pend.j) * D;
            if (w == 0) {
                __nv_bfloat16 *dv = static_cast<__nv_bfloat16 *>(p.out1) + rowoff;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t a[32];
                    tmem_ld32(lane_base + C::COL_DV + cc * 32, a);
                    tmem_ld_wait(a);
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        x[e] = __uint_as_float(a[e]);
                    if (s < pend.tl)
                        store_row32_bf16(dv + cc * 32, x);
                }
            } else {
                __nv_bfloat16 *dkp = static_cast<__nv_bfloat16 *>(p.out0) + rowoff;
                epilogue_inverse_rope<D>(lane_base + C::COL_DK, p.scale, static_cast<uint32_t>(s),
                                         p.rope, dkp, s < pend.tl);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bar_acc_free));
            pend_k = -1;
            return true;
        };
        for (int k = 0; ok; ++k) {
            const int u = snake_unit(k, cta, P);
            if (u >= NU)
                break;
            const DkvUnit un = dkv_unit<VAR>(u, p);
            for (int it = 0; it < un.nitems; ++it, ++gi) {
                const int st = gi % ST, su = gi / ST;
                const int mt = un.n + it / p.G;
                if (!mbar_wait_warp(smem_u32(&bar_q_ready[st]), su & 1, wc) ||
                    !mbar_wait_warp(smem_u32(&bar_s_full), gi & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sv[2][32], pv[2][32];
                tmem_ld32(lane_base + C::COL_S + 64 * w, sv[0]);
                tmem_ld32(lane_base + C::COL_S + 64 * w + 32, sv[1]);
                tmem_ld32(lane_base + C::COL_DP + 64 * w, pv[0]);
                tmem_ld32(lane_base + C::COL_DP + 64 * w + 32, pv[1]);
                tmem_ld_wait_only();
                tmem_tie(sv[0]);
                tmem_tie(sv[1]);
                tmem_tie(pv[0]);
                tmem_tie(pv[1]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_s_empty));

                const float4 *ld4 =
                    reinterpret_cast<const float4 *>(lsed + st * 2 * kRows + 2 * 64 * w);
                uint32_t pp[32], dk[32];
                const uint64_t sl2x2 = f32x2(p.scale_log2, p.scale_log2);
                // sliding window: query columns c >= wmin (query >= key + W)
                // are masked
                int wmin = 1 << 30;
                if constexpr (WIN)
                    wmin = un.n * kRows + r + p.window - mt * kRows;
                // column pair (c, c+1): P = 2^(S sl2 - l2), dS = P (dP - D) on
                // packed fp32 pairs; masked entries (query column c before key
                // row r on the diagonal tile, or outside the window) get P = 0
                const bool masked = mt == un.n || (WIN && __any_sync(0xffffffffu, wmin < kRows));
                const int clo = (!WIN || mt == un.n) ? r : -1;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float4 a = ld4[(32 * h + e) >> 1];   // -l2, -l2', -D, -D'
                        const uint64_t x2 = fma_f32x2(
                            f32x2(__uint_as_float(sv[h][e]), __uint_as_float(sv[h][e + 1])), sl2x2,
                            f32x2(a.x, a.y));
                        float x0, x1;
                        f32x2_split(x2, x0, x1);
                        float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        if (masked) {
                            const int c = 64 * w + 32 * h + e;
                            p0 = (c < clo || (WIN && c >= wmin)) ? 0.f : p0;
                            p1 = (c + 1 < clo || (WIN && c + 1 >= wmin)) ? 0.f : p1;
                        }
                        const uint64_t pr2 = f32x2(p0, p1);
                        const uint64_t ds2 = mul_f32x2(
                            pr2, add_f32x2(f32x2(__uint_as_float(pv[h][e]),
                                                 __uint_as_float(pv[h][e + 1])),
                                           f32x2(a.z, a.w)));
                        float d0, d1;
                        f32x2_split(ds2, d0, d1);
                        maxds = fmax3(maxds, fabsf(d0), fabsf(d1));
                        pp[16 * h + e / 2] = pack_bf16x2(p0, p1);
                        dk[16 * h + e / 2] = pack_f16x2(d0, d1);
                    }
                if (gi >= 1 && !mbar_wait_warp(smem_u32(&bar_pds_empty), (gi - 1) & 1, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_st32(lane_base + C::col_p(w), pp);
                tmem_st32(lane_base + C::col_ds(w), dk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&bar_pds_full));
                if (it == 0 && pend_k >= 0 && !epilogue()) {
                    ok = false;
                    break;
                }
            }
            if (!ok)
                break;
            pend_k = k;      // dV, dK of this unit: out at the next unit's first item
            pend = un;
        }
        if (ok && pend_k >= 0)
            ok = epilogue();
        if (maxds > kFp16Max)
            atomicOr(p.status, kDevRange);
        teardown();
    }
}

// ------------------------------------------------------------- launch ---

template <int D, int GC, int ST, bool WIN, bool VAR>
static cudaError_t launch_dq_w(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                               const CUtensorMap &dO, const CUtensorMap &dq,
                               const AttnParams &p0, cudaStream_t stream)
{
    using C = DqCfg<D, GC, ST>;
    auto kern = dq_kernel<D, GC, ST, WIN, VAR>;
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
    return launch_pdl(kern, grid, 384, C::SMEM_BYTES, stream, q, k, v, dO, dq, p);
}

template <int D, int GC, int ST>
static cudaError_t launch_dq_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                               const CUtensorMap &dO, const CUtensorMap &dq, const AttnParams &p,
                               cudaStream_t stream)
{
    if (p.window > 0)
        return launch_dq_w<D, GC, ST, true, false>(q, k, v, dO, dq, p, stream);
    if (p.units)
        return launch_dq_w<D, GC, ST, false, true>(q, k, v, dO, dq, p, stream);
    return launch_dq_w<D, GC, ST, false, false>(q, k, v, dO, dq, p, stream);
}

cudaError_t launch_bwd_dq(int d, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                          const CUtensorMap &dO, const CUtensorMap &dq, const AttnParams &p,
                          cudaStream_t stream)
{
    switch (d) {
    case 32:
        switch (p.GC) {
        case 1: return launch_dq_t<32, 1, 4>(q, k, v, dO, dq, p, stream);
        case 2: return launch_dq_t<32, 2, 4>(q, k, v, dO, dq, p, stream);
        case 3: return launch_dq_t<32, 3, 4>(q, k, v, dO, dq, p, stream);
        case 4: return launch_dq_t<32, 4, 4>(q, k, v, dO, dq, p, stream);
        default: break;
        }
        break;
    case 64:
        switch (p.GC) {
        case 1: return launch_dq_t<64, 1, 3>(q, k, v, dO, dq, p, stream);
        case 2: return launch_dq_t<64, 2, 3>(q, k, v, dO, dq, p, stream);
        case 3: return launch_dq_t<64, 3, 3>(q, k, v, dO, dq, p, stream);
        default: break;
        }
        break;
    case 128:
        if (p.GC == 1)
            return launch_dq_t<128, 1, 2>(q, k, v, dO, dq, p, stream);
        break;
    default: break;
    }
    return cudaErrorInvalidValue;
}

template <int D, int ST, bool WIN, bool VAR>
static cudaError_t launch_dkdv_w(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                 const CUtensorMap &dO, const AttnParams &p0, cudaStream_t stream)
{
    using C = DkvCfg<D, ST>;
    auto kern = dkdv_kernel<D, ST, WIN, VAR>;
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
        p.num_units = p.M * p.B * p.Hkv;   // varlen: the table's length
    // a count in device memory is unknown here: one CTA per SM
    const int nu = (VAR && p.unit_count != nullptr) ? sms : p.num_units;
    const unsigned grid = static_cast<unsigned>(nu < sms ? nu : sms);
    return launch_pdl(kern, grid, 512, C::SMEM_BYTES, stream, q, k, v, dO, p);
}

template <int D, int ST>
static cudaError_t launch_dkdv_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                 const CUtensorMap &dO, const AttnParams &p, cudaStream_t stream)
{
    if (p.window > 0)
        return launch_dkdv_w<D, ST, true, false>(q, k, v, dO, p, stream);
    if (p.units)
        return launch_dkdv_w<D, ST, false, true>(q, k, v, dO, p, stream);
    return launch_dkdv_w<D, ST, false, false>(q, k, v, dO, p, stream);
}

cudaError_t launch_bwd_dkdv(int d, const CUtensorMap &q, const CUtensorMap &k,
                            const CUtensorMap &v, const CUtensorMap &dO, const AttnParams &p,
                            cudaStream_t stream)
{
    switch (d) {
    case 32: return launch_dkdv_t<32, 4>(q, k, v, dO, p, stream);
    case 64: return launch_dkdv_t<64, 4>(q, k, v, dO, p, stream);
    case 128: return launch_dkdv_t<128, 1>(q, k, v, dO, p, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace ne
