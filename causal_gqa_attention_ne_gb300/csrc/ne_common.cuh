// ne_common.cuh -- tile geometry, RoPE helpers and launch parameters shared by
// the forward and backward attention kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"

namespace ne {

constexpr int kRows = 128;          // query rows and key rows per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kFp16Max = 65504.0f;

// Kernels that allocate all 512 TMEM columns request at least this much
// dynamic shared memory, so two of their CTAs never share an SM (the second
// would otherwise stall in tcgen05.alloc until the first exits).
constexpr int kOneCtaPerSmSmem = 116 * 1024;
constexpr int smem_one_cta(int bytes) { return bytes > kOneCtaPerSmSmem ? bytes : kOneCtaPerSmSmem; }

// Geometry of one 128-row tile of head dimension D in shared memory, exactly
// as TMA lands it: the D columns are split into NB column blocks of SWB bytes
// per row (SWB = 128 for D >= 64, 64 for D = 32); each block is 128 rows of
// SWB bytes with the matching TMA/UMMA swizzle (128-byte or 64-byte).
template <int D>
struct Tile {
    static constexpr int SWB = (2 * D < 128) ? 2 * D : 128;
    static constexpr int NB = 2 * D / SWB;
    static constexpr int BLOCK = kRows * SWB;        // bytes per column block
    static constexpr int BYTES = kRows * 2 * D;      // bytes per tile
    static constexpr uint32_t LAYOUT = (SWB == 128) ? 2u : 4u;
    static constexpr int BOX_COLS = SWB / 2;         // TMA box width in elements
    static constexpr int NPV = (D < 64) ? D : 64;    // N of one MN-major MMA (one swizzle atom)
};

// Physical byte offset of logical byte `lin` of a swizzled block whose rows
// are `swb` bytes: 16-byte chunk bits [4,6|7) are XOR-ed with address bits
// [7,9|10).
template <int SWB>
__device__ __forceinline__ uint32_t swz(uint32_t lin)
{
    constexpr uint32_t mask = (SWB == 128) ? 7u : 3u;
    return lin ^ (((lin >> 7) & mask) << 4);
}

// Byte offset of the 16-byte chunk holding elements [8c, 8c+8) of row r of a
// D-wide tile.
template <int D>
__device__ __forceinline__ uint32_t tile_chunk(int r, int c)
{
    using TL = Tile<D>;
    constexpr int CPB = TL::SWB / 16;   // chunks per block row
    return (c / CPB) * TL::BLOCK + swz<TL::SWB>(r * TL::SWB + (c % CPB) * 16);
}

// Byte offset of chunk c (8 keys) of row r of a 128x128 16-bit tile (P, dS):
// two column blocks of 64 elements, 128-byte swizzle.
__device__ __forceinline__ uint32_t ptile_chunk(int r, int c)
{
    return (c >> 3) * (kRows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// K-major operand descriptor of a D-wide tile for K step kk (16 elements).
template <int D>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile_addr, int kk)
{
    using TL = Tile<D>;
    const int byte = kk * 32;
    return smem_desc(tile_addr + (byte / TL::SWB) * TL::BLOCK + (byte % TL::SWB), 16,
                     8 * TL::SWB, TL::LAYOUT);
}

// K-major descriptor of a 128x128 16-bit tile (P or dS) for K step kk.
__device__ __forceinline__ uint64_t desc_ptile(uint32_t tile_addr, int kk)
{
    return smem_desc(tile_addr + (kk >> 2) * (kRows * 128) + (kk & 3) * 32, 16, 1024, 2u);
}

// MN-major descriptor of a D-wide tile used as the B operand with N = the
// tile's columns and K = its rows: N chunk nc (one swizzle atom, NPV
// columns), K step kk (16 rows).  The operand never spans two atoms along N,
// so only the K-direction stride between 8-row groups matters; it is written
// into both offset fields.
template <int D>
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile_addr, int nc, int kk)
{
    using TL = Tile<D>;
    return smem_desc(tile_addr + nc * TL::BLOCK + kk * 16 * TL::SWB, 8 * TL::SWB, 8 * TL::SWB,
                     TL::LAYOUT);
}

// RoPE angles.  Frequency i is passed as a 32-bit fixed-point number of turns
// per position, F_i = round(2^32 * theta^(-2i/d) / (2 pi)).  The angle of
// position p is then p * F_i modulo 2^32 turns (exact integer wrap-around),
// mapped to [-pi, pi) before the hardware sine/cosine.
struct RopeFreqs {
    uint32_t turn[64];
};

__device__ __forceinline__ void rope_sincos(uint32_t pos, uint32_t f, float &s, float &c)
{
    const int32_t t = static_cast<int32_t>(pos * f);
    const float ang = static_cast<float>(t) * 1.4629180792671596e-09f;   // 2 pi / 2^32
    __sincosf(ang, &s, &c);
}

// Rotate row r of a bf16 tile in place, writing fp16 (the score-side operand
// type).  x'_i = x_i cos - x_{i+D/2} sin, x'_{i+D/2} = x_{i+D/2} cos + x_i sin.
// Returns the largest |x'| seen (for the fp16 range check).
template <int D>
__device__ __forceinline__ float rope_row_to_f16(uint8_t *tile, int r, uint32_t pos,
                                                 const RopeFreqs &fr)
{
    constexpr int HC = D / 16;   // chunks in the first half of the row
    float mx = 0.f;
#pragma unroll
    for (int c = 0; c < HC; ++c) {
        uint4 *pa = reinterpret_cast<uint4 *>(tile + tile_chunk<D>(r, c));
        uint4 *pb = reinterpret_cast<uint4 *>(tile + tile_chunk<D>(r, c + HC));
        const uint4 a = *pa, b = *pb;
        const uint32_t av[4] = {a.x, a.y, a.z, a.w};
        const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
        uint32_t ao[4], bo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float s0, c0, s1, c1;
            rope_sincos(pos, fr.turn[8 * c + 2 * e], s0, c0);
            rope_sincos(pos, fr.turn[8 * c + 2 * e + 1], s1, c1);
            const float x0 = bf16_lo(av[e]), x1 = bf16_hi(av[e]);
            const float y0 = bf16_lo(bv[e]), y1 = bf16_hi(bv[e]);
            const float u0 = x0 * c0 - y0 * s0, w0 = y0 * c0 + x0 * s0;
            const float u1 = x1 * c1 - y1 * s1, w1 = y1 * c1 + x1 * s1;
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(u0), fabsf(w0)), fmaxf(fabsf(u1), fabsf(w1))));
            ao[e] = pack_f16x2(u0, u1);
            bo[e] = pack_f16x2(w0, w1);
        }
        *pa = make_uint4(ao[0], ao[1], ao[2], ao[3]);
        *pb = make_uint4(bo[0], bo[1], bo[2], bo[3]);
    }
    return mx;
}

// ---- table-driven RoPE (no special-function unit work per element) ----
//
// A CTA keeps float2 tab[j][r] = (cos, sin)(r * theta_j) for the 128 rows r
// of a tile and the D/2 frequencies j, and per rotated tile the 64 values
// base[j] = (cos, sin)(p0 * theta_j) of the tile's first position p0.  The
// angle of row r is p0*theta_j + r*theta_j; its cosine and sine come from the
// angle-addition formulas (four multiply-adds).  Both tables come from the
// hardware sine/cosine on the exactly reduced angle in [-pi, pi), where its
// absolute error is below 4e-7 (far below the fp16 rounding of the result).

__device__ __forceinline__ float2 rope_cs(uint32_t pos, uint32_t f)
{
    float s, c;
    rope_sincos(pos, f, s, c);
    return make_float2(c, s);
}

// Thread r (0..127) fills row r of the table.
template <int D>
__device__ __forceinline__ void rope_table_fill(float2 *tab, int r, const RopeFreqs &fr)
{
#pragma unroll 4
    for (int j = 0; j < D / 2; ++j)
        tab[j * kRows + r] = rope_cs(static_cast<uint32_t>(r), fr.turn[j]);
}

// Rotate row r of a bf16 tile in place to fp16 using the table and the
// tile's base; returns the largest |x'| (fp16 range check).
template <int D>
__device__ __forceinline__ float rope_row_table(uint8_t *tile, int r, const float2 *tab,
                                                const float2 *base)
{
    constexpr int HC = D / 16;
    float mx = 0.f;
#pragma unroll
    for (int c = 0; c < HC; ++c) {
        uint4 *pa = reinterpret_cast<uint4 *>(tile + tile_chunk<D>(r, c));
        uint4 *pb = reinterpret_cast<uint4 *>(tile + tile_chunk<D>(r, c + HC));
        const uint4 a = *pa, b = *pb;
        const uint32_t av[4] = {a.x, a.y, a.z, a.w};
        const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
        uint32_t ao[4], bo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float u[2], w[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = 8 * c + 2 * e + h;
                const float2 t = tab[j * kRows + r];
                const float2 bs = base[j];
                const float cs = bs.x * t.x - bs.y * t.y;
                const float sn = bs.y * t.x + bs.x * t.y;
                const float x = h ? bf16_hi(av[e]) : bf16_lo(av[e]);
                const float y = h ? bf16_hi(bv[e]) : bf16_lo(bv[e]);
                u[h] = x * cs - y * sn;
                w[h] = y * cs + x * sn;
                mx = fmaxf(mx, fmaxf(fabsf(u[h]), fabsf(w[h])));
            }
            ao[e] = pack_f16x2(u[0], u[1]);
            bo[e] = pack_f16x2(w[0], w[1]);
        }
        *pa = make_uint4(ao[0], ao[1], ao[2], ao[3]);
        *pb = make_uint4(bo[0], bo[1], bo[2], bo[3]);
    }
    return mx;
}

// Rotate row r of a bf16 tile in place to fp16 with the hardware sine/cosine
// per pair, loading a batch of up to four chunk pairs before computing so the
// shared-memory and special-function latencies overlap.  Returns max |x'|.
template <int D>
__device__ __forceinline__ float rope_row_ilp(uint8_t *tile, int r, uint32_t pos,
                                              const RopeFreqs &fr)
{
    constexpr int HC = D / 16;
    constexpr int BATCH = HC < 2 ? HC : 2;
    float mx = 0.f;
#pragma unroll
    for (int c0 = 0; c0 < HC; c0 += BATCH) {
        uint4 a[BATCH], b[BATCH];
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            a[i] = *reinterpret_cast<const uint4 *>(tile + tile_chunk<D>(r, c0 + i));
            b[i] = *reinterpret_cast<const uint4 *>(tile + tile_chunk<D>(r, c0 + i + HC));
        }
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            uint32_t av[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
            uint32_t bv[4] = {b[i].x, b[i].y, b[i].z, b[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float u[2], w[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float sn, cs;
                    rope_sincos(pos, fr.turn[8 * (c0 + i) + 2 * e + h], sn, cs);
                    const float x = h ? bf16_hi(av[e]) : bf16_lo(av[e]);
                    const float y = h ? bf16_hi(bv[e]) : bf16_lo(bv[e]);
                    u[h] = x * cs - y * sn;
                    w[h] = y * cs + x * sn;
                    mx = fmaxf(mx, fmaxf(fabsf(u[h]), fabsf(w[h])));
                }
                av[e] = pack_f16x2(u[0], u[1]);
                bv[e] = pack_f16x2(w[0], w[1]);
            }
            a[i] = make_uint4(av[0], av[1], av[2], av[3]);
            b[i] = make_uint4(bv[0], bv[1], bv[2], bv[3]);
        }
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            *reinterpret_cast<uint4 *>(tile + tile_chunk<D>(r, c0 + i)) = a[i];
            *reinterpret_cast<uint4 *>(tile + tile_chunk<D>(r, c0 + i + HC)) = b[i];
        }
    }
    return mx;
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

// Inverse rotation (by -angle) of a pair of fp32 values held in registers.
__device__ __forceinline__ void rope_inverse_pair(float &x, float &y, uint32_t pos, uint32_t f)
{
    float s, c;
    rope_sincos(pos, f, s, c);
    const float u = x * c + y * s;
    const float w = y * c - x * s;
    x = u;
    y = w;
}

// Raises a kernel's dynamic shared-memory limit once per device (not on
// every launch, so launches stay cheap and capturable in CUDA graphs).
// `done` must be a flag array owned by exactly one kernel instantiation.
template <typename Kernel>
inline cudaError_t ensure_smem_attr(Kernel kern, int bytes, bool (&done)[64])
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < 64 && done[dev])
        return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64)
        done[dev] = true;
    return e;
}

// Launches `kern` with programmatic stream serialization: the grid may be
// scheduled while the previous kernel in the stream is still finishing (as
// soon as every CTA of that kernel has run griddep_launch_dependents or
// exited).  Every kernel of this library runs griddep_wait() after its
// shared-memory / TMEM prologue and before its first global-memory access,
// so only the prologue and the launch latency overlap the previous kernel.
// After a kernel that never triggers early (any kernel not from this
// library) the launch behaves like a plain one.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                              cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Descriptor offsets (in the descriptor's 16-byte address units) of the K
// step kk of a K-major D-wide tile, and of (N chunk nc, K step kk) of an
// MN-major one, relative to the tile's base descriptor.  Compile-time
// constants, so each MMA needs one add.
template <int D>
__host__ __device__ constexpr uint32_t kmajor_off(int kk)
{
    return static_cast<uint32_t>(((kk * 32) / Tile<D>::SWB * Tile<D>::BLOCK +
                                  (kk * 32) % Tile<D>::SWB) >> 4);
}
template <int D>
__host__ __device__ constexpr uint32_t mnmajor_off(int nc, int kk)
{
    return static_cast<uint32_t>((nc * Tile<D>::BLOCK + kk * 16 * Tile<D>::SWB) >> 4);
}
template <int D>
__device__ __forceinline__ uint64_t desc_kmajor_base(uint32_t tile_addr)
{
    return smem_desc(tile_addr, 16, 8 * Tile<D>::SWB, Tile<D>::LAYOUT);
}
template <int D>
__device__ __forceinline__ uint64_t desc_mnmajor_base(uint32_t tile_addr)
{
    return smem_desc(tile_addr, 8 * Tile<D>::SWB, 8 * Tile<D>::SWB, Tile<D>::LAYOUT);
}

// Persistent-CTA work order: CTA c of P takes units c, 2P-1-c, 2P+c, 4P-1-c,
// ... (a snake over a list sorted by decreasing cost), which balances the
// causal work across CTAs without any shared counter.
__device__ __forceinline__ int snake_unit(int k, int c, int P)
{
    return (k & 1) ? k * P + (P - 1 - c) : k * P + c;
}

// Launch parameters (everything except the TMA descriptors).
struct AttnParams {
    int B, T, Hq, Hkv, G, M;     // M = number of 128-row tiles along T
    int GC, nchunks;             // query heads per CTA, CTAs per KV group (Q-major kernels)
    float scale_log2;            // log2(e) / sqrt(d)
    float scale;                 // 1 / sqrt(d)
    const void *o_in;            // backward: forward output O (preprocess)
    const void *do_in;           // backward: dO (preprocess)
    void *out0;                  // forward: O; backward: dq / dk
    void *out1;                  // backward: dv
    float *lse;                  // forward: written; backward: read
    float *Dws;                  // backward: D = rowsum(dO * O), [B][Hq][T]
    uint32_t *status;            // device status word
    int num_units;               // persistent kernels: work units in the launch
    uint64_t wait_limit_ns;
    int save_rot;                // forward: also store Q' and K' (fp16) for the backward
    int window;                  // 0: causal; W > 0: query t sees keys t-W+1 .. t
    // padded variable-length batches (varlen instantiations only): the live
    // work units of the launch (indices into the full enumeration, num_units
    // of them) and the valid length of every sequence, both in device memory
    const int *units;
    const int *seqlen;
    RopeFreqs rope;
};

// Sliding window: the first key tile any row of query tile m sees (0 without
// a window: its first row t = 128 m sees keys >= t - W + 1), and the last
// query tile any key of key tile n is visible to (t <= 128 n + 127 + W - 1).
__host__ __device__ inline int key_tile_lo(int m, int window)
{
    if (window <= 0)
        return 0;
    const int lo_key = m * kRows - window + 1;
    return lo_key <= 0 ? 0 : lo_key / kRows;
}
__host__ __device__ inline int query_tile_hi(int n, int window, int M)
{
    if (window <= 0)
        return M - 1;
    const int hi = (n * kRows + kRows - 2 + window) / kRows;
    return hi < M - 1 ? hi : M - 1;
}

} // namespace ne
