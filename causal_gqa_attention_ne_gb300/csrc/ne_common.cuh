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

// RoPE angles.  Frequency i is passed as a 64-bit fixed-point number of
// turns per position, F_i = round(2^64 * theta^(-2i/d) / (2 pi)) mod 2^64,
// split into its high and low 32-bit words.  The angle of position p, in
// turns modulo 1, is p * F_i mod 2^64; its top 32 bits are
// p * hi + floor(p * lo / 2^32) (mod 2^32): integer arithmetic, exact but for
// the dropped low word (under 2^-32 turn).  That top word, read as a signed
// fraction of a turn, is the angle in [-pi, pi) before the hardware
// sine/cosine, so the error of the angle does not grow with the position.
struct RopeFreqs {
    uint32_t hi[64];
    uint32_t lo[64];
};

__device__ __forceinline__ void rope_sincos(uint32_t pos, const RopeFreqs &fr, int i, float &s,
                                            float &c)
{
    const int32_t t = static_cast<int32_t>(pos * fr.hi[i] + __umulhi(pos, fr.lo[i]));
    const float ang = static_cast<float>(t) * 1.4629180792671596e-09f;   // 2 pi / 2^32
    __sincosf(ang, &s, &c);
}

// One rotate-half pair (x, y) rotated by the angle with cosine c and sine s:
// (x c - y s, y c + x s).  The operations are rounded explicitly (one
// product, then a fused multiply-add), so the forward, the backward's
// preprocess and the exact-score path produce the same bits for the same
// input, whatever contractions the compiler would choose in each kernel.
__device__ __forceinline__ void rope_rotate(float x, float y, float c, float s, float &u,
                                            float &w)
{
    u = __fmaf_rn(x, c, -__fmul_rn(y, s));
    w = __fmaf_rn(y, c, __fmul_rn(x, s));
}

// Rotate row r of a bf16 tile in place to fp16 with the hardware sine/cosine
// per pair, loading a batch of up to four chunk pairs before computing so the
// shared-memory and special-function latencies overlap.  Returns max |x'|
// (the fp16 range check) and sets ss to the sum of x'^2 over the row (fp32,
// before rounding).
template <int D>
__device__ __forceinline__ float rope_row_ilp(uint8_t *tile, int r, uint32_t pos,
                                              const RopeFreqs &fr, float &ss)
{
    constexpr int HC = D / 16;
    constexpr int BATCH = HC < 2 ? HC : 2;
    float mx = 0.f;
    ss = 0.f;
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
                    rope_sincos(pos, fr, 8 * (c0 + i) + 2 * e + h, sn, cs);
                    const float x = h ? bf16_hi(av[e]) : bf16_lo(av[e]);
                    const float y = h ? bf16_hi(bv[e]) : bf16_lo(bv[e]);
                    rope_rotate(x, y, cs, sn, u[h], w[h]);
                    mx = fmaxf(mx, fmaxf(fabsf(u[h]), fabsf(w[h])));
                    ss = fmaf(u[h], u[h], fmaf(w[h], w[h], ss));
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
__device__ __forceinline__ void rope_inverse_pair(float &x, float &y, uint32_t pos,
                                                  const RopeFreqs &fr, int i)
{
    float s, c;
    rope_sincos(pos, fr, i, s, c);
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
    const void *q_in, *k_in, *v_in;   // forward: bf16 q, k, v (re-read to repair large rows)
    const void *o_in;            // backward: forward output O (preprocess)
    const void *do_in;           // backward: dO (preprocess)
    void *out0;                  // forward: O; backward: dq / dk
    void *out1;                  // backward: dv
    float *lse;                  // forward: written; backward: read
    float *Dws;                  // backward: D = rowsum(dO * O), [B][Hq][T]
    uint32_t *status;            // device status word
    int num_units;               // persistent kernels: work units in the launch
    const int *unit_count;       // varlen planned on the device: num_units there instead
    uint64_t wait_limit_ns;
    int save_rot;                // forward: also store Q' and K' (fp16) for the backward
    int window;                  // 0: causal; W > 0: query t sees keys t-W+1 .. t
    // padded variable-length batches (varlen instantiations only): the live
    // work units of the launch (indices into the full enumeration, num_units
    // of them) and the valid length of every sequence, both in device memory
    const int *units;
    const int *seqlen;
    // packed variable-length batches (varlen instantiations with cu set):
    // the sequences are concatenated along the rows of one batch entry
    // (B = 1 in memory, T = the total row count), sequence b starting at row
    // cu[b]; the launch's B is the sequence count
    const int *cu;
    int nseq;                    // packed: the number of sequences (cu has nseq + 1 entries)
    RopeFreqs rope;
};

// Work units of a persistent launch: num_units, or (variable-length batches
// planned on the device) the count the plan kernel wrote.  Read after the
// grid dependency wait.
template <bool VAR>
__device__ __forceinline__ int unit_total(const AttnParams &p)
{
    if constexpr (VAR) {
        if (p.unit_count != nullptr)
            return *p.unit_count;
    }
    return p.num_units;
}

// Where sequence b of a launch lives: the TMA batch coordinate bc and first
// row base of its rows, and its valid rows len.  Plain and padded batches:
// bc = b, base = 0 (len = T, or the sequence's length); packed batches:
// bc = 0, base = cu[b].
struct SeqLoc {
    int bc, base, len;
};
template <bool VAR>
__device__ __forceinline__ SeqLoc seq_loc(const AttnParams &p, int b)
{
    if constexpr (VAR) {
        const int len = __ldg(p.seqlen + b);
        if (p.cu != nullptr)
            return SeqLoc{0, __ldg(p.cu + b), len};
        return SeqLoc{b, 0, len};
    }
    return SeqLoc{b, 0, p.T};
}

// Row t of a sequence in the [B][T] row space of a tensor (T = p.T).
__device__ __forceinline__ size_t seq_row(const AttnParams &p, const SeqLoc &s, int t)
{
    return static_cast<size_t>(s.bc) * p.T + s.base + t;
}

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
