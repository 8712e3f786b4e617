// ne_varlen.cu -- padded variable-length batches: the host-side tables of
// live work units, and the fill of padding rows.
//
// The NanoEuler SFT stage pads every instruction/response pair to the context
// length and masks the loss on prompt and padding ("Rebuilding GPT-2 in one
// 100KB C/CUDA file", section 3.2, SFT stage).  Attention over a padded batch
// with per-sequence lengths L_b is one causal problem per sequence over its
// first L_b rows; a padding row attends to nothing (O = 0, lse = -inf) and
// padding positions get zero gradients.  The persistent kernels run such a
// batch from a table of their live units: a query tile (forward, dq) or key
// tile (dk/dv) that lies wholly past L_b does no work at all, and a dk/dv unit
// stops at its sequence's last query tile.  The kernels compute the padding
// rows of a live tile like any other row; pad_fill_kernel then writes the
// defined values over every padding row.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "ne_common.cuh"
#include "ne_kernels.h"

namespace ne {

// Rows t >= seqlen[b] of up to three [B][T][row] tensors are set to zero and
// lse[b][h][t] (if given) to -inf.  Block i serves sequence i / per and part
// i % per of its padding; 16-byte stores.
__global__ void __launch_bounds__(256) pad_fill_kernel(const PadFillParams p, int per)
{
    griddep_wait();
    const int b = static_cast<int>(blockIdx.x) / per;
    const int part = static_cast<int>(blockIdx.x) % per;
    const int L = p.seqlen[b];
    const int npad = p.T - L;
    if (npad > 0) {
        const size_t tid = static_cast<size_t>(part) * blockDim.x + threadIdx.x;
        const size_t nthr = static_cast<size_t>(per) * blockDim.x;
        for (int i = 0; i < p.ntensors; ++i) {
            const size_t row16 = static_cast<size_t>(p.row_bytes[i]) / 16;
            uint4 *pad = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.x[i]) +
                                                   (static_cast<size_t>(b) * p.T + L) *
                                                       p.row_bytes[i]);
            const size_t n = static_cast<size_t>(npad) * row16;
            for (size_t c = tid; c < n; c += nthr)
                pad[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (p.lse) {
            const size_t n = static_cast<size_t>(p.Hq) * npad;
            for (size_t c = tid; c < n; c += nthr) {
                const size_t h = c / npad, t = L + c % npad;
                p.lse[(static_cast<size_t>(b) * p.Hq + h) * p.T + t] = -INFINITY;
            }
        }
    }
    griddep_launch_dependents();
}

cudaError_t launch_pad_fill(const PadFillParams &p, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    // about four blocks per SM in all, at least one per sequence
    const int per = std::max(1, (4 * sms + p.B - 1) / p.B);
    const unsigned grid = static_cast<unsigned>(static_cast<size_t>(p.B) * per);
    return launch_pdl(pad_fill_kernel, grid, 256, 0, stream, p, per);
}

// The live units, as indices into each kernel's full enumeration (the decode
// functions in ne_fwd.cu and ne_bwd.cu):
//   forward / dq: u -> m = M-1 - u / (B Hkv nchunks), then chunk, j, b; live
//                 iff query tile m has a valid row, 128 m < L_b; the
//                 enumeration is by decreasing m, i.e. decreasing work, and
//                 the filtered list keeps that order;
//   dk/dv:        u -> n = u / (B Hkv), then j, b; live iff 128 n < L_b; its
//                 work is the ceil(L_b / 128) - n query tiles it visits, so
//                 the list is sorted by that (stable), largest first.
// The persistent kernels deal the list out in a snake over their CTAs, which
// balances a list sorted by decreasing work.
int varlen_plan(const int *seqlen, int B, int T, int Hq, int Hkv, int d, int *fwd_units,
                int *dq_units, int *dkv_units, const size_t caps[3], int counts[3])
{
    const int G = Hq / Hkv, M = (T + kRows - 1) / kRows;
    std::vector<int> mt(static_cast<size_t>(B));
    for (int b = 0; b < B; ++b)
        mt[static_cast<size_t>(b)] = (seqlen[b] + kRows - 1) / kRows;
    int *tables[2] = {fwd_units, dq_units};
    const int chunks[2] = {G / fwd_heads_per_cta(d, G), G / dq_heads_per_cta(d, G)};
    for (int k = 0; k < 2; ++k) {
        const int nch = chunks[k];
        const size_t per_m = static_cast<size_t>(B) * Hkv * nch;
        size_t n = 0;
        for (size_t u = 0; u < static_cast<size_t>(M) * per_m; ++u) {
            const int m = M - 1 - static_cast<int>(u / per_m);
            const int b = static_cast<int>((u % per_m) / nch / Hkv);
            if (m < mt[static_cast<size_t>(b)]) {
                if (tables[k] && n < caps[k])
                    tables[k][n] = static_cast<int>(u);
                ++n;
            }
        }
        counts[k] = static_cast<int>(n);
    }
    const size_t per_n = static_cast<size_t>(B) * Hkv;
    std::vector<int> live;
    for (size_t u = 0; u < static_cast<size_t>(M) * per_n; ++u) {
        const int n = static_cast<int>(u / per_n);
        const int b = static_cast<int>((u % per_n) / Hkv);
        if (n < mt[static_cast<size_t>(b)])
            live.push_back(static_cast<int>(u));
    }
    auto work = [&](int u) {
        const int n = static_cast<int>(static_cast<size_t>(u) / per_n);
        const int b = static_cast<int>((static_cast<size_t>(u) % per_n) / Hkv);
        return mt[static_cast<size_t>(b)] - n;
    };
    std::stable_sort(live.begin(), live.end(), [&](int a, int c) { return work(a) > work(c); });
    if (dkv_units)
        for (size_t i = 0; i < live.size() && i < caps[2]; ++i)
            dkv_units[i] = live[i];
    counts[2] = static_cast<int>(live.size());
    return 0;
}

// ----------------------------------------------------- device-side plan ---
// The same tables, built on the GPU from lengths in device memory, so a
// variable-length call can be captured into a CUDA graph and replayed with
// other lengths.  One CTA of kPlanThreads threads.  Forward and dq tables:
// the live units of each enumeration, compacted in order (a block-wide
// scan per slice of the enumeration).  dk/dv table: the stable sort by
// decreasing work has a closed form.  Unit u = n (B Hkv) + b Hkv + j is live
// iff n < mt_b (mt_b = ceil(L_b / 128)) and has work w = mt_b - n; among the
// units of work w, ordered by u, the one of (b, j) comes after the units of
// every b' with w <= mt_b' < mt_b, then those of every b' < b with
// mt_b' = mt_b, then j of its own.  With C(w) = #{b : mt_b >= w}:
//   pos = Hkv sum_{w' > w} C(w') + Hkv (C(w) - C(mt_b) + eq_b) + j,
// eq_b = #{b' < b : mt_b' = mt_b}.  Lengths outside [0, T] are clamped and
// recorded in the status word.  Packed batches (cu_in set): the prefix
// array is made monotone within [0, T = total] (starting at 0, ending at
// total; any change recorded) and written out, since the kernels address
// rows through it, and the lengths are its differences.
constexpr int kPlanThreads = 1024;

// Exclusive scan of one int per thread over the block; returns the block's
// total through *total.
__device__ int block_excl_scan(int x, int *warp_sums, int *total)
{
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = kPlanThreads / 32;
        int v = lane < nw ? warp_sums[lane] : 0;
        int w_incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w_incl, o);
            if (lane >= o)
                w_incl += y;
        }
        if (lane < nw)
            warp_sums[lane] = w_incl - v;   // exclusive
        if (lane == nw - 1)
            *total = w_incl;
    }
    __syncthreads();
    const int r = warp_sums[warp] + incl - x;
    __syncthreads();   // warp_sums is reused by the next call
    return r;
}

__global__ void __launch_bounds__(kPlanThreads, 1) varlen_plan_kernel(const DevicePlanParams p)
{
    __shared__ int warp_sums[kPlanThreads / 32];
    __shared__ int total_s;
    const int tid = threadIdx.x;
    const int M = p.M;
    int *mt = p.scratch;                  // [B]
    int *eq = mt + p.B;                   // [B]
    int *cge = eq + p.B;                  // [M + 2]: C(w)
    int *start = cge + (M + 2);           // [M + 2]: Hkv sum_{w' > w} C(w')
    griddep_wait();
    // lengths (clamped), tiles, and the histogram of tiles (into cge)
    for (int i = tid; i < M + 2; i += kPlanThreads)
        cge[i] = 0;
    if (p.cu_in != nullptr && tid == 0) {
        // one pass: the running maximum, clipped to the pack
        bool bad = p.cu_in[0] != 0 || p.cu_in[p.B] != p.T;
        int prev = 0;
        p.cu_out[0] = 0;
        for (int b = 1; b <= p.B; ++b) {
            int c = p.cu_in[b];
            bad = bad || c < prev;
            c = c < prev ? prev : (c > p.T ? p.T : c);
            if (b == p.B)
                c = p.T;
            p.cu_out[b] = c;
            prev = c;
        }
        if (bad)
            atomicOr(p.status, kDevArg);
    }
    __syncthreads();
    for (int b = tid; b < p.B; b += kPlanThreads) {
        int L;
        if (p.cu_in != nullptr) {
            L = p.cu_out[b + 1] - p.cu_out[b];
        } else {
            L = p.seqlens_in[b];
            if (L < 0 || L > p.T) {
                atomicOr(p.status, kDevArg);
                L = L < 0 ? 0 : p.T;
            }
        }
        p.seqlen_out[b] = L;
        mt[b] = (L + kRows - 1) / kRows;
        if (mt[b] > M) {   // a packed length above the tile bound cannot occur
            atomicOr(p.status, kDevArg);
            mt[b] = M;
        }
        atomicAdd(cge + mt[b], 1);
    }
    __syncthreads();
    // eq_b: earlier sequences with as many tiles
    for (int b = tid; b < p.B; b += kPlanThreads) {
        int c = 0;
        for (int b2 = 0; b2 < b; ++b2)
            c += mt[b2] == mt[b] ? 1 : 0;
        eq[b] = c;
    }
    // C(w) = sum_{L >= w} hist(L): a suffix scan (reversed exclusive scan
    // plus the element), slice by slice from the top
    {
        int carry = 0;
        for (int i0 = 0; i0 < M + 2; i0 += kPlanThreads) {
            const int w = M + 1 - (i0 + tid);           // descending
            const int h = w >= 0 ? cge[w] : 0;
            const int ex = block_excl_scan(h, warp_sums, &total_s);
            if (w >= 0)
                cge[w] = carry + ex + h;
            carry += total_s;
            __syncthreads();
        }
    }
    __syncthreads();
    // start(w) = Hkv sum_{w' > w, w' >= 1} C(w') (works 1..M)
    {
        int carry = 0;
        for (int i0 = 0; i0 < M + 2; i0 += kPlanThreads) {
            const int w = M + 1 - (i0 + tid);
            const int c = (w >= 1 && w <= M) ? cge[w] : 0;
            const int ex = block_excl_scan(c, warp_sums, &total_s);
            if (w >= 0)
                start[w] = p.Hkv * (carry + ex);
            carry += total_s;
            __syncthreads();
        }
        if (tid == 0)
            p.counts[2] = p.Hkv * carry;
    }
    __syncthreads();
    // forward and dq tables: the live units in enumeration order
    for (int k = 0; k < 2; ++k) {
        const int nch = k == 0 ? p.nch_fwd : p.nch_dq;
        int *table = k == 0 ? p.fwd_units : p.dq_units;
        const long long per_m = static_cast<long long>(p.B) * p.Hkv * nch;
        const long long n = per_m * M;
        int base = 0;
        for (long long i0 = 0; i0 < n; i0 += kPlanThreads) {
            const long long u = i0 + tid;
            bool live = false;
            if (u < n) {
                const int m = M - 1 - static_cast<int>(u / per_m);
                const int b = static_cast<int>((u % per_m) / nch / p.Hkv);
                live = m < mt[b];
            }
            const int ex = block_excl_scan(live ? 1 : 0, warp_sums, &total_s);
            if (live)
                table[base + ex] = static_cast<int>(u);
            base += total_s;
            __syncthreads();
        }
        if (tid == 0)
            p.counts[k] = base;
    }
    // dk/dv table: each live unit straight to its position
    const long long per_n = static_cast<long long>(p.B) * p.Hkv;
    for (long long u = tid; u < per_n * M; u += kPlanThreads) {
        const int n = static_cast<int>(u / per_n);
        const int b = static_cast<int>((u % per_n) / p.Hkv);
        const int j = static_cast<int>(u % p.Hkv);
        if (n < mt[b]) {
            const int w = mt[b] - n;
            p.dkv_units[start[w] + p.Hkv * (cge[w] - cge[mt[b]] + eq[b]) + j] =
                static_cast<int>(u);
        }
    }
    griddep_launch_dependents();
}

cudaError_t launch_varlen_plan(const DevicePlanParams &p, cudaStream_t stream)
{
    return launch_pdl(varlen_plan_kernel, 1, kPlanThreads, 0, stream, p);
}

} // namespace ne
