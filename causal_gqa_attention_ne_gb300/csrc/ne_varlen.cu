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

} // namespace ne
