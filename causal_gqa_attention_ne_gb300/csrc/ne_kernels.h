// ne_kernels.h -- internal launchers of the attention kernels (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "ne_common.cuh"

namespace ne {

// Forward: persistent CTAs of 512 threads over M * B * Hkv * nchunks units;
// `o` is the tensor map of the output (same layout as q) with a box of
// kFwdOStoreRows rows: each softmax warp stores its own rows of a head.
// `qs` / `ks` map the fp16 Q' / K' regions of a backward workspace; they are
// written only when p.save_rot is set.
constexpr int kFwdOStoreRows = 32;
cudaError_t launch_fwd(int d, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                       const CUtensorMap &o, const CUtensorMap &qs, const CUtensorMap &ks,
                       const AttnParams &p, cudaStream_t stream);

// Backward preprocess: D[b][h][t] = sum_c dO[b,t,h,c] * O[b,t,h,c], and the
// rotated Q' = R(t) q, K' = R(s) k as fp16 (same layouts) into qrot / krot.
cudaError_t launch_bwd_pre(int d, const AttnParams &p, const void *q, void *qrot, const void *k,
                           void *krot, cudaStream_t stream);

// Backward dQ (query-tile major, recomputes S and dP); `dq` is the tensor
// map of the output (same layout as q) with a box of kDqStoreRows rows, used
// by its TMA stores (d <= 64): each row warp stores its own rows of a head.
constexpr int kDqStoreRows = 32;
cudaError_t launch_bwd_dq(int d, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                          const CUtensorMap &dO, const CUtensorMap &dq, const AttnParams &p,
                          cudaStream_t stream);

// Backward dK, dV (key-tile major; dK and dV summed over the query heads of
// each KV head inside the CTA).  `q` and `k` are the fp16 rotated Q' / K' maps.
cudaError_t launch_bwd_dkdv(int d, const CUtensorMap &q, const CUtensorMap &k,
                            const CUtensorMap &v, const CUtensorMap &dO, const AttnParams &p,
                            cudaStream_t stream);

// Heads per CTA the Q-major kernels support for head dim d and group size G.
int fwd_heads_per_cta(int d, int G);
int dq_heads_per_cta(int d, int G);

// Decode against a key/value cache: one query row per (b, h) at position
// Tk - 1 over Tk cached keys.  Split over chunks of decode_chunk_keys() keys;
// part_o [B][Hq][nchunks][d] and part_ml [B][Hq][nchunks][2] (fp32) hold the
// chunks' partial results, merged by a second kernel into o and lse.
constexpr int kMaxDecodeGroup = 16;   // query heads per key/value head
struct DecodeParams {
    int B, Tk, Hq, Hkv, G, nchunks;
    float scale_log2;
    const void *q, *k, *v;
    void *o;
    float *lse;
    float *part_o, *part_ml;
    uint32_t *status;          // device status word (bounded waits)
    uint64_t wait_limit_ns;
    RopeFreqs rope;
};
// `k`, `v`: 4-D tensor maps of the caches (the layout of the training
// kernels' k and v maps, T = Tk).
cudaError_t launch_decode(int d, const CUtensorMap &k, const CUtensorMap &v,
                          const DecodeParams &p, cudaStream_t stream);
int decode_chunk_keys();

// Padded variable-length batches.  varlen_plan lists the live work units of
// the forward, dq and dk/dv kernels for per-sequence lengths seqlen[B] (host
// array, 0 <= seqlen[b] <= T) as indices into each kernel's full unit
// enumeration, writing at most caps[i] entries into table i (a null table is
// only counted) and the three counts; the kernels take a table through
// AttnParams::units with num_units = its count.  launch_pad_fill writes the
// padding rows t >= seqlen[b]: zero in up to three [B][T][row_bytes] tensors
// (row_bytes a multiple of 16, 16-byte aligned bases) and -inf in lse
// [B][Hq][T] when lse is not null.  seqlen is a device array there.
struct PadFillParams {
    void *x[3];
    int row_bytes[3];
    int ntensors;
    float *lse;
    int B, T, Hq;
    const int *seqlen;
};
int varlen_plan(const int *seqlen, int B, int T, int Hq, int Hkv, int d, int *fwd_units,
                int *dq_units, int *dkv_units, const size_t caps[3], int counts[3]);
// Device-side plan of a padded variable-length batch: the tables of
// varlen_plan (forward, dq, dk/dv, same contents and order) and the three
// counts, from lengths in device memory, clamped to [0, T] (kDevArg recorded
// for a length outside), copied to seqlen_out; or from a packed batch's
// prefix array (sanitised into cu_out).  M: the tiles of the enumeration.
// scratch holds 2 B + 2 (M + 2) ints.
struct DevicePlanParams {
    const int *seqlens_in;      // padded: lengths [B]
    const int *cu_in;           // packed: prefix array [B + 1] (seqlens_in unused)
    int *seqlen_out, *cu_out, *fwd_units, *dq_units, *dkv_units, *counts, *scratch;
    int B, T, M, Hkv, nch_fwd, nch_dq;   // packed: B = sequences, T = total rows
    uint32_t *status;
};
cudaError_t launch_varlen_plan(const DevicePlanParams &p, cudaStream_t stream);
cudaError_t launch_pad_fill(const PadFillParams &p, cudaStream_t stream);

// One-block kernel whose wait can never complete (checks the timeout path).
cudaError_t launch_timeout_selftest(uint32_t *status, uint64_t limit_ns, cudaStream_t stream);

} // namespace ne
