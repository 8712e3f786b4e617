// ne_api.cu -- the C ABI of include/ne_attn.h: argument validation, TMA
// descriptor construction, launch sequencing and the device status word.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ne_attn.h"
#include "ne_common.cuh"
#include "ne_kernels.h"

namespace {

// One status word per device (module-scope device variable): bounded waits
// that run out and fp16 range overflows are OR-ed into it by the kernels.
__device__ uint32_t g_status_word;

// Bound on device-side waits for launches made by this host thread (each
// thread has its own value, so a thread changing it never affects another
// thread's launches).
thread_local uint64_t g_wait_limit_ns = 2000000000ull;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;

constexpr int kMaxDevices = 64;
struct DeviceState {
    bool probed = false;
    bool supported = false;
    uint32_t *status = nullptr;
};
DeviceState g_dev[kMaxDevices];

EncodeTiledFn encode_fn()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

// Returns NE_OK and the device's status-word address, or an error status.
int device_state(uint32_t **status)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return NE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &s = g_dev[dev];
    if (!s.probed) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return NE_ERR_CUDA;
        s.supported = (major == 10 && minor == 3);
        if (s.supported) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess)
                return NE_ERR_CUDA;
            s.status = static_cast<uint32_t *>(p);
        }
        s.probed = true;
    }
    if (!s.supported)
        return NE_ERR_UNSUPPORTED;
    *status = s.status;
    return NE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_shape(int B, int T, int Hq, int Hkv, int d, float theta)
{
    if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
        return NE_ERR_SHAPE;
    if (d != 32 && d != 64 && d != 128)
        return NE_ERR_UNSUPPORTED;
    if (!(theta > 0.f) || !std::isfinite(theta))
        return NE_ERR_ARG;
    // Grid sizes and 32-bit row positions must not overflow.
    const long long M = (T + 127) / 128;
    if (T > (1 << 24) || M * B * Hq > 0x7fffffffLL)
        return NE_ERR_SHAPE;
    return NE_OK;
}

// 4-D TMA descriptor over a contiguous [B][T][H][d] 16-bit tensor; box is
// (one swizzle span of columns, 1 head, 128 rows, 1 batch).
int make_map(CUtensorMap *m, const void *ptr, int B, int T, int H, int d, bool fp16 = false,
             int box_rows = 128)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return NE_ERR_CUDA;
    const int swb = (2 * d < 128) ? 2 * d : 128;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2,
                             static_cast<cuuint64_t>(T) * H * d * 2};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(swb / 2), 1, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     4, const_cast<void *>(ptr), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NE_OK : NE_ERR_CUDA;
}

// Fixed-point RoPE frequencies: F_i = round(2^64 * theta^(-2i/d) / (2 pi))
// mod 2^64 as two 32-bit words.  The fraction f (in [0, 1)) is a double, so
// F_i carries its 53 significant bits: an error below 2^-54 turn per
// position, 2^-30 turn at position 2^24.  Scaling by 2^32 and taking the
// integer part are exact in double arithmetic.
void fill_rope(ne::RopeFreqs &fr, int d, float theta)
{
    std::memset(&fr, 0, sizeof(fr));
    const double two_pi = 6.283185307179586476925286766559;
    for (int i = 0; i < d / 2; ++i) {
        double f = std::pow(static_cast<double>(theta), -2.0 * i / d) / two_pi;
        f -= std::floor(f);
        const double top = std::floor(f * 4294967296.0);          // high word
        const double rest = f * 4294967296.0 - top;               // in [0, 1)
        unsigned long long hi = static_cast<unsigned long long>(top);
        unsigned long long lo = static_cast<unsigned long long>(std::llround(rest * 4294967296.0));
        if (lo > 0xffffffffull) {   // rounded up to the next high word
            lo = 0;
            ++hi;
        }
        fr.hi[i] = static_cast<uint32_t>(hi & 0xffffffffull);
        fr.lo[i] = static_cast<uint32_t>(lo);
    }
}

// Backward workspace: [D: fp32 B*Hq*T][Q': fp16 B*T*Hq*d][K': fp16 B*T*Hkv*d],
// each 256-aligned.
size_t ws_d_bytes(int B, int T, int Hq)
{
    return ((static_cast<size_t>(B) * Hq * T * sizeof(float)) + 255) & ~static_cast<size_t>(255);
}
size_t ws_q_bytes(int B, int T, int Hq, int d)
{
    return ((static_cast<size_t>(B) * T * Hq * d * 2) + 255) & ~static_cast<size_t>(255);
}

ne::AttnParams base_params(int B, int T, int Hq, int Hkv, int d, float theta, uint32_t *status)
{
    ne::AttnParams p;
    std::memset(&p, 0, sizeof(p));
    p.B = B;
    p.T = T;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.M = (T + 127) / 128;
    p.scale = 1.0f / std::sqrt(static_cast<float>(d));
    p.scale_log2 = p.scale * 1.4426950408889634f;
    p.status = status;
    p.wait_limit_ns = g_wait_limit_ns;
    fill_rope(p.rope, d, theta);
    return p;
}

int largest_divisor_at_most(int G, int cap)
{
    for (int g = cap; g >= 1; --g)
        if (G % g == 0)
            return g;
    return 1;
}

__global__ void timeout_selftest_kernel(uint32_t *status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        ne::mbar_init(ne::smem_u32(&bar), 1);
        ne::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const ne::WaitCtl wc{&abort_flag, status, limit_ns};
        // Nothing ever arrives on `bar`: this wait can only end by its limit.
        ne::mbar_wait(ne::smem_u32(&bar), 0, wc);
    }
}

} // namespace

namespace ne {

int fwd_heads_per_cta(int d, int G) { return largest_divisor_at_most(G, d == 32 ? 4 : d == 64 ? 3 : 2); }
int dq_heads_per_cta(int d, int G)
{
    return d == 128 ? 1 : largest_divisor_at_most(G, d == 64 ? 3 : 4);
}

cudaError_t launch_timeout_selftest(uint32_t *status, uint64_t limit_ns, cudaStream_t stream)
{
    timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

} // namespace ne

namespace {

// The forward; with a workspace it also stores the rotated Q' and K' (fp16)
// into the workspace's Q' and K' regions for ne_attn_bwd_saved.
int fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse, void *workspace,
             size_t workspace_bytes, bool save, int B, int T, int Hq, int Hkv, int d,
             float rope_theta, void *stream, int window = 0)
{
    if (!q || !k || !v || !o || !lse || (save && !workspace))
        return NE_ERR_NULL;
    int rc = check_shape(B, T, Hq, Hkv, d, rope_theta);
    if (rc != NE_OK)
        return rc;
    if (window < 0)
        return NE_ERR_ARG;
    if (save && workspace_bytes < ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d))
        return NE_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
        (save && !aligned16(workspace)))
        return NE_ERR_ALIGN;
    uint32_t *status = nullptr;
    if ((rc = device_state(&status)) != NE_OK)
        return rc;
    ne::AttnParams p = base_params(B, T, Hq, Hkv, d, rope_theta, status);
    p.GC = ne::fwd_heads_per_cta(d, p.G);
    p.nchunks = p.G / p.GC;
    p.out0 = o;
    p.lse = lse;
    p.q_in = q;
    p.k_in = k;
    p.v_in = v;
    p.save_rot = save ? 1 : 0;
    p.window = window;
    CUtensorMap mq, mk, mv, mo, mqs, mks;
    if (make_map(&mq, q, B, T, Hq, d) || make_map(&mk, k, B, T, Hkv, d) ||
        make_map(&mv, v, B, T, Hkv, d) ||
        make_map(&mo, o, B, T, Hq, d, false, ne::kFwdOStoreRows))
        return NE_ERR_CUDA;
    if (save) {
        void *qrot = static_cast<uint8_t *>(workspace) + ws_d_bytes(B, T, Hq);
        void *krot = static_cast<uint8_t *>(qrot) + ws_q_bytes(B, T, Hq, d);
        if (make_map(&mqs, qrot, B, T, Hq, d, true) || make_map(&mks, krot, B, T, Hkv, d, true))
            return NE_ERR_CUDA;
    } else {
        mqs = mq;   // not used
        mks = mk;
    }
    cudaError_t e =
        ne::launch_fwd(d, mq, mk, mv, mo, mqs, mks, p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

} // namespace

extern "C" {

int ne_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int T,
                int Hq, int Hkv, int d, float rope_theta, void *stream)
{
    return fwd_impl(q, k, v, o, lse, nullptr, 0, false, B, T, Hq, Hkv, d, rope_theta, stream);
}

int ne_attn_fwd_save(const void *q, const void *k, const void *v, void *o, float *lse,
                     void *workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                     float rope_theta, int window, void *stream)
{
    return fwd_impl(q, k, v, o, lse, workspace, workspace_bytes, true, B, T, Hq, Hkv, d,
                    rope_theta, stream, window);
}

size_t ne_attn_bwd_workspace_size(int B, int T, int Hq, int Hkv, int d)
{
    if (check_shape(B, T, Hq, Hkv, d, 1.0f) != NE_OK)
        return 0;
    return ws_d_bytes(B, T, Hq) + ws_q_bytes(B, T, Hq, d) + ws_q_bytes(B, T, Hkv, d);
}

int ne_attn_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                       int T, int Hq, int Hkv, int d, float rope_theta, int window, void *stream)
{
    return fwd_impl(q, k, v, o, lse, nullptr, 0, false, B, T, Hq, Hkv, d, rope_theta, stream,
                    window);
}

} // extern "C"

namespace {

// Validation shared by the backward entry points; fills the common params.
int bwd_setup(const void *q, const void *k, const void *v, const float *lse, const void *dO,
              void *workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
              float rope_theta, ne::AttnParams *p, CUtensorMap *mq, CUtensorMap *mk,
              CUtensorMap *mv, CUtensorMap *mdo, CUtensorMap *mqr, CUtensorMap *mkr)
{
    if (!q || !k || !v || !lse || !dO)
        return NE_ERR_NULL;
    int rc = check_shape(B, T, Hq, Hkv, d, rope_theta);
    if (rc != NE_OK)
        return rc;
    if (!workspace || workspace_bytes < ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d))
        return NE_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned4(lse) ||
        !aligned16(workspace))
        return NE_ERR_ALIGN;
    uint32_t *status = nullptr;
    if ((rc = device_state(&status)) != NE_OK)
        return rc;
    *p = base_params(B, T, Hq, Hkv, d, rope_theta, status);
    p->do_in = dO;
    p->lse = const_cast<float *>(lse);
    p->Dws = static_cast<float *>(workspace);
    void *qrot = static_cast<uint8_t *>(workspace) + ws_d_bytes(B, T, Hq);
    void *krot = static_cast<uint8_t *>(qrot) + ws_q_bytes(B, T, Hq, d);
    if (make_map(mq, q, B, T, Hq, d) || make_map(mk, k, B, T, Hkv, d) ||
        make_map(mv, v, B, T, Hkv, d) || make_map(mdo, dO, B, T, Hq, d) ||
        make_map(mqr, qrot, B, T, Hq, d, true) || make_map(mkr, krot, B, T, Hkv, d, true))
        return NE_ERR_CUDA;
    return NE_OK;
}

int run_dq(int d, const ne::AttnParams &base, void *dq, const CUtensorMap &mq,
           const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mdo, cudaStream_t st)
{
    ne::AttnParams p = base;
    p.GC = ne::dq_heads_per_cta(d, p.G);
    p.nchunks = p.G / p.GC;
    p.out0 = dq;
    CUtensorMap mdq;
    // packed batches: one batch entry in memory (p.B counts the sequences)
    if (make_map(&mdq, dq, p.cu != nullptr ? 1 : p.B, p.T, p.Hq, d, false, ne::kDqStoreRows))
        return NE_ERR_CUDA;
    return ne::launch_bwd_dq(d, mq, mk, mv, mdo, mdq, p, st) == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

int run_dkdv(int d, const ne::AttnParams &base, void *dk, void *dv, const CUtensorMap &mq,
             const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mdo,
             cudaStream_t st)
{
    ne::AttnParams p = base;
    p.out0 = dk;
    p.out1 = dv;
    return ne::launch_bwd_dkdv(d, mq, mk, mv, mdo, p, st) == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

} // namespace

extern "C" {

int ne_attn_bwd_preprocess(const void *q, const void *k, const void *o, const void *dO,
                           void *workspace, size_t workspace_bytes, int B, int T, int Hq,
                           int Hkv, int d, float rope_theta, void *stream)
{
    if (!q || !k || !o || !dO)
        return NE_ERR_NULL;
    int rc = check_shape(B, T, Hq, Hkv, d, rope_theta);
    if (rc != NE_OK)
        return rc;
    if (!workspace || workspace_bytes < ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d))
        return NE_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(o) || !aligned16(dO) ||
        !aligned16(workspace))
        return NE_ERR_ALIGN;
    uint32_t *status = nullptr;
    if ((rc = device_state(&status)) != NE_OK)
        return rc;
    ne::AttnParams p = base_params(B, T, Hq, Hkv, d, rope_theta, status);
    p.o_in = o;
    p.do_in = dO;
    p.Dws = static_cast<float *>(workspace);
    void *qrot = static_cast<uint8_t *>(workspace) + ws_d_bytes(B, T, Hq);
    void *krot = static_cast<uint8_t *>(qrot) + ws_q_bytes(B, T, Hq, d);
    return ne::launch_bwd_pre(d, p, q, qrot, k, krot, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? NE_OK
               : NE_ERR_CUDA;
}

int ne_attn_bwd_preprocess_d(const void *o, const void *dO, void *workspace,
                             size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                             void *stream)
{
    if (!o || !dO)
        return NE_ERR_NULL;
    int rc = check_shape(B, T, Hq, Hkv, d, 1.0f);
    if (rc != NE_OK)
        return rc;
    if (!workspace || workspace_bytes < ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d))
        return NE_ERR_WORKSPACE;
    if (!aligned16(o) || !aligned16(dO) || !aligned16(workspace))
        return NE_ERR_ALIGN;
    uint32_t *status = nullptr;
    if ((rc = device_state(&status)) != NE_OK)
        return rc;
    ne::AttnParams p = base_params(B, T, Hq, Hkv, d, 1.0f, status);
    p.o_in = o;
    p.do_in = dO;
    p.Dws = static_cast<float *>(workspace);
    return ne::launch_bwd_pre(d, p, nullptr, nullptr, nullptr, nullptr,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? NE_OK
               : NE_ERR_CUDA;
}

int ne_attn_bwd_dq(const void *q, const void *k, const void *v, const float *lse,
                   const void *dO, void *dq, const void *workspace, size_t workspace_bytes,
                   int B, int T, int Hq, int Hkv, int d, float rope_theta, void *stream)
{
    if (!dq)
        return NE_ERR_NULL;
    if (!aligned16(dq))
        return NE_ERR_ALIGN;
    ne::AttnParams p;
    CUtensorMap mq, mk, mv, mdo, mqr, mkr;
    int rc = bwd_setup(q, k, v, lse, dO, const_cast<void *>(workspace), workspace_bytes, B, T,
                       Hq, Hkv, d, rope_theta, &p, &mq, &mk, &mv, &mdo, &mqr, &mkr);
    if (rc != NE_OK)
        return rc;
    return run_dq(d, p, dq, mqr, mkr, mv, mdo, static_cast<cudaStream_t>(stream));
}

int ne_attn_bwd_dkdv(const void *q, const void *k, const void *v, const float *lse,
                     const void *dO, void *dk, void *dv, const void *workspace,
                     size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                     float rope_theta, void *stream)
{
    if (!dk || !dv)
        return NE_ERR_NULL;
    if (!aligned16(dk) || !aligned16(dv))
        return NE_ERR_ALIGN;
    ne::AttnParams p;
    CUtensorMap mq, mk, mv, mdo, mqr, mkr;
    int rc = bwd_setup(q, k, v, lse, dO, const_cast<void *>(workspace), workspace_bytes, B, T,
                       Hq, Hkv, d, rope_theta, &p, &mq, &mk, &mv, &mdo, &mqr, &mkr);
    if (rc != NE_OK)
        return rc;
    return run_dkdv(d, p, dk, dv, mqr, mkr, mv, mdo, static_cast<cudaStream_t>(stream));
}

int ne_attn_bwd_window(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dO, void *dq, void *dk, void *dv,
                       void *workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv,
                       int d, float rope_theta, int window, void *stream);

int ne_attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                const void *dO, void *dq, void *dk, void *dv, void *workspace,
                size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d, float rope_theta,
                void *stream)
{
    return ne_attn_bwd_window(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, T,
                              Hq, Hkv, d, rope_theta, 0, stream);
}

int ne_attn_bwd_window(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dO, void *dq, void *dk, void *dv,
                       void *workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv,
                       int d, float rope_theta, int window, void *stream)
{
    if (window < 0)
        return NE_ERR_ARG;
    if (!o || !dq || !dk || !dv)
        return NE_ERR_NULL;
    if (!aligned16(o) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return NE_ERR_ALIGN;
    ne::AttnParams p;
    CUtensorMap mq, mk, mv, mdo, mqr, mkr;
    int rc = bwd_setup(q, k, v, lse, dO, workspace, workspace_bytes, B, T, Hq, Hkv, d,
                       rope_theta, &p, &mq, &mk, &mv, &mdo, &mqr, &mkr);
    if (rc != NE_OK)
        return rc;
    p.window = window;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    p.o_in = o;
    void *qrot = static_cast<uint8_t *>(workspace) + ws_d_bytes(B, T, Hq);
    void *krot = static_cast<uint8_t *>(qrot) + ws_q_bytes(B, T, Hq, d);
    if (ne::launch_bwd_pre(d, p, q, qrot, k, krot, st) != cudaSuccess)
        return NE_ERR_CUDA;
    if ((rc = run_dq(d, p, dq, mqr, mkr, mv, mdo, st)) != NE_OK)
        return rc;
    return run_dkdv(d, p, dk, dv, mqr, mkr, mv, mdo, st);
}

int ne_attn_bwd_saved(const void *q, const void *k, const void *v, const void *o,
                      const float *lse, const void *dO, void *dq, void *dk, void *dv,
                      void *workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv,
                      int d, float rope_theta, int window, void *stream)
{
    if (window < 0)
        return NE_ERR_ARG;
    if (!o || !dq || !dk || !dv)
        return NE_ERR_NULL;
    if (!aligned16(o) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return NE_ERR_ALIGN;
    ne::AttnParams p;
    CUtensorMap mq, mk, mv, mdo, mqr, mkr;
    int rc = bwd_setup(q, k, v, lse, dO, workspace, workspace_bytes, B, T, Hq, Hkv, d,
                       rope_theta, &p, &mq, &mk, &mv, &mdo, &mqr, &mkr);
    if (rc != NE_OK)
        return rc;
    p.window = window;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    p.o_in = o;
    // Q' and K' are already in the workspace: the preprocess computes D only
    if (ne::launch_bwd_pre(d, p, q, nullptr, k, nullptr, st) != cudaSuccess)
        return NE_ERR_CUDA;
    if ((rc = run_dq(d, p, dq, mqr, mkr, mv, mdo, st)) != NE_OK)
        return rc;
    return run_dkdv(d, p, dk, dv, mqr, mkr, mv, mdo, st);
}

size_t ne_attn_decode_workspace_size(int B, int Tk, int Hq, int Hkv, int d)
{
    if (check_shape(B, Tk, Hq, Hkv, d, 1.0f) != NE_OK)
        return 0;
    const size_t nchunks = (static_cast<size_t>(Tk) + ne::decode_chunk_keys() - 1) /
                           ne::decode_chunk_keys();
    const size_t rows = static_cast<size_t>(B) * Hq * nchunks;
    const size_t part_o = (rows * d * sizeof(float) + 255) & ~static_cast<size_t>(255);
    const size_t part_ml = (rows * 2 * sizeof(float) + 255) & ~static_cast<size_t>(255);
    return part_o + part_ml;
}

int ne_attn_decode(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                   void *workspace, size_t workspace_bytes, int B, int Tk, int Hq, int Hkv, int d,
                   float rope_theta, void *stream)
{
    if (!q || !k_cache || !v_cache || !o || !lse)
        return NE_ERR_NULL;
    int rc = check_shape(B, Tk, Hq, Hkv, d, rope_theta);
    if (rc != NE_OK)
        return rc;
    if (Hq / Hkv > ne::kMaxDecodeGroup)
        return NE_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < ne_attn_decode_workspace_size(B, Tk, Hq, Hkv, d))
        return NE_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
        !aligned4(lse) || !aligned16(workspace))
        return NE_ERR_ALIGN;
    uint32_t *status = nullptr;
    if ((rc = device_state(&status)) != NE_OK)
        return rc;
    ne::DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.B = B;
    p.Tk = Tk;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.nchunks = (Tk + ne::decode_chunk_keys() - 1) / ne::decode_chunk_keys();
    p.scale_log2 = 1.4426950408889634f / std::sqrt(static_cast<float>(d));
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.o = o;
    p.lse = lse;
    const size_t rows = static_cast<size_t>(B) * Hq * p.nchunks;
    p.part_o = static_cast<float *>(workspace);
    p.part_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                          ((rows * d * sizeof(float) + 255) &
                                           ~static_cast<size_t>(255)));
    p.status = status;
    p.wait_limit_ns = g_wait_limit_ns;
    fill_rope(p.rope, d, rope_theta);
    CUtensorMap mk, mv;
    if (make_map(&mk, k_cache, B, Tk, Hkv, d) || make_map(&mv, v_cache, B, Tk, Hkv, d))
        return NE_ERR_CUDA;
    return ne::launch_decode(d, mk, mv, p, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? NE_OK
               : NE_ERR_CUDA;
}

int ne_attn_get_error(void *stream)
{
    uint32_t *status = nullptr;
    int rc = device_state(&status);
    if (rc != NE_OK)
        return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return NE_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)) != cudaSuccess)
        return NE_ERR_CUDA;
    if (word) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
            return NE_ERR_CUDA;
    }
    if (word & ne::kDevTimeout)
        return NE_ERR_TIMEOUT;
    if (word & ne::kDevRange)
        return NE_ERR_RANGE;
    if (word & ne::kDevArg)
        return NE_ERR_ARG;
    if (word & ne::kDevPrecision)
        return NE_WARN_PRECISION;
    return NE_OK;
}

const char *ne_attn_status_string(int status)
{
    switch (status) {
    case NE_OK: return "ok";
    case NE_ERR_NULL: return "a required pointer is NULL";
    case NE_ERR_SHAPE: return "invalid shape (B, T, Hq, Hkv) or Hq % Hkv != 0";
    case NE_ERR_UNSUPPORTED: return "unsupported head dim or device (needs d in {32,64,128}, sm_103)";
    case NE_ERR_ALIGN: return "pointer misaligned (tensors need 16 bytes, lse 4 bytes)";
    case NE_ERR_WORKSPACE: return "workspace missing or too small";
    case NE_ERR_CUDA: return "CUDA call or kernel launch failed";
    case NE_ERR_TIMEOUT: return "a device-side bounded wait ran out";
    case NE_ERR_RANGE: return "an fp16 tensor-core operand exceeded 65504";
    case NE_ERR_ARG:
        return "invalid argument (rope_theta must be finite and > 0; a window, sequence length "
               "or cu_seqlens out of range)";
    case NE_ERR_TOO_LARGE:
        return "shape needs more scratch than ne_attn_bwd_noalloc's fixed buffer holds";
    case NE_WARN_PRECISION:
        return "a CTA of the forward met more large-norm rows than it repairs";
    default: return "unknown status";
    }
}

void ne_attn_set_wait_limit_ns(uint64_t limit_ns)
{
    g_wait_limit_ns = limit_ns ? limit_ns : 1;
}

int ne_attn_selftest_timeout(uint64_t limit_ns, void *stream)
{
    uint32_t *status = nullptr;
    int rc = device_state(&status);
    if (rc != NE_OK)
        return rc;
    cudaError_t e = ne::launch_timeout_selftest(status, limit_ns ? limit_ns : 1,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

} // extern "C"

// ------------------------------------------------------------------------
// Padded variable-length batches.  Workspace: the unit tables [seqlen: int32
// B][forward units][dq units][dk/dv units], each region 256-byte aligned and
// sized for every unit of the padded shape, then the device-side plan's
// counts (int32 [4]) and scratch (int32 [2 B + 2 (M + 2)]), then (backward)
// the backward workspace of ne_attn_bwd.
namespace {

struct VarlenLayout {
    size_t off_fwd, off_dq, off_dkv, off_cnt, off_scr, tables, total;
};

VarlenLayout varlen_layout(int B, int T, int Hq, int Hkv, int d)
{
    auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const int G = Hq / Hkv;
    const size_t tiles = static_cast<size_t>((T + 127) / 128) * B * Hkv;
    const size_t nf = tiles * static_cast<size_t>(G / ne::fwd_heads_per_cta(d, G));
    const size_t nq = tiles * static_cast<size_t>(G / ne::dq_heads_per_cta(d, G));
    VarlenLayout L;
    L.off_fwd = al(sizeof(int32_t) * static_cast<size_t>(B));
    L.off_dq = L.off_fwd + al(sizeof(int32_t) * nf);
    L.off_dkv = L.off_dq + al(sizeof(int32_t) * nq);
    L.off_cnt = L.off_dkv + al(sizeof(int32_t) * tiles);
    L.off_scr = L.off_cnt + al(sizeof(int32_t) * 4);
    const size_t M = static_cast<size_t>((T + 127) / 128);
    L.tables = L.off_scr + al(sizeof(int32_t) * (2 * static_cast<size_t>(B) + 2 * (M + 2)));
    L.total = L.tables + ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d);
    return L;
}

int check_seqlens(const int32_t *seqlens, int B, int T)
{
    if (!seqlens)
        return NE_ERR_NULL;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > T)
            return NE_ERR_ARG;
    return NE_OK;
}

// The workspace's table region as the host builds it: the lengths, then each
// table at its offset, filled up to its own region's capacity.
int build_table_image(const int32_t *seqlens, int B, int T, int Hq, int Hkv, int d,
                      const VarlenLayout &L, std::vector<int32_t> &img, int counts[3])
{
    const size_t w = sizeof(int32_t);
    img.assign(L.tables / w, 0);
    std::memcpy(img.data(), seqlens, w * static_cast<size_t>(B));
    const size_t caps[3] = {(L.off_dq - L.off_fwd) / w, (L.off_dkv - L.off_dq) / w,
                            (L.tables - L.off_dkv) / w};
    ne::varlen_plan(seqlens, B, T, Hq, Hkv, d, img.data() + L.off_fwd / w,
                    img.data() + L.off_dq / w, img.data() + L.off_dkv / w, caps, counts);
    for (int i = 0; i < 3; ++i)
        if (static_cast<size_t>(counts[i]) > caps[i])
            return NE_ERR_ARG;   // cannot happen: every region holds all units of its kernel
    return NE_OK;
}

// Builds the table image and copies it into the workspace on `st`.  The copy
// is from pageable memory: it is staged before cudaMemcpyAsync returns, so
// the host buffer may go away afterwards.
int upload_tables(const int32_t *seqlens, int B, int T, int Hq, int Hkv, int d,
                  const VarlenLayout &L, void *workspace, cudaStream_t st, int counts[3])
{
    std::vector<int32_t> img;
    const int rc = build_table_image(seqlens, B, T, Hq, Hkv, d, L, img, counts);
    if (rc != NE_OK)
        return rc;
    return cudaMemcpyAsync(workspace, img.data(), L.tables, cudaMemcpyHostToDevice, st) ==
                   cudaSuccess
               ? NE_OK
               : NE_ERR_CUDA;
}

const int *ws_int(void *workspace, size_t off)
{
    return reinterpret_cast<const int *>(static_cast<uint8_t *>(workspace) + off);
}

// The plan kernel: the tables, counts and lengths of `seqlens` (device
// memory) into the workspace on `st`.
int plan_on_device(const int32_t *seqlens, int B, int T, int Hq, int Hkv, int d,
                   const VarlenLayout &L, void *workspace, uint32_t *status, cudaStream_t st)
{
    auto at = [&](size_t off) { return const_cast<int *>(ws_int(workspace, off)); };
    const int G = Hq / Hkv;
    ne::DevicePlanParams q;
    std::memset(&q, 0, sizeof(q));
    q.seqlens_in = seqlens;
    q.seqlen_out = at(0);
    q.fwd_units = at(L.off_fwd);
    q.dq_units = at(L.off_dq);
    q.dkv_units = at(L.off_dkv);
    q.counts = at(L.off_cnt);
    q.scratch = at(L.off_scr);
    q.B = B;
    q.T = T;
    q.M = (T + 127) / 128;
    q.Hkv = Hkv;
    q.nch_fwd = G / ne::fwd_heads_per_cta(d, G);
    q.nch_dq = G / ne::dq_heads_per_cta(d, G);
    q.status = status;
    return ne::launch_varlen_plan(q, st) == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

} // namespace

extern "C" {

size_t ne_attn_varlen_workspace_size(int B, int T, int Hq, int Hkv, int d)
{
    if (check_shape(B, T, Hq, Hkv, d, 1.0f) != NE_OK)
        return 0;
    return varlen_layout(B, T, Hq, Hkv, d).total;
}

int ne_attn_varlen_plan(const int32_t *seqlens, int B, int T, int Hq, int Hkv, int d,
                        int32_t *fwd_units, int32_t *dq_units, int32_t *dkv_units, size_t cap,
                        int32_t *counts)
{
    if (!counts)
        return NE_ERR_NULL;
    int rc = check_shape(B, T, Hq, Hkv, d, 1.0f);
    if (rc != NE_OK)
        return rc;
    if ((rc = check_seqlens(seqlens, B, T)) != NE_OK)
        return rc;
    // the very image the varlen entry points copy into the workspace
    const VarlenLayout L = varlen_layout(B, T, Hq, Hkv, d);
    std::vector<int32_t> img;
    int c[3];
    if ((rc = build_table_image(seqlens, B, T, Hq, Hkv, d, L, img, c)) != NE_OK)
        return rc;
    int32_t *out[3] = {fwd_units, dq_units, dkv_units};
    const size_t off[3] = {L.off_fwd, L.off_dq, L.off_dkv};
    for (int i = 0; i < 3; ++i) {
        counts[i] = c[i];
        if (out[i])
            std::memcpy(out[i], img.data() + off[i] / sizeof(int32_t),
                        sizeof(int32_t) * std::min(cap, static_cast<size_t>(c[i])));
    }
    return NE_OK;
}

} // extern "C"

namespace {

// The padded variable-length forward and backward.  With dev_lengths the
// lengths are in device memory and the plan kernel builds the tables (the
// calls can be captured into a graph); otherwise the host builds them from
// host lengths and copies them in.
int fwd_varlen_impl(const void *q, const void *k, const void *v, void *o, float *lse,
                    const int32_t *seqlens, bool dev_lengths, void *workspace,
                    size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                    float rope_theta, void *stream)
{
    if (!q || !k || !v || !o || !lse || !workspace)
        return NE_ERR_NULL;
    int rc = check_shape(B, T, Hq, Hkv, d, rope_theta);
    if (rc != NE_OK)
        return rc;
    // device lengths are checked by the plan kernel (NE_ERR_ARG through
    // ne_attn_get_error)
    if (dev_lengths && !seqlens)
        return NE_ERR_NULL;
    if (!dev_lengths && (rc = check_seqlens(seqlens, B, T)) != NE_OK)
        return rc;
    const VarlenLayout L = varlen_layout(B, T, Hq, Hkv, d);
    if (workspace_bytes < L.tables)
        return NE_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
        !aligned16(workspace) || (dev_lengths && !aligned4(seqlens)))
        return NE_ERR_ALIGN;
    uint32_t *status = nullptr;
    if ((rc = device_state(&status)) != NE_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ne::AttnParams p = base_params(B, T, Hq, Hkv, d, rope_theta, status);
    p.GC = ne::fwd_heads_per_cta(d, p.G);
    p.nchunks = p.G / p.GC;
    p.out0 = o;
    p.lse = lse;
    p.q_in = q;
    p.k_in = k;
    p.v_in = v;
    CUtensorMap mq, mk, mv, mo;
    if (make_map(&mq, q, B, T, Hq, d) || make_map(&mk, k, B, T, Hkv, d) ||
        make_map(&mv, v, B, T, Hkv, d) ||
        make_map(&mo, o, B, T, Hq, d, false, ne::kFwdOStoreRows))
        return NE_ERR_CUDA;
    int counts[3] = {1, 1, 1};
    if (dev_lengths)
        rc = plan_on_device(seqlens, B, T, Hq, Hkv, d, L, workspace, status, st);
    else
        rc = upload_tables(seqlens, B, T, Hq, Hkv, d, L, workspace, st, counts);
    if (rc != NE_OK)
        return rc;
    p.seqlen = ws_int(workspace, 0);
    p.units = ws_int(workspace, L.off_fwd);
    p.num_units = counts[0];
    if (dev_lengths)
        p.unit_count = ws_int(workspace, L.off_cnt);
    if (counts[0] > 0 && ne::launch_fwd(d, mq, mk, mv, mo, mq, mk, p, st) != cudaSuccess)
        return NE_ERR_CUDA;
    ne::PadFillParams f;
    std::memset(&f, 0, sizeof(f));
    f.x[0] = o;
    f.row_bytes[0] = Hq * d * 2;
    f.ntensors = 1;
    f.lse = lse;
    f.B = B;
    f.T = T;
    f.Hq = Hq;
    f.seqlen = p.seqlen;
    return ne::launch_pad_fill(f, st) == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

int bwd_varlen_impl(const void *q, const void *k, const void *v, const void *o,
                    const float *lse, const void *dO, void *dq, void *dk, void *dv,
                    const int32_t *seqlens, bool dev_lengths, void *workspace,
                    size_t workspace_bytes, int B, int T, int Hq, int Hkv, int d,
                    float rope_theta, void *stream)
{
    if (!o || !dq || !dk || !dv || !workspace)
        return NE_ERR_NULL;
    int rc = check_shape(B, T, Hq, Hkv, d, rope_theta);
    if (rc != NE_OK)
        return rc;
    if (dev_lengths && !seqlens)
        return NE_ERR_NULL;
    if (!dev_lengths && (rc = check_seqlens(seqlens, B, T)) != NE_OK)
        return rc;
    const VarlenLayout L = varlen_layout(B, T, Hq, Hkv, d);
    if (workspace_bytes < L.total)
        return NE_ERR_WORKSPACE;
    if (!aligned16(o) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        !aligned16(workspace) || (dev_lengths && !aligned4(seqlens)))
        return NE_ERR_ALIGN;
    void *bws = static_cast<uint8_t *>(workspace) + L.tables;
    ne::AttnParams p;
    CUtensorMap mq, mk, mv, mdo, mqr, mkr;
    rc = bwd_setup(q, k, v, lse, dO, bws, workspace_bytes - L.tables, B, T, Hq, Hkv, d,
                   rope_theta, &p, &mq, &mk, &mv, &mdo, &mqr, &mkr);
    if (rc != NE_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int counts[3] = {1, 1, 1};
    if (dev_lengths)
        rc = plan_on_device(seqlens, B, T, Hq, Hkv, d, L, workspace, p.status, st);
    else
        rc = upload_tables(seqlens, B, T, Hq, Hkv, d, L, workspace, st, counts);
    if (rc != NE_OK)
        return rc;
    p.o_in = o;
    // the lengths let the preprocess skip padding rows
    p.seqlen = ws_int(workspace, 0);
    void *qrot = static_cast<uint8_t *>(bws) + ws_d_bytes(B, T, Hq);
    void *krot = static_cast<uint8_t *>(qrot) + ws_q_bytes(B, T, Hq, d);
    if (ne::launch_bwd_pre(d, p, q, qrot, k, krot, st) != cudaSuccess)
        return NE_ERR_CUDA;
    p.units = ws_int(workspace, L.off_dq);
    p.num_units = counts[1];
    if (dev_lengths)
        p.unit_count = ws_int(workspace, L.off_cnt) + 1;
    if (counts[1] > 0 && (rc = run_dq(d, p, dq, mqr, mkr, mv, mdo, st)) != NE_OK)
        return rc;
    p.units = ws_int(workspace, L.off_dkv);
    p.num_units = counts[2];
    if (dev_lengths)
        p.unit_count = ws_int(workspace, L.off_cnt) + 2;
    if (counts[2] > 0 && (rc = run_dkdv(d, p, dk, dv, mqr, mkr, mv, mdo, st)) != NE_OK)
        return rc;
    ne::PadFillParams f;
    std::memset(&f, 0, sizeof(f));
    f.x[0] = dq;
    f.x[1] = dk;
    f.x[2] = dv;
    f.row_bytes[0] = Hq * d * 2;
    f.row_bytes[1] = Hkv * d * 2;
    f.row_bytes[2] = Hkv * d * 2;
    f.ntensors = 3;
    f.B = B;
    f.T = T;
    f.Hq = Hq;
    f.seqlen = p.seqlen;
    return ne::launch_pad_fill(f, st) == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

} // namespace

extern "C" {

int ne_attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                       const int32_t *seqlens, void *workspace, size_t workspace_bytes, int B,
                       int T, int Hq, int Hkv, int d, float rope_theta, void *stream)
{
    return fwd_varlen_impl(q, k, v, o, lse, seqlens, false, workspace, workspace_bytes, B, T, Hq,
                           Hkv, d, rope_theta, stream);
}

int ne_attn_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dO, void *dq, void *dk, void *dv,
                       const int32_t *seqlens, void *workspace, size_t workspace_bytes, int B,
                       int T, int Hq, int Hkv, int d, float rope_theta, void *stream)
{
    return bwd_varlen_impl(q, k, v, o, lse, dO, dq, dk, dv, seqlens, false, workspace,
                           workspace_bytes, B, T, Hq, Hkv, d, rope_theta, stream);
}

int ne_attn_fwd_varlen_dev(const void *q, const void *k, const void *v, void *o, float *lse,
                           const int32_t *seqlens_dev, void *workspace, size_t workspace_bytes,
                           int B, int T, int Hq, int Hkv, int d, float rope_theta, void *stream)
{
    return fwd_varlen_impl(q, k, v, o, lse, seqlens_dev, true, workspace, workspace_bytes, B, T,
                           Hq, Hkv, d, rope_theta, stream);
}

int ne_attn_bwd_varlen_dev(const void *q, const void *k, const void *v, const void *o,
                           const float *lse, const void *dO, void *dq, void *dk, void *dv,
                           const int32_t *seqlens_dev, void *workspace, size_t workspace_bytes,
                           int B, int T, int Hq, int Hkv, int d, float rope_theta, void *stream)
{
    return bwd_varlen_impl(q, k, v, o, lse, dO, dq, dk, dv, seqlens_dev, true, workspace,
                           workspace_bytes, B, T, Hq, Hkv, d, rope_theta, stream);
}

} // extern "C"

// ------------------------------------------------------------------------
// Packed variable-length batches: the sequences concatenated along the rows
// of one batch entry (q [total][Hq][d], lse [Hq][total]), sequence b at rows
// cu[b] .. cu[b+1]-1 with positions restarting at 0.  The kernels are the
// padded variable-length instantiations with the sequences' first rows
// (cu) added: a unit's TMA coordinates start at its sequence's first row,
// rows past the sequence inside its last tile are masked like padding and
// stored row by row, so a tile never writes the next sequence's rows.
// Workspace: [lengths int32 nseq][cu int32 nseq+1][forward units][dq
// units][dk/dv units][device-side plan: counts, scratch], each region
// 256-byte aligned, then (backward) the backward workspace of a [1][total]
// batch.
namespace {

struct PackedLayout {
    size_t off_cu, off_fwd, off_dq, off_dkv, off_cnt, off_scr, tables, total;
};

PackedLayout packed_layout(int nseq, int total, int Hq, int Hkv, int d)
{
    auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const int G = Hq / Hkv;
    // live tiles per KV head: sum over sequences of ceil(L_b / 128) is at
    // most floor(total / 128) + nseq
    const size_t tiles = (static_cast<size_t>(total) / 128 + nseq) * Hkv;
    const size_t nf = tiles * static_cast<size_t>(G / ne::fwd_heads_per_cta(d, G));
    const size_t nq = tiles * static_cast<size_t>(G / ne::dq_heads_per_cta(d, G));
    PackedLayout L;
    L.off_cu = al(sizeof(int32_t) * static_cast<size_t>(nseq));
    L.off_fwd = L.off_cu + al(sizeof(int32_t) * (static_cast<size_t>(nseq) + 1));
    L.off_dq = L.off_fwd + al(sizeof(int32_t) * nf);
    L.off_dkv = L.off_dq + al(sizeof(int32_t) * nq);
    // the device-side plan: counts, then scratch for M = ceil(total / 128)
    L.off_cnt = L.off_dkv + al(sizeof(int32_t) * tiles);
    L.off_scr = L.off_cnt + al(sizeof(int32_t) * 4);
    const size_t M = static_cast<size_t>((total + 127) / 128);
    L.tables = L.off_scr + al(sizeof(int32_t) * (2 * static_cast<size_t>(nseq) + 2 * (M + 2)));
    L.total = L.tables + ne_attn_bwd_workspace_size(1, total, Hq, Hkv, d);
    return L;
}

// Shape and cu_seqlens checks; on success *maxlen is the longest sequence.
int check_packed(const int32_t *cu, int nseq, int total, int Hq, int Hkv, int d, float theta,
                 int *maxlen)
{
    if (!cu)
        return NE_ERR_NULL;
    if (nseq < 1)
        return NE_ERR_SHAPE;
    int rc = check_shape(1, total, Hq, Hkv, d, theta);
    if (rc != NE_OK)
        return rc;
    if (cu[0] != 0 || cu[nseq] != total)
        return NE_ERR_ARG;
    int mx = 0;
    for (int b = 0; b < nseq; ++b) {
        if (cu[b + 1] < cu[b])
            return NE_ERR_ARG;
        mx = std::max(mx, cu[b + 1] - cu[b]);
    }
    if ((rc = check_shape(nseq, mx > 0 ? mx : 1, Hq, Hkv, d, theta)) != NE_OK)
        return rc;
    *maxlen = mx;
    return NE_OK;
}

// Builds [lengths][cu][tables] and copies it into the workspace on `st` (a
// copy from pageable memory, staged before cudaMemcpyAsync returns).
int upload_packed_tables(const int32_t *cu, int nseq, int maxlen, int Hq, int Hkv, int d,
                         const PackedLayout &L, void *workspace, cudaStream_t st, int counts[3])
{
    const size_t w = sizeof(int32_t);
    std::vector<int32_t> img(L.tables / w, 0);
    for (int b = 0; b < nseq; ++b)
        img[static_cast<size_t>(b)] = cu[b + 1] - cu[b];
    std::memcpy(img.data() + L.off_cu / w, cu, w * (static_cast<size_t>(nseq) + 1));
    const size_t caps[3] = {(L.off_dq - L.off_fwd) / w, (L.off_dkv - L.off_dq) / w,
                            (L.tables - L.off_dkv) / w};
    ne::varlen_plan(img.data(), nseq, maxlen > 0 ? maxlen : 1, Hq, Hkv, d, img.data() + L.off_fwd / w,
                    img.data() + L.off_dq / w, img.data() + L.off_dkv / w, caps, counts);
    for (int i = 0; i < 3; ++i)
        if (static_cast<size_t>(counts[i]) > caps[i])
            return NE_ERR_ARG;   // cannot happen: the regions bound every live unit
    return cudaMemcpyAsync(workspace, img.data(), L.tables, cudaMemcpyHostToDevice, st) ==
                   cudaSuccess
               ? NE_OK
               : NE_ERR_CUDA;
}

// The launch parameters of a packed batch's kernels: the sequence count as
// the batch of the unit enumeration, the longest sequence's tiles as M, the
// pack's rows as T.
void set_packed(ne::AttnParams &p, void *workspace, const PackedLayout &L, int nseq, int maxlen)
{
    p.B = nseq;
    p.M = (maxlen + 127) / 128;
    p.seqlen = ws_int(workspace, 0);
    p.cu = ws_int(workspace, L.off_cu);
    p.nseq = nseq;
}

} // namespace

extern "C" {

size_t ne_attn_packed_workspace_size(int nseq, int total, int Hq, int Hkv, int d)
{
    if (nseq < 1 || check_shape(1, total, Hq, Hkv, d, 1.0f) != NE_OK)
        return 0;
    return packed_layout(nseq, total, Hq, Hkv, d).total;
}

} // extern "C"

namespace {

// The plan kernel on a packed batch's prefix array (device memory).
int plan_packed_on_device(const int32_t *cu, int nseq, int total, int Hq, int Hkv, int d,
                          const PackedLayout &L, void *workspace, uint32_t *status,
                          cudaStream_t st)
{
    auto at = [&](size_t off) { return const_cast<int *>(ws_int(workspace, off)); };
    const int G = Hq / Hkv;
    ne::DevicePlanParams q;
    std::memset(&q, 0, sizeof(q));
    q.cu_in = cu;
    q.cu_out = at(L.off_cu);
    q.seqlen_out = at(0);
    q.fwd_units = at(L.off_fwd);
    q.dq_units = at(L.off_dq);
    q.dkv_units = at(L.off_dkv);
    q.counts = at(L.off_cnt);
    q.scratch = at(L.off_scr);
    q.B = nseq;
    q.T = total;
    q.M = (total + 127) / 128;
    q.Hkv = Hkv;
    q.nch_fwd = G / ne::fwd_heads_per_cta(d, G);
    q.nch_dq = G / ne::dq_heads_per_cta(d, G);
    q.status = status;
    return ne::launch_varlen_plan(q, st) == cudaSuccess ? NE_OK : NE_ERR_CUDA;
}

// Host-side checks of a packed call; with a prefix array in device memory
// only its pointer and the shape (the plan kernel checks the contents), and
// the tile bound is that of one sequence of `total` rows.
int check_packed_args(const int32_t *cu, bool dev_cu, int nseq, int total, int Hq, int Hkv,
                      int d, float theta, int *maxlen)
{
    if (!dev_cu)
        return check_packed(cu, nseq, total, Hq, Hkv, d, theta, maxlen);
    if (!cu)
        return NE_ERR_NULL;
    if (nseq < 1)
        return NE_ERR_SHAPE;
    int rc = check_shape(1, total, Hq, Hkv, d, theta);
    if (rc != NE_OK)
        return rc;
    if ((rc = check_shape(nseq, total, Hq, Hkv, d, theta)) != NE_OK)
        return rc;
    *maxlen = total;
    return NE_OK;
}

int fwd_packed_impl(const void *q, const void *k, const void *v, void *o, float *lse,
                    const int32_t *cu_seqlens, bool dev_cu, void *workspace,
                    size_t workspace_bytes, int nseq, int total, int Hq, int Hkv, int d,
                    float rope_theta, void *stream)
{
    if (!q || !k || !v || !o || !lse || !workspace)
        return NE_ERR_NULL;
    int maxlen = 0;
    int rc = check_packed_args(cu_seqlens, dev_cu, nseq, total, Hq, Hkv, d, rope_theta, &maxlen);
    if (rc != NE_OK)
        return rc;
    const PackedLayout L = packed_layout(nseq, total, Hq, Hkv, d);
    if (workspace_bytes < L.tables)
        return NE_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
        !aligned16(workspace) || (dev_cu && !aligned4(cu_seqlens)))
        return NE_ERR_ALIGN;
    uint32_t *status = nullptr;
    if ((rc = device_state(&status)) != NE_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ne::AttnParams p = base_params(1, total, Hq, Hkv, d, rope_theta, status);
    p.GC = ne::fwd_heads_per_cta(d, p.G);
    p.nchunks = p.G / p.GC;
    p.out0 = o;
    p.lse = lse;
    p.q_in = q;
    p.k_in = k;
    p.v_in = v;
    CUtensorMap mq, mk, mv, mo;
    if (make_map(&mq, q, 1, total, Hq, d) || make_map(&mk, k, 1, total, Hkv, d) ||
        make_map(&mv, v, 1, total, Hkv, d) ||
        make_map(&mo, o, 1, total, Hq, d, false, ne::kFwdOStoreRows))
        return NE_ERR_CUDA;
    int counts[3] = {1, 1, 1};
    if (dev_cu)
        rc = plan_packed_on_device(cu_seqlens, nseq, total, Hq, Hkv, d, L, workspace, status, st);
    else
        rc = upload_packed_tables(cu_seqlens, nseq, maxlen, Hq, Hkv, d, L, workspace, st,
                                  counts);
    if (rc != NE_OK)
        return rc;
    set_packed(p, workspace, L, nseq, maxlen);
    p.units = ws_int(workspace, L.off_fwd);
    p.num_units = counts[0];
    if (dev_cu)
        p.unit_count = ws_int(workspace, L.off_cnt);
    if (counts[0] > 0 && ne::launch_fwd(d, mq, mk, mv, mo, mq, mk, p, st) != cudaSuccess)
        return NE_ERR_CUDA;
    return NE_OK;
}

int bwd_packed_impl(const void *q, const void *k, const void *v, const void *o,
                    const float *lse, const void *dO, void *dq, void *dk, void *dv,
                    const int32_t *cu_seqlens, bool dev_cu, void *workspace,
                    size_t workspace_bytes, int nseq, int total, int Hq, int Hkv, int d,
                    float rope_theta, void *stream)
{
    if (!o || !dq || !dk || !dv || !workspace)
        return NE_ERR_NULL;
    int maxlen = 0;
    int rc = check_packed_args(cu_seqlens, dev_cu, nseq, total, Hq, Hkv, d, rope_theta, &maxlen);
    if (rc != NE_OK)
        return rc;
    const PackedLayout L = packed_layout(nseq, total, Hq, Hkv, d);
    if (workspace_bytes < L.total)
        return NE_ERR_WORKSPACE;
    if (!aligned16(o) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        !aligned16(workspace) || (dev_cu && !aligned4(cu_seqlens)))
        return NE_ERR_ALIGN;
    void *bws = static_cast<uint8_t *>(workspace) + L.tables;
    ne::AttnParams p;
    CUtensorMap mq, mk, mv, mdo, mqr, mkr;
    rc = bwd_setup(q, k, v, lse, dO, bws, workspace_bytes - L.tables, 1, total, Hq, Hkv, d,
                   rope_theta, &p, &mq, &mk, &mv, &mdo, &mqr, &mkr);
    if (rc != NE_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int counts[3] = {1, 1, 1};
    if (dev_cu)
        rc = plan_packed_on_device(cu_seqlens, nseq, total, Hq, Hkv, d, L, workspace, p.status,
                                   st);
    else
        rc = upload_packed_tables(cu_seqlens, nseq, maxlen, Hq, Hkv, d, L, workspace, st,
                                  counts);
    if (rc != NE_OK)
        return rc;
    // the preprocess streams over the pack's rows (B = 1 in memory) and
    // finds each row's position in its sequence through cu
    p.o_in = o;
    p.cu = ws_int(workspace, L.off_cu);
    p.nseq = nseq;
    void *qrot = static_cast<uint8_t *>(bws) + ws_d_bytes(1, total, Hq);
    void *krot = static_cast<uint8_t *>(qrot) + ws_q_bytes(1, total, Hq, d);
    if (ne::launch_bwd_pre(d, p, q, qrot, k, krot, st) != cudaSuccess)
        return NE_ERR_CUDA;
    set_packed(p, workspace, L, nseq, maxlen);
    p.units = ws_int(workspace, L.off_dq);
    p.num_units = counts[1];
    if (dev_cu)
        p.unit_count = ws_int(workspace, L.off_cnt) + 1;
    if (counts[1] > 0 && (rc = run_dq(d, p, dq, mqr, mkr, mv, mdo, st)) != NE_OK)
        return rc;
    p.units = ws_int(workspace, L.off_dkv);
    p.num_units = counts[2];
    if (dev_cu)
        p.unit_count = ws_int(workspace, L.off_cnt) + 2;
    if (counts[2] > 0 && (rc = run_dkdv(d, p, dk, dv, mqr, mkr, mv, mdo, st)) != NE_OK)
        return rc;
    return NE_OK;
}

} // namespace

extern "C" {

int ne_attn_fwd_packed(const void *q, const void *k, const void *v, void *o, float *lse,
                       const int32_t *cu_seqlens, void *workspace, size_t workspace_bytes,
                       int nseq, int total, int Hq, int Hkv, int d, float rope_theta,
                       void *stream)
{
    return fwd_packed_impl(q, k, v, o, lse, cu_seqlens, false, workspace, workspace_bytes, nseq,
                           total, Hq, Hkv, d, rope_theta, stream);
}

int ne_attn_bwd_packed(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dO, void *dq, void *dk, void *dv,
                       const int32_t *cu_seqlens, void *workspace, size_t workspace_bytes,
                       int nseq, int total, int Hq, int Hkv, int d, float rope_theta,
                       void *stream)
{
    return bwd_packed_impl(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens, false, workspace,
                           workspace_bytes, nseq, total, Hq, Hkv, d, rope_theta, stream);
}

int ne_attn_fwd_packed_dev(const void *q, const void *k, const void *v, void *o, float *lse,
                           const int32_t *cu_seqlens_dev, void *workspace,
                           size_t workspace_bytes, int nseq, int total, int Hq, int Hkv, int d,
                           float rope_theta, void *stream)
{
    return fwd_packed_impl(q, k, v, o, lse, cu_seqlens_dev, true, workspace, workspace_bytes,
                           nseq, total, Hq, Hkv, d, rope_theta, stream);
}

int ne_attn_bwd_packed_dev(const void *q, const void *k, const void *v, const void *o,
                           const float *lse, const void *dO, void *dq, void *dk, void *dv,
                           const int32_t *cu_seqlens_dev, void *workspace,
                           size_t workspace_bytes, int nseq, int total, int Hq, int Hkv, int d,
                           float rope_theta, void *stream)
{
    return bwd_packed_impl(q, k, v, o, lse, dO, dq, dk, dv, cu_seqlens_dev, true, workspace,
                           workspace_bytes, nseq, total, Hq, Hkv, d, rope_theta, stream);
}

} // extern "C"

// ------------------------------------------------------------------------
// Backward without any allocation.  Its scratch (the D rows and the rotated
// Q'/K' that ne_attn_bwd keeps in the caller's workspace) lives in one fixed
// array that is part of this library's device image, so every GPU that
// loads the library holds it until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(32) << 20;   // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (cudaGetSymbolAddress with that device current).
int noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return NE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
            return NE_ERR_CUDA;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return NE_OK;
}

} // namespace

extern "C" {

size_t ne_attn_bwd_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

int ne_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                        const float *lse, const void *dO, void *dq, void *dk, void *dv, int B,
                        int T, int Hq, int Hkv, int d, float rope_theta, void *stream)
{
    // The checks run in ne_attn_bwd's order, with the scratch limit where
    // ne_attn_bwd checks the workspace, so the same arguments give the same
    // status.
    if (!o || !dq || !dk || !dv)
        return NE_ERR_NULL;
    if (!aligned16(o) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return NE_ERR_ALIGN;
    if (!q || !k || !v || !lse || !dO)
        return NE_ERR_NULL;
    int rc = check_shape(B, T, Hq, Hkv, d, rope_theta);
    if (rc != NE_OK)
        return rc;
    if (ne_attn_bwd_workspace_size(B, T, Hq, Hkv, d) > kNoAllocScratchBytes)
        return NE_ERR_TOO_LARGE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned4(lse))
        return NE_ERR_ALIGN;
    uint32_t *status = nullptr;
    if ((rc = device_state(&status)) != NE_OK)
        return rc;
    void *scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch)) != NE_OK)
        return rc;
    // Every part of the scratch the kernels read is written earlier in the same
    // call, so nothing has to be cleared between calls.
    return ne_attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, scratch, kNoAllocScratchBytes, B, T, Hq,
                       Hkv, d, rope_theta, stream);
}

} // extern "C"
