// zp_noalloc.cu -- paged decode attention for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc at all: an allocator or memory-pool
// callback (allocating there would re-enter the allocator), a plug-in loaded
// into a host process that owns all device memory, or a real-time path that
// must not block on the driver's allocator.  This entry point needs no
// zp_cache handle (whose creation allocates) and allocates nothing: its
// split-K partial results live in a fixed file-scope device array, created
// when the library's device code is loaded into a context (usually at the
// first call there) and held until the process exits.
//
// The kernels here are a plain CUDA-core variant of the split-K decode
// attention in zp_decode.cu: one CTA per (request, query head, split); a warp
// takes 32 / (d / 8) tokens at a time, d / 8 lanes per token row reading 16
// bytes each, with a shuffle-reduced dot product and an online softmax per
// token group, merged within the warp and then across warps; a log-sum-exp
// combine over the splits.
#include <mutex>

#include "zp_internal.cuh"

namespace {

constexpr int kNaThreads = 128;
constexpr int kNaWarps = kNaThreads / 32;
constexpr int kNaMaxSplits = 16;
// Maximum (request, query head, split) partial slots the array holds; with
// head_dim up to 128 each slot is 130 floats, so the array is ~16.3 MiB.
constexpr int kNaSlots = 32768;
constexpr int kNaSlotFloats = 128 + 2;

static __device__ __align__(256) float g_na_part[static_cast<size_t>(kNaSlots) * kNaSlotFloats];

struct NaArgs {
    const __nv_bfloat16 *kpool, *vpool, *q;
    const int32_t *tables, *lengths, *req_idx;
    int32_t stride, num_rows, num_blocks, R, Hkv, Hq, splits, tps;  // tps: tokens per split
    float logit_scale;  // scale * log2(e)
    float *part;        // the device address of g_na_part
    __nv_bfloat16 *out;
    int32_t *status;    // nullable
};

template <int D>
__global__ void __launch_bounds__(kNaThreads) na_decode_split(const NaArgs a)
{
    constexpr int LPR = D / 8;     // lanes per row: 16 bytes (8 elements) each
    constexpr int TPW = 32 / LPR;  // tokens a warp takes at a time
    __shared__ float s_m[kNaWarps], s_l[kNaWarps];
    __shared__ float s_o[kNaWarps][D];
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    const int sub = lane / LPR, sl = lane % LPR;  // token of the warp's group, lane in the row
    const int split = blockIdx.x, hq = blockIdx.y, r = blockIdx.z;
    const int G = a.Hq / a.Hkv, h = hq / G;
    int row = a.req_idx ? a.req_idx[r] : r;
    const bool row_ok = row >= 0 && row < a.num_rows;
    int len = row_ok ? a.lengths[row] : 0;
    if (!row_ok || len < 0 || len > a.stride * zp::kBlk) {
        if (threadIdx.x == 0 && split == 0 && a.status)
            atomicCAS(a.status, 0, row_ok ? ZP_ERR_DEVICE_CHECK : ZP_ERR_INVALID_ARG);
        len = 0;
        row = 0;
    }
    float qv[8];
    const __nv_bfloat16 *qrow = a.q + ((size_t)r * a.Hq + hq) * D + sl * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        qv[i] = __bfloat162float(qrow[i]);
    const int t_begin = split * a.tps, t_end = min(len, t_begin + a.tps);
    float m = -1e30f, l = 0.f, o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        o[i] = 0.f;
    // the warp takes TPW consecutive tokens at a time, LPR lanes per token
    for (int t0 = t_begin + wi * TPW; t0 < t_end; t0 += kNaWarps * TPW) {
        const int t = t0 + sub;
        bool valid = t < t_end;
        size_t off = 0;
        if (valid) {
            const int blk = a.tables[(size_t)row * a.stride + t / zp::kBlk];
            if (blk < 0 || blk >= a.num_blocks) {
                if (sl == 0 && a.status)
                    atomicCAS(a.status, 0, ZP_ERR_DEVICE_CHECK);
                valid = false;
            } else {
                off = (((size_t)blk * a.Hkv + h) * zp::kBlk + t % zp::kBlk) * D + sl * 8;
            }
        }
        uint4 kr = make_uint4(0u, 0u, 0u, 0u), vr = make_uint4(0u, 0u, 0u, 0u);
        if (valid) {
            kr = zp::ld_global_nc_v4(a.kpool + off);
            vr = zp::ld_global_nc_v4(a.vpool + off);
        }
        const __nv_bfloat162 *kh = reinterpret_cast<const __nv_bfloat162 *>(&kr);
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 kf = __bfloat1622float2(kh[i]);
            dot += qv[2 * i] * kf.x + qv[2 * i + 1] * kf.y;
        }
#pragma unroll
        for (int s = LPR / 2; s > 0; s >>= 1)
            dot += __shfl_xor_sync(0xffffffffu, dot, s);
        const float x = valid ? dot * a.logit_scale : -INFINITY;
        const float m_new = fmaxf(m, x);
        const float corr = exp2f(m - m_new), p = valid ? exp2f(x - m_new) : 0.f;
        l = l * corr + p;
        const __nv_bfloat162 *vh = reinterpret_cast<const __nv_bfloat162 *>(&vr);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 vf = __bfloat1622float2(vh[i]);
            o[2 * i] = o[2 * i] * corr + p * vf.x;
            o[2 * i + 1] = o[2 * i + 1] * corr + p * vf.y;
        }
        m = m_new;
    }
    // the warp's token groups merged: lanes sl of every group hold the same columns
#pragma unroll
    for (int s = LPR; s < 32; s <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, s);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, s);
        const float mm = fmaxf(m, m2);
        const float f1 = exp2f(m - mm), f2 = exp2f(m2 - mm);
        l = l * f1 + l2 * f2;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float o2 = __shfl_xor_sync(0xffffffffu, o[i], s);
            o[i] = o[i] * f1 + o2 * f2;
        }
        m = mm;
    }
    if (lane == 0) {
        s_m[wi] = m;
        s_l[wi] = l;
    }
    if (sub == 0)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            s_o[wi][sl * 8 + i] = o[i];
    __syncthreads();
    float *p = a.part + (((size_t)r * a.Hq + hq) * a.splits + split) * kNaSlotFloats;
    float M = -1e30f;
#pragma unroll
    for (int w = 0; w < kNaWarps; ++w)
        M = fmaxf(M, s_m[w]);
    for (int c = threadIdx.x; c < D; c += kNaThreads) {
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kNaWarps; ++w) {
            const float f = exp2f(s_m[w] - M);
            L += s_l[w] * f;
            O += s_o[w][c] * f;
        }
        p[c] = O;
        if (c == 0) {
            p[D] = M;
            p[D + 1] = L;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(D) na_decode_combine(const NaArgs a)
{
    const int rh = blockIdx.x, c = threadIdx.x;
    const float *base = a.part + (size_t)rh * a.splits * kNaSlotFloats;
    float M = -1e30f;
    for (int s = 0; s < a.splits; ++s)
        M = fmaxf(M, base[s * kNaSlotFloats + D]);
    float L = 0.f, O = 0.f;
    for (int s = 0; s < a.splits; ++s) {
        const float f = exp2f(base[s * kNaSlotFloats + D] - M);
        L += base[s * kNaSlotFloats + D + 1] * f;
        O += base[s * kNaSlotFloats + c] * f;
    }
    a.out[(size_t)rh * D + c] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
}

// The device address of g_na_part belongs to a CUDA context: the module (and
// with it the array) is loaded once per context, so another context on the
// same device, or the new primary context after cudaDeviceReset, has its own
// copy at its own address.  Outside a stream capture every call asks the
// runtime for the current context's address (a host-side lookup) and records
// it against the context; inside a capture, where the lookup could load the
// module, only a recorded address is used.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);

CtxGetCurrentFn ctx_get_current()
{
    static CtxGetCurrentFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrentFn>(p);
        return static_cast<CtxGetCurrentFn>(nullptr);
    }();
    return fn;
}

constexpr int kNaCtxSlots = 64;
std::mutex g_na_mu;
CUcontext g_na_ctx[kNaCtxSlots];
float *g_na_addr[kNaCtxSlots];
int g_na_used = 0;

// ZP_OK with *out set, ZP_ERR_UNSUPPORTED when `stream` is being captured and
// this context has no recorded address yet, ZP_ERR_CUDA on a runtime error.
zp_status na_scratch(cudaStream_t stream, float **out)
{
    CtxGetCurrentFn get = ctx_get_current();
    if (!get)
        return ZP_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess)
        return ZP_ERR_CUDA;
    if (cap == cudaStreamCaptureStatusNone) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_na_part) != cudaSuccess)
            return ZP_ERR_CUDA;
        CUcontext ctx = nullptr;
        if (get(&ctx) != CUDA_SUCCESS || !ctx)
            return ZP_ERR_CUDA;
        std::lock_guard<std::mutex> lock(g_na_mu);
        int i = 0;
        while (i < g_na_used && g_na_ctx[i] != ctx)
            ++i;
        if (i == g_na_used && g_na_used < kNaCtxSlots)
            g_na_ctx[g_na_used++] = ctx;
        if (i < g_na_used)
            g_na_addr[i] = static_cast<float *>(ptr);
        *out = static_cast<float *>(ptr);
        return ZP_OK;
    }
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS || !ctx)
        return ZP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_na_mu);
    for (int i = 0; i < g_na_used; ++i)
        if (g_na_ctx[i] == ctx) {
            *out = g_na_addr[i];
            return ZP_OK;
        }
    return ZP_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" zp_status zp_paged_decode_attn_noalloc(
    const void *k_pool, const void *v_pool, int32_t num_blocks, int32_t num_kv_heads,
    int32_t num_q_heads, int32_t head_dim, const void *q, const int32_t *block_tables,
    int32_t bt_stride, int32_t num_rows, const int32_t *lengths, const int32_t *req_idx, int32_t R,
    float scale, void *out, int32_t *status, void *stream)
{
    if (!k_pool || !v_pool || !q || !block_tables || !lengths || !out)
        return ZP_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(k_pool) % 16 || reinterpret_cast<uintptr_t>(v_pool) % 16)
        return ZP_ERR_INVALID_ARG;  // pool rows are read 16 bytes at a time
    if (num_blocks < 1 || num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads ||
        R < 0 || num_rows < 1 || bt_stride < 1 || !(scale == scale))
        return ZP_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128)
        return ZP_ERR_UNSUPPORTED;
    if (static_cast<long long>(R) * num_q_heads > kNaSlots)
        return ZP_ERR_UNSUPPORTED;  // more (request, head) pairs than the fixed array holds
    if (static_cast<long long>(bt_stride) * zp::kBlk >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    if (R == 0)
        return ZP_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float *part = nullptr;
    const zp_status scratch = na_scratch(s, &part);
    if (scratch != ZP_OK)
        return scratch;
    int device = 0, sms = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return ZP_ERR_CUDA;

    // splits: about four CTAs per SM, bounded by the array and by 16
    const int heads = R * num_q_heads;
    int splits = (4 * sms + heads - 1) / heads;
    splits = splits < 1 ? 1 : splits > kNaMaxSplits ? kNaMaxSplits : splits;
    while (splits > 1 && static_cast<long long>(heads) * splits > kNaSlots)
        --splits;
    const int max_tokens = bt_stride * zp::kBlk;
    NaArgs a{};
    a.kpool = static_cast<const __nv_bfloat16 *>(k_pool);
    a.vpool = static_cast<const __nv_bfloat16 *>(v_pool);
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.tables = block_tables;
    a.lengths = lengths;
    a.req_idx = req_idx;
    a.stride = bt_stride;
    a.num_rows = num_rows;
    a.num_blocks = num_blocks;
    a.R = R;
    a.Hkv = num_kv_heads;
    a.Hq = num_q_heads;
    a.splits = splits;
    a.tps = (max_tokens + splits - 1) / splits;
    a.logit_scale = scale * 1.4426950408889634f;
    a.part = part;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.status = status;
    const dim3 grid(static_cast<unsigned>(splits), static_cast<unsigned>(num_q_heads),
                    static_cast<unsigned>(R));
    if (head_dim == 64) {
        na_decode_split<64><<<grid, kNaThreads, 0, s>>>(a);
        na_decode_combine<64><<<static_cast<unsigned>(heads), 64, 0, s>>>(a);
    } else {
        na_decode_split<128><<<grid, kNaThreads, 0, s>>>(a);
        na_decode_combine<128><<<static_cast<unsigned>(heads), 128, 0, s>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? ZP_OK : ZP_ERR_CUDA;
}
