// zp_noalloc.cu -- paged decode attention for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc at all: an allocator or memory-pool
// callback (allocating there would re-enter the allocator), a plug-in loaded
// into a host process that owns all device memory, or a real-time path that
// must not block on the driver's allocator.  This entry point needs no
// zp_cache handle (whose creation allocates) and allocates nothing: it runs
// the handle path's split-K decode kernel (zp_decode.cu) with the two pools'
// tensor maps passed by value in the launch parameters (encoded on the host
// for each call), and its split-K partial results live in a fixed
// file-scope device array, created when the library's device code is loaded
// into a context (usually at the first call there) and held until the
// process exits.  The array's last word is the status word of calls that
// pass none.  With the same splits as the handle path, the results are the
// handle path's bit for bit.
#include <mutex>

#include "zp_internal.cuh"

namespace {

// The fixed array: 32,768 partial slots of a (request, query head, split) at
// head_dim 128 (130 floats each: m, l, o[d]; ~16.3 MiB); calls are limited to
// R * Hq <= kNaSlots pairs, and the splits to what the array holds.
constexpr int kNaSlots = 32768;
constexpr int kNaSlotFloats = 128 + 2;
constexpr size_t kNaFloats = static_cast<size_t>(kNaSlots) * kNaSlotFloats;

static __device__ __align__(256) float g_na_part[kNaFloats];

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
    if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(out) % 2)
        return ZP_ERR_INVALID_ARG;  // query rows are read 16 bytes at a time
    if ((head_dim != 64 && head_dim != 128) || num_q_heads / num_kv_heads > 16)
        return ZP_ERR_UNSUPPORTED;  // (up to 16 query heads share a kv head)
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

    zp::DecodeArgs a{};
    if (!zp::encode_pool_map(&a.kmap_v, k_pool, num_blocks, num_kv_heads, head_dim) ||
        !zp::encode_pool_map(&a.vmap_v, v_pool, num_blocks, num_kv_heads, head_dim))
        return ZP_ERR_UNSUPPORTED;
    // the handle path's splits, fewer if the array cannot hold their partials
    // (its last word stays free: the status of calls that pass none)
    int bps = 0;
    int splits = zp::decode_splits(static_cast<long long>(R) * num_kv_heads, bt_stride, sms, &bps);
    while (splits > 1 && static_cast<size_t>(R) * num_q_heads * splits * (head_dim + 2) >=
                             kNaFloats) {
        bps = (bt_stride + splits - 2) / (splits - 1);
        splits = (bt_stride + bps - 1) / bps;
    }
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.tables = block_tables;
    a.stride = bt_stride;
    a.num_rows = num_rows;
    a.lengths = lengths;
    a.req_idx = req_idx;
    a.R = R;
    a.Hkv = num_kv_heads;
    a.Hq = num_q_heads;
    a.num_blocks = num_blocks;
    a.splits = splits;
    a.bps = bps;
    a.logit_scale = scale * 1.4426950408889634f;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.part = part;
    a.sticky = status ? status : reinterpret_cast<int32_t *>(part + kNaFloats - 1);
    if (zp::launch_decode_mapv(a, head_dim, s) != cudaSuccess)
        return ZP_ERR_CUDA;
    return ZP_OK;
}
