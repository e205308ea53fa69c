// zp_api.cu -- the C ABI declared in include/zp.h: handle, argument checks,
// TMA tensor maps, launches.  Host code only.
#include <nvtx3/nvToolsExt.h>  // header-only; the ranges cost a pointer test without a profiler

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "zp_aux.cuh"
#include "zp_internal.cuh"

using zp::Workspace;

namespace {

constexpr int kMaxSplits = 16;

// NVTX range around one entry point (host side: the argument checks and the
// launches it enqueues), named after it, for timeline profilers.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

struct Alloc {
    size_t off = 0;
    size_t take(size_t bytes, size_t align = 256)
    {
        off = (off + align - 1) / align * align;
        const size_t o = off;
        off += bytes;
        return o;
    }
};

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace zp {

// One split per pair whenever the pairs alone give every SM a CTA (the
// hardware scheduler balances the waves; a split adds partials and a combine
// launch), else enough to give every SM one, at most kMaxSplits, never fewer
// than 4 blocks per split.
int decode_splits(long long pairs, int bt_stride, int num_sms, int *bps)
{
    const long long target = num_sms;
    int splits = static_cast<int>(
        std::min<long long>(kMaxSplits, std::max<long long>(1, (target + pairs - 1) / pairs)));
    splits = std::min(splits, std::max(1, bt_stride / 4));
    *bps = (bt_stride + splits - 1) / splits;
    return (bt_stride + *bps - 1) / *bps;
}

}  // namespace zp

struct zp_cache {
    int device = 0;
    int L = 0, Hkv = 0, Hq = 0, d = 0, b = 0, num_blocks = 0;
    int max_requests = 0, max_blocks = 0;
    int num_sms = 0;
    std::vector<void *> kpools, vpools;  // host copies of the pool pointers
    void *base = nullptr;
    Workspace ws{};
};

extern "C" {

const char *zp_status_string(zp_status s)
{
    switch (s) {
    case ZP_OK: return "ok";
    case ZP_ERR_INVALID_ARG: return "invalid argument";
    case ZP_ERR_UNSUPPORTED: return "unsupported shape or size";
    case ZP_ERR_OUT_OF_BLOCKS: return "free stack too short";
    case ZP_ERR_DEVICE_CHECK: return "inconsistent cache state found on the device";
    case ZP_ERR_CUDA: return "CUDA runtime error";
    case ZP_ERR_TIMEOUT: return "bounded device wait gave up";
    default: return "unknown status";
    }
}

zp_status zp_cache_create(const zp_cache_desc *desc, zp_cache **out)
{
    NvtxRange nvtx("zp_cache_create");
    if (!desc || !out)
        return ZP_ERR_INVALID_ARG;
    const zp_cache_desc &D = *desc;
    if (D.num_layers < 1 || D.num_kv_heads < 1 || D.num_q_heads < 1 || D.num_blocks < 1 ||
        D.max_requests < 1 || D.max_blocks_per_req < 2 || !D.k_pools || !D.v_pools)
        return ZP_ERR_INVALID_ARG;
    if (D.num_q_heads % D.num_kv_heads != 0)
        return ZP_ERR_INVALID_ARG;
    if (D.head_dim != 64 && D.head_dim != 128)
        return ZP_ERR_UNSUPPORTED;
    if (D.block_size != zp::kBlk)
        return ZP_ERR_UNSUPPORTED;
    if (D.num_q_heads / D.num_kv_heads > 16)
        return ZP_ERR_UNSUPPORTED;
    const uint64_t rows = static_cast<uint64_t>(D.num_blocks) * D.num_kv_heads * zp::kBlk;
    if (rows >= (1ull << 31))
        return ZP_ERR_UNSUPPORTED;
    for (int l = 0; l < D.num_layers; ++l)
        if (!D.k_pools[l] || !D.v_pools[l] || !aligned(D.k_pools[l], 16) ||
            !aligned(D.v_pools[l], 16))
            return ZP_ERR_INVALID_ARG;

    zp_cache *c = new (std::nothrow) zp_cache();
    if (!c)
        return ZP_ERR_CUDA;
    c->L = D.num_layers;
    c->Hkv = D.num_kv_heads;
    c->Hq = D.num_q_heads;
    c->d = D.head_dim;
    c->b = D.block_size;
    c->num_blocks = D.num_blocks;
    c->max_requests = D.max_requests;
    c->max_blocks = D.max_blocks_per_req;
    if (cudaGetDevice(&c->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) !=
            cudaSuccess) {
        delete c;
        return ZP_ERR_CUDA;
    }

    const size_t entries = static_cast<size_t>(D.max_requests) * D.max_blocks_per_req;
    const size_t part = static_cast<size_t>(D.max_requests) * D.num_q_heads * kMaxSplits *
                        (D.head_dim + 2);
    Alloc A;
    const size_t o_sticky = A.take(4);
    const size_t o_call = A.take(4);
    const size_t o_gens = A.take(8);
    const size_t o_smw = A.take(4 * 3 * zp::kSmSlots);
    const size_t o_kmaps = A.take(sizeof(CUtensorMap) * D.num_layers, 128);
    const size_t o_vmaps = A.take(sizeof(CUtensorMap) * D.num_layers, 128);
    const size_t o_krmaps = A.take(sizeof(CUtensorMap) * D.num_layers, 128);
    const size_t o_vrmaps = A.take(sizeof(CUtensorMap) * D.num_layers, 128);
    const size_t o_kp = A.take(sizeof(void *) * D.num_layers);
    const size_t o_vp = A.take(sizeof(void *) * D.num_layers);
    const size_t o_dst = A.take(4 * entries);
    const size_t o_push = A.take(4 * entries);
    const size_t o_cnt = A.take(16);
    const size_t o_occ = A.take(4 * static_cast<size_t>(D.num_blocks));
    const size_t o_last = A.take(4 * static_cast<size_t>(D.num_blocks));
    const size_t o_rowmark = A.take(4 * static_cast<size_t>(D.max_requests));
    const size_t o_part = A.take(4 * part);
    const size_t o_ap_call = A.take(4);
    const size_t o_ap_cnt = A.take(16);
    const size_t o_ap_rowmark = A.take(4 * static_cast<size_t>(D.max_requests));
    const size_t o_ap_occ = A.take(4 * static_cast<size_t>(D.num_blocks));
    const size_t o_ap_last = A.take(4 * static_cast<size_t>(D.num_blocks));
    const size_t o_ap_plan = A.take(16 * static_cast<size_t>(D.max_requests));
    const size_t total = A.take(0);

    if (cudaMalloc(&c->base, total) != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return ZP_ERR_CUDA;
    }
    uint8_t *b = static_cast<uint8_t *>(c->base);
    Workspace &ws = c->ws;
    ws.sticky = reinterpret_cast<int32_t *>(b + o_sticky);
    ws.call = reinterpret_cast<int32_t *>(b + o_call);
    ws.gens = reinterpret_cast<int32_t *>(b + o_gens);
    ws.smwave = reinterpret_cast<uint32_t *>(b + o_smw);
    ws.kmaps = reinterpret_cast<CUtensorMap *>(b + o_kmaps);
    ws.vmaps = reinterpret_cast<CUtensorMap *>(b + o_vmaps);
    ws.krmaps = reinterpret_cast<CUtensorMap *>(b + o_krmaps);
    ws.vrmaps = reinterpret_cast<CUtensorMap *>(b + o_vrmaps);
    ws.kpools = reinterpret_cast<void **>(b + o_kp);
    ws.vpools = reinterpret_cast<void **>(b + o_vp);
    ws.dst_table = reinterpret_cast<int32_t *>(b + o_dst);
    ws.push_list = reinterpret_cast<int32_t *>(b + o_push);
    ws.counters = reinterpret_cast<int32_t *>(b + o_cnt);
    ws.occ = reinterpret_cast<int32_t *>(b + o_occ);
    ws.last = reinterpret_cast<int32_t *>(b + o_last);
    ws.rowmark = reinterpret_cast<int32_t *>(b + o_rowmark);
    ws.dec_part = reinterpret_cast<float *>(b + o_part);
    ws.dec_part_floats = part;
    ws.ap_call = reinterpret_cast<int32_t *>(b + o_ap_call);
    ws.ap_counters = reinterpret_cast<int32_t *>(b + o_ap_cnt);
    ws.ap_rowmark = reinterpret_cast<int32_t *>(b + o_ap_rowmark);
    ws.ap_occ = reinterpret_cast<int32_t *>(b + o_ap_occ);
    ws.ap_last = reinterpret_cast<int32_t *>(b + o_ap_last);
    ws.ap_plan = reinterpret_cast<int4 *>(b + o_ap_plan);
    c->kpools.assign(D.k_pools, D.k_pools + D.num_layers);
    c->vpools.assign(D.v_pools, D.v_pools + D.num_layers);

    std::vector<CUtensorMap> kmaps(D.num_layers), vmaps(D.num_layers), krmaps(D.num_layers),
        vrmaps(D.num_layers);
    bool ok = true;
    for (int l = 0; l < D.num_layers && ok; ++l) {
        ok = zp::encode_pool_map(&kmaps[l], D.k_pools[l], D.num_blocks, D.num_kv_heads,
                                 D.head_dim) &&
             zp::encode_pool_map(&vmaps[l], D.v_pools[l], D.num_blocks, D.num_kv_heads, D.head_dim) &&
             zp::encode_row_map(&krmaps[l], D.k_pools[l], D.num_blocks, D.num_kv_heads, D.head_dim) &&
             zp::encode_row_map(&vrmaps[l], D.v_pools[l], D.num_blocks, D.num_kv_heads, D.head_dim);
    }
    ok = ok && cudaMemset(c->base, 0, o_kmaps) == cudaSuccess &&
         cudaMemset(b + o_rowmark, 0, 4 * static_cast<size_t>(D.max_requests)) == cudaSuccess &&
         cudaMemset(b + o_ap_call, 0, o_ap_occ - o_ap_call) == cudaSuccess &&
         cudaMemcpy(ws.kmaps, kmaps.data(), sizeof(CUtensorMap) * D.num_layers,
                    cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(ws.vmaps, vmaps.data(), sizeof(CUtensorMap) * D.num_layers,
                    cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(ws.krmaps, krmaps.data(), sizeof(CUtensorMap) * D.num_layers,
                    cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(ws.vrmaps, vrmaps.data(), sizeof(CUtensorMap) * D.num_layers,
                    cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(ws.kpools, D.k_pools, sizeof(void *) * D.num_layers,
                    cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(ws.vpools, D.v_pools, sizeof(void *) * D.num_layers,
                    cudaMemcpyHostToDevice) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        cudaFree(c->base);
        delete c;
        return ZP_ERR_CUDA;
    }
    *out = c;
    return ZP_OK;
}

void zp_cache_destroy(zp_cache *cache)
{
    if (!cache)
        return;
    if (cache->base)
        cudaFree(cache->base);
    delete cache;
}

static bool on_device(const zp_cache *c)
{
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev == c->device;
}

zp_status zp_compress(zp_cache *c, int32_t *block_tables, int32_t bt_stride, int32_t num_rows,
                      int32_t *lengths, const int32_t *req_idx, int32_t R, const void *window_q,
                      int32_t n_max, int32_t window, float lambda, const zp_block_pool *pool,
                      void *stream, float *scores_out, int32_t *kept_out)
{
    NvtxRange nvtx("zp_compress");
    if (!c || !block_tables || !lengths || !window_q || !pool || !pool->free_ids ||
        !pool->free_count || !pool->refcount)
        return ZP_ERR_INVALID_ARG;
    if (R < 0 || num_rows < 1 || num_rows > c->max_requests || R > num_rows)
        return ZP_ERR_INVALID_ARG;
    if (n_max < 2 || bt_stride < n_max || pool->capacity < 1)
        return ZP_ERR_INVALID_ARG;
    if (window < 1 || window > c->b || !std::isfinite(lambda))
        return ZP_ERR_INVALID_ARG;
    if (!aligned(window_q, 16) || !aligned(scores_out, 4) || !aligned(kept_out, 4))
        return ZP_ERR_INVALID_ARG;
    const int G = c->Hq / c->Hkv;
    const int T = n_max * c->b;
    const int rows = window * G;
    const int cs = zp::compress_cluster_size(T);
    if (n_max > c->max_blocks || cs == 0 || rows > zp::kMaxRows)
        return ZP_ERR_UNSUPPORTED;
    if (R == 0)
        return ZP_OK;
    if (!on_device(c))
        return ZP_ERR_INVALID_ARG;
    const int mt = rows <= 16 ? 1 : rows <= 32 ? 2 : 4;
    const long long units = static_cast<long long>(R) * c->L * c->Hkv;
    if (units * cs >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    zp::PlanArgs pa{};
    pa.tables = block_tables;
    pa.stride = bt_stride;
    pa.num_rows = num_rows;
    pa.lengths = lengths;
    pa.req_idx = req_idx;
    pa.R = R;
    pa.N = n_max;
    pa.M = n_max;
    pa.prefill = 0;
    pa.num_blocks = c->num_blocks;
    pa.refcount = pool->refcount;
    pa.free_ids = pool->free_ids;
    pa.free_count = pool->free_count;
    pa.capacity = pool->capacity;
    pa.ws = c->ws;
    if (zp::launch_plan(pa, s) != cudaSuccess)
        return ZP_ERR_CUDA;

    zp::CompressArgs ca{};
    ca.kmaps = c->ws.kmaps;
    ca.kpools = c->ws.kpools;
    ca.vpools = c->ws.vpools;
    ca.tables = block_tables;
    ca.stride = bt_stride;
    ca.req_idx = req_idx;
    ca.dst_table = c->ws.dst_table;
    ca.window_q = static_cast<const __nv_bfloat16 *>(window_q);
    ca.scores_out = scores_out;
    ca.kept_out = kept_out;
    ca.call = c->ws.call;
    ca.cstat = c->ws.counters + 2;
    ca.sticky = c->ws.sticky;
    ca.smwave = c->ws.smwave;
    ca.L = c->L;
    ca.Hkv = c->Hkv;
    ca.Hq = c->Hq;
    ca.R = R;
    ca.N = n_max;
    ca.w = window;
    ca.rows = rows;
    ca.cs = cs;
    ca.num_rows = num_rows;
    ca.num_blocks = c->num_blocks;
    ca.lambda = lambda;
    ca.inv_rows = 1.0f / static_cast<float>(rows);
    ca.logit_scale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c->d)));
    if (zp::launch_compress(ca, c->d, mt, static_cast<int>(units), s) != cudaSuccess)
        return ZP_ERR_CUDA;

    zp::FinalizeArgs fa{};
    fa.tables = block_tables;
    fa.stride = bt_stride;
    fa.lengths = lengths;
    fa.req_idx = req_idx;
    fa.R = R;
    fa.N = n_max;
    fa.M = n_max;
    fa.prefill = 0;
    fa.refcount = pool->refcount;
    fa.free_ids = pool->free_ids;
    fa.free_count = pool->free_count;
    fa.ws = c->ws;
    if (zp::launch_finalize(fa, s) != cudaSuccess)
        return ZP_ERR_CUDA;
    return ZP_OK;
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

zp_status zp_compress_prefill_workspace_size(const zp_cache *c, int32_t R, int32_t bt_stride,
                                             size_t *bytes)
{
    if (!c || !bytes || R < 0 || bt_stride < 1)
        return ZP_ERR_INVALID_ARG;
    const size_t units = static_cast<size_t>(R) * c->L * c->Hkv;
    const size_t T_cap = static_cast<size_t>(bt_stride) * c->b;
    const size_t NC = (T_cap + zp::kPrefillChunk - 1) / zp::kPrefillChunk;
    *bytes = align256(units * NC * zp::kMaxRows * sizeof(float2)) +  // chunk statistics
             2 * align256(units * T_cap * 4) +                        // redundancy, scores
             align256(units * T_cap * 4);                             // kept positions
    return ZP_OK;
}

zp_status zp_compress_prefill(zp_cache *c, int32_t *block_tables, int32_t bt_stride,
                              int32_t num_rows, int32_t *lengths, const int32_t *req_idx,
                              int32_t R, const void *window_q, int32_t n_max, int32_t window,
                              float lambda, const zp_block_pool *pool, void *workspace,
                              size_t workspace_bytes, void *stream, float *scores_out,
                              int32_t *kept_out)
{
    NvtxRange nvtx("zp_compress_prefill");
    if (!c || !block_tables || !lengths || !window_q || !pool || !pool->free_ids ||
        !pool->free_count || !pool->refcount)
        return ZP_ERR_INVALID_ARG;
    if (R < 0 || num_rows < 1 || num_rows > c->max_requests || R > num_rows)
        return ZP_ERR_INVALID_ARG;
    if (n_max < 2 || bt_stride < n_max || pool->capacity < 1)
        return ZP_ERR_INVALID_ARG;
    if (window < 1 || window > c->b || !std::isfinite(lambda))
        return ZP_ERR_INVALID_ARG;
    if (!aligned(window_q, 16) || !aligned(scores_out, 4) || !aligned(kept_out, 4) ||
        !aligned(workspace, 256))
        return ZP_ERR_INVALID_ARG;
    const int G = c->Hq / c->Hkv;
    const int rows = window * G;
    if (bt_stride > c->max_blocks || static_cast<long long>(bt_stride) * c->b > zp::kPrefillMaxTokens ||
        rows > zp::kMaxRows)
        return ZP_ERR_UNSUPPORTED;
    size_t need = 0;
    zp_compress_prefill_workspace_size(c, R, bt_stride, &need);
    if (R > 0 && (!workspace || workspace_bytes < need))
        return ZP_ERR_INVALID_ARG;
    if (R == 0)
        return ZP_OK;
    if (!on_device(c))
        return ZP_ERR_INVALID_ARG;
    const long long units = static_cast<long long>(R) * c->L * c->Hkv;
    if (units >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int mt = rows <= 16 ? 1 : rows <= 32 ? 2 : 4;
    const int T_cap = bt_stride * c->b;
    const int NC = (T_cap + zp::kPrefillChunk - 1) / zp::kPrefillChunk;

    zp::PlanArgs pa{};
    pa.tables = block_tables;
    pa.stride = bt_stride;
    pa.num_rows = num_rows;
    pa.lengths = lengths;
    pa.req_idx = req_idx;
    pa.R = R;
    pa.N = n_max;
    pa.M = bt_stride;
    pa.prefill = 1;
    pa.num_blocks = c->num_blocks;
    pa.refcount = pool->refcount;
    pa.free_ids = pool->free_ids;
    pa.free_count = pool->free_count;
    pa.capacity = pool->capacity;
    pa.ws = c->ws;
    if (zp::launch_plan(pa, s) != cudaSuccess)
        return ZP_ERR_CUDA;

    uint8_t *w = static_cast<uint8_t *>(workspace);
    const size_t U = static_cast<size_t>(units);
    zp::PrefillArgs a{};
    a.kmaps = c->ws.kmaps;
    a.krmaps = c->ws.krmaps;
    a.vrmaps = c->ws.vrmaps;
    a.kpools = c->ws.kpools;
    a.vpools = c->ws.vpools;
    a.tables = block_tables;
    a.stride = bt_stride;
    a.lengths = lengths;
    a.req_idx = req_idx;
    a.dst_table = c->ws.dst_table;
    a.window_q = static_cast<const __nv_bfloat16 *>(window_q);
    a.stats = reinterpret_cast<float2 *>(w);
    w += align256(U * NC * zp::kMaxRows * sizeof(float2));
    a.red = reinterpret_cast<float *>(w);
    w += align256(U * T_cap * 4);
    a.scores = scores_out ? scores_out : reinterpret_cast<float *>(w);
    w += align256(U * T_cap * 4);
    a.kept = kept_out ? kept_out : reinterpret_cast<int32_t *>(w);
    a.call = c->ws.call;
    a.sticky = c->ws.sticky;
    a.L = c->L;
    a.Hkv = c->Hkv;
    a.Hq = c->Hq;
    a.R = R;
    a.N = n_max;
    a.w = window;
    a.rows = rows;
    a.T_cap = T_cap;
    a.NC = NC;
    a.lambda = lambda;
    a.inv_rows = 1.0f / static_cast<float>(rows);
    a.logit_scale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c->d)));
    if (zp::launch_prefill(a, c->d, mt, static_cast<int>(units), s) != cudaSuccess)
        return ZP_ERR_CUDA;

    zp::FinalizeArgs fa{};
    fa.tables = block_tables;
    fa.stride = bt_stride;
    fa.lengths = lengths;
    fa.req_idx = req_idx;
    fa.R = R;
    fa.N = n_max;
    fa.M = bt_stride;
    fa.prefill = 1;
    fa.refcount = pool->refcount;
    fa.free_ids = pool->free_ids;
    fa.free_count = pool->free_count;
    fa.ws = c->ws;
    if (zp::launch_finalize(fa, s) != cudaSuccess)
        return ZP_ERR_CUDA;
    return ZP_OK;
}

zp_status zp_paged_decode_attn(zp_cache *c, int32_t layer, const void *q,
                               const int32_t *block_tables, int32_t bt_stride, int32_t num_rows,
                               const int32_t *lengths, const int32_t *req_idx, int32_t R,
                               float scale, void *out, void *stream)
{
    NvtxRange nvtx("zp_paged_decode_attn");
    if (!c || !q || !block_tables || !lengths || !out)
        return ZP_ERR_INVALID_ARG;
    if (layer < 0 || layer >= c->L || R < 0 || R > c->max_requests || num_rows < 1 ||
        bt_stride < 1 || !std::isfinite(scale))
        return ZP_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 2))
        return ZP_ERR_INVALID_ARG;
    if (static_cast<long long>(bt_stride) * c->b >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    if (R == 0)
        return ZP_OK;
    if (!on_device(c))
        return ZP_ERR_INVALID_ARG;

    int bps = 0;
    const int splits = zp::decode_splits(static_cast<long long>(R) * c->Hkv, bt_stride,
                                         c->num_sms, &bps);

    zp::DecodeArgs da{};
    // the per-layer maps live in device memory; kernels take their address
    da.kmap = c->ws.kmaps + layer;
    da.vmap = c->ws.vmaps + layer;
    da.q = static_cast<const __nv_bfloat16 *>(q);
    da.tables = block_tables;
    da.stride = bt_stride;
    da.num_rows = num_rows;
    da.lengths = lengths;
    da.req_idx = req_idx;
    da.R = R;
    da.Hkv = c->Hkv;
    da.Hq = c->Hq;
    da.num_blocks = c->num_blocks;
    da.splits = splits;
    da.bps = bps;
    da.logit_scale = scale * 1.4426950408889634f;
    da.out = static_cast<__nv_bfloat16 *>(out);
    da.part = c->ws.dec_part;
    da.sticky = c->ws.sticky;
    if (zp::launch_decode(da, c->d, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ZP_ERR_CUDA;
    return ZP_OK;
}

zp_status zp_append_slots(zp_cache *c, int32_t *block_tables, int32_t bt_stride,
                          int32_t num_rows, int32_t *lengths, const int32_t *req_idx, int32_t R,
                          int32_t n_max, const zp_block_pool *pool, void *stream,
                          int32_t *trigger_rows, int32_t *trigger_count)
{
    NvtxRange nvtx("zp_append_slots");
    if (!c || !block_tables || !lengths || !pool || !pool->free_ids || !pool->free_count ||
        !pool->refcount)
        return ZP_ERR_INVALID_ARG;
    if (R < 0 || num_rows < 1 || num_rows > c->max_requests || R > num_rows || bt_stride < 1 ||
        n_max < 0 || pool->capacity < 1)
        return ZP_ERR_INVALID_ARG;
    if (!aligned(trigger_rows, 4) || !aligned(trigger_count, 4))
        return ZP_ERR_INVALID_ARG;
    if (static_cast<long long>(bt_stride) * c->b >= (1ll << 31) ||
        static_cast<long long>(n_max) * c->b >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    if (!on_device(c))
        return ZP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (R == 0) {
        if (trigger_count && cudaMemsetAsync(trigger_count, 0, 4, s) != cudaSuccess)
            return ZP_ERR_CUDA;
        return ZP_OK;
    }
    zp::AppendArgs a{};
    a.tables = block_tables;
    a.stride = bt_stride;
    a.num_rows = num_rows;
    a.lengths = lengths;
    a.req_idx = req_idx;
    a.R = R;
    a.n_max = n_max;
    a.num_blocks = c->num_blocks;
    a.L = c->L;
    a.Hkv = c->Hkv;
    a.d = c->d;
    a.refcount = pool->refcount;
    a.free_ids = pool->free_ids;
    a.free_count = pool->free_count;
    a.capacity = pool->capacity;
    a.trigger_rows = trigger_rows;
    a.trigger_count = trigger_count;
    a.ws = c->ws;
    return zp::launch_append_slots(a, s) == cudaSuccess ? ZP_OK : ZP_ERR_CUDA;
}

zp_status zp_append_kv(zp_cache *c, int32_t layer, const void *k_new, const void *v_new,
                       const int32_t *block_tables, int32_t bt_stride, int32_t num_rows,
                       const int32_t *lengths, const int32_t *req_idx, int32_t R, void *stream)
{
    NvtxRange nvtx("zp_append_kv");
    if (!c || !k_new || !v_new || !block_tables || !lengths)
        return ZP_ERR_INVALID_ARG;
    if (layer < 0 || layer >= c->L || R < 0 || R > c->max_requests || num_rows < 1 ||
        bt_stride < 1)
        return ZP_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
        return ZP_ERR_INVALID_ARG;
    if (static_cast<long long>(bt_stride) * c->b >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    if (R == 0)
        return ZP_OK;
    if (!on_device(c))
        return ZP_ERR_INVALID_ARG;
    zp::AppendKvArgs a{};
    a.kpool = static_cast<__nv_bfloat16 *>(c->kpools[layer]);
    a.vpool = static_cast<__nv_bfloat16 *>(c->vpools[layer]);
    a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    a.tables = block_tables;
    a.stride = bt_stride;
    a.num_rows = num_rows;
    a.lengths = lengths;
    a.req_idx = req_idx;
    a.R = R;
    a.Hkv = c->Hkv;
    a.d = c->d;
    a.num_blocks = c->num_blocks;
    a.sticky = c->ws.sticky;
    return zp::launch_append_kv(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ZP_OK
                                                                                      : ZP_ERR_CUDA;
}

static zp_status rows_checks(const zp_cache *c, const int32_t *block_tables, int32_t bt_stride,
                             int32_t num_rows, const int32_t *lengths, int32_t R,
                             const zp_block_pool *pool)
{
    if (!c || !block_tables || !lengths || !pool || !pool->free_ids || !pool->free_count ||
        !pool->refcount || pool->capacity < 1)
        return ZP_ERR_INVALID_ARG;
    if (R < 0 || num_rows < 1 || num_rows > c->max_requests || R > num_rows || bt_stride < 1)
        return ZP_ERR_INVALID_ARG;
    if (static_cast<long long>(bt_stride) * c->b >= (1ll << 31) ||
        static_cast<long long>(R) * bt_stride >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    return ZP_OK;
}

zp_status zp_alloc_rows(zp_cache *c, int32_t *block_tables, int32_t bt_stride, int32_t num_rows,
                        int32_t *lengths, const int32_t *req_idx, int32_t R,
                        const int32_t *counts, const zp_block_pool *pool, void *stream)
{
    NvtxRange nvtx("zp_alloc_rows");
    zp_status st = rows_checks(c, block_tables, bt_stride, num_rows, lengths, R, pool);
    if (st != ZP_OK)
        return st;
    if (!counts)
        return ZP_ERR_INVALID_ARG;
    if (R == 0)
        return ZP_OK;
    if (!on_device(c))
        return ZP_ERR_INVALID_ARG;
    return zp::launch_alloc_rows(c->ws, block_tables, bt_stride, num_rows, lengths, req_idx, R,
                                 counts, c->num_blocks, pool,
                                 static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ZP_OK
               : ZP_ERR_CUDA;
}

zp_status zp_release_rows(zp_cache *c, int32_t *block_tables, int32_t bt_stride,
                          int32_t num_rows, int32_t *lengths, const int32_t *req_idx, int32_t R,
                          const zp_block_pool *pool, void *stream)
{
    NvtxRange nvtx("zp_release_rows");
    zp_status st = rows_checks(c, block_tables, bt_stride, num_rows, lengths, R, pool);
    if (st != ZP_OK)
        return st;
    if (R == 0)
        return ZP_OK;
    if (!on_device(c))
        return ZP_ERR_INVALID_ARG;
    return zp::launch_release_rows(c->ws, block_tables, bt_stride, num_rows, lengths, req_idx, R,
                                   c->num_blocks, pool,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ZP_OK
               : ZP_ERR_CUDA;
}

zp_status zp_fork_rows(zp_cache *c, int32_t *block_tables, int32_t bt_stride, int32_t num_rows,
                       int32_t *lengths, const int32_t *src_rows, const int32_t *dst_rows,
                       int32_t n, int32_t *refcount, void *stream)
{
    NvtxRange nvtx("zp_fork_rows");
    if (!c || !block_tables || !lengths || !refcount || (n > 0 && (!src_rows || !dst_rows)))
        return ZP_ERR_INVALID_ARG;
    if (n < 0 || num_rows < 1 || num_rows > c->max_requests || n > num_rows || bt_stride < 1)
        return ZP_ERR_INVALID_ARG;
    if (static_cast<long long>(n) * bt_stride >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    if (n == 0)
        return ZP_OK;
    if (!on_device(c))
        return ZP_ERR_INVALID_ARG;
    return zp::launch_fork_rows(c->ws, block_tables, bt_stride, num_rows, lengths, src_rows,
                                dst_rows, n, c->num_blocks, refcount,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ZP_OK
               : ZP_ERR_CUDA;
}

zp_status zp_global_redundancy(zp_cache *c, const int32_t *block_tables, int32_t bt_stride,
                               int32_t num_rows, const int32_t *lengths, const int32_t *req_idx,
                               int32_t R, float *red_out, void *stream)
{
    NvtxRange nvtx("zp_global_redundancy");
    if (!c || !block_tables || !lengths || !red_out || !aligned(red_out, 4))
        return ZP_ERR_INVALID_ARG;
    if (R < 0 || R > c->max_requests || num_rows < 1 || bt_stride < 1)
        return ZP_ERR_INVALID_ARG;
    if (static_cast<long long>(bt_stride) * c->b >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    const long long units = static_cast<long long>(R) * c->L * c->Hkv;
    if (units >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    if (R == 0)
        return ZP_OK;
    if (!on_device(c))
        return ZP_ERR_INVALID_ARG;
    zp::GlobalRedArgs a{};
    a.kpools = reinterpret_cast<__nv_bfloat16 *const *>(c->ws.kpools);
    a.tables = block_tables;
    a.stride = bt_stride;
    a.num_rows = num_rows;
    a.lengths = lengths;
    a.req_idx = req_idx;
    a.R = R;
    a.Hkv = c->Hkv;
    a.num_blocks = c->num_blocks;
    a.T_cap = bt_stride * c->b;
    a.red_out = red_out;
    a.sticky = c->ws.sticky;
    return zp::launch_global_redundancy(a, c->d, static_cast<int>(units),
                                        static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ZP_OK
               : ZP_ERR_CUDA;
}

zp_status zp_global_redundancy_gram(zp_cache *c, const int32_t *block_tables,
                                    int32_t bt_stride, int32_t num_rows, const int32_t *lengths,
                                    const int32_t *req_idx, int32_t R, float *red_out,
                                    void *stream)
{
    NvtxRange nvtx("zp_global_redundancy_gram");
    if (!c || !block_tables || !lengths || !red_out || !aligned(red_out, 4))
        return ZP_ERR_INVALID_ARG;
    if (R < 0 || R > c->max_requests || num_rows < 1 || bt_stride < 1)
        return ZP_ERR_INVALID_ARG;
    if (static_cast<long long>(bt_stride) * c->b >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    const long long units = static_cast<long long>(R) * c->L * c->Hkv;
    const int T_cap = bt_stride * c->b;
    const int row_tiles = zp::gram_row_tiles(T_cap);
    if (units * row_tiles >= (1ll << 31))
        return ZP_ERR_UNSUPPORTED;
    if (R == 0)
        return ZP_OK;
    if (!on_device(c))
        return ZP_ERR_INVALID_ARG;
    zp::GramRedArgs a{};
    a.kmaps = c->ws.kmaps;
    a.tables = block_tables;
    a.stride = bt_stride;
    a.num_rows = num_rows;
    a.lengths = lengths;
    a.req_idx = req_idx;
    a.R = R;
    a.Hkv = c->Hkv;
    a.num_blocks = c->num_blocks;
    a.T_cap = T_cap;
    a.row_tiles = row_tiles;
    a.red_out = red_out;
    a.sticky = c->ws.sticky;
    return zp::launch_gram_redundancy(a, c->d, static_cast<int>(units), c->num_sms,
                                      static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ZP_OK
               : ZP_ERR_CUDA;
}

zp_status zp_cache_status(zp_cache *c, void *stream, int32_t *out_status)
{
    NvtxRange nvtx("zp_cache_status");
    if (!c || !out_status)
        return ZP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, c->ws.sticky, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(c->ws.sticky, 0, 4, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return ZP_ERR_CUDA;
    *out_status = v;
    return ZP_OK;
}

}  // extern "C"
