// zp_internal.cuh -- shared device helpers and launch-argument structs of the
// sm_103a Compressed PagedAttention library.  Internal: not part of the C ABI.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; no driver-API link)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zp.h"

namespace zp {

constexpr int kBlk = 16;            // tokens per block (the only supported size)
constexpr int kMaxRows = 64;        // window rows per unit: w * (Hq / Hkv)
constexpr int kMaxCluster = 16;     // CTAs per unit in the compression kernel
constexpr uint32_t kWaitSpins = 1u << 22;  // bound on every mbarrier wait
constexpr int kPlanThreads = 1024;  // the one-CTA bookkeeping kernels
constexpr int kSmSlots = 256;       // SM ids tracked by the compression kernel's pairing

// ----------------------------------------------------------------- workspace
// Device memory the handle owns (allocated once in zp_cache_create).
struct Workspace {
    int32_t *sticky;     // [1]  first device-detected error since last read
    int32_t *call;       // [1]  status of the compression call in flight
    int32_t *gens;       // [2]  generation counters of the duplicate-row stamps
                         //      (compression, reservation), advanced on the device so
                         //      that a captured CUDA graph stamps afresh on every replay
    uint32_t *smwave;    // [3 * kSmSlots] per SM id, within one compression call: first
                         //      and second CTA claims, the first CTA's pass-1 flag;
                         //      zeroed by the finalize kernel
    CUtensorMap *kmaps;  // [L]  K pool maps, 128B swizzle, box {64, 16}
    CUtensorMap *vmaps;  // [L]  V pool maps, same
    CUtensorMap *krmaps; // [L]  K pool maps, no swizzle, box {d, 1}: one pool row (row gathers)
    CUtensorMap *vrmaps; // [L]  V pool maps, same
    void **kpools;       // [L]  device copies of the pool pointers
    void **vpools;       // [L]
    int32_t *dst_table;  // [max_requests * max_blocks] plan: destination blocks
    int32_t *push_list;  // [max_requests * max_blocks] plan: blocks to free, in order
    int32_t *counters;   // [4]  plan: pops, pushes; [2] the compaction's own status
    int32_t *occ;        // [num_blocks] plan: holders of a replaced block in this call
    int32_t *last;       // [num_blocks] plan: last (request, block) entry of such a block
    int32_t *rowmark;    // [max_requests] generation stamps (duplicate-row check)
    float *dec_part;     // decode split partials
    size_t dec_part_floats;
    // slot reservation (zp_append_slots) keeps its own scratch
    int32_t *ap_call;     // [1]  status of the reservation call in flight
    int32_t *ap_counters; // [4]  pops, triggers, free count after the pops
    int32_t *ap_rowmark;  // [max_requests] generation stamps
    int32_t *ap_occ;      // [num_blocks] writers of a block in this call
    int32_t *ap_last;     // [num_blocks] last writer of a block in this call
    int4 *ap_plan;        // [max_requests] tail block, fresh block, rows to copy, trigger slot
};

// ------------------------------------------------------------ launch args
// The plan and finalize kernels serve both compressions: at N_max full
// blocks (M = N, every request exactly N*b tokens) and at admission (prefill:
// M = the table stride, N*b <= T <= M*b, blocks N .. of a request released).
struct PlanArgs {
    const int32_t *tables;
    int32_t stride, num_rows;
    const int32_t *lengths;
    const int32_t *req_idx;
    int32_t R, N, M, prefill, num_blocks;
    const int32_t *refcount;
    const int32_t *free_ids;
    const int32_t *free_count;
    int32_t capacity;
    Workspace ws;
};

struct FinalizeArgs {
    int32_t *tables;
    int32_t stride;
    int32_t *lengths;
    const int32_t *req_idx;
    int32_t R, N, M, prefill;
    int32_t *refcount;
    int32_t *free_ids;
    int32_t *free_count;
    Workspace ws;
};

struct CompressArgs {
    const CUtensorMap *kmaps;
    void *const *kpools;
    void *const *vpools;
    const int32_t *tables;
    int32_t stride;
    const int32_t *req_idx;
    const int32_t *dst_table;
    const __nv_bfloat16 *window_q;
    float *scores_out;
    int32_t *kept_out;
    int32_t *call;   // the plan's verdict: only the plan writes it
    int32_t *cstat;  // the compaction's own status (a bounded wait that gave up)
    int32_t *sticky;
    uint32_t *smwave;  // Workspace::smwave (null: no pairing)
    int32_t L, Hkv, Hq, R, N, w, rows, cs;
    int32_t num_rows, num_blocks;  // bounds for reads made before the plan's verdict
    float lambda;
    float inv_rows;       // 1 / (w * G)
    float logit_scale;    // log2(e) / sqrt(d): logits are kept in base 2
};

struct DecodeArgs {
    const CUtensorMap *kmap;
    const CUtensorMap *vmap;
    const __nv_bfloat16 *q;
    const int32_t *tables;
    int32_t stride, num_rows;
    const int32_t *lengths;
    const int32_t *req_idx;
    int32_t R, Hkv, Hq, num_blocks;
    int32_t splits, bps;  // splits per (request, kv head), blocks per split
    float logit_scale;    // scale * log2(e)
    __nv_bfloat16 *out;
    float *part;          // [R][Hq][splits][2 + d] (m, l, o[d]) when splits > 1
    int32_t *sticky;
    // launches that take the maps by value (launch_decode_mapv): the K and V
    // tensor maps in the kernel's parameter space, for a caller with no
    // device memory to hold them; kmap / vmap are then unused
    CUtensorMap kmap_v, vmap_v;
};

// Compression at admission (zp_prefill.cu); units u = (l*R + r)*Hkv + h.
struct PrefillArgs {
    const CUtensorMap *kmaps;
    void *const *kpools;
    void *const *vpools;
    const int32_t *tables;
    int32_t stride;
    const int32_t *lengths;
    const int32_t *req_idx;
    const int32_t *dst_table;  // [R][stride] from the plan
    const __nv_bfloat16 *window_q;
    float2 *stats;             // [units][NC][kMaxRows] per-chunk (max, sum), base 2
    float *red;                // [units][T_cap]
    float *scores;             // [units][T_cap] (the caller's scores_out when given)
    int32_t *kept;             // [units][(N-1)*b] (the caller's kept_out when given)
    int32_t *call;
    int32_t *sticky;
    int32_t L, Hkv, Hq, R, N, w, rows, T_cap, NC;
    float lambda;
    float inv_rows;
    float logit_scale;
    const CUtensorMap *krmaps, *vrmaps;  // per layer: one pool row per box (row gathers)
};

struct AppendArgs {
    int32_t *tables;
    int32_t stride, num_rows;
    int32_t *lengths;
    const int32_t *req_idx;
    int32_t R, n_max, num_blocks, L, Hkv, d;
    int32_t *refcount;
    const int32_t *free_ids;
    int32_t *free_count;
    int32_t capacity;
    int32_t *trigger_rows;   // nullable
    int32_t *trigger_count;  // nullable
    Workspace ws;
};

struct AppendKvArgs {
    __nv_bfloat16 *kpool, *vpool;
    const __nv_bfloat16 *k_new, *v_new;
    const int32_t *tables;
    int32_t stride, num_rows;
    const int32_t *lengths;
    const int32_t *req_idx;
    int32_t R, Hkv, d, num_blocks;
    int32_t *sticky;
};

// Launchers (defined next to their kernels).
cudaError_t launch_append_slots(const AppendArgs &a, cudaStream_t s);
// Scoring, selection and compaction of a compression at admission.
cudaError_t launch_prefill(const PrefillArgs &a, int d, int mt, int units, cudaStream_t s);
constexpr int kPrefillChunk = 2048;     // tokens per scoring CTA
constexpr int kPrefillMaxTokens = 32768;  // scores of one unit fit in shared memory
cudaError_t launch_append_kv(const AppendKvArgs &a, cudaStream_t s);
cudaError_t launch_plan(const PlanArgs &a, cudaStream_t s);
cudaError_t launch_finalize(const FinalizeArgs &a, cudaStream_t s);
// CTAs per unit of the fused compression kernel for T tokens (0: unsupported).
int compress_cluster_size(int T);
cudaError_t launch_compress(const CompressArgs &a, int d, int mt, int units, cudaStream_t s);
cudaError_t launch_compress_d64(const CompressArgs &a, int mt, int units, cudaStream_t s);
cudaError_t launch_compress_d128(const CompressArgs &a, int mt, int units, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs &a, int d, cudaStream_t s);
cudaError_t launch_decode_mapv(const DecodeArgs &a, int d, cudaStream_t s);
// Splits per (request, kv head) of a decode over `pairs` (request, kv head)
// pairs and tables of bt_stride blocks on `num_sms` SMs; *bps: blocks per split.
int decode_splits(long long pairs, int bt_stride, int num_sms, int *bps);
// The swizzled 2D tensor map of a pool [num_blocks][hkv][b][d] that the
// decode and compression kernels load (box: 64 columns x b rows).
bool encode_pool_map(CUtensorMap *map, const void *pool, int num_blocks, int hkv, int d);
// The same view with a box of one whole row and no swizzle (tile::gather4).
bool encode_row_map(CUtensorMap *map, const void *pool, int num_blocks, int hkv, int d);

// ------------------------------------------------------------ device helpers
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_error(int32_t *word, int32_t code)
{
    atomicCAS(word, 0, code);
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before its predecessor on the stream finishes;
// griddepcontrol.wait blocks until the predecessor grid has completed and its
// memory operations are visible (a no-op when launched without it), and
// launch_dependents lets the successor start once every CTA issued it.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// block scan ----------------------------------------------------------------
// Exclusive prefix sum over the threads of a CTA in thread order.  `scratch`
// holds NW + 1 ints.  Returns the exclusive prefix; `total` gets the sum.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int *scratch, int &total)
{
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        scratch[wi] = x;
    __syncthreads();
    if (wi == 0) {
        int s = lane < NW ? scratch[lane] : 0;
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += y;
        }
        if (lane < NW)
            scratch[lane] = incl - s;
        if (lane == NW - 1)
            scratch[NW] = incl;
    }
    __syncthreads();
    const int res = scratch[wi] + x - v;
    total = scratch[NW];
    __syncthreads();
    return res;
}

// mbarrier ------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Bounded wait on a phase of an mbarrier; false when the bound was hit.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    const uint32_t addr = smem_u32(bar);
    for (uint32_t i = 0; i < kWaitSpins; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}\n"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done)
            return true;
        if (i > 64)
            __nanosleep(64);
    }
    return false;
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA / bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA: 2D tile load global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// TMA row gather: four rows y0..y3 (a box one row high) of a 2D tensor map,
// columns from x, land one after the other at dst; completion counted on an
// mbarrier.
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *map, int x, int y0,
                                            int y1, int y2, int y3, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar))
        : "memory");
}

// Waits until at most N committed bulk groups of this thread still read their
// shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until every committed bulk group of this thread is complete.
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Bulk (untiled) copy global -> shared; 16-byte aligned, size multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every committed bulk copy of this thread has read its source.
__device__ __forceinline__ void bulk_wait_read0()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// L2 cache policies for the copies below.
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int x, int y,
                                                 uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_s2g_hint(void *dst, const void *src, uint32_t bytes,
                                              uint64_t policy)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                 ::"l"(dst), "r"(smem_u32(src)), "r"(bytes), "l"(policy)
                 : "memory");
}

// Plain arrive (no transaction bytes) on a barrier of this CTA.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Arrive on the barrier at a shared::cluster address (another CTA's barrier).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// Bounded wait with cluster-scope acquire (pairs with mbar_arrive_remote).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity)
{
    const uint32_t addr = smem_u32(bar);
    for (uint32_t i = 0; i < kWaitSpins; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}\n"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done)
            return true;
        if (i > 64)
            __nanosleep(64);
    }
    return false;
}

// Barrier over the first `threads` threads of the CTA (named barrier 1).
__device__ __forceinline__ void named_sync(uint32_t threads)
{
    asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

// ldmatrix / mma ---------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `ch` (8 bf16) of row `row` in a [rows][d] bf16
// tile stored as d/64 column panels of [rows][128 B] with the 128-byte
// swizzle (chunk index XOR row % 8) -- the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B into a 1024-byte aligned buffer.
__device__ __forceinline__ uint32_t swz(int row, int ch, int rows)
{
    return static_cast<uint32_t>((ch >> 3) * rows * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// cluster --------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync()
{
    cluster_arrive();
    cluster_wait();
}

// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void *local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float2 ld_dsmem_f32x2(uint32_t addr)
{
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

// Starts moving [p, p + bytes) from global memory into L2 (no completion).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t ld_dsmem_u64(uint32_t addr)
{
    uint64_t v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ int32_t ld_dsmem_s32(uint32_t addr)
{
    int32_t v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// global / shared 16-byte moves ------------------------------------------------
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_global_v4(void *p, uint4 v)
{
    asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// 2^x by the PTX instruction ex2.approx.ftz.f32 (relative error about 2^-22,
// subnormal arguments and results flushed to zero, 2^-inf = +0): the
// exponentials of the online softmax, whose sums tolerate both.
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t sm_id()
{
    uint32_t v;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
    return v;
}

// fp32 -> u32 map that preserves order (-0.0 sorts just below +0.0).
__device__ __forceinline__ uint32_t f32_order(float f)
{
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

#endif  // __CUDACC__

}  // namespace zp
