// zp_blocks.cu -- whole-request block allocation, release and fork.
//
// "Paged KV cache and continuous batching for LLMs" ("How it works"): blocks
// are taken from the pool only as a request's tokens need them, a block's
// reference counter counts the tables that point at it, finished (or
// preempted) requests leave the batch and give their blocks back, and
// parallel samples of one prompt share its blocks.
//
// Each call is one launch of one CTA: every check first, then -- only if all
// pass -- every write, so a failed call changes nothing.  Pops and pushes keep
// the order of a sequential pass over (request, block): block scans over
// per-thread contiguous ranges number them.
#include "zp_aux.cuh"

namespace zp {

struct RowsArgs {
    int32_t *tables;
    int32_t stride, num_rows;
    int32_t *lengths;
    const int32_t *req_idx;
    const int32_t *counts;  // alloc only
    int32_t R, num_blocks;
    int32_t *refcount;
    int32_t *free_ids;
    int32_t *free_count;
    int32_t capacity;
    Workspace ws;
};

// Advances the generation of the duplicate-row stamps (thread 0, once per call).
__device__ __forceinline__ int row_stamp_gen(const RowsArgs &a)
{
    const int g = a.ws.gens[1];
    const int ng = g >= 0x7ffffff0 ? 1 : g + 1;
    a.ws.gens[1] = ng;
    return ng;
}

__global__ void __launch_bounds__(kPlanThreads) zp_alloc_rows_kernel(const RowsArgs a)
{
    __shared__ int s_err, s_fc, s_gen;
    __shared__ int s_scan[kPlanThreads / 32 + 1];
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_gen = row_stamp_gen(a);
        s_err = 0;
        s_fc = *a.free_count;
        if (s_fc < 0 || s_fc > a.capacity)
            s_err = ZP_ERR_DEVICE_CHECK;
    }
    __syncthreads();
    const int fc = s_fc;
    const int per = (a.R + kPlanThreads - 1) / kPlanThreads;
    const int i0 = min(a.R, tid * per), i1 = min(a.R, i0 + per);
    int my_need = 0;
    for (int i = i0; i < i1; ++i) {
        const int row = a.req_idx ? a.req_idx[i] : i;
        const int n = a.counts[i];
        if (row < 0 || row >= a.num_rows || n < 0 || n > a.stride * kBlk) {
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
            continue;
        }
        if (atomicExch(&a.ws.ap_rowmark[row], s_gen) == s_gen || a.lengths[row] != 0)
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
        const int nb = (n + kBlk - 1) / kBlk;
        for (int p = 0; p < nb; ++p)
            if (a.tables[(size_t)row * a.stride + p] >= 0)
                atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
        my_need += nb;
    }
    int need;
    const int k0 = block_excl_scan<kPlanThreads>(my_need, s_scan, need);
    if (tid == 0 && need > fc)
        atomicCAS(&s_err, 0, ZP_ERR_OUT_OF_BLOCKS);
    __syncthreads();
    if (s_err == 0) {
        // the k-th block needed pops free_ids[fc - 1 - k]
        for (int k = k0; k < k0 + my_need; ++k) {
            const int t = a.free_ids[fc - 1 - k];
            if (t < 0 || t >= a.num_blocks || a.refcount[t] != 0)
                atomicCAS(&s_err, 0, ZP_ERR_DEVICE_CHECK);
        }
    }
    __syncthreads();
    if (s_err != 0) {
        if (tid == 0)
            set_error(a.ws.sticky, s_err);
        return;
    }
    int k = k0;
    for (int i = i0; i < i1; ++i) {
        const int row = a.req_idx ? a.req_idx[i] : i;
        const int n = a.counts[i];
        const int nb = (n + kBlk - 1) / kBlk;
        for (int p = 0; p < nb; ++p, ++k) {
            const int t = a.free_ids[fc - 1 - k];
            a.refcount[t] = 1;
            a.tables[(size_t)row * a.stride + p] = t;
        }
        a.lengths[row] = n;
    }
    if (tid == 0)
        *a.free_count = fc - need;
}

__global__ void __launch_bounds__(kPlanThreads) zp_release_rows_kernel(const RowsArgs a)
{
    __shared__ int s_err, s_fc, s_gen;
    __shared__ int s_scan[kPlanThreads / 32 + 1];
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_gen = row_stamp_gen(a);
        s_err = 0;
        s_fc = *a.free_count;
        if (s_fc < 0 || s_fc > a.capacity)
            s_err = ZP_ERR_DEVICE_CHECK;
    }
    __syncthreads();
    const int fc = s_fc;
    for (int i = tid; i < a.R; i += kPlanThreads) {
        const int row = a.req_idx ? a.req_idx[i] : i;
        if (row < 0 || row >= a.num_rows) {
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
            continue;
        }
        if (atomicExch(&a.ws.ap_rowmark[row], s_gen) == s_gen)
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
    }
    __syncthreads();
    if (s_err != 0) {
        if (tid == 0)
            set_error(a.ws.sticky, s_err);
        return;
    }

    // entries e = i * stride + p, thread-contiguous; holders of each block
    const int E = a.R * a.stride;
    const int per = (E + kPlanThreads - 1) / kPlanThreads;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    auto blk_of = [&](int e) {
        const int i = e / a.stride, p = e - i * a.stride;
        const int row = a.req_idx ? a.req_idx[i] : i;
        return a.tables[(size_t)row * a.stride + p];
    };
    int *occ = a.ws.ap_occ, *last = a.ws.ap_last;
    for (int e = e0; e < e1; ++e) {
        const int blk = blk_of(e);
        if (blk >= a.num_blocks)
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
        else if (blk >= 0) {
            occ[blk] = 0;
            last[blk] = -1;
        }
    }
    __syncthreads();
    for (int e = e0; e < e1; ++e) {
        const int blk = blk_of(e);
        if (blk >= 0 && blk < a.num_blocks) {
            atomicAdd(&occ[blk], 1);
            atomicMax(&last[blk], e);
        }
    }
    __syncthreads();
    int my_push = 0;
    for (int e = e0; e < e1; ++e) {
        const int blk = blk_of(e);
        if (blk >= 0 && blk < a.num_blocks && last[blk] == e) {
            const int rc = a.refcount[blk];
            if (occ[blk] > rc)
                atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);  // more holders than references
            my_push += occ[blk] == rc;
        }
    }
    int pushes;
    int pos = block_excl_scan<kPlanThreads>(my_push, s_scan, pushes);
    if (tid == 0 && s_err == 0 && fc + pushes > a.capacity)
        atomicCAS(&s_err, 0, ZP_ERR_DEVICE_CHECK);
    __syncthreads();
    if (s_err != 0) {
        if (tid == 0)
            set_error(a.ws.sticky, s_err);
        return;
    }
    // a block loses all its released references at its last holder and is
    // pushed there when that empties it (the order of a sequential pass)
    for (int e = e0; e < e1; ++e) {
        const int blk = blk_of(e);
        if (blk >= 0 && last[blk] == e) {
            const int left = a.refcount[blk] - occ[blk];
            a.refcount[blk] = left;
            if (left == 0)
                a.free_ids[fc + pos++] = blk;
        }
    }
    __syncthreads();  // every entry read before any is cleared
    for (int e = e0; e < e1; ++e) {
        const int i = e / a.stride, p = e - i * a.stride;
        const int row = a.req_idx ? a.req_idx[i] : i;
        a.tables[(size_t)row * a.stride + p] = -1;
    }
    for (int i = tid; i < a.R; i += kPlanThreads)
        a.lengths[a.req_idx ? a.req_idx[i] : i] = 0;
    if (tid == 0)
        *a.free_count = fc + pushes;
}

// Rows dst[i] become copies of rows src[i]: same entries, same length, one
// more reference per block entry (atomics: several forks may share a block).
__global__ void __launch_bounds__(kPlanThreads) zp_fork_rows_kernel(const RowsArgs a,
                                                                    const int32_t *src,
                                                                    const int32_t *dst, int n)
{
    __shared__ int s_err, s_gen;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_gen = row_stamp_gen(a);
        s_err = 0;
    }
    __syncthreads();
    for (int i = tid; i < n; i += kPlanThreads) {
        const int s = src[i], d = dst[i];
        if (s < 0 || s >= a.num_rows || d < 0 || d >= a.num_rows || s == d) {
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
            continue;
        }
        if (atomicExch(&a.ws.ap_rowmark[d], s_gen) == s_gen || a.lengths[d] != 0)
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
    }
    __syncthreads();
    // every (pair, entry): destinations empty, sources valid and referenced;
    // no destination is also a source of this call
    for (int e = tid; e < n * a.stride && s_err == 0; e += kPlanThreads) {
        const int i = e / a.stride, p = e - i * a.stride;
        const int s = src[i], d = dst[i];
        if (p == 0 && a.ws.ap_rowmark[s] == s_gen)
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
        const int blk = a.tables[(size_t)s * a.stride + p];
        if (a.tables[(size_t)d * a.stride + p] >= 0 || blk >= a.num_blocks ||
            (blk >= 0 && a.refcount[blk] < 1))
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
    }
    __syncthreads();
    if (s_err != 0) {
        if (tid == 0)
            set_error(a.ws.sticky, s_err);
        return;
    }
    for (int e = tid; e < n * a.stride; e += kPlanThreads) {
        const int i = e / a.stride, p = e - i * a.stride;
        const int blk = a.tables[(size_t)src[i] * a.stride + p];
        a.tables[(size_t)dst[i] * a.stride + p] = blk;
        if (blk >= 0)
            atomicAdd(&a.refcount[blk], 1);
    }
    for (int i = tid; i < n; i += kPlanThreads)
        a.lengths[dst[i]] = a.lengths[src[i]];
}

}  // namespace zp

namespace {

zp::RowsArgs rows_args(zp::Workspace ws, int32_t *block_tables, int32_t bt_stride,
                       int32_t num_rows, int32_t *lengths, const int32_t *req_idx, int32_t R,
                       const int32_t *counts, int32_t num_blocks, const zp_block_pool *pool)
{
    zp::RowsArgs a{};
    a.tables = block_tables;
    a.stride = bt_stride;
    a.num_rows = num_rows;
    a.lengths = lengths;
    a.req_idx = req_idx;
    a.counts = counts;
    a.R = R;
    a.num_blocks = num_blocks;
    a.refcount = pool->refcount;
    a.free_ids = pool->free_ids;
    a.free_count = pool->free_count;
    a.capacity = pool->capacity;
    a.ws = ws;
    return a;
}

}  // namespace

namespace zp {

cudaError_t launch_alloc_rows(const Workspace &ws, int32_t *block_tables, int32_t bt_stride,
                              int32_t num_rows, int32_t *lengths, const int32_t *req_idx,
                              int32_t R, const int32_t *counts, int32_t num_blocks,
                              const zp_block_pool *pool, cudaStream_t s)
{
    zp_alloc_rows_kernel<<<1, kPlanThreads, 0, s>>>(
        rows_args(ws, block_tables, bt_stride, num_rows, lengths, req_idx, R, counts, num_blocks,
                  pool));
    return cudaGetLastError();
}

cudaError_t launch_fork_rows(const Workspace &ws, int32_t *block_tables, int32_t bt_stride,
                             int32_t num_rows, int32_t *lengths, const int32_t *src,
                             const int32_t *dst, int32_t n, int32_t num_blocks, int32_t *refcount,
                             cudaStream_t s)
{
    zp_block_pool pool{};
    pool.refcount = refcount;
    zp_fork_rows_kernel<<<1, kPlanThreads, 0, s>>>(
        rows_args(ws, block_tables, bt_stride, num_rows, lengths, nullptr, 0, nullptr, num_blocks,
                  &pool),
        src, dst, n);
    return cudaGetLastError();
}

cudaError_t launch_release_rows(const Workspace &ws, int32_t *block_tables, int32_t bt_stride,
                                int32_t num_rows, int32_t *lengths, const int32_t *req_idx,
                                int32_t R, int32_t num_blocks, const zp_block_pool *pool,
                                cudaStream_t s)
{
    zp_release_rows_kernel<<<1, kPlanThreads, 0, s>>>(
        rows_args(ws, block_tables, bt_stride, num_rows, lengths, req_idx, R, nullptr, num_blocks,
                  pool));
    return cudaGetLastError();
}

}  // namespace zp
