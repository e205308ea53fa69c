// zp_compress.cu -- compression of full requests: plan, fused score/select/
// compact, finalize.
//
// Method: "Zipage: Maintain High Request Concurrency for LLM Reasoning through
// Compressed PagedAttention" (gist.science summaries).  Dutch "Methodologie"
// §1 (N_max blocks, trigger on a full last block, compaction into the first
// N_max-1 blocks, the last block reserved), §3 (shared prefixes compress into
// new target blocks), §5 (Lightning Redundancy Score: similarity only inside a
// block); Korean "방법론" A (token-wise eviction per layer and head, the
// observation window of the last w queries, always kept), C (target blocks,
// refcounts maintained), E (O(N b^2) redundancy).
//
// One compression call is three launches on the caller's stream:
//   zp_plan_kernel      1 CTA: validates, picks destination blocks, computes
//                       the refcount/free-stack update; writes nothing the
//                       caller owns.
//   zp_compress_stream_kernel  (zp_compress_stream.cuh) one thread-block
//                       cluster of `cs` CTAs per unit
//                       (request, layer, kv head); CTA c owns tokens
//                       [c*TPC, (c+1)*TPC).  K chunk -> shared memory by TMA
//                       (128B swizzle); window logits and the intra-block
//                       Gram on the tensor cores (mma.sync bf16, fp32
//                       accumulate); softmax statistics and the b lowest
//                       scores (warp radix select on the fp32 score bits,
//                       merged per CTA and then per cluster) exchanged over
//                       distributed shared memory; kept rows scattered to
//                       their destination slots.
//   zp_finalize_kernel  1 CTA: commits tables, lengths, refcounts, free stack.
#include "zp_internal.cuh"

namespace zp {

// ================================================================== plan

__global__ void __launch_bounds__(kPlanThreads) zp_plan_kernel(const PlanArgs a)
{
    // the fused kernel may start now: it reads nothing of this plan before
    // its own griddepcontrol.wait
    pdl_launch_dependents();
    __shared__ int s_err;
    __shared__ int s_fc, s_gen;
    __shared__ int s_scan[kPlanThreads / 32 + 1];
    const int tid = threadIdx.x;
    if (tid == 0) {
        a.ws.counters[2] = 0;  // the compaction's status, set by it only on a failed wait
        const int g = a.ws.gens[0];
        s_gen = g >= 0x7ffffff0 ? 1 : g + 1;
        a.ws.gens[0] = s_gen;
        s_err = 0;
        s_fc = *a.free_count;
        if (s_fc < 0 || s_fc > a.capacity)
            s_err = ZP_ERR_DEVICE_CHECK;
    }
    __syncthreads();
    const int fc = s_fc;

    // rows: in range, distinct, full (the trigger needs N_max full blocks;
    // at admission at least N_max*b tokens, within the table row)
    for (int r = tid; r < a.R; r += kPlanThreads) {
        const int row = a.req_idx ? a.req_idx[r] : r;
        if (row < 0 || row >= a.num_rows) {
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
            continue;
        }
        if (atomicExch(&a.ws.rowmark[row], s_gen) == s_gen)
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
        const int len = a.lengths[row];
        if (a.prefill ? (len < a.N * kBlk || len > a.stride * kBlk) : len != a.N * kBlk)
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
    }
    __syncthreads();
    if (s_err != 0) {
        if (tid == 0)
            *a.ws.call = s_err;
        return;
    }

    // destinations: refcount 1 -> in place, > 1 -> pop a fresh target.  The
    // k-th needing entry in (request, block) order pops free_ids[fc-1-k].
    // Entries at block N_max and beyond (admission only) are released: their
    // destination is -1.  Entries past a request's blocks are not entries.
    // Thread t owns the contiguous entries [t*per, (t+1)*per): its loads are
    // independent, and one block scan orders the pops.
    const int E = a.R * a.M;
    const int per = (E + kPlanThreads - 1) / kPlanThreads;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    auto src_of = [&](int e) {
        const int r = e / a.M, p = e - r * a.M;
        const int row = a.req_idx ? a.req_idx[r] : r;
        return a.tables[(size_t)row * a.stride + p];
    };
    // 0: not an entry, 1: destination block (p < N), 2: released (p >= N)
    auto kind_of = [&](int e) {
        if (!a.prefill)
            return 1;
        const int r = e / a.M, p = e - r * a.M;
        const int row = a.req_idx ? a.req_idx[r] : r;
        const int nblk = (a.lengths[row] + kBlk - 1) / kBlk;
        return p >= nblk ? 0 : p < a.N ? 1 : 2;
    };
    int my_need = 0;
#pragma unroll 8
    for (int e = e0; e < e1; ++e) {
        const int kind = kind_of(e);
        if (kind == 0)
            continue;
        const int blk = src_of(e);
        if (blk < 0 || blk >= a.num_blocks) {
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
            continue;
        }
        const int rc = a.refcount[blk];
        if (rc < 1)
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
        my_need += kind == 1 && rc > 1;
    }
    int pops;
    int k = block_excl_scan<kPlanThreads>(my_need, s_scan, pops);
    if (s_err == 0 && pops > fc) {
        if (tid == 0)
            atomicCAS(&s_err, 0, ZP_ERR_OUT_OF_BLOCKS);
    }
    __syncthreads();
    if (s_err != 0) {
        if (tid == 0)
            *a.ws.call = s_err;
        return;
    }
#pragma unroll 8
    for (int e = e0; e < e1; ++e) {
        const int kind = kind_of(e);
        const int blk = src_of(e);
        int dst = kind == 2 ? -1 : blk;
        if (kind == 1 && a.refcount[blk] > 1) {
            dst = a.free_ids[fc - 1 - k];
            ++k;
            if (dst < 0 || dst >= a.num_blocks || a.refcount[dst] != 0)
                atomicCAS(&s_err, 0, ZP_ERR_DEVICE_CHECK);
        }
        a.ws.dst_table[e] = dst;
    }
    __syncthreads();
    if (s_err != 0 || (pops == 0 && !a.prefill)) {
        // nothing shared: no reference is released, nothing is pushed
        if (tid == 0) {
            a.ws.counters[0] = pops;
            a.ws.counters[1] = 0;
            *a.ws.call = s_err;
        }
        return;
    }

    // released blocks: a replaced block loses one reference per holder in this
    // call; it is freed at its last holder when that empties it.
    for (int e = e0; e < e1; ++e) {
        const int src = src_of(e);
        if (a.ws.dst_table[e] != src) {
            a.ws.occ[src] = 0;
            a.ws.last[src] = -1;
        }
    }
    __syncthreads();
    for (int e = e0; e < e1; ++e) {
        const int src = src_of(e);
        if (a.ws.dst_table[e] != src) {
            atomicAdd(&a.ws.occ[src], 1);
            atomicMax(&a.ws.last[src], e);
        }
    }
    __syncthreads();
    int my_push = 0;
    for (int e = e0; e < e1; ++e) {
        const int src = src_of(e);
        if (a.ws.dst_table[e] != src && a.ws.last[src] == e) {
            const int occ = a.ws.occ[src], rc = a.refcount[src];
            if (occ > rc)
                atomicCAS(&s_err, 0, ZP_ERR_DEVICE_CHECK);
            my_push += occ == rc;
        }
    }
    int pushes;
    int pos = block_excl_scan<kPlanThreads>(my_push, s_scan, pushes);
    for (int e = e0; e < e1; ++e) {
        const int src = src_of(e);
        if (a.ws.dst_table[e] != src && a.ws.last[src] == e && a.ws.occ[src] == a.refcount[src])
            a.ws.push_list[pos++] = src;
    }
    __syncthreads();
    if (tid == 0) {
        if (fc - pops + pushes > a.capacity)
            atomicCAS(&s_err, 0, ZP_ERR_DEVICE_CHECK);
        a.ws.counters[0] = pops;
        a.ws.counters[1] = pushes;
        *a.ws.call = s_err;
    }
}

// ============================================================== finalize

__global__ void __launch_bounds__(kPlanThreads) zp_finalize_kernel(const FinalizeArgs a)
{
    __shared__ int s_fc;
    const int tid = threadIdx.x;
    pdl_wait();  // every write of the kernels before it is visible
    for (int i = tid; i < 3 * kSmSlots; i += kPlanThreads)
        a.ws.smwave[i] = 0u;  // the compression kernel's per-SM pairing, for the next call
    int st = *(volatile int32_t *)a.ws.call;
    if (st == 0)
        st = *(volatile int32_t *)(a.ws.counters + 2);
    if (st != 0) {
        if (tid == 0)
            set_error(a.ws.sticky, st);
        return;
    }
    if (tid == 0)
        s_fc = *a.free_count;
    __syncthreads();
    const int pops = a.ws.counters[0], pushes = a.ws.counters[1];
    // nothing shared and nothing released: tables unchanged
    const int E = pops > 0 || a.prefill ? a.R * a.M : 0;
    for (int e = tid; e < E; e += kPlanThreads) {
        const int r = e / a.M, p = e - r * a.M;
        const int row = a.req_idx ? a.req_idx[r] : r;
        int32_t *slot = a.tables + (size_t)row * a.stride + p;
        const int src = *slot, dst = a.ws.dst_table[e];
        if (dst != src) {
            if (a.ws.last[src] == e)
                a.refcount[src] -= a.ws.occ[src];
            if (dst >= 0)
                a.refcount[dst] = 1;
            *slot = dst;
        }
    }
    for (int r = tid; r < a.R; r += kPlanThreads) {
        const int row = a.req_idx ? a.req_idx[r] : r;
        a.lengths[row] = (a.N - 1) * kBlk;
    }
    const int top = s_fc - pops;
    for (int i = tid; i < pushes; i += kPlanThreads)
        a.free_ids[top + i] = a.ws.push_list[i];
    __syncthreads();
    if (tid == 0)
        *a.free_count = top + pushes;
}

// ============================================================== launchers

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t s)
{
    zp_plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeArgs &a, cudaStream_t s)
{
    // launched early (programmatic serialisation); it waits at its start
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kPlanThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, zp_finalize_kernel, a);
}

int compress_cluster_size(int T)
{
    // the fewest CTAs per unit with at most ZP_STREAM_MAX_TC tokens each, every chunk a
    // whole number of 128-token stages
#ifndef ZP_STREAM_MAX_TC
#define ZP_STREAM_MAX_TC 2048
#endif
    for (int cs = 1; cs <= kMaxCluster; ++cs)
        if (T % cs == 0 && T / cs <= ZP_STREAM_MAX_TC && (T / cs) % 128 == 0)
            return cs;
    return 0;
}

cudaError_t launch_compress(const CompressArgs &a, int d, int mt, int units, cudaStream_t s)
{
    if (d == 64)
        return launch_compress_d64(a, mt, units, s);
    if (d == 128)
        return launch_compress_d128(a, mt, units, s);
    return cudaErrorInvalidValue;
}

}  // namespace zp
