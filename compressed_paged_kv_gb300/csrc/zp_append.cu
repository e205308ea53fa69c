// zp_append.cu -- decode-side slot reservation and new-token writes.
//
// "Paged KV cache and continuous batching for LLMs" ("How it works"): a
// request's next token goes into its last block; a block is taken from the
// free stack only when the previous ones are full; a request about to write
// into a shared block (refcount > 1) first copies it to a fresh block and
// drops one reference to the original (block-level copy-on-write).  Zipage
// (gist.science, Dutch "Methodologie" §1): a request whose cache holds N_max
// full blocks is due for compression; those rows are listed on the device for
// the next zp_compress.
//
// zp_append_slots is two launches on the caller's stream:
//   zp_append_plan_kernel   1 CTA: checks; the copy-on-write rule, which is
//                           defined request after request, resolved for all
//                           requests at once; pops; trigger slots.  Writes
//                           nothing the caller owns.
//   zp_append_apply_kernel  one CTA per listed request: copies the filled
//                           slots of a shared tail block (every layer, kv
//                           head, K and V) into its fresh block with 16-byte
//                           vectors, then commits the table entry, refcounts,
//                           length and trigger row.
// zp_append_kv is one launch per layer: one warp per (request, kv head)
// stores the K and V rows of the new token with 16-byte stores.
//
// The copy-on-write rule in parallel.  Taken request after request, the k-th
// writer (k = 0, 1, ...) of a block whose refcount is c at the start finds
// c - k references and copies iff c - k > 1.  Each writer holds one of the c
// references, so a call has m <= c writers of the block: all of them copy
// when m < c, and all but the last when m == c.  A writer therefore copies
// unless it is the block's last writer in the call AND m == c.
#include "zp_internal.cuh"

namespace zp {

constexpr int kApplyThreads = 256;
constexpr int kKvThreads = 128;

__global__ void __launch_bounds__(kPlanThreads) zp_append_plan_kernel(const AppendArgs a)
{
    __shared__ int s_err;
    __shared__ int s_fc, s_gen;
    __shared__ int s_scan[kPlanThreads / 32 + 1];
    const int tid = threadIdx.x;
    if (tid == 0) {
        const int g = a.ws.gens[1];
        s_gen = g >= 0x7ffffff0 ? 1 : g + 1;
        a.ws.gens[1] = s_gen;
        s_err = 0;
        s_fc = *a.free_count;
        if (s_fc < 0 || s_fc > a.capacity)
            s_err = ZP_ERR_DEVICE_CHECK;
    }
    __syncthreads();
    const int fc = s_fc;
    int4 *plan = a.ws.ap_plan;
    int *occ = a.ws.ap_occ;
    int *last = a.ws.ap_last;

    // thread t owns the contiguous requests [i0, i1), so the scans below
    // number pops and triggers in list order
    const int per = (a.R + kPlanThreads - 1) / kPlanThreads;
    const int i0 = min(a.R, tid * per), i1 = min(a.R, i0 + per);

    // checks; plan[i] = (tail block or -1, position of the new token, -, -)
    for (int i = i0; i < i1; ++i) {
        plan[i] = make_int4(-1, 0, 0, -1);
        const int row = a.req_idx ? a.req_idx[i] : i;
        if (row < 0 || row >= a.num_rows) {
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
            continue;
        }
        if (atomicExch(&a.ws.ap_rowmark[row], s_gen) == s_gen)
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
        const int p = a.lengths[row];
        if (p < 0 || p >= a.stride * kBlk || (a.n_max > 0 && p >= a.n_max * kBlk)) {
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
            continue;
        }
        const int blk = a.tables[(size_t)row * a.stride + p / kBlk];
        if (blk >= a.num_blocks || (blk < 0 && p % kBlk != 0) ||
            (blk >= 0 && a.refcount[blk] < 1)) {
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
            continue;
        }
        plan[i] = make_int4(blk < 0 ? -1 : blk, p, 0, -1);
    }
    __syncthreads();
    if (s_err != 0) {
        if (tid == 0)
            *a.ws.ap_call = s_err;
        return;
    }

    // writers per block and the last of them
    for (int i = i0; i < i1; ++i) {
        const int blk = plan[i].x;
        if (blk >= 0) {
            occ[blk] = 0;
            last[blk] = -1;
        }
    }
    __syncthreads();
    for (int i = i0; i < i1; ++i) {
        const int blk = plan[i].x;
        if (blk >= 0) {
            atomicAdd(&occ[blk], 1);
            atomicMax(&last[blk], i);
        }
    }
    __syncthreads();

    auto needs_block = [&](int i, int blk) {
        return blk < 0 || !(last[blk] == i && occ[blk] == a.refcount[blk]);
    };
    const int trig_len = a.n_max > 0 ? a.n_max * kBlk : -1;
    int my_need = 0, my_trig = 0;
    for (int i = i0; i < i1; ++i) {
        const int4 e = plan[i];
        if (e.x >= 0 && occ[e.x] > a.refcount[e.x])
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);  // more writers than references
        my_need += needs_block(i, e.x);
        my_trig += e.y + 1 == trig_len;
    }
    int pops, trigs;
    int k = block_excl_scan<kPlanThreads>(my_need, s_scan, pops);
    int t = block_excl_scan<kPlanThreads>(my_trig, s_scan, trigs);
    if (tid == 0 && pops > fc)
        atomicCAS(&s_err, 0, ZP_ERR_OUT_OF_BLOCKS);
    __syncthreads();
    if (s_err != 0) {
        if (tid == 0)
            *a.ws.ap_call = s_err;
        return;
    }

    // plan[i] = (tail block or -1, fresh block or -1, rows to copy, trigger slot or -1);
    // the k-th request needing a block pops free_ids[fc - 1 - k]
    for (int i = i0; i < i1; ++i) {
        const int4 e = plan[i];
        int fresh = -1, rows = 0;
        if (needs_block(i, e.x)) {
            fresh = a.free_ids[fc - 1 - k];
            ++k;
            if (fresh < 0 || fresh >= a.num_blocks || a.refcount[fresh] != 0)
                atomicCAS(&s_err, 0, ZP_ERR_DEVICE_CHECK);
            rows = e.x >= 0 ? e.y % kBlk : 0;
        }
        const int trig = e.y + 1 == trig_len ? t++ : -1;
        plan[i] = make_int4(e.x, fresh, rows, trig);
    }
    __syncthreads();
    if (tid == 0) {
        a.ws.ap_counters[0] = pops;
        a.ws.ap_counters[1] = trigs;
        a.ws.ap_counters[2] = fc - pops;
        *a.ws.ap_call = s_err;
    }
}

__global__ void __launch_bounds__(kApplyThreads) zp_append_apply_kernel(const AppendArgs a)
{
    const int st = *(volatile int32_t *)a.ws.ap_call;
    if (st != 0) {
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            set_error(a.ws.sticky, st);
            if (a.trigger_count)
                *a.trigger_count = 0;
        }
        return;
    }
    const int i = blockIdx.x;
    const int4 e = a.ws.ap_plan[i];

    // copy-on-write: slots 0 .. rows-1 of every (layer, kv head, K/V) slab
    if (e.z > 0) {
        const int vpr = a.d / 8;  // 16-byte vectors per token row
        const int per_slab = e.z * vpr;
        const int total = a.L * a.Hkv * 2 * per_slab;
        const size_t slab = (size_t)kBlk * vpr;
        for (int v = threadIdx.x; v < total; v += kApplyThreads) {
            int q = v / per_slab;
            const int off = v - q * per_slab;
            const int kv = q & 1;
            q >>= 1;
            const int h = q % a.Hkv, l = q / a.Hkv;
            uint4 *pool = static_cast<uint4 *>(kv ? a.ws.vpools[l] : a.ws.kpools[l]);
            const uint4 x = ld_global_nc_v4(pool + ((size_t)e.x * a.Hkv + h) * slab + off);
            pool[((size_t)e.y * a.Hkv + h) * slab + off] = x;
        }
    }
    if (threadIdx.x == 0) {
        const int row = a.req_idx ? a.req_idx[i] : i;
        const int p = a.lengths[row];
        if (e.y >= 0) {
            a.tables[(size_t)row * a.stride + p / kBlk] = e.y;
            a.refcount[e.y] = 1;
            if (e.x >= 0)
                atomicSub(&a.refcount[e.x], 1);
        }
        a.lengths[row] = p + 1;
        if (e.w >= 0 && a.trigger_rows)
            a.trigger_rows[e.w] = row;
        if (i == 0) {
            *a.free_count = a.ws.ap_counters[2];
            if (a.trigger_count)
                *a.trigger_count = a.ws.ap_counters[1];
        }
    }
}

__global__ void __launch_bounds__(kKvThreads) zp_append_kv_kernel(const AppendKvArgs a)
{
    pdl_wait();  // launched early: the reservation's writes are visible from here
    pdl_launch_dependents();
    const int warp = (blockIdx.x * kKvThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= a.R * a.Hkv)
        return;
    const int i = warp / a.Hkv, h = warp - i * a.Hkv;
    const int row = a.req_idx ? a.req_idx[i] : i;
    bool ok = row >= 0 && row < a.num_rows;
    const int p = ok ? a.lengths[row] - 1 : -1;
    ok = ok && p >= 0 && p < a.stride * kBlk;
    const int blk = ok ? a.tables[(size_t)row * a.stride + p / kBlk] : -1;
    if (!ok || blk < 0 || blk >= a.num_blocks) {
        if (lane == 0)
            set_error(a.sticky, ZP_ERR_DEVICE_CHECK);
        return;
    }
    const int vpr = a.d / 8;  // 16-byte vectors per token row: lanes [0, vpr) K, [vpr, 2 vpr) V
    const size_t dst = (((size_t)blk * a.Hkv + h) * kBlk + p % kBlk) * vpr;
    const size_t src = ((size_t)i * a.Hkv + h) * vpr;
    if (lane < vpr)
        reinterpret_cast<uint4 *>(a.kpool)[dst + lane] =
            ld_global_nc_v4(reinterpret_cast<const uint4 *>(a.k_new) + src + lane);
    else if (lane < 2 * vpr)
        reinterpret_cast<uint4 *>(a.vpool)[dst + lane - vpr] =
            ld_global_nc_v4(reinterpret_cast<const uint4 *>(a.v_new) + src + lane - vpr);
}

cudaError_t launch_append_slots(const AppendArgs &a, cudaStream_t s)
{
    zp_append_plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
    zp_append_apply_kernel<<<static_cast<unsigned>(a.R), kApplyThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_append_kv(const AppendKvArgs &a, cudaStream_t s)
{
    const long long threads = static_cast<long long>(a.R) * a.Hkv * 32;
    const unsigned grid = static_cast<unsigned>((threads + kKvThreads - 1) / kKvThreads);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kKvThreads, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, zp_append_kv_kernel, a);
}

}  // namespace zp
