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
//   zp_compress_kernel  one thread-block cluster of `cs` CTAs per unit
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

// ============================================================ block scans

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

// ================================================================== plan

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) zp_plan_kernel(const PlanArgs a)
{
    __shared__ int s_err;
    __shared__ int s_fc;
    __shared__ int s_scan[kPlanThreads / 32 + 1];
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_err = 0;
        s_fc = *a.free_count;
        if (s_fc < 0 || s_fc > a.capacity)
            s_err = ZP_ERR_DEVICE_CHECK;
    }
    __syncthreads();
    const int fc = s_fc;

    // rows: in range, distinct, full (the trigger needs N_max full blocks)
    for (int r = tid; r < a.R; r += kPlanThreads) {
        const int row = a.req_idx ? a.req_idx[r] : r;
        if (row < 0 || row >= a.num_rows) {
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
            continue;
        }
        if (atomicExch(&a.ws.rowmark[row], a.gen) == a.gen)
            atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
        if (a.lengths[row] != a.N * kBlk)
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
    const int E = a.R * a.N;
    int pops = 0;
    for (int base = 0; base < E; base += kPlanThreads) {
        const int e = base + tid;
        int need = 0, blk = -1;
        if (e < E) {
            const int r = e / a.N, p = e - r * a.N;
            const int row = a.req_idx ? a.req_idx[r] : r;
            blk = a.tables[(size_t)row * a.stride + p];
            if (blk < 0 || blk >= a.num_blocks) {
                atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
                blk = -1;
            } else {
                const int rc = a.refcount[blk];
                if (rc < 1)
                    atomicCAS(&s_err, 0, ZP_ERR_INVALID_ARG);
                need = rc > 1;
            }
        }
        int total;
        const int k = block_excl_scan<kPlanThreads>(need, s_scan, total) + pops;
        if (blk >= 0) {
            int dst = blk;
            if (need) {
                if (k >= fc) {
                    atomicCAS(&s_err, 0, ZP_ERR_OUT_OF_BLOCKS);
                } else {
                    dst = a.free_ids[fc - 1 - k];
                    if (dst < 0 || dst >= a.num_blocks || a.refcount[dst] != 0)
                        atomicCAS(&s_err, 0, ZP_ERR_DEVICE_CHECK);
                }
            }
            a.ws.dst_table[e] = dst;
        }
        pops += total;
    }
    __syncthreads();
    if (s_err != 0) {
        if (tid == 0)
            *a.ws.call = s_err;
        return;
    }

    // released blocks: a replaced block loses one reference per holder in this
    // call; it is freed at its last holder when that empties it.
    for (int e = tid; e < E; e += kPlanThreads) {
        const int r = e / a.N, p = e - r * a.N;
        const int row = a.req_idx ? a.req_idx[r] : r;
        const int src = a.tables[(size_t)row * a.stride + p];
        if (a.ws.dst_table[e] != src) {
            a.ws.occ[src] = 0;
            a.ws.last[src] = -1;
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kPlanThreads) {
        const int r = e / a.N, p = e - r * a.N;
        const int row = a.req_idx ? a.req_idx[r] : r;
        const int src = a.tables[(size_t)row * a.stride + p];
        if (a.ws.dst_table[e] != src) {
            atomicAdd(&a.ws.occ[src], 1);
            atomicMax(&a.ws.last[src], e);
        }
    }
    __syncthreads();
    int pushes = 0;
    for (int base = 0; base < E; base += kPlanThreads) {
        const int e = base + tid;
        int flag = 0, src = -1;
        if (e < E) {
            const int r = e / a.N, p = e - r * a.N;
            const int row = a.req_idx ? a.req_idx[r] : r;
            src = a.tables[(size_t)row * a.stride + p];
            if (a.ws.dst_table[e] != src && a.ws.last[src] == e) {
                const int occ = a.ws.occ[src], rc = a.refcount[src];
                if (occ > rc)
                    atomicCAS(&s_err, 0, ZP_ERR_DEVICE_CHECK);
                flag = occ == rc;
            }
        }
        int total;
        const int pos = block_excl_scan<kPlanThreads>(flag, s_scan, total) + pushes;
        if (flag)
            a.ws.push_list[pos] = src;
        pushes += total;
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
    const int st = *(volatile int32_t *)a.ws.call;
    if (st != 0) {
        if (tid == 0)
            set_error(a.ws.sticky, st);
        return;
    }
    if (tid == 0)
        s_fc = *a.free_count;
    __syncthreads();
    const int pops = a.ws.counters[0], pushes = a.ws.counters[1];
    const int E = a.R * a.N;
    for (int e = tid; e < E; e += kPlanThreads) {
        const int r = e / a.N, p = e - r * a.N;
        const int row = a.req_idx ? a.req_idx[r] : r;
        int32_t *slot = a.tables + (size_t)row * a.stride + p;
        const int src = *slot, dst = a.ws.dst_table[e];
        if (dst != src) {
            if (a.ws.last[src] == e)
                a.refcount[src] -= a.ws.occ[src];
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

// ============================================================ fused kernel

// Warp radix select: the k smallest of the 32*KPL distinct 64-bit keys held
// KPL per lane (slot s of lane l is entry l + 32 s), MSB first, one bit per
// step: at each bit the keys with a 0 are counted by ballot; if they cover
// the remaining demand the search continues among them, else all of them are
// taken and it continues among the 1s.  chosen[s] is the ballot mask of the
// selected entries of slot s (the same in every lane).  Entries equal to ~0
// are padding; if any are needed they are taken in entry order.
template <int KPL>
__device__ __forceinline__ void warp_select_smallest(const uint64_t (&key)[KPL], int k,
                                                     uint32_t (&chosen)[KPL])
{
    uint32_t active[KPL];
    int n_active = 0;
#pragma unroll
    for (int s = 0; s < KPL; ++s) {
        active[s] = 0xffffffffu;
        chosen[s] = 0u;
        n_active += 32;
    }
    int need = k;
    for (int bit = 63; bit >= 0 && need > 0 && need < n_active; --bit) {
        uint32_t zeros[KPL];
        int nz = 0;
#pragma unroll
        for (int s = 0; s < KPL; ++s) {
            zeros[s] = __ballot_sync(0xffffffffu, ((key[s] >> bit) & 1ull) == 0ull) & active[s];
            nz += __popc(zeros[s]);
        }
        if (nz >= need) {
#pragma unroll
            for (int s = 0; s < KPL; ++s)
                active[s] = zeros[s];
            n_active = nz;
        } else {
#pragma unroll
            for (int s = 0; s < KPL; ++s) {
                chosen[s] |= zeros[s];
                active[s] &= ~zeros[s];
            }
            need -= nz;
            n_active -= nz;
        }
    }
    if (need > 0 && need >= n_active) {
#pragma unroll
        for (int s = 0; s < KPL; ++s)
            chosen[s] |= active[s];
        need -= n_active;
    }
    // equal (padding) keys left over: take the first `need` in entry order
#pragma unroll
    for (int s = 0; s < KPL; ++s) {
        while (need > 0 && active[s] & ~chosen[s]) {
            const uint32_t m = active[s] & ~chosen[s];
            chosen[s] |= m & (~m + 1u);
            --need;
        }
    }
}

// Writes the selected keys to dst[0..) in entry order (slot, then lane).
template <int KPL>
__device__ __forceinline__ void warp_compact_keys(const uint64_t (&key)[KPL],
                                                  const uint32_t (&chosen)[KPL], uint64_t *dst)
{
    const int lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    int base = 0;
#pragma unroll
    for (int s = 0; s < KPL; ++s) {
        if ((chosen[s] >> lane) & 1u)
            dst[base + __popc(chosen[s] & lt)] = key[s];
        base += __popc(chosen[s]);
    }
}

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int D, int TW, int MT>
struct CompressSmem {
    static constexpr int TPC = kWarps * TW * 16;  // tokens per CTA
    static constexpr int NBLK = TPC / kBlk;
    static constexpr int ROWS = MT * 16;
    static constexpr int K_BYTES = TPC * D * 2;
    static constexpr int Q_BYTES = ROWS * D * 2;
    static constexpr int VT_BYTES = kBlk * D * 2;
    static constexpr int off_k = 0;
    static constexpr int off_q = off_k + K_BYTES;
    static constexpr int off_vt = off_q + Q_BYTES;
    static constexpr int off_rowa = off_vt + VT_BYTES;              // float [NW][ROWS]
    static constexpr int off_statm = off_rowa + kWarps * ROWS * 4;  // float [ROWS] (remote-read)
    static constexpr int off_stats = off_statm + ROWS * 4;          // float [ROWS] (remote-read)
    static constexpr int off_gm = off_stats + ROWS * 4;             // float [ROWS]
    static constexpr int off_ginv = off_gm + ROWS * 4;              // float [ROWS]
    static constexpr int off_score = off_ginv + ROWS * 4;           // float [TPC]
    static constexpr int off_red = off_score + TPC * 4;             // float [TPC]
    static constexpr int off_diag = off_red + TPC * 4;              // float [TPC]
    static constexpr int off_doff = off_diag + TPC * 4;             // int [TPC]
    static constexpr int off_cand = off_doff + TPC * 4;             // u64 [NW][b]
    static constexpr int off_pub = off_cand + kWarps * kBlk * 8;    // u64 [b] (remote-read)
    static constexpr int off_ev = off_pub + kBlk * 8;               // int [b]
    static constexpr int off_misc = off_ev + kBlk * 4;              // int [8]
    static constexpr int off_bmove = off_misc + 8 * 4;              // int [NBLK]
    static constexpr int off_bar = (off_bmove + NBLK * 4 + 15) / 16 * 16;  // 2 mbarriers
    static constexpr int BYTES = off_bar + 16;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024 B
};

template <int D, int TW, int MT>
__global__ void __launch_bounds__(kThreads, 1) zp_compress_kernel(const CompressArgs a)
{
    using S = CompressSmem<D, TW, MT>;
    constexpr int TPC = S::TPC, NBLK = S::NBLK, ROWS = S::ROWS;
    constexpr int HALVES = D / 64;
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    constexpr int KPT = (TPC + kThreads - 1) / kThreads;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sK = sm + S::off_k;
    uint8_t *sQ = sm + S::off_q;
    uint8_t *sVt = sm + S::off_vt;
    float *sRowA = reinterpret_cast<float *>(sm + S::off_rowa);
    float *sStatM = reinterpret_cast<float *>(sm + S::off_statm);
    float *sStatS = reinterpret_cast<float *>(sm + S::off_stats);
    float *sGm = reinterpret_cast<float *>(sm + S::off_gm);
    float *sGinv = reinterpret_cast<float *>(sm + S::off_ginv);
    float *sScore = reinterpret_cast<float *>(sm + S::off_score);
    float *sRed = reinterpret_cast<float *>(sm + S::off_red);
    float *sDiag = reinterpret_cast<float *>(sm + S::off_diag);
    int *sDoff = reinterpret_cast<int *>(sm + S::off_doff);
    uint64_t *sCand = reinterpret_cast<uint64_t *>(sm + S::off_cand);
    uint64_t *sPub = reinterpret_cast<uint64_t *>(sm + S::off_pub);
    int *sEv = reinterpret_cast<int *>(sm + S::off_ev);
    int *sMisc = reinterpret_cast<int *>(sm + S::off_misc);
    int *sBMove = reinterpret_cast<int *>(sm + S::off_bmove);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::off_bar);

    const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5;
    const int cs = a.cs;
    const uint32_t crank = cluster_ctarank();
    const int unit = blockIdx.x / cs;
    const int h = unit % a.Hkv;
    const int l = (unit / a.Hkv) % a.L;
    const int r = unit / (a.Hkv * a.L);

    // A failed plan makes the whole grid exit here, uniformly per cluster.
    if (*reinterpret_cast<volatile int32_t *>(a.call) != 0)
        return;

    const int row = a.req_idx ? a.req_idx[r] : r;
    const int32_t *src_row = a.tables + (size_t)row * a.stride;
    const int32_t *dst_row = a.dst_table + (size_t)r * a.N;
    const int T = a.N * kBlk, C = T - a.w;
    const int t0 = static_cast<int>(crank) * TPC;
    const int blk0 = t0 / kBlk;
    const int G = a.Hq / a.Hkv;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    for (int q = tid; q < NBLK; q += kThreads)
        sBMove[q] = 0;
    __syncthreads();

    // ---- loads: K chunk (TMA, swizzled), the V rows of the last block of the
    // chunk (bulk copy; the next CTA may overwrite them in place later), and
    // the window queries (plain loads into the same swizzled layout).
    if (wi == 0) {
        const CUtensorMap *kmap = a.kmaps + l;
        if (lane == 0)
            mbar_arrive_expect_tx(&bars[0], S::K_BYTES + S::VT_BYTES);
        __syncwarp();
        for (int q = lane; q < NBLK; q += 32) {
            const int blk = src_row[blk0 + q];
            const int y = (blk * a.Hkv + h) * kBlk;
#pragma unroll
            for (int hf = 0; hf < HALVES; ++hf)
                tma_load_2d(sK + hf * TPC * 128 + q * kBlk * 128, kmap, hf * 64, y, &bars[0]);
        }
        if (lane == 0) {
            const int blk = src_row[blk0 + NBLK - 1];
            const __nv_bfloat16 *vsrc = static_cast<const __nv_bfloat16 *>(a.vpools[l]) +
                                        ((size_t)blk * a.Hkv + h) * kBlk * D;
            bulk_g2s(sVt, vsrc, S::VT_BYTES, &bars[0]);
        }
    }
    {
        const __nv_bfloat16 *qsrc =
            a.window_q + ((((size_t)l * a.R + r) * a.Hq + (size_t)h * G) * a.w) * D;
        const uint32_t q_base = smem_u32(sQ);
        for (int c = tid; c < ROWS * CPR; c += kThreads) {
            const int rr = c / CPR, ch = c - rr * CPR;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (rr < a.rows)
                v = ld_global_nc_v4(qsrc + (size_t)rr * D + ch * 8);
            st_shared_v4(q_base + swz(rr, ch, ROWS), v);
        }
    }
    bool bad = !mbar_wait(&bars[0], 0);
    bad = __syncthreads_or(bad);

    // ---- window logits (base 2) and the intra-block Gram, on the tensor cores
    float acc[MT][TW][2][4];
    float gram[TW][2][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int tt = 0; tt < TW; ++tt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[mt][tt][nt][e] = 0.f;
#pragma unroll
    for (int tt = 0; tt < TW; ++tt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                gram[tt][nt][e] = 0.f;
    {
        const uint32_t kb_base = smem_u32(sK), qb_base = smem_u32(sQ);
        const int mi = lane >> 3;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t qa[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                ldsm_x4(qb_base + swz(mt * 16 + (mi & 1) * 8 + (lane & 7), ks * 2 + (mi >> 1), ROWS),
                        qa[mt]);
#pragma unroll
            for (int tt = 0; tt < TW; ++tt) {
                const int key0 = (wi * TW + tt) * 16;
                uint32_t kb[4];
                ldsm_x4(kb_base + swz(key0 + (mi >> 1) * 8 + (lane & 7), ks * 2 + (mi & 1), TPC), kb);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    mma_bf16(acc[mt][tt][0], qa[mt][0], qa[mt][1], qa[mt][2], qa[mt][3], kb[0], kb[1]);
                    mma_bf16(acc[mt][tt][1], qa[mt][0], qa[mt][1], qa[mt][2], qa[mt][3], kb[2], kb[3]);
                }
                mma_bf16(gram[tt][0], kb[0], kb[2], kb[1], kb[3], kb[0], kb[1]);
                mma_bf16(gram[tt][1], kb[0], kb[2], kb[1], kb[3], kb[2], kb[3]);
            }
        }
    }

    // scale to base 2 and apply the causal mask of the window rows
    int slot_of[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int rr = mt * 16 + (lane >> 2) + hh * 8;
            slot_of[mt][hh] = rr < a.rows ? rr % a.w : -1;
        }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int tt = 0; tt < TW; ++tt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int slot = slot_of[mt][e >> 1];
                    const int tok = t0 + (wi * TW + tt) * 16 + nt * 8 + (lane & 3) * 2 + (e & 1);
                    float v = acc[mt][tt][nt][e] * a.logit_scale;
                    if (slot >= 0 && tok > C + slot)
                        v = -INFINITY;
                    acc[mt][tt][nt][e] = v;
                }

    // row max over this CTA's keys
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float m = -INFINITY;
#pragma unroll
            for (int tt = 0; tt < TW; ++tt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    m = fmaxf(m, fmaxf(acc[mt][tt][nt][hh * 2], acc[mt][tt][nt][hh * 2 + 1]));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            if ((lane & 3) == 0)
                sRowA[wi * ROWS + mt * 16 + (lane >> 2) + hh * 8] = m;
        }
    __syncthreads();
    if (tid < ROWS) {
        float m = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2)
            m = fmaxf(m, sRowA[w2 * ROWS + tid]);
        sGm[tid] = m;
    }
    __syncthreads();
    // row sum of exp2(l - m_cta)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const float m = sGm[mt * 16 + (lane >> 2) + hh * 8];
            float s = 0.f;
#pragma unroll
            for (int tt = 0; tt < TW; ++tt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    s += exp2f(acc[mt][tt][nt][hh * 2] - m) + exp2f(acc[mt][tt][nt][hh * 2 + 1] - m);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if ((lane & 3) == 0)
                sRowA[wi * ROWS + mt * 16 + (lane >> 2) + hh * 8] = s;
        }

    // Lightning Redundancy Score from the Gram fragments: element e of n-tile
    // nt is G[j][k], j = lane/4 + 8*(e/2), k = 8*nt + 2*(lane%4) + e%2.
#pragma unroll
    for (int tt = 0; tt < TW; ++tt) {
        const int key0 = (wi * TW + tt) * 16;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = (lane >> 2) + (e >> 1) * 8, k = nt * 8 + (lane & 3) * 2 + (e & 1);
                if (j == k)
                    sDiag[key0 + j] = gram[tt][nt][e];
            }
    }
    __syncwarp();
#pragma unroll
    for (int tt = 0; tt < TW; ++tt) {
        const int key0 = (wi * TW + tt) * 16;
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = (lane >> 2) + (e >> 1) * 8, k = nt * 8 + (lane & 3) * 2 + (e & 1);
                const float dk = sDiag[key0 + k];
                const float inv_k = dk > 0.f ? 1.0f / sqrtf(dk) : 0.f;
                if (j != k)
                    rs[e >> 1] += gram[tt][nt][e] * inv_k;
            }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float s = rs[hh];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if ((lane & 3) == 0) {
                const int j = (lane >> 2) + hh * 8;
                const float dj = sDiag[key0 + j];
                const float inv_j = dj > 0.f ? 1.0f / sqrtf(dj) : 0.f;
                sRed[key0 + j] = inv_j * s * (1.0f / (kBlk - 1));
            }
        }
    }
    __syncthreads();
    if (tid < ROWS) {
        float s = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2)
            s += sRowA[w2 * ROWS + tid];
        sStatM[tid] = sGm[tid];
        sStatS[tid] = s;
    }
    cluster_sync();  // (1) per-CTA softmax statistics published

    if (tid < ROWS) {
        // all remote loads first, so they are in flight together
        float mv[kMaxCluster], sv[kMaxCluster];
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c) {
            mv[c] = c < cs ? ld_dsmem_f32(dsmem_addr(sStatM + tid, c)) : -INFINITY;
            sv[c] = c < cs ? ld_dsmem_f32(dsmem_addr(sStatS + tid, c)) : 0.f;
        }
        float m = -INFINITY;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            m = fmaxf(m, mv[c]);
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c)
            if (c < cs)
                s += sv[c] * exp2f(mv[c] - m);
        sGm[tid] = m;
        sGinv[tid] = tid < a.rows ? 1.0f / s : 0.f;
    }
    __syncthreads();

    // importance: mean over window rows of the softmax probabilities; score
#pragma unroll
    for (int tt = 0; tt < TW; ++tt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int ee = 0; ee < 2; ++ee) {
                float s = 0.f;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int rr = mt * 16 + (lane >> 2) + hh * 8;
                        s += exp2f(acc[mt][tt][nt][hh * 2 + ee] - sGm[rr]) * sGinv[rr];
                    }
                s += __shfl_xor_sync(0xffffffffu, s, 4);
                s += __shfl_xor_sync(0xffffffffu, s, 8);
                s += __shfl_xor_sync(0xffffffffu, s, 16);
                if (lane < 4) {
                    const int key = (wi * TW + tt) * 16 + nt * 8 + lane * 2 + ee;
                    sScore[key] = s * a.inv_rows - a.lambda * sRed[key];
                }
            }
    __syncthreads();

    // ---- select: the b lowest candidates under (score ascending, index
    // descending) are evicted.  Each candidate carries a distinct 64-bit key:
    // the order-preserving image of its fp32 score bits above the complement
    // of its index.  A warp radix select (MSB first, one bit per step, by
    // ballot) keeps each warp's b smallest keys, warp 0 keeps the CTA's b
    // smallest of those, and after one cluster barrier warp 0 of every CTA
    // selects the unit's b smallest among the cluster's candidates.
    {
        constexpr int KW = 16 * TW;              // keys per warp
        constexpr int KPL = (KW + 31) / 32;      // keys per lane
        uint64_t key[KPL];
#pragma unroll
        for (int s = 0; s < KPL; ++s) {
            const int kk = lane + 32 * s;
            key[s] = ~0ull;
            if (kk < KW) {
                const int k = wi * KW + kk, tok = t0 + k;
                const uint32_t hi = tok < C ? f32_order(sScore[k]) : 0xffffffffu;
                key[s] = (static_cast<uint64_t>(hi) << 32) | (0xffffffffu - static_cast<uint32_t>(tok));
            }
        }
        uint32_t chosen[KPL];
        warp_select_smallest<KPL>(key, kBlk, chosen);
        warp_compact_keys<KPL>(key, chosen, sCand + wi * kBlk);
    }
    __syncthreads();
    if (wi == 0) {
        uint64_t key[4];
#pragma unroll
        for (int s = 0; s < 4; ++s)
            key[s] = sCand[lane + 32 * s];
        uint32_t chosen[4];
        warp_select_smallest<4>(key, kBlk, chosen);
        warp_compact_keys<4>(key, chosen, sPub);
    }
    cluster_sync();  // (2) each CTA's b candidates published
    if (wi == 0) {
        uint64_t key[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const int e = lane + 32 * s, c = e >> 4;
            key[s] = c < cs ? ld_dsmem_u64(dsmem_addr(sPub + (e & 15), c)) : ~0ull;
        }
        uint32_t chosen[4];
        warp_select_smallest<4>(key, kBlk, chosen);
        warp_compact_keys<4>(key, chosen, sCand);  // the unit's b evicted keys
        __syncwarp();
        if (lane < kBlk) {
            const uint32_t mine = 0xffffffffu - static_cast<uint32_t>(sCand[lane]);
            int rank = 0;
#pragma unroll
            for (int i = 0; i < kBlk; ++i)
                rank += (0xffffffffu - static_cast<uint32_t>(sCand[i])) < mine;
            sEv[rank] = static_cast<int>(mine);
        }
    }
    cluster_arrive();  // no remote shared-memory reads after this point
    __syncthreads();

    {
        const size_t uo = ((size_t)l * a.R + r) * a.Hkv + h;
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
            const int k = tid * KPT + j;
            if (k >= TPC)
                continue;
            const int tok = t0 + k;
            int before = 0;
            bool ev = false;
#pragma unroll
            for (int i = 0; i < kBlk; ++i) {
                const int e = sEv[i];
                before += e < tok;
                ev |= e == tok;
            }
            int doff = -1;
            if (!ev) {
                const int dp = tok - before;
                const int dblk = dst_row[dp >> 4];
                const int sblk = src_row[tok >> 4];
                if (dp != tok || dblk != sblk) {
                    doff = (dblk * a.Hkv + h) * kBlk + (dp & 15);
                    sBMove[k >> 4] = 1;
                }
                if (a.kept_out)
                    a.kept_out[uo * (size_t)(T - kBlk) + dp] = tok;
            }
            sDoff[k] = doff;
            if (a.scores_out)
                a.scores_out[uo * (size_t)T + tok] = (tok < C) ? sScore[k] : INFINITY;
        }
    }
    __syncthreads();

    // ---- compaction.  K rows come from shared memory.  Exactly b tokens are
    // evicted, so destination j reads source kept[j] with j <= kept[j] <= j+b:
    // in-place writes by the next CTA only reach this CTA's last block, whose
    // V rows were staged before the first cluster barrier; every CTA read its
    // K before that barrier too.
    if (!bad) {
        __nv_bfloat16 *kpool = static_cast<__nv_bfloat16 *>(a.kpools[l]);
        const uint32_t kb_base = smem_u32(sK);
        for (int c = tid; c < TPC * CPR; c += kThreads) {
            const int k = c / CPR, ch = c - k * CPR;
            const int doff = sDoff[k];
            if (doff < 0)
                continue;
            const uint4 v = ld_shared_v4(kb_base + swz(k, ch, TPC));
            st_global_v4(kpool + (size_t)doff * D + ch * 8, v);
        }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // V rows of the moved tokens: stage the source blocks (except the last,
    // already staged) into the K buffer, then scatter.
    if (wi == 0) {
        int nv = 0;
        for (int q = lane; q < NBLK - 1; q += 32)
            nv += (!bad && sBMove[q]) ? 1 : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            nv += __shfl_xor_sync(0xffffffffu, nv, o);
        if (lane == 0) {
            sMisc[4] = nv;
            if (nv > 0)
                mbar_arrive_expect_tx(&bars[1], nv * kBlk * D * 2);
        }
        __syncwarp();
        if (nv > 0) {
            for (int q = lane; q < NBLK - 1; q += 32) {
                if (!sBMove[q])
                    continue;
                const int blk = src_row[blk0 + q];
                const __nv_bfloat16 *vsrc = static_cast<const __nv_bfloat16 *>(a.vpools[l]) +
                                            ((size_t)blk * a.Hkv + h) * kBlk * D;
                bulk_g2s(sK + q * kBlk * D * 2, vsrc, kBlk * D * 2, &bars[1]);
            }
        }
    }
    __syncthreads();
    if (sMisc[4] > 0)
        bad |= !mbar_wait(&bars[1], 0);
    bad = __syncthreads_or(bad);
    if (!bad) {
        __nv_bfloat16 *vpool = static_cast<__nv_bfloat16 *>(a.vpools[l]);
        const uint32_t v_base = smem_u32(sK), vt_base = smem_u32(sVt);
        for (int c = tid; c < TPC * CPR; c += kThreads) {
            const int k = c / CPR, ch = c - k * CPR;
            const int doff = sDoff[k];
            if (doff < 0)
                continue;
            const uint32_t src = (k >= TPC - kBlk) ? vt_base + ((k - (TPC - kBlk)) * CPR + ch) * 16
                                                   : v_base + (k * CPR + ch) * 16;
            st_global_v4(vpool + (size_t)doff * D + ch * 8, ld_shared_v4(src));
        }
    } else if (tid == 0) {
        set_error(a.call, ZP_ERR_TIMEOUT);
        set_error(a.sticky, ZP_ERR_TIMEOUT);
    }
    cluster_wait();  // peers may still read this CTA's counts until here
}

// ============================================================== launchers

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t s)
{
    zp_plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeArgs &a, cudaStream_t s)
{
    zp_finalize_kernel<<<1, kPlanThreads, 0, s>>>(a);
    return cudaGetLastError();
}

int compress_tile_words(int T)
{
    // smallest tiles-per-warp (1, 2 or 4) that splits T into <= 8 CTAs
    const int tws[3] = {1, 2, 4};
    for (int i = 0; i < 3; ++i) {
        const int tpc = kWarps * 16 * tws[i];
        if (T % tpc == 0 && T / tpc <= kMaxCluster)
            return tws[i];
    }
    return 0;
}

template <int D, int TW, int MT>
static cudaError_t launch_compress_t(const CompressArgs &a, int units, cudaStream_t s)
{
    using Sm = CompressSmem<D, TW, MT>;
    auto kern = zp_compress_kernel<D, TW, MT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Sm::ALLOC);
    if (err != cudaSuccess)
        return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * a.cs), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Sm::ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int D, int TW>
static cudaError_t dispatch_mt(const CompressArgs &a, int mt, int units, cudaStream_t s)
{
    switch (mt) {
    case 1: return launch_compress_t<D, TW, 1>(a, units, s);
    case 2: return launch_compress_t<D, TW, 2>(a, units, s);
    case 4: return launch_compress_t<D, TW, 4>(a, units, s);
    default: return cudaErrorInvalidValue;
    }
}

template <int D>
static cudaError_t dispatch_tw(const CompressArgs &a, int tw, int mt, int units, cudaStream_t s)
{
    switch (tw) {
    case 1: return dispatch_mt<D, 1>(a, mt, units, s);
    case 2: return dispatch_mt<D, 2>(a, mt, units, s);
    case 4: return dispatch_mt<D, 4>(a, mt, units, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_compress(const CompressArgs &a, int d, int tw, int mt, int units,
                            cudaStream_t s)
{
    if (d == 64)
        return dispatch_tw<64>(a, tw, mt, units, s);
    if (d == 128)
        return dispatch_tw<128>(a, tw, mt, units, s);
    return cudaErrorInvalidValue;
}

}  // namespace zp
