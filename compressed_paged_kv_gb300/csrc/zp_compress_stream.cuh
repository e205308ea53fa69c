// zp_compress_stream.cuh -- the fused score / select / compact kernel of one
// compression call (instantiated per head dim in zp_compress_d64.cu and
// zp_compress_d128.cu).
//
// Method: "Zipage: Maintain High Request Concurrency for LLM Reasoning through
// Compressed PagedAttention" (gist.science summaries; Dutch "Methodologie"
// §1, §3, §5, Korean "방법론" A, C, E).
//
// One unit = (request, layer, kv head) = T = N_max * b cached tokens.  A
// cluster of `cs` CTAs owns the unit (cs = 1 up to 2048 tokens); CTA c owns
// the chunk of TC = T / cs tokens starting at c * TC.  Each CTA is 8
// consumer warps (two groups of four taking alternate stages) and one
// producer warp.  The producer streams the chunk through a ring of NS
// shared-memory stages with TMA in three passes:
//   pass 1  K blocks (tensor maps, 128-byte swizzle, kept in L2 for the
//           next passes where the reuse distance allows it): window logits
//           and the b x b Gram of every block on
//           the tensor cores (mma.sync m16n8k16 bf16, fp32 accumulate);
//           online row max / sum per window row; Lightning Redundancy Score;
//   pass 2  the same K blocks again, in reverse order so that they come from
//           L2 (an LRU cache reused cyclically would evict each block just
//           before its reuse): logits again, importance =
//           mean over the w*G window rows of exp(l - m) / S with the
//           statistics of all T keys, score = importance - lambda * redundancy;
//   pass 3  K and V slabs (bulk copies, plain layout): the kept rows of each
//           block leave for their destination slots, one bulk copy per run of
//           consecutive rows with consecutive destinations.
// Between the passes the cluster exchanges the per-CTA softmax statistics
// and the per-CTA candidates over distributed shared memory, signalled with
// remote mbarrier arrivals (the producer never waits on them).  The b evicted
// tokens: over 64-bit keys = order-preserving image of the fp32 score bits
// above the complemented index, a threshold (the largest of the warps' two
// smallest keys) leaves a few dozen candidates that are ranked by brute force
// (a warp radix select per warp when more than 256 remain), and a merge of
// the cluster's sorted lists (ranks by binary search for up to four lists,
// else b steps of a k-way merge).
//
// Launch: the kernel may start while the one-CTA plan kernel still runs
// (programmatic dependent launch).  Passes 1 and 2 need nothing from the
// plan; griddepcontrol.wait comes right after pass 1 (consumers: the plan's
// destinations load during the statistics merge, before any global write)
// and before pass 3's bulk reads (producer), and the plan's
// verdict word, written by nobody else, decides uniformly whether the CTA
// selects and compacts.  Until then only bounds-safe reads happen: TMA loads
// (bounded by the tensor map) and bounds-checked table rows and block ids.
//
// In-place safety: exactly b tokens are evicted, so destination j reads
// source kept[j] with j <= kept[j] <= j + b.  Pass 3 handles the chunk's
// blocks in ascending order and writes a block's rows only after the stage
// holding that block has landed, so a block is overwritten only after it was
// read; the first rows of CTA c+1 land in CTA c's last block, which CTA c
// stages before it lets the cluster start pass 3.
#pragma once

#include "zp_internal.cuh"

namespace zp {

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
        while (need > 0 && (active[s] & ~chosen[s])) {
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

// Number of entries of the ascending 16-entry list `a` below `key`.
__device__ __forceinline__ int count_below16(const uint64_t *a, uint64_t key)
{
    int p = 0;
    if (a[p + 7] < key)
        p += 8;
    if (a[p + 3] < key)
        p += 4;
    if (a[p + 1] < key)
        p += 2;
    if (a[p] < key)
        p += 1;
    if (p == 15 && a[15] < key)
        p = 16;
    return p;
}

// Merge of two online-softmax partials (m, s) in base 2 (-inf m: empty).
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2)
{
    const float M = fmaxf(m, m2);
    if (M == -INFINITY)
        return;
    s = (m == -INFINITY ? 0.f : s * exp2f(m - M)) + (m2 == -INFINITY ? 0.f : s2 * exp2f(m2 - M));
    m = M;
}

constexpr int kSW = 8;                     // consumer warps, in two groups of four
constexpr int kSGroupWarps = 4;            // the groups take alternate stages
constexpr int kSThreads = (kSW + 1) * 32;  // + one producer warp
constexpr int kSScoreBlocks = 4;           // blocks per stage in passes 1 and 2 (one per warp)
constexpr int kSMoveBlocks = 2;            // blocks per stage in pass 3 (K and V slabs)
#ifndef ZP_STREAM_MAX_TC
#define ZP_STREAM_MAX_TC 2048
#endif
constexpr int kSMaxTC = ZP_STREAM_MAX_TC;  // tokens per CTA at most
constexpr int kSKeysPerLane = kSMaxTC / kSW / 32;

template <int D, int MT, int NS>
struct StreamSmem {
    static constexpr int ROWS = MT * 16;
    static constexpr int SLAB = kBlk * D * 2;          // one (block, kv head) slab
    static constexpr int STAGE = kSScoreBlocks * SLAB;  // 16 KB at d = 128
    static constexpr int off_ring = 0;
    static constexpr int off_q = off_ring + NS * STAGE;         // bf16 [ROWS][D], swizzled
    static constexpr int off_tail = off_q + ROWS * D * 2;       // K slab, V slab of the last block
    static constexpr int off_red = off_tail + 2 * SLAB;         // float [kSMaxTC]
    static constexpr int off_score = off_red + kSMaxTC * 4;     // float [kSMaxTC]
    static constexpr int off_rm = off_score + kSMaxTC * 4;      // float [kSW][ROWS]
    static constexpr int off_rs = off_rm + kSW * ROWS * 4;      // float [kSW][ROWS]
    static constexpr int off_stat = off_rs + kSW * ROWS * 4;    // float2 [ROWS] (remote-read)
    static constexpr int off_gm = off_stat + ROWS * 8;          // float [ROWS]
    static constexpr int off_ginv = off_gm + ROWS * 4;          // float [ROWS]
    static constexpr int off_inv = off_ginv + ROWS * 4;         // float [kSW][b]
    static constexpr int off_cand = off_inv + kSW * kBlk * 4;   // u64 [kSW * b]
    static constexpr int off_pub = off_cand + kSW * kBlk * 8;   // u64 [b] sorted (remote-read)
    static constexpr int off_all = off_pub + kBlk * 8;          // u64 [kMaxCluster * b]
    static constexpr int off_ev = off_all + kMaxCluster * kBlk * 8;  // int [b]
    static constexpr int off_sblk = off_ev + kBlk * 4;          // int [kSMaxTC / b] source blocks
    static constexpr int off_dblk = off_sblk + kSMaxTC / kBlk * 4;  // int [.. + 1] destinations
    static constexpr int off_nsel = off_dblk + (kSMaxTC / kBlk + 1) * 4;  // int: candidates
    static constexpr int off_role = off_nsel + 4;  // int: first-wave pairing role, SM id
    static constexpr int off_bar = (off_role + 4 + 7) / 8 * 8;
    static constexpr int NBAR = 2 * NS + 3;  // full[NS], empty[NS], tail, exchange 1, exchange 2
    static constexpr int BYTES = off_bar + NBAR * 8;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024 B
};

// Byte offset of 16-byte chunk `ch` of row `row` (< 16) in one K block staged
// by TMA with the 128-byte swizzle: d/64 panels of [16 rows][128 B].
__device__ __forceinline__ uint32_t blk_swz(int row, int ch)
{
    return static_cast<uint32_t>((ch >> 3) * 2048 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

template <int D, int MT, int NS>
__global__ void __launch_bounds__(kSThreads, 2) zp_compress_stream_kernel(const CompressArgs a)
{
    // a stage is always consumed by the same group of warps (idx and g have the
    // same parity in every pass), which the parity waits on its barriers need
    static_assert(NS % 2 == 0, "the two consumer groups take alternate stages");
    using S = StreamSmem<D, MT, NS>;
    constexpr int ROWS = S::ROWS, SLAB = S::SLAB, STAGE = S::STAGE;
    constexpr int HALVES = D / 64;
    constexpr int CPR = D / 8;
    constexpr uint32_t ROW_BYTES = D * 2;
    constexpr int NCT = kSW * 32;  // consumer threads

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sRing = sm + S::off_ring;
    uint8_t *sQ = sm + S::off_q;
    uint8_t *sTail = sm + S::off_tail;
    float *sRed = reinterpret_cast<float *>(sm + S::off_red);
    float *sScore = reinterpret_cast<float *>(sm + S::off_score);
    float *sRM = reinterpret_cast<float *>(sm + S::off_rm);
    float *sRS = reinterpret_cast<float *>(sm + S::off_rs);
    float2 *sStat = reinterpret_cast<float2 *>(sm + S::off_stat);
    float *sGm = reinterpret_cast<float *>(sm + S::off_gm);
    float *sGinv = reinterpret_cast<float *>(sm + S::off_ginv);
    float *sInv = reinterpret_cast<float *>(sm + S::off_inv);
    uint64_t *sCand = reinterpret_cast<uint64_t *>(sm + S::off_cand);
    uint64_t *sPub = reinterpret_cast<uint64_t *>(sm + S::off_pub);
    uint64_t *sAll = reinterpret_cast<uint64_t *>(sm + S::off_all);
    int *sEv = reinterpret_cast<int *>(sm + S::off_ev);
    int *sSblk = reinterpret_cast<int *>(sm + S::off_sblk);  // chunk block q -> source block
    int *sDblk = reinterpret_cast<int *>(sm + S::off_dblk);  // dst block of chunk block q-1+i
    int *sNsel = reinterpret_cast<int *>(sm + S::off_nsel);
    int *sRole = reinterpret_cast<int *>(sm + S::off_role);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::off_bar);
    uint64_t *full = bars, *empty = bars + NS;
    uint64_t *tailb = bars + 2 * NS, *xb1 = tailb + 1, *xb2 = tailb + 2;

    const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5;
    const int cs = a.cs;
    const int crank = static_cast<int>(cluster_ctarank());
    const int unit = blockIdx.x / cs;
    const int h = unit % a.Hkv;
    const int l = (unit / a.Hkv) % a.L;
    const int r = unit / (a.Hkv * a.L);

    // This kernel may start while the plan kernel still runs (programmatic
    // dependent launch).  Until its griddepcontrol.wait it reads no plan
    // output and writes no global memory; reads taken from the caller's
    // tables are bounds-checked (TMA loads are by the tensor map), and a bad
    // row or block, which the plan reports, only stops this unit.
    const int row = a.req_idx ? a.req_idx[r] : r;
    if (row < 0 || row >= a.num_rows)
        return;  // uniform per cluster: its CTAs share the unit
    const int32_t *src_row = a.tables + (size_t)row * a.stride;
    const int32_t *dst_row = a.dst_table + (size_t)r * a.N;
    const int T = a.N * kBlk, C = T - a.w;
    const int TC = T / cs;
    const int t0 = crank * TC;
    const int blk0 = t0 / kBlk;
    const int nblk = TC / kBlk;
    const int n_score = TC / (kSScoreBlocks * kBlk);
    const int n_move = TC / (kSMoveBlocks * kBlk);
    const int G = a.Hq / a.Hkv;
    const __nv_bfloat16 *kpool_in = static_cast<const __nv_bfloat16 *>(a.kpools[l]);
    const __nv_bfloat16 *vpool_in = static_cast<const __nv_bfloat16 *>(a.vpools[l]);

    // the chunk's block ids, read once: source blocks of chunk blocks 0..nblk-1
    // and destination blocks of logical blocks blk0-1 .. blk0+nblk-1 (a row
    // moves at most one block down)
    for (int q = tid; q < nblk; q += kSThreads)
        sSblk[q] = src_row[blk0 + q];
    if (tid == 0) {
        // First-wave pairing (one-CTA units).  At the start of a call every
        // resident CTA would run the same phase at the same time, HBM idling
        // while all of them score from L2.  The second CTA of this call on an
        // SM therefore waits (at most 100 us) until the first has consumed
        // pass 1, and the two run out of phase from then on.  Later
        // CTAs, and CTAs whose partner has already finished, do not wait.
        int role = 0;
        const uint32_t smid = sm_id();
        if (cs == 1 && a.smwave && smid < static_cast<uint32_t>(kSmSlots)) {
            if (atomicCAS(a.smwave + smid, 0u, 1u) == 0u) {
                role = 1;
            } else if (atomicCAS(a.smwave + kSmSlots + smid, 0u, 1u) == 0u) {
                role = 2;
                const volatile uint32_t *flag = a.smwave + 2 * kSmSlots + smid;
                const uint64_t t_start = globaltimer_ns();
                while (*flag == 0u && globaltimer_ns() - t_start < 100000ull)
                    __nanosleep(256);
            }
        }
        *sRole = role | static_cast<int>(smid << 2);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kSGroupWarps);
        }
        mbar_init(tailb, 1);
        mbar_init(xb1, cs);
        mbar_init(xb2, cs);
        fence_mbar_init();
    }
    __syncthreads();
    // Peers' barriers must exist before a remote arrive: every thread arrives
    // here and waits only right before its first remote access, so the
    // producer starts streaming at once.
    if (cs > 1)
        cluster_arrive();

    if (wi == kSW) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t keep = policy_evict_last(), once = policy_evict_first();
            bool ok = true;
            if (cs > 1) {
                const int blk = sSblk[nblk - 1];
                if (blk >= 0 && blk < a.num_blocks) {
                    const size_t off = ((size_t)blk * a.Hkv + h) * kBlk * D;
                    mbar_arrive_expect_tx(tailb, 2 * SLAB);
                    bulk_g2s_hint(sTail, kpool_in + off, SLAB, tailb, once);
                    bulk_g2s_hint(sTail + SLAB, vpool_in + off, SLAB, tailb, once);
                } else {
                    mbar_arrive_expect_tx(tailb, 0);  // a bad id: the plan fails the call
                }
            }
            const CUtensorMap *kmap = a.kmaps + l;
            int idx = 0;
            for (int pass = 0; pass < 2; ++pass) {
                for (int g = 0; g < n_score; ++g, ++idx) {
                    const int s = idx % NS;
                    if (idx >= NS)
                        ok &= mbar_wait(&empty[s], ((idx / NS) - 1) & 1);
                    mbar_arrive_expect_tx(&full[s], STAGE);
                    uint8_t *dst = sRing + s * STAGE;
                    // pass 2 walks the chunk backwards: it starts on the blocks
                    // pass 1 read last (still in L2), and pass 3, forwards,
                    // starts on the blocks pass 2 read last
                    const int gg = pass == 0 ? g : n_score - 1 - g;
                    // L2 priority by the distance to the next read of the block:
                    // pass 1 -> pass 2 it is short for the last blocks, pass 2 ->
                    // pass 3 short for the first ones.  The lines a read cannot
                    // keep until then (the first quarter read in pass 1, the
                    // first half read in pass 2) leave first and do not displace
                    // those that can be kept.
                    const uint64_t pol =
                        (pass == 0 ? g < n_score / 4 : g < n_score / 2) ? once : keep;
                    for (int i = 0; i < kSScoreBlocks; ++i) {
                        const int blk = sSblk[gg * kSScoreBlocks + i];
                        const int y = (blk * a.Hkv + h) * kBlk;
#pragma unroll
                        for (int hf = 0; hf < HALVES; ++hf)
                            tma_load_2d_hint(dst + i * SLAB + hf * 2048, kmap, hf * 64, y,
                                             &full[s], pol);
                    }
                }
            }
            // pass 3 reads the blocks with plain bulk copies: only after the
            // plan has checked every id (and not at all if it failed)
            pdl_wait();
            const int n_move_live =
                *reinterpret_cast<volatile int32_t *>(a.call) == 0 ? n_move : 0;
            for (int g = 0; g < n_move_live; ++g, ++idx) {
                const int s = idx % NS;
                if (idx >= NS)
                    ok &= mbar_wait(&empty[s], ((idx / NS) - 1) & 1);
                int nb = 0;
                for (int i = 0; i < kSMoveBlocks; ++i)
                    nb += !(cs > 1 && g * kSMoveBlocks + i == nblk - 1);
                mbar_arrive_expect_tx(&full[s], nb * 2 * SLAB);
                uint8_t *dst = sRing + s * STAGE;
                for (int i = 0; i < kSMoveBlocks; ++i) {
                    const int q = g * kSMoveBlocks + i;
                    if (cs > 1 && q == nblk - 1)
                        continue;  // the staged last block stands in for it
                    const int blk = sSblk[q];
                    const size_t off = ((size_t)blk * a.Hkv + h) * kBlk * D;
                    bulk_g2s_hint(dst + i * SLAB, kpool_in + off, SLAB, &full[s], once);
                    bulk_g2s_hint(dst + (kSMoveBlocks + i) * SLAB, vpool_in + off, SLAB, &full[s],
                                  once);
                }
            }
            if (!ok) {
                set_error(a.cstat, ZP_ERR_TIMEOUT);
                set_error(a.sticky, ZP_ERR_TIMEOUT);
            }
        }
        __syncwarp();
        if (cs > 1)
            cluster_wait();  // (the arrive right after set-up)
    } else {
        // ------------------------------------------------------- consumers
        {
            const __nv_bfloat16 *qsrc =
                a.window_q + ((((size_t)l * a.R + r) * a.Hq + (size_t)h * G) * a.w) * D;
            const uint32_t q_base = smem_u32(sQ);
            for (int c = tid; c < ROWS * CPR; c += NCT) {
                const int rr = c / CPR, ch = c - rr * CPR;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (rr < a.rows)
                    v = ld_global_nc_v4(qsrc + (size_t)rr * D + ch * 8);
                st_shared_v4(q_base + swz(rr, ch, ROWS), v);
            }
        }
        named_sync(NCT);

        bool bad = false;
        int idx = 0;
        const int mi = lane >> 3;
        const int grp = wi / kSGroupWarps, gw = wi % kSGroupWarps;  // group, warp in group
        const uint32_t qb_base = smem_u32(sQ);
        const float ls = a.logit_scale;  // base-2 logit scale, applied in the exponents
        int slot_of[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int rr = mt * 16 + (lane >> 2) + hh * 8;
                slot_of[mt][hh] = rr < a.rows ? rr % a.w : -1;
            }

        // logits of the window rows against the block of this warp in stage s
        // (unscaled: the base-2 scale enters each exponent; causal mask
        // applied); optionally the block's Gram too
        auto block_logits = [&](int s, int key0, float (&acc)[MT][2][4], float (&gram)[2][4],
                                bool with_gram) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc[mt][nt][e] = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    gram[nt][e] = 0.f;
            const uint32_t kb = smem_u32(sRing + s * STAGE + gw * SLAB);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t kf[4];
                ldsm_x4(kb + blk_swz((mi >> 1) * 8 + (lane & 7), ks * 2 + (mi & 1)), kf);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t qa[4];
                    ldsm_x4(qb_base + swz(mt * 16 + (mi & 1) * 8 + (lane & 7), ks * 2 + (mi >> 1),
                                          ROWS),
                            qa);
                    mma_bf16(acc[mt][0], qa[0], qa[1], qa[2], qa[3], kf[0], kf[1]);
                    mma_bf16(acc[mt][1], qa[0], qa[1], qa[2], qa[3], kf[2], kf[3]);
                }
                if (with_gram) {
                    mma_bf16(gram[0], kf[0], kf[2], kf[1], kf[3], kf[0], kf[1]);
                    mma_bf16(gram[1], kf[0], kf[2], kf[1], kf[3], kf[2], kf[3]);
                }
            }
            const bool masked_block = t0 + key0 + kBlk - 1 > C;  // holds window keys
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (masked_block) {
                            const int slot = slot_of[mt][e >> 1];
                            const int tok = t0 + key0 + nt * 8 + (lane & 3) * 2 + (e & 1);
                            if (slot >= 0 && tok > C + slot)
                                acc[mt][nt][e] = -INFINITY;
                        }
                    }
        };

        // ---- pass 1: online row statistics and the redundancy of every key
        float rm[MT][2], rsum[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                rm[mt][hh] = -INFINITY;
                rsum[mt][hh] = 0.f;
            }
        for (int g = 0; g < n_score; ++g, ++idx) {
            if ((g & 1) != grp)
                continue;
            const int s = idx % NS;
            bad |= !mbar_wait(&full[s], (idx / NS) & 1);
            const int key0 = (g * kSScoreBlocks + gw) * kBlk;
            float acc[MT][2][4], gram[2][4];
            block_logits(s, key0, acc, gram, true);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s]);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float bm = fmaxf(fmaxf(acc[mt][0][hh * 2], acc[mt][0][hh * 2 + 1]),
                                           fmaxf(acc[mt][1][hh * 2], acc[mt][1][hh * 2 + 1]));
                    const float m_new = fmaxf(rm[mt][hh], bm);
                    // no branch: while every key so far is masked, any finite
                    // reference gives exp2(-inf) = 0 for all of them
                    const float mref = m_new == -INFINITY ? 0.f : m_new * ls;
                    float sum = rsum[mt][hh] * ex2_approx(fmaf(rm[mt][hh], ls, -mref));
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
                        sum += ex2_approx(fmaf(acc[mt][nt][hh * 2], ls, -mref)) +
                               ex2_approx(fmaf(acc[mt][nt][hh * 2 + 1], ls, -mref));
                    rm[mt][hh] = m_new;
                    rsum[mt][hh] = sum;
                }
            // redundancy: G[j][k] = element e of n-tile nt with j = lane/4 + 8(e/2),
            // k = 8 nt + 2 (lane%4) + e%2; 1/|k_j| once per key from the diagonal
            float *inv = sInv + wi * kBlk;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = (lane >> 2) + (e >> 1) * 8, k = nt * 8 + (lane & 3) * 2 + (e & 1);
                    if (j == k)
                        inv[j] = gram[nt][e];
                }
            __syncwarp();
            if (lane < kBlk) {
                const float dj = inv[lane];
                inv[lane] = dj > 0.f ? rsqrtf(dj) : 0.f;
            }
            __syncwarp();
            float rs[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = (lane >> 2) + (e >> 1) * 8, k = nt * 8 + (lane & 3) * 2 + (e & 1);
                    if (j != k)
                        rs[e >> 1] += gram[nt][e] * inv[k];
                }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float v = rs[hh];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                if ((lane & 3) == 0) {
                    const int j = (lane >> 2) + hh * 8;
                    sRed[key0 + j] = inv[j] * v * (1.0f / (kBlk - 1));
                }
            }
            __syncwarp();
        }
        if (tid == 0 && (*sRole & 3) == 1) {
            // pass 1 consumed: the SM's second CTA of this call may start
            __threadfence();
            *reinterpret_cast<volatile uint32_t *>(a.smwave + 2 * kSmSlots + (*sRole >> 2)) = 1u;
        }

        // the plan's verdict and destinations (the plan kernel may have run
        // alongside pass 1); the loads overlap the statistics merge
        pdl_wait();
        const bool live = *reinterpret_cast<volatile int32_t *>(a.call) == 0;
        constexpr int kDblkPerThread = (kSMaxTC / kBlk + 1 + NCT - 1) / NCT;
        int dblk_ld[kDblkPerThread];
#pragma unroll
        for (int i = 0; i < kDblkPerThread; ++i) {
            const int q = tid + i * NCT, lb = blk0 - 1 + q;
            dblk_ld[i] = (q <= nblk && live && lb >= 0 && lb < a.N - 1) ? dst_row[lb] : -1;
        }

        // per-warp statistics: combine the four lanes of each row
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float m = rm[mt][hh] * ls, sum = rsum[mt][hh];
#pragma unroll
                for (int o = 1; o <= 2; o <<= 1) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
                    const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
                    lse_merge(m, sum, m2, s2);
                }
                if ((lane & 3) == 0) {
                    const int rr = mt * 16 + (lane >> 2) + hh * 8;
                    sRM[wi * ROWS + rr] = m;
                    sRS[wi * ROWS + rr] = sum;
                }
            }
        named_sync(NCT);
        // ... of the CTA; with a cluster, of all its CTAs
        if (tid < ROWS) {
            float m = -INFINITY, sum = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kSW; ++w2)
                lse_merge(m, sum, sRM[w2 * ROWS + tid], sRS[w2 * ROWS + tid]);
            if (cs > 1) {
                sStat[tid] = make_float2(m, sum);
            } else {
                sGm[tid] = m;
                sGinv[tid] = tid < a.rows && sum > 0.f ? 1.0f / sum : 0.f;
            }
        }
        if (cs > 1) {
            named_sync(NCT);
            cluster_wait();  // (the arrive right after set-up)
            if (tid == 0)
                for (int c = 0; c < cs; ++c)
                    mbar_arrive_remote(dsmem_addr(xb1, c));
            bad |= !mbar_wait_cluster(xb1, 0);
            if (tid < ROWS) {
                float m = -INFINITY, sum = 0.f;
                float2 v[kMaxCluster];
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c)
                    v[c] = c < cs ? ld_dsmem_f32x2(dsmem_addr(sStat + tid, c))
                                  : make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c)
                    lse_merge(m, sum, v[c].x, v[c].y);
                sGm[tid] = m;
                sGinv[tid] = tid < a.rows && sum > 0.f ? 1.0f / sum : 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < kDblkPerThread; ++i)
            if (tid + i * NCT <= nblk)
                sDblk[tid + i * NCT] = dblk_ld[i];
        named_sync(NCT);

        // ---- pass 2: importance and score of every key
        const size_t uo = ((size_t)l * a.R + r) * a.Hkv + h;
        float gm[MT][2], ginv[MT][2];  // statistics of this lane's rows
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int rr = mt * 16 + (lane >> 2) + hh * 8;
                gm[mt][hh] = sGm[rr];
                ginv[mt][hh] = sGinv[rr];
            }
        for (int g = 0; g < n_score; ++g, ++idx) {
            if ((g & 1) != grp)
                continue;
            const int s = idx % NS;
            bad |= !mbar_wait(&full[s], (idx / NS) & 1);
            const int key0 = ((n_score - 1 - g) * kSScoreBlocks + gw) * kBlk;  // backwards
            float acc[MT][2][4], gram[2][4];
            block_logits(s, key0, acc, gram, false);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int ee = 0; ee < 2; ++ee) {
                    float v = 0.f;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
                            v += ex2_approx(fmaf(acc[mt][nt][hh * 2 + ee], ls, -gm[mt][hh])) * ginv[mt][hh];
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    if (lane < 4) {
                        const int key = key0 + nt * 8 + lane * 2 + ee;
                        const float sc = v * a.inv_rows - a.lambda * sRed[key];
                        sScore[key] = sc;
                        if (a.scores_out && live)
                            a.scores_out[uo * (size_t)T + t0 + key] =
                                (t0 + key < C) ? sc : INFINITY;
                    }
                }
        }
        named_sync(NCT);
        if (!live) {
            // a failed plan: nothing is written; wait for the staged tail
            // block before leaving (no copy may target freed shared memory)
            if (cs > 1 && tid == 0)
                bad |= !mbar_wait(tailb, 0);
        } else {
            // ---- select the b evicted tokens: the CTA's b smallest keys (order
            // image of the score above the complemented token index), sorted,
            // into sPub.  The largest of the warps' two smallest keys has at
            // least 2 kSW = b keys at or below it, so the b smallest are among
            // the keys at or below it (usually a few dozen), which are ranked by
            // brute force; above kCand of them each warp radix-selects its b
            // smallest and those are ranked.
            {
                static_assert(2 * kSW == kBlk, "two keys per warp make the threshold");
                constexpr int kCand = kMaxCluster * kBlk;  // candidate list in sAll
                const int KW = TC / kSW;  // keys of this warp
                uint64_t key[kSKeysPerLane];
                uint64_t m1 = ~0ull, m2 = ~0ull;
#pragma unroll
                for (int s2 = 0; s2 < kSKeysPerLane; ++s2) {
                    const int kk = lane + 32 * s2;
                    key[s2] = ~0ull;
                    if (kk < KW) {
                        const int k = wi * KW + kk, tok = t0 + k;
                        const uint32_t hi = tok < C ? f32_order(sScore[k]) : 0xffffffffu;
                        key[s2] = (static_cast<uint64_t>(hi) << 32) |
                                  (0xffffffffu - static_cast<uint32_t>(tok));
                    }
                    if (key[s2] < m1) {
                        m2 = m1;
                        m1 = key[s2];
                    } else if (key[s2] < m2) {
                        m2 = key[s2];
                    }
                }
                uint64_t g1 = m1;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const uint64_t x = __shfl_xor_sync(0xffffffffu, g1, o);
                    g1 = x < g1 ? x : g1;
                }
                uint64_t g2 = m1 == g1 ? m2 : m1;  // keys are distinct
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const uint64_t x = __shfl_xor_sync(0xffffffffu, g2, o);
                    g2 = x < g2 ? x : g2;
                }
                if (lane == 0)
                    sCand[wi] = g2;
                if (tid == 0)
                    *sNsel = 0;
                named_sync(NCT);
                uint64_t theta = 0ull;
#pragma unroll
                for (int w2 = 0; w2 < kSW; ++w2)
                    theta = sCand[w2] > theta ? sCand[w2] : theta;
#pragma unroll
                for (int s2 = 0; s2 < kSKeysPerLane; ++s2) {
                    const bool take = key[s2] <= theta;
                    const uint32_t bal = __ballot_sync(0xffffffffu, take);
                    int base = 0;
                    if (lane == 0 && bal)
                        base = atomicAdd(sNsel, __popc(bal));
                    base = __shfl_sync(0xffffffffu, base, 0);
                    const int pos = base + __popc(bal & ((1u << lane) - 1u));
                    if (take && pos < kCand)
                        sAll[pos] = key[s2];
                }
                named_sync(NCT);
                const int n = *sNsel;
                if (n <= kCand) {
                    for (int t = tid; t < n; t += NCT) {
                        const uint64_t k0 = sAll[t];
                        int rank = 0;
                        for (int s2 = 0; s2 < n; ++s2)
                            rank += sAll[s2] < k0;
                        if (rank < kBlk)
                            sPub[rank] = k0;
                    }
                } else {
                    uint32_t chosen[kSKeysPerLane];
                    warp_select_smallest<kSKeysPerLane>(key, kBlk, chosen);
                    warp_compact_keys<kSKeysPerLane>(key, chosen, sCand + wi * kBlk);
                    named_sync(NCT);
                    for (int t = tid; t < kSW * kBlk; t += NCT) {
                        const uint64_t k0 = sCand[t];
                        int rank = 0;
#pragma unroll 8
                        for (int s2 = 0; s2 < kSW * kBlk; ++s2)
                            rank += sCand[s2] < k0;
                        if (rank < kBlk)
                            sPub[rank] = k0;
                    }
                }
            }
            named_sync(NCT);
            if (cs > 1) {
                if (tid == 0) {
                    // this CTA's last block is staged: peers may now write into it
                    bad |= !mbar_wait(tailb, 0);
                    for (int c = 0; c < cs; ++c)
                        mbar_arrive_remote(dsmem_addr(xb2, c));
                }
                bad |= !mbar_wait_cluster(xb2, 0);
                for (int e = tid; e < cs * kBlk; e += NCT)
                    sAll[e] = ld_dsmem_u64(dsmem_addr(sPub + (e & (kBlk - 1)), e / kBlk));
                named_sync(NCT);
                if (cs <= 4) {
                    // rank of each candidate: its place in its own sorted list plus
                    // a binary search in each other list
                    for (int e = tid; e < cs * kBlk; e += NCT) {
                        const uint64_t k0 = sAll[e];
                        const int c0 = e / kBlk;
                        int rank = e % kBlk;
                        for (int c = 0; c < cs; ++c)
                            if (c != c0)
                                rank += count_below16(sAll + c * kBlk, k0);
                        if (rank < kBlk)
                            sEv[rank] = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k0));
                    }
                } else if (wi == 0) {  // b steps of a k-way merge of the sorted lists
                    int ptr = 0;
                    for (int step = 0; step < kBlk; ++step) {
                        const uint64_t head =
                            (lane < cs && ptr < kBlk) ? sAll[lane * kBlk + ptr] : ~0ull;
                        const uint32_t hi = static_cast<uint32_t>(head >> 32);
                        const uint32_t lo = static_cast<uint32_t>(head);
                        const uint32_t mhi = __reduce_min_sync(0xffffffffu, hi);
                        const uint32_t mlo =
                            __reduce_min_sync(0xffffffffu, hi == mhi ? lo : 0xffffffffu);
                        if (lane < cs && hi == mhi && lo == mlo)
                            ++ptr;
                        if (lane == 0)
                            sEv[step] = static_cast<int>(0xffffffffu - mlo);
                    }
                }
            } else if (tid < kBlk) {
                sEv[tid] = static_cast<int>(0xffffffffu - static_cast<uint32_t>(sPub[tid]));
            }
            named_sync(NCT);

            // ---- pass 3: compaction, a half block per warp
            pdl_launch_dependents();  // the finalize kernel may be scheduled
            __nv_bfloat16 *kpool = static_cast<__nv_bfloat16 *>(a.kpools[l]);
            __nv_bfloat16 *vpool = static_cast<__nv_bfloat16 *>(a.vpools[l]);
            const uint64_t once = policy_evict_first();
            for (int g = 0; g < n_move; ++g, ++idx) {
                if ((g & 1) != grp)
                    continue;
                const int s = idx % NS;
                bad |= !mbar_wait(&full[s], (idx / NS) & 1);
                const int bi = gw >> 1;              // block of the stage
                const int q = g * kSMoveBlocks + bi;  // block of the chunk
                const int r8 = (gw & 1) * 8 + lane;   // row of the block (lanes 0..7)
                const bool tail = cs > 1 && q == nblk - 1;
                int dp = 0, dblk = -1;
                bool moved = false;
                if (lane < 8) {
                    const int tok = t0 + q * kBlk + r8;
                    int before = 0;
                    bool ev = false;
    #pragma unroll
                    for (int i = 0; i < kBlk; ++i) {
                        const int e = sEv[i];
                        before += e < tok;
                        ev |= e == tok;
                    }
                    if (!ev) {
                        dp = tok - before;
                        dblk = sDblk[(dp >> 4) - blk0 + 1];
                        moved = dp != tok || dblk != sSblk[q];
                        if (a.kept_out)
                            a.kept_out[uo * (size_t)(T - kBlk) + dp] = tok;
                    }
                }
                const int dp_prev = __shfl_up_sync(0xffffffffu, dp, 1);
                const int dblk_prev = __shfl_up_sync(0xffffffffu, dblk, 1);
                const bool moved_prev = __shfl_up_sync(0xffffffffu, moved ? 1 : 0, 1) != 0;
                const bool cont = moved && lane > 0 && moved_prev && dblk_prev == dblk &&
                                  dp_prev + 1 == dp;
                const uint32_t cont_mask = __ballot_sync(0xffffffffu, cont);
                if (moved && !cont && !bad) {
                    const uint32_t rest = ~(cont_mask >> (lane + 1));
                    const int len = __ffs(rest);  // 1 + continuing lanes after this one
                    const size_t goff = ((size_t)dblk * a.Hkv + h) * kBlk + (dp & (kBlk - 1));
                    const uint8_t *ksrc = tail ? sTail + r8 * ROW_BYTES
                                               : sRing + s * STAGE + bi * SLAB + r8 * ROW_BYTES;
                    const uint8_t *vsrc = tail ? sTail + SLAB + r8 * ROW_BYTES
                                               : sRing + s * STAGE + (kSMoveBlocks + bi) * SLAB +
                                                     r8 * ROW_BYTES;
                    bulk_s2g_hint(kpool + goff * D, ksrc, len * ROW_BYTES, once);
                    bulk_s2g_hint(vpool + goff * D, vsrc, len * ROW_BYTES, once);
                }
                bulk_commit();
                bulk_wait_read0();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[s]);
            }
        }
        if (bad && tid == 0) {
            set_error(a.cstat, ZP_ERR_TIMEOUT);
            set_error(a.sticky, ZP_ERR_TIMEOUT);
        }
    }
    if (cs > 1)
        cluster_sync();  // peers may read this CTA's shared memory until here
}

// Chunking: the fewest CTAs per unit with at most kSMaxTC tokens each, the
// chunk a multiple of 128 tokens (one score stage) and of 64 (a move stage).
inline int stream_cluster_size(int T)
{
    for (int cs = 1; cs <= kMaxCluster; ++cs) {
        if (T % cs)
            continue;
        const int tc = T / cs;
        if (tc <= kSMaxTC && tc % (kSScoreBlocks * kBlk) == 0)
            return cs;
    }
    return 0;
}

template <int D, int MT, int NS>
cudaError_t launch_stream_t(const CompressArgs &a, int units, cudaStream_t s)
{
    using Sm = StreamSmem<D, MT, NS>;
    auto kern = zp_compress_stream_kernel<D, MT, NS>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Sm::ALLOC);
    if (err == cudaSuccess && a.cs > 8)
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess)
        return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * a.cs), 1, 1);
    cfg.blockDim = dim3(kSThreads, 1, 1);
    cfg.dynamicSmemBytes = Sm::ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(a.cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start while the plan kernel runs; it waits before using the plan
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int D>
cudaError_t launch_stream_for_d(const CompressArgs &a, int mt, int units, cudaStream_t s)
{
    constexpr int NS = 4;  // four 16 KB stages: two CTAs fit on an SM
    switch (mt) {
    case 1: return launch_stream_t<D, 1, NS>(a, units, s);
    case 2: return launch_stream_t<D, 2, NS>(a, units, s);
    case 4: return launch_stream_t<D, 4, NS>(a, units, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace zp
