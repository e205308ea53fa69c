// zp_compress_kernel.cuh -- the fused score / select / compact kernel of one
// compression call (instantiated per head dim in zp_compress_d64.cu and
// zp_compress_d128.cu).
//
// Method: "Zipage: Maintain High Request Concurrency for LLM Reasoning through
// Compressed PagedAttention" (gist.science summaries; Dutch "Methodologie"
// §1, §3, §5, Korean "방법론" A, C, E).
//
// One unit = (request, layer, kv head) = T = N_max * b cached tokens.  A
// thread-block cluster of `cs` CTAs owns the unit; CTA c owns tokens
// [c*TPC, (c+1)*TPC) and keeps their K rows in shared memory (TMA, 128-byte
// swizzle).  Steps:
//   1. logits of the w*G window rows against the CTA's keys and the b x b
//      Gram of every block, on the tensor cores (mma.sync m16n8k16 bf16,
//      fp32 accumulate), logits kept in registers in base 2;
//   2. per-CTA row max / sum, merged over the cluster through distributed
//      shared memory into the softmax statistics of all T keys (window row i
//      sees keys up to its own position);
//   3. importance = mean over the w*G rows of the probabilities; Lightning
//      Redundancy Score = mean cosine to the other b-1 keys of the block;
//      score = importance - lambda * redundancy (candidates only);
//   4. the b lowest candidates under (score ascending, index descending):
//      each warp radix-selects its b smallest 64-bit keys (order-preserving
//      image of the fp32 score bits above the complemented index), the CTA
//      ranks its warps' candidates into a sorted list, and b steps of a
//      k-way merge of the cluster's sorted lists give the unit's b;
//   5. kept rows are written to their destination slots: K from shared
//      memory, V through a staging copy (its blocks are prefetched into L2
//      when the CTA starts).  Exactly b tokens are evicted, so
//      destination j reads source kept[j] with j <= kept[j] <= j + b.  In-place
//      writes of the next CTA can only reach this CTA's last block, whose V
//      rows are staged before the first cluster barrier; every K row is in
//      shared memory before that barrier too.
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

template <int D, int NW, int TW, int MT>
struct CompressSmem {
    static constexpr int NT = NW * 32;
    static constexpr int TPC = NW * TW * 16;  // tokens per CTA
    static constexpr int NBLK = TPC / kBlk;
    static constexpr int ROWS = MT * 16;
    static constexpr int K_BYTES = TPC * D * 2;
    static constexpr int Q_BYTES = ROWS * D * 2;
    static constexpr int VT_BYTES = kBlk * D * 2;
    static constexpr int off_k = 0;
    static constexpr int off_q = off_k + K_BYTES;
    static constexpr int off_vt = off_q + Q_BYTES;
    static constexpr int off_rowa = off_vt + VT_BYTES;              // float [NW][ROWS]
    static constexpr int NG = NT / ROWS > 0 ? NT / ROWS : 1;    // stats merge thread groups
    static constexpr int RA = (NW > NG ? NW : NG) * ROWS;           // sRowA / sPart entries
    static constexpr int off_stat = off_rowa + RA * 4;              // float2 [ROWS] (remote-read)
    static constexpr int off_part = off_stat + ROWS * 8;            // float [RA]
    static constexpr int off_gm = off_part + RA * 4;                // float [ROWS]
    static constexpr int off_ginv = off_gm + ROWS * 4;              // float [ROWS]
    static constexpr int off_score = off_ginv + ROWS * 4;           // float [TPC]
    static constexpr int off_red = off_score + TPC * 4;             // float [TPC]
    static constexpr int off_invn = off_red + TPC * 4;              // float [TPC]
    static constexpr int off_doff = off_invn + TPC * 4;             // int [TPC]
    static constexpr int off_cand = off_doff + TPC * 4;             // u64 [NW * b]
    static constexpr int off_pub = off_cand + NW * kBlk * 8;        // u64 [b] sorted (remote-read)
    static constexpr int off_all = off_pub + kBlk * 8;              // u64 [kMaxCluster * b]
    static constexpr int off_ev = off_all + kMaxCluster * kBlk * 8;  // int [b]
    static constexpr int off_misc = off_ev + kBlk * 4;              // int [8]
    static constexpr int off_bmove = off_misc + 8 * 4;              // int [NBLK]
    static constexpr int off_bar = (off_bmove + NBLK * 4 + 15) / 16 * 16;  // 2 mbarriers
    static constexpr int BYTES = off_bar + 16;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024 B
    static constexpr int MIN_BLOCKS = NW == 4 ? (TW <= 2 ? 4 : 2) : (TW <= 2 ? 2 : 1);
};

template <int D, int NW, int TW, int MT>
__global__ void __launch_bounds__(NW * 32, (CompressSmem<D, NW, TW, MT>::MIN_BLOCKS))
    zp_compress_kernel(const CompressArgs a)
{
    using S = CompressSmem<D, NW, TW, MT>;
    constexpr int NT = S::NT, TPC = S::TPC, NBLK = S::NBLK, ROWS = S::ROWS;
    constexpr int HALVES = D / 64;
    constexpr int CPR = D / 8;           // 16-byte chunks per row
    constexpr int KPT = TPC / NT;        // keys per thread (TW / 2)
    static_assert(TW % 2 == 0 && KPT >= 1, "two or more 16-key tiles per warp");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sK = sm + S::off_k;
    uint8_t *sQ = sm + S::off_q;
    uint8_t *sVt = sm + S::off_vt;
    float *sRowA = reinterpret_cast<float *>(sm + S::off_rowa);
    float2 *sStat = reinterpret_cast<float2 *>(sm + S::off_stat);
    float *sPart = reinterpret_cast<float *>(sm + S::off_part);
    float *sGm = reinterpret_cast<float *>(sm + S::off_gm);
    float *sGinv = reinterpret_cast<float *>(sm + S::off_ginv);
    float *sScore = reinterpret_cast<float *>(sm + S::off_score);
    float *sRed = reinterpret_cast<float *>(sm + S::off_red);
    float *sInvN = reinterpret_cast<float *>(sm + S::off_invn);
    int *sDoff = reinterpret_cast<int *>(sm + S::off_doff);
    uint64_t *sCand = reinterpret_cast<uint64_t *>(sm + S::off_cand);
    uint64_t *sPub = reinterpret_cast<uint64_t *>(sm + S::off_pub);
    uint64_t *sAll = reinterpret_cast<uint64_t *>(sm + S::off_all);
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
    for (int q = tid; q < NBLK; q += NT)
        sBMove[q] = 0;
    __syncthreads();

    // ---- loads: K chunk (TMA, swizzled), the V rows of the chunk's last
    // block (bulk copy; the next CTA may overwrite them in place later), and
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
        // the other V blocks are staged much later: start their trip to L2 now
        for (int q = lane; q < NBLK - 1; q += 32) {
            const int blk = src_row[blk0 + q];
            prefetch_l2(static_cast<const __nv_bfloat16 *>(a.vpools[l]) +
                            ((size_t)blk * a.Hkv + h) * kBlk * D,
                        kBlk * D * 2);
        }
    }
    {
        const __nv_bfloat16 *qsrc =
            a.window_q + ((((size_t)l * a.R + r) * a.Hq + (size_t)h * G) * a.w) * D;
        const uint32_t q_base = smem_u32(sQ);
        for (int c = tid; c < ROWS * CPR; c += NT) {
            const int rr = c / CPR, ch = c - rr * CPR;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (rr < a.rows)
                v = ld_global_nc_v4(qsrc + (size_t)rr * D + ch * 8);
            st_shared_v4(q_base + swz(rr, ch, ROWS), v);
        }
    }
    bool bad = !mbar_wait(&bars[0], 0);
    bad = __syncthreads_or(bad);

    // ---- 1. window logits (base 2) and intra-block Gram on the tensor cores
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

    // ---- 2. row max / sum over this CTA's keys
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
    // Gram fragments: element e of n-tile nt is G[j][k], j = lane/4 + 8*(e/2),
    // k = 8*nt + 2*(lane%4) + e%2.  1/|k_j| once per key, from the diagonal.
#pragma unroll
    for (int tt = 0; tt < TW; ++tt) {
        const int key0 = (wi * TW + tt) * 16;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = (lane >> 2) + (e >> 1) * 8, k = nt * 8 + (lane & 3) * 2 + (e & 1);
                if (j == k)
                    sInvN[key0 + j] = gram[tt][nt][e];  // |k_j|^2 for now
            }
    }
    __syncwarp();
#pragma unroll
    for (int s = 0; s < TW / 2; ++s) {  // one key per lane
        const int key = wi * TW * 16 + s * 32 + lane;
        const float dj = sInvN[key];
        sInvN[key] = dj > 0.f ? 1.0f / sqrtf(dj) : 0.f;
    }
    __syncthreads();
    if (tid < ROWS) {
        float m = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2)
            m = fmaxf(m, sRowA[w2 * ROWS + tid]);
        sGm[tid] = m;
    }
    // redundancy: mean cosine to the other b-1 keys of the block
#pragma unroll
    for (int tt = 0; tt < TW; ++tt) {
        const int key0 = (wi * TW + tt) * 16;
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = (lane >> 2) + (e >> 1) * 8, k = nt * 8 + (lane & 3) * 2 + (e & 1);
                if (j != k)
                    rs[e >> 1] += gram[tt][nt][e] * sInvN[key0 + k];
            }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float s = rs[hh];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if ((lane & 3) == 0) {
                const int j = (lane >> 2) + hh * 8;
                sRed[key0 + j] = sInvN[key0 + j] * s * (1.0f / (kBlk - 1));
            }
        }
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
    __syncthreads();
    if (tid < ROWS) {
        float s = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2)
            s += sRowA[w2 * ROWS + tid];
        sStat[tid] = make_float2(sGm[tid], s);
    }
    cluster_sync();  // (1) per-CTA softmax statistics published

    // merge over the cluster: thread group g takes CTAs g, g+NG, ... (all
    // remote loads first, so they are in flight together)
    {
        constexpr int NG = NT / ROWS > 0 ? NT / ROWS : 1;
        constexpr int PER = (kMaxCluster + NG - 1) / NG;
        for (int t = tid; t < ROWS * NG; t += NT) {
            const int rr = t % ROWS, g = t / ROWS;
            float2 v[PER];
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int c = g + i * NG;
                v[i] = c < cs ? ld_dsmem_f32x2(dsmem_addr(sStat + rr, c))
                              : make_float2(-INFINITY, 0.f);
            }
            float m = -INFINITY;
#pragma unroll
            for (int i = 0; i < PER; ++i)
                m = fmaxf(m, v[i].x);
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < PER; ++i)
                if (v[i].y > 0.f)
                    sum += v[i].y * exp2f(v[i].x - m);
            sRowA[g * ROWS + rr] = m;
            sPart[g * ROWS + rr] = sum;
        }
        __syncthreads();
        if (tid < ROWS) {
            float m = -INFINITY;
#pragma unroll
            for (int g = 0; g < NG; ++g)
                m = fmaxf(m, sRowA[g * ROWS + tid]);
            float sum = 0.f;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const float sg = sPart[g * ROWS + tid];
                if (sg > 0.f)
                    sum += sg * exp2f(sRowA[g * ROWS + tid] - m);
            }
            sGm[tid] = m;
            sGinv[tid] = tid < a.rows ? 1.0f / sum : 0.f;
        }
    }
    __syncthreads();

    // ---- 3. importance = mean over window rows of the probabilities; score
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
    __syncwarp();

    // ---- 4. select the b evicted tokens
    {
        constexpr int KW = 16 * TW;   // keys per warp
        constexpr int KPL = KW / 32;  // keys per lane
        uint64_t key[KPL];
#pragma unroll
        for (int s = 0; s < KPL; ++s) {
            const int k = wi * KW + lane + 32 * s, tok = t0 + k;
            const uint32_t hi = tok < C ? f32_order(sScore[k]) : 0xffffffffu;
            key[s] = (static_cast<uint64_t>(hi) << 32) | (0xffffffffu - static_cast<uint32_t>(tok));
        }
        uint32_t chosen[KPL];
        warp_select_smallest<KPL>(key, kBlk, chosen);
        warp_compact_keys<KPL>(key, chosen, sCand + wi * kBlk);
    }
    __syncthreads();
    // the CTA's b smallest, sorted: rank of each warp candidate among all
    for (int t = tid; t < NW * kBlk; t += NT) {
        const uint64_t k0 = sCand[t];
        int rank = 0;
#pragma unroll 8
        for (int s2 = 0; s2 < NW * kBlk; ++s2)
            rank += sCand[s2] < k0;
        if (rank < kBlk)
            sPub[rank] = k0;
    }
    cluster_sync();  // (2) each CTA's sorted candidates published
    for (int e = tid; e < cs * kBlk; e += NT)
        sAll[e] = ld_dsmem_u64(dsmem_addr(sPub + (e & (kBlk - 1)), e / kBlk));
    cluster_arrive();  // no remote shared-memory reads after this point
    __syncthreads();
    // the unit's b smallest: b steps of a k-way merge of the sorted per-CTA
    // lists, lane c holding the head of list c
    if (wi == 0) {
        int ptr = 0;
        for (int step = 0; step < kBlk; ++step) {
            const uint64_t head = (lane < cs && ptr < kBlk) ? sAll[lane * kBlk + ptr] : ~0ull;
            const uint32_t hi = static_cast<uint32_t>(head >> 32), lo = static_cast<uint32_t>(head);
            const uint32_t mhi = __reduce_min_sync(0xffffffffu, hi);
            const uint32_t mlo = __reduce_min_sync(0xffffffffu, hi == mhi ? lo : 0xffffffffu);
            if (lane < cs && hi == mhi && lo == mlo)
                ++ptr;
            if (lane == 0)
                sEv[step] = static_cast<int>(0xffffffffu - mlo);
        }
    }
    __syncthreads();

    {
        const size_t uo = ((size_t)l * a.R + r) * a.Hkv + h;
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
            const int k = tid * KPT + j;
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

    // ---- 5. compaction: K rows from shared memory
    if (!bad) {
        __nv_bfloat16 *kpool = static_cast<__nv_bfloat16 *>(a.kpools[l]);
        const uint32_t kb_base = smem_u32(sK);
        for (int c = tid; c < TPC * CPR; c += NT) {
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
        for (int c = tid; c < TPC * CPR; c += NT) {
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
    cluster_wait();  // peers may still read this CTA's shared memory until here
}

template <int D, int NW, int TW, int MT>
cudaError_t launch_compress_t(const CompressArgs &a, int units, cudaStream_t s)
{
    using Sm = CompressSmem<D, NW, TW, MT>;
    auto kern = zp_compress_kernel<D, NW, TW, MT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           Sm::ALLOC);
    if (err == cudaSuccess && a.cs > 8)
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess)
        return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * a.cs), 1, 1);
    cfg.blockDim = dim3(Sm::NT, 1, 1);
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

// Whether clusters of 16 CTAs of the 4-warp kernel can be resident at all.
template <int D>
bool cluster16_ok_t()
{
    using Sm = CompressSmem<D, 4, 2, 2>;
    auto kern = zp_compress_kernel<D, 4, 2, 2>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::ALLOC) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16 * 64, 1, 1);
    cfg.blockDim = dim3(Sm::NT, 1, 1);
    cfg.dynamicSmemBytes = Sm::ALLOC;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return n > 0;
}

template <int D>
cudaError_t launch_compress_for_d(const CompressArgs &a, CompressShape sh, int mt, int units,
                                  cudaStream_t s)
{
#define ZP_CASE(NW_, TW_, MT_)                                        \
    if (sh.nw == NW_ && sh.tw == TW_ && mt == MT_)                     \
        return launch_compress_t<D, NW_, TW_, MT_>(a, units, s);
    ZP_CASE(4, 2, 1) ZP_CASE(4, 2, 2) ZP_CASE(4, 2, 4)
    ZP_CASE(4, 4, 1) ZP_CASE(4, 4, 2) ZP_CASE(4, 4, 4)
    ZP_CASE(8, 2, 1) ZP_CASE(8, 2, 2) ZP_CASE(8, 2, 4)
    ZP_CASE(8, 4, 1) ZP_CASE(8, 4, 2) ZP_CASE(8, 4, 4)
#undef ZP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace zp
