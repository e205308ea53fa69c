// zp_prefill.cu -- compression at admission of requests longer than the budget.
//
// Zipage (gist.science, Dutch "Methodologie" §1): the kept entries move into
// the first N_max-1 blocks, the N_max-th block is reserved for decoding, and
// the excess blocks are released; §3: shared blocks compress into fresh target
// blocks; §5 and Korean "방법론" E: the Lightning Redundancy Score compares the
// keys of one block only.  The scores are those of zp_compress computed over
// each request's own T >= N_max*b tokens (the window is its last w tokens); the
// selection keeps (N_max-1)*b - w candidates, so T - (N_max-1)*b tokens go --
// a number that varies per request and can be most of the request.
//
// Launches, between the shared plan and finalize kernels (zp_compress.cu):
//   zp_prefill_pass_kernel<.., false>  grid (unit, chunk of 2048 tokens), four
//       warps each streaming their blocks through a private two-stage TMA
//       ring: window logits and the Gram of each block on mma.sync, the
//       chunk's softmax statistics of every window row, the redundancy of
//       every key (over the filled slots of its block) -> workspace.
//   zp_prefill_pass_kernel<.., true>   same grid: the statistics of all
//       chunks of the unit merged, logits again, importance and score.
//   zp_prefill_select_kernel  one CTA of 256 threads per unit: radix
//       select (digit passes over bits 31-21, 20-10 and 9-0 of the
//       order-preserving image of the fp32 scores held in shared memory,
//       each digit found by a block-wide scan of the histogram) of the
//       K_keep-th largest score; ties at the threshold go to the lower
//       index; the kept positions in ascending order by block scans, then
//       the window.
//   zp_prefill_gather_kernel  one CTA per unit: the source pool row of every
//       destination row resolved into shared memory, then the destination
//       blocks in ascending order through a ring of shared-memory stages:
//       TMA row gathers (tile::gather4, four arbitrary pool rows per load)
//       of each block's 16 K and 16 V rows, written back as the block's two
//       contiguous slabs by bulk stores.  Every later block reads sources at
//       or after its own position (kept[j] >= j), which no earlier block's
//       store writes -- so compacting in place is safe with loads running
//       ahead of the stores.
#include "zp_internal.cuh"

namespace zp {

constexpr int kPW = 4;                       // warps of a scoring CTA
constexpr int kPThreads = kPW * 32;
constexpr int kPStages = 2;                  // TMA stages per warp
constexpr int kPChunk = kPrefillChunk;       // tokens per scoring CTA
constexpr int kPBlocks = kPChunk / kBlk;
constexpr int kSelThreads = 256;
constexpr int kSelBins = 2048;                 // digits of the selection's widest pass
constexpr int kCmpSeg = 2048;                // destination rows whose indices are staged at once

template <int D, int MT>
struct PrefillSmem {
    static constexpr int ROWS = MT * 16;
    static constexpr int SLAB = kBlk * D * 2;
    static constexpr int off_ring = 0;                              // [kPW][kPStages][SLAB]
    static constexpr int off_q = off_ring + kPW * kPStages * SLAB;  // bf16 [ROWS][D], swizzled
    static constexpr int off_rm = off_q + ROWS * D * 2;             // float [kPW][ROWS]
    static constexpr int off_rs = off_rm + kPW * ROWS * 4;          // float [kPW][ROWS]
    static constexpr int off_gm = off_rs + kPW * ROWS * 4;          // float [ROWS]
    static constexpr int off_ginv = off_gm + ROWS * 4;              // float [ROWS]
    static constexpr int off_inv = off_ginv + ROWS * 4;             // float [kPW][b]
    static constexpr int off_bar = (off_inv + kPW * kBlk * 4 + 7) / 8 * 8;
    static constexpr int BYTES = off_bar + kPW * kPStages * 8;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024 B
};

// Merges the softmax statistics (m, s) of two key sets (base 2); (-inf, 0) is
// the empty set.
__device__ __forceinline__ void stat_merge(float &m, float &s, float m2, float s2)
{
    if (m2 == -INFINITY)
        return;
    if (m == -INFINITY) {
        m = m2;
        s = s2;
        return;
    }
    const float mn = fmaxf(m, m2);
    s = s * exp2f(m - mn) + s2 * exp2f(m2 - mn);
    m = mn;
}

template <int D, int MT, bool SCORE>
__global__ void __launch_bounds__(kPThreads) zp_prefill_pass_kernel(const PrefillArgs a)
{
    using S = PrefillSmem<D, MT>;
    constexpr int ROWS = S::ROWS, SLAB = S::SLAB, HALVES = D / 64, CPR = D / 8;
    if (*(volatile int32_t *)a.call != 0)
        return;
    const int u = blockIdx.x, chunk = blockIdx.y;
    const int h = u % a.Hkv, r = (u / a.Hkv) % a.R, l = u / (a.Hkv * a.R);
    const int row = a.req_idx ? a.req_idx[r] : r;
    const int T = a.lengths[row];  // checked by the plan
    const int C = T - a.w;
    const int t0 = chunk * kPChunk;
    if (t0 >= T)
        return;
    const int nblk = min(kPBlocks, (T - t0 + kBlk - 1) / kBlk);
    const int G = a.Hq / a.Hkv;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = sm + S::off_q;
    float *sRM = reinterpret_cast<float *>(sm + S::off_rm);
    float *sRS = reinterpret_cast<float *>(sm + S::off_rs);
    float *sGm = reinterpret_cast<float *>(sm + S::off_gm);
    float *sGinv = reinterpret_cast<float *>(sm + S::off_ginv);
    float *sInv = reinterpret_cast<float *>(sm + S::off_inv);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::off_bar);
    const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5, mi = lane >> 3;

    if (tid < kPW * kPStages)
        mbar_init(&bars[tid], 1);
    if (tid == 0)
        fence_mbar_init();
    __syncthreads();

    // this warp's blocks of the chunk: wi, wi + kPW, ...; the first loads are
    // issued before anything else, so the queries and statistics below are
    // read while they are in flight
    const int my_n = wi < nblk ? (nblk - wi + kPW - 1) / kPW : 0;
    uint8_t *ring = sm + S::off_ring + wi * kPStages * SLAB;
    uint64_t *bar = bars + wi * kPStages;
    const int32_t *trow = a.tables + (size_t)row * a.stride;
    const CUtensorMap *kmap = a.kmaps + l;
    // the block ids of this warp's blocks, one per lane, read once (the TMA
    // issue of every block then waits on no global load)
    static_assert(kPBlocks / kPW <= 32, "one block id per lane");
    const int my_blk = lane < my_n ? trow[t0 / kBlk + wi + lane * kPW] : 0;  // checked by the plan
    auto issue = [&](int i, int blk) {
        const int s = i % kPStages;
        mbar_arrive_expect_tx(&bar[s], SLAB);
        const int y = (blk * a.Hkv + h) * kBlk;
#pragma unroll
        for (int hf = 0; hf < HALVES; ++hf)
            tma_load_2d(ring + s * SLAB + hf * kBlk * 128, kmap, hf * 64, y, &bar[s]);
    };
#pragma unroll
    for (int i = 0; i < kPStages; ++i) {
        const int blk = __shfl_sync(0xffffffffu, my_blk, i);
        if (lane == 0 && i < my_n)
            issue(i, blk);
    }

    // window queries -> shared memory (swizzled, rows past w*G zero)
    {
        const __nv_bfloat16 *qsrc =
            a.window_q + ((((size_t)l * a.R + r) * a.Hq + (size_t)h * G) * a.w) * D;
        const uint32_t qb = smem_u32(sQ);
        for (int c = tid; c < ROWS * CPR; c += kPThreads) {
            const int rr = c / CPR, ch = c - rr * CPR;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (rr < a.rows)
                v = ld_global_nc_v4(qsrc + (size_t)rr * D + ch * 8);
            st_shared_v4(qb + swz(rr, ch, ROWS), v);
        }
    }
    if (SCORE && tid < ROWS) {
        // statistics of all keys of the unit: merge the chunks (their loads
        // four at a time, independent of one another)
        const int nc = (T + kPChunk - 1) / kPChunk;
        const float2 *st = a.stats + (size_t)u * a.NC * kMaxRows + tid;
        float m = -INFINITY, s = 0.f;
        for (int c0 = 0; c0 < nc; c0 += 4) {
            float2 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                v[k] = c0 + k < nc ? st[(size_t)(c0 + k) * kMaxRows] : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                stat_merge(m, s, v[k].x, v[k].y);
        }
        sGm[tid] = m;
        sGinv[tid] = tid < a.rows && s > 0.f ? 1.0f / s : 0.f;
    }
    __syncthreads();

    int slot_of[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int rr = mt * 16 + (lane >> 2) + hh * 8;
            slot_of[mt][hh] = rr < a.rows ? rr % a.w : -1;
        }
    float rm[MT][2], rsum[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            rm[mt][hh] = -INFINITY;
            rsum[mt][hh] = 0.f;
        }
    const size_t ubase = (size_t)u * a.T_cap;
    const uint32_t qb = smem_u32(sQ);
    const float ls = a.logit_scale;  // base-2 logit scale
    bool ok = true;
    // scoring: the merged statistics of this thread's rows in registers, and
    // the redundancy of each block's keys (lane j: slot j) read one block ahead
    float gm[MT][2], ginv[MT][2];
    float red_cur = 0.f;
    auto red_of = [&](int i) {
        const int key = t0 + (wi + i * kPW) * kBlk + (lane & 15);
        return lane < kBlk && i < my_n && key < C ? a.red[ubase + key] : 0.f;
    };
    if (SCORE) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int rr = mt * 16 + (lane >> 2) + hh * 8;
                gm[mt][hh] = sGm[rr];
                ginv[mt][hh] = sGinv[rr];
            }
        red_cur = red_of(0);
    }

    for (int i = 0; i < my_n; ++i) {
        const int s = i % kPStages;
        const float red_nxt = SCORE ? red_of(i + 1) : 0.f;
        ok &= mbar_wait(&bar[s], (i / kPStages) & 1);
        const int key0 = t0 + (wi + i * kPW) * kBlk;  // token of the block's slot 0
        const uint32_t kb = smem_u32(ring + s * SLAB);
        float acc[MT][2][4], gram[2][4];
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
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t kf[4];
            ldsm_x4(kb + swz((mi >> 1) * 8 + (lane & 7), ks * 2 + (mi & 1), kBlk), kf);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t qa[4];
                ldsm_x4(qb + swz(mt * 16 + (mi & 1) * 8 + (lane & 7), ks * 2 + (mi >> 1), ROWS),
                        qa);
                mma_bf16(acc[mt][0], qa[0], qa[1], qa[2], qa[3], kf[0], kf[1]);
                mma_bf16(acc[mt][1], qa[0], qa[1], qa[2], qa[3], kf[2], kf[3]);
            }
            if (!SCORE) {
                mma_bf16(gram[0], kf[0], kf[2], kf[1], kf[3], kf[0], kf[1]);
                mma_bf16(gram[1], kf[0], kf[2], kf[1], kf[3], kf[2], kf[3]);
            }
        }
        __syncwarp();
        {
            const int blk = __shfl_sync(0xffffffffu, my_blk, (i + kPStages) & 31);
            if (lane == 0 && i + kPStages < my_n) {
                fence_proxy_async_smem();
                issue(i + kPStages, blk);
            }
        }
        // window row of slot i sees keys up to C + i, which also hides the
        // unfilled slots of a partial last block (only blocks reaching past C
        // hold such keys); the logits stay unscaled here, the base-2 scale
        // enters each exponent below
        if (key0 + kBlk - 1 > C) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int slot = slot_of[mt][e >> 1];
                        const int tok = key0 + nt * 8 + (lane & 3) * 2 + (e & 1);
                        if (slot >= 0 ? tok > C + slot : tok >= T)
                            acc[mt][nt][e] = -INFINITY;
                    }
        }

        if (!SCORE) {
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
            // redundancy over the f filled slots: G[j][k] is element e of
            // n-tile nt with j = lane/4 + 8(e/2), k = 8 nt + 2 (lane%4) + e%2
            const int f = min(kBlk, T - key0);
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
                inv[lane] = lane < f && dj > 0.f ? rsqrtf(dj) : 0.f;
            }
            __syncwarp();
            float rs[2] = {0.f, 0.f};
            const float rf1 = f > 1 ? __frcp_rn(static_cast<float>(f - 1)) : 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = (lane >> 2) + (e >> 1) * 8, k = nt * 8 + (lane & 3) * 2 + (e & 1);
                    if (j != k && k < f)
                        rs[e >> 1] += gram[nt][e] * inv[k];
                }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float v = rs[hh];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                const int j = (lane >> 2) + hh * 8;
                if ((lane & 3) == 0 && j < f)
                    a.red[ubase + key0 + j] = inv[j] * v * rf1;
            }
            __syncwarp();
        } else {
            // importance = mean over the window rows of the softmax probability
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
                    const float rd = __shfl_sync(0xffffffffu, red_cur, nt * 8 + (lane & 3) * 2 + ee);
                    const int key = key0 + nt * 8 + lane * 2 + ee;
                    if (lane < 4 && key < T)
                        a.scores[ubase + key] = key < C ? v * a.inv_rows - a.lambda * rd : INFINITY;
                }
        }
        red_cur = red_nxt;
    }
    if (!ok && lane == 0)
        set_error(a.sticky, ZP_ERR_TIMEOUT);

    if (!SCORE) {
        // the chunk's statistics of every row: lanes, then warps
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float m = rm[mt][hh] * ls, s = rsum[mt][hh];
#pragma unroll
                for (int o = 1; o <= 2; o <<= 1) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
                    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
                    stat_merge(m, s, m2, s2);
                }
                if ((lane & 3) == 0) {
                    const int rr = mt * 16 + (lane >> 2) + hh * 8;
                    sRM[wi * ROWS + rr] = m;
                    sRS[wi * ROWS + rr] = s;
                }
            }
        __syncthreads();
        if (tid < ROWS) {
            float m = -INFINITY, s = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kPW; ++w2)
                stat_merge(m, s, sRM[w2 * ROWS + tid], sRS[w2 * ROWS + tid]);
            a.stats[((size_t)u * a.NC + chunk) * kMaxRows + tid] = make_float2(m, s);
        }
    }
}

__global__ void __launch_bounds__(kSelThreads) zp_prefill_select_kernel(const PrefillArgs a)
{
    if (*(volatile int32_t *)a.call != 0)
        return;
    extern __shared__ uint32_t sKey[];  // [T_cap] order images of the scores
    __shared__ int hist[kSelBins];
    __shared__ int s_scan[kSelThreads / 32 + 1];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;
    const int tid = threadIdx.x;
    const int u = blockIdx.x;
    const int r = (u / a.Hkv) % a.R;
    const int row = a.req_idx ? a.req_idx[r] : r;
    const int T = a.lengths[row];
    const int C = T - a.w;
    const int KT = (a.N - 1) * kBlk, keep = KT - a.w;  // 0 <= keep < C since T >= N*b
    const float *sc = a.scores + (size_t)u * a.T_cap;
    for (int j = tid; j < C; j += kSelThreads)
        sKey[j] = f32_order(sc[j]);
    if (tid == 0) {
        s_prefix = 0u;
        s_need = keep;
    }

    // the keep-th largest order image, one digit at a time from the top:
    // bits 31-21, 20-10, 9-0
    uint32_t mask = 0u;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
        const int nb = pass == 2 ? 1024 : 2048;  // digits of this pass
        for (int i = tid; i < nb; i += kSelThreads)
            hist[i] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        const int need = s_need;
        for (int j = tid; j < C; j += kSelThreads) {
            const uint32_t k = sKey[j];
            if ((k & mask) == prefix)
                atomicAdd(&hist[(k >> shift) & static_cast<uint32_t>(nb - 1)], 1);
        }
        __syncthreads();
        // thread t holds the digits hi, hi - 1, .., hi - bpt + 1 (larger
        // digits at smaller t); the keys above its digits come from a scan
        const int bpt = nb / kSelThreads;
        const int hi = nb - 1 - tid * bpt;
        int c = 0;
        for (int i = 0; i < bpt; ++i)
            c += hist[hi - i];
        int total;
        const int above = block_excl_scan<kSelThreads>(c, s_scan, total);
        // the digit at which the count from the top reaches need (need <= 0
        // only when nothing is kept: the top digit then, nothing above it)
        if (need <= 0 ? tid == 0 : (above < need && need <= above + c)) {
            int run = above, i = 0;
            while (i < bpt - 1 && run + hist[hi - i] < need)
                run += hist[hi - i++];
            s_prefix = prefix | (static_cast<uint32_t>(hi - i) << shift);
            s_need = need - run;
        }
        mask |= static_cast<uint32_t>(nb - 1) << shift;
        __syncthreads();
    }
    const uint32_t thr = s_prefix;
    const int take_eq = s_need;  // keys equal to thr to keep: the lowest indices

    // keep j iff key > thr, or key == thr among the first take_eq such indices
    const int per = (C + kSelThreads - 1) / kSelThreads;
    const int j0 = min(C, tid * per), j1 = min(C, j0 + per);
    int my_eq = 0;
    for (int j = j0; j < j1; ++j)
        my_eq += sKey[j] == thr;
    int total;
    int eq_before = block_excl_scan<kSelThreads>(my_eq, s_scan, total);
    int my_keep = 0;
    {
        int e = eq_before;
        for (int j = j0; j < j1; ++j) {
            const uint32_t k = sKey[j];
            my_keep += k > thr || (k == thr && e++ < take_eq);
        }
    }
    int pos = block_excl_scan<kSelThreads>(my_keep, s_scan, total);
    int32_t *kept = a.kept + (size_t)u * KT;
    {
        int e = eq_before;
        for (int j = j0; j < j1; ++j) {
            const uint32_t k = sKey[j];
            if (k > thr || (k == thr && e++ < take_eq)) {
                if (pos < keep)  // holds by construction; guards the neighbour's slice
                    kept[pos] = j;
                ++pos;
            }
        }
    }
    for (int i = tid; i < a.w; i += kSelThreads)
        kept[keep + i] = C + i;
    if (tid == 0 && total != keep)
        set_error(a.sticky, ZP_ERR_DEVICE_CHECK);
}

// Compaction by TMA row gathers: one CTA per unit.  The source pool row of
// every destination row is resolved into shared memory first (all threads);
// then one thread streams the destination blocks in ascending order through
// a ring of kGatStages shared-memory stages: a stage takes a destination
// block's 16 K rows and 16 V rows with eight tile::gather4 loads (four
// arbitrary pool rows each, one row per box) and leaves as two bulk stores,
// the block's contiguous K and V slabs.  Loads run kGatAhead blocks ahead of
// the store.  In place this is safe: the sources of destination block p lie
// at positions >= 16 p (kept[j] >= j), so block p's slab is written only
// after every load that reads it -- its own and all earlier blocks' -- has
// landed, and the blocks loaded ahead read only later positions.  A block
// whose 16 rows all stay where they are is skipped.
constexpr int kGatThreads = 256;
constexpr int kGatStages = 8;
constexpr int kGatAhead = 5;
static_assert(kGatAhead < kGatStages, "a stage is reused only after its store read it");

template <int D>
__global__ void __launch_bounds__(kGatThreads) zp_prefill_gather_kernel(const PrefillArgs a)
{
    constexpr int SLAB = kBlk * D * 2;  // one (block, kv head) slab of K or of V
    __shared__ uint32_t sSrc[kCmpSeg];               // source pool row of each destination row
    __shared__ uint8_t sMove[kCmpSeg / kBlk];        // the destination block moves a row
    __shared__ __align__(8) uint64_t full[kGatStages];
    extern __shared__ uint8_t smem_raw[];            // [kGatStages][K slab, V slab]
    uint8_t *stage = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    if (*(volatile int32_t *)a.call != 0)
        return;
    const int u = blockIdx.x;
    const int h = u % a.Hkv, r = (u / a.Hkv) % a.R, l = u / (a.Hkv * a.R);
    const int row = a.req_idx ? a.req_idx[r] : r;
    const int T = a.lengths[row];
    const int KT = (a.N - 1) * kBlk;
    const int32_t *kept = a.kept + (size_t)u * KT;
    const int32_t *trow = a.tables + (size_t)row * a.stride;
    const int32_t *drow = a.dst_table + (size_t)r * a.stride;
    uint8_t *const kpool = static_cast<uint8_t *>(a.kpools[l]);
    uint8_t *const vpool = static_cast<uint8_t *>(a.vpools[l]);
    const CUtensorMap *kmap = a.krmaps + l, *vmap = a.vrmaps + l;
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < kGatStages; ++s)
            mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    bool ok = true;
    int g = 0;  // destination blocks streamed so far (all segments)
    for (int s0 = 0; s0 < KT; s0 += kCmpSeg) {
        const int n = min(kCmpSeg, KT - s0);  // a multiple of 16
        const int nb = n / kBlk;
        __syncthreads();  // the previous segment's rows are issued
        for (int q = tid; q < nb; q += kGatThreads)
            sMove[q] = 0;
        __syncthreads();
        for (int jj = tid; jj < n; jj += kGatThreads) {
            const int j = s0 + jj, src = kept[j];
            const uint32_t dr =
                (static_cast<uint32_t>(drow[j / kBlk]) * a.Hkv + h) * kBlk + j % kBlk;
            uint32_t sr = dr;  // a row that stays is gathered from where it is
            if (src < j || src >= T) {  // kept[j] >= j holds for any valid selection
                set_error(a.sticky, ZP_ERR_DEVICE_CHECK);
            } else {
                sr = (static_cast<uint32_t>(trow[src / kBlk]) * a.Hkv + h) * kBlk + src % kBlk;
            }
            sSrc[jj] = sr;
            if (sr != dr)
                sMove[jj / kBlk] = 1;
        }
        __syncthreads();
        if (tid == 0) {
            if (s0 > 0)
                bulk_wait_read<0>();  // stage reuse across segments: every earlier store read
            int issued = 0, stored = 0;  // blocks of the segment loaded, stored
            for (int step = 0; step < nb + kGatAhead && ok; ++step) {
                const int pl = step, ps = step - kGatAhead;
                if (pl < nb) {
                    ++issued;
                    const int gi = g + pl, st = gi % kGatStages;
                    // the store that last read this stage was committed kGatStages -
                    // kGatAhead steps ago: at most that many minus one groups may read on
                    if (gi >= kGatStages)
                        bulk_wait_read<kGatStages - kGatAhead - 1>();
                    uint8_t *ks = stage + st * 2 * SLAB;
                    if (sMove[pl]) {
                        mbar_arrive_expect_tx(&full[st], 2 * SLAB);
                        const uint32_t *rs = sSrc + pl * kBlk;
#pragma unroll
                        for (int i = 0; i < kBlk; i += 4) {
                            tma_gather4(ks + i * D * 2, kmap, 0, rs[i], rs[i + 1], rs[i + 2],
                                        rs[i + 3], &full[st]);
                            tma_gather4(ks + SLAB + i * D * 2, vmap, 0, rs[i], rs[i + 1],
                                        rs[i + 2], rs[i + 3], &full[st]);
                        }
                    } else {
                        mbar_arrive_expect_tx(&full[st], 0);
                    }
                }
                if (ps >= 0) {
                    const int gi = g + ps, st = gi % kGatStages;
                    ok &= mbar_wait(&full[st], (gi / kGatStages) & 1);
                    if (ok && sMove[ps]) {
                        const int p = s0 / kBlk + ps;
                        const size_t off = ((static_cast<size_t>(drow[p]) * a.Hkv + h) * kBlk) *
                                           (size_t)(D * 2);
                        uint8_t *ks = stage + st * 2 * SLAB;
                        bulk_s2g_hint(kpool + off, ks, SLAB, policy_evict_first());
                        bulk_s2g_hint(vpool + off, ks + SLAB, SLAB, policy_evict_first());
                    }
                    bulk_commit();
                    ++stored;
                }
            }
            if (!ok) {
                set_error(a.sticky, ZP_ERR_TIMEOUT);
                // loads still in flight land before the stages go away
                for (int pl = stored; pl < issued; ++pl)
                    mbar_wait(&full[(g + pl) % kGatStages], ((g + pl) / kGatStages) & 1);
            }
            g += nb;
            bulk_wait_all();
        }
    }
}

template <int D, int MT>
static cudaError_t launch_passes(const PrefillArgs &a, int units, cudaStream_t s)
{
    using S = PrefillSmem<D, MT>;
    auto k1 = zp_prefill_pass_kernel<D, MT, false>;
    auto k2 = zp_prefill_pass_kernel<D, MT, true>;
    cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, S::ALLOC);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, S::ALLOC);
    if (e != cudaSuccess)
        return e;
    const dim3 grid(static_cast<unsigned>(units), static_cast<unsigned>(a.NC));
    k1<<<grid, kPThreads, S::ALLOC, s>>>(a);
    k2<<<grid, kPThreads, S::ALLOC, s>>>(a);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_for_d(const PrefillArgs &a, int mt, int units, cudaStream_t s)
{
    cudaError_t e = mt == 1   ? launch_passes<D, 1>(a, units, s)
                    : mt == 2 ? launch_passes<D, 2>(a, units, s)
                              : launch_passes<D, 4>(a, units, s);
    if (e != cudaSuccess)
        return e;
    const int sel_smem = a.T_cap * 4;
    e = cudaFuncSetAttribute(zp_prefill_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             sel_smem);
    if (e != cudaSuccess)
        return e;
    zp_prefill_select_kernel<<<static_cast<unsigned>(units), kSelThreads, sel_smem, s>>>(a);
    constexpr int gat_smem = kGatStages * 2 * kBlk * D * 2 + 128;
    e = cudaFuncSetAttribute(zp_prefill_gather_kernel<D>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, gat_smem);
    if (e != cudaSuccess)
        return e;
    zp_prefill_gather_kernel<D><<<static_cast<unsigned>(units), kGatThreads, gat_smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs &a, int d, int mt, int units, cudaStream_t s)
{
    if (d == 64)
        return launch_for_d<64>(a, mt, units, s);
    if (d == 128)
        return launch_for_d<128>(a, mt, units, s);
    return cudaErrorInvalidValue;
}

}  // namespace zp
