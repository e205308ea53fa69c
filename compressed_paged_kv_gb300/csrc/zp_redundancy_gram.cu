// zp_redundancy_gram.cu -- the all-keys redundancy of every key computed the
// way the original score pays for it: from the dense T x T Gram matrix of
// each (request, layer, kv head) unit, O(T^2 d), on the 5th-generation tensor
// cores.  The Lightning Redundancy Score of the compression kernels replaces
// this O(N^2 b^2) score by an O(N b^2) one (Zipage, gist.science: Dutch
// "Methodologie" §5, Korean "방법론" E); zp_redundancy_global.cu computes the
// same quantity in O(T d) through the sum of the normalised keys.  Result:
// red_t = mean over the other keys k of the unit of cos(K_t, K_k), a zero key
// having cosine 0 with every key.
//
// Work items are (unit, 256 keys t): A = those 256 key rows as two halves of
// 128, B = the unit's keys 128 at a time, D_g = A_g B^T (128 x 128 fp32 per
// half, two buffers: all 512 tensor-memory columns), and
//   sum_t = sum_k D[t][k] / |K_k|,   red_t = (sum_t / |K_t| - 1) / (T - 1)
// (the k = t term is the 1 removed; columns past T are skipped).  Each B tile
// feeds both halves: 256 rows of products per byte staged.  The kernel is
// persistent: one CTA per SM takes a contiguous range of items, so a unit's
// row tiles run back to back on one SM (its keys stay in L2 between them, and
// the inverse norms of its keys, computed by its first item there, in shared
// memory for the next ones); it keeps its tensor memory for the whole launch
// and runs the pipelines below continuously from one item into the next.
// Eighteen warps:
//   warp 0     TMA producer: each item's A once it is free (its last products
//              done and its row norms taken), B through four stages (the K
//              pool maps, 128-byte swizzle, one 16-row box per cache block
//              and 64 dims);
//   warp 1     allocates the tensor memory, one lane issues tcgen05.mma
//              (kind::f16, bf16 x bf16 -> fp32, M 128, N 128, K 16) for both
//              halves and commits to mbarriers;
//   warps 2-17 two sets of 8 (one per accumulator buffer, so consecutive
//              tiles are reduced at the same time): the inverse norms of the
//              set's B stages (one key per thread; for units of up to 4,096
//              keys in a unit's first item only), then tcgen05.ld of 32 lanes
//              of one half and weighted row sums in registers, the two sets'
//              sums added at the end of the item.
// The accumulators alternate between two buffers, so the products of one B
// tile overlap the reduction of the previous one.
// Every wait is bounded; after a timeout a warp records ZP_ERR_TIMEOUT and
// stops waiting (it still passes every barrier its set passes, doing no
// work), the producer waits for its copies in flight and the MMA lane for its
// products before the tensor memory is freed.
#include "zp_aux.cuh"

namespace zp {

namespace {

constexpr int kGramH = 128;                // keys t per accumulator (tensor-memory lanes)
constexpr int kGramM = 2 * kGramH;         // keys t per CTA
constexpr int kGramN = 128;                // keys k per product (accumulator columns)
constexpr int kGramNS = 4;                 // B stages
constexpr int kGramEW = 16;                // reducing warps: 2 sets (one per buffer) of 8
constexpr int kGramThreads = (2 + kGramEW) * 32;
constexpr int kTmemCols = 4 * kGramN;      // [buffer][half] accumulators
constexpr int kGramUMax = 4096;            // longest unit whose key norms stay in shared memory

template <int D>
struct GramSmem {
    static constexpr int PANELS = D / 64;                 // 128-byte rows per key
    static constexpr int A_PANEL = kGramH * 128;          // bytes of one half, one panel
    static constexpr int B_PANEL = kGramN * 128;
    static constexpr int A_BYTES = 2 * PANELS * A_PANEL;
    static constexpr int B_STAGE = PANELS * B_PANEL;
    static constexpr int off_a = 0;                       // [half][panel]
    static constexpr int off_b = off_a + A_BYTES;         // kGramNS stages
    static constexpr int off_inv = off_b + kGramNS * B_STAGE;  // float [kGramNS][kGramN]
    static constexpr int off_invu = off_inv + kGramNS * kGramN * 4;  // float [kGramUMax]
    static constexpr int off_part = off_invu + kGramUMax * 4;       // float [2][2][kGramM]
    static constexpr int off_bar = off_part + 4 * kGramM * 4;
    // fullA, fullB[NS], emptyB[NS], accFull[2], accEmpty[2], emptyA, done
    static constexpr int NBAR = 1 + 2 * kGramNS + 4 + 2;
    static constexpr int off_tmem = off_bar + NBAR * 8;   // u32: tensor-memory base
    static constexpr int BYTES = off_tmem + 16;
    static constexpr int ALLOC = BYTES + 1024;            // room to align the base to 1024 B
};

// Shared-memory matrix descriptor of a K-major operand stored as 128-byte
// rows with the 128-byte swizzle (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3ffffu) >> 4);       // start address
    d |= static_cast<uint64_t>(16 >> 4) << 16;                 // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;               // stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                       // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                       // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 accumulator,
// both operands K-major, M = 128, N = 128.
constexpr uint32_t kGramIdesc = (1u << 4)                       // D fp32
                                | (1u << 7)                     // A bf16
                                | (1u << 10)                    // B bf16
                                | (static_cast<uint32_t>(kGramN >> 3) << 17)
                                | (static_cast<uint32_t>(kGramH >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kGramIdesc), "r"(accumulate)
        : "memory");
}

// Arrives once on `bar` when every tcgen05.mma this thread issued before is done.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void named_sync_id(uint32_t id, uint32_t threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void tmem_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's accumulator lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Sum of squares of the key row `row` of a staged operand (its 128-byte
// rows; the swizzle permutes 16-byte chunks within a row, which a sum over
// the row does not see).  The chunks are visited starting at row % 8, so
// that neighbouring threads (neighbouring rows, 128 bytes apart) read
// different banks.
template <int PANELS>
__device__ __forceinline__ float row_sq(const uint8_t *base, int panel_bytes, int row)
{
    float s = 0.f;
#pragma unroll
    for (int p = 0; p < PANELS; ++p) {
        const uint32_t a = smem_u32(base + p * panel_bytes + row * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 v = ld_shared_v4(a + ((j + row) & 7) * 16);
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h[i]);
                s = fmaf(f.x, f.x, s);
                s = fmaf(f.y, f.y, s);
            }
        }
    }
    return s;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kGramThreads, 1) zp_gram_redundancy_kernel(const GramRedArgs a)
{
    using S = GramSmem<D>;
    constexpr int PANELS = S::PANELS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = sm + S::off_a;
    uint8_t *sB = sm + S::off_b;
    float *sInv = reinterpret_cast<float *>(sm + S::off_inv);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::off_bar);
    uint64_t *fullA = bars, *fullB = bars + 1, *emptyB = bars + 1 + kGramNS,
             *accFull = bars + 1 + 2 * kGramNS, *accEmpty = accFull + 2, *emptyA = accEmpty + 2,
             *done = emptyA + 1;
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(sm + S::off_tmem);

    const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5;
    const int n_items = a.units * a.row_tiles;
    // a contiguous range of items per CTA: a unit's row tiles run back to back
    // on one SM (its keys then stay in L2 between them, and their inverse
    // norms in shared memory)
    const int per = (n_items + gridDim.x - 1) / gridDim.x;
    const int w_begin = min(n_items, static_cast<int>(blockIdx.x) * per);
    const int w_end = min(n_items, w_begin + per);

    if (tid == 0) {
        mbar_init(fullA, 1);
        mbar_init(emptyA, 2);  // the item's last products and its row norms taken
        mbar_init(done, 1);
        for (int s = 0; s < kGramNS; ++s) {
            mbar_init(&fullB[s], 1);
            mbar_init(&emptyB[s], 2);  // the products' commit and the norms' arrival
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accFull[b], 1);
            mbar_init(&accEmpty[b], kGramEW / 2);  // one arrival per warp of its set
        }
        fence_mbar_init();
    }
    if (wi == 1) {  // the whole warp: allocation is warp-wide
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(sTmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tmem = *sTmem;
    bool bad = false;

    // Item w: unit u = w / row_tiles (h fastest, then the request, then the
    // layer), keys t0 .. t0 + 255.  Every role walks the same items in the
    // same order, so the pipeline counters agree without communication.
    struct Item {
        int u, h, l, t0, T, nblk, n_tiles;
        const int32_t *trow;
        int state;  // 0 work, 1 nothing to do (t0 >= T), 2 bad length, 3 bad request index
    };
    auto decode = [&](int w) {
        Item it;
        it.u = w / a.row_tiles;
        it.h = it.u % a.Hkv;
        const int r = (it.u / a.Hkv) % a.R;
        it.l = it.u / (a.Hkv * a.R);
        it.t0 = (w - it.u * a.row_tiles) * kGramM;
        const int row = a.req_idx ? a.req_idx[r] : r;
        const bool row_ok = row >= 0 && row < a.num_rows;
        it.T = row_ok ? a.lengths[row] : 0;
        it.trow = a.tables + (size_t)(row_ok ? row : 0) * a.stride;
        it.nblk = (it.T + kBlk - 1) / kBlk;  // cache blocks holding the unit's keys
        it.n_tiles = (it.T + kGramN - 1) / kGramN;
        it.state = !row_ok ? 3 : (it.T < 0 || it.T > a.stride * kBlk) ? 2 : it.t0 >= it.T ? 1 : 0;
        return it;
    };

    if (wi == 0) {
        // ------------------------------------------------------- producer
        // the whole warp: lane q reads the id of the q-th block of a tile (one
        // round trip for all of them), lane 0 issues the loads
        constexpr int QA = kGramM / kBlk, QB = kGramN / kBlk;  // blocks per A, per B tile
        static_assert(QA * PANELS <= 32 && QB * PANELS <= 32, "one box per lane");
        // the y coordinate (pool row) of cache block q of the item's unit, or
        // a negative one past the unit's blocks (the load then fills zeros)
        auto block_y = [&](const Item &it, int q) {
            if (q >= it.nblk)
                return -kBlk;
            const int blk = it.trow[q];
            if (blk < 0 || blk >= a.num_blocks) {
                set_error(a.sticky, ZP_ERR_DEVICE_CHECK);
                return -kBlk;
            }
            return (blk * a.Hkv + it.h) * kBlk;
        };
        uint32_t ia = 0, gt = 0;  // items loaded, B tiles loaded (over all items)
        for (int w = w_begin; w < w_end && !bad; ++w) {
            const Item it = decode(w);
            if (it.state != 0) {
                if (it.state >= 2 && it.t0 == 0 && lane == 0)
                    set_error(a.sticky, it.state == 2 ? ZP_ERR_DEVICE_CHECK : ZP_ERR_INVALID_ARG);
                continue;
            }
            const CUtensorMap *kmap = a.kmaps + it.l;
            const int ya = lane < QA ? block_y(it, it.t0 / kBlk + lane) : 0;
            if (lane == 0) {
                bad = ia > 0 && !mbar_wait(emptyA, (ia - 1) & 1);
                if (!bad)
                    mbar_arrive_expect_tx(fullA, S::A_BYTES);
            }
            bad = __shfl_sync(0xffffffffu, bad, 0);
            if (bad)
                break;
            {  // one box (a block's 16 rows, 64 dims) per lane
                const int q = lane / PANELS, p = lane % PANELS;
                const int y = __shfl_sync(0xffffffffu, ya, q & 31);
                const int g = q / (kGramH / kBlk), qq = q % (kGramH / kBlk);
                if (q < QA)
                    tma_load_2d(sA + (g * PANELS + p) * S::A_PANEL + qq * kBlk * 128, kmap,
                                p * 64, y, fullA);
            }
            ++ia;
            for (int t = 0; t < it.n_tiles; ++t) {
                const int s = gt % kGramNS;
                const int yb = lane < QB ? block_y(it, t * QB + lane) : 0;
                if (lane == 0) {
                    bad = gt >= kGramNS && !mbar_wait(&emptyB[s], ((gt / kGramNS) - 1) & 1);
                    if (!bad)
                        mbar_arrive_expect_tx(&fullB[s], S::B_STAGE);
                }
                bad = __shfl_sync(0xffffffffu, bad, 0);
                if (bad)
                    break;
                uint8_t *dst = sB + s * S::B_STAGE;
                {  // one box per lane
                    const int q = lane / PANELS, p = lane % PANELS;
                    const int y = __shfl_sync(0xffffffffu, yb, q & 31);
                    if (q < QB)
                        tma_load_2d(dst + p * S::B_PANEL + q * kBlk * 128, kmap, p * 64, y,
                                    &fullB[s]);
                }
                ++gt;
            }
        }
        // every copy issued has landed before the CTA may exit (immediate
        // unless a consumer gave up)
        if (lane == 0) {
            bool ok = ia == 0 || mbar_wait(fullA, (ia - 1) & 1);
            for (uint32_t j = gt > kGramNS ? gt - kGramNS : 0; j < gt; ++j)
                ok &= mbar_wait(&fullB[j % kGramNS], (j / kGramNS) & 1);
            bad |= !ok;
        }
    } else if (wi == 1) {
        // ------------------------------------------------------- products
        if (lane == 0) {
            uint32_t ia = 0, gt = 0, use[2] = {0u, 0u};
            for (int w = w_begin; w < w_end && !bad; ++w) {
                const Item it = decode(w);
                if (it.state != 0)
                    continue;
                if (!mbar_wait(fullA, ia & 1)) {
                    bad = true;
                    break;
                }
                for (int t = 0; t < it.n_tiles; ++t, ++gt) {
                    const int s = gt % kGramNS, b = t & 1;
                    const uint32_t j = use[b]++;
                    if (!mbar_wait(&fullB[s], (gt / kGramNS) & 1) ||
                        (j > 0 && !mbar_wait(&accEmpty[b], (j - 1) & 1))) {
                        bad = true;
                        break;
                    }
                    tmem_fence_after();
                    const uint32_t bBase = smem_u32(sB + s * S::B_STAGE);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t koff = (ks & 3) * 32u;  // 16 dims within a 128-byte row
                        const uint64_t bd = sw128_desc(bBase + (ks >> 2) * S::B_PANEL + koff);
#pragma unroll
                        for (int g = 0; g < 2; ++g) {
                            const uint64_t ad = sw128_desc(
                                smem_u32(sA + (g * PANELS + (ks >> 2)) * S::A_PANEL) + koff);
                            umma_bf16(tmem + static_cast<uint32_t>((b * 2 + g) * kGramN), ad, bd,
                                      ks > 0);
                        }
                    }
                    umma_commit(&emptyB[s]);    // this stage's operands are read
                    umma_commit(&accFull[b]);  // both halves of buffer b are complete
                }
                if (bad)
                    break;
                umma_commit(emptyA);  // the item's products no longer read A
                ++ia;
            }
            // every product issued is done before the tensor memory is freed
            umma_commit(done);
            bad |= !mbar_wait(done, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- reduction
        // two sets of 8 warps, set b reducing the tiles t = b, b + 2, ... of
        // each item (accumulator buffer b), each warp 32 lanes of one 128-key
        // half.  The barriers a set passes depend only on the items, never on
        // a timeout, so a warp that gave up still passes all of them.
        constexpr int NSET = kGramEW / 2 * 32;   // threads per set
        const int w2 = wi - 2;                   // 0 .. 15
        const int set = w2 >> 3;
        const int es = (w2 & 7) * 32 + lane;     // 0 .. 255 within the set
        const int quarter = wi & 3;              // tensor-memory lanes 32*quarter ..
        const int g = (w2 & 7) >> 2;             // accumulator half (of the item's keys)
        const int tr = quarter * 32 + lane;      // this thread's key t0 + g*128 + tr
        float *sPart = reinterpret_cast<float *>(sm + S::off_part);
        float *sInvU = reinterpret_cast<float *>(sm + S::off_invu);
        uint32_t ia = 0, gt = 0, use = 0, ic = 0;
        int cur_u = -1;  // the unit whose key norms sInvU holds
        for (int w = w_begin; w < w_end; ++w) {
            const Item it = decode(w);
            if (it.state != 0)
                continue;
            const int T = it.T;
            // a unit's first item here computes the inverse norms of all its
            // keys (each set those of its tiles) into sInvU, the next ones
            // read them; units too long for it take them per stage
            const bool cached = T <= kGramUMax;
            const bool fresh = !cached || it.u != cur_u;
            cur_u = cached ? it.u : -1;
            float inv_t = 0.f;
            if (set == 0) {
                // the norm of this thread's key t, before A is released (only
                // set 0 waits for A: its arrival gates the next load, so the
                // phase it waits for cannot be overtaken)
                if (!bad)
                    bad = !mbar_wait(fullA, ia & 1);
                ++ia;
                if (!bad) {
                    const float sq_t =
                        row_sq<PANELS>(sA + g * PANELS * S::A_PANEL, S::A_PANEL, tr);
                    inv_t = sq_t > 0.f ? rsqrtf(sq_t) : 0.f;
                }
                named_sync_id(1, NSET);
                if (es == 0)
                    mbar_arrive(emptyA);
            }
            float sum = 0.f;
            for (int t = 0; t < it.n_tiles; ++t, ++gt) {
                if ((t & 1) != set)
                    continue;
                const int s = gt % kGramNS, b = set;
                const uint32_t j = use++;
                float *inv_row = cached ? sInvU + t * kGramN : sInv + s * kGramN;
                if (fresh) {
                    if (!bad)
                        bad = !mbar_wait(&fullB[s], (gt / kGramNS) & 1);
                    if (es < kGramN) {  // inverse norm of this stage's key es
                        const int k = t * kGramN + es;
                        const float sq =
                            bad ? 0.f : row_sq<PANELS>(sB + s * S::B_STAGE, S::B_PANEL, es);
                        inv_row[es] = (k < T && sq > 0.f) ? rsqrtf(sq) : 0.f;
                    }
                    named_sync_id(1 + set, NSET);
                    if (es == 0)
                        mbar_arrive(&emptyB[s]);
                } else if (es == 0) {
                    // nothing of the stage is read here: release it once it
                    // holds this tile (an earlier arrival could close the
                    // stage's previous phase)
                    if (!bad)
                        bad = !mbar_wait(&fullB[s], (gt / kGramNS) & 1);
                    mbar_arrive(&emptyB[s]);
                }
                if (!bad)
                    bad = !mbar_wait(&accFull[b], j & 1);
                tmem_fence_after();
                bad = __any_sync(0xffffffffu, bad);  // tcgen05.ld is warp-collective
                if (!bad) {
                    const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                           static_cast<uint32_t>((b * 2 + g) * kGramN);
                    const float4 *inv = reinterpret_cast<const float4 *>(inv_row);
                    const int lim = T - t * kGramN;  // columns at and past it are not keys
#pragma unroll 1
                    for (int ch = 0; ch < kGramN / 32; ++ch) {
                        float v[32];
                        tmem_ld32(tbase + ch * 32, v);
                        if (ch * 32 + 32 <= lim) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float4 wv = inv[ch * 8 + i];
                                sum = fmaf(v[4 * i], wv.x, sum);
                                sum = fmaf(v[4 * i + 1], wv.y, sum);
                                sum = fmaf(v[4 * i + 2], wv.z, sum);
                                sum = fmaf(v[4 * i + 3], wv.w, sum);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (ch * 32 + i < lim)
                                    sum = fmaf(v[i], inv_row[ch * 32 + i], sum);
                        }
                    }
                }
                tmem_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&accEmpty[b]);
            }
            // the two sets' partial sums, double-buffered by item: a set can
            // be at most one item ahead of the other at this barrier
            float *part = sPart + (ic & 1) * 2 * kGramM;
            part[set * kGramM + g * kGramH + tr] = sum;
            named_sync_id(3, 2 * NSET);
            const int tt = it.t0 + g * kGramH + tr;
            if (set == 0 && tt < T && !bad) {
                const float tot = part[g * kGramH + tr] + part[kGramM + g * kGramH + tr];
                const float pairs = T > 1 ? 1.0f / static_cast<float>(T - 1) : 0.f;
                a.red_out[(size_t)it.u * a.T_cap + tt] =
                    inv_t > 0.f ? (tot * inv_t - 1.0f) * pairs : 0.f;
            }
            ++ic;
        }
    }
    if (bad)
        set_error(a.sticky, ZP_ERR_TIMEOUT);
    tmem_fence_before();
    __syncthreads();
    if (wi == 1) {
        tmem_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

template <int D>
static cudaError_t launch_gram_t(const GramRedArgs &a, int ctas, cudaStream_t s)
{
    using S = GramSmem<D>;
    auto kern = zp_gram_redundancy_kernel<D>;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               S::ALLOC);
    if (e != cudaSuccess)
        return e;
    kern<<<static_cast<unsigned>(ctas), kGramThreads, S::ALLOC, s>>>(a);
    return cudaGetLastError();
}

int gram_row_tiles(int T_cap) { return (T_cap + kGramM - 1) / kGramM; }

cudaError_t launch_gram_redundancy(const GramRedArgs &a, int d, int units, int sms,
                                   cudaStream_t s)
{
    const long long items = static_cast<long long>(units) * a.row_tiles;
    if (items >= (1ll << 31) || sms < 1)
        return cudaErrorInvalidValue;
    GramRedArgs b = a;
    b.units = units;
    const int ctas = static_cast<int>(items < sms ? items : sms);  // one CTA per SM
    if (ctas < 1)
        return cudaSuccess;
    if (d == 64)
        return launch_gram_t<64>(b, ctas, s);
    if (d == 128)
        return launch_gram_t<128>(b, ctas, s);
    return cudaErrorInvalidValue;
}

}  // namespace zp
