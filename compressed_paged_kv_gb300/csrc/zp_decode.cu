// zp_decode.cu -- paged decode attention over block tables.
//
// "Paged KV cache and continuous batching for LLMs" ("How it works"): a
// request's KV cache lives in fixed-size blocks that need not be contiguous,
// reached through its block table.  One query token per request attends to
// its lengths[row] cached tokens.
//
// Grid (split, kv head, request), 4 warps per CTA.  A CTA owns a contiguous
// range of `bps` blocks of one (request, kv head); warp w takes every fourth
// block of that range.  Each warp runs its own TMA pipeline (3 stages of one
// K block + one V block, 128-byte swizzle) and keeps an online softmax for
// the G query heads of the group (padded to the 16 rows of an mma tile):
// S = Q K^T and O += P V on the tensor cores (mma.sync bf16, fp32
// accumulate, P rounded to bf16 for the second product).  Warps merge in
// shared memory; with more than one split the CTA writes (m, l, o) partials
// that zp_decode_combine merges with a log-sum-exp.  The two tensor maps come
// from device memory (the handle's per-layer maps) or, for the allocation-
// free entry point, by value in the launch parameters.
#include "zp_internal.cuh"

namespace zp {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecStages = 3;

template <int D>
struct DecodeSmem {
    static constexpr int Q_BYTES = 16 * D * 2;
    static constexpr int KV_BYTES = kBlk * D * 2;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int off_q = 0;
    static constexpr int off_stage = off_q + Q_BYTES;
    static constexpr int STAGES_BYTES = kDecWarps * kDecStages * STAGE_BYTES;
    // merge area (reuses the stages once every load has been consumed)
    static constexpr int MERGE_BYTES = kDecWarps * 16 * (D + 2) * 4;
    static_assert(MERGE_BYTES <= STAGES_BYTES, "merge area must fit in the stage area");
    static constexpr int off_bar = off_stage + STAGES_BYTES;
    static constexpr int BYTES = off_bar + kDecWarps * kDecStages * 8;
    static constexpr int ALLOC = BYTES + 1024;
};

// MAPV: the tensor maps come by value in the parameters (a.kmap_v, a.vmap_v)
template <int D, bool MAPV>
__global__ void __launch_bounds__(kDecThreads, 2)
    zp_decode_kernel(const __grid_constant__ DecodeArgs a)
{
    pdl_wait();  // launched early: everything of the kernels before it is visible from here
    using S = DecodeSmem<D>;
    constexpr int CPR = D / 8;
    constexpr int HALVES = D / 64;
    constexpr int KS = D / 16;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = sm + S::off_q;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + S::off_bar);

    const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5;
    const int split = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
    const int G = a.Hq / a.Hkv;
    int row = a.req_idx ? a.req_idx[r] : r;
    bool row_ok = row >= 0 && row < a.num_rows;
    int len = row_ok ? a.lengths[row] : 0;
    if (!row_ok || len < 0 || len > a.stride * kBlk) {
        if (tid == 0 && split == 0 && h == 0)
            set_error(a.sticky, row_ok ? ZP_ERR_DEVICE_CHECK : ZP_ERR_INVALID_ARG);
        len = 0;
        row = 0;
    }
    const int nblk = (len + kBlk - 1) / kBlk;
    const int b_begin = split * a.bps;
    const int b_end = min(nblk, b_begin + a.bps);

    // query rows of the group -> shared memory (swizzled), then A fragments
    {
        const __nv_bfloat16 *qsrc = a.q + ((size_t)r * a.Hq + (size_t)h * G) * D;
        const uint32_t qb = smem_u32(sQ);
        for (int c = tid; c < 16 * CPR; c += kDecThreads) {
            const int rr = c / CPR, ch = c - rr * CPR;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (rr < G)
                v = ld_global_nc_v4(qsrc + (size_t)rr * D + ch * 8);
            st_shared_v4(qb + swz(rr, ch, 16), v);
        }
    }
    if (tid < kDecWarps * kDecStages)
        mbar_init(&bars[tid], 1);
    if (tid == 0)
        fence_mbar_init();
    __syncthreads();

    uint32_t qa[KS][4];
    {
        const uint32_t qb = smem_u32(sQ);
        const int mi = lane >> 3;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
            ldsm_x4(qb + swz((mi & 1) * 8 + (lane & 7), ks * 2 + (mi >> 1), 16), qa[ks]);
    }

    const int first = b_begin + wi;
    const int my_n = first < b_end ? (b_end - first + kDecWarps - 1) / kDecWarps : 0;
    uint8_t *my_stage = sm + S::off_stage + wi * kDecStages * S::STAGE_BYTES;
    uint64_t *my_bar = bars + wi * kDecStages;
    const int32_t *trow = a.tables + (size_t)row * a.stride;
    const CUtensorMap *kmap = MAPV ? &a.kmap_v : a.kmap;
    const CUtensorMap *vmap = MAPV ? &a.vmap_v : a.vmap;

    auto issue = [&](int i) {
        int blk = trow[first + i * kDecWarps];
        if (blk < 0 || blk >= a.num_blocks) {
            set_error(a.sticky, ZP_ERR_DEVICE_CHECK);
            blk = 0;
        }
        const int s = i % kDecStages;
        uint8_t *kd = my_stage + s * S::STAGE_BYTES;
        uint8_t *vd = kd + S::KV_BYTES;
        mbar_arrive_expect_tx(&my_bar[s], S::STAGE_BYTES);
        const int y = (blk * a.Hkv + h) * kBlk;
#pragma unroll
        for (int hf = 0; hf < HALVES; ++hf) {
            tma_load_2d(kd + hf * kBlk * 128, kmap, hf * 64, y, &my_bar[s]);
            tma_load_2d(vd + hf * kBlk * 128, vmap, hf * 64, y, &my_bar[s]);
        }
    };
    if (lane == 0)
        for (int i = 0; i < my_n && i < kDecStages; ++i)
            issue(i);

    float m_run[2] = {-1e30f, -1e30f};
    float l_run[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            o[nt][e] = 0.f;
    bool ok = true;

    for (int i = 0; i < my_n; ++i) {
        const int s = i % kDecStages;
        ok &= mbar_wait(&my_bar[s], (i / kDecStages) & 1);
        const int tok0 = (first + i * kDecWarps) * kBlk;
        if (len - tok0 < kBlk) {
            // the slots past the length of a partial last block: their keys get
            // probability 0, but 0 times a NaN or infinite V element (stale or
            // never-written pool bytes) is NaN, so their V rows are cleared
            uint8_t *vd = my_stage + s * S::STAGE_BYTES + S::KV_BYTES;
            const int fill = len - tok0;  // >= 1: the block holds a token below len
            constexpr int CPR2 = D / 8;   // 16-byte chunks per row (over the 64-dim panels)
            for (int c = lane; c < (kBlk - fill) * CPR2; c += 32) {
                const int rr = fill + c / CPR2, ch = c % CPR2;
                st_shared_v4(smem_u32(vd + (ch >> 3) * kBlk * 128 + rr * 128 + (ch & 7) * 16),
                             make_uint4(0u, 0u, 0u, 0u));
            }
            __syncwarp();
        }
        const uint32_t kb_base = smem_u32(my_stage + s * S::STAGE_BYTES);
        const uint32_t vb_base = kb_base + S::KV_BYTES;
        const int mi = lane >> 3;

        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t kb[4];
            ldsm_x4(kb_base + swz((mi >> 1) * 8 + (lane & 7), ks * 2 + (mi & 1), kBlk), kb);
            mma_bf16(sacc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], kb[0], kb[1]);
            mma_bf16(sacc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], kb[2], kb[3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = nt * 8 + (lane & 3) * 2 + (e & 1);
                float v = sacc[nt][e] * a.logit_scale;
                if (tok0 + key >= len)
                    v = -INFINITY;
                sacc[nt][e] = v;
            }
        // online softmax, rows lane/4 (hh = 0) and lane/4 + 8 (hh = 1)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float mx = fmaxf(fmaxf(sacc[0][hh * 2], sacc[0][hh * 2 + 1]),
                             fmaxf(sacc[1][hh * 2], sacc[1][hh * 2 + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run[hh], mx);
            const float corr = ex2_approx(m_run[hh] - m_new);
            m_run[hh] = m_new;
            l_run[hh] *= corr;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                o[nt][hh * 2] *= corr;
                o[nt][hh * 2 + 1] *= corr;
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                sacc[nt][hh * 2] = ex2_approx(sacc[nt][hh * 2] - m_new);
                sacc[nt][hh * 2 + 1] = ex2_approx(sacc[nt][hh * 2 + 1] - m_new);
                l_run[hh] += sacc[nt][hh * 2] + sacc[nt][hh * 2 + 1];
            }
        }
        const uint32_t pa0 = pack_bf16x2(sacc[0][0], sacc[0][1]);
        const uint32_t pa1 = pack_bf16x2(sacc[0][2], sacc[0][3]);
        const uint32_t pa2 = pack_bf16x2(sacc[1][0], sacc[1][1]);
        const uint32_t pa3 = pack_bf16x2(sacc[1][2], sacc[1][3]);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
            uint32_t vb[4];
            ldsm_x4_t(vb_base + swz((mi & 1) * 8 + (lane & 7), dp * 2 + (mi >> 1), kBlk), vb);
            mma_bf16(o[2 * dp], pa0, pa1, pa2, pa3, vb[0], vb[1]);
            mma_bf16(o[2 * dp + 1], pa0, pa1, pa2, pa3, vb[2], vb[3]);
        }
        __syncwarp();
        if (lane == 0 && i + kDecStages < my_n) {
            fence_proxy_async_smem();
            issue(i + kDecStages);
        }
    }
    if (!ok && lane == 0)
        set_error(a.sticky, ZP_ERR_TIMEOUT);
    pdl_launch_dependents();  // the combine kernel may be scheduled
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 1);
        l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 2);
    }
    __syncthreads();  // every stage consumed: reuse the area for the merge

    float *mrg = reinterpret_cast<float *>(sm + S::off_stage);  // [warp][16][D + 2]
    {
        float *mine = mrg + wi * 16 * (D + 2);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int rr = (lane >> 2) + hh * 8;
            if ((lane & 3) == 0) {
                mine[rr * (D + 2) + D] = m_run[hh];
                mine[rr * (D + 2) + D + 1] = l_run[hh];
            }
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                const int c = nt * 8 + (lane & 3) * 2;
                mine[rr * (D + 2) + c] = o[nt][hh * 2];
                mine[rr * (D + 2) + c + 1] = o[nt][hh * 2 + 1];
            }
        }
    }
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += kDecThreads) {
        const int g = idx / D, c = idx - g * D;
        float M = -1e30f;
#pragma unroll
        for (int w2 = 0; w2 < kDecWarps; ++w2)
            M = fmaxf(M, mrg[(w2 * 16 + g) * (D + 2) + D]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kDecWarps; ++w2) {
            const float *src = mrg + (w2 * 16 + g) * (D + 2);
            const float f = exp2f(src[D] - M);
            L += src[D + 1] * f;
            O += src[c] * f;
        }
        const int hq = h * G + g;
        if (a.splits == 1) {
            a.out[((size_t)r * a.Hq + hq) * D + c] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
        } else {
            float *p = a.part + (((size_t)r * a.Hq + hq) * a.splits + split) * (D + 2);
            p[c] = O;
            if (c == 0) {
                p[D] = M;
                p[D + 1] = L;
            }
        }
    }
}

template <int D>
__global__ void __launch_bounds__(D) zp_decode_combine(const DecodeArgs a)
{
    pdl_wait();
    const int rh = blockIdx.x;  // r * Hq + hq
    const int c = threadIdx.x;
    const float *base = a.part + (size_t)rh * a.splits * (D + 2);
    float M = -1e30f;
    for (int s = 0; s < a.splits; ++s)
        M = fmaxf(M, base[s * (D + 2) + D]);
    float L = 0.f, O = 0.f;
    for (int s = 0; s < a.splits; ++s) {
        const float f = exp2f(base[s * (D + 2) + D] - M);
        L += base[s * (D + 2) + D + 1] * f;
        O += base[s * (D + 2) + c] * f;
    }
    a.out[(size_t)rh * D + c] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
}

template <int D, bool MAPV>
static cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t s)
{
    using Sm = DecodeSmem<D>;
    cudaError_t err = cudaFuncSetAttribute(zp_decode_kernel<D, MAPV>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::ALLOC);
    if (err != cudaSuccess)
        return err;
    // both launched early (programmatic serialisation); each waits at its start
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.splits), static_cast<unsigned>(a.Hkv),
                       static_cast<unsigned>(a.R));
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.dynamicSmemBytes = Sm::ALLOC;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, zp_decode_kernel<D, MAPV>, a);
    if (err != cudaSuccess || a.splits == 1)
        return err;
    cfg.gridDim = dim3(static_cast<unsigned>(a.R * a.Hq), 1, 1);
    cfg.blockDim = dim3(D, 1, 1);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, zp_decode_combine<D>, a);
}

cudaError_t launch_decode(const DecodeArgs &a, int d, cudaStream_t s)
{
    if (d == 64)
        return launch_decode_t<64, false>(a, s);
    if (d == 128)
        return launch_decode_t<128, false>(a, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_mapv(const DecodeArgs &a, int d, cudaStream_t s)
{
    if (d == 64)
        return launch_decode_t<64, true>(a, s);
    if (d == 128)
        return launch_decode_t<128, true>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace zp
