// zp_redundancy_global.cu -- redundancy of every key against ALL keys of its
// unit: the O(N^2 b^2) score that the Lightning Redundancy Score replaces
// (Zipage, gist.science: Dutch "Methodologie" §5, Korean "방법론" E), kept as
// an ablation next to the block-local score of the compression kernels.
//
// With the mean-cosine definition the pairwise sum collapses: for a key with
// nonzero norm, sum_{k != j} cos(K_j, K_k) = k^_j . S - 1 with k^ = K/|K| and
// S = sum over the unit's nonzero keys of k^ (a zero key adds nothing to S and
// has redundancy 0).  One CTA per (request, layer, kv head) therefore makes
// two passes over the unit's T keys, O(T d) each: S, then every key's dot
// with S.  A row of d bf16 is d/8 lanes of 16-byte loads; the norms are
// reduced across those lanes with shuffles.
#include "zp_aux.cuh"

namespace zp {

constexpr int kGrThreads = 256;

template <int D>
__global__ void __launch_bounds__(kGrThreads) zp_global_redundancy_kernel(const GlobalRedArgs a)
{
    constexpr int LPR = D / 8;            // lanes per key row (16-byte chunks)
    constexpr int GROUPS = kGrThreads / LPR;
    __shared__ float s_part[GROUPS][D];
    __shared__ float s_sum[D];
    const int u = blockIdx.x;
    const int h = u % a.Hkv, r = (u / a.Hkv) % a.R, l = u / (a.Hkv * a.R);
    int row = a.req_idx ? a.req_idx[r] : r;
    const bool row_ok = row >= 0 && row < a.num_rows;
    int T = row_ok ? a.lengths[row] : 0;
    if (!row_ok || T < 0 || T > a.stride * kBlk) {
        if (threadIdx.x == 0)
            set_error(a.sticky, row_ok ? ZP_ERR_DEVICE_CHECK : ZP_ERR_INVALID_ARG);
        return;
    }
    const int32_t *trow = a.tables + (size_t)row * a.stride;
    const __nv_bfloat16 *pool = a.kpools[l];
    const int lane = threadIdx.x & 31, sub = lane % LPR;
    const int grp = threadIdx.x / LPR;  // one key row at a time per lane group

    // the 8 elements of key t this lane holds, widened; false past the pool
    auto load = [&](int t, float (&x)[8]) {
        const int blk = trow[t / kBlk];
        if (blk < 0 || blk >= a.num_blocks) {
            set_error(a.sticky, ZP_ERR_DEVICE_CHECK);
            return false;
        }
        const uint4 v = ld_global_nc_v4(pool + (((size_t)blk * a.Hkv + h) * kBlk + t % kBlk) * D +
                                        sub * 8);
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(p[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
        return true;
    };
    // sum over the lanes of one row group
    auto row_sum = [&](float v) {
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1)
            v += __shfl_xor_sync(0xffffffffu, v, o);
        return v;
    };
    const int steps = (T + GROUPS - 1) / GROUPS;  // uniform trip count: shuffles need whole warps

    // pass 1: S = sum of the normalised nonzero keys
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int it = 0; it < steps; ++it) {
        const int t = it * GROUPS + grp;
        float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const bool ok = t < T && load(t, x);
        float n2 = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            n2 += x[i] * x[i];
        n2 = row_sum(n2);
        const float inv = ok && n2 > 0.f ? rsqrtf(n2) : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] += x[i] * inv;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        s_part[grp][sub * 8 + i] = acc[i];
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kGrThreads) {
        float v = 0.f;
        for (int g = 0; g < GROUPS; ++g)
            v += s_part[g][c];
        s_sum[c] = v;
    }
    __syncthreads();
    float sv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        sv[i] = s_sum[sub * 8 + i];

    // pass 2: red_j = (k^_j . S - 1) / (T - 1) for a nonzero key, else 0
    const float inv_pairs = T > 1 ? 1.0f / static_cast<float>(T - 1) : 0.f;
    float *out = a.red_out + (size_t)u * a.T_cap;
    for (int it = 0; it < steps; ++it) {
        const int t = it * GROUPS + grp;
        float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const bool ok = t < T && load(t, x);
        float n2 = 0.f, dot = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            n2 += x[i] * x[i];
            dot += x[i] * sv[i];
        }
        n2 = row_sum(n2);
        dot = row_sum(dot);
        if (ok && sub == 0)
            out[t] = n2 > 0.f ? (dot * rsqrtf(n2) - 1.0f) * inv_pairs : 0.f;
    }
}

cudaError_t launch_global_redundancy(const GlobalRedArgs &a, int d, int units, cudaStream_t s)
{
    if (d == 64)
        zp_global_redundancy_kernel<64><<<static_cast<unsigned>(units), kGrThreads, 0, s>>>(a);
    else if (d == 128)
        zp_global_redundancy_kernel<128><<<static_cast<unsigned>(units), kGrThreads, 0, s>>>(a);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace zp
