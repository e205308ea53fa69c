// zp_aux.cuh -- launch arguments and launchers of the kernels off the
// compression path: the all-keys redundancy ablation (zp_redundancy_global.cu)
// and whole-request block allocation / release / fork (zp_blocks.cu).  Internal: not
// part of the C ABI.
#pragma once

#include "zp_internal.cuh"

namespace zp {

// units u = (l*R + r)*Hkv + h
struct GlobalRedArgs {
    __nv_bfloat16 *const *kpools;  // device array of the L K pools
    const int32_t *tables;
    int32_t stride, num_rows;
    const int32_t *lengths;
    const int32_t *req_idx;
    int32_t R, Hkv, num_blocks, T_cap;
    float *red_out;  // [units][T_cap]
    int32_t *sticky;
};

cudaError_t launch_global_redundancy(const GlobalRedArgs &a, int d, int units, cudaStream_t s);

// The same score from the dense Gram of every unit (zp_redundancy_gram.cu).
struct GramRedArgs {
    const CUtensorMap *kmaps;  // [L] the K pool maps (128-byte swizzle, box {64, 16})
    const int32_t *tables;
    int32_t stride, num_rows;
    const int32_t *lengths;
    const int32_t *req_idx;
    int32_t R, Hkv, num_blocks, T_cap;
    int32_t row_tiles;  // work items per unit: ceil(T_cap / 256)
    int32_t units;      // (request, layer, kv head) units; set by the launcher
    float *red_out;     // [units][T_cap]
    int32_t *sticky;
};

int gram_row_tiles(int T_cap);
cudaError_t launch_gram_redundancy(const GramRedArgs &a, int d, int units, int sms,
                                   cudaStream_t s);  // one CTA per SM (sms of them at most)

cudaError_t launch_alloc_rows(const Workspace &ws, int32_t *block_tables, int32_t bt_stride,
                              int32_t num_rows, int32_t *lengths, const int32_t *req_idx,
                              int32_t R, const int32_t *counts, int32_t num_blocks,
                              const zp_block_pool *pool, cudaStream_t s);
cudaError_t launch_fork_rows(const Workspace &ws, int32_t *block_tables, int32_t bt_stride,
                             int32_t num_rows, int32_t *lengths, const int32_t *src,
                             const int32_t *dst, int32_t n, int32_t num_blocks, int32_t *refcount,
                             cudaStream_t s);
cudaError_t launch_release_rows(const Workspace &ws, int32_t *block_tables, int32_t bt_stride,
                                int32_t num_rows, int32_t *lengths, const int32_t *req_idx,
                                int32_t R, int32_t num_blocks, const zp_block_pool *pool,
                                cudaStream_t s);

}  // namespace zp
