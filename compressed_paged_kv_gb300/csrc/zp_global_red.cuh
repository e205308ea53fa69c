// zp_global_red.cuh -- launch arguments of the all-keys redundancy kernel
// (zp_redundancy_global.cu).  Internal: not part of the C ABI.
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

}  // namespace zp
