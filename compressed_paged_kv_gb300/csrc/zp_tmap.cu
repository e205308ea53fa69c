// zp_tmap.cu -- the TMA tensor maps of the K and V pools (host code).  A
// pool [num_blocks][Hkv][b][d] bf16 is seen as a 2D tensor of
// num_blocks * Hkv * b rows of d elements.
#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include "zp_internal.cuh"

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

namespace zp {

// Box {64 columns, b rows}, 128-byte swizzle: one (block, kv head) slab is
// loaded as d/64 boxes.  L2 promotion to 128 bytes, the box rows' own size
// (256-byte promotion measured ~0.7 % slower on the compression).
bool encode_pool_map(CUtensorMap *map, const void *pool, int num_blocks, int hkv, int d)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d),
                          static_cast<cuuint64_t>(num_blocks) * hkv * zp::kBlk};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(zp::kBlk)};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

// The same 2D view with a box of one whole row ({d columns, 1 row}) and no
// swizzle: the compaction gathers four arbitrary pool rows per load
// (tile::gather4, whose box is one row high) into a [16][d] destination slab.
bool encode_row_map(CUtensorMap *map, const void *pool, int num_blocks, int hkv, int d)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d),
                          static_cast<cuuint64_t>(num_blocks) * hkv * zp::kBlk};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(d), 1};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS;
}

}  // namespace zp
