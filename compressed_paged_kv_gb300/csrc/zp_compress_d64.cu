// zp_compress_d64.cu -- fused compression kernels for head dim 64.
#include "zp_compress_kernel.cuh"

namespace zp {

cudaError_t launch_compress_d64(const CompressArgs &a, CompressShape shape, int mt, int units,
                                cudaStream_t s)
{
    return launch_compress_for_d<64>(a, shape, mt, units, s);
}

}  // namespace zp
