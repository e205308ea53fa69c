// zp_compress_d64.cu -- fused compression kernels for head dim 64.
#include "zp_compress_kernel.cuh"

namespace zp {

cudaError_t launch_compress_d64(const CompressArgs &a, CompressShape shape, int mt, int units,
                                cudaStream_t s)
{
    return launch_compress_for_d<64>(a, shape, mt, units, s);
}

int resident_clusters_d64(CompressShape shape, int mt)
{
    return resident_clusters_for_d<64>(shape, mt);
}

}  // namespace zp
