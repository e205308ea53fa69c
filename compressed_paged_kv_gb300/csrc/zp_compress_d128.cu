// zp_compress_d128.cu -- fused compression kernels for head dim 128, and the
// device check of 16-CTA cluster residency.
#include "zp_compress_kernel.cuh"

namespace zp {

cudaError_t launch_compress_d128(const CompressArgs &a, CompressShape shape, int mt, int units,
                                 cudaStream_t s)
{
    return launch_compress_for_d<128>(a, shape, mt, units, s);
}

bool compress_cluster16_ok()
{
    static int cached = -1;
    if (cached < 0)
        cached = cluster16_ok_t<128>() && cluster16_ok_t<64>() ? 1 : 0;
    return cached == 1;
}

}  // namespace zp
