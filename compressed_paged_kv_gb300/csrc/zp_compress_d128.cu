// zp_compress_d128.cu -- the fused compression kernels for head dim 128.
#include "zp_compress_stream.cuh"

namespace zp {

cudaError_t launch_compress_d128(const CompressArgs &a, int mt, int units, cudaStream_t s)
{
    return launch_stream_for_d<128>(a, mt, units, s);
}

}  // namespace zp
