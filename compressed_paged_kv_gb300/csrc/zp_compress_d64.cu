// zp_compress_d64.cu -- the fused compression kernels for head dim 64.
#include "zp_compress_stream.cuh"

namespace zp {

cudaError_t launch_compress_d64(const CompressArgs &a, int mt, int units, cudaStream_t s)
{
    return launch_stream_for_d<64>(a, mt, units, s);
}

}  // namespace zp
