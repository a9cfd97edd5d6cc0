// Kernel variants of the tensor-core conv3d with the IG3_EPI_TANH_MISH epilogue (one
// translation unit per epilogue so the variants compile in parallel).
#include "conv3d_tc_kernel.cuh"

namespace ig3 {
namespace tc {
template int launch_kernel<IG3_EPI_TANH_MISH>(const TcParams&, size_t, int, cudaStream_t);
}  // namespace tc
}  // namespace ig3
