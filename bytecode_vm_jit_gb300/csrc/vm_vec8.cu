// vm_vec8.cu — the VEC interpreter instantiated for 8 elements per lane
// (one warp moves 512 bytes of the narrowest dtype of a launch).
#include "vm_vec.cuh"

namespace dvm {
template cudaError_t launch_vec<8>(const LaunchParams&, int, size_t, bool, cudaStream_t);
}  // namespace dvm
