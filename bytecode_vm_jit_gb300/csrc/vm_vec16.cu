// vm_vec16.cu — the VEC interpreter instantiated for 16 elements per lane
// (one warp moves 512 bytes of the narrowest dtype of a launch).
#include "vm_vec.cuh"

namespace dvm {
template cudaError_t launch_vec<16>(const LaunchParams&, int, size_t, bool, cudaStream_t);
}  // namespace dvm
