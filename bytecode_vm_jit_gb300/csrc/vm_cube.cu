// vm_cube.cu — placeholder until the CUBE (tcgen05) interpreter lands.
#include "dvm_internal.h"
#include <cstdio>
namespace dvm {
int cube_launch(DeviceState*, const uint8_t*, size_t, void* const*, int, void*, char* msg, size_t cap) {
  std::snprintf(msg, cap, "the CUBE kernel type is not built yet");
  return -2;
}
}  // namespace dvm
