#include "mla_device.cuh"
#include "mla_launch.h"
namespace mla {
int launch_pair(int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, int,
                cudaStream_t) {
  return MLA_ERR_UNSUPPORTED;
}
}  // namespace mla
