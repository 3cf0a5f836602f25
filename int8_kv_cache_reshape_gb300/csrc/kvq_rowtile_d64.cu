// kvq_rowtile_d64.cu -- row-tile attention kernels for head_dim 64 (one
// translation unit per head_dim keeps the build parallel).
#include "kvq_rowtile.cuh"

namespace kvq {
int launch_rowtile_d64(const AttnParams& p, int dtype, int ntiles, int64_t item_offset,
                      int64_t num_items, void* stream) {
  return launch_rowtile_d<64>(p, dtype, ntiles, item_offset, num_items,
                             static_cast<cudaStream_t>(stream));
}
}  // namespace kvq
