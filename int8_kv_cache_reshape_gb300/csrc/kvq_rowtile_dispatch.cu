// kvq_rowtile_dispatch.cu -- head_dim dispatch of the row-tile attention
// kernels (one translation unit per head_dim holds the instances).
#include "kvq_internal.h"

namespace kvq {

int launch_rowtile_d64(const AttnParams&, int, int, int64_t, int64_t, void*);
int launch_rowtile_d128(const AttnParams&, int, int, int64_t, int64_t, void*);
int launch_rowtile_d256(const AttnParams&, int, int, int64_t, int64_t, void*);

int launch_rowtile(const AttnParams& p, int dtype, int head_dim, int ntiles,
                   int64_t item_offset, int64_t num_items, void* stream) {
  if (num_items <= 0) return KVQ_OK;
  switch (head_dim) {
    case 64: return launch_rowtile_d64(p, dtype, ntiles, item_offset, num_items, stream);
    case 128: return launch_rowtile_d128(p, dtype, ntiles, item_offset, num_items, stream);
    case 256: return launch_rowtile_d256(p, dtype, ntiles, item_offset, num_items, stream);
    default: return KVQ_E_UNSUPPORTED;
  }
}

}  // namespace kvq
