// kvq_decode_dispatch.cu -- head_dim dispatch of the split-KV decode and the
// tensor-core prefill kernels (one translation unit per head_dim holds the
// instances).
#include "kvq_internal.h"

namespace kvq {

int launch_decode_d64(const AttnParams&, int, int, void*);
int launch_decode_d128(const AttnParams&, int, int, void*);
int launch_decode_d256(const AttnParams&, int, int, void*);
int launch_prefill_d64(const AttnParams&, const PrefillMaps&, int, int64_t, void*);
int launch_prefill_d128(const AttnParams&, const PrefillMaps&, int, int64_t, void*);
int launch_prefill_d256(const AttnParams&, const PrefillMaps&, int, int64_t, void*);

int launch_decode(const AttnParams& p, int dtype, int head_dim, int ntiles, void* stream) {
  if (p.num_chunks <= 0) return KVQ_OK;
  switch (head_dim) {
    case 64: return launch_decode_d64(p, dtype, ntiles, stream);
    case 128: return launch_decode_d128(p, dtype, ntiles, stream);
    case 256: return launch_decode_d256(p, dtype, ntiles, stream);
    default: return KVQ_E_UNSUPPORTED;
  }
}

int launch_prefill(const AttnParams& p, const PrefillMaps& maps, int dtype, int head_dim,
                   int64_t num_tiles, void* stream) {
  if (num_tiles <= 0) return KVQ_OK;
  switch (head_dim) {
    case 64: return launch_prefill_d64(p, maps, dtype, num_tiles, stream);
    case 128: return launch_prefill_d128(p, maps, dtype, num_tiles, stream);
    case 256: return launch_prefill_d256(p, maps, dtype, num_tiles, stream);
    default: return KVQ_E_UNSUPPORTED;
  }
}

}  // namespace kvq
