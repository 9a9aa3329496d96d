// Block size 8 instantiations of the paged decode kernel, INT8 per-group (see
// kvq_decode_impl.cuh: each 16-token tile is made of two 8-token pages).
#include "kvq_decode_impl.cuh"
#include "kvq_internal.h"

namespace kvq {

cudaError_t launch_decode_bs8_group(const DecodeLaunch& l) {
  return run_decode_group<FMT_INT8_GROUP, true>(l);
}

}  // namespace kvq
