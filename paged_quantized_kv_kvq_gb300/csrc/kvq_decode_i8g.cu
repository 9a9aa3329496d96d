// INT8 per-group instantiations of the paged decode kernel (see
// kvq_decode_impl.cuh).  NG = head_dim / group scale groups per head.
#include "kvq_decode_impl.cuh"
#include "kvq_internal.h"

namespace kvq {

cudaError_t launch_decode_int8_group(const DecodeLaunch& l) {
  return run_decode_group<FMT_INT8_GROUP>(l);
}

}  // namespace kvq
