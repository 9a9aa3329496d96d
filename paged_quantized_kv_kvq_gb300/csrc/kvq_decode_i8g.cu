// INT8 per-group instantiations of the paged decode kernel (see
// kvq_decode_impl.cuh).  NG = head_dim / group scale groups per head.
#include "kvq_decode_impl.cuh"
#include "kvq_internal.h"

namespace kvq {

cudaError_t launch_decode_int8_group(const DecodeLaunch& l) {
  const int D = l.p.pool.D, ng = l.p.pool.ng;
  if (D == 64) {
    switch (ng) {
      case 1: return run_decode<FMT_INT8_GROUP, 64, 1>(l);
      case 2: return run_decode<FMT_INT8_GROUP, 64, 2>(l);
      case 4: return run_decode<FMT_INT8_GROUP, 64, 4>(l);
    }
  } else if (D == 128) {
    switch (ng) {
      case 1: return run_decode<FMT_INT8_GROUP, 128, 1>(l);
      case 2: return run_decode<FMT_INT8_GROUP, 128, 2>(l);
      case 4: return run_decode<FMT_INT8_GROUP, 128, 4>(l);
      case 8: return run_decode<FMT_INT8_GROUP, 128, 8>(l);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
