// kvq_decode_i4g.cu -- decode kernel instantiations for INT4 per-group pools
// (kvq_decode_impl.cuh), one translation unit so they compile in parallel.
#include "kvq_decode_impl.cuh"
#include "kvq_internal.h"

namespace kvq {

cudaError_t launch_decode_int4_group(const DecodeLaunch& l) {
  const int D = l.p.pool.D, ng = l.p.pool.ng;
  if (D == 64) {
    switch (ng) {
      case 1: return run_decode<FMT_INT4_GROUP, 64, 1>(l);
      case 2: return run_decode<FMT_INT4_GROUP, 64, 2>(l);
      case 4: return run_decode<FMT_INT4_GROUP, 64, 4>(l);
    }
  } else if (D == 128) {
    switch (ng) {
      case 1: return run_decode<FMT_INT4_GROUP, 128, 1>(l);
      case 2: return run_decode<FMT_INT4_GROUP, 128, 2>(l);
      case 4: return run_decode<FMT_INT4_GROUP, 128, 4>(l);
      case 8: return run_decode<FMT_INT4_GROUP, 128, 8>(l);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
