// Block size 8 instantiations of the paged decode kernel: FP16, per-token
// INT8 / FP8 e4m3, per-channel INT8 and FP8 e5m2 (see kvq_decode_impl.cuh).
#include "kvq_decode_impl.cuh"
#include "kvq_internal.h"

namespace kvq {

cudaError_t launch_decode_bs8_misc(const DecodeLaunch& l) {
  switch (l.p.pool.fmt) {
    case FMT_FP16: return run_decode_d<FMT_FP16, true>(l);
    case FMT_INT8_TOKEN: return run_decode_d<FMT_INT8_TOKEN, true>(l);
    case FMT_FP8_TOKEN: return run_decode_d<FMT_FP8_TOKEN, true>(l);
    case FMT_INT8_CHANNEL: return run_decode_d<FMT_INT8_CHANNEL, true>(l);
    case FMT_FP8_E5M2: return run_decode_d<FMT_FP8_E5M2, true>(l);
  }
  return cudaErrorInvalidValue;  // INT4 packs tokens t and t+8 in one word: no 8-token pages
}

}  // namespace kvq
