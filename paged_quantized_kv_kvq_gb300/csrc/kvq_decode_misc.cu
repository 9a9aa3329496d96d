// FP16, per-token (INT8 / FP8 e4m3) and per-channel INT8 instantiations of the
// paged decode kernel (see kvq_decode_impl.cuh).
#include "kvq_decode_impl.cuh"
#include "kvq_internal.h"

namespace kvq {

cudaError_t launch_decode_fp16(const DecodeLaunch& l) { return run_decode_d<FMT_FP16>(l); }

cudaError_t launch_decode_token(const DecodeLaunch& l) {
  return l.p.pool.fmt == FMT_FP8_TOKEN ? run_decode_d<FMT_FP8_TOKEN>(l)
                                       : run_decode_d<FMT_INT8_TOKEN>(l);
}

cudaError_t launch_decode_channel(const DecodeLaunch& l) { return run_decode_d<FMT_INT8_CHANNEL>(l); }

cudaError_t launch_decode_e5m2(const DecodeLaunch& l) { return run_decode_d<FMT_FP8_E5M2>(l); }

}  // namespace kvq
