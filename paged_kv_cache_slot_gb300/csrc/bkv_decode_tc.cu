// bkv_decode_tc.cu -- tensor-core (tcgen05) partition kernel for the paged
// decode.  Placeholder until the kernel lands: reports every shape as
// unsupported so the generic kernel runs.
#include "bkv_decode.cuh"

namespace bkv {

bool decode_tc_supported(const DecodeArgs &) { return false; }

int launch_decode_tc(const DecodeArgs &, cudaStream_t) { return BKV_ERR_UNSUPPORTED; }

}  // namespace bkv
