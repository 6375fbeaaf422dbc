// bkv_ragged_tc.cu -- tensor-core prefill kernel of the mixed-step attention
// (placeholder until the tcgen05 kernel lands: no shape is taken yet).
#include "bkv_ragged.cuh"

namespace bkv {

bool prepare_ragged_tc(const RaggedArgs &, RaggedTc *) { return false; }

int launch_ragged_tc(const RaggedArgs &, const RaggedTc &, cudaStream_t) { return BKV_ERR_UNSUPPORTED; }

}  // namespace bkv
