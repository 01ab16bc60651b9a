// gla_tc.cu — tensor-core (tcgen05 / TMEM / TMA) chunked Simple GLA forward.
#include "gla_common.cuh"

GLA_DEFINE_STATUS(tc)

namespace gla {

bool tc_chunk_supported(int, int, int) { return false; }

int tc_chunk_fwd_bf16(const void *, const void *, const void *, const float *, const float *, void *, float *,
                      int, int, int, int, int, const int32_t *, cudaStream_t) {
    return GLA_ERR_UNSUPPORTED;
}

}  // namespace gla
