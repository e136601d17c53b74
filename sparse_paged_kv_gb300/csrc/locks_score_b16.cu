// The locks_select score kernel for page size B = 16 (its own translation
// unit, so the two page sizes compile in parallel).
#include "locks_score.cuh"

namespace locks {

int launch_score_b16(const SelectParams& p, int G, int RP, int dtype, int n_ctas,
                     cudaStream_t stream) {
  return launch_score_pb<16>(p, G, RP, dtype, n_ctas, stream);
}

}  // namespace locks
