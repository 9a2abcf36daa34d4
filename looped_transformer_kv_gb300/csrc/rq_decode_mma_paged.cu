// ResidualQuant decode attention: the paged-cache kernel variants (the kernel template is in
// rq_decode_mma.cuh; compiled apart from the contiguous variants so that both build in parallel).
#include "rq_decode_mma.cuh"

namespace rq {

KernelFn pick_paged(int D, bool res4, int nr, bool packed) {
  return packed ? pick_pg<true, true>(D, res4, nr) : pick_pg<true, false>(D, res4, nr);
}

}  // namespace rq
