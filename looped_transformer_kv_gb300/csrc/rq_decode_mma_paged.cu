// ResidualQuant decode attention: the paged-cache kernel variants (the kernel template is in
// rq_decode_mma.cuh; compiled apart from the contiguous variants so that both build in parallel).
#include "rq_decode_mma.cuh"

namespace rq {

KernelFn pick_paged(int D, bool res4, int nr, int pk) {
  if (pk == 2) return pick_pg<true, 2>(D, res4, nr);
  return pk == 1 ? pick_pg<true, 1>(D, res4, nr) : pick_pg<true, 0>(D, res4, nr);
}

}  // namespace rq
