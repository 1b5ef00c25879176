// Sparse verification attention: K/V rows gathered by the index set
// (Stage 2 of the "dustin-long-context" notes, section 2.2 / Fig. 5).
#include "attn_host.cuh"

namespace dustin {

cudaError_t launch_attn_sparse(const AttnArgs& a, int d, int mt, bool paged,
                               cudaStream_t st) {
  return AttnHost::launch(a, d, mt, paged, st);
}

int occupancy_attn_sparse(int d, int mt) { return AttnHost::occupancy(d, mt); }

cudaError_t take_attn_sparse_flags(unsigned* flags) {
  return AttnHost::take_flags(flags);
}

}  // namespace dustin
