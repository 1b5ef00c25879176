// Full-cache verification attention: the dense in-run baseline (the "Full
// Cache" bar of the "dustin-long-context" notes, section 3, Fig. 7).
#include "attn_host.cuh"

namespace dustin {

cudaError_t launch_attn_dense(const AttnArgs& a, int d, int mt, bool paged,
                              cudaStream_t st) {
  return AttnHost<true>::launch(a, d, mt, paged, st);
}

int occupancy_attn_dense(int d, int mt) {
  return AttnHost<true>::occupancy(d, mt);
}

cudaError_t take_attn_dense_flags(unsigned* flags) {
  return AttnHost<true>::take_flags(flags);
}

}  // namespace dustin
