// Full-cache verification attention: the dense in-run baseline (the "Full
// Cache" bar of the "dustin-long-context" notes, section 3, Fig. 7), on the
// stream-K kernel of attn_streamk.cuh.
#include "attn_streamk.cuh"
#include "internal.h"

namespace dustin {
namespace {

template <int D, int MT, bool PAGED, bool WIN>
cudaError_t prepare() {
  using C = SkCfg<D, MT>;
  static std::atomic<uint64_t> done{0};
  if constexpr (C::REBALANCE) {
    static std::atomic<int> checked{0};
    cudaError_t e = check_register_split<C>(verify_attn_sk_kernel<D, MT, PAGED, WIN>, checked);
    if (e != cudaSuccess) return e;
  }
  return ensure_smem_attr(verify_attn_sk_kernel<D, MT, PAGED, WIN>, C::SMEM, done);
}

template <int D, int MT, bool PAGED, bool WIN>
cudaError_t run(const AttnSkArgs& a, cudaStream_t st) {
  using C = SkCfg<D, MT>;
  cudaError_t e = prepare<D, MT, PAGED, WIN>();
  if (e != cudaSuccess) return e;
  e = launch_pdl(verify_attn_sk_kernel<D, MT, PAGED, WIN>, dim3((unsigned)a.grid),
                 dim3(C::NT), C::SMEM, st, a);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

template <int D, bool PAGED, bool WIN>
cudaError_t by_mt(const AttnSkArgs& a, int mt, cudaStream_t st) {
  switch (mt) {
    case 1: return run<D, 1, PAGED, WIN>(a, st);
    case 2: return run<D, 2, PAGED, WIN>(a, st);
    case 3: return run<D, 3, PAGED, WIN>(a, st);
    default: return run<D, 4, PAGED, WIN>(a, st);
  }
}

template <int D, bool PAGED>
cudaError_t by_win(const AttnSkArgs& a, int mt, cudaStream_t st) {
  return a.has_win ? by_mt<D, PAGED, true>(a, mt, st) : by_mt<D, PAGED, false>(a, mt, st);
}

template <int D, int MT>
int occ() {
  if (prepare<D, MT, false, false>() != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, verify_attn_sk_kernel<D, MT, false, false>, SkCfg<D, MT>::NT,
          SkCfg<D, MT>::SMEM) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

}  // namespace

cudaError_t launch_attn_dense(const AttnSkArgs& a, int d, int mt, bool paged,
                              cudaStream_t st) {
  if (d == 64) return paged ? by_win<64, true>(a, mt, st) : by_win<64, false>(a, mt, st);
  return paged ? by_win<128, true>(a, mt, st) : by_win<128, false>(a, mt, st);
}

int occupancy_attn_dense(int d, int mt) {
  if (d == 64) {
    switch (mt) {
      case 1: return occ<64, 1>();
      case 2: return occ<64, 2>();
      case 3: return occ<64, 3>();
      default: return occ<64, 4>();
    }
  }
  switch (mt) {
    case 1: return occ<128, 1>();
    case 2: return occ<128, 2>();
    case 3: return occ<128, 3>();
    default: return occ<128, 4>();
  }
}

cudaError_t take_attn_dense_flags(unsigned* flags) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_sk_dev_flags, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_attn_sk_dev_flags, &zero, sizeof(zero));
  *flags |= v;
  return e;
}

}  // namespace dustin
