// Sparse verification attention of many layers in one persistent launch
// (attn_multilayer.cuh).
#include "attn_multilayer.cuh"
#include "internal.h"

namespace dustin {
namespace {

template <int D, int MT, bool PAGED>
cudaError_t prepare() {
  using C = SkCfg<D, MT>;
  static std::atomic<uint64_t> done{0};
  if constexpr (C::REBALANCE) {
    static std::atomic<int> checked{0};
    cudaError_t e = check_register_split<C>(verify_attn_ml_kernel<D, MT, PAGED>, checked);
    if (e != cudaSuccess) return e;
  }
  return ensure_smem_attr(verify_attn_ml_kernel<D, MT, PAGED>, C::SMEM, done);
}

template <int D, int MT, bool PAGED>
cudaError_t run(const AttnMlArgs& a, int grid, cudaStream_t st) {
  using C = SkCfg<D, MT>;
  cudaError_t e = prepare<D, MT, PAGED>();
  if (e != cudaSuccess) return e;
  e = launch_pdl(verify_attn_ml_kernel<D, MT, PAGED>, dim3((unsigned)grid),
                 dim3(C::NT), C::SMEM, st, a);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

template <int D, bool PAGED>
cudaError_t by_mt(const AttnMlArgs& a, int mt, int grid, cudaStream_t st) {
  switch (mt) {
    case 1: return run<D, 1, PAGED>(a, grid, st);
    case 2: return run<D, 2, PAGED>(a, grid, st);
    case 3: return run<D, 3, PAGED>(a, grid, st);
    default: return run<D, 4, PAGED>(a, grid, st);
  }
}

}  // namespace

cudaError_t launch_attn_ml(const AttnMlArgs& a, int d, int mt, bool paged, int grid,
                           cudaStream_t st) {
  if (d == 64) return paged ? by_mt<64, true>(a, mt, grid, st) : by_mt<64, false>(a, mt, grid, st);
  return paged ? by_mt<128, true>(a, mt, grid, st) : by_mt<128, false>(a, mt, grid, st);
}

cudaError_t take_attn_ml_flags(unsigned* flags) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_ml_dev_flags, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_attn_ml_dev_flags, &zero, sizeof(zero));
  *flags |= v;
  return e;
}

}  // namespace dustin
