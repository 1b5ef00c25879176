// Host-side launch of the sparse verification-attention kernel and its
// split combine (attn.cuh).
#pragma once

#include <atomic>

#include "attn.cuh"
#include "internal.h"

namespace dustin {

struct AttnHost {
  template <int D, int MT, bool PAGED, bool WIN, bool WIDE>
  static cudaError_t prepare() {
    using C = AttnCfg<D, MT>;
    static std::atomic<uint64_t> done{0};
    if constexpr (C::REBALANCE) {
      static std::atomic<int> checked{0};
      cudaError_t e = check_register_split<C>(verify_attn_kernel<D, MT, PAGED, WIN, WIDE>, checked);
      if (e != cudaSuccess) return e;
    }
    return ensure_smem_attr(verify_attn_kernel<D, MT, PAGED, WIN, WIDE>, C::SMEM, done);
  }

  template <int D, int MT, bool PAGED, bool WIN, bool WIDE>
  static cudaError_t run(const AttnArgs& a, cudaStream_t st) {
    using C = AttnCfg<D, MT>;
    cudaError_t e = prepare<D, MT, PAGED, WIN, WIDE>();
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)a.b * a.hkv * a.row_blocks;
    e = launch_pdl(verify_attn_kernel<D, MT, PAGED, WIN, WIDE>,
                   dim3((unsigned)(blocks * a.splits)), dim3(C::NT), C::SMEM, st, a);
    if (e != cudaSuccess) return e;
    note_launches(1);
    if (a.splits > 1) {
      const long long warps = blocks * C::ROWS;
      e = launch_pdl(attn_combine_kernel<D, MT>, dim3((unsigned)((warps + 7) / 8)),
                     dim3(256), 0, st, a);
      if (e != cudaSuccess) return e;
      note_launches(1);
    }
    return cudaSuccess;
  }

  template <int D, bool PAGED, bool WIN, bool WIDE>
  static cudaError_t by_mt(const AttnArgs& a, int mt, cudaStream_t st) {
    switch (mt) {
      case 1: return run<D, 1, PAGED, WIN, WIDE>(a, st);
      case 2: return run<D, 2, PAGED, WIN, WIDE>(a, st);
      case 3: return run<D, 3, PAGED, WIN, WIDE>(a, st);
      default: return run<D, 4, PAGED, WIN, WIDE>(a, st);
    }
  }

  // The window variant always uses the 64-bit table (the host splits).
  template <int D, bool PAGED>
  static cudaError_t by_win(const AttnArgs& a, int mt, cudaStream_t st) {
    if (a.has_win) return by_mt<D, PAGED, true, false>(a, mt, st);
    return a.wide ? by_mt<D, PAGED, false, true>(a, mt, st)
                  : by_mt<D, PAGED, false, false>(a, mt, st);
  }

  static cudaError_t launch(const AttnArgs& a, int d, int mt, bool paged,
                            cudaStream_t st) {
    if (d == 64) return paged ? by_win<64, true>(a, mt, st) : by_win<64, false>(a, mt, st);
    return paged ? by_win<128, true>(a, mt, st) : by_win<128, false>(a, mt, st);
  }

  template <int D, int MT>
  static int occ() {
    if (prepare<D, MT, false, false, false>() != cudaSuccess) return 1;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, verify_attn_kernel<D, MT, false, false, false>, AttnCfg<D, MT>::NT,
            AttnCfg<D, MT>::SMEM) != cudaSuccess)
      return 1;
    return n > 0 ? n : 1;
  }

  static int occupancy(int d, int mt) {
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

  static cudaError_t take_flags(unsigned* flags) {
    unsigned v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_attn_dev_flags, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_attn_dev_flags, &zero, sizeof(zero));
    *flags |= v;
    return e;
  }
};

}  // namespace dustin
