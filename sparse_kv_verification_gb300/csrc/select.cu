// Hybrid combination and global per-sequence Top-K (the verification set
// I_verify of the "dustin-long-context" notes, sections 2.2 and 2.3):
// protected sink and recent positions, then the top of the hybrid score
// (alpha mode) or draft top-m followed by target top-(rest) (m mode).
//
// One CTA of 1024 threads per sequence.  Scores become order-preserving
// uint32 keys (NaN lowest, -0 folded onto +0), computed once into shared
// memory when the row fits (n <= 49152), else recomputed from global memory
// in every pass.  A three-pass radix select (11 + 11 + 10 bits, one shared
// histogram; lanes of a warp that hit the same bucket are merged with
// __match_any_sync so each distinct bucket costs one atomic, which matters
// because scores concentrate in few buckets; a block scan finds the bucket
// holding the r-th key from the top) fixes the threshold key T and how many
// keys equal to T to take; a marking pass over positions in ascending order
// takes every key > T and the lowest-position keys == T into a shared-memory
// bitmap.  A final ordered compaction writes the kept positions (protected
// or marked) in ascending order.
#include "device_common.cuh"
#include "internal.h"

namespace dustin {

namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN: below everything
  if (u == 0x80000000u) u = 0u;                      // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan of v over the block; *total receives the block sum.
__device__ int block_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int base = warp ? warp_sums[warp - 1] : 0;
  *total = warp_sums[31];
  __syncthreads();
  return base + x - v;
}

__device__ double block_sum_f64(double v, double* buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) buf[warp] = v;
  __syncthreads();
  double t = 0.0;
  if (warp == 0) {
    t = buf[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) buf[32] = t;
  }
  __syncthreads();
  t = buf[32];
  __syncthreads();
  return t;
}

struct Shared {
  int hist[2048];
  int warp_sums[32];
  int pick[2];
  double dbuf[33];
};

// Marks the top-r eligible positions by key (ties: lower position first).
template <class KeyF, class EligF>
__device__ void select_mark(int r, int n, KeyF key, EligF elig, uint32_t* bits,
                            Shared& sh) {
  if (r <= 0) return;
  uint32_t prefix = 0, mask = 0;
  int need = r;
  const int tid = threadIdx.x;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int i = tid; i < 2048; i += kThreads) sh.hist[i] = 0;
    __syncthreads();
    // n is padded to whole warps so that __match_any_sync sees full warps.
    const int n_pad = (n + 31) & ~31;
    for (int j = tid; j < n_pad; j += kThreads) {
      bool hit = false;
      uint32_t bin = 0;
      if (j < n && elig(j)) {
        const uint32_t kj = key(j);
        hit = (kj & mask) == prefix;
        bin = (kj >> shift) & (nb - 1);
      }
      const unsigned hits = __ballot_sync(0xffffffffu, hit);
      if (hits == 0u) continue;
      const unsigned same = __match_any_sync(0xffffffffu, hit ? bin : 0xffffffffu);
      const int lane = threadIdx.x & 31;
      if (hit && (__ffs(same) - 1) == lane) atomicAdd(&sh.hist[bin], __popc(same));
    }
    __syncthreads();
    // Thread u owns the bins nb-1-u*bpt-q (q < bpt), i.e. bins from the top.
    const int bpt = nb / kThreads;
    int cnt[2] = {0, 0};
    int sum = 0;
    for (int q = 0; q < bpt; ++q) {
      cnt[q] = sh.hist[nb - 1 - tid * bpt - q];
      sum += cnt[q];
    }
    int total;
    int acc = block_scan(sum, sh.warp_sums, &total);
    for (int q = 0; q < bpt; ++q) {
      if (acc < need && need <= acc + cnt[q]) {
        sh.pick[0] = nb - 1 - tid * bpt - q;
        sh.pick[1] = acc;
      }
      acc += cnt[q];
    }
    __syncthreads();
    prefix |= (uint32_t)sh.pick[0] << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    need -= sh.pick[1];
    __syncthreads();
  }
  // Take keys > T, and the first `need` keys == T in position order.
  const uint32_t T = prefix;
  int eq_before = 0;
#pragma unroll 1
  for (int base = 0; base < n; base += kThreads) {
    const int j = base + tid;
    const bool e = j < n && elig(j);
    const uint32_t kj = e ? key(j) : 0u;
    const bool gt = e && kj > T;
    const bool eq = e && kj == T;
    int tot;
    const int rank = block_scan(eq ? 1 : 0, sh.warp_sums, &tot);
    if (gt || (eq && eq_before + rank < need)) atomicOr(&bits[j >> 5], 1u << (j & 31));
    eq_before += tot;
  }
  __syncthreads();
}

constexpr int kSmemKeysMaxN = 49152;

template <bool SMEM_KEYS>
__global__ void __launch_bounds__(kThreads) select_kernel(const SelectArgs a) {
  extern __shared__ uint32_t bits[];
  __shared__ Shared sh;
  uint32_t* skeys = bits + ((a.n + 31) / 32);   // only with SMEM_KEYS
  const int tid = threadIdx.x;
  const int n = a.n, k = a.k;
  int32_t* out = a.idx + (long long)blockIdx.x * min(k, n);
  const float* sd = a.sd ? a.sd + (long long)blockIdx.x * n : nullptr;
  const float* st = a.st ? a.st + (long long)blockIdx.x * n : nullptr;
  griddep_wait();
  griddep_launch_dependents();
  if (k >= n) {
    for (int j = tid; j < n; j += kThreads) out[j] = j;
    return;
  }
  const int ns = min(max(a.n_sink, 0), n);
  const int hi = n - min(max(a.n_recent, 0), n);
  auto forced = [&](int j) { return j < ns || j >= hi; };
  const int n_forced = hi <= ns ? n : ns + (n - hi);
  const int budget = k - n_forced;  // >= 0, checked on the host
  for (int i = tid; i < (n + 31) / 32; i += kThreads) bits[i] = 0u;
  __syncthreads();

  auto not_forced = [&](int j) { return !forced(j); };
  if (a.m < 0) {
    const bool hasD = sd != nullptr && a.alpha != 0.0;
    const bool hasT = st != nullptr && (1.0 - a.alpha) != 0.0;
    double cd = a.alpha, ct = 1.0 - a.alpha;
    if (a.norm == 1) {
      if (hasD) {
        double s = 0.0;
        for (int j = tid; j < n; j += kThreads) s += (double)sd[j];
        s = block_sum_f64(s, sh.dbuf);
        if (s > 0.0 && isfinite(s)) cd = cd / s;
      }
      if (hasT) {
        double s = 0.0;
        for (int j = tid; j < n; j += kThreads) s += (double)st[j];
        s = block_sum_f64(s, sh.dbuf);
        if (s > 0.0 && isfinite(s)) ct = ct / s;
      }
    }
    const float fd = (float)cd, ft = (float)ct;
    auto mix = [&](int j) -> uint32_t {
      float c;
      if (hasD && hasT)
        c = __fadd_rn(__fmul_rn(fd, sd[j]), __fmul_rn(ft, st[j]));
      else if (hasD)
        c = __fmul_rn(fd, sd[j]);
      else if (hasT)
        c = __fmul_rn(ft, st[j]);
      else
        c = 0.f;
      return order_key(c);
    };
    if constexpr (SMEM_KEYS) {
      for (int j = tid; j < n; j += kThreads) skeys[j] = mix(j);
      __syncthreads();
      auto cached = [&](int j) { return skeys[j]; };
      select_mark(budget, n, cached, not_forced, bits, sh);
    } else {
      select_mark(budget, n, mix, not_forced, bits, sh);
    }
  } else {
    const int m_eff = min(a.m, budget);
    auto free_pos = [&](int j) {
      return !forced(j) && !((bits[j >> 5] >> (j & 31)) & 1u);
    };
    if constexpr (SMEM_KEYS) {
      auto cached = [&](int j) { return skeys[j]; };
      if (m_eff > 0) {
        for (int j = tid; j < n; j += kThreads) skeys[j] = order_key(sd[j]);
        __syncthreads();
        select_mark(m_eff, n, cached, not_forced, bits, sh);
      }
      if (budget - m_eff > 0) {
        for (int j = tid; j < n; j += kThreads) skeys[j] = order_key(st[j]);
        __syncthreads();
        select_mark(budget - m_eff, n, cached, free_pos, bits, sh);
      }
    } else {
      if (m_eff > 0) {
        auto kd = [&](int j) { return order_key(sd[j]); };
        select_mark(m_eff, n, kd, not_forced, bits, sh);
      }
      if (budget - m_eff > 0) {
        auto kt = [&](int j) { return order_key(st[j]); };
        select_mark(budget - m_eff, n, kt, free_pos, bits, sh);
      }
    }
  }

  // Ordered compaction of protected + marked positions.
  int written = 0;
#pragma unroll 1
  for (int base = 0; base < n; base += kThreads) {
    const int j = base + tid;
    const bool keep = j < n && (forced(j) || ((bits[j >> 5] >> (j & 31)) & 1u));
    int tot;
    const int pos = block_scan(keep ? 1 : 0, sh.warp_sums, &tot);
    if (keep && written + pos < k) out[written + pos] = j;
    written += tot;
  }
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st) {
  const int words = (a.n + 31) / 32;
  const bool cache = a.n <= kSmemKeysMaxN && a.k < a.n;
  const int smem = words * 4 + (cache ? a.n * 4 : 0);
  auto kern = cache ? select_kernel<true> : select_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(a.b), dim3(kThreads), smem, st, a);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace dustin
