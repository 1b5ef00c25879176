// Hybrid combination and global per-sequence Top-K (the verification set
// I_verify of the "dustin-long-context" notes, sections 2.2 and 2.3):
// protected sink and recent positions, then the top of the hybrid score
// (alpha mode) or draft top-m followed by target top-(rest) (m mode).
//
// One thread-block cluster of C <= 8 CTAs (1024 threads each) per sequence;
// CTA r owns the positions [r seg, r seg + seg), seg a multiple of 32, so a
// 32k-position row keeps 8 SMs busy instead of one.  Many short rows take
// one 256-thread CTA each instead (the same code, fewer threads).  Cluster-wide values
// pass through distributed shared memory: the CTAs publish partial results
// in their own shared memory, barrier.cluster, then every CTA reads all the
// partials in the same rank order, so every CTA derives the same values.
//
//  * alpha mode with L1 normalisation: the sums of S_D and S_T, per thread
//    and per CTA as float-float pairs (TwoSum: about 44 significant bits;
//    fp64 arithmetic is slow on this GPU), per cluster in fp64 in rank
//    order; one thread forms the mixing coefficients in fp64 and rounds them
//    to fp32, and c = fl32(fl32(a_D S_D) + fl32(a_T S_T)).  (A partial sum
//    past the fp32 range reads as infinite and leaves its vector unscaled.)
//  * Scores become order-preserving uint32 keys (NaN lowest, -0 folded onto
//    +0), cached in shared memory when the segment fits (the raw scores are
//    staged there during the one read of global memory).
//  * A three-pass radix select (11 + 11 + 10 bits) finds the threshold key
//    T and how many keys equal to T to take: each CTA builds the histogram
//    of its segment with one shared-memory atomic per key (each group of 8
//    warps has its own copy; measured here, this beats merging equal
//    buckets first with __match_any_sync or a warp sort, 1.3 against 5-6 us
//    for a pass over 8192 keys that concentrate in few buckets),
//    the copies are folded, the CTAs sum the cluster's folded histograms bin
//    by bin, and a block scan finds the bucket holding the r-th key from the
//    top.  Two folded buffers alternate, so one cluster barrier per pass
//    suffices.
//  * Marking: keys > T are taken, and keys == T in ascending position order
//    until the count is met.  Each warp owns a 32-aligned run of positions
//    and walks it 32 at a time, so a step covers one word of the bitmap of
//    marks; the rank of an equal key is its CTA's offset (published counts
//    of the lower ranks) + its warp's offset (one scan of the warp counts)
//    + the count in earlier steps and lower lanes.
//  * Compaction: protected or marked positions are written in ascending
//    order the same way (CTA offset + warp offset + running count).
// A final cluster barrier keeps every CTA's shared memory alive until the
// others have read it.
#include <cooperative_groups.h>

#include "device_common.cuh"
#include "internal.h"

namespace dustin {

namespace {

namespace cg = cooperative_groups;

// Threads per CTA: 1024 for the cluster kernel of long rows; 256 for many
// short rows (one CTA each, several CTAs per SM).
constexpr int kThreads = 1024;
constexpr int kThreadsShort = 256;
constexpr int kShortRowsMinRows = 304;   // two 1024-thread CTAs on each of 152 SMs
constexpr int kMaxWarps = kThreads / 32;
// Build-time tunable: the largest cluster (CTAs per sequence).
#ifndef DUSTIN_SELECT_CLUSTER
#define DUSTIN_SELECT_CLUSTER 8
#endif
constexpr int kMaxCluster = DUSTIN_SELECT_CLUSTER;
constexpr int kSegPerCta = 4096;          // positions per CTA that call for
                                          // another CTA in the cluster
constexpr int kSmemKeysMaxSeg = 20480;    // cached keys + raw S_T per CTA (160 KB)

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN: below everything
  if (u == 0x80000000u) u = 0u;                      // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sub-histograms of a CTA (8 warps each).
__host__ __device__ constexpr int hist_copies(int threads) {
  return threads >= 1024 ? 4 : 1;
}

struct Shared {
  int warp_vals[kMaxWarps];
  float coef[2];          // fp32 mixing coefficients (alpha mode)
  int pick[3];            // bucket, keys above it, keys in it
  int xchg[4];            // counts this CTA publishes to its cluster
  double dpart[2];        // this CTA's L1 partial sums (draft, target)
  float4 fbuf[kMaxWarps + 1];
};

// Exclusive scan of v over the block of WARPS warps; *total receives the
// block sum.
template <int WARPS>
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
    int w = lane < WARPS ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < WARPS) warp_sums[lane] = w;
  }
  __syncthreads();
  const int base = warp ? warp_sums[warp - 1] : 0;
  *total = warp_sums[WARPS - 1];
  __syncthreads();
  return base + x - v;
}

// Scan of one warp-uniform count per warp: (exclusive prefix of this warp,
// block total).  Every warp scans the 32 counts itself.
template <int WARPS>
__device__ int2 scan_warp_counts(int c, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();                 // the previous scan's reads are done
  if (lane == 0) sh.warp_vals[warp] = c;
  __syncthreads();
  const int v = lane < WARPS ? sh.warp_vals[lane] : 0;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  const int excl = __shfl_sync(0xffffffffu, x - v, warp);
  const int total = __shfl_sync(0xffffffffu, x, 31);
  return make_int2(excl, total);
}

// hi + lo += x exactly (Knuth's TwoSum: the rounding error of hi + x goes
// to lo).  Per-thread partial sums run in this float-float form and only
// the per-thread totals in fp64, which is slow on this GPU.
__device__ __forceinline__ void two_sum_acc(float2& acc, float x) {
  const float s = __fadd_rn(acc.x, x);
  const float bp = __fsub_rn(s, acc.x);
  const float err = __fadd_rn(__fsub_rn(acc.x, __fsub_rn(s, bp)), __fsub_rn(x, bp));
  acc.x = s;
  acc.y = __fadd_rn(acc.y, err);
}

// (a.x + a.y) + (b.x + b.y) as a float-float pair.
__device__ __forceinline__ float2 ff_add(float2 a, float2 b) {
  float2 r = a;
  two_sum_acc(r, b.x);
  r.y = __fadd_rn(r.y, b.y);
  return r;
}

// Block sum of two float-float values, returned to every thread.
template <int WARPS>
__device__ float4 block_sum_ff2(float2 d, float2 t, float4* buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    d = ff_add(d, make_float2(__shfl_xor_sync(0xffffffffu, d.x, o),
                              __shfl_xor_sync(0xffffffffu, d.y, o)));
    t = ff_add(t, make_float2(__shfl_xor_sync(0xffffffffu, t.x, o),
                              __shfl_xor_sync(0xffffffffu, t.y, o)));
  }
  if (lane == 0) buf[warp] = make_float4(d.x, d.y, t.x, t.y);
  __syncthreads();
  if (warp == 0) {
    const float4 v = lane < WARPS ? buf[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    d = make_float2(v.x, v.y);
    t = make_float2(v.z, v.w);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      d = ff_add(d, make_float2(__shfl_xor_sync(0xffffffffu, d.x, o),
                                __shfl_xor_sync(0xffffffffu, d.y, o)));
      t = ff_add(t, make_float2(__shfl_xor_sync(0xffffffffu, t.x, o),
                                __shfl_xor_sync(0xffffffffu, t.y, o)));
    }
    if (lane == 0) buf[WARPS] = make_float4(d.x, d.y, t.x, t.y);
  }
  __syncthreads();
  const float4 r = buf[WARPS];
  __syncthreads();
  return r;
}

// Sum of slot `slot` of xchg over the cluster ranks below `rank` (every lane
// of the calling warp gets it).
__device__ int lower_ranks_sum(cg::cluster_group& cl, Shared& sh, int slot,
                               int rank) {
  const int lane = threadIdx.x & 31;
  int v = 0;
  if (lane < rank) v = cl.map_shared_rank(sh.xchg, lane)[slot];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// This CTA's positions, and the run of them that warp w walks.
struct Seg {
  int lo, len;   // [lo, lo + len)
  int cw;        // positions per warp (multiple of 32)
};

// Marks the top-r eligible positions of the sequence by key (ties: lower
// position first) in `bits` (this CTA's segment).  Called by every CTA of
// the cluster with the same r; xslot is this call's exchange slot (the
// m-split makes two calls, draft quota then target).
template <int THREADS, class KeyF, class EligF>
__device__ void select_mark(cg::cluster_group& cl, int rank, int C, int r,
                            const Seg& sg, KeyF key, EligF elig,
                            uint32_t* bits, int* fold, int* copies, Shared& sh,
                            int xslot) {
  if (r <= 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, mask = 0;
  int need = r;
  // Set when the bucket holding the r-th key holds exactly the keys still
  // needed: every key whose top bits match is taken, whatever its lower
  // bits, so the remaining passes and the ranking of equal keys are
  // skipped (the same set: the order among them no longer matters).
  bool whole = false;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    // Each group of 8 warps counts into its own copy of the histogram (fewer
    // atomics on the few hot buckets), the copies are folded into one of two
    // alternating buffers, and the cluster reads the folded ones.
    constexpr int HC = hist_copies(THREADS);
    int* h = fold + (pass & 1) * 2048;
    int* mine = copies + (warp % HC) * 2048;
    for (int i = tid; i < HC * 2048; i += THREADS) copies[i] = 0;
    __syncthreads();
    for (int p = tid; p < sg.len; p += THREADS) {
      const int j = sg.lo + p;
      if (elig(j)) {
        const uint32_t kj = key(j);
        if ((kj & mask) == prefix) atomicAdd(&mine[(kj >> shift) & (nb - 1)], 1);
      }
    }
    __syncthreads();
    for (int i = tid; i < nb; i += THREADS) {
      int c = 0;
#pragma unroll
      for (int q = 0; q < HC; ++q) c += copies[q * 2048 + i];
      h[i] = c;
    }
    cl.sync();   // every CTA's histogram is complete
    // Thread u owns the bins nb-1-u*bpt-q (q < bpt), i.e. bins from the top,
    // summed over the cluster in rank order.
    const int bpt = nb / THREADS;
    int cnt[2048 / THREADS] = {};
    int sum = 0;
    for (int q = 0; q < bpt; ++q) {
      const int bin = nb - 1 - tid * bpt - q;
      int c = 0;
#pragma unroll
      for (int rr = 0; rr < kMaxCluster; ++rr)
        if (rr < C) c += cl.map_shared_rank(h, rr)[bin];
      cnt[q] = c;
      sum += c;
    }
    int total;
    int acc = block_scan<THREADS / 32>(sum, sh.warp_vals, &total);
    for (int q = 0; q < bpt; ++q) {
      if (acc < need && need <= acc + cnt[q]) {
        sh.pick[0] = nb - 1 - tid * bpt - q;
        sh.pick[1] = acc;
        sh.pick[2] = cnt[q];
      }
      acc += cnt[q];
    }
    __syncthreads();
    prefix |= (uint32_t)sh.pick[0] << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    need -= sh.pick[1];
    whole = sh.pick[2] == need;   // the same in every CTA of the cluster
    __syncthreads();
    if (whole) break;
  }

  if (whole) {
    // Take every eligible key whose top bits are at least the prefix.
    const int w0 = warp * sg.cw, w1 = min(sg.len, w0 + sg.cw);
    for (int i = w0; i < w0 + sg.cw; i += 32) {
      const int p = i + lane;
      bool take = false;
      if (p < w1) {
        const int j = sg.lo + p;
        take = elig(j) && (key(j) & mask) >= prefix;
      }
      const unsigned word = __ballot_sync(0xffffffffu, take);
      if (lane == 0 && word) bits[i >> 5] |= word;
    }
    // The other CTAs have read this CTA's histograms before any later call
    // writes them again.
    cl.sync();
    __syncthreads();
    return;
  }

  // Take keys > T, and the first `need` keys == T in position order.
  const uint32_t T = prefix;
  const int w0 = warp * sg.cw, w1 = min(sg.len, w0 + sg.cw);
  int eq_count = 0;
  for (int i = w0; i < w0 + sg.cw; i += 32) {
    const int p = i + lane;
    bool eq = false;
    if (p < w1) {
      const int j = sg.lo + p;
      eq = elig(j) && key(j) == T;
    }
    eq_count += __popc(__ballot_sync(0xffffffffu, eq));
  }
  const int2 ws = scan_warp_counts<THREADS / 32>(eq_count, sh);
  if (tid == 0) sh.xchg[xslot] = ws.y;
  cl.sync();   // the CTAs' counts of equal keys are published
  int running = lower_ranks_sum(cl, sh, xslot, rank) + ws.x;
  const unsigned lower = (1u << lane) - 1u;
  for (int i = w0; i < w0 + sg.cw; i += 32) {
    const int p = i + lane;
    bool gt = false, eq = false;
    if (p < w1) {
      const int j = sg.lo + p;
      if (elig(j)) {
        const uint32_t kj = key(j);
        gt = kj > T;
        eq = kj == T;
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, eq);
    const bool take = gt || (eq && running + __popc(bal & lower) < need);
    const unsigned word = __ballot_sync(0xffffffffu, take);
    if (lane == 0 && word) bits[i >> 5] |= word;
    running += __popc(bal);
  }
  __syncthreads();
}

template <bool SMEM_KEYS, int THREADS>
__global__ void __launch_bounds__(THREADS) select_kernel(const SelectArgs a,
                                                         const int seg) {
  constexpr int WARPS = THREADS / 32;
  constexpr int HC = hist_copies(THREADS);
  extern __shared__ uint32_t bits[];
  __shared__ Shared sh;
  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int row = blockIdx.x / C;
  // Dynamic shared memory: mark bitmap | 2 folded histograms | histogram
  // copies | keys | raw S_T (the last two only with SMEM_KEYS).
  int* fold = reinterpret_cast<int*>(bits + seg / 32);
  int* copies = fold + 2 * 2048;
  uint32_t* skeys = reinterpret_cast<uint32_t*>(copies + HC * 2048);
  float* sraw = reinterpret_cast<float*>(skeys + seg);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.n, k = a.k;
  int32_t* out = a.idx + (long long)row * min(k, n);
  const float* sd = a.sd ? a.sd + (long long)row * n : nullptr;
  const float* st = a.st ? a.st + (long long)row * n : nullptr;
  Seg sg;
  sg.lo = min(n, rank * seg);
  sg.len = min(n, sg.lo + seg) - sg.lo;
  sg.cw = ((sg.len + 32 * WARPS - 1) / (32 * WARPS)) * 32;
  griddep_wait();
  griddep_launch_dependents();
  if (k >= n) {   // uniform over the cluster: no barriers on this path
    for (int p = tid; p < sg.len; p += THREADS) out[sg.lo + p] = sg.lo + p;
    return;
  }
  const int ns = min(max(a.n_sink, 0), n);
  const int hi = n - min(max(a.n_recent, 0), n);
  auto forced = [&](int j) { return j < ns || j >= hi; };
  const int n_forced = hi <= ns ? n : ns + (n - hi);
  const int budget = k - n_forced;  // >= 0, checked on the host
  for (int i = tid; i < seg / 32; i += THREADS) bits[i] = 0u;
  __syncthreads();
  auto marked = [&](int j) { return (bits[(j - sg.lo) >> 5] >> ((j - sg.lo) & 31)) & 1u; };
  auto not_forced = [&](int j) { return !forced(j); };

  if (a.m < 0) {
    const bool hasD = sd != nullptr && a.alpha != 0.0;
    const bool hasT = st != nullptr && (1.0 - a.alpha) != 0.0;
    const bool sums = a.norm == 1 && (hasD || hasT);
    double cd = a.alpha, ct = 1.0 - a.alpha;
    // One read of the segment's scores: the raw values go to shared memory
    // (S_D's bits in skeys, S_T in sraw) when the keys are cached, and the
    // L1 partial sums are taken on the way.
    float2 pd = make_float2(0.f, 0.f), pt = make_float2(0.f, 0.f);
    if (SMEM_KEYS || sums) {
#pragma unroll 4
      for (int p = tid; p < sg.len; p += THREADS) {
        const float x = hasD ? __ldg(sd + sg.lo + p) : 0.f;
        const float y = hasT ? __ldg(st + sg.lo + p) : 0.f;
        if constexpr (SMEM_KEYS) {
          skeys[p] = __float_as_uint(x);
          sraw[p] = y;
        }
        if (sums) {
          two_sum_acc(pd, x);
          two_sum_acc(pt, y);
        }
      }
    }
    if (sums) {
      const float4 part = block_sum_ff2<WARPS>(pd, pt, sh.fbuf);
      if (tid == 0) {
        sh.dpart[0] = (double)part.x + (double)part.y;
        sh.dpart[1] = (double)part.z + (double)part.w;
      }
      cl.sync();   // the partial sums are published
      if (tid == 0) {
        double tot_d = 0.0, tot_t = 0.0;
        for (int rr = 0; rr < C; ++rr) {   // rank order: the same in every CTA
          const double* dp = cl.map_shared_rank(sh.dpart, rr);
          tot_d += dp[0];
          tot_t += dp[1];
        }
        if (hasD && tot_d > 0.0 && isfinite(tot_d)) cd = cd / tot_d;
        if (hasT && tot_t > 0.0 && isfinite(tot_t)) ct = ct / tot_t;
        sh.coef[0] = (float)cd;
        sh.coef[1] = (float)ct;
      }
      __syncthreads();
    } else if (tid == 0) {
      sh.coef[0] = (float)cd;
      sh.coef[1] = (float)ct;
    }
    __syncthreads();
    const float fd = sh.coef[0], ft = sh.coef[1];
    auto mix_of = [&](float x, float y) -> uint32_t {
      float c;
      if (hasD && hasT)
        c = __fadd_rn(__fmul_rn(fd, x), __fmul_rn(ft, y));
      else if (hasD)
        c = __fmul_rn(fd, x);
      else if (hasT)
        c = __fmul_rn(ft, y);
      else
        c = 0.f;
      return order_key(c);
    };
    if constexpr (SMEM_KEYS) {
      for (int p = tid; p < sg.len; p += THREADS)
        skeys[p] = mix_of(__uint_as_float(skeys[p]), sraw[p]);
      __syncthreads();
      auto cached = [&](int j) { return skeys[j - sg.lo]; };
      select_mark<THREADS>(cl, rank, C, budget, sg, cached, not_forced, bits, fold, copies, sh, 0);
    } else {
      auto mix = [&](int j) -> uint32_t {
        return mix_of(hasD ? __ldg(sd + j) : 0.f, hasT ? __ldg(st + j) : 0.f);
      };
      select_mark<THREADS>(cl, rank, C, budget, sg, mix, not_forced, bits, fold, copies, sh, 0);
    }
  } else {
    const int m_eff = min(a.m, budget);
    auto free_pos = [&](int j) { return !forced(j) && !marked(j); };
    if constexpr (SMEM_KEYS) {
      auto cached = [&](int j) { return skeys[j - sg.lo]; };
      if (m_eff > 0) {
        for (int p = tid; p < sg.len; p += THREADS) skeys[p] = order_key(sd[sg.lo + p]);
        __syncthreads();
        select_mark<THREADS>(cl, rank, C, m_eff, sg, cached, not_forced, bits, fold, copies, sh, 0);
      }
      if (budget - m_eff > 0) {
        for (int p = tid; p < sg.len; p += THREADS) skeys[p] = order_key(st[sg.lo + p]);
        __syncthreads();
        select_mark<THREADS>(cl, rank, C, budget - m_eff, sg, cached, free_pos, bits, fold, copies, sh, 1);
      }
    } else {
      if (m_eff > 0) {
        auto kd = [&](int j) { return order_key(sd[j]); };
        select_mark<THREADS>(cl, rank, C, m_eff, sg, kd, not_forced, bits, fold, copies, sh, 0);
      }
      if (budget - m_eff > 0) {
        auto kt = [&](int j) { return order_key(st[j]); };
        select_mark<THREADS>(cl, rank, C, budget - m_eff, sg, kt, free_pos, bits, fold, copies, sh, 1);
      }
    }
  }

  // Ordered compaction of protected + marked positions.
  const int w0 = warp * sg.cw, w1 = min(sg.len, w0 + sg.cw);
  int kept = 0;
  for (int i = w0; i < w0 + sg.cw; i += 32) {
    const int p = i + lane;
    const bool keep = p < w1 && (forced(sg.lo + p) || marked(sg.lo + p));
    kept += __popc(__ballot_sync(0xffffffffu, keep));
  }
  const int2 ws = scan_warp_counts<WARPS>(kept, sh);
  if (tid == 0) sh.xchg[2] = ws.y;
  cl.sync();   // the CTAs' kept counts are published
  int running = lower_ranks_sum(cl, sh, 2, rank) + ws.x;
  const unsigned lower = (1u << lane) - 1u;
  for (int i = w0; i < w0 + sg.cw; i += 32) {
    const int p = i + lane;
    const bool keep = p < w1 && (forced(sg.lo + p) || marked(sg.lo + p));
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    const int pos = running + __popc(bal & lower);
    if (keep && pos < k) out[pos] = sg.lo + p;
    running += __popc(bal);
  }
  cl.sync();   // nobody reads this CTA's shared memory any more
}

int smem_bytes(int seg, bool cache, int threads = kThreads) {
  return seg / 32 * 4 + (2 + hist_copies(threads)) * 2048 * 4 + (cache ? 2 * seg * 4 : 0);
}

// Clusters of `c` select CTAs that fit on the current device at once
// (cached per device and cluster size).
int max_active_clusters(int c, bool cache) {
  static std::atomic<int> memo[64][kMaxCluster + 1][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  std::atomic<int>& m = memo[dev][c][cache ? 1 : 0];
  int v = m.load(std::memory_order_relaxed);
  if (v > 0) return v;
  auto kern = cache ? select_kernel<true, kThreads> : select_kernel<false, kThreads>;
  const int smem = smem_bytes(kSmemKeysMaxSeg, cache);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(c * 64));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&v, kern, &cfg) != cudaSuccess || v < 1)
    v = 1;
  m.store(v, std::memory_order_relaxed);
  return v;
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st) {
  // C CTAs per sequence, each owning seg positions (a multiple of 32): as
  // many as the row calls for (4096 positions a CTA), halved while the
  // sequences' clusters would not all be resident at once.
  int C = std::min(kMaxCluster, std::max(1, (a.n + kSegPerCta - 1) / kSegPerCta));
  auto seg_of = [&](int c) { return std::max(32, (((a.n + c - 1) / c) + 31) & ~31); };
  while (C > 1 && a.b > max_active_clusters(C, seg_of(C) <= kSmemKeysMaxSeg && a.k < a.n))
    C /= 2;
  const int seg = seg_of(C);
  const bool cache = seg <= kSmemKeysMaxSeg && a.k < a.n;
  // Many short rows (one CTA each, more rows than two 1024-thread CTAs per
  // SM hold at once): 256-thread CTAs with one histogram copy, several per
  // SM.  Measured on 1024 rows of 2048 page scores: 42 us against 82 us
  // with 1024-thread CTAs.
  const bool short_rows = C == 1 && a.n <= kSegPerCta && a.b >= kShortRowsMinRows;
  const int threads = short_rows ? kThreadsShort : kThreads;
  const int smem = smem_bytes(seg, cache, threads);
  auto kern = short_rows ? (cache ? select_kernel<true, kThreadsShort>
                                  : select_kernel<false, kThreadsShort>)
                         : (cache ? select_kernel<true, kThreads>
                                  : select_kernel<false, kThreads>);
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl_cluster(kern, dim3((unsigned)(a.b * C)), dim3(threads), smem, st,
                         (unsigned)C, a, seg);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace dustin
