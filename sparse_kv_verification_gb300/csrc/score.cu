// Importance scoring on the scored (layer, head) pairs: S_Target and
// S_Draft of the "dustin-long-context" notes, section 2.2 (attention summed
// over heads, layers and query rows), restricted to a few heads as in
// section 2.4 / Fig. 6.
//
//   S[b][j] = sum_p sum_r softmax_j(scale * q[p][b][r] . K_p[b][g_p][j])
//
// Two passes.  Pass 1 computes each row's logits (log2 units) with bf16
// mma.sync (fp32 accumulate), writes them to the workspace and keeps an
// online (max, sum of 2^(l - max)) per row and 512-position chunk: the
// persistent TMA kernel (score_logits_tma_kernel, below) for contiguous
// caches and for pages of 16, 32 or 64 positions; otherwise
// score_logits_kernel, one CTA per (pair, sequence, chunk) streaming the
// chunk's key rows through a 4-stage cp.async pipeline into swizzled shared
// memory.
// Pass 2 (score_reduce_kernel): combines the chunk statistics into each
// row's log2-sum-exp and writes S[b][j] = sum_{p,r} 2^(l - lse2), summed
// in a fixed order (pair-major, then row) in fp32, four positions per
// thread with the logits loads batched ahead of the sums.
// The logits are scratch that pass 2 reads once: when n is a multiple of 32
// (and the workspace 128-byte aligned) pass 1 writes them under an
// evict-last L2 policy and pass 2 drops each 128-byte line from L2 after
// reading it, so they are read from L2 and never written back to DRAM
// (72B-shaped step: target scoring 93.1 -> 89.0 us, draft 57.0 -> 56.3 us).
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <mutex>

#include "device_common.cuh"
#include "dustin.h"
#include "internal.h"

namespace dustin {

namespace {

constexpr int kTile = 64;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 4;
constexpr int kMaxTab = 2048;

template <int D>
struct ScoreCfg {
  static constexpr int CPR = D / 8;
  static constexpr int KS = D / 16;
  static constexpr int TILE_BYTES = kTile * D * 2;
  static constexpr int Q_BYTES = 16 * D * 2;
  static constexpr int SMEM = Q_BYTES + kStages * TILE_BYTES + kMaxTab * 8 +
                              kWarps * 16 * 8;
};

__device__ unsigned int g_score_dev_flags;

template <int D, bool PAGED>
__global__ void __launch_bounds__(kThreads)
    score_logits_kernel(const ScoreArgs a) {
  using C = ScoreCfg<D>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sK = sQ + C::Q_BYTES;
  long long* tab = reinterpret_cast<long long*>(sK + kStages * C::TILE_BYTES);
  float2* red = reinterpret_cast<float2*>(tab + kMaxTab);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x % a.nchunks;
  const int bb = (blockIdx.x / a.nchunks) % a.b;
  const int p = blockIdx.x / (a.nchunks * a.b);
  const ScorePair& pr = a.pairs[p];
  const KvView& kv = pr.kv;

  const int p_begin = c * a.chunk;
  const int p_end = min(a.n, p_begin + a.chunk);
  const int len = max(0, p_end - p_begin);
  const int ntiles = (len + kTile - 1) / kTile;
  const long long unit_off = (long long)bb * kv.sb + (long long)pr.kv_head * kv.sh;
  griddep_wait();
  griddep_launch_dependents();

  // Query rows of this (pair, sequence): q[p][b][r][D], zero past `rows`.
  const __nv_bfloat16* qb = a.q + ((long long)p * a.b + bb) * a.rows * D;
  for (int i = tid; i < 16 * C::CPR; i += kThreads) {
    const int r = i / C::CPR, ch = i % C::CPR;
    const bool ok = r < a.rows;
    cp_async_16(smem_u32(sQ + swz<D>(r, ch)), qb + (ok ? r * D + ch * 8 : 0),
                ok ? 16 : 0);
  }
  cp_async_commit();

  if constexpr (PAGED) {
    const int pg0 = p_begin / kv.page_size;
    const int npg = len > 0 ? (p_end - 1) / kv.page_size - pg0 + 1 : 0;
    for (int i = tid; i < npg; i += kThreads) {
      const int pg = __ldg(kv.page_table + (long long)bb * kv.pages_per_seq + pg0 + i);
      long long off = -1;
      if (pg < 0 || pg >= kv.num_pages)
        atomicOr(&g_score_dev_flags, 2u);
      else
        off = (long long)pg * kv.sb + (long long)pr.kv_head * kv.sh;
      tab[i] = off;
    }
  }
  __syncthreads();

  auto row_offset = [&](int i) -> long long {
    const int j = p_begin + i;
    if constexpr (PAGED) {
      const long long base = tab[j / kv.page_size - p_begin / kv.page_size];
      return base < 0 ? -1 : base + (long long)(j % kv.page_size) * kv.sn;
    } else {
      return unit_off + (long long)j * kv.sn;
    }
  };

  auto issue_tile = [&](int t) {
    if (t < ntiles) {
      const uint32_t dk = smem_u32(sK + (t % kStages) * C::TILE_BYTES);
      for (int i = tid; i < kTile * C::CPR; i += kThreads) {
        const int r = i / C::CPR, ch = i % C::CPR;
        const int pos = t * kTile + r;
        const long long off = pos < len ? row_offset(pos) : -1;
        const bool ok = off >= 0;
        cp_async_16(dk + swz<D>(r, ch), kv.k + (ok ? off + ch * 8 : 0), ok ? 16 : 0);
      }
    }
    cp_async_commit();
  };

  for (int t = 0; t < kStages - 1; ++t) issue_tile(t);
  cp_async_wait<kStages - 1>();
  __syncthreads();
  uint32_t qf[C::KS][4];
#pragma unroll
  for (int ks = 0; ks < C::KS; ++ks)
    ldmatrix_x4(smem_u32(sQ + swz<D>(lane & 15, ks * 2 + (lane >> 4))), qf[ks][0],
                qf[ks][1], qf[ks][2], qf[ks][3]);

  const int gq = lane >> 2, tq = lane & 3;
  const bool rowA = gq < a.rows, rowB = gq + 8 < a.rows;
  float* outA = a.logits + (((long long)p * a.rows + gq) * a.b + bb) * a.n;
  float* outB = a.logits + (((long long)p * a.rows + gq + 8) * a.b + bb) * a.n;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    issue_tile(t + kStages - 1);
    const unsigned char* tk = sK + (t % kStages) * C::TILE_BYTES;

    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      const int r = warp * 16 + ((lane >> 4) << 3) + (lane & 7);
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4(smem_u32(tk + swz<D>(r, ks * 2 + ((lane >> 3) & 1))), b0, b1,
                  b2, b3);
      mma_bf16(s[0], qf[ks], b0, b1);
      mma_bf16(s[1], qf[ks], b2, b3);
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = t * kTile + warp * 16 + j * 8 + 2 * tq + e;
        bool ok = i < len;
        if constexpr (PAGED) ok = ok && row_offset(i) >= 0;
        const float va = ok ? s[j][e] * a.scale_log2 : -INFINITY;
        const float vb = ok ? s[j][e + 2] * a.scale_log2 : -INFINITY;
        s[j][e] = va;
        s[j][e + 2] = vb;
        if (i < len) {  // failed page checks store -inf: probability 0
          if (rowA) outA[p_begin + i] = va;
          if (rowB) outB[p_begin + i] = vb;
        }
        mx0 = fmaxf(mx0, va);
        mx1 = fmaxf(mx1, vb);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      ps0 += ex2(s[j][0] - u0) + ex2(s[j][1] - u0);
      ps1 += ex2(s[j][2] - u1) + ex2(s[j][3] - u1);
    }
    l0 = l0 * ex2(m0 - u0) + ps0;
    l1 = l1 * ex2(m1 - u1) + ps1;
    m0 = n0;
    m1 = n1;
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  cp_async_wait<0>();
  if (tq == 0) {
    red[warp * 16 + gq] = make_float2(m0, l0);
    red[warp * 16 + gq + 8] = make_float2(m1, l1);
  }
  __syncthreads();
  if (tid < a.rows) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red[w * 16 + tid].x);
    const float u = M == -INFINITY ? 0.f : M;
    float L = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float2 v = red[w * 16 + tid];
      L += v.y * ex2(v.x - u);
    }
    a.stats[(((long long)p * a.rows + tid) * a.b + bb) * a.nchunks + c] =
        make_float2(M, L);
  }
}

// One thread per 4 consecutive positions j of one sequence (16-byte loads
// when n % 4 == 0, 16-byte stores when S is 16-byte aligned too), 1024 per
// CTA.  The logits of the first kReduceRows rows
// are requested before the row statistics are combined, so their latency
// overlaps that step; later rows follow in batches of the same size, every
// batch's loads issued before any of its sums.  S is summed per position in
// row order, as a single chain.  The row statistics are combined by teams
// of 16 lanes, one row per team, 16 rows at once (draft scoring at the 72B
// shape: 56.4 -> 54.7 us against one warp per row, two rows per warp).
constexpr int kReduceRows = 8;   // (measured: 16 rows per batch is slower)

__global__ void __launch_bounds__(256) score_reduce_kernel(const ScoreArgs a) {
  __shared__ float lse2[1024];
  const int bb = blockIdx.y;
  const int prs = a.n_pairs * a.rows;
  const int lane = threadIdx.x & 31;
  const long long j0 = (long long)blockIdx.x * 1024 + threadIdx.x * 4;
  const bool vec = (a.n & 3) == 0;   // logits rows start 16-byte aligned
  const bool vec_out = vec && (reinterpret_cast<uintptr_t>(a.s_out) & 15u) == 0;
  griddep_wait();
  griddep_launch_dependents();

  auto load_batch = [&](int i0, float4 (&v)[kReduceRows]) {
#pragma unroll
    for (int u = 0; u < kReduceRows; ++u) {
      const int i = i0 + u;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i >= prs || j0 >= a.n) continue;
      const float* row = a.logits + ((long long)i * a.b + bb) * a.n;
      if (vec) {
        v[u] = __ldg(reinterpret_cast<const float4*>(row + j0));
      } else {
        v[u].x = __ldg(row + j0);
        if (j0 + 1 < a.n) v[u].y = __ldg(row + j0 + 1);
        if (j0 + 2 < a.n) v[u].z = __ldg(row + j0 + 2);
        if (j0 + 3 < a.n) v[u].w = __ldg(row + j0 + 3);
      }
    }
  };
  float4 v[kReduceRows];
  load_batch(0, v);

  // Row i's log2-sum-exp from its chunk statistics: a team of 16 lanes per
  // row (16 rows at once), the lanes over the chunks.
  {
    const int team = threadIdx.x >> 4, tl = threadIdx.x & 15;
    for (int i0 = 0; i0 < prs; i0 += 16) {
      const int i = i0 + team;
      const bool live = i < prs;
      const float2* st = a.stats + ((long long)(live ? i : 0) * a.b + bb) * a.nchunks;
      float M = -INFINITY;
      if (live)
        for (int c = tl; c < a.nchunks; c += 16) M = fmaxf(M, st[c].x);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float u = M == -INFINITY ? 0.f : M;
      float Z = 0.f;
      if (live)
        for (int c = tl; c < a.nchunks; c += 16) Z += st[c].y * ex2(st[c].x - u);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
      // An all-masked row contributes nothing.
      if (live && tl == 0) lse2[i] = Z > 0.f ? u + log2f(Z) : INFINITY;
    }
  }
  __syncthreads();

  // n a multiple of 32 and the logits on a 128-byte boundary: every
  // 128-byte line of a logits row belongs to the eight consecutive threads
  // of this CTA that read it; once they have, the first of them drops the
  // line from L2 (the logits are dead).
  const bool drop = (a.n & 31) == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 127u) == 0;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = 0; i0 < prs; i0 += kReduceRows) {
    if (i0 > 0) load_batch(i0, v);
#pragma unroll
    for (int u = 0; u < kReduceRows; ++u) {
      if (i0 + u >= prs) break;
      const float L = lse2[i0 + u];
      acc.x += ex2(v[u].x - L);
      acc.y += ex2(v[u].y - L);
      acc.z += ex2(v[u].z - L);
      acc.w += ex2(v[u].w - L);
    }
    if (drop) {
      __syncwarp();
      if ((lane & 7) == 0 && j0 < a.n) {
#pragma unroll
        for (int u = 0; u < kReduceRows; ++u)
          if (i0 + u < prs) discard_l2_line(a.logits + ((long long)(i0 + u) * a.b + bb) * a.n + j0);
      }
    }
  }
  if (j0 >= a.n) return;
  float* out = a.s_out + (long long)bb * a.n;
  if (vec_out) {
    *reinterpret_cast<float4*>(out + j0) = acc;
  } else {
    out[j0] = acc.x;
    if (j0 + 1 < a.n) out[j0 + 1] = acc.y;
    if (j0 + 2 < a.n) out[j0 + 2] = acc.z;
    if (j0 + 3 < a.n) out[j0 + 3] = acc.w;
  }
}

// ---- Contiguous key caches: the logits pass on TMA.
//
// A persistent kernel (one CTA per SM for d = 128, two for d = 64) takes the
// work items (pair, sequence, chunk) round-robin.  One producer warp loads
// each item's query rows (cp.async, handed over through q_full / q_empty)
// and, from lane 0, each 64-position tile of keys with tiled TMA loads of
// 64 x 64 boxes (one per 64 channels) into 128B-swizzled stages; the
// tensor map of a pair views its kv head of the cache as [b][n][d], so rows
// past n come back as zeros.  Four consumer warps take 16 positions each per
// tile, as in the cp.async kernel, and release the stage through its
// "empty" mbarrier.  Every wait is bounded and raises flag 0x4 on timeout.
// Paged caches (page size 16, 32 or 64): the tensor map of a pair views its
// kv head of the page pool as [P][page][d], and a tile is 64 / page boxes of
// one page each, whose ids the producer lanes read from the page table once
// per item (one page per lane); a page id outside the pool raises flag 0x2,
// its box is filled with zeros (an out-of-range coordinate) and its rows
// are left out through a per-stage mask, as in the cp.async kernel.
struct ScoreTmaArgs {
  ScoreArgs s;
  CUtensorMap maps[kMaxPairs];   // per pair: kv head kv_head as [b][n][d]
                                 // (paged: [P][page][d])
};

// Build-time tunables: TMA pipeline depth per CTA (several CTAs share an
// SM, each consuming its own tile).  Measured at the 72B shape: d = 64 with
// 3 stages 65.2 us per draft scoring call against 67.6 with 4, 69.3 with 6.
#ifndef DUSTIN_SCORE_STAGES128
#define DUSTIN_SCORE_STAGES128 3
#endif
#ifndef DUSTIN_SCORE_STAGES64
#define DUSTIN_SCORE_STAGES64 3
#endif

template <int D>
struct TmaCfg {
  static constexpr int STAGES = D == 128 ? DUSTIN_SCORE_STAGES128 : DUSTIN_SCORE_STAGES64;
  static constexpr int HALVES = D / 64;
  static constexpr int TILE_BYTES = kTile * D * 2;
  static constexpr int Q_BYTES = 16 * D * 2;
  static constexpr int OFF_Q = STAGES * TILE_BYTES;          // 1 KB multiple
  static constexpr int OFF_RED = OFF_Q + Q_BYTES;
  static constexpr int OFF_BAR = OFF_RED + kWarps * 16 * 8;
  static constexpr int NBARS = 2 * STAGES + 2;
  static constexpr int OFF_BAD = OFF_BAR + NBARS * 8;        // paged: bad-page mask / stage
  static constexpr int SMEM = OFF_BAD + STAGES * 4 + 1024;   // + alignment slack
  static constexpr int NT = (kWarps + 1) * 32;
};

template <int D, bool PAGED>
__global__ void __launch_bounds__(TmaCfg<D>::NT)
    score_logits_tma_kernel(const __grid_constant__ ScoreTmaArgs ta) {
  using C = ScoreCfg<D>;
  using T = TmaCfg<D>;
  const ScoreArgs& a = ta.s;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // The 128B swizzle pattern is a function of the address: stages start on
  // 1 KB boundaries.
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  unsigned char* sQ = smem + T::OFF_Q;
  float2* red = reinterpret_cast<float2*>(smem + T::OFF_RED);
  const uint32_t bar0 = smem_u32(smem + T::OFF_BAR);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (T::STAGES + s); };
  const uint32_t q_full = bar0 + 8u * (2 * T::STAGES);
  const uint32_t q_empty = q_full + 8u;
  unsigned* sBad = reinterpret_cast<unsigned*>(smem + T::OFF_BAD);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tpi = a.chunk / kTile;
  const long long n_items = (long long)a.n_pairs * a.b * a.nchunks;
  struct Item {
    int p, bb, c;
  };
  auto item_of = [&](long long it) {
    Item x;
    x.c = (int)(it % a.nchunks);
    x.bb = (int)((it / a.nchunks) % a.b);
    x.p = (int)(it / ((long long)a.nchunks * a.b));
    return x;
  };

  griddep_wait();
  griddep_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < T::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kWarps);
    }
    mbar_init(q_full, 32);
    mbar_init(q_empty, kWarps);
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ============================ producer warp ============================
    int t = 0, k = 0;
    bool ok_run = true;
    for (long long it = blockIdx.x; it < n_items && ok_run; it += gridDim.x, ++k) {
      const Item x = item_of(it);
      if (k > 0 && !mbar_wait(q_empty, (k - 1) & 1, kWaitLimitCycles)) {
        if (lane == 0) atomicOr(&g_score_dev_flags, 4u);
        break;
      }
      const __nv_bfloat16* qb = a.q + ((long long)x.p * a.b + x.bb) * a.rows * D;
      for (int i = lane; i < 16 * C::CPR; i += 32) {
        const int r = i / C::CPR, ch = i % C::CPR;
        const bool ok = r < a.rows;
        cp_async_16(smem_u32(sQ + swz<D>(r, ch)), qb + (ok ? r * D + ch * 8 : 0),
                    ok ? 16 : 0);
      }
      cp_async_mbar_arrive(q_full);
      const void* map = &ta.maps[x.p];
      // Paged: lane l holds the pool page of the chunk's l-th page (-1: past
      // n, or failed its check: read as zeros at an out-of-range page).
      int my_pid = -1;
      unsigned bad_pages = 0;
      int ps = kTile, pool = 0;
      if constexpr (PAGED) {
        const KvView& kv = a.pairs[x.p].kv;
        ps = kv.page_size;
        pool = kv.num_pages;
        const int pi = x.c * (a.chunk / ps) + lane;
        bool bad = false;
        if (lane < a.chunk / ps && (long long)pi * ps < a.n) {
          const int pid = __ldg(kv.page_table + (long long)x.bb * kv.pages_per_seq + pi);
          if (pid < 0 || pid >= kv.num_pages) {
            bad = true;
            atomicOr(&g_score_dev_flags, 2u);
          } else {
            my_pid = pid;
          }
        }
        bad_pages = __ballot_sync(0xffffffffu, bad);
      }
      // Keys read by one pair only are read once: evict them first, so the
      // logits written meanwhile are still in L2 when the second pass reads
      // them.  When pairs share keys (GQA sibling heads of one layer), the
      // next pair re-reads them soon after, so they get the normal policy
      // (measured, all 64 heads of each 72B layer scored: 99 ms per step
      // with evict-first against 71 ms without).
      const uint64_t pol = a.keys_shared ? policy_evict_normal() : policy_evict_first();
      for (int tt = 0; tt < tpi; ++tt, ++t) {
        const int st = t % T::STAGES;
        if (t >= T::STAGES &&
            !mbar_wait(empty_bar(st), ((t / T::STAGES) & 1) ^ 1, kWaitLimitCycles)) {
          if (lane == 0) atomicOr(&g_score_dev_flags, 4u);
          ok_run = false;
          break;
        }
        const uint32_t dst = smem_u32(smem + st * T::TILE_BYTES);
        if constexpr (PAGED) {
          const int ppt = kTile / ps;   // pages per tile
          const int pid = __shfl_sync(0xffffffffu, my_pid, tt * ppt + lane % ppt);
          if (lane == 0) {
            sBad[st] = (bad_pages >> (tt * ppt)) & ((1u << ppt) - 1u);
            mbar_arrive_expect_tx(full_bar(st), T::TILE_BYTES);
          }
          __syncwarp();
          if (lane < ppt) {
#pragma unroll
            for (int h = 0; h < T::HALVES; ++h)
              tma_load_3d_hint(dst + h * (kTile * 128) + lane * ps * 128, map, h * 64, 0,
                               pid >= 0 ? pid : pool, full_bar(st), pol);
          }
        } else if (lane == 0) {
          mbar_arrive_expect_tx(full_bar(st), T::TILE_BYTES);
          const int j0 = x.c * a.chunk + tt * kTile;
#pragma unroll
          for (int h = 0; h < T::HALVES; ++h)
            tma_load_3d_hint(dst + h * (kTile * 128), map, h * 64, j0, x.bb, full_bar(st),
                             pol);
        }
        __syncwarp();
      }
    }
    cp_async_wait<0>();
    return;
  }

  // ============================ consumer warps =============================
  const int gq = lane >> 2, tq = lane & 3;
  int t = 0, k = 0;
  bool dead = false;
  auto wait_or_die = [&](uint32_t bar, uint32_t parity) {
    if (dead) return;
    if (!mbar_wait(bar, parity, kWaitLimitCycles)) {
      dead = true;
      if (lane == 0) atomicOr(&g_score_dev_flags, 4u);
    }
  };
  for (long long it = blockIdx.x; it < n_items; it += gridDim.x, ++k) {
    const Item x = item_of(it);
    wait_or_die(q_full, k & 1);
    uint32_t qf[C::KS][4];
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks)
      ldmatrix_x4(smem_u32(sQ + swz<D>(lane & 15, ks * 2 + (lane >> 4))), qf[ks][0],
                  qf[ks][1], qf[ks][2], qf[ks][3]);
    __syncwarp();
    if (lane == 0) mbar_arrive(q_empty);
    const bool rowA = gq < a.rows, rowB = gq + 8 < a.rows;
    float* outA = a.logits + (((long long)x.p * a.rows + gq) * a.b + x.bb) * a.n;
    float* outB = a.logits + (((long long)x.p * a.rows + gq + 8) * a.b + x.bb) * a.n;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    // Logits rows of an even n take 8-byte stores; when n is a multiple of
    // 32 and the logits start on a 128-byte boundary the second pass
    // discards each 128-byte line after reading it, so the rows are written
    // to stay in L2 until then (evict-last) and never go back to DRAM.
    const bool pair_stores = (a.n & 1) == 0;
    const bool dropped = (a.n & 31) == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 127u) == 0;
    const uint64_t out_pol = dropped ? policy_evict_last() : policy_evict_normal();
    // Paged: log2 of the page size (16, 32 or 64), for the bad-page mask.
    const int page_shift = PAGED ? 31 - __clz(a.pairs[x.p].kv.page_size) : 6;

    for (int tt = 0; tt < tpi; ++tt, ++t) {
      const int st = t % T::STAGES;
      wait_or_die(full_bar(st), (t / T::STAGES) & 1);
      const unsigned char* tk = smem + st * T::TILE_BYTES;
      const int p0 = x.c * a.chunk + tt * kTile;
      const unsigned bad = PAGED ? sBad[st] : 0u;   // read before the stage is released
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int r = warp * 16 + ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
        // 16-byte chunk cg of row r, in the 64-channel box cg / 8, at its
        // 128B-swizzled place.
        const int cg = ks * 2 + ((lane >> 3) & 1);
        const uint32_t addr = smem_u32(tk + (cg >> 3) * (kTile * 128) + r * 128 +
                                       (((cg & 7) ^ (r & 7)) << 4));
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(addr, b0, b1, b2, b3);
        mma_bf16(sc[0], qf[ks], b0, b1);
        mma_bf16(sc[1], qf[ks], b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(st));
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pos = warp * 16 + jj * 8 + 2 * tq + e;   // in the tile
          const int j = p0 + pos;
          bool ok = j < a.n;
          if constexpr (PAGED) ok = ok && !((bad >> (pos >> page_shift)) & 1u);
          const float va = ok ? sc[jj][e] * a.scale_log2 : -INFINITY;
          const float vb = ok ? sc[jj][e + 2] * a.scale_log2 : -INFINITY;
          sc[jj][e] = va;
          sc[jj][e + 2] = vb;
          if (!pair_stores && j < a.n) {   // failed page checks store -inf
            if (rowA) outA[j] = va;
            if (rowB) outB[j] = vb;
          }
          mx0 = fmaxf(mx0, va);
          mx1 = fmaxf(mx1, vb);
        }
        // Positions j, j + 1 of a row as one 8-byte store (n even: j + 1 < n
        // whenever j < n), under the policy that keeps them in L2 for the
        // second pass.
        const int j = p0 + warp * 16 + jj * 8 + 2 * tq;
        if (pair_stores && j < a.n) {
          if (rowA) st_global_v2_hint(outA + j, sc[jj][0], sc[jj][1], out_pol);
          if (rowB) st_global_v2_hint(outB + j, sc[jj][2], sc[jj][3], out_pol);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        ps0 += ex2(sc[jj][0] - u0) + ex2(sc[jj][1] - u0);
        ps1 += ex2(sc[jj][2] - u1) + ex2(sc[jj][3] - u1);
      }
      l0 = l0 * ex2(m0 - u0) + ps0;
      l1 = l1 * ex2(m1 - u1) + ps1;
      m0 = n0;
      m1 = n1;
    }
    // Item end: per-row (max, sum) over the four warps.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (tq == 0) {
      red[warp * 16 + gq] = make_float2(m0, l0);
      red[warp * 16 + gq + 8] = make_float2(m1, l1);
    }
    named_bar_sync(1, kWarps * 32);
    if (tid < a.rows) {
      float M = -INFINITY;
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red[w * 16 + tid].x);
      const float u = M == -INFINITY ? 0.f : M;
      float L = 0.f;
      for (int w = 0; w < kWarps; ++w) {
        const float2 v = red[w * 16 + tid];
        L += v.y * ex2(v.x - u);
      }
      a.stats[(((long long)x.p * a.rows + tid) * a.b + x.bb) * a.nchunks + x.c] =
          make_float2(M, L);
    }
    named_bar_sync(1, kWarps * 32);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); null if unavailable.
EncodeTiledFn encode_tiled() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  static std::atomic<int> tried{0};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (f || tried.load()) return f;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                       cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess && p) {
    f = reinterpret_cast<EncodeTiledFn>(p);
    fn.store(f, std::memory_order_release);
  }
  tried.store(1);
  return f;
}

// Tensor maps of every pair; false if one cannot be encoded (or, paged, if
// a page size is not 16, 32 or 64: those pairs go to the cp.async kernel).
template <int D, bool PAGED>
bool make_maps(const ScoreArgs& a, ScoreTmaArgs& ta) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  for (int p = 0; p < a.n_pairs; ++p) {
    const KvView& kv = a.pairs[p].kv;
    void* base = const_cast<__nv_bfloat16*>(kv.k + (long long)a.pairs[p].kv_head * kv.sh);
    if (PAGED && !(kv.page_size == 16 || kv.page_size == 32 || kv.page_size == 64))
      return false;
    // Contiguous: the kv head as [b][n][d], 64-row boxes.  Paged: the kv
    // head of the pool as [P][page][d], one page a box.
    const cuuint64_t dims[3] = {(cuuint64_t)D,
                                (cuuint64_t)(PAGED ? kv.page_size : a.n),
                                (cuuint64_t)(PAGED ? kv.num_pages : a.b)};
    const cuuint64_t strides[2] = {(cuuint64_t)kv.sn * 2, (cuuint64_t)kv.sb * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)(PAGED ? kv.page_size : kTile), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&ta.maps[p], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

template <int D, bool PAGED>
cudaError_t run_score_tma(const ScoreArgs& a, cudaStream_t st, bool* used) {
  using T = TmaCfg<D>;
  *used = false;
  static ScoreTmaArgs ta;   // large: kept off the stack; guarded below
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  ta.s = a;
  if (!make_maps<D, PAGED>(a, ta)) return cudaSuccess;
  auto kern = score_logits_tma_kernel<D, PAGED>;
  static std::atomic<int> slots_memo[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) dev = 0;
  int slots = slots_memo[dev].load(std::memory_order_relaxed);
  if (slots <= 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
    if (e != cudaSuccess) return e;
    int occ = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, T::NT, T::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    slots = std::max(1, occ) * std::max(1, sms);
    slots_memo[dev].store(slots, std::memory_order_relaxed);
  }
  const long long items = (long long)a.n_pairs * a.b * a.nchunks;
  const long long grid = std::min<long long>(items, slots);
  e = launch_pdl(kern, dim3((unsigned)grid), dim3(T::NT), T::SMEM, st, ta);
  if (e != cudaSuccess) return e;
  note_launches(1);
  *used = true;
  return cudaSuccess;
}

template <int D, bool PAGED>
cudaError_t run_score_cp(const ScoreArgs& a, cudaStream_t st);

template <int D, bool PAGED>
cudaError_t run_score(const ScoreArgs& a, cudaStream_t st) {
  bool used = false;
  cudaError_t e = run_score_tma<D, PAGED>(a, st, &used);
  if (e != cudaSuccess) return e;
  if (used) {
    dim3 g2((unsigned)((a.n + 1023) / 1024), (unsigned)a.b);
    e = launch_pdl(score_reduce_kernel, g2, dim3(256), 0, st, a);
    if (e == cudaSuccess) note_launches(1);
    return e;
  }
  return run_score_cp<D, PAGED>(a, st);
}

template <int D, bool PAGED>
cudaError_t run_score_cp(const ScoreArgs& a, cudaStream_t st) {
  using C = ScoreCfg<D>;
  auto kern = score_logits_kernel<D, PAGED>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)a.n_pairs * a.b * a.nchunks;
  e = launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), C::SMEM, st, a);
  if (e != cudaSuccess) return e;
  note_launches(1);
  dim3 g2((unsigned)((a.n + 1023) / 1024), (unsigned)a.b);
  e = launch_pdl(score_reduce_kernel, g2, dim3(256), 0, st, a);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace

int score_chunk() { return 512; }

cudaError_t launch_score(const ScoreArgs& a, int d, bool paged,
                         cudaStream_t st) {
  if (d == 64) return paged ? run_score<64, true>(a, st) : run_score<64, false>(a, st);
  return paged ? run_score<128, true>(a, st) : run_score<128, false>(a, st);
}

cudaError_t take_score_flags(unsigned* flags) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_score_dev_flags, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_score_dev_flags, &zero, sizeof(zero));
  *flags |= v;
  return e;
}

}  // namespace dustin

// ------------------------------------------------------------------------
// Scoring without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they score: a serving
// loop that has handed all of HBM to the KV cache (cudaMalloc would fail or
// stall the step), or a plugin whose host framework owns the allocator and
// passes only input and output buffers.  dustin_score_heads_noalloc gives
// them the scoring call with its scratch in a fixed array compiled into this
// library.  Every GPU that loads the library holds the array until the
// process exits.
namespace dustin {
namespace {

static __device__ __align__(256) unsigned char
    g_noalloc_scratch[DUSTIN_NOALLOC_SCRATCH_BYTES];

// The current context's id through the runtime's driver entry points (no
// link against the driver library); 0 when there is no current context or
// the entry points are missing.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

unsigned long long current_context_id() {
  static std::atomic<void*> get_current{nullptr}, get_id{nullptr};
  static std::atomic<int> tried{0};
  if (!tried.load(std::memory_order_acquire)) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current.store(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id.store(p);
    tried.store(1, std::memory_order_release);
  }
  auto cur = reinterpret_cast<CtxGetCurrentFn>(get_current.load());
  auto id = reinterpret_cast<CtxGetIdFn>(get_id.load());
  CUcontext ctx = nullptr;
  unsigned long long v = 0;
  if (!cur || !id || cur(&ctx) != CUDA_SUCCESS || !ctx || id(ctx, &v) != CUDA_SUCCESS) return 0;
  return v;
}

// Device address of the array, per device, remembered together with the
// context it was looked up in: a new context on that device (after
// cudaDeviceReset, say) looks the address up again.  In host code the
// array's name is only a host-side stand-in, so the kernels always get this
// address.
struct NoallocSlot {
  void* ptr = nullptr;
  unsigned long long ctx = 0;
};
NoallocSlot g_noalloc_slot[64];
std::mutex g_noalloc_mutex;

cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocSlot& slot = g_noalloc_slot[dev];
  const unsigned long long ctx = current_context_id();
  if (slot.ptr == nullptr || ctx == 0 || ctx != slot.ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    slot.ptr = p;
    slot.ctx = current_context_id();   // the lookup made the context current
  }
  *out = slot.ptr;
  return cudaSuccess;
}

}  // namespace
}  // namespace dustin

extern "C" size_t dustin_score_heads_noalloc_capacity(void) {
  return (size_t)DUSTIN_NOALLOC_SCRATCH_BYTES;
}

extern "C" int dustin_score_heads_noalloc(int b, int n, int d, int n_pairs,
                                          int rows, const void* q,
                                          const dustin_kv* kv,
                                          const int32_t* kv_head, float scale,
                                          float* s_out, void* stream) {
  using namespace dustin;
  const char* what = "dustin_score_heads_noalloc";
  bool paged = false, empty = false;
  const int rc = check_score_args(b, n, d, n_pairs, rows, q, kv, kv_head, scale, s_out,
                                  what, &paged, &empty);
  if (rc || empty) return rc;
  const size_t need = dustin_score_heads_workspace_size(b, n, n_pairs, rows);
  if (need > (size_t)DUSTIN_NOALLOC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "%s: this call needs %zu bytes of scratch; the built-in array holds %zu "
             "(use dustin_score_heads with a workspace)",
             what, need, (size_t)DUSTIN_NOALLOC_SCRATCH_BYTES);
    return record_error(DUSTIN_ERR_WORKSPACE, msg);
  }
  void* ws = nullptr;
  cudaError_t e = noalloc_scratch(&ws);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "%s: cudaGetSymbolAddress: %s", what, cudaGetErrorString(e));
    return record_error(DUSTIN_ERR_CUDA, msg);
  }
  return dustin_score_heads(b, n, d, n_pairs, rows, q, kv, kv_head, scale,
                            s_out, ws, (size_t)DUSTIN_NOALLOC_SCRATCH_BYTES,
                            stream);
}
