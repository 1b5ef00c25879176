// Quest page scoring, the page-level baseline selector the notes compare
// against ("dustin-long-context" notes, section 1 and related work; the
// "Quest-16" curve of Fig. 8): per-page, per-channel min/max key statistics
// and, for each query head, the page score
//   score[b][h][p] = sum_c max(q_c * min_c, q_c * max_c),
// the largest q . k over the page's channel box.
//
//  * quest_stats_kernel: one warp per (sequence, kv head, page); each lane
//    owns D/32 channels and folds the page's rows into fp32 minima and
//    maxima, written back as bf16 (exact: they are bf16 inputs).  Stats
//    layout [b][h_kv][P][2][D] (minimum row, then maximum row).
//  * quest_score_kernel: one warp per 32 pages of one (sequence, kv head),
//    for all G query heads of that kv head; each lane owns D/32 channels of
//    a page's two stat rows (coalesced loads) and of the G query rows (fp32
//    in shared memory), forms q_c * (q_c >= 0 ? mx_c : mn_c) summed over its
//    channels, and the heads' sums over the lanes are taken eight at a time
//    by a shuffle reduce-scatter; results leave as one store per head and
//    32 pages.
#include "device_common.cuh"
#include "dustin.h"
#include "internal.h"

namespace dustin {

namespace {

__device__ unsigned int g_quest_dev_flags;

template <int D, bool PAGED>
__global__ void __launch_bounds__(256) quest_stats_kernel(const QuestArgs a) {
  constexpr int CPL = D / 32;   // channels per lane
  const int lane = threadIdx.x & 31;
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const long long total = (long long)a.b * a.hkv * a.n_pages;
  griddep_wait();
  griddep_launch_dependents();
  if (gw >= total) return;
  const int p = (int)(gw % a.n_pages);
  const int g = (int)((gw / a.n_pages) % a.hkv);
  const int bb = (int)(gw / ((long long)a.n_pages * a.hkv));
  const int r0 = p * a.page, r1 = min(a.n, r0 + a.page);
  float mn[CPL], mx[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    mn[c] = INFINITY;
    mx[c] = -INFINITY;
  }
  for (int j = r0; j < r1; ++j) {
    long long off;
    if constexpr (PAGED) {
      const int pg = __ldg(a.kv.page_table + (long long)bb * a.kv.pages_per_seq +
                           j / a.kv.page_size);
      if (pg < 0 || pg >= a.kv.num_pages) {
        if (lane == 0) atomicOr(&g_quest_dev_flags, 2u);
        continue;
      }
      off = (long long)pg * a.kv.sb + (long long)g * a.kv.sh +
            (long long)(j % a.kv.page_size) * a.kv.sn;
    } else {
      off = (long long)bb * a.kv.sb + (long long)g * a.kv.sh + (long long)j * a.kv.sn;
    }
    const __nv_bfloat16* row = a.kv.k + off + lane * CPL;
    __nv_bfloat16 v[CPL];
    if constexpr (CPL == 4) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(row));
      memcpy(v, &u, sizeof(u));
    } else {
      const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(row));
      memcpy(v, &u, sizeof(u));
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const float f = __bfloat162float(v[c]);
      mn[c] = fminf(mn[c], f);
      mx[c] = fmaxf(mx[c], f);
    }
  }
  __nv_bfloat16 omn[CPL], omx[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    omn[c] = __float2bfloat16_rn(mn[c]);
    omx[c] = __float2bfloat16_rn(mx[c]);
  }
  __nv_bfloat16* dst = a.stats + gw * 2 * D + lane * CPL;
  if constexpr (CPL == 4) {
    uint2 u;
    memcpy(&u, omn, sizeof(u));
    *reinterpret_cast<uint2*>(dst) = u;
    memcpy(&u, omx, sizeof(u));
    *reinterpret_cast<uint2*>(dst + D) = u;
  } else {
    uint32_t u;
    memcpy(&u, omn, sizeof(u));
    *reinterpret_cast<uint32_t*>(dst) = u;
    memcpy(&u, omx, sizeof(u));
    *reinterpret_cast<uint32_t*>(dst + D) = u;
  }
}

constexpr int kScoreWarps = 8;
constexpr int kPagesPerWarp = 32;
constexpr int kPagesPerCta = kScoreWarps * kPagesPerWarp;
constexpr int kHeadChunk = 8;

// Sum over the 32 lanes of eight values per lane, leaving the sum of value
// (lane >> 2) & 7 on every lane (nine shuffles: halves exchanged at lane
// distances 16, 8, 4, then a plain sum over distances 2 and 1).
__device__ __forceinline__ float reduce8(const float (&v)[kHeadChunk], int lane) {
  float a[4], b[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 16;
    const float mine = hi ? v[i + 4] : v[i], other = hi ? v[i] : v[i + 4];
    a[i] = mine + __shfl_xor_sync(0xffffffffu, other, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 8;
    const float mine = hi ? a[i + 2] : a[i], other = hi ? a[i] : a[i + 2];
    b[i] = mine + __shfl_xor_sync(0xffffffffu, other, 8);
  }
  const bool hi = lane & 4;
  float c = (hi ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, hi ? b[0] : b[1], 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

// One warp per 32 consecutive pages of one (sequence, kv head); lane l owns
// channels [l D/32, (l + 1) D/32) of each page's two stat rows (coalesced
// loads), forms its part of every head's bound, and the eight heads of a
// chunk are summed over the lanes together (reduce8).  A page's bounds go
// to shared memory and each head's 32 pages leave as one 128-byte store.
template <int D>
__global__ void __launch_bounds__(kScoreWarps * 32)
    quest_score_kernel(const QuestArgs a) {
  constexpr int CPL = D / 32;   // channels per lane
  extern __shared__ float sq[];  // [G][D] fp32 query rows, then [warps][8][32]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int blocks_per_head = (a.n_pages + kPagesPerCta - 1) / kPagesPerCta;
  const int pb = blockIdx.x % blocks_per_head;
  const int g = (blockIdx.x / blocks_per_head) % a.hkv;
  const int bb = blockIdx.x / (blocks_per_head * a.hkv);
  const int group = a.hq / a.hkv;
  float* res = sq + group * D + warp * kHeadChunk * 32;
  griddep_wait();
  griddep_launch_dependents();
  for (int i = tid; i < group * D; i += kScoreWarps * 32) {
    const int h = g * group + i / D;
    sq[i] = __bfloat162float(a.q[((long long)bb * a.hq + h) * D + i % D]);
  }
  __syncthreads();
  const int p0 = pb * kPagesPerCta + warp * kPagesPerWarp;
  if (p0 >= a.n_pages) return;
  const int np = min(kPagesPerWarp, a.n_pages - p0);
  const __nv_bfloat16* st0 =
      a.stats_in + (((long long)bb * a.hkv + g) * a.n_pages + p0) * 2 * D + lane * CPL;
  for (int h0 = 0; h0 < group; h0 += kHeadChunk) {
    const int nh = min(kHeadChunk, group - h0);
    float qv[kHeadChunk][CPL];
#pragma unroll
    for (int h = 0; h < kHeadChunk; ++h)
#pragma unroll
      for (int c = 0; c < CPL; ++c)
        qv[h][c] = h < nh ? sq[(h0 + h) * D + lane * CPL + c] : 0.f;
    for (int pp = 0; pp < np; ++pp) {
      const __nv_bfloat16* st = st0 + (long long)pp * 2 * D;
      __nv_bfloat16 vmn[CPL], vmx[CPL];
      if constexpr (CPL == 4) {
        const uint2 umn = __ldg(reinterpret_cast<const uint2*>(st));
        const uint2 umx = __ldg(reinterpret_cast<const uint2*>(st + D));
        memcpy(vmn, &umn, 8);
        memcpy(vmx, &umx, 8);
      } else {
        const uint32_t umn = __ldg(reinterpret_cast<const uint32_t*>(st));
        const uint32_t umx = __ldg(reinterpret_cast<const uint32_t*>(st + D));
        memcpy(vmn, &umn, 4);
        memcpy(vmx, &umx, 4);
      }
      float part[kHeadChunk];
#pragma unroll
      for (int h = 0; h < kHeadChunk; ++h) {
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const float qc = qv[h][c];
          acc = fmaf(qc, __bfloat162float(qc >= 0.f ? vmx[c] : vmn[c]), acc);
        }
        part[h] = acc;
      }
      const float sum = reduce8(part, lane);
      if ((lane & 3) == 0) res[((lane >> 2) & 7) * 32 + pp] = sum;
    }
    __syncwarp();
    for (int h = 0; h < nh; ++h)
      if (lane < np)
        a.scores[((long long)bb * a.hq + g * group + h0 + h) * a.n_pages + p0 + lane] =
            res[h * 32 + lane];
    __syncwarp();
  }
}

template <int D, bool PAGED>
cudaError_t run_stats(const QuestArgs& a, cudaStream_t st) {
  const long long total = (long long)a.b * a.hkv * a.n_pages;
  cudaError_t e = launch_pdl(quest_stats_kernel<D, PAGED>, dim3((unsigned)((total + 7) / 8)),
                             dim3(256), 0, st, a);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

template <int D>
cudaError_t run_scores(const QuestArgs& a, cudaStream_t st) {
  const int bph = (a.n_pages + kPagesPerCta - 1) / kPagesPerCta;
  const long long grid = (long long)a.b * a.hkv * bph;
  const int smem = ((a.hq / a.hkv) * D + kScoreWarps * kHeadChunk * 32) * 4;
  cudaError_t e = cudaFuncSetAttribute(quest_score_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(quest_score_kernel<D>, dim3((unsigned)grid), dim3(kScoreWarps * 32), smem,
                 st, a);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

}  // namespace

cudaError_t launch_quest_stats(const QuestArgs& a, int d, bool paged, cudaStream_t st) {
  if (d == 64) return paged ? run_stats<64, true>(a, st) : run_stats<64, false>(a, st);
  return paged ? run_stats<128, true>(a, st) : run_stats<128, false>(a, st);
}

cudaError_t launch_quest_scores(const QuestArgs& a, int d, cudaStream_t st) {
  return d == 64 ? run_scores<64>(a, st) : run_scores<128>(a, st);
}

cudaError_t take_quest_flags(unsigned* flags) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_quest_dev_flags, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_quest_dev_flags, &zero, sizeof(zero));
  *flags |= v;
  return e;
}

}  // namespace dustin
