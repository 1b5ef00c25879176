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
//  * quest_score_kernel: one thread per page of one (sequence, kv head),
//    for all G query heads of that kv head; the G query rows sit in shared
//    memory as fp32 and are read as broadcasts, the page's two stat rows
//    stream through 16-byte loads.  max(q_c mn_c, q_c mx_c) is taken as
//    q_c * (q_c >= 0 ? mx_c : mn_c), summed over channels in ascending order.
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

constexpr int kScoreThreads = 128;
constexpr int kHeadChunk = 8;

template <int D>
__global__ void __launch_bounds__(kScoreThreads)
    quest_score_kernel(const QuestArgs a) {
  extern __shared__ float sq[];   // [G][D] fp32 query rows of this kv head
  const int tid = threadIdx.x;
  const int blocks_per_head = (a.n_pages + kScoreThreads - 1) / kScoreThreads;
  const int pb = blockIdx.x % blocks_per_head;
  const int g = (blockIdx.x / blocks_per_head) % a.hkv;
  const int bb = blockIdx.x / (blocks_per_head * a.hkv);
  const int group = a.hq / a.hkv;
  griddep_wait();
  griddep_launch_dependents();
  for (int i = tid; i < group * D; i += kScoreThreads) {
    const int h = g * group + i / D;
    sq[i] = __bfloat162float(a.q[((long long)bb * a.hq + h) * D + i % D]);
  }
  __syncthreads();
  const int p = pb * kScoreThreads + tid;
  if (p >= a.n_pages) return;
  const __nv_bfloat16* st =
      a.stats_in + (((long long)bb * a.hkv + g) * a.n_pages + p) * 2 * D;
  for (int h0 = 0; h0 < group; h0 += kHeadChunk) {
    const int nh = min(kHeadChunk, group - h0);
    float acc[kHeadChunk];
#pragma unroll
    for (int h = 0; h < kHeadChunk; ++h) acc[h] = 0.f;
    for (int c0 = 0; c0 < D; c0 += 8) {
      const uint4 umn = __ldg(reinterpret_cast<const uint4*>(st + c0));
      const uint4 umx = __ldg(reinterpret_cast<const uint4*>(st + D + c0));
      __nv_bfloat16 vmn[8], vmx[8];
      memcpy(vmn, &umn, 16);
      memcpy(vmx, &umx, 16);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float fmn = __bfloat162float(vmn[c]), fmx = __bfloat162float(vmx[c]);
#pragma unroll
        for (int h = 0; h < kHeadChunk; ++h) {
          if (h < nh) {
            const float qc = sq[(h0 + h) * D + c0 + c];
            acc[h] = fmaf(qc, qc >= 0.f ? fmx : fmn, acc[h]);
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < kHeadChunk; ++h)
      if (h < nh)
        a.scores[(((long long)bb * a.hq + g * group + h0 + h) * a.n_pages) + p] = acc[h];
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
  const int bph = (a.n_pages + kScoreThreads - 1) / kScoreThreads;
  const long long grid = (long long)a.b * a.hkv * bph;
  const int smem = (a.hq / a.hkv) * D * 4;
  cudaError_t e = cudaFuncSetAttribute(quest_score_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(quest_score_kernel<D>, dim3((unsigned)grid), dim3(kScoreThreads), smem,
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
