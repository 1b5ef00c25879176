// Host-side declarations shared by the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "device_common.cuh"

struct dustin_kv;

namespace dustin {

// ---- scoring
constexpr int kMaxPairs = 64;

struct ScorePair {
  KvView kv;
  int kv_head;
};

struct ScoreArgs {
  const __nv_bfloat16* q;  // [n_pairs][b][rows][d]
  float* s_out;            // [b][n]
  float* logits;           // workspace [n_pairs][rows][b][n], log2 units
  float2* stats;           // workspace [n_pairs][rows][b][nchunks]
  int b, n, n_pairs, rows;
  int chunk, nchunks;
  float scale_log2;
  int keys_shared;         // two pairs read the same keys (same cache, kv head)
  ScorePair pairs[kMaxPairs];
};

int score_chunk();
int check_score_args(int b, int n, int d, int n_pairs, int rows, const void* q,
                     const ::dustin_kv* kv, const int32_t* kv_head, float scale,
                     const float* s_out, const char* what, bool* paged, bool* empty);
cudaError_t launch_score(const ScoreArgs& a, int d, bool paged, cudaStream_t st);
cudaError_t take_score_flags(unsigned* flags);

// ---- Quest page scoring (baseline selector)
struct QuestArgs {
  KvView kv;                     // keys (stats pass)
  __nv_bfloat16* stats;          // [b][hkv][P][2][d] out (stats pass)
  const __nv_bfloat16* stats_in; // the same, in (score pass)
  const __nv_bfloat16* q;        // [b][hq][d] (score pass)
  float* scores;                 // [b][hq][P] (score pass)
  int b, hq, hkv, n, page, n_pages;
};
cudaError_t launch_quest_stats(const QuestArgs& a, int d, bool paged, cudaStream_t st);
cudaError_t launch_quest_scores(const QuestArgs& a, int d, cudaStream_t st);
cudaError_t take_quest_flags(unsigned* flags);

// ---- selection
struct SelectArgs {
  const float* sd;
  const float* st;
  int32_t* idx;
  double alpha;
  int b, n, k, n_sink, n_recent, m, norm;
};
constexpr int kSelectMaxN = 1 << 20;
cudaError_t launch_select(const SelectArgs& a, cudaStream_t st);

// ---- verification attention (AttnArgs in attn.cuh, AttnSkArgs in
// attn_streamk.cuh)
struct AttnArgs;
struct AttnSkArgs;
cudaError_t launch_attn_sparse(const AttnArgs& a, int d, int mt, bool paged,
                               cudaStream_t st);
cudaError_t launch_attn_dense(const AttnSkArgs& a, int d, int mt, bool paged,
                              cudaStream_t st);
struct AttnMlArgs;
cudaError_t launch_attn_ml(const AttnMlArgs& a, int d, int mt, bool paged, int grid,
                           cudaStream_t st);
cudaError_t take_attn_ml_flags(unsigned* flags);
int occupancy_attn_sparse(int d, int mt);
int occupancy_attn_dense(int d, int mt);
cudaError_t take_attn_sparse_flags(unsigned* flags);
cudaError_t take_attn_dense_flags(unsigned* flags);

// ---- bookkeeping (api.cu)
void note_launches(int count);
int record_error(int status, const char* message);  // sets dustin_last_error()

}  // namespace dustin
