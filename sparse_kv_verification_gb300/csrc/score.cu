// Importance scoring on the scored (layer, head) pairs: S_Target and
// S_Draft of the "dustin-long-context" notes, section 2.2 (attention summed
// over heads, layers and query rows), restricted to a few heads as in
// section 2.4 / Fig. 6.
//
//   S[b][j] = sum_p sum_r softmax_j(scale * q[p][b][r] . K_p[b][g_p][j])
//
// Two passes.  Pass 1 (score_logits_kernel): one CTA per (pair, sequence,
// 2048-position chunk) streams the chunk's key rows through a 4-stage
// cp.async pipeline into swizzled shared memory, computes the rows' logits
// with bf16 mma.sync (fp32 accumulate), writes them (log2 units) to the
// workspace and keeps an online (max, sum of 2^(l - max)) per row.
// Pass 2 (score_reduce_kernel): combines the chunk statistics into each
// row's log2-sum-exp and writes S[b][j] = sum_{p,r} 2^(l - lse2), summed
// in a fixed order (pair-major, then row) in fp32.
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

__global__ void __launch_bounds__(256) score_reduce_kernel(const ScoreArgs a) {
  __shared__ float lse2[1024];
  const int bb = blockIdx.y;
  const int prs = a.n_pairs * a.rows;
  griddep_wait();
  griddep_launch_dependents();
  for (int i = threadIdx.x; i < prs; i += blockDim.x) {
    const float2* st = a.stats + ((long long)i * a.b + bb) * a.nchunks;
    float M = -INFINITY;
    for (int c = 0; c < a.nchunks; ++c) M = fmaxf(M, st[c].x);
    const float u = M == -INFINITY ? 0.f : M;
    float Z = 0.f;
    for (int c = 0; c < a.nchunks; ++c) Z += st[c].y * ex2(st[c].x - u);
    // An all-masked row contributes nothing.
    lse2[i] = Z > 0.f ? u + log2f(Z) : INFINITY;
  }
  __syncthreads();
  const long long base = (long long)blockIdx.x * 1024;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const long long j = base + q * 256 + threadIdx.x;
    if (j >= a.n) continue;
    float acc = 0.f;
    for (int i = 0; i < prs; ++i)
      acc += ex2(a.logits[((long long)i * a.b + bb) * a.n + j] - lse2[i]);
    a.s_out[(long long)bb * a.n + j] = acc;
  }
}

template <int D, bool PAGED>
cudaError_t run_score(const ScoreArgs& a, cudaStream_t st) {
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

int score_chunk() { return 2048; }

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

std::atomic<void*> g_noalloc_ptr[64];
std::mutex g_noalloc_mutex;

// Device address of the array on the current device, looked up once per
// device (with that device current).  In host code the array's name is only
// a host-side stand-in, so the kernels always get this address.
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return e;
      g_noalloc_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace dustin

extern "C" int dustin_score_heads_noalloc(int b, int n, int d, int n_pairs,
                                          int rows, const void* q,
                                          const dustin_kv* kv,
                                          const int32_t* kv_head, float scale,
                                          float* s_out, void* stream) {
  using namespace dustin;
  const size_t need = dustin_score_heads_workspace_size(b, n, n_pairs, rows);
  if (need > (size_t)DUSTIN_NOALLOC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "dustin_score_heads_noalloc: this call needs %zu bytes of scratch; "
             "the built-in array holds %zu (use dustin_score_heads with a "
             "workspace)",
             need, (size_t)DUSTIN_NOALLOC_SCRATCH_BYTES);
    return record_error(DUSTIN_ERR_WORKSPACE, msg);
  }
  if (need == 0)  // empty or invalid sizes: the checks of the main entry point
    return dustin_score_heads(b, n, d, n_pairs, rows, q, kv, kv_head, scale,
                              s_out, nullptr, 0, stream);
  void* ws = nullptr;
  cudaError_t e = noalloc_scratch(&ws);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "dustin_score_heads_noalloc: cudaGetSymbolAddress: %s",
             cudaGetErrorString(e));
    return record_error(DUSTIN_ERR_CUDA, msg);
  }
  return dustin_score_heads(b, n, d, n_pairs, rows, q, kv, kv_head, scale,
                            s_out, ws, (size_t)DUSTIN_NOALLOC_SCRATCH_BYTES,
                            stream);
}
