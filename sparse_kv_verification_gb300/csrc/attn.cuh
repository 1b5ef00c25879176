// Verification attention for Dustin's Stage 2 (sparse verification over the
// selected KV; "dustin-long-context" notes section 2.2, Fig. 5) and the
// full-cache baseline (notes section 3, Fig. 7).
//
// One CTA handles one (sequence b, kv head g, row block, split): the G*w
// query rows that share kv head g (query heads g*G .. g*G+G-1, w window
// rows each: a contiguous [G*w][d] block of q) against a contiguous range
// of the unit's positions.  Positions are idx[b][i] (sparse) or i (dense).
//
// Pipeline: K and V rows of 64-position tiles are gathered with 16-byte
// cp.async into XOR-swizzled shared memory, STAGES tiles deep.  Warp
// (wm, wn) owns query rows [16 wm, 16 wm + 16) and a 64/WN-position slice of
// every tile: S = Q K^T and O += P V run on bf16 mma.sync m16n8k16 with
// fp32 accumulators, with an online (base-2) softmax in registers.  At the
// end the WN slices are merged through shared memory; a single split writes
// O (bf16) and LSE directly, several splits write fp32 partials that
// attn_combine_kernel merges.
#pragma once

#include "device_common.cuh"

namespace dustin {

struct AttnArgs {
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;
  KvView kv;
  const int* idx;   // [b][npos] (sparse) or nullptr (dense)
  int b, hq, hkv, w, n;
  int npos;         // positions per (b, kv head): k or n
  int group;        // hq / hkv
  int rows;         // group * w
  int row_blocks;   // ceil(rows / (16 * MT))
  int splits;
  int chunk;        // positions per split (multiple of 64)
  float scale_log2; // scale * log2(e)
  float* ws_o;      // [blocks][splits][16 MT][D] (splits > 1)
  float2* ws_ml;    // [blocks][splits][16 MT]    (m in log2 units, l)
};

template <int D, int MT>
struct AttnCfg {
  static constexpr int WN = (MT == 1) ? 4 : 2;
  static constexpr int NWARP = MT * WN;
  static constexpr int NT = NWARP * 32;
  static constexpr int TILE = 64;
  static constexpr int PW = TILE / WN;   // positions per warp per tile
  static constexpr int NT8 = PW / 8;     // n8 tiles of S per warp
  static constexpr int KS = D / 16;      // k16 steps over d
  static constexpr int DT = D / 8;       // n8 tiles of O over d
  static constexpr int CPR = D / 8;      // 16-byte chunks per row
  static constexpr int ROWS = 16 * MT;
  static constexpr int STAGES = 4;
  static constexpr int TILE_BYTES = TILE * D * 2;
  static constexpr int Q_BYTES = ROWS * D * 2;
  static constexpr int MAX_TAB = 2048;   // offset-table entries
  static constexpr int SMEM = Q_BYTES + 2 * STAGES * TILE_BYTES + MAX_TAB * 8;
  static constexpr int MERGE_FLOATS = (WN - 1) * MT * 32 * (DT * 4 + 4);
  static_assert(MERGE_FLOATS * 4 <= STAGES * TILE_BYTES, "merge buffer");
};

// Device-side check flags of this translation unit.
static __device__ unsigned int g_attn_dev_flags;

template <int D, int MT, bool PAGED, bool DENSE>
__global__ void __launch_bounds__(AttnCfg<D, MT>::NT, 1)
    verify_attn_kernel(const AttnArgs a) {
  using C = AttnCfg<D, MT>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sK = sQ + C::Q_BYTES;
  unsigned char* sV = sK + C::STAGES * C::TILE_BYTES;
  long long* tab = reinterpret_cast<long long*>(sV + C::STAGES * C::TILE_BYTES);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int wm = warp / C::WN;
  const int wn = warp % C::WN;

  // Block -> (b, kv head, row block, split).
  int blk = blockIdx.x;
  const int split = blk % a.splits;
  blk /= a.splits;
  const int rb = blk % a.row_blocks;
  const int unit = blk / a.row_blocks;
  const int g = unit % a.hkv;
  const int bb = unit / a.hkv;

  const int p_begin = split * a.chunk;
  const int p_end = min(a.npos, p_begin + a.chunk);
  const int len = max(0, p_end - p_begin);
  const int ntiles = (len + C::TILE - 1) / C::TILE;

  const long long unit_off = (long long)bb * a.kv.sb + (long long)g * a.kv.sh;
  const long long row_base =
      ((long long)bb * a.hq + (long long)g * a.group) * a.w;  // first q row
  const int r_lo = rb * C::ROWS;                               // first row here

  // ---- Q rows into shared memory (zero rows past G*w).
  for (int c = tid; c < C::ROWS * C::CPR; c += C::NT) {
    const int r = c / C::CPR, ch = c % C::CPR;
    const int R = r_lo + r;
    const bool ok = R < a.rows;
    const __nv_bfloat16* src = a.q + (ok ? (row_base + R) * D + ch * 8 : 0);
    cp_async_16(smem_u32(sQ + swz<D>(r, ch)), src, ok ? 16 : 0);
  }
  cp_async_commit();

  // ---- Offset table: element offset of each position's K/V row (sparse),
  // or of each page (dense, paged).  -1 marks a position that failed a check.
  if constexpr (!DENSE) {
    for (int i = tid; i < len; i += C::NT) {
      const int j = __ldg(a.idx + (long long)bb * a.npos + p_begin + i);
      long long off = -1;
      if (j < 0 || j >= a.n) {
        atomicOr(&g_attn_dev_flags, 1u);
      } else if constexpr (PAGED) {
        const int pg = __ldg(a.kv.page_table + (long long)bb * a.kv.pages_per_seq +
                             j / a.kv.page_size);
        if (pg < 0 || pg >= a.kv.num_pages) {
          atomicOr(&g_attn_dev_flags, 2u);
        } else {
          off = (long long)pg * a.kv.sb + (long long)g * a.kv.sh +
                (long long)(j % a.kv.page_size) * a.kv.sn;
        }
      } else {
        off = unit_off + (long long)j * a.kv.sn;
      }
      tab[i] = off;
    }
  } else if constexpr (PAGED) {
    const int pg0 = p_begin / a.kv.page_size;
    const int npg = len > 0 ? (p_end - 1) / a.kv.page_size - pg0 + 1 : 0;
    for (int i = tid; i < npg; i += C::NT) {
      const int pg = __ldg(a.kv.page_table + (long long)bb * a.kv.pages_per_seq +
                           pg0 + i);
      long long off = -1;
      if (pg < 0 || pg >= a.kv.num_pages) {
        atomicOr(&g_attn_dev_flags, 2u);
      } else {
        off = (long long)pg * a.kv.sb + (long long)g * a.kv.sh;
      }
      tab[i] = off;
    }
  }
  __syncthreads();

  auto row_offset = [&](int i) -> long long {
    if constexpr (!DENSE) {
      return tab[i];
    } else if constexpr (PAGED) {
      const int j = p_begin + i;
      const long long base = tab[j / a.kv.page_size - p_begin / a.kv.page_size];
      return base < 0 ? -1 : base + (long long)(j % a.kv.page_size) * a.kv.sn;
    } else {
      return unit_off + (long long)(p_begin + i) * a.kv.sn;
    }
  };

  auto issue_tile = [&](int t) {
    if (t < ntiles) {
      const int stage = t % C::STAGES;
      const uint32_t dk = smem_u32(sK + stage * C::TILE_BYTES);
      const uint32_t dv = smem_u32(sV + stage * C::TILE_BYTES);
      for (int c = tid; c < C::TILE * C::CPR; c += C::NT) {
        const int r = c / C::CPR, ch = c % C::CPR;
        const int i = t * C::TILE + r;
        long long off = (i < len) ? row_offset(i) : -1;
        const bool ok = off >= 0;
        const long long e = ok ? off + ch * 8 : 0;
        cp_async_16(dk + swz<D>(r, ch), a.kv.k + e, ok ? 16 : 0);
        cp_async_16(dv + swz<D>(r, ch), a.kv.v + e, ok ? 16 : 0);
      }
    }
    cp_async_commit();
  };

  for (int t = 0; t < C::STAGES - 1; ++t) issue_tile(t);

  // ---- Q fragments (A operand) into registers.
  cp_async_wait<C::STAGES - 1>();  // the Q group is the oldest
  __syncthreads();
  uint32_t qf[C::KS][4];
#pragma unroll
  for (int ks = 0; ks < C::KS; ++ks) {
    const int r = wm * 16 + (lane & 15);
    const int ch = ks * 2 + (lane >> 4);
    ldmatrix_x4(smem_u32(sQ + swz<D>(r, ch)), qf[ks][0], qf[ks][1], qf[ks][2],
                qf[ks][3]);
  }

  float oacc[C::DT][4];
#pragma unroll
  for (int i = 0; i < C::DT; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[i][e] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  const int gq = lane >> 2, tq = lane & 3;

  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<C::STAGES - 2>();
    __syncthreads();
    issue_tile(t + C::STAGES - 1);

    const int stage = t % C::STAGES;
    const unsigned char* tk = sK + stage * C::TILE_BYTES;
    const unsigned char* tv = sV + stage * C::TILE_BYTES;

    // S = Q K^T over this warp's PW positions.
    float s[C::NT8][4];
#pragma unroll
    for (int j = 0; j < C::NT8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
#pragma unroll
      for (int j = 0; j < C::NT8; j += 2) {
        const int r = wn * C::PW + j * 8 + ((lane >> 4) << 3) + (lane & 7);
        const int ch = ks * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(smem_u32(tk + swz<D>(r, ch)), b0, b1, b2, b3);
        mma_bf16(s[j], qf[ks], b0, b1);
        mma_bf16(s[j + 1], qf[ks], b2, b3);
      }
    }

    // Scale into log2 units, mask positions past the range or failed checks.
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < C::NT8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = t * C::TILE + wn * C::PW + j * 8 + 2 * tq + e;
        bool ok = i < len;
        if constexpr (!DENSE) ok = ok && tab[i] >= 0;
        if constexpr (DENSE && PAGED) ok = ok && row_offset(i) >= 0;
        s[j][e] = ok ? s[j][e] * a.scale_log2 : -INFINITY;
        s[j][e + 2] = ok ? s[j][e + 2] * a.scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, s[j][e]);
        mx1 = fmaxf(mx1, s[j][e + 2]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float u0 = (n0 == -INFINITY) ? 0.f : n0;   // subtrahend
    const float u1 = (n1 == -INFINITY) ? 0.f : n1;
    const float c0 = ex2(m0 - u0), c1 = ex2(m1 - u1);
    m0 = n0;
    m1 = n1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int j = 0; j < C::NT8; ++j) {
      s[j][0] = ex2(s[j][0] - u0);
      s[j][1] = ex2(s[j][1] - u0);
      s[j][2] = ex2(s[j][2] - u1);
      s[j][3] = ex2(s[j][3] - u1);
      ps0 += s[j][0] + s[j][1];
      ps1 += s[j][2] + s[j][3];
    }
    l0 = l0 * c0 + ps0;
    l1 = l1 * c1 + ps1;
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt) {
      oacc[dt][0] *= c0;
      oacc[dt][1] *= c0;
      oacc[dt][2] *= c1;
      oacc[dt][3] *= c1;
    }

    // O += P V.
#pragma unroll
    for (int kk = 0; kk < C::PW / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dt = 0; dt < C::DT; dt += 2) {
        const int r = wn * C::PW + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int ch = dt + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(smem_u32(tv + swz<D>(r, ch)), b0, b1, b2, b3);
        mma_bf16(oacc[dt], pa, b0, b1);
        mma_bf16(oacc[dt + 1], pa, b2, b3);
      }
    }
  }

  // ---- Row sums over the quad, then merge the WN position slices.
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  cp_async_wait<0>();
  __syncthreads();
  if constexpr (C::WN > 1) {
    float* mb = reinterpret_cast<float*>(sK);
    constexpr int SLOTS = C::DT * 4 + 4;
    if (wn > 0) {
      float* p = mb + ((wn - 1) * MT + wm) * 32 * SLOTS + lane;
      p[0] = m0;
      p[32] = m1;
      p[64] = l0;
      p[96] = l1;
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) p[(4 + dt * 4 + e) * 32] = oacc[dt][e];
    }
    __syncthreads();
    if (wn == 0) {
#pragma unroll 1
      for (int o = 1; o < C::WN; ++o) {
        const float* p = mb + ((o - 1) * MT + wm) * 32 * SLOTS + lane;
        const float om0 = p[0], om1 = p[32], ol0 = p[64], ol1 = p[96];
        const float M0 = fmaxf(m0, om0), M1 = fmaxf(m1, om1);
        const float v0 = (M0 == -INFINITY) ? 0.f : M0;
        const float v1 = (M1 == -INFINITY) ? 0.f : M1;
        const float a0 = ex2(m0 - v0), b0 = ex2(om0 - v0);
        const float a1 = ex2(m1 - v1), b1 = ex2(om1 - v1);
        l0 = l0 * a0 + ol0 * b0;
        l1 = l1 * a1 + ol1 * b1;
        m0 = M0;
        m1 = M1;
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt) {
          oacc[dt][0] = oacc[dt][0] * a0 + p[(4 + dt * 4 + 0) * 32] * b0;
          oacc[dt][1] = oacc[dt][1] * a0 + p[(4 + dt * 4 + 1) * 32] * b0;
          oacc[dt][2] = oacc[dt][2] * a1 + p[(4 + dt * 4 + 2) * 32] * b1;
          oacc[dt][3] = oacc[dt][3] * a1 + p[(4 + dt * 4 + 3) * 32] * b1;
        }
      }
    }
  }
  if (wn != 0) return;

  // ---- Write: rows r = 16 wm + gq (+8) of this row block.
  const int rA = wm * 16 + gq, rB = rA + 8;
  const int RA = r_lo + rA, RB = r_lo + rB;
  if (a.splits == 1) {
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f;
    const float i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt) {
      const int col = dt * 8 + 2 * tq;
      if (RA < a.rows)
        *reinterpret_cast<uint32_t*>(a.o + (row_base + RA) * D + col) =
            pack_bf16(oacc[dt][0] * i0, oacc[dt][1] * i0);
      if (RB < a.rows)
        *reinterpret_cast<uint32_t*>(a.o + (row_base + RB) * D + col) =
            pack_bf16(oacc[dt][2] * i1, oacc[dt][3] * i1);
    }
    if (tq == 0) {
      if (RA < a.rows)
        a.lse[row_base + RA] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
      if (RB < a.rows)
        a.lse[row_base + RB] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
    }
  } else {
    const long long pb = ((long long)blockIdx.x) * C::ROWS;  // (blk, split)
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt) {
      const int col = dt * 8 + 2 * tq;
      *reinterpret_cast<float2*>(a.ws_o + (pb + rA) * D + col) =
          make_float2(oacc[dt][0], oacc[dt][1]);
      *reinterpret_cast<float2*>(a.ws_o + (pb + rB) * D + col) =
          make_float2(oacc[dt][2], oacc[dt][3]);
    }
    if (tq == 0) {
      a.ws_ml[pb + rA] = make_float2(m0, l0);
      a.ws_ml[pb + rB] = make_float2(m1, l1);
    }
  }
}

// Merge split partials: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,
// LSE = (M + log2 sum_s 2^(m_s - M) l_s) ln 2.  One warp per query row.
template <int D, int MT>
__global__ void __launch_bounds__(256)
    attn_combine_kernel(const AttnArgs a) {
  using C = AttnCfg<D, MT>;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int nblk = a.b * a.hkv * a.row_blocks;
  if (warp >= nblk * C::ROWS) return;
  const int r = warp % C::ROWS;
  const int blk = warp / C::ROWS;
  const int rb = blk % a.row_blocks;
  const int unit = blk / a.row_blocks;
  const int g = unit % a.hkv;
  const int bb = unit / a.hkv;
  const int R = rb * C::ROWS + r;
  if (R >= a.rows) return;
  const long long row = ((long long)bb * a.hq + (long long)g * a.group) * a.w + R;

  float M = -INFINITY;
  for (int s = 0; s < a.splits; ++s)
    M = fmaxf(M, a.ws_ml[((long long)blk * a.splits + s) * C::ROWS + r].x);
  const float u = (M == -INFINITY) ? 0.f : M;
  constexpr int E = D / 32;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int s = 0; s < a.splits; ++s) {
    const long long pr = ((long long)blk * a.splits + s) * C::ROWS + r;
    const float2 ml = a.ws_ml[pr];
    const float f = ex2(ml.x - u);
    wsum += f * ml.y;
    const float* po = a.ws_o + pr * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] += f * po[e];
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    *reinterpret_cast<uint32_t*>(a.o + row * D + lane * E + e) =
        pack_bf16(acc[e] * inv, acc[e + 1] * inv);
  if (lane == 0) a.lse[row] = wsum > 0.f ? (M + log2f(wsum)) * kLn2 : -INFINITY;
}

}  // namespace dustin
