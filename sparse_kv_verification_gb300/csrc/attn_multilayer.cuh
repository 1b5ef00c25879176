// Sparse verification attention of many layers in one persistent launch
// (Stage 2 of the "dustin-long-context" notes, section 2.2 / Fig. 5, for
// several layers whose queries are all ready; one global index set serves
// every layer and head).
//
// A work item is (layer, sequence b, kv head g, row block): the G*w query
// rows of kv head g against the k selected positions of that layer's cache.
// The L x units items are dealt round-robin to the CTAs (one per SM), so at
// 80 layers x 128 units on 152 SMs every SM gets 67 or 68 whole items and
// nothing is split or merged across CTAs.  Inside a CTA one warp-specialised
// pipeline runs across all its items without draining: the producer
// warpgroup loads each item's query rows (handed to the consumers through a
// q_full / q_empty mbarrier pair), builds the item's offset table from idx
// (each producer warp the entries of the rows it fetches; the consumers are
// still busy with the previous item's tiles in the stages), then streams the
// item's tiles exactly as the per-layer kernel does; the consumers run the same
// math per tile, merge their position slices through a small buffer at each
// item's end and write O and LSE of that layer.  Every mbarrier wait is
// bounded (about one second) and raises a flag on timeout.
#pragma once

#include "attn_streamk.cuh"

namespace dustin {

constexpr int kMlMaxLayers = 128;   // layers per launch (kernel parameters)

struct MlLayer {
  const __nv_bfloat16* q;   // [b][hq][w][d]
  __nv_bfloat16* o;         // [b][hq][w][d]
  float* lse;               // [b][hq][w]
  KvView kv;                // this layer's K/V cache
};

struct AttnMlArgs {
  const int* idx;   // [b][k], shared by every layer
  int layers, b, hq, hkv, w, n, k;
  int group, rows, row_blocks, units, tpu;
  float scale_log2;
  MlLayer layer[kMlMaxLayers];
};

// Device-side check flags of this translation unit.
static __device__ unsigned int g_attn_ml_dev_flags;

template <int D, int MT, bool PAGED>
__global__ void __launch_bounds__(SkCfg<D, MT>::NT, 1)
    verify_attn_ml_kernel(const __grid_constant__ AttnMlArgs a) {
  using C = SkCfg<D, MT>;
  static_assert(C::MAX_TAB >= 2048, "offset table of one item");
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sK = smem + C::OFF_K;
  unsigned char* sV = smem + C::OFF_V;
  float* sMerge = reinterpret_cast<float*>(smem + C::OFF_MERGE);
  long long* tab = reinterpret_cast<long long*>(smem + C::OFF_TAB);
  unsigned long long* sMask64 =
      reinterpret_cast<unsigned long long*>(smem + C::OFF_MASK);
  const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  const uint32_t q_full = bar0 + 8u * (2 * C::STAGES);
  const uint32_t q_empty = q_full + 8u;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const long long n_items = (long long)a.layers * a.units;

  struct Item {
    int layer, bb, g, rb;
    long long row_base;
  };
  auto item_of = [&](long long it) {
    Item x;
    x.layer = (int)(it / a.units);
    const int u = (int)(it - (long long)x.layer * a.units);
    x.rb = u % a.row_blocks;
    const int ug = u / a.row_blocks;
    x.g = ug % a.hkv;
    x.bb = ug / a.hkv;
    x.row_base = ((long long)x.bb * a.hq + (long long)x.g * a.group) * a.w;
    return x;
  };

  griddep_wait();
  griddep_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), C::NPW * 32 + C::NPW);  // copies + mask arrives
      mbar_init(empty_bar(s), C::NCW);
    }
    mbar_init(q_full, C::NPW * 32);
    mbar_init(q_empty, C::NCW);
    mbar_fence_init();
  }
  __syncthreads();

  if (warp >= C::NCW) {
    // =========================== producer warps ==========================
    if constexpr (C::REBALANCE)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(C::PRODUCER_REGS));
    const int pw = warp - C::NCW;
    const int ptid = tid - C::NCW * 32;
    const int my_row = pw * C::RPW + (lane % C::RPW);
    static_assert(C::RPW <= 32, "one offset per lane");
    constexpr int LPR = 2 * C::CPR;   // lanes per row: K chunks, then V chunks
    constexpr int RPI = 32 / LPR;     // rows per warp instruction
    const int sub = lane / LPR;
    const int l2 = lane % LPR;
    const bool is_v = l2 >= C::CPR;
    const int ch = l2 % C::CPR;
    unsigned char* dst_base = is_v ? sV : sK;
    constexpr int PT = C::NPW * 32;   // producer threads

    int t = 0;   // tile counter over all items (stage, phase)
    int s = 0;   // item counter
    bool ok_run = true;
    for (long long it = blockIdx.x; it < n_items && ok_run; it += gridDim.x, ++s) {
      const Item x = item_of(it);
      const MlLayer& Ld = a.layer[x.layer];
      // Query rows of the item, once the consumers hold the previous ones.
      if (s > 0 && !mbar_wait(q_empty, (s - 1) & 1, kWaitLimitCycles)) {
        if (lane == 0) atomicOr(&g_attn_ml_dev_flags, 4u);
        break;
      }
      for (int c = ptid; c < C::ROWS * C::CPR; c += PT) {
        const int r = c / C::CPR, cc = c % C::CPR;
        const int R = x.rb * C::ROWS + r;
        const bool ok = R < a.rows;
        cp_async_16(smem_u32(sQ + r * C::RS + cc * 16),
                    Ld.q + (ok ? (x.row_base + R) * D + cc * 8 : 0), ok ? 16 : 0);
      }
      cp_async_mbar_arrive(q_full);
      // Offset table of the item.  Warp pw fetches rows RPW pw .. RPW pw +
      // RPW - 1 of every tile, so it builds (and alone reads) exactly those
      // entries: no barrier beyond the warp, and the entries of the previous
      // item are no longer needed once this warp has issued its tiles.
      {
        const int* idx_row = a.idx + (long long)x.bb * a.k;
        constexpr int TPL = 32 / C::RPW;           // tiles per lane step
        constexpr int PER = 2048 / (C::TILE * TPL);  // steps to cover k <= 2048
        const int r_in = lane % C::RPW;
        int jv[PER];
#pragma unroll
        for (int r = 0; r < PER; ++r) {
          const int e = (r * TPL + lane / C::RPW) * C::TILE + pw * C::RPW + r_in;
          jv[r] = e < a.k ? __ldg(idx_row + e) : 0;
        }
        const long long head = (long long)x.g * Ld.kv.sh;
#pragma unroll
        for (int r = 0; r < PER; ++r) {
          const int e = (r * TPL + lane / C::RPW) * C::TILE + pw * C::RPW + r_in;
          if (e >= a.k) continue;
          const int j = jv[r];
          long long off = -1;
          if (j < 0 || j >= a.n) {
            atomicOr(&g_attn_ml_dev_flags, 1u);
          } else if constexpr (PAGED) {
            const int pg = __ldg(Ld.kv.page_table +
                                 (long long)x.bb * Ld.kv.pages_per_seq + j / Ld.kv.page_size);
            if (pg < 0 || pg >= Ld.kv.num_pages)
              atomicOr(&g_attn_ml_dev_flags, 2u);
            else
              off = (long long)pg * Ld.kv.sb + head +
                    (long long)(j % Ld.kv.page_size) * Ld.kv.sn;
          } else {
            off = (long long)x.bb * Ld.kv.sb + head + (long long)j * Ld.kv.sn;
          }
          tab[e] = off;
        }
        __syncwarp();
      }
      const __nv_bfloat16* src_base = is_v ? Ld.kv.v : Ld.kv.k;
      const uint64_t pol = policy_evict_first();   // K/V rows are read once
      // The kv heads of a sequence share idx: start head g at tile
      // g tpu / hkv so that they do not read the same positions together.
      const int rot = DUSTIN_ATTN_ROTATE ? (int)(((long long)x.g * a.tpu) / a.hkv) : 0;
      for (int lt = 0; lt < a.tpu; ++lt, ++t) {
        const int st = t % C::STAGES;
        if (t >= C::STAGES &&
            !mbar_wait(empty_bar(st), ((t / C::STAGES) & 1) ^ 1, kWaitLimitCycles)) {
          if (lane == 0) atomicOr(&g_attn_ml_dev_flags, 4u);
          ok_run = false;
          break;
        }
        int pt = lt + rot;
        pt = pt >= a.tpu ? pt - a.tpu : pt;
        const int i = pt * C::TILE + my_row;
        const long long my_off = i < a.k ? tab[i] : -1;
        const unsigned vm = __ballot_sync(0xffffffffu, my_off >= 0) &
                            (C::RPW == 32 ? 0xffffffffu : ((1u << C::RPW) - 1u));
        unsigned char* dst = dst_base + st * C::TILE_BYTES + ch * 16;
#pragma unroll 8
        for (int q = 0; q < C::RPW / RPI; ++q) {
          const int rr = q * RPI + sub;             // row within this warp's rows
          const long long off = __shfl_sync(0xffffffffu, my_off, rr);
          const bool ok = off >= 0;
          cp_async_16_hint(smem_u32(dst + (pw * C::RPW + rr) * C::RS),
                           src_base + (ok ? off + ch * 8 : 0), ok ? 16 : 0, pol);
        }
        cp_async_mbar_arrive(full_bar(st));
        if (lane == 0) {
          if constexpr (C::RPW == 16)
            reinterpret_cast<unsigned short*>(sMask64 + st)[pw] = (unsigned short)vm;
          else if constexpr (C::RPW == 8)
            reinterpret_cast<unsigned char*>(sMask64 + st)[pw] = (unsigned char)vm;
          else
            reinterpret_cast<unsigned*>(sMask64 + st)[pw] = vm;
          mbar_arrive(full_bar(st));
        }
      }
    }
    // Every copy of this thread lands before the CTA may exit.
    cp_async_wait<0>();
    return;
  }

  // ============================ consumer warps ============================
  if constexpr (C::REBALANCE)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(C::CONSUMER_REGS));
  const int wm = warp / C::WN;
  const int wn = warp % C::WN;
  const int gq = lane >> 2, tq = lane & 3;
  int t = 0;
  bool dead = false;
  auto wait_or_die = [&](uint32_t bar, uint32_t parity) {
    if (dead) return;
    if (!mbar_wait(bar, parity, kWaitLimitCycles)) {
      dead = true;
      if (lane == 0) atomicOr(&g_attn_ml_dev_flags, 4u);
    }
  };

  int s = 0;
  for (long long it = blockIdx.x; it < n_items; it += gridDim.x, ++s) {
    wait_or_die(q_full, s & 1);
    uint32_t qf[C::KS][4];
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      const int r = wm * 16 + (lane & 15);
      const int cc = ks * 2 + (lane >> 4);
      ldmatrix_x4(smem_u32(sQ + r * C::RS + cc * 16), qf[ks][0], qf[ks][1],
                  qf[ks][2], qf[ks][3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(q_empty);

    float oacc[C::DT][4];
#pragma unroll
    for (int i = 0; i < C::DT; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[i][e] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int lt = 0; lt < a.tpu; ++lt, ++t) {
      const int st = t % C::STAGES;
      wait_or_die(full_bar(st), (t / C::STAGES) & 1);
      const unsigned char* tk = sK + st * C::TILE_BYTES;
      const unsigned char* tv = sV + st * C::TILE_BYTES;
      const unsigned long long vmask = sMask64[st];

      // S = Q K^T over this warp's PW positions.
      float sc[C::NT8][4];
#pragma unroll
      for (int j = 0; j < C::NT8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[j][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
#pragma unroll
        for (int j = 0; j < C::NT8; j += 2) {
          const int r = wn * C::PW + j * 8 + ((lane >> 4) << 3) + (lane & 7);
          const int cc = ks * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(smem_u32(tk + r * C::RS + cc * 16), b0, b1, b2, b3);
          mma_bf16(sc[j], qf[ks], b0, b1);
          mma_bf16(sc[j + 1], qf[ks], b2, b3);
        }
      }
      // Rows left out get -inf; the scale (> 0) enters the exponent below.
      if (vmask != ~0ull) {
#pragma unroll
        for (int j = 0; j < C::NT8; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int pos = wn * C::PW + j * 8 + 2 * tq + e;
            const bool ok = (vmask >> pos) & 1ull;
            sc[j][e] = ok ? sc[j][e] : -INFINITY;
            sc[j][e + 2] = ok ? sc[j][e + 2] : -INFINITY;
          }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < C::NT8; ++j) {
        mx0 = fmaxf(mx0, fmaxf(sc[j][0], sc[j][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[j][2], sc[j][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      mx0 *= a.scale_log2;
      mx1 *= a.scale_log2;
      // Lazy rescale (exact): move a row's reference maximum only when the
      // tile's maximum exceeds it by more than 2^kLazyRescale.
      const bool up0 = mx0 > m0 + kLazyRescale, up1 = mx1 > m1 + kLazyRescale;
      if (__any_sync(0xffffffffu, up0 || up1)) {
        const float n0 = up0 ? mx0 : m0, n1 = up1 ? mx1 : m1;
        const float c0 = up0 ? ex2(m0 - n0) : 1.f;
        const float c1 = up1 ? ex2(m1 - n1) : 1.f;
        m0 = n0;
        m1 = n1;
        l0 *= c0;
        l1 *= c1;
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt) {
          oacc[dt][0] *= c0;
          oacc[dt][1] *= c0;
          oacc[dt][2] *= c1;
          oacc[dt][3] *= c1;
        }
      }
      const float u0 = (m0 == -INFINITY) ? 0.f : m0;
      const float u1 = (m1 == -INFINITY) ? 0.f : m1;
      const float cs = a.scale_log2;
#pragma unroll
      for (int j = 0; j < C::NT8; ++j) {
        sc[j][0] = ex2(fmaf(sc[j][0], cs, -u0));
        sc[j][1] = ex2(fmaf(sc[j][1], cs, -u0));
        sc[j][2] = ex2(fmaf(sc[j][2], cs, -u1));
        sc[j][3] = ex2(fmaf(sc[j][3], cs, -u1));
        l0 += sc[j][0] + sc[j][1];
        l1 += sc[j][2] + sc[j][3];
      }
      // O += P V.
#pragma unroll
      for (int kk = 0; kk < C::PW / 16; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
        pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
        pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
        for (int dt = 0; dt < C::DT; dt += 2) {
          const int r = wn * C::PW + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int cc = dt + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(smem_u32(tv + r * C::RS + cc * 16), b0, b1, b2, b3);
          mma_bf16(oacc[dt], pa, b0, b1);
          mma_bf16(oacc[dt + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(st));
    }

    // ---- Item end: row sums over the quad, merge the WN slices through
    // the small buffer (the producers are already streaming the next item).
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if constexpr (C::WN > 1) {
      float* mb = sMerge + wm * 32 * C::MSLOTS + lane;
#pragma unroll 1
      for (int o = 1; o < C::WN; ++o) {
        float a0 = 1.f, a1 = 1.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (wn == o) {
            if (half == 0) {
              mb[0] = m0;
              mb[32] = m1;
              mb[64] = l0;
              mb[96] = l1;
            }
#pragma unroll
            for (int dt = 0; dt < C::DT / 2; ++dt)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                mb[(4 + dt * 4 + e) * 32] = oacc[half * (C::DT / 2) + dt][e];
          }
          named_bar_sync(1, C::NCW * 32);
          if (wn == 0) {
            if (half == 0) {
              const float om0 = mb[0], om1 = mb[32], ol0 = mb[64], ol1 = mb[96];
              const float M0 = fmaxf(m0, om0), M1 = fmaxf(m1, om1);
              const float v0 = (M0 == -INFINITY) ? 0.f : M0;
              const float v1 = (M1 == -INFINITY) ? 0.f : M1;
              a0 = ex2(m0 - v0);
              b0 = ex2(om0 - v0);
              a1 = ex2(m1 - v1);
              b1 = ex2(om1 - v1);
              l0 = l0 * a0 + ol0 * b0;
              l1 = l1 * a1 + ol1 * b1;
              m0 = M0;
              m1 = M1;
            }
#pragma unroll
            for (int dt = 0; dt < C::DT / 2; ++dt) {
              const int d0 = half * (C::DT / 2) + dt;
              oacc[d0][0] = oacc[d0][0] * a0 + mb[(4 + dt * 4 + 0) * 32] * b0;
              oacc[d0][1] = oacc[d0][1] * a0 + mb[(4 + dt * 4 + 1) * 32] * b0;
              oacc[d0][2] = oacc[d0][2] * a1 + mb[(4 + dt * 4 + 2) * 32] * b1;
              oacc[d0][3] = oacc[d0][3] * a1 + mb[(4 + dt * 4 + 3) * 32] * b1;
            }
          }
          named_bar_sync(1, C::NCW * 32);
        }
      }
    }
    if (wn != 0) continue;
    const Item x = item_of(it);
    const MlLayer& Ld = a.layer[x.layer];
    const int RA = x.rb * C::ROWS + wm * 16 + gq, RB = RA + 8;
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f;
    const float i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt) {
      const int col = dt * 8 + 2 * tq;
      if (RA < a.rows)
        *reinterpret_cast<uint32_t*>(Ld.o + (x.row_base + RA) * D + col) =
            pack_bf16(oacc[dt][0] * i0, oacc[dt][1] * i0);
      if (RB < a.rows)
        *reinterpret_cast<uint32_t*>(Ld.o + (x.row_base + RB) * D + col) =
            pack_bf16(oacc[dt][2] * i1, oacc[dt][3] * i1);
    }
    if (tq == 0) {
      if (RA < a.rows)
        Ld.lse[x.row_base + RA] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
      if (RB < a.rows)
        Ld.lse[x.row_base + RB] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
    }
  }
}

}  // namespace dustin
