// Full-cache verification attention: the dense in-run baseline (the "Full
// Cache" bar of the "dustin-long-context" notes, section 3, Fig. 7), every
// query row of the window against every cached position.
//
// Work units are (sequence b, kv head g, row block): the G*w query rows that
// share kv head g (query heads g*G .. g*G+G-1, w window rows each: one
// contiguous [G*w][d] block of q) against the unit's n positions, cut into
// 64-position tiles.  A dense unit is long (512 tiles at n = 32768) and the
// units rarely fill the SMs evenly (128 units on 152 SMs at the 72B shape),
// so the tiles are shared out stream-K style:
//
// the units' tiles are laid end to end and CTA c takes the contiguous range
// [c*T/G, (c+1)*T/G) of the T tiles, G being the number of CTAs resident at
// once, so every SM gets the same number of tiles.  A CTA walks its range
// as segments, one per unit it touches.  A segment that covers its whole
// unit writes O and LSE directly.  A unit split between CTAs: each of its
// segments leaves a partial (O unnormalised, max, sum) in workspace slot
// 2c + 1 (the segment that starts the unit) or 2c (any other segment; a CTA
// owns at most one of each), then counts itself on the unit's counter; the
// CTA that completes the count merges the partials, in CTA order, and writes
// the unit.  No CTA ever waits for another.  The counter word holds
// (call epoch << 24 | count): a word from another call, or garbage, reads as
// zero, and the merging CTA resets the word, so the workspace needs no
// initialisation and a replayed launch starts from zero.
//
// Inside a CTA, the warp-specialised pipeline of the sparse kernel (same
// tiles, shared-memory layout and math): a producer warpgroup streams each
// tile's K and V rows with 16-byte cp.async into padded rows (contiguous
// rows here; a paged cache goes through a per-CTA table of page offsets, one
// entry per 16 positions, since pages hold a multiple of 16 positions), and
// MT*WN consumer warps run S = Q K^T and O += P V on bf16 mma.sync with an
// online base-2 softmax and a lazy reference maximum.  The producers also
// load each later segment's query rows, handing them over through a
// q_full / q_empty mbarrier pair.  At a segment's end the WN position slices
// are merged: through the K stages at the range's last segment (nothing is
// in flight any more), otherwise through a small buffer of their own, one
// partner and half of d at a time.  With 16 warps the producers hand
// registers to the consumers with setmaxnreg (64 / 144 of a 128-register
// launch).  Every mbarrier wait is bounded (about one second): after a
// timeout a warp stops waiting but keeps the same barrier sequence, raises
// a flag, and the call's outputs are void.
#pragma once

#include "device_common.cuh"

namespace dustin {

struct AttnSkArgs {
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;
  KvView kv;
  int b, hq, hkv, w, n;
  int group;        // hq / hkv
  int rows;         // group * w
  int row_blocks;   // ceil(rows / (16 * MT))
  int units;        // b * hkv * row_blocks
  int tph;          // history tiles per unit: ceil(n / 64)
  int tpu;          // tiles per unit: max(1, tph + has_win)
  int grid;         // CTAs (G)
  float scale_log2; // scale * log2(e)
  int kv_ready;     // the page table and K/V may be read before the wait
  KvView win;       // the window's own K/V [b][hkv][w][d] (has_win)
  int has_win;      // a unit's last tile is its window tile (causal;
                    // selects the WIN instance of the kernel)
  float* ws_o;      // [2 G][16 MT][D] partial O   (when some unit is split)
  float2* ws_ml;    // [2 G][16 MT] (m in log2 units, l)
  unsigned long long* counters;  // [units] (epoch << 24 | count)
  unsigned long long epoch;      // 40-bit, nonzero, distinct per call
};

// Build-time tunables (nvcc -D): producer warps (4 or 8), pipeline depth
// for d = 128, and split accumulators for S = Q K^T (two half-depth chains
// per n8 tile instead of one, for instruction-level parallelism).
#ifndef DUSTIN_ATTN_NPW
#define DUSTIN_ATTN_NPW 4
#endif
#ifndef DUSTIN_ATTN_STAGES128
#define DUSTIN_ATTN_STAGES128 5
#endif
// Registers of a producer thread when the consumers take the rest.
#ifndef DUSTIN_ATTN_PRODUCER_REGS
#define DUSTIN_ATTN_PRODUCER_REGS 64
#endif
// Rotate each unit's tile order by its kv head (see the kernel).
#ifndef DUSTIN_ATTN_ROTATE
#define DUSTIN_ATTN_ROTATE 1
#endif

template <int D, int MT>
struct SkCfg {
  static constexpr int WN = (MT == 4) ? 2 : 4;
  static constexpr int NCW = MT * WN;            // consumer warps
  static constexpr int NPW = DUSTIN_ATTN_NPW;    // producer warps
  static_assert(NPW == 4 || NPW == 8, "producer warps: whole warpgroups");
  static constexpr int NT = (NCW + NPW) * 32;
  static constexpr int RPW = 64 / NPW;           // tile rows per producer warp
  // Above 384 threads the register file is tight: the producer warpgroups
  // drop to 64 registers and the consumer warpgroups take the rest, e.g.
  // 16 warps (128 at launch): 64*128 + 144*384 <= 128*512.
  static constexpr bool REBALANCE = (NT > 384);
  static constexpr int PRODUCER_REGS = DUSTIN_ATTN_PRODUCER_REGS;
  static constexpr int LAUNCH_REGS = (65536 / NT) & ~7;
  static constexpr int CONSUMER_REGS =
      ((LAUNCH_REGS * NT - PRODUCER_REGS * NPW * 32) / (NCW * 32)) & ~7;
  static constexpr int TILE = 64;
  static constexpr int PW = TILE / WN;           // positions per warp per tile
  static constexpr int NT8 = PW / 8;             // n8 tiles of S per warp
  static constexpr int KS = D / 16;              // k16 steps over d
  static constexpr int DT = D / 8;               // n8 tiles of O over d
  static constexpr int CPR = D / 8;              // 16-byte chunks per row
  static constexpr int ROWS = 16 * MT;
  static constexpr int RS = D * 2 + 16;          // padded row stride, bytes
  static constexpr int STAGES = (D == 128) ? DUSTIN_ATTN_STAGES128 : 8;
  static constexpr int TILE_BYTES = TILE * RS;
  static constexpr int Q_BYTES = ROWS * RS;
  static constexpr int MAX_TAB = 2048;           // offset-table entries
  // Tiles one CTA may own: one page-table entry per 16-row group.
  static constexpr int MAX_TILES = MAX_TAB / (TILE / 16);
  static constexpr int MSLOTS = DT * 2 + 4;      // merge slots: half of O + m, l
  static constexpr int MERGE_FLOATS = MT * 32 * MSLOTS;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * TILE_BYTES;
  static constexpr int OFF_MERGE = OFF_V + STAGES * TILE_BYTES;
  static constexpr int OFF_TAB = OFF_MERGE + MERGE_FLOATS * 4;
  static constexpr int OFF_MASK = OFF_TAB + MAX_TAB * 8;
  static constexpr int OFF_BAR = OFF_MASK + STAGES * 8;  // 64-bit mask / stage
  static constexpr int NBARS = 2 * STAGES + 2;  // full, empty, q_full, q_empty
  static constexpr int OFF_FLAG = OFF_BAR + NBARS * 8;
  static constexpr int SMEM = OFF_FLAG + 32;   // flag, then [T0, T1)
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Device-side check flags of this translation unit.
static __device__ unsigned int g_attn_sk_dev_flags;


// First tile of CTA c's range, and the CTA whose range holds tile x: the
// largest c with floor(c T / G) <= x, i.e. floor(((x + 1) G - 1) / T).
__host__ __device__ inline long long sk_begin(long long c, long long T, long long G) {
  return c * T / G;
}
__host__ __device__ inline int sk_owner(long long x, long long T, long long G) {
  return (int)(((x + 1) * G - 1) / T);
}

template <int D, int MT, bool PAGED, bool WIN>
__global__ void __launch_bounds__(SkCfg<D, MT>::NT, 1)
    verify_attn_sk_kernel(const AttnSkArgs a) {
  using C = SkCfg<D, MT>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sK = smem + C::OFF_K;
  unsigned char* sV = smem + C::OFF_V;
  float* sMerge = reinterpret_cast<float*>(smem + C::OFF_MERGE);
  long long* tab = reinterpret_cast<long long*>(smem + C::OFF_TAB);
  unsigned long long* sMask64 =
      reinterpret_cast<unsigned long long*>(smem + C::OFF_MASK);
  int* sFlag = reinterpret_cast<int*>(smem + C::OFF_FLAG);
  volatile long long* sRange = reinterpret_cast<long long*>(smem + C::OFF_FLAG + 16);
  const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  const uint32_t q_full = bar0 + 8u * (2 * C::STAGES);
  const uint32_t q_empty = q_full + 8u;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  const long long T = (long long)a.units * a.tpu;
  const long long T0 = sk_begin(blockIdx.x, T, a.grid);
  const long long T1 = sk_begin(blockIdx.x + 1, T, a.grid);
  const int ntiles = (int)(T1 - T0);
  const int u_first = (int)(T0 / a.tpu);
  const int nseg = ntiles > 0 ? (int)((T1 - 1) / a.tpu) - u_first + 1 : 0;

  struct Unit {
    int bb, g, rb;
    long long kv_off, row_base;
  };
  auto unit_of = [&](int u) {
    Unit x;
    x.rb = u % a.row_blocks;
    const int ug = u / a.row_blocks;
    x.g = ug % a.hkv;
    x.bb = ug / a.hkv;
    x.kv_off = (long long)x.bb * a.kv.sb + (long long)x.g * a.kv.sh;
    x.row_base = ((long long)x.bb * a.hq + (long long)x.g * a.group) * a.w;
    return x;
  };
  // Position tile of a unit's local tile lt.  The kv heads of a sequence
  // share its index set, so without a rotation the CTAs of one sequence
  // would read the same positions of eight K/V slabs a power of two apart
  // at the same moments; starting head g at tile g tpu / hkv spreads them.
  // (History tiles only: lt < tph.)
  auto phys_tile = [&](int lt, int g) {
    if (!DUSTIN_ATTN_ROTATE) return lt;
    const long long gt = (long long)g * a.tph;
    const int t = lt + (gt <= 0x7fffffffLL ? (int)gt / a.hkv : (int)(gt / a.hkv));
    return t >= a.tph ? t - a.tph : t;
  };
  // Unit u and local tile range [lt0, lt1) of segment s.
  // (Reads the range back from shared memory, so that the pipelines do not
  // hold it in registers.)
  auto seg_range = [&](int s, int& u, int& lt0, int& lt1) {
    const long long r0 = sRange[0], r1 = sRange[1];
    u = (int)(r0 / a.tpu) + s;
    const long long ub = (long long)u * a.tpu;
    lt0 = (int)(max(r0, ub) - ub);
    lt1 = (int)(min(r1, ub + a.tpu) - ub);
  };

  // Programmatic dependent launch, as in the sparse kernel: normally every
  // thread waits for the previous kernel first; with kv_ready the page
  // table and the first STAGES tiles are fetched before the wait, and only
  // q (and every write) waits.  A thread triggers the next launch only after
  // its own wait.
  if (!a.kv_ready) {
    griddep_wait();
    griddep_launch_dependents();
  }

  // ---- Query rows of a unit into shared memory (zero past G*w).
  auto load_q = [&](int u, int first, int step) {
    const Unit x = unit_of(u);
    for (int c = first; c < C::ROWS * C::CPR; c += step) {
      const int r = c / C::CPR, ch = c % C::CPR;
      const int R = x.rb * C::ROWS + r;
      const bool ok = R < a.rows;
      cp_async_16(smem_u32(sQ + r * C::RS + ch * 16),
                  a.q + (ok ? (x.row_base + R) * D + ch * 8 : 0), ok ? 16 : 0);
    }
  };
  if (nseg > 0 && !a.kv_ready) load_q(u_first, tid, C::NT);
  cp_async_commit();
  if (tid == 0) {
    sRange[0] = T0;
    sRange[1] = T1;
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), C::NPW * 32 + C::NPW);  // copies + mask arrives
      mbar_init(empty_bar(s), C::NCW);
    }
    mbar_init(q_full, C::NPW * 32);
    mbar_init(q_empty, C::NCW);
    mbar_fence_init();
  }

  // ---- Paged cache: page offsets of every 16-position group of the range
  // (-1: a page that failed its check).  First one thread per tile decodes
  // the tile's sequence, kv head and first position into shared memory (the
  // K stages, unused until the pipeline starts); then every thread loads
  // the page numbers of all its entries before converting them, so that the
  // loads overlap.
  if constexpr (PAGED) {
    constexpr int PER_TILE = C::TILE / 16;
    constexpr int PER_THREAD = (C::MAX_TAB + C::NT - 1) / C::NT;
    int4* tinfo = reinterpret_cast<int4*>(sK);   // {b, g, first position}
    static_assert(C::MAX_TILES * 16 <= C::STAGES * C::TILE_BYTES, "tile info");
    {
      const int u0 = (int)(T0 / a.tpu);
      const int lt_first = (int)(T0 - (long long)u0 * a.tpu);
      for (int tt = tid; tt < ntiles; tt += C::NT) {
        const int x = lt_first + tt;
        const int ug = (u0 + x / a.tpu) / a.row_blocks;
        const int g = ug % a.hkv;
        const int lt = x % a.tpu;   // the window tile has no page entries
        tinfo[tt] = make_int4(ug / a.hkv, g,
                              lt < a.tph ? phys_tile(lt, g) * C::TILE : -(1 << 30), 0);
      }
    }
    __syncthreads();
    const int n_ent = ntiles * PER_TILE;
    int key[PER_THREAD];   // page number
#pragma unroll
    for (int r = 0; r < PER_THREAD; ++r) {
      const int i = tid + r * C::NT;
      key[r] = -1;
      if (i < n_ent) {
        const int4 ti = tinfo[i / PER_TILE];
        const int p = ti.z + (i % PER_TILE) * 16;
        if (p >= 0 && p < a.n)
          key[r] = __ldg(a.kv.page_table + (long long)ti.x * a.kv.pages_per_seq +
                         p / a.kv.page_size);
      }
    }
#pragma unroll
    for (int r = 0; r < PER_THREAD; ++r) {
      const int i = tid + r * C::NT;
      if (i >= n_ent) continue;
      const int4 ti = tinfo[i / PER_TILE];
      const int p = ti.z + (i % PER_TILE) * 16;
      long long off = -1;
      if (p >= 0 && p < a.n) {
        const int pg = key[r];
        if (pg < 0 || pg >= a.kv.num_pages)
          atomicOr(&g_attn_sk_dev_flags, 2u);
        else
          off = (long long)pg * a.kv.sb + (long long)ti.y * a.kv.sh +
                (long long)(p % a.kv.page_size) * a.kv.sn;
      }
      tab[i] = off;
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  if (warp >= C::NCW) {
    // =========================== producer warps ==========================
    // Warp pw fetches rows [RPW pw, RPW pw + RPW) of every tile.  Lane l
    // looks up the offset of row RPW pw + l % RPW (-1: leave the row out);
    // the copies of row rr use lane rr's offset through a shuffle.
    if constexpr (C::REBALANCE)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(C::PRODUCER_REGS));
    const int pw = warp - C::NCW;
    const int my_row = pw * C::RPW + (lane % C::RPW);
    static_assert(C::RPW <= 32, "one offset per lane");
    constexpr int LPR = 2 * C::CPR;   // lanes per row: K chunks, then V chunks
    constexpr int RPI = 32 / LPR;     // rows per warp instruction
    const int sub = lane / LPR;
    const int l2 = lane % LPR;
    const bool is_v = l2 >= C::CPR;
    const int ch = l2 % C::CPR;
    const __nv_bfloat16* src_base = is_v ? a.kv.v : a.kv.k;
    unsigned char* dst_base = is_v ? sV : sK;

    int t = 0;   // tile counter over the whole range (stage, phase)
    bool ok_run = true;
    bool waited = !a.kv_ready;   // kv_ready: wait after the first STAGES tiles
    auto ensure_wait = [&]() {
      if (!waited) {
        griddep_wait();
        griddep_launch_dependents();
        waited = true;
      }
    };
    for (int s = 0; s < nseg && ok_run; ++s) {
      int u, lt0, lt1;
      seg_range(s, u, lt0, lt1);
      const int ug = u / a.row_blocks;
      const int rot = (!WIN || a.tph > 0) ? phys_tile(0, ug % a.hkv) : 0;
      long long kv_off = 0;
      if constexpr (!PAGED) kv_off = unit_of(u).kv_off;
      long long win_off = 0;
      if constexpr (WIN)
        win_off = (long long)(ug / a.hkv) * a.win.sb + (long long)(ug % a.hkv) * a.win.sh;
      if (s > 0) {
        ensure_wait();
        // The consumers took the previous query rows into registers.
        if (!mbar_wait(q_empty, (s - 1) & 1, kWaitLimitCycles)) {
          if (lane == 0) atomicOr(&g_attn_sk_dev_flags, 4u);
          break;
        }
        load_q(u, pw * 32 + lane, C::NPW * 32);
        cp_async_mbar_arrive(q_full);
      }
      const uint64_t pol = policy_evict_first();   // K/V are read once
      for (int lt = lt0; lt < lt1; ++lt, ++t) {
        const int st = t % C::STAGES;
        if (t >= C::STAGES) ensure_wait();
        if (t >= C::STAGES &&
            !mbar_wait(empty_bar(st), ((t / C::STAGES) & 1) ^ 1, kWaitLimitCycles)) {
          if (lane == 0) atomicOr(&g_attn_sk_dev_flags, 4u);
          ok_run = false;
          break;
        }
        long long my_off = -1;
        const bool wtile = WIN && lt == a.tph;
        if (wtile) {   // the window rows, read (like q) only after the wait
          ensure_wait();
          if (my_row < a.w) my_off = win_off + (long long)my_row * a.win.sn;
        } else {
          int pt = lt + rot;
          pt = pt >= a.tph ? pt - a.tph : pt;
          const int p = pt * C::TILE + my_row;  // position in the unit
          if (p < a.n) {
            if constexpr (PAGED) {
              const long long base = tab[t * (C::TILE / 16) + my_row / 16];
              my_off = base < 0 ? -1 : base + (long long)(my_row % 16) * a.kv.sn;
            } else {
              my_off = kv_off + (long long)p * a.kv.sn;
            }
          }
        }
        const __nv_bfloat16* src = wtile ? (is_v ? a.win.v : a.win.k) : src_base;
        const unsigned vm = __ballot_sync(0xffffffffu, my_off >= 0) &
                            (C::RPW == 32 ? 0xffffffffu : ((1u << C::RPW) - 1u));
        unsigned char* dst = dst_base + st * C::TILE_BYTES + ch * 16;
#pragma unroll 8
        for (int it = 0; it < C::RPW / RPI; ++it) {
          const int rr = it * RPI + sub;            // row within this warp's rows
          const long long off = __shfl_sync(0xffffffffu, my_off, rr);
          const bool ok = off >= 0;
          cp_async_16_hint(smem_u32(dst + (pw * C::RPW + rr) * C::RS),
                           src + (ok ? off + ch * 8 : 0), ok ? 16 : 0, pol);
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
    ensure_wait();
    // Every copy of this thread lands before the CTA may exit.
    cp_async_wait<0>();
    return;
  }

  // ============================ consumer warps ============================
  if constexpr (C::REBALANCE)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(C::CONSUMER_REGS));
  const int wm = warp / C::WN;
  const int wn = warp % C::WN;
  if (a.kv_ready) {
    griddep_wait();
    griddep_launch_dependents();
    if (nseg > 0) load_q(u_first, tid, C::NCW * 32);
    cp_async_commit();
    cp_async_wait<0>();
    named_bar_sync(1, C::NCW * 32);
  }
  const int gq = lane >> 2, tq = lane & 3;
  int t = 0;
  bool dead = false;
  auto wait_or_die = [&](uint32_t bar, uint32_t parity) {
    if (dead) return;
    if (!mbar_wait(bar, parity, kWaitLimitCycles)) {
      dead = true;
      if (lane == 0) atomicOr(&g_attn_sk_dev_flags, 4u);
    }
  };

  for (int sgi = 0; sgi < nseg; ++sgi) {
    int seg_tiles, seg_lt0, tA = 0, tB = 0;
    {
      int u, lt0, lt1;
      seg_range(sgi, u, lt0, lt1);
      seg_tiles = lt1 - lt0;
      seg_lt0 = lt0;
      if (WIN) {   // window position of rows 16 wm + gq and + 8
        const int r0 = (u % a.row_blocks) * C::ROWS + wm * 16 + gq;
        tA = r0 % a.w;
        tB = (r0 + 8) % a.w;
      }
    }
    if (sgi > 0) wait_or_die(q_full, (sgi - 1) & 1);
    uint32_t qf[C::KS][4];
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      const int r = wm * 16 + (lane & 15);
      const int ch = ks * 2 + (lane >> 4);
      ldmatrix_x4(smem_u32(sQ + r * C::RS + ch * 16), qf[ks][0], qf[ks][1],
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

    for (int i = 0; i < seg_tiles; ++i, ++t) {
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
      // Two accumulator chains (even and odd k16 steps), summed after the
      // loop: half the dependent mma depth (measured 340 -> 327 us per
      // 72B-shaped dense layer).
      float sc2[C::NT8][4];
#pragma unroll
      for (int j = 0; j < C::NT8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc2[j][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks) {
#pragma unroll
        for (int j = 0; j < C::NT8; j += 2) {
          const int r = wn * C::PW + j * 8 + ((lane >> 4) << 3) + (lane & 7);
          const int ch = ks * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(smem_u32(tk + r * C::RS + ch * 16), b0, b1, b2, b3);
          if (ks & 1) {
            mma_bf16(sc2[j], qf[ks], b0, b1);
            mma_bf16(sc2[j + 1], qf[ks], b2, b3);
            continue;
          }
          mma_bf16(sc[j], qf[ks], b0, b1);
          mma_bf16(sc[j + 1], qf[ks], b2, b3);
        }
      }
#pragma unroll
      for (int j = 0; j < C::NT8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[j][e] += sc2[j][e];

      // Rows left out of the tile get -inf.  Scores stay unscaled here: the
      // scale (> 0) is folded into the exponent below, so the maximum is
      // taken on raw scores and converted once per row.
      if (WIN && seg_lt0 + i == a.tph) {   // the window: causal
#pragma unroll
        for (int j = 0; j < C::NT8; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int pos = wn * C::PW + j * 8 + 2 * tq + e;
            sc[j][e] = pos <= tA ? sc[j][e] : -INFINITY;
            sc[j][e + 2] = pos <= tB ? sc[j][e + 2] : -INFINITY;
          }
      } else if (vmask != ~0ull) {
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
      mx0 *= a.scale_log2;   // log2 units (-inf stays -inf)
      mx1 *= a.scale_log2;
      // Lazy rescale: move a row's reference maximum only when the tile's
      // maximum exceeds it by more than 2^kLazyRescale.
      const bool up0 = mx0 > m0 + kLazyRescale, up1 = mx1 > m1 + kLazyRescale;
      if (__any_sync(0xffffffffu, up0 || up1)) {
        const float n0 = up0 ? mx0 : m0, n1 = up1 ? mx1 : m1;
        const float c0 = up0 ? ex2(m0 - n0) : 1.f;   // ex2(-inf) = 0
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
          const int ch = dt + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(smem_u32(tv + r * C::RS + ch * 16), b0, b1, b2, b3);
          mma_bf16(oacc[dt], pa, b0, b1);
          mma_bf16(oacc[dt + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(st));
    }

    // ---- Segment end: row sums over the quad, merge the WN slices.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if constexpr (C::WN > 1) {
      if (sgi == nseg - 1) {
        // The range's last segment: every copy has landed and none follows,
        // so the K stages hold all WN - 1 slices at once (one exchange).
        named_bar_sync(1, C::NCW * 32);
        constexpr int SLOTS = C::DT * 4 + 4;
        static_assert((C::WN - 1) * MT * 32 * SLOTS * 4 <= C::STAGES * C::TILE_BYTES,
                      "merge slices");
        float* mb = reinterpret_cast<float*>(sK);
        if (wn > 0) {
          float* pp = mb + ((wn - 1) * MT + wm) * 32 * SLOTS + lane;
          pp[0] = m0;
          pp[32] = m1;
          pp[64] = l0;
          pp[96] = l1;
#pragma unroll
          for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
            for (int e = 0; e < 4; ++e) pp[(4 + dt * 4 + e) * 32] = oacc[dt][e];
        }
        named_bar_sync(1, C::NCW * 32);
        if (wn == 0) {
#pragma unroll 1
          for (int o = 1; o < C::WN; ++o) {
            const float* pp = mb + ((o - 1) * MT + wm) * 32 * SLOTS + lane;
            const float om0 = pp[0], om1 = pp[32], ol0 = pp[64], ol1 = pp[96];
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
              oacc[dt][0] = oacc[dt][0] * a0 + pp[(4 + dt * 4 + 0) * 32] * b0;
              oacc[dt][1] = oacc[dt][1] * a0 + pp[(4 + dt * 4 + 1) * 32] * b0;
              oacc[dt][2] = oacc[dt][2] * a1 + pp[(4 + dt * 4 + 2) * 32] * b1;
              oacc[dt][3] = oacc[dt][3] * a1 + pp[(4 + dt * 4 + 3) * 32] * b1;
            }
          }
        }
      } else {
        // A segment with more to follow: the producers are filling the
        // stages already, so the slices pass through a small buffer of
        // their own, one partner and half of d at a time.
        float* mb = sMerge + wm * 32 * C::MSLOTS + lane;
#pragma unroll 1
        for (int o = 1; o < C::WN; ++o) {
          // Weights of the two sides, from the maxima (shared by both halves).
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
    }

    // ---- Write rows r = 16 wm + gq (+8) of this unit's row block.
    int u, lt0, lt1;
    seg_range(sgi, u, lt0, lt1);
    const Unit x = unit_of(u);
    const int rA = wm * 16 + gq, rB = rA + 8;
    const int RA = x.rb * C::ROWS + rA, RB = RA + 8;
    if (lt0 == 0 && lt1 == a.tpu) {
      if (wn == 0) {
        const float i0 = l0 > 0.f ? 1.f / l0 : 0.f;
        const float i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt) {
          const int col = dt * 8 + 2 * tq;
          if (RA < a.rows)
            *reinterpret_cast<uint32_t*>(a.o + (x.row_base + RA) * D + col) =
                pack_bf16(oacc[dt][0] * i0, oacc[dt][1] * i0);
          if (RB < a.rows)
            *reinterpret_cast<uint32_t*>(a.o + (x.row_base + RB) * D + col) =
                pack_bf16(oacc[dt][2] * i1, oacc[dt][3] * i1);
        }
        if (tq == 0) {
          if (RA < a.rows)
            a.lse[x.row_base + RA] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
          if (RB < a.rows)
            a.lse[x.row_base + RB] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
        }
      }
      continue;
    }

    // Split unit: leave this segment's partial, count it, and let the CTA
    // that completes the count merge the unit.
    const long long slot = 2LL * blockIdx.x + (lt0 == 0 ? 1 : 0);
    if (wn == 0) {
      const long long pb = slot * C::ROWS;
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
      __threadfence();
    }
    const long long x0 = (long long)u * a.tpu;
    const int c_first = sk_owner(x0, T, a.grid);
    const int c_last = sk_owner(x0 + a.tpu - 1, T, a.grid);
    named_bar_sync(1, C::NCW * 32);
    if (warp == 0 && lane == 0) {
      unsigned long long* cw = a.counters + u;
      unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(cw);
      unsigned long long mine = 0;
      bool done = false;
      for (int it = 0; it < 4096 && !done; ++it) {
        const unsigned long long cnt = ((old >> 24) == a.epoch) ? (old & 0xffffffull) : 0ull;
        mine = (a.epoch << 24) | (cnt + 1);
        const unsigned long long seen = atomicCAS(cw, old, mine);
        done = seen == old;
        old = seen;
      }
      const int count = done ? (int)(mine & 0xffffffull) : 0;
      if (!done) atomicOr(&g_attn_sk_dev_flags, 4u);
      const bool last = count == c_last - c_first + 1;
      if (last) {
        __threadfence();
        atomicExch(cw, 0ull);   // ready for the next call or replay
      }
      *sFlag = last ? 1 : 0;
    }
    named_bar_sync(1, C::NCW * 32);
    if (*sFlag == 0 || wn != 0) continue;
    __threadfence();
    // Merge the unit's partials, rows rA, rB of this warp:
    //   O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c,  M = max_c m_c,
    // summed in CTA order whichever CTA merges, so the result is the same
    // bits every run.  The first term is this CTA's own partial (still in
    // registers) when it holds the unit's first tiles, the usual case.
    auto slot_of = [&](int c) { return (c == c_first ? 2LL * c + 1 : 2LL * c) * C::ROWS; };
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll 4
    for (int c = c_first; c <= c_last; ++c) {
      M0 = fmaxf(M0, __ldcg(&a.ws_ml[slot_of(c) + rA].x));
      M1 = fmaxf(M1, __ldcg(&a.ws_ml[slot_of(c) + rB].x));
    }
    const float v0 = (M0 == -INFINITY) ? 0.f : M0;
    const float v1 = (M1 == -INFINITY) ? 0.f : M1;
    float L0, L1;
    {
      const long long pb = slot_of(c_first);
      const float2 mlA = __ldcg(&a.ws_ml[pb + rA]);
      const float2 mlB = __ldcg(&a.ws_ml[pb + rB]);
      const float fA = ex2(mlA.x - v0), fB = ex2(mlB.x - v1);
      L0 = __fmul_rn(fA, mlA.y);
      L1 = __fmul_rn(fB, mlB.y);
      const bool mine = c_first == (int)blockIdx.x;
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt) {
        const int col = dt * 8 + 2 * tq;
        float2 pA, pB;
        if (mine) {
          pA = make_float2(oacc[dt][0], oacc[dt][1]);
          pB = make_float2(oacc[dt][2], oacc[dt][3]);
        } else {
          pA = __ldcg(reinterpret_cast<const float2*>(a.ws_o + (pb + rA) * D + col));
          pB = __ldcg(reinterpret_cast<const float2*>(a.ws_o + (pb + rB) * D + col));
        }
        oacc[dt][0] = __fmul_rn(fA, pA.x);
        oacc[dt][1] = __fmul_rn(fA, pA.y);
        oacc[dt][2] = __fmul_rn(fB, pB.x);
        oacc[dt][3] = __fmul_rn(fB, pB.y);
      }
    }
    for (int c = c_first + 1; c <= c_last; ++c) {
      const long long pb = slot_of(c);
      const float2 mlA = __ldcg(&a.ws_ml[pb + rA]);
      const float2 mlB = __ldcg(&a.ws_ml[pb + rB]);
      const float fA = ex2(mlA.x - v0), fB = ex2(mlB.x - v1);
      L0 = fmaf(fA, mlA.y, L0);
      L1 = fmaf(fB, mlB.y, L1);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float2 pA[C::DT / 2], pB[C::DT / 2];
#pragma unroll
        for (int dt = 0; dt < C::DT / 2; ++dt) {
          const int col = (half * (C::DT / 2) + dt) * 8 + 2 * tq;
          pA[dt] = __ldcg(reinterpret_cast<const float2*>(a.ws_o + (pb + rA) * D + col));
          pB[dt] = __ldcg(reinterpret_cast<const float2*>(a.ws_o + (pb + rB) * D + col));
        }
#pragma unroll
        for (int dt = 0; dt < C::DT / 2; ++dt) {
          float* o4 = oacc[half * (C::DT / 2) + dt];
          o4[0] = fmaf(fA, pA[dt].x, o4[0]);
          o4[1] = fmaf(fA, pA[dt].y, o4[1]);
          o4[2] = fmaf(fB, pB[dt].x, o4[2]);
          o4[3] = fmaf(fB, pB[dt].y, o4[3]);
        }
      }
    }
    const float i0 = L0 > 0.f ? 1.f / L0 : 0.f;
    const float i1 = L1 > 0.f ? 1.f / L1 : 0.f;
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt) {
      const int col = dt * 8 + 2 * tq;
      if (RA < a.rows)
        *reinterpret_cast<uint32_t*>(a.o + (x.row_base + RA) * D + col) =
            pack_bf16(oacc[dt][0] * i0, oacc[dt][1] * i0);
      if (RB < a.rows)
        *reinterpret_cast<uint32_t*>(a.o + (x.row_base + RB) * D + col) =
            pack_bf16(oacc[dt][2] * i1, oacc[dt][3] * i1);
    }
    if (tq == 0) {
      if (RA < a.rows)
        a.lse[x.row_base + RA] = L0 > 0.f ? (M0 + log2f(L0)) * kLn2 : -INFINITY;
      if (RB < a.rows)
        a.lse[x.row_base + RB] = L1 > 0.f ? (M1 + log2f(L1)) * kLn2 : -INFINITY;
    }
  }
}

}  // namespace dustin
