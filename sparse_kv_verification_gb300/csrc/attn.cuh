// Sparse verification attention, Dustin's Stage 2 (verification over the
// selected KV; "dustin-long-context" notes section 2.2, Fig. 5): every query
// row of the window against the k positions idx[b][0..k) of its sequence.
//
// One CTA handles one (sequence b, kv head g, row block, split): the G*w
// query rows that share kv head g (query heads g*G .. g*G+G-1, w window
// rows each: a contiguous [G*w][d] block of q) against a contiguous range
// of the selected positions.  A sparse unit is short (32 tiles of 64 at
// k = 2048), so one CTA per unit is the fastest schedule whenever the units
// come near filling the GPU (128 on 152 SMs at the 72B shape): splitting a
// unit across CTAs only adds a merge to a loop already near the gather
// ceiling.  When they do not, the positions are split into `splits` equal
// ranges and attn_combine_kernel merges the partials.
//
// Warp-specialised pipeline:
//  * a producer warpgroup (4 warps) gathers each 64-position tile, 16 rows
//    per warp: one warp instruction of 16-byte cp.async copies a whole K row
//    and V row (d = 128; two rows for d = 64) into padded shared-memory rows
//    (2*d + 16 bytes, so ldmatrix of eight rows is conflict-free).  Each
//    producer thread then arms cp.async.mbarrier.arrive on the stage's
//    "full" mbarrier, and lane 0 publishes the warp's valid-row mask with a
//    plain (release) arrive.  Row offsets come from a shared-memory table
//    that every thread of the CTA fills once from idx (and the page table)
//    before the pipeline starts, so no global-load latency sits inside the
//    producer loop.  Rows that fail a check, and rows past the range, are
//    zero-filled by the copy (source size 0) and left out through the valid
//    mask.  (Measured on a 72B-shaped gather of 256-byte rows: 16-byte
//    cp.async reaches 4.3, 5.0 and 5.2 TB/s with 2, 4 and 8 producer warps,
//    per-row TMA bulk copies 1.1 TB/s and TMA tile::gather4 1.8 TB/s, so
//    cp.async does the gather.)  With 16 warps (three consumer warpgroups)
//    the producers hand registers to the consumers with setmaxnreg (40 / 152
//    of a 128-register launch).
//  * MT*WN consumer warps: warp (wm, wn) owns query rows [16 wm, 16 wm + 16)
//    and a 64/WN-position slice of every tile.  S = Q K^T and O += P V run on
//    bf16 mma.sync m16n8k16 with fp32 accumulators; the softmax is online in
//    base 2 with a lazy reference maximum (O and l are rescaled only when a
//    row maximum grows by more than 2^8), which is exact: the reference only
//    has to bound the exponents.  Consumers release a stage through its
//    "empty" mbarrier.
// STAGES tiles are in flight.  Every mbarrier wait is bounded (about one
// second): on timeout the kernel raises a flag and winds down.  At the end
// the WN position slices are merged through shared memory; a single split
// writes O (bf16) and LSE directly, several splits write fp32 partials that
// attn_combine_kernel merges.
#pragma once

#include "device_common.cuh"

namespace dustin {

struct AttnArgs {
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;
  KvView kv;
  const int* idx;   // [b][npos]
  int b, hq, hkv, w, n;
  int npos;         // selected positions per sequence: k
  int group;        // hq / hkv
  int rows;         // group * w
  int row_blocks;   // ceil(rows / (16 * MT))
  int splits;
  int chunk;        // positions per split (multiple of 64)
  float scale_log2; // scale * log2(e)
  int kv_ready;     // idx, page table and K/V may be read before the wait
  KvView win;       // the window's own K/V [b][hkv][w][d] (has_win)
  int has_win;      // merge the window's causal block (last split only;
                    // selects the WIN instance of the kernel)
  int wide;         // 32-bit row codes (selects the WIDE instance)
  float* ws_o;      // [blocks][splits][16 MT][D] (splits > 1)
  float2* ws_ml;    // [blocks][splits][16 MT]    (m in log2 units, l)
};

// Build-time tunables (nvcc -D): producer warps (4 or 8) and pipeline depth
// for d = 128.
#ifndef DUSTIN_ATTN_NPW
#define DUSTIN_ATTN_NPW 4
#endif
#ifndef DUSTIN_ATTN_STAGES128
#define DUSTIN_ATTN_STAGES128 5
#endif
#ifndef DUSTIN_ATTN_ROTATE
#define DUSTIN_ATTN_ROTATE 1
#endif
#ifndef DUSTIN_ATTN_PLAIN_CP
#define DUSTIN_ATTN_PLAIN_CP 0
#endif

template <int D, int MT>
struct AttnCfg {
  static constexpr int WN = (MT == 4) ? 2 : 4;
  static constexpr int NCW = MT * WN;            // consumer warps
  static constexpr int NPW = DUSTIN_ATTN_NPW;    // producer warps
  static_assert(NPW == 4 || NPW == 8, "producer warps: whole warpgroups");
  static constexpr int NT = (NCW + NPW) * 32;
  static constexpr int RPW = 64 / NPW;           // tile rows per producer warp
  // Above 384 threads the register file is tight: the producer warpgroups
  // drop to 40 registers and the consumer warpgroups take the rest, e.g.
  // 16 warps (128 at launch): 40*128 + 152*384 <= 128*512.
  static constexpr bool REBALANCE = (NT > 384);
  static constexpr int PRODUCER_REGS = 40;
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
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * TILE_BYTES;
  static constexpr int OFF_MASK = OFF_V + STAGES * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_MASK + STAGES * 8;   // 64-bit mask / stage
  // Row table of one CTA's positions: TAB_BYTES of shared memory holding
  // either the 64-bit element offset of each row (TAB64 positions) or, in
  // the WIDE kernel variant for longer ranges, a 32-bit row code (TAB32
  // positions).  Four row tiles leave room for half as much.
  static constexpr int TAB_BYTES = MT == 4 ? 16384 : 32768;
  static constexpr int TAB64 = TAB_BYTES / 8;
  static constexpr int TAB32 = TAB_BYTES / 4;
  static constexpr int OFF_TAB = OFF_BAR + 2 * STAGES * 8;
  static constexpr int SMEM = OFF_TAB + TAB_BYTES;
  static constexpr int MERGE_FLOATS = (WN - 1) * MT * 32 * (DT * 4 + 4);
  static_assert(MERGE_FLOATS * 4 <= 2 * STAGES * TILE_BYTES, "merge buffer");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Device-side check flags of this translation unit.
static __device__ unsigned int g_attn_dev_flags;


template <int D, int MT, bool PAGED, bool WIN, bool WIDE>
__global__ void __launch_bounds__(AttnCfg<D, MT>::NT, 1)
    verify_attn_kernel(const AttnArgs a) {
  using C = AttnCfg<D, MT>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sQ = smem;
  unsigned char* sK = smem + C::OFF_K;
  unsigned char* sV = smem + C::OFF_V;
  unsigned long long* sMask64 =
      reinterpret_cast<unsigned long long*>(smem + C::OFF_MASK);
  long long* tab = reinterpret_cast<long long*>(smem + C::OFF_TAB);   // !WIDE
  int* tab32 = reinterpret_cast<int*>(smem + C::OFF_TAB);              // WIDE
  const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

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
  const int ntiles = (len + C::TILE - 1) / C::TILE;   // history tiles
  // With the window merged in, the last split runs one more tile: the w
  // window rows, causal (row t sees window positions 0..t).
  const int ntot = ntiles + ((WIN && split == a.splits - 1) ? 1 : 0);

  const long long unit_off = (long long)bb * a.kv.sb + (long long)g * a.kv.sh;
  // The kv heads of a sequence share one index set, so their CTAs would
  // gather the same positions from planes a fixed stride apart at the same
  // moment.  Each kv head starts at a different tile instead (the order of
  // tiles does not change the result beyond fp32 rounding).
  const int rot = DUSTIN_ATTN_ROTATE ? (int)(((long long)g * ntiles) / a.hkv) : 0;
  auto tile_of = [&](int t) { int u = t + rot; return u >= ntiles ? u - ntiles : u; };
  const long long row_base =
      ((long long)bb * a.hq + (long long)g * a.group) * a.w;  // first q row
  const int r_lo = rb * C::ROWS;

  // Programmatic dependent launch: the kernel before this one on the stream
  // may still be running until griddepcontrol.wait returns.  Normally every
  // thread waits first.  With kv_ready the caller guarantees that idx, the
  // page table and K/V were not written by that kernel: the table is built
  // and the first STAGES tiles are fetched before the wait, and only q (and
  // every write) waits.  A thread triggers the next launch only after its
  // own wait, so a kernel never starts early while its predecessor's
  // predecessor may still be running.
  if (!a.kv_ready) {
    griddep_wait();
    griddep_launch_dependents();
  }

  // ---- Q rows into shared memory (zero rows past G*w), barriers.
  auto load_q = [&](int first, int step) {
    for (int c = first; c < C::ROWS * C::CPR; c += step) {
      const int r = c / C::CPR, ch = c % C::CPR;
      const int R = r_lo + r;
      const bool ok = R < a.rows;
      cp_async_16(smem_u32(sQ + r * C::RS + ch * 16),
                  a.q + (ok ? (row_base + R) * D + ch * 8 : 0), ok ? 16 : 0);
    }
  };
  if (!a.kv_ready) load_q(tid, C::NT);
  cp_async_commit();
  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), C::NPW * 32 + C::NPW);  // copies + mask arrives
      mbar_init(empty_bar(s), C::NCW);
    }
    mbar_fence_init();
  }
  // Row table: for each selected position, its element offset, or (WIDE)
  // its row code: the position j in a contiguous cache, the pool row
  // page * page_size + j % page_size in a paged one; -1 for a row that
  // failed a check.
  const int* idx_row = a.idx + (long long)bb * a.npos + p_begin;
  if constexpr (PAGED) {
    // Paged: the page-table read depends on the idx read, so a batch of
    // TB entries per thread issues all its idx loads, then all its page
    // loads (two memory latencies per batch instead of two per entry).
    constexpr int TB = 4;
    for (int i0 = tid; i0 < len; i0 += TB * C::NT) {
      int j[TB], pg[TB];
#pragma unroll
      for (int u = 0; u < TB; ++u) {
        const int i = i0 + u * C::NT;
        j[u] = i < len ? __ldg(idx_row + i) : 0;
      }
#pragma unroll
      for (int u = 0; u < TB; ++u) {
        const bool in = i0 + u * C::NT < len && j[u] >= 0 && j[u] < a.n;
        pg[u] = in ? __ldg(a.kv.page_table + (long long)bb * a.kv.pages_per_seq +
                           j[u] / a.kv.page_size)
                   : 0;
      }
#pragma unroll
      for (int u = 0; u < TB; ++u) {
        const int i = i0 + u * C::NT;
        if (i >= len) break;
        long long off = -1;
        int code = -1;
        if (j[u] < 0 || j[u] >= a.n) {
          atomicOr(&g_attn_dev_flags, 1u);
        } else if (pg[u] < 0 || pg[u] >= a.kv.num_pages) {
          atomicOr(&g_attn_dev_flags, 2u);
        } else {
          const int jp = j[u] % a.kv.page_size;
          off = (long long)pg[u] * a.kv.sb + (long long)g * a.kv.sh + (long long)jp * a.kv.sn;
          code = pg[u] * a.kv.page_size + jp;   // < 2^31 (host check)
        }
        if constexpr (WIDE)
          tab32[i] = code;
        else
          tab[i] = off;
      }
    }
  } else {
    // Contiguous: one entry per thread at a time (measured faster here than
    // batching the loads).
    for (int i = tid; i < len; i += C::NT) {
      const int j = __ldg(idx_row + i);
      long long off = -1;
      int code = -1;
      if (j < 0 || j >= a.n) {
        atomicOr(&g_attn_dev_flags, 1u);
      } else {
        off = unit_off + (long long)j * a.kv.sn;
        code = j;
      }
      if constexpr (WIDE)
        tab32[i] = code;
      else
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

    // Element offset of tile row r (-1: leave the row out).
    auto row_offset = [&](int t, int r) -> long long {
      const int i = t * C::TILE + r;
      if constexpr (!WIDE) {
        return i < len ? tab[i] : -1;
      } else {
        const int code = i < len ? tab32[i] : -1;
        if (code < 0) return -1;
        if constexpr (PAGED) {
          const int pg = code / a.kv.page_size;
          return (long long)pg * a.kv.sb + (long long)g * a.kv.sh +
                 (long long)(code - pg * a.kv.page_size) * a.kv.sn;
        } else {
          return unit_off + (long long)code * a.kv.sn;
        }
      }
    };

    // kv_ready: the first n_pre history tiles go out before this thread's
    // wait (the window tile, like q, is read only after it).
    const int n_pre = a.kv_ready ? min(ntiles, C::STAGES) : -1;
    // K/V rows are read once per launch: fetched under an evict-first L2
    // policy they leave idx, q and the outputs in L2 (measured: 28.1 ->
    // 27.8 us per back-to-back layer at the 72B shape).
    const uint64_t pol = policy_evict_first();
    for (int t = 0; t < ntot; ++t) {
      const int s = t % C::STAGES;
      if (t == n_pre) {
        griddep_wait();
        griddep_launch_dependents();
      }
      if (t >= C::STAGES &&
          !mbar_wait(empty_bar(s), ((t / C::STAGES) & 1) ^ 1, kWaitLimitCycles)) {
        if (lane == 0) atomicOr(&g_attn_dev_flags, 4u);
        break;
      }
      const bool wtile = WIN && t == ntiles;
      long long my_off;
      if (!wtile)
        my_off = row_offset(tile_of(t), my_row);
      else
        my_off = my_row < a.w ? (long long)bb * a.win.sb + (long long)g * a.win.sh +
                                    (long long)my_row * a.win.sn
                              : -1;
      const __nv_bfloat16* src = wtile ? (is_v ? a.win.v : a.win.k) : src_base;
      const unsigned vm = __ballot_sync(0xffffffffu, my_off >= 0) &
                          (C::RPW == 32 ? 0xffffffffu : ((1u << C::RPW) - 1u));
      unsigned char* dst = dst_base + s * C::TILE_BYTES + ch * 16;
      // Eight rows' shuffles and copies in flight at once: the producers'
      // issue rate sets part of the tile period (72B layer back to back:
      // 27.85 -> 26.65 us against four; sixteen 26.76; the row offset read
      // from shared memory instead of shuffled 36.0; 32-bit row codes
      // shuffled and the address formed after 29.1).
#pragma unroll 8
      for (int it = 0; it < C::RPW / RPI; ++it) {
        const int rr = it * RPI + sub;            // row within this warp's rows
        const long long off = __shfl_sync(0xffffffffu, my_off, rr);
        const uint32_t d = smem_u32(dst + (pw * C::RPW + rr) * C::RS);
#if DUSTIN_ATTN_PLAIN_CP
        if (off >= 0)
          cp_async_16_full(d, src + off + ch * 8);
        else
          cp_async_16(d, src, 0);                 // zero-fill a left-out row
#else
        const bool ok = off >= 0;
        cp_async_16_hint(d, src + (ok ? off + ch * 8 : 0), ok ? 16 : 0, pol);
#endif
      }
      cp_async_mbar_arrive(full_bar(s));
      if (lane == 0) {
        if constexpr (C::RPW == 16)
          reinterpret_cast<unsigned short*>(sMask64 + s)[pw] = (unsigned short)vm;
        else if constexpr (C::RPW == 8)
          reinterpret_cast<unsigned char*>(sMask64 + s)[pw] = (unsigned char)vm;
        else
          reinterpret_cast<unsigned*>(sMask64 + s)[pw] = vm;
        mbar_arrive(full_bar(s));
      }
    }
    if (n_pre >= ntot) {   // kv_ready, and every tile went out early
      griddep_wait();
      griddep_launch_dependents();
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
  if (a.kv_ready) {
    griddep_wait();
    griddep_launch_dependents();
    load_q(tid, C::NCW * 32);
    cp_async_commit();
    cp_async_wait<0>();
    named_bar_sync(1, C::NCW * 32);
  }
  uint32_t qf[C::KS][4];
#pragma unroll
  for (int ks = 0; ks < C::KS; ++ks) {
    const int r = wm * 16 + (lane & 15);
    const int ch = ks * 2 + (lane >> 4);
    ldmatrix_x4(smem_u32(sQ + r * C::RS + ch * 16), qf[ks][0], qf[ks][1],
                qf[ks][2], qf[ks][3]);
  }

  float oacc[C::DT][4];
#pragma unroll
  for (int i = 0; i < C::DT; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[i][e] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int gq = lane >> 2, tq = lane & 3;

  for (int t = 0; t < ntot; ++t) {
    const int s = t % C::STAGES;
    if (!mbar_wait(full_bar(s), (t / C::STAGES) & 1, kWaitLimitCycles)) {
      if (lane == 0) atomicOr(&g_attn_dev_flags, 4u);
      break;
    }
    const unsigned char* tk = sK + s * C::TILE_BYTES;
    const unsigned char* tv = sV + s * C::TILE_BYTES;
    const unsigned long long vmask = sMask64[s];

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
        const int ch = ks * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(smem_u32(tk + r * C::RS + ch * 16), b0, b1, b2, b3);
        mma_bf16(sc[j], qf[ks], b0, b1);
        mma_bf16(sc[j + 1], qf[ks], b2, b3);
      }
    }

    // Rows left out of the tile get -inf.  Scores stay unscaled here: the
    // scale (> 0) is folded into the exponent below, so the maximum is taken
    // on raw scores and converted once per row.
    if (WIN && t == ntiles) {   // the window tile: causal within the window
      // Window position of rows 16 wm + gq and + 8 (rows past G*w: unused),
      // formed here so that they hold no registers through the loop.
      const int tA = (r_lo + wm * 16 + gq) % a.w;
      const int tB = (r_lo + wm * 16 + gq + 8) % a.w;
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
    const float c = a.scale_log2;
#pragma unroll
    for (int j = 0; j < C::NT8; ++j) {
      sc[j][0] = ex2(fmaf(sc[j][0], c, -u0));
      sc[j][1] = ex2(fmaf(sc[j][1], c, -u0));
      sc[j][2] = ex2(fmaf(sc[j][2], c, -u1));
      sc[j][3] = ex2(fmaf(sc[j][3], c, -u1));
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
    if (lane == 0) mbar_arrive(empty_bar(s));
  }

  // ---- Row sums over the quad, then merge the WN position slices.
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  if constexpr (C::WN == 4) {
    // ---- Merge the WN position slices; every consumer warp takes part
    // (72B layer back to back: 26.56 -> 25.77 us against the merge by the
    // wn = 0 warps below, which the two-slice instance keeps).
    // Every warp parks its (m, l) and partial O in shared memory (the stages
    // are free: every issued copy was waited for); warp (wm, wn) then owns
    // the d tiles [wn OWN, wn OWN + OWN) of its row tile and folds slices
    // 1 .. WN-1 into slice 0 in slice order for them, with the pairwise rule
    //   M' = max(M, m_o),  a = 2^(M - M'),  b = 2^(m_o - M'),
    //   L' = L a + l_o b,  O' = O a + O_o b
    // that every warp of the row tile evaluates on the same (m, l) table.
    // The normalised bf16 rows go through shared memory (the Q rows, no
    // longer read) so that the global writes are whole 16-byte chunks.
    constexpr int OWN = C::DT / C::WN;
    static_assert(MT * C::WN * (C::DT + 1) * 32 * 16 <= 2 * C::STAGES * C::TILE_BYTES,
                  "slice exchange buffer");
    const int rA = wm * 16 + gq, rB = rA + 8;
    named_bar_sync(1, C::NCW * 32);
    float4* xo = reinterpret_cast<float4*>(sK);                 // [MT][WN][DT][32]
    float4* xml = xo + MT * C::WN * C::DT * 32;                 // [MT][WN][32]
    const float4* mine = xo + (wm * C::WN) * C::DT * 32 + lane; // slice 0 of the row tile
    xml[(wm * C::WN + wn) * 32 + lane] = make_float4(m0, m1, l0, l1);
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt)
      xo[((wm * C::WN + wn) * C::DT + dt) * 32 + lane] =
          make_float4(oacc[dt][0], oacc[dt][1], oacc[dt][2], oacc[dt][3]);
    named_bar_sync(1, C::NCW * 32);
    float M0, M1, L0, L1;
    {
      const float4 v = xml[(wm * C::WN) * 32 + lane];
      M0 = v.x;
      M1 = v.y;
      L0 = v.z;
      L1 = v.w;
    }
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt) {
      if (dt / OWN != wn) continue;
      const float4 v = mine[dt * 32];
      oacc[dt][0] = v.x;
      oacc[dt][1] = v.y;
      oacc[dt][2] = v.z;
      oacc[dt][3] = v.w;
    }
#pragma unroll 1
    for (int o = 1; o < C::WN; ++o) {
      const float4 v = xml[(wm * C::WN + o) * 32 + lane];
      const float N0 = fmaxf(M0, v.x), N1 = fmaxf(M1, v.y);
      const float u0 = (N0 == -INFINITY) ? 0.f : N0;
      const float u1 = (N1 == -INFINITY) ? 0.f : N1;
      const float a0 = ex2(M0 - u0), b0 = ex2(v.x - u0);
      const float a1 = ex2(M1 - u1), b1 = ex2(v.y - u1);
      L0 = __fmaf_rn(L0, a0, __fmul_rn(v.z, b0));
      L1 = __fmaf_rn(L1, a1, __fmul_rn(v.w, b1));
      M0 = N0;
      M1 = N1;
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt) {
        if (dt / OWN != wn) continue;
        const float4 w = mine[(o * C::DT + dt) * 32];
        oacc[dt][0] = __fmaf_rn(oacc[dt][0], a0, __fmul_rn(w.x, b0));
        oacc[dt][1] = __fmaf_rn(oacc[dt][1], a0, __fmul_rn(w.y, b0));
        oacc[dt][2] = __fmaf_rn(oacc[dt][2], a1, __fmul_rn(w.z, b1));
        oacc[dt][3] = __fmaf_rn(oacc[dt][3], a1, __fmul_rn(w.w, b1));
      }
    }

    if (a.splits == 1) {
      const float i0 = L0 > 0.f ? 1.f / L0 : 0.f;
      const float i1 = L1 > 0.f ? 1.f / L1 : 0.f;
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt) {
        if (dt / OWN != wn) continue;
        const int col = dt * 8 + 2 * tq;
        *reinterpret_cast<uint32_t*>(sQ + rA * C::RS + col * 2) =
            pack_bf16(oacc[dt][0] * i0, oacc[dt][1] * i0);
        *reinterpret_cast<uint32_t*>(sQ + rB * C::RS + col * 2) =
            pack_bf16(oacc[dt][2] * i1, oacc[dt][3] * i1);
      }
      if (wn == 0 && tq == 0) {
        const int RA = r_lo + rA, RB = r_lo + rB;
        if (RA < a.rows)
          a.lse[row_base + RA] = L0 > 0.f ? (M0 + log2f(L0)) * kLn2 : -INFINITY;
        if (RB < a.rows)
          a.lse[row_base + RB] = L1 > 0.f ? (M1 + log2f(L1)) * kLn2 : -INFINITY;
      }
      named_bar_sync(1, C::NCW * 32);
      for (int c = tid; c < C::ROWS * C::CPR; c += C::NCW * 32) {
        const int r = c / C::CPR, ch = c % C::CPR;
        if (r_lo + r < a.rows)
          *reinterpret_cast<uint4*>(a.o + (row_base + r_lo + r) * D + ch * 8) =
              *reinterpret_cast<const uint4*>(sQ + r * C::RS + ch * 16);
      }
    } else {
      const long long pb = ((long long)blockIdx.x) * C::ROWS;  // (blk, split)
#pragma unroll
      for (int dt = 0; dt < C::DT; ++dt) {
        if (dt / OWN != wn) continue;
        const int col = dt * 8 + 2 * tq;
        *reinterpret_cast<float2*>(a.ws_o + (pb + rA) * D + col) =
            make_float2(oacc[dt][0], oacc[dt][1]);
        *reinterpret_cast<float2*>(a.ws_o + (pb + rB) * D + col) =
            make_float2(oacc[dt][2], oacc[dt][3]);
      }
      if (wn == 0 && tq == 0) {
        a.ws_ml[pb + rA] = make_float2(M0, L0);
        a.ws_ml[pb + rB] = make_float2(M1, L1);
      }
    }
  } else {
    // Every issued copy was waited for, so the stages are free to reuse.
    named_bar_sync(1, C::NCW * 32);
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
      named_bar_sync(1, C::NCW * 32);
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
  griddep_wait();
  griddep_launch_dependents();
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
