// C-ABI of the Dustin sparse-verification library (declared in
// include/dustin.h): host-side validation, launch planning and dispatch.
// Nothing here allocates device memory; scratch comes from the caller.
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "attn.cuh"
#include "attn_streamk.cuh"
#include "attn_multilayer.cuh"
#include "dustin.h"
#include "internal.h"

namespace dustin {

namespace {

std::atomic<uint64_t> g_launches{0};
thread_local char g_err[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(DUSTIN_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
      cudaSuccess)
    return 1;
  return sms > 0 ? sms : 1;
}

// Resident CTAs of the (non-paged) attention kernel times the SM count,
// cached per device, kernel family, head dim and row tile count.
int attn_slots(bool dense, int d, int mt) {
  static std::atomic<int> cache[64][2][2][5];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  std::atomic<int>& c = cache[dev][dense ? 1 : 0][d == 128 ? 1 : 0][mt];
  int v = c.load(std::memory_order_relaxed);
  if (v > 0) return v;
  const int occ = dense ? occupancy_attn_dense(d, mt) : occupancy_attn_sparse(d, mt);
  v = sm_count() * (occ > 0 ? occ : 1);
  c.store(v, std::memory_order_relaxed);
  return v;
}

KvView to_view(const dustin_kv& kv) {
  KvView v;
  v.k = static_cast<const __nv_bfloat16*>(kv.k);
  v.v = static_cast<const __nv_bfloat16*>(kv.v);
  v.sb = kv.stride_b;
  v.sh = kv.stride_h;
  v.sn = kv.stride_n;
  v.page_table = kv.page_table;
  v.page_size = kv.page_size;
  v.pages_per_seq = kv.pages_per_seq;
  v.num_pages = kv.num_pages;
  return v;
}

// Checks a KV descriptor for `b` sequences of `n` positions with head dim d.
int check_kv(const dustin_kv* kv, int b, int n, int d, bool need_v,
             const char* what) {
  if (!kv) return fail(DUSTIN_ERR_INVALID_ARG, "%s: kv is NULL", what);
  if (!kv->k) return fail(DUSTIN_ERR_INVALID_ARG, "%s: kv.k is NULL", what);
  if (need_v && !kv->v)
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: kv.v is NULL", what);
  if (!aligned16(kv->k) || (need_v && !aligned16(kv->v)))
    return fail(DUSTIN_ERR_ALIGNMENT, "%s: kv base not 16-byte aligned", what);
  if (kv->stride_b < 0 || kv->stride_h < 0 || kv->stride_n < d)
    return fail(DUSTIN_ERR_SHAPE, "%s: bad kv strides (%lld, %lld, %lld)", what,
                (long long)kv->stride_b, (long long)kv->stride_h,
                (long long)kv->stride_n);
  if (kv->stride_b % 8 || kv->stride_h % 8 || kv->stride_n % 8)
    return fail(DUSTIN_ERR_ALIGNMENT,
                "%s: kv strides must be multiples of 8 elements", what);
  if (kv->page_table) {
    if (kv->page_size < 16 || kv->page_size % 16)
      return fail(DUSTIN_ERR_UNSUPPORTED,
                  "%s: page_size %d (must be a positive multiple of 16)", what,
                  kv->page_size);
    if (kv->num_pages < 1)
      return fail(DUSTIN_ERR_SHAPE, "%s: num_pages %d", what, kv->num_pages);
    const long long need = ((long long)n + kv->page_size - 1) / kv->page_size;
    if (kv->pages_per_seq < need)
      return fail(DUSTIN_ERR_SHAPE, "%s: pages_per_seq %d < %lld", what,
                  kv->pages_per_seq, need);
    if ((reinterpret_cast<uintptr_t>(kv->page_table) & 3u) != 0)
      return fail(DUSTIN_ERR_ALIGNMENT, "%s: page_table misaligned", what);
  }
  (void)b;
  return DUSTIN_OK;
}

// ---- attention planning
// Shared by both kernels: a unit is (sequence, kv head, row block of at
// most 64 query rows, in 16-row tiles).
struct AttnPlan {
  int mt, row_blocks, tpu, tph;
  long long units;
  // sparse: positions split `splits` ways, `chunk` positions each.
  int splits, chunk;
  bool wide;   // 32-bit row table (sparse)
  // dense: stream-K over `grid` CTAs; `split` when some unit is shared.
  long long grid;
  bool split;
  size_t ws_o, ws_ml, ws_cnt;
  size_t workspace() const { return ws_o + ws_ml + ws_cnt; }
};

AttnPlan plan_units(int hq, int hkv, int w, int b, int npos) {
  AttnPlan p{};
  const long long rows = (long long)(hq / hkv) * w;
  p.mt = (int)std::min<long long>(4, std::max<long long>(1, (rows + 15) / 16));
  p.row_blocks = (int)((rows + 16 * p.mt - 1) / (16 * p.mt));
  p.units = (long long)b * hkv * p.row_blocks;
  p.tpu = std::max(1, (npos + 63) / 64);
  return p;
}

// Sparse: one CTA per unit; when the units leave SMs idle, or a unit has
// more positions than one CTA's row table holds (8192, or 4096 with four
// row tiles), the positions of each unit are split into equal ranges and
// merged by a combine kernel.
// Row-table bytes of the sparse kernel's CTA for (d, row tiles), taken
// from the kernel's configuration so that host planning and shared-memory
// layout cannot drift apart.
long long attn_tab_bytes(int d, int mt) {
  if (d == 64) {
    switch (mt) {
      case 1: return AttnCfg<64, 1>::TAB_BYTES;
      case 2: return AttnCfg<64, 2>::TAB_BYTES;
      case 3: return AttnCfg<64, 3>::TAB_BYTES;
      default: return AttnCfg<64, 4>::TAB_BYTES;
    }
  }
  switch (mt) {
    case 1: return AttnCfg<128, 1>::TAB_BYTES;
    case 2: return AttnCfg<128, 2>::TAB_BYTES;
    case 3: return AttnCfg<128, 3>::TAB_BYTES;
    default: return AttnCfg<128, 4>::TAB_BYTES;
  }
}

AttnPlan plan_sparse(int b, int hq, int hkv, int d, int w, int k, bool win) {
  AttnPlan p = plan_units(hq, hkv, w, b, k);
  const int tiles = (k + 63) / 64;
  p.splits = 1;
  p.chunk = 64;
  p.wide = false;
  if (tiles > 0 && p.units > 0) {
    const long long slots = (long long)attn_slots(false, d, p.mt);
    long long s = p.units >= slots ? 1 : slots / p.units;
    s = std::min<long long>(s, tiles);
    // Row table of one CTA (the kernel's own TAB_BYTES): 64-bit offsets for
    // up to cap64 tiles, 32-bit row codes (the WIDE variant; not with the
    // window) for up to cap32.
    const long long tab_bytes = attn_tab_bytes(d, p.mt);
    const long long cap64 = tab_bytes / 8 / 64, cap32 = tab_bytes / 4 / 64;
    long long ct = (tiles + s - 1) / s;
    if (ct > cap64) {
      if (win) {
        ct = cap64;
      } else {
        p.wide = true;
        ct = std::min(ct, cap32);
      }
    }
    p.splits = (int)((tiles + ct - 1) / ct);
    p.chunk = (int)(ct * 64);
  }
  if (p.splits > 1) {
    const size_t prows = (size_t)p.units * p.splits * 16 * p.mt;
    p.ws_o = align256(prows * d * sizeof(float));
    p.ws_ml = align256(prows * sizeof(float2));
  }
  return p;
}

// Build-time tunable: an upper bound on the CTAs one dense launch keeps
// resident (0: all that fit).
#ifndef DUSTIN_ATTN_GRID_CAP
#define DUSTIN_ATTN_GRID_CAP 0
#endif

// Dense: stream-K over tiles.  G is the number of CTAs resident at once,
// raised where a CTA's range would overflow its page table (512 tiles).
AttnPlan plan_dense(int b, int hq, int hkv, int d, int w, int n, bool win) {
  AttnPlan p = plan_units(hq, hkv, w, b, n);
  // History tiles, then (with the window merged in) one window tile.
  p.tph = (n + 63) / 64;
  p.tpu = std::max(1, p.tph + (win ? 1 : 0));
  const long long T = p.units * p.tpu;
  if (T <= 0) return p;
  long long slots = (long long)attn_slots(true, d, p.mt);
#if DUSTIN_ATTN_GRID_CAP > 0
  slots = std::min<long long>(slots, DUSTIN_ATTN_GRID_CAP);
#endif
  const long long cap = SkCfg<128, 3>::MAX_TILES;   // tiles one CTA's page table holds
  p.grid = std::max(std::min(slots, T), (T + cap - 1) / cap);
  // Every range boundary c T / G falls on a unit boundary when G divides
  // the unit count (conservatively "split" otherwise).
  p.split = p.tpu > 1 && p.units % p.grid != 0;
  if (p.split) {
    const size_t prows = (size_t)(2 * p.grid) * 16 * p.mt;
    p.ws_o = align256(prows * d * sizeof(float));
    p.ws_ml = align256(prows * sizeof(float2));
    p.ws_cnt = align256((size_t)p.units * sizeof(unsigned long long));
  }
  return p;
}

// A fresh nonzero 40-bit tag per dense call, so counter words left by
// earlier calls (or never written) read as zero.
unsigned long long next_epoch() {
  static std::atomic<unsigned long long> ctr{
      (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count()};
  constexpr unsigned long long kMask = (1ull << 40) - 1;
  unsigned long long e;
  do {
    e = ctr.fetch_add(1) & kMask;
  } while (e == 0);
  return e;
}

int check_attn_shape(int b, int hq, int hkv, int d, int w, int n,
                     const char* what) {
  if (b < 0 || n < 0 || w < 1 || hq < 1 || hkv < 1)
    return fail(DUSTIN_ERR_SHAPE, "%s: b=%d n=%d w=%d h_q=%d h_kv=%d", what, b,
                n, w, hq, hkv);
  if (hq % hkv)
    return fail(DUSTIN_ERR_SHAPE, "%s: h_q %d not a multiple of h_kv %d", what,
                hq, hkv);
  if (d != 64 && d != 128)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: d=%d (64 or 128)", what, d);
  const long long blocks = (long long)b * hkv *
                           (((long long)(hq / hkv) * w + 63) / 64);
  if (blocks > (1LL << 24))
    return fail(DUSTIN_ERR_SHAPE, "%s: problem too large", what);
  return DUSTIN_OK;
}

// The window's own K/V: [b][h_kv][w][d] through a contiguous descriptor.
int check_win(const dustin_kv* win, int d, const char* what) {
  if (!win->k || !win->v)
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: win.k and win.v are required", what);
  if (!aligned16(win->k) || !aligned16(win->v))
    return fail(DUSTIN_ERR_ALIGNMENT, "%s: win base not 16-byte aligned", what);
  if (win->page_table)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: the window cannot be paged", what);
  if (win->stride_b < 0 || win->stride_h < 0 || win->stride_n < d)
    return fail(DUSTIN_ERR_SHAPE, "%s: bad win strides", what);
  if (win->stride_b % 8 || win->stride_h % 8 || win->stride_n % 8)
    return fail(DUSTIN_ERR_ALIGNMENT,
                "%s: win strides must be multiples of 8 elements", what);
  return DUSTIN_OK;
}

int run_attn(bool dense, int b, int hq, int hkv, int d, int w, int n, int k,
             const void* q, const dustin_kv* kv, const int32_t* idx,
             const dustin_kv* win, float scale, void* o, float* lse, void* ws,
             size_t ws_bytes, unsigned flags, void* stream) {
  const char* what = dense ? (win ? "dustin_full_verify_attn_window" : "dustin_full_verify_attn")
                           : (win ? "dustin_sparse_verify_attn_window"
                                  : "dustin_sparse_verify_attn");
  int rc = check_attn_shape(b, hq, hkv, d, w, n, what);
  if (rc) return rc;
  if (!dense && (k < 0 || k > n))
    return fail(DUSTIN_ERR_SHAPE, "%s: k=%d must be in [0, n=%d]", what, k, n);
  if (b == 0) return DUSTIN_OK;
  if (!q || !o || !lse)
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: q, o and lse are required", what);
  if (!dense && k > 0 && !idx)
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: idx is NULL", what);
  if (!aligned16(q) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (idx && (reinterpret_cast<uintptr_t>(idx) & 3u)))
    return fail(DUSTIN_ERR_ALIGNMENT, "%s: q/o need 16-byte, lse/idx 4-byte alignment",
                what);
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: scale must be finite and > 0", what);
  if (flags & ~DUSTIN_ATTN_KV_READY)
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: unknown flags 0x%x", what, flags);
  rc = check_kv(kv, b, n, d, true, what);
  if (rc) return rc;
  if (win && (rc = check_win(win, d, what))) return rc;
  const bool paged = kv->page_table != nullptr;
  cudaError_t e;
  if (!dense) {
    if (paged && (long long)kv->num_pages * kv->page_size > 0x7fffffffLL)
      return fail(DUSTIN_ERR_UNSUPPORTED, "%s: page pool of 2^31 rows or more", what);
    const AttnPlan p = plan_sparse(b, hq, hkv, d, w, k, win != nullptr);
    if (p.units * p.splits > 0x7fffffffLL)
      return fail(DUSTIN_ERR_SHAPE, "%s: grid too large", what);
    const size_t need = p.workspace();
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws)))
      return fail(DUSTIN_ERR_WORKSPACE,
                  "%s: workspace %zu bytes, need %zu (16-byte aligned)", what,
                  ws_bytes, need);
    AttnArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.o = static_cast<__nv_bfloat16*>(o);
    a.lse = lse;
    a.kv = to_view(*kv);
    a.idx = idx;
    a.b = b;
    a.hq = hq;
    a.hkv = hkv;
    a.w = w;
    a.n = n;
    a.npos = k;
    a.group = hq / hkv;
    a.rows = a.group * w;
    a.row_blocks = p.row_blocks;
    a.splits = p.splits;
    a.chunk = p.chunk;
    a.scale_log2 = scale * kLog2e;
    a.kv_ready = (flags & DUSTIN_ATTN_KV_READY) ? 1 : 0;
    a.has_win = win ? 1 : 0;
    a.wide = p.wide ? 1 : 0;
    if (win) a.win = to_view(*win);
    a.ws_o = need ? static_cast<float*>(ws) : nullptr;
    a.ws_ml = need ? reinterpret_cast<float2*>(static_cast<char*>(ws) + p.ws_o)
                   : nullptr;
    e = launch_attn_sparse(a, d, p.mt, paged, (cudaStream_t)stream);
  } else {
    const AttnPlan p = plan_dense(b, hq, hkv, d, w, n, win != nullptr);
    const long long T = p.units * p.tpu;
    if (p.units > 0x7fffffffLL || p.grid > 0x7fffffffLL || T > (1LL << 40) ||
        p.grid * T > (1LL << 62) ||
        p.tpu / std::max(1LL, T / std::max(1LL, p.grid)) + 2 > (1LL << 24) - 1)
      return fail(DUSTIN_ERR_SHAPE, "%s: problem too large", what);
    const size_t need = p.workspace();
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws)))
      return fail(DUSTIN_ERR_WORKSPACE,
                  "%s: workspace %zu bytes, need %zu (16-byte aligned)", what,
                  ws_bytes, need);
    AttnSkArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.o = static_cast<__nv_bfloat16*>(o);
    a.lse = lse;
    a.kv = to_view(*kv);
    a.b = b;
    a.hq = hq;
    a.hkv = hkv;
    a.w = w;
    a.n = n;
    a.group = hq / hkv;
    a.rows = a.group * w;
    a.row_blocks = p.row_blocks;
    a.units = (int)p.units;
    a.tpu = p.tpu;
    a.tph = p.tph;
    a.has_win = win ? 1 : 0;
    if (win) a.win = to_view(*win);
    a.grid = (int)p.grid;
    a.scale_log2 = scale * kLog2e;
    a.kv_ready = (flags & DUSTIN_ATTN_KV_READY) ? 1 : 0;
    char* wsb = static_cast<char*>(ws);
    a.ws_o = need ? reinterpret_cast<float*>(wsb) : nullptr;
    a.ws_ml = need ? reinterpret_cast<float2*>(wsb + p.ws_o) : nullptr;
    a.counters = need ? reinterpret_cast<unsigned long long*>(wsb + p.ws_o + p.ws_ml)
                      : nullptr;
    a.epoch = next_epoch();
    e = launch_attn_dense(a, d, p.mt, paged, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, what);
  return DUSTIN_OK;
}

}  // namespace

// Argument checks of the scoring calls (everything but the workspace):
// DUSTIN_OK with *empty set when there is nothing to do.
int check_score_args(int b, int n, int d, int n_pairs, int rows, const void* q,
                     const dustin_kv* kv, const int32_t* kv_head, float scale,
                     const float* s_out, const char* what, bool* paged, bool* empty) {
  *paged = false;
  *empty = false;
  if (b < 0 || n < 0) return fail(DUSTIN_ERR_SHAPE, "%s: b=%d n=%d", what, b, n);
  if (d != 64 && d != 128)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: d=%d (64 or 128)", what, d);
  if (n_pairs < 1 || n_pairs > kMaxPairs)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: n_pairs=%d (1..%d)", what, n_pairs,
                kMaxPairs);
  if (rows < 1 || rows > 16)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: rows=%d (1..16)", what, rows);
  if (n_pairs * rows > 1024)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: n_pairs*rows > 1024", what);
  if (b == 0 || n == 0) {
    *empty = true;
    return DUSTIN_OK;
  }
  if (!q || !kv || !kv_head || !s_out)
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: q, kv, kv_head, s_out required", what);
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(s_out) & 3u))
    return fail(DUSTIN_ERR_ALIGNMENT, "%s: q needs 16-byte alignment", what);
  if (!std::isfinite(scale))
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: scale is not finite", what);
  if ((long long)n_pairs * b * ((n + score_chunk() - 1) / score_chunk()) > 0x7fffffffLL ||
      (long long)b > 65535)
    return fail(DUSTIN_ERR_SHAPE, "%s: problem too large", what);
  for (int p = 0; p < n_pairs; ++p) {
    int rc = check_kv(&kv[p], b, n, d, false, what);
    if (rc) return rc;
    if (kv_head[p] < 0)
      return fail(DUSTIN_ERR_SHAPE, "%s: kv_head[%d]=%d", what, p, kv_head[p]);
    if (p > 0 && ((kv[p].page_table != nullptr) != *paged))
      return fail(DUSTIN_ERR_UNSUPPORTED, "%s: mixed paged/contiguous pairs", what);
    *paged = kv[p].page_table != nullptr;
  }
  return DUSTIN_OK;
}

void note_launches(int count) { g_launches.fetch_add((uint64_t)count); }

int record_error(int status, const char* message) {
  return fail(status, "%s", message);
}

}  // namespace dustin

using namespace dustin;

extern "C" {

const char* dustin_status_string(int status) {
  switch (status) {
    case DUSTIN_OK: return "ok";
    case DUSTIN_ERR_INVALID_ARG: return "invalid argument";
    case DUSTIN_ERR_SHAPE: return "bad shape";
    case DUSTIN_ERR_UNSUPPORTED: return "unsupported configuration";
    case DUSTIN_ERR_WORKSPACE: return "workspace missing or too small";
    case DUSTIN_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case DUSTIN_ERR_CUDA: return "CUDA error";
    case DUSTIN_ERR_DEVICE: return "device-side check failed";
    default: return "unknown status";
  }
}

const char* dustin_last_error(void) { return g_err; }

int dustin_version(void) { return 100; }

uint64_t dustin_launch_count(void) { return g_launches.load(); }

namespace dustin {
namespace {

__device__ unsigned int g_selftest_flags;

// One warp waits on an mbarrier that expects one arrival nobody makes.
__global__ void wait_selftest_kernel(long long limit) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_fence_init();
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  if (!mbar_wait(b, 0, limit) && threadIdx.x == 0)
    atomicOr(&g_selftest_flags, DUSTIN_DEVFLAG_WAIT_TIMEOUT);
}

cudaError_t take_selftest_flags(unsigned* flags) {
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_selftest_flags, sizeof(v));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_selftest_flags, &zero, sizeof(zero));
  *flags |= v;
  return e;
}

}  // namespace
}  // namespace dustin

int dustin_wait_selftest(int64_t limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles > (1LL << 31))
    return fail(DUSTIN_ERR_SHAPE, "dustin_wait_selftest: limit %lld cycles",
                (long long)limit_cycles);
  cudaError_t e = launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0,
                             (cudaStream_t)stream, (long long)limit_cycles);
  if (e != cudaSuccess) return cuda_fail(e, "dustin_wait_selftest");
  note_launches(1);
  return DUSTIN_OK;
}

int dustin_device_status(uint32_t* flags) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "dustin_device_status");
  unsigned f = 0;
  if ((e = take_selftest_flags(&f)) != cudaSuccess ||
      (e = take_attn_sparse_flags(&f)) != cudaSuccess ||
      (e = take_attn_dense_flags(&f)) != cudaSuccess ||
      (e = take_attn_ml_flags(&f)) != cudaSuccess ||
      (e = take_quest_flags(&f)) != cudaSuccess ||
      (e = take_score_flags(&f)) != cudaSuccess)
    return cuda_fail(e, "dustin_device_status");
  if (flags) *flags = f;
  if (f) return fail(DUSTIN_ERR_DEVICE, "device flags 0x%x", f);
  return DUSTIN_OK;
}

size_t dustin_score_heads_workspace_size(int b, int n, int n_pairs, int rows) {
  if (b <= 0 || n <= 0 || n_pairs <= 0 || rows <= 0) return 0;
  const long long chunk = score_chunk();
  const long long nch = (n + chunk - 1) / chunk;
  const size_t prs = (size_t)n_pairs * rows * b;
  return align256(prs * n * sizeof(float)) + align256(prs * nch * sizeof(float2));
}

int dustin_score_heads(int b, int n, int d, int n_pairs, int rows,
                       const void* q, const dustin_kv* kv,
                       const int32_t* kv_head, float scale, float* s_out,
                       void* ws, size_t ws_bytes, void* stream) {
  const char* what = "dustin_score_heads";
  bool paged = false, empty = false;
  const int rc = check_score_args(b, n, d, n_pairs, rows, q, kv, kv_head, scale, s_out,
                                  what, &paged, &empty);
  if (rc || empty) return rc;
  const size_t need = dustin_score_heads_workspace_size(b, n, n_pairs, rows);
  if (!ws || ws_bytes < need || !aligned16(ws))
    return fail(DUSTIN_ERR_WORKSPACE, "%s: workspace %zu bytes, need %zu", what,
                ws_bytes, need);
  ScoreArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.s_out = s_out;
  a.b = b;
  a.n = n;
  a.n_pairs = n_pairs;
  a.rows = rows;
  a.chunk = score_chunk();
  a.nchunks = (n + a.chunk - 1) / a.chunk;
  a.scale_log2 = scale * kLog2e;
  const size_t prs = (size_t)n_pairs * rows * b;
  a.logits = static_cast<float*>(ws);
  a.stats = reinterpret_cast<float2*>(static_cast<char*>(ws) +
                                      align256(prs * n * sizeof(float)));
  for (int p = 0; p < n_pairs; ++p) {
    a.pairs[p].kv = to_view(kv[p]);
    a.pairs[p].kv_head = kv_head[p];
    for (int q = 0; q < p; ++q)
      if (kv[q].k == kv[p].k && kv_head[q] == kv_head[p]) a.keys_shared = 1;
  }
  cudaError_t e = launch_score(a, d, paged, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return DUSTIN_OK;
}

int dustin_hybrid_topk(int b, int n, int k, int n_sink, int n_recent,
                       double alpha, int m, int norm, const float* s_draft,
                       const float* s_target, int32_t* idx, void* stream) {
  const char* what = "dustin_hybrid_topk";
  if (b < 0 || n < 0 || k < 0)
    return fail(DUSTIN_ERR_SHAPE, "%s: b=%d n=%d k=%d", what, b, n, k);
  if (n > kSelectMaxN)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: n=%d > %d", what, n, kSelectMaxN);
  if (norm != DUSTIN_NORM_NONE && norm != DUSTIN_NORM_L1)
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: norm=%d", what, norm);
  if (!std::isfinite(alpha))
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: alpha not finite", what);
  if (b == 0 || n == 0 || k == 0) return DUSTIN_OK;
  if (!idx) return fail(DUSTIN_ERR_INVALID_ARG, "%s: idx is NULL", what);
  if (k < n) {
    if (!s_draft && !s_target)
      return fail(DUSTIN_ERR_INVALID_ARG, "%s: both score vectors NULL", what);
    const int ns = std::min(std::max(n_sink, 0), n);
    const int hi = n - std::min(std::max(n_recent, 0), n);
    const int forced = hi <= ns ? n : ns + (n - hi);
    if (forced > k)
      return fail(DUSTIN_ERR_SHAPE, "%s: %d protected positions exceed k=%d", what,
                  forced, k);
    if (m >= 0) {
      const int budget = k - forced;
      const int m_eff = std::min(m, budget);
      if (m_eff > 0 && !s_draft)
        return fail(DUSTIN_ERR_INVALID_ARG, "%s: m mode needs s_draft", what);
      if (budget - m_eff > 0 && !s_target)
        return fail(DUSTIN_ERR_INVALID_ARG, "%s: m mode needs s_target", what);
    }
  }
  SelectArgs a;
  a.sd = s_draft;
  a.st = s_target;
  a.idx = idx;
  a.alpha = alpha;
  a.b = b;
  a.n = n;
  a.k = k;
  a.n_sink = n_sink;
  a.n_recent = n_recent;
  a.m = m;
  a.norm = norm;
  cudaError_t e = launch_select(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return DUSTIN_OK;
}

size_t dustin_sparse_verify_attn_workspace_size(int b, int h_q, int h_kv, int d,
                                                int w, int k) {
  if (b <= 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv || w <= 0 || k < 0 ||
      (d != 64 && d != 128))
    return 0;
  // Covers the call with and without the window merged in.
  return std::max(plan_sparse(b, h_q, h_kv, d, w, k, false).workspace(),
                  plan_sparse(b, h_q, h_kv, d, w, k, true).workspace());
}

int dustin_sparse_verify_attn(int b, int h_q, int h_kv, int d, int w, int n,
                              int k, const void* q, const dustin_kv* kv,
                              const int32_t* idx, float scale, void* o,
                              float* lse, void* ws, size_t ws_bytes,
                              unsigned flags, void* stream) {
  return run_attn(false, b, h_q, h_kv, d, w, n, k, q, kv, idx, nullptr, scale, o,
                  lse, ws, ws_bytes, flags, stream);
}

int dustin_sparse_verify_attn_window(int b, int h_q, int h_kv, int d, int w,
                                     int n, int k, const void* q,
                                     const dustin_kv* kv, const int32_t* idx,
                                     const dustin_kv* win, float scale, void* o,
                                     float* lse, void* ws, size_t ws_bytes,
                                     unsigned flags, void* stream) {
  if (!win) return fail(DUSTIN_ERR_INVALID_ARG, "dustin_sparse_verify_attn_window: win is NULL");
  return run_attn(false, b, h_q, h_kv, d, w, n, k, q, kv, idx, win, scale, o, lse,
                  ws, ws_bytes, flags, stream);
}

int dustin_sparse_verify_attn_layers(int n_layers, int b, int h_q, int h_kv, int d,
                                     int w, int n, int k, const void* const* q,
                                     const dustin_kv* kv, const int32_t* idx,
                                     float scale, void* const* o, float* const* lse,
                                     unsigned flags, void* stream) {
  const char* what = "dustin_sparse_verify_attn_layers";
  if (n_layers < 0) return fail(DUSTIN_ERR_SHAPE, "%s: n_layers=%d", what, n_layers);
  int rc = check_attn_shape(b, h_q, h_kv, d, w, n, what);
  if (rc) return rc;
  if (k < 0 || k > n)
    return fail(DUSTIN_ERR_SHAPE, "%s: k=%d must be in [0, n=%d]", what, k, n);
  constexpr int kMlMaxK = SkCfg<128, 3>::MAX_TAB;   // offset-table entries of one item
  if (k > kMlMaxK)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: k=%d (at most %d per call)", what, k, kMlMaxK);
  if (n_layers == 0 || b == 0) return DUSTIN_OK;
  if (!q || !kv || !o || !lse)
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: q, kv, o and lse arrays are required", what);
  if (k > 0 && !idx) return fail(DUSTIN_ERR_INVALID_ARG, "%s: idx is NULL", what);
  if (idx && (reinterpret_cast<uintptr_t>(idx) & 3u))
    return fail(DUSTIN_ERR_ALIGNMENT, "%s: idx needs 4-byte alignment", what);
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: scale must be finite and > 0", what);
  if (flags & ~DUSTIN_ATTN_KV_READY)
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: unknown flags 0x%x", what, flags);
  const bool paged = kv[0].page_table != nullptr;
  for (int l = 0; l < n_layers; ++l) {
    if (!q[l] || !o[l] || !lse[l])
      return fail(DUSTIN_ERR_INVALID_ARG, "%s: layer %d: q, o and lse are required", what, l);
    if (!aligned16(q[l]) || !aligned16(o[l]) || (reinterpret_cast<uintptr_t>(lse[l]) & 3u))
      return fail(DUSTIN_ERR_ALIGNMENT, "%s: layer %d: q/o need 16-byte, lse 4-byte alignment",
                  what, l);
    if ((rc = check_kv(&kv[l], b, n, d, true, what))) return rc;
    if ((kv[l].page_table != nullptr) != paged)
      return fail(DUSTIN_ERR_INVALID_ARG, "%s: layers mix paged and contiguous caches", what);
  }
  const AttnPlan p = plan_units(h_q, h_kv, w, b, k);
  const long long slots = (long long)attn_slots(true, d, p.mt);
  for (int l0 = 0; l0 < n_layers; l0 += kMlMaxLayers) {
    const int nl = std::min(kMlMaxLayers, n_layers - l0);
    AttnMlArgs a;
    a.idx = idx;
    a.layers = nl;
    a.b = b;
    a.hq = h_q;
    a.hkv = h_kv;
    a.w = w;
    a.n = n;
    a.k = k;
    a.group = h_q / h_kv;
    a.rows = a.group * w;
    a.row_blocks = p.row_blocks;
    a.units = (int)p.units;
    a.tpu = p.tpu;
    a.scale_log2 = scale * kLog2e;
    for (int l = 0; l < nl; ++l) {
      a.layer[l].q = static_cast<const __nv_bfloat16*>(q[l0 + l]);
      a.layer[l].o = static_cast<__nv_bfloat16*>(o[l0 + l]);
      a.layer[l].lse = lse[l0 + l];
      a.layer[l].kv = to_view(kv[l0 + l]);
    }
    const long long items = (long long)nl * p.units;
    const int grid = (int)std::min(slots, items);
    cudaError_t e = launch_attn_ml(a, d, p.mt, paged, grid, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, what);
  }
  return DUSTIN_OK;
}

size_t dustin_quest_stats_size(int b, int h_kv, int d, int n, int page) {
  if (b <= 0 || h_kv <= 0 || n < 0 || page <= 0 || (d != 64 && d != 128)) return 0;
  const size_t pages = ((size_t)n + page - 1) / page;
  return (size_t)b * h_kv * pages * 2 * d * sizeof(uint16_t);
}

int dustin_quest_page_stats(int b, int h_kv, int d, int n, int page,
                            const dustin_kv* kv, void* stats, void* stream) {
  const char* what = "dustin_quest_page_stats";
  if (b < 0 || h_kv < 1 || n < 0 || page < 1)
    return fail(DUSTIN_ERR_SHAPE, "%s: b=%d h_kv=%d n=%d page=%d", what, b, h_kv, n, page);
  if (d != 64 && d != 128)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: d=%d (64 or 128)", what, d);
  if (b == 0 || n == 0) return DUSTIN_OK;
  if (!stats || !aligned16(stats))
    return fail(DUSTIN_ERR_ALIGNMENT, "%s: stats must be 16-byte aligned", what);
  int rc = check_kv(kv, b, n, d, false, what);
  if (rc) return rc;
  QuestArgs a{};
  a.kv = to_view(*kv);
  a.stats = static_cast<__nv_bfloat16*>(stats);
  a.b = b;
  a.hkv = h_kv;
  a.n = n;
  a.page = page;
  a.n_pages = (n + page - 1) / page;
  cudaError_t e = launch_quest_stats(a, d, kv->page_table != nullptr, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return DUSTIN_OK;
}

int dustin_quest_page_scores(int b, int h_q, int h_kv, int d, int n, int page,
                             const void* q, const void* stats, float* scores,
                             void* stream) {
  const char* what = "dustin_quest_page_scores";
  if (b < 0 || h_q < 1 || h_kv < 1 || h_q % h_kv || n < 0 || page < 1)
    return fail(DUSTIN_ERR_SHAPE, "%s: b=%d h_q=%d h_kv=%d n=%d page=%d", what, b, h_q,
                h_kv, n, page);
  if (d != 64 && d != 128)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: d=%d (64 or 128)", what, d);
  if (h_q / h_kv > 64)
    return fail(DUSTIN_ERR_UNSUPPORTED, "%s: more than 64 query heads per kv head", what);
  if (b == 0 || n == 0) return DUSTIN_OK;
  if (!q || !stats || !scores)
    return fail(DUSTIN_ERR_INVALID_ARG, "%s: q, stats and scores are required", what);
  if (!aligned16(stats) || (reinterpret_cast<uintptr_t>(q) & 1u) ||
      (reinterpret_cast<uintptr_t>(scores) & 3u))
    return fail(DUSTIN_ERR_ALIGNMENT, "%s: stats 16-byte, q 2-byte, scores 4-byte aligned",
                what);
  QuestArgs a{};
  a.stats_in = static_cast<const __nv_bfloat16*>(stats);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.scores = scores;
  a.b = b;
  a.hq = h_q;
  a.hkv = h_kv;
  a.n = n;
  a.page = page;
  a.n_pages = (n + page - 1) / page;
  cudaError_t e = launch_quest_scores(a, d, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, what);
  return DUSTIN_OK;
}

size_t dustin_full_verify_attn_workspace_size(int b, int h_q, int h_kv, int d,
                                              int w, int n) {
  if (b <= 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv || w <= 0 || n < 0 ||
      (d != 64 && d != 128))
    return 0;
  // Covers the call with and without the window merged in.
  return std::max(plan_dense(b, h_q, h_kv, d, w, n, false).workspace(),
                  plan_dense(b, h_q, h_kv, d, w, n, true).workspace());
}

int dustin_full_verify_attn(int b, int h_q, int h_kv, int d, int w, int n,
                            const void* q, const dustin_kv* kv, float scale,
                            void* o, float* lse, void* ws, size_t ws_bytes,
                            unsigned flags, void* stream) {
  return run_attn(true, b, h_q, h_kv, d, w, n, n, q, kv, nullptr, nullptr, scale, o,
                  lse, ws, ws_bytes, flags, stream);
}

int dustin_full_verify_attn_window(int b, int h_q, int h_kv, int d, int w, int n,
                                   const void* q, const dustin_kv* kv,
                                   const dustin_kv* win, float scale, void* o,
                                   float* lse, void* ws, size_t ws_bytes,
                                   unsigned flags, void* stream) {
  if (!win) return fail(DUSTIN_ERR_INVALID_ARG, "dustin_full_verify_attn_window: win is NULL");
  return run_attn(true, b, h_q, h_kv, d, w, n, n, q, kv, nullptr, win, scale, o, lse,
                  ws, ws_bytes, flags, stream);
}

}  // extern "C"
