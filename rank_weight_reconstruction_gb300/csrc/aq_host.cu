// aq_host.cu -- the C ABI declared in include/aq.h: argument validation, work planning
// (tile sizes, grid, pipeline depth), TMA descriptor encoding and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>

#include "aq.h"
#include "aq_internal.h"

using namespace aq;

namespace {

thread_local std::string t_err;
thread_local int32_t t_last_path = 0;
thread_local int32_t t_launches = 0;
std::atomic<int> g_path{AQ_PATH_AUTO};
// aq_selftest_prefill_timeout: on this thread, the next prefill GEMM waits for a t-flag count
// no tile reaches, with this limit (0: the normal plan)
thread_local uint64_t t_test_unreachable_t_ns = 0;

constexpr int kDecodeMaxM = kDecMaxTok;               // mma.sync decode kernel up to this M
constexpr int kDec2Staged = 1;   // cluster decode: x and V in the W0 stages (no gated input)
// The swapped-operand GEMM (output rows as accumulator lanes) is taken automatically where it was
// measured faster than the token-lane GEMM (bench.py --sweep, gate-like 6912 x 1152 and down-like
// 1152 x 6912, r = 0..256): calls of at least this many tokens whose families have few 128-row
// tiles over a deep K (down-like at 4096 tokens: 54-99 us against 74-116 us). At 64-512 tokens
// the token-lane GEMM was as fast or faster on both shapes, and at 8192 tokens too (the
// Gemma-3-1B down projection at r = 64: 122 us against 149 us).
constexpr int64_t kSwapMinM = 1024;
constexpr int64_t kSwapMaxM = 4096;
constexpr int64_t kSwapMaxRowTiles = 16;
constexpr int kSwapMinK = 4096;
constexpr int kGemmMinMBigW0 = 16;                    // ... but from this M the GEMM takes calls
constexpr int64_t kGemmBigW0Bytes = 128ll << 20;      // whose W0 has at least this many bytes
constexpr uint64_t kTimeoutNs = 1000ull * 1000 * 1000;  // limit of one in-kernel wait: 1 s
constexpr size_t kSmemSlack = 1024;                   // room to align the dynamic smem base

aq_status fail(aq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_err = buf;
  return st;
}

aq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(AQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------------
// per-device facts, queried once
// ---------------------------------------------------------------------------------
struct DevInfo {
  bool ready = false;
  int sms = 0;
  size_t smem_optin = 0;
  int gemm_pairs = 0;   // CTA pairs of the prefill GEMM that fit at once (0: no pairs)
  int32_t* status = nullptr;
};

std::mutex g_dev_mu;
DevInfo g_dev[64];

aq_status device_info(DevInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(AQ_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0, smem = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) ||
        (e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)))
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
      return fail(AQ_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a (GB300)",
                  dev, major, minor);
    if ((e = configure_kernels(dev, static_cast<size_t>(smem))))
      return cuda_fail(e, "cudaFuncSetAttribute");
    int32_t* st = device_status_ptr(dev, &e);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    int pairs = 0;
    if (static_cast<size_t>(smem) < kGemmPairMinSmem || gemm_max_clusters(kGemmPairMinSmem, 2, &pairs) != cudaSuccess)
      pairs = 0;
    cudaGetLastError();   // a failed occupancy query only disables the pairs
    d.gemm_pairs = pairs;
    d.sms = sms;
    d.smem_optin = static_cast<size_t>(smem);
    d.status = st;
    d.ready = true;
  }
  *out = &d;
  return AQ_OK;
}

// ---------------------------------------------------------------------------------
// TMA descriptors
// ---------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(aq_status* st) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  *st = fn ? AQ_OK : fail(AQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  return fn;
}

// bf16 matrix [outer, inner] with row stride ld (elements); box {64, box_outer}; 128-byte
// swizzle; out-of-bounds elements read as zero.
aq_status tmap_2d(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t ld,
                  int box_outer, const char* what) {
  aq_status st;
  EncodeTiledFn fn = encode_fn(&st);
  if (!fn) return st;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2u};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(AQ_ERR_CUDA, "cuTensorMapEncodeTiled(%s: %lld x %lld, ld %lld, box rows %d) failed: %d", what,
                (long long)outer, (long long)inner, (long long)ld, box_outer, (int)r);
  return AQ_OK;
}

// bf16 matrix [outer, inner] with row stride ld, box {box_inner, box_outer}, no swizzle
// (rows land densely in shared memory); out-of-bounds elements read as zero.
aq_status tmap_2d_plain(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t ld, int box_inner,
                        int box_outer, const char* what) {
  aq_status st;
  EncodeTiledFn fn = encode_fn(&st);
  if (!fn) return st;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2u};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(AQ_ERR_CUDA, "cuTensorMapEncodeTiled(%s: %lld x %lld, ld %lld, box %d x %d) failed: %d", what,
                (long long)outer, (long long)inner, (long long)ld, box_outer, box_inner, (int)r);
  return AQ_OK;
}

// bf16 matrix [outer, inner] (inner a multiple of 64) seen as [outer, inner / 64, 64], box
// {64, box_mid, box_outer}, 128-byte swizzle: one request fetches box_mid consecutive
// 64-wide blocks of box_outer rows.
aq_status tmap_3d(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t ld, int box_mid,
                  int box_outer, const char* what) {
  aq_status st;
  EncodeTiledFn fn = encode_fn(&st);
  if (!fn) return st;
  cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(inner / 64), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[2] = {128u, static_cast<cuuint64_t>(ld) * 2u};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_mid), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(AQ_ERR_CUDA, "cuTensorMapEncodeTiled(%s 3-D: %lld x %lld, ld %lld, box %d x %d) failed: %d", what,
                (long long)outer, (long long)inner, (long long)ld, box_outer, box_mid, (int)r);
  return AQ_OK;
}

// ---------------------------------------------------------------------------------
// validation helpers
// ---------------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bytes spanned by a row-strided bf16 matrix.
struct Span {
  uintptr_t base = 0;
  int64_t rows = 0, cols = 0, ld = 0;
  const char* name = "";
  bool empty() const { return base == 0 || rows <= 0 || cols <= 0; }
  uintptr_t lo() const { return base; }
  uintptr_t hi() const { return base + static_cast<uintptr_t>(((rows - 1) * ld + cols) * 2); }
};

Span span(const void* p, int64_t rows, int64_t cols, int64_t ld, const char* name) {
  Span s;
  s.base = reinterpret_cast<uintptr_t>(p);
  s.rows = rows;
  s.cols = cols;
  s.ld = ld;
  s.name = name;
  return s;
}

// Exact for equal leading dimensions (e.g. q/k/v outputs as column slices of one
// buffer); conservative otherwise.
bool overlaps(const Span& a, const Span& b) {
  if (a.empty() || b.empty()) return false;
  if (a.hi() <= b.lo() || b.hi() <= a.lo()) return false;
  if (a.ld != b.ld || a.ld <= 0) return true;
  const int64_t diff = static_cast<int64_t>(b.base) - static_cast<int64_t>(a.base);
  if (diff % 2 != 0) return true;
  const int64_t l = a.ld;
  const int64_t d = diff / 2;
  const int64_t c = ((d % l) + l) % l;  // column of b's first element within a's row grid
  // b covers columns [c, c + b.cols) modulo l; a covers [0, a.cols)
  if (b.cols >= l || a.cols >= l) return true;
  auto inter = [](int64_t x0, int64_t x1, int64_t y0, int64_t y1) { return x0 < y1 && y0 < x1; };
  if (c + b.cols <= l) return inter(c, c + b.cols, 0, a.cols);
  return inter(c, l, 0, a.cols) || inter(0, c + b.cols - l, 0, a.cols);
}

aq_status check_theta(const aq_theta* th, const char* who) {
  if (!th) return fail(AQ_ERR_INVALID_ARG, "%s: theta is NULL", who);
  if (!th->W0 || !th->s) return fail(AQ_ERR_INVALID_ARG, "%s: W0 and s must be non-NULL", who);
  if (th->out < 1 || th->in < 1) return fail(AQ_ERR_SHAPE, "%s: out=%d in=%d must be >= 1", who, th->out, th->in);
  if (th->in > 65536 * 64) return fail(AQ_ERR_SHAPE, "%s: in=%d exceeds the supported maximum", who, th->in);
  if (th->r < 0) return fail(AQ_ERR_SHAPE, "%s: r=%d is negative", who, th->r);
  if (th->r > AQ_MAX_RANK)
    return fail(AQ_ERR_UNSUPPORTED, "%s: r=%d exceeds AQ_MAX_RANK=%d", who, th->r, AQ_MAX_RANK);
  if (th->ld_w0 < th->in) return fail(AQ_ERR_SHAPE, "%s: ld_w0=%lld < in=%d", who, (long long)th->ld_w0, th->in);
  if (!aligned16(th->W0) || !aligned16(th->s) || th->ld_w0 % 8 != 0)
    return fail(AQ_ERR_ALIGNMENT, "%s: W0/s must be 16-byte aligned and ld_w0 a multiple of 8", who);
  if (th->r > 0) {
    if (!th->U || !th->V) return fail(AQ_ERR_INVALID_ARG, "%s: U and V must be non-NULL when r=%d > 0", who, th->r);
    if (th->ld_u < th->r || th->ld_v < th->r)
      return fail(AQ_ERR_SHAPE, "%s: ld_u=%lld / ld_v=%lld must be >= r=%d", who, (long long)th->ld_u,
                  (long long)th->ld_v, th->r);
    if (!aligned16(th->U) || !aligned16(th->V) || th->ld_u % 8 != 0 || th->ld_v % 8 != 0)
      return fail(AQ_ERR_ALIGNMENT, "%s: U/V must be 16-byte aligned and ld_u, ld_v multiples of 8", who);
  }
  return AQ_OK;
}

void theta_spans(const aq_theta* th, Span* out4) {
  out4[0] = span(th->W0, th->out, th->in, th->ld_w0, "W0");
  out4[1] = span(th->s, 1, th->out, th->out, "s");
  out4[2] = span(th->r > 0 ? th->U : nullptr, th->out, th->r, th->ld_u, "U");
  out4[3] = span(th->r > 0 ? th->V : nullptr, th->in, th->r, th->ld_v, "V");
}

// ---------------------------------------------------------------------------------
// workspace layout of aq_linear / aq_linear_qkv
//   [0, kSyncBytes)   sync region: zero before first use, left zero by every decode call
//                     (tile arrival counters, fp32 t accumulator)
//   [kSyncBytes, ..)  scratch, no initialisation needed (prefill: t [M, ld_t] bf16, then
//                     V^T of every family stacked as [ld_t, ldvt]: family j at row t_col[j],
//                     like its columns of t); decode uses only the sync region
// ---------------------------------------------------------------------------------
struct WsLayout {
  int64_t ld_t = 0;              // prefill: row stride of t [M, sum round_up(r_j, 8)]
  int64_t t_col[kMaxSeg] = {};   // prefill: column of family j in t
  int32_t dec_t_col[kMaxSeg] = {};  // decode: column of family j in the fp32 t accumulator
  int32_t r_total = 0;
  size_t vt_off[kMaxSeg] = {};   // prefill: byte offset of V^T of family j
  int64_t ldvt = 0;
  size_t decode_scratch = 0;
  size_t prefill_scratch = 0;
  size_t total = 0;              // what a call needs at least
  bool any_r = false;
  // split K (prefill with few output tiles over a deep K): fp32 partial sums after the rest,
  // per slice [M][ld_pz] of W0 x (family j at column pz_col[j]) then [M][ld_t] of x V
  int64_t ld_pz = 0;
  int64_t pz_col[kMaxSeg] = {};
  size_t split_base = 0;
  size_t split_slice = 0;        // bytes per slice
  int32_t split_max = 1;         // slices the preferred size holds
  size_t total_split = 0;        // preferred size: total plus split_max slices of partials
};

// Most SMs of any sm_103 part, for sizing the split partials without querying a device.
constexpr int kSplitSmsBound = 192;

// The most K slices any sm_103 part would take for this call (see the planner in
// linear_impl): only calls whose fewest possible output tiles fill at most half of the SMs.
int split_bound(const aq_theta* const* th, int n, int64_t M) {
  for (int j = 0; j < n; ++j)
    if (th[j]->r > kSplitMaxRank) return 1;
  const int64_t nkb = ceil_div(th[0]->in, kBK);
  const int64_t tok_tiles = ceil_div(M, kMmaM);
  int64_t min_tiles = 0;
  for (int j = 0; j < n; ++j) min_tiles += tok_tiles * ceil_div(th[j]->out, 256);
  if (min_tiles * 2 > kSplitSmsBound || nkb < 2 * kSplitMinKb) return 1;
  const int64_t sp = std::min<int64_t>({kMaxSplit, nkb / kSplitMinKb, kSplitSmsBound / min_tiles});
  return sp >= 2 ? static_cast<int>(sp) : 1;
}

WsLayout ws_layout(const aq_theta* const* th, int n, int64_t M) {
  WsLayout w;
  for (int j = 0; j < n; ++j) {
    w.t_col[j] = w.ld_t;
    w.dec_t_col[j] = w.r_total;
    if (th[j]->r > 0) {
      w.any_r = true;
      w.ld_t += round_up(th[j]->r, 8);
      w.r_total += th[j]->r;
    }
  }
  if (M <= 0) return w;
  if (w.any_r) {
    const size_t off = static_cast<size_t>(round_up(M * w.ld_t * 2, 256));
    w.ldvt = round_up(th[0]->in, 8);
    for (int j = 0; j < n; ++j) w.vt_off[j] = kSyncBytes + off + static_cast<size_t>(w.t_col[j] * w.ldvt * 2);
    w.prefill_scratch = off + static_cast<size_t>(round_up(w.ld_t * w.ldvt * 2, 256));
  }
  if (M <= kDecodeMaxM || w.any_r) w.total = kSyncBytes + std::max(w.decode_scratch, w.prefill_scratch);
  w.total_split = w.total;
  for (int j = 0; j < n; ++j) {
    w.pz_col[j] = w.ld_pz;
    w.ld_pz += round_up(th[j]->out, 4);
  }
  w.split_max = split_bound(th, n, M);
  w.split_base = static_cast<size_t>(round_up(static_cast<int64_t>(w.total), 256));
  w.split_slice = static_cast<size_t>(M) * static_cast<size_t>(w.ld_pz + (w.any_r ? w.ld_t : 0)) * 4u;
  if (w.split_max > 1) w.total_split = w.split_base + static_cast<size_t>(w.split_max) * w.split_slice;
  return w;
}

// ---------------------------------------------------------------------------------
// planners
// ---------------------------------------------------------------------------------
uint32_t tmem_cols_for(int n) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(n)) c <<= 1;
  return c;
}

int stages_for(uint32_t stage_bytes, size_t smem_cap, size_t fixed) {
  const size_t budget = std::min<size_t>(smem_cap, 227 * 1024) - fixed;
  int st = static_cast<int>(budget / stage_bytes);
  return std::max(2, std::min(st, kMaxStages));
}

// Prefill N tile: minimise waves x the cost of one tile.
int prefill_row_tile(const aq_theta* const* th, int n, int64_t n_tok_tiles, int sms) {
  // multiples of 64 only: the epilogue writes y in 64-column bulk stores
  static const int cand[] = {256, 192, 128, 64};
  int best = 256;
  double best_cost = 1e300;
  for (int bn : cand) {
    int64_t tiles = 0;
    for (int j = 0; j < n; ++j) tiles += n_tok_tiles * ceil_div(th[j]->out, bn);
    // A tcgen05.mma of M = 128, K = 16 costs about (N + 230) / 486 of an N = 256 one on this
    // part (measured on the 31B-class prefill: 128-wide tiles take 1.48x, 64-wide 2.8x the
    // time of 256-wide ones for the same work), so narrow tiles only pay when they save waves.
    const double cost = static_cast<double>(ceil_div(tiles, sms)) * (bn + 230);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

aq_status launch_or_fail(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_fail(e, what);
  ++t_launches;
  return AQ_OK;
}

// Cluster decode plan (M <= 16). Returns false when the call does not fit it (the caller then
// plans the row-owning decode kernel); otherwise launches and reports the launch's status.
//   * C = cluster size = K slices of about nine 64-wide k blocks each;
//   * one CTA per SM: SMs / C clusters, shared among the families in proportion to their rows,
//     rc <= 256 rows per cluster;
//   * every region in half of an SM's shared memory, so that consecutive calls' CTAs co-reside.
bool plan_decode2(const aq_theta* const* th, int n, const void* x, int64_t M, int64_t ldx, void* const* ys,
                  const int64_t* ldys, const DevInfo* dev, cudaStream_t cs, aq_status* st, const void* x2, int act) {
  const int K = th[0]->in;
  if (M < 1 || M > 16 || K % kBK != 0) return false;
  int max_r16 = 0;
  int64_t rows_total = 0;
  for (int j = 0; j < n; ++j) {
    if (th[j]->r > 32) return false;
    max_r16 = std::max(max_r16, static_cast<int>(round_up(th[j]->r, 16)));
    rows_total += th[j]->out;
  }
  const int nkb = K / kBK;
  const size_t half = std::min<size_t>(dev->smem_optin, 227 * 1024) / 2 - 1024;
  Dec2Params dp = {};
  size_t smem = 0;
  int clusters = 0;
  bool fits = false;
  // Slices of about nine 64-wide k blocks (measured on the Gemma-3-1B decode step: one slice per
  // CTA, i.e. no cluster, was twice as slow for the q/k/v and o projections), more when the plan
  // does not fit half of an SM. After the loop the CTAs push their partial sums into each
  // other's receive areas (distributed shared-memory stores), so the exchange costs one cluster
  // barrier and no remote read.
  for (int want = std::max(1, std::min(kDec2MaxC, (nkb + 4) / 9)); want <= kDec2MaxC && !fits; ++want) {
    dp = Dec2Params{};
    dp.M = static_cast<int32_t>(M);
    dp.K = K;
    dp.nkb = nkb;
    dp.kb_per = static_cast<int32_t>(ceil_div(nkb, want));
    const int C = static_cast<int>(ceil_div(nkb, dp.kb_per));   // no empty slice
    if (C != want) continue;
    dp.C = C;
    // clusters: one CTA per SM, at least 8 rows per cluster, every family at least one
    const int64_t n_cl = std::max<int64_t>(n, std::min<int64_t>(dev->sms / C, ceil_div(rows_total, 8)));
    int64_t cnt[kMaxSeg] = {};
    int64_t used = 0;
    for (int j = 0; j < n; ++j) {
      cnt[j] = std::max<int64_t>(1, n_cl * th[j]->out / rows_total);
      used += cnt[j];
    }
    while (used < n_cl) {
      int best = 0;
      for (int j = 1; j < n; ++j)
        if (static_cast<int64_t>(th[j]->out) * cnt[best] > static_cast<int64_t>(th[best]->out) * cnt[j]) best = j;
      ++cnt[best];
      ++used;
    }
    int rc_max = 0, kg_max = 1;
    bool rc_ok = true;
    clusters = 0;
    for (int j = 0; j < n; ++j) {
      Dec2Seg& sg = dp.seg[dp.nseg++];
      sg.rc = static_cast<int32_t>(ceil_div(th[j]->out, cnt[j]));
      if (sg.rc > 256) rc_ok = false;
      cnt[j] = ceil_div(th[j]->out, sg.rc);
      sg.cl_begin = clusters;
      clusters += static_cast<int>(cnt[j]);
      sg.s = static_cast<const uint16_t*>(th[j]->s);
      sg.U = static_cast<const uint16_t*>(th[j]->U);
      sg.ldu = th[j]->ld_u;
      sg.y = static_cast<uint16_t*>(ys[j]);
      sg.ldy = ldys[j];
      sg.rows = th[j]->out;
      sg.r = th[j]->r;
      sg.r16 = static_cast<int32_t>(round_up(th[j]->r, 16));
      rc_max = std::max(rc_max, static_cast<int>(sg.rc));
      const int nslab = static_cast<int>(ceil_div(sg.rc, 16));
      kg_max = std::max(kg_max, nslab >= 8 ? 1 : 8 / nslab);
    }
    if (!rc_ok) continue;
    // shared memory: header, x slice, V slice, U rows and s of the finished rows, t, W0 ring
    // (x box odd where the tensor has the block: its eight token rows of an ldmatrix then land
    // in distinct banks)
    dp.xkb = (dp.kb_per | 1) <= nkb ? (dp.kb_per | 1) : dp.kb_per;
    dp.vrow = max_r16;
    const int64_t kslice = static_cast<int64_t>(dp.kb_per) * kBK;
    const int64_t nvb = ceil_div(kslice, 256);
    const int64_t rf_max = ceil_div(rc_max, C);
    dp.u_bytes = max_r16 > 0 ? static_cast<uint32_t>(round_up(rf_max * max_r16 * 2, 1024)) : 0u;
    dp.s_bytes = static_cast<uint32_t>(round_up((rf_max + 15) / 8 * 16, 1024));
    dp.tf_bytes = max_r16 > 0 ? static_cast<uint32_t>(round_up(static_cast<int64_t>(max_r16) * M * 4, 1024)) : 0u;
    dp.rx_bytes = static_cast<uint32_t>(round_up(static_cast<int64_t>(C) * (round_up(rf_max, 4) + max_r16) * M * 4, 1024));
    // The W0 ring of one layout: x and V resident (staged = 0), or riding in every stage behind
    // its W0 box (staged = 1: x after the dependency wait, no resident slices). k blocks per
    // stage: the largest odd count (conflict-free ldmatrix rows, at most nine) that leaves two
    // stages (measured: many one-block stages are slower than fewer larger ones, even with
    // more of W0 in flight).
    struct Ring {
      bool ok = false;
      int kbox = 0, stages = 0;
      size_t sb = 0, wb = 0, xb = 0, fixed = 0;
    };
    auto ring_for = [&](bool staged) {
      Ring g;
      const size_t xres = staged ? 0 : static_cast<size_t>(round_up(static_cast<int64_t>(dp.xkb) * M * 128, 1024));
      const size_t x2res = act >= 0 ? xres : 0;
      const size_t vres = (max_r16 > 0 && !staged)
                              ? static_cast<size_t>(round_up(nvb * round_up(ceil_div(kslice, nvb), 16) * dp.vrow * 2, 1024))
                              : 0;
      g.fixed = kHeaderBytes + kSmemSlack + xres + x2res + vres + dp.u_bytes + dp.s_bytes + dp.tf_bytes + dp.rx_bytes;
      if (g.fixed >= half) return g;
      const size_t ring = half - g.fixed;
      int kb_start = std::min(9, static_cast<int>(dp.kb_per));
      if (kb_start % 2 == 0) --kb_start;   // odd, and never past the slice
      for (int kb = kb_start; kb >= 1; kb -= 2) {
        const size_t wb = static_cast<size_t>(round_up(static_cast<int64_t>(kb) * rc_max * 128, 1024));
        const size_t xb = staged ? static_cast<size_t>(round_up(static_cast<int64_t>(kb) * M * 128, 1024)) : 0;
        const size_t vb = (staged && max_r16 > 0) ? static_cast<size_t>(round_up(static_cast<int64_t>(kb) * kBK * dp.vrow * 2, 1024)) : 0;
        const size_t sb = wb + xb + vb;
        if (ring / sb >= 2 || kb == 1) {
          g.kbox = kb;
          g.stages = static_cast<int>(std::min<size_t>(kMaxStages, ring / sb));
          g.sb = sb;
          g.wb = wb;
          g.xb = xb;
          g.ok = g.stages >= 2;
          break;
        }
      }
      return g;
    };
    // Resident x and V unless the ring then holds less of the slice than riding them in the
    // stages would (a gated input keeps both x slices resident: the activation is formed over
    // them once, before the loop). Measured: riding costs the small calls whose slice fits the
    // ring either way (q/k/v, o) about 0.4 us, and gains where the slice does not fit.
    const Ring rr = ring_for(false);
    const Ring rs = (act < 0 && kDec2Staged) ? ring_for(true) : Ring{};
    const auto held = [&](const Ring& g) { return g.ok ? std::min(g.kbox * g.stages, static_cast<int>(dp.kb_per)) : 0; };
    const bool use_staged = rs.ok && (!rr.ok || (held(rr) < dp.kb_per && held(rs) > held(rr)));
    const Ring& g = use_staged ? rs : rr;
    if (!g.ok) continue;
    dp.staged = use_staged ? 1 : 0;
    dp.x_bytes = dp.staged ? 0u : static_cast<uint32_t>(round_up(static_cast<int64_t>(dp.xkb) * M * 128, 1024));
    dp.x2_bytes = act >= 0 ? dp.x_bytes : 0u;   // a gated input stages both slices
    dp.vbox = dp.staged ? kBK : static_cast<int32_t>(round_up(ceil_div(kslice, nvb), 16));
    dp.v_bytes = (max_r16 > 0 && !dp.staged) ? static_cast<uint32_t>(round_up(nvb * dp.vbox * dp.vrow * 2, 1024)) : 0u;
    const size_t fixed = g.fixed;
    dp.kbox = g.kbox;
    dp.stages = g.stages;
    dp.stage_bytes = static_cast<uint32_t>(g.sb);
    dp.sx_off = static_cast<uint32_t>(g.wb);
    dp.sv_off = static_cast<uint32_t>(g.wb + g.xb);
    if (dp.kbox < 1 || dp.kbox > dp.kb_per || dp.stages < 2) continue;
    // the partial sums of W0 x and t reuse the ring once the loop is done
    const size_t exch = (static_cast<size_t>(kg_max) * rc_max * M + static_cast<size_t>(8) * max_r16 * M) * 4;
    const size_t ring_used = static_cast<size_t>(dp.stages) * dp.stage_bytes;
    if (exch > ring_used) continue;
    smem = fixed + ring_used;
    fits = true;
  }
  if (!fits) return false;
  const int C = dp.C;
  // tensor maps
  if ((*st = tmap_3d(&dp.tm_x, x, K, M, ldx, dp.staged ? dp.kbox : dp.xkb, static_cast<int>(M), "x")) != AQ_OK)
    return true;
  dp.act = act;
  if (act >= 0) {
    if ((*st = tmap_3d(&dp.tm_x2, x2, K, M, ldx, dp.xkb, static_cast<int>(M), "x (gated)")) != AQ_OK) return true;
    dp.x2 = static_cast<const uint16_t*>(x2);
  }
  for (int j = 0; j < n; ++j) {
    Dec2Seg& sg = dp.seg[j];
    if ((*st = tmap_3d(&sg.tm_w, th[j]->W0, K, th[j]->out, th[j]->ld_w0, dp.kbox, sg.rc, "W0")) != AQ_OK) return true;
    if (th[j]->r > 0 &&
        (*st = tmap_2d_plain(&sg.tm_v, th[j]->V, th[j]->r, K, th[j]->ld_v, dp.vrow, dp.vbox, "V")) != AQ_OK)
      return true;
  }
  dp.x = static_cast<const uint16_t*>(x);
  dp.ldx = ldx;
  dp.status = dev->status;
  dp.timeout_ns = kTimeoutNs;
  *st = launch_or_fail(launch_decode2(dp, clusters * C, smem, cs, true), "launch cluster decode kernel");
  if (*st == AQ_OK) t_last_path = AQ_PATH_DECODE;
  return true;
}

// x2 / act: a gated input, act(x) * x2 elementwise (the down projection of the fused MLP), which
// only the cluster decode kernel takes (the caller falls back to a separate activation pass).
aq_status linear_impl(const aq_theta* const* th, int n, const void* x, int64_t M, int64_t ldx,
                      void* const* ys, const int64_t* ldys, void* ws, size_t ws_bytes, void* stream,
                      const void* x2 = nullptr, int act = -1) {
  const char* who = n == 1 ? "aq_linear" : "aq_linear_qkv";
  t_launches = 0;
  for (int j = 0; j < n; ++j) {
    aq_status st = check_theta(th[j], who);
    if (st != AQ_OK) return st;
    if (th[j]->in != th[0]->in)
      return fail(AQ_ERR_SHAPE, "%s: family %d has in=%d but family 0 has in=%d", who, j, th[j]->in, th[0]->in);
  }
  const int K = th[0]->in;
  if (M < 0) return fail(AQ_ERR_SHAPE, "%s: M=%lld is negative", who, (long long)M);
  if (M > (int64_t(1) << 31) - 1) return fail(AQ_ERR_SHAPE, "%s: M=%lld is too large", who, (long long)M);
  if (M == 0) return AQ_OK;
  if (!x) return fail(AQ_ERR_INVALID_ARG, "%s: x is NULL", who);
  if (ldx < K || ldx % 8 != 0 || !aligned16(x))
    return fail(ldx < K ? AQ_ERR_SHAPE : AQ_ERR_ALIGNMENT, "%s: x must be 16-byte aligned with ldx (%lld) >= in and a multiple of 8",
                who, (long long)ldx);
  for (int j = 0; j < n; ++j) {
    if (!ys[j]) return fail(AQ_ERR_INVALID_ARG, "%s: output %d is NULL", who, j);
    if (ldys[j] < th[j]->out) return fail(AQ_ERR_SHAPE, "%s: ldy of output %d (%lld) < out=%d", who, j, (long long)ldys[j], th[j]->out);
    if (ldys[j] % 8 != 0 || !aligned16(ys[j]))
      return fail(AQ_ERR_ALIGNMENT, "%s: output %d must be 16-byte aligned with ldy a multiple of 8", who, j);
  }
  const WsLayout wl = ws_layout(th, n, M);
  if (wl.total > 0) {
    if (!ws) return fail(AQ_ERR_WORKSPACE, "%s: workspace of %zu bytes required, got NULL", who, wl.total);
    if (ws_bytes < wl.total) return fail(AQ_ERR_WORKSPACE, "%s: workspace of %zu bytes required, got %zu", who, wl.total, ws_bytes);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(AQ_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", who);
  }
  // overlap checks
  {
    Span ins[1 + 4 * kMaxSeg];
    int ni = 0;
    ins[ni++] = span(x, M, K, ldx, "x");
    for (int j = 0; j < n; ++j) {
      theta_spans(th[j], ins + ni);
      ni += 4;
    }
    // the bytes this call may touch: what it needs, and the split partials the workspace holds
    const size_t ws_touch = ws ? std::max(wl.total, std::min(ws_bytes, wl.total_split)) : 0;
    Span wsp = span(ws_touch ? ws : nullptr, 1, static_cast<int64_t>(ws_touch / 2), static_cast<int64_t>(ws_touch / 2), "workspace");
    for (int j = 0; j < n; ++j) {
      Span yj = span(ys[j], M, th[j]->out, ldys[j], "y");
      for (int i = 0; i < ni; ++i)
        if (overlaps(yj, ins[i])) return fail(AQ_ERR_OVERLAP, "%s: output %d overlaps input %s", who, j, ins[i].name);
      if (overlaps(yj, wsp)) return fail(AQ_ERR_OVERLAP, "%s: output %d overlaps the workspace", who, j);
      for (int k = 0; k < j; ++k)
        if (overlaps(yj, span(ys[k], M, th[k]->out, ldys[k], "y")))
          return fail(AQ_ERR_OVERLAP, "%s: outputs %d and %d overlap", who, k, j);
    }
    for (int i = 0; i < ni; ++i)
      if (overlaps(wsp, ins[i])) return fail(AQ_ERR_OVERLAP, "%s: the workspace overlaps input %s", who, ins[i].name);
    if (act >= 0) {
      if (!x2 || !aligned16(x2)) return fail(AQ_ERR_ALIGNMENT, "%s: the gated input must be 16-byte aligned", who);
      const Span x2s = span(x2, M, K, ldx, "x2");
      for (int j = 0; j < n; ++j)
        if (overlaps(span(ys[j], M, th[j]->out, ldys[j], "y"), x2s))
          return fail(AQ_ERR_OVERLAP, "%s: output %d overlaps the gated input", who, j);
    }
  }

  const int path_cfg = t_test_unreachable_t_ns ? static_cast<int>(AQ_PATH_PREFILL) : g_path.load();
  // From 16 tokens on, a call with a large W0 runs faster on the tcgen05 GEMM than on the
  // mma.sync decode kernel, whose issue rate then bounds it (measured on the 31B-class
  // 21504 x 5376 projection: 50.9 vs 62.3 us at M = 16, 50.7 vs 84.8 us at M = 32); at
  // 5376 x 5376 and on the Gemma-3-1B shapes the decode kernel is as fast or faster.
  int64_t w0_bytes = 0;
  for (int j = 0; j < n; ++j) w0_bytes += static_cast<int64_t>(th[j]->out) * K * 2;
  const bool gemm_pays = M >= kGemmMinMBigW0 && w0_bytes >= kGemmBigW0Bytes;
  const bool decode = path_cfg == AQ_PATH_DECODE || (path_cfg == AQ_PATH_AUTO && M <= kDecodeMaxM && !gemm_pays);
  // the tcgen05 GEMM with output rows as accumulator lanes and the tokens as N
  int64_t row_tiles128 = 0;
  for (int j = 0; j < n; ++j) row_tiles128 += ceil_div(th[j]->out, kMmaM);
  const bool swap_pays = M >= kSwapMinM && M <= kSwapMaxM && row_tiles128 <= kSwapMaxRowTiles && K >= kSwapMinK;
  const bool midm = !decode && (path_cfg == AQ_PATH_MIDM || (path_cfg == AQ_PATH_AUTO && swap_pays));
  if (decode && M > kDecodeMaxM)
    return fail(AQ_ERR_UNSUPPORTED, "%s: the decode kernel handles at most %d tokens (M=%lld)", who, kDecodeMaxM,
                (long long)M);
  if (decode && static_cast<int64_t>(M) * wl.r_total > kMaxTAcc)
    return fail(AQ_ERR_UNSUPPORTED, "%s: M x total rank = %lld exceeds the decode limit %d", who,
                (long long)(M * wl.r_total), kMaxTAcc);
  DevInfo* dev = nullptr;
  aq_status st = device_info(&dev);
  if (st != AQ_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);

  if (decode) {
    if (plan_decode2(th, n, x, M, ldx, ys, ldys, dev, cs, &st, x2, act)) return st;
    if (act >= 0) return fail(AQ_ERR_UNSUPPORTED, "%s: a gated input needs the cluster decode kernel", who);
    // ---- one launch: W0 streamed by row-owning CTAs, t = V^T x by a few extra CTAs ----
    DecodeParams dp = {};
    dp.x = static_cast<const uint16_t*>(x);
    dp.ldx = ldx;
    dp.M = static_cast<int32_t>(M);
    dp.K = K;
    dp.nkb = static_cast<int32_t>(ceil_div(K, kBK));
    // tokens per mma tile: every 8 tokens cost one more mma per 16 x 16 slice of W0
    dp.tok_tile = M <= 8 ? 8 : M <= 16 ? 16 : 32;
    dp.r_total = wl.r_total;
    dp.w3d = (K % kBK) == 0 ? 1 : 0;
    int max_r8 = 0;
    for (int j = 0; j < n; ++j) max_r8 = std::max(max_r8, static_cast<int>(round_up(th[j]->r, 8)));
    const int64_t kp = static_cast<int64_t>(dp.nkb) * kBK;
    dp.xs_ld = static_cast<int32_t>(kp + 8);
    dp.x_res = M * (kp + 8) * 2 <= 64 * 1024 ? 1 : 0;
    {
      int64_t call_w0_bytes = 0;
      for (int j = 0; j < n; ++j) call_w0_bytes += static_cast<int64_t>(th[j]->out) * K * 2;
      dp.l2_prefetch = call_w0_bytes <= 48ll * 1024 * 1024 ? 1 : 0;   // L2 is 126 MB
    }
    dp.xres_bytes = dp.x_res ? static_cast<uint32_t>(round_up(M * (kp + 8) * 2, 1024)) : 0u;
    // t = V^T x: computed by every streaming CTA for its own family when that family's V
    // is small (no cross-CTA dependency at all), else by t CTAs publishing through the
    // workspace's sync region.
    dp.vbox = static_cast<int32_t>(std::min<int64_t>(256, round_up(K, 16)));
    const int64_t vres = round_up(ceil_div(K, dp.vbox) * dp.vbox * max_r8 * 2, 1024);
    dp.t_local = (wl.r_total > 0 && dp.x_res && max_r8 <= kDecLocalMaxR8 && vres <= 40 * 1024) ? 1 : 0;
    dp.vres_bytes = dp.t_local ? static_cast<uint32_t>(vres) : 0u;
    int64_t v_bytes = 0;
    for (int j = 0; j < n; ++j) v_bytes += static_cast<int64_t>(th[j]->r) * K * 2;
    // t CTAs: about 32 KB of V each, at most kDecMaxTCtas, at least 8 rows of `in` each
    dp.t_ctas = (wl.r_total > 0 && !dp.t_local)
                    ? static_cast<int32_t>(std::max<int64_t>(
                          1, std::min<int64_t>({kDecMaxTCtas, ceil_div(v_bytes, 32 * 1024), ceil_div(K, 8)})))
                    : 0;
    // x streamed with every stage, or read by the t CTAs: the next call's weight prefetch
    // would delay those reads, so it is released after them (measured: down projections and
    // the 31B-class call at M = 32 gain 0.4-14 us; calls running from resident x and local t
    // lose up to 1.6 us and keep the early release)
    dp.late_release = (!dp.x_res || dp.t_ctas > 0) ? 1 : 0;
    int64_t rows_total = 0;
    for (int j = 0; j < n; ++j) rows_total += th[j]->out;
    // streaming CTAs: one per remaining SM, at least 8 rows each, shared among the families
    // in proportion to their rows (every family gets at least one)
    // A call whose W0 is many MB deep runs two of its own CTAs per SM: the mma.sync loop is
    // latency-bound at one CTA (8 consumer warps) per SM, and two halve-size rings keep
    // the same bytes in flight.
    const bool dual = ceil_div(rows_total, 8) >= 2 * dev->sms && rows_total * K * 2 > 64ll * 1024 * 1024 &&
                      M * (round_up(K, kBK) + 8) * 2 <= 64 * 1024;   // x resident: stages hold only W0
    const int G = static_cast<int>(std::max<int64_t>(
        n, std::min<int64_t>((dual ? 2 : 1) * dev->sms - dp.t_ctas, ceil_div(rows_total, 8))));
    int cnt[kMaxSeg] = {};
    int used = 0;
    for (int j = 0; j < n; ++j) {
      cnt[j] = std::max(1, static_cast<int>(static_cast<int64_t>(G) * th[j]->out / rows_total));
      used += cnt[j];
    }
    while (used < G) {  // hand the remainder to the family with the most rows per CTA
      int best = 0;
      for (int j = 1; j < n; ++j)
        if (static_cast<int64_t>(th[j]->out) * cnt[best] > static_cast<int64_t>(th[best]->out) * cnt[j]) best = j;
      ++cnt[best];
      ++used;
    }
    int max_rows = 8, max_r = 0;
    int cta_begin = 0;
    int64_t max_share = 0;
    for (int j = 0; j < n; ++j) {
      DecodeSeg& sg = dp.seg[dp.nseg++];
      const int64_t per = ceil_div(th[j]->out, cnt[j]);
      // A CTA whose share of W0 is many rings deep streams it in chunks of at most 32
      // rows, so that a stage can span 8 k blocks: 1 KB contiguous per row, which is what
      // keeps HBM near its copy rate. Smaller shares keep one chunk (one epilogue).
      // and U rows of a chunk staged in shared memory stay within 16 KB
      const int64_t r16 = round_up(th[j]->r, 16);
      const int64_t u_cap = r16 > 0 ? std::max<int64_t>(16, (16 * 1024) / (r16 * 2) / 16 * 16) : kMmaM;
      const int64_t row_cap = std::min<int64_t>(per * K * 2 > 256 * 1024 ? 32 : kMmaM, u_cap);
      sg.chunks = static_cast<int32_t>(ceil_div(per, row_cap));
      sg.chunk_rows = static_cast<int32_t>(ceil_div(th[j]->out, static_cast<int64_t>(cnt[j]) * sg.chunks));
      cnt[j] = static_cast<int>(ceil_div(th[j]->out, static_cast<int64_t>(sg.chunk_rows) * sg.chunks));  // CTAs with rows
      sg.s = static_cast<const uint16_t*>(th[j]->s);
      sg.U = static_cast<const uint16_t*>(th[j]->U);
      sg.ldu = th[j]->ld_u;
      sg.V = static_cast<const uint16_t*>(th[j]->V);
      sg.ldv = th[j]->ld_v;
      sg.y = static_cast<uint16_t*>(ys[j]);
      sg.ldy = ldys[j];
      sg.rows = th[j]->out;
      sg.r = th[j]->r;
      sg.r8 = static_cast<int32_t>(round_up(th[j]->r, 8));
      sg.r16 = static_cast<int32_t>(r16);
      sg.t_col = wl.dec_t_col[j];
      sg.cta_begin = cta_begin;
      cta_begin += cnt[j];
      max_rows = std::max(max_rows, static_cast<int>(sg.chunk_rows));
      max_r = std::max(max_r, th[j]->r);
      dp.r8_total += sg.r8;
      max_share = std::max<int64_t>(max_share, static_cast<int64_t>(sg.chunk_rows) * sg.chunks * K * 2);
    }
    // 2-D boxes must start on 1 KB (128-byte swizzle atoms of 8 rows): round rows to 8
    dp.wbox_bytes = static_cast<uint32_t>(round_up(max_rows, 8) * 128);
    // epilogue staging: the warps' row sums (or, first, their partial t) then t itself
    dp.ts_off = std::max<int32_t>(8 * 16 * dp.tok_tile, dp.t_local ? 8 * round_up(dp.tok_tile, 16) * max_r8 : 0);
    const int64_t max_r16 = round_up(max_r, 16);
    // t_hi / t_lo and staged U rows are r16 wide plus 8 elements of padding (bank spread)
    const int64_t rs16 = max_r > 0 ? max_r16 + 8 : 0;
    dp.epi_bytes = static_cast<uint32_t>(round_up(static_cast<int64_t>(dp.ts_off) * 4 + 2 * dp.tok_tile * rs16 * 2, 1024));
    // U rows of a chunk staged in shared memory (two buffers when CTAs have several chunks)
    int max_chunks = 1;
    for (int j = 0; j < n; ++j) max_chunks = std::max(max_chunks, static_cast<int>(dp.seg[j].chunks));
    dp.ubuf_bytes = static_cast<uint32_t>(round_up(static_cast<int64_t>(max_rows) * rs16 * 2, 128));
    dp.ures_bytes = max_r > 0 ? static_cast<uint32_t>(round_up((max_chunks > 1 ? 2 : 1) * dp.ubuf_bytes, 1024)) : 0u;
    // Two CTAs per SM when a CTA's W0 share is small (the next call's CTAs then stream W0
    // while this call's finish), with smaller stages if that is what it takes to fit three;
    // one CTA with a deep ring when the share is large.
    const size_t fixed = kHeaderBytes + kSmemSlack + dp.epi_bytes + dp.xres_bytes + dp.vres_bytes + dp.ures_bytes;
    const size_t cap = std::min<size_t>(dev->smem_optin, 227 * 1024);
    const size_t half = cap / 2 - 1024;
    // With 3-D boxes a stage row is (row, k block) = row * kbox + b and the 128-byte
    // swizzle keys on that index mod 8; ldmatrix reads 8 rows at one k block, which land
    // on 8 different bank groups only when kbox is odd. 2-D boxes split K evenly.
    auto pick_kbox = [&](int64_t kb) -> int64_t {
      if (!dp.w3d) return ceil_div(dp.nkb, ceil_div(dp.nkb, kb));
      int64_t best = 1, best_waste = INT64_MAX;
      for (int64_t k = (kb % 2) ? kb : kb - 1; k >= std::max<int64_t>(1, kb - 4); k -= 2) {
        const int64_t waste = ceil_div(dp.nkb, k) * k - dp.nkb;
        if (waste < best_waste) best = k, best_waste = waste;
      }
      return best;
    };
    auto set_kbox = [&](int64_t kb) {
      dp.kbox = static_cast<int32_t>(pick_kbox(kb));
      // a 3-D box is kbox x rows lines of 128 bytes, packed; 2-D boxes start on 1 KB each
      dp.wregion = static_cast<uint32_t>(round_up(static_cast<int64_t>(dp.kbox) *
                                                      (dp.w3d ? static_cast<int64_t>(max_rows) * 128 : dp.wbox_bytes),
                                                  1024));
      dp.stage_bytes = static_cast<uint32_t>(
          round_up(dp.wregion + (dp.x_res ? 0 : static_cast<int64_t>(dp.kbox) * dp.tok_tile * 128), 1024));
      return fixed < half ? static_cast<int>((half - fixed) / dp.stage_bytes) : 0;
    };
    const int64_t kb0 = std::max<int64_t>(1, std::min<int64_t>({9, (36 * 1024) / dp.wbox_bytes, dp.nkb}));
    int stages2 = 0;
    bool two = false;
    // (boxes of fewer than 3 k blocks stall TMA on request rate: below that, one CTA per SM)
    const int64_t kb_min = std::min<int64_t>(3, kb0);
    if (max_share <= 128 * 1024 || dual)
      for (int64_t kb = kb0; kb >= kb_min && !two; --kb) {
        stages2 = set_kbox(kb);
        two = stages2 >= 3 || (stages2 >= 2 && kb == kb_min);
      }
    if (two) {
      dp.stages = std::min(stages2, kMaxStages);
    } else {
      set_kbox(kb0);
      dp.stages = stages_for(dp.stage_bytes, dev->smem_optin, fixed);
    }
    size_t smem = fixed + static_cast<size_t>(dp.stages) * dp.stage_bytes;
    if (smem > cap) return fail(AQ_ERR_UNSUPPORTED, "%s: decode plan needs %zu bytes of shared memory", who, smem);
    if (dp.t_ctas > 0) {
      // A t CTA stages its whole slice of V (all families) and x at once, in boxes of vbox
      // rows, after its fp32 t [M][r_total]; add t CTAs until a slice fits, and when even
      // the thinnest slice does not, give the launch the shared memory it needs.
      const int64_t tacc_bytes = round_up(M * wl.r_total * 4, 1024);
      const int64_t tspace = static_cast<int64_t>(smem) - kHeaderBytes - kSmemSlack - tacc_bytes;
      const int64_t max_t = std::max<int64_t>(1, ceil_div(K, 16));
      for (;;) {
        const int64_t ks = round_up(ceil_div(K, dp.t_ctas), 16);   // the kernel's slice length
        const int64_t nvb = ceil_div(ks, 256);
        dp.vbox = static_cast<int32_t>(round_up(ceil_div(ks, nvb), 16));
        // per box: V rows of every family, then x [M][vbox] padded to 128 bytes
        const int64_t per_box = static_cast<int64_t>(dp.vbox) * dp.r8_total * 2 + round_up(dp.vbox * M * 2, 128);
        if (nvb * per_box <= tspace) break;
        if (dp.t_ctas >= max_t) {
          const size_t need = kHeaderBytes + kSmemSlack + static_cast<size_t>(tacc_bytes + nvb * per_box);
          if (need > cap)
            return fail(AQ_ERR_UNSUPPORTED, "%s: M x total rank too large for the decode kernel's shared memory", who);
          smem = need;
          break;
        }
        ++dp.t_ctas;
      }
      // the t CTAs' fixed-order reduction parks up to 256 x 16 fp32 partials after t
      smem = std::max<size_t>(smem, kHeaderBytes + kSmemSlack + static_cast<size_t>(tacc_bytes) + 256 * 16 * 4);
      if (smem > cap) return fail(AQ_ERR_UNSUPPORTED, "%s: decode plan needs %zu bytes of shared memory", who, smem);
      if ((st = tmap_2d_plain(&dp.tm_xt, x, K, M, ldx, dp.vbox, static_cast<int>(M), "x (t)")) != AQ_OK) return st;
    }
    for (int j = 0; j < n; ++j) {
      DecodeSeg& sg = dp.seg[j];
      if (dp.w3d) {
        if ((st = tmap_3d(&sg.tm_w, th[j]->W0, K, th[j]->out, th[j]->ld_w0, dp.kbox, sg.chunk_rows, "W0")) != AQ_OK)
          return st;
      } else if ((st = tmap_2d(&sg.tm_w, th[j]->W0, K, th[j]->out, th[j]->ld_w0, sg.chunk_rows, "W0")) != AQ_OK) {
        return st;
      }
      if (th[j]->r > 0 && (st = tmap_2d_plain(&sg.tm_v, th[j]->V, th[j]->r, K, th[j]->ld_v, sg.r8, dp.vbox, "V")) != AQ_OK)
        return st;
    }
    if (!dp.x_res) {
      if (dp.w3d) {
        if ((st = tmap_3d(&dp.tm_x, x, K, M, ldx, dp.kbox, static_cast<int>(M), "x")) != AQ_OK) return st;
      } else if ((st = tmap_2d(&dp.tm_x, x, K, M, ldx, static_cast<int>(M), "x")) != AQ_OK) {
        return st;
      }
    }
    dp.counters = reinterpret_cast<int32_t*>(wsb);
    dp.t_acc = reinterpret_cast<float*>(wsb + kSyncTAccOffset);
    dp.status = dev->status;
    dp.timeout_ns = kTimeoutNs;
    // every TMA destination in shared memory must be 128-byte aligned (1 KB for the
    // swizzled W0 / x stages): the regions above are sized so; refuse a plan that is not
    if (dp.epi_bytes % 1024 || dp.xres_bytes % 1024 || dp.vres_bytes % 1024 || dp.ures_bytes % 1024 ||
        dp.ubuf_bytes % 16 || dp.stage_bytes % 1024 ||
        dp.wregion % 1024 || dp.wbox_bytes % 1024 || (static_cast<int64_t>(dp.vbox) * 8 * 2) % 128)
      return fail(AQ_ERR_UNSUPPORTED, "%s: decode plan breaks shared-memory alignment", who);
    const int grid = dp.t_ctas + cta_begin;
    if ((st = launch_or_fail(launch_decode(dp, grid, smem, cs, true), "launch decode kernel")) != AQ_OK) return st;
    t_last_path = AQ_PATH_DECODE;
    return AQ_OK;
  }

  if (act >= 0) return fail(AQ_ERR_UNSUPPORTED, "%s: a gated input needs the cluster decode kernel", who);
  uint16_t* tbuf = reinterpret_cast<uint16_t*>(wsb + kSyncBytes);
  // ---- plan of the prefill GEMM with the fused reconstruction epilogue ----
  GemmParams gp = {};
  gp.M = static_cast<int32_t>(M);
  gp.K = K;
  if (midm) {
    // 128 output rows per tile as the accumulator lanes; all tokens (in tiles of at most 256,
    // balanced, multiples of 16) as the MMA N
    gp.swap = 1;
    gp.row_tile = kMmaM;
    gp.n_tok_tiles = static_cast<int32_t>(ceil_div(M, 256));
    gp.tok_tile = static_cast<int32_t>(round_up(ceil_div(M, gp.n_tok_tiles), 16));
    gp.n_mma = gp.tok_tile;
  } else {
    gp.tok_tile = kMmaM;
    gp.n_tok_tiles = static_cast<int32_t>(ceil_div(M, kMmaM));
    gp.row_tile = prefill_row_tile(th, n, gp.n_tok_tiles, dev->sms);
    gp.n_mma = gp.row_tile;
  }
  // Split K: when the output tiles fill at most half of the SMs and K is deep, the K of every
  // tile is cut into slices that separate CTAs sum into fp32 partials (no scale, no rank-r
  // part), and a small kernel finishes y = RN(s * sum z + U * sum t). The slices stop where
  // the caller's workspace does.
  const int64_t nkb = ceil_div(K, kBK);
  int64_t main_tiles = 0;
  for (int j = 0; j < n; ++j) main_tiles += gp.n_tok_tiles * ceil_div(th[j]->out, gp.row_tile);
  int split = 1;
  int call_max_r = 0;
  for (int j = 0; j < n; ++j) call_max_r = std::max(call_max_r, th[j]->r);
  if (main_tiles * 2 <= dev->sms && nkb >= 2 * kSplitMinKb && call_max_r <= kSplitMaxRank && M <= 65535 && ws &&
      (reinterpret_cast<uintptr_t>(ws) & 255u) == 0 && wl.split_slice > 0) {
    // as many slices as keep all tiles (the t tiles included) within one wave
    const size_t room = ws_bytes > wl.split_base ? ws_bytes - wl.split_base : 0;
    const int64_t tiles = main_tiles + (wl.any_r ? gp.n_tok_tiles * ceil_div(wl.ld_t, gp.row_tile) : 0);
    const int64_t sp = std::min<int64_t>({dev->sms / tiles, nkb / kSplitMinKb, kMaxSplit, wl.split_max,
                                          static_cast<int64_t>(room / wl.split_slice)});
    if (sp >= 2) split = static_cast<int>(sp);
  }
  int kb_per = static_cast<int>(nkb);
  if (split > 1) {
    kb_per = static_cast<int>(ceil_div(nkb, split));
    split = static_cast<int>(ceil_div(nkb, kb_per));   // every slice holds at least one k block
  }
  float* const pz_base = split > 1 ? reinterpret_cast<float*>(wsb + wl.split_base) : nullptr;
  float* const pt_base = split > 1 ? pz_base + static_cast<int64_t>(split) * M * wl.ld_pz : nullptr;
  // CTA pairs (2-SM MMAs, M = 256) on adjacent token tiles: each CTA holds half of the N
  // rows of B, so a stage is 32 KB instead of 48 and shared memory moves a third less per
  // MMA, which bounds this GEMM. Pairs need two token tiles and one CTA per SM; each half of
  // B is a whole number of 8-row swizzle atoms.
  size_t smem = 0;
  // (the swapped layout writes y straight from registers: no output staging)
  const size_t ystage = midm ? 0 : kYStageTotal;
  for (int cl = (!midm && split == 1 && gp.n_tok_tiles >= 2 && dev->gemm_pairs > 0 && gp.row_tile % 16 == 0) ? 2 : 1;
       cl >= 1; --cl) {
    gp.cluster = cl;
    // a stage: the 128-lane operand (A) and the N-row operand (B, or this CTA's half of it)
    gp.stage_bytes = static_cast<uint32_t>(round_up(kStageA + (gp.n_mma / cl) * 128, 1024));
    gp.stages = stages_for(gp.stage_bytes, dev->smem_optin, kHeaderBytes + kGemmSBufBytes + kSmemSlack + ystage);
    smem = kSmemSlack + kHeaderBytes + kGemmSBufBytes + ystage + static_cast<size_t>(gp.stages) * gp.stage_bytes;
    if (cl == 1 || smem >= kGemmPairMinSmem) break;
  }
  gp.n_tok_units = static_cast<int32_t>(ceil_div(gp.n_tok_tiles, gp.cluster));
  // Walk order: the larger operand streams once, the smaller is re-read from L2. More tokens
  // than output rows (the Gemma-sized families at thousands of tokens) walk a token unit's row
  // tiles first; otherwise (the 31B-class rows) a row tile's token units first.
  {
    int64_t rows_total = 0;
    for (int j = 0; j < n; ++j) rows_total += th[j]->out;
    gp.tok_major = (!midm && M > rows_total) ? 1 : 0;
  }
  const int box_rows = gp.row_tile / gp.cluster;
  // t = x V as the first tiles of the same launch, when the sync region holds a flag per
  // token tile; otherwise as a GEMM launch of its own before it
  const int64_t n_flags = static_cast<int64_t>(gp.n_tok_units) * gp.cluster;
  const bool fused_t = wl.any_r && (split > 1 || 1 + n_flags <= static_cast<int64_t>(kSyncBytes / 4));
  if (midm && wl.any_r && !fused_t)
    return fail(AQ_ERR_UNSUPPORTED, "%s: M=%lld has too many token tiles for the mid-M path", who, (long long)M);

  if (wl.any_r) {
    // V^T into the workspace: the t tiles read it K-major
    TransposeParams tp = {};
    tp.K = K;
    int max_r = 0;
    for (int j = 0; j < n; ++j) {
      if (th[j]->r == 0) continue;
      TransposeSeg& s = tp.seg[tp.nseg++];
      s.V = static_cast<const uint16_t*>(th[j]->V);
      s.ldv = th[j]->ld_v;
      s.Vt = reinterpret_cast<uint16_t*>(wsb + wl.vt_off[j]);
      s.ldvt = wl.ldvt;
      s.r = th[j]->r;
      max_r = std::max(max_r, th[j]->r);
    }
    if ((st = launch_or_fail(launch_transpose(tp, max_r, cs, true), "launch V transpose")) != AQ_OK) return st;
  }
  if (wl.any_r && !fused_t) {
    GemmParams tg = {};
    tg.M = static_cast<int32_t>(M);
    tg.K = K;
    tg.tok_tile = kMmaM;
    tg.n_tok_tiles = static_cast<int32_t>(ceil_div(M, kMmaM));
    int rt = 16;
    for (int j = 0; j < n; ++j) rt = std::max<int>(rt, static_cast<int>(round_up(th[j]->r, 16)));
    tg.row_tile = rt;
    tg.n_mma = rt;
    if ((st = tmap_2d(&tg.tm_x, x, K, M, ldx, kMmaM, "x")) != AQ_OK) return st;
    int tiles = 0;
    for (int j = 0; j < n; ++j) {
      if (th[j]->r == 0) continue;
      GemmSeg& s = tg.seg[tg.nseg++];
      if ((st = tmap_2d(&s.tm_w, wsb + wl.vt_off[j], K, th[j]->r, wl.ldvt, rt, "V^T")) != AQ_OK) return st;
      s.s = nullptr;
      s.y = tbuf + wl.t_col[j];
      s.ldy = wl.ld_t;
      s.rows = th[j]->r;
      s.r = 0;
      s.n_row_tiles = 1;
      s.tile_begin = tiles;
      s.n_mma = rt;
      tiles += tg.n_tok_tiles;
    }
    tg.cluster = 1;
    tg.n_tok_units = tg.n_tok_tiles;
    tg.head_kb = kGemmHeadKb;
    tg.total_tiles = tiles;
    tg.prefetch_w = 0;  // V^T comes from the transpose kernel just before
    tg.stage_bytes = static_cast<uint32_t>(round_up(kStageA + tg.n_mma * 128, 1024));
    tg.stages = stages_for(tg.stage_bytes, dev->smem_optin, kHeaderBytes + kGemmSBufBytes + kSmemSlack);
    tg.tmem_cols = tmem_cols_for(2 * tg.n_mma);
    tg.status = dev->status;
    tg.timeout_ns = kTimeoutNs;
    const size_t tsmem = kSmemSlack + kHeaderBytes + kGemmSBufBytes + static_cast<size_t>(tg.stages) * tg.stage_bytes;
    const int tgrid = std::min(tiles, dev->sms);
    if ((st = launch_or_fail(launch_gemm(tg, tgrid, tsmem, cs, true), "launch t GEMM")) != AQ_OK) return st;
  }

  if ((st = tmap_2d(&gp.tm_x, x, K, M, ldx, gp.tok_tile, "x")) != AQ_OK) return st;
  int tiles = 0;
  if (fused_t) {
    // one t segment first: t [M, ld_t] = x [V_0 | V_1 | ...] over the stacked V^T (rows of
    // padding between families feed only padding columns of t, which nothing reads), no
    // scale, no rank-r part
    GemmSeg& s = gp.seg[gp.nseg++];
    if ((st = tmap_2d(&s.tm_w, wsb + wl.vt_off[0], K, wl.ld_t, wl.ldvt, box_rows, "V^T")) != AQ_OK) return st;
    s.s = nullptr;
    s.y = tbuf;
    s.ldy = wl.ld_t;
    s.rows = static_cast<int32_t>(wl.ld_t);
    s.r = 0;
    s.t_seg = 1;
    s.n_row_tiles = static_cast<int32_t>(ceil_div(wl.ld_t, gp.row_tile));
    s.n_mma = midm ? gp.n_mma : static_cast<int32_t>(std::min<int64_t>(round_up(wl.ld_t, 16), gp.row_tile));
    s.tile_begin = tiles;
    tiles += s.n_row_tiles * gp.n_tok_units;
    if (split > 1) {
      // partial sums of t; nothing in this launch waits for them (the families' tiles have no
      // rank-r part), so no flags. t_seg stays set: V^T comes from the previous kernel.
      s.y = nullptr;
      s.part = pt_base;
      s.ld_part = wl.ld_t;
    } else {
      gp.t_need = s.n_row_tiles;
      gp.t_flags = reinterpret_cast<int32_t*>(wsb);
      gp.n_flags = static_cast<int32_t>(n_flags);
    }
  }
  for (int j = 0; j < n; ++j) {
    GemmSeg& s = gp.seg[gp.nseg++];
    if ((st = tmap_2d(&s.tm_w, th[j]->W0, K, th[j]->out, th[j]->ld_w0, box_rows, "W0")) != AQ_OK) return st;
    if (th[j]->r > 0) {
      if ((st = tmap_2d(&s.tm_u, th[j]->U, th[j]->r, th[j]->out, th[j]->ld_u, box_rows, "U")) != AQ_OK) return st;
      if ((st = tmap_2d(&s.tm_t, tbuf + wl.t_col[j], th[j]->r, M, wl.ld_t, gp.tok_tile, "t")) != AQ_OK) return st;
    }
    s.s = static_cast<const uint16_t*>(th[j]->s);
    s.y = static_cast<uint16_t*>(ys[j]);
    s.ldy = ldys[j];
    s.rows = th[j]->out;
    s.r = th[j]->r;
    s.n_row_tiles = static_cast<int32_t>(ceil_div(th[j]->out, gp.row_tile));
    s.n_mma = gp.n_mma;
    // bulk tensor stores of y need whole 64-column boxes per tile: a partial box would write
    // into the next tile's columns (the tensor map clips only at the family's last row)
    s.tma_y = (!midm && gp.row_tile % 64 == 0) ? 1 : 0;
    if (split > 1) {   // fp32 partials of W0 x; s and U t are the finalize kernel's
      s.s = nullptr;
      s.y = nullptr;
      s.r = 0;
      s.tma_y = 0;
      s.part = pz_base + wl.pz_col[j];
      s.ld_part = wl.ld_pz;
    }
    if (s.tma_y && (st = tmap_2d(&s.tm_y, ys[j], th[j]->out, M, ldys[j], 32, "y")) != AQ_OK) return st;
    s.tile_begin = tiles;
    tiles += s.n_row_tiles * gp.n_tok_units;
  }
  gp.total_tiles = tiles * split;
  gp.ksplit = split;
  gp.kb_per = kb_per;
  gp.prefetch_w = 1;
  gp.head_kb = kGemmHeadKb;
  gp.tmem_cols = tmem_cols_for(2 * gp.n_mma);   // two accumulator buffers
  gp.status = dev->status;
  gp.timeout_ns = kTimeoutNs;
  if (t_test_unreachable_t_ns) {
    if (!gp.t_flags || gp.cluster != 1)
      return fail(AQ_ERR_UNSUPPORTED, "aq_selftest_prefill_timeout: the call must wait on t flags in unpaired CTAs");
    gp.t_need = 1 << 30;
    gp.timeout_ns = t_test_unreachable_t_ns;
  }
  const int grid = gp.cluster > 1 ? 2 * std::min(tiles, dev->gemm_pairs) : std::min(gp.total_tiles, dev->sms);
  if ((st = launch_or_fail(launch_gemm(gp, grid, smem, cs, true), "launch reconstruction GEMM")) != AQ_OK) return st;
  if (split > 1) {
    FinalizeParams fp = {};
    fp.nseg = n;
    fp.M = static_cast<int32_t>(M);
    fp.ksplit = split;
    fp.ld_pz = wl.ld_pz;
    fp.ld_pt = wl.ld_t;
    fp.pz_slice = M * wl.ld_pz;
    fp.pt_slice = M * wl.ld_t;
    int blocks = 0;
    for (int j = 0; j < n; ++j) {
      FinalizeSeg& f = fp.seg[j];
      f.pz = pz_base + wl.pz_col[j];
      f.pt = th[j]->r > 0 ? pt_base + wl.t_col[j] : nullptr;
      f.s = static_cast<const uint16_t*>(th[j]->s);
      f.U = static_cast<const uint16_t*>(th[j]->U);
      f.ldu = th[j]->ld_u;
      f.y = static_cast<uint16_t*>(ys[j]);
      f.ldy = ldys[j];
      f.rows = th[j]->out;
      f.r = th[j]->r;
      f.block_begin = blocks;
      blocks += static_cast<int>(ceil_div(th[j]->out, kFinRows));
    }
    if ((st = launch_or_fail(launch_finalize(fp, blocks, cs, true), "launch split-K finalize")) != AQ_OK) return st;
  }
  t_last_path = midm ? AQ_PATH_MIDM : AQ_PATH_PREFILL;
  return AQ_OK;
}

}  // namespace

namespace aq {
size_t linear_workspace_min_bytes(const aq_theta* th, int32_t n_theta, int64_t M);
}  // namespace aq

size_t aq::linear_workspace_min_bytes(const aq_theta* th, int32_t n_theta, int64_t M) {
  if (!th || n_theta < 1 || n_theta > AQ_MAX_FAMILIES || M < 0) return static_cast<size_t>(-1);
  const aq_theta* ptrs[kMaxSeg];
  for (int j = 0; j < n_theta; ++j) {
    if (th[j].r < 0 || th[j].r > AQ_MAX_RANK || th[j].in < 1) return static_cast<size_t>(-1);
    ptrs[j] = &th[j];
  }
  return ws_layout(ptrs, n_theta, M).total;
}

int aq::set_last_error(int status, const char* message) {
  t_err = message ? message : "";
  return status;
}

// =====================================================================================
// exported C ABI
// =====================================================================================
extern "C" {

size_t aq_linear_workspace_bytes(const aq_theta* th, int32_t n_theta, int64_t M) {
  if (!th || n_theta < 1 || n_theta > AQ_MAX_FAMILIES || M < 0) return static_cast<size_t>(-1);
  const aq_theta* ptrs[kMaxSeg];
  for (int j = 0; j < n_theta; ++j) {
    if (th[j].r < 0 || th[j].r > AQ_MAX_RANK || th[j].in < 1) return static_cast<size_t>(-1);
    ptrs[j] = &th[j];
  }
  return ws_layout(ptrs, n_theta, M).total_split;
}

aq_status aq_linear(const aq_theta* th, const void* x, int64_t M, int64_t ldx, void* y, int64_t ldy,
                    void* workspace, size_t workspace_bytes, void* stream) {
  if (!th) return fail(AQ_ERR_INVALID_ARG, "aq_linear: theta is NULL");
  const aq_theta* ptrs[1] = {th};
  void* ys[1] = {y};
  int64_t lds[1] = {ldy};
  return linear_impl(ptrs, 1, x, M, ldx, ys, lds, workspace, workspace_bytes, stream);
}

aq_status aq_linear_qkv(const aq_theta th[3], const void* x, int64_t M, int64_t ldx, void* const y[3],
                        const int64_t ldy[3], void* workspace, size_t workspace_bytes, void* stream) {
  if (!th || !y || !ldy) return fail(AQ_ERR_INVALID_ARG, "aq_linear_qkv: NULL array argument");
  const aq_theta* ptrs[3] = {&th[0], &th[1], &th[2]};
  return linear_impl(ptrs, 3, x, M, ldx, y, ldy, workspace, workspace_bytes, stream);
}

aq_status aq_linear_multi(const aq_theta* th, int32_t n, const void* x, int64_t M, int64_t ldx, void* const* y,
                          const int64_t* ldy, void* workspace, size_t workspace_bytes, void* stream) {
  if (!th || !y || !ldy) return fail(AQ_ERR_INVALID_ARG, "aq_linear_multi: NULL array argument");
  if (n < 1 || n > AQ_MAX_FAMILIES)
    return fail(AQ_ERR_INVALID_ARG, "aq_linear_multi: n=%d outside [1, %d]", n, AQ_MAX_FAMILIES);
  const aq_theta* ptrs[AQ_MAX_FAMILIES] = {};
  for (int j = 0; j < n; ++j) ptrs[j] = &th[j];
  return linear_impl(ptrs, n, x, M, ldx, y, ldy, workspace, workspace_bytes, stream);
}

// ---- fused MLP: y = down( act(gate(x)) * up(x) ) ----
namespace {
struct MlpLayout {
  size_t lin = 0;      // workspace of the linear calls (shared: they run one after another)
  size_t g_off = 0, u_off = 0;
  int64_t ldg = 0;
  size_t total = 0;
};

size_t mlp_layout(const aq_theta* gate, const aq_theta* up, const aq_theta* down, int64_t M, MlpLayout* out) {
  const aq_theta pair[2] = {*gate, *up};
  const size_t a = aq_linear_workspace_bytes(pair, 2, M);
  const size_t b = aq_linear_workspace_bytes(down, 1, M);
  if (a == static_cast<size_t>(-1) || b == static_cast<size_t>(-1)) return static_cast<size_t>(-1);
  MlpLayout l;
  l.lin = static_cast<size_t>(round_up(static_cast<int64_t>(std::max(a, b)), 256));
  l.ldg = round_up(gate->out, 8);
  const size_t gbytes = static_cast<size_t>(round_up(M * l.ldg * 2, 256));
  l.g_off = l.lin;
  l.u_off = l.g_off + gbytes;
  l.total = l.u_off + gbytes;
  if (out) *out = l;
  return l.total;
}
}  // namespace

size_t aq_mlp_workspace_bytes(const aq_theta* gate, const aq_theta* up, const aq_theta* down, int64_t M) {
  if (!gate || !up || !down || M < 0) return static_cast<size_t>(-1);
  return mlp_layout(gate, up, down, M, nullptr);
}

aq_status aq_mlp(const aq_theta* gate, const aq_theta* up, const aq_theta* down, aq_act act, const void* x,
                 int64_t M, int64_t ldx, void* y, int64_t ldy, void* workspace, size_t workspace_bytes,
                 void* stream) {
  t_launches = 0;
  if (!gate || !up || !down) return fail(AQ_ERR_INVALID_ARG, "aq_mlp: NULL bundle");
  if (act != AQ_ACT_GELU_TANH && act != AQ_ACT_SILU) return fail(AQ_ERR_INVALID_ARG, "aq_mlp: unknown activation %d", (int)act);
  if (gate->out != up->out || gate->in != up->in || down->in != gate->out)
    return fail(AQ_ERR_SHAPE, "aq_mlp: gate and up must share [out, in] and down.in must equal their out "
                "(gate %d x %d, up %d x %d, down %d x %d)", gate->out, gate->in, up->out, up->in, down->out, down->in);
  if (M < 0) return fail(AQ_ERR_SHAPE, "aq_mlp: M=%lld is negative", (long long)M);
  if (M == 0) return AQ_OK;
  MlpLayout l;
  if (mlp_layout(gate, up, down, M, &l) == static_cast<size_t>(-1)) return fail(AQ_ERR_INVALID_ARG, "aq_mlp: bad bundle");
  if (!workspace || workspace_bytes < l.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(AQ_ERR_WORKSPACE, "aq_mlp: workspace of %zu bytes (256-byte aligned) required, got %zu", l.total,
                workspace_bytes);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  uint16_t* g = reinterpret_cast<uint16_t*>(wsb + l.g_off);
  uint16_t* u = reinterpret_cast<uint16_t*>(wsb + l.u_off);
  // gate and up over one x in one launch
  const aq_theta* gu[2] = {gate, up};
  void* gys[2] = {g, u};
  const int64_t glds[2] = {l.ldg, l.ldg};
  aq_status st = linear_impl(gu, 2, x, M, ldx, gys, glds, workspace, l.lin, stream);
  if (st != AQ_OK) return st;
  int launches = t_launches;
  // down over act(g) * u: fused into the cluster decode kernel's input when it takes the call,
  // else one activation pass in place of g first
  const aq_theta* dn[1] = {down};
  void* dys[1] = {y};
  const int64_t dlds[1] = {ldy};
  const int32_t saved_path = g_path.load();
  if (M <= 16 && saved_path != AQ_PATH_PREFILL && saved_path != AQ_PATH_MIDM) {
    st = linear_impl(dn, 1, g, M, l.ldg, dys, dlds, workspace, l.lin, stream, u, static_cast<int>(act));
    if (st == AQ_OK) {
      t_launches += launches;
      return AQ_OK;
    }
    if (st != AQ_ERR_UNSUPPORTED) return st;
  }
  cudaError_t e = launch_gated_act(g, u, l.ldg, M, gate->out, static_cast<int32_t>(act), static_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return cuda_fail(e, "aq_mlp: launch activation");
  ++launches;
  st = linear_impl(dn, 1, g, M, l.ldg, dys, dlds, workspace, l.lin, stream);
  if (st == AQ_OK) t_launches += launches;
  return st;
}

constexpr int kPrePfAhead = 4;   // precompute: W0 tiles of a CTA prefetched into L2 ahead
constexpr int kPreNvfp4Keep = 3;  // NVFP4 frees its W0 buffers on read: three suffice (2-4 measured equal)

// Tiles, tensor maps and shared-memory budget of the precompute kernel (any output kind).
static aq_status plan_precompute(const aq_theta* th, DevInfo* dev, PrecomputeParams* pp, size_t* smem,
                                 int* grid, int out_kind, const char* who) {
  pp->out = th->out;
  pp->in = th->in;
  pp->r = th->r;
  pp->bn = 128;
  pp->s = static_cast<const uint16_t*>(th->s);
  pp->n_row_tiles = static_cast<int32_t>(ceil_div(th->out, kMmaM));
  pp->n_col_tiles = static_cast<int32_t>(ceil_div(th->in, pp->bn));
  pp->total_tiles = pp->n_row_tiles * pp->n_col_tiles;
  aq_status st;
  if ((st = tmap_2d(&pp->tm_w0, th->W0, th->in, th->out, th->ld_w0, kMmaM, "W0")) != AQ_OK) return st;
  if (th->r > 0) {
    if ((st = tmap_2d(&pp->tm_u, th->U, th->r, th->out, th->ld_u, kMmaM, "U")) != AQ_OK) return st;
    if ((st = tmap_2d(&pp->tm_v, th->V, th->r, th->in, th->ld_v, pp->bn, "V")) != AQ_OK) return st;
  }
  pp->stage_bytes = static_cast<uint32_t>(round_up(kStageA + pp->bn * 128, 1024));
  // Shared memory: W0 / W_eff tile buffers (four kept before the ring grows: measured best
  // for r = 128, where four buffers and a three-stage ring beat three and four), the U / V
  // ring (two tiles' chunks where they fit, so that the next tile's chunks arrive from L2
  // while this tile's MMAs run) and the NVFP4 table of 1/d.
  const size_t cbuf_bytes = static_cast<size_t>(pp->bn) * 256u;
  const size_t cap = std::min<size_t>(dev->smem_optin, 227 * 1024);
  const size_t staging = out_kind == kPreNvfp4 ? kNvfp4TableBytes : 0u;
  const size_t base = kSmemSlack + kHeaderBytes + staging;
  const int nkb = static_cast<int>(ceil_div(th->r, kBK));
  if (th->r > 0) {
    const size_t keep = (out_kind == kPreBf16 ? 4 : kPreNvfp4Keep) * cbuf_bytes;
    const size_t room = cap > base + keep ? cap - base - keep : 0;
    pp->stages = static_cast<int32_t>(std::max<size_t>(2, std::min<size_t>(2 * nkb, room / pp->stage_bytes)));
  } else {
    pp->stages = 0;
  }
  const size_t fixed = base + static_cast<size_t>(pp->stages) * pp->stage_bytes;
  pp->cbufs = static_cast<int32_t>(std::min<size_t>(8, (cap - fixed) / cbuf_bytes));
  // W0 tiles prefetched into L2 ahead of the tile buffers (beyond what shared memory holds)
  pp->pf_ahead = out_kind == kPreBf16 ? kPrePfAhead : 0;   // measured: helps bf16 only
  pp->tmem_cols = th->r > 0 ? tmem_cols_for(2 * pp->bn) : 32;
  pp->status = dev->status;
  pp->timeout_ns = kTimeoutNs;
  *smem = fixed + static_cast<size_t>(pp->cbufs) * cbuf_bytes;
  if (pp->cbufs < 2) return fail(AQ_ERR_UNSUPPORTED, "%s: shared memory holds %d tile buffers", who, pp->cbufs);
  if (*smem > dev->smem_optin) return fail(AQ_ERR_UNSUPPORTED, "%s: needs %zu bytes of shared memory", who, *smem);
  *grid = std::min(pp->total_tiles, dev->sms);
  return AQ_OK;
}

aq_status aq_precompute(const aq_theta* th, void* W_eff, int64_t ld_weff, void* stream) {
  t_launches = 0;
  aq_status st = check_theta(th, "aq_precompute");
  if (st != AQ_OK) return st;
  if (!W_eff) return fail(AQ_ERR_INVALID_ARG, "aq_precompute: W_eff is NULL");
  if (ld_weff < th->in) return fail(AQ_ERR_SHAPE, "aq_precompute: ld_weff=%lld < in=%d", (long long)ld_weff, th->in);
  if (ld_weff % 8 != 0 || !aligned16(W_eff))
    return fail(AQ_ERR_ALIGNMENT, "aq_precompute: W_eff must be 16-byte aligned with ld_weff a multiple of 8");
  {
    Span ins[4];
    theta_spans(th, ins);
    Span we = span(W_eff, th->out, th->in, ld_weff, "W_eff");
    for (int i = 0; i < 4; ++i)
      if (overlaps(we, ins[i])) return fail(AQ_ERR_OVERLAP, "aq_precompute: W_eff overlaps %s", ins[i].name);
  }
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != AQ_OK) return st;
  PrecomputeParams pp = {};
  size_t smem = 0;
  int grid = 0;
  if ((st = plan_precompute(th, dev, &pp, &smem, &grid, kPreBf16, "aq_precompute")) != AQ_OK) return st;
  if ((st = tmap_2d(&pp.tm_we, W_eff, th->in, th->out, ld_weff, kMmaM, "W_eff")) != AQ_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  return launch_or_fail(launch_precompute(pp, grid, smem, cs, true), "launch precompute");
}

size_t aq_precompute_nvfp4_workspace_bytes(void) { return kNvfp4Partials * sizeof(float); }

aq_status aq_precompute_nvfp4(const aq_theta* th, void* q, int64_t ldq, void* sf, int sf_layout,
                              float* global_scale, int scale_mode, void* workspace, size_t workspace_bytes,
                              void* stream) {
  t_launches = 0;
  const char* who = "aq_precompute_nvfp4";
  aq_status st = check_theta(th, who);
  if (st != AQ_OK) return st;
  if (!q || !sf || !global_scale) return fail(AQ_ERR_INVALID_ARG, "%s: q, sf and global_scale must be non-NULL", who);
  if (sf_layout != AQ_SF_LINEAR && sf_layout != AQ_SF_128X4)
    return fail(AQ_ERR_INVALID_ARG, "%s: sf_layout=%d is not AQ_SF_LINEAR or AQ_SF_128X4", who, sf_layout);
  if (scale_mode != AQ_NVFP4_SCALE_FROM_AMAX && scale_mode != AQ_NVFP4_SCALE_GIVEN)
    return fail(AQ_ERR_INVALID_ARG, "%s: scale_mode=%d is not a aq_nvfp4_scale value", who, scale_mode);
  if (th->in % 16 != 0) return fail(AQ_ERR_SHAPE, "%s: in=%d is not a multiple of 16", who, th->in);
  if (ldq < th->in / 2) return fail(AQ_ERR_SHAPE, "%s: ldq=%lld < in/2=%d", who, (long long)ldq, th->in / 2);
  if (ldq % 8 != 0 || (reinterpret_cast<uintptr_t>(q) & 7u) != 0 || !aligned16(sf) ||
      (reinterpret_cast<uintptr_t>(global_scale) & 3u) != 0)
    return fail(AQ_ERR_ALIGNMENT, "%s: q and ldq must be 8-byte aligned, sf 16-byte, global_scale 4-byte", who);
  const bool from_amax = scale_mode == AQ_NVFP4_SCALE_FROM_AMAX;
  if (from_amax) {
    if (!workspace) return fail(AQ_ERR_INVALID_ARG, "%s: workspace is NULL", who);
    if (workspace_bytes < aq_precompute_nvfp4_workspace_bytes())
      return fail(AQ_ERR_WORKSPACE, "%s: workspace of %zu bytes < %zu", who, workspace_bytes,
                  aq_precompute_nvfp4_workspace_bytes());
    if ((reinterpret_cast<uintptr_t>(workspace) & 3u) != 0)
      return fail(AQ_ERR_ALIGNMENT, "%s: workspace must be 4-byte aligned", who);
  }
  const int64_t sf_bytes = sf_layout == AQ_SF_LINEAR
                               ? static_cast<int64_t>(th->out) * (th->in / 16)
                               : ceil_div(th->out, 128) * 128 * (ceil_div(th->in / 16, 4) * 4);
  {
    // byte ranges as spans of 2-byte elements (ldq is even)
    Span outs[4] = {span(q, th->out, (th->in / 2 + 1) / 2, ldq / 2, "q"),
                    span(sf, 1, (sf_bytes + 1) / 2, (sf_bytes + 1) / 2, "sf"),
                    span(global_scale, 1, 2, 2, "global_scale"),
                    span(from_amax ? workspace : nullptr, 1, kNvfp4Partials * 2, kNvfp4Partials * 2,
                         "workspace")};
    Span ins[4];
    theta_spans(th, ins);
    for (int a = 0; a < 4; ++a) {
      for (int i = 0; i < 4; ++i)
        if (overlaps(outs[a], ins[i])) return fail(AQ_ERR_OVERLAP, "%s: %s overlaps %s", who, outs[a].name, ins[i].name);
      for (int b = a + 1; b < 4; ++b)
        if (overlaps(outs[a], outs[b])) return fail(AQ_ERR_OVERLAP, "%s: %s overlaps %s", who, outs[a].name, outs[b].name);
    }
  }
  DevInfo* dev = nullptr;
  if ((st = device_info(&dev)) != AQ_OK) return st;
  PrecomputeParams pp = {};
  size_t smem = 0;
  int grid = 0;
  if ((st = plan_precompute(th, dev, &pp, &smem, &grid, kPreNvfp4, who)) != AQ_OK) return st;
  if (grid > kNvfp4Partials) return fail(AQ_ERR_UNSUPPORTED, "%s: %d CTAs exceed the partial maxima", who, grid);
  pp.q = static_cast<uint8_t*>(q);
  pp.ldq = ldq;
  pp.sf = static_cast<uint8_t*>(sf);
  pp.sf_layout = sf_layout;
  pp.sf_cols = th->in / 16;
  pp.sf_ktiles = static_cast<int32_t>(ceil_div(th->in / 16, 4));
  pp.gscale = global_scale;
  pp.partials = static_cast<float*>(workspace);
  pp.n_partials = grid;
  pp.scale_given = from_amax ? 0 : 1;
  pp.reverse = from_amax ? 1 : 0;
  pp.q16 = (ldq % 16 == 0 && (reinterpret_cast<uintptr_t>(q) & 15u) == 0) ? 1 : 0;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (from_amax) {
    if ((st = launch_or_fail(launch_precompute(pp, grid, smem, cs, true, kPreAmax), "launch W_eff amax")) != AQ_OK)
      return st;
  }
  return launch_or_fail(launch_precompute(pp, grid, smem, cs, true, kPreNvfp4), "launch NVFP4 precompute");
}

aq_status aq_device_status(void* stream) {
  DevInfo* dev = nullptr;
  aq_status st = device_info(&dev);
  if (st != AQ_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int32_t v = 0;
  if ((e = cudaMemcpy(&v, dev->status, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read device status");
  if ((e = cudaMemset(dev->status, 0, sizeof v)) != cudaSuccess) return cuda_fail(e, "clear device status");
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  if (v == AQ_OK) return AQ_OK;
  if (v == AQ_ERR_TIMEOUT) return fail(AQ_ERR_TIMEOUT, "a bounded wait inside a kernel expired");
  if (v == AQ_ERR_BOUNDS) return fail(AQ_ERR_BOUNDS, "checked build: a kernel skipped a store outside its output");
  return fail(AQ_ERR_CUDA, "unexpected device status %d", v);
}

aq_status aq_selftest_bounded_wait(uint32_t timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000)
    return fail(AQ_ERR_INVALID_ARG, "aq_selftest_bounded_wait: timeout_us=%u outside [1, 1000000]", timeout_us);
  DevInfo* dev = nullptr;
  aq_status st = device_info(&dev);
  if (st != AQ_OK) return st;
  t_launches = 0;
  return launch_or_fail(launch_bounded_wait_selftest(dev->status, uint64_t(timeout_us) * 1000u,
                                                     static_cast<cudaStream_t>(stream)),
                        "launch bounded-wait self test");
}

aq_status aq_selftest_bounds_check(void* stream) {
  DevInfo* dev = nullptr;
  aq_status st = device_info(&dev);
  if (st != AQ_OK) return st;
  t_launches = 0;
  return launch_or_fail(launch_bounds_selftest(dev->status, static_cast<cudaStream_t>(stream)),
                        "launch bounds-check self test");
}

int32_t aq_checked_build(void) {
#ifdef AQ_DEBUG_CHECKS
  return 1;
#else
  return 0;
#endif
}

aq_status aq_selftest_prefill_timeout(const aq_theta* th, const void* x, int64_t M, int64_t ldx, void* y, int64_t ldy,
                                      void* workspace, size_t workspace_bytes, uint32_t timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000)
    return fail(AQ_ERR_INVALID_ARG, "aq_selftest_prefill_timeout: timeout_us=%u outside [1, 1000000]", timeout_us);
  if (!th || th->r <= 0) return fail(AQ_ERR_INVALID_ARG, "aq_selftest_prefill_timeout: needs a bundle with r > 0");
  t_test_unreachable_t_ns = static_cast<uint64_t>(timeout_us) * 1000u;
  const aq_status st = aq_linear(th, x, M, ldx, y, ldy, workspace, workspace_bytes, stream);
  t_test_unreachable_t_ns = 0;
  return st;
}

aq_status aq_set_path(aq_path path) {
  if (path != AQ_PATH_AUTO && path != AQ_PATH_DECODE && path != AQ_PATH_PREFILL && path != AQ_PATH_MIDM)
    return fail(AQ_ERR_INVALID_ARG, "aq_set_path: unknown path %d", (int)path);
  g_path.store(path);
  return AQ_OK;
}

int32_t aq_decode_max_m(void) { return kDecodeMaxM; }
int32_t aq_last_path(void) { return t_last_path; }
int32_t aq_last_launch_count(void) { return t_launches; }
int32_t aq_abi_version(void) { return AQ_ABI_VERSION; }

const char* aq_status_string(aq_status s) {
  switch (s) {
    case AQ_OK: return "AQ_OK";
    case AQ_ERR_INVALID_ARG: return "AQ_ERR_INVALID_ARG";
    case AQ_ERR_SHAPE: return "AQ_ERR_SHAPE";
    case AQ_ERR_ALIGNMENT: return "AQ_ERR_ALIGNMENT";
    case AQ_ERR_UNSUPPORTED: return "AQ_ERR_UNSUPPORTED";
    case AQ_ERR_WORKSPACE: return "AQ_ERR_WORKSPACE";
    case AQ_ERR_OVERLAP: return "AQ_ERR_OVERLAP";
    case AQ_ERR_CUDA: return "AQ_ERR_CUDA";
    case AQ_ERR_TIMEOUT: return "AQ_ERR_TIMEOUT";
    case AQ_ERR_NUMERIC: return "AQ_ERR_NUMERIC";
    case AQ_ERR_BOUNDS: return "AQ_ERR_BOUNDS";
  }
  return "AQ_ERR_UNKNOWN";
}

const char* aq_last_error(void) { return t_err.c_str(); }

}  // extern "C"
