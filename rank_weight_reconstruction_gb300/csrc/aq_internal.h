// aq_internal.h -- parameter blocks shared by the host planner (aq_host.cu) and the
// kernels (aq_kernels.cu). Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace aq {

constexpr int kBK = 64;            // K elements per pipeline stage: one 128-byte swizzle row
constexpr int kUmmaK = 16;         // K of one tcgen05.mma kind::f16
constexpr int kMmaM = 128;         // accumulator lanes (tokens or output rows)
constexpr int kMaxSeg = 3;         // projection families batched into one launch
constexpr int kGemmEpiWarps = 8;   // prefill GEMM epilogue: two warps per TMEM lane quadrant
constexpr int kGemmThreads = 64 + 32 * kGemmEpiWarps;  // warp 0 TMA producer, warp 1 MMA issuer, then the epilogue
constexpr int kPreThreads = 576;   // precompute: warps 2-17 epilogue, four per TMEM lane quadrant
constexpr int kStageA = kMmaM * 128;  // bytes of the A tile of one stage (128 rows x 128 B)
constexpr int kHeaderBytes = 1024;    // barriers + TMEM address at the start of shared memory
constexpr int kGemmSBufBytes = 1024;  // prefill GEMM: s of the current tile (fp32, n_mma <= 256)
constexpr int kMaxStages = 16;

// One projection family (segment) of a batched GEMM launch.
struct GemmSeg {
  CUtensorMap tm_w;  // "row" operand over the K loop: W0 [rows, K] (or V^T for the t GEMM)
  CUtensorMap tm_u;  // low-rank row operand U [rows, r]
  CUtensorMap tm_t;  // low-rank token operand t [M, r]
  CUtensorMap tm_y;  // output y for bulk stores: box {64 rows of the row operand, 32 tokens}
  const uint16_t* s; // [rows] bf16 scale, or nullptr for 1
  uint16_t* y;       // output [M, rows] bf16, row stride ldy
  int64_t ldy;
  int32_t rows;      // valid rows of this family
  int32_t r;         // rank (0: no low-rank blocks)
  int32_t n_row_tiles;
  int32_t tile_begin;  // first global tile index of this segment
  int32_t n_mma;     // MMA N of this segment's tiles (<= GemmParams::n_mma)
  int32_t tma_y;     // 1: y leaves through shared memory and bulk tensor stores
  int32_t t_seg;     // 1: computes t = x V (row operand V^T from the workspace, written by the
                     //    previous kernel); its tiles publish per-token-tile flags
  float* part;       // split K: fp32 partial sums [ksplit][M][ld_part] instead of y (no s, r = 0)
  int64_t ld_part;
};

// Segments of one prefill GEMM launch: the families, and before them their t = x V parts.
constexpr int kMaxGemmSeg = 2 * kMaxSeg;

// Tile mapping: the accumulator is D[token, col] = sum_k x[token, k] * W[col, k], with 128
// tokens per tile as the accumulator lanes and `row_tile` rows of the row operand as N.
struct GemmParams {
  CUtensorMap tm_x;  // tokens operand x [M, K]
  GemmSeg seg[kMaxGemmSeg];
  int32_t nseg;
  int32_t M;
  int32_t K;
  int32_t row_tile;     // rows of the row operand per tile (box rows of tm_w / tm_u)
  int32_t tok_tile;     // tokens per tile (box rows of tm_x / tm_t)
  int32_t n_tok_tiles;
  int32_t cluster;      // 1, or 2: CTA pairs take adjacent token tiles of one row tile; each
                        //    CTA loads half of the row operand (its own TMA loads, no
                        //    multicast) and the pair's 2-SM MMAs read both halves
  int32_t n_tok_units;  // ceil(n_tok_tiles / cluster): token tiles per row tile, in pairs
  int32_t tok_major;    // 1: units walk a token unit's row tiles first (x read once, the row
                        //    operand kept in L2); 0: a row tile's token units first
  int32_t total_tiles;  // work units: row tiles x n_tok_units, summed over the segments
  int32_t n_mma;        // MMA N: round_up(row_tile, 16)
  int32_t stages;
  int32_t prefetch_w;   // 1: the row operand is a weight and may be loaded before the
                        //    previous grid completes; 0: it is produced by that grid
  uint32_t stage_bytes; // kStageA + n_mma * 128, rounded to 1024
  uint32_t tmem_cols;   // power of two >= 2 * n_mma: two accumulator buffers
  int32_t* t_flags;     // t segments present: [0] CTAs finished, [1 + i] t tiles done for
                        // token tile i (workspace sync region; zero before, zero after)
  int32_t t_need;       // t tiles per token tile (summed over the t segments)
  int32_t n_flags;      // token tiles with a flag: n_tok_units * cluster
  int32_t head_kb;      // k blocks of tile i+1 issued before the rank-r blocks of tile i
  int32_t* status;      // device status word
  uint64_t timeout_ns;
  int32_t ksplit;       // K slices per tile (1: none); work item = unit * ksplit + slice
  int32_t kb_per;       // k blocks per slice (the last slice may have fewer)
  int32_t swap;         // 1: the row operand's 128-row tiles are the accumulator lanes and the
                        //    tokens (tok_tile <= 256 of them) the MMA N; row_tile = 128,
                        //    n_mma = tok_tile (the mid-M bucket)
};
static_assert(sizeof(GemmParams) <= 4096, "kernel parameters are limited to 4 KB");

// Split-K finalize: y = RN(s * sum_k z_k + U * sum_k t_k) from the fp32 partials of a split
// GEMM, the slices summed in order.
struct FinalizeSeg {
  const float* pz;       // [ksplit][M][ld_pz] partial sums of W0 x for this family's rows
  const float* pt;       // [ksplit][M][ld_pt] partial sums of x V, at this family's columns
  const uint16_t* s;     // [rows] bf16
  const uint16_t* U;     // [rows, ldu] bf16, r columns
  int64_t ldu;
  uint16_t* y;
  int64_t ldy;
  int32_t rows;
  int32_t r;
  int32_t block_begin;   // first blockIdx.x of this family
};
struct FinalizeParams {
  FinalizeSeg seg[kMaxSeg];
  int32_t nseg;
  int32_t M;
  int32_t ksplit;
  int64_t ld_pz;
  int64_t ld_pt;
  int64_t pz_slice;      // elements between slices of pz (M * ld_pz)
  int64_t pt_slice;
};
constexpr int kFinRows = 256;      // outputs per finalize block: consecutive rows of one token
constexpr int kFinMaxR = 256;      // largest rank the finalize stages in shared memory
constexpr int kSplitMinKb = 4;     // k blocks per slice at least
constexpr int kMaxSplit = 16;
// Largest rank for which K is split: the finalize sums the slices' partials of t and of W0 x
// with dependent global loads and runs U t on the FP32 pipes, which pays for itself only at
// small r (measured on 1152 x 6912 at M = 64 and 512: 1.2-2.5x faster for r <= 16, slower
// than the unsplit GEMM for r = 64 and 256).
constexpr int kSplitMaxRank = 16;

// Decode (M <= kDecMaxTok tokens): each W0-streaming CTA owns a contiguous range of
// output rows of one family over the full K; a few extra CTAs compute t = V^T x.
constexpr int kDecThreads = 288;        // warp 0 TMA producer, warps 1..8 mma.sync consumers
constexpr int kDecConsumers = 256;
constexpr int kDecMaxTok = 32;          // tokens the decode kernel handles
constexpr int kDecMaxEpiBytes = 48 * 1024;  // largest epilogue staging (sums + t)
constexpr int kDecMaxTCtas = 16;        // most CTAs that compute t = V^T x
constexpr int kDecLocalMaxR8 = 32;      // largest r8 for which streaming CTAs compute t themselves
constexpr int kEarlyTMax = 512;      // largest t tile (tokens x r16) warp 0 fetches during the W0 loop
// Two buffers for a chunk's s (up to 128 rows + 8 of alignment) in the kernel's header,
// after its mbarriers and flags.
constexpr int kSBufOffset = 384;
constexpr int kSBufBytes = 320;
// Workspace: [0, kSyncBytes) must be zero before first use and is left zero by every decode
// call (counters and the fp32 t accumulator); scratch that needs no initialisation follows.
constexpr size_t kSyncBytes = 128 * 1024;
constexpr size_t kSyncTAccOffset = 32 * 1024;   // t accumulator inside the sync region
constexpr int kMaxTAcc = static_cast<int>((kSyncBytes - kSyncTAccOffset) / 4);

struct DecodeSeg {
  CUtensorMap tm_w;    // W0: 3-D view {64, K/64, rows} with box {64, kbox, chunk_rows} when w3d,
                       // else 2-D [rows, K] with box {64, chunk_rows}; 128-byte swizzle
  CUtensorMap tm_v;    // V [in, r]: 2-D, no swizzle, box {r8, vbox}
  const uint16_t* s;
  const uint16_t* U;
  int64_t ldu;
  const uint16_t* V;
  int64_t ldv;
  uint16_t* y;
  int64_t ldy;
  int32_t rows;
  int32_t r;
  int32_t r8;          // round_up(r, 8): width of this family's V rows in a t CTA's staging
  int32_t r16;         // round_up(r, 16): K of the U t mma (staged U rows and t_hi / t_lo)
  int32_t t_col;       // first column of this family in t [M, r_total]
  int32_t cta_begin;   // first W0-streaming CTA of this family (counted after the t CTAs)
  int32_t chunk_rows;  // rows per chunk (TMA box rows), <= 128
  int32_t chunks;      // chunks per CTA
};

struct DecodeParams {
  CUtensorMap tm_x;    // x per stage (when !x_res): like tm_w with M rows
  CUtensorMap tm_xt;   // x for t CTAs: 2-D, no swizzle, box {vbox, M}
  DecodeSeg seg[kMaxSeg];
  const uint16_t* x;
  int64_t ldx;
  int32_t nseg;
  int32_t M;
  int32_t K;
  int32_t nkb;         // 64-wide k blocks
  int32_t kbox;        // k blocks per pipeline stage
  int32_t w3d;         // 1: W0 / x stages are single 3-D boxes (K is a multiple of 64)
  int32_t x_res;       // 1: x resident in shared memory for the whole call
  int32_t late_release; // 1: release the next kernel only once this CTA's activations arrived
  int32_t l2_prefetch; // 1: before the dependency wait, pull the W0 stages that do not fit the
                       // ring into L2 (calls whose W0 fits comfortably in L2)
  int32_t xs_ld;       // row stride (elements) of resident x: round_up(K, 64) + 8
  int32_t tok_tile;    // 16 or 32
  int32_t r_total;
  int32_t t_local;     // 1: every streaming CTA computes its family's t itself from V staged
                       // in its shared memory (small V); 0: t CTAs, see t_ctas
  int32_t t_ctas;      // CTAs [0, t_ctas) compute t into the sync region; the rest stream W0
  int32_t vbox;        // rows of `in` per V (and t-CTA x) box: a multiple of 16, <= 256
  int32_t r8_total;    // sum of r8 over the families
  int32_t ts_off;      // float offset of t_hi in the epilogue staging
  int32_t stages;
  uint32_t stage_bytes;
  uint32_t wregion;    // bytes of the W0 part of a stage: kbox * wbox_bytes, 1 KB aligned
  uint32_t wbox_bytes; // bytes of one 64-wide k block of W0 rows: round_up(max chunk_rows, 8) * 128
  uint32_t epi_bytes;  // epilogue staging: warp sums [8][16][tok_tile] (or, when t_local, the
                       // warps' partial t [8][tok_tile][r8]), then at ts_off t_hi and t_lo,
                       // bf16 [tok_tile][r16] each; 1 KB aligned
  uint32_t xres_bytes; // resident x bytes (0 if !x_res), 1 KB aligned
  uint32_t vres_bytes; // staged V of the CTA's family when t_local: [ceil(in/vbox)*vbox][r8]
  uint32_t ures_bytes; // staged U rows of a chunk, [chunk_rows][r16] per buffer, two buffers
                       // when a CTA has several chunks
  uint32_t ubuf_bytes; // bytes of one U buffer
  int32_t* counters;   // sync region: [0] t arrivals, [1] finished CTAs
  float* t_acc;        // sync region: [M][r_total]
  int32_t* status;
  uint64_t timeout_ns;
};

// Cluster decode kernel (M <= 16): a cluster of C CTAs owns `rc` rows of one family, CTA q of
// the cluster covers K slice q (k blocks [q * kb_per, (q + 1) * kb_per)); t = V^T x is formed in
// the same mma loop; partial sums are added across the cluster through distributed shared
// memory.
constexpr int kDec2MaxC = 8;   // largest cluster (K slices) of the cluster decode kernel
constexpr int kDec2Batch = 4;  // outputs per thread whose remote partial sums are loaded together
struct Dec2Seg {
  CUtensorMap tm_w;    // W0 as {64, K/64, rows}, box {64, kbox, rc}, 128-byte swizzle
  CUtensorMap tm_v;    // V [in, r]: 2-D, no swizzle, box {vrow, vbox} (zero past r)
  const uint16_t* s;
  const uint16_t* U;
  int64_t ldu;
  uint16_t* y;
  int64_t ldy;
  int32_t rows;
  int32_t r;
  int32_t r16;         // round_up(r, 16): rows of V^T in the mma tiles, width of staged U rows
  int32_t rc;          // rows per cluster (<= 256)
  int32_t cl_begin;    // first cluster of this family
};

struct Dec2Params {
  CUtensorMap tm_x;    // x as {64, K/64, M}, box {64, xkb, M}, 128-byte swizzle
  CUtensorMap tm_x2;   // gated input (act >= 0): the up projection's output, same view as tm_x
  Dec2Seg seg[kMaxSeg];
  const uint16_t* x;   // for L2 prefetch hints
  int64_t ldx;
  int32_t nseg;
  int32_t M;
  int32_t K;           // a multiple of 64
  int32_t nkb;
  int32_t C;           // cluster size = K slices
  int32_t kb_per;      // k blocks per slice
  int32_t kbox;        // k blocks per W0 stage (odd: conflict-free ldmatrix rows)
  int32_t xkb;         // k blocks of the x box (>= kb_per, odd)
  int32_t vrow;        // elements per staged V row (>= every family's r16)
  int32_t vbox;        // V rows per TMA box (multiple of 16, <= 256)
  int32_t stages;
  uint32_t stage_bytes;  // kbox * max rc * 128, 1 KB aligned
  uint32_t x_bytes, v_bytes, u_bytes, s_bytes, tf_bytes;  // shared-memory regions, 1 KB aligned
  uint32_t rx_bytes;     // receive area of the cluster exchange: [C][M][round_up(rf, 4)] + [C][r16][M] fp32
  uint32_t x2_bytes;     // the second x slice of a gated input (0 without one)
  int32_t act;           // gated input: -1 none; else the input is act(x) * x2 (kAct* below)
  const uint16_t* x2;    // for L2 prefetch hints
  int32_t staged;        // 1: x and V ride in every stage behind its W0 box (x box {64, kbox, M},
                         //    V rows {vrow, 64} per k block); no resident x or V slice
  uint32_t sx_off;       // staged: byte offset of a stage's x box
  uint32_t sv_off;       // staged: byte offset of a stage's V rows
  int32_t* status;
  uint64_t timeout_ns;
};
static_assert(sizeof(Dec2Params) <= 4096, "kernel parameters are limited to 4 KB");

// Activations of the fused MLP (aq_act in aq.h).
constexpr int kActGeluTanh = 0;
constexpr int kActSilu = 1;

// V [in, r] -> Vt [r, in] (bf16) for the prefill t GEMM.
struct TransposeSeg {
  const uint16_t* V;
  int64_t ldv;
  uint16_t* Vt;
  int64_t ldvt;
  int32_t r;
};

struct TransposeParams {
  TransposeSeg seg[kMaxSeg];
  int32_t nseg;
  int32_t K;
};

// W_eff = s * W0 + U V^T.
struct PrecomputeParams {
  CUtensorMap tm_u;   // U [out, r], box {64, 128}
  CUtensorMap tm_v;   // V [in, r],  box {64, bn}
  CUtensorMap tm_w0;  // W0 [out, in], box {64, 128}
  CUtensorMap tm_we;  // W_eff [out, in], box {64, 128}
  const uint16_t* s;
  int32_t out;
  int32_t in;
  int32_t r;
  int32_t bn;          // columns of W_eff per tile (multiple of 64, <= 256)
  int32_t n_row_tiles;
  int32_t n_col_tiles;
  int32_t total_tiles;
  int32_t stages;      // operand ring depth (U/V chunks)
  int32_t cbufs;       // W0 / W_eff tile buffers (<= 8): W0 tiles in flight while others are
                       // in the epilogue or being stored
  uint32_t stage_bytes;
  uint32_t tmem_cols;
  int32_t* status;
  uint64_t timeout_ns;
  // NVFP4 output (kPreNvfp4) and the W_eff amax pass before it (kPreAmax)
  uint8_t* q;          // codes [out, in/2] bytes, row stride ldq
  int64_t ldq;
  uint8_t* sf;         // E4M3 block scales, layout sf_layout
  int32_t sf_layout;   // AQ_SF_LINEAR or AQ_SF_128X4
  int32_t sf_cols;     // in / 16
  int32_t sf_ktiles;   // ceil(in / 64): 4-scale column tiles of the 128x4 layout
  int32_t scale_given; // 1: g read from *gscale; 0: g from the amax pass's partial maxima
  int32_t n_partials;  // partial maxima written by the amax pass (its grid)
  int32_t reverse;     // walk the tiles last to first (re-reads the amax pass's L2 tail first)
  float* gscale;       // the fp32 global decode scale g
  float* partials;     // one max|W_eff| per CTA of the amax pass
  int32_t q16;         // q and ldq 16-byte aligned: codes leave in 16-byte stores
  int32_t pf_ahead;    // W0 tiles of this CTA prefetched into L2 ahead of the TMA loads (0: off)
};

// Output of aq_precompute_kernel: bf16 W_eff, max|W_eff| partials, or NVFP4 codes + scales.
constexpr int kPreBf16 = 0;
constexpr int kPreAmax = 1;
constexpr int kPreNvfp4 = 2;
constexpr int kNvfp4Partials = 1024;   // partial maxima a workspace holds (>= any grid)
// NVFP4: 128 floats of 1/d, one per scale byte, after the operand ring
constexpr int kNvfp4TableBytes = 128 * 4;

// Launch helpers implemented in aq_kernels.cu; each returns the CUDA error of the launch.
cudaError_t launch_gemm(const GemmParams& p, int grid, size_t smem, cudaStream_t st, bool pdl);
// Most clusters of `cluster` aq_gemm_kernel CTAs with `smem` bytes each that fit at once.
cudaError_t gemm_max_clusters(size_t smem, int cluster, int* n);
// Shared memory from which one aq_gemm_kernel CTA fills an SM (CTA pairs need that: the pair
// count is taken at this size).
constexpr size_t kGemmPairMinSmem = 120 * 1024;
// k blocks of the next tile the MMA warp issues while the epilogue scales a tile by s (sized
// when four epilogue warps took about five 64-wide k blocks of a 256-wide tile for the scale
// pass; with eight it takes about half that, and the head is kept as measured)
constexpr int kGemmHeadKb = 6;
// Output staging of the prefill epilogue: per epilogue warp one buffer of 32 tokens x 64
// columns of bf16 (128-byte swizzled rows), after the ring
constexpr int kYStageBytes = 32 * 128;
constexpr int kYStageTotal = kGemmEpiWarps * kYStageBytes;
cudaError_t launch_finalize(const FinalizeParams& p, int blocks, cudaStream_t st, bool pdl);
cudaError_t launch_decode(const DecodeParams& p, int grid, size_t smem, cudaStream_t st, bool pdl);
cudaError_t configure_decode(size_t max_smem);
cudaError_t launch_decode2(const Dec2Params& p, int grid, size_t smem, cudaStream_t st, bool pdl);
// h[m, i] = RN_bf16(act(g[m, i]) * u[m, i]) in place of g (rows of `n` elements, stride ld).
cudaError_t launch_gated_act(uint16_t* g, const uint16_t* u, int64_t ld, int64_t M, int32_t n, int32_t act,
                             cudaStream_t st, bool pdl);
cudaError_t configure_decode2(size_t max_smem);
cudaError_t launch_transpose(const TransposeParams& p, int max_r, cudaStream_t st, bool pdl);
cudaError_t launch_precompute(const PrecomputeParams& p, int grid, size_t smem, cudaStream_t st,
                              bool pdl, int out_kind = kPreBf16);
cudaError_t launch_bounded_wait_selftest(int32_t* status, uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_bounds_selftest(int32_t* status, cudaStream_t st);
cudaError_t configure_kernels(int device, size_t max_smem);
// Records the message aq_last_error() returns on this thread and passes the status through.
int set_last_error(int status, const char* message);
int32_t* device_status_ptr(int device, cudaError_t* err);

}  // namespace aq
