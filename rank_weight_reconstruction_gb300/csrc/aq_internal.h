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
constexpr int kGemmThreads = 192;  // warp 0 TMA producer, warp 1 MMA issuer, warps 2-5 epilogue
constexpr int kStageA = kMmaM * 128;  // bytes of the A tile of one stage (128 rows x 128 B)
constexpr int kHeaderBytes = 1024;    // barriers + TMEM address at the start of shared memory
constexpr int kMaxStages = 16;

// One projection family (segment) of a batched GEMM launch.
struct GemmSeg {
  CUtensorMap tm_w;  // "row" operand over the K loop: W0 [rows, K] (or V^T for the t GEMM)
  CUtensorMap tm_u;  // low-rank row operand U [rows, r]
  CUtensorMap tm_t;  // low-rank token operand t [M, r]
  const uint16_t* s; // [rows] bf16 scale, or nullptr for 1
  uint16_t* y;       // output [M, rows] bf16, row stride ldy
  int64_t ldy;
  int32_t rows;      // valid rows of this family
  int32_t r;         // rank (0: no low-rank blocks)
  int32_t n_row_tiles;
  int32_t tile_begin;  // first global tile index of this segment
};

// Tile mapping: the accumulator is D[lane, col] = sum_k A[lane, k] * B[col, k].
//   swap (decode):  A = row operand (W0 rows, `row_tile` valid lanes), B = tokens (x)
//   normal (prefill): A = tokens (x, 128 lanes), B = row operand (`row_tile` columns)
struct GemmParams {
  CUtensorMap tm_x;  // tokens operand x [M, K]
  GemmSeg seg[kMaxSeg];
  int32_t nseg;
  int32_t M;
  int32_t K;
  int32_t row_tile;     // rows of the row operand per tile (box rows of tm_w / tm_u)
  int32_t tok_tile;     // tokens per tile (box rows of tm_x / tm_t)
  int32_t n_tok_tiles;
  int32_t total_tiles;
  int32_t n_mma;        // MMA N: swap -> round_up(tok_tile, 16); normal -> round_up(row_tile, 16)
  int32_t stages;
  int32_t prefetch_w;   // 1: the row operand is a weight and may be loaded before the
                        //    previous grid completes; 0: it is produced by that grid
  uint32_t stage_bytes; // kStageA + n_mma * 128, rounded to 1024
  uint32_t tmem_cols;   // power of two >= 2 * n_mma (or n_mma without a low-rank term)
  int32_t* status;      // device status word
  uint64_t timeout_ns;
};

// t = V^T x for small M on CUDA cores, one thread-block cluster per (family, 32
// columns of t, 16 tokens); the cluster splits `in` and reduces through DSMEM.
struct DownSeg {
  const uint16_t* V;
  int64_t ldv;
  int32_t r;
  uint16_t* t;   // t [M, r] bf16 at column offset, row stride ldt
  int32_t kchunks;
  int32_t block_begin;  // first blockIdx.y of this family
};

struct DownParams {
  const uint16_t* x;
  int64_t ldx;
  int64_t ldt;
  int32_t M;
  int32_t K;
  int32_t mgroups;
  int32_t nseg;
  int32_t csize;   // cluster size (CTAs splitting K)
  int32_t kslice;  // K rows per CTA (multiple of 8)
  DownSeg seg[kMaxSeg];
};

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
  uint32_t stage_bytes;
  uint32_t tmem_cols;
  int32_t* status;
  uint64_t timeout_ns;
};

// Launch helpers implemented in aq_kernels.cu; each returns the CUDA error of the launch.
cudaError_t launch_gemm(const GemmParams& p, bool swap, int grid, size_t smem, cudaStream_t st,
                        bool pdl);
cudaError_t launch_down(const DownParams& p, int grid_y, cudaStream_t st, bool pdl);
cudaError_t launch_transpose(const TransposeParams& p, int max_r, cudaStream_t st, bool pdl);
cudaError_t launch_precompute(const PrecomputeParams& p, int grid, size_t smem, cudaStream_t st,
                              bool pdl);
cudaError_t launch_bounded_wait_selftest(int32_t* status, uint64_t timeout_ns, cudaStream_t st);
cudaError_t configure_kernels(int device, size_t max_smem);
// Records the message aq_last_error() returns on this thread and passes the status through.
int set_last_error(int status, const char* message);
int32_t* device_status_ptr(int device, cudaError_t* err);

}  // namespace aq
