/*
 * aq.h -- C ABI of the theta-bundle reconstruction linear on GB300 (sm_103a).
 *
 * A theta bundle replaces one projection's dense [out, in] weight by
 *   W0 [out, in]  a dense block shared by the layers of a projection family,
 *   s  [out]      a per-output-row scale,
 *   U  [out, r], V [in, r]  a rank-r delta,
 * ("How attnquant works", section "The theta bundle"). The projection is rebuilt by
 * the reconstruction identity y = s . (W0 x) + U (V^T x) and its load-time form
 * W_eff = diag(s) . W0 + U . V^T ("How attnquant works", "The reconstruction
 * identity"; "Execution paths", "Precompute-outside: the production path").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor is bfloat16, row-major, with an explicit leading dimension (in
 *   elements). Orientation follows "Execution paths", "The GEMM formulation":
 *   x [M, in], y [M, out], W0 [out, in], V [in, r], U [out, r]; s scales y's columns.
 * - Every tensor pointer is a DEVICE pointer owned by the caller; the library keeps
 *   no reference after a call returns and allocates no device memory. (The one array
 *   it owns is the fixed scratch of aq_linear_noalloc, compiled into the library.)
 * - Alignment: pointers 16-byte aligned, every leading dimension a multiple of 8
 *   elements (rows start on 16-byte boundaries: the kernels move operands with TMA).
 * - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t; NULL is
 *   the legacy default stream). They return once the work is enqueued. They may be
 *   captured into CUDA graphs. Kernels are launched with programmatic dependent
 *   launch so that a call's weight prefetch overlaps the tail of the previous one;
 *   activations and the workspace are touched only after the previous kernel in the
 *   stream finished. Weights (W0, s, U, V) may be read before then, so they must not
 *   be written by a kernel that is still running and has released its dependents
 *   early (griddepcontrol.launch_dependents). This library's own kernels release
 *   early only when their outputs are activations; aq_precompute does not, so its
 *   W_eff may serve as the very next call's W0 on the same stream.
 * - Errors: argument errors are detected on the host before anything is enqueued and
 *   returned as an aq_status; aq_last_error() then describes them (thread-local).
 *   No C++ exception crosses this interface. Faults detected on the device (a bounded
 *   wait that expired) are recorded in a per-device status word read by
 *   aq_device_status().
 * - Rounding: products accumulate in fp32; each output element is rounded to bf16
 *   once (nearest-even). On the prefill path t = V^T x is held in bf16 between the
 *   tiles that produce it and those that consume it; on the decode path it stays fp32
 *   and enters U t as a pair of bf16 values (about 16 significant bits).
 */
#ifndef AQ_H_
#define AQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AQ_ABI_VERSION 1

/* Largest supported rank r. ("Execution paths", "The custom op": a path refuses ranks
 * beyond what its layout supports and says so; here the limit is 256.) */
#define AQ_MAX_RANK 256

typedef enum aq_status {
  AQ_OK = 0,
  AQ_ERR_INVALID_ARG = 1,  /* NULL pointer where one is required, negative size, bad value */
  AQ_ERR_SHAPE = 2,        /* out/in/r inconsistent, leading dimension too small, size limits */
  AQ_ERR_ALIGNMENT = 3,    /* pointer not 16-byte aligned or leading dimension not a multiple of 8 */
  AQ_ERR_UNSUPPORTED = 4,  /* r > AQ_MAX_RANK, or the current device is not sm_103 */
  AQ_ERR_WORKSPACE = 5,    /* workspace missing, misaligned or smaller than required */
  AQ_ERR_OVERLAP = 6,      /* an output buffer overlaps an input buffer */
  AQ_ERR_CUDA = 7,         /* a CUDA runtime or driver call failed (message in aq_last_error) */
  AQ_ERR_TIMEOUT = 8,      /* device side: a bounded wait inside a kernel expired */
  AQ_ERR_NUMERIC = 9,      /* aq_randomized_svd: a factorisation met a non-positive pivot */
  AQ_ERR_BOUNDS = 10       /* checked build only: a kernel skipped a store outside its output */
} aq_status;

/* One projection's theta bundle. All pointers are device pointers to bf16 data.
 *   W0    [out, in], row stride ld_w0 >= in
 *   s     [out], contiguous
 *   U     [out, r], row stride ld_u >= r     (may be NULL iff r == 0)
 *   V     [in, r],  row stride ld_v >= r     (may be NULL iff r == 0)
 * r == 0 means U and V are empty and the weight is the scaled shared block alone
 * ("How attnquant works", "How the decomposition produces s, U, and V").
 * Limits: 1 <= out, 1 <= in, both < 2^31 and in <= 65536 * 64; 0 <= r <= AQ_MAX_RANK. */
typedef struct aq_theta {
  const void* W0;
  int64_t ld_w0;
  const void* s;
  const void* U;
  int64_t ld_u;
  const void* V;
  int64_t ld_v;
  int32_t out;
  int32_t in;
  int32_t r;
} aq_theta;

/* Workspace of aq_linear / aq_linear_qkv / aq_linear_multi. Its first
 * AQ_WORKSPACE_SYNC_BYTES hold the counters and the fp32 accumulator of t = V^T x that the
 * CTAs of the decode kernel share, and the per-token-tile flags of the prefill kernel:
 * that part must be zero before the workspace is first used (e.g. cudaMemset once after
 * allocating it), and every call that completes leaves it zero again, so one workspace
 * can serve any sequence of calls, shapes and paths on a stream. The rest is scratch
 * that needs no initialisation (the decode kernel uses none of it; t in bf16 and a
 * transposed copy of V at prefill; and, when a prefill call splits K, the fp32 partial
 * sums of every K slice). After a call whose bounded wait expired
 * (aq_device_status() == AQ_ERR_TIMEOUT) the sync part must be zeroed again. */
#define AQ_WORKSPACE_SYNC_BYTES (128u * 1024u)

/* Bytes of device workspace for aq_linear (n_theta == 1), aq_linear_qkv (n_theta == 3,
 * pass the three bundles) or aq_linear_multi (n_theta == n) over M tokens, on either path,
 * including room for the fp32 partial sums of a prefill call that splits K (see aq_linear).
 * A smaller workspace that still holds the call's minimum is accepted: the call then splits
 * K into fewer slices, or not at all. Returns 0 if the call needs none and splits nothing
 * (M == 0, or M above the decode limit with r == 0 and too many output tiles to split), and
 * (size_t)-1 for invalid arguments. */
size_t aq_linear_workspace_bytes(const aq_theta* th, int32_t n_theta, int64_t M);

/* y[m, o] = RN_bf16( s[o] * sum_i W0[o,i] x[m,i] + sum_k U[o,k] * t[m,k] ),
 *           t[m, k] = sum_i V[i,k] x[m,i]
 * ("How attnquant works", "The reconstruction identity"; axes as in "Execution paths",
 * "The GEMM formulation").
 *   th        the bundle (host pointer to the struct; the struct's pointers are device)
 *   x         [M, in] device, row stride ldx >= in
 *   y         [M, out] device, row stride ldy >= out; must not overlap x, W0, s, U, V
 *   workspace device, aq_linear_workspace_bytes(th, 1, M) bytes (a smaller one that holds
 *             the call's minimum also works; the error names that minimum), 256-byte
 *             aligned, first AQ_WORKSPACE_SYNC_BYTES zero (see above); NULL when no
 *             workspace is needed
 *   stream    cudaStream_t
 * M == 0 is a no-op returning AQ_OK. Decode (M <= aq_decode_max_m() = 32) is one
 * launch that streams W0 once, split evenly over the SMs. The mid-M and prefill GEMMs (see
 * aq_set_path) transpose V and run one tcgen05 GEMM whose first tiles compute t = x V. All
 * fuse s and the rank-r term into the epilogue. A GEMM call whose output tiles fill at most
 * half of the SMs over a deep K, with r <= 16, instead splits K over more CTAs that write
 * fp32 partial sums, and a third launch computes y from them in a fixed order. Concurrent
 * calls sharing one workspace must be ordered on the GPU. */
aq_status aq_linear(const aq_theta* th, const void* x, int64_t M, int64_t ldx,
                    void* y, int64_t ldy, void* workspace, size_t workspace_bytes,
                    void* stream);

/* The three attention projections of one layer over the same x in one pass
 * ("Execution paths", "Precompute-outside: the production path" and "The GEMM
 * formulation": Q/K/V batched into one dispatch). th[0..2] are the q, k and v
 * bundles (all with the same `in`; out and r may differ); y[j] is [M, th[j].out] with
 * row stride ldy[j]. Passing y[1] = y[0] + out_q, y[2] = y[1] + out_k and a common
 * ldy = out_q + out_k + out_v yields the concatenated [M, q|k|v] layout. Outputs must
 * not overlap each other or any input. workspace: aq_linear_workspace_bytes(th, 3, M). */
aq_status aq_linear_qkv(const aq_theta th[3], const void* x, int64_t M, int64_t ldx,
                        void* const y[3], const int64_t ldy[3],
                        void* workspace, size_t workspace_bytes, void* stream);

/* Up to AQ_MAX_FAMILIES projections over the same x in one pass: aq_linear_qkv for any
 * n in [1, AQ_MAX_FAMILIES] -- gate and up of an MLP (n = 2) are the other pair the pages
 * batch ("Execution paths", "Precompute-outside: the production path": Q/K/V and gate-up
 * fusion). th[0..n-1] share `in`; y[j] is [M, th[j].out] with row stride ldy[j]; outputs
 * must not overlap each other or any input. workspace: aq_linear_workspace_bytes(th, n, M).
 * n outside [1, AQ_MAX_FAMILIES] returns AQ_ERR_INVALID_ARG. */
#define AQ_MAX_FAMILIES 3
aq_status aq_linear_multi(const aq_theta* th, int32_t n, const void* x, int64_t M, int64_t ldx,
                          void* const* y, const int64_t* ldy, void* workspace, size_t workspace_bytes,
                          void* stream);

/* aq_linear for callers that may not allocate device memory. The paper has no
 * counterpart: this entry point exists for callers such as plugins inside a runtime that
 * owns all device memory, or serving loops that forbid allocation after start-up.
 * Same arguments and results as aq_linear, minus the workspace: its scratch comes from one
 * array of AQ_NOALLOC_WORKSPACE_BYTES compiled into the library, which every GPU that uses
 * the library keeps allocated until the process exits. The caller still passes x and y.
 *   - A call whose minimum scratch need exceeds AQ_NOALLOC_WORKSPACE_BYTES is rejected
 *     with AQ_ERR_WORKSPACE (message in aq_last_error) before anything is enqueued. Split-K
 *     partial sums use what the array has beyond that minimum (for r = 0 too, whose
 *     minimum is zero), so such a call may split K into fewer slices than with a full
 *     workspace.
 *   - The first call on a device looks up the array's device address on that device;
 *     make that first call before capturing a stream into a CUDA graph. The address is
 *     looked up again when the device's current context has changed since (after
 *     cudaDeviceReset, for example); a call that does so must not be captured either.
 *   - All calls on a device share the one array and it keeps the previous call's
 *     contents. Its sync part (see AQ_WORKSPACE_SYNC_BYTES) starts at zero when the
 *     library is loaded and every completed call leaves it zero; after an expired wait
 *     (AQ_ERR_TIMEOUT) results of later calls are undefined. Calls that can overlap on
 *     the GPU -- on different streams without ordering between them -- race on the
 *     array; order them.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine. */
#define AQ_NOALLOC_WORKSPACE_BYTES (8u * 1024u * 1024u)
aq_status aq_linear_noalloc(const aq_theta* th, const void* x, int64_t M, int64_t ldx,
                            void* y, int64_t ldy, void* stream);

/* Test hook for aq_linear_noalloc (no counterpart in the paper): copies `bytes` of the
 * built-in scratch array of the current device, starting at `offset`, to `dst` (host or
 * device memory), ordered on `stream`, and returns once the copy is done. Lets a test check
 * that the array's sync part reads back zero after a series of calls. A range outside the
 * array returns AQ_ERR_INVALID_ARG. Allocates nothing. */
aq_status aq_noalloc_scratch_read(void* dst, size_t offset, size_t bytes, void* stream);

/* The fused MLP of one layer ("Execution paths", "The custom op": gate, up, activation and down
 * of a layer in one dispatch), every projection a reconstruction linear:
 *   y = down( RN_bf16( act(g) * u ) ),  g = RN_bf16(gate(x)), u = RN_bf16(up(x))
 * The pages do not name the activation. AQ_ACT_GELU_TANH is the tanh approximation of GELU,
 * v/2 (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))), the MLP activation of Gemma 3 (whose shapes the
 * benchmark uses); AQ_ACT_SILU is v / (1 + e^-v). gate and up share [inter, in]; down is
 * [out, inter]. x [M, in], y [M, out] as for aq_linear. gate and up run as one batched launch.
 * When the cluster decode kernel takes the down projection with both of its input slices (g and
 * u) staged (up to 16 tokens, and the slices within its shared memory: up to 4 tokens at
 * inter = 6912), the activation is formed inside that kernel as it loads its input: two
 * launches in all. Otherwise one activation pass runs between them.
 * workspace: aq_mlp_workspace_bytes(gate, up, down, M) bytes, 256-byte aligned, its first
 * AQ_WORKSPACE_SYNC_BYTES zero before first use (as for aq_linear); it also holds g and u. */
typedef enum aq_act { AQ_ACT_GELU_TANH = 0, AQ_ACT_SILU = 1 } aq_act;
size_t aq_mlp_workspace_bytes(const aq_theta* gate, const aq_theta* up, const aq_theta* down, int64_t M);
aq_status aq_mlp(const aq_theta* gate, const aq_theta* up, const aq_theta* down, aq_act act, const void* x,
                 int64_t M, int64_t ldx, void* y, int64_t ldy, void* workspace, size_t workspace_bytes,
                 void* stream);

/* W_eff[o, i] = RN_bf16( s[o] * W0[o,i] + sum_k U[o,k] * V[i,k] )
 * ("Execution paths", "Precompute-outside: the production path": built once per
 * layer at load). W_eff is [out, in] device, row stride ld_weff >= in, and must not
 * overlap W0, s, U or V. Needs no workspace. The sum over k accumulates in fp32 on
 * the tensor cores; s * W0 is exact in fp32; one final rounding. */
aq_status aq_precompute(const aq_theta* th, void* W_eff, int64_t ld_weff, void* stream);

/* W_eff quantized to NVFP4 as it is formed, never written in bf16 ("Execution paths",
 * "Precompute-outside: the production path": each W_eff quantized to 4 bits at load;
 * "Internals and extension", "Nvfp4Spec": two E2M1 values per byte, so the [out, in]
 * weight is held as [out, in/2] bytes, one FP8-E4M3 scale per 16 values along in, one
 * fp32 global scale; scales in a linear [out, in/16] layout or a "128x4" layout padded to
 * [ceil(out,128), ceil(in/16,4)] for Blackwell GEMMs).
 *
 * The value quantized is the fp32 W_eff of aq_precompute before its bf16 rounding. The
 * rule, each step one fp32 operation rounded to nearest even (the pages state none):
 *   g = global scale (decode multiplier: weight = e2m1 * e4m3 * g)
 *   per 16 values x along in: a = max|x|; scale = E4M3(a * (1/(6 g))), ties to even,
 *   clamped to 448 (1/(6 g) formed once); d = scale * g; code = E2M1(x * (1/d)), ties to the
 *   even code, clamped to +-6, sign of x kept (a d of 0 gives +0 codes).
 * Codes: byte j of a row holds columns 2j (low nibble) and 2j+1 (high nibble).
 *
 * q: [out, in/2] bytes, device, row stride ldq >= in/2 bytes, ldq and q 8-byte aligned.
 * in must be a multiple of 16 (AQ_ERR_SHAPE otherwise).
 * sf: device, 16-byte aligned; sf_layout AQ_SF_LINEAR: out * (in/16) bytes, row o at
 *   o * (in/16); AQ_SF_128X4: ceil(out,128) * ceil(in/16,4) bytes in tiles of 128 rows by 4
 *   scale columns (512 bytes each, tiles of one row band consecutive along in, bands
 *   consecutive), the scale of row r, column k of a tile at 16 (r mod 32) + 4 (r div 32) + k;
 *   padding entries are written as 0. (The pages give the padded shape, not this order.)
 * global_scale: one fp32 in device memory. scale_mode AQ_NVFP4_SCALE_GIVEN: read as g (one
 *   launch). AQ_NVFP4_SCALE_FROM_AMAX: written with g = RN(max|W_eff| / 2688) (2688 = 6 * 448:
 *   the largest block lands on the largest E4M3 scale); a first launch finds max|W_eff|
 *   (each CTA's maximum into `workspace`, aq_precompute_nvfp4_workspace_bytes() bytes,
 *   4-byte aligned, no initial contents needed), a second quantizes, walking the tiles in
 *   reverse so that the W0 tail still in L2 is read first. workspace may be NULL when given.
 * None of q, sf, global_scale, workspace may overlap each other or W0, s, U, V. */
typedef enum aq_sf_layout { AQ_SF_LINEAR = 0, AQ_SF_128X4 = 1 } aq_sf_layout;
typedef enum aq_nvfp4_scale { AQ_NVFP4_SCALE_FROM_AMAX = 0, AQ_NVFP4_SCALE_GIVEN = 1 } aq_nvfp4_scale;
size_t aq_precompute_nvfp4_workspace_bytes(void);
aq_status aq_precompute_nvfp4(const aq_theta* th, void* q, int64_t ldq, void* sf, int sf_layout,
                              float* global_scale, int scale_mode, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Synchronises `stream`, then returns the device status word of the current device
 * (AQ_OK, AQ_ERR_TIMEOUT if a kernel's bounded wait expired since the last clear, or in the
 * checked build AQ_ERR_BOUNDS if a kernel skipped an out-of-range store)
 * and clears it. A kernel whose wait expires stops its work (its outputs are then
 * undefined), releases its tensor memory and exits; the CUDA context stays usable.
 *
 * Residency contract. The CTAs of one decode launch hand t = V^T x to each other through
 * the workspace (t CTAs publish it, the W0-streaming CTAs wait for it, one CTA waits for
 * all of them before it clears the sync region), and the prefill GEMM's tiles wait for the
 * t tiles of the same launch. These launches are sized to fit on the GPU at once, so every
 * wait ends when the launch has the device to itself or shares it with other work of this
 * process that completes. If SMs are held for longer by another context, an MPS client or a
 * green context, some CTAs may not run until the waits of others expire: such a call ends
 * with AQ_ERR_TIMEOUT in the status word and undefined outputs, and reports nothing else.
 * Callers that share the GPU that way should poll aq_device_status() after a batch of
 * calls (it synchronises the stream) and recompute the batch when it reports a timeout.
 * The cluster decode kernel (M <= 16) is not subject to this: its CTAs wait only on the
 * other CTAs of their thread-block cluster, which the hardware schedules together. */
aq_status aq_device_status(void* stream);

/* Test hook for the bounded-wait path: launches one block that waits on a barrier no
 * thread ever arrives on, with a limit of timeout_us microseconds (1..1000000). The
 * wait expires, the block records AQ_ERR_TIMEOUT in the device status word and
 * exits; aq_device_status() then reports it. No fault, trap or hang is involved. */
aq_status aq_selftest_bounded_wait(uint32_t timeout_us, void* stream);

/* Checked build (compiled with AQ_DEBUG_CHECKS; libaq_gb300_debug.so): every plain output store
 * of the hot-path kernels (decode y, the GEMM's column and partial-sum stores, NVFP4 codes and
 * scales) checks its index against the extent of the output it addresses; a violation skips
 * the store and sets the device status word to AQ_ERR_BOUNDS. TMA stores are bounded by their
 * tensor maps in every build. aq_checked_build() is 1 in that build, 0 otherwise.
 * aq_selftest_bounds_check launches one thread that checks two indices outside their extents
 * (nothing is accessed): afterwards aq_device_status() reports AQ_ERR_BOUNDS in the checked
 * build and AQ_OK in the normal one. */
int32_t aq_checked_build(void);
aq_status aq_selftest_bounds_check(void* stream);

/* Test hook for the bounded waits of a real kernel: runs aq_linear on the prefill GEMM with
 * its wait for the t tiles of the same launch set to a count no tile reaches and a limit of
 * timeout_us microseconds (1..1000000). Needs r > 0, a call that takes the t tiles inside the
 * GEMM launch and unpaired CTAs (one token tile, no split of K), else AQ_ERR_UNSUPPORTED. The
 * waits expire; each CTA records AQ_ERR_TIMEOUT, lets its issued copies land and its issued
 * MMAs finish (bounded), frees its tensor memory, counts itself out (the last CTA returns the
 * workspace's sync region to zero) and exits. y is undefined afterwards; aq_device_status()
 * reports the timeout and the context stays usable. No fault, trap or hang is involved. */
aq_status aq_selftest_prefill_timeout(const aq_theta* th, const void* x, int64_t M, int64_t ldx, void* y, int64_t ldy,
                                      void* workspace, size_t workspace_bytes, uint32_t timeout_us, void* stream);

/* Path selection for aq_linear / aq_linear_qkv / aq_linear_multi. Three kernels serve the
 * three token buckets of one call:
 *   AQ_PATH_DECODE   the mma.sync streaming kernel, M <= aq_decode_max_m() = 32: W0 split by
 *                    output rows over the SMs, x resident, t = V^T x within the launch;
 *   AQ_PATH_MIDM     the tcgen05 GEMM with 128 output rows per tile as the accumulator lanes
 *                    and the tokens (up to 256 per tile) as the MMA N, so that each W0 tile is
 *                    read once for all tokens; a transpose of V and t = x V inside the launch;
 *   AQ_PATH_PREFILL  the tcgen05 GEMM with 128 tokens per tile as the accumulator lanes and
 *                    output rows as N (CTA pairs, 2-SM MMAs), for large M.
 * AQ_PATH_AUTO picks by M and size, as measured on GB300: decode up to 32 tokens, except that
 * from 16 tokens a call whose W0 (summed over its families) holds 128 MB or more takes the
 * prefill GEMM; above 32 tokens the prefill GEMM, except that calls of 1024 to 4096 tokens
 * whose families have at most 16 tiles of 128 rows over K >= 4096 take the AQ_PATH_MIDM GEMM.
 * The other values force a path for tests: mid-M and prefill work for every M, decode for
 * M <= aq_decode_max_m() (larger M returns AQ_ERR_UNSUPPORTED). Process-wide setting. */
typedef enum aq_path { AQ_PATH_AUTO = 0, AQ_PATH_DECODE = 1, AQ_PATH_PREFILL = 2, AQ_PATH_MIDM = 3 } aq_path;
aq_status aq_set_path(aq_path path);
int32_t aq_decode_max_m(void);
/* Path the last aq_linear / aq_linear_qkv / aq_linear_multi call on this thread took (an
 * aq_path value other than AQ_PATH_AUTO; 0 if none). */
int32_t aq_last_path(void);

/* Number of kernel launches the last successful aq_* call on this thread enqueued. */
int32_t aq_last_launch_count(void);

/* ---------------------------------------------------------------------------------
 * The decomposition that produces a bundle ("How attnquant works", "How the decomposition
 * produces s, U, and V"), run on the GPU in double precision. It is a load-time step: every
 * call is stream-ordered like the others, and aq_randomized_svd synchronises its stream at
 * the end to report a numerical breakdown.
 * --------------------------------------------------------------------------------- */

/* W0 of one band: W0[o, i] = RN_bf16( (sum over l of weights[l][o, i]) / L ), the sum in fp64
 * in layer order ("W0 is the mean of the projection weights across the layers that share it").
 *   weights  host array of L device pointers to bf16 [out, in] matrices, row stride ld
 *   W0       device bf16 [out, in], row stride ld_w0
 * 1 <= L <= 256. */
aq_status aq_band_mean(const void* const* weights, int32_t L, int32_t out, int32_t in, int64_t ld, void* W0,
                       int64_t ld_w0, void* stream);

/* Per-row least-squares scale of W0 toward one layer's weight and the residual it leaves:
 *   s[o]       = RN_bf16( (w[o] . W0[o]) / (W0[o] . W0[o]) ), 1 for a W0 row of zeros
 *   resid[o,i] = w[o,i] - s[o] * W0[o,i]   (fp64, against the stored bf16 s)
 * The dot products accumulate in fp64 in a fixed order. weight and W0 are device bf16 [out, in]
 * with row strides ldw and ld_w0, s device bf16 [out], resid device fp64 [out, ld_r]. */
aq_status aq_ls_residual(const void* weight, int64_t ldw, const void* W0, int64_t ld_w0, int32_t out, int32_t in,
                         void* s, double* resid, int64_t ld_r, void* stream);

/* Rank-r factors of A [m, n] (device fp64, row stride lda) by the randomized SVD the pages name
 * (Halko, Martinsson and Tropp, 2009): Y = A Omega, Q = orth(Y), power_iters times
 * Q = orth(A orth(A^T Q)), B = Q^T A = W S Vb^T; U = Q W[:, :r] S[:r] (bf16 [m, ld_u]) and
 * V = Vb[:, :r] (bf16 [n, ld_v]), so U V^T approximates A. Omega [n, k] (device fp64, row stride
 * ld_omega) is the caller's random test matrix, k = r + oversampling, r <= k <= min(m, n) and
 * k <= 256; k = min(m, n) captures the whole range, which makes the factors the exact rank-r
 * truncation (the pages' fallback for min(m, n) <= 256). orth() is CholeskyQR2, the small SVD
 * comes from a Jacobi eigen-decomposition of B B^T, all in fp64. Factors are unique only up to
 * the sign of each pair of columns (and the order of equal singular values): compare U V^T.
 * workspace: device, aq_randomized_svd_workspace_bytes(m, n, k, r) bytes, 16-byte aligned.
 * Returns AQ_ERR_NUMERIC if a Cholesky pivot is not positive (A Omega rank deficient). */
size_t aq_randomized_svd_workspace_bytes(int32_t m, int32_t n, int32_t k, int32_t r);
aq_status aq_randomized_svd(const double* A, int64_t lda, int32_t m, int32_t n, int32_t r, const double* omega,
                            int64_t ld_omega, int32_t k, int32_t power_iters, void* U, int64_t ld_u, void* V,
                            int64_t ld_v, void* workspace, size_t workspace_bytes, void* stream);

const char* aq_status_string(aq_status status);
/* Thread-local description of the last error returned on this thread ("" if none). */
const char* aq_last_error(void);
int32_t aq_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AQ_H_ */
