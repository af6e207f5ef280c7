/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 skinny GEMM library.
 *
 *   Y[M][N] (bf16) = X[M][K] (bf16) . dequant(W)[N][K]^T,  fp32 accumulation,
 *   dequant(W)[n][k] = scale[n][k / G] * (code(n, k) - 8),  G = group_size.
 *
 * The op: "[ROCm][Kernel] W4A16 skinny GEMM: hand-asm kernel for gfx1151"
 * (opening paragraph: int4 weights, bf16 activations, N x K weight shapes;
 * section 1 "Magic-constant bf16 dequant": weight = scale * (n - 8)).  The
 * packing rule (low nibble = even k), the atomic-free split-K workspace
 * [SPLIT_K][M][N] and the device-side grouped row starts come from "Add
 * Triton BF16xINT4 rowwise GEMM for ROCm gfx942/gfx950", section
 * "Implementation" (paragraphs "Fused A-operand dot", "Split-K without
 * atomics", "Native fused grouped kernel").
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev, X, Y, W_*, scales, workspace and out are DEVICE
 *    pointers; `stream` is a cudaStream_t passed as void* (NULL = legacy
 *    default stream).  All buffers are owned by the caller.
 *  - Matrices are dense and row-major.  bf16 values travel as their raw
 *    16-bit patterns (w4a16_bf16).
 *  - The library never allocates, frees or synchronises, and never copies
 *    between host and device inside a call; kernels are enqueued on `stream`
 *    and the call returns.  (The one exception is the checking call
 *    w4a16_read_error_word, which is not on the GEMM's path.)  No entry point
 *    reads the environment.
 *  - Arguments are validated on the host before anything is enqueued; a
 *    failed check returns an error status and launches nothing.  A launch
 *    failure returns W4A16_ERR_CUDA.  Kernels never trap.
 *  - group_size G (columns per scale) is 128, 64 or 32
 *    (W4A16_ERR_UNSUPPORTED otherwise; the gfx1151 page's "Benchmark results
 *    (per-GEMM)" use group_size=32); scales are bf16 [N][K/G].  K must be a
 *    positive multiple of 128 whatever G is; N >= 1; M >= 0 (M == 0 launches
 *    nothing).
 *  - X, W_packed and workspace must be 16-byte aligned; scales and Y 2-byte
 *    aligned (W4A16_ERR_INVALID_ARG otherwise).
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t w4a16_bf16; /* raw bf16 bit pattern */

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = 1,          /* null pointer, bad shape, misalignment */
    W4A16_ERR_UNSUPPORTED = 2,          /* group_size not 128, 64 or 32, or an option not available */
    W4A16_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below what the call needs */
    W4A16_ERR_CUDA = 4                  /* a CUDA runtime call or launch failed */
} w4a16_status;

/* Which kernel family computes a plain (non-grouped) call. */
typedef enum {
    W4A16_ARM_AUTO = 0,     /* dispatcher decides (M <= 16: decode, else tensor) */
    W4A16_ARM_DECODE = 1,   /* register-dequant mma.sync streaming arm */
    W4A16_ARM_TENSOR = 2    /* TMA + TMEM + tcgen05.mma arm */
} w4a16_arm;

/* w4a16_options.flags bits. */
enum {
    /* W_packed, scales and zero points are resident: no kernel still running
     * on the stream when the call is made writes them (they were written
     * before that kernel started, e.g. when the model was loaded).  The call's
     * kernel is launched with programmatic dependent launch and may then start
     * streaming the weights into shared memory while the previous kernel on
     * the stream is still running; X is read, and Y and the workspace are
     * written, only after that kernel has completed.  Without the flag nothing
     * is read before it has completed.  The decode arm uses it; the tensor arm
     * (one large CTA per SM, which cannot start beside the previous call's)
     * reads nothing before the previous kernel has completed either way.  Do
     * not set it when W_packed, scales or zero points alias the output or
     * workspace of a call just before on the same stream. */
    W4A16_FLAG_RESIDENT_WEIGHTS = 1,
    /* Decode-arm kernel choice (for tests and tuning; by default the
     * dispatcher chooses).  WHOLE_K: the kernel in which every CTA covers all
     * of K for a few 16-row blocks of W, its warps split K among themselves
     * and add their partial sums in shared memory, so K is never split across
     * CTAs (no workspace, no reduce kernel); it takes up to 16 tokens whose X
     * rows fit its shared-memory ring next to the CTA's scales (at least three
     * stages of 16 KB of weights and their X columns), with 128-wide scale
     * groups; otherwise the call returns W4A16_ERR_UNSUPPORTED.  K_SLICES:
     * never that kernel.  Setting
     * both is W4A16_ERR_INVALID_ARG. */
    W4A16_FLAG_DECODE_WHOLE_K = 2,
    W4A16_FLAG_DECODE_K_SLICES = 4,
    /* Plan for the zero-point variant (w4a16_plan / w4a16_workspace_bytes
     * queries; w4a16_gemm_zp sets it itself).  Passing it to any other call
     * is W4A16_ERR_INVALID_ARG. */
    W4A16_FLAG_ZERO_POINTS = 8,
    /* Test only: exercises the failure path without faulting the GPU.  The
     * decode arm's K-slice kernel is launched with no weight copies and with
     * its bounded waits cut from 2 s to 1 ms, so every CTA gives up: the call
     * returns W4A16_OK (the launch itself succeeds), every output it owns
     * (Y, or the split-K workspace and through the reduce Y) becomes NaN, and
     * the device error word gets W4A16_ERROR_WAIT_TIMEOUT.  With the tensor
     * arm or the whole-K kernel the call returns W4A16_ERR_UNSUPPORTED. */
    W4A16_FLAG_TEST_STALL = 16
};

/* Bits of the device error word (w4a16_read_error_word). */
enum {
    /* A bounded wait inside a kernel ran out (2 s without progress): the CTA
     * stopped, let its copies in flight land, released its tensor memory and
     * wrote NaN to every output it owned, so the call's result holds NaN
     * where it is incomplete. */
    W4A16_ERROR_WAIT_TIMEOUT = 1
};

/* Overrides for tests and tuning.  Zero-initialised = automatic. */
typedef struct {
    int arm;          /* w4a16_arm */
    int split_k;      /* 0 = automatic, else the requested number of K slices, clamped to
                         K/128.  The decode arm rounds it up to the nearest count whose
                         slices hold 1, 2, 4, 8 or (up to 8 tokens) 16 of the 128-wide
                         blocks each (with G < 128, at most 16 (8 tokens) or 8 scale
                         groups per slice). */
    int tile_tokens;  /* tensor arm only: 0 = automatic, else tokens per tile (32..256, multiple of 32) */
    int flags;        /* W4A16_FLAG_* bits; unknown bits are rejected (W4A16_ERR_INVALID_ARG) */
} w4a16_options;

/* What the dispatcher chose for a shape on the current device. */
typedef struct {
    int arm;              /* w4a16_arm actually used (never AUTO) */
    int split_k;          /* K slices (1 = no workspace, output written directly) */
    int tile_tokens;      /* tokens per tile (decode arm: 8 or 16 per pass) */
    int ctas;             /* CTAs in the main launch */
    size_t workspace_bytes;
    int whole_k;          /* 1: the decode arm's whole-K kernel (see W4A16_FLAG_DECODE_WHOLE_K) */
} w4a16_plan_info;

/* Human-readable name of a status code (static string, never NULL). */
const char *w4a16_status_string(int status);

/* The device-side error word of the current device: the OR of the
 * W4A16_ERROR_* bits that this library's kernels have recorded since it was
 * last cleared (kernels never trap; a pipeline that cannot make progress
 * records a bit and ends).  *out receives the word; clear != 0 resets it to 0.
 * Host only and synchronous: it waits for all work on the device
 * (cudaDeviceSynchronize) and copies the word back, so it is a checking call,
 * not one for the GEMM's path, and it cannot be captured in a CUDA graph.  The
 * pages have no counterpart (their kernels report nothing on the device); this
 * is the library's own failure report. */
w4a16_status w4a16_read_error_word(int *out, int clear);

/* Version of the packed-weight layout written by w4a16_pack_weights.  A packed
 * buffer is only valid for a library reporting the same version. */
int w4a16_layout_version(void);

/* Bytes of the packed weight buffer for an N x K matrix: N rounded up to a
 * multiple of 128, times K/2.  Returns 0 when N < 1 or K is not a positive
 * multiple of 128.  Host only. */
size_t w4a16_packed_weight_bytes(int N, int K);

/* Rearrange canonical int4 weights into the kernels' layout.
 *  w_canon:  device, uint8 [N][K/2]; byte j of row n holds the code of
 *            k = 2j in bits 0-3 and of k = 2j+1 in bits 4-7 ("Add Triton
 *            BF16xINT4 ...", "Fused A-operand dot": low nibble <-> even K).
 *  w_packed: device, w4a16_packed_weight_bytes(N, K) bytes, written fully
 *            (padding rows hold code 8, i.e. weight 0).  Must not overlap
 *            w_canon.  The packed layout does not depend on the group size,
 *            and the scales need no repacking: every entry point takes them
 *            as bf16 [N][K/G].
 * The CUTLASS path that page mentions also preshuffles the weights; this
 * layout is this library's own. */
w4a16_status w4a16_pack_weights(const uint8_t *w_canon, uint8_t *w_packed, int N, int K,
                                void *stream);

/* Plan a plain call on the current device (host only, no launch): fills
 * *info (may be NULL) and, when bytes != NULL, the workspace size the call
 * needs (0 when no split).  `opts` may be NULL. */
w4a16_status w4a16_plan(int M, int N, int K, int group_size, const w4a16_options *opts,
                        w4a16_plan_info *info);

/* Workspace bytes w4a16_gemm needs for this shape on the current device
 * (the split-K partial sums, fp32 [SPLIT_K][M][N]; 0 when no split). */
w4a16_status w4a16_workspace_bytes(int M, int N, int K, int group_size, size_t *bytes);

/* Y = X . dequant(W)^T.
 *  X:        device bf16 [M][K].          Y: device bf16 [M][N].
 *  W_packed: output of w4a16_pack_weights for (N, K).
 *  scales:   device bf16 [N][K/G], G = group_size.
 *  workspace/workspace_bytes: device scratch of at least
 *            w4a16_workspace_bytes(M, N, K, G) bytes (may be NULL when
 *            that is 0).  Its contents need no initialisation.
 * Split-K calls enqueue two kernels (partial products into the workspace,
 * then a reduce that sums the slices in order 0..SPLIT_K-1 and rounds to
 * bf16); the result does not depend on timing.  Output rounding is
 * round-to-nearest-even. */
w4a16_status w4a16_gemm(const w4a16_bf16 *X, const uint8_t *W_packed, const w4a16_bf16 *scales,
                        w4a16_bf16 *Y, int M, int N, int K, int group_size, void *workspace,
                        size_t workspace_bytes, void *stream);

/* w4a16_gemm with overrides (`opts` may be NULL = automatic).  The workspace
 * requirement is the one w4a16_plan reports for the same opts. */
w4a16_status w4a16_gemm_ex(const w4a16_bf16 *X, const uint8_t *W_packed,
                           const w4a16_bf16 *scales, w4a16_bf16 *Y, int M, int N, int K,
                           int group_size, void *workspace, size_t workspace_bytes,
                           const w4a16_options *opts, void *stream);

/* Only the first launch of w4a16_gemm_ex: when the plan for (M, N, K, opts)
 * has SPLIT_K > 1 it writes the fp32 partial sums of every slice to
 * workspace as [SPLIT_K][M][N] (slice s covers K groups [s*P, s*P + P), P
 * from the plan) and leaves Y untouched; with one slice it writes Y exactly
 * as w4a16_gemm_ex does.  Following it with w4a16_splitk_reduce(workspace,
 * Y, SPLIT_K, M, N) gives the same bits as w4a16_gemm_ex.  Lets a caller
 * time or fuse the two launches separately.  *split_k_out (may be NULL)
 * receives SPLIT_K. */
w4a16_status w4a16_gemm_partials(const w4a16_bf16 *X, const uint8_t *W_packed,
                                 const w4a16_bf16 *scales, w4a16_bf16 *Y, int M, int N, int K,
                                 int group_size, void *workspace, size_t workspace_bytes,
                                 const w4a16_options *opts, int *split_k_out, void *stream);

/* Batched product ("Add Triton BF16xINT4 rowwise GEMM for ROCm gfx942/gfx950",
 * "bf16i4bf16_shuffled_batched": B independent products of one shape in one
 * launch): for b < batch, Y[b] = X[b] . dequant(W[b])^T.
 *  X:        device bf16 [batch][M][K].      Y: device bf16 [batch][M][N].
 *  W_packed: batch consecutive blocks, each w4a16_packed_weight_bytes(N, K).
 *  scales:   device bf16 [batch][N][K/G].
 *  workspace/workspace_bytes: at least the workspace_bytes w4a16_plan_batched
 *            reports (split-K partials [SPLIT_K][batch][M][N]; 0 without a
 *            split); contents need no initialisation.
 *  opts:     as for w4a16_gemm_ex (may be NULL).
 * The dispatcher plans the whole batch at once (the decode arm for M <= 16
 * with the CTA slots shared among the entries, else the tensor arm walking
 * every entry's tiles); each entry's result equals the product computed on its
 * own within the GEMM tolerance.  1 <= batch <= 1024, batch * M <= 2^24;
 * M == 0 launches nothing. */
w4a16_status w4a16_plan_batched(int batch, int M, int N, int K, int group_size,
                                const w4a16_options *opts, w4a16_plan_info *info);

/* Host-only planning for a device with `sms` streaming multiprocessors (152 on
 * GB300) instead of the current device: the plan w4a16_plan_batched (batch > 1)
 * or w4a16_plan (batch == 1) would make there.  sms == 0 queries the current
 * device.  Needs no GPU when sms > 0 (plan tables built ahead of time, tests).
 * 0 <= sms <= 4096, else W4A16_ERR_INVALID_ARG. */
w4a16_status w4a16_plan_for_sms(int sms, int batch, int M, int N, int K, int group_size,
                                const w4a16_options *opts, w4a16_plan_info *info);
w4a16_status w4a16_gemm_batched(const w4a16_bf16 *X, const uint8_t *W_packed,
                                const w4a16_bf16 *scales, w4a16_bf16 *Y, int batch, int M, int N,
                                int K, int group_size, void *workspace, size_t workspace_bytes,
                                const w4a16_options *opts, void *stream);

/* Zero-point variant: Y = X . dequant(W)^T with
 *   dequant(W)[n][k] = scale[n][k/G] * (code(n, k) - z[n][k/G]).
 * The pages describe only the symmetric form (z = 8); this is the usual int4
 * convention of a 4-bit integer zero point per row and scale group, a reading
 * for the asymmetric case.
 *  zeros:    device uint8 [N][K/G]; the low four bits of each byte are z
 *            (all z = 8 gives the symmetric result).
 *  Other arguments as for w4a16_gemm_ex; the workspace is what w4a16_plan
 *  reports with W4A16_FLAG_ZERO_POINTS in opts->flags.  The decode arm always
 *  uses its K-slice kernel.  w4a16_gemm_batched_zp and w4a16_gemm_grouped_zp
 *  below are the batched and grouped forms. */
w4a16_status w4a16_gemm_zp(const w4a16_bf16 *X, const uint8_t *W_packed, const w4a16_bf16 *scales,
                           const uint8_t *zeros, w4a16_bf16 *Y, int M, int N, int K,
                           int group_size, void *workspace, size_t workspace_bytes,
                           const w4a16_options *opts, void *stream);

/* Batched product with zero points (w4a16_gemm_batched with the dequant of
 * w4a16_gemm_zp): zeros is device uint8 [batch][N][K/G], entry b's block
 * following entry b - 1's as for the scales.  The workspace is what
 * w4a16_plan_batched reports with W4A16_FLAG_ZERO_POINTS in opts->flags. */
w4a16_status w4a16_gemm_batched_zp(const w4a16_bf16 *X, const uint8_t *W_packed,
                                   const w4a16_bf16 *scales, const uint8_t *zeros, w4a16_bf16 *Y,
                                   int batch, int M, int N, int K, int group_size, void *workspace,
                                   size_t workspace_bytes, const w4a16_options *opts,
                                   void *stream);

/* Workspace bytes of a grouped call: 16 bytes holding the device status word
 * (see w4a16_gemm_grouped).  Host only. */
w4a16_status w4a16_grouped_workspace_bytes(int num_groups, int M_total, int N, int K,
                                           int group_size, size_t *bytes);

/* Grouped product in one launch ("Add Triton BF16xINT4 ...", "Native fused
 * grouped kernel"): group g owns rows [start_g, start_g + M_sizes[g]) of X
 * and Y, start_g = sum of M_sizes[j] for j < g, and uses weight block g and
 * scale block g.
 *  X:         device bf16 [M_total][K].   Y: device bf16 [M_total][N].
 *  W_packed:  num_groups consecutive blocks, each w4a16_packed_weight_bytes(N, K).
 *  scales:    device bf16 [num_groups][N][K/G].
 *  M_sizes_dev: device int32 [num_groups]; read only by the kernel (the host
 *             never reads it, so the call needs no synchronisation).
 *  workspace: >= w4a16_grouped_workspace_bytes(...) bytes.  The kernel writes
 *             an int32 status word at workspace[0]: 0 = consistent; bit 0 =
 *             a negative size (treated as 0); bit 1 = the sizes sum past
 *             M_total (rows at or past M_total are not computed).  Rows no
 *             group covers are left unwritten.
 * 1 <= num_groups <= 1024. */
w4a16_status w4a16_gemm_grouped(const w4a16_bf16 *X, const uint8_t *W_packed,
                                const w4a16_bf16 *scales, const int32_t *M_sizes_dev,
                                w4a16_bf16 *Y, int num_groups, int M_total, int N, int K,
                                int group_size, void *workspace, size_t workspace_bytes,
                                void *stream);

/* Grouped product with zero points: w4a16_gemm_grouped with the dequant of
 * w4a16_gemm_zp; zeros is device uint8 [num_groups][N][K/G] (group g's block
 * after group g - 1's, as for the scales).  Same workspace and status word. */
w4a16_status w4a16_gemm_grouped_zp(const w4a16_bf16 *X, const uint8_t *W_packed,
                                   const w4a16_bf16 *scales, const uint8_t *zeros,
                                   const int32_t *M_sizes_dev, w4a16_bf16 *Y, int num_groups,
                                   int M_total, int N, int K, int group_size, void *workspace,
                                   size_t workspace_bytes, void *stream);

/* Dequantise a packed weight to fp32: out[n][k] = float(scale[n][k/G]) *
 * (code - 8), computed with the same in-register bit trick the GEMM arms use
 * (the code is OR-ed into the bf16 pattern of 128 + n and 136 is subtracted
 * exactly, "[ROCm][Kernel] W4A16 ...", section 1).  Exact: the product of an
 * 8-bit and a 4-bit significand fits binary32.  out: device fp32 [N][K]. */
w4a16_status w4a16_dequant_fp32(const uint8_t *W_packed, const w4a16_bf16 *scales, float *out,
                                int N, int K, int group_size, void *stream);

/* Dequantise to the bf16 operand the tensor arm feeds its MMAs:
 * out[n][k] = bf16_rne(scale[n][k/G] * (code - 8)).  out: device bf16 [N][K]. */
w4a16_status w4a16_dequant_bf16(const uint8_t *W_packed, const w4a16_bf16 *scales,
                                w4a16_bf16 *out, int N, int K, int group_size, void *stream);

/* The same two probes for the zero-point variant: scale * (code - z), z the
 * low four bits of zeros[n][k/G] (device uint8 [N][K/G]); fp32 exact, bf16
 * rounded once (the tensor arm's operand). */
w4a16_status w4a16_dequant_zp_fp32(const uint8_t *W_packed, const w4a16_bf16 *scales,
                                   const uint8_t *zeros, float *out, int N, int K, int group_size,
                                   void *stream);
w4a16_status w4a16_dequant_zp_bf16(const uint8_t *W_packed, const w4a16_bf16 *scales,
                                   const uint8_t *zeros, w4a16_bf16 *out, int N, int K,
                                   int group_size, void *stream);

/* The split-K reduce on its own: Y[i] = bf16_rne(sum over s = 0..splits-1 of
 * ws[s][i]) for i < M*N, slices summed in fp32 in ascending order ("Add Triton
 * BF16xINT4 ...", "Split-K without atomics").  ws: device fp32
 * [splits][M][N] (16-byte aligned); Y: device bf16 [M][N]. */
w4a16_status w4a16_splitk_reduce(const float *ws, w4a16_bf16 *Y, int splits, int M, int N,
                                 void *stream);

/* w4a16_gemm for callers that cannot allocate device memory on the GEMM's
 * path -- e.g. a framework plugin that receives only its inputs and outputs
 * while the framework keeps the rest of device memory for its own arena, or
 * code being captured into a CUDA graph, where cudaMalloc is not allowed.
 * The pages have no counterpart of this entry point; it is this library's own.
 * Arguments and result are those of w4a16_gemm minus the workspace: split-K
 * partial sums go to a 4 MiB scratch array inside the library image (a
 * file-scope __device__ array, held by every GPU that loads the library until
 * the process exits).  Nothing is allocated or freed.
 *  - Shapes whose plan needs more than 4 MiB of scratch (w4a16_workspace_bytes)
 *    return W4A16_ERR_WORKSPACE_TOO_SMALL and launch nothing.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture on the device.
 *  - All calls on a device share the one array and it keeps the last call's
 *    contents, so calls that may overlap on the GPU (different streams without
 *    ordering between them) race; order them on one stream or by events. */
w4a16_status w4a16_gemm_noalloc(const w4a16_bf16 *X, const uint8_t *W_packed,
                                const w4a16_bf16 *scales, w4a16_bf16 *Y, int M, int N, int K,
                                int group_size, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
