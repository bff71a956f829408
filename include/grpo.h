/*
 * libgrpo -- fused memory-efficient ("linear") GRPO loss for one NVIDIA GB300
 * (sm_103a).  C ABI: plain pointers and sizes, no framework types.
 *
 * The operation ("Long-context GRPO", sections 2-4; "Train your own R1
 * reasoning model with Unsloth", section 3):
 *
 *   For every completion token t (row t of the hidden-state matrices),
 *     z_pol = h_pol[t] . W^T      z_ref = h_ref[t] . W^T      (V logits each)
 *     q_t = z_pol[tok_t] - logsumexp(z_pol)    policy log-prob of the sampled token
 *     p_t = z_ref[tok_t] - logsumexp(z_ref)    frozen-reference log-prob
 *     ell_t = -[ exp(q_t - sg(q_t)) * A_i - beta * (exp(p_t-q_t) - (p_t-q_t) - 1) ]
 *   with A_i the group-relative advantage of the completion (sequence) i that
 *   row t belongs to, and the loss is the mean of ell_t over masked rows.
 *   The backward gives dH = d loss / d h_pol and dW = d loss / d W through the
 *   policy logits (the reference is a frozen constant).
 *
 *   The (rows x V) logits are never stored: extra device memory is
 *   O(chunk_rows * V + rows), never O(rows * V).
 *
 * Conventions shared by every entry point
 *   - All data pointers are caller-owned DEVICE memory; the library never
 *     allocates or frees device memory and keeps no pointer after a call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; 0 = legacy default
 *     stream).  The return value reports argument validation and launch
 *     errors only; errors found while the kernels run are written to the
 *     caller's device word `status` (same codes), which the call resets to 0
 *     before its first kernel.
 *   - Matrices are row-major.  h_pol, h_ref: [N x d]; W: [V x d] (the layout of
 *     an nn.Linear weight), element type given by grpo_shape.dtype.  Every
 *     matrix base pointer must be 16-byte aligned (the kernels read them with
 *     the tensor memory accelerator).
 *   - Row t = i*L + j is position j of completion i; completion i belongs to
 *     prompt group i / G.  N = n_groups * G * L.
 *   - All hidden-state rows, masked or not, must hold finite values.
 *   - Several host threads may call the entry points at once, each call with
 *     its own workspace and outputs.  grpo_loss_fwd_noalloc is the exception
 *     (its calls share one array; see there).
 *   - Nothing throws, aborts or exits the process.
 */
#ifndef GRPO_H
#define GRPO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes (return values and the device `status` word) */
enum {
    GRPO_OK = 0,
    GRPO_ERR_POINTER = 1,    /* null or misaligned pointer */
    GRPO_ERR_SHAPE = 2,      /* bad shape or a token id outside [0, V) */
    GRPO_ERR_WORKSPACE = 3,  /* workspace smaller than grpo_workspace_bytes() */
    GRPO_ERR_LAUNCH = 4,     /* a CUDA launch or driver call failed */
    GRPO_ERR_DTYPE = 5,      /* dtype not supported */
    GRPO_ERR_TIMEOUT = 6,    /* a device-side wait ran out of time (kernel gave up, no hang) */
    GRPO_ERR_DEVICE = 7,     /* device is not sm_103 / lacks the needed shared memory */
    GRPO_ERR_BOUNDS = 8      /* a device-side index check failed; only the checked build
                                (libgrpo_checked.so, see grpo_device_checks) makes them */
};

typedef enum { GRPO_BF16 = 0, GRPO_FP16 = 1, GRPO_E4M3 = 2, GRPO_E5M2 = 3 } grpo_dtype;

typedef struct CUstream_st* grpo_stream_t;   /* the same type as cudaStream_t */

/* Problem description.
 *   n_groups, G : prompts and completions per prompt (G >= 1)
 *   L           : rows per completion (max completion length)
 *   d           : hidden size, a multiple of 64
 *   V           : vocabulary size (>= 1)
 *   dtype       : storage/compute type of h_pol, h_ref, W (and of dH);
 *                 GRPO_E4M3 / GRPO_E5M2 only with grpo_loss_fwd_fp8
 *   beta        : KL coefficient (0.04 in the pages' setting)
 *   eps         : added to the group std in grpo_group_advantages
 *   std_unbiased: 1 -> group std with divisor G-1, 0 -> divisor G
 *   chunk_rows  : masked rows processed per backward chunk, rounded up to a
 *                 multiple of 128 and capped at N.  0 picks the default: 38
 *                 tiles of 128 rows (4864) when its dH work divides evenly
 *                 over the 76 SM pairs (d/256 a multiple of 4, e.g. d = 4096
 *                 or 5120), else 76 tiles (9728); 76 tiles for 8-bit shapes.
 *                 grpo_chunk_rows tells.
 *   loss_mode   : GRPO_TOKEN_MEAN -- mean of ell_t over all masked rows;
 *                 GRPO_SEQUENCE_MEAN -- mean over completions (with at least
 *                 one masked row) of each completion's mean over its rows
 *   objective   : the per-token objective ("Long-context GRPO", section 4:
 *                 the four-way experiment; the pages' formula images are
 *                 lost, so each variant is the reading stated here), with
 *                 x = p_t - q_t and ell_t = -A + beta * pen_t:
 *                 GRPO_OBJ_GRPO        detached exp(q - sg(q)) * A, pen = e^x - x - 1
 *                 GRPO_OBJ_NO_DETACH   same value, but exp(q - q) carries no
 *                                      gradient: d ell/d q = beta (1 - e^x)
 *                 GRPO_OBJ_REVERSE_KL_Q  pen = e^q (e^x - x - 1): the penalty
 *                                      multiplied by the token's policy probability
 *                 GRPO_OBJ_FORWARD_KL  pen = e^-x + x - 1 */
typedef struct {
    int n_groups, G, L, d, V;
    grpo_dtype dtype;
    float beta;
    float eps;
    int std_unbiased;
    int chunk_rows;
    int loss_mode;
    int objective;
} grpo_shape;

enum { GRPO_TOKEN_MEAN = 0, GRPO_SEQUENCE_MEAN = 1 };
enum { GRPO_OBJ_GRPO = 0, GRPO_OBJ_NO_DETACH = 1, GRPO_OBJ_REVERSE_KL_Q = 2, GRPO_OBJ_FORWARD_KL = 3 };

/* Fills a grpo_shape with the pages' defaults (beta 0.04, eps 1e-4, unbiased
 * std, token mean, the GRPO objective). */
void grpo_shape_init(grpo_shape* s, int n_groups, int G, int L, int d, int V, grpo_dtype dtype);

/* Bytes of device workspace grpo_loss_fwd / grpo_loss_fwd_bwd need for this
 * shape: O(chunk_rows * (V + d) + N), independent of how many rows are
 * masked.  Returns 0 for an invalid shape. */
size_t grpo_workspace_bytes(const grpo_shape* shape);

/* Rows per backward chunk that grpo_loss_fwd / grpo_loss_fwd_bwd use for this
 * shape (the chunk_rows field resolved as described above).  Returns 0 for
 * an invalid shape.  The pages have no counterpart: it is this library's
 * memory/throughput knob. */
int grpo_chunk_rows(const grpo_shape* shape);

/* Group-relative advantages ("Train your own R1 reasoning model with
 * Unsloth", section 3, steps 3-5: score each response, take the group mean,
 * compare every score with it).
 *   rewards [n_groups*G] fp32 (device, read)    adv_out [n_groups*G] fp32 (device, written)
 *   adv = (r - mean_group(r)) / (std_group(r) + eps), computed in fp64 with a
 *   fixed summation order and rounded once to fp32 (bit-reproducible).
 *   A group whose std divisor is 0 (G == 1 with std_unbiased) has std 0. */
int grpo_group_advantages(const float* rewards, int n_groups, int G, float eps, int std_unbiased,
                          float* adv_out, grpo_stream_t stream);

/* Completion mask from completion lengths: mask[i*L + j] = (j < lengths[i]).
 *   lengths [n_groups*G] int32 (device)   mask_out [N] uint8 (device, written) */
int grpo_build_mask(const int32_t* lengths, const grpo_shape* shape, uint8_t* mask_out,
                    grpo_stream_t stream);

/* Indices of the masked-in rows in ascending order and their count.
 *   mask [N] uint8 (device)   rows_out [N] int32 (device; first *n_valid entries written)
 *   n_valid_out: one int32 (device).  workspace as for grpo_loss_fwd. */
int grpo_valid_rows(const uint8_t* mask, const grpo_shape* shape, int32_t* rows_out,
                    int32_t* n_valid_out, void* workspace, size_t ws_bytes, grpo_stream_t stream);

/* Forward pass of the linear GRPO loss ("Long-context GRPO", section 2: the
 * memory-efficient linear algorithm; section 4: the objective, the detach
 * factor and the logsumexp trick).  Runs the same chunked kernels as
 * grpo_loss_fwd_bwd, without the backward.
 *   h_pol, h_ref [N x d], W [V x d]          (dtype; device, read)
 *   tokens [N] int32 in [0, V)               (device, read; masked rows too)
 *   mask [N] uint8, nonzero = completion token (device, read)
 *   adv [n_groups*G] fp32, one per completion (device, read)
 *   workspace: >= grpo_workspace_bytes(shape) bytes of device memory, 256-byte aligned
 *   loss_out: one fp32 (device) <- the mean of ell_t chosen by loss_mode (0 if
 *             no row is masked in)
 *   row_stats: NULL or [N x 5] fp32 (device) <- (lse_pol, lse_ref, q, p, pen)
 *              per row; zeros on masked rows
 *   status: one int32 (device) <- 0 or an error code
 * The result is bitwise reproducible from run to run. */
int grpo_loss_fwd(const void* h_pol, const void* h_ref, const void* W, const int32_t* tokens,
                  const uint8_t* mask, const float* adv, const grpo_shape* shape,
                  void* workspace, size_t ws_bytes, float* loss_out, float* row_stats,
                  int32_t* status, grpo_stream_t stream);

/* Forward and backward.  Same inputs and outputs as grpo_loss_fwd, plus
 *   loss_scale: gradients are multiplied by it (1 for bf16; the fp16 loss
 *               scale otherwise -- "Long-context GRPO", section 3: mixed
 *               precision with automatic loss scaling breaks a naive linear
 *               cross entropy unless handled)
 *   dH [N x d] (dtype; device, written, 32-byte aligned): loss_scale *
 *               d loss / d h_pol; exactly 0 on masked rows
 *   dW [V x d] fp32 (device, overwritten, 32-byte aligned): loss_scale *
 *               d loss / d W
 *   (the gradient epilogues write whole 32-byte sectors; a dH or dW that is
 *   only 16-byte aligned is refused with GRPO_ERR_POINTER)
 *   found_inf: one int32 (device) <- 1 if any scaled gradient value (the
 *               16-bit dlogits, dH or dW) is not finite, else 0.  The caller
 *               lowers the scale and calls again when it is set.
 * The loss and row_stats equal grpo_loss_fwd's bit for bit; every output is
 * bitwise reproducible from run to run (fixed reduction orders, no
 * floating-point atomics). */
int grpo_loss_fwd_bwd(const void* h_pol, const void* h_ref, const void* W, const int32_t* tokens,
                      const uint8_t* mask, const float* adv, const grpo_shape* shape,
                      float loss_scale, void* workspace, size_t ws_bytes, float* loss_out,
                      void* dH, float* dW, int32_t* found_inf, float* row_stats,
                      int32_t* status, grpo_stream_t stream);

/* ---- data-parallel shards ---------------------------------------------
 * A batch of prompt groups split over several GPUs, each holding W and whole
 * prompt groups (so advantages need no exchange).  The loss is still the
 * mean over the completion tokens of the WHOLE batch ("Long-context GRPO",
 * section 4: the objective averaged over completion tokens); the pages
 * describe one GPU, so the split itself is this library's.  Protocol:
 *   1. each shard: grpo_shard_counts(mask) -> its two counts (device);
 *   2. the caller sums the counts over the shards (e.g. an all-reduce);
 *   3. each shard: grpo_loss_fwd_bwd_shard(..., global_counts, ...);
 *   4. the caller sums loss_out and dW over the shards.
 * Every shard's weights use the global counts, so the summed loss and dW equal
 * a one-GPU call on the whole batch up to rounding, and each shard's dH rows
 * are exactly the whole batch's dH rows.
 *
 * grpo_shard_counts: counts_out [2] int32 (device, written) <- (masked-in
 * rows, completions with at least one masked-in row) of this shard's mask
 * [n_groups*G*L] uint8 (device).  Asynchronous on `stream`. */
int grpo_shard_counts(const uint8_t* mask, const grpo_shape* shape, int32_t* counts_out, grpo_stream_t stream);

/* One shard's forward (+ backward): the arguments of grpo_loss_fwd /
 * grpo_loss_fwd_bwd for this shard's rows (shape describes the shard:
 * n_groups is its own group count), plus
 *   global_counts [2] int32 (device, read): the sums over all shards of
 *     grpo_shard_counts, i.e. (N_v of the batch, active completions of the batch)
 * and with these meanings of the outputs:
 *   loss_out: this shard's share of the batch loss, i.e. the sum of its rows'
 *     weighted objectives divided by the batch's divisor; the shares add up
 *     to the batch loss
 *   dW: this shard's share of the batch gradient (sum over shards = dW)
 *   dH: the batch gradient of this shard's rows (no sum needed)
 * Global counts below this shard's own counts set *status to GRPO_ERR_SHAPE.
 * Workspace, alignment and every other rule are those of grpo_loss_fwd_bwd. */
int grpo_loss_fwd_shard(const void* h_pol, const void* h_ref, const void* W, const int32_t* tokens,
                        const uint8_t* mask, const float* adv, const grpo_shape* shape,
                        const int32_t* global_counts, void* workspace, size_t ws_bytes, float* loss_out,
                        float* row_stats, int32_t* status, grpo_stream_t stream);
int grpo_loss_fwd_bwd_shard(const void* h_pol, const void* h_ref, const void* W, const int32_t* tokens,
                            const uint8_t* mask, const float* adv, const grpo_shape* shape,
                            const int32_t* global_counts, float loss_scale, void* workspace, size_t ws_bytes,
                            float* loss_out, void* dH, float* dW, int32_t* found_inf, float* row_stats,
                            int32_t* status, grpo_stream_t stream);

/* Forward pass on 8-bit inputs ("Long-context GRPO", section 3: linear cross
 * entropy under float8 mixed precision).  h_pol, h_ref and W hold OCP FP8
 * codes of one format, shape->dtype: GRPO_E4M3 (4 exponent bits, 3 mantissa
 * bits) or GRPO_E5M2 (5 and 2), one byte per element, same row-major layouts;
 * element values are code * scale with one scale per tensor (scale_h_pol,
 * scale_h_ref, scale_w > 0).  The logits come from 8-bit tensor-core products
 * accumulated in fp32 and multiplied by scale_h * scale_w; everything after
 * that is as in grpo_loss_fwd.  d must be a multiple of 128; the workspace is
 * grpo_workspace_bytes(shape) (for an 8-bit shape it includes the buffers of
 * grpo_loss_fwd_bwd_fp8, which this call leaves unused). */
int grpo_loss_fwd_fp8(const void* h_pol, const void* h_ref, const void* W, float scale_h_pol, float scale_h_ref,
                      float scale_w, const int32_t* tokens, const uint8_t* mask, const float* adv,
                      const grpo_shape* shape, void* workspace, size_t ws_bytes, float* loss_out, float* row_stats,
                      int32_t* status, grpo_stream_t stream);

/* Forward and backward on 8-bit inputs ("Long-context GRPO", section 3: a
 * linear cross entropy under float8 mixed precision with automatic scaling
 * breaks unless the scaling is handled).  Inputs as grpo_loss_fwd_fp8; the
 * outputs as grpo_loss_fwd_bwd without loss scaling:
 *   dH [N x d] bf16 (device, written, 32-byte aligned): d loss / d h_pol,
 *      exactly 0 on masked rows
 *   dW [V x d] fp32 (device, overwritten, 32-byte aligned): d loss / d W
 * (gradients with respect to the decoded values code * scale).  Both backward
 * GEMMs run on 8-bit codes.  The dlogits g (onehot(tok) - softmax) are split:
 * the one-hot part, which holds the largest entry of every row, is added
 * exactly in the GEMM epilogues from the decoded inputs; only the softmax part
 * g * softmax goes through 8-bit codes of the input format, with one scale per
 * dlogit row for dH and one per 32 vocabulary rows for dW (scales along the
 * GEMMs' M dimension, so no K-block scales are needed).  Chunks hold at most
 * 16384 rows (larger chunk_rows give GRPO_ERR_SHAPE).  The workspace is
 * grpo_workspace_bytes(shape) for the 8-bit shape. */
int grpo_loss_fwd_bwd_fp8(const void* h_pol, const void* h_ref, const void* W, float scale_h_pol, float scale_h_ref,
                          float scale_w, const int32_t* tokens, const uint8_t* mask, const float* adv,
                          const grpo_shape* shape, void* workspace, size_t ws_bytes, float* loss_out, void* dH,
                          float* dW, float* row_stats, int32_t* status, grpo_stream_t stream);

/* Forward loss for callers that cannot allocate device memory -- for
 * instance a training step that shares the GPU with an inference engine
 * which has already reserved all free memory for its own pool, or code that
 * cannot afford cudaMalloc's device-wide synchronisation inside its step.
 * The pages have no counterpart of this entry point; it is a property of
 * this library, not of the method.
 *
 * Same inputs and outputs as grpo_loss_fwd, without the workspace: the
 * library uses an 8 MiB array of its own, held on every GPU that loads the
 * library until the process exits.  It allocates nothing and calls no
 * allocating routine.  It runs all rows at once on single-SM kernels, so its
 * results equal grpo_loss_fwd's up to fp32 rounding (the vocabulary is split
 * differently).
 *   Limit: N = n_groups*G*L <= 32768 rows; larger shapes are rejected with
 *   GRPO_ERR_WORKSPACE before anything is launched.
 *   The first call on a device looks up the array's device address (a
 *   synchronous runtime call).  Under lazy module loading (the CUDA default)
 *   that first call is also when the CUDA driver loads this library's device code
 *   and places the array in device memory, so make it before the device's
 *   free memory is handed to anything else (an inference engine's pool), and
 *   before any stream capture; later calls need no new memory.
 *   Every call uses the same array, so calls that can overlap on the GPU
 *   (other streams, other host threads) race; serialise them.  Nothing
 *   carries over between calls: each call writes every word it reads. */
int grpo_loss_fwd_noalloc(const void* h_pol, const void* h_ref, const void* W, const int32_t* tokens,
                          const uint8_t* mask, const float* adv, const grpo_shape* shape,
                          float* loss_out, float* row_stats, int32_t* status, grpo_stream_t stream);

/* ---- diagnostics ------------------------------------------------------
 * Per-kernel device time.  While enabled, the library records a CUDA event
 * pair on the launching stream around every kernel it launches.
 * grpo_profile_collect waits for the recorded events, adds the elapsed
 * milliseconds of each kernel kind into ms[kind] and the launch count into
 * launches[kind] (arrays of at least GRPO_PROF_KINDS entries, caller-owned
 * host memory), and clears the records.  Meant for benchmarks: the
 * records of every thread's launches go into one list, and while profiling
 * is on, launches from different threads take turns on a lock.
 * grpo_kernel_launches counts every kernel launched by the library since it
 * was loaded, profiling on or off. */
enum {
    GRPO_PROF_ADVANTAGES = 0,
    GRPO_PROF_MASK,
    GRPO_PROF_INDEX,
    GRPO_PROF_FWD,
    GRPO_PROF_MERGE,
    GRPO_PROF_CLEAR,
    GRPO_PROF_GATHER,
    GRPO_PROF_DLOGITS,
    GRPO_PROF_DH,
    GRPO_PROF_DW,
    GRPO_PROF_F8_PREP,   /* the 8-bit backward's group bounds and token sort */
    GRPO_PROF_KINDS
};
int grpo_profile_enable(int on);
int grpo_profile_collect(double* ms, long long* launches, int n_kinds);
unsigned long long grpo_kernel_launches(void);

/* Device-side index checks.  The library is also built as
 * libgrpo_checked.so, whose kernels check every global index they take from
 * device data (the valid-row list) and the offset arithmetic of the chunk
 * buffers: a failing check skips the access and sets *status to
 * GRPO_ERR_BOUNDS.  It stands in for a memory checker; the pages have no
 * counterpart.  grpo_device_checks() returns 1 in that build, 0 in the normal
 * one.  grpo_selftest_bounds_check makes one such check fail on purpose (a
 * guarded store one past a 16-element shared array, refused by the check):
 * *status (device int32) then reads GRPO_ERR_BOUNDS.  In the normal build it
 * launches nothing and returns GRPO_ERR_DEVICE. */
int grpo_device_checks(void);
int grpo_selftest_bounds_check(int32_t* status, grpo_stream_t stream);

/* Self-test of the bounded device waits: one CTA waits, with the wait the
 * kernels use, on an mbarrier that nothing completes.  It gives up after about
 * a second and writes GRPO_ERR_TIMEOUT to *status (device int32, set to 0 by
 * the caller beforehand) and the nanoseconds it waited to *waited_ns (device
 * uint64).  The context stays usable.  The pages have no counterpart; it
 * checks the library's own guarantee that no kernel waits forever. */
int grpo_selftest_wait_timeout(int32_t* status, unsigned long long* waited_ns, grpo_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* grpo_status_string(int status);

/* Library version, as major*10000 + minor*100 + patch. */
int grpo_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GRPO_H */
