/*
 * blasst.h - C ABI of the GB300 (sm_103a) Skip-Softmax (BLASST) attention forward.
 *
 * The operation ("Skip-Softmax" design doc, vLLM-Omni, section "Algorithm";
 * "Skip-Softmax" on docs.vllm.ai, sections "The online-softmax pass" and
 * "The skip test"):
 *
 *   FlashAttention's single streaming pass over key tiles of 128. Per query row
 *   it keeps m (largest score so far), l = sum exp(s - m) and O = sum exp(s - m) v
 *   and returns O / l. For key tile j the scores S_j = Q . K_j^T . scale are
 *   always computed. If, for EVERY query row i of the 128-row query tile,
 *       tile_max[i] - running_max[i] < ln(lambda),
 *   the tile's exponentials, its l / O update and its P . V product are dropped.
 *   lambda = factor / Sk ("From configuration to the kernel threshold": the
 *   kernel takes threshold_scale_factor and divides it by the KV length).
 *   factor = 0 skips nothing and gives dense attention.
 *
 * Conventions for every entry point below:
 *   - Tensors are contiguous, row-major, [B, S, H, d] for q / k / v / o (token
 *     major, then head, then the d features), in bf16. lse is [B, H, Sq] fp32.
 *   - d must be 128.
 *   - All tensor pointers are DEVICE pointers on the current CUDA device, owned
 *     by the caller; the library keeps no reference after the call returns.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream) and
 *     return once the work is enqueued. No call allocates device memory.
 *   - Errors are reported by the return code only; nothing is enqueued when an
 *     argument is rejected. No C++ exception crosses this interface.
 */
#ifndef BLASST_H_
#define BLASST_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* a cudaStream_t is a `struct CUstream_st *` */

typedef enum blasst_status {
  BLASST_OK = 0,
  BLASST_ERR_INVALID_ARG = 1,        /* an argument is outside the documented domain */
  BLASST_ERR_UNSUPPORTED_DEVICE = 2, /* the current device is not compute capability 10.3 */
  BLASST_ERR_LAUNCH = 3,             /* the CUDA runtime refused a launch, copy or set-up step */
  BLASST_ERR_TIMEOUT = 4,            /* a device-side wait gave up (see blasst_device_error) */
  BLASST_ERR_TOO_LARGE = 5           /* the problem does not fit a fixed-size library buffer */
} blasst_status;

/*
 * Skip-Softmax attention forward.
 *
 *   q            [B, Sq, H, 128] bf16, 16-byte aligned.
 *   k, v         [B, Sk, H, 128] bf16, 16-byte aligned.
 *   o            [B, Sq, H, 128] bf16 output, 16-byte aligned: O / l over the kept tiles.
 *   lse          [B, H, Sq] fp32 output or NULL: m + ln(l) (natural log, scaled scores,
 *                kept tiles only).
 *   B, H         1 .. 65535.   Sq, Sk >= 1.   d == 128.
 *   scale        score scale, finite and > 0 (typically 1/sqrt(128)).
 *   factor       threshold_scale_factor, finite and >= 0; lambda = factor / Sk.
 *   stream       CUDA stream the work is enqueued on.
 *   skip_counts  [B * H] uint32 output or NULL: per (b, h), the number of
 *                (query tile, key tile) pairs that were skipped. Overwritten
 *                (zeroed on `stream`, then counted), never accumulated across calls.
 *   skip_mask_dbg [B, H, ceil(Sq/128), ceil(Sk/128)] uint8 output or NULL: 1 where the
 *                pair was skipped, 0 where it was computed. Every entry is written.
 *
 * Tiles are 128 query rows by 128 keys; key tiles are visited in ascending
 * order; query rows past Sq do not vote and are not stored; keys past Sk are
 * excluded from tile_max and from the softmax. The first key tile of every
 * query tile is always computed.
 *
 * Returns BLASST_OK once enqueued, BLASST_ERR_INVALID_ARG (nothing enqueued),
 * BLASST_ERR_UNSUPPORTED_DEVICE or BLASST_ERR_LAUNCH.
 */
blasst_status blasst_attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int H, int Sq, int Sk, int d, float scale, float factor,
                              struct CUstream_st *stream, uint32_t *skip_counts,
                              uint8_t *skip_mask_dbg);

/*
 * Extended call: every argument of blasst_attn_fwd plus
 *
 *   max_prob      [B, H, Sq] fp32 output or NULL (packed documents: [H, total_q]): per row
 *                 the largest softmax weight, exp(m - m) / l = 1 / l with l relative to the
 *                 row max m over the kept keys ("video-attention" blog, "max_prob = 1 / l_i,
 *                 and why it is free": a row-peakedness signal the pass already holds).
 *   packed documents (variable length): cu_seqlens_q and cu_seqlens_k, DEVICE arrays of
 *                 B + 1 int32 token offsets (non-decreasing, starting at 0), turn q / o into
 *                 [Sq, H, 128] and k / v into [Sk, H, 128] tensors of Sq / Sk tokens in all,
 *                 holding B documents; document b attends to its own keys only. lse and
 *                 max_prob become [H, Sq]. max_seqlen_q / max_seqlen_k are the longest
 *                 document lengths and max_seqlen_k is the KV length lambda is normalised by
 *                 (lambda = factor / max_seqlen_k for every document, the design doc's
 *                 max_kv_len, so that a threshold keeps its meaning in mixed batches).
 *                 skip_mask_dbg must be NULL; skip_counts is [B * H]. Offsets that are out of
 *                 order, out of the tensors or longer than the stated maxima are clamped and
 *                 raise an error bit that blasst_device_error reports.
 *   min_seq_len   documents (or batch entries) with fewer keys than this run dense (0 = off),
 *                 the per-document dense fallback of packed batches.
 *   qk_format     BLASST_QK_BF16 (0): q and k are bf16 as above. BLASST_QK_E4M3 (1): q and k
 *                 are FP8 e4m3 (OCP "e4m3fn": 1 sign, 4 exponent, 3 mantissa bits, no
 *                 infinities), one byte per element in the same layout, 16-byte aligned; the
 *                 score product Q . K^T runs on the FP8 tensor cores with fp32 accumulation while
 *                 v, P . V and o stay bf16. The scores are then S = (Q_e4m3 . K_e4m3^T) * scale *
 *                 q_descale * k_descale, with q_descale / k_descale (finite, > 0, read only in
 *                 this mode) the factors that undo the caller's per-tensor quantisation. The
 *                 "video-attention" blog (section "First, the hardware ceiling") notes that the
 *                 two products cost the same and only the score product tolerates the low
 *                 precision there; the score product is the part skipping never removes.
 *   status        DEVICE uint32 word or NULL, owned by the caller: zeroed on `stream` by the
 *                 call, then OR-ed with the error bits of every CTA whose bounded wait gave up
 *                 (1 producer, 2 MMA issuer, 4 softmax warps, 8 exit drain) or whose
 *                 packed-document offsets were invalid (16). A stream-ordered copy of it after the
 *                 call tells the caller whether o / lse are complete, without synchronizing the
 *                 device (blasst_device_error reports the same bits device-wide).
 *
 * struct_size must be sizeof(blasst_fwd_args); the size of the layout without `status` (the
 * offset of that member) is also accepted, with status taken as NULL. Same return codes as
 * blasst_attn_fwd.
 */
typedef struct blasst_fwd_args {
  uint32_t struct_size;
  const void *q, *k, *v;
  void *o;
  float *lse;
  float *max_prob;
  int B, H, Sq, Sk, d;
  float scale, factor;
  struct CUstream_st *stream;
  uint32_t *skip_counts;
  uint8_t *skip_mask_dbg;
  const int32_t *cu_seqlens_q, *cu_seqlens_k;
  int max_seqlen_q, max_seqlen_k;
  int min_seq_len;
  int qk_format;
  float q_descale, k_descale;
  uint32_t *status;
} blasst_fwd_args;

enum { BLASST_QK_BF16 = 0, BLASST_QK_E4M3 = 1 };

blasst_status blasst_attn_fwd_ex(const blasst_fwd_args *args);

/*
 * Host-buffer call: blasst_attn_fwd on fixed-length tensors that live in HOST memory. The heads
 * are streamed through a caller-provided device workspace in groups of heads_per_group: the
 * host-to-device copies of one group overlap the kernel on the previous group and the
 * device-to-host copies of the group before that; the kernels of consecutive groups run on
 * two streams, so one can start while the other finishes. (The attention of a head does not depend on
 * any other head, so the outputs equal those of blasst_attn_fwd bit for bit.)
 *
 *   q            HOST [B, Sq, H, 128] bf16.   k, v   HOST [B, Sk, H, 128] bf16.
 *   o            HOST [B, Sq, H, 128] bf16 output.   lse   HOST [B, H, Sq] fp32 output or NULL.
 *                Page-locked (pinned) host memory lets the copies overlap the kernels; pageable
 *                memory works but serialises them.
 *   workspace    DEVICE buffer, 256-byte aligned, of at least
 *                blasst_host_workspace_bytes(B, H, Sq, Sk, heads_per_group) bytes, owned by the
 *                caller; it must not be used by any other call until this one has completed.
 *   heads_per_group  1 .. H (H need not be a multiple of it): the largest group. Group sizes
 *                grow 1, 2, 3, 5, 8, ... (about 1.5 times the previous) up to it and the last
 *                group holds a single head, which shortens the pipeline's fill and drain.
 *   stream       the call starts after earlier work on `stream`, and work enqueued on `stream`
 *                afterwards starts after the last copy back: the host outputs are complete and the
 *                host inputs and the workspace free once `stream` reaches that point.
 *
 * The library owns four streams and seven events per device for this call, created at its first
 * use on the device; calls on one device are enqueued one at a time (a library mutex). No
 * device memory is allocated. Per-head skip counts and the skip mask are not available here.
 * Same argument rules and return codes as blasst_attn_fwd; struct_size must be
 * sizeof(blasst_host_args).
 */
typedef struct blasst_host_args {
  uint32_t struct_size;
  const void *q, *k, *v;
  void *o;
  float *lse;
  int B, H, Sq, Sk, d;
  float scale, factor;
  void *workspace;
  size_t workspace_bytes;
  int heads_per_group;
  struct CUstream_st *stream;
} blasst_host_args;

/* Device workspace the host-buffer call needs (two groups of q, k, v, o and lse), or 0 when an
 * argument is outside its domain. */
size_t blasst_host_workspace_bytes(int B, int H, int Sq, int Sk, int heads_per_group);

blasst_status blasst_attn_fwd_host(const blasst_host_args *args);

/*
 * Host-buffer call that allocates nothing. It has no counterpart in the method or on the pages
 * that describe it: it exists for callers that cannot call cudaMalloc. Examples are a plug-in
 * loaded into a host application that keeps all of the GPU's memory in its own pool and hands
 * out no raw device buffers, and a latency-critical loop that must not call cudaMalloc or
 * cudaFree, which can synchronize the whole device.
 *
 * The call is blasst_attn_fwd_host with its device workspace taken from a buffer of
 * BLASST_NOALLOC_SCRATCH_BYTES bytes that the library itself holds: a fixed-size __device__
 * array. The CUDA runtime reserves it on a device when it loads the library's code there and
 * releases it only when the process exits. With lazy module loading (the CUDA default) that
 * happens at this entry point's first call on the device; with eager loading, when the context
 * is created.
 *
 *   args   as for blasst_attn_fwd_host, except that workspace must be NULL and workspace_bytes
 *          0. heads_per_group (1 .. H) is the largest head group wanted: the call lowers it to
 *          the largest group whose two workspace slots fit the buffer.
 *
 * The call returns BLASST_ERR_TOO_LARGE, with nothing enqueued, when even a group of one head
 * does not fit, that is when blasst_host_workspace_bytes(B, H, Sq, Sk, 1) exceeds
 * BLASST_NOALLOC_SCRATCH_BYTES. Otherwise it returns what blasst_attn_fwd_host returns. It
 * never calls cudaMalloc, cudaFree or any library routine that allocates device memory.
 *
 * Set-up: the first call on a device, made with that device current, looks up the buffer's
 * device address there (cudaGetSymbolAddress). That lookup loads the library's code on the
 * device if it is not loaded yet. Make that first call before any stream capture begins.
 *
 * Sharing: every call on a device uses the same buffer, and the buffer keeps the last call's
 * contents. Each call writes every byte of the buffer it reads before reading it (its copies of
 * q, k and v; the kernel writes all of o and lse), so nothing needs clearing between calls.
 * Calls whose GPU work overlaps race on the buffer. A call starts after earlier work on its
 * `stream`, so calls on one stream are safe. Calls on different streams, or from different
 * threads, must be ordered by the caller.
 */
#define BLASST_NOALLOC_SCRATCH_BYTES ((size_t)256 << 20)
blasst_status blasst_attn_fwd_host_noalloc(const blasst_host_args *args);

/* A static, human-readable name for a status code. */
const char *blasst_status_string(blasst_status s);

/*
 * Reads the device-side error word of the current device, which a kernel sets
 * when one of its bounded waits gives up (every wait in the kernel is limited
 * in time; a kernel that gives up writes no further output and returns).
 * Synchronizes the device. *word receives 0 when no wait gave up since the
 * last clear; `clear` != 0 resets the word afterwards.
 * Returns BLASST_OK, BLASST_ERR_TIMEOUT (word != 0), BLASST_ERR_INVALID_ARG
 * (word == NULL) or BLASST_ERR_LAUNCH.
 */
blasst_status blasst_device_error(uint32_t *word, int clear);

/*
 * Host-side controls (no CUDA call). They turn user settings into the factor the kernel
 * takes, following the "Skip-Softmax" design doc (vLLM-Omni), sections "From
 * configuration to the kernel threshold", "Timestep gating" and "Mapping the cutoff to
 * denoising steps". Every output pointer is a host pointer owned by the caller; on
 * BLASST_ERR_INVALID_ARG nothing is written.
 */

/* Direct control: *factor = threshold * max_kv_len, so lambda = factor / max_kv_len is the
 * threshold itself at any sequence length. threshold finite and >= 0; max_kv_len >= 1. */
blasst_status blasst_factor_from_threshold(double threshold, int64_t max_kv_len, double *factor);

/* Calibrated control: *factor = a * exp(b * target_sparsity), a point on the curve fitted per
 * model. Rejected unless the result is finite and >= 0. */
blasst_status blasst_factor_from_target_sparsity(double a, double b, double target_sparsity,
                                                 double *factor);

/* Timestep gate for one attention call. disabled_until_timestep == 0 switches the gate off
 * (t is not read; *out = factor). Otherwise *out = 0 (dense) while t > disabled_until_timestep,
 * and also when t_published == 0, in which case *warn = 1 so that the caller can log once;
 * once t <= disabled_until_timestep, *out = factor. warn may be NULL. factor and
 * disabled_until_timestep finite and >= 0; t finite when published. */
blasst_status blasst_gate_factor(double factor, double disabled_until_timestep, int t_published,
                                 double t, double *out, int *warn);

/* *dense_steps = count(t[i] > disabled_until_timestep) for i < n (t: host array of n values). */
blasst_status blasst_dense_steps(const double *t, int n, double disabled_until_timestep,
                                 int *dense_steps);

/* Flow-shifted rectified-flow schedule: t_out[i] = s u / (1 + (s - 1) u) at the num_points
 * uniform positions u = 1 - i / (num_points - 1) (from 1 down to 0). shift > 0,
 * num_points >= 2; t_out holds num_points values. */
blasst_status blasst_flow_shift_schedule(double shift, int num_points, double *t_out);

/* Library version as major * 10000 + minor * 100 + patch. */
int blasst_version(void);

/*
 * Test hook for the bounded device waits (no counterpart in the method): from the next call
 * on, in every process-wide kernel launch, the TMA producer never issues the copy of key tile
 * `tile`, so the waits on it run out after their time limit, the CTAs leave through their
 * abort path and the error bits show in `status` and blasst_device_error. -1 (the initial
 * state) switches it off. Returns BLASST_ERR_INVALID_ARG for tile < -1.
 */
blasst_status blasst_debug_withhold_key_tile(int tile);

/*
 * Number of TMA tensor descriptors this process has encoded so far. Each call needs one for
 * q, k and v; they are kept in a small per-process cache keyed by (address, shape, format),
 * so repeated calls on the same tensors encode none.
 */
uint64_t blasst_tensor_map_encodes(void);

#ifdef __cplusplus
}
#endif

#endif /* BLASST_H_ */
