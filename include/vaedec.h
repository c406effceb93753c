/*
 * vaedec -- layerwise height-row-band VAE decode on one GPU (sm_103a).
 *
 * What it computes.  A diffusion VAE decoder (an AutoencoderKL-style 2D CNN or a
 * WanDecoder3d-style causal 3D CNN) run layer by layer over height row bands, as
 * ChituDiffusion's pages "VAEP：VAE 并行解码" (section 按高度分片，逐层解码) and
 * "Static Layer-Wise VAE Decode" (table "Semantics and Communication") define it:
 *   - the latent height is cut into disjoint row bands; uneven bands keep their
 *     lengths, and every 2x upsample doubles each band's rows;
 *   - every conv reads kernel-radius halo rows of the neighbouring band, with zero
 *     padding only at the global image edges (section 卷积：交换边界行);
 *   - GroupNorm merges per-part central moments with the element-count-weighted
 *     rule mean = sum w_i mean_i, var = sum w_i (var_i + (mean_i - mean)^2), in
 *     fp32 (section GroupNorm：合并全局统计量);
 *   - mid-block attention keeps Q band-local and attends over all K/V
 *     (section Attention：本地 Q，全局 K/V);
 *   - SiLU, channel RMSNorm and nearest-2x upsample are local.
 * On one GPU every band lives in the same device memory: halo rows are read in
 * place, statistics are merged by a kernel, K/V are already resident.  The result
 * equals the unbanded decode, and on this library it is bit-identical for every
 * band count.
 *
 * Threading and streams.  A handle may be used from one host thread at a time.
 * Calls are stream-ordered and asynchronous unless stated otherwise.  Two decodes
 * on one handle must be ordered on the same stream (they share the handle's
 * workspace).
 *
 * Errors.  Every entry point returns a vaedec_status; the message of the calling
 * thread's last failure is available from vaedec_last_error().  Kernel-side
 * failures (a bounded wait that ran out) are recorded in a device status word and
 * reported by vaedec_sync() or the next synchronous call.
 */
#ifndef VAEDEC_H_
#define VAEDEC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define VAEDEC_ABI_VERSION 2
#define VAEDEC_MAX_STAGES 6

typedef struct vaedec vaedec_t; /* opaque: device weights + workspace */

typedef enum {
  VAEDEC_OK = 0,
  VAEDEC_ERR_INVALID_ARG = 1, /* bad shape, dtype, band count, pointer, size */
  VAEDEC_ERR_UNSUPPORTED = 2, /* geometry outside the method's scope (see below) */
  VAEDEC_ERR_OOM = 3,         /* device allocation failed */
  VAEDEC_ERR_CUDA = 4,        /* a CUDA call failed (message holds the CUDA error) */
  VAEDEC_ERR_TIMEOUT = 5,     /* a kernel's bounded wait ran out (device status word) */
  VAEDEC_ERR_STOPPED = 6      /* debug run stopped at the requested op (not a failure) */
} vaedec_status;

enum { VAEDEC_FAMILY_KL2D = 1, VAEDEC_FAMILY_WAN3D = 2 };
enum { VAEDEC_DTYPE_F32 = 1, VAEDEC_DTYPE_BF16 = 2 };
enum { VAEDEC_UP_NONE = 0, VAEDEC_UP_SPATIAL = 1, VAEDEC_UP_SPATIOTEMPORAL = 2 };

/* A named HOST tensor, contiguous row-major, read only during vaedec_create. */
typedef struct {
  const char* name;   /* Diffusers state-dict key, e.g. "mid_block.resnets.0.conv1.weight" */
  const void* data;   /* host pointer */
  int dtype;          /* VAEDEC_DTYPE_F32 or VAEDEC_DTYPE_BF16 */
  int ndim;
  int64_t shape[5];
} vaedec_tensor;

/*
 * Decoder description.  conv_in maps latent_channels -> mid_channels; the mid block
 * is [resnet, attention, resnet] at mid_channels; stage s runs stage_resnets[s]
 * residual blocks to stage_channels[s] channels, then an optional upsample whose
 * 3x3 conv maps to stage_up_channels[s]; a final norm, SiLU and 3x3 conv_out map to
 * out_channels.  KL2D uses GroupNorm(norm_groups, eps); WAN3D uses channel RMSNorm
 * and causal 3x3x3 convs.
 * max_latent = {B, T, H, W} upper bounds (T = 1 for KL2D): the workspace is sized
 * for them once at create time.
 */
typedef struct {
  int family;
  int dtype; /* bf16: tensor-core path; f32: CUDA-core fp32 path (checks only) */
  int latent_channels, mid_channels, out_channels;
  int n_stages;
  int stage_channels[VAEDEC_MAX_STAGES];
  int stage_resnets[VAEDEC_MAX_STAGES];
  int stage_upsample[VAEDEC_MAX_STAGES]; /* VAEDEC_UP_* */
  int stage_up_channels[VAEDEC_MAX_STAGES];
  int norm_groups;
  float eps;
  int64_t max_latent[4];
  /* AutoencoderKLFlux2 latent front-end ("VAEP：VAE 并行解码", 不同模型如何复用: keep the latent
   * BatchNorm and patch conversion), KL2D only.  latent_patch 0 or 1: none.  latent_patch 2: the
   * decode input is the transformer-side latent, 4 * latent_channels channels on an (H, W) grid
   * normalised by an inference BatchNorm without affine terms (weights "bn.running_mean" and
   * "bn.running_var", 4 * latent_channels values each, eps latent_bn_eps); the decode first computes
   * x * sqrt(var + eps) + mean per channel and unpatchifies channel c*4 + py*2 + px to pixel
   * (2y + py, 2x + px) of channel c, then runs the decoder on the (2H, 2W) grid.  Latent shapes,
   * max_latent and output shapes are in the input's (H, W) units; bands split the (2H, 2W) grid. */
  int latent_patch;
  float latent_bn_eps;
} vaedec_config;

/*
 * Create a decoder on the current CUDA device.  Every later call that launches work or reads the
 * handle's device memory (decode, decode_bands, decode_host, sync, profile_read, the debug runs)
 * must be made with that device current; otherwise it returns VAEDEC_ERR_INVALID_ARG and launches
 * nothing.  vaedec_destroy switches to the handle's device to free it and restores the caller's.  Copies and repacks every weight
 * (host memory, any of the two dtypes) into device layouts owned by the handle and
 * allocates the workspace for config->max_latent.  Synchronous.
 * Errors: INVALID_ARG (missing/extra-shaped weight, bad config), UNSUPPORTED
 * (channel counts the kernels cannot tile), OOM, CUDA.  On error *out is NULL and
 * nothing is leaked.
 */
vaedec_status vaedec_create(const vaedec_config* config, const vaedec_tensor* weights, int n_weights,
                            vaedec_t** out);

/* Release every device allocation of the handle.  Synchronises the device first.  NULL is a no-op. */
void vaedec_destroy(vaedec_t* h);

/* Decoded output shape for a latent shape (ndim 4: B,C,H,W; ndim 5: B,C,T,H,W). */
vaedec_status vaedec_output_shape(const vaedec_t* h, const int64_t* latent_shape, int ndim, int64_t* out_shape);

/* Bytes of device workspace the handle owns (weights excluded). */
vaedec_status vaedec_workspace_bytes(const vaedec_t* h, size_t* bytes);

/* The workspace a handle created with `config` would own, computed on the host (no CUDA call, no
 * weights).  The band scheduler keeps every activation and the attention's scratch in one arena:
 * a dry walk of the decode at config->max_latent lists each tensor with the span of the walk in
 * which it is alive (from its producer to its last reader), and each is placed at the lowest
 * 256-byte-aligned offset whose bytes no tensor alive at the same time holds, largest first.
 * Bounded memory is the pages' concern for a single-GPU decode ("Static Layer-Wise VAE Decode",
 * Pretrained GPU Measurements: extra peak allocation); here the bound is the live set of the
 * largest layer, not a whole-image buffer per role.  The walk creates tensors in the same order
 * for every latent shape up to max_latent, so the layout holds for all of them.
 *   bytes            total workspace (= vaedec_workspace_bytes of the created handle)
 *   arena_bytes      the arena within it (may be NULL)
 *   peak_live_bytes  the largest sum of arena tensors alive at once, a lower bound on the arena (may be NULL)
 * INVALID_ARG / UNSUPPORTED as vaedec_create for a bad config. */
vaedec_status vaedec_plan_workspace(const vaedec_config* config, size_t* bytes, size_t* arena_bytes,
                                    size_t* peak_live_bytes);

/*
 * Decode on `stream` (a cudaStream_t; NULL = legacy default stream).
 * latent: DEVICE pointer, channels-first (NCHW or NCTHW), contiguous, model dtype.
 * out:    DEVICE pointer, caller-allocated, channels-first, model dtype, shape from
 *         vaedec_output_shape.
 * n_bands in [1, latent H]: band b holds floor(H/n) latent rows, the first H mod n
 * bands one more.  The output does not depend on n_bands (bit-identical).
 * Asynchronous: returns after enqueueing.  Errors: INVALID_ARG (shape above
 * max_latent, wrong ndim, channel mismatch, n_bands out of range, NULL pointer),
 * CUDA (launch failure).
 */
vaedec_status vaedec_decode(vaedec_t* h, const void* latent, const int64_t* latent_shape, int ndim, void* out,
                            int n_bands, void* stream);

/*
 * Band split axis ("VAE Parallel", Strategy Selection Contract: spatial_shard_height,
 * spatial_shard_width, auto).  On one GPU a band only decides which queries one attention pass
 * holds; no result depends on the axis or the band count.
 */
enum { VAEDEC_BANDS_HEIGHT = 0, VAEDEC_BANDS_WIDTH = 1, VAEDEC_BANDS_AUTO = 2 };

/*
 * The axis a request is split along ("VAE Parallel", Spatially-Sharded Decode): HEIGHT or WIDTH as
 * asked when that latent axis holds n_bands bands (at least one latent row or column each); AUTO:
 * the longer latent axis that can, width on ties.  latent_shape as for vaedec_decode (only its last
 * two entries, H and W, are read).  *axis_out receives VAEDEC_BANDS_HEIGHT or VAEDEC_BANDS_WIDTH.
 * Host only, no handle or device needed.  Errors: INVALID_ARG (NULL pointer, ndim not 4 or 5,
 * unknown axis, n_bands < 1, or no allowed axis can hold n_bands).
 */
vaedec_status vaedec_band_axis(const int64_t* latent_shape, int ndim, int n_bands, int axis, int* axis_out);

/*
 * vaedec_decode with the band split axis `axis` (VAEDEC_BANDS_*; AUTO resolved as in
 * vaedec_band_axis).  Width band b holds floor(W/n) latent columns, the first W mod n bands one
 * more; its queries are gathered into a dense buffer and its attention output scattered back.  The
 * output is bit-identical for every axis and band count.  Same arguments, ownership and errors as
 * vaedec_decode (n_bands must fit the chosen axis).
 */
vaedec_status vaedec_decode_bands(vaedec_t* h, const void* latent, const int64_t* latent_shape, int ndim, void* out,
                                  int n_bands, int axis, void* stream);

/*
 * Same as vaedec_decode with HOST buffers: copies the latent host->device, decodes,
 * copies the output device->host, and synchronises `stream` before returning.
 * Host buffers should be pinned for full copy bandwidth.  Also reports kernel-side
 * failures (TIMEOUT).
 */
vaedec_status vaedec_decode_host(vaedec_t* h, const void* latent_host, const int64_t* latent_shape, int ndim,
                                 void* out_host, int n_bands, void* stream);

/* Synchronise `stream` and report the device status word (TIMEOUT if a kernel gave up waiting); clears it. */
vaedec_status vaedec_sync(vaedec_t* h, void* stream);

/* Message of the calling thread's last failure ("" if none). */
const char* vaedec_last_error(void);

/* Number of kernel launches this handle has enqueued since vaedec_create. */
vaedec_status vaedec_launch_count(const vaedec_t* h, uint64_t* n);

/* ---- Per-op timing (profiling) -------------------------------------------------------
 * When enabled, each op of a decode (see the inspection calls below) is bracketed by
 * CUDA events recorded on the decode stream; the events cost a few microseconds of
 * host time per op and nothing on the device.  vaedec_profile_read waits for the last
 * profiled decode's events and writes each op's device milliseconds, in op order.
 */
vaedec_status vaedec_profile_enable(vaedec_t* h, int enable);
vaedec_status vaedec_profile_read(vaedec_t* h, float* ms, int max_ops, int* n_ops);

/* ---- GroupNorm without device allocation --------------------------------------------
 * The pages have no counterpart for this entry point; it serves callers that cannot
 * allocate device memory while they run: plugin hosts and inference servers that give
 * a plugin only its input/output buffers and forbid cudaMalloc inside their enqueue
 * callback, real-time pipelines whose memory is fixed at start-up, and code living
 * under another allocator.  It runs the same GroupNorm kernels as the decoder
 * (fixed one-row chunks of central moments, the weighted merge, scale/shift + optional
 * SiLU) on one channels-last tensor, with all scratch in one fixed 2.25 MiB array
 * compiled into this library.  It calls no cudaMalloc, cudaFree or allocating routine.
 *
 *   x      DEVICE [B][rows][W][C], in_dtype (VAEDEC_DTYPE_F32 or VAEDEC_DTYPE_BF16), 16-byte aligned
 *   y      DEVICE [B][rows][W][C], out_dtype (f32->bf16, f32->f32 or bf16->bf16), 16-byte aligned
 *   gamma, beta  DEVICE fp32 [C];  groups G divide C;  C a multiple of 8, at most 2048
 *   stream a cudaStream_t (NULL = legacy default stream); asynchronous
 * Limits of the fixed scratch: B * rows * G <= 131072 and B * C <= 32768; larger sizes
 * return VAEDEC_ERR_INVALID_ARG with a message naming the limit, before any launch.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current) and caches it under the current context's unique id; a call
 * in a context not seen before (after cudaDeviceReset, or in a caller's own driver-API
 * context) looks it up again.  Make the first call on each device, and in each new
 * context, before any stream capture.  Every call shares the array and leaves its last contents there; nothing in
 * it has to start at zero (each call writes every word it reads), but calls whose
 * kernels overlap on the GPU (e.g. on two streams) race on it and must be ordered by
 * the caller.  Every GPU that loads this library holds the array until process exit.
 */
vaedec_status vaedec_groupnorm_noalloc(int in_dtype, int out_dtype, const void* x, void* y, int B, int rows, int W,
                                       int C, int G, const float* gamma, const float* beta, float eps, int silu,
                                       void* stream);

/* ---- Band attention core ------------------------------------------------------------
 * The fused kernel the bf16 decode runs for its mid-block attention, on caller buffers:
 *   O[q, :] = softmax_k(Q[q, :] . K[k, :] / sqrt(C)) V[k, :]
 * for every query row q of F frames of ntok = grid_h * grid_w tokens, each query against every
 * key and value of its own frame ("VAEP：VAE 并行解码", Attention：本地 Q，全局 K/V).  The query
 * rows of a frame are split into n_bands height bands of the grid_h x grid_w token grid (band b:
 * floor(grid_h / n_bands) grid rows, the first grid_h mod n_bands bands one more); query tiles
 * never cross a band.  The result does not depend on n_bands, bit for bit.
 *   q, k   DEVICE bf16 [F][ntok][C] (token-major, channels contiguous)
 *   vt     DEVICE bf16 [F][C][ntok] (V transposed: tokens contiguous)
 *   o      DEVICE bf16 [F][ntok][C]; must not overlap q, k, vt or work
 *   C a multiple of 128, at most 512; ntok a multiple of 8; 1 <= n_bands <= grid_h; all device
 *   pointers 16-byte aligned
 *   work   DEVICE scratch of work_bytes >= vaedec_band_attention_work_bytes(F, grid_h, grid_w, C)
 *          (fp32 partials of the key splits; may be NULL when that size is 0)
 *   status DEVICE int the kernel ORs a nonzero error bit into if one of its bounded waits runs out
 *          (read it after the stream completes; the caller owns and clears it)
 *   stream a cudaStream_t (NULL = legacy default stream); asynchronous, allocates nothing
 * INVALID_ARG for a NULL pointer, a size or alignment outside these limits or too small a work
 * buffer (before any launch); CUDA for a failed launch. */
vaedec_status vaedec_band_attention_work_bytes(int F, int grid_h, int grid_w, int C, size_t* bytes);
vaedec_status vaedec_band_attention(const void* q, const void* k, const void* vt, void* o, int F, int grid_h,
                                    int grid_w, int C, int n_bands, void* work, size_t work_bytes, int* status,
                                    void* stream);

/* ---- Inspection (tests and profiling) ------------------------------------------------
 * The decode is a fixed list of ops (latent layout, conv, groupnorm, rmsnorm,
 * attention block, temporal upsample).  These calls describe that list for a latent
 * shape and band count, and run the decode up to one op, copying the op's input,
 * auxiliary input (a conv's residual, else nothing) and output activations into
 * caller DEVICE buffers (channels-last [B][T][H][W][C] in the model dtype, except
 * the final conv's channels-first output).
 */
vaedec_status vaedec_debug_num_ops(vaedec_t* h, const int64_t* latent_shape, int ndim, int n_bands, int* n_ops);
/* One line "key=value ..." describing op `op`; INVALID_ARG if buf is too small. */
vaedec_status vaedec_debug_op_desc(vaedec_t* h, const int64_t* latent_shape, int ndim, int n_bands, int op,
                                   char* buf, int buf_len);
/* Runs ops [0, op], copies, synchronises `stream`, returns OK (or the first error). */
vaedec_status vaedec_debug_run_until(vaedec_t* h, const void* latent, const int64_t* latent_shape, int ndim,
                                     int n_bands, int op, void* dst_in, size_t in_bytes, void* dst_aux,
                                     size_t aux_bytes, void* dst_out, size_t out_bytes, void* stream);

/* ---- failure injection (no counterpart on the pages; they test exception cleanup and
 * buffer release on failure: "Static Layer-Wise VAE Decode", Tests).  Process-wide, for tests.
 *
 * vaedec_debug_inject_fault: kind 0 = off; 1 = the nth device allocation made by any
 * vaedec_create from now on fails (create returns VAEDEC_ERR_OOM after releasing everything it
 * allocated); 2 = at the nth kernel launch of any decode from now on the decode records a
 * failure, enqueues nothing after that kernel and returns VAEDEC_ERR_CUDA (kernels already
 * enqueued complete).  nth >= 1.
 * The fault fires once, then injection switches itself off.  INVALID_ARG for other kinds.
 *
 * vaedec_debug_set_wait_limit: the limit of every bounded wait inside the library's kernels,
 * in nanoseconds (0 restores the default of 2 s).  With a tiny limit the waits run out: the
 * kernels record a status bit, let their issued copies land, free their TMEM and return, and the
 * decode returns VAEDEC_ERR_TIMEOUT; the handle stays usable.  Applies to the current device. */
vaedec_status vaedec_debug_inject_fault(int kind, int nth);
vaedec_status vaedec_debug_set_wait_limit(uint64_t ns);
/* Enqueues on `stream` (NULL: the legacy default stream) one kernel that waits, through the
 * same bounded wait as the decode kernels, on a barrier nothing ever completes: after the wait
 * limit it records a timeout in the handle's status word and returns, so the next vaedec_sync
 * returns VAEDEC_ERR_TIMEOUT and the handle stays usable. */
vaedec_status vaedec_debug_wait_probe(vaedec_t* h, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* VAEDEC_H_ */
