// Host-side launchers of every kernel in the library (internal interface).
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include <string>

#include "conv.h"

namespace vd {

enum DType : int { kF32 = 1, kBF16 = 2 };

// ---------------------------------------------------------------- latent front-end
// Inverse latent BatchNorm (x * scale[cp] + shift[cp] per patched channel cp) and p x p unpatchify
// of a channels-first [B][C*p*p][Hp][Wp] latent into channels-last [B][p*Hp][p*Wp][C].
cudaError_t launch_latent_frontend(int dtype, const void* zp, void* y, int B, int C, int Hp, int Wp, int p,
                                   const float* scale, const float* shift, cudaStream_t stream);

// ---------------------------------------------------------------- width bands
// Copy the width band [c0, c0 + nc) of a channels-last frame [H][W][C] into a dense
// [H][nc][C] buffer (to_band = 1) or back (to_band = 0).  C * element size must be a
// multiple of 16 and both pointers 16-byte aligned.
cudaError_t launch_band_cols(int dtype, const void* src, void* dst, int H, int W, int C, int c0, int nc, int to_band,
                             cudaStream_t stream);

// ---------------------------------------------------------------- convolution
// Tensor-core implicit GEMM (bf16 in, fp32 accumulate, bf16/fp32 out).
// `wts` is [w_rows][ntaps_w][Cin] bf16 (K-major per output channel).  `out2`
// (optional) receives a bf16 copy of a channels-last output.
const char* conv_tc_plan(const ConvGeom& g, int* bk_out);

// A 1x1 convolution summed into a 3x3 conv's accumulators (a resnet's shortcut fused
// into its conv2): `in` channels-last bf16 [B][T][H][W][cin] on the conv's grid,
// `w` [w_rows][1][cin] bf16.  The caller folds the shortcut bias into the conv bias.
struct ConvShortcut {
  const void* in = nullptr;
  const void* w = nullptr;
  int cin = 0;
  int w_rows = 0;
};
// When g.gn_part is set and the chosen kernel can, the epilogue also writes the
// GroupNorm central moments of its output in fixed chunks and *gn_chunks receives
// the number of chunks per sample (0 when no moments were written).
cudaError_t launch_conv_tc(const ConvGeom& g, const void* in, const void* wts, int ntaps_w, int w_rows,
                           const float* bias, const void* residual, const float* rowscale, void* out, void* out2,
                           int* status, cudaStream_t stream, const char** why, int* gn_chunks = nullptr,
                           const ConvShortcut* sc = nullptr);

// Halo-tile variant (R output rows per CTA, activations staged once per channel
// chunk for all 3x3 taps); launch_conv_tc dispatches to it when applicable.
bool conv_halo_applicable(const ConvGeom& g);
cudaError_t launch_conv_halo(const ConvGeom& g, const void* in, const void* wts, int ntaps_w, int w_rows,
                             const float* bias, const void* residual, void* out, void* out2, int* status,
                             cudaStream_t stream, const char** why);

// Channel-major halo variant (output channels on M, up to 256 pixels on N).
bool conv_halo_t_applicable(const ConvGeom& g);
// Whether a shortcut of `sc_cin` input channels can be fused into this conv.
bool conv_halo_t_shortcut_ok(const ConvGeom& g, int sc_cin);
cudaError_t launch_conv_halo_t(const ConvGeom& g, const void* in, const void* wts, int ntaps_w, int w_rows,
                               const float* bias, const void* residual, void* out, void* out2, int* status,
                               cudaStream_t stream, const char** why, int* gn_chunks,
                               const ConvShortcut* sc = nullptr);

// Narrow-output 3x3 / causal 3x3x3 conv (C_out = 3): the three kernel rows share the
// MMA's N dimension.  `w_narrow` is [16][kt * 3 (frame, kernel column)][Cin] bf16 with row
// n = kernel_row * C_out + co (rows beyond 3 * C_out zero).
bool conv_narrow_applicable(const ConvGeom& g);
cudaError_t launch_conv_narrow(const ConvGeom& g, const void* in, const void* w_narrow, const float* bias,
                               void* out, int* status, cudaStream_t stream, const char** why);

// CUDA-core fp32 direct convolution over the same ConvGeom (the fp32 path).
// `wts` is [w_rows][ntaps_w][Cin] fp32.
cudaError_t launch_conv_simple_f32(const ConvGeom& g, const float* in, const float* wts, int ntaps_w,
                                   const float* bias, const float* residual, const float* rowscale, float* out,
                                   cudaStream_t stream);

// ---------------------------------------------------------------- GroupNorm
// Central moments of one fixed row chunk and one group: count, mean, sum of
// squared deviations.
struct GnPartial {
  float n, mean, m2, pad;
};

// Phase 1: per (sample, row chunk, group) central moments of a channels-last
// [B][rows][W][C] tensor (rows = T*H for video; chunk = `chunk_rows` rows), stored
// [sample][group][chunk] (the conv epilogue writes the same layout).
cudaError_t launch_gn_partials(int dtype, const void* x, int B, int rows, int W, int C, int G, int chunk_rows,
                               GnPartial* part, cudaStream_t stream);
// Phase 2: merge the chunks of each (sample, group) with the weighted rule and
// fold mean, variance, gamma and beta into a per-(sample, channel) scale/shift.
cudaError_t launch_gn_finalize(const GnPartial* part, int B, int n_chunks, int C, int G, const float* gamma,
                               const float* beta, float eps, float* scale, float* shift, cudaStream_t stream);
// y = x * scale[b, c] + shift[b, c], then SiLU when `silu`; x in `in_dtype`,
// y in `out_dtype`; `y_raw` (optional, `out_dtype`) receives x itself, cast.
cudaError_t launch_gn_apply(int in_dtype, int out_dtype, const void* x, void* y, void* y_raw,
                            long long pixels_per_sample, int B, int C, const float* scale, const float* shift,
                            int silu, cudaStream_t stream);

// Channel RMSNorm (Wan): y = x / max(||x||_2, 1e-12) * sqrt(C) * gamma, then SiLU
// when `silu`; dtypes and `y_raw` as for launch_gn_apply.
cudaError_t launch_rms_norm(int in_dtype, int out_dtype, const void* x, void* y, void* y_raw, long long pixels,
                            int C, const float* gamma, int silu, cudaStream_t stream);

// ---------------------------------------------------------------- GEMM
// D[m, n] = scale * scale_n[n] * sum_k A[m, k] B[n, k] + bias_m[m] + bias_n[n]
// (+ residual), stored channel-major: out[n * ldo + m].  A is [M][lda] and B
// [N][ldb] bf16, K contiguous, rows 16-byte aligned.  With splits > 1 the K range
// is divided among `splits` CTAs that write fp32 partials to
// out + s * split_stride (for the caller to sum in split order).
struct GemmArgs {
  const void* A = nullptr;
  long long lda = 0;
  const void* B = nullptr;
  long long ldb = 0;
  int M = 0, N = 0, K = 0;
  void* out = nullptr;
  long long ldo = 0;
  int out_f32 = 1;
  int splits = 1;
  long long split_stride = 0;
  const float* bias_m = nullptr;
  const float* bias_n = nullptr;
  const float* scale_n = nullptr;
  float scale = 1.f;
  const void* residual = nullptr;   // same layout and ldo as out
  int res_f32 = 0;
  void* out2 = nullptr;             // optional bf16 copy of out
};
cudaError_t launch_gemm_cm(const GemmArgs& a, int* status, cudaStream_t stream, const char** why);

// ---------------------------------------------------------------- attention
// Row softmax numerators of the fp32 path: P[r, k] = exp(S[r, k] - max_k S[r, :]), inv_l[r] =
// 1 / sum_k P[r, k]; S and P fp32 (p_dtype must be kF32).
cudaError_t launch_softmax_rows(int p_dtype, const float* S, void* P, float* inv_l, int rows, int nk,
                                cudaStream_t stream);

// Fused (flash-style) band attention, bf16 operands, fp32 softmax and accumulation:
//   O[q, :] = softmax_k(Q[q, :] . K[k, :] / sqrt(C)) V[k, :]
// for every query row q of `q` ([F * ntok][C] channels-last, frame f's rows at f * ntok) against
// every key of its own frame (`k` [F][ntok][C]; `vt` = V transposed, [F][C][ntok]).  The queries of
// a frame form n_seg consecutive band segments: the first seg_rem hold (seg_q + 1) * U rows, the
// others seg_q * U; query tiles never cross a segment.  A query row's arithmetic depends only on its
// row and on ntok, not on the segments.  Output bf16 [F * ntok][C] at `out` (the same row index as
// the query).  With flash_splits(ntok) > 1 the keys are split into that many ranges whose fp32
// partial outputs (`part`, [splits][F * ntok][C]) and row maxima/sums (`ml`, [splits][F * ntok]
// float2) are merged in split order by a second kernel.  C a multiple of 128 up to 512, ntok a
// multiple of 8, all pointers 16-byte aligned.
struct FlashArgs {
  const void* q = nullptr;
  const void* k = nullptr;
  const void* vt = nullptr;
  void* out = nullptr;
  float* part = nullptr;
  void* ml = nullptr;
  int F = 0;
  long long ntok = 0;
  int C = 0;
  int U = 0, seg_q = 0, seg_rem = 0, n_seg = 0;
};
int flash_splits(long long ntok);
// Bytes of `part` plus `ml` that launch_attn_flash needs (0 when flash_splits(ntok) == 1).
size_t flash_work_bytes(int F, long long ntok, int C);
// The attention kernel, then (a separate launch, nothing when there is one split) the merge of the
// key splits into `out`.
cudaError_t launch_attn_flash(const FlashArgs& a, int* status, cudaStream_t stream, const char** why);
cudaError_t launch_attn_combine(const FlashArgs& a, cudaStream_t stream);
cudaError_t set_wait_limit_attn_flash(unsigned long long ns);

// ---------------------------------------------------------------- layout
// [B][C][S] -> [B][S][C] (same dtype).
cudaError_t launch_to_channels_last(int dtype, const void* x, void* y, int B, int C, long long spatial,
                                    cudaStream_t stream);

// Lower (ns > 0) or restore (ns == 0) the bounded-wait limit of each source's kernels.
cudaError_t set_wait_limit_conv_tc(unsigned long long ns);
cudaError_t set_wait_limit_conv_halo(unsigned long long ns);
cudaError_t set_wait_limit_conv_halo_t(unsigned long long ns);
cudaError_t set_wait_limit_conv_narrow(unsigned long long ns);
cudaError_t set_wait_limit_gemm_cm(unsigned long long ns);

// One thread waits (bounded) on a barrier nothing completes; records kErrTimeoutFull in *status.
cudaError_t launch_wait_probe(int* status, cudaStream_t stream);

// Message returned by vaedec_last_error() on the calling thread.
void record_last_error(const std::string& message);

}  // namespace vd
