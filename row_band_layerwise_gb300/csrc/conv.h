// Convolution / GEMM problem description shared by the host planner and the
// conv kernels (tensor-core bf16 and CUDA-core fp32).
//
// Every convolution of the decode is an implicit GEMM
//   out[p, co] = sum_{tap, ci} W[co, tap, ci] * in[p + offset(tap), ci]
// over output pixels p of a (B, T, H, W) grid with channels-last activations.
// A centred 3x3 conv reads offsets (dy, dx) in {-1, 0, 1}^2 and gets its zero
// padding from out-of-range reads, which are zero (the tensor-memory-access
// unit fills them); a causal 3x3x3 conv adds dt in {-2, -1, 0}.  A nearest-2x
// upsample followed by a 3x3 conv is computed on the low-resolution input as
// four output phases (py, px), each reading low-resolution offsets
// floor((p + k - 1) / 2), so the upsampled tensor never exists.  Plain GEMMs
// (attention projections, scores, probabilities times values) are 1-tap
// "convs" over a 1-row grid.
#pragma once
#include <cstdint>

namespace vd {

constexpr int kMaxTaps = 27;
constexpr int kMaxPhases = 4;

struct ConvTap {
  int8_t dt, dy, dx, wtap;   // input offsets and the weight tap they multiply
};

struct ConvGeom {
  // Input tensor (channels-last [B][T][H][W][Cin]) = the output grid.
  int B, T, H, W;
  int Cin;
  int Cout;                  // GEMM N (real output channels)
  int nphase;                // 1, or 4 for a fused nearest-2x upsample
  int ntaps;                 // taps per phase
  ConvTap taps[kMaxPhases][kMaxTaps];
  // Output tensor.
  int oT, oH, oW, oC;        // output dims (channels-last) or [B][oC][oT][oH][oW] (channels-first)
  int osy, osx;              // output = grid * (osy, osx) + phase offset
  int time_up_c;             // >0: temporal upsample, column co -> frame 1+2t+(co>=c), channel co%c
  int out_chfirst;           // 1: channels-first store
  int out_f32;               // 1: fp32 output, 0: bf16
  int res_f32;               // 1: the residual is fp32, 0: bf16
  float scale;               // v = acc * scale (* rowscale[p]) + bias + residual
  // Optional GroupNorm chunk moments of the stored output (kernels that support it):
  // `gn_part` points to {n, mean, M2, pad} float4 records, `gn_groups` groups.
  void* gn_part;
  int gn_groups;
};

}  // namespace vd
