// fp32 CUDA-core direct convolution (the fp32 debug path).  One thread per
// (output pixel, phase, output channel): sum over taps and input channels in
// fp32, taps outside the input read nothing (zero padding), then the same
// scale / row-scale / bias / residual epilogue and output mapping as the
// tensor-core kernel.
#include <cuda_runtime.h>

#include "conv.h"
#include "kernels.h"
#include "ptx.cuh"
#include "launch.h"

namespace vd {

__global__ void conv_simple_f32_kernel(const ConvGeom g, const float* __restrict__ in,
                                       const float* __restrict__ w, int ntaps_w, const float* __restrict__ bias,
                                       const float* __restrict__ residual, const float* __restrict__ rowscale,
                                       float* __restrict__ out, long long total) {
  pdl_wait();   // the previous kernel on the stream has finished (programmatic launch)
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    long long r = idx;
    const int co = static_cast<int>(r % g.Cout);
    r /= g.Cout;
    const int phase = static_cast<int>(r % g.nphase);
    r /= g.nphase;
    const int x = static_cast<int>(r % g.W);
    r /= g.W;
    const int y = static_cast<int>(r % g.H);
    r /= g.H;
    const int t = static_cast<int>(r % g.T);
    const int b = static_cast<int>(r / g.T);
    float acc = 0.f;
    for (int k = 0; k < g.ntaps; ++k) {
      const ConvTap tp = g.taps[phase][k];
      const int ti = t + tp.dt, yi = y + tp.dy, xi = x + tp.dx;
      if (ti < 0 || ti >= g.T || yi < 0 || yi >= g.H || xi < 0 || xi >= g.W) continue;
      const float* ip = in + ((((long long)b * g.T + ti) * g.H + yi) * g.W + xi) * g.Cin;
      const float* wp = w + ((long long)co * ntaps_w + tp.wtap) * g.Cin;
      for (int ci = 0; ci < g.Cin; ++ci) acc = fmaf(ip[ci], wp[ci], acc);
    }
    const long long grid_pix = (((long long)b * g.T + t) * g.H + y) * g.W + x;
    float v = acc * g.scale;
    if (rowscale != nullptr) v *= rowscale[grid_pix];
    if (bias != nullptr) v += bias[co];
    int to = t, ch = co;
    if (g.time_up_c > 0) {
      const int half = co >= g.time_up_c ? 1 : 0;
      to = 1 + 2 * t + half;
      ch = co - half * g.time_up_c;
    }
    const int yo = y * g.osy + (g.nphase > 1 ? (phase >> 1) : 0);
    const int xo = x * g.osx + (g.nphase > 1 ? (phase & 1) : 0);
    const long long opix = (((long long)b * g.oT + to) * g.oH + yo) * g.oW + xo;
    if (!g.out_chfirst) {
      const long long a = opix * g.oC + ch;
      if (residual != nullptr) v += residual[a];
      out[a] = v;
    } else {
      const long long plane = (long long)g.oT * g.oH * g.oW;
      const long long sp = ((long long)to * g.oH + yo) * g.oW + xo;
      out[((long long)b * g.oC + ch) * plane + sp] = v;
    }
  }
}

cudaError_t launch_conv_simple_f32(const ConvGeom& g, const float* in, const float* wts, int ntaps_w,
                                   const float* bias, const float* residual, const float* rowscale, float* out,
                                   cudaStream_t stream) {
  const long long total = (long long)g.B * g.T * g.H * g.W * g.nphase * g.Cout;
  if (total <= 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  const int grid = static_cast<int>(blocks < 152LL * 64 ? blocks : 152LL * 64);
  launch_pdl(conv_simple_f32_kernel, grid, threads, 0, stream, g, in, wts, ntaps_w, bias, residual, rowscale, out, total);
  return cudaGetLastError();
}

}  // namespace vd
