// Attention softmax for band-local queries against global keys
// ("VAEP：VAE 并行解码", section Attention：本地 Q，全局 K/V): the scores of one
// band's query rows against every key are normalised row by row.
// Also the small layout kernel that turns the caller's channels-first latent
// into the channels-last activation layout.
#include <cuda_runtime.h>
#include <algorithm>
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "launch.h"

namespace vd {

namespace {

constexpr int kSmThreads = 256;

__device__ __forceinline__ float block_reduce_max(float v, float* sh) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  float r = sh[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, sh[i]);
  return r;
}

__device__ __forceinline__ float block_reduce_sum(float v, float* sh) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  float r = sh[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r += sh[i];
  return r;
}

template <typename P>
__device__ __forceinline__ float store_p(P* p, float v);
template <>
__device__ __forceinline__ float store_p<float>(float* p, float v) {
  *p = v;
  return v;
}

__device__ __forceinline__ float load_s(const float* p) { return *p; }

// Four consecutive scores (16-byte aligned), streamed once.
__device__ __forceinline__ float4 load_s4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }

template <typename SIn, typename P>
__global__ void __launch_bounds__(kSmThreads) softmax_rows_kernel(const SIn* __restrict__ S, P* __restrict__ Pm,
                                                                  float* __restrict__ inv_l, int nk) {
  pdl_wait();   // the previous kernel on the stream has finished (programmatic launch)
  __shared__ float red[32];
  const long long row = blockIdx.x;
  const SIn* s = S + row * nk;
  P* p = Pm + row * nk;
  float m = -INFINITY;
  for (int k = threadIdx.x; k < nk; k += blockDim.x) m = fmaxf(m, load_s(s + k));
  m = block_reduce_max(m, red);
  float l = 0.f;
  for (int k = threadIdx.x; k < nk; k += blockDim.x) l += store_p<P>(p + k, __expf(load_s(s + k) - m));
  l = block_reduce_sum(l, red);
  if (threadIdx.x == 0) inv_l[row] = 1.f / l;
}

// Single-read variant: the row stays in registers (NV float4 per thread, rows of
// at most 1024 * NV scores, nk a multiple of 4), so S is read from memory once.
// Same definition as softmax_rows_kernel (max, exp of the difference, sum of the
// stored values, one reciprocal); the sum is taken four values at a time.
template <typename P>
__device__ __forceinline__ float store_p4(P* p, float4 v);
template <>
__device__ __forceinline__ float store_p4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
  return (v.x + v.y) + (v.z + v.w);
}

template <typename SIn, typename P, int NV>
__global__ void __launch_bounds__(kSmThreads) softmax_rows_reg_kernel(const SIn* __restrict__ S, P* __restrict__ Pm,
                                                                      float* __restrict__ inv_l, int nk) {
  pdl_wait();   // the previous kernel on the stream has finished (programmatic launch)
  __shared__ float red[32];
  const long long row = blockIdx.x;
  const SIn* srow = S + row * nk;
  P* p = Pm + row * nk;
  const int n4 = nk >> 2;
  float4 v[NV];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = threadIdx.x + i * kSmThreads;
    if (idx < n4) {
      v[i] = load_s4(srow + 4 * idx);
      m = fmaxf(m, fmaxf(fmaxf(v[i].x, v[i].y), fmaxf(v[i].z, v[i].w)));
    }
  }
  m = block_reduce_max(m, red);
  float l = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = threadIdx.x + i * kSmThreads;
    if (idx < n4) {
      float4 e;
      e.x = __expf(v[i].x - m);
      e.y = __expf(v[i].y - m);
      e.z = __expf(v[i].z - m);
      e.w = __expf(v[i].w - m);
      l += store_p4<P>(p + 4 * idx, e);
    }
  }
  l = block_reduce_sum(l, red);
  if (threadIdx.x == 0) inv_l[row] = 1.f / l;
}

template <typename T>
__global__ void to_channels_last_kernel(const T* __restrict__ x, T* __restrict__ y, int C, long long spatial,
                                        long long total) {
  pdl_wait();   // the previous kernel on the stream has finished (programmatic launch)
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = static_cast<int>(i % C);
    const long long r = i / C;
    const long long sp = r % spatial;
    const long long b = r / spatial;
    y[i] = x[(b * C + c) * spatial + sp];
  }
}

template <typename SIn>
cudaError_t softmax_rows_t(const SIn* S, float* P, float* inv_l, int rows, int nk, cudaStream_t stream) {
  if (nk % 4 == 0 && nk <= 16 * 4 * kSmThreads) {
    const int nv = (nk + 4 * kSmThreads - 1) / (4 * kSmThreads);
#define VD_SOFTMAX_REG(NV)                                                                                \
  if (nv <= NV) {                                                                                         \
    launch_pdl(softmax_rows_reg_kernel<SIn, float, NV>, rows, kSmThreads, 0, stream, S, P, inv_l, nk);    \
    return cudaGetLastError();                                                                            \
  }
    VD_SOFTMAX_REG(2)
    VD_SOFTMAX_REG(4)
    VD_SOFTMAX_REG(8)
    VD_SOFTMAX_REG(16)
#undef VD_SOFTMAX_REG
  }
  launch_pdl(softmax_rows_kernel<SIn, float>, rows, kSmThreads, 0, stream, S, P, inv_l, nk);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_softmax_rows(int p_dtype, const float* S, void* P, float* inv_l, int rows, int nk,
                                cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (p_dtype != kF32) return cudaErrorInvalidValue;   // the fp32 path's probabilities
  return softmax_rows_t(S, static_cast<float*>(P), inv_l, rows, nk, stream);
}

cudaError_t launch_to_channels_last(int dtype, const void* x, void* y, int B, int C, long long spatial,
                                    cudaStream_t stream) {
  const long long total = (long long)B * C * spatial;
  if (total <= 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 152LL * 32) blocks = 152LL * 32;
  if (dtype == kBF16)
    launch_pdl(to_channels_last_kernel<__nv_bfloat16>, (int)blocks, threads, 0, stream, 
        static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), C, spatial, total);
  else
    launch_pdl(to_channels_last_kernel<float>, (int)blocks, threads, 0, stream, static_cast<const float*>(x),
                                                                       static_cast<float*>(y), C, spatial, total);
  return cudaGetLastError();
}


namespace {

// Copy one width band of a channels-last frame [H][W][C] to or from a dense [H][nc][C] buffer
// (16-byte vectors; C * sizeof(T) is a multiple of 16).
template <typename T>
__global__ void band_cols_kernel(const T* __restrict__ src, T* __restrict__ dst, int H, int W, int C, int c0, int nc,
                                 int to_band) {
  pdl_wait();   // the previous kernel on the stream has finished (programmatic launch)
  const int vpp = C * static_cast<int>(sizeof(T)) / 16;   // vectors per pixel
  const long long n = static_cast<long long>(H) * nc * vpp;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(i % vpp);
    const long long px = i / vpp;
    const int j = static_cast<int>(px % nc);
    const int h = static_cast<int>(px / nc);
    const long long band_off = (static_cast<long long>(h) * nc + j) * vpp + v;
    const long long full_off = (static_cast<long long>(h) * W + c0 + j) * vpp + v;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    if (to_band)
      d4[band_off] = s4[full_off];
    else
      d4[full_off] = s4[band_off];
  }
}

}  // namespace

cudaError_t launch_band_cols(int dtype, const void* src, void* dst, int H, int W, int C, int c0, int nc, int to_band,
                             cudaStream_t stream) {
  const int es = dtype == kBF16 ? 2 : 4;
  if ((C * es) % 16 != 0 || c0 < 0 || nc < 1 || c0 + nc > W) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) return cudaErrorInvalidValue;
  const long long n = static_cast<long long>(H) * nc * (C * es / 16);
  if (n <= 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = std::min<long long>((n + threads - 1) / threads, 152LL * 16);
  if (dtype == kBF16)
    launch_pdl(band_cols_kernel<__nv_bfloat16>, (int)blocks, threads, 0, stream,
               static_cast<const __nv_bfloat16*>(src), static_cast<__nv_bfloat16*>(dst), H, W, C, c0, nc, to_band);
  else
    launch_pdl(band_cols_kernel<float>, (int)blocks, threads, 0, stream, static_cast<const float*>(src),
               static_cast<float*>(dst), H, W, C, c0, nc, to_band);
  return cudaGetLastError();
}


namespace {

// AutoencoderKLFlux2 front-end: undo the inference BatchNorm of the patchified latent (per patched
// channel: x * scale + shift with scale = sqrt(var + eps), shift = mean) and unpatchify channel
// c*p*p + py*p + px of the (Hp, Wp) grid to pixel (p*y + py, p*x + px) of channel c, written
// channels-last on the (p*Hp, p*Wp) grid.  fp32 arithmetic, one rounding to T.
template <typename T>
__global__ void latent_frontend_kernel(const T* __restrict__ zp, T* __restrict__ y, int B, int C, int Hp, int Wp,
                                       int p, const float* __restrict__ scale, const float* __restrict__ shift) {
  pdl_wait();   // the previous kernel on the stream has finished (programmatic launch)
  const int H = Hp * p, W = Wp * p;
  const long long n = static_cast<long long>(B) * H * W * C;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % C);
    const long long px = i / C;
    const int X = static_cast<int>(px % W);
    const int Y = static_cast<int>((px / W) % H);
    const int b = static_cast<int>(px / (static_cast<long long>(W) * H));
    const int cp = (c * p + Y % p) * p + X % p;
    const long long src = ((static_cast<long long>(b) * C * p * p + cp) * Hp + Y / p) * Wp + X / p;
    const float v = static_cast<float>(zp[src]) * scale[cp] + shift[cp];
    y[i] = static_cast<T>(v);
  }
}

}  // namespace

cudaError_t launch_latent_frontend(int dtype, const void* zp, void* y, int B, int C, int Hp, int Wp, int p,
                                   const float* scale, const float* shift, cudaStream_t stream) {
  const long long n = static_cast<long long>(B) * Hp * p * Wp * p * C;
  if (n <= 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = std::min<long long>((n + threads - 1) / threads, 152LL * 16);
  if (dtype == kBF16)
    launch_pdl(latent_frontend_kernel<__nv_bfloat16>, (int)blocks, threads, 0, stream,
               static_cast<const __nv_bfloat16*>(zp), static_cast<__nv_bfloat16*>(y), B, C, Hp, Wp, p, scale, shift);
  else
    launch_pdl(latent_frontend_kernel<float>, (int)blocks, threads, 0, stream, static_cast<const float*>(zp),
               static_cast<float*>(y), B, C, Hp, Wp, p, scale, shift);
  return cudaGetLastError();
}

}  // namespace vd
