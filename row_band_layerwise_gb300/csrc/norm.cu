// GroupNorm in two phases, plus the Wan channel RMSNorm.
//
// GroupNorm statistics span the whole image, so every band must use the same
// merged mean and variance ("VAEP：VAE 并行解码", section GroupNorm：合并全局统计量;
// "Static Layer-Wise VAE Decode", "Semantics and Communication").  Here:
//   phase 1  one CTA per (sample, fixed row chunk): central moments
//            (count, mean, sum of squared deviations) per group, in fp32,
//            from per-channel shifted sums merged across threads in a fixed
//            order.  Chunks never depend on the band split, so the result
//            is bit-identical for every band count.
//   phase 2  one warp per (sample, group): merge the chunks with the pages'
//            weighted rule  mean = sum w_i mean_i,
//            var = sum w_i (var_i + (mean_i - mean)^2),  w_i = n_i / N,
//            then fold gamma / beta into a per-(sample, channel) scale/shift.
//   apply    y = x * scale + shift (+ SiLU), 16-byte vectors, HBM-bound.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "kernels.h"

namespace vd {

namespace {

template <typename T>
struct Vec8;
template <>
struct Vec8<float> {
  __device__ static void load(const float* p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  __device__ static void store(float* p, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};
template <>
struct Vec8<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h[j]);
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 a;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&a);
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
    *reinterpret_cast<uint4*>(p) = a;
  }
};

// Chan et al. pairwise merge of (n, mean, M2).
__device__ __forceinline__ void merge_into(float& n, float& mean, float& m2, float nb, float meanb, float m2b) {
  if (nb == 0.f) return;
  if (n == 0.f) {
    n = nb;
    mean = meanb;
    m2 = m2b;
    return;
  }
  const float nt = n + nb;
  const float d = meanb - mean;
  mean = mean + d * (nb / nt);
  m2 = m2 + m2b + d * d * (n * nb / nt);
  n = nt;
}

constexpr int kGnThreads = 256;

// Shared layout: per thread 8 channels x (n, mean, M2).
template <typename T>
__global__ void __launch_bounds__(kGnThreads) gn_partials_kernel(const T* __restrict__ x, int rows, int W, int C,
                                                                 int G, int chunk_rows, int n_chunks,
                                                                 GnPartial* __restrict__ part) {
  extern __shared__ float sh[];   // [nthreads][8][3]
  const int chunk = blockIdx.x, b = blockIdx.y;
  const int vpp = C / 8;                        // vectors per pixel
  const int lanes = kGnThreads / vpp;           // pixels processed in parallel
  const int nthreads = lanes * vpp;
  const int tid = threadIdx.x;
  const int r0 = chunk * chunk_rows;
  const int r1 = min(rows, r0 + chunk_rows);
  const long long npix = (long long)(r1 - r0) * W;
  const T* base = x + ((long long)b * rows + r0) * W * C;

  float cnt = 0.f, k[8], s1[8], s2[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) { k[j] = 0.f; s1[j] = 0.f; s2[j] = 0.f; }
  if (tid < nthreads) {
    const int v = tid % vpp;
    const int pl = tid / vpp;
    bool first = true;
    for (long long pix = pl; pix < npix; pix += lanes) {
      float val[8];
      Vec8<T>::load(base + pix * C + v * 8, val);
      if (first) {
#pragma unroll
        for (int j = 0; j < 8; ++j) k[j] = val[j];
        first = false;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = val[j] - k[j];
        s1[j] += d;
        s2[j] = fmaf(d, d, s2[j]);
      }
      cnt += 1.f;
    }
  }
  // per-channel central moments
  float* my = sh + tid * 24;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float mean_off = cnt > 0.f ? s1[j] / cnt : 0.f;
    my[3 * j + 0] = cnt;
    my[3 * j + 1] = k[j] + mean_off;
    my[3 * j + 2] = cnt > 0.f ? fmaxf(s2[j] - s1[j] * mean_off, 0.f) : 0.f;
  }
  __syncthreads();
  // one thread per group merges its channels over all pixel lanes in a fixed order
  const int cg = C / G;
  for (int g = tid; g < G; g += blockDim.x) {
    float n = 0.f, mean = 0.f, m2 = 0.f;
    for (int pl = 0; pl < lanes; ++pl) {
      for (int c = g * cg; c < (g + 1) * cg; ++c) {
        const int t = pl * vpp + c / 8;
        const float* e = sh + t * 24 + 3 * (c % 8);
        merge_into(n, mean, m2, e[0], e[1], e[2]);
      }
    }
    GnPartial o;
    o.n = n;
    o.mean = mean;
    o.m2 = m2;
    o.pad = 0.f;
    part[((long long)b * n_chunks + chunk) * G + g] = o;
  }
}

// One CTA per (sample, group), in one pass over the chunk moments.  Thread t folds
// chunks t, t + 512, ... in order into (n, mean, M2) with the two-part form of the
// weighted rule (for parts a, b: mean = w_a mean_a + w_b mean_b and
// M2 = M2_a + M2_b + (mean_b - mean_a)^2 n_a n_b / n, which is the rule
// var = sum w_i (var_i + (mean_i - mean)^2) for two parts times n); the 512
// thread results are then combined with the same two-part rule along a fixed
// tree.  Every step is fixed by the chunk geometry, so the result does not
// depend on how the tensor was produced (band count, tile order).
constexpr int kFinThreads = 512;

__global__ void __launch_bounds__(kFinThreads) gn_finalize_kernel(const GnPartial* __restrict__ part, int B,
                                                                  int n_chunks, int C, int G,
                                                                  const float* __restrict__ gamma,
                                                                  const float* __restrict__ beta, float eps,
                                                                  float* __restrict__ scale,
                                                                  float* __restrict__ shift) {
  __shared__ float sn[kFinThreads], sm[kFinThreads], s2[kFinThreads];
  const int b = blockIdx.x / G, g = blockIdx.x % G;
  const int t = threadIdx.x;
  const GnPartial* pp = part + (long long)b * n_chunks * G + g;
  float n = 0.f, mean = 0.f, m2 = 0.f;
  int c = t;
  // four loads in flight per step, folded in chunk order
  for (; c + 3 * kFinThreads < n_chunks; c += 4 * kFinThreads) {
    GnPartial e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = pp[(long long)(c + i * kFinThreads) * G];
#pragma unroll
    for (int i = 0; i < 4; ++i) merge_into(n, mean, m2, e[i].n, e[i].mean, e[i].m2);
  }
  for (; c < n_chunks; c += kFinThreads) {
    const GnPartial e = pp[(long long)c * G];
    merge_into(n, mean, m2, e.n, e.mean, e.m2);
  }
  sn[t] = n;
  sm[t] = mean;
  s2[t] = m2;
  __syncthreads();
  for (int half = kFinThreads / 2; half > 0; half >>= 1) {
    if (t < half) {
      float na = sn[t], ma = sm[t], m2a = s2[t];
      merge_into(na, ma, m2a, sn[t + half], sm[t + half], s2[t + half]);
      sn[t] = na;
      sm[t] = ma;
      s2[t] = m2a;
    }
    __syncthreads();
  }
  const float var = sn[0] > 0.f ? s2[0] / sn[0] : 0.f;
  const float rstd = rsqrtf(var + eps);
  const float gmean = sm[0];
  const int cg = C / G;
  for (int ch = g * cg + t; ch < (g + 1) * cg; ch += kFinThreads) {
    const float a = gamma[ch] * rstd;
    scale[(long long)b * C + ch] = a;
    shift[(long long)b * C + ch] = beta[ch] - gmean * a;
  }
}

// SiLU(v) = v / (1 + exp(-v)) with CUDA's fast exponential and fast division
// (the result is rounded to bf16 or feeds fp32 storage; both intrinsics are
// within a few ulp, and exp(-v) = inf for very negative v gives 0 as it should).
__device__ __forceinline__ float silu_f(float v) { return __fdividef(v, 1.f + __expf(-v)); }

__device__ __forceinline__ void load8f(const float* p, float (&o)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) gn_apply_kernel(const Tin* __restrict__ x, Tout* __restrict__ y,
                                                       Tout* __restrict__ y_raw, long long nvec,
                                                       long long vec_per_sample, int C,
                                                       const float* __restrict__ scale,
                                                       const float* __restrict__ shift, int silu) {
  const int vpp = C / 8;
  const long long step = (long long)gridDim.x * blockDim.x;
  // two 8-element vectors per thread and iteration: more loads in flight
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nvec; i += 2 * step) {
    const long long i2 = i + step;
    const bool has2 = i2 < nvec;
    float v[8], w[8];
    Vec8<Tin>::load(x + i * 8, v);
    if (has2) Vec8<Tin>::load(x + i2 * 8, w);
    {
      if (y_raw != nullptr) Vec8<Tout>::store(y_raw + i * 8, v);
      const int b = static_cast<int>(i / vec_per_sample);
      const int c0 = static_cast<int>(i % vpp) * 8;
      float a[8], sh[8], o[8];
      load8f(scale + (long long)b * C + c0, a);
      load8f(shift + (long long)b * C + c0, sh);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float t = fmaf(v[j], a[j], sh[j]);
        o[j] = silu ? silu_f(t) : t;
      }
      Vec8<Tout>::store(y + i * 8, o);
    }
    if (has2) {
      if (y_raw != nullptr) Vec8<Tout>::store(y_raw + i2 * 8, w);
      const int b = static_cast<int>(i2 / vec_per_sample);
      const int c0 = static_cast<int>(i2 % vpp) * 8;
      float a[8], sh[8], o[8];
      load8f(scale + (long long)b * C + c0, a);
      load8f(shift + (long long)b * C + c0, sh);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float t = fmaf(w[j], a[j], sh[j]);
        o[j] = silu ? silu_f(t) : t;
      }
      Vec8<Tout>::store(y + i2 * 8, o);
    }
  }
}

// One warp per pixel.
template <typename Tin, typename Tout>
__global__ void rms_norm_kernel(const Tin* __restrict__ x, Tout* __restrict__ y, Tout* __restrict__ y_raw,
                                long long pixels, int C, const float* __restrict__ gamma, int silu) {
  const long long wid = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  const int nv = C / 8;
  const float sc = sqrtf(static_cast<float>(C));
  for (long long pix = wid; pix < pixels; pix += nw) {
    const Tin* xp = x + pix * C;
    float v[2][8];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int vi = lane + 32 * k;
      if (vi < nv) {
        Vec8<Tin>::load(xp + vi * 8, v[k]);
#pragma unroll
        for (int j = 0; j < 8; ++j) ss = fmaf(v[k][j], v[k][j], ss);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = sc / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int vi = lane + 32 * k;
      if (vi < nv) {
        if (y_raw != nullptr) Vec8<Tout>::store(y_raw + pix * C + vi * 8, v[k]);
        float o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float t = v[k][j] * inv * __ldg(gamma + vi * 8 + j);
          o[j] = silu ? silu_f(t) : t;
        }
        Vec8<Tout>::store(y + pix * C + vi * 8, o);
      }
    }
  }
}

int grid_for(long long work, int threads) {
  const long long b = (work + threads - 1) / threads;
  return static_cast<int>(b < 152LL * 8 ? (b < 1 ? 1 : b) : 152LL * 8);
}

}  // namespace

cudaError_t launch_gn_partials(int dtype, const void* x, int B, int rows, int W, int C, int G, int chunk_rows,
                               GnPartial* part, cudaStream_t stream) {
  if (C % 8 != 0 || C / 8 > kGnThreads || C % G != 0 || chunk_rows < 1) return cudaErrorInvalidValue;
  const int n_chunks = (rows + chunk_rows - 1) / chunk_rows;
  dim3 grid(n_chunks, B);
  const size_t smem = kGnThreads * 24 * sizeof(float);
  if (dtype == kBF16)
    gn_partials_kernel<__nv_bfloat16><<<grid, kGnThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16*>(x), rows, W, C, G, chunk_rows, n_chunks, part);
  else
    gn_partials_kernel<float><<<grid, kGnThreads, smem, stream>>>(static_cast<const float*>(x), rows, W, C, G,
                                                                  chunk_rows, n_chunks, part);
  return cudaGetLastError();
}

cudaError_t launch_gn_finalize(const GnPartial* part, int B, int n_chunks, int C, int G, const float* gamma,
                               const float* beta, float eps, float* scale, float* shift, cudaStream_t stream) {
  gn_finalize_kernel<<<B * G, kFinThreads, 0, stream>>>(part, B, n_chunks, C, G, gamma, beta, eps, scale, shift);
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
void gn_apply_t(const void* x, void* y, void* y_raw, long long nvec, long long vps, int C, const float* scale,
                const float* shift, int silu, cudaStream_t stream) {
  const int threads = 256;
  gn_apply_kernel<Tin, Tout><<<grid_for(nvec, threads), threads, 0, stream>>>(
      static_cast<const Tin*>(x), static_cast<Tout*>(y), static_cast<Tout*>(y_raw), nvec, vps, C, scale, shift,
      silu);
}

cudaError_t launch_gn_apply(int in_dtype, int out_dtype, const void* x, void* y, void* y_raw,
                            long long pixels_per_sample, int B, int C, const float* scale, const float* shift,
                            int silu, cudaStream_t stream) {
  if (C % 8 != 0) return cudaErrorInvalidValue;
  const long long vps = pixels_per_sample * (C / 8);
  const long long nvec = vps * B;
  if (nvec <= 0) return cudaSuccess;
  if (in_dtype == kF32 && out_dtype == kBF16)
    gn_apply_t<float, __nv_bfloat16>(x, y, y_raw, nvec, vps, C, scale, shift, silu, stream);
  else if (in_dtype == kF32 && out_dtype == kF32)
    gn_apply_t<float, float>(x, y, y_raw, nvec, vps, C, scale, shift, silu, stream);
  else if (in_dtype == kBF16 && out_dtype == kBF16)
    gn_apply_t<__nv_bfloat16, __nv_bfloat16>(x, y, y_raw, nvec, vps, C, scale, shift, silu, stream);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
void rms_t(const void* x, void* y, void* y_raw, long long pixels, int C, const float* gamma, int silu,
           cudaStream_t stream) {
  const int threads = 256;
  rms_norm_kernel<Tin, Tout><<<grid_for(pixels * 32, threads), threads, 0, stream>>>(
      static_cast<const Tin*>(x), static_cast<Tout*>(y), static_cast<Tout*>(y_raw), pixels, C, gamma, silu);
}

cudaError_t launch_rms_norm(int in_dtype, int out_dtype, const void* x, void* y, void* y_raw, long long pixels,
                            int C, const float* gamma, int silu, cudaStream_t stream) {
  if (C % 8 != 0 || C > 512) return cudaErrorInvalidValue;
  if (pixels <= 0) return cudaSuccess;
  if (in_dtype == kF32 && out_dtype == kBF16)
    rms_t<float, __nv_bfloat16>(x, y, y_raw, pixels, C, gamma, silu, stream);
  else if (in_dtype == kF32 && out_dtype == kF32)
    rms_t<float, float>(x, y, y_raw, pixels, C, gamma, silu, stream);
  else if (in_dtype == kBF16 && out_dtype == kBF16)
    rms_t<__nv_bfloat16, __nv_bfloat16>(x, y, y_raw, pixels, C, gamma, silu, stream);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace vd
