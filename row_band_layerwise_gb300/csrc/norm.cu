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
#include "ptx.cuh"
#include "launch.h"

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
  // streaming load: the data is read once, keep it from displacing reused lines in L2
  __device__ static void load_stream(const float* p, float (&v)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
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
  __device__ static void load_stream(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 a = __ldcs(reinterpret_cast<const uint4*>(p));
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
  pdl_wait();   // the previous kernel on the stream has finished (programmatic launch)
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
    part[((long long)b * G + g) * n_chunks + chunk] = o;
  }
}

// One CTA per (sample, group), in one pass over the chunk moments.  Thread t folds
// chunks t, t + 1024, ... in order into (n, mean, M2) with the two-part form of the
// weighted rule (for parts a, b: mean = w_a mean_a + w_b mean_b and
// M2 = M2_a + M2_b + (mean_b - mean_a)^2 n_a n_b / n, which is the rule
// var = sum w_i (var_i + (mean_i - mean)^2) for two parts times n); the 1024
// thread results are then combined with the same two-part rule along a fixed
// tree.  Every step is fixed by the chunk geometry, so the result does not
// depend on how the tensor was produced (band count, tile order).
constexpr int kFinThreads = 1024;   // with eight loads in flight per thread: one pass of latency

__global__ void __launch_bounds__(kFinThreads) gn_finalize_kernel(const GnPartial* __restrict__ part, int B,
                                                                  int n_chunks, int C, int G,
                                                                  const float* __restrict__ gamma,
                                                                  const float* __restrict__ beta, float eps,
                                                                  float* __restrict__ scale,
                                                                  float* __restrict__ shift) {
  pdl_wait();   // the previous kernel on the stream has finished (programmatic launch)
  __shared__ float sn[kFinThreads], sm[kFinThreads], s2[kFinThreads];
  const int b = blockIdx.x / G, g = blockIdx.x % G;
  const int t = threadIdx.x;
  const GnPartial* pp = part + ((long long)b * G + g) * n_chunks;   // [sample][group][chunk]
  float n = 0.f, mean = 0.f, m2 = 0.f;
  int c = t;
  // eight loads in flight per step, folded in chunk order
  for (; c + 7 * kFinThreads < n_chunks; c += 8 * kFinThreads) {
    GnPartial e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = pp[c + i * kFinThreads];
#pragma unroll
    for (int i = 0; i < 8; ++i) merge_into(n, mean, m2, e[i].n, e[i].mean, e[i].m2);
  }
  for (; c < n_chunks; c += kFinThreads) {
    const GnPartial e = pp[c];
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
__global__ void __launch_bounds__(1024) gn_apply_kernel(const Tin* __restrict__ x, Tout* __restrict__ y,
                                                       Tout* __restrict__ y_raw, uint32_t nvec,
                                                       uint32_t vec_per_sample, int C, int vpp_log2,
                                                       const float* __restrict__ scale,
                                                       const float* __restrict__ shift, int silu) {
  pdl_wait();   // the previous kernel on the stream has finished (programmatic launch)
  // 32-bit vector indices (the launcher guarantees nvec < 2^31); the channel of a vector is a
  // mask when C / 8 is a power of two (every GroupNorm width here), else a 32-bit remainder
  const uint32_t vpp = static_cast<uint32_t>(C / 8);
  const uint32_t step = gridDim.x * blockDim.x;
  // a thread's channels stay the same on every iteration when the grid stride is a multiple of C / 8
  // (launchers use multiples of 256 threads, C / 8 <= 64); with one sample its scale and shift are
  // then fixed and loaded once
  const bool fixed = vec_per_sample == nvec && vpp_log2 >= 0 && (step & (vpp - 1)) == 0;
  float fa[8], fsh[8];
  if (fixed) {
    const uint32_t c0 = ((blockIdx.x * blockDim.x + threadIdx.x) & (vpp - 1)) * 8;
    load8f(scale + c0, fa);
    load8f(shift + c0, fsh);
  }
  // two 8-element vectors per thread and iteration: more loads in flight
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += 2 * step) {
    const uint32_t i2 = i + step;
    const bool has2 = i2 < nvec;
    float v[8], w[8];
    Vec8<Tin>::load_stream(x + static_cast<size_t>(i) * 8, v);
    if (has2) Vec8<Tin>::load_stream(x + static_cast<size_t>(i2) * 8, w);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (h == 1 && !has2) break;
      const uint32_t iv = h == 0 ? i : i2;
      float (&u)[8] = h == 0 ? v : w;
      if (y_raw != nullptr) Vec8<Tout>::store(y_raw + static_cast<size_t>(iv) * 8, u);
      float a[8], sh[8], o[8];
      if (fixed) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          a[j] = fa[j];
          sh[j] = fsh[j];
        }
      } else {
        const uint32_t bs = vec_per_sample == nvec ? 0u : iv / vec_per_sample;
        const uint32_t c0 = (vpp_log2 >= 0 ? (iv & (vpp - 1)) : iv % vpp) * 8;
        load8f(scale + static_cast<size_t>(bs) * C + c0, a);
        load8f(shift + static_cast<size_t>(bs) * C + c0, sh);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float t = fmaf(u[j], a[j], sh[j]);
        o[j] = silu ? silu_f(t) : t;
      }
      Vec8<Tout>::store(y + static_cast<size_t>(iv) * 8, o);
    }
  }
}

// Four consecutive channels.
template <typename T>
struct Vec4;
template <>
struct Vec4<float> {
  __device__ static float4 load(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
  __device__ static void store(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
};
template <>
struct Vec4<__nv_bfloat16> {
  __device__ static float4 load(const __nv_bfloat16* p) {
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
  __device__ static void store(__nv_bfloat16* p, float4 v) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
  }
};

// A group of GS lanes per pixel (GS a power of two dividing 32), each lane holding V four-channel
// vectors (C = 4 * GS * V), so a warp covers 32 / GS consecutive pixels with every lane busy and
// each warp-wide access touches 512 contiguous bytes.  Sum of squares: per lane in a fixed order,
// then a shuffle tree inside the group.
template <typename Tin, typename Tout, int V>
__global__ void __launch_bounds__(256) rms_norm_kernel(const Tin* __restrict__ x, Tout* __restrict__ y,
                                                       Tout* __restrict__ y_raw, long long pixels, int C, int gs,
                                                       const float* __restrict__ gamma, int silu) {
  pdl_wait();   // the previous kernel on the stream has finished (programmatic launch)
  const int lane = threadIdx.x & 31;
  const int j = lane & (gs - 1);          // position in the group
  const int ppw = 32 / gs;                // pixels per warp step
  const long long warp_id = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const float sc = sqrtf(static_cast<float>(C));
  float4 gm[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const float* gp = gamma + 4 * (j + gs * i);
    gm[i] = make_float4(__ldg(gp), __ldg(gp + 1), __ldg(gp + 2), __ldg(gp + 3));
  }
  for (long long p0 = warp_id * ppw; p0 < pixels; p0 += nwarps * ppw) {
    const long long pix = p0 + lane / gs;
    const bool ok = pix < pixels;
    float4 v[V];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      v[i] = ok ? Vec4<Tin>::load(x + pix * C + 4 * (j + gs * i)) : make_float4(0.f, 0.f, 0.f, 0.f);
      ss = fmaf(v[i].x, v[i].x, ss);
      ss = fmaf(v[i].y, v[i].y, ss);
      ss = fmaf(v[i].z, v[i].z, ss);
      ss = fmaf(v[i].w, v[i].w, ss);
    }
    for (int off = 1; off < gs; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = sc / fmaxf(sqrtf(ss), 1e-12f);
    if (ok) {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const long long e = pix * C + 4 * (j + gs * i);
        if (y_raw != nullptr) Vec4<Tout>::store(y_raw + e, v[i]);
        float4 o;
        o.x = v[i].x * inv * gm[i].x;
        o.y = v[i].y * inv * gm[i].y;
        o.z = v[i].z * inv * gm[i].z;
        o.w = v[i].w * inv * gm[i].w;
        if (silu) {
          o.x = silu_f(o.x);
          o.y = silu_f(o.y);
          o.z = silu_f(o.z);
          o.w = silu_f(o.w);
        }
        Vec4<Tout>::store(y + e, o);
      }
    }
  }
}

int sm_count() {
  static const int n = [] {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
      sms = 1;
    return sms;
  }();
  return n;
}

// Blocks of `threads` that are resident on one SM at once for `kernel` (its registers decide).
template <typename KernelT>
int blocks_per_sm(KernelT kernel, int threads) {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, 0) != cudaSuccess || occ < 1) occ = 1;
  return occ;
}

// Grid for a grid-stride loop over `work` items: no more blocks than are resident at once, so
// every block loops over an equal share and no partial second wave runs at low occupancy.
int grid_for(long long work, int threads, int resident_per_sm) {
  const long long b = (work + threads - 1) / threads;
  const long long cap = static_cast<long long>(sm_count()) * resident_per_sm;
  return static_cast<int>(b < cap ? (b < 1 ? 1 : b) : cap);
}

}  // namespace

cudaError_t launch_gn_partials(int dtype, const void* x, int B, int rows, int W, int C, int G, int chunk_rows,
                               GnPartial* part, cudaStream_t stream) {
  if (C % 8 != 0 || C / 8 > kGnThreads || C % G != 0 || chunk_rows < 1) return cudaErrorInvalidValue;
  const int n_chunks = (rows + chunk_rows - 1) / chunk_rows;
  dim3 grid(n_chunks, B);
  const size_t smem = kGnThreads * 24 * sizeof(float);
  if (dtype == kBF16)
    launch_pdl(gn_partials_kernel<__nv_bfloat16>, grid, kGnThreads, smem, stream, 
        static_cast<const __nv_bfloat16*>(x), rows, W, C, G, chunk_rows, n_chunks, part);
  else
    launch_pdl(gn_partials_kernel<float>, grid, kGnThreads, smem, stream, static_cast<const float*>(x), rows, W, C, G,
                                                                  chunk_rows, n_chunks, part);
  return cudaGetLastError();
}

cudaError_t launch_gn_finalize(const GnPartial* part, int B, int n_chunks, int C, int G, const float* gamma,
                               const float* beta, float eps, float* scale, float* shift, cudaStream_t stream) {
  launch_pdl(gn_finalize_kernel, B * G, kFinThreads, 0, stream, part, B, n_chunks, C, G, gamma, beta, eps, scale, shift);
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
void gn_apply_t(const void* x, void* y, void* y_raw, long long nvec, long long vps, int C, const float* scale,
                const float* shift, int silu, cudaStream_t stream) {
  const int threads = 256;
  const int vpp = C / 8;
  const int vpp_log2 = (vpp & (vpp - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(vpp)) : -1;
  static const int occ = blocks_per_sm(gn_apply_kernel<Tin, Tout>, threads);
  if (nvec < (8LL << 20)) {
    // tensors of the small layers (input mostly still in L2): one 1024-thread CTA per SM starts and
    // drains faster than five 256-thread ones (measured 2.161 -> 2.127 ms for the 1024x1024 decode's
    // GroupNorms); the kernel is grid-stride, so the result does not depend on the grid
    launch_pdl(gn_apply_kernel<Tin, Tout>, sm_count(), 1024, 0, stream, static_cast<const Tin*>(x),
               static_cast<Tout*>(y), static_cast<Tout*>(y_raw), static_cast<uint32_t>(nvec),
               static_cast<uint32_t>(vps), C, vpp_log2, scale, shift, silu);
    return;
  }
  launch_pdl(gn_apply_kernel<Tin, Tout>, grid_for(nvec, threads, occ), threads, 0, stream, 
      static_cast<const Tin*>(x), static_cast<Tout*>(y), static_cast<Tout*>(y_raw), static_cast<uint32_t>(nvec),
      static_cast<uint32_t>(vps), C, vpp_log2, scale, shift, silu);
}

cudaError_t launch_gn_apply(int in_dtype, int out_dtype, const void* x, void* y, void* y_raw,
                            long long pixels_per_sample, int B, int C, const float* scale, const float* shift,
                            int silu, cudaStream_t stream) {
  if (C % 8 != 0) return cudaErrorInvalidValue;
  const long long vps = pixels_per_sample * (C / 8);
  if ((long long)B * vps >= (1LL << 31)) return cudaErrorInvalidValue;   // 32-bit vector indices
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

template <typename Tin, typename Tout, int V>
void rms_launch(const Tin* x, Tout* y, Tout* y_raw, long long warps, long long pixels, int C, int gs,
                const float* gamma, int silu, cudaStream_t stream) {
  const int threads = 256;
  static const int occ = blocks_per_sm(rms_norm_kernel<Tin, Tout, V>, threads);
  launch_pdl(rms_norm_kernel<Tin, Tout, V>, grid_for(warps * 32, threads, occ), threads, 0, stream, x, y, y_raw, pixels, C, gs,
                                                                                            gamma, silu);
}

template <typename Tin, typename Tout>
void rms_t(const void* x, void* y, void* y_raw, long long pixels, int C, const float* gamma, int silu,
           cudaStream_t stream) {
  // lanes per pixel: the largest power of two <= 32 dividing C / 4, leaving at most 8 vectors per lane
  const int nv4 = C / 4;
  int gs = 32;
  while (nv4 % gs != 0) gs >>= 1;
  const int v = nv4 / gs;
  const long long warps = (pixels + (32 / gs) - 1) / (32 / gs);
  const Tin* xi = static_cast<const Tin*>(x);
  Tout* yo = static_cast<Tout*>(y);
  Tout* yr = static_cast<Tout*>(y_raw);
  switch (v) {
    case 1: rms_launch<Tin, Tout, 1>(xi, yo, yr, warps, pixels, C, gs, gamma, silu, stream); break;
    case 2: rms_launch<Tin, Tout, 2>(xi, yo, yr, warps, pixels, C, gs, gamma, silu, stream); break;
    case 3: rms_launch<Tin, Tout, 3>(xi, yo, yr, warps, pixels, C, gs, gamma, silu, stream); break;
    case 4: rms_launch<Tin, Tout, 4>(xi, yo, yr, warps, pixels, C, gs, gamma, silu, stream); break;
    case 5: rms_launch<Tin, Tout, 5>(xi, yo, yr, warps, pixels, C, gs, gamma, silu, stream); break;
    case 6: rms_launch<Tin, Tout, 6>(xi, yo, yr, warps, pixels, C, gs, gamma, silu, stream); break;
    case 7: rms_launch<Tin, Tout, 7>(xi, yo, yr, warps, pixels, C, gs, gamma, silu, stream); break;
    default: rms_launch<Tin, Tout, 8>(xi, yo, yr, warps, pixels, C, gs, gamma, silu, stream); break;
  }
}

cudaError_t launch_rms_norm(int in_dtype, int out_dtype, const void* x, void* y, void* y_raw, long long pixels,
                            int C, const float* gamma, int silu, cudaStream_t stream) {
  if (C % 8 != 0 || C > 512) return cudaErrorInvalidValue;   // C / 4 = (lanes per pixel) x (vectors <= 8)
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
