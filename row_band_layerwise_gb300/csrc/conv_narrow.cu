// Tensor-core 3x3 (and causal 3x3x3) convolution for very few output channels (the
// decoder's final conv: 3 output channels).
//
// With C_out = 3 a channel-major tile would waste 125 of 128 MMA rows and a
// pixel-major tile with N = C_out reruns the same activation operand nine times
// for a 16-wide product.  Here the kernel row dy moves into N instead:
//   Y[s][x][dy * C_out + co] = sum_{dt, dx, ci} W[co][dt][dy][dx][ci] * in[t + dt][y0 - 1 + s][x + dx][ci]
// for every staged input row s, so one MMA (M = 128 pixels, N = 16 >= 3 * C_out,
// K = 16 channels) serves all three kernel rows, dx and the causal frames stay in
// K (the staged rows are read through descriptors shifted by whole pixels, as in
// the channel-major halo kernel), and the epilogue forms each output row from the
// three staged rows around it:
//   out[y0 + r][x][co] = bias[co] + sum_dy Y[r + dy][x][dy * C_out + co],
// which stays inside one TMEM lane (one pixel).  Halo rows of neighbouring bands are
// read in place and the global-edge zero padding comes from the TMA unit's
// out-of-bounds fill ("VAEP：VAE 并行解码", 卷积：交换边界行).
//
// Roles (224 threads): warp 0 TMA producer, warp 1 MMA issuer + TMEM owner, warp 2
// waiter (polls the stage barriers and releases the MMA warp through a named barrier),
// warps 3..6 epilogue (one TMEM lane quarter each).  Persistent over tiles of R output
// rows x 128 pixels, two TMEM accumulator buffers.  Every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "conv.h"
#include "kernels.h"
#include "ptx.cuh"
#include "tma_host.h"
#include "launch.h"

namespace vd {

namespace {

constexpr int kThreadsN = 224;
constexpr int kRowsN = 6;          // output rows per tile (R + 2 = 8 staged rows, 128 TMEM columns)
constexpr int kNN = 16;            // MMA N: 3 kernel rows x C_out, padded
constexpr int kCoutN = 3;          // output channels (the decoder's RGB output)
constexpr int kPipeBytesN = 200 * 1024;

struct NarrowParams {
  CUtensorMap tmX;                 // activations 5D (Cin, W, H, T, B), box (BK, half, 1, 1, 1)
  CUtensorMap tmW;                 // narrow weights 3D (Cin, kt * 3, 16), box (BK, 1, 16)
  ConvGeom g;
  int kt;                          // causal frames (1 for 2D)
  int half;                        // pixels per staging box (two boxes per staged row)
  int tiles_x, tiles_y, ntiles, n_kchunks;
  uint32_t row_bytes, x_stage_bytes, w_dx_bytes, stage_bytes, stage_stride;
  const float* bias;
  void* out;
  int* status;
};

template <int BK>
struct SwzN {
  static constexpr uint32_t kSbo = BK * 2 * 8;
  static constexpr uint32_t kMode = BK == 64 ? 2u : (BK == 32 ? 4u : 6u);
};

__device__ __forceinline__ bool handoff_n(bool aborted) { return bar_sync_or(1, 64, aborted); }

template <int BK>
__global__ void __launch_bounds__(kThreadsN, 1) conv_narrow_kernel(const __grid_constant__ NarrowParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[2], empty_bar[2];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const ConvGeom& g = p.g;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nchunk = p.kt * p.n_kchunks;   // (frame, channel chunk) stages per tile
  constexpr int kAcc = (kRowsN + 2) * kNN;  // TMEM columns per accumulator buffer

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmX);
    tma_prefetch_desc(&p.tmW);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 2 * kAcc);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the previous kernel on the stream has finished and its writes are visible from here on
  pdl_wait();
  const uint32_t tmem = tmem_base_sh;

  // tile t -> (tx, ty, frame, sample)
  auto tile_of = [&](int t, int& x0, int& y0, int& tt, int& bb) {
    x0 = (t % p.tiles_x) * 128;
    t /= p.tiles_x;
    y0 = (t % p.tiles_y) * kRowsN;
    t /= p.tiles_y;
    tt = t % g.T;
    bb = t / g.T;
  };

  if (warp == 0) {
    // ---- TMA producer: per stage the 8 staged rows of one (frame, channel chunk) and its weights
    if (lane == 0) {
      int gs = 0;   // stages issued so far
      for (int t = blockIdx.x; t < p.ntiles && !abort_flag; t += gridDim.x) {
        int x0, y0, tt, bb;
        tile_of(t, x0, y0, tt, bb);
        for (int c = 0; c < nchunk && !abort_flag; ++c, ++gs) {
          const int dti = c / p.n_kchunks;
          const int kc = c - dti * p.n_kchunks;
          const int dt = dti - (p.kt - 1);
          const int s = gs & 1;
          if (gs >= 2 && !mbar_wait(&empty_bar[s], (static_cast<uint32_t>(gs >> 1) & 1u) ^ 1u, p.status,
                                    kErrTimeoutEmpty, &abort_flag))
            break;
          mbar_arrive_expect_tx(&full_bar[s], p.stage_bytes);
          uint8_t* xs = smem + s * p.stage_stride;
          uint8_t* ws = xs + p.x_stage_bytes;
          for (int rb = 0; rb < kRowsN + 2; ++rb) {
            tma_load_5d(xs + rb * p.row_bytes, &p.tmX, &full_bar[s], kc * BK, x0 - 1, y0 - 1 + rb, tt + dt, bb);
            tma_load_5d(xs + rb * p.row_bytes + p.half * BK * 2, &p.tmX, &full_bar[s], kc * BK, x0 - 1 + p.half,
                        y0 - 1 + rb, tt + dt, bb);
          }
          for (int dx = 0; dx < 3; ++dx)
            tma_load_3d(ws + dx * p.w_dx_bytes, &p.tmW, &full_bar[s], kc * BK, dti * 3 + dx, 0);
        }
      }
      if (abort_flag) {
        // let the copies already issued land before the CTA exits
        for (int i = max(0, gs - 2); i < gs; ++i) mbar_drain(&full_bar[i & 1], static_cast<uint32_t>(i >> 1) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---- waiter: one hand-off per stage (the first of a tile also covers its accumulator buffer)
    int gs = 0, it = 0;
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
      const int buf = it & 1;
      for (int c = 0; c < nchunk; ++c, ++gs) {
        bool ab = false;
        if (lane == 0) {
          if (!abort_flag) {
            if (c == 0 && it >= 2)
              mbar_wait(&acc_empty[buf], (static_cast<uint32_t>(it >> 1) & 1u) ^ 1u, p.status, kErrTimeoutEmpty,
                        &abort_flag);
            mbar_wait(&full_bar[gs & 1], static_cast<uint32_t>(gs >> 1) & 1u, p.status, kErrTimeoutFull,
                      &abort_flag);
          }
          ab = abort_flag != 0;
        }
        __syncwarp();
        handoff_n(ab);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: per stage, every staged row s x 3 pixel shifts x BK/16 channel steps
    const uint32_t idesc = idesc_bf16_f32(128, kNN);
    const uint64_t dX0 = smem_desc_kmajor(smem_u32(smem), SwzN<BK>::kSbo, SwzN<BK>::kMode);
    const uint64_t dW0 = smem_desc_kmajor(smem_u32(smem) + p.x_stage_bytes, SwzN<BK>::kSbo, SwzN<BK>::kMode);
    const uint32_t stage16 = p.stage_stride >> 4, row16 = p.row_bytes >> 4;
    const uint32_t wdx16 = p.w_dx_bytes >> 4;
    int gs = 0, it = 0;
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
      const int buf = it & 1;
      const uint32_t dcol = tmem + static_cast<uint32_t>(buf * kAcc);
      for (int c = 0; c < nchunk; ++c, ++gs) {
        const int s = gs & 1;
        const bool aborted = handoff_n(false);
        tc_fence_after();
        if (lane == 0) {
          if (!aborted) {
            const uint64_t dXs = dX0 + static_cast<uint64_t>(s * stage16);
            const uint64_t dWs = dW0 + static_cast<uint64_t>(s * stage16);
#pragma unroll
            for (int dx = 0; dx < 3; ++dx)
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
#pragma unroll
                for (int r = 0; r < kRowsN + 2; ++r)
                  tc_mma_bf16(dcol + static_cast<uint32_t>(r * kNN), dXs + r * row16 + dx * (BK * 2 / 16) + 2 * k,
                              dWs + dx * wdx16 + 2 * k, idesc, (c | dx | k) != 0 ? 1u : 0u);
          }
          tc_commit(&empty_bar[s]);
          if (c == nchunk - 1) tc_commit(&acc_full[buf]);
        }
        __syncwarp();
      }
    }
    // every MMA issued has completed before the CTA releases TMEM (also after a timeout)
    if (lane == 0) {
      tc_commit(&mma_done);
      mbar_drain(&mma_done, 0);
    }
    __syncwarp();
  } else {
    // ---- epilogue (warps 3..6): TMEM lane = pixel; out[y0 + r] = bias + sum_dy Y[r + dy][dy * Cout + co]
    const int q = warp & 3;
    constexpr int cout = kCoutN;
    int it = 0;
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
      int x0, y0, tt, bb;
      tile_of(t, x0, y0, tt, bb);
      const int buf = it & 1;
      const int x = x0 + q * 32 + lane;
      const bool ok = mbar_wait(&acc_full[buf], static_cast<uint32_t>(it >> 1) & 1u, p.status, kErrTimeoutAccum,
                                &abort_flag);
      tc_fence_after();
      if (!__all_sync(0xffffffffu, ok && !abort_flag)) break;
      const uint32_t lane_addr = tmem + static_cast<uint32_t>(buf * kAcc) + (static_cast<uint32_t>(q * 32) << 16);
      // Y of the 8 staged rows for this pixel (16 columns each)
      float yv[kRowsN + 2][kNN];
#pragma unroll
      for (int s = 0; s < kRowsN + 2; ++s) {
        uint32_t rr[16];
        tmem_ld_16x_32x32b(lane_addr + static_cast<uint32_t>(s * kNN), rr);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < kNN; ++j) yv[s][j] = __uint_as_float(rr[j]);
      }
      // the accumulator buffer is free once its values are in registers
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
#pragma unroll
      for (int r = 0; r < kRowsN; ++r) {
        const int y = y0 + r;
        if (y >= g.H || x >= g.W) continue;
#pragma unroll
        for (int co = 0; co < cout; ++co) {
          const float v = (p.bias != nullptr ? __ldg(p.bias + co) : 0.f) + yv[r][co] + yv[r + 1][cout + co] +
                          yv[r + 2][2 * cout + co];
          long long e;
          if (g.out_chfirst)
            e = (((static_cast<long long>(bb) * g.oC + co) * g.oT + tt) * g.oH + y) * static_cast<long long>(g.oW) + x;
          else
            e = (((static_cast<long long>(bb) * g.oT + tt) * g.oH + y) * static_cast<long long>(g.oW) + x) * g.oC + co;
          if (g.out_f32)
            static_cast<float*>(p.out)[e] = v;
          else
            static_cast<__nv_bfloat16*>(p.out)[e] = __float2bfloat16_rn(v);
        }
      }
      __syncwarp();
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kAcc);
  }
}

int round_up_n(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace

// 3x3 spatial taps in the standard order (kernel row, then column), optionally times causal
// frames; 3 output channels (3 kernel rows x 3 fit the 16-wide N); no upsample phases or
// temporal interleave (the caller passes no residual).
bool conv_narrow_applicable(const ConvGeom& g) {
  if (g.nphase != 1 || g.time_up_c > 0) return false;
  if (g.ntaps != 9 && g.ntaps != 27) return false;
  if (g.Cout != kCoutN) return false;
  if (g.Cin % 16 != 0) return false;
  if (g.osx != 1 || g.osy != 1) return false;
  const int kt = g.ntaps / 9;
  for (int k = 0; k < g.ntaps; ++k) {
    const ConvTap t = g.taps[0][k];
    const int s = k / 9, i = (k % 9) / 3, j = k % 3;
    if (t.dt != s - (kt - 1) || t.dy != i - 1 || t.dx != j - 1 || t.wtap != k) return false;
  }
  return true;
}

cudaError_t launch_conv_narrow(const ConvGeom& g, const void* in, const void* w_narrow, const float* bias,
                               void* out, int* status, cudaStream_t stream, const char** why) {
  *why = nullptr;
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return cudaErrorNotSupported;
  }
  NarrowParams p;
  std::memset(&p, 0, sizeof(p));
  p.g = g;
  p.kt = g.ntaps / 9;
  p.half = round_up_n(128 + 2, 16) / 2;   // 72: two boxes cover the 130 pixels a 128-pixel tile reads
  p.tiles_x = (g.W + 127) / 128;
  p.tiles_y = (g.H + kRowsN - 1) / kRowsN;
  const long long ntiles = (long long)g.B * g.T * p.tiles_y * p.tiles_x;
  if (ntiles <= 0) return cudaSuccess;
  if (ntiles > 0x7fffffffLL) {
    *why = "grid too large";
    return cudaErrorInvalidValue;
  }
  p.ntiles = static_cast<int>(ntiles);
  int bk = 0;
  for (int cand : {64, 32, 16}) {
    if (g.Cin % cand != 0) continue;
    const int row = 2 * p.half * cand * 2;
    const int stage = round_up_n((kRowsN + 2) * row + 3 * kNN * cand * 2, 1024);
    if (2 * stage <= kPipeBytesN) {
      bk = cand;
      break;
    }
  }
  if (bk == 0) {
    *why = "no narrow conv tile fits shared memory";
    return cudaErrorInvalidValue;
  }
  p.n_kchunks = g.Cin / bk;
  p.row_bytes = static_cast<uint32_t>(2 * p.half * bk * 2);
  p.x_stage_bytes = static_cast<uint32_t>((kRowsN + 2) * p.row_bytes);
  p.w_dx_bytes = static_cast<uint32_t>(kNN * bk * 2);
  p.stage_bytes = p.x_stage_bytes + 3 * p.w_dx_bytes;   // bytes the TMA unit delivers per stage
  p.bias = bias;
  p.out = out;
  p.status = status;
  p.stage_stride = static_cast<uint32_t>(round_up_n(static_cast<int>(p.stage_bytes), 1024));
  const cuuint32_t ones[5] = {1, 1, 1, 1, 1};
  {
    const cuuint64_t dims[5] = {(cuuint64_t)g.Cin, (cuuint64_t)g.W, (cuuint64_t)g.H, (cuuint64_t)g.T,
                                (cuuint64_t)g.B};
    const cuuint64_t strides[4] = {dims[0] * 2, dims[0] * dims[1] * 2, dims[0] * dims[1] * dims[2] * 2,
                                   dims[0] * dims[1] * dims[2] * dims[3] * 2};
    const cuuint32_t box[5] = {(cuuint32_t)bk, (cuuint32_t)p.half, 1, 1, 1};
    if (enc(&p.tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(in), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "narrow conv activation tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)g.Cin, (cuuint64_t)(p.kt * 3), (cuuint64_t)kNN};
    const cuuint64_t strides[2] = {dims[0] * 2, dims[0] * dims[1] * 2};
    const cuuint32_t box[3] = {(cuuint32_t)bk, 1, (cuuint32_t)kNN};
    if (enc(&p.tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w_narrow), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "narrow conv weight tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  const size_t smem = 2 * (size_t)p.stage_stride + 1024;   // two stages at stage_stride spacing
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(std::min<long long>(ntiles, std::max(1, sms)));
  switch (bk) {
    case 64:
      e = cudaFuncSetAttribute(conv_narrow_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) launch_pdl(conv_narrow_kernel<64>, grid, kThreadsN, smem, stream, p);
      break;
    case 32:
      e = cudaFuncSetAttribute(conv_narrow_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) launch_pdl(conv_narrow_kernel<32>, grid, kThreadsN, smem, stream, p);
      break;
    default:
      e = cudaFuncSetAttribute(conv_narrow_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) launch_pdl(conv_narrow_kernel<16>, grid, kThreadsN, smem, stream, p);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

VD_WAIT_LIMIT_SETTER(set_wait_limit_conv_narrow)

}  // namespace vd
