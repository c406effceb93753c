// Channel-major GEMM on tcgen05 tensor cores:  D[m, n] = sum_k A[m, k] * B[n, k],
// stored at out[n * ldo + m].
//
// Used for the attention products (scores = keys x queries, probabilities x
// values with the sum over keys split across tiles) and the 1x1 convolutions.  A
// tile is 128 (m) x NB (n, up to 256); every TMEM lane is one m, so each epilogue
// store instruction writes 32 consecutive m of one n: coalesced.  The kernel is
// persistent (one CTA per SM, tiles dealt round-robin) with two accumulator
// buffers in TMEM: the epilogue of tile i overlaps the MMAs of tile i + 1, and the
// producer streams the next tile's K chunks while the current one finishes.
//
// Roles (352 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA issuer,
// warp 2 stage waiter, warps 3..10 epilogue.  The waiter polls the stage
// mbarriers and hands each landed stage to the MMA warp through one hardware
// named barrier that both warps sync on once per stage, so the MMA-issuing thread
// never polls shared memory while the tensor pipe is busy (it sleeps in the
// barrier instead), and the waiter polls stage i+1 while the MMAs of stage i run.
// Both warps pass the barrier exactly once per stage, also after a timeout, so
// neither can block on it.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "kernels.h"
#include "ptx.cuh"
#include "tma_host.h"
#include "launch.h"

namespace vd {

namespace {

constexpr int kGThreads = 352;
constexpr int kGMaxStages = 4;
constexpr int kGBK = 64;   // K chunk (128B swizzle)
constexpr int kGCols = 16; // accumulator columns per epilogue step
constexpr int kGEpiWarps = 8;
constexpr int kGStageO = 128 * 32 * 4;   // one output staging buffer (32 columns of fp32)

struct GemmParams {
  CUtensorMap tmA;   // (K, M) box (64, 128)
  CUtensorMap tmB;   // (K, N) box (64, NB)
  CUtensorMap tmO;   // output (M, N, splits) box (128, 32, 1), when tma_out
  int tma_out;       // 1: the epilogue stages 32-column chunks in shared memory and stores them with TMA
  int M, N, K, NB, n_mtiles, n_ntiles, nk, splits, nb, ntiles;
  uint32_t a_stage, b_stage, acc_cols, tmem_cols;
  void* out;
  long long ldo, split_stride;
  int out_f32, res_f32;   // output fp32, else bf16
  const float* bias_m;
  const float* bias_n;
  const float* scale_n;
  float scale;
  const void* residual;
  __nv_bfloat16* out2;
  int* status;
};

struct GTile {
  int m0, n0, split, k_begin, nks;
};

// Tile t: m tile fastest (tiles running at the same time share their B rows), then n tile, then split.
__device__ __forceinline__ GTile gemm_tile(const GemmParams& p, int t) {
  GTile d;
  const int mt = t % p.n_mtiles;
  t /= p.n_mtiles;
  const int nt = t % p.n_ntiles;
  d.split = t / p.n_ntiles;
  d.m0 = mt * 128;
  d.n0 = nt * p.NB;
  d.k_begin = static_cast<int>((long long)d.split * p.nk / p.splits);
  d.nks = static_cast<int>((long long)(d.split + 1) * p.nk / p.splits) - d.k_begin;
  return d;
}

// Named barrier 1, shared by the waiter warp and the MMA warp (64 threads); returns true when the
// waiter saw the abort flag raised.
__device__ __forceinline__ bool stage_handoff(bool aborted) { return bar_sync_or(1, 64, aborted); }

// Named barrier `id` over the 128 threads of one epilogue half (four warps).
__device__ __forceinline__ void half_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }
// The same barrier, returning the AND of `v` over its 128 threads.
__device__ __forceinline__ bool half_and(int id, bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred pv, pr;\n\tsetp.ne.s32 pv, %1, 0;\n\tbar.red.and.pred pr, %2, 128, pv;\n\t"
      "selp.s32 %0, 1, 0, pr;\n\t}"
      : "=r"(r)
      : "r"(static_cast<int>(v)), "r"(id)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kGThreads, 1) gemm_cm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kGMaxStages], empty_bar[kGMaxStages];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + p.nb * p.a_stage;
  uint8_t* smO = smB + p.nb * p.b_stage;   // two 16 KB output staging buffers (tma_out)

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.nb; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kGEpiWarps);
    }
    mbar_init(&mma_done, 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
    if (p.tma_out) tma_prefetch_desc(&p.tmO);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the previous kernel on the stream has finished and its writes are visible from here on
  pdl_wait();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ---- TMA producer: K chunks of every tile of this CTA, through the stage ring
    if (lane == 0) {
      const uint32_t tx = p.a_stage + static_cast<uint32_t>(p.NB * kGBK * 2);
      int g = 0;   // stages issued so far
      for (int t = blockIdx.x; t < p.ntiles && !abort_flag; t += gridDim.x) {
        const GTile d = gemm_tile(p, t);
        for (int i = 0; i < d.nks && !abort_flag; ++i, ++g) {
          const int s = g % p.nb;
          if (g >= p.nb && !mbar_wait(&empty_bar[s], (static_cast<uint32_t>(g / p.nb) & 1u) ^ 1u, p.status,
                                      kErrTimeoutEmpty, &abort_flag))
            break;
          mbar_arrive_expect_tx(&full_bar[s], tx);
          const int kc = (d.k_begin + i) * kGBK;
          tma_load_3d(smA + s * p.a_stage, &p.tmA, &full_bar[s], kc, d.m0, 0);
          tma_load_3d(smB + s * p.b_stage, &p.tmB, &full_bar[s], kc, d.n0, 0);
        }
      }
      if (abort_flag) {
        // let the copies already issued land before the CTA exits
        for (int i = max(0, g - p.nb); i < g; ++i) mbar_drain(&full_bar[i % p.nb], static_cast<uint32_t>(i / p.nb) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---- waiter: one hand-off per stage of every tile, always (also after an abort); the first of a
    // tile also covers the tile's accumulator buffer
    int g = 0, it = 0;
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
      const int nks = gemm_tile(p, t).nks;
      const int buf = it & 1;
      for (int i = 0; i < nks; ++i, ++g) {
        bool ab = false;
        if (lane == 0) {
          if (!abort_flag) {
            if (i == 0 && it >= 2)
              mbar_wait(&acc_empty[buf], (static_cast<uint32_t>(it >> 1) & 1u) ^ 1u, p.status, kErrTimeoutEmpty,
                        &abort_flag);
            mbar_wait(&full_bar[g % p.nb], static_cast<uint32_t>(g / p.nb) & 1u, p.status, kErrTimeoutFull,
                      &abort_flag);
          }
          ab = abort_flag != 0;
        }
        __syncwarp();
        stage_handoff(ab);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: tile i accumulates into TMEM buffer i & 1; same stage sequence as the waiter
    const uint32_t idesc = idesc_bf16_f32(128, p.NB);
    // base descriptors; a stage / K step only adds to the start-address field (16-byte units)
    const uint64_t dA0 = smem_desc_kmajor(smem_u32(smA), 1024, 2);
    const uint64_t dB0 = smem_desc_kmajor(smem_u32(smB), 1024, 2);
    const uint32_t a_stage16 = p.a_stage >> 4, b_stage16 = p.b_stage >> 4;
    int g = 0, it = 0, s = 0;
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
      const int nks = gemm_tile(p, t).nks;
      const int buf = it & 1;
      const uint32_t dbase = tmem + static_cast<uint32_t>(buf) * p.acc_cols;
      for (int i = 0; i < nks; ++i, ++g) {
        const bool aborted = stage_handoff(false);
        tc_fence_after();
        if (lane == 0) {
          if (!aborted) {
            const uint64_t da = dA0 + static_cast<uint64_t>(s * a_stage16);
            const uint64_t db = dB0 + static_cast<uint64_t>(s * b_stage16);
#pragma unroll
            for (int k = 0; k < kGBK / 16; ++k) tc_mma_bf16(dbase, da + 2 * k, db + 2 * k, idesc, (i | k) != 0 ? 1u : 0u);
          }
          tc_commit(&empty_bar[s]);
        }
        __syncwarp();
        s = (s + 1 == p.nb) ? 0 : s + 1;
      }
      if (lane == 0) tc_commit(&acc_full[buf]);
      __syncwarp();
    }
    // every MMA issued has completed before the CTA releases TMEM (also after a timeout)
    if (lane == 0) {
      tc_commit(&mma_done);
      mbar_drain(&mma_done, 0);
    }
    __syncwarp();
  } else {
    // ---- epilogue warps 3..10: quarter q of the TMEM lanes, half `sub` of the column chunks
    const int q = warp & 3;
    const int sub = (warp - 3) >> 2;
    if (p.tma_out) {
      // 32-column chunks: the four warps of a half stage [32 n][128 m] in shared memory, then
      // one thread stores the chunk with TMA (rows and columns outside the output are clipped)
      const int bar_id = 2 + sub;
      const bool leader = q == 0 && lane == 0;
      const bool per_col = p.scale_n != nullptr || p.bias_n != nullptr;
      uint8_t* stg = smO + sub * kGStageO;
      int it = 0;
      for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
        const GTile d = gemm_tile(p, t);
        const int buf = it & 1;
        const int ml = q * 32 + lane;
        const int m = d.m0 + ml;
        const bool mvalid = m < p.M;
        const float bm = (p.bias_m != nullptr && mvalid) ? p.bias_m[m] : 0.f;
        const bool ok = mbar_wait(&acc_full[buf], static_cast<uint32_t>(it >> 1) & 1u, p.status, kErrTimeoutAccum,
                                  &abort_flag);
        tc_fence_after();
        if (!half_and(bar_id, ok && !abort_flag)) break;   // the same decision in all four warps
        const uint32_t lane_addr =
            tmem + static_cast<uint32_t>(buf) * p.acc_cols + (static_cast<uint32_t>(q * 32) << 16);
        for (int c0 = sub * 32; c0 < p.NB && d.nks > 0; c0 += 64) {
          const int nvalid = min(32, p.N - (d.n0 + c0));
          if (nvalid <= 0) break;   // uniform across the half
          uint32_t rr[32];
          tmem_ld_32x32b_x32(lane_addr + static_cast<uint32_t>(c0), rr);
          tmem_ld_wait();
          float v[32];
          if (per_col) {
            // column j's scale and bias: lane j loads them, a shuffle hands them to every lane
            const float lsc = (lane < nvalid && p.scale_n != nullptr) ? __ldg(p.scale_n + d.n0 + c0 + lane) : 1.f;
            const float lbn = (lane < nvalid && p.bias_n != nullptr) ? __ldg(p.bias_n + d.n0 + c0 + lane) : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              v[j] = fmaf(__uint_as_float(rr[j]), p.scale * __shfl_sync(0xffffffffu, lsc, j),
                          bm + __shfl_sync(0xffffffffu, lbn, j));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = fmaf(__uint_as_float(rr[j]), p.scale, bm);
          }
          if (p.residual != nullptr && mvalid) {
            // all 32 loads issued before the first use
            const long long e0 = static_cast<long long>(d.n0 + c0) * p.ldo + m;
            float rv[32];
            if (p.res_f32) {
              const float* rp = static_cast<const float*>(p.residual) + e0;
#pragma unroll
              for (int j = 0; j < 32; ++j) rv[j] = (j < nvalid) ? __ldg(rp + j * p.ldo) : 0.f;
            } else {
              const __nv_bfloat16* rp = static_cast<const __nv_bfloat16*>(p.residual) + e0;
#pragma unroll
              for (int j = 0; j < 32; ++j) rv[j] = (j < nvalid) ? __bfloat162float(rp[j * p.ldo]) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += rv[j];
          }
          // the staging buffer is free once the previous store from it has read it
          if (leader) bulk_wait_group_read0();
          half_sync(bar_id);
          if (p.out_f32) {
            float* sp = reinterpret_cast<float*>(stg) + ml;
#pragma unroll
            for (int j = 0; j < 32; ++j) sp[j * 128] = v[j];
          } else {
            __nv_bfloat16* sp = reinterpret_cast<__nv_bfloat16*>(stg) + ml;
#pragma unroll
            for (int j = 0; j < 32; ++j) sp[j * 128] = __float2bfloat16_rn(v[j]);
          }
          fence_proxy_async_smem();   // make the staged values visible to the TMA unit
          half_sync(bar_id);
          if (leader) {
            tma_store_3d(&p.tmO, stg, d.m0, d.n0 + c0, d.split);
            bulk_commit_group();
          }
          __syncwarp();
        }
        // hand the accumulator buffer back to the MMA issuer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
      if (leader) bulk_wait_group0();
      __syncwarp();
    } else {
      int it = 0;
      for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
        const GTile d = gemm_tile(p, t);
        const int buf = it & 1;
        const int m = d.m0 + q * 32 + lane;
        const bool mvalid = m < p.M;
        const float bm = (p.bias_m != nullptr && mvalid) ? p.bias_m[m] : 0.f;
        const bool ok = mbar_wait(&acc_full[buf], static_cast<uint32_t>(it >> 1) & 1u, p.status, kErrTimeoutAccum,
                                  &abort_flag);
        tc_fence_after();
        if (!__all_sync(0xffffffffu, ok && !abort_flag)) break;
        const uint32_t lane_addr = tmem + static_cast<uint32_t>(buf) * p.acc_cols + (static_cast<uint32_t>(q * 32) << 16);
        char* outp = static_cast<char*>(p.out) + (p.out_f32 ? 4 : 2) * d.split * p.split_stride;
        for (int c0 = sub * kGCols; c0 < p.NB && d.nks > 0; c0 += 2 * kGCols) {
          const int nvalid = min(kGCols, p.N - (d.n0 + c0));
          if (nvalid <= 0) break;   // uniform across the warp
          uint32_t rr[kGCols];
          tmem_ld_16x_32x32b(lane_addr + static_cast<uint32_t>(c0), rr);
          tmem_ld_wait();
          float v[kGCols];
#pragma unroll
          for (int j = 0; j < kGCols; ++j) {
            const int n = d.n0 + c0 + j;
            float sc = p.scale;
            float bn = 0.f;
            if (j < nvalid) {
              if (p.scale_n != nullptr) sc *= __ldg(p.scale_n + n);
              if (p.bias_n != nullptr) bn = __ldg(p.bias_n + n);
            }
            v[j] = __uint_as_float(rr[j]) * sc + bm + bn;
          }
          const long long e0 = static_cast<long long>(d.n0 + c0) * p.ldo + m;
          if (mvalid) {
            if (p.residual != nullptr) {
              if (p.res_f32) {
                const float* rp = static_cast<const float*>(p.residual) + e0;
#pragma unroll
                for (int j = 0; j < kGCols; ++j)
                  if (j < nvalid) v[j] += rp[j * p.ldo];
              } else {
                const __nv_bfloat16* rp = static_cast<const __nv_bfloat16*>(p.residual) + e0;
#pragma unroll
                for (int j = 0; j < kGCols; ++j)
                  if (j < nvalid) v[j] += __bfloat162float(rp[j * p.ldo]);
              }
            }
            if (p.out_f32) {
              float* op = reinterpret_cast<float*>(outp) + e0;
#pragma unroll
              for (int j = 0; j < kGCols; ++j)
                if (j < nvalid) op[j * p.ldo] = v[j];
            } else {
              __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(outp) + e0;
#pragma unroll
              for (int j = 0; j < kGCols; ++j)
                if (j < nvalid) op[j * p.ldo] = __float2bfloat16_rn(v[j]);
            }
            if (p.out2 != nullptr) {
              __nv_bfloat16* op = p.out2 + e0;
#pragma unroll
              for (int j = 0; j < kGCols; ++j)
                if (j < nvalid) op[j * p.ldo] = __float2bfloat16_rn(v[j]);
            }
          }
          __syncwarp();   // reconverge before the next warp-wide TMEM load
        }
        // hand the accumulator buffer back to the MMA issuer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

int round_up_g(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace

cudaError_t launch_gemm_cm(const GemmArgs& a, int* status, cudaStream_t stream, const char** why) {
  *why = nullptr;
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return cudaErrorNotSupported;
  }
  if (a.M < 1 || a.N < 1 || a.K < 1 || a.splits < 1) return cudaSuccess;
  if ((a.lda % 8) || (a.ldb % 8) || a.lda < a.K || a.ldb < a.K) {
    *why = "GEMM operand rows must be 16-byte aligned and at least K long";
    return cudaErrorInvalidValue;
  }
  if ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) & 15) {
    *why = "GEMM operands must be 16-byte aligned";
    return cudaErrorInvalidValue;
  }
  if (a.splits > 1 && !a.out_f32) {
    *why = "split-K GEMM needs fp32 partial output";
    return cudaErrorInvalidValue;
  }
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.NB = std::min(256, round_up_g(a.N, 16));
  p.n_mtiles = (a.M + 127) / 128;
  p.n_ntiles = (a.N + p.NB - 1) / p.NB;
  p.nk = (a.K + kGBK - 1) / kGBK;
  p.splits = std::min(a.splits, p.nk);
  p.a_stage = 128 * kGBK * 2;
  p.b_stage = static_cast<uint32_t>(round_up_g(p.NB * kGBK * 2, 1024));
  // TMA-stored output: rows 16-byte aligned, no second output copy
  const size_t oes = a.out_f32 ? 4 : 2;
  p.tma_out = a.out2 == nullptr && (reinterpret_cast<uintptr_t>(a.out) % 16) == 0 && (a.ldo * oes) % 16 == 0 &&
              (a.splits <= 1 || (a.split_stride * oes) % 16 == 0) && a.ldo >= a.M;
  // one persistent CTA per SM: a deep stage ring, two accumulator buffers, two output staging buffers
  const int stage_budget = 227 * 1024 - 1024 - 512 - (p.tma_out ? 2 * kGStageO : 0);
  p.nb = std::min(kGMaxStages, static_cast<int>(stage_budget / (p.a_stage + p.b_stage)));
  p.acc_cols = 32;
  while (p.acc_cols < static_cast<uint32_t>(p.NB)) p.acc_cols <<= 1;
  p.tmem_cols = 2 * p.acc_cols;
  p.out = a.out;
  p.ldo = a.ldo;
  p.split_stride = a.split_stride;
  p.out_f32 = a.out_f32;
  p.res_f32 = a.res_f32;
  p.bias_m = a.bias_m;
  p.bias_n = a.bias_n;
  p.scale_n = a.scale_n;
  p.scale = a.scale;
  p.residual = a.residual;
  p.out2 = static_cast<__nv_bfloat16*>(a.out2);
  p.status = status;
  const cuuint32_t ones[3] = {1, 1, 1};
  {
    const cuuint64_t dims[3] = {(cuuint64_t)a.K, (cuuint64_t)a.M, 1};
    const cuuint64_t strides[2] = {(cuuint64_t)a.lda * 2, (cuuint64_t)a.lda * 2 * a.M};
    const cuuint32_t box[3] = {kGBK, 128, 1};
    if (enc(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.A), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "GEMM A tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)a.K, (cuuint64_t)a.N, 1};
    const cuuint64_t strides[2] = {(cuuint64_t)a.ldb * 2, (cuuint64_t)a.ldb * 2 * a.N};
    const cuuint32_t box[3] = {kGBK, (cuuint32_t)p.NB, 1};
    if (enc(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.B), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "GEMM B tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  if (p.tma_out) {
    const cuuint64_t dims[3] = {(cuuint64_t)a.M, (cuuint64_t)a.N, (cuuint64_t)p.splits};
    const cuuint64_t strides[2] = {(cuuint64_t)(a.ldo * oes),
                                   (cuuint64_t)(p.splits > 1 ? a.split_stride * oes : a.ldo * oes * a.N)};
    const cuuint32_t box[3] = {128, 32, 1};
    const CUtensorMapDataType odt = a.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (enc(&p.tmO, odt, 3, a.out, dims,
            strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "GEMM output tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  const size_t smem = (size_t)p.nb * (p.a_stage + p.b_stage) + (p.tma_out ? 2 * kGStageO : 0) + 1024;
  cudaError_t e = cudaFuncSetAttribute(gemm_cm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long ntiles = (long long)p.n_mtiles * p.n_ntiles * p.splits;
  if (ntiles > 0x7fffffffLL) {
    *why = "GEMM has too many tiles";
    return cudaErrorInvalidValue;
  }
  p.ntiles = static_cast<int>(ntiles);
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(std::min<long long>(ntiles, std::max(1, sms)));
  launch_pdl(gemm_cm_kernel, grid, kGThreads, smem, stream, p);
  return cudaGetLastError();
}

VD_WAIT_LIMIT_SETTER(set_wait_limit_gemm_cm)

}  // namespace vd
