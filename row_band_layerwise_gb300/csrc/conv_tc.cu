// Implicit-GEMM convolution on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// One CTA computes a 128-pixel x BN-channel output tile:
//   warp 0      TMA producer: per K step (tap, 64/32/16-channel chunk) loads the
//               shifted 128-pixel activation box and the weight box into a
//               swizzled shared-memory stage.  Out-of-range boxes read zeros,
//               which is the conv's zero padding at the global image edges (and
//               the causal zero frames in time); rows of a neighbouring band are
//               in range and read their real values (the conv halo of
//               "VAEP：VAE 并行解码", section 卷积：交换边界行).
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=BN, K=16) from
//               one thread, accumulating fp32 in TMEM; commits free each stage.
//   warps 2..5  epilogue: tcgen05.ld the accumulator (one TMEM lane per pixel),
//               scale, add bias and residual in fp32, round once, store.
// Every wait is bounded (see ptx.cuh); on timeout the CTA records an error,
// drains its own copies, frees TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdio>
#include <cstring>

#include "conv.h"
#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tma_host.h"
#include "launch.h"

namespace vd {

struct ConvTcParams {
  CUtensorMap tmA;       // activations [B][T][H][W][Cin] as 5D (Cin, W, H, T, B)
  CUtensorMap tmB;       // weights [rows][ntaps_w][Cin] as 3D (Cin, ntaps_w, rows)
  ConvGeom g;
  int BX, BY;            // pixel tile: BY rows x BX columns, BX * BY = 128
  int tiles_x, tiles_y;
  int BN, n_ntiles;
  int n_kchunks, stages;
  uint32_t stage_a_bytes, stage_b_bytes, tmem_cols;
  const float* bias;     // [Cout] or null
  const void* residual;  // channels-last (fp32 or bf16, see g.res_f32), same index as out, or null
  const float* rowscale; // per output pixel (flat grid index), or null
  void* out;
  __nv_bfloat16* out2;   // optional bf16 copy of a channels-last output
  int* status;
};

constexpr int kThreads = 192;
constexpr int kBM = 128;

template <int BK>
struct SwizzleOf {
  // row pitch BK*2 bytes; 8-row swizzle atom
  static constexpr uint32_t kSbo = BK * 2 * 8;
  static constexpr uint32_t kMode = BK == 64 ? 2u : (BK == 32 ? 4u : 6u);
};

template <int BK>
__global__ void __launch_bounds__(kThreads) conv_tc_kernel(const __grid_constant__ ConvTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[8];
  __shared__ __align__(8) uint64_t empty_bar[8];
  __shared__ __align__(8) uint64_t accum_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ float bias_sh[256];

  const ConvGeom& g = p.g;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + p.stages * p.stage_a_bytes;

  // ---- tile coordinates
  int bid = blockIdx.x;
  const int ntile = bid % p.n_ntiles;
  bid /= p.n_ntiles;
  const int phase = bid % g.nphase;
  bid /= g.nphase;
  const int tx = bid % p.tiles_x;
  bid /= p.tiles_x;
  const int ty = bid % p.tiles_y;
  bid /= p.tiles_y;
  const int tt = bid % g.T;
  const int bb = bid / g.T;
  const int x0 = tx * p.BX, y0 = ty * p.BY, n0 = ntile * p.BN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&accum_bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, p.tmem_cols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    for (int i = threadIdx.x - 64; i < p.BN; i += 128) {
      const int co = n0 + i;
      bias_sh[i] = (p.bias != nullptr && co < g.Cout) ? p.bias[co] : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the previous kernel on the stream has finished and its writes are visible from here on
  pdl_wait();
  const uint32_t tmem = tmem_base_sh;

  const int ksteps = g.ntaps * p.n_kchunks;

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t tx_bytes = static_cast<uint32_t>(kBM * BK * 2 + p.BN * BK * 2);
      int issued = 0;
      for (int ks = 0; ks < ksteps; ++ks) {
        const int s = ks % p.stages;
        const uint32_t ph = static_cast<uint32_t>(ks / p.stages) & 1u;
        if (ks >= p.stages && !mbar_wait(&empty_bar[s], ph ^ 1u, p.status, kErrTimeoutEmpty, &abort_flag)) break;
        const int tap = ks / p.n_kchunks;
        const int kc = ks - tap * p.n_kchunks;
        const ConvTap tp = g.taps[phase][tap];
        mbar_arrive_expect_tx(&full_bar[s], tx_bytes);
        tma_load_5d(smA + s * p.stage_a_bytes, &p.tmA, &full_bar[s], kc * BK, x0 + tp.dx, y0 + tp.dy, tt + tp.dt, bb);
        tma_load_3d(smB + s * p.stage_b_bytes, &p.tmB, &full_bar[s], kc * BK, tp.wtap, n0);
        issued = ks + 1;
      }
      if (abort_flag) {
        // Drain: wait (bounded) until every stage this thread filled has landed.
        for (int ks = max(0, issued - p.stages); ks < issued; ++ks) {
          const int s = ks % p.stages;
          mbar_drain(&full_bar[s], static_cast<uint32_t>(ks / p.stages) & 1u);
        }
      }
    }
    __syncwarp();   // reconverge warp 0 before the CTA-wide barrier
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, p.BN);
      const uint32_t a_base = smem_u32(smA), b_base = smem_u32(smB);
      for (int ks = 0; ks < ksteps; ++ks) {
        const int s = ks % p.stages;
        const uint32_t ph = static_cast<uint32_t>(ks / p.stages) & 1u;
        if (!mbar_wait(&full_bar[s], ph, p.status, kErrTimeoutFull, &abort_flag)) break;
        tc_fence_after();
        const uint32_t a0 = a_base + s * p.stage_a_bytes;
        const uint32_t b0 = b_base + s * p.stage_b_bytes;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t da = smem_desc_kmajor(a0 + k * 32, SwizzleOf<BK>::kSbo, SwizzleOf<BK>::kMode);
          const uint64_t db = smem_desc_kmajor(b0 + k * 32, SwizzleOf<BK>::kSbo, SwizzleOf<BK>::kMode);
          tc_mma_bf16(tmem, da, db, idesc, (ks | k) != 0 ? 1u : 0u);
        }
        tc_commit(&empty_bar[s]);
      }
      tc_commit(&accum_bar);
      // every MMA issued has completed before the CTA releases TMEM (also after a timeout,
      // when the epilogue stops waiting for the accumulator)
      mbar_drain(&accum_bar, 0);
    }
    __syncwarp();
  } else {
    // ---- epilogue: warps 2..5 cover TMEM lane quarters (warp % 4)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int ly = row / p.BX, lx = row - ly * p.BX;
    const int y = y0 + ly, x = x0 + lx;
    const bool valid = (y < g.H) && (x < g.W);
    const bool ok = mbar_wait(&accum_bar, 0, p.status, kErrTimeoutAccum, &abort_flag);
    tc_fence_after();
    // warp-uniform decision: tcgen05.ld is a warp-collective instruction
    const bool go = __all_sync(0xffffffffu, ok && !abort_flag);
    if (go) {
      const int py = phase >> 1, px = phase & 1;
      const int grid_pix = ((bb * g.T + tt) * g.H + y) * g.W + x;
      const float rs = (p.rowscale != nullptr && valid) ? p.rowscale[grid_pix] : 1.f;
      const int yo = y * g.osy + (g.nphase > 1 ? py : 0);
      const int xo = x * g.osx + (g.nphase > 1 ? px : 0);
      for (int c0 = 0; c0 < p.BN; c0 += 16) {
        uint32_t r[16];
        tmem_ld_16x_32x32b(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, r);
        tmem_ld_wait();
        const int co0 = n0 + c0;
        if (!valid || co0 >= g.Cout) continue;
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]) * g.scale * rs + bias_sh[c0 + j];
        epilogue_store16(g, v, bb, tt, yo, xo, co0, p.residual, p.out, p.out2);
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ---------------------------------------------------------------- host side
EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

CUtensorMapSwizzle swizzle_for(int bk) {
  return bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : (bk == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

namespace {

int round_up(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace

const char* conv_tc_plan(const ConvGeom& g, int* bk_out) {
  if (g.Cin % 8 != 0) return "tensor-core conv needs C_in a multiple of 8";
  if (g.Cout < 1) return "C_out must be positive";
  if (g.ntaps < 1 || g.ntaps > kMaxTaps || g.nphase < 1 || g.nphase > kMaxPhases) return "bad tap table";
  // BK: the largest chunk whose padded K is within 5% of the tightest one.
  int best = 1 << 30;
  for (int bk : {64, 32, 16}) best = std::min(best, round_up(g.Cin, bk));
  int bk = 16;
  for (int cand : {64, 32, 16}) {
    if (round_up(g.Cin, cand) * 100 <= best * 105) {
      bk = cand;
      break;
    }
  }
  *bk_out = bk;
  return nullptr;
}

cudaError_t launch_conv_tc(const ConvGeom& g, const void* in, const void* wts, int ntaps_w, int w_rows,
                           const float* bias, const void* residual, const float* rowscale, void* out, void* out2,
                           int* status, cudaStream_t stream, const char** why, int* gn_chunks,
                           const ConvShortcut* sc) {
  *why = nullptr;
  if (gn_chunks != nullptr) *gn_chunks = 0;
  if (sc != nullptr) {
    // a fused shortcut exists only in the channel-major halo kernel
    if (rowscale != nullptr || !conv_halo_t_applicable(g) || !conv_halo_t_shortcut_ok(g, sc->cin)) {
      *why = "shortcut fusion not supported for this conv";
      return cudaErrorInvalidValue;
    }
    return launch_conv_halo_t(g, in, wts, ntaps_w, w_rows, bias, residual, out, out2, status, stream, why,
                              gn_chunks, sc);
  }
  int bk = 64;
  if (const char* e = conv_tc_plan(g, &bk)) {
    *why = e;
    return cudaErrorInvalidValue;
  }
  if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(wts) & 15)) {
    *why = "conv operands must be 16-byte aligned";
    return cudaErrorInvalidValue;
  }
  if (rowscale == nullptr && conv_halo_t_applicable(g))
    return launch_conv_halo_t(g, in, wts, ntaps_w, w_rows, bias, residual, out, out2, status, stream, why,
                              gn_chunks);
  if (rowscale == nullptr && conv_halo_applicable(g))
    return launch_conv_halo(g, in, wts, ntaps_w, w_rows, bias, residual, out, out2, status, stream, why);
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return cudaErrorNotSupported;
  }
  if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(wts) & 15)) {
    *why = "conv operands must be 16-byte aligned";
    return cudaErrorInvalidValue;
  }
  ConvTcParams p;
  std::memset(&p, 0, sizeof(p));
  p.g = g;

  // Pixel tile: BY x BX = 128, BX a power of two chosen to waste the fewest pixels.
  long long best_cost = -1;
  for (int bx = 128; bx >= 8; bx >>= 1) {
    const int by = 128 / bx;
    const long long cost = static_cast<long long>((g.W + bx - 1) / bx) * bx * ((g.H + by - 1) / by) * by;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      p.BX = bx;
      p.BY = by;
    }
  }
  p.tiles_x = (g.W + p.BX - 1) / p.BX;
  p.tiles_y = (g.H + p.BY - 1) / p.BY;
  p.n_ntiles = (g.Cout + 255) / 256;
  p.BN = round_up((g.Cout + p.n_ntiles - 1) / p.n_ntiles, 16);
  p.n_kchunks = (g.Cin + bk - 1) / bk;
  p.stage_a_bytes = kBM * bk * 2;
  p.stage_b_bytes = static_cast<uint32_t>(round_up(p.BN * bk * 2, 1024));
  const int stage_bytes = static_cast<int>(p.stage_a_bytes + p.stage_b_bytes);
  p.stages = std::min(8, (200 * 1024) / stage_bytes);
  // narrow tiles do little MMA work per stage: keep the CTA small so that several
  // CTAs share an SM and cover each other's stage waits
  if (p.BN <= 64) p.stages = std::min(p.stages, 4);
  p.stages = std::min(p.stages, std::max(2, g.ntaps * ((g.Cin + bk - 1) / bk)));
  if (p.stages < 2) {
    *why = "tile does not fit shared memory";
    return cudaErrorInvalidValue;
  }
  p.tmem_cols = 32;
  while (p.tmem_cols < static_cast<uint32_t>(p.BN)) p.tmem_cols <<= 1;
  p.bias = bias;
  p.residual = residual;
  p.out2 = static_cast<__nv_bfloat16*>(out2);
  if (out2 != nullptr && g.out_chfirst) {
    *why = "a second output needs a channels-last store";
    return cudaErrorInvalidValue;
  }
  p.rowscale = rowscale;
  p.out = out;
  p.status = status;

  const cuuint32_t ones[5] = {1, 1, 1, 1, 1};
  {
    const cuuint64_t dims[5] = {static_cast<cuuint64_t>(g.Cin), static_cast<cuuint64_t>(g.W),
                                static_cast<cuuint64_t>(g.H), static_cast<cuuint64_t>(g.T),
                                static_cast<cuuint64_t>(g.B)};
    const cuuint64_t es = 2;
    const cuuint64_t strides[4] = {dims[0] * es, dims[0] * dims[1] * es, dims[0] * dims[1] * dims[2] * es,
                                   dims[0] * dims[1] * dims[2] * dims[3] * es};
    const cuuint32_t box[5] = {static_cast<cuuint32_t>(bk), static_cast<cuuint32_t>(p.BX),
                               static_cast<cuuint32_t>(p.BY), 1, 1};
    CUresult r = enc(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(in), dims, strides, box, ones,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *why = "activation tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.Cin), static_cast<cuuint64_t>(ntaps_w),
                                static_cast<cuuint64_t>(w_rows)};
    const cuuint64_t strides[2] = {dims[0] * 2, dims[0] * dims[1] * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(bk), 1, static_cast<cuuint32_t>(p.BN)};
    CUresult r = enc(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(wts), dims, strides, box, ones,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *why = "weight tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  const long long nblocks =
      static_cast<long long>(g.B) * g.T * p.tiles_y * p.tiles_x * g.nphase * p.n_ntiles;
  if (nblocks <= 0) return cudaSuccess;
  if (nblocks > 0x7fffffffLL) {
    *why = "grid too large";
    return cudaErrorInvalidValue;
  }
  const size_t smem = static_cast<size_t>(p.stages) * stage_bytes + 1024;
  cudaError_t e = cudaSuccess;
  switch (bk) {
    case 64:
      e = cudaFuncSetAttribute(conv_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) launch_pdl(conv_tc_kernel<64>, (unsigned)nblocks, kThreads, smem, stream, p);
      break;
    case 32:
      e = cudaFuncSetAttribute(conv_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) launch_pdl(conv_tc_kernel<32>, (unsigned)nblocks, kThreads, smem, stream, p);
      break;
    default:
      e = cudaFuncSetAttribute(conv_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) launch_pdl(conv_tc_kernel<16>, (unsigned)nblocks, kThreads, smem, stream, p);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

namespace {

// Waits, with the library's bounded wait, on a barrier that nothing ever completes: the wait
// runs out after the current limit, records kErrTimeoutFull in *status and the kernel returns.
__global__ void wait_probe_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    mbar_wait(&bar, 0, status, kErrTimeoutFull, &abort_flag);
  }
}

}  // namespace

cudaError_t launch_wait_probe(int* status, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

VD_WAIT_LIMIT_SETTER(set_wait_limit_conv_tc)

}  // namespace vd
