// Halo-tile implicit-GEMM convolution on tcgen05 tensor cores.
//
// A CTA computes R output rows x 128 pixels x BN output channels, one TMEM
// accumulator (128 lanes x BN fp32 columns) per output row.  For every input
// channel chunk (and causal frame) it stages the R + 2 input rows the tile needs
// -- 136 pixels each, starting one pixel left of the tile -- once, with one TMA
// box per row: boxes outside the image read zeros (the conv's zero padding at the
// global edges), rows of neighbouring bands read their real values (the halo of
// "VAEP：VAE 并行解码", 卷积：交换边界行).  All 3x3 taps then read that stage:
// tap (dy, dx) of output row r is the 128-pixel window of staged row r + dy + 1
// starting at pixel dx + 1, i.e. the shared-memory descriptor of the staged row
// advanced by whole pixel rows.  Compared with loading one shifted box per tap,
// the activations cross L2 -> SM once per chunk instead of nine times, and each
// weight chunk is reused for R output rows.
//
// Roles (192 threads): warp 0 issues TMA (activation stages double-buffered,
// weight stages NB-deep), warp 1 owns TMEM and issues tcgen05.mma, warps 2..5
// run the epilogue.  Waits are bounded (ptx.cuh).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "conv.h"
#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tma_host.h"
#include "launch.h"

namespace vd {

namespace {

constexpr int kHaloThreads = 192;
constexpr int kHaloPix = 136;     // staged pixels per row: 128 + 2 halo, rounded up to a multiple of 8
constexpr int kMaxNB = 8;
constexpr int kPipeBytes = 184 * 1024;   // activation + weight stages; 16 KB more for the epilogue stages

struct HaloParams {
  CUtensorMap tmA;               // activations as 5D (Cin, W, H, T, B), box (BK, 136, 1, 1, 1)
  CUtensorMap tmB;               // weights as 3D (Cin, ntaps_w, rows), box (BK, 1, BN)
  ConvGeom g;
  int R;                         // output rows per CTA
  int tiles_x, tiles_y, BN, n_ntiles, n_kchunks, ndt, nb;
  uint32_t rowbuf_bytes, a_stage_bytes, b_stage_bytes, tmem_cols;
  const float* bias;
  const void* residual;
  void* out;
  __nv_bfloat16* out2;
  int* status;
};

template <int BK>
struct Swz {
  static constexpr uint32_t kSbo = BK * 2 * 8;
  static constexpr uint32_t kMode = BK == 64 ? 2u : (BK == 32 ? 4u : 6u);
};

// Descriptor of a K-major operand that starts at any whole pixel row of a staged
// row buffer.  The tensor cores apply the swizzle to absolute shared-memory
// address bits (the same rule the TMA unit used when it wrote the stage), so a
// start shifted by whole rows needs no base-offset correction (field left 0).
template <int BK>
__device__ __forceinline__ uint64_t desc_at(uint32_t addr) {
  return smem_desc_kmajor(addr, Swz<BK>::kSbo, Swz<BK>::kMode);
}

template <int BK>
__global__ void __launch_bounds__(kHaloThreads, 1) conv_halo_kernel(const __grid_constant__ HaloParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t a_full[2], a_empty[2];
  __shared__ __align__(8) uint64_t b_full[kMaxNB], b_empty[kMaxNB];
  __shared__ __align__(8) uint64_t accum_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ float bias_sh[256];

  const ConvGeom& g = p.g;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + 2 * p.a_stage_bytes;

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
  const int x0 = tx * 128, y0 = ty * p.R, n0 = ntile * p.BN;
  const int nsp = g.ntaps / p.ndt;    // spatial taps per causal frame (9)

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < p.nb; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
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
  const int nac = p.ndt * p.n_kchunks;

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t a_tx = static_cast<uint32_t>((p.R + 2) * kHaloPix * BK * 2);
      const uint32_t b_tx = static_cast<uint32_t>(p.BN * BK * 2);
      int kb = 0, issued_a = 0, issued_b = 0;
      for (int ac = 0; ac < nac && !abort_flag; ++ac) {
        const int dti = ac / p.n_kchunks;
        const int kc = ac - dti * p.n_kchunks;
        const int dt = g.taps[phase][dti * nsp].dt;
        const int sa = ac & 1;
        if (ac >= 2 && !mbar_wait(&a_empty[sa], (static_cast<uint32_t>(ac >> 1) & 1u) ^ 1u, p.status,
                                  kErrTimeoutEmpty, &abort_flag))
          break;
        mbar_arrive_expect_tx(&a_full[sa], a_tx);
        for (int rb = 0; rb < p.R + 2; ++rb)
          tma_load_5d(smA + sa * p.a_stage_bytes + rb * p.rowbuf_bytes, &p.tmA, &a_full[sa], kc * BK, x0 - 1,
                      y0 - 1 + rb, tt + dt, bb);
        issued_a = ac + 1;
        for (int s = 0; s < nsp; ++s, ++kb) {
          const int sb = kb % p.nb;
          if (kb >= p.nb && !mbar_wait(&b_empty[sb], (static_cast<uint32_t>(kb / p.nb) & 1u) ^ 1u, p.status,
                                       kErrTimeoutEmpty, &abort_flag))
            break;
          mbar_arrive_expect_tx(&b_full[sb], b_tx);
          tma_load_3d(smB + sb * p.b_stage_bytes, &p.tmB, &b_full[sb], kc * BK, g.taps[phase][dti * nsp + s].wtap,
                      n0);
          issued_b = kb + 1;
        }
      }
      if (abort_flag) {
        // drain: every stage this thread filled lands before the CTA exits (bounded)
        for (int ac = max(0, issued_a - 2); ac < issued_a; ++ac)
          mbar_drain(&a_full[ac & 1], static_cast<uint32_t>(ac >> 1) & 1u);
        for (int k = max(0, issued_b - p.nb); k < issued_b; ++k)
          mbar_drain(&b_full[k % p.nb], static_cast<uint32_t>(k / p.nb) & 1u);
      }
    }
    __syncwarp();   // reconverge warp 0 before the CTA-wide barrier
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, p.BN);
      const uint32_t a_base0 = smem_u32(smA), b_base0 = smem_u32(smB);
      int kb = 0;
      bool ok = true;
      for (int ac = 0; ac < nac && ok; ++ac) {
        const int dti = ac / p.n_kchunks;
        const int sa = ac & 1;
        if (!mbar_wait(&a_full[sa], static_cast<uint32_t>(ac >> 1) & 1u, p.status, kErrTimeoutFull, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = a_base0 + sa * p.a_stage_bytes;
        for (int s = 0; s < nsp; ++s, ++kb) {
          const int sb = kb % p.nb;
          if (!mbar_wait(&b_full[sb], static_cast<uint32_t>(kb / p.nb) & 1u, p.status, kErrTimeoutFull,
                         &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const ConvTap tp = g.taps[phase][dti * nsp + s];
          const uint32_t b_addr = b_base0 + sb * p.b_stage_bytes;
          for (int r = 0; r < p.R; ++r) {
            const uint32_t a_addr =
                a_base + (r + tp.dy + 1) * p.rowbuf_bytes + static_cast<uint32_t>((tp.dx + 1) * BK * 2);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t da = desc_at<BK>(a_addr + k * 32);
              const uint64_t db = smem_desc_kmajor(b_addr + k * 32, Swz<BK>::kSbo, Swz<BK>::kMode);
              tc_mma_bf16(tmem + static_cast<uint32_t>(r * p.BN), da, db, idesc, (ac | s | k) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&b_empty[sb]);
        }
        tc_commit(&a_empty[sa]);
      }
      tc_commit(&accum_bar);
      // every MMA issued has completed before the CTA releases TMEM (also after a timeout,
      // when the epilogue stops waiting for the accumulator)
      mbar_drain(&accum_bar, 0);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    uint8_t* stage = smB + p.nb * p.b_stage_bytes + q * kEpiStageBytes;
    const int x = x0 + q * 32 + lane;
    const bool xvalid = x < g.W;
    const bool ok = mbar_wait(&accum_bar, 0, p.status, kErrTimeoutAccum, &abort_flag);
    tc_fence_after();
    const bool go = __all_sync(0xffffffffu, ok && !abort_flag);
    if (go) {
      const int py = phase >> 1, px = phase & 1;
      const int xo = x * g.osx + (g.nphase > 1 ? px : 0);
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
      for (int r = 0; r < p.R; ++r) {
        const int y = y0 + r;
        const bool valid = xvalid && y < g.H;
        const int yo = y * g.osy + (g.nphase > 1 ? py : 0);
        const long long opix = ((static_cast<long long>(bb) * g.oT + tt) * g.oH + yo) * g.oW + xo;
        for (int c0 = 0; c0 < p.BN; c0 += 32) {
          const int co0 = n0 + c0;
          const int nc = min(32, min(p.BN - c0, g.Cout - co0));   // warp-uniform
          if (nc <= 0) break;
          uint32_t rr[32];
          if (nc > 16) {
            tmem_ld_32x32b_x32(lane_addr + static_cast<uint32_t>(r * p.BN + c0), rr);
          } else {
            uint32_t (&h)[16] = *reinterpret_cast<uint32_t(*)[16]>(rr);
            tmem_ld_16x_32x32b(lane_addr + static_cast<uint32_t>(r * p.BN + c0), h);
          }
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(rr[j]) * g.scale + bias_sh[(c0 + j) & 255];
          if (g.out_chfirst) {
            if (valid) {
              float* h0 = v;
              epilogue_store16(g, *reinterpret_cast<float(*)[16]>(h0), bb, tt, yo, xo, co0, p.residual, p.out, p.out2);
              if (nc > 16)
                epilogue_store16(g, *reinterpret_cast<float(*)[16]>(h0 + 16), bb, tt, yo, xo, co0 + 16, p.residual,
                                 p.out, p.out2);
            }
          } else if (nc > 16) {
            epi_chunk_cl<32>(g, v, opix * g.oC + co0, valid, p.residual, p.out, p.out2, stage, lane);
          } else {
            epi_chunk_cl<16>(g, v, opix * g.oC + co0, valid, p.residual, p.out, p.out2, stage, lane);
          }
        }
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

int round_up_i(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace

// The halo kernel applies to centred 3x3 taps (optionally grouped by causal frame,
// or as four upsample phases) on grids at least 128 pixels wide whose 128-pixel
// row tiles waste at most 12% of the MMA rows.
bool conv_halo_applicable(const ConvGeom& g) {
  if (g.ntaps != 9 && g.ntaps != 27) return false;
  if (g.out_chfirst || g.Cout < 64) return false;   // narrow N: the one-tile kernel is faster
  if (g.W < 128) return false;
  const int tiles = (g.W + 127) / 128;
  if (tiles * 128 * 100 > g.W * 112) return false;
  const int ndt = g.ntaps / 9;
  for (int ph = 0; ph < g.nphase; ++ph)
    for (int d = 0; d < ndt; ++d)
      for (int s = 0; s < 9; ++s) {
        const ConvTap t = g.taps[ph][d * 9 + s];
        if (t.dt != g.taps[ph][d * 9].dt) return false;
        if (t.dy < -1 || t.dy > 1 || t.dx < -1 || t.dx > 1) return false;
      }
  return true;
}

cudaError_t launch_conv_halo(const ConvGeom& g, const void* in, const void* wts, int ntaps_w, int w_rows,
                             const float* bias, const void* residual, void* out, void* out2, int* status,
                             cudaStream_t stream, const char** why) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return cudaErrorNotSupported;
  }
  HaloParams p;
  std::memset(&p, 0, sizeof(p));
  p.g = g;
  p.n_ntiles = (g.Cout + 255) / 256;
  p.BN = round_up_i((g.Cout + p.n_ntiles - 1) / p.n_ntiles, 16);
  // rows per CTA: as many accumulators as TMEM holds (at most 4)
  p.R = std::max(1, std::min(4, 512 / p.BN));
  while (p.R > 1 && p.R > g.H) --p.R;
  // K chunk: the largest that divides C_in (allowing 5% padding) and fits two activation stages
  // plus at least four weight stages in 200 KB
  int bk = 0;
  for (int cand : {64, 32, 16}) {
    if (round_up_i(g.Cin, cand) * 100 > g.Cin * 105) continue;
    const int a_stage = (p.R + 2) * kHaloPix * cand * 2;
    const int b_stage = round_up_i(p.BN * cand * 2, 1024);
    if (2 * a_stage + 4 * b_stage <= kPipeBytes) {
      bk = cand;
      break;
    }
  }
  if (bk == 0) {
    *why = "no halo tile fits shared memory";
    return cudaErrorInvalidValue;
  }
  p.n_kchunks = (g.Cin + bk - 1) / bk;
  p.ndt = g.ntaps / 9;
  p.rowbuf_bytes = static_cast<uint32_t>(kHaloPix * bk * 2);
  p.a_stage_bytes = static_cast<uint32_t>((p.R + 2) * p.rowbuf_bytes);
  p.b_stage_bytes = static_cast<uint32_t>(round_up_i(p.BN * bk * 2, 1024));
  p.nb = std::min(kMaxNB, static_cast<int>((kPipeBytes - 2 * p.a_stage_bytes) / p.b_stage_bytes));
  p.tiles_x = (g.W + 127) / 128;
  p.tiles_y = (g.H + p.R - 1) / p.R;
  p.tmem_cols = 32;
  while (p.tmem_cols < static_cast<uint32_t>(p.R * p.BN)) p.tmem_cols <<= 1;
  p.bias = bias;
  p.residual = residual;
  p.out = out;
  p.out2 = static_cast<__nv_bfloat16*>(out2);
  p.status = status;

  const cuuint32_t ones[5] = {1, 1, 1, 1, 1};
  {
    const cuuint64_t dims[5] = {(cuuint64_t)g.Cin, (cuuint64_t)g.W, (cuuint64_t)g.H, (cuuint64_t)g.T,
                                (cuuint64_t)g.B};
    const cuuint64_t strides[4] = {dims[0] * 2, dims[0] * dims[1] * 2, dims[0] * dims[1] * dims[2] * 2,
                                   dims[0] * dims[1] * dims[2] * dims[3] * 2};
    const cuuint32_t box[5] = {(cuuint32_t)bk, (cuuint32_t)kHaloPix, 1, 1, 1};
    if (enc(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(in), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "halo activation tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)g.Cin, (cuuint64_t)ntaps_w, (cuuint64_t)w_rows};
    const cuuint64_t strides[2] = {dims[0] * 2, dims[0] * dims[1] * 2};
    const cuuint32_t box[3] = {(cuuint32_t)bk, 1, (cuuint32_t)p.BN};
    if (enc(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(wts), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "halo weight tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  const long long nblocks = (long long)g.B * g.T * p.tiles_y * p.tiles_x * g.nphase * p.n_ntiles;
  if (nblocks <= 0) return cudaSuccess;
  if (nblocks > 0x7fffffffLL) {
    *why = "grid too large";
    return cudaErrorInvalidValue;
  }
  const size_t smem = 2 * (size_t)p.a_stage_bytes + (size_t)p.nb * p.b_stage_bytes + 4 * kEpiStageBytes + 1024;
  cudaError_t e;
  switch (bk) {
    case 64:
      e = cudaFuncSetAttribute(conv_halo_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) launch_pdl(conv_halo_kernel<64>, (unsigned)nblocks, kHaloThreads, smem, stream, p);
      break;
    case 32:
      e = cudaFuncSetAttribute(conv_halo_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) launch_pdl(conv_halo_kernel<32>, (unsigned)nblocks, kHaloThreads, smem, stream, p);
      break;
    default:
      e = cudaFuncSetAttribute(conv_halo_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) launch_pdl(conv_halo_kernel<16>, (unsigned)nblocks, kHaloThreads, smem, stream, p);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

VD_WAIT_LIMIT_SETTER(set_wait_limit_conv_halo)

}  // namespace vd
