// Channel-major halo-tile convolution on tcgen05 tensor cores.
//
// The GEMM is laid out with output channels on M (128 per CTA) and pixels on N
// (one image row segment of up to 256 pixels): D[co, x] += W[co, tap, ci] *
// in[x + offset(tap), ci].  As in the pixel-major halo kernel, every input
// channel chunk stages the R + 2 input rows a tile needs once (zero-filled
// outside the image: the global-edge padding; real rows across band boundaries:
// the halo of "VAEP：VAE 并行解码", 卷积：交换边界行), and each 3x3 tap reads those
// rows through a shared-memory descriptor shifted by whole pixels.  Putting
// pixels on N gives 256-wide MMAs for every layer (also the 128-channel ones),
// which keeps the tensor pipe at its full rate, and makes every TMEM lane one
// output channel, so each epilogue store instruction writes 32 consecutive
// channels of one pixel: fully coalesced, with residual reads batched 32 deep.
//
// Roles (352 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warp 2 waiter,
// warps 3..10 epilogue (two warps per TMEM lane quarter).  The waiter polls the stage and
// accumulator barriers in the MMA warp's order and releases the MMA warp through a named barrier,
// so the MMA-issuing thread never polls shared memory while the tensor pipe saturates it (a poll
// then costs about a thousand cycles, more than a one-row weight stage's 768 cycles of MMAs).  A
// weight stage holds the three taps of one kernel row.  Every wait is bounded (ptx.cuh); the waiter
// and the MMA warp pass the named barrier the same number of times on every path.
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

constexpr int kThreadsT = 352;   // warp 0 TMA, warp 1 MMA, warp 2 waiter, warps 3..10 epilogue (two per TMEM lane quarter)
constexpr int kEpiWarpsT = 8;
constexpr int kMaxWStages = 4;
constexpr int kPipeBytesT = 212 * 1024;
constexpr int kStageOutBytes = 16 * 32 * 4;   // one epilogue warp's [16 px][32 ch] fp32 staging
constexpr int kResBufs = 3;                    // staging buffers per warp when the residual comes by TMA
constexpr int kStageOut2Bytes = 16 * 32 * 2;   // one epilogue warp's [16 px][32 ch] bf16 copy staging
constexpr int kMaxDynSmemT = 227 * 1024 - 512;   // per-CTA limit, less room for the static barriers (336 B)

struct HaloTParams {
  CUtensorMap tmX;               // activations 5D (Cin, W, H, T, B), box (BK, half, 1, 1, 1)
  CUtensorMap tmW;               // weights 3D (Cin, ntaps_w, rows), box (BK, 1, 128)
  ConvGeom g;
  int R;                         // output rows per CTA
  int npx;                       // pixels per tile (MMA N)
  int half;                      // pixels per staging box (two boxes per staged row)
  int tiles_x, tiles_y, n_mtiles, n_kchunks, ndt, nw, ntiles;
  int nbuf;                      // accumulator buffers in TMEM (2: a tile's epilogue overlaps the next tile's MMAs)
  int acc_cols;                  // TMEM columns per buffer
  int csplit;                    // 2: the two epilogue warp halves split a row's pixels (R == 1), else 1
  uint32_t row_bytes, x_stage_bytes, w_tap_bytes, w_stage_bytes, tmem_cols;
  const float* bias;
  const void* residual;
  void* out;
  __nv_bfloat16* out2;
  int* status;
  GnPartial* gn_part;            // GroupNorm chunk moments of the output, or null
  int gn_cg;                     // channels per group (divides 32)
  // fused 1x1 shortcut (R == 1 only): its input's centre row staged in up to three channel chunks
  // per stage, beside the matching weight chunks in the three tap slots of a weight stage
  CUtensorMap tmX2;              // shortcut input 5D (sc_cin, W, H, T, B), box (BK, half, 1, 1, 1)
  CUtensorMap tmW2;              // shortcut weights 3D (sc_cin, 1, rows), box (BK, 1, 128)
  int sc_chunks;                 // shortcut channel chunks (sc_cin / BK), 0 = no shortcut
  int n_sc;                      // shortcut stages per tile: ceil(sc_chunks / 3)
  // fp32 output through shared memory and TMA tensor stores (each epilogue warp stages 16 pixels x
  // its 32 channels, then one thread stores them), instead of one 4-byte store per value
  CUtensorMap tmO;               // output 3D (oC, oW, B * oT * oH), box (32, 16, 1)
  CUtensorMap tmR;               // fp32 residual, same geometry as tmO (loaded with TMA when tma_out == 2)
  CUtensorMap tmO2;              // bf16 copy of the output, same geometry (tma_out == 1 with out2)
  int tma_out;                   // 0: direct stores; 1: TMA stores; 2: also TMA residual loads (one-row tiles)
  uint32_t stage_out_off;        // byte offset of the epilogue staging buffers (2 KB each) in the pipeline
};

template <int BK>
struct SwzT {
  static constexpr uint32_t kSbo = BK * 2 * 8;
  static constexpr uint32_t kMode = BK == 64 ? 2u : (BK == 32 ? 4u : 6u);
};

// Chan's merge of central moments: (n, mean, M2) of part a, then part b.
__device__ __forceinline__ void moments_merge(float na, float ma, float m2a, float nb, float mb, float m2b, float& n,
                                              float& m, float& m2) {
  if (nb == 0.f) {
    n = na; m = ma; m2 = m2a;
    return;
  }
  if (na == 0.f) {
    n = nb; m = mb; m2 = m2b;
    return;
  }
  const float nt = na + nb;
  const float d = mb - ma;
  m = ma + d * (nb / nt);
  m2 = m2a + m2b + d * d * (na * nb / nt);
  n = nt;
}

struct TileT {
  int mtile, phase, tx, ty, tt, bb, x0, y0, m0;
};

__device__ __forceinline__ TileT decode_tile(const HaloTParams& p, int t) {
  TileT d;
  d.mtile = t % p.n_mtiles;
  t /= p.n_mtiles;
  d.phase = t % p.g.nphase;
  t /= p.g.nphase;
  d.tx = t % p.tiles_x;
  t /= p.tiles_x;
  d.ty = t % p.tiles_y;
  t /= p.tiles_y;
  d.tt = t % p.g.T;
  d.bb = t / p.g.T;
  d.x0 = d.tx * p.npx;
  d.y0 = d.ty * p.R;
  d.m0 = d.mtile * 128;
  return d;
}

// Shifted GroupNorm sums of v[0..15] (the first nvalid values): four interleaved partial sums per
// moment, the pairs of each group of four added as packed f32x2 (the same roundings, in the same
// order, as four scalar accumulators), then folded in a fixed tree.
__device__ __forceinline__ void gn_sums16(const float (&v)[16], int nvalid, float kshift, float& s1, float& s2,
                                          float& cnt) {
  float2 a1l = make_float2(0.f, 0.f), a1h = a1l, a2l = a1l, a2h = a1l;
  if (nvalid == 16) {
    const float2 nk = make_float2(-kshift, -kshift);
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
      const float2 dl = __fadd2_rn(make_float2(v[j], v[j + 1]), nk);
      const float2 dh = __fadd2_rn(make_float2(v[j + 2], v[j + 3]), nk);
      a1l = __fadd2_rn(a1l, dl);
      a1h = __fadd2_rn(a1h, dh);
      a2l = __ffma2_rn(dl, dl, a2l);
      a2h = __ffma2_rn(dh, dh, a2h);
    }
  } else {
    float a1[4] = {0.f, 0.f, 0.f, 0.f}, a2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float dv = (j < nvalid) ? v[j] - kshift : 0.f;
      a1[j & 3] += dv;
      a2[j & 3] = fmaf(dv, dv, a2[j & 3]);
    }
    a1l = make_float2(a1[0], a1[1]);
    a1h = make_float2(a1[2], a1[3]);
    a2l = make_float2(a2[0], a2[1]);
    a2h = make_float2(a2[2], a2[3]);
  }
  s1 += (a1l.x + a1l.y) + (a1h.x + a1h.y);
  s2 += (a2l.x + a2l.y) + (a2h.x + a2h.y);
  cnt += static_cast<float>(nvalid);
}

// GroupNorm chunk moments of output channel `co` over tile row r, from sums shifted by kshift, merged
// over the group's gn_cg consecutive lanes and stored by the group's first lane.
__device__ __forceinline__ void gn_store(const HaloTParams& p, const TileT& d, int r, int co, bool cvalid, int lane,
                                         int sub, float kshift, float s1, float s2, float cnt) {
  const ConvGeom& g = p.g;
  const int py = d.phase >> 1, px = d.phase & 1;
  // this channel's (count, mean, centred sum of squares) over the row
  float sn = cnt, smean = 0.f, sm2 = 0.f;
  if (cnt > 0.f) {
    const float d1 = s1 / cnt;
    smean = kshift + d1;
    sm2 = fmaxf(s2 - s1 * d1, 0.f);
  }
  // merge the group's channels (gn_cg consecutive lanes), lower lane first
  for (int off = 1; off < p.gn_cg; off <<= 1) {
    const float on = __shfl_xor_sync(0xffffffffu, sn, off);
    const float om = __shfl_xor_sync(0xffffffffu, smean, off);
    const float o2 = __shfl_xor_sync(0xffffffffu, sm2, off);
    if (lane & off)
      moments_merge(on, om, o2, sn, smean, sm2, sn, smean, sm2);
    else
      moments_merge(sn, smean, sm2, on, om, o2, sn, smean, sm2);
  }
  if (cvalid && (lane % p.gn_cg) == 0) {
    // chunk = (output row, phase column, pixel tile, column half), fixed by the geometry alone
    const int yo = (d.y0 + r) * g.osy + (g.nphase > 1 ? py : 0);
    const int npxp = g.nphase > 1 ? 2 : 1;
    const long long orow = static_cast<long long>(d.tt) * g.oH + yo;
    const long long chunk = ((orow * npxp + (g.nphase > 1 ? px : 0)) * p.tiles_x + d.tx) * p.csplit +
                            (p.csplit == 2 ? sub : 0);
    const long long n_chunks = static_cast<long long>(g.oT) * g.oH * npxp * p.tiles_x * p.csplit;
    GnPartial o;
    o.n = sn;
    o.mean = smean;
    o.m2 = sm2;
    o.pad = 0.f;
    // [sample][group][chunk]: a group's chunks are contiguous for the merge
    p.gn_part[(static_cast<long long>(d.bb) * g.gn_groups + co / p.gn_cg) * n_chunks + chunk] = o;
  }
}

// Named barrier 1, shared by the waiter warp and the MMA warp (64 threads); returns true when the
// waiter saw the abort flag raised.
__device__ __forceinline__ bool stage_handoff(bool aborted) { return bar_sync_or(1, 64, aborted); }

// kNsp: spatial taps per causal frame, 9 (three kernel rows of 3), or 7 for an upsample conv in its exact
// two-by-two phase form (weight stages of 3, 3 and 1 taps).  A compile-time count keeps the MMA issue
// loop free of per-stage tap tests.
template <int BK, int kOut, int kNsp>
__global__ void __launch_bounds__(kThreadsT, 1) conv_halo_t_kernel(const __grid_constant__ HaloTParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t x_full[2], x_empty[2];
  __shared__ __align__(8) uint64_t w_full[kMaxWStages], w_empty[kMaxWStages];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ __align__(8) uint64_t res_full[kEpiWarpsT * kResBufs];   // residual TMA loads (tma_out == 2)
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const ConvGeom& g = p.g;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smX = smem;
  uint8_t* smW = smem + 2 * p.x_stage_bytes;
  const int nsp = g.ntaps / p.ndt;   // 9 spatial taps per causal frame (kernel rows of 3), or 7

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 1);
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarpsT);
    }
    for (int i = 0; i < p.nw; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&w_empty[i], 1);
    }
    mbar_init(&mma_done, 1);
    for (int i = 0; i < kEpiWarpsT * kResBufs; ++i) mbar_init(&res_full[i], 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmX);
    tma_prefetch_desc(&p.tmW);
    if (p.tma_out != 0) tma_prefetch_desc(&p.tmO);
    if (p.tma_out == 2) tma_prefetch_desc(&p.tmR);
    if (p.n_sc > 0) {
      tma_prefetch_desc(&p.tmX2);
      tma_prefetch_desc(&p.tmW2);
    }
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
  const int nac = p.ndt * p.n_kchunks;   // staged activation chunks per tile
  const int ngrp = (nsp + 2) / 3;        // weight stages per chunk (up to 3 taps each)

  if (warp == 0) {
    // ---- TMA producer: activation chunks (R + 2 rows) and weight stages (3 taps), tile after tile
    if (lane == 0) {
      const uint32_t x_tx = static_cast<uint32_t>((p.R + 2) * 2 * p.half * BK * 2);
      const uint32_t w_tx = static_cast<uint32_t>(3 * 128 * BK * 2);
      int acg = 0, kbg = 0;   // chunks / weight stages issued so far (all tiles)
      int sw = 0;             // weight slot of stage kbg (kbg % nw, kept as a running count)
      uint32_t wpar = 1u;     // parity of the empty phase that frees slot sw for stage kbg
      for (int t = blockIdx.x; t < p.ntiles && !abort_flag; t += gridDim.x) {
        const TileT d = decode_tile(p, t);
        for (int ac = 0; ac < nac && !abort_flag; ++ac) {
          const int dti = ac / p.n_kchunks;
          const int kc = ac - dti * p.n_kchunks;
          const int dt = g.taps[d.phase][dti * nsp].dt;
          const int sx = acg & 1;
          if (acg >= 2 && !mbar_wait(&x_empty[sx], (static_cast<uint32_t>(acg >> 1) & 1u) ^ 1u, p.status,
                                     kErrTimeoutEmpty, &abort_flag))
            break;
          mbar_arrive_expect_tx(&x_full[sx], x_tx);
          uint8_t* xs = smX + sx * p.x_stage_bytes;
          for (int rb = 0; rb < p.R + 2; ++rb) {
            tma_load_5d(xs + rb * p.row_bytes, &p.tmX, &x_full[sx], kc * BK, d.x0 - 1, d.y0 - 1 + rb, d.tt + dt,
                        d.bb);
            tma_load_5d(xs + rb * p.row_bytes + p.half * BK * 2, &p.tmX, &x_full[sx], kc * BK, d.x0 - 1 + p.half,
                        d.y0 - 1 + rb, d.tt + dt, d.bb);
          }
          ++acg;
          for (int gi = 0; gi < ngrp; ++gi) {
            const int ntp = kNsp == 9 ? 3 : min(3, nsp - 3 * gi);   // taps in this weight stage
            if (kbg >= p.nw && !mbar_wait(&w_empty[sw], wpar, p.status, kErrTimeoutEmpty, &abort_flag)) break;
            mbar_arrive_expect_tx(&w_full[sw], kNsp == 9 ? w_tx : static_cast<uint32_t>(ntp) * p.w_tap_bytes);
            uint8_t* ws = smW + sw * p.w_stage_bytes;
            for (int tp = 0; tp < ntp; ++tp)
              tma_load_3d(ws + tp * p.w_tap_bytes, &p.tmW, &w_full[sw], kc * BK,
                          g.taps[d.phase][dti * nsp + gi * 3 + tp].wtap, d.m0);
            ++kbg;
            if (++sw == p.nw) {
              sw = 0;
              wpar ^= 1u;
            }
          }
        }
        for (int sc = 0; sc < p.n_sc && !abort_flag; ++sc) {
          // fused shortcut: centre row (y0, R == 1) of up to three channel chunks, and their weights
          const int cnt = min(3, p.sc_chunks - 3 * sc);
          const int sx = acg & 1;
          if (acg >= 2 && !mbar_wait(&x_empty[sx], (static_cast<uint32_t>(acg >> 1) & 1u) ^ 1u, p.status,
                                     kErrTimeoutEmpty, &abort_flag))
            break;
          mbar_arrive_expect_tx(&x_full[sx], static_cast<uint32_t>(cnt * 2 * p.half * BK * 2));
          uint8_t* xs = smX + sx * p.x_stage_bytes;
          for (int sl = 0; sl < cnt; ++sl) {
            const int kc = 3 * sc + sl;
            tma_load_5d(xs + sl * p.row_bytes, &p.tmX2, &x_full[sx], kc * BK, d.x0 - 1, d.y0, d.tt, d.bb);
            tma_load_5d(xs + sl * p.row_bytes + p.half * BK * 2, &p.tmX2, &x_full[sx], kc * BK, d.x0 - 1 + p.half,
                        d.y0, d.tt, d.bb);
          }
          ++acg;
          if (kbg >= p.nw && !mbar_wait(&w_empty[sw], wpar, p.status, kErrTimeoutEmpty, &abort_flag)) break;
          mbar_arrive_expect_tx(&w_full[sw], static_cast<uint32_t>(cnt) * p.w_tap_bytes);
          uint8_t* ws = smW + sw * p.w_stage_bytes;
          for (int sl = 0; sl < cnt; ++sl) tma_load_3d(ws + sl * p.w_tap_bytes, &p.tmW2, &w_full[sw], (3 * sc + sl) * BK, 0, d.m0);
          ++kbg;
          if (++sw == p.nw) {
            sw = 0;
            wpar ^= 1u;
          }
        }
      }
      if (abort_flag) {
        // let the copies already issued land before the CTA exits
        for (int i = max(0, acg - 2); i < acg; ++i)
          mbar_drain(&x_full[i & 1], static_cast<uint32_t>(i >> 1) & 1u);
        for (int k = max(0, kbg - p.nw); k < kbg; ++k)
          mbar_drain(&w_full[k % p.nw], static_cast<uint32_t>(k / p.nw) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---- waiter: polls the barriers the MMA warp consumes, in the MMA warp's order, and hands each
    // weight stage over through the named barrier (one hand-off per stage, also after an abort)
    // (slot, parity) of every ring advance as running counts: no divisions in the loop
    int acg = 0, it = 0, buf = 0, sw = 0;
    uint32_t wpar = 0u, apar = 1u;   // full parity of slot sw; empty parity of accumulator buf
    bool ab = false;                 // abort seen (lane 0)
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
      for (int ac = 0; ac < nac; ++ac, ++acg) {
        for (int gi = 0; gi < ngrp; ++gi) {
          if (lane == 0 && !ab) {
            // the first hand-off of a tile also covers its accumulator buffer, the first of a chunk its rows
            if (ac == 0 && gi == 0 && it >= p.nbuf)
              mbar_wait(&acc_empty[buf], apar, p.status, kErrTimeoutEmpty, &abort_flag);
            if (gi == 0)
              mbar_wait(&x_full[acg & 1], static_cast<uint32_t>(acg >> 1) & 1u, p.status, kErrTimeoutFull,
                        &abort_flag);
            mbar_wait(&w_full[sw], wpar, p.status, kErrTimeoutFull, &abort_flag);
            ab = abort_flag != 0;
          }
          __syncwarp();
          stage_handoff(ab);
          if (++sw == p.nw) {
            sw = 0;
            wpar ^= 1u;
          }
        }
      }
      for (int sc = 0; sc < p.n_sc; ++sc, ++acg) {
        if (lane == 0 && !ab) {
          mbar_wait(&x_full[acg & 1], static_cast<uint32_t>(acg >> 1) & 1u, p.status, kErrTimeoutFull, &abort_flag);
          mbar_wait(&w_full[sw], wpar, p.status, kErrTimeoutFull, &abort_flag);
          ab = abort_flag != 0;
        }
        __syncwarp();
        stage_handoff(ab);
        if (++sw == p.nw) {
          sw = 0;
          wpar ^= 1u;
        }
      }
      if (++buf == p.nbuf) {
        buf = 0;
        apar ^= 1u;
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: tile i accumulates into TMEM buffer i % nbuf.  It never reads shared memory:
    // the waiter warp releases it through the named barrier once a stage (or buffer) is ready, and
    // hands over the abort state in the same barrier.  The
    // issue loop only adds precomputed offsets to two base descriptors (the start-address field is
    // in 16-byte units), so one thread issues faster than the tensor pipe executes.
    const uint32_t idesc = idesc_bf16_f32(128, p.npx);
    const uint64_t dA0 = smem_desc_kmajor(smem_u32(smW), SwzT<BK>::kSbo, SwzT<BK>::kMode);
    const uint64_t dB0 = smem_desc_kmajor(smem_u32(smX), SwzT<BK>::kSbo, SwzT<BK>::kMode);
    const uint32_t w_stage16 = p.w_stage_bytes >> 4, w_tap16 = p.w_tap_bytes >> 4;
    const uint32_t x_stage16 = p.x_stage_bytes >> 4, row16 = p.row_bytes >> 4;
    const bool one_row = p.R == 1;
    int it = 0, sw = 0, acg = 0;
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
      const int phase = decode_tile(p, t).phase;
      // per spatial tap (the same for every causal frame): offset of its shifted rows
      uint32_t xoff[9];
#pragma unroll
      for (int i = 0; i < 9; ++i) {
        const ConvTap tap = g.taps[phase][i];
        xoff[i] = static_cast<uint32_t>(((tap.dy + 1) * static_cast<int>(p.row_bytes) + (tap.dx + 1) * BK * 2) >> 4);
      }
      const int buf = it % p.nbuf;
      const uint32_t dcol = tmem + static_cast<uint32_t>(buf * p.acc_cols);
      for (int ac = 0; ac < nac; ++ac, ++acg) {
        const int sx = acg & 1;
        const uint64_t dBs = dB0 + static_cast<uint64_t>(sx * x_stage16);
#pragma unroll
        for (int gi = 0; gi < 3; ++gi) {
          const int ntp = (kNsp == 9 || gi < 2) ? 3 : kNsp - 6;   // taps of this stage (compile time)
          const bool aborted = stage_handoff(false);
          tc_fence_after();
          if (lane == 0) {
            if (!aborted) {
              const uint64_t dAs = dA0 + static_cast<uint64_t>(sw * w_stage16);
              if (one_row) {
                // one-row tiles: the stage's MMAs back to back with no test between them (the tensor
                // pipe queues few MMAs, so work between two issues can leave it idle)
#pragma unroll
                for (int tp = 0; tp < 3; ++tp) {
                  if (tp >= ntp) continue;   // resolved at compile time in the unrolled loop
                  const uint64_t dAt = dAs + tp * w_tap16;
                  const uint64_t dBt = dBs + xoff[gi * 3 + tp];
#pragma unroll
                  for (int k = 0; k < BK / 16; ++k)
                    tc_mma_bf16(dcol, dAt + 2 * k, dBt + 2 * k, idesc, (ac | gi | tp | k) != 0 ? 1u : 0u);
                }
              } else {
#pragma unroll
                for (int tp = 0; tp < 3; ++tp) {
                  if (tp >= ntp) continue;
                  const uint64_t dAt = dAs + tp * w_tap16;
                  const uint64_t dBt = dBs + xoff[gi * 3 + tp];
#pragma unroll
                  for (int r = 0; r < 4; ++r) {
                    if (r < p.R) {
#pragma unroll
                      for (int k = 0; k < BK / 16; ++k)
                        tc_mma_bf16(dcol + static_cast<uint32_t>(r * p.npx), dAt + 2 * k, dBt + r * row16 + 2 * k,
                                    idesc, (ac | gi | tp | k) != 0 ? 1u : 0u);
                    }
                  }
                }
              }
            }
            tc_commit(&w_empty[sw]);
          }
          __syncwarp();
          sw = (sw + 1 == p.nw) ? 0 : sw + 1;
        }
        if (lane == 0) tc_commit(&x_empty[sx]);
        __syncwarp();
      }
      for (int sc = 0; sc < p.n_sc; ++sc, ++acg) {
        // fused shortcut: slot i holds channel chunk 3 sc + i of the centre row and its weights
        const int cnt = min(3, p.sc_chunks - 3 * sc);
        const int sx = acg & 1;
        const uint64_t dBs = dB0 + static_cast<uint64_t>(sx * x_stage16) + (BK * 2 / 16);   // centre pixel
        const bool aborted = stage_handoff(false);
        tc_fence_after();
        if (lane == 0) {
          if (!aborted) {
            const uint64_t dAs = dA0 + static_cast<uint64_t>(sw * w_stage16);
#pragma unroll
            for (int sl = 0; sl < 3; ++sl)
              if (sl < cnt) {
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                  tc_mma_bf16(dcol, dAs + sl * w_tap16 + 2 * k, dBs + sl * row16 + 2 * k, idesc, 1u);
              }
          }
          tc_commit(&w_empty[sw]);
          tc_commit(&x_empty[sx]);
        }
        __syncwarp();
        sw = (sw + 1 == p.nw) ? 0 : sw + 1;
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
    // ---- epilogue (warps 3..10): TMEM lane = output channel; columns = pixels of a tile row
    const int q = warp & 3;
    const int sub = (warp - 3) >> 2;   // csplit 1: rows r with r % 2 == sub; csplit 2: half `sub` of the row
    const int hc = p.csplit == 2 ? (((p.npx + 1) / 2 + 31) & ~31) : p.npx;
    const int r_begin = p.csplit == 2 ? 0 : sub, r_step = p.csplit == 2 ? 1 : 2;
    const int c_begin = p.csplit == 2 ? sub * hc : 0, c_end = p.csplit == 2 ? min(p.npx, (sub + 1) * hc) : p.npx;
    const long long stride = static_cast<long long>(g.osx) * g.oC;   // elements between neighbouring pixels
    const bool res_f32 = g.res_f32 != 0;
    const int rsize = res_f32 ? 4 : 2;
    // tma_out == 2: this warp's ring of kResBufs staging buffers; the residual of a 16-pixel sub-chunk is
    // loaded into a buffer two sub-chunks ahead, the output overwrites it in place and is stored from it
    uint8_t* rbuf0 = smem + p.stage_out_off + (warp - 3) * kResBufs * kStageOutBytes;
    uint64_t* rbar = res_full + (warp - 3) * kResBufs;
    int ld_slot = 0, use_slot = 0, pending = 0;   // next slot to load / to consume; loads not yet consumed
    uint32_t use_par = 0u;
    int it = 0;
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++it) {
      const TileT d = decode_tile(p, t);
      const int buf = it % p.nbuf;
      // tma_out == 2 (one-row tiles): this warp's residual sub-chunks, the first two loaded before the
      // accumulator is ready
      const int orow0 = (d.bb * g.oT + d.tt) * g.oH + d.y0;
      const int c_lim = min(c_end, g.W - d.x0);
      const int nsc = (kOut == 2 && d.y0 < g.H && c_lim > c_begin) ? (c_lim - c_begin + 15) / 16 : 0;
      auto issue_res = [&](int i) {   // lane 0: residual of sub-chunk i into the next slot
        bulk_wait_group_read1();      // the store that last used the slot (all but the newest) has read it
        mbar_arrive_expect_tx(&rbar[ld_slot], kStageOutBytes);
        tma_load_3d(rbuf0 + ld_slot * kStageOutBytes, &p.tmR, &rbar[ld_slot], d.m0 + q * 32, d.x0 + c_begin + 16 * i,
                    orow0);
        ld_slot = ld_slot + 1 == kResBufs ? 0 : ld_slot + 1;
        ++pending;
      };
      if (kOut == 2 && lane == 0) {
        for (int i = 0; i < 2 && i < nsc; ++i) issue_res(i);
      }
      const int co = d.m0 + q * 32 + lane;
      const bool cvalid = co < g.Cout;
      const float bias = (p.bias != nullptr && cvalid) ? p.bias[co] : 0.f;
      const int py = d.phase >> 1, px = d.phase & 1;
      auto row_first = [&](int r) -> long long {   // element (first pixel of the tile row, channel 0)
        const int yo = (d.y0 + r) * g.osy + (g.nphase > 1 ? py : 0);
        const long long row_pix =
            ((static_cast<long long>(d.bb) * g.oT + d.tt) * g.oH + yo) * static_cast<long long>(g.oW);
        return (row_pix + static_cast<long long>(d.x0) * g.osx + (g.nphase > 1 ? px : 0)) * g.oC;
      };
      if (p.residual != nullptr && warp == 3 && lane == 0) {
        // pull this tile's residual rows into L2 while its MMAs run (whole pixels, all channels: contiguous)
        const int nv = min(p.npx, g.W - d.x0);
        for (int r = 0; r < p.R && d.y0 + r < g.H; ++r) {
          const char* base = static_cast<const char*>(p.residual) + row_first(r) * rsize;
          const long long bytes = (static_cast<long long>(nv - 1) * stride + g.oC) * rsize;
          for (long long off = 0; off < bytes; off += 32768)
            l2_prefetch_bulk(base + off, static_cast<uint32_t>(min(32768LL, bytes - off)));
        }
      }
      const bool ok = mbar_wait(&acc_full[buf], static_cast<uint32_t>(it / p.nbuf) & 1u, p.status, kErrTimeoutAccum,
                                &abort_flag);
      tc_fence_after();
      if (!__all_sync(0xffffffffu, ok && !abort_flag)) break;
      const uint32_t lane_addr = tmem + static_cast<uint32_t>(buf * p.acc_cols) + (static_cast<uint32_t>(q * 32) << 16);
      const bool has_res = p.residual != nullptr && cvalid;
      for (int r = r_begin; r < p.R; r += r_step) {
        if (d.y0 + r >= g.H) break;   // uniform across the warp
        const long long erow = row_first(r) + co;
        if constexpr (kOut == 2) {
          // one-row tiles: residual and output both pass through this warp's staging ring
          float kshift = 0.f, s1 = 0.f, s2 = 0.f, cnt = 0.f;
          const uint32_t lane4 = 4u * lane;
          for (int i = 0; i < nsc; ++i) {
            const int c0 = c_begin + 16 * i;
            const int nvalid = min(16, c_lim - c0);
            uint32_t rr[16];
            tmem_ld_16x_32x32b(lane_addr + static_cast<uint32_t>(c0), rr);
            uint8_t* sb = rbuf0 + use_slot * kStageOutBytes;
            const uint32_t sa = smem_u32(sb) + lane4;
            const bool okr = mbar_wait(&rbar[use_slot], use_par, p.status, kErrTimeoutAccum, &abort_flag);
            tmem_ld_wait();
            if (!__all_sync(0xffffffffu, okr)) break;
            float v[16];
            const float2 sc2 = make_float2(g.scale, g.scale), b2 = make_float2(bias, bias);
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              float r0, r1;
              asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r0) : "r"(sa + 128u * j) : "memory");
              asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r1) : "r"(sa + 128u * (j + 1)) : "memory");
              float2 t = __ffma2_rn(make_float2(__uint_as_float(rr[j]), __uint_as_float(rr[j + 1])), sc2, b2);
              t = __fadd2_rn(t, cvalid ? make_float2(r0, r1) : make_float2(0.f, 0.f));
              v[j] = t.x;
              v[j + 1] = t.y;
            }
            if (p.gn_part != nullptr) {
              if (i == 0) kshift = v[0];
              gn_sums16(v, nvalid, kshift, s1, s2, cnt);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j)
              asm volatile("st.shared.f32 [%0], %1;" ::"r"(sa + 128u * j), "f"(v[j]) : "memory");
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              // pixels beyond the image width are clipped by the store
              tma_store_3d(&p.tmO, sb, d.m0 + q * 32, d.x0 + c0, orow0);
              bulk_commit_group();
              if (i + 2 < nsc) issue_res(i + 2);
            }
            --pending;
            use_slot = use_slot + 1 == kResBufs ? 0 : use_slot + 1;
            if (use_slot == 0) use_par ^= 1u;
            __syncwarp();   // reconverge before the next warp-wide TMEM load
          }
          if (p.gn_part != nullptr) gn_store(p, d, r, co, cvalid, lane, sub, kshift, s1, s2, cnt);
          continue;
        }
        if constexpr (kOut == 1) {
          // 16-pixel sub-chunks: TMEM -> registers -> this warp's staging rows -> TMA tensor store
          uint8_t* stg = smem + p.stage_out_off + (warp - 3) * kStageOutBytes;
          const uint32_t stg_lane = smem_u32(stg) + 4u * lane;
          uint8_t* stg2 = smem + p.stage_out_off + kEpiWarpsT * kStageOutBytes + (warp - 3) * kStageOut2Bytes;
          const uint32_t stg2_lane = smem_u32(stg2) + 2u * lane;
          const int orow = (d.bb * g.oT + d.tt) * g.oH + (d.y0 + r);
          float rv[16], rn[16];
          auto load_res16 = [&](int c0, float (&dst)[16]) {
            const int nvalid = min(16, min(c_end - c0, g.W - (d.x0 + c0)));
            const float* rp = static_cast<const float*>(p.residual) + erow + static_cast<long long>(c0) * stride;
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[j] = (j < nvalid) ? rp[j * stride] : 0.f;
          };
          if (has_res && c_begin < c_end && d.x0 + c_begin < g.W) load_res16(c_begin, rv);
          float kshift = 0.f, s1 = 0.f, s2 = 0.f, cnt = 0.f;
          for (int c0 = c_begin; c0 < c_end; c0 += 16) {
            const int nvalid = min(16, min(c_end - c0, g.W - (d.x0 + c0)));
            if (nvalid <= 0) break;   // uniform across the warp
            uint32_t rr[16];
            tmem_ld_16x_32x32b(lane_addr + static_cast<uint32_t>(r * p.npx + c0), rr);
            if (has_res && c0 + 16 < c_end && d.x0 + c0 + 16 < g.W) load_res16(c0 + 16, rn);
            tmem_ld_wait();
            float v[16];
            const float2 sc2 = make_float2(g.scale, g.scale), b2 = make_float2(bias, bias);
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              float2 t = __ffma2_rn(make_float2(__uint_as_float(rr[j]), __uint_as_float(rr[j + 1])), sc2, b2);
              if (has_res) t = __fadd2_rn(t, make_float2(rv[j], rv[j + 1]));
              v[j] = t.x;
              v[j + 1] = t.y;
            }
            if (has_res) {
#pragma unroll
              for (int j = 0; j < 16; ++j) rv[j] = rn[j];
            }
            if (p.gn_part != nullptr) {
              if (c0 == c_begin) kshift = v[0];
              gn_sums16(v, nvalid, kshift, s1, s2, cnt);
            }
            // the previous store from this buffer has finished reading it
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              asm volatile("st.shared.f32 [%0], %1;" ::"r"(stg_lane + 128u * j), "f"(v[j]) : "memory");
            if (p.out2 != nullptr) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                asm volatile("st.shared.b16 [%0], %1;" ::"r"(stg2_lane + 64u * j),
                             "h"(__bfloat16_as_ushort(__float2bfloat16_rn(v[j])))
                             : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            // pixels beyond the image width are clipped by the store
            if (lane == 0) {
              tma_store_3d(&p.tmO, stg, d.m0 + q * 32, d.x0 + c0, orow);
              if (p.out2 != nullptr) tma_store_3d(&p.tmO2, stg2, d.m0 + q * 32, d.x0 + c0, orow);
              bulk_commit_group();
            }
            __syncwarp();   // reconverge before the next warp-wide TMEM load
          }
          if (p.gn_part != nullptr) gn_store(p, d, r, co, cvalid, lane, sub, kshift, s1, s2, cnt);
          continue;
        }
        // residual of chunk c0 in rv; the next chunk's loads are issued before this one is used
        float rv[32], rn[32];
        auto load_res = [&](int c0, float (&dst)[32]) {
          const int nvalid = min(32, min(c_end - c0, g.W - (d.x0 + c0)));
          const long long e0 = erow + static_cast<long long>(c0) * stride;
          if (res_f32) {
            const float* rp = static_cast<const float*>(p.residual) + e0;
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[j] = (j < nvalid) ? rp[j * stride] : 0.f;
          } else {
            const __nv_bfloat16* rp = static_cast<const __nv_bfloat16*>(p.residual) + e0;
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[j] = (j < nvalid) ? __bfloat162float(rp[j * stride]) : 0.f;
          }
        };
        if (has_res && c_begin < c_end && d.x0 + c_begin < g.W) load_res(c_begin, rv);
        // GroupNorm moments of this channel over the tile row: sums shifted by the row's first value
        float kshift = 0.f, s1 = 0.f, s2 = 0.f, cnt = 0.f;
        for (int c0 = c_begin; c0 < c_end; c0 += 32) {
          const int nvalid = min(32, min(c_end - c0, g.W - (d.x0 + c0)));
          if (nvalid <= 0) break;   // uniform across the warp
          uint32_t rr[32];
          tmem_ld_32x32b_x32(lane_addr + static_cast<uint32_t>(r * p.npx + c0), rr);
          if (has_res && c0 + 32 < c_end && d.x0 + c0 + 32 < g.W) load_res(c0 + 32, rn);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(rr[j]) * g.scale + bias;
          if (has_res) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += rv[j];
#pragma unroll
            for (int j = 0; j < 32; ++j) rv[j] = rn[j];
          }
          if (p.gn_part != nullptr) {
            if (c0 == c_begin) kshift = v[0];
            float a1[4] = {0.f, 0.f, 0.f, 0.f}, a2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float dv = (j < nvalid) ? v[j] - kshift : 0.f;
              a1[j & 3] += dv;
              a2[j & 3] = fmaf(dv, dv, a2[j & 3]);
            }
            s1 += (a1[0] + a1[1]) + (a1[2] + a1[3]);
            s2 += (a2[0] + a2[1]) + (a2[2] + a2[3]);
            cnt += static_cast<float>(nvalid);
          }
          if (cvalid) {
            const long long e0 = erow + static_cast<long long>(c0) * stride;
            if (g.out_f32) {
              float* op = reinterpret_cast<float*>(p.out) + e0;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < nvalid) op[j * stride] = v[j];
            } else {
              __nv_bfloat16* op = reinterpret_cast<__nv_bfloat16*>(p.out) + e0;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < nvalid) op[j * stride] = __float2bfloat16_rn(v[j]);
            }
            if (p.out2 != nullptr) {
              __nv_bfloat16* op = p.out2 + e0;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < nvalid) op[j * stride] = __float2bfloat16_rn(v[j]);
            }
          }
          __syncwarp();   // reconverge before the next warp-wide TMEM load
        }
        if (p.gn_part != nullptr) gn_store(p, d, r, co, cvalid, lane, sub, kshift, s1, s2, cnt);
      }
      // hand the accumulator buffer back to the MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
    // every staged store has completed before the CTA exits
    if (kOut == 2 && lane == 0) {
      // residual loads issued but not consumed (a stopped decode) land before the CTA exits
      for (; pending > 0; --pending) {
        mbar_drain(&rbar[use_slot], use_par);
        use_slot = use_slot + 1 == kResBufs ? 0 : use_slot + 1;
        if (use_slot == 0) use_par ^= 1u;
      }
    }
    if (kOut != 0 && lane == 0) bulk_wait_group0();
    __syncwarp();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}
int round_up_t(int a, int b) { return (a + b - 1) / b * b; }

}  // namespace

// Channel-major halo kernel: 3x3 spatial taps (in groups of three per kernel row,
// optionally per causal frame or per upsample phase), channels-last output, and
// rows wide enough for at least 96-pixel tiles.
bool conv_halo_t_applicable(const ConvGeom& g) {
  if (g.out_chfirst || g.time_up_c > 0) return false;
  if (g.ntaps != 9 && g.ntaps != 27 && !(g.ntaps == 7 && g.nphase == 4)) return false;
  if (g.W < 96) return false;
  if (g.Cout % 16 != 0 || g.Cin % 16 != 0) return false;
  const int ndt = g.ntaps == 27 ? 3 : 1;
  const int nsp = g.ntaps / ndt;
  for (int ph = 0; ph < g.nphase; ++ph)
    for (int d = 0; d < ndt; ++d)
      for (int s = 0; s < nsp; ++s) {
        const ConvTap t = g.taps[ph][d * nsp + s];
        if (t.dt != g.taps[ph][d * nsp].dt) return false;
        if (t.dy < -1 || t.dy > 1 || t.dx < -1 || t.dx > 1) return false;
      }
  return true;
}

bool conv_halo_t_shortcut_ok(const ConvGeom& g, int sc_cin) {
  // 2D 3x3 convs only (the shortcut stages the tile's centre row); channel chunks of any BK
  return g.ntaps == 9 && g.nphase == 1 && g.T >= 1 && sc_cin > 0 && sc_cin % 64 == 0;
}

cudaError_t launch_conv_halo_t(const ConvGeom& g, const void* in, const void* wts, int ntaps_w, int w_rows,
                               const float* bias, const void* residual, void* out, void* out2, int* status,
                               cudaStream_t stream, const char** why, int* gn_chunks, const ConvShortcut* sc) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return cudaErrorNotSupported;
  }
  HaloTParams p;
  std::memset(&p, 0, sizeof(p));
  p.g = g;
  // pixel tile: split the row into equal tiles of at most 256 pixels (multiple of 16).  Where tiles
  // have at least 192 pixels and the layer is not an upsample, a tile is one row in one of two
  // 256-column accumulator buffers, so its epilogue overlaps the next tile's MMAs; measured on the
  // decoders' layers this wins everywhere except for wide rows (> 256 px) read with more than 256
  // input channels and no residual, where R rows sharing one buffer of up to 512 columns (twice
  // the pixels per weight fetch, fewer re-read halo rows) keep the loads below the TMA rate.
  // Narrower tiles also take R rows (narrower MMAs are shared-memory bound).
  const int ntx = (g.W + 255) / 256;
  p.npx = round_up_t((g.W + ntx - 1) / ntx, 16);
  p.tiles_x = (g.W + p.npx - 1) / p.npx;
  p.half = round_up_t(p.npx + 2, 16) / 2;          // two boxes per staged row, multiple of 8 pixels each
  const bool one_row = g.nphase == 1 && (g.Cin <= 256 || residual != nullptr || g.W <= 256);
  if ((p.npx >= 192 && one_row) || sc != nullptr) {   // a fused shortcut needs one-row tiles
    p.nbuf = 2;
    p.R = 1;
  } else {
    p.nbuf = 1;
    p.R = std::max(1, std::min(4, 512 / p.npx));
  }
  p.acc_cols = 512 / p.nbuf;
  while (p.R > 1 && p.R > g.H) --p.R;
  p.csplit = p.R == 1 ? 2 : 1;
  p.n_mtiles = (g.Cout + 127) / 128;   // weight rows beyond w_rows read as zeros
  int bk = 0;
  for (int cand : {64, 32, 16}) {
    if (g.Cin % cand != 0) continue;
    const int x_stage = (p.R + 2) * 2 * p.half * cand * 2;
    const int w_stage = 3 * 128 * cand * 2;
    if (2 * x_stage + 2 * w_stage <= kPipeBytesT) {
      bk = cand;
      break;
    }
  }
  if (bk == 0) {
    *why = "no channel-major halo tile fits shared memory";
    return cudaErrorInvalidValue;
  }
  p.n_kchunks = g.Cin / bk;
  p.ndt = g.ntaps == 27 ? 3 : 1;
  p.row_bytes = static_cast<uint32_t>(2 * p.half * bk * 2);
  p.x_stage_bytes = static_cast<uint32_t>((p.R + 2) * p.row_bytes);
  p.w_tap_bytes = static_cast<uint32_t>(128 * bk * 2);
  p.w_stage_bytes = 3 * p.w_tap_bytes;
  p.nw = std::min(kMaxWStages, static_cast<int>((kPipeBytesT - 2 * p.x_stage_bytes) / p.w_stage_bytes));
  p.tiles_y = (g.H + p.R - 1) / p.R;
  p.tmem_cols = 512;
  p.bias = bias;
  p.residual = residual;
  p.out = out;
  p.out2 = static_cast<__nv_bfloat16*>(out2);
  p.status = status;
  if (g.gn_part != nullptr && g.gn_groups > 0 && g.out_f32 && g.Cout % g.gn_groups == 0) {
    const int cg = g.Cout / g.gn_groups;
    if (cg <= 32 && 32 % cg == 0) {
      p.gn_part = static_cast<GnPartial*>(g.gn_part);
      p.gn_cg = cg;
      if (gn_chunks != nullptr) *gn_chunks = g.oT * g.oH * (g.nphase > 1 ? 2 : 1) * p.tiles_x * p.csplit;
    }
  }

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
      *why = "channel-major halo activation tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)g.Cin, (cuuint64_t)ntaps_w, (cuuint64_t)w_rows};
    const cuuint64_t strides[2] = {dims[0] * 2, dims[0] * dims[1] * 2};
    const cuuint32_t box[3] = {(cuuint32_t)bk, 1, 128};
    if (enc(&p.tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(wts), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "channel-major halo weight tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  if (sc != nullptr) {
    if (p.R != 1 || sc->cin % bk != 0 || (reinterpret_cast<uintptr_t>(sc->in) & 15) ||
        (reinterpret_cast<uintptr_t>(sc->w) & 15)) {
      *why = "shortcut fusion needs one-row tiles and 16-byte aligned operands";
      return cudaErrorInvalidValue;
    }
    p.sc_chunks = sc->cin / bk;
    p.n_sc = (p.sc_chunks + 2) / 3;
    {
      const cuuint64_t dims[5] = {(cuuint64_t)sc->cin, (cuuint64_t)g.W, (cuuint64_t)g.H, (cuuint64_t)g.T,
                                  (cuuint64_t)g.B};
      const cuuint64_t strides[4] = {dims[0] * 2, dims[0] * dims[1] * 2, dims[0] * dims[1] * dims[2] * 2,
                                     dims[0] * dims[1] * dims[2] * dims[3] * 2};
      const cuuint32_t box[5] = {(cuuint32_t)bk, (cuuint32_t)p.half, 1, 1, 1};
      if (enc(&p.tmX2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(sc->in), dims, strides, box, ones,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        *why = "shortcut input tensor map rejected";
        return cudaErrorInvalidValue;
      }
    }
    {
      const cuuint64_t dims[3] = {(cuuint64_t)sc->cin, 1, (cuuint64_t)sc->w_rows};
      const cuuint64_t strides[2] = {dims[0] * 2, dims[0] * 2};
      const cuuint32_t box[3] = {(cuuint32_t)bk, 1, 128};
      if (enc(&p.tmW2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(sc->w), dims, strides, box, ones,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(bk), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        *why = "shortcut weight tensor map rejected";
        return cudaErrorInvalidValue;
      }
    }
  }
  // fp32 channels-last output with whole 32-channel quarters: store through shared memory with TMA
  size_t smem = 2 * (size_t)p.x_stage_bytes + (size_t)p.nw * p.w_stage_bytes + 1024;
  // (not where a residual is read in a serial epilogue: there the 32-pixel chunks' deeper residual
  // loads of the direct stores win)
  const size_t stage1 = (size_t)kEpiWarpsT * (kStageOutBytes + (out2 != nullptr ? kStageOut2Bytes : 0));
  if (g.out_f32 && g.nphase == 1 && g.osx == 1 && g.osy == 1 && g.Cout % 32 == 0 &&
      (p.nbuf == 2 || residual == nullptr) &&
      g.oC == g.Cout && (residual == nullptr || g.res_f32) && (reinterpret_cast<uintptr_t>(out) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(out2) & 15) == 0 && smem + stage1 <= (size_t)kMaxDynSmemT) {
    const cuuint64_t dims[3] = {(cuuint64_t)g.oC, (cuuint64_t)g.oW, (cuuint64_t)g.B * g.oT * g.oH};
    const cuuint64_t strides[2] = {dims[0] * 4, dims[0] * dims[1] * 4};
    const cuuint32_t box[3] = {32, 16, 1};
    if (enc(&p.tmO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      p.tma_out = 1;
      // one-row tiles with an fp32 residual: the residual also comes by TMA, through a ring of three
      // staging buffers per warp (room taken from the fourth weight stage)
      const int nw3 = std::min(p.nw, 3);
      const size_t smem3 = 2 * (size_t)p.x_stage_bytes + (size_t)nw3 * p.w_stage_bytes + 1024 +
                           (size_t)kEpiWarpsT * kResBufs * kStageOutBytes;
      if (out2 != nullptr) {
        const cuuint64_t strides2[2] = {dims[0] * 2, dims[0] * dims[1] * 2};
        if (enc(&p.tmO2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out2, dims, strides2, box, ones,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
          p.tma_out = 0;
      }
      if (p.tma_out == 1 && out2 == nullptr && residual != nullptr && p.nbuf == 2 && p.R == 1 && p.csplit == 2 &&
          nw3 >= 3 &&
          (reinterpret_cast<uintptr_t>(residual) & 15) == 0 && smem3 <= (size_t)kMaxDynSmemT &&
          enc(&p.tmR, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(residual), dims, strides, box, ones,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
        p.tma_out = 2;
        p.nw = nw3;
        smem = smem3;
      } else if (p.tma_out == 1) {
        smem += stage1;
      }
      p.stage_out_off = 2 * p.x_stage_bytes + static_cast<uint32_t>(p.nw) * p.w_stage_bytes;
    }
  }
  const long long ntiles = (long long)g.B * g.T * p.tiles_y * p.tiles_x * g.nphase * p.n_mtiles;
  if (ntiles <= 0) return cudaSuccess;
  if (ntiles > 0x7fffffffLL) {
    *why = "grid too large";
    return cudaErrorInvalidValue;
  }
  p.ntiles = static_cast<int>(ntiles);
  // persistent: one CTA per SM (the pipeline fills shared memory), tiles dealt round-robin
  int dev = 0, sms = 0;
  cudaError_t ea = cudaGetDevice(&dev);
  if (ea == cudaSuccess) ea = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ea != cudaSuccess) return ea;
  const long long nblocks = std::min<long long>(ntiles, std::max(1, sms));
  cudaError_t e;
  auto go = [&](auto kern) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (r == cudaSuccess) launch_pdl(kern, (unsigned)nblocks, kThreadsT, smem, stream, p);
    return r;
  };
  if (g.ntaps == 7) {
    // upsample convs in the two-by-two phase form: the serial epilogue (no TMA stores)
    if (p.tma_out != 0) {
      *why = "the two-by-two upsample form has no TMA-store epilogue";
      return cudaErrorInvalidValue;
    }
    switch (bk) {
      case 64: e = go(conv_halo_t_kernel<64, 0, 7>); break;
      case 32: e = go(conv_halo_t_kernel<32, 0, 7>); break;
      default: e = go(conv_halo_t_kernel<16, 0, 7>); break;
    }
  } else {
    switch (bk * 4 + p.tma_out) {
      case 64 * 4 + 0: e = go(conv_halo_t_kernel<64, 0, 9>); break;
      case 64 * 4 + 1: e = go(conv_halo_t_kernel<64, 1, 9>); break;
      case 64 * 4 + 2: e = go(conv_halo_t_kernel<64, 2, 9>); break;
      case 32 * 4 + 0: e = go(conv_halo_t_kernel<32, 0, 9>); break;
      case 32 * 4 + 1: e = go(conv_halo_t_kernel<32, 1, 9>); break;
      case 32 * 4 + 2: e = go(conv_halo_t_kernel<32, 2, 9>); break;
      case 16 * 4 + 0: e = go(conv_halo_t_kernel<16, 0, 9>); break;
      case 16 * 4 + 1: e = go(conv_halo_t_kernel<16, 1, 9>); break;
      default: e = go(conv_halo_t_kernel<16, 2, 9>); break;
    }
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

VD_WAIT_LIMIT_SETTER(set_wait_limit_conv_halo_t)

}  // namespace vd
