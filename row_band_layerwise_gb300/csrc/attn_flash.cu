// Fused band attention on tcgen05 tensor cores: softmax(Q K^T / sqrt(C)) V with band-local queries
// against every key and value of the frame ("VAEP：VAE 并行解码", section Attention：本地 Q，全局 K/V;
// "Static Layer-Wise VAE Decode", Semantics: attention keeps Q local and K/V global).
//
// One work item is (query tile of 128 rows, channel half of the output, key range).  The scores of a
// 128-query x 128-key block are computed into tensor memory, exponentiated in registers (one query
// row per thread, running maximum and row sum in fp32) and written back over their own scores as
// bf16 probabilities, which the probabilities x values MMA reads straight from tensor memory into
// the output accumulator; the accumulator stays in tensor memory for the whole key range, and
// nothing of size queries x keys ever reaches shared or global memory.  At C = 512 a 128-row output
// accumulator would fill all 512 TMEM columns, so each item owns one channel half (256 columns) next
// to two 128-column score buffers, and the two halves of a tile compute the same scores
// (bit-identical: the same MMAs on the same operands).
//
// The running maximum is updated lazily: the probabilities of a block are taken against the largest
// score seen so far only when it exceeds the maximum in use by more than 2^8 (in the exponent's
// units); until then the old maximum stays, the probabilities stay below 2^8, and no rescaling of
// the accumulator is needed.  Softmax is invariant to the shift, and the row sum is taken over the
// same stored (bf16-rounded) probabilities the product uses.  Every decision depends on the query
// row's own scores only, so a row's result is the same whatever band or tile holds it.
//
// Roles (256 threads): warp 0 streams the query tile and the key stages through the key ring, warp 2
// the value stages through the value ring; warp 1 (TMEM owner) issues the score MMAs, up to two
// blocks ahead of the softmax (two score buffers), and warp 3 the probabilities x values MMAs as soon
// as a block's probabilities are in tensor memory; warps 4..7 run the softmax and the output (warp w
// owns TMEM lanes 32 (w % 4) ...).  Keys and values have rings of their own, so the keys of the next
// blocks keep streaming while a block's values wait for its probabilities.  Every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "kernels.h"
#include "ptx.cuh"
#include "tma_host.h"
#include "launch.h"

namespace vd {

namespace {

constexpr int kFThreads = 256;
constexpr int kFSlot = 16384;         // one 128-byte-swizzled atom column: 128 rows x 64 bf16
constexpr int kFKSlot = 2 * kFSlot;   // key slot: 128 keys x 128 channels (8 MMAs per commit)
constexpr int kFMaxStages = 8;
constexpr uint32_t kFSCol = 256;      // TMEM column of score buffer 0 (buffer 1 at + 128)
constexpr float kFRescale = 8.f;      // lazy-maximum threshold, log2 units

struct FlashParams {
  CUtensorMap tmQ;   // (C, F * ntok) box (64, 128)
  CUtensorMap tmK;   // (C, ntok, F) box (64, 128, 1)
  CUtensorMap tmV;   // (ntok, C, F) box (64, C / 2, 1)
  int C, half_c, ck, kst;   // ck 64-channel atoms of Q; kst key stages (128 channels) per block
  long long ntok, rows;
  int nkb, splits, F;
  int U, seg_q, seg_rem, n_seg, t_big, t_small, tiles_per_frame;
  int n_tiles, n_items, nk, nv;   // key and value ring slots
  uint32_t vslot;                  // value slot bytes: C/2 channels x 64 keys
  float scale_log2;
  __nv_bfloat16* out;
  float* part;
  float2* ml;
  int* status;
};

struct FItem {
  long long q0;
  int nq, f, half, split, kb0, kb1;
};

// Item t: channel half fastest, then query tile, then key split.
__device__ __forceinline__ FItem flash_item(const FlashParams& p, int t) {
  FItem d;
  d.half = t & 1;
  t >>= 1;
  const int tile = t % p.n_tiles;
  d.split = t / p.n_tiles;
  d.f = tile / p.tiles_per_frame;
  const int tt = tile - d.f * p.tiles_per_frame;
  const int big = p.seg_rem * p.t_big;
  int seg, tis;
  if (tt < big) {
    seg = tt / p.t_big;
    tis = tt - seg * p.t_big;
  } else {
    const int r = tt - big;
    seg = p.seg_rem + r / p.t_small;
    tis = r - (seg - p.seg_rem) * p.t_small;
  }
  const long long seg_start = (long long)seg * p.seg_q + min(seg, p.seg_rem);
  const long long seg_len = (long long)(p.seg_q + (seg < p.seg_rem ? 1 : 0)) * p.U;
  d.q0 = (long long)d.f * p.ntok + seg_start * p.U + (long long)tis * 128;
  d.nq = static_cast<int>(min(128LL, seg_len - (long long)tis * 128));
  d.kb0 = static_cast<int>((long long)d.split * p.nkb / p.splits);
  d.kb1 = static_cast<int>((long long)(d.split + 1) * p.nkb / p.splits);
  return d;
}

// Named barrier 1 over the 128 softmax threads (warps 4..7), returning the AND of `v` over them.
__device__ __forceinline__ bool softmax_and(bool v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred pv, pr;\n\tsetp.ne.s32 pv, %1, 0;\n\tbar.red.and.pred pr, 1, 128, pv;\n\t"
      "selp.s32 %0, 1, 0, pr;\n\t}"
      : "=r"(r)
      : "r"(static_cast<int>(v))
      : "memory");
  return r != 0;
}

// 2^x with the hardware's approximate base-2 exponential (PTX ex2.approx.ftz.f32).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi, float& sum) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  const float2 r = __bfloat1622float2(h);
  sum += r.x;
  sum += r.y;
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kFThreads, 1) attn_flash_kernel(const __grid_constant__ FlashParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t kfull[kFMaxStages], kempty[kFMaxStages], vfull[kFMaxStages], vempty[kFMaxStages];
  __shared__ __align__(8) uint64_t q_full, q_empty, s_full[2], p_free[2], p_full[2], o_full, o_free;
  __shared__ __align__(8) uint64_t s_done, v_done;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smQ = smem;                        // ck atoms of 128 rows x 64 channels
  uint8_t* kring = smQ + p.ck * kFSlot;       // nk slots of 128 keys x 128 channels
  uint8_t* vring = kring + p.nk * kFKSlot;    // nv slots of C/2 channels x 64 keys

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.nk; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < p.nv; ++i) {
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
    }
    mbar_init(&q_full, 1);
    mbar_init(&q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_free[i], 1);
      // probabilities ready, per block parity: the softmax can finish block g + 1 before the product
      // has observed block g (block g + 2 needs block g's product), so one barrier could run two
      // phases ahead of the product's parity wait
      mbar_init(&p_full[i], 1);
    }
    mbar_init(&o_full, 1);
    mbar_init(&o_free, 1);
    mbar_init(&s_done, 1);
    mbar_init(&v_done, 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmQ);
    tma_prefetch_desc(&p.tmK);
  }
  if (warp == 2 && lane == 0) tma_prefetch_desc(&p.tmV);
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();   // the previous kernel on the stream has finished and its writes are visible
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ---- K producer: each item's query tile, then the key stages of every block in order
    if (lane == 0) {
      int g = 0, it = 0, qn = 0;   // key stages and query tiles issued
      int s = 0;                   // slot of key stage g and the parity of the empty phase that frees it
      uint32_t epar = 1u;
      for (int t = blockIdx.x; t < p.n_items && !abort_flag; t += gridDim.x, ++it) {
        const FItem d = flash_item(p, t);
        if (it >= 1 && !mbar_wait(&q_empty, static_cast<uint32_t>(it - 1) & 1u, p.status, kErrTimeoutEmpty,
                                  &abort_flag))
          break;
        if (abort_flag) break;
        mbar_arrive_expect_tx(&q_full, static_cast<uint32_t>(p.ck) * kFSlot);
        for (int i = 0; i < p.ck; ++i)
          tma_load_3d(smQ + i * kFSlot, &p.tmQ, &q_full, i * 64, static_cast<int>(d.q0), 0);
        ++qn;
        bool stop = false;
        for (int kb = d.kb0; kb < d.kb1 && !stop; ++kb) {
          for (int kc = 0; kc < p.kst; ++kc) {
            if ((g >= p.nk && !mbar_wait(&kempty[s], epar, p.status, kErrTimeoutEmpty, &abort_flag)) || abort_flag) {
              stop = true;
              break;
            }
            mbar_arrive_expect_tx(&kfull[s], kFKSlot);
            tma_load_3d(kring + s * kFKSlot, &p.tmK, &kfull[s], kc * 128, kb * 128, d.f);
            tma_load_3d(kring + s * kFKSlot + kFSlot, &p.tmK, &kfull[s], kc * 128 + 64, kb * 128, d.f);
            ++g;
            if (++s == p.nk) {
              s = 0;
              epar ^= 1u;
            }
          }
        }
        if (stop) break;
      }
      if (abort_flag) {
        // let the copies already issued land before the CTA exits
        for (int i = max(0, g - p.nk); i < g; ++i) mbar_drain(&kfull[i % p.nk], static_cast<uint32_t>(i / p.nk) & 1u);
        if (qn > 0) mbar_drain(&q_full, static_cast<uint32_t>(qn - 1) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ---- V producer: the value stages of every block (the item's channel half, keys 64 b ..)
    if (lane == 0) {
      const uint32_t v_tx = p.vslot;
      int g = 0;
      int s = 0;              // slot of value stage g and the parity of the empty phase that frees it
      uint32_t epar = 1u;
      bool stop = false;
      for (int t = blockIdx.x; t < p.n_items && !abort_flag && !stop; t += gridDim.x) {
        const FItem d = flash_item(p, t);
        for (int kb = d.kb0; kb < d.kb1 && !stop; ++kb) {
          for (int v = 0; v < 2; ++v) {
            if ((g >= p.nv && !mbar_wait(&vempty[s], epar, p.status, kErrTimeoutEmpty, &abort_flag)) || abort_flag) {
              stop = true;
              break;
            }
            mbar_arrive_expect_tx(&vfull[s], v_tx);
            tma_load_3d(vring + s * p.vslot, &p.tmV, &vfull[s], kb * 128 + v * 64, d.half * p.half_c, d.f);
            ++g;
            if (++s == p.nv) {
              s = 0;
              epar ^= 1u;
            }
          }
        }
      }
      if (abort_flag)
        for (int i = max(0, g - p.nv); i < g; ++i) mbar_drain(&vfull[i % p.nv], static_cast<uint32_t>(i / p.nv) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- score MMAs: S(g) = Q K^T into buffer g & 1, as soon as block g - 2's probabilities in that
    // buffer have been used
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, 128);
      const uint64_t dQ0 = smem_desc_kmajor(smem_u32(smQ), 1024, 2);
      const uint64_t dK0 = smem_desc_kmajor(smem_u32(kring), 1024, 2);
      int it = 0;
      int s = 0;              // key slot of the next stage, and the parity of its full phase: running
      uint32_t kpar = 0u;     // counts, so the issue loop has no division between two MMA groups
      long long sg = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x, ++it) {
        const FItem d = flash_item(p, t);
        ok = mbar_wait(&q_full, static_cast<uint32_t>(it) & 1u, p.status, kErrTimeoutFull, &abort_flag);
        for (int kb = d.kb0; kb < d.kb1 && ok; ++kb, ++sg) {
          if (sg >= 2)   // the probabilities this buffer held (block sg - 2) have been multiplied out
            ok = mbar_wait(&p_free[sg & 1], (static_cast<uint32_t>(sg >> 1) & 1u) ^ 1u, p.status, kErrTimeoutEmpty,
                           &abort_flag);
          const uint32_t dS = tmem + kFSCol + static_cast<uint32_t>(sg & 1) * 128u;
          for (int kc = 0; kc < p.kst && ok; ++kc) {
            ok = mbar_wait(&kfull[s], kpar, p.status, kErrTimeoutFull, &abort_flag);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t da = dQ0 + static_cast<uint64_t>((2 * kc + h) * (kFSlot >> 4));
              const uint64_t db = dK0 + static_cast<uint64_t>((s * 2 + h) * (kFSlot >> 4));
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tc_mma_bf16(dS, da + 2 * k, db + 2 * k, idesc_s, (kc | h | k) != 0 ? 1u : 0u);
            }
            tc_commit(&kempty[s]);
            if (++s == p.nk) {
              s = 0;
              kpar ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit(&s_full[sg & 1]);
          if (kb == d.kb1 - 1) tc_commit(&q_empty);
        }
      }
      // every MMA issued has completed before the CTA releases TMEM (also after a timeout)
      tc_commit(&s_done);
      mbar_drain(&s_done, 0);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ---- probabilities x values MMAs: O += P[:, keys 64 b ..] V^T[half, keys 64 b ..]^T (N = C/2), P read
    // from tensor memory
    if (lane == 0) {
      const uint32_t idesc_v = idesc_bf16_f32(128, p.half_c);
      const uint64_t dV0 = smem_desc_kmajor(smem_u32(vring), 1024, 2);
      int it = 0;
      int s = 0;              // value slot of the next stage and the parity of its full phase (running counts)
      uint32_t vpar = 0u;
      long long pg = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.n_items && ok; t += gridDim.x, ++it) {
        const FItem d = flash_item(p, t);
        for (int kb = d.kb0; kb < d.kb1 && ok; ++kb, ++pg) {
          const bool first = kb == d.kb0;
          // the block's probabilities are in tensor memory (and the accumulator rescaled); before the
          // item's first block, the previous item's output has also been read out of the accumulator
          ok = mbar_wait(&p_full[pg & 1], static_cast<uint32_t>(pg >> 1) & 1u, p.status, kErrTimeoutFull, &abort_flag);
          if (ok && first && it >= 1)
            ok = mbar_wait(&o_free, static_cast<uint32_t>(it - 1) & 1u, p.status, kErrTimeoutEmpty, &abort_flag);
          for (int b = 0; b < 2 && ok; ++b) {
            ok = mbar_wait(&vfull[s], vpar, p.status, kErrTimeoutFull, &abort_flag);
            if (!ok) break;
            tc_fence_after();
            // P of the block: 64 columns of its score buffer, keys 2c and 2c + 1 in column c
            const uint32_t ta = tmem + kFSCol + static_cast<uint32_t>(pg & 1) * 128u + static_cast<uint32_t>(b * 32);
            const uint64_t db = dV0 + static_cast<uint64_t>(s * (p.vslot >> 4));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_bf16_tmem_a(tmem, ta + 8 * k, db + 2 * k, idesc_v, (!first || b != 0 || k != 0) ? 1u : 0u);
            tc_commit(&vempty[s]);
            if (++s == p.nv) {
              s = 0;
              vpar ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit(&p_free[pg & 1]);
          if (kb == d.kb1 - 1) tc_commit(&o_full);
        }
      }
      tc_commit(&v_done);
      mbar_drain(&v_done, 0);
    }
    __syncwarp();
  } else {
    // ---- softmax and output, warps 4..7: query row r = TMEM lane.  A failed (timed-out) wait only
    // marks `ok` false and skips the tensor-memory work that depended on it; the four warps decide to
    // leave together at the block's sync point (an AND over their 128 threads), so none of them can
    // be left waiting at the named barrier.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl = p.scale_log2;
    long long sg = 0;
    int it = 0;
    bool ok = true, dead = false;
    for (int t = blockIdx.x; t < p.n_items && !dead; t += gridDim.x, ++it) {
      const FItem d = flash_item(p, t);
      const int nb = d.kb1 - d.kb0;
      float m_use = 0.f, l = 0.f;
      for (int jj = 0; jj < nb; ++jj) {
        if (ok) ok = mbar_wait(&s_full[sg & 1], static_cast<uint32_t>(sg >> 1) & 1u, p.status, kErrTimeoutAccum,
                               &abort_flag);
        ok = __all_sync(0xffffffffu, ok && !abort_flag);
        const uint32_t sbuf = lane_base + kFSCol + static_cast<uint32_t>(sg & 1) * 128u;
        uint32_t sr[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) sr[i] = 0u;
        if (ok) {
          tc_fence_after();
          uint32_t (&c0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sr[0]);
          uint32_t (&c1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sr[32]);
          uint32_t (&c2)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sr[64]);
          uint32_t (&c3)[32] = *reinterpret_cast<uint32_t (*)[32]>(&sr[96]);
          tmem_ld_32x32b_x32(sbuf, c0);
          tmem_ld_32x32b_x32(sbuf + 32, c1);
          tmem_ld_32x32b_x32(sbuf + 64, c2);
          tmem_ld_32x32b_x32(sbuf + 96, c3);
          tmem_ld_wait();
        }
        // keys past the end of the frame (the last block) take no weight
        const long long kbase = (long long)(d.kb0 + jj) * 128;
        if (kbase + 128 > p.ntok) {
          const int nvalid = static_cast<int>(p.ntok - kbase);
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= nvalid) sr[i] = __float_as_uint(-INFINITY);
        }
        // block maximum: eight independent chains, then a fixed tree
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = __uint_as_float(sr[i]);
#pragma unroll
        for (int i = 8; i < 128; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[i]));
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float mt = mx * sl;
        bool resc = false;
        float alpha = 1.f;
        if (jj == 0) {
          m_use = mt;
          l = 0.f;
        } else if (mt > m_use + kFRescale) {
          alpha = ex2(m_use - mt);
          m_use = mt;
          l *= alpha;
          resc = true;
        }
        // probabilities of the block as bf16, and their sum (of the stored values) in four chains
        const float nm = -m_use;
        uint32_t pw[64];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 64; ++i)
          pw[i] = pack_bf16(ex2(fmaf(__uint_as_float(sr[2 * i]), sl, nm)),
                            ex2(fmaf(__uint_as_float(sr[2 * i + 1]), sl, nm)), ls[i & 3]);
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // P replaces the scores in their buffer (this thread's row, columns 0..63)
        if (ok) {
          const uint32_t (&p0)[32] = *reinterpret_cast<const uint32_t (*)[32]>(&pw[0]);
          const uint32_t (&p1)[32] = *reinterpret_cast<const uint32_t (*)[32]>(&pw[32]);
          tmem_st_32x32b_x32(sbuf, p0);
          tmem_st_32x32b_x32(sbuf + 32, p1);
          tmem_st_wait();
        }
        // block sg - 1's product (its buffer's p_free phase) must have finished before the accumulator
        // is rescaled
        const long long pv = sg - 1;
        const uint32_t pv_par = static_cast<uint32_t>(pv >> 1) & 1u;
        bool waited = false;
        if (ok && jj >= 1 && __any_sync(0xffffffffu, resc)) {
          ok = mbar_wait(&p_free[pv & 1], pv_par, p.status, kErrTimeoutAccum, &abort_flag);
          ok = __all_sync(0xffffffffu, ok && !abort_flag);
          waited = true;
          if (ok) {
            tc_fence_after();
            // rows whose maximum moved multiply their accumulator row by alpha (the others by 1)
            for (int c0 = 0; c0 < p.half_c; c0 += 32) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(c0), o);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st_32x32b_x32(lane_base + static_cast<uint32_t>(c0), o);
            }
            tmem_st_wait();
          }
        }
        // all four warps have written (and rescaled) their rows before one thread signals the block:
        // arrivals never run ahead into the next block's phase
        tc_fence_before();
        if (!softmax_and(ok)) {
          dead = true;
          break;
        }
        if (r == 0) mbar_arrive(&p_full[sg & 1]);
        if (jj >= 1 && !waited) {
          // keep step with the barrier: one wait per phase (nothing later can complete it again first);
          // a failure here is acted on at the next sync point
          ok = mbar_wait(&p_free[pv & 1], pv_par, p.status, kErrTimeoutAccum, &abort_flag);
          ok = __all_sync(0xffffffffu, ok && !abort_flag);
        }
        ++sg;
      }
      if (dead) break;
      // ---- output of the item; the last product (its buffer's p_free phase) completed with o_full
      if (ok) ok = mbar_wait(&o_full, static_cast<uint32_t>(it) & 1u, p.status, kErrTimeoutAccum, &abort_flag);
      if (ok)
        ok = mbar_wait(&p_free[(sg - 1) & 1], static_cast<uint32_t>((sg - 1) >> 1) & 1u, p.status, kErrTimeoutAccum,
                       &abort_flag);
      ok = __all_sync(0xffffffffu, ok && !abort_flag);
      if (ok) {
        tc_fence_after();
        const bool valid = r < d.nq;
        const long long row = d.q0 + r;
        if (p.splits == 1) {
          const float inv = 1.f / l;
          __nv_bfloat16* orow = p.out + row * p.C + d.half * p.half_c;
          for (int c0 = 0; c0 < p.half_c; c0 += 32) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(c0), o);
            tmem_ld_wait();
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(o[q * 8 + 2 * i]) * inv,
                                                                 __uint_as_float(o[q * 8 + 2 * i + 1]) * inv);
                  w[i] = *reinterpret_cast<const uint32_t*>(&h);
                }
                dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
          }
        } else {
          float* prow = p.part + ((long long)d.split * p.rows + row) * p.C + d.half * p.half_c;
          for (int c0 = 0; c0 < p.half_c; c0 += 32) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(c0), o);
            tmem_ld_wait();
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(prow + c0);
#pragma unroll
              for (int q = 0; q < 8; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            }
          }
          if (valid && d.half == 0) p.ml[(long long)d.split * p.rows + row] = make_float2(m_use, l);
        }
      }
      tc_fence_before();
      if (!softmax_and(ok)) break;
      if (r == 0) mbar_arrive(&o_free);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// out[row, c] = sum_s 2^(m_s - M) O_s[row, c] / sum_s 2^(m_s - M) l_s, M = max_s m_s, splits in order.
__global__ void attn_combine_kernel(const float* __restrict__ part, const float2* __restrict__ ml,
                                    __nv_bfloat16* __restrict__ out, long long rows, int C, int splits) {
  pdl_wait();
  const int c4 = C >> 2;
  const long long n = rows * c4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / c4;
    const int c = static_cast<int>(i - row * c4) * 4;
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, ml[s * rows + row].x);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < splits; ++s) {
      const float2 q = ml[s * rows + row];
      const float w = exp2f(q.x - M);
      den = fmaf(w, q.y, den);
      const float4 v = *reinterpret_cast<const float4*>(part + (s * rows + row) * C + c);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    const float inv = 1.f / den;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + row * C + c) = u;
  }
}

}  // namespace

// Key splits: a function of the key count only (every band plan merges the same partials in the
// same order); one split per 2048 keys, at most 4.
int flash_splits(long long ntok) { return static_cast<int>(std::max(1LL, std::min(4LL, ntok / 2048))); }

size_t flash_work_bytes(int F, long long ntok, int C) {
  const int s = flash_splits(ntok);
  if (s <= 1) return 0;
  const size_t rows = static_cast<size_t>(F) * static_cast<size_t>(ntok);
  return static_cast<size_t>(s) * rows * (static_cast<size_t>(C) * sizeof(float) + sizeof(float2));
}

cudaError_t launch_attn_flash(const FlashArgs& a, int* status, cudaStream_t stream, const char** why) {
  *why = nullptr;
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return cudaErrorNotSupported;
  }
  if (a.F < 1 || a.ntok < 1) return cudaSuccess;
  if (a.C < 128 || a.C > 512 || a.C % 128 != 0) {
    *why = "fused attention needs C a multiple of 128, at most 512";
    return cudaErrorInvalidValue;
  }
  if (a.ntok % 8 != 0) {
    *why = "fused attention needs a multiple of 8 keys per frame";
    return cudaErrorInvalidValue;
  }
  if (a.U < 1 || a.n_seg < 1 || a.seg_q < 1 || a.seg_rem < 0 || a.seg_rem >= a.n_seg ||
      (long long)(a.seg_q * (long long)a.n_seg + a.seg_rem) * a.U != a.ntok) {
    *why = "fused attention: band segments do not cover the frame";
    return cudaErrorInvalidValue;
  }
  if ((reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) | reinterpret_cast<uintptr_t>(a.vt) |
       reinterpret_cast<uintptr_t>(a.out)) & 15) {
    *why = "fused attention operands must be 16-byte aligned";
    return cudaErrorInvalidValue;
  }
  FlashParams p;
  std::memset(&p, 0, sizeof(p));
  p.C = a.C;
  p.half_c = a.C / 2;
  p.ck = a.C / 64;
  p.kst = a.C / 128;
  p.ntok = a.ntok;
  p.F = a.F;
  p.rows = (long long)a.F * a.ntok;
  p.nkb = static_cast<int>((a.ntok + 127) / 128);
  p.splits = std::min(flash_splits(a.ntok), p.nkb);
  if (p.splits > 1 && (a.part == nullptr || a.ml == nullptr ||
                       ((reinterpret_cast<uintptr_t>(a.part) | reinterpret_cast<uintptr_t>(a.ml)) & 15))) {
    *why = "fused attention needs 16-byte aligned partial buffers for its key splits";
    return cudaErrorInvalidValue;
  }
  p.U = a.U;
  p.seg_q = a.seg_q;
  p.seg_rem = a.seg_rem;
  p.n_seg = a.n_seg;
  p.t_big = static_cast<int>(((long long)(a.seg_q + 1) * a.U + 127) / 128);
  p.t_small = static_cast<int>(((long long)a.seg_q * a.U + 127) / 128);
  p.tiles_per_frame = a.seg_rem * p.t_big + (a.n_seg - a.seg_rem) * p.t_small;
  const long long n_tiles = (long long)a.F * p.tiles_per_frame;
  const long long n_items = n_tiles * 2 * p.splits;
  if (n_items > 0x7fffffffLL || p.rows > 0x7fffffffLL) {
    *why = "fused attention has too many query tiles";
    return cudaErrorInvalidValue;
  }
  p.n_tiles = static_cast<int>(n_tiles);
  p.n_items = static_cast<int>(n_items);
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt((double)a.C));
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.part = a.part;
  p.ml = static_cast<float2*>(a.ml);
  p.status = status;
  const size_t fixed = static_cast<size_t>(p.ck) * kFSlot + 1024;
  const long long budget = 227LL * 1024 - 1024 - (long long)fixed;   // 1 KB for the static shared memory
  // two key slots, the rest for values (C = 512: one value slot, C = 384: two)
  p.vslot = static_cast<uint32_t>(p.half_c) * 128u;
  p.nk = 2;
  p.nv = static_cast<int>(std::min<long long>(kFMaxStages, (budget - 2LL * kFKSlot) / p.vslot));
  if (p.nv < 1) {
    *why = "fused attention does not fit in shared memory";
    return cudaErrorInvalidValue;
  }
  const cuuint32_t ones[3] = {1, 1, 1};
  {
    const cuuint64_t dims[3] = {(cuuint64_t)a.C, (cuuint64_t)p.rows, 1};
    const cuuint64_t strides[2] = {(cuuint64_t)a.C * 2, (cuuint64_t)a.C * 2 * p.rows};
    const cuuint32_t box[3] = {64, 128, 1};
    if (enc(&p.tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "fused attention query tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)a.C, (cuuint64_t)a.ntok, (cuuint64_t)a.F};
    const cuuint64_t strides[2] = {(cuuint64_t)a.C * 2, (cuuint64_t)a.C * 2 * a.ntok};
    const cuuint32_t box[3] = {64, 128, 1};
    if (enc(&p.tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.k), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "fused attention key tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)a.ntok, (cuuint64_t)a.C, (cuuint64_t)a.F};
    const cuuint64_t strides[2] = {(cuuint64_t)a.ntok * 2, (cuuint64_t)a.ntok * 2 * a.C};
    const cuuint32_t box[3] = {64, (cuuint32_t)p.half_c, 1};
    if (enc(&p.tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.vt), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      *why = "fused attention value tensor map rejected";
      return cudaErrorInvalidValue;
    }
  }
  const size_t smem = fixed + static_cast<size_t>(p.nk) * kFKSlot + static_cast<size_t>(p.nv) * p.vslot;
  cudaError_t e = cudaFuncSetAttribute(attn_flash_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.n_items, std::max(1, sms));
  return launch_pdl(attn_flash_kernel, grid, kFThreads, smem, stream, p);
}

cudaError_t launch_attn_combine(const FlashArgs& a, cudaStream_t stream) {
  const int nkb = static_cast<int>((a.ntok + 127) / 128);
  const int splits = std::min(flash_splits(a.ntok), nkb);
  if (splits <= 1 || a.F < 1 || a.ntok < 1) return cudaSuccess;
  const long long rows = (long long)a.F * a.ntok;
  const long long n = rows * (a.C / 4);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, (long long)std::max(1, sms) * 8));
  return launch_pdl(attn_combine_kernel, blocks, 256, 0, stream, static_cast<const float*>(a.part),
                    static_cast<const float2*>(a.ml), static_cast<__nv_bfloat16*>(a.out), rows, a.C, splits);
}

VD_WAIT_LIMIT_SETTER(set_wait_limit_attn_flash)

}  // namespace vd
