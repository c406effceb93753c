// Epilogue helpers shared by the tensor-core conv kernels: 16 consecutive output
// channels of one pixel are scaled, biased, summed with a residual (fp32 or bf16)
// and stored channels-last (fp32 or bf16, optionally also as a bf16 copy) or
// channels-first, following the ConvGeom output mapping.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "conv.h"

namespace vd {

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 16 consecutive channels of one pixel: 64-byte (fp32) or 32-byte (bf16) vector
// accesses when all 16 are valid, scalar otherwise.
__device__ __forceinline__ void add_f32x16(float (&v)[16], const float* r, int n) {
  if (n == 16) {
    const float4* r4 = reinterpret_cast<const float4*>(r);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 a = r4[j];
      v[4 * j] += a.x;
      v[4 * j + 1] += a.y;
      v[4 * j + 2] += a.z;
      v[4 * j + 3] += a.w;
    }
  } else {
    for (int j = 0; j < n; ++j) v[j] += r[j];
  }
}

__device__ __forceinline__ void add_bf16x16(float (&v)[16], const __nv_bfloat16* r, int n) {
  if (n == 16) {
    const uint4* rp = reinterpret_cast<const uint4*>(r);
    uint4 r0 = rp[0], r1 = rp[1];
    const __nv_bfloat16* h0 = reinterpret_cast<const __nv_bfloat16*>(&r0);
    const __nv_bfloat16* h1 = reinterpret_cast<const __nv_bfloat16*>(&r1);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] += __bfloat162float(h0[j]);
      v[8 + j] += __bfloat162float(h1[j]);
    }
  } else {
    for (int j = 0; j < n; ++j) v[j] += __bfloat162float(r[j]);
  }
}

__device__ __forceinline__ void store_f32x16(float* o, const float (&v)[16], int n) {
  if (n == 16) {
    float4* o4 = reinterpret_cast<float4*>(o);
#pragma unroll
    for (int j = 0; j < 4; ++j) o4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  } else {
    for (int j = 0; j < n; ++j) o[j] = v[j];
  }
}

__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* o, const float (&v)[16], int n) {
  if (n == 16) {
    uint4 w0, w1;
    w0.x = pack_bf16x2(v[0], v[1]);
    w0.y = pack_bf16x2(v[2], v[3]);
    w0.z = pack_bf16x2(v[4], v[5]);
    w0.w = pack_bf16x2(v[6], v[7]);
    w1.x = pack_bf16x2(v[8], v[9]);
    w1.y = pack_bf16x2(v[10], v[11]);
    w1.z = pack_bf16x2(v[12], v[13]);
    w1.w = pack_bf16x2(v[14], v[15]);
    reinterpret_cast<uint4*>(o)[0] = w0;
    reinterpret_cast<uint4*>(o)[1] = w1;
  } else {
    for (int j = 0; j < n; ++j) o[j] = __float2bfloat16_rn(v[j]);
  }
}


// Store 16 accumulator values (already scaled and biased) of output pixel
// (bb, grid frame tt, output row yo, output column xo), channels co0..co0+15.
__device__ __forceinline__ void epilogue_store16(const ConvGeom& g, float (&v)[16], int bb, int tt, int yo, int xo,
                                                 int co0, const void* residual, void* out, __nv_bfloat16* out2) {
  int to = tt, ch0 = co0;
  if (g.time_up_c > 0) {
    const int half = co0 >= g.time_up_c ? 1 : 0;
    to = 1 + 2 * tt + half;
    ch0 = co0 - half * g.time_up_c;
  }
  const long long opix = ((static_cast<long long>(bb) * g.oT + to) * g.oH + yo) * g.oW + xo;
  const int nvalid = min(16, g.Cout - co0);
  if (!g.out_chfirst) {
    const long long base = opix * g.oC + ch0;
    if (residual != nullptr) {
      if (g.res_f32)
        add_f32x16(v, reinterpret_cast<const float*>(residual) + base, nvalid);
      else
        add_bf16x16(v, reinterpret_cast<const __nv_bfloat16*>(residual) + base, nvalid);
    }
    if (g.out_f32)
      store_f32x16(reinterpret_cast<float*>(out) + base, v, nvalid);
    else
      store_bf16x16(reinterpret_cast<__nv_bfloat16*>(out) + base, v, nvalid);
    if (out2 != nullptr) store_bf16x16(out2 + base, v, nvalid);
  } else {
    // channels-first [B][oC][oT][oH][oW]
    const long long plane = static_cast<long long>(g.oT) * g.oH * g.oW;
    const long long sp = (static_cast<long long>(to) * g.oH + yo) * g.oW + xo;
    for (int j = 0; j < nvalid; ++j) {
      const long long a = (static_cast<long long>(bb) * g.oC + ch0 + j) * plane + sp;
      if (g.out_f32)
        reinterpret_cast<float*>(out)[a] = v[j];
      else
        reinterpret_cast<__nv_bfloat16*>(out)[a] = __float2bfloat16_rn(v[j]);
    }
  }
}

}  // namespace vd

namespace vd {

// ---------------------------------------------------------------------------
// Warp-cooperative channels-last epilogue.
//
// A warp holds 32 output pixels (one per lane) x NC consecutive channels.  Each
// lane's NC values are one contiguous row in global memory (NC * 4 B fp32 or
// NC * 2 B bf16), but rows of neighbouring lanes are C_out channels apart, so
// lane-direct vector stores would touch 32 separate sectors per instruction.
// Instead the rows go through a per-warp shared-memory stage (32 rows, 16-byte
// chunks XOR-swizzled by row) and are written with lanes spread along the rows:
// every store instruction then covers whole 128-byte lines.  Residual rows are
// read the same way.
// ---------------------------------------------------------------------------
constexpr int kEpiStageBytes = 32 * 128;   // per warp

__device__ __forceinline__ uint4* stage_chunk(uint8_t* stage, int row, int chunk, int nchunks) {
  return reinterpret_cast<uint4*>(stage + row * nchunks * 16 + ((chunk ^ (row & (nchunks - 1))) * 16));
}

// Move 32 rows of `nchunks` 16-byte chunks between global memory (row of lane p
// starts at that lane's `grow`) and the stage.  kStore: stage -> global.
template <bool kStore>
__device__ __forceinline__ void coalesced_rows(uint8_t* stage, char* grow, bool valid, int nchunks, int lane) {
  const int rows_per_step = 32 / nchunks;
  for (int s = 0; s < nchunks; ++s) {
    const int p = s * rows_per_step + lane / nchunks;
    const int j = lane % nchunks;
    char* gp = reinterpret_cast<char*>(__shfl_sync(0xffffffffu, reinterpret_cast<long long>(grow), p));
    const int ok = __shfl_sync(0xffffffffu, valid ? 1 : 0, p);
    if (ok) {
      if (kStore)
        *reinterpret_cast<uint4*>(gp + j * 16) = *stage_chunk(stage, p, j, nchunks);
      else
        *stage_chunk(stage, p, j, nchunks) = *reinterpret_cast<const uint4*>(gp + j * 16);
    }
  }
}

__device__ __forceinline__ void put_row_f32(uint8_t* stage, int lane, const float* v, int nc) {
  const int nch = nc / 4;
  for (int j = 0; j < nch; ++j)
    *reinterpret_cast<float4*>(stage_chunk(stage, lane, j, nch)) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

__device__ __forceinline__ void put_row_bf16(uint8_t* stage, int lane, const float* v, int nc) {
  const int nch = nc / 8;
  for (int j = 0; j < nch; ++j) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * j], v[8 * j + 1]);
    w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
    w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
    w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
    *stage_chunk(stage, lane, j, nch) = w;
  }
}

// Channels-last epilogue of one NC-column chunk (NC = 16 or 32) for the 32 pixels of a warp.
// `v` holds this lane's accumulator values already scaled and biased; `base` is the element
// offset of this lane's pixel at the chunk's first output channel; `valid` masks pixels outside
// the image.  All lanes of the warp must call this together.
template <int NC>
__device__ __forceinline__ void epi_chunk_cl(const ConvGeom& g, float (&v)[32], long long base, bool valid,
                                             const void* residual, void* out, __nv_bfloat16* out2, uint8_t* stage,
                                             int lane) {
  if (residual != nullptr) {
    if (g.res_f32) {
      coalesced_rows<false>(stage, reinterpret_cast<char*>(const_cast<float*>(reinterpret_cast<const float*>(residual) + base)),
                            valid, NC / 4, lane);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < NC / 4; ++j) {
        const float4 f = *reinterpret_cast<const float4*>(stage_chunk(stage, lane, j, NC / 4));
        v[4 * j] += f.x;
        v[4 * j + 1] += f.y;
        v[4 * j + 2] += f.z;
        v[4 * j + 3] += f.w;
      }
    } else {
      coalesced_rows<false>(stage, reinterpret_cast<char*>(const_cast<__nv_bfloat16*>(reinterpret_cast<const __nv_bfloat16*>(residual) + base)),
                            valid, NC / 8, lane);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < NC / 8; ++j) {
        const uint4 u = *stage_chunk(stage, lane, j, NC / 8);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(h[k]);
          v[8 * j + 2 * k] += f.x;
          v[8 * j + 2 * k + 1] += f.y;
        }
      }
    }
    __syncwarp();
  }
  if (g.out_f32) {
    put_row_f32(stage, lane, v, NC);
    __syncwarp();
    coalesced_rows<true>(stage, reinterpret_cast<char*>(reinterpret_cast<float*>(out) + base), valid, NC / 4, lane);
  } else {
    put_row_bf16(stage, lane, v, NC);
    __syncwarp();
    coalesced_rows<true>(stage, reinterpret_cast<char*>(reinterpret_cast<__nv_bfloat16*>(out) + base), valid, NC / 8,
                         lane);
  }
  __syncwarp();
  if (out2 != nullptr) {
    put_row_bf16(stage, lane, v, NC);
    __syncwarp();
    coalesced_rows<true>(stage, reinterpret_cast<char*>(out2 + base), valid, NC / 8, lane);
    __syncwarp();
  }
}

}  // namespace vd
