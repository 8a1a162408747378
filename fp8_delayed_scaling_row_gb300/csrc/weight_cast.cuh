// The weight casts of a forward call, carried by the LayerNorm forward launch
// (layernorm.cu): code = fp8(w * scale) for every element of up to two bf16
// weight tensors, with max|w| folded into each tensor's running amax (TE
// tutorial, code block 1: the module casts its weight to FP8 with the scale
// of its forward state every step). The casts and the LayerNorm are
// independent and both HBM-bound, so one launch runs both: each CTA of the
// LayerNorm grid first takes its share of the weights' 128 x 64 tiles (the
// loads of its first LayerNorm rows already in flight), then normalises rows.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace lnfp8 {

constexpr int kWTileRows = 128;
constexpr int kWTileCols = 64;
constexpr int kWThreads = 256;  // the block size of every kernel that calls weight_cast_tiles

// Tiles t = blockIdx.x, blockIdx.x + gridDim.x, ... of the job (tensor 0's
// tiles first). Thread t owns the 8-column vector t % 8 of a tile and its rows
// t / 8 + 32 h, h < 4; all four 16-byte loads are issued before any convert.
template <int DT>
__device__ inline void weight_cast_tiles(const WeightCastJob& j) {
  __shared__ uint32_t wred[2][kWThreads / 32];
  const int t = threadIdx.x, cv = t & 7, rr = t >> 3;
  const int64_t total = j.tiles[0] + j.tiles[1];
  uint32_t am0 = 0u, am1 = 0u;
  for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
    // tensor k's fields by selects (a runtime index into the parameter arrays would copy them to local memory)
    const bool k = tile >= j.tiles[0];
    const int64_t lt = k ? tile - j.tiles[0] : tile;
    const int64_t cols = k ? j.cols[1] : j.cols[0], rows = k ? j.rows[1] : j.rows[0];
    const int64_t strips = (cols + kWTileCols - 1) / kWTileCols;
    const int64_t c = (lt % strips) * kWTileCols + cv * 8;
    const int64_t r0 = (lt / strips) * kWTileRows + rr;
    if (c >= cols) continue;
    const uint16_t* __restrict__ in = k ? j.in[1] : j.in[0];
    uint8_t* __restrict__ out = k ? j.out[1] : j.out[0];
    uint4 u[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int64_t r = r0 + 32 * h;
      u[h] = r < rows ? *reinterpret_cast<const uint4*>(in + r * cols + c) : make_uint4(0u, 0u, 0u, 0u);
    }
    const float s = k ? *j.scale[1] : *j.scale[0];
    uint32_t m = 0u;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int64_t r = r0 + 32 * h;
      if (r >= rows) continue;
      const uint32_t w[4] = {u[h].x, u[h].y, u[h].z, u[h].w};
      float v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
        v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) m = max(m, abs_bits(v[i]));
      *reinterpret_cast<uint2*>(out + r * cols + c) = cvt_fp8x8<DT>(v, s);
    }
    if (k) am1 = max(am1, m);
    else am0 = max(am0, m);
  }
  // both tensors' block maxima in one exchange round, then one atomic each
  const int w = t >> 5, l = t & 31;
  am0 = warp_max_u32(am0);
  am1 = warp_max_u32(am1);
  if (l == 0) {
    wred[0][w] = am0;
    wred[1][w] = am1;
  }
  __syncthreads();
  if (w < 2) {
    uint32_t v = l < kWThreads / 32 ? wred[w][l] : 0u;
    v = warp_max_u32(v);
    float* amax = w ? j.amax[1] : j.amax[0];
    if (l == 0 && v != 0u && (w ? j.tiles[1] : j.tiles[0]) > 0) atomic_max_amax(amax, v);
  }
  __syncthreads();
}

}  // namespace lnfp8
