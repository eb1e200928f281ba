// The writer's arithmetic for one 64-channel group of one token, shared by the
// stand-alone writer kernel and the decode kernel's fused append.
//
// QuantMLA, Figure 8 caption: every incoming token is packed as it arrives.
// One warp quantises one group: lane l holds channels (2l, 2l+1) as a bf16
// pair; a warp-wide min/max gives the fp16 scale and min (float32 arithmetic
// with explicitly rounded intrinsics, so the bytes are independent of
// compiler contraction), codes are rounded half to even, clamped and packed.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace mlalb {

// Online rotation of one 64-channel content group held by a warp as bf16 pairs
// (lane l: channels 2l, 2l+1): R x with R = H_64 / 8, float32 butterflies in
// the layout's order (stage h pairs element i, bit h clear, with i + h into
// (a + b, a - b); h = 1 inside the lane, h >= 2 across lanes l ^ h/2), then
// x 1/8 (exact), rounded to bf16 (nearest even).  All 32 lanes must call it.
__device__ __forceinline__ uint32_t rotate_group_bf16(uint32_t v, int lane) {
  const float a = bf16lo_to_f32(v), b = bf16hi_to_f32(v);
  float x0 = __fadd_rn(a, b), x1 = __fsub_rn(a, b);
#pragma unroll
  for (int hl = 1; hl < 32; hl <<= 1) {
    const float p0 = __shfl_xor_sync(0xffffffffu, x0, hl);
    const float p1 = __shfl_xor_sync(0xffffffffu, x1, hl);
    if (lane & hl) {  // this element is the second of its pair: partner - own
      x0 = __fsub_rn(p0, x0);
      x1 = __fsub_rn(p1, x1);
    } else {
      x0 = __fadd_rn(x0, p0);
      x1 = __fadd_rn(x1, p1);
    }
  }
  const __nv_bfloat162 r = __floats2bfloat162_rn(x0 * 0.125f, x1 * 0.125f);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Quantise and store group g (0..7 content, 8 RoPE) of the token in row `row`
// of the packed page at `page_base`.  All 32 lanes of the warp must call it.
template <int CB>
__device__ __forceinline__ void write_packed_group(uint8_t* page_base, int row, int g, int lane,
                                                   uint32_t v) {
  constexpr PageGeom G = page_geom(CB);
  const int bits = g < 8 ? CB : 4;
  const int levels = (1 << bits) - 1;
  const float x0 = bf16lo_to_f32(v), x1 = bf16hi_to_f32(v);
  float mn = fminf(x0, x1), mx = fmaxf(x0, x1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  mn = __fadd_rn(mn, 0.0f);  // a zero minimum is stored as +0
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), (float)levels);
  const __half s16 = __float2half_rn(fminf(s32, 65504.0f));
  const __half m16 = __float2half_rn(fminf(fmaxf(mn, -65504.0f), 65504.0f));
  const float sf = __half2float(s16), mf = __half2float(m16);
  int c0 = 0, c1 = 0;
  if (sf != 0.0f) {
    c0 = __float2int_rn(__fdiv_rn(__fsub_rn(x0, mf), sf));
    c1 = __float2int_rn(__fdiv_rn(__fsub_rn(x1, mf), sf));
    c0 = min(max(c0, 0), levels);
    c1 = min(max(c1, 0), levels);
  }
  uint8_t* seg;
  if (g < 8)
    seg = page_base + G.content_off + row * G.content_row + g * (G.content_row / 8);
  else
    seg = page_base + G.rope_off + row * G.rope_row;
  if (bits == 4) {
    seg[lane] = static_cast<uint8_t>(c0 | (c1 << 4));
  } else {
    const int nib = c0 | (c1 << 2);
    const int other = __shfl_down_sync(0xffffffffu, nib, 1);
    if ((lane & 1) == 0) seg[lane >> 1] = static_cast<uint8_t>(nib | (other << 4));
  }
  if (lane == 0) {
    const uint32_t meta = static_cast<uint32_t>(__half_as_ushort(s16)) |
                          (static_cast<uint32_t>(__half_as_ushort(m16)) << 16);
    *reinterpret_cast<uint32_t*>(page_base + G.meta_off + row * G.meta_row + g * 4) = meta;
  }
}

}  // namespace mlalb
