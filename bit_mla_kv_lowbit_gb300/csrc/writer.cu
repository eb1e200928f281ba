// Fused cache writer.
//
// QuantMLA, Figure 8 caption: the writer packs each token as it arrives, all
// tokens alike, and keeps the unquantised bf16 values of the protected sink
// and recent tokens in separate buffers.  One warp handles one
// 64-channel group of one token (9 warps per token): a warp-wide min/max,
// fp16 scale and min, round-half-to-even codes, nibble/crumb packing, and the
// bf16 copies.  The arithmetic is the float32 definition in mla_lowbit.h, done
// with explicitly rounded intrinsics so that it is bit-exact regardless of
// compiler contraction.
#include "common.cuh"

namespace mlalb {

template <int CB>
__global__ void __launch_bounds__(kGroups * 32) writer_kernel(WriterArgs a) {
  constexpr PageGeom G = page_geom(CB);
  const int i = blockIdx.x;
  const int g = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int s = a.seq_idx ? a.seq_idx[i] : i;
  const int p = a.pos[i];
  if (s < 0 || s >= a.num_seqs) {
    if (threadIdx.x == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_SEQ);
    return;
  }
  if (p < 0 || p >= a.max_pages * kPageTokens) {
    if (threadIdx.x == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_POS);
    return;
  }
  const long long page = a.block_table[(long long)s * a.max_pages + p / kPageTokens];
  if (page < 0 || page >= a.num_pages) {
    if (threadIdx.x == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
    return;
  }
  const int row = p % kPageTokens;
  uint8_t* base = a.pool + page * G.page_bytes;

  // Lane holds channels (2*lane, 2*lane+1) of this group.
  const uint32_t v = g < 8 ? a.ckv[(long long)i * (kLatent / 2) + g * 32 + lane]
                           : a.krope[(long long)i * (kRope / 2) + lane];

  if constexpr (CB == 16) {
    reinterpret_cast<uint32_t*>(base + row * G.content_row)[g * 32 + lane] = v;
    return;
  } else {
    // bf16 copies of protected tokens.
    if (p < kSink) a.sink[((long long)s * kSink + p) * (kDim / 2) + g * 32 + lane] = v;
    const int len_after = a.lens_after ? a.lens_after[s] : p + 1;
    if (p >= len_after - kLocal)
      a.recent[((long long)s * kLocal + p % kLocal) * (kDim / 2) + g * 32 + lane] = v;

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
      seg = base + G.content_off + row * G.content_row + g * (G.content_row / 8);
    else
      seg = base + G.rope_off + row * G.rope_row;
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
      *reinterpret_cast<uint32_t*>(base + G.meta_off + row * G.meta_row + g * 4) = meta;
    }
  }
}

cudaError_t launch_writer(int cbits, const WriterArgs& a, cudaStream_t stream) {
  if (a.n_tokens == 0) return cudaSuccess;
  dim3 grid(a.n_tokens), block(kGroups * 32);
  switch (cbits) {
    case 4: writer_kernel<4><<<grid, block, 0, stream>>>(a); break;
    case 2: writer_kernel<2><<<grid, block, 0, stream>>>(a); break;
    case 16: writer_kernel<16><<<grid, block, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mlalb
