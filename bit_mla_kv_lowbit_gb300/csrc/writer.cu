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
#include "writer_common.cuh"

namespace mlalb {

template <int CB>
__global__ void __launch_bounds__(kGroups * 32) writer_kernel(WriterArgs a) {
  constexpr PageGeom G = page_geom(CB);
  const int i = blockIdx.x;
  const int g = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int s = a.seq_idx ? a.seq_idx[i] : i;
  if (!a.pos && (s < 0 || s >= a.num_seqs)) {  // appending: token i is sequence i's
    if (threadIdx.x == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_SEQ);
    return;
  }
  const int p = a.pos ? a.pos[i] : a.lens_after[s] - 1;
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
  uint32_t v = g < 8 ? a.ckv[(long long)i * (kLatent / 2) + g * 32 + lane]
                     : a.krope[(long long)i * (kRope / 2) + lane];
  if (a.rotate && g < 8) v = rotate_group_bf16(v, lane);  // whole warp: g is warp-uniform

  if constexpr (CB == 16) {
    reinterpret_cast<uint32_t*>(base + row * G.content_row)[g * 32 + lane] = v;
    return;
  } else {
    // bf16 copies of protected tokens.
    if (p < kSink) a.sink[((long long)s * kSink + p) * (kDim / 2) + g * 32 + lane] = v;
    const int len_after = a.lens_after ? a.lens_after[s] : p + 1;
    if (p >= len_after - kLocal)
      a.recent[((long long)s * kLocal + p % kLocal) * (kDim / 2) + g * 32 + lane] = v;

    write_packed_group<CB>(base, row, g, lane, v);
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
