// Shared definitions of the low-bit MLA decode kernels (sm_103a).
//
// Geometry of the packed page (QuantMLA, Figure 3 / Figure 8 captions: packed
// content and RoPE codes with per-group metadata; the byte layout itself is
// this library's choice and is documented in include/mla_lowbit.h).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mla_lowbit.h"

namespace mlalb {

constexpr int kLatent = 512;
constexpr int kRope = 64;
constexpr int kDim = kLatent + kRope;  // 576
constexpr int kGroup = 64;
constexpr int kGroups = kDim / kGroup;  // 9: 8 content + 1 RoPE
constexpr int kPageTokens = 64;
constexpr int kSink = 4;
constexpr int kLocal = 128;
constexpr int kProtected = kSink + kLocal;

// Byte offsets inside one page for content bits 4 / 2 / 16 (bf16 page).
struct PageGeom {
  int content_off, content_row, rope_off, rope_row, meta_off, meta_row, page_bytes;
};

__host__ __device__ constexpr PageGeom page_geom(int cbits) {
  return cbits == 16
             ? PageGeom{0, kDim * 2, 0, 0, 0, 0, kPageTokens * kDim * 2}
             : PageGeom{0,
                        kLatent * cbits / 8,
                        kPageTokens * (kLatent * cbits / 8),
                        kRope / 2,
                        kPageTokens * (kLatent * cbits / 8) + kPageTokens * (kRope / 2),
                        kGroups * 4,
                        kPageTokens * (kLatent * cbits / 8) + kPageTokens * (kRope / 2) +
                            kPageTokens * kGroups * 4};
}

static_assert(page_geom(4).page_bytes == 20736, "C4R4 page");
static_assert(page_geom(2).page_bytes == 12544, "C2R4 page");
static_assert(page_geom(16).page_bytes == 73728, "bf16 page");

__device__ __forceinline__ void set_error(int32_t* err, int bits) {
  if (err) atomicOr(reinterpret_cast<int*>(err), bits);
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) {
  return __uint_as_float(v & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D += A(16x16, row) * B(16x8, col), fp16 inputs, fp32 accumulate.  A pure
// register operation (not volatile), so the compiler may interleave
// independent accumulation chains.
__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t* r, const void* p) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, const void* p) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

// Split planning shared by host and device.
//
// Pages of a sequence that hold at least one packed-served token (for bf16
// pages: every page).
__host__ __device__ inline int packed_pages_of(int L, bool packed) {
  if (L <= 0) return 0;
  if (!packed) return (L + kPageTokens - 1) / kPageTokens;
  if (L <= kProtected) return 0;
  // packed-served tokens are 4 .. L-129
  return (L - kLocal - 1) / kPageTokens + 1;
}
// Protected tokens a packed layout serves from its bf16 buffers: the sink
// tokens 0 .. min(L,4)-1, then the recent tokens max(4, L-128) .. L-1.
__host__ __device__ inline int bf16_tokens_of(int L, bool packed) {
  if (!packed || L <= 0) return 0;
  const int n_sink = L < kSink ? L : kSink;
  const int rec_start = L - kLocal > kSink ? L - kLocal : kSink;
  return n_sink + (L > rec_start ? L - rec_start : 0);
}
// Work units of a sequence: its pages (above), one unit each, then its
// protected bf16 tokens in 64-token tiles of kBf16TileUnits units each (a tile
// of bf16 rows read from the bf16 buffers costs about that many packed pages).
// Splits cut the units into chunks of chunk_pages; a bf16 tile belongs to the
// split that holds its first unit.
constexpr int kBf16TileUnits = 3;
__host__ __device__ inline int bf16_tiles_of(int L, bool packed) {
  return (bf16_tokens_of(L, packed) + kPageTokens - 1) / kPageTokens;
}
__host__ __device__ inline int units_of(int L, bool packed) {
  return packed_pages_of(L, packed) + kBf16TileUnits * bf16_tiles_of(L, packed);
}
__host__ __device__ inline int splits_of(int L, bool packed, int chunk_pages) {
  const int s = (units_of(L, packed) + chunk_pages - 1) / chunk_pages;
  return s > 0 ? s : 1;
}

// Kernel argument blocks (filled by the host ABI in api.cu).
struct WriterArgs {
  const uint32_t* ckv;    // [n][512] bf16, read as bf16 pairs
  const uint32_t* krope;  // [n][64] bf16
  const int32_t* seq_idx;
  const int32_t* pos;
  const int32_t* lens_after;
  const int32_t* block_table;
  uint8_t* pool;
  uint32_t* sink;    // [S][4][576] bf16 as pairs
  uint32_t* recent;  // [S][128][576] bf16 as pairs
  int32_t* err;
  long long num_pages;
  int n_tokens, num_seqs, max_pages;
  int rotate = 0;  // online Hadamard rotation of the content latent (layout field)
};

struct DecodeArgs {
  const uint16_t* q;  // [B][H][576] bf16
  const uint8_t* pool;
  long long num_pages;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const uint16_t* sink;    // [B][4][576] bf16
  const uint16_t* recent;  // [B][128][576] bf16
  float* part_o;           // [total_splits][H][512]
  float* part_ml;          // [total_splits][H][2] (running max in log2 units, sum)
  int32_t* seq_split;      // [B][2] (first split, split count)
  int32_t* err;
  int B, H, max_pages, chunk_pages, total_splits;
  float scale_log2;  // softmax_scale * log2(e)
  // Queries per sequence: the H rows of a sequence are n_q blocks of H / n_q
  // heads, query i at position seq_lens[b] - n_q + i (causal among them).
  int n_q = 1;
  int rotate = 0;  // the cache's content latent is stored rotated (layout field)
  // Bounded waits of the tcgen05 kernels give up after this many SM clock
  // cycles (about one second by default).  fault = 1 (self-test only) makes
  // the 128-row kernel's unpack warps skip their first hand-off, so that the
  // waits downstream of it run out.
  long long wait_cycles = 2000000000LL;
  int fault = 0;
  // Fused append (mla_lowbit_write_decode): the token at position
  // seq_lens[b] - 1 of every sequence, written by the sequence's bf16 split of
  // head chunk 0 and read from here by every bf16 split.  Null for a plain decode.
  const uint32_t* new_ckv = nullptr;  // [B][256] bf16 pairs
  const uint32_t* new_kr = nullptr;   // [B][32] bf16 pairs
  uint8_t* pool_w = nullptr;          // the page pool, writable
  uint32_t* sink_w = nullptr;         // [B][4][288] bf16 pairs
  uint32_t* recent_w = nullptr;       // [B][128][288] bf16 pairs
};

cudaError_t launch_writer(int cbits, const WriterArgs& a, cudaStream_t stream);
cudaError_t launch_decode(int cbits, const DecodeArgs& a, float* out, float* lse,
                          cudaStream_t stream);
// True when launch_decode can append each sequence's new token itself (the
// DecodeArgs new_* fields): the default split kernel on a packed layout.
bool decode_fuses_append(int cbits, int rotate, int rows);
// CTAs that process one split (head chunks of 16, or one 2-CTA cluster per
// 128-row block for the tcgen05 kernel): the planner sizes chunks so that all
// fit one wave.
int decode_ctas_per_split(int cbits, int rows, int rotate);
// Most work units (pages) one split may hold: it bounds the number of
// accumulating MMAs into one fp32 tensor-core output (whose adds are not
// round-to-nearest) and the split's page list in shared memory.
int decode_max_split_pages(int cbits, int rows, int rotate);
cudaError_t launch_decode_wide(int cbits, const DecodeArgs& a, cudaStream_t stream);
// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (device, kernel): the limit is a per-device attribute.
// Thread-safe.
cudaError_t ensure_smem_limit(const void* kernel, int bytes);

}  // namespace mlalb
