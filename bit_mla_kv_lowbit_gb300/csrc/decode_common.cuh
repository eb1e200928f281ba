// Device helpers shared by the decode kernels: the channel pairing of the
// nibble/crumb unpack, the unpack itself, hi/lo splitting and the split lookup.
#pragma once

#include "common.cuh"

namespace mlalb {

constexpr int kHC = 16;  // heads per CTA

// ---------------------------------------------------------------- pairing
// The unpack of one thread's 16 channels (16j..16j+15 of a group) yields 8
// fp16 pairs P_0..P_7.  INT4 ("type A"): P_i = (8(i>>2) + (i&3), +4).  INT2
// ("type B"): P_i = (i, i+8).  mma k-step s takes b0 = P_2s, b1 = P_2s+1.

__device__ __forceinline__ int phys_of_logical(int k, bool typeB) {
  const int s = k >> 4, h = (k >> 3) & 1, j = (k >> 1) & 3, e = k & 1;
  const int i = 2 * s + h;
  return typeB ? 16 * j + i + 8 * e : 16 * j + 8 * (i >> 2) + (i & 3) + 4 * e;
}

// Inverse of phys_of_logical.
__device__ __forceinline__ int logical_of_phys(int p, bool typeB) {
  const int j = p >> 4, rem = p & 15;
  int i, e;
  if (typeB) {
    e = rem >> 3;
    i = rem & 7;
  } else {
    e = (rem >> 2) & 1;
    i = 4 * (rem >> 3) + (rem & 3);
  }
  return 16 * (i >> 1) + 8 * (i & 1) + 2 * j + e;
}

// Physical channel of PV output column n (0..7) of tile chunk c (0..7).
__device__ __forceinline__ int phys_of_chunk(int c, int n, bool typeB) {
  const int jj = c >> 1, wd = c & 1, r = n >> 1, e = n & 1, i = 4 * wd + r;
  return typeB ? 16 * jj + i + 8 * e : 16 * jj + 8 * wd + r + 4 * e;
}

__device__ __forceinline__ uint32_t h2fma(uint32_t x, uint32_t m, uint32_t a) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<__half2*>(&m),
                      *reinterpret_cast<__half2*>(&a));
  return *reinterpret_cast<uint32_t*>(&r);
}

constexpr uint32_t kMagic = 0x64006400u;  // fp16 1024 in both halves

// Codes are centred before they reach the tensor cores (INT4: c - 8 in
// [-8, 7]; INT2: c - 2 in [-2, 1]) and the min is moved by the same amount
// (m' = m + 8s or m + 2s).  The products stay exact; the point is that the MMA
// sums over thousands of tokens then have mixed signs, so the fp32 tensor-core
// accumulation, whose adds are not round-to-nearest, does not drift.
constexpr int kCentre4 = 8;
constexpr int kCentre2 = 2;

// 8 nibbles (channels 0..7 of the word) -> (c0,c4) (c1,c5) (c2,c6) (c3,c7), minus 8.
__device__ __forceinline__ void unpack_int4(uint32_t w, uint32_t* p) {
  const uint32_t w8 = w >> 8;
  p[0] = h2fma((w & 0x000F000Fu) | kMagic, 0x3C003C00u, 0xE408E408u);   // x*1 - 1032
  p[1] = h2fma((w & 0x00F000F0u) | kMagic, 0x2C002C00u, 0xD480D480u);   // x/16 - 72
  p[2] = h2fma((w8 & 0x000F000Fu) | kMagic, 0x3C003C00u, 0xE408E408u);
  p[3] = h2fma((w8 & 0x00F000F0u) | kMagic, 0x2C002C00u, 0xD480D480u);
}

// 16 crumbs (channels 0..15) -> (c0,c8) (c1,c9) ... (c7,c15), minus 2.
__device__ __forceinline__ void unpack_int2(uint32_t w, uint32_t* p) {
  const uint32_t w8 = w >> 8;
  p[0] = h2fma((w & 0x00030003u) | kMagic, 0x3C003C00u, 0xE402E402u);   // x - 1026
  p[1] = h2fma((w & 0x000C000Cu) | kMagic, 0x34003400u, 0xDC08DC08u);   // x/4 - 258
  p[2] = h2fma((w & 0x00300030u) | kMagic, 0x2C002C00u, 0xD420D420u);   // x/16 - 66
  p[3] = h2fma((w & 0x00C000C0u) | kMagic, 0x24002400u, 0xCC80CC80u);   // x/64 - 18
  p[4] = h2fma((w8 & 0x00030003u) | kMagic, 0x3C003C00u, 0xE402E402u);
  p[5] = h2fma((w8 & 0x000C000Cu) | kMagic, 0x34003400u, 0xDC08DC08u);
  p[6] = h2fma((w8 & 0x00300030u) | kMagic, 0x2C002C00u, 0xD420D420u);
  p[7] = h2fma((w8 & 0x00C000C0u) | kMagic, 0x24002400u, 0xCC80CC80u);
}

// 16 bf16 values (v[k] = channels 2k, 2k+1) -> fp16 pairs in the given pairing.
template <bool kB>
__device__ __forceinline__ void pairs_from_bf16(const uint32_t* v, uint32_t* p) {
  float f[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    f[2 * k] = bf16lo_to_f32(v[k]);
    f[2 * k + 1] = bf16hi_to_f32(v[k]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int a = kB ? i : 8 * (i >> 2) + (i & 3);
    const int b = kB ? i + 8 : a + 4;
    p[i] = pack_half2(f[a], f[b]);
  }
}

__device__ __forceinline__ void split_hi_lo(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_half2(a - hf.x, b - hf.y);
}

// ---------------------------------------------------------------- split work
// Units [split * chunk, (split + 1) * chunk) of a sequence of length L: packed
// pages page_begin .. page_begin + n_pages - 1, then bf16 tiles bf_begin ..
// bf_begin + n_bf - 1 (the tiles whose first unit falls in the range); bf16
// tile k holds protected tokens 64k .. 64k + 63 of the list (sink tokens
// 0 .. n_sink - 1, then recent tokens from rec_start), n_tok in all, in
// bf_total tiles.  has_last: the split holds the last protected token.
struct SplitWork {
  int page_begin, n_pages, bf_begin, n_bf, n_sink, rec_start, n_tok, bf_total;
  bool has_last;
};
__device__ __forceinline__ SplitWork split_work(int L, int split, int chunk, bool packed) {
  SplitWork w;
  const int pages = packed_pages_of(L, packed);
  const int u0 = split * chunk, u1 = min(units_of(L, packed), u0 + chunk);
  w.page_begin = u0;
  w.n_pages = max(0, min(u1, pages) - u0);
  w.bf_total = bf16_tiles_of(L, packed);
  // first unit of tile k is pages + kBf16TileUnits * k
  const int k0 = max(0, (u0 - pages + kBf16TileUnits - 1) / kBf16TileUnits);
  const int k1 = min(w.bf_total, max(0, (u1 - pages + kBf16TileUnits - 1) / kBf16TileUnits));
  w.bf_begin = min(k0, w.bf_total);
  w.n_bf = max(0, k1 - w.bf_begin);
  w.n_sink = packed ? min(L, kSink) : 0;
  w.rec_start = max(kSink, L - kLocal);
  w.n_tok = bf16_tokens_of(L, packed);
  w.has_last = w.n_bf > 0 && w.bf_begin + w.n_bf == w.bf_total;
  return w;
}

// Position of entry idx of the protected-token list.
__device__ __forceinline__ int bf16_pos(const SplitWork& w, int idx) {
  return idx < w.n_sink ? idx : w.rec_start + (idx - w.n_sink);
}

// ---------------------------------------------------------------- plan lookup
// Every CTA recomputes the per-sequence split counts (same integer formula as
// the host) and finds which (sequence, split) its blockIdx.x names.
// `target` is the split's global index (blockIdx.x by default).
template <int kThreads>
__device__ void find_split(const DecodeArgs& a, bool packed, int* scan, int& b_out,
                           int& split_out, int& nsplit_out, int target_index = -1) {
  constexpr int kCtaWarps = kThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (a.B + kThreads - 1) / kThreads;
  const int b0 = min(a.B, tid * per), b1 = min(a.B, b0 + per);
  const int max_tok = a.max_pages * kPageTokens;
  int local = 0;
  for (int b = b0; b < b1; ++b) {
    int L = a.seq_lens[b];
    if (L < 0 || L > max_tok) L = 0;
    local += splits_of(L, packed, a.chunk_pages);
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) scan[warp] = incl;
  if (tid == 0) scan[kCtaWarps] = -1;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int w = 0; w < kCtaWarps; ++w) {
      const int t = scan[w];
      scan[w] = acc;
      acc += t;
    }
    scan[kCtaWarps + 1] = acc;  // device-side total
  }
  __syncthreads();
  const int excl = scan[warp] + incl - local;
  const int target = target_index >= 0 ? target_index : (int)blockIdx.x;
  if (target >= excl && target < excl + local) {
    int acc = excl;
    for (int b = b0; b < b1; ++b) {
      int L = a.seq_lens[b];
      if (L < 0 || L > max_tok) L = 0;
      const int n = splits_of(L, packed, a.chunk_pages);
      if (target < acc + n) {
        scan[kCtaWarps + 2] = b;
        scan[kCtaWarps + 3] = target - acc;
        scan[kCtaWarps + 4] = n;
        scan[kCtaWarps] = 1;
        break;
      }
      acc += n;
    }
  }
  __syncthreads();
  if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) {
    if (scan[kCtaWarps + 1] != a.total_splits) set_error(a.err, MLA_LOWBIT_DEV_PLAN);
    for (int b = 0; b < a.B; ++b) {
      const int L = a.seq_lens[b];
      if (L < 0 || L > max_tok) set_error(a.err, MLA_LOWBIT_DEV_BAD_LEN);
    }
  }
  if (scan[kCtaWarps] == 1) {
    b_out = scan[kCtaWarps + 2];
    split_out = scan[kCtaWarps + 3];
    nsplit_out = scan[kCtaWarps + 4];
  } else {
    b_out = -1;
  }
}

}  // namespace mlalb
