// Split-KV low-bit MLA decode (one CTA per (split, 16-head chunk)) and the
// log-sum-exp combine of the splits.
//
// QuantMLA (Abstract) integrates unpacking and dequantisation into attention;
// the Figure 8 caption has the reconstructed content tile serve both matching
// (QK) and latent aggregation (PV), bf16 values for protected tokens, and one
// global softmax over all valid tokens.  The page-level kernel design is this
// library's own (the pages give none):
//
// * Codes stay exact integers.  With x = s*c + m per (token, group),
//     QK:  z = sum_g s_g * (q_g . c_g) + sum_g m_g * sum(q_g)
//     PV:  o[c] = sum_t (p_t s_t,g) c_t,c + sum_t p_t m_t,g
//   so the tensor cores only see exact fp16 codes, and the per-group scale and
//   min are applied in fp32 (on the QK accumulator and on P).  P*s is split
//   into an fp16 high and low part (two MMAs), which keeps the 22-bit product
//   precision the outlier channels need.
// * A 64-token tile (one page) per step.  Warp w unpacks tokens 8w..8w+7 of
//   all 9 groups straight into mma B fragments (nibble -> fp16 by the
//   exponent-bias trick of Kim et al. 2022, "Who Says Elephants Can't Run"),
//   runs QK for them, and stores the content codes to a swizzled shared tile.
//   After a block-wide max, warp w runs PV for content group w over all 64
//   tokens, reading the tile with ldmatrix.trans.
// * The contraction dimension is permuted inside each group so that the
//   unpack's natural pair order is the mma fragment order; q is staged in the
//   same permuted order and the output channels are un-permuted at the end.
// * The sink/recent bf16 tokens are one more split of the same sequence, so
//   the combine kernel folds them into the one softmax.
#include <cfloat>

#include "common.cuh"

namespace mlalb {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kHC = 16;                 // heads per CTA
constexpr int kTileRow = 1024;          // bytes per token row of the content tile
constexpr int kQStride = kDim + 8;      // fp16 per q row in shared memory
constexpr int kPStride = 72;            // floats per P row
constexpr int kOffTile = 0;
constexpr int kOffQ = kOffTile + kPageTokens * kTileRow;
constexpr int kOffP = kOffQ + kHC * kQStride * 2;
constexpr int kOffS = kOffP + kHC * kPStride * 4;
constexpr int kOffM = kOffS + 8 * kPageTokens * 4;
constexpr int kOffMax = kOffM + 8 * kPageTokens * 4;
constexpr int kOffQsum = kOffMax + kWarps * kHC * 4;
constexpr int kOffScan = kOffQsum + kGroups * kHC * 4;
constexpr int kSmemBytes = kOffScan + (kThreads + 64) * 4;

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

// ---------------------------------------------------------------- plan lookup
// Every CTA recomputes the per-sequence split counts (same integer formula as
// the host) and finds which (sequence, split) its blockIdx.x names.
__device__ void find_split(const DecodeArgs& a, bool packed, int* scan, int& b_out,
                           int& split_out, int& nsplit_out) {
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
  if (tid == 0) scan[kWarps] = -1;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int t = scan[w];
      scan[w] = acc;
      acc += t;
    }
    scan[kWarps + 1] = acc;  // device-side total
  }
  __syncthreads();
  const int excl = scan[warp] + incl - local;
  const int target = blockIdx.x;
  if (target >= excl && target < excl + local) {
    int acc = excl;
    for (int b = b0; b < b1; ++b) {
      int L = a.seq_lens[b];
      if (L < 0 || L > max_tok) L = 0;
      const int n = splits_of(L, packed, a.chunk_pages);
      if (target < acc + n) {
        scan[kWarps + 2] = b;
        scan[kWarps + 3] = target - acc;
        scan[kWarps + 4] = n;
        scan[kWarps] = 1;
        break;
      }
      acc += n;
    }
  }
  __syncthreads();
  if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) {
    if (scan[kWarps + 1] != a.total_splits) set_error(a.err, MLA_LOWBIT_DEV_PLAN);
    for (int b = 0; b < a.B; ++b) {
      const int L = a.seq_lens[b];
      if (L < 0 || L > max_tok) set_error(a.err, MLA_LOWBIT_DEV_BAD_LEN);
    }
  }
  if (scan[kWarps] == 1) {
    b_out = scan[kWarps + 2];
    split_out = scan[kWarps + 3];
    nsplit_out = scan[kWarps + 4];
  } else {
    b_out = -1;
  }
}

// ---------------------------------------------------------------- split kernel
template <int CB>
__global__ void __launch_bounds__(kThreads, 2) decode_split_kernel(DecodeArgs a) {
  constexpr bool kPacked = CB != 16;
  constexpr bool kTypeB = CB == 2;  // pairing of the content groups
  constexpr PageGeom G = page_geom(CB);
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* tile = smem + kOffTile;
  __half* qs = reinterpret_cast<__half*>(smem + kOffQ);
  float* P = reinterpret_cast<float*>(smem + kOffP);
  float* smS = reinterpret_cast<float*>(smem + kOffS);
  float* smM = reinterpret_cast<float*>(smem + kOffM);
  float* smax = reinterpret_cast<float*>(smem + kOffMax);
  float* qsum = reinterpret_cast<float*>(smem + kOffQsum);
  int* scan = reinterpret_cast<int*>(smem + kOffScan);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = lane & 3, rn = lane >> 2;
  const int h0 = rn;  // rows h0 and h0 + 8 of the 16-head chunk

  int b, split, nsplit;
  find_split(a, kPacked, scan, b, split, nsplit);
  if (b < 0) return;
  const int hc = blockIdx.y;
  const int L = [&] {
    const int v = a.seq_lens[b];
    return (v < 0 || v > a.max_pages * kPageTokens) ? 0 : v;
  }();
  if (split == 0 && hc == 0 && tid == 0) {
    a.seq_split[2 * b] = blockIdx.x;
    a.seq_split[2 * b + 1] = nsplit;
  }

  // ---- stage q (fp16, permuted contraction order) and its group sums: thread
  // t < 144 owns (group g, head h), loads its 64 values with 8 vector loads and
  // sums them in a fixed order.
  {
    for (int idx = tid; idx < kPageTokens * kTileRow / 16; idx += kThreads)
      reinterpret_cast<uint4*>(tile)[idx] = make_uint4(0, 0, 0, 0);
    if (tid < kGroups * kHC) {
      const int g = tid / kHC, h = tid % kHC;
      const bool tb = g < 8 ? kTypeB : false;
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + ((long long)b * a.H + hc * kHC + h) * kDim + g * 64);
      uint4 v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) v[c] = src[c];
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int p = c * 8 + e;
          const float f = (e & 1) ? bf16hi_to_f32(w[e >> 1]) : bf16lo_to_f32(w[e >> 1]);
          const __half hv = __float2half_rn(f);
          acc += __half2float(hv);
          qs[h * kQStride + g * 64 + logical_of_phys(p, tb)] = hv;
        }
      }
      qsum[g * kHC + h] = acc;
    }
    __syncthreads();
  }

  // ---- work of this split
  const bool bf16_split = kPacked && split == nsplit - 1;
  int n_tiles, page_begin = 0, n_sink = 0, rec_start = 0, n_tok = 0;
  if (bf16_split) {
    n_sink = min(L, kSink);
    rec_start = max(kSink, L - kLocal);
    n_tok = n_sink + max(0, L - rec_start);
    n_tiles = (n_tok + kPageTokens - 1) / kPageTokens;
  } else {
    const int pages = packed_pages_of(L, kPacked);
    page_begin = split * a.chunk_pages;
    n_tiles = max(0, min(a.chunk_pages, pages - page_begin));
  }
  const int valid_lo = kPacked ? kSink : 0;
  const int valid_hi = kPacked ? L - kLocal : L;  // packed-served tokens [lo, hi)

  float O[8][4];
#pragma unroll
  for (int c = 0; c < 8; ++c) O[c][0] = O[c][1] = O[c][2] = O[c][3] = 0.f;
  float m_run0 = -INFINITY, m_run1 = -INFINITY;
  float accm0 = 0.f, accm1 = 0.f, l0 = 0.f, l1 = 0.f;

  const int rowB = warp * 8 + rn;   // tile row of this thread's B fragment
  const int tC0 = warp * 8 + 2 * j;  // tile rows of this thread's C columns

  for (int tile_i = 0; tile_i < n_tiles; ++tile_i) {
    // ================= phase 1: unpack + QK for tokens 8w..8w+7
    float S[4] = {0.f, 0.f, 0.f, 0.f};
    bool v0, v1;  // validity of tokens tC0, tC0+1
    bool use_packed = false;
    if constexpr (kPacked) use_packed = !bf16_split;
    if (use_packed) {
      if constexpr (kPacked) {
      const int page_idx = page_begin + tile_i;
      const long long page = a.block_table[(long long)b * a.max_pages + page_idx];
      const bool page_ok = page >= 0 && page < a.num_pages;
      if (!page_ok && tid == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
      const int tok0 = page_idx * kPageTokens;
      v0 = page_ok && tok0 + tC0 >= valid_lo && tok0 + tC0 < valid_hi;
      v1 = page_ok && tok0 + tC0 + 1 >= valid_lo && tok0 + tC0 + 1 < valid_hi;
      if (page_ok) {
        const uint8_t* pb = a.pool + page * G.page_bytes;
        uint32_t cw[kGroups][2];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          if constexpr (CB == 4) {
            const uint2 t = *reinterpret_cast<const uint2*>(pb + G.content_off +
                                                             rowB * G.content_row + g * 32 + j * 8);
            cw[g][0] = t.x;
            cw[g][1] = t.y;
          } else {
            cw[g][0] = *reinterpret_cast<const uint32_t*>(pb + G.content_off +
                                                          rowB * G.content_row + g * 16 + j * 4);
            cw[g][1] = 0;
          }
        }
        {
          const uint2 t =
              *reinterpret_cast<const uint2*>(pb + G.rope_off + rowB * G.rope_row + j * 8);
          cw[8][0] = t.x;
          cw[8][1] = t.y;
        }
        uint32_t mt0[kGroups], mt1[kGroups];
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          mt0[g] = *reinterpret_cast<const uint32_t*>(pb + G.meta_off + tC0 * G.meta_row + g * 4);
          mt1[g] =
              *reinterpret_cast<const uint32_t*>(pb + G.meta_off + (tC0 + 1) * G.meta_row + g * 4);
        }
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          uint32_t bq[8];
          if (g < 8 && CB == 2) {
            unpack_int2(cw[g][0], bq);
          } else {
            unpack_int4(cw[g][0], bq);
            unpack_int4(cw[g][1], bq + 4);
          }
          float D[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            uint32_t af[4];
            ldmatrix_x4(af, qs + (lane & 15) * kQStride + g * 64 + s * 16 + (lane >> 4) * 8);
            mma_16816(D, af, bq[2 * s], bq[2 * s + 1]);
          }
          const float centre = (g < 8 && CB == 2) ? float(kCentre2) : float(kCentre4);
          const float s0 = __half2float(__ushort_as_half(static_cast<unsigned short>(mt0[g])));
          const float s1 = __half2float(__ushort_as_half(static_cast<unsigned short>(mt1[g])));
          const float m0 = fmaf(centre, s0,
              __half2float(__ushort_as_half(static_cast<unsigned short>(mt0[g] >> 16))));
          const float m1 = fmaf(centre, s1,
              __half2float(__ushort_as_half(static_cast<unsigned short>(mt1[g] >> 16))));
          const float q0 = qsum[g * kHC + h0], q1 = qsum[g * kHC + h0 + 8];
          S[0] += s0 * D[0] + m0 * q0;
          S[1] += s1 * D[1] + m1 * q0;
          S[2] += s0 * D[2] + m0 * q1;
          S[3] += s1 * D[3] + m1 * q1;
          if (g < 8) {
            uint8_t* rowp = tile + rowB * kTileRow;
            const int c0 = (8 * g + 2 * j) ^ (rowB & 7), c1 = (8 * g + 2 * j + 1) ^ (rowB & 7);
            *reinterpret_cast<uint4*>(rowp + c0 * 16) = make_uint4(bq[0], bq[1], bq[2], bq[3]);
            *reinterpret_cast<uint4*>(rowp + c1 * 16) = make_uint4(bq[4], bq[5], bq[6], bq[7]);
            if (rn == 0) {
              smS[g * kPageTokens + tC0] = v0 ? s0 : 0.f;
              smS[g * kPageTokens + tC0 + 1] = v1 ? s1 : 0.f;
              smM[g * kPageTokens + tC0] = v0 ? m0 : 0.f;
              smM[g * kPageTokens + tC0 + 1] = v1 ? m1 : 0.f;
            }
          }
        }
      } else if (rn == 0) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          smS[g * kPageTokens + tC0] = smS[g * kPageTokens + tC0 + 1] = 0.f;
          smM[g * kPageTokens + tC0] = smM[g * kPageTokens + tC0 + 1] = 0.f;
        }
      }
      }
    } else {
      // bf16 rows: protected tokens of a packed cache, or bf16 pages.
      const uint16_t* rowptr = nullptr;
      if (bf16_split) {
        const int i = tile_i * kPageTokens + rowB;
        if (i < n_tok) {
          const int pos = i < n_sink ? i : rec_start + (i - n_sink);
          rowptr = pos < kSink ? a.sink + ((long long)b * kSink + pos) * kDim
                               : a.recent + ((long long)b * kLocal + pos % kLocal) * kDim;
        }
        v0 = tile_i * kPageTokens + tC0 < n_tok;
        v1 = tile_i * kPageTokens + tC0 + 1 < n_tok;
      } else {
        const int page_idx = page_begin + tile_i;
        const long long page = a.block_table[(long long)b * a.max_pages + page_idx];
        const bool page_ok = page >= 0 && page < a.num_pages;
        if (!page_ok && tid == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
        const int tok0 = page_idx * kPageTokens;
        if (page_ok)
          rowptr = reinterpret_cast<const uint16_t*>(a.pool + page * G.page_bytes) + rowB * kDim;
        v0 = page_ok && tok0 + tC0 < L;
        v1 = page_ok && tok0 + tC0 + 1 < L;
      }
#pragma unroll 1
      for (int g = 0; g < kGroups; ++g) {
        uint32_t vv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (rowptr) {
          const uint4* src = reinterpret_cast<const uint4*>(rowptr + g * 64 + j * 16);
          const uint4 t0 = src[0], t1 = src[1];
          vv[0] = t0.x; vv[1] = t0.y; vv[2] = t0.z; vv[3] = t0.w;
          vv[4] = t1.x; vv[5] = t1.y; vv[6] = t1.z; vv[7] = t1.w;
        }
        uint32_t bq[8];
        if (kTypeB && g < 8)
          pairs_from_bf16<true>(vv, bq);
        else
          pairs_from_bf16<false>(vv, bq);
        float D[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          uint32_t af[4];
          ldmatrix_x4(af, qs + (lane & 15) * kQStride + g * 64 + s * 16 + (lane >> 4) * 8);
          mma_16816(D, af, bq[2 * s], bq[2 * s + 1]);
        }
        S[0] += D[0];
        S[1] += D[1];
        S[2] += D[2];
        S[3] += D[3];
        if (g < 8) {
          uint8_t* rowp = tile + rowB * kTileRow;
          const int c0 = (8 * g + 2 * j) ^ (rowB & 7), c1 = (8 * g + 2 * j + 1) ^ (rowB & 7);
          *reinterpret_cast<uint4*>(rowp + c0 * 16) = make_uint4(bq[0], bq[1], bq[2], bq[3]);
          *reinterpret_cast<uint4*>(rowp + c1 * 16) = make_uint4(bq[4], bq[5], bq[6], bq[7]);
          if (rn == 0) {
            smS[g * kPageTokens + tC0] = v0 ? 1.f : 0.f;
            smS[g * kPageTokens + tC0 + 1] = v1 ? 1.f : 0.f;
            smM[g * kPageTokens + tC0] = 0.f;
            smM[g * kPageTokens + tC0 + 1] = 0.f;
          }
        }
      }
    }

    // ---- mask, scale to log2 units, block max per head
    S[0] = v0 ? S[0] * a.scale_log2 : -INFINITY;
    S[1] = v1 ? S[1] * a.scale_log2 : -INFINITY;
    S[2] = v0 ? S[2] * a.scale_log2 : -INFINITY;
    S[3] = v1 ? S[3] * a.scale_log2 : -INFINITY;
    float mx0 = fmaxf(S[0], S[1]), mx1 = fmaxf(S[2], S[3]);
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    if (j == 0) {
      smax[warp * kHC + h0] = mx0;
      smax[warp * kHC + h0 + 8] = mx1;
    }
    __syncthreads();
    float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      t0 = fmaxf(t0, smax[w * kHC + h0]);
      t1 = fmaxf(t1, smax[w * kHC + h0 + 8]);
    }
    const float mn0 = fmaxf(m_run0, t0), mn1 = fmaxf(m_run1, t1);
    const float alpha0 = mn0 == -INFINITY ? 1.f : fast_exp2(m_run0 - mn0);
    const float alpha1 = mn1 == -INFINITY ? 1.f : fast_exp2(m_run1 - mn1);
    m_run0 = mn0;
    m_run1 = mn1;
    {
      const float p0 = S[0] == -INFINITY ? 0.f : fast_exp2(S[0] - mn0);
      const float p1 = S[1] == -INFINITY ? 0.f : fast_exp2(S[1] - mn0);
      const float p2 = S[2] == -INFINITY ? 0.f : fast_exp2(S[2] - mn1);
      const float p3 = S[3] == -INFINITY ? 0.f : fast_exp2(S[3] - mn1);
      *reinterpret_cast<float2*>(&P[h0 * kPStride + tC0]) = make_float2(p0, p1);
      *reinterpret_cast<float2*>(&P[(h0 + 8) * kPStride + tC0]) = make_float2(p2, p3);
    }
    __syncthreads();

    // ================= phase 2: PV for content group g = warp
    {
      const int g = warp;
      if (alpha0 != 1.f) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          O[c][0] *= alpha0;
          O[c][1] *= alpha0;
        }
        accm0 *= alpha0;
        l0 *= alpha0;
      }
      if (alpha1 != 1.f) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          O[c][2] *= alpha1;
          O[c][3] *= alpha1;
        }
        accm1 *= alpha1;
        l1 *= alpha1;
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int t = ks * 16 + 2 * j;
        const float2 pa = *reinterpret_cast<const float2*>(&P[h0 * kPStride + t]);
        const float2 pb = *reinterpret_cast<const float2*>(&P[(h0 + 8) * kPStride + t]);
        const float2 pc = *reinterpret_cast<const float2*>(&P[h0 * kPStride + t + 8]);
        const float2 pd = *reinterpret_cast<const float2*>(&P[(h0 + 8) * kPStride + t + 8]);
        const float2 sA = *reinterpret_cast<const float2*>(&smS[g * kPageTokens + t]);
        const float2 sB = *reinterpret_cast<const float2*>(&smS[g * kPageTokens + t + 8]);
        const float2 mA = *reinterpret_cast<const float2*>(&smM[g * kPageTokens + t]);
        const float2 mB = *reinterpret_cast<const float2*>(&smM[g * kPageTokens + t + 8]);
        uint32_t ahi[4], alo[4];
        split_hi_lo(pa.x * sA.x, pa.y * sA.y, ahi[0], alo[0]);
        split_hi_lo(pb.x * sA.x, pb.y * sA.y, ahi[1], alo[1]);
        split_hi_lo(pc.x * sB.x, pc.y * sB.y, ahi[2], alo[2]);
        split_hi_lo(pd.x * sB.x, pd.y * sB.y, ahi[3], alo[3]);
        accm0 += pa.x * mA.x + pa.y * mA.y + pc.x * mB.x + pc.y * mB.y;
        accm1 += pb.x * mA.x + pb.y * mA.y + pd.x * mB.x + pd.y * mB.y;
        l0 += (pa.x + pa.y) + (pc.x + pc.y);
        l1 += (pb.x + pb.y) + (pd.x + pd.y);
        const int tok = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int c = 0; c < 8; c += 2) {
          const int chunk = 8 * g + c + (lane >> 4);
          uint32_t bf[4];
          ldmatrix_x4_trans(bf, tile + tok * kTileRow + ((chunk ^ (tok & 7)) << 4));
          mma_16816(O[c], ahi, bf[0], bf[1]);
          mma_16816(O[c], alo, bf[0], bf[1]);
          mma_16816(O[c + 1], ahi, bf[2], bf[3]);
          mma_16816(O[c + 1], alo, bf[2], bf[3]);
        }
      }
    }
    __syncthreads();
  }

  // ---- epilogue: finish the min term, write the partial (O, max, sum)
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    accm0 += __shfl_xor_sync(0xffffffffu, accm0, o);
    accm1 += __shfl_xor_sync(0xffffffffu, accm1, o);
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  const int g = warp;
  const long long sidx = blockIdx.x;
  const int hg0 = hc * kHC + h0, hg1 = hg0 + 8;
  float* o0 = a.part_o + (sidx * a.H + hg0) * kLatent + g * 64;
  float* o1 = a.part_o + (sidx * a.H + hg1) * kLatent + g * 64;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    o0[phys_of_chunk(c, 2 * j, kTypeB)] = O[c][0] + accm0;
    o0[phys_of_chunk(c, 2 * j + 1, kTypeB)] = O[c][1] + accm0;
    o1[phys_of_chunk(c, 2 * j, kTypeB)] = O[c][2] + accm1;
    o1[phys_of_chunk(c, 2 * j + 1, kTypeB)] = O[c][3] + accm1;
  }
  if (warp == 0 && j == 0) {
    a.part_ml[(sidx * a.H + hg0) * 2] = m_run0;
    a.part_ml[(sidx * a.H + hg0) * 2 + 1] = l0;
    a.part_ml[(sidx * a.H + hg1) * 2] = m_run1;
    a.part_ml[(sidx * a.H + hg1) * 2 + 1] = l1;
  }
}

// ---------------------------------------------------------------- combine
struct CombineArgs {
  const float* part_o;
  const float* part_ml;
  const int32_t* seq_split;
  float* out;
  float* lse;
  int B, H, total_splits;
};

constexpr int kCombineThreads = 128;
constexpr int kCombineMaxW = 1024;  // split weights kept in shared memory

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float t = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, t) : v + t;
  }
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
  for (int w = 1; w < kCombineThreads / 32; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
  return v;
}

// One block per (sequence, head): the split weights 2^(m_s - M) go to shared
// memory once, then every thread sums its 4 channels over the splits with
// independent (unrolled, branch-free) loads.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineArgs a) {
  __shared__ float wsm[kCombineMaxW];
  __shared__ float red[kCombineThreads / 32];
  const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
  int off = a.seq_split[2 * b], n = a.seq_split[2 * b + 1];
  off = min(max(off, 0), a.total_splits);
  n = min(max(n, 0), a.total_splits - off);
  const float* ml = a.part_ml + ((long long)off * a.H + h) * 2;
  const long long mstride = (long long)a.H * 2;
  float M = -INFINITY;
  for (int s = threadIdx.x; s < n; s += kCombineThreads)
    if (ml[s * mstride + 1] > 0.f) M = fmaxf(M, ml[s * mstride]);
  M = block_reduce(M, true, red);
  float den = 0.f;
  for (int s = threadIdx.x; s < n; s += kCombineThreads) {
    const float l = ml[s * mstride + 1];
    const float w = l > 0.f ? fast_exp2(ml[s * mstride] - M) : 0.f;
    den += w * l;
    if (s < kCombineMaxW) wsm[s] = w;
  }
  den = block_reduce(den, false, red);
  const int c = threadIdx.x * 4;
  const float* o = a.part_o + ((long long)off * a.H + h) * kLatent + c;
  const long long ostride = (long long)a.H * kLatent;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int s = 0; s < n; ++s) {
    float w;
    if (s < kCombineMaxW) {
      w = wsm[s];
    } else {
      const float l = ml[s * mstride + 1];
      w = l > 0.f ? fast_exp2(ml[s * mstride] - M) : 0.f;
    }
    const float4 v = *reinterpret_cast<const float4*>(o + s * ostride);
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  *reinterpret_cast<float4*>(a.out + ((long long)b * a.H + h) * kLatent + c) =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (a.lse && threadIdx.x == 0)
    a.lse[(long long)b * a.H + h] = den > 0.f ? (M + log2f(den)) * 0.69314718055994531f
                                              : -INFINITY;
}

cudaError_t launch_decode(int cbits, const DecodeArgs& a, float* out, float* lse,
                          cudaStream_t stream) {
  static bool configured[3] = {false, false, false};
  const int k = cbits == 4 ? 0 : cbits == 2 ? 1 : 2;
  cudaError_t e = cudaSuccess;
  if (!configured[k]) {
    switch (cbits) {
      case 4: e = cudaFuncSetAttribute(decode_split_kernel<4>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes); break;
      case 2: e = cudaFuncSetAttribute(decode_split_kernel<2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes); break;
      default: e = cudaFuncSetAttribute(decode_split_kernel<16>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    }
    if (e != cudaSuccess) return e;
    configured[k] = true;
  }
  dim3 grid(a.total_splits, a.H / kHC), block(kThreads);
  switch (cbits) {
    case 4: decode_split_kernel<4><<<grid, block, kSmemBytes, stream>>>(a); break;
    case 2: decode_split_kernel<2><<<grid, block, kSmemBytes, stream>>>(a); break;
    default: decode_split_kernel<16><<<grid, block, kSmemBytes, stream>>>(a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CombineArgs ca{a.part_o, a.part_ml, a.seq_split, out, lse, a.B, a.H, a.total_splits};
  combine_kernel<<<a.B * a.H, kCombineThreads, 0, stream>>>(ca);
  return cudaGetLastError();
}

}  // namespace mlalb
