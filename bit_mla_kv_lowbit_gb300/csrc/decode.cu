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
// * The sink/recent bf16 tokens are more 64-token tiles of the same split
//   work list (after the sequence's pages, see split_work), so the combine
//   kernel folds them into the one softmax.
#include <cfloat>

#include "decode_common.cuh"
#include "writer_common.cuh"

namespace mlalb {

constexpr int kTeams = 2;                 // independent 8-warp teams per CTA
constexpr int kTeamWarps = 8;
constexpr int kTeamThreads = kTeamWarps * 32;
constexpr int kCtaWarps = kTeams * kTeamWarps;
constexpr int kThreads = kCtaWarps * 32;
constexpr int kTileRow = 1024;          // bytes per token row of the content tile
constexpr int kQStride = kDim + 8;      // fp16 per q row in shared memory
constexpr int kPStride = 72;            // floats per P row
// shared by both teams
constexpr int kOffQ = 0;
constexpr int kQBytes = kHC * kQStride * 2;
constexpr int kOffQsum = kOffQ + kQBytes;
constexpr int kOffScan = kOffQsum + kGroups * kHC * 4;
constexpr int kOffPages = kOffScan + 64 * 4;  // [64] page ids of the split
constexpr int kOffTeam = ((kOffPages + 64 * 4) + 127) / 128 * 128;
// per team
constexpr int kTOffTile = 0;
constexpr int kTOffP = kTOffTile + kPageTokens * kTileRow;
constexpr int kTOffS = kTOffP + kHC * kPStride * 4;
constexpr int kTOffM = kTOffS + 8 * kPageTokens * 4;
constexpr int kTOffMax = kTOffM + 8 * kPageTokens * 4;
constexpr int kTOffStage = kTOffMax + kTeamWarps * kHC * 4;
static_assert(kTOffMax % 16 == 0, "tile maxima are read as float4");
__host__ __device__ constexpr int team_bytes(int cbits) {
  return kTOffStage + (cbits == 16 ? 0 : page_geom(cbits).page_bytes);
}
// a rotated q keeps its low fp16 parts after the two teams, then the rotated
// content latent of the appended token
__host__ __device__ constexpr int smem_bytes(int cbits, bool rot = false) {
  return kOffTeam + kTeams * team_bytes(cbits) + (rot ? kQBytes + kLatent * 2 : 0);
}
static_assert(smem_bytes(4, true) <= 227 * 1024, "shared memory budget");

// ---------------------------------------------------------------- split kernel
__device__ __forceinline__ void team_sync(int team) {
  asm volatile("bar.sync %0, %1;" ::"r"(team + 1), "r"(kTeamThreads) : "memory");
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// XOR applied to the 16-byte chunk index of content row r in the staging copy:
// it spreads the rows a half-warp reads over all 32 banks.
template <int CB>
__device__ __forceinline__ int stage_swizzle(int r) {
  return CB == 4 ? ((r & 3) << 1) : (r & 3);
}

// One CTA per (split, 16-head chunk), one CTA per SM.  Two independent teams
// of 8 warps take alternate pages of the split, each with its own running max,
// sum and output, and merge at the end.  Packed pages are copied into a
// per-team staging buffer with cp.async one page ahead.
// kRot: the cache holds the online-rotated content latent; q's content groups
// are rotated here (float32) and kept as fp16 high + low parts, so QK runs a
// second MMA per content k-step on the low parts.
template <int CB, bool kRot>
__global__ void __launch_bounds__(kThreads, 1) decode_split_kernel(DecodeArgs a) {
  constexpr bool kPacked = CB != 16;
  static_assert(!kRot || kPacked, "rotation needs a packed layout");
  constexpr bool kTypeB = CB == 2;  // pairing of the content groups
  constexpr PageGeom G = page_geom(CB);
  extern __shared__ __align__(128) uint8_t smem[];
  __half* qs = reinterpret_cast<__half*>(smem + kOffQ);
  __half* qs_lo = reinterpret_cast<__half*>(smem + kOffTeam + kTeams * team_bytes(CB));
  uint32_t* new_rot = reinterpret_cast<uint32_t*>(smem + kOffTeam + kTeams * team_bytes(CB) + kQBytes);
  float* qsum = reinterpret_cast<float*>(smem + kOffQsum);
  int* scan = reinterpret_cast<int*>(smem + kOffScan);

  const int tid = threadIdx.x, lane = tid & 31;
  const int team = tid / kTeamThreads, ttid = tid % kTeamThreads, warp = ttid >> 5;
  uint8_t* tbase = smem + kOffTeam + team * team_bytes(CB);
  uint8_t* tile = tbase + kTOffTile;
  float* P = reinterpret_cast<float*>(tbase + kTOffP);
  float* smS = reinterpret_cast<float*>(tbase + kTOffS);
  float* smM = reinterpret_cast<float*>(tbase + kTOffM);
  float* smax = reinterpret_cast<float*>(tbase + kTOffMax);
  uint8_t* stage = tbase + kTOffStage;
  int* s_pages = reinterpret_cast<int*>(smem + kOffPages);
  const int j = lane & 3, rn = lane >> 2;
  const int h0 = rn;  // rows h0 and h0 + 8 of the 16-head chunk

  int b, split, nsplit;
  find_split<kThreads>(a, kPacked, scan, b, split, nsplit);
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

  // ---- work of this split: pages, then 64-token tiles of the protected bf16
  // tokens (packed layouts); tile_i < n_pages is a page
  const SplitWork sw = split_work(L, split, a.chunk_pages, kPacked);
  const int n_pages = sw.n_pages, page_begin = sw.page_begin;
  int n_tiles = n_pages + sw.n_bf;
  if (n_tiles > 64) {  // the planner caps splits at 64 units
    if (tid == 0) set_error(a.err, MLA_LOWBIT_DEV_PLAN);
    n_tiles = 0;
  }
  const int valid_lo = kPacked ? kSink : 0;
  const int valid_hi = kPacked ? L - kLocal : L;  // packed-served tokens [lo, hi)
  // query blocks: this head chunk's query does not see the sequence's last
  // n_masked tokens (all inside the recent window)
  const int n_masked = a.n_q - 1 - (hc * kHC) / (a.H / a.n_q);

  // Copy part of packed page `tile_i` of this split into the team's staging
  // buffer: the thread's 16-byte chunks ttid + kTeamThreads * i for i in
  // [i0, i1).  The whole page is the parts i in [0, kStageIters); a commit
  // closes it.
  constexpr int kStageIters = (G.page_bytes / 16 + kTeamThreads - 1) / kTeamThreads;
  auto stage_part = [&](int tile_i, int i0, int i1) {
    if constexpr (kPacked) {
      const long long page = s_pages[tile_i];
      if (page >= 0 && page < a.num_pages) {
        const uint8_t* src = a.pool + page * G.page_bytes;
        constexpr int kChunks = G.page_bytes / 16;
        constexpr int kRowChunks = G.content_row / 16;
        constexpr int kContentChunks = kPageTokens * kRowChunks;
        for (int i = i0; i < i1; ++i) {
          const int k = ttid + kTeamThreads * i;
          if (k >= kChunks) break;
          int dst = k * 16;
          if (k < kContentChunks) {
            const int r = k / kRowChunks, c = k % kRowChunks;
            dst = G.content_off + r * G.content_row + ((c ^ stage_swizzle<CB>(r)) << 4);
          }
          cp_async16(stage + dst, src + k * 16);
        }
      }
    }
  };
  auto stage_page = [&](int tile_i) {
    stage_part(tile_i, 0, kStageIters);
    cp_async_commit();
  };

  // ---- stage q (fp16, permuted contraction order) and its group sums: thread
  // t < 144 owns (group g, head h), loads its 64 values with 8 vector loads and
  // sums them in a fixed order.  Each team zeroes its content tile.
  {
    for (int idx = ttid; idx < kPageTokens * kTileRow / 16; idx += kTeamThreads)
      reinterpret_cast<uint4*>(tile)[idx] = make_uint4(0, 0, 0, 0);
    if (tid < kGroups * kHC) {
      const int g = tid / kHC, h = tid % kHC;
      const bool tb = g < 8 ? kTypeB : false;
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + ((long long)b * a.H + hc * kHC + h) * kDim + g * 64);
      uint4 v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) v[c] = src[c];
      float f[64];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
          f[c * 8 + e] = (e & 1) ? bf16hi_to_f32(w[e >> 1]) : bf16lo_to_f32(w[e >> 1]);
      }
      if (kRot && g < 8) {
        // R q for this content group: the same orthonormal Hadamard rotation
        // as the stored latent (the order of operations does not matter here)
#pragma unroll
        for (int hh = 1; hh < 64; hh <<= 1) {
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            if (i & hh) continue;
            const float x = f[i], y = f[i + hh];
            f[i] = x + y;
            f[i + hh] = x - y;
          }
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) f[i] *= 0.125f;
      }
      float acc = 0.f;
#pragma unroll
      for (int p = 0; p < 64; ++p) {
        const __half hv = __float2half_rn(f[p]);
        const __half lv = __float2half_rn(f[p] - __half2float(hv));
        acc += __half2float(hv);
        if (kRot) acc += __half2float(lv);
        qs[h * kQStride + g * 64 + logical_of_phys(p, tb)] = hv;
        if (kRot) qs_lo[h * kQStride + g * 64 + logical_of_phys(p, tb)] = lv;
      }
      qsum[g * kHC + h] = acc;
    }
    if (kPacked && tid < n_pages && tid < 64)
      s_pages[tid] = a.block_table[(long long)b * a.max_pages + page_begin + tid];
    if constexpr (kPacked) {
      // the bf16 rows of this split's protected-token tiles come last and are
      // read straight from the bf16 buffers: start moving them into L2 now
      const int first = 64 * sw.bf_begin, end = min(sw.n_tok, 64 * (sw.bf_begin + sw.n_bf));
      for (int k = tid; k < (end - first) * (kDim * 2 / 128); k += kThreads) {
        const int pos = bf16_pos(sw, first + k / (kDim * 2 / 128));
        const uint16_t* row = pos < kSink ? a.sink + ((long long)b * kSink + pos) * kDim
                                          : a.recent + ((long long)b * kLocal + pos % kLocal) * kDim;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row + (k % (kDim * 2 / 128)) * 64));
      }
    }
    __syncthreads();  // page ids visible
    if (kPacked && team < n_pages) stage_page(team);
    __syncthreads();
  }

  // fused append: the sequence's new token (position L - 1) is packed into its
  // page and copied to the bf16 buffers by head chunk 0's bf16 split, one warp
  // per group.  No split reads those bytes in this call: the token is inside
  // the recent window, and every bf16 split reads it from the input below (a
  // rotated cache: the split's rotated copy of it in shared memory).
  if constexpr (kPacked) {
    if (kRot && sw.has_last && a.new_ckv && L >= 1) {
      if ((tid >> 5) < 8) {
        const int gwp = tid >> 5;
        new_rot[gwp * 32 + lane] =
            rotate_group_bf16(a.new_ckv[(long long)b * (kLatent / 2) + gwp * 32 + lane], lane);
      }
      __syncthreads();  // CTA-uniform condition
    }
    if (sw.has_last && a.new_ckv && hc == 0 && L >= 1 && (tid >> 5) < kGroups) {
      const int gwp = tid >> 5, pos = L - 1;
      const long long page = a.block_table[(long long)b * a.max_pages + pos / kPageTokens];
      if (page >= 0 && page < a.num_pages) {
        const uint32_t v = gwp < 8 ? (kRot ? new_rot[gwp * 32 + lane]
                                           : a.new_ckv[(long long)b * (kLatent / 2) + gwp * 32 + lane])
                                   : a.new_kr[(long long)b * (kRope / 2) + lane];
        if (pos < kSink) a.sink_w[((long long)b * kSink + pos) * (kDim / 2) + gwp * 32 + lane] = v;
        a.recent_w[((long long)b * kLocal + pos % kLocal) * (kDim / 2) + gwp * 32 + lane] = v;
        write_packed_group<CB>(a.pool_w + page * G.page_bytes, pos % kPageTokens, gwp, lane, v);
      } else if (tid == 0) {
        set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
      }
    }
  }

  float O[8][4];
#pragma unroll
  for (int c = 0; c < 8; ++c) O[c][0] = O[c][1] = O[c][2] = O[c][3] = 0.f;
  float m_run0 = -INFINITY, m_run1 = -INFINITY;
  float accm0 = 0.f, accm1 = 0.f, l0 = 0.f, l1 = 0.f;

  const int rowB = warp * 8 + rn;    // tile row of this thread's B fragment
  const int tC0 = warp * 8 + 2 * j;  // tile rows of this thread's C columns

  for (int tile_i = team; tile_i < n_tiles; tile_i += kTeams) {
    const bool use_stage = kPacked && tile_i < n_pages;  // a staged packed page
    if (use_stage) cp_async_wait_all();
    team_sync(team);
    // ================= phase 1: unpack + QK for tokens 8w..8w+7
    float S[4] = {0.f, 0.f, 0.f, 0.f};
    bool v0, v1;  // validity of tokens tC0, tC0+1
    if (use_stage) {
      if constexpr (kPacked) {
        const int page_idx = page_begin + tile_i;
        const long long page = s_pages[tile_i];
        const bool page_ok = page >= 0 && page < a.num_pages;
        if (!page_ok && ttid == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
        const int tok0 = page_idx * kPageTokens;
        v0 = page_ok && tok0 + tC0 >= valid_lo && tok0 + tC0 < valid_hi;
        v1 = page_ok && tok0 + tC0 + 1 >= valid_lo && tok0 + tC0 + 1 < valid_hi;
        if (page_ok) {
          const uint8_t* sb = stage;
          const int sw = stage_swizzle<CB>(rowB);
          uint32_t cw[kGroups][2];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            if constexpr (CB == 4) {
              const int c = 2 * g + (j >> 1);
              const uint2 t = *reinterpret_cast<const uint2*>(
                  sb + G.content_off + rowB * G.content_row + ((c ^ sw) << 4) + 8 * (j & 1));
              cw[g][0] = t.x;
              cw[g][1] = t.y;
            } else {
              cw[g][0] = *reinterpret_cast<const uint32_t*>(
                  sb + G.content_off + rowB * G.content_row + ((g ^ sw) << 4) + 4 * j);
              cw[g][1] = 0;
            }
          }
          {
            const uint2 t =
                *reinterpret_cast<const uint2*>(sb + G.rope_off + rowB * G.rope_row + j * 8);
            cw[8][0] = t.x;
            cw[8][1] = t.y;
          }
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            const uint32_t mt0 =
                *reinterpret_cast<const uint32_t*>(sb + G.meta_off + tC0 * G.meta_row + g * 4);
            const uint32_t mt1 =
                *reinterpret_cast<const uint32_t*>(sb + G.meta_off + (tC0 + 1) * G.meta_row + g * 4);
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
              if (kRot && g < 8) {
                ldmatrix_x4(af, qs_lo + (lane & 15) * kQStride + g * 64 + s * 16 + (lane >> 4) * 8);
                mma_16816(D, af, bq[2 * s], bq[2 * s + 1]);
              }
            }
            const float centre = (g < 8 && CB == 2) ? float(kCentre2) : float(kCentre4);
            const float2 sm0 = __half22float2(*reinterpret_cast<const __half2*>(&mt0));
            const float2 sm1 = __half22float2(*reinterpret_cast<const __half2*>(&mt1));
            const float s0 = sm0.x, s1 = sm1.x;
            const float m0 = fmaf(centre, s0, sm0.y), m1 = fmaf(centre, s1, sm1.y);
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
                *reinterpret_cast<float2*>(&smS[g * kPageTokens + tC0]) =
                    make_float2(v0 ? s0 : 0.f, v1 ? s1 : 0.f);
                *reinterpret_cast<float2*>(&smM[g * kPageTokens + tC0]) =
                    make_float2(v0 ? m0 : 0.f, v1 ? m1 : 0.f);
              }
            }
          }
        } else if (rn == 0) {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            *reinterpret_cast<float2*>(&smS[g * kPageTokens + tC0]) = make_float2(0.f, 0.f);
            *reinterpret_cast<float2*>(&smM[g * kPageTokens + tC0]) = make_float2(0.f, 0.f);
          }
        }
      }
    } else {
      // bf16 rows: protected tokens of a packed cache, or bf16 pages.
      const uint16_t* rowptr = nullptr;
      const uint16_t* rope_ptr = nullptr;  // RoPE channels, when not at rowptr + 512
      if (kPacked) {
        // protected tokens: tile (bf_begin + tile_i - n_pages) of the bf16 list
        const int bt = sw.bf_begin + tile_i - n_pages;
        const int i = bt * kPageTokens + rowB;
        if (i < sw.n_tok) {
          const int pos = bf16_pos(sw, i);
          if (a.new_ckv && pos == L - 1) {
            rowptr = kRot ? reinterpret_cast<const uint16_t*>(new_rot)
                          : reinterpret_cast<const uint16_t*>(a.new_ckv) + (long long)b * kLatent;
            rope_ptr = reinterpret_cast<const uint16_t*>(a.new_kr) + (long long)b * kRope;
          } else {
            rowptr = pos < kSink ? a.sink + ((long long)b * kSink + pos) * kDim
                                 : a.recent + ((long long)b * kLocal + pos % kLocal) * kDim;
          }
        }
        // the protected-token list is in position order: the masked tokens are
        // its last n_masked entries
        const int visible = sw.n_tok - n_masked;
        v0 = bt * kPageTokens + tC0 < visible;
        v1 = bt * kPageTokens + tC0 + 1 < visible;
      } else {
        const int page_idx = page_begin + tile_i;
        const long long page = a.block_table[(long long)b * a.max_pages + page_idx];
        const bool page_ok = page >= 0 && page < a.num_pages;
        if (!page_ok && ttid == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
        const int tok0 = page_idx * kPageTokens;
        if (page_ok)
          rowptr = reinterpret_cast<const uint16_t*>(a.pool + page * G.page_bytes) + rowB * kDim;
        v0 = page_ok && tok0 + tC0 < L - n_masked;
        v1 = page_ok && tok0 + tC0 + 1 < L - n_masked;
      }
#pragma unroll 1
      for (int g = 0; g < kGroups; ++g) {
        uint32_t vv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (rowptr) {
          const uint16_t* chan = (g == 8 && rope_ptr) ? rope_ptr : rowptr + g * 64;
          const uint4* src = reinterpret_cast<const uint4*>(chan + j * 16);
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
          if (kRot && g < 8) {
            ldmatrix_x4(af, qs_lo + (lane & 15) * kQStride + g * 64 + s * 16 + (lane >> 4) * 8);
            mma_16816(D, af, bq[2 * s], bq[2 * s + 1]);
          }
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
            *reinterpret_cast<float2*>(&smS[g * kPageTokens + tC0]) =
                make_float2(v0 ? 1.f : 0.f, v1 ? 1.f : 0.f);
            *reinterpret_cast<float2*>(&smM[g * kPageTokens + tC0]) = make_float2(0.f, 0.f);
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
    if (j == 0) {  // [head][warp]: a head's 8 warp maxima are two 16-byte words
      smax[h0 * kTeamWarps + warp] = mx0;
      smax[(h0 + 8) * kTeamWarps + warp] = mx1;
    }
    team_sync(team);
    // the staging buffer is free again: this team's next page is fetched in
    // parts between the PV k-steps below, where the copies overlap the MMAs
    // instead of stalling every warp of the team on the load/store queue
    const bool stage_next = kPacked && tile_i + kTeams < n_pages;
    float t0, t1;
    {
      static_assert(kTeamWarps == 8, "two float4 per head");
      const float4* r0 = reinterpret_cast<const float4*>(smax + h0 * kTeamWarps);
      const float4* r1 = reinterpret_cast<const float4*>(smax + (h0 + 8) * kTeamWarps);
      const float4 a0 = r0[0], b0 = r0[1], a1 = r1[0], b1 = r1[1];
      t0 = fmaxf(fmaxf(fmaxf(a0.x, a0.y), fmaxf(a0.z, a0.w)), fmaxf(fmaxf(b0.x, b0.y), fmaxf(b0.z, b0.w)));
      t1 = fmaxf(fmaxf(fmaxf(a1.x, a1.y), fmaxf(a1.z, a1.w)), fmaxf(fmaxf(b1.x, b1.y), fmaxf(b1.z, b1.w)));
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
    team_sync(team);

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
        constexpr int kPart = (kStageIters + 2) / 3;
        if (stage_next && ks < 3)
          stage_part(tile_i + kTeams, kPart * ks, min(kPart * (ks + 1), kStageIters));
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
    cp_async_commit();  // the next page's parts (an empty group when none)
  }

  // ---- epilogue: finish the min term, merge the two teams, write the partial
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    accm0 += __shfl_xor_sync(0xffffffffu, accm0, o);
    accm1 += __shfl_xor_sync(0xffffffffu, accm1, o);
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    O[c][0] += accm0;
    O[c][1] += accm0;
    O[c][2] += accm1;
    O[c][3] += accm1;
  }
  // team 1 hands its state to team 0 through team 1's content tile
  float* xch = reinterpret_cast<float*>(smem + kOffTeam + team_bytes(CB) + kTOffTile) + ttid * 36;
  __syncthreads();
  if (team == 1) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<float4*>(xch + 4 * c) = make_float4(O[c][0], O[c][1], O[c][2], O[c][3]);
    *reinterpret_cast<float4*>(xch + 32) = make_float4(m_run0, m_run1, l0, l1);
  }
  __syncthreads();
  if (team == 1) return;
  {
    const float4 ml = *reinterpret_cast<const float4*>(xch + 32);
    const float M0 = fmaxf(m_run0, ml.x), M1 = fmaxf(m_run1, ml.y);
    const float a0 = M0 == -INFINITY ? 0.f : fast_exp2(m_run0 - M0);
    const float b0 = M0 == -INFINITY ? 0.f : fast_exp2(ml.x - M0);
    const float a1 = M1 == -INFINITY ? 0.f : fast_exp2(m_run1 - M1);
    const float b1 = M1 == -INFINITY ? 0.f : fast_exp2(ml.y - M1);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 o = *reinterpret_cast<const float4*>(xch + 4 * c);
      O[c][0] = a0 * O[c][0] + b0 * o.x;
      O[c][1] = a0 * O[c][1] + b0 * o.y;
      O[c][2] = a1 * O[c][2] + b1 * o.z;
      O[c][3] = a1 * O[c][3] + b1 * o.w;
    }
    m_run0 = M0;
    m_run1 = M1;
    l0 = a0 * l0 + b0 * ml.z;
    l1 = a1 * l1 + b1 * ml.w;
  }
  const int g = warp;
  const long long sidx = blockIdx.x;
  const int hg0 = hc * kHC + h0, hg1 = hg0 + 8;
  float* o0 = a.part_o + (sidx * a.H + hg0) * kLatent + g * 64;
  float* o1 = a.part_o + (sidx * a.H + hg1) * kLatent + g * 64;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    o0[phys_of_chunk(c, 2 * j, kTypeB)] = O[c][0];
    o0[phys_of_chunk(c, 2 * j + 1, kTypeB)] = O[c][1];
    o1[phys_of_chunk(c, 2 * j, kTypeB)] = O[c][2];
    o1[phys_of_chunk(c, 2 * j + 1, kTypeB)] = O[c][3];
  }
  if (warp == 0 && j == 0) {
    a.part_ml[(sidx * a.H + hg0) * 2] = m_run0;
    a.part_ml[(sidx * a.H + hg0) * 2 + 1] = l0;
    a.part_ml[(sidx * a.H + hg1) * 2] = m_run1;
    a.part_ml[(sidx * a.H + hg1) * 2 + 1] = l1;
  }
  // this CTA's partial is written: the combine may be launched
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- combine
struct CombineArgs {
  const float* part_o;
  const float* part_ml;
  const int32_t* seq_split;
  float* out;
  float* lse;
  int B, H, total_splits;
  int rotate;  // the splits hold R o for each content group: apply R (= R^T) back
};

constexpr int kCombineWarps = 2;  // 128-channel quarters per block
constexpr int kCombineThreads = kCombineWarps * 32;

// One warp per (sequence, head, 128-channel quarter).  Lane s holds the
// weights 2^(m_s - M) of splits s and s + 32 (splits beyond 64 recompute
// theirs); every lane then sums its 4 channels over the splits with the
// weight broadcast by shuffle: no shared memory and no block barrier.  Launched as a programmatic dependent
// of the split kernel, it waits for the split kernel's results before reading
// them.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (item >= a.B * a.H * 4) return;
  const int quarter = item & 3, bh = item >> 2, b = bh / a.H, h = bh % a.H;
  int off = a.seq_split[2 * b], n = a.seq_split[2 * b + 1];
  off = min(max(off, 0), a.total_splits);
  n = min(max(n, 0), a.total_splits - off);
  const float* ml = a.part_ml + ((long long)off * a.H + h) * 2;
  const long long mstride = (long long)a.H * 2;
  // lane s holds splits s and s + 32 (weights by shuffle); splits from 64 on
  // recompute theirs
  float m1 = -INFINITY, l1 = 0.f, m2 = -INFINITY, l2 = 0.f;
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) {
    const float2 v = *reinterpret_cast<const float2*>(ml + s * mstride);
    if (s < 32) {
      m1 = v.x;
      l1 = v.y;
    } else if (s < 64) {
      m2 = v.x;
      l2 = v.y;
    }
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w1 = (l1 > 0.f && M != -INFINITY) ? fast_exp2(m1 - M) : 0.f;
  const float w2 = (l2 > 0.f && M != -INFINITY) ? fast_exp2(m2 - M) : 0.f;
  float den = w1 * l1 + w2 * l2;
  for (int s = lane + 64; s < n; s += 32) {
    const float2 v = *reinterpret_cast<const float2*>(ml + s * mstride);
    den += v.y > 0.f ? fast_exp2(v.x - M) * v.y : 0.f;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const int c = quarter * 128 + lane * 4;
  const float* o = a.part_o + ((long long)off * a.H + h) * kLatent + c;
  const long long ostride = (long long)a.H * kLatent;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  // the first 64 splits in batches of 16 loads issued together (the partials
  // are L2-resident: latency, not bandwidth, sets the time)
  constexpr int kBatch = 16;
  const int n64 = min(n, 64);
  for (int s0 = 0; s0 < n64; s0 += kBatch) {
    float4 v[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      if (s0 + k < n64) v[k] = *reinterpret_cast<const float4*>(o + (s0 + k) * ostride);
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (s0 + k < n64) {
        const int sk = s0 + k;
        const float w = __shfl_sync(0xffffffffu, sk < 32 ? w1 : w2, sk & 31);
        acc.x = fmaf(w, v[k].x, acc.x);
        acc.y = fmaf(w, v[k].y, acc.y);
        acc.z = fmaf(w, v[k].z, acc.z);
        acc.w = fmaf(w, v[k].w, acc.w);
      }
    }
  }
  for (int s = 64; s < n; ++s) {
    const float2 mv = *reinterpret_cast<const float2*>(ml + s * mstride);
    const float w = mv.y > 0.f ? fast_exp2(mv.x - M) : 0.f;
    const float4 v = *reinterpret_cast<const float4*>(o + s * ostride);
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  if (a.rotate) {
    // Sylvester H64 / 8 over the group of 16 lanes (4 channels each) this
    // lane belongs to: stages 1 and 2 inside the lane, 4..32 across lanes
    float x[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int hh = 1; hh < 4; hh <<= 1)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (!(i & hh)) {
          const float u = x[i], v = x[i + hh];
          x[i] = u + v;
          x[i + hh] = u - v;
        }
#pragma unroll
    for (int lb = 1; lb < 16; lb <<= 1)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = __shfl_xor_sync(0xffffffffu, x[i], lb);
        x[i] = (lane & lb) ? p - x[i] : x[i] + p;
      }
    acc = make_float4(x[0] * 0.125f, x[1] * 0.125f, x[2] * 0.125f, x[3] * 0.125f);
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  *reinterpret_cast<float4*>(a.out + ((long long)b * a.H + h) * kLatent + c) =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (a.lse && quarter == 0 && lane == 0)
    a.lse[(long long)b * a.H + h] = den > 0.f ? (M + log2f(den)) * 0.69314718055994531f
                                              : -INFINITY;
}

// Launch the combine as a programmatic dependent of the kernel just queued on
// `stream`, so that its launch overlaps the split kernel's last CTAs.
static cudaError_t launch_combine(const CombineArgs& ca, cudaStream_t stream) {
  const int items = ca.B * ca.H * 4;
  if (items == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((items + kCombineWarps - 1) / kCombineWarps);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, ca);
}

// Kernel for a layout and a row count (n_q * heads), fixed by those alone:
// a multiple of 128 rows without rotation takes the 2-CTA tcgen05 kernel
// (decode_wide.cu, one cluster per split and 128-row block; packed or bf16
// pages); everything else the mma.sync kernel above in 16-row chunks.
static bool use_wide(int cbits, int rotate, int rows) {
  (void)cbits;
  return !rotate && rows % 128 == 0;
}

// 128 pages for the cluster kernel (8,192 tokens: max-abs 7.4e-4 against the
// fp64 oracle on a 131,072-token sequence with 128 heads, against 4.3e-4 at
// 64), 64 for the 16-row kernel.
int decode_max_split_pages(int cbits, int rows, int rotate) { return use_wide(cbits, rotate, rows) ? 128 : 64; }
int decode_ctas_per_split(int cbits, int rows, int rotate) {
  return use_wide(cbits, rotate, rows) ? 2 * (rows / 128) : rows / kHC;
}

bool decode_fuses_append(int cbits, int rotate, int rows) {
  return cbits != 16 && !use_wide(cbits, rotate, rows);
}

cudaError_t launch_decode(int cbits, const DecodeArgs& a, float* out, float* lse,
                          cudaStream_t stream) {
  if (use_wide(cbits, a.rotate, a.H)) {
    const cudaError_t et = launch_decode_wide(cbits, a, stream);
    if (et != cudaSuccess) return et;
    CombineArgs ca{a.part_o, a.part_ml, a.seq_split, out, lse, a.B, a.H, a.total_splits, 0};
    return launch_combine(ca, stream);
  }
  const bool rot = a.rotate && cbits != 16;
  void (*kern)(DecodeArgs) = cbits == 4   ? (rot ? decode_split_kernel<4, true> : decode_split_kernel<4, false>)
                             : cbits == 2 ? (rot ? decode_split_kernel<2, true> : decode_split_kernel<2, false>)
                                          : decode_split_kernel<16, false>;
  const int smem = smem_bytes(cbits, rot);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.total_splits, a.H / kHC), block(kThreads);
  kern<<<grid, block, smem, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CombineArgs ca{a.part_o, a.part_ml, a.seq_split, out, lse, a.B, a.H, a.total_splits, rot ? 1 : 0};
  return launch_combine(ca, stream);
}

}  // namespace mlalb
