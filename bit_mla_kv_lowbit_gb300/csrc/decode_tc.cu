// Split-KV low-bit MLA decode on the 5th-generation tensor cores (tcgen05,
// accumulators in tensor memory) for packed caches, 16 heads per CTA.
//
// What it computes is the same as decode.cu (QuantMLA, Abstract and Figure 8
// caption; exact integer codes, fp32 per-group scale/min, P*scale split into
// fp16 high and low parts).  The difference is how the contractions are laid
// out for tcgen05, whose small MMAs are bound by the issue rate of each issuing
// thread (about one MMA per 150 cycles) rather than by arithmetic:
//
// * A tile is 32 tokens (half a page).  The unpacked codes of group g form a
//   32 x 64 fp16 "plane" (128-byte rows, 128-byte swizzle).  Four consecutive
//   planes form a 128-row K-major operand, so one QK MMA (M=128, N=64, K=16)
//   multiplies groups g..g+3 against the queries of the same four groups; the
//   useful results are the diagonal blocks, and TMEM lane quadrant q holds
//   group g+q for the 32 tokens.  12 MMAs per tile cover all 9 groups.
// * PV for groups (2p, 2p+1): the same planes read as an MN-major operand
//   (M=128 channels, K=tokens) times B = [P*s_2p hi | lo | P*s_2p+1 hi | lo]
//   (N=64), accumulating in TMEM over the whole split.  8 MMAs per tile.
// * The min term sum_t p_t m'_t,g and the softmax denominator come from one
//   more small MMA: A = [m' hi (8 groups) ; m' lo ; ones] per token, B = [P hi | P lo].
//
// Warp roles (512 threads, one CTA per SM):
//   warps 0-3   unpack: packed bytes (cp.async staging) -> fp16 planes,
//               metadata, min matrix;
//   warps 4-11  softmax: read QK accumulators (two warps per TMEM lane
//               quadrant, 8 heads each), fold scales, online softmax, write
//               the P*s operands;
//   warps 12-15 MMA issue (one lane each), and warp 12 owns the TMEM
//               allocation.
// Hand-offs use mbarriers; every wait is bounded and, if it gives up, the CTA
// records MLA_LOWBIT_DEV_PIPELINE, skips the remaining work and still frees its
// tensor memory.
#include "decode_common.cuh"
#include "tc_util.cuh"

namespace mlalb {
namespace tc {

constexpr int kThreads = 512;
constexpr int kTok = 32;                 // tokens per tile
constexpr int kNB = 3;                   // operand ring depth
constexpr int kPlane = kTok * 128;       // 4096 B: 32 rows x 64 fp16
constexpr int kABuf = 10 * kPlane;       // planes 0..8 + min matrix
constexpr int kQPlane = 16 * 128;        // 2048 B: 16 heads x 64 fp16
constexpr float kLazy = 2.0f;            // rescale O only when the max grows by more (log2 units)

// shared memory layout (bytes); the A ring is followed directly by the q planes
// so that the junk rows of the last QK group quad read valid memory.
constexpr int kOffA = 0;
constexpr int kOffQ = kOffA + kNB * kABuf;
constexpr int kOffPs = kOffQ + 12 * kQPlane;        // P*s operands: 4 pairs x 32 rows x 128 B
constexpr int kOffPm = kOffPs + 4 * kPlane;         // [P hi | P lo | 0]: 32 rows x 128 B
constexpr int kOffMeta = kOffPm + kPlane;           // [NB][9][32] raw (s16, m16)
constexpr int kXStride = 20;                          // floats per exchange row (padded)
constexpr int kOffX = kOffMeta + kNB * 9 * kTok * 4;  // S partials [4][32][20] fp32
constexpr int kOffTmax = kOffX + 4 * kTok * kXStride * 4;  // [16] fp32
constexpr int kOffMt = kOffTmax + 64;                 // min-term rows [17][16] (16 = denominator)
constexpr int kOffQsum = kOffMt + 17 * 16 * 4;
constexpr int kOffScan = kOffQsum + 9 * 16 * 4;
constexpr int kOffBar = kOffScan + 64 * 4;          // mbarriers (8 B each)
constexpr int kOffMisc = kOffBar + 16 * 8;          // tmem base, abort flag
constexpr int kStages = 3;                          // cp.async staging ring of the unpack warps
constexpr int kStageBytes = 6 * 2048;               // 6 x 16 B per unpack thread (SoA)
constexpr int kOffStage = kOffMisc + 64;
constexpr int kOffValid = kOffStage + kStages * kStageBytes;
constexpr int kSmem = kOffValid + kStages * 128;
static_assert(kSmem + 1024 <= 227 * 1024, "shared memory budget (with 1 KB alignment slack)");

// mbarrier slots
constexpr int kBarAFull = 0;   // [kNB] count 128 (unpack threads)
constexpr int kBarAFree = 3;   // [kNB] count 4 (issuer commits of PV + min term)
constexpr int kBarQK = 6;      // count 3 (QK issuer commits)
constexpr int kBarDFree = 7;   // count 256 (softmax threads)
constexpr int kBarPFull = 8;   // count 256 (softmax threads)
constexpr int kBarPV = 9;      // count 4 (issuer commits)
constexpr int kBarFlush = 10;  // [4] count 1 each (final drain of issuer k)

// TMEM columns
constexpr uint32_t kColQK = 0;     // 3 quads x 64
constexpr uint32_t kColO = 192;    // 4 pairs x 64
constexpr uint32_t kColM = 448;    // 64
constexpr uint32_t kTmemCols = 512;

template <int CB>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(DecodeArgs a) {
  constexpr bool kTypeB = CB == 2;
  constexpr PageGeom G = page_geom(CB);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle is a function of absolute shared addresses: align to 1 KB
  uint8_t* smem = smem_raw + ((1024 - (su32(smem_raw) & 1023)) & 1023);
  uint8_t* sA = smem + kOffA;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sPs = smem + kOffPs;
  uint8_t* sPm = smem + kOffPm;
  uint32_t* sMeta = reinterpret_cast<uint32_t*>(smem + kOffMeta);
  float* sX = reinterpret_cast<float*>(smem + kOffX);
  float* sTmax = reinterpret_cast<float*>(smem + kOffTmax);
  float* sMt = reinterpret_cast<float*>(smem + kOffMt);
  float* qsum = reinterpret_cast<float*>(smem + kOffQsum);
  int* scan = reinterpret_cast<int*>(smem + kOffScan);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  uint8_t* sStage = smem + kOffStage;
  uint8_t* sValid = smem + kOffValid;
  auto bar = [&](int i) { return su32(&bars[i]); };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int b, split, nsplit;
  find_split<kThreads>(a, true, scan, b, split, nsplit);
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

  // ---- work of this split: packed pages (two tiles each), then the
  // protected bf16 tokens of its bf16 units in 32-token tiles
  const SplitWork sw = split_work(L, split, a.chunk_pages, true);
  const int page_begin = sw.page_begin, n_pk = 2 * sw.n_pages;
  const int bf_first = 64 * sw.bf_begin;  // first protected-token index of the split
  const int bf_end = min(sw.n_tok, 64 * (sw.bf_begin + sw.n_bf));
  const int n_tiles = n_pk + max(0, (bf_end - bf_first + kTok - 1) / kTok);

  // ---- set-up: barriers, TMEM, q planes, zero regions
  if (tid == 0) {
    for (int i = 0; i < kNB; ++i) {
      bar_init(bar(kBarAFull + i), 128);
      bar_init(bar(kBarAFree + i), 4);
    }
    bar_init(bar(kBarQK), 3);
    bar_init(bar(kBarDFree), 256);
    bar_init(bar(kBarPFull), 256);
    bar_init(bar(kBarPV), 4);
    for (int k = 0; k < 4; ++k) bar_init(bar(kBarFlush + k), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 12) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // zero: min-matrix planes (rows 17..63 stay zero), Pm (columns 32..63 stay
  // zero), q planes 9..11
  for (int i = tid; i < kNB * kPlane / 16; i += kThreads) {
    const int buf = i / (kPlane / 16), off = i % (kPlane / 16);
    reinterpret_cast<uint4*>(sA + buf * kABuf + 9 * kPlane)[off] = make_uint4(0, 0, 0, 0);
  }
  for (int i = tid; i < kPlane / 16; i += kThreads)
    reinterpret_cast<uint4*>(sPm)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < 3 * kQPlane / 16; i += kThreads)
    reinterpret_cast<uint4*>(sQ + 9 * kQPlane)[i] = make_uint4(0, 0, 0, 0);
  // q planes 0..8 in the unpack's permuted channel order, and the group sums
  if (tid < kGroups * kHC) {
    const int g = tid / kHC, h = tid % kHC;
    const bool tb = g < 8 ? kTypeB : false;
    const uint16_t* src = a.q + ((long long)b * a.H + hc * kHC + h) * kDim + g * 64;
    uint4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = reinterpret_cast<const uint4*>(src)[c];
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(v);
    float acc = 0.f;
    uint8_t* plane = sQ + g * kQPlane;
    for (int c = 0; c < 8; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const int p0 = chan_of_pos(c, 2 * e2, tb), p1 = chan_of_pos(c, 2 * e2 + 1, tb);
        const __half h0 = __float2half_rn(__uint_as_float((uint32_t)vs[p0] << 16));
        const __half h1 = __float2half_rn(__uint_as_float((uint32_t)vs[p1] << 16));
        acc += __half2float(h0) + __half2float(h1);
        w[e2] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
      }
      *reinterpret_cast<uint4*>(plane + sw_chunk(h, c)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    qsum[g * kHC + h] = acc;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // =====================================================================
  if (warp < 4) {
    // ---------------- unpack warps: thread (token t = lane, part q = warp)
    // handles content groups q and q + 4, RoPE channels 16q..16q+15 and the
    // metadata words of those groups.  Packed bytes arrive by cp.async in a
    // per-thread staging ring (structure of arrays: conflict-free reads),
    // two tiles ahead.
    const int t = lane, q = warp, u = tid;
    auto stage_at = [&](int s, int unit) { return sStage + s * kStageBytes + unit * 2048 + u * 16; };
    auto issue = [&](int i) {
      uint8_t okb = 0;
      if (i < n_pk) {
        const int page_idx = page_begin + (i >> 1);
        const int r = (i & 1) * kTok + t;
        const long long page = a.block_table[(long long)b * a.max_pages + page_idx];
        const int pos = page_idx * kPageTokens + r;
        if (page < 0 || page >= a.num_pages) {
          if (u == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
        } else {
          okb = 1 | ((pos >= kSink && pos < L - kLocal) ? 2 : 0);
          const uint8_t* pb = a.pool + page * G.page_bytes;
          const int s = i % kStages;
          const uint8_t* crow = pb + G.content_off + r * G.content_row;
          if constexpr (CB == 4) {
            cp_async(stage_at(s, 0), crow + 32 * q, 16);
            cp_async(stage_at(s, 1), crow + 32 * q + 16, 16);
            cp_async(stage_at(s, 2), crow + 32 * (q + 4), 16);
            cp_async(stage_at(s, 3), crow + 32 * (q + 4) + 16, 16);
          } else {
            cp_async(stage_at(s, 0), crow + 16 * q, 16);
            cp_async(stage_at(s, 2), crow + 16 * (q + 4), 16);
          }
          cp_async(stage_at(s, 4), pb + G.rope_off + r * G.rope_row + 8 * q, 8);
          const uint8_t* mrow = pb + G.meta_off + r * G.meta_row;
          cp_async(stage_at(s, 5), mrow + 4 * q, 4);
          cp_async(stage_at(s, 5) + 4, mrow + 4 * (q + 4), 4);
          if (q == 0) cp_async(stage_at(s, 5) + 8, mrow + 32, 4);
        }
      }
      if (i < n_tiles) sValid[(i % kStages) * 128 + u] = okb;
      cp_async_commit();
    };
    issue(0);
    issue(1);
    for (int i = 0; i < n_tiles; ++i) {
      const int buf = i % kNB;
      if (i >= kNB && !bar_wait(bar(kBarAFree + buf), ((i / kNB) - 1) & 1, abort_flag, a.err))
        break;
      uint8_t* A = sA + buf * kABuf;
      uint32_t* meta = sMeta + buf * 9 * kTok;
      uint8_t* mm = A + 9 * kPlane;
      const float centre = kTypeB ? float(kCentre2) : float(kCentre4);
      issue(i + 2);
      if (i < n_pk) {
        cp_async_wait<2>();
        const int s = i % kStages;
        const uint8_t okb = sValid[s * 128 + u];
        const bool sok = okb & 1, okt = okb & 2;
        uint4 cc[4];
        uint2 rr;
        uint32_t mw[3];
        if (sok) {
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) cc[k2] = *reinterpret_cast<const uint4*>(stage_at(s, k2));
          rr = *reinterpret_cast<const uint2*>(stage_at(s, 4));
          const uint4 m4 = *reinterpret_cast<const uint4*>(stage_at(s, 5));
          mw[0] = m4.x;
          mw[1] = m4.y;
          mw[2] = m4.z;
        } else {
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) cc[k2] = make_uint4(0, 0, 0, 0);
          rr = make_uint2(0, 0);
          mw[0] = mw[1] = mw[2] = 0;
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int g = q + 4 * half;
          uint8_t* plane = A + g * kPlane;
          if constexpr (CB == 4) {
            const uint4 c0 = cc[2 * half], c1 = cc[2 * half + 1];
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {
              uint32_t p[4];
              unpack_int4(w[k2], p);
              *reinterpret_cast<uint4*>(plane + sw_chunk(t, k2)) = make_uint4(p[0], p[1], p[2], p[3]);
            }
          } else {
            const uint4 c0 = cc[2 * half];
            const uint32_t w[4] = {c0.x, c0.y, c0.z, c0.w};
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              uint32_t p[8];
              unpack_int2(w[k2], p);
              *reinterpret_cast<uint4*>(plane + sw_chunk(t, 2 * k2)) = make_uint4(p[0], p[1], p[2], p[3]);
              *reinterpret_cast<uint4*>(plane + sw_chunk(t, 2 * k2 + 1)) = make_uint4(p[4], p[5], p[6], p[7]);
            }
          }
          const uint32_t mword = mw[half];
          meta[g * kTok + t] = okt ? mword : 0u;
          const float2 sm = __half22float2(*reinterpret_cast<const __half2*>(&mword));
          const float mp = okt ? fmaf(centre, sm.x, sm.y) : 0.f;
          const __half hi = __float2half_rn(mp);
          const __half lo = __float2half_rn(mp - __half2float(hi));
          *reinterpret_cast<__half*>(mm + sw_off(t, g)) = hi;
          *reinterpret_cast<__half*>(mm + sw_off(t, 8 + g)) = lo;
        }
        {
          // RoPE channels 16q..16q+15: two words -> chunks 2q, 2q+1 of plane 8
          uint32_t p[4];
          unpack_int4(rr.x, p);
          *reinterpret_cast<uint4*>(A + 8 * kPlane + sw_chunk(t, 2 * q)) = make_uint4(p[0], p[1], p[2], p[3]);
          unpack_int4(rr.y, p);
          *reinterpret_cast<uint4*>(A + 8 * kPlane + sw_chunk(t, 2 * q + 1)) = make_uint4(p[0], p[1], p[2], p[3]);
        }
        if (q == 0) {
          meta[8 * kTok + t] = okt ? mw[2] : 0u;
          *reinterpret_cast<__half*>(mm + sw_off(t, 16)) = __float2half(okt ? 1.f : 0.f);
        }
      } else {
        // bf16 rows (protected tokens): values in place of codes, scale 1, min 0
        const int idx = bf_first + (i - n_pk) * kTok + t;
        const bool okt = idx < bf_end;
        const uint16_t* rp = nullptr;
        if (okt) {
          const int pos = bf16_pos(sw, idx);
          rp = pos < kSink ? a.sink + ((long long)b * kSink + pos) * kDim
                           : a.recent + ((long long)b * kLocal + pos % kLocal) * kDim;
        }
#pragma unroll 1
        for (int gi = 0; gi < 3; ++gi) {
          const int g = gi == 2 ? 8 : q + 4 * gi;
          if (gi == 2 && q != 0) {
            // plane 8 is split: thread q writes channels 16q..16q+15
          }
          const bool tb = g < 8 ? kTypeB : false;
          uint8_t* plane = A + g * kPlane;
          // channels handled by this thread in group g: all 64 for content
          // groups q, q+4; 16q..16q+15 for the RoPE group
          const int c_lo = g == 8 ? 16 * q : 0, c_hi = g == 8 ? 16 * q + 16 : 64;
          for (int ch0 = c_lo; ch0 < c_hi; ch0 += 8) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (okt) v = *reinterpret_cast<const uint4*>(rp + g * 64 + ch0);
            const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float f = (e & 1) ? bf16hi_to_f32(vv[e >> 1]) : bf16lo_to_f32(vv[e >> 1]);
              const int ch = ch0 + e;
              int c, pos;
              if (!tb) {
                c = ch >> 3;
                pos = 2 * (ch & 3) + ((ch & 4) ? 1 : 0);
              } else {
                const int r16 = ch & 15;
                c = 2 * (ch >> 4) + ((r16 & 4) ? 1 : 0);
                pos = 2 * (r16 & 3) + (r16 >= 8 ? 1 : 0);
              }
              *reinterpret_cast<__half*>(plane + sw_off(t, 8 * c + pos)) = __float2half_rn(f);
            }
          }
          if (g < 8) {
            meta[g * kTok + t] = okt ? 0x00003C00u : 0u;  // (s = 1, m = 0)
            *reinterpret_cast<__half*>(mm + sw_off(t, g)) = __float2half(0.f);
            *reinterpret_cast<__half*>(mm + sw_off(t, 8 + g)) = __float2half(0.f);
          }
        }
        if (q == 0) {
          meta[8 * kTok + t] = okt ? 0x00003C00u : 0u;
          *reinterpret_cast<__half*>(mm + sw_off(t, 16)) = __float2half(okt ? 1.f : 0.f);
        }
      }
      fence_async_smem();
      bar_arrive(bar(kBarAFull + buf));
    }
    cp_async_wait<0>();
  } else if (warp < 12) {
    // ---------------- softmax warps: quadrant qd, heads 8hh..8hh+7, token t = lane
    const int qd = warp & 3, hh = (warp - 4) >> 2, t = lane, f = tid - 128;
    const int h0 = 8 * hh;
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
    float m_run[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) m_run[h] = -INFINITY;
    // min-term rows held by this lane (quadrant 0 lanes 0..15, quadrant 1 lane
    // 0 = denominator), for heads h0..h0+7, summed in fp32 across tiles
    float accm[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) accm[h] = 0.f;
    auto add_mterm = [&]() {
      if (qd < 2) {
        float v[8], w[8];
        tmem_ld8(tl + kColM + h0, v);
        tmem_ld8(tl + kColM + 16 + h0, w);
#pragma unroll
        for (int h = 0; h < 8; ++h) accm[h] += v[h] + w[h];
      }
    };
    const float centre_bf = 0.f;
    for (int i = 0; i < n_tiles; ++i) {
      const int buf = i % kNB;
      if (!bar_wait(bar(kBarQK), i & 1, abort_flag, a.err)) break;
      tc_fence_after();
      float S[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) S[h] = 0.f;
      const uint32_t* meta = sMeta + buf * 9 * kTok;
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int g = 4 * k + qd;
        if (g > 8) break;
        float D[8];
        tmem_ld8(tl + kColQK + 64 * k + 16 * qd + h0, D);
        const uint32_t mw = meta[g * kTok + t];
        const float2 sm = __half22float2(*reinterpret_cast<const __half2*>(&mw));
        const float centre = i >= n_pk ? centre_bf
                             : ((g < 8 && kTypeB) ? float(kCentre2) : float(kCentre4));
        const float s = sm.x, mp = fmaf(centre, sm.x, sm.y);
        const float4 qa = *reinterpret_cast<const float4*>(qsum + g * kHC + h0);
        const float4 qb = *reinterpret_cast<const float4*>(qsum + g * kHC + h0 + 4);
        const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
        for (int h = 0; h < 8; ++h) S[h] += s * D[h] + mp * qv[h];
      }
      tc_fence_before();
      bar_arrive(bar(kBarDFree));
      // exchange partial logits across the four quadrants (heads h0..h0+7)
      {
        float4* x4 = reinterpret_cast<float4*>(sX + (qd * kTok + t) * kXStride + h0);
        x4[0] = make_float4(S[0], S[1], S[2], S[3]);
        x4[1] = make_float4(S[4], S[5], S[6], S[7]);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
#pragma unroll
      for (int h = 0; h < 8; ++h) S[h] = 0.f;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const float4* y4 = reinterpret_cast<const float4*>(sX + (qq * kTok + t) * kXStride + h0);
        const float4 y0 = y4[0], y1 = y4[1];
        S[0] += y0.x; S[1] += y0.y; S[2] += y0.z; S[3] += y0.w;
        S[4] += y1.x; S[5] += y1.y; S[6] += y1.z; S[7] += y1.w;
      }
      const bool okt =
          __half2float(*reinterpret_cast<const __half*>(sA + buf * kABuf + 9 * kPlane + sw_off(t, 16))) != 0.f;
#pragma unroll
      for (int h = 0; h < 8; ++h) S[h] = okt ? S[h] * a.scale_log2 : -INFINITY;
      // tile max: warp (qd, hh) reduces heads h0 + 2qd, h0 + 2qd + 1 over the tokens
#pragma unroll
      for (int hx = 0; hx < 2; ++hx) {
        float v = S[2 * qd + hx];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) sTmax[h0 + 2 * qd + hx] = v;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      bool need = false;
#pragma unroll
      for (int h = 0; h < 16; ++h) need |= (m_run[h] != -INFINITY) && (sTmax[h] > m_run[h] + kLazy);
      if (i > 0) {
        // PV of the previous tile must be done: the P operands are reused and O
        // may need rescaling
        if (!bar_wait(bar(kBarPV), (i - 1) & 1, abort_flag, a.err)) break;
        tc_fence_after();
        add_mterm();  // previous tile's min term, at the previous scale
      }
      if (need) {
        // raise the running max of every head whose tile max exceeds it and
        // rescale what has been accumulated so far
        float alpha[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float mu = fmaxf(m_run[h], sTmax[h]);
          alpha[h] = (m_run[h] == -INFINITY || mu == -INFINITY) ? 1.f : fast_exp2(m_run[h] - mu);
          m_run[h] = mu;
        }
#pragma unroll
        for (int h = 0; h < 8; ++h) accm[h] *= alpha[h0 + h];
        // O of my lane: blocks 8hh..8hh+7 (16 columns = heads 0..15 each)
        for (int c = 0; c < 8; ++c) {
          const uint32_t col = kColO + 16 * (8 * hh + c);
          float v[16];
          tmem_ld16(tl + col, v);
#pragma unroll
          for (int h = 0; h < 16; ++h) v[h] *= alpha[h];
          tmem_st16(tl + col, v);
        }
      } else {
#pragma unroll
        for (int h = 0; h < 16; ++h)
          if (m_run[h] == -INFINITY) m_run[h] = sTmax[h];
      }
      // p and P*s operands: row t of pair qd, heads h0..h0+7
      float p[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) p[h] = S[h] == -INFINITY ? 0.f : fast_exp2(S[h] - m_run[h0 + h]);
      {
        uint8_t* ps = sPs + qd * kPlane;
#pragma unroll
        for (int gg = 0; gg < 2; ++gg) {
          const int g = 2 * qd + gg;
          const uint32_t mw = meta[g * kTok + t];
          const float s = __half2float(*reinterpret_cast<const __half*>(&mw));
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int h2 = 0; h2 < 4; ++h2) split_hi_lo(p[2 * h2] * s, p[2 * h2 + 1] * s, hi[h2], lo[h2]);
          *reinterpret_cast<uint4*>(ps + sw_chunk(t, 4 * gg + hh)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(ps + sw_chunk(t, 4 * gg + 2 + hh)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        if (qd == 0) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int h2 = 0; h2 < 4; ++h2) split_hi_lo(p[2 * h2], p[2 * h2 + 1], hi[h2], lo[h2]);
          *reinterpret_cast<uint4*>(sPm + sw_chunk(t, hh)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(sPm + sw_chunk(t, 2 + hh)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      fence_async_smem();
      tc_fence_before();  // my TMEM accesses precede the next MMAs
      bar_arrive(bar(kBarPFull));
    }
    // ---- epilogue: wait for the last PV, assemble the partial
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const bool have = n_tiles > 0;
    const bool done = have && bar_wait(bar(kBarPV), (n_tiles - 1) & 1, abort_flag, a.err);
    const long long sidx = blockIdx.x;
    if (done) {
      tc_fence_after();
      add_mterm();
      if (qd < 2) {
        const int row = qd == 0 ? (lane < 16 ? lane : -1) : (lane == 0 ? 16 : -1);
        if (row >= 0) {
#pragma unroll
          for (int h = 0; h < 8; ++h) sMt[row * 16 + h0 + h] = accm[h];
        }
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const int L_lane = 32 * qd + lane;  // TMEM lane = channel within the pair
      const int half = L_lane >> 6, ch = L_lane & 63;
      const int logical_c = ch >> 3, e = ch & 7;
#pragma unroll 1
      for (int pr = 0; pr < 4; ++pr) {
        const int g = 2 * pr + half;
        float oh[8], ol[8];
        tmem_ld8(tl + kColO + 64 * pr + 32 * half + h0, oh);
        tmem_ld8(tl + kColO + 64 * pr + 32 * half + 16 + h0, ol);
        const int phys = g * 64 + chan_of_pos(logical_c, e, kTypeB);
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float mt = sMt[g * 16 + h0 + h] + sMt[(8 + g) * 16 + h0 + h];
          a.part_o[(sidx * a.H + hc * kHC + h0 + h) * kLatent + phys] = oh[h] + ol[h] + mt;
        }
      }
      if (f < 16) {
        a.part_ml[(sidx * a.H + hc * kHC + f) * 2] = m_run[f];
        a.part_ml[(sidx * a.H + hc * kHC + f) * 2 + 1] = sMt[16 * 16 + f];
      }
    } else {
      // no tokens in this split (or a time-out): an empty partial
      for (int i = f; i < kHC * kLatent; i += 256)
        a.part_o[(sidx * a.H + hc * kHC + i / kLatent) * kLatent + i % kLatent] = 0.f;
      if (f < 16) {
        a.part_ml[(sidx * a.H + hc * kHC + f) * 2] = -INFINITY;
        a.part_ml[(sidx * a.H + hc * kHC + f) * 2 + 1] = 0.f;
      }
    }
  } else {
    // ---------------- MMA issue warps: issuer k = warp - 12, lane 0.  QK of
    // the next tile is issued before PV of the current one, so the softmax
    // warps find their logits ready.
    const int k = warp - 12;
    if (lane == 0) {
      const uint32_t id_qk = idesc(128, 64, 0, 0);   // A K-major, B K-major
      const uint32_t id_pv = idesc(128, 64, 1, 1);   // A MN-major, B MN-major
      const uint32_t id_m = idesc(64, 64, 1, 1);
      auto issue_qk = [&](int i) {
        const uint32_t A = su32(sA + (i % kNB) * kABuf);
        const uint32_t qa = su32(sQ + 4 * k * kQPlane);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma(tmem + kColQK + 64 * k, desc(A + 4 * k * kPlane + 32 * ks, 16, 1024),
              desc(qa + 32 * ks, 16, 1024), id_qk, ks > 0);
        commit(bar(kBarQK));
      };
      bool ok = n_tiles > 0 && bar_wait(bar(kBarAFull), 0, abort_flag, a.err);
      if (ok) {
        tc_fence_after();
        if (k < 3) issue_qk(0);
      }
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int buf = i % kNB;
        if (i + 1 < n_tiles) {
          const int nb = (i + 1) % kNB;
          if (!bar_wait(bar(kBarAFull + nb), ((i + 1) / kNB) & 1, abort_flag, a.err)) break;
          if (!bar_wait(bar(kBarDFree), i & 1, abort_flag, a.err)) break;
          tc_fence_after();
          if (k < 3) issue_qk(i + 1);
        }
        if (!bar_wait(bar(kBarPFull), i & 1, abort_flag, a.err)) break;
        tc_fence_after();
        const uint32_t A = su32(sA + buf * kABuf);
        const uint32_t pa = A + 2 * k * kPlane;  // planes 2k, 2k+1
        const uint32_t pb = su32(sPs + k * kPlane);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          mma(tmem + kColO + 64 * k, desc(pa + 2048 * ks, kPlane, 1024),
              desc(pb + 2048 * ks, 1024, 1024), id_pv, (i > 0 || ks > 0));
        if (k == 3) {
          const uint32_t ma = A + 9 * kPlane;
          const uint32_t mb = su32(sPm);
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            mma(tmem + kColM, desc(ma + 2048 * ks, 1024, 1024), desc(mb + 2048 * ks, 1024, 1024),
                id_m, ks > 0);
        }
        commit(bar(kBarPV));
        commit(bar(kBarAFree + buf));
      }
      // drain: wait (bounded, regardless of the abort flag) for this issuer's
      // own MMAs before the CTA frees tensor memory
      commit(bar(kBarFlush + k));
      const long long t0 = clock64();
      for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar(kBarFlush + k)), "r"(0)
            : "memory");
        if (ok) break;
        if (clock64() - t0 > kWaitCycles) {
          set_error(a.err, MLA_LOWBIT_DEV_PIPELINE);
          break;
        }
      }
    }
  }

  // ---- teardown: every issuer has drained its MMAs; free tensor memory
  tc_fence_before();
  __syncthreads();
  // the partial of this CTA is written: the combine may be launched
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 12) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

}  // namespace tc

cudaError_t launch_decode_tc(int cbits, const DecodeArgs& a, cudaStream_t stream) {
  static bool configured[2] = {false, false};
  const int k = cbits == 4 ? 0 : 1;
  cudaError_t e = cudaSuccess;
  if (!configured[k]) {
    e = cbits == 4 ? cudaFuncSetAttribute(tc::decode_tc_kernel<4>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmem + 1024)
                   : cudaFuncSetAttribute(tc::decode_tc_kernel<2>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmem + 1024);
    if (e != cudaSuccess) return e;
    configured[k] = true;
  }
  dim3 grid(a.total_splits, a.H / kHC), block(tc::kThreads);
  if (cbits == 4)
    tc::decode_tc_kernel<4><<<grid, block, tc::kSmem + 1024, stream>>>(a);
  else
    tc::decode_tc_kernel<2><<<grid, block, tc::kSmem + 1024, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlalb
