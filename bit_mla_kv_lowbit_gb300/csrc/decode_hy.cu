// Split-KV low-bit MLA decode for packed caches: QK on mma.sync in the warps
// that unpack, PV on the tcgen05 tensor cores with its accumulators in tensor
// memory.  One CTA per (split, 16-head chunk), one CTA per SM.
//
// What it computes is the same as decode.cu (QuantMLA, Abstract and Figure 8
// caption): exact integer codes on the tensor cores, the per-group fp32 scale
// and min applied outside them, P*scale split into fp16 high and low parts for
// PV, and one softmax over all valid tokens.  The split of the work follows
// the cost of each contraction on this GPU: QK has only 16 heads per token, a
// shape the register-fed mma.sync path handles well straight out of the
// unpack, while PV (512 channels x 32 hi/lo head columns per group) suits a
// 128-row tcgen05 MMA that runs asynchronously and costs the unpacking warps
// no issue slots.
//
// Per page of 64 tokens:
//   compute warps 0-7 (warp w owns tokens 8w..8w+7)
//     1. unpack the page (cp.async staging, two pages ahead), QK with mma.sync,
//        fold in s and m' per group, and store the centred fp16 codes into
//        128-byte-swizzled planes (one 64x64 plane per content group);
//     2. page max per head; the running max moves only when a head's page max
//        exceeds it by more than kLazy (then O in tensor memory is rescaled);
//     3. p = 2^(z - m), the min term sum_t p m' and the denominator in
//        registers, and the PV operand P*s (hi, lo) for every (token, group);
//   MMA warp 8 (one lane)
//     4. 16 MMAs M=128 (channels of a group pair) x N=64 ([hi|lo] x 16 heads
//        for both groups) x K=16 tokens into tensor memory, then a commit.
// Planes are double-buffered, so the compute warps unpack page i+1 while the
// tensor cores run PV of page i.  Every wait is bounded; on time-out the CTA
// records MLA_LOWBIT_DEV_PIPELINE, stops at a point all compute warps agree on,
// drains its MMAs and frees its tensor memory.
#include "decode_common.cuh"
#include "tc_util.cuh"

namespace mlalb {
namespace hy {

using namespace tc;

constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kThreads = kComputeThreads + 32;  // + the MMA warp
constexpr int kMmaWarp = kComputeWarps;
constexpr int kPlane = kPageTokens * 128;       // 64 tokens x 64 fp16 (one group)
constexpr int kPlaneSet = 8 * kPlane;           // the 8 content groups of one page
constexpr int kPStride = 20;                    // floats per row of the p buffer (padded)
constexpr uint32_t kTmemCols = 256;             // O: 4 group pairs x 64 columns
// The running max of a head moves only when a page max exceeds it by more
// than kLazy (log2 units), so p = 2^(z - m) stays below 2^kLazy and the costly
// rescale of O in tensor memory is rare.  P*s must stay finite in fp16: that
// holds for s below kBigScale; a page holding a larger scale moves the running
// max (then p <= 1).
constexpr float kLazy = 8.0f;
constexpr float kBigScale = 65504.0f / 256.0f;
static_assert(kLazy <= 8.0f, "kBigScale assumes p <= 2^8");

// shared memory (bytes from a 1024-byte-aligned base)
constexpr int kOffPlanes = 0;                                // [2][8][64 rows][128 B]
constexpr int kOffPs = kOffPlanes + 2 * kPlaneSet;           // [4 pairs][64 rows][128 B]
constexpr int kOffQ = kOffPs + 4 * kPlane;                   // [16][576] fp16, 16 B chunks XOR-swizzled
constexpr int kOffP = kOffQ + kHC * kDim * 2;                // [64][kPStride] fp32; set-up and epilogue scratch
constexpr int kOffS = kOffP + kPageTokens * kPStride * 4;    // [8 groups][64] fp32 scales (0 = invalid)
constexpr int kOffPmax = kOffS + 8 * kPageTokens * 4;        // [8 warps][16] page max, [16] alpha
constexpr int kOffFlags = kOffPmax + (kComputeWarps + 1) * kHC * 4;  // [8] per-warp vote words
constexpr int kOffBar = kOffFlags + kComputeWarps * 4;       // mbarriers
constexpr int kOffMisc = kOffBar + 8 * 8;                    // tmem base, abort flag
constexpr int kOffPages = kOffMisc + 16;                     // [64] page ids of the split
constexpr int kOffStage = kOffPages + 64 * 4;                // [2][page bytes]
__host__ __device__ constexpr int smem_bytes(int cbits) {
  return kOffStage + 2 * page_geom(cbits).page_bytes;
}
static_assert(smem_bytes(4) <= 227 * 1024, "shared memory budget");
static_assert(kOffStage % 16 == 0, "cp.async alignment");
static_assert(kComputeWarps * kHC * 9 * 4 + kHC * 9 * 4 <= kPlaneSet, "epilogue scratch");

// mbarriers
constexpr int kBarPReady = 0;  // count 256: planes and P*s of the page are written
constexpr int kBarPVDone = 1;  // [2] count 1: PV of the pages using plane set 0 / 1 finished
constexpr int kBarFlush = 3;   // count 1: final drain of the MMA warp

// q element e (0..575) of head h, fp16, 16-byte chunks swizzled against the row
__device__ __forceinline__ int q_off(int h, int e) {
  return h * kDim + ((((e >> 3) ^ (h & 7))) << 3) + (e & 7);
}

// XOR applied to the 16-byte chunk index of content row r in the staging copy
template <int CB>
__device__ __forceinline__ int stage_swizzle(int r) {
  return CB == 4 ? ((r & 3) << 1) : (r & 3);
}

__device__ __forceinline__ void bar_sync_compute() {
  asm volatile("bar.sync 1, %0;" ::"n"(kComputeThreads) : "memory");
}

template <int CB>
__global__ void __launch_bounds__(kThreads, 1) decode_hy_kernel(DecodeArgs a) {
  constexpr bool kTypeB = CB == 2;
  constexpr PageGeom G = page_geom(CB);
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the 128-byte swizzle of the MMA operands is a function of the absolute
  // shared address; the dynamic shared window starts 1 KB aligned
  if ((su32(smem) & 1023) != 0) {
    if (tid == 0) set_error(a.err, MLA_LOWBIT_DEV_PIPELINE);
    return;
  }
  uint8_t* planes0 = smem + kOffPlanes;
  uint8_t* sPs = smem + kOffPs;
  __half* qs = reinterpret_cast<__half*>(smem + kOffQ);
  float* pbuf = reinterpret_cast<float*>(smem + kOffP);
  float* smS = reinterpret_cast<float*>(smem + kOffS);
  float* pmax = reinterpret_cast<float*>(smem + kOffPmax);
  int* flags = reinterpret_cast<int*>(smem + kOffFlags);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  uint8_t* stage0 = smem + kOffStage;
  int* s_pages = reinterpret_cast<int*>(smem + kOffPages);
  auto bar = [&](int i) { return su32(&bars[i]); };

  int b, split, nsplit;
  find_split<kThreads>(a, true, reinterpret_cast<int*>(pbuf), b, split, nsplit);
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

  // ---- work of this split: packed pages, then 64-token tiles of the
  // protected bf16 tokens; tile i < n_pages is a page
  const SplitWork sw = split_work(L, split, a.chunk_pages, true);
  const int n_pages = sw.n_pages, page_begin = sw.page_begin;
  int n_tiles = n_pages + sw.n_bf;
  const int valid_lo = kSink, valid_hi = L - kLocal;  // packed-served tokens [lo, hi)
  if (n_tiles > 64) {  // the planner caps splits at 64 pages
    if (tid == 0) set_error(a.err, MLA_LOWBIT_DEV_PLAN);
    n_tiles = 0;
  }

  const int ct = tid;  // compute-thread index (valid for warp < 8)
  auto stage_page = [&](int tile_i) {
    if (tile_i < n_pages) {
      const long long page = s_pages[tile_i];
      if (page >= 0 && page < a.num_pages) {
        const uint8_t* src = a.pool + page * G.page_bytes;
        uint8_t* dst0 = stage0 + (tile_i & 1) * G.page_bytes;
        constexpr int kChunks = G.page_bytes / 16;
        constexpr int kRowChunks = G.content_row / 16;
        constexpr int kContentChunks = kPageTokens * kRowChunks;
        for (int k = ct; k < kChunks; k += kComputeThreads) {
          int dst = k * 16;
          if (k < kContentChunks) {
            const int r = k / kRowChunks, c = k % kRowChunks;
            dst = G.content_off + r * G.content_row + ((c ^ stage_swizzle<CB>(r)) << 4);
          }
          cp_async(dst0 + dst, src + k * 16, 16);
        }
      }
    }
    cp_async_commit();  // one group per page slot, possibly empty
  };

  // ---- set-up: barriers, tensor memory, q (fp16, permuted contraction
  // order, swizzled rows) and its group sums, the first two pages
  if (tid == 0) {
    bar_init(bar(kBarPReady), kComputeThreads);
    bar_init(bar(kBarPVDone), 1);
    bar_init(bar(kBarPVDone + 1), 1);
    bar_init(bar(kBarFlush), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  __syncthreads();  // the scan scratch (p buffer) is free again
  float* qsum_s = pbuf;  // [9][16], read into registers before the first page
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
        qs[q_off(h, g * 64 + logical_of_phys(p, tb))] = hv;
      }
    }
    qsum_s[g * kHC + h] = acc;
  }
  if (tid < n_pages && tid < 64)
    s_pages[tid] = a.block_table[(long long)b * a.max_pages + page_begin + tid];
  __syncthreads();  // page ids visible
  if (warp < kComputeWarps) {
    stage_page(0);
    stage_page(1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long sidx = blockIdx.x;

  if (warp < kComputeWarps) {
    // ======================= compute warps
    const int j = lane & 3, rn = lane >> 2;
    const int h0 = rn;                 // heads h0 and h0 + 8
    const int rowB = warp * 8 + rn;    // page row of this thread's B fragment
    const int tC0 = warp * 8 + 2 * j;  // page rows of this thread's C columns
    float qs0[kGroups], qs1[kGroups];
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      qs0[g] = qsum_s[g * kHC + h0];
      qs1[g] = qsum_s[g * kHC + h0 + 8];
    }
    float m_run0 = -INFINITY, m_run1 = -INFINITY;
    float accm0[8], accm1[8], l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int g = 0; g < 8; ++g) accm0[g] = accm1[g] = 0.f;
    bool local_abort = false;
    int done_tiles = 0;  // pages whose PV has been issued to the MMA warp

    for (int i = 0; i < n_tiles; ++i) {
      const int buf = i & 1;
      uint8_t* planes = planes0 + buf * kPlaneSet;
      cp_async_wait<1>();
      // plane set `buf` is free once PV of page i - 2 has finished
      if (i >= 2 && !local_abort &&
          !bar_wait(bar(kBarPVDone + buf), ((i - 2) >> 1) & 1, abort_flag, a.err))
        local_abort = true;
      bar_sync_compute();  // B0: the staged page is visible to every compute thread

      // -------- 1. unpack + QK + fold, codes to the planes
      float S[4] = {0.f, 0.f, 0.f, 0.f};
      float mp0[8], mp1[8];  // m' of tokens tC0, tC0 + 1 (0 when invalid)
      bool v0, v1, big = false;
      if (i < n_pages) {
        const int page_idx = page_begin + i;
        const long long page = s_pages[i];
        const bool page_ok = page >= 0 && page < a.num_pages;
        if (!page_ok && ct == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
        const int tok0 = page_idx * kPageTokens;
        v0 = page_ok && tok0 + tC0 >= valid_lo && tok0 + tC0 < valid_hi;
        v1 = page_ok && tok0 + tC0 + 1 >= valid_lo && tok0 + tC0 + 1 < valid_hi;
        const uint8_t* sb = stage0 + buf * G.page_bytes;
        const int sw = stage_swizzle<CB>(rowB);
        uint32_t cw[kGroups][2];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          if constexpr (CB == 4) {
            const int c = 2 * g + (j >> 1);
            const uint2 t = *reinterpret_cast<const uint2*>(
                sb + G.content_off + rowB * G.content_row + ((c ^ sw) << 4) + 8 * (j & 1));
            cw[g][0] = page_ok ? t.x : 0u;
            cw[g][1] = page_ok ? t.y : 0u;
          } else {
            const uint32_t t = *reinterpret_cast<const uint32_t*>(
                sb + G.content_off + rowB * G.content_row + ((g ^ sw) << 4) + 4 * j);
            cw[g][0] = page_ok ? t : 0u;
            cw[g][1] = 0;
          }
        }
        {
          const uint2 t = *reinterpret_cast<const uint2*>(sb + G.rope_off + rowB * G.rope_row + j * 8);
          cw[8][0] = page_ok ? t.x : 0u;
          cw[8][1] = page_ok ? t.y : 0u;
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
            const int hr = lane & 15;
            ldmatrix_x4(af, qs + q_off(hr, g * 64 + s * 16 + (lane >> 4) * 8));
            mma_16816(D, af, bq[2 * s], bq[2 * s + 1]);
          }
          const float centre = (g < 8 && CB == 2) ? float(kCentre2) : float(kCentre4);
          const float2 sm0 = __half22float2(*reinterpret_cast<const __half2*>(&mt0));
          const float2 sm1 = __half22float2(*reinterpret_cast<const __half2*>(&mt1));
          const float s0 = v0 ? sm0.x : 0.f, s1 = v1 ? sm1.x : 0.f;
          const float m0 = v0 ? fmaf(centre, sm0.x, sm0.y) : 0.f;
          const float m1 = v1 ? fmaf(centre, sm1.x, sm1.y) : 0.f;
          S[0] += s0 * D[0] + m0 * qs0[g];
          S[1] += s1 * D[1] + m1 * qs0[g];
          S[2] += s0 * D[2] + m0 * qs1[g];
          S[3] += s1 * D[3] + m1 * qs1[g];
          if (g < 8) {
            big |= fmaxf(fabsf(s0), fabsf(s1)) > kBigScale;
            mp0[g] = m0;
            mp1[g] = m1;
            uint8_t* rowp = planes + g * kPlane + rowB * 128;
            const int c0 = (2 * j) ^ (rowB & 7), c1 = (2 * j + 1) ^ (rowB & 7);
            *reinterpret_cast<uint4*>(rowp + c0 * 16) = make_uint4(bq[0], bq[1], bq[2], bq[3]);
            *reinterpret_cast<uint4*>(rowp + c1 * 16) = make_uint4(bq[4], bq[5], bq[6], bq[7]);
            if (rn == 0) *reinterpret_cast<float2*>(&smS[g * kPageTokens + tC0]) = make_float2(s0, s1);
          }
        }
      } else {
        // bf16 rows of the protected tokens: values in place of codes, s = 1, m = 0
        const uint16_t* rowptr = nullptr;
        const int bt = sw.bf_begin + i - n_pages;
        const int idx = bt * kPageTokens + rowB;
        if (idx < sw.n_tok) {
          const int pos = bf16_pos(sw, idx);
          rowptr = pos < kSink ? a.sink + ((long long)b * kSink + pos) * kDim
                               : a.recent + ((long long)b * kLocal + pos % kLocal) * kDim;
        }
        v0 = bt * kPageTokens + tC0 < sw.n_tok;
        v1 = bt * kPageTokens + tC0 + 1 < sw.n_tok;
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
            const int hr = lane & 15;
            ldmatrix_x4(af, qs + q_off(hr, g * 64 + s * 16 + (lane >> 4) * 8));
            mma_16816(D, af, bq[2 * s], bq[2 * s + 1]);
          }
          S[0] += D[0];
          S[1] += D[1];
          S[2] += D[2];
          S[3] += D[3];
          if (g < 8) {
            uint8_t* rowp = planes + g * kPlane + rowB * 128;
            const int c0 = (2 * j) ^ (rowB & 7), c1 = (2 * j + 1) ^ (rowB & 7);
            *reinterpret_cast<uint4*>(rowp + c0 * 16) = make_uint4(bq[0], bq[1], bq[2], bq[3]);
            *reinterpret_cast<uint4*>(rowp + c1 * 16) = make_uint4(bq[4], bq[5], bq[6], bq[7]);
            if (rn == 0)
              *reinterpret_cast<float2*>(&smS[g * kPageTokens + tC0]) =
                  make_float2(v0 ? 1.f : 0.f, v1 ? 1.f : 0.f);
          }
        }
#pragma unroll
        for (int g = 0; g < 8; ++g) mp0[g] = mp1[g] = 0.f;
      }

      // -------- 2. mask, scale to log2 units, page max; vote on rescale / abort
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
      const bool over = (m_run0 != -INFINITY && mx0 > m_run0 + kLazy) ||
                        (m_run1 != -INFINITY && mx1 > m_run1 + kLazy);
      const unsigned vote_need = __ballot_sync(0xffffffffu, over || big);
      const unsigned vote_abort = __ballot_sync(0xffffffffu, local_abort);
      if (j == 0) {
        pmax[warp * kHC + h0] = mx0;
        pmax[warp * kHC + h0 + 8] = mx1;
      }
      if (lane == 0) flags[warp] = (vote_need ? 1 : 0) | (vote_abort ? 2 : 0);
      bar_sync_compute();  // B1
      // the staged page has been read by every compute thread: fetch page i + 2
      stage_page(i + 2);
      int fl = 0;
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) fl |= flags[w];
      if (fl & 2) break;  // uniform across the compute warps
      float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) {
        t0 = fmaxf(t0, pmax[w * kHC + h0]);
        t1 = fmaxf(t1, pmax[w * kHC + h0 + 8]);
      }
      bool waited_prev = false;
      if (fl & 1) {
        // move the running max of every head to the page max (when higher) and
        // rescale what tensor memory and the registers hold
        const float mn0 = fmaxf(m_run0, t0), mn1 = fmaxf(m_run1, t1);
        const float al0 = (m_run0 == -INFINITY || mn0 == -INFINITY) ? 1.f : fast_exp2(m_run0 - mn0);
        const float al1 = (m_run1 == -INFINITY || mn1 == -INFINITY) ? 1.f : fast_exp2(m_run1 - mn1);
        m_run0 = mn0;
        m_run1 = mn1;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          accm0[g] *= al0;
          accm1[g] *= al1;
        }
        l0 *= al0;
        l1 *= al1;
        float* alpha = pmax + kComputeWarps * kHC;
        if (warp == 0 && j == 0) {
          alpha[h0] = al0;
          alpha[h0 + 8] = al1;
        }
        if (i > 0) {
          if (!local_abort &&
              !bar_wait(bar(kBarPVDone + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag, a.err))
            local_abort = true;
          waited_prev = true;
          tc_fence_after();
        }
        bar_sync_compute();  // alpha visible
        // tcgen05.ld/st are warp-collective: the whole warp rescales or none of it
        if (i > 0 && __all_sync(0xffffffffu, !local_abort)) {
          float al[16];
#pragma unroll
          for (int h = 0; h < 16; ++h) al[h] = alpha[h];
          const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            const uint32_t col = 128 * (warp >> 2) + 16 * c;
            float v[16];
            tmem_ld16(tl + col, v);
#pragma unroll
            for (int h = 0; h < 16; ++h) v[h] *= al[h];
            tmem_st16(tl + col, v);
          }
        }
      } else {
        if (m_run0 == -INFINITY) m_run0 = t0;
        if (m_run1 == -INFINITY) m_run1 = t1;
      }

      // -------- 3. p, min term, denominator, P*s operand
      const float p0 = S[0] == -INFINITY ? 0.f : fast_exp2(S[0] - m_run0);
      const float p1 = S[1] == -INFINITY ? 0.f : fast_exp2(S[1] - m_run0);
      const float p2 = S[2] == -INFINITY ? 0.f : fast_exp2(S[2] - m_run1);
      const float p3 = S[3] == -INFINITY ? 0.f : fast_exp2(S[3] - m_run1);
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        accm0[g] += p0 * mp0[g] + p1 * mp1[g];
        accm1[g] += p2 * mp0[g] + p3 * mp1[g];
      }
      l0 += p0 + p1;
      l1 += p2 + p3;
      pbuf[tC0 * kPStride + h0] = p0;
      pbuf[(tC0 + 1) * kPStride + h0] = p1;
      pbuf[tC0 * kPStride + h0 + 8] = p2;
      pbuf[(tC0 + 1) * kPStride + h0 + 8] = p3;
      // the P*s operand is single-buffered: PV of page i - 1 must be done
      if (i > 0 && !waited_prev && !local_abort &&
          !bar_wait(bar(kBarPVDone + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag, a.err))
        local_abort = true;
      bar_sync_compute();  // B2: p of the page visible
      {
        // thread (token t, group pair k) writes row t of the pair's operand:
        // [g hi h0-7, g hi h8-15, g lo .., g lo .., g+1 hi .., .., g+1 lo .., ..]
        const int t = ct & 63, k = ct >> 6;
        float pv[16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 x = *reinterpret_cast<const float4*>(pbuf + t * kPStride + 4 * q4);
          pv[4 * q4] = x.x;
          pv[4 * q4 + 1] = x.y;
          pv[4 * q4 + 2] = x.z;
          pv[4 * q4 + 3] = x.w;
        }
        uint8_t* row = sPs + k * kPlane + t * 128;
#pragma unroll
        for (int gg = 0; gg < 2; ++gg) {
          const float sv = smS[(2 * k + gg) * kPageTokens + t];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              split_hi_lo(pv[8 * hh + 2 * e] * sv, pv[8 * hh + 2 * e + 1] * sv, hi[e], lo[e]);
            const int chi = (4 * gg + hh) ^ (t & 7), clo = (4 * gg + 2 + hh) ^ (t & 7);
            *reinterpret_cast<uint4*>(row + chi * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(row + clo * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      bar_arrive(bar(kBarPReady));
      done_tiles = i + 1;
    }
    cp_async_wait<0>();

    // -------- epilogue: wait for the last PV, reduce the register terms,
    // write the partial
    const bool have = done_tiles > 0 && done_tiles == n_tiles;
    bool ok = have;
    if (have) {
      const int last = n_tiles - 1;
      ok = bar_wait(bar(kBarPVDone + (last & 1)), (last >> 1) & 1, abort_flag, a.err);
      tc_fence_after();
    }
    ok = __all_sync(0xffffffffu, ok);  // warp-uniform before the collective TMEM loads
    bar_sync_compute();  // every compute thread is past its last PV wait
    // the plane sets are free now: reduction scratch
    float* red = reinterpret_cast<float*>(planes0);          // [8 warps][16][9]
    float* fin = red + kComputeWarps * kHC * 9;              // [16][9]
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        accm0[g] += __shfl_xor_sync(0xffffffffu, accm0[g], o);
        accm1[g] += __shfl_xor_sync(0xffffffffu, accm1[g], o);
      }
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    if (j == 0) {
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        red[(warp * kHC + h0) * 9 + g] = accm0[g];
        red[(warp * kHC + h0 + 8) * 9 + g] = accm1[g];
      }
      red[(warp * kHC + h0) * 9 + 8] = l0;
      red[(warp * kHC + h0 + 8) * 9 + 8] = l1;
    }
    bar_sync_compute();
    if (ct < kHC * 9) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kComputeWarps; ++w) v += red[w * kHC * 9 + ct];
      fin[ct] = v;
    }
    bar_sync_compute();
    if (ok) {
      const int q = warp & 3, gg = q >> 1;
      const int cpos = 32 * (q & 1) + lane;  // position inside the group's plane row
      const int phys = chan_of_pos(cpos >> 3, cpos & 7, kTypeB);
      const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
      for (int kk = 0; kk < 2; ++kk) {
        const int k = 2 * (warp >> 2) + kk, g = 2 * k + gg;
        float oh[16], ol[16];
        tmem_ld16(tl + 64 * k + 32 * gg, oh);
        tmem_ld16(tl + 64 * k + 32 * gg + 16, ol);
#pragma unroll
        for (int h = 0; h < 16; ++h)
          a.part_o[(sidx * a.H + hc * kHC + h) * kLatent + g * 64 + phys] =
              oh[h] + ol[h] + fin[h * 9 + g];
      }
      if (warp == 0 && j == 0) {
        a.part_ml[(sidx * a.H + hc * kHC + h0) * 2] = m_run0;
        a.part_ml[(sidx * a.H + hc * kHC + h0) * 2 + 1] = fin[h0 * 9 + 8];
        a.part_ml[(sidx * a.H + hc * kHC + h0 + 8) * 2] = m_run1;
        a.part_ml[(sidx * a.H + hc * kHC + h0 + 8) * 2 + 1] = fin[(h0 + 8) * 9 + 8];
      }
    } else {
      // no tokens in this split, or a time-out: an empty partial
      for (int i = ct; i < kHC * kLatent; i += kComputeThreads)
        a.part_o[(sidx * a.H + hc * kHC + i / kLatent) * kLatent + i % kLatent] = 0.f;
      if (ct < kHC) {
        a.part_ml[(sidx * a.H + hc * kHC + ct) * 2] = -INFINITY;
        a.part_ml[(sidx * a.H + hc * kHC + ct) * 2 + 1] = 0.f;
      }
    }
  } else if (lane == 0) {
    // ======================= MMA warp: PV of every page, then a bounded drain
    const uint32_t id_pv = idesc(128, 64, 1, 1);  // A and B MN-major
    const uint32_t pl0 = su32(planes0), ps = su32(sPs);
    for (int i = 0; i < n_tiles; ++i) {
      if (!bar_wait(bar(kBarPReady), i & 1, abort_flag, a.err)) break;
      tc_fence_after();
      const uint32_t pl = pl0 + (i & 1) * kPlaneSet;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma(tmem + 64 * k, desc(pl + 2 * k * kPlane + 2048 * ks, kPlane, 1024),
              desc(ps + k * kPlane + 2048 * ks, 1024, 1024), id_pv, (i > 0 || ks > 0));
      }
      commit(bar(kBarPVDone + (i & 1)));
    }
    commit(bar(kBarFlush));
    const long long t0 = clock64();
    for (;;) {
      uint32_t done;
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
          " selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(bar(kBarFlush)), "r"(0)
          : "memory");
      if (done) break;
      if (clock64() - t0 > kWaitCycles) {
        set_error(a.err, MLA_LOWBIT_DEV_PIPELINE);
        break;
      }
    }
  }

  // ---- teardown: the MMA warp has drained; free tensor memory
  tc_fence_before();
  __syncthreads();
  // the partial of this CTA is written: the combine may be launched
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

}  // namespace hy

cudaError_t launch_decode_hy(int cbits, const DecodeArgs& a, cudaStream_t stream) {
  static bool configured[2] = {false, false};
  const int k = cbits == 4 ? 0 : 1;
  cudaError_t e = cudaSuccess;
  if (!configured[k]) {
    e = cbits == 4 ? cudaFuncSetAttribute(hy::decode_hy_kernel<4>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, hy::smem_bytes(4))
                   : cudaFuncSetAttribute(hy::decode_hy_kernel<2>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, hy::smem_bytes(2));
    if (e != cudaSuccess) return e;
    configured[k] = true;
  }
  dim3 grid(a.total_splits, a.H / kHC), block(hy::kThreads);
  if (cbits == 4)
    hy::decode_hy_kernel<4><<<grid, block, hy::smem_bytes(4), stream>>>(a);
  else
    hy::decode_hy_kernel<2><<<grid, block, hy::smem_bytes(2), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlalb
