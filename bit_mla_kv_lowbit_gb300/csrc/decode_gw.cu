// Split-KV low-bit MLA decode with two warps per content group ("group per
// warp"), for packed caches.  One CTA per (16-head chunk, split), 16 warps.
//
// Same arithmetic as decode.cu (QuantMLA, Abstract and Figure 8 caption:
// exact integer codes on the tensor cores, per-group fp32 scale and min outside
// them, P*scale split into fp16 high and low parts for PV, one softmax over all
// valid tokens).  The work is laid out to keep shared-memory traffic low,
// which bounds the one-team-per-page layout of decode.cu:
//
// * Warp (g, hf) owns content group g for the 32 tokens of page half hf.  Its
//   q fragments (16 heads x 64 channels of group g) live in registers for the
//   whole split, so q is never re-read; each warp also takes one 16-channel
//   k-step of the RoPE group for two of its four token blocks.
// * The warp unpacks its group's codes straight into mma.sync B fragments,
//   runs QK, and writes its partial logits s_g * (q_g . c_g) + m'_g * sum(q_g)
//   to a small buffer; after a barrier warp h sums the 8 group partials of head
//   h for all 64 tokens and does the head's online-softmax bookkeeping.
// * For PV the same registers are reused: movmatrix transposes each 8x8 block
//   of codes from the QK layout (token rows) to the PV layout (channel rows),
//   so the code tile never goes through shared memory.  O[16 heads][64
//   channels of group g] over the warp's half stays in registers and is
//   rescaled every page (p <= 1); the two halves are added once per split.
#include "decode_common.cuh"

namespace mlalb {
namespace gw {

constexpr int kWarps = 16;             // 8 groups x 2 token halves
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;      // page staging ring (prefetch distance 2)
constexpr int kZStride = 72;    // floats per (warp, head) row of the partial-logit buffer
constexpr int kPStride = 72;    // floats per head row of the p buffer

// shared memory (bytes)
constexpr int kOffQ = 0;                                         // [16][576] fp16, swizzled rows
constexpr int kOffZ = kOffQ + kHC * kDim * 2;                    // [8 groups][16][kZStride] fp32
constexpr int kOffP = kOffZ + 8 * kHC * kZStride * 4;            // [16][kPStride] fp32
constexpr int kOffAlpha = kOffP + kHC * kPStride * 4;            // [16] fp32
constexpr int kOffScan = kOffAlpha + kHC * 4;                    // [64] int
constexpr int kOffPages = kOffScan + 64 * 4;                     // [64] page ids of the split
constexpr int kOffStage = kOffPages + 64 * 4;                    // [kStages][page bytes]
__host__ __device__ constexpr int smem_bytes(int cbits) {
  return kOffStage + kStages * page_geom(cbits).page_bytes;
}
static_assert(kOffStage % 16 == 0, "cp.async alignment");
static_assert(smem_bytes(4) <= 227 * 1024, "shared memory budget");
static_assert(8 * 32 * 32 <= 8 * kHC * kZStride, "epilogue exchange fits the logit buffer");

// q element e (0..575) of head h: 16-byte chunks swizzled against the row
__device__ __forceinline__ int q_off(int h, int e) {
  return h * kDim + ((((e >> 3) ^ (h & 7))) << 3) + (e & 7);
}
// staging: 16-byte chunk c of content row r is stored at chunk c ^ swz(r), so
// the 8 rows a warp reads for one group start in different banks
template <int CB>
__device__ __forceinline__ int stage_swz(int r) {
  return CB == 4 ? ((r & 7) << 1) : (r & 7);
}

__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src)
               : "memory");
}

template <int CB>
__global__ void __launch_bounds__(kThreads, 1) decode_gw_kernel(DecodeArgs a) {
  constexpr bool kTypeB = CB == 2;
  constexpr PageGeom G = page_geom(CB);
  extern __shared__ __align__(128) uint8_t smem[];
  __half* qs = reinterpret_cast<__half*>(smem + kOffQ);
  float* zbuf = reinterpret_cast<float*>(smem + kOffZ);
  float* pbuf = reinterpret_cast<float*>(smem + kOffP);
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  int* scan = reinterpret_cast<int*>(smem + kOffScan);
  int* s_pages = reinterpret_cast<int*>(smem + kOffPages);
  uint8_t* stage0 = smem + kOffStage;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j = lane & 3, rn = lane >> 2;
  const int h0 = rn;  // C/A fragment rows: heads h0 and h0 + 8
  const int hc = blockIdx.x;
  const int sidx = blockIdx.y;  // the split's global index

  int b, split, nsplit;
  find_split<kThreads>(a, true, scan, b, split, nsplit, sidx);
  if (b < 0) return;
  const int L = [&] {
    const int v = a.seq_lens[b];
    return (v < 0 || v > a.max_pages * kPageTokens) ? 0 : v;
  }();
  if (split == 0 && hc == 0 && tid == 0) {
    a.seq_split[2 * b] = sidx;
    a.seq_split[2 * b + 1] = nsplit;
  }

  // ---- work of this split: packed pages, then 64-token tiles of the
  // protected bf16 tokens; tile i < n_pages is a page
  const SplitWork sw = split_work(L, split, a.chunk_pages, true);
  const int n_pages = sw.n_pages, page_begin = sw.page_begin;
  int n_tiles = n_pages + sw.n_bf;
  if (n_tiles > 64) {  // the planner caps splits at 64 pages
    if (tid == 0) set_error(a.err, MLA_LOWBIT_DEV_PLAN);
    n_tiles = 0;
  }
  const int valid_lo = kSink, valid_hi = L - kLocal;  // packed-served tokens [lo, hi)

  auto stage_page = [&](int tile_i) {
    if (tile_i < n_pages) {
      const long long page = s_pages[tile_i];
      if (page >= 0 && page < a.num_pages) {
        const uint8_t* src = a.pool + page * G.page_bytes;
        uint8_t* dst0 = stage0 + (tile_i % kStages) * G.page_bytes;
        constexpr int kChunks = G.page_bytes / 16;
        constexpr int kRowChunks = G.content_row / 16;
        constexpr int kContentChunks = kPageTokens * kRowChunks;
        for (int k = tid; k < kChunks; k += kThreads) {
          int dst = k * 16;
          if (k < kContentChunks) {
            const int r = k / kRowChunks, c = k % kRowChunks;
            dst = G.content_off + r * G.content_row + ((c ^ stage_swz<CB>(r)) << 4);
          }
          cp_async16(dst0 + dst, src + k * 16);
        }
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  // ---- set-up: q (fp16, permuted contraction order) and its group sums
  float* qsum_s = pbuf;  // [9][16] scratch until the first page
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
      const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int p = c * 8 + e;
        const float f = (e & 1) ? bf16hi_to_f32(w4[e >> 1]) : bf16lo_to_f32(w4[e >> 1]);
        const __half hv = __float2half_rn(f);
        acc += __half2float(hv);
        qs[q_off(h, g * 64 + logical_of_phys(p, tb))] = hv;
      }
    }
    qsum_s[g * kHC + h] = acc;
  }
  if (tid < n_pages && tid < 64)
    s_pages[tid] = a.block_table[(long long)b * a.max_pages + page_begin + tid];
  __syncthreads();
  stage_page(0);
  stage_page(1);

  // warp (g, hf): content group g for the 32 tokens of half hf, plus RoPE
  // k-step rk for two of its four token blocks (rsb picks which two)
  const int g = warp & 7, hf = warp >> 3, rk = warp & 3, rsb = (warp >> 2) & 1;
  uint32_t af[4][4], afr[4];
#pragma unroll
  for (int s = 0; s < 4; ++s)
    ldmatrix_x4(af[s], qs + q_off(lane & 15, g * 64 + s * 16 + (lane >> 4) * 8));
  ldmatrix_x4(afr, qs + q_off(lane & 15, 512 + rk * 16 + (lane >> 4) * 8));
  const float qw0 = qsum_s[g * kHC + h0], qw1 = qsum_s[g * kHC + h0 + 8];
  const float qr0 = qsum_s[8 * kHC + h0], qr1 = qsum_s[8 * kHC + h0 + 8];
  const float centre = kTypeB ? float(kCentre2) : float(kCentre4);

  float O[8][4];
#pragma unroll
  for (int k = 0; k < 8; ++k) O[k][0] = O[k][1] = O[k][2] = O[k][3] = 0.f;
  float accm0 = 0.f, accm1 = 0.f;
  // softmax state of head hs = warp (tokens 2*lane, 2*lane + 1 of each page)
  const int hs = warp;
  float m_run = -INFINITY, l_run = 0.f;

  for (int i = 0; i < n_tiles; ++i) {
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();  // B0: page i staged; buffers of page i - 1 free
    stage_page(i + 2);

    // -------- A. unpack, QK, partial logits, codes transposed for PV
    uint32_t bq[4][8];
    float sv[4][2], mv[4][2];  // s and m' of this thread's C-fragment tokens, group g
    const int tok0 = (page_begin + i) * kPageTokens;
    bool page_ok = true;
    const bool bf_tile = i >= n_pages;
    const int bt = sw.bf_begin + i - n_pages;  // bf16 tile index when bf_tile
    if (!bf_tile) {
      const long long page = s_pages[i];
      page_ok = page >= 0 && page < a.num_pages;
      if (!page_ok && tid == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
      const uint8_t* sb = stage0 + (i % kStages) * G.page_bytes;
#pragma unroll
      for (int nl = 0; nl < 4; ++nl) {
        const int nb = 4 * hf + nl;
        const int r = 8 * nb + rn;  // B-fragment token
        const int t0 = 8 * nb + 2 * j;
        if constexpr (CB == 4) {
          const int c = 2 * g + (j >> 1);
          const uint2 x = *reinterpret_cast<const uint2*>(
              sb + G.content_off + r * G.content_row + ((c ^ stage_swz<CB>(r)) << 4) + 8 * (j & 1));
          unpack_int4(page_ok ? x.x : 0u, bq[nl]);
          unpack_int4(page_ok ? x.y : 0u, bq[nl] + 4);
        } else {
          const uint32_t x = *reinterpret_cast<const uint32_t*>(
              sb + G.content_off + r * G.content_row + ((g ^ stage_swz<CB>(r)) << 4) + 4 * j);
          unpack_int2(page_ok ? x : 0u, bq[nl]);
        }
        const uint32_t mt0 =
            *reinterpret_cast<const uint32_t*>(sb + G.meta_off + t0 * G.meta_row + g * 4);
        const uint32_t mt1 =
            *reinterpret_cast<const uint32_t*>(sb + G.meta_off + (t0 + 1) * G.meta_row + g * 4);
        const bool v0 = page_ok && tok0 + t0 >= valid_lo && tok0 + t0 < valid_hi;
        const bool v1 = page_ok && tok0 + t0 + 1 >= valid_lo && tok0 + t0 + 1 < valid_hi;
        const float2 sm0 = __half22float2(*reinterpret_cast<const __half2*>(&mt0));
        const float2 sm1 = __half22float2(*reinterpret_cast<const __half2*>(&mt1));
        sv[nl][0] = v0 ? sm0.x : 0.f;
        sv[nl][1] = v1 ? sm1.x : 0.f;
        mv[nl][0] = v0 ? fmaf(centre, sm0.x, sm0.y) : 0.f;
        mv[nl][1] = v1 ? fmaf(centre, sm1.x, sm1.y) : 0.f;
        float D[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 4; ++s) mma_16816(D, af[s], bq[nl][2 * s], bq[nl][2 * s + 1]);
        float z0 = sv[nl][0] * D[0] + mv[nl][0] * qw0;
        float z1 = sv[nl][1] * D[1] + mv[nl][1] * qw0;
        float z2 = sv[nl][0] * D[2] + mv[nl][0] * qw1;
        float z3 = sv[nl][1] * D[3] + mv[nl][1] * qw1;
        if ((nl >> 1) == rsb) {
          // RoPE k-step rk of token r: word rk >> 1 of this thread's 16 channels
          const uint2 x = *reinterpret_cast<const uint2*>(sb + G.rope_off + r * G.rope_row + j * 8);
          uint32_t rp[4];
          unpack_int4(page_ok ? ((rk >> 1) ? x.y : x.x) : 0u, rp);
          const uint32_t rb0 = (rk & 1) ? rp[2] : rp[0], rb1 = (rk & 1) ? rp[3] : rp[1];
          float Dr[4] = {0.f, 0.f, 0.f, 0.f};
          mma_16816(Dr, afr, rb0, rb1);
          const uint32_t rt0 =
              *reinterpret_cast<const uint32_t*>(sb + G.meta_off + t0 * G.meta_row + 8 * 4);
          const uint32_t rt1 =
              *reinterpret_cast<const uint32_t*>(sb + G.meta_off + (t0 + 1) * G.meta_row + 8 * 4);
          const float2 r0 = __half22float2(*reinterpret_cast<const __half2*>(&rt0));
          const float2 r1 = __half22float2(*reinterpret_cast<const __half2*>(&rt1));
          const float rs0 = v0 ? r0.x : 0.f, rs1 = v1 ? r1.x : 0.f;
          z0 += rs0 * Dr[0];
          z1 += rs1 * Dr[1];
          z2 += rs0 * Dr[2];
          z3 += rs1 * Dr[3];
          if (rk == 0) {
            const float rm0 = v0 ? fmaf(float(kCentre4), r0.x, r0.y) : 0.f;
            const float rm1 = v1 ? fmaf(float(kCentre4), r1.x, r1.y) : 0.f;
            z0 += rm0 * qr0;
            z1 += rm1 * qr0;
            z2 += rm0 * qr1;
            z3 += rm1 * qr1;
          }
        }
        *reinterpret_cast<float2*>(zbuf + (g * kHC + h0) * kZStride + t0) = make_float2(z0, z1);
        *reinterpret_cast<float2*>(zbuf + (g * kHC + h0 + 8) * kZStride + t0) = make_float2(z2, z3);
#pragma unroll
        for (int k = 0; k < 8; ++k) bq[nl][k] = transpose8x8(bq[nl][k]);
      }
    } else {
      // bf16 rows of the protected tokens: values in place of codes, s = 1, m = 0
#pragma unroll
      for (int nl = 0; nl < 4; ++nl) {
        const int nb = 4 * hf + nl;
        const int r = 8 * nb + rn;
        const int t0 = 8 * nb + 2 * j;
        const int idx = bt * kPageTokens + r;
        const uint16_t* rowp = nullptr;
        if (idx < sw.n_tok) {
          const int pos = bf16_pos(sw, idx);
          rowp = pos < kSink ? a.sink + ((long long)b * kSink + pos) * kDim
                             : a.recent + ((long long)b * kLocal + pos % kLocal) * kDim;
        }
        const bool v0 = bt * kPageTokens + t0 < sw.n_tok, v1 = bt * kPageTokens + t0 + 1 < sw.n_tok;
        uint32_t vv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (rowp) {
          const uint4* src = reinterpret_cast<const uint4*>(rowp + g * 64 + j * 16);
          const uint4 x0 = src[0], x1 = src[1];
          vv[0] = x0.x; vv[1] = x0.y; vv[2] = x0.z; vv[3] = x0.w;
          vv[4] = x1.x; vv[5] = x1.y; vv[6] = x1.z; vv[7] = x1.w;
        }
        pairs_from_bf16<kTypeB>(vv, bq[nl]);
        sv[nl][0] = v0 ? 1.f : 0.f;
        sv[nl][1] = v1 ? 1.f : 0.f;
        mv[nl][0] = mv[nl][1] = 0.f;
        float D[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 4; ++s) mma_16816(D, af[s], bq[nl][2 * s], bq[nl][2 * s + 1]);
        if ((nl >> 1) == rsb) {
          uint32_t rv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          if (rowp) {
            const uint4* src = reinterpret_cast<const uint4*>(rowp + 512 + j * 16);
            const uint4 x0 = src[0], x1 = src[1];
            rv[0] = x0.x; rv[1] = x0.y; rv[2] = x0.z; rv[3] = x0.w;
            rv[4] = x1.x; rv[5] = x1.y; rv[6] = x1.z; rv[7] = x1.w;
          }
          uint32_t rq[8];
          pairs_from_bf16<false>(rv, rq);
          const uint32_t rb0 = rk == 0 ? rq[0] : rk == 1 ? rq[2] : rk == 2 ? rq[4] : rq[6];
          const uint32_t rb1 = rk == 0 ? rq[1] : rk == 1 ? rq[3] : rk == 2 ? rq[5] : rq[7];
          mma_16816(D, afr, rb0, rb1);
        }
        *reinterpret_cast<float2*>(zbuf + (g * kHC + h0) * kZStride + t0) = make_float2(D[0], D[1]);
        *reinterpret_cast<float2*>(zbuf + (g * kHC + h0 + 8) * kZStride + t0) = make_float2(D[2], D[3]);
#pragma unroll
        for (int k = 0; k < 8; ++k) bq[nl][k] = transpose8x8(bq[nl][k]);
      }
    }
    __syncthreads();  // B1: partial logits of all groups written

    // -------- B. logits of (head hs, tokens 2*lane, 2*lane + 1), online softmax, p
    {
      float z[2] = {0.f, 0.f};
#pragma unroll
      for (int gg = 0; gg < 8; ++gg) {
        const float2 x = *reinterpret_cast<const float2*>(zbuf + (gg * kHC + hs) * kZStride + 2 * lane);
        z[0] += x.x;
        z[1] += x.y;
      }
      float tmax = -INFINITY;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 2 * lane + e;
        const bool valid = bf_tile ? (bt * kPageTokens + t < sw.n_tok)
                                      : (page_ok && tok0 + t >= valid_lo && tok0 + t < valid_hi);
        z[e] = valid ? z[e] * a.scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, z[e]);
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_new = fmaxf(m_run, tmax);
      const float alpha = (m_run == -INFINITY || m_new == -INFINITY) ? 1.f : fast_exp2(m_run - m_new);
      const float p0 = z[0] == -INFINITY ? 0.f : fast_exp2(z[0] - m_new);
      const float p1 = z[1] == -INFINITY ? 0.f : fast_exp2(z[1] - m_new);
      float lsum = p0 + p1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
      l_run = l_run * alpha + lsum;
      m_run = m_new;
      *reinterpret_cast<float2*>(pbuf + hs * kPStride + 2 * lane) = make_float2(p0, p1);
      if (lane == 0) alpha_s[hs] = alpha;
    }
    __syncthreads();  // B2: p and the rescale factors of the page visible

    // -------- C. PV of group g over the tokens of half hf (and its min term)
    {
      const float al0 = alpha_s[h0], al1 = alpha_s[h0 + 8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        O[k][0] *= al0;
        O[k][1] *= al0;
        O[k][2] *= al1;
        O[k][3] *= al1;
      }
      accm0 *= al0;
      accm1 *= al1;
#pragma unroll
      for (int kl = 0; kl < 2; ++kl) {
        const int t0 = 32 * hf + 16 * kl + 2 * j;
        const float2 pa = *reinterpret_cast<const float2*>(pbuf + h0 * kPStride + t0);
        const float2 pb = *reinterpret_cast<const float2*>(pbuf + (h0 + 8) * kPStride + t0);
        const float2 pc = *reinterpret_cast<const float2*>(pbuf + h0 * kPStride + t0 + 8);
        const float2 pd = *reinterpret_cast<const float2*>(pbuf + (h0 + 8) * kPStride + t0 + 8);
        const float sA0 = sv[2 * kl][0], sA1 = sv[2 * kl][1];
        const float sB0 = sv[2 * kl + 1][0], sB1 = sv[2 * kl + 1][1];
        uint32_t ahi[4], alo[4];
        split_hi_lo(pa.x * sA0, pa.y * sA1, ahi[0], alo[0]);
        split_hi_lo(pb.x * sA0, pb.y * sA1, ahi[1], alo[1]);
        split_hi_lo(pc.x * sB0, pc.y * sB1, ahi[2], alo[2]);
        split_hi_lo(pd.x * sB0, pd.y * sB1, ahi[3], alo[3]);
        const float mA0 = mv[2 * kl][0], mA1 = mv[2 * kl][1];
        const float mB0 = mv[2 * kl + 1][0], mB1 = mv[2 * kl + 1][1];
        accm0 += pa.x * mA0 + pa.y * mA1 + pc.x * mB0 + pc.y * mB1;
        accm1 += pb.x * mA0 + pb.y * mA1 + pd.x * mB0 + pd.y * mB1;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          mma_16816(O[k], ahi, bq[2 * kl][k], bq[2 * kl + 1][k]);
          mma_16816(O[k], alo, bq[2 * kl][k], bq[2 * kl + 1][k]);
        }
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  // ---- epilogue: min term into every channel of the group; the two halves of
  // each group are added (half 1 hands its sums over through shared memory),
  // channels un-permuted, partial stored
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    accm0 += __shfl_xor_sync(0xffffffffu, accm0, o);
    accm1 += __shfl_xor_sync(0xffffffffu, accm1, o);
  }
  float* xch = zbuf + (g * 32 + lane) * 32;  // [8 groups][32 lanes][32]
  __syncthreads();  // every thread is past the last read of zbuf
  if (hf == 1) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      *reinterpret_cast<float4*>(xch + 4 * k) =
          make_float4(O[k][0] + accm0, O[k][1] + accm0, O[k][2] + accm1, O[k][3] + accm1);
  }
  __syncthreads();
  if (hf == 0) {
    const int hg0 = hc * kHC + h0, hg1 = hg0 + 8;
    float* o0 = a.part_o + ((long long)sidx * a.H + hg0) * kLatent + g * 64;
    float* o1 = a.part_o + ((long long)sidx * a.H + hg1) * kLatent + g * 64;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 y = *reinterpret_cast<const float4*>(xch + 4 * k);
      const int ph0 = phys_of_logical(8 * k + 2 * j, kTypeB);
      const int ph1 = phys_of_logical(8 * k + 2 * j + 1, kTypeB);
      o0[ph0] = O[k][0] + accm0 + y.x;
      o0[ph1] = O[k][1] + accm0 + y.y;
      o1[ph0] = O[k][2] + accm1 + y.z;
      o1[ph1] = O[k][3] + accm1 + y.w;
    }
  }
  if (lane == 0) {
    a.part_ml[((long long)sidx * a.H + hc * kHC + hs) * 2] = m_run;
    a.part_ml[((long long)sidx * a.H + hc * kHC + hs) * 2 + 1] = l_run;
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace gw

cudaError_t launch_decode_gw(int cbits, const DecodeArgs& a, cudaStream_t stream) {
  static bool configured[2] = {false, false};
  const int k = cbits == 4 ? 0 : 1;
  if (!configured[k]) {
    const cudaError_t e =
        cbits == 4 ? cudaFuncSetAttribute(gw::decode_gw_kernel<4>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, gw::smem_bytes(4))
                   : cudaFuncSetAttribute(gw::decode_gw_kernel<2>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, gw::smem_bytes(2));
    if (e != cudaSuccess) return e;
    configured[k] = true;
  }
  if (a.total_splits > 65535) return cudaErrorInvalidConfiguration;  // grid.y limit
  dim3 grid(a.H / kHC, a.total_splits), block(gw::kThreads);
  if (cbits == 4)
    gw::decode_gw_kernel<4><<<grid, block, gw::smem_bytes(4), stream>>>(a);
  else
    gw::decode_gw_kernel<2><<<grid, block, gw::smem_bytes(2), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlalb
