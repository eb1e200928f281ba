// Split-KV low-bit MLA decode for query rows in blocks of 128 per sequence
// (128 heads, n_q query blocks of 128 / n_q heads, or n_q blocks of 128 heads)
// on the 5th-generation tensor cores, one 2-CTA cluster per (split, 128-row
// block), for packed caches and (a template variant) bf16 pages.
//
// Same arithmetic as decode.cu (QuantMLA, Abstract and Figure 8 caption:
// exact integer codes on the tensor cores, per-group fp16 scale and min, one
// softmax over all valid tokens), laid out so that both contractions run on
// tcgen05 with 128 rows as M:
//
// * The two CTAs of a cluster split the channels.  Rank r owns content groups
//   4r..4r+3 and RoPE channels 32r..32r+31: it unpacks only those parts of
//   each page (so both ranks carry the same work) and owns output channels
//   256r..256r+255.
// * The scale is carried by the B operand.  Each code c (centred) is written
//   twice, as s_hi * c and s_lo * c, where s_hi is the fp16 scale cut to 7
//   significant bits and s_lo the exact remainder (at most 4 bits): both
//   products are exact in fp16.  So QK accumulates every group of a tile into
//   one tensor-memory accumulator (q . (s c) = q . (s_hi c) + q . (s_lo c)),
//   and PV runs with one operand P for all groups of the CTA (N = 256):
//   O += P_hi (s_hi c) + P_lo (s_hi c) + P_hi (s_lo c), with P split into fp16
//   high and low parts once per row and token.  The min terms (m' = m + centre
//   s) of the logits run on the tensor core too, as two bf16 k-steps of QK
//   (factors split in three bf16 parts); those of the output are rank-one
//   sums done in fp32 on the CUDA cores.  A token whose scale
//   would take s c past the fp16 range has both planes scaled by 2^-4 and its
//   logit and P scaled back by 2^4 (exact powers of two).
// * q of the content groups lives in tensor memory and is the A operand of
//   QK; the partial logits cross the cluster with st.async into the peer's
//   shared memory, each softmax warp with the peer's warp of the same rows
//   and tokens through a barrier pair of its own (the sum is commutative, so
//   both CTAs hold bit-identical logits and make the same online-softmax
//   decisions); P is written by the
//   softmax warps straight into tensor memory as the A operand of PV; O
//   (128 x 256 fp32) stays in tensor memory for the whole split and is
//   rescaled only when a row's running max grows by more than kLazy.
//
// bf16 pages need none of the scale machinery: the planes are the cache's own
// bf16 rows (one per group, no s_lo planes, no min terms), loaded by the
// tensor-memory accelerator into a 4-deep ring; QK and PV run as bf16 MMAs
// with P in bf16 high and low parts.
//
// Packed caches run 48-token tiles in a 3-deep ring of plane sets (s_hi and
// s_lo planes, 60 KB a set), so the unpack of a tile waits for the PV of the
// tile three back; bf16 pages run 64-token tiles in a 4-deep ring.
//
// Warp roles (448 threads, one CTA per SM):
//   warps 0-3   unpack: two threads per token (one per half of the CTA's
//               groups), 64 tokens (a page) per step into 48-token tiles; the
//               next page's bytes are loaded into registers while a plane
//               buffer drains (bf16 pages: one thread issues the tensor copies,
//               the warps clear rows past the sequence);
//   warps 4-11  softmax: TMEM lane quadrant w & 3 (32 rows), token half
//               (w - 4) >> 2 (24 or 32 tokens);
//   warp 12     QK issue (one lane) and the TMEM allocation;
//   warp 13     PV issue (one lane): a tile's PV starts as soon as its P is in
//               tensor memory, whatever the next tile's QK is waiting for.
// Every wait is bounded; on a time-out the CTA records MLA_LOWBIT_DEV_PIPELINE,
// the softmax warps of a quadrant leave the tile loop together, the partial is
// written empty, and tensor memory is still freed.
#include <cuda.h>  // CUtensorMap and its encoding enums (the encoder comes through the runtime)
#include <cudaTypedefs.h>

#include <mutex>

#include "decode_common.cuh"
#include "tc_util.cuh"

namespace mlalb {
namespace wide {

using namespace tc;

constexpr int kRows = 128;
constexpr int kThreads = 448;
constexpr int kSoftWarp0 = 4;
constexpr int kSoftThreads = 256;
constexpr int kIssuerWarp = 12;      // QK
constexpr int kPvWarp = 13;          // PV
constexpr int kMaxOwn = 5;              // QK groups of a CTA
constexpr int kQBlock = kRows * 128;    // 128 rows x 64 fp16
constexpr float kLazy = 8.0f;           // log2 units
constexpr float kShiftAbove = 32768.f;  // |s c| bound beyond which a token's planes are scaled by 2^-4
constexpr int kQPitch = 41;             // uint4 per row of the q staging (5 groups x 8 + 1)
constexpr int kOPitch = 260;            // floats per row of the output staging (16-byte stores at 4 wavefronts)
constexpr int kNumBars = 33;
constexpr int kMaxSmem = 227 * 1024;

// Tile geometry and shared-memory layout (bytes, from a 1 KB aligned base) by
// layout.  Packed caches use 48-token tiles, so that three sets of s_hi and
// s_lo planes fit (a tile's planes live from its unpack to the end of its PV,
// and the ring depth divides that lifetime); bf16 pages use 64-token tiles
// (one page, one tensor-copy box per plane) in a 4-deep ring of s_hi-only sets.
template <int CB>
struct Geo {
  static constexpr bool kBF = CB == 16;
  static constexpr int kTok = kBF ? 64 : 48;              // tokens per tile
  static constexpr int kTW = kTok / 2;                    // tokens of a tile per softmax warp
  static constexpr int kNB = kBF ? 4 : 3;                 // plane-set ring depth
  static constexpr int kPlane = kTok * 128;               // kTok tokens x 64 fp16 (128-byte rows)
  static constexpr int kABuf = (kBF ? 1 : 2) * kMaxOwn * kPlane;  // s_hi planes, then s_lo planes
  static constexpr int kXChunks = kTW / 4;                // 4-token chunks of a softmax warp
  static constexpr int kOffA = 0;                         // [kNB] plane sets
  static constexpr int kOffQR = kOffA + kNB * kABuf;      // RoPE q block
  // exchange buffer: [2 token halves][kXChunks chunks of 4 tokens][128 rows]
  // float4, so that a warp's 16-byte stores (and loads) of one chunk are 512
  // contiguous bytes
  static constexpr int kOffX = kOffQR + kQBlock;
  static constexpr int kOffMeta = kOffX + 2 * kXChunks * kRows * 16;  // [kNB][4][kTok] fp32 m' (content groups)
  static constexpr int kOffShift = kOffMeta + kNB * 4 * kTok * 4;     // [kNB][kTok] token factor
  static constexpr int kOffValid = kOffShift + kNB * kTok * 4;        // [kNB][4] 16-token masks
  static constexpr int kOffMax = kOffValid + kNB * 4 * 4;             // [2][2][128] fp32
  static constexpr int kOffScan = kOffMax + 2 * 2 * kRows * 4;        // [32] int
  static constexpr int kOffPages = kOffScan + 32 * 4;                 // [128] page ids of the split
  static constexpr int kOffBar = kOffPages + 128 * 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;             // tmem base, abort flag
  static constexpr int kSmem = kOffMisc + 64;
  static constexpr int kLaunch = kSmem + 1024;  // the layout plus room to align the base to 1 KB
  static_assert(kOffQR % 1024 == 0 && kPlane % 1024 == 0 && kABuf % 1024 == 0,
                "swizzled operands need 1 KB alignment");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert(kLaunch <= kMaxSmem, "shared memory budget");
  static_assert(kRows * kOPitch * 4 <= kNB * kABuf, "output staging fits the plane buffers");
  static_assert(kRows * kQPitch * 16 <= kNB * kABuf, "q staging fits the plane buffers");
  static_assert(kTok % 16 == 0 && kTW % 8 == 0, "MMA N and P k-steps");
};

// mbarriers
constexpr int kBarAFull = 0;    // [kNB] count 2 kTok (unpack or copy threads)
constexpr int kBarAFree = 4;    // [kNB] count 1 (issuer commit after the tile's PV)
constexpr int kBarDFull = 8;    // count 1: the tile's QK is complete
constexpr int kBarDFree = 9;    // count 256: the softmax warps have read it
constexpr int kBarPFull = 10;   // count 256: P of the tile is in tensor memory
constexpr int kBarPFree = 11;   // count 1: the tile's PV is complete
constexpr int kBarFlush = 12;   // count 2: final drain of both issuers
constexpr int kBarXFull = 13;   // [8] per softmax warp w: count 1 + the partial's bytes, the peer's
                                //     warp w has written its partial logits into my buffer
constexpr int kBarXFree = 21;   // [8] per softmax warp w: count 1, the peer's warp w has read its buffer
constexpr int kBarTFull = 29;   // [kNB] bf16 pages: count 1 + 40 KB of tensor-copy transactions

// tensor memory columns
constexpr uint32_t kColO = 0;     // [4 groups][64 channels] fp32
constexpr uint32_t kColD = 256;   // [kTok tokens] fp32 QK accumulator
constexpr uint32_t kColP = 320;   // [hi kTok/2 | lo kTok/2] fp16 pairs: P of kTok tokens
constexpr uint32_t kColQ = 384;   // [4 content groups][32] fp16 pairs: q
constexpr uint32_t kTmemCols = 512;

// v[t] *= f[t] for the tokens of a softmax warp's half tile (the factor 16
// of tokens whose planes were stored scaled by 2^-4); called only for tiles
// that hold such a token.
template <int N>
__device__ __forceinline__ void scale_by_token(float (&v)[N], const float4* f4) {
#pragma unroll
  for (int t4 = 0; t4 < N / 4; ++t4) {
    const float4 f = f4[t4];
    v[4 * t4] *= f.x;
    v[4 * t4 + 1] *= f.y;
    v[4 * t4 + 2] *= f.z;
    v[4 * t4 + 3] *= f.w;
  }
}

// One 2-D box of a tensor map into shared memory (the tensor-memory
// accelerator), completing `bytes` of transactions on the barrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Bounded wait on a barrier phase that ignores the abort flag (copies in
// flight must land before the CTA leaves).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!tc::bar_test(bar, parity))
    if (clock64() - t0 > limit) break;
}

// OR of `pred` over the 256 softmax threads (named barrier 1).
__device__ __forceinline__ bool soft_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// OR of `pred` over the two softmax warps of TMEM lane quadrant qd (named
// barrier 2 + qd, 64 threads).
__device__ __forceinline__ bool pair_any(bool pred, int qd) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, %2, 64, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(2 + qd)
      : "memory");
  return r != 0;
}
// Wait results made warp-uniform before any .sync.aligned tensor-memory access.
__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// fp16 bits of the two parts of a scale: hi keeps 7 significant bits, lo is the
// exact remainder (at most 4 bits); both scaled by 2^-4 when `shift`.
__device__ __forceinline__ void scale_parts(uint32_t s16, bool shift, uint32_t& hi2, uint32_t& lo2) {
  const __half s = __ushort_as_half((unsigned short)s16);
  const __half hi = __ushort_as_half((unsigned short)(s16 & 0xFFF0u));
  __half lo = __hsub(s, hi);
  __half h2 = hi;
  if (shift) {
    h2 = __hmul(hi, __float2half(0.0625f));
    lo = __hmul(lo, __float2half(0.0625f));
  }
  hi2 = (uint32_t)__half_as_ushort(h2) * 0x00010001u;
  lo2 = (uint32_t)__half_as_ushort(lo) * 0x00010001u;
}

// Min terms on the tensor core.  The logit's min terms sum_j qs_j m'_j over
// the CTA's groups (qs_j: the row's q summed over group j; m'_j = m + centre s:
// the token's dequantised value at the centre code of group j, where the
// planes' centred codes are 0) run as two bf16 k-steps of QK, in
// the RoPE k-steps this rank leaves unused (both in the RoPE q block and in
// the RoPE s_hi plane).  Each factor is split in three bf16 parts (h + m + l,
// 24 significant bits; bf16 has the fp32 exponent range), and the two
// k-steps carry the six products hh, hm, mh, hl, lh, mm of the five groups:
//   k-step X  A: qh0-4 qh0-4 qm0-4 0    B: mh0-4 mm0-4 mh0-4 0
//   k-step Y  A: qh0-4 ql0-4 qm0-4 0    B: ml0-4 mh0-4 mm0-4 0
__device__ __forceinline__ float bf16_round(float x) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(0.f), "f"(x));
  return __uint_as_float(d << 16);
}
__device__ __forceinline__ void split3_bf16(float x, float& h, float& m, float& l) {
  h = bf16_round(x);
  const float r1 = x - h;  // exact
  m = bf16_round(r1);
  l = bf16_round(r1 - m);  // r1 - m exact
}
// two floats that are bf16 values -> one bf16x2 word (lo in the low half)
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  return (__float_as_uint(hi) & 0xFFFF0000u) | (__float_as_uint(lo) >> 16);
}
// The 16-byte chunks of k-step X (c = 0, 1) and Y (c = 2, 3) for a row of
// the RoPE q block (x = q parts) or a token of the plane (x = m' parts).
__device__ __forceinline__ uint4 min_chunk_a(int c, const float* h, const float* m, const float* l) {
  switch (c) {
    case 0: return make_uint4(bf16x2_bits(h[0], h[1]), bf16x2_bits(h[2], h[3]), bf16x2_bits(h[4], h[0]),
                              bf16x2_bits(h[1], h[2]));
    case 1: return make_uint4(bf16x2_bits(h[3], h[4]), bf16x2_bits(m[0], m[1]), bf16x2_bits(m[2], m[3]),
                              bf16x2_bits(m[4], 0.f));
    case 2: return make_uint4(bf16x2_bits(h[0], h[1]), bf16x2_bits(h[2], h[3]), bf16x2_bits(h[4], l[0]),
                              bf16x2_bits(l[1], l[2]));
    default: return make_uint4(bf16x2_bits(l[3], l[4]), bf16x2_bits(m[0], m[1]), bf16x2_bits(m[2], m[3]),
                               bf16x2_bits(m[4], 0.f));
  }
}
__device__ __forceinline__ uint4 min_chunk_b(int c, const float* h, const float* m, const float* l) {
  switch (c) {
    case 0: return make_uint4(bf16x2_bits(h[0], h[1]), bf16x2_bits(h[2], h[3]), bf16x2_bits(h[4], m[0]),
                              bf16x2_bits(m[1], m[2]));
    case 1: return make_uint4(bf16x2_bits(m[3], m[4]), bf16x2_bits(h[0], h[1]), bf16x2_bits(h[2], h[3]),
                              bf16x2_bits(h[4], 0.f));
    case 2: return make_uint4(bf16x2_bits(l[0], l[1]), bf16x2_bits(l[2], l[3]), bf16x2_bits(l[4], h[0]),
                              bf16x2_bits(h[1], h[2]));
    default: return make_uint4(bf16x2_bits(h[3], h[4]), bf16x2_bits(m[0], m[1]), bf16x2_bits(m[2], m[3]),
                               bf16x2_bits(m[4], 0.f));
  }
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Channel position (0..63, chunk-major) -> channel of the group, for a plane or
// q row in the unpack's order.
__device__ __forceinline__ int chan_at(int p, bool tb) { return tc::chan_of_pos(p >> 3, p & 7, tb); }

template <int CB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_wide_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmap) {
  using GG = Geo<CB>;
  constexpr bool kBF = GG::kBF;      // bf16 pages: planes are the values themselves
  constexpr int NB = GG::kNB;        // plane-set ring depth
  constexpr int ABUF = GG::kABuf;    // bytes per plane set (bf16: no s_lo planes)
  constexpr int TOK = GG::kTok;      // tokens per tile
  constexpr int TW = GG::kTW;        // tokens of a tile per softmax warp
  constexpr int PL = GG::kPlane;     // bytes per plane
  constexpr bool kTypeB = CB == 2;
  constexpr PageGeom G = page_geom(CB);
  constexpr float kCentreC = kTypeB ? float(kCentre2) : float(kCentre4);
  constexpr float kCmaxC = kTypeB ? 2.f : 8.f;  // largest |code - centre| of a content group
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (tc::su32(smem_raw) & 1023)) & 1023);
  uint8_t* sA = smem + GG::kOffA;
  uint8_t* sQR = smem + GG::kOffQR;
  float* sX = reinterpret_cast<float*>(smem + GG::kOffX);
  float* sMeta = reinterpret_cast<float*>(smem + GG::kOffMeta);
  float* sShift = reinterpret_cast<float*>(smem + GG::kOffShift);
  uint32_t* sMask = reinterpret_cast<uint32_t*>(smem + GG::kOffValid);
  float* sMax = reinterpret_cast<float*>(smem + GG::kOffMax);
  int* scan = reinterpret_cast<int*>(smem + GG::kOffScan);
  int* s_pages = reinterpret_cast<int*>(smem + GG::kOffPages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GG::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + GG::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + GG::kOffMisc + 4);
  auto bar = [&](int i) { return tc::su32(&bars[i]); };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = (int)cluster_rank();
  const uint32_t peer = r ^ 1;
  const int sidx = blockIdx.x >> 1;  // the split's global index
  const int hb = kRows * blockIdx.y;  // first query row of this cluster

  int b, split, nsplit;
  find_split<kThreads>(a, !kBF, scan, b, split, nsplit, sidx);
  if (b < 0) return;  // both CTAs of the cluster name the same split
  const int L = [&] {
    const int v = a.seq_lens[b];
    return (v < 0 || v > a.max_pages * kPageTokens) ? 0 : v;
  }();
  if (split == 0 && r == 0 && blockIdx.y == 0 && tid == 0) {
    a.seq_split[2 * b] = sidx;
    a.seq_split[2 * b + 1] = nsplit;
  }
  const SplitWork sw = split_work(L, split, a.chunk_pages, !kBF);
  const int n_pk = sw.n_pages;
  // tiles of the split's run of paged tokens (packed: 48-token tiles over its
  // n_pk pages, the last one ragged), then tiles of its protected tokens
  const int n_pt = (n_pk * kPageTokens + TOK - 1) / TOK;
  const int bf_first = 64 * sw.bf_begin;
  const int bf_end = min(sw.n_tok, 64 * (sw.bf_begin + sw.n_bf));
  const int n_tiles = n_pt + max(0, (bf_end - bf_first + TOK - 1) / TOK);

  // ---- set-up: barriers, TMEM, page ids, RoPE q block
  if (tid == 0) {
    for (int i = 0; i < NB; ++i) {
      tc::bar_init(bar(kBarAFull + i), 2 * TOK);
      tc::bar_init(bar(kBarAFree + i), 1);
      tc::bar_init(bar(kBarTFull + i), 1);
    }
    tc::bar_init(bar(kBarDFull), 1);
    tc::bar_init(bar(kBarDFree), kSoftThreads);
    tc::bar_init(bar(kBarPFull), kSoftThreads);
    tc::bar_init(bar(kBarPFree), 1);
    for (int w = 0; w < kSoftThreads / 32; ++w) {
      tc::bar_init(bar(kBarXFull + w), 1);
      tc::bar_init(bar(kBarXFree + w), 1);
    }
    tc::bar_init(bar(kBarFlush), 2);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kIssuerWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     tc::su32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // page ids of the split's packed pages (the planner caps a split at 128)
  for (int k = tid; k < min(n_pk, 128); k += kThreads)
    s_pages[k] = a.block_table[(long long)b * a.max_pages + sw.page_begin + k];
  // this CTA's q rows (its four content groups and the RoPE group, 640 bytes a
  // row) staged in the plane buffers with one round of coalesced loads;
  // the softmax warps convert them below, before any plane is written.  Row
  // pitch 656 bytes: a warp's 16-byte loads of 32 rows take four wavefronts.
  // (all loads are issued before the first store: the compiler cannot move a
  // global load past a shared store it might alias)
  uint4* sQ = reinterpret_cast<uint4*>(sA);
  {
    constexpr int kQU = (kRows * 40 + kThreads - 1) / kThreads;
    uint4 qv[kQU];
#pragma unroll
    for (int k = 0; k < kQU; ++k) {
      const int u = tid + k * kThreads;
      if (u < kRows * 40) {
        const int h = u / 40, rem = u - 40 * h, j = rem >> 3;
        const int g = j < 4 ? 4 * r + j : 8;
        qv[k] = reinterpret_cast<const uint4*>(a.q + ((long long)b * a.H + hb + h) * kDim + 64 * g)[rem & 7];
      }
    }
#pragma unroll
    for (int k = 0; k < kQU; ++k) {
      const int u = tid + k * kThreads;
      if (u < kRows * 40) sQ[(u / 40) * kQPitch + u % 40] = qv[k];
    }
  }
  // RoPE q block: row h, chunk c holds the channels in the unpack's order (each
  // rank multiplies only its half of them)
  if constexpr (kBF) {
    // bf16 pages: the row's RoPE channels in their own order, unconverted
    for (int u = tid; u < kRows * 8; u += kThreads) {
      const int h = u >> 3, c = u & 7;
      *reinterpret_cast<uint4*>(sQR + tc::sw_chunk(h, c)) =
          reinterpret_cast<const uint4*>(a.q + ((long long)b * a.H + hb + h) * kDim + 512)[c];
    }
  } else {
    for (int u = tid; u < kRows * 4; u += kThreads) {
      const int h = u >> 2, cc = u & 3;
      const uint4* src = reinterpret_cast<const uint4*>(a.q + ((long long)b * a.H + hb + h) * kDim + 512 + 16 * cc);
      const uint4 v0 = src[0], v1 = src[1];
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int c = 2 * cc + c2;
        uint32_t o[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int p0 = tc::chan_of_pos(c, 2 * e2, false) - 16 * cc;
          const int p1 = tc::chan_of_pos(c, 2 * e2 + 1, false) - 16 * cc;
          const float f0 = (p0 & 1) ? bf16hi_to_f32(w[p0 >> 1]) : bf16lo_to_f32(w[p0 >> 1]);
          const float f1 = (p1 & 1) ? bf16hi_to_f32(w[p1 >> 1]) : bf16lo_to_f32(w[p1 >> 1]);
          o[e2] = pack_half2(f0, f1);
        }
        *reinterpret_cast<uint4*>(sQR + tc::sw_chunk(h, c)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  tc::fence_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // softmax warps: q of content groups 2th, 2th+1 into tensor memory (row h =
  // lane of quadrant qd), and the group sums of the row's q for the min terms
  float qs[kMaxOwn] = {0.f, 0.f, 0.f, 0.f, 0.f};
  if (warp >= kSoftWarp0 && warp < kSoftWarp0 + 8) {
    const int qd = warp & 3, th = (warp - kSoftWarp0) >> 2, h = 32 * qd + lane;
#pragma unroll
    for (int j = 0; j < kMaxOwn; ++j) {
      const bool tb = j < 4 && kTypeB;
      uint32_t w[32];
      const uint4* src = sQ + h * kQPitch + 8 * j;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 v = src[k];
        w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
      }
      uint32_t o[32];
      float acc = 0.f;
#pragma unroll
      for (int p2 = 0; p2 < 32; ++p2) {
        if constexpr (kBF) {  // bf16 pages: q stays bf16, channels in order
          o[p2] = w[p2];
          continue;
        }
        const int c0 = tb ? chan_at(2 * p2, true) : chan_at(2 * p2, false);
        const int c1 = tb ? chan_at(2 * p2 + 1, true) : chan_at(2 * p2 + 1, false);
        const float f0 = (c0 & 1) ? bf16hi_to_f32(w[c0 >> 1]) : bf16lo_to_f32(w[c0 >> 1]);
        const float f1 = (c1 & 1) ? bf16hi_to_f32(w[c1 >> 1]) : bf16lo_to_f32(w[c1 >> 1]);
        o[p2] = pack_half2(f0, f1);
        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&o[p2]));
        acc += hf.x + hf.y;
      }
      qs[j] = j < 4 || r == 1 ? acc : 0.f;  // the RoPE group's min term is rank 1's
      if (j < 4 && (j >> 1) == th) {
        const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
        tmem_st8_nowait(tl + kColQ + 32 * j, o);
        tmem_st8_nowait(tl + kColQ + 32 * j + 8, o + 8);
        tmem_st8_nowait(tl + kColQ + 32 * j + 16, o + 16);
        tmem_st8_nowait(tl + kColQ + 32 * j + 24, o + 24);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
    }
    if (th == 0 && !kBF) {
      float qh[kMaxOwn], qm[kMaxOwn], ql[kMaxOwn];
#pragma unroll
      for (int j = 0; j < kMaxOwn; ++j) split3_bf16(qs[j], qh[j], qm[j], ql[j]);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(sQR + tc::sw_chunk(h, 4 * (1 - r) + c)) = min_chunk_a(c, qh, qm, ql);
      tc::fence_async_smem();
    }
  }
  // the q staging's reads (generic proxy) come before any tensor copy
  // (async proxy) into the same plane buffers
  tc::fence_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive or store

  if (warp < 4 && kBF) {
    // ---------------- copy (bf16 pages): thread 0 loads each tile's five
    // planes (the CTA's four content groups and the RoPE group, 64 tokens x 64
    // channels each) with the tensor-memory accelerator, NB - 1 tiles ahead,
    // 128-byte swizzled as the MMAs read them; a bad page is read past the
    // map's end (zeros).  Once a tile has landed, the token rows past the
    // sequence are cleared (thread half gh: planes 2gh, 2gh+1 and half the RoPE
    // plane of row t), and the tile is handed over.
    const int t = tid >> 1, gh = tid & 1;
    int issued = 0;
    auto issue = [&](int i) {  // thread 0
      const int buf = i % NB;
      const long long page = s_pages[i];
      const bool ok_p = page >= 0 && page < a.num_pages;
      if (!ok_p) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
      const int y = ok_p ? (int)(page * kPageTokens) : -kPageTokens;
      const uint32_t dst = tc::su32(sA + buf * ABUF), tb = bar(kBarTFull + buf);
      expect_tx(tb, 5 * PL);
#pragma unroll
      for (int j = 0; j < 4; ++j) tma_load_2d(dst + j * PL, &tmap, 64 * (4 * r + j), y, tb);
      tma_load_2d(dst + 4 * PL, &tmap, kLatent, y, tb);
    };
    if (tid == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
      for (; issued < min(NB - 1, n_pk); ++issued) issue(issued);
    }
    int consumed = 0;
    for (int i = 0; i < n_tiles; ++i) {
      const int buf = i % NB;
      if (!wait(bar(kBarTFull + buf), (i / NB) & 1, abort_flag, a.err, a.wait_cycles)) break;
      consumed = i + 1;
      const long long page = s_pages[i];
      const bool okt = page >= 0 && page < a.num_pages && (sw.page_begin + i) * kPageTokens + t < L;
      if (!okt) {
        uint8_t* A = sA + buf * ABUF;
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(A + (2 * gh + jj) * PL + tc::sw_chunk(t, c)) = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(A + 4 * PL + tc::sw_chunk(t, 4 * gh + c)) = make_uint4(0, 0, 0, 0);
      }
      tc::fence_async_smem();
      uint32_t mk = __ballot_sync(0xffffffffu, okt) & 0x55555555u;
      mk = (mk | (mk >> 1)) & 0x33333333u;
      mk = (mk | (mk >> 2)) & 0x0F0F0F0Fu;
      mk = (mk | (mk >> 4)) & 0x00FF00FFu;
      mk = (mk | (mk >> 8)) & 0x0000FFFFu;
      if (lane == 0) sMask[buf * 4 + warp] = mk;
      // self-test of the bounded waits: the first tile's hand-off is withheld
      if (!(a.fault == 1 && i == 0)) tc::bar_arrive(bar(kBarAFull + buf));
      // refill: tile i + NB - 1 goes to the buffer of tile i - 1, free once
      // that tile's PV is complete
      const int nxt = i + NB - 1;
      if (nxt < n_pk) {
        const bool free_ok =
            i < 1 || wait(bar(kBarAFree + (i - 1) % NB), ((i - 1) / NB) & 1, abort_flag, a.err, a.wait_cycles);
        if (!__all_sync(0xffffffffu, free_ok)) break;
        if (tid == 0) {
          issue(nxt);
          issued = nxt + 1;
        }
      }
    }
    // copies issued but not waited for (an early exit) land before the CTA leaves
    if (tid == 0)
      for (int i = consumed; i < issued; ++i) drain_wait(bar(kBarTFull + i % NB), (i / NB) & 1, a.wait_cycles);
  } else if (warp < 4) {
    // ---------------- unpack, over the split's tokens in batches of 64 (batch
    // b of the run of pages is page b): token u of every batch, two threads
    // per token; thread half gh takes content groups 2gh, 2gh+1 and RoPE words
    // 4r+2gh, 4r+2gh+1 (16 channels).  Position s = 64b + u is row s mod 48 of
    // tile s / 48, so a tile spans two batches; a warp's 16 tokens always lie
    // in one tile (48 and 64 are multiples of 16) and it waits for that tile's
    // buffer alone.
    const int u = tid >> 1, gh = tid & 1;
    uint4 nc[4];
    uint2 nr = make_uint2(0, 0);
    uint32_t nm[3];
    bool n_ok = false, n_okt = false;
    auto fetch = [&](int pi) {  // row u of page pi of the split's run
      const int row = u;
      const bool in_run = pi < n_pk;
      const long long page = in_run ? s_pages[pi] : 0;
      const int pos = (sw.page_begin + pi) * kPageTokens + row;
      const bool page_ok = page >= 0 && page < a.num_pages;
      if (in_run && !page_ok && gh == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
      n_ok = in_run && page_ok;
      n_okt = n_ok && pos >= kSink && pos < L - kLocal;
      const uint8_t* pb = a.pool + (n_ok ? page : 0) * (long long)G.page_bytes;
      const uint8_t* crow = pb + G.content_off + row * G.content_row;
      const uint8_t* mrow = pb + G.meta_off + row * G.meta_row;
#pragma unroll
      for (int k = 0; k < 4; ++k) nc[k] = make_uint4(0, 0, 0, 0);
      nr = make_uint2(0, 0);
      nm[0] = nm[1] = nm[2] = 0u;
      if (n_ok) {
        // groups 4r + 2gh, 4r + 2gh + 1 are contiguous in the row
        const uint4* cs = reinterpret_cast<const uint4*>(crow + (CB == 4 ? 32 : 16) * (4 * r + 2 * gh));
        // thread gh = 1 walks the chunks from the middle (bank spread, below):
        // its words come in that order, so that the loop indexes them directly
        if constexpr (CB == 4) {
#pragma unroll
          for (int k = 0; k < 4; ++k) nc[k] = cs[k ^ gh];
        } else {
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint4 v = cs[k];
            nc[k] = gh ? make_uint4(v.z, v.w, v.x, v.y) : v;
          }
        }
        nr = *reinterpret_cast<const uint2*>(pb + G.rope_off + row * G.rope_row + 16 * r + 8 * gh);
      }
      if (n_okt) {
        nm[0] = *reinterpret_cast<const uint32_t*>(mrow + 4 * (4 * r + 2 * gh));
        nm[1] = *reinterpret_cast<const uint32_t*>(mrow + 4 * (4 * r + 2 * gh + 1));
        nm[2] = *reinterpret_cast<const uint32_t*>(mrow + 32);
      }
    };
    if (u < TOK * n_pt) fetch(0);
    for (int bb = 0;; ++bb) {
      const int s = 64 * bb + u;  // position in the split's tiles
      if (s >= TOK * n_tiles) break;
      const int i = s / TOK, t = s - i * TOK;  // tile, row
      const int buf = i % NB;
      uint4 cc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) cc[k] = nc[k];
      const uint2 rr = nr;
      const uint32_t mw0 = nm[0], mw1 = nm[1], mw2 = nm[2];
      const bool okt_cur = n_okt;
      if (s + 64 < TOK * n_pt) fetch(bb + 1);  // in flight while the buffer drains
      const bool packed = i < n_pt;
      // What needs only this tile's metadata is done before the buffer is
      // free: the token factor, the scale parts, m', the min-term chunks, the
      // RoPE codes and the validity mask.
      bool shift = false;
      uint32_t hiA = 0u, loA = 0u, hiB = 0u, loB = 0u, hiR = 0u, loR = 0u;
      float mqA = 0.f, mqB = 0.f;  // m' of the two content groups, in order
      uint32_t rc[8];              // the two RoPE words' centred codes
      uint4 mc0 = make_uint4(0, 0, 0, 0), mc1 = mc0;
      if (packed) {
        // one factor per token: 2^-4 on both planes when some group's s * |c|
        // could leave the fp16 range (decided with the token's other half)
        float smax = 0.f;
        const uint32_t mws[3] = {mw0, mw1, mw2};
#pragma unroll
        for (int jj = 0; jj < 3; ++jj) {
          const float sv = __half2float(__ushort_as_half((unsigned short)(mws[jj] & 0xFFFFu)));
          smax = fmaxf(smax, sv * (jj < 2 ? kCmaxC : 8.f));
        }
        smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 1));
        shift = smax > kShiftAbove;
        scale_parts(mw0 & 0xFFFFu, shift, hiA, loA);
        scale_parts(mw1 & 0xFFFFu, shift, hiB, loB);
        scale_parts(mw2 & 0xFFFFu, shift, hiR, loR);
        const float2 smA = __half22float2(*reinterpret_cast<const __half2*>(&mw0));
        const float2 smB = __half22float2(*reinterpret_cast<const __half2*>(&mw1));
        mqA = fmaf(kCentreC, smA.x, smA.y);
        mqB = fmaf(kCentreC, smB.x, smB.y);
        unpack_int4(rr.x, rc);
        unpack_int4(rr.y, rc + 4);
        // min-term k-steps of the token (B side): m' of the CTA's content
        // groups (two from each thread of the token) and, on rank 1, of the
        // RoPE group, times the token's plane factor; thread gh writes the
        // chunks of k-step X (gh = 0) or Y (gh = 1)
        const float2 smr = __half22float2(*reinterpret_cast<const __half2*>(&mw2));
        const float pa = __shfl_xor_sync(0xffffffffu, mqA, 1);
        const float pb = __shfl_xor_sync(0xffffffffu, mqB, 1);
        const float f = shift ? 0.0625f : 1.f;
        const float mv[kMaxOwn] = {gh ? pa : mqA, gh ? pb : mqB, gh ? mqA : pa, gh ? mqB : pb,
                                   r ? fmaf(float(kCentre4), smr.x, smr.y) : 0.f};
        float mh[kMaxOwn], mm[kMaxOwn], ml[kMaxOwn];
#pragma unroll
        for (int j = 0; j < kMaxOwn; ++j) split3_bf16(mv[j] * f, mh[j], mm[j], ml[j]);
        mc0 = min_chunk_b(2 * gh, mh, mm, ml);
        mc1 = min_chunk_b(2 * gh + 1, mh, mm, ml);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) rc[k] = 0u;
      }
      const bool okt = packed ? okt_cur : bf_first + (i - n_pt) * TOK + t < bf_end;
      // validity of the warp's 16 tokens (lanes 2k and 2k+1 hold token k);
      // bit 31: some token of the 16 has its planes scaled by 2^-4
      const bool any_shift = __any_sync(0xffffffffu, shift);
      uint32_t mk = __ballot_sync(0xffffffffu, okt) & 0x55555555u;
      mk = (mk | (mk >> 1)) & 0x33333333u;
      mk = (mk | (mk >> 2)) & 0x0F0F0F0Fu;
      mk = (mk | (mk >> 4)) & 0x00FF00FFu;
      mk = (mk | (mk >> 8)) & 0x0000FFFFu;
      // the buffer: free once the PV of tile i - NB is complete (the lanes of
      // a warp leave together)
      const bool free_ok = i < NB || wait(bar(kBarAFree + buf), ((i / NB) - 1) & 1, abort_flag, a.err, a.wait_cycles);
      if (!__all_sync(0xffffffffu, free_ok)) break;
      uint8_t* A = sA + buf * ABUF;
      float* meta = sMeta + buf * 4 * TOK;
      if (packed) {
        if (gh == 0) sShift[buf * TOK + t] = shift ? 16.f : 1.f;
        // the thread's two content groups in a rolled loop (code size): the
        // group in hand is always cc[0..] with hiA/loA/mqA, shifted down afterwards
#pragma unroll 1
        for (int jj = 0; jj < 2; ++jj) {
          const int j = 2 * gh + jj;
          uint8_t* p1 = A + j * PL;
          uint8_t* p2 = A + (kMaxOwn + j) * PL;
          // the token's two threads write the same positions of planes 8 KB
          // apart (same banks): the second one walks the chunks in another
          // order, so that their stores never meet in one bank
          if constexpr (CB == 4) {
            const uint4 c0 = cc[0], c1 = cc[1];
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {
              const int kk = k2 ^ (gh << 2);
              uint32_t p[4];
              unpack_int4(w[k2], p);
              *reinterpret_cast<uint4*>(p1 + tc::sw_chunk(t, kk)) =
                  make_uint4(hmul2u(p[0], hiA), hmul2u(p[1], hiA), hmul2u(p[2], hiA), hmul2u(p[3], hiA));
              *reinterpret_cast<uint4*>(p2 + tc::sw_chunk(t, kk)) =
                  make_uint4(hmul2u(p[0], loA), hmul2u(p[1], loA), hmul2u(p[2], loA), hmul2u(p[3], loA));
            }
          } else {
            const uint4 c0 = cc[0];
            const uint32_t w[4] = {c0.x, c0.y, c0.z, c0.w};
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              const int kk = k2 ^ (gh << 1);
              uint32_t p[8];
              unpack_int2(w[k2], p);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                *reinterpret_cast<uint4*>(p1 + tc::sw_chunk(t, 2 * kk + hh)) =
                    make_uint4(hmul2u(p[4 * hh], hiA), hmul2u(p[4 * hh + 1], hiA),
                               hmul2u(p[4 * hh + 2], hiA), hmul2u(p[4 * hh + 3], hiA));
                *reinterpret_cast<uint4*>(p2 + tc::sw_chunk(t, 2 * kk + hh)) =
                    make_uint4(hmul2u(p[4 * hh], loA), hmul2u(p[4 * hh + 1], loA),
                               hmul2u(p[4 * hh + 2], loA), hmul2u(p[4 * hh + 3], loA));
              }
            }
          }
          meta[j * TOK + t] = mqA;
          mqA = mqB;
          hiA = hiB;
          loA = loB;
          if constexpr (CB == 4) {
            cc[0] = cc[2];
            cc[1] = cc[3];
          } else {
            cc[0] = cc[1];
          }
        }
        {
          // RoPE words 4r + 2gh, 4r + 2gh + 1 -> chunks of the same index
          uint8_t* p1 = A + 4 * PL;
          uint8_t* p2 = A + (kMaxOwn + 4) * PL;
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int c = 4 * r + 2 * gh + k2;
            const uint32_t* p = rc + 4 * k2;
            *reinterpret_cast<uint4*>(p1 + tc::sw_chunk(t, c)) =
                make_uint4(hmul2u(p[0], hiR), hmul2u(p[1], hiR), hmul2u(p[2], hiR), hmul2u(p[3], hiR));
            *reinterpret_cast<uint4*>(p2 + tc::sw_chunk(t, c)) =
                make_uint4(hmul2u(p[0], loR), hmul2u(p[1], loR), hmul2u(p[2], loR), hmul2u(p[3], loR));
          }
          *reinterpret_cast<uint4*>(p1 + tc::sw_chunk(t, 4 * (1 - r) + 2 * gh)) = mc0;
          *reinterpret_cast<uint4*>(p1 + tc::sw_chunk(t, 4 * (1 - r) + 2 * gh + 1)) = mc1;
        }
      } else {
        // protected tokens: bf16 values as the s_hi plane, zero s_lo plane, min 0
        const int idx = bf_first + (i - n_pt) * TOK + t;
        const uint16_t* rp = nullptr;
        if (okt) {
          const int pos = bf16_pos(sw, idx);
          rp = pos < kSink ? a.sink + ((long long)b * kSink + pos) * kDim
                           : a.recent + ((long long)b * kLocal + pos % kLocal) * kDim;
        }
        if (gh == 0) sShift[buf * TOK + t] = 1.f;
        // 16-channel blocks: 4 per content group (2 groups), then RoPE block 2r + gh
#pragma unroll 1
        for (int blk = 0; blk < 9; ++blk) {
          const int j = blk < 8 ? 2 * gh + (blk >> 2) : 4;
          const int cc16 = blk < 8 ? (blk & 3) : 2 * r + gh;
          const int g = j < 4 ? 4 * r + j : 8;
          const bool tb = j < 4 && kTypeB;
          uint8_t* p1 = A + j * PL;
          uint8_t* p2 = A + (kMaxOwn + j) * PL;
          uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
          if (rp) {
            v0 = reinterpret_cast<const uint4*>(rp + g * 64 + 16 * cc16)[0];
            v1 = reinterpret_cast<const uint4*>(rp + g * 64 + 16 * cc16)[1];
          }
          const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const int c = 2 * cc16 + c2;
            uint32_t o[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const int q0 = tc::chan_of_pos(c, 2 * e2, tb) - 16 * cc16;
              const int q1 = tc::chan_of_pos(c, 2 * e2 + 1, tb) - 16 * cc16;
              const float f0 = (q0 & 1) ? bf16hi_to_f32(w[q0 >> 1]) : bf16lo_to_f32(w[q0 >> 1]);
              const float f1 = (q1 & 1) ? bf16hi_to_f32(w[q1 >> 1]) : bf16lo_to_f32(w[q1 >> 1]);
              o[e2] = pack_half2(f0, f1);
            }
            *reinterpret_cast<uint4*>(p1 + tc::sw_chunk(t, c)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(p2 + tc::sw_chunk(t, c)) = make_uint4(0, 0, 0, 0);
          }
        }
        meta[(2 * gh) * TOK + t] = 0.f;
        meta[(2 * gh + 1) * TOK + t] = 0.f;
        // no min terms: zero min-term k-steps
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2)
          *reinterpret_cast<uint4*>(A + 4 * PL + tc::sw_chunk(t, 4 * (1 - r) + 2 * gh + c2)) =
              make_uint4(0, 0, 0, 0);
      }
      if (lane == 0) sMask[buf * 4 + t / 16] = mk | (any_shift ? 0x80000000u : 0u);
      tc::fence_async_smem();
      // self-test of the bounded waits: the first tile's hand-off is withheld
      if (!(a.fault == 1 && i == 0)) tc::bar_arrive(bar(kBarAFull + buf));
    }
  } else if (warp == kIssuerWarp || warp == kPvWarp) {
    // ---------------- MMA issue (lane 0 of two warps): QK of each tile as soon
    // as its planes are in and the softmax warps have read the previous tile's
    // logits; PV of each tile once its P is in tensor memory.  Each issuer
    // commits its own MMAs (a commit tracks the issuing thread's operations).
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc(128, TOK, 0, 0);   // A K-major, B K-major
      // the same shape with bf16 A and B (bits 7-9, 10-12: format 1) for the
      // min-term k-steps
      const uint32_t id_min = id_qk | (1u << 7) | (1u << 10);
      const uint32_t id_pv = tc::idesc(128, 256, 0, 1);   // A (tensor memory), B MN-major
      const uint32_t id_pv_bf = id_pv | (1u << 7) | (1u << 10);
      auto tile_ready = [&](int i) {
        const bool r2 = wait(bar(kBarAFull + i % NB), (i / NB) & 1, abort_flag, a.err, a.wait_cycles);
        if (r2) tc::tc_fence_after();
        return r2;
      };
      // descriptors differ only in their start address (16-byte units in the
      // low bits, no carry for shared-memory addresses)
      const uint64_t kq0 = tc::desc(tc::su32(sA), 16, 1024);
      const uint64_t kp0 = tc::desc(tc::su32(sA), PL, 1024);
      const uint64_t qr0 = tc::desc(tc::su32(sQR), 16, 1024);
      // (the issue loops are unrolled: with the descriptors folded to
      // constants an MMA issues every ~46 cycles, against ~60 from a rolled loop)
      if (warp == kIssuerWarp) {
        for (int k = 0; k < n_tiles; ++k) {
          if (!(tile_ready(k) && (k == 0 || wait(bar(kBarDFree), (k - 1) & 1, abort_flag, a.err, a.wait_cycles))))
            break;
          tc::tc_fence_after();
          const uint64_t d = kq0 + (uint64_t)(((k % NB) * ABUF) >> 4);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint32_t qa = tmem + kColQ + 32 * j + 8 * ks;
              if constexpr (kBF) {  // bf16 q and values: one product, exact in fp32
                mma_tmem_a(tmem + kColD, qa, d + (uint64_t)((j * PL + 32 * ks) >> 4), id_min, (j | ks) != 0);
              } else {
                mma_tmem_a(tmem + kColD, qa, d + (uint64_t)((j * PL + 32 * ks) >> 4), id_qk, (j | ks) != 0);
                mma_tmem_a(tmem + kColD, qa, d + (uint64_t)(((kMaxOwn + j) * PL + 32 * ks) >> 4), id_qk, 1);
              }
            }
          }
          // this rank's half of the RoPE channels: k-steps 2r, 2r + 1
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2) {
            const int ks = 2 * r + k2;
            if constexpr (kBF) {
              tc::mma(tmem + kColD, qr0 + (uint64_t)((32 * ks) >> 4),
                      d + (uint64_t)((4 * PL + 32 * ks) >> 4), id_min, 1);
            } else {
              tc::mma(tmem + kColD, qr0 + (uint64_t)((32 * ks) >> 4),
                      d + (uint64_t)((4 * PL + 32 * ks) >> 4), id_qk, 1);
              tc::mma(tmem + kColD, qr0 + (uint64_t)((32 * ks) >> 4),
                      d + (uint64_t)(((kMaxOwn + 4) * PL + 32 * ks) >> 4), id_qk, 1);
            }
          }
          // the min terms: the other rank's RoPE k-steps, in bf16
          if constexpr (!kBF) {
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
              const int ks = 2 * (1 - r) + k2;
              tc::mma(tmem + kColD, qr0 + (uint64_t)((32 * ks) >> 4),
                      d + (uint64_t)((4 * PL + 32 * ks) >> 4), id_min, 1);
            }
          }
          tc::commit(bar(kBarDFull));
        }
      } else {
        for (int k = 0; k < n_tiles; ++k) {
          // P of tile k is in tensor memory; its planes were complete before
          // its QK (tested again here: an acquire in this thread too)
          if (!(wait(bar(kBarPFull), k & 1, abort_flag, a.err, a.wait_cycles) && tile_ready(k))) break;
          tc::tc_fence_after();
          const uint64_t d = kp0 + (uint64_t)(((k % NB) * ABUF) >> 4);
#pragma unroll
          for (int ks = 0; ks < TOK / 16; ++ks) {
            // the four content groups' planes side by side: N = 256 channels
            const uint64_t b1 = d + (uint64_t)((2048 * ks) >> 4);
            const uint64_t b2 = d + (uint64_t)((kMaxOwn * PL + 2048 * ks) >> 4);
            const uint32_t phi = tmem + kColP + 8 * ks, plo = tmem + kColP + TOK / 2 + 8 * ks;
            if constexpr (kBF) {  // P in bf16 high and low parts, bf16 values
              mma_tmem_a(tmem + kColO, phi, b1, id_pv_bf, (k > 0 || ks > 0));
              mma_tmem_a(tmem + kColO, plo, b1, id_pv_bf, 1);
            } else {
              mma_tmem_a(tmem + kColO, phi, b1, id_pv, (k > 0 || ks > 0));
              mma_tmem_a(tmem + kColO, plo, b1, id_pv, 1);
              mma_tmem_a(tmem + kColO, phi, b2, id_pv, 1);
            }
          }
          tc::commit(bar(kBarPFree));
          tc::commit(bar(kBarAFree + k % NB));
        }
      }
      // drain (bounded, regardless of the abort flag) before TMEM is freed:
      // the barrier completes once both issuers' operations are done
      tc::commit(bar(kBarFlush));
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
        if (clock64() - t0 > a.wait_cycles) {
          set_error(a.err, MLA_LOWBIT_DEV_PIPELINE);
          break;
        }
      }
    }
  } else if (warp >= kSoftWarp0) {
    // ---------------- softmax: row h (TMEM lane), tokens TW*th .. TW*th+TW-1
    const int qd = warp & 3, th = (warp - kSoftWarp0) >> 2, h = 32 * qd + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
    const uint32_t x_peer = map_peer(tc::su32(sX), peer);
    // warp w exchanges with the peer's warp w only (same rows, same tokens),
    // through a pair of barriers of its own
    const int sw_idx = warp - kSoftWarp0;
    const uint32_t xfull_peer = map_peer(bar(kBarXFull + sw_idx), peer);
    const uint32_t xfree_peer = map_peer(bar(kBarXFree + sw_idx), peer);
    // rows of query block qb see all but the last n_q - 1 - qb protected tokens
    const int n_masked = a.n_q - 1 - (hb + h) / (a.H / a.n_q);
    float m_run = -INFINITY, l = 0.f;
    float accm[4] = {0.f, 0.f, 0.f, 0.f};
    bool ok = true;
    int done_tiles = 0;
    for (int i = 0; i < n_tiles; ++i) {
      const int buf = i % NB;
      const bool packed_tile = i < n_pt;
      const float* meta = sMeta + buf * 4 * TOK + TW * th;
      const float4* f4 = reinterpret_cast<const float4*>(sShift + buf * TOK + TW * th);
      float S[TW];
      // partial logits of my groups: the accumulator (scaled back per token)
      // plus the min terms.  The unpack warps' metadata of this tile is read
      // after an acquire on its plane-ready barrier (complete by now: QK ran).
      if (ok) ok = wait(bar(kBarDFull), i & 1, abort_flag, a.err, a.wait_cycles);
      if (ok) ok = wait(bar(kBarAFull + buf), (i / NB) & 1, abort_flag, a.err, a.wait_cycles);
      uint64_t vm64 = 0;
      uint32_t mk_or = 0;
#pragma unroll
      for (int w = 0; w < TOK / 16; ++w) {
        const uint32_t mk = sMask[buf * 4 + w];
        vm64 |= (uint64_t)(mk & 0xFFFFu) << (16 * w);
        mk_or |= mk;
      }
      const bool shifted = (mk_or >> 31) != 0;  // some token's logit and P take a factor 16
      constexpr uint32_t kAll = TW == 32 ? 0xFFFFFFFFu : (1u << TW) - 1u;
      uint32_t vmask = (uint32_t)(vm64 >> (TW * th)) & kAll;
      ok = warp_all(ok);
      if (ok) {
        tc::tc_fence_after();
        if constexpr (TW == 32) {
          tmem_ld32(tl + kColD + TW * th, S);
        } else {
          tmem_ld24(tl + kColD + TW * th, S);
        }
        tc::tc_fence_before();
        tc::bar_arrive(bar(kBarDFree));
        // the accumulator holds the min terms too (scaled like the planes)
        if (shifted) scale_by_token(S, f4);
      }
      // exchange with the peer: my partial of my TW tokens goes to the
      // peer's buffer (once the peer has read the previous tile's), the peer's
      // partial of the same tokens arrives in mine
      if (ok && i >= 1) ok = bar_wait_cluster(bar(kBarXFree + sw_idx), (i - 1) & 1, abort_flag, a.err, a.wait_cycles);
      if (ok) {
#pragma unroll
        for (int k = 0; k < TW / 4; ++k)
          st_async4(x_peer + (uint32_t)(((th * (TW / 4) + k) * kRows + h) * 16), S[4 * k], S[4 * k + 1],
                    S[4 * k + 2], S[4 * k + 3], xfull_peer);
        if (lane == 0) expect_tx(bar(kBarXFull + sw_idx), 32 * TW * 4);
        ok = wait(bar(kBarXFull + sw_idx), i & 1, abort_flag, a.err, a.wait_cycles);
      }
      if (ok) {
        const float4* src = reinterpret_cast<const float4*>(sX);
#pragma unroll
        for (int k = 0; k < TW / 4; ++k) {
          const float4 v = src[(th * (TW / 4) + k) * kRows + h];
          S[4 * k] += v.x;
          S[4 * k + 1] += v.y;
          S[4 * k + 2] += v.z;
          S[4 * k + 3] += v.w;
        }
      }
      // validity, log2 scale, tile max over both halves.  In bf16 tiles the
      // row's query block also masks the last protected tokens.
      if (!packed_tile) {
        const int lim = sw.n_tok - n_masked - (bf_first + (i - n_pt) * TOK + TW * th);
        vmask &= lim <= 0 ? 0u : lim >= TW ? kAll : (1u << lim) - 1u;
      } else if (kBF && n_masked > 0) {
        // bf16 pages hold the last tokens too: the row's query block does not
        // see the sequence's last n_masked of them
        const int lim = L - n_masked - ((sw.page_begin + i) * kPageTokens + TW * th);
        vmask &= lim <= 0 ? 0u : lim >= TW ? kAll : (1u << lim) - 1u;
      }
      // (the max of the raw logits, scaled once: the scale is positive and
      // rounding is monotonic, so this is the max of the scaled logits)
      // (four independent chains: the max does not depend on the order)
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (vmask == kAll) {
#pragma unroll
        for (int t = 0; t < TW; ++t) mx4[t & 3] = fmaxf(mx4[t & 3], S[t]);
      } else {
#pragma unroll
        for (int t = 0; t < TW; ++t) {
          S[t] = ((vmask >> t) & 1u) ? S[t] : -INFINITY;
          mx4[t & 3] = fmaxf(mx4[t & 3], S[t]);
        }
      }
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      sMax[((i & 1) * 2 + th) * kRows + h] = mx * a.scale_log2;
      if (pair_any(!ok, qd)) break;  // both warps of the rows leave at the same tile
      // my reads of the peer's partial are done: one arrival per warp, issued
      // after the tile max so that it does not queue ahead of local accesses
      __syncwarp();
      if (lane == 0) arrive_peer_relaxed(xfree_peer);
      const float tmax = fmaxf(sMax[((i & 1) * 2) * kRows + h], sMax[((i & 1) * 2 + 1) * kRows + h]);
      // lazy running max: moved only when the tile max exceeds it by kLazy
      const bool need = m_run != -INFINITY && tmax > m_run + kLazy;
      const float m_new = (m_run == -INFINITY || need) ? tmax : m_run;
      // the previous tile's PV must be complete: P is reused, and O may be rescaled
      if (ok && i >= 1) ok = wait(bar(kBarPFree), (i - 1) & 1, abort_flag, a.err, a.wait_cycles);
      ok = warp_all(ok);
      if (ok && __any_sync(0xffffffffu, need)) {
        tc::tc_fence_after();
        const float alpha = need ? fast_exp2(m_run - m_new) : 1.f;
        l *= alpha;
#pragma unroll
        for (int j = 0; j < 4; ++j) accm[j] *= alpha;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const uint32_t col = kColO + 128 * th + 32 * c;
          float v[32];
          tmem_ld32(tl + col, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] *= alpha;
          tmem_st32(tl + col, v);
        }
      }
      m_run = m_new;
      // p = 2^(scale * S - m) in one rounding; masked tokens (S = -inf) give 0,
      // also while no token of the row has been valid yet (m = -inf)
      const float mneg = m_run == -INFINITY ? 0.f : -m_run;
      // (the tile's sum in four partial sums: short dependency chains)
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int t = 0; t < TW; ++t) {
        S[t] = fast_exp2(fmaf(S[t], a.scale_log2, mneg));
        ls4[t & 3] += S[t];
      }
      l += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
      // min terms of my four PV groups (unscaled P).  The loop stays rolled
      // (the per-tile code of all warp roles has to fit the instruction
      // caches): the four sums rotate one place per group, back in order
      // after the fourth.
#pragma unroll 1
      for (int j = 0; j < (kBF ? 0 : 4); ++j) {
        const float4* m4 = reinterpret_cast<const float4*>(meta + j * TOK);
        float am[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int t4 = 0; t4 < TW / 4; ++t4) {
          const float4 mv = m4[t4];
          am[0] = fmaf(S[4 * t4], mv.x, am[0]);
          am[1] = fmaf(S[4 * t4 + 1], mv.y, am[1]);
          am[2] = fmaf(S[4 * t4 + 2], mv.z, am[2]);
          am[3] = fmaf(S[4 * t4 + 3], mv.w, am[3]);
        }
        const float a0 = accm[0] + ((am[0] + am[1]) + (am[2] + am[3]));
        accm[0] = accm[1];
        accm[1] = accm[2];
        accm[2] = accm[3];
        accm[3] = a0;
      }
      // P (times each token's plane factor) as fp16 high and low parts
      if (ok) {
        tc::tc_fence_after();
        uint32_t hi[TW / 2], lo[TW / 2];
        if (shifted) scale_by_token(S, f4);
#pragma unroll
        for (int t2 = 0; t2 < TW / 2; ++t2) {
          if constexpr (kBF) {
            split_trunc_bf16(S[2 * t2], S[2 * t2 + 1], hi[t2], lo[t2]);
          } else {
            split_trunc(S[2 * t2], S[2 * t2 + 1], hi[t2], lo[t2]);
          }
        }
        if constexpr (TW == 32) {
          tmem_st16_nowait(tl + kColP + (TW / 2) * th, hi);
          tmem_st16_nowait(tl + kColP + TOK / 2 + (TW / 2) * th, lo);
        } else {
          tmem_st12_nowait(tl + kColP + (TW / 2) * th, hi);
          tmem_st12_nowait(tl + kColP + TOK / 2 + (TW / 2) * th, lo);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc::tc_fence_before();
        tc::bar_arrive(bar(kBarPFull));
      }
      done_tiles = i + 1;
    }
    // ---- epilogue: the halves' l and min terms through the exchange buffer
    // (no more traffic from the peer), then my 128 output columns (groups 2th, 2th+1)
    soft_sync();
    bool done = ok && n_tiles > 0 && done_tiles == n_tiles &&
                wait(bar(kBarPFree), (n_tiles - 1) & 1, abort_flag, a.err, a.wait_cycles);
    done = !soft_any(!done);  // one decision for all softmax warps
    sX[(th * 5) * kRows + h] = l;
#pragma unroll
    for (int j = 0; j < 4; ++j) sX[(th * 5 + 1 + j) * kRows + h] = accm[j];
    soft_sync();
    const float l_tot = sX[h] + sX[5 * kRows + h];
    float* orow = a.part_o + ((long long)sidx * a.H + hb + h) * kLatent;
    if (done) {
      tc::tc_fence_after();
      // my 128 columns of row h go to shared memory in channel order (the
      // plane buffers are free: every MMA has completed and the unpack warps
      // are done), then the CTA's 128 rows x 256 channels leave as coalesced
      // 16-byte stores.  Positions 0, 2, 4, 6 of a chunk hold four adjacent
      // channels and positions 1, 3, 5, 7 the next four.
      float* sO = reinterpret_cast<float*>(sA);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const int j = 2 * th + (c >> 1);
        const float mt = sX[(1 + j) * kRows + h] + sX[(6 + j) * kRows + h];
        float v[32];
        tmem_ld32(tl + kColO + 128 * th + 32 * c, v);
        float* dst = sO + h * kOPitch + j * 64;
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {
          const int ck = 4 * (c & 1) + k8;  // chunk of the group
          const float* u = v + 8 * k8;
          if constexpr (kBF) {  // bf16 pages: channels in order
            *reinterpret_cast<float4*>(dst + 8 * ck) = make_float4(u[0], u[1], u[2], u[3]);
            *reinterpret_cast<float4*>(dst + 8 * ck + 4) = make_float4(u[4], u[5], u[6], u[7]);
          } else {
            *reinterpret_cast<float4*>(dst + tc::chan_of_pos(ck, 0, kTypeB)) =
                make_float4(u[0] + mt, u[2] + mt, u[4] + mt, u[6] + mt);
            *reinterpret_cast<float4*>(dst + tc::chan_of_pos(ck, 1, kTypeB)) =
                make_float4(u[1] + mt, u[3] + mt, u[5] + mt, u[7] + mt);
          }
        }
      }
      soft_sync();
      const int st = tid - kSoftWarp0 * 32;  // 0..255
      float* obase = a.part_o + ((long long)sidx * a.H + hb) * kLatent + 256 * r;
#pragma unroll 4
      for (int k = 0; k < kRows * 64 / kSoftThreads; ++k) {
        const int idx = st + kSoftThreads * k;  // row idx / 64, float4 column idx % 64
        const int row = idx >> 6, c4 = idx & 63;
        *reinterpret_cast<float4*>(obase + (long long)row * kLatent + 4 * c4) =
            *reinterpret_cast<const float4*>(sO + row * kOPitch + 4 * c4);
      }
      if (r == 0 && th == 0) {
        a.part_ml[((long long)sidx * a.H + hb + h) * 2] = m_run;
        a.part_ml[((long long)sidx * a.H + hb + h) * 2 + 1] = l_tot;
      }
    } else {
      for (int c = 0; c < 128; ++c) orow[(4 * r + 2 * th) * 64 + c] = 0.f;
      if (r == 0 && th == 0) {
        a.part_ml[((long long)sidx * a.H + hb + h) * 2] = -INFINITY;
        a.part_ml[((long long)sidx * a.H + hb + h) * 2 + 1] = 0.f;
      }
    }
  }

  // ---- teardown
  tc::tc_fence_before();
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == kIssuerWarp) {
    tc::tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
  cluster_sync();  // no remote access to this CTA's shared memory after it exits
}

}  // namespace wide

// The driver's tensor-map encoder, looked up once through the runtime.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

cudaError_t launch_decode_wide(int cbits, const DecodeArgs& a, cudaStream_t stream) {
  const int smem = cbits == 16 ? wide::Geo<16>::kLaunch : wide::Geo<4>::kLaunch;
  void (*kern)(DecodeArgs, CUtensorMap) = cbits == 4   ? wide::decode_wide_kernel<4>
                                          : cbits == 2 ? wide::decode_wide_kernel<2>
                                                       : wide::decode_wide_kernel<16>;
  const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  // bf16 pages: a 2-D map of the pool, [pages * 64 token rows][576 channels],
  // boxes of 64 x 64 (one plane) with the 128-byte swizzle of the MMA operands
  CUtensorMap tmap;
  memset(&tmap, 0, sizeof(tmap));
  if (cbits == 16) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)a.num_pages * kPageTokens};
    const cuuint64_t strides[1] = {(cuuint64_t)kDim * 2};
    const cuuint32_t box[2] = {64, kPageTokens};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint8_t*>(a.pool), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  dim3 grid(2 * a.total_splits, a.H / wide::kRows), block(wide::kThreads);
  kern<<<grid, block, smem, stream>>>(a, tmap);
  return cudaGetLastError();
}

}  // namespace mlalb
