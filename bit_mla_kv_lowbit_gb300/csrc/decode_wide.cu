// Split-KV low-bit MLA decode for 128 query rows per sequence (128 heads, or
// n_q query blocks of 128 / n_q heads) on the 5th-generation tensor cores, one
// 2-CTA cluster per split, for packed caches.
//
// Same arithmetic as decode.cu (QuantMLA, Abstract and Figure 8 caption:
// exact integer codes on the tensor cores, fp32 per-group scale and min folded
// outside them, P*scale split into fp16 high and low parts for PV, one
// softmax over all valid tokens).  With 128 rows the heads fill the M = 128
// dimension of a tcgen05 MMA, so every contraction runs there:
//
// * The two CTAs of a cluster split the channels.  Rank r owns content groups
//   4r..4r+3 (and rank 1 the RoPE group): it holds q for those channels in
//   shared memory, unpacks only those groups of each page, and computes the
//   partial logits sum_g s_g (q_g . c_g) + m'_g sum(q_g) over them (QK: M=128
//   rows, N=64 tokens, K=16 per MMA; one TMEM accumulator per group, folded
//   by the softmax warps).  The partials are exchanged through distributed
//   shared memory, so both CTAs hold the same logits and run the same online
//   softmax.
// * Rank r then accumulates O for its 256 output channels: per group, A =
//   P*s_g (fp16 high and low) written by the softmax warps straight into
//   tensor memory, B = the group's code plane read as an MN-major operand.
//   The A operand never passes through shared memory, which is what bounds
//   small-N MMAs whose A comes from there.
// * O (128 x 256 fp32) lives in tensor memory for the whole split and is
//   rescaled only when a row's running max grows by more than kLazy.
//
// Warp roles (672 threads, one CTA per SM):
//   warps 0-3   unpack: packed bytes -> fp16 code planes and metadata; the
//               next tile's bytes are loaded into registers while a plane
//               buffer is still in use;
//   warps 4-19  softmax: TMEM lane quadrant w & 3 (32 rows), token quarter
//               (w - 4) >> 2 (16 tokens); fold, exchange, softmax, P*s
//               operands;
//   warp 20     MMA issue (one lane) and the TMEM allocation.
// Every wait is bounded; on a time-out the CTA records MLA_LOWBIT_DEV_PIPELINE,
// the softmax warps leave the tile loop together (barrier reduction), the
// partial is written empty, and tensor memory is still freed.
#include "decode_common.cuh"
#include "tc_util.cuh"

namespace mlalb {
namespace wide {

constexpr int kRows = 128;
constexpr int kThreads = 672;
constexpr int kSoftThreads = 512;
constexpr int kTW = 16;                 // tokens of a tile per softmax warp
constexpr int kIssuerWarp = 20;
constexpr int kNB = 2;                  // code-plane ring depth (tiles)
constexpr int kMaxOwn = 5;              // QK groups of a CTA
constexpr int kPlane = 64 * 128;        // 64 tokens x 64 fp16 (128-byte rows)
constexpr int kQBlock = kRows * 128;    // 128 rows x 64 fp16
constexpr float kLazy = 8.0f;           // log2 units

// shared memory (bytes, from a 1 KB aligned base)
constexpr int kOffQ = 0;                                     // [5] q blocks
constexpr int kOffA = kOffQ + kMaxOwn * kQBlock;             // [kNB][5] planes
constexpr int kXStride = 20;                                 // floats per exchange row (padded)
constexpr int kOffX = kOffA + kNB * kMaxOwn * kPlane;        // [4 quarters][128 rows][kXStride] fp32
constexpr int kOffMeta = kOffX + 4 * kRows * kXStride * 4;   // [kNB][5][64] fp32 (s, m')
constexpr int kOffValid = kOffMeta + kNB * kMaxOwn * 64 * 8; // [kNB][2] token masks
constexpr int kOffSmax = kOffValid + kNB * 2 * 4;            // [kNB][4] largest PV scale per unpack warp
constexpr int kOffMax = kOffSmax + kNB * 4 * 4;              // [2][4][128] fp32
constexpr int kOffScan = kOffMax + 2 * 4 * kRows * 4;        // [32] int
constexpr int kOffPages = kOffScan + 32 * 4;                 // [64] page ids of the split
constexpr int kOffBar = kOffPages + 64 * 4;
constexpr int kNumBars = 20;
constexpr int kOffMisc = kOffBar + kNumBars * 8;             // tmem base, abort flag
constexpr int kSmem = kOffMisc + 64;
static_assert(kOffA % 1024 == 0 && kPlane % 1024 == 0, "swizzled operands need 1 KB alignment");
static_assert(kOffBar % 8 == 0, "mbarrier alignment");
static_assert(kSmem + 1024 <= 227 * 1024, "shared memory budget (with 1 KB alignment slack)");

// mbarriers
constexpr int kBarAFull = 0;    // [kNB] count 128 (unpack threads)
constexpr int kBarAFree = 3;    // [kNB] count 1 (issuer commit after the tile's PV)
constexpr int kBarDFull = 6;    // [2] count 1 (QK commit)
constexpr int kBarDFree = 8;    // [2] count 512 (softmax threads)
constexpr int kBarPsFull = 10;  // [2] count 512
constexpr int kBarPsFree = 12;  // [2] count 1 (PV commit)
constexpr int kBarPV = 14;      // count 1: a tile's PV is complete
constexpr int kBarXFull = 15;   // count 1 + 32 KB of transactions: the peer's partial logits are in my buffer
constexpr int kBarXFree = 16;   // count 512: the peer has read its buffer
constexpr int kBarFlush = 17;   // count 1: final drain of the issuer

// tensor memory columns
constexpr uint32_t kColO = 0;     // [4 groups][64 channels]
constexpr uint32_t kColD = 256;   // [2 slots][64 tokens] QK accumulators
constexpr uint32_t kColPs = 384;  // [2 slots][hi 32 | lo 32] P*s operands (fp16 pairs)
constexpr uint32_t kTmemCols = 512;

__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id,
                                           int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void tmem_st8_nowait(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// 32 consecutive columns of this thread's lane, one wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  tc::tmem_st16(taddr, v);
  tc::tmem_st16(taddr + 16, v + 16);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t peer) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(peer));
  return r;
}
// 16 bytes into the peer's shared memory, counted as transaction bytes on the
// peer's mbarrier (no fence: the barrier's phase completes once the bytes land).
__device__ __forceinline__ void st_async4(uint32_t addr, float a0, float a1, float a2, float a3,
                                          uint32_t bar_cluster_addr) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1,%2,%3,%4}, [%5];" ::"r"(addr),
      "f"(a0), "f"(a1), "f"(a2), "f"(a3), "r"(bar_cluster_addr)
      : "memory");
}
__device__ __forceinline__ void expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Arrival on the peer's barrier that orders nothing: it only reports that this
// thread's reads of its buffer have returned.
__device__ __forceinline__ void arrive_peer_relaxed(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr)
               : "memory");
}
// Bounded wait for arrivals from the peer that carry no data.
__device__ __forceinline__ bool bar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort,
                                                 int32_t* err) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.relaxed.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(200000u)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (clock64() - t0 > tc::kWaitCycles) {
      *abort = 1;
      set_error(err, MLA_LOWBIT_DEV_PIPELINE);
      return false;
    }
  }
}
// Bounded wait on a local mbarrier phase; the thread sleeps in the barrier
// (up to kSuspendNs per try) instead of spinning, so waiting warps leave the
// issue slots to the working ones.
constexpr uint32_t kSuspendNs = 200000;
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* err) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendNs)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (clock64() - t0 > tc::kWaitCycles) {
      *abort = 1;
      set_error(err, MLA_LOWBIT_DEV_PIPELINE);
      return false;
    }
  }
}

// OR of `pred` over the 512 softmax threads (named barrier 1).
__device__ __forceinline__ bool soft_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 1, 512, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
// OR of `pred` over the four softmax warps of TMEM lane quadrant qd (named
// barrier 2 + qd, 128 threads).
__device__ __forceinline__ bool quad_any(bool pred, int qd) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(2 + qd)
      : "memory");
  return r != 0;
}
// Wait results made warp-uniform before any .sync.aligned tensor-memory access.
__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// x = hi + lo with hi = x cut to 11 significant bits (exact in fp16 over its
// normal range) and lo = the exact float32 remainder rounded to fp16: x to
// about 2^-21 relative, in fewer instructions than rounding hi.
__device__ __forceinline__ void split_trunc(float a, float b, uint32_t& hi, uint32_t& lo) {
  const float ha = __uint_as_float(__float_as_uint(a) & 0xFFFFE000u);
  const float hb = __uint_as_float(__float_as_uint(b) & 0xFFFFE000u);
  hi = pack_half2(ha, hb);
  lo = pack_half2(a - ha, b - hb);
}

// Global group of local QK group j of rank r.
__device__ __forceinline__ int group_of(int r, int j) { return j < 4 ? 4 * r + j : 8; }

template <int CB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_wide_kernel(DecodeArgs a) {
  constexpr bool kTypeB = CB == 2;
  constexpr PageGeom G = page_geom(CB);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (tc::su32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sA = smem + kOffA;
  float* sX = reinterpret_cast<float*>(smem + kOffX);
  float2* sMeta = reinterpret_cast<float2*>(smem + kOffMeta);
  uint32_t* sMask = reinterpret_cast<uint32_t*>(smem + kOffValid);
  float* sMax = reinterpret_cast<float*>(smem + kOffMax);
  float* sSmax = reinterpret_cast<float*>(smem + kOffSmax);
  int* scan = reinterpret_cast<int*>(smem + kOffScan);
  int* s_pages = reinterpret_cast<int*>(smem + kOffPages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  auto bar = [&](int i) { return tc::su32(&bars[i]); };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = (int)cluster_rank();
  const uint32_t peer = r ^ 1;
  const int sidx = blockIdx.x >> 1;  // the split's global index

  int b, split, nsplit;
  find_split<kThreads>(a, true, scan, b, split, nsplit, sidx);
  if (b < 0) return;  // both CTAs of the cluster name the same split
  const int L = [&] {
    const int v = a.seq_lens[b];
    return (v < 0 || v > a.max_pages * kPageTokens) ? 0 : v;
  }();
  if (split == 0 && r == 0 && tid == 0) {
    a.seq_split[2 * b] = sidx;
    a.seq_split[2 * b + 1] = nsplit;
  }
  const SplitWork sw = split_work(L, split, a.chunk_pages, true);
  const int n_pk = sw.n_pages;
  const int bf_first = 64 * sw.bf_begin;
  const int bf_end = min(sw.n_tok, 64 * (sw.bf_begin + sw.n_bf));
  const int n_tiles = n_pk + max(0, (bf_end - bf_first + 63) / 64);
  const int n_own = 4 + r;

  // ---- set-up: barriers, TMEM, q blocks
  if (tid == 0) {
    for (int i = 0; i < kNB; ++i) {
      tc::bar_init(bar(kBarAFull + i), 128);
      tc::bar_init(bar(kBarAFree + i), 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::bar_init(bar(kBarDFull + s), 1);
      tc::bar_init(bar(kBarDFree + s), kSoftThreads);
      tc::bar_init(bar(kBarPsFull + s), kSoftThreads);
      tc::bar_init(bar(kBarPsFree + s), 1);
    }
    tc::bar_init(bar(kBarPV), 1);
    tc::bar_init(bar(kBarXFull), 1);
    tc::bar_init(bar(kBarXFree), kSoftThreads);
    tc::bar_init(bar(kBarFlush), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kIssuerWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     tc::su32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // q block j: row h, chunk c holds the group's channels in the unpack's order
  for (int u = tid; u < n_own * kRows * 4; u += kThreads) {
    const int j = u / (kRows * 4), h = (u >> 2) % kRows, cc = u & 3;
    const int g = group_of(r, j);
    const bool tb = g < 8 && kTypeB;
    const uint4* src = reinterpret_cast<const uint4*>(
        a.q + ((long long)b * a.H + h) * kDim + g * 64 + 16 * cc);
    const uint4 v0 = src[0], v1 = src[1];
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      const int c = 2 * cc + c2;
      uint32_t o[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const int p0 = tc::chan_of_pos(c, 2 * e2, tb) - 16 * cc;
        const int p1 = tc::chan_of_pos(c, 2 * e2 + 1, tb) - 16 * cc;
        const float f0 = (p0 & 1) ? bf16hi_to_f32(w[p0 >> 1]) : bf16lo_to_f32(w[p0 >> 1]);
        const float f1 = (p1 & 1) ? bf16hi_to_f32(w[p1 >> 1]) : bf16lo_to_f32(w[p1 >> 1]);
        o[e2] = pack_half2(f0, f1);
      }
      *reinterpret_cast<uint4*>(sQ + j * kQBlock + tc::sw_chunk(h, c)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  // page ids of the split's packed pages (the planner caps a split at 64)
  for (int k = tid; k < min(n_pk, 64); k += kThreads)
    s_pages[k] = a.block_table[(long long)b * a.max_pages + sw.page_begin + k];
  tc::fence_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive or store
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ---------------- unpack: token t, part pp (local groups 2pp, 2pp+1 and
    // RoPE channels 32pp..32pp+31 on rank 1)
    const int t = tid & 63, pp = tid >> 6;
    // registers of the next packed tile: codes of the thread's two content
    // groups, its RoPE quarter (rank 1) and the metadata words
    uint4 nc[4], nr = make_uint4(0, 0, 0, 0);
    uint32_t nm[3] = {0u, 0u, 0u};
    bool n_ok = false, n_okt = false;
    auto fetch = [&](int i) {
      const int page_idx = sw.page_begin + i;
      const long long page = s_pages[i];
      const int pos = page_idx * kPageTokens + t;
      n_ok = page >= 0 && page < a.num_pages;
      if (!n_ok && tid == 0) set_error(a.err, MLA_LOWBIT_DEV_BAD_PAGE);
      n_okt = n_ok && pos >= kSink && pos < L - kLocal;
      const uint8_t* pb = a.pool + (n_ok ? page : 0) * (long long)G.page_bytes;
      const uint8_t* crow = pb + G.content_off + t * G.content_row;
      const uint8_t* mrow = pb + G.meta_off + t * G.meta_row;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int g = 4 * r + 2 * pp + jj;
        nc[2 * jj] = nc[2 * jj + 1] = make_uint4(0, 0, 0, 0);
        nm[jj] = 0u;
        if (n_ok) {
          if constexpr (CB == 4) {
            nc[2 * jj] = *reinterpret_cast<const uint4*>(crow + 32 * g);
            nc[2 * jj + 1] = *reinterpret_cast<const uint4*>(crow + 32 * g + 16);
          } else {
            nc[2 * jj] = *reinterpret_cast<const uint4*>(crow + 16 * g);
          }
        }
        if (n_okt) nm[jj] = *reinterpret_cast<const uint32_t*>(mrow + 4 * g);
      }
      nr = make_uint4(0, 0, 0, 0);
      nm[2] = 0u;
      if (r == 1) {
        if (n_ok) nr = *reinterpret_cast<const uint4*>(pb + G.rope_off + t * G.rope_row + 16 * pp);
        if (n_okt && pp == 0) nm[2] = *reinterpret_cast<const uint32_t*>(mrow + 32);
      }
    };
    if (n_pk > 0) fetch(0);
    for (int i = 0; i < n_tiles; ++i) {
      const int buf = i % kNB;
      const uint4 cc0 = nc[0], cc1 = nc[1], cc2 = nc[2], cc3 = nc[3], rr = nr;
      const uint32_t mw0 = nm[0], mw1 = nm[1], mw2 = nm[2];
      const bool okt_cur = n_okt;
      if (i + 1 < n_pk) fetch(i + 1);  // in flight while the buffer drains
      if (i >= kNB && !wait(bar(kBarAFree + buf), ((i / kNB) - 1) & 1, abort_flag, a.err))
        break;
      uint8_t* A = sA + buf * kMaxOwn * kPlane;
      float2* meta = sMeta + buf * kMaxOwn * 64;
      // (s, m' = m + centre * s) of a metadata word, as the softmax warps use them
      auto sm_of = [](uint32_t w, float centre) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
        return make_float2(f.x, fmaf(centre, f.x, f.y));
      };
      if (i < n_pk) {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int j = 2 * pp + jj;
          uint8_t* plane = A + j * kPlane;
          const uint4 c0 = jj ? cc2 : cc0, c1 = jj ? cc3 : cc1;
          if constexpr (CB == 4) {
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {
              uint32_t p[4];
              unpack_int4(w[k2], p);
              *reinterpret_cast<uint4*>(plane + tc::sw_chunk(t, k2)) = make_uint4(p[0], p[1], p[2], p[3]);
            }
          } else {
            const uint32_t w[4] = {c0.x, c0.y, c0.z, c0.w};
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
              uint32_t p[8];
              unpack_int2(w[k2], p);
              *reinterpret_cast<uint4*>(plane + tc::sw_chunk(t, 2 * k2)) = make_uint4(p[0], p[1], p[2], p[3]);
              *reinterpret_cast<uint4*>(plane + tc::sw_chunk(t, 2 * k2 + 1)) = make_uint4(p[4], p[5], p[6], p[7]);
            }
          }
          meta[j * 64 + t] = sm_of(jj ? mw1 : mw0, kTypeB ? float(kCentre2) : float(kCentre4));
        }
        if (r == 1) {
          const uint32_t w[4] = {rr.x, rr.y, rr.z, rr.w};
          uint8_t* plane = A + 4 * kPlane;
#pragma unroll
          for (int k2 = 0; k2 < 4; ++k2) {
            uint32_t p[4];
            unpack_int4(w[k2], p);
            *reinterpret_cast<uint4*>(plane + tc::sw_chunk(t, 4 * pp + k2)) = make_uint4(p[0], p[1], p[2], p[3]);
          }
          if (pp == 0) meta[4 * 64 + t] = sm_of(mw2, float(kCentre4));
        }
        const uint32_t mk = __ballot_sync(0xffffffffu, okt_cur);
        if (pp == 0 && lane == 0) sMask[buf * 2 + (t >> 5)] = mk;
        // largest scale of the PV groups in this tile (bounds P * s in fp16)
        float smx = fmaxf(meta[(2 * pp) * 64 + t].x, meta[(2 * pp + 1) * 64 + t].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) smx = fmaxf(smx, __shfl_xor_sync(0xffffffffu, smx, o));
        if (lane == 0) sSmax[buf * 4 + warp] = smx;
      } else {
        // protected tokens: bf16 values in place of codes, scale 1, min 0
        const int idx = bf_first + (i - n_pk) * 64 + t;
        const bool okt = idx < bf_end;
        const uint16_t* rp = nullptr;
        if (okt) {
          const int pos = bf16_pos(sw, idx);
          rp = pos < kSink ? a.sink + ((long long)b * kSink + pos) * kDim
                           : a.recent + ((long long)b * kLocal + pos % kLocal) * kDim;
        }
        auto put16 = [&](uint8_t* plane, const uint16_t* src16, int cc, bool tb) {
          // channels 16cc..16cc+15 of a group -> chunks 2cc, 2cc+1
          uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
          if (src16) {
            v0 = reinterpret_cast<const uint4*>(src16)[0];
            v1 = reinterpret_cast<const uint4*>(src16)[1];
          }
          const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            const int c = 2 * cc + c2;
            uint32_t o[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const int p0 = tc::chan_of_pos(c, 2 * e2, tb) - 16 * cc;
              const int p1 = tc::chan_of_pos(c, 2 * e2 + 1, tb) - 16 * cc;
              const float f0 = (p0 & 1) ? bf16hi_to_f32(w[p0 >> 1]) : bf16lo_to_f32(w[p0 >> 1]);
              const float f1 = (p1 & 1) ? bf16hi_to_f32(w[p1 >> 1]) : bf16lo_to_f32(w[p1 >> 1]);
              o[e2] = pack_half2(f0, f1);
            }
            *reinterpret_cast<uint4*>(plane + tc::sw_chunk(t, c)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        };
#pragma unroll 1
        for (int jj = 0; jj < 2; ++jj) {
          const int j = 2 * pp + jj, g = 4 * r + j;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc)
            put16(A + j * kPlane, rp ? rp + g * 64 + 16 * cc : nullptr, cc, kTypeB);
          meta[j * 64 + t] = make_float2(okt ? 1.f : 0.f, 0.f);  // (s = 1, m = 0)
        }
        if (r == 1) {
#pragma unroll 1
          for (int cc = 2 * pp; cc < 2 * pp + 2; ++cc)
            put16(A + 4 * kPlane, rp ? rp + 512 + 16 * cc : nullptr, cc, false);
          if (pp == 0) meta[4 * 64 + t] = make_float2(okt ? 1.f : 0.f, 0.f);
        }
        const uint32_t mk = __ballot_sync(0xffffffffu, okt);
        if (pp == 0 && lane == 0) sMask[buf * 2 + (t >> 5)] = mk;
        if (lane == 0) sSmax[buf * 4 + warp] = 1.f;
      }
      tc::fence_async_smem();
      tc::bar_arrive(bar(kBarAFull + buf));
    }
  } else if (warp < kIssuerWarp) {
    // ---------------- softmax: row h (TMEM lane), tokens kTW*tq .. kTW*tq+kTW-1
    const int qd = warp & 3, tq = (warp - 4) >> 2, h = 32 * qd + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
    const uint32_t x_peer = map_peer(tc::su32(sX), peer);
    const uint32_t xfull_peer = map_peer(bar(kBarXFull), peer);
    const uint32_t xfree_peer = map_peer(bar(kBarXFree), peer);
    // group sums of this row's q (fp16 values, as the MMA sees them)
    float qs[kMaxOwn];
#pragma unroll
    for (int j = 0; j < kMaxOwn; ++j) {
      float acc = 0.f;
      if (j < n_own) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(sQ + j * kQBlock + tc::sw_chunk(h, c));
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
            acc += f.x + f.y;
          }
        }
      }
      qs[j] = acc;
    }
    // rows of query block qb see all but the last n_q - 1 - qb protected tokens
    const int n_masked = a.n_q - 1 - h / (kRows / a.n_q);
    float m_run = -INFINITY, l = 0.f;
    float accm[4] = {0.f, 0.f, 0.f, 0.f};
    bool ok = true;
    int kq = 0;
    int done_tiles = 0;
    for (int i = 0; i < n_tiles; ++i) {
      const int buf = i % kNB;
      const bool packed_tile = i < n_pk;
      const float2* meta = sMeta + buf * kMaxOwn * 64;
      float S[kTW];
#pragma unroll
      for (int t = 0; t < kTW; ++t) S[t] = 0.f;
      // fold the partial logits of my groups
#pragma unroll
      for (int j = 0; j < kMaxOwn; ++j) {
        if (j >= n_own) break;
        const int slot = kq & 1;
        if (ok) ok = wait(bar(kBarDFull + slot), (kq >> 1) & 1, abort_flag, a.err);
        ok = warp_all(ok);
        if (ok) {
          tc::tc_fence_after();
          float D[kTW];
          tc::tmem_ld16(tl + kColD + 64 * slot + kTW * tq, D);
          tc::tc_fence_before();
          tc::bar_arrive(bar(kBarDFree + slot));
          const float4* m4 = reinterpret_cast<const float4*>(meta + j * 64 + kTW * tq);
#pragma unroll
          for (int t2 = 0; t2 < kTW / 2; ++t2) {
            const float4 mv = m4[t2];  // (s, m') of tokens 2 t2, 2 t2 + 1
            S[2 * t2] = fmaf(mv.x, D[2 * t2], fmaf(mv.y, qs[j], S[2 * t2]));
            S[2 * t2 + 1] = fmaf(mv.z, D[2 * t2 + 1], fmaf(mv.w, qs[j], S[2 * t2 + 1]));
          }
        }
        ++kq;
      }
      // exchange with the peer: my partial of my kTW tokens goes to the
      // peer's buffer (once the peer has read the previous tile's), the peer's
      // partial of the same tokens arrives in mine
      if (ok && i >= 1) ok = bar_wait_cluster(bar(kBarXFree), (i - 1) & 1, abort_flag, a.err);
      if (ok) {
        const uint32_t dst = x_peer + (uint32_t)((tq * kRows + h) * kXStride) * 4u;
#pragma unroll
        for (int k = 0; k < kTW / 4; ++k)
          st_async4(dst + 16 * k, S[4 * k], S[4 * k + 1], S[4 * k + 2], S[4 * k + 3], xfull_peer);
        if (tid == 128) expect_tx(bar(kBarXFull), kSoftThreads * kTW * 4);
        ok = wait(bar(kBarXFull), i & 1, abort_flag, a.err);
      }
      if (ok) {
        const float4* src = reinterpret_cast<const float4*>(sX + (tq * kRows + h) * kXStride);
#pragma unroll
        for (int k = 0; k < kTW / 4; ++k) {
          const float4 v = src[k];
          S[4 * k] += v.x;
          S[4 * k + 1] += v.y;
          S[4 * k + 2] += v.z;
          S[4 * k + 3] += v.w;
        }
        arrive_peer_relaxed(xfree_peer);
      }
      // validity, log2 scale, tile max over the four quarters
      const int tok0 = bf_first + (i - n_pk) * 64 + kTW * tq;                   // bf16 tiles
      const uint32_t vmask = sMask[buf * 2 + (tq >> 1)] >> (kTW * (tq & 1));  // packed tiles
      float mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < kTW; ++t) {
        const bool v = packed_tile ? ((vmask >> t) & 1u) != 0
                                   : (tok0 + t < bf_end && tok0 + t < sw.n_tok - n_masked);
        S[t] = v ? S[t] * a.scale_log2 : -INFINITY;
        mx = fmaxf(mx, S[t]);
      }
      sMax[((i & 1) * 4 + tq) * kRows + h] = mx;
      if (quad_any(!ok, qd)) break;  // the four warps of the rows leave at the same tile
      const float tmax = fmaxf(fmaxf(sMax[((i & 1) * 4) * kRows + h], sMax[((i & 1) * 4 + 1) * kRows + h]),
                               fmaxf(sMax[((i & 1) * 4 + 2) * kRows + h], sMax[((i & 1) * 4 + 3) * kRows + h]));
      // lazy max: moved only when the tile max exceeds it by kLazy, or by less
      // when the tile's largest scale s would take P * s <= 2^kLazy * s past
      // the fp16 range
      const float smax = fmaxf(fmaxf(sSmax[buf * 4], sSmax[buf * 4 + 1]),
                               fmaxf(sSmax[buf * 4 + 2], sSmax[buf * 4 + 3]));
      const float lim = smax > 0.f ? fmaxf(0.f, fminf(kLazy, log2f(32768.f / smax))) : kLazy;
      const bool need = m_run != -INFINITY && tmax > m_run + lim;
      const float m_new = (m_run == -INFINITY || need) ? tmax : m_run;
      if (__any_sync(0xffffffffu, need)) {
        // rescale what PV has accumulated so far (previous tile's PV done)
        if (ok) ok = wait(bar(kBarPV), (i - 1) & 1, abort_flag, a.err);
        ok = warp_all(ok);
        if (ok) {
          tc::tc_fence_after();
          const float alpha = need ? fast_exp2(m_run - m_new) : 1.f;
          l *= alpha;
#pragma unroll
          for (int j = 0; j < 4; ++j) accm[j] *= alpha;
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            const uint32_t col = kColO + 64 * tq + 32 * c;
            float v[32];
            tmem_ld32(tl + col, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] *= alpha;
            tmem_st32(tl + col, v);
          }
        }
      }
      m_run = m_new;
      float lsum = 0.f;
#pragma unroll
      for (int t = 0; t < kTW; ++t) {
        S[t] = S[t] == -INFINITY ? 0.f : fast_exp2(S[t] - m_run);
        lsum += S[t];
      }
      l += lsum;
      // P * s_j operands of my four PV groups, high and low fp16 parts
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int kp = 4 * i + j, pslot = kp & 1;
        if (ok && kp >= 2) ok = wait(bar(kBarPsFree + pslot), ((kp >> 1) - 1) & 1, abort_flag, a.err);
        ok = warp_all(ok);
        if (!ok) continue;
        tc::tc_fence_after();
        const float4* m4 = reinterpret_cast<const float4*>(meta + j * 64 + kTW * tq);
        uint32_t hi[kTW / 2], lo[kTW / 2];
        float am = 0.f;
#pragma unroll
        for (int t2 = 0; t2 < kTW / 2; ++t2) {
          const float4 mv = m4[t2];  // (s, m') of tokens 2 t2, 2 t2 + 1
          const float p0 = S[2 * t2], p1 = S[2 * t2 + 1];
          am = fmaf(p0, mv.y, fmaf(p1, mv.w, am));
          split_trunc(p0 * mv.x, p1 * mv.z, hi[t2], lo[t2]);
        }
        accm[j] += am;
        tmem_st8_nowait(tl + kColPs + 64 * pslot + (kTW / 2) * tq, hi);
        tmem_st8_nowait(tl + kColPs + 64 * pslot + 32 + (kTW / 2) * tq, lo);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc::tc_fence_before();
        tc::bar_arrive(bar(kBarPsFull + pslot));
      }
      done_tiles = i + 1;
    }
    // ---- epilogue: halves' l and min terms through the exchange buffer (no
    // more traffic from the peer), then my 128 output columns
    soft_sync();
    bool done = ok && n_tiles > 0 && done_tiles == n_tiles &&
                wait(bar(kBarPV), (n_tiles - 1) & 1, abort_flag, a.err);
    done = !soft_any(!done);  // one decision for all softmax warps
    sX[(tq * 5) * kRows + h] = l;
#pragma unroll
    for (int j = 0; j < 4; ++j) sX[(tq * 5 + 1 + j) * kRows + h] = accm[j];
    soft_sync();
    float l_tot = 0.f, mt[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      l_tot += sX[(k * 5) * kRows + h];
#pragma unroll
      for (int j = 0; j < 4; ++j) mt[j] += sX[(k * 5 + 1 + j) * kRows + h];
    }
    float* orow = a.part_o + ((long long)sidx * a.H + h) * kLatent;
    if (done) {
      tc::tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const int col = 64 * tq + 32 * c;
        float v[32];
        tmem_ld32(tl + kColO + col, v);
        const int j = col >> 6, g = 4 * r + j;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int cc = (col & 63) + e;
          orow[g * 64 + tc::chan_of_pos(cc >> 3, cc & 7, kTypeB)] = v[e] + mt[j];
        }
      }
      if (r == 0 && tq == 0) {
        a.part_ml[((long long)sidx * a.H + h) * 2] = m_run;
        a.part_ml[((long long)sidx * a.H + h) * 2 + 1] = l_tot;
      }
    } else {
      for (int c = 0; c < 64; ++c) orow[(4 * r + tq) * 64 + c] = 0.f;
      if (r == 0 && tq == 0) {
        a.part_ml[((long long)sidx * a.H + h) * 2] = -INFINITY;
        a.part_ml[((long long)sidx * a.H + h) * 2 + 1] = 0.f;
      }
    }
  } else {
    // ---------------- MMA issue (lane 0): QK of the next tile's first two
    // groups, then PV of this tile, then the rest of the next tile's QK
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc(128, 64, 0, 0);  // A K-major, B K-major
      const uint32_t id_pv = tc::idesc(128, 64, 0, 1);  // A (tensor memory), B MN-major
      int kq = 0;
      auto issue_qk = [&](int i, int j) -> bool {
        const int slot = kq & 1;
        if (kq >= 2 && !wait(bar(kBarDFree + slot), ((kq >> 1) - 1) & 1, abort_flag, a.err))
          return false;
        tc::tc_fence_after();
        const uint32_t qa = tc::su32(sQ + j * kQBlock);
        const uint32_t pb = tc::su32(sA + (i % kNB) * kMaxOwn * kPlane + j * kPlane);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma(tmem + kColD + 64 * slot, tc::desc(qa + 32 * ks, 16, 1024),
                  tc::desc(pb + 32 * ks, 16, 1024), id_qk, ks > 0);
        tc::commit(bar(kBarDFull + slot));
        ++kq;
        return true;
      };
      auto tile_ready = [&](int i) {
        const bool r2 = wait(bar(kBarAFull + i % kNB), (i / kNB) & 1, abort_flag, a.err);
        if (r2) tc::tc_fence_after();
        return r2;
      };
      bool ok = n_tiles > 0 && tile_ready(0);
      for (int j = 0; ok && j < n_own; ++j) ok = issue_qk(0, j);
      auto issue_pv = [&](int i, int j) -> bool {
        const int kp = 4 * i + j, pslot = kp & 1;
        if (!wait(bar(kBarPsFull + pslot), (kp >> 1) & 1, abort_flag, a.err)) return false;
        tc::tc_fence_after();
        const uint32_t pb = tc::su32(sA + (i % kNB) * kMaxOwn * kPlane + j * kPlane);
        const uint32_t ps = tmem + kColPs + 64 * pslot;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bd = tc::desc(pb + 2048 * ks, 1024, 1024);
          mma_tmem_a(tmem + kColO + 64 * j, ps + 8 * ks, bd, id_pv, (i > 0 || ks > 0));
          mma_tmem_a(tmem + kColO + 64 * j, ps + 32 + 8 * ks, bd, id_pv, 1);
        }
        tc::commit(bar(kBarPsFree + pslot));
        return true;
      };
      // order per tile: the next tile's first two QK groups, PV of groups 0
      // and 1, the rest of the next tile's QK (its slots are freed by the
      // softmax warps' fold, which follows their P*s writes for this tile),
      // then PV of groups 2 and 3
      for (int i = 0; ok && i < n_tiles; ++i) {
        const bool nxt = i + 1 < n_tiles;
        if (nxt) {
          ok = tile_ready(i + 1);
          for (int j = 0; ok && j < 2; ++j) ok = issue_qk(i + 1, j);
        }
        for (int j = 0; ok && j < 2; ++j) ok = issue_pv(i, j);
        for (int j = 2; ok && nxt && j < n_own; ++j) ok = issue_qk(i + 1, j);
        for (int j = 2; ok && j < 4; ++j) ok = issue_pv(i, j);
        if (!ok) break;
        tc::commit(bar(kBarPV));
        tc::commit(bar(kBarAFree + i % kNB));
      }
      // drain (bounded, regardless of the abort flag) before TMEM is freed
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
        if (clock64() - t0 > tc::kWaitCycles) {
          set_error(a.err, MLA_LOWBIT_DEV_PIPELINE);
          break;
        }
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

cudaError_t launch_decode_wide(int cbits, const DecodeArgs& a, cudaStream_t stream) {
  static bool configured[2] = {false, false};
  const int k = cbits == 4 ? 0 : 1;
  const int smem = wide::kSmem + 1024;
  cudaError_t e = cudaSuccess;
  if (!configured[k]) {
    e = cbits == 4 ? cudaFuncSetAttribute(wide::decode_wide_kernel<4>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                   : cudaFuncSetAttribute(wide::decode_wide_kernel<2>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[k] = true;
  }
  dim3 grid(2 * a.total_splits), block(wide::kThreads);
  if (cbits == 4)
    wide::decode_wide_kernel<4><<<grid, block, smem, stream>>>(a);
  else
    wide::decode_wide_kernel<2><<<grid, block, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mlalb
