// Host side of the C ABI declared in include/mla_lowbit.h: argument checks,
// split planning and kernel launches.  No device memory is allocated here.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace mlalb {

namespace {

constexpr int kMaxHeads = 128;
constexpr int kMaxQueries = 16;                    // queries per sequence (multi-query decode)
constexpr int kMaxRows = kMaxHeads * kMaxQueries;  // rows of a sequence in a plan
constexpr int kCtasPerSm = 1;

int check_layout(const mla_lowbit_layout* l) {
  if (!l) return MLA_LOWBIT_ENULL;
  const bool ok_bits = (l->content_bits == 4 && l->rope_bits == 4) ||
                       (l->content_bits == 2 && l->rope_bits == 4) ||
                       (l->content_bits == 16 && l->rope_bits == 16);
  if (!ok_bits || l->group != kGroup || l->sink != kSink || l->local != kLocal ||
      l->page_tokens != kPageTokens || l->latent != kLatent || l->rope != kRope)
    return MLA_LOWBIT_EINVAL;
  if (l->rotate != 0 && (l->rotate != 1 || l->content_bits == 16)) return MLA_LOWBIT_EINVAL;
  return MLA_LOWBIT_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Self-test settings of the tcgen05 kernels' bounded waits (mla_lowbit_set_fault_injection).
std::atomic<int> g_fault_mode{0};
std::atomic<long long> g_wait_cycles{0};

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

cudaError_t ensure_smem_limit(const void* kernel, int bytes) {
  // (device, kernel, bytes) triples already applied; a handful of kernels per device
  struct Entry { int dev; const void* kernel; int bytes; };
  static Entry done[256];
  static int n_done = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].dev == dev && done[i].kernel == kernel && done[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (n_done < 256) done[n_done++] = Entry{dev, kernel, bytes};
  return cudaSuccess;
}

}  // namespace mlalb

using namespace mlalb;

extern "C" {

size_t mla_lowbit_page_bytes(const mla_lowbit_layout* layout) {
  if (check_layout(layout) != MLA_LOWBIT_OK) return 0;
  return static_cast<size_t>(page_geom(layout->content_bits).page_bytes);
}

size_t mla_lowbit_bytes_per_token(const mla_lowbit_layout* layout) {
  if (check_layout(layout) != MLA_LOWBIT_OK) return 0;
  return mla_lowbit_page_bytes(layout) / kPageTokens;
}

int mla_lowbit_write(const mla_lowbit_layout* layout, int n_tokens, const void* ckv,
                     const void* krope, const int32_t* seq_idx, const int32_t* pos,
                     const int32_t* seq_lens_after, int num_seqs, const int32_t* block_table,
                     int max_pages, void* page_pool, int64_t num_pages, void* sink_buf,
                     void* recent_buf, int32_t* err_word, void* stream) {
  int st = check_layout(layout);
  if (st != MLA_LOWBIT_OK) return st;
  if (n_tokens < 0 || num_seqs < 0 || max_pages < 0 || num_pages < 0) return MLA_LOWBIT_ESIZE;
  if (n_tokens == 0) return MLA_LOWBIT_OK;
  if (num_seqs == 0 || max_pages == 0 || num_pages == 0) return MLA_LOWBIT_ESIZE;
  if ((long long)max_pages * kPageTokens > INT32_MAX) return MLA_LOWBIT_ESIZE;
  const bool packed = layout->content_bits != 16;
  if (!ckv || !krope || !pos || !block_table || !page_pool || !err_word) return MLA_LOWBIT_ENULL;
  if (!seq_idx && n_tokens > num_seqs) return MLA_LOWBIT_EINVAL;
  if (packed && (!sink_buf || !recent_buf)) return MLA_LOWBIT_ENULL;
  if (!aligned16(ckv) || !aligned16(krope) || !aligned16(page_pool) ||
      (packed && (!aligned16(sink_buf) || !aligned16(recent_buf))))
    return MLA_LOWBIT_EALIGN;
  WriterArgs a;
  a.ckv = static_cast<const uint32_t*>(ckv);
  a.krope = static_cast<const uint32_t*>(krope);
  a.seq_idx = seq_idx;
  a.pos = pos;
  a.lens_after = seq_lens_after;
  a.block_table = block_table;
  a.pool = static_cast<uint8_t*>(page_pool);
  a.sink = static_cast<uint32_t*>(sink_buf);
  a.recent = static_cast<uint32_t*>(recent_buf);
  a.err = err_word;
  a.num_pages = num_pages;
  a.n_tokens = n_tokens;
  a.num_seqs = num_seqs;
  a.max_pages = max_pages;
  a.rotate = layout->rotate;
  cudaError_t e = launch_writer(layout->content_bits, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_LOWBIT_OK : MLA_LOWBIT_ECUDA;
}

int mla_lowbit_decode_plan(const mla_lowbit_layout* layout, int num_seqs, int heads,
                           const int32_t* seq_lens_host, int num_sms, int* total_splits,
                           int* chunk_pages, size_t* workspace_bytes) {
  int st = check_layout(layout);
  if (st != MLA_LOWBIT_OK) return st;
  if (num_seqs <= 0 || heads <= 0 || heads % 16 != 0 || heads > kMaxRows) return MLA_LOWBIT_ESIZE;
  if (!seq_lens_host || !total_splits || !chunk_pages || !workspace_bytes) return MLA_LOWBIT_ENULL;
  if (num_sms <= 0) num_sms = device_sm_count();
  if (num_sms <= 0) return MLA_LOWBIT_ECUDA;
  const bool packed = layout->content_bits != 16;
  long long work = 0;
  for (int b = 0; b < num_seqs; ++b) {
    if (seq_lens_host[b] < 0) return MLA_LOWBIT_EINVAL;
    work += units_of(seq_lens_host[b], packed);
  }
  const long long head_chunks =
      decode_ctas_per_split(layout->content_bits, heads, layout->rotate);
  const long long max_chunk = decode_max_split_pages(layout->content_bits, heads, layout->rotate);
  const long long slots = (long long)num_sms * kCtasPerSm;
  // equal chunks of work units (pages, then the protected tokens' bf16 tiles)
  // so that all splits of all head chunks fit one wave when they can
  long long chunk = (work * head_chunks + slots - 1) / slots;
  if (chunk < 1) chunk = 1;
  // a split accumulates at most max_chunk * 64 tokens in fp32 tensor-core
  // accumulators (whose adds are not round-to-nearest; 64 or 128 pages by
  // kernel); longer sequences get more splits, merged in fp32 by the combine
  // kernel.  For a wave count, the work is spread evenly over all its waves
  // (no sliver for the last one): the smallest chunk, from the even share
  // up, whose splits fit.
  auto splits_for = [&](long long c) {
    long long t = 0;
    for (int b = 0; b < num_seqs; ++b) t += splits_of(seq_lens_host[b], packed, (int)c);
    return t;
  };
  auto fit = [&](long long w, long long& c_out, long long& t_out) {
    long long c = (work * head_chunks + slots * w - 1) / (slots * w);
    c = std::min(std::max(c, 1LL), max_chunk);
    for (;;) {
      const long long t = splits_for(c);
      if (t * head_chunks <= slots * w || c >= max_chunk) {
        c_out = c;
        t_out = t;
        return t * head_chunks <= slots * w;
      }
      ++c;
    }
  };
  // the fewest waves that the capped chunk allows, then more until one fits
  // (or the chunk is down to one page)
  long long total = splits_for(max_chunk);
  long long waves = (chunk + max_chunk - 1) / max_chunk;
  waves = std::max(waves, (total * head_chunks + slots - 1) / slots);
  for (;; ++waves)
    if (fit(waves, chunk, total) || chunk == 1) break;
  // A CTA's time is about its split's units plus a fixed set-up and epilogue
  // (about kWaveUnits units), so the step takes waves * (chunk + kWaveUnits):
  // one or two more waves of smaller chunks are taken when that is at least
  // 5 % less (the per-sequence rounding can force a large chunk into the
  // fewest waves; more splits also cost the combine a little).
  constexpr long long kWaveUnits = 3;
  for (long long w = waves + 1; w <= waves + 2; ++w) {
    long long c2 = 0, t2 = 0;
    if (fit(w, c2, t2) && 20 * w * (c2 + kWaveUnits) < 19 * waves * (chunk + kWaveUnits)) {
      waves = w;
      chunk = c2;
      total = t2;
    }
  }
  if (total > INT32_MAX / 2) return MLA_LOWBIT_ESIZE;
  *total_splits = (int)total;
  *chunk_pages = (int)chunk;
  const size_t part = (size_t)total * heads * (kLatent + 2) * sizeof(float);
  *workspace_bytes = part + (size_t)num_seqs * 2 * sizeof(int32_t);
  return MLA_LOWBIT_OK;
}

// Decode, optionally appending one token per sequence first (ckv_new and
// krope_new non-null): fused into the decode launch when the split kernel
// supports it, else the writer kernel runs first on the same stream.
static int decode_impl(const mla_lowbit_layout* layout, int num_seqs, int n_q, int heads,
                       float softmax_scale, const void* q, const void* ckv_new,
                       const void* krope_new, void* page_pool, int64_t num_pages,
                       const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                       const int32_t* seq_lens_host, void* sink_buf, void* recent_buf, float* out,
                       float* lse, void* workspace, size_t workspace_bytes, int32_t* err_word,
                       void* stream) {
  int st = check_layout(layout);
  if (st != MLA_LOWBIT_OK) return st;
  if (num_seqs <= 0 || heads <= 0 || heads % 16 != 0 || heads > kMaxHeads || max_pages <= 0 ||
      num_pages <= 0 || n_q < 1 || n_q > kMaxQueries)
    return MLA_LOWBIT_ESIZE;
  if ((long long)max_pages * kPageTokens > INT32_MAX) return MLA_LOWBIT_ESIZE;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return MLA_LOWBIT_EINVAL;
  const bool packed = layout->content_bits != 16;
  const bool append = ckv_new || krope_new;
  if (!q || !page_pool || !block_table || !seq_lens || !seq_lens_host || !out || !workspace ||
      !err_word)
    return MLA_LOWBIT_ENULL;
  if (append && (!ckv_new || !krope_new)) return MLA_LOWBIT_ENULL;
  if (packed && (!sink_buf || !recent_buf)) return MLA_LOWBIT_ENULL;
  if (!aligned16(q) || !aligned16(page_pool) || !aligned16(out) || !aligned16(workspace) ||
      (packed && (!aligned16(sink_buf) || !aligned16(recent_buf))) ||
      (append && (!aligned16(ckv_new) || !aligned16(krope_new))))
    return MLA_LOWBIT_EALIGN;
  for (int b = 0; b < num_seqs; ++b) {
    if (seq_lens_host[b] < 0 || (long long)seq_lens_host[b] > (long long)max_pages * kPageTokens)
      return MLA_LOWBIT_EINVAL;
    if (append && seq_lens_host[b] < 1) return MLA_LOWBIT_EINVAL;
    if (n_q > 1 && seq_lens_host[b] < n_q) return MLA_LOWBIT_EINVAL;  // queries' tokens cached
  }
  const int rows = n_q * heads;  // rows of a sequence: n_q blocks of `heads`
  int total = 0, chunk = 0;
  size_t need = 0;
  st = mla_lowbit_decode_plan(layout, num_seqs, rows, seq_lens_host, 0, &total, &chunk, &need);
  if (st != MLA_LOWBIT_OK) return st;
  if (workspace_bytes < need) return MLA_LOWBIT_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool fused = append && n_q == 1 &&
                     decode_fuses_append(layout->content_bits, layout->rotate, heads);
  if (append && !fused) {
    WriterArgs w;
    w.ckv = static_cast<const uint32_t*>(ckv_new);
    w.krope = static_cast<const uint32_t*>(krope_new);
    w.seq_idx = nullptr;
    w.pos = nullptr;  // position seq_lens[b] - 1
    w.lens_after = seq_lens;
    w.block_table = block_table;
    w.pool = static_cast<uint8_t*>(page_pool);
    w.sink = static_cast<uint32_t*>(sink_buf);
    w.recent = static_cast<uint32_t*>(recent_buf);
    w.err = err_word;
    w.num_pages = num_pages;
    w.n_tokens = num_seqs;
    w.num_seqs = num_seqs;
    w.max_pages = max_pages;
    w.rotate = layout->rotate;
    if (launch_writer(layout->content_bits, w, s) != cudaSuccess) return MLA_LOWBIT_ECUDA;
  }
  DecodeArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.pool = static_cast<const uint8_t*>(page_pool);
  a.num_pages = num_pages;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.sink = static_cast<const uint16_t*>(sink_buf);
  a.recent = static_cast<const uint16_t*>(recent_buf);
  a.part_o = static_cast<float*>(workspace);
  a.part_ml = a.part_o + (size_t)total * rows * kLatent;
  a.seq_split = reinterpret_cast<int32_t*>(a.part_ml + (size_t)total * rows * 2);
  a.err = err_word;
  a.B = num_seqs;
  a.H = rows;
  a.n_q = n_q;
  a.rotate = layout->rotate;
  a.max_pages = max_pages;
  a.chunk_pages = chunk;
  a.total_splits = total;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.fault = g_fault_mode.load();
  if (const long long wc = g_wait_cycles.load(); wc > 0) a.wait_cycles = wc;
  if (fused) {
    a.new_ckv = static_cast<const uint32_t*>(ckv_new);
    a.new_kr = static_cast<const uint32_t*>(krope_new);
    a.pool_w = static_cast<uint8_t*>(page_pool);
    a.sink_w = static_cast<uint32_t*>(sink_buf);
    a.recent_w = static_cast<uint32_t*>(recent_buf);
  }
  cudaError_t e = launch_decode(layout->content_bits, a, out, lse, s);
  return e == cudaSuccess ? MLA_LOWBIT_OK : MLA_LOWBIT_ECUDA;
}

int mla_lowbit_decode(const mla_lowbit_layout* layout, int num_seqs, int heads,
                      float softmax_scale, const void* q, const void* page_pool,
                      int64_t num_pages, const int32_t* block_table, int max_pages,
                      const int32_t* seq_lens, const int32_t* seq_lens_host,
                      const void* sink_buf, const void* recent_buf, float* out, float* lse,
                      void* workspace, size_t workspace_bytes, int32_t* err_word,
                      void* stream) {
  return decode_impl(layout, num_seqs, 1, heads, softmax_scale, q, nullptr, nullptr,
                     const_cast<void*>(page_pool), num_pages, block_table, max_pages, seq_lens,
                     seq_lens_host, const_cast<void*>(sink_buf), const_cast<void*>(recent_buf), out,
                     lse, workspace, workspace_bytes, err_word, stream);
}

int mla_lowbit_write_decode(const mla_lowbit_layout* layout, int num_seqs, int heads,
                            float softmax_scale, const void* q, const void* ckv_new,
                            const void* krope_new, void* page_pool, int64_t num_pages,
                            const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                            const int32_t* seq_lens_host, void* sink_buf, void* recent_buf,
                            float* out, float* lse, void* workspace, size_t workspace_bytes,
                            int32_t* err_word, void* stream) {
  if (!ckv_new || !krope_new) return MLA_LOWBIT_ENULL;
  return decode_impl(layout, num_seqs, 1, heads, softmax_scale, q, ckv_new, krope_new, page_pool,
                     num_pages, block_table, max_pages, seq_lens, seq_lens_host, sink_buf,
                     recent_buf, out, lse, workspace, workspace_bytes, err_word, stream);
}

int mla_lowbit_decode_multi(const mla_lowbit_layout* layout, int num_seqs, int queries_per_seq,
                            int heads, float softmax_scale, const void* q, const void* page_pool,
                            int64_t num_pages, const int32_t* block_table, int max_pages,
                            const int32_t* seq_lens, const int32_t* seq_lens_host,
                            const void* sink_buf, const void* recent_buf, float* out, float* lse,
                            void* workspace, size_t workspace_bytes, int32_t* err_word,
                            void* stream) {
  return decode_impl(layout, num_seqs, queries_per_seq, heads, softmax_scale, q, nullptr, nullptr,
                     const_cast<void*>(page_pool), num_pages, block_table, max_pages, seq_lens,
                     seq_lens_host, const_cast<void*>(sink_buf), const_cast<void*>(recent_buf), out,
                     lse, workspace, workspace_bytes, err_word, stream);
}

int mla_lowbit_set_fault_injection(int mode, int64_t wait_cycles) {
  if (mode < 0 || mode > 1 || wait_cycles < 0) return MLA_LOWBIT_EINVAL;
  g_fault_mode.store(mode);
  g_wait_cycles.store(wait_cycles);
  return MLA_LOWBIT_OK;
}

int mla_lowbit_read_error(const int32_t* err_word, int32_t* code_out) {
  if (!err_word || !code_out) return MLA_LOWBIT_ENULL;
  return cudaMemcpy(code_out, err_word, sizeof(int32_t), cudaMemcpyDeviceToHost) == cudaSuccess
             ? MLA_LOWBIT_OK
             : MLA_LOWBIT_ECUDA;
}

const char* mla_lowbit_strerror(int status) {
  switch (status) {
    case MLA_LOWBIT_OK: return "ok";
    case MLA_LOWBIT_EINVAL: return "invalid layout or argument value";
    case MLA_LOWBIT_ENULL: return "required pointer is NULL";
    case MLA_LOWBIT_EALIGN: return "pointer is not 16-byte aligned";
    case MLA_LOWBIT_ESIZE: return "size outside the supported range";
    case MLA_LOWBIT_EWORKSPACE: return "workspace smaller than the decode plan needs";
    case MLA_LOWBIT_ECUDA: return "CUDA runtime call or kernel launch failed";
    default: return "unknown status";
  }
}

int mla_lowbit_version(void) { return 100; }

}  // extern "C"
