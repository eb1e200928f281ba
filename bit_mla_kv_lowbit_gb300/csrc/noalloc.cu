// Decode entry point for callers that cannot allocate device memory.
//
// Some hosts hand this library only their input and output buffers: a serving
// engine that has already reserved nearly all of HBM for its own KV-cache pool,
// a plug-in interface that offers no workspace argument, or a latency-critical
// loop where the device-wide synchronisation of cudaMalloc is not acceptable.
// For them, mla_lowbit_decode_noalloc runs the same split + combine kernels as
// mla_lowbit_decode, with the split partials placed in a fixed array that the
// library itself owns in device memory (below), so the caller passes no
// workspace and nothing is allocated per call.
#include <mutex>

#include "common.cuh"

namespace mlalb {
namespace {

// Largest workspace this entry point can serve.  Every GPU that loads the
// library keeps this array for the lifetime of the process.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch, looked up once per device.  In host code
// the array's name is only a host-side stand-in, never a device address.
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return MLA_LOWBIT_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return MLA_LOWBIT_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_LOWBIT_OK;
}

}  // namespace
}  // namespace mlalb

using namespace mlalb;

extern "C" {

int mla_lowbit_decode_noalloc(const mla_lowbit_layout* layout, int num_seqs, int heads,
                              float softmax_scale, const void* q, const void* page_pool,
                              int64_t num_pages, const int32_t* block_table, int max_pages,
                              const int32_t* seq_lens, const int32_t* seq_lens_host,
                              const void* sink_buf, const void* recent_buf, float* out,
                              float* lse, int32_t* err_word, void* stream) {
  if (!layout || !seq_lens_host) return MLA_LOWBIT_ENULL;
  int total = 0, chunk = 0;
  size_t need = 0;
  int st = mla_lowbit_decode_plan(layout, num_seqs, heads, seq_lens_host, 0, &total, &chunk,
                                  &need);
  if (st != MLA_LOWBIT_OK) return st;
  if (need > kNoAllocScratchBytes) return MLA_LOWBIT_ESIZE;
  void* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != MLA_LOWBIT_OK) return st;
  // Every byte of the workspace that the kernels read is written earlier in
  // the same call, so the array needs no clearing between calls.
  return mla_lowbit_decode(layout, num_seqs, heads, softmax_scale, q, page_pool, num_pages,
                           block_table, max_pages, seq_lens, seq_lens_host, sink_buf, recent_buf,
                           out, lse, scratch, kNoAllocScratchBytes, err_word, stream);
}

}  // extern "C"
