/*
 * mla_lowbit.h -- C ABI of the low-bit MLA decode library (one GB300, sm_103a).
 *
 * What it computes follows "QuantMLA: Function-Aligned Dual-Path Quantization
 * for Low-Bit MLA KV Caching":
 *   - Abstract: the content latent (c_kv, 512 channels) is cached at INT4 or
 *     INT2 and the decoupled RoPE key (64 channels) at INT4; a native low-bit
 *     MLA attention kernel unpacks and dequantises inside attention;
 *   - Figure 3 caption: the backend stores packed cache representations and
 *     serves protected sink and recent tokens from bf16 buffers;
 *   - Figure 8 caption: a fused writer packs every incoming token and keeps the
 *     bf16 values of protected tokens; attention uses the bf16 values for
 *     protected tokens and dequantised values otherwise; the reconstructed
 *     content tile serves both matching (QK) and latent aggregation (PV); all
 *     valid tokens share one softmax normalisation;
 *   - Figure 5 / Table 9 captions: the protection policy is sink 4 / local 128.
 * The pages leave the quantiser open; this library fixes it as per-token
 * asymmetric quantisation over 64-channel groups with an fp16 scale and an fp16
 * min per group and round-half-to-even codes (details at mla_lowbit_write).
 *
 * Conventions for every call:
 *   - All tensors are device pointers unless marked "host".  The caller owns
 *     all memory; the library never allocates or frees device memory.
 *   - Calls are asynchronous on the caller's stream (`stream` is a
 *     cudaStream_t; NULL means the legacy default stream).
 *   - Return value: MLA_LOWBIT_OK or a negative MLA_LOWBIT_E* status for errors
 *     found on the host (bad layout, NULL pointer, misalignment, size, small
 *     workspace, launch failure).  Nothing is launched when a call fails.
 *   - Errors that only the device can see (a page id outside the pool, a
 *     position outside the block table, a sequence length out of range) are
 *     OR-ed into the int32 `err_word` (device memory, MLA_LOWBIT_DEV_* bits);
 *     the offending work is skipped, never trapped.  Read it with
 *     mla_lowbit_read_error.
 *   - Pointers to the page pool, bf16 buffers, queries, outputs and the
 *     workspace must be 16-byte aligned.
 */
#ifndef MLA_LOWBIT_H
#define MLA_LOWBIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Cache layout.  Supported (content_bits, rope_bits): (4,4) "C4R4", (2,4)
 * "C2R4", (16,16) unquantised bf16 pages.  The other fields must hold the
 * values shown (they are checked, so a caller states its assumptions). */
typedef struct mla_lowbit_layout {
  int content_bits; /* 4, 2, or 16 (bf16 pages) */
  int rope_bits;    /* 4, or 16 with bf16 pages */
  int group;        /* 64: channels per quantisation group */
  int sink;         /* 4: leading tokens kept in bf16 */
  int local;        /* 128: trailing tokens kept in bf16 */
  int page_tokens;  /* 64: tokens per page */
  int latent;       /* 512: content latent width (kv_lora_rank) */
  int rope;         /* 64: RoPE key width (qk_rope_head_dim) */
  int rotate;       /* 0, or 1 (packed layouts): online Hadamard rotation of the content
                       latent -- the writer replaces each 64-channel content group x by
                       R x, R = H_64 / 8 (orthonormal Sylvester-Hadamard; float32
                       butterfly stages h = 1, 2, .., 32, element i (bit h clear) and
                       i + h becoming (a + b, a - b), then x 1/8), rounded to bf16, for the
                       packed codes and the bf16 copies alike; decode rotates the
                       queries' content channels by R and rotates outputs back, so the
                       result is attention over R^T of the stored keys.  RoPE keys are
                       not rotated.  (QuantMLA, Table 1: QuaRot as an MLA-adapted
                       baseline; the pages' own transforms are fused offline -- this is
                       the un-fused variant.) */
} mla_lowbit_layout;

enum {
  MLA_LOWBIT_OK = 0,
  MLA_LOWBIT_EINVAL = -1,     /* bad layout or argument value */
  MLA_LOWBIT_ENULL = -2,      /* required pointer is NULL */
  MLA_LOWBIT_EALIGN = -3,     /* pointer not 16-byte aligned */
  MLA_LOWBIT_ESIZE = -4,      /* size outside the supported range */
  MLA_LOWBIT_EWORKSPACE = -5, /* workspace smaller than the plan needs */
  MLA_LOWBIT_ECUDA = -6       /* a CUDA runtime call or launch failed */
};

/* Bits OR-ed into the device error word. */
enum {
  MLA_LOWBIT_DEV_BAD_SEQ = 1,   /* writer: sequence index outside [0, num_seqs) */
  MLA_LOWBIT_DEV_BAD_POS = 2,   /* position < 0 or >= max_pages * 64 */
  MLA_LOWBIT_DEV_BAD_PAGE = 4,  /* block-table entry outside [0, num_pages) */
  MLA_LOWBIT_DEV_BAD_LEN = 8,   /* decode: seq_len < 0 or > max_pages * 64 */
  MLA_LOWBIT_DEV_PLAN = 16,     /* decode: device lengths disagree with seq_lens_host */
  MLA_LOWBIT_DEV_PIPELINE = 32  /* decode: an internal pipeline step failed -- a bounded wait gave up
                                  or shared memory was misaligned (the output is invalid) */
};

/* Bytes of one 64-token page: 20736 (C4R4), 12544 (C2R4), 73728 (bf16).
 * Page layout (every region starts on a 128-byte boundary):
 *   packed: content codes [64][latent*content_bits/8] u8, then RoPE codes
 *           [64][rope*rope_bits/8] u8, then metadata [64][9] x {fp16 scale,
 *           fp16 min} (groups 0..7 content, 8 RoPE);
 *           INT4: channel 2i -> low nibble of byte i, 2i+1 -> high nibble;
 *           INT2: channel 4i+j -> bits 2j..2j+1 of byte i;
 *   bf16:   [64][576] bf16 (content then RoPE), no metadata.
 * Returns 0 for an unsupported layout. */
size_t mla_lowbit_page_bytes(const mla_lowbit_layout* layout);

/* Packed bytes per cached token: 324 (C4R4), 196 (C2R4), 1152 (bf16). */
size_t mla_lowbit_bytes_per_token(const mla_lowbit_layout* layout);

/* Fused cache writer (Figure 8 caption: each arriving token is packed, and the
 * bf16 values of protected tokens are kept in their own buffers).
 *
 * Token i (0 <= i < n_tokens) has content latent ckv[i][512] and RoPE key
 * krope[i][64] (bf16, already rotated), sequence seq_idx[i] (or i when seq_idx
 * is NULL) and position pos[i].  It is stored in page block_table[s][pos/64],
 * row pos%64.  For packed layouts each of its 9 groups of 64 channels is
 * quantised with bits b (content_bits for groups 0..7, rope_bits for group 8):
 *   mn, mx = min, max of the group (float32);
 *   s16 = fp16_rn(min((mx - mn) / (2^b - 1), 65504)), m16 = fp16_rn(mn clamped
 *   to +-65504), both float32 operations rounded to nearest;
 *   code = clamp(round_half_even((x - m16) / s16), 0, 2^b - 1) with float32
 *   subtraction and true division; every code is 0 when s16 == 0.
 * A packed copy is written for every token, protected or not.  In addition
 * (packed layouts only) a token with pos < 4 is copied to sink_buf[s][pos] and
 * a token with pos >= seq_lens_after[s] - 128 to recent_buf[s][pos % 128]
 * (seq_lens_after == NULL means pos[i] + 1, the one-token decode step).  Within
 * one call the positions of a sequence must be distinct.
 *
 *   ckv            [n_tokens][512] bf16        krope   [n_tokens][64] bf16
 *   seq_idx        [n_tokens] int32 or NULL    pos     [n_tokens] int32
 *   seq_lens_after [num_seqs] int32 or NULL
 *   block_table    [num_seqs][max_pages] int32 (physical page ids)
 *   page_pool      [num_pages][page_bytes] u8
 *   sink_buf       [num_seqs][4][576] bf16, recent_buf [num_seqs][128][576]
 *                  bf16 (may be NULL for bf16 pages)
 *   err_word       int32 (device), OR-ed MLA_LOWBIT_DEV_* bits
 */
int mla_lowbit_write(const mla_lowbit_layout* layout, int n_tokens, const void* ckv,
                     const void* krope, const int32_t* seq_idx, const int32_t* pos,
                     const int32_t* seq_lens_after, int num_seqs, const int32_t* block_table,
                     int max_pages, void* page_pool, int64_t num_pages, void* sink_buf,
                     void* recent_buf, int32_t* err_word, void* stream);

/* Split-KV plan of one decode call.  The work of a sequence is a list of
 * units: one per 64-token page that holds a packed-served token (bf16 pages:
 * every page), then, for packed layouts, its protected bf16 tokens (sink and
 * recent) in 64-token tiles of 3 units each.  The list is cut into splits of
 * `chunk_pages` units, chosen from the total work and the SM count: the
 * fewest waves of CTAs (one per SM) that the cap allows, or one or two more
 * waves of smaller chunks when the estimated time, waves x (chunk + 3), drops
 * by at least 5 %; the smallest chunk whose splits fit the waves.  The cap is
 * 128 units for the 128-row cluster kernel (query rows a multiple of 128,
 * no rotation) and 64 for the 16-row kernel; it bounds the tokens one split
 * accumulates in fp32 tensor-core outputs.  A bf16 tile belongs to the split
 * that holds its first unit.  Writes the number of splits and the workspace
 * bytes the call needs.  num_sms == 0 asks the current CUDA device. */
int mla_lowbit_decode_plan(const mla_lowbit_layout* layout, int num_seqs, int heads,
                           const int32_t* seq_lens_host, int num_sms, int* total_splits,
                           int* chunk_pages, size_t* workspace_bytes);

/* Low-bit MLA decode attention in absorbed form (Abstract: unpacking and
 * dequantisation inside attention; Figure 8 caption: bf16 values for
 * protected tokens, one global softmax, the content tile used for QK and PV).
 *
 * For sequence s with L = seq_lens[s] cached tokens and head h:
 *   key_t  = bf16 value of token t if t < 4 or t >= L - 128 (sink/recent
 *            buffers), else s16*code + m16 from its packed page (bf16 pages:
 *            always the page value);
 *   z_t    = softmax_scale * dot(q[s][h][0:576], key_t[0:576]);
 *   out[s][h][c] = sum_t softmax(z)_t * key_t[c],  c < 512 (value = latent);
 *   lse[s][h]    = log(sum_t exp(z_t)) (natural log; -inf and out = 0 when L = 0).
 * heads must be a multiple of 16, at most 128 (mla_lowbit_decode_plan takes
 * the rows of a sequence: heads, or n * heads for mla_lowbit_decode_multi,
 * at most 2048).
 *
 *   q             [num_seqs][heads][576] bf16
 *   page_pool     [num_pages][page_bytes] u8 (as written by mla_lowbit_write)
 *   block_table   [num_seqs][max_pages] int32
 *   seq_lens      [num_seqs] int32 (device) and seq_lens_host (host, same
 *                 values; used to plan the split grid)
 *   sink_buf, recent_buf as for the writer (ignored for bf16 pages)
 *   out           [num_seqs][heads][512] float32
 *   lse           [num_seqs][heads] float32, or NULL
 *   workspace     at least the bytes mla_lowbit_decode_plan reports
 *   err_word      int32 (device), OR-ed MLA_LOWBIT_DEV_* bits
 * Launches the split kernel and the log-sum-exp combine kernel on `stream`.
 * The split kernel is fixed by the layout and the row count: packed,
 * unrotated layouts with a multiple of 128 rows per sequence run on tcgen05
 * tensor cores as 2-CTA clusters; every other call runs on mma.sync
 * tensor-core instructions in 16-row chunks. */
int mla_lowbit_decode(const mla_lowbit_layout* layout, int num_seqs, int heads,
                      float softmax_scale, const void* q, const void* page_pool,
                      int64_t num_pages, const int32_t* block_table, int max_pages,
                      const int32_t* seq_lens, const int32_t* seq_lens_host,
                      const void* sink_buf, const void* recent_buf, float* out, float* lse,
                      void* workspace, size_t workspace_bytes, int32_t* err_word,
                      void* stream);

/* One decode step with its append (QuantMLA, Figure 8 caption: the writer packs
 * every incoming token and attention runs over the packed cache and the bf16
 * buffers): writes the token at position seq_lens[s] - 1 of every sequence
 * exactly as mla_lowbit_write does with pos = seq_lens[s] - 1 and
 * seq_lens_after = seq_lens, then decodes exactly as mla_lowbit_decode over
 * seq_lens[s] tokens.  Results (pool bytes, bf16 buffers, out, lse) are
 * identical to that pair of calls.  For packed layouts on the default split
 * kernel both happen in the decode launch (the new token is inside the recent
 * window, so no packed split reads the bytes being written, and the bf16
 * split reads the new values from ckv_new/krope_new, rotating the content
 * latent itself on a rotated layout); otherwise the writer kernel runs first
 * on `stream`.
 *
 *   ckv_new    [num_seqs][512] bf16, krope_new [num_seqs][64] bf16 (16-byte aligned)
 *   seq_lens   device, every entry >= 1 (seq_lens_host the same values)
 *   page_pool, sink_buf, recent_buf are written (as by mla_lowbit_write)
 * Other arguments, errors and the workspace as for mla_lowbit_decode;
 * seq_lens_host entries < 1 return MLA_LOWBIT_EINVAL. */
int mla_lowbit_write_decode(const mla_lowbit_layout* layout, int num_seqs, int heads,
                            float softmax_scale, const void* q, const void* ckv_new,
                            const void* krope_new, void* page_pool, int64_t num_pages,
                            const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                            const int32_t* seq_lens_host, void* sink_buf, void* recent_buf,
                            float* out, float* lse, void* workspace, size_t workspace_bytes,
                            int32_t* err_word, void* stream);

/* Multi-token query decode (several new tokens per sequence at once, as for
 * multi-token prediction or speculative verification): queries_per_seq = n
 * queries per sequence at positions L - n .. L - 1 (L = seq_lens[s], all n
 * tokens already written), each attending causally: query i sees tokens
 * 0 .. L - n + i.  Same arithmetic, tolerance and errors as mla_lowbit_decode
 * otherwise; the n queries run as n blocks of `heads` rows over one pass of the
 * cache (the masked tokens are all inside the recent window, 1 <= n <= 16).
 *
 *   q      [num_seqs][n][heads][576] bf16
 *   out    [num_seqs][n][heads][512] float32; lse [num_seqs][n][heads] or NULL
 *   seq_lens_host entries >= n
 *   workspace  mla_lowbit_decode_plan with heads = n * heads
 * The split kernel is chosen as for mla_lowbit_decode from the row count
 * n * heads (so 128-row blocks run on tcgen05). */
int mla_lowbit_decode_multi(const mla_lowbit_layout* layout, int num_seqs, int queries_per_seq,
                            int heads, float softmax_scale, const void* q, const void* page_pool,
                            int64_t num_pages, const int32_t* block_table, int max_pages,
                            const int32_t* seq_lens, const int32_t* seq_lens_host,
                            const void* sink_buf, const void* recent_buf, float* out, float* lse,
                            void* workspace, size_t workspace_bytes, int32_t* err_word,
                            void* stream);

/* mla_lowbit_decode for callers that cannot allocate device memory.  The
 * pages have no counterpart to this entry point: it exists because some hosts
 * give a kernel only its inputs and outputs -- a serving engine that has
 * already reserved almost all of HBM for its own cache pool, a plug-in
 * interface without a workspace argument, or a loop that cannot afford the
 * device-wide synchronisation of cudaMalloc.
 *
 * Same arguments, results and error handling as mla_lowbit_decode, minus the
 * workspace: the split partials live in a fixed 32 MiB device array owned by
 * the library (every GPU that loads the library holds it until the process
 * exits).  Calls whose plan needs more than 32 MiB (see
 * mla_lowbit_decode_plan) return MLA_LOWBIT_ESIZE and launch nothing.  The
 * call allocates and frees nothing.
 *
 * The first call on a device looks up that device's address of the array
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  All calls share the one array and it keeps the
 * last call's contents (nothing in it needs to start at zero: each call writes
 * every byte it reads).  Calls that overlap on the GPU -- on different streams,
 * or from different threads without ordering -- race on the array; issue them
 * on one stream or order them yourself. */
int mla_lowbit_decode_noalloc(const mla_lowbit_layout* layout, int num_seqs, int heads,
                              float softmax_scale, const void* q, const void* page_pool,
                              int64_t num_pages, const int32_t* block_table, int max_pages,
                              const int32_t* seq_lens, const int32_t* seq_lens_host,
                              const void* sink_buf, const void* recent_buf, float* out,
                              float* lse, int32_t* err_word, void* stream);

/* Self-test of the failure path of the tcgen05 decode kernels (the pages have
 * no counterpart to it; it checks this library's own error handling).  Those
 * kernels hand work between warp roles through mbarriers, and every wait on
 * one is bounded: when it runs out the CTA sets MLA_LOWBIT_DEV_PIPELINE in the
 * error word, its warps leave their loops together, the tensor-core work
 * already issued drains, tensor memory is freed and the kernel returns (no
 * trap, the context stays usable; the call's output is invalid).
 *
 * This sets, for every later decode call of the process (all threads):
 *   mode        0: normal operation; 1: the 128-row (tcgen05) decode kernel's
 *               unpack warps withhold their first hand-off, so that the waits
 *               behind it run out -- a fault made on purpose, for tests only;
 *   wait_cycles the wait limit in SM clock cycles; 0 restores the default
 *               (about one second).
 * Returns MLA_LOWBIT_EINVAL for a mode other than 0 or 1 or a negative limit.
 * The mma.sync kernel has no such waits and ignores both settings. */
int mla_lowbit_set_fault_injection(int mode, int64_t wait_cycles);

/* Synchronously copies the device error word to *code_out (a blocking
 * cudaMemcpy: it waits for prior work on the legacy default stream). */
int mla_lowbit_read_error(const int32_t* err_word, int32_t* code_out);

/* Human-readable text for a status code; never NULL. */
const char* mla_lowbit_strerror(int status);

/* Library version, major*10000 + minor*100 + patch. */
int mla_lowbit_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_LOWBIT_H */
