// Internal interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace kvgqa {

// cuTensorMapEncodeTiled from the driver (looked up once); nullptr if absent.
PFN_cuTensorMapEncodeTiled_v12000 tma_encoder();

constexpr int kMaxHeadDim = 128;
constexpr int kMaxActiveRows = 1024;  // decode attention keeps per-row tables of A+1 ints in smem

// ------------------------------------------------------------------ RoPE + store
// The RoPE frequencies f_i = theta^(-2i/D) (each a double computed on the
// host), stored as the angle a position step adds in quarter turns,
// f_i * 2/pi: its fraction as a 64-bit fixed-point number (rounded down) and
// its integer part mod 4.  pos * f_i then reduces modulo pi/2 with integer
// arithmetic (rope_math.cuh).
struct RopeFreqs {
  uint64_t frac[kMaxHeadDim / 2];
  uint8_t quad[kMaxHeadDim / 2];
};

struct RopeStoreParams {
  const uint16_t* q;         // decode [A,H_q,D]; prefill [A,T,H_q,D]
  const uint16_t* k;         // decode [A,H_kv,D]; prefill [A,T,H_kv,D]
  const uint16_t* v;
  const int32_t* positions;  // decode [A]; prefill: nullptr (positions are 0..T-1)
  const int32_t* cache_rows; // [A]
  const int32_t* offsets;    // varlen prefill [A]: position of each prompt's first token
  const int32_t* lengths;    // varlen prefill [A]: tokens of each prompt (<= T)
  uint16_t* q_out;           // rotated Q, same layout as q
  int32_t* item_order;       // varlen prefill: (query tile, prompt) pairs, longest first (written by CTA 0)
  uint16_t* k_cache;         // [S,H_kv,max_seq,D]
  uint16_t* v_cache;
  int32_t* status;
  int A, T, H_q, H_kv, D, S, max_seq;
  int f16;                   // storage: 0 BF16, 1 IEEE binary16
  RopeFreqs freqs;           // the D/2 frequencies theta^(-2i/D)
};

// mode 0: decode (token a at positions[a]); 1: equal-length prefill (one CTA
// per position 0..T-1, all prompts); 2: varlen prefill (token t of prompt a at
// offsets[a] + t, t < lengths[a]).  Mode 0 gives each token four CTAs, each
// with a quarter of the frequencies (H_kv * D / 8 must divide by 4); mode 2
// walks the real tokens in groups of 8 per CTA (up to 2048 prompts; with
// more, the padded tokens with four CTAs each, as mode 0).
cudaError_t launch_rope_kv_store(const RopeStoreParams& p, int mode, cudaStream_t stream);

// ------------------------------------------------------------------ decode attention
struct DecodeParams {
  const uint16_t* q;          // [A,H_q,D] rotated queries (attention call) or raw queries (fused step)
  const uint16_t* k_cache;    // [S,H_kv,max_seq,D]
  const uint16_t* v_cache;
  const int32_t* positions;   // [A]
  const int32_t* cache_rows;  // [A]
  uint16_t* out;              // [A,H_q,D]
  float* partials;            // split-K partial results (workspace)
  int32_t* counters;          // per (row, KV head): partials written so far (zero between calls)
  int32_t* status;
  int A, H_q, H_kv, G, D, S, max_seq;
  int num_ctas;               // grid size of the split-K kernel
  int f16;                    // storage: 0 BF16, 1 IEEE binary16
  float scale_log2;           // scale * log2(e)
  // Early start (whole-step call only, where the previous kernel in the
  // stream is that call's own store kernel, which writes only the rotated
  // queries and each active row's new cell): cache tiles without a new cell
  // are loaded before the store kernel ends.
  int early;
  // Fused decode step only (fused != 0): the kernel rotates q itself and
  // stores the rotated new K and raw new V into each row's cell at positions[a].
  int fused;
  const uint16_t* k_new;      // [A,H_kv,D]
  const uint16_t* v_new;      // [A,H_kv,D]
  uint16_t* k_cache_w;        // the same caches, written
  uint16_t* v_cache_w;
  RopeFreqs freqs;            // the D/2 frequencies theta^(-2i/D)
};

// Padded group size used by the decode kernels: the next power of two >= G.
int decode_group_pad(int G);
// Workspace of the decode attention behind the status block: per-segment
// counters (A * H_kv ints, rounded up to 256 bytes), then the split-K
// partials of the grid the kernel uses on `device`.
struct DecodeLayout {
  int num_ctas;
  size_t counter_bytes, partial_bytes;
};
cudaError_t decode_layout(int device, int D, int GP, int64_t A, int64_t H_kv, DecodeLayout* out);
cudaError_t launch_cached_gqa_attention(const DecodeParams& p, cudaStream_t stream);
// The same for IEEE binary16 storage (called by the above when p.f16 is set).
cudaError_t launch_cached_gqa_attention_f16(const DecodeParams& p, cudaStream_t stream);

// Size of the library's own device scratch array (status block + partials)
// used by the entry point for callers that cannot allocate, and its device
// address on `device` (looked up once per device; `device` must be current).
constexpr size_t kStaticScratchBytes = 4u << 20;
cudaError_t static_scratch_address(int device, void** ptr);

// ------------------------------------------------------------------ prefill attention
struct PrefillParams {
  const uint16_t* q_rot;      // [A,T,H_q,D] rotated queries (workspace)
  const uint16_t* k_cache;    // [S,H_kv,max_seq,D]
  const uint16_t* v_cache;
  const int32_t* cache_rows;  // [A]
  const int32_t* offsets;     // [A] or nullptr (all 0): position of each prompt's first token
  const int32_t* lengths;     // [A] or nullptr (all T): tokens of each prompt
  // Prompts at offsets: the pairs c = qt * A + a (query tile qt of prompt a)
  // ordered by their key tiles, most first (see kPrefillTile); nullptr for
  // the equal-length prefill, whose query tile index already orders them.
  const int32_t* item_order;
  uint16_t* out;              // [A,T,H_q,D]
  int32_t* status;
  int A, T, H_q, H_kv, G, D, S, max_seq;
  float scale_log2;
  int f16;                    // storage: 0 BF16, 1 IEEE binary16
  int out_32b;                // out is 32-byte aligned (set by the launcher): whole-sector stores
};

cudaError_t launch_prefill_attention(const PrefillParams& p, cudaStream_t stream);

// Query and key tile of the prefill attention kernel; the varlen prefill's
// item order has one entry per (query tile, prompt) pair.
constexpr int kPrefillTile = 128;
inline int64_t prefill_order_entries(int64_t A, int64_t T) { return A * ((T + kPrefillTile - 1) / kPrefillTile); }

// ------------------------------------------------------------------ bounded-wait check
// One CTA whose only wait can never complete (kvgqa_check_bounded_wait).
cudaError_t launch_bounded_wait_check(int32_t* status, cudaStream_t stream);

}  // namespace kvgqa
