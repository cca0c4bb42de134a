// K2: split-K flash-decode over the shared slot KV cache on tcgen05 tensor
// cores, with K3, the combine of split segments, run by the CTA that finishes
// a segment last.
//
// microLLM-rocm ARCHITECTURE.md, section "Tensor ownership boundary": each
// survivor token attends to its own row's cached prefix, with device
// positions[A] and cache_rows[A].  Section "Attention layout boundary": with
// GQA one K/V head serves a group of query heads (the zero-stride idea: K/V
// are never expanded).  operator-development.md, "Public interfaces": low
// precision softmax keeps FP32 reductions and rounds only the caller output.
//
// Work split.  Segment (a, g) is the prefix of KV head g in row cache_rows[a]:
// n_a = positions[a] + 1 keys, contiguous in memory.  A tile holds up to TK
// keys (128, or 256 at head width 64: 64 KB of K and V either way).  A tile
// costs about the same whether it is whole or a short tail (its softmax and
// P.V round trip dominate), so work is balanced in a
// virtual key space where segment (a, g) occupies ceil(n_a / TK) * TK + SEG_V
// * TK / 128 keys: its n_a real keys first, then padding that stands for the
// cost of its tail tile and its end.  CTA b
// of the persistent grid (one CTA per SM) takes the virtual range
// [b*W, (b+1)*W), W = ceil(V_tot / grid), and processes the real keys in it.
// A segment whose real keys lie inside one CTA is finished there (output in the storage type
// written); a segment cut by a CTA boundary leaves FP32 partials (m, l, o):
// the CTA where it starts writes slot 1, each later CTA slot 0.  The combine
// (K3) runs in whichever of those CTAs finishes last: each counts its partial
// in a per-segment counter, and the one that completes the count merges the
// segment's partials, writes the output (storage type) and resets the counter to zero.
//
// Inside a CTA, per tile of up to TK keys of one segment (below for TK = 128;
// a 256-key tile is two 128-key blocks, each its own S MMA chain into its own
// TMEM columns and one key per softmax thread, and one P.V over both):
//   warp 4     TMA producer: K and V tiles (128B swizzle; a whole tile in one
//              128-row box per 64-column half, a short tail in 32-row boxes so
//              it reads at most 31 rows past the prefix) and the group's query
//              rows (16 rows: the G heads, the rest padding) into a 3-stage
//              ring (fewer TMA instructions per tile: the producer's issue
//              time was part of each tile's period);
//   warp 5     one thread issues tcgen05.mma: S^T = K Q_g^T (M = 128 keys,
//              N = 16 heads) into one of two TMEM buffers (the next tile's
//              while the softmax works on this one; in the attention call only
//              if that tile has landed, else after this tile's P.V), then
//              O^T += V^T P^T (M = D, N = 16; V is an MN-major operand) into a
//              TMEM accumulator;
//   warps 0-3  one thread per key: S^T row from TMEM, FP32 online softmax per
//              head (a warp reduction instruction + a 4-warp exchange for the
//              tile maximum; each thread keeps its keys' share of the row sums,
//              summed over the CTA once, at the segment end), P^T in the
//              storage type into 128B-swizzled shared memory; the O^T
//              rescale (TMEM load/scale/store, one lane per d) happens only when
//              a head's maximum grew by more than 2^8; at a segment end each
//              lane d writes O^T[d][h] / l[h] (or the partial).
// The tensor cores do the two contractions, so the CUDA cores only run the
// softmax: the kernel is bound by the HBM stream of K and V.
#ifndef KVGQA_DECODE_F16
#define KVGQA_DECODE_F16 0  // 1: the IEEE binary16 build of these kernels
#endif

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "elem.cuh"
#include "kvgqa_internal.h"
#include "rope_math.cuh"
#include "tcgen05.cuh"

namespace kvgqa {
namespace {

// Storage type of this translation unit's kernels (flash_decode_f16.cu
// compiles the same kernels for IEEE binary16).
constexpr bool kF16 = KVGQA_DECODE_F16 != 0;
using E = Elem<kF16>;
constexpr CUtensorMapDataType kTmaElem = kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

constexpr int BN = 128;                 // keys per block (= MMA M = TMEM lanes = softmax threads)
constexpr int NQ = 16;                  // MMA N: query heads of a group, padded
constexpr int BOX_ROWS = 32;            // rows per TMA box of a K or V tile
constexpr int SUB = BN * 128;           // one [128 rows x 64 16-bit values] swizzled block
constexpr int QSUB = NQ * 128;          // one [16 rows x 64 16-bit values] swizzled sub-tile
// 4 softmax warps + producer + MMA, plus the query/cell prep warp of the fused step
__host__ __device__ constexpr int threads_of(bool fused) { return fused ? 224 : 192; }
constexpr int W_MIN = 256;              // fewest (virtual) keys a CTA is given, per 128-key block of a tile
constexpr int SEG_V = 128;              // virtual keys charged for a segment end, per block of a tile
constexpr unsigned FULL = 0xffffffffu;

// One split-K partial result: o[GP][D], then m[GP], then l[GP] (each of the
// last two padded to at least 2 floats) so that every slot starts on a
// 16-byte boundary for the float4 accesses.
__host__ __device__ constexpr int slot_floats(int GP, int D) { return GP * D + 2 * (GP < 2 ? 2 : GP); }
__host__ __device__ constexpr int slot_l_offset(int GP, int D) { return GP * D + (GP < 2 ? 2 : GP); }
constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int D, bool FUSED>
struct Cfg {
  static constexpr int NSUB = D / 64;
  // Keys per tile: one 128-key block, or two at D = 64, so that a tile
  // carries 64 KB of K and V at either width (the per-tile chain of S MMA,
  // softmax and P.V, not the bytes, bounded 32 KB tiles).  A block is one
  // M = 128 MMA and one key per softmax thread.  Every form of the call (the
  // attention call, the early-start and the fused step) uses the same tiles,
  // so that their FP32 sums, and hence their outputs, are bit-identical.
  static constexpr int KB = D == 64 ? 2 : 1;
  static constexpr int TK = KB * BN;
  static constexpr int SUBK = KB * SUB;                // one [TK rows x 64 values] swizzled sub-tile
  static constexpr int NS = D == 128 || KB == 2 ? 3 : 4;  // stages
  static constexpr int K_OFF = 0;                      // inside a stage
  static constexpr int V_OFF = NSUB * SUBK;
  // Attention call: each stage also carries the segment's (rotated) query
  // tile, loaded with every K/V tile.  Fused step: the query tile is rotated
  // in shared memory once per segment, in a ring of QR buffers, one more than
  // the stages, so the producer (at most NS tiles, hence NS segments, ahead)
  // never waits for a query buffer and no per-segment barrier of the ring can
  // run two phases ahead of its waiter.
  static constexpr int Q_OFF = 2 * NSUB * SUBK;
  static constexpr int STAGE = FUSED ? 2 * NSUB * SUBK : 2 * NSUB * SUBK + NSUB * QSUB;  // multiple of 1024
  static constexpr int QR = FUSED ? NS + 1 : 0;
  static constexpr int QB_OFF = NS * STAGE;            // fused: query tiles [QR][16 x D]
  static constexpr int QBUF = NSUB * QSUB;
  static constexpr int PBUF = TK / 64 * QSUB;                 // P^T [16 x TK keys]: 64-key swizzled sub-tiles
  static constexpr int P_OFF = QB_OFF + QR * QBUF;             // P^T x2 buffers
  static constexpr int RED_OFF = P_OFF + 2 * PBUF;             // [3][4 warps][16] floats: maxima x2, sums
  static constexpr int PREFIX_OFF = RED_OFF + 3 * 4 * NQ * 4;  // [kMaxActiveRows + 1] ints
  static constexpr int NKEYS_OFF = PREFIX_OFF + (kMaxActiveRows + 1) * 4;  // [kMaxActiveRows] ints
  static constexpr int BAR_OFF = align_up(NKEYS_OFF + kMaxActiveRows * 4, 16);
  // kv_full[NS], kv_empty[NS], s_full[2], p_full[2], o_done[2], q_free[QR],
  // prep_done[QR], patch_done[QR], last_full[QR], q_full[QR], drain
  static constexpr int NBAR = 2 * NS + 7 + 5 * QR;
  static constexpr int SLOT_OFF = BAR_OFF + NBAR * 8;
  static constexpr int FLAG_OFF = SLOT_OFF + 8;
  static constexpr int SMEM = FLAG_OFF + 16 + 1024;            // + alignment slack
  static constexpr int TMEM_COLS = KB == 1 ? 64 : 128;        // S^T x2 (KB x 16 cols each) + O^T (16 cols)
  static constexpr int O_COL = 2 * KB * NQ;                    // TMEM column of O^T
  static_assert(STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct DecodeMaps {
  CUtensorMap kc;  // cache [S*H_kv][max_seq][D], box {64, 32, 1}
  CUtensorMap vc;
  CUtensorMap kcf;  // the same with box {64, 128, 1}: a whole tile per sub-tile
  CUtensorMap vcf;
  CUtensorMap q;   // q_rot [A*H_q][D], box {64, 16}
};

// Virtual length of a segment of n real keys in tiles of TK keys (0 for an
// invalid row).
template <int TK>
__device__ __forceinline__ int seg_vlen(int n) { return n == 0 ? 0 : (n + TK - 1) / TK * TK + SEG_V * (TK / BN); }

// Running sum over rows of H_kv * seg_vlen(n_a): prefix[a] is the virtual
// start of row a's first segment.  Invalid metadata -> an empty row.
template <int TK>
__device__ void build_prefix(const DecodeParams& p, int* prefix, int* nkeys, bool flag) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    int carry = 0, bad = 0;
    for (int base = 0; base < p.A; base += 32) {
      const int a = base + lane;
      int n = 0;
      if (a < p.A) {
        const int pos = p.positions[a];
        const int row = p.cache_rows[a];
        const bool pos_ok = pos >= 0 && pos < p.max_seq;
        const bool row_ok = row >= 0 && row < p.S;
        if (pos_ok && row_ok) n = seg_vlen<TK>(pos + 1) * p.H_kv;
        nkeys[a] = pos_ok && row_ok ? pos + 1 : 0;
        bad |= (pos_ok ? 0 : KVGQA_FLAG_POSITION_RANGE) | (row_ok ? 0 : KVGQA_FLAG_ROW_RANGE);
      }
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(FULL, incl, off);
        if (lane >= off) incl += t;
      }
      if (a < p.A) prefix[a + 1] = carry + incl;
      carry += __shfl_sync(FULL, incl, 31);
    }
    if (lane == 0) prefix[0] = 0;
    for (int off = 16; off; off >>= 1) bad |= __shfl_xor_sync(FULL, bad, off);
    if (flag && lane == 0 && bad) atomicOr(p.status, bad);
  }
  __syncthreads();
}

template <int TK>
__device__ __forceinline__ int keys_per_cta(int k_tot, int num_ctas) {
  const int w = (k_tot + num_ctas - 1) / num_ctas;
  return w < W_MIN * (TK / BN) ? W_MIN * (TK / BN) : w;
}

// Walks the tiles of one CTA's virtual range [v0, v1): segment by segment, the
// real keys of each in tiles of at most TK.  Every role runs its own copy.
template <int TK>
struct Cursor {
  const int* prefix;
  const int* nkeys;
  int H_kv, A, v0, v1;
  int a, g, n, vlen, vlo;  // current segment: row, head, real keys, virtual length and start
  int x, x_end;            // next real key of the segment and the end of this CTA's part
  int k_first;             // first real key of this CTA's part of the segment

  __device__ __forceinline__ int row_vlen(int r) const { return (prefix[r + 1] - prefix[r]) / H_kv; }

  // Enter segment (a, g): clip its real keys to [v0, v1); false if none.
  __device__ __forceinline__ bool enter() {
    n = nkeys[a];
    vlen = row_vlen(a);
    vlo = prefix[a] + g * vlen;
    const int lo = max(v0, vlo), hi = min(v1, vlo + n);
    x = lo - vlo;
    x_end = hi - vlo;
    k_first = x;
    return lo < hi;
  }
  // Step to the next segment that starts before v1; false when there is none.
  __device__ __forceinline__ bool next_segment() {
    for (;;) {
      if (++g == H_kv) {
        g = 0;
        do { ++a; } while (a < A && row_vlen(a) == 0);
        if (a >= A) return false;
      }
      if (prefix[a] + g * row_vlen(a) >= v1) return false;
      if (enter()) return true;
    }
  }
  __device__ void init(const int* pf, const int* nk, int h_kv, int rows, int lo, int hi) {
    prefix = pf; nkeys = nk; H_kv = h_kv; A = rows; v0 = lo; v1 = hi;
    int l = 0, r = A - 1;  // last row with prefix[row] <= v0
    while (l < r) {
      const int mid = (l + r + 1) >> 1;
      if (prefix[mid] <= lo) l = mid; else r = mid - 1;
    }
    a = l;
    while (row_vlen(a) == 0) ++a;
    g = (lo - prefix[a]) / row_vlen(a);
    if (!enter()) {
      if (!next_segment()) x = x_end = 0, done_ = true;
    }
  }
  bool done_ = false;
  __device__ __forceinline__ bool more() const { return !done_; }
  __device__ __forceinline__ int k0() const { return x; }
  __device__ __forceinline__ int nt() const { return min(TK, x_end - x); }
  __device__ __forceinline__ bool first() const { return x == k_first; }
  __device__ __forceinline__ bool last() const { return x + nt() == x_end; }
  __device__ __forceinline__ bool whole() const { return vlo >= v0 && vlo + n <= v1; }
  __device__ __forceinline__ int slot() const { return vlo < v0 ? 0 : 1; }
  // Another tile follows in this CTA (used to run S of the next tile early).
  __device__ __forceinline__ bool has_next() const {
    if (!last()) return true;
    Cursor c = *this;
    return c.next_segment();
  }
  __device__ void advance() {
    if (!last()) { x += nt(); return; }
    if (!next_segment()) done_ = true;
  }
  // Skip the rest of the current segment (a walk over segments only).
  __device__ void advance_segment() {
    if (!next_segment()) done_ = true;
  }
};

// K3, the combine: merge the partials of CTAs b0..b1 for segment (a, g) and
// write the output of its G query heads.  One thread per d (d < D) of
// the 128 softmax threads.  Partials of other CTAs are read past L1, in
// batches of kMaxParts partials whose loads (all heads) are issued before any
// is used: one L2 round trip per batch instead of one per partial and head.
template <int D, int GP>
__device__ void combine_segment(const DecodeParams& p, int a, int g, int b0, int b1, int d) {
  if (d >= D) return;
  constexpr size_t SLOT = slot_floats(GP, D);
  constexpr int kMaxParts = GP >= 16 ? 1 : (GP >= 8 ? 2 : 4);  // bounded by registers
  float M[GP], lsum[GP], acc[GP];
#pragma unroll
  for (int h = 0; h < GP; ++h) { M[h] = -INFINITY; lsum[h] = 0.f; acc[h] = 0.f; }
  for (int bb = b0; bb <= b1; bb += kMaxParts) {
    float m[kMaxParts][GP], lb[kMaxParts][GP], ob[kMaxParts][GP];
#pragma unroll
    for (int j = 0; j < kMaxParts; ++j) {
      const int b = bb + j;
      const float* sp = p.partials + (static_cast<size_t>(b) * 2 + (b == b0 ? 1 : 0)) * SLOT;
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const bool use = b <= b1 && h < p.G;
        m[j][h] = use ? __ldcg(sp + GP * D + h) : -INFINITY;
        lb[j][h] = use ? __ldcg(sp + slot_l_offset(GP, D) + h) : 0.f;
        ob[j][h] = use ? __ldcg(sp + h * D + d) : 0.f;
      }
    }
    // one pass over the batch, rescaling the running sums as the maximum grows
#pragma unroll
    for (int j = 0; j < kMaxParts; ++j) {
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        if (m[j][h] == -INFINITY) continue;  // unused entry
        const float mn = fmaxf(M[h], m[j][h]);
        const float s_old = exp2f(M[h] - mn), s_new = exp2f(m[j][h] - mn);
        lsum[h] = lsum[h] * s_old + lb[j][h] * s_new;
        acc[h] = acc[h] * s_old + ob[j][h] * s_new;
        M[h] = mn;
      }
    }
  }
#pragma unroll
  for (int h = 0; h < GP; ++h)
    if (h < p.G) p.out[(static_cast<size_t>(a) * p.H_q + g * p.G + h) * D + d] = E::from_f32(acc[h] / lsum[h]);
}

// Atomic add with release and acquire semantics at GPU scope.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* ptr, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
  return old;
}

template <int D, int GP, bool FUSED, bool EARLY>
__global__ void __launch_bounds__(threads_of(FUSED), 1)
flash_decode_splitk_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap map_k,
                           const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_q,
                           const __grid_constant__ CUtensorMap map_kf, const __grid_constant__ CUtensorMap map_vf) {
  static_assert(!(FUSED && EARLY), "the fused step has no store kernel before it");
  using C = Cfg<D, FUSED>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  int* prefix = reinterpret_cast<int*>(smem + C::PREFIX_OFF);
  int* nkeys = reinterpret_cast<int*>(smem + C::NKEYS_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::NS;
  uint64_t* s_full = bars + 2 * C::NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  // per segment k, slot k % QR, phase k / QR:
  uint64_t* q_free = o_done + 2;           // the segment's S MMAs are complete
  uint64_t* prep_done = q_free + C::QR;    // fused step: its query tile is rotated
  uint64_t* patch_done = prep_done + C::QR;  // fused step: the new key is in its last tile
  uint64_t* last_full = patch_done + C::QR;  // fused step: the TMA of the tile with the new key landed
  uint64_t* q_full = last_full + C::QR;    // fused step: the segment's raw query tile landed
  uint64_t* drain = q_full + C::QR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SLOT_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::FLAG_OFF);
  volatile int* merge_flag = abort_flag + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);  // one arrival per softmax warp
      mbar_init(&o_done[b], 1);
    }
    for (int b = 0; b < C::QR; ++b) {
      mbar_init(&q_free[b], 1);
      mbar_init(&prep_done[b], 1);
      mbar_init(&patch_done[b], 1);
      mbar_init(&last_full[b], 1);
      mbar_init(&q_full[b], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // The producer's descriptors are fetched and its L2 policies created while
  // the CTA sets up (creating the two policies took about 0.35 us when the
  // producer did it after the set-up).
  uint64_t pol_kv = 0, pol_q = 0;
  if (threadIdx.x == 32 * 4) {
    tma_prefetch_map(&map_k);
    tma_prefetch_map(&map_v);
    tma_prefetch_map(&map_q);
    pol_kv = l2_evict_first_policy();
    pol_q = l2_evict_last_policy();
  }
  // Everything past pdl_wait() may read what the previous kernel wrote.  With
  // an early start only the producer waits, before the first query tile or
  // tile with a new cell it loads: the positions and rows read here are inputs
  // of the whole step, which its store kernel does not write.
  if constexpr (!EARLY) pdl_wait();
  pdl_trigger();  // the next kernel in the stream may launch and set itself up
  build_prefix<C::TK>(p, prefix, nkeys, blockIdx.x == 0);  // ends with __syncthreads

  const int v_tot = prefix[p.A];
  const int W = keys_per_cta<C::TK>(v_tot, p.num_ctas);
  const int v0 = blockIdx.x * W;
  const int v1 = min(v0 + W, v_tot);
  Cursor<C::TK> cur;
  if (v0 < v_tot) cur.init(prefix, nkeys, p.H_kv, p.A, v0, v1);
  if (v0 >= v_tot || !cur.more()) return;  // uniform: nothing allocated yet

  // The tensor-memory address reaches the warps that use it through a
  // named barrier the producer (warp 4) does not join: it needs no tensor
  // memory, and starts its copies without waiting for the allocation.
  if (warp == 5) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  uint32_t tmem = 0;
  if (warp != 4) {
    tc_fence_before();
    named_bar_sync(2, threads_of(FUSED) - 32);
    tc_fence_after();
    tmem = *tmem_slot;
  }
  const uint32_t sbase = smem_u32(smem);

  if (warp == 4) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      if constexpr (!FUSED) {
        // each tile brings its K and V rows and the segment's rotated query tile
        int it = 0;
        // Early start: the K/V rows of the first tiles (at most one per stage,
        // up to the first that holds a new cell) are loaded before waiting for
        // the store kernel, their query tiles right after it.  The loops stay
        // rolled: unrolled, this once-per-CTA code measured about 4 us slower
        // over the whole kernel on GB300.
        if constexpr (EARLY) {
          int qrow[C::NS];
          int n_early = 0;
#pragma unroll 1
          for (; n_early < C::NS && cur.more() && !(cur.last() && cur.x_end == cur.n); cur.advance(), ++n_early) {
            const int nb = (cur.nt() + BOX_ROWS - 1) / BOX_ROWS;
            unsigned char* st = smem + n_early * C::STAGE;
            const int kv_row = p.cache_rows[cur.a] * p.H_kv + cur.g;
            mbar_arrive_expect_tx(&kv_full[n_early], static_cast<uint32_t>(C::NSUB) * (2u * nb * BOX_ROWS * 128u + QSUB));
#pragma unroll 1
            for (int sub = 0; sub < C::NSUB; ++sub) {
              if (nb * BOX_ROWS == C::TK) {  // a whole tile: one box per 128-key block
#pragma unroll 1
                for (int kb = 0; kb < C::KB; ++kb) {
                  tma_load_3d(st + C::K_OFF + sub * C::SUBK + kb * SUB, &map_kf, sub * 64, cur.k0() + kb * BN, kv_row,
                              &kv_full[n_early], pol_kv);
                  tma_load_3d(st + C::V_OFF + sub * C::SUBK + kb * SUB, &map_vf, sub * 64, cur.k0() + kb * BN, kv_row,
                              &kv_full[n_early], pol_kv);
                }
                continue;
              }
#pragma unroll 1
              for (int b = 0; b < nb; ++b) {
                tma_load_3d(st + C::K_OFF + sub * C::SUBK + b * BOX_ROWS * 128, &map_k, sub * 64,
                            cur.k0() + b * BOX_ROWS, kv_row, &kv_full[n_early], pol_kv);
                tma_load_3d(st + C::V_OFF + sub * C::SUBK + b * BOX_ROWS * 128, &map_v, sub * 64,
                            cur.k0() + b * BOX_ROWS, kv_row, &kv_full[n_early], pol_kv);
              }
            }
            qrow[n_early] = cur.a * p.H_q + cur.g * p.G;
          }
          pdl_wait();
#pragma unroll 1
          for (int i = 0; i < n_early; ++i)
#pragma unroll 1
            for (int sub = 0; sub < C::NSUB; ++sub)
              tma_load_3d(smem + i * C::STAGE + C::Q_OFF + sub * QSUB, &map_q, sub * 64, qrow[i], 0, &kv_full[i],
                          pol_q);
          it = n_early;
        }
        for (; cur.more(); cur.advance(), ++it) {
          const int s = it % C::NS;
          if (it >= C::NS && !mbar_wait_bounded(&kv_empty[s], ((it / C::NS) - 1) & 1, abort_flag, p.status)) break;
          const int nb = (cur.nt() + BOX_ROWS - 1) / BOX_ROWS;
          const uint32_t bytes = static_cast<uint32_t>(C::NSUB) * (2u * nb * BOX_ROWS * 128u + QSUB);
          unsigned char* st = smem + s * C::STAGE;
          const int kv_row = p.cache_rows[cur.a] * p.H_kv + cur.g;
          mbar_arrive_expect_tx(&kv_full[s], bytes);
          for (int sub = 0; sub < C::NSUB; ++sub) {
            if (nb * BOX_ROWS == C::TK) {  // a whole tile: one box per 128-key block
#pragma unroll
              for (int kb = 0; kb < C::KB; ++kb) {
                tma_load_3d(st + C::K_OFF + sub * C::SUBK + kb * SUB, &map_kf, sub * 64, cur.k0() + kb * BN, kv_row,
                            &kv_full[s], pol_kv);
                tma_load_3d(st + C::V_OFF + sub * C::SUBK + kb * SUB, &map_vf, sub * 64, cur.k0() + kb * BN, kv_row,
                            &kv_full[s], pol_kv);
              }
            } else {
              for (int b = 0; b < nb; ++b) {
                tma_load_3d(st + C::K_OFF + sub * C::SUBK + b * BOX_ROWS * 128, &map_k, sub * 64,
                            cur.k0() + b * BOX_ROWS, kv_row, &kv_full[s], pol_kv);
                tma_load_3d(st + C::V_OFF + sub * C::SUBK + b * BOX_ROWS * 128, &map_v, sub * 64,
                            cur.k0() + b * BOX_ROWS, kv_row, &kv_full[s], pol_kv);
              }
            }
            tma_load_3d(st + C::Q_OFF + sub * QSUB, &map_q, sub * 64, cur.a * p.H_q + cur.g * p.G, 0, &kv_full[s],
                        pol_q);
          }
        }
        if (*abort_flag) {
          volatile int none = 0;
          for (int t = it - C::NS < 0 ? 0 : it - C::NS; t < it; ++t)
            mbar_wait_bounded(&kv_full[t % C::NS], (t / C::NS) & 1, &none, nullptr);
        }
      } else {
        // The segment's raw query tile is loaded ahead of its first K/V tile,
        // on its own barrier, into ring slot kseg % QR once the S MMAs of
        // segment kseg - QR are done; the prep warp rotates it in place,
        // usually before the K/V tile lands.  The tile that holds the new key lands on
        // the segment's own barrier (last_full), which the prep warp waits for
        // before patching the key in (kv_full of a stage could be several
        // phases ahead of it); kv_full[s] gets a plain arrival so its phases
        // stay in step, and the MMA warp waits for the patch instead.
        int it = 0, kseg = -1;
        int nk_recent = -1;  // the most recent segment whose new-key tile was issued
        int q_recent = -1;   // the most recent segment whose query tile was issued
        for (; cur.more(); cur.advance(), ++it) {
          const int s = it % C::NS;
          if (cur.first()) ++kseg;
          if (it >= C::NS && !mbar_wait_bounded(&kv_empty[s], ((it / C::NS) - 1) & 1, abort_flag, p.status)) break;
          const bool load_q = cur.first();
          if (load_q && kseg >= C::QR &&
              !mbar_wait_bounded(&q_free[kseg % C::QR], (kseg / C::QR - 1) & 1, abort_flag, p.status))
            break;
          const int nb = (cur.nt() + BOX_ROWS - 1) / BOX_ROWS;
          const uint32_t bytes = static_cast<uint32_t>(C::NSUB) * (2u * nb * BOX_ROWS * 128u);
          unsigned char* st = smem + s * C::STAGE;
          unsigned char* qb = smem + C::QB_OFF + (kseg % C::QR) * C::QBUF;
          const int kv_row = p.cache_rows[cur.a] * p.H_kv + cur.g;
          if (load_q) {
            uint64_t* qbar = &q_full[kseg % C::QR];
            mbar_arrive_expect_tx(qbar, static_cast<uint32_t>(C::NSUB) * QSUB);
            for (int sub = 0; sub < C::NSUB; ++sub)
              tma_load_3d(qb + sub * QSUB, &map_q, sub * 64, cur.a * p.H_q + cur.g * p.G, 0, qbar, pol_q);
            q_recent = kseg;
          }
          const bool newkey_tile = cur.last() && cur.x_end == cur.n;
          uint64_t* bar = newkey_tile ? &last_full[kseg % C::QR] : &kv_full[s];
          mbar_arrive_expect_tx(bar, bytes);
          if (newkey_tile) {
            mbar_arrive(&kv_full[s]);
            nk_recent = kseg;
          }
          for (int sub = 0; sub < C::NSUB; ++sub) {
            if (nb * BOX_ROWS == C::TK) {  // a whole tile: one box per 128-key block
#pragma unroll
              for (int kb = 0; kb < C::KB; ++kb) {
                tma_load_3d(st + C::K_OFF + sub * C::SUBK + kb * SUB, &map_kf, sub * 64, cur.k0() + kb * BN, kv_row,
                            bar, pol_kv);
                tma_load_3d(st + C::V_OFF + sub * C::SUBK + kb * SUB, &map_vf, sub * 64, cur.k0() + kb * BN, kv_row,
                            bar, pol_kv);
              }
            } else {
              for (int b = 0; b < nb; ++b) {
                tma_load_3d(st + C::K_OFF + sub * C::SUBK + b * BOX_ROWS * 128, &map_k, sub * 64,
                            cur.k0() + b * BOX_ROWS, kv_row, bar, pol_kv);
                tma_load_3d(st + C::V_OFF + sub * C::SUBK + b * BOX_ROWS * 128, &map_v, sub * 64,
                            cur.k0() + b * BOX_ROWS, kv_row, bar, pol_kv);
              }
            }
          }
        }
        if (*abort_flag) {
          volatile int none = 0;
          for (int t = it - C::NS < 0 ? 0 : it - C::NS; t < it; ++t)
            mbar_wait_bounded(&kv_full[t % C::NS], (t / C::NS) & 1, &none, nullptr);
          // the new-key tiles still in flight belong to the last (at most NS)
          // new-key segments, which are consecutive
          for (int k = nk_recent; k >= 0 && k > nk_recent - C::NS; --k)
            mbar_wait_bounded(&last_full[k % C::QR], (k / C::QR) & 1, &none, nullptr);
          // and the query tiles of the last (at most QR) segments
          for (int k = q_recent; k >= 0 && k > q_recent - C::QR; --k)
            mbar_wait_bounded(&q_full[k % C::QR], (k / C::QR) & 1, &none, nullptr);
        }
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_f16kind_f32(E::kMmaFormat, BN, NQ, 0, 0);
      constexpr uint32_t IDESC_O = idesc_f16kind_f32(E::kMmaFormat, BN, NQ, 0, 1);
      constexpr uint32_t V_LBO = D == 128 ? C::SUBK : 0;  // D = 64: the second M half repeats the first
      const uint32_t p_addr = sbase + C::P_OFF;
      bool issued = false;
      // S^T of tile t, its K/V (and query) tile already landed.  Attention call: the query tile rides in the tile's
      // stage.  Fused step: it is ring slot kq % QR of segment kq, rotated by
      // the prep warp; the slot is released after the segment's last S, and a
      // tile that holds the new key waits for the prep warp's patch.
      auto issue_s_ready = [&](int t, int kq, bool seg_first, bool seg_last, bool new_key) -> bool {
        if constexpr (FUSED) {
          if (seg_first && !mbar_wait_bounded(&prep_done[kq % C::QR], (kq / C::QR) & 1, abort_flag, p.status))
            return false;
          if (new_key && !mbar_wait_bounded(&patch_done[kq % C::QR], (kq / C::QR) & 1, abort_flag, p.status))
            return false;
        }
        tc_fence_after();
        const uint32_t st = sbase + (t % C::NS) * C::STAGE;
        const uint32_t qb = FUSED ? sbase + C::QB_OFF + (kq % C::QR) * C::QBUF : st + C::Q_OFF;
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {  // one M = 128 MMA chain per block of 128 keys
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t koff = (ks / 4) * C::SUBK + kb * SUB + (ks % 4) * 32;
            const uint32_t qoff = (ks / 4) * QSUB + (ks % 4) * 32;
            umma_f16_ss(tmem + ((t & 1) * C::KB + kb) * NQ, smem_desc_sw128(st + C::K_OFF + koff, 16, 1024),
                        smem_desc_sw128(qb + qoff, 16, 1024), IDESC_S, ks > 0);
          }
        }
        umma_commit(&s_full[t & 1]);
        if constexpr (FUSED) {
          if (seg_last) umma_commit(&q_free[kq % C::QR]);
        }
        issued = true;
        return true;
      };
      auto issue_s = [&](int t, int kq, bool seg_first, bool seg_last, bool new_key) -> bool {
        if (!mbar_wait_bounded(&kv_full[t % C::NS], (t / C::NS) & 1, abort_flag, p.status)) return false;
        return issue_s_ready(t, kq, seg_first, seg_last, new_key);
      };
      int it = 0, kseg = -1;
      bool s_next = false;  // S of the next tile is still to be issued (its tile was late)
      int s_kq = 0;
      bool s_first = false, s_last = false, s_key = false;
      for (; cur.more(); cur.advance(), ++it) {
        if (cur.first()) ++kseg;
        if (it == 0 && !issue_s(0, 0, true, cur.last(), cur.last() && cur.x_end == cur.n)) break;
        // another tile follows: overlap its S with this softmax (the next
        // segment's facts are needed only when this tile ends a segment)
        if (cur.has_next()) {
          bool n_last, n_key;
          if (!cur.last()) {
            n_last = cur.x_end - (cur.x + cur.nt()) <= C::TK;
            n_key = n_last && cur.x_end == cur.n;
          } else {
            Cursor<C::TK> nx = cur;
            nx.advance();
            n_last = nx.last();
            n_key = n_last && nx.x_end == nx.n;
          }
          // Issued now only if its tile has landed; otherwise after this
          // tile's P.V, which is not held up behind the copy (a late P.V
          // delays the refill of its stage and the end of a segment).
          // (The attention call only: the whole step's early-start and fused
          // forms measured faster issuing S first.)
          constexpr bool kDeferLateS = !EARLY && !FUSED;
          if (!kDeferLateS) {
            if (!issue_s(it + 1, cur.last() ? kseg + 1 : kseg, cur.last(), n_last, n_key)) break;
          } else if (mbar_test(&kv_full[(it + 1) % C::NS], ((it + 1) / C::NS) & 1)) {
            if (!issue_s_ready(it + 1, cur.last() ? kseg + 1 : kseg, cur.last(), n_last, n_key)) break;
          } else {
            s_next = true;
            s_kq = cur.last() ? kseg + 1 : kseg;
            s_first = cur.last();
            s_last = n_last;
            s_key = n_key;
          }
        }
        if (!mbar_wait_bounded(&p_full[it & 1], (it >> 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t v_addr = sbase + (it % C::NS) * C::STAGE + C::V_OFF;
        const uint32_t pb_addr = p_addr + (it & 1) * C::PBUF;
        const uint32_t acc0 = cur.first() ? 0u : 1u;
#pragma unroll
        for (int ks = 0; ks < C::TK / 16; ++ks) {
          umma_f16_ss(tmem + C::O_COL, smem_desc_sw128(v_addr + ks * 2048, V_LBO, 1024),
                      smem_desc_sw128(pb_addr + (ks / 4) * QSUB + (ks % 4) * 32, 16, 1024), IDESC_O,
                      ks > 0 ? 1u : acc0);
        }
        umma_commit(&o_done[it & 1]);
        umma_commit(&kv_empty[it % C::NS]);
        if (s_next) {
          s_next = false;
          if (!issue_s(it + 1, s_kq, s_first, s_last, s_key)) break;
        }
      }
      if (*abort_flag && issued) {
        umma_commit(drain);
        volatile int none = 0;
        mbar_wait_bounded(drain, 0, &none, nullptr);
      }
    }
  } else if (FUSED && warp == 6) {
    // ---------------------------------------------------------- query / cell prep (fused step)
    // Per segment of this CTA, in order: rotate the group's G raw query rows
    // (loaded ahead of the segment's first tile into query buffer k % QR,
    // 128B swizzled, K-major) in place at the row's position; and if this CTA
    // holds the segment's last key, rotate the new K, store it with the new V
    // into the row's cell at that position, and write the same row into the
    // last K/V tile in shared memory (the TMA loaded the stale cell).  Lane l
    // owns the frequency pairs j = l + 32u.
    if constexpr (FUSED) {
      constexpr int HALF = D / 2;
      constexpr int NU = HALF / 32;
      auto cell = [&](unsigned char* base, int row, int c) -> uint16_t* {  // 128B-swizzled [rows][64] sub-tiles
        const int cc = c & 63, chunk = cc >> 3;
        return reinterpret_cast<uint16_t*>(base + (row * 128 + ((chunk ^ (row & 7)) << 4) + (cc & 7) * 2));
      };
      // cos/sin depend on the row's position only: the KV heads of one row
      // are consecutive segments, so they are evaluated (the costly part)
      // once per row, not once per segment.
      CosSin cs[NU];
      int cs_row = -1, t_first = 0;
      for (int k = 0; cur.more(); ++k) {
        const int b = k % C::QR, ph = (k / C::QR) & 1;
        const int pos = nkeys[cur.a] - 1;
        Cursor<C::TK> c = cur;  // find the segment's last tile in this CTA
        int t_last = t_first;
        while (!c.last()) { c.advance(); ++t_last; }
        const bool new_key = cur.x_end == cur.n;
        const size_t src_off = (static_cast<size_t>(cur.a) * p.H_kv + cur.g) * D;
        uint16_t kn[2 * NU], vn[D / 32];
        if (new_key) {  // issue the loads of the new K/V early
#pragma unroll
          for (int u = 0; u < NU; ++u) {
            kn[2 * u] = p.k_new[src_off + lane + 32 * u];
            kn[2 * u + 1] = p.k_new[src_off + lane + 32 * u + HALF];
          }
#pragma unroll
          for (int e = 0; e < D / 32; ++e) vn[e] = p.v_new[src_off + lane + 32 * e];
        }
        if (cur.a != cs_row) {
#pragma unroll
          for (int u = 0; u < NU; ++u)
            cs[u] = rope_cos_sin(pos, p.freqs.frac[lane + 32 * u], p.freqs.quad[lane + 32 * u]);
          cs_row = cur.a;
        }
        // the raw query tile, on its own barrier
        if (!__all_sync(FULL, mbar_wait_bounded(&q_full[b], ph, abort_flag, p.status))) break;
        unsigned char* qb = smem + C::QB_OFF + b * C::QBUF;
        for (int h = 0; h < p.G; ++h) {
#pragma unroll
          for (int u = 0; u < NU; ++u) {
            const int j = lane + 32 * u;
            uint16_t* c1 = cell(qb + (j >> 6) * QSUB, h, j);
            uint16_t* c2 = cell(qb + ((j + HALF) >> 6) * QSUB, h, j + HALF);
            const float x1 = E::to_f32(*c1), x2 = E::to_f32(*c2);
            *c1 = E::from_f32(rot_first(x1, x2, cs[u]));
            *c2 = E::from_f32(rot_second(x1, x2, cs[u]));
          }
        }
        fence_proxy_async_smem();  // the query tile is read by the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(&prep_done[b]);
        if (new_key) {
          uint16_t kr[2 * NU];
#pragma unroll
          for (int u = 0; u < NU; ++u) {
            const float x1 = E::to_f32(kn[2 * u]), x2 = E::to_f32(kn[2 * u + 1]);
            kr[2 * u] = E::from_f32(rot_first(x1, x2, cs[u]));
            kr[2 * u + 1] = E::from_f32(rot_second(x1, x2, cs[u]));
          }
          const size_t cell_off = ((static_cast<size_t>(p.cache_rows[cur.a]) * p.H_kv + cur.g) * p.max_seq + pos) * D;
#pragma unroll
          for (int u = 0; u < NU; ++u) {
            p.k_cache_w[cell_off + lane + 32 * u] = kr[2 * u];
            p.k_cache_w[cell_off + lane + 32 * u + HALF] = kr[2 * u + 1];
          }
#pragma unroll
          for (int e = 0; e < D / 32; ++e) p.v_cache_w[cell_off + lane + 32 * e] = vn[e];
          // the last tile (rows k0.. of this segment) holds the stale cell at row pos - k0
          if (!__all_sync(FULL, mbar_wait_bounded(&last_full[b], ph, abort_flag, p.status))) break;
          const int row = pos - c.k0();
          unsigned char* st = smem + (t_last % C::NS) * C::STAGE;
#pragma unroll
          for (int u = 0; u < NU; ++u) {
            const int j = lane + 32 * u;
            *cell(st + C::K_OFF + (j >> 6) * C::SUBK, row, j) = kr[2 * u];
            *cell(st + C::K_OFF + ((j + HALF) >> 6) * C::SUBK, row, j + HALF) = kr[2 * u + 1];
          }
#pragma unroll
          for (int e = 0; e < D / 32; ++e) {
            const int j = lane + 32 * e;
            *cell(st + C::V_OFF + (j >> 6) * C::SUBK, row, j) = vn[e];
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&patch_done[b]);
        }
        t_first = t_last + 1;
        cur.advance_segment();
      }
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------- softmax (warps 0-3)
    const int r = threadIdx.x;  // key row of the tile == TMEM lane == d of O^T
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // Per-warp maxima of a tile, in one of two buffers by tile parity: a warp
    // writes tile t+2's into the buffer of tile t only after passing tile
    // t+1's exchange, which every warp reaches after reading tile t's.
    float* red_max2 = reinterpret_cast<float*>(smem + C::RED_OFF);
    float* red_sum = red_max2 + 2 * 4 * NQ;
    unsigned char* pt0 = smem + C::P_OFF;
    // m_ref: the reference maximum of each head (the same in every thread);
    // l: this thread's share of each head's row sum (its keys' weights), all
    // rescaled together and summed over the CTA once, at the segment end.
    float m_ref[GP], l[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) { m_ref[h] = -INFINITY; l[h] = 0.f; }
    int it = 0;
    for (; cur.more(); cur.advance(), ++it) {
      const int nt = cur.nt();
      const bool first = cur.first();
      if (!__all_sync(FULL, mbar_wait_bounded(&s_full[it & 1], (it >> 1) & 1, abort_flag, p.status))) break;
      tc_fence_after();
      // key kb * 128 + r of the tile, for each 128-key block kb
      uint32_t u[C::KB][16];
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) tmem_ld16(tmem + lane_base + ((it & 1) * C::KB + kb) * NQ, u[kb]);
      tmem_wait_ld();
      float* red_max = red_max2 + (it & 1) * 4 * NQ;
      float x[C::KB][GP], mt[GP];
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        float xm = -INFINITY;
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
          x[kb][h] = (kb * BN + r < nt && h < p.G) ? __uint_as_float(u[kb][h]) * p.scale_log2 : -INFINITY;
          xm = fmaxf(xm, x[kb][h]);
        }
        float m;  // the warp's maximum in one instruction
        asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(xm));
        if (lane == 0) red_max[warp * NQ + h] = m;
      }
      named_bar_sync(1, BN);
      bool grow_any = false;
      float alpha[GP];
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        mt[h] = fmaxf(fmaxf(red_max[h], red_max[NQ + h]), fmaxf(red_max[2 * NQ + h], red_max[3 * NQ + h]));
        const bool grow = mt[h] > m_ref[h] + 8.f || first;
        alpha[h] = 1.f;
        if (grow) {
          const float mn = first ? mt[h] : fmaxf(m_ref[h], mt[h]);
          alpha[h] = first ? 0.f : exp2f(m_ref[h] - mn);
          m_ref[h] = mn;
          grow_any |= !first;
        }
        l[h] = first ? 0.f : l[h] * alpha[h];
      }
      // P^T buffer it&1 was last read by the P.V of tile it-2; an O^T rescale
      // needs the P.V of tile it-1 to be complete.
      if (it > 1 && !__all_sync(FULL, mbar_wait_bounded(&o_done[it & 1], ((it - 2) >> 1) & 1, abort_flag, p.status))) break;
      if (grow_any && it > 0 &&
          !__all_sync(FULL, mbar_wait_bounded(&o_done[(it - 1) & 1], ((it - 1) >> 1) & 1, abort_flag, p.status)))
        break;
      tc_fence_after();
      if (grow_any) {  // uniform across the CTA: every thread saw the same maxima
        uint32_t o[16];
        tmem_ld16(tmem + lane_base + C::O_COL, o);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < GP; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
        tmem_st16(tmem + lane_base + C::O_COL, o);
        tmem_wait_st();
      }
      // P^T[h][key] in the storage type (K-major B operand: 16 rows of TK keys in
      // 64-key swizzled sub-tiles); padded heads and invalid keys are zero.
      const int chunk = (r & 63) >> 3, e = r & 7;
      unsigned char* pt = pt0 + (it & 1) * C::PBUF;
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) {
        const int sub = (kb * BN + r) >> 6;
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
          uint16_t b = 0;
          if (h < GP) {
            const float pv = x[kb][h] == -INFINITY ? 0.f : exp2f(x[kb][h] - m_ref[h]);
            b = E::from_f32(pv);
            l[h] += E::to_f32(b);  // the weight P.V actually uses
          }
          *reinterpret_cast<uint16_t*>(pt + sub * QSUB + h * 128 + ((chunk ^ (h & 7)) << 4) + e * 2) = b;
        }
        if (kb * BN + r >= nt) {  // rows past the tile's keys: zero V so P = 0 meets no stale NaN
          unsigned char* vrow = smem + (it % C::NS) * C::STAGE + C::V_OFF + (kb * BN + r) * 128;
#pragma unroll
          for (int sb = 0; sb < C::NSUB; ++sb)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(vrow + sb * C::SUBK + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      // Each warp's P^T stores and TMEM reads are done and fenced before it
      // synchronises; then one lane arrives (four arrivals in all, instead
      // of a CTA-wide barrier or 128 serialised ones).
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[it & 1]);

      if (cur.last()) {
        // ---------------------------------------------------- segment end
        // the row sums of the whole segment part: summed over the CTA's keys
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          float ps = l[h];
#pragma unroll
          for (int off = 16; off; off >>= 1) ps += __shfl_xor_sync(FULL, ps, off);
          if (lane == 0) red_sum[warp * NQ + h] = ps;
        }
        named_bar_sync(1, BN);
#pragma unroll
        for (int h = 0; h < GP; ++h)
          l[h] = (red_sum[h] + red_sum[NQ + h]) + (red_sum[2 * NQ + h] + red_sum[3 * NQ + h]);
        if (!__all_sync(FULL, mbar_wait_bounded(&o_done[it & 1], (it >> 1) & 1, abort_flag, p.status))) break;
        tc_fence_after();
        uint32_t o[16];
        tmem_ld16(tmem + lane_base + C::O_COL, o);
        tmem_wait_ld();
        const int d = r;
        if (d < D) {
          if (cur.whole()) {
            uint16_t* dst = p.out + (static_cast<size_t>(cur.a) * p.H_q + cur.g * p.G) * D + d;
#pragma unroll
            for (int h = 0; h < GP; ++h)
              if (h < p.G) dst[h * D] = E::from_f32(__uint_as_float(o[h]) / l[h]);
          } else {
            float* slotp = p.partials + static_cast<size_t>(blockIdx.x * 2 + cur.slot()) * slot_floats(GP, D);
#pragma unroll
            for (int h = 0; h < GP; ++h) slotp[h * D + d] = __uint_as_float(o[h]);
            if (d < GP) {
#pragma unroll
              for (int h = 0; h < GP; ++h)
                if (h == d) {
                  slotp[GP * D + h] = m_ref[h];
                  slotp[slot_l_offset(GP, D) + h] = l[h];
                }
            }
          }
        }
        if (!cur.whole()) {
          // Count this CTA's partial; the CTA that completes the count merges.
          const int b0 = cur.vlo / W, b1 = (cur.vlo + cur.n - 1) / W;
          int* cnt = p.counters + cur.a * p.H_kv + cur.g;
          // The barrier orders every thread's partial stores before thread 0's
          // release-acquire count; the merging CTA's acquire makes the other
          // CTAs' partials visible, and the next barrier hands that on.
          named_bar_sync(1, BN);
          if (r == 0) *merge_flag = atomic_add_acq_rel_gpu(cnt, 1) == b1 - b0;
          named_bar_sync(1, BN);
          if (*merge_flag) {
            combine_segment<D, GP>(p, cur.a, cur.g, b0, b1, r);
            if (r == 0) *cnt = 0;  // ready for the next call
          }
          named_bar_sync(1, BN);  // merge_flag is reused at the next segment end
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, C::TMEM_COLS);
}

cudaError_t make_decode_maps(const DecodeParams& p, DecodeMaps* m) {
  auto enc = tma_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t D = p.D;
  cuuint64_t dims[3] = {D, static_cast<cuuint64_t>(p.max_seq), static_cast<cuuint64_t>(p.S) * p.H_kv};
  cuuint64_t strides[2] = {D * 2, D * 2 * static_cast<cuuint64_t>(p.max_seq)};
  cuuint32_t es[3] = {1, 1, 1};
  for (int t = 0; t < 4; ++t) {
    cuuint32_t bx[3] = {64, t < 2 ? static_cast<cuuint32_t>(BOX_ROWS) : static_cast<cuuint32_t>(BN), 1};
    CUtensorMap* dst = t == 0 ? &m->kc : t == 1 ? &m->vc : t == 2 ? &m->kcf : &m->vcf;
    if (enc(dst, kTmaElem, 3, const_cast<uint16_t*>((t & 1) == 0 ? p.k_cache : p.v_cache), dims, strides, bx, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Queries as rows of D; a group reads 16 rows (its G heads, then padding
  // that is never used; rows past the tensor read as zeros).
  cuuint64_t qdims[3] = {D, static_cast<cuuint64_t>(p.A) * p.H_q, 1};
  cuuint64_t qstrides[2] = {D * 2, D * 2 * static_cast<cuuint64_t>(p.A) * p.H_q};
  cuuint32_t qbox[3] = {64, NQ, 1};
  if (enc(&m->q, kTmaElem, 3, const_cast<uint16_t*>(p.q), qdims, qstrides, qbox, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

template <int D, int GP>
struct Kernels {
  static cudaError_t prepare(int device, int* num_ctas) {
    static std::once_flag flags[64];
    static cudaError_t errs[64];
    static int ctas[64];
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::call_once(flags[device], [&]() {
      errs[device] = cudaFuncSetAttribute(flash_decode_splitk_kernel<D, GP, false, false>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, false>::SMEM);
      if (errs[device] == cudaSuccess)
        errs[device] = cudaFuncSetAttribute(flash_decode_splitk_kernel<D, GP, false, true>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, false>::SMEM);
      if (errs[device] == cudaSuccess)
        errs[device] = cudaFuncSetAttribute(flash_decode_splitk_kernel<D, GP, true, false>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, true>::SMEM);
      int sms = 0;
      if (errs[device] == cudaSuccess)
        errs[device] = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
      ctas[device] = sms;  // one CTA per SM (the shared-memory ring fills an SM)
    });
    *num_ctas = ctas[device];
    return errs[device];
  }
  template <bool FUSED, bool EARLY>
  static cudaError_t launch_mode(const DecodeParams& p, const DecodeMaps& m, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_ctas);
    cfg.blockDim = dim3(threads_of(FUSED));
    cfg.dynamicSmemBytes = Cfg<D, FUSED>::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, flash_decode_splitk_kernel<D, GP, FUSED, EARLY>, p, m.kc, m.vc, m.q, m.kcf, m.vcf);
  }
  static cudaError_t launch(const DecodeParams& p, const DecodeMaps& m, cudaStream_t stream) {
    if (p.fused) return launch_mode<true, false>(p, m, stream);
    return p.early ? launch_mode<false, true>(p, m, stream) : launch_mode<false, false>(p, m, stream);
  }
};

template <typename F>
cudaError_t dispatch(int D, int GP, F&& f) {
  if (D == 128) {
    switch (GP) {
      case 1: return f(Kernels<128, 1>{});
      case 2: return f(Kernels<128, 2>{});
      case 4: return f(Kernels<128, 4>{});
      case 8: return f(Kernels<128, 8>{});
      case 16: return f(Kernels<128, 16>{});
    }
  } else if (D == 64) {
    switch (GP) {
      case 1: return f(Kernels<64, 1>{});
      case 2: return f(Kernels<64, 2>{});
      case 4: return f(Kernels<64, 4>{});
      case 8: return f(Kernels<64, 8>{});
      case 16: return f(Kernels<64, 16>{});
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace

#if KVGQA_DECODE_F16
cudaError_t launch_cached_gqa_attention_f16(const DecodeParams& p, cudaStream_t stream) {
  DecodeMaps m;
  cudaError_t e = make_decode_maps(p, &m);
  if (e != cudaSuccess) return e;
  const int GP = decode_group_pad(p.G);
  int device = 0, n = 0;
  e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  return dispatch(p.D, GP, [&](auto k) {
    const cudaError_t pe = decltype(k)::prepare(device, &n);
    return pe != cudaSuccess ? pe : decltype(k)::launch(p, m, stream);
  });
}
#else
int decode_group_pad(int G) {
  int gp = 1;
  while (gp < G) gp <<= 1;
  return gp;
}

cudaError_t decode_layout(int device, int D, int GP, int64_t A, int64_t H_kv, DecodeLayout* out) {
  int n = 0;
  const cudaError_t e = dispatch(D, GP, [&](auto k) { return decltype(k)::prepare(device, &n); });
  if (e != cudaSuccess) return e;
  out->num_ctas = n;
  out->counter_bytes = (static_cast<size_t>(A) * H_kv * sizeof(int32_t) + 255) / 256 * 256;
  out->partial_bytes = static_cast<size_t>(n) * 2 * slot_floats(GP, D) * sizeof(float);
  return cudaSuccess;
}

// Scratch for callers that cannot allocate device memory themselves: the
// split-K partials (and the status word in front of them) live in this
// file-scope device array instead of a caller workspace.  Every GPU that
// loads the library holds it until the process exits; all calls share it.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

cudaError_t static_scratch_address(int device, void** ptr) {
  static std::once_flag flags[64];
  static void* addr[64];
  static cudaError_t errs[64];
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  // Runs once per device, with that device current (the caller's current device).
  std::call_once(flags[device], [&] { errs[device] = cudaGetSymbolAddress(&addr[device], g_static_scratch); });
  *ptr = addr[device];
  return errs[device];
}

cudaError_t launch_cached_gqa_attention(const DecodeParams& p, cudaStream_t stream) {
  if (p.A == 0) return cudaSuccess;
  if (p.f16) return launch_cached_gqa_attention_f16(p, stream);
  DecodeMaps m;
  const cudaError_t e = make_decode_maps(p, &m);
  if (e != cudaSuccess) return e;
  const int GP = decode_group_pad(p.G);
  return dispatch(p.D, GP, [&](auto k) { return decltype(k)::launch(p, m, stream); });
}
#endif  // KVGQA_DECODE_F16

}  // namespace kvgqa
