// K4: causal GQA attention of the equal-length prefill, on tcgen05 tensor
// cores with the accumulators in tensor memory.
//
// microLLM-rocm ARCHITECTURE.md, section "Tensor ownership boundary": equal-
// length pending prompts run as one batch and each prefix is mapped into its
// target empty shared-cache row; section "Attention layout boundary": Q/K/V
// leave the projection token-major (BTHD) and context is written back
// token-major; with GQA one K/V head serves G query heads without expansion.
// The rotated K and V have already been stored into the target cache rows
// (K1), so this kernel reads them straight from the cache.
//
// A persistent grid (one CTA per SM) walks items (128-query tile qt, prompt a,
// pair of query heads of one KV group), longest first, dealt round-robin.
// Both heads of a pair read the same K/V tiles, so each tile staged in shared
// memory feeds four MMAs.  Per item:
//   warp 8      TMA: the two Q tiles, then 128-key K tiles (2-stage ring);
//   warp 9      TMA: the matching V tiles (2-stage ring);
//   warp 10     one thread issues tcgen05.mma: S_x = Q_x K^T into TMEM and
//               O_x += P_x V with P_x read from TMEM (x = A, B);
//   warps 0-3   softmax of head A, warps 4-7 softmax of head B, one thread
//               per query row: S row from TMEM, scale and causal mask (on the
//               tiles that reach past the row's query), FP32 online softmax, P
//               in the storage type written back over the S columns, O
//               rescaled in TMEM only when the row maximum grew by more than
//               2^8 (otherwise the old base is kept; O / l stays exact); at the
//               item end O / l is rounded to the storage type, staged in shared
//               memory per warp and stored by the TMA unit.
// While one head's softmax group works on its scores, the MMAs of the other
// head run.  MMAs issued by one thread complete in order and a commit covers
// every earlier MMA, so S_x of tile t being ready means P_x of tile t-1 has
// been consumed.
// Key tiles past the diagonal are never visited; tensor maps bound the key and
// query ranges by T so rows past the prompt read as zeros.  With an odd group
// size, items hold one head (the B group idles).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "kvgqa_internal.h"
#include "elem.cuh"
#include "tcgen05.cuh"

namespace kvgqa {
namespace {

constexpr int BM = 128;        // query rows per tile
constexpr int BN = 128;        // keys per tile
static_assert(BM == kPrefillTile && BN == kPrefillTile, "the varlen item order counts tiles of this size");
constexpr int SUB = 16384;     // one [128 rows x 64 16-bit values] swizzled sub-tile
constexpr int NWARPS = 12;     // 2 x 4 softmax + Q/K producer + V producer + MMA + spare
constexpr int THREADS = NWARPS * 32;
constexpr int W_QK = 8, W_V = 9, W_MMA = 10;
// Register split (setmaxnreg): the launch gives every thread kLaunchRegs; the
// third warpgroup (producers, MMA issuer) drops to kRoleRegs so the two
// softmax warpgroups can rise to kSoftmaxRegs and hold a whole score row.
// The sum stays within the launch's registers (checked on the host against
// the compiled kernel before every launch).
constexpr int kLaunchRegs = 168, kRoleRegs = 72, kSoftmaxRegs = 216;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kRoleRegs <= THREADS * kLaunchRegs, "register split");
constexpr int TMEM_COLS = 512; // S_A, S_B, O_A, O_B: 128 columns each
constexpr unsigned FULLMASK = 0xffffffffu;

template <int D>
struct PCfg {
  static constexpr int NSUB = D / 64;               // 64-wide sub-tiles per row
  static constexpr int TILE = NSUB * SUB;           // one Q, K or V tile
  static constexpr int NK = D == 128 ? 2 : 4;       // K stages
  static constexpr int NV = D == 128 ? 2 : 4;       // V stages
  static constexpr int Q_OFF = 0;                   // Q_A, Q_B
  static constexpr int K_OFF = 2 * TILE;
  static constexpr int V_OFF = K_OFF + NK * TILE;
  // Output staging: one [32 rows x 64 values] 128B-swizzled box per softmax
  // warp, written by the warp and stored by the TMA unit.
  static constexpr int STG = 32 * 128;
  static constexpr int STG_OFF = V_OFF + NV * TILE;
  static constexpr int BAR_OFF = STG_OFF + 8 * STG;
  // q_full[2], q_empty[2], k_full[NK], k_empty[NK], v_full[NV], v_empty[NV],
  // s_full[2], p_full[2], o_done[2], drain (index [2] = head A / B)
  static constexpr int NBAR = 4 + 2 * NK + 2 * NV + 7;
  static constexpr int SLOT_OFF = BAR_OFF + NBAR * 8;
  static constexpr int FLAG_OFF = SLOT_OFF + 8;
  static constexpr int SMEM = FLAG_OFF + 16 + 1024;  // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct PrefillMaps {
  CUtensorMap q;  // [A][T][H_q][D] rotated queries
  CUtensorMap k;  // cache [S*H_kv][T(bounded)][D]
  CUtensorMap v;
  CUtensorMap o;  // [A][T][H_q][D] output, box of 32 rows x 64 values
};


template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// One lane of a converged warp (the same one every lane agrees on).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Maximum of three values (one instruction on sm_100 and later; NaN inputs
// are ignored like fmaxf does).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// One 32-byte store (eight 32-bit words, a whole sector) to global memory,
// 32-byte aligned, marked as streaming (written once, not read again here).
// Each softmax thread writes its own output row, so a warp's 16-byte stores
// would each fill half of 32 different sectors: whole sectors halved the
// cost of the item epilogue's stores.
__device__ __forceinline__ void stg256_stream(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// 2^x on the special-function unit (flushes results below 2^-126 to zero,
// which no 16-bit probability needs).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The work of the persistent grid: items (query tile qt, prompt a, head pair),
// longest first (by query tile for the equal-length prefill, by the item
// order the store kernel wrote for prompts at offsets; query tile qt of
// prompt a covers queries [qt*BM, qt*BM+BM)
// at positions off_a + t and visits the key tiles up to its last query's
// position), dealt in snake order (round k gives item k*grid + b to CTA b on
// even rounds and to CTA grid-1-b on odd ones, which evens out the sums of a
// list sorted longest first much better than plain round-robin); every role
// of a CTA walks the same sequence,
// key tile by key tile.  Prompt a holds len_a tokens at positions
// off_a .. off_a+len_a-1 of its row (the equal-length prefill: off 0, len T).
struct TileWalk {
  const PrefillParams* p;     // the launch's parameters (read in place)
  int i;                      // current item index
  int cta, grid, round;       // this CTA, the grid size, the dealing round of item i
  int qt, a, hA, hB, kv_row;  // current item (hB < 0: single head)
  int off, len, nkt, kend;    // its prompt's offset and length, its key tiles, its last key + 1
  int j;                      // key tile within the item
  bool ok;                    // false past the last item

  // Two heads of one KV group per item when G is even.
  __device__ __forceinline__ bool pairs() const { return (p->G % 2) == 0; }
  __device__ __forceinline__ int per_tok() const { return pairs() ? p->H_q / 2 : p->H_q; }
  __device__ __forceinline__ int units() const { return p->A * per_tok(); }
  __device__ __forceinline__ int n_items() const { return (p->T + BM - 1) / BM * units(); }
  // Prompt a of item i.
  __device__ __forceinline__ int prompt_of(int item) const {
    return p->item_order ? p->item_order[item / per_tok()] % p->A : item % units() / per_tok();
  }

  __device__ bool load_item() {
    const int nqt = (p->T + BM - 1) / BM, u = units(), pt = per_tok(), n = nqt * u;
    while (i < n) {
      int k;
      if (p->item_order) {  // prompts at offsets: pairs (qt, a) longest first, then the head pairs
        const int c = p->item_order[i / pt];
        qt = c / p->A;
        a = c % p->A;
        k = i % pt;
      } else {              // equal length: query tiles from the last (longest) down
        qt = nqt - 1 - i / u;
        const int rem = i % u;
        a = rem / pt;
        k = rem % pt;
      }
      hA = pairs() ? 2 * k : k;
      hB = pairs() ? 2 * k + 1 : -1;
      const int r = p->cache_rows[a];
      const int o = p->offsets ? p->offsets[a] : 0;
      const int L = p->lengths ? p->lengths[a] : p->T;
      const bool meta_ok = L >= 0 && L <= p->T && o >= 0 && o <= p->max_seq - L;
      if (r >= 0 && r < p->S && meta_ok && qt * BM < L) {
        off = o;
        len = L;
        const int q_end = min(L, qt * BM + BM);
        kend = o + q_end;
        nkt = (kend + BN - 1) / BN;  // key tiles holding positions 0 .. kend - 1
        kv_row = r * p->H_kv + hA / p->G;
        j = 0;
        return true;
      }
      // prompts with an invalid row or metadata are skipped (and flagged by
      // the store kernel); query tiles past a prompt's length have no work
      next_index();
    }
    return false;
  }
  __device__ __forceinline__ void next_index() {
    ++round;
    i = round * grid + ((round & 1) ? grid - 1 - cta : cta);
  }
  __device__ void init(const PrefillParams* params, int first, int step) {
    p = params;
    cta = first;
    grid = step;
    round = 0;
    i = first;
    ok = load_item();
  }
  __device__ __forceinline__ bool first_tile() const { return j == 0; }
  __device__ __forceinline__ bool last_tile() const { return j == nkt - 1; }
  // First cache position of the key tile: j * BN, except that with prompts at
  // offsets a last tile reaching past kend is moved back to end at kend, so
  // it reads no cell past the prompt (those may hold anything, and a zero
  // weight times a NaN is still a NaN); its columns before j * BN were
  // covered by tile j - 1 and are masked.  (The equal-length prefill's
  // key map ends at T, so its positions past the prompt read as zeros.)
  __device__ __forceinline__ int kstart() const {
    return (p->offsets && j == nkt - 1 && (j + 1) * BN > kend) ? kend - BN : j * BN;
  }
  // Query row r of the tile sees key column c iff
  // mask_lo() <= c <= mask_base() + r.
  __device__ __forceinline__ int mask_base() const { return off + qt * BM - kstart(); }
  __device__ __forceinline__ int mask_lo() const { return j * BN - kstart(); }
  __device__ void advance() {
    if (j < nkt - 1) { ++j; return; }
    next_index();
    ok = load_item();
  }
};

template <int D, bool F16>
__global__ void __launch_bounds__(THREADS, 1)
prefill_attention_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                         const __grid_constant__ CUtensorMap map_o) {
  using C = PCfg<D>;
  using E = Elem<F16>;  // storage type of Q, K, V, P and the output
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;       // [head]
  uint64_t* q_empty = bars + 2;  // [head]
  uint64_t* k_full = bars + 4;
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* v_full = k_empty + C::NK;
  uint64_t* v_empty = v_full + C::NV;
  uint64_t* s_full = v_empty + C::NV;  // [head]
  uint64_t* p_full = s_full + 2;       // [head]
  uint64_t* o_done = p_full + 2;       // [head]
  uint64_t* drain = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::SLOT_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::FLAG_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Launched behind the store kernel with programmatic dependent launch: the
  // CTA starts while the store's last CTAs drain and waits here before it
  // reads anything that kernel writes (the item order, the rotated queries
  // and the cache cells).
  pdl_wait();
  TileWalk walk;
  walk.init(&p, blockIdx.x, gridDim.x);
  if (!walk.ok) {  // uniform: this CTA has no valid item
    if (threadIdx.x == 0) {
      for (int i = blockIdx.x; i < walk.n_items(); i += gridDim.x) {
        const int r = p.cache_rows[walk.prompt_of(i)];
        if (r < 0 || r >= p.S) { atomicOr(p.status, KVGQA_FLAG_ROW_RANGE); break; }
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_full[x], 1);
      mbar_init(&q_empty[x], 1);
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 4);  // one arrival per softmax warp
      mbar_init(&o_done[x], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  if (warp >= 8) {
  regs_dec<kRoleRegs>();
  if (warp == W_QK) {
    // ------------------------------------------------------------ Q and K producer
    if (lane == 0) {
      const uint64_t pol_q = l2_evict_first_policy();
      const uint64_t pol_kv = l2_evict_last_policy();  // K/V tiles are re-read by the group's heads
      for (int i = blockIdx.x; i < walk.n_items(); i += gridDim.x) {
        const int r = p.cache_rows[walk.prompt_of(i)];
        if (r < 0 || r >= p.S) { atomicOr(p.status, KVGQA_FLAG_ROW_RANGE); break; }
      }
      // Per item: Q_A, the first K tile, Q_B (the order the MMAs need them).
      int it = 0, qa = 0, qb = 0;  // K tiles and Q tiles (per head) loaded so far
      auto load_q = [&](int x, int& qn) -> bool {
        if (qn >= 1 && !mbar_wait_bounded(&q_empty[x], (qn - 1) & 1, abort_flag, p.status)) return false;
        mbar_arrive_expect_tx(&q_full[x], BM * D * 2);
        for (int sub = 0; sub < C::NSUB; ++sub)
          tma_load_4d(smem + C::Q_OFF + x * C::TILE + sub * SUB, &map_q, sub * 64, x ? walk.hB : walk.hA,
                      walk.qt * BM, walk.a, &q_full[x], pol_q);
        ++qn;
        return true;
      };
      for (; walk.ok; walk.advance()) {
        const bool fresh = walk.first_tile();
        if (fresh && !load_q(0, qa)) break;
        const int s = it % C::NK;
        if (it >= C::NK && !mbar_wait_bounded(&k_empty[s], ((it / C::NK) - 1) & 1, abort_flag, p.status)) break;
        unsigned char* st = smem + C::K_OFF + s * C::TILE;
        mbar_arrive_expect_tx(&k_full[s], BN * D * 2);
        for (int sub = 0; sub < C::NSUB; ++sub)
          tma_load_3d(st + sub * SUB, &map_k, sub * 64, walk.kstart(), walk.kv_row, &k_full[s], pol_kv);
        ++it;
        if (fresh && walk.hB >= 0 && !load_q(1, qb)) break;
      }
      if (*abort_flag) {
        volatile int none = 0;
        if (qa >= 1) mbar_wait_bounded(&q_full[0], (qa - 1) & 1, &none, nullptr);
        if (qb >= 1) mbar_wait_bounded(&q_full[1], (qb - 1) & 1, &none, nullptr);
        for (int t = it - C::NK < 0 ? 0 : it - C::NK; t < it; ++t)
          mbar_wait_bounded(&k_full[t % C::NK], (t / C::NK) & 1, &none, nullptr);
      }
    }
  } else if (warp == W_V) {
    // ------------------------------------------------------------ V producer
    if (lane == 0) {
      const uint64_t pol_kv = l2_evict_last_policy();
      int it = 0;
      for (; walk.ok; walk.advance()) {
        const int s = it % C::NV;
        if (it >= C::NV && !mbar_wait_bounded(&v_empty[s], ((it / C::NV) - 1) & 1, abort_flag, p.status)) break;
        unsigned char* st = smem + C::V_OFF + s * C::TILE;
        mbar_arrive_expect_tx(&v_full[s], BN * D * 2);
        for (int sub = 0; sub < C::NSUB; ++sub)
          tma_load_3d(st + sub * SUB, &map_v, sub * 64, walk.kstart(), walk.kv_row, &v_full[s], pol_kv);
        ++it;
      }
      if (*abort_flag) {
        volatile int none = 0;
        for (int t = it - C::NV < 0 ? 0 : it - C::NV; t < it; ++t)
          mbar_wait_bounded(&v_full[t % C::NV], (t / C::NV) & 1, &none, nullptr);
      }
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop (uniform control flow); one elected
    // lane issues each group of MMAs and its commits.
    {
      constexpr uint32_t IDESC_QK = idesc_f16kind_f32(E::kMmaFormat, BM, BN, 0);
      constexpr uint32_t IDESC_PV = idesc_f16kind_f32(E::kMmaFormat, BM, D, 1);
      const bool pairs = walk.pairs();
      const int nh = pairs ? 2 : 1;
      bool issued = false;
      int qn = 0;             // items whose Q tiles have been consumed
      TileWalk ahead = walk;  // the tile whose S is issued next
      bool ok = true;
      bool first_next = true; // first-tile flag of the newest tile whose S was issued
      // Returns whether every lane's wait succeeded (a timeout anywhere stops the warp).
#define KVGQA_WAIT(bar, parity) (ok = ok && __all_sync(FULLMASK, mbar_wait_bounded((bar), (parity), abort_flag, p.status)))
      for (int t = -1; ok; ++t) {
        // ---- P.V of tile t (t >= 0) interleaved with S of tile t + 1, head by head.
        // The K tile of tile t + 1 is waited for before the first P.V so that no
        // wait separates the groups (the tensor pipe's queue is short; a stalled
        // issuer leaves it idle).
        const bool first = first_next, more = ahead.ok;
        const int sv = t % C::NV, kn = (t + 1) % C::NK;
        if (t >= 0) KVGQA_WAIT(&v_full[sv], (t / C::NV) & 1);
        if (more) KVGQA_WAIT(&k_full[kn], ((t + 1) / C::NK) & 1);
        const uint32_t v_addr = sbase + C::V_OFF + sv * C::TILE;
        const uint32_t k_addr = sbase + C::K_OFF + kn * C::TILE;
        const bool a_first = ahead.first_tile(), a_last = ahead.last_tile();
        for (int x = 0; x < nh && ok; ++x) {
          if (t >= 0) {
            // O_x += P_x V, P_x read from TMEM over S_x's first half
            KVGQA_WAIT(&p_full[x], t & 1);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
#pragma unroll
              for (int ks = 0; ks < BN / 16; ++ks)
                umma_f16_ts(tmem + (2 + x) * BN, tmem + x * BN + ks * 8, smem_desc_sw128(v_addr + ks * 2048, SUB, 1024),
                            IDESC_PV, (ks > 0 || !first) ? 1u : 0u);
              umma_commit(&o_done[x]);
              if (x == nh - 1) umma_commit(&v_empty[sv]);
            }
            __syncwarp();
          }
          if (more) {
            // S_x = Q_x K^T of tile t + 1; the last head frees the K stage, and
            // after an item's last tile Q_x is freed, once the MMAs complete
            if (a_first) KVGQA_WAIT(&q_full[x], qn & 1);
            if (!ok) break;
            tc_fence_after();
            const uint32_t q_addr = sbase + C::Q_OFF + x * C::TILE;
            if (elect_one()) {
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t off = (ks / 4) * SUB + (ks % 4) * 32;
                umma_f16_ss(tmem + x * BN, smem_desc_sw128(q_addr + off, 16, 1024),
                            smem_desc_sw128(k_addr + off, 16, 1024), IDESC_QK, ks > 0);
              }
              umma_commit(&s_full[x]);
              if (a_last) umma_commit(&q_empty[x]);
              if (x == nh - 1) umma_commit(&k_empty[kn]);
            }
            __syncwarp();
            issued = true;
          }
        }
        if (!more) break;
        first_next = a_first;
        if (a_first) ++qn;
        ahead.advance();
      }
#undef KVGQA_WAIT
      if (*abort_flag && issued) {
        // let every MMA issued so far finish before TMEM is released
        if (elect_one()) umma_commit(drain);
        __syncwarp();
        volatile int none = 0;
        mbar_wait_bounded(drain, 0, &none, nullptr);
      }
    }
  }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    regs_inc<kSoftmaxRegs>();
    const int x = warp >> 2;           // head of the pair this group serves
    const int r = threadIdx.x & 127;   // query row in the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_base + x * BN;
    const uint32_t o_col = tmem + lane_base + (2 + x) * BN;
    const float c = p.scale_log2;
    const float ce = c > 0.f ? c : 1.f;
    float m_ref = -INFINITY, l = 0.f;
    for (int t = 0; walk.ok; ++t, walk.advance()) {
      if (x == 1 && walk.hB < 0) continue;  // single-head item: the B group has nothing to do
      const bool first = walk.first_tile(), last = walk.last_tile();
      const int mbase = walk.mask_base(), mlo = walk.mask_lo();
      if (!__all_sync(FULLMASK, mbar_wait_bounded(&s_full[x], t & 1, abort_flag, p.status))) break;
      tc_fence_after();
      // Scores enter the softmax as s * ce with ce > 0 (a non-positive scale is
      // folded into the scores first, a path no usual caller takes).  On the
      // tiles that reach past a query's position (the diagonal), keys after
      // the query become -inf, so they weigh zero.  Every query sees key 0 in
      // tile 0; a later tile may hold no key a row sees (with offsets), and
      // then the row's maximum stays and its weights there are zero.
      uint32_t u[BN];
#pragma unroll
      for (int q = 0; q < BN / 32; ++q) tmem_ld32(s_col + q * 32, *reinterpret_cast<uint32_t(*)[32]>(u + q * 32));
      tmem_wait_ld();
      float* sv = reinterpret_cast<float*>(u);
      if (c <= 0.f) {
#pragma unroll
        for (int i = 0; i < BN; ++i) sv[i] *= c;
      }
      if (mlo > 0) {  // a moved last tile: a band
        const int thr = mbase + r;
#pragma unroll
        for (int i = 0; i < BN; ++i) sv[i] = (i >= mlo && i <= thr) ? sv[i] : -INFINITY;
      } else if (mbase < BN - 1) {
        const int thr = mbase + r;
#pragma unroll
        for (int i = 0; i < BN; ++i) sv[i] = i <= thr ? sv[i] : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = fmaxf(sv[2 * k], sv[2 * k + 1]);
#pragma unroll
      for (int i = 16; i < BN; i += 16) {
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = fmax3(mx[k], sv[i + 2 * k], sv[i + 2 * k + 1]);
      }
      const float mraw = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      const float mt = mraw * ce;                    // tile maximum of the scaled scores
      const bool grow = first || mt > m_ref + 8.f;   // keep the old base unless it grew by 2^8
      float alpha = 1.f;
      if (grow) {
        alpha = first ? 0.f : ex2(m_ref - mt);
        m_ref = mt;
        l *= alpha;
      }
      // S_x of this tile being ready means the P.V of the previous tile is
      // complete, so O_x may be rescaled here without a further wait.
      if (__any_sync(FULLMASK, grow && !first)) {
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t u[32];
          tmem_ld32(o_col + q * 32, u);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
          tmem_st32(o_col + q * 32, u);
        }
      }
      // P as pairs of the storage type over the first 64 columns of S_x (the A
      // operand of P.V, which must have V's type).
      float2 ls = make_float2(0.f, 0.f);
      const float2 c2 = make_float2(ce, ce), nm2 = make_float2(-m_ref, -m_ref);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int i0 = half * 64 + 2 * e;
          const float2 xx = ffma2(make_float2(sv[i0], sv[i0 + 1]), c2, nm2);
          const float2 pr = make_float2(ex2(xx.x), ex2(xx.y));
          ls = fadd2(ls, pr);
          w[e] = E::pack2(pr.x, pr.y);
        }
        tmem_st32(s_col + half * 32, w);
      }
      tmem_wait_st();
      l += ls.x + ls.y;
      // Each warp arrives once (128 single-thread arrivals on one barrier
      // serialise): every lane's TMEM stores are complete (wait::st) and
      // fenced before the warp synchronises, then lane 0 arrives.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&p_full[x]);
      }

      if (last) {
        // ---------------------------------------------------- item epilogue
        if (!__all_sync(FULLMASK, mbar_wait_bounded(&o_done[x], t & 1, abort_flag, p.status))) break;
        tc_fence_after();
        const int tq = walk.qt * BM + r;
        const float inv = 1.f / l;
        const int h = x ? walk.hB : walk.hA;
        // This warp's 32 rows go out through shared memory and a TMA store
        // (coalesced, and off the softmax's path) when all of them lie inside
        // the prompt; in a query tile that reaches past the prompt's end the
        // rows take direct stores, and those past the end stay unwritten.
        const int row0 = walk.qt * BM + (warp & 3) * 32;
        const bool via_tma = row0 + 32 <= walk.len;
        unsigned char* stg = smem + C::STG_OFF + warp * C::STG;
        uint16_t* dst = p.out + ((static_cast<size_t>(walk.a) * p.T + tq) * p.H_q + h) * D;
#pragma unroll
        for (int sub = 0; sub < C::NSUB; ++sub) {  // 64 output values of the row at a time
          uint32_t u[64];
          tmem_ld32(o_col + sub * 64, *reinterpret_cast<uint32_t(*)[32]>(u));  // warp-wide
          tmem_ld32(o_col + sub * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
          tmem_wait_ld();
          uint32_t w[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) w[k] = E::pack2(__uint_as_float(u[2 * k]) * inv, __uint_as_float(u[2 * k + 1]) * inv);
          if (via_tma) {
            if (lane == 0) bulk_wait_group_read<0>();  // the previous store has read the buffer
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c)  // 16-byte chunk c of row `lane` at its 128B-swizzled place
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                  make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_4d(&map_o, stg, sub * 64, h, row0, walk.a);
              bulk_commit_group();
            }
          } else if (tq < walk.len) {
#pragma unroll
            for (int q16 = 0; q16 < 4; ++q16) {  // 16 values: a whole 32-byte sector
              uint16_t* o = dst + sub * 64 + q16 * 16;
              const uint32_t(&w8)[8] = *reinterpret_cast<const uint32_t(*)[8]>(w + 8 * q16);
              if (p.out_32b) {
                stg256_stream(o, w8);
              } else {
                *reinterpret_cast<uint4*>(o) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
                *reinterpret_cast<uint4*>(o + 8) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
              }
            }
          }
        }
      }
    }
  }

  if (warp < 8 && lane == 0) bulk_wait_group<0>();  // this warp's output stores are complete
  __syncwarp();  // the role warps reconverge (their lane 0 worked alone)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

cudaError_t make_maps(const PrefillParams& p, PrefillMaps* m) {
  auto enc = tma_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t D = p.D;
  const CUtensorMapDataType elem_type = p.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  {
    cuuint64_t dims[4] = {D, static_cast<cuuint64_t>(p.H_q), static_cast<cuuint64_t>(p.T),
                          static_cast<cuuint64_t>(p.A)};
    cuuint64_t strides[3] = {D * 2, D * 2 * p.H_q, D * 2 * p.H_q * p.T};
    cuuint32_t box[4] = {64, 1, BM, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&m->q, elem_type, 4, const_cast<uint16_t*>(p.q_rot), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Keys: positions [0, T) of each (slot, kv head) for the equal-length
  // prefill (positions >= T are outside the map and read as zeros), the whole
  // row for prompts at offsets (keys past a query's position are masked).
  const cuuint64_t key_extent = p.offsets ? static_cast<cuuint64_t>(p.max_seq) : static_cast<cuuint64_t>(p.T);
  cuuint64_t dims[3] = {D, key_extent, static_cast<cuuint64_t>(p.S) * p.H_kv};
  cuuint64_t strides[2] = {D * 2, D * 2 * static_cast<cuuint64_t>(p.max_seq)};
  cuuint32_t box[3] = {64, BN, 1};
  cuuint32_t es[3] = {1, 1, 1};
  if (enc(&m->k, elem_type, 3, const_cast<uint16_t*>(p.k_cache), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (enc(&m->v, elem_type, 3, const_cast<uint16_t*>(p.v_cache), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  {
    cuuint64_t odims[4] = {D, static_cast<cuuint64_t>(p.H_q), static_cast<cuuint64_t>(p.T),
                           static_cast<cuuint64_t>(p.A)};
    cuuint64_t ostrides[3] = {D * 2, D * 2 * p.H_q, D * 2 * p.H_q * p.T};
    cuuint32_t obox[4] = {64, 1, 32, 1};
    cuuint32_t oes[4] = {1, 1, 1, 1};
    if (enc(&m->o, elem_type, 4, p.out, odims, ostrides, obox, oes, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <int D, bool F16>
cudaError_t launch_d(const PrefillParams& p, const PrefillMaps& m, cudaStream_t stream) {
  static std::once_flag flags[64];
  static cudaError_t errs[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(flags[dev], [&] {
    errs[dev] = cudaFuncSetAttribute(prefill_attention_kernel<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     PCfg<D>::SMEM);
    // The in-kernel register split needs the launch to hand out kLaunchRegs
    // per thread; with fewer, setmaxnreg.inc could never be satisfied.
    cudaFuncAttributes attr;
    if (errs[dev] == cudaSuccess) errs[dev] = cudaFuncGetAttributes(&attr, prefill_attention_kernel<D, F16>);
    if (errs[dev] == cudaSuccess && attr.numRegs < kLaunchRegs) errs[dev] = cudaErrorInvalidConfiguration;
  });
  if (errs[dev] != cudaSuccess) return errs[dev];
  static int sms[64];
  static std::once_flag sm_flags[64];
  std::call_once(sm_flags[dev], [&] {
    if (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms[dev] = 0;
  });
  if (sms[dev] <= 0) return cudaErrorInvalidDevice;
  const int per_tok = p.G % 2 == 0 ? p.H_q / 2 : p.H_q;  // head pairs when the group size is even
  const long long items = static_cast<long long>((p.T + BM - 1) / BM) * p.A * per_tok;
  const unsigned grid = static_cast<unsigned>(items < sms[dev] ? items : sms[dev]);  // one CTA per SM
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = PCfg<D>::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_attention_kernel<D, F16>, p, m.q, m.k, m.v, m.o);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tma_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

cudaError_t launch_prefill_attention(const PrefillParams& params, cudaStream_t stream) {
  if (params.A == 0 || params.T == 0) return cudaSuccess;
  PrefillParams p = params;
  p.out_32b = reinterpret_cast<uintptr_t>(p.out) % 32 == 0;  // every output row then starts on 32 bytes too
  PrefillMaps m;
  cudaError_t e = make_maps(p, &m);
  if (e != cudaSuccess) return e;
  if (p.D == 128) return p.f16 ? launch_d<128, true>(p, m, stream) : launch_d<128, false>(p, m, stream);
  if (p.D == 64) return p.f16 ? launch_d<64, true>(p, m, stream) : launch_d<64, false>(p, m, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvgqa
