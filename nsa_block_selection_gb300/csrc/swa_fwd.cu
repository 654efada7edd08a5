// GQA sliding-window attention forward for sm_103a on the 5th-generation
// tensor cores (tcgen05 MMAs, accumulators in tensor memory, TMA operands).
//
// Operation ("[Kernel][MI350] Add 8 wave GQA sliding-window attention
// kernel", sections "Summary" and "What it does"): grouped-query attention,
// H / H_kv consecutive query heads per KV head; dense, or with a
// (LEFT, RIGHT) window: query i attends to keys [i - LEFT, i + RIGHT]
// (a negative side is unbounded); online softmax; bf16 (or fp16) in and out,
// head dim 64 or 128. Q [B,M,H,D], K and V [B,N,H_kv,D], O [B,M,H,D],
// optional LSE [B,H,M] (natural log, fp32).
//
// Two kernels. With an even number of query heads per KV head,
// swa_fwd_pair_kernel (below) takes two heads per work item, one softmax
// warpgroup each, so that one head's exponentials overlap the other head's
// MMAs. Otherwise (an odd number) swa_fwd_kernel:
// one CTA per (b, head, tile of 128 queries); 6 warps with fixed roles:
//  * warp 0, one lane: TMA producer. Loads the Q tile once and streams the
//    K and V tiles of 128 keys that the window of the query tile touches
//    through a 3-stage ring (each tile two 128B-swizzled boxes of 64 dims);
//  * warp 1: allocates 512 tensor-memory columns; one lane issues the MMAs:
//    S_i = Q K_i^T (M = 128 queries, N = 128 keys, K = D; both operands
//    K-major) into one of two S buffers, then O += P_i V_i (M = 128,
//    N = D, K = 128 keys; P from tensor memory, V MN-major straight from
//    its [keys][D] tile). The order is S_0, S_1, PV_0, S_2, PV_1, ... so the
//    softmax of one tile overlaps the QK^T of the next;
//  * warps 2-5: softmax, one thread per query row (a warp reads the
//    tensor-memory lanes of its quarter). Each reads its row of S_i, masks
//    it on edge tiles, keeps a reference max that moves only when a score
//    exceeds it by more than 8 (log2 units; O in tensor memory is then
//    rescaled in place, after the previous PV has completed), writes
//    P = 2^(x - ref) rounded to the input type into one of two tensor-memory
//    P buffers (two 16-bit values per column) and arrives on its barrier:
//    with two buffers the exponentials of tile i overlap both the PV of
//    tile i - 1 and the QK^T of tile i + 1. Keeping P out of shared memory
//    leaves room for the third K/V stage, which the L2 latency needs at
//    full MMA rate. The epilogue reads O, divides by the row sum and stores
//    the row and its LSE.
// Every mbarrier wait is bounded (1 s); a role that gives up sets the status
// word and leaves its loop, so every role reaches the teardown, which frees
// the tensor memory.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "nsa_sel_attn.h"
#include "ptx.cuh"
#include "sel_attn_fwd.cuh"
#include "status.cuh"
#include "tc.cuh"

namespace nsa {
namespace {

constexpr int kSwaQ = 128;     // queries per work item (MMA M)
constexpr int kSwaKeys = 128;  // keys per tile
constexpr int kSwaThreads = 192;
constexpr uint32_t kSwaTmemCols = 512;
constexpr uint32_t kColS = 0;    // S buffers at columns 0 and 128
constexpr uint32_t kColO = 256;  // D columns
constexpr uint32_t kColP = 384;  // two P buffers of 64 columns (128 keys, 16-bit pairs)
constexpr float kSwaSlack = 8.0f;

// One barrier per ring slot / buffer, so that no barrier can complete twice
// before its waiter has seen the first completion. Tiles are counted across
// the CTA's work items (g); Q buffers and the O accumulator by work item (n).
enum SwaBar : int {
  kQFull = 0,    // 2 Q buffers
  kQEmpty = 2,   // 2: every QK^T of the item that used Q buffer b has completed
  kKFull = 4,    // 2 K stages
  kKEmpty = 6,   // 2
  kVFull = 8,    // 2 V stages
  kVEmpty = 10,  // 2
  kSFull = 12,   // 2 S buffers (tensor memory)
  kPFull = 14,   // 2 P buffers (tensor memory)
  kPvDone = 16,  // 2: PV of the tile that used P buffer b has completed
  kOEmpty = 18,     // the softmax warps have read O of the previous item
  kOStaged = 19,    // the softmax warps have written this item's O tile to shared memory
  kOSmemFree = 20,  // the previous item's O tile store has read shared memory
  kNumBars = 21
};

template <int D>
struct SwaCfg {
  static constexpr int kAtoms = D / 64;                 // 64-element swizzle columns
  static constexpr int kAtomBytes = kSwaQ * 128;         // 128 rows x 128 B
  static constexpr int kQBytes = kSwaQ * D * 2;          // one Q buffer
  static constexpr int kKVBytes = kSwaKeys * D * 2;      // one K (or V) stage
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQBytes;
  static constexpr int kOffV = kOffK + 2 * kKVBytes;
  static constexpr int kOffO = kOffV + 2 * kKVBytes;  // O tile, staged for a TMA store
  static constexpr int kOffBar = kOffO + kQBytes;
  static constexpr int kOffTmem = kOffBar + kNumBars * 8;
  // at least 116 KB so that one CTA holds an SM (all 512 tensor-memory columns)
  static constexpr int kUsed = kOffTmem + 16 + 1024;
  static constexpr int kSmemBytes = kUsed > 118784 ? kUsed : 118784;
};

struct SwaProblem {
  void* O;  // [B, M, H, D] in the inputs' type (read by the head-pair kernel)
  float* LSE;
  int B, M, N, H, Hkv, hpg, qtiles;
  int left, right;  // clamped to [0, M + N]: M + N is unbounded in effect
  float sl2;        // scale * log2(e)
  int64_t items;    // B * H * qtiles
  bool o32;         // O 32-byte aligned: 32-byte stores of O rows (head-pair kernel)
};

// One work item: a tile of 128 queries of one head, and the keys its
// windows touch, in whole tiles of 128.
struct SwaItem {
  int b, g, h, q0, q_last, t0, nt, in_lo, in_hi;
};

// Items in the order (b, KV head, query tile, head within the group), the
// head fastest: the CTAs working at the same time share K/V tiles in L2.
// items < 2^31 (host check): 32-bit arithmetic.
__device__ __forceinline__ SwaItem swa_item(const SwaProblem& p, int64_t item) {
  SwaItem it;
  uint32_t x = static_cast<uint32_t>(item);
  const int hh = static_cast<int>(x % static_cast<uint32_t>(p.hpg));
  x /= static_cast<uint32_t>(p.hpg);
  const int qt = static_cast<int>(x % static_cast<uint32_t>(p.qtiles));
  x /= static_cast<uint32_t>(p.qtiles);
  it.g = static_cast<int>(x % static_cast<uint32_t>(p.Hkv));
  it.b = static_cast<int>(x / static_cast<uint32_t>(p.Hkv));
  it.h = it.g * p.hpg + hh;
  it.q0 = qt * kSwaQ;
  it.q_last = min(it.q0 + kSwaQ, p.M) - 1;
  const int jlo = max(0, it.q0 - p.left);
  const int jhi = min(p.N - 1, it.q_last + p.right);
  it.t0 = jlo / kSwaKeys;
  it.nt = jhi >= jlo ? jhi / kSwaKeys - it.t0 + 1 : 0;
  // keys every row of the item sees (tiles inside need no mask)
  it.in_lo = max(0, it.q_last - p.left);
  it.in_hi = min(p.N - 1, it.q0 + p.right);
  return it;
}

// Per-warpgroup register budget (all four warps of a warpgroup execute it).
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N) : "memory");
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return pack2_t<BF16>(lo, hi);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kSwaThreads, 1)
    swa_fwd_kernel(const SwaProblem p, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmO) {
  using C = SwaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);  // generic pointer to `base`
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  auto bar = [&](int i) { return base + C::kOffBar + 8u * static_cast<uint32_t>(i); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kQFull + s), 1);
      mbar_init(bar(kQEmpty + s), 1);
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 1);
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kPFull + s), 4 * 32);
      mbar_init(bar(kPvDone + s), 1);
    }
    mbar_init(bar(kOEmpty), 4 * 32);
    mbar_init(bar(kOStaged), 4 * 32);
    mbar_init(bar(kOSmemFree), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc_alloc(base + C::kOffTmem, kSwaTmemCols);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kOffTmem);
  bool failed = false;
  // Work items are dealt in rounds of gridDim.x, in snake order (the
  // direction reverses every round) so that no CTA takes the same position
  // -- the same query-tile offset, the same amount of work -- in every round.
  const int64_t nrounds = (p.items + gridDim.x - 1) / gridDim.x;
  auto item_of = [&](int64_t k) -> int64_t {
    const int64_t pos = (k & 1) ? gridDim.x - 1 - blockIdx.x : blockIdx.x;
    return k * gridDim.x + pos;  // may be >= p.items in the last round
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer ----
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t once = l2_policy_evict_first();
      int64_t gt = 0;  // tiles loaded so far
      int n = 0;       // items with keys so far
      for (int64_t k = 0; k < nrounds && !failed; ++k) {
        const int64_t x = item_of(k);
        if (x >= p.items) continue;
        const SwaItem it = swa_item(p, x);
        if (it.nt == 0) continue;
        const int qb = n & 1;
        if (n >= 2 && !wait_phase(bar(kQEmpty + qb), ((n - 2) >> 1) & 1, kWaitLimitNs)) {
          failed = true;
          break;
        }
        mbar_arrive_expect_tx(bar(kQFull + qb), C::kQBytes);
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_4d(base + C::kOffQ + qb * C::kQBytes + a * C::kAtomBytes, &tmQ,
                      bar(kQFull + qb), a * 64, it.h, it.q0, it.b, once);
        for (int i = 0; i < it.nt; ++i) {
          const int64_t gi = gt + i;
          const int s = static_cast<int>(gi & 1);
          const uint32_t prev = static_cast<uint32_t>(((gi - 2) >> 1) & 1);
          const int j0 = (it.t0 + i) * kSwaKeys;
          if (gi >= 2 && !wait_phase(bar(kKEmpty + s), prev, kWaitLimitNs)) {
            failed = true;
            break;
          }
          mbar_arrive_expect_tx(bar(kKFull + s), C::kKVBytes);
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_4d(base + C::kOffK + s * C::kKVBytes + a * C::kAtomBytes, &tmK,
                        bar(kKFull + s), a * 64, it.g, j0, it.b, keep);
          if (gi >= 2 && !wait_phase(bar(kVEmpty + s), prev, kWaitLimitNs)) {
            failed = true;
            break;
          }
          mbar_arrive_expect_tx(bar(kVFull + s), C::kKVBytes);
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_4d(base + C::kOffV + s * C::kKVBytes + a * C::kAtomBytes, &tmV,
                        bar(kVFull + s), a * 64, it.g, j0, it.b, keep);
        }
        gt += it.nt;
        ++n;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: the tiles of all items as one stream ----
      constexpr uint32_t idesc_s = umma_idesc_f16(kSwaQ, kSwaKeys, BF16, false);
      constexpr uint32_t idesc_o = umma_idesc_f16(kSwaQ, D, BF16, true);
      auto issue_s = [&](int64_t gi, int qb) -> bool {
        const int s = static_cast<int>(gi & 1);
        if (!wait_phase(bar(kKFull + s), static_cast<uint32_t>((gi >> 1) & 1), kWaitLimitNs))
          return false;
        tc_fence_after();
        const uint32_t d = tmem + kColS + static_cast<uint32_t>(s) * kSwaKeys;
        const uint32_t qbase = base + C::kOffQ + qb * C::kQBytes;
        const uint32_t kb = base + C::kOffK + s * C::kKVBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * C::kAtomBytes + (k & 3) * 32;
          tc_mma(d, umma_desc_sw128(qbase + off, 16), umma_desc_sw128(kb + off, 16), idesc_s,
                 k > 0 ? 1u : 0u);
        }
        tc_commit(bar(kKEmpty + s));
        tc_commit(bar(kSFull + s));
        return true;
      };
      // PV of global tile gi; `first`: the item's first tile (O starts from
      // zero, after the softmax warps have read the previous item's O)
      auto issue_pv = [&](int64_t gi, bool first, int n) -> bool {
        const int s = static_cast<int>(gi & 1);  // V stage and P buffer
        const uint32_t ph = static_cast<uint32_t>((gi >> 1) & 1);
        if (!wait_phase(bar(kPFull + s), ph, kWaitLimitNs)) return false;
        if (!wait_phase(bar(kVFull + s), ph, kWaitLimitNs)) return false;
        if (first && n >= 1 && !wait_phase(bar(kOEmpty), (n - 1) & 1, kWaitLimitNs))
          return false;
        tc_fence_after();
        const uint32_t vb = base + C::kOffV + s * C::kKVBytes;
        const uint32_t pcol = tmem + kColP + static_cast<uint32_t>(s) * (kSwaKeys / 2);
#pragma unroll
        for (int kk = 0; kk < kSwaKeys / 16; ++kk)
          tc_mma_ts(tmem + kColO, pcol + 8 * kk, umma_desc_sw128(vb + kk * 2048, C::kAtomBytes),
                    idesc_o, (!first || kk > 0) ? 1u : 0u);
        tc_commit(bar(kVEmpty + s));
        tc_commit(bar(kPvDone + s));
        return true;
      };
      bool ok = true;
      int64_t gt = 0;
      int n = 0;
      int64_t pend = -1;  // global tile whose PV is still to be issued
      bool pend_first = false;
      int pend_n = 0;
      for (int64_t k = 0; k < nrounds && ok; ++k) {
        const int64_t x = item_of(k);
        if (x >= p.items) continue;
        const SwaItem it = swa_item(p, x);
        if (it.nt == 0) continue;
        const int qb = n & 1;
        ok = wait_phase(bar(kQFull + qb), (n >> 1) & 1, kWaitLimitNs);
        for (int i = 0; i < it.nt && ok; ++i) {
          ok = issue_s(gt + i, qb);
          if (ok && i == it.nt - 1) tc_commit(bar(kQEmpty + qb));
          if (ok && pend >= 0) ok = issue_pv(pend, pend_first, pend_n);
          pend = gt + i;
          pend_first = i == 0;
          pend_n = n;
        }
        gt += it.nt;
        ++n;
      }
      if (ok && pend >= 0) ok = issue_pv(pend, pend_first, pend_n);
      failed = !ok;
    }
  } else {
    // ---- softmax (warps 2..5): thread <-> query row of each item ----
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.sl2;
    // waits are decided warp-wide (tcgen05.ld/st are warp-collective)
    auto wait_all = [&](int b, uint32_t parity) {
      return __all_sync(kFull, wait_phase(bar(b), parity, kWaitLimitNs));
    };
    int64_t gt = 0;
    int n = 0;
    int e = 0;  // epilogues (O tiles stored) so far
    for (int64_t k = 0; k < nrounds && !failed; ++k) {
      const int64_t x = item_of(k);
      if (x >= p.items) continue;
      const SwaItem it = swa_item(p, x);
      const int iq = it.q0 + row;
      const int lo_i = max(0, iq - p.left);
      const int hi_i = min(p.N - 1, iq + p.right);
      float ref = -INFINITY, neg = 0.f, l = 0.f;  // ref, neg in the log2 domain
      for (int i = 0; i < it.nt; ++i) {
        const int64_t gi = gt + i;
        const int sb = static_cast<int>(gi & 1);  // S buffer and P buffer of this tile
        if (!wait_all(kSFull + sb, static_cast<uint32_t>((gi >> 1) & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
        uint32_t sr[kSwaKeys];
#pragma unroll
        for (int c = 0; c < kSwaKeys / 32; ++c)
          tc_ld32(lane_addr + kColS + sb * kSwaKeys + 32 * c,
                  *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tc_wait_ld();
        const int j0 = (it.t0 + i) * kSwaKeys;
        if (j0 < it.in_lo || j0 + kSwaKeys - 1 > it.in_hi) {  // edge tile (CTA-uniform)
#pragma unroll
          for (int j = 0; j < kSwaKeys; ++j)
            if (j0 + j < lo_i || j0 + j > hi_i) sr[j] = __float_as_uint(-INFINITY);
        }
        // row max of the raw scores (scale > 0 commutes with max), 8 chains
        float m8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) m8[j] = __uint_as_float(sr[j]);
#pragma unroll
        for (int j = 8; j < kSwaKeys; ++j) m8[j & 7] = fmaxf(m8[j & 7], __uint_as_float(sr[j]));
        const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
        const bool move = mx > ref + kSwaSlack;
        if (__any_sync(kFull, move)) {
          // alpha = 0 while a row has seen nothing (its O row is still 0).
          // O may be rescaled only once the previous tile's PV has completed.
          const float alpha = move ? ex2(ref - mx) : 1.f;
          if (i > 0) {
            if (!wait_all(kPvDone + static_cast<int>((gi - 1) & 1),
                          static_cast<uint32_t>(((gi - 1) >> 1) & 1))) {
              failed = true;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tc_ld32(lane_addr + kColO + 32 * c, o);
              tc_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
              tc_st32(lane_addr + kColO + 32 * c, o);
            }
            tc_wait_st();
          }
          if (move) {
            l *= alpha;
            ref = mx;
            neg = -mx;
          }
        }
        // P buffer sb was last read by the PV of tile gi - 2
        if (gi >= 2 && !wait_all(kPvDone + sb, static_cast<uint32_t>(((gi - 2) >> 1) & 1))) {
          failed = true;
          break;
        }
        // P = 2^(s * scale * log2e - ref) into tensor-memory P buffer sb:
        // column c holds keys 2c (low half) and 2c + 1
        float l8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) l8[j] = 0.f;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t pw[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int j = 64 * h2 + 2 * c;
            const float e0 = ex2(fmaf(__uint_as_float(sr[j]), sl2, neg));
            const float e1 = ex2(fmaf(__uint_as_float(sr[j + 1]), sl2, neg));
            l8[(2 * c) & 7] += e0;
            l8[(2 * c + 1) & 7] += e1;
            pw[c] = pack2<BF16>(e0, e1);
          }
          tc_st32(lane_addr + kColP + sb * (kSwaKeys / 2) + 32 * h2, pw);
        }
        l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kPFull + sb));
      }
      if (failed) break;
      // epilogue: read O into registers and release it to the next item's
      // PVs; normalise, stage the tile in shared memory (128B-swizzled rows)
      // and let one thread store it with TMA; LSE is stored directly
      uint32_t o[D];
      if (it.nt > 0) {
        const int64_t gl = gt + it.nt - 1;
        if (!wait_all(kPvDone + static_cast<int>(gl & 1), static_cast<uint32_t>((gl >> 1) & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          tc_ld32(lane_addr + kColO + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&o[32 * c]));
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(kOEmpty));
      } else {
#pragma unroll
        for (int j = 0; j < D; ++j) o[j] = 0u;
      }
      const bool leader = warp == 2 && lane == 0;
      if (e >= 1) {  // the previous tile's store must have read the staging buffer
        if (leader) {
          bulk_wait_group_read0();
          mbar_arrive(bar(kOSmemFree));
        }
        if (!wait_all(kOSmemFree, static_cast<uint32_t>((e - 1) & 1))) {
          failed = true;
          break;
        }
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint8_t* const orow = gbase + C::kOffO + row * 128;
#pragma unroll
      for (int q = 0; q < D / 8; ++q) {
        uint4 w;
        w.x = pack2<BF16>(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
        w.y = pack2<BF16>(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
        w.z = pack2<BF16>(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
        w.w = pack2<BF16>(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
        *reinterpret_cast<uint4*>(orow + (q >> 3) * C::kAtomBytes + (((q & 7) ^ (row & 7)) << 4)) =
            w;
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kOStaged));
      bool staged = true;
      if (leader) {
        staged = wait_phase(bar(kOStaged), static_cast<uint32_t>(e & 1), kWaitLimitNs);
        if (staged) {
          for (int a = 0; a < C::kAtoms; ++a)
            tma_store_4d(&tmO, base + C::kOffO + a * C::kAtomBytes, a * 64, it.h, it.q0, it.b);
          bulk_commit_group();
        }
      }
      if (!__all_sync(kFull, staged)) failed = true;  // warp-wide, like every other decision
      if (iq < p.M && p.LSE != nullptr) {
        constexpr float kLn2 = 0.69314718055994530942f;
        p.LSE[(static_cast<int64_t>(it.b) * p.H + it.h) * p.M + iq] =
            l > 0.f ? (ref + __log2f(l)) * kLn2 : -INFINITY;
      }
      ++e;
      gt += it.nt;
      if (it.nt > 0) ++n;
    }
  }

  // teardown: every role is here; the O stores have completed; the tensor
  // memory is freed
  if (warp == 2 && lane == 0) bulk_wait_group0();
  if (failed) report_timeout();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, kSwaTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Head-pair variant (hpg even). A
// work item is one tile of 128 queries of two heads of the same KV group:
// both read the same K/V tiles under the same masks. Each head has its own softmax warpgroup, so one
// head's exponentials run while the tensor cores work on the other's tiles:
//   S_A(i), S_B(i), PV_A(i), S_A(i + 1), PV_B(i), S_B(i + 1), PV_A(i + 1) ...
// Tensor memory: S_A at 0, S_B at 128 (P is written over the first 64
// columns of its S once S has been read: the tensor pipe runs the MMAs in
// issue order, so the next S of that head is issued after the PV that reads
// P), O_A at 256, O_B at 256 + D. Shared memory holds one Q pair, so the
// next item's Q waits for the last QK^T of the current one. For long
// windows the softmax warps write O rows straight to global memory; for
// short ones (TMA_O) they stage them in a shared buffer that warp 10 stores
// with TMA tensor stores.
// Warpgroups: 0 softmax and epilogue of head A (warps 0-3), 1 of head B
// (warps 4-7), 2 producer (warp 8), MMA issuer (warp 9), O store warp
// (warp 10, TMA_O) and an idle warp.
// ---------------------------------------------------------------------------

enum SwaPairBar : int {
  kPQFull = 0,     // the Q pair of the item has landed
  kPQEmpty = 1,    // every QK^T of the item has completed
  kPKFull = 2,     // 2 K stages
  kPKEmpty = 4,    // 2
  kPVFull = 6,     // 2 V stages
  kPVEmpty = 8,    // 2
  kPSFull = 10,    // 2 (head A, head B): S of the head's current tile
  kPPFull = 12,    // 2: P written over that S
  kPOFull = 14,    // 2: the item's last PV of the head has completed
  kPOEmpty = 16,   // 2: the head's softmax warps have read its O
  kPOStaged = 18,  // 2 (TMA_O): the head's softmax warps have staged its O tile
  kPOSmemFree = 20,  // (TMA_O) the last O tile store has read the staging buffer
  kPNumBars = 21
};

constexpr int kSwaPairThreads = 384;

// TMA_O: the O tiles go through one shared staging buffer (heads A, B in
// turn) and are written by TMA tensor stores from an otherwise idle warp;
// otherwise each softmax thread stores its own O row. The first pays at
// short windows (many items per key), the second at long ones (it keeps the
// softmax path free of the staging protocol's registers).
template <int D, bool TMA_O>
struct SwaPairCfg {
  static constexpr int kAtoms = D / 64;
  static constexpr int kAtomBytes = kSwaQ * 128;
  static constexpr int kQBytes = kSwaQ * D * 2;      // one head's Q tile
  static constexpr int kKVBytes = kSwaKeys * D * 2;  // one K (or V) stage
  static constexpr int kOffQ = 0;                    // Q_A, Q_B
  static constexpr int kOffK = kOffQ + 2 * kQBytes;
  static constexpr int kOffV = kOffK + 2 * kKVBytes;
  static constexpr int kOffO = kOffV + 2 * kKVBytes;  // (TMA_O) one head's O tile, staged
  static constexpr int kOffBar = kOffO + (TMA_O ? kQBytes : 0);
  static constexpr int kOffTmem = kOffBar + kPNumBars * 8;
  static constexpr int kUsed = kOffTmem + 16 + 1024;
  static constexpr int kSmemBytes = kUsed > 118784 ? kUsed : 118784;
  static_assert(kSmemBytes <= 232448, "fits one SM");
};

// Windows up to this many keys per query tile use the TMA_O variant.
constexpr int64_t kSwaPairTmaOMaxKeys = 1152;

// Item -> (b, KV group, query tile, head pair), the pair fastest.
__device__ __forceinline__ SwaItem swa_item_pair(const SwaProblem& p, int64_t item) {
  const int pairs = p.hpg / 2;
  uint32_t x = static_cast<uint32_t>(item);
  const int pp = static_cast<int>(x % static_cast<uint32_t>(pairs));
  x /= static_cast<uint32_t>(pairs);
  // the same decode as swa_item with the head index 2 pp
  const uint32_t rest = x;  // (b * Hkv + g) * qtiles + qt
  return swa_item(p, static_cast<int64_t>(rest) * p.hpg + 2 * pp);
}

template <int D, bool BF16, bool TMA_O>
__global__ void __launch_bounds__(kSwaPairThreads, 1)
    swa_fwd_pair_kernel(const SwaProblem p, const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO) {
  using C = SwaPairCfg<D, TMA_O>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) { return base + C::kOffBar + 8u * static_cast<uint32_t>(i); };
  if (threadIdx.x == 0) {
    mbar_init(bar(kPQFull), 1);
    mbar_init(bar(kPQEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kPKFull + s), 1);
      mbar_init(bar(kPKEmpty + s), 1);
      mbar_init(bar(kPVFull + s), 1);
      mbar_init(bar(kPVEmpty + s), 1);
      mbar_init(bar(kPSFull + s), 1);
      mbar_init(bar(kPPFull + s), 4 * 32);
      mbar_init(bar(kPOFull + s), 1);
      mbar_init(bar(kPOEmpty + s), 4 * 32);
      mbar_init(bar(kPOStaged + s), 4 * 32);
    }
    mbar_init(bar(kPOSmemFree), 1);
    fence_mbar_init();
  }
  if (warp == 9) {
    tc_alloc(base + C::kOffTmem, kSwaTmemCols);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kOffTmem);
  bool failed = false;
  const int64_t nrounds = (p.items + gridDim.x - 1) / gridDim.x;
  auto item_of = [&](int64_t k) -> int64_t {
    const int64_t pos = (k & 1) ? gridDim.x - 1 - blockIdx.x : blockIdx.x;
    return k * gridDim.x + pos;
  };
  constexpr uint32_t kColSA = 0, kColSB = 128, kColOA = 256, kColOB = 256 + D;

  // Registers: the block starts at 168 a thread; warpgroup 2 gives part of
  // its share to the softmax warpgroups: 128 x (200 + 200 + 104) = 64,512 =
  // 384 x 168, and 200 + 200 + 104 <= 512 per sub-partition (one warp of
  // each warpgroup).
  if (warp >= 8) {
    setmaxnreg_dec<104>();  // every warp of warpgroup 2, converged
    if (warp == 8 && lane == 0) {
      // ---- TMA producer ----
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t once = l2_policy_evict_first();
      int64_t gt = 0;
      int n = 0;
      for (int64_t k = 0; k < nrounds && !failed; ++k) {
        const int64_t x = item_of(k);
        if (x >= p.items) continue;
        const SwaItem it = swa_item_pair(p, x);
        if (it.nt == 0) continue;
        if (n >= 1 && !wait_phase(bar(kPQEmpty), (n - 1) & 1, kWaitLimitNs)) {
          failed = true;
          break;
        }
        mbar_arrive_expect_tx(bar(kPQFull), 2 * C::kQBytes);
        for (int hx = 0; hx < 2; ++hx)
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_4d(base + C::kOffQ + hx * C::kQBytes + a * C::kAtomBytes, &tmQ,
                        bar(kPQFull), a * 64, it.h + hx, it.q0, it.b, once);
        for (int i = 0; i < it.nt; ++i) {
          const int64_t gi = gt + i;
          const int s = static_cast<int>(gi & 1);
          const uint32_t prev = static_cast<uint32_t>(((gi - 2) >> 1) & 1);
          const int j0 = (it.t0 + i) * kSwaKeys;
          if (gi >= 2 && !wait_phase(bar(kPKEmpty + s), prev, kWaitLimitNs)) {
            failed = true;
            break;
          }
          mbar_arrive_expect_tx(bar(kPKFull + s), C::kKVBytes);
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_4d(base + C::kOffK + s * C::kKVBytes + a * C::kAtomBytes, &tmK,
                        bar(kPKFull + s), a * 64, it.g, j0, it.b, keep);
          if (gi >= 2 && !wait_phase(bar(kPVEmpty + s), prev, kWaitLimitNs)) {
            failed = true;
            break;
          }
          mbar_arrive_expect_tx(bar(kPVFull + s), C::kKVBytes);
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_4d(base + C::kOffV + s * C::kKVBytes + a * C::kAtomBytes, &tmV,
                        bar(kPVFull + s), a * 64, it.g, j0, it.b, keep);
        }
        gt += it.nt;
        ++n;
      }
    } else if (warp == 9 && lane == 0) {
      // ---- MMA issuer ----
      constexpr uint32_t idesc_s = umma_idesc_f16(kSwaQ, kSwaKeys, BF16, false);
      constexpr uint32_t idesc_o = umma_idesc_f16(kSwaQ, D, BF16, true);
      // S_X of global tile gi (hx: head 0 = A, 1 = B)
      auto issue_s = [&](int64_t gi, int hx) {
        const int s = static_cast<int>(gi & 1);
        const uint32_t d = tmem + (hx ? kColSB : kColSA);
        const uint32_t qbase = base + C::kOffQ + hx * C::kQBytes;
        const uint32_t kb = base + C::kOffK + s * C::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kAtomBytes + (kk & 3) * 32;
          tc_mma(d, umma_desc_sw128(qbase + off, 16), umma_desc_sw128(kb + off, 16), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(kPSFull + hx));
      };
      int n = 0;  // items with keys so far
      // PV_X of global tile gi (`first`: the item's first tile, O from zero,
      // once the head's softmax warps have read the previous item's O)
      auto issue_pv = [&](int64_t gi, int hx, bool first) -> bool {
        if (first && n >= 1 &&
            !wait_phase(bar(kPOEmpty + hx), static_cast<uint32_t>((n - 1) & 1), kWaitLimitNs))
          return false;
        tc_fence_after();
        const int s = static_cast<int>(gi & 1);
        const uint32_t vb = base + C::kOffV + s * C::kKVBytes;
        const uint32_t pcol = tmem + (hx ? kColSB : kColSA);
        const uint32_t o = tmem + (hx ? kColOB : kColOA);
#pragma unroll
        for (int kk = 0; kk < kSwaKeys / 16; ++kk)
          tc_mma_ts(o, pcol + 8 * kk, umma_desc_sw128(vb + kk * 2048, C::kAtomBytes), idesc_o,
                    (!first || kk > 0) ? 1u : 0u);
        return true;
      };
      auto wait_ok = [&](int b, uint32_t parity) { return wait_phase(bar(b), parity, kWaitLimitNs); };
      bool ok = true;
      int64_t gt = 0;
      for (int64_t k = 0; k < nrounds && ok; ++k) {
        const int64_t x = item_of(k);
        if (x >= p.items) continue;
        const SwaItem it = swa_item_pair(p, x);
        if (it.nt == 0) continue;
        ok = wait_ok(kPQFull, n & 1);
        for (int i = 0; i < it.nt && ok; ++i) {
          const int64_t gi = gt + i;
          const int s = static_cast<int>(gi & 1);
          const uint32_t ph = static_cast<uint32_t>((gi >> 1) & 1);
          ok = wait_ok(kPKFull + s, ph);
          if (!ok) break;
          tc_fence_after();
          // S_A(i) follows PV_A(i - 1) in issue order (it overwrites P_A)
          if (i > 0) {
            ok = wait_ok(kPPFull + 0, static_cast<uint32_t>((gi - 1) & 1)) &&
                 wait_ok(kPVFull + ((gi - 1) & 1), static_cast<uint32_t>(((gi - 1) >> 1) & 1)) &&
                 issue_pv(gi - 1, 0, i == 1);
            if (!ok) break;
          }
          issue_s(gi, 0);
          if (i > 0) {
            ok = wait_ok(kPPFull + 1, static_cast<uint32_t>((gi - 1) & 1)) &&
                 issue_pv(gi - 1, 1, i == 1);
            if (!ok) break;
            tc_commit(bar(kPVEmpty + ((gi - 1) & 1)));
          }
          issue_s(gi, 1);
          tc_commit(bar(kPKEmpty + s));
          if (i == it.nt - 1) tc_commit(bar(kPQEmpty));
        }
        if (!ok) break;
        // the item's last PVs
        const int64_t gl = gt + it.nt - 1;
        for (int hx = 0; hx < 2 && ok; ++hx) {
          ok = wait_ok(kPPFull + hx, static_cast<uint32_t>(gl & 1)) &&
               (hx == 1 || wait_ok(kPVFull + (gl & 1), static_cast<uint32_t>((gl >> 1) & 1))) &&
               issue_pv(gl, hx, it.nt == 1);
          if (!ok) break;
          tc_commit(bar(kPOFull + hx));
        }
        if (ok) tc_commit(bar(kPVEmpty + (gl & 1)));
        gt += it.nt;
        ++n;
      }
      failed = !ok;
    } else if (TMA_O && warp == 10 && lane == 0) {
      // ---- O tile stores: the heads' staged tiles in the order A, B of
      // every item, one TMA tensor store each; the staging buffer is handed
      // back once the store has read it ----
      tma_prefetch_desc(&tmO);
      int ne = 0;  // items so far
      for (int64_t k = 0; k < nrounds && !failed; ++k) {
        const int64_t x = item_of(k);
        if (x >= p.items) continue;
        const SwaItem it = swa_item_pair(p, x);
        for (int hx = 0; hx < 2; ++hx) {
          if (!wait_phase(bar(kPOStaged + hx), static_cast<uint32_t>(ne & 1), kWaitLimitNs)) {
            failed = true;
            break;
          }
          for (int a = 0; a < C::kAtoms; ++a)
            tma_store_4d(&tmO, base + C::kOffO + a * C::kAtomBytes, a * 64, it.h + hx, it.q0, it.b);
          bulk_commit_group();
          bulk_wait_group_read0();
          mbar_arrive(bar(kPOSmemFree));
        }
        ++ne;
      }
      bulk_wait_group0();  // the stores have completed
    }
  } else {
    setmaxnreg_inc<200>();  // every warp of warpgroups 0 and 1, converged
    // ---- softmax and epilogue of head hx (warps 4 hx .. 4 hx + 3) ----
    const int hx = warp >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t col_s = hx ? kColSB : kColSA, col_o = hx ? kColOB : kColOA;
    const float sl2 = p.sl2;
    auto wait_all = [&](int b, uint32_t parity) {
      return __all_sync(kFull, wait_phase(bar(b), parity, kWaitLimitNs));
    };
    int64_t gt = 0;
    int n = 0;   // items with keys so far
    int ne = 0;  // (TMA_O) items so far: O tiles staged by this head
    for (int64_t k = 0; k < nrounds && !failed; ++k) {
      const int64_t x = item_of(k);
      if (x >= p.items) continue;
      const SwaItem it = swa_item_pair(p, x);
      const int h = it.h + hx;
      const int iq = it.q0 + row;
      const int lo_i = max(0, iq - p.left);
      const int hi_i = min(p.N - 1, iq + p.right);
      float ref = -INFINITY, neg = 0.f, l = 0.f;
      for (int i = 0; i < it.nt; ++i) {
        const int64_t gi = gt + i;
        if (!wait_all(kPSFull + hx, static_cast<uint32_t>(gi & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
        uint32_t sr[kSwaKeys];
#pragma unroll
        for (int c = 0; c < kSwaKeys / 32; ++c)
          tc_ld32(lane_addr + col_s + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tc_wait_ld();
        const int j0 = (it.t0 + i) * kSwaKeys;
        // The tile's softmax, compiled twice: interior tiles (every key
        // visible to every row) without any mask code, edge tiles with it.
        auto tile = [&](auto edge_c) {
          // 32-key chunks of an edge tile, decided for the warp's 32 rows at
          // once (the window bounds grow with the row): every key visible to
          // every row, to none, or per element. Keys of empty chunks are
          // neither maximised nor exponentiated (P = 0).
          uint32_t empty = 0u;
          if constexpr (decltype(edge_c)::value) {
            const int qa = it.q0 + quarter * 32, qb = qa + 31;
            const int lo_a = max(0, qa - p.left), lo_b = max(0, qb - p.left);
            const int hi_a = min(p.N - 1, qa + p.right), hi_b = min(p.N - 1, qb + p.right);
#pragma unroll
            for (int c = 0; c < kSwaKeys / 32; ++c) {
              const int cs = j0 + 32 * c, ce = cs + 31;
              if (hi_b < cs || lo_a > ce) {
                empty |= 1u << c;
              } else if (lo_b > cs || hi_a < ce) {
#pragma unroll
                for (int j = 32 * c; j < 32 * c + 32; ++j)
                  if (j0 + j < lo_i || j0 + j > hi_i) sr[j] = __float_as_uint(-INFINITY);
              }
            }
          }
          float m8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) m8[j] = -INFINITY;
#pragma unroll
          for (int c = 0; c < kSwaKeys / 32; ++c) {
            if ((empty >> c) & 1u) continue;
#pragma unroll
            for (int j = 32 * c; j < 32 * c + 32; ++j)
              m8[j & 7] = fmaxf(m8[j & 7], __uint_as_float(sr[j]));
          }
          const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
          const bool move = mx > ref + kSwaSlack;
          if (__any_sync(kFull, move)) {
            const float alpha = move ? ex2(ref - mx) : 1.f;
            if (i > 0) {
              // PV of the previous tile has completed: this tile's S was
              // committed after it
#pragma unroll 1
              for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tc_ld32(lane_addr + col_o + 32 * c, o);
                tc_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                tc_st32(lane_addr + col_o + 32 * c, o);
              }
              tc_wait_st();
            }
            if (move) {
              l *= alpha;
              ref = mx;
              neg = -mx;
            }
          }
          float l8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) l8[j] = 0.f;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t pw[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              if ((empty >> (2 * h2 + half)) & 1u) {
#pragma unroll
                for (int c = 16 * half; c < 16 * half + 16; ++c) pw[c] = 0u;
                continue;
              }
#pragma unroll
              for (int c = 16 * half; c < 16 * half + 16; ++c) {
                const int j = 64 * h2 + 2 * c;
                const float e0 = ex2(fmaf(__uint_as_float(sr[j]), sl2, neg));
                const float e1 = ex2(fmaf(__uint_as_float(sr[j + 1]), sl2, neg));
                l8[(2 * c) & 7] += e0;
                l8[(2 * c + 1) & 7] += e1;
                pw[c] = pack2<BF16>(e0, e1);
              }
            }
            tc_st32(lane_addr + col_s + 32 * h2, pw);  // P over the S just read
          }
          l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
          tc_wait_st();
          tc_fence_before();
  mbar_arrive(bar(kPPFull + hx));
        };
        if (j0 < it.in_lo || j0 + kSwaKeys - 1 > it.in_hi)
          tile(std::true_type{});
        else
          tile(std::false_type{});
      }
      if (failed) break;
      // epilogue: O of this head once the item's last PV has completed
      uint32_t o[D];
      if (it.nt > 0) {
        if (!wait_all(kPOFull + hx, static_cast<uint32_t>(n & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          tc_ld32(lane_addr + col_o + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&o[32 * c]));
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(kPOEmpty + hx));
      } else {
#pragma unroll
        for (int j = 0; j < D; ++j) o[j] = 0u;
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if constexpr (TMA_O) {
        // stage the O row (128B-swizzled, one 64-column atom after the
        // other) once the previous tile store, of either head, has read the
        // buffer: the tiles go A, B of every item
        const int e = 2 * ne + hx;
        if (e >= 1 && !wait_all(kPOSmemFree, static_cast<uint32_t>((e - 1) & 1))) {
          failed = true;
          break;
        }
        uint8_t* const srow = gbase + C::kOffO + row * 128;
#pragma unroll
        for (int q = 0; q < D / 8; ++q) {
          uint4 w;
          w.x = pack2<BF16>(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
          w.y = pack2<BF16>(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
          w.z = pack2<BF16>(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
          w.w = pack2<BF16>(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
          *reinterpret_cast<uint4*>(srow + (q >> 3) * C::kAtomBytes +
                                    (((q & 7) ^ (row & 7)) << 4)) = w;
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kPOStaged + hx));
        ++ne;
      }
      if (iq < p.M) {
        uint16_t* const orow =
            static_cast<uint16_t*>(p.O) + ((static_cast<int64_t>(it.b) * p.M + iq) * p.H + h) * D;
        if constexpr (TMA_O) {
          // O went through the staging buffer
        } else if (p.o32) {
          // 32-byte stores: whole sectors, half the store instructions
#pragma unroll
          for (int q = 0; q < D / 16; ++q) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w[e] = pack2<BF16>(__uint_as_float(o[16 * q + 2 * e]) * inv,
                                 __uint_as_float(o[16 * q + 2 * e + 1]) * inv);
            asm volatile(
                "st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n" ::"l"(orow + 16 * q),
                "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                "r"(w[7])
                : "memory");
          }
        } else {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int q = 0; q < D / 8; ++q) {
            uint4 w;
            w.x = pack2<BF16>(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
            w.y = pack2<BF16>(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
            w.z = pack2<BF16>(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
            w.w = pack2<BF16>(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
            dst[q] = w;
          }
        }
        if (p.LSE != nullptr) {
          constexpr float kLn2 = 0.69314718055994530942f;
          p.LSE[(static_cast<int64_t>(it.b) * p.H + h) * p.M + iq] =
              l > 0.f ? (ref + __log2f(l)) * kLn2 : -INFINITY;
        }
      }
      gt += it.nt;
      if (it.nt > 0) ++n;
    }
  }

  if (failed) report_timeout();
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, kSwaTmemCols);
  }
}

template <int D, bool BF16>
int launch_swa(const SwaProblem& p, const void* Q, const void* K, const void* V, void* O,
               cudaStream_t st) {
  using C = SwaCfg<D>;
  constexpr CUtensorMapDataType dt =
      BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tq, tk, tv, to;
  if (!encode_kv_map(&tq, Q, p.B, p.M, p.H, D, kSwaQ, dt) ||
      !encode_kv_map(&to, O, p.B, p.M, p.H, D, kSwaQ, dt))
    return NSA_ERR_LAUNCH;
  if (p.N > 0) {
    if (!encode_kv_map(&tk, K, p.B, p.N, p.Hkv, D, kSwaKeys, dt) ||
        !encode_kv_map(&tv, V, p.B, p.N, p.Hkv, D, kSwaKeys, dt))
      return NSA_ERR_LAUNCH;
  } else {
    memset(&tk, 0, sizeof(tk));  // no key: no tile is ever loaded
    memset(&tv, 0, sizeof(tv));
  }
  auto kern = swa_fwd_kernel<D, BF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return NSA_ERR_LAUNCH;
  // persistent: one CTA per SM, work items dealt round-robin
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return NSA_ERR_LAUNCH;
  const int64_t blocks = p.items < sms ? p.items : sms;
  kern<<<static_cast<unsigned>(blocks), kSwaThreads, C::kSmemBytes, st>>>(p, tq, tk, tv, to);
  return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
}

template <int D, bool BF16, bool TMA_O>
int launch_swa_pair(SwaProblem p, const void* Q, const void* K, const void* V,
                    cudaStream_t st) {
  using C = SwaPairCfg<D, TMA_O>;
  constexpr CUtensorMapDataType dt =
      BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tq, tk, tv, to;
  if (!encode_kv_map(&tq, Q, p.B, p.M, p.H, D, kSwaQ, dt) ||
      !encode_kv_map(&tk, K, p.B, p.N, p.Hkv, D, kSwaKeys, dt) ||
      !encode_kv_map(&tv, V, p.B, p.N, p.Hkv, D, kSwaKeys, dt))
    return NSA_ERR_LAUNCH;
  if (TMA_O) {
    if (!encode_kv_map(&to, p.O, p.B, p.M, p.H, D, kSwaQ, dt)) return NSA_ERR_LAUNCH;
  } else {
    memset(&to, 0, sizeof(to));  // never read
  }
  auto kern = swa_fwd_pair_kernel<D, BF16, TMA_O>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return NSA_ERR_LAUNCH;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return NSA_ERR_LAUNCH;
  p.items /= 2;  // items of two heads (hpg is even)
  const int64_t blocks = p.items < sms ? p.items : sms;
  kern<<<static_cast<unsigned>(blocks), kSwaPairThreads, C::kSmemBytes, st>>>(p, tq, tk, tv, to);
  return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
}

}  // namespace

int swa_read_and_clear_status(unsigned int* value) { return read_and_clear_status(value); }

}  // namespace nsa

extern "C" int nsa_swa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                           int64_t B, int64_t M, int64_t N, int64_t H, int64_t H_kv, int64_t D,
                           int64_t window_left, int64_t window_right, float scale, int dtype,
                           void* stream) {
  using namespace nsa;
  if (B < 0 || M < 0 || N < 0 || H <= 0 || H_kv <= 0) return NSA_ERR_SHAPE;
  if (H % H_kv != 0) return NSA_ERR_GROUPS;
  if (D != 64 && D != 128) return NSA_ERR_HEAD_DIM;
  if (dtype != NSA_F16 && dtype != NSA_BF16) return NSA_ERR_DTYPE;
  const int64_t lim = (int64_t(1) << 30);
  if (M > lim || N > lim || H > 65536 || B > 65536) return NSA_ERR_SHAPE;
  const int64_t qtiles = (M + kSwaQ - 1) / kSwaQ;
  if (B * H * qtiles > (int64_t(1) << 31) - 1) return NSA_ERR_SHAPE;
  if (B == 0 || M == 0) return NSA_OK;
  if (!Q || !O) return NSA_ERR_NULL;
  if (N > 0 && (!K || !V)) return NSA_ERR_NULL;
  auto mis = [](const void* ptr, uintptr_t a) {
    return ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
  };
  if (mis(Q, 16) || mis(K, 16) || mis(V, 16) || mis(O, 16) || mis(LSE, 4)) return NSA_ERR_ALIGN;
  SwaProblem p;
  p.LSE = LSE;
  p.B = static_cast<int>(B);
  p.items = B * H * qtiles;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.H = static_cast<int>(H);
  p.Hkv = static_cast<int>(H_kv);
  p.hpg = static_cast<int>(H / H_kv);
  p.qtiles = static_cast<int>(qtiles);
  const int64_t unb = M + N;  // a window side this wide reaches every key
  p.left = static_cast<int>(window_left < 0 || window_left > unb ? unb : window_left);
  p.right = static_cast<int>(window_right < 0 || window_right > unb ? unb : window_right);
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  p.sl2 = sc * 1.4426950408889634f;
  p.O = O;
  p.o32 = (reinterpret_cast<uintptr_t>(O) & 31u) == 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf = dtype == NSA_BF16;
  // an even number of heads per KV group: the head-pair kernel (for every
  // window: at (256, 0) it runs 550 TFLOP/s against the one-head kernel's
  // 426, at (128, 0) 293-312 against 260)
  const int64_t span = static_cast<int64_t>(p.left) + p.right + kSwaQ;  // keys a query tile touches
  if (p.hpg % 2 == 0 && N > 0) {
    if (span <= kSwaPairTmaOMaxKeys) {  // short windows: O by TMA stores
      if (D == 64)
        return bf ? launch_swa_pair<64, true, true>(p, Q, K, V, st)
                  : launch_swa_pair<64, false, true>(p, Q, K, V, st);
      return bf ? launch_swa_pair<128, true, true>(p, Q, K, V, st)
                : launch_swa_pair<128, false, true>(p, Q, K, V, st);
    }
    if (D == 64)
      return bf ? launch_swa_pair<64, true, false>(p, Q, K, V, st)
                : launch_swa_pair<64, false, false>(p, Q, K, V, st);
    return bf ? launch_swa_pair<128, true, false>(p, Q, K, V, st)
              : launch_swa_pair<128, false, false>(p, Q, K, V, st);
  }
  if (D == 64)
    return bf ? launch_swa<64, true>(p, Q, K, V, O, st) : launch_swa<64, false>(p, Q, K, V, O, st);
  return bf ? launch_swa<128, true>(p, Q, K, V, O, st)
            : launch_swa<128, false>(p, Q, K, V, O, st);
}
