// Two-pass NSA selection-attention forward: the blocks that every query of a
// tile of 16 consecutive queries selects are gathered once per tile and
// attended to on the 5th-generation tensor cores; the gather kernel then
// attends to the rest of each query's blocks, starting from that partial
// softmax state.
//
// Operation ("[wave] NSA: selection attention forward kernel", sections
// "Operation" and "Algorithm"): per (b, m, g) one online softmax over the keys
// of the selected blocks, causally masked. The softmax is a sum over keys, so
// it may be split over disjoint key sets and merged: the first pass leaves the
// normalised partial O and its LSE, which is the state (O, row sum 1,
// reference LSE) the online softmax of the second pass continues from. Index
// rows that always keep the initial block and the most recent blocks of a
// query (the top-k selection with forced blocks produces such rows) give
// consecutive queries those blocks in common; gathered once per tile, they
// no longer cross from L2 to the SMs once per query, which is the traffic the
// gather kernel is bound by.
//
// List pass (shared_blocks_kernel, one warp per (b, g, tile)): the blocks
// listed by every query of the tile, taken in the order the tile's first
// query lists them, up to kSharedMax, and only blocks whose first key is
// visible to the tile's first query and whose keys all lie below both M and
// N. Every query of the tile then sees at least one key of each such block;
// the tile-shared pass masks the keys after a row's query (in the block the
// tile's queries sit in), and a key it reads past a row's query is a key
// row of the sequence (< M), never a row past its end. The record
// {count, ids} per tile is the workspace both other passes read.
//
// Tile-shared pass (sel_attn_shared_kernel): persistent, one CTA per SM
// taking the tiles round-robin (tiles with an empty record are skipped), 11
// warps with fixed roles; the next tile's loads overlap the current tile's
// softmax and epilogue:
//  * warp 0, one lane: TMA producer of Q and K. The Q tile is 16 queries x 8
//    heads = 128 rows (row = 8 * query + head, 128B-swizzled boxes of 64
//    dims) in one of two buffers; the K blocks (block_size keys each) go
//    through a 4-stage ring that runs across tiles, a slot freed as soon as
//    its QK^T has completed, so the next QK^T rarely waits for a load;
//  * warp 10, one lane: TMA producer of V, a 2-stage ring freed by the PVs;
//  * warp 1: allocates the 512 tensor-memory columns; one lane issues
//    S_j = Q K_j^T (M = 128, N = block_size, K = 128) into one of two S
//    buffers and O += P_j V_j (M = 128, N = 128, K = block_size; P from tensor
//    memory, written over the first half of S_j; V MN-major from its
//    [keys][d] tile) into one of two O buffers (tiles alternate), in the
//    order S_0, S_1, PV_0, S_2, PV_1, ... over all blocks of all its tiles;
//  * warps 2-5: softmax, one row per thread, with the lazily moved reference
//    of the gather kernel (O rescaled in tensor memory after the previous PV
//    completed); at the end of a tile the row's (ref, l) go to two
//    tensor-memory columns of the tile's O buffer;
//  * warps 6-9: epilogue, while the softmax warps go on with the next tile:
//    O read out of tensor memory (the buffer is then released to the tile
//    after next), O / l staged in shared memory and stored by one TMA tensor
//    store per tile; LSE directly.
// Every wait is bounded (1 s); a role that gives up sets the status word and
// leaves its loop; the teardown always frees the tensor memory.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "nsa_sel_attn.h"
#include "ptx.cuh"
#include "sel_attn_fwd.cuh"
#include "status.cuh"
#include "tc.cuh"

namespace nsa {
namespace {

constexpr int kShHeads = 8;                       // heads per KV group served
constexpr int kShRows = kSharedTileQ * kShHeads;  // 128: the MMA's M
constexpr int kShD = 128;
constexpr int kShThreads = 352;  // K producer, MMA, softmax and epilogue warpgroups, V producer
constexpr int kKStages = 4;  // K ring: a slot is free once its QK^T has completed
constexpr int kVStages = 2;  // V ring: a slot is free once its PV has completed
constexpr uint32_t kShTmemCols = 512;
constexpr uint32_t kColS = 0;    // S buffers at columns 0 and 64 (P over their first half)
constexpr uint32_t kColO = 128;  // two O buffers of 128 columns (tiles alternate)
constexpr uint32_t kColStats = 384;  // per O buffer two columns: the row's ref and l
constexpr float kShSlack = 8.0f;

// One barrier per buffer or ring slot, so that none can complete twice
// before its waiter has seen the first completion. Blocks are counted across
// the CTA's tiles (gi), tiles by n.
constexpr int kQFull = 0;                    // 2 Q buffers
constexpr int kQEmpty = 2;                   // 2: every QK^T of the tile that used the buffer has completed
constexpr int kSFull = 4;                    // 2 S buffers
constexpr int kPFull = 6;                    // 2: P written over that S
constexpr int kODone = 8;                    // 2 O buffers: the tile's last PV has completed
constexpr int kOEmpty = 10;                  // 2: the epilogue warps have read the O buffer
constexpr int kPvDone = 12;                  // one completion per PV
constexpr int kEnd = 13;                     // every MMA of the CTA has completed
constexpr int kOStaged = 14;                 // the epilogue warps have staged the tile's O
constexpr int kOSmemFree = 15;               // the previous tile's O store has read the staging buffer
constexpr int kStats = 16;                   // 2 O buffers: the softmax warps have written (ref, l)
constexpr int kKFull = 18;                   // kKStages
constexpr int kKFree = kKFull + kKStages;    // kKStages: the QK^T that read the slot has completed
constexpr int kVFull = kKFree + kKStages;    // kVStages
constexpr int kVFree = kVFull + kVStages;    // kVStages: the PV that read the slot has completed
constexpr int kNumBars = kVFree + kVStages;

template <int BS>
struct ShCfg {
  static constexpr int kQBox = kShRows * 128;  // 128 rows x 64 d x 2 B
  static constexpr int kQBytes = 2 * kQBox;    // one Q buffer
  static constexpr int kKVBox = BS * 128;      // BS keys x 64 d x 2 B
  static constexpr int kKVBytes = 2 * kKVBox;  // one K (or V) block
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKVBytes;
  static constexpr int kOBox = kShRows * 128;  // 128 rows x 32 fp32
  static constexpr int kOffO = kOffV + kVStages * kKVBytes;  // O tile staged for the TMA store
  static constexpr int kOffBar = kOffO + (kShD / 32) * kOBox;
  static constexpr int kOffTmem = kOffBar + kNumBars * 8;
  // at least 116 KB so that one CTA holds an SM (all 512 tensor-memory columns)
  static constexpr int kUsed = kOffTmem + 16 + 1024;
  static constexpr int kSmemBytes = kUsed > 118784 ? kUsed : 118784;
};

struct ListProblem {
  const int32_t* idx;
  int32_t* lists;
  int64_t M, N, G, T, ntiles, units;
  int bs, nblk;
};

// One warp per (b, g, tile): the record of the blocks every query of the tile
// lists whose first key the tile's first query sees and whose keys all lie
// below M and N.
__global__ void __launch_bounds__(128) shared_blocks_kernel(const ListProblem p) {
  const int lane = threadIdx.x & 31;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (unit >= p.units) return;
  const int64_t tile = unit % p.ntiles;
  const int64_t bg = unit / p.ntiles;
  const int64_t g = bg % p.G;
  const int64_t b = bg / p.G;
  const int64_t m0 = tile * kSharedTileQ;
  const int R = static_cast<int>(p.M - m0 < kSharedTileQ ? p.M - m0 : kSharedTileQ);
  // block e qualifies when e * bs <= m0 (the tile's first query sees its
  // first key) and (e + 1) * bs <= min(M, N) (all its keys exist, below M)
  const int64_t lim = p.M < p.N ? p.M : p.N;
  const int64_t qstride = p.G * p.T;  // between the index rows of consecutive queries
  const int32_t* row0 = p.idx + ((b * p.M + m0) * p.G + g) * p.T;
  int cnt = 0, mine = -1;  // lane j < cnt holds recorded id j
  for (int64_t w = 0; w < p.T && cnt < kSharedMax; w += 32) {
    const int64_t j = w + lane;
    const int e = j < p.T ? __ldg(row0 + j) : -1;
    bool cand = e >= 0 && e < p.nblk && static_cast<int64_t>(e) * p.bs <= m0 &&
                static_cast<int64_t>(e + 1) * p.bs <= lim;
    // an id repeated in the window counts at its first lane; recorded ids once
    const unsigned same = __match_any_sync(kFull, e);
    cand = cand && (same & ((1u << lane) - 1u)) == 0u;
    for (int k = 0; k < cnt; ++k) {
      const int r = __shfl_sync(kFull, mine, k);  // every lane shuffles
      cand = cand && e != r;
    }
    for (int q = 1; q < R && __any_sync(kFull, cand); ++q) {
      const int32_t* rq = row0 + q * qstride;
      bool found = false;
      for (int64_t v = 0; v < p.T; v += 32) {
        const int x = v + lane < p.T ? __ldg(rq + v + lane) : -1;
        const int nv = static_cast<int>(p.T - v < 32 ? p.T - v : 32);
        for (int s = 0; s < nv; ++s) {
          const int y = __shfl_sync(kFull, x, s);  // every lane shuffles
          found = found || e == y;
        }
        if (__all_sync(kFull, found || !cand)) break;
      }
      cand = cand && found;
    }
    unsigned bal = __ballot_sync(kFull, cand);
    while (bal != 0u && cnt < kSharedMax) {
      const int src = __ffs(bal) - 1;
      bal &= bal - 1u;
      const int id = __shfl_sync(kFull, e, src);
      if (lane == cnt) mine = id;
      ++cnt;
    }
  }
  int32_t* rec = p.lists + unit * kSharedRec;
  if (lane == 0) rec[0] = cnt;
  if (lane < kSharedMax) rec[1 + lane] = lane < cnt ? mine : -1;
}

struct ShProblem {
  const int32_t* lists;
  float* O;
  float* LSE;
  int64_t M, H, G, ntiles, units;
  float sl2;  // scale * log2(e)
};

// Tiles are dealt round-robin: CTA c takes tiles c, c + gridDim.x, ...; a
// tile whose record is empty is skipped by every role alike.
__device__ __forceinline__ int tile_count(const ShProblem& p, int64_t x) {
  const int c = __ldg(p.lists + x * kSharedRec);
  return c < kSharedMax ? c : kSharedMax;
}

template <int BS, bool BF16>
__global__ void __launch_bounds__(kShThreads, 1)
    sel_attn_shared_kernel(const ShProblem p, const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmO) {
  using C = ShCfg<BS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  auto bar = [&](int i) { return base + C::kOffBar + 8u * static_cast<uint32_t>(i); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kQFull + s), 1);
      mbar_init(bar(kQEmpty + s), 1);
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kPFull + s), 4 * 32);
      mbar_init(bar(kODone + s), 1);
      mbar_init(bar(kOEmpty + s), 4 * 32);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKFree + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVFree + s), 1);
    }
    mbar_init(bar(kPvDone), 1);
    mbar_init(bar(kEnd), 1);
    mbar_init(bar(kOStaged), 4 * 32);
    mbar_init(bar(kOSmemFree), 1);
    mbar_init(bar(kStats), 4 * 32);
    mbar_init(bar(kStats + 1), 4 * 32);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc_alloc(base + C::kOffTmem, kShTmemCols);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kOffTmem);
  bool failed = false;
  const int64_t step = gridDim.x;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer: Q of each tile (two buffers), its K blocks (ring) ----
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t once = l2_policy_evict_first();
      int64_t gi = 0;  // blocks loaded so far
      int n = 0;       // tiles loaded so far
      for (int64_t x = blockIdx.x; x < p.units && !failed; x += step) {
        const int cnt = tile_count(p, x);
        if (cnt == 0) continue;
        const int g = static_cast<int>((x / p.ntiles) % p.G);
        const int b = static_cast<int>(x / p.ntiles / p.G);
        const int m0 = static_cast<int>((x % p.ntiles) * kSharedTileQ);
        const int qb = n & 1;
        if (n >= 2 &&
            !wait_phase(bar(kQEmpty + qb), static_cast<uint32_t>(((n - 2) >> 1) & 1), kWaitLimitNs)) {
          failed = true;
          break;
        }
        mbar_arrive_expect_tx(bar(kQFull + qb), C::kQBytes);
        for (int a = 0; a < 2; ++a)
          tma_load_4d(base + C::kOffQ + qb * C::kQBytes + a * C::kQBox, &tmQ, bar(kQFull + qb),
                      a * 64, g * kShHeads, m0, b, once);
        const int32_t* ids = p.lists + x * kSharedRec + 1;
        for (int i = 0; i < cnt; ++i, ++gi) {
          const int st = static_cast<int>(gi % kKStages);
          if (gi >= kKStages &&
              !wait_phase(bar(kKFree + st), static_cast<uint32_t>(((gi - kKStages) / kKStages) & 1),
                          kWaitLimitNs)) {
            failed = true;
            break;
          }
          const int key0 = __ldg(ids + i) * BS;
          mbar_arrive_expect_tx(bar(kKFull + st), C::kKVBytes);
          for (int a = 0; a < 2; ++a)
            tma_load_4d(base + C::kOffK + st * C::kKVBytes + a * C::kKVBox, &tmK, bar(kKFull + st),
                        a * 64, g, key0, b, keep);
        }
        ++n;
      }
      // the copies in flight land before the CTA may exit
      for (int j = n >= 2 ? n - 2 : 0; j < n; ++j)
        wait_phase(bar(kQFull + (j & 1)), static_cast<uint32_t>((j >> 1) & 1), kWaitLimitNs);
      for (int64_t j = gi >= kKStages ? gi - kKStages : 0; j < gi; ++j)
        wait_phase(bar(kKFull + static_cast<int>(j % kKStages)),
                   static_cast<uint32_t>((j / kKStages) & 1), kWaitLimitNs);
    }
  } else if (warp == 10) {
    if (lane == 0) {
      // ---- TMA producer of the V blocks (ring), ahead of the PVs ----
      tma_prefetch_desc(&tmV);
      const uint64_t keep = l2_policy_evict_last();
      int64_t gi = 0;  // blocks loaded so far
      for (int64_t x = blockIdx.x; x < p.units && !failed; x += step) {
        const int cnt = tile_count(p, x);
        if (cnt == 0) continue;
        const int g = static_cast<int>((x / p.ntiles) % p.G);
        const int b = static_cast<int>(x / p.ntiles / p.G);
        const int32_t* ids = p.lists + x * kSharedRec + 1;
        for (int i = 0; i < cnt; ++i, ++gi) {
          const int st = static_cast<int>(gi % kVStages);
          if (gi >= kVStages &&
              !wait_phase(bar(kVFree + st), static_cast<uint32_t>(((gi - kVStages) / kVStages) & 1),
                          kWaitLimitNs)) {
            failed = true;
            break;
          }
          const int key0 = __ldg(ids + i) * BS;
          mbar_arrive_expect_tx(bar(kVFull + st), C::kKVBytes);
          for (int a = 0; a < 2; ++a)
            tma_load_4d(base + C::kOffV + st * C::kKVBytes + a * C::kKVBox, &tmV, bar(kVFull + st),
                        a * 64, g, key0, b, keep);
        }
      }
      for (int64_t j = gi >= kVStages ? gi - kVStages : 0; j < gi; ++j)
        wait_phase(bar(kVFull + static_cast<int>(j % kVStages)),
                   static_cast<uint32_t>((j / kVStages) & 1), kWaitLimitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: the blocks of all tiles as one stream ----
      // S_0, S_1, PV_0, S_2, PV_1, ...: S of block j is issued after PV of
      // block j - 2 (which read the P written over the same S buffer) and
      // before PV of block j - 1.
      constexpr uint32_t idesc_s = umma_idesc_f16(kShRows, BS, BF16, false);
      constexpr uint32_t idesc_o = umma_idesc_f16(kShRows, kShD, BF16, true);
      auto issue_s = [&](int64_t gi, int qb) -> bool {
        const int st = static_cast<int>(gi % kKStages);
        if (!wait_phase(bar(kKFull + st), static_cast<uint32_t>((gi / kKStages) & 1), kWaitLimitNs))
          return false;
        tc_fence_after();
        const uint32_t d = tmem + kColS + static_cast<uint32_t>(gi & 1) * 64;
        const uint32_t qbase = base + C::kOffQ + qb * C::kQBytes;
        const uint32_t kb = base + C::kOffK + st * C::kKVBytes;
#pragma unroll
        for (int k = 0; k < kShD / 16; ++k) {
          const uint32_t qa = qbase + (k >> 2) * C::kQBox + (k & 3) * 32;
          const uint32_t ka = kb + (k >> 2) * C::kKVBox + (k & 3) * 32;
          tc_mma(d, umma_desc_sw128(qa, 16), umma_desc_sw128(ka, 16), idesc_s, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(kKFree + st));
        tc_commit(bar(kSFull + static_cast<int>(gi & 1)));
        return true;
      };
      // PV of block gi into the O buffer of tile n; `first` / `last`: the
      // tile's first / last block; `nk`: its 16-key steps that reach a key
      // some row of the tile sees (the keys past the tile's last query are
      // left out: their P is 0, and their V rows are never multiplied)
      auto issue_pv = [&](int64_t gi, int n, bool first, bool last, int nk) -> bool {
        const int st = static_cast<int>(gi % kVStages);
        const int sb = static_cast<int>(gi & 1);
        const int ob = n & 1;
        if (!wait_phase(bar(kPFull + sb), static_cast<uint32_t>((gi >> 1) & 1), kWaitLimitNs))
          return false;
        if (!wait_phase(bar(kVFull + st), static_cast<uint32_t>((gi / kVStages) & 1), kWaitLimitNs))
          return false;
        if (first && n >= 2 &&
            !wait_phase(bar(kOEmpty + ob), static_cast<uint32_t>(((n - 2) >> 1) & 1), kWaitLimitNs))
          return false;
        tc_fence_after();
        const uint32_t vb = base + C::kOffV + st * C::kKVBytes;
        const uint32_t pcol = tmem + kColS + static_cast<uint32_t>(sb) * 64;
        const uint32_t ocol = tmem + kColO + static_cast<uint32_t>(ob) * kShD;
        for (int kk = 0; kk < nk; ++kk)
          tc_mma_ts(ocol, pcol + 8 * kk, umma_desc_sw128(vb + kk * 2048, C::kKVBox), idesc_o,
                    (!first || kk > 0) ? 1u : 0u);
        tc_commit(bar(kVFree + st));
        tc_commit(bar(kPvDone));
        if (last) tc_commit(bar(kODone + ob));
        return true;
      };
      bool ok = true;
      int64_t gi = 0;
      int n = 0;
      int64_t pend = -1;  // block whose PV is still to be issued
      int pend_n = 0, pend_nk = BS / 16;
      bool pend_first = false, pend_last = false;
      for (int64_t x = blockIdx.x; x < p.units && ok; x += step) {
        const int cnt = tile_count(p, x);
        if (cnt == 0) continue;
        const int qb = n & 1;
        const int64_t m0 = (x % p.ntiles) * kSharedTileQ;
        const int64_t last_q = m0 + kSharedTileQ - 1 < p.M - 1 ? m0 + kSharedTileQ - 1 : p.M - 1;
        ok = wait_phase(bar(kQFull + qb), static_cast<uint32_t>((n >> 1) & 1), kWaitLimitNs);
        for (int i = 0; i < cnt && ok; ++i) {
          ok = issue_s(gi + i, qb);
          if (ok && i == cnt - 1) tc_commit(bar(kQEmpty + qb));
          if (ok && pend >= 0) ok = issue_pv(pend, pend_n, pend_first, pend_last, pend_nk);
          // keys e * BS .. last_q of block e (e * BS <= m0 <= last_q)
          const int64_t span = last_q + 1 - static_cast<int64_t>(__ldg(p.lists + x * kSharedRec + 1 + i)) * BS;
          pend = gi + i;
          pend_n = n;
          pend_nk = span >= BS ? BS / 16 : static_cast<int>((span + 15) / 16);
          pend_first = i == 0;
          pend_last = i == cnt - 1;
        }
        gi += cnt;
        ++n;
      }
      if (ok && pend >= 0) ok = issue_pv(pend, pend_n, pend_first, pend_last, pend_nk);
      // every MMA issued has completed once kEnd completes
      tc_commit(bar(kEnd));
      if (!wait_phase(bar(kEnd), 0, kWaitLimitNs)) ok = false;
      failed = !ok;
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---- softmax (warps 2..5): thread <-> row 8 * query + head (the
    // tensor-memory lane 32 * (warp % 4) + lane) ----
    const int quarter = warp & 3;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.sl2;
    // waits are decided warp-wide (tcgen05.ld/st are warp-collective)
    auto wait_all = [&](int bi, uint32_t parity) {
      return __all_sync(kFull, wait_phase(bar(bi), parity, kWaitLimitNs));
    };
    int64_t gi = 0;
    int n = 0;
    for (int64_t x = blockIdx.x; x < p.units && !failed; x += step) {
      const int cnt = tile_count(p, x);
      if (cnt == 0) continue;
      const int ob = n & 1;
      const uint32_t ocol = lane_addr + kColO + static_cast<uint32_t>(ob) * kShD;
      float ref = -INFINITY, neg = 0.f, l = 0.f;  // ref, neg in the log2 domain
      for (int i = 0; i < cnt; ++i, ++gi) {
        const int sb = static_cast<int>(gi & 1);
        if (!wait_all(kSFull + sb, static_cast<uint32_t>((gi >> 1) & 1))) {
          failed = true;
          break;
        }
        tc_fence_after();
        const uint32_t scol = lane_addr + kColS + static_cast<uint32_t>(sb) * 64;
        uint32_t sr[BS];
#pragma unroll
        for (int c = 0; c < BS / 32; ++c)
          tc_ld32(scol + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tc_wait_ld();
        // keys after the row's query (only in a block that reaches past the
        // tile's first query) are masked; every row sees the block's first key
        {
          const int e = __ldg(p.lists + x * kSharedRec + 1 + i);
          const int m0 = static_cast<int>((x % p.ntiles) * kSharedTileQ);
          if ((e + 1) * BS - 1 > m0) {  // CTA-uniform
            const int thr = m0 + (quarter * 32 + lane) / kShHeads - e * BS;  // last visible j
#pragma unroll
            for (int j = 0; j < BS; ++j)
              if (j > thr) sr[j] = __float_as_uint(-INFINITY);
          }
        }
        float m8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) m8[j] = __uint_as_float(sr[j]);
#pragma unroll
        for (int j = 8; j < BS; ++j) m8[j & 7] = fmaxf(m8[j & 7], __uint_as_float(sr[j]));
        const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))) * sl2;
        const bool move = mx > ref + kShSlack;
        if (__any_sync(kFull, move)) {
          const float alpha = move ? ex2(ref - mx) : 1.f;
          if (i > 0) {
            // S of this block was issued after the PV two blocks back: the
            // PV of the previous block is the one to wait for
            if (!wait_all(kPvDone, static_cast<uint32_t>((gi - 1) & 1))) {
              failed = true;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < kShD / 32; ++c) {
              uint32_t o[32];
              tc_ld32(ocol + 32 * c, o);
              tc_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
              tc_st32(ocol + 32 * c, o);
            }
            tc_wait_st();
          }
          if (move) {
            l *= alpha;
            ref = mx;
            neg = -mx;
          }
        }
        // P = 2^(s * scale * log2e - ref), two 16-bit values per column, over
        // the first half of S buffer sb
        float l8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) l8[j] = 0.f;
        uint32_t pw[BS / 2];
#pragma unroll
        for (int c = 0; c < BS / 2; ++c) {
          const float e0 = ex2(fmaf(__uint_as_float(sr[2 * c]), sl2, neg));
          const float e1 = ex2(fmaf(__uint_as_float(sr[2 * c + 1]), sl2, neg));
          l8[(2 * c) & 7] += e0;
          l8[(2 * c + 1) & 7] += e1;
          pw[c] = pack2_t<BF16>(e0, e1);
        }
        if constexpr (BS == 64) {
          tc_st32(scol, pw);
        } else {
          tc_st16(scol, pw);
        }
        l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kPFull + sb));
      }
      if (failed) break;
      // hand the row's (ref, l) to the epilogue warps through two tensor-memory
      // columns of this O buffer; they were last read by the epilogue of the
      // tile before last, which released the O buffer after reading them
      if (n >= 2 &&
          !wait_all(kOEmpty + ob, static_cast<uint32_t>(((n - 2) >> 1) & 1))) {
        failed = true;
        break;
      }
      const uint32_t scol = lane_addr + kColStats + 2u * static_cast<uint32_t>(ob);
      tc_st1(scol, __float_as_uint(ref));
      tc_st1(scol + 1, __float_as_uint(l));
      tc_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kStats + ob));
      ++n;
    }
  } else if (warp >= 6) {
    // ---- epilogue (warps 6..9): O of each tile out of tensor memory, O / l
    // staged in shared memory (128B-swizzled rows, four boxes of 32 columns)
    // and stored by one TMA tensor store per tile (rows past M are clipped);
    // LSE directly. Runs while the softmax warps work on the next tile.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    auto wait_all = [&](int bi, uint32_t parity) {
      return __all_sync(kFull, wait_phase(bar(bi), parity, kWaitLimitNs));
    };
    const bool leader = warp == 6 && lane == 0;
    int n = 0;
    for (int64_t x = blockIdx.x; x < p.units && !failed; x += step) {
      const int cnt = tile_count(p, x);
      if (cnt == 0) continue;
      const int ob = n & 1;
      const uint32_t ocol = lane_addr + kColO + static_cast<uint32_t>(ob) * kShD;
      const uint32_t ph = static_cast<uint32_t>((n >> 1) & 1);
      if (!wait_all(kStats + ob, ph) || !wait_all(kODone + ob, ph)) {
        failed = true;
        break;
      }
      tc_fence_after();
      const uint32_t scol = lane_addr + kColStats + 2u * static_cast<uint32_t>(ob);
      const float ref = __uint_as_float(tc_ld1(scol));
      const float l = __uint_as_float(tc_ld1(scol + 1));
      tc_wait_ld();
      if (n >= 1) {  // the previous tile's store must have read the staging buffer
        if (leader) {
          bulk_wait_group_read0();
          mbar_arrive(bar(kOSmemFree));
        }
        if (!wait_all(kOSmemFree, static_cast<uint32_t>((n - 1) & 1))) {
          failed = true;
          break;
        }
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < kShD / 32; ++c) {
        uint32_t o[32];
        tc_ld32(ocol + 32 * c, o);
        tc_wait_ld();
        if (c == kShD / 32 - 1) {
          // O and the stats slot of this buffer are read: release both
          tc_fence_before();
          mbar_arrive(bar(kOEmpty + ob));
        }
        uint8_t* const orow = gbase + C::kOffO + c * C::kOBox + row * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float4*>(orow + ((j ^ (row & 7)) << 4)) =
              make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                          __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kOStaged));
      const int g = static_cast<int>((x / p.ntiles) % p.G);
      const int b = static_cast<int>(x / p.ntiles / p.G);
      const int m0 = static_cast<int>((x % p.ntiles) * kSharedTileQ);
      bool staged = true;
      if (leader) {
        staged = wait_phase(bar(kOStaged), static_cast<uint32_t>(n & 1), kWaitLimitNs);
        if (staged) {
          for (int c = 0; c < kShD / 32; ++c)
            tma_store_4d(&tmO, base + C::kOffO + c * C::kOBox, c * 32, g * kShHeads, m0, b);
          bulk_commit_group();
        }
      }
      if (!__all_sync(kFull, staged)) failed = true;  // warp-wide, like every other decision
      const int64_t m = m0 + (row >> 3);
      if (m < p.M) {
        constexpr float kLn2 = 0.69314718055994530942f;
        p.LSE[(static_cast<int64_t>(b) * p.H + static_cast<int64_t>(g) * kShHeads + (row & 7)) *
                  p.M + m] = l > 0.f ? (ref + __log2f(l)) * kLn2 : -INFINITY;
      }
      ++n;
    }
  }

  // teardown: every role is here; the O stores have completed; the tensor
  // memory is freed
  if (warp == 6 && lane == 0) bulk_wait_group0();
  if (failed) report_timeout();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, kShTmemCols);
  }
}

// Q [B, M, H, D] contiguous as a 4-D map (d, h, m, b); box = 64 d x 8 heads x
// 16 queries x 1: 128 rows of 128 bytes, row = 8 * query + head.
bool encode_q_tile_map(CUtensorMap* tm, const void* ptr, int64_t B, int64_t M, int64_t H,
                       CUtensorMapDataType dt) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kShD), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kShD * 2),
                                 static_cast<cuuint64_t>(H * kShD * 2),
                                 static_cast<cuuint64_t>(M * H * kShD * 2)};
  const cuuint32_t box[4] = {64, kShHeads, kSharedTileQ, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return enc(tm, dt, 4, const_cast<void*>(ptr), dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// O [B, M, H, D] fp32 contiguous as a 4-D map (d, h, m, b); box = 32 d x 8
// heads x 16 queries x 1: 128 rows of 128 bytes, the staged O tile's layout.
bool encode_o_tile_map(CUtensorMap* tm, void* ptr, int64_t B, int64_t M, int64_t H) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kShD), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kShD * 4),
                                 static_cast<cuuint64_t>(H * kShD * 4),
                                 static_cast<cuuint64_t>(M * H * kShD * 4)};
  const cuuint32_t box[4] = {32, kShHeads, kSharedTileQ, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BS, bool BF16>
int launch_shared_kernel(const ShProblem& p, int64_t units, const void* Q, const void* K,
                         const void* V, int64_t B, int64_t M, int64_t N, int64_t H, int64_t G,
                         cudaStream_t st) {
  using C = ShCfg<BS>;
  constexpr CUtensorMapDataType dt =
      BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tq, tk, tv, to;
  if (!encode_q_tile_map(&tq, Q, B, M, H, dt) || !encode_o_tile_map(&to, p.O, B, M, H) ||
      !encode_kv_map(&tk, K, B, N, G, kShD, BS, dt) || !encode_kv_map(&tv, V, B, N, G, kShD, BS, dt))
    return NSA_ERR_LAUNCH;
  auto kern = sel_attn_shared_kernel<BS, BF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return NSA_ERR_LAUNCH;
  // persistent: one CTA per SM, tiles dealt round-robin
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return NSA_ERR_LAUNCH;
  const int64_t blocks = units < sms ? units : sms;
  kern<<<static_cast<unsigned>(blocks), kShThreads, C::kSmemBytes, st>>>(p, tq, tk, tv, to);
  return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
}

}  // namespace

int64_t shared_workspace_bytes(int64_t B, int64_t M, int64_t G) {
  if (B < 0 || M < 0 || G <= 0) return NSA_ERR_SHAPE;
  const int64_t lim = (int64_t(1) << 31) - 1;
  const int64_t ntiles = (M + kSharedTileQ - 1) / kSharedTileQ;
  if (B > 0 && ntiles > 0 && (B > lim / G || B * G > lim / ntiles)) return NSA_ERR_SHAPE;
  const int64_t bytes = B * G * ntiles * kSharedRec * 4;
  return (bytes + 255) / 256 * 256;
}

bool shared_pass_eligible(int64_t H, int64_t G, int64_t D, int o_dtype, const int64_t* strides,
                          int64_t m_off) {
  return D == kShD && G > 0 && H == G * kShHeads && o_dtype == NSA_F32 && strides == nullptr &&
         m_off == 0;
}

bool shared_pass_sizes_ok(int64_t M, int64_t N, int64_t T, int block_size) {
  // 64-key blocks only: three common blocks of 64 keys are about a fifth of
  // a 16-block row's bytes and the gather kernel saves more than the two
  // extra passes cost; at 32 keys they are about a tenth of a 32-block row
  // and the passes cost more than they save (6.27 against 6.19 ms one-pass
  // at B=2, M=32k, T=32).
  // Tensor-map boxes (16 queries, block_size keys) stay within the tensors.
  return block_size == 64 && M >= kSharedTileQ && N >= block_size && T > 0;
}

int launch_shared_passes(const void* Q, const void* K, const void* V, const int32_t* idx,
                         float* O, float* LSE, int64_t B, int64_t M, int64_t N, int64_t H,
                         int64_t G, int64_t T, int block_size, float sl2, bool bf16,
                         int32_t* lists, cudaStream_t st) {
  const int64_t ntiles = (M + kSharedTileQ - 1) / kSharedTileQ;
  const int64_t units = B * G * ntiles;  // < 2^31 (shared_workspace_bytes)
  ListProblem lp;
  lp.idx = idx;
  lp.lists = lists;
  lp.M = M;
  lp.N = N;
  lp.G = G;
  lp.T = T;
  lp.ntiles = ntiles;
  lp.units = units;
  lp.bs = block_size;
  lp.nblk = static_cast<int>((N + block_size - 1) / block_size);
  shared_blocks_kernel<<<static_cast<unsigned>((units + 3) / 4), 128, 0, st>>>(lp);
  if (cudaGetLastError() != cudaSuccess) return NSA_ERR_LAUNCH;

  ShProblem sp;
  sp.lists = lists;
  sp.O = O;
  sp.LSE = LSE;
  sp.M = M;
  sp.H = H;
  sp.G = G;
  sp.ntiles = ntiles;
  sp.units = units;
  sp.sl2 = sl2;
  // block_size == 64 (shared_pass_sizes_ok)
  return bf16 ? launch_shared_kernel<64, true>(sp, units, Q, K, V, B, M, N, H, G, st)
              : launch_shared_kernel<64, false>(sp, units, Q, K, V, B, M, N, H, G, st);
}

int shared_read_and_clear_status(unsigned int* value) { return read_and_clear_status(value); }

}  // namespace nsa
