// Top-k block selection for sm_103a: block_indices [B,M,G,T] from one score
// per (b, m, g, key block).
//
// Operation: "[wave] NSA: selection attention forward kernel", section
// "Depends on" names a top-k selection kernel as the producer of
// block_indices, whose layout section "Operation" fixes (T blocks per
// query) and which section "Requirements" shares across the heads of a GQA
// group (one row per (b, m, g)). Per row:
//  * candidates: blocks t = 0..c holding a key visible to query m,
//    c = floor(min(m, N-1) / block_size);
//  * if c + 1 <= T every candidate is selected; otherwise the first n_init
//    and the last n_local candidates are forced and the other
//    T - n_init - n_local slots go to the highest scores (equal scores to
//    the lower block; -0.0 equals +0.0; NaN below every number);
//  * the row is written in ascending block order, -1 padded.
//
// Kernel shape (HBM-bound: each score is read at most once):
//  * one warp per row, rows grid-stride. A row's candidate scores arrive in
//    the warp's shared-memory row buffer by one bulk copy (TMA, mbarrier
//    with a bounded wait); the next row's copy starts once this row's
//    survivors are out of the buffer;
//  * fast path: lane l holds the 4 nqo consecutive blocks from 4 nqo l
//    (nqo = ceil((c + 1) / 128) rounded up to odd, for conflict-free
//    16-byte shared loads), so lane order is block order. A threshold t0
//    from the lane (or group) maxima has at least k scores at or above it;
//    those few survivors are marked with one bit each, placed in block
//    order (per-lane counts, a warp scan) and the S - k smallest of them
//    are dropped one at a time with a warp minimum;
//  * general path (more than 32 free picks, fewer than k groups holding a
//    number, or more than 64 survivors -- ties, clustered scores): lane l
//    holds blocks 128q + 32i + l as order-preserving 32-bit keys; a search
//    over the key range brackets the k-th largest key with one counting
//    pass per step, and the chosen blocks (forced, keys above the
//    threshold, and the first ties at it in block order) are written with
//    ballot compaction.

#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "nsa_sel_attn.h"
#include "ptx.cuh"

namespace nsa {
namespace {

constexpr int kTopkWarps = 8;
constexpr int kTopkMaxBlocks = 4096;  // 32 lanes x 128 keys
constexpr int kSurvivors = 64;        // fast path: scores kept for the exact ranking
constexpr uint32_t kNanBits = 0x7fc00000u;

// n / d for 0 <= n < 2^31 and 1 <= d < 2^31 as (n * mul) >> shift with
// shift = 31 + ceil(log2 d) and mul = ceil(2^shift / d) < 2^32 (division by
// an invariant integer by multiplication, Granlund and Montgomery 1994):
// mul = (2^shift + e) / d with 0 <= e < d, so n * mul / 2^shift exceeds n / d
// by less than 2^(31 - shift) <= 1/d and the floor is exact.
struct FastDiv {
  uint32_t mul;
  uint32_t shift;
};

inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  FastDiv f;
  f.shift = 31 + l;
  f.mul = static_cast<uint32_t>(((uint64_t(1) << f.shift) + d - 1) / d);
  return f;
}

__device__ __forceinline__ uint32_t fastdiv(uint32_t n, FastDiv f) {
  return static_cast<uint32_t>((static_cast<uint64_t>(n) * f.mul) >> f.shift);
}

struct TopkProblem {
  const float* scores;  // [rows, nblk]
  int32_t* idx;         // [rows, T]
  int64_t rows;         // B * M * G
  int64_t M, N;
  int G, T, bs, nblk, n_init, n_local;
  bool vec;  // nblk % 4 == 0 and 16-byte aligned scores: 16-byte copies
  FastDiv div_g, div_m, div_bs;
};

// Per-warp shared memory.
struct TopkSmem {
  uint32_t key[kSurvivors];
  int blk[kSurvivors];
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t r;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
  return r;
}

// A key whose unsigned order is the order of the scores: positive floats
// get the sign bit set, negative ones are complemented; -0.0 becomes +0.0
// and every NaN becomes 1, below -inf (0x007fffff). 0 marks "not a free
// candidate".
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  const uint32_t mag = u & 0x7fffffffu;
  if (mag > 0x7f800000u) return 1u;
  if (mag == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Per-row quantities shared by the load and the selection of one row.
struct TopkRow {
  int64_t row;
  int c;         // last candidate block (-1: none)
  int lo_local;  // forced: t < n_init or lo_local <= t <= c
  int nq;        // quads of key slots in use (warp-uniform)
  int nqo;       // nq rounded up to odd: quads per lane in the row buffer
  bool trivial;  // at most T candidates: all of them, no scores read
};

__device__ __forceinline__ TopkRow topk_row_info(const TopkProblem& p, int64_t row) {
  TopkRow r;
  r.row = row;
  // rows < 2^31 and M, N < 2^31 (host checks): 32-bit index arithmetic
  const uint32_t bm = fastdiv(static_cast<uint32_t>(row), p.div_g);  // b * M + m
  const uint32_t m = bm - fastdiv(bm, p.div_m) * static_cast<uint32_t>(p.M);
  const uint32_t last = static_cast<uint32_t>(p.N) - 1u;  // N > 0 unless c = -1 below
  r.c = p.N > 0 ? static_cast<int>(fastdiv(m < last ? m : last, p.div_bs)) : -1;
  r.trivial = r.c + 1 <= p.T;
  r.lo_local = r.c - p.n_local + 1;
  r.nq = (r.c + 1 + 127) >> 7;
  r.nqo = r.nq | 1;
  return r;
}

// Raw score bits of the free candidates of one row into registers (slot j
// of lane l is block 32j + l). Loads only: nothing reads the registers until
// topk_keys, so the loads stay in flight while the previous row is selected.
template <int J>
__device__ __forceinline__ void topk_load(const TopkProblem& p, const TopkRow& r, int lane,
                                          uint32_t (&key)[J]) {
#pragma unroll
  for (int j = 0; j < J; ++j) key[j] = 0u;
  if (r.trivial) return;
  const float* srow = p.scores + r.row * p.nblk;
#pragma unroll
  for (int q = 0; q < J / 4; ++q) {
    if (q >= r.nq) break;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 128 * q + 32 * i + lane;
      if (t >= p.n_init && t < r.lo_local) key[4 * q + i] = __float_as_uint(__ldcs(srow + t));
    }
  }
}

// Raw bits -> keys of the free candidates; 0 in every other slot.
template <int J>
__device__ __forceinline__ void topk_keys(const TopkProblem& p, const TopkRow& r, int lane,
                                          uint32_t (&key)[J]) {
#pragma unroll
  for (int q = 0; q < J / 4; ++q) {
    if (q >= r.nq) break;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 128 * q + 32 * i + lane;
      key[4 * q + i] =
          (t >= p.n_init && t < r.lo_local) ? order_key(__uint_as_float(key[4 * q + i])) : 0u;
    }
  }
}

// Bracket [lo, hi) of the k-th largest of a set of keys, with
// count(>= lo) = clo >= k > count(>= hi) = chi. A pivot is interpolated where
// the k-th key should sit, or is the midpoint right after an interpolation
// step that failed to halve the bracket, so the bracket at least halves
// every two steps. Any pivot inside the bracket keeps it exact.
struct KeyBracket {
  uint32_t lo, hi;
  int clo, chi;
  bool bisect;

  __device__ __forceinline__ uint32_t pivot(int k) const {
    const uint32_t w = hi - lo;
    if (bisect) return lo + (w >> 1);
    const float f = __fdividef(static_cast<float>(k - chi), static_cast<float>(clo - chi));
    uint32_t d = __float2uint_rz(static_cast<float>(w) * f);
    d = min(max(d, 1u), w - 1u);
    return hi - d;  // in [lo + 1, hi - 1]
  }

  __device__ __forceinline__ void update(uint32_t piv, int cnt, uint32_t w, int k) {
    if (cnt >= k) {
      lo = piv;
      clo = cnt;
    } else {
      hi = piv;
      chi = cnt;
    }
    bisect = !bisect && (hi - lo > (w >> 1));
  }
};

// General path: selects and writes one row from its keys (layout 32j + l).
//  * The k-th largest free key is bracketed (KeyBracket: one counting pass
//    and one warp reduction per step, at most 64 steps); the search stops
//    when a pivot splits off exactly k keys or the bracket holds one value.
//  * Once at most 32 keys are >= lo, they are compacted in block order into
//    one (key, block) pair per lane (through 256 bytes of shared memory per
//    warp): the remaining steps are a ballot each, and only the survivors
//    are written. Otherwise (ties, clustered scores) the steps and the
//    output run over all key slots.
template <int J>
__device__ __forceinline__ void topk_select(const TopkProblem& p, const TopkRow& r, int lane,
                                            uint32_t (&key)[J], uint32_t* s_key, int* s_blk) {
  int32_t* out = p.idx + r.row * p.T;
  const uint32_t below = lanemask_lt();
  if (r.trivial) {
    for (int t = lane; t < p.T; t += 32) out[t] = t <= r.c ? t : -1;
    return;
  }
  topk_keys<J>(p, r, lane, key);
  // here c + 1 > T >= n_init + n_local: the forced blocks are distinct candidates
  const int k = p.T - p.n_init - p.n_local;  // free picks
  // forced blocks: the first n_init at 0.., the last n_local at T - n_local..
  for (int t = lane; t < p.n_init; t += 32) out[t] = t;
  for (int t = lane; t < p.n_local; t += 32) out[p.T - p.n_local + t] = r.lo_local + t;
  if (k == 0) return;

  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int q = 0; q < J / 4; ++q) {
    if (q >= r.nq) break;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x = key[4 * q + i];
      kmax = max(kmax, x);
      kmin = min(kmin, x ? x : 0xffffffffu);
    }
  }
  KeyBracket br;
  br.lo = __reduce_min_sync(kFull, kmin);
  br.hi = __reduce_max_sync(kFull, kmax) + 1u;  // keys <= 0xff800000: no wrap
  br.clo = r.c + 1 - p.n_init - p.n_local;       // every free candidate (> k of them)
  br.chi = 0;
  br.bisect = false;
  int it = 0;
  // phase 1: over all key slots while more than 32 keys are >= lo
  for (; it < 80 && br.clo != k && br.hi - br.lo > 1u && br.clo > 32; ++it) {
    const uint32_t w = br.hi - br.lo;
    const uint32_t piv = br.pivot(k);
    int cnt = 0;
#pragma unroll
    for (int q = 0; q < J / 4; ++q) {
      if (q >= r.nq) break;
      cnt += (key[4 * q] >= piv) + (key[4 * q + 1] >= piv) + (key[4 * q + 2] >= piv) +
             (key[4 * q + 3] >= piv);
    }
    br.update(piv, __reduce_add_sync(kFull, cnt), w, k);
  }
  if (br.clo <= 32) {
    // phase 2: compact the br.clo keys >= lo (ascending blocks) to one per lane
    int base = 0;
#pragma unroll
    for (int q = 0; q < J / 4; ++q) {
      if (q >= r.nq) break;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x = key[4 * q + i];
        const bool keep = x >= br.lo;  // free keys only: lo >= 1
        const uint32_t kb = __ballot_sync(kFull, keep);
        if (keep) {
          const int pos = base + __popc(kb & below);
          s_key[pos] = x;
          s_blk[pos] = 128 * q + 32 * i + lane;
        }
        base += __popc(kb);
      }
    }
    __syncwarp();
    const uint32_t mine = lane < br.clo ? s_key[lane] : 0u;
    const int blk = lane < br.clo ? s_blk[lane] : 0;
    __syncwarp();
    for (; it < 80 && br.clo != k && br.hi - br.lo > 1u; ++it) {
      const uint32_t w = br.hi - br.lo;
      const uint32_t piv = br.pivot(k);
      br.update(piv, __popc(__ballot_sync(kFull, mine >= piv)), w, k);
    }
    const uint32_t tau = br.lo;
    const int need = k - __popc(__ballot_sync(kFull, mine > tau));  // ties at tau, in block order
    const uint32_t tb = __ballot_sync(kFull, mine == tau && mine != 0u);
    const bool take = mine > tau || ((tb >> lane) & 1u && __popc(tb & below) < need);
    const uint32_t sb = __ballot_sync(kFull, take);
    if (take) out[p.n_init + __popc(sb & below)] = blk;
    return;
  }
  // ties or clustered scores: finish over all key slots
  for (; it < 80 && br.clo != k && br.hi - br.lo > 1u; ++it) {
    const uint32_t w = br.hi - br.lo;
    const uint32_t piv = br.pivot(k);
    int cnt = 0;
#pragma unroll
    for (int q = 0; q < J / 4; ++q) {
      if (q >= r.nq) break;
      cnt += (key[4 * q] >= piv) + (key[4 * q + 1] >= piv) + (key[4 * q + 2] >= piv) +
             (key[4 * q + 3] >= piv);
    }
    br.update(piv, __reduce_add_sync(kFull, cnt), w, k);
  }
  const uint32_t tau = br.lo;
  int gt = 0;
#pragma unroll
  for (int q = 0; q < J / 4; ++q) {
    if (q >= r.nq) break;
    gt += (key[4 * q] > tau) + (key[4 * q + 1] > tau) + (key[4 * q + 2] > tau) +
          (key[4 * q + 3] > tau);
  }
  int need = k - __reduce_add_sync(kFull, gt);
  int base = 0;
#pragma unroll
  for (int q = 0; q < J / 4; ++q) {
    if (q >= r.nq) break;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x = key[4 * q + i];
      bool take = x > tau;  // free keys only (tau >= 1)
      if (need > 0) {  // warp-uniform
        const uint32_t tb = __ballot_sync(kFull, x == tau);
        take = take || (x == tau && __popc(tb & below) < need);
        need -= __popc(tb);
      }
      const uint32_t sb = __ballot_sync(kFull, take);
      const int pos = base + __popc(sb & below);
      if (take && pos < k) out[p.n_init + pos] = 128 * q + 32 * i + lane;
      base += __popc(sb);
    }
  }
}

// 4-byte asynchronous copy global -> shared (cached in L1 and L2).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}

// Starts copying the scores of blocks 0..c of a row into a row buffer, in
// block order. Lane l of the fast path reads blocks 4 nqo l .. 4 nqo l +
// 4 nqo - 1 as nqo 16-byte quads from byte 16 nqo l; nqo is odd, so the 8
// lanes of a quarter-warp load from distinct bank groups. 16-byte aligned
// rows of a multiple of 4 blocks (p.vec): one bulk copy issued by lane 0,
// completion counted on the buffer's mbarrier `bar`; other rows: coalesced
// 4-byte cp.async copies, one commit group. Bytes past block c are not
// written (the fast path masks them).
template <int J>
__device__ __forceinline__ void topk_prefetch(const TopkProblem& p, const TopkRow& r, int lane,
                                              uint32_t sbuf, uint32_t bar) {
  const float* src = p.scores + r.row * p.nblk;
  if (p.vec) {
    if (lane == 0) {
      if (r.trivial) {
        mbar_arrive(bar);
      } else {
        // 4 ceil((c + 1) / 4) <= nblk blocks: inside the row
        const uint32_t bytes = 16u * static_cast<uint32_t>((r.c + 4) >> 2);
        fence_proxy_async_smem();  // the buffer's earlier reads come first
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(sbuf, src, bytes, bar);
      }
    }
  } else {
    if (!r.trivial)
      for (int t = lane; t <= r.c; t += 32) cp_async_4(sbuf + 4 * t, src + t);
    cp_async_commit();
  }
}

// Waits for the copies of the row in the buffer: its mbarrier phase
// `parity` (bulk copy, bounded wait) or the cp.async group.
__device__ __forceinline__ bool topk_wait(const TopkProblem& p, uint32_t bar, uint32_t parity) {
  if (p.vec) return wait_phase(bar, parity, kWaitLimitNs);
  cp_async_wait<0>();
  return true;
}

__device__ __forceinline__ void ld_shared_v4f(uint32_t addr, float (&v)[4]) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
               : "r"(addr));
}

// Descending sort of one 32-bit key per lane across the warp (bitonic
// network, 15 compare-exchange steps); lane i ends with the (i+1)-th largest.
__device__ __forceinline__ uint32_t warp_sort_desc(uint32_t v, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t o = __shfl_xor_sync(kFull, v, stride);
      const bool keep_max = ((lane & size) == 0) == ((lane & stride) == 0);
      v = keep_max ? max(v, o) : min(v, o);
    }
  }
  return v;
}

// Bits [lo, hi) of word w of a per-lane element mask (element e is bit
// e mod 32 of word e / 32); lo and hi may lie outside the word.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int w) {
  const int a = max(lo - 32 * w, 0);
  const int b = min(hi - 32 * w, 32);
  if (b <= a) return 0u;
  const uint32_t upto_b = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
  return upto_b & ~((1u << a) - 1u);  // a <= 31 here
}

// Fast path for one row whose scores are in the row buffer `sbuf` (copies
// complete). Returns false, having written at most the forced blocks, when
// the row needs the general path. `pending`: the next row's copies are to
// be issued into the buffer once this row no longer reads it; cleared when
// issued.
//  * Element e of lane l is block 4 nqo l + e (at byte 4 (4 nqo l + e) of
//    the buffer). Forced blocks and blocks past c are masked to NaN (a
//    per-lane bit mask of the free ones), which no comparison passes.
//  * t0 = the k-th largest lane maximum (k <= 16), else the lower end of a
//    KeyBracket over the 128 group maxima (group = lane and e mod 4),
//    stopped once at most k + 8 groups are >= it: the scores >= t0 hold
//    every pick.
//  * Survivors (scores >= t0): one bit per element, a warp scan of the
//    per-lane counts, then each lane copies its own survivors from the row
//    buffer, in block order, to one slot each (S of them, k <= S <=
//    kSurvivors).
//  * S <= 32: the S - k smallest survivors (by score, then the later block
//    first) are dropped one at a time with a warp minimum; the rest are the
//    picks. S > 32: tau = the k-th largest survivor key by a KeyBracket over
//    two keys per lane, and the picks are the keys above tau and the first
//    ties at tau in block order.
template <int J>
__device__ __forceinline__ bool topk_select_fast(const TopkProblem& p, const TopkRow& r,
                                                 const TopkRow& next, bool& pending, int lane,
                                                 uint32_t sbuf, uint32_t bar, TopkSmem& sm) {
  constexpr int Q = J / 4 + 1;         // quads per lane at most (nqo <= Q)
  constexpr int W = (4 * Q + 31) / 32;  // survivor bit words per lane
  int32_t* out = p.idx + r.row * p.T;
  const uint32_t below = lanemask_lt();
  auto release = [&]() {
    if (pending) {  // warp-uniform
      __syncwarp();
      topk_prefetch<J>(p, next, lane, sbuf, bar);
      pending = false;
    }
  };
  if (r.trivial) {
    release();
    for (int t = lane; t < p.T; t += 32) out[t] = t <= r.c ? t : -1;
    return true;
  }
  const int k = p.T - p.n_init - p.n_local;
  if (p.n_init <= 32 && p.n_local <= 32) {
    if (lane < p.n_init) out[lane] = lane;
    if (lane < p.n_local) out[p.T - p.n_local + lane] = r.lo_local + lane;
  } else {
    for (int t = lane; t < p.n_init; t += 32) out[t] = t;
    for (int t = lane; t < p.n_local; t += 32) out[p.T - p.n_local + t] = r.lo_local + t;
  }
  if (k == 0 || k > 32) {
    release();
    return k == 0;
  }

  const int seg = 4 * r.nqo * lane;
  const uint32_t base = sbuf + 16 * r.nqo * lane;  // element e at base + 4 e
  uint32_t vm[W];  // free candidates: blocks n_init <= t < lo_local
#pragma unroll
  for (int w = 0; w < W; ++w) vm[w] = range_bits(p.n_init - seg, r.lo_local - seg, w);
  float gm[4] = {__uint_as_float(kNanBits), __uint_as_float(kNanBits), __uint_as_float(kNanBits),
                 __uint_as_float(kNanBits)};
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    if (q >= r.nqo) break;
    float v[4];
    ld_shared_v4f(base + 16 * q, v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * q + i;
      gm[i] = fmaxf(gm[i], (vm[e >> 5] >> (e & 31)) & 1u ? v[i] : __uint_as_float(kNanBits));
    }
  }

  uint32_t t0key = 0u;
  bool have_t0 = false;
  if (k <= 16) {
    const float lmx = fmaxf(fmaxf(gm[0], gm[1]), fmaxf(gm[2], gm[3]));
    const uint32_t v = lmx == lmx ? order_key(lmx) : 0u;  // 0: the lane holds no number
    if (__popc(__ballot_sync(kFull, v != 0u)) >= k) {
      t0key = __shfl_sync(kFull, warp_sort_desc(v, lane), k - 1);
      have_t0 = true;
    }
  }
  if (!have_t0) {
    uint32_t kg[4];
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    int nz = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kg[i] = gm[i] == gm[i] ? order_key(gm[i]) : 0u;  // 0: the group holds no number
      nz += kg[i] != 0u;
      kmax = max(kmax, kg[i]);
      kmin = min(kmin, kg[i] ? kg[i] : 0xffffffffu);
    }
    KeyBracket br;
    br.clo = __reduce_add_sync(kFull, nz);
    if (br.clo < k) {
      release();
      return false;
    }
    br.lo = __reduce_min_sync(kFull, kmin);
    br.hi = __reduce_max_sync(kFull, kmax) + 1u;
    br.chi = 0;
    br.bisect = false;
    for (int it = 0; it < 80 && br.clo > k + 8 && br.hi - br.lo > 1u; ++it) {
      const uint32_t w = br.hi - br.lo;
      const uint32_t piv = br.pivot(k);
      const int cnt = (kg[0] >= piv) + (kg[1] >= piv) + (kg[2] >= piv) + (kg[3] >= piv);
      br.update(piv, __reduce_add_sync(kFull, cnt), w, k);
    }
    t0key = br.lo;
  }
  // the float whose key is t0key (>= key(-inf) > 1: a number)
  const float t0 = __uint_as_float((t0key & 0x80000000u) ? (t0key & 0x7fffffffu) : ~t0key);

  // survivors: a bit per element (the row read again from the buffer; the
  // mask drops forced blocks and blocks past c), counts scanned across lanes
  uint32_t bits[W];
#pragma unroll
  for (int w = 0; w < W; ++w) bits[w] = 0u;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    if (q >= r.nqo) break;
    float v[4];
    ld_shared_v4f(base + 16 * q, v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * q + i;
      if (v[i] >= t0) bits[e >> 5] |= 1u << (e & 31);
    }
  }
  int cnt = 0;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    bits[w] &= vm[w];
    cnt += __popc(bits[w]);
  }
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, d);
    if (lane >= d) incl += v;
  }
  const int S = __shfl_sync(kFull, incl, 31);
  if (S > kSurvivors) {
    release();
    return false;
  }
  // each lane copies its survivors (raw score bits) in block order
  int pos = incl - cnt;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    uint32_t b = bits[w];
    while (b) {
      const int e = 32 * w + __ffs(b) - 1;
      b &= b - 1u;
      sm.key[pos] = __float_as_uint(ld_shared_f32(base + 4 * e));
      sm.blk[pos] = seg + e;
      ++pos;
    }
  }
  __syncwarp();
  release();
  if (S <= 32) {
    uint32_t key = lane < S ? order_key(__uint_as_float(sm.key[lane])) : 0xffffffffu;
    const int blk = lane < S ? sm.blk[lane] : 0;
    bool keep = lane < S;
    __syncwarp();  // the next row may overwrite the arrays
    // survivor keys are at most key(+inf) < 0xffffffff, the mark of a free slot
    for (int d = S - k; d > 0; --d) {
      const uint32_t m = __reduce_min_sync(kFull, key);
      const uint32_t eq = __ballot_sync(kFull, key == m);
      if (lane == 31 - __clz(eq)) {  // the latest block among the smallest
        key = 0xffffffffu;
        keep = false;
      }
    }
    const uint32_t s0 = __ballot_sync(kFull, keep);
    if (keep) out[p.n_init + __popc(s0 & below)] = blk;
    return true;
  }
  const uint32_t k0 = order_key(__uint_as_float(sm.key[lane]));  // S > 32: every lane holds one
  const int b0 = sm.blk[lane];
  const uint32_t k1 = lane + 32 < S ? order_key(__uint_as_float(sm.key[lane + 32])) : 0u;
  const int b1 = lane + 32 < S ? sm.blk[lane + 32] : 0;
  __syncwarp();  // the next row may overwrite the arrays
  KeyBracket bs;
  bs.lo = __reduce_min_sync(kFull, min(k0, k1 ? k1 : 0xffffffffu));
  bs.hi = __reduce_max_sync(kFull, max(k0, k1)) + 1u;
  bs.clo = S;
  bs.chi = 0;
  bs.bisect = false;
  for (int it = 0; it < 80 && bs.clo != k && bs.hi - bs.lo > 1u; ++it) {
    const uint32_t w = bs.hi - bs.lo;
    const uint32_t piv = bs.pivot(k);
    bs.update(piv, __popc(__ballot_sync(kFull, k0 >= piv)) + __popc(__ballot_sync(kFull, k1 >= piv)),
              w, k);
  }
  const uint32_t tau = bs.lo;
  const int need =
      k - __popc(__ballot_sync(kFull, k0 > tau)) - __popc(__ballot_sync(kFull, k1 > tau));
  const uint32_t e0 = __ballot_sync(kFull, k0 == tau);
  const uint32_t e1 = __ballot_sync(kFull, k1 == tau && k1 != 0u);
  const bool take0 = k0 > tau || (((e0 >> lane) & 1u) && __popc(e0 & below) < need);
  const bool take1 =
      k1 > tau || (((e1 >> lane) & 1u) && __popc(e0) + __popc(e1 & below) < need);
  const uint32_t s0 = __ballot_sync(kFull, take0);
  const uint32_t s1 = __ballot_sync(kFull, take1);
  if (take0) out[p.n_init + __popc(s0 & below)] = b0;
  if (take1) out[p.n_init + __popc(s0) + __popc(s1 & below)] = b1;
  return true;
}

// The general path, on its own load of the row. Not inlined: the fast path
// keeps its registers, and only this rare call pays for saving them.
template <int J>
__device__ __noinline__ void topk_general(const TopkProblem* p, const TopkRow r, int lane,
                                          TopkSmem* sm) {
  uint32_t key[J];
  topk_load<J>(*p, r, lane, key);
  topk_select<J>(*p, r, lane, key, sm->key, sm->blk);
}

// J: keys per lane (a multiple of 4), covering nblk <= 32 * J.

template <int J>
__host__ __device__ constexpr int topk_ctas_per_sm() {
  return J <= 8 ? 4 : (J <= 32 ? 3 : (J <= 64 ? 2 : 1));
}

// Row buffer: 32 lanes x nqo quads (nqo <= J/4 + 1), then its mbarrier.
// A copy fills at most the first 4 nblk <= 128 J bytes; the lanes' reads
// past block c land in the rest and are masked.
template <int J>
__host__ __device__ constexpr int topk_buffer_bytes() {
  return J * 32 * 4 + 512 + 16;
}

template <int J>
__host__ __device__ constexpr int topk_smem_bytes() {
  return kTopkWarps * (topk_buffer_bytes<J>() + static_cast<int>(sizeof(TopkSmem)));
}

// One warp per row, rows grid-stride, one row buffer per warp: the next
// row's copy starts as soon as this row's survivors are out of the buffer
// (topk_select_fast), so it is in flight during the exact selection and the
// output. (Two buffers per warp, the next row copied while this one is
// read, measured slower with cp.async and with bulk copies alike.)
template <int J>
__global__ void __launch_bounds__(kTopkWarps * 32, topk_ctas_per_sm<J>())
    topk_blocks_kernel(const __grid_constant__ TopkProblem p) {
  constexpr int kBar = J * 32 * 4 + 512;  // mbarrier offset inside the buffer
  extern __shared__ __align__(16) uint8_t topk_smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbuf = smem_u32(topk_smem_raw) + warp * topk_buffer_bytes<J>();
  const uint32_t bar = sbuf + kBar;
  TopkSmem& sm =
      reinterpret_cast<TopkSmem*>(topk_smem_raw + kTopkWarps * topk_buffer_bytes<J>())[warp];
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kTopkWarps;
  int64_t row = static_cast<int64_t>(blockIdx.x) * kTopkWarps + warp;
  if (row >= p.rows) return;
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  TopkRow r = topk_row_info(p, row);
  topk_prefetch<J>(p, r, lane, sbuf, bar);
  for (uint32_t parity = 0;; parity ^= 1u) {  // the buffer's mbarrier phase of this row
    const int64_t r1 = row + stride;
    const bool more = r1 < p.rows;
    const TopkRow next = more ? topk_row_info(p, r1) : r;
    // decided warp-wide: the selection below is warp-collective
    if (!__all_sync(kFull, topk_wait(p, bar, parity))) {
      if (lane == 0) report_timeout();  // the row's scores never arrived: stop (outputs undefined)
      return;
    }
    __syncwarp();  // (cp.async rows) every lane's copies are visible to the others
    bool pending = more;
    if (!topk_select_fast<J>(p, r, next, pending, lane, sbuf, bar, sm))
      topk_general<J>(&p, r, lane, &sm);
    if (pending) {  // not issued by the fast path
      __syncwarp();
      topk_prefetch<J>(p, next, lane, sbuf, bar);
    }
    __syncwarp();  // the buffer and the shared arrays are free for the next row
    if (!more) break;
    r = next;
    row = r1;
  }
}

template <int J>
int launch_topk(const TopkProblem& p, cudaStream_t st) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return NSA_ERR_LAUNCH;
  constexpr int smem = topk_smem_bytes<J>();
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(topk_blocks_kernel<J>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return NSA_ERR_LAUNCH;
  const int64_t need = (p.rows + kTopkWarps - 1) / kTopkWarps;
  const int64_t resident = static_cast<int64_t>(sms) * topk_ctas_per_sm<J>();
  const int64_t blocks = need < resident ? need : resident;
  topk_blocks_kernel<J><<<static_cast<unsigned>(blocks), kTopkWarps * 32, smem, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
}

}  // namespace

int topk_read_and_clear_status(unsigned int* value) { return read_and_clear_status(value); }

}  // namespace nsa

extern "C" int nsa_topk_blocks(const float* scores, int32_t* block_indices, int64_t B, int64_t M,
                               int64_t N, int64_t G, int64_t T, int block_size, int n_init,
                               int n_local, void* stream) {
  using namespace nsa;
  if (B < 0 || M < 0 || N < 0 || T < 0 || G <= 0) return NSA_ERR_SHAPE;
  if (block_size <= 0) return NSA_ERR_BLOCK_SIZE;
  if (n_init < 0 || n_local < 0 || static_cast<int64_t>(n_init) + n_local > T)
    return NSA_ERR_SHAPE;
  const int64_t nblk = (N + block_size - 1) / block_size;
  const int64_t lim = (int64_t(1) << 31) - 1024;
  if (nblk > kTopkMaxBlocks || T > lim || M > lim || N > lim) return NSA_ERR_SHAPE;
  const int64_t rows = B * M * G;
  if (B > 0 && M > 0 && (G > lim / M || B > lim / (M * G))) return NSA_ERR_SHAPE;
  if (rows == 0 || T == 0) return NSA_OK;
  if (!block_indices || (nblk > 0 && !scores)) return NSA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(block_indices) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(scores) & 3u) != 0)
    return NSA_ERR_ALIGN;
  TopkProblem p;
  p.scores = scores;
  p.idx = block_indices;
  p.rows = rows;
  p.M = M;
  p.N = N;
  p.G = static_cast<int>(G);
  p.T = static_cast<int>(T);
  p.bs = block_size;
  p.nblk = static_cast<int>(nblk);
  p.n_init = n_init;
  p.n_local = n_local;
  p.vec = nblk % 4 == 0 && (reinterpret_cast<uintptr_t>(scores) & 15u) == 0;
  p.div_g = make_fastdiv(static_cast<uint32_t>(G));
  p.div_m = make_fastdiv(static_cast<uint32_t>(M));
  p.div_bs = make_fastdiv(static_cast<uint32_t>(block_size));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (nblk <= 256) return launch_topk<8>(p, st);
  if (nblk <= 1024) return launch_topk<32>(p, st);
  if (nblk <= 2048) return launch_topk<64>(p, st);
  return launch_topk<128>(p, st);
}
