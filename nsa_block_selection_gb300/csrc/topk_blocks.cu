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
//  * one warp per row, rows grid-stride. While a row is selected, the next
//    row's scores are already being copied (cp.async) into the warp's
//    shared-memory row buffer;
//  * fast path: lane l holds the 4 nq consecutive blocks from 4 nq l
//    (nq = ceil((c + 1) / 128)), so lane order is block order. g_j = the
//    maximum of group j (lane, slot mod 4). The k-th largest g_j is at most
//    the k-th largest score, so every pick is among the scores at or above
//    it. Those few survivors are compacted in block order (per-lane counts,
//    a warp scan) and the exact k-th largest of them is found by a ballot
//    search;
//  * general path (more than 32 free picks, fewer than k groups holding a
//    number, or more than 64 survivors -- ties, clustered scores): lane l
//    holds blocks 128q + 32i + l as order-preserving 32-bit keys; a search over the key range
//    brackets the k-th largest key with one counting pass per step, and the
//    chosen blocks (forced, keys above the threshold, and the first ties at
//    it in block order) are written with ballot compaction.

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

// Starts copying the scores of blocks 0..c of a row into the warp's row
// buffer. Lane l's segment is the 4 nq blocks from 4 nq l; its quad q
// (blocks 4 nq l + 4q .. + 3) lands at 16-byte slot 32q + l, so each lane
// reads a quad with one conflict-free 16-byte load. Slots past c are not
// written.
template <int J>
__device__ __forceinline__ void topk_prefetch(const TopkProblem& p, const TopkRow& r, int lane,
                                              uint32_t sbuf) {
  const int seg = 4 * r.nq * lane;
  if (!r.trivial && seg <= r.c) {
    const float* src = p.scores + r.row * p.nblk + seg;
#pragma unroll
    for (int q = 0; q < J / 4; ++q) {
      if (q >= r.nq) break;
      const int b0 = seg + 4 * q;
      const uint32_t dst = sbuf + (32 * q + lane) * 16;
      if (p.vec) {
        // b0 % 4 == 0 and nblk % 4 == 0: the 16 bytes lie inside the row
        if (b0 <= r.c) cp_async_16(dst, src + 4 * q, 16);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (b0 + i <= r.c) cp_async_4(dst + 4 * i, src + 4 * q + i);
      }
    }
  }
  cp_async_commit();
}

// Fast path for one row whose scores are in the row buffer; issues the next
// row's copies once the buffer is read. Returns false, having written at
// most the forced blocks, when the row needs the general path.
//  * Forced blocks and blocks past c become NaN, which no comparison passes.
//  * t0 = the k-th largest lane maximum (k <= 16), else the lower end of a
//    KeyBracket over the group-maximum keys, stopped once at most k + 8
//    groups are >= it: the scores >= t0 hold every pick.
//  * The scores >= t0 (S of them, k <= S <= kSurvivors) are compacted in
//    block order; a KeyBracket over them (one ballot per step) finds the k-th
//    largest key tau; the picks are the keys above tau and the first ties at
//    tau in block order.
template <int J>
__device__ __forceinline__ bool topk_select_fast(const TopkProblem& p, const TopkRow& r,
                                                 const TopkRow& next, bool more, int lane,
                                                 uint32_t (&raw)[J], uint32_t sbuf,
                                                 TopkSmem& sm) {
  int32_t* out = p.idx + r.row * p.T;
  const uint32_t below = lanemask_lt();
  const int seg = 4 * r.nq * lane;
  float gm[4] = {__uint_as_float(kNanBits), __uint_as_float(kNanBits), __uint_as_float(kNanBits),
                 __uint_as_float(kNanBits)};
  if (!r.trivial) {
    cp_async_wait<0>();
    __syncwarp();
    const bool edge = seg < p.n_init || seg + 4 * r.nq > r.lo_local;
#pragma unroll
    for (int q = 0; q < J / 4; ++q) {
      if (q >= r.nq) break;
      uint32_t v[4];
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                   : "r"(sbuf + (32 * q + lane) * 16));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = seg + 4 * q + i;
        if (edge && (t < p.n_init || t >= r.lo_local)) v[i] = kNanBits;
        raw[4 * q + i] = v[i];
        gm[i] = fmaxf(gm[i], __uint_as_float(v[i]));
      }
    }
  }
  __syncwarp();  // every lane has read the buffer
  if (more) topk_prefetch<J>(p, next, lane, sbuf);

  if (r.trivial) {
    for (int t = lane; t < p.T; t += 32) out[t] = t <= r.c ? t : -1;
    return true;
  }
  const int k = p.T - p.n_init - p.n_local;
  for (int t = lane; t < p.n_init; t += 32) out[t] = t;
  for (int t = lane; t < p.n_local; t += 32) out[p.T - p.n_local + t] = r.lo_local + t;
  if (k == 0) return true;
  if (k > 32) return false;

  // t0: with k <= 16 and at least k lanes holding a number, the k-th
  // largest lane maximum (a warp bitonic sort of 32 keys); otherwise a
  // KeyBracket over the 128 group maxima, stopped once at most k + 8 groups
  // are >= it. Either way at least k scores are >= t0.
  uint32_t t0key = 0u;
  bool have_t0 = false;
  if (k <= 16) {
    const float lmx = fmaxf(fmaxf(gm[0], gm[1]), fmaxf(gm[2], gm[3]));
    uint32_t v = lmx == lmx ? order_key(lmx) : 0u;  // 0: the lane holds no number
    if (__popc(__ballot_sync(kFull, v != 0u)) >= k) {
#pragma unroll
      for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          const uint32_t o = __shfl_xor_sync(kFull, v, stride);
          const bool keep_max = ((lane & size) == 0) == ((lane & stride) == 0);
          v = keep_max ? max(v, o) : min(v, o);  // descending overall
        }
      }
      t0key = __shfl_sync(kFull, v, k - 1);
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
    if (br.clo < k) return false;
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

  // survivors in block order: count per lane, scan across lanes, write
  int cnt = 0;
#pragma unroll
  for (int q = 0; q < J / 4; ++q) {
    if (q >= r.nq) break;
#pragma unroll
    for (int i = 0; i < 4; ++i) cnt += __uint_as_float(raw[4 * q + i]) >= t0;
  }
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, d);
    if (lane >= d) incl += v;
  }
  const int S = __shfl_sync(kFull, incl, 31);
  if (S > kSurvivors) return false;
  if (cnt) {
    int pos = incl - cnt;
#pragma unroll
    for (int q = 0; q < J / 4; ++q) {
      if (q >= r.nq) break;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (__uint_as_float(raw[4 * q + i]) >= t0) {
          sm.key[pos] = raw[4 * q + i];  // raw bits; keys are formed below
          sm.blk[pos] = seg + 4 * q + i;
          ++pos;
        }
      }
    }
  }
  __syncwarp();
  const uint32_t k0 = lane < S ? order_key(__uint_as_float(sm.key[lane])) : 0u;
  const int b0 = lane < S ? sm.blk[lane] : 0;
  const uint32_t k1 = lane + 32 < S ? order_key(__uint_as_float(sm.key[lane + 32])) : 0u;
  const int b1 = lane + 32 < S ? sm.blk[lane + 32] : 0;
  __syncwarp();  // the next row may overwrite the arrays
  KeyBracket bs;
  bs.lo = __reduce_min_sync(kFull, min(k0 ? k0 : 0xffffffffu, k1 ? k1 : 0xffffffffu));
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
  const uint32_t e0 = __ballot_sync(kFull, k0 == tau && k0 != 0u);
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
constexpr int topk_ctas_per_sm() {
  return J <= 8 ? 4 : (J <= 32 ? 3 : (J <= 64 ? 2 : 1));
}

template <int J>
constexpr int topk_smem_bytes() {
  return kTopkWarps * (J * 32 * 4 + static_cast<int>(sizeof(TopkSmem)));
}

template <int J>
__global__ void __launch_bounds__(kTopkWarps * 32, topk_ctas_per_sm<J>())
    topk_blocks_kernel(const __grid_constant__ TopkProblem p) {
  extern __shared__ __align__(16) uint8_t topk_smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbuf = smem_u32(topk_smem_raw) + warp * (J * 32 * 4);
  TopkSmem& sm = reinterpret_cast<TopkSmem*>(topk_smem_raw + kTopkWarps * (J * 32 * 4))[warp];
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kTopkWarps;
  int64_t row = static_cast<int64_t>(blockIdx.x) * kTopkWarps + warp;
  if (row >= p.rows) return;
  uint32_t raw[J];
  TopkRow r = topk_row_info(p, row);
  topk_prefetch<J>(p, r, lane, sbuf);
  for (;;) {
    const int64_t r1 = row + stride;
    const bool more = r1 < p.rows;
    const TopkRow next = more ? topk_row_info(p, r1) : r;
    if (!topk_select_fast<J>(p, r, next, more, lane, raw, sbuf, sm))
      topk_general<J>(&p, r, lane, &sm);
    __syncwarp();  // the shared arrays are free for the next row
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
