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
//  * one warp per row, 8 rows per CTA; lane l holds the scores of blocks
//    32j + l (coalesced 128-byte loads, streaming cache hint) as
//    order-preserving 32-bit keys in registers -- forced blocks and
//    non-candidates hold key 0, below every score;
//  * the k-th largest key is bracketed by an interpolation search over the
//    key range (one counting pass and one warp reduction per step, bisection
//    as a safeguard); it stops as soon as a pivot splits off exactly k keys;
//  * the chosen blocks (forced, keys above the threshold, and the first
//    ties at it in block order) are written with ballot compaction, which
//    keeps them in ascending order.

#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "nsa_sel_attn.h"

namespace nsa {
namespace {

constexpr int kTopkWarps = 8;
constexpr int kTopkMaxBlocks = 4096;  // 32 lanes x 128 keys

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
  FastDiv div_g, div_m, div_bs;
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

// J: keys per lane (a multiple of 4), covering nblk <= 32 * J.
template <int J>
__global__ void __launch_bounds__(kTopkWarps * 32, J <= 32 ? 4 : 1)
    topk_blocks_kernel(const TopkProblem p) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // rows < 2^31 and M, N < 2^31 (host checks): 32-bit index arithmetic
  const uint32_t row = blockIdx.x * kTopkWarps + warp;
  if (row >= static_cast<uint64_t>(p.rows)) return;
  const uint32_t bm = fastdiv(row, p.div_g);  // b * M + m
  const uint32_t m = bm - fastdiv(bm, p.div_m) * static_cast<uint32_t>(p.M);
  int32_t* out = p.idx + static_cast<int64_t>(row) * p.T;
  const uint32_t last = static_cast<uint32_t>(p.N) - 1u;  // N > 0 unless c = -1 below
  const int c = p.N > 0 ? static_cast<int>(fastdiv(m < last ? m : last, p.div_bs)) : -1;
  if (c + 1 <= p.T) {
    for (int t = lane; t < p.T; t += 32) out[t] = t <= c ? t : -1;
    return;
  }
  // here c + 1 > T >= n_init + n_local: the forced blocks are distinct candidates
  const int k = p.T - p.n_init - p.n_local;  // free picks
  const int lo_local = c - p.n_local + 1;    // forced: t < n_init or t >= lo_local
  const int nq = (c + 1 + 127) >> 7;         // quads of key slots in use (warp-uniform)
  const float* srow = p.scores + static_cast<int64_t>(row) * p.nblk;

  uint32_t key[J];
#pragma unroll
  for (int j = 0; j < J; ++j) key[j] = 0u;
#pragma unroll
  for (int q = 0; q < J / 4; ++q) {
    if (q >= nq) break;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 128 * q + 32 * i + lane;
      if (t >= p.n_init && t < lo_local) key[4 * q + i] = order_key(__ldcs(srow + t));
    }
  }

  // threshold: the k-th largest key, or a key that already splits off
  // exactly k keys. Bracket [lo, hi) with count(>= lo) = clo >= k >
  // count(>= hi) = chi; each step counts the keys >= a pivot inside it (one
  // pass, one warp reduction) and keeps the half holding the k-th key. The
  // pivot interpolates where the k-th key should sit, except right after an
  // interpolation step that failed to halve the bracket, which is followed
  // by a bisection -- so the bracket at least halves every two steps (at
  // most 64 steps over 32-bit keys; about 5 for i.i.d. scores). Any pivot
  // inside the bracket keeps the result exact. k == 0 selects no free block.
  uint32_t tau = 0xffffffffu;
  if (k > 0) {
    uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
    for (int q = 0; q < J / 4; ++q) {
      if (q >= nq) break;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x = key[4 * q + i];
        kmax = max(kmax, x);
        kmin = min(kmin, x ? x : 0xffffffffu);
      }
    }
    uint32_t lo = __reduce_min_sync(kFull, kmin);
    uint32_t hi = __reduce_max_sync(kFull, kmax) + 1u;  // keys <= 0xff800000: no wrap
    int clo = c + 1 - p.n_init - p.n_local;  // every free candidate (> k of them)
    int chi = 0;
    bool bisect = false;
    for (int it = 0; it < 80 && clo != k && hi - lo > 1u; ++it) {
      const uint32_t w = hi - lo;
      uint32_t piv;
      if (bisect) {
        piv = lo + (w >> 1);
      } else {
        const float f = __fdividef(static_cast<float>(k - chi), static_cast<float>(clo - chi));
        uint32_t d = __float2uint_rz(static_cast<float>(w) * f);
        d = min(max(d, 1u), w - 1u);
        piv = hi - d;  // in [lo + 1, hi - 1]
      }
      int cnt = 0;
#pragma unroll
      for (int q = 0; q < J / 4; ++q) {
        if (q >= nq) break;
        cnt += (key[4 * q] >= piv) + (key[4 * q + 1] >= piv) + (key[4 * q + 2] >= piv) +
               (key[4 * q + 3] >= piv);
      }
      cnt = __reduce_add_sync(kFull, cnt);
      if (cnt >= k) {
        lo = piv;
        clo = cnt;
      } else {
        hi = piv;
        chi = cnt;
      }
      bisect = !bisect && (hi - lo > (w >> 1));
    }
    tau = lo;
  }
  int gt = 0;
#pragma unroll
  for (int q = 0; q < J / 4; ++q) {
    if (q >= nq) break;
    gt += (key[4 * q] > tau) + (key[4 * q + 1] > tau) + (key[4 * q + 2] > tau) +
          (key[4 * q + 3] > tau);
  }
  int need = k - __reduce_add_sync(kFull, gt);  // ties at tau, taken in block order

  // ascending block order: slot 4q + i of lane l is block 128q + 32i + l.
  // Free keys are >= 1 and tau >= 1 when k > 0, so "key > tau" never takes
  // a non-candidate.
  const uint32_t below = lanemask_lt();
  int base = 0;
#pragma unroll
  for (int q = 0; q < J / 4; ++q) {
    if (q >= nq) break;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x = key[4 * q + i];
      const int t = 128 * q + 32 * i + lane;
      bool take = (t < p.n_init || (t >= lo_local && t <= c)) || x > tau;
      if (need > 0) {  // warp-uniform; only when ties straddle the threshold
        const uint32_t tb = __ballot_sync(kFull, x == tau);
        take = take || (x == tau && __popc(tb & below) < need);
        need -= __popc(tb);
      }
      const uint32_t sb = __ballot_sync(kFull, take);
      const int pos = base + __popc(sb & below);
      if (take && pos < p.T) out[pos] = t;  // exactly T are taken; the test only bounds writes
      base += __popc(sb);
    }
  }
}

template <int J>
int launch_topk(const TopkProblem& p, cudaStream_t st) {
  const int64_t blocks = (p.rows + kTopkWarps - 1) / kTopkWarps;
  topk_blocks_kernel<J><<<static_cast<unsigned>(blocks), kTopkWarps * 32, 0, st>>>(p);
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
  p.div_g = make_fastdiv(static_cast<uint32_t>(G));
  p.div_m = make_fastdiv(static_cast<uint32_t>(M));
  p.div_bs = make_fastdiv(static_cast<uint32_t>(block_size));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (nblk <= 256) return launch_topk<8>(p, st);
  if (nblk <= 1024) return launch_topk<32>(p, st);
  if (nblk <= 2048) return launch_topk<64>(p, st);
  return launch_topk<128>(p, st);
}
