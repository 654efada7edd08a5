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

// Selects and writes one row from its keys.
//  * The k-th largest free key is bracketed in [lo, hi) with
//    count(>= lo) = clo >= k > count(>= hi) = chi; each step counts the keys
//    >= a pivot (interpolated where the k-th key should sit, or a bisection
//    right after an interpolation step that failed to halve the bracket,
//    so the bracket at least halves every two steps: at most 64 steps) and
//    keeps the half holding the k-th key. Any pivot inside the bracket keeps
//    the result exact; the search stops when a pivot splits off exactly k
//    keys or the bracket holds one value.
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
  uint32_t lo = __reduce_min_sync(kFull, kmin);
  uint32_t hi = __reduce_max_sync(kFull, kmax) + 1u;  // keys <= 0xff800000: no wrap
  int clo = r.c + 1 - p.n_init - p.n_local;            // every free candidate (> k of them)
  int chi = 0;
  bool bisect = false;
  auto pivot = [&]() -> uint32_t {
    const uint32_t w = hi - lo;
    if (bisect) return lo + (w >> 1);
    const float f = __fdividef(static_cast<float>(k - chi), static_cast<float>(clo - chi));
    uint32_t d = __float2uint_rz(static_cast<float>(w) * f);
    d = min(max(d, 1u), w - 1u);
    return hi - d;  // in [lo + 1, hi - 1]
  };
  auto update = [&](uint32_t piv, int cnt, uint32_t w) {
    if (cnt >= k) {
      lo = piv;
      clo = cnt;
    } else {
      hi = piv;
      chi = cnt;
    }
    bisect = !bisect && (hi - lo > (w >> 1));
  };
  int it = 0;
  // phase 1: over all key slots while more than 32 keys are >= lo
  for (; it < 80 && clo != k && hi - lo > 1u && clo > 32; ++it) {
    const uint32_t w = hi - lo;
    const uint32_t piv = pivot();
    int cnt = 0;
#pragma unroll
    for (int q = 0; q < J / 4; ++q) {
      if (q >= r.nq) break;
      cnt += (key[4 * q] >= piv) + (key[4 * q + 1] >= piv) + (key[4 * q + 2] >= piv) +
             (key[4 * q + 3] >= piv);
    }
    update(piv, __reduce_add_sync(kFull, cnt), w);
  }
  if (clo <= 32) {
    // phase 2: compact the clo keys >= lo (ascending blocks) to one per lane
    int base = 0;
#pragma unroll
    for (int q = 0; q < J / 4; ++q) {
      if (q >= r.nq) break;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x = key[4 * q + i];
        const bool keep = x >= lo;  // free keys only: lo >= 1
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
    const uint32_t mine = lane < clo ? s_key[lane] : 0u;
    const int blk = lane < clo ? s_blk[lane] : 0;
    __syncwarp();
    for (; it < 80 && clo != k && hi - lo > 1u; ++it) {
      const uint32_t w = hi - lo;
      const uint32_t piv = pivot();
      update(piv, __popc(__ballot_sync(kFull, mine >= piv)), w);
    }
    const uint32_t tau = lo;
    const int need = k - __popc(__ballot_sync(kFull, mine > tau));  // ties at tau, in block order
    const uint32_t tb = __ballot_sync(kFull, mine == tau && mine != 0u);
    const bool take = mine > tau || ((tb >> lane) & 1u && __popc(tb & below) < need);
    const uint32_t sb = __ballot_sync(kFull, take);
    if (take) out[p.n_init + __popc(sb & below)] = blk;
    return;
  }
  // ties or clustered scores: finish over all key slots
  for (; it < 80 && clo != k && hi - lo > 1u; ++it) {
    const uint32_t w = hi - lo;
    const uint32_t piv = pivot();
    int cnt = 0;
#pragma unroll
    for (int q = 0; q < J / 4; ++q) {
      if (q >= r.nq) break;
      cnt += (key[4 * q] >= piv) + (key[4 * q + 1] >= piv) + (key[4 * q + 2] >= piv) +
             (key[4 * q + 3] >= piv);
    }
    update(piv, __reduce_add_sync(kFull, cnt), w);
  }
  const uint32_t tau = lo;
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

// J: keys per lane (a multiple of 4), covering nblk <= 32 * J. Each warp
// takes rows grid-stride; with PIPE the loads of its next row are issued
// before the current row is selected (two key sets in registers).
template <int J>
constexpr int topk_ctas_per_sm() {
  return J <= 8 ? 4 : (J <= 32 ? 2 : 1);
}

template <int J, bool PIPE>
__global__ void __launch_bounds__(kTopkWarps * 32, topk_ctas_per_sm<J>())
    topk_blocks_kernel(const TopkProblem p) {
  __shared__ uint32_t s_key[kTopkWarps][32];
  __shared__ int s_blk[kTopkWarps][32];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kTopkWarps;
  int64_t row = static_cast<int64_t>(blockIdx.x) * kTopkWarps + warp;
  if (row >= p.rows) return;
  uint32_t ka[J];
  TopkRow ra = topk_row_info(p, row);
  topk_load<J>(p, ra, lane, ka);
  if constexpr (PIPE) {
    // one call site (the selection code is large): after each row the
    // prefetched raw bits move into the working set; they have had a whole
    // selection to arrive
    uint32_t kb[J];
    for (;;) {
      const int64_t r1 = row + stride;
      const bool more = r1 < p.rows;
      TopkRow rb = ra;
      if (more) {
        rb = topk_row_info(p, r1);
        topk_load<J>(p, rb, lane, kb);
      }
      topk_select<J>(p, ra, lane, ka, s_key[warp], s_blk[warp]);
      if (!more) break;
#pragma unroll
      for (int j = 0; j < J; ++j) ka[j] = kb[j];
      ra = rb;
      row = r1;
    }
  } else {
    for (;;) {
      topk_select<J>(p, ra, lane, ka, s_key[warp], s_blk[warp]);
      row += stride;
      if (row >= p.rows) break;
      ra = topk_row_info(p, row);
      topk_load<J>(p, ra, lane, ka);
    }
  }
}

template <int J, bool PIPE>
int launch_topk(const TopkProblem& p, cudaStream_t st) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return NSA_ERR_LAUNCH;
  const int64_t need = (p.rows + kTopkWarps - 1) / kTopkWarps;
  const int64_t resident = static_cast<int64_t>(sms) * topk_ctas_per_sm<J>();
  const int64_t blocks = need < resident ? need : resident;
  topk_blocks_kernel<J, PIPE><<<static_cast<unsigned>(blocks), kTopkWarps * 32, 0, st>>>(p);
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
  if (nblk <= 256) return launch_topk<8, true>(p, st);
  if (nblk <= 1024) return launch_topk<32, true>(p, st);
  if (nblk <= 2048) return launch_topk<64, true>(p, st);
  return launch_topk<128, false>(p, st);
}
