// Pieces shared by the selection-attention kernels (forward and backward):
// constants, the bounded mbarrier wait and the per-translation-unit status
// word it reports to, the index-row tile walker, and the host-side encoding
// of the K/V tensor maps.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "nsa_sel_attn.h"
#include "ptx.cuh"

namespace nsa {

// Query heads one warp serves (the N of its MMAs). A KV group with fewer
// heads pads the rest; a group with more (a multiple of 8) is split into
// sub-groups of 8 that share the group's K/V and index row.
constexpr int kHeadsPerGroup = 8;

// Sub-groups of 8 heads for `hpg` heads per KV group (1 when hpg <= 8).
__host__ __device__ inline int head_subgroups(int64_t hpg) {
  return static_cast<int>((hpg + kHeadsPerGroup - 1) / kHeadsPerGroup);
}
constexpr int kTileKeys = 16;
// Two-pass forward: queries per tile whose common blocks are gathered once
// (16 queries x 8 heads = 128 rows, the M of one tcgen05 MMA), and the
// per-tile record the passes share: {count, ids[kSharedMax]} as int32.
constexpr int kSharedTileQ = 16;
constexpr int kSharedMax = 7;
constexpr int kSharedRec = 8;
constexpr int kBoxCols = 64;                   // d columns per TMA box: 128-byte rows
constexpr int kBoxBytes = kTileKeys * 128;     // one box: 16 keys x 64 d x fp16
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr unsigned kFull = 0xffffffffu;

// Bit 0 set by a kernel of this translation unit whose bounded wait gave up.
static __device__ unsigned int g_status_word = 0u;

__device__ __forceinline__ void report_timeout() { atomicOr(&g_status_word, 1u); }

// Bit 1: a check of the NSA_DEBUG_BOUNDS build found an address outside
// what the operation may touch (the access itself is still bounded: TMA
// reads outside a tensor map return zeros).
__device__ __forceinline__ void report_bounds() { atomicOr(&g_status_word, 2u); }

// Reads and clears this translation unit's status word (current device).
static inline int read_and_clear_status(unsigned int* value) {
  if (cudaMemcpyFromSymbol(value, g_status_word, sizeof(*value)) != cudaSuccess)
    return NSA_ERR_LAUNCH;
  if (*value != 0u) {
    const unsigned int zero = 0u;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess)
      return NSA_ERR_LAUNCH;
  }
  return NSA_OK;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait on an mbarrier phase; false after `limit_ns` without it.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Warp-uniform walk over the 16-key tiles one index row selects, in the
// order the row lists its blocks. Padding (< 0 or >= nblk) and blocks that
// start after the last visible key are skipped, as are tiles of a block that
// start after it, and the blocks of an optional skip list (lane j holds id j
// of skip_n ids: blocks another pass has already attended to).
struct TileWalk {
  const int32_t* row;
  int T, nblk, bs, lastkey;
  int win;        // start of the next 32-entry window
  unsigned mask;  // lanes of the current window still to visit
  int lane_val;   // this lane's entry of the current window
  int n0, nend;   // next tile start, end of the visible keys of the block
  int skip_val, skip_n;

  __device__ __forceinline__ void init(const int32_t* r, int T_, int nblk_, int bs_,
                                       int lastkey_) {
    row = r;
    T = T_;
    nblk = nblk_;
    bs = bs_;
    lastkey = lastkey_;
    win = 0;
    mask = 0u;
    lane_val = -1;
    n0 = 0;
    nend = 0;
    skip_val = -1;
    skip_n = 0;
  }

  __device__ __forceinline__ void set_skip(int lane_id, int n) {
    skip_val = lane_id;
    skip_n = n;
  }

  __device__ __forceinline__ bool next(int& out) {
    while (n0 >= nend) {
      while (mask == 0u) {
        if (win >= T) return false;
        const int j = win + (threadIdx.x & 31);
        const int t = (j < T) ? __ldg(row + j) : -1;
        bool ok = t >= 0 && t < nblk && t * bs <= lastkey;
        for (int k = 0; k < skip_n; ++k) {
          const int sk = __shfl_sync(kFull, skip_val, k);  // every lane shuffles
          ok = ok && t != sk;
        }
        mask = __ballot_sync(kFull, ok);
        lane_val = t;
        win += 32;
      }
      const int src = __ffs(mask) - 1;
      mask &= mask - 1u;
      const int t = __shfl_sync(kFull, lane_val, src);
      n0 = t * bs;
      nend = min(n0 + bs, lastkey + 1);
    }
    out = n0;
    n0 += kTileKeys;
    return true;
  }
};

// ---- host: tensor maps over K / V -------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// A [B, N, G, D] 16-bit tensor with element strides (sb, sn, sg) for b, n, g
// (d contiguous) as a 4-D map (d, g, n, b); box = 64 d x 1 x rows x 1. A
// stride of an extent-1 dimension is never used and is replaced by the
// contiguous value (the encoder wants every stride a positive multiple of
// 16 bytes).
static inline bool encode_kv_map_strided(CUtensorMap* tm, const void* ptr, int64_t B, int64_t N,
                                         int64_t G, int64_t D, int rows, CUtensorMapDataType dt,
                                         int64_t sb, int64_t sn, int64_t sg) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  if (G == 1) sg = D;
  if (N == 1) sn = G * sg;
  if (B == 1) sb = N * sn;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(G),
                              static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(sg * 2), static_cast<cuuint64_t>(sn * 2),
                                 static_cast<cuuint64_t>(sb * 2)};
  const cuuint32_t box[4] = {kBoxCols, 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return enc(tm, dt, 4, const_cast<void*>(ptr), dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K or V [B, N, G, D] contiguous as a 4-D map (d, g, n, b); box = 64 d x 1 x rows x 1.
static inline bool encode_kv_map(CUtensorMap* tm, const void* ptr, int64_t B, int64_t N,
                                 int64_t G, int64_t D, int rows = kTileKeys,
                                 CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(G),
                              static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D * 2),
                                 static_cast<cuuint64_t>(G * D * 2),
                                 static_cast<cuuint64_t>(N * G * D * 2)};
  const cuuint32_t box[4] = {kBoxCols, 1, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return enc(tm, dt, 4, const_cast<void*>(ptr), dims, strides, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major fp16 matrix [rows, D] as a 2-D map; box = 64 columns x `rows_per_box`
// rows, 128-byte swizzle (used for the 8 head rows of one (b, m, g)).
static inline bool encode_rows_map(CUtensorMap* tm, const void* ptr, int64_t rows, int64_t D,
                                   int rows_per_box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D * 2)};
  const cuuint32_t box[2] = {kBoxCols, static_cast<cuuint32_t>(rows_per_box)};
  const cuuint32_t estride[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace nsa
