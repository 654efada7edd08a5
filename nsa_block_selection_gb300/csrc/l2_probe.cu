// Gather-bandwidth probe: the ceiling the selection forward's block gather
// meets once the selected K/V blocks live in L2.
//
// The gather ("[wave] NSA: selection attention forward kernel", section
// "MI350 considerations": the irregular block gather is the most
// performance-critical part) moves whole 16-key tiles of the selected blocks
// of one KV group from L2 into shared memory, as TMA boxes of 16 key rows x
// 64 dims with the 128-byte swizzle and an L2 evict_last hint. This kernel
// issues exactly those copies, for randomly chosen blocks, and does nothing
// else: lane 0 of each warp keeps `slots` tiles in flight in the warp's own
// shared-memory ring and re-issues a slot as soon as its copy has landed
// (the whole warp waits, as in the forward).
// The bytes it moves per second over a long run are the most any kernel
// moving the same boxes with the same in-flight depth can reach on the GPU
// it runs on, so the forward's gathered bytes per second divided by the
// probe's best figure is its fraction of the ceiling that binds it.
//
// Tile i of a warp: pair j = i / 2 of (K tile, V tile) covers key rows
// [blk * bs + 16 * (j mod bs/16), +16) of block blk, a hash of (seed, warp,
// j / (bs/16)) mod floor(N / bs); i even reads K, odd reads V. The KV group
// is `g`, or a hash of the block draw when g < 0 (all groups interleaved).
//
// Every wait is bounded (1 s of %globaltimer): on timeout lane 0 sets this
// translation unit's status word, waits (bounded) for its copies still in
// flight and stops; nsa_sync_status() reports NSA_ERR_TIMEOUT.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "nsa_sel_attn.h"
#include "ptx.cuh"
#include "sel_attn_fwd.cuh"
#include "status.cuh"

namespace nsa {

constexpr int kProbeMaxWarps = 32;
constexpr int kProbeMaxSlots = 16;

struct ProbeArgs {
  int64_t loads;  // tiles per warp
  int64_t* rec;   // optional [gridDim.x, 3]: SM id, start ns, end ns
  int nblk, bs, G, g, slots;
  int rows;       // key rows per TMA box (16, 32 or 64; at most bs)
  uint32_t seed;
};

// 32-bit integer hash: two xorshift-multiply rounds (the "lowbias32"
// constants published by C. Wellons, hash-prospector).
__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

template <int D>
__global__ void __launch_bounds__(kProbeMaxWarps * 32)
    l2_gather_probe_kernel(const ProbeArgs a, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV) {
  constexpr int kBoxes = D / kBoxCols;
  const uint32_t kBox = static_cast<uint32_t>(a.rows) * 128u;  // one box: rows x 64 d
  const uint32_t kTile = kBoxes * kBox;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t ring = base + static_cast<uint32_t>(warp * a.slots) * kTile;
  const uint32_t bars =
      base + static_cast<uint32_t>(warps * a.slots) * kTile + static_cast<uint32_t>(warp * a.slots) * 8u;

  if (threadIdx.x == 0 && a.rec != nullptr) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;\n" : "=r"(smid));
    a.rec[3 * blockIdx.x] = smid;
    a.rec[3 * blockIdx.x + 1] = static_cast<int64_t>(globaltimer_ns());
  }
  if (lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int s = 0; s < a.slots; ++s) mbar_init(bars + 8u * s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  // The whole warp runs the loop (lane 0 issues, every lane waits), as the
  // forward's warps do: a lone lane spinning while its warp's other lanes
  // sit at a CTA barrier is not the forward's issue pattern.
  const uint64_t keep = l2_policy_evict_last();
  const uint32_t gw = blockIdx.x * static_cast<uint32_t>(warps) + warp;
  const int tpb = a.bs / a.rows;
  auto issue = [&](int s, int64_t i) {
    if (lane != 0) return;
    const int64_t j = i >> 1;
    const uint32_t h = mix32(a.seed ^ mix32(gw * 0x9e3779b9u + static_cast<uint32_t>(j / tpb)));
    const int blk = static_cast<int>(h % static_cast<uint32_t>(a.nblk));
    const int grp = a.g >= 0 ? a.g : static_cast<int>(mix32(h) % static_cast<uint32_t>(a.G));
    const int n0 = blk * a.bs + static_cast<int>(j % tpb) * a.rows;
    const CUtensorMap* tm = (i & 1) ? &tmV : &tmK;
    const uint32_t dst = ring + static_cast<uint32_t>(s) * kTile, bar = bars + 8u * s;
    mbar_arrive_expect_tx(bar, kTile);
#pragma unroll
    for (int x = 0; x < kBoxes; ++x)
      tma_load_4d(dst + x * kBox, tm, bar, x * kBoxCols, grp, n0, 0, keep);
  };
  const int64_t first = a.loads < a.slots ? a.loads : a.slots;
  for (int s = 0; s < first; ++s) issue(s, s);
  int64_t i = 0;
  bool ok = true;
  for (; i < a.loads; ++i) {
    const int s = static_cast<int>(i % a.slots);
    if (!__all_sync(kFull, wait_phase(bars + 8u * s, static_cast<uint32_t>((i / a.slots) & 1),
                                      kWaitLimitNs))) {
      ok = false;
      break;
    }
    __syncwarp();
    if (i + a.slots < a.loads) issue(s, i + a.slots);
  }
  if (!ok && lane == 0) {
    report_timeout();
    // tiles i .. i + slots - 1 (those issued) may still be landing in this ring
    const int64_t end = i + a.slots < a.loads ? i + a.slots : a.loads;
    for (int64_t k = i; k < end; ++k)
      wait_phase(bars + 8u * static_cast<uint32_t>(k % a.slots),
                 static_cast<uint32_t>((k / a.slots) & 1), kWaitLimitNs);
  }
  __syncthreads();
  if (threadIdx.x == 0 && a.rec != nullptr)
    a.rec[3 * blockIdx.x + 2] = static_cast<int64_t>(globaltimer_ns());
}

// The same copies driven by an index tensor: the forward's own tiles, in
// the forward's order, and nothing else. Warp w walks units u = w, w + W,
// w + 2W, ... (W warps in the grid; unit u = (b, g, m) with m fastest, as in
// the forward's grid), and each unit's row with the forward's TileWalk; the
// K tile and then the V tile of every 16-key tile go through the warp's ring
// of `slots` copies, with no gap between one unit's tiles and the next's.
struct RowsProbeArgs {
  const int32_t* idx;
  int64_t M, N, G, T, units;
  int nblk, bs, slots;
};

template <int D>
__global__ void __launch_bounds__(kProbeMaxWarps * 32)
    gather_rows_probe_kernel(const RowsProbeArgs a, const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV) {
  constexpr int kBoxes = D / kBoxCols;
  constexpr uint32_t kTile = kBoxes * kBoxBytes;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t ring = base + static_cast<uint32_t>(warp * a.slots) * kTile;
  const uint32_t bars = base + static_cast<uint32_t>(warps * a.slots) * kTile +
                        static_cast<uint32_t>(warp * a.slots) * 8u;
  if (lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int s = 0; s < a.slots; ++s) mbar_init(bars + 8u * s, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t keep = l2_policy_evict_last();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * warps;
  int64_t u = static_cast<int64_t>(blockIdx.x) * warps + warp;
  int b = 0, g = 0;
  TileWalk walk;
  auto start_unit = [&]() -> bool {
    if (u >= a.units) return false;
    const int64_t m = u % a.M;
    const int64_t bg = u / a.M;
    g = static_cast<int>(bg % a.G);
    b = static_cast<int>(bg / a.G);
    const int lastkey = static_cast<int>(m < a.N - 1 ? m : a.N - 1);
    walk.init(a.idx + ((b * a.M + m) * a.G + g) * a.T, static_cast<int>(a.T), a.nblk, a.bs,
              lastkey);
    return true;
  };
  bool live = start_unit();
  int pn0 = 0, pb = 0, pg = 0;
  bool pend_v = false;  // the V tile of (pn0, pb, pg) is the next copy
  // the next copy into slot s (warp-uniform); false once every unit is done
  auto issue_next = [&](int s) -> bool {
    if (!pend_v) {
      bool got = false;
      while (live && !got) {
        got = walk.next(pn0);
        if (!got) {
          u += stride;
          live = start_unit();
        }
      }
      if (!got) return false;
      pb = b;
      pg = g;
    }
    if (lane == 0) {
      const uint32_t dst = ring + static_cast<uint32_t>(s) * kTile, bar = bars + 8u * s;
      const CUtensorMap* tm = pend_v ? &tmV : &tmK;
      mbar_arrive_expect_tx(bar, kTile);
#pragma unroll
      for (int x = 0; x < kBoxes; ++x)
        tma_load_4d(dst + x * kBoxBytes, tm, bar, x * kBoxCols, pg, pn0, pb, keep);
    }
    pend_v = !pend_v;
    return true;
  };
  int64_t issued = 0;
  for (int s = 0; s < a.slots; ++s) {
    if (!issue_next(s)) break;
    ++issued;
  }
  int64_t i = 0;
  bool ok = true;
  for (; i < issued; ++i) {
    const int s = static_cast<int>(i % a.slots);
    if (!__all_sync(kFull, wait_phase(bars + 8u * s, static_cast<uint32_t>((i / a.slots) & 1),
                                      kWaitLimitNs))) {
      ok = false;
      break;
    }
    __syncwarp();
    if (issue_next(s)) ++issued;  // copy number i + slots, into the slot just freed
  }
  if (!ok && lane == 0) {
    report_timeout();
    for (int64_t k = i; k < issued; ++k)
      wait_phase(bars + 8u * static_cast<uint32_t>(k % a.slots),
                 static_cast<uint32_t>((k / a.slots) & 1), kWaitLimitNs);
  }
}

// The backward's dQ reductions alone: each warp adds 4 KB rows (the 8 head
// rows of one query and KV group: 8 x 128 fp32, contiguous) into rows drawn
// at random from `rows` rows spaced `stride` floats apart, 16 bytes per lane
// per instruction (red.global.add.v4.f32), as the backward's dQ warps do.
__global__ void reduce_rows_probe_kernel(float* buf, int64_t rows, int64_t stride, int64_t iters,
                                         uint32_t seed) {
  const int lane = threadIdx.x & 31;
  const uint32_t gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (int64_t i = 0; i < iters; ++i) {
    const uint32_t r = mix32(seed ^ mix32(gw * 0x9e3779b9u + static_cast<uint32_t>(i))) %
                       static_cast<uint32_t>(rows);
    float* row = buf + static_cast<int64_t>(r) * stride;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float* q = row + (k * 32 + lane) * 4;
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(q), "f"(0.f), "f"(0.f),
                   "f"(0.f), "f"(0.f)
                   : "memory");
    }
  }
}

static int64_t probe_smem_bytes(int64_t D, int64_t warps, int64_t slots, int64_t rows = kTileKeys) {
  return warps * slots * (D / kBoxCols) * rows * 128 + warps * slots * 8 + 1024;
}

template <int D>
static int launch_probe(const ProbeArgs& a, const void* K, const void* V, int64_t N, int64_t G,
                        int64_t ctas, int warps, cudaStream_t st) {
  CUtensorMap tk, tv;
  if (!encode_kv_map(&tk, K, 1, N, G, D, a.rows) || !encode_kv_map(&tv, V, 1, N, G, D, a.rows))
    return NSA_ERR_LAUNCH;
  const int smem = static_cast<int>(probe_smem_bytes(D, warps, a.slots, a.rows));
  auto kern = l2_gather_probe_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return NSA_ERR_LAUNCH;
  kern<<<static_cast<unsigned>(ctas), warps * 32, smem, st>>>(a, tk, tv);
  return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
}

template <int D>
static int launch_rows_probe(const RowsProbeArgs& a, const void* K, const void* V, int64_t B,
                             int64_t ctas, int warps, int64_t pad, cudaStream_t st) {
  CUtensorMap tk, tv;
  if (!encode_kv_map(&tk, K, B, a.N, a.G, D) || !encode_kv_map(&tv, V, B, a.N, a.G, D))
    return NSA_ERR_LAUNCH;
  const int smem = static_cast<int>(probe_smem_bytes(D, warps, a.slots) + pad);
  auto kern = gather_rows_probe_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return NSA_ERR_LAUNCH;
  kern<<<static_cast<unsigned>(ctas), warps * 32, smem, st>>>(a, tk, tv);
  return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
}

int probe_read_and_clear_status(unsigned int* value) { return read_and_clear_status(value); }

}  // namespace nsa

extern "C" {

int64_t nsa_probe_l2_gather_bytes(int64_t D, int64_t ctas, int warps_per_cta,
                                  int64_t loads_per_warp, int rows_per_box) {
  if ((D != 64 && D != 128) || ctas < 0 || warps_per_cta < 0 || loads_per_warp < 0 ||
      (rows_per_box != 16 && rows_per_box != 32 && rows_per_box != 64))
    return NSA_ERR_SHAPE;
  return ctas * warps_per_cta * loads_per_warp * (D / nsa::kBoxCols) * rows_per_box * 128;
}

int nsa_probe_l2_gather(const void* K, const void* V, int64_t N, int64_t G, int64_t D,
                        int64_t g, int block_size, int64_t ctas, int warps_per_cta,
                        int slots_per_warp, int64_t loads_per_warp, int rows_per_box,
                        uint32_t seed, int64_t* cta_record, void* stream) {
  using namespace nsa;
  if (!K || !V) return NSA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V)) & 15u)
    return NSA_ERR_ALIGN;
  if (D != 64 && D != 128) return NSA_ERR_HEAD_DIM;
  if (block_size != 32 && block_size != 64) return NSA_ERR_BLOCK_SIZE;
  const int64_t lim = (int64_t(1) << 31) - 1024;
  if (N < block_size || N > lim || G < 1 || G > lim || g < -1 || g >= G) return NSA_ERR_SHAPE;
  if (ctas < 1 || ctas > lim || warps_per_cta < 1 || warps_per_cta > kProbeMaxWarps ||
      slots_per_warp < 1 || slots_per_warp > kProbeMaxSlots || loads_per_warp < 0 ||
      loads_per_warp > (int64_t(1) << 40))
    return NSA_ERR_SHAPE;
  if ((rows_per_box != 16 && rows_per_box != 32 && rows_per_box != 64) ||
      rows_per_box > block_size)
    return NSA_ERR_SHAPE;
  if (probe_smem_bytes(D, warps_per_cta, slots_per_warp, rows_per_box) > 227 * 1024)
    return NSA_ERR_SHAPE;
  if (cta_record != nullptr && (reinterpret_cast<uintptr_t>(cta_record) & 7u))
    return NSA_ERR_ALIGN;
  ProbeArgs a;
  a.rows = rows_per_box;
  a.loads = loads_per_warp;
  a.rec = cta_record;
  a.nblk = static_cast<int>(N / block_size);
  a.bs = block_size;
  a.G = static_cast<int>(G);
  a.g = static_cast<int>(g);
  a.slots = slots_per_warp;
  a.seed = seed;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  return D == 64 ? launch_probe<64>(a, K, V, N, G, ctas, warps_per_cta, st)
                 : launch_probe<128>(a, K, V, N, G, ctas, warps_per_cta, st);
}

int nsa_probe_gather_rows(const void* K, const void* V, const int32_t* block_indices, int64_t B,
                          int64_t M, int64_t N, int64_t G, int64_t D, int64_t T, int block_size,
                          int64_t ctas, int warps_per_cta, int slots_per_warp,
                          int64_t extra_smem_bytes, void* stream) {
  using namespace nsa;
  const int chk = check_sizes(B, M, N, G, G, D, T, block_size);
  if (chk != NSA_OK) return chk;
  if (ctas < 1 || ctas > (int64_t(1) << 31) - 1 || warps_per_cta < 1 ||
      warps_per_cta > kProbeMaxWarps || slots_per_warp < 1 || slots_per_warp > kProbeMaxSlots)
    return NSA_ERR_SHAPE;
  if (extra_smem_bytes < 0 ||
      probe_smem_bytes(D, warps_per_cta, slots_per_warp) + extra_smem_bytes > 227 * 1024)
    return NSA_ERR_SHAPE;
  if (B == 0 || M == 0 || N == 0 || T == 0) return NSA_OK;
  if (!K || !V || !block_indices) return NSA_ERR_NULL;
  if (((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V)) & 15u) ||
      (reinterpret_cast<uintptr_t>(block_indices) & 3u))
    return NSA_ERR_ALIGN;
  RowsProbeArgs a;
  a.idx = block_indices;
  a.M = M;
  a.N = N;
  a.G = G;
  a.T = T;
  a.units = B * G * M;
  a.nblk = static_cast<int>((N + block_size - 1) / block_size);
  a.bs = block_size;
  a.slots = slots_per_warp;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  return D == 64 ? launch_rows_probe<64>(a, K, V, B, ctas, warps_per_cta, extra_smem_bytes, st)
                 : launch_rows_probe<128>(a, K, V, B, ctas, warps_per_cta, extra_smem_bytes, st);
}

int nsa_probe_reduce_rows(float* buf, int64_t rows, int64_t stride, int64_t ctas,
                          int warps_per_cta, int64_t iters_per_warp, uint32_t seed,
                          void* stream) {
  using namespace nsa;
  if (!buf) return NSA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(buf) & 15u) return NSA_ERR_ALIGN;
  if (rows < 1 || rows > (int64_t(1) << 31) - 1 || stride < 1024 || stride % 4 != 0 ||
      ctas < 1 || ctas > (int64_t(1) << 31) - 1 || warps_per_cta < 1 ||
      warps_per_cta > kProbeMaxWarps || iters_per_warp < 0 || iters_per_warp > (int64_t(1) << 40))
    return NSA_ERR_SHAPE;
  reduce_rows_probe_kernel<<<static_cast<unsigned>(ctas), warps_per_cta * 32, 0,
                             static_cast<cudaStream_t>(stream)>>>(buf, rows, stride,
                                                                  iters_per_warp, seed);
  return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
}

}  // extern "C"
