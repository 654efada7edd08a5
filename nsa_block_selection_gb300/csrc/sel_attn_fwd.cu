// NSA selection-attention forward for sm_103a, and the library's C ABI.
//
// Operation ("[wave] NSA: selection attention forward kernel", sections
// "Operation", "Algorithm", "Requirements"): for every (b, m, g) the heads of
// KV group g attend, with one online softmax, over the keys of the blocks
// block_indices[b, m, g, :] selects, causally masked; O [B,M,H,D] and the
// natural-log LSE [B,H,M] are written.
//
// Kernel shape (one warp per (b, m, g) work unit):
//  * the warp walks its index row and streams the selected keys in tiles of
//    16 keys (K tile + V tile, 2 x 16 x D fp16) through a private ring of
//    NSTAGE shared-memory stages filled with 16-byte cp.async copies; key rows
//    past the query's last visible key are zero-filled and never read;
//  * S^T = K Q^T on the tensor cores (mma.sync m16n8k16, fp16 in, fp32 acc):
//    16 keys x 8 heads, so the group's 8 heads are exactly the MMA's N;
//  * scores are scaled into the log2 domain, causally masked, and folded into
//    a running (max, sum) per head; the probabilities are rounded to fp16,
//    transposed in registers (movmatrix) into the B operand of
//    O^T += V^T P^T, whose A operand comes from ldmatrix.trans;
//  * the epilogue normalises O, writes it as fp32 and writes LSE.
// Shared-memory rows are XOR-swizzled in 16-byte units so every ldmatrix
// phase touches 8 distinct bank groups.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "nsa_sel_attn.h"
#include "ptx.cuh"

#ifndef NSA_WARPS
#define NSA_WARPS 4
#endif
#ifndef NSA_STAGES
#define NSA_STAGES 3
#endif

namespace nsa {

constexpr int kHeadsPerGroup = 8;
constexpr int kTileKeys = 16;

struct Problem {
  const __half* Q;
  const __half* K;
  const __half* V;
  const int32_t* idx;
  float* O;
  float* LSE;
  int64_t B, M, N, H, G, T;
  int64_t units;  // B * G * M
  int bs;
  int nblk;       // ceil(N / bs)
  float sl2;      // scale * log2(e)
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Warp-uniform walk over the 16-key tiles one index row selects, in the
// order the row lists its blocks. Padding (< 0 or >= nblk) and blocks that
// start after the last visible key are skipped, as are tiles of a block that
// start after it.
struct TileWalk {
  const int32_t* row;
  int T, nblk, bs, lastkey;
  int win;        // start of the next 32-entry window
  unsigned mask;  // lanes of the current window still to visit
  int lane_val;   // this lane's entry of the current window
  int n0, nend;   // next tile start, end of the visible keys of the block

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
  }

  __device__ __forceinline__ bool next(int& out) {
    while (n0 >= nend) {
      while (mask == 0u) {
        if (win >= T) return false;
        const int j = win + (threadIdx.x & 31);
        const int t = (j < T) ? __ldg(row + j) : -1;
        const bool ok = t >= 0 && t < nblk && t * bs <= lastkey;
        mask = __ballot_sync(0xffffffffu, ok);
        lane_val = t;
        win += 32;
      }
      const int src = __ffs(mask) - 1;
      mask &= mask - 1u;
      const int t = __shfl_sync(0xffffffffu, lane_val, src);
      n0 = t * bs;
      nend = min(n0 + bs, lastkey + 1);
    }
    out = n0;
    n0 += kTileKeys;
    return true;
  }
};

template <int D, int WARPS, int NSTAGE>
struct WarpKernelCfg {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kPiecesPerRow = D / 8;  // 16-byte pieces
  static constexpr int kTileBytes = kTileKeys * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K tile + V tile
  static constexpr int kWarpBytes = NSTAGE * kStageBytes;
  static constexpr int kSmemBytes = WARPS * kWarpBytes;
  static constexpr int kCopiesPerLane = kTileKeys * kPiecesPerRow / 32;
  static constexpr int kSteps = D / 16;
};

template <int D, int WARPS, int NSTAGE>
__global__ void __launch_bounds__(WARPS * 32)
    sel_attn_fwd_warp_kernel(const Problem p) {
  using C = WarpKernelCfg<D, WARPS, NSTAGE>;
  extern __shared__ __align__(128) uint8_t smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * WARPS + warp;
  if (unit >= p.units) return;
  const int64_t m = unit % p.M;
  const int64_t bg = unit / p.M;
  const int64_t g = bg % p.G;
  const int64_t b = bg / p.G;
  const int gid = lane >> 2;  // MMA group id (row within an 8-row slab)
  const int tig = lane & 3;   // thread in group

  const uint32_t wsm = smem_u32(smem) + warp * C::kWarpBytes;
  const int64_t hbase = g * kHeadsPerGroup;

  // Q^T as the B operand of S^T = K Q^T: head gid, dims 16k + 2tig (+1, +8, +9).
  uint32_t qf[C::kSteps][2];
  {
    const __half* q = p.Q + ((b * p.M + m) * p.H + hbase + gid) * D + 2 * tig;
#pragma unroll
    for (int k = 0; k < C::kSteps; ++k) {
      qf[k][0] = __ldg(reinterpret_cast<const unsigned int*>(q + 16 * k));
      qf[k][1] = __ldg(reinterpret_cast<const unsigned int*>(q + 16 * k + 8));
    }
  }

  const int lastkey = static_cast<int>(m < p.N - 1 ? m : p.N - 1);
  const int32_t* irow = p.idx + ((b * p.M + m) * p.G + g) * p.T;
  const int64_t kv_stride = p.G * D;  // elements between consecutive keys
  const __half* kb = p.K + (b * p.N * p.G + g) * D;
  const __half* vb = p.V + (b * p.N * p.G + g) * D;
  const uint64_t keep = l2_policy_evict_last();

  auto issue = [&](int slot, int n0) {
    const uint32_t sk = wsm + slot * C::kStageBytes;
    const uint32_t sv = sk + C::kTileBytes;
#pragma unroll
    for (int i = 0; i < C::kCopiesPerLane; ++i) {
      const int piece = i * 32 + lane;
      const int r = piece / C::kPiecesPerRow;
      const int c = piece % C::kPiecesPerRow;
      const int n = n0 + r;
      const bool ok = n <= lastkey;
      const int64_t off = static_cast<int64_t>(ok ? n : 0) * kv_stride + c * 8;
      const uint32_t so = r * C::kRowBytes + ((c ^ (r & 7)) << 4);
      cp_async_16_hint(sk + so, kb + off, ok ? 16 : 0, keep);
      cp_async_16_hint(sv + so, vb + off, ok ? 16 : 0, keep);
    }
  };

  TileWalk prod, cons;
  prod.init(irow, static_cast<int>(p.T), p.nblk, p.bs, lastkey);
  cons.init(irow, static_cast<int>(p.T), p.nblk, p.bs, lastkey);

  int issued = 0;
#pragma unroll
  for (int s = 0; s < NSTAGE - 1; ++s) {
    int n0;
    if (prod.next(n0)) {
      issue(issued % NSTAGE, n0);
      ++issued;
    }
    cp_async_commit();
  }

  float acc[C::kSteps][4];
#pragma unroll
  for (int i = 0; i < C::kSteps; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float mrun0 = -INFINITY, mrun1 = -INFINITY;  // heads 2tig, 2tig+1 (log2 domain)
  float l0 = 0.f, l1 = 0.f;                    // this lane's share of the row sums

  // ldmatrix row addresses: K tiles (row-major A), V tiles (transposed A).
  const int ka_row = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int ka_hi = lane >> 4;
  const int va_row = (lane & 7) + (lane >> 4) * 8;
  const int va_hi = (lane >> 3) & 1;
  const int sw = lane & 7;  // row & 7 for both

  int consumed = 0;
  int n0;
  while (cons.next(n0)) {
    {
      int nn;
      if (prod.next(nn)) {
        issue(issued % NSTAGE, nn);
        ++issued;
      }
      cp_async_commit();
    }
    cp_async_wait<NSTAGE - 1>();
    __syncwarp();

    const uint32_t sk = wsm + (consumed % NSTAGE) * C::kStageBytes;
    const uint32_t sv = sk + C::kTileBytes;

    // S^T (16 keys x 8 heads) = K_tile Q^T
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < C::kSteps; ++k) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sk + ka_row * C::kRowBytes + (((2 * k + ka_hi) ^ sw) << 4), a0, a1, a2, a3);
      mma_16816(s, a0, a1, a2, a3, qf[k][0], qf[k][1]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j] *= p.sl2;
    if (n0 + kTileKeys - 1 > lastkey) {  // causal edge or end of keys
      if (n0 + gid > lastkey) s[0] = s[1] = -INFINITY;
      if (n0 + gid + 8 > lastkey) s[2] = s[3] = -INFINITY;
    }

    // online softmax, per head
    float mx0 = fmaxf(s[0], s[2]);
    float mx1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(mrun0, mx0);
    const float mn1 = fmaxf(mrun1, mx1);
    const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float al0 = fast_exp2(mrun0 - mu0);
    const float al1 = fast_exp2(mrun1 - mu1);
    const float p0 = fast_exp2(s[0] - mu0);
    const float p1 = fast_exp2(s[1] - mu1);
    const float p2 = fast_exp2(s[2] - mu0);
    const float p3 = fast_exp2(s[3] - mu1);
    l0 = l0 * al0 + (p0 + p2);
    l1 = l1 * al1 + (p1 + p3);
    mrun0 = mn0;
    mrun1 = mn1;
#pragma unroll
    for (int i = 0; i < C::kSteps; ++i) {
      acc[i][0] *= al0;
      acc[i][1] *= al1;
      acc[i][2] *= al0;
      acc[i][3] *= al1;
    }

    // P^T as the B operand: (keys 2tig.., head gid) from (key gid, heads 2tig..)
    const uint32_t pb0 = movmatrix_t(pack_half2(p0, p1));
    const uint32_t pb1 = movmatrix_t(pack_half2(p2, p3));

    // O^T (D x 8 heads) += V_tile^T P^T
#pragma unroll
    for (int i = 0; i < C::kSteps; ++i) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(sv + va_row * C::kRowBytes + (((2 * i + va_hi) ^ sw) << 4), a0, a1, a2, a3);
      mma_16816(acc[i], a0, a1, a2, a3, pb0, pb1);
    }
    ++consumed;
    __syncwarp();
  }
  cp_async_wait<0>();

  // epilogue: finish the row sums, normalise, store O (fp32) and LSE
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  float* o = p.O + ((b * p.M + m) * p.H + hbase + 2 * tig) * D + gid;
#pragma unroll
  for (int i = 0; i < C::kSteps; ++i) {
    o[16 * i] = acc[i][0] * inv0;
    o[D + 16 * i] = acc[i][1] * inv1;
    o[16 * i + 8] = acc[i][2] * inv0;
    o[D + 16 * i + 8] = acc[i][3] * inv1;
  }
  if (gid == 0) {
    constexpr float kLn2 = 0.69314718055994530942f;
    float* L = p.LSE + (b * p.H + hbase + 2 * tig) * p.M + m;
    L[0] = l0 > 0.f ? (mrun0 + log2f(l0)) * kLn2 : -INFINITY;
    L[p.M] = l1 > 0.f ? (mrun1 + log2f(l1)) * kLn2 : -INFINITY;
  }
}

template <int D>
static int launch_warp_kernel(const Problem& p, cudaStream_t stream) {
  constexpr int W = NSA_WARPS;
  constexpr int S = NSA_STAGES;
  using C = WarpKernelCfg<D, W, S>;
  auto kern = sel_attn_fwd_warp_kernel<D, W, S>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return NSA_ERR_LAUNCH;
  const int64_t blocks = (p.units + W - 1) / W;
  kern<<<static_cast<unsigned>(blocks), W * 32, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
}

}  // namespace nsa

extern "C" {

const char* nsa_status_string(int status) {
  switch (status) {
    case NSA_OK: return "ok";
    case NSA_ERR_NULL: return "null pointer";
    case NSA_ERR_SHAPE: return "invalid shape";
    case NSA_ERR_BLOCK_SIZE: return "block_size must be 32 or 64";
    case NSA_ERR_HEAD_DIM: return "head dim D must be 64 or 128";
    case NSA_ERR_GROUPS: return "H must be 8 * G (8 query heads per KV group)";
    case NSA_ERR_ALIGN: return "misaligned pointer";
    case NSA_ERR_LAUNCH: return "CUDA launch failed";
    case NSA_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int nsa_version(void) { return 100; }

int nsa_sel_attn_fwd(const void* Q, const void* K, const void* V, const int32_t* block_indices,
                     float* O, float* LSE, int64_t B, int64_t M, int64_t N, int64_t H, int64_t G,
                     int64_t D, int64_t T, int block_size, float scale, void* stream) {
  using namespace nsa;
  if (B < 0 || M < 0 || N < 0 || T < 0 || H <= 0 || G <= 0 || D <= 0) return NSA_ERR_SHAPE;
  if (H % G != 0 || H / G != kHeadsPerGroup) return NSA_ERR_GROUPS;
  if (D != 64 && D != 128) return NSA_ERR_HEAD_DIM;
  if (block_size != 32 && block_size != 64) return NSA_ERR_BLOCK_SIZE;
  // 32-bit key and index arithmetic inside the kernel; grid of B*G*M warps
  const int64_t lim = (int64_t(1) << 31) - 1024;
  if (M > lim || N > lim || T > lim || G > lim) return NSA_ERR_SHAPE;
  if (B > 0 && M > 0 && B * G > lim / M) return NSA_ERR_SHAPE;
  if (B == 0 || M == 0) return NSA_OK;
  if (!Q || !O || !LSE) return NSA_ERR_NULL;
  if (N > 0 && (!K || !V)) return NSA_ERR_NULL;
  if (T > 0 && !block_indices) return NSA_ERR_NULL;
  auto mis = [](const void* ptr, uintptr_t a) {
    return ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
  };
  if (mis(Q, 16) || mis(K, 16) || mis(V, 16) || mis(O, 16) || mis(LSE, 4) ||
      mis(block_indices, 4))
    return NSA_ERR_ALIGN;

  Problem p;
  p.Q = static_cast<const __half*>(Q);
  p.K = static_cast<const __half*>(K);
  p.V = static_cast<const __half*>(V);
  p.idx = block_indices;
  p.O = O;
  p.LSE = LSE;
  p.B = B;
  p.M = M;
  p.N = N;
  p.H = H;
  p.G = G;
  p.T = T;
  p.units = B * G * M;
  p.bs = block_size;
  p.nblk = static_cast<int>((N + block_size - 1) / block_size);
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  p.sl2 = sc * 1.4426950408889634f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return D == 64 ? launch_warp_kernel<64>(p, st) : launch_warp_kernel<128>(p, st);
}

}  // extern "C"
