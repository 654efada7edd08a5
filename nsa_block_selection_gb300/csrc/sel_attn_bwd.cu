// NSA selection-attention backward for sm_103a: dQ, dK, dV from dO.
//
// The forward ("[wave] NSA: selection attention forward kernel", sections
// "Operation" / "Algorithm") returns LSE because the backward needs it
// (section "Requirements"). Per (b, m, g) row and head h, over its visible
// keys n, with p_n = exp(scale q.k_n - LSE), dP_n = dO . v_n and
// delta = dO . O:
//   dS_n = p_n (dP_n - delta);  dQ = scale sum_n dS_n k_n;
//   dK[n] += scale dS_n q;      dV[n] += p_n dO.
//
// Stages:
//  1. D = 64: query-major kernel (one warp per (b, m, g), same TMA tile
//     gather as the forward): recomputes S^T = K Q^T, P, dP^T = V dO^T and dS
//     on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32
//     accumulate) and accumulates dQ^T += K^T dS^T in registers; it also
//     writes delta. D = 128: a small kernel writes only the per-row inputs of
//     the tensor-core kernels (16-bit dO, LSE, delta).
//  2. transposed index: for every (b, g, block) the list of queries whose row
//     selects it (count: warp row walks with combined atomics; one-CTA scan;
//     fill with atomics in index order, so lists keep rough query order).
//     With D = 128 the entries of each query's own block c and of block
//     c - 1 stay out of the lists (recorded per row for stage 3a), and the
//     stage runs on a second stream of the call beside stage 1 and 3a.
//  3a. D = 128: local-block kernel, one CTA per (b, block row, g): the two
//     blocks a block row shares, loaded once; each dQ row summed over both
//     on the tensor cores (tcgen05) and stored once, so dQ needs no zeroing;
//     dK / dV of both blocks summed over the block row.
//  3. key-major kernel: one CTA per chunk of <= kQueriesPerChunk queries of a
//     list; the block's K / V are loaded once and each query's S, P, dP, dS
//     recomputed against them. D = 64: bs/16 warps each own 16 keys and use
//     mma.sync m16n8k8 (the C layout of S^T is already the A layout of that
//     MMA) for dV += P^T dO and dK += dS^T Q, added with fp32 atomics at the
//     end of a chunk. D = 128: tcgen05 MMAs with tensor-memory accumulators
//     on 128-row batches of (query, head) rows, which also give dQ = dS K per
//     batch, added into global memory with fp32 reductions; dK / dV are
//     staged in shared memory at the end of a chunk (and of a block row in
//     3a) and added by 512-byte bulk reductions. Summation orders follow the
//     atomics and reductions.
// Masked keys get exact zero weights by select (never multiplied through).
// In stage 1 (D = 64), K / V rows past a query's last visible key are zeroed
// in shared memory before they enter a product; with D = 128 the whole
// block's K rows enter dQ = dS K with dS = 0 for masked keys (and, in 3a,
// for queries of the block row that do not take the block), so those rows
// must hold finite values.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "common.cuh"
#include "nsa_sel_attn.h"
#include "ptx.cuh"
#include "sel_attn_fwd.cuh"
#include "status.cuh"
#include "tc.cuh"

namespace nsa {

// Queries per chunk of a list (the key-major kernels' unit of work): larger
// chunks mean fewer block loads and dK / dV epilogues per list (m64k_bs64
// backward: 64 / 128 / 256 / 384 / 448 queries measured 19.4 / 15.4 / 12.37
// / 11.93 / 11.79 ms). 448 keeps the tensor-core kernel's shared memory
// (query ids included) within 227 KB.
constexpr int kQueriesPerChunk = 448;

// D = A(16x8, row) * B(8x8, col) + D, bf16 inputs, fp32 accumulate: the
// bf16 twin of mma_1688, used only by the key-major dK / dV products.
__device__ __forceinline__ void mma_1688_bf16(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

template <bool BF16>
__device__ __forceinline__ void mma_1688_t(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  if constexpr (BF16)
    mma_1688_bf16(d, a0, a1, b0);
  else
    mma_1688(d, a0, a1, b0);
}

struct BwdProblem {
  const uint16_t* Q;   // fp16 or bf16
  const int32_t* idx;
  const float* O;
  const float* LSE;
  const float* dO;
  float* dQ;
  float* dK;
  float* dV;
  uint16_t* dO16;      // [B, M, H, D] 16-bit copy of dO, in the inputs' type (stage 1 -> 3)
  float* rec;          // [B * M * G * nsub][16]: LSE * log2(e) of 8 heads, then delta
  const int* offs;     // [L + 1] list starts (L = B * G * nblk)
  const int* choffs;   // [L + 1] chunk starts
  const int* chunk_list;  // [chunks] the list of each chunk
  const int* chunk_order;  // [chunks] launch order of the chunks (D = 128), or null
  const int* lists;    // query ids, list by list
  int2* lfirst;        // [B * M * G] per row, the entry index of its first entry of block c
                       // and of block c - 1 (-1: none), taken by the local-block kernel
                       // (D = 128); null otherwise
  int64_t B, M, N, H, G, T;
  int64_t units;       // B * G * nsub * M
  int hpg, nsub;       // heads per KV group, sub-groups of 8 heads
  int bs, nblk, L;
  float sl2;           // scale * log2(e)
  float scale;
};

// 16-byte fp32 reduction into global memory (no return value).
__device__ __forceinline__ void red_add_v4(float* p, float x, float y, float z, float w) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(x), "f"(y), "f"(z),
               "f"(w)
               : "memory");
}


// Bulk fp32 add of `bytes` (a multiple of 16) from shared memory into global
// memory, both addresses 16-byte aligned; tracked by the issuing thread's
// bulk group.
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;\n" ::"l"(
                   dst),
               "r"(src), "r"(bytes)
               : "memory");
}

// Spin limit of the MMA issuers' polling loops, in SM clock cycles (about 2 s
// at 2 GHz): the loop reads the SM clock, which is cheap, rather than the
// global timer on every pass.
constexpr long long kSpinLimitCycles = 4000000000LL;

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Tensor-map element type of the inputs (fp16 or bf16).
static inline CUtensorMapDataType map_dtype(bool bf16) {
  return bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// A row-major 16-bit matrix [rows, D] of element type `dt` as a 2-D map;
// box = 64 columns x `rows_per_box` rows, 128-byte swizzle.
static inline bool encode_rows_map_t(CUtensorMap* tm, const void* ptr, int64_t rows, int64_t D,
                                     int rows_per_box, CUtensorMapDataType dt) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D * 2)};
  const cuuint32_t box[2] = {kBoxCols, static_cast<cuuint32_t>(rows_per_box)};
  const cuuint32_t estride[2] = {1, 1};
  return enc(tm, dt, 2, const_cast<void*>(ptr), dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Stage 1 for D = 64: dQ (query-major)
// ---------------------------------------------------------------------------

template <int D, int WARPS>
struct DqCfg {
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kWarpBytes = 3 * kTileBytes;  // K slot 0, K slot 1, V slot
  static constexpr int kBarOffset = WARPS * kWarpBytes;
  static constexpr int kSmemBytes = kBarOffset + WARPS * 3 * 8 + 1024;
  static constexpr int kSteps = D / 16;
};

template <int D, int WARPS, bool BF16>
__global__ void __launch_bounds__(WARPS * 32, 4)
    sel_attn_bwd_dq_kernel(const BwdProblem p, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV) {
  using C = DqCfg<D, WARPS>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * WARPS + warp;
  if (unit >= p.units) return;
  const int64_t m = unit % p.M;
  const int64_t r = unit / p.M;
  const int sub = static_cast<int>(r % p.nsub);
  const int64_t bg = r / p.nsub;
  const int g = static_cast<int>(bg % p.G);
  const int b = static_cast<int>(bg / p.G);
  const int gid = lane >> 2;
  const int tig = lane & 3;
  // heads hbase + j, j < hw; MMA columns j >= hw are padding
  const int hw = p.hpg - sub * kHeadsPerGroup < kHeadsPerGroup ? p.hpg - sub * kHeadsPerGroup
                                                                : kHeadsPerGroup;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t slots = base + warp * C::kWarpBytes;  // K0, K1, V
  const uint32_t bars = base + C::kBarOffset + warp * 24;
  if (lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    mbar_init(bars, 1);
    mbar_init(bars + 8, 1);
    mbar_init(bars + 16, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncwarp();

  const int64_t hbase = static_cast<int64_t>(g) * p.hpg + sub * kHeadsPerGroup;
  const int64_t row = (b * p.M + m) * p.H + hbase;  // first head of this warp
  // Q^T and dO^T as B operands (head gid, dims 16k + 2tig (+1, +8, +9));
  // delta of head gid from the same dO elements against O (fp32); padding
  // columns are zero
  uint32_t qf[C::kSteps][2], df[C::kSteps][2];
  float dpart = 0.f;
  {
    const bool real = gid < hw;
    const uint16_t* q = p.Q + (row + gid) * D + 2 * tig;
    const float* dob = p.dO + (row + gid) * D + 2 * tig;
    const float* ob = p.O + (row + gid) * D + 2 * tig;
#pragma unroll
    for (int k = 0; k < C::kSteps; ++k) {
      qf[k][0] = real ? __ldg(reinterpret_cast<const unsigned int*>(q + 16 * k)) : 0u;
      qf[k][1] = real ? __ldg(reinterpret_cast<const unsigned int*>(q + 16 * k + 8)) : 0u;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float2 d2 =
            real ? __ldg(reinterpret_cast<const float2*>(dob + 16 * k + 8 * h)) : float2{0.f, 0.f};
        const float2 o2 =
            real ? __ldg(reinterpret_cast<const float2*>(ob + 16 * k + 8 * h)) : float2{0.f, 0.f};
        df[k][h] = pack2_t<BF16>(d2.x, d2.y);
        dpart = fmaf(d2.x, o2.x, fmaf(d2.y, o2.y, dpart));
      }
    }
  }
  dpart += __shfl_xor_sync(kFull, dpart, 1);
  dpart += __shfl_xor_sync(kFull, dpart, 2);  // delta of head gid
  const float dla = __shfl_sync(kFull, dpart, (2 * tig) * 4);      // head 2tig
  const float dlb = __shfl_sync(kFull, dpart, (2 * tig + 1) * 4);  // head 2tig+1
  constexpr float kLog2e = 1.4426950408889634f;
  // padding columns: LSE = +inf makes their probabilities exactly 0
  const float lsa =
      2 * tig < hw ? p.LSE[(b * p.H + hbase + 2 * tig) * p.M + m] * kLog2e : INFINITY;
  const float lsb =
      2 * tig + 1 < hw ? p.LSE[(b * p.H + hbase + 2 * tig + 1) * p.M + m] * kLog2e : INFINITY;
  {
    // for stage 3: dO as fp16 rows, and one 64-byte record per (b, m, g, sub)
    if (gid < hw) {
      uint32_t* d16 = reinterpret_cast<uint32_t*>(p.dO16 + (row + gid) * D + 2 * tig);
#pragma unroll
      for (int k = 0; k < C::kSteps; ++k) {
        d16[8 * k] = df[k][0];
        d16[8 * k + 4] = df[k][1];
      }
    }
    if (tig == 0) {
      float* rec = p.rec + (((b * p.M + m) * p.G + g) * p.nsub + sub) * 16;
      rec[gid] = gid < hw ? p.LSE[(b * p.H + hbase + gid) * p.M + m] * kLog2e : INFINITY;
      rec[8 + gid] = dpart;
    }
  }

  const int lastkey = static_cast<int>(m < p.N - 1 ? m : p.N - 1);
  const int32_t* irow = p.idx + ((b * p.M + m) * p.G + g) * p.T;
  const uint64_t keep = l2_policy_evict_last();
  auto tma_tile = [&](uint32_t dst, uint32_t bar, const CUtensorMap* tm, int n0) {
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, C::kTileBytes);
#pragma unroll
    for (int h = 0; h < C::kBoxes; ++h)
      tma_load_4d(dst + h * kBoxBytes, tm, bar, h * kBoxCols, g, n0, b, keep);
  };
  const uint32_t sv = slots + 2 * C::kTileBytes;
  const uint32_t bar_v = bars + 16;

  TileWalk walk;
  walk.init(irow, static_cast<int>(p.T), p.nblk, p.bs, lastkey);
  int nA = 0, nB = 0;
  bool hA = walk.next(nA);
  bool hB = hA && walk.next(nB);
  if (lane == 0) {
    if (hA) {
      tma_tile(slots, bars, &tmK, nA);
      tma_tile(sv, bar_v, &tmV, nA);
    }
    if (hB) tma_tile(slots + C::kTileBytes, bars + 8, &tmK, nB);
  }

  float acc[C::kSteps][4];
#pragma unroll
  for (int i = 0; i < C::kSteps; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const float sl2 = p.sl2;
  const uint32_t ka = (lane & 7) * 128 + ((lane & 8) ? 8 * 128 : 0);
  const int ka_hi = lane >> 4;
  const uint32_t ta = (lane & 7) * 128 + ((lane & 16) ? 8 * 128 : 0);
  const int ta_hi = (lane >> 3) & 1;
  const int sw = lane & 7;

  // x^T (16 keys x 8 heads) = X_tile B with B given as fragments (two chains)
  auto rows_times = [&](uint32_t slot, const uint32_t(&bf)[C::kSteps][2], float (&x)[4]) {
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < C::kSteps; k += 2) {
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      ldsm_x4(slot + ka + (k >> 2) * kBoxBytes + ((((k & 3) * 2 + ka_hi) ^ sw) << 4), a0, a1,
              a2, a3);
      ldsm_x4(slot + ka + ((k + 1) >> 2) * kBoxBytes +
                  (((((k + 1) & 3) * 2 + ka_hi) ^ sw) << 4),
              b0, b1, b2, b3);
      mma_16816_t<BF16>(s, a0, a1, a2, a3, bf[k][0], bf[k][1]);
      mma_16816_t<BF16>(t, b0, b1, b2, b3, bf[k + 1][0], bf[k + 1][1]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = s[j] + t[j];
  };

  int i = 0;
  int fail = 0;  // 1: K of tile i missing, 2: V of tile i missing
  while (hA) {
    const int n0 = nA;
    const int ks = i & 1;
    const uint32_t sk = slots + ks * C::kTileBytes;
    if (!__all_sync(kFull, wait_phase(bars + 8 * ks, (i >> 1) & 1, kWaitLimitNs))) {
      fail = 1;
      break;
    }
    float x[4];
    rows_times(sk, qf, x);
    if (!__all_sync(kFull, wait_phase(bar_v, i & 1, kWaitLimitNs))) {
      fail = 2;
      break;
    }
    const bool edge = n0 + kTileKeys - 1 > lastkey;
    if (edge) {
      // zero K and V rows past the last visible key: both enter products
#pragma unroll
      for (int e = lane; e < 2 * kTileKeys * (D / 8); e += 32) {
        const int r = (e >> 1) / (D / 8), c = (e >> 1) % (D / 8);
        if (n0 + r > lastkey)
          st_shared_zero16(((e & 1) ? sv : sk) + (c >> 3) * kBoxBytes + r * 128 +
                           (((c & 7) ^ (r & 7)) << 4));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (n0 + gid > lastkey) x[0] = x[1] = -INFINITY;
      if (n0 + gid + 8 > lastkey) x[2] = x[3] = -INFINITY;
    }
    float dp[4];
    rows_times(sv, df, dp);
    __syncwarp();
    if (hB && lane == 0) tma_tile(sv, bar_v, &tmV, nB);  // V slot is free
    // P = exp(s*scale - LSE), dS = P (dP - delta); masked keys: exactly 0
    float ds[4];
    ds[0] = x[0] == -INFINITY ? 0.f : ex2(fmaf(x[0], sl2, -lsa)) * (dp[0] - dla);
    ds[1] = x[1] == -INFINITY ? 0.f : ex2(fmaf(x[1], sl2, -lsb)) * (dp[1] - dlb);
    ds[2] = x[2] == -INFINITY ? 0.f : ex2(fmaf(x[2], sl2, -lsa)) * (dp[2] - dla);
    ds[3] = x[3] == -INFINITY ? 0.f : ex2(fmaf(x[3], sl2, -lsb)) * (dp[3] - dlb);
    const uint32_t db0 = movmatrix_t(pack2_t<BF16>(ds[0], ds[1]));
    const uint32_t db1 = movmatrix_t(pack2_t<BF16>(ds[2], ds[3]));
    // dQ^T (D x 8 heads) += K_tile^T dS^T
#pragma unroll
    for (int d = 0; d < C::kSteps; ++d) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(sk + ta + (d >> 2) * kBoxBytes + ((((d & 3) * 2 + ta_hi) ^ sw) << 4), a0, a1, a2,
                a3);
      mma_16816_t<BF16>(acc[d], a0, a1, a2, a3, db0, db1);
    }
    __syncwarp();
    int nC = 0;
    const bool hC = hB && walk.next(nC);
    if (hC && lane == 0) tma_tile(sk, bars + 8 * ks, &tmK, nC);  // this K slot is free
    nA = nB;
    hA = hB;
    nB = nC;
    hB = hC;
    ++i;
  }
  if (fail) {
    if (lane == 0) report_timeout();
    if (fail == 1) wait_phase(bars + 8 * (i & 1), (i >> 1) & 1, kWaitLimitNs);
    wait_phase(bar_v, i & 1, kWaitLimitNs);
    if (hB) wait_phase(bars + 8 * ((i + 1) & 1), ((i + 1) >> 1) & 1, kWaitLimitNs);
    return;
  }
  float* o = p.dQ + (row + 2 * tig) * D + gid;
  const bool ha = 2 * tig < hw, hb = 2 * tig + 1 < hw;
#pragma unroll
  for (int d = 0; d < C::kSteps; ++d) {
    if (ha) {
      o[16 * d] = acc[d][0] * p.scale;
      o[16 * d + 8] = acc[d][2] * p.scale;
    }
    if (hb) {
      o[D + 16 * d] = acc[d][1] * p.scale;
      o[D + 16 * d + 8] = acc[d][3] * p.scale;
    }
  }
}

// ---------------------------------------------------------------------------
// Stage 1 for D = 128: per-row inputs
// ---------------------------------------------------------------------------

// Per-row inputs of the key-major kernel when it also produces dQ (D = 128):
// one warp per (b, m, g, head sub-group): dO as fp16 rows, and the 64-byte
// record (LSE * log2(e) of its 8 heads, then delta = dO . O of each head;
// padding heads get LSE = +inf and delta = 0, so their probabilities are 0).
template <int D, bool BF16>
__global__ void __launch_bounds__(256) sel_attn_bwd_prep_kernel(const BwdProblem p) {
  static_assert(D == 128, "one float4 per lane and head row");
  constexpr int kPer = D / 32;  // dims per lane
  const int lane = threadIdx.x & 31;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (unit >= p.units) return;
  const int sub = static_cast<int>(unit % p.nsub);
  const int64_t bmg = unit / p.nsub;  // (b * M + m) * G + g
  const int g = static_cast<int>(bmg % p.G);
  const int64_t bm = bmg / p.G;
  const int64_t m = bm % p.M, b = bm / p.M;
  const int hw = p.hpg - sub * kHeadsPerGroup < kHeadsPerGroup ? p.hpg - sub * kHeadsPerGroup
                                                                : kHeadsPerGroup;
  const int64_t hbase = static_cast<int64_t>(g) * p.hpg + sub * kHeadsPerGroup;
  float dl = 0.f;  // lane h < 8: delta of head h
  for (int h = 0; h < hw; ++h) {
    const int64_t at = (bm * p.H + hbase + h) * D + kPer * lane;
    float part = 0.f;
    uint32_t w[kPer / 2];
#pragma unroll
    for (int v = 0; v < kPer / 4; ++v) {
      const float4 d4 = __ldg(reinterpret_cast<const float4*>(p.dO + at) + v);
      const float4 o4 = __ldg(reinterpret_cast<const float4*>(p.O + at) + v);
      part = fmaf(d4.x, o4.x, fmaf(d4.y, o4.y, fmaf(d4.z, o4.z, fmaf(d4.w, o4.w, part))));
      w[2 * v] = pack2_t<BF16>(d4.x, d4.y);
      w[2 * v + 1] = pack2_t<BF16>(d4.z, d4.w);
    }
    *reinterpret_cast<uint2*>(p.dO16 + at) = make_uint2(w[0], w[1]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
    if (lane == h) dl = part;
  }
  if (lane < kHeadsPerGroup) {
    constexpr float kLog2e = 1.4426950408889634f;
    float* rec = p.rec + unit * 16;
    rec[lane] = lane < hw ? p.LSE[(b * p.H + hbase + lane) * p.M + m] * kLog2e : INFINITY;
    rec[8 + lane] = lane < hw ? dl : 0.f;
  }
}

// ---------------------------------------------------------------------------
// Stage 2: transposed index (who selected each (b, g, block))
// ---------------------------------------------------------------------------

// The local blocks of a query in block row c (queries c*bs .. c*bs + bs - 1):
// slot 0 = its own block c, slot 1 = block c - 1; -1 for any other block.
__device__ __forceinline__ int local_slot(int t, int c) {
  if (t == c) return 0;
  if (t == c - 1) return 1;
  return -1;
}

// The count walks the index in units of (b, g, 32 consecutive queries):
// lane l takes query m0 + l and its row's entries in order. Entry j -> the
// list it files into, or -1: padding, out of range, wholly in the query's
// future, or taken by the local-block kernel (with lfirst: the row's first
// entry of each local block, recorded in `first`).
struct RowWalk {
  int64_t b, m, row;  // row = (b * M + m) * G + g
  int g, c, lastkey;
  bool live;
  int first[2];
  __device__ __forceinline__ RowWalk(const BwdProblem& p, int64_t unit, int lane) {
    const int64_t nmw = (p.M + 31) / 32;
    const int64_t bg = unit / nmw;
    g = static_cast<int>(bg % p.G);
    b = bg / p.G;
    m = (unit % nmw) * 32 + lane;
    live = m < p.M;
    row = (b * p.M + m) * p.G + g;
    c = static_cast<int>(m / p.bs);
    lastkey = static_cast<int>(m < p.N - 1 ? m : p.N - 1);
    first[0] = first[1] = -1;
  }
  __device__ __forceinline__ int list_of(const BwdProblem& p, int j) {
    if (!live) return -1;
    const int t = __ldg(p.idx + row * p.T + j);
    if (t < 0 || t >= p.nblk || static_cast<int64_t>(t) * p.bs > lastkey) return -1;
    if (p.lfirst != nullptr) {
      const int s = local_slot(t, c);
      if (s >= 0 && first[s] < 0) {
        first[s] = j;
        return -1;
      }
    }
    return static_cast<int>((b * p.G + g) * p.nblk + t);
  }
};

// Per list, the number of entries it gets. Lanes filing into the same list
// (block 0 and the local blocks, which neighbouring queries share) add with
// one atomic. With lfirst, each row's local entries are recorded there.
__global__ void csr_count_kernel(const BwdProblem p, int* count) {
  const int lane = threadIdx.x & 31;
  const int64_t nu = p.B * p.G * ((p.M + 31) / 32);
  for (int64_t u = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; u < nu;
       u += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
    RowWalk w(p, u, lane);
    for (int j = 0; j < p.T; ++j) {
      const int l = w.list_of(p, j);
      const unsigned peers = __match_any_sync(kFull, l);
      if (l >= 0 && lane == __ffs(peers) - 1) atomicAdd(count + l, __popc(peers));
    }
    if (w.live && p.lfirst != nullptr) p.lfirst[w.row] = make_int2(w.first[0], w.first[1]);
  }
}

// Exclusive scans of count[] and of ceil(count / chunk) over L lists, one CTA
// of 1024 threads walking the array in tiles; offs[L] and choffs[L] get totals.
__global__ void __launch_bounds__(1024) csr_scan_kernel(const int* count, int* offs, int* choffs,
                                                        int L, int chunk) {
  __shared__ int wsum[2][32];
  __shared__ int carry[2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry[0] = carry[1] = 0;
  __syncthreads();
  for (int base = 0; base < L; base += 1024) {
    const int i = base + threadIdx.x;
    const int c = i < L ? count[i] : 0;
    const int k = (c + chunk - 1) / chunk;
    int sc = c, sk = k;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int a = __shfl_up_sync(kFull, sc, off), bb = __shfl_up_sync(kFull, sk, off);
      if (lane >= off) {
        sc += a;
        sk += bb;
      }
    }
    if (lane == 31) {
      wsum[0][warp] = sc;
      wsum[1][warp] = sk;
    }
    __syncthreads();
    if (warp == 0) {
      int a = wsum[0][lane], bb = wsum[1][lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int x = __shfl_up_sync(kFull, a, off), y = __shfl_up_sync(kFull, bb, off);
        if (lane >= off) {
          a += x;
          bb += y;
        }
      }
      wsum[0][lane] = a;
      wsum[1][lane] = bb;
    }
    __syncthreads();
    const int pc = carry[0] + (warp ? wsum[0][warp - 1] : 0) + sc - c;
    const int pk = carry[1] + (warp ? wsum[1][warp - 1] : 0) + sk - k;
    if (i < L) {
      offs[i] = pc;
      choffs[i] = pk;
    }
    __syncthreads();
    if (threadIdx.x == 1023) {
      carry[0] = pc + c;
      carry[1] = pk + k;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    offs[L] = carry[0];
    choffs[L] = carry[1];
  }
}

// chunk -> the list it belongs to (chunks of list l: choffs[l] .. choffs[l + 1])
__global__ void csr_chunk_list_kernel(const int* choffs, int L, int* chunk_list) {
  for (int l = blockIdx.x * blockDim.x + threadIdx.x; l < L; l += gridDim.x * blockDim.x)
    for (int c = choffs[l]; c < choffs[l + 1]; ++c) chunk_list[c] = l;
}

// Launch order of the key-major tensor-core kernel's chunks (D = 128).
// Numbered list by list, the CTAs in flight at any moment would work on ~150
// consecutive blocks, whose queries span the whole sequence: the dQ rows they
// add into (one 4 KB row per query and head group) would be scattered over
// all of dQ, and every fp32 reduction would be a read-modify-write in HBM.
// Ordered by the mean query position of each chunk (in buckets of
// kOrderQueries positions, per (b, g)), the CTAs in flight add into a band of
// dQ rows that L2 can hold, so most of a row's reductions from its blocks
// meet in L2. Lists fill in roughly increasing query order (the fill walks
// the index tensor in order), so a chunk covers a contiguous stretch of its
// list's queries.
#ifndef NSA_BWD_ORDER_QUERIES
#define NSA_BWD_ORDER_QUERIES 512
#endif
constexpr int kOrderQueries = NSA_BWD_ORDER_QUERIES;

// One warp per chunk: its bucket (b, g, mean query / kOrderQueries), counted.
__global__ void chunk_key_kernel(const BwdProblem p, int nbkt, int* key, int* bcount) {
  const int64_t c = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (c >= p.choffs[p.L]) return;
  const int l = __ldg(p.chunk_list + c);
  const int q0 = p.offs[l] + (static_cast<int>(c) - p.choffs[l]) * kQueriesPerChunk;
  const int nq = min(q0 + kQueriesPerChunk, p.offs[l + 1]) - q0;  // >= 1
  long long sum = 0;
  for (int i = lane; i < nq; i += 32) sum += __ldg(p.lists + q0 + i);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
  if (lane == 0) {
    const int bg = l / p.nblk;
    const int bk = static_cast<int>(sum / nq) / kOrderQueries;
    const int k = bg * nbkt + min(bk, nbkt - 1);
    key[c] = k;
    atomicAdd(bcount + k, 1);
  }
}

__global__ void chunk_order_fill_kernel(const BwdProblem p, const int* key, const int* boffs,
                                        int* bcursor, int* order) {
  const int nch = p.choffs[p.L];
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < nch; c += gridDim.x * blockDim.x) {
    const int k = key[c];
    order[boffs[k] + atomicAdd(bcursor + k, 1)] = c;
  }
}

// Each list's entries (query ids). Threads take the index entries in order
// (grid-stride), so the few hundred rows in flight at a time keep every
// list in roughly increasing query order, which the chunks' launch order
// relies on. Entries the count recorded in lfirst are left out.
__global__ void csr_fill_kernel(const BwdProblem p, int* cursor, int* lists) {
  const int64_t total = p.B * p.M * p.G * p.T;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = e / p.T;  // (b * M + m) * G + g
    const int j = static_cast<int>(e - r * p.T);
    const int g = static_cast<int>(r % p.G);
    const int64_t bm = r / p.G;
    const int64_t m = bm % p.M, b = bm / p.M;
    const int t = __ldg(p.idx + e);
    const int64_t lastkey = m < p.N - 1 ? m : p.N - 1;
    if (t < 0 || t >= p.nblk || static_cast<int64_t>(t) * p.bs > lastkey) continue;
    if (p.lfirst != nullptr) {
      const int s = local_slot(t, static_cast<int>(m / p.bs));
      if (s >= 0) {
        const int2 f = p.lfirst[r];
        if ((s == 0 ? f.x : f.y) == j) continue;
      }
    }
    const int l = static_cast<int>((b * p.G + g) * p.nblk + t);
    lists[p.offs[l] + atomicAdd(cursor + l, 1)] = static_cast<int>(m);
  }
}

// ---------------------------------------------------------------------------
// Stage 3 for D = 64: dK, dV (key-major)
// ---------------------------------------------------------------------------

template <int D, int KT>
struct DkvCfg {
  static constexpr int kWarps = 2 * KT;                       // (16-key tile, half of D)
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kBoxBytesBlk = KT * kTileKeys * 128;   // one box of bs rows
  static constexpr int kBlockBytes = kBoxes * kBoxBytesBlk;   // K (or V) block
  static constexpr int kRowBox = 8 * 128;                     // 8 head rows x 64 dims
  static constexpr int kRecOffset = 2 * kBoxes * kRowBox;     // after the Q and dO boxes
  static constexpr int kStageBytes = kRecOffset + 1024;       // record, keeps 1 KB alignment
  // queries in flight: their Q / dO rows sit at random places in memory, so
  // the ring must cover a DRAM round trip of several query iterations
  static constexpr int kStages = 16;
  static constexpr int kStageOffset = 2 * kBlockBytes;
  static constexpr int kBarOffset = kStageOffset + kStages * kStageBytes;
  static constexpr int kListOffset = kBarOffset + (1 + 2 * kStages) * 8;
  static constexpr int kSmemBytes = kListOffset + kQueriesPerChunk * 4 + 1024;
  static constexpr int kSteps = D / 16;
  static constexpr int kHalfTiles = D / 16;                   // 8-dim n-tiles per half of D
};

// SPLIT: the group has more than 8 heads (items are (query, sub-group) pairs);
// otherwise one item per query.
template <int D, int KT, bool SPLIT, bool BF16>
__global__ void __launch_bounds__(2 * KT * 32, 1)
    sel_attn_bwd_dkv_kernel(const BwdProblem p, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmD) {
  using C = DkvCfg<D, KT>;
  extern __shared__ uint8_t smem_raw[];
  const int c = blockIdx.x;
  if (c >= p.choffs[p.L]) return;
  const int l = __ldg(p.chunk_list + c);  // the list of this chunk
  const int q0 = p.offs[l] + (c - p.choffs[l]) * kQueriesPerChunk;
  const int nq = min(q0 + kQueriesPerChunk, p.offs[l + 1]) - q0;
  const int nsub = SPLIT ? p.nsub : 1;
  const int nitems = nq * nsub;  // (query, sub-group of 8 heads) pairs
  const int t = l % p.nblk;
  const int bg = l / p.nblk;
  const int g = bg % static_cast<int>(p.G);
  const int b = bg / static_cast<int>(p.G);
  const int64_t hgroup = static_cast<int64_t>(g) * p.hpg;  // first head of the group
  const int hw0 = p.hpg < kHeadsPerGroup ? p.hpg : kHeadsPerGroup;  // head rows per item

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kt = warp >> 1;  // 16-key tile of the block
  const int dh = warp & 1;   // half of D this warp accumulates
  const int gid = lane >> 2;
  const int tig = lane & 3;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = base, sV = base + C::kBlockBytes;
  const uint32_t stages = base + C::kStageOffset;
  const uint32_t bar_blk = base + C::kBarOffset;
  const uint32_t full = bar_blk + 8, empty = full + 8 * C::kStages;
  const int n_blk = t * p.bs;  // first key of the block
  const float* stage_rec = reinterpret_cast<const float*>(smem_raw + (base - smem_u32(smem_raw)) +
                                                          C::kStageOffset + C::kRecOffset);

  int* qlist = reinterpret_cast<int*>(smem_raw + (base - smem_u32(smem_raw)) + C::kListOffset);
  // item i of the chunk -> stage i % kStages (its Q and dO head rows, record)
  auto issue_query = [&](int i) {
    const int s = i % C::kStages;
    const uint32_t st = stages + s * C::kStageBytes;
    const int m = qlist[SPLIT ? i / nsub : i];
    const int sub = SPLIT ? i % nsub : 0;
    const int qrow = static_cast<int>((b * p.M + m) * p.H + hgroup + sub * kHeadsPerGroup);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(full + 8 * s, 2 * C::kBoxes * hw0 * 128 + 64);
#pragma unroll
    for (int h = 0; h < C::kBoxes; ++h) {
      tma_load_2d(st + h * C::kRowBox, &tmQ, full + 8 * s, h * kBoxCols, qrow);
      tma_load_2d(st + (C::kBoxes + h) * C::kRowBox, &tmD, full + 8 * s, h * kBoxCols, qrow);
    }
    bulk_load(st + C::kRecOffset, p.rec + (((b * p.M + m) * p.G + g) * nsub + sub) * 16, 64,
              full + 8 * s);
  };

  for (int j = threadIdx.x; j < nq; j += blockDim.x) qlist[j] = __ldg(p.lists + q0 + j);
  if (hw0 < kHeadsPerGroup) {
    // head rows the copies never write (groups of fewer than 8 heads): zero,
    // so the padding columns multiply zeros
    const int per_stage = 2 * C::kBoxes * (kHeadsPerGroup - hw0) * 8;  // 16-byte pieces
    for (int e = threadIdx.x; e < C::kStages * per_stage; e += blockDim.x) {
      const int s = e / per_stage, r = e % per_stage;
      const int box = r / ((kHeadsPerGroup - hw0) * 8);
      const int row = hw0 + (r / 8) % (kHeadsPerGroup - hw0);
      st_shared_zero16(stages + s * C::kStageBytes + box * C::kRowBox + row * 128 + (r % 8) * 16);
    }
  }
  if (threadIdx.x == 0) {
    const uint64_t keep = l2_policy_evict_last();
    mbar_init(bar_blk, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, C::kWarps);
    }
    fence_mbar_init();
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar_blk, 2 * C::kBlockBytes);
#pragma unroll
    for (int h = 0; h < C::kBoxes; ++h) {
      tma_load_4d(sK + h * C::kBoxBytesBlk, &tmK, bar_blk, h * kBoxCols, g, n_blk, b, keep);
      tma_load_4d(sV + h * C::kBoxBytesBlk, &tmV, bar_blk, h * kBoxCols, g, n_blk, b, keep);
    }
  }
  __syncthreads();  // barriers initialised, query list in shared memory
  if (threadIdx.x == 0)
    for (int i = 0; i < nitems && i < C::kStages; ++i) issue_query(i);
  int issued = nitems < C::kStages ? nitems : C::kStages;  // meaningful in warp 0 only
  bool ok = __all_sync(kFull, wait_phase(bar_blk, 0, kWaitLimitNs));

  // this warp's 16 keys of K and V as cached A fragments (all of D)
  const int nw0 = n_blk + kt * kTileKeys;
  uint32_t kf[C::kSteps][4], vf[C::kSteps][4];
  if (ok) {
    const uint32_t ka = (lane & 7) * 128 + ((lane & 8) ? 8 * 128 : 0);
    const int ka_hi = lane >> 4;
    const int sw = lane & 7;
#pragma unroll
    for (int k = 0; k < C::kSteps; ++k) {
      const uint32_t off = kt * kTileKeys * 128 + ka + (k >> 2) * C::kBoxBytesBlk +
                           ((((k & 3) * 2 + ka_hi) ^ sw) << 4);
      ldsm_x4(sK + off, kf[k][0], kf[k][1], kf[k][2], kf[k][3]);
      ldsm_x4(sV + off, vf[k][0], vf[k][1], vf[k][2], vf[k][3]);
    }
  }
  const float sl2 = p.sl2;
  float dk[C::kHalfTiles][4], dv[C::kHalfTiles][4];
#pragma unroll
  for (int j = 0; j < C::kHalfTiles; ++j)
    dk[j][0] = dk[j][1] = dk[j][2] = dk[j][3] = dv[j][0] = dv[j][1] = dv[j][2] = dv[j][3] = 0.f;
  // ldmatrix of a stage's head rows: tile = lane >> 3, row = head lane & 7
  const int qrow_l = lane & 7;
  const int qtile = lane >> 3;

  using Frag = uint32_t[C::kSteps][2];
  // Query i's Q / dO fragments, record and position into registers; the stage
  // is released right away (and warp 0 refills it) so that the next query's
  // copy overlaps this one's arithmetic.
  auto fetch = [&](int i, Frag& qf, Frag& df, float (&rc)[4], int& m) -> bool {
    const int s = i % C::kStages;
    const uint32_t ph = (i / C::kStages) & 1;
    const uint32_t st = stages + s * C::kStageBytes;
    if (!__all_sync(kFull, wait_phase(full + 8 * s, ph, kWaitLimitNs))) return false;
#pragma unroll
    for (int k = 0; k < C::kSteps; k += 2) {
      const int cc = 2 * k + qtile;  // 16-byte column chunk of D
      const uint32_t off = (cc >> 3) * C::kRowBox + qrow_l * 128 + (((cc & 7) ^ qrow_l) << 4);
      ldsm_x4(st + off, qf[k][0], qf[k][1], qf[k + 1][0], qf[k + 1][1]);
      ldsm_x4(st + C::kBoxes * C::kRowBox + off, df[k][0], df[k][1], df[k + 1][0], df[k + 1][1]);
    }
    const float* rec = stage_rec + s * (C::kStageBytes / 4);
    rc[0] = rec[2 * tig];
    rc[1] = rec[2 * tig + 1];
    rc[2] = rec[8 + 2 * tig];
    rc[3] = rec[8 + 2 * tig + 1];
    m = qlist[SPLIT ? i / nsub : i];
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + 8 * s);
    if (warp == 0 && i + C::kStages < nitems) {
      // refill the stage once every warp has taken its copy
      if (!__all_sync(kFull, wait_phase(empty + 8 * s, ph, kWaitLimitNs))) return false;
      if (lane == 0) issue_query(i + C::kStages);
      issued = i + C::kStages + 1;
    }
    return true;
  };

  auto compute = [&](const Frag& qf, const Frag& df, const float (&rc)[4], int m) {
    const int lastkey = static_cast<int>(m < p.N - 1 ? m : p.N - 1);
    if (nw0 > lastkey) return;  // all of this warp's keys are in the query's future
    // S^T and dP^T (16 keys x 8 heads), two chains each
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < C::kSteps; k += 2) {
      mma_16816_t<BF16>(s0, kf[k][0], kf[k][1], kf[k][2], kf[k][3], qf[k][0], qf[k][1]);
      mma_16816_t<BF16>(d0, vf[k][0], vf[k][1], vf[k][2], vf[k][3], df[k][0], df[k][1]);
      mma_16816_t<BF16>(s1, kf[k + 1][0], kf[k + 1][1], kf[k + 1][2], kf[k + 1][3], qf[k + 1][0],
                qf[k + 1][1]);
      mma_16816_t<BF16>(d1, vf[k + 1][0], vf[k + 1][1], vf[k + 1][2], vf[k + 1][3], df[k + 1][0],
                df[k + 1][1]);
    }
    const bool va = nw0 + gid <= lastkey, vb = nw0 + gid + 8 <= lastkey;
    float pr[4], ds[4];
    pr[0] = va ? ex2(fmaf(s0[0] + s1[0], sl2, -rc[0])) : 0.f;
    pr[1] = va ? ex2(fmaf(s0[1] + s1[1], sl2, -rc[1])) : 0.f;
    pr[2] = vb ? ex2(fmaf(s0[2] + s1[2], sl2, -rc[0])) : 0.f;
    pr[3] = vb ? ex2(fmaf(s0[3] + s1[3], sl2, -rc[1])) : 0.f;
    ds[0] = va ? pr[0] * (d0[0] + d1[0] - rc[2]) : 0.f;
    ds[1] = va ? pr[1] * (d0[1] + d1[1] - rc[3]) : 0.f;
    ds[2] = vb ? pr[2] * (d0[2] + d1[2] - rc[2]) : 0.f;
    ds[3] = vb ? pr[3] * (d0[3] + d1[3] - rc[3]) : 0.f;
    // A operands (16 keys x 8 heads): the C layout of S^T is the A layout of
    // m16n8k8; B operands (8 heads x 8 dims) are transposed Q / dO fragments
    const uint32_t pa0 = pack2_t<BF16>(pr[0], pr[1]), pa1 = pack2_t<BF16>(pr[2], pr[3]);
    const uint32_t sa0 = pack2_t<BF16>(ds[0], ds[1]), sa1 = pack2_t<BF16>(ds[2], ds[3]);
    // this warp's half of D (branch on the warp-uniform half so that every
    // fragment index is a compile-time constant)
    auto accumulate = [&](auto half) {
      constexpr int h0 = decltype(half)::value * C::kHalfTiles;
#pragma unroll
      for (int jj = 0; jj < C::kHalfTiles; ++jj) {
        const int j = h0 + jj;  // 8-dim tile of D
        mma_1688_t<BF16>(dv[jj], pa0, pa1, movmatrix_t(df[j >> 1][j & 1]));
        mma_1688_t<BF16>(dk[jj], sa0, sa1, movmatrix_t(qf[j >> 1][j & 1]));
      }
    };
    if (dh == 0)
      accumulate(std::integral_constant<int, 0>{});
    else
      accumulate(std::integral_constant<int, 1>{});
  };

  // queries alternate between two register sets (A, B): query i+1 is fetched
  // before query i is computed
  uint32_t qa[C::kSteps][2], da[C::kSteps][2], qb[C::kSteps][2], db[C::kSteps][2];
  float ra[4], rb[4];
  int ma = 0, mb = 0;
  int i = 0;         // next query to compute
  int failed_at = -1;
  if (ok && nitems > 0 && !fetch(0, qa, da, ra, ma)) failed_at = 0;
  if (!ok) failed_at = 0;
  while (failed_at < 0 && i < nitems) {
    if (i + 1 < nitems && !fetch(i + 1, qb, db, rb, mb)) {
      failed_at = i + 1;
      break;
    }
    compute(qa, da, ra, ma);
    if (++i >= nitems) break;
    if (i + 1 < nitems && !fetch(i + 1, qa, da, ra, ma)) {
      failed_at = i + 1;
      break;
    }
    compute(qb, db, rb, mb);
    ++i;
  }
  if (failed_at >= 0) {
    // let every copy this CTA requested land before it can exit
    if (lane == 0) report_timeout();
    if (threadIdx.x == 0) {
      wait_phase(bar_blk, 0, kWaitLimitNs);
      for (int j = failed_at; j < issued; ++j)
        wait_phase(full + 8 * (j % C::kStages), (j / C::kStages) & 1, kWaitLimitNs);
    }
    return;
  }

  // add this chunk's partial sums into dK / dV (rows past N are not written)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int n = nw0 + gid + 8 * r;
    if (n >= p.N) continue;
    float* dkr = p.dK + ((b * p.N + n) * p.G + g) * D + dh * (D / 2) + 2 * tig;
    float* dvr = p.dV + ((b * p.N + n) * p.G + g) * D + dh * (D / 2) + 2 * tig;
#pragma unroll
    for (int jj = 0; jj < C::kHalfTiles; ++jj) {
      atomicAdd(reinterpret_cast<float2*>(dkr + 8 * jj),
                make_float2(dk[jj][2 * r] * p.scale, dk[jj][2 * r + 1] * p.scale));
      atomicAdd(reinterpret_cast<float2*>(dvr + 8 * jj),
                make_float2(dv[jj][2 * r], dv[jj][2 * r + 1]));
    }
  }
}

// ---------------------------------------------------------------------------
// Stage 3 on the 5th-generation tensor cores (D = 128): dK, dV and dQ
// (key-major)
// ---------------------------------------------------------------------------
//
// One CTA per chunk of <= kQueriesPerChunk items of a list (as above). The
// items (query, head sub-group) are taken 16 at a time: their 8 head rows
// each are exactly one 1024-byte 128B-swizzled group, so 16 items gathered
// by TMA form 128-row Q and dO operand tiles without any reshuffling.
// Per batch of 128 rows, with the block's 64 keys (a block of 32 is read as
// 32 rows of a 64-row tile whose other rows are zero):
//   S  = Q_R K^T,  dP = dO_R V^T       (M = 128 rows, N = 64 keys, K = D)
//   P  = 2^(S scale log2e - LSE log2e), dS = P (dP - delta)  (softmax warps,
//        one row per thread; masked and padding rows give exact zeros)
//   dV^T += dO_R^T P,  dK^T += Q_R^T dS  (M = D = 128, N = 64, K = 128 rows;
//        the Q / dO tiles serve again as MN-major A operands, P and dS are
//        written to shared memory as MN-major B operands)
//   dQ_R = dS K  (M = 128 rows, N = D, K = 64 keys; dS read as a K-major A
//        operand, the K tile as an MN-major B operand)
// with S / dP double-buffered in tensor memory and the Q / dO tiles in a
// 2-stage ring, so the next batch's S and dP overlap this batch's softmax.
// The softmax warps read each batch's dQ_R out of tensor memory after the
// next batch's softmax, stage it through their rows of the batch's (then
// free) P / dS buffer and add it into dQ with 16-byte fp32 reductions, 16
// lanes per 256 contiguous bytes. dV^T and dK^T accumulate in tensor memory
// over the chunk and are added into dK / dV with fp32 atomics at the end
// (lane = d, coalesced per key).
// Warps: 0 producer (one lane), 1 tensor-memory owner and MMA issuer (one
// lane), 2-5 softmax and epilogue. Every wait is bounded.

// A row-major fp16 matrix [rows, 128] as a 3-D map (64 columns, rows, 2
// column halves); box = 64 x `rows_per_box` x 2: one copy brings both halves
// of `rows_per_box` rows, landing as two consecutive 128B-swizzled groups
// (half 0's rows, then half 1's).
static inline bool encode_rows_halves_map(CUtensorMap* tm, const void* ptr, int64_t rows,
                                          int rows_per_box, CUtensorMapDataType dt) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), 2};
  const cuuint64_t strides[2] = {128 * 2, 64 * 2};  // next row, next half (bytes)
  const cuuint32_t box[3] = {kBoxCols, static_cast<cuuint32_t>(rows_per_box), 2};
  const cuuint32_t estride[3] = {1, 1, 1};
  return enc(tm, dt, 3, const_cast<void*>(ptr), dims, strides, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kTcBatch = 16;  // items per batch: 128 rows
enum DkvBar : int {
  kBlkFull = 0,
  kQdFull = 1,    // 2 stages
  kQdEmpty = 3,   // 2
  kSdFull = 5,    // 2 S / dP buffers
  kPdsFull = 7,   // 2 P / dS buffers
  kPdsFree = 9,   // 2
  kAccDone = 11,
  kDqFull = 12,   // dQ of a batch is in tensor memory
  kDqFree = 13,   // the dQ warps have read it
  kStaged = 14,   // the chunk's dV / dK staged in shared memory
  kDkvBars = 15
};

// Q / dO tiles of a batch: item j's 8 head rows at j * 2048, dims 0-63 in
// the first 1024 bytes and dims 64-127 in the next (one 3-D copy per item);
// 8-row groups of one column half are 2048 bytes apart.
struct DkvTcCfg {
  static constexpr int kAtom = 128 * 128;    // 128 rows x 128 B
  static constexpr int kItemBytes = 2048;    // 8 rows x 2 halves x 128 B
  static constexpr int kBlkAtom = 64 * 128;  // 64 keys x 128 B
  static constexpr int kOffK = 0;            // 2 atoms (d 0-63, 64-127)
  static constexpr int kOffV = kOffK + 2 * kBlkAtom;
  static constexpr int kOffStage = kOffV + 2 * kBlkAtom;
  static constexpr int kStageBytes = 4 * kAtom;  // Q tile (2 atoms), dO tile (2 atoms)
  static constexpr int kOffPds = kOffStage + 2 * kStageBytes;
  static constexpr int kPdsBytes = 2 * 128 * 128;  // P tile, dS tile (128 rows x 64 keys)
  static constexpr int kOffBar = kOffPds + 2 * kPdsBytes;
  static constexpr int kOffTmem = kOffBar + kDkvBars * 8;
  static constexpr int kOffList = kOffTmem + 16;  // the chunk's query ids
  static constexpr int kSmemBytes = kOffList + kQueriesPerChunk * 4 + 1024;
  static constexpr uint32_t kColS = 0, kColDp = 128, kColDv = 256, kColDk = 320, kColDq = 384;
};
static_assert(DkvTcCfg::kSmemBytes <= 232448, "one CTA per SM within 227 KB");

constexpr int kDkvTcThreads = 320;

template <bool SPLIT, bool BF16>
__global__ void __launch_bounds__(kDkvTcThreads, 1)
    sel_attn_bwd_dkv_tc_kernel(const BwdProblem p, const __grid_constant__ CUtensorMap tmK,
                               const __grid_constant__ CUtensorMap tmV,
                               const __grid_constant__ CUtensorMap tmQ,
                               const __grid_constant__ CUtensorMap tmD) {
  using C = DkvTcCfg;
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  if (static_cast<int>(blockIdx.x) >= p.choffs[p.L]) return;  // before any tensor memory is taken
  const int c = p.chunk_order ? __ldg(p.chunk_order + blockIdx.x) : static_cast<int>(blockIdx.x);
  const int l = __ldg(p.chunk_list + c);
  const int q0 = p.offs[l] + (c - p.choffs[l]) * kQueriesPerChunk;
  const int nq = min(q0 + kQueriesPerChunk, p.offs[l + 1]) - q0;
  const int nsub = SPLIT ? p.nsub : 1;
  const int nitems = nq * nsub;
  const int nbat = (nitems + kTcBatch - 1) / kTcBatch;
  const int t = l % p.nblk;
  const int bg = l / p.nblk;
  const int g = bg % static_cast<int>(p.G);
  const int b = bg / static_cast<int>(p.G);
  const int64_t hgroup = static_cast<int64_t>(g) * p.hpg;
  const int hw0 = p.hpg < kHeadsPerGroup ? p.hpg : kHeadsPerGroup;  // head rows per item
  const int n_blk = t * p.bs;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  auto bar = [&](int i) { return base + C::kOffBar + 8u * static_cast<uint32_t>(i); };
  int* const qlist = reinterpret_cast<int*>(gbase + C::kOffList);
  for (int j = threadIdx.x; j < nq; j += blockDim.x) qlist[j] = __ldg(p.lists + q0 + j);
  auto item_query = [&](int item, int& m, int& sub) {
    m = qlist[SPLIT ? item / nsub : item];
    sub = SPLIT ? item % nsub : 0;
  };

  if (hw0 < kHeadsPerGroup) {
    // head rows the copies never write (groups of fewer than 8 heads): zero,
    // so the padding rows multiply zeros
    // (stage, tensor, item, half) groups x (8 - hw0) rows x 8 pieces of 16 bytes
    const int per = 2 * 2 * kTcBatch * 2 * (kHeadsPerGroup - hw0) * 8;
    for (int e = threadIdx.x; e < per; e += blockDim.x) {
      const int piece = e % 8, rr = e / 8;
      const int row = hw0 + rr % (kHeadsPerGroup - hw0);
      const int grp = rr / (kHeadsPerGroup - hw0);  // 1024-byte group: item-half of a tile
      st_shared_zero16(base + C::kOffStage + grp * 1024 + row * 128 + piece * 16);
    }
    fence_proxy_async_smem();
  }
  if (p.bs < 64) {
    // a block of 32 keys arrives as 32 rows of each K / V column half; the
    // other 32 rows stay zero (dQ multiplies every row of the tile)
    const int per = 4 * (64 - p.bs) * 8;  // (tensor, half) x rows x 16-byte pieces
    for (int e = threadIdx.x; e < per; e += blockDim.x) {
      const int piece = e % 8, rr = e / 8;
      const int row = p.bs + rr % (64 - p.bs), atom = rr / (64 - p.bs);  // K0, K1, V0, V1
      st_shared_zero16(base + C::kOffK + atom * C::kBlkAtom + row * 128 + piece * 16);
    }
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(kBlkFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kQdFull + s), 1);
      mbar_init(bar(kQdEmpty + s), 1);
      mbar_init(bar(kSdFull + s), 1);
      mbar_init(bar(kPdsFull + s), 4 * 32);
      mbar_init(bar(kPdsFree + s), 1);
    }
    mbar_init(bar(kAccDone), 1);
    mbar_init(bar(kDqFull), 1);
    mbar_init(bar(kDqFree), 4 * 32);
    mbar_init(bar(kStaged), 4 * 32);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc_alloc(base + C::kOffTmem, 512);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kOffTmem);
  bool failed = false;

  if (warp == 0) {
    // ---- producer: the block's K / V (64 keys), then Q / dO rows per batch;
    // lane j < 16 issues the copies of item j of a batch ----
    const uint64_t keep = l2_policy_evict_last();
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(kBlkFull), 4 * p.bs * 128);
      for (int a = 0; a < 2; ++a) {
        tma_load_4d(base + C::kOffK + a * C::kBlkAtom, &tmK, bar(kBlkFull), a * kBoxCols, g,
                    n_blk, b, keep);
        tma_load_4d(base + C::kOffV + a * C::kBlkAtom, &tmV, bar(kBlkFull), a * kBoxCols, g,
                    n_blk, b, keep);
      }
    }
    // the rows of batch i into L2 (lane j: item j), ahead of their copies
    auto prefetch = [&](int i) {
      if (i < nbat && lane < kTcBatch) {
        int m, sub;
        item_query(min(i * kTcBatch + lane, nitems - 1), m, sub);
        const int qrow = static_cast<int>((b * p.M + m) * p.H + hgroup + sub * kHeadsPerGroup);
        if (hw0 == kHeadsPerGroup) {
          tma_prefetch_l2_3d(&tmQ, 0, qrow, 0);
          tma_prefetch_l2_3d(&tmD, 0, qrow, 0);
        } else {
          for (int a = 0; a < 2; ++a) {
            tma_prefetch_l2_2d(&tmQ, a * kBoxCols, qrow);
            tma_prefetch_l2_2d(&tmD, a * kBoxCols, qrow);
          }
        }
      }
    };
    // batch i's copies first, then the L2 prefetches of the batches two
    // ahead, so the chunk's first copies do not queue behind prefetches
    for (int i = 0; i < nbat && !failed; ++i) {
      const int s = i & 1;
      if (i >= 2 &&
          !__all_sync(kFull, wait_phase(bar(kQdEmpty + s), ((i - 2) >> 1) & 1, kWaitLimitNs))) {
        failed = true;
        break;
      }
      const uint32_t st = base + C::kOffStage + s * C::kStageBytes;
      if (lane == 0) mbar_arrive_expect_tx(bar(kQdFull + s), kTcBatch * 4 * hw0 * 128);
      __syncwarp();
      if (lane < kTcBatch) {
        // items past the chunk repeat its last item (their rows are masked)
        const int item = min(i * kTcBatch + lane, nitems - 1);
        int m, sub;
        item_query(item, m, sub);
        const int qrow = static_cast<int>((b * p.M + m) * p.H + hgroup + sub * kHeadsPerGroup);
        const uint32_t dq = st + lane * C::kItemBytes, dd = dq + 2 * C::kAtom;
        if (hw0 == kHeadsPerGroup) {  // both column halves in one 3-D copy
          tma_load_3d(dq, &tmQ, bar(kQdFull + s), 0, qrow, 0);
          tma_load_3d(dd, &tmD, bar(kQdFull + s), 0, qrow, 0);
        } else {  // fewer head rows: one 2-D copy per column half
          for (int a = 0; a < 2; ++a) {
            tma_load_2d(dq + a * 1024, &tmQ, bar(kQdFull + s), a * kBoxCols, qrow);
            tma_load_2d(dd + a * 1024, &tmD, bar(kQdFull + s), a * kBoxCols, qrow);
          }
        }
      }
      if (i == 0) prefetch(1);
      prefetch(i + 2);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      constexpr uint32_t idesc_sd = umma_idesc_f16(128, 64, BF16, false);   // K-major A, B
      constexpr uint32_t idesc_acc =
          umma_idesc_f16(128, 64, BF16, true) | (1u << 15);  // MN-major A and B
      bool ok = wait_phase(bar(kBlkFull), 0, kWaitLimitNs);
      // S / dP of batch i: its Q / dO rows have landed (caller checked)
      auto issue_sd = [&](int i) {
        const int s = i & 1;
        tc_fence_after();
        const uint32_t st = base + C::kOffStage + s * C::kStageBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t offa = (k >> 2) * 1024 + (k & 3) * 32;  // column half, then 16 dims
          const uint32_t offb = (k >> 2) * C::kBlkAtom + (k & 3) * 32;
          tc_mma(tmem + C::kColS + 64 * s, umma_desc_sw128(st + offa, 16, C::kItemBytes),
                 umma_desc_sw128(base + C::kOffK + offb, 16), idesc_sd, k > 0 ? 1u : 0u);
          tc_mma(tmem + C::kColDp + 64 * s,
                 umma_desc_sw128(st + 2 * C::kAtom + offa, 16, C::kItemBytes),
                 umma_desc_sw128(base + C::kOffV + offb, 16), idesc_sd, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(kSdFull + s));
      };
      // dV / dK / dQ of batch i: its P / dS are written and dQ of batch i - 1
      // has been read out of tensor memory (caller checked)
      constexpr uint32_t idesc_dq =
          umma_idesc_f16(128, 128, BF16, true);  // dS K-major A, K MN-major B
      auto issue_acc = [&](int i) {
        const int s = i & 1;
        tc_fence_after();
        const uint32_t st = base + C::kOffStage + s * C::kStageBytes;
        const uint32_t pds = base + C::kOffPds + s * C::kPdsBytes;
        // dQ_R (128 rows x D) = dS (rows x 64 keys) K (keys x D) first, so the
        // dQ warps can start: A = dS rows, 16 keys (32 bytes) per step; B = the
        // K tile read N-major, the two 64-column halves 8 KB apart, 16 keys
        // (2 row groups) per step
#pragma unroll
        for (int k = 0; k < 64 / 16; ++k)
          tc_mma(tmem + C::kColDq, umma_desc_sw128(pds + 128 * 128 + k * 32, 16),
                 umma_desc_sw128(base + C::kOffK + k * 2048, C::kBlkAtom), idesc_dq,
                 k > 0 ? 1u : 0u);
        tc_commit(bar(kDqFull));
#pragma unroll
        for (int k = 0; k < 128 / 16; ++k) {  // 16 rows per step
          const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
          // A: 16 rows = 2 items per step; column halves 1024 bytes apart
          tc_mma(tmem + C::kColDv,
                 umma_desc_sw128(st + 2 * C::kAtom + k * 2 * C::kItemBytes, 1024, C::kItemBytes),
                 umma_desc_sw128(pds + k * 2048, 16), idesc_acc, acc);
          tc_mma(tmem + C::kColDk, umma_desc_sw128(st + k * 2 * C::kItemBytes, 1024, C::kItemBytes),
                 umma_desc_sw128(pds + 128 * 128 + k * 2048, 16), idesc_acc, acc);
        }
        tc_commit(bar(kQdEmpty + s));
        tc_commit(bar(kPdsFree + s));
      };
      // Issue whichever is ready first: S / dP of the next batch once its rows
      // have landed (and the S / dP buffer is free: dV / dK of two batches
      // before issued), dV / dK / dQ of the oldest batch once its P / dS are
      // written and the previous dQ has been read -- so the dV / dK of batch
      // i never waits for the rows of batch i + 1. One bounded wait: about
      // 2 s (kSpinLimitCycles) without progress fails.
      int nsd = 0, nacc = 0;
      long long t_last = clock64();
      while (ok && nacc < nbat) {
        bool progressed = false;
        if (nsd < nbat && nsd <= nacc + 1 &&
            mbar_test_wait(bar(kQdFull + (nsd & 1)), (nsd >> 1) & 1)) {
          issue_sd(nsd++);
          progressed = true;
        }
        if (nacc < nsd && mbar_test_wait(bar(kPdsFull + (nacc & 1)), (nacc >> 1) & 1) &&
            (nacc == 0 || mbar_test_wait(bar(kDqFree), (nacc - 1) & 1))) {
          issue_acc(nacc++);
          progressed = true;
        }
        if (progressed) {
          t_last = clock64();
        } else if (clock64() - t_last > kSpinLimitCycles) {
          ok = false;
        }
      }
      if (ok) tc_commit(bar(kAccDone));
      failed = !ok;
    }
  } else if (warp >= 6) {
    // ---- dQ out (warps 6..9): each batch's dQ_R from tensor memory, scaled,
    // added into dQ with 16-byte fp32 reductions. A .16x256b load gives
    // thread (g8 = lane / 4, c4 = lane % 4) columns 2 c4, 2 c4 + 1 (+ 8 per
    // repetition) of rows g8 and g8 + 8 of a 16-row slice; shuffles among
    // the 4 threads of a row turn that into columns 16k + 4 c4 .. + 3, so
    // one reduction instruction covers 64 contiguous bytes of each of 8
    // rows. This thread: head g8 of items 16 j + 4 quarter + a, a = 0..3
    // (rows 32 quarter + g8 + 8 a). ----
    const int quarter = warp & 3;
    const int g8 = lane >> 2, c4 = lane & 3;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int src_lo = (lane & ~3) | (2 * (c4 & 1));  // holds columns 4 c4 % 8, + 1
    const bool upper = c4 >= 2;                        // wants the odd repetition
    for (int j = 0; j < nbat; ++j) {
      float* rowp[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int item = j * kTcBatch + quarter * 4 + a;
        rowp[a] = nullptr;
        if (item < nitems && g8 < hw0) {
          int m, sub;
          item_query(item, m, sub);
          rowp[a] = p.dQ + ((b * p.M + m) * p.H + hgroup + sub * kHeadsPerGroup + g8) * D + 4 * c4;
        }
      }
      if (!__all_sync(kFull, wait_phase(bar(kDqFull), j & 1, kWaitLimitNs))) {
        failed = true;
        break;
      }
      tc_fence_after();
      // all four pieces (16-row slice, 64-column half) first: the tensor
      // memory is released before the reductions
      uint32_t v[4][32];
#pragma unroll
      for (int piece = 0; piece < 4; ++piece)
        tc_ld_16x256b_x8(lane_addr + (static_cast<uint32_t>(16 * (piece >> 1)) << 16) +
                             C::kColDq + 64 * (piece & 1),
                         v[piece]);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(kDqFree));
#pragma unroll
      for (int piece = 0; piece < 4; ++piece) {
        const int slice = piece >> 1, half = piece & 1;
#pragma unroll
        for (int up = 0; up < 2; ++up) {  // rows g8 and g8 + 8 of the slice: items a = 2 slice + up
          float* const dst = rowp[2 * slice + up];
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // columns 16k .. 16k + 15 of the half
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int src = src_lo + (e >> 1);
              const float x =
                  __shfl_sync(kFull, __uint_as_float(v[piece][8 * k + 2 * up + (e & 1)]), src);
              const float y =
                  __shfl_sync(kFull, __uint_as_float(v[piece][8 * k + 4 + 2 * up + (e & 1)]), src);
              o[e] = (upper ? y : x) * p.scale;
            }
            if (dst) red_add_v4(dst + 64 * half + 16 * k, o[0], o[1], o[2], o[3]);
          }
        }
      }
    }
  } else {
    // ---- softmax (warps 2..5): thread <-> row (item r / 8, head r % 8) ----
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.sl2;
    auto wait_all = [&](int bb, uint32_t parity) {
      return __all_sync(kFull, wait_phase(bar(bb), parity, kWaitLimitNs));
    };
    // this row's query position and record of batch i; the next batch's are
    // requested before this batch is processed
    auto row_of = [&](int i, int& m, float& lse2, float& delta) {
      const int item = i * kTcBatch + r / 8;
      m = -1;
      lse2 = INFINITY;
      delta = 0.f;
      if (i < nbat && item < nitems) {
        int sub;
        item_query(item, m, sub);
        const float* rec = p.rec + (((b * p.M + m) * p.G + g) * nsub + sub) * 16;
        lse2 = __ldg(rec + (r & 7));
        delta = __ldg(rec + 8 + (r & 7));
      }
    };
    int m_next;
    float lse_next, delta_next;
    row_of(0, m_next, lse_next, delta_next);
    for (int i = 0; i < nbat; ++i) {
      const int s = i & 1;
      const int m = m_next;
      const float lse2 = lse_next, delta = delta_next;
      const bool valid = m >= 0;
      row_of(i + 1, m_next, lse_next, delta_next);
      const int lastkey = static_cast<int>(m < p.N - 1 ? m : p.N - 1);
      // keys n_blk + j visible: j < block size and n_blk + j <= lastkey
      const int nvis = valid ? min(p.bs, lastkey - n_blk + 1) : 0;
      if (!wait_all(kSdFull + s, (i >> 1) & 1)) {
        failed = true;
        break;
      }
      tc_fence_after();
      uint32_t sv[64], dv[64];
      tc_ld32(lane_addr + C::kColS + 64 * s, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tc_ld32(lane_addr + C::kColS + 64 * s + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tc_ld32(lane_addr + C::kColDp + 64 * s, *reinterpret_cast<uint32_t(*)[32]>(&dv[0]));
      tc_ld32(lane_addr + C::kColDp + 64 * s + 32, *reinterpret_cast<uint32_t(*)[32]>(&dv[32]));
      tc_wait_ld();
      if (i >= 2 && !wait_all(kPdsFree + s, ((i - 2) >> 1) & 1)) {
        failed = true;
        break;
      }
      uint8_t* const prow = gbase + C::kOffPds + s * C::kPdsBytes + r * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t pw[4], dw[4];
#pragma unroll
        for (int h2 = 0; h2 < 4; ++h2) {
          const int j = 8 * cc + 2 * h2;
          const bool v0 = j < nvis, v1 = j + 1 < nvis;
          const float p0 = v0 ? ex2(fmaf(__uint_as_float(sv[j]), sl2, -lse2)) : 0.f;
          const float p1 = v1 ? ex2(fmaf(__uint_as_float(sv[j + 1]), sl2, -lse2)) : 0.f;
          const float d0 = v0 ? p0 * (__uint_as_float(dv[j]) - delta) : 0.f;
          const float d1 = v1 ? p1 * (__uint_as_float(dv[j + 1]) - delta) : 0.f;
          pw[h2] = pack2_t<BF16>(p0, p1);
          dw[h2] = pack2_t<BF16>(d0, d1);
        }
        const uint32_t off = ((cc ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(prow + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        *reinterpret_cast<uint4*>(prow + 128 * 128 + off) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kPdsFull + s));
    }
    // epilogue: the chunk's dV and dK (scaled) staged in a free Q / dO stage
    // as key rows of D floats (lane = d), then added into global memory by
    // one 512-byte bulk reduction per key row
    if (!failed && nbat > 0) {
      if (!wait_all(kAccDone, 0)) {
        failed = true;
      } else {
        tc_fence_after();
        const int d = r;
        float* const stg_f = reinterpret_cast<float*>(gbase + C::kOffStage);  // dV rows, dK rows
        for (int half = 0; half < 2; ++half) {
          uint32_t vv[32], kv[32];
          tc_ld32(lane_addr + C::kColDv + 32 * half, vv);
          tc_ld32(lane_addr + C::kColDk + 32 * half, kv);
          tc_wait_ld();
          float* const rv = stg_f + (32 * half) * D + d;
          float* const rk = stg_f + (64 + 32 * half) * D + d;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            rv[j * D] = __uint_as_float(vv[j]);
            rk[j * D] = __uint_as_float(kv[j]) * p.scale;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kStaged));
        if (!wait_all(kStaged, 0)) {
          failed = true;
        } else {
          const int kidx = r & 63;  // thread r: key row kidx of dV (r < 64) or dK
          const int n = n_blk + kidx;
          if (kidx < p.bs && n < p.N) {
            bulk_reduce_add_f32((r < 64 ? p.dV : p.dK) + ((b * p.N + n) * p.G + g) * D,
                                base + C::kOffStage + static_cast<uint32_t>(r) * (D * 4), D * 4);
            bulk_commit_group();
            bulk_wait_group_read0();  // the staging row has been read
          }
        }
      }
    }
  }

  if (failed) report_timeout();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Stage 3a (D = 128): the local blocks of every block row
// ---------------------------------------------------------------------------
//
// The queries of block row c (positions c*bs .. c*bs + bs - 1) share their
// two local blocks, block c and block c - 1 (local_slot). The list kernels
// leave those entries out of the query lists and record them per row in
// lfirst; this kernel takes them, one CTA per (b, block row, g). The CTA
// owns the dQ rows of its queries: their contributions from both blocks
// are summed in tensor memory and stored once (rows that take neither block
// get zeros), so dQ needs no zeroing and the key-major kernel's fp32
// reductions shrink by two of each row's blocks. The blocks' dK and dV
// accumulate in tensor memory over the block row; at the end they are
// staged in shared memory and added by 512-byte bulk fp32 reductions.
//
// Steps: (batch of 16 items, active slot), batch by batch. Per step the
// MMA warp issues S = Q K^T and dP = dO V^T into 128 tensor-memory
// columns; the softmax warps load them (which frees the columns for the
// next step's S / dP) and write P and dS to shared memory; the MMA warp
// then adds dQ_R += dS K into the batch's dQ columns and dV^T += dO^T P,
// dK^T += Q^T dS into the slot's columns. After a batch's last slot the
// dQ warps read its dQ_R out, scale it and store it. K / V of the two
// blocks arrive once, the Q / dO tiles of each batch in two stages.
enum LocBar : int {
  kLKvFull = 0,    // 2: K / V of each active slot (loaded once)
  kLQdFull = 2,    // 2 Q / dO stages
  kLQdEmpty = 4,   // 2
  kLSdFull = 6,    // S / dP of the step are in tensor memory
  kLTFree = 7,     // the softmax warps have loaded them
  kLPdsFull = 8,   // P / dS written
  kLPdsFree = 9,   // the MMAs that read P / dS are done
  kLDqFull = 10,   // dQ_R of a batch is complete
  kLDqFree = 11,   // the dQ warps have read it
  kLAccDone = 12,  // every MMA of the CTA is done
  kLStaged = 13,   // dV / dK of the block row staged in shared memory
  kLocBars = 14
};

struct LocalCfg {
  static constexpr int kAtom = 128 * 128;    // 128 rows x 128 B
  static constexpr int kItemBytes = 2048;    // 8 rows x 2 halves x 128 B
  static constexpr int kBlkAtom = 64 * 128;  // 64 keys x 128 B
  static constexpr int kKvBytes = 4 * kBlkAtom;  // K (2 atoms: d 0-63, 64-127), then V
  static constexpr int kOffKv = 0;               // slot k at k * kKvBytes
  static constexpr int kOffStage = kOffKv + 2 * kKvBytes;
  static constexpr int kStageBytes = 4 * kAtom;  // Q tile (2 atoms), dO tile (2 atoms)
  static constexpr int kOffPds = kOffStage + 2 * kStageBytes;
  static constexpr int kPdsBytes = 2 * 128 * 128;  // P tile, dS tile (128 rows x 64 keys)
  static constexpr int kOffBar = kOffPds + kPdsBytes;
  static constexpr int kOffTmem = kOffBar + kLocBars * 8;
  static constexpr int kSmemBytes = kOffTmem + 16 + 1024;
  // slot k: dV^T at columns 128 k .. + 63, dK^T at 128 k + 64 .. + 127
  static constexpr uint32_t kColT = 256;   // S (64 columns), dP (64)
  static constexpr uint32_t kColDq = 384;  // dQ_R of the batch (128 rows x D)
};
static_assert(LocalCfg::kSmemBytes <= 232448, "one CTA per SM");

template <bool SPLIT, bool BF16>
__global__ void __launch_bounds__(kDkvTcThreads, 1)
    sel_attn_bwd_local_kernel(const BwdProblem p, const __grid_constant__ CUtensorMap tmK,
                              const __grid_constant__ CUtensorMap tmV,
                              const __grid_constant__ CUtensorMap tmQ,
                              const __grid_constant__ CUtensorMap tmD) {
  using C = LocalCfg;
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  const int nrow = static_cast<int>((p.M + p.bs - 1) / p.bs);
  const int g = static_cast<int>(blockIdx.x % p.G);
  const int64_t bc = blockIdx.x / p.G;
  const int c = static_cast<int>(bc % nrow);
  const int64_t b = bc / nrow;
  const int m0 = c * p.bs;
  const int nq = static_cast<int>(p.M - m0 < p.bs ? p.M - m0 : p.bs);
  const int nsub = SPLIT ? p.nsub : 1;
  const int nitems = nq * nsub;
  const int nbat = (nitems + kTcBatch - 1) / kTcBatch;
  const int64_t hgroup = static_cast<int64_t>(g) * p.hpg;
  const int hw0 = p.hpg < kHeadsPerGroup ? p.hpg : kHeadsPerGroup;  // head rows per item
  const int64_t mrow0 = (b * p.M + m0) * p.G + g;                  // row of query m0

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  auto bar = [&](int i) { return base + C::kOffBar + 8u * static_cast<uint32_t>(i); };

  if (threadIdx.x == 32) {  // the tensor maps' descriptors, while the CTA sets up
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmD);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  // the slots some query of the block row takes here, in slot order
  uint32_t any = 0;
  for (int q = threadIdx.x; q < nq; q += blockDim.x) {
    const int2 f = p.lfirst[mrow0 + q * p.G];
    any |= (f.x >= 0 ? 1u : 0u) | (f.y >= 0 ? 2u : 0u);
  }
  const int act = (__syncthreads_or(any & 1u) ? 1 : 0) | (__syncthreads_or(any & 2u) ? 2 : 0);
  const int nsl = __popc(act);
  auto slot_at = [&](int k) { return act == 2 ? 1 : k; };  // k-th active slot
  auto block_of = [&](int s) { return c - s; };
  const int nsteps = nbat * nsl;

  auto item_row = [&](int item, int& m, int& sub) {
    m = m0 + (SPLIT ? item / nsub : item);
    sub = SPLIT ? item % nsub : 0;
  };

  if (hw0 < kHeadsPerGroup) {
    // head rows the copies never write: zero, so the padding rows multiply zeros
    const int per = 2 * 2 * kTcBatch * 2 * (kHeadsPerGroup - hw0) * 8;
    for (int e = threadIdx.x; e < per; e += blockDim.x) {
      const int piece = e % 8, rr = e / 8;
      const int row = hw0 + rr % (kHeadsPerGroup - hw0);
      const int grp = rr / (kHeadsPerGroup - hw0);
      st_shared_zero16(base + C::kOffStage + grp * 1024 + row * 128 + piece * 16);
    }
    fence_proxy_async_smem();
  }
  if (p.bs < 64) {
    // 32-key blocks fill 32 rows of each K / V column half; the other rows stay zero
    const int per = 2 * 4 * (64 - p.bs) * 8;  // (buffer, tensor, half) x rows x 16-byte pieces
    for (int e = threadIdx.x; e < per; e += blockDim.x) {
      const int piece = e % 8, rr = e / 8;
      const int row = p.bs + rr % (64 - p.bs), atom = rr / (64 - p.bs);
      st_shared_zero16(base + C::kOffKv + atom * C::kBlkAtom + row * 128 + piece * 16);
    }
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kLKvFull + s), 1);
      mbar_init(bar(kLQdFull + s), 1);
      mbar_init(bar(kLQdEmpty + s), 1);
    }
    mbar_init(bar(kLSdFull), 1);
    mbar_init(bar(kLTFree), 4 * 32);
    mbar_init(bar(kLPdsFull), 4 * 32);
    mbar_init(bar(kLPdsFree), 1);
    mbar_init(bar(kLDqFull), 1);
    mbar_init(bar(kLDqFree), 4 * 32);
    mbar_init(bar(kLAccDone), 1);
    mbar_init(bar(kLStaged), 4 * 32);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc_alloc(base + C::kOffTmem, 512);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + C::kOffTmem);
  bool failed = false;

  if (warp == 0) {
    // ---- producer: the K / V blocks of the active slots once (lane 0),
    // per batch its Q / dO rows (lane j < 16: item j) ----
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();
      for (int k = 0; k < nsl; ++k) {
        const int n_blk = block_of(slot_at(k)) * p.bs;
        const uint32_t kvb = base + C::kOffKv + k * C::kKvBytes;
        mbar_arrive_expect_tx(bar(kLKvFull + k), 4 * p.bs * 128);
        for (int a = 0; a < 2; ++a) {
          tma_load_4d(kvb + a * C::kBlkAtom, &tmK, bar(kLKvFull + k), a * kBoxCols, g, n_blk,
                      static_cast<int>(b), keep);
          tma_load_4d(kvb + (2 + a) * C::kBlkAtom, &tmV, bar(kLKvFull + k), a * kBoxCols, g,
                      n_blk, static_cast<int>(b), keep);
        }
      }
    }
    for (int i = 0; i < nbat && nsl > 0; ++i) {
      const int s = i & 1;
      if (i >= 2 &&
          !__all_sync(kFull, wait_phase(bar(kLQdEmpty + s), ((i - 2) >> 1) & 1, kWaitLimitNs))) {
        failed = true;
        break;
      }
      const uint32_t st = base + C::kOffStage + s * C::kStageBytes;
      if (lane == 0) mbar_arrive_expect_tx(bar(kLQdFull + s), kTcBatch * 4 * hw0 * 128);
      __syncwarp();
      if (lane < kTcBatch) {
        // items past the block row repeat its last item (their rows are masked)
        int m, sub;
        item_row(min(i * kTcBatch + lane, nitems - 1), m, sub);
        const int qrow = static_cast<int>((b * p.M + m) * p.H + hgroup + sub * kHeadsPerGroup);
        const uint32_t dq = st + lane * C::kItemBytes, dd = dq + 2 * C::kAtom;
        if (hw0 == kHeadsPerGroup) {
          tma_load_3d(dq, &tmQ, bar(kLQdFull + s), 0, qrow, 0);
          tma_load_3d(dd, &tmD, bar(kLQdFull + s), 0, qrow, 0);
        } else {
          for (int a = 0; a < 2; ++a) {
            tma_load_2d(dq + a * 1024, &tmQ, bar(kLQdFull + s), a * kBoxCols, qrow);
            tma_load_2d(dd + a * 1024, &tmD, bar(kLQdFull + s), a * kBoxCols, qrow);
          }
        }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: S / dP of a step as soon as the softmax warps have
      // loaded the previous one (and its rows have landed); dQ_R, dV and dK
      // of the oldest step whose P / dS are written (the first slot of a
      // batch once the dQ warps have read the previous batch's dQ_R). One
      // bounded wait: about 2 s (kSpinLimitCycles) without progress fails. ----
      constexpr uint32_t idesc_sd = umma_idesc_f16(128, 64, BF16, false);  // K-major A, B
      constexpr uint32_t idesc_acc =
          umma_idesc_f16(128, 64, BF16, true) | (1u << 15);  // MN-major A and B
      constexpr uint32_t idesc_dq =
          umma_idesc_f16(128, 128, BF16, true);  // dS K-major A, K MN-major B
      const uint32_t pds = base + C::kOffPds;
      auto issue_sd = [&](int j) {
        const int i = j / nsl, k = j - i * nsl;
        tc_fence_after();
        const uint32_t st = base + C::kOffStage + (i & 1) * C::kStageBytes;
        const uint32_t kvb = base + C::kOffKv + k * C::kKvBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offa = (kk >> 2) * 1024 + (kk & 3) * 32;  // column half, then 16 dims
          const uint32_t offb = (kk >> 2) * C::kBlkAtom + (kk & 3) * 32;
          tc_mma(tmem + C::kColT, umma_desc_sw128(st + offa, 16, C::kItemBytes),
                 umma_desc_sw128(kvb + offb, 16), idesc_sd, kk > 0 ? 1u : 0u);
          tc_mma(tmem + C::kColT + 64, umma_desc_sw128(st + 2 * C::kAtom + offa, 16, C::kItemBytes),
                 umma_desc_sw128(kvb + 2 * C::kBlkAtom + offb, 16), idesc_sd, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(kLSdFull));
      };
      auto issue_acc = [&](int j) {
        const int i = j / nsl, k = j - i * nsl;
        tc_fence_after();
        const uint32_t st = base + C::kOffStage + (i & 1) * C::kStageBytes;
        const uint32_t kvb = base + C::kOffKv + k * C::kKvBytes;
        // dQ_R (128 rows x D) += dS K: A = dS rows, 16 keys per step; B = the K
        // tile read N-major, the two 64-column halves 8 KB apart
#pragma unroll
        for (int kk = 0; kk < 64 / 16; ++kk)
          tc_mma(tmem + C::kColDq, umma_desc_sw128(pds + 128 * 128 + kk * 32, 16),
                 umma_desc_sw128(kvb + kk * 2048, C::kBlkAtom), idesc_dq,
                 (k > 0 || kk > 0) ? 1u : 0u);
        const uint32_t cdv = tmem + 128u * static_cast<uint32_t>(k);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk) {  // 16 rows (2 items) per step
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          tc_mma(cdv,
                 umma_desc_sw128(st + 2 * C::kAtom + kk * 2 * C::kItemBytes, 1024, C::kItemBytes),
                 umma_desc_sw128(pds + kk * 2048, 16), idesc_acc, acc);
          tc_mma(cdv + 64, umma_desc_sw128(st + kk * 2 * C::kItemBytes, 1024, C::kItemBytes),
                 umma_desc_sw128(pds + 128 * 128 + kk * 2048, 16), idesc_acc, acc);
        }
        tc_commit(bar(kLPdsFree));
        if (k == nsl - 1) {
          tc_commit(bar(kLQdEmpty + (i & 1)));
          tc_commit(bar(kLDqFull));
        }
      };
      bool ok = true;
      int nsd = 0, nacc = 0;
      long long t_last = clock64();
      while (nacc < nsteps) {
        bool progressed = false;
        if (nsd < nsteps) {
          const int i = nsd / nsl, k = nsd - i * nsl;
          if ((nsd == 0 || mbar_test_wait(bar(kLTFree), (nsd - 1) & 1)) &&
              (k != 0 || mbar_test_wait(bar(kLQdFull + (i & 1)), (i >> 1) & 1)) &&
              mbar_test_wait(bar(kLKvFull + k), 0)) {
            issue_sd(nsd++);
            progressed = true;
          }
        }
        if (nacc < nsd) {
          const int i = nacc / nsl, k = nacc - i * nsl;
          if (mbar_test_wait(bar(kLPdsFull), nacc & 1) &&
              (k != 0 || i == 0 || mbar_test_wait(bar(kLDqFree), (i - 1) & 1))) {
            issue_acc(nacc++);
            progressed = true;
          }
        }
        if (progressed) {
          t_last = clock64();
        } else if (clock64() - t_last > kSpinLimitCycles) {
          ok = false;
          break;
        }
      }
      if (ok) tc_commit(bar(kLAccDone));
      failed = !ok;
    }
  } else if (warp >= 6) {
    // ---- dQ out (warps 6..9): each batch's dQ_R from tensor memory (the
    // .16x256b layout: thread (g8 = lane / 4, c4 = lane % 4) gets columns
    // 2 c4, 2 c4 + 1 (+ 8 per repetition) of rows g8 and g8 + 8 of a 16-row
    // slice), scaled, regrouped by shuffles into 16-byte pieces of 4
    // consecutive columns and stored. This thread: head g8 of items
    // 16 i + 4 quarter + a. ----
    const int quarter = warp & 3;
    const int g8 = lane >> 2, c4 = lane & 3;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int src_lo = (lane & ~3) | (2 * (c4 & 1));  // holds columns 4 c4 % 8, + 1
    const bool upper = c4 >= 2;                        // wants the odd repetition
    for (int i = 0; i < nbat; ++i) {
      uint32_t v[4][32];
      if (nsl > 0) {
        if (!__all_sync(kFull, wait_phase(bar(kLDqFull), i & 1, kWaitLimitNs))) {
          failed = true;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int piece = 0; piece < 4; ++piece)
          tc_ld_16x256b_x8(lane_addr + (static_cast<uint32_t>(16 * (piece >> 1)) << 16) +
                               C::kColDq + 64 * (piece & 1),
                           v[piece]);
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(kLDqFree));
      } else {  // no local block in the block row: its rows start at zero
#pragma unroll
        for (int piece = 0; piece < 4; ++piece)
#pragma unroll
          for (int e = 0; e < 32; ++e) v[piece][e] = 0u;
      }
      float* rowp[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int item = i * kTcBatch + quarter * 4 + a;
        rowp[a] = nullptr;
        if (item < nitems && g8 < hw0) {
          int m, sub;
          item_row(item, m, sub);
          rowp[a] = p.dQ + ((b * p.M + m) * p.H + hgroup + sub * kHeadsPerGroup + g8) * D + 4 * c4;
        }
      }
#pragma unroll
      for (int piece = 0; piece < 4; ++piece) {
        const int slice = piece >> 1, half = piece & 1;
#pragma unroll
        for (int up = 0; up < 2; ++up) {  // rows g8 and g8 + 8 of the slice: items a = 2 slice + up
          float* const dst = rowp[2 * slice + up];
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // columns 16k .. 16k + 15 of the half
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int src = src_lo + (e >> 1);
              const float x =
                  __shfl_sync(kFull, __uint_as_float(v[piece][8 * k + 2 * up + (e & 1)]), src);
              const float y =
                  __shfl_sync(kFull, __uint_as_float(v[piece][8 * k + 4 + 2 * up + (e & 1)]), src);
              o[e] = (upper ? y : x) * p.scale;
            }
            if (dst)
              *reinterpret_cast<float4*>(dst + 64 * half + 16 * k) = make_float4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    }
  } else if (warp >= 2) {
    // ---- softmax (warps 2..5): thread <-> row (item r / 8, head r % 8) ----
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.sl2;
    auto wait_all = [&](int bb, uint32_t parity) {
      return __all_sync(kFull, wait_phase(bar(bb), parity, kWaitLimitNs));
    };
    for (int i = 0; i < nbat && !failed && nsl > 0; ++i) {
      const int item = i * kTcBatch + r / 8;
      int m = -1;
      float lse2 = INFINITY, delta = 0.f;
      uint32_t rmask = 0;
      if (item < nitems) {
        int sub;
        item_row(item, m, sub);
        const int64_t row = (b * p.M + m) * p.G + g;
        const float* rec = p.rec + (row * nsub + sub) * 16;
        lse2 = __ldg(rec + (r & 7));
        delta = __ldg(rec + 8 + (r & 7));
        const int2 f = p.lfirst[row];
        rmask = (f.x >= 0 ? 1u : 0u) | (f.y >= 0 ? 2u : 0u);
      }
      const int lastkey = static_cast<int>(m < p.N - 1 ? m : p.N - 1);
      for (int k = 0; k < nsl; ++k) {
        const int j = i * nsl + k;
        const int sl = slot_at(k);
        const int n_blk = block_of(sl) * p.bs;
        // keys n_blk + jj visible: the row takes this block here, jj < block
        // size and n_blk + jj <= lastkey
        const bool valid = m >= 0 && ((rmask >> sl) & 1u);
        const int nvis = valid ? min(p.bs, lastkey - n_blk + 1) : 0;
        if (!wait_all(kLSdFull, j & 1)) {
          failed = true;
          break;
        }
        tc_fence_after();
        uint32_t sv[64], dv[64];
        tc_ld32(lane_addr + C::kColT, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tc_ld32(lane_addr + C::kColT + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tc_ld32(lane_addr + C::kColT + 64, *reinterpret_cast<uint32_t(*)[32]>(&dv[0]));
        tc_ld32(lane_addr + C::kColT + 96, *reinterpret_cast<uint32_t(*)[32]>(&dv[32]));
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(kLTFree));  // the next step's S / dP may go
        // the P / dS tiles are free once the previous step's MMAs are done
        if (j >= 1 && !wait_all(kLPdsFree, (j - 1) & 1)) {
          failed = true;
          break;
        }
        uint8_t* const prow = gbase + C::kOffPds + r * 128;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t pw[4], dw[4];
#pragma unroll
          for (int h2 = 0; h2 < 4; ++h2) {
            const int jj = 8 * cc + 2 * h2;
            const bool v0 = jj < nvis, v1 = jj + 1 < nvis;
            const float p0 = v0 ? ex2(fmaf(__uint_as_float(sv[jj]), sl2, -lse2)) : 0.f;
            const float p1 = v1 ? ex2(fmaf(__uint_as_float(sv[jj + 1]), sl2, -lse2)) : 0.f;
            const float d0 = v0 ? p0 * (__uint_as_float(dv[jj]) - delta) : 0.f;
            const float d1 = v1 ? p1 * (__uint_as_float(dv[jj + 1]) - delta) : 0.f;
            pw[h2] = pack2_t<BF16>(p0, p1);
            dw[h2] = pack2_t<BF16>(d0, d1);
          }
          const uint32_t off = ((cc ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(prow + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
          *reinterpret_cast<uint4*>(prow + 128 * 128 + off) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kLPdsFull));
      }
    }
    // epilogue: each slot's dV and dK (scaled) staged in the free Q / dO
    // stages as key rows of D floats (lane = d), then added into global
    // memory by one 512-byte bulk reduction per key row
    if (!failed && nsteps > 0) {
      if (!wait_all(kLAccDone, 0)) {
        failed = true;
      } else {
        tc_fence_after();
        const int d = r;
        const uint32_t stg = base + C::kOffStage;  // (2 k + tensor) * 64 + key rows of 512 B
        float* const stg_f = reinterpret_cast<float*>(gbase + C::kOffStage);
        for (int k = 0; k < nsl; ++k) {
          for (int half = 0; half < 2; ++half) {
            uint32_t vv[32], kv[32];
            tc_ld32(lane_addr + 128 * k + 32 * half, vv);
            tc_ld32(lane_addr + 128 * k + 64 + 32 * half, kv);
            tc_wait_ld();
            float* const rv = stg_f + ((2 * k) * 64 + 32 * half) * D + d;
            float* const rk = stg_f + ((2 * k + 1) * 64 + 32 * half) * D + d;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              rv[jj * D] = __uint_as_float(vv[jj]);
              rk[jj * D] = __uint_as_float(kv[jj]) * p.scale;
            }
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kLStaged));
        if (!wait_all(kLStaged, 0)) {
          failed = true;
        } else {
          for (int q = r; q < 2 * nsl * 64; q += 128) {
            const int tk = q >> 6, kidx = q & 63;  // tk = 2 k + tensor
            const int n = block_of(slot_at(tk >> 1)) * p.bs + kidx;
            if (kidx < p.bs && n < p.N)
              bulk_reduce_add_f32((tk & 1 ? p.dK : p.dV) + ((b * p.N + n) * p.G + g) * D,
                                  stg + static_cast<uint32_t>(q) * (D * 4), D * 4);
          }
          bulk_commit_group();
          bulk_wait_group_read0();  // the staging rows have been read
        }
      }
    }
  }

  if (failed) report_timeout();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------

struct BwdPlan {
  size_t off_do16, off_rec, off_count, off_cursor, off_offs, off_choffs, off_lists,
      off_chunk_list, off_order, off_key, off_bcount, off_bcursor, off_boffs, off_bscratch,
      off_lfirst, total;
  int64_t L, entries, max_chunks, nkeys, nbkt;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static BwdPlan bwd_plan(int64_t B, int64_t M, int64_t N, int64_t H, int64_t G, int64_t D,
                        int64_t T, int bs) {
  BwdPlan pl;
  const int64_t nsub = G > 0 ? head_subgroups(H / G) : 1;
  const int64_t nblk = (N + bs - 1) / bs;
  pl.L = B * G * nblk;
  pl.entries = B * M * G * T;
  size_t at = 0;
  pl.off_do16 = at;
  at += align256(static_cast<size_t>(B * M * H * D) * 2);
  pl.off_rec = at;
  at += align256(static_cast<size_t>(B * M * G * nsub) * 64);
  pl.off_count = at;
  at += align256(static_cast<size_t>(pl.L) * 4);
  pl.off_cursor = at;
  at += align256(static_cast<size_t>(pl.L) * 4);
  pl.off_offs = at;
  at += align256(static_cast<size_t>(pl.L + 1) * 4);
  pl.off_choffs = at;
  at += align256(static_cast<size_t>(pl.L + 1) * 4);
  pl.off_lists = at;
  at += align256(static_cast<size_t>(pl.entries) * 4);
  // chunks: sum over lists of ceil(count / chunk) <= entries / chunk + L
  pl.max_chunks = (pl.entries + kQueriesPerChunk - 1) / kQueriesPerChunk + pl.L;
  pl.off_chunk_list = at;
  at += align256(static_cast<size_t>(pl.max_chunks) * 4);
  // chunk launch order (D = 128): per chunk its order slot and bucket key;
  // per (b, g, bucket of kOrderQueries queries) a count, cursor and offset
  pl.nbkt = (M + kOrderQueries - 1) / kOrderQueries;
  if (pl.nbkt < 1) pl.nbkt = 1;
  pl.nkeys = B * G * pl.nbkt;
  pl.off_order = at;
  at += align256(static_cast<size_t>(pl.max_chunks) * 4);
  pl.off_key = at;
  at += align256(static_cast<size_t>(pl.max_chunks) * 4);
  pl.off_bcount = at;
  at += align256(static_cast<size_t>(pl.nkeys) * 4);
  pl.off_bcursor = at;
  at += align256(static_cast<size_t>(pl.nkeys) * 4);
  pl.off_boffs = at;
  at += align256(static_cast<size_t>(pl.nkeys + 1) * 4);
  pl.off_bscratch = at;
  at += align256(static_cast<size_t>(pl.nkeys + 1) * 4);
  // per (b, m, g) row: the entries the local-block kernel takes (D = 128)
  pl.off_lfirst = at;
  at += align256(static_cast<size_t>(B * M * G) * 8);
  pl.total = at;
  return pl;
}

// A second stream and its fork / join events for one call, released when
// the call returns (CUDA defers the release until the queued work is done).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, mid = nullptr, back = nullptr;
  bool ok = false;
  explicit SideStream(bool wanted) {
    if (!wanted) return;  // ok stays false: everything runs on the caller's stream
    // the highest priority: its few CTAs are scheduled as soon as SM slots
    // free up, beside the long grid already running on the caller's stream
    int lo = 0, hi = 0;
    if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess) hi = 0;
    ok = cudaStreamCreateWithPriority(&s, cudaStreamNonBlocking, hi) == cudaSuccess &&
         cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&join, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&mid, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&back, cudaEventDisableTiming) == cudaSuccess;
  }
  // `st` waits for everything queued on the side stream; if that cannot be
  // arranged, the side stream is waited for here, so no queued work outlives
  // an error return. False in that case.
  bool join_into(cudaStream_t st) {
    if (cudaEventRecord(join, s) == cudaSuccess && cudaStreamWaitEvent(st, join, 0) == cudaSuccess)
      return true;
    cudaStreamSynchronize(s);
    return false;
  }
  ~SideStream() {
    if (back) cudaEventDestroy(back);
    if (mid) cudaEventDestroy(mid);
    if (join) cudaEventDestroy(join);
    if (fork) cudaEventDestroy(fork);
    if (s) cudaStreamDestroy(s);
  }
};

template <int D, bool BF16>
static int launch_bwd(BwdProblem& p, const void* K, const void* V, uint8_t* ws,
                      const BwdPlan& pl, cudaStream_t st, bool second_stream) {
  constexpr int W = 4;
  using Cq = DqCfg<D, W>;
  int* count = reinterpret_cast<int*>(ws + pl.off_count);
  int* cursor = reinterpret_cast<int*>(ws + pl.off_cursor);
  int* offs = reinterpret_cast<int*>(ws + pl.off_offs);
  int* choffs = reinterpret_cast<int*>(ws + pl.off_choffs);
  int* lists = reinterpret_cast<int*>(ws + pl.off_lists);
  p.dO16 = reinterpret_cast<uint16_t*>(ws + pl.off_do16);
  p.rec = reinterpret_cast<float*>(ws + pl.off_rec);
  p.offs = offs;
  p.choffs = choffs;
  p.lists = lists;
  int* chunk_list = reinterpret_cast<int*>(ws + pl.off_chunk_list);
  p.chunk_list = chunk_list;
  p.chunk_order = nullptr;
  // D = 128: the local blocks of each block row go to their own kernel
  p.lfirst = D == 128 ? reinterpret_cast<int2*>(ws + pl.off_lfirst) : nullptr;
  const int64_t B = p.units / (p.M * p.G * p.nsub);
  // dK and dV start at zero (the stage-3 kernels add into them); with D =
  // 128 and a query to process, stage 2 zeroes them on its stream
  auto zero_dkv = [&](cudaStream_t s) {
    return p.N <= 0 ||
           (cudaMemsetAsync(p.dK, 0, static_cast<size_t>(B * p.N * p.G * D) * 4, s) ==
                cudaSuccess &&
            cudaMemsetAsync(p.dV, 0, static_cast<size_t>(B * p.N * p.G * D) * 4, s) ==
                cudaSuccess);
  };
  if ((D != 128 || p.N <= 0 || p.T == 0) && !zero_dkv(st)) return NSA_ERR_LAUNCH;
  const int64_t chunks = pl.max_chunks;
  int* order = reinterpret_cast<int*>(ws + pl.off_order);

  // stage 2 on stream s2: the transposed index and, with D = 128, the
  // chunks' launch order. It reads only the index tensor. 2a: per list its
  // count (and per row its local entries; with D = 128 also dK = dV = 0),
  // which is all the local-block kernel needs; 2b: the scans, the lists,
  // the chunk -> list table and the chunks' order.
  // Grids: grid-stride, `per_sm` CTAs per SM. Beside the prep and the
  // local-block kernel one CTA per SM disturbs those least and still
  // finishes in their shadow; run alone, four keep more atomics in flight.
  auto stage2a = [&](cudaStream_t s2, int per_sm) -> int {
    if (cudaMemsetAsync(count, 0, static_cast<size_t>(pl.L) * 4, s2) != cudaSuccess ||
        cudaMemsetAsync(cursor, 0, static_cast<size_t>(pl.L) * 4, s2) != cudaSuccess)
      return NSA_ERR_LAUNCH;
    if (p.lfirst != nullptr && !zero_dkv(s2)) return NSA_ERR_LAUNCH;
    // one warp per (b, g, 32 queries)
    const int64_t units = B * p.G * ((p.M + 31) / 32);
    const int64_t grid_u = (units + 7) / 8 < 152 * per_sm ? (units + 7) / 8 : 152 * per_sm;
    csr_count_kernel<<<static_cast<unsigned>(grid_u), 256, 0, s2>>>(p, count);
    return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
  };
  auto stage2b = [&](cudaStream_t s2, int per_sm) -> int {
    csr_scan_kernel<<<1, 1024, 0, s2>>>(count, offs, choffs, static_cast<int>(pl.L),
                                        kQueriesPerChunk);
    const int64_t grid_e =
        (pl.entries + 255) / 256 < 152 * per_sm ? (pl.entries + 255) / 256 : 152 * per_sm;
    csr_fill_kernel<<<static_cast<unsigned>(grid_e), 256, 0, s2>>>(p, cursor, lists);
    csr_chunk_list_kernel<<<static_cast<unsigned>((pl.L + 255) / 256), 256, 0, s2>>>(
        choffs, static_cast<int>(pl.L), chunk_list);
    if constexpr (D == 128) {
      // launch order of the chunks: by mean query position, bucketed per (b, g)
      int* key = reinterpret_cast<int*>(ws + pl.off_key);
      int* bcount = reinterpret_cast<int*>(ws + pl.off_bcount);
      int* bcursor = reinterpret_cast<int*>(ws + pl.off_bcursor);
      int* boffs = reinterpret_cast<int*>(ws + pl.off_boffs);
      int* bscratch = reinterpret_cast<int*>(ws + pl.off_bscratch);
      if (cudaMemsetAsync(bcount, 0, static_cast<size_t>(pl.nkeys) * 4, s2) != cudaSuccess ||
          cudaMemsetAsync(bcursor, 0, static_cast<size_t>(pl.nkeys) * 4, s2) != cudaSuccess)
        return NSA_ERR_LAUNCH;
      chunk_key_kernel<<<static_cast<unsigned>((chunks + 7) / 8), 256, 0, s2>>>(
          p, static_cast<int>(pl.nbkt), key, bcount);
      csr_scan_kernel<<<1, 1024, 0, s2>>>(bcount, boffs, bscratch, static_cast<int>(pl.nkeys),
                                          1);
      chunk_order_fill_kernel<<<static_cast<unsigned>((chunks + 255) / 256), 256, 0, s2>>>(
          p, key, boffs, bcursor, order);
    }
    return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
  };

  CUtensorMap tk, tv, tkb, tvb;
  const bool have_keys = p.N > 0;
  if (have_keys) {
    if (!encode_kv_map(&tk, K, B, p.N, p.G, D, kTileKeys, map_dtype(BF16)) ||
        !encode_kv_map(&tv, V, B, p.N, p.G, D, kTileKeys, map_dtype(BF16)) ||
        !encode_kv_map(&tkb, K, B, p.N, p.G, D, p.bs, map_dtype(BF16)) ||
        !encode_kv_map(&tvb, V, B, p.N, p.G, D, p.bs, map_dtype(BF16)))
      return NSA_ERR_LAUNCH;
  } else {
    memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv));
    memset(&tkb, 0, sizeof(tkb));
    memset(&tvb, 0, sizeof(tvb));
  }
  // Q / dO rows of the stage-3 kernels
  CUtensorMap tq, tdo;
  const int hw0 = p.hpg < kHeadsPerGroup ? p.hpg : kHeadsPerGroup;
  if (!encode_rows_map_t(&tq, p.Q, B * p.M * p.H, D, hw0, map_dtype(BF16)) ||
      !encode_rows_map_t(&tdo, p.dO16, B * p.M * p.H, D, hw0, map_dtype(BF16)))
    return NSA_ERR_LAUNCH;
  const bool split = p.nsub > 1;

  if constexpr (D == 128) {
    if (!have_keys || p.T == 0) {  // dQ = dK = dV = 0
      return cudaMemsetAsync(p.dQ, 0, static_cast<size_t>(B * p.M * p.H * D) * 4, st) ==
                     cudaSuccess
                 ? NSA_OK
                 : NSA_ERR_LAUNCH;
    }
    // the tensor-core (tcgen05) kernels: block K / V read as one box per
    // column half, the Q / dO rows of an item as one 3-D box (both column
    // halves)
    CUtensorMap tk64, tv64, tq3 = tq, tdo3 = tdo;
    if (!encode_kv_map(&tk64, K, B, p.N, p.G, D, p.bs, map_dtype(BF16)) ||
        !encode_kv_map(&tv64, V, B, p.N, p.G, D, p.bs, map_dtype(BF16)))
      return NSA_ERR_LAUNCH;
    if (hw0 == kHeadsPerGroup &&
        (!encode_rows_halves_map(&tq3, p.Q, B * p.M * p.H, hw0, map_dtype(BF16)) ||
         !encode_rows_halves_map(&tdo3, p.dO16, B * p.M * p.H, hw0, map_dtype(BF16))))
      return NSA_ERR_LAUNCH;
    auto kl = split ? sel_attn_bwd_local_kernel<true, BF16> : sel_attn_bwd_local_kernel<false, BF16>;
    auto kk = split ? sel_attn_bwd_dkv_tc_kernel<true, BF16> : sel_attn_bwd_dkv_tc_kernel<false, BF16>;
    if (cudaFuncSetAttribute(kl, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             LocalCfg::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DkvTcCfg::kSmemBytes) != cudaSuccess)
      return NSA_ERR_LAUNCH;
    // Stage 2 runs on a second stream: 2a beside stage 1 (prep: 16-bit dO,
    // LSE, delta), which streams dO and O through HBM; 2b after stage 1,
    // beside the local-block kernel (one CTA of its fill fits beside each of
    // that kernel's CTAs), so the prep has the SMs to itself but for 2a.
    // Neither stage touches what the other writes. The local-block kernel
    // waits for stage 1 and stage 2a; the key-major kernel for everything.
    SideStream side(second_stream);
    const bool on_side = side.ok && cudaEventRecord(side.fork, st) == cudaSuccess &&
                         cudaStreamWaitEvent(side.s, side.fork, 0) == cudaSuccess;
    cudaStream_t s2 = on_side ? side.s : st;  // no second stream: in order on st
    const int per_sm = on_side ? 1 : 4;
    int rc2 = stage2a(s2, per_sm);
    const bool mid_ok = on_side && rc2 == NSA_OK && cudaEventRecord(side.mid, s2) == cudaSuccess;
    sel_attn_bwd_prep_kernel<D, BF16><<<static_cast<unsigned>((p.units + 7) / 8), 256, 0, st>>>(p);
    bool rc1 = cudaGetLastError() == cudaSuccess;
    // 2b after the prep (if that order cannot be arranged, 2b runs beside it)
    if (on_side && cudaEventRecord(side.back, st) == cudaSuccess)
      cudaStreamWaitEvent(s2, side.back, 0);
    if (rc2 == NSA_OK) rc2 = stage2b(s2, per_sm);
    if (on_side) {
      // the local-block kernel needs stage 2a only; if that wait cannot be
      // arranged, it waits for all of stage 2
      if (!(mid_ok && cudaStreamWaitEvent(st, side.mid, 0) == cudaSuccess) &&
          !side.join_into(st))
        return NSA_ERR_LAUNCH;
    }
    if (rc2 != NSA_OK || !rc1) {
      if (on_side) side.join_into(st);  // no queued work outlives the call
      return rc2 != NSA_OK ? rc2 : NSA_ERR_LAUNCH;
    }
    // the local blocks of every block row first: it stores each dQ row once,
    // then the key-major kernel adds the rest of the row's blocks
    const int64_t lgrid = B * p.G * ((p.M + p.bs - 1) / p.bs);  // < 2^31: B * M * G * T is
    if (lgrid > 0)
      kl<<<static_cast<unsigned>(lgrid), kDkvTcThreads, LocalCfg::kSmemBytes, st>>>(p, tk64, tv64,
                                                                                   tq3, tdo3);
    rc1 = cudaGetLastError() == cudaSuccess;
    if (on_side && !side.join_into(st)) return NSA_ERR_LAUNCH;
    if (!rc1) return NSA_ERR_LAUNCH;
    p.chunk_order = order;  // written by stage 2b
    kk<<<static_cast<unsigned>(chunks), kDkvTcThreads, DkvTcCfg::kSmemBytes, st>>>(
        p, tk64, tv64, tq3, tdo3);
    return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
  } else {
    // stage 1: dQ and delta
    auto kq = sel_attn_bwd_dq_kernel<D, W, BF16>;
    if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, Cq::kSmemBytes) !=
        cudaSuccess)
      return NSA_ERR_LAUNCH;
    kq<<<static_cast<unsigned>((p.units + W - 1) / W), W * 32, Cq::kSmemBytes, st>>>(p, tk, tv);
    if (cudaGetLastError() != cudaSuccess) return NSA_ERR_LAUNCH;
    if (!have_keys || p.T == 0) return NSA_OK;  // dK = dV = 0
    // stage 2 after stage 1, on the caller's stream
    int rc2 = stage2a(st, 4);
    if (rc2 == NSA_OK) rc2 = stage2b(st, 4);
    if (rc2 != NSA_OK) return rc2;
    // stage 3: dK, dV; grid bound: sum over lists of ceil(count / chunk)
    auto run = [&](auto kt, auto sp) -> int {
      constexpr int KT = decltype(kt)::value;
      using Ck = DkvCfg<D, KT>;
      auto kd = sel_attn_bwd_dkv_kernel<D, KT, decltype(sp)::value, BF16>;
      if (cudaFuncSetAttribute(kd, cudaFuncAttributeMaxDynamicSharedMemorySize, Ck::kSmemBytes) !=
          cudaSuccess)
        return NSA_ERR_LAUNCH;
      kd<<<static_cast<unsigned>(chunks), Ck::kWarps * 32, Ck::kSmemBytes, st>>>(p, tkb, tvb, tq,
                                                                               tdo);
      return NSA_OK;
    };
    using I2 = std::integral_constant<int, 2>;
    using I4 = std::integral_constant<int, 4>;
    using Yes = std::true_type;
    using No = std::false_type;
    int rc;
    if (p.bs == 64)
      rc = split ? run(I4{}, Yes{}) : run(I4{}, No{});
    else
      rc = split ? run(I2{}, Yes{}) : run(I2{}, No{});
    if (rc != NSA_OK) return rc;
    return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
  }
}

int bwd_read_and_clear_status(unsigned int* value) { return read_and_clear_status(value); }

// ---- fixed scratch for callers that cannot allocate --------------------------
//
// Some callers of this library may not allocate device memory at all: a
// plugin inside a host application that owns every device allocation
// through its own pool and hands plugins no allocator, or a service that
// reserves all of its memory at start-up and forbids allocation while it
// serves. nsa_sel_attn_bwd_noalloc gives them the backward without a
// caller-provided workspace: its scratch (delta, list counts and offsets,
// the query lists) lives in this file-scope device array, which every GPU
// that loads the library holds until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch in the current device's context. In
// host code the array's name is only a host-side handle, never a device
// address. The address is looked up on every call (a host-side query that
// allocates nothing and does not synchronise), so a context created anew
// after cudaDeviceReset is never served a stale address.
static void* noalloc_scratch_address() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
  return ptr;
}

// Size checks of both backward entry points; fills the scratch plan.
static int bwd_check_sizes(int64_t B, int64_t M, int64_t N, int64_t H, int64_t G, int64_t D,
                           int64_t T, int block_size, BwdPlan* pl) {
  const int chk = check_sizes(B, M, N, H, G, D, T, block_size);
  if (chk != NSA_OK) return chk;
  if (B * M * G * T > (int64_t(1) << 31) - 1) return NSA_ERR_SHAPE;
  *pl = bwd_plan(B, M, N, H, G, D, T, block_size);
  if (pl->L > (int64_t(1) << 31) - 2) return NSA_ERR_SHAPE;
  return NSA_OK;
}

// Pointer checks of both backward entry points for a problem with queries
// (B, M > 0): NSA_ERR_NULL, NSA_ERR_ALIGN or NSA_OK. `workspace` is checked
// for alignment when given.
static int bwd_check_pointers(const void* Q, const void* K, const void* V, const int32_t* idx,
                              const float* O, const float* LSE, const float* dO, const float* dQ,
                              const float* dK, const float* dV, int64_t N, int64_t T,
                              const void* workspace) {
  if (!Q || !O || !LSE || !dO || !dQ) return NSA_ERR_NULL;
  if (N > 0 && (!K || !V || !dK || !dV)) return NSA_ERR_NULL;
  if (T > 0 && !idx) return NSA_ERR_NULL;
  auto mis = [](const void* ptr, uintptr_t a) {
    return ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
  };
  if (mis(Q, 16) || mis(K, 16) || mis(V, 16) || mis(O, 16) || mis(dO, 16) || mis(dQ, 16) ||
      mis(dK, 16) || mis(dV, 16) || mis(LSE, 4) || mis(idx, 4) || mis(workspace, 256))
    return NSA_ERR_ALIGN;
  return NSA_OK;
}

// Validated arguments -> the kernels' problem description, then the launch
// of the stages with `ws` as scratch.
static int run_bwd(const void* Q, const void* K, const void* V, const int32_t* idx,
                   const float* O, const float* LSE, const float* dO, float* dQ, float* dK,
                   float* dV, int64_t B, int64_t M, int64_t N, int64_t H, int64_t G, int64_t D,
                   int64_t T, int block_size, float scale, bool bf16, const BwdPlan& pl,
                   uint8_t* ws, cudaStream_t st, bool second_stream) {
  BwdProblem p;
  p.Q = static_cast<const uint16_t*>(Q);
  p.idx = idx;
  p.O = O;
  p.LSE = LSE;
  p.dO = dO;
  p.dQ = dQ;
  p.dK = dK;
  p.dV = dV;
  p.M = M;
  p.N = N;
  p.H = H;
  p.G = G;
  p.T = T;
  p.B = B;
  p.hpg = static_cast<int>(H / G);
  p.nsub = head_subgroups(p.hpg);
  p.units = B * G * p.nsub * M;
  p.bs = block_size;
  p.nblk = static_cast<int>((N + block_size - 1) / block_size);
  p.L = static_cast<int>(pl.L);
  p.scale = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  p.sl2 = p.scale * 1.4426950408889634f;
  if (D == 64)
    return bf16 ? launch_bwd<64, true>(p, K, V, ws, pl, st, second_stream)
                : launch_bwd<64, false>(p, K, V, ws, pl, st, second_stream);
  return bf16 ? launch_bwd<128, true>(p, K, V, ws, pl, st, second_stream)
              : launch_bwd<128, false>(p, K, V, ws, pl, st, second_stream);
}

}  // namespace nsa

extern "C" {

int64_t nsa_sel_attn_bwd_workspace_bytes(int64_t B, int64_t M, int64_t N, int64_t H, int64_t G,
                                         int64_t D, int64_t T, int block_size) {
  nsa::BwdPlan pl;
  const int chk = nsa::bwd_check_sizes(B, M, N, H, G, D, T, block_size, &pl);
  if (chk != NSA_OK) return chk;
  return static_cast<int64_t>(pl.total);
}

int nsa_sel_attn_bwd_ex(const void* Q, const void* K, const void* V,
                        const int32_t* block_indices, const float* O, const float* LSE,
                        const float* dO, float* dQ, float* dK, float* dV, int64_t B, int64_t M,
                        int64_t N, int64_t H, int64_t G, int64_t D, int64_t T, int block_size,
                        float scale, int qkv_dtype, void* workspace, int64_t workspace_bytes,
                        void* stream) {
  using namespace nsa;
  if (qkv_dtype != NSA_F16 && qkv_dtype != NSA_BF16) return NSA_ERR_DTYPE;
  BwdPlan pl;
  const int chk = bwd_check_sizes(B, M, N, H, G, D, T, block_size, &pl);
  if (chk != NSA_OK) return chk;
  if (B == 0 || (M == 0 && N == 0)) return NSA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M == 0) {  // no query: every key gradient is zero
    if (!dK || !dV) return NSA_ERR_NULL;
    if (cudaMemsetAsync(dK, 0, static_cast<size_t>(B * N * G * D) * 4, st) != cudaSuccess ||
        cudaMemsetAsync(dV, 0, static_cast<size_t>(B * N * G * D) * 4, st) != cudaSuccess)
      return NSA_ERR_LAUNCH;
    return NSA_OK;
  }
  int rc = bwd_check_pointers(Q, K, V, block_indices, O, LSE, dO, dQ, dK, dV, N, T, nullptr);
  if (rc != NSA_OK) return rc;
  if (!workspace || workspace_bytes < static_cast<int64_t>(pl.total)) return NSA_ERR_WORKSPACE;
  rc = bwd_check_pointers(Q, K, V, block_indices, O, LSE, dO, dQ, dK, dV, N, T, workspace);
  if (rc != NSA_OK) return rc;
  return run_bwd(Q, K, V, block_indices, O, LSE, dO, dQ, dK, dV, B, M, N, H, G, D, T,
                 block_size, scale, qkv_dtype == NSA_BF16, pl, static_cast<uint8_t*>(workspace),
                 st, true);
}

int nsa_sel_attn_bwd(const void* Q, const void* K, const void* V, const int32_t* block_indices,
                     const float* O, const float* LSE, const float* dO, float* dQ, float* dK,
                     float* dV, int64_t B, int64_t M, int64_t N, int64_t H, int64_t G, int64_t D,
                     int64_t T, int block_size, float scale, void* workspace,
                     int64_t workspace_bytes, void* stream) {
  return nsa_sel_attn_bwd_ex(Q, K, V, block_indices, O, LSE, dO, dQ, dK, dV, B, M, N, H, G, D, T,
                             block_size, scale, NSA_F16, workspace, workspace_bytes, stream);
}

int nsa_sel_attn_bwd_noalloc(const void* Q, const void* K, const void* V,
                             const int32_t* block_indices, const float* O, const float* LSE,
                             const float* dO, float* dQ, float* dK, float* dV, int64_t B,
                             int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                             int block_size, float scale, void* stream) {
  using namespace nsa;
  BwdPlan pl;
  const int chk = bwd_check_sizes(B, M, N, H, G, D, T, block_size, &pl);
  if (chk != NSA_OK) return chk;
  if (B == 0 || M == 0) {
    // no query, so no scratch: the workspace entry point zeroes dK and dV
    return nsa_sel_attn_bwd(Q, K, V, block_indices, O, LSE, dO, dQ, dK, dV, B, M, N, H, G, D, T,
                            block_size, scale, nullptr, 0, stream);
  }
  if (pl.total > kNoAllocScratchBytes) return NSA_ERR_SCRATCH;
  const int rc =
      bwd_check_pointers(Q, K, V, block_indices, O, LSE, dO, dQ, dK, dV, N, T, nullptr);
  if (rc != NSA_OK) return rc;
  void* scratch = noalloc_scratch_address();
  if (scratch == nullptr) return NSA_ERR_LAUNCH;
  return run_bwd(Q, K, V, block_indices, O, LSE, dO, dQ, dK, dV, B, M, N, H, G, D, T,
                 block_size, scale, false, pl, static_cast<uint8_t*>(scratch),
                 static_cast<cudaStream_t>(stream), false);
}

}  // extern "C"
