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
// One CTA per (b, head, tile of 128 queries); 6 warps with fixed roles:
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

#include "common.cuh"
#include "nsa_sel_attn.h"
#include "ptx.cuh"
#include "sel_attn_fwd.cuh"
#include "tc.cuh"

namespace nsa {
namespace {

constexpr int kSwaQ = 128;     // queries per CTA (MMA M)
constexpr int kSwaKeys = 128;  // keys per tile
constexpr int kSwaThreads = 192;
constexpr uint32_t kSwaTmemCols = 512;
constexpr uint32_t kColS = 0;  // S buffers at columns 0 and 128
constexpr uint32_t kColO = 256;  // D columns
constexpr uint32_t kColP = 384;  // two P buffers of 64 columns (128 keys, 16-bit pairs)
constexpr int kSwaStages = 3;    // K/V ring
constexpr float kSwaSlack = 8.0f;

// One barrier per ring slot / buffer, so that no barrier can complete twice
// before its waiter has seen the first completion.
enum SwaBar : int {
  kQFull = 0,
  kKFull = 1,    // 3 stages
  kKEmpty = 4,   // 3
  kVFull = 7,    // 3
  kVEmpty = 10,  // 3
  kSFull = 13,   // 2 S buffers (tensor memory)
  kPFull = 15,   // 2 P buffers (tensor memory)
  kPvDone = 17,  // 2: PV of the tile that used P buffer b has completed
  kNumBars = 19
};

template <int D>
struct SwaCfg {
  static constexpr int kAtoms = D / 64;                 // 64-element swizzle columns
  static constexpr int kAtomBytes = kSwaQ * 128;         // 128 rows x 128 B
  static constexpr int kQBytes = kSwaQ * D * 2;
  static constexpr int kKVBytes = kSwaKeys * D * 2;      // one K (or V) stage
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kSwaStages * kKVBytes;
  static constexpr int kOffBar = kOffV + kSwaStages * kKVBytes;
  static constexpr int kOffTmem = kOffBar + kNumBars * 8;
  // at least 116 KB so that one CTA holds an SM (all 512 tensor-memory columns)
  static constexpr int kUsed = kOffTmem + 16 + 1024;
  static constexpr int kSmemBytes = kUsed > 118784 ? kUsed : 118784;
};

struct SwaProblem {
  void* O;
  float* LSE;
  int M, N, H, Hkv, hpg, qtiles;
  int left, right;  // clamped to [0, M + N]: M + N is unbounded in effect
  float sl2;        // scale * log2(e)
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return pack2_t<BF16>(lo, hi);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kSwaThreads, 1)
    swa_fwd_kernel(const SwaProblem p, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV) {
  using C = SwaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);  // generic pointer to `base`
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // (b, KV head, query tile, head within the group), the head fastest: the
  // CTAs in flight share their K/V tiles through L2
  uint32_t x = blockIdx.x;
  const int hh = static_cast<int>(x % p.hpg);
  x /= p.hpg;
  const int qt = static_cast<int>(x % p.qtiles);
  x /= p.qtiles;
  const int g = static_cast<int>(x % p.Hkv);
  const int b = static_cast<int>(x / p.Hkv);
  const int h = g * p.hpg + hh;
  const int q0 = qt * kSwaQ;
  const int q_last = min(q0 + kSwaQ, p.M) - 1;
  // keys the tile's windows touch, in whole tiles of 128
  const int jlo = max(0, q0 - p.left);
  const int jhi = min(p.N - 1, q_last + p.right);
  const int t0 = jlo / kSwaKeys;
  const int nt = jhi >= jlo ? jhi / kSwaKeys - t0 + 1 : 0;
  // keys every row of the tile sees (tiles inside need no mask)
  const int in_lo = max(0, q_last - p.left);
  const int in_hi = min(p.N - 1, q0 + p.right);

  auto bar = [&](int i) { return base + C::kOffBar + 8u * static_cast<uint32_t>(i); };
  if (threadIdx.x == 0) {
    mbar_init(bar(kQFull), 1);
    for (int s = 0; s < kSwaStages; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 1);
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(bar(kSFull + s), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kPFull + s), 4 * 32);
      mbar_init(bar(kPvDone + s), 1);
    }
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

  if (warp == 0) {
    if (lane == 0 && nt > 0) {
      // ---- TMA producer ----
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint64_t keep = l2_policy_evict_last();
      mbar_arrive_expect_tx(bar(kQFull), C::kQBytes);
      for (int a = 0; a < C::kAtoms; ++a)
        tma_load_4d(base + C::kOffQ + a * C::kAtomBytes, &tmQ, bar(kQFull), a * 64, h, q0, b,
                    l2_policy_evict_first());
      for (int i = 0; i < nt && !failed; ++i) {
        const int s = i % kSwaStages;
        const int j0 = (t0 + i) * kSwaKeys;
        const uint32_t prev = ((i - kSwaStages) / kSwaStages) & 1;  // phase of tile i - 3
        if (i >= kSwaStages && !wait_phase(bar(kKEmpty + s), prev, kWaitLimitNs)) {
          failed = true;
          break;
        }
        mbar_arrive_expect_tx(bar(kKFull + s), C::kKVBytes);
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_4d(base + C::kOffK + s * C::kKVBytes + a * C::kAtomBytes, &tmK,
                      bar(kKFull + s), a * 64, g, j0, b, keep);
        if (i >= kSwaStages && !wait_phase(bar(kVEmpty + s), prev, kWaitLimitNs)) {
          failed = true;
          break;
        }
        mbar_arrive_expect_tx(bar(kVFull + s), C::kKVBytes);
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_4d(base + C::kOffV + s * C::kKVBytes + a * C::kAtomBytes, &tmV,
                      bar(kVFull + s), a * 64, g, j0, b, keep);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nt > 0) {
      // ---- MMA issuer ----
      constexpr uint32_t idesc_s = umma_idesc_f16(kSwaQ, kSwaKeys, BF16, false);
      constexpr uint32_t idesc_o = umma_idesc_f16(kSwaQ, D, BF16, true);
      bool ok = wait_phase(bar(kQFull), 0, kWaitLimitNs);
      auto issue_s = [&](int i) -> bool {
        const int s = i % kSwaStages;
        if (!wait_phase(bar(kKFull + s), (i / kSwaStages) & 1, kWaitLimitNs)) return false;
        tc_fence_after();
        const uint32_t d = tmem + kColS + static_cast<uint32_t>(i & 1) * kSwaKeys;
        const uint32_t kb = base + C::kOffK + s * C::kKVBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * C::kAtomBytes + (k & 3) * 32;
          tc_mma(d, umma_desc_sw128(base + C::kOffQ + off, 16),
                 umma_desc_sw128(kb + off, 16), idesc_s, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(kKEmpty + s));
        tc_commit(bar(kSFull + (i & 1)));
        return true;
      };
      auto issue_pv = [&](int i) -> bool {
        const int s = i % kSwaStages;  // V stage
        const int pbuf = i & 1;        // P buffer
        if (!wait_phase(bar(kPFull + pbuf), (i >> 1) & 1, kWaitLimitNs)) return false;
        if (!wait_phase(bar(kVFull + s), (i / kSwaStages) & 1, kWaitLimitNs)) return false;
        tc_fence_after();
        const uint32_t vb = base + C::kOffV + s * C::kKVBytes;
        const uint32_t pcol = tmem + kColP + static_cast<uint32_t>(pbuf) * (kSwaKeys / 2);
#pragma unroll
        for (int kk = 0; kk < kSwaKeys / 16; ++kk) {
          tc_mma_ts(tmem + kColO, pcol + 8 * kk, umma_desc_sw128(vb + kk * 2048, C::kAtomBytes),
                    idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(kVEmpty + s));
        tc_commit(bar(kPvDone + pbuf));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int i = 1; i <= nt && ok; ++i) {
        if (i < nt) ok = issue_s(i);
        if (ok) ok = issue_pv(i - 1);
      }
      failed = !ok;
    }
  } else {
    // ---- softmax (warps 2..5): thread <-> query row ----
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int iq = q0 + row;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int lo_i = max(0, iq - p.left);
    const int hi_i = min(p.N - 1, iq + p.right);
    float ref = -INFINITY, neg = 0.f, l = 0.f;  // ref, neg in the log2 domain
    const float sl2 = p.sl2;
    // waits are decided warp-wide (tcgen05.ld/st are warp-collective)
    auto wait_all = [&](int b, int parity) {
      return __all_sync(kFull, wait_phase(bar(b), parity, kWaitLimitNs));
    };
    for (int i = 0; i < nt; ++i) {
      const int sb = i & 1;  // S buffer and P buffer of this tile
      if (!wait_all(kSFull + sb, (i >> 1) & 1)) {
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
      const int j0 = (t0 + i) * kSwaKeys;
      if (j0 < in_lo || j0 + kSwaKeys - 1 > in_hi) {  // edge tile (CTA-uniform)
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
          if (!wait_all(kPvDone + ((i - 1) & 1), ((i - 1) >> 1) & 1)) {
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
      // P buffer sb was last read by the PV of tile i - 2
      if (i >= 2) {
        if (!wait_all(kPvDone + sb, ((i - 2) >> 1) & 1)) {
          failed = true;
          break;
        }
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
    // epilogue
    if (!failed && nt > 0) {
      if (!wait_all(kPvDone + ((nt - 1) & 1), ((nt - 1) >> 1) & 1)) failed = true;
      tc_fence_after();
    }
    if (!failed) {  // warp-uniform: the tensor-memory loads are collective
      const bool store = iq < p.M;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* orow = static_cast<uint16_t*>(p.O) +
                       ((static_cast<int64_t>(b) * p.M + (store ? iq : 0)) * p.H + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (nt > 0) {
          tc_ld32(lane_addr + kColO + 32 * c, o);
          tc_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0u;
        }
        if (!store) continue;
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack2<BF16>(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
          w.y = pack2<BF16>(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
          w.z = pack2<BF16>(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
          w.w = pack2<BF16>(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
          dst[q] = w;
        }
      }
      if (store && p.LSE != nullptr) {
        constexpr float kLn2 = 0.69314718055994530942f;
        p.LSE[(static_cast<int64_t>(b) * p.H + h) * p.M + iq] =
            l > 0.f ? (ref + __log2f(l)) * kLn2 : -INFINITY;
      }
    }
  }

  // teardown: every role is here; the tensor memory is freed
  if (failed) report_timeout();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tc_dealloc(tmem, kSwaTmemCols);
  }
}

template <int D, bool BF16>
int launch_swa(const SwaProblem& p, const void* Q, const void* K, const void* V, int64_t B,
               cudaStream_t st) {
  using C = SwaCfg<D>;
  constexpr CUtensorMapDataType dt =
      BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tq, tk, tv;
  if (!encode_kv_map(&tq, Q, B, p.M, p.H, D, kSwaQ, dt)) return NSA_ERR_LAUNCH;
  if (p.N > 0) {
    if (!encode_kv_map(&tk, K, B, p.N, p.Hkv, D, kSwaKeys, dt) ||
        !encode_kv_map(&tv, V, B, p.N, p.Hkv, D, kSwaKeys, dt))
      return NSA_ERR_LAUNCH;
  } else {
    memset(&tk, 0, sizeof(tk));  // no key: no tile is ever loaded
    memset(&tv, 0, sizeof(tv));
  }
  auto kern = swa_fwd_kernel<D, BF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return NSA_ERR_LAUNCH;
  const int64_t blocks = B * p.H * p.qtiles;
  kern<<<static_cast<unsigned>(blocks), kSwaThreads, C::kSmemBytes, st>>>(p, tq, tk, tv);
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
  p.O = O;
  p.LSE = LSE;
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf = dtype == NSA_BF16;
  if (D == 64)
    return bf ? launch_swa<64, true>(p, Q, K, V, B, st) : launch_swa<64, false>(p, Q, K, V, B, st);
  return bf ? launch_swa<128, true>(p, Q, K, V, B, st) : launch_swa<128, false>(p, Q, K, V, B, st);
}
