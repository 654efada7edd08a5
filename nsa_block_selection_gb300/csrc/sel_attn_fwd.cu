// NSA selection-attention forward for sm_103a, and the library's C ABI.
//
// Operation ("[wave] NSA: selection attention forward kernel", sections
// "Operation", "Algorithm", "Requirements"): for every (b, m, g) the heads of
// KV group g attend, with one online softmax, over the keys of the blocks
// block_indices[b, m, g, :] selects, causally masked; O [B,M,H,D] and the
// natural-log LSE [B,H,M] are written.
//
// Kernel shape (one warp per (b, m, g) work unit, warps independent):
//  * the warp walks its index row and streams the selected keys in tiles of
//    16 keys through two private shared-memory slots (K tile, V tile); lane 0
//    fills a slot with TMA bulk-tensor copies (128-byte swizzled rows) that
//    complete on the slot's mbarrier, and refills it with the next tile's K
//    (or V) as soon as QK^T (or PV) has read it;
//  * S^T = K Q^T on the tensor cores (mma.sync m16n8k16, fp16 in, fp32 acc):
//    16 keys x 8 heads, so the group's 8 heads are exactly the MMA's N; the
//    k-steps run as two independent MMA chains;
//  * scores are scaled into the log2 domain; probabilities are
//    exp2(x - ref) with a per-head reference that only moves when a score
//    exceeds it by more than 8 (so the max reduction and the O rescale run
//    on few tiles);
//  * P is rounded to fp16, transposed in registers (movmatrix) into the B
//    operand of O^T += V^T P^T, whose A operand comes from ldmatrix.trans;
//  * the epilogue normalises O, writes it as fp32 and writes LSE.
// Keys past the query's last visible key (causal edge, or n >= N) are masked
// by select; V rows there are zeroed in shared memory before the PV product,
// so whatever those rows hold never reaches the output. Rows n >= N are
// outside the tensor map and arrive as zeros.
//
// Every mbarrier wait is bounded (1 s of %globaltimer). On timeout the warp
// sets bit 0 of the device status word, waits (bounded) for its own copies in
// flight, and returns without writing its outputs; nsa_sync_status() reports
// it as NSA_ERR_TIMEOUT.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "nsa_sel_attn.h"
#include "ptx.cuh"
#include "sel_attn_fwd.cuh"
#include "status.cuh"

#ifndef NSA_WARPS
#define NSA_WARPS 4
#endif
#ifndef NSA_MIN_BLOCKS
#define NSA_MIN_BLOCKS 4
#endif

namespace nsa {

struct Problem {
  const uint16_t* Q;  // fp16 or bf16
  const int32_t* idx;
  void* O;            // fp32, or the inputs' 16-bit type
  float* LSE;
  int64_t M, N, H, G, T;
  int64_t q_sb, q_sm, q_sh;  // element strides of Q over b, m, h (d contiguous)
  int64_t o_sb, o_sm, o_sh;  // element strides of O over b, m, h (d contiguous)
  int64_t m_off;  // query position of row 0 (a chunk of a longer sequence)
  int64_t units;  // B * G * nsub * M
  const int32_t* shared;  // two-pass path: per-tile records of the blocks already attended to
  int64_t ntiles;         // query tiles per (b, g) of those records
  int hpg;        // query heads per KV group
  int nsub;       // sub-groups of 8 heads per KV group
  int bs;
  int nblk;       // ceil(N / bs)
  float sl2;      // scale * log2(e)
};

template <int D, int WARPS, bool SHARED = false>
struct Cfg {
  static constexpr int kBoxes = D / kBoxCols;            // TMA boxes per tile
  static constexpr int kTileBytes = kBoxes * kBoxBytes;  // one K (or V) tile = one slot
  static constexpr int kWarpBytes = 2 * kTileBytes;      // slot 0: K, slot 1: V
  static constexpr int kBarOffset = WARPS * kWarpBytes;
  // two-pass gather kernel: per warp, the tile-shared pass's partial O of its
  // 8 heads (fp32, contiguous) and the barrier its bulk copy completes on
  static constexpr int kPartBytes = SHARED ? kHeadsPerGroup * D * 4 : 0;
  static constexpr int kPartBarOffset = kBarOffset + WARPS * 2 * 8;
  static constexpr int kPartOffset = kPartBarOffset + (SHARED ? WARPS * 8 : 0);
  static constexpr int kSmemBytes = kPartOffset + WARPS * kPartBytes + 1024;  // + align slack
  static constexpr int kSteps = D / 16;
};

// Raise the running max only when a scaled score exceeds it by more than
// 2^8: probabilities stay <= 256 (exact in the sums, fine for fp16) and the
// shuffle reduction and O rescale run on few tiles. LSE and O use the same
// reference, so the result does not depend on it.
constexpr float kMaxSlack = 8.0f;

// BF16: Q/K/V are bf16 (else fp16); P is rounded to the same type for the PV
// product. O16: O is written in that 16-bit type (else fp32). SHARED (fp32 O,
// 8 heads per group): the tile-shared pass has attended to the blocks its
// record lists and left the normalised partial O and its LSE in the outputs;
// the warp skips those blocks and starts from that state (O = the partial O,
// row sum 1, reference = its LSE in log2 units).
template <int D, int WARPS, bool BF16, bool O16, bool SHARED = false>
__global__ void __launch_bounds__(WARPS * 32, NSA_MIN_BLOCKS)
    sel_attn_fwd_kernel(const Problem p, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV) {
  using C = Cfg<D, WARPS, SHARED>;
  extern __shared__ uint8_t smem_raw[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * WARPS + warp;
  if (unit >= p.units) return;
  // unit -> (b, g, sub-group, m), m fastest: the warps in flight share one
  // group's K/V
  const int64_t m = unit % p.M;
  const int64_t r = unit / p.M;
  const int sub = static_cast<int>(r % p.nsub);
  const int64_t bg = r / p.nsub;
  const int g = static_cast<int>(bg % p.G);
  const int b = static_cast<int>(bg / p.G);
  // heads of this warp: hbase + j for j < hw (MMA columns j >= hw are padding)
  const int hw = p.hpg - sub * kHeadsPerGroup < kHeadsPerGroup ? p.hpg - sub * kHeadsPerGroup
                                                                : kHeadsPerGroup;
  const int gid = lane >> 2;  // MMA group id (row within an 8-row slab)
  const int tig = lane & 3;   // thread in group
  // two-pass path: the record of this query's tile ({count, ids}), loaded
  // first so that its latency overlaps the setup below
  int rec_v = 0;
  if constexpr (SHARED) {
    const int32_t* rec = p.shared + (bg * p.ntiles + m / kSharedTileQ) * kSharedRec;
    if (lane < kSharedRec) rec_v = __ldg(rec + lane);
  }

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t slots = base + warp * C::kWarpBytes;
  const uint32_t bars = base + C::kBarOffset + warp * 2 * 8;
  const uint32_t part_bar = base + C::kPartBarOffset + warp * 8;  // two-pass only
  const uint32_t part = base + C::kPartOffset + warp * C::kPartBytes;

  if (lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    mbar_init(bars, 1);
    mbar_init(bars + 8, 1);
    if constexpr (SHARED) mbar_init(part_bar, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncwarp();

  const int64_t hbase = static_cast<int64_t>(g) * p.hpg + sub * kHeadsPerGroup;
  // Q^T as the B operand of S^T = K Q^T: head gid, dims 16k + 2tig (+1, +8, +9);
  // zero for padding columns
  uint32_t qf[C::kSteps][2];
  {
    const uint16_t* q = p.Q + b * p.q_sb + m * p.q_sm + (hbase + gid) * p.q_sh + 2 * tig;
#pragma unroll
    for (int k = 0; k < C::kSteps; ++k) {
      qf[k][0] = gid < hw ? __ldg(reinterpret_cast<const unsigned int*>(q + 16 * k)) : 0u;
      qf[k][1] = gid < hw ? __ldg(reinterpret_cast<const unsigned int*>(q + 16 * k + 8)) : 0u;
    }
  }

  const int64_t mpos = m + p.m_off;  // the query's position in the key sequence
  const int lastkey = static_cast<int>(mpos < p.N - 1 ? mpos : p.N - 1);
  const int32_t* irow = p.idx + ((b * p.M + m) * p.G + g) * p.T;
  const uint64_t keep = l2_policy_evict_last();

  // Two slots: slot 0 holds the K tile, slot 1 the V tile of the same 16
  // keys. The K tile of the next 16 keys is requested as soon as QK^T has
  // read slot 0, its V tile as soon as PV has read slot 1; both barriers
  // complete once per tile, so the phase parity is the tile count's low bit.
  const uint32_t sk = slots;
  const uint32_t sv = slots + C::kTileBytes;
  const uint32_t bar_k = bars, bar_v = bars + 8;
  auto issue = [&](uint32_t dst, uint32_t bar, const CUtensorMap* tm, int n0) {
#ifdef NSA_DEBUG_BOUNDS
    // a tile the row may read: on a 16-key boundary, at or before the last
    // visible key, inside a block of the index range
    if (lane == 0 && (n0 < 0 || n0 % kTileKeys != 0 || n0 > lastkey || n0 / p.bs >= p.nblk))
      report_bounds();
#endif
    if (lane == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, C::kTileBytes);
#pragma unroll
      for (int h = 0; h < C::kBoxes; ++h)
        tma_load_4d(dst + h * kBoxBytes, tm, bar, h * kBoxCols, g, n0, b, keep);
    }
  };

  TileWalk walk;
  walk.init(irow, static_cast<int>(p.T), p.nblk, p.bs, lastkey);
  int shared_cnt = 0;
  if constexpr (SHARED) {
    // lane j takes id j of the record
    shared_cnt = __shfl_sync(kFull, rec_v, 0);
    const int id = __shfl_sync(kFull, rec_v, (lane + 1) & 31);
    if (shared_cnt > 0) walk.set_skip(id, shared_cnt < kSharedMax ? shared_cnt : kSharedMax);
  }
  int n_next = 0;
  bool have = walk.next(n_next);
  if (have) {
    issue(sk, bar_k, &tmK, n_next);
    issue(sv, bar_v, &tmV, n_next);
  }

  float acc[C::kSteps][4];
#pragma unroll
  for (int i = 0; i < C::kSteps; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m2a = -INFINITY, m2b = -INFINITY;  // reference max, scaled (x = s * sl2), heads 2tig, 2tig+1
  float nega = 0.f, negb = 0.f;            // -reference (0 while a head has seen nothing)
  float la = 0.f, lb = 0.f;                // this lane's share of the row sums
  const float sl2 = p.sl2;
  // two-pass: the tile-shared pass's normalised partial O (8 head rows, 4 KB
  // contiguous) is copied into this warp's shared buffer now and its LSE
  // read into registers; both are merged into the result in the epilogue,
  // so their latency hides behind the whole gather
  float lsa = -INFINITY, lsb = -INFINITY;
  if constexpr (SHARED) {
    if (shared_cnt > 0) {
      if (lane == 0) {
        const float* o = static_cast<const float*>(p.O) + b * p.o_sb + m * p.o_sm + hbase * p.o_sh;
        mbar_arrive_expect_tx(part_bar, C::kPartBytes);
        bulk_load(part, o, C::kPartBytes, part_bar);
      }
      const float* L = p.LSE + (b * p.H + hbase + 2 * tig) * p.M + m;
      lsa = L[0];
      lsb = L[p.M];
    }
  }

  // ldmatrix row addresses: K tiles (row-major A), V tiles (transposed A).
  const uint32_t ka = sk + (lane & 7) * 128 + ((lane & 8) ? 8 * 128 : 0);
  const int ka_hi = lane >> 4;
  const uint32_t va = sv + (lane & 7) * 128 + ((lane & 16) ? 8 * 128 : 0);
  const int va_hi = (lane >> 3) & 1;
  const int sw = lane & 7;  // key row & 7 for both

  uint32_t phase = 0;
  int timed_out = 0;  // 1: K tile missing, 2: V tile missing
  while (have) {
    const int n0 = n_next;
    if (!__all_sync(kFull, wait_phase(bar_k, phase, kWaitLimitNs))) {
      timed_out = 1;
      break;
    }
    // S^T (16 keys x 8 heads) = K_tile Q^T, raw dot products, two MMA chains
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < C::kSteps; k += 2) {
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      ldsm_x4(ka + (k >> 2) * kBoxBytes + ((((k & 3) * 2 + ka_hi) ^ sw) << 4), a0, a1, a2, a3);
      ldsm_x4(ka + ((k + 1) >> 2) * kBoxBytes + (((((k + 1) & 3) * 2 + ka_hi) ^ sw) << 4), b0,
              b1, b2, b3);
      mma_16816_t<BF16>(s, a0, a1, a2, a3, qf[k][0], qf[k][1]);
      mma_16816_t<BF16>(t, b0, b1, b2, b3, qf[k + 1][0], qf[k + 1][1]);
    }
    __syncwarp();
    have = walk.next(n_next);
    if (have) issue(sk, bar_k, &tmK, n_next);  // slot 0 is free

    float x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = (s[j] + t[j]) * sl2;
    const bool edge = n0 + kTileKeys - 1 > lastkey;  // warp-uniform
    if (edge) {
      if (n0 + gid > lastkey) x[0] = x[1] = -INFINITY;
      if (n0 + gid + 8 > lastkey) x[2] = x[3] = -INFINITY;
    }
    // online softmax per head: move the reference only on a large excess
    float mxa = fmaxf(x[0], x[2]);
    float mxb = fmaxf(x[1], x[3]);
    if (__any_sync(kFull, (mxa > m2a + kMaxSlack) || (mxb > m2b + kMaxSlack))) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mxa = fmaxf(mxa, __shfl_xor_sync(kFull, mxa, off));
        mxb = fmaxf(mxb, __shfl_xor_sync(kFull, mxb, off));
      }
      const float mna = fmaxf(m2a, mxa);
      const float mnb = fmaxf(m2b, mxb);
      const float ua = (mna == -INFINITY) ? 0.f : mna;
      const float ub = (mnb == -INFINITY) ? 0.f : mnb;
      const float ala = ex2(m2a - ua);
      const float alb = ex2(m2b - ub);
      m2a = mna;
      m2b = mnb;
      nega = -ua;
      negb = -ub;
      la *= ala;
      lb *= alb;
#pragma unroll
      for (int i = 0; i < C::kSteps; ++i) {
        acc[i][0] *= ala;
        acc[i][1] *= alb;
        acc[i][2] *= ala;
        acc[i][3] *= alb;
      }
    }
    const float p0 = ex2(x[0] + nega);
    const float p1 = ex2(x[1] + negb);
    const float p2 = ex2(x[2] + nega);
    const float p3 = ex2(x[3] + negb);
    la += p0 + p2;
    lb += p1 + p3;
    // P^T as the B operand: (keys 2tig.., head gid) from (key gid, heads 2tig..)
    const uint32_t pb0 = movmatrix_t(pack2_t<BF16>(p0, p1));
    const uint32_t pb1 = movmatrix_t(pack2_t<BF16>(p2, p3));

    if (!__all_sync(kFull, wait_phase(bar_v, phase, kWaitLimitNs))) {
      timed_out = 2;
      break;
    }
    if (edge) {
      // zero the V rows past the last visible key (they may hold anything)
#pragma unroll
      for (int e = lane; e < kTileKeys * (D / 8); e += 32) {
        const int r = e / (D / 8), c = e % (D / 8);
        if (n0 + r > lastkey)
          st_shared_zero16(sv + (c >> 3) * kBoxBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    // O^T (D x 8 heads) += V_tile^T P^T
#pragma unroll
    for (int i = 0; i < C::kSteps; ++i) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(va + (i >> 2) * kBoxBytes + ((((i & 3) * 2 + va_hi) ^ sw) << 4), a0, a1, a2, a3);
      mma_16816_t<BF16>(acc[i], a0, a1, a2, a3, pb0, pb1);
    }
    __syncwarp();
    if (have) issue(sv, bar_v, &tmV, n_next);  // slot 1 is free
    phase ^= 1u;
  }

  if (timed_out) {
    // copies still in flight target this warp's slots: let them land first
    if (lane == 0) report_timeout();
    if constexpr (SHARED) {
      if (shared_cnt > 0) wait_phase(part_bar, 0, kWaitLimitNs);
    }
    if (timed_out == 1) {
      wait_phase(bar_k, phase, kWaitLimitNs);
      wait_phase(bar_v, phase, kWaitLimitNs);
    } else {
      if (have) wait_phase(bar_k, phase ^ 1u, kWaitLimitNs);
      wait_phase(bar_v, phase, kWaitLimitNs);
    }
    return;
  }

  // epilogue: finish the row sums, normalise, store O and LSE
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    la += __shfl_xor_sync(kFull, la, off);
    lb += __shfl_xor_sync(kFull, lb, off);
  }
  if constexpr (SHARED) {
    if (shared_cnt > 0) {
      // merge the partial state: O_s (normalised, weight 2^Ls in log2 units)
      // with this warp's (acc, l) relative to 2^ref
      if (!__all_sync(kFull, wait_phase(part_bar, 0, kWaitLimitNs))) {
        if (lane == 0) report_timeout();
        return;
      }
      constexpr float kLog2e = 1.4426950408889634f;
      float ga = 1.f, sa = 0.f, gb = 1.f, sb = 0.f;  // gather and partial weights
      if (lsa > -INFINITY) {
        const float ls = lsa * kLog2e;
        const float r = fmaxf(m2a, ls);
        ga = m2a == -INFINITY ? 0.f : ex2(m2a - r);
        sa = ex2(ls - r);
        m2a = r;
        la = la * ga + sa;
      }
      if (lsb > -INFINITY) {
        const float ls = lsb * kLog2e;
        const float r = fmaxf(m2b, ls);
        gb = m2b == -INFINITY ? 0.f : ex2(m2b - r);
        sb = ex2(ls - r);
        m2b = r;
        lb = lb * gb + sb;
      }
      // acc[i][0 / 2]: head 2 tig, dims 16 i + gid (+ 8); [1 / 3]: head 2 tig + 1
      const uint32_t pa = part + (2 * tig) * (D * 4) + gid * 4;
      const uint32_t pbh = pa + D * 4;
#pragma unroll
      for (int i = 0; i < C::kSteps; ++i) {
        acc[i][0] = fmaf(acc[i][0], ga, sa * ld_shared_f32(pa + 64 * i));
        acc[i][2] = fmaf(acc[i][2], ga, sa * ld_shared_f32(pa + 64 * i + 32));
        acc[i][1] = fmaf(acc[i][1], gb, sb * ld_shared_f32(pbh + 64 * i));
        acc[i][3] = fmaf(acc[i][3], gb, sb * ld_shared_f32(pbh + 64 * i + 32));
      }
    }
  }
  const float inva = la > 0.f ? 1.f / la : 0.f;
  const float invb = lb > 0.f ? 1.f / lb : 0.f;
  if constexpr (O16) {
    // round, then transpose each 8x8 (dim x head) quarter in registers so a
    // lane holds two adjacent dims of head gid: one 4-byte store per pair
    uint32_t* o = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.O) + b * p.o_sb +
                                              m * p.o_sm + (hbase + gid) * p.o_sh) +
                  tig;
#pragma unroll
    for (int i = 0; i < C::kSteps; ++i) {
      const uint32_t lo = movmatrix_t(pack2_t<BF16>(acc[i][0] * inva, acc[i][1] * invb));
      const uint32_t hi = movmatrix_t(pack2_t<BF16>(acc[i][2] * inva, acc[i][3] * invb));
      if (gid < hw) {
        o[8 * i] = lo;
        o[8 * i + 4] = hi;
      }
    }
  } else {
    const bool ha = 2 * tig < hw, hb = 2 * tig + 1 < hw;  // real heads, not padding
    float* o = static_cast<float*>(p.O) + b * p.o_sb + m * p.o_sm + (hbase + 2 * tig) * p.o_sh +
               gid;
    float* o2 = o + p.o_sh;  // head 2 tig + 1
#pragma unroll
    for (int i = 0; i < C::kSteps; ++i) {
      if (ha) {
        o[16 * i] = acc[i][0] * inva;
        o[16 * i + 8] = acc[i][2] * inva;
      }
      if (hb) {
        o2[16 * i] = acc[i][1] * invb;
        o2[16 * i + 8] = acc[i][3] * invb;
      }
    }
  }
  if (gid == 0) {
    const bool ha = 2 * tig < hw, hb = 2 * tig + 1 < hw;
    constexpr float kLn2 = 0.69314718055994530942f;
    float* L = p.LSE + (b * p.H + hbase + 2 * tig) * p.M + m;
    if (ha) L[0] = la > 0.f ? (m2a + __log2f(la)) * kLn2 : -INFINITY;
    if (hb) L[p.M] = lb > 0.f ? (m2b + __log2f(lb)) * kLn2 : -INFINITY;
  }
}

// A one-warp kernel whose mbarrier never completes: exercises the bounded
// wait and the status word without touching any other memory.
__global__ void selftest_timeout_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(a, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = wait_phase(a, 0, limit_ns);
  if (!__all_sync(kFull, ok) && threadIdx.x == 0) report_timeout();
}

// ---- host side ---------------------------------------------------------------

template <int D, bool BF16, bool O16, bool SHARED = false>
static int launch_fwd(const Problem& p, const void* K, const void* V, int64_t B,
                      const int64_t (&ks)[3], const int64_t (&vs)[3], cudaStream_t stream) {
  constexpr int W = NSA_WARPS;
  using C = Cfg<D, W, SHARED>;
  constexpr CUtensorMapDataType dt =
      BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tk, tv;
  if (p.N > 0) {
    if (!encode_kv_map_strided(&tk, K, B, p.N, p.G, D, kTileKeys, dt, ks[0], ks[1], ks[2]) ||
        !encode_kv_map_strided(&tv, V, B, p.N, p.G, D, kTileKeys, dt, vs[0], vs[1], vs[2]))
      return NSA_ERR_LAUNCH;
  } else {
    memset(&tk, 0, sizeof(tk));  // no key: no tile is ever loaded
    memset(&tv, 0, sizeof(tv));
  }
  auto kern = sel_attn_fwd_kernel<D, W, BF16, O16, SHARED>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return NSA_ERR_LAUNCH;
  const int64_t blocks = (p.units + W - 1) / W;
  kern<<<static_cast<unsigned>(blocks), W * 32, C::kSmemBytes, stream>>>(p, tk, tv);
  return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
}

}  // namespace nsa

namespace nsa {

int check_sizes(int64_t B, int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                int block_size) {
  if (B < 0 || M < 0 || N < 0 || T < 0 || H <= 0 || G <= 0 || D <= 0) return NSA_ERR_SHAPE;
  // heads per group: up to 8 (padded), or a multiple of 8 (sub-groups)
  if (H % G != 0) return NSA_ERR_GROUPS;
  const int64_t hpg = H / G;
  if (hpg > kHeadsPerGroup && hpg % kHeadsPerGroup != 0) return NSA_ERR_GROUPS;
  if (D != 64 && D != 128) return NSA_ERR_HEAD_DIM;
  if (block_size != 32 && block_size != 64) return NSA_ERR_BLOCK_SIZE;
  // 32-bit key / coordinate arithmetic inside the kernel; grid of
  // B*G*(sub-groups)*M warps; 2-D tensor maps over B*M*H head rows
  const int64_t lim = (int64_t(1) << 31) - 1024;
  if (M > lim || N > lim || T > lim || H > lim || B > lim) return NSA_ERR_SHAPE;
  if (B > 0 && M > 0 && B * H > lim / M) return NSA_ERR_SHAPE;
  return NSA_OK;
}

int launch_forward(const void* Q, const void* K, const void* V, const int32_t* block_indices,
                   void* O, float* LSE, int64_t B, int64_t M, int64_t N, int64_t H, int64_t G,
                   int64_t D, int64_t T, int64_t m_off, int block_size, float scale,
                   int qkv_dtype, int o_dtype, const int64_t* strides, cudaStream_t st,
                   const SharedPass* shared) {
  const int chk = check_sizes(B, M, N, H, G, D, T, block_size);
  if (chk != NSA_OK) return chk;
  if ((qkv_dtype != NSA_F16 && qkv_dtype != NSA_BF16) ||
      (o_dtype != NSA_F32 && o_dtype != qkv_dtype))
    return NSA_ERR_DTYPE;
  if (m_off < 0 || m_off > ((int64_t(1) << 31) - 1024) - M) return NSA_ERR_SHAPE;
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
  if (shared != nullptr) {
    const int64_t need = shared_workspace_bytes(B, M, G);
    if (need < 0) return static_cast<int>(need);
    if (shared->workspace == nullptr || shared->workspace_bytes < need) return NSA_ERR_WORKSPACE;
    if (mis(shared->workspace, 16)) return NSA_ERR_ALIGN;
  }
  // element strides (b, m|n, h|g) of Q, K, V, O; d is contiguous
  int64_t sq[3] = {M * H * D, H * D, D}, sk[3] = {N * G * D, G * D, D};
  int64_t sv[3] = {sk[0], sk[1], sk[2]}, so[3] = {sq[0], sq[1], sq[2]};
  if (strides != nullptr) {
    for (int i = 0; i < 3; ++i) {
      sq[i] = strides[i];
      sk[i] = strides[3 + i];
      sv[i] = strides[6 + i];
      so[i] = strides[9 + i];
    }
    // every row start stays 16-byte aligned (TMA, vector loads and stores)
    for (int i = 0; i < 12; ++i) {
      if (strides[i] < 0 || strides[i] > (int64_t(1) << 40)) return NSA_ERR_SHAPE;
      if (strides[i] % 8 != 0) return NSA_ERR_ALIGN;
    }
  }

  Problem p;
  p.Q = static_cast<const uint16_t*>(Q);
  p.idx = block_indices;
  p.O = O;
  p.LSE = LSE;
  p.M = M;
  p.N = N;
  p.H = H;
  p.G = G;
  p.T = T;
  p.q_sb = sq[0];
  p.q_sm = sq[1];
  p.q_sh = sq[2];
  p.o_sb = so[0];
  p.o_sm = so[1];
  p.o_sh = so[2];
  p.m_off = m_off;
  p.hpg = static_cast<int>(H / G);
  p.nsub = head_subgroups(p.hpg);
  p.units = B * G * p.nsub * M;
  p.bs = block_size;
  p.nblk = static_cast<int>((N + block_size - 1) / block_size);
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D));
  p.sl2 = sc * 1.4426950408889634f;
  p.shared = nullptr;
  p.ntiles = 0;
  const bool bf = qkv_dtype == NSA_BF16, o16 = o_dtype != NSA_F32;
  if (shared != nullptr && shared_pass_sizes_ok(M, N, T, block_size) &&
      shared_pass_eligible(H, G, D, o_dtype, strides, m_off)) {
    int32_t* lists = static_cast<int32_t*>(shared->workspace);
    const int rc = launch_shared_passes(Q, K, V, block_indices, static_cast<float*>(O), LSE, B,
                                        M, N, H, G, T, block_size, p.sl2, bf, lists, st);
    if (rc != NSA_OK) return rc;
    p.shared = lists;
    p.ntiles = (M + kSharedTileQ - 1) / kSharedTileQ;
    return bf ? launch_fwd<128, true, false, true>(p, K, V, B, sk, sv, st)
              : launch_fwd<128, false, false, true>(p, K, V, B, sk, sv, st);
  }
  if (D == 64) {
    if (bf) return o16 ? launch_fwd<64, true, true>(p, K, V, B, sk, sv, st)
                       : launch_fwd<64, true, false>(p, K, V, B, sk, sv, st);
    return o16 ? launch_fwd<64, false, true>(p, K, V, B, sk, sv, st)
               : launch_fwd<64, false, false>(p, K, V, B, sk, sv, st);
  }
  if (bf) return o16 ? launch_fwd<128, true, true>(p, K, V, B, sk, sv, st)
                     : launch_fwd<128, true, false>(p, K, V, B, sk, sv, st);
  return o16 ? launch_fwd<128, false, true>(p, K, V, B, sk, sv, st)
             : launch_fwd<128, false, false>(p, K, V, B, sk, sv, st);
}

int fwd_read_and_clear_status(unsigned int* value) { return read_and_clear_status(value); }

}  // namespace nsa

extern "C" {

int nsa_sel_attn_fwd(const void* Q, const void* K, const void* V, const int32_t* block_indices,
                     float* O, float* LSE, int64_t B, int64_t M, int64_t N, int64_t H, int64_t G,
                     int64_t D, int64_t T, int block_size, float scale, void* stream) {
  return nsa::launch_forward(Q, K, V, block_indices, O, LSE, B, M, N, H, G, D, T, 0, block_size,
                             scale, NSA_F16, NSA_F32, nullptr, static_cast<cudaStream_t>(stream));
}

int nsa_sel_attn_fwd_ex(const void* Q, const void* K, const void* V,
                        const int32_t* block_indices, void* O, float* LSE, int64_t B, int64_t M,
                        int64_t N, int64_t H, int64_t G, int64_t D, int64_t T, int block_size,
                        float scale, int qkv_dtype, int o_dtype, void* stream) {
  return nsa::launch_forward(Q, K, V, block_indices, O, LSE, B, M, N, H, G, D, T, 0, block_size,
                             scale, qkv_dtype, o_dtype, nullptr, static_cast<cudaStream_t>(stream));
}

int nsa_sel_attn_fwd_strided(const void* Q, const void* K, const void* V,
                             const int32_t* block_indices, void* O, float* LSE, int64_t B,
                             int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                             int block_size, float scale, int qkv_dtype, int o_dtype,
                             const int64_t* strides, void* stream) {
  return nsa::launch_forward(Q, K, V, block_indices, O, LSE, B, M, N, H, G, D, T, 0, block_size,
                             scale, qkv_dtype, o_dtype, strides,
                             static_cast<cudaStream_t>(stream));
}

int64_t nsa_sel_attn_fwd_shared_workspace_bytes(int64_t B, int64_t M, int64_t G) {
  return nsa::shared_workspace_bytes(B, M, G);
}

int nsa_sel_attn_fwd_shared(const void* Q, const void* K, const void* V,
                            const int32_t* block_indices, float* O, float* LSE, int64_t B,
                            int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                            int block_size, float scale, int qkv_dtype, void* workspace,
                            int64_t workspace_bytes, void* stream) {
  const nsa::SharedPass sp{workspace, workspace_bytes};
  return nsa::launch_forward(Q, K, V, block_indices, O, LSE, B, M, N, H, G, D, T, 0, block_size,
                             scale, qkv_dtype, NSA_F32, nullptr,
                             static_cast<cudaStream_t>(stream), &sp);
}

int nsa_selftest_wait_timeout(int64_t limit_ns, void* stream) {
  if (limit_ns < 1000 || limit_ns > 2000000000) return NSA_ERR_SHAPE;
  nsa::selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? NSA_OK : NSA_ERR_LAUNCH;
}

}  // extern "C"
