// Host-buffer entry point: chunked upload / forward / download pipeline.
//
// The queries are cut into chunks of chunk_m positions. Chunk c uses buffer
// slot c % 2 of the caller's device workspace:
//   upload stream   : K/V rows [kv_done, min(N, end_c)) (each key row once),
//                     Q rows and index rows of the chunk          -> event up[c%2]
//   compute streams : forward kernel over the chunk (query positions start
//                     at the chunk's first position); even chunks on the
//                     caller's stream, odd chunks on a second one  -> event fw[c%2]
//   download stream : O rows and LSE columns of the chunk         -> event dn[c%2]
// Slot reuse is ordered by events: the upload of chunk c waits fw of chunk
// c-2 (its Q/index slot has been read), the kernel of chunk c waits dn of
// chunk c-2 (its O/LSE slot has been copied out). Every copy is one plain
// cudaMemcpy2DAsync (strided rows for B > 1 and for LSE's [B, H, M] layout).
//
// A kernel only reads keys up to its queries' last visible position, all of
// which were uploaded before it starts; the rest of the K/V workspace may be
// stale or in the middle of a later upload, and the kernel's masking keeps
// such rows out of the result.

#include <cuda_runtime.h>

#include <cstdint>

#include "nsa_sel_attn.h"
#include "sel_attn_fwd.cuh"

namespace nsa {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct HostPlan {
  int64_t chunk;        // queries per chunk
  int64_t nchunks;
  size_t off_k, off_v;  // full K and V
  size_t off_q[2], off_idx[2], off_o[2], off_lse[2];
  size_t total;
};

int64_t default_chunk(int64_t M) {
  int64_t c = (M + 31) / 32;
  c = (c + 63) / 64 * 64;
  if (c < 64) c = 64;
  return c < M ? c : M;
}

HostPlan make_plan(int64_t B, int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                   int64_t chunk_m) {
  HostPlan pl;
  // chunks start at multiples of 64 positions, so a chunk's kernel groups its
  // queries exactly as a single launch over all M would (bit-identical output)
  const int64_t c64 = chunk_m > 0 ? (chunk_m + 63) / 64 * 64 : 0;
  pl.chunk = c64 > 0 ? (c64 < M ? c64 : M) : default_chunk(M);
  if (pl.chunk < 1) pl.chunk = 1;
  pl.nchunks = M > 0 ? (M + pl.chunk - 1) / pl.chunk : 0;
  const size_t kv = align_up(static_cast<size_t>(B * N * G * D) * 2);
  const size_t q = align_up(static_cast<size_t>(B * pl.chunk * H * D) * 2);
  const size_t ix = align_up(static_cast<size_t>(B * pl.chunk * G * T) * 4);
  const size_t o = align_up(static_cast<size_t>(B * pl.chunk * H * D) * 4);
  const size_t l = align_up(static_cast<size_t>(B * H * pl.chunk) * 4);
  size_t at = 0;
  pl.off_k = at;
  at += kv;
  pl.off_v = at;
  at += kv;
  for (int s = 0; s < 2; ++s) {
    pl.off_q[s] = at;
    at += q;
    pl.off_idx[s] = at;
    at += ix;
    pl.off_o[s] = at;
    at += o;
    pl.off_lse[s] = at;
    at += l;
  }
  pl.total = at;
  return pl;
}

// Streams and events of one call; released (deferred by CUDA until their
// work completes) when the call returns.
struct CallResources {
  cudaStream_t up = nullptr, dn = nullptr, fw2 = nullptr;
  cudaEvent_t start = nullptr, up_ev[2] = {nullptr, nullptr}, fw_ev[2] = {nullptr, nullptr},
              dn_ev[2] = {nullptr, nullptr}, join[3] = {nullptr, nullptr, nullptr};
  bool ok = true;

  CallResources() {
    ok = cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking) == cudaSuccess &&
         cudaStreamCreateWithFlags(&dn, cudaStreamNonBlocking) == cudaSuccess &&
         cudaStreamCreateWithFlags(&fw2, cudaStreamNonBlocking) == cudaSuccess &&
         cudaEventCreateWithFlags(&start, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < 3 && ok; ++i)
      ok = cudaEventCreateWithFlags(&join[i], cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; s < 2 && ok; ++s)
      ok = cudaEventCreateWithFlags(&up_ev[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&fw_ev[s], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&dn_ev[s], cudaEventDisableTiming) == cudaSuccess;
  }
  ~CallResources() {
    for (int s = 0; s < 2; ++s) {
      if (up_ev[s]) cudaEventDestroy(up_ev[s]);
      if (fw_ev[s]) cudaEventDestroy(fw_ev[s]);
      if (dn_ev[s]) cudaEventDestroy(dn_ev[s]);
    }
    for (int i = 0; i < 3; ++i)
      if (join[i]) cudaEventDestroy(join[i]);
    if (start) cudaEventDestroy(start);
    if (up) cudaStreamDestroy(up);
    if (dn) cudaStreamDestroy(dn);
    if (fw2) cudaStreamDestroy(fw2);
  }
};

// Copies `height` rows of `width` bytes between pitched buffers.
bool copy2d(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, size_t height,
            cudaMemcpyKind kind, cudaStream_t st) {
  if (width == 0 || height == 0) return true;
  return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, kind, st) == cudaSuccess;
}

}  // namespace
}  // namespace nsa

extern "C" {

int64_t nsa_sel_attn_fwd_host_workspace_bytes(int64_t B, int64_t M, int64_t N, int64_t H,
                                              int64_t G, int64_t D, int64_t T, int block_size,
                                              int64_t chunk_m) {
  const int chk = nsa::check_sizes(B, M, N, H, G, D, T, block_size);
  if (chk != NSA_OK) return chk;
  return static_cast<int64_t>(nsa::make_plan(B, M, N, H, G, D, T, chunk_m).total);
}

int nsa_sel_attn_fwd_host_ex(const void* Q, const void* K, const void* V,
                             const int32_t* block_indices, void* O, float* LSE, int64_t B,
                             int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                             int block_size, float scale, int qkv_dtype, int o_dtype,
                             void* workspace, int64_t workspace_bytes, int64_t chunk_m,
                             void* stream) {
  using namespace nsa;
  const int chk = check_sizes(B, M, N, H, G, D, T, block_size);
  if (chk != NSA_OK) return chk;
  if ((qkv_dtype != NSA_F16 && qkv_dtype != NSA_BF16) ||
      (o_dtype != NSA_F32 && o_dtype != qkv_dtype))
    return NSA_ERR_DTYPE;
  if (B == 0 || M == 0) return NSA_OK;
  if (!Q || !O || !LSE) return NSA_ERR_NULL;
  if (N > 0 && (!K || !V)) return NSA_ERR_NULL;
  if (T > 0 && !block_indices) return NSA_ERR_NULL;
  const HostPlan pl = make_plan(B, M, N, H, G, D, T, chunk_m);
  if (!workspace || workspace_bytes < static_cast<int64_t>(pl.total)) return NSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return NSA_ERR_ALIGN;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CallResources r;
  if (!r.ok) return NSA_ERR_LAUNCH;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* dK = ws + pl.off_k;
  void* dV = ws + pl.off_v;
  const size_t kv_row = static_cast<size_t>(G * D) * 2;       // one key, all groups
  const size_t q_row = static_cast<size_t>(H * D) * 2;        // one query, all heads
  const size_t i_row = static_cast<size_t>(G * T) * 4;        // one query's index rows
  const size_t o_row = static_cast<size_t>(H * D) * (o_dtype == NSA_F32 ? 4 : 2);  // one query's O rows
  const uint8_t* hK = static_cast<const uint8_t*>(K);
  const uint8_t* hV = static_cast<const uint8_t*>(V);
  const uint8_t* hQ = static_cast<const uint8_t*>(Q);
  const uint8_t* hI = reinterpret_cast<const uint8_t*>(block_indices);
  uint8_t* hO = reinterpret_cast<uint8_t*>(O);
  uint8_t* hL = reinterpret_cast<uint8_t*>(LSE);

  bool ok = cudaEventRecord(r.start, st) == cudaSuccess &&
            cudaStreamWaitEvent(r.up, r.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(r.dn, r.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(r.fw2, r.start, 0) == cudaSuccess;
  int status = NSA_OK;
  int64_t kv_done = 0;
  for (int64_t c = 0; c < pl.nchunks && ok; ++c) {
    const int s = static_cast<int>(c & 1);
    const int64_t m0 = c * pl.chunk;
    const int64_t mc = (M - m0) < pl.chunk ? (M - m0) : pl.chunk;
    uint8_t* dQ = ws + pl.off_q[s];
    uint8_t* dI = ws + pl.off_idx[s];
    void* dO = ws + pl.off_o[s];  // sized for fp32: a 16-bit O uses half
    float* dL = reinterpret_cast<float*>(ws + pl.off_lse[s]);

    // upload: visible K/V rows not yet on the device, then this chunk's rows
    if (c >= 2) ok = ok && cudaStreamWaitEvent(r.up, r.fw_ev[s], 0) == cudaSuccess;
    const int64_t kv_need = (m0 + mc) < N ? (m0 + mc) : N;
    if (kv_need > kv_done) {
      const size_t off = static_cast<size_t>(kv_done) * kv_row;
      const size_t w = static_cast<size_t>(kv_need - kv_done) * kv_row;
      const size_t pitch = static_cast<size_t>(N) * kv_row;
      ok = ok && copy2d(static_cast<uint8_t*>(dK) + off, pitch, hK + off, pitch, w, B,
                        cudaMemcpyHostToDevice, r.up);
      ok = ok && copy2d(static_cast<uint8_t*>(dV) + off, pitch, hV + off, pitch, w, B,
                        cudaMemcpyHostToDevice, r.up);
      kv_done = kv_need;
    }
    ok = ok && copy2d(dQ, mc * q_row, hQ + m0 * q_row, M * q_row, mc * q_row, B,
                      cudaMemcpyHostToDevice, r.up);
    if (T > 0)
      ok = ok && copy2d(dI, mc * i_row, hI + m0 * i_row, M * i_row, mc * i_row, B,
                        cudaMemcpyHostToDevice, r.up);
    ok = ok && cudaEventRecord(r.up_ev[s], r.up) == cudaSuccess;

    // forward: chunks are independent (disjoint queries), so even chunks run
    // on the caller's stream and odd ones on a second stream, letting one
    // kernel's last wave overlap the next kernel
    cudaStream_t fs = s == 0 ? st : r.fw2;
    ok = ok && cudaStreamWaitEvent(fs, r.up_ev[s], 0) == cudaSuccess;
    if (c >= 2) ok = ok && cudaStreamWaitEvent(fs, r.dn_ev[s], 0) == cudaSuccess;
    if (!ok) break;
    const int rc = launch_forward(dQ, N > 0 ? dK : nullptr, N > 0 ? dV : nullptr,
                                  T > 0 ? reinterpret_cast<const int32_t*>(dI) : nullptr, dO,
                                  dL, B, mc, N, H, G, D, T, m0, block_size, scale, qkv_dtype,
                                  o_dtype, nullptr, fs);
    if (rc != NSA_OK) {
      status = rc;
      break;
    }
    ok = cudaEventRecord(r.fw_ev[s], fs) == cudaSuccess;

    // download: O rows [m0, m0+mc) of every batch, LSE columns of every (b, h)
    ok = ok && cudaStreamWaitEvent(r.dn, r.fw_ev[s], 0) == cudaSuccess;
    ok = ok && copy2d(hO + m0 * o_row, M * o_row, dO, mc * o_row, mc * o_row, B,
                      cudaMemcpyDeviceToHost, r.dn);
    ok = ok && copy2d(hL + m0 * 4, M * 4, dL, mc * 4, mc * 4, B * H, cudaMemcpyDeviceToHost,
                      r.dn);
    ok = ok && cudaEventRecord(r.dn_ev[s], r.dn) == cudaSuccess;
  }
  // The caller's stream completes only after everything this call queued on
  // its internal streams, on every path: copies that read or write the
  // caller's host buffers are never left in flight behind an error return.
  // If the join itself fails, the internal streams are waited for here.
  const cudaStream_t internal[3] = {r.up, r.fw2, r.dn};
  bool joined = true;
  for (int i = 0; i < 3; ++i)
    joined = joined && cudaEventRecord(r.join[i], internal[i]) == cudaSuccess &&
             cudaStreamWaitEvent(st, r.join[i], 0) == cudaSuccess;
  if (!joined)
    for (int i = 0; i < 3; ++i) cudaStreamSynchronize(internal[i]);
  if (status != NSA_OK) return status;
  return ok && joined ? NSA_OK : NSA_ERR_LAUNCH;
}

int nsa_sel_attn_fwd_host(const void* Q, const void* K, const void* V,
                          const int32_t* block_indices, float* O, float* LSE, int64_t B,
                          int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                          int block_size, float scale, void* workspace, int64_t workspace_bytes,
                          int64_t chunk_m, void* stream) {
  return nsa_sel_attn_fwd_host_ex(Q, K, V, block_indices, O, LSE, B, M, N, H, G, D, T,
                                  block_size, scale, NSA_F16, NSA_F32, workspace, workspace_bytes,
                                  chunk_m, stream);
}

}  // extern "C"
