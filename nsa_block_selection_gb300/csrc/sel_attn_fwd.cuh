// Internal interface of the forward kernel, shared by the library's entry
// points (device buffers, host buffers). Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace nsa {

// Size checks common to every entry point; NSA_OK or a negative nsa_status.
int check_sizes(int64_t B, int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                int block_size);

// Validates and launches the forward over query rows [0, M) of Q / indices /
// O / LSE, whose positions in the key sequence are m_off .. m_off + M - 1.
// K and V hold the whole key sequence [B, N, G, D]; LSE is [B, H, M].
// qkv_dtype / o_dtype are nsa_dtype values (Q/K/V fp16 or bf16; O fp32 or
// the 16-bit type of Q/K/V). `strides`: NULL (contiguous) or 12 element
// strides, (b, m, h) of Q, (b, n, g) of K and of V, (b, m, h) of O.
//
// `shared`: NULL, or the workspace of the two-pass path (nsa_sel_attn_fwd_shared):
// where shared_pass_eligible() holds, the blocks common to each tile of
// kSharedTileQ queries are attended to first by the tile-shared pass, which
// leaves its partial O / LSE in the outputs, and the gather kernel skips them
// and continues from that state.
struct SharedPass {
  void* workspace;
  int64_t workspace_bytes;
};

int launch_forward(const void* Q, const void* K, const void* V, const int32_t* block_indices,
                   void* O, float* LSE, int64_t B, int64_t M, int64_t N, int64_t H, int64_t G,
                   int64_t D, int64_t T, int64_t m_off, int block_size, float scale,
                   int qkv_dtype, int o_dtype, const int64_t* strides, cudaStream_t st,
                   const SharedPass* shared = nullptr);

// ---- two-pass path (sel_attn_shared.cu) ----

// Workspace of the two-pass path: one record per (b, g, query tile), or a
// negative nsa_status for invalid sizes.
int64_t shared_workspace_bytes(int64_t B, int64_t M, int64_t G);

// Sizes and types the tile-shared pass serves: D = 128, 8 query heads per KV
// group, fp32 O, contiguous tensors, the whole query sequence (m_off = 0).
bool shared_pass_eligible(int64_t H, int64_t G, int64_t D, int o_dtype,
                          const int64_t* strides, int64_t m_off);

// Sizes the two-pass path takes (else the one-pass kernel runs): at least one
// full query tile, one full block of keys, and an index row.
bool shared_pass_sizes_ok(int64_t M, int64_t N, int64_t T, int block_size);

// Enqueues the list pass (per tile: the blocks every query of the tile lists
// and sees whole) and the tile-shared pass (their partial softmax for all
// 128 rows of the tile, written to O and LSE). Arguments were validated by
// launch_forward. Returns NSA_OK or NSA_ERR_LAUNCH.
int launch_shared_passes(const void* Q, const void* K, const void* V, const int32_t* idx,
                         float* O, float* LSE, int64_t B, int64_t M, int64_t N, int64_t H,
                         int64_t G, int64_t T, int block_size, float sl2, bool bf16,
                         int32_t* lists, cudaStream_t st);

}  // namespace nsa
