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
int launch_forward(const void* Q, const void* K, const void* V, const int32_t* block_indices,
                   void* O, float* LSE, int64_t B, int64_t M, int64_t N, int64_t H, int64_t G,
                   int64_t D, int64_t T, int64_t m_off, int block_size, float scale,
                   int qkv_dtype, int o_dtype, const int64_t* strides, cudaStream_t st);

}  // namespace nsa
