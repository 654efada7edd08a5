/*
 * nsa_sel_attn.h -- C ABI of the NSA selection-attention forward library
 * (libnsa_sel_attn.so, sm_103a).
 *
 * The operation is the one stated in "[wave] NSA: selection attention forward
 * kernel":
 *   section "Operation"    -- Q [B,M,H,D], K [B,N,G,D], V [B,N,G,D],
 *                             block_indices [B,M,G,T] in; O_slc [B,M,H,D],
 *                             LSE_slc [B,H,M] out; T = selected blocks/query;
 *   section "Algorithm"    -- for query m and each selected block t, the keys
 *                             [t*block_size, (t+1)*block_size) are gathered,
 *                             scored against q[m] (QK^T), causally masked and
 *                             softmaxed; V is accumulated with an online
 *                             softmax (running max + log-sum-exp); O and LSE
 *                             are stored;
 *   section "Requirements" -- the heads of a GQA group share block_indices;
 *                             online softmax across all T blocks; causal mask
 *                             inside gathered blocks; FP16 matmuls with FP32
 *                             accumulation; LSE returned for the backward
 *                             pass; block_size 64 and 32.
 *
 * Conventions where the pages are silent (the library's contract):
 *   - head h belongs to KV group h / (H/G) (contiguous heads per group);
 *   - key n is visible to query m iff n <= m and n < N;
 *   - scores are multiplied by `scale` (pass <= 0 for 1/sqrt(D));
 *   - block_indices entries < 0 or >= ceil(N/block_size) are padding and may
 *     sit anywhere in a row; a row must not list a block twice (a top-k
 *     output never does; a repeated block is counted twice);
 *   - a row with no visible key yields O = 0 and LSE = -inf;
 *   - LSE is the natural log of sum(exp(scale * q.k)) over visible keys.
 *
 * Every buffer is contiguous row-major in the layout given, owned by the
 * caller, and not retained after the call returns. Key/value rows that no
 * index selects are never read; rows after a query inside its own 16-key
 * tile may be read but never reach the output (whatever they hold).
 */
#ifndef NSA_SEL_ATTN_H
#define NSA_SEL_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. Values < 0 are errors; nothing was launched when an argument
 * check fails. */
typedef enum nsa_status {
  NSA_OK = 0,
  NSA_ERR_NULL = -1,        /* a required pointer is NULL                     */
  NSA_ERR_SHAPE = -2,       /* a size is negative or the sizes are too large */
  NSA_ERR_BLOCK_SIZE = -3,  /* block_size not in {32, 64}                     */
  NSA_ERR_HEAD_DIM = -4,    /* D not in {64, 128}                             */
  NSA_ERR_GROUPS = -5,      /* H % G != 0, or H/G > 8 and not a multiple of 8 */
  NSA_ERR_ALIGN = -6,       /* Q, K, V or O not 16-byte aligned, LSE or
                               block_indices not 4-byte aligned               */
  NSA_ERR_LAUNCH = -7,      /* the CUDA runtime refused the launch or a copy
                               (no device, no sm_103a image, bad stream ...) */
  NSA_ERR_TIMEOUT = -8,     /* a bounded device-side wait gave up (reported by
                               nsa_sync_status)                               */
  NSA_ERR_WORKSPACE = -9,   /* workspace NULL or smaller than required        */
  NSA_ERR_SCRATCH = -10,    /* problem needs more scratch than the fixed
                               buffer of nsa_sel_attn_bwd_noalloc (64 MiB)    */
  NSA_ERR_DTYPE = -11,      /* element type combination not supported by
                               nsa_sel_attn_fwd_ex                            */
  NSA_ERR_BOUNDS = -12      /* (library built with NSA_DEBUG_BOUNDS only) a
                               kernel's own bounds check found a tile outside
                               the keys its row may read; reported by
                               nsa_sync_status                                */
} nsa_status;

/* Element types of nsa_sel_attn_fwd_ex. */
typedef enum nsa_dtype {
  NSA_F16 = 0,   /* IEEE binary16                                  */
  NSA_BF16 = 1,  /* bfloat16 (the upper 16 bits of an IEEE binary32) */
  NSA_F32 = 2    /* IEEE binary32                                  */
} nsa_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* nsa_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int nsa_version(void);

/*
 * nsa_sel_attn_fwd -- selection-attention forward on the GPU.
 *
 *   Q              device, IEEE fp16, [B, M, H, D]
 *   K, V           device, IEEE fp16, [B, N, G, D]
 *   block_indices  device, int32,     [B, M, G, T]; block ids, -1 = padding
 *   O              device, fp32,      [B, M, H, D]   (output)
 *   LSE            device, fp32,      [B, H, M]      (output, natural log)
 *   B, M, N, T     >= 0; an empty problem (B*M == 0) returns NSA_OK at once
 *   H, G, D        > 0, H % G == 0, D in {64, 128}; H/G (query heads per
 *                  KV group) is 1..8, or a multiple of 8 -- a warp serves up to
 *                  8 heads of a group: fewer are padded, more are split into
 *                  sub-groups of 8 that share the group's K/V and index row
 *   block_size     32 or 64
 *   scale          score multiplier; <= 0 selects 1/sqrt(D)
 *   stream         cudaStream_t to launch on (NULL = legacy default stream)
 *
 * Asynchronous: validates the arguments on the host, enqueues one kernel on
 * `stream` and returns without synchronising. K and V are fetched with TMA
 * through tensor maps encoded on the host for each call. It allocates
 * nothing, frees nothing and keeps no state between calls (the per-device
 * status word of nsa_sync_status aside); concurrent calls on different
 * streams are safe. Returns NSA_OK, or a negative nsa_status. Errors that
 * surface only when the kernel runs are reported by the next CUDA call that
 * synchronises with `stream`, as for any CUDA launch.
 */
int nsa_sel_attn_fwd(const void* Q, const void* K, const void* V,
                     const int32_t* block_indices, float* O, float* LSE,
                     int64_t B, int64_t M, int64_t N, int64_t H, int64_t G,
                     int64_t D, int64_t T, int block_size, float scale,
                     void* stream);

/*
 * nsa_sel_attn_fwd_ex -- nsa_sel_attn_fwd with a choice of element types.
 *
 *   qkv_dtype  NSA_F16 or NSA_BF16: the type of Q, K and V (all three alike)
 *   o_dtype    NSA_F32, or qkv_dtype: the type O is written in
 *
 * Every other argument, layout, check and property is that of
 * nsa_sel_attn_fwd; LSE stays fp32. nsa_sel_attn_fwd is this call with
 * (NSA_F16, NSA_F32). With bf16 inputs both products run as bf16 MMAs with
 * fp32 accumulation, so the probabilities are rounded to bf16 (8 significant
 * bits) before the PV product -- the bf16 reading of the "FP16 matmuls, FP32
 * accumulation" requirement ("[wave] NSA: selection attention forward
 * kernel", section "Requirements"). Scores, running max and row sums are
 * fp32 in every combination; a 16-bit O is the fp32 result rounded to
 * nearest even. Any other combination returns NSA_ERR_DTYPE before launch.
 */
int nsa_sel_attn_fwd_ex(const void* Q, const void* K, const void* V,
                        const int32_t* block_indices, void* O, float* LSE,
                        int64_t B, int64_t M, int64_t N, int64_t H, int64_t G,
                        int64_t D, int64_t T, int block_size, float scale,
                        int qkv_dtype, int o_dtype, void* stream);

/*
 * nsa_sel_attn_fwd_strided -- nsa_sel_attn_fwd_ex on strided tensors.
 *
 *   strides  host array of 12 element strides, or NULL for contiguous:
 *            [0..2]  Q over (b, m, h)     [3..5]  K over (b, n, g)
 *            [6..8]  V over (b, n, g)     [9..11] O over (b, m, h)
 *            The last dimension (d) of Q, K, V and O is contiguous; LSE and
 *            block_indices are contiguous as in nsa_sel_attn_fwd.
 *
 * Lets Q, K and V be views into one fused projection (for example
 * [B, M, H + 2G, D] with Q the first H heads) and O a slice of a larger
 * buffer, without copies. Every stride must be a multiple of 8 elements (so
 * every row starts 16-byte aligned; else NSA_ERR_ALIGN) and in
 * [0, 2^40] (else NSA_ERR_SHAPE); the strides must describe memory the
 * caller owns, and O must not overlap Q, K or V. Everything else is
 * nsa_sel_attn_fwd_ex.
 */
int nsa_sel_attn_fwd_strided(const void* Q, const void* K, const void* V,
                             const int32_t* block_indices, void* O, float* LSE,
                             int64_t B, int64_t M, int64_t N, int64_t H, int64_t G,
                             int64_t D, int64_t T, int block_size, float scale,
                             int qkv_dtype, int o_dtype, const int64_t* strides,
                             void* stream);

/*
 * nsa_sel_attn_fwd_shared_workspace_bytes -- device workspace of
 * nsa_sel_attn_fwd_shared: one 32-byte record per (b, g, tile of 16
 * queries), rounded up to 256 bytes. Negative nsa_status for invalid sizes
 * (B * G * ceil(M/16) must stay below 2^31). Pure host arithmetic.
 */
int64_t nsa_sel_attn_fwd_shared_workspace_bytes(int64_t B, int64_t M, int64_t G);

/*
 * nsa_sel_attn_fwd_shared -- the forward of nsa_sel_attn_fwd_ex (O fp32) in
 * two passes over the blocks that consecutive queries share.
 *
 *   qkv_dtype   NSA_F16 or NSA_BF16
 *   workspace   device memory of at least
 *               nsa_sel_attn_fwd_shared_workspace_bytes(B, M, G) bytes,
 *               16-byte aligned, owned by the caller (else NSA_ERR_WORKSPACE
 *               or NSA_ERR_ALIGN); on return it holds the per-tile records
 *
 * Index rows that keep the initial block and the most recent blocks of
 * every query (as nsa_topk_blocks with n_init, n_local > 0 writes them) give
 * the queries of a tile of 16 consecutive positions some blocks in common.
 * Per (b, g, tile) a list pass records up to 7
 * blocks that every query of the tile lists, whose first key the tile's
 * first query sees and whose keys all lie below M and N, in the order the
 * tile's first query lists them. A tile-shared pass gathers those blocks
 * once and computes, on the tcgen05 tensor cores, the softmax of all
 * 16 x 8 (query, head) rows over their keys (each row masked to the keys
 * at or before its query); it writes the normalised partial O and its LSE
 * into O and LSE. The gather kernel of
 * nsa_sel_attn_fwd then skips the recorded blocks and continues the online
 * softmax from that state, so its outputs cover every selected key once.
 * The result is the same operation as nsa_sel_attn_fwd_ex with the same
 * tolerance (the partial sums are added in another order; outputs are not
 * bit-identical to the one-pass call). Three kernels are enqueued on
 * `stream`; nothing is allocated or synchronised.
 *
 * The two-pass path serves block_size = 64, D = 128, H/G = 8, M >= 16,
 * N >= block_size and T >= 1; any other valid problem runs the one-pass
 * kernel (the workspace is then unused). With 32-key blocks the common
 * blocks are too small a share of a row's bytes for the extra passes to pay
 * (measured slower than one pass), so those problems take the one-pass
 * kernel too. Every other argument, layout, check and property is that
 * of nsa_sel_attn_fwd_ex, with one difference in what non-finite inputs
 * may do: NaN or Inf in K/V rows past every query (>= M), in blocks no
 * query lists, and in the keys of a tile's own block past the tile's last
 * query never reach an output (as for the one-pass call), but a non-finite
 * V row between two queries of the same 16-query tile reaches the earlier
 * query's output too (the tile's rows share one P.V product over those
 * keys).
 */
int nsa_sel_attn_fwd_shared(const void* Q, const void* K, const void* V,
                            const int32_t* block_indices, float* O, float* LSE, int64_t B,
                            int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                            int block_size, float scale, int qkv_dtype, void* workspace,
                            int64_t workspace_bytes, void* stream);

/*
 * nsa_sel_attn_fwd_host_workspace_bytes -- device workspace that
 * nsa_sel_attn_fwd_host needs for these sizes and query chunk length
 * (chunk_m <= 0 selects the default). Returns the byte count, or a negative
 * nsa_status for invalid sizes. Pure host arithmetic; no CUDA call.
 */
int64_t nsa_sel_attn_fwd_host_workspace_bytes(int64_t B, int64_t M, int64_t N, int64_t H,
                                              int64_t G, int64_t D, int64_t T, int block_size,
                                              int64_t chunk_m);

/*
 * nsa_sel_attn_fwd_host -- the same forward with HOST buffers in and out.
 *
 *   Q, K, V, block_indices   host memory, layouts as in nsa_sel_attn_fwd
 *   O, LSE                   host memory, written
 *   workspace                device memory of at least
 *                            nsa_sel_attn_fwd_host_workspace_bytes(...) bytes,
 *                            256-byte aligned, owned by the caller
 *   chunk_m                  queries per pipeline chunk, rounded up to a
 *                            multiple of 64 (<= 0: default, about M/32)
 *   stream                   caller's stream: the call's work starts after
 *                            the work already queued on it, and it waits for
 *                            all of the call's work
 *
 * The queries are processed in chunks of chunk_m positions. For each chunk
 * the call enqueues, on an internal upload stream, the copies of its Q rows,
 * its index rows and the K/V rows it can see (keys below the chunk's end,
 * each copied once); the kernel (even chunks on `stream`, odd chunks on an
 * internal second compute stream); and on an internal download
 * stream, the copies of its O rows and LSE columns. Chunk buffers are double
 * buffered in the workspace, so uploads, kernels and downloads of adjacent
 * chunks overlap. Copies overlap only if the host buffers are page-locked
 * (pinned); with pageable memory they are correct but serial.
 *
 * Returns after enqueueing; `stream` is made to wait for every copy, so the
 * outputs are complete once `stream` is synchronised. Results are
 * bit-identical to nsa_sel_attn_fwd on the same inputs. It allocates no
 * memory (the internal streams and events are created and released by the
 * call). Errors: as nsa_sel_attn_fwd, plus NSA_ERR_WORKSPACE.
 */
int nsa_sel_attn_fwd_host(const void* Q, const void* K, const void* V,
                          const int32_t* block_indices, float* O, float* LSE, int64_t B,
                          int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                          int block_size, float scale, void* workspace,
                          int64_t workspace_bytes, int64_t chunk_m, void* stream);

/*
 * nsa_sel_attn_fwd_host_ex -- nsa_sel_attn_fwd_host with the element types of
 * nsa_sel_attn_fwd_ex: Q, K, V in host memory as qkv_dtype (NSA_F16 or
 * NSA_BF16), O written as o_dtype (NSA_F32 or qkv_dtype); LSE fp32. Any
 * other combination returns NSA_ERR_DTYPE before anything is enqueued. The
 * workspace of nsa_sel_attn_fwd_host_workspace_bytes (sized for fp32 O)
 * suffices for every combination. Results are bit-identical to
 * nsa_sel_attn_fwd_ex on the same inputs; everything else is
 * nsa_sel_attn_fwd_host.
 */
int nsa_sel_attn_fwd_host_ex(const void* Q, const void* K, const void* V,
                             const int32_t* block_indices, void* O, float* LSE, int64_t B,
                             int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                             int block_size, float scale, int qkv_dtype, int o_dtype,
                             void* workspace, int64_t workspace_bytes, int64_t chunk_m,
                             void* stream);

/*
 * nsa_sel_attn_bwd_workspace_bytes -- device workspace nsa_sel_attn_bwd
 * needs: an fp16 copy of dO, one 64-byte (LSE, delta) record per (b, m, g,
 * 8-head sub-group), the per-(b, g, block) query lists (at most B*M*G*T
 * entries) and their counts and offsets, and 8 bytes per (b, m, g) row
 * for the row's local entries. Negative nsa_status for invalid sizes
 * (B*M*G*T must stay below 2^31). Pure host arithmetic.
 */
int64_t nsa_sel_attn_bwd_workspace_bytes(int64_t B, int64_t M, int64_t N, int64_t H,
                                         int64_t G, int64_t D, int64_t T, int block_size);

/*
 * nsa_sel_attn_bwd -- gradients of nsa_sel_attn_fwd (the section
 * "Requirements" returns LSE for this pass).
 *
 *   Q, K, V, block_indices   as for the forward (device)
 *   O, LSE                   the forward's outputs (device, fp32)
 *   dO                       upstream gradient of O, fp32 [B, M, H, D]
 *   dQ                       fp32 [B, M, H, D]   (written)
 *   dK, dV                   fp32 [B, N, G, D]   (written; zeroed first)
 *   workspace                device memory of at least
 *                            nsa_sel_attn_bwd_workspace_bytes() bytes,
 *                            256-byte aligned
 *
 * With p = exp(scale q.k - LSE), dP = dO.v and delta = dO.O per row and head:
 * dS = p (dP - delta), dQ = scale sum dS k, dK += scale dS q, dV += p dO over
 * every visible (query, head, key). Stages on `stream`: per-row inputs
 * (delta, an fp16 copy of dO; with D = 64 also dQ, from a query-major
 * kernel); a transposed index listing, per (b, g, block), the queries that
 * selected it; a key-major kernel that loads each block once per chunk of
 * its list and adds its dK / dV partial sums. With D = 128, the entries
 * of each query's own block c and of block c - 1 go to a local-block
 * kernel instead (one CTA per block row of 32 or 64 queries: their dQ rows
 * summed on the tensor cores and stored once, dK / dV of the two blocks
 * summed over the block row), and the key-major kernel also forms dQ =
 * dS K for the other entries and adds it with fp32 reductions; dK / dV are
 * added with fp32 atomics (D = 64) or bulk fp32 reductions (D = 128). dK /
 * dV (and dQ when D = 128) sum in an order set by atomics (equal within
 * rounding from run to run). With D = 128 every key of a block some query
 * selects may enter the dQ of the queries that share its block row or its
 * chunk (with weight 0 where a query does not select or see it), so K
 * must be finite in every selected block, including keys after a query's
 * position. With D = 128 the index transpose runs on a second stream that
 * the call creates and releases, beside the per-row stage and the
 * local-block kernel; `stream` waits for it. Asynchronous, allocates no
 * device memory; errors as nsa_sel_attn_fwd plus NSA_ERR_WORKSPACE.
 * Pointers must be 16-byte aligned (LSE and block_indices 4-byte).
 */
int nsa_sel_attn_bwd(const void* Q, const void* K, const void* V,
                     const int32_t* block_indices, const float* O, const float* LSE,
                     const float* dO, float* dQ, float* dK, float* dV, int64_t B, int64_t M,
                     int64_t N, int64_t H, int64_t G, int64_t D, int64_t T, int block_size,
                     float scale, void* workspace, int64_t workspace_bytes, void* stream);

/*
 * nsa_sel_attn_bwd_ex -- nsa_sel_attn_bwd with a choice of input type.
 *
 *   qkv_dtype  NSA_F16 or NSA_BF16: the type of Q, K and V (else
 *              NSA_ERR_DTYPE before anything is enqueued)
 *
 * With bf16 inputs every tensor-core product takes bf16 operands (the 16-bit
 * copy of dO, P and dS are rounded to bf16) with fp32 accumulation -- the
 * bf16 reading of "FP16 matmuls, FP32 accumulation" that nsa_sel_attn_fwd_ex
 * takes for the forward. O, LSE, dO and the gradients stay fp32. Everything
 * else, the workspace included, is nsa_sel_attn_bwd; nsa_sel_attn_bwd is
 * this call with NSA_F16.
 */
int nsa_sel_attn_bwd_ex(const void* Q, const void* K, const void* V,
                        const int32_t* block_indices, const float* O, const float* LSE,
                        const float* dO, float* dQ, float* dK, float* dV, int64_t B, int64_t M,
                        int64_t N, int64_t H, int64_t G, int64_t D, int64_t T, int block_size,
                        float scale, int qkv_dtype, void* workspace, int64_t workspace_bytes,
                        void* stream);

/*
 * nsa_sel_attn_bwd_noalloc -- nsa_sel_attn_bwd for callers that cannot
 * allocate device memory. The pages have no counterpart to this entry point.
 *
 * Some callers may not allocate at all: a plugin inside a host application
 * that owns every device allocation through its own pool and hands plugins
 * no allocator, or a service that reserves all of its memory at start-up and
 * forbids allocation while it serves. They still pass every input and
 * output; the scratch the backward needs (delta, the per-block query lists
 * and their offsets) comes from a fixed 64 MiB array inside the library,
 * which every GPU that loads the library holds until the process exits.
 *
 * Arguments, layouts and results are those of nsa_sel_attn_bwd without the
 * workspace. A problem whose scratch (nsa_sel_attn_bwd_workspace_bytes)
 * exceeds 64 MiB is rejected with NSA_ERR_SCRATCH before anything is
 * launched; a problem without queries (B == 0 or M == 0) needs no scratch
 * and only zeroes dK and dV. The call allocates and frees nothing and creates
 * no stream: all of its stages run in order on `stream`. Every
 * call looks up the array's device address in the current device's context
 * (cudaGetSymbolAddress: a host-side query, no allocation, no
 * synchronisation), so a context created anew after cudaDeviceReset gets
 * its own array. The first lookup on a device may load the library's
 * device code: make the first call on each device before any stream
 * capture. Every call uses the same array and finds the previous call's
 * contents in it; the parts that must start at zero are cleared on the
 * call's stream. Calls whose work overlaps on the GPU (on different
 * streams, or from different threads on one device) race on the array:
 * serialise them.
 */
int nsa_sel_attn_bwd_noalloc(const void* Q, const void* K, const void* V,
                             const int32_t* block_indices, const float* O, const float* LSE,
                             const float* dO, float* dQ, float* dK, float* dV, int64_t B,
                             int64_t M, int64_t N, int64_t H, int64_t G, int64_t D, int64_t T,
                             int block_size, float scale, void* stream);

/*
 * nsa_topk_blocks -- top-k block selection: block_indices from block scores.
 *
 * The selection-attention issue takes block_indices from a top-k selection
 * kernel ("[wave] NSA: selection attention forward kernel", section
 * "Depends on"); its section "Operation" fixes the output [B,M,G,T] and
 * section "Requirements" one row per GQA group. The pages do not say how
 * blocks are scored, so the scores are the input:
 *
 *   scores         device, fp32,  [B, M, G, ceil(N/block_size)]; the score
 *                  of key block t for query (b, m) and KV group g. Only
 *                  entries of free candidate blocks (below) are read.
 *   block_indices  device, int32, [B, M, G, T] (output)
 *   B, M, N, T     >= 0; G > 0; ceil(N/block_size) <= 4096
 *   block_size     >= 1 (keys per block, as in nsa_sel_attn_fwd)
 *   n_init,        >= 0 with n_init + n_local <= T: the first n_init and the
 *   n_local        last n_local candidate blocks of a row are always chosen
 *   stream         cudaStream_t to launch on
 *
 * Row (b, m, g): the candidates are the blocks t = 0..c holding a key
 * visible to query m, c = floor(min(m, N-1) / block_size) (none if N = 0).
 * With at most T candidates all are chosen. Otherwise the forced blocks are
 * chosen and the remaining T - n_init - n_local slots go to the other
 * candidates with the highest scores; equal scores choose the lower block
 * (-0.0 equals +0.0) and NaN ranks below every number. The row is written
 * in ascending block order and padded with -1, so it is a valid
 * block_indices row for nsa_sel_attn_fwd (distinct, causal).
 *
 * Asynchronous: one kernel on `stream`, no allocation, no synchronisation.
 * Returns NSA_ERR_SHAPE (bad sizes, n_init/n_local out of range, too many
 * blocks), NSA_ERR_BLOCK_SIZE, NSA_ERR_NULL, NSA_ERR_ALIGN (a pointer not
 * 4-byte aligned) before launch; an empty output returns NSA_OK at once.
 * A row copy that does not arrive within 1 s makes nsa_sync_status report
 * NSA_ERR_TIMEOUT; the outputs of that launch are then undefined.
 */
int nsa_topk_blocks(const float* scores, int32_t* block_indices, int64_t B, int64_t M,
                    int64_t N, int64_t G, int64_t T, int block_size, int n_init,
                    int n_local, void* stream);

/*
 * nsa_swa_fwd -- GQA sliding-window (or dense) attention forward, the
 * second workload on the pages ("[Kernel][MI350] Add 8 wave GQA
 * sliding-window attention kernel", sections "Summary" and "What it does").
 *
 *   Q              device, [B, M, H, D],    fp16 or bf16 (dtype)
 *   K, V           device, [B, N, H_kv, D], same type
 *   O              device, [B, M, H, D],    same type (output)
 *   LSE            device, fp32 [B, H, M] (output, natural log), or NULL
 *   H % H_kv == 0  query head h reads KV head h / (H / H_kv)
 *   D              64 or 128
 *   window_left,   query i attends to keys j with i - window_left <= j <=
 *   window_right   i + window_right and 0 <= j < N; a negative value leaves
 *                  that side unbounded: (-1, -1) is dense attention, (-1, 0)
 *                  causal, (L, 0) causal with L keys of history
 *   scale          score multiplier; <= 0 selects 1/sqrt(D)
 *   dtype          NSA_F16 or NSA_BF16
 *
 * Query i is aligned with key i. Both products run on the 5th-generation
 * tensor cores (tcgen05, fp32 accumulation in tensor memory). P is rounded
 * to the input type before the PV product, and O is the fp32 result rounded
 * once. A row with no visible key gets O = 0 and LSE = -inf. The call is
 * asynchronous and allocates nothing. Each CTA holds 512 tensor-memory
 * columns of its SM for its lifetime. Errors returned before launch:
 * NSA_ERR_SHAPE, NSA_ERR_GROUPS, NSA_ERR_HEAD_DIM, NSA_ERR_DTYPE,
 * NSA_ERR_NULL, NSA_ERR_ALIGN (Q, K, V, O not 16-byte aligned, LSE not
 * 4-byte aligned). A timed-out device wait is reported by nsa_sync_status.
 */
int nsa_swa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                int64_t B, int64_t M, int64_t N, int64_t H, int64_t H_kv, int64_t D,
                int64_t window_left, int64_t window_right, float scale, int dtype,
                void* stream);

/*
 * nsa_sync_status -- wait for `stream`, then read and clear the device status
 * word of the current device.
 *
 * Every device-side wait of this library's kernels is bounded (1 s). A warp
 * whose wait gives up records it in a per-device status word, lets its own
 * copies in flight land, and returns without writing its outputs. This call
 * returns NSA_ERR_TIMEOUT if that happened in any launch since the last call,
 * NSA_ERR_LAUNCH if synchronising the stream reports a CUDA error, NSA_OK
 * otherwise. A library built with NSA_DEBUG_BOUNDS also checks, before every
 * K/V tile copy of the selection forward, that the tile starts on a 16-key
 * boundary, at or before the query's last visible key, inside a block of the
 * index range; a failed check is returned here as NSA_ERR_BOUNDS (ahead of a
 * timeout). It synchronises; it allocates nothing.
 */
int nsa_sync_status(void* stream);

/*
 * nsa_selftest_wait_timeout -- test hook for the bounded waits.
 *
 * Launches one warp on `stream` that waits on a barrier nothing will ever
 * complete; after `limit_ns` (1e3 .. 2e9) it gives up and sets the status
 * word, so the next nsa_sync_status() returns NSA_ERR_TIMEOUT. Touches no
 * other memory. Returns NSA_ERR_SHAPE for a limit out of range.
 */
int nsa_selftest_wait_timeout(int64_t limit_ns, void* stream);

/*
 * nsa_probe_l2_gather -- measurement kernel: the gather of
 * nsa_sel_attn_fwd with nothing else, to measure the ceiling that gather
 * meets ("[wave] NSA: selection attention forward kernel", section "MI350
 * considerations": the irregular block gather is the most
 * performance-critical part of the kernel).
 *
 *   K, V            device, IEEE fp16, [N, G, D] (one batch), 16-byte aligned
 *   N               >= block_size; blocks 0 .. floor(N/block_size)-1 are drawn
 *   G, g            KV groups; the group read (0 <= g < G), or -1 for a
 *                   group drawn with every block (all groups interleaved)
 *   D               64 or 128
 *   block_size      32 or 64
 *   ctas            grid size (1 .. 2^31); size it as SMs x CTAs per SM
 *   warps_per_cta   1 .. 32
 *   slots_per_warp  1 .. 16 tiles each warp keeps in flight
 *   loads_per_warp  tiles each warp copies (>= 0)
 *   rows_per_box    key rows per TMA box and per tile: 16 (the forward's), 32
 *                   or 64, at most block_size
 *   seed            block draw seed
 *   cta_record      device int64 [ctas, 3] written with (SM id, start ns,
 *                   end ns) of every CTA (%globaltimer), or NULL
 *
 * Each warp copies loads_per_warp tiles of rows_per_box key rows x D (TMA
 * boxes of rows_per_box x 64, 128-byte swizzle, L2 evict_last: with 16 rows,
 * the forward's copies) into
 * shared memory, alternating K and V and walking the 16-key tiles of
 * randomly drawn blocks, keeping slots_per_warp copies in flight and doing
 * nothing with the data. The bytes moved, nsa_probe_l2_gather_bytes(), over
 * the kernel's time is the gather bandwidth this GPU delivers for that
 * access pattern and in-flight depth. Shared memory per CTA is
 * warps x slots x D/64 x rows_per_box x 128 B (+ 1 KB + barriers), within
 * 227 KB (else NSA_ERR_SHAPE). Asynchronous; allocates nothing. Errors:
 * NSA_ERR_NULL, NSA_ERR_ALIGN, NSA_ERR_HEAD_DIM, NSA_ERR_BLOCK_SIZE,
 * NSA_ERR_SHAPE, NSA_ERR_LAUNCH. A timed-out wait is reported by
 * nsa_sync_status.
 */
int nsa_probe_l2_gather(const void* K, const void* V, int64_t N, int64_t G, int64_t D,
                        int64_t g, int block_size, int64_t ctas, int warps_per_cta,
                        int slots_per_warp, int64_t loads_per_warp, int rows_per_box,
                        uint32_t seed, int64_t* cta_record, void* stream);

/* Bytes nsa_probe_l2_gather moves for these arguments (negative nsa_status
 * for invalid ones). Pure host arithmetic. */
int64_t nsa_probe_l2_gather_bytes(int64_t D, int64_t ctas, int warps_per_cta,
                                  int64_t loads_per_warp, int rows_per_box);

/*
 * nsa_probe_gather_rows -- measurement kernel: exactly the copies
 * nsa_sel_attn_fwd makes for these index rows, and nothing else.
 *
 *   K, V, block_indices, B, M, N, G, D, T, block_size
 *                   as for nsa_sel_attn_fwd (H plays no part: the copies are
 *                   per (b, m, g) row); same checks and errors
 *   ctas            grid size (1 .. 2^31 - 1)
 *   warps_per_cta   1 .. 32
 *   slots_per_warp  1 .. 16 copies each warp keeps in flight
 *   extra_smem_bytes  >= 0: unused shared memory added to each CTA, to
 *                   measure how the gather rate depends on the shared
 *                   memory a kernel reserves (total within 227 KB)
 *
 * Every warp takes the (b, g, m) rows w, w + W, w + 2W, ... (W warps in the
 * grid, m fastest) and walks each row as the forward does -- padding,
 * out-of-range ids and blocks after the query skipped, the 16-key tiles of
 * each selected block that start at or before the query -- copying the K
 * tile and then the V tile of every 16-key tile into shared memory (TMA
 * boxes of 16 x 64, 128-byte swizzle, L2 evict_last). It moves the bytes of
 * every whole 16-key tile the forward gathers, back to back across rows,
 * so the forward's gathered bytes over this kernel's time bound the
 * forward's gather rate from above for these rows. Shared memory and
 * asynchrony as nsa_probe_l2_gather; allocates nothing.
 */
int nsa_probe_gather_rows(const void* K, const void* V, const int32_t* block_indices, int64_t B,
                          int64_t M, int64_t N, int64_t G, int64_t D, int64_t T, int block_size,
                          int64_t ctas, int warps_per_cta, int slots_per_warp,
                          int64_t extra_smem_bytes, void* stream);

/*
 * nsa_probe_reduce_rows -- measurement kernel: the backward's dQ reductions
 * alone, to measure the rate they can reach on this GPU.
 *
 *   buf             device fp32, at least rows * stride floats, 16-byte
 *                   aligned; its contents are left unchanged (zeros are added)
 *   rows, stride    rows of 1024 floats (4 KB: 8 head rows of 128 dims, one
 *                   query and KV group of dQ), `stride` floats apart
 *                   (>= 1024, a multiple of 4); dQ of one KV group is
 *                   rows = B*M, stride = H*128
 *   ctas, warps_per_cta  grid (warps_per_cta 1 .. 32)
 *   iters_per_warp  rows each warp adds into
 *
 * Each warp adds one 4 KB row at a time into a row drawn at random, with
 * 16-byte fp32 reductions (red.global.add.v4.f32), as the key-major backward
 * kernel adds its dQ partial sums. Bytes reduced = ctas x warps x iters x
 * 4096. Asynchronous; allocates nothing. Errors: NSA_ERR_NULL,
 * NSA_ERR_ALIGN, NSA_ERR_SHAPE, NSA_ERR_LAUNCH.
 */
int nsa_probe_reduce_rows(float* buf, int64_t rows, int64_t stride, int64_t ctas,
                          int warps_per_cta, int64_t iters_per_warp, uint32_t seed,
                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NSA_SEL_ATTN_H */
