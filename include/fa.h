/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * What is computed (FlashAttention: Fast and Memory-Efficient Exact Attention
 * with IO-Awareness, hackmd summary, section "Standard Attention
 * Implementation"): for every batch b and head h, with Q, K, V in R^{N x d},
 *     S = scale * Q K^T,   P = softmax(S + mask) row by row,   O = P V.
 * The library never forms S or P in memory: the forward walks K/V tile by
 * tile with a running row max and row sum ("Tiling"), and the backward
 * rebuilds S and P from Q, K, V and the stored statistic ("Recomputation").
 * The stored statistic is the natural-log logsumexp lse_i = m_i + ln l_i.
 *
 * Conventions shared by every call
 *   Tensors      bf16, contiguous [B, H, N, d] (each (b, h) slice is the
 *                pages' N x d matrix); lse and D are fp32 [B, H, N].
 *   Pointers     device pointers.  q, k, v, o, dO, dq, dk, dv and the
 *                workspace must be 16-byte aligned (TMA / vector access);
 *                lse 4-byte aligned.  Misalignment -> FA_ERR_MISALIGNED.
 *   Sizes        B, H, N >= 1; d in {64, 128} (else FA_ERR_UNSUPPORTED);
 *                B*H*N*d < 2^31.  scale finite and > 0.
 *   Masks        causal != 0 keeps key j for query i iff j <= i.  Block
 *                masks are uint8 [mask_heads, nT, nT] in device memory,
 *                nT = ceil(N / 128); a nonzero byte keeps that 128 x 128
 *                tile; mask_heads is 1 (shared by all heads) or H.
 *                A query row with no kept key gets O = 0, lse = -inf and
 *                zero gradients.
 *   Ownership    the caller allocates every buffer, including workspaces;
 *                the library allocates no device memory and keeps no state
 *                between calls except one status word per device.
 *   Streams      work is enqueued on `stream` and the call returns without
 *                waiting.  The return value reports argument and launch
 *                errors; no kernel is launched when it is not FA_OK.
 *                A device-side wait that exceeds its time limit records
 *                FA_ERR_TIMEOUT, read with fa_get_device_status().
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad scale   */
  FA_ERR_UNSUPPORTED = 2, /* head dim not in {64, 128}, sizes too large    */
  FA_ERR_MISALIGNED = 3,  /* pointer alignment below the stated minimum    */
  FA_ERR_WORKSPACE = 4,   /* workspace smaller than the *_workspace_size   */
  FA_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed          */
  FA_ERR_TIMEOUT = 6      /* a device-side wait ran past its limit         */
} fa_status;

/* Short English description of a status code (static storage). */
const char* fa_status_string(fa_status s);

/*
 * Forward pass ("Tiling"; "Kernel Fusion": one kernel does
 * matmul -> mask -> softmax -> matmul).
 *   in : q, k, v   bf16 [B, H, N, d]
 *   out: o         bf16 [B, H, N, d]   O = softmax(scale*QK^T + mask) V
 *        lse       fp32 [B, H, N]      natural-log logsumexp of each row
 * The extra memory is O(N) per head ("Theorem 1"): only o and lse.
 */
fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int N, int d, float scale, int causal, cudaStream_t stream);

/* Bytes of workspace fa_backward needs: D (fp32 [B,H,N]) and the fp32 dQ
 * accumulator ([B,H,N,d]), each 256-byte aligned; for d = 128 with more
 * than 64 key tiles (B*H*ceil(N/128)) also min(tiles/2, 96) slots of
 * 128 KiB plus 8 bytes each (at most 12 MiB): fp32 dK, dV partial sums
 * of key tiles whose query-tile walk the last round of the persistent
 * backward splits between two SMs; then one int (the block-sparse
 * backward's next-unit counter).  O(B*H*N*d), never O(N^2). */
size_t fa_backward_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass by recomputation ("Recomputation": the forward kept only O
 * and the softmax statistics; S and P are rebuilt block by block).
 *   in : q, k, v, o, dO   bf16 [B, H, N, d];  lse fp32 [B, H, N] from
 *        fa_forward with the same q, k, v, scale and causal
 *   out: dq, dk, dv       bf16 [B, H, N, d], gradients of sum(O o dO)
 *   workspace / workspace_bytes: caller-owned device scratch of at least
 *        fa_backward_workspace_size(B, H, N, d) bytes; its contents on
 *        entry do not matter.
 * Enqueues three kernels: fa_backward_preprocess, fa_backward_main,
 * fa_backward_dq_convert (also exported separately, below).  dq is summed
 * with fp32 atomics, so it is not bit-reproducible from run to run.
 */
fa_status fa_backward(const void* q, const void* k, const void* v, const void* o, const void* dO,
                      const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                      float scale, int causal, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/* Backward step 1: D_i = <dO_i, O_i> (fp32) into the workspace and zero the
 * workspace's dQ accumulator and its counters. */
fa_status fa_backward_preprocess(const void* o, const void* dO, int B, int H, int N, int d,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Backward step 2: the fused recompute kernel.  Reads D from the workspace,
 * writes dk and dv, and adds unscaled dS K into the workspace's dQ
 * accumulator.  Run it once after each fa_backward_preprocess of the same
 * problem on the same workspace: the preprocess also clears the counters
 * with which split key tiles of the last round hand over their partial
 * dK, dV sums (and the block-sparse backward hands out its units), and a
 * second run on the same workspace would find them used. */
fa_status fa_backward_main(const void* q, const void* k, const void* v, const void* dO,
                           const float* lse, void* dk, void* dv, int B, int H, int N, int d,
                           float scale, int causal, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* Backward step 3: dq = bf16(scale * dQ accumulator). */
fa_status fa_backward_dq_convert(void* dq, int B, int H, int N, int d, float scale,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_backward without a workspace argument, for callers that cannot
 * allocate device memory: a host framework that hands a plugin no workspace,
 * or code that must not call cudaMalloc once running (it can synchronise the
 * device and can fail under memory pressure mid-job).  The paper has no
 * counterpart; this is a packaging variant of fa_backward, same arguments
 * and results minus the workspace.
 *   Scratch: one file-scope device array of 32 MiB (2^25 bytes) per GPU,
 *            held from library load until process exit.  Problems whose
 *            fa_backward_workspace_size(B, H, N, d) exceeds 2^25 bytes return
 *            FA_ERR_WORKSPACE with nothing launched (d = 64: about 129k rows
 *            B*H*N; d = 128: about 40k rows).
 *   Sharing: every call on a device uses the same array, which keeps the last
 *            call's contents; each call clears what must start at zero (the
 *            dQ accumulator) itself.  Calls whose kernels overlap on the GPU
 *            race on the array: order them on one stream.
 *   Set-up:  the first call on each device looks up the array's device
 *            address (cudaGetSymbolAddress, that device current) and caches
 *            it; make that first call before any stream capture.
 * Allocates nothing: no cudaMalloc / cudaFree, no allocating library call.
 */
fa_status fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                              int H, int N, int d, float scale, int causal, cudaStream_t stream);

/*
 * Grouped key/value heads (multi-head-attention variants, hackmd summary,
 * "Future Directions": multi-query / grouped-query attention).  H query
 * heads share Hkv key/value heads, H % Hkv == 0 (Hkv = 1: one key/value
 * head for all); query head h reads key/value head h / (H / Hkv).
 *   q, o, dO, dq  bf16 [B, H, N, d];   lse fp32 [B, H, N]
 *   k, v, dk, dv  bf16 [B, Hkv, N, d]; dk, dv sum over the H / Hkv query
 *                 heads that read each key/value head
 * Workspace as fa_backward_workspace_size(B, H, N, d).  Other rules as
 * fa_forward / fa_backward; Hkv outside [1, H] or not dividing H gives
 * FA_ERR_INVALID_ARG.
 */
fa_status fa_forward_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int Hkv, int N, int d, float scale, int causal,
                         cudaStream_t stream);
fa_status fa_backward_gqa(const void* q, const void* k, const void* v, const void* o,
                          const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                          int H, int Hkv, int N, int d, float scale, int causal, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);

/*
 * Packed variable-length batch (hackmd summary, section 4.4: attention over
 * a batch of unequal lengths, which padding would waste work on).  The B
 * sequences are packed back to back along the row axis; sequence b holds rows
 * cu_seqlens[b] .. cu_seqlens[b+1]-1 and attends only within itself (causal:
 * row i of a sequence sees that sequence's rows 0..i).
 *   q, o, dO, dq  bf16 [H, total, d];   lse fp32 [H, total]
 *   k, v, dk, dv  bf16 [Hkv, total, d]  (Hkv = H: ordinary multi-head;
 *                 otherwise grouped heads as fa_forward_gqa)
 *   cu_seqlens    int32 [B+1], DEVICE memory, cu_seqlens[0] = 0,
 *                 nondecreasing, cu_seqlens[B] = total; empty sequences
 *                 (equal neighbours) are allowed and produce nothing
 *   max_seqlen    >= every length (it sizes the grid); 1 <= max_seqlen <= total
 * The array is read only on the device.  The kernels clamp its entries to
 * [0, total] and lengths to max_seqlen: an array that breaks the rules gives
 * unspecified values in the outputs but no access outside the tensors.
 * total = 0 returns FA_OK with nothing launched.  Workspace (backward):
 * fa_backward_workspace_size(1, H, total, d).  p_drop, seed, offset:
 * dropout on P as fa_forward_dropout, sequence b taking the place of batch
 * b (p_drop = 0: none).  Other rules as fa_forward / fa_backward;
 * H * total * d must stay below 2^31.
 */
fa_status fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens, int B, int max_seqlen, int total, int H,
                            int Hkv, int d, float scale, int causal, float p_drop,
                            unsigned long long seed, unsigned offset, cudaStream_t stream);
fa_status fa_backward_varlen(const void* q, const void* k, const void* v, const void* o,
                             const void* dO, const float* lse, void* dq, void* dk, void* dv,
                             const int* cu_seqlens, int B, int max_seqlen, int total, int H,
                             int Hkv, int d, float scale, int causal, float p_drop,
                             unsigned long long seed, unsigned offset, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/*
 * Deterministic backward: dQ, dK, dV identical bit for bit from run to run
 * (fa_backward sums dQ with unordered fp32 atomic adds, so its dQ may differ
 * in the last bits between runs).  Two passes after the D preprocess:
 *   key-tile pass   per key tile: S, P, dP, dS, dV += P^T dO, dK += dS^T Q
 *                   (fixed order inside one CTA), no dQ product
 *   query-tile pass per query tile: S, P, dP, dS recomputed, dQ += dS K over
 *                   the key tiles in ascending order; bf16(scale * dQ)
 *                   written directly
 * It recomputes S and dP once more (7 tile products per (query, key) tile
 * pair instead of 5), the price of the fixed order ("Recomputation" leaves
 * the summation order open).  Same arguments and results as fa_backward;
 * the workspace needs only align256(4 * B*H*N) bytes (D); any size from
 * fa_backward_workspace_size works.
 */
fa_status fa_backward_deterministic(const void* q, const void* k, const void* v, const void* o,
                                    const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                    int B, int H, int N, int d, float scale, int causal,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Dropout on the attention weights, fused into both passes (hackmd summary,
 * "Kernel Fusion": masking and dropout are applied inside the kernel; the
 * section 4.4 benchmark runs with dropout).  Inverted dropout of P:
 *   O = (z o P) V / (1 - p'),   lse = the undropped row's logsumexp
 * The keep indicator z_ij of query row i, key j of (batch b, head h) is
 *   byte (j mod 16) of Philox4x32-10(counter = (j/16, i, b*H + h, offset),
 *                                    key = (seed mod 2^32, seed / 2^32))
 *   (output word (j/4) mod 4, byte j mod 4, little-endian)  >=  t,
 *   t = rint(256 * p_drop),  p' = t / 256
 * (Philox: Salmon, Moraes, Dror, Shaw, SC 2011).  Decisions are integer
 * and reproducible bit for bit; the backward regenerates them from the same
 * (seed, offset), which must match the forward's.  p_drop is rounded to a
 * multiple of 1/256; p_drop outside [0, 1), or rounding to 1, gives
 * FA_ERR_INVALID_ARG.  p_drop = 0 computes the undropped result.  Layouts,
 * workspace and other rules as fa_forward / fa_backward.
 */
fa_status fa_forward_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int N, int d, float scale, int causal, float p_drop,
                             unsigned long long seed, unsigned offset, cudaStream_t stream);
fa_status fa_backward_dropout(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal, float p_drop,
                              unsigned long long seed, unsigned offset, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* Bytes of workspace the block-sparse calls need: the CSR and CSC tile
 * lists of the mask (4 * mask_heads * (2*(nT+1) + 2*nT*nT + nT + 1) bytes,
 * rounded up to 256) followed by the fa_backward workspace.  The forward uses
 * only the list part. */
size_t fa_blocksparse_workspace_size(int B, int H, int N, int d, int mask_heads);

/*
 * Block-sparse tile lists ("Block-sparse FlashAttention": only the nonzero
 * blocks of the block mask are read and computed).  Writes into the
 * workspace, at offset 0:
 *   row_ptr int32 [mask_heads, nT+1]   head-local CSR offsets
 *   col_ptr int32 [mask_heads, nT+1]   head-local CSC offsets
 *   col_idx int32 [mask_heads, nT*nT]  ascending key tiles of each query tile
 *   row_idx int32 [mask_heads, nT*nT]  ascending query tiles of each key tile
 *   order   int32 [mask_heads, nT]     key tiles by descending row_idx list
 *                                      length, ties by index
 *   nlong   int32 [mask_heads]         how many key tiles have more than
 *                                      twice the mean list length
 * The backward takes the nlong longest key tiles of every head first, then
 * each head's other key tiles in that order, head by head.
 * Integer work, bit-exact.  nT must be <= 8192.
 */
fa_status fa_blocksparse_build_lists(const uint8_t* block_mask, int mask_heads, int N,
                                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Block-sparse forward: builds the lists into the workspace, then runs the
 * forward over kept tiles only; skipped tiles contribute exactly zero.
 * causal may be combined with the mask (intersection). */
fa_status fa_blocksparse_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int N, int d, float scale, int causal,
                                 const uint8_t* block_mask, int mask_heads, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/* Block-sparse backward: lists, preprocess, recompute kernel over kept
 * tiles, dq conversion.  workspace as fa_blocksparse_workspace_size. */
fa_status fa_blocksparse_backward(const void* q, const void* k, const void* v, const void* o,
                                  const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                  int B, int H, int N, int d, float scale, int causal,
                                  const uint8_t* block_mask, int mask_heads, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/* Synchronises `stream`, then reads and clears the status word of the
 * current device.  FA_OK, FA_ERR_TIMEOUT (a device wait gave up; outputs of
 * the calls since the last check are undefined) or FA_ERR_CUDA. */
fa_status fa_get_device_status(cudaStream_t stream);

/* Time limit of every device-side wait, in nanoseconds (default 2e9, also
 * settable with the FA_WAIT_LIMIT_NS environment variable).  0 restores the
 * default.  Applies to calls made after it returns. */
fa_status fa_set_wait_limit_ns(unsigned long long ns);

/* ---------------------------------------------------------------- tests */

/* Launches one CTA that waits on an mbarrier nothing completes; the bounded
 * wait gives up after limit_ns and records FA_ERR_TIMEOUT in the status
 * word.  Exercises the timeout path without faulting or hanging. */
fa_status fa_debug_wait_timeout(unsigned long long limit_ns, cudaStream_t stream);

/*
 * Exports the tile schedules the kernels walk (integer, bit-exact):
 *   fwd_counts int32 [heads, nT], fwd_lists int32 [heads, nT, nT]:
 *       for each query tile, the key tiles the forward visits, in order;
 *   bwd_counts int32 [heads, nT], bwd_lists int32 [heads, nT, nT]:
 *       for each key tile, the query tiles the backward visits, in order.
 * heads = mask_heads with a block mask (the lists are built into the
 * workspace first), else 1.  All outputs are device memory.
 */
fa_status fa_debug_schedule(int N, int causal, const uint8_t* block_mask, int mask_heads,
                            void* workspace, size_t workspace_bytes, int* fwd_counts,
                            int* bwd_counts, int* fwd_lists, int* bwd_lists, cudaStream_t stream);

/*
 * fa_forward with its tile configuration chosen by the caller (the block-size
 * experiment of the hackmd summary, "IO Complexity Analysis": changing the
 * block size B_c changes the IO, and the runtime with it, until compute
 * bounds it).
 *   rows_per_cta  128 (one query tile per CTA) or 256 (two; fa_forward's
 *                 choice)
 *   key_tile      keys per key tile, B_c: 64, 128 (fa_forward's) or 256;
 *                 256 needs rows_per_cta = 128 (tensor memory holds S and O
 *                 of one query tile then)
 *   kv_stages     K/V shared-memory ring depth, one key or value tile per
 *                 slot:
 *                   d = 128: key_tile 128: 2..5 (5 is fa_forward's);
 *                            64: 4 or 8; 256: 2
 *                   d = 64:  key_tile 128: 2, 4 or 8 (8 is fa_forward's);
 *                            64: 8 or 16; 256: 2 or 4
 * Dense or causal, no grouped K/V.  Other arguments and results as
 * fa_forward; unsupported choices give FA_ERR_UNSUPPORTED.
 */
fa_status fa_debug_forward_config(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int H, int N, int d, float scale, int causal,
                                  int rows_per_cta, int key_tile, int kv_stages,
                                  cudaStream_t stream);

/*
 * One-tile tcgen05 check of the operand layouts the kernels use.
 *   mode 0: c[128x128] = a b^T, a and b bf16 [128 x 128]
 *   mode 1: c[128xn]   = a b,   a bf16 [128 x 128], b bf16 [128 x n]
 *   mode 2: c[128xn]   = a^T b, a bf16 [128 x 128], b bf16 [128 x n]
 *   mode 3: c[128xn]   = a b,   as mode 1 with a held in tensor memory
 * n in {64, 128}; c fp32 row-major; all device pointers, 16-byte aligned.
 */
fa_status fa_debug_mma_probe(const void* a, const void* b, float* c, int mode, int n,
                             cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
