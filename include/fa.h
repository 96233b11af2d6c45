/*
 * fa.h -- C ABI of libfa.so: exact, IO-aware tiled attention forward on GB300
 * (sm_103a), written for tcgen05 tensor cores, tensor memory and TMA.
 *
 * The operation ("Flash Attention 3 principles (guijiagi)", section 1.2 for
 * standard attention, section 2.2 for the online-softmax recurrence the kernel
 * uses, section 5.2 for the varlen call with `causal` and `softmax_scale`):
 *
 *   for every sequence b, head h and query row i of that sequence,
 *     s_ij  = scale * sum_d Q[i,h,d] K[j,h,d]        for visible keys j
 *     O[i,h,:] = sum_j exp(s_ij - m_i) V[j,h,:] / sum_j exp(s_ij - m_i)
 *     LSE[i,h] = m_i + ln sum_j exp(s_ij - m_i)        (natural log)
 *   with m_i the row max; visible keys are j < Lk, and with `causal` only
 *   j <= i + Lk - Lq (mask aligned to the bottom-right corner; for Lq = Lk
 *   this is j <= i). A row with no visible key gets O = 0 and LSE = -inf.
 *
 * Conventions shared by every entry point:
 *   - All tensor arguments are DEVICE pointers on the current CUDA device.
 *     The caller owns every buffer; the library keeps none of them.
 *   - Q/K/V/O layout: contiguous [tokens, H, D] (row-major, D fastest), i.e.
 *     (B, S, H, D) for fixed length (tokens = B*S, batch-major) or packed
 *     sequences for varlen. Base pointers must be 16-byte aligned.
 *   - D (head dimension) is 64, 128 or 256.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *     call is asynchronous on it; argument errors are reported synchronously
 *     by the return value, errors found on the device by
 *     fa_get_device_status().
 *   - Return value: FA_OK (0) or a negative FA_ERR_* code (fa_strerror()).
 *   - The library allocates no device memory: scratch that a call needs is
 *     passed in. Its device state, present on every device that loads the
 *     library until the process exits, is static __device__ arrays: one
 *     status word, 64 pairs of tile-scheduler counters, and the fixed 64 MiB
 *     scratch array that only fa_fwd_splitkv_noalloc (below) uses.
 *   - The first call on a device sets up the library's host-side state for it:
 *     it looks up the device addresses of those arrays and creates one CUDA
 *     event per scheduler slot (64). Make that first call before any stream
 *     capture. The addresses are kept for the life of the process; they do
 *     not survive cudaDeviceReset, so do not call the library on a device
 *     after resetting it.
 *   - Concurrency: every kernel that schedules work tiles dynamically holds
 *     one of the device's 64 scheduler slots until it finishes (an event
 *     recorded after its launch says when). When all 64 are held by
 *     launches in flight, over all streams and host threads, a new launch
 *     reuses the slot handed out longest ago, and its stream first waits on
 *     the GPU (cudaStreamWaitEvent) until that slot's previous launch has
 *     finished: the call does not block the host, but with more than 64
 *     launches in flight a launch may wait for one on another stream. A
 *     launch captured into a CUDA graph is not tracked: it takes the next
 *     slot in turn at capture time and keeps it for every replay, so
 *     replays must not overlap one another or other launches of the library
 *     on that device. FA_ERR_BUSY: the stream wait could not be issued;
 *     nothing is launched.
 *   - The status word is per device, not per stream or call:
 *     fa_get_device_status() reports (and clears) what any kernel of the
 *     library on that device recorded since the last read.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_OK 0
#define FA_ERR_INVALID_ARG -1     /* a size, pointer or flag is out of range   */
#define FA_ERR_UNSUPPORTED -2     /* valid request this build does not support */
#define FA_ERR_ALIGNMENT -3       /* a pointer is not 16-byte aligned          */
#define FA_ERR_CUDA -4            /* a CUDA runtime / driver call failed       */
#define FA_ERR_DEVICE_TIMEOUT -5  /* a kernel wait gave up (see status)        */
#define FA_ERR_DEVICE_SEQLENS -6  /* a cu_seqlens entry broke its bounds       */
#define FA_ERR_NO_DEVICE -7       /* no sm_100-family device is current        */
#define FA_ERR_SCRATCH_LIMIT -8   /* needs more than the built-in scratch      */
#define FA_ERR_BUSY -9            /* no scheduler slot could be given          */

typedef enum { FA_FP16 = 0, FA_BF16 = 1, FA_FP8_E4M3 = 2 } fa_dtype;

/*
 * fa_fwd -- attention forward for 16-bit inputs (FA_FP16 or FA_BF16).
 *
 *   q            [Tq, H, D] 16-bit, Tq = B*Sq (fixed) or total_q (varlen)
 *   k, v         [Tk, H, D] same type, Tk = B*Sk or total_k
 *   o            [Tq, H, D] output, same type as q (written)
 *   lse          fp32 output: [B, H, Sq] (fixed) or [H, total_q] (varlen)
 *   B            number of sequences (fixed: batch size)
 *   H, D         heads, head dimension
 *   Sq, Sk       fixed: query / key length of every sequence;
 *                varlen: upper bounds of the lengths (max_seqlen_q / _k)
 *   scale        softmax scale, finite and >= 0 (1/sqrt(D) in the pages)
 *   causal       0 or 1
 *   cu_seqlens_q, cu_seqlens_k
 *                NULL for fixed length; for varlen both are device int32
 *                arrays of B+1 nondecreasing prefix sums starting at 0
 *   total_q, total_k
 *                varlen only: rows of q/o and of k/v (cu_seqlens[B] may not
 *                exceed them); ignored for fixed length
 *   dtype        FA_FP16 or FA_BF16 (FA_FP8_E4M3 -> FA_ERR_UNSUPPORTED; the
 *                8-bit path is fa_fp8_prep + fa_fwd_fp8 below)
 *
 * A varlen sequence whose lengths break the bounds is skipped on the device
 * and reported as FA_ERR_DEVICE_SEQLENS by fa_get_device_status(). A query
 * row that sees no key (a sequence with no keys, or causal rows before the
 * first visible key) gets O = 0 and LSE = -inf. With no key rows at all
 * (Tk = 0), k and v are not read and may be NULL. With no query rows
 * (B = 0, Sq = 0 or Tq = 0) the call does nothing and returns FA_OK.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int Sq, int Sk, int D, float scale, int causal,
           const int* cu_seqlens_q, const int* cu_seqlens_k, int total_q, int total_k,
           int dtype, void* stream);

/*
 * fa_fwd_splitkv -- the same forward with the keys of every (sequence, head)
 * cut into ranges that run as separate work tiles, then merged: each range r
 * gives a self-normalised partial O_r and LSE_r, and the rows over all keys
 * are LSE = ln sum_r exp(LSE_r), O = sum_r exp(LSE_r - LSE) O_r (the partial
 * softmax of FlashDecoding, in the lineage of the "FlashAttention-3
 * (lukebest wiki)" page). It fills the GPU when B * H * ceil(Sq/256) work
 * tiles alone would not (short Sq, long Sk).
 *
 *   arguments as fa_fwd, fixed length only (no cu_seqlens)
 *   num_splits   key ranges; <= 0 picks the count with the least estimated
 *                time: whole waves of work tiles over the SMs, the key blocks
 *                of a tile plus a per-tile overhead, and the merge of the
 *                partial results (so a call whose tiles already fill the GPU
 *                keeps one range). It is capped at 256 and at ceil(Sk/128),
 *                and trimmed so that no range is empty.
 *   workspace    device scratch of at least
 *                fa_fwd_splitkv_workspace_size(B, H, Sq, Sk, D, num_splits)
 *                bytes, 256-byte aligned, owned by the caller; its contents
 *                on entry do not matter and are overwritten (partial O in
 *                fp32, then partial LSE). Calls that share a workspace and
 *                overlap on the GPU race.
 *
 * Returns FA_ERR_INVALID_ARG if the workspace is missing or too small.
 */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int Sq, int Sk, int D, int num_splits);
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int Sq, int Sk, int D, float scale, int causal,
                   int num_splits, void* workspace, size_t workspace_bytes, int dtype,
                   void* stream);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv for callers that cannot allocate
 * device memory (no cudaMalloc where they run, or an allocator that must not
 * grow). It takes no workspace: the scratch is a fixed 64 MiB array inside
 * the library, present on every device that loads the library until the
 * process exits. The pages have no counterpart of this entry point.
 *
 *   arguments as fa_fwd_splitkv, without workspace and workspace_bytes
 *
 * Returns FA_ERR_SCRATCH_LIMIT, before touching any pointer, when
 * fa_fwd_splitkv_workspace_size(B, H, Sq, Sk, D, num_splits) exceeds 64 MiB
 * (ask for fewer key ranges, or use fa_fwd_splitkv). The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) and, if
 * no other entry point has run on the device yet, sets up the library's
 * per-device state (see the conventions above); make that first call before
 * any stream capture. All calls share the one array:
 * calls that overlap on the GPU (other streams, other threads) race and give
 * wrong results. Nothing in it needs clearing between calls: every byte a
 * call reads, the same call has written. Allocates nothing.
 */
int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int Sq, int Sk, int D, float scale, int causal,
                           int num_splits, int dtype, void* stream);

/*
 * fa_fwd_paged -- fa_fwd with K and V read from a paged cache
 * ("Flash Attention 3 principles (guijiagi)" section 5.3: PagedAttention
 * keeps a sequence's keys in fixed-size pages named by a block table). That
 * section gathers a sequence's pages into a contiguous buffer before
 * attention; here the kernel's TMA loads read each page in place, so there
 * is no gather pass and no extra copy.
 *
 *   q            [B*Sq, H, D] (fixed query length Sq per sequence), or
 *                packed [total_q, H, D] when cu_seqlens_q is given
 *   k_cache, v_cache  [num_pages, page_size, H, D], same 16-bit type as q
 *   block_table  device int32 [B, max_pages]: page of each page_size-key
 *                block of each sequence
 *   seqlens_k    device int32 [B]: keys of each sequence (<= max_pages *
 *                page_size); key j of sequence b is row j % page_size of
 *                page block_table[b][j / page_size]
 *   o, lse       as fa_fwd: [B*Sq, H, D] and [B, H, Sq], or with packed
 *                queries [total_q, H, D] and [H, total_q]
 *   cu_seqlens_q device int32 [B + 1] query prefix sums (Sq then bounds every
 *                query length), or NULL for fixed-length queries; total_q =
 *                rows of q. Packed queries take num_splits = 1
 *                (FA_ERR_UNSUPPORTED otherwise).
 *   page_size    16, 32, 64 or a multiple of 128
 *   num_splits   key ranges as fa_fwd_splitkv: 1 = none (workspace unused),
 *                0 = automatic, > 1 = that many; the workspace is
 *                fa_fwd_splitkv_workspace_size(B, H, Sq, max_pages *
 *                page_size, D, num_splits) bytes when more than one range
 *                is used (NULL allowed otherwise)
 *   causal       bottom-right aligned per sequence (a sequence's queries
 *                are the last positions of its seqlens_k[b] keys)
 *
 * Only the table entries of a sequence's first ceil(seqlens_k[b] /
 * page_size) blocks are read. Every row of those pages must hold finite
 * values, the rows past the sequence's length in its last page included:
 * their scores are masked, but their V rows still meet a zero weight in the
 * tensor-core product. An entry outside [0, num_pages) or a bad length is
 * not dereferenced (its keys read as zeros) and is reported as
 * FA_ERR_DEVICE_SEQLENS by fa_get_device_status; that sequence's outputs are
 * then undefined.
 */
int fa_fwd_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                 const int* seqlens_k, void* o, float* lse, int B, int H, int Sq, int D,
                 int num_pages, int page_size, int max_pages, float scale, int causal,
                 const int* cu_seqlens_q, int total_q,
                 int num_splits, void* workspace, size_t workspace_bytes, int dtype, void* stream);

/*
 * fa_fp8_prep -- FP8 preparation of the inputs ("FlashAttention-3 (lukebest
 * wiki)", technique 3: block quantisation and incoherent processing).
 *
 *   q, k, v      16-bit inputs, [B*Sq, H, D] and [B*Sk, H, D] (in_dtype
 *                FA_FP16 or FA_BF16), fixed length
 *   q8, k8, v8   e4m3 outputs, same shapes, one byte per element (written)
 *   q_scale      fp32 [B, H, ceil(Sq/128)] (written); k_scale, v_scale
 *                fp32 [B, H, ceil(Sk/128)] (written)
 *   sigma        device int8 [D] of +-1, or NULL for no rotation
 *   D            64, 128 or 256
 *
 * Q' = Q M and K' = K M with M = diag(sigma) H_D / sqrt(D) (H_D the
 * Sylvester Hadamard matrix in natural order; M is orthogonal so
 * Q'K'^T = QK^T); V is not rotated. For every 128-row block of every
 * (sequence, head) of Q', K' and V: scale = amax / 448 (1.0 for an all-zero
 * block) and code = e4m3(x / scale), round to nearest even, saturating at
 * +-448 (the "fn" encoding, no infinities). Sq = 0 or Sk = 0 skips those
 * tensors (their pointers may then be NULL).
 */
int fa_fp8_prep(const void* q, const void* k, const void* v, int in_dtype,
                void* q8, void* k8, void* v8, float* q_scale, float* k_scale, float* v_scale,
                const signed char* sigma, int B, int H, int Sq, int Sk, int D, void* stream);

/*
 * fa_fwd_fp8 -- attention forward on the output of fa_fp8_prep: the same
 * operation as fa_fwd on the dequantised values (code * block scale), with
 * the block scales folded into the softmax constant and into P, and P
 * rounded to e4m3 before it multiplies V.
 *
 *   q8, k8, v8 and the three scale arrays as written by fa_fp8_prep
 *   o            bf16 [B*Sq, H, D] (written); lse fp32 [B, H, Sq] (written)
 *   D            64, 128 or 256 (at D = 64 a 64-byte row of codes is one
 *                TMA box in the 64-byte swizzle)
 *   scale, causal as for fa_fwd. Fixed length (varlen: fa_fwd_fp8_varlen).
 *   Rows that see no key get O = 0 and LSE = -inf; with Sk = 0, k8, v8 and
 *   their scales are not read and may be NULL.
 */
int fa_fwd_fp8(const void* q8, const void* k8, const void* v8,
               const float* q_scale, const float* k_scale, const float* v_scale,
               void* o, float* lse, int B, int H, int Sq, int Sk, int D,
               float scale, int causal, void* stream);

/*
 * fa_varlen_blocks -- block offsets of the variable-length e4m3 layout.
 *
 *   cu_seqlens   device int32 [B + 1], token prefix sums (as for fa_fwd)
 *   cu_blocks    device int32 [B + 1] (written): cu_blocks[0] = 0,
 *                cu_blocks[b + 1] = cu_blocks[b] + ceil(L_b / 128),
 *                L_b = cu_seqlens[b + 1] - cu_seqlens[b] (a negative L_b
 *                counts as 0 and is reported later by the kernels that use it)
 *
 * One small kernel on `stream`; nothing is read on the host. The varlen
 * scales of a tensor are fp32 [n_blocks, H]: row cu_blocks[b] + j holds the
 * scales of block j of sequence b for every head. cu_blocks[B] never exceeds
 * floor(total / 128) + B, the number of rows to allocate when the host does
 * not know the lengths.
 */
int fa_varlen_blocks(const int* cu_seqlens, int B, int* cu_blocks, void* stream);

/*
 * fa_fp8_prep_varlen -- fa_fp8_prep over packed variable-length sequences
 * ("FlashAttention-3 (lukebest wiki)", technique 3, applied per sequence).
 *
 *   q, k, v      16-bit [total_q, H, D] and [total_k, H, D]
 *   q8, k8, v8   e4m3 outputs of the same shapes (written)
 *   cu_seqlens_q/k  device int32 [B + 1] token prefix sums
 *   cu_blocks_q/k   device int32 [B + 1] from fa_varlen_blocks on them
 *   q_scale      fp32 [cu_blocks_q[B], H] (written); k_scale, v_scale
 *                fp32 [cu_blocks_k[B], H] (written)
 *   max_seqlen_q/k  bounds on the lengths; 0 skips that side (Q, or K and
 *                V), whose pointers may then be NULL -- K and V of a cache
 *                are prepared once and reused with every new Q
 *
 * Blocks are the 128-row blocks of each sequence, counted from its first
 * token; a sequence's last block may be short. A sequence whose entries break
 * the bounds (negative or decreasing offsets, beyond total, longer than
 * max_seqlen, or cu_blocks not matching the lengths) is skipped and reported
 * as FA_ERR_DEVICE_SEQLENS by fa_get_device_status.
 */
int fa_fp8_prep_varlen(const void* q, const void* k, const void* v, int in_dtype,
                       void* q8, void* k8, void* v8, float* q_scale, float* k_scale, float* v_scale,
                       const signed char* sigma, int B, int H,
                       const int* cu_seqlens_q, const int* cu_seqlens_k,
                       const int* cu_blocks_q, const int* cu_blocks_k,
                       int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int D, void* stream);

/*
 * fa_fwd_fp8_varlen -- fa_fwd_fp8 over packed variable-length sequences, on
 * the output of fa_fp8_prep_varlen.
 *
 *   o            bf16 [total_q, H, D] (written); lse fp32 [H, total_q]
 *                (written)
 *   cu_*, total_*, max_seqlen_* as for fa_fp8_prep_varlen (all required)
 *   D            64, 128 or 256; scale, causal as for fa_fwd (the causal
 *                diagonal is bottom-right aligned per sequence)
 *
 * Bad sequences are skipped (their rows left unwritten) and reported as
 * FA_ERR_DEVICE_SEQLENS by fa_get_device_status.
 */
int fa_fwd_fp8_varlen(const void* q8, const void* k8, const void* v8,
                      const float* q_scale, const float* k_scale, const float* v_scale,
                      void* o, float* lse, int B, int H,
                      const int* cu_seqlens_q, const int* cu_seqlens_k,
                      const int* cu_blocks_q, const int* cu_blocks_k,
                      int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int D,
                      float scale, int causal, void* stream);

/*
 * fa_bwd_workspace_size -- bytes of device scratch fa_bwd needs: two fp32
 * values per (query token, head), rounded up to 256. 0 when there is nothing
 * to do.
 */
size_t fa_bwd_workspace_size(int H, int total_q);

/*
 * fa_bwd -- gradients of fa_fwd: dQ, dK, dV for an upstream gradient dO.
 *
 * The pages define the forward only ("Flash Attention 3 principles
 * (guijiagi)" section 1.2 with the section 2.2 softmax; the FlashAttention-3
 * wiki's table reports the backward's speed). This is the exact derivative of
 * that forward, with P recomputed from the forward's LSE:
 *   dV = P^T dO,  dS = P * (dO V^T - rowsum(dO * O)),  dQ = scale dS K,
 *   dK = scale dS^T Q.
 *
 *   q, k, v, o   the forward's inputs and output, layouts as fa_fwd
 *   dout         dO, same shape and type as o
 *   lse          the forward's LSE (fp32, [B, H, Sq] or varlen [H, total_q])
 *   dq, dk, dv   outputs, shapes and type of q, k, v (written; every row of
 *                every sequence, 0 where no pair is visible)
 *   B..dtype     as fa_fwd; D = 64, 128 or 256
 *   workspace    device scratch of at least fa_bwd_workspace_size(H, total_q)
 *                bytes, 256-byte aligned; holds the per-row constants
 *
 * P and dS are rounded to the input type before they enter the tensor-core
 * products (as P is in the forward); accumulation is fp32. Deterministic: no
 * atomics, every output row is written by one CTA. Three kernels on `stream`
 * (row constants, dK/dV, dQ), four at D = 256 (row constants, dV, dK, dQ:
 * the dK and dV accumulators do not fit tensor memory together). Bad varlen
 * sequences are skipped and reported as FA_ERR_DEVICE_SEQLENS by
 * fa_get_device_status.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D,
           float scale, int causal, const int* cu_seqlens_q, const int* cu_seqlens_k,
           int total_q, int total_k, void* workspace, size_t workspace_bytes, int dtype,
           void* stream);

/*
 * fa_get_device_status -- synchronise `stream`, then read and clear the
 * current device's status word (shared by every stream and call on the
 * device: a code may come from a kernel on another stream). Returns FA_OK, FA_ERR_DEVICE_TIMEOUT (a
 * kernel's bounded wait expired; the kernel left early and its outputs are
 * incomplete), FA_ERR_DEVICE_SEQLENS, or FA_ERR_CUDA. `raw` (may be NULL)
 * receives the raw word for diagnosis.
 */
int fa_get_device_status(void* stream, int* raw);

/* Human-readable text of a status code (static storage). */
const char* fa_strerror(int status);

/* ABI version of this header, (major << 16) | minor. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
