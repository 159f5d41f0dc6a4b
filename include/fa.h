/*
 * fa.h -- C ABI of libfa.so: exact scaled-dot-product attention on GB300
 * (sm_103a), computed tile by tile with the online-softmax recurrence.
 *
 * What every call computes (the pages' definition; the kernels never write an
 * S x S matrix to device memory):
 *
 *   S = scale * Q K^T,  P = softmax(S) over the visible keys of each row,
 *   O = P V,  LSE_i = ln sum_j exp(S_ij)  (natural log, scale included)
 *
 *   -- "Flash Attention" history page, sections 1.1 (the attention formula),
 *      1.2 (running max m, denominator l, rescaled output), 1.3 (tiles live on
 *      chip and are discarded), 2.1 (parallelism over the query sequence,
 *      causal tiles skipped); FlashAttention_01 page, "online softmax
 *      derivation" (m, l, unnormalised u, divide once at the end; mask before
 *      the max; an explicit rule for rows with no visible key) and "backward
 *      recomputation" (save one logsumexp per row, rebuild P from it).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  * Tensors are bf16 (IEEE bfloat16 bit patterns), contiguous, layout
 *    [B, H, S, d] with d innermost.  Q, O, dO, dQ: [B, Hq, Sq, d].
 *    K, V, dK, dV: [B, Hkv, Sk, d].  LSE: fp32 [B, Hq, Sq].
 *  * Every pointer is a DEVICE pointer of the current CUDA device, 16-byte
 *    aligned.  The caller owns every buffer and the stream; the library never
 *    allocates, frees or retains device memory (scratch comes from the
 *    caller's workspace argument).
 *  * Grouped K/V heads (GQA/MQA, "Flash Attention" practitioner page 2.3):
 *    Hq % Hkv == 0 and query head h reads KV head h / (Hq / Hkv).
 *  * Visibility of key j to query row i of batch row b:
 *        k_start[b] <= j < k_end[b]   and   (causal == 0  or  j <= i + Sk - Sq)
 *    The causal rule is aligned to the bottom-right corner (for Sq == Sk it is
 *    the usual lower triangle).  k_start / k_end are optional device int32[B]
 *    arrays (NULL means 0 and Sk); values outside [0, Sk] are clamped.
 *  * A row with no visible key gets O = 0 and LSE = -inf, and contributes zero
 *    gradient; no -inf - (-inf) is ever evaluated.
 *  * d (head dimension) must be 64 or 128 (FA_ERR_UNSUPPORTED otherwise).
 *  * scale must be finite and >= 0 (FA_ERR_INVALID_ARG otherwise); scale 0
 *    gives uniform weights over the visible keys.
 *  * Calls are asynchronous: they validate, enqueue kernels on `stream` and
 *    return.  A validation failure returns before any launch and writes
 *    nothing.  Launch failures return FA_ERR_CUDA.  fa_last_error_detail()
 *    gives a one-line reason for the last non-OK status of the calling thread.
 *  * Device-side pipeline waits are bounded (1 s).  A wait that runs out
 *    records FA_ERR_TIMEOUT in a device status word and the kernel returns
 *    early; fa_device_status() reads (and optionally clears) that word.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* bad size, null or misaligned pointer, Hq % Hkv != 0 */
  FA_ERR_UNSUPPORTED = 2, /* head dimension other than 64 or 128, or no sm_103a device */
  FA_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than the *_workspace_size query */
  FA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  FA_ERR_TIMEOUT = 5      /* a device pipeline wait ran out (see fa_device_status) */
} fa_status;

/*
 * Forward pass.  O = softmax(scale * Q K^T) V over visible keys, and per-row
 * LSE (natural log, scale included).  lse may be NULL when the caller does
 * not need it; the backward needs it.
 *   q [B,Hq,Sq,d], k/v [B,Hkv,Sk,d], o [B,Hq,Sq,d] (written), lse [B,Hq,Sq]
 *   (written).  B, Hq, Hkv, Sq, Sk >= 1.
 * Follows: "Flash Attention" history page 1.2-1.3 and 2.1; FlashAttention_01
 * page, online-softmax derivation and the large-score worked example.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                 int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                 const int32_t* k_start, const int32_t* k_end, cudaStream_t stream);

/* Bytes of device workspace fa_bwd needs: an fp32 dQ accumulator
   [B,Hq,Sq,d] and the fp32 row terms D_i = rowsum(dO * O) [B,Hq,Sq]. */
size_t fa_bwd_workspace_size(int B, int Hq, int Sq, int d);

/*
 * Backward pass by recomputation.  Given the forward's inputs, its bf16
 * output o and its lse, and the upstream gradient dout:
 *   D_i = rowsum(dO * O),  P = exp(scale * Q K^T - LSE) on visible entries,
 *   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
 *   dQ = scale * dS K,  dK = scale * dS^T Q,
 * with dK/dV of a KV head summed over its query heads.  dq [B,Hq,Sq,d],
 * dk/dv [B,Hkv,Sk,d] are written (bf16).  The mask arguments, causal flag and
 * scale must be the ones the forward used.  workspace must hold at least
 * fa_bwd_workspace_size(B, Hq, Sq, d) bytes; its contents on entry are
 * ignored and on return are unspecified.
 * Follows: FlashAttention_01 page, "why the backward can recompute" and the
 * chain-rule section (dV, dP, dS, dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d)).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
                 int Sk, int d, int causal, float scale, const int32_t* k_start,
                 const int32_t* k_end, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream);

/*
 * Per-key boolean masks and packed ragged ("varlen") sequences.
 * Follows: FlashAttention_01 page, "interface and implementation constraints"
 * (masks and ragged layouts are part of the kernel contract; statistics cover
 * only valid rows; a ragged layout tells logical row numbers from packed ones).
 *
 * Key mask bits: key j of mask row r is visible iff bit (j % 32) of word
 * bits[r * fa_key_mask_words(Sk) + j / 32] is set.  A hidden key is treated
 * like a key outside [k_start, k_end): it gets weight 0 in the softmax and
 * zero dK/dV.  A row that sees no key gives O = 0, LSE = -inf.  The bits
 * buffer is caller-owned device memory, 16-byte aligned; bits past Sk are
 * ignored.  fa_pack_key_mask builds it from one byte per key.
 */
size_t fa_key_mask_words(int Sk); /* uint32 words per mask row: 4 * ceil(Sk / 128) */

/* bits[rows][fa_key_mask_words(Sk)] = packed (mask[rows][Sk] != 0); device
   buffers, asynchronous on stream.  mask needs no alignment. */
fa_status fa_pack_key_mask(const uint8_t* mask, uint32_t* bits, int rows, int Sk,
                           cudaStream_t stream);

/* fa_fwd with a per-(batch row, key) mask: key_mask_bits has B mask rows
   (NULL = no mask, exactly fa_fwd). */
fa_status fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                        const int32_t* k_start, const int32_t* k_end,
                        const uint32_t* key_mask_bits, cudaStream_t stream);

/* fa_bwd with the same key mask the forward used (NULL = exactly fa_bwd). */
fa_status fa_bwd_masked(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                        int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                        const int32_t* k_start, const int32_t* k_end,
                        const uint32_t* key_mask_bits, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/*
 * Packed ragged forward.  nseq sequences are concatenated along the row
 * axis: q/o [Hq, total_q, d], k/v [Hkv, total_k, d], lse [Hq, total_q].
 * Sequence s owns packed query rows [cu_seqlens_q[s], cu_seqlens_q[s+1]) and
 * packed keys [cu_seqlens_k[s], cu_seqlens_k[s+1]) and attends only within
 * itself; the causal rule is bottom-right within the sequence (logical key
 * j' <= logical row i' + Sk_s - Sq_s).  cu_seqlens_* are device int32[nseq+1],
 * non-decreasing, from 0 to total_q / total_k (values are clamped to
 * [0, total]).  max_seqlen_q/k are host upper bounds on the sequences'
 * query and key counts; they size the grid, and rows or keys of a sequence
 * past them are not processed (their outputs are left unwritten).  Packed
 * rows or keys that belong to no sequence are not written either.
 * Rows of a sequence without keys get O = 0 and LSE = -inf.  key_mask_bits
 * (nullable) is one mask row over the packed keys.
 */
fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                        int Hkv, int d, int causal, float scale, const uint32_t* key_mask_bits,
                        cudaStream_t stream);

/*
 * Packed ragged backward, the layout and arguments of fa_fwd_varlen: dq
 * [Hq, total_q, d] and dk/dv [Hkv, total_k, d] are written; workspace holds
 * fa_bwd_workspace_size(1, Hq, total_q, d) bytes.
 */
fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int nseq,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                        int Hkv, int d, int causal, float scale, const uint32_t* key_mask_bits,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Dropout on the attention weights, with the random mapping fixed as part of
 * the forward/backward contract (FlashAttention_01 page, "why the backward
 * can recompute", "interface and implementation constraints" and "training
 * configuration and misuse boundaries": recomputation needs the same mask,
 * statistics, scale and dropout mapping).
 *   O_i = sum_j P_ij * keep_ij * r * v_j,  P the undropped softmax;
 *   LSE is the undropped one (what the backward needs to rebuild P).
 *   keep_ij <=> the 16-bit half (j mod 2) (0: low, 1: high) of word
 *   ((j mod 8) / 2) of Philox4x32-10 (Salmon et al., SC 2011) at counter
 *   (j / 8, i, b * Hq + h, offset) under key (seed & 0xffffffff, seed >> 32)
 *   is >= thr = floor(dropout_p * 2^16); i is the query row and j the key
 *   index within batch row b.  The keep probability is thus 1 - thr / 2^16,
 *   and kept weights are scaled by its reciprocal r = 2^16 / (2^16 - thr),
 *   so E[keep_ij * r] = 1 exactly (p below 2^-16: thr = 0, nothing is dropped
 *   and r = 1).
 * dropout_p must lie in [0, 1) (0 = no dropout); the backward must get the
 * forward's dropout_p, seed and offset.  Otherwise these are fa_fwd_masked /
 * fa_bwd_masked (key_mask_bits may be NULL).
 */
fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                         const int32_t* k_start, const int32_t* k_end,
                         const uint32_t* key_mask_bits, float dropout_p,
                         unsigned long long seed, unsigned int offset, cudaStream_t stream);

fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                         int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                         const int32_t* k_start, const int32_t* k_end,
                         const uint32_t* key_mask_bits, float dropout_p,
                         unsigned long long seed, unsigned int offset, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/*
 * FP8 forward ("Flash Attention" history page 2.2: FA3 runs attention in
 * FP8).  q [B,Hq,Sq,128], k [B,Hkv,Sk,128] and vt [B,Hkv,128,Sk] (V
 * transposed: each head's value matrix stored head-dimension-major) hold
 * e4m3 (OCP FP8 E4M3, bias 7, max 448) bytes; the attention is computed for
 * Q = q_descale * q, K = k_descale * k, V = v_descale * v with the bf16
 * forward's visibility rules (key interval, causal, GQA).  o (bf16
 * [B,Hq,Sq,128]) and lse are written as by fa_fwd.  Both matrix products run
 * in FP8 with fp32 accumulation; the softmax weights are rounded to e4m3 for
 * the second product (O is normalised by the sum of the rounded weights, the
 * LSE uses the exact fp32 sum).  d must be 128 (FA_ERR_UNSUPPORTED
 * otherwise), Sk a multiple of 16, and the descale factors finite and > 0.
 */
fa_status fa_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B,
                     int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                     float q_descale, float k_descale, float v_descale, const int32_t* k_start,
                     const int32_t* k_end, cudaStream_t stream);

/* Bytes of device workspace fa_decode needs for a cache of Sk_max positions:
   per (b, query head, split) partial outputs and logsumexps. */
size_t fa_decode_workspace_size(int B, int Hq, int Sk_max, int d);

/*
 * Single-query decode (Sq = 1) over a padded KV cache with split-KV and a
 * logsumexp merge.  q [B,Hq,1,d]; k_cache/v_cache [B,Hkv,Sk_max,d] of which
 * the first seqlens_k[b] positions of batch row b are valid; seqlens_k is a
 * device int32[B] (values clamped to [0, Sk_max]; 0 gives O = 0, LSE = -inf).
 * o [B,Hq,1,d] is written; lse [B,Hq] is written when not NULL.  The split
 * plan depends only on (B, Hq, Hkv, Sk_max, d), never on the values in
 * seqlens_k, so the call never reads device memory on the host.
 * workspace must hold fa_decode_workspace_size(B, Hq, Sk_max, d) bytes.
 * Follows: FlashAttention_01 page, "performance validation" (prefill with
 * Sq = Sk and decode with Sq = 1 are measured separately); the merge applies
 * the rescale rule of the "Flash Attention" history page 1.2 to whole
 * per-chunk states.
 */
fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache, void* o,
                    float* lse, const int32_t* seqlens_k, int B, int Hq, int Hkv, int Sk_max,
                    int d, float scale, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream);

/* Size of the scratch array built into the library for fa_decode_noalloc. */
#define FA_DECODE_NOALLOC_MAX_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * fa_decode without a workspace argument, for callers that cannot allocate
 * device memory: callers whose interface only carries the input and output
 * buffers (a fixed operator or plugin signature with no workspace slot), and
 * callers that run where allocating is not possible or not wanted (a host
 * framework that owns all device memory through its own pool, or a
 * latency-critical loop that cannot pay for cudaMalloc and the device
 * synchronisation it implies).  The pages have no counterpart: it is an
 * interface variant of fa_decode, with the same arguments, results and errors
 * minus workspace/workspace_bytes.
 *
 * Scratch comes from one array of FA_DECODE_NOALLOC_MAX_SCRATCH_BYTES (64 MiB)
 * compiled into the library; each GPU on which it is used keeps that array
 * until the process exits.  No device memory is allocated by the call.
 *   - Problems whose fa_decode_workspace_size(B, Hq, Sk_max, d) exceeds the
 *     array are rejected with FA_ERR_WORKSPACE before any device work.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is tied to the device's CUDA context: after cudaDeviceReset
 *     (or with another context current) the next call looks it up again, so
 *     that call, too, should come before any capture.
 *   - All calls on a device share the array: calls that can overlap on the GPU
 *     (different streams without ordering between them) race and corrupt each
 *     other's results.  Calls ordered on one stream are safe; nothing in the
 *     array needs to start at zero.
 */
fa_status fa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o,
                            float* lse, const int32_t* seqlens_k, int B, int Hq, int Hkv,
                            int Sk_max, int d, float scale, cudaStream_t stream);

/* Reads the device status words of the current device (this synchronises the
   device).  Returns FA_OK or FA_ERR_TIMEOUT; *code_out (may be NULL) receives
   the raw word (low 16 bits: error code, high 16 bits: wait site).  When
   clear != 0 the words are reset to 0 afterwards. */
fa_status fa_device_status(unsigned int* code_out, int clear);

/* Self-test of the bounded device waits behind FA_ERR_TIMEOUT.  Enqueues on
   `stream` one small kernel whose two warps wait, with the helpers every
   attention kernel uses, on barriers that nothing arrives on: the first
   wait runs out after its 1 s limit, records the timeout at wait site 0x7e
   in the device status word and raises the kernel's abort flag; the second
   gives up on seeing the flag (no second record).  The kernel then returns
   normally and the context stays usable.  result is a device array of two
   unsigned ints (16-byte aligned), set to 1 for each wait that reported
   failure.  Afterwards fa_device_status() returns FA_ERR_TIMEOUT with the
   word 0x007e0001.  Takes about one second; for tests of the failure path
   only. */
fa_status fa_selftest_wait_timeout(unsigned int* result, cudaStream_t stream);

/* Profiling hook (the pages ask that a timing confirm which kernel actually
   ran).  start/stop are cudaEvent_t handles created by the caller.  The next
   fa_fwd, fa_bwd or fa_decode call made on this host thread records `start`
   on its stream right before its main kernel (fa_fwd: the attention kernel;
   fa_bwd: the key-tile kernel, not the preprocess or dQ-convert kernels;
   fa_decode: the split partial kernel, not the merge) and `stop` right after
   it, then the hook disarms itself.  Passing NULL for both disarms it.  The
   events are not owned by the library. */
fa_status fa_profile_next_launch(cudaEvent_t start, cudaEvent_t stop);

/* Static text for a status code. */
const char* fa_status_string(fa_status s);

/* One-line detail of the last non-OK status returned on the calling thread
   ("" when none). */
const char* fa_last_error_detail(void);

/* Library version string. */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
