/*
 * fattn.h -- C ABI of libfattn: exact fused attention forward, its backward, and split-KV decode
 * for sm_103a.
 *
 * The operation is the one the pages define: O = softmax(scale * Q K^T + mask) V, computed tile by
 * tile with the online-softmax recurrence (running max m, running sum l, unnormalised O rescaled by
 * exp(m_old - m_new)), so that the N x N score and probability matrices never reach device memory,
 * and L = m + log(l) emitted per query row.
 *   - "Flash Attention: The Hidden Gem", sections Background, Online Softmax, The Algorithm
 *     (steps 3-7) and The Correction Factor.
 *   - "FlashAttention: attention was never compute-bound", section The one formula.
 *   - "Understanding FlashAttention", section Attention: Q and the output are [N, D], K and V are
 *     [M, D]; decoding one token is N = 1 against M cached keys; batch and heads only repeat
 *     independent problems.
 *
 * Conventions shared by every entry point
 *   - Tensors live in device memory, are contiguous and row-major, and are owned by the caller.
 *     The library allocates no device memory in any call and keeps no pointer after a call returns.
 *   - bf16 means IEEE-style bfloat16 (1-8-7), stored as 16-bit words.  Accumulation is fp32.
 *   - `stream` is a cudaStream_t passed as void*; NULL means the legacy default stream.  Calls are
 *     asynchronous and stream-ordered: they return after enqueueing work.
 *   - Every argument is checked on the host before anything is launched.  A rejected call returns
 *     FATTN_ERR_INVALID_ARG or FATTN_ERR_UNSUPPORTED and launches nothing.
 *   - Device pointers must be 16-byte aligned.
 *   - A returned FATTN_ERR_CUDA means a launch was refused by the CUDA runtime; the runtime's own
 *     error state is left for the caller to read.
 */
#ifndef FATTN_H_
#define FATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fattn_status {
  FATTN_OK = 0,
  FATTN_ERR_INVALID_ARG = 1, /* a null/misaligned pointer, a non-positive size, a bad scale ... */
  FATTN_ERR_UNSUPPORTED = 2, /* a head dimension other than 64 or 128 */
  FATTN_ERR_CUDA = 3,        /* the CUDA runtime refused a launch or an attribute call */
  FATTN_ERR_TIMEOUT = 4,     /* a bounded on-device wait gave up (see fattn_last_error) */
  FATTN_ERR_DEBUG = 5        /* debug builds only: a device-side check failed (see fattn_debug_take) */
} fattn_status;

/*
 * fattn_fwd -- fused attention forward ("Flash Attention: The Hidden Gem", The Algorithm).
 *
 *   q    bf16 [B, H, Nq, d]      queries
 *   k    bf16 [B, H, Nk, d]      keys
 *   v    bf16 [B, H, Nk, d]      values
 *   o    bf16 [B, H, Nq, d]      output, written: O_i = diag(l_i)^-1 * O_i (step 6)
 *   lse  fp32 [B, H, Nq] or NULL log-sum-exp per row, natural log of sum_j exp(scale * q_i.k_j)
 *                                over the visible keys, i.e. L = m + log(l) (step 6)
 *   B, H, Nq, Nk >= 1; d in {64, 128}
 *   causal  0 or 1.  With 1, query row i sees key j iff j <= i + (Nk - Nq) (bottom-right
 *           alignment; the usual lower triangle when Nq == Nk).  Requires Nq <= Nk, so that every
 *           row sees at least one key.
 *   scale   finite and > 0 (typically 1/sqrt(d)).
 *
 * The kernel reads Q, K and V and writes O and L; no score or probability tile leaves the chip.
 *
 * Numerics: each row's exponent reference is the max of its first key tile with a visible key
 * and is not raised afterwards (softmax is unchanged by the choice of reference, The Correction
 * Factor).  A row whose weights then leave a safe range (weight sum above 2^64, i.e. scores more
 * than about 64 log2-units above those of its first tile, or a non-finite output) marks its
 * 128-row query tile, and the kernel computes the marked tiles again on the tensor cores, after
 * its other work, with the running max and the O rescale of The Correction Factor (at most about
 * twice the time when every tile is marked); the result is within the same tolerance either way.
 * fattn_fwd_recomputed_rows counts such rows.
 */
fattn_status fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                       int Nq, int Nk, int d, int causal, float scale, void* stream);

/*
 * fattn_fwd_masked -- fattn_fwd with a banded mask ("Understanding FlashAttention", Attention: a
 * mask is elementwise and independent of the scores, causal masking being one kind among others;
 * What is left to the implementation, point 2: rows whose keys are all masked).
 *
 * With off = Nk - Nq, query row i sees key j iff
 *     i + off - window_left  <=  j  <=  i + off + window_right,
 * where -1 leaves that side unbounded.  No mask is (-1, -1), causal is (-1, 0) (the same as
 * fattn_fwd with causal = 1), a sliding window of the last W keys is (W - 1, 0).  Any Nq, Nk >= 1
 * is accepted.  A row with no visible key gets o = 0 and L = -inf (log of an empty sum).
 * Returns FATTN_ERR_INVALID_ARG for a window side below -1; other arguments as for fattn_fwd.
 */
fattn_status fattn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                              int Nq, int Nk, int d, int window_left, int window_right, float scale,
                              void* stream);

/*
 * fattn_fwd_mask -- fattn_fwd_masked with an element mask on top of the band ("Understanding
 * FlashAttention", Attention: a mask is elementwise and independent of the scores; What is left to
 * the implementation, point 2: rows whose keys are all masked).  O = softmax(scale * Q K^T + mask) V
 * where the mask gives -inf to the pairs (i, j) that the band or the element mask hides.
 *
 *   mask      device memory, 16-byte aligned, owned by the caller: a bit per (query, key) pair.  Row
 *             i of head (b, h) is fattn_mask_row_words(Nk) 32-bit words starting at word
 *             b * mask_stride_b + h * mask_stride_h + i * fattn_mask_row_words(Nk); key j is bit
 *             (j & 31) of its word j >> 5, set = the key may be seen.  Bits past Nk are ignored.
 *   mask_stride_b, mask_stride_h   in 32-bit words, >= 0 and multiples of 4; 0 shares one mask over
 *             that dimension (one mask for every head: mask_stride_h = 0).
 *   window_left, window_right   the band of fattn_fwd_masked ((-1, -1) for the element mask alone).
 *   workspace device memory of at least fattn_mask_workspace_size(B, H, Nq, Nk) bytes, owned by the
 *             caller: it receives the mask's tile summary, two bits per 128-query by 128-key tile
 *             telling whether the mask hides all, some or none of it, written once per distinct
 *             mask (once in all for mask_stride_b = mask_stride_h = 0).  Tiles it hides entirely are
 *             skipped (no loads, no products); only partly hidden tiles read the mask bits.  Calls
 *             sharing a workspace must not overlap.
 *
 * A row with no visible key gets o = 0 and L = -inf.  Two kernels run on `stream`: the tile summary,
 * then the forward.  Returns FATTN_ERR_INVALID_ARG for a null or misaligned mask, a negative or
 * unaligned stride, or a short workspace; other arguments as for fattn_fwd_masked.
 */
int fattn_mask_row_words(int Nk); /* 4 * ceil(Nk / 128): whole 16-byte groups per row; -1 if Nk < 1 */
size_t fattn_mask_workspace_size(int B, int H, int Nq, int Nk);
fattn_status fattn_fwd_mask(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                            int Nk, int d, const void* mask, long long mask_stride_b, long long mask_stride_h,
                            int window_left, int window_right, float scale, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * fattn_bwd -- gradients of the attention forward ("Flash Attention: The Hidden Gem", Phase 2:
 * Chain Rule Through a Matrix Multiply, The Softmax Jacobian, The D Shortcut, The Algorithm).
 *
 * For O = softmax(scale * Q K^T + mask) V and an upstream gradient dO it writes
 *   dV = P^T dO,   dQ = scale * dS K,   dK = scale * dS^T Q,
 * where P = exp(scale * Q K^T - L) is recomputed from the forward's L, dP = dO V^T,
 * D = rowsum(dO o O) and dS = P o (dP - D).  The pages state the gradients without the scale; the
 * factor on dQ and dK is the chain rule through S = scale * Q K^T.
 *
 *   q, k, v  bf16, as given to fattn_fwd
 *   o        bf16 [B, H, Nq, d]  the forward output for these q, k, v (only D = rowsum(dO o O) uses it)
 *   lse      fp32 [B, H, Nq]     the forward's L (natural log), as fattn_fwd writes it
 *   dout     bf16 [B, H, Nq, d]  upstream gradient dO
 *   dq       bf16 [B, H, Nq, d]  written
 *   dk, dv   bf16 [B, H, Nk, d]  written
 *   B, H, Nq, Nk, d, causal, scale   as for fattn_fwd (the same mask must be used)
 *   workspace        device memory of at least fattn_bwd_workspace_size(B, H, Nq, d) bytes,
 *                    256-byte aligned, owned by the caller; its contents on entry do not matter
 *                    and it holds the fp32 dQ accumulator and the per-row terms of D and L on return
 *
 * Three kernels run in order on `stream`: a pre-pass (D per row, the accumulator cleared), the fused
 * kernel (one CTA per 128-key tile of a head; dK and dV stay on chip, dQ is added into the fp32
 * accumulator), and a pass that scales and rounds dQ.  Calls sharing a workspace must not overlap.
 * Accumulation is fp32; P and dS are rounded to bf16 before the products that consume them, and
 * dQ's accumulation order across key tiles is not fixed, so dQ is not bitwise reproducible.
 */
size_t fattn_bwd_workspace_size(int B, int H, int Nq, int d);
fattn_status fattn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                       int causal, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fattn_bwd_masked -- fattn_bwd for the banded masks of fattn_fwd_masked (same window_left,
 * window_right, o and lse as that call produced).  Rows with no visible key get dq = 0; keys that
 * no query sees get dk = dv = 0.
 */
fattn_status fattn_bwd_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                              int window_left, int window_right, float scale, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * fattn_bwd_mask -- fattn_bwd_masked for the element mask of fattn_fwd_mask (same mask, strides, band,
 * o and lse as that call produced).  Rows with no visible key get dq = 0; keys that no query sees get
 * dk = dv = 0; query tiles the mask hides from a key tile entirely are skipped for it.
 *
 *   workspace  device memory of at least fattn_bwd_mask_workspace_size(B, H, Nq, Nk, d) bytes,
 *              256-byte aligned, owned by the caller: the backward's workspace
 *              (fattn_bwd_workspace_size) followed by the mask's tile summary
 *              (fattn_mask_workspace_size).
 * Returns FATTN_ERR_INVALID_ARG for a null or misaligned mask, a negative or unaligned stride, or a
 * short workspace; other arguments as for fattn_bwd_masked.
 */
size_t fattn_bwd_mask_workspace_size(int B, int H, int Nq, int Nk, int d);
fattn_status fattn_bwd_mask(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                            const void* mask, long long mask_stride_b, long long mask_stride_h, int window_left,
                            int window_right, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fattn_decode_num_splits -- the number of key splits fattn_decode uses for a request.
 *
 * The cached keys are cut into blocks of 64; nblk = ceil(Nk / 64).  `num_splits` = 0 asks for the
 * default: splits of about 8 blocks (512 keys), or more of them, up to one per block, while fewer
 * than 8192 (b, h, split) work items would be left for the GPU:
 *     S = min(nblk, max(ceil(nblk / 8), ceil(8192 / (B H)))).
 * A value in [1, nblk] is used as given; split s then covers blocks [s*nblk/S, (s+1)*nblk/S).
 * Returns the resolved count, or -1 if the request is invalid (B, H or Nk < 1, or num_splits
 * outside [0, nblk]).
 */
int fattn_decode_num_splits(int B, int H, int Nk, int num_splits);

/*
 * fattn_decode_workspace_size -- bytes of scratch fattn_decode needs for these sizes.
 *
 * The workspace holds one partial state (m, l, unnormalised O[d]) in fp32 per (b, h, split).
 * Returns 0 if the sizes are invalid.
 */
size_t fattn_decode_workspace_size(int B, int H, int Nk, int d, int num_splits);

/*
 * fattn_decode -- one query token per (b, h) against a KV cache (Nq = 1; "Understanding
 * FlashAttention", Attention: decoding a single token is the case of one query row).  No mask:
 * every cached key is visible.
 *
 *   q        bf16 [B, H, 1, d]
 *   k_cache  bf16 [B, H, Nk, d]
 *   v_cache  bf16 [B, H, Nk, d]
 *   o        bf16 [B, H, 1, d]       output
 *   lse      fp32 [B, H, 1] or NULL  natural-log log-sum-exp of the scaled scores
 *   workspace  device scratch of at least fattn_decode_workspace_size(B, H, Nk, d, num_splits)
 *              bytes, 16-byte aligned, owned by the caller; its contents on entry do not matter and
 *              on return are unspecified.  Two calls in flight at once must not share it.
 *
 * Two kernels run on `stream`: a split kernel that streams each split's keys and values once and
 * leaves a partial (m, l, O) per split, and a combine kernel that merges the partials with the
 * correction-factor rule (m = max m_s, l = sum exp(m_s - m) l_s, O = sum exp(m_s - m) O_s / l;
 * "Flash Attention: The Hidden Gem", The Correction Factor) and writes O and L.
 */
fattn_status fattn_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                          int B, int H, int Nk, int d, float scale, int num_splits, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * fattn_decode_masked -- fattn_decode under the banded masks of fattn_fwd_masked.  The one query of
 * each (b, h) sits at position Nk - 1 (bottom-right alignment), so it sees the keys
 * [Nk - 1 - window_left, Nk - 1] (all of them for window_left = -1 or >= Nk - 1); window_right
 * cannot exclude a key and only has to be >= -1.  This is the decode step of a sliding-window model:
 * window (W - 1, 0) attends to the last W cached keys.  num_splits and its 64-key blocks count
 * the visible keys; the workspace needs fattn_decode_workspace_size(B, H, W_visible, d, num_splits)
 * bytes, which the size for all Nk keys always covers.  Other arguments as for fattn_decode.
 */
fattn_status fattn_decode_masked(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                                 int B, int H, int Nk, int d, int window_left, int window_right, float scale,
                                 int num_splits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fattn_decode_static -- fattn_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point: it exists for users of this library who are
 * handed only their inputs, outputs and a stream and may not call cudaMalloc -- for example a
 * plugin inside a host framework that owns every device allocation, or a latency-critical path
 * where an allocation's implicit device synchronisation is not acceptable.  It computes the same
 * result as fattn_decode with the same arguments, minus the workspace: the partial (m, l, O)
 * states live in a fixed scratch array compiled into the library (FATTN_DECODE_STATIC_WORKSPACE_BYTES
 * of device memory on every GPU that loads the library, held until the process exits).  Nothing is
 * allocated, by this library or by any library it calls.
 *
 *   num_splits  0 starts from fattn_decode_num_splits's default and lowers it until the partial
 *               states fit in the array; an explicit count must fit in the array too.
 *   Returns FATTN_ERR_INVALID_ARG, launching nothing, when the partial states for these sizes do
 *   not fit (B * H * num_splits * (d + 2) floats, each of the two arrays rounded up to 256 bytes,
 *   must not exceed FATTN_DECODE_STATIC_WORKSPACE_BYTES; with num_splits = 0 this only fails when
 *   a single split per (b, h) does not fit).  The other arguments are checked as in fattn_decode.
 *
 * Set-up: the array is created with the library's device code, which CUDA's lazy module loading
 * (the default) loads at the first call of any libfattn entry point on a device; that call may
 * synchronise.  The first call of this entry point on each device also looks up the array's device
 * address, with that device current.  Make both first calls during set-up, before any stream
 * capture begins; later calls allocate nothing and do not synchronise.
 * Sharing: every call on a device uses the same array and leaves its contents behind.  No part of
 * it needs clearing: each call writes every partial state it later reads.  Two calls whose work
 * overlaps on the GPU (different streams, or other host threads) race on the array and may return
 * wrong results; serialise them.
 */
#define FATTN_DECODE_STATIC_WORKSPACE_BYTES (8u << 20)
fattn_status fattn_decode_static(const void* q, const void* k_cache, const void* v_cache, void* o,
                                 float* lse, int B, int H, int Nk, int d, float scale, int num_splits,
                                 void* stream);

/*
 * fattn_fwd_fp8 -- the attention forward on FP8 operands ("Flash Attention: The Hidden Gem", section
 * FA1, FA2, FA3: FP8 support doubles the tensor-core rate at some cost in precision).  The pages
 * state no accuracy contract for it; this one is stated from the arithmetic.
 *
 *   q        e4m3 [B, H, Nq, d]   (OCP FP8 E4M3: 1 sign, 4 exponent, 3 mantissa bits, bias 7)
 *   k, v     e4m3 [B, H, Nk, d]
 *   o        bf16 [B, H, Nq, d]; lse fp32 [B, H, Nq] or NULL, as for fattn_fwd_masked
 *   q_descale, k_descale, v_descale   finite, > 0: the call computes the attention of the dequantised
 *            tensors q * q_descale, k * k_descale, v * v_descale, with the band of fattn_fwd_masked
 *            and the given scale
 *   d        64 or 128 (FATTN_ERR_UNSUPPORTED otherwise)
 *   workspace  device memory of at least fattn_fwd_fp8_workspace_size(B, H, Nk, d) bytes, 256-byte
 *            aligned, owned by the caller: it receives V transposed ([B*H][d][Nk rounded up to 16]),
 *            because 8-bit operands are read by the tensor core with the reduced dimension contiguous.
 *
 * Both products are e4m3 x e4m3 with fp32 accumulation, so S is exact up to fp32 summation.  The
 * probabilities enter P V rounded to e4m3 (relative error at most 2^-4 for weights above 2^-6 of the
 * stored scale, an absolute error below 2^-10 of it under that); L and the normalisation use the
 * fp32 weights.  Per output element, with p the exact probabilities of the dequantised problem:
 *     |o - o_exact| <= 2^-4 * sum_j p_j |v_j| + 2^-9 |o_exact| + (2^-15 * n_j + 2^-16) * max_j |v_j|,
 * n_j the row's visible keys (the last term covers weights stored below e4m3's normal range and the
 * fp32 arithmetic); |lse - lse_exact| <= 2^-20 |lse| + 1e-5.  Calls sharing a workspace must not
 * overlap.
 */
size_t fattn_fwd_fp8_workspace_size(int B, int H, int Nk, int d);
fattn_status fattn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                           int Nk, int d, int window_left, int window_right, float scale, float q_descale,
                           float k_descale, float v_descale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fattn_fwd_host / fattn_decode_host -- the same computations with the inputs and outputs in HOST
 * memory.  The pages put the cost of attention in moving data between memory levels ("Flash
 * Attention: The Hidden Gem", Background; "FlashAttention: attention was never compute-bound",
 * The one formula); these entry points extend that to the host link: the (b, h) problems are cut
 * into chunks of `heads_per_chunk` consecutive heads of the flattened [B * H] index, and chunk c + 1
 * is copied to the device while chunk c is computed and chunk c - 1 is copied back, through two
 * slots of a caller-owned device workspace.
 *
 *   q_host ... lse_host   host memory, same shapes and layouts as the device calls; lse_host may be
 *                         NULL.  Page-locked memory (cudaHostAlloc / cudaHostRegister) lets the
 *                         copies run asynchronously and overlap; pageable memory is accepted and
 *                         gives the same results with less overlap.  No alignment is required.
 *   window_left, window_right   the band of fattn_fwd_masked ((-1, 0) is causal, (-1, -1) none).
 *                         For the decode only window_left matters (fattn_decode_masked): just the
 *                         visible keys [Nk - 1 - window_left, Nk - 1] of each head are copied.
 *   heads_per_chunk       0 picks a default (about four chunks for the forward, eight for the
 *                         decode); otherwise 1 .. B * H.
 *   workspace             device memory of at least the matching *_workspace_size bytes for the
 *                         same arguments, 256-byte aligned, owned by the caller.
 *   stream                the compute stream.  The copies run on two streams the library creates
 *                         once per device and keeps for the life of the process, ordered against
 *                         `stream` with events: the call's first copy waits for the work enqueued on
 *                         `stream` before the call, and `stream` waits for the call's last copy.
 *                         Synchronise `stream` before reading the host outputs.
 *
 * The kernels are those of the device calls, applied to each chunk as its own problem (B = 1,
 * H = heads in the chunk), so the outputs equal the device calls' outputs for the same inputs.
 * Calls that share a workspace, or that run from several host threads at once, must be serialised
 * by the caller.  Returns the device calls' statuses, and FATTN_ERR_CUDA if a copy or an event call
 * is refused.
 */
size_t fattn_fwd_host_workspace_size(int B, int H, int Nq, int Nk, int d, int heads_per_chunk);
fattn_status fattn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                            float* lse_host, int B, int H, int Nq, int Nk, int d, int window_left,
                            int window_right, float scale, int heads_per_chunk, void* workspace,
                            size_t workspace_bytes, void* stream);
size_t fattn_decode_host_workspace_size(int B, int H, int Nk, int d, int window_left, int heads_per_chunk);
fattn_status fattn_decode_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                               float* lse_host, int B, int H, int Nk, int d, int window_left, int window_right,
                               float scale, int heads_per_chunk, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * fattn_last_error -- wait for `stream`, then read and clear the library's on-device status word on
 * the current device.  Returns FATTN_OK, FATTN_ERR_TIMEOUT if some kernel's bounded wait gave up
 * since the last read (its outputs are then unspecified), or FATTN_ERR_CUDA if the stream reported
 * an error.
 */
fattn_status fattn_last_error(void* stream);

/*
 * fattn_fwd_recomputed_rows -- the number of rows of fattn_fwd and fattn_fwd_masked that failed the
 * fast path's range check on the current device since the library was loaded, and whose query
 * tiles were therefore computed again with a running max (a diagnostic; see fattn_fwd, Numerics).
 * Waits for all work on the current device first.  *out must not be NULL
 * (FATTN_ERR_INVALID_ARG); FATTN_ERR_CUDA if the device reported an error.
 */
fattn_status fattn_fwd_recomputed_rows(unsigned long long* out);

/*
 * Debug builds.  The library can be built with device-side checks (libfattn_debug.so, compiled with
 * -DFATTN_DEBUG): before every TMA copy, bulk copy, mbarrier operation, tensor-memory load or store
 * and tcgen05.mma the kernels check the operands against the hardware's rules (shared-memory and
 * barrier alignment; a TMA copy's innermost coordinate a multiple of 16 elements, and no store or
 * reduce starting below 0; a warp's tensor-memory accesses inside its 32-lane quarter and the 512
 * allocated columns), and every output store against its tensor's extent.  An operation that
 * breaks a rule is not issued; the rule is recorded instead, so that a bad index is reported and
 * does not fault the GPU (a copy left out leaves its barrier incomplete, and the bounded waits end
 * the kernel).  In debug builds every entry point waits for its stream after launching and returns
 * FATTN_ERR_DEBUG when a check failed, and fattn_last_error reports it too.  The arithmetic is the
 * release build's: results are bit-identical.
 *
 * fattn_debug_build -- 1 for a library built with the device-side checks, 0 otherwise.
 * fattn_debug_take  -- (debug builds: wait for the device, then) read and clear the checks' record:
 *   *rules = the OR of the rules broken since the last call (bit 0 shared-memory or barrier
 *   alignment, bit 1 TMA coordinate, bit 2 tensor-memory lane, bit 3 tensor-memory column, bit 4
 *   bulk-copy size or address, bit 5 output store out of range), *first = the first failure as
 *   block << 32 | thread << 8 | (index of its lowest rule bit + 1), 0 if none.  Release builds
 *   report 0 and 0 and touch no device.  FATTN_ERR_INVALID_ARG for a NULL pointer.
 */
int fattn_debug_build(void);
fattn_status fattn_debug_take(unsigned int* rules, unsigned long long* first);

/* fattn_status_string -- a static, human-readable name for a status code (never NULL). */
const char* fattn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H_ */
