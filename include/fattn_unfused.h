/*
 * fattn_unfused.h -- C ABI of libfattn_unfused: standard attention as three kernels, the baseline
 * that the fused forward's memory-traffic argument is measured against.  It is not on the fused
 * path; libfattn does not use it.
 *
 * "Flash Attention: The Hidden Gem", section Background: a standard implementation writes the score
 * matrix S = Q K^T * scale to HBM (step 1), reads it back for the row softmax and writes
 * P = softmax(S) to HBM (step 2), and reads P again for O = P V (step 3); section Enter Flash
 * Attention: each step is a separate kernel that reads its input from HBM and writes its output
 * there.  "FlashAttention: attention was never compute-bound", section Where the time actually goes,
 * counts that traffic as 4 n^2 + 4 n d elements per head.
 *
 * Conventions are libfattn's (fattn.h): caller-owned, contiguous, row-major device tensors, 16-byte
 * aligned; bf16 inputs and output; stream-ordered asynchronous calls; every argument checked on the
 * host before anything is launched.
 */
#ifndef FATTN_UNFUSED_H_
#define FATTN_UNFUSED_H_

#include <stddef.h>

#include "fattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fattn_unfused_workspace_size -- bytes of device workspace fattn_fwd_unfused needs: the score
 * matrix S in fp32 and the probability matrix P in bf16, [B, H, Nq, ld] each with
 * ld = Nk rounded up to a multiple of 8, each region rounded up to 256 bytes.  0 for a size < 1.
 */
size_t fattn_unfused_workspace_size(int B, int H, int Nq, int Nk);

/*
 * fattn_fwd_unfused -- the same result as fattn_fwd, computed the standard way.
 *
 *   q, k, v   bf16 [B, H, Nq|Nk, d]; o bf16 [B, H, Nq, d]; lse fp32 [B, H, Nq] or NULL
 *   B, H, Nq, Nk >= 1; d a multiple of 8 from 8 to 256; Nk <= 32768 (one CTA holds a score row)
 *   causal    0 or 1, with fattn_fwd's bottom-right alignment; causal requires Nq <= Nk
 *   scale     finite and > 0
 *   workspace at least fattn_unfused_workspace_size(B, H, Nq, Nk) bytes, 16-byte aligned, owned by
 *             the caller; on return it holds S and P
 *
 * Kernels, in stream order:
 *   1. S = scale * Q K^T, a cuBLAS bf16 GEMM (fp32 accumulation, strided-batched over B*H) that
 *      writes S in fp32;
 *   2. a softmax kernel, one CTA per row: reads the row of S once, applies the mask, writes P
 *      (normalised, bf16; masked keys 0) and L = m + log(l);
 *   3. O = P V, a cuBLAS bf16 GEMM that writes O in bf16.
 *
 * The first call on a device creates that device's cuBLAS handle and a 32 MiB cuBLAS workspace and
 * keeps them for the life of the process; later calls allocate no device memory.  (Capture of these
 * calls in a CUDA graph is not covered by the tests.)  Returns FATTN_ERR_INVALID_ARG or FATTN_ERR_UNSUPPORTED for rejected arguments (nothing
 * launched) and FATTN_ERR_CUDA when cuBLAS or the runtime refuses a call.
 */
fattn_status fattn_fwd_unfused(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                               int Nq, int Nk, int d, int causal, float scale, void* workspace, size_t ws_bytes,
                               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_UNFUSED_H_ */
