// fattn_internal.h -- launcher interfaces shared by the host entry points and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "fattn.h"

namespace fattn {

// Status bits the kernels may set in the library's device status word.
constexpr unsigned int kStatusTimeout = 1u;

struct FwdProblem {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, Nq, Nk, d;
  // Band mask, bottom-right aligned: row i sees key j iff i+off-window_left <= j <= i+off+window_right
  // with off = Nk - Nq; -1 leaves that side unbounded.  No mask (-1, -1); causal (-1, 0).
  int window_left, window_right;
  float scale;
  // Failure-detection testing only (never set in normal use): the key tile of this block index is
  // not loaded, so the waits for it must give up and report a timeout.  -1 = off.
  int drop_kv_block;
  // Device counter of rows that failed the fixed-reference range check (incremented by the kernel).
  unsigned long long* recomputed;
  // Element mask (null: none).  Bit j & 31 of word (j >> 5) of row i of head (b, h) at
  // mask + b * mask_sb + h * mask_sh + i * mask_words (32-bit words), set = visible.  `tiles` is its
  // summary by query tile, as written by launch_mask_tiles.
  const void* mask = nullptr;
  long long mask_sb = 0, mask_sh = 0;
  int mask_words = 0;
  const unsigned long long* tiles = nullptr;
};

struct DecodeProblem {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, Nk, d;
  float scale;
  int num_splits;    // resolved, in [1, nblk]
  float* ws_o;       // [B*H*num_splits, d] partial unnormalised outputs
  float* ws_ml;      // [B*H*num_splits, 2] partial (m, l), m in log2 units of the scaled score
  int key_lo;        // first visible key (a sliding window keeps keys [key_lo, Nk)); 0 = all
};

struct BwdProblem {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  int B, H, Nq, Nk, d;
  int window_left, window_right;  // band mask as in FwdProblem
  float scale;
  float* ws_dq;    // [B*H][Nq_pad][d] fp32 dQ accumulator
  void* ws_ext_q;   // [B*H][Nq_pad][16] bf16: three terms of -L / scale (per query row)
  void* ws_ext_do;  // [B*H][Nq_pad][16] bf16: three terms of -D
  // Failure-detection testing only (never set in normal use): the key and value tiles are not
  // loaded, so the kernel's waits for them must give up and report a timeout.
  int drop_kv;
  // Element mask (null: none), laid out as in FwdProblem, with its tile summary by key tile.
  const void* mask = nullptr;
  long long mask_sb = 0, mask_sh = 0;
  int mask_words = 0;
  const unsigned long long* tiles = nullptr;
};

// Query rows of the backward workspace per head: Nq rounded up to the 128-row query tile.
inline int bwd_padded_rows(int Nq) { return (Nq + 127) / 128 * 128; }

// Keys per decode block: the unit a split is made of.
constexpr int kDecodeBlockKeys = 64;

// Prefill: the three tensor maps describe q, k, v as 3-D [B*H][N][d] bf16 tensors with
// 64-element (128-byte) inner boxes of 128 rows and 128-byte swizzle.
cudaError_t launch_prefill(const FwdProblem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, unsigned int* status, unsigned long long timeout_ns,
                           cudaStream_t stream);

cudaError_t launch_decode(const DecodeProblem& p, cudaStream_t stream);

// Debug builds (-DFATTN_DEBUG): each kernel file's record of device-side checks that failed (the
// rule bits, and the first failure as block << 32 | thread << 8 | rule + 1), read and optionally
// cleared; release builds report zeros.
cudaError_t debug_take_prefill(unsigned int* rules, unsigned long long* first, bool clear);
cudaError_t debug_take_fp8(unsigned int* rules, unsigned long long* first, bool clear);
cudaError_t debug_take_backward(unsigned int* rules, unsigned long long* first, bool clear);
cudaError_t debug_take_decode(unsigned int* rules, unsigned long long* first, bool clear);
// All files' records combined (rules OR-ed, the first non-empty first-failure record).
cudaError_t debug_collect(unsigned int* rules, unsigned long long* first, bool clear);
// Debug builds: wait for `stream` after a call's launches and turn a failed device-side check into
// FATTN_ERR_DEBUG (the records stay for fattn_debug_take).  Release builds return `s` unchanged.
fattn_status debug_after(void* stream, fattn_status s);

// Element-mask summary.  The mask is judged per 128 x 128 tile (query rows 128 i.., keys 128 j..,
// inside Nq x Nk) once per slice: one slice per (b, h) the mask's strides tell apart (a zero stride
// shares a slice), slice (b' * nh + h') with b' = mask_sb ? b : 0, h' = mask_sh ? h : 0 and
// nh = mask_sh ? H : 1.  Each slice holds, per "major" tile (the query tile i by_key == false, the
// key tile j when true), `words` 64-bit words of live bits (the tile has a visible key) followed by
// `words` of partial bits (visible and hidden keys both), bit t & 63 of word t >> 6 for minor tile t
// (the key tile, or the query tile).  words = ceil(minor tiles / 64).
__host__ __device__ inline int mask_summary_words(int minor_tiles) { return (minor_tiles + 63) / 64; }
inline size_t mask_summary_bytes(long long slices, int Nq, int Nk, bool by_key) {
  const int tq = (Nq + 127) / 128, tk = (Nk + 127) / 128;
  const int major = by_key ? tk : tq, minor = by_key ? tq : tk;
  return static_cast<size_t>(slices) * major * 2 * mask_summary_words(minor) * sizeof(unsigned long long);
}
// The summary's strides over b and h in 64-bit words (0 where the mask is shared).
inline void mask_summary_strides(long long mask_sb, long long mask_sh, int H, int Nq, int Nk, bool by_key,
                                 long long& sb, long long& sh) {
  const int tq = (Nq + 127) / 128, tk = (Nk + 127) / 128;
  const long long per_slice =
      static_cast<long long>(by_key ? tk : tq) * 2 * mask_summary_words(by_key ? tq : tk);
  sh = mask_sh != 0 ? per_slice : 0;
  sb = mask_sb != 0 ? (mask_sh != 0 ? H : 1) * per_slice : 0;
}
cudaError_t launch_mask_tiles(const uint32_t* mask, long long mask_sb, long long mask_sh, int mask_words, int B,
                              int H, int Nq, int Nk, bool by_key, unsigned long long* tiles, cudaStream_t stream);

// Backward: q, k, v, dout as for the prefill; tdq describes ws_dq as a 3-D [B*H][Nq_pad][d] fp32
// tensor with 32-element (128-byte) inner boxes of 128 rows and 128-byte swizzle.
cudaError_t launch_backward(const BwdProblem& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, unsigned int* status,
                            unsigned long long timeout_ns, cudaStream_t stream);

// FP8 forward (d = 64 or 128): q, k, v are e4m3 [B*H][N][d]; the attention is that of q * q_descale,
// k * k_descale, v * v_descale.  vt is V transposed, [B*H][d][fp8_padded_keys(Nk)].
struct Fp8Problem {
  const void* q;
  const void* k;
  const void* vt;
  void* o;
  float* lse;
  int B, H, Nq, Nk, d;
  int window_left, window_right;
  float scale, q_descale, k_descale, v_descale;
  int drop_kv_block;  // failure-detection testing only: key tile never loaded (-1 = off)
};

int fp8_padded_keys(int Nk);
cudaError_t launch_vt_transpose(const void* v, void* vt, int BH, int Nk, int d, cudaStream_t stream);
// tq, tk: [B*H][N][d] e4m3, d x 128-row boxes (128-byte swizzle for d = 128, 64-byte for d = 64);
// tvt: [B*H][d][Nk_pad] e4m3, 128-key x d-row boxes, 128-byte swizzle.
cudaError_t launch_prefill_fp8(const Fp8Problem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tvt, unsigned int* status, unsigned long long timeout_ns,
                               cudaStream_t stream);

}  // namespace fattn
