// fattn_api.cu -- the C ABI of libfattn: argument checks, TMA descriptors, launches, status.
//
// Every entry point validates its arguments on the host and launches nothing when they are bad;
// no entry point allocates device memory.  The declarations and their contracts are in fattn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>
#include <mutex>

#include "fattn.h"
#include "fattn_internal.h"

namespace fattn {
namespace {

// Status word the kernels raise bits in (bounded waits that gave up).  One copy per device.
__device__ unsigned int g_device_status;
// Rows of fattn_fwd that failed the prefill kernel's range check, whose tiles it computed again
// with a running max (cumulative).
__device__ unsigned long long g_recomputed_rows;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

unsigned long long wait_timeout_ns() {
  static unsigned long long ns = [] {
    const char* s = getenv("FATTN_WAIT_TIMEOUT_MS");
    long long ms = s ? atoll(s) : 0;
    if (ms <= 0) ms = 4000;
    return static_cast<unsigned long long>(ms) * 1000000ull;
  }();
  return ns;
}

// Failure-detection testing only: FATTN_TEST_DROP_KV_BLOCK=<j> makes the prefill kernel skip the
// load of key tile j, so that its bounded waits give up and report FATTN_ERR_TIMEOUT.
int test_drop_kv_block() {
  static int j = [] {
    const char* s = getenv("FATTN_TEST_DROP_KV_BLOCK");
    return s ? atoi(s) : -1;
  }();
  return j;
}

// Failure-detection testing only: FATTN_TEST_DROP_BWD_KV=1 makes the backward kernel skip its key
// and value loads, so that its bounded waits give up and report FATTN_ERR_TIMEOUT.
int test_drop_bwd_kv() {
  static int on = [] {
    const char* s = getenv("FATTN_TEST_DROP_BWD_KV");
    return s ? atoi(s) : 0;
  }();
  return on;
}

// Device address of g_device_status for the current device, looked up once per device.
cudaError_t device_status_ptr(unsigned int** out) {
  static std::mutex mu;
  static unsigned int* cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && cache[dev] != nullptr) {
    *out = cache[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_device_status);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev] = static_cast<unsigned int*>(p);
  *out = static_cast<unsigned int*>(p);
  return cudaSuccess;
}

// Device address of g_recomputed_rows for the current device, looked up once per device.
cudaError_t recomputed_rows_ptr(unsigned long long** out) {
  static std::mutex mu;
  static unsigned long long* cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && cache[dev] != nullptr) {
    *out = cache[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_recomputed_rows);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev] = static_cast<unsigned long long*>(p);
  *out = static_cast<unsigned long long*>(p);
  return cudaSuccess;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// [BH][N][d] bf16, 128-row x 64-column boxes, 128-byte swizzle; out-of-range rows read as zero.
bool make_map(CUtensorMap* map, const void* base, int BH, int N, int d) {
  EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                  estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [BH][rows][d] fp32 (the backward's dQ accumulator), 128-row x 32-column boxes, 128-byte swizzle.
bool make_map_f32(CUtensorMap* map, void* base, int BH, int rows, int d) {
  EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(rows) * d * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D byte tensor [BH][rows][cols] (e4m3 operands), boxes of box_rows rows x box_cols bytes (128 or
// 64) with the swizzle of the same span; out-of-range elements read as zero.  cols and the row pitch
// are multiples of 16 bytes.
bool make_map_u8(CUtensorMap* map, const void* base, int BH, int rows, int cols, int box_cols, int box_rows) {
  EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  if (box_cols != 128 && box_cols != 64) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows) * cols};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estride[3] = {1, 1, 1};
  const CUtensorMapSwizzle sw = box_cols == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool positive_sizes(long long a, long long b, long long c, long long d) {
  return a >= 1 && b >= 1 && c >= 1 && d >= 1;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace
}  // namespace fattn

using namespace fattn;

extern "C" {

const char* fattn_status_string(int status) {
  switch (status) {
    case FATTN_OK: return "FATTN_OK";
    case FATTN_ERR_INVALID_ARG: return "FATTN_ERR_INVALID_ARG";
    case FATTN_ERR_UNSUPPORTED: return "FATTN_ERR_UNSUPPORTED";
    case FATTN_ERR_CUDA: return "FATTN_ERR_CUDA";
    case FATTN_ERR_TIMEOUT: return "FATTN_ERR_TIMEOUT";
    case FATTN_ERR_DEBUG: return "FATTN_ERR_DEBUG";
    default: return "FATTN_UNKNOWN_STATUS";
  }
}

}  // extern "C"

namespace fattn {

cudaError_t debug_collect(unsigned int* rules, unsigned long long* first, bool clear) {
  cudaError_t (*const parts[])(unsigned int*, unsigned long long*, bool) = {debug_take_prefill, debug_take_fp8,
                                                                            debug_take_backward, debug_take_decode};
  *rules = 0u;
  *first = 0ull;
  for (auto take : parts) {
    unsigned int r = 0u;
    unsigned long long f = 0ull;
    const cudaError_t e = take(&r, &f, clear);
    if (e != cudaSuccess) return e;
    *rules |= r;
    if (*first == 0ull) *first = f;
  }
  return cudaSuccess;
}

fattn_status debug_after(void* stream, fattn_status s) {
#ifdef FATTN_DEBUG
  if (s != FATTN_OK) return s;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FATTN_ERR_CUDA;
  unsigned int rules = 0u;
  unsigned long long first = 0ull;
  if (debug_collect(&rules, &first, false) != cudaSuccess) return FATTN_ERR_CUDA;
  return rules != 0u ? FATTN_ERR_DEBUG : FATTN_OK;
#else
  (void)stream;
  return s;
#endif
}

namespace {

// Bytes of an element mask's tile summary with one slice per head, in the larger of its two layouts
// (a mask shared over heads or batch entries uses less of it).
size_t mask_tiles_bytes(int B, int H, int Nq, int Nk) {
  const long long slices = static_cast<long long>(B) * H;
  const size_t by_query = mask_summary_bytes(slices, Nq, Nk, false);
  const size_t by_key = mask_summary_bytes(slices, Nq, Nk, true);
  return align_up(by_query > by_key ? by_query : by_key, 256);
}

struct MaskArg {
  const void* mask = nullptr;  // null: no element mask
  long long sb = 0, sh = 0;
  void* workspace = nullptr;
  size_t workspace_bytes = 0;
};

fattn_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                      int Nk, int d, int wl, int wr, float scale, void* stream, const MaskArg& mk = MaskArg()) {
  if (!q || !k || !v || !o) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FATTN_ERR_INVALID_ARG;
  if (!positive_sizes(B, H, Nq, Nk)) return FATTN_ERR_INVALID_ARG;
  if (wl < -1 || wr < -1) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 0x7fffffffLL / 64) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;

  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, BH, Nq, d) || !make_map(&tk, k, BH, Nk, d) || !make_map(&tv, v, BH, Nk, d))
    return FATTN_ERR_CUDA;
  unsigned int* status = nullptr;
  unsigned long long* recomputed = nullptr;
  if (device_status_ptr(&status) != cudaSuccess || recomputed_rows_ptr(&recomputed) != cudaSuccess)
    return FATTN_ERR_CUDA;
  FwdProblem p{q, k, v, o, lse, B, H, Nq, Nk, d, wl, wr, scale, test_drop_kv_block(), recomputed};
  if (mk.mask != nullptr) {
    p.mask = mk.mask;
    p.mask_sb = mk.sb;
    p.mask_sh = mk.sh;
    p.mask_words = fattn_mask_row_words(Nk);
    p.tiles = static_cast<const unsigned long long*>(mk.workspace);
    if (launch_mask_tiles(static_cast<const uint32_t*>(mk.mask), mk.sb, mk.sh, p.mask_words, B, H, Nq, Nk, false,
                          static_cast<unsigned long long*>(mk.workspace), static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
      return FATTN_ERR_CUDA;
  }
  if (launch_prefill(p, tq, tk, tv, status, wait_timeout_ns(), static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return FATTN_ERR_CUDA;
  return debug_after(stream, FATTN_OK);
}

fattn_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, int wl,
                      int wr, float scale, void* workspace, size_t workspace_bytes, void* stream,
                      const MaskArg& mk = MaskArg()) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FATTN_ERR_INVALID_ARG;
  if (!positive_sizes(B, H, Nq, Nk)) return FATTN_ERR_INVALID_ARG;
  if (wl < -1 || wr < -1) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 0x7fffffffLL / 256) return FATTN_ERR_INVALID_ARG;
  if (Nq > 0x7fffffff - 128) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  const size_t need = fattn_bwd_workspace_size(B, H, Nq, d);
  if (need == 0 || workspace_bytes < need) return FATTN_ERR_INVALID_ARG;

  const int BH = B * H;
  const int Nq_pad = bwd_padded_rows(Nq);
  const size_t rows = static_cast<size_t>(BH) * Nq_pad;
  char* ws = static_cast<char*>(workspace);
  float* ws_dq = reinterpret_cast<float*>(ws);
  void* ws_ext_q = ws + align_up(rows * d * sizeof(float), 256);
  void* ws_ext_do = ws + align_up(rows * d * sizeof(float), 256) + align_up(rows * 32, 256);
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_map(&tq, q, BH, Nq, d) || !make_map(&tk, k, BH, Nk, d) || !make_map(&tv, v, BH, Nk, d) ||
      !make_map(&tdo, dout, BH, Nq, d) || !make_map_f32(&tdq, ws_dq, BH, Nq_pad, d))
    return FATTN_ERR_CUDA;
  unsigned int* status = nullptr;
  if (device_status_ptr(&status) != cudaSuccess) return FATTN_ERR_CUDA;
  BwdProblem p{q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, wl, wr, scale, ws_dq, ws_ext_q, ws_ext_do,
               test_drop_bwd_kv()};
  if (mk.mask != nullptr) {
    p.mask = mk.mask;
    p.mask_sb = mk.sb;
    p.mask_sh = mk.sh;
    p.mask_words = fattn_mask_row_words(Nk);
    p.tiles = static_cast<const unsigned long long*>(mk.workspace);
    if (launch_mask_tiles(static_cast<const uint32_t*>(mk.mask), mk.sb, mk.sh, p.mask_words, B, H, Nq, Nk, true,
                          static_cast<unsigned long long*>(mk.workspace), static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
      return FATTN_ERR_CUDA;
  }
  if (launch_backward(p, tq, tk, tv, tdo, tdq, status, wait_timeout_ns(), static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return FATTN_ERR_CUDA;
  return debug_after(stream, FATTN_OK);
}

}  // namespace
}  // namespace fattn

extern "C" {

fattn_status fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                       int Nq, int Nk, int d, int causal, float scale, void* stream) {
  if (causal != 0 && causal != 1) return FATTN_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return FATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, -1, causal ? 0 : -1, scale, stream);
}

fattn_status fattn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                              int Nq, int Nk, int d, int window_left, int window_right, float scale, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, window_left, window_right, scale, stream);
}

int fattn_mask_row_words(int Nk) {
  if (Nk < 1) return -1;
  return 4 * ((Nk + 127) / 128);
}

size_t fattn_mask_workspace_size(int B, int H, int Nq, int Nk) {
  if (!positive_sizes(B, H, Nq, Nk)) return 0;
  return mask_tiles_bytes(B, H, Nq, Nk);
}

fattn_status fattn_fwd_mask(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                            int Nk, int d, const void* mask, long long mask_stride_b, long long mask_stride_h,
                            int window_left, int window_right, float scale, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (mask == nullptr || !aligned16(mask) || workspace == nullptr) return FATTN_ERR_INVALID_ARG;
  if (mask_stride_b < 0 || mask_stride_h < 0 || (mask_stride_b & 3) || (mask_stride_h & 3))
    return FATTN_ERR_INVALID_ARG;
  if (!positive_sizes(B, H, Nq, Nk)) return FATTN_ERR_INVALID_ARG;
  const size_t need = fattn_mask_workspace_size(B, H, Nq, Nk);
  if (need == 0 || workspace_bytes < need) return FATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * ((Nq + 127) / 128) * ((Nk + 127) / 128) / 8 > 0x7fffffffLL)
    return FATTN_ERR_INVALID_ARG;
  MaskArg mk;
  mk.mask = mask;
  mk.sb = mask_stride_b;
  mk.sh = mask_stride_h;
  mk.workspace = workspace;
  mk.workspace_bytes = workspace_bytes;
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, window_left, window_right, scale, stream, mk);
}

size_t fattn_bwd_workspace_size(int B, int H, int Nq, int d) {
  if (!positive_sizes(B, H, Nq, d)) return 0;
  const size_t rows = static_cast<size_t>(B) * H * bwd_padded_rows(Nq);
  return align_up(rows * d * sizeof(float), 256) + 2 * align_up(rows * 32, 256);
}

fattn_status fattn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                       int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (causal != 0 && causal != 1) return FATTN_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return FATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, -1, causal ? 0 : -1, scale, workspace,
                  workspace_bytes, stream);
}

fattn_status fattn_bwd_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                              int window_left, int window_right, float scale, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, window_left, window_right, scale, workspace,
                  workspace_bytes, stream);
}

size_t fattn_bwd_mask_workspace_size(int B, int H, int Nq, int Nk, int d) {
  const size_t a = fattn_bwd_workspace_size(B, H, Nq, d), b = fattn_mask_workspace_size(B, H, Nq, Nk);
  return a == 0 || b == 0 ? 0 : a + b;
}

fattn_status fattn_bwd_mask(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
                            const void* mask, long long mask_stride_b, long long mask_stride_h, int window_left,
                            int window_right, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (mask == nullptr || !aligned16(mask) || workspace == nullptr) return FATTN_ERR_INVALID_ARG;
  if (mask_stride_b < 0 || mask_stride_h < 0 || (mask_stride_b & 3) || (mask_stride_h & 3))
    return FATTN_ERR_INVALID_ARG;
  if (!positive_sizes(B, H, Nq, Nk)) return FATTN_ERR_INVALID_ARG;
  const size_t need = fattn_bwd_mask_workspace_size(B, H, Nq, Nk, d);
  if (need == 0 || workspace_bytes < need) return FATTN_ERR_INVALID_ARG;
  // The backward's own workspace first, the tile summary after it (both multiples of 256 bytes).
  const size_t bwd_bytes = fattn_bwd_workspace_size(B, H, Nq, d);
  MaskArg mk;
  mk.mask = mask;
  mk.sb = mask_stride_b;
  mk.sh = mask_stride_h;
  mk.workspace = static_cast<char*>(workspace) + bwd_bytes;
  mk.workspace_bytes = workspace_bytes - bwd_bytes;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, window_left, window_right, scale, workspace,
                  bwd_bytes, stream, mk);
}

int fattn_decode_num_splits(int B, int H, int Nk, int num_splits) {
  if (B < 1 || H < 1 || Nk < 1) return -1;
  const int nblk = (Nk + kDecodeBlockKeys - 1) / kDecodeBlockKeys;
  if (num_splits == 0) {
    // Splits of about 8 blocks, or more of them (up to one per block) while fewer than 8192
    // (b, h, split) warps would be left to spread over the GPU.
    const long long bh = static_cast<long long>(B) * H;
    const long long by_length = (nblk + 7) / 8;
    const long long by_width = (8192 + bh - 1) / bh;
    return static_cast<int>(std::min<long long>(nblk, std::max(by_length, by_width)));
  }
  if (num_splits < 0 || num_splits > nblk) return -1;
  return num_splits;
}

size_t fattn_decode_workspace_size(int B, int H, int Nk, int d, int num_splits) {
  if (!positive_sizes(B, H, Nk, d)) return 0;
  const int S = fattn_decode_num_splits(B, H, Nk, num_splits);
  if (S < 1) return 0;
  const size_t parts = static_cast<size_t>(B) * H * S;
  return align_up(parts * d * sizeof(float), 256) + align_up(parts * 2 * sizeof(float), 256);
}

fattn_status fattn_decode_masked(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                                 int B, int H, int Nk, int d, int window_left, int window_right, float scale,
                                 int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  if (window_left < -1 || window_right < -1) return FATTN_ERR_INVALID_ARG;
  if (Nk < 1) return FATTN_ERR_INVALID_ARG;
  // The one query sits at position Nk - 1 (bottom-right): it sees keys [Nk - 1 - window_left, Nk - 1];
  // window_right cannot exclude anything, and the last key is always visible.
  const int key_lo = window_left >= 0 && window_left < Nk - 1 ? Nk - 1 - window_left : 0;
  if (!q || !k_cache || !v_cache || !o || !workspace) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      !aligned16(workspace) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FATTN_ERR_INVALID_ARG;
  if (!positive_sizes(B, H, Nk, 1)) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  const int S = fattn_decode_num_splits(B, H, Nk - key_lo, num_splits);
  if (S < 1) return FATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * S > 0x7fffffffLL) return FATTN_ERR_INVALID_ARG;
  const size_t need = fattn_decode_workspace_size(B, H, Nk - key_lo, d, num_splits);
  if (need == 0 || workspace_bytes < need) return FATTN_ERR_INVALID_ARG;
  const size_t parts = static_cast<size_t>(B) * H * S;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          align_up(parts * d * sizeof(float), 256));
  DecodeProblem p{q, k_cache, v_cache, o, lse, B, H, Nk, d, scale, S, ws_o, ws_ml, key_lo};
  if (launch_decode(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FATTN_ERR_CUDA;
  return debug_after(stream, FATTN_OK);
}

fattn_status fattn_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                          int B, int H, int Nk, int d, float scale, int num_splits, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !o || !workspace) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      !aligned16(workspace) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FATTN_ERR_INVALID_ARG;
  if (!positive_sizes(B, H, Nk, 1)) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  const int S = fattn_decode_num_splits(B, H, Nk, num_splits);
  if (S < 1) return FATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * S > 0x7fffffffLL) return FATTN_ERR_INVALID_ARG;
  const size_t need = fattn_decode_workspace_size(B, H, Nk, d, num_splits);
  if (need == 0 || workspace_bytes < need) return FATTN_ERR_INVALID_ARG;
  const size_t parts = static_cast<size_t>(B) * H * S;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          align_up(parts * d * sizeof(float), 256));
  DecodeProblem p{q, k_cache, v_cache, o, lse, B, H, Nk, d, scale, S, ws_o, ws_ml, 0};
  if (launch_decode(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FATTN_ERR_CUDA;
  return debug_after(stream, FATTN_OK);
}

}  // extern "C"

extern "C" {

size_t fattn_fwd_fp8_workspace_size(int B, int H, int Nk, int d) {
  if (!positive_sizes(B, H, Nk, 1) || (d != 128 && d != 64)) return 0;
  return align_up(static_cast<size_t>(B) * H * d * fp8_padded_keys(Nk), 256);
}

fattn_status fattn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                           int Nk, int d, int window_left, int window_right, float scale, float q_descale,
                           float k_descale, float v_descale, void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !workspace) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FATTN_ERR_INVALID_ARG;
  if (!positive_sizes(B, H, Nq, Nk) || window_left < -1 || window_right < -1) return FATTN_ERR_INVALID_ARG;
  for (float x : {scale, q_descale, k_descale, v_descale})
    if (!(x > 0.f) || !isfinite(x)) return FATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 0x7fffffffLL / 64 || Nk > 0x7fffffff - 128) return FATTN_ERR_INVALID_ARG;
  if (d != 128 && d != 64) return FATTN_ERR_UNSUPPORTED;
  const size_t need = fattn_fwd_fp8_workspace_size(B, H, Nk, d);
  if (need == 0 || workspace_bytes < need) return FATTN_ERR_INVALID_ARG;
  const int BH = B * H;
  const int Nk_pad = fp8_padded_keys(Nk);
  CUtensorMap tq, tk, tvt;
  if (!make_map_u8(&tq, q, BH, Nq, d, d, 128) || !make_map_u8(&tk, k, BH, Nk, d, d, 128) ||
      !make_map_u8(&tvt, workspace, BH, d, Nk_pad, 128, d))
    return FATTN_ERR_CUDA;
  unsigned int* status = nullptr;
  if (device_status_ptr(&status) != cudaSuccess) return FATTN_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_vt_transpose(v, workspace, BH, Nk, d, s) != cudaSuccess) return FATTN_ERR_CUDA;
  Fp8Problem p{q, k, workspace, o, lse, B, H, Nq, Nk, d, window_left, window_right, scale, q_descale, k_descale,
               v_descale, test_drop_kv_block()};
  if (launch_prefill_fp8(p, tq, tk, tvt, status, wait_timeout_ns(), s) != cudaSuccess) return FATTN_ERR_CUDA;
  return debug_after(stream, FATTN_OK);
}

}  // extern "C"

// ------------------------------------------------------------------------------------------------
// Allocation-free decode: the partial states live in a fixed array compiled into the library.
// ------------------------------------------------------------------------------------------------
namespace fattn {
namespace {

static __device__ __align__(256) unsigned char g_decode_static_ws[FATTN_DECODE_STATIC_WORKSPACE_BYTES];

// The array's host-side name is only a stand-in for the symbol; the kernels need its device
// address, looked up once per device with that device current.
cudaError_t decode_static_ws_ptr(void** out) {
  static std::mutex mu;
  static void* cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && cache[dev] != nullptr) {
    *out = cache[dev];
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_static_ws);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev] = p;
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace fattn

extern "C" {

fattn_status fattn_decode_static(const void* q, const void* k_cache, const void* v_cache, void* o,
                                 float* lse, int B, int H, int Nk, int d, float scale, int num_splits,
                                 void* stream) {
  if (!q || !k_cache || !v_cache || !o) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FATTN_ERR_INVALID_ARG;
  if (!positive_sizes(B, H, Nk, 1)) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  const size_t cap = FATTN_DECODE_STATIC_WORKSPACE_BYTES;
  int S = fattn_decode_num_splits(B, H, Nk, num_splits);
  if (S < 1) return FATTN_ERR_INVALID_ARG;
  if (num_splits == 0) {
    // largest split count (at most one per 64-key block) whose partial states fit
    while (S > 1 && fattn_decode_workspace_size(B, H, Nk, d, S) > cap) {
      const size_t per_split = static_cast<size_t>(B) * H * (d + 2) * sizeof(float);
      const int guess = static_cast<int>(cap / per_split);
      S = (guess >= 1 && guess < S) ? guess : S - 1;
    }
  }
  const size_t need = fattn_decode_workspace_size(B, H, Nk, d, S);
  if (need == 0 || need > cap) return FATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * S > 0x7fffffffLL) return FATTN_ERR_INVALID_ARG;
  void* ws = nullptr;
  if (decode_static_ws_ptr(&ws) != cudaSuccess) return FATTN_ERR_CUDA;
  const size_t parts = static_cast<size_t>(B) * H * S;
  float* ws_o = static_cast<float*>(ws);
  float* ws_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + align_up(parts * d * sizeof(float), 256));
  DecodeProblem p{q, k_cache, v_cache, o, lse, B, H, Nk, d, scale, S, ws_o, ws_ml, 0};
  if (launch_decode(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FATTN_ERR_CUDA;
  return debug_after(stream, FATTN_OK);
}

fattn_status fattn_fwd_recomputed_rows(unsigned long long* out) {
  if (out == nullptr) return FATTN_ERR_INVALID_ARG;
  unsigned long long* p = nullptr;
  if (recomputed_rows_ptr(&p) != cudaSuccess) return FATTN_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return FATTN_ERR_CUDA;
  if (cudaMemcpy(out, p, sizeof(*out), cudaMemcpyDeviceToHost) != cudaSuccess) return FATTN_ERR_CUDA;
  return FATTN_OK;
}

fattn_status fattn_last_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FATTN_ERR_CUDA;
  unsigned int* status = nullptr;
  if (device_status_ptr(&status) != cudaSuccess) return FATTN_ERR_CUDA;
  unsigned int h = 0;
  if (cudaMemcpy(&h, status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FATTN_ERR_CUDA;
  if (h != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return FATTN_ERR_CUDA;
  }
#ifdef FATTN_DEBUG
  unsigned int rules = 0;
  unsigned long long first = 0;
  if (debug_collect(&rules, &first, false) != cudaSuccess) return FATTN_ERR_CUDA;
  if (rules != 0) return FATTN_ERR_DEBUG;
#endif
  return (h & kStatusTimeout) ? FATTN_ERR_TIMEOUT : FATTN_OK;
}

int fattn_debug_build(void) {
#ifdef FATTN_DEBUG
  return 1;
#else
  return 0;
#endif
}

fattn_status fattn_debug_take(unsigned int* rules, unsigned long long* first) {
  if (rules == nullptr || first == nullptr) return FATTN_ERR_INVALID_ARG;
#ifdef FATTN_DEBUG
  if (cudaDeviceSynchronize() != cudaSuccess) return FATTN_ERR_CUDA;
#endif
  return debug_collect(rules, first, true) == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA;
}

}  // extern "C"
