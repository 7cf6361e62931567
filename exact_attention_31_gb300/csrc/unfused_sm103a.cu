// Standard (unfused) attention: the three-kernel form the fused kernels replace, kept as the
// measured baseline of the IO argument.
//
// "Flash Attention: The Hidden Gem", section Background, lists what a standard implementation does:
// S = Q K^T / sqrt(d) is too large for on-chip memory and goes to HBM (step 1), the row softmax reads
// S back and writes P = softmax(S) to HBM (step 2), and O = P V reads P once more (step 3); section
// Enter Flash Attention adds that these are three separate kernels, each reading its input from HBM
// and writing its output there.  "FlashAttention: attention was never compute-bound", section Where
// the time actually goes, counts the resulting traffic: 4 n^2 + 4 n d elements per head, almost all
// of it the n x n matrices.
//
// Here the two products are cuBLAS bf16 GEMMs with fp32 accumulation (strided-batched over B*H) and
// the softmax is the kernel below.  S is stored in fp32 and P in bf16 (the tensor-core GEMM that
// multiplies P by the bf16 V takes both operands in one type); both rows are padded to ld = Nk
// rounded up to 8 elements so that every row starts on a 16-byte boundary.  The causal mask is
// applied in the softmax, as an elementwise mask of the full score matrix.

#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fattn_unfused.h"

namespace {

constexpr int kVec = 8;            // float4 chunks of the score row held by each softmax thread
constexpr int kMaxThreads = 1024;  // one CTA per row: rows up to 4 * kVec * kMaxThreads = 32768 keys
constexpr size_t kCublasWorkspace = 32ull << 20;

long long row_ld(int Nk) { return (static_cast<long long>(Nk) + 7) / 8 * 8; }

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Max (op 0) or sum (op 1) over the CTA; every thread gets the result.
template <int Op>
__device__ __forceinline__ float block_reduce(float x, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, warps = blockDim.x >> 5;
  x = Op == 0 ? warp_max(x) : warp_sum(x);
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float y = lane < warps ? red[lane] : (Op == 0 ? -INFINITY : 0.f);
  y = Op == 0 ? warp_max(y) : warp_sum(y);
  __syncthreads();  // red is reused by the next reduction
  return y;
}

// One CTA per score row r = (b*H + h)*Nq + i: read the row of S once, mask it, take its max and
// the sum of its exponentials, write the normalised row of P (bf16; masked keys and the padding to
// ld get 0) and L = m + log(l).  A row that sees no key gets P = 0 and L = -inf.
__global__ void __launch_bounds__(kMaxThreads) unfused_softmax_kernel(const float* __restrict__ S,
                                                                      __nv_bfloat16* __restrict__ P,
                                                                      float* __restrict__ lse, int Nq, int Nk,
                                                                      long long ld, int causal) {
  __shared__ float red[32];
  const long long r = blockIdx.x;
  const int i = static_cast<int>(r % Nq);
  // last visible key: bottom-right-aligned causal mask, or every key
  const long long hi = causal ? static_cast<long long>(i) + (Nk - Nq) : static_cast<long long>(Nk) - 1;
  const float4* row = reinterpret_cast<const float4*>(S + r * ld);
  const long long chunks = ld / 4;

  float x[kVec][4];
  float mx = -INFINITY;
#pragma unroll
  for (int t = 0; t < kVec; ++t) {
    const long long c = threadIdx.x + static_cast<long long>(t) * blockDim.x;
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < chunks) f = __ldcs(row + c);  // streamed: every score is read once
    const float e4[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      // a select, not arithmetic: the padding columns hold whatever the GEMM left there
      x[t][e] = (c < chunks && 4 * c + e <= hi) ? e4[e] : -INFINITY;
      mx = fmaxf(mx, x[t][e]);
    }
  }
  mx = block_reduce<0>(mx, red);

  constexpr float kLog2e = 1.4426950408889634f;
  const float ref = mx == -INFINITY ? 0.f : mx * kLog2e;
  float l = 0.f;
#pragma unroll
  for (int t = 0; t < kVec; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[t][e] = x[t][e] == -INFINITY ? 0.f : exp2f(fmaf(x[t][e], kLog2e, -ref));
      l += x[t][e];
    }
  l = block_reduce<1>(l, red);
  const float inv = l > 0.f ? 1.f / l : 0.f;

  __nv_bfloat16* prow = P + r * ld;
#pragma unroll
  for (int t = 0; t < kVec; ++t) {
    const long long c = threadIdx.x + static_cast<long long>(t) * blockDim.x;
    if (c >= chunks) continue;
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[t][0] * inv, x[t][1] * inv);
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[t][2] * inv, x[t][3] * inv);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&a);
    w.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(prow + 4 * c) = w;
  }
  if (lse != nullptr && threadIdx.x == 0) lse[r] = l > 0.f ? mx + logf(l) : -INFINITY;
}

// One cuBLAS handle per device, created by the first call on that device together with a fixed
// workspace, so that later calls allocate nothing and can be captured in a CUDA graph.
struct Handles {
  std::mutex mu;
  cublasHandle_t h[64] = {};
};

Handles& handles() {
  static Handles hs;
  return hs;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" size_t fattn_unfused_workspace_size(int B, int H, int Nq, int Nk) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return 0;
  const size_t rows = static_cast<size_t>(B) * H * Nq, ld = static_cast<size_t>(row_ld(Nk));
  return round256(rows * ld * sizeof(float)) + round256(rows * ld * sizeof(__nv_bfloat16));
}

extern "C" fattn_status fattn_fwd_unfused(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                          int H, int Nq, int Nk, int d, int causal, float scale, void* workspace,
                                          size_t ws_bytes, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || workspace == nullptr)
    return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace) ||
      (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return FATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || (causal != 0 && causal != 1) || (causal && Nq > Nk))
    return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (d < 8 || d > 256 || d % 8 != 0) return FATTN_ERR_UNSUPPORTED;
  const long long ld = row_ld(Nk);
  if (ld > 4LL * kVec * kMaxThreads) return FATTN_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(B) * H * Nq;
  if (rows > INT_MAX || static_cast<long long>(B) * H > INT_MAX) return FATTN_ERR_UNSUPPORTED;
  if (ws_bytes < fattn_unfused_workspace_size(B, H, Nq, Nk)) return FATTN_ERR_INVALID_ARG;

  float* S = static_cast<float*>(workspace);
  __nv_bfloat16* P = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(workspace) +
                                                      round256(static_cast<size_t>(rows) * ld * sizeof(float)));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FATTN_ERR_CUDA;

  Handles& hs = handles();
  std::lock_guard<std::mutex> lock(hs.mu);
  if (hs.h[dev] == nullptr) {
    cublasHandle_t h = nullptr;
    void* ws = nullptr;
    if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return FATTN_ERR_CUDA;
    if (cudaMalloc(&ws, kCublasWorkspace) != cudaSuccess ||
        cublasSetWorkspace(h, ws, kCublasWorkspace) != CUBLAS_STATUS_SUCCESS) {
      if (ws != nullptr) cudaFree(ws);
      cublasDestroy(h);
      return FATTN_ERR_CUDA;
    }
    hs.h[dev] = h;
  }
  cublasHandle_t h = hs.h[dev];
  if (cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS) return FATTN_ERR_CUDA;

  // cuBLAS is column-major: a row-major [rows, cols] matrix is its column-major transpose.
  // Step 1, S = scale * Q K^T: column-major S^T [Nk, Nq] (ld) = (K as [d, Nk])^T * (Q as [d, Nq]).
  const int BH = B * H;
  const float alpha_s = scale, one = 1.f, zero = 0.f;
  if (cublasGemmStridedBatchedEx(h, CUBLAS_OP_T, CUBLAS_OP_N, Nk, Nq, d, &alpha_s, k, CUDA_R_16BF, d,
                                 static_cast<long long>(Nk) * d, q, CUDA_R_16BF, d, static_cast<long long>(Nq) * d,
                                 &zero, S, CUDA_R_32F, static_cast<int>(ld), static_cast<long long>(Nq) * ld, BH,
                                 CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return FATTN_ERR_CUDA;

  // Step 2, P = softmax(S) row by row (and L).
  const int threads = static_cast<int>(std::min<long long>(
      kMaxThreads, std::max<long long>(32, ((ld / 4 + kVec - 1) / kVec + 31) / 32 * 32)));
  unfused_softmax_kernel<<<static_cast<unsigned>(rows), threads, 0, st>>>(S, P, lse, Nq, Nk, ld, causal);
  if (cudaGetLastError() != cudaSuccess) return FATTN_ERR_CUDA;

  // Step 3, O = P V: column-major O^T [d, Nq] = (V as [d, Nk]) * (P as [ld, Nq], first Nk rows).
  if (cublasGemmStridedBatchedEx(h, CUBLAS_OP_N, CUBLAS_OP_N, d, Nq, Nk, &one, v, CUDA_R_16BF, d,
                                 static_cast<long long>(Nk) * d, P, CUDA_R_16BF, static_cast<int>(ld),
                                 static_cast<long long>(Nq) * ld, &zero, o, CUDA_R_16BF, d,
                                 static_cast<long long>(Nq) * d, BH, CUBLAS_COMPUTE_32F,
                                 CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
    return FATTN_ERR_CUDA;
  return FATTN_OK;
}
