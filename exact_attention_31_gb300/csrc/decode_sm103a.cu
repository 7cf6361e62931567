// decode_sm103a.cu -- split-KV attention for one query token per (b, h) against a KV cache.
//
// Decoding is N = 1 against M cached keys ("Understanding FlashAttention", Attention).  The work is
// a single pass over K and V, so the path is bound by device-memory bandwidth: every cached byte is
// read exactly once with 128-bit loads, and the only other traffic is one small partial state per
// split.
//
// Split kernel: one warp per (b, h, split).  A split is a run of 64-key blocks.  Lane l owns the
// 16-byte chunk (l mod d/8) of the rows of key sub-stream (l div d/8), so one warp-wide load covers
// 32/(d/8) consecutive key rows (512 contiguous bytes).  Each lane carries the online-softmax state
// (m, l, o[8]) of its sub-stream over groups of keys ("Flash Attention: The Hidden Gem", Online
// Softmax; "FlashAttention: attention was never compute-bound", The one formula), and at the end of
// the split the sub-streams are merged with the same correction rule and written as one partial
// (m, l, O[d]).
//
// Combine kernel: one CTA per (b, h) merges its partials to M = max m_s, l = sum exp(m_s - M) l_s,
// O = sum exp(m_s - M) O_s / l, L = M + log(l) ("Flash Attention: The Hidden Gem", The Correction
// Factor), pairwise with the same rule so that no separate pass for M is needed (exact by
// exp(a-c) = exp(a-b) exp(b-c)).
//
// All exponents are base 2 on scores pre-multiplied by c = scale * log2(e).
#include <cuda_bf16.h>
#include <math.h>

#include "fattn_internal.h"
#include "sm103a_ptx.cuh"

namespace fattn {
namespace {

constexpr int kSplitWarps = 4;           // warps per CTA in the split kernel
constexpr int kCombineThreads = 256;

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = bf16lo_to_f32(u.x);
  f[1] = bf16hi_to_f32(u.x);
  f[2] = bf16lo_to_f32(u.y);
  f[3] = bf16hi_to_f32(u.y);
  f[4] = bf16lo_to_f32(u.z);
  f[5] = bf16hi_to_f32(u.z);
  f[6] = bf16lo_to_f32(u.w);
  f[7] = bf16hi_to_f32(u.w);
}

// D/8 lanes share one key row; KPI key rows per warp-wide load; G keys per lane per step.
template <int D>
struct SplitCfg {
  static constexpr int kLanesPerRow = D / 8;
  static constexpr int kRowsPerLoad = 32 / kLanesPerRow;
  static constexpr int kKeysPerLane = 8;                            // per step
  static constexpr int kKeysPerStep = kRowsPerLoad * kKeysPerLane;  // 16 (d=128) or 32 (d=64)
};

template <int D>
__global__ void __launch_bounds__(kSplitWarps * 32)
    decode_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                        const __nv_bfloat16* __restrict__ v, float* __restrict__ ws_o,
                        float* __restrict__ ws_ml, int BH, int Nk, int key_lo, int nblk, int S, float c_log2) {
  using C = SplitCfg<D>;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kSplitWarps + (threadIdx.x >> 5);
  if (gw >= BH * S) return;
  const int bh = gw / S;
  const int s = gw - bh * S;
  // split s covers 64-key blocks [s*nblk/S, (s+1)*nblk/S) of the visible keys [key_lo, Nk)
  const int key_begin = key_lo + static_cast<int>((static_cast<long long>(s) * nblk / S) * kDecodeBlockKeys);
  const int key_end =
      min(Nk, key_lo + static_cast<int>((static_cast<long long>(s + 1) * nblk / S) * kDecodeBlockKeys));
  const int chunk = lane % C::kLanesPerRow;
  const int sub = lane / C::kLanesPerRow;

  float qf[8];
  unpack8(*reinterpret_cast<const uint4*>(q + static_cast<size_t>(bh) * D + chunk * 8), qf);
#pragma unroll
  for (int i = 0; i < 8; ++i) qf[i] *= c_log2;

  const size_t head = static_cast<size_t>(bh) * Nk * D;
  const __nv_bfloat16* kp = k + head + chunk * 8;
  const __nv_bfloat16* vp = v + head + chunk * 8;

  float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;

  for (int key0 = key_begin; key0 < key_end; key0 += C::kKeysPerStep) {
    uint4 kr[C::kKeysPerLane], vr[C::kKeysPerLane];
#pragma unroll
    for (int g = 0; g < C::kKeysPerLane; ++g) {
      const int key = key0 + g * C::kRowsPerLoad + sub;
      if (key < key_end) {
        kr[g] = ld_nc_v4(kp + static_cast<size_t>(key) * D);
        vr[g] = ld_nc_v4(vp + static_cast<size_t>(key) * D);
      } else {
        kr[g] = make_uint4(0, 0, 0, 0);
        vr[g] = make_uint4(0, 0, 0, 0);
      }
    }
    float x[C::kKeysPerLane];
#pragma unroll
    for (int g = 0; g < C::kKeysPerLane; ++g) {
      float kf[8];
      unpack8(kr[g], kf);
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) dot = fmaf(qf[i], kf[i], dot);
#pragma unroll
      for (int off = C::kLanesPerRow / 2; off > 0; off >>= 1)
        dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const int key = key0 + g * C::kRowsPerLoad + sub;
      x[g] = (key < key_end) ? dot : -INFINITY;
    }
    float mx = x[0];
#pragma unroll
    for (int g = 1; g < C::kKeysPerLane; ++g) mx = fmaxf(mx, x[g]);
    const float m_new = fmaxf(m, mx);
    if (m_new == -INFINITY) continue;  // this sub-stream saw no key in the step
    const float corr = ex2_approx(m - m_new);  // 0 while m is still -inf
    l *= corr;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] *= corr;
#pragma unroll
    for (int g = 0; g < C::kKeysPerLane; ++g) {
      const float p = ex2_approx(x[g] - m_new);
      l += p;
      float vf[8];
      unpack8(vr[g], vf);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vf[i], acc[i]);
    }
    m = m_new;
  }

  // Merge the sub-streams (lanes that hold the same chunk of different key rows).
#pragma unroll
  for (int off = C::kLanesPerRow; off < 32; off <<= 1) {
    const float m_o = __shfl_xor_sync(0xffffffffu, m, off);
    const float l_o = __shfl_xor_sync(0xffffffffu, l, off);
    const float mm = fmaxf(m, m_o);
    const float a = (mm == -INFINITY) ? 0.f : ex2_approx(m - mm);
    const float b = (mm == -INFINITY) ? 0.f : ex2_approx(m_o - mm);
    l = l * a + l_o * b;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float acc_o = __shfl_xor_sync(0xffffffffu, acc[i], off);
      acc[i] = acc[i] * a + acc_o * b;
    }
    m = mm;
  }
  const size_t part = static_cast<size_t>(bh) * S + s;
  if (!dbg_in(static_cast<long long>(part), static_cast<long long>(BH) * S)) return;
  if (sub == 0) {
    float4* dst = reinterpret_cast<float4*>(ws_o + part * D + chunk * 8);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  if (lane == 0) {
    ws_ml[2 * part] = m;
    ws_ml[2 * part + 1] = l;
  }
}

// Merge of partial states (m_a, l_a, acc_a) <- (m_b, l_b, acc_b) by the correction-factor rule.
__device__ __forceinline__ void merge_state(float& m, float& l, float4& acc, float mb, float lb, float4 ob) {
  const float mm = fmaxf(m, mb);
  const float wa = (mm == -INFINITY) ? 0.f : ex2_approx(m - mm);
  const float wb = (mm == -INFINITY) ? 0.f : ex2_approx(mb - mm);
  l = fmaf(l, wa, lb * wb);
  acc.x = fmaf(acc.x, wa, ob.x * wb);
  acc.y = fmaf(acc.y, wa, ob.y * wb);
  acc.z = fmaf(acc.z, wa, ob.z * wb);
  acc.w = fmaf(acc.w, wa, ob.w * wb);
  m = mm;
}

// One CTA per (b, h).  D/4 threads cover one partial O_s (a float4 each); the CTA's groups of D/4
// threads walk the splits in one pass, each keeping its own running (m, l, O) and loading
// kUnroll partial states ahead, then the groups' states are merged through shared memory.
template <int D>
__global__ void __launch_bounds__(kCombineThreads)
    decode_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_ml,
                          __nv_bfloat16* __restrict__ o, float* __restrict__ lse, int S) {
  constexpr int kLanesPerRow = D / 4;                       // float4 per thread
  constexpr int kGroups = kCombineThreads / kLanesPerRow;   // splits handled in parallel
  constexpr int kUnroll = 4;
  __shared__ float4 part_acc[kGroups][kLanesPerRow];
  __shared__ float2 part_ml[kGroups];
  const int bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int g = tid / kLanesPerRow, c = tid % kLanesPerRow;
  const float2* ml = reinterpret_cast<const float2*>(ws_ml) + static_cast<size_t>(bh) * S;
  const float* base = ws_o + static_cast<size_t>(bh) * S * D + 4 * c;

  float m = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = g; s0 < S; s0 += kGroups * kUnroll) {
    float2 st[kUnroll];
    float4 ov[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int s = s0 + u * kGroups;
      if (s < S) {
        st[u] = ml[s];
        ov[u] = *reinterpret_cast<const float4*>(base + static_cast<size_t>(s) * D);
      } else {
        st[u] = make_float2(-INFINITY, 0.f);
        ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) merge_state(m, l, acc, st[u].x, st[u].y, ov[u]);
  }
  part_acc[g][c] = acc;
  if (c == 0) part_ml[g] = make_float2(m, l);
  __syncthreads();
  if (g == 0) {
#pragma unroll
    for (int gg = 1; gg < kGroups; ++gg) merge_state(m, l, acc, part_ml[gg].x, part_ml[gg].y, part_acc[gg][c]);
    const float inv = 1.f / l;
    const uint32_t lo = pack_bf16x2(acc.x * inv, acc.y * inv);
    const uint32_t hi = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(o + static_cast<size_t>(bh) * D + 4 * c) = make_uint2(lo, hi);
    if (c == 0 && lse != nullptr) lse[bh] = (m + __log2f(l)) * 0.6931471805599453f;
  }
}

template <int D>
cudaError_t launch_decode_d(const DecodeProblem& p, cudaStream_t stream) {
  const int BH = p.B * p.H;
  const int nblk = (p.Nk - p.key_lo + kDecodeBlockKeys - 1) / kDecodeBlockKeys;
  const long long warps = static_cast<long long>(BH) * p.num_splits;
  const unsigned int grid = static_cast<unsigned int>((warps + kSplitWarps - 1) / kSplitWarps);
  decode_split_kernel<D><<<grid, kSplitWarps * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(p.q), static_cast<const __nv_bfloat16*>(p.k),
      static_cast<const __nv_bfloat16*>(p.v), p.ws_o, p.ws_ml, BH, p.Nk, p.key_lo, nblk, p.num_splits,
      p.scale * 1.4426950408889634f);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<D><<<BH, kCombineThreads, 0, stream>>>(
      p.ws_o, p.ws_ml, static_cast<__nv_bfloat16*>(p.o), p.lse, p.num_splits);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeProblem& p, cudaStream_t stream) {
  if (p.d == 64) return launch_decode_d<64>(p, stream);
  return launch_decode_d<128>(p, stream);
}

// Debug builds: read (and optionally clear) this file's device-side check record.
FATTN_DEBUG_ACCESSOR(decode)

}  // namespace fattn
