// prefill_fp8_sm103a.cu -- fused exact attention forward on FP8 (e4m3) operands, d = 64 or 128, sm_103a.
//
// The computation is the same tiled online-softmax forward as the bf16 kernel ("Flash Attention:
// The Hidden Gem", The Algorithm; "FlashAttention: attention was never compute-bound", The one
// formula), on inputs given as e4m3 with one dequantisation factor per tensor: the attention of
// q * q_descale, k * k_descale and v * v_descale.  Both products run as tcgen05.mma kind::f8f6f4
// with fp32 accumulation ("Flash Attention: The Hidden Gem", section FA1, FA2, FA3: FP8 operands
// trade precision for twice the tensor-core rate):
//   S_t = Q_t K_j^T    A = Q_t (smem, K-major), B = K_j (smem, K-major), 32 elements per K step
//   O_t += P_t V_j     A = P_t in TMEM as e4m3 (four keys per 32-bit column), B = V_j^T (smem, K-major)
// 8-bit operands are read K-major only, so V is transposed once per call into a workspace
// ([B*H][d][Nk rounded up to 16] e4m3, keys past Nk zero) by fwd_fp8_vt_kernel.  A Q or K tile is
// 128 rows of d bytes: with d = 128 it is stored with the 128-byte swizzle, with d = 64 with the
// 64-byte one (a row is one 64-byte swizzle span).  A V^T tile is d rows of 128 keys, 128-byte swizzle.
//
// Layout per CTA (persistent, one per SM, 320 threads): warps 0-3 and 4-7 the softmax of two
// 128-row query tiles (one thread per row), warp 8 the TMA producer, warp 9 the MMA issuer and TMEM
// owner.  TMEM: S_t at columns 128t, O_t at 256 + 128t; P_t (32 columns) overwrites the first
// columns of S_t once they are in registers, so S_t(j+1) is issued after P_t(j) V_j (issue order).
//
// P is rounded to e4m3 from 2^(s c - m_ref + 5): the reference is raised when a tile's max exceeds
// it by more than 2^3, so the stored weights are at most 2^8 (e4m3's largest finite value is 448),
// and the factor 2^5 keeps weights down to 2^-14 of the row's largest out of e4m3's flush-to-zero
// range.  The fp32 row sum l uses the same scaled weights, so the factor cancels in O / l and is
// taken out of L.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "fattn_internal.h"
#include "sm103a_ptx.cuh"

namespace fattn {
namespace {

constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kTiles = 2;
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleLog2 = 3.0f;
constexpr float kPScaleLog2 = 5.0f;
constexpr uint32_t kTmemCols = 512;
constexpr int kSlots = 8;  // K/V^T ring

struct F8Cfg {
  static constexpr int kQFull = 0;     // [2]
  static constexpr int kSFull = 2;     // [2]
  static constexpr int kPFull = 4;     // [2] one arrival per softmax warp
  static constexpr int kOFull = 6;     // [2]
  static constexpr int kQFree = 8;     // [2]
  static constexpr int kOFree = 10;    // [2] one arrival per softmax warp
  static constexpr int kDrain = 12;
  static constexpr int kKVFull = 13;   // [kSlots]
  static constexpr int kKVEmpty = 13 + kSlots;
  static constexpr int kNumBars = 13 + 2 * kSlots;
  __host__ __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + 128u * t; }
};
using C = F8Cfg;

// Shared memory of the head dimension D: two Q tiles, then the K/V^T ring, then the barriers.
template <int D>
struct F8Smem {
  static constexpr uint32_t kTileBytes = kBlockM * D;  // a Q or K tile (128 x D), or a V^T tile (D x 128)
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKVOff = kQOff + kTiles * kTileBytes;
  static constexpr uint32_t kBarOff = kKVOff + kSlots * kTileBytes;
  static constexpr uint32_t kMiscOff = kBarOff + C::kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;
  static_assert(kTileBytes % 1024 == 0, "tiles stay on 1024-byte swizzle-atom boundaries");
};

struct F8Args {
  __nv_bfloat16* o;
  float* lse;
  int BH, Nq, Nk;
  int wl, wr, off;
  int units_per_head, total_units;
  float c_log2;     // scale * q_descale * k_descale * log2(e)
  float v_descale;
  unsigned int* status;
  unsigned long long timeout_ns;
  int drop_kv_block;  // failure-detection testing only; -1 = off
};

// Key tiles [jb, je) that query tile [r0, r0 + 128) visits (empty past Nq or outside the band).
__device__ __forceinline__ void key_tiles(int r0, const F8Args& a, int& jb, int& je) {
  jb = je = 0;
  if (r0 >= a.Nq) return;
  const int r1 = min(r0 + kBlockM, a.Nq) - 1;
  const long long lo = a.wl >= 0 ? max(0LL, static_cast<long long>(r0) + a.off - a.wl) : 0LL;
  const long long hi = a.wr >= 0 ? min(static_cast<long long>(a.Nk) - 1, static_cast<long long>(r1) + a.off + a.wr)
                                 : static_cast<long long>(a.Nk) - 1;
  if (lo > hi) return;
  jb = static_cast<int>(lo / kBlockN);
  je = static_cast<int>(hi / kBlockN) + 1;
}

struct Unit {
  int bh, row0;
  int jb[2], je[2];
};
__device__ __forceinline__ int union_begin(const Unit& u) {
  int b = 0x7fffffff;
  for (int t = 0; t < kTiles; ++t)
    if (u.je[t] > u.jb[t]) b = min(b, u.jb[t]);
  return b;
}
__device__ __forceinline__ int union_end(const Unit& u) {
  int e = 0;
  for (int t = 0; t < kTiles; ++t)
    if (u.je[t] > u.jb[t]) e = max(e, u.je[t]);
  return e;
}

// The k-th unit (two adjacent query tiles of one head) of this CTA: rounds of gridDim.x units,
// heaviest first, every other round walked backwards.
__device__ __forceinline__ bool cta_unit(int k, const F8Args& a, Unit& u) {
  const int G = static_cast<int>(gridDim.x), cid = static_cast<int>(blockIdx.x);
  const long long idx = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - cid) : cid);
  if (idx >= a.total_units) return false;
  const int i = static_cast<int>(idx);
  u.bh = i % a.BH;
  u.row0 = (a.units_per_head - 1 - i / a.BH) * kTiles * kBlockM;
  key_tiles(u.row0, a, u.jb[0], u.je[0]);
  key_tiles(u.row0 + kBlockM, a, u.jb[1], u.je[1]);
  return true;
}

__device__ __forceinline__ void wait_dep(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
        "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
        "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])::"memory");
}

struct Abort {
  volatile uint32_t* flag;
  unsigned int* status;
  uint64_t deadline;
  __device__ void raise() const {
    *flag = 1u;
    atomicOr(status, kStatusTimeout);
  }
  __device__ void renew(unsigned long long timeout_ns) { deadline = globaltimer_ns() + timeout_ns; }
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Abort& ab) {
  bool ok = mbar_wait_bounded(bar, parity, ab.flag, ab.deadline);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) ab.raise();
  return ok;
}

__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, const Abort& ab) {
  const bool ok = mbar_wait_bounded(bar, parity, ab.flag, ab.deadline);
  if (!ok) ab.raise();
  return ok;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (o0, o1) = (a0, a1) * b + c
__device__ __forceinline__ void ffma2_bc(float& o0, float& o1, float a0, float a1, float b, float c) {
  asm("{\n\t.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\tmov.b64 z, {%5, %5};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(o0), "=f"(o1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

__device__ __forceinline__ void fadd2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y, w;\n\t"
      "mov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "add.rn.f32x2 w, x, y;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// Four fp32 weights rounded to e4m3 (round to nearest even, saturating at 448), lowest key in the
// lowest byte -- the order the tensor core reads an A operand from TMEM.
__device__ __forceinline__ uint32_t pack_e4m3x4(float e0, float e1, float e2, float e3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(e0), "f"(e1), "f"(e2), "f"(e3));
  return r;
}

// Instruction descriptor of kind::f8f6f4: fp32 D, e4m3 A and B (format code 0), both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((static_cast<uint32_t>(N) >> 3) << 17) | ((static_cast<uint32_t>(M) >> 4) << 24);
}

// Max of a row's 128 scores as a balanced tree of three-input maxes: 66 instructions, five deep (every
// step waits on it before its exponentials).
__device__ __forceinline__ float max128_tree(const uint32_t (&s)[4][32]) {
  auto at = [&](int e) { return __uint_as_float(s[e >> 5][e & 31]); };
  float a[43];
#pragma unroll
  for (int i = 0; i < 42; ++i) a[i] = max3f(at(3 * i), at(3 * i + 1), at(3 * i + 2));
  a[42] = fmaxf(at(126), at(127));
  float b[15];
#pragma unroll
  for (int i = 0; i < 14; ++i) b[i] = max3f(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
  b[14] = a[42];
  float c5[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) c5[i] = max3f(b[3 * i], b[3 * i + 1], b[3 * i + 2]);
  return fmaxf(max3f(c5[0], c5[1], c5[2]), fmaxf(c5[3], c5[4]));
}

// ------------------------------------------------------------------------------------------------
// Softmax group: one thread per query row.  g counts tile t's steps over the CTA's units (phases
// of S_full / P_full); done counts its non-empty units (phases of O_full / O_free).
// ------------------------------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ bool softmax_unit(int t, int jb, int n_tiles, int row0, int bh, uint32_t tmem,
                                             uint32_t sbar, const F8Args& a, const Abort& ab, int& g, int& done) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int q_row = row0 + t * kBlockM + quarter * 32 + lane;
  const long long c_row = static_cast<long long>(q_row) + a.off;
  const int hi = static_cast<int>(a.wr >= 0 ? min(c_row + a.wr, static_cast<long long>(a.Nk) - 1)
                                            : static_cast<long long>(a.Nk) - 1);
  const int lo = static_cast<int>(a.wl >= 0 ? max(c_row - a.wl, -1LL) : -1LL);
  const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = tmem + lane_field + C::col_s(t);
  const uint32_t tO = tmem + lane_field + C::col_o(t);
  const float c = a.c_log2;

  float m_ref = -INFINITY;  // exponent reference, log2 units
  float l = 0.f;            // sum of the stored-scale fp32 weights
  bool ok = true;
  for (int step = 0; step < n_tiles; ++step, ++g) {
    const int j = jb + step;
    if (!warp_wait(sbar + 8 * (C::kSFull + t), g & 1, ab)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t s[4][32];
    tmem_ld_32x32b_x128(tS, s);  // one load of the 128 columns (fewer than four 32-column loads)
#pragma unroll
    for (int h = 0; h < 4; ++h) wait_dep(s[h]);
    const int kv0 = j * kBlockN;
    if (__any_sync(0xffffffffu, kv0 + kBlockN - 1 > hi || kv0 < lo)) {
      // Keys outside this row's visible range, as offsets into the tile: one compare with an
      // immediate per key and side, and only the sides that cut into this tile for some row of the
      // warp (a causal diagonal tile or a band's upper edge: the upper side; a band's lower edge:
      // the lower side).
      const int vhi = hi - kv0, vlo = lo - kv0;
      const bool cut_lo = __any_sync(0xffffffffu, vlo > 0);
      const bool cut_hi = __any_sync(0xffffffffu, vhi < kBlockN - 1);
      if (!cut_lo) {
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * h + i > vhi) s[h][i] = __float_as_uint(-INFINITY);
      } else if (!cut_hi) {
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * h + i < vlo) s[h][i] = __float_as_uint(-INFINITY);
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * h + i > vhi || 32 * h + i < vlo) s[h][i] = __float_as_uint(-INFINITY);
      }
    }
    const float mx = max128_tree(s);
    const float m_new = fmaxf(m_ref, mx * c);
    const bool need = m_new > m_ref + kRescaleLog2;
    float corr = 1.f;
    if (need) {
      corr = ex2_approx(m_ref - m_new);  // 0 on the first tile
      m_ref = m_new;
      l *= corr;
    }
    // stored weight 2^(s c - m_ref + kPScaleLog2)
    const float nm = (m_ref == -INFINITY) ? 0.f : kPScaleLog2 - m_ref;
    uint32_t p[32];
    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float x0, x1, x2, x3;
        ffma2_bc(x0, x1, __uint_as_float(s[h][4 * i]), __uint_as_float(s[h][4 * i + 1]), c, nm);
        ffma2_bc(x2, x3, __uint_as_float(s[h][4 * i + 2]), __uint_as_float(s[h][4 * i + 3]), c, nm);
        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1), e2 = ex2_approx(x2), e3 = ex2_approx(x3);
        p[8 * h + i] = pack_e4m3x4(e0, e1, e2, e3);
        fadd2(ls[0], ls[1], e0, e1);
        fadd2(ls[2], ls[3], e2, e3);
      }
    }
    // P_t over the first 32 columns of S_t (already in registers); the next S_t is issued after
    // this tile's P V, which reads them.
    tmem_st_32x32b_x32(tS, p);
    l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
    if (step > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int h = 0; h < D / 32; ++h) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + 32 * h, o);
        wait_dep(o);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float y0, y1;
          ffma2_bc(y0, y1, __uint_as_float(o[i]), __uint_as_float(o[i + 1]), corr, 0.f);
          o[i] = __float_as_uint(y0);
          o[i + 1] = __float_as_uint(y1);
        }
        tmem_st_32x32b_x32(tO + 32 * h, o);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbar + 8 * (C::kPFull + t));
  }
  if (!ok) return false;
  const bool store =
      q_row < a.Nq && dbg_in(static_cast<long long>(bh) * a.Nq + q_row, static_cast<long long>(a.BH) * a.Nq);
  __nv_bfloat16* orow = a.o + (static_cast<size_t>(bh) * a.Nq + (store ? q_row : 0)) * D;
  if (n_tiles == 0) {
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      if (a.lse != nullptr) a.lse[static_cast<size_t>(bh) * a.Nq + q_row] = -INFINITY;
    }
    return true;
  }
  if (!warp_wait(sbar + 8 * (C::kOFull + t), done & 1, ab)) return false;
  tc_fence_after();
  const float f = l > 0.f ? a.v_descale / l : 0.f;
#pragma unroll
  for (int h = 0; h < D / 32; ++h) {
    uint32_t o[32];
    tmem_ld_32x32b_x32(tO + 32 * h, o);
    wait_dep(o);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * f, __uint_as_float(o[2 * i + 1]) * f);
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(orow + 32 * h);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(sbar + 8 * (C::kOFree + t));
  ++done;
  if (store && a.lse != nullptr)
    a.lse[static_cast<size_t>(bh) * a.Nq + q_row] =
        l > 0.f ? (m_ref - kPScaleLog2 + __log2f(l)) * 0.6931471805599453f : -INFINITY;
  return true;
}

template <int D>
__device__ __forceinline__ void softmax_role(int t, uint32_t tmem, uint32_t sbar, const F8Args& a, Abort ab) {
  int g = 0, done = 0;
  Unit u;
  for (int k = 0; cta_unit(k, a, u); ++k) {
    ab.renew(a.timeout_ns);
    if (!softmax_unit<D>(t, u.jb[t], u.je[t] - u.jb[t], u.row0, u.bh, tmem, sbar, a, ab, g, done)) return;
  }
}

// ------------------------------------------------------------------------------------------------
// TMA producer (one thread): Q tiles once per unit, then K_j and V_j^T through the ring.
// ------------------------------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tvt,
                                              uint32_t sbase, const F8Args& a, Abort ab) {
  using M = F8Smem<D>;
  const uint32_t sbar = sbase + M::kBarOff;
  tma_prefetch_desc(tq);
  tma_prefetch_desc(tk);
  tma_prefetch_desc(tvt);
  int ring = 0, issued = 0;
  int dropped = -1;  // ring index of the load skipped for failure-detection testing
  int qloads[2] = {0, 0};
  bool ok = true;
  Unit u;
  for (int k = 0; ok && cta_unit(k, a, u); ++k) {
    ab.renew(a.timeout_ns);
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      if (u.je[t] == u.jb[t]) continue;
      if (qloads[t] > 0 && !thread_wait(sbar + 8 * (C::kQFree + t), (qloads[t] - 1) & 1, ab)) {
        ok = false;
        break;
      }
      const uint32_t bar = sbar + 8 * (C::kQFull + t);
      mbar_arrive_expect_tx(bar, M::kTileBytes);
      tma_load_3d(sbase + M::kQOff + t * M::kTileBytes, tq, bar, 0, u.row0 + t * kBlockM, u.bh);
      ++qloads[t];
    }
    if (!ok) break;
    const int J0 = union_begin(u), J1 = union_end(u);
    for (int j = J0; j < J1 && ok; ++j) {
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const int idx = ring + 2 * (j - J0) + w;
        const int slot = idx % kSlots, round = idx / kSlots;
        if (round > 0 && !thread_wait(sbar + 8 * (C::kKVEmpty + slot), (round - 1) & 1, ab)) {
          ok = false;
          break;
        }
        if (w == 0 && j == a.drop_kv_block) {  // testing only: this tile never arrives
          dropped = idx;
          issued = idx + 1;
          continue;
        }
        const uint32_t bar = sbar + 8 * (C::kKVFull + slot);
        mbar_arrive_expect_tx(bar, M::kTileBytes);
        const uint32_t dst = sbase + M::kKVOff + slot * M::kTileBytes;
        if (w == 0) tma_load_3d(dst, tk, bar, 0, j * kBlockN, u.bh);   // K_j: 128 keys x d
        else tma_load_3d(dst, tvt, bar, j * kBlockN, 0, u.bh);         // V_j^T: d rows x 128 keys
        issued = idx + 1;
      }
    }
    if (J1 > J0) ring += 2 * (J1 - J0);
  }
  if (!ok) {
    const uint64_t until = globaltimer_ns() + 50ull * 1000 * 1000;
    volatile uint32_t never = 0;
    for (int idx = max(0, issued - kSlots); idx < issued; ++idx)
      if (idx != dropped)
        mbar_wait_bounded(sbar + 8 * (C::kKVFull + idx % kSlots), (idx / kSlots) & 1, &never, until);
#pragma unroll
    for (int t = 0; t < kTiles; ++t)
      if (qloads[t] > 0) mbar_wait_bounded(sbar + 8 * (C::kQFull + t), (qloads[t] - 1) & 1, &never, until);
  }
}

// ------------------------------------------------------------------------------------------------
// MMA issuer: the whole warp runs the schedule, one elected lane issues.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate, uint32_t lead) {
  FATTN_DBG_SKIP_IF(dbg_mma_d(d_tmem, idesc));
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(lead)
      : "memory");
}
__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate, uint32_t lead) {
  FATTN_DBG_SKIP_IF(dbg_mma_d(d_tmem, idesc) | ((a_tmem & 0xFFFFu) + 8u > kTmemColumns ? kDbgTmemCol : 0u));
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(lead)
      : "memory");
}

// K-major descriptor of a Q or K tile (128 rows of D bytes): 128-byte swizzle with 1024-byte atoms
// for D = 128, 64-byte swizzle with 512-byte atoms for D = 64.
template <int D>
__device__ __forceinline__ uint64_t qk_desc(uint32_t addr) {
  if constexpr (D == 128) return smem_desc_sw128(addr, 16, 1024);
  else return smem_desc_sw64(addr);
}

template <int D>
struct MmaCtx {
  using M = F8Smem<D>;
  uint32_t tmem, sbar, lead;
  uint64_t dq[kTiles], dk0, dv0;
  __device__ __forceinline__ void init(uint32_t tmem_, uint32_t sbase) {
    tmem = tmem_;
    sbar = sbase + M::kBarOff;
#pragma unroll
    for (int t = 0; t < kTiles; ++t) dq[t] = qk_desc<D>(sbase + M::kQOff + t * M::kTileBytes);
    dk0 = qk_desc<D>(sbase + M::kKVOff);
    dv0 = smem_desc_sw128(sbase + M::kKVOff, 16, 1024);
    lead = elect_lane();
  }
  __device__ __forceinline__ static uint64_t slot_adv(int slot) {
    return static_cast<uint64_t>(slot) * (M::kTileBytes >> 4);
  }
  // S_t = Q_t K^T: D / 32 K steps of 32 e4m3 (32 bytes) along d
  __device__ __forceinline__ void issue_s(int t, int slot) const {
    constexpr uint32_t id = idesc_e4m3(kBlockM, kBlockN);
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk)
      mma_f8_ss(tmem + C::col_s(t), dq[t] + 2 * kk, dk0 + slot_adv(slot) + 2 * kk, id, kk > 0 ? 1u : 0u, lead);
  }
  // O_t += P_t V: four K steps of 32 keys; P_t's 32 keys of a step are 8 TMEM columns
  __device__ __forceinline__ void issue_pv(int t, int slot, bool first) const {
    constexpr uint32_t id = idesc_e4m3(kBlockM, D);
#pragma unroll
    for (int kk = 0; kk < kBlockN / 32; ++kk)
      mma_f8_ts(tmem + C::col_o(t), tmem + C::col_s(t) + 8 * kk, dv0 + slot_adv(slot) + 2 * kk, id,
                (!first || kk > 0) ? 1u : 0u, lead);
  }
  __device__ __forceinline__ void commit(int bar) const { mma_commit_lead(sbar + 8 * bar, lead); }
  __device__ __forceinline__ bool wait(int bar, int parity, const Abort& ab) const {
    return warp_wait(sbar + 8 * bar, parity & 1, ab);
  }
};

struct MmaState {
  int ring = 0;
  int s_issued[2] = {0, 0};
  int p_seen[2] = {0, 0};
  int units[2] = {0, 0};
  int q_seen[2] = {0, 0};
};

// Unit schedule: for j = J0 .. J1, first P_t(j-1) V_{j-1}, then S_t(j), per tile; K_j's slot is
// released after the S(j), V_{j-1}'s after the P V(j-1).  Ring index of K_j is ring + 2 (j - J0).
template <int D>
__device__ __forceinline__ bool mma_unit(const Unit& u, const MmaCtx<D>& m, MmaState& st, const Abort& ab) {
  const int J0 = union_begin(u), J1 = union_end(u);
  if (J0 >= J1) return true;
  auto active = [&](int t, int j) { return u.jb[t] <= j && j < u.je[t]; };
  const int r0 = st.ring;
  for (int j = J0; j <= J1; ++j) {
    const int r = r0 + 2 * (j - J0);
    if (j < J1 && !m.wait(C::kKVFull + r % kSlots, r / kSlots, ab)) return false;
    if (j > J0 && !m.wait(C::kKVFull + (r - 1) % kSlots, (r - 1) / kSlots, ab)) return false;
    tc_fence_after();
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      if (j > J0 && active(t, j - 1)) {
        const bool first = (j - 1 == u.jb[t]);
        if (!m.wait(C::kPFull + t, st.p_seen[t]++, ab)) return false;
        if (first && st.units[t] > 0 && !m.wait(C::kOFree + t, st.units[t] - 1, ab)) return false;
        tc_fence_after();
        m.issue_pv(t, (r - 1) % kSlots, first);
        if (j - 1 == u.je[t] - 1) {
          m.commit(C::kOFull + t);
          ++st.units[t];
        }
      }
      if (j < J1 && active(t, j)) {
        m.issue_s(t, r % kSlots);
        m.commit(C::kSFull + t);
        if (j == u.je[t] - 1) m.commit(C::kQFree + t);
        ++st.s_issued[t];
      }
    }
    if (j < J1) m.commit(C::kKVEmpty + r % kSlots);
    if (j > J0) m.commit(C::kKVEmpty + (r - 1) % kSlots);
  }
  st.ring = r0 + 2 * (J1 - J0);
  return true;
}

template <int D>
__device__ __forceinline__ void mma_role(uint32_t tmem, uint32_t sbase, const F8Args& a, Abort ab) {
  MmaCtx<D> m;
  m.init(tmem, sbase);
  MmaState st;
  bool ok = true;
  Unit u;
  for (int k = 0; ok && cta_unit(k, a, u); ++k) {
    ab.renew(a.timeout_ns);
#pragma unroll
    for (int t = 0; t < kTiles; ++t)
      if (u.je[t] > u.jb[t] && ok) ok = m.wait(C::kQFull + t, st.q_seen[t]++, ab);
    if (ok) ok = mma_unit(u, m, st, ab);
  }
  m.commit(C::kDrain);
  volatile uint32_t never = 0;
  const uint64_t until = ok ? ab.deadline : globaltimer_ns() + 50ull * 1000 * 1000;
  mbar_wait_bounded(m.sbar + 8 * C::kDrain, 0, &never, until);
  __syncwarp();
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_vt, const F8Args a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  using M = F8Smem<D>;
  const uint32_t sbar = sbase + M::kBarOff;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + M::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + M::kMiscOff + 4);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(sbar + 8 * (C::kQFull + t), 1);
      mbar_init(sbar + 8 * (C::kSFull + t), 1);
      mbar_init(sbar + 8 * (C::kPFull + t), kBlockM / 32);
      mbar_init(sbar + 8 * (C::kOFull + t), 1);
      mbar_init(sbar + 8 * (C::kQFree + t), 1);
      mbar_init(sbar + 8 * (C::kOFree + t), kBlockM / 32);
    }
    mbar_init(sbar + 8 * C::kDrain, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(sbar + 8 * (C::kKVFull + s), 1);
      mbar_init(sbar + 8 * (C::kKVEmpty + s), 1);
    }
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  Abort ab{abort_flag, a.status, globaltimer_ns() + a.timeout_ns};
  if (warp < 8) {
    softmax_role<D>(warp >> 2, tmem, sbar, a, ab);
  } else if (warp == kProducerWarp) {
    if ((threadIdx.x & 31) == 0) producer_role<D>(&tm_q, &tm_k, &tm_vt, sbase, a, ab);
    __syncwarp();
  } else {
    mma_role<D>(tmem, sbase, a, ab);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// V [BH][Nk][D] -> V^T [BH][D][Nk_pad] (e4m3 bytes), keys Nk .. Nk_pad - 1 written as zero.
// One block of 2 D threads per (128-key tile, head): the tile is read with 16-byte loads into shared
// memory; thread (key block kb of 16 keys, word w = 4 d values) reads its 16 words (conflict-free:
// the D / 4 words of a row, and for D = 64 two rows 16 banks apart, per warp), transposes four 4 x 4
// byte blocks with byte permutes, and writes 16 keys of each of its 4 d rows as one 16-byte store.
template <int D>
__global__ void __launch_bounds__(2 * D) fwd_fp8_vt_kernel(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt,
                                                           int Nk, int Nk_pad) {
  constexpr int kWords = D / 4;                // 32-bit words of a key row
  __shared__ uint32_t tile[128][kWords + 1];  // [key][d / 4], padded
  const int kt = blockIdx.x, bh = blockIdx.y;
  const int key0 = kt * 128;
  const uint8_t* src = v + static_cast<size_t>(bh) * Nk * D;
  for (int i = threadIdx.x; i < 128 * (D / 16); i += 2 * D) {
    const int key = i / (D / 16), c = i % (D / 16);  // 16-byte chunk c of row key
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (key0 + key < Nk) w = reinterpret_cast<const uint4*>(src + static_cast<size_t>(key0 + key) * D)[c];
    tile[key][4 * c] = w.x;
    tile[key][4 * c + 1] = w.y;
    tile[key][4 * c + 2] = w.z;
    tile[key][4 * c + 3] = w.w;
  }
  __syncthreads();
  const int w = threadIdx.x % kWords, kb = threadIdx.x / kWords;  // d values 4w .. 4w + 3, keys 16kb .. 16kb + 15
  if (key0 + 16 * kb >= Nk_pad) return;
  uint32_t out[4][4];  // [d row r][word: 4 keys]
#pragma unroll
  for (int b4 = 0; b4 < 4; ++b4) {
    const uint32_t a0 = tile[16 * kb + 4 * b4][w], a1 = tile[16 * kb + 4 * b4 + 1][w];
    const uint32_t a2 = tile[16 * kb + 4 * b4 + 2][w], a3 = tile[16 * kb + 4 * b4 + 3][w];
    const uint32_t t0 = __byte_perm(a0, a1, 0x5140), t1 = __byte_perm(a0, a1, 0x7362);
    const uint32_t t2 = __byte_perm(a2, a3, 0x5140), t3 = __byte_perm(a2, a3, 0x7362);
    out[0][b4] = __byte_perm(t0, t2, 0x5410);
    out[1][b4] = __byte_perm(t0, t2, 0x7632);
    out[2][b4] = __byte_perm(t1, t3, 0x5410);
    out[3][b4] = __byte_perm(t1, t3, 0x7632);
  }
  uint8_t* dst = vt + static_cast<size_t>(bh) * D * Nk_pad + key0 + 16 * kb;
#pragma unroll
  for (int r = 0; r < 4; ++r)
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(4 * w + r) * Nk_pad) =
        make_uint4(out[r][0], out[r][1], out[r][2], out[r][3]);
}

}  // namespace

int fp8_padded_keys(int Nk) { return (Nk + 15) / 16 * 16; }

cudaError_t launch_vt_transpose(const void* v, void* vt, int BH, int Nk, int d, cudaStream_t stream) {
  const int Nk_pad = fp8_padded_keys(Nk);
  dim3 grid(static_cast<unsigned int>((Nk_pad + 127) / 128), static_cast<unsigned int>(BH));
  const uint8_t* src = static_cast<const uint8_t*>(v);
  uint8_t* dst = static_cast<uint8_t*>(vt);
  if (d == 128) fwd_fp8_vt_kernel<128><<<grid, 256, 0, stream>>>(src, dst, Nk, Nk_pad);
  else if (d == 64) fwd_fp8_vt_kernel<64><<<grid, 128, 0, stream>>>(src, dst, Nk, Nk_pad);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

namespace {
template <int D>
cudaError_t launch_fp8_d(const F8Args& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                         cudaStream_t stream) {
  static bool attr_set[64] = {};
  static int sm_count[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_fp8_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(F8Smem<D>::kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (sm_count[dev] == 0) {
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  const unsigned int grid = static_cast<unsigned int>(min(a.total_units, sm_count[dev]));
  prefill_fp8_kernel<D><<<grid, kThreads, F8Smem<D>::kSmemBytes, stream>>>(tq, tk, tvt, a);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_prefill_fp8(const Fp8Problem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tvt, unsigned int* status, unsigned long long timeout_ns,
                               cudaStream_t stream) {
  F8Args a;
  a.o = static_cast<__nv_bfloat16*>(p.o);
  a.lse = p.lse;
  a.BH = p.B * p.H;
  a.Nq = p.Nq;
  a.Nk = p.Nk;
  a.wl = p.window_left;
  a.wr = p.window_right;
  a.off = p.Nk - p.Nq;
  a.units_per_head = (p.Nq + kTiles * kBlockM - 1) / (kTiles * kBlockM);
  a.total_units = a.units_per_head * a.BH;
  a.c_log2 = p.scale * p.q_descale * p.k_descale * 1.4426950408889634f;
  a.v_descale = p.v_descale;
  a.status = status;
  a.timeout_ns = timeout_ns;
  a.drop_kv_block = p.drop_kv_block;
  if (p.d == 128) return launch_fp8_d<128>(a, tq, tk, tvt, stream);
  if (p.d == 64) return launch_fp8_d<64>(a, tq, tk, tvt, stream);
  return cudaErrorInvalidValue;
}

// Debug builds: read (and optionally clear) this file's device-side check record.
FATTN_DEBUG_ACCESSOR(fp8)

}  // namespace fattn
