// backward_sm103a.cu -- attention backward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes is the FlashAttention-2 backward pass ("Flash Attention: The Hidden Gem",
// Phase 2).  Given Q, K, V, the forward's L (log-sum-exp per query row) and O, and the upstream
// gradient dO:
//   D   = rowsum(dO o O)                              (The D Shortcut)
//   P   = exp(scale * Q K^T - L)                      (recomputed from L, The Algorithm step 11)
//   dV  = P^T dO,  dP = dO V^T                        (Chain Rule Through a Matrix Multiply)
//   dS  = P o (dP - D)                                (The Softmax Jacobian)
//   dQ  = scale * dS K,  dK = scale * dS^T Q          (the scale comes from S = scale * Q K^T)
// with the key/value tile in the outer loop and query tiles in the inner loop (step 5): dK_j and
// dV_j stay in tensor memory for the whole inner loop and are written once; dQ_i is accumulated in
// an fp32 array in device memory by every key tile that sees it.
//
// Three kernels run in stream order:
//   bwd_prep_kernel  per query row, -L_i / scale and -D_i, each split into three bf16 terms (see
//                    below), into a padded workspace; rows past Nq get -inf and 0 so that their P is
//                    exactly 0; zeroes the dQ array
//   bwd_kernel       one CTA per (head, 128-key tile); walks the query tiles that can see its keys
//   bwd_dq_kernel    dQ = scale * accumulated array, rounded to bf16
//
// bwd_kernel works on transposed tiles so that one thread owns one key: S^T = K Q^T and
// dP^T = V dO^T land in tensor memory with keys on the 128 lanes and the 128 queries of the tile
// along the columns.  Thread layout (480 threads):
//   warps 0-7    compute: warp w reads lanes 32*(w%4).. and the query half w/4 of S^T and dP^T,
//                forms P^T = exp2(S^T * scale*log2e - L*log2e) and dS^T = P^T o (dP^T - D), writes
//                P^T (bf16) back into tensor memory and dS^T (bf16) into shared memory
//   warp  8      TMA producer: K_j and V_j once, then Q_i, dO_i, -L_i*log2e, -D_i per query tile
//   warp  9      MMA issuer (dP^T, dV, dK, dQ; with d = 128 also S^T) and tensor-memory owner
//   warps 10-13  dQ drain: one thread per query row reads dQ_i from tensor memory, stages it in
//                shared memory and adds it into the fp32 array with a TMA reduce
//   warp  14     (d = 64) issues S^T = K Q_i^T for every tile as soon as its buffer is free, so the
//                main MMA warp never waits for the dQ drain
// The five products per query tile are tcgen05.mma with M = 128:
//   S^T  = K Q^T        A = K (K-major)          B = Q (K-major)
//   dP^T = V dO^T       A = V (K-major)          B = dO (K-major)
//   dV  += P^T dO       A = P^T in TMEM          B = dO read MN-major
//   dK  += dS^T Q       A = dS^T (K-major)       B = Q read MN-major
//   dQ   = dS K         A = dS^T read MN-major   B = K read MN-major
// so one shared-memory copy of dS^T serves both of its products.
//
// The per-query terms enter through the tensor core, not through shared-memory loads in the compute
// warps: S^T and dP^T get one more K step of 16 columns whose A side is a constant block of ones and
// whose B side holds, per query, the three bf16 terms of -L_i / scale (for S) or -D_i (for dP), each
// halved and written into both 8-column halves of the step.  The products come out as
// S'^T = S^T - L / scale and dP'^T = dP^T - D, so the compute warps form P^T = exp2(S'^T * scale *
// log2(e)) and dS^T = P^T o dP'^T with one multiply each.  Three bf16 terms carry an fp32 value to
// within 2^-24 of its magnitude; halving is exact.
//
// Tensor memory (512 columns):
//   d = 64:  S^T buffers at 0 and 128 (two query tiles in flight), dP^T at 256, dV at 384, dK at
//            448.  After the compute warps have read S^T they overwrite it with P^T packed as bf16
//            pairs: queries 0-63 in columns 0-31, queries 64-127 in columns 96-127.  Columns 32-95
//            are then free and receive dQ_i (64 fp32 columns).
//   d = 128: one S^T buffer at 0, dP^T at 128, dV at 256, dK at 384; dQ_i (128 columns) goes to
//            the dP^T columns once the compute warps have read them.  The next tile's dP^T is then
//            computed in two 64-query halves (N = 64), each as soon as the drain warps have read
//            the 64 dQ columns under it, and the compute warps form P^T from S^T before they wait
//            for their half of dP^T, so that the exponentials overlap the drain.
#include <cuda_bf16.h>
#include <math.h>

#include "fattn_internal.h"
#include "sm103a_ptx.cuh"

namespace fattn {
namespace {

constexpr int kBM = 128;  // queries per inner step (columns of S^T)
constexpr int kBN = 128;  // keys per CTA (TMEM lanes)
constexpr int kThreads = 480;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kDrainWarp0 = 10;
constexpr int kSWarp = 14;  // issues the S^T products (d = 64)
constexpr int kDrainBarrier = 1;  // named barrier id of the four drain warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAtom = 128 * 128;  // 128 rows x 128 bytes: one swizzled 64-column chunk of a tile
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BCfg {
  static constexpr bool kTwoS = (D == 64);
  static constexpr int kSBufs = kTwoS ? 2 : 1;
  // Q_i and dO_i buffers: d = 64 two Q and three dO (the dO reload is on the path to the next dP^T),
  // d = 128 one of each.
  static constexpr int kQStages = kTwoS ? 2 : 1;
  static constexpr int kOStages = kTwoS ? 3 : 1;
  static constexpr int kDSBufs = 1;               // dS^T buffers
  static constexpr int kChunks = D / 64;
  static constexpr uint32_t kTile = kBM * D * 2;  // one 128-row bf16 tile of Q, K, V or dO
  static constexpr uint32_t kKOff = 0;
  static constexpr uint32_t kVOff = kTile;
  static constexpr uint32_t kStageOff = 2 * kTile;  // Q stages, then dO stages
  __host__ __device__ static constexpr uint32_t q_off(int st) { return kStageOff + static_cast<uint32_t>(st) * kTile; }
  __host__ __device__ static constexpr uint32_t do_off(int st) {
    return kStageOff + static_cast<uint32_t>(kQStages + st) * kTile;
  }
  static constexpr uint32_t kDSBytes = kBN * kBM * 2;
  static constexpr uint32_t kDSOff = kStageOff + (kQStages + kOStages) * kTile;
  static constexpr uint32_t kDQOff = kDSOff + kDSBufs * kDSBytes;  // 64 columns of dQ at a time
  static constexpr uint32_t kDQBytes = kBM * 64 * 4;
  static constexpr uint32_t kOnesOff = kDQOff + kDQBytes;  // [128 rows][16] bf16 of the constant A block
  static constexpr uint32_t kExtBytes = kBM * 32;             // [128 rows][16] bf16
  static constexpr uint32_t kExtOff = kOnesOff + kExtBytes;   // Q terms per Q stage, then dO terms per dO stage
  __host__ __device__ static constexpr uint32_t ext_q_off(int st) { return kExtOff + static_cast<uint32_t>(st) * kExtBytes; }
  __host__ __device__ static constexpr uint32_t ext_do_off(int st) {
    return kExtOff + static_cast<uint32_t>(kQStages + st) * kExtBytes;
  }
  static constexpr uint32_t kBarOff = kExtOff + (kQStages + kOStages) * kExtBytes;
  // barrier indices
  static_assert(kQStages <= 4 && kOStages <= 4, "barrier slots");
  static constexpr int kKVFull = 0;
  static constexpr int kQFull = 1;     // [kQStages] Q_i and its extra K-step block landed
  static constexpr int kOFull = 5;     // [kOStages] dO_i and its extra K-step block landed
  static constexpr int kQEmpty = 9;    // [kQStages] Q_i's last reader (dK_i) done
  static constexpr int kOEmpty = 13;   // [kOStages] dO_i's last reader (dV_i) done
  static constexpr int kSFull = 17;    // [2] S^T of a buffer computed
  static constexpr int kDPFull = 19;   // dP^T computed
  static constexpr int kCDone = 20;    // compute warps done with a tile (one arrival per warp)
  static constexpr int kDSEmpty = 21;  // [2] dK_i and dQ_i have read a dS^T buffer
  static constexpr int kDQFull = 23;   // [2] dQ_i in tensor memory
  static constexpr int kDQFree = 25;   // [2] dQ_i read out of tensor memory (one arrival per drain warp)
  static constexpr int kAccDone = 27;  // every MMA of the CTA done: dK, dV final
  static constexpr int kDrain = 28;
  static constexpr int kDPFree = 29;   // compute warps have read dP^T (one arrival per warp)
  static constexpr int kDrainS = 30;
  static constexpr int kDPFullB = 31;  // d = 128: dP^T of queries 64-127 computed (kDPFull: queries 0-63)
  static constexpr int kNumBars = 32;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kMiscOff + 16 + 1024;  // + slack to align the base
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // tensor-memory columns
  __host__ __device__ static constexpr uint32_t col_s(int b) { return 128u * b; }
  static constexpr uint32_t kColDP = kTwoS ? 256u : 128u;
  static constexpr uint32_t kColDV = kTwoS ? 384u : 256u;
  static constexpr uint32_t kColDK = kTwoS ? 448u : 384u;
  __host__ __device__ static constexpr uint32_t col_dq(int b) { return kTwoS ? col_s(b) + 32u : kColDP; }
};

// Packed P^T columns: queries [64h + 32c, 64h + 32c + 32) of a tile go to 16 columns at this
// offset from the S^T buffer.  Each compute warp only overwrites columns it has already read.
__host__ __device__ constexpr uint32_t p_col(int half, int chunk) {
  return half ? 96u + 16u * chunk : 16u * chunk;
}
// ... and 16 queries (K step kk of dV += P^T dO) start at this column.
__host__ __device__ constexpr uint32_t p_step_col(int kk) { return kk < 4 ? 8u * kk : 96u + 8u * (kk - 4); }

constexpr long long kL2GroupBytes = 64ll << 20;

struct BArgs {
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const __nv_bfloat16* ext_q;   // [BH][Nq_pad][16]  terms of -L / scale
  const __nv_bfloat16* ext_do;  // [BH][Nq_pad][16]  terms of -D
  int BH, Nq, Nk, Nq_pad, NqT;
  int wl, wr, off;  // mask band: key j visible to query i iff i+off-wl <= j <= i+off+wr (-1 = unbounded)
  float c_log2;  // scale * log2(e)
  float scale;
  unsigned int* status;
  unsigned long long timeout_ns;
  int drop_kv;  // failure-detection testing only: K_j and V_j are never loaded
  int nkt;      // key tiles per head
  int group;    // heads per CTA group (1 .. BH)
  // Element mask (masked instantiation only), laid out as for the forward: bit j & 31 of word j >> 5
  // of query row i of head (b, h) at mask + b * mask_sb + h * mask_sh + i * mask_words, set = visible.
  // Its summary by key tile: for key tile j of head (b, h), at tiles + b * tiles_sb + h * tiles_sh +
  // j * 2 * tiles_w, tiles_w 64-bit words with bit i & 63 of word i >> 6 set when query tile i sees
  // a key of the tile, then tiles_w words with the bit set when some of those keys are hidden from it.
  int H;
  const uint32_t* mask;
  long long mask_sb, mask_sh;
  int mask_words;
  const unsigned long long* tiles;
  long long tiles_sb, tiles_sh;
  int tiles_w;
};

// Under an element mask: the summary words of key tile jt of head bh.
__device__ __forceinline__ const unsigned long long* key_tile_bits(const BArgs& a, int bh, int jt) {
  return a.tiles + (bh / a.H) * a.tiles_sb + (bh % a.H) * a.tiles_sh + static_cast<long long>(jt) * 2 * a.tiles_w;
}

// Under an element mask, whether query tile qt sees some but not all of the key tile's keys.
__device__ __forceinline__ bool partly_hidden(const BArgs& a, const unsigned long long* bits, int qt) {
  return (__ldg(bits + a.tiles_w + (qt >> 6)) >> (qt & 63)) & 1ull;
}

// The query tile after qt (from it0 - 1 on) that this key tile computes: every one without a mask,
// the ones the mask does not hide entirely with one (the next set bit of the key tile's live words).
template <bool M>
__device__ __forceinline__ int next_qtile(const BArgs& a, const unsigned long long* bits, int qt) {
  ++qt;
  if constexpr (M) {
    while ((qt >> 6) < a.tiles_w) {
      const unsigned long long rest = __ldg(bits + (qt >> 6)) >> (qt & 63);
      if (rest != 0ull) return qt + __ffsll(static_cast<long long>(rest)) - 1;
      qt = (qt | 63) + 1;
    }
  }
  return qt;
}

struct Abort {
  volatile uint32_t* flag;
  unsigned int* status;
  uint64_t deadline;
  __device__ void raise() const {
    *flag = 1u;
    atomicOr(status, kStatusTimeout);
  }
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

__device__ __forceinline__ void wait_dep(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
        "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
        "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])::"memory");
}

// (o0, o1) = (a0, a1) * (b0, b1)
__device__ __forceinline__ void fmul2(float& o0, float& o1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y, w;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 w, x, y;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(o0), "=f"(o1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// ------------------------------------------------------------------------------------------------
// Compute warps: one thread per key; each warp covers 64 of the tile's 128 queries.
// ------------------------------------------------------------------------------------------------
template <int D, bool M>
__device__ __forceinline__ void compute_role(int n, int it0, int n0, int bh, uint32_t tmem, uint32_t sbase,
                                             const uint8_t* smem, const BArgs& a, const Abort& ab) {
  using C = BCfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int kr = quarter * 32 + lane;  // key row within the tile = TMEM lane
  const int kidx = n0 + kr;
  const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t sbar = sbase + C::kBarOff;
  const float c = a.c_log2;
  bool ok = true;
  int qt = it0 - 1;  // element mask: the query tile of step i
  const unsigned long long* bits = M ? key_tile_bits(a, bh, n0 / kBN) : nullptr;
  for (int i = 0; i < n; ++i) {
    const int b = i % C::kSBufs;
    const int dsb = i % C::kDSBufs;
    if constexpr (M) qt = next_qtile<M>(a, bits, qt);
    if (!warp_wait(sbar + 8 * (C::kSFull + b), (i / C::kSBufs) & 1, ab) ||
        (C::kTwoS && !warp_wait(sbar + 8 * C::kDPFull, i & 1, ab)) ||
        (!C::kTwoS && i >= C::kDSBufs && !warp_wait(sbar + 8 * (C::kDSEmpty + dsb), ((i / C::kDSBufs) - 1) & 1, ab))) {
      ok = false;
      break;
    }
    tc_fence_after();
    const int q0 = (M ? qt : it0 + i) * kBM;
    const bool partial = M && partly_hidden(a, bits, qt);  // the same for the whole tile
    const uint32_t tS = tmem + lane_field + C::col_s(b);
    const uint32_t tDP = tmem + lane_field + C::kColDP;
    const uint32_t ds_row = sbase + C::kDSOff + dsb * C::kDSBytes + half * kAtom + kr * 128;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int ch = half ? 1 - cc : cc;  // the upper half writes its packed P^T over chunk 1 first
      const int qa = 64 * half + 32 * ch;
      uint32_t s[32], dp[32];
      tmem_ld_32x32b_x32(tS + qa, s);
      if constexpr (C::kTwoS) tmem_ld_32x32b_x32(tDP + qa, dp);
      wait_dep(s);
      if constexpr (C::kTwoS) wait_dep(dp);
      if (C::kTwoS && cc == 1) {
        // dP^T is in registers: the next tile's dP^T may be computed into the same columns.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sbar + 8 * C::kDPFree);
      }
      // s = S'^T = S^T - L / scale and dp = dP'^T = dP^T - D for queries [q0 + qa, q0 + qa + 32).
      // Key kidx is visible to query q iff kidx - off - wr <= q <= kidx - off + wl: elements e of
      // this chunk outside [e_lo, e_hi] are masked.
      const int e_lo = a.wr >= 0 ? kidx - a.off - a.wr - (q0 + qa) : -1;
      const int e_hi = a.wl >= 0 ? kidx - a.off + a.wl - (q0 + qa) : 32;
      const bool mask = __any_sync(0xffffffffu, e_lo > 0 || e_hi < 31);
      // Element mask on a partly hidden tile: lane e loads the word of query q0 + qa + e that holds
      // this warp's 32 keys, and 32 ballots turn those rows into columns, so that bit e of `vis` says
      // whether this thread's key is visible to query q0 + qa + e.
      uint32_t vis = ~0u;
      if constexpr (M) {
        if (partial) {
          const int qrow = q0 + qa + lane;
          const uint32_t word = qrow < a.Nq ? __ldg(a.mask + (bh / a.H) * a.mask_sb + (bh % a.H) * a.mask_sh +
                                                        static_cast<long long>(qrow) * a.mask_words + (kidx >> 5))
                                            : 0u;
#pragma unroll
          for (int kb = 0; kb < 32; ++kb) {
            const uint32_t col = __ballot_sync(0xffffffffu, (word >> kb) & 1u);
            if (lane == kb) vis = col;
          }
        }
      }
      uint32_t pp[16], pd[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float x0, x1;
        fmul2(x0, x1, __uint_as_float(s[e]), __uint_as_float(s[e + 1]), c, c);
        float p0 = ex2_approx(x0);
        float p1 = ex2_approx(x1);
        if (mask) {
          p0 = (e < e_lo || e > e_hi) ? 0.f : p0;
          p1 = (e + 1 < e_lo || e + 1 > e_hi) ? 0.f : p1;
        }
        if constexpr (M) {
          if (partial) {
            p0 = ((vis >> e) & 1u) ? p0 : 0.f;
            p1 = ((vis >> (e + 1)) & 1u) ? p1 : 0.f;
          }
        }
        pp[e >> 1] = pack_bf16x2(p0, p1);
        if constexpr (C::kTwoS) {
          float d0, d1;
          fmul2(d0, d1, p0, p1, __uint_as_float(dp[e]), __uint_as_float(dp[e + 1]));
          pd[e >> 1] = pack_bf16x2(d0, d1);
        } else {
          s[e] = __float_as_uint(p0);
          s[e + 1] = __float_as_uint(p1);
        }
      }
      tmem_st_32x32b_x16(tS + p_col(half, ch), pp);
      if constexpr (!C::kTwoS) {
        // d = 128: P of this chunk is done; its dS needs this query half's dP^T, which the MMA warp
        // issues once the drain warps have read the dQ columns under it.
        if (cc == 0) {
          if (!warp_wait(sbar + 8 * (half ? C::kDPFullB : C::kDPFull), i & 1, ab)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        tmem_ld_32x32b_x32(tDP + qa, dp);
        wait_dep(dp);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float d0, d1;
          fmul2(d0, d1, __uint_as_float(s[e]), __uint_as_float(s[e + 1]), __uint_as_float(dp[e]),
                __uint_as_float(dp[e + 1]));
          pd[e >> 1] = pack_bf16x2(d0, d1);
        }
      }
      // The dS^T buffer is free once the previous user's dK and dQ products have read it.  At d = 64
      // waiting here rather than at the top of the tile overlaps the first chunk's loads and
      // exponentials with those products (8.7 % faster); at d = 128 the next S^T and dP^T are issued
      // after dQ anyway, and the wait stays at the top (1.7 % faster there).
      if (C::kTwoS && cc == 0 && i >= C::kDSBufs &&
          !warp_wait(sbar + 8 * (C::kDSEmpty + dsb), ((i / C::kDSBufs) - 1) & 1, ab)) {
        ok = false;
        break;
      }
      // dS^T row kr, queries [qa, qa + 32): 16-byte units 4*ch .. 4*ch + 3 of this half's 128-byte
      // row, 128-byte swizzled like a TMA tile.
#pragma unroll
      for (int u = 0; u < 4; ++u)
        st_shared_v4(ds_row + ((static_cast<uint32_t>(4 * ch + u) ^ static_cast<uint32_t>(kr & 7)) << 4),
                     pd[4 * u], pd[4 * u + 1], pd[4 * u + 2], pd[4 * u + 3]);
    }
    tmem_wait_st();
    if (!ok) break;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbar + 8 * C::kCDone);
  }
  if (!ok) return;

  // Epilogue: dV and scale * dK rows of this warp's keys, this warp's half of the columns.
  if (!warp_wait(sbar + 8 * C::kAccDone, 0, ab)) return;
  tc_fence_after();
  const bool store =
      kidx < a.Nk && dbg_in(static_cast<long long>(bh) * a.Nk + kidx, static_cast<long long>(a.BH) * a.Nk);
  const size_t row = (static_cast<size_t>(bh) * a.Nk + (store ? kidx : 0)) * D;
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const uint32_t tcol = tmem + lane_field + (w ? C::kColDK : C::kColDV);
    __nv_bfloat16* out = (w ? a.dk : a.dv) + row;
    const float f = w ? a.scale : 1.f;
#pragma unroll
    for (int e = 0; e < D / 64; ++e) {
      const int col = half * (D / 2) + 32 * e;
      uint32_t r[32];
      tmem_ld_32x32b_x32(tcol + col, r);
      wait_dep(r);
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) pk[k] = pack_bf16x2(__uint_as_float(r[2 * k]) * f, __uint_as_float(r[2 * k + 1]) * f);
      if (store) {
        uint4* dst = reinterpret_cast<uint4*>(out + col);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// TMA producer (one thread)
// ------------------------------------------------------------------------------------------------
template <int D, bool M>
__device__ __forceinline__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                                              const CUtensorMap* tdo, int n, int it0, int n0, int bh,
                                              uint32_t sbase, const BArgs& a, const Abort& ab) {
  using C = BCfg<D>;
  const uint32_t sbar = sbase + C::kBarOff;
  tma_prefetch_desc(tq);
  tma_prefetch_desc(tk);
  tma_prefetch_desc(tv);
  tma_prefetch_desc(tdo);
  if (!a.drop_kv) {
    mbar_arrive_expect_tx(sbar + 8 * C::kKVFull, 2 * C::kTile);
#pragma unroll
    for (int ch = 0; ch < C::kChunks; ++ch) {
      tma_load_3d(sbase + C::kKOff + ch * kAtom, tk, sbar + 8 * C::kKVFull, 64 * ch, n0, bh);
      tma_load_3d(sbase + C::kVOff + ch * kAtom, tv, sbar + 8 * C::kKVFull, 64 * ch, n0, bh);
    }
  }
  // Q_i (with its -L / scale terms) and dO_i (with its -D terms) are loaded separately: Q_i's stage
  // is free once dK_i has read it, dO_i's once dV_i has.
  int issued = 0;
  bool ok = true;
  int qt = it0 - 1;  // element mask: the query tile of step i
  const unsigned long long* bits = M ? key_tile_bits(a, bh, n0 / kBN) : nullptr;
  for (int i = 0; i < n && ok; ++i) {
    if constexpr (M) qt = next_qtile<M>(a, bits, qt);
    const int q0 = (M ? qt : it0 + i) * kBM;
    const size_t r0 = (static_cast<size_t>(bh) * a.Nq_pad + q0) * 16;
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const int stages = w ? C::kOStages : C::kQStages;
      const int st = i % stages, use = i / stages;
      if (use > 0 && !thread_wait(sbar + 8 * ((w ? C::kOEmpty : C::kQEmpty) + st), (use - 1) & 1, ab)) {
        ok = false;
        break;
      }
      const uint32_t bar = sbar + 8 * ((w ? C::kOFull : C::kQFull) + st);
      const uint32_t dst = sbase + (w ? C::do_off(st) : C::q_off(st));
      mbar_arrive_expect_tx(bar, C::kTile + C::kExtBytes);
#pragma unroll
      for (int ch = 0; ch < C::kChunks; ++ch) tma_load_3d(dst + ch * kAtom, w ? tdo : tq, bar, 64 * ch, q0, bh);
      bulk_load(sbase + (w ? C::ext_do_off(st) : C::ext_q_off(st)), (w ? a.ext_do : a.ext_q) + r0, C::kExtBytes, bar);
      issued = 2 * i + w + 1;
    }
  }
  if (!ok) {
    // Let the copies already in flight land before the CTA's shared memory goes away: the last
    // loads of each kind, as many as it has buffers.
    const uint64_t until = globaltimer_ns() + 50ull * 1000 * 1000;
    volatile uint32_t never = 0;
    if (!a.drop_kv) mbar_wait_bounded(sbar + 8 * C::kKVFull, 0, &never, until);
    for (int idx = max(0, issued - 2 * max(C::kQStages, C::kOStages)); idx < issued; ++idx) {
      const int i = idx >> 1, w = idx & 1;
      const int stages = w ? C::kOStages : C::kQStages;
      if (i < (issued - 1 - w) / 2 + 1 - stages) continue;  // an older load of a buffer reused since
      mbar_wait_bounded(sbar + 8 * ((w ? C::kOFull : C::kQFull) + i % stages), (i / stages) & 1, &never, until);
    }
  }
}

// ------------------------------------------------------------------------------------------------
// MMA issuer: the whole warp runs the schedule, one elected lane issues.
// ------------------------------------------------------------------------------------------------
template <int D>
struct BMma {
  using C = BCfg<D>;
  uint32_t tmem, sbar;
  uint64_t k_kmaj, v_kmaj, k_mn;   // K_j, V_j
  uint64_t q_kmaj0, do_kmaj0;      // stage 0 Q_i, dO_i as K-major operands
  uint64_t q_mn0, do_mn0;          // ... and as MN-major operands
  uint64_t ds_kmaj0, ds_mn0;       // dS^T buffer 0, K-major (for dK) and MN-major (for dQ)
  uint64_t ones, ext_q0, ext_do0;  // the extra K step: constant A block, stage 0 B blocks
  uint32_t lead;

  __device__ __forceinline__ void init(uint32_t tmem_, uint32_t sbase) {
    tmem = tmem_;
    sbar = sbase + C::kBarOff;
    k_kmaj = smem_desc_sw128(sbase + C::kKOff, 16, 1024);
    v_kmaj = smem_desc_sw128(sbase + C::kVOff, 16, 1024);
    k_mn = smem_desc_sw128(sbase + C::kKOff, kAtom, 1024);
    q_kmaj0 = smem_desc_sw128(sbase + C::q_off(0), 16, 1024);
    do_kmaj0 = smem_desc_sw128(sbase + C::do_off(0), 16, 1024);
    q_mn0 = smem_desc_sw128(sbase + C::q_off(0), kAtom, 1024);
    do_mn0 = smem_desc_sw128(sbase + C::do_off(0), kAtom, 1024);
    ds_kmaj0 = smem_desc_sw128(sbase + C::kDSOff, 16, 1024);
    ds_mn0 = smem_desc_sw128(sbase + C::kDSOff, kAtom, 1024);
    ones = smem_desc_sw32(sbase + C::kOnesOff);
    ext_q0 = smem_desc_sw32(sbase + C::ext_q_off(0));
    ext_do0 = smem_desc_sw32(sbase + C::ext_do_off(0));
    lead = elect_lane();
  }
  // start-address advances, in 16-byte units
  __host__ __device__ static constexpr uint64_t q_adv(int st) { return static_cast<uint64_t>(C::q_off(st) - C::q_off(0)) >> 4; }
  __host__ __device__ static constexpr uint64_t do_adv(int st) { return static_cast<uint64_t>(C::do_off(st) - C::do_off(0)) >> 4; }
  __host__ __device__ static constexpr uint64_t ds_adv(int b) { return static_cast<uint64_t>(b) * (C::kDSBytes >> 4); }
  // K-major operand, K step kk of 16 elements: 4 steps per 128-byte row, then the next 64-column chunk
  __host__ __device__ static constexpr uint64_t kmaj_adv(int kk) { return static_cast<uint64_t>((kk >> 2) * kAtom + (kk & 3) * 32) >> 4; }
  // MN-major operand, K step kk of 16 rows
  __host__ __device__ static constexpr uint64_t mn_adv(int kk) { return static_cast<uint64_t>(kk * 16 * 128) >> 4; }

  __host__ __device__ static constexpr uint64_t ext_q_adv(int st) {
    return static_cast<uint64_t>(C::ext_q_off(st) - C::ext_q_off(0)) >> 4;
  }
  __host__ __device__ static constexpr uint64_t ext_do_adv(int st) {
    return static_cast<uint64_t>(C::ext_do_off(st) - C::ext_do_off(0)) >> 4;
  }
  // S'^T = K Q^T + ones (terms of -L / scale)^T
  __device__ __forceinline__ void issue_s(int b, int st) const {
    constexpr uint32_t id = mma_idesc_bf16_f32(kBN, kBM, false);
    const uint64_t bq = q_kmaj0 + q_adv(st);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_ss_lead(tmem + C::col_s(b), k_kmaj + kmaj_adv(kk), bq + kmaj_adv(kk), id, kk > 0 ? 1u : 0u, lead);
    mma_ss_lead(tmem + C::col_s(b), ones, ext_q0 + ext_q_adv(st), id, 1u, lead);
  }
  // dP'^T = V dO^T + ones (terms of -D)^T
  __device__ __forceinline__ void issue_dp(int st) const {
    constexpr uint32_t id = mma_idesc_bf16_f32(kBN, kBM, false);
    const uint64_t bd = do_kmaj0 + do_adv(st);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_ss_lead(tmem + C::kColDP, v_kmaj + kmaj_adv(kk), bd + kmaj_adv(kk), id, kk > 0 ? 1u : 0u, lead);
    mma_ss_lead(tmem + C::kColDP, ones, ext_do0 + ext_do_adv(st), id, 1u, lead);
  }
  // dP'^T of queries [64 h, 64 h + 64) only, into those 64 columns (N = 64): d = 128, where each half
  // goes as soon as the drain warps have read the dQ columns under it.
  __device__ __forceinline__ void issue_dp_half(int st, int h) const {
    constexpr uint32_t id = mma_idesc_bf16_f32(kBN, kBM / 2, false);
    const uint64_t bd = do_kmaj0 + do_adv(st) + static_cast<uint64_t>(h * (kBM / 2) * 128 >> 4);
    const uint64_t be = ext_do0 + ext_do_adv(st) + static_cast<uint64_t>(h * (kBM / 2) * 32 >> 4);
    const uint32_t dcol = tmem + C::kColDP + (kBM / 2) * h;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_ss_lead(dcol, v_kmaj + kmaj_adv(kk), bd + kmaj_adv(kk), id, kk > 0 ? 1u : 0u, lead);
    mma_ss_lead(dcol, ones, be, id, 1u, lead);
  }
  __device__ __forceinline__ void issue_dv(int b, int st, bool first) const {
    constexpr uint32_t id = mma_idesc_bf16_f32(kBN, D, true);
    const uint64_t bd = do_mn0 + do_adv(st);
#pragma unroll
    for (int kk = 0; kk < kBM / 16; ++kk)
      mma_ts_lead(tmem + C::kColDV, tmem + C::col_s(b) + p_step_col(kk), bd + mn_adv(kk), id,
                  (!first || kk > 0) ? 1u : 0u, lead);
  }
  __device__ __forceinline__ void issue_dk(int dsb, int st, bool first) const {
    constexpr uint32_t id = mma_idesc_bf16_f32(kBN, D, true);
    const uint64_t aa = ds_kmaj0 + ds_adv(dsb), bq = q_mn0 + q_adv(st);
#pragma unroll
    for (int kk = 0; kk < kBM / 16; ++kk)
      mma_ss_lead(tmem + C::kColDK, aa + kmaj_adv(kk), bq + mn_adv(kk), id, (!first || kk > 0) ? 1u : 0u, lead);
  }
  __device__ __forceinline__ void issue_dq(int b, int dsb) const {
    constexpr uint32_t id = mma_idesc_bf16_f32(kBM, D, true, true);
    const uint64_t aa = ds_mn0 + ds_adv(dsb);
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk)
      mma_ss_lead(tmem + C::col_dq(b), aa + mn_adv(kk), k_mn + mn_adv(kk), id, kk > 0 ? 1u : 0u, lead);
  }
  // dQ columns [64 h, 64 h + 64) only (d = 128): the drain's first pass starts while the second half
  // is still being computed.
  __device__ __forceinline__ void issue_dq_half(int dsb, int h) const {
    constexpr uint32_t id = mma_idesc_bf16_f32(kBM, 64, true, true);
    const uint64_t aa = ds_mn0 + ds_adv(dsb), bk = k_mn + static_cast<uint64_t>(h * kAtom >> 4);
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk)
      mma_ss_lead(tmem + C::kColDP + 64 * h, aa + mn_adv(kk), bk + mn_adv(kk), id, kk > 0 ? 1u : 0u, lead);
  }
  __device__ __forceinline__ void commit(int bar) const { mma_commit_lead(sbar + 8 * bar, lead); }
  __device__ __forceinline__ bool wait(int bar, int parity, const Abort& ab) const {
    return warp_wait(sbar + 8 * bar, parity & 1, ab);
  }
};

// d = 64, main MMA warp: dP^T of the next tile as soon as the compute warps have read this tile's,
// then this tile's dV, dK and dQ once its P^T and dS^T are written.  S^T is the other warp's.
template <int D>
__device__ __forceinline__ bool mma_schedule_two(int n, const BMma<D>& m, const Abort& ab) {
  using C = BCfg<D>;
  if (!m.wait(C::kKVFull, 0, ab) || !m.wait(C::kOFull, 0, ab)) return false;
  tc_fence_after();
  m.issue_dp(0);
  m.commit(C::kDPFull);
  for (int i = 0; i < n; ++i) {
    const int b = i & 1, qs = i % C::kQStages, os = i % C::kOStages, dsb = i % C::kDSBufs;
    if (i + 1 < n) {
      if (!m.wait(C::kDPFree, i, ab) || !m.wait(C::kOFull + (i + 1) % C::kOStages, (i + 1) / C::kOStages, ab))
        return false;
      tc_fence_after();
      m.issue_dp((i + 1) % C::kOStages);
      m.commit(C::kDPFull);
    }
    if (!m.wait(C::kCDone, i, ab)) return false;
    tc_fence_after();
    // dK_i and dQ_i first: they release the one dS^T buffer, which the compute warps of tile i+1
    // are about to refill; then dV_i.  (Measured: 2 % faster than dV, dK, dQ with three Q/dO stages.)
    m.issue_dk(dsb, qs, i == 0);
    m.commit(C::kQEmpty + qs);
    m.issue_dq(b, dsb);
    m.commit(C::kDQFull + b);
    m.commit(C::kDSEmpty + dsb);
    m.issue_dv(b, os, i == 0);
    m.commit(C::kOEmpty + os);
  }
  m.commit(C::kAccDone);
  return true;
}

// d = 64, S^T warp: S^T of tile t into buffer t % 2 once tile t-2 is done with it -- dV_{t-2} has read
// P^T_{t-2} (the dO stage of tile t-2 is released after dV_{t-2}) and the drain warps have read dQ_{t-2}
// -- and Q_t has landed.
template <int D>
__device__ __forceinline__ bool mma_schedule_s(int n, const BMma<D>& m, const Abort& ab) {
  using C = BCfg<D>;
  if (!m.wait(C::kKVFull, 0, ab)) return false;
  for (int t = 0; t < n; ++t) {
    const int b = t & 1;
    if (t >= 2) {
      const int u = t - 2;
      if (!m.wait(C::kDQFree + b, u / 2, ab) || !m.wait(C::kOEmpty + u % C::kOStages, u / C::kOStages, ab))
        return false;
    }
    if (!m.wait(C::kQFull + t % C::kQStages, t / C::kQStages, ab)) return false;
    tc_fence_after();
    m.issue_s(b, t % C::kQStages);
    m.commit(C::kSFull + b);
  }
  return true;
}

// d = 128, one MMA warp: one S^T buffer, dQ in the dP^T columns.
template <int D>
__device__ __forceinline__ bool mma_schedule_one(int n, const BMma<D>& m, const Abort& ab) {
  using C = BCfg<D>;
  if (!m.wait(C::kKVFull, 0, ab) || !m.wait(C::kQFull, 0, ab) || !m.wait(C::kOFull, 0, ab)) return false;
  tc_fence_after();
  m.issue_s(0, 0);
  m.commit(C::kSFull);
  m.issue_dp_half(0, 0);
  m.commit(C::kDPFull);
  m.issue_dp_half(0, 1);
  m.commit(C::kDPFullB);
  for (int i = 0; i < n; ++i) {
    const int dsb = i % C::kDSBufs;
    if (!m.wait(C::kCDone, i, ab)) return false;
    tc_fence_after();
    // dK_i, dV_i, then dQ_i: Q_i's stage is released first, so Q_{i+1} is in place when the next S^T
    // is issued; with one S^T buffer that S^T waits for dV_i anyway, and dO_{i+1} is needed only
    // after the dQ drain.  (Measured: dK first 1.0 % faster than dV first, dQ first 7 % slower.)
    m.issue_dk(dsb, 0, i == 0);
    m.commit(C::kQEmpty);
    m.issue_dv(0, 0, i == 0);
    m.commit(C::kOEmpty);
    // dQ_i into the dP^T columns (read by the compute warps already), in two halves of 64 columns
    m.issue_dq_half(dsb, 0);
    m.commit(C::kDQFull);
    m.issue_dq_half(dsb, 1);
    m.commit(C::kDQFull + 1);
    m.commit(C::kDSEmpty + dsb);
    if (i + 1 < n) {
      // S^T of the next tile after dV_i has read P^T from the same columns (issue order).
      if (!m.wait(C::kQFull, i + 1, ab)) return false;
      tc_fence_after();
      m.issue_s(0, 0);
      m.commit(C::kSFull);
      // dP^T of the next tile in two query halves, each as soon as the drain warps have read the
      // 64 dQ columns it overwrites (the first half after the drain's first pass).
      if (!m.wait(C::kDQFree, i, ab) || !m.wait(C::kOFull, i + 1, ab)) return false;
      tc_fence_after();
      m.issue_dp_half(0, 0);
      m.commit(C::kDPFull);
      if (!m.wait(C::kDQFree + 1, i, ab)) return false;
      tc_fence_after();
      m.issue_dp_half(0, 1);
      m.commit(C::kDPFullB);
    }
  }
  m.commit(C::kAccDone);
  return true;
}

template <int D>
__device__ __forceinline__ void mma_role(int n, uint32_t tmem, uint32_t sbase, bool s_warp, const Abort& ab) {
  using C = BCfg<D>;
  BMma<D> m;
  m.init(tmem, sbase);
  bool ok;
  if constexpr (C::kTwoS) ok = s_warp ? mma_schedule_s<D>(n, m, ab) : mma_schedule_two<D>(n, m, ab);
  else ok = mma_schedule_one<D>(n, m, ab);
  // Every MMA (and every arrival its commits make) completes before the CTA winds down.
  const int drain = s_warp ? C::kDrainS : C::kDrain;
  m.commit(drain);
  volatile uint32_t never = 0;
  const uint64_t until = ok ? ab.deadline : globaltimer_ns() + 50ull * 1000 * 1000;
  mbar_wait_bounded(m.sbar + 8 * drain, 0, &never, until);
  __syncwarp();
}

// ------------------------------------------------------------------------------------------------
// dQ drain warps: one thread per query row of the tile.
// ------------------------------------------------------------------------------------------------
template <int D, bool M>
__device__ __forceinline__ void drain_role(const CUtensorMap* tdq, int n, int it0, int n0, int bh, uint32_t tmem,
                                           uint32_t sbase, const BArgs& a, const Abort& ab) {
  using C = BCfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t sbar = sbase + C::kBarOff;
  const bool issuer = (warp == kDrainWarp0) && lane == 0;
  const uint32_t stg = sbase + C::kDQOff;  // two [128 rows][32 fp32] boxes, 128-byte swizzled
  if (issuer) tma_prefetch_desc(tdq);
  int qt = it0 - 1;  // element mask: the query tile of step i
  const unsigned long long* bits = M ? key_tile_bits(a, bh, n0 / kBN) : nullptr;
  for (int i = 0; i < n; ++i) {
    const int b = i % C::kSBufs;
    if constexpr (M) qt = next_qtile<M>(a, bits, qt);
    // d = 64: one dQ buffer per tile; d = 128: dQ in two 64-column halves, one per pass
    bool fail = C::kTwoS && !warp_wait(sbar + 8 * (C::kDQFull + b), (i / C::kSBufs) & 1, ab);
    if (C::kTwoS && !fail) tc_fence_after();
    const int q0 = (M ? qt : it0 + i) * kBM;
#pragma unroll 1
    for (int pass = 0; pass < D / 64; ++pass) {
      uint32_t v[2][32];
      if (!C::kTwoS && !fail) {
        fail = !warp_wait(sbar + 8 * (C::kDQFull + pass), i & 1, ab);
        if (!fail) tc_fence_after();
      }
      if (!fail) {
        const uint32_t t = tmem + lane_field + C::col_dq(b) + 64 * pass;
        tmem_ld_32x32b_x32(t, v[0]);
        tmem_ld_32x32b_x32(t + 32, v[1]);
        wait_dep(v[0]);
        wait_dep(v[1]);
        if (!C::kTwoS || pass == D / 64 - 1) {
          // d = 128: each pass's 64 columns are released on their own barrier (the next tile's dP^T
          // of one query half goes there); d = 64: the buffer, after its only pass.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(sbar + 8 * (C::kDQFree + (C::kTwoS ? b : pass)));
        }
      }
      if (issuer) bulk_wait_read_all();  // the previous reduce has finished reading the staging area
      fail = named_bar_or(kDrainBarrier, 128, fail);
      if (fail) break;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t rbase = stg + h * (kBM * 128) + row * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(rbase + ((static_cast<uint32_t>(u) ^ static_cast<uint32_t>(row & 7)) << 4), v[h][4 * u],
                       v[h][4 * u + 1], v[h][4 * u + 2], v[h][4 * u + 3]);
      }
      fence_proxy_async_smem();
      named_bar_sync(kDrainBarrier, 128);
      if (issuer) {
        tma_reduce_add_3d(tdq, stg, 64 * pass, q0, bh);
        tma_reduce_add_3d(tdq, stg + kBM * 128, 64 * pass + 32, q0, bh);
        bulk_commit_group();
      }
    }
    if (fail) break;
  }
  if (issuer) bulk_wait_all();
}

template <int D, bool M>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dq, const BArgs a) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t sbar = sbase + C::kBarOff;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff + 4);
  const int warp = threadIdx.x >> 5;

  // CTAs walk the heads in groups of a.group, sized so that a group's Q, dO and fp32 dQ accumulator
  // stay in L2; within a group, key tiles with the most query tiles (the first ones, under a causal
  // mask) are launched first.
  const int blk = static_cast<int>(blockIdx.x);
  const int g0 = blk / (a.group * a.nkt) * a.group;
  const int gsz = min(a.group, a.BH - g0);
  const int within = blk - g0 * a.nkt;
  const int jt = within / gsz;
  const int bh = g0 + within % gsz;
  const int n0 = jt * kBN;
  // Query tiles holding a query that sees any of keys [n0, n0 + 128): q in
  // [n0 - off - wr, k_last - off + wl] clipped to [0, Nq).  None (n = 0) is possible with a band.
  const int k_last = min(n0 + kBN, a.Nk) - 1;
  const long long q_lo = a.wr >= 0 ? max(0LL, static_cast<long long>(n0) - a.off - a.wr) : 0LL;
  const long long q_hi = a.wl >= 0 ? min(static_cast<long long>(a.Nq) - 1, static_cast<long long>(k_last) - a.off + a.wl)
                                   : static_cast<long long>(a.Nq) - 1;
  const int it0 = q_lo <= q_hi ? static_cast<int>(q_lo / kBM) : 0;
  int n = q_lo <= q_hi ? static_cast<int>(q_hi / kBM) + 1 - it0 : 0;
  if constexpr (M) {
    // Only the query tiles the element mask does not hide entirely.
    const unsigned long long* bits = key_tile_bits(a, bh, jt);
    int live = 0;
    for (int wi = it0 >> 6; n > 0 && wi <= (it0 + n - 1) >> 6; ++wi) {
      const int lo = max(it0 - 64 * wi, 0), hi = min(it0 + n - 64 * wi, 64);
      const unsigned long long span = (hi == 64 ? ~0ull : (1ull << hi) - 1ull) & (~0ull << lo);
      live += __popcll(__ldg(bits + wi) & span);
    }
    n = live;
  }

  if (threadIdx.x == 0) {
    mbar_init(sbar + 8 * C::kKVFull, 1);
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(sbar + 8 * (C::kQFull + s), 1);
      mbar_init(sbar + 8 * (C::kQEmpty + s), 1);
    }
    for (int s = 0; s < C::kOStages; ++s) {
      mbar_init(sbar + 8 * (C::kOFull + s), 1);
      mbar_init(sbar + 8 * (C::kOEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(sbar + 8 * (C::kSFull + s), 1);
      mbar_init(sbar + 8 * (C::kDSEmpty + s), 1);
      mbar_init(sbar + 8 * (C::kDQFull + s), 1);
      mbar_init(sbar + 8 * (C::kDQFree + s), 4);  // one arrival per drain warp
    }
    mbar_init(sbar + 8 * C::kDPFull, 1);
    mbar_init(sbar + 8 * C::kDPFullB, 1);
    mbar_init(sbar + 8 * C::kCDone, 8);  // one arrival per compute warp
    mbar_init(sbar + 8 * C::kAccDone, 1);
    mbar_init(sbar + 8 * C::kDrain, 1);
    mbar_init(sbar + 8 * C::kDPFree, 8);  // one arrival per compute warp
    mbar_init(sbar + 8 * C::kDrainS, 1);
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x < 2 * kBN) {
    // The constant A block of the extra K step: every 16-byte half of every row is (1, 1, 1, 0, ..., 0)
    // in bf16, so its layout does not depend on the swizzle pattern.
    st_shared_v4(sbase + C::kOnesOff + 16 * threadIdx.x, 0x3F803F80u, 0x00003F80u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  Abort ab{abort_flag, a.status, globaltimer_ns() + a.timeout_ns};

  if (n == 0) {
    // No query sees these keys: dK = dV = 0, nothing else to do.
    if (warp < 8) {
      const int kidx = n0 + (warp & 3) * 32 + (threadIdx.x & 31);
      if (kidx < a.Nk) {
        const size_t row = (static_cast<size_t>(bh) * a.Nk + kidx) * D + (warp >> 2) * (D / 2);
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
          reinterpret_cast<uint4*>(a.dk + row)[i] = make_uint4(0u, 0u, 0u, 0u);
          reinterpret_cast<uint4*>(a.dv + row)[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
  } else if (warp < 8) {
    compute_role<D, M>(n, it0, n0, bh, tmem, sbase, smem, a, ab);
  } else if (warp == kProducerWarp) {
    if ((threadIdx.x & 31) == 0) producer_role<D, M>(&tm_q, &tm_k, &tm_v, &tm_do, n, it0, n0, bh, sbase, a, ab);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    mma_role<D>(n, tmem, sbase, false, ab);
  } else if (warp == kSWarp) {
    if (C::kTwoS) mma_role<D>(n, tmem, sbase, true, ab);
  } else {
    drain_role<D, M>(&tm_dq, n, it0, n0, bh, tmem, sbase, a, ab);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------------------------------------
// Pre- and post-passes (memory-bound, plain loads and stores)
// ------------------------------------------------------------------------------------------------
// D/8 threads per padded query row: each reads 8 elements of O and dO, the group reduces
// D_i = sum(dO_i * O_i); the group also zeroes the row of the dQ array.
// One 32-byte row of the extra K step's B block: the value y as three bf16 terms t0 + t1 + t2 (each
// the rounding of what the previous ones left), halved, in columns 0-2 and again in columns 8-10.
// y = -inf gives (-inf, 0, 0).
__device__ __forceinline__ void write_terms(__nv_bfloat16* row, float y) {
  float t[3] = {y, 0.f, 0.f};
  if (isfinite(y)) {
    float r = y;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      t[j] = __bfloat162float(__float2bfloat16_rn(r));
      r -= t[j];
    }
  }
  const uint32_t w0 = pack_bf16x2(0.5f * t[0], 0.5f * t[1]);
  const uint32_t w1 = pack_bf16x2(0.5f * t[2], 0.f);
  uint4* dst = reinterpret_cast<uint4*>(row);
  dst[0] = make_uint4(w0, w1, 0u, 0u);
  dst[1] = make_uint4(w0, w1, 0u, 0u);
}

template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const float* __restrict__ lse, __nv_bfloat16* __restrict__ ext_q,
                                                       __nv_bfloat16* __restrict__ ext_do, float* __restrict__ dq_acc,
                                                       int BH, int Nq, int Nq_pad, float inv_scale) {
  constexpr int G = D / 8;  // threads per row (8 or 16)
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long r = t / G;
  const int g = static_cast<int>(t % G);
  const bool live = r < static_cast<long long>(BH) * Nq_pad;
  const long long bh = live ? r / Nq_pad : 0;
  const int i = live ? static_cast<int>(r % Nq_pad) : 0;
  float acc = 0.f;
  const bool valid = live && i < Nq;
  if (valid) {
    const size_t off = (static_cast<size_t>(bh) * Nq + i) * D + 8 * g;
    const uint4 a = *reinterpret_cast<const uint4*>(o + off);
    const uint4 b = *reinterpret_cast<const uint4*>(dout + off);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = fmaf(bf16lo_to_f32(av[k]), bf16lo_to_f32(bv[k]), acc);
      acc = fmaf(bf16hi_to_f32(av[k]), bf16hi_to_f32(bv[k]), acc);
    }
  }
#pragma unroll
  for (int s = G / 2; s >= 1; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (!live || !dbg_in(bh * Nq_pad + i, static_cast<long long>(BH) * Nq_pad)) return;
  float4* z = reinterpret_cast<float4*>(dq_acc + (static_cast<size_t>(bh) * Nq_pad + i) * D + 8 * g);
  z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
  z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (g == 0) {
    const size_t ri = (static_cast<size_t>(bh) * Nq_pad + i) * 16;
    // A row with no visible key (L = -inf) must give P = 0 on every key: its term is -inf as well.
    const float L = valid ? lse[static_cast<size_t>(bh) * Nq + i] : -INFINITY;
    write_terms(ext_q + ri, L > -INFINITY ? -L * inv_scale : -INFINITY);
    write_terms(ext_do + ri, valid ? -acc : 0.f);
  }
}

// dQ = scale * accumulated dQ, 8 elements per thread.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq,
                                                     int BH, int Nq, int Nq_pad, float scale) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(BH) * Nq * (D / 8);
  if (t >= total) return;
  const long long r = t / (D / 8);
  const int g = static_cast<int>(t % (D / 8));
  const long long bh = r / Nq;
  const int i = static_cast<int>(r % Nq);
  if (!dbg_in(r, static_cast<long long>(BH) * Nq)) return;
  const float4* src = reinterpret_cast<const float4*>(dq_acc + (static_cast<size_t>(bh) * Nq_pad + i) * D + 8 * g);
  const float4 x = src[0], y = src[1];
  uint4 out;
  out.x = pack_bf16x2(x.x * scale, x.y * scale);
  out.y = pack_bf16x2(x.z * scale, x.w * scale);
  out.z = pack_bf16x2(y.x * scale, y.y * scale);
  out.w = pack_bf16x2(y.z * scale, y.w * scale);
  *reinterpret_cast<uint4*>(dq + static_cast<size_t>(r) * D + 8 * g) = out;
}

template <int D, bool M>
cudaError_t launch_bwd_d(const BwdProblem& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, unsigned int* status,
                         unsigned long long timeout_ns, cudaStream_t stream) {
  using C = BCfg<D>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(bwd_kernel<D, M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int BH = p.B * p.H;
  const int Nq_pad = bwd_padded_rows(p.Nq);
  {
    const long long threads = static_cast<long long>(BH) * Nq_pad * (D / 8);
    const unsigned int grid = static_cast<unsigned int>((threads + 255) / 256);
    bwd_prep_kernel<D><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(p.o),
                                                  static_cast<const __nv_bfloat16*>(p.dout), p.lse,
                                                  static_cast<__nv_bfloat16*>(p.ws_ext_q),
                                                  static_cast<__nv_bfloat16*>(p.ws_ext_do), p.ws_dq, BH, p.Nq,
                                                  Nq_pad, 1.f / p.scale);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  BArgs a;
  a.dk = static_cast<__nv_bfloat16*>(p.dk);
  a.dv = static_cast<__nv_bfloat16*>(p.dv);
  a.ext_q = static_cast<const __nv_bfloat16*>(p.ws_ext_q);
  a.ext_do = static_cast<const __nv_bfloat16*>(p.ws_ext_do);
  a.BH = BH;
  a.Nq = p.Nq;
  a.Nk = p.Nk;
  a.Nq_pad = Nq_pad;
  a.NqT = Nq_pad / kBM;
  a.wl = p.window_left;
  a.wr = p.window_right;
  a.off = p.Nk - p.Nq;
  a.c_log2 = p.scale * kLog2e;
  a.scale = p.scale;
  a.status = status;
  a.timeout_ns = timeout_ns;
  a.drop_kv = p.drop_kv;
  a.nkt = (p.Nk + kBN - 1) / kBN;
  a.H = p.H;
  a.mask = static_cast<const uint32_t*>(p.mask);
  a.mask_sb = p.mask_sb;
  a.mask_sh = p.mask_sh;
  a.mask_words = p.mask_words;
  a.tiles = p.tiles;
  mask_summary_strides(p.mask_sb, p.mask_sh, p.H, p.Nq, p.Nk, true, a.tiles_sb, a.tiles_sh);
  a.tiles_w = mask_summary_words((p.Nq + kBM - 1) / kBM);
  {
    // Heads per group: as many as keep Q, dO (bf16) and the dQ accumulator (fp32) of the group within
    // 64 MiB, about half of L2 (B1 H32 N8192: 16 heads at d = 64, 8 at d = 128).
    const long long per_head = static_cast<long long>(Nq_pad) * D * 8;
    a.group = static_cast<int>(std::max(1LL, std::min<long long>(BH, kL2GroupBytes / per_head)));
  }
  const unsigned int grid = static_cast<unsigned int>(a.nkt) * static_cast<unsigned int>(BH);
  bwd_kernel<D, M><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    const long long threads = static_cast<long long>(BH) * p.Nq * (D / 8);
    const unsigned int g2 = static_cast<unsigned int>((threads + 255) / 256);
    bwd_dq_kernel<D><<<g2, 256, 0, stream>>>(p.ws_dq, static_cast<__nv_bfloat16*>(p.dq), BH, p.Nq, Nq_pad, p.scale);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BwdProblem& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, unsigned int* status,
                            unsigned long long timeout_ns, cudaStream_t stream) {
  if (p.tiles != nullptr) {
    if (p.d == 64) return launch_bwd_d<64, true>(p, tq, tk, tv, tdo, tdq, status, timeout_ns, stream);
    return launch_bwd_d<128, true>(p, tq, tk, tv, tdo, tdq, status, timeout_ns, stream);
  }
  if (p.d == 64) return launch_bwd_d<64, false>(p, tq, tk, tv, tdo, tdq, status, timeout_ns, stream);
  return launch_bwd_d<128, false>(p, tq, tk, tv, tdo, tdq, status, timeout_ns, stream);
}

// Debug builds: read (and optionally clear) this file's device-side check record.
FATTN_DEBUG_ACCESSOR(backward)

}  // namespace fattn
