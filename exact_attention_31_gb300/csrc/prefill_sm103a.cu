// prefill_sm103a.cu -- fused exact attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes is the FlashAttention-2 forward loop nest ("Flash Attention: The Hidden Gem",
// The Algorithm, steps 3-7): for each query tile, carry an exponent reference m, a running sum l and
// an unnormalised output O per row; for each key/value tile compute S = Q K^T, add P = exp(S - m)
// to l and P V to O; after the last tile write O / l and L = m + log(l).  S and P live only in
// tensor memory.  The pages raise m to the running max at every tile and rescale l and O by
// exp(m_old - m_new) (The Correction Factor); here m is set once per row and the rows whose weights
// would leave the safe range are recomputed (see below), which gives the same result.
//
// The grid is persistent: at most one CTA per SM, each working through units (two adjacent 128-row
// query tiles of one (b, h)) in rounds, heaviest causal units first.  Every barrier counts its
// phases over all of a CTA's units, so the next unit's Q tiles, K/V tiles and first S are fetched
// and computed while the current unit finishes; two barriers guard the hand-over (the last S_t has
// read Q_t before Q_t is reloaded; the epilogue has read O_t before the next P_t V overwrites it).
//
// How it maps onto one SM (one CTA per SM, 352 threads):
//   warps 0-3  softmax group for query tile 0 (one thread per query row / TMEM lane)
//   warps 4-7  softmax group for query tile 1
//   warp  8    TMA producer: Q tiles once, then K_j, V_j through a ring of shared-memory slots
//   warp  9    MMA issuer and TMEM owner; with d = 64 it issues query tile 0's products only
//   warp  10   (d = 64) MMA issuer of query tile 1's products
// With d = 64 each query tile has an MMA warp of its own, so one tile's next S never waits in the
// issue order behind the other tile's P V; a key/value slot is released once both warps' products
// that read it have completed.
// Tensor memory (512 columns x 128 lanes, fp32): S_t at columns 128t and O_t at 256 + 128t.  The
// bf16 probabilities P_t are fed to the second MMA straight from TMEM.  With d = 64, O_t uses only
// half of its 128 columns and P_t gets the other half, so S_t(j+1) = Q_t K_{j+1}^T can be issued
// as soon as the softmax group has read S_t(j) into registers: the tensor core computes the next
// scores while the current ones are exponentiated.  With d = 128 tensor memory is full and P_t is
// written over the first 64 columns of S_t, so S_t(j+1) follows P_t(j) V_j.  Two query tiles per
// CTA let the tensor core work on one tile while the other tile's softmax runs.
//
// Scores are handled in log2 units: with c = scale * log2(e), exp(scale * s - scale * m) is
// exp2(s * c - m * c), one FFMA and one ex2 per element.  The exponent reference m of a row is the
// max of its first key tile that holds a visible key, and it stays there: the result is the same
// for any reference as long as l, O and L use the same one (exp(a-c) = exp(a-b) exp(b-c),
// "FlashAttention: attention was never compute-bound", On the maths anxiety), and fp32 and bf16
// keep their relative precision over the whole normal range, so a later key tile whose scores rise
// above m only makes its weights larger than 1.  That saves the row max and the O correction of
// every later step.  What it gives up is a bound on the weights, so each row is checked when its
// unit ends: with the reference in place its weight sum l is at least 1 (the first max has weight
// 1), and the row is accepted when l <= 2^64 and every output is finite.  A row that fails (its
// scores rose by more than about 64 / c over those of its first tile) marks its 128-row query tile
// in a per-CTA bitmask and is counted in a device counter.  When the CTA has worked through its
// units, every role meets at one barrier and the marked tiles are computed again on the tensor
// cores, as units of their own through the same pipeline, by a softmax that carries the running
// max and multiplies l and O (in tensor memory) by exp2(m_old - m_new) whenever the max rises, as
// the pages' correction factor does (the redo phase).  The redo phase's code lives in functions that
// are not inlined: with it inlined the compiler lays out the main loop differently, and the main
// loop is the time that matters.  One row sum
// l of the fp32 weights gives both O / l and L = m + log(l); P V sees the weights rounded to bf16,
// so O carries a relative bias of at most 2^-9 (one rounding of the dominant weight) on rows with
// one dominant key.  The per-row arithmetic uses packed fp32x2 FMA/add and three-input max with
// several independent accumulators, so one thread's row is not a single long dependency chain.
#include <cuda_bf16.h>

#include <algorithm>
#include <math.h>

#include "fattn_internal.h"
#include "sm103a_ptx.cuh"

namespace fattn {
namespace {

constexpr int kBlockM = 128;       // query rows per tile (= TMEM lanes)
constexpr int kBlockN = 128;       // keys per key/value tile
constexpr int kTiles = 2;          // query tiles per CTA
constexpr int kThreads = 352;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;   // tile 0 (d = 64) or both tiles (d = 128); TMEM owner
constexpr int kMmaWarp1 = 10; // tile 1 (d = 64)
constexpr float kWeightSumMax = 0x1p64f;  // a row whose weight sum exceeds this is recomputed
constexpr float kRescaleLog2 = 0.f;        // redo phase: the running max moves when it rises by more
constexpr int kRedoWords = 256;            // bitmask of marked query tiles, 2 bits per unit of a CTA
constexpr int kMaxUnitsPerCta = kRedoWords * 16;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAtomBytes = kBlockM * 128;  // one 128-row x 128-byte swizzled chunk

template <int D>
struct Cfg {
  static constexpr bool kSepP = (D == 64);  // P_t has TMEM columns of its own (see above)
  static constexpr int kChunks = D / 64;
  static constexpr uint32_t kTileBytes = kBlockM * D * 2;
  static constexpr int kSlots = (D == 64) ? 6 : 4;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKVOff = kQOff + kTiles * kTileBytes;
  static constexpr uint32_t kBarOff = kKVOff + kSlots * kTileBytes;
  // barrier indices
  static constexpr int kQFull = 0;              // [2] Q_t landed
  static constexpr int kSFull = 2;              // [2] S_t computed
  static constexpr int kSFree = 4;              // [2] S_t read into registers (separate-P only)
  static constexpr int kPFull = 6;              // [2] P_t written
  static constexpr int kPVDone = 8;             // [2] O_t += P_t V done (separate-P only)
  static constexpr int kOFull = 10;             // [2] last P V of tile t done
  static constexpr int kQFree = 12;             // [2] the unit's last S_t has read Q_t
  static constexpr int kOFree = 14;             // [2] O_t read out by the epilogue (one arrival per warp)
  static constexpr int kDrain = 16;             // [1] wind-down of MMA warp 9
  static constexpr int kKVFull = 17;            // [kSlots]
  static constexpr int kKVEmpty = 17 + kSlots;  // [kSlots]
  static constexpr int kDrain1 = 17 + 2 * kSlots;  // [1] wind-down of MMA warp 10
  static constexpr int kNumBars = 18 + 2 * kSlots;
  static constexpr int kMmaWarps = kSepP ? 2 : 1;   // commits that release a K/V slot
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kRedoOff = kMiscOff + 16;  // kRedoWords words: tiles to compute again
  static constexpr uint32_t kSmemBytes = kRedoOff + kRedoWords * 4 + 1024;  // + slack to align the base
  // tensor-memory columns
  __host__ __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + 128u * t; }
  __host__ __device__ static constexpr uint32_t col_p(int t) { return kSepP ? 256u + 128u * t + 64u : 128u * t; }
};

struct Args {
  __nv_bfloat16* o;
  float* lse;
  int BH, H, Nq, Nk;
  int wl, wr, off;     // mask band: key j visible to row i iff i+off-wl <= j <= i+off+wr (-1 = unbounded)
  int units_per_head;  // ceil(Nq / 256)
  int unit_base;       // this launch works on units [unit_base, unit_end) of the BH * units_per_head
  int unit_end;
  float c_log2;        // scale * log2(e)
  unsigned int* status;
  unsigned long long* recomputed;  // rows that failed the range check (diagnostic counter)
  unsigned long long timeout_ns;
  int drop_kv_block;  // failure-detection testing only; -1 = off
  // Element mask (masked instantiation only): bit j & 31 of word (j >> 5) of row i of head (b, h) at
  // mask + b * mask_sb + h * mask_sh + i * mask_words, set = visible.  Its summary by query tile: for
  // query tile i of head (b, h), at tiles + b * tiles_sb + h * tiles_sh + i * 2 * tiles_w, tiles_w
  // 64-bit words with bit j & 63 of word j >> 6 set when key tile j holds a visible key of the tile,
  // then tiles_w words with the bit set when it holds hidden ones too.
  const uint32_t* mask;
  long long mask_sb, mask_sh;
  int mask_words;
  const unsigned long long* tiles;
  long long tiles_sb, tiles_sh;
  int tiles_w;
  // One-tile items: the units from half_unit0 on are taken one query tile at a time, item
  // half_unit0 + s being tile s % 2 of unit half_unit0 + s / 2 (unit_end counts items); the other
  // tile is another CTA's and is marked absent (je < jb).  half_unit0 = unit_end: none.
  int half_unit0;
};

// Key/value tiles [jb, je) that query tile [r0, r0 + 128) must visit: those holding a key visible to
// any of its rows.  Empty (jb == je) when the tile is past Nq or the band leaves it no key.
__device__ __forceinline__ void key_tiles(int r0, const Args& a, int& jb, int& je) {
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

// First and one-past-last key tile of the union of the CTA's two query tiles' ranges (J0 >= J1 when
// both are empty).  Each range [jb_t, je_t) is an interval, and they overlap or touch because the
// band moves monotonically with the row.
__host__ __device__ __forceinline__ int union_begin(const int (&jb)[2], const int (&je)[2]) {
  int b = 0x7fffffff;
  for (int t = 0; t < kTiles; ++t)
    if (je[t] > jb[t]) b = min(b, jb[t]);
  return b;
}
__host__ __device__ __forceinline__ int union_end(const int (&jb)[2], const int (&je)[2]) {
  int e = 0;
  for (int t = 0; t < kTiles; ++t)
    if (je[t] > jb[t]) e = max(e, je[t]);
  return e;
}

// One unit of work: two adjacent 128-row query tiles of one (b, h), with each tile's key-tile range.
struct Unit {
  int bh, row0;
  int jb[2], je[2];
};

// Under an element mask: the summary words of query tile qt of head bh.
__device__ __forceinline__ const unsigned long long* tile_bits(const Args& a, int bh, int qt) {
  return a.tiles + (bh / a.H) * a.tiles_sb + (bh % a.H) * a.tiles_sh + static_cast<long long>(qt) * 2 * a.tiles_w;
}

// Bits of tiles [b, e) among the 64 from 64 wi on.
__device__ __forceinline__ unsigned long long span_bits(int b, int e, int wi) {
  const int lo = max(b - 64 * wi, 0), hi = min(e - 64 * wi, 64);
  if (lo >= hi) return 0ull;
  return (hi == 64 ? ~0ull : (1ull << hi) - 1ull) & (~0ull << lo);
}

// Under an element mask, the key tiles [64 wi, 64 wi + 64) each query tile of a unit computes: its
// summary word cut to its key range, loaded as a walk over the range reaches a new word.  Scalars,
// not an array, so that a warp whose tile index is a run-time value keeps them in registers.
struct LiveWords {
  int wi = -1;
  unsigned long long w0 = 0ull, w1 = 0ull;
};

__device__ __forceinline__ void live_words(const Args& a, const Unit& u, LiveWords& lw, int wi) {
  if (lw.wi == wi) return;
  lw.wi = wi;
  const int qt = u.row0 / kBlockM;
  lw.w0 = u.je[0] > u.jb[0] ? __ldg(tile_bits(a, u.bh, qt) + wi) & span_bits(u.jb[0], u.je[0], wi) : 0ull;
  lw.w1 = u.je[1] > u.jb[1] ? __ldg(tile_bits(a, u.bh, qt + 1) + wi) & span_bits(u.jb[1], u.je[1], wi) : 0ull;
}

// Whether query tile t of the unit computes key tile j: inside its range and, under an element mask,
// not a tile the mask leaves empty.
template <bool M>
__device__ __forceinline__ bool live(const Args& a, const Unit& u, LiveWords& lw, int t, int j) {
  if constexpr (M) {
    live_words(a, u, lw, j >> 6);
    return ((t ? lw.w1 : lw.w0) >> (j & 63)) & 1ull;
  }
  return t ? (u.jb[1] <= j && j < u.je[1]) : (u.jb[0] <= j && j < u.je[0]);
}

// The key tile after j that either query tile of the unit computes (J1 when none is left).
template <bool M>
__device__ __forceinline__ int next_live(const Args& a, const Unit& u, LiveWords& lw, int j, int J1) {
  ++j;
  if constexpr (M) {
    while (j < J1) {
      live_words(a, u, lw, j >> 6);
      const unsigned long long rest = (lw.w0 | lw.w1) >> (j & 63);
      if (rest != 0ull) return j + __ffsll(static_cast<long long>(rest)) - 1;
      j = (j | 63) + 1;
    }
    return J1;
  }
  return j;
}

// Key tiles query tile t of the unit computes.
template <bool M>
__device__ __forceinline__ int live_count(const Args& a, const Unit& u, int t) {
  if constexpr (M) {
    if (u.je[t] <= u.jb[t]) return 0;
    const unsigned long long* bits = tile_bits(a, u.bh, u.row0 / kBlockM + t);
    int n = 0;
    for (int wi = u.jb[t] >> 6; wi <= (u.je[t] - 1) >> 6; ++wi)
      n += __popcll(__ldg(bits + wi) & span_bits(u.jb[t], u.je[t], wi));
    return n;
  }
  return u.je[t] - u.jb[t];
}

// The k-th unit of this CTA.  The grid is persistent (at most one CTA per SM); units are taken in
// rounds of gridDim.x, heaviest causal units (last query rows) first, and every other round is
// walked backwards so that each CTA's total is closer to the others'.  Returns false past the end.
template <bool M, bool H>
__device__ __forceinline__ bool cta_unit(int k, const Args& a, Unit& u) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const long long idx = a.unit_base + static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
  if (idx >= a.unit_end) return false;
  int i = static_cast<int>(idx);
  int keep = -1;  // a one-tile item: the query tile it computes
  if constexpr (H) {
    if (i >= a.half_unit0) {
      keep = (i - a.half_unit0) & 1;
      i = a.half_unit0 + ((i - a.half_unit0) >> 1);
    }
  }
  u.bh = i % a.BH;
  u.row0 = (a.units_per_head - 1 - i / a.BH) * kTiles * kBlockM;
  key_tiles(u.row0, a, u.jb[0], u.je[0]);
  key_tiles(u.row0 + kBlockM, a, u.jb[1], u.je[1]);
  if constexpr (H) {
    if (keep == 0) {
      u.jb[1] = 0;
      u.je[1] = -1;
    } else if (keep == 1) {
      u.jb[0] = 0;
      u.je[0] = -1;
    }
  }
  if constexpr (M) {
    // Narrow each range to its first and last key tile with a visible key; a tile left with none
    // is empty (its rows get o = 0 and L = -inf).
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      if (u.je[t] <= u.jb[t]) continue;
      const unsigned long long* bits = tile_bits(a, u.bh, u.row0 / kBlockM + t);
      int b = -1, e = 0;
      for (int wi = u.jb[t] >> 6; wi <= (u.je[t] - 1) >> 6; ++wi) {
        const unsigned long long w = __ldg(bits + wi) & span_bits(u.jb[t], u.je[t], wi);
        if (w == 0ull) continue;
        if (b < 0) b = 64 * wi + __ffsll(static_cast<long long>(w)) - 1;
        e = 64 * wi + 64 - __clzll(static_cast<long long>(w));
      }
      u.jb[t] = b >= 0 ? b : 0;
      u.je[t] = b >= 0 ? e : 0;
    }
  }
  return true;
}

// Unit k of the CTA again, for the redo phase: only the query tiles marked in `redo` (2 bits per
// unit; the others emptied).  False when neither is marked.
__device__ __forceinline__ bool redo_unit(int k, const uint32_t* redo, Unit& u) {
  const uint32_t bits = (redo[k >> 4] >> ((k & 15) * 2)) & 3u;
  if (!(bits & 1u)) u.jb[0] = u.je[0] = 0;
  if (!(bits & 2u)) u.jb[1] = u.je[1] = 0;
  return bits != 0u;
}

// Every thread of the CTA calls this once, after its role's main phase: by then every role has issued,
// and the softmax groups have finished, all of the main phase's work (or some wait gave up and set
// the abort word), and the marks are visible to every thread.  True when the redo phase runs: some
// tile was marked (the word after the abort word, set by mark_row) and no wait gave up.
__device__ __noinline__ bool redo_begin(bool ok, volatile uint32_t* abort_flag) {
  __syncwarp();
  named_bar_sync(1, kThreads);
  return abort_flag[1] != 0u && ok && abort_flag[0] == 0u;
}

__device__ __forceinline__ void wait_dep(uint32_t (&r)[32]) {
  // tcgen05.wait::ld that also ties the loaded registers, so no use can be scheduled above it
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
  // A CTA works through many units; each role gives its waits a fresh limit at every unit.
  __device__ void renew(unsigned long long timeout_ns) { deadline = globaltimer_ns() + timeout_ns; }
};

// Every thread of a warp waits; the outcome is made warp-uniform so the warp stays converged for
// the .sync.aligned tensor-memory instructions that follow.
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

// ------------------------------------------------------------------------------------------------
// Packed fp32 helpers (sm_100+): two lanes of fp32 per instruction.
// ------------------------------------------------------------------------------------------------
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

// (a0, a1) += (b0, b1)
__device__ __forceinline__ void fadd2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y, w;\n\t"
      "mov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "add.rn.f32x2 w, x, y;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// Marks query tile t of the CTA's unit k for the redo phase (bit 2k + t of the shared-memory
// bitmask) and counts the row.  Out of line, like any rare path here, so that the main loop's code
// does not change with it.
template <int D>
__device__ __noinline__ void mark_row(const Args& a, uint32_t sbar, int k, int t) {
  const uint32_t word = sbar - Cfg<D>::kBarOff + Cfg<D>::kRedoOff + 4u * static_cast<uint32_t>(k >> 4);
  asm volatile("red.shared.or.b32 [%0], %1;" ::"r"(word), "r"(1u << ((k & 15) * 2 + t)) : "memory");
  const uint32_t any = sbar - Cfg<D>::kBarOff + Cfg<D>::kMiscOff + 8u;  // "some tile is marked"
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(any), "r"(1u) : "memory");
  atomicAdd(a.recomputed, 1ull);
}

// Bits i of a 32-bit word with lo <= i <= hi (either bound may lie outside [0, 31]).
__device__ __forceinline__ uint32_t bits_between(int lo, int hi) {
  const int l = max(lo, 0), h = min(hi, 31);
  if (l > h) return 0u;
  return (0xffffffffu >> (31 - h)) & (0xffffffffu << l);
}

// Max of a row's 128 scores in eight independent chains of three-input maxes: fewer live temporaries
// than the tree below (the redo phase takes it at every step, with all 128 scores live).
__device__ __forceinline__ float max128_chains(const uint32_t (&s)[4][32]) {
  float mx8[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(__uint_as_float(s[0][2 * k]), __uint_as_float(s[0][2 * k + 1]));
#pragma unroll
  for (int e = 16; e < 128; e += 16) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      mx8[k] = max3f(mx8[k], __uint_as_float(s[(e + 2 * k) >> 5][(e + 2 * k) & 31]),
                     __uint_as_float(s[(e + 2 * k + 1) >> 5][(e + 2 * k + 1) & 31]));
  }
  return fmaxf(max3f(mx8[0], mx8[1], mx8[2]), fmaxf(max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
}

// Max of a row's 128 scores as a balanced tree of three-input maxes: 66 instructions, five deep (the
// first step of a unit waits on it, so its depth matters more than its count).
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
// Softmax group: one thread per query row.
// ------------------------------------------------------------------------------------------------
// g counts tile t's steps over all units of this CTA (the phase of S_full, P_full, PV_done);
// done counts its non-empty units (the phase of O_full and O_free).
//
// kRunning = false (the main phase): the exponent reference is fixed at the max of the row's first
// tile with a visible key; a tile with a row that fails the range check at the end is marked in
// `redo` (bit 2k + t, k the CTA's unit index) for the redo phase.
// kRunning = true (the redo phase): every step takes the tile's row max, and when it exceeds the
// reference by more than kRescaleLog2 the reference moves up to it and l and O are multiplied by
// exp2(m_old - m_new) ("Flash Attention: The Hidden Gem", The Correction Factor), so every weight
// stays below 2^kRescaleLog2.  With kRescaleLog2 = 0 the row's largest weight is exactly 1, which
// bf16 holds exactly: the rows that land here are the ones whose large weights come late, and a
// rounded dominant weight would bias their O by up to 2^-9 of its size.
template <int D, bool M, bool kRunning>
__device__ __forceinline__ bool softmax_unit(int t, int k, int jb, int n_tiles, int row0, int bh, uint32_t tmem,
                                             uint32_t sbar, const Args& a, const Abort& ab, int& g, int& done) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int q_row = row0 + t * kBlockM + quarter * 32 + lane;
  // this row's visible keys: [lo, hi] (lo may be negative, hi may be below lo)
  const long long c_row = static_cast<long long>(q_row) + a.off;
  const int hi = static_cast<int>(a.wr >= 0 ? min(c_row + a.wr, static_cast<long long>(a.Nk) - 1)
                                            : static_cast<long long>(a.Nk) - 1);
  const int lo = static_cast<int>(a.wl >= 0 ? max(c_row - a.wl, -1LL) : -1LL);
  const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = tmem + lane_field + C::col_s(t);
  const uint32_t tO = tmem + lane_field + C::col_o(t);
  const uint32_t tP = tmem + lane_field + C::col_p(t);
  const float c = a.c_log2;

  float m_ref = -INFINITY;  // exponent reference, log2 units of the scaled score
  float l = 0.f;            // sum of the fp32 weights: O = O / l, L = m + log(l)
  bool ok = true;
  // Element mask: this tile's summary words and this row's mask words (rows past Nq read none).  The
  // walk visits the key tiles whose live bit is set; a tile's partial bit (the same for the whole
  // tile) says whether the row's 128 bits for it are needed.
  const unsigned long long* bits = nullptr;
  const uint4* mrow = nullptr;
  if constexpr (M) {
    bits = tile_bits(a, bh, row0 / kBlockM + t);
    if (q_row < a.Nq)
      mrow = reinterpret_cast<const uint4*>(a.mask + (bh / a.H) * a.mask_sb + (bh % a.H) * a.mask_sh +
                                            static_cast<long long>(q_row) * a.mask_words);
  }
  int jm = jb;  // element mask: the key tile of this step (the tiles the mask leaves empty are skipped)
  for (int step = 0; step < n_tiles; ++step, ++g) {
    const int j = M ? jm : jb + step;
    uint4 mw = make_uint4(~0u, ~0u, ~0u, ~0u);  // the row's 128 mask bits for key tile j
    bool partial = false;
    unsigned long long live_w = 0ull, part_w = 0ull;
    if constexpr (M) {
      live_w = __ldg(bits + (j >> 6));
      part_w = __ldg(bits + a.tiles_w + (j >> 6));
    }
    if (!warp_wait(sbar + 8 * (C::kSFull + t), g & 1, ab)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t s[4][32];
    tmem_ld_32x32b_x128(tS, s);  // one load of the 128 columns (fewer than four 32-column loads)
#pragma unroll
    for (int h = 0; h < 4; ++h) wait_dep(s[h]);
    if constexpr (C::kSepP) {
      // S_t is in registers: the MMA warp may compute the next S_t into the same columns.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sbar + 8 * (C::kSFree + t));
    }

    const int kv0 = j * kBlockN;
    if constexpr (M) {
      // Band and element mask in one pass: bit i of vis[h] says whether key kv0 + 32 h + i is
      // visible to this row; only tiles the band cuts or the mask partly hides take it.
      const bool cut = __any_sync(0xffffffffu, kv0 + kBlockN - 1 > hi || kv0 < lo);
      partial = (part_w >> (j & 63)) & 1ull;
      if (partial && mrow != nullptr) mw = __ldg(mrow + j);
      if (cut || partial) {
        uint32_t vis[4] = {mw.x, mw.y, mw.z, mw.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) vis[h] &= bits_between(lo - kv0 - 32 * h, hi - kv0 - 32 * h);
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (!((vis[h] >> i) & 1u)) s[h][i] = __float_as_uint(-INFINITY);
      }
    } else {
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
    }
    float corr = 1.f;  // redo phase: factor for l and O when the reference moved in this step
    bool moved = false;
    if constexpr (kRunning) {
      const float m_new = fmaxf(m_ref, max128_chains(s) * c);
      if (m_new > m_ref + kRescaleLog2) {
        corr = ex2_approx(m_ref - m_new);  // 0 while no key has been seen
        m_ref = m_new;
        l *= corr;
        moved = true;
      }
    } else {
      // The reference is the max of the row's first key tile that holds a visible key; later tiles
      // leave it in place.
      if (__any_sync(0xffffffffu, m_ref == -INFINITY)) {
        const float mx = max128_tree(s);
        if (m_ref == -INFINITY) m_ref = mx * c;
      }
    }
    const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;

    // P in two halves of 64 keys, each stored to TMEM as soon as it is packed.
    uint32_t ph[32];
    float ls[4] = {0.f, 0.f, 0.f, 0.f};  // two packed pairs of fp32 partial sums
    bool pv_ok = true;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float x0, x1;
        ffma2_bc(x0, x1, __uint_as_float(s[h][2 * i]), __uint_as_float(s[h][2 * i + 1]), c, neg_m);
        const float e0 = ex2_approx(x0);
        const float e1 = ex2_approx(x1);
        ph[(h & 1) * 16 + i] = pack_bf16x2(e0, e1);
        const int acc = (i & 1) * 2;
        fadd2(ls[acc], ls[acc + 1], e0, e1);
      }
      if (h & 1) {
        if (C::kSepP && h == 1 && g > 0) {
          // P_t is still read by the previous P_t V until it completes.
          pv_ok = warp_wait(sbar + 8 * (C::kPVDone + t), (g - 1) & 1, ab);
          if (!pv_ok) break;
          tc_fence_after();
        }
        tmem_st_32x32b_x32(tP + 32 * (h >> 1), ph);
      }
    }
    if (!pv_ok) {
      ok = false;
      break;
    }
    if constexpr (kRunning) {
      // O_t was last written by P_t(j-1) V_{j-1}, which has completed: with a separate P its
      // completion was awaited before the P store above; with P over S, S_t(j) was issued after it.
      if (step > 0 && __any_sync(0xffffffffu, moved)) {
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
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sbar + 8 * (C::kPFull + t));
    // The row sum is not needed by the hand-off: P_t goes to the MMA warp first.
    l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
    if constexpr (M) {
      if (step + 1 < n_tiles) {
        // The next live tile: in j's word or a later one.
        const unsigned long long rest = (live_w >> (j & 63)) >> 1;
        if (rest != 0ull) {
          jm = j + __ffsll(static_cast<long long>(rest));
        } else {
          for (int w = (j >> 6) + 1; w < a.tiles_w; ++w) {
            const unsigned long long x = __ldg(bits + w);
            if (x != 0ull) {
              jm = 64 * w + __ffsll(static_cast<long long>(x)) - 1;
              break;
            }
          }
        }
      }
    }
  }
  if (!ok) return false;
  const bool store =
      q_row < a.Nq && dbg_in(static_cast<long long>(bh) * a.Nq + q_row, static_cast<long long>(a.BH) * a.Nq);
  __nv_bfloat16* orow = a.o + (static_cast<size_t>(bh) * a.Nq + (store ? q_row : 0)) * D;
  if (n_tiles == 0) {
    // No key is visible to any row of this tile: o = 0, L = log(0) = -inf.
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
  // A row that saw no key has l = 0 and m = -inf: o = 0 and L = -inf.
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  // Sum of the outputs / 256 (not finite iff one of them is not), in four independent partial sums.
  float fin = 0.f, fin1 = 0.f, fin2 = 0.f, fin3 = 0.f;
  uint32_t oall[D / 32][32];  // O_t's D columns of this row, in one load
  if constexpr (D == 128) tmem_ld_32x32b_x128(tO, oall);
  else tmem_ld_32x32b_x64(tO, oall);
#pragma unroll
  for (int h = 0; h < D / 32; ++h) wait_dep(oall[h]);
#pragma unroll
  for (int h = 0; h < D / 32; ++h) {
    const uint32_t(&o)[32] = oall[h];
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float y0 = __uint_as_float(o[2 * i]) * inv_l, y1 = __uint_as_float(o[2 * i + 1]) * inv_l;
      if constexpr (!kRunning) {
        if (i & 1) {
          fin2 = fmaf(y0, 0x1p-8f, fin2);
          fin3 = fmaf(y1, 0x1p-8f, fin3);
        } else {
          fin = fmaf(y0, 0x1p-8f, fin);
          fin1 = fmaf(y1, 0x1p-8f, fin1);
        }
      }
      pk[i] = pack_bf16x2(y0, y1);
    }
    if (store) {
      uint4* dst = reinterpret_cast<uint4*>(orow + 32 * h);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
  }
  fin = (fin + fin1) + (fin2 + fin3);
  // O_t has been read: the next unit's first P_t V may overwrite it.
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(sbar + 8 * (C::kOFree + t));
  ++done;
  if (store && a.lse != nullptr) {
    a.lse[static_cast<size_t>(bh) * a.Nq + q_row] = l > 0.f ? (m_ref + __log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
  if constexpr (!kRunning) {
    // A row with a visible key has l >= 1 (the reference's own weight); it is accepted when l stayed
    // within kWeightSumMax (no weight overflowed or approached the fp32 range) and its outputs are
    // finite.  Otherwise the tile is computed again in the redo phase.
    const int k_lo = max(lo, 0);
    const bool accepted = l >= 0.5f && l <= kWeightSumMax && fabsf(fin) <= 3.4028234663852886e38f;
    if (store && k_lo <= hi && !accepted) mark_row<D>(a, sbar, k, t);
  }
  __syncwarp();
  return true;
}

// The redo phase of softmax group t (a function of its own, so that its code does not change the
// main phase's): the marked tiles again with a running max, barrier phases continued from g, done.
template <int D, bool M>
__device__ __noinline__ bool softmax_unit_running(int t, int k, int jb, int n_tiles, int row0, int bh, uint32_t tmem,
                                                  uint32_t sbar, const Args& a, const Abort& ab, int& g, int& done) {
  return softmax_unit<D, M, true>(t, k, jb, n_tiles, row0, bh, tmem, sbar, a, ab, g, done);
}

template <int D, bool M, bool H>
__device__ __noinline__ void softmax_tail(int t, uint32_t tmem, uint32_t sbar, const Args& a, Abort ab, int g,
                                          int done, uint32_t* redo, bool ok) {
  if (!redo_begin(ok, ab.flag)) return;
  Unit u;
  for (int k = 0; cta_unit<M, H>(k, a, u); ++k) {
    if (!redo_unit(k, redo, u) || u.je[t] == u.jb[t]) continue;
    ab.renew(a.timeout_ns);
    if (!softmax_unit_running<D, M>(t, k, u.jb[t], live_count<M>(a, u, t), u.row0, u.bh, tmem, sbar, a, ab, g, done))
      return;
  }
}

template <int D, bool M, bool H>
__device__ __forceinline__ void softmax_role(int t, uint32_t tmem, uint32_t sbar, const Args& a, Abort ab,
                                             uint32_t* redo) {
  int g = 0, done = 0;
  bool ok = true;
  Unit u;
  for (int k = 0; cta_unit<M, H>(k, a, u); ++k) {
    if constexpr (H) {
      if (u.je[t] < u.jb[t]) continue;  // a one-tile item's other tile: another CTA's rows
    }
    ab.renew(a.timeout_ns);
    if (!softmax_unit<D, M, false>(t, k, u.jb[t], live_count<M>(a, u, t), u.row0, u.bh, tmem, sbar, a, ab, g, done)) {
      ok = false;
      break;
    }
  }
  softmax_tail<D, M, H>(t, tmem, sbar, a, ab, g, done, redo, ok);
}

// ------------------------------------------------------------------------------------------------
// TMA producer (one thread)
// ------------------------------------------------------------------------------------------------
struct ProducerState {
  int ring = 0;            // K/V ring index of the unit's first key tile (2 per key tile, over all units)
  int qloads[2] = {0, 0};  // Q_t loads issued so far (the phase of Q_full / Q_free)
  int issued = 0;          // ring index one past the last K/V load issued
  int dropped = -1;        // ring index of the load skipped for failure-detection testing
};

// One unit's loads: Q of its non-empty tiles, then K_j and V_j for the union of the two tiles' ranges
// (ring index ring + 2 (j - J0) + w).  False when a wait gave up.
template <int D, bool M>
__device__ __forceinline__ bool producer_unit(const Unit& u, const CUtensorMap* tq, const CUtensorMap* tk,
                                              const CUtensorMap* tv, uint32_t sbase, const Args& a,
                                              const Abort& ab, ProducerState& ps) {
  using C = Cfg<D>;
  const uint32_t sbar = sbase + C::kBarOff;
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    if (u.je[t] <= u.jb[t]) continue;  // empty, or (a one-tile item) another CTA's
    // Q_t's buffer is free once the previous unit's last S_t has read it.
    if (ps.qloads[t] > 0 && !thread_wait(sbar + 8 * (C::kQFree + t), (ps.qloads[t] - 1) & 1, ab)) return false;
    const uint32_t bar = sbar + 8 * (C::kQFull + t);
    mbar_arrive_expect_tx(bar, C::kTileBytes);
#pragma unroll
    for (int ch = 0; ch < C::kChunks; ++ch)
      tma_load_3d(sbase + C::kQOff + t * C::kTileBytes + ch * kAtomBytes, tq, bar, ch * 64, u.row0 + t * kBlockM,
                  u.bh);
    ++ps.qloads[t];
  }
  const int J0 = union_begin(u.jb, u.je), J1 = union_end(u.jb, u.je);
  int n = 0;  // key tiles loaded for this unit (ring index ring + 2 n + w)
  LiveWords lw;
  for (int j = J0; j < J1; j = next_live<M>(a, u, lw, j, J1), ++n) {
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const int idx = ps.ring + 2 * n + w;
      const int slot = idx % C::kSlots;
      const int round = idx / C::kSlots;
      if (round > 0 && !thread_wait(sbar + 8 * (C::kKVEmpty + slot), (round - 1) & 1, ab)) return false;
      ps.issued = idx + 1;
      if (w == 0 && j == a.drop_kv_block) {  // testing only: this tile never arrives
        ps.dropped = idx;
        continue;
      }
      const uint32_t bar = sbar + 8 * (C::kKVFull + slot);
      mbar_arrive_expect_tx(bar, C::kTileBytes);
#pragma unroll
      for (int ch = 0; ch < C::kChunks; ++ch)
        tma_load_3d(sbase + C::kKVOff + slot * C::kTileBytes + ch * kAtomBytes, w ? tv : tk, bar, ch * 64,
                    j * kBlockN, u.bh);
    }
  }
  ps.ring += 2 * n;
  return true;
}

template <int D, bool M>
__device__ __noinline__ bool producer_unit_redo(const Unit& u, const CUtensorMap* tq, const CUtensorMap* tk,
                                                const CUtensorMap* tv, uint32_t sbase, const Args& a, const Abort& ab,
                                                ProducerState& ps) {
  return producer_unit<D, M>(u, tq, tk, tv, sbase, a, ab, ps);
}

// The producer's redo phase and wind-down (whole warp; lane 0 issues).  After a wait gave up, the
// copies already in flight land before the CTA's shared memory goes away.
template <int D, bool M, bool H>
__device__ __noinline__ void producer_tail(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                                           uint32_t sbase, const Args& a, Abort ab, ProducerState ps, bool ok,
                                           uint32_t* redo) {
  using C = Cfg<D>;
  const uint32_t sbar = sbase + C::kBarOff;
  const bool lead = (threadIdx.x & 31) == 0;
  if (redo_begin(ok, ab.flag) && lead) {
    Unit u;
    for (int k = 0; cta_unit<M, H>(k, a, u); ++k) {
      if (!redo_unit(k, redo, u)) continue;
      ab.renew(a.timeout_ns);
      if (!producer_unit_redo<D, M>(u, tq, tk, tv, sbase, a, ab, ps)) {
        ok = false;
        break;
      }
    }
  }
  if (lead && !ok) {
    const uint64_t until = globaltimer_ns() + 50ull * 1000 * 1000;
    volatile uint32_t never = 0;
    for (int idx = max(0, ps.issued - C::kSlots); idx < ps.issued; ++idx) {
      if (idx == ps.dropped) continue;
      const int slot = idx % C::kSlots;
      mbar_wait_bounded(sbar + 8 * (C::kKVFull + slot), (idx / C::kSlots) & 1, &never, until);
    }
#pragma unroll
    for (int t = 0; t < kTiles; ++t)
      if (ps.qloads[t] > 0) mbar_wait_bounded(sbar + 8 * (C::kQFull + t), (ps.qloads[t] - 1) & 1, &never, until);
  }
  __syncwarp();
}

// Whole warp; lane 0 issues the main phase's loads.
template <int D, bool M, bool H>
__device__ __forceinline__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                                              uint32_t sbase, const Args& a, Abort ab, uint32_t* redo) {
  ProducerState ps;
  bool ok = true;
  if ((threadIdx.x & 31) == 0) {
    tma_prefetch_desc(tq);
    tma_prefetch_desc(tk);
    tma_prefetch_desc(tv);
    Unit u;
    for (int k = 0; cta_unit<M, H>(k, a, u); ++k) {
      ab.renew(a.timeout_ns);
      if (!producer_unit<D, M>(u, tq, tk, tv, sbase, a, ab, ps)) {
        ok = false;
        break;
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  producer_tail<D, M, H>(tq, tk, tv, sbase, a, ab, ps, ok, redo);
}

// ------------------------------------------------------------------------------------------------
// MMA issuer: the whole warp runs the schedule (its waits and indices are warp-uniform) and one
// elected lane issues the tcgen05 instructions.  Every shared-memory descriptor is built once; a
// step of K only adds a constant to the start-address field, so issuing an MMA is one 64-bit add.
// ------------------------------------------------------------------------------------------------
template <int D>
struct MmaCtx {
  using C = Cfg<D>;
  uint32_t tmem, sbar;
  uint64_t dq[kTiles];  // Q_t, K-major
  uint64_t dk0;         // slot 0 as a K-major operand (K_j)
  uint64_t dv0;         // slot 0 as an MN-major operand (V_j)
  uint32_t lead;  // non-zero in the one lane that issues

  __device__ __forceinline__ void init(uint32_t tmem_, uint32_t sbase) {
    tmem = tmem_;
    sbar = sbase + C::kBarOff;
#pragma unroll
    for (int t = 0; t < kTiles; ++t) dq[t] = smem_desc_sw128(sbase + C::kQOff + t * C::kTileBytes, 16, 1024);
    dk0 = smem_desc_sw128(sbase + C::kKVOff, 16, 1024);
    dv0 = smem_desc_sw128(sbase + C::kKVOff, kAtomBytes, 1024);
    lead = elect_lane();
  }
  // start-address field advance (16-byte units)
  __host__ __device__ static constexpr uint64_t slot_adv(int slot) { return static_cast<uint64_t>(slot) * (C::kTileBytes >> 4); }
  __host__ __device__ static constexpr uint64_t kmajor_adv(int kk) { return static_cast<uint64_t>((kk >> 2) * kAtomBytes + (kk & 3) * 32) >> 4; }
  __host__ __device__ static constexpr uint64_t vstep_adv(int kk) { return static_cast<uint64_t>(kk * 16 * 128) >> 4; }

  // S_t = Q_t K^T: both operands K-major, 16 elements of d per instruction.
  __device__ __forceinline__ void issue_s(int t, int kslot) const {
    constexpr uint32_t kIdS = mma_idesc_bf16_f32(kBlockM, kBlockN, false);
    const uint64_t a = dq[t], b = dk0 + slot_adv(kslot);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_ss_lead(tmem + C::col_s(t), a + kmajor_adv(kk), b + kmajor_adv(kk), kIdS, kk > 0 ? 1u : 0u, lead);
  }
  // O_t += P_t V: A from TMEM (bf16 pairs packed per column), B = V MN-major, 16 keys per step.
  __device__ __forceinline__ void issue_pv(int t, int vslot, bool first) const {
    constexpr uint32_t kIdPV = mma_idesc_bf16_f32(kBlockM, D, true);
    const uint64_t b = dv0 + slot_adv(vslot);
#pragma unroll
    for (int kk = 0; kk < kBlockN / 16; ++kk)
      mma_ts_lead(tmem + C::col_o(t), tmem + C::col_p(t) + 8 * kk, b + vstep_adv(kk), kIdPV,
                  (!first || kk > 0) ? 1u : 0u, lead);
  }
  __device__ __forceinline__ void commit(int bar) const { mma_commit_lead(sbar + 8 * bar, lead); }
  // KV ring index of K_j is 2j, of V_j is 2j + 1.
  __device__ __forceinline__ bool wait_kv(int idx, const Abort& ab) const {
    return warp_wait(sbar + 8 * (C::kKVFull + idx % C::kSlots), (idx / C::kSlots) & 1, ab);
  }
  __device__ __forceinline__ bool wait(int bar, int parity, const Abort& ab) const {
    return warp_wait(sbar + 8 * bar, parity & 1, ab);
  }
};

// Barrier phases of the MMA warp over all units of the CTA.
struct MmaState {
  int ring = 0;              // K/V ring index of the current unit's first key tile
  int s_issued[2] = {0, 0};  // S_t issued (S_full commits); S_t number n waits S_free number n-1
  int p_seen[2] = {0, 0};    // P_full phases consumed
  int units[2] = {0, 0};     // non-empty units finished per tile (O_full commits, O_free phases)
  int q_seen[2] = {0, 0};    // Q_full phases consumed
};

// S_t for key tile j.  The columns are free once the softmax warps have read the previous S_t (d = 64;
// with d = 128 the previous P_t V, issued earlier by this warp, reads P_t from them).  The unit's
// last S_t releases Q_t.
template <int D>
__device__ __forceinline__ bool issue_s_step(int t, int slot, bool last, const MmaCtx<D>& m, MmaState& st,
                                             const Abort& ab) {
  using C = Cfg<D>;
  if (C::kSepP && st.s_issued[t] > 0) {
    if (!m.wait(C::kSFree + t, st.s_issued[t] - 1, ab)) return false;
    tc_fence_after();
  }
  m.issue_s(t, slot);
  m.commit(C::kSFull + t);
  if (last) m.commit(C::kQFree + t);
  ++st.s_issued[t];
  return true;
}

// O_t += P_t V_j.  The unit's first P_t V overwrites O_t: the previous unit's epilogue must have read it.
template <int D>
__device__ __forceinline__ bool issue_pv_step(int t, int slot, bool first, bool last, const MmaCtx<D>& m,
                                              MmaState& st, const Abort& ab) {
  using C = Cfg<D>;
  if (!m.wait(C::kPFull + t, st.p_seen[t]++, ab)) return false;
  if (first && st.units[t] > 0 && !m.wait(C::kOFree + t, st.units[t] - 1, ab)) return false;
  tc_fence_after();
  m.issue_pv(t, slot, first);
  if (C::kSepP) m.commit(C::kPVDone + t);
  if (last) {
    m.commit(C::kOFull + t);
    ++st.units[t];
  }
  return true;
}

// Separate P (d = 64), one warp per query tile t: S_t(j+1) is issued once S_t(j) has been read,
// P_t(j) V_j once P_t(j) is written.  The warp waits for every K/V tile of the unit's union range
// and commits once per tile to its slot's K/V-empty barrier (two arrivals release a slot), whether
// or not tile t uses it; a commit for a slot's next use can only follow that use's load, which
// itself waited for both of the previous use's arrivals.  Ring index of K_j is ring + 2 (j - J0),
// of V_j one more.
// The MMA warps' look-ahead (d = 64, one warp per query tile): the CTA's next unit (and a fresh wait
// limit for it), computed once the current unit's first S is issued, while the warp would otherwise
// wait, rather than between units where it delays the next unit's first S.  (With d = 128's one
// interleaved warp it measured 0.5 % slower and is not used there.)
struct NoNext {
  __device__ __forceinline__ void operator()() const {}
};
template <bool M, bool H>
struct NextUnit {
  const Args* a;
  int k;
  Unit* u;
  bool* have;
  Abort* ab;
  __device__ __forceinline__ void operator()() const {
    *have = cta_unit<M, H>(k, *a, *u);
    ab->renew(a->timeout_ns);
  }
};

template <int D, bool M, class N = NoNext>
__device__ __forceinline__ bool mma_unit_tile(int t, const Unit& u, const MmaCtx<D>& m, MmaState& st,
                                              const Abort& ab, const Args& a, const N& next = N()) {
  using C = Cfg<D>;
  const int J0 = union_begin(u.jb, u.je), J1 = union_end(u.jb, u.je);
  if (J0 >= J1) {
    next();
    return true;
  }
  const int jb = t ? u.jb[1] : u.jb[0], je = t ? u.je[1] : u.je[0];
  const int r0 = st.ring;
  if constexpr (M) {
    // The same schedule over the key tiles either query tile computes (n-th loaded: ring r0 + 2 n).
    LiveWords lw;
    if (!m.wait_kv(r0, ab)) return false;
    tc_fence_after();
    if (live<M>(a, u, lw, t, J0) && !issue_s_step<D>(t, r0 % C::kSlots, J0 == je - 1, m, st, ab)) return false;
    m.commit(C::kKVEmpty + r0 % C::kSlots);
    next();
    int n = 0;
    for (int j = J0; j < J1; ++n) {
      const int jn = next_live<M>(a, u, lw, j, J1);
      if (jn < J1) {
        const int kidx = r0 + 2 * (n + 1);
        if (!m.wait_kv(kidx, ab)) return false;
        if (live<M>(a, u, lw, t, jn) && !issue_s_step<D>(t, kidx % C::kSlots, jn == je - 1, m, st, ab)) return false;
        m.commit(C::kKVEmpty + kidx % C::kSlots);
      }
      const int vidx = r0 + 2 * n + 1;
      if (!m.wait_kv(vidx, ab)) return false;
      if (live<M>(a, u, lw, t, j) && !issue_pv_step<D>(t, vidx % C::kSlots, j == jb, j == je - 1, m, st, ab)) return false;
      m.commit(C::kKVEmpty + vidx % C::kSlots);
      j = jn;
    }
    st.ring = r0 + 2 * n;
    return true;
  }
  if (!m.wait_kv(r0, ab)) return false;
  tc_fence_after();
  if (jb <= J0 && J0 < je && !issue_s_step<D>(t, r0 % C::kSlots, J0 == je - 1, m, st, ab)) return false;
  m.commit(C::kKVEmpty + r0 % C::kSlots);  // K_{J0} is free once S_t(J0) is done
  next();
  for (int j = J0; j < J1; ++j) {
    if (j + 1 < J1) {
      const int kidx = r0 + 2 * (j + 1 - J0);
      if (!m.wait_kv(kidx, ab)) return false;
      if (jb <= j + 1 && j + 1 < je && !issue_s_step<D>(t, kidx % C::kSlots, j + 1 == je - 1, m, st, ab))
        return false;
      m.commit(C::kKVEmpty + kidx % C::kSlots);
    }
    const int vidx = r0 + 2 * (j - J0) + 1;
    if (!m.wait_kv(vidx, ab)) return false;
    if (jb <= j && j < je && !issue_pv_step<D>(t, vidx % C::kSlots, j == jb, j == je - 1, m, st, ab)) return false;
    m.commit(C::kKVEmpty + vidx % C::kSlots);
  }
  st.ring = r0 + 2 * (J1 - J0);
  return true;
}

// P aliased over S (d = 128): S_t(j+1) is issued after P_t(j) V_j, which reads P_t from the same
// columns (tcgen05.mma operations of one CTA execute in issue order).
template <int D, bool M>
__device__ __forceinline__ bool mma_unit_aliased_p(const Unit& u, const MmaCtx<D>& m, MmaState& st,
                                                   const Abort& ab, const Args& a) {
  using C = Cfg<D>;
  const int J0 = union_begin(u.jb, u.je), J1 = union_end(u.jb, u.je);
  if (J0 >= J1) return true;
  auto active = [&](int t, int j) { return u.jb[t] <= j && j < u.je[t]; };
  const int r0 = st.ring;
  if constexpr (M) {
    // The same schedule over the key tiles either query tile computes: the n-th loaded tile j (ring
    // r0 + 2 n) after the previous one jp.
    int j = J0, jp = -1, n = 0;
    LiveWords lw;
    for (;;) {
      const int r = r0 + 2 * n;
      if (j < J1 && !m.wait_kv(r, ab)) return false;
      if (n > 0 && !m.wait_kv(r - 1, ab)) return false;  // V_jp
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        if (n > 0 && live<M>(a, u, lw, t, jp) &&
            !issue_pv_step<D>(t, (r - 1) % C::kSlots, jp == u.jb[t], jp == u.je[t] - 1, m, st, ab))
          return false;
        if (j < J1 && live<M>(a, u, lw, t, j) && !issue_s_step<D>(t, r % C::kSlots, j == u.je[t] - 1, m, st, ab))
          return false;
      }
      if (j < J1) m.commit(C::kKVEmpty + r % C::kSlots);
      if (n > 0) m.commit(C::kKVEmpty + (r - 1) % C::kSlots);
      if (j >= J1) break;
      jp = j;
      j = next_live<M>(a, u, lw, j, J1);
      ++n;
    }
    st.ring = r0 + 2 * n;
    return true;
  }
  for (int j = J0; j <= J1; ++j) {
    const int r = r0 + 2 * (j - J0);  // ring index of K_j
    if (j < J1 && !m.wait_kv(r, ab)) return false;
    if (j > J0 && !m.wait_kv(r - 1, ab)) return false;  // V_{j-1}
    tc_fence_after();
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      if (j > J0 && active(t, j - 1) &&
          !issue_pv_step<D>(t, (r - 1) % C::kSlots, j - 1 == u.jb[t], j - 1 == u.je[t] - 1, m, st, ab))
        return false;
      if (j < J1 && active(t, j) && !issue_s_step<D>(t, r % C::kSlots, j == u.je[t] - 1, m, st, ab)) return false;
    }
    if (j < J1) m.commit(C::kKVEmpty + r % C::kSlots);
    if (j > J0) m.commit(C::kKVEmpty + (r - 1) % C::kSlots);
  }
  st.ring = r0 + 2 * (J1 - J0);
  return true;
}

template <int D, bool M>
__device__ __noinline__ bool mma_unit_redo(int tt, const Unit& u, const MmaCtx<D>& m, MmaState& st, const Abort& ab,
                                           const Args& a) {
  using C = Cfg<D>;
  bool ok = true;
#pragma unroll
  for (int t = 0; t < kTiles; ++t)
    if ((!C::kSepP || t == tt) && u.je[t] > u.jb[t] && ok) ok = m.wait(C::kQFull + t, st.q_seen[t]++, ab);
  if (ok) ok = C::kSepP ? mma_unit_tile<D, M>(tt, u, m, st, ab, a) : mma_unit_aliased_p<D, M>(u, m, st, ab, a);
  return ok;
}

// The MMA warp's redo phase and wind-down: before the CTA winds down, every MMA (and every arrival
// its commits make on this CTA's barriers) has completed, on the normal path and after a timeout
// alike.
template <int D, bool M, bool H>
__device__ __noinline__ void mma_tail(int tt, const MmaCtx<D>& m, MmaState st, const Args& a, Abort ab, bool ok,
                                      uint32_t* redo) {
  using C = Cfg<D>;
  if (redo_begin(ok, ab.flag)) {
    Unit u;
    for (int k = 0; ok && cta_unit<M, H>(k, a, u); ++k) {
      if (!redo_unit(k, redo, u)) continue;
      ab.renew(a.timeout_ns);
      ok = mma_unit_redo<D, M>(tt, u, m, st, ab, a);
    }
  }
  const int drain = tt ? C::kDrain1 : C::kDrain;
  m.commit(drain);
  volatile uint32_t never = 0;
  const uint64_t until = ok ? ab.deadline : globaltimer_ns() + 50ull * 1000 * 1000;
  mbar_wait_bounded(m.sbar + 8 * drain, 0, &never, until);
  __syncwarp();
}

// Whole warp.  `tt` is the query tile of this warp (d = 64); with d = 128 the one MMA warp (tt = 0)
// issues both tiles' products.
template <int D, bool M, bool H>
__device__ __forceinline__ void mma_role(int tt, uint32_t tmem, uint32_t sbase, const Args& a, Abort ab,
                                         uint32_t* redo) {
  using C = Cfg<D>;
  MmaCtx<D> m;
  m.init(tmem, sbase);
  MmaState st;
  bool ok = true;
  Unit u, un;
  bool have = cta_unit<M, H>(0, a, u);
  ab.renew(a.timeout_ns);
  for (int k = 0; ok && have; ++k) {
#pragma unroll
    for (int t = 0; t < kTiles; ++t)
      if ((!C::kSepP || t == tt) && u.je[t] > u.jb[t] && ok) ok = m.wait(C::kQFull + t, st.q_seen[t]++, ab);
    bool have_next = false;
    if constexpr (C::kSepP) {
      const NextUnit<M, H> next{&a, k + 1, &un, &have_next, &ab};
      if (ok) ok = mma_unit_tile<D, M>(tt, u, m, st, ab, a, next);
    } else {
      if (ok) ok = mma_unit_aliased_p<D, M>(u, m, st, ab, a);
      if (ok) {
        have_next = cta_unit<M, H>(k + 1, a, un);
        ab.renew(a.timeout_ns);
      }
    }
    u = un;
    have = have_next;
  }
  mma_tail<D, M, H>(tt, m, st, a, ab, ok, redo);
}

template <int D, bool M, bool H>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Args a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t sbar = sbase + C::kBarOff;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff + 4);
  uint32_t* redo = reinterpret_cast<uint32_t*>(smem + C::kRedoOff);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(sbar + 8 * (C::kQFull + t), 1);
      mbar_init(sbar + 8 * (C::kSFull + t), 1);
      mbar_init(sbar + 8 * (C::kSFree + t), kBlockM / 32);  // one arrival per softmax warp
      mbar_init(sbar + 8 * (C::kPFull + t), kBlockM / 32);
      mbar_init(sbar + 8 * (C::kPVDone + t), 1);
      mbar_init(sbar + 8 * (C::kOFull + t), 1);
      mbar_init(sbar + 8 * (C::kQFree + t), 1);
      mbar_init(sbar + 8 * (C::kOFree + t), kBlockM / 32);  // one arrival per softmax warp
    }
    mbar_init(sbar + 8 * C::kDrain, 1);
    mbar_init(sbar + 8 * C::kDrain1, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(sbar + 8 * (C::kKVFull + s), 1);
      mbar_init(sbar + 8 * (C::kKVEmpty + s), C::kMmaWarps);
    }
    *abort_flag = 0u;
    abort_flag[1] = 0u;  // "some tile is marked"
    fence_mbarrier_init();
  }
  for (int w = threadIdx.x; w < kRedoWords; w += kThreads) redo[w] = 0u;
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  Abort ab{abort_flag, a.status, globaltimer_ns() + a.timeout_ns};

  // Each role works through the CTA's units, then meets the others at one barrier (redo_begin) and
  // computes the marked tiles again.
  if (warp < 8) {
    softmax_role<D, M, H>(warp >> 2, tmem, sbar, a, ab, redo);
  } else if (warp == kProducerWarp) {
    producer_role<D, M, H>(&tm_q, &tm_k, &tm_v, sbase, a, ab, redo);
  } else if (warp == kMmaWarp) {
    mma_role<D, M, H>(0, tmem, sbase, a, ab, redo);
  } else if (C::kSepP && warp == kMmaWarp1) {
    mma_role<D, M, H>(1, tmem, sbase, a, ab, redo);
  } else {
    redo_begin(true, abort_flag);  // (d = 128: the spare warp only takes part in the barrier)
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool M, bool H>
cudaError_t launch_d(const FwdProblem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, unsigned int* status, unsigned long long timeout_ns,
                     cudaStream_t stream) {
  using C = Cfg<D>;
  static bool attr_set[64] = {};  // per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_kernel<D, M, H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  Args a;
  a.o = static_cast<__nv_bfloat16*>(p.o);
  a.lse = p.lse;
  a.BH = p.B * p.H;
  a.H = p.H;
  a.Nq = p.Nq;
  a.Nk = p.Nk;
  a.wl = p.window_left;
  a.wr = p.window_right;
  a.off = p.Nk - p.Nq;
  a.units_per_head = (p.Nq + kTiles * kBlockM - 1) / (kTiles * kBlockM);
  a.c_log2 = p.scale * 1.4426950408889634f;
  a.status = status;
  a.recomputed = p.recomputed;
  a.timeout_ns = timeout_ns;
  a.drop_kv_block = p.drop_kv_block;
  a.mask = static_cast<const uint32_t*>(p.mask);
  a.mask_sb = p.mask_sb;
  a.mask_sh = p.mask_sh;
  a.mask_words = p.mask_words;
  a.tiles = p.tiles;
  mask_summary_strides(p.mask_sb, p.mask_sh, p.H, p.Nq, p.Nk, false, a.tiles_sb, a.tiles_sh);
  a.tiles_w = mask_summary_words((p.Nk + kBlockN - 1) / kBlockN);
  // Persistent: one CTA per SM (each holds all of an SM's tensor memory), looping over the units.
  static int sm_count[64] = {};
  if (dev < 0 || dev >= 64 || sm_count[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) sm_count[dev] = n;
    else return cudaErrorInvalidDevice;
  }
  // A CTA marks the tiles to compute again in a bitmask of kMaxUnitsPerCta units, so one launch
  // covers at most grid * kMaxUnitsPerCta units; larger problems take several launches.
  const long long total = static_cast<long long>(a.units_per_head) * a.BH;
  const int sms = sm_count[dev];
  // One-tile items where two-tile units would leave SMs idle: when there are fewer units than SMs,
  // every unit is taken one query tile at a time; without a band (units of equal length), when the
  // last round of units fills at most half of the SMs, that round's units are (under a band the
  // last round holds the lightest units, and the rounds' balance is better left as it is).  A CTA
  // with one tile computes it faster than its share of a unit, and each tile still writes its own O
  // and L, so nothing is merged afterwards.  The kernel for them is a separate instantiation, so
  // that the one for whole units is unchanged.  (Without an element mask only.)
  long long half0 = total;
  if (total <= kMaxUnitsPerCta * static_cast<long long>(sms)) {
    if (2 * total <= sms) half0 = 0;
    else if (total > sms && 2 * (total % sms) <= sms && p.window_left < 0 && p.window_right < 0)
      half0 = total - total % sms;
  }
  if constexpr (!M && !H) {
    if (half0 < total) return launch_d<D, false, true>(p, tq, tk, tv, status, timeout_ns, stream);
  }
  a.half_unit0 = static_cast<int>(std::min<long long>(half0, 0x7fffffffLL));
  if constexpr (H) {
    const long long items = total + (total - half0);
    a.unit_base = 0;
    a.unit_end = static_cast<int>(items);
    prefill_kernel<D, M, H><<<static_cast<unsigned int>(std::min<long long>(items, sms)), kThreads,
                              C::kSmemBytes, stream>>>(tq, tk, tv, a);
    return cudaGetLastError();
  }
  const long long grid = std::min<long long>(total, sms);
  const long long per_launch = grid * kMaxUnitsPerCta;
  for (long long base = 0; base < total; base += per_launch) {
    a.unit_base = static_cast<int>(base);
    a.unit_end = static_cast<int>(std::min(total, base + per_launch));
    const unsigned int g = static_cast<unsigned int>(std::min<long long>(grid, a.unit_end - a.unit_base));
    prefill_kernel<D, M, H><<<g, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_prefill(const FwdProblem& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, unsigned int* status, unsigned long long timeout_ns,
                           cudaStream_t stream) {
  if (p.tiles != nullptr) {
    if (p.d == 64) return launch_d<64, true, false>(p, tq, tk, tv, status, timeout_ns, stream);
    return launch_d<128, true, false>(p, tq, tk, tv, status, timeout_ns, stream);
  }
  if (p.d == 64) return launch_d<64, false, false>(p, tq, tk, tv, status, timeout_ns, stream);
  return launch_d<128, false, false>(p, tq, tk, tv, status, timeout_ns, stream);
}

// Debug builds: read (and optionally clear) this file's device-side check record.
FATTN_DEBUG_ACCESSOR(prefill)

}  // namespace fattn
