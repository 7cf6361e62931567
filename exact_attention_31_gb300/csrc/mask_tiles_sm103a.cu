// mask_tiles_sm103a.cu -- per-tile summary of an element mask.
//
// A mask is elementwise and independent of the scores ("Understanding FlashAttention", Attention),
// so whole 128 x 128 tiles of it can be judged before any score is computed: a tile with no visible
// key is never loaded or multiplied, a tile with every key visible needs no per-element work, and
// only the tiles in between read the mask bits during the softmax.  This kernel writes that judgement
// as two bit sets, `live` (some key of the tile visible) and `partial` (some visible and some
// hidden), in the layout fattn_internal.h describes: by query tile for the forward, whose CTAs walk
// key tiles, and by key tile for the backward, whose CTAs walk query tiles.  A mask shared over
// heads or batch entries (a zero stride) is one slice and is judged once.
#include "fattn_internal.h"

namespace fattn {
namespace {

constexpr int kRows = 128;       // query rows per tile (one thread each)
constexpr int kKeys = 128;       // keys per tile (four 32-bit words per row)
constexpr int kTilesPerCta = 8;  // key tiles one CTA judges, one after another (divides 64)

// One CTA per (slice, query tile, group of kTilesPerCta key tiles); thread r reads row r's four words
// of each key tile and the block's OR and AND give the tile's state, which thread 0 ORs into the
// summary (cleared beforehand).  Bits of keys >= Nk and rows >= Nq do not count.
__global__ void __launch_bounds__(kRows) mask_tiles_kernel(const uint32_t* mask, long long sb, long long sh,
                                                           int words, int mask_nh, int Nq, int Nk, int tq, int tk,
                                                           int groups, bool by_key, unsigned long long* tiles) {
  const long long cta = blockIdx.x;
  const int grp = static_cast<int>(cta % groups);
  const long long rest = cta / groups;
  const int qt = static_cast<int>(rest % tq);
  const int slice = static_cast<int>(rest / tq);
  const int row = qt * kRows + static_cast<int>(threadIdx.x);
  const uint4* mrow = nullptr;
  if (row < Nq)
    mrow = reinterpret_cast<const uint4*>(mask + (slice / mask_nh) * sb + (slice % mask_nh) * sh +
                                          static_cast<long long>(row) * words);
  const int w_key = mask_summary_words(tk), w_query = mask_summary_words(tq);
  unsigned long long live = 0ull, part = 0ull;  // by query tile: this group's bits within its word
  const int j_end = min(tk, (grp + 1) * kTilesPerCta);
  for (int j = grp * kTilesPerCta; j < j_end; ++j) {
    bool any = false, all = true;
    if (mrow != nullptr) {
      const uint4 w4 = __ldg(mrow + j);
      const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int valid_keys = Nk - (j * kKeys + 32 * h);
        const uint32_t valid = valid_keys >= 32 ? ~0u : (valid_keys <= 0 ? 0u : ((1u << valid_keys) - 1u));
        any |= (w[h] & valid) != 0u;
        all &= (w[h] & valid) == valid;
      }
    }
    const bool tile_any = __syncthreads_or(any) != 0;
    const bool tile_all = __syncthreads_and(all) != 0;
    if (by_key) {
      if (threadIdx.x == 0 && tile_any) {
        unsigned long long* col = tiles + (static_cast<long long>(slice) * tk + j) * 2 * w_query + (qt >> 6);
        atomicOr(col, 1ull << (qt & 63));
        if (!tile_all) atomicOr(col + w_query, 1ull << (qt & 63));
      }
    } else {
      if (tile_any) live |= 1ull << (j & 63);
      if (tile_any && !tile_all) part |= 1ull << (j & 63);
    }
  }
  if (!by_key && threadIdx.x == 0) {
    unsigned long long* base =
        tiles + (static_cast<long long>(slice) * tq + qt) * 2 * w_key + (grp * kTilesPerCta) / 64;
    if (live) atomicOr(base, live);
    if (part) atomicOr(base + w_key, part);
  }
}

}  // namespace

cudaError_t launch_mask_tiles(const uint32_t* mask, long long mask_sb, long long mask_sh, int mask_words, int B,
                              int H, int Nq, int Nk, bool by_key, unsigned long long* tiles, cudaStream_t stream) {
  const int mask_nb = mask_sb != 0 ? B : 1, mask_nh = mask_sh != 0 ? H : 1;
  const int tq = (Nq + kRows - 1) / kRows;
  const int tk = (Nk + kKeys - 1) / kKeys;
  const int groups = (tk + kTilesPerCta - 1) / kTilesPerCta;
  const long long ctas = static_cast<long long>(mask_nb) * mask_nh * tq * groups;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(tiles, 0, mask_summary_bytes(mask_nb * mask_nh, Nq, Nk, by_key), stream);
  if (e != cudaSuccess) return e;
  mask_tiles_kernel<<<static_cast<unsigned int>(ctas), kRows, 0, stream>>>(mask, mask_sb, mask_sh, mask_words,
                                                                           mask_nh, Nq, Nk, tq, tk, groups, by_key,
                                                                           tiles);
  return cudaGetLastError();
}

}  // namespace fattn
