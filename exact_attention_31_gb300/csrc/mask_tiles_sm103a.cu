// mask_tiles_sm103a.cu -- per-tile summary of an element mask.
//
// A mask is elementwise and independent of the scores ("Understanding FlashAttention", Attention),
// so whole 128 x 128 tiles of it can be judged before any score is computed: a tile with no visible
// key is never loaded or multiplied, a tile with every key visible needs no per-element work, and
// only the tiles in between read the mask bits during the softmax.  This kernel writes that judgement
// (0 = none visible, 1 = some, 2 = all) for every (head, query tile, key tile); the masked forward and
// backward read it.
#include "fattn_internal.h"

namespace fattn {
namespace {

constexpr int kRows = 128;      // query rows per tile (one thread each)
constexpr int kKeys = 128;      // keys per tile (four 32-bit words per row)
constexpr int kTilesPerCta = 8;  // key tiles one CTA judges, one after another

// One CTA per (head, query tile, group of kTilesPerCta key tiles); thread r reads row r's four words
// of each key tile.  Bits of keys >= Nk and rows >= Nq do not count.
__global__ void __launch_bounds__(kRows) mask_tiles_kernel(const uint32_t* mask, long long sb, long long sh,
                                                           int words, int H, int Nq, int Nk, int tq, int tk,
                                                           int groups, uint8_t* tiles) {
  const long long cta = blockIdx.x;
  const int grp = static_cast<int>(cta % groups);
  const long long rest = cta / groups;
  const int qt = static_cast<int>(rest % tq);
  const int bh = static_cast<int>(rest / tq);
  const int row = qt * kRows + static_cast<int>(threadIdx.x);
  const uint4* mrow = nullptr;
  if (row < Nq)
    mrow = reinterpret_cast<const uint4*>(mask + (bh / H) * sb + (bh % H) * sh + static_cast<long long>(row) * words);
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
    if (threadIdx.x == 0)
      tiles[(static_cast<long long>(bh) * tq + qt) * tk + j] = tile_any ? (tile_all ? 2 : 1) : 0;
  }
}

}  // namespace

cudaError_t launch_mask_tiles(const uint32_t* mask, long long mask_sb, long long mask_sh, int mask_words, int B,
                              int H, int Nq, int Nk, uint8_t* tiles, cudaStream_t stream) {
  const int tq = (Nq + kRows - 1) / kRows;
  const int tk = (Nk + kKeys - 1) / kKeys;
  const int groups = (tk + kTilesPerCta - 1) / kTilesPerCta;
  const long long ctas = static_cast<long long>(B) * H * tq * groups;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  mask_tiles_kernel<<<static_cast<unsigned int>(ctas), kRows, 0, stream>>>(mask, mask_sb, mask_sh, mask_words, H, Nq,
                                                                           Nk, tq, tk, groups, tiles);
  return cudaGetLastError();
}

}  // namespace fattn
