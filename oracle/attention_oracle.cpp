// attention_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, fp64 CPU statement of what the fused attention path computes.  It is the
// parity oracle for the CUDA library and shares no code with it.  Only the test suite, the
// package's smoke check and the benchmark's CPU-baseline leg may load it.
//
// Every function is written from the definitions on the pages it cites:
//   [FA-GEM]  "Flash Attention: The Hidden Gem" (ashishkpokharel.com.np/blogs/flash-attention)
//   [FA-IO]   "FlashAttention: attention was never compute-bound" (paperfordummies.in)
//   [FA-UND]  "Understanding FlashAttention" (jimwang99.github.io)
//
// Arithmetic is fp64 throughout, sums are sequential in key order, and fused multiply-add
// contraction is disabled at build time so the results are the same on every host.
//
// Parity status: every exported function is pinned by tests that do not call back into this
// file's arithmetic (closed forms, printed values from [FA-IO] demo 2, a 50-digit brute force,
// and independent restatements of the per-key and tiled recurrences).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <limits>
#include <thread>
#include <vector>

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

// Banded visibility, bottom-right aligned.  With off = Nk - Nq, query row i of Nq may see key j of
// Nk iff  i + off - window_left <= j <= i + off + window_right,  where a negative window means "no
// bound on that side".  No mask is (-1, -1); causal is (-1, 0), the lower triangle j <= i when
// Nq == Nk; a sliding window of W keys is (W - 1, 0).  The pages say only that masks are
// elementwise and independent of the scores, and that causal masking is one of several kinds
// ([FA-UND] "Attention"; [FA-GEM] opening code, is_causal=True); the band family and the
// alignment for Nq != Nk are this file's reading.
inline bool visible(int64_t i, int64_t j, int64_t Nq, int64_t Nk, int64_t wl, int64_t wr) {
    const int64_t c = i + (Nk - Nq);
    if (wr >= 0 && j > c + wr) return false;
    if (wl >= 0 && j < c - wl) return false;
    return true;
}

// One query row of the attention definition, three logical passes as in safe softmax
// ([FA-GEM] "Safe Softmax" and "Why is Flash Attention needed?"; [FA-UND] "Safe softmax"):
//   x_j = scale * <q, k_j>            for every visible key j
//   m   = max_j x_j                   (pass 1)
//   l   = sum_j exp(x_j - m)          (pass 2)
//   o   = sum_j exp(x_j - m) / l * v_j  (pass 3)
//   lse = m + log(l)                  ([FA-GEM] step 6: L = m + log(l))
// Masked keys are excluded outright (their weight is exactly zero).  `mrow`, when given, is an
// element mask for this row over the Nk keys (nonzero = the key may be seen), applied on top of the
// band: a mask is elementwise and independent of the scores ([FA-UND] "Attention").  Returns the
// number of visible keys.  With none visible the max is -inf and -inf minus -inf is undefined ([FA-UND]
// "What is left to the implementation", point 2); such a row gets no weight anywhere: o = 0 and
// lse = log(0) = -inf (this file's reading).
int64_t attention_row(const double* q, const double* k, const double* v, int64_t i, int64_t Nq,
                      int64_t Nk, int64_t d, int64_t wl, int64_t wr, const uint8_t* mrow, double scale,
                      double* x_scratch, double* o, double* lse) {
    int64_t nvis = 0;
    for (int64_t j = 0; j < Nk; ++j) {
        if (!visible(i, j, Nq, Nk, wl, wr) || (mrow != nullptr && mrow[j] == 0)) {
            x_scratch[j] = kNegInf;
            continue;
        }
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t) dot += q[t] * k[j * d + t];
        x_scratch[j] = scale * dot;
        ++nvis;
    }
    if (nvis == 0) {
        for (int64_t t = 0; t < d; ++t) o[t] = 0.0;
        *lse = kNegInf;
        return 0;
    }
    double m = kNegInf;  // pass 1
    for (int64_t j = 0; j < Nk; ++j) m = std::max(m, x_scratch[j]);
    double l = 0.0;  // pass 2
    for (int64_t j = 0; j < Nk; ++j)
        if (x_scratch[j] != kNegInf) l += std::exp(x_scratch[j] - m);
    for (int64_t t = 0; t < d; ++t) o[t] = 0.0;  // pass 3
    for (int64_t j = 0; j < Nk; ++j) {
        if (x_scratch[j] == kNegInf) continue;
        const double p = std::exp(x_scratch[j] - m) / l;
        for (int64_t t = 0; t < d; ++t) o[t] += p * v[j * d + t];
    }
    *lse = m + std::log(l);
    return nvis;
}

template <class F>
void parallel_for(int64_t n, int nthreads, F&& f) {
    if (nthreads <= 1 || n <= 1) {
        for (int64_t r = 0; r < n; ++r) f(r);
        return;
    }
    const int T = static_cast<int>(std::min<int64_t>(nthreads, n));
    std::vector<std::thread> pool;
    pool.reserve(T);
    for (int w = 0; w < T; ++w) {
        pool.emplace_back([&, w]() {
            for (int64_t r = w; r < n; r += T) f(r);
        });
    }
    for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Safe softmax over one vector, three logical passes ([FA-GEM] "Safe Softmax";
// [FA-UND] "Safe softmax"): max, then the exp-sum, then the division.
void oracle_softmax(const double* x, int64_t n, double* y) {
    double m = kNegInf;
    for (int64_t j = 0; j < n; ++j) m = std::max(m, x[j]);
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) l += std::exp(x[j] - m);
    for (int64_t j = 0; j < n; ++j) y[j] = std::exp(x[j] - m) / l;
}

// Online softmax streamed block by block ([FA-IO] "The one formula" and "Online softmax: the
// whole idea"; [FA-GEM] "Online Softmax").  A running max m and running sum l are carried over
// blocks of `block` scores; when a block raises the max, the old sum is multiplied by
// exp(m_old - m_new) before the block's terms exp(x - m_new) are added.  With rescale == 0 that
// multiplication is dropped, which is the deliberately broken variant the page uses to show
// that the correction is load-bearing.  The output vector is exp(x - m_final) / l_final.
void oracle_online_softmax(const double* x, int64_t n, int64_t block, int rescale, double* y) {
    double m = kNegInf;
    double l = 0.0;
    for (int64_t j0 = 0; j0 < n; j0 += block) {
        const int64_t j1 = std::min(n, j0 + block);
        double m_new = m;
        for (int64_t j = j0; j < j1; ++j) m_new = std::max(m_new, x[j]);
        if (rescale && m != kNegInf) l = l * std::exp(m - m_new);
        for (int64_t j = j0; j < j1; ++j) l += std::exp(x[j] - m_new);
        m = m_new;
    }
    for (int64_t j = 0; j < n; ++j) y[j] = std::exp(x[j] - m) / l;
}

// The per-element online normalizer ([FA-UND] "Online softmax"; Milakov & Gimelshein as cited
// there): g_i = max(g_{i-1}, x_i), s_i = s_{i-1} * exp(g_{i-1} - g_i) + exp(x_i - g_i), started
// from g_1 = x_1, s_1 = 1.  Writes the final pair (g_N, s_N).
void oracle_online_normalizer(const double* x, int64_t n, double* g_out, double* s_out) {
    if (n <= 0) {
        *g_out = kNegInf;
        *s_out = 0.0;
        return;
    }
    double g = x[0];
    double s = 1.0;
    for (int64_t i = 1; i < n; ++i) {
        const double g_new = std::max(g, x[i]);
        s = s * std::exp(g - g_new) + std::exp(x[i] - g_new);
        g = g_new;
    }
    *g_out = g;
    *s_out = s;
}

// Attention by its definition, O = softmax(scale * Q K^T + mask) V, plus L = m + log(l) per row
// ([FA-GEM] "Background" and step 6; [FA-UND] "Attention" for the [N,D]/[M,D] shapes and the
// note that batch and heads only repeat independent problems).
//   q: [B,H,Nq,d], k,v: [B,H,Nk,d], o: [B,H,Nq,d], lse: [B,H,Nq]; all row-major fp64.
// The mask is the band (window_left, window_right) described at visible(), and, when `mask` is not
// null, also the element mask [B*H][Nq][Nk] (uint8, nonzero = visible).  Returns the number of rows
// that had no visible key.
int64_t oracle_attention(const double* q, const double* k, const double* v, double* o, double* lse,
                         int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, int64_t window_left,
                         int64_t window_right, const uint8_t* mask, double scale, int nthreads) {
    const int64_t rows = B * H * Nq;
    std::vector<int64_t> empty(static_cast<size_t>(std::max<int64_t>(rows, 1)), 0);
    parallel_for(rows, nthreads, [&](int64_t r) {
        thread_local std::vector<double> xs;
        xs.resize(static_cast<size_t>(Nk));
        const int64_t bh = r / Nq, i = r % Nq;
        const int64_t n = attention_row(q + r * d, k + bh * Nk * d, v + bh * Nk * d, i, Nq, Nk, d,
                                        window_left, window_right, mask ? mask + r * Nk : nullptr, scale,
                                        xs.data(), o + r * d, lse + r);
        empty[static_cast<size_t>(r)] = (n == 0);
    });
    int64_t n_empty = 0;
    for (int64_t r = 0; r < rows; ++r) n_empty += empty[static_cast<size_t>(r)];
    return n_empty;
}

// The same definition for a chosen subset of rows (flat indices into B*H*Nq), so that very
// large problems can be checked on sampled outputs one row at a time.  Row n of the result is
// written to o_rows[n*d ...] and lse_rows[n].
int64_t oracle_attention_rows(const double* q, const double* k, const double* v, const int64_t* rows,
                              int64_t nrows, double* o_rows, double* lse_rows, int64_t B, int64_t H,
                              int64_t Nq, int64_t Nk, int64_t d, int64_t window_left,
                              int64_t window_right, const uint8_t* mask, double scale, int nthreads) {
    (void)B;
    (void)H;
    std::vector<int64_t> empty(static_cast<size_t>(std::max<int64_t>(nrows, 1)), 0);
    parallel_for(nrows, nthreads, [&](int64_t n) {
        thread_local std::vector<double> xs;
        xs.resize(static_cast<size_t>(Nk));
        const int64_t r = rows[n];
        const int64_t bh = r / Nq, i = r % Nq;
        const int64_t cnt = attention_row(q + r * d, k + bh * Nk * d, v + bh * Nk * d, i, Nq, Nk, d,
                                          window_left, window_right, mask ? mask + r * Nk : nullptr, scale,
                                          xs.data(), o_rows + n * d, lse_rows + n);
        empty[static_cast<size_t>(n)] = (cnt == 0);
    });
    int64_t n_empty = 0;
    for (int64_t n = 0; n < nrows; ++n) n_empty += empty[static_cast<size_t>(n)];
    return n_empty;
}

// The probability matrix of one head, P = softmax(scale * Q K^T + mask), row by row with the
// same three passes ([FA-GEM] "Why is Flash Attention needed?", steps 1-2).  p: [Nq, Nk];
// masked entries are exactly 0, and so is every entry of a row with no visible key.  `mask`, when
// not null, is the head's element mask [Nq][Nk] (nonzero = visible), on top of the band.
void oracle_attention_probs(const double* q, const double* k, int64_t Nq, int64_t Nk, int64_t d,
                            int64_t window_left, int64_t window_right, const uint8_t* mask, double scale,
                            double* p) {
    std::vector<double> xs(static_cast<size_t>(Nk));
    for (int64_t i = 0; i < Nq; ++i) {
        double m = kNegInf;
        for (int64_t j = 0; j < Nk; ++j) {
            if (!visible(i, j, Nq, Nk, window_left, window_right) || (mask != nullptr && mask[i * Nk + j] == 0)) {
                xs[j] = kNegInf;
                continue;
            }
            double dot = 0.0;
            for (int64_t t = 0; t < d; ++t) dot += q[i * d + t] * k[j * d + t];
            xs[j] = scale * dot;
            m = std::max(m, xs[j]);
        }
        double l = 0.0;
        for (int64_t j = 0; j < Nk; ++j)
            if (xs[j] != kNegInf) l += std::exp(xs[j] - m);
        for (int64_t j = 0; j < Nk; ++j)
            p[i * Nk + j] = (xs[j] == kNegInf) ? 0.0 : std::exp(xs[j] - m) / l;
    }
}

// Gradients of attention by its definition ("Flash Attention: The Hidden Gem", Phase 2: Gradient
// and the Jacobian, Chain Rule Through a Matrix Multiply, The Softmax Jacobian).  With
// P = softmax(X + mask), X = scale * Q K^T, O = P V and an upstream gradient dO:
//   dV = P^T dO,  dP = dO V^T,  dX_ij = P_ij (dP_ij - D_i)  with  D_i = sum_k dP_ik P_ik,
//   dQ = scale * dX K,  dK = scale * dX^T Q.
// D is computed from the Jacobian form (rowsum(dP o P)), not from the rowsum(dO o O) shortcut, so
// that the shortcut can be checked against it.  The pages write the backward without the scale;
// the factor scale on dQ and dK is the chain rule through X = scale * Q K^T.
//   q, dq: [B,H,Nq,d]; k, v, dk, dv: [B,H,Nk,d]; do_: [B,H,Nq,d]; fp64, row-major.
// Heads are independent and run in parallel.  Masked entries have P = 0, hence dX = 0; a row with
// no visible key has P = 0 throughout and gets dQ = 0.  `mask`, when not null, is the element mask
// [B*H][Nq][Nk] (nonzero = visible), on top of the band.
void oracle_attention_backward(const double* q, const double* k, const double* v, const double* do_,
                               double* dq, double* dk, double* dv, int64_t B, int64_t H, int64_t Nq,
                               int64_t Nk, int64_t d, int64_t window_left, int64_t window_right,
                               const uint8_t* mask, double scale, int nthreads) {
  parallel_for(B * H, nthreads, [&](int64_t bh) {
    const double* Q = q + bh * Nq * d;
    const double* K = k + bh * Nk * d;
    const double* V = v + bh * Nk * d;
    const double* dO = do_ + bh * Nq * d;
    double* dQ = dq + bh * Nq * d;
    double* dK = dk + bh * Nk * d;
    double* dV = dv + bh * Nk * d;
    std::vector<double> P(static_cast<size_t>(Nq * Nk));
    oracle_attention_probs(Q, K, Nq, Nk, d, window_left, window_right, mask ? mask + bh * Nq * Nk : nullptr,
                           scale, P.data());
    for (int64_t x = 0; x < Nk * d; ++x) {
      dK[x] = 0.0;
      dV[x] = 0.0;
    }
    std::vector<double> dP(static_cast<size_t>(Nk));
    std::vector<double> dX(static_cast<size_t>(Nk));
    for (int64_t i = 0; i < Nq; ++i) {
      const double* p = P.data() + i * Nk;
      // dV += P^T dO (row i's contribution)
      for (int64_t j = 0; j < Nk; ++j)
        for (int64_t t = 0; t < d; ++t) dV[j * d + t] += p[j] * dO[i * d + t];
      // dP_i = dO_i V^T
      for (int64_t j = 0; j < Nk; ++j) {
        double acc = 0.0;
        for (int64_t t = 0; t < d; ++t) acc += dO[i * d + t] * V[j * d + t];
        dP[j] = acc;
      }
      // D_i = sum_k dP_ik P_ik; dX_ij = P_ij (dP_ij - D_i)
      double Di = 0.0;
      for (int64_t j = 0; j < Nk; ++j) Di += dP[j] * p[j];
      for (int64_t j = 0; j < Nk; ++j) dX[j] = p[j] * (dP[j] - Di);
      // dQ_i = scale * dX_i K;  dK += scale * dX_i^T Q_i
      for (int64_t t = 0; t < d; ++t) {
        double acc = 0.0;
        for (int64_t j = 0; j < Nk; ++j) acc += dX[j] * K[j * d + t];
        dQ[i * d + t] = scale * acc;
      }
      for (int64_t j = 0; j < Nk; ++j)
        for (int64_t t = 0; t < d; ++t) dK[j * d + t] += scale * dX[j] * Q[i * d + t];
    }
  });
}

}  // extern "C"
