// host_staging.cu -- fattn_fwd_host and fattn_decode_host: the device entry points applied to chunks
// of consecutive heads staged through two slots of a caller-owned device workspace, with the host
// copies of one chunk overlapping the kernels of the next.  Contracts are in fattn.h.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "fattn.h"

namespace {

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Two copy streams (host to device, device to host) and the events of two slots, created once per
// device with that device current and kept for the life of the process.
struct Staging {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t in[2] = {nullptr, nullptr};    // a slot's inputs are on the device
  cudaEvent_t out[2] = {nullptr, nullptr};   // a slot's kernels are done
  cudaEvent_t free[2] = {nullptr, nullptr};  // a slot's outputs are back on the host
};

cudaError_t staging(Staging** out) {
  static std::mutex mu;
  static Staging cache[64];
  static bool ready[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  Staging& s = cache[dev];
  if (!ready[dev]) {
    if ((e = cudaStreamCreateWithFlags(&s.h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&s.d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&s.start, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int i = 0; i < 2; ++i) {
      if ((e = cudaEventCreateWithFlags(&s.in[i], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&s.out[i], cudaEventDisableTiming)) != cudaSuccess) return e;
      if ((e = cudaEventCreateWithFlags(&s.free[i], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    ready[dev] = true;
  }
  *out = &s;
  return cudaSuccess;
}

// Heads per chunk: the request, or B*H / `chunks` rounded up.  0 for an invalid request.
long long resolve_chunk(long long BH, int heads_per_chunk, int chunks) {
  if (BH < 1 || heads_per_chunk < 0 || heads_per_chunk > BH) return 0;
  if (heads_per_chunk > 0) return heads_per_chunk;
  return (BH + chunks - 1) / chunks;
}

// Byte offsets of one slot of the forward's workspace, for `hc` heads.
struct FwdSlot {
  size_t q, k, v, o, lse, bytes;
};
FwdSlot fwd_slot(long long hc, long long Nq, long long Nk, long long d) {
  FwdSlot s;
  s.q = 0;
  s.k = s.q + align256(static_cast<size_t>(hc * Nq * d * 2));
  s.v = s.k + align256(static_cast<size_t>(hc * Nk * d * 2));
  s.o = s.v + align256(static_cast<size_t>(hc * Nk * d * 2));
  s.lse = s.o + align256(static_cast<size_t>(hc * Nq * d * 2));
  s.bytes = s.lse + align256(static_cast<size_t>(hc * Nq * 4));
  return s;
}

// ... and of the decode's, for `hc` heads of which only the last `nk` keys are copied.
struct DecSlot {
  size_t q, k, v, o, lse, ws, ws_bytes, bytes;
  int splits;  // split count of a full chunk, used for every chunk so that each fits the slot
};
DecSlot dec_slot(long long hc, long long nk, int d) {
  DecSlot s;
  s.q = 0;
  s.k = s.q + align256(static_cast<size_t>(hc * d * 2));
  s.v = s.k + align256(static_cast<size_t>(hc * nk * d * 2));
  s.o = s.v + align256(static_cast<size_t>(hc * nk * d * 2));
  s.lse = s.o + align256(static_cast<size_t>(hc * d * 2));
  s.ws = s.lse + align256(static_cast<size_t>(hc * 4));
  s.splits = fattn_decode_num_splits(1, static_cast<int>(hc), static_cast<int>(nk), 0);
  s.ws_bytes = fattn_decode_workspace_size(1, static_cast<int>(hc), static_cast<int>(nk), d, s.splits);
  s.bytes = s.ws + align256(s.ws_bytes);
  return s;
}

// The decode copies the keys [key_lo, Nk) of each head.
int decode_key_lo(int Nk, int window_left) {
  return window_left >= 0 && window_left < Nk - 1 ? Nk - 1 - window_left : 0;
}

}  // namespace

namespace {

// Chunk c (slot c % 2): inputs copied on the H2D stream, the device call on `stream`, outputs copied
// back on the D2H stream; a slot is refilled only after its previous chunk's outputs are home.
template <class CopyIn, class Compute, class CopyOut>
fattn_status run_chunks(long long BH, long long hc, char* ws, size_t slot_bytes, cudaStream_t stream,
                        CopyIn copy_in, Compute compute, CopyOut copy_out) {
  Staging* st = nullptr;
  if (staging(&st) != cudaSuccess) return FATTN_ERR_CUDA;
  if (cudaEventRecord(st->start, stream) != cudaSuccess) return FATTN_ERR_CUDA;
  if (cudaStreamWaitEvent(st->h2d, st->start, 0) != cudaSuccess) return FATTN_ERR_CUDA;
  const long long nchunks = (BH + hc - 1) / hc;
  for (long long c = 0; c < nchunks; ++c) {
    const int s = static_cast<int>(c & 1);
    const long long bh0 = c * hc;
    const long long n = BH - bh0 < hc ? BH - bh0 : hc;
    char* slot = ws + s * slot_bytes;
    if (c >= 2 && cudaStreamWaitEvent(st->h2d, st->free[s], 0) != cudaSuccess) return FATTN_ERR_CUDA;
    if (copy_in(slot, bh0, n, st->h2d) != cudaSuccess) return FATTN_ERR_CUDA;
    if (cudaEventRecord(st->in[s], st->h2d) != cudaSuccess) return FATTN_ERR_CUDA;
    if (cudaStreamWaitEvent(stream, st->in[s], 0) != cudaSuccess) return FATTN_ERR_CUDA;
    const fattn_status r = compute(slot, n, stream);
    if (r != FATTN_OK) return r;
    if (cudaEventRecord(st->out[s], stream) != cudaSuccess) return FATTN_ERR_CUDA;
    if (cudaStreamWaitEvent(st->d2h, st->out[s], 0) != cudaSuccess) return FATTN_ERR_CUDA;
    if (copy_out(slot, bh0, n, st->d2h) != cudaSuccess) return FATTN_ERR_CUDA;
    if (cudaEventRecord(st->free[s], st->d2h) != cudaSuccess) return FATTN_ERR_CUDA;
  }
  for (long long c = nchunks - 1; c >= 0 && c >= nchunks - 2; --c)
    if (cudaStreamWaitEvent(stream, st->free[c & 1], 0) != cudaSuccess) return FATTN_ERR_CUDA;
  return FATTN_OK;
}

bool sizes_ok(int B, int H, int N1, int N2) { return B >= 1 && H >= 1 && N1 >= 1 && N2 >= 1; }

}  // namespace

extern "C" {

size_t fattn_fwd_host_workspace_size(int B, int H, int Nq, int Nk, int d, int heads_per_chunk) {
  if (!sizes_ok(B, H, Nq, Nk) || (d != 64 && d != 128)) return 0;
  const long long hc = resolve_chunk(static_cast<long long>(B) * H, heads_per_chunk, 4);
  if (hc == 0) return 0;
  return 2 * fwd_slot(hc, Nq, Nk, d).bytes;
}

fattn_status fattn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                            float* lse_host, int B, int H, int Nq, int Nk, int d, int window_left,
                            int window_right, float scale, int heads_per_chunk, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!q_host || !k_host || !v_host || !o_host || !workspace) return FATTN_ERR_INVALID_ARG;
  if (!sizes_ok(B, H, Nq, Nk) || window_left < -1 || window_right < -1) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 0x7fffffffLL / 64) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FATTN_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long hc = resolve_chunk(BH, heads_per_chunk, 4);
  if (hc == 0) return FATTN_ERR_INVALID_ARG;
  const FwdSlot sl = fwd_slot(hc, Nq, Nk, d);
  if (workspace_bytes < 2 * sl.bytes) return FATTN_ERR_INVALID_ARG;
  const size_t qrow = static_cast<size_t>(Nq) * d * 2, krow = static_cast<size_t>(Nk) * d * 2;
  const char* qh = static_cast<const char*>(q_host);
  const char* kh = static_cast<const char*>(k_host);
  const char* vh = static_cast<const char*>(v_host);
  char* oh = static_cast<char*>(o_host);
  auto copy_in = [&](char* slot, long long bh0, long long n, cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(slot + sl.q, qh + bh0 * qrow, n * qrow, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(slot + sl.k, kh + bh0 * krow, n * krow, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(slot + sl.v, vh + bh0 * krow, n * krow, cudaMemcpyHostToDevice, s);
    return e;
  };
  auto compute = [&](char* slot, long long n, cudaStream_t s) {
    return fattn_fwd_masked(slot + sl.q, slot + sl.k, slot + sl.v, slot + sl.o,
                            reinterpret_cast<float*>(slot + sl.lse), 1, static_cast<int>(n), Nq, Nk, d,
                            window_left, window_right, scale, s);
  };
  auto copy_out = [&](char* slot, long long bh0, long long n, cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(oh + bh0 * qrow, slot + sl.o, n * qrow, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && lse_host)
      e = cudaMemcpyAsync(lse_host + bh0 * Nq, slot + sl.lse, n * Nq * sizeof(float), cudaMemcpyDeviceToHost, s);
    return e;
  };
  return run_chunks(BH, hc, static_cast<char*>(workspace), sl.bytes, static_cast<cudaStream_t>(stream), copy_in,
                    compute, copy_out);
}

size_t fattn_decode_host_workspace_size(int B, int H, int Nk, int d, int window_left, int heads_per_chunk) {
  if (!sizes_ok(B, H, Nk, 1) || (d != 64 && d != 128) || window_left < -1) return 0;
  const long long hc = resolve_chunk(static_cast<long long>(B) * H, heads_per_chunk, 8);
  if (hc == 0) return 0;
  const DecSlot sl = dec_slot(hc, Nk - decode_key_lo(Nk, window_left), d);
  if (sl.ws_bytes == 0) return 0;
  return 2 * sl.bytes;
}

fattn_status fattn_decode_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                               float* lse_host, int B, int H, int Nk, int d, int window_left, int window_right,
                               float scale, int heads_per_chunk, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (!q_host || !k_host || !v_host || !o_host || !workspace) return FATTN_ERR_INVALID_ARG;
  if (!sizes_ok(B, H, Nk, 1) || window_left < -1 || window_right < -1) return FATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FATTN_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long hc = resolve_chunk(BH, heads_per_chunk, 8);
  if (hc == 0) return FATTN_ERR_INVALID_ARG;
  const int key_lo = decode_key_lo(Nk, window_left);
  const int nk = Nk - key_lo;
  const DecSlot sl = dec_slot(hc, nk, d);
  if (sl.ws_bytes == 0 || workspace_bytes < 2 * sl.bytes) return FATTN_ERR_INVALID_ARG;
  if (hc * ((nk + 63) / 64) > 0x7fffffffLL) return FATTN_ERR_INVALID_ARG;
  const size_t qrow = static_cast<size_t>(d) * 2;
  const size_t kpitch = static_cast<size_t>(Nk) * d * 2, kwidth = static_cast<size_t>(nk) * d * 2;
  const char* qh = static_cast<const char*>(q_host);
  const char* kh = static_cast<const char*>(k_host) + static_cast<size_t>(key_lo) * d * 2;
  const char* vh = static_cast<const char*>(v_host) + static_cast<size_t>(key_lo) * d * 2;
  char* oh = static_cast<char*>(o_host);
  auto copy_in = [&](char* slot, long long bh0, long long n, cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(slot + sl.q, qh + bh0 * qrow, n * qrow, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(slot + sl.k, kwidth, kh + bh0 * kpitch, kpitch, kwidth, n, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(slot + sl.v, kwidth, vh + bh0 * kpitch, kpitch, kwidth, n, cudaMemcpyHostToDevice, s);
    return e;
  };
  auto compute = [&](char* slot, long long n, cudaStream_t s) {
    return fattn_decode(slot + sl.q, slot + sl.k, slot + sl.v, slot + sl.o, reinterpret_cast<float*>(slot + sl.lse),
                        1, static_cast<int>(n), nk, d, scale, sl.splits, slot + sl.ws, sl.ws_bytes, s);
  };
  auto copy_out = [&](char* slot, long long bh0, long long n, cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(oh + bh0 * qrow, slot + sl.o, n * qrow, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && lse_host)
      e = cudaMemcpyAsync(lse_host + bh0, slot + sl.lse, n * sizeof(float), cudaMemcpyDeviceToHost, s);
    return e;
  };
  return run_chunks(BH, hc, static_cast<char*>(workspace), sl.bytes, static_cast<cudaStream_t>(stream), copy_in,
                    compute, copy_out);
}

}  // extern "C"
