// attn_host.cu — the forward pass over host buffers: copies the inputs into
// caller-owned device staging memory, runs attn_prefill_fwd_chunk there and
// copies O and LSE back, all enqueued on the caller's stream. (A deployment
// convenience; the attention itself is the device entry point's.)
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_prefill.h"

namespace gb300_host {
// attn_prefill.cu: every check of attn_prefill_fwd_chunk short of the launch,
// including the device's first-call set-up.
attn_status_t forward_preflight(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, int64_t B, int64_t Lq, int64_t Lk,
                                int32_t n_q, int32_t n_kv, int32_t d_h, int32_t causal,
                                float scale, cudaStream_t stream);
}  // namespace gb300_host

namespace {

constexpr int64_t kAlign = 256;

int64_t round_up(int64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Staging {
  int64_t q, k, v, o, lse, total;   // byte offsets of the regions and the total size
};

// Region layout [q | k | v | o | lse], each 256-byte aligned; total -1 when
// the sizes are invalid.
Staging staging_layout(int64_t B, int64_t Lq, int64_t Lk, int32_t n_q, int32_t n_kv,
                       int32_t d_h) {
  Staging s{0, 0, 0, 0, 0, -1};
  if (B < 1 || Lq < 1 || Lk < Lq || n_q < 1 || n_kv < 1 || n_q % n_kv != 0 ||
      (d_h != 64 && d_h != 128) || Lk > (int64_t{1} << 30) || B > (int64_t{1} << 30))
    return s;
  // keep every byte count far from int64 overflow
  if (static_cast<double>(B) * static_cast<double>(Lk) * (n_q + n_kv) * d_h * 2.0 > 0x1p60)
    return s;
  const int64_t qb = B * Lq * n_q * d_h * 2, kvb = B * Lk * n_kv * d_h * 2;
  const int64_t lb = B * n_q * Lq * 4;
  s.k = round_up(qb);
  s.v = s.k + round_up(kvb);
  s.o = s.v + round_up(kvb);
  s.lse = s.o + round_up(qb);
  s.total = s.lse + round_up(lb);
  return s;
}

}  // namespace

extern "C" {

int64_t attn_prefill_host_staging_bytes(int64_t B, int64_t Lq, int64_t Lk, int32_t n_q,
                                        int32_t n_kv, int32_t d_h) {
  return staging_layout(B, Lq, Lk, n_q, n_kv, d_h).total;
}

attn_status_t attn_prefill_fwd_host(const void* q, const void* k, const void* v, void* o,
                                    float* lse, void* staging, int64_t staging_bytes, int64_t B,
                                    int64_t Lq, int64_t Lk, int32_t n_q, int32_t n_kv,
                                    int32_t d_h, int32_t causal, float scale, void* stream_ptr) {
  if (!q || !k || !v || !o || !lse || !staging) return ATTN_ERR_INVALID_ARG;
  if ((causal != 0 && causal != 1) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(staging) & (kAlign - 1)) != 0) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Lq < 1 || Lk < Lq || n_q < 1 || n_kv < 1 || n_q % n_kv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return ATTN_ERR_UNSUPPORTED;
  const Staging s = staging_layout(B, Lq, Lk, n_q, n_kv, d_h);
  if (s.total < 0) return ATTN_ERR_UNSUPPORTED;
  if (staging_bytes < s.total) return ATTN_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* base = static_cast<uint8_t*>(staging);
  const size_t qb = static_cast<size_t>(B * Lq * n_q * d_h * 2);
  const size_t kvb = static_cast<size_t>(B * Lk * n_kv * d_h * 2);
  const size_t lb = static_cast<size_t>(B * n_q * Lq * 4);
  // Everything the forward could refuse (sizes, the device, a first call
  // during capture) is settled before the first copy is enqueued, so an error
  // return leaves nothing half done on the stream.
  const attn_status_t pre = gb300_host::forward_preflight(
      base + s.q, base + s.k, base + s.v, base + s.o, reinterpret_cast<float*>(base + s.lse), B,
      Lq, Lk, n_q, n_kv, d_h, causal, scale, stream);
  if (pre != ATTN_OK) return pre;
  // one copy per tensor, in, then the forward, then one copy per result, out
  if (cudaMemcpyAsync(base + s.q, q, qb, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(base + s.k, k, kvb, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(base + s.v, v, kvb, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const attn_status_t st = attn_prefill_fwd_chunk(
      base + s.q, base + s.k, base + s.v, base + s.o, reinterpret_cast<float*>(base + s.lse), B,
      Lq, Lk, n_q, n_kv, d_h, causal, scale, stream_ptr);
  if (st != ATTN_OK) return st;
  if (cudaMemcpyAsync(o, base + s.o, qb, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaMemcpyAsync(lse, base + s.lse, lb, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // extern "C"
