// attn_backward.cu — gradients of the causal GQA attention forward on GB300
// (sm_103a), by recomputation from the saved log-sum-exp.
//
// The backward pass rebuilds each score tile from Q, K and the forward's row
// statistics instead of storing the L x L table ("Long-Context Attention
// Explained" (sevydevy), "What FlashAttention does not change"). With
// P = exp(scale*S - LSE), D_i = dO_i . O_i:
//
//   dV_j = sum_i P_ij dO_i        dP = dO V^T        dS = P * (dP - D)
//   dK_j = scale sum_i dS_ij Q_i  dQ_i = scale sum_j dS_ij K_j
//
// Three kernels, no atomics:
//   rowdot  per query row: -LSE*log2(e) and -D = -dO . O, padded to whole
//           128-row tiles (-inf / 0) so tiles can be fetched with bulk copies;
//   dkdv    one CTA per (b, K/V head, 128-key tile j): loops over the g query
//           heads of the group and the query tiles that see tile j; with the
//           key dimension on the TMEM lanes it computes S^T = K Q^T and
//           dP^T = V dO^T (tcgen05, both operands from shared memory, K_j and
//           V_j resident), turns them into P^T and dS^T (bf16, written back
//           into TMEM) and accumulates dV += P^T dO and dK += dS^T Q (A from
//           TMEM); dK and dV for the whole group stay in TMEM until the end;
//   dq      persistent (one CTA per SM), walking (b, query head, 128-row
//           tile i) units longest first in snake order: S = Q K^T (Q_i in
//           TMEM) and dP = dO V^T (dO_i in shared memory), dS in its own TMEM
//           columns, dQ += dS K over the key tiles it sees; the next unit's
//           K/V tiles stream in while the current unit drains.
// Both tile kernels step over whole 128-column score tiles (128 queries of a
// query tile in dkdv, 128 keys of a key tile in dq), so every product is
// N = 128 (or D) wide, and order their products so that the tensor cores run
// the next tile's scores while the compute warps turn this tile's into P/dS.
//
// Each kernel has a TMA producer warp, an MMA warp (warp-wide loop, one elected
// issuing lane) and kComputeWGs compute warpgroups that split the 128 columns
// of a tile (thread = TMEM lane = tile row; warpgroup w owns columns
// [w*C, w*C + C), C = 128 / kComputeWGs). A warpgroup writes its bf16 P (and
// in dkdv dS) back over the first C/2 of its own, already consumed, fp32
// columns, so no warpgroup ever overwrites columns another one still has to
// read; the products that consume P/dS take their A operand K-step by K-step
// from there.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_prefill.h"
#include "sm103_ptx.cuh"

namespace gb300_host {
attn_status_t device_status_word(cudaStream_t stream, int** status);
}

namespace {

using namespace gb300;

constexpr int kT = 128;                  // rows per query tile and keys per key tile
// One bf16 tile of 128 rows x D (D = 64 or 128 head dimensions): D / 64
// chunks of 128 rows x 128 bytes, 128-byte swizzled.
template <int D>
__host__ __device__ constexpr int tile_bytes() { return kT * D * 2; }
constexpr int kComputeWGs = 2;           // compute warpgroups
constexpr int kColsQ = kT / kComputeWGs;     // dQ: key-tile columns per warpgroup
constexpr int kComputeThreads = 128 * kComputeWGs;
constexpr int kLoadWarp = 4 * kComputeWGs, kMmaWarp = kLoadWarp + 1;
// producer and MMA warps plus two idle warps: registers are granted per
// four warps, so the CTA is a whole number of warpgroups
constexpr int kThreads = kComputeThreads + 128;
constexpr long long kSpinLimit = 1ll << 31;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int L, n_q, n_kv, g, T;   // T = 128-row tiles per sequence
  int causal;
  float c;                  // scale * log2(e)
  float scale;
  const float* nlse2;       // [B, n_q, T*128] -LSE * log2(e), -inf past L
  const float* nrowdot;     // [B, n_q, T*128] -D, 0 past L
  uint16_t* dq;             // bf16 [B, L, n_q, 128]
  uint16_t* dk;             // bf16 [B, L, n_kv, 128]
  uint16_t* dv;
  int* status;
  int q_units;              // dQ work units: B * n_q * T query tiles
};

constexpr int kStages = 3;               // dQ: ring of streamed K/V tiles
constexpr int kStagesKV = 2;             // dK/dV: ring of streamed Q/dO tiles (V_j is resident)

struct Sync {
  uint64_t a_ready;                 // the CTA's fixed A operands are in TMEM
  uint64_t fixed_full;              // dK/dV: V_j has landed in shared memory
  uint64_t full[kStages], empty[kStages];
  uint64_t s_full[2], p_full[2];    // scores ready (commit) / P or dS ready (compute threads)
  uint64_t dp_full, ds_full;        // dP (dP^T) ready (commit) / dS (dS^T) ready (compute threads)
  uint64_t dp_free, dq_done;        // dQ: dP read out (compute threads) / dQ += dS K done (commit)
  uint64_t done, drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, Sync& sy,
                                             const BwdParams& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = clock64_now();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&sy.abort)) return false;
    if (static_cast<long long>(clock64_now() - t0) > kSpinLimit) {
      *reinterpret_cast<volatile int*>(&sy.abort) = 1;
      atomicOr(p.status, 1);
      return false;
    }
  }
}

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = clock64_now();
  while (!mbar_try_wait(bar, parity))
    if (static_cast<long long>(clock64_now() - t0) > kSpinLimit) return;
}

// Plain (non-tensor) bulk copy global -> shared, completion on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
        "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
        "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// TMEM column (relative to the score tile's base) holding the bf16 A operand
// for K step kk (tile columns 16*kk .. 16*kk + 15): warpgroup w packs its
// columns [w*C, w*C + C) two per 32-bit column starting at column w*C.
template <int C>
__host__ __device__ constexpr uint32_t a_col(int kk) {
  return static_cast<uint32_t>((16 * kk / C) * C + (16 * kk % C) / 2);
}

// This thread's row of a bf16 [B, L, H, D] tensor into D/2 TMEM columns of
// its lane, as a tcgen05 A operand (column c = elements 2c, 2c+1, the lower in
// the low half, which is the row's memory order); rows past L become zeros.
template <int D>
__device__ __forceinline__ void row_to_tmem(uint32_t taddr, const uint16_t* src, bool valid) {
#pragma unroll
  for (int half = 0; half < D / 64; ++half) {
    uint32_t w[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (valid) x = reinterpret_cast<const uint4*>(src)[8 * half + q];
      w[4 * q] = x.x;
      w[4 * q + 1] = x.y;
      w[4 * q + 2] = x.z;
      w[4 * q + 3] = x.w;
    }
    tmem_st32(taddr + 32 * half, w);
  }
}

// Scores of a whole tile: D[128 x 128] = A B^T over K = 128, A a fixed operand
// in TMEM, B a [128 rows x 128] K-major tile in shared memory.
template <int D>
__device__ __forceinline__ void mma_scores_full(bool leader, uint32_t d_tmem, uint32_t a_tmem,
                                                uint32_t b_smem) {
  constexpr uint32_t idesc = idesc_bf16_f32(kT, kT, false);
  const uint64_t b0 = sdesc_sw128(b_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * (kT * 128) + (kk & 3) * 32;
    if (leader) mma_ts(d_tmem, a_tmem + 8 * kk, b0 + (off >> 4), idesc, kk > 0 ? 1u : 0u);
  }
}

// D[128 x 128] (+)= A B over K = 128: A the bf16 dS of a whole tile in TMEM
// (a_col<kColsQ> layout), B a [128 rows x 128] tile used MN-major.
template <int D>
__device__ __forceinline__ void mma_accum_full(bool leader, uint32_t d_tmem, uint32_t a_tmem,
                                               uint32_t b_smem, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kT, D, true);
  const uint64_t b0 = sdesc_sw128(b_smem, kT * 128, 1024);
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk)
    if (leader)
      mma_ts(d_tmem, a_tmem + a_col<kColsQ>(kk), b0 + ((kk * 16 * 128) >> 4), idesc,
             (accumulate || kk > 0) ? 1u : 0u);
}

// dQ[128 x D] (+)= dS K over K = 128 keys: dS bf16 in TMEM, packed two keys
// per column (K step kk at column 8*kk), K a [128 keys x D] tile used MN-major.
template <int D>
__device__ __forceinline__ void mma_accum_dq(bool leader, uint32_t d_tmem, uint32_t a_tmem,
                                             uint32_t b_smem, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kT, D, true);
  const uint64_t b0 = sdesc_sw128(b_smem, kT * 128, 1024);
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk)
    if (leader)
      mma_ts(d_tmem, a_tmem + 8 * kk, b0 + ((kk * 16 * 128) >> 4), idesc,
             (accumulate || kk > 0) ? 1u : 0u);
}

// D[128 x 128] = A B^T over K = D: A a [128 rows x D] K-major tile in shared
// memory (dO), B a [128 rows x D] K-major tile (V).
template <int D>
__device__ __forceinline__ void mma_scores_full_ss(bool leader, uint32_t d_tmem, uint32_t a_smem,
                                                   uint32_t b_smem) {
  constexpr uint32_t idesc = idesc_bf16_f32(kT, kT, false);
  const uint64_t a0 = sdesc_sw128(a_smem, 16, 1024);
  const uint64_t b0 = sdesc_sw128(b_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * (kT * 128) + (kk & 3) * 32) >> 4;
    if (leader) mma_ss(d_tmem, a0 + off, b0 + off, idesc, kk > 0 ? 1u : 0u);
  }
}

__device__ __forceinline__ void setup(Sync& sy) {
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&sy.a_ready), kComputeThreads);
    mbar_init(smem_addr(&sy.fixed_full), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&sy.full[s]), 1);
      mbar_init(smem_addr(&sy.empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&sy.s_full[s]), 1);
      mbar_init(smem_addr(&sy.p_full[s]), kComputeThreads);
    }
    mbar_init(smem_addr(&sy.dp_full), 1);
    mbar_init(smem_addr(&sy.ds_full), kComputeThreads);
    mbar_init(smem_addr(&sy.dp_free), kComputeThreads);
    mbar_init(smem_addr(&sy.dq_done), 1);
    mbar_init(smem_addr(&sy.done), 1);
    mbar_init(smem_addr(&sy.drain), 1);
    sy.abort = 0;
    fence_mbar_init();
  }
  if ((threadIdx.x >> 5) == kMmaWarp) {
    tmem_alloc(smem_addr(&sy.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
}

__device__ __forceinline__ void teardown(Sync& sy, const BwdParams& p, bool leader_mma) {
  if ((threadIdx.x >> 5) == kMmaWarp) {
    if (leader_mma) mma_commit(smem_addr(&sy.drain));
    wait_drain(smem_addr(&sy.drain), 0);
    __syncwarp();
  }
  tc_fence_before_sync();
  __syncthreads();
  if ((threadIdx.x >> 5) == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(sy.tmem_base, 512);
  }
}

// 32 bf16 outputs of this thread's row from 32 fp32 TMEM columns, times `mul`.
__device__ __forceinline__ void store_chunk(uint32_t taddr, uint16_t* dst, float mul, bool valid) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
  tmem_wait_ld(v);
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    w[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
  if (valid) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) d4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}

// dK/dV phase 1 for one warpgroup: P^T = 2^(c S^T + nl) for its kColsQ query
// columns of this thread's key row (S^T read from TMEM at `taddr`, the row
// statistics nl from shared memory), kept in `pr` and written back as bf16
// over the first consumed columns. kMask: the diagonal tile, where query
// column q0 + k is masked when q0 + k < r (q_minus_r = q0 - r).
template <bool kMask>
__device__ __forceinline__ void pt_from_st(uint32_t taddr, const float4* nl4, uint64_t c2,
                                           int q_minus_r, float (&pr)[kColsQ]) {
#pragma unroll
  for (int cc = 0; cc < kColsQ / 32; ++cc) {
    uint32_t sv[32];
    tmem_ld32(taddr + 32 * cc, sv);
    tmem_wait_ld(sv);
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float4 nl = nl4[8 * cc + e];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int jj = 4 * e + 2 * h2;
        const uint64_t x = ffma2(f32x2_pack(__uint_as_float(sv[jj]), __uint_as_float(sv[jj + 1])),
                                 c2, h2 ? f32x2_pack(nl.z, nl.w) : f32x2_pack(nl.x, nl.y));
        float x0, x1;
        f32x2_unpack(x, x0, x1);
        float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        if (kMask) {
          if (q_minus_r + 32 * cc + jj < 0) p0 = 0.0f;
          if (q_minus_r + 32 * cc + jj + 1 < 0) p1 = 0.0f;
        }
        pr[32 * cc + jj] = p0;
        pr[32 * cc + jj + 1] = p1;
        pk[jj / 2] = pack_bf16x2(p0, p1);
      }
    }
    tmem_st16(taddr + 16 * cc, pk);
  }
}

// dQ phase 1 for one warpgroup: P = 2^(c S + nl) for its kColsQ key columns
// [k0, k0 + kColsQ) of this thread's query row, kept in `pr`. kMask: keys
// after in-tile index `keep` are masked (the diagonal tile, or keys past L).
template <bool kMask>
__device__ __forceinline__ void p_from_s(uint32_t taddr, uint64_t c2, uint64_t nl2, int k0,
                                         int keep, float (&pr)[kColsQ]) {
#pragma unroll
  for (int c = 0; c < kColsQ / 32; ++c) {
    uint32_t sv[32];
    tmem_ld32(taddr + 32 * c, sv);
    tmem_wait_ld(sv);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint64_t x = ffma2(
          f32x2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), c2, nl2);
      float x0, x1;
      f32x2_unpack(x, x0, x1);
      float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      if (kMask) {
        if (k0 + 32 * c + 2 * e > keep) p0 = 0.0f;
        if (k0 + 32 * c + 2 * e + 1 > keep) p1 = 0.0f;
      }
      pr[32 * c + 2 * e] = p0;
      pr[32 * c + 2 * e + 1] = p1;
    }
  }
}

// ------------------------------------------------------------------ rowdot

// Half a warp per padded row (b, h, t), t < Lp: 16 lanes x 8 dimensions, with
// 16-byte loads; a warp takes four rows at a time so that its loads of all
// four are in flight together, and walks the rows grid-stride (at most eight
// blocks per SM: a long-lived grid instead of thousands of short blocks).
// Rows past L get -inf and 0 without touching O or dO. The dK/dV kernel is
// launched as this grid's programmatic dependent and waits for it before it
// reads the statistics.
constexpr int kRowdotRowsPerWarp = 4;
__device__ __forceinline__ float dot2_bf16(uint32_t a, uint32_t d, float acc) {
  acc = fmaf(__uint_as_float(a << 16), __uint_as_float(d << 16), acc);
  return fmaf(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(d & 0xFFFF0000u), acc);
}
__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 d) {
  float acc = __uint_as_float(a.x << 16) * __uint_as_float(d.x << 16);
  acc = fmaf(__uint_as_float(a.x & 0xFFFF0000u), __uint_as_float(d.x & 0xFFFF0000u), acc);
  acc = fmaf(__uint_as_float(a.y << 16), __uint_as_float(d.y << 16), acc);
  acc = fmaf(__uint_as_float(a.y & 0xFFFF0000u), __uint_as_float(d.y & 0xFFFF0000u), acc);
  acc = fmaf(__uint_as_float(a.z << 16), __uint_as_float(d.z << 16), acc);
  acc = fmaf(__uint_as_float(a.z & 0xFFFF0000u), __uint_as_float(d.z & 0xFFFF0000u), acc);
  acc = fmaf(__uint_as_float(a.w << 16), __uint_as_float(d.w << 16), acc);
  acc = fmaf(__uint_as_float(a.w & 0xFFFF0000u), __uint_as_float(d.w & 0xFFFF0000u), acc);
  return acc;
}

// Lanes of a half-warp hold D / 16 dimensions each (8 for D = 128: one
// 16-byte load; 4 for D = 64: the first half of it).
template <int D>
__global__ void rowdot_kernel(const uint16_t* o, const uint16_t* dout, const float* lse,
                              float* nlse2, float* nrowdot, int B, int L, int n_q, int Lp) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t total = static_cast<int64_t>(B) * n_q * Lp;
  const int64_t warps = (total + kRowdotRowsPerWarp - 1) / kRowdotRowsPerWarp;
  const int64_t wstride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int half = (threadIdx.x >> 4) & 1, l16 = threadIdx.x & 15;
  for (int64_t warp_id = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       warp_id < warps; warp_id += wstride) {
  uint4 a[kRowdotRowsPerWarp / 2], d[kRowdotRowsPerWarp / 2];
  bool live[kRowdotRowsPerWarp / 2];
#pragma unroll
  for (int k = 0; k < kRowdotRowsPerWarp / 2; ++k) {
    const int64_t row = warp_id * kRowdotRowsPerWarp + 2 * k + half;
    live[k] = false;
    a[k] = d[k] = make_uint4(0u, 0u, 0u, 0u);
    if (row < total) {
      const int t = static_cast<int>(row % Lp);
      const int64_t bh = row / Lp;
      if (t < L) {
        const int h = static_cast<int>(bh % n_q);
        const int b = static_cast<int>(bh / n_q);
        const size_t off = ((static_cast<size_t>(b) * L + t) * n_q + h) * D + (D / 16) * l16;
        if (D == 128) {
          a[k] = *reinterpret_cast<const uint4*>(o + off);
          d[k] = *reinterpret_cast<const uint4*>(dout + off);
        } else {
          const uint2 a2 = *reinterpret_cast<const uint2*>(o + off);
          const uint2 d2 = *reinterpret_cast<const uint2*>(dout + off);
          a[k] = make_uint4(a2.x, a2.y, 0u, 0u);
          d[k] = make_uint4(d2.x, d2.y, 0u, 0u);
        }
        live[k] = true;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kRowdotRowsPerWarp / 2; ++k) {
    float dd = 0.0f;
    if (live[k]) dd = (D == 128) ? dot8_bf16(a[k], d[k])
                                 : dot2_bf16(a[k].y, d[k].y, dot2_bf16(a[k].x, d[k].x, 0.0f));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, off);
    const int64_t row = warp_id * kRowdotRowsPerWarp + 2 * k + half;
    if (l16 == 0 && row < total) {
      const int t = static_cast<int>(row % Lp);
      nrowdot[row] = -dd;
      nlse2[row] = (t < L) ? -lse[(row / Lp) * L + t] * kLog2e : -INFINITY;
    }
  }
  }
}

// -------------------------------------------------------------------- dK, dV

// Producer side shared by both tile kernels: drains the ring so that no copy is
// still in flight when the CTA exits; `issued` tiles were put in flight.
template <int S>
__device__ __forceinline__ void drain_ring(Sync& sy, int issued) {
  for (int s = 0; s < S && s < issued; ++s) {
    const int last = s + ((issued - 1 - s) / S) * S;
    wait_drain(smem_addr(&sy.full[s]), (last / S) & 1);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
            const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
            const BwdParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Sync sy;
  // smem: K_j | V_j | kStagesKV x [Q_i | dO_i | -LSE*log2 e [128] | -D [128]]
  constexpr int kTileBytes = tile_bytes<D>();
  const uint32_t base = (smem_addr(dyn_smem) + 1023u) & ~1023u;
  const uint32_t sK = base, sV = base + kTileBytes, sRing = base + 2 * kTileBytes;
  constexpr uint32_t kStage = 2 * kTileBytes + 1024;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = static_cast<int>(gridDim.x) / p.T;
  const int j = blockIdx.x / groups;                  // key tile (ascending = most work first)
  const int grp = blockIdx.x - j * groups;
  const int b = grp / p.n_kv, kvh = grp - b * p.n_kv;
  const int i0 = p.causal ? j : 0;
  const int nsteps = p.g * (p.T - i0);                 // (head, query tile) pairs
  setup(sy);
  // Launched as the row kernel's programmatic dependent: the set-up above
  // overlaps its end; the row statistics are read only after it completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The dQ kernel (this grid's programmatic dependent) reads nothing this
  // kernel writes: its CTAs may take SMs as soon as every CTA here is past
  // the wait above (so the row statistics are complete when dQ starts).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t tmem = sy.tmem_base;
  // TMEM columns: S^T 0..127 (P^T, bf16, is written over it), dP^T 128..255
  // (dS^T over it), dV at 256 and dK at 256 + D (D columns each). Each step
  // is a whole 128-query tile, so every product has N = 128 (or D): the
  // tensor cores get 64-cycle MMAs, which one issuing thread keeps up with.
  constexpr uint32_t cS = 0, cP = 128, cDV = 256, cDK = 256 + D;

  if (warp == kLoadWarp) {
    if (lane == 0) {
      const uint32_t fb = smem_addr(&sy.fixed_full);
      mbar_arrive_expect_tx(fb, 2 * kTileBytes);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_4d(sK + c * kT * 128, &tmK, fb, c * 64, kvh, j * kT, b);
        tma_load_4d(sV + c * kT * 128, &tmV, fb, c * 64, kvh, j * kT, b);
      }
      int t = 0;
      for (; t < nsteps; ++t) {
        const int st = t % kStagesKV, use = t / kStagesKV;
        if (use > 0 && !wait_bounded(smem_addr(&sy.empty[st]), (use - 1) & 1, sy, p)) break;
        const int h = kvh * p.g + t / (p.T - i0);
        const int i = i0 + t % (p.T - i0);
        const uint32_t dst = sRing + st * kStage, bar = smem_addr(&sy.full[st]);
        mbar_arrive_expect_tx(bar, 2 * kTileBytes + 1024);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(dst + c * kT * 128, &tmQ, bar, c * 64, h, i * kT, b);
          tma_load_4d(dst + kTileBytes + c * kT * 128, &tmdO, bar, c * 64, h, i * kT, b);
        }
        const size_t row0 = (static_cast<size_t>(b) * p.n_q + h) * (p.T * kT) + i * kT;
        bulk_load(dst + 2 * kTileBytes, p.nlse2 + row0, 512, bar);
        bulk_load(dst + 2 * kTileBytes + 512, p.nrowdot + row0, 512, bar);
      }
      wait_drain(fb, 0);
      drain_ring<kStagesKV>(sy, t);
    }
  } else if (warp == kMmaWarp) {
    const bool leader = elect_one();
    bool ok = __all_sync(0xffffffffu, wait_bounded(smem_addr(&sy.fixed_full), 0, sy, p));
    tc_fence_after_sync();
    auto stage_of = [&](int t) { return sRing + (t % kStagesKV) * kStage; };
    auto wait_stage = [&](int t) -> bool {
      if (!__all_sync(0xffffffffu, wait_bounded(smem_addr(&sy.full[t % kStagesKV]),
                                                (t / kStagesKV) & 1, sy, p)))
        return false;
      tc_fence_after_sync();
      return true;
    };
    auto wait_all = [&](uint64_t& bar, int t) -> bool {
      if (!__all_sync(0xffffffffu, wait_bounded(smem_addr(&bar), t & 1, sy, p))) return false;
      tc_fence_after_sync();
      return true;
    };
    if (ok && (ok = wait_stage(0))) {
      mma_scores_full_ss<D>(leader, tmem + cS, sK, stage_of(0));                  // S^T  = K Q^T
      if (leader) mma_commit(smem_addr(&sy.s_full[0]));
      mma_scores_full_ss<D>(leader, tmem + cP, sV, stage_of(0) + kTileBytes);     // dP^T = V dO^T
      if (leader) mma_commit(smem_addr(&sy.dp_full));
    }
    for (int t = 0; t < nsteps && ok; ++t) {
      const uint32_t sQ = stage_of(t), sdO = sQ + kTileBytes;
      const bool more = t + 1 < nsteps;
      if (!wait_all(sy.p_full[0], t)) break;
      mma_accum_full<D>(leader, tmem + cDV, tmem + cS, sdO, t > 0);              // dV += P^T dO
      // S^T(t+1) overwrites P^T(t), which the dV product issued above reads first
      if (more) {
        if (!wait_stage(t + 1)) break;
        mma_scores_full_ss<D>(leader, tmem + cS, sK, stage_of(t + 1));
        if (leader) mma_commit(smem_addr(&sy.s_full[0]));
      }
      if (!wait_all(sy.ds_full, t)) break;
      mma_accum_full<D>(leader, tmem + cDK, tmem + cP, sQ, t > 0);               // dK += dS^T Q
      if (leader) mma_commit(smem_addr(&sy.empty[t % kStagesKV]));
      if (more) {
        mma_scores_full_ss<D>(leader, tmem + cP, sV, stage_of(t + 1) + kTileBytes);
        if (leader) mma_commit(smem_addr(&sy.dp_full));
      }
    }
    if (leader) mma_commit(smem_addr(&sy.done));
    teardown(sy, p, leader);
    return;
  } else if (warp < 4 * kComputeWGs) {
    // compute warpgroups: thread r = key row r of the tile = TMEM lane r;
    // warpgroup cw takes query columns [cw*kColsQ, cw*kColsQ + kColsQ) of a step
    const int cw = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int krow = j * kT + r;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const size_t koff = ((static_cast<size_t>(b) * p.L + krow) * p.n_kv + kvh) * D;
    const uint64_t c2 = f32x2_pack(p.c, p.c);
    const int q0 = cw * kColsQ;                        // first query column (in the tile)
    bool ok = true;
    for (int t = 0; t < nsteps; ++t) {
      const int st = t % kStagesKV;
      const int i = i0 + t % (p.T - i0);
      if (!__all_sync(0xffffffffu, wait_bounded(smem_addr(&sy.s_full[0]), t & 1, sy, p)) ||
          // the staged row statistics arrived with the stage's copies
          !__all_sync(0xffffffffu,
                      wait_bounded(smem_addr(&sy.full[st]), (t / kStagesKV) & 1, sy, p))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float4* nl4 = reinterpret_cast<const float4*>(
          dyn_smem + (sRing + st * kStage + 2 * kTileBytes - smem_addr(dyn_smem))) + q0 / 4;
      const float4* nd4 = nl4 + 32;
      const bool diag = p.causal && i == j;           // query c < key r is masked
      // phase 1: P^T from S^T, kept in registers for phase 2, and written (bf16)
      // over this warpgroup's first consumed S^T columns
      float pr[kColsQ];
      // the causal mask only touches the diagonal tile: a separate copy of the
      // loop keeps its compares and selects out of every other tile
      if (diag) pt_from_st<true>(lane_base + cS + q0, nl4, c2, q0 - r, pr);
      else pt_from_st<false>(lane_base + cS + q0, nl4, c2, q0 - r, pr);
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(smem_addr(&sy.p_full[0]));
      // phase 2: dS^T = P^T * (dP^T - D), over this warpgroup's consumed dP^T columns
      if (!__all_sync(0xffffffffu, wait_bounded(smem_addr(&sy.dp_full), t & 1, sy, p))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
#pragma unroll
      for (int cc = 0; cc < kColsQ / 32; ++cc) {
        uint32_t dpv[32];
        tmem_ld32(lane_base + cP + q0 + 32 * cc, dpv);
        tmem_wait_ld(dpv);
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 nd = nd4[8 * cc + e];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int jj = 4 * e + 2 * h2;
            const uint64_t dd = fadd2(
                f32x2_pack(__uint_as_float(dpv[jj]), __uint_as_float(dpv[jj + 1])),
                h2 ? f32x2_pack(nd.z, nd.w) : f32x2_pack(nd.x, nd.y));
            float d0, d1;
            f32x2_unpack(fmul2(f32x2_pack(pr[32 * cc + jj], pr[32 * cc + jj + 1]), dd), d0, d1);
            dk[jj / 2] = pack_bf16x2(d0, d1);
          }
        }
        tmem_st16(lane_base + cP + q0 + 16 * cc, dk);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(smem_addr(&sy.ds_full));
    }
    if (ok && __all_sync(0xffffffffu, wait_bounded(smem_addr(&sy.done), 0, sy, p))) {
      tc_fence_after_sync();
      const bool valid = krow < p.L;
      // 2*D/32 chunks of 32 columns (dV then dK) shared out over the warpgroups
      constexpr int kOut = 2 * D / 32, kPer = kOut / kComputeWGs, kHalfOut = D / 32;
#pragma unroll 1
      for (int q = cw * kPer; q < (cw + 1) * kPer; ++q) {
        const int col = (q % kHalfOut) * 32;
        if (q < kHalfOut) store_chunk(lane_base + cDV + col, p.dv + koff + col, 1.0f, valid);
        else store_chunk(lane_base + cDK + col, p.dk + koff + col, p.scale, valid);
      }
    }
  }
  teardown(sy, p, false);
}

// ------------------------------------------------------------------------ dQ

// dQ unit u (longest first): query tile i = T - 1 - u / groups of head
// (b, h) = u % groups, groups = B * n_q.
struct DqUnit {
  int b, h, i, n;
};
__device__ __forceinline__ DqUnit dq_unit(int u, const BwdParams& p) {
  const int groups = p.q_units / p.T;
  DqUnit x;
  x.i = p.T - 1 - u / groups;
  const int grp = u - (p.T - 1 - x.i) * groups;
  x.b = grp / p.n_q;
  x.h = grp - x.b * p.n_q;
  x.n = p.causal ? x.i + 1 : p.T;
  return x;
}

// Persistent: one CTA per SM walks the units in snake order (round r takes
// units r*G .. r*G+G-1, left to right on even rounds, right to left on odd
// ones), so each CTA's set-up happens once and the next unit's K/V tiles
// stream in while the current one drains.
__device__ __forceinline__ int dq_snake(int r) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
dq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
          const __grid_constant__ CUtensorMap tmdO, const uint16_t* __restrict__ q_rows,
          const BwdParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Sync sy;
  // smem: dO_i | kStages x [K_t | V_t]
  constexpr int kTileBytes = tile_bytes<D>();
  const uint32_t base = (smem_addr(dyn_smem) + 1023u) & ~1023u;
  const uint32_t sdO = base, sRing = base + kTileBytes;
  constexpr uint32_t kStage = 2 * kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = p.q_units;
  const int G = static_cast<int>(gridDim.x);
  setup(sy);
  const uint32_t tmem = sy.tmem_base;
  // TMEM columns: Q_i at 0 (D/2 columns, the A operand of S), S 64..191,
  // dP 192..319, dS 320..383 (bf16, two keys per column), dQ 384..511.
  // dP is read out before dS is formed and dS has its own columns, so per key
  // tile t the tensor cores run S(t+1) and dP(t+1) while the compute warps
  // still work on tile t, and dQ(t) as soon as dS(t) is in. Barrier phases
  // count tiles and units over the CTA's whole walk.
  constexpr uint32_t cQ = 0, cS = 64, cP = 192, cDS = 320, cDQ = 384;

  if (warp == kLoadWarp) {
    if (lane == 0) {
      const uint32_t fb = smem_addr(&sy.fixed_full);
      int it = 0, uc = 0;
      bool ok = true;
      for (int r = 0; r * G < units && ok; ++r) {
        const int u = dq_snake(r);
        if (u >= units) continue;
        const DqUnit x = dq_unit(u, p);
        const int kvh = x.h / p.g;
        // The first ring's worth of this unit's K/V tiles goes out while the
        // previous unit still runs; dO_i's buffer is free only once every
        // product of the previous unit is done.
        const int pre = x.n < kStages ? x.n : kStages;
        for (int t = 0; t < x.n; ++t, ++it) {
          if (t == pre) {
            if (uc > 0 && !wait_bounded(smem_addr(&sy.done), (uc - 1) & 1, sy, p)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(fb, kTileBytes);
            for (int c = 0; c < D / 64; ++c)
              tma_load_4d(sdO + c * kT * 128, &tmdO, fb, c * 64, x.h, x.i * kT, x.b);
            ++uc;
          }
          const int st = it % kStages, use = it / kStages;
          if (use > 0 && !wait_bounded(smem_addr(&sy.empty[st]), (use - 1) & 1, sy, p)) {
            ok = false;
            break;
          }
          const uint32_t dst = sRing + st * kStage, bar = smem_addr(&sy.full[st]);
          mbar_arrive_expect_tx(bar, 2 * kTileBytes);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_4d(dst + c * kT * 128, &tmK, bar, c * 64, kvh, t * kT, x.b);
            tma_load_4d(dst + kTileBytes + c * kT * 128, &tmV, bar, c * 64, kvh, t * kT, x.b);
          }
        }
        if (ok && pre == x.n) {
          // every tile fitted in the ring ahead of dO
          if (uc > 0 && !wait_bounded(smem_addr(&sy.done), (uc - 1) & 1, sy, p)) break;
          mbar_arrive_expect_tx(fb, kTileBytes);
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(sdO + c * kT * 128, &tmdO, fb, c * 64, x.h, x.i * kT, x.b);
          ++uc;
        }
      }
      if (uc > 0) wait_drain(fb, (uc - 1) & 1);
      drain_ring<kStages>(sy, it);
    }
  } else if (warp == kMmaWarp) {
    const bool leader = elect_one();
    int it = 0, gt = 0, uc = 0;      // ring items, tiles, units consumed so far
    bool ok = true;
    auto wait_all = [&](uint64_t& bar, int ph) -> bool {
      if (!__all_sync(0xffffffffu, wait_bounded(smem_addr(&bar), ph & 1, sy, p))) return false;
      tc_fence_after_sync();
      return true;
    };
    for (int r = 0; r * G < units && ok; ++r) {
      const int u = dq_snake(r);
      if (u >= units) continue;
      const int n = dq_unit(u, p).n;
      auto stage_of = [&](int t) { return sRing + ((it + t) % kStages) * kStage; };
      auto wait_stage = [&](int t) -> bool {
        return wait_all(sy.full[(it + t) % kStages], (it + t) / kStages);
      };
      // Q_i in TMEM (compute threads) and dO_i in shared memory
      if (!wait_all(sy.a_ready, uc) || !wait_all(sy.fixed_full, uc) || !wait_stage(0)) {
        ok = false;
        break;
      }
      mma_scores_full<D>(leader, tmem + cS, tmem + cQ, stage_of(0));           // S  = Q K^T
      if (leader) mma_commit(smem_addr(&sy.s_full[0]));
      mma_scores_full_ss<D>(leader, tmem + cP, sdO, stage_of(0) + kTileBytes);  // dP = dO V^T
      if (leader) mma_commit(smem_addr(&sy.dp_full));
      for (int t = 0; t < n; ++t) {
        const bool more = t + 1 < n;
        // S(t) read out: the next tile's scores may overwrite it
        if (!wait_all(sy.p_full[0], gt + t)) { ok = false; break; }
        if (more) {
          if (!wait_stage(t + 1)) { ok = false; break; }
          mma_scores_full<D>(leader, tmem + cS, tmem + cQ, stage_of(t + 1));
          if (leader) mma_commit(smem_addr(&sy.s_full[0]));
        }
        // dP(t) read out: the next tile's dP may overwrite it
        if (!wait_all(sy.dp_free, gt + t)) { ok = false; break; }
        if (more) {
          mma_scores_full_ss<D>(leader, tmem + cP, sdO, stage_of(t + 1) + kTileBytes);
          if (leader) mma_commit(smem_addr(&sy.dp_full));
        }
        if (!wait_all(sy.ds_full, gt + t)) { ok = false; break; }
        mma_accum_dq<D>(leader, tmem + cDQ, tmem + cDS, stage_of(t), t > 0);      // dQ += dS K
        if (leader) mma_commit(smem_addr(&sy.dq_done));
        if (leader) mma_commit(smem_addr(&sy.empty[(it + t) % kStages]));
      }
      if (!ok) break;
      if (leader) mma_commit(smem_addr(&sy.done));
      it += n;
      gt += n;
      ++uc;
    }
    teardown(sy, p, leader);
    return;
  } else if (warp < 4 * kComputeWGs) {
    // compute warpgroups: thread r = query row r of the tile = TMEM lane r;
    // warpgroup cw takes key columns [cw*kColsQ, cw*kColsQ + kColsQ)
    const int cw = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint64_t c2 = f32x2_pack(p.c, p.c);
    const int k0 = cw * kColsQ;                        // first key column (in the tile)
    int gt = 0, uc = 0;
    bool ok = true;
    for (int rr = 0; rr * G < units && ok; ++rr) {
      const int u = dq_snake(rr);
      if (u >= units) continue;
      const DqUnit x = dq_unit(u, p);
      const int i = x.i, n = x.n;
      const int row = i * kT + r;
      const size_t qoff = ((static_cast<size_t>(x.b) * p.L + row) * p.n_q + x.h) * D;
      // Q_i becomes the A operand of S in TMEM (first warpgroup); the previous
      // unit's products are all done (its epilogue waited for them)
      if (cw == 0) row_to_tmem<D>(lane_base + cQ, q_rows + qoff, row < p.L);
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(smem_addr(&sy.a_ready));
      const size_t srow = (static_cast<size_t>(x.b) * p.n_q + x.h) * (p.T * kT) + row;
      const float nl = p.nlse2[srow], nd = p.nrowdot[srow];
      const uint64_t nl2 = f32x2_pack(nl, nl), nd2 = f32x2_pack(nd, nd);
      for (int t = 0; t < n; ++t) {
        // phase 1: P from S, kept in registers
        if (!__all_sync(0xffffffffu, wait_bounded(smem_addr(&sy.s_full[0]), (gt + t) & 1, sy, p))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        // keys after `keep` (in-tile) are masked: the diagonal tile, or keys past L
        const bool masked = p.causal ? (t == i) : (p.L - t * kT < kT);
        const int keep = p.causal ? r : p.L - 1 - t * kT;
        float pr[kColsQ];
        if (masked) p_from_s<true>(lane_base + cS + k0, c2, nl2, k0, keep, pr);
        else p_from_s<false>(lane_base + cS + k0, c2, nl2, k0, keep, pr);
        tc_fence_before_sync();
        mbar_arrive(smem_addr(&sy.p_full[0]));
        // phase 2: dP read out (its columns are then free for the next tile),
        // dS = P * (dP - D) into the dS columns once dQ(t-1) has read them
        if (!__all_sync(0xffffffffu, wait_bounded(smem_addr(&sy.dp_full), (gt + t) & 1, sy, p))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t dk[kColsQ / 2];
#pragma unroll
        for (int c = 0; c < kColsQ / 32; ++c) {
          uint32_t dpv[32];
          tmem_ld32(lane_base + cP + k0 + 32 * c, dpv);
          tmem_wait_ld(dpv);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t dd = fadd2(
                f32x2_pack(__uint_as_float(dpv[2 * e]), __uint_as_float(dpv[2 * e + 1])), nd2);
            float d0, d1;
            f32x2_unpack(fmul2(f32x2_pack(pr[32 * c + 2 * e], pr[32 * c + 2 * e + 1]), dd), d0, d1);
            dk[16 * c + e] = pack_bf16x2(d0, d1);
          }
        }
        tc_fence_before_sync();
        mbar_arrive(smem_addr(&sy.dp_free));
        if (t > 0 && !__all_sync(0xffffffffu, wait_bounded(smem_addr(&sy.dq_done), (gt + t - 1) & 1, sy, p))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < kColsQ / 32; ++c)
          tmem_st16(lane_base + cDS + k0 / 2 + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(dk + 16 * c));
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(smem_addr(&sy.ds_full));
      }
      if (!ok || !__all_sync(0xffffffffu, wait_bounded(smem_addr(&sy.done), uc & 1, sy, p))) break;
      tc_fence_after_sync();
      constexpr int kPer = (D / 32) / kComputeWGs;    // chunks of 32 dQ columns per warpgroup
#pragma unroll 1
      for (int q = cw * kPer; q < (cw + 1) * kPer; ++q)
        store_chunk(lane_base + cDQ + 32 * q, p.dq + qoff + 32 * q, p.scale, row < p.L);
      gt += n;
      ++uc;
    }
  }
  teardown(sy, p, false);
  // This grid started while dK/dV still ran (it reads nothing dK/dV writes);
  // it ends only once dK/dV has ended (one waiting thread keeps the CTA
  // alive; every thread waiting cost 1.4 %), so that a programmatic dependent
  // of this grid (the stream's next kernel) finds dK and dV complete as well.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// --------------------------------------------------------------------- host

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
constexpr int kMaxDevices = 64;
std::mutex g_bwd_mutex;
bool g_bwd_ready[kMaxDevices];
EncodeTiledFn g_bwd_encode = nullptr;
template <int D>
constexpr int dkdv_smem() { return 2 * tile_bytes<D>() + kStagesKV * (2 * tile_bytes<D>() + 1024) + 1024; }
template <int D>
constexpr int dq_smem() { return tile_bytes<D>() + kStages * (2 * tile_bytes<D>()) + 1024; }

attn_status_t bwd_device_ready(cudaStream_t stream, int** status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  // device check, tensor-map encoder and status word come from the forward's set-up
  const attn_status_t ds = gb300_host::device_status_word(stream, status);
  if (ds != ATTN_OK) return ds;
  std::lock_guard<std::mutex> lock(g_bwd_mutex);
  if (!g_bwd_ready[dev]) {
    // one-time set-up: not inside a stream capture
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
      cudaGetLastError();
      return ATTN_ERR_UNSUPPORTED;
    }
    if (!g_bwd_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return ATTN_ERR_CUDA;
      g_bwd_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (cudaFuncSetAttribute(dkdv_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dkdv_smem<128>()) != cudaSuccess ||
        cudaFuncSetAttribute(dq_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dq_smem<128>()) != cudaSuccess ||
        cudaFuncSetAttribute(dkdv_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dkdv_smem<64>()) != cudaSuccess ||
        cudaFuncSetAttribute(dq_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dq_smem<64>()) != cudaSuccess)
      return ATTN_ERR_CUDA;
    g_bwd_ready[dev] = true;
  }
  return ATTN_OK;
}

// dK/dV is launched as the row kernel's programmatic dependent: its CTAs set
// up while the row kernel finishes and wait for it before reading anything.
template <int D>
cudaError_t launch_dkdv(unsigned grid, cudaStream_t stream, const CUtensorMap& mq,
                        const CUtensorMap& mdo, const CUtensorMap& mk, const CUtensorMap& mv,
                        const BwdParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dkdv_smem<D>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dkdv_kernel<D>, mq, mdo, mk, mv, p);
}

// dQ is launched as the dK/dV kernel's programmatic dependent: it reads only
// the inputs and the row statistics (complete once dK/dV's CTAs are past their
// wait, which is when they let dQ launch), so it needs no grid-dependency wait
// and its persistent CTAs take the SMs that dK/dV's last CTAs free.
template <int D>
cudaError_t launch_dq(unsigned grid, cudaStream_t stream, const CUtensorMap& mk,
                      const CUtensorMap& mv, const CUtensorMap& mdo, const uint16_t* qh,
                      const BwdParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dq_smem<D>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dq_kernel<D>, mk, mv, mdo, qh, p);
}

bool encode_tile_map(CUtensorMap* map, const void* ptr, int D, int H, int64_t L, int64_t B) {
  const cuuint64_t d = static_cast<cuuint64_t>(D);
  const cuuint64_t dims[4] = {d, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {d * 2, static_cast<cuuint64_t>(H) * d * 2,
                                 static_cast<cuuint64_t>(L) * H * d * 2};
  const cuuint32_t box[4] = {64, 1, kT, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return g_bwd_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                      strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

int64_t attn_prefill_bwd_workspace_bytes(int64_t B, int64_t L, int32_t n_q, int32_t n_kv,
                                         int32_t d_h) {
  if (B < 1 || L < 1 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0 || (d_h != 64 && d_h != 128)) return -1;
  const int64_t T = (L + kT - 1) / kT;
  return 2 * B * n_q * T * kT * 4;
}

attn_status_t attn_prefill_bwd(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               void* workspace, int64_t workspace_bytes, int64_t B, int64_t L,
                               int32_t n_q, int32_t n_kv, int32_t d_h, int32_t causal,
                               float scale, void* stream_ptr) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || L < 1 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0) return ATTN_ERR_INVALID_ARG;
  if ((causal != 0 && causal != 1) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void* ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
  };
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
      misaligned(dout, 16) || misaligned(dq, 16) || misaligned(dk, 16) || misaligned(dv, 16) ||
      misaligned(lse, 4) || misaligned(workspace, 16))
    return ATTN_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return ATTN_ERR_UNSUPPORTED;
  const int64_t T = (L + kT - 1) / kT;
  // 32-bit tile indexing, and the row kernel's grid (128 rows x B*n_q*T / 32)
  if (L > (int64_t{1} << 30) || B * n_kv * T > INT32_MAX || B * n_q * T > INT32_MAX / 4)
    return ATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < attn_prefill_bwd_workspace_bytes(B, L, n_q, n_kv, d_h))
    return ATTN_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int* status = nullptr;
  const attn_status_t ds = bwd_device_ready(stream, &status);
  if (ds != ATTN_OK) return ds;

  CUtensorMap mq, mk, mv, mdo;
  if (!encode_tile_map(&mq, q, d_h, n_q, L, B) || !encode_tile_map(&mk, k, d_h, n_kv, L, B) ||
      !encode_tile_map(&mv, v, d_h, n_kv, L, B) || !encode_tile_map(&mdo, dout, d_h, n_q, L, B))
    return ATTN_ERR_CUDA;
  BwdParams p;
  p.L = static_cast<int>(L);
  p.n_q = n_q;
  p.n_kv = n_kv;
  p.g = n_q / n_kv;
  p.T = static_cast<int>(T);
  p.causal = causal;
  p.c = scale * kLog2e;
  p.scale = scale;
  float* nlse2 = static_cast<float*>(workspace);
  float* nrowdot = nlse2 + B * n_q * T * kT;
  p.nlse2 = nlse2;
  p.nrowdot = nrowdot;
  p.dq = static_cast<uint16_t*>(dq);
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  p.status = status;
  p.q_units = static_cast<int>(B * n_q * T);

  const int64_t rows = B * n_q * T * kT;
  constexpr int kRowdotRowsPerBlock = 8 * kRowdotRowsPerWarp;   // 256 threads
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    sms = 1;
  const int64_t need_blocks = (rows + kRowdotRowsPerBlock - 1) / kRowdotRowsPerBlock;
  const unsigned row_blocks = static_cast<unsigned>(need_blocks < 8 * sms ? need_blocks : 8 * sms);
  const uint16_t* oh = static_cast<const uint16_t*>(o);
  const uint16_t* qh = static_cast<const uint16_t*>(q);
  const uint16_t* doh = static_cast<const uint16_t*>(dout);
  const int Lp = static_cast<int>(T * kT);
  const unsigned kv_tiles = static_cast<unsigned>(B * n_kv * T);
  const unsigned dq_grid = static_cast<unsigned>(B * n_q * T < sms ? B * n_q * T : sms);
  if (d_h == 128) {
    rowdot_kernel<128><<<row_blocks, 256, 0, stream>>>(oh, doh, lse, nlse2, nrowdot,
                                                       static_cast<int>(B), p.L, n_q, Lp);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    if (launch_dkdv<128>(kv_tiles, stream, mq, mdo, mk, mv, p) != cudaSuccess) return ATTN_ERR_CUDA;
    if (launch_dq<128>(dq_grid, stream, mk, mv, mdo, qh, p) != cudaSuccess) return ATTN_ERR_CUDA;
  } else {
    rowdot_kernel<64><<<row_blocks, 256, 0, stream>>>(oh, doh, lse, nlse2, nrowdot,
                                                      static_cast<int>(B), p.L, n_q, Lp);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    if (launch_dkdv<64>(kv_tiles, stream, mq, mdo, mk, mv, p) != cudaSuccess) return ATTN_ERR_CUDA;
    if (launch_dq<64>(dq_grid, stream, mk, mv, mdo, qh, p) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
