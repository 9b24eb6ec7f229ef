// attn_decode.cu — decode attention (one new query token per sequence) for
// GB300 (sm_103a), split over the key range.
//
// Decode attends one query row per head to the whole K/V cache; its work per
// byte is the GQA group size g, so it is bound by HBM bandwidth, not by the
// tensor cores ("Long-Context Attention Explained" (sevydevy), prefill vs
// decode: each decode step reads the whole KV cache; "Memory-bound vs
// compute-bound" lesson (Pranay), "Attention itself": decode attention is a
// batched matrix-vector product whose time is cache size over bandwidth).
// So the kernel is built to stream K and V once at the copy rate, and it
// hands both products to the tensor cores only to keep the SM's issue slots
// free for that stream:
//
//   split kernel  persistent, one CTA per SM. The B * n_kv * T key tiles
//                 (T = ceil(Lk / 128) per K/V head) are cut into equal
//                 contiguous ranges, one per CTA; a range that crosses a head
//                 boundary becomes one segment per head. Per segment the CTA
//                 streams its K and V tiles through a 6-stage TMA ring and
//                 computes, with the keys on the TMEM lanes and the g <= 16
//                 query heads of the group as the N = 16 columns,
//                   S^T = K Q^T          (tcgen05, both operands in smem)
//                   O^T += V^T P^T       (tcgen05, V used MN-major)
//                 with an online softmax over the key lanes in between (one
//                 thread per key; the running maximum moves lazily, so the
//                 cross-thread maximum is only taken when a score exceeds it
//                 by the threshold). It writes the segment's normalised partial
//                 output and log-sum-exp to the workspace.
//   combine       one CTA per (b, query head) merges the head's segments
//                 through their log-sum-exps into bf16 O and fp32 LSE.
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

constexpr int kDim = 128;            // head dimension handled here
constexpr int kKeys = 128;           // keys per tile (= TMEM lanes of S^T)
constexpr int kHeadsPad = 16;        // N of both products: the group's heads, padded
constexpr int kMaxG = 16;            // query heads per K/V head
constexpr int kRing = 6;             // K/V ring slots (K and V tiles alternate)
constexpr int kTileBytes = kKeys * kDim * 2;          // 32 KiB: two 128 x 64 swizzled chunks
constexpr int kChunkBytes = kKeys * 128;              // 16 KiB
constexpr int kQBytes = kHeadsPad * kDim * 2;         // 4 KiB: two 16 x 64 chunks
constexpr int kPBytes = kHeadsPad * kKeys * 2;        // 4 KiB: P as 16 heads x 128 keys
constexpr int kSmallChunk = kHeadsPad * 128;          // 2 KiB: one 16-row swizzled chunk
constexpr int kSmemBytes = kRing * kTileBytes + 2 * kQBytes + 2 * kPBytes + 1024;
constexpr int kDecodeCtas = 152;     // one CTA per SM on a 152-SM GB300
constexpr int kThreads = 192;        // warps 0-3 softmax, 4 TMA producer, 5 MMA issuer
constexpr int kLoadWarp = 4, kMmaWarp = 5;
constexpr uint32_t kTmemCols = 64;
constexpr uint32_t kColS = 0;        // S^T buffers at columns 0 and 16
constexpr uint32_t kColO = 32;       // O^T accumulator
constexpr float kRescale = 8.0f;     // lazy running-max threshold (log2 units)
constexpr int kStatusTimeout = 1;

struct DecodeParams {
  float* part_o;         // fp32 [G * P_max * g, 128] normalised partial outputs
  float* part_lse;       // fp32 [G * P_max * g] partial log-sum-exp (natural log)
  int* status;           // per-device status word (timeouts)
  int Lk, n_q, n_kv, g;
  int T;                 // key tiles per K/V head
  long long W;           // B * n_kv * T
  int G, P_max;          // CTAs and segment slots per CTA
  float c;               // scale * log2(e)
  long long spin_limit;
};

struct DecodeCtl {
  uint64_t full[kRing], empty[kRing];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_done, o_free, drain;
  uint32_t tmem_base;
  int abort;
  float red_m[4][kHeadsPad];
  float red_l[4][kHeadsPad];
};

// First global tile of CTA c's range, and the CTA whose range holds tile x.
__host__ __device__ __forceinline__ long long range_start(long long c, long long W, long long G) {
  return c * W / G;
}
__host__ __device__ __forceinline__ long long cta_of(long long x, long long W, long long G) {
  return ((x + 1) * G - 1) / W;
}

// Segment slots per CTA: a range of at most ceil(W / G) tiles touches at most
// this many heads.
long long segment_slots(long long W, long long G, long long T) {
  return ((W + G - 1) / G - 1) / T + 2;
}

__device__ __forceinline__ bool spin_wait(uint32_t bar, uint32_t parity, DecodeCtl& ctl,
                                          const DecodeParams& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = clock64_now();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&ctl.abort)) return false;
    if (static_cast<long long>(clock64_now() - t0) > p.spin_limit) {
      *reinterpret_cast<volatile int*>(&ctl.abort) = 1;
      if (p.status) atomicOr(p.status, kStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, DecodeCtl& ctl,
                                          const DecodeParams& p) {
  return __all_sync(0xffffffffu, spin_wait(bar, parity, ctl, p));
}

// Wait used while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const DecodeParams& p) {
  const uint64_t t0 = clock64_now();
  while (!mbar_try_wait(bar, parity))
    if (static_cast<long long>(clock64_now() - t0) > p.spin_limit) return;
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
        "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
      :
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

// Generic-proxy shared-memory writes of this thread become visible to the
// tensor cores (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier 1 over the 128 softmax threads; the OR of `v` over them.
__device__ __forceinline__ void bar_softmax() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool bar_softmax_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* desc, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];"
      ::"r"(dst), "l"(desc), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// One segment of a CTA's tile range: K/V head `hd` (= b * n_kv + kv head),
// key tiles [t0, t0 + n), written to segment slot `slot` of the CTA.
struct Segment {
  int hd, t0, n, slot;
};

// Walks CTA c's range segment by segment (every role takes the same walk).
struct SegmentWalk {
  long long x, end;
  int T, slot;
  __device__ SegmentWalk(const DecodeParams& p, int c)
      : x(range_start(c, p.W, p.G)), end(range_start(c + 1, p.W, p.G)), T(p.T), slot(0) {}
  __device__ bool next(Segment& s) {
    if (x >= end) return false;
    const long long hd = x / T, base = hd * T;
    const long long t1 = (end - base < T) ? end - base : T;
    s.hd = static_cast<int>(hd);
    s.t0 = static_cast<int>(x - base);
    s.n = static_cast<int>(t1 - (x - base));
    s.slot = slot++;
    x = base + t1;
    return true;
  }
};

}  // namespace

namespace {

// GP: the group's query heads padded to 4, 8 or 16 (g <= GP); the loops over
// heads unroll to GP and skip h >= g.
template <int GP>
__global__ void __launch_bounds__(kThreads, 1)
attn_decode_split_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ DecodeCtl ctl;
  // smem: kRing K/V tiles | Q[2] (16 heads x 128, two 2 KiB chunks) | P[2]
  const uint32_t base = (smem_addr(dyn_smem) + 1023u) & ~1023u;   // swizzle atoms need 1 KiB
  const uint32_t sRing = base, sQ = base + kRing * kTileBytes, sP = sQ + 2 * kQBytes;
  uint8_t* const pgen = dyn_smem + (sP - smem_addr(dyn_smem));      // generic address of P[0]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = static_cast<int>(blockIdx.x);
  // The combine kernel (launched as this grid's programmatic dependent) may
  // start now; it waits for this grid to complete before reading anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(smem_addr(&ctl.full[s]), 1);
      mbar_init(smem_addr(&ctl.empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&ctl.q_full[s]), 1);
      mbar_init(smem_addr(&ctl.q_empty[s]), 1);
      mbar_init(smem_addr(&ctl.s_full[s]), 1);
      mbar_init(smem_addr(&ctl.p_full[s]), 128);
      mbar_init(smem_addr(&ctl.pv_done[s]), 1);
    }
    mbar_init(smem_addr(&ctl.o_done), 1);
    mbar_init(smem_addr(&ctl.o_free), 128);
    mbar_init(smem_addr(&ctl.drain), 1);
    ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(&ctl.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4) {
    // P rows g..15 are never written again: they stay zero, so the padded
    // columns of O^T stay zero.
    uint4* pz = reinterpret_cast<uint4*>(pgen);
    for (int i = threadIdx.x; i < 2 * kPBytes / 16; i += 128) pz[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;
  // Launched as the programmatic dependent of the stream's previous kernel
  // (the previous call's combine, or whatever wrote Q, K and V): the set-up
  // above overlaps it; global memory is touched only after it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == kLoadWarp) {
    if (lane == 0) {
      SegmentWalk walk(p, cta);
      Segment sg;
      uint32_t it = 0;   // ring items issued (K_t and V_t alternate)
      uint32_t qn = 0;   // Q tiles issued (one per segment)
      bool ok = true;
      while (ok && walk.next(sg)) {
        const int b = sg.hd / p.n_kv, kvh = sg.hd - b * p.n_kv;
        const uint32_t qb = qn & 1;
        if (qn >= 2 && !spin_wait(smem_addr(&ctl.q_empty[qb]), ((qn >> 1) - 1) & 1, ctl, p)) {
          ok = false;
          break;
        }
        const uint32_t qbar = smem_addr(&ctl.q_full[qb]);
        mbar_arrive_expect_tx(qbar, kQBytes);
        // rows kvh*g .. kvh*g + 15: the group's heads first (rows past n_q read as zero)
        for (int ch = 0; ch < 2; ++ch)
          tma_load_3d(sQ + qb * kQBytes + ch * kSmallChunk, &tmQ, qbar, ch * 64, kvh * p.g, b);
        ++qn;
        for (int t = 0; t < sg.n && ok; ++t) {
          for (int kind = 0; kind < 2; ++kind) {
            const uint32_t slot = it % kRing, use = it / kRing;
            if (use > 0 && !spin_wait(smem_addr(&ctl.empty[slot]), (use - 1) & 1, ctl, p)) {
              ok = false;
              break;
            }
            const uint32_t bar = smem_addr(&ctl.full[slot]);
            mbar_arrive_expect_tx(bar, kTileBytes);
            for (int ch = 0; ch < 2; ++ch)
              tma_load_4d(sRing + slot * kTileBytes + ch * kChunkBytes, kind ? &tmV : &tmK, bar,
                          ch * 64, kvh, (sg.t0 + t) * kKeys, b);
            ++it;
          }
        }
      }
      if (!ok) {
        // Let every copy this thread started land before the CTA can exit.
        for (uint32_t s = 0; s < 2 && s < qn; ++s) {
          const uint32_t last = s + ((qn - 1 - s) / 2) * 2;
          drain_wait(smem_addr(&ctl.q_full[s]), (last >> 1) & 1, p);
        }
        for (uint32_t s = 0; s < kRing && s < it; ++s) {
          const uint32_t last = s + ((it - 1 - s) / kRing) * kRing;
          drain_wait(smem_addr(&ctl.full[s]), (last / kRing) & 1, p);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // The whole warp runs the loop (warp-uniform control flow); one elected
    // lane issues every tcgen05 instruction and commit.
    const bool leader = elect_one();
    // S^T = K Q^T: M = 128 keys, N = 16 heads, both K-major (K = head dim).
    constexpr uint32_t kIdS = idesc_bf16_f32(kKeys, kHeadsPad, false);
    // O^T = V^T P^T: M = 128 dims with V read MN-major (bit 15), B = P K-major.
    constexpr uint32_t kIdO = idesc_bf16_f32(kDim, kHeadsPad, false) | (1u << 15);
    SegmentWalk walk(p, cta);
    Segment sg;
    uint32_t it = 0, gt = 0, sn = 0;
    bool ok = true;
    auto wait_item = [&](uint32_t item) {
      const bool r = wait_warp(smem_addr(&ctl.full[item % kRing]), (item / kRing) & 1, ctl, p);
      tc_fence_after_sync();
      return r;
    };
    auto issue_s = [&](uint32_t kitem, uint32_t qb, uint32_t sbuf) {
      const uint32_t k_smem = sRing + (kitem % kRing) * kTileBytes, q_smem = sQ + qb * kQBytes;
#pragma unroll
      for (int kk = 0; kk < kDim / 16; ++kk) {
        const uint64_t a = sdesc_sw128(k_smem + (kk >> 2) * kChunkBytes + (kk & 3) * 32, 16, 1024);
        const uint64_t bq = sdesc_sw128(q_smem + (kk >> 2) * kSmallChunk + (kk & 3) * 32, 16, 1024);
        if (leader) mma_ss(tmem + kColS + 16 * sbuf, a, bq, kIdS, kk > 0 ? 1u : 0u);
      }
      if (leader) mma_commit(smem_addr(&ctl.s_full[sbuf]));
      if (leader) mma_commit(smem_addr(&ctl.empty[kitem % kRing]));
    };
    while (ok && walk.next(sg)) {
      const uint32_t qb = sn & 1, it0 = it;
      if (!wait_warp(smem_addr(&ctl.q_full[qb]), (sn >> 1) & 1, ctl, p) || !wait_item(it0)) {
        ok = false;
        break;
      }
      issue_s(it0, qb, gt & 1);
      if (sg.n == 1 && leader) mma_commit(smem_addr(&ctl.q_empty[qb]));
      for (int t = 0; t < sg.n; ++t, ++gt) {
        // scores of the next tile run while the softmax works on this one
        if (t + 1 < sg.n) {
          if (!wait_item(it0 + 2 * (t + 1))) { ok = false; break; }
          issue_s(it0 + 2 * (t + 1), qb, (gt + 1) & 1);
          if (t + 2 == sg.n && leader) mma_commit(smem_addr(&ctl.q_empty[qb]));
        }
        // O^T of the previous segment must have been read out first
        if (t == 0 && sn > 0 && !wait_warp(smem_addr(&ctl.o_free), (sn - 1) & 1, ctl, p)) {
          ok = false;
          break;
        }
        if (!wait_warp(smem_addr(&ctl.p_full[gt & 1]), (gt >> 1) & 1, ctl, p) ||
            !wait_item(it0 + 2 * t + 1)) {
          ok = false;
          break;
        }
        const uint32_t vitem = it0 + 2 * t + 1;
        const uint32_t v_smem = sRing + (vitem % kRing) * kTileBytes;
        const uint32_t p_smem = sP + (gt & 1) * kPBytes;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          // V^T: a K step of 16 keys spans 16 rows (2 KiB); the two 64-dim
          // chunks are kChunkBytes apart. P: 32 bytes per K step.
          const uint64_t a = sdesc_sw128(v_smem + kk * 16 * 128, kChunkBytes, 1024);
          const uint64_t bp = sdesc_sw128(p_smem + (kk >> 2) * kSmallChunk + (kk & 3) * 32, 16, 1024);
          if (leader) mma_ss(tmem + kColO, a, bp, kIdO, (t > 0 || kk > 0) ? 1u : 0u);
        }
        if (leader) mma_commit(smem_addr(&ctl.pv_done[gt & 1]));
        if (leader) mma_commit(smem_addr(&ctl.empty[vitem % kRing]));
      }
      if (!ok) break;
      if (leader) mma_commit(smem_addr(&ctl.o_done));
      it = it0 + 2 * sg.n;
      ++sn;
    }
    // No MMA may still be running when TMEM is released.
    if (leader) mma_commit(smem_addr(&ctl.drain));
    drain_wait(smem_addr(&ctl.drain), 0, p);
    __syncwarp();
  } else if (warp < 4) {
    // softmax warps: thread r is key r of a tile (S^T lane) and dimension r
    // of the output (O^T lane)
    const int r = threadIdx.x;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    // where key r of a tile goes in a P buffer: 128-byte swizzled rows of 64
    // keys, chunk r / 64, 16-byte unit (r % 64) / 8 XOR (head % 8)
    const int p_chunk = (r >> 6) * kSmallChunk, p_unit = (r & 63) >> 3, p_byte = (r & 7) * 2;
    SegmentWalk walk(p, cta);
    Segment sg;
    uint32_t gt = 0, sn = 0;
    bool ok = true;
    // Every wait of these four warps ends in a vote over all 128 threads, so
    // they leave together when one of them gives up and none is left alone
    // at a named barrier.
    auto waited = [&](uint32_t bar, uint32_t parity) {
      const bool fail = bar_softmax_any(!spin_wait(bar, parity, ctl, p));
      tc_fence_after_sync();
      return !fail;
    };
    while (ok && walk.next(sg)) {
      float m_run[GP], l_thr[GP];
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        m_run[h] = -INFINITY;
        l_thr[h] = 0.0f;
      }
      for (int t = 0; t < sg.n; ++t, ++gt) {
        if (!waited(smem_addr(&ctl.s_full[gt & 1]), (gt >> 1) & 1)) {
          ok = false;
          break;
        }
        uint32_t sv[16];
        tmem_ld16(lane_base + kColS + 16 * (gt & 1), sv);
        tmem_wait_ld16(sv);
        const bool valid = (sg.t0 + t) * kKeys + r < p.Lk;
        float x[GP];
        bool need = false;
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          x[h] = valid ? __uint_as_float(sv[h]) * p.c : -INFINITY;
          if (h < p.g) need |= x[h] > m_run[h] + kRescale;
        }
        if (bar_softmax_any(need)) {
          // exact maximum of this tile per head, then move the running maxima
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            if (h >= p.g) break;
            float v = x[h];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
            if (lane == 0) ctl.red_m[warp][h] = v;
          }
          bar_softmax();
          float alpha[GP];
          bool scaled = false;
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            alpha[h] = 1.0f;
            if (h >= p.g) continue;
            const float tm = fmaxf(fmaxf(ctl.red_m[0][h], ctl.red_m[1][h]),
                                   fmaxf(ctl.red_m[2][h], ctl.red_m[3][h]));
            const float mn = fmaxf(m_run[h], tm);
            if (mn != m_run[h]) {
              alpha[h] = (m_run[h] == -INFINITY) ? 0.0f : ex2_approx(m_run[h] - mn);
              m_run[h] = mn;
              scaled = true;
            }
            l_thr[h] *= alpha[h];
          }
          if (t > 0 && scaled) {
            // rescale O^T once the previous tile's product has landed
            const uint32_t pg = gt - 1;
            if (!waited(smem_addr(&ctl.pv_done[pg & 1]), (pg >> 1) & 1)) {
              ok = false;
              break;
            }
            uint32_t ov[16];
            tmem_ld16(lane_base + kColO, ov);
            tmem_wait_ld16(ov);
#pragma unroll
            for (int h = 0; h < GP; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
            tmem_st16(lane_base + kColO, ov);
            tmem_wait_st();
          }
        }
        // P into buffer gt & 1, free once the product of tile gt - 2 is done
        if (gt >= 2 && !waited(smem_addr(&ctl.pv_done[gt & 1]), ((gt >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        uint8_t* pb = pgen + (gt & 1) * kPBytes + p_chunk + p_byte;
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          if (h >= p.g) break;
          const float e = valid ? ex2_approx(x[h] - m_run[h]) : 0.0f;
          l_thr[h] += e;
          *reinterpret_cast<uint16_t*>(pb + h * 128 + ((p_unit ^ (h & 7)) << 4)) =
              static_cast<uint16_t>(pack_bf16x2(e, 0.0f) & 0xFFFFu);
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        mbar_arrive(smem_addr(&ctl.p_full[gt & 1]));
      }
      if (!ok) break;
      // epilogue: O^T / l and the log-sum-exp of this segment
      if (!waited(smem_addr(&ctl.o_done), sn & 1)) break;
      uint32_t ov[16];
      tmem_ld16(lane_base + kColO, ov);
      tmem_wait_ld16(ov);
      tc_fence_before_sync();
      mbar_arrive(smem_addr(&ctl.o_free));
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        if (h >= p.g) break;
        float v = l_thr[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) ctl.red_l[warp][h] = v;
      }
      bar_softmax();
      const size_t row0 = (static_cast<size_t>(cta) * p.P_max + sg.slot) * p.g;
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        if (h >= p.g) break;
        const float l = ctl.red_l[0][h] + ctl.red_l[1][h] + ctl.red_l[2][h] + ctl.red_l[3][h];
        p.part_o[(row0 + h) * kDim + r] = __uint_as_float(ov[h]) / l;
        if (r == h) p.part_lse[row0 + h] = (m_run[h] + log2f(l)) * 0.69314718055994530942f;
      }
      ++sn;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One CTA of kCombineWarps warps per (b, query head): O = sum_s w_s O_s,
// w_s = exp(lse_s - LSE) over the head's segments (the CTAs whose tile ranges
// cover its K/V head). One pass: the warps take interleaved segments and merge
// them against a running maximum, each lane four dimensions; the warps' states
// are merged in shared memory.
constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(32 * kCombineWarps)
attn_decode_combine_kernel(uint16_t* o, float* lse, const DecodeParams p) {
  __shared__ float red_m[kCombineWarps], red_w[kCombineWarps];
  __shared__ float4 red_o[kCombineWarps][32];
  const int row = blockIdx.x;                       // b * n_q + query head
  const int b = row / p.n_q, h = row - b * p.n_q;
  const int r = h % p.g;
  const long long hd = static_cast<long long>(b) * p.n_kv + h / p.g;
  const long long c0 = cta_of(hd * p.T, p.W, p.G);
  const int ns = static_cast<int>(cta_of(hd * p.T + p.T - 1, p.W, p.G) - c0 + 1);
  // The head is segment slot `slot0` of CTA c0; every later CTA's range starts
  // inside the head (each range holds at least one tile), so it is their slot 0.
  const long long slot0 = hd - range_start(c0, p.W, p.G) / p.T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The next kernel in the stream (the next call's split kernel) may launch
  // and set up now; it waits for this grid to complete before touching
  // global memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Launched early behind the split kernel: wait until it has completed and
  // its partial results are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float m = -INFINITY, wsum = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 4
  for (int s = warp; s < ns; s += kCombineWarps) {
    const size_t sr = static_cast<size_t>(((c0 + s) * p.P_max + (s == 0 ? slot0 : 0)) * p.g + r);
    const float ls = p.part_lse[sr];
    const float4 v = *reinterpret_cast<const float4*>(p.part_o + sr * kDim + 4 * lane);
    const float mn = fmaxf(m, ls);
    const float a = (m == -INFINITY) ? 0.0f : __expf(m - mn);
    const float w = __expf(ls - mn);
    m = mn;
    wsum = fmaf(wsum, a, w);
    acc.x = fmaf(w, v.x, acc.x * a);
    acc.y = fmaf(w, v.y, acc.y * a);
    acc.z = fmaf(w, v.z, acc.z * a);
    acc.w = fmaf(w, v.w, acc.w * a);
  }
  red_o[warp][lane] = acc;
  if (lane == 0) {
    red_m[warp] = m;
    red_w[warp] = wsum;
  }
  __syncthreads();
  if (warp == 0) {
    float mx = red_m[0];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) mx = fmaxf(mx, red_m[w]);
    float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float ws = 0.0f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      const float a = (red_m[w] == -INFINITY) ? 0.0f : __expf(red_m[w] - mx);
      const float4 u = red_o[w][lane];
      t.x = fmaf(a, u.x, t.x);
      t.y = fmaf(a, u.y, t.y);
      t.z = fmaf(a, u.z, t.z);
      t.w = fmaf(a, u.w, t.w);
      ws = fmaf(a, red_w[w], ws);
    }
    const float inv = 1.0f / ws;
    const uint32_t w0 = pack_bf16x2(t.x * inv, t.y * inv);
    const uint32_t w1 = pack_bf16x2(t.z * inv, t.w * inv);
    *reinterpret_cast<uint2*>(o + static_cast<size_t>(row) * kDim + 4 * lane) = make_uint2(w0, w1);
    if (lane == 0) lse[row] = mx + logf(ws);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;
std::mutex g_decode_mutex;
bool g_decode_ready[kMaxDevices] = {};
EncodeTiledFn g_decode_encode = nullptr;

template <int GP>
bool set_smem() {
  return cudaFuncSetAttribute(attn_decode_split_kernel<GP>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes) == cudaSuccess;
}

attn_status_t decode_device_ready(cudaStream_t stream, int** status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  // device check (sm_103) and the status word come from the forward's set-up
  const attn_status_t ds = gb300_host::device_status_word(stream, status);
  if (ds != ATTN_OK) return ds;
  std::lock_guard<std::mutex> lock(g_decode_mutex);
  if (g_decode_ready[dev]) return ATTN_OK;
  // one-time set-up: not inside a stream capture
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return ATTN_ERR_UNSUPPORTED;
  }
  if (!g_decode_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return ATTN_ERR_CUDA;
    g_decode_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  if (!set_smem<4>() || !set_smem<8>() || !set_smem<16>()) return ATTN_ERR_CUDA;
  g_decode_ready[dev] = true;
  return ATTN_OK;
}

// K or V [B, Lk, H, 128] bf16 as (D, H, L, B): 64 x 1 x 128 x 1 boxes,
// 128-byte swizzle (the tensor cores' operand layout).
bool encode_kv(CUtensorMap* map, const void* ptr, int H, int64_t Lk, int64_t B) {
  const cuuint64_t dims[4] = {kDim, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(Lk),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {kDim * 2, static_cast<cuuint64_t>(H) * kDim * 2,
                                 static_cast<cuuint64_t>(Lk) * H * kDim * 2};
  const cuuint32_t box[4] = {64, 1, kKeys, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return g_decode_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                         strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q [B, 1, n_q, 128] bf16 as (D, n_q, B): 64 x 16 x 1 boxes (16 heads from
// the group's first), 128-byte swizzle.
bool encode_q(CUtensorMap* map, const void* ptr, int n_q, int64_t B) {
  const cuuint64_t dims[3] = {kDim, static_cast<cuuint64_t>(n_q), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {kDim * 2, static_cast<cuuint64_t>(n_q) * kDim * 2};
  const cuuint32_t box[3] = {64, kHeadsPad, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  return g_decode_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                         strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool decode_sizes_ok(int64_t B, int64_t Lk, int32_t n_q, int32_t n_kv, int32_t d_h) {
  return B >= 1 && Lk >= 1 && n_q >= 1 && n_kv >= 1 && n_q % n_kv == 0 && d_h >= 1;
}

// The partition of the B * n_kv * T key tiles over the split kernel's CTAs.
struct DecodeShape {
  int64_t T, W, G, P_max;
};
DecodeShape decode_shape(int64_t B, int64_t Lk, int32_t n_kv) {
  DecodeShape s;
  s.T = (Lk + kKeys - 1) / kKeys;
  s.W = B * n_kv * s.T;
  s.G = s.W < kDecodeCtas ? s.W : kDecodeCtas;
  s.P_max = segment_slots(s.W, s.G, s.T);
  return s;
}

}  // namespace

extern "C" {

int64_t attn_decode_workspace_bytes(int64_t B, int64_t Lk, int32_t n_q, int32_t n_kv,
                                    int32_t d_h) {
  if (!decode_sizes_ok(B, Lk, n_q, n_kv, d_h) || d_h != kDim || n_q / n_kv > kMaxG) return -1;
  if (Lk > (int64_t{1} << 30) || B * n_kv > (int64_t{1} << 24)) return -1;
  const DecodeShape s = decode_shape(B, Lk, n_kv);
  const int64_t rows = s.G * s.P_max * (n_q / n_kv);
  return rows * kDim * 4 + rows * 4;
}

attn_status_t attn_decode_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                              void* workspace, int64_t workspace_bytes, int64_t B, int64_t Lk,
                              int32_t n_q, int32_t n_kv, int32_t d_h, float scale,
                              void* stream_ptr) {
  if (!q || !k || !v || !o || !lse || !workspace) return ATTN_ERR_INVALID_ARG;
  if (!decode_sizes_ok(B, Lk, n_q, n_kv, d_h) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void* ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
  };
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
      misaligned(lse, 4) || misaligned(workspace, 16))
    return ATTN_ERR_INVALID_ARG;
  if (d_h != kDim || n_q / n_kv > kMaxG) return ATTN_ERR_UNSUPPORTED;
  if (Lk > (int64_t{1} << 30) || B * n_kv > (int64_t{1} << 24)) return ATTN_ERR_UNSUPPORTED;
  const DecodeShape s = decode_shape(B, Lk, n_kv);
  if (s.W > (int64_t{1} << 31) - 1 || B * n_q > (int64_t{1} << 31) - 1) return ATTN_ERR_UNSUPPORTED;
  const int64_t need = attn_decode_workspace_bytes(B, Lk, n_q, n_kv, d_h);
  if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int* status = nullptr;
  const attn_status_t ds = decode_device_ready(stream, &status);
  if (ds != ATTN_OK) return ds;

  CUtensorMap mq, mk, mv;
  if (!encode_q(&mq, q, n_q, B) || !encode_kv(&mk, k, n_kv, Lk, B) ||
      !encode_kv(&mv, v, n_kv, Lk, B))
    return ATTN_ERR_CUDA;
  DecodeParams p;
  const int64_t rows = s.G * s.P_max * (n_q / n_kv);
  p.part_o = static_cast<float*>(workspace);
  p.part_lse = p.part_o + rows * kDim;
  p.status = status;
  p.Lk = static_cast<int>(Lk);
  p.n_q = n_q;
  p.n_kv = n_kv;
  p.g = n_q / n_kv;
  p.T = static_cast<int>(s.T);
  p.W = s.W;
  p.G = static_cast<int>(s.G);
  p.P_max = static_cast<int>(s.P_max);
  p.c = scale * 1.4426950408889634f;
  p.spin_limit = 1ll << 31;   // about a second at 2 GHz
  // Both kernels are launched as programmatic dependents of the kernel before
  // them in the stream: the split kernel's set-up overlaps the previous
  // kernel's end, and the combine's CTAs are scheduled while the split kernel
  // still runs. Each waits (griddepcontrol.wait) before touching memory.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.G));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (p.g <= 4)
    e = cudaLaunchKernelEx(&cfg, attn_decode_split_kernel<4>, mq, mk, mv, p);
  else if (p.g <= 8)
    e = cudaLaunchKernelEx(&cfg, attn_decode_split_kernel<8>, mq, mk, mv, p);
  else
    e = cudaLaunchKernelEx(&cfg, attn_decode_split_kernel<16>, mq, mk, mv, p);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  cfg.gridDim = dim3(static_cast<unsigned>(B * n_q));
  cfg.blockDim = dim3(32 * kCombineWarps);
  cfg.dynamicSmemBytes = 0;
  uint16_t* o16 = static_cast<uint16_t*>(o);
  if (cudaLaunchKernelEx(&cfg, attn_decode_combine_kernel, o16, lse, p) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
