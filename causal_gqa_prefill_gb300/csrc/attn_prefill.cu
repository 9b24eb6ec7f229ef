// attn_prefill.cu — causal GQA prefill attention forward for GB300 (sm_103a).
//
// One persistent, warp-specialised kernel computes O = softmax(scale*Q K^T +
// causal mask) V tile by tile with an online softmax, so the L x L scores live
// only in tensor memory ("Long-Context Attention Explained" (sevydevy),
// sections "Tiling" and "Online softmax"; "Why Attention Scaling Breaks"
// (shivam2003), section "Flash Attention: the tiling insight").
//
// Work unit: two 128-row query tiles that read the same K/V head (two heads of
// one GQA group at the same query tile, or, when a group has one head, two
// neighbouring tiles of that head). Each K/V tile is fetched once by TMA and
// used by both query tiles ("prefill-attention" flop record (phantomic12),
// "Arithmetic intensity": GQA raises reuse of every K/V byte by g). Causal
// units visit only key tiles 0..i (skipping fully masked tiles, "Long-Context
// Attention Explained", FlashAttention-2 paragraph on causal block skipping),
// and units are handed out longest first over a persistent grid.
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3   softmax for query tile 0    (thread = tile row = TMEM lane)
//   warps 4-7   softmax for query tile 1
//   warp  8     TMA producer (Q tiles, K/V ring)
//   warp  9     tcgen05 MMA issuer (the whole warp runs the loop warp-uniformly,
//               one elected lane issues); owns the TMEM allocation
//   warps 10-11 idle
// The softmax warpgroups raise their register limit to 224 and the third
// warpgroup lowers its to 56 (setmaxnreg), so each softmax thread holds its
// whole 128-score row in registers without spilling.
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,128)   S0 scores, later P0 (bf16, packed two per column, cols 0..63)
//   [128,256) S1 / P1
//   [256,384) O0 accumulator (D columns)
//   [384,512) O1 accumulator
// Shared memory (d_h = 128, bf16): Q0 and Q1 (32 KiB each), a 4-stage K/V
// ring (32 KiB per tile) and 4 KiB per softmax warp through which the
// epilogue turns each thread's O row into row-contiguous global stores.
//
// MMA issue order per key tile j (ping-pong between the two query tiles, so
// one tile's softmax overlaps the other tile's matrix products):
//   S0_j = Q0 K_j^T ; O1 += P1_{j-1} V_{j-1} ; S1_j = Q1 K_j^T ; O0 += P0_j V_j
// tcgen05 operations from one thread execute in issue order, so a commit that
// signals S_t,j ready also implies O_t holds every tile before j.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn_prefill.h"
#include "sm103_ptx.cuh"

namespace {

using namespace gb300;

constexpr int kBM = 128;          // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;          // keys per K/V tile
constexpr int kThreads = 384;
constexpr int kSoftmaxRegs = 224;   // per thread, warpgroups 0 and 1
constexpr int kOtherRegs = 56;      // per thread, warpgroup 2
// The split must fit the registers the CTA is launched with (168 per thread
// at 384 threads and one CTA per SM); the host checks the compiled count.
constexpr int kRegBudget = 2 * 128 * kSoftmaxRegs + 128 * kOtherRegs;
static_assert(kRegBudget <= kThreads * 168, "setmaxnreg split exceeds the launch allocation");
constexpr int kLoadWarp = 8;
constexpr int kOStageWarpBytes = 32 * 128;           // 32 rows x 128 bytes per softmax warp
constexpr int kOStageBytes = 8 * kOStageWarpBytes;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
static_assert(kColS0 + kBN <= kColS1 && kColS1 + kBN <= kColO0 && kColO0 + 128 <= kColO1 &&
                  kColO1 + 128 <= kTmemCols,
              "TMEM column regions overlap or exceed the allocation");
// A row's running maximum is only moved (and O rescaled) once the tile maximum
// exceeds it by this many log2 units; exponentials stay <= 2^8 meanwhile, and
// the final O / l and LSE use the same stale maximum, so the result is exact.
constexpr float kRescaleThreshold = 8.0f;
constexpr int kStatusTimeout = 1;
constexpr int kStatusCheck = 2;     // a consistency check of the ATTN_DEBUG build failed
constexpr long long kSpinLimitCycles = 1ll << 31;   // about a second at 2 GHz
// Smallest batch of (b, kv-head) groups in the unit order, in rounds of the
// persistent grid (decode_unit).
constexpr int kBatchRounds = 8;

// D = head dim; F8: Q, K, V (and P) in fp8 e4m3 instead of bf16.
template <int D, bool F8>
struct Tile {
  static constexpr int kElemBytes = F8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElemBytes;
  static constexpr int kChunks = kRowBytes / 128;       // 128-byte swizzle column chunks
  static constexpr int kChunkElems = 128 / kElemBytes;  // elements per chunk row
  static constexpr int kQBytes = kBM * kRowBytes;
  static constexpr int kKVBytes = kBN * kRowBytes;
  static constexpr int kStages = (kKVBytes == 32768) ? 4 : 8;   // K/V ring depth (K and V share it)
  // two Q tiles, the K/V ring, and 4 KiB per softmax warp to stage O rows
  // for coalesced stores
  static constexpr int kSmemBytes = 2 * kQBytes + kStages * kKVBytes + kOStageBytes + 1024;
  // MMA K step: 16 bf16 or 32 e4m3 elements, 32 bytes either way.
  static constexpr int kKStep = 32 / kElemBytes;
  static_assert(kRowBytes % 128 == 0, "rows must fill whole 128-byte swizzle chunks");
};

struct Params {
  uint16_t* o;          // bf16 [B, L, n_q, D]
  float* lse;           // fp32 [B, n_q, L]
  int* status;          // per-device status word
  int Lq, Lk;           // query rows (chunk length) and keys
  int offset;           // absolute position of query row 0 = Lk - Lq
  int n_q, n_kv, g;
  int Tq, Tk;           // 128-row query tiles and 128-key tiles
  int causal;
  int scale_pos;        // 1 when c > 0
  float c;              // scale * log2(e) (times the Q and K descale factors for fp8)
  float o_scale;        // multiplies O / l in the epilogue (the V descale for fp8, else 1)
  int groups;           // B * n_kv
  int units;            // pairs per group * groups
  int pairs;            // pairs (units) per group
  int batch;            // groups per batch (see decode_unit)
  long long spin_limit;
};

#ifdef ATTN_DEBUG
// Debug build: how many phases each barrier's producer has started (TMA loads
// issued, commits issued, arrival rounds begun), and how many phases each
// waiter has consumed. A parity wait for phase k is only sound while no more
// than phase k + 1 has been started; every wait checks that. `checks` counts
// the checks run.
struct DbgShadow {
  unsigned int q_full, q_empty, kv_full[8], kv_empty[8], s_full[2], p_full[2], o_done[2];
  unsigned int checks;
};
#endif

struct Ctl {
  uint64_t q_full, q_empty;
  uint64_t kv_full[8], kv_empty[8];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
#ifdef ATTN_DEBUG
  DbgShadow dbg;
#endif
};

// Consistency checks of the ATTN_DEBUG build. The statement macros below
// expand to nothing in the release build, whose kernels are therefore the
// same code as without them. A failed check raises the abort flag and the
// check bit of the status word, and the caller leaves through the same path
// as after a wait timeout.
#ifdef ATTN_DEBUG
__device__ unsigned long long g_dbg_checks;   // checks run, summed at CTA exit

__device__ __forceinline__ bool dbg_ok(bool cond, Ctl& ctl, const Params& p) {
  atomicAdd(&ctl.dbg.checks, 1u);
  if (!cond) {
    *reinterpret_cast<volatile int*>(&ctl.abort) = 1;
    atomicOr(p.status, kStatusCheck);
  }
  return cond;
}
// the parity wait for phase k of `field`'s barrier is sound
#define DBG_PHASE_OK(field, k) \
  dbg_ok(*reinterpret_cast<volatile unsigned int*>(&ctl.dbg.field) <= (k) + 1u, ctl, p)
#define DBG_ISSUE(field) atomicAdd(&ctl.dbg.field, 1u)
#define DBG_BREAK_UNLESS(cond) \
  if (!(cond)) {               \
    ok = false;                \
    break;                     \
  }
#define DBG_RETURN_UNLESS(cond) \
  if (!(cond)) return;
#else
#define DBG_ISSUE(field)
#define DBG_BREAK_UNLESS(cond)
#define DBG_RETURN_UNLESS(cond)
#endif

struct Unit {
  int b, kvh, nkv;
  int head[2], qtile[2], n[2];
};

// Unit u -> (batch, K/V head, two query tiles). The (b, kv-head) groups are
// taken in batches of p.batch consecutive groups (the last batch may be
// smaller); within a batch units are ordered by pair index first, so
// ascending u means descending causal length (longest first) batch by batch,
// and only one batch's K/V is streamed at a time. The host batches only when
// the K/V of all groups exceeds 1.5 times the L2: a batch is as many groups as
// fit half of the L2, but at least kBatchRounds rounds of the persistent
// grid, so the snake order still balances it. Otherwise there is one batch
// and the order is pair-major over all groups.
// Query row i of the chunk sits at absolute position offset + i (the chunk is
// the end of the key range; offset = 0 for square prefill).
// Within one (b, kv-head) group the g*T query tiles are listed longest first
// and paired neighbour by neighbour: slot 1 holds the longer (or equal) tile,
// slot 0 the next one, and their key-tile counts differ by at most one.
__device__ __forceinline__ Unit decode_unit(int u, const Params& p) {
  Unit x;
  const int per_batch = p.batch * p.pairs;
  const int bi = u / per_batch;
  const int v = u - bi * per_batch;
  const int g0 = bi * p.batch;
  const int nb = min(p.batch, p.groups - g0);
  const int pair = v / nb;
  const int grp = g0 + (v - pair * nb);
  x.b = grp / p.n_kv;
  x.kvh = grp - x.b * p.n_kv;
  const int total = p.g * p.Tq;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int k = 2 * pair + (1 - s);
    if (k < total) {
      const int i = p.Tq - 1 - k / p.g;
      x.head[s] = x.kvh * p.g + (k % p.g);
      x.qtile[s] = i;
      // Causal: key tiles up to the one holding the tile's last query position.
      const int last_row = min(i * kBM + kBM - 1, p.Lq - 1);
      x.n[s] = p.causal ? min(p.Tk, (p.offset + last_row) / kBN + 1) : p.Tk;
    } else {
      x.head[s] = 0;
      x.qtile[s] = 0;
      x.n[s] = 0;
    }
  }
  x.nkv = x.n[1];
  return x;
}

// Persistent schedule: round r of the grid takes units r*grid .. r*grid+grid-1
// of the longest-first list, left to right on even rounds and right to left
// on odd rounds (snake order), which balances the triangular causal work
// without any shared counter.
__device__ __forceinline__ int snake_unit(int r) {
  const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return r * g + ((r & 1) ? (g - 1 - c) : c);
}

// Bounded wait: true when the phase completed; false if another role aborted
// or this wait ran past the limit (then it raises the abort flag and the
// device status word so the host sees ATTN_ERR_TIMEOUT).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, Ctl& ctl,
                                           const Params& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = clock64_now();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&ctl.abort)) return false;
    if (static_cast<long long>(clock64_now() - t0) > p.spin_limit) {
      *reinterpret_cast<volatile int*>(&ctl.abort) = 1;
      atomicOr(p.status, kStatusTimeout);
      return false;
    }
  }
}

// Wait used only while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const Params& p) {
  const uint64_t t0 = clock64_now();
  while (!mbar_try_wait(bar, parity)) {
    if (static_cast<long long>(clock64_now() - t0) > p.spin_limit) return;
  }
}

// Bounded wait taken by a whole warp; the result is the same on every lane.
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, Ctl& ctl, const Params& p) {
  return __all_sync(0xffffffffu, wait_phase(bar, parity, ctl, p));
}

// Diagnostic kernel for the wait limit: warp 0 waits on an mbarrier that
// nothing ever completes and must give up after p.spin_limit cycles, raising
// the abort flag and the device status word; warp 1 waits on a second such
// barrier and must leave through the abort flag (or its own limit). Both use
// the same wait routine as the attention roles.
__global__ void __launch_bounds__(64, 1) wait_selftest_kernel(const Params p) {
  __shared__ Ctl ctl;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&ctl.q_full), 1);
    mbar_init(smem_addr(&ctl.q_empty), 1);
    ctl.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t bar = smem_addr((threadIdx.x >> 5) == 0 ? &ctl.q_full : &ctl.q_empty);
  wait_all(bar, 0, ctl, p);
  __syncthreads();
}

// ------------------------------------------------------------------ producer

template <int D, bool F8>
__device__ void load_role(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                          const CUtensorMap* tmV, Ctl& ctl, const Params& p,
                          uint32_t sQ0, uint32_t sQ1, uint32_t sKV, uint32_t smem_end) {
  using TL = Tile<D, F8>;
  // Run by lane 0 alone: a whole warp polling the ring barriers would cost
  // the softmax warps on this SM sub-partition more issue slots than it saves.
  uint32_t it = 0;       // K/V ring items issued
  uint32_t q_issued = 0;
  bool ok = true;
  int uc = 0;
#ifdef ATTN_DEBUG
  // a copy's tile must start inside its tensor (x aligned to 16 bytes) and
  // land inside the CTA's shared memory
  const int nB = p.groups / p.n_kv;
  auto tma_ok = [&](uint32_t dst, int c0, int c1, int H, int c2, int rows, int c3) -> bool {
    return dbg_ok((c0 * TL::kElemBytes) % 16 == 0 && c0 >= 0 && c0 < D && c1 >= 0 && c1 < H &&
                      c2 >= 0 && c2 < rows && c3 >= 0 && c3 < nB && dst >= sQ0 &&
                      dst + kBM * 128 <= smem_end,
                  ctl, p);
  };
#endif
  for (int r = 0; r * static_cast<int>(gridDim.x) < p.units; ++r) {
    const int u = snake_unit(r);
    if (u >= p.units) continue;
    const Unit x = decode_unit(u, p);
    if (uc > 0 && !wait_phase(smem_addr(&ctl.q_empty), (uc - 1) & 1, ctl, p)) { ok = false; break; }
    DBG_BREAK_UNLESS(uc == 0 || DBG_PHASE_OK(q_empty, static_cast<uint32_t>(uc - 1)))
    ++uc;
    const uint32_t qbar = smem_addr(&ctl.q_full);
    mbar_arrive_expect_tx(qbar, (x.n[0] > 0 ? 2u : 1u) * TL::kQBytes);
    ++q_issued;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      if (x.n[s] == 0) continue;
      const uint32_t dst = s ? sQ1 : sQ0;
#pragma unroll
      for (int c = 0; c < TL::kChunks; ++c) {
        DBG_BREAK_UNLESS(tma_ok(dst + c * kBM * 128, c * TL::kChunkElems, x.head[s], p.n_q,
                                x.qtile[s] * kBM, p.Lq, x.b))
        tma_load_4d(dst + c * kBM * 128, tmQ, qbar, c * TL::kChunkElems, x.head[s], x.qtile[s] * kBM,
                    x.b);
      }
    }
#ifdef ATTN_DEBUG
    if (!ok) break;
#endif
    DBG_ISSUE(q_full);
    for (int j = 0; j < x.nkv && ok; ++j) {
#pragma unroll
      for (int kind = 0; kind < 2; ++kind) {
        const uint32_t slot = it % TL::kStages, use = it / TL::kStages;
        if (use > 0 && !wait_phase(smem_addr(&ctl.kv_empty[slot]), (use - 1) & 1, ctl, p)) {
          ok = false;
          break;
        }
        DBG_BREAK_UNLESS(use == 0 || DBG_PHASE_OK(kv_empty[slot], use - 1))
        const uint32_t bar = smem_addr(&ctl.kv_full[slot]);
        const uint32_t dst = sKV + slot * TL::kKVBytes;
#ifdef ATTN_DEBUG
        bool coords = true;
        for (int c = 0; c < TL::kChunks; ++c)
          coords = coords && tma_ok(dst + c * kBN * 128, c * TL::kChunkElems, x.kvh, p.n_kv,
                                    j * kBN, p.Lk, x.b);
        DBG_BREAK_UNLESS(coords)
#endif
        mbar_arrive_expect_tx(bar, TL::kKVBytes);
#pragma unroll
        for (int c = 0; c < TL::kChunks; ++c)
          tma_load_4d(dst + c * kBN * 128, kind ? tmV : tmK, bar, c * TL::kChunkElems, x.kvh, j * kBN,
                      x.b);
        DBG_ISSUE(kv_full[slot]);
        ++it;
      }
    }
    if (!ok) break;
  }
  if (!ok) {
    // Let every copy this thread started land before the CTA can exit.
    if (q_issued) drain_wait(smem_addr(&ctl.q_full), (q_issued - 1) & 1, p);
    for (uint32_t s = 0; s < TL::kStages && s < it; ++s) {
      const uint32_t last = s + ((it - 1 - s) / TL::kStages) * TL::kStages;
      drain_wait(smem_addr(&ctl.kv_full[s]), (last / TL::kStages) & 1, p);
    }
  }
}

// ---------------------------------------------------------------- MMA issuer

template <int D, bool F8>
__device__ __forceinline__ void issue_qk(bool leader, uint32_t d_tmem, uint32_t q_smem,
                                         uint32_t k_smem) {
  using TL = Tile<D, F8>;
  constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(kBM, kBN, false) : idesc_bf16_f32(kBM, kBN, false);
#pragma unroll
  for (int kk = 0; kk < TL::kRowBytes / 32; ++kk) {
    // K step kk: 32 bytes (16 bf16 or 32 e4m3) inside chunk kk/4 of the swizzled tile.
    const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
    const uint64_t a = sdesc_sw128(q_smem + off, 16, 1024);
    const uint64_t b = sdesc_sw128(k_smem + off, 16, 1024);
    if (leader) {
      if (F8) mma_ss_e4m3(d_tmem, a, b, idesc, kk > 0 ? 1u : 0u);
      else mma_ss(d_tmem, a, b, idesc, kk > 0 ? 1u : 0u);
    }
  }
}

template <int D, bool F8>
__device__ __forceinline__ void issue_pv(bool leader, uint32_t d_tmem, uint32_t p_tmem,
                                         uint32_t v_smem, bool accumulate) {
  using TL = Tile<D, F8>;
  constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(kBM, D, true) : idesc_bf16_f32(kBM, D, true);
#pragma unroll
  for (int kk = 0; kk < kBN / TL::kKStep; ++kk) {
    // V tile is [keys][D] with D contiguous (MN-major for this product): a K
    // step of 16 (bf16) or 32 (e4m3) keys spans that many 128-byte rows;
    // 128-byte column chunks are kBN*128 bytes apart. P takes 8 TMEM columns
    // per K step either way (2 bf16 or 4 e4m3 per column).
    const uint64_t b = sdesc_sw128(v_smem + kk * TL::kKStep * 128, kBN * 128, 1024);
    if (leader) {
      if (F8) mma_ts_e4m3(d_tmem, p_tmem + kk * 8, b, idesc, (accumulate || kk > 0) ? 1u : 0u);
      else mma_ts(d_tmem, p_tmem + kk * 8, b, idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
  }
}

template <int D, bool F8>
__device__ void mma_role(Ctl& ctl, const Params& p, uint32_t tmem, uint32_t sQ0, uint32_t sQ1,
                         uint32_t sKV, uint32_t smem_end) {
  using TL = Tile<D, F8>;
  // The whole warp runs this loop (so its control flow and descriptor math
  // stay warp-uniform); one elected lane issues every tcgen05 instruction,
  // which keeps all commits on the thread that issued the MMAs.
  const bool leader = elect_one();
  uint32_t it = 0;
  uint32_t ph_p0 = 0, ph_p1 = 0;
  int uc = 0;
#ifdef ATTN_DEBUG
  // the allocation starts at lane 0, column 0; operand tiles lie inside the
  // CTA's shared memory; phases consumed per P-ready barrier
  uint32_t n_p0 = 0, n_p1 = 0;
  auto smem_ok = [&](uint32_t a, uint32_t bytes) -> bool {
    return dbg_ok(a >= sQ0 && a + bytes <= smem_end, ctl, p);
  };
  const bool tmem_ok = dbg_ok(tmem == 0u, ctl, p);
#endif
  for (int r = 0; r * static_cast<int>(gridDim.x) < p.units; ++r) {
    const int u = snake_unit(r);
    if (u >= p.units) continue;
    const Unit x = decode_unit(u, p);
#ifdef ATTN_DEBUG
    if (!tmem_ok) break;
#endif
    if (!wait_all(smem_addr(&ctl.q_full), uc & 1, ctl, p)) break;
#ifdef ATTN_DEBUG
    if (!DBG_PHASE_OK(q_full, static_cast<uint32_t>(uc))) break;
#endif
    ++uc;
    tc_fence_after_sync();
    uint32_t v_prev = 0;
    bool ok = true;
    for (int j = 0; j < x.nkv; ++j) {
      const uint32_t ks = it % TL::kStages;
      if (!wait_all(smem_addr(&ctl.kv_full[ks]), (it / TL::kStages) & 1, ctl, p)) { ok = false; break; }
      DBG_BREAK_UNLESS(DBG_PHASE_OK(kv_full[ks], it / TL::kStages))
      ++it;
      tc_fence_after_sync();
      const uint32_t k_smem = sKV + ks * TL::kKVBytes;
      DBG_BREAK_UNLESS(smem_ok(k_smem, TL::kKVBytes) && smem_ok(sQ0, TL::kQBytes) &&
                       smem_ok(sQ1, TL::kQBytes))
      if (j < x.n[0]) {
        issue_qk<D, F8>(leader, tmem + kColS0, sQ0, k_smem);
        if (leader) mma_commit(smem_addr(&ctl.s_full[0]));
#ifdef ATTN_DEBUG
        if (leader) DBG_ISSUE(s_full[0]);
#endif
      }
      if (j > 0) {
        if (!wait_all(smem_addr(&ctl.p_full[1]), ph_p1, ctl, p)) { ok = false; break; }
        ph_p1 ^= 1;
#ifdef ATTN_DEBUG
        DBG_BREAK_UNLESS(DBG_PHASE_OK(p_full[1], n_p1))
        ++n_p1;
#endif
        tc_fence_after_sync();
        issue_pv<D, F8>(leader, tmem + kColO1, tmem + kColS1, sKV + v_prev * TL::kKVBytes, j - 1 > 0);
        if (leader) mma_commit(smem_addr(&ctl.kv_empty[v_prev]));
#ifdef ATTN_DEBUG
        if (leader) DBG_ISSUE(kv_empty[v_prev]);
#endif
      }
      issue_qk<D, F8>(leader, tmem + kColS1, sQ1, k_smem);
      if (leader) mma_commit(smem_addr(&ctl.s_full[1]));
      if (leader) mma_commit(smem_addr(&ctl.kv_empty[ks]));
      if (leader && j == x.nkv - 1) mma_commit(smem_addr(&ctl.q_empty));
#ifdef ATTN_DEBUG
      if (leader) {
        DBG_ISSUE(s_full[1]);
        DBG_ISSUE(kv_empty[ks]);
        if (j == x.nkv - 1) DBG_ISSUE(q_empty);
      }
#endif

      const uint32_t vs = it % TL::kStages;
      if (!wait_all(smem_addr(&ctl.kv_full[vs]), (it / TL::kStages) & 1, ctl, p)) { ok = false; break; }
      DBG_BREAK_UNLESS(DBG_PHASE_OK(kv_full[vs], it / TL::kStages) &&
                       smem_ok(sKV + vs * TL::kKVBytes, TL::kKVBytes))
      ++it;
      tc_fence_after_sync();
      if (j < x.n[0]) {
        if (!wait_all(smem_addr(&ctl.p_full[0]), ph_p0, ctl, p)) { ok = false; break; }
        ph_p0 ^= 1;
#ifdef ATTN_DEBUG
        DBG_BREAK_UNLESS(DBG_PHASE_OK(p_full[0], n_p0))
        ++n_p0;
#endif
        tc_fence_after_sync();
        issue_pv<D, F8>(leader, tmem + kColO0, tmem + kColS0, sKV + vs * TL::kKVBytes, j > 0);
        if (leader && j == x.n[0] - 1) mma_commit(smem_addr(&ctl.o_done[0]));
#ifdef ATTN_DEBUG
        if (leader && j == x.n[0] - 1) DBG_ISSUE(o_done[0]);
#endif
      }
      v_prev = vs;
    }
    if (!ok) break;
    if (!wait_all(smem_addr(&ctl.p_full[1]), ph_p1, ctl, p)) break;
    ph_p1 ^= 1;
#ifdef ATTN_DEBUG
    if (!DBG_PHASE_OK(p_full[1], n_p1)) break;
    ++n_p1;
#endif
    tc_fence_after_sync();
    issue_pv<D, F8>(leader, tmem + kColO1, tmem + kColS1, sKV + v_prev * TL::kKVBytes, x.nkv - 1 > 0);
    if (leader) mma_commit(smem_addr(&ctl.o_done[1]));
    if (leader) mma_commit(smem_addr(&ctl.kv_empty[v_prev]));
#ifdef ATTN_DEBUG
    if (leader) {
      DBG_ISSUE(o_done[1]);
      DBG_ISSUE(kv_empty[v_prev]);
    }
#endif
  }
  // No MMA may still be running when TMEM is released.
  if (leader) mma_commit(smem_addr(&ctl.drain));
  drain_wait(smem_addr(&ctl.drain), 0, p);
  __syncwarp();
}

// ------------------------------------------------------------------- softmax

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Row maximum of 128 scores with three-input max instructions.
__device__ __forceinline__ float row_max128(const float* v) {
  float m[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) m[t] = v[t];
#pragma unroll
  for (int i = 8; i < 128; i += 16)
#pragma unroll
    for (int t = 0; t < 8; ++t) m[t] = max3(m[t], v[i + t], v[i + 8 + t]);
  return max3(max3(m[0], m[1], m[2]), max3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

template <int D, bool F8, bool kPos>
__device__ void softmax_role(int slot, Ctl& ctl, const Params& p, uint32_t tmem,
                             uint32_t o_stage) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (warp & 3) * 32 + lane;                         // tile row = TMEM lane
  const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const uint32_t tS = lane_base + (slot ? kColS1 : kColS0);
  const uint32_t tO = lane_base + (slot ? kColO1 : kColO0);
  const uint32_t bar_s = smem_addr(&ctl.s_full[slot]);
  const uint32_t bar_p = smem_addr(&ctl.p_full[slot]);
  const uint32_t bar_o = smem_addr(&ctl.o_done[slot]);
  const float cc = kPos ? p.c : 1.0f;
  const uint64_t cc2 = f32x2_pack(cc, cc);
  uint32_t ph_s = 0, ph_o = 0;
#ifdef ATTN_DEBUG
  // the allocation starts at lane 0, column 0, so this warp's loads and
  // stores use its own lane quarter; phases consumed per barrier
  uint32_t n_s = 0, n_o = 0;
  DBG_RETURN_UNLESS(dbg_ok(tmem == 0u, ctl, p))
#endif

  for (int rr = 0; rr * static_cast<int>(gridDim.x) < p.units; ++rr) {
    const int u = snake_unit(rr);
    if (u >= p.units) continue;
    const Unit x = decode_unit(u, p);
    // this warpgroup's query tile (selected, not indexed: a runtime index
    // would put the unit in local memory)
    const int n = slot ? x.n[1] : x.n[0];
    if (n == 0) continue;
    const int qtile = slot ? x.qtile[1] : x.qtile[0];
    const int head = slot ? x.head[1] : x.head[0];
    const int row = qtile * kBM + r;                            // chunk row
    const int qrow0 = p.offset + qtile * kBM;                   // absolute position of row 0
    float m_run = -INFINITY, l_run = 0.0f;
    for (int j = 0; j < n; ++j) {
      if (!__all_sync(0xffffffffu, wait_phase(bar_s, ph_s, ctl, p))) return;
      ph_s ^= 1;
#ifdef ATTN_DEBUG
      DBG_RETURN_UNLESS(__all_sync(0xffffffffu, DBG_PHASE_OK(s_full[slot], n_s)))
      ++n_s;
#endif
      tc_fence_after_sync();
      float s[128];
      {
        uint32_t* sr = reinterpret_cast<uint32_t*>(s);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * c));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_after_wait(*reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        tmem_after_wait(*reinterpret_cast<uint32_t(*)[32]>(sr + 64));
        tmem_after_wait(*reinterpret_cast<uint32_t(*)[32]>(sr + 96));
      }
      if (!kPos) {
        // Non-positive scale (its own kernel instance): fold it in first so
        // that masking and the maximum below work on the scaled scores (then
        // cc = 1).
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] *= p.c;
      }
      // Keys after in-tile index `keep` are masked: past the row's absolute
      // position (causal; the diagonal tile, or the last two tiles when the
      // chunk offset is not a multiple of the tile), or past the last key.
      const bool masked = p.causal ? (j * kBN + kBN - 1 > qrow0) : (p.Lk - j * kBN < kBN);
      if (masked) {
        const int keep = p.causal ? qrow0 + r - j * kBN : p.Lk - 1 - j * kBN;
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i > keep) s[i] = -INFINITY;
      }
      const float m_tile = row_max128(s) * cc;
      const float m_new = fmaxf(m_run, m_tile);
      const bool need = m_new > m_run + kRescaleThreshold;
      float alpha = 1.0f;
      if (need) {
        alpha = ex2_approx(m_run - m_new);
        m_run = m_new;
      }
      // P = 2^(c*s - m) into the first columns of this tile's S region (every
      // score of the row is already in registers): bf16 pairs in [0, 64), or
      // e4m3 quadruples in [0, 32). Two scores per packed FMA / add.
      const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
      const uint64_t negm2 = f32x2_pack(-m_use, -m_use);
      uint64_t sum2 = f32x2_pack(0.0f, 0.0f);
      if (F8) {
        // e4m3 P, four scores per TMEM column (first key in the lowest byte),
        // columns [0, 32). The row sum keeps the unrounded fp32 values.
        uint64_t sum2b = sum2;
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint64_t xa = ffma2(f32x2_pack(s[4 * i], s[4 * i + 1]), cc2, negm2);
          const uint64_t xb = ffma2(f32x2_pack(s[4 * i + 2], s[4 * i + 3]), cc2, negm2);
          float x0, x1, x2, x3;
          f32x2_unpack(xa, x0, x1);
          f32x2_unpack(xb, x2, x3);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
          sum2 = fadd2(sum2, f32x2_pack(p0, p1));
          sum2b = fadd2(sum2b, f32x2_pack(p2, p3));
          pk[i] = pack_e4m3x4(p0, p1, p2, p3);
        }
        tmem_st32(tS, pk);
        sum2 = fadd2(sum2, sum2b);
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint64_t xa = ffma2(f32x2_pack(s[64 * h + 2 * i], s[64 * h + 2 * i + 1]), cc2, negm2);
            float x0, x1;
            f32x2_unpack(xa, x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            const uint64_t pp = f32x2_pack(p0, p1);
            sum2 = fadd2(sum2, pp);
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st32(tS + 32 * h, pk);
        }
      }
      float sa, sb;
      f32x2_unpack(sum2, sa, sb);
      l_run = l_run * alpha + (sa + sb);
      // O <- O * 2^(m_old - m_new) when some row's maximum moved (rare): done
      // after P, when the row's scores are no longer held in registers, and
      // before the P-ready arrival that lets O += P V run (O already holds
      // every earlier tile: S of this tile was issued after the last P V).
      if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t ov[32];
          tmem_ld32(tO + c, ov);
          tmem_wait_ld(ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st32(tO + c, ov);
        }
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(bar_p);
#ifdef ATTN_DEBUG
      if (r == 0) DBG_ISSUE(p_full[slot]);
#endif
    }
    // Epilogue: O = acc / l (bf16, round to nearest even) and LSE in natural log.
    if (!__all_sync(0xffffffffu, wait_phase(bar_o, ph_o, ctl, p))) return;
    ph_o ^= 1;
#ifdef ATTN_DEBUG
    DBG_RETURN_UNLESS(__all_sync(0xffffffffu, DBG_PHASE_OK(o_done[slot], n_o)))
    ++n_o;
#endif
    tc_fence_after_sync();
    const float inv_l = p.o_scale / l_run;
    const bool valid = row < p.Lq;
    // O rows leave through this warp's 4 KiB of shared memory, 64 columns (128
    // bytes of bf16) at a time: each thread writes its own row's 128 bytes
    // (16-byte unit u at u ^ (row % 8), so a warp's stores hit all banks), then
    // each store to global memory covers four whole rows' 128-byte pieces
    // (eight threads per row) instead of 32 scattered 16-byte pieces.
    const uint32_t stg = o_stage + warp * kOStageWarpBytes;
    const int row0 = qtile * kBM + (warp & 3) * 32;             // first row of this warp
    const size_t hstride = static_cast<size_t>(p.n_q) * D;     // elements between rows
    uint16_t* obase = p.o + (static_cast<size_t>(x.b) * p.Lq * p.n_q + head) *
                                static_cast<size_t>(D);
#pragma unroll 1
    for (int hh = 0; hh < D / 64; ++hh) {
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t ov[32];
        tmem_ld32(tO + 64 * hh + 32 * c2, ov);
        tmem_wait_ld(ov);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
#pragma unroll
        for (int u = 4 * c2; u < 4 * c2 + 4; ++u)
          st_shared_v4(stg + lane * 128 + ((u ^ (lane & 7)) << 4), w[4 * u - 16 * c2],
                       w[4 * u - 16 * c2 + 1], w[4 * u - 16 * c2 + 2], w[4 * u - 16 * c2 + 3]);
      }
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int rr = 4 * k + (lane >> 3), u = lane & 7;
        const uint4 v = ld_shared_v4(stg + rr * 128 + ((u ^ (rr & 7)) << 4));
        if (row0 + rr < p.Lq)
          *reinterpret_cast<uint4*>(obase + static_cast<size_t>(row0 + rr) * hstride + 64 * hh + 8 * u) = v;
      }
      __syncwarp();
    }
    if (valid) {
      const float m_fin = (m_run == -INFINITY) ? 0.0f : m_run;
      p.lse[(static_cast<size_t>(x.b) * p.n_q + head) * p.Lq + row] =
          (m_fin + log2f(l_run)) * 0.69314718055994530942f;
    }
  }
}

// -------------------------------------------------------------------- kernel

template <int D, bool F8, bool kPos>
__global__ void __launch_bounds__(kThreads, 1)
attn_prefill_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const Params p) {
  using TL = Tile<D, F8>;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Ctl ctl;
  const uint32_t base = (smem_addr(dyn_smem) + 1023u) & ~1023u;   // swizzle atoms need 1 KiB
  const uint32_t sQ0 = base, sQ1 = base + TL::kQBytes, sKV = base + 2 * TL::kQBytes;
  const uint32_t smem_end = smem_addr(dyn_smem) + TL::kSmemBytes;   // checked in debug builds
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&ctl.q_full), 1);
    mbar_init(smem_addr(&ctl.q_empty), 1);
    for (int s = 0; s < TL::kStages; ++s) {
      mbar_init(smem_addr(&ctl.kv_full[s]), 1);
      mbar_init(smem_addr(&ctl.kv_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&ctl.s_full[s]), 1);
      mbar_init(smem_addr(&ctl.p_full[s]), 128);
      mbar_init(smem_addr(&ctl.o_done[s]), 1);
    }
    mbar_init(smem_addr(&ctl.drain), 1);
    ctl.abort = 0;
#ifdef ATTN_DEBUG
    memset(&ctl.dbg, 0, sizeof(ctl.dbg));
#endif
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
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl.tmem_base;

  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    softmax_role<D, F8, kPos>(warp >> 2, ctl, p, tmem, sKV + TL::kStages * TL::kKVBytes);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (warp == kLoadWarp) {
      if (lane == 0) load_role<D, F8>(&tmQ, &tmK, &tmV, ctl, p, sQ0, sQ1, sKV, smem_end);
    } else if (warp == kMmaWarp) {
      mma_role<D, F8>(ctl, p, tmem, sQ0, sQ1, sKV, smem_end);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
#ifdef ATTN_DEBUG
  if (threadIdx.x == 0) atomicAdd(&g_dbg_checks, static_cast<unsigned long long>(ctl.dbg.checks));
#endif
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int l2 = 0;              // L2 cache bytes
  int* status = nullptr;
};

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

// The softmax warpgroups raise their register limit with setmaxnreg; that
// only succeeds if the CTA was launched with at least kRegBudget registers,
// so refuse to launch a build whose register count does not cover the split.
template <int D, bool F8, bool kPos>
bool configure_kernel() {
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, attn_prefill_fwd_kernel<D, F8, kPos>) != cudaSuccess ||
      fa.numRegs * kThreads < kRegBudget)
    return false;
  return cudaFuncSetAttribute(attn_prefill_fwd_kernel<D, F8, kPos>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Tile<D, F8>::kSmemBytes) == cudaSuccess;
}

// Register-split check and shared-memory limit for every kernel instance.
bool configure_kernels() {
  return configure_kernel<64, false, true>() && configure_kernel<128, false, true>() &&
         configure_kernel<128, true, true>() && configure_kernel<64, false, false>() &&
         configure_kernel<128, false, false>() && configure_kernel<128, true, false>();
}

attn_status_t device_state(cudaStream_t stream, DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    // The set-up allocates and clears the status word on `stream`; neither
    // may happen inside a stream capture, so a first call there is refused
    // (and leaves nothing half set up).
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
      cudaGetLastError();
      return ATTN_ERR_UNSUPPORTED;
    }
    int major = 0, minor = 0, sms = 0, l2 = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;   // built for sm_103a only
    if (!configure_kernels()) return ATTN_ERR_UNSUPPORTED;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return ATTN_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    int* status = nullptr;
    if (cudaMalloc(&status, 256) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemsetAsync(status, 0, 256, stream) != cudaSuccess) {
      cudaFree(status);
      return ATTN_ERR_CUDA;
    }
    st.sms = sms;
    st.l2 = l2;
    st.status = status;
    st.ready = true;
  }
  *out = &st;
  return ATTN_OK;
}

// [B, L, H, D] (bf16, or e4m3 bytes when f8) as a 4-D tensor (D, H, L, B);
// boxes of one 128-byte row chunk x 1 x 128 x 1 with 128-byte swizzle. Rows
// past L read as zeros.
bool encode_bhld(CUtensorMap* map, const void* ptr, int D, int H, int64_t L, int64_t B,
                 bool f8 = false) {
  const cuuint64_t eb = f8 ? 1 : 2;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * eb,
                                 static_cast<cuuint64_t>(H) * D * eb,
                                 static_cast<cuuint64_t>(L) * H * D * eb};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb), 1, kBM, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return g_encode(map, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void*>(ptr), dims, strides,
                  box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Sizes -> work units; returns false when they exceed 32-bit tile indexing.
bool count_units(int64_t B, int64_t Lq, int64_t Lk, int32_t n_q, int32_t n_kv, int* Tq_out,
                 int* units_out) {
  const int64_t Tq = (Lq + kBM - 1) / kBM;
  const int64_t g = n_q / n_kv;
  const int64_t pairs = (g * Tq + 1) / 2;
  const int64_t units = pairs * B * n_kv;
  if (Lq > (int64_t{1} << 30) || Lk > (int64_t{1} << 30) || B > (int64_t{1} << 30) ||
      g * Tq > INT32_MAX || units > INT32_MAX || B * n_kv > INT32_MAX)
    return false;
  *Tq_out = static_cast<int>(Tq);
  *units_out = static_cast<int>(units);
  return true;
}

attn_status_t validate(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, int64_t B, int64_t Lq, int64_t Lk, int32_t n_q,
                       int32_t n_kv, int32_t d_h, int32_t causal, float scale) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Lq < 1 || Lk < Lq || n_q < 1 || n_kv < 1 || n_q % n_kv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  auto misaligned = [](const void* ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
  };
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
      misaligned(lse, 4))
    return ATTN_ERR_INVALID_ARG;
  if (d_h != 64 && d_h != 128) return ATTN_ERR_UNSUPPORTED;
  int Tq = 0, units = 0;
  if (!count_units(B, Lq, Lk, n_q, n_kv, &Tq, &units)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// One launch of the kernel instance for (f8, d_h) and the sign of the scale:
// a positive scale multiplies inside the exponent's FMA, any other is applied
// to the scores first (separate instances, so neither pays for the other).
template <bool kPos>
void launch_instance(int grid, cudaStream_t stream, const CUtensorMap& mq, const CUtensorMap& mk,
                     const CUtensorMap& mv, const Params& p, bool f8, int d_h) {
  if (f8)
    attn_prefill_fwd_kernel<128, true, kPos>
        <<<grid, kThreads, Tile<128, true>::kSmemBytes, stream>>>(mq, mk, mv, p);
  else if (d_h == 128)
    attn_prefill_fwd_kernel<128, false, kPos>
        <<<grid, kThreads, Tile<128, false>::kSmemBytes, stream>>>(mq, mk, mv, p);
  else
    attn_prefill_fwd_kernel<64, false, kPos>
        <<<grid, kThreads, Tile<64, false>::kSmemBytes, stream>>>(mq, mk, mv, p);
}

// Encodes the tensor maps, fills the parameters and launches (arguments
// already validated). `status` is the device status word the kernel reports
// wait timeouts into; `sms` the device's multiprocessor count.
// f8: Q, K, V are e4m3 with the given descale factors (real value = stored
// value * descale); otherwise bf16 and the descales are 1.
attn_status_t launch_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                             int64_t B, int64_t Lq, int64_t Lk, int32_t n_q, int32_t n_kv,
                             int32_t d_h, int32_t causal, float scale, cudaStream_t stream,
                             int* status, int sms, int l2, bool f8 = false,
                             float qk_descale = 1.0f,
                             float v_descale = 1.0f) {
  int Tq = 0, units = 0;
  count_units(B, Lq, Lk, n_q, n_kv, &Tq, &units);
  CUtensorMap mq, mk, mv;
  if (!encode_bhld(&mq, q, d_h, n_q, Lq, B, f8) || !encode_bhld(&mk, k, d_h, n_kv, Lk, B, f8) ||
      !encode_bhld(&mv, v, d_h, n_kv, Lk, B, f8))
    return ATTN_ERR_CUDA;

  Params p;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  p.status = status;
  p.Lq = static_cast<int>(Lq);
  p.Lk = static_cast<int>(Lk);
  p.offset = static_cast<int>(Lk - Lq);
  p.n_q = n_q;
  p.n_kv = n_kv;
  p.g = n_q / n_kv;
  p.Tq = Tq;
  p.Tk = static_cast<int>((Lk + kBN - 1) / kBN);
  p.causal = causal;
  p.c = scale * qk_descale * 1.4426950408889634f;
  p.o_scale = v_descale;
  p.scale_pos = p.c > 0.0f ? 1 : 0;
  p.groups = static_cast<int>(B * n_kv);
  p.units = units;
  p.pairs = units / p.groups;
  p.batch = p.groups;
  {
    // Batches of groups only when the K/V of all groups is well beyond the
    // L2 (more than 1.5 times its size): then as many groups as fit half of
    // it, but at least kBatchRounds rounds of the grid's units per batch.
    const int64_t kv_group = 2 * Lk * static_cast<int64_t>(d_h) * (f8 ? 1 : 2);
    if (2 * kv_group * p.groups > 3 * static_cast<int64_t>(l2)) {
      const int64_t grid_ctas = units < sms ? units : sms;
      const int64_t by_rounds = (kBatchRounds * grid_ctas + p.pairs - 1) / p.pairs;
      const int64_t by_l2 = (l2 / 2) / kv_group;
      int64_t want = by_rounds > by_l2 ? by_rounds : by_l2;
      if (want < 1) want = 1;
      p.batch = static_cast<int>(want < p.groups ? want : p.groups);
    }
  }
  p.spin_limit = kSpinLimitCycles;

  const int grid = units < sms ? units : sms;
  if (p.scale_pos)
    launch_instance<true>(grid, stream, mq, mk, mv, p, f8, d_h);
  else
    launch_instance<false>(grid, stream, mq, mk, mv, p, f8, d_h);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

// ----------------------------------------------------- allocation-free variant
//
// For callers that cannot allocate device memory: code running inside a
// memory pool or arena that must own every allocation (a cudaMalloc behind
// its back escapes its accounting and limits), or a host framework that
// forbids the library from touching the allocator. The only global memory the
// kernel needs beyond its inputs and outputs is its status word; here that
// word lives in the fixed array below, part of the library's own device image
// (zero when the library is loaded; the kernel only sets bits in it, and
// attn_device_check reads and clears it).

constexpr size_t kNoAllocScratchBytes = 256;            // stated maximum scratch
constexpr size_t kNoAllocScratchNeeded = sizeof(int);   // one status word, any problem size
static_assert(kNoAllocScratchNeeded <= kNoAllocScratchBytes,
              "the allocation-free variant's scratch exceeds its fixed array");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

struct NoAllocState {
  bool ready = false;
  int sms = 0;
  int l2 = 0;
  int* scratch = nullptr;    // device address of g_noalloc_scratch on this device
};

NoAllocState g_noalloc[kMaxDevices];

// Once per device, with that device current: resolve the device address of
// the static scratch array (the host-side symbol is only a stand-in and must
// never be handed to a kernel), query the device, set the kernels'
// shared-memory limit and resolve the tensor-map encoder. Nothing here
// allocates. Like the allocating path's set-up, a first call made while
// `stream` is being captured is refused (ATTN_ERR_UNSUPPORTED) and sets up
// nothing: the module look-ups it makes are not stream work and have no place
// in a graph.
attn_status_t noalloc_state(cudaStream_t stream, NoAllocState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  NoAllocState& st = g_noalloc[dev];
  if (!st.ready) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
      cudaGetLastError();
      return ATTN_ERR_UNSUPPORTED;
    }
    int major = 0, minor = 0, sms = 0, l2 = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;
    if (!configure_kernels()) return ATTN_ERR_UNSUPPORTED;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return ATTN_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    void* scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || scratch == nullptr)
      return ATTN_ERR_CUDA;
    st.sms = sms;
    st.l2 = l2;
    st.scratch = static_cast<int*>(scratch);
    st.ready = true;
  }
  *out = &st;
  return ATTN_OK;
}

// Reads a status word (synchronously) and clears it when set; *word gets its
// value. Allocates nothing.
attn_status_t read_and_clear(int* status, int* word) {
  *word = 0;
  if (cudaMemcpy(word, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (*word != 0 && cudaMemset(status, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace

// The per-device status word (allocated on first use) for the other kernels of
// this library, so that attn_device_check reports their timeouts as well.
namespace gb300_host {
attn_status_t device_status_word(cudaStream_t stream, int** status) {
  DeviceState* st = nullptr;
  const attn_status_t ds = device_state(stream, &st);
  if (ds != ATTN_OK) return ds;
  *status = st->status;
  return ATTN_OK;
}

// Every check attn_prefill_fwd_chunk makes before it launches (arguments,
// sizes, the device and the first-call set-up), without launching: the host
// entry point runs it on its staging pointers before enqueueing any copy.
attn_status_t forward_preflight(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, int64_t B, int64_t Lq, int64_t Lk,
                                int32_t n_q, int32_t n_kv, int32_t d_h, int32_t causal,
                                float scale, cudaStream_t stream) {
  const attn_status_t bad = validate(q, k, v, o, lse, B, Lq, Lk, n_q, n_kv, d_h, causal, scale);
  if (bad != ATTN_OK) return bad;
  DeviceState* st = nullptr;
  return device_state(stream, &st);
}
}  // namespace gb300_host

extern "C" {

attn_status_t attn_prefill_fwd_chunk(const void* q, const void* k, const void* v, void* o,
                                     float* lse, int64_t B, int64_t Lq, int64_t Lk, int32_t n_q,
                                     int32_t n_kv, int32_t d_h, int32_t causal, float scale,
                                     void* stream_ptr) {
  const attn_status_t bad = validate(q, k, v, o, lse, B, Lq, Lk, n_q, n_kv, d_h, causal, scale);
  if (bad != ATTN_OK) return bad;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  DeviceState* st = nullptr;
  const attn_status_t ds = device_state(stream, &st);
  if (ds != ATTN_OK) return ds;
  return launch_forward(q, k, v, o, lse, B, Lq, Lk, n_q, n_kv, d_h, causal, scale, stream,
                        st->status, st->sms, st->l2);
}

attn_status_t attn_prefill_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                               int64_t B, int64_t L, int32_t n_q, int32_t n_kv, int32_t d_h,
                               int32_t causal, float scale, void* stream_ptr) {
  return attn_prefill_fwd_chunk(q, k, v, o, lse, B, L, L, n_q, n_kv, d_h, causal, scale,
                                stream_ptr);
}

attn_status_t attn_prefill_fwd_fp8(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int64_t B, int64_t Lq, int64_t Lk, int32_t n_q,
                                   int32_t n_kv, int32_t d_h, int32_t causal, float scale,
                                   float q_descale, float k_descale, float v_descale,
                                   void* stream_ptr) {
  const attn_status_t bad = validate(q, k, v, o, lse, B, Lq, Lk, n_q, n_kv, d_h, causal, scale);
  if (bad != ATTN_OK) return bad;
  if (!std::isfinite(q_descale) || !std::isfinite(k_descale) || !std::isfinite(v_descale) ||
      !std::isfinite(scale * q_descale * k_descale))
    return ATTN_ERR_INVALID_ARG;
  if (d_h != 128) return ATTN_ERR_UNSUPPORTED;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  DeviceState* st = nullptr;
  const attn_status_t ds = device_state(stream, &st);
  if (ds != ATTN_OK) return ds;
  return launch_forward(q, k, v, o, lse, B, Lq, Lk, n_q, n_kv, d_h, causal, scale, stream,
                        st->status, st->sms, st->l2, true, q_descale * k_descale,
                        v_descale);
}

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG: invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED: unsupported size, head dim or device";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: CUDA call or kernel launch failed";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a device-side wait exceeded its limit";
    case ATTN_ERR_CHECK:
      return "ATTN_ERR_CHECK: a device-side consistency check of the debug build failed";
  }
  return "ATTN_ERR_UNKNOWN";
}

attn_status_t attn_device_check(void* stream_ptr) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  int* status = nullptr;
  int* noalloc_status = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_dev[dev].ready) status = g_dev[dev].status;
    if (g_noalloc[dev].ready) noalloc_status = g_noalloc[dev].scratch;
  }
  // the allocating entry points' word, then the allocation-free variant's
  int word = 0, noalloc_word = 0;
  if (status && read_and_clear(status, &word) != ATTN_OK) return ATTN_ERR_CUDA;
  if (noalloc_status && read_and_clear(noalloc_status, &noalloc_word) != ATTN_OK)
    return ATTN_ERR_CUDA;
  const int any = word | noalloc_word;
  if (any == 0) return ATTN_OK;
  return (any & kStatusCheck) ? ATTN_ERR_CHECK : ATTN_ERR_TIMEOUT;
}

int64_t attn_debug_check_count(void) {
#ifdef ATTN_DEBUG
  unsigned long long n = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpyFromSymbol(&n, g_dbg_checks, sizeof(n)) != cudaSuccess)
    return -1;
  return static_cast<int64_t>(n);
#else
  return -1;
#endif
}

attn_status_t attn_selftest_wait_timeout(int64_t spin_cycles, void* stream_ptr) {
  if (spin_cycles < 1 || spin_cycles > kSpinLimitCycles) return ATTN_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  DeviceState* st = nullptr;
  const attn_status_t ds = device_state(stream, &st);
  if (ds != ATTN_OK) return ds;
  Params p{};
  p.status = st->status;
  p.spin_limit = spin_cycles;
  wait_selftest_kernel<<<1, 64, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int64_t attn_prefill_grid_size(int64_t B, int64_t L, int32_t n_q, int32_t n_kv, int32_t d_h,
                               int32_t causal) {
  if (B < 1 || L < 1 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0 || (causal != 0 && causal != 1) ||
      (d_h != 64 && d_h != 128))
    return -1;
  int T = 0, units = 0;
  if (!count_units(B, L, L, n_q, n_kv, &T, &units)) return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  return units < sms ? units : sms;
}

}  // extern "C"

// ------------------------------------------ allocation-free entry points

extern "C" attn_status_t attn_prefill_fwd_noalloc(const void* q, const void* k, const void* v,
                                                  void* o, float* lse, int64_t B, int64_t L,
                                                  int32_t n_q, int32_t n_kv, int32_t d_h,
                                                  int32_t causal, float scale, void* stream_ptr) {
  const attn_status_t bad = validate(q, k, v, o, lse, B, L, L, n_q, n_kv, d_h, causal, scale);
  if (bad != ATTN_OK) return bad;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  NoAllocState* st = nullptr;
  const attn_status_t ds = noalloc_state(stream, &st);
  if (ds != ATTN_OK) return ds;
  // The status word is not cleared here: like the allocating path's word it
  // collects every wait timeout since attn_device_check last read it.
  return launch_forward(q, k, v, o, lse, B, L, L, n_q, n_kv, d_h, causal, scale, stream,
                        st->scratch, st->sms, st->l2);
}

extern "C" attn_status_t attn_selftest_wait_timeout_noalloc(int64_t spin_cycles,
                                                            void* stream_ptr) {
  if (spin_cycles < 1 || spin_cycles > kSpinLimitCycles) return ATTN_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  NoAllocState* st = nullptr;
  const attn_status_t ds = noalloc_state(stream, &st);
  if (ds != ATTN_OK) return ds;
  Params p{};
  p.status = st->scratch;
  p.spin_limit = spin_cycles;
  wait_selftest_kernel<<<1, 64, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
