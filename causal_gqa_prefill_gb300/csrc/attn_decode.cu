// attn_decode.cu — decode attention (one new query token per sequence) for
// GB300 (sm_103a), split over the key range.
//
// Decode attends one query row per head to the whole K/V cache; its work per
// byte is the GQA group size g, so it is bound by HBM bandwidth, not by the
// tensor cores ("Long-Context Attention Explained" (sevydevy), prefill vs
// decode: each decode step reads the whole KV cache; "Memory-bound vs
// compute-bound" lesson (Pranay), "Attention itself": decode attention is a
// batched matrix-vector product whose time is cache size over bandwidth).
// The kernel therefore streams K and V once through a TMA ring in shared
// memory and computes on the CUDA cores:
//
//   split kernel  grid = B * n_kv * S CTAs; CTA (b, kv head, split s) streams
//                 keys [s*R, (s+1)*R) of that head through a 4-stage ring of
//                 64-key K and V tiles (warp 8, lane 0 issues the copies) and
//                 eight compute warps run an online softmax for all g <= 8
//                 query heads of the group: each half-warp takes one key row,
//                 each lane 8 of the 128 dimensions; head dot products are
//                 finished with an 8-shuffle butterfly. The CTA writes its
//                 normalised partial output and log-sum-exp to the workspace.
//   combine       one CTA per (b, query head) merges the S partial results
//                 through their log-sum-exps into bf16 O and fp32 LSE.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_prefill.h"
#include "sm103_ptx.cuh"

namespace {

using namespace gb300;

constexpr int kDim = 128;            // head dimension handled here
constexpr int kRows = 64;            // keys per ring stage
constexpr int kStages = 4;
// Compute warps per CTA: as many as the registers allow (per-lane state
// grows with the group size), to hide the shuffle and FMA latency.
template <int G>
struct Warps {
  static constexpr int value = G <= 4 ? 16 : 8;
};
constexpr int kMaxComputeWarps = 16;
constexpr int kMaxG = 8;             // query heads per K/V head
constexpr int kTileBytes = kRows * kDim * 2;                  // one K or V stage tile
constexpr int kSmemBytes = kStages * 2 * kTileBytes + 1024;
constexpr int kMinSplitKeys = 256;
constexpr int kWaveCtas = 152;       // one CTA per SM on a 152-SM GB300
constexpr int kMaxWaves = 8;
constexpr long long kSpinLimit = 1ll << 31;
constexpr float kRescale = 8.0f;     // lazy running-max threshold (log2 units)

struct DecodeParams {
  const uint16_t* q;     // bf16 [B, 1, n_q, 128]
  float* part_o;         // fp32 [B, n_q, S, 128] normalised partial outputs
  float* part_lse;       // fp32 [B, n_q, S] partial log-sum-exp (natural log)
  int* status;           // unused slot for symmetry with prefill (may be null)
  int Lk, n_q, n_kv, g, S, keys_per_split;
  float c;               // scale * log2(e)
};

// Per-warp partial state for the final merge: kMaxComputeWarps * 4 heads or
// 8 warps * 8 heads, whichever the instance uses, fit in 16 KiB of outputs.
struct DecodeCtl {
  uint64_t full[kStages], empty[kStages];
  float m[kMaxComputeWarps][kMaxG], l[kMaxComputeWarps][kMaxG];
  float o[kMaxComputeWarps * kMaxG / 2][kDim];
};

// Heads rounded up to a power of two for the butterfly.
template <int G>
struct Pow2 {
  static constexpr int value = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8;
};

// Lane holding head h's full dot product after the butterfly over GP (a power
// of two) heads: the i-th halving step (offset 8 >> i) keeps the upper half of
// the remaining heads on lanes with that offset bit set.
template <int GP>
__device__ __forceinline__ int butterfly_owner(int h) {
  int lane = 0;
  int bit = GP >> 1, off = 8;
  while (bit > 0) {
    if (h & bit) lane |= off;
    bit >>= 1;
    off >>= 1;
  }
  return lane;
}

// Number of key splits S (CTAs = B * n_kv * S). Chooses the S whose CTAs
// fill whole waves of one CTA per SM (152 SMs) best, over at most kMaxWaves
// waves and with at least kMinSplitKeys keys per split; ties go to fewer
// waves. A pure function of the sizes, so the workspace size needs no device.
int64_t decode_splits(int64_t B, int64_t Lk, int32_t n_kv) {
  const int64_t heads = B * n_kv;
  const int64_t cap = (Lk + kMinSplitKeys - 1) / kMinSplitKeys;
  int64_t best = 1;
  double best_eff = -1.0;
  for (int64_t s = 1; s <= cap; ++s) {
    const int64_t ctas = heads * s;
    const int64_t waves = (ctas + kWaveCtas - 1) / kWaveCtas;
    if (waves > kMaxWaves) break;
    const double eff = static_cast<double>(ctas) / static_cast<double>(waves * kWaveCtas);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

__device__ __forceinline__ bool spin_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = clock64_now();
  while (!mbar_try_wait(bar, parity))
    if (static_cast<long long>(clock64_now() - t0) > kSpinLimit) return false;
  return true;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// G: query heads per K/V head (1..8).
template <int G>
__global__ void __launch_bounds__(32 * (Warps<G>::value + 1), 1)
attn_decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  constexpr int kComputeWarps = Warps<G>::value;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ DecodeCtl ctl;
  const uint32_t base = (smem_addr(dyn_smem) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x % p.S;
  const int grp = blockIdx.x / p.S;              // b * n_kv + kv head
  const int b = grp / p.n_kv, kvh = grp - b * p.n_kv;
  const int k_begin = split * p.keys_per_split;
  const int k_end = min(p.Lk, k_begin + p.keys_per_split);
  const int n_tiles = (k_end - k_begin + kRows - 1) / kRows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&ctl.full[s]), 1);
      mbar_init(smem_addr(&ctl.empty[s]), kComputeWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    // Producer: K and V tiles of 64 keys (two 64-dimension boxes each).
    if (lane == 0) {
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kStages, use = t / kStages;
        if (use > 0 && !spin_wait(smem_addr(&ctl.empty[s]), (use - 1) & 1)) break;
        const uint32_t bar = smem_addr(&ctl.full[s]);
        const uint32_t dk = base + s * 2 * kTileBytes, dv = dk + kTileBytes;
        mbar_arrive_expect_tx(bar, 2 * kTileBytes);
        const int row = k_begin + t * kRows;
        for (int c = 0; c < 2; ++c) {
          tma_load_4d(dk + c * (kTileBytes / 2), &tmK, bar, c * 64, kvh, row, b);
          tma_load_4d(dv + c * (kTileBytes / 2), &tmV, bar, c * 64, kvh, row, b);
        }
      }
      // let the last copies land before the CTA can exit
      for (int s = 0; s < kStages && s < n_tiles; ++s) {
        const int last = s + ((n_tiles - 1 - s) / kStages) * kStages;
        spin_wait(smem_addr(&ctl.full[s]), (last / kStages) & 1);
      }
    }
    return;
  }

  // ---- compute warps
  const int half = lane >> 4;            // which of the warp's two key rows
  const int L = lane & 15;               // dimension slice: [8L, 8L + 8)
  const int chunk = L >> 3;              // 64-dimension box of the slice
  const int coff = (L & 7) * 16;         // byte offset of the slice inside a box row
  float q[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint4 w = *reinterpret_cast<const uint4*>(
        p.q + (static_cast<size_t>(b) * p.n_q + kvh * G + h) * kDim + 8 * L);
    // scale * log2(e) folded into q: dot products come out in log2 units
    q[h][0] = bf16_lo(w.x) * p.c; q[h][1] = bf16_hi(w.x) * p.c;
    q[h][2] = bf16_lo(w.y) * p.c; q[h][3] = bf16_hi(w.y) * p.c;
    q[h][4] = bf16_lo(w.z) * p.c; q[h][5] = bf16_hi(w.z) * p.c;
    q[h][6] = bf16_lo(w.w) * p.c; q[h][7] = bf16_hi(w.w) * p.c;
  }
  constexpr int GP = Pow2<G>::value;
  // After the butterfly this lane holds the full score of head `mine` (lanes
  // 16/GP apart share a head); it alone keeps that head's running max and sum
  // and computes its weight, which the row's lanes then broadcast.
  int mine = 0;
#pragma unroll
  for (int h = 0; h < GP; ++h)
    if (butterfly_owner<GP>(h) == (L & (16 - 16 / GP))) mine = h;
  float m_own = -INFINITY, l_own = 0.0f;
  float o[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) o[h][i] = 0.0f;

  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % kStages;
    if (!spin_wait(smem_addr(&ctl.full[s]), (t / kStages) & 1)) break;
    const uint32_t sk = base + s * 2 * kTileBytes, sv = sk + kTileBytes;
    // this warp's 16 rows of the tile, two per step
    for (int rr = 0; rr < kRows / kComputeWarps; rr += 2) {
      const int r = warp * (kRows / kComputeWarps) + rr + half;
      const int key = k_begin + t * kRows + r;
      uint4 kw, vw;
      const uint32_t off = chunk * (kTileBytes / 2) + r * 128 + coff;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(kw.x), "=r"(kw.y), "=r"(kw.z), "=r"(kw.w) : "r"(sk + off));
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(vw.x), "=r"(vw.y), "=r"(vw.z), "=r"(vw.w) : "r"(sv + off));
      const float kf[8] = {bf16_lo(kw.x), bf16_hi(kw.x), bf16_lo(kw.y), bf16_hi(kw.y),
                           bf16_lo(kw.z), bf16_hi(kw.z), bf16_lo(kw.w), bf16_hi(kw.w)};
      // partial dot products of this lane's 8 dimensions, all heads (packed
      // pairs of dimensions, folded at the end); heads past G are zero
      float part[GP];
#pragma unroll
      for (int h = G; h < GP; ++h) part[h] = 0.0f;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        uint64_t a = f32x2_pack(q[h][0] * kf[0], q[h][1] * kf[1]);
#pragma unroll
        for (int i = 2; i < 8; i += 2)
          a = ffma2(f32x2_pack(q[h][i], q[h][i + 1]), f32x2_pack(kf[i], kf[i + 1]), a);
        float a0, a1;
        f32x2_unpack(a, a0, a1);
        part[h] = a0 + a1;
      }
      // butterfly over the 16 lanes of this row: each halving step sends half
      // of the remaining heads across, so after log2(G) steps a lane holds one
      // head summed over 16 / G lanes, and the remaining offsets finish the sum
#pragma unroll
      for (int off = 8, nv = GP; off >= 1; off >>= 1) {
        if (nv > 1) {
          const int hn = nv >> 1;
          const bool up = L & off;
#pragma unroll
          for (int i = 0; i < hn; ++i) {
            const float send = up ? part[i] : part[i + hn];
            const float keep = up ? part[i + hn] : part[i];
            part[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
          }
          nv = hn;
        } else {
          part[0] += __shfl_xor_sync(0xffffffffu, part[0], off);
        }
      }
      // the owner lane's online-softmax step for its head (log2 units); keys
      // past this split (or past the cache) get weight 0
      const float x = part[0];
      const bool valid = key < k_end && mine < G;
      const bool grow = valid && x > m_own + kRescale;   // lazy running max: rare after the first keys
      if (__any_sync(0xffffffffu, grow)) {
        const float alpha = grow ? ex2_approx(m_own - x) : 1.0f;
        if (grow) {
          m_own = x;
          l_own *= alpha;
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float ah = __shfl_sync(0xffffffffu, alpha, (half << 4) | butterfly_owner<GP>(h));
#pragma unroll
          for (int i = 0; i < 8; ++i) o[h][i] *= ah;
        }
      }
      const float pw_own = valid ? ex2_approx(x - m_own) : 0.0f;
      l_own += pw_own;
      const float vf[8] = {bf16_lo(vw.x), bf16_hi(vw.x), bf16_lo(vw.y), bf16_hi(vw.y),
                           bf16_lo(vw.z), bf16_hi(vw.z), bf16_lo(vw.w), bf16_hi(vw.w)};
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pw = __shfl_sync(0xffffffffu, pw_own, (half << 4) | butterfly_owner<GP>(h));
        const uint64_t pw2 = f32x2_pack(pw, pw);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const uint64_t r2 = ffma2(pw2, f32x2_pack(vf[i], vf[i + 1]), f32x2_pack(o[h][i], o[h][i + 1]));
          f32x2_unpack(r2, o[h][i], o[h][i + 1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl.empty[s]));
  }

  // every lane takes each head's running max and sum from that head's owner
  float m[G], l[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = __shfl_sync(0xffffffffu, m_own, (half << 4) | butterfly_owner<GP>(h));
    l[h] = __shfl_sync(0xffffffffu, l_own, (half << 4) | butterfly_owner<GP>(h));
  }
  // merge the warp's two rows (lanes L and L+16 hold the same dimensions)
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float mo = __shfl_xor_sync(0xffffffffu, m[h], 16);
    const float lo = __shfl_xor_sync(0xffffffffu, l[h], 16);
    const float mn = fmaxf(m[h], mo);
    const float a = (m[h] == -INFINITY) ? 0.0f : ex2_approx(m[h] - mn);
    const float bb = (mo == -INFINITY) ? 0.0f : ex2_approx(mo - mn);
    l[h] = l[h] * a + lo * bb;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float oo = __shfl_xor_sync(0xffffffffu, o[h][i], 16);
      o[h][i] = o[h][i] * a + oo * bb;
    }
    m[h] = mn;
  }
  if (half == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (L == 0) {
        ctl.m[warp][h] = m[h];
        ctl.l[warp][h] = l[h];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ctl.o[warp * G + h][8 * L + i] = o[h][i];
    }
  }
  // merge the compute warps (named barrier over those warps only; the
  // producer warp has left)
  asm volatile("bar.sync 1, %0;" ::"r"(32 * kComputeWarps) : "memory");
  for (int hd = threadIdx.x; hd < p.g * kDim; hd += 32 * kComputeWarps) {
    const int h = hd / kDim, d = hd - h * kDim;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) mx = fmaxf(mx, ctl.m[w][h]);
    float lt = 0.0f, ot = 0.0f;
#pragma unroll
    for (int w = 0; w < kComputeWarps; ++w) {
      const float a = (ctl.m[w][h] == -INFINITY) ? 0.0f : ex2_approx(ctl.m[w][h] - mx);
      lt += ctl.l[w][h] * a;
      ot += ctl.o[w * G + h][d] * a;
    }
    const size_t row = (static_cast<size_t>(b) * p.n_q + kvh * p.g + h) * p.S + split;
    p.part_o[row * kDim + d] = (lt > 0.0f) ? ot / lt : 0.0f;
    if (d == 0)
      p.part_lse[row] = (lt > 0.0f) ? (mx + log2f(lt)) * 0.69314718055994530942f : -INFINITY;
  }
}

// One CTA of kCombineWarps warps per (b, query head): O = sum_s w_s O_s,
// w_s = exp(lse_s - LSE). The warps take interleaved splits (independent
// loads, so many are in flight at once), each lane four dimensions; the warps'
// sums are added in shared memory.
constexpr int kCombineWarps = 8;
__global__ void __launch_bounds__(32 * kCombineWarps)
attn_decode_combine_kernel(const float* part_o, const float* part_lse, uint16_t* o, float* lse,
                           int S) {
  __shared__ float red_m[kCombineWarps], red_w[kCombineWarps];
  __shared__ float4 red_o[kCombineWarps][32];
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* pl = part_lse + static_cast<size_t>(row) * S;
  float mx = -INFINITY;
  for (int s = threadIdx.x; s < S; s += blockDim.x) mx = fmaxf(mx, pl[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red_m[warp] = mx;
  __syncthreads();
  mx = red_m[0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) mx = fmaxf(mx, red_m[w]);
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  float wsum = 0.0f;
#pragma unroll 4
  for (int s = warp; s < S; s += kCombineWarps) {
    const float ls = pl[s];
    const float w = (ls == -INFINITY) ? 0.0f : __expf(ls - mx);
    const float4 v = *reinterpret_cast<const float4*>(part_o + (static_cast<size_t>(row) * S + s) *
                                                                   kDim + 4 * lane);
    wsum += w;
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  red_o[warp][lane] = acc;
  if (lane == 0) red_w[warp] = wsum;
  __syncthreads();
  if (warp == 0) {
    float4 t = red_o[0][lane];
    float ws = red_w[0];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) {
      const float4 u = red_o[w][lane];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
      ws += red_w[w];
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

struct DecodeDevice {
  bool ready = false;
  int sms = 0;
};
constexpr int kMaxDevices = 64;
std::mutex g_decode_mutex;
DecodeDevice g_decode_dev[kMaxDevices];
EncodeTiledFn g_decode_encode = nullptr;

template <int G>
void launch_split(unsigned grid, cudaStream_t stream, const CUtensorMap& mk, const CUtensorMap& mv,
                  const DecodeParams& p) {
  attn_decode_split_kernel<G><<<grid, 32 * (Warps<G>::value + 1), kSmemBytes, stream>>>(mk, mv, p);
}

template <int G>
bool set_smem() {
  return cudaFuncSetAttribute(attn_decode_split_kernel<G>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes) == cudaSuccess;
}

attn_status_t decode_device_ready() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_decode_mutex);
  DecodeDevice& st = g_decode_dev[dev];
  if (st.ready) return ATTN_OK;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;
  if (!g_decode_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return ATTN_ERR_CUDA;
    g_decode_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  if (!set_smem<1>() || !set_smem<2>() || !set_smem<3>() || !set_smem<4>() || !set_smem<5>() ||
      !set_smem<6>() || !set_smem<7>() || !set_smem<8>())
    return ATTN_ERR_CUDA;
  st.ready = true;
  return ATTN_OK;
}

// K or V [B, Lk, H, 128] bf16 as (D, H, L, B), 64 x 1 x 64 x 1 boxes, no swizzle.
bool encode_kv(CUtensorMap* map, const void* ptr, int H, int64_t Lk, int64_t B) {
  const cuuint64_t dims[4] = {kDim, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(Lk),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {kDim * 2, static_cast<cuuint64_t>(H) * kDim * 2,
                                 static_cast<cuuint64_t>(Lk) * H * kDim * 2};
  const cuuint32_t box[4] = {64, 1, kRows, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return g_decode_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                         strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool decode_sizes_ok(int64_t B, int64_t Lk, int32_t n_q, int32_t n_kv, int32_t d_h) {
  return B >= 1 && Lk >= 1 && n_q >= 1 && n_kv >= 1 && n_q % n_kv == 0 && d_h >= 1;
}

}  // namespace

extern "C" {

int64_t attn_decode_workspace_bytes(int64_t B, int64_t Lk, int32_t n_q, int32_t n_kv,
                                    int32_t d_h) {
  if (!decode_sizes_ok(B, Lk, n_q, n_kv, d_h) || d_h != kDim) return -1;
  const int64_t S = decode_splits(B, Lk, n_kv);
  const int64_t rows = B * n_q * S;
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
  const int64_t need = attn_decode_workspace_bytes(B, Lk, n_q, n_kv, d_h);
  if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  const attn_status_t ds = decode_device_ready();
  if (ds != ATTN_OK) return ds;

  const int64_t S = decode_splits(B, Lk, n_kv);
  CUtensorMap mk, mv;
  if (!encode_kv(&mk, k, n_kv, Lk, B) || !encode_kv(&mv, v, n_kv, Lk, B)) return ATTN_ERR_CUDA;
  DecodeParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.part_o = static_cast<float*>(workspace);
  p.part_lse = p.part_o + B * n_q * S * kDim;
  p.status = nullptr;
  p.Lk = static_cast<int>(Lk);
  p.n_q = n_q;
  p.n_kv = n_kv;
  p.g = n_q / n_kv;
  p.S = static_cast<int>(S);
  const int64_t per = (Lk + S - 1) / S;
  p.keys_per_split = static_cast<int>(((per + kRows - 1) / kRows) * kRows);
  p.c = scale * 1.4426950408889634f;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int64_t ctas = B * n_kv * S;
  const unsigned grid = static_cast<unsigned>(ctas);
  switch (p.g) {
    case 1: launch_split<1>(grid, stream, mk, mv, p); break;
    case 2: launch_split<2>(grid, stream, mk, mv, p); break;
    case 3: launch_split<3>(grid, stream, mk, mv, p); break;
    case 4: launch_split<4>(grid, stream, mk, mv, p); break;
    case 5: launch_split<5>(grid, stream, mk, mv, p); break;
    case 6: launch_split<6>(grid, stream, mk, mv, p); break;
    case 7: launch_split<7>(grid, stream, mk, mv, p); break;
    default: launch_split<8>(grid, stream, mk, mv, p); break;
  }
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  const int rows = static_cast<int>(B * n_q);
  attn_decode_combine_kernel<<<rows, 32 * kCombineWarps, 0, stream>>>(
      p.part_o, p.part_lse, static_cast<uint16_t*>(o), lse, p.S);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
