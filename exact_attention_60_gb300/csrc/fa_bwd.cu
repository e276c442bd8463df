// fa_bwd.cu -- FlashAttention-2 backward for GB300 (sm_103a), and its C ABI.
//
// What is computed (per batch b, head h), given Q, K, V, the forward output O, its
// row statistic LSE and the loss gradient dO:
//   P_ij  = exp(scale * Q_i.K_j - LSE_i)          (recomputed, never stored)
//   dV_j  = sum_i P_ij dO_i
//   dP_ij = dO_i . V_j
//   dS_ij = P_ij (dP_ij - Delta_i),  Delta_i = dO_i . O_i  (= sum_j P_ij dP_ij)
//   dQ_i  = scale sum_j dS_ij K_j,   dK_j = scale sum_i dS_ij Q_i
// over the allowed pairs (all j < Lk, j <= i when causal, or the band and key-padding
// mask of the strided forward).  The principle --
// keep the per-row statistic from the forward pass and recompute P from it
// instead of storing the score matrix -- is the one the wsisp.com post
// "FlashAttention-2 forward in Triton" states for the backward pass, which it
// leaves to later work; the formulas are the chain rule through O = P V, the row
// softmax and S = scale Q K^T.
//
// Three kernels on one stream:
//   fa_bwd_delta_kernel : Delta = rowsum(dO * O), fp32, memory-bound.
//   fa_bwd_dkdv_kernel  : one unit = one 128-key tile of one head; streams the
//                         query tiles that see it.  TMEM: S^T | dP^T | dV | dK.
//                           S^T  = K Q^T,  dP^T = V dO^T        (A, B in smem)
//                           dV  += P^T dO, dK  += dS^T Q        (A = P^T / dS^T in TMEM)
//                         Two warpgroups (thread = key row, 64 columns each) turn
//                         S^T into P^T (bf16, over S^T) and dP^T into dS^T (bf16,
//                         over dP^T).
//   fa_bwd_dq_kernel    : one unit = one 128-query tile; streams its key tiles.
//                         TMEM: S | dP | dQ.  S = Q K^T, dP = dO V^T, dQ += dS K.
// Splitting dQ from dK/dV costs two extra GEMMs per tile pair but needs no
// atomics and no dQ accumulator in global memory.  Roles per CTA (320 threads):
// warps 0-7 two compute warpgroups sharing each row's columns, warp 8 TMA loads, warp
// 9 MMA issue (the whole warp runs the loop; one elected lane issues each tcgen05.mma /
// commit).  Every wait
// is bounded in time; a wait that runs out records FA_ERR_TIMEOUT in this file's
// status word (read by fa_last_device_status) and every role drains and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fab {

namespace ptx = fa::ptx;

__device__ unsigned int g_bwd_status;

constexpr int kBlk = 128;          // rows per tile (queries or keys), one M=128 MMA
constexpr int kThreads = 320;     // two compute warpgroups, load warp, MMA warp
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kComputeThreads = 256;

// The per-element work of the backward pass (P from S and the saved LSE, dS from P, dP
// and Delta) needs no reduction along a row, so the two compute warpgroups share each
// row: warpgroup g takes columns [64g, 64g + 64) of S (dP) and writes its 32 packed
// bf16 columns of P (dS) over the first half of that range, which only it has read.
// The A operand of the next MMA (K = 128) is then columns [0, 32) and [64, 96).
__device__ __forceinline__ uint32_t packed_col(int kk) {   // TMEM column of K-slice kk (16 rows)
  return kk < 4 ? 8u * kk : 64u + 8u * (kk - 4);
}
constexpr unsigned long long kDefaultWaitNs = 1000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

enum Site : uint32_t { kSiteLoad = 1, kSiteMma = 2, kSiteCompute = 3, kSiteEpilogue = 4 };

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned long long limit_ns, uint32_t site) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicCAS(&g_bwd_status, 0u, static_cast<unsigned>(FA_ERR_TIMEOUT) | (site << 8));
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long limit_ns, uint32_t site) {
  return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, limit_ns, site));
}

__device__ __noinline__ bool drain_phase(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// tcgen05 instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major or (b_mn_major) MN-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major, bool f16 = false) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Two floats to the packed 16-bit pair of the I/O type, and back.
template <bool kF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kF16) return ptx::pack_f16x2(lo, hi);
  else return ptx::pack_bf16x2(lo, hi);
}
template <bool kF16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  if constexpr (kF16) {
    __half2 h;
    memcpy(&h, &v, 4);
    return __half22float2(h);
  } else {
    return ptx::unpack_bf16x2(v);
  }
}

// Element (bh, row) of a [B,H,L,D] tensor with element strides st.
__device__ __forceinline__ long long row_offset(const long long* st, int H, int bh, long long row) {
  const int b = bh / H, h = bh - b * H;
  return b * st[0] + h * st[1] + row * st[2];
}

// Shared-memory descriptor of a 128B-swizzled operand (see the forward kernel).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

struct BwdParams {
  CUtensorMap tm_q;    // 4-D views [B][H][L][D] (caller's strides), box 64 x 128 x 1 x 1, 128B swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  const float* delta;  // [B*H][nq*128] rowsum(dO * O), 0 past Lq
  const float* lse2;   // [B*H][nq*128] LSE * log2(e), +inf past Lq
  uint16_t* dq;        // bf16 or fp16 elements, written through the strides below
  uint16_t* dk;
  uint16_t* dv;
  long long dq_s[3], dk_s[3], dv_s[3];   // element strides {batch, head, row}
  int dq_v8, dkv_v8;   // dQ / dK and dV: base and strides multiples of 32 bytes (32-byte stores)
  int bh_count;
  int H;
  int Lq;
  int Lk;
  int win_left;        // key j allowed for query i iff i - win_left <= j <= i + win_right
  int win_right;       //   (-1: unbounded side); causal is (-1, 0), the full mask (-1, -1)
  const int* kv_len;   // per-batch valid keys (key padding), device memory; nullptr = none
  int nq;              // query tiles: ceil(Lq / 128)
  int nk;              // key tiles:   ceil(Lk / 128)
  int n_units;
  int group_heads;     // causal-like orders: heads per group (a group's streamed tiles stay in L2)
  int* unit_ctr;       // units drawn after each CTA's first, zeroed by the Delta kernel
  float scale;
  float scale_log2;    // scale * log2(e)
  uint32_t flags;      // test hooks (fa_debug_set): bit 0 withholds the first V tile of dK/dV
  unsigned long long wait_limit_ns;
};

template <int HD>
struct Tiles {
  static constexpr int kTileBytes = kBlk * HD * 2;   // one 128 x HD bf16 tile
  static constexpr int kRegionBytes = kBlk * 128;    // 128 rows x 64 bf16: one swizzle column
  static constexpr int kRegions = HD / 64;
};

// Valid (unpadded) keys of head bh's batch.
__device__ __forceinline__ int batch_keys(const BwdParams& p, int bh) {
  return p.kv_len ? min(max(__ldg(p.kv_len + bh / p.H), 0), p.Lk) : p.Lk;
}

// The query tiles a dK/dV unit (key tile kt) streams, [*qa, *qa + *n): those holding a query
// q with q - left <= k <= q + right for some unpadded key k of the tile.
__device__ __forceinline__ void dkdv_range(const BwdParams& p, int kt, int kvl, int* qa, int* n) {
  const long long k0 = static_cast<long long>(kt) * kBlk, k1 = min(k0 + kBlk - 1, static_cast<long long>(kvl) - 1);
  const long long q_lo = p.win_right < 0 ? 0 : max(0ll, k0 - p.win_right);
  const long long q_hi = p.win_left < 0 ? p.Lq - 1 : min(static_cast<long long>(p.Lq) - 1, k1 + p.win_left);
  *qa = 0;
  *n = 0;
  if (k1 < k0 || q_hi < q_lo) return;
  *qa = static_cast<int>(q_lo / kBlk);
  *n = static_cast<int>(q_hi / kBlk) - *qa + 1;
}

// The key tiles a dQ unit (query tile qt) streams, [*ka, *ka + *n): those holding an
// allowed key of some query of the tile.
__device__ __forceinline__ void dq_range(const BwdParams& p, int qt, int kvl, int* ka, int* n) {
  const long long q0 = static_cast<long long>(qt) * kBlk, q1 = min(q0 + kBlk - 1, static_cast<long long>(p.Lq) - 1);
  const long long lo = p.win_left < 0 ? 0 : max(0ll, q0 - p.win_left);
  const long long lim = p.win_right < 0 ? kvl : min(static_cast<long long>(kvl), q1 + p.win_right + 1);
  *ka = 0;
  *n = 0;
  if (lim <= lo) return;
  *ka = static_cast<int>(lo / kBlk);
  *n = static_cast<int>((lim - 1) / kBlk) - *ka + 1;
}

// Unit order.  Causal-like masks (the first key tiles are seen by the most queries, the
// last query tiles see the most keys) go heaviest first within groups of group_heads
// heads, one group after another: the units in flight then share a group's streamed
// tiles in L2 instead of every head's at once.  Other masks go head by head.  Units are
// handed out dynamically (below), so the heavy-first order also balances the CTAs.
__device__ __forceinline__ void grouped_unit(const BwdParams& p, int idx, int n_tiles, int& bh, int& t) {
  const int per_group = p.group_heads * n_tiles;
  const int grp = idx / per_group;
  const int i = idx - grp * per_group;
  const int h0 = grp * p.group_heads;
  const int hc = min(p.group_heads, p.bh_count - h0);   // the last group may be smaller
  t = i / hc;
  bh = h0 + (i - t * hc);
}
__device__ __forceinline__ void dkdv_unit(const BwdParams& p, int idx, int& bh, int& kt) {
  if (p.win_left < 0 && p.win_right >= 0) {
    grouped_unit(p, idx, p.nk, bh, kt);
  } else {
    bh = idx / p.nk;
    kt = idx % p.nk;
  }
}
__device__ __forceinline__ void dq_unit(const BwdParams& p, int idx, int& bh, int& qt) {
  if (p.win_left < 0 && p.win_right >= 0) {
    int i;
    grouped_unit(p, idx, p.nq, bh, i);
    qt = p.nq - 1 - i;
  } else {
    bh = idx / p.nq;
    qt = idx % p.nq;
  }
}

// Dynamic unit hand-out.  Each CTA's first unit is its block index; the load warp draws
// every later one from a global counter and passes it to the MMA warp and the compute
// warps through a ring of shared-memory slots (full: count 1, the load warp; empty:
// count 9, the eight compute warps and the MMA warp).  A drawn index >= n_units ends
// every role's loop.  Both functions are warp-uniform.
constexpr int kUnitRing = 4;
constexpr int kUnitConsumers = 9;
constexpr int kCtrStride = 32;   // the two counters sit 128 bytes apart in the workspace's last 256

__device__ __forceinline__ bool unit_produce(const BwdParams& p, uint32_t full0, uint32_t empty0,
                                             volatile int* slots, int r, int& idx, volatile int* abort_flag,
                                             unsigned long long limit, uint32_t site) {
  const int s = r % kUnitRing;
  if (!wait_warp(empty0 + 8u * s, ((r / kUnitRing) & 1) ^ 1u, abort_flag, limit, site)) return false;
  int v = 0;
  if ((threadIdx.x & 31) == 0) {
    v = r == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(p.unit_ctr, 1);
    slots[s] = v;
    ptx::mbar_arrive(full0 + 8u * s);   // release: the slot's value is visible to the waiters
  }
  idx = __shfl_sync(0xffffffffu, v, 0);
  return true;
}

__device__ __forceinline__ bool unit_consume(uint32_t full0, uint32_t empty0, const volatile int* slots, int r,
                                             int& idx, volatile int* abort_flag, unsigned long long limit,
                                             uint32_t site) {
  const int s = r % kUnitRing;
  if (!wait_warp(full0 + 8u * s, (r / kUnitRing) & 1, abort_flag, limit, site)) return false;
  idx = slots[s];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(empty0 + 8u * s);
  return true;
}

// ------------------------------------------------------------------ Delta = rowsum(dO * O)
// Rows are numbered over whole 128-row tiles (row = bh * Lpad + q, Lpad = nq * 128), so
// both outputs can be copied into shared memory a tile at a time with bulk copies:
// delta[row] = dO_q . O_q and lse2[row] = LSE_q * log2(e) for q < Lq; 0 and +inf past Lq
// (+inf makes every recomputed probability of a padded query exactly 0).
// Rows of O and dO are read through their strides (o_s, do_s: {batch, head, row}).
struct DeltaArgs {
  const uint16_t* O;
  const uint16_t* dO;
  const float* lse;
  float* delta;
  float* lse2;
  long long o_s[3], do_s[3];
  long long rows_pad;
  int* unit_ctr;   // the dK/dV and dQ kernels' unit counters, zeroed here
  int Lq, Lpad, H;
};

template <int HD, bool kF16>
__global__ void __launch_bounds__(256) fa_bwd_delta_kernel(const __grid_constant__ DeltaArgs a) {
  // Launched as a programmatic dependent for short problems: the previous kernel (possibly
  // the last backward's dQ kernel, which reads this workspace) completes before any access.
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  constexpr int kT = HD / 8;   // threads per row, 8 elements (16 bytes) each
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = tid / kT;
  const int part = static_cast<int>(tid % kT);
  const int bh = static_cast<int>(row / a.Lpad);
  const int q = static_cast<int>(row - static_cast<long long>(bh) * a.Lpad);
  const bool valid = row < a.rows_pad && q < a.Lq;
  if (tid == 0) {
    a.unit_ctr[0] = 0;
    a.unit_ctr[kCtrStride] = 0;
  }
  float acc = 0.0f;
  if (valid) {
    const uint4 x4 = __ldg(reinterpret_cast<const uint4*>(a.O + row_offset(a.o_s, a.H, bh, q)) + part);
    const uint4 y4 = __ldg(reinterpret_cast<const uint4*>(a.dO + row_offset(a.do_s, a.H, bh, q)) + part);
    const uint32_t xv[4] = {x4.x, x4.y, x4.z, x4.w}, yv[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = unpack2<kF16>(xv[e]), y = unpack2<kF16>(yv[e]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int off = kT / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (part == 0 && row < a.rows_pad) {
    a.delta[row] = valid ? acc : 0.0f;
    a.lse2[row] = valid ? __ldg(a.lse + static_cast<long long>(bh) * a.Lq + q) * kLog2e : INFINITY;
  }
}

// ------------------------------------------------------------------ dK, dV
template <int HD>
struct DkdvLayout {
  using T = Tiles<HD>;
  static constexpr int kStages = (HD == 128) ? 2 : 4;           // (Q, dO, LSE, Delta) ring
  static constexpr int kOffK = 0;
  static constexpr int kOffV = T::kTileBytes;
  static constexpr int kOffStage = 2 * T::kTileBytes;
  static constexpr int kStageBytes = 2 * T::kTileBytes + 1024;   // Q | dO | lse2[128] | delta[128]
  static constexpr int kOffBar = kOffStage + kStages * kStageBytes;
  static constexpr int kBarKvFull = 0, kBarKvEmpty = 1;
  static constexpr int kBarQFull = 2;                           // [kStages] Q and LSE*log2e
  static constexpr int kBarDoFull = kBarQFull + kStages;        // [kStages] dO and Delta
  static constexpr int kBarQdEmpty = kBarDoFull + kStages;      // [kStages]
  static constexpr int kBarSFull = kBarQdEmpty + kStages;
  static constexpr int kBarDpFull = kBarSFull + 1;
  static constexpr int kBarPFull = kBarDpFull + 1;              // count 256 (compute threads)
  static constexpr int kBarDsFull = kBarPFull + 1;              // count 256 (compute threads)
  static constexpr int kBarAccFull = kBarDsFull + 1;
  static constexpr int kBarAccEmpty = kBarAccFull + 1;          // count 256 (compute threads)
  static constexpr int kBarDrain = kBarAccEmpty + 1;
  static constexpr int kBarUnitFull = kBarDrain + 1;                // [kUnitRing]
  static constexpr int kBarUnitEmpty = kBarUnitFull + kUnitRing;    // [kUnitRing]
  static constexpr int kNumBars = kBarUnitEmpty + kUnitRing;
  static constexpr int kOffAbort = kOffBar + kNumBars * 8;
  static constexpr int kOffTmemSlot = kOffAbort + 4;
  static constexpr int kOffUnits = kOffTmemSlot + 4;                // int[kUnitRing]
  static constexpr int kBytes = kOffUnits + 4 * kUnitRing;
  static constexpr int kAlloc = kBytes + 1024;
  // TMEM columns: S^T | dP^T | dV | dK (P^T and dS^T as bf16 over the first 64 columns of S^T / dP^T)
  static constexpr uint32_t kColS = 0, kColDp = 128, kColDv = 256, kColDk = 256 + HD;
  static constexpr uint32_t kTmemCols = 512;
};
static_assert(DkdvLayout<128>::kAlloc <= 232448, "dK/dV shared memory (D=128)");
static_assert(DkdvLayout<64>::kAlloc <= 232448, "dK/dV shared memory (D=64)");

template <int HD, bool kF16>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using L = DkdvLayout<HD>;
  using T = Tiles<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_addr(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  volatile int* unit_slots = reinterpret_cast<volatile int*>(smem + L::kOffUnits);
  auto bar = [&](int idx) -> uint32_t { return sbase + L::kOffBar + 8u * idx; };
  auto stage_off = [&](int s) -> uint32_t { return L::kOffStage + s * L::kStageBytes; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(L::kBarKvFull), 1);
    ptx::mbar_init(bar(L::kBarKvEmpty), 1);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(L::kBarQFull + s), 1);
      ptx::mbar_init(bar(L::kBarDoFull + s), 1);
      ptx::mbar_init(bar(L::kBarQdEmpty + s), 1);
    }
    ptx::mbar_init(bar(L::kBarSFull), 1);
    ptx::mbar_init(bar(L::kBarDpFull), 1);
    ptx::mbar_init(bar(L::kBarPFull), kComputeThreads);
    ptx::mbar_init(bar(L::kBarDsFull), kComputeThreads);
    ptx::mbar_init(bar(L::kBarAccFull), 1);
    ptx::mbar_init(bar(L::kBarAccEmpty), kComputeThreads);
    ptx::mbar_init(bar(L::kBarDrain), 1);
    for (int s = 0; s < kUnitRing; ++s) {
      ptx::mbar_init(bar(L::kBarUnitFull + s), 1);
      ptx::mbar_init(bar(L::kBarUnitEmpty + s), kUnitConsumers);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), L::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const unsigned long long limit = p.wait_limit_ns;
  // Launched as a programmatic dependent for short problems: the set-up above overlapped the
  // previous kernel; nothing in global memory is touched before it completes.
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  if (warp < 8) {
    // ------------------------------------------------ compute warpgroups: thread = key row
    const int g = warp >> 2;                   // columns [64g, 64g + 64) of the row
    const int rw = warp & 3;                   // TMEM lane quarter this warp may access
    const int row = rw * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(rw * 32) << 16;
    const uint32_t t_s = tmem + lane_off + L::kColS + 64 * g;
    const uint32_t t_dp = tmem + lane_off + L::kColDp + 64 * g;
    const float sl2 = p.scale_log2;
    uint32_t it = 0;          // query tiles processed (s_full, dp_full phases; ring position)
    uint32_t acc_count = 0;   // units whose accumulators were read
    bool ok = true;
    int idx;
    for (int r = 0; ok; ++r) {
      ok = unit_consume(bar(L::kBarUnitFull), bar(L::kBarUnitEmpty), unit_slots, r, idx, abort_flag,
                        limit, kSiteCompute);
      if (!ok || idx >= p.n_units) break;
      int bh, kt;
      dkdv_unit(p, idx, bh, kt);
      const int kvl = batch_keys(p, bh);
      int q_first, n;
      dkdv_range(p, kt, kvl, &q_first, &n);
      const int k = kt * kBlk + row;   // this thread's key
      // warpgroup 0 writes dV, 1 writes dK
      uint16_t* mine = g ? p.dk + row_offset(p.dk_s, p.H, bh, k < p.Lk ? k : 0)
                         : p.dv + row_offset(p.dv_s, p.H, bh, k < p.Lk ? k : 0);
      if (n == 0) {   // no query sees these keys: their gradients are zero
        if (k < p.Lk)
          for (int c = 0; c < HD; c += 8) *reinterpret_cast<uint4*>(mine + c) = make_uint4(0, 0, 0, 0);
        continue;
      }
      for (int t = 0; t < n; ++t, ++it) {
        const int qt = q_first + t;
        const int s = static_cast<int>(it % L::kStages);
        const float* lse2 = reinterpret_cast<const float*>(smem + stage_off(s) + 2 * T::kTileBytes) + 64 * g;
        const float* dlt = lse2 + kBlk;
        // LSE (a bulk copy that lands with Q, the stage's first half) is read here: wait
        // for that half and for S^T, which the MMA warp commits; Delta comes with dO
        ok = __all_sync(0xffffffffu, wait_phase(bar(L::kBarQFull + s), (it / L::kStages) & 1, abort_flag,
                                                limit, kSiteCompute) &&
                                         wait_phase(bar(L::kBarSFull), it & 1, abort_flag, limit, kSiteCompute));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[64];
        ptx::tmem_ld32x32b_x64(t_s, sr);   // one load, one wait for the warpgroup's 64 columns
        // P^T_kq = exp2(sl2 * S - lse_q * log2e); padded queries carry lse2 = +inf (P = 0).
        // Key k is seen by query q iff k - right <= q <= k + left and k < kvl; only tiles the
        // band or the padding cuts are masked (a query without keys, LSE = -inf, is always in
        // such a tile).
        const int qb = qt * kBlk;   // first query of the tile
        const int kmin = kt * kBlk, kmax = kmin + kBlk - 1;
        const bool cut = kmax >= kvl || (p.win_right >= 0 && qb < kmax - p.win_right) ||
                         (p.win_left >= 0 && qb + kBlk - 1 > kmin + p.win_left);
        const int base = qb + 64 * g;   // query of column 0 of this warpgroup
        const int c_lo = (p.win_right < 0 ? 0 : k - p.win_right) - base;
        const int c_hi = (p.win_left < 0 ? INT_MAX / 2 : k + p.win_left) - base;
        const bool key_ok = k < kvl;
        float pr[64];
#pragma unroll
        for (int c = 0; c < 64; c += 4) {   // LSE * log2e of four queries per shared-memory load
          const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c);
          pr[c] = ptx::ex2_approx(fmaf(__uint_as_float(sr[c]), sl2, -l4.x));
          pr[c + 1] = ptx::ex2_approx(fmaf(__uint_as_float(sr[c + 1]), sl2, -l4.y));
          pr[c + 2] = ptx::ex2_approx(fmaf(__uint_as_float(sr[c + 2]), sl2, -l4.z));
          pr[c + 3] = ptx::ex2_approx(fmaf(__uint_as_float(sr[c + 3]), sl2, -l4.w));
        }
        if (cut) {
#pragma unroll
          for (int c = 0; c < 64; ++c) pr[c] = (key_ok && c >= c_lo && c <= c_hi) ? pr[c] : 0.0f;
        }
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = pack2<kF16>(pr[2 * c], pr[2 * c + 1]);
        ptx::tmem_st32x32b_x32(t_s, pk);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarPFull));
        // dS^T_kq = P^T_kq (dP^T_kq - Delta_q); the packed result lands over this warpgroup's
        // first 32 dP^T columns, after both halves have been read.  Delta came with dO.
        ok = __all_sync(0xffffffffu, wait_phase(bar(L::kBarDoFull + s), (it / L::kStages) & 1, abort_flag, limit,
                                                kSiteCompute) &&
                                         wait_phase(bar(L::kBarDpFull), it & 1, abort_flag, limit, kSiteCompute));
        if (!ok) break;
        ptx::tc_fence_after();
        ptx::tmem_ld32x32b_x64(t_dp, sr);
#pragma unroll
        for (int c = 0; c < 32; c += 2) {   // Delta of four queries per shared-memory load
          const float4 d4 = *reinterpret_cast<const float4*>(dlt + 2 * c);
          pk[c] = pack2<kF16>(pr[2 * c] * (__uint_as_float(sr[2 * c]) - d4.x),
                              pr[2 * c + 1] * (__uint_as_float(sr[2 * c + 1]) - d4.y));
          pk[c + 1] = pack2<kF16>(pr[2 * c + 2] * (__uint_as_float(sr[2 * c + 2]) - d4.z),
                                  pr[2 * c + 3] * (__uint_as_float(sr[2 * c + 3]) - d4.w));
        }
        ptx::tmem_st32x32b_x32(t_dp, pk);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarDsFull));
      }
      if (!ok) break;
      // Epilogue: warpgroup 0 writes dV, warpgroup 1 scale * dK, of this thread's key row.
      ok = __all_sync(0xffffffffu, wait_phase(bar(L::kBarAccFull), acc_count & 1, abort_flag, limit, kSiteEpilogue));
      if (!ok) break;
      ++acc_count;
      ptx::tc_fence_after();
      {
        // The whole accumulator row first, released at once (the next unit's first dV / dK
        // MMA may overwrite it), then scaled, packed and stored from registers.
        const uint32_t t_acc = tmem + lane_off + (g ? L::kColDk : L::kColDv);
        const float mul = g ? p.scale : 1.0f;
        uint32_t a[HD / 32][32];
#pragma unroll
        for (int k2 = 0; k2 < HD / 32; ++k2) ptx::tmem_ld32x32b_x32(t_acc + 32 * k2, a[k2]);
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarAccEmpty));
#pragma unroll
        for (int k2 = 0; k2 < HD / 32; ++k2) {
          uint32_t pk16[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk16[c] = pack2<kF16>(__uint_as_float(a[k2][2 * c]) * mul, __uint_as_float(a[k2][2 * c + 1]) * mul);
          if (k < p.Lk) {
            if (p.dkv_v8) {
              ptx::st_global_v8(mine + 32 * k2, pk16);
              ptx::st_global_v8(mine + 32 * k2 + 16, pk16 + 8);
            } else {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                reinterpret_cast<uint4*>(mine + 32 * k2)[v] = make_uint4(pk16[4 * v], pk16[4 * v + 1], pk16[4 * v + 2], pk16[4 * v + 3]);
            }
          }
        }
      }
    }
  } else if (warp == kLoadWarp) {
    // ------------------------------------------------ load warp
    if (lane == 0) {
      ptx::prefetch_tensormap(&p.tm_q);
      ptx::prefetch_tensormap(&p.tm_k);
      ptx::prefetch_tensormap(&p.tm_v);
      ptx::prefetch_tensormap(&p.tm_do);
    }
    uint32_t it = 0, units = 0;
    int last_fill[L::kStages];
    for (int s = 0; s < L::kStages; ++s) last_fill[s] = -1;
    bool ok = true;
    int idx;
    for (int r = 0; ok; ++r) {
      ok = unit_produce(p, bar(L::kBarUnitFull), bar(L::kBarUnitEmpty), unit_slots, r, idx, abort_flag,
                        limit, kSiteLoad);
      if (!ok || idx >= p.n_units) break;
      int bh, kt;
      dkdv_unit(p, idx, bh, kt);
      int q_first, n;
      dkdv_range(p, kt, batch_keys(p, bh), &q_first, &n);
      if (units > 0) {
        ok = wait_warp(bar(L::kBarKvEmpty), (units - 1) & 1, abort_flag, limit, kSiteLoad);
        if (!ok) break;
      }
      if (lane == 0) {
        // test hook (bit 0): the first unit's V tile is never loaded, so kv_full never
        // completes and the waits on it run out (FA_ERR_TIMEOUT) instead of the kernel hanging
        const bool withhold_v = (p.flags & 1u) && units == 0;
        ptx::mbar_arrive_expect_tx(bar(L::kBarKvFull), 2 * T::kTileBytes);
        for (int rg = 0; rg < T::kRegions; ++rg) {
          ptx::tma_load_4d(sbase + L::kOffK + rg * T::kRegionBytes, &p.tm_k, bar(L::kBarKvFull), 64 * rg, kt * kBlk, bh - (bh / p.H) * p.H, bh / p.H);
          if (!withhold_v)
            ptx::tma_load_4d(sbase + L::kOffV + rg * T::kRegionBytes, &p.tm_v, bar(L::kBarKvFull), 64 * rg, kt * kBlk, bh - (bh / p.H) * p.H, bh / p.H);
        }
      }
      ++units;
      for (int t = 0; t < n; ++t, ++it) {
        const int qt = q_first + t;
        const int s = static_cast<int>(it % L::kStages);
        ok = wait_warp(bar(L::kBarQdEmpty + s), ((it / L::kStages) & 1) ^ 1u, abort_flag, limit, kSiteLoad);
        if (!ok) break;
        if (lane == 0) {
          // Q and LSE first (S^T of the tile needs them), then dO and Delta (needed from
          // dP^T on), each half on its own barrier
          const uint32_t qfull = bar(L::kBarQFull + s), dofull = bar(L::kBarDoFull + s);
          const size_t rowp = (static_cast<size_t>(bh) * p.nq + qt) * kBlk;   // padded row of the tile
          ptx::mbar_arrive_expect_tx(qfull, T::kTileBytes + kBlk * 4);
          for (int rg = 0; rg < T::kRegions; ++rg)
            ptx::tma_load_4d(sbase + stage_off(s) + rg * T::kRegionBytes, &p.tm_q, qfull, 64 * rg, qt * kBlk, bh - (bh / p.H) * p.H, bh / p.H);
          ptx::bulk_load(sbase + stage_off(s) + 2 * T::kTileBytes, p.lse2 + rowp, kBlk * 4, qfull);
          ptx::mbar_arrive_expect_tx(dofull, T::kTileBytes + kBlk * 4);
          for (int rg = 0; rg < T::kRegions; ++rg)
            ptx::tma_load_4d(sbase + stage_off(s) + T::kTileBytes + rg * T::kRegionBytes, &p.tm_do, dofull, 64 * rg, qt * kBlk, bh - (bh / p.H) * p.H, bh / p.H);
          ptx::bulk_load(sbase + stage_off(s) + 2 * T::kTileBytes + kBlk * 4, p.delta + rowp, kBlk * 4, dofull);
        }
        last_fill[s] = static_cast<int>(it);
      }
    }
    // Drain: every copy this warp started has landed before the CTA exits.
    if (units > 0) drain_phase(bar(L::kBarKvFull), (units - 1) & 1, limit);
    for (int s = 0; s < L::kStages; ++s)
      if (last_fill[s] >= 0) {
        drain_phase(bar(L::kBarQFull + s), (last_fill[s] / L::kStages) & 1, limit);
        drain_phase(bar(L::kBarDoFull + s), (last_fill[s] / L::kStages) & 1, limit);
      }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA warp (warp-uniform, elected issue)
    constexpr uint32_t kIdescS = make_idesc(kBlk, kBlk, false, kF16);   // S^T, dP^T: 128 x 128, K = HD
    constexpr uint32_t kIdescAcc = make_idesc(kBlk, HD, true, kF16);    // dV, dK: 128 x HD, K = 128 queries
    const uint64_t desc_k = sw128_desc(sbase + L::kOffK, 16, 1024);
    const uint64_t desc_v = sw128_desc(sbase + L::kOffV, 16, 1024);
    auto kmaj = [&](uint32_t off) { return sw128_desc(sbase + off, 16, 1024); };
    auto mnmaj = [&](uint32_t off) { return sw128_desc(sbase + off, T::kRegionBytes, 1024); };
    // X^T = A B^T with A (keys) and B (queries) both K-major over HD.
    auto issue_rows = [&](uint32_t d_col, uint64_t a, uint64_t b) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * T::kRegionBytes + (kk & 3) * 32) >> 4;
        ptx::mma_ss_warp(tmem + d_col, a + off, b + off, kIdescS, kk > 0 ? 1u : 0u);
      }
    };
    // acc (+)= X^T B, X^T (bf16) in TMEM columns a_col, B MN-major [128 queries x HD].
    auto issue_acc = [&](uint32_t d_col, uint32_t a_col, uint64_t b, bool accumulate) {
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk)   // X^T packed by the two warpgroups
        ptx::mma_ts_warp(tmem + d_col, tmem + a_col + packed_col(kk), b + ((kk * 16 * 128) >> 4),
                         kIdescAcc, (accumulate || kk > 0) ? 1u : 0u);
    };
    uint32_t it = 0, units = 0, acc_units = 0;
    bool ok = true;
    int idx;
    for (int r = 0; ok; ++r) {
      ok = unit_consume(bar(L::kBarUnitFull), bar(L::kBarUnitEmpty), unit_slots, r, idx, abort_flag,
                        limit, kSiteMma);
      if (!ok || idx >= p.n_units) break;
      int bh, kt;
      dkdv_unit(p, idx, bh, kt);
      int qa_unused, n;
      dkdv_range(p, kt, batch_keys(p, bh), &qa_unused, &n);
      ok = wait_warp(bar(L::kBarKvFull), units & 1, abort_flag, limit, kSiteMma);
      if (!ok) break;
      ++units;
      if (n == 0) {   // nothing reads K, V: release them
        ptx::mma_commit_warp(bar(L::kBarKvEmpty));
        continue;
      }
      ptx::tc_fence_after();
      {
        const int s0 = static_cast<int>(it % L::kStages);
        ok = wait_warp(bar(L::kBarQFull + s0), (it / L::kStages) & 1, abort_flag, limit, kSiteMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_rows(L::kColS, desc_k, kmaj(stage_off(s0)));
        ptx::mma_commit_warp(bar(L::kBarSFull));
        ok = wait_warp(bar(L::kBarDoFull + s0), (it / L::kStages) & 1, abort_flag, limit, kSiteMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_rows(L::kColDp, desc_v, kmaj(stage_off(s0) + T::kTileBytes));
        ptx::mma_commit_warp(bar(L::kBarDpFull));
      }
      for (int t = 0; t < n && ok; ++t, ++it) {
        const int s = static_cast<int>(it % L::kStages);
        const int s1 = static_cast<int>((it + 1) % L::kStages);
        if (t == 0 && acc_units > 0) {   // the previous unit's epilogue has read dV, dK
          ok = wait_warp(bar(L::kBarAccEmpty), (acc_units - 1) & 1, abort_flag, limit, kSiteMma);
          if (!ok) break;
        }
        ok = wait_warp(bar(L::kBarPFull), it & 1, abort_flag, limit, kSiteMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_acc(L::kColDv, L::kColS, mnmaj(stage_off(s) + T::kTileBytes), t > 0);   // dV += P^T dO
        if (t + 1 < n) {   // next S^T overwrites P^T: issued after the MMA that reads it
          // A tile that TMA landed in shared memory needs no tcgen05 fence after its wait
          // (that fence, which orders MMAs after TMEM hand-offs between threads, costs the
          // tensor pipe about 80 cycles)
          ok = wait_warp(bar(L::kBarQFull + s1), ((it + 1) / L::kStages) & 1, abort_flag, limit, kSiteMma);
          if (!ok) break;
          issue_rows(L::kColS, desc_k, kmaj(stage_off(s1)));
          ptx::mma_commit_warp(bar(L::kBarSFull));
        }
        ok = wait_warp(bar(L::kBarDsFull), it & 1, abort_flag, limit, kSiteMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_acc(L::kColDk, L::kColDp, mnmaj(stage_off(s)), t > 0);                   // dK += dS^T Q
        // Q, dO (and LSE, Delta) of stage s read.  Released by this commit, not by a compute
        // thread once dP^T(t + 1) is done (as the dQ kernel's rings are): with two stages the
        // later release leaves the next query tile unloaded when S^T(t + 2) is due.
        ptx::mma_commit_warp(bar(L::kBarQdEmpty + s));
        if (t + 1 < n) {
          ok = wait_warp(bar(L::kBarDoFull + s1), ((it + 1) / L::kStages) & 1, abort_flag, limit, kSiteMma);
          if (!ok) break;   // TMA data: no fence (above)
          issue_rows(L::kColDp, desc_v, kmaj(stage_off(s1) + T::kTileBytes));
          ptx::mma_commit_warp(bar(L::kBarDpFull));
        }
      }
      if (!ok) break;
      ptx::mma_commit_warp(bar(L::kBarAccFull));
      ptx::mma_commit_warp(bar(L::kBarKvEmpty));
      ++acc_units;
    }
    ptx::mma_commit_warp(bar(L::kBarDrain));
    drain_phase(bar(L::kBarDrain), 0, limit);
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ------------------------------------------------------------------ dQ
template <int HD>
struct DqLayout {
  using T = Tiles<HD>;
  // Separate K and V rings: K is read twice per key tile (S early, dQ last) and V once
  // (dP), so K gets the deeper ring and each V slot is freed as soon as its dP is done.
  static constexpr int kKStages = (HD == 128) ? 3 : 4;
  static constexpr int kVStages = (HD == 128) ? 2 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDo = T::kTileBytes;
  static constexpr int kOffK = 2 * T::kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * T::kTileBytes;
  static constexpr int kOffBar = kOffV + kVStages * T::kTileBytes;
  static constexpr int kBarQdFull = 0, kBarQdEmpty = 1;
  static constexpr int kBarKFull = 2;                           // [kKStages]
  static constexpr int kBarKEmpty = kBarKFull + kKStages;       // [kKStages]
  static constexpr int kBarVFull = kBarKEmpty + kKStages;       // [kVStages]
  static constexpr int kBarVEmpty = kBarVFull + kVStages;       // [kVStages]
  static constexpr int kBarSFull = kBarVEmpty + kVStages;
  static constexpr int kBarSFree = kBarSFull + 1;               // count 256 (compute threads)
  static constexpr int kBarDpFull = kBarSFree + 1;
  static constexpr int kBarDsFull = kBarDpFull + 1;             // count 256 (compute threads)
  static constexpr int kBarAccFull = kBarDsFull + 1;
  static constexpr int kBarAccEmpty = kBarAccFull + 1;          // count 256 (compute threads)
  static constexpr int kBarDrain = kBarAccEmpty + 1;
  static constexpr int kBarUnitFull = kBarDrain + 1;                // [kUnitRing]
  static constexpr int kBarUnitEmpty = kBarUnitFull + kUnitRing;    // [kUnitRing]
  static constexpr int kNumBars = kBarUnitEmpty + kUnitRing;
  static constexpr int kOffAbort = kOffBar + kNumBars * 8;
  static constexpr int kOffTmemSlot = kOffAbort + 4;
  static constexpr int kOffUnits = kOffTmemSlot + 4;                // int[kUnitRing]
  static constexpr int kBytes = kOffUnits + 4 * kUnitRing;
  static constexpr int kAlloc = kBytes + 1024;
  // TMEM columns: S | dP | dQ (dS as bf16 over the first 64 columns of dP)
  static constexpr uint32_t kColS = 0, kColDp = 128, kColDq = 256;
  static constexpr uint32_t kTmemCols = 512;
};
static_assert(DqLayout<128>::kAlloc <= 232448, "dQ shared memory (D=128)");
static_assert(DqLayout<64>::kAlloc <= 232448, "dQ shared memory (D=64)");

template <int HD, bool kF16>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using L = DqLayout<HD>;
  using T = Tiles<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_addr(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  volatile int* unit_slots = reinterpret_cast<volatile int*>(smem + L::kOffUnits);
  auto bar = [&](int idx) -> uint32_t { return sbase + L::kOffBar + 8u * idx; };
  auto k_off = [&](int s) -> uint32_t { return L::kOffK + s * T::kTileBytes; };
  auto v_off = [&](int s) -> uint32_t { return L::kOffV + s * T::kTileBytes; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(L::kBarQdFull), 1);
    ptx::mbar_init(bar(L::kBarQdEmpty), 1);
    for (int s = 0; s < L::kKStages; ++s) {
      ptx::mbar_init(bar(L::kBarKFull + s), 1);
      ptx::mbar_init(bar(L::kBarKEmpty + s), 1);
    }
    for (int s = 0; s < L::kVStages; ++s) {
      ptx::mbar_init(bar(L::kBarVFull + s), 1);
      ptx::mbar_init(bar(L::kBarVEmpty + s), 1);
    }
    ptx::mbar_init(bar(L::kBarSFull), 1);
    ptx::mbar_init(bar(L::kBarSFree), kComputeThreads);
    ptx::mbar_init(bar(L::kBarDpFull), 1);
    ptx::mbar_init(bar(L::kBarDsFull), kComputeThreads);
    ptx::mbar_init(bar(L::kBarAccFull), 1);
    ptx::mbar_init(bar(L::kBarAccEmpty), kComputeThreads);
    ptx::mbar_init(bar(L::kBarDrain), 1);
    for (int s = 0; s < kUnitRing; ++s) {
      ptx::mbar_init(bar(L::kBarUnitFull + s), 1);
      ptx::mbar_init(bar(L::kBarUnitEmpty + s), kUnitConsumers);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), L::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const unsigned long long limit = p.wait_limit_ns;
  // Always launched as a programmatic dependent of the dK/dV kernel.  What dQ reads (the
  // inputs, Delta, LSE * log2 e, its unit counter) was complete before that kernel let
  // this one launch: the dK/dV kernel allows it only after its own wait for the Delta
  // kernel.  So this kernel starts on the SMs that the dK/dV kernel's last units leave
  // free, and waits for the dK/dV kernel only before it exits, so that its completion
  // still implies both (the next call may read dK or dV).
  ptx::grid_launch_dependents();

  if (warp < 8) {
    // ------------------------------------------------ compute warpgroups: thread = query row
    const int g = warp >> 2;                   // columns [64g, 64g + 64) of the row
    const int rw = warp & 3;
    const int row = rw * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(rw * 32) << 16;
    const uint32_t t_s = tmem + lane_off + L::kColS + 64 * g;
    const uint32_t t_dp = tmem + lane_off + L::kColDp + 64 * g;
    const float sl2 = p.scale_log2;
    uint32_t it = 0, acc_count = 0;
    bool ok = true;
    int idx;
    for (int r = 0; ok; ++r) {
      ok = unit_consume(bar(L::kBarUnitFull), bar(L::kBarUnitEmpty), unit_slots, r, idx, abort_flag,
                        limit, kSiteCompute);
      if (!ok || idx >= p.n_units) break;
      int bh, qt;
      dq_unit(p, idx, bh, qt);
      const int kvl = batch_keys(p, bh);
      int ka, n;
      dq_range(p, qt, kvl, &ka, &n);
      const int q = qt * kBlk + row;   // this thread's query
      const bool valid = q < p.Lq;
      const size_t gp = (static_cast<size_t>(bh) * p.nq + qt) * kBlk + row;   // padded row
      const float lse2 = valid ? p.lse2[gp] : 0.0f;
      const float dlt = p.delta[gp];
      // keys allowed for this row: key_lo <= k < key_lim (a row without keys gets dQ = 0)
      auto lo_of = [&](int qq) { return p.win_left < 0 ? 0 : qq - p.win_left; };
      auto lim_of = [&](int qq) {
        return p.win_right < 0 ? kvl
                               : static_cast<int>(min(static_cast<long long>(kvl),
                                                      static_cast<long long>(qq) + p.win_right + 1));
      };
      const int key_lo = lo_of(q), key_lim = lim_of(q);
      // a key tile needs masking only where the band's left edge (of the tile's last row)
      // or its right edge and the padding (of its first row) cut it; rows without keys
      // always lie in such tiles
      const int lo_last = lo_of(qt * kBlk + kBlk - 1), lim_first = lim_of(qt * kBlk);
      if (n == 0) {   // no query of the tile has a key: dQ = 0, no MMA
        if (valid)
          for (int c = 0; c < HD / 2; c += 8)
            *reinterpret_cast<uint4*>(p.dq + row_offset(p.dq_s, p.H, bh, q) + (HD / 2) * g + c) =
                make_uint4(0, 0, 0, 0);
        continue;
      }
      for (int t = 0; t < n; ++t, ++it) {
        ok = __all_sync(0xffffffffu, wait_phase(bar(L::kBarSFull), it & 1, abort_flag, limit, kSiteCompute));
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[64];
        ptx::tmem_ld32x32b_x64(t_s, sr);   // one load, one wait for the warpgroup's 64 columns
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarSFree));   // S is in registers: the next S may overwrite it
        const int kb = (ka + t) * kBlk;
        const bool cut = kb < lo_last || kb + kBlk > lim_first;
        const int base = kb + 64 * g;   // key of this warpgroup's column 0
        const int lo_c = key_lo - base, lim_c = key_lim - base;   // columns lo_c <= c < lim_c are allowed
        float pr[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) pr[c] = ptx::ex2_approx(fmaf(__uint_as_float(sr[c]), sl2, -lse2));
        if (cut) {
#pragma unroll
          for (int c = 0; c < 64; ++c) pr[c] = (c >= lo_c && c < lim_c) ? pr[c] : 0.0f;
        }
        ok = __all_sync(0xffffffffu, wait_phase(bar(L::kBarDpFull), it & 1, abort_flag, limit, kSiteCompute));
        if (!ok) break;
        ptx::tc_fence_after();
        ptx::tmem_ld32x32b_x64(t_dp, sr);
        // Ring slots are released here rather than by MMA commits (each commit costs the
        // tensor pipe about 90 cycles): dP(t) was V(t)'s only reader, and dP(t) was issued
        // after dQ(t - 1), K(t - 1)'s last reader.
        if (threadIdx.x == 0) {
          ptx::mbar_arrive(bar(L::kBarVEmpty + static_cast<int>(it % L::kVStages)));
          if (t > 0) ptx::mbar_arrive(bar(L::kBarKEmpty + static_cast<int>((it - 1) % L::kKStages)));
        }
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c)
          pk[c] = pack2<kF16>(pr[2 * c] * (__uint_as_float(sr[2 * c]) - dlt),
                              pr[2 * c + 1] * (__uint_as_float(sr[2 * c + 1]) - dlt));
        ptx::tmem_st32x32b_x32(t_dp, pk);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarDsFull));
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, wait_phase(bar(L::kBarAccFull), acc_count & 1, abort_flag, limit, kSiteEpilogue));
      if (!ok) break;
      ++acc_count;
      ptx::tc_fence_after();
      // every MMA of the unit is complete: the K slot of its last key tile is free
      if (threadIdx.x == 0) ptx::mbar_arrive(bar(L::kBarKEmpty + static_cast<int>((it - 1) % L::kKStages)));
      // Epilogue: each warpgroup writes its half of the row's columns.
      uint16_t* dst = p.dq + row_offset(p.dq_s, p.H, bh, valid ? q : 0) + (HD / 2) * g;
      // This warpgroup's half of the row first, released at once, then stored.
      uint32_t a[HD / 64][32];
#pragma unroll
      for (int k2 = 0; k2 < HD / 64; ++k2)
        ptx::tmem_ld32x32b_x32(tmem + lane_off + L::kColDq + (HD / 2) * g + 32 * k2, a[k2]);
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::kBarAccEmpty));
#pragma unroll
      for (int k2 = 0; k2 < HD / 64; ++k2) {
        uint32_t pk16[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk16[c] = pack2<kF16>(__uint_as_float(a[k2][2 * c]) * p.scale, __uint_as_float(a[k2][2 * c + 1]) * p.scale);
        if (valid) {
          if (p.dq_v8) {
            ptx::st_global_v8(dst + 32 * k2, pk16);
            ptx::st_global_v8(dst + 32 * k2 + 16, pk16 + 8);
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              reinterpret_cast<uint4*>(dst + 32 * k2)[v] = make_uint4(pk16[4 * v], pk16[4 * v + 1], pk16[4 * v + 2], pk16[4 * v + 3]);
          }
        }
      }
    }
  } else if (warp == kLoadWarp) {
    // ------------------------------------------------ load warp
    if (lane == 0) {
      ptx::prefetch_tensormap(&p.tm_q);
      ptx::prefetch_tensormap(&p.tm_k);
      ptx::prefetch_tensormap(&p.tm_v);
      ptx::prefetch_tensormap(&p.tm_do);
    }
    uint32_t it = 0, units = 0;
    int last_k[L::kKStages], last_v[L::kVStages];
    for (int s = 0; s < L::kKStages; ++s) last_k[s] = -1;
    for (int s = 0; s < L::kVStages; ++s) last_v[s] = -1;
    bool ok = true;
    int idx;
    for (int r = 0; ok; ++r) {
      ok = unit_produce(p, bar(L::kBarUnitFull), bar(L::kBarUnitEmpty), unit_slots, r, idx, abort_flag,
                        limit, kSiteLoad);
      if (!ok || idx >= p.n_units) break;
      int bh, qt;
      dq_unit(p, idx, bh, qt);
      int ka, n;
      dq_range(p, qt, batch_keys(p, bh), &ka, &n);
      if (n == 0) continue;   // no keys: nothing to load
      if (units > 0) {
        ok = wait_warp(bar(L::kBarQdEmpty), (units - 1) & 1, abort_flag, limit, kSiteLoad);
        if (!ok) break;
      }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar(L::kBarQdFull), 2 * T::kTileBytes);
        for (int rg = 0; rg < T::kRegions; ++rg) {
          ptx::tma_load_4d(sbase + L::kOffQ + rg * T::kRegionBytes, &p.tm_q, bar(L::kBarQdFull), 64 * rg, qt * kBlk, bh - (bh / p.H) * p.H, bh / p.H);
          ptx::tma_load_4d(sbase + L::kOffDo + rg * T::kRegionBytes, &p.tm_do, bar(L::kBarQdFull), 64 * rg, qt * kBlk, bh - (bh / p.H) * p.H, bh / p.H);
        }
      }
      ++units;
      for (int t = 0; t < n; ++t, ++it) {
        const int sk = static_cast<int>(it % L::kKStages), sv = static_cast<int>(it % L::kVStages);
        ok = wait_warp(bar(L::kBarKEmpty + sk), ((it / L::kKStages) & 1) ^ 1u, abort_flag, limit, kSiteLoad);
        if (!ok) break;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(bar(L::kBarKFull + sk), T::kTileBytes);
          for (int rg = 0; rg < T::kRegions; ++rg)
            ptx::tma_load_4d(sbase + k_off(sk) + rg * T::kRegionBytes, &p.tm_k, bar(L::kBarKFull + sk), 64 * rg, (ka + t) * kBlk, bh - (bh / p.H) * p.H, bh / p.H);
        }
        last_k[sk] = static_cast<int>(it);
        ok = wait_warp(bar(L::kBarVEmpty + sv), ((it / L::kVStages) & 1) ^ 1u, abort_flag, limit, kSiteLoad);
        if (!ok) break;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(bar(L::kBarVFull + sv), T::kTileBytes);
          for (int rg = 0; rg < T::kRegions; ++rg)
            ptx::tma_load_4d(sbase + v_off(sv) + rg * T::kRegionBytes, &p.tm_v, bar(L::kBarVFull + sv), 64 * rg, (ka + t) * kBlk, bh - (bh / p.H) * p.H, bh / p.H);
        }
        last_v[sv] = static_cast<int>(it);
      }
    }
    if (lane == 0) {
      if (units > 0) drain_phase(bar(L::kBarQdFull), (units - 1) & 1, limit);
      for (int s = 0; s < L::kKStages; ++s)
        if (last_k[s] >= 0) drain_phase(bar(L::kBarKFull + s), (last_k[s] / L::kKStages) & 1, limit);
      for (int s = 0; s < L::kVStages; ++s)
        if (last_v[s] >= 0) drain_phase(bar(L::kBarVFull + s), (last_v[s] / L::kVStages) & 1, limit);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA warp (warp-uniform, elected issue)
    constexpr uint32_t kIdescS = make_idesc(kBlk, kBlk, false, kF16);
    constexpr uint32_t kIdescAcc = make_idesc(kBlk, HD, true, kF16);
    const uint64_t desc_q = sw128_desc(sbase + L::kOffQ, 16, 1024);
    const uint64_t desc_do = sw128_desc(sbase + L::kOffDo, 16, 1024);
    auto kmaj = [&](uint32_t off) { return sw128_desc(sbase + off, 16, 1024); };
    auto mnmaj = [&](uint32_t off) { return sw128_desc(sbase + off, T::kRegionBytes, 1024); };
    auto issue_rows = [&](uint32_t d_col, uint64_t a, uint64_t b) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * T::kRegionBytes + (kk & 3) * 32) >> 4;
        ptx::mma_ss_warp(tmem + d_col, a + off, b + off, kIdescS, kk > 0 ? 1u : 0u);
      }
    };
    auto issue_acc = [&](uint64_t b, bool accumulate) {   // dQ (+)= dS K, dS packed by both warpgroups
#pragma unroll
      for (int kk = 0; kk < kBlk / 16; ++kk)
        ptx::mma_ts_warp(tmem + L::kColDq, tmem + L::kColDp + packed_col(kk), b + ((kk * 16 * 128) >> 4),
                         kIdescAcc, (accumulate || kk > 0) ? 1u : 0u);
    };
    uint32_t it = 0, units = 0, acc_units = 0;
    bool ok = true;
    int idx;
    for (int r = 0; ok; ++r) {
      ok = unit_consume(bar(L::kBarUnitFull), bar(L::kBarUnitEmpty), unit_slots, r, idx, abort_flag,
                        limit, kSiteMma);
      if (!ok || idx >= p.n_units) break;
      int bh, qt;
      dq_unit(p, idx, bh, qt);
      int ka_unused, n;
      dq_range(p, qt, batch_keys(p, bh), &ka_unused, &n);
      if (n == 0) continue;   // no keys: nothing to issue
      ok = wait_warp(bar(L::kBarQdFull), units & 1, abort_flag, limit, kSiteMma);
      if (!ok) break;
      ++units;
      {
        const int k0 = static_cast<int>(it % L::kKStages), v0 = static_cast<int>(it % L::kVStages);
        ok = wait_warp(bar(L::kBarKFull + k0), (it / L::kKStages) & 1, abort_flag, limit, kSiteMma);
        if (ok) ok = wait_warp(bar(L::kBarVFull + v0), (it / L::kVStages) & 1, abort_flag, limit, kSiteMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_rows(L::kColS, desc_q, kmaj(k_off(k0)));
        ptx::mma_commit_warp(bar(L::kBarSFull));
        issue_rows(L::kColDp, desc_do, kmaj(v_off(v0)));
        ptx::mma_commit_warp(bar(L::kBarDpFull));
      }
      for (int t = 0; t < n && ok; ++t, ++it) {
        const int sk = static_cast<int>(it % L::kKStages);
        const int k1 = static_cast<int>((it + 1) % L::kKStages), v1 = static_cast<int>((it + 1) % L::kVStages);
        if (t + 1 < n) {   // next S as soon as this S has left TMEM
          ok = wait_warp(bar(L::kBarSFree), it & 1, abort_flag, limit, kSiteMma);
          if (ok) ok = wait_warp(bar(L::kBarKFull + k1), ((it + 1) / L::kKStages) & 1, abort_flag, limit, kSiteMma);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_rows(L::kColS, desc_q, kmaj(k_off(k1)));
          ptx::mma_commit_warp(bar(L::kBarSFull));
        }
        if (t == 0 && acc_units > 0) {
          ok = wait_warp(bar(L::kBarAccEmpty), (acc_units - 1) & 1, abort_flag, limit, kSiteMma);
          if (!ok) break;
        }
        ok = wait_warp(bar(L::kBarDsFull), it & 1, abort_flag, limit, kSiteMma);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_acc(mnmaj(k_off(sk)), t > 0);
        if (t + 1 < n) {   // next dP overwrites dS: issued after the MMA that reads it
          // V landed by TMA: no tcgen05 fence after its wait (the fence orders MMAs after
          // TMEM hand-offs between threads and costs the tensor pipe about 80 cycles)
          ok = wait_warp(bar(L::kBarVFull + v1), ((it + 1) / L::kVStages) & 1, abort_flag, limit, kSiteMma);
          if (!ok) break;
          issue_rows(L::kColDp, desc_do, kmaj(v_off(v1)));
          ptx::mma_commit_warp(bar(L::kBarDpFull));
        }
      }
      if (!ok) break;
      ptx::mma_commit_warp(bar(L::kBarAccFull));
      ptx::mma_commit_warp(bar(L::kBarQdEmpty));
      ++acc_units;
    }
    ptx::mma_commit_warp(bar(L::kBarDrain));
    drain_phase(bar(L::kBarDrain), 0, limit);
    __syncwarp();
  }

  ptx::grid_dependency_wait();   // the dK/dV kernel ahead has completed
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::kTmemCols);
  }
}

// Zero the rows of a strided [B,H,L,D] tensor (the key gradients when there is no query).
__global__ void __launch_bounds__(256) fa_bwd_zero_kernel(uint16_t* base, long long s0, long long s1,
                                                          long long s2, int H, int L, long long rows,
                                                          int D) {
  const int per = D / 8;   // 16-byte chunks per row
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < rows * per;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / per;
    const int c = static_cast<int>(i - r * per) * 8;
    const long long bh = r / L, l = r - bh * L;
    const long long b = bh / H, h = bh - b * H;
    *reinterpret_cast<uint4*>(base + b * s0 + h * s1 + l * s2 + c) = make_uint4(0, 0, 0, 0);
  }
}

}  // namespace fab

// ============================================================================ host side
namespace {

using fab::BwdParams;

std::mutex g_bwd_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_bwd_encode = nullptr;
bool g_bwd_ready[64][2][2] = {};   // [device][D == 128][fp16]: shared-memory opt-in done

// Problems with fewer key tiles than SMs run the dQ kernel on a second stream beside the
// dK/dV kernel (see the launch sequence below): one stream and two events per device,
// owned by the library and created at first use.  An event's record and the wait that
// reads it are made together under `mu`, so concurrent callers cannot interleave them.
struct BwdFork {
  cudaStream_t aux = nullptr;
  cudaEvent_t fork = nullptr;   // recorded on the caller's stream after the Delta kernel
  cudaEvent_t join = nullptr;   // recorded on `aux` after the dQ kernel
  std::mutex mu;
};
BwdFork g_bwd_fork[64];

// The device's fork state, created on first use; nullptr if it cannot be created.
BwdFork* bwd_fork(int dev) {
  if (dev < 0 || dev >= 64) return nullptr;
  BwdFork& f = g_bwd_fork[dev];
  std::lock_guard<std::mutex> lock(f.mu);
  if (!f.aux) {
    cudaStream_t aux = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaStreamCreateWithFlags(&aux, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&e0, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&e1, cudaEventDisableTiming) != cudaSuccess) {
      if (e0) cudaEventDestroy(e0);
      cudaStreamDestroy(aux);
      return nullptr;
    }
    f.fork = e0;
    f.join = e1;
    f.aux = aux;
  }
  return &f;
}

using BwdKernel = void (*)(const BwdParams);
BwdKernel dkdv_kernel(int D, bool f16) {
  if (D == 128) return f16 ? fab::fa_bwd_dkdv_kernel<128, true> : fab::fa_bwd_dkdv_kernel<128, false>;
  return f16 ? fab::fa_bwd_dkdv_kernel<64, true> : fab::fa_bwd_dkdv_kernel<64, false>;
}
BwdKernel dq_kernel(int D, bool f16) {
  if (D == 128) return f16 ? fab::fa_bwd_dq_kernel<128, true> : fab::fa_bwd_dq_kernel<128, false>;
  return f16 ? fab::fa_bwd_dq_kernel<64, true> : fab::fa_bwd_dq_kernel<64, false>;
}
using DeltaKernel = void (*)(const fab::DeltaArgs);
DeltaKernel delta_kernel(int D, bool f16) {
  if (D == 128) return f16 ? fab::fa_bwd_delta_kernel<128, true> : fab::fa_bwd_delta_kernel<128, false>;
  return f16 ? fab::fa_bwd_delta_kernel<64, true> : fab::fa_bwd_delta_kernel<64, false>;
}

// Element strides {batch, head, row} of every tensor of one backward call.
struct BwdStrides {
  long long q[3], k[3], v[3], o[3], dO[3], dq[3], dk[3], dv[3];
};

void contiguous3(long long H, long long L, int D, long long* st) {
  st[2] = D;
  st[1] = L * D;
  st[0] = H * L * D;
}

BwdStrides contiguous_bwd(int H, int Lq, int Lk, int D) {
  BwdStrides sd;
  contiguous3(H, Lq, D, sd.q);
  contiguous3(H, Lk, D, sd.k);
  contiguous3(H, Lk, D, sd.v);
  contiguous3(H, Lq, D, sd.o);
  contiguous3(H, Lq, D, sd.dO);
  contiguous3(H, Lq, D, sd.dq);
  contiguous3(H, Lk, D, sd.dk);
  contiguous3(H, Lk, D, sd.dv);
  return sd;
}

bool bwd_overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return na && nb && pa < pb + nb && pb < pa + na;
}

size_t bwd_round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
constexpr size_t kBwdCounterBytes = 256;   // the kernels' two unit counters

// Heads per unit group: as many as keep a group's streamed tensors (bytes_per_head each)
// within 32 MiB of L2, at least one.
int bwd_group_heads(long long bytes_per_head, long long bh) {
  const long long g = (32ll << 20) / std::max(1ll, bytes_per_head);
  return static_cast<int>(std::max(1ll, std::min(g, bh)));
}

fa_status bwd_prepare(int D, bool f16, int* sm_count) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  // Make the device's primary context current on this thread: a thread that has only
  // selected the device (a worker thread, autograd's backward thread) has none yet, and
  // tensor-map encoding needs one.
  if (cudaSetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_bwd_mutex);
  if (!g_bwd_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return FA_ERR_CUDA;
    g_bwd_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const int di = (D == 128) ? 1 : 0, ti = f16 ? 1 : 0;
  if (!g_bwd_ready[dev][di][ti]) {
    const int dkdv_smem = D == 128 ? fab::DkdvLayout<128>::kAlloc : fab::DkdvLayout<64>::kAlloc;
    const int dq_smem = D == 128 ? fab::DqLayout<128>::kAlloc : fab::DqLayout<64>::kAlloc;
    if (cudaFuncSetAttribute(dkdv_kernel(D, f16), cudaFuncAttributeMaxDynamicSharedMemorySize, dkdv_smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(dq_kernel(D, f16), cudaFuncAttributeMaxDynamicSharedMemorySize, dq_smem) !=
            cudaSuccess)
      return FA_ERR_CUDA;
    g_bwd_ready[dev][di][ti] = true;
  }
  return FA_OK;
}

// 4-D tensor map [B][H][L][D] over element strides st = {batch, head, row} (as the forward's;
// a size-1 dimension's stride addresses nothing and is replaced by a valid one).
bool bwd_encode_map(CUtensorMap* map, const void* base, long long B, long long H, long long L, int D,
                    const long long* st, bool f16) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  const long long row = L > 1 ? st[2] : D;
  const long long head = H > 1 ? st[1] : row * L;
  const long long batch = B > 1 ? st[0] : head * H;
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(row) * 2, static_cast<cuuint64_t>(head) * 2,
                           static_cast<cuuint64_t>(batch) * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estrides[4] = {1, 1, 1, 1};
  return g_bwd_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                      const_cast<void*>(base), dims, strides, box, estrides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Size checks shared by fa_bwd and fa_bwd_workspace_size; *rows = B*H*Lq.
fa_status bwd_check_sizes(int B, int H, int Lq, int Lk, int D, long long* rows, long long* bh) {
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (Lq > INT_MAX - 128) return FA_ERR_INVALID_ARG;   // rows are padded to whole 128-row tiles
  *bh = static_cast<long long>(B) * H;
  *rows = *bh * Lq;
  if (*rows == 0) return FA_OK;
  if (Lk < 1) return FA_ERR_INVALID_ARG;
  if (*rows * D > (1ll << 40) || *bh * Lk * D > (1ll << 40)) return FA_ERR_INVALID_ARG;
  const long long nq = (Lq + 127) / 128, nk = (Lk + 127) / 128;
  if (*bh > INT_MAX || *bh * nq > INT_MAX || *bh * nk > INT_MAX) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

}  // namespace

unsigned fa_bwd_take_device_status() {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, fab::g_bwd_status, sizeof(v)) != cudaSuccess) return FA_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(fab::g_bwd_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return v;
}

extern "C" fa_status fa_bwd_workspace_size(int B, int H, int Lq, int Lk, int D, int causal, size_t* bytes) {
  (void)causal;
  if (!bytes) return FA_ERR_INVALID_ARG;
  *bytes = 0;
  long long rows = 0, bh = 0;
  const fa_status st = bwd_check_sizes(B, H, Lq, Lk, D, &rows, &bh);
  if (st != FA_OK) return st;
  const size_t rows_pad = static_cast<size_t>(bh) * ((Lq + 127) / 128) * 128;
  *bytes = 2 * bwd_round256(rows_pad * sizeof(float)) + kBwdCounterBytes;
  return FA_OK;
}

namespace {
fa_status bwd_impl(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                   const float* LSE, void* dQ, void* dK, void* dV, const int* kv_len, int B, int H,
                   int Lq, int Lk, int D, int window_left, int window_right, float scale, bool f16,
                   const BwdStrides& sd, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  using fa_layout::no_self_overlap;
  using fa_layout::span_bytes;
  using fa_layout::strides_ok;
  long long rows = 0, bh = 0;
  fa_status st = bwd_check_sizes(B, H, Lq, Lk, D, &rows, &bh);
  if (st != FA_OK) return st;
  if (bh * Lk == 0) return FA_OK;
  if (rows == 0) {   // no query rows: every key gradient is zero
    if (!dK || !dV || (reinterpret_cast<uintptr_t>(dK) | reinterpret_cast<uintptr_t>(dV)) & 15u)
      return FA_ERR_INVALID_ARG;
    if (!strides_ok(B, H, Lk, D, sd.dk) || !strides_ok(B, H, Lk, D, sd.dv) ||
        !no_self_overlap(B, H, Lk, D, sd.dk) || !no_self_overlap(B, H, Lk, D, sd.dv))
      return FA_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;
    const long long krows = bh * Lk;
    const unsigned blocks = static_cast<unsigned>(std::min<long long>((krows * (D / 8) + 255) / 256, 65535));
    for (int which = 0; which < 2; ++which) {
      const long long* s3 = which ? sd.dv : sd.dk;
      cudaLaunchConfig_t zc = {};
      zc.gridDim = dim3(blocks);
      zc.blockDim = dim3(256);
      zc.stream = stream;
      if (cudaLaunchKernelEx(&zc, fab::fa_bwd_zero_kernel, static_cast<uint16_t*>(which ? dV : dK), s3[0],
                             s3[1], s3[2], H, Lk, krows, D) != cudaSuccess)
        return FA_ERR_CUDA;
    }
    return FA_OK;
  }
  if (!(scale > 0.0f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  const void* in[6] = {Q, K, V, O, dO, LSE};
  void* out[3] = {dQ, dK, dV};
  uintptr_t bits = reinterpret_cast<uintptr_t>(workspace);
  for (const void* x : in) {
    if (!x) return FA_ERR_INVALID_ARG;
    bits |= reinterpret_cast<uintptr_t>(x);
  }
  for (void* x : out) {
    if (!x) return FA_ERR_INVALID_ARG;
    bits |= reinterpret_cast<uintptr_t>(x);
  }
  if (bits & 15u) return FA_ERR_INVALID_ARG;
  if (!strides_ok(B, H, Lq, D, sd.q) || !strides_ok(B, H, Lk, D, sd.k) || !strides_ok(B, H, Lk, D, sd.v) ||
      !strides_ok(B, H, Lq, D, sd.o) || !strides_ok(B, H, Lq, D, sd.dO) || !strides_ok(B, H, Lq, D, sd.dq) ||
      !strides_ok(B, H, Lk, D, sd.dk) || !strides_ok(B, H, Lk, D, sd.dv) ||
      !no_self_overlap(B, H, Lq, D, sd.dq) || !no_self_overlap(B, H, Lk, D, sd.dk) ||
      !no_self_overlap(B, H, Lk, D, sd.dv))
    return FA_ERR_INVALID_ARG;
  const size_t bytes_l = static_cast<size_t>(rows) * 4;
  const long long nq_ll = (Lq + 127) / 128;
  const size_t rows_pad = static_cast<size_t>(bh) * nq_ll * 128;
  const size_t half_ws = bwd_round256(rows_pad * sizeof(float));
  const size_t need_ws = 2 * half_ws + kBwdCounterBytes;
  if (!workspace || workspace_bytes < need_ws || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FA_ERR_INVALID_ARG;
  // Inputs may share memory (they are only read); outputs and the workspace meet nothing.
  const size_t in_bytes[6] = {span_bytes(B, H, Lq, D, sd.q), span_bytes(B, H, Lk, D, sd.k),
                              span_bytes(B, H, Lk, D, sd.v), span_bytes(B, H, Lq, D, sd.o),
                              span_bytes(B, H, Lq, D, sd.dO), bytes_l};
  const size_t out_bytes[4] = {span_bytes(B, H, Lq, D, sd.dq), span_bytes(B, H, Lk, D, sd.dk),
                               span_bytes(B, H, Lk, D, sd.dv), need_ws};
  void* outs[4] = {dQ, dK, dV, workspace};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (bwd_overlaps(outs[a], out_bytes[a], in[b], in_bytes[b])) return FA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (bwd_overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b])) return FA_ERR_INVALID_ARG;
  }
  int sm_count = 0;
  st = bwd_prepare(D, f16, &sm_count);
  if (st != FA_OK) return st;

  BwdParams p;
  if (!bwd_encode_map(&p.tm_q, Q, B, H, Lq, D, sd.q, f16) || !bwd_encode_map(&p.tm_k, K, B, H, Lk, D, sd.k, f16) ||
      !bwd_encode_map(&p.tm_v, V, B, H, Lk, D, sd.v, f16) || !bwd_encode_map(&p.tm_do, dO, B, H, Lq, D, sd.dO, f16))
    return FA_ERR_CUDA;
  float* delta = static_cast<float*>(workspace);
  float* lse2 = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + half_ws);
  int* unit_ctr = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + 2 * half_ws);
  p.delta = delta;
  p.lse2 = lse2;
  p.dq = static_cast<uint16_t*>(dQ);
  p.dk = static_cast<uint16_t*>(dK);
  p.dv = static_cast<uint16_t*>(dV);
  auto v8_ok = [](const void* base, const long long* st) {
    return reinterpret_cast<uintptr_t>(base) % 32 == 0 && (st[0] * 2) % 32 == 0 &&
           (st[1] * 2) % 32 == 0 && (st[2] * 2) % 32 == 0;
  };
  p.dq_v8 = v8_ok(dQ, sd.dq) ? 1 : 0;
  p.dkv_v8 = (v8_ok(dK, sd.dk) && v8_ok(dV, sd.dv)) ? 1 : 0;
  for (int i = 0; i < 3; ++i) {
    p.dq_s[i] = sd.dq[i];
    p.dk_s[i] = sd.dk[i];
    p.dv_s[i] = sd.dv[i];
  }
  p.bh_count = static_cast<int>(bh);
  p.Lq = Lq;
  p.Lk = Lk;
  p.H = H;
  p.win_left = window_left >= Lq - 1 ? -1 : window_left;   // a side covering every key is unbounded
  p.win_right = window_right >= Lk - 1 ? -1 : window_right;
  p.kv_len = kv_len;
  p.nq = (Lq + 127) / 128;
  p.nk = (Lk + 127) / 128;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  const unsigned long long lim = fa_internal_wait_limit_ns();
  p.wait_limit_ns = lim ? lim : fab::kDefaultWaitNs;
  p.flags = fa_internal_debug_flags();
  if (p.flags & 2u) return FA_ERR_CUDA;   // test hook: simulated launch failure

  // Short problems launch the Delta and dK/dV kernels as programmatic dependents: each
  // one's set-up (barriers, TMEM) overlaps the kernel ahead of it, which it waits for
  // before touching memory.  Long ones launch them plainly (the forward measured bimodal
  // times with dependent launches of long kernels).  Work per CTA: the query-key tile
  // pairs of the problem.  The dQ kernel, which does not read what dK/dV writes, is a
  // dependent of the dK/dV kernel and fills the SMs its last units leave.  With fewer key
  // tiles than SMs, the dK/dV grid leaves SMs idle from the start and its units end at
  // very different times.  A dependent grid that fits beside it starts at once, but one
  // that does not was measured to take none of the SMs the dK/dV units free early (one
  // causal head of 16K tokens: 323 us, against 320 us launched plainly after dK/dV).
  // Those problems fork instead: the dQ kernel goes to a second stream that waits for the
  // Delta kernel only, and the caller's stream waits for it at the end (189 us; two heads
  // of 8K 180 -> 105 us).  Where both grids fit at once the fork only adds its events
  // (one head of 8K or 4K: 2-7 % slower), so it is not taken there.
  const long long pairs_per_cta = bh * static_cast<long long>(p.nq) * p.nk / std::max(1, sm_count);
  const bool dependent = pairs_per_cta <= 256;
  const long long grid_kv = bh * static_cast<long long>(p.nk);
  const long long grid_q = std::min<long long>(bh * static_cast<long long>(p.nq), sm_count);
  BwdFork* fk = nullptr;
  if (grid_kv < sm_count && grid_kv + grid_q > sm_count) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || !(fk = bwd_fork(dev))) return FA_ERR_CUDA;
  }
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;

  // 1. Delta = rowsum(dO * O) and LSE * log2(e), padded to whole tiles.  Launch errors
  // come from the launch call itself (not cudaGetLastError, which would also report an
  // earlier error of the calling thread).
  {
    fab::DeltaArgs da;
    da.O = static_cast<const uint16_t*>(O);
    da.dO = static_cast<const uint16_t*>(dO);
    da.lse = LSE;
    da.delta = delta;
    da.lse2 = lse2;
    for (int i = 0; i < 3; ++i) {
      da.o_s[i] = sd.o[i];
      da.do_s[i] = sd.dO[i];
    }
    da.rows_pad = static_cast<long long>(rows_pad);
    da.unit_ctr = unit_ctr;
    da.Lq = Lq;
    da.Lpad = static_cast<int>(nq_ll * 128);
    da.H = H;
    const long long threads = static_cast<long long>(rows_pad) * (D / 8);
    cudaLaunchConfig_t dc = {};
    dc.gridDim = dim3(static_cast<unsigned>((threads + 255) / 256));
    dc.blockDim = dim3(256);
    dc.stream = stream;
    dc.attrs = pdl;
    dc.numAttrs = dependent ? 1 : 0;
    if (cudaLaunchKernelEx(&dc, delta_kernel(D, f16), da) != cudaSuccess) return FA_ERR_CUDA;
  }
  if (fk) {   // the dQ kernel's stream starts after the Delta kernel
    std::lock_guard<std::mutex> lock(fk->mu);
    if (cudaEventRecord(fk->fork, stream) != cudaSuccess ||
        cudaStreamWaitEvent(fk->aux, fk->fork, 0) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  // 2. dK, dV (one unit per key tile) and 3. dQ (one unit per query tile)
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(fab::kThreads);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = (dependent && !fk) ? 1 : 0;   // an event record now separates it from Delta
  p.n_units = static_cast<int>(bh * p.nk);
  p.unit_ctr = unit_ctr;
  p.group_heads = bwd_group_heads(4ll * Lq * D, bh);   // dK/dV streams Q and dO
  cfg.gridDim = dim3(static_cast<unsigned>(std::min(p.n_units, sm_count)));
  cfg.dynamicSmemBytes = (D == 128) ? fab::DkdvLayout<128>::kAlloc : fab::DkdvLayout<64>::kAlloc;
  if (cudaLaunchKernelEx(&cfg, dkdv_kernel(D, f16), p) != cudaSuccess) return FA_ERR_CUDA;
  p.n_units = static_cast<int>(bh * p.nq);
  p.unit_ctr = unit_ctr + fab::kCtrStride;
  p.group_heads = bwd_group_heads(4ll * Lk * D, bh);   // dQ streams K and V
  cfg.gridDim = dim3(static_cast<unsigned>(std::min(p.n_units, sm_count)));
  cfg.dynamicSmemBytes = (D == 128) ? fab::DqLayout<128>::kAlloc : fab::DqLayout<64>::kAlloc;
  if (fk) {
    cfg.stream = fk->aux;
    cfg.numAttrs = 0;
  } else {
    cfg.numAttrs = 1;   // dependent launch, whatever the problem's length
  }
  if (cudaLaunchKernelEx(&cfg, dq_kernel(D, f16), p) != cudaSuccess) return FA_ERR_CUDA;
  if (fk) {   // the caller's stream continues once dQ is done
    std::lock_guard<std::mutex> lock(fk->mu);
    if (cudaEventRecord(fk->join, fk->aux) != cudaSuccess ||
        cudaStreamWaitEvent(stream, fk->join, 0) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  return FA_OK;
}
}  // namespace

extern "C" fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                            const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Lq, int Lk,
                            int D, int causal, float scale, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, nullptr, B, H, Lq, Lk, D, -1, causal ? 0 : -1, scale,
                  false, contiguous_bwd(H, Lq, Lk, D), workspace, workspace_bytes, stream);
}

extern "C" fa_status fa_bwd_masked(const void* Q, const void* K, const void* V, const void* O,
                                   const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                                   const int* kv_len, int B, int H, int Lq, int Lk, int D,
                                   int window_left, int window_right, float scale, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream) {
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, kv_len, B, H, Lq, Lk, D, window_left, window_right,
                  scale, false, contiguous_bwd(H, Lq, Lk, D), workspace, workspace_bytes, stream);
}

extern "C" fa_status fa_bwd_strided(const void* Q, const long long* q_stride, const void* K,
                                    const long long* k_stride, const void* V, const long long* v_stride,
                                    const void* O, const long long* o_stride, const void* dO,
                                    const long long* do_stride, const float* LSE, void* dQ,
                                    const long long* dq_stride, void* dK, const long long* dk_stride,
                                    void* dV, const long long* dv_stride, const int* kv_len, int B,
                                    int H, int Lq, int Lk, int D, int window_left, int window_right,
                                    float scale, int dtype, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;
  const long long* arrays[8] = {q_stride, k_stride, v_stride, o_stride, do_stride, dq_stride, dk_stride,
                                dv_stride};
  for (const long long* a : arrays)
    if (!a) return FA_ERR_INVALID_ARG;
  BwdStrides sd;
  for (int i = 0; i < 3; ++i) {
    sd.q[i] = q_stride[i];
    sd.k[i] = k_stride[i];
    sd.v[i] = v_stride[i];
    sd.o[i] = o_stride[i];
    sd.dO[i] = do_stride[i];
    sd.dq[i] = dq_stride[i];
    sd.dk[i] = dk_stride[i];
    sd.dv[i] = dv_stride[i];
  }
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, kv_len, B, H, Lq, Lk, D, window_left, window_right,
                  scale, dtype == FA_DTYPE_FP16, sd, workspace, workspace_bytes, stream);
}
