// fa_fwd.cu -- FlashAttention-2 forward for GB300 (sm_103a), and its C ABI.
//
// What is computed (per batch b, head h, query row i):
//   O[i,:] = sum_j softmax_j(scale * Q[i,:].K[j,:]) V[j,:],  LSE[i] = ln sum_j exp(scale * Q[i,:].K[j,:])
// over all keys j < Lk, or only j <= i when causal.  The method is the one of the
// wsisp.com post "FlashAttention-2 forward in Triton": each query tile streams
// the K/V tiles of its head through an online softmax (running row max m,
// running exp-sum l, unnormalised fp32 accumulator rescaled when m grows), the
// score matrix never reaches global memory, and the epilogue writes O / l and
// m + log(l).  Causal runs skip the tiles past the diagonal and mask only the
// diagonal tile ("flash-attention-kernel" skill card, causal tips; the post's
// STAGE 1/2 split).  exp is taken as exp2 with log2(e) folded into the scale
// ("Triton Ascend Attention", 在线 Softmax 算法, which multiplies by 1.44269504).
//
// How it runs on sm_103a.  The grid is persistent: one CTA per SM (shared memory
// allows no more), each walking a static list of units.  A unit is a pair of
// 128-row query tiles of one (batch, head); units are numbered heaviest first and
// dealt out in boustrophedon order so the per-CTA totals stay balanced.
//   warp 8      : load warp.  TMA brings Q (once per unit) and a ring of K/V tiles
//                 into shared memory, 128B-swizzled, completing on mbarriers.
//   warp 9      : MMA warp.  One thread issues tcgen05.mma:
//                   S_i = Q_i K_j^T   (A and B from shared memory)  -> TMEM
//                   O_i += P_i V_j    (A = P from TMEM, B = V from shared memory)
//                 and tcgen05.commit signals completion on mbarriers.  It also
//                 owns the TMEM allocation (512 columns).
//   warps 0-3/4-7: softmax warpgroups, one per query tile; thread r owns row r
//                 (TMEM lane r): reads its S row, masks, takes the row max,
//                 exponentiates, writes P (bf16) back over S, rescales its O row
//                 in TMEM when the max grew by more than 2^8 (lazy rescale),
//                 and finally writes O / l (bf16) and the LSE.
//   warps 10-11 : spare (they give their registers to the softmax warpgroups).
// The two tiles alternate on the tensor cores: while one warpgroup turns S into
// P, the MMA warp runs the other tile's GEMMs.  Between units, the next unit's
// Q loads and first S GEMMs overlap the current unit's epilogue.
//
// Every pipeline wait is bounded in time.  A wait that runs out sets the
// library's device status word (FA_ERR_TIMEOUT), all roles stop, wait for
// their own copies and MMAs still in flight, free the TMEM and return.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>
#include <atomic>
#include <climits>
#include <mutex>
#include <utility>
#include <vector>
#include <queue>

#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// Device status word: 0, or an fa_status code in bits 0..7 and the wait site in bits 8..15.
__device__ unsigned int g_status;

constexpr int kBlockM = 128;        // query rows per tile (one tcgen05 M=128 MMA)
constexpr int kBlockN = 128;        // keys per K/V tile
constexpr int kThreads = 384;       // 8 softmax warps, load warp, MMA warp, 2 spare warps
// Register split between the warpgroups (setmaxnreg): each softmax thread holds a
// whole 128-column score row; the load/MMA warpgroup needs far fewer registers.
// 256 * kRegsSoftmax + 128 * kRegsOther must not exceed 384 * (registers at launch).
constexpr uint32_t kRegsSoftmax = 192;
constexpr uint32_t kRegsOther = 112;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold on the running max (log2 units)
constexpr unsigned long long kDefaultWaitNs = 1000000000ull;  // one second per wait

// Work schedules, one kernel instantiation each (template parameter kS).
//   kSchedWhole: whole units, every query tile starts at key tile 0 (full or causal mask).
//   kSchedSplit: key ranges cut across CTAs, merged by fa_combine_kernel.
//   kSchedBand : local (sliding-window) attention; each query tile covers its own band
//                of key tiles, and only tiles cut by the band's edges are masked.
//   kSchedTable: whole units in an order computed on the host (causal problems whose K/V
//                outgrow the L2 cache): heads in groups whose K/V fit in L2, each group's
//                units dealt heaviest first to the least-loaded CTA.
//   kSchedWholeList: kSchedWhole with the CTA's units listed in shared memory when the
//     kernel starts (D = 64, at most kMaxParts units per CTA): the unit arithmetic then
//     stays out of the roles' loops, which at D = 64 made the load and MMA warps spill.
enum Sched : int { kSchedWhole = 0, kSchedSplit = 1, kSchedBand = 2, kSchedTable = 3, kSchedWholeList = 4 };

enum WaitSite : uint32_t {
  kSiteLoadKV = 1, kSiteMmaQ, kSiteMmaK, kSiteMmaV, kSiteMmaP, kSiteSoftS, kSiteSoftO,
  kSiteMmaSFree, kSiteSoftPV, kSiteStage
};

template <int HD>
struct Layout {
  static constexpr int kTileBytes = kBlockM * HD * 2;    // one 128 x HD bf16 tile
  static constexpr int kRegionBytes = kBlockM * 128;     // 128 rows x 128 B (64 bf16): one swizzle column
  static constexpr int kRegions = HD / 64;
  static constexpr int kStages = (HD == 128) ? 4 : 8;    // K/V ring slots
  // D = 64 has shared memory to spare: two Q buffers per tile (the next unit's Q loads
  // while the current unit runs) and one O staging tile per query tile (the epilogue
  // writes O / l there and one TMA store moves the tile to global memory).
  static constexpr int kQBufs = (HD == 64) ? 2 : 1;
  static constexpr bool kTmaStoreO = (HD == 64);
  // D = 128: three Q buffers used as a ring by both tiles (a unit takes the next one or
  // two), so the next unit's Q_0 loads at any time and its Q_1 once tile 0 of the current
  // unit is done.
  static constexpr bool kQRing = (HD == 128);
  static constexpr int kQSlots = kQRing ? 3 : 2 * kQBufs;
  static constexpr int kOffQ = 0;                        // Q buffer b at kOffQ + b * kTileBytes
  static constexpr int kOffKV = kQSlots * kTileBytes;
  static constexpr int kOffStage = kOffKV + kStages * kTileBytes;   // [2] O staging (D = 64)
  static constexpr int kOffBar = kOffStage + (kTmaStoreO ? 2 : 0) * kTileBytes;
  static constexpr int kBarQFull = 0;                    // [kQSlots]  Q buffer landed
  static constexpr int kBarQEmpty = kQSlots;             // [kQSlots]  last MMA reading it done
  static constexpr int kBarKVFull = 2 * kQSlots;         // [kStages]
  static constexpr int kBarKVEmpty = kBarKVFull + kStages;
  static constexpr int kBarSFull = kBarKVEmpty + kStages;   // [2] S_i in TMEM
  static constexpr int kBarPFull = kBarSFull + 2;           // [2] P_i in TMEM, O_i rescaled
  static constexpr int kBarOFull = kBarPFull + 2;           // [2] last P_i V MMA of a unit done
  static constexpr int kBarOEmpty = kBarOFull + 2;          // [2] epilogue has read O_i
  static constexpr int kBarDrain = kBarOEmpty + 2;
  // Decoupled pipeline only (kDecoupled): S_i read out of TMEM into registers, and
  // the last P_i V MMA issued so far done (P_i columns free, O_i stable).
  static constexpr int kBarSFree = kBarDrain + 1;           // [2]
  static constexpr int kBarPVDone = kBarSFree + 2;          // [2]
  // D = 128 only: P_i is handed over in halves, p_full for its first 32 packed columns
  // (K-slices 0-3 of the P V MMA) and p_half for the other 32.
  static constexpr int kBarPHalf = kBarPVDone + 2;          // [2]
  // D = 64 epilogue: tile i's O staging buffer may be written (the previous TMA store has
  // read it; one arrival by the storing thread), and has been written (128 arrivals).
  static constexpr int kBarStageFree = kBarPHalf + 2;       // [2]
  static constexpr int kBarStageFull = kBarStageFree + 2;   // [2]
  static constexpr int kNumBars = kBarStageFull + 2;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  // Split schedule: the CTA's parts (kMaxParts x 8 ints: bh, q0, kv0, nblk[0] | nblk[1],
  // nmax, partial, slot), listed once when the kernel starts.  Every role reads its next
  // part from here: the search through the step space stays out of the roles' loops
  // (inlined there it made every key-tile step about 20 % slower).
  static constexpr int kMaxParts = 24;
  static constexpr int kOffNParts = kOffAbort + 4;
  static constexpr int kOffParts = (kOffNParts + 4 + 15) & ~15;
  static constexpr int kBytes = kOffParts + kMaxParts * 32;
  static constexpr int kAlloc = kBytes + 1024;           // slack to align the base to 1 KB
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: S_0 | S_1 | O_0 | O_1.  At D = 128 P_i (bf16 pairs) overwrites the
  // first 64 columns of S_i, so S_i(j+1) can only be computed after P_i(j) V.  At D = 64
  // the 128 columns left over hold P_0 | P_1 (kDecoupled): S_i(j+1) is computed as
  // soon as the softmax has read S_i(j), while it still works on that tile.
  static constexpr bool kDecoupled = (HD == 64);
  __host__ __device__ static constexpr uint32_t col_s(int i) { return 128u * i; }
  __host__ __device__ static constexpr uint32_t col_o(int i) { return 256u + HD * i; }
  __host__ __device__ static constexpr uint32_t col_p(int i) {
    return kDecoupled ? 256u + 2u * HD + 64u * i : 128u * i;
  }
};
static_assert(256 + 2 * 64 + 2 * 64 <= 512, "D = 64 TMEM budget: S, O and P of two tiles");

static_assert(Layout<128>::kAlloc <= 232448, "shared memory budget (D=128)");
static_assert(Layout<64>::kAlloc <= 232448, "shared memory budget (D=64)");

struct Params {
  CUtensorMap tm_q;   // 4-D views [B][H][L][D] of Q, K, V (caller's strides); box 64 x 128 x 1 x 1
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;   // D = 64: 4-D view of O for the epilogue's TMA stores (same box)
  uint16_t* o;        // bf16 or fp16 elements
  long long o_sb, o_sh, o_sl;   // O strides in elements (batch, head, row); features contiguous
  int o_v8;           // O's base and strides are 32-byte multiples: the epilogue stores 32 B a time
  float* lse;         // contiguous [B*H][Lq]
  int bh_count;
  int H;
  int Lq;
  int Lk;
  int causal;
  int n_pairs;        // ceil(Lq / 256)
  int n_units;        // n_pairs * bh_count
  int nkv;            // key tiles per unit: ceil(Lk / 128)
  int split;          // 0: whole units, boustrophedon; 1: split key ranges (stream-K)
  long long total_steps;   // split schedule: key-tile steps of all units plus unit_cost per unit
  int unit_cost;           // split schedule: virtual steps in front of each unit
  float* ws_o;        // split schedule: partial O rows   [2 * grid][2 tiles][128 rows][D] fp32
  float* ws_ml;       //                 partial (m, l)   [2 * grid][2 tiles][128 rows][2] fp32
  int win_left;       // band schedule: key j allowed for row i iff i - win_left <= j <= i + win_right,
  int win_right;      //   -1 = unbounded on that side; both are below Lq / Lk
  int band_desc;      // band schedule: 1 = units in descending query order (heavier last tiles)
  const int* kv_len;  // band schedule: per-batch count of valid keys (keys j >= kv_len[b] are
                      //   padding), device memory; nullptr = none
  float scale_log2;   // scale * log2(e)
  uint32_t flags;     // test hooks (fa_debug_set)
  unsigned long long wait_limit_ns;
};

// The host-computed order of kSchedTable, passed with the launch: CTA g takes the units
// tab_units[tab_off[g] .. tab_off[g + 1]) in that order.
constexpr int kTabMaxGrid = 256;
constexpr int kTabMaxUnits = 4096;
struct TableParams : Params {
  uint16_t tab_off[kTabMaxGrid + 1];
  uint32_t tab_units[kTabMaxUnits];   // (bh << 12) | index of the pair of query tiles
};
template <int kS> struct ParamsOf { using type = Params; };
template <> struct ParamsOf<kSchedTable> { using type = TableParams; };

// A unit of work: two consecutive 128-row query tiles of one (batch, head).
// Units are numbered heaviest first (causal: the last query tiles attend to the
// most keys); a CTA takes units in boustrophedon order over the grid (round r:
// CTA g takes unit r*G + g when r is even, r*G + G-1-g when odd), which keeps
// the per-CTA totals within a few percent of each other for causal loads.
//
// Split schedule: the units' key tiles form one sequence of T steps (head after head,
// each head's pairs in order; nkv per unit for the full mask, the key tiles up to the
// diagonal with the causal mask) and CTA g takes the steps [T*g/G, T*(g+1)/G).  A unit cut by a CTA boundary is processed in parts; each
// part leaves its rows' partial state (unnormalised O, running max m, sum l) in
// the workspace, and a second kernel on the same stream merges the parts of every
// split unit into the final O and LSE.  No CTA ever waits for another.
struct Unit {
  int bh;
  int q0;
  int kv0;       // first key tile of this (part of a) unit
  int nblk[2];   // key tiles of query tile 0 and 1 in this part (0 = tile absent)
  int first[2];  // band schedule: key tile (relative to kv0) where query tile i starts
  int nmax;      // key tiles loaded for the unit: the union of the tiles' ranges
  int kvl;       // band schedule: valid keys of the unit's batch (Lk without padding)
  int partial;   // 1: a part of a unit split across CTAs
  int slot;      // workspace slot of this part: 2 * CTA + (first part of the CTA ? 0 : 1)
};

__device__ __forceinline__ long long split_lo(const Params& p, int g) {
  return p.total_steps * g / static_cast<int>(gridDim.x);
}

// Split schedule step space: the units of a head are its pairs of query tiles in order
// (pair p = rows [256p, 256p + 256)), heads one after the other; a unit's steps are the key
// tiles of its longer tile: all nkv of them for the full mask, with the causal mask the
// tiles up to the diagonal of its last present tile.  Each unit is preceded by `cost`
// virtual steps that stand for what a part costs besides its key tiles (loading its Q
// tiles, its first S, parking its rows), so that a CTA whose range holds many short units
// gets fewer key tiles.  A part is the intersection of a CTA's range with a unit's key
// tiles; a range that meets only a unit's virtual steps holds no part of it.
__host__ __device__ inline long long pair_steps(int pair, int nkv, int Lq, int causal) {
  if (!causal) return nkv;
  const int last = (pair * 2 * kBlockM + kBlockM < Lq) ? 2 * pair + 2 : 2 * pair + 1;
  return last < nkv ? last : nkv;
}
// Steps of pairs [0, P) of one head (P <= n_pairs), `cost` virtual steps per pair included.
__host__ __device__ inline long long head_prefix(int P, int nkv, int Lq, int n_pairs, int causal,
                                                 int cost) {
  const long long virt = static_cast<long long>(P) * cost;
  if (!causal) return static_cast<long long>(P) * nkv + virt;
  const long long c = nkv / 2;   // pairs p with 2p + 2 <= nkv
  long long s = (P <= c) ? static_cast<long long>(P) * (P + 1)
                         : c * (c + 1) + static_cast<long long>(P - c) * nkv;
  if (P == n_pairs && n_pairs > 0) {   // the head's last pair may lack its second tile
    const long long full = 2ll * (n_pairs - 1) + 2 < nkv ? 2ll * (n_pairs - 1) + 2 : nkv;
    s -= full - pair_steps(n_pairs - 1, nkv, Lq, causal);
  }
  return s + virt;
}
// The unit whose steps (virtual ones included) contain step x: its head, pair, first step
// (its first virtual step) and number of key-tile steps.
__host__ __device__ inline void split_locate(long long x, int nkv, int Lq, int n_pairs, int causal,
                                             int cost, int* bh, int* pair, long long* start,
                                             long long* steps) {
  const long long per_head = head_prefix(n_pairs, nkv, Lq, n_pairs, causal, cost);
  const long long h = x / per_head, xh = x - h * per_head;
  int lo = 0, hi = n_pairs - 1;   // the last pair whose first step is <= xh
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (head_prefix(mid, nkv, Lq, n_pairs, causal, cost) <= xh) lo = mid;
    else hi = mid - 1;
  }
  *bh = static_cast<int>(h);
  *pair = lo;
  *start = h * per_head + head_prefix(lo, nkv, Lq, n_pairs, causal, cost);
  *steps = pair_steps(lo, nkv, Lq, causal);
}

__device__ __forceinline__ void unit_rows(const Params& p, int idx, Unit& u) {
  if (p.causal) {   // heaviest first: the last query tiles of every head come first
    const int pair = p.n_pairs - 1 - idx / p.bh_count;
    u.bh = idx % p.bh_count;
    u.q0 = pair * 2 * kBlockM;
  } else {          // equal costs: the units of one head are neighbours, so they run together
    u.bh = idx / p.n_pairs;
    u.q0 = (idx % p.n_pairs) * 2 * kBlockM;
  }
}

// Band schedule: allowed keys of row q are [band_lo(q), band_lim(q, kvl)), where kvl is
// the number of valid (unpadded) keys of the row's batch.
__device__ __forceinline__ int band_lo(const Params& p, int q) {
  return p.win_left < 0 ? 0 : max(0, q - p.win_left);
}
__device__ __forceinline__ int band_lim(const Params& p, int q, int kvl) {
  return p.win_right < 0
             ? kvl
             : static_cast<int>(min(static_cast<long long>(kvl),
                                    static_cast<long long>(q) + p.win_right + 1));
}

template <int kS, class P>
__device__ __forceinline__ bool unit_of(const P& p, int r, Unit& u) {
  const int G = static_cast<int>(gridDim.x);
  const int g = static_cast<int>(blockIdx.x);
  if constexpr (kS == kSchedTable) {
    const int e = p.tab_off[g] + r;
    if (e >= p.tab_off[g + 1]) return false;
    const uint32_t t = p.tab_units[e];
    u.bh = static_cast<int>(t >> 12);
    u.q0 = static_cast<int>(t & 0xfffu) * 2 * kBlockM;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int qi = u.q0 + i * kBlockM;
      u.nblk[i] = (qi >= p.Lq) ? 0 : (p.causal ? min(p.nkv, qi / kBlockN + 1) : p.nkv);
    }
    u.nmax = max(u.nblk[0], u.nblk[1]);
    u.kv0 = 0;
    u.first[0] = u.first[1] = 0;
    u.partial = 0;
    return true;
  } else if constexpr (kS == kSchedBand) {
    // Units in the order that puts the heaviest first: descending query order
    // when the band is bounded on the right or open on the left (the last tiles
    // see the most keys), ascending when only the left side is bounded.
    const int idx = r * G + ((r & 1) ? (G - 1 - g) : g);
    if (idx >= p.n_units) return false;
    const int pi = idx / p.bh_count;
    const int pair = p.band_desc ? p.n_pairs - 1 - pi : pi;
    u.bh = idx % p.bh_count;
    u.q0 = pair * 2 * kBlockM;
    u.kvl = p.kv_len ? min(max(__ldg(p.kv_len + u.bh / p.H), 0), p.Lk) : p.Lk;
    // Tile i covers key tiles a[i]..b[i]: from the band's left edge at its first
    // row to its right edge at its last stored row (both edges only move right as the
    // row grows).  The two ranges overlap or touch, so the unit loads one contiguous
    // run of key tiles.  With key padding a tile's range can be empty (b < a).
    int a[2], b[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int qt = u.q0 + i * kBlockM;
      if (qt >= p.Lq) {   // tile 1 absent (tile 0 never is)
        a[i] = a[0];
        b[i] = a[0] - 1;
        continue;
      }
      const int last = min(qt + kBlockM, p.Lq) - 1;   // last row that is stored
      const int lo = band_lo(p, qt), lim = band_lim(p, last, u.kvl);
      a[i] = lo / kBlockN;
      b[i] = lim > lo ? (lim - 1) / kBlockN : a[i] - 1;
    }
    u.kv0 = a[0];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      u.nblk[i] = max(0, b[i] - a[i] + 1);   // 0 when the tile is absent or has no keys
      u.first[i] = u.nblk[i] > 0 ? a[i] - a[0] : 0;
    }
    u.nmax = max(u.nblk[0], u.first[1] + u.nblk[1]);
    u.partial = 0;
    return true;
  } else if constexpr (kS == kSchedWhole || kS == kSchedWholeList) {
    const int idx = r * G + ((r & 1) ? (G - 1 - g) : g);
    if (idx >= p.n_units) return false;
    unit_rows(p, idx, u);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int qi = u.q0 + i * kBlockM;
      u.nblk[i] = (qi >= p.Lq) ? 0 : (p.causal ? min(p.nkv, qi / kBlockN + 1) : p.nkv);
    }
    u.nmax = max(u.nblk[0], u.nblk[1]);
    u.kv0 = 0;
    u.first[0] = u.first[1] = 0;
    u.partial = 0;
    return true;
  } else {
  const long long lo = split_lo(p, g), hi = split_lo(p, g + 1);
  long long x = lo;
  int bh = 0, pair = 0, k = 0;
  long long start = 0, steps = 0, ra = 0, rb = 0;
  for (; x < hi; x = min(start + p.unit_cost + steps, hi)) {   // the r-th part of the range
    split_locate(x, p.nkv, p.Lq, p.n_pairs, p.causal, p.unit_cost, &bh, &pair, &start, &steps);
    const long long ks = start + p.unit_cost;   // the unit's first key-tile step
    ra = max(x, ks);
    rb = min(ks + steps, hi);
    if (ra < rb && k++ == r) break;
  }
  if (x >= hi) return false;
  const int a = static_cast<int>(ra - (start + p.unit_cost));
  const int len = static_cast<int>(rb - ra);
  u.bh = bh;
  u.q0 = pair * 2 * kBlockM;
#pragma unroll
  for (int i = 0; i < 2; ++i) {   // the tile's key tiles that fall in this part's [a, a + len)
    const int qi = u.q0 + i * kBlockM;
    const int all = p.causal ? min(p.nkv, qi / kBlockN + 1) : p.nkv;
    u.nblk[i] = (qi >= p.Lq) ? 0 : max(0, min(all, a + len) - a);
  }
  u.nmax = len;
  u.kv0 = a;
  u.first[0] = u.first[1] = 0;
  u.partial = (len != steps);
  // A cut unit is its range's first or last part (the ones between are whole).
  if (u.partial) u.slot = 2 * g + (r == 0 ? 0 : 1);
  return true;
  }
}

// tcgen05 instruction descriptor, kind::f16: fp32 accumulator, A and B both bf16 (or
// both fp16 with f16), A K-major, B K-major or (b_mn_major) MN-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major, bool f16 = false) {
  return (1u << 4)                            // D format: f32
         | ((f16 ? 0u : 1u) << 7)             // A format: bf16 (1) or f16 (0)
         | ((f16 ? 0u : 1u) << 10)            // B format: the same as A
         | ((b_mn_major ? 1u : 0u) << 16)     // B major-ness
         | (static_cast<uint32_t>(N >> 3) << 17)
         | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128B-swizzled operand (tcgen05 format).
// lbo/sbo in bytes: for K-major operands sbo is the distance between 8-row
// groups (1024 B) and lbo is unused; for MN-major operands lbo is the distance
// between 64-element column blocks and sbo the distance between 8-row K groups.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu)
         | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16)
         | (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32)
         | (1ull << 46)     // descriptor version for tcgen05
         | (2ull << 61);    // 128-byte swizzle
}

// Bounded wait on an mbarrier phase (inlined: it sits on every pipeline handoff).
// Gives up when another role aborted or after `limit_ns`, in which case it
// records FA_ERR_TIMEOUT and raises the CTA abort flag.
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
        atomicCAS(&g_status, 0u, static_cast<unsigned>(FA_ERR_TIMEOUT) | (site << 8));
        return false;
      }
    }
  }
}

// wait_phase for a whole warp that must stay converged: true only if every lane's
// wait succeeded.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long limit_ns, uint32_t site) {
  return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, limit_ns, site));
}

// Bounded wait used while draining: ignores the abort flag (the copy or MMA being
// waited for completes on its own), still limited in time.
__device__ __noinline__ bool drain_phase(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// kS selects the schedule at compile time, so the whole-unit kernel carries none
// of the other schedules' code.
// exp2 of a pair, packed as the I/O type (P has the type of V in the P V MMA).
template <bool kF16>
__device__ __forceinline__ uint32_t exp2_pair(float x0, float x1, uint64_t k2, uint64_t c2, uint64_t& acc) {
  if constexpr (kF16) return ptx::exp2_pair_f16(x0, x1, k2, c2, acc);
  else return ptx::exp2_pair_bf16(x0, x1, k2, c2, acc);
}

// Two floats to the packed 16-bit element pair of the I/O type.
template <bool kF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kF16) return ptx::pack_f16x2(lo, hi);
  else return ptx::pack_bf16x2(lo, hi);
}

template <int HD, int kS, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_kernel(const __grid_constant__ typename ParamsOf<kS>::type p) {
  using L = Layout<HD>;
  constexpr bool kSplit = kS == kSchedSplit;
  constexpr bool kBand = kS == kSchedBand;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_addr(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  auto bar = [&](int idx) -> uint32_t { return sbase + L::kOffBar + 8u * idx; };
  volatile int* s_nparts = reinterpret_cast<volatile int*>(smem + L::kOffNParts);
  int4* s_parts = reinterpret_cast<int4*>(smem + L::kOffParts);
  // The r-th unit of this CTA (false: none left).  Split parts and listed whole units come
  // from the list that thread 0 writes before the CTA-wide barrier below; the other
  // schedules find their units directly.
  auto unit_at = [&](int r, Unit& u) -> bool {
    if constexpr (kSplit || kS == kSchedWholeList) {
      if (r >= *s_nparts) return false;
      const int4 a = s_parts[2 * r], b = s_parts[2 * r + 1];
      u.bh = a.x;
      u.q0 = a.y;
      u.kv0 = a.z;
      u.nblk[0] = a.w;
      u.nblk[1] = b.x;
      u.nmax = b.y;
      u.partial = b.z;
      u.slot = b.w;
      u.first[0] = u.first[1] = 0;
      return true;
    } else {
      return unit_of<kS>(p, r, u);
    }
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < L::kQSlots; ++i) {
      ptx::mbar_init(bar(L::kBarQFull + i), 1);
      ptx::mbar_init(bar(L::kBarQEmpty + i), 1);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(L::kBarSFull + i), 1);
      ptx::mbar_init(bar(L::kBarPFull + i), 4 * 32);
      ptx::mbar_init(bar(L::kBarPHalf + i), 4 * 32);
      ptx::mbar_init(bar(L::kBarOFull + i), 1);
      ptx::mbar_init(bar(L::kBarOEmpty + i), 4 * 32);
    }
#pragma unroll
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(L::kBarKVFull + s), 1);
      ptx::mbar_init(bar(L::kBarKVEmpty + s), 1);
    }
    ptx::mbar_init(bar(L::kBarDrain), 1);
    if constexpr (kSplit || kS == kSchedWholeList) {
      // The host takes these schedules only when no CTA has more than kMaxParts units.
      int n = 0;
      Unit t;
      while (n < L::kMaxParts && unit_of<kS>(p, n, t)) {
        s_parts[2 * n] = make_int4(t.bh, t.q0, t.kv0, t.nblk[0]);
        s_parts[2 * n + 1] = make_int4(t.nblk[1], t.nmax, t.partial, t.partial ? t.slot : 0);
        ++n;
      }
      // More units than the list holds would be a host planning error: report it and do
      // nothing rather than drop units silently.
      if (n == L::kMaxParts && unit_of<kS>(p, n, t)) {
        atomicCAS(&g_status, 0u, static_cast<unsigned>(FA_ERR_UNSUPPORTED));
        n = 0;
      }
      *s_nparts = n;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(L::kBarStageFree + i), 1);
      ptx::mbar_init(bar(L::kBarStageFull + i), 4 * 32);
    }
    if constexpr (L::kDecoupled) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        ptx::mbar_init(bar(L::kBarSFree + i), 4 * 32);
        ptx::mbar_init(bar(L::kBarPVDone + i), 1);
      }
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
  // While the previous kernel finishes, warm L2 with this CTA's first Q and K/V tiles: a
  // prefetch only reads, and L2 is where the previous kernel's writes land, so a tile it
  // writes is still read fresh after the wait below.  (Key padding reads its counts from
  // memory to find the unit, so that schedule skips it.)
  if (warp == kLoadWarp && lane == 0 && !(kBand && p.kv_len)) {
    Unit u0;
    if (unit_at(0, u0)) {
      const int ub = u0.bh / p.H, uh = u0.bh - ub * p.H;
#pragma unroll
      for (int rg = 0; rg < L::kRegions; ++rg) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (u0.nblk[i] > 0) ptx::tma_prefetch_l2_4d(&p.tm_q, 64 * rg, u0.q0 + i * kBlockM, uh, ub);
        if (u0.nmax > 0) {
          ptx::tma_prefetch_l2_4d(&p.tm_k, 64 * rg, u0.kv0 * kBlockN, uh, ub);
          ptx::tma_prefetch_l2_4d(&p.tm_v, 64 * rg, u0.kv0 * kBlockN, uh, ub);
        }
      }
    }
  }
  // Launched as a programmatic dependent of the previous kernel in the stream: the set-up
  // above overlapped its tail; nothing in global memory is touched before it completes.
  // The next kernel may be scheduled now (it waits the same way before touching memory).
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();

  if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroups
    ptx::setmaxnreg_inc<kRegsSoftmax>();
    const int wg = warp >> 2;           // query tile 0 or 1 of each unit
    const int rw = warp & 3;            // TMEM lane quarter this warp may access
    const int row = rw * 32 + lane;     // row of the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(rw * 32) << 16;
    const uint32_t t_s = tmem + lane_off + L::col_s(wg);
    const uint32_t t_o = tmem + lane_off + L::col_o(wg);
    const uint32_t t_p = tmem + lane_off + L::col_p(wg);
    const float sl2 = p.scale_log2;
    uint32_t s_base = 0;    // S_i tiles consumed in earlier units (s_full / p_full phase)
    uint32_t o_count = 0;   // units finished by this warpgroup (o_full phase)
    uint32_t n_stage = 0;   // epilogues through the O staging buffer (stage_free / stage_full phase)
    bool ok = true;
    Unit u;
    for (int r = 0; ok && unit_at(r, u); ++r) {
      const int n_blocks = wg ? u.nblk[1] : u.nblk[0];
      if constexpr (kSplit) {
        // Causal split: a part can hold no key tile of the first (shorter) query tile; its
        // slot then holds an empty partial state (O = 0, m = -inf, l = 0) for the merge.
        if (n_blocks == 0 && u.partial && u.q0 + wg * kBlockM < p.Lq) {
          const size_t rowi = static_cast<size_t>(u.slot * 2 + wg) * kBlockM + row;
          float* so = p.ws_o + rowi * HD;
#pragma unroll
          for (int c = 0; c < HD; c += 4) *reinterpret_cast<float4*>(so + c) = make_float4(0.f, 0.f, 0.f, 0.f);
          p.ws_ml[rowi * 2] = -INFINITY;
          p.ws_ml[rowi * 2 + 1] = 0.0f;
          continue;
        }
      }
      if (n_blocks == 0) {
        // Band schedule: a present tile whose rows have no allowed key (key padding):
        // O = 0 and LSE = -inf, written here without any MMA.
        if constexpr (kBand) {
          const int qz = u.q0 + wg * kBlockM + row;
          if (qz < p.Lq) {
            const int zb = u.bh / p.H, zh = u.bh - zb * p.H;
            uint16_t* zrow = p.o + zb * p.o_sb + zh * p.o_sh + static_cast<long long>(qz) * p.o_sl;
#pragma unroll
            for (int c = 0; c < HD; c += 8) *reinterpret_cast<uint4*>(zrow + c) = make_uint4(0, 0, 0, 0);
            p.lse[static_cast<size_t>(u.bh) * p.Lq + qz] = -INFINITY;
          }
        }
        continue;
      }
      const int bh = u.bh;
      const int qt = u.q0 + wg * kBlockM;
      const int q = qt + row;
      const int key_lim = kBand ? band_lim(p, q, u.kvl) : (p.causal ? min(p.Lk, q + 1) : p.Lk);
      const int first_diag = p.causal ? qt / kBlockN : INT_MAX;
      // Band: row q keeps keys [key_lo, key_lim); a key tile needs masking when the
      // band's left edge (of the tile's last row) or right edge (of its first row) cuts it.
      const int key_lo = kBand ? band_lo(p, q) : 0;
      const int lo_last = kBand ? band_lo(p, qt + kBlockM - 1) : 0;
      const int lim_first = kBand ? band_lim(p, qt, u.kvl) : 0;
      const int jb0 = kBand ? u.kv0 + (wg ? u.first[1] : u.first[0]) : (kSplit ? u.kv0 : 0);
      float m = -INFINITY;   // running max of scaled scores, log2 units (possibly stale by < 8)
      float l = 0.0f;        // running sum of exp2(s*sl2 - m)
      for (int j = 0; j < n_blocks; ++j) {
        ok = wait_phase(bar(L::kBarSFull + wg), (s_base + j) & 1, abort_flag, limit, kSiteSoftS);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ptx::tc_fence_after();
        uint32_t sr[128];
        ptx::tmem_ld32x32b_x128(t_s, sr);
        if constexpr (L::kDecoupled) {   // S_i is in registers: the MMA may overwrite it
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(L::kBarSFree + wg));
        }
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
        const int jb = jb0 + j;   // key tile index
        if constexpr (kBand) {
          if (jb * kBlockN < lo_last || (jb + 1) * kBlockN > lim_first) {
            const int lo = key_lo - jb * kBlockN;    // columns lo <= c < lim are allowed keys
            const int lim = key_lim - jb * kBlockN;
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = (c >= lo && c < lim) ? s[c] : -INFINITY;
          }
        } else if (jb >= first_diag || (jb + 1) * kBlockN > p.Lk) {
          const int lim = key_lim - jb * kBlockN;   // columns c < lim are allowed keys
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
        }
        float mx[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) mx[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
        for (int c = 8; c < 128; c += 8) {
#pragma unroll
          for (int k = 0; k < 4; ++k) mx[k] = ptx::fmax3(mx[k], s[c + 2 * k], s[c + 2 * k + 1]);
        }
        const float rmax = ptx::fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
        const float m_new = fmaxf(m, rmax * sl2);
        const bool rescale = m_new > m + kRescaleLog2;
        float alpha = 1.0f;
        if (rescale) {
          alpha = ptx::ex2_approx(m - m_new);
          m = m_new;
        }
        const float neg_m = (m == -INFINITY) ? 0.0f : -m;
        const uint64_t k2 = ptx::pack_f32x2(sl2, sl2);
        const uint64_t c2 = ptx::pack_f32x2(neg_m, neg_m);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        if constexpr (L::kDecoupled) {
          // P_i(j) may only be stored once P_i(j-1) V has been computed (P_i columns
          // free, O_i no longer being accumulated): the first half of the row is
          // exponentiated before that wait, the second half while the first is stored.
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c)
            pk[c] = exp2_pair<kF16>(s[2 * c], s[2 * c + 1], k2, c2, acc[c & 3]);
          if (j > 0) {
            ok = wait_phase(bar(L::kBarPVDone + wg), (s_base + j - 1) & 1, abort_flag, limit,
                            kSiteSoftPV);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
              for (int c0 = 0; c0 < HD; c0 += 32) {
                uint32_t o[32];
                ptx::tmem_ld32x32b_x32(t_o + c0, o);
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                ptx::tmem_st32x32b_x32(t_o + c0, o);
              }
            }
          }
          ptx::tmem_st32x32b_x32(t_p, pk);
#pragma unroll
          for (int c = 0; c < 32; ++c)
            pk[c] = exp2_pair<kF16>(s[64 + 2 * c], s[64 + 2 * c + 1], k2, c2, acc[c & 3]);
          ptx::tmem_st32x32b_x32(t_p + 32, pk);
          float2 a0 = ptx::unpack_f32x2(acc[0]), a1 = ptx::unpack_f32x2(acc[1]);
          float2 a2 = ptx::unpack_f32x2(acc[2]), a3 = ptx::unpack_f32x2(acc[3]);
          l = l * alpha + (((a0.x + a0.y) + (a1.x + a1.y)) + ((a2.x + a2.y) + (a3.x + a3.y)));
        } else {
          // P_i in halves: the MMA warp starts P V on the first while the second is computed.
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c)
              pk[c] = exp2_pair<kF16>(s[64 * h + 2 * c], s[64 * h + 2 * c + 1], k2, c2, acc[c & 3]);
            ptx::tmem_st32x32b_x32(t_s + 32 * h, pk);
            // O_i was last written by P_i(j-1) V, complete since S_i(j) is: rescale it
            // before the first half is handed over, as that half's MMAs accumulate into O_i.
            if (h == 0 && j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
              for (int c0 = 0; c0 < HD; c0 += 32) {
                uint32_t o[32];
                ptx::tmem_ld32x32b_x32(t_o + c0, o);
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                ptx::tmem_st32x32b_x32(t_o + c0, o);
              }
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar((h == 0 ? L::kBarPFull : L::kBarPHalf) + wg));
          }
          float2 a0 = ptx::unpack_f32x2(acc[0]), a1 = ptx::unpack_f32x2(acc[1]);
          float2 a2 = ptx::unpack_f32x2(acc[2]), a3 = ptx::unpack_f32x2(acc[3]);
          l = l * alpha + (((a0.x + a0.y) + (a1.x + a1.y)) + ((a2.x + a2.y) + (a3.x + a3.y)));
        }
        if constexpr (L::kDecoupled) {
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(L::kBarPFull + wg));
        }
      }
      if (!ok) break;
      s_base += n_blocks;
      ok = wait_phase(bar(L::kBarOFull + wg), o_count & 1, abort_flag, limit, kSiteSoftO);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++o_count;
      ptx::tc_fence_after();
      if (kSplit && u.partial) {
        // A part of a split unit: park this row's state (unnormalised O, m, l) for
        // the combine kernel that runs after this one.
        const size_t rowi = static_cast<size_t>(u.slot * 2 + wg) * kBlockM + row;
        float* so = p.ws_o + rowi * HD;   // 32-byte aligned: 256-byte base, HD * 4-byte rows
        // The whole row first, O released at once, then whole 32-byte sectors from registers.
        uint32_t o[HD / 32][32];
#pragma unroll
        for (int k = 0; k < HD / 32; ++k) ptx::tmem_ld32x32b_x32(t_o + 32 * k, o[k]);
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarOEmpty + wg));
#pragma unroll
        for (int k = 0; k < HD / 32; ++k)
#pragma unroll
          for (int v = 0; v < 4; ++v) ptx::st_global_v8(so + 32 * k + 8 * v, o[k] + 8 * v);
        p.ws_ml[rowi * 2] = m;
        p.ws_ml[rowi * 2 + 1] = l;
        continue;
      }
      // Epilogue: O / l as bf16 rows, LSE = ln2 * (m + log2 l); rows >= Lq are not stored.
      // (band schedule: a row with no allowed key has l = 0 and gets O = 0, LSE = -inf)
      const float inv_l = kBand ? (l > 0.0f ? 1.0f / l : 0.0f) : 1.0f / l;
      const bool store = q < p.Lq;
      const int ob = bh / p.H, oh = bh - ob * p.H;
      if constexpr (L::kTmaStoreO) {
        // D = 64: each thread writes its row into this tile's staging buffer in the
        // 128-byte-swizzled layout of the O tensor map (16-byte chunk c of row r at chunk
        // position c ^ (r % 8)), and one thread stores the 128 x 64 tile with TMA; rows
        // past Lq lie outside the tensor and are not written.
        const uint32_t stage = sbase + L::kOffStage + wg * L::kTileBytes;
        const bool leader = (threadIdx.x & 127) == 0;
        if (leader) {
          ptx::bulk_wait_read_all();   // the previous store has read the buffer
          ptx::mbar_arrive(bar(L::kBarStageFree + wg));
        }
        ok = wait_phase(bar(L::kBarStageFree + wg), n_stage & 1, abort_flag, limit, kSiteStage);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint32_t row_addr = stage + row * 128;
#pragma unroll
        for (int c0 = 0; c0 < HD; c0 += 32) {
          uint32_t o[32];
          ptx::tmem_ld32x32b_x32(t_o + c0, o);
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = pack2<kF16>(__uint_as_float(o[2 * c]) * inv_l,
                                __uint_as_float(o[2 * c + 1]) * inv_l);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t chunk = static_cast<uint32_t>((c0 >> 3) + v);
            ptx::st_shared_v4(row_addr + ((chunk ^ static_cast<uint32_t>(row & 7)) << 4), pk[4 * v],
                              pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
        // O_i has been read into registers: the next unit's P_i V MMA may overwrite it.
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::kBarOEmpty + wg));
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(bar(L::kBarStageFull + wg));
        if (leader) {
          if (wait_phase(bar(L::kBarStageFull + wg), n_stage & 1, abort_flag, limit, kSiteStage)) {
            ptx::tma_store_4d(&p.tm_o, stage, 0, qt, oh, ob);
            ptx::bulk_commit_group();
          } else {
            ok = false;
          }
        }
        ok = __all_sync(0xffffffffu, ok);
        ++n_stage;
      } else {
      uint16_t* orow = p.o + ob * p.o_sb + oh * p.o_sh + static_cast<long long>(store ? q : 0) * p.o_sl;
      // Read the whole row of O first and release O_i (the next unit's first P_i V MMA
      // may overwrite it), then normalise and store from registers.
      uint32_t o[HD / 32][32];
#pragma unroll
      for (int k = 0; k < HD / 32; ++k) ptx::tmem_ld32x32b_x32(t_o + 32 * k, o[k]);
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::kBarOEmpty + wg));
#pragma unroll
      for (int k = 0; k < HD / 32; ++k) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack2<kF16>(__uint_as_float(o[k][2 * c]) * inv_l,
                              __uint_as_float(o[k][2 * c + 1]) * inv_l);
        if (store) {
          // Each warp store writes 32 rows: 32-byte pieces halve the instructions when O's
          // layout allows them (measured 0.5-2.7 % on whole launches at D = 128).
          if (p.o_v8) {
            ptx::st_global_v8(orow + 32 * k, pk);
            ptx::st_global_v8(orow + 32 * k + 16, pk + 8);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * k);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      }
      }
      if (store) {
        p.lse[static_cast<size_t>(bh) * p.Lq + q] = (m + log2f(l)) * 0.69314718055994531f;
      }
    }
  } else if (warp == kLoadWarp) {
    // ------------------------------------------------------------ load warp
    ptx::setmaxnreg_dec<kRegsOther>();
    if (lane == 0) {
      ptx::prefetch_tensormap(&p.tm_q);
      ptx::prefetch_tensormap(&p.tm_k);
      ptx::prefetch_tensormap(&p.tm_v);
      uint32_t q_count[2] = {0, 0};   // Q_i loads issued so far
      uint32_t q_pos = 0;             // Q ring position of the next load (kQRing)
      uint32_t it = 0;                // K/V ring position (K_j and V_j alternate)
      int last_fill[L::kStages];
#pragma unroll
      for (int s = 0; s < L::kStages; ++s) last_fill[s] = -1;
      bool ok = true;
      bool first = true;
      Unit u;
      for (int r = 0; ok && unit_at(r, u); ++r) {
        const int ub = u.bh / p.H, uh = u.bh - ub * p.H;   // batch and head of the unit
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (u.nblk[i] == 0) continue;
          // Buffers alternate between units (D = 64); a buffer is refilled once the MMAs of
          // its previous unit have read it.  uses = earlier loads into this buffer.
          int qi;
          uint32_t uses;
          if constexpr (L::kQRing) {
            qi = static_cast<int>(q_pos % 3u);
            uses = q_pos / 3u;
            ++q_pos;
          } else {
            qi = 2 * (L::kQBufs == 2 ? static_cast<int>(q_count[i] & 1) : 0) + i;
            uses = L::kQBufs == 2 ? (q_count[i] >> 1) : q_count[i];
          }
          if (uses > 0 && !wait_phase(bar(L::kBarQEmpty + qi), (uses - 1) & 1,
                                      abort_flag, limit, kSiteLoadKV)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(bar(L::kBarQFull + qi), L::kTileBytes);
#pragma unroll
          for (int rg = 0; rg < L::kRegions; ++rg)
            ptx::tma_load_4d(sbase + L::kOffQ + qi * L::kTileBytes + rg * L::kRegionBytes, &p.tm_q,
                             bar(L::kBarQFull + qi), 64 * rg, u.q0 + i * kBlockM, uh, ub);
          ++q_count[i];
        }
        for (int j = 0; j < u.nmax && ok; ++j) {
#pragma unroll
          for (int t = 0; t < 2; ++t, ++it) {   // t = 0: K_j, t = 1: V_j
            const int s = it % L::kStages;
            const uint32_t ph = (it / L::kStages) & 1;
            if (!wait_phase(bar(L::kBarKVEmpty + s), ph ^ 1u, abort_flag, limit, kSiteLoadKV)) {
              ok = false;
              break;
            }
            if ((p.flags & 1u) && first && j == 0 && t == 1) continue;   // test hook: withhold V_0
            ptx::mbar_arrive_expect_tx(bar(L::kBarKVFull + s), L::kTileBytes);
#pragma unroll
            for (int rg = 0; rg < L::kRegions; ++rg)
              ptx::tma_load_4d(sbase + L::kOffKV + s * L::kTileBytes + rg * L::kRegionBytes,
                               t ? &p.tm_v : &p.tm_k, bar(L::kBarKVFull + s), 64 * rg,
                               (u.kv0 + j) * kBlockN, uh, ub);
            last_fill[s] = static_cast<int>(it);
          }
        }
        first = false;
      }
      // Drain: every copy this thread started has landed before the CTA may exit.
#pragma unroll
      for (int s = 0; s < L::kStages; ++s)
        if (last_fill[s] >= 0)
          drain_phase(bar(L::kBarKVFull + s), (last_fill[s] / L::kStages) & 1, limit);
      if constexpr (L::kQRing) {
#pragma unroll
        for (int b = 0; b < 3; ++b) {   // loads into ring buffer b: positions b, b + 3, ...
          const uint32_t n = (q_pos + 2u - b) / 3u;
          if (n > 0) drain_phase(bar(L::kBarQFull + b), (n - 1) & 1, limit);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
          for (int b = 0; b < L::kQBufs; ++b) {
            // loads into buffer b of tile i: every kQBufs-th load, starting with load b
            const uint32_t n = (q_count[i] + L::kQBufs - 1 - b) / L::kQBufs;
            if (n > 0) drain_phase(bar(L::kBarQFull + 2 * b + i), (n - 1) & 1, limit);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA warp
    ptx::setmaxnreg_dec<kRegsOther>();
    {   // The whole warp runs the loop, so its state stays warp-uniform; one elected
        // lane issues every MMA and commit.
      constexpr uint32_t kIdescS = make_idesc(kBlockM, kBlockN, false, kF16);
      constexpr uint32_t kIdescPV = make_idesc(kBlockM, HD, true, kF16);
      // Descriptors of the first operand blocks; later blocks differ only in the
      // start-address field (bits 0..13, address >> 4), which never carries over.
      const uint64_t desc_q0 = sw128_desc(sbase + L::kOffQ, 16, 1024);
      const uint64_t desc_kv0 = sw128_desc(sbase + L::kOffKV, 16, 1024);
      const uint64_t desc_v0 = sw128_desc(sbase + L::kOffKV, L::kRegionBytes, 1024);
      uint32_t q_count[2] = {0, 0};   // units in which tile i was present (o_empty phase)
      uint32_t q_pos = 0;             // Q ring position of the next unit's first tile (kQRing)
      // Buffer of Q_i in the current unit and the phase of its q_full (the number of
      // earlier loads into it): ring positions in load order (kQRing), else buffer
      // 2b + i with b alternating between units when kQBufs = 2.
      int qb[2] = {0, 1};
      uint32_t qp[2] = {0, 0};
      auto set_q = [&](const int* nb) {
        if constexpr (L::kQRing) {
          uint32_t pos = q_pos;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (nb[i] > 0) {
              qb[i] = static_cast<int>(pos % 3u);
              qp[i] = (pos / 3u) & 1u;
              ++pos;
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            qb[i] = 2 * (L::kQBufs == 2 ? static_cast<int>(q_count[i] & 1u) : 0) + i;
            qp[i] = (L::kQBufs == 2 ? (q_count[i] >> 1) : q_count[i]) & 1u;
          }
        }
      };
      auto q_buf = [&](int i) -> int { return qb[i]; };
      auto q_phase = [&](int i) -> uint32_t { return qp[i]; };
      auto issue_s = [&](int i, int slot) {
        const uint64_t a = desc_q0 + ((q_buf(i) * L::kTileBytes) >> 4);
        const uint64_t b = desc_kv0 + ((slot * L::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kRegionBytes + (kk & 3) * 32) >> 4;
          ptx::mma_ss_warp(tmem + L::col_s(i), a + off, b + off, kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      // P_i V over K-slices [k0, k1) (16 keys each)
      auto issue_pv_part = [&](int i, int slot, bool accumulate, int k0, int k1) {
        const uint64_t b = desc_v0 + ((slot * L::kTileBytes) >> 4);
#pragma unroll
        for (int kk = k0; kk < k1; ++kk) {
          ptx::mma_ts_warp(tmem + L::col_o(i), tmem + L::col_p(i) + kk * 8, b + ((kk * 16 * 128) >> 4),
                      kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int i, int slot, bool accumulate) { issue_pv_part(i, slot, accumulate, 0, kBlockN / 16); };
      uint32_t p_base[2] = {0, 0};    // S_i tiles of earlier units (p_full phase)
      uint32_t it_base = 0;           // K/V ring position of this unit's K_0
      bool ok = true;
      Unit u;
      if constexpr (L::kDecoupled) {
        // Per key tile j: first the S GEMMs of key tile j+1 (each as soon as the
        // softmax has read the tile's previous S), then the P V GEMMs of key tile j.
        uint32_t s_iss[2] = {0, 0};   // S_i GEMMs issued so far (s_free phase)
        for (int r = 0; ok && unit_at(r, u); ++r) {
          if (kBand && u.nmax == 0) continue;   // no keys at all (key padding): nothing to issue
          const int nblk[2] = {u.nblk[0], u.nblk[1]};
          const int nmax = u.nmax;
          const int fst[2] = {0, kBand ? u.first[1] : 0};
          set_q(nblk);
#pragma unroll
          for (int i = 0; i < 2; ++i)
            if (ok && nblk[i] > 0)
              ok = wait_warp(bar(L::kBarQFull + q_buf(i)), q_phase(i), abort_flag, limit, kSiteMmaQ);
          const int slot_k0 = it_base % L::kStages;
          if (ok) ok = wait_warp(bar(L::kBarKVFull + slot_k0), (it_base / L::kStages) & 1,
                                  abort_flag, limit, kSiteMmaK);
          if (!ok) break;
          ptx::tc_fence_after();
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (nblk[i] > 0 && fst[i] == 0) {   // S_i of the unit's first key tile
              issue_s(i, slot_k0);
              ptx::mma_commit_warp(bar(L::kBarSFull + i));
              ++s_iss[i];
              if (nblk[i] == 1) ptx::mma_commit_warp(bar(L::kBarQEmpty + q_buf(i)));
            }
          }
          ptx::mma_commit_warp(bar(L::kBarKVEmpty + slot_k0));
          for (int j = 0; j < nmax && ok; ++j) {
            const uint32_t it_v = it_base + 2 * j + 1;
            const int slot_v = it_v % L::kStages;
            const uint32_t it_k = it_v + 1;
            const int slot_k = it_k % L::kStages;
            bool k_ready = false;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int t = j + 1 - fst[i];   // tile i's step that key tile j+1 is
              if (t < 0 || t >= nblk[i]) continue;
              if (t > 0) {   // S_i(t-1) must have left TMEM
                if (!wait_warp(bar(L::kBarSFree + i), (s_iss[i] - 1) & 1, abort_flag, limit,
                                kSiteMmaSFree)) {
                  ok = false;
                  break;
                }
              }
              if (!k_ready) {
                if (!wait_warp(bar(L::kBarKVFull + slot_k), (it_k / L::kStages) & 1, abort_flag,
                                limit, kSiteMmaK)) {
                  ok = false;
                  break;
                }
                k_ready = true;
              }
              ptx::tc_fence_after();
              issue_s(i, slot_k);
              ptx::mma_commit_warp(bar(L::kBarSFull + i));
              ++s_iss[i];
              if (t == nblk[i] - 1) ptx::mma_commit_warp(bar(L::kBarQEmpty + q_buf(i)));   // Q_i read for the last time
            }
            if (!ok) break;
            if (k_ready) ptx::mma_commit_warp(bar(L::kBarKVEmpty + slot_k));
            if (!wait_warp(bar(L::kBarKVFull + slot_v), (it_v / L::kStages) & 1, abort_flag, limit,
                            kSiteMmaV)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int jl = j - fst[i];
              if (jl < 0 || jl >= nblk[i]) continue;
              // The first P_i V MMA of a unit overwrites O_i: the previous epilogue must
              // have read it.
              if (jl == 0 && q_count[i] > 0 &&
                  !wait_warp(bar(L::kBarOEmpty + i), (q_count[i] - 1) & 1, abort_flag, limit,
                              kSiteMmaP)) {
                ok = false;
                break;
              }
              if (!wait_warp(bar(L::kBarPFull + i), (p_base[i] + jl) & 1, abort_flag, limit,
                              kSiteMmaP)) {
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              issue_pv(i, slot_v, jl > 0);
              ptx::mma_commit_warp(bar(L::kBarPVDone + i));
              if (jl == nblk[i] - 1) ptx::mma_commit_warp(bar(L::kBarOFull + i));
            }
            if (!ok) break;
            ptx::mma_commit_warp(bar(L::kBarKVEmpty + slot_v));
          }
          it_base += 2 * nmax;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            p_base[i] += nblk[i];
            if (nblk[i] > 0) ++q_count[i];
          }
          if constexpr (L::kQRing) q_pos += (nblk[0] > 0 ? 1u : 0u) + (nblk[1] > 0 ? 1u : 0u);
        }
      }
      for (int r = 0; !L::kDecoupled && ok && unit_at(r, u); ++r) {
        if (kBand && u.nmax == 0) continue;   // no keys at all (key padding): nothing to issue
        const int nb0 = u.nblk[0], nb1 = u.nblk[1], nmax = u.nmax;
        const int nblk[2] = {nb0, nb1};
        set_q(nblk);
        // Step j of the unit (key tile kv0 + j) is step j - fst[i] of query tile i.
        const int fst[2] = {0, kBand ? u.first[1] : 0};
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (ok && nblk[i] > 0)
            ok = wait_warp(bar(L::kBarQFull + q_buf(i)), q_phase(i), abort_flag, limit, kSiteMmaQ);
        const int slot_k0 = it_base % L::kStages;
        if (ok) ok = wait_warp(bar(L::kBarKVFull + slot_k0), (it_base / L::kStages) & 1,
                                abort_flag, limit, kSiteMmaK);
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (nblk[i] > 0 && fst[i] == 0) {
            issue_s(i, slot_k0);
            ptx::mma_commit_warp(bar(L::kBarSFull + i));
            if (nblk[i] == 1) ptx::mma_commit_warp(bar(L::kBarQEmpty + q_buf(i)));
          }
        }
        ptx::mma_commit_warp(bar(L::kBarKVEmpty + slot_k0));
        // The first P_i V MMA of a unit overwrites O_i: the previous unit's epilogue
        // must have read it.
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (ok && nblk[i] > 0 && q_count[i] > 0)
            ok = wait_warp(bar(L::kBarOEmpty + i), (q_count[i] - 1) & 1, abort_flag, limit,
                            kSiteMmaP);
        for (int j = 0; j < nmax && ok; ++j) {
          const uint32_t it_v = it_base + 2 * j + 1;
          const int slot_v = it_v % L::kStages;
          if (!wait_warp(bar(L::kBarKVFull + slot_v), (it_v / L::kStages) & 1, abort_flag, limit,
                          kSiteMmaV)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t it_k = it_v + 1;
          const int slot_k = it_k % L::kStages;
          bool k_ready = false;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int jl = j - fst[i];
            if (jl < 0 || jl >= nblk[i]) continue;
            if (!wait_warp(bar(L::kBarPFull + i), (p_base[i] + jl) & 1, abort_flag, limit,
                            kSiteMmaP)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            issue_pv_part(i, slot_v, jl > 0, 0, kBlockN / 32);   // first half of P_i
            if (!wait_warp(bar(L::kBarPHalf + i), (p_base[i] + jl) & 1, abort_flag, limit,
                            kSiteMmaP)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            issue_pv_part(i, slot_v, true, kBlockN / 32, kBlockN / 16);
            if (jl == nblk[i] - 1) {
              ptx::mma_commit_warp(bar(L::kBarOFull + i));
              if (nblk[i] > 1) ptx::mma_commit_warp(bar(L::kBarQEmpty + q_buf(i)));   // Q_i no longer read
            }
            if (jl + 1 < nblk[i]) {
              if (!k_ready) {
                if (!wait_warp(bar(L::kBarKVFull + slot_k), (it_k / L::kStages) & 1, abort_flag,
                                limit, kSiteMmaK)) {
                  ok = false;
                  break;
                }
                ptx::tc_fence_after();
                k_ready = true;
              }
              issue_s(i, slot_k);
              ptx::mma_commit_warp(bar(L::kBarSFull + i));
            }
          }
          if constexpr (kBand) {
            // A query tile whose band starts at the next key tile: its first S GEMM.
            if (ok && nblk[1] > 0 && fst[1] == j + 1) {
              if (!k_ready) {
                if (!wait_warp(bar(L::kBarKVFull + slot_k), (it_k / L::kStages) & 1, abort_flag,
                                limit, kSiteMmaK)) {
                  ok = false;
                } else {
                  ptx::tc_fence_after();
                  k_ready = true;
                }
              }
              if (ok) {
                issue_s(1, slot_k);
                ptx::mma_commit_warp(bar(L::kBarSFull + 1));
                if (nblk[1] == 1) ptx::mma_commit_warp(bar(L::kBarQEmpty + q_buf(1)));
              }
            }
          }
          if (!ok) break;
          ptx::mma_commit_warp(bar(L::kBarKVEmpty + slot_v));
          if (k_ready) ptx::mma_commit_warp(bar(L::kBarKVEmpty + slot_k));
        }
        it_base += 2 * nmax;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          p_base[i] += nblk[i];
          if (nblk[i] > 0) ++q_count[i];
        }
        if constexpr (L::kQRing) q_pos += (nblk[0] > 0 ? 1u : 0u) + (nblk[1] > 0 ? 1u : 0u);
      }
      // Drain: every MMA issued has completed before TMEM is freed.
      ptx::mma_commit_warp(bar(L::kBarDrain));
      drain_phase(bar(L::kBarDrain), 0, limit);
    }
    __syncwarp();
  } else {
    ptx::setmaxnreg_dec<kRegsOther>();   // the two spare warps of the load/MMA warpgroup
  }

  // The epilogue's TMA stores (D = 64) must be complete before the CTA exits.
  if (L::kTmaStoreO && warp < 8 && (threadIdx.x & 127) == 0) ptx::bulk_wait_all();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::kTmemCols);
  }
}

// Parameters of the combine kernel that finishes split units (split schedule).
struct CombineParams {
  const float* ws_o;
  const float* ws_ml;
  uint16_t* o;
  long long o_sb, o_sh, o_sl;
  int H;
  float* lse;
  long long total_steps;
  int unit_cost;     // virtual steps in front of each unit (as in Params)
  int grid;          // CTAs of the attention kernel that made the parts
  int nkv;
  int n_pairs;
  int bh_count;
  int Lq;
  int causal;
};

// One CTA per (CTA boundary of the attention kernel, query tile, group of 16
// rows).  The boundary that is the first one inside a unit finishes that unit:
// for each row it merges the unit's parts k in one pass, the same update the
// online softmax applies per key tile:
//   m' = max(m, m_k),  l' = l 2^(m - m') + l_k 2^(m_k - m'),
//   O' = O 2^(m - m') + O_k 2^(m_k - m'),
// and writes O = O'/l' and LSE = ln2 (m' + log2 l').  Each warp merges 4 rows,
// interleaved so their loads overlap; its lanes cover the D columns.
constexpr int kCombineRowsPerWarp = 4;
constexpr int kCombineRows = 4 * kCombineRowsPerWarp;   // rows per CTA (4 warps)
constexpr int kCombineMaxParts = 256;                   // parts come from distinct CTAs

template <int HD, bool kF16>
__global__ void __launch_bounds__(128) fa_combine_kernel(const __grid_constant__ CombineParams c) {
  __shared__ int s_slot[kCombineMaxParts];
  __shared__ int s_nparts, s_bh, s_q0;
  const int b = blockIdx.x + 1;   // boundary between CTA b-1 and CTA b
  const int tile = blockIdx.y;
  // Which parts this CTA merges follows from the launch's sizes alone: found while the
  // attention kernel ahead may still be running (under a dependent launch).
  if (threadIdx.x == 0) {
    const long long G = c.grid;
    auto lo = [&](long long g) { return c.total_steps * g / G; };
    const long long xb = lo(b);
    int bh, pair;
    long long step0, steps;
    split_locate(xb, c.nkv, c.Lq, c.n_pairs, c.causal, c.unit_cost, &bh, &pair, &step0, &steps);
    const long long ks = step0 + c.unit_cost, ke = ks + steps;   // the unit's key-tile steps
    int n = 0;
    // Nothing to do unless this boundary cuts the unit's key tiles and no earlier one does.
    // The unit's parts are those of CTA b-1 (its first part when nothing precedes the unit
    // in its range) and of the CTAs after it whose ranges start inside the unit.
    if (xb > ks && !(b >= 2 && lo(b - 1) > ks)) {
      for (long long g = b - 1; g < G && lo(g) < ke && n < kCombineMaxParts; ++g)
        s_slot[n++] = static_cast<int>(2 * g + (lo(g) >= step0 ? 0 : 1));
    }
    s_nparts = n;
    s_bh = bh;
    s_q0 = pair * 2 * kBlockM + tile * kBlockM;
  }
  __syncthreads();
  // The parts come from the attention kernel ahead.  Every CTA waits for it, even one with
  // nothing to merge, so that this kernel's completion implies that kernel's.  A dependent
  // launch after this one may start its set-up now (it waits for this kernel in turn).
  ptx::grid_dependency_wait();
  ptx::grid_launch_dependents();
  const int nparts = s_nparts;
  if (nparts == 0 || s_q0 >= c.Lq) return;
  constexpr int kPerLane = HD / 32;   // 4 (D = 128) or 2 (D = 64) columns per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.z * kCombineRows + warp * kCombineRowsPerWarp;
  float m[kCombineRowsPerWarp], l[kCombineRowsPerWarp], acc[kCombineRowsPerWarp][kPerLane];
#pragma unroll
  for (int rr = 0; rr < kCombineRowsPerWarp; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.0f;
#pragma unroll
    for (int e = 0; e < kPerLane; ++e) acc[rr][e] = 0.0f;
  }
  for (int k = 0; k < nparts; ++k) {
    const size_t base = static_cast<size_t>(s_slot[k] * 2 + tile) * kBlockM + r0;
#pragma unroll
    for (int rr = 0; rr < kCombineRowsPerWarp; ++rr) {
      const size_t row = base + rr;
      const float2 ml = __ldg(reinterpret_cast<const float2*>(c.ws_ml) + row);
      const float* src = c.ws_o + row * HD + lane * kPerLane;
      float x[kPerLane];
      if constexpr (kPerLane == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(src));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
      } else {
        const float2 v = __ldg(reinterpret_cast<const float2*>(src));
        x[0] = v.x; x[1] = v.y;
      }
      const float m_new = fmaxf(m[rr], ml.x);
      if (m_new == -INFINITY) continue;   // no key of this row so far (an empty part)
      const float a = ptx::ex2_approx(m[rr] - m_new);   // 0 on the first part (m = -inf)
      const float w = ptx::ex2_approx(ml.x - m_new);
      l[rr] = l[rr] * a + ml.y * w;
#pragma unroll
      for (int e = 0; e < kPerLane; ++e) acc[rr][e] = acc[rr][e] * a + x[e] * w;
      m[rr] = m_new;
    }
  }
#pragma unroll
  for (int rr = 0; rr < kCombineRowsPerWarp; ++rr) {
    const int q = s_q0 + r0 + rr;
    if (q >= c.Lq) continue;
    const float inv_l = 1.0f / l[rr];
    const int ob = s_bh / c.H, oh = s_bh - ob * c.H;
    uint16_t* dst = c.o + ob * c.o_sb + oh * c.o_sh + static_cast<long long>(q) * c.o_sl + lane * kPerLane;
    if constexpr (kPerLane == 4) {
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(pack2<kF16>(acc[rr][0] * inv_l, acc[rr][1] * inv_l),
                     pack2<kF16>(acc[rr][2] * inv_l, acc[rr][3] * inv_l));
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack2<kF16>(acc[rr][0] * inv_l, acc[rr][1] * inv_l);
    }
    if (lane == 0)
      c.lse[static_cast<size_t>(s_bh) * c.Lq + q] = (m[rr] + log2f(l[rr])) * 0.69314718055994531f;
  }
}

}  // namespace fa

// ============================================================================ host side
namespace {

using fa::Params;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  bool attr[2][5][2] = {};   // [D == 128][schedule][fp16]: shared-memory opt-in done
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<unsigned> g_debug_flags{0};
std::atomic<unsigned long long> g_wait_limit_ns{0};

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return na && nb && pa < pb + nb && pb < pa + na;
}

// The attention kernel instance for head dimension D, schedule `sched` (fa::Sched) and
// element type (bf16, or fp16 with f16).
using KernelFn = void (*)(const Params);
template <bool kF16>
KernelFn attention_kernel_t(int D, int sched) {
  if (D == 64)
    return sched == fa::kSchedBand        ? fa::fa_fwd_kernel<64, fa::kSchedBand, kF16>
           : sched == fa::kSchedSplit     ? fa::fa_fwd_kernel<64, fa::kSchedSplit, kF16>
           : sched == fa::kSchedWholeList ? fa::fa_fwd_kernel<64, fa::kSchedWholeList, kF16>
                                          : fa::fa_fwd_kernel<64, fa::kSchedWhole, kF16>;
  return sched == fa::kSchedBand    ? fa::fa_fwd_kernel<128, fa::kSchedBand, kF16>
         : sched == fa::kSchedSplit ? fa::fa_fwd_kernel<128, fa::kSchedSplit, kF16>
                                    : fa::fa_fwd_kernel<128, fa::kSchedWhole, kF16>;
}
KernelFn attention_kernel(int D, int sched, bool f16) {
  return f16 ? attention_kernel_t<true>(D, sched) : attention_kernel_t<false>(D, sched);
}
using TableKernelFn = void (*)(const fa::TableParams);
TableKernelFn table_kernel(int D, bool f16) {
  if (D == 64)
    return f16 ? fa::fa_fwd_kernel<64, fa::kSchedTable, true> : fa::fa_fwd_kernel<64, fa::kSchedTable, false>;
  return f16 ? fa::fa_fwd_kernel<128, fa::kSchedTable, true> : fa::fa_fwd_kernel<128, fa::kSchedTable, false>;
}

// Shared-memory opt-in for one kernel instance, and a check that the registers it
// is launched with cover the warpgroups' register split (setmaxnreg.inc would
// otherwise wait forever for registers that do not exist).
template <class Fn>
fa_status configure_kernel(Fn kernel, int smem_bytes) {
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, kernel) != cudaSuccess) return FA_ERR_CUDA;
  const long long launched = static_cast<long long>(attr.numRegs) * fa::kThreads;
  const long long split = 256ll * fa::kRegsSoftmax + 128ll * fa::kRegsOther;
  if (launched < split) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Per-device set-up: capability check, kernel attributes, encoder entry point.
// On success *sm_count holds the device's number of SMs.
fa_status prepare_device(int dev, int D, int* sm_count, bool f16 = false) {
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& info = g_devices[dev];
  if (!info.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    info.supported = (major == 10 && minor == 3);
    info.ready = true;
  }
  if (!info.supported) return FA_ERR_UNSUPPORTED;
  *sm_count = info.sm_count;
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return FA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const int di = (D == 128) ? 1 : 0, ti = f16 ? 1 : 0;
  for (int sc = 0; sc < 5; ++sc) {
    if (info.attr[di][sc][ti]) continue;
    const int smem = D == 64 ? fa::Layout<64>::kAlloc : fa::Layout<128>::kAlloc;
    const fa_status st = sc == fa::kSchedTable ? configure_kernel(table_kernel(D, f16), smem)
                                               : configure_kernel(attention_kernel(D, sc, f16), smem);
    if (st != FA_OK) return st;
    info.attr[di][sc][ti] = true;
  }
  return FA_OK;
}

// 4-D tensor map [B][H][L][D] over a tensor with element strides st = {batch, head, row}
// (features contiguous); box = 64 features x 128 rows x 1 head x 1 batch.  A size-1
// dimension's stride is never used to address anything and is replaced by a valid one.
bool encode_map(CUtensorMap* map, const void* base, long long B, long long H, long long L, int D,
                const long long* st, bool f16) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  const long long row = L > 1 ? st[2] : D;
  const long long head = H > 1 ? st[1] : row * L;
  const long long batch = B > 1 ? st[0] : head * H;
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(row) * 2, static_cast<cuuint64_t>(head) * 2,
                           static_cast<cuuint64_t>(batch) * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estrides[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              4, const_cast<void*>(base), dims, strides, box, estrides,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

namespace {

// A validated problem (argument checks shared by every entry point).
struct Problem {
  const void* Q;
  const void* K;
  const void* V;
  void* O;
  float* LSE;
  int Lq, Lk, D, causal;
  float scale;
  long long bh;
  int n_pairs, n_units, nkv;
  size_t bytes_q, bytes_k, bytes_lse;
  bool band = false;     // local attention over the band below (fa_fwd_window)
  int win_left = -1;     // key j allowed for row i iff i - win_left <= j <= i + win_right
  int win_right = -1;    //   (-1: unbounded side)
  bool f16 = false;      // fp16 instead of bf16 inputs and output
  const int* kv_len = nullptr;   // per-batch valid keys (device), band schedule only
  int B = 0, H = 0;
  long long qs[3] = {0, 0, 0}, ks[3] = {0, 0, 0}, vs[3] = {0, 0, 0}, os[3] = {0, 0, 0};   // element strides {batch, head, row}
};

// Contiguous [B,H,L,D] strides.
void contiguous_strides(long long H, long long L, int D, long long* st) {
  st[2] = D;
  st[1] = L * D;
  st[0] = H * L * D;
}

// FA_OK with *empty = true means there is nothing to compute (no launch).
fa_status check_problem(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                        int H, int Lq, int Lk, int D, int causal, float scale, Problem* pr,
                        bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  const long long rows_q = bh * Lq;
  if (rows_q == 0) {
    *empty = true;
    return FA_OK;
  }
  if (Lk < 1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  const uintptr_t align_bits = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                               reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O) |
                               reinterpret_cast<uintptr_t>(LSE);
  if (align_bits & 15u) return FA_ERR_INVALID_ARG;
  const long long elems_q = rows_q * D, elems_k = bh * Lk * D;
  if (elems_q > (1ll << 40) || elems_k > (1ll << 40)) return FA_ERR_INVALID_ARG;
  const size_t bytes_q = static_cast<size_t>(elems_q) * 2, bytes_k = static_cast<size_t>(elems_k) * 2;
  const size_t bytes_lse = static_cast<size_t>(rows_q) * 4;
  if (overlaps(O, bytes_q, Q, bytes_q) || overlaps(O, bytes_q, K, bytes_k) ||
      overlaps(O, bytes_q, V, bytes_k) || overlaps(O, bytes_q, LSE, bytes_lse) ||
      overlaps(LSE, bytes_lse, Q, bytes_q) || overlaps(LSE, bytes_lse, K, bytes_k) ||
      overlaps(LSE, bytes_lse, V, bytes_k))
    return FA_ERR_INVALID_ARG;
  const long long n_pairs = (Lq + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM);
  if (bh > INT_MAX || n_pairs * bh > INT_MAX) return FA_ERR_INVALID_ARG;
  *pr = Problem{Q, K, V, O, LSE, Lq, Lk, D, causal ? 1 : 0, scale, bh,
                static_cast<int>(n_pairs), static_cast<int>(n_pairs * bh),
                (Lk + fa::kBlockN - 1) / fa::kBlockN, bytes_q, bytes_k, bytes_lse};
  pr->B = B;
  pr->H = H;
  contiguous_strides(H, Lq, D, pr->qs);
  contiguous_strides(H, Lk, D, pr->ks);
  contiguous_strides(H, Lk, D, pr->vs);
  contiguous_strides(H, Lq, D, pr->os);
  return FA_OK;
}

// Schedule choice.  Causal units have different costs and are balanced by the
// heaviest-first boustrophedon order (or the host-computed table order); only when
// the longest unit dwarfs an even share are their key ranges split (see below).
// Non-causal units all cost the same; when
// whole units would keep at most half of the SM-rounds busy (a quarter for D = 64,
// whose parts are cheaper to compute and so relatively dearer to merge) and a unit
// has at least two key tiles, the key ranges are split across CTAs (needs a
// workspace).  The thresholds come from measurements: splitting paid 3.1-3.6x at
// 21 % fill and 61 % at 42 % fill (D = 128), and lost 9-36 % at 84 % fill.
struct Plan {
  bool split;
  bool band;
  int grid;
  size_t off_ml, ws_bytes;
};

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Key-tile steps of all units in the split schedule's step space.
// Virtual steps in front of each unit of the split step space: what a part costs besides
// its key tiles (its Q loads, first S and parked rows took about four key-tile steps in a
// trace of one long causal head), so that ranges holding many short units carry fewer key
// tiles.  Causal units differ in length and the short ones gather in a few ranges; measured
// side by side, 5 at D = 128 and 3 at D = 64 ran 15-23 % faster than no cost on one to four
// long causal heads (higher and lower values slower).  Non-causal units are all alike and
// take none (a cost measured 0-1 % slower there).
int split_unit_cost(const Problem& pr) { return pr.causal ? (pr.D == 128 ? 5 : 3) : 0; }

// Steps of all units in the split schedule's step space, `cost` virtual steps per unit
// included (0: key-tile steps only).
long long split_total_steps(const Problem& pr, int cost) {
  return pr.bh * fa::head_prefix(pr.n_pairs, pr.nkv, pr.Lq, pr.n_pairs, pr.causal, cost);
}

// The most parts any CTA of a split launch with `grid` CTAs takes: the units whose key tiles
// meet its step range [T g / G, T (g + 1) / G) (the kernel's own division of the step space).
int split_max_parts(const Problem& pr, int grid, int cost) {
  const long long T = split_total_steps(pr, cost);
  // Every unit takes at least 1 + cost steps, so a range of R steps meets at most
  // R / (1 + cost) + 2 of them; when that bound is small enough the walk below is skipped.
  const long long range = (T + grid - 1) / grid;
  const long long bound = range / (1 + cost) + 2;
  if (bound <= fa::Layout<128>::kMaxParts) return static_cast<int>(bound);
  long long most = 0;
  for (int g = 0; g < grid; ++g) {
    const long long a = T * g / grid, b = T * (g + 1) / grid;
    long long n = 0;
    for (long long x = a; x < b;) {
      int bh, pair;
      long long start, steps;
      fa::split_locate(x, pr.nkv, pr.Lq, pr.n_pairs, pr.causal, cost, &bh, &pair, &start, &steps);
      const long long ks = start + cost, ke = ks + steps;
      if (std::max(x, ks) < std::min(ke, b)) ++n;
      x = std::min(ke, b);
    }
    most = std::max(most, n);
  }
  return static_cast<int>(std::min<long long>(most, INT_MAX));
}

Plan plan_schedule(const Problem& pr, int sm_count) {
  Plan pl{};
  const long long rounds = (pr.n_units + sm_count - 1) / sm_count;
  const double fill = static_cast<double>(pr.n_units) / (static_cast<double>(rounds) * sm_count);
  if (!pr.causal) {
    // Cut key ranges when at most half of the last round of units would be filled
    // (measured side by side: at D = 64 a fill of 0.42 ran 80 % faster split; at D = 128 a
    // fill of 0.63 ran 1 % slower split).
    pl.split = pr.nkv >= 2 && fill <= 0.5;
  } else {
    // Causal units grow along the sequence; whole units finish no sooner than the longest
    // one.  When that unit is well above an even share of all steps (few heads, long
    // sequences), the key ranges are cut across CTAs as for the full mask.  Each part
    // reloads its Q tiles and parks fp32 partial rows, and a merge kernel follows, so the
    // split pays only when the longest unit is at least twice the share: measured side by
    // side, one or two heads of 16K-32K tokens (2.3-2.4x) ran 29-42 % faster split and four
    // heads of 8K (2.3x) 10 %, while shapes at 1.6-1.8x ran 6-9 % slower.  Short sequences
    // (units under 16 key tiles) and problems under two steps per SM stay whole.
    const long long longest = fa::pair_steps(pr.n_pairs - 1, pr.nkv, pr.Lq, 1);
    const long long total = split_total_steps(pr, 0);
    const double share = static_cast<double>(total) / sm_count;
    pl.split = longest >= 16 && total >= 2ll * sm_count && static_cast<double>(longest) >= 2.0 * share;
  }
  if (!pl.split) {
    pl.grid = std::min(pr.n_units, sm_count);
    return pl;
  }
  const long long steps = split_total_steps(pr, 0);
  pl.grid = static_cast<int>(std::min<long long>(steps, sm_count));
  // Each CTA lists its parts in shared memory (at most kMaxParts); a problem whose step
  // ranges would cut more units than that (many tiny causal units in one range) keeps
  // whole units.
  if (split_max_parts(pr, pl.grid, split_unit_cost(pr)) > fa::Layout<128>::kMaxParts) {
    pl.split = false;
    pl.grid = std::min(pr.n_units, sm_count);
    return pl;
  }
  const size_t rows = static_cast<size_t>(pl.grid) * 2 * 2 * fa::kBlockM;   // 2 slots x 2 tiles
  pl.off_ml = round256(rows * pr.D * sizeof(float));
  pl.ws_bytes = pl.off_ml + round256(rows * 2 * sizeof(float));
  return pl;
}

// ---------------------------------------------------------------- schedule table (kSchedTable)
// Causal units are dealt heaviest first so the CTAs finish together; with the formula order
// (all heads' last query tiles first) every head's K/V is in flight at once, and K/V tiles
// leave the L2 cache between the units of a head that read them (DRAM reads measured at
// 2.6x the compulsory bytes at 4K tokens, 64 heads).  When the heads' K/V outgrow the L2,
// the host orders the units instead: heads in groups whose K/V take about 32 MiB, group
// after group, each group's units heaviest first, each unit to the CTA with the least work
// so far (greedy longest-processing-time).  The per-CTA lists go to the kernel with the
// launch.  A one-entry cache per device keeps the last table.
constexpr long long kTableGroupBytes = 32ll << 20;   // K/V bytes of one head group
constexpr long long kTableMinBytes = 48ll << 20;     // below this the heads' K/V stay in L2

bool table_eligible(const Problem& pr, const Plan& pl) {
  if (pl.split || pl.band || !pr.causal || (g_debug_flags.load() & 16u)) return false;
  const long long kv_head = 4ll * pr.Lk * pr.D;   // K and V bytes of one head (16-bit elements)
  return pr.n_units <= fa::kTabMaxUnits && pl.grid <= fa::kTabMaxGrid && pr.n_pairs <= 4096 &&
         pr.bh < (1ll << 20) && pr.bh * kv_head > kTableMinBytes;
}

struct TableCache {
  bool valid = false;
  long long bh = 0;
  int Lq = 0, Lk = 0, D = 0, grid = 0;
  std::vector<uint16_t> off;
  std::vector<uint32_t> units;
};
std::mutex g_table_mutex;
TableCache g_table_cache[kMaxDevices];

void build_table(const Problem& pr, int G, TableCache& tc) {
  const long long kv_head = 4ll * pr.Lk * pr.D;
  const long long group = std::max(1ll, kTableGroupBytes / kv_head);
  std::vector<std::vector<uint32_t>> lists(G);
  using Load = std::pair<long long, int>;   // (work so far, CTA): least work first, then lowest index
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int g = 0; g < G; ++g) heap.push({0, g});
  for (long long h0 = 0; h0 < pr.bh; h0 += group) {
    const long long h1 = std::min(pr.bh, h0 + group);
    for (int pair = pr.n_pairs - 1; pair >= 0; --pair) {
      // Cost: key tiles of the pair's two query tiles, plus two for the unit's fill and drain.
      const int q0 = pair * 2 * fa::kBlockM;
      const int n0 = std::min(pr.nkv, q0 / fa::kBlockN + 1);
      const int n1 = q0 + fa::kBlockM >= pr.Lq ? 0 : std::min(pr.nkv, (q0 + fa::kBlockM) / fa::kBlockN + 1);
      const long long cost = n0 + n1 + 2;
      for (long long h = h0; h < h1; ++h) {
        const Load least = heap.top();
        heap.pop();
        lists[least.second].push_back(static_cast<uint32_t>((h << 12) | pair));
        heap.push({least.first + cost, least.second});
      }
    }
  }
  tc.off.assign(G + 1, 0);
  tc.units.clear();
  for (int g = 0; g < G; ++g) {
    tc.off[g] = static_cast<uint16_t>(tc.units.size());
    tc.units.insert(tc.units.end(), lists[g].begin(), lists[g].end());
  }
  tc.off[G] = static_cast<uint16_t>(tc.units.size());
  tc.bh = pr.bh;
  tc.Lq = pr.Lq;
  tc.Lk = pr.Lk;
  tc.D = pr.D;
  tc.grid = G;
  tc.valid = true;
}

// Fills the table part of *tp for this problem (from the cache when it matches).
fa_status fill_table(const Problem& pr, int G, fa::TableParams* tp) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_table_mutex);
  TableCache& tc = g_table_cache[dev];
  if (!tc.valid || tc.bh != pr.bh || tc.Lq != pr.Lq || tc.Lk != pr.Lk || tc.D != pr.D || tc.grid != G)
    build_table(pr, G, tc);
  std::copy(tc.off.begin(), tc.off.end(), tp->tab_off);
  std::copy(tc.units.begin(), tc.units.end(), tp->tab_units);
  return FA_OK;
}

// allow_dependent = false keeps the kernel from starting before the operation ahead of it
// in the stream has completed (needed when that operation is an event wait, which a
// programmatic dependent launch does not order).
fa_status launch(const Problem& pr, int sm_count, const Plan& pl, void* ws, cudaStream_t stream,
                 bool allow_dependent = true) {
  Params p;
  if (!encode_map(&p.tm_q, pr.Q, pr.B, pr.H, pr.Lq, pr.D, pr.qs, pr.f16) ||
      !encode_map(&p.tm_k, pr.K, pr.B, pr.H, pr.Lk, pr.D, pr.ks, pr.f16) ||
      !encode_map(&p.tm_v, pr.V, pr.B, pr.H, pr.Lk, pr.D, pr.vs, pr.f16))
    return FA_ERR_CUDA;
  // D = 64 stores O through a tensor map as well (TMA stores from the epilogue's staging).
  if (pr.D == 64 ? !encode_map(&p.tm_o, pr.O, pr.B, pr.H, pr.Lq, pr.D, pr.os, pr.f16)
                 : (memset(&p.tm_o, 0, sizeof(p.tm_o)), false))
    return FA_ERR_CUDA;
  p.o = static_cast<uint16_t*>(pr.O);
  p.o_sb = pr.os[0];
  p.o_sh = pr.os[1];
  p.o_sl = pr.os[2];
  p.o_v8 = (reinterpret_cast<uintptr_t>(pr.O) % 32 == 0 && (pr.os[0] * 2) % 32 == 0 &&
            (pr.os[1] * 2) % 32 == 0 && (pr.os[2] * 2) % 32 == 0) ? 1 : 0;
  p.H = pr.H;
  p.lse = pr.LSE;
  p.bh_count = static_cast<int>(pr.bh);
  p.Lq = pr.Lq;
  p.Lk = pr.Lk;
  p.causal = pr.causal;
  p.n_pairs = pr.n_pairs;
  p.n_units = pr.n_units;
  p.nkv = pr.nkv;
  p.split = pl.split ? 1 : 0;
  p.win_left = pr.win_left;
  p.win_right = pr.win_right;
  // Heaviest units first: the last query tiles unless only the left side is bounded.
  p.band_desc = (pr.win_left >= 0 && pr.win_right < 0) ? 0 : 1;
  p.kv_len = pr.kv_len;
  p.unit_cost = split_unit_cost(pr);
  p.total_steps = split_total_steps(pr, p.unit_cost);
  p.ws_o = nullptr;
  p.ws_ml = nullptr;
  if (pl.split) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    p.ws_o = reinterpret_cast<float*>(base);
    p.ws_ml = reinterpret_cast<float*>(base + pl.off_ml);
  }
  p.scale_log2 = static_cast<float>(static_cast<double>(pr.scale) * 1.4426950408889634);
  p.flags = g_debug_flags.load();
  const unsigned long long lim = g_wait_limit_ns.load();
  p.wait_limit_ns = lim ? lim : fa::kDefaultWaitNs;
  if (p.flags & 2u) return FA_ERR_CUDA;   // test hook: simulated launch failure
  (void)sm_count;

  cudaLaunchConfig_t cfg = {};
  // Persistent launch: one CTA per SM (shared memory allows no more), each
  // walking its share of the work.
  cfg.gridDim = dim3(static_cast<unsigned>(pl.grid));
  cfg.blockDim = dim3(fa::kThreads);
  cfg.stream = stream;
  cfg.dynamicSmemBytes = (pr.D == 64) ? fa::Layout<64>::kAlloc : fa::Layout<128>::kAlloc;
  // Programmatic dependent launch for short kernels: the kernel's set-up may overlap the
  // previous kernel in the stream (it waits for it with griddepcontrol.wait before
  // touching memory), which hides the launch gap.  Used when a CTA's share of the work
  // is at most 256 key-tile steps (about a quarter of a millisecond): side by side it
  // gained 11-13 % on 1K-token D = 64 batches and 2 % on 4K causal, while on 16K causal
  // (about 430 steps per CTA) it gave 1620-1784 TFLOP/s against a steady 1761-1782.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  const long long steps_per_cta =
      static_cast<long long>(pr.n_units) * pr.nkv / std::max(1, pl.grid);
  const bool dependent_launch = steps_per_cta <= 256;
  cfg.attrs = attr;
  cfg.numAttrs = (dependent_launch && allow_dependent) ? 1 : 0;
  int sched = pl.band ? fa::kSchedBand : pl.split ? fa::kSchedSplit : fa::kSchedWhole;
  // D = 64 whole units read from a per-CTA list when it holds them all (bit-identical;
  // measured on 1K-token batches: +2.4 % with the full mask, +7 % causal).  The same list
  // left the D = 128 kernels unchanged and made the D = 64 table order 4 % slower.
  if (sched == fa::kSchedWhole && pr.D == 64 &&
      (pr.n_units + pl.grid - 1) / std::max(1, pl.grid) <= fa::Layout<64>::kMaxParts)
    sched = fa::kSchedWholeList;
  cudaError_t err;
  if (table_eligible(pr, pl)) {
    fa::TableParams tp;
    static_cast<Params&>(tp) = p;
    const fa_status ts = fill_table(pr, pl.grid, &tp);
    if (ts != FA_OK) return ts;
    err = cudaLaunchKernelEx(&cfg, table_kernel(pr.D, pr.f16), tp);
  } else {
    err = cudaLaunchKernelEx(&cfg, attention_kernel(pr.D, sched, pr.f16), p);
  }
  if (err != cudaSuccess) return FA_ERR_CUDA;
  if (pl.split && pl.grid > 1) {
    // Merge the parts of every split unit (same stream: runs after the parts exist).
    fa::CombineParams c;
    c.ws_o = p.ws_o;
    c.ws_ml = p.ws_ml;
    c.o = p.o;
    c.o_sb = p.o_sb;
    c.o_sh = p.o_sh;
    c.o_sl = p.o_sl;
    c.H = p.H;
    c.lse = p.lse;
    c.total_steps = p.total_steps;
    c.unit_cost = p.unit_cost;
    c.grid = pl.grid;
    c.nkv = pr.nkv;
    c.n_pairs = pr.n_pairs;
    c.bh_count = static_cast<int>(pr.bh);
    c.Lq = pr.Lq;
    c.causal = pr.causal;
    cudaLaunchConfig_t cc = {};
    cc.gridDim = dim3(static_cast<unsigned>(pl.grid - 1), 2, fa::kBlockM / fa::kCombineRows);
    cc.blockDim = dim3(128);
    cc.stream = stream;
    cc.attrs = attr;
    cc.numAttrs = dependent_launch ? 1 : 0;
    if (pr.f16)
      err = (pr.D == 64) ? cudaLaunchKernelEx(&cc, fa::fa_combine_kernel<64, true>, c)
                         : cudaLaunchKernelEx(&cc, fa::fa_combine_kernel<128, true>, c);
    else
      err = (pr.D == 64) ? cudaLaunchKernelEx(&cc, fa::fa_combine_kernel<64, false>, c)
                         : cudaLaunchKernelEx(&cc, fa::fa_combine_kernel<128, false>, c);
    if (err != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}

fa_status current_device(int D, int* sm_count) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  // Make the device's primary context current on this thread (a thread that has only
  // selected the device has none yet, and tensor-map encoding needs one).
  if (cudaSetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;
  return prepare_device(dev, D, sm_count);
}

}  // namespace

extern "C" fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            int B, int H, int Lq, int Lk, int D, int causal, float scale,
                            cudaStream_t stream) {
  Problem pr;
  bool empty = false;
  const fa_status st = check_problem(Q, K, V, O, LSE, B, H, Lq, Lk, D, causal, scale, &pr, &empty);
  if (st != FA_OK || empty) return st;
  int sm_count = 0;
  const fa_status prep = current_device(D, &sm_count);
  if (prep != FA_OK) return prep;
  Plan pl = plan_schedule(pr, sm_count);
  if (pl.split) {   // no workspace here: whole units only
    pl.split = false;
    pl.grid = std::min(pr.n_units, sm_count);
  }
  return launch(pr, sm_count, pl, nullptr, stream);
}

namespace {
// The problem fa_fwd_ws would plan, from sizes alone (no pointers).  *empty = true: no work.
fa_status sized_problem(int B, int H, int Lq, int Lk, int D, int causal, Problem* pr,
                        int* sm_count, bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  if (bh * Lq == 0) {
    *empty = true;
    return FA_OK;
  }
  if (Lk < 1) return FA_ERR_INVALID_ARG;
  const long long n_pairs = (Lq + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM);
  if (bh > INT_MAX || n_pairs * bh > INT_MAX) return FA_ERR_INVALID_ARG;
  const fa_status prep = current_device(D, sm_count);
  if (prep != FA_OK) return prep;
  *pr = Problem{};
  pr->Lq = Lq;
  pr->Lk = Lk;
  pr->D = D;
  pr->causal = causal ? 1 : 0;
  pr->bh = bh;
  pr->n_pairs = static_cast<int>(n_pairs);
  pr->n_units = static_cast<int>(n_pairs * bh);
  pr->nkv = (Lk + fa::kBlockN - 1) / fa::kBlockN;
  pr->B = B;
  pr->H = H;
  return FA_OK;
}
}  // namespace

extern "C" fa_status fa_fwd_workspace_size(int B, int H, int Lq, int Lk, int D, int causal,
                                           size_t* bytes) {
  if (!bytes) return FA_ERR_INVALID_ARG;
  *bytes = 0;
  Problem pr;
  int sm_count = 0;
  bool empty = false;
  const fa_status st = sized_problem(B, H, Lq, Lk, D, causal, &pr, &sm_count, &empty);
  if (st != FA_OK || empty) return st;
  const Plan pl = plan_schedule(pr, sm_count);
  *bytes = pl.split ? pl.ws_bytes : 0;
  return FA_OK;
}

extern "C" fa_status fa_fwd_schedule(int B, int H, int Lq, int Lk, int D, int causal,
                                     int* schedule) {
  if (!schedule) return FA_ERR_INVALID_ARG;
  *schedule = FA_SCHED_WHOLE;
  Problem pr;
  int sm_count = 0;
  bool empty = false;
  const fa_status st = sized_problem(B, H, Lq, Lk, D, causal, &pr, &sm_count, &empty);
  if (st != FA_OK || empty) return st;
  const Plan pl = plan_schedule(pr, sm_count);
  *schedule = pl.split ? FA_SCHED_SPLIT : table_eligible(pr, pl) ? FA_SCHED_TABLE : FA_SCHED_WHOLE;
  return FA_OK;
}

extern "C" fa_status fa_fwd_ws(const void* Q, const void* K, const void* V, void* O, float* LSE,
                               int B, int H, int Lq, int Lk, int D, int causal, float scale,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Problem pr;
  bool empty = false;
  const fa_status st = check_problem(Q, K, V, O, LSE, B, H, Lq, Lk, D, causal, scale, &pr, &empty);
  if (st != FA_OK || empty) return st;
  int sm_count = 0;
  const fa_status prep = current_device(D, &sm_count);
  if (prep != FA_OK) return prep;
  const Plan pl = plan_schedule(pr, sm_count);
  if (pl.split) {
    if (!workspace || workspace_bytes < pl.ws_bytes) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_INVALID_ARG;
    if (overlaps(workspace, pl.ws_bytes, Q, pr.bytes_q) ||
        overlaps(workspace, pl.ws_bytes, K, pr.bytes_k) ||
        overlaps(workspace, pl.ws_bytes, V, pr.bytes_k) ||
        overlaps(workspace, pl.ws_bytes, O, pr.bytes_q) ||
        overlaps(workspace, pl.ws_bytes, LSE, pr.bytes_lse))
      return FA_ERR_INVALID_ARG;
  }
  return launch(pr, sm_count, pl, workspace, stream);
}

extern "C" fa_status fa_fwd_window(const void* Q, const void* K, const void* V, void* O,
                                   float* LSE, int B, int H, int Lq, int Lk, int D,
                                   int window_left, int window_right, float scale,
                                   cudaStream_t stream) {
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  Problem pr;
  bool empty = false;
  const fa_status st = check_problem(Q, K, V, O, LSE, B, H, Lq, Lk, D, 0, scale, &pr, &empty);
  if (st != FA_OK || empty) return st;
  // A side of the band that reaches past every row's first or last key is unbounded.
  int left = window_left, right = window_right;
  if (left >= Lq - 1) left = -1;
  if (right >= Lk - 1) right = -1;
  // Every row needs an allowed key: the last row's band starts at Lq - 1 - left.
  if (left >= 0 && Lq - 1 - left > Lk - 1) return FA_ERR_INVALID_ARG;
  int sm_count = 0;
  const fa_status prep = current_device(D, &sm_count);
  if (prep != FA_OK) return prep;
  const bool force_band = (g_debug_flags.load() & 4u) != 0;
  if (!force_band && left < 0 && (right < 0 || right == 0)) {
    pr.causal = (right == 0) ? 1 : 0;   // the full or the causal mask: whole units
  } else {
    pr.band = true;
    pr.win_left = left;
    pr.win_right = right;
  }
  Plan pl{};
  pl.band = pr.band;
  pl.grid = std::min(pr.n_units, sm_count);
  return launch(pr, sm_count, pl, nullptr, stream);
}

// ---------------------------------------------------------------- strided / fp16 entry point
using fa_layout::no_self_overlap;
using fa_layout::span_bytes;
using fa_layout::strides_ok;

extern "C" fa_status fa_fwd_strided(const void* Q, const long long* q_stride, const void* K,
                                    const long long* k_stride, const void* V,
                                    const long long* v_stride, void* O, const long long* o_stride,
                                    float* LSE, const int* kv_len, int B, int H, int Lq, int Lk,
                                    int D, int window_left, int window_right, float scale,
                                    int dtype, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  if (bh * Lq == 0) return FA_OK;
  if (Lk < 1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.0f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (!Q || !K || !V || !O || !LSE || !q_stride || !k_stride || !v_stride || !o_stride)
    return FA_ERR_INVALID_ARG;
  const uintptr_t align_bits = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                               reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O) |
                               reinterpret_cast<uintptr_t>(LSE);
  if (align_bits & 15u) return FA_ERR_INVALID_ARG;
  if (!strides_ok(B, H, Lq, D, q_stride) || !strides_ok(B, H, Lk, D, k_stride) ||
      !strides_ok(B, H, Lk, D, v_stride) || !strides_ok(B, H, Lq, D, o_stride) ||
      !no_self_overlap(B, H, Lq, D, o_stride))
    return FA_ERR_INVALID_ARG;
  const long long n_pairs = (Lq + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM);
  if (bh > INT_MAX || n_pairs * bh > INT_MAX) return FA_ERR_INVALID_ARG;
  // Q, K and V may share memory (they are only read); O must not meet any input or the LSE.
  const size_t sq = span_bytes(B, H, Lq, D, q_stride), sk = span_bytes(B, H, Lk, D, k_stride);
  const size_t sv = span_bytes(B, H, Lk, D, v_stride), so = span_bytes(B, H, Lq, D, o_stride);
  const size_t sl = static_cast<size_t>(bh * Lq) * 4;
  if (overlaps(O, so, Q, sq) || overlaps(O, so, K, sk) || overlaps(O, so, V, sv) ||
      overlaps(O, so, LSE, sl) || overlaps(LSE, sl, Q, sq) || overlaps(LSE, sl, K, sk) ||
      overlaps(LSE, sl, V, sv))
    return FA_ERR_INVALID_ARG;
  int left = window_left, right = window_right;
  if (left >= Lq - 1) left = -1;
  if (right >= Lk - 1) right = -1;
  // A row without keys is an argument error, except with key padding, where lengths in
  // device memory can empty any row and such rows get O = 0, LSE = -inf.
  if (!kv_len && left >= 0 && Lq - 1 - left > Lk - 1) return FA_ERR_INVALID_ARG;
  if (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u)) return FA_ERR_INVALID_ARG;

  Problem pr{};
  pr.Q = Q;
  pr.K = K;
  pr.V = V;
  pr.O = O;
  pr.LSE = LSE;
  pr.Lq = Lq;
  pr.Lk = Lk;
  pr.D = D;
  pr.scale = scale;
  pr.bh = bh;
  pr.n_pairs = static_cast<int>(n_pairs);
  pr.n_units = static_cast<int>(n_pairs * bh);
  pr.nkv = (Lk + fa::kBlockN - 1) / fa::kBlockN;
  pr.B = B;
  pr.H = H;
  pr.f16 = dtype == FA_DTYPE_FP16;
  for (int i = 0; i < 3; ++i) {
    pr.qs[i] = q_stride[i];
    pr.ks[i] = k_stride[i];
    pr.vs[i] = v_stride[i];
    pr.os[i] = o_stride[i];
  }
  int sm_count = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaSetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;   // primary context current here
  const fa_status prep = prepare_device(dev, D, &sm_count, pr.f16);
  if (prep != FA_OK) return prep;
  const bool force_band = (g_debug_flags.load() & 4u) != 0;
  Plan pl{};
  pr.kv_len = kv_len;
  if (!kv_len && !force_band && left < 0 && (right < 0 || right == 0)) {
    pr.causal = (right == 0) ? 1 : 0;
    pl = plan_schedule(pr, sm_count);
    if (pl.split) {   // the split schedule only with a workspace that fits
      const bool ws_ok = workspace && workspace_bytes >= pl.ws_bytes &&
                         !(reinterpret_cast<uintptr_t>(workspace) & 255u) &&
                         !overlaps(workspace, pl.ws_bytes, Q, sq) &&
                         !overlaps(workspace, pl.ws_bytes, K, sk) &&
                         !overlaps(workspace, pl.ws_bytes, V, sv) &&
                         !overlaps(workspace, pl.ws_bytes, O, so) &&
                         !overlaps(workspace, pl.ws_bytes, LSE, sl);
      if (!ws_ok) {
        if (workspace) return FA_ERR_INVALID_ARG;   // given but unusable
        pl.split = false;
        pl.grid = std::min(pr.n_units, sm_count);
      }
    }
  } else {
    pr.band = true;
    pr.win_left = left;
    pr.win_right = right;
    pl.band = true;
    pl.grid = std::min(pr.n_units, sm_count);
  }
  return launch(pr, sm_count, pl, workspace, stream);
}

// ---------------------------------------------------------------- no-allocation entry point
// Scratch for fa_fwd_noalloc: the split schedule's workspace, held in device
// memory that the CUDA runtime reserves when this library's module is loaded on a
// GPU, so the call itself never allocates.  42 MiB covers the split schedule at
// D = 128 on up to 165 SMs (GB300 has 152) and at D = 64 on up to 325 SMs.
constexpr size_t kNoAllocScratchBytes = 42ull << 20;
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_fa_noalloc_scratch on device `dev` (which must be current).
// The name g_fa_noalloc_scratch in host code only stands in for the symbol; the
// address comes from cudaGetSymbolAddress, once per device.
fa_status scratch_address(int dev, void** addr) {
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_fa_noalloc_scratch) != cudaSuccess || !a) return FA_ERR_CUDA;
    g_scratch_addr[dev] = a;
  }
  *addr = g_scratch_addr[dev];
  return FA_OK;
}
}  // namespace

extern "C" fa_status fa_fwd_noalloc(const void* Q, const void* K, const void* V, void* O,
                                    float* LSE, int B, int H, int Lq, int Lk, int D, int causal,
                                    float scale, cudaStream_t stream) {
  Problem pr;
  bool empty = false;
  const fa_status st = check_problem(Q, K, V, O, LSE, B, H, Lq, Lk, D, causal, scale, &pr, &empty);
  if (st != FA_OK || empty) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaSetDevice(dev) != cudaSuccess) return FA_ERR_CUDA;   // primary context current here
  int sm_count = 0;
  const fa_status prep = prepare_device(dev, D, &sm_count);
  if (prep != FA_OK) return prep;
  const Plan pl = plan_schedule(pr, sm_count);
  if (!pl.split) return launch(pr, sm_count, pl, nullptr, stream);
  if (pl.ws_bytes > kNoAllocScratchBytes) return FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const fa_status sa = scratch_address(dev, &scratch);
  if (sa != FA_OK) return sa;
  return launch(pr, sm_count, pl, scratch, stream);
}

// ---------------------------------------------------------------- host-buffer entry point
// fa_fwd_host: Q, K, V in host memory, O and LSE back to host memory, with the copies and
// the kernels overlapped.  The (batch, head) slices are cut into chunks of whole heads;
// chunk c travels to the GPU on an upload stream while chunk c-1 is computed on the
// caller's stream and chunk c-2 travels back on a download stream, ordered by events.
// Every device buffer lives in the caller's workspace, so the call allocates nothing.
namespace {

constexpr int kHostMaxChunks = 8;   // chunks of heads, plus possibly one single-head last chunk

struct HostPipe {
  bool ready = false;
  cudaStream_t up = nullptr;
  cudaStream_t down = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t end = nullptr;
  cudaEvent_t up_done[kHostMaxChunks + 1] = {};
  cudaEvent_t cmp_done[kHostMaxChunks + 1] = {};
};

std::mutex g_host_mutex[kMaxDevices];
HostPipe g_host_pipe[kMaxDevices];

// The device's upload/download streams and events, created on first use (the device's
// mutex must be held).
fa_status host_pipe(int dev, HostPipe** out) {
  HostPipe& hp = g_host_pipe[dev];
  if (!hp.ready) {
    bool ok = cudaStreamCreateWithFlags(&hp.up, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.down, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.end, cudaEventDisableTiming) == cudaSuccess;
    for (int c = 0; ok && c < kHostMaxChunks + 1; ++c)
      ok = cudaEventCreateWithFlags(&hp.up_done[c], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.cmp_done[c], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      if (hp.up) cudaStreamDestroy(hp.up);
      if (hp.down) cudaStreamDestroy(hp.down);
      for (cudaEvent_t e : {hp.start, hp.end}) if (e) cudaEventDestroy(e);
      for (int c = 0; c < kHostMaxChunks + 1; ++c) {
        if (hp.up_done[c]) cudaEventDestroy(hp.up_done[c]);
        if (hp.cmp_done[c]) cudaEventDestroy(hp.cmp_done[c]);
      }
      hp = HostPipe{};
      return FA_ERR_CUDA;
    }
    hp.ready = true;
  }
  *out = &hp;
  return FA_OK;
}

// A validated host-buffer problem and the layout of its device workspace.
struct HostPlan {
  Problem pr;          // sizes, mask and scale; the pointers are the caller's host buffers
  int chunks = 1;
  long long bounds[kHostMaxChunks + 2] = {};   // chunk c holds the heads [bounds[c], bounds[c + 1])
  size_t off_q = 0, off_k = 0, off_v = 0, off_o = 0, off_lse = 0, off_split = 0;
  size_t split_bytes = 0;
  size_t total = 0;
};

long long chunk_lo(const HostPlan& hp, int c) { return hp.bounds[c]; }

// The chunk of heads [a, b) as a problem of its own: B = 1, H = b - a, on the workspace copies.
Problem chunk_problem(const HostPlan& hp, uint8_t* ws, long long a, long long b) {
  Problem c = hp.pr;
  const long long n = b - a;
  const size_t q_row = static_cast<size_t>(hp.pr.Lq) * hp.pr.D * 2;
  const size_t k_row = static_cast<size_t>(hp.pr.Lk) * hp.pr.D * 2;
  c.Q = ws ? ws + hp.off_q + a * q_row : nullptr;
  c.K = ws ? ws + hp.off_k + a * k_row : nullptr;
  c.V = ws ? ws + hp.off_v + a * k_row : nullptr;
  c.O = ws ? ws + hp.off_o + a * q_row : nullptr;
  c.LSE = ws ? reinterpret_cast<float*>(ws + hp.off_lse) + a * hp.pr.Lq : nullptr;
  c.B = 1;
  c.H = static_cast<int>(n);
  c.bh = n;
  c.n_units = static_cast<int>(n * hp.pr.n_pairs);
  c.bytes_q = n * q_row;
  c.bytes_k = n * k_row;
  c.bytes_lse = static_cast<size_t>(n) * hp.pr.Lq * 4;
  contiguous_strides(c.H, c.Lq, c.D, c.qs);
  contiguous_strides(c.H, c.Lk, c.D, c.ks);
  contiguous_strides(c.H, c.Lk, c.D, c.vs);
  contiguous_strides(c.H, c.Lq, c.D, c.os);
  return c;
}

// Checks the arguments of fa_fwd_host / fa_fwd_host_workspace_size and lays out the
// workspace.  *empty = true: nothing to compute.
fa_status host_plan(int B, int H, int Lq, int Lk, int D, int window_left, int window_right,
                    float scale, bool check_scale, HostPlan* hp, int* sm_count, bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (window_left < -1 || window_right < -1) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  if (bh * Lq == 0) {
    *empty = true;
    return FA_OK;
  }
  if (Lk < 1) return FA_ERR_INVALID_ARG;
  if (check_scale && (!(scale > 0.0f) || !isfinite(scale))) return FA_ERR_INVALID_ARG;
  const long long n_pairs = (Lq + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM);
  if (bh > INT_MAX || n_pairs * bh > INT_MAX) return FA_ERR_INVALID_ARG;
  if (bh * Lq * D > (1ll << 40) || bh * Lk * D > (1ll << 40)) return FA_ERR_INVALID_ARG;
  int left = window_left, right = window_right;
  if (left >= Lq - 1) left = -1;
  if (right >= Lk - 1) right = -1;
  if (left >= 0 && Lq - 1 - left > Lk - 1) return FA_ERR_INVALID_ARG;   // a row without keys
  const fa_status prep = current_device(D, sm_count);
  if (prep != FA_OK) return prep;

  Problem& pr = hp->pr;
  pr = Problem{};
  pr.Lq = Lq;
  pr.Lk = Lk;
  pr.D = D;
  pr.scale = scale;
  pr.bh = bh;
  pr.n_pairs = static_cast<int>(n_pairs);
  pr.n_units = static_cast<int>(n_pairs * bh);
  pr.nkv = (Lk + fa::kBlockN - 1) / fa::kBlockN;
  pr.B = B;
  pr.H = H;
  if (left < 0 && (right < 0 || right == 0)) {
    pr.causal = right == 0 ? 1 : 0;   // the full or the causal mask: whole units or split
  } else {
    pr.band = true;
    pr.win_left = left;
    pr.win_right = right;
  }
  // Chunks: enough to overlap the copies with the kernels, few enough that each chunk's
  // kernel still spreads over the GPU (at least 256 query-tile pairs per chunk).  Test
  // hook (fa_debug_set bit 3): as many chunks as there are heads, up to the maximum.
  const long long chunks = (g_debug_flags.load() & 8u)
                               ? std::min<long long>(kHostMaxChunks, bh)
                               : std::min<long long>({kHostMaxChunks, pr.n_units / 256, bh});
  hp->chunks = static_cast<int>(std::max<long long>(1, chunks));
  for (int c = 0; c <= hp->chunks; ++c) hp->bounds[c] = bh * c / hp->chunks;
  // A causal chunk takes as long as its longest unit, which its last head alone also has:
  // the last chunk's kernel is what remains once the last input has arrived.  When one head
  // by itself would take the split-key schedule (its longest unit spread over every SM), the
  // last chunk is that one head.
  if (pr.causal && hp->chunks >= 2 && bh > hp->chunks) {
    Problem one = pr;
    one.B = 1;
    one.H = 1;
    one.bh = 1;
    one.n_units = pr.n_pairs;
    if (plan_schedule(one, *sm_count).split) {
      const int rest = hp->chunks;   // the other heads keep the chunk count
      for (int c = 0; c <= rest; ++c) hp->bounds[c] = (bh - 1) * c / rest;
      hp->chunks = rest + 1;
      hp->bounds[hp->chunks] = bh;
    }
  }
  pr.bytes_q = static_cast<size_t>(bh) * Lq * D * 2;
  pr.bytes_k = static_cast<size_t>(bh) * Lk * D * 2;
  pr.bytes_lse = static_cast<size_t>(bh) * Lq * 4;
  hp->off_q = 0;
  hp->off_k = hp->off_q + round256(pr.bytes_q);
  hp->off_v = hp->off_k + round256(pr.bytes_k);
  hp->off_o = hp->off_v + round256(pr.bytes_k);
  hp->off_lse = hp->off_o + round256(pr.bytes_q);
  hp->off_split = hp->off_lse + round256(pr.bytes_lse);
  hp->split_bytes = 0;
  if (!pr.band) {   // the largest split-schedule workspace any chunk needs
    for (int c = 0; c < hp->chunks; ++c) {
      const Problem cp = chunk_problem(*hp, nullptr, chunk_lo(*hp, c), chunk_lo(*hp, c + 1));
      const Plan pl = plan_schedule(cp, *sm_count);
      if (pl.split) hp->split_bytes = std::max(hp->split_bytes, pl.ws_bytes);
    }
  }
  hp->total = hp->off_split + hp->split_bytes;
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_fwd_host_workspace_size(int B, int H, int Lq, int Lk, int D,
                                                int window_left, int window_right, size_t* bytes) {
  if (!bytes) return FA_ERR_INVALID_ARG;
  *bytes = 0;
  HostPlan hp;
  int sm_count = 0;
  bool empty = false;
  const fa_status st = host_plan(B, H, Lq, Lk, D, window_left, window_right, 0.0f, false, &hp,
                                 &sm_count, &empty);
  if (st != FA_OK || empty) return st;
  *bytes = hp.total;
  return FA_OK;
}

extern "C" fa_status fa_fwd_host(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                 int B, int H, int Lq, int Lk, int D, int window_left,
                                 int window_right, float scale, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  HostPlan hp;
  int sm_count = 0;
  bool empty = false;
  const fa_status st = host_plan(B, H, Lq, Lk, D, window_left, window_right, scale, true, &hp,
                                 &sm_count, &empty);
  if (st != FA_OK || empty) return st;
  const Problem& pr = hp.pr;
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  // O and LSE are written while later chunks of Q, K, V are still being read.
  if (overlaps(O, pr.bytes_q, Q, pr.bytes_q) || overlaps(O, pr.bytes_q, K, pr.bytes_k) ||
      overlaps(O, pr.bytes_q, V, pr.bytes_k) || overlaps(O, pr.bytes_q, LSE, pr.bytes_lse) ||
      overlaps(LSE, pr.bytes_lse, Q, pr.bytes_q) || overlaps(LSE, pr.bytes_lse, K, pr.bytes_k) ||
      overlaps(LSE, pr.bytes_lse, V, pr.bytes_k))
    return FA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < hp.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return FA_ERR_INVALID_ARG;
  const void* host[5] = {Q, K, V, O, LSE};
  const size_t host_bytes[5] = {pr.bytes_q, pr.bytes_k, pr.bytes_k, pr.bytes_q, pr.bytes_lse};
  for (int i = 0; i < 5; ++i)
    if (overlaps(workspace, hp.total, host[i], host_bytes[i])) return FA_ERR_INVALID_ARG;
  if (g_debug_flags.load() & 2u) return FA_ERR_CUDA;   // test hook: simulated launch failure

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_host_mutex[dev]);
  HostPipe* pipe = nullptr;
  const fa_status ps = host_pipe(dev, &pipe);
  if (ps != FA_OK) return ps;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* hq = static_cast<const uint8_t*>(Q);
  const uint8_t* hk = static_cast<const uint8_t*>(K);
  const uint8_t* hv = static_cast<const uint8_t*>(V);
  uint8_t* ho = static_cast<uint8_t*>(O);
  const size_t q_row = static_cast<size_t>(pr.Lq) * pr.D * 2;
  const size_t k_row = static_cast<size_t>(pr.Lk) * pr.D * 2;
  const size_t l_row = static_cast<size_t>(pr.Lq) * 4;
  // The copies start after the work queued on `stream` so far (the caller may still be
  // producing the inputs or using the outputs there).
  if (cudaEventRecord(pipe->start, stream) != cudaSuccess ||
      cudaStreamWaitEvent(pipe->up, pipe->start, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  auto copy = [](void* dst, const void* src, size_t n, cudaStream_t s) {
    return cudaMemcpyAsync(dst, src, n, cudaMemcpyDefault, s) == cudaSuccess;
  };
  for (int c = 0; c < hp.chunks; ++c) {
    const long long a = chunk_lo(hp, c), b = chunk_lo(hp, c + 1);
    const size_t n = static_cast<size_t>(b - a);
    if (!copy(ws + hp.off_q + a * q_row, hq + a * q_row, n * q_row, pipe->up) ||
        !copy(ws + hp.off_k + a * k_row, hk + a * k_row, n * k_row, pipe->up) ||
        !copy(ws + hp.off_v + a * k_row, hv + a * k_row, n * k_row, pipe->up) ||
        cudaEventRecord(pipe->up_done[c], pipe->up) != cudaSuccess ||
        cudaStreamWaitEvent(stream, pipe->up_done[c], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    const Problem cp = chunk_problem(hp, ws, a, b);
    Plan pl{};
    if (cp.band) {
      pl.band = true;
      pl.grid = std::min(cp.n_units, sm_count);
    } else {
      pl = plan_schedule(cp, sm_count);
    }
    // Not a programmatic dependent launch: the operation ahead of it is the event wait.
    const fa_status ls = launch(cp, sm_count, pl, pl.split ? ws + hp.off_split : nullptr, stream,
                                /*allow_dependent=*/false);
    if (ls != FA_OK) return ls;
    if (cudaEventRecord(pipe->cmp_done[c], stream) != cudaSuccess ||
        cudaStreamWaitEvent(pipe->down, pipe->cmp_done[c], 0) != cudaSuccess ||
        !copy(ho + a * q_row, ws + hp.off_o + a * q_row, n * q_row, pipe->down) ||
        !copy(LSE + a * pr.Lq, ws + hp.off_lse + a * l_row, n * l_row, pipe->down))
      return FA_ERR_CUDA;
  }
  // `stream` completes only after the last download.
  if (cudaEventRecord(pipe->end, pipe->down) != cudaSuccess ||
      cudaStreamWaitEvent(stream, pipe->end, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

extern "C" const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported head dim or device";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel pipeline wait ran out of time";
  }
  return "unknown fa_status";
}

extern "C" fa_status fa_last_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, fa::g_status, sizeof(v)) != cudaSuccess) return FA_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(fa::g_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
  }
  const unsigned vb = fa_bwd_take_device_status();   // the backward kernels' word
  if (!v) v = vb;
  return static_cast<fa_status>(v & 0xffu);
}

unsigned long long fa_internal_wait_limit_ns() { return g_wait_limit_ns.load(); }
unsigned fa_internal_debug_flags() { return g_debug_flags.load(); }

extern "C" fa_status fa_debug_set(unsigned int flags, unsigned long long wait_limit_ns) {
  g_debug_flags.store(flags);
  g_wait_limit_ns.store(wait_limit_ns);
  return FA_OK;
}
