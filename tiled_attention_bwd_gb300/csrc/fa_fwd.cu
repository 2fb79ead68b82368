// fa_fwd.cu -- forward attention kernel for sm_103a.
//
// O = softmax(scale * Q K^T [+ causal mask]) V and LSE per row, computed
// tile by tile with an online softmax so the N x N scores never leave the SM
// ("RTX Flash Attention Implementation COMPLETE", "CUDA Kernel Design: Flash
// Attention Forward Kernel" and "Online Softmax Algorithm"; the TMA /
// warp-specialised pipeline of "GPU Performance Optimization Batch 1 --
// Design Spec", Item 3, sections "TMA" and "Warp Specialization").
//
// Persistent blocks (one per SM) take work items of two 128-row Q tiles of
// one (batch, head), or of one tile when a problem has fewer pairs than
// SMs, and stream the 128-row K/V tiles past them:
//   warp 8      TMA producer: Q0, Q1 once per item (three rotating
//               buffers, q_buf); K_j, V_j through a ring.
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM, then
//               O_t += P_t V_j with P_t read straight from TMEM.
//   warps 0-3   softmax for Q tile 0, warps 4-7 for Q tile 1; thread = row.
//               exp2 with the scale folded in, lazy rescaling of O (only when
//               the row max grows by more than 2^8), P written back to TMEM
//               as bf16 over the S columns it came from.
// At the end of an item each softmax thread writes its row of O: by TMA
// store through a per-warp box in shared memory in the dynamic-schedule and
// windowed kernels, in 32-byte (else 16-byte) stores from registers in the
// others.
// While one softmax group works on its tile the tensor core runs the other
// tile's MMAs (ping-pong).  Causal blocks stop at the diagonal tile; only the
// diagonal (and a ragged last tile) is masked.
//
// Two variants the pages list as future work are folded in: grouped /
// multi-query attention (H query heads share Hkv key/value heads; query
// head h reads K/V head h / (H / Hkv)) and a sliding window (key j visible
// to query i only if |i - j| <= window).  A window narrows each Q tile's key
// tiles to the band and masks the tiles its edges cross; without one (and
// with Hkv = H) the kernel is the plain operation.
//
// TMEM columns (512 allocated): S0, S1 | O0, O1 (see FwdLayout).
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

// Warps 0-3: softmax for Q tile 0; 4-7: tile 1; 8: TMA producer; 9: MMA
// issuer.  With kSplitRegs the block has 12 warps (three warpgroups; 10 and
// 11 idle): launched at kLaunchRegs registers per thread, the control group
// drops to kCtrlRegs and the softmax groups rise to kSoftmaxRegs, with
// 2 * 128 * kSoftmaxRegs + 128 * kCtrlRegs <= 384 * kLaunchRegs.  Without it
// the block has 10 warps at 168 registers each (65536 / 320, rounded down to
// a multiple of 8 and limited by the three warps on two of the four
// schedulers).
constexpr bool kSplitRegs = true;
constexpr int kFwdThreads = kSplitRegs ? 384 : 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kLaunchRegs = 168;
constexpr bool kInl = kSplitRegs;  // waits inline: no calls under setmaxnreg
constexpr int kCtrlRegs = 96;
constexpr int kSoftmaxRegs = 200;
static_assert(!kSplitRegs || 2 * 128 * kSoftmaxRegs + 128 * kCtrlRegs <=
                                  kFwdThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: factor 256

// Shared memory: three Q tile buffers (see q_buf) and a ring of K/V tiles,
// all 128 rows.
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [256+d,256+2d);
// P_t (bf16 pairs) is written over the first 64 columns of S_t.
//
// Measured on this part: in a chain of M=128 tcgen05 MMAs as an earlier
// probe issued them, both operands in smem ran at about 40% of peak and A in
// TMEM at full rate; MMAs with N or K of 64 ran well below it; and the
// forward's interleaving of S = Q K^T (smem x smem) with O += P V (TMEM x
// smem) ran at full rate.  Issued back to back with no waits, every form runs
// at full rate, so the smem x smem cost is latency on a dependent path.
// Hence 128-key tiles, P kept in TMEM, and two Q tiles whose MMAs interleave.
// QBUFS: 3 Q buffers for the rotation of q_buf, 2 for the banded (WINDOW)
// kernels, which keep tile t in buffer t.  Those include the kernels with
// per-sequence lengths, whose balanced item table takes the shared memory
// left after the tiles: about 32 KB with two buffers, 1.8 KB with three.
// OSTG: O leaves through shared memory by TMA store, one [32 rows][64
// columns] bf16 box (4 KB, 128-byte swizzle) per softmax warp.  With three
// Q buffers at d = 128 the K/V ring gives up a stage for it (measured no
// slower with the dynamic schedule, whose K/V come from DRAM; the static
// one lost 6.5% at 4x32x1024, so it keeps four stages and stores O from
// registers); the banded kernels' two Q buffers leave room for it.
template <int D, int QBUFS = 3, bool OSTG = false>
struct FwdLayout {
  static constexpr int kSub = D / 64;             // 64-column sub-tiles
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = (D == 128) ? ((OSTG && QBUFS == 3) ? 3 : 4) : 6;
  static constexpr int kQOff = 0;
  static constexpr int kQBufs = QBUFS;
  static constexpr int kKVOff = kQBufs * kTileBytes;
  static constexpr int kOStgOff = kKVOff + kStages * kTileBytes;
  static constexpr int kOStgBoxBytes = 32 * 128;
  static constexpr int kBarOff = kOStgOff + (OSTG ? 8 * kOStgBoxBytes : 0);
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // + align slack
};
// Bytes reserved for the barriers; the item table of the VARLEN kernels
// follows them.
constexpr int kFwdBarBytes = 256;

// Kernels whose O leaves by TMA store: bf16, with the dynamic schedule or a
// window (not per-sequence lengths, whose padding rows stay untouched and
// whose item table takes the shared memory).
template <bool WINDOW, bool FP8, bool VARLEN, bool DYN>
constexpr bool fwd_ostg() { return !FP8 && !VARLEN && (DYN || WINDOW); }

template <int STAGES>
struct FwdBars {
  uint64_t q_full[3];    // per Q buffer
  uint64_t q_empty[3];
  uint64_t kv_full[STAGES];
  uint64_t kv_empty[STAGES];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t mma_done;
  uint64_t sched_full[2];   // work item t published in sched_item[t % 2]
  uint64_t sched_empty[2];  // ... and read by the MMA thread and 8 warps
  int sched_item[2];
  uint32_t tmem_base;
  uint32_t abort;
};

// Where-codes of bounded waits (recorded when a wait expires).
enum : uint32_t {
  kWFwdProdEmpty = 0x101,
  kWFwdProdQ = 0x102,
  kWFwdProdSched = 0x103,
  kWFwdMmaSched = 0x204,
  kWFwdSmSched = 0x303,
  kWFwdMmaQ = 0x201,
  kWFwdMmaKV = 0x202,
  kWFwdMmaP = 0x203,
  kWFwdSmS = 0x301,
  kWFwdSmO = 0x302,
};

// Q buffer of tile t (0, 1) of the n-th item (with work) a block runs.
// Tile 0 takes the buffer the item before left spare, tile 1 that item's
// tile-0 buffer, which is freed a key tile before its tile-1 buffer (causal
// pairs end one key tile apart).  So both loads of the next item can be
// issued while the current item's last key tiles run, instead of waiting
// for its tile 1 to let go of its buffer: buffers (t0, t1, spare) run
// (0, 1, 2), (2, 0, 1), (1, 2, 0), ...  The banded (WINDOW) kernels keep
// two buffers, tile t in buffer t (see FwdLayout): the rotation cost them
// 3-4%.
__device__ __forceinline__ int q_buf(uint32_t n, int t) {
  const int r = (int)(n % 3u);
  return (t == 0 ? 3 - r : 4 - r) % 3;
}

// S_t = Q_t K^T: M = N = 128, K = d; both operands K-major in smem.  The
// descriptors are those of the tiles' first bytes; each 16-wide K step is
// 32 bytes further along the 128-byte rows, each 64-column sub-tile 16 KB.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint64_t q_desc,
                                         uint64_t k_desc) {
  constexpr uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    const uint32_t off = (s >> 2) * kSubTileBytes + (s & 3) * 32;
    mma_ss(s_tmem, sdesc_adv(q_desc, off), sdesc_adv(k_desc, off), id,
           s > 0 ? 1u : 0u);
  }
}

// FP8 path: S_t = Q8_t K8^T with E4M3 operands, K = 128 in four steps
// of 32 elements (32 bytes) along one 128-byte row; scales are applied by
// the softmax.
__device__ __forceinline__ void issue_qk_fp8(uint32_t s_tmem, uint64_t q_desc,
                                             uint64_t k_desc) {
  constexpr uint32_t id = idesc_e4m3(128, 128);
#pragma unroll
  for (int s = 0; s < 4; ++s)
    mma_ss_f8(s_tmem, sdesc_adv(q_desc, s * 32), sdesc_adv(k_desc, s * 32), id,
              s > 0 ? 1u : 0u);
}

// O_t (+)= P_t V: M = 128, N = d, K = 128 keys; A = P from TMEM, B = V
// read MN-major (d contiguous in smem; 16 keys = 2048 bytes per K step).
// v_desc: MN-major descriptor of V's first byte.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem,
                                         uint64_t v_desc, bool accumulate) {
  constexpr uint32_t id = idesc_bf16(128, D, false, true);
#pragma unroll
  for (int s = 0; s < kTile / 16; ++s) {
    mma_ts(o_tmem, p_tmem + s * 8, sdesc_adv(v_desc, s * 2048), id,
           (accumulate || s > 0) ? 1u : 0u);
  }
}

// Key tiles [lo, hi] that Q tile qt must visit.  Query i sees key j when
// j <= i (causal) and |i - j| <= window (window >= 0); rows and keys past N
// are handled by the masks.  `window` is below N here (a wider band is the
// same as none and is passed as -1, or as N - 1 with per-sequence lengths).
template <bool CAUSAL>
__device__ __forceinline__ void key_range(int qt, int n_tiles, int window,
                                          int& lo, int& hi) {
  const long long q0 = (long long)qt * kTile, q1 = q0 + kTile - 1;
  lo = (window >= 0 && q0 > window) ? (int)((q0 - window) / kTile) : 0;
  if (CAUSAL) {
    hi = qt;
  } else if (window >= 0) {
    const long long h = (q1 + window) / kTile;
    hi = h < n_tiles - 1 ? (int)h : n_tiles - 1;
  } else {
    hi = n_tiles - 1;
  }
}

// One work item = (query head, pair of Q tiles).  Tile t visits key tiles
// lo_t..hi_t; the K/V stream covers jb..je, the union of both ranges (a
// missing second tile has hi1 = -1).  K/V come from the item's key/value
// head: query head h of a batch entry reads head h / (H / Hkv).
struct FwdItem {
  int bh, kvh, qt0, qt1, lo0, hi0, lo1, hi1, jb, je;
  int len;  // rows of this batch entry's sequence (N without lengths)
};
// Items come in groups of heads whose K and V fit in L2 together, heaviest
// first within a group (pair index slow, head fast; causal pairs from the
// last one down).
// Balanced item order with per-sequence lengths.  The plain order assumes
// that every head has the same items; with lengths, items past a sequence's
// end are empty and the dealing of the remaining ones to blocks loses its
// balance.  So each block first builds, in shared memory, the same compact
// list of non-empty items in decreasing cost:
//   np[b]    pairs of Q tiles of sequence b (ceil(tiles / 2));
//   order[s] sequences by decreasing np (ties by index: every block gets the
//            same order, so the item lists agree), by a counting sort;
//   pref[x]  item counts before group x, where a group is a pair index from
//            the last one down (causal: a pair's cost is the same for every
//            sequence that has it, and the sequences that have pair p are the
//            first ones of `order`) or a sequence in `order` (otherwise: a
//            sequence's pairs all cost its length).
// Returns the number of items.  All threads of the block take part.
template <bool CAUSAL>
__device__ int build_item_table(int* tab, const FwdArgs& a, int n_pairs) {
  const int B = a.BH / a.H;
  const int X = CAUSAL ? n_pairs : B;
  int* np = tab;
  int* order = tab + B;
  int* pref = tab + 2 * B;
  int* start = pref + X + 1;  // [n_pairs + 1]: counting-sort bins
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int v = tid; v <= n_pairs; v += nt) start[v] = 0;
  for (int b = tid; b < B; b += nt) {
    const int tiles = (seq_len_of(a.seq_lens, b, a.N) + kTile - 1) / kTile;
    np[b] = (tiles + 1) / 2;  // <= n_pairs: lengths are clamped to N
  }
  __syncthreads();
  for (int b = tid; b < B; b += nt) atomicAdd(&start[np[b]], 1);
  __syncthreads();
  // Stable counting sort by decreasing np, by one warp: start[v] becomes the
  // number of sequences with more pairs than v, then 32 sequences are placed
  // per step in index order (equal values ranked by lane), so every block
  // builds the same order.
  if (tid < 32) {
    const int V = n_pairs + 1;  // bins, taken from the largest value down
    const int chunk = (V + 31) / 32;
    const int r0 = tid * chunk, r1 = min(V, r0 + chunk);
    int sum = 0;
    for (int r = r0; r < r1; ++r) sum += start[n_pairs - r];
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (tid >= off) incl += t;
    }
    int run = incl - sum;
    for (int r = r0; r < r1; ++r) {
      const int c = start[n_pairs - r];
      start[n_pairs - r] = run;
      run += c;
    }
    __syncwarp();
    for (int c0 = 0; c0 < B; c0 += 32) {
      const int b = c0 + tid;
      const int v = b < B ? np[b] : -1;
      const unsigned grp = __match_any_sync(0xffffffffu, v);
      const int rank = __popc(grp & ((1u << tid) - 1u));
      const int base = b < B ? start[v] : 0;
      __syncwarp();
      if (b < B) {
        order[base + rank] = b;
        if (rank == 0) start[v] = base + __popc(grp);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int x = tid; x < X; x += nt) {
    int cnt;
    if (CAUSAL) {  // sequences with more than p pairs: a prefix of `order`
      const int p = n_pairs - 1 - x;
      int lo = 0, hi = B;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (np[order[mid]] > p) lo = mid + 1; else hi = mid;
      }
      cnt = lo;
    } else {
      cnt = np[order[x]];
    }
    pref[x + 1] = cnt * a.H;
  }
  __syncthreads();
  if (tid < 32) {  // inclusive scan of pref[1..X]: one chunk per lane
    const int chunk = (X + 31) / 32;
    const int x0 = tid * chunk, x1 = min(X, x0 + chunk);
    int sum = 0;
    for (int x = x0; x < x1; ++x) sum += pref[x + 1];
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (tid >= off) incl += t;
    }
    int run = incl - sum;
    for (int x = x0; x < x1; ++x) {
      run += pref[x + 1];
      pref[x + 1] = run;
    }
    if (tid == 0) pref[0] = 0;
  }
  __syncthreads();
  return pref[X];
}

// Query head and pair index of compact item c (see build_item_table).
template <bool CAUSAL>
__device__ __forceinline__ void table_item(int c, const int* tab, int B,
                                           int H, int n_pairs, int& bh,
                                           int& pair) {
  const int* order = tab + B;
  const int* pref = tab + 2 * B;
  int lo = 0, hi = (CAUSAL ? n_pairs : B) - 1;  // last group with pref <= c
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= c) lo = mid; else hi = mid - 1;
  }
  const int k = c - pref[lo];
  int s, h;
  if (CAUSAL) {
    pair = n_pairs - 1 - lo;
    s = k / H;
    h = k - s * H;
  } else {
    s = lo;
    pair = k / H;
    h = k - pair * H;
  }
  bh = order[s] * H + h;
}

// Per-sequence lengths are honoured by the VARLEN instantiations only, which
// are windowed ones (the host runs a call with lengths and no window as one
// with a window of N - 1, which hides nothing): in the other instantiations
// the length's per-item arithmetic cost registers and about 5% of the time.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ FwdItem fwd_item(int w, int n_tiles, int n_pairs,
                                            const FwdArgs& a, const int* tab) {
  FwdItem it;
  int pair;
  if (VARLEN && tab) {
    table_item<CAUSAL>(w, tab, a.BH / a.H, a.H, n_pairs, it.bh, pair);
  } else {
    // Groups of a.group heads whose K and V fit in L2 together; within a
    // group the pair index is slow (heaviest first) and the head fast.
    const int per_group = a.group * n_pairs;
    const int grp = w / per_group;
    const int rr = w - grp * per_group;
    const int rest = a.BH - grp * a.group;
    const int heads = rest < a.group ? rest : a.group;
    const int rank = rr / heads;
    pair = CAUSAL ? (n_pairs - 1 - rank) : rank;
    it.bh = grp * a.group + (rr - rank * heads);
  }
  const int b = it.bh / a.H, h = it.bh - b * a.H;
  it.kvh = b * a.Hkv + h / (a.H / a.Hkv);
  // A single-tile item has no tile 1 (qt1 past the last tile).
  it.qt0 = a.single ? pair : 2 * pair;
  it.qt1 = a.single ? n_tiles : 2 * pair + 1;
  // With per-sequence lengths, tiles at or past the sequence's end are not
  // visited; an item with no tile left is empty (hi0 = -1) for every role.
  it.len = VARLEN ? seq_len_of(a.seq_lens, b, a.N) : a.N;
  const int tiles_b = VARLEN ? (it.len + kTile - 1) / kTile : n_tiles;
  if (VARLEN && it.qt0 >= tiles_b) {
    it.lo0 = it.lo1 = it.jb = 0;
    it.hi0 = it.hi1 = it.je = -1;
    return it;
  }
  key_range<CAUSAL>(it.qt0, tiles_b, a.window, it.lo0, it.hi0);
  if (it.qt1 < tiles_b) {
    key_range<CAUSAL>(it.qt1, tiles_b, a.window, it.lo1, it.hi1);
  } else {
    it.lo1 = 0;
    it.hi1 = -1;
  }
  it.jb = it.lo0;  // lo1 >= lo0
  it.je = it.hi0 > it.hi1 ? it.hi0 : it.hi1;
  return it;
}

// Work items are handed out in one of two ways.  When every head's K and V
// fit in L2 together, in rounds of gridDim.x items dealt to the blocks
// alternately forwards and backwards, so that with items sorted by
// decreasing cost every block gets a similar total.  Otherwise dynamically
// (the DYN instantiations): block b starts with item b and then claims the next
// unclaimed one from a counter in device memory, so that the head groups
// cost no balance.  The counter belongs to this call (a slot of a ring the
// host hands out); the last block to finish sets it back to zero for the
// slot's next call.  Either way the producer thread publishes each item in
// a two-slot ring in shared memory, which the MMA thread and the softmax
// warps read in the same order.
__device__ __forceinline__ int fwd_round_item(int r) {
  const int g = (int)gridDim.x, b = (int)blockIdx.x;
  return r * g + ((r & 1) ? (g - 1 - b) : b);
}

// Item t of this block: the alternating rounds, computed locally, or (with
// DYN) the one the producer published.
template <bool DYN, int S>
__device__ __forceinline__ bool fwd_take(FwdBars<S>* bars, int t, bool warp_wide,
                                         const WaitCtl& wc, uint32_t where, int& w) {
  if constexpr (!DYN) {
    w = fwd_round_item(t);
    return true;
  }
  const int sl = t & 1;
  const uint32_t par = (uint32_t)(t >> 1) & 1u;
  bool ok = wait_bar<true>(&bars->sched_full[sl], par, wc, where);
  if (warp_wide) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return false;
  w = *reinterpret_cast<volatile int*>(&bars->sched_item[sl]);
  if (warp_wide) warp_arrive(&bars->sched_empty[sl]);
  else mbar_arrive(&bars->sched_empty[sl]);
  return true;
}

// Persistent: one block per SM takes items one after another.  Barrier
// phases run on across items, so the producer fetches the next item's Q and
// K/V while the current one finishes, and the next item's first Q K^T
// overlaps the softmax warps' epilogue.
template <int D, bool CAUSAL, bool WINDOW, bool FP8, bool VARLEN, bool DYN,
          bool HOOK>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v,
               const __grid_constant__ CUtensorMap tm_o, const FwdArgs a) {
  constexpr bool OSTG = fwd_ostg<WINDOW, FP8, VARLEN, DYN>();
  using L = FwdLayout<D, WINDOW ? 2 : 3, OSTG>;
  constexpr int S = L::kStages;
  // Bytes and 128-byte-wide TMA boxes of one Q or K tile: bf16, or E4M3 on
  // the FP8 path: one byte per element in rows of 128 bytes (at d = 64 the
  // upper half of each row is zero, so the product is that of d = 128), a
  // single box.
  static_assert(!FP8 || D == 128 || D == 64, "the FP8 path needs d = 64 or 128");
  constexpr uint32_t kQKBytes = FP8 ? kTile * 128 : L::kTileBytes;
  constexpr int kQKBoxes = FP8 ? 1 : L::kSub;
  static_assert(sizeof(FwdBars<S>) <= kFwdBarBytes, "barrier block");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  auto* bars = reinterpret_cast<FwdBars<S>*>(smem + L::kBarOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  // Work items ("pairs" below) per head: pairs of Q tiles, or single tiles.
  const int n_pairs = a.single ? n_tiles : (n_tiles + 1) / 2;
  int n_items = a.BH * n_pairs;
  const int* tab = nullptr;
  if constexpr (VARLEN) {
    if (a.sched) {
      int* t = reinterpret_cast<int*>(smem + L::kBarOff + kFwdBarBytes);
      n_items = build_item_table<CAUSAL>(t, a, n_pairs);
      tab = t;
    }
  }

  if (threadIdx.x == 0) {
    bars->abort = *reinterpret_cast<volatile unsigned int*>(&a.st->abort);
    for (int b = 0; b < L::kQBufs; ++b) {
      mbar_init(&bars->q_full[b], 1);
      mbar_init(&bars->q_empty[b], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 4);   // one arrival per warp
      mbar_init(&bars->o_done[t], 1);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->mma_done, 1);
    for (int sl = 0; sl < 2; ++sl) {
      mbar_init(&bars->sched_full[sl], 1);
      mbar_init(&bars->sched_empty[sl], 9);  // MMA thread + 8 softmax warps
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool run = ld_volatile_u32(&bars->abort) == 0;
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{a.st, &bars->abort, a.timeout_ns};

  // Each role's code sits inside the branch that sets its register count,
  // so that the compiler sizes it for that count.
  if (kSplitRegs && warp >= 8) reg_dealloc<kCtrlRegs>();
  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0 && run) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      if constexpr (OSTG) prefetch_tmap(&tm_o);
      int last_par[S];
#pragma unroll
      for (int s = 0; s < S; ++s) last_par[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      // Per Q buffer (bit b): parity of the loads issued into it, and
      // whether it has had one.
      uint32_t q_par = 0, q_used = 0;
      uint32_t n_done = 0;   // items with work so far
      bool ok = true;
      for (int ti = 0; ok; ++ti) {
        FwdItem itm;
        int w;
        if constexpr (!DYN) {
          // Alternating rounds: every role computes the same sequence.
          w = fwd_round_item(ti);
          if (w >= n_items) break;
          itm = fwd_item<CAUSAL, VARLEN>(w, n_tiles, n_pairs, a, tab);
          if (VARLEN && itm.hi0 < 0) continue;  // empty (past its sequence's end)
        } else {
          // Claim the next item with work (with per-sequence lengths some
          // are empty) and publish it; n_items or more tells the others to
          // stop.
          w = ti > 0 ? (int)gridDim.x + (int)atomicAdd(a.work_next, 1u)
                     : (int)blockIdx.x;
          while (w < n_items) {
            itm = fwd_item<CAUSAL, VARLEN>(w, n_tiles, n_pairs, a, tab);
            if (!VARLEN || itm.hi0 >= 0) break;
            w = (int)gridDim.x + (int)atomicAdd(a.work_next, 1u);
          }
          ok = wait_bar<kInl, HOOK>(&bars->sched_empty[ti & 1],
                              ((uint32_t)(ti >> 1) & 1u) ^ 1u, wc, kWFwdProdSched);
          if (!ok) break;
          *reinterpret_cast<volatile int*>(&bars->sched_item[ti & 1]) = w;
          mbar_arrive(&bars->sched_full[ti & 1]);
          if (w >= n_items) break;
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok || (t == 1 && itm.hi1 < 0)) break;
          const int b = WINDOW ? t : q_buf(n_done, t);
          // The buffer must no longer be read by an earlier item's Q K^T.
          ok = wait_bar<kInl, HOOK>(&bars->q_empty[b], ((q_par >> b) & 1u) ^ 1u, wc,
                                    kWFwdProdQ);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars->q_full[b], kQKBytes);
#pragma unroll
          for (int sb = 0; sb < kQKBoxes; ++sb)
            tma_load_3d(smem + L::kQOff + b * L::kTileBytes + sb * kSubTileBytes,
                        &tm_q, &bars->q_full[b], sb * 64,
                        (t ? itm.qt1 : itm.qt0) * kTile, itm.bh);
          q_par ^= 1u << b;
          q_used |= 1u << b;
        }
        ++n_done;
        for (int j = itm.jb; j <= itm.je && ok; ++j) {
          for (int kv = 0; kv < 2; ++kv) {  // 0: K_j, 1: V_j
            ok = wait_bar<kInl, HOOK>(&bars->kv_empty[stage], phase ^ 1u, wc, kWFwdProdEmpty);
            if (!ok) break;
            const CUtensorMap* m = kv ? &tm_v : &tm_k;
            const int boxes = kv ? L::kSub : kQKBoxes;
            mbar_arrive_expect_tx(&bars->kv_full[stage],
                                  kv ? (uint32_t)L::kTileBytes : kQKBytes);
            for (int sb = 0; sb < boxes; ++sb)
              tma_load_3d(smem + L::kKVOff + stage * L::kTileBytes +
                              sb * kSubTileBytes,
                          m, &bars->kv_full[stage], sb * 64, j * kTile, itm.kvh);
            last_par[stage] = (int)phase;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // Stopping: let every copy this thread started land before exit.
        for (int b = 0; b < L::kQBufs; ++b)
          if ((q_used >> b) & 1u)
            drain_bar<kInl>(&bars->q_full[b], ((q_par >> b) & 1u) ^ 1u, a.timeout_ns);
        for (int s = 0; s < S; ++s)
          if (last_par[s] >= 0)
            drain_bar<kInl>(&bars->kv_full[s], (uint32_t)last_par[s], a.timeout_ns);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0 && run) {
      // Per-tile addresses are computed, not indexed, so that nothing of
      // this thread's state lives in local memory.
      const uint32_t q_base = smem_addr(smem + L::kQOff);
      const uint32_t kv_addr = smem_addr(smem + L::kKVOff);
      // Descriptors of every operand tile, fixed for the kernel's lifetime:
      // Q_t K-major; ring stage st read K-major (as K) or MN-major (as V).
      const uint64_t q_desc0 = sdesc_sw128(q_base, 16, 1024);
      const uint64_t kv_desc_k = sdesc_sw128(kv_addr, 16, 1024);
      const uint64_t kv_desc_v = sdesc_sw128(kv_addr, kSubTileBytes, 1024);
      auto q_desc = [&](int b) { return sdesc_adv(q_desc0, b * L::kTileBytes); };
      auto k_desc = [&](int st) { return sdesc_adv(kv_desc_k, st * L::kTileBytes); };
      auto v_desc = [&](int st) { return sdesc_adv(kv_desc_v, st * L::kTileBytes); };
      auto tS = [&](int t) { return tmem + (uint32_t)(t * 128); };
      auto tO = [&](int t) { return tmem + (uint32_t)(256 + t * D); };
      int stage = 0;
      uint32_t phase = 0;
      uint32_t q_par = 0;    // per Q buffer (bit b): parity of its next load
      uint32_t n_done = 0;   // items with work so far
      uint32_t p_cnt0 = 0, p_cnt1 = 0;
      bool ok = true;
      auto next_kv = [&](int& st) -> bool {
        st = stage;
        const bool rr = wait_bar<kInl, HOOK>(&bars->kv_full[stage], phase, wc, kWFwdMmaKV);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
        return rr;
      };
      // Q K^T for tile t (in Q buffer b) and key tile x; after the tile's
      // last one (hi_t), the buffer is released to the producer (in-order
      // completion).
      auto qk = [&](int t, int b, int x, int hi_t, int k_st) {
        if constexpr (FP8)
          issue_qk_fp8(tS(t), q_desc(b), k_desc(k_st));
        else
          issue_qk<D>(tS(t), q_desc(b), k_desc(k_st));
        mma_commit(&bars->s_full[t]);
        if (x == hi_t) mma_commit(&bars->q_empty[b]);
      };
      for (int ti = 0; ok; ++ti) {
        int w;
        ok = fwd_take<DYN>(bars, ti, false, wc, kWFwdMmaSched, w);
        if (!ok || w >= n_items) break;
        const FwdItem itm = fwd_item<CAUSAL, VARLEN>(w, n_tiles, n_pairs, a, tab);
        if (VARLEN && itm.hi0 < 0) continue;  // empty item (alternating rounds)
        auto act0 = [&](int x) { return x <= itm.hi0; };  // x >= lo0 = jb
        auto act1 = [&](int x) { return x >= itm.lo1 && x <= itm.hi1; };
        const int qb0 = WINDOW ? 0 : q_buf(n_done, 0);
        const int qb1 = WINDOW ? 1 : q_buf(n_done, 1);
        ++n_done;
        ok = wait_bar<kInl, HOOK>(&bars->q_full[qb0], (q_par >> qb0) & 1u, wc, kWFwdMmaQ);
        q_par ^= 1u << qb0;
        if (ok && itm.hi1 >= 0) {
          ok = wait_bar<kInl, HOOK>(&bars->q_full[qb1], (q_par >> qb1) & 1u, wc, kWFwdMmaQ);
          q_par ^= 1u << qb1;
        }
        int k_stage = 0;
        if (ok) ok = next_kv(k_stage);
        if (!ok) break;
        tc_fence_after();
        qk(0, qb0, itm.jb, itm.hi0, k_stage);
        if (act1(itm.jb)) qk(1, qb1, itm.jb, itm.hi1, k_stage);
        mma_commit(&bars->kv_empty[k_stage]);
        for (int j = itm.jb; j <= itm.je && ok; ++j) {
          int v_stage = 0;
          ok = next_kv(v_stage);
          if (!ok) break;
          tc_fence_after();
          const uint64_t vd = v_desc(v_stage);
          int kn_stage = -1;
          // Tile 0: P V for key tile j, then Q K^T for key tile j+1.
          if (act0(j)) {
            ok = wait_bar<kInl, HOOK>(&bars->p_full[0], p_cnt0 & 1u, wc, kWFwdMmaP);
            ++p_cnt0;
            if (!ok) break;
            tc_fence_after();
            issue_pv<D>(tO(0), tS(0), vd, j > itm.lo0);
          }
          if (j < itm.je) {
            ok = next_kv(kn_stage);
            if (!ok) break;
            tc_fence_after();
          }
          if (act0(j + 1))
            qk(0, qb0, j + 1, itm.hi0, kn_stage);
          else if (j == itm.hi0)
            mma_commit(&bars->o_done[0]);
          // Tile 1: the same; V_j is released after both tiles used it.
          if (act1(j)) {
            ok = wait_bar<kInl, HOOK>(&bars->p_full[1], p_cnt1 & 1u, wc, kWFwdMmaP);
            ++p_cnt1;
            if (!ok) break;
            tc_fence_after();
            issue_pv<D>(tO(1), tS(1), vd, j > itm.lo1);
          }
          mma_commit(&bars->kv_empty[v_stage]);
          if (act1(j + 1))
            qk(1, qb1, j + 1, itm.hi1, kn_stage);
          else if (j == itm.hi1)
            mma_commit(&bars->o_done[1]);
          if (kn_stage >= 0) mma_commit(&bars->kv_empty[kn_stage]);
        }
      }
      // Every MMA issued above must finish before TMEM is released.
      mma_commit(&bars->mma_done);
      drain_bar<kInl>(&bars->mma_done, 0, a.timeout_ns);
    }
  } else if (warp < 8) {
    // ------------------------------------------------- softmax (thread = row)
    if constexpr (kSplitRegs) reg_alloc<kSoftmaxRegs>();
    const int t = warp >> 2, quarter = warp & 3;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t tS = tl + t * 128;
    const uint32_t tO = tl + 256 + t * D;
    const float c = a.scale_log2;
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ostg_pending = false;  // this warp's O box is being stored
    bool ok = run;
    for (int ti = 0; ok; ++ti) {
      int w;
      ok = fwd_take<DYN>(bars, ti, true, wc, kWFwdSmSched, w);
      if (!ok || w >= n_items) break;
      const FwdItem itm = fwd_item<CAUSAL, VARLEN>(w, n_tiles, n_pairs, a, tab);
      const int lo_t = t ? itm.lo1 : itm.lo0;
      const int hi_t = t ? itm.hi1 : itm.hi0;
      if (hi_t < 0) continue;
      const int q0 = (t ? itm.qt1 : itm.qt0) * kTile;
      const int qrow = q0 + quarter * 32 + lane;
      // Visible keys of a row: j <= i (causal), |i - j| <= window, j < N.
      // Without a window only the last key tile can need the mask (the
      // diagonal, or keys past a ragged N).  With one, a key tile needs it
      // if it reaches below the Q tile's largest lower bound or above its
      // smallest upper bound; the window is below N, so none of these sums
      // overflows.
      // Everything the masks need is derived here, once per item, so that
      // the loop keeps as few values live as possible: without a window,
      // the last tile's bound (uniform over the warp without causality);
      // with one, the row's own visible key range.
      const int win = a.window, nm1 = itm.len - 1;
      const int klo_max = WINDOW ? q0 + kTile - 1 - win : -1;
      const int khi_min =
          CAUSAL ? q0 : (WINDOW ? (q0 > nm1 - win ? nm1 : q0 + win) : nm1);
      const int lim_last = (CAUSAL ? qrow : nm1) - hi_t * kTile;
      const int row_lo = qrow > win ? qrow - win : 0;
      const int row_hi = CAUSAL ? qrow : (qrow > nm1 - win ? nm1 : qrow + win);
      // FP8: scores are in units of sq(row block) * sk(key block); the row's
      // factor is folded into its exponent scale.
      float cr = c;
      if constexpr (FP8) cr = c * a.q_scale[(size_t)itm.bh * a.n_sblk + (qrow >> 4)];
      float m_ref = -INFINITY, l = 0.f;
      for (int j = lo_t; j <= hi_t; ++j) {
        float4 ska, skb;  // FP8: the 8 key-block scales of tile j
        if constexpr (FP8) {
          const float4* ks = reinterpret_cast<const float4*>(
              a.k_scale + (size_t)itm.kvh * a.n_sblk + (size_t)j * 8);
          ska = ks[0];
          skb = ks[1];
        }
        ok = wait_bar_warp<kInl>(&bars->s_full[t], s_cnt & 1u, wc, kWFwdSmS);
        ++s_cnt;
        if (!ok) break;
        tc_fence_after();
        uint32_t s[128];
        tmem_ld32(tS + 0, s);
        tmem_ld32(tS + 32, s + 32);
        tmem_ld32(tS + 64, s + 64);
        tmem_ld32(tS + 96, s + 96);
        tmem_wait_ld();
        reg_fence32(s);
        reg_fence32(s + 32);
        reg_fence32(s + 64);
        reg_fence32(s + 96);
        if constexpr (!WINDOW) {
          if (j == hi_t && (CAUSAL || lim_last < kTile - 1)) {
#pragma unroll
            for (int e = 0; e < 128; ++e)
              if (e > lim_last) s[e] = __float_as_uint(-INFINITY);
          }
        } else {
          const int kb = j * kTile;
          if (kb < klo_max || kb + kTile - 1 > khi_min) {
            const int e_lo = row_lo - kb, e_hi = row_hi - kb;
#pragma unroll
            for (int e = 0; e < 128; ++e)
              if (e < e_lo || e > e_hi) s[e] = __float_as_uint(-INFINITY);
          }
        }
        // Row max: four independent chains of three-input maxima (one long
        // dependent chain dominated the softmax latency).  FP8: one maximum
        // per 16-key group, each times its positive scale.
        float m_tile;
        float w[8];  // FP8: exponent scale of each 16-key group
        if constexpr (!FP8) {
          float mx4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mx4[k] = fmaxf(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1]));
#pragma unroll
          for (int e = 8; e < 128; e += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mx4[k] = max3(mx4[k], __uint_as_float(s[e + 2 * k]),
                            __uint_as_float(s[e + 2 * k + 1]));
          const float mx = max3(max3(mx4[0], mx4[1], mx4[2]), mx4[3], mx4[3]);
          m_tile = mx * c;
        } else {
          w[0] = cr * ska.x; w[1] = cr * ska.y; w[2] = cr * ska.z; w[3] = cr * ska.w;
          w[4] = cr * skb.x; w[5] = cr * skb.y; w[6] = cr * skb.z; w[7] = cr * skb.w;
          float mg[8];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            float m = fmaxf(__uint_as_float(s[16 * g]), __uint_as_float(s[16 * g + 1]));
#pragma unroll
            for (int e = 16 * g + 2; e < 16 * g + 16; e += 2)
              m = max3(m, __uint_as_float(s[e]), __uint_as_float(s[e + 1]));
            mg[g] = m * w[g];
          }
          m_tile = max3(max3(mg[0], mg[1], mg[2]), max3(mg[3], mg[4], mg[5]),
                        fmaxf(mg[6], mg[7]));
        }
        // Lazy rescale: keep the reference max until the row max exceeds it
        // by more than the threshold; exp2(x - m_ref) <= 2^8 meanwhile.
        const bool bump = m_tile > m_ref + kRescaleThreshold;
        float alpha = 1.f;
        if (bump) {
          alpha = ex2(m_ref - m_tile);
          m_ref = m_tile;
        }
        l *= alpha;
        // With a window a row may have seen no visible key yet (m_ref =
        // -inf): its P is 0, not exp2(-inf + inf).
        float neg_m = -m_ref;
        if constexpr (WINDOW) neg_m = (m_ref == -INFINITY) ? 0.f : neg_m;
        const uint64_t c2 = bcast2(c), nm2 = bcast2(neg_m);
        uint64_t w2[8];
        if constexpr (FP8) {
#pragma unroll
          for (int g = 0; g < 8; ++g) w2[g] = bcast2(w[g]);
        }
        // Scores to exponents two at a time (packed fp32 FMA), row sum in
        // four packed partial sums; P is packed in place: pair (e, e+1) goes
        // to s[e/2], a slot whose score has already been consumed.
        float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 128; e += 2) {
          float x0, x1;
          fma2_bcast(x0, x1, __uint_as_float(s[e]), __uint_as_float(s[e + 1]),
                     FP8 ? w2[e / 16] : c2, nm2);
          const float p0 = ex2(x0), p1 = ex2(x1);
          add2_acc(la[(e >> 1) & 3], lb[(e >> 1) & 3], p0, p1);
          s[e / 2] = pack_bf16(p0, p1);
        }
        l += ((la[0] + lb[0]) + (la[1] + lb[1])) + ((la[2] + lb[2]) + (la[3] + lb[3]));
        tmem_st32(tS + 0, s);
        tmem_st32(tS + 32, s + 32);
        if (j > lo_t && __any_sync(0xffffffffu, bump)) {
          // Rescale O_t, which holds P V for tiles < j (the S_t(j) commit
          // came after them); done after P is stored so that the scores are
          // no longer live.  P V for tile j waits for p_full below.
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32(tO + ch * 32, o);
            tmem_wait_ld();
            reg_fence32(o);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + ch * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&bars->p_full[t]);
      }
      if (!ok) break;
      ok = wait_bar_warp<kInl>(&bars->o_done[t], o_cnt & 1u, wc, kWFwdSmO);
      ++o_cnt;
      if (!ok) break;
      tc_fence_after();
      const float inv_l = 1.0f / l;
      // The length is read again rather than kept live through the loop.
      const bool valid =
          qrow < (VARLEN ? seq_len_of(a.seq_lens, itm.bh / a.H, a.N) : a.N);
      if constexpr (OSTG) {
        // 64 columns at a time: the row goes into this warp's box (row =
        // lane, 16-byte pieces in the 128-byte swizzle) and the box leaves
        // by TMA store, which clips rows past N.  The box is rewritten only
        // after the previous store has read it.
        uint8_t* const box = smem + L::kOStgOff + warp * L::kOStgBoxBytes;
        uint8_t* const brow = box + lane * 128;
#pragma unroll 1
        for (int hb = 0; hb < D / 64; ++hb) {
          if (ostg_pending) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + hb * 64 + c * 32, o);
            tmem_wait_ld();
            reg_fence32(o);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv_l,
                                __uint_as_float(o[2 * e + 1]) * inv_l);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              *reinterpret_cast<uint4*>(brow + (((c * 4 + v4) ^ (lane & 7)) * 16)) =
                  make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tm_o, box, hb * 64, q0 + quarter * 32, itm.bh);
            bulk_commit_group();
          }
          ostg_pending = true;
        }
      } else {
        __nv_bfloat16* orow = a.o + ((size_t)itm.bh * a.N + (valid ? qrow : 0)) * D;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(tO + ch * 32, o);
          tmem_wait_ld();
          reg_fence32(o);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv_l,
                              __uint_as_float(o[2 * e + 1]) * inv_l);
          if (valid) {
            if (a.o_wide) {  // whole 32-byte sectors (rows are d * 2 bytes apart)
              st_global_v8(orow + ch * 32, pk);
              st_global_v8(orow + ch * 32 + 16, pk + 8);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2],
                                     pk[4 * v4 + 3]);
            }
          }
        }
      }
      if (valid) a.lse[(size_t)itm.bh * a.N + qrow] = (m_ref + lg2(l)) * kLn2;
      // The next item's first P V (which overwrites O_t) is issued only after
      // this warp group's next p_full arrival, so O_t is read out first.
      tc_fence_before();
    }
    // O stores complete (and done reading shared memory) before exit.
    if (OSTG && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // Every block has stopped claiming; the last one out resets the counter.
  if (DYN && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.work_done, 1u) == gridDim.x - 1) {
      atomicExch(a.work_next, 0u);
      atomicExch(a.work_done, 0u);
    }
  }
}

template <int D, bool CAUSAL, bool WINDOW, bool FP8, bool VARLEN = false,
          bool DYN = false, bool HOOK = false>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& to,
                         const FwdArgs& a, int BH, int grid_blocks,
                         cudaStream_t stream) {
  using L = FwdLayout<D, WINDOW ? 2 : 3, fwd_ostg<WINDOW, FP8, VARLEN, DYN>()>;
  static_assert(!VARLEN || (WINDOW && !FP8), "lengths run windowed, bf16");
  static_assert(!DYN || !WINDOW, "banded calls use the alternating rounds");
  // The failure-path test hook has its own instantiation, for d = 128 bf16
  // without a window, lengths or the dynamic schedule only.
  if constexpr (D == 128 && !WINDOW && !FP8 && !VARLEN && !DYN && !HOOK) {
    if (a.hook)
      return launch_fwd_t<D, CAUSAL, WINDOW, FP8, VARLEN, false, true>(
          tq, tk, tv, to, a, BH, grid_blocks, stream);
  }
  // The dynamic schedule exists only without a window: the host asks for it
  // (a.dynamic) only there.
  if constexpr (!WINDOW && !DYN && !HOOK) {
    if (a.dynamic)
      return launch_fwd_t<D, CAUSAL, WINDOW, FP8, VARLEN, true>(tq, tk, tv, to, a, BH,
                                                              grid_blocks, stream);
  }
  auto kern = fwd_kernel<D, CAUSAL, WINDOW, FP8, VARLEN, DYN, HOOK>;
  cudaError_t e;
  if constexpr (kSplitRegs) {
    // The register split inside the kernel assumes exactly kLaunchRegs per
    // thread at launch; with fewer the softmax groups' setmaxnreg.inc could
    // never be granted, so such a build is refused here.
    cudaFuncAttributes fa_attr{};
    e = cudaFuncGetAttributes(&fa_attr, kern);
    if (e != cudaSuccess) return e;
    if (fa_attr.numRegs != kLaunchRegs) return cudaErrorInvalidKernelImage;
  }
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const int n_pairs = a.single ? n_tiles : (n_tiles + 1) / 2;
  FwdArgs args = a;
  size_t smem_bytes = L::kSmemBytes;
  args.sched = 0;
  if constexpr (VARLEN) {
    // The balanced item table (np, order: B ints each; pref: groups + 1;
    // sort bins: pairs + 1) when it fits in the shared memory left by the
    // tiles.
    const long long B = a.BH / a.H;
    const long long groups = CAUSAL ? n_pairs : B;
    const long long table = 4 * (2 * B + groups + 1 + n_pairs + 1);
    int dev = 0, optin = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&optin,
                                 cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    if ((long long)L::kSmemBytes + table <= optin) {
      smem_bytes = L::kSmemBytes + (size_t)table;
      args.sched = 1;
    }
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_bytes);
  if (e != cudaSuccess) return e;
  const int n_items = BH * n_pairs;
  const int blocks = n_items < grid_blocks ? n_items : grid_blocks;
  kern<<<blocks, kFwdThreads, smem_bytes, stream>>>(tq, tk, tv, to, args);
  return cudaGetLastError();
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_w(const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& to,
                         const FwdArgs& a, int BH, int grid_blocks,
                         cudaStream_t stream) {
  if (a.seq_lens)  // the host passes a window (N - 1 at widest) with lengths
    return a.window >= 0
               ? launch_fwd_t<D, CAUSAL, true, false, true>(tq, tk, tv, to, a, BH, grid_blocks, stream)
               : cudaErrorInvalidValue;
  return a.window >= 0
             ? launch_fwd_t<D, CAUSAL, true, false>(tq, tk, tv, to, a, BH, grid_blocks, stream)
             : launch_fwd_t<D, CAUSAL, false, false>(tq, tk, tv, to, a, BH, grid_blocks, stream);
}

// E4M3 quantisation, one warp per 16-row block of one head: amax of the
// block, scale = amax / 448 (1 for an all-zero block), codes = round to
// nearest even of x / scale with saturation.  Both divisions are IEEE
// round-to-nearest, so the codes are those of the same float32 arithmetic
// anywhere.  Lane l holds columns [l*D/32, (l+1)*D/32) of every row.  Code
// rows are `pitch` bytes apart (pitch >= D); bytes D .. pitch - 1 of a row
// are written as zero (the FP8 forward pads d = 64 rows to 128 bytes).
template <int D>
__global__ void __launch_bounds__(256) quant_e4m3_kernel(
    const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
    float* __restrict__ scales, int BH, int N, int n_sblk, int pitch) {
  constexpr int kPer = D / 32;
  const int lane = threadIdx.x & 31;
  const long long n_blk = (long long)BH * n_sblk;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long blk = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       blk < n_blk; blk += warps) {
    const int bh = (int)(blk / n_sblk);
    const int r0 = (int)(blk - (long long)bh * n_sblk) * 16;
    const int rows = N - r0 < 16 ? N - r0 : 16;
    if (rows <= 0) {  // padding block past N
      if (lane == 0) scales[blk] = 1.0f;
      continue;
    }
    const size_t base = ((size_t)bh * N + r0) * D + lane * kPer;
    const size_t cbase = ((size_t)bh * N + r0) * pitch + lane * kPer;
    float v[16][kPer];
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      if (r < rows) {
        if constexpr (kPer == 4) {
          const uint2 u = *reinterpret_cast<const uint2*>(x + base + (size_t)r * D);
          v[r][0] = bf16_lo(u.x); v[r][1] = bf16_hi(u.x);
          v[r][2] = bf16_lo(u.y); v[r][3] = bf16_hi(u.y);
        } else {
          const uint32_t u = *reinterpret_cast<const uint32_t*>(x + base + (size_t)r * D);
          v[r][0] = bf16_lo(u); v[r][1] = bf16_hi(u);
        }
      } else {
#pragma unroll
        for (int e = 0; e < kPer; ++e) v[r][e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < kPer; ++e) amax = fmaxf(amax, fabsf(v[r][e]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      if (r >= rows) break;
      uint8_t* dst = codes + cbase + (size_t)r * pitch;
      for (int c = D; c < pitch; c += 32 * kPer)  // zero padding of the row
        for (int e = 0; e < kPer; ++e) dst[c + e] = 0;
      if constexpr (kPer == 4) {
        const uint32_t lo = pack_e4m3(__fdiv_rn(v[r][0], sc), __fdiv_rn(v[r][1], sc));
        const uint32_t hi = pack_e4m3(__fdiv_rn(v[r][2], sc), __fdiv_rn(v[r][3], sc));
        *reinterpret_cast<uint32_t*>(dst) = lo | (hi << 16);
      } else {
        *reinterpret_cast<uint16_t*>(dst) =
            pack_e4m3(__fdiv_rn(v[r][0], sc), __fdiv_rn(v[r][1], sc));
      }
    }
    if (lane == 0) scales[blk] = sc;
  }
}

}  // namespace

cudaError_t launch_quant_e4m3(const __nv_bfloat16* x, uint8_t* codes,
                              float* scales, int BH, int N, int d, int n_sblk,
                              int pitch, int grid_blocks, cudaStream_t stream) {
  if (d == 128)
    quant_e4m3_kernel<128><<<grid_blocks, 256, 0, stream>>>(x, codes, scales, BH, N,
                                                           n_sblk, pitch);
  else
    quant_e4m3_kernel<64><<<grid_blocks, 256, 0, stream>>>(x, codes, scales, BH, N,
                                                          n_sblk, pitch);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to,
                           const FwdArgs& a, int BH, int d, bool causal,
                           int grid_blocks, cudaStream_t stream) {
  if (d == 64)
    return causal ? launch_fwd_t<64, true, false, true>(tq, tk, tv, to, a, BH, grid_blocks, stream)
                  : launch_fwd_t<64, false, false, true>(tq, tk, tv, to, a, BH, grid_blocks, stream);
  return causal ? launch_fwd_t<128, true, false, true>(tq, tk, tv, to, a, BH, grid_blocks, stream)
                : launch_fwd_t<128, false, false, true>(tq, tk, tv, to, a, BH, grid_blocks, stream);
}

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to,
                       const FwdArgs& a, int BH, int d, bool causal,
                       int grid_blocks, cudaStream_t stream) {
  if (d == 128)
    return causal ? launch_fwd_w<128, true>(tq, tk, tv, to, a, BH, grid_blocks, stream)
                  : launch_fwd_w<128, false>(tq, tk, tv, to, a, BH, grid_blocks, stream);
  return causal ? launch_fwd_w<64, true>(tq, tk, tv, to, a, BH, grid_blocks, stream)
                : launch_fwd_w<64, false>(tq, tk, tv, to, a, BH, grid_blocks, stream);
}

cudaError_t set_expire_site_fwd(uint32_t site) {
  return cudaMemcpyToSymbol(c_expire_site, &site, sizeof(site));
}

}  // namespace fa
