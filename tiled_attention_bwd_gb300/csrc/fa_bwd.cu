// fa_bwd.cu -- backward attention kernels for sm_103a.
//
// Gradients of O = softmax(scale Q K^T [+ mask]) V with P recomputed from the
// saved LSE instead of stored ("GPU Performance Optimization Batch 1 -- Design
// Spec", Item 3, backward paragraph; "RTX Flash Attention Implementation
// COMPLETE", "Flash Attention Backward Kernel": gradient recomputation,
// atomic memory operations, dQ/dK/dV updates).  With D_i = dO_i . O_i:
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  dQ = scale dS K,
//   dK = scale dS^T Q.
//
// Three launches on one stream:
//   pre   D_i and LSE2_i = -LSE_i*log2(e) per row (padded to whole tiles:
//         D = 0 and LSE2 = -inf past N, which zeroes P there); dQ
//         accumulator := 0.
//   main  persistent, one thread block per SM walking work items (batch,
//         head, 128-key tile j).  K_j, V_j stay
//         in smem; dK_j, dV_j accumulate in TMEM; Q_i (two stages) and dO_i
//         (one buffer) stream in by TMA (causal: only i >= j).  Per Q tile, five tcgen05
//         MMAs: S^T = K Q^T, dP^T = V dO^T, dV += P^T dO (P^T from TMEM),
//         dK += dS^T Q (dS^T from TMEM) and dQ_i = dS K (dS from smem, read
//         MN-major).  dQ_i leaves TMEM and is added into the fp32
//         accumulator by TMA reduce-add.
//   post  dQ = scale * accumulator, rounded to bf16.
//
// Warps of the main kernel:
//   0-3  thread = key row: P^T = exp2(S^T c + LSE2), then dS^T = P^T (dP^T - D);
//        at the end of an item the dK_j read-out, staged in the dS tile and
//        sent by TMA store
//   4-7  thread = query row: drain dQ_i from TMEM, stage it box by box
//        through two 4 KB boxes per warp and add it into the fp32
//        accumulator with TMA reduce-add; at the end of an item the dV_j
//        read-out, staged in the same boxes and sent by TMA store
//   8    TMA producer,  9  MMA issuer (one thread) and TMEM owner.
// TMEM columns (512 allocated): S^T/P^T [0,128)  dP^T, then dS^T (bf16
// pairs in [128,192)), then dQ [128,256)  dK [256, 256+d)  dV [256+d, 256+2d).
// Measured on this part: issued back to back, every MMA form runs at the
// full tensor rate; on a dependent chain (each product waiting for the one
// before) one with both operands in smem takes about 2.4 times as long as
// one with A in TMEM.  So every product whose A operand can live in TMEM
// takes it from there.
#include <climits>

#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

constexpr int kBwdThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;

template <int D>
struct BwdLayout {
  static constexpr int kSub = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  // Two Q stages, each Q_i followed by LSE2_i[128] and D_i[128] (fp32).
  static constexpr int kQOff = 2 * kTileBytes;
  static constexpr int kQStageBytes = kTileBytes + 2 * kTile * 4;
  // One dO buffer: dO_i is free once dV_i is done and dO_{i+1} is first
  // needed one dK/dQ pair later.
  static constexpr int kDOOff = kQOff + 2 * kQStageBytes;
  static constexpr int kDSOff = kDOOff + kTileBytes;
  static constexpr int kDSBytes = kTile * kTile * 2;  // 2 sub-tiles [128][64]
  // dQ staging: per drain warp two [32 rows][32 fp32] boxes of 4 KB, used
  // alternately (4 warps x 2 x 4 KB).
  static constexpr int kStgOff = kDSOff + kDSBytes;
  static constexpr int kStgBoxBytes = 32 * 128;
  static constexpr int kBarOff = kStgOff + 8 * kStgBoxBytes;
  // d = 128 uses 231,680 of the 232,448 bytes a block may have, so the base
  // is taken as is (checked at run time); d = 64 keeps alignment slack.
  static constexpr int kSlack = (D == 128) ? 0 : 1024;
  static constexpr int kSmemBytes = kBarOff + 256 + kSlack;
};

struct BwdBars {
  uint64_t k_full;      // K_j of the block's current work item landed
  uint64_t v_full;      // V_j landed
  uint64_t k_empty;     // the item's last MMA reading K_j is done
  uint64_t v_empty;     // the item's last MMA reading V_j is done
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t do_full;
  uint64_t do_empty;
  uint64_t s_full;
  uint64_t dp_full;
  uint64_t p_full;
  uint64_t ds_full;
  uint64_t dq_full;
  uint64_t dq_free;
  uint64_t ds_free;
  uint64_t acc_done;    // the item's dK_j, dV_j are complete in TMEM
  uint64_t acc_free;    // ... and have been read out (8 warps arrive)
  uint64_t mma_done;
  uint64_t sched_full[2];   // work item t published in sched_item[t % 2]
  uint64_t sched_empty[2];  // ... and read by the MMA thread and 8 warps
  int sched_item[2];
  uint32_t tmem_base;
  uint32_t abort;
};

enum : uint32_t {
  kWBwdProdQEmpty = 0x111,
  kWBwdProdDoEmpty = 0x112,
  kWBwdProdKEmpty = 0x113,
  kWBwdProdVEmpty = 0x114,
  kWBwdProdSched = 0x115,
  kWBwdMmaSched = 0x218,
  kWBwdCmpSched = 0x316,
  kWBwdDqSched = 0x413,
  kWBwdMmaAccFree = 0x217,
  kWBwdMmaKV = 0x211,
  kWBwdMmaQ = 0x212,
  kWBwdMmaDqFree = 0x213,
  kWBwdMmaP = 0x214,
  kWBwdMmaDs = 0x215,
  kWBwdMmaDo = 0x216,
  kWBwdCmpQ = 0x311,
  kWBwdCmpS = 0x312,
  kWBwdCmpDp = 0x313,
  kWBwdCmpDsFree = 0x314,
  kWBwdCmpAcc = 0x315,
  kWBwdDqFull = 0x411,
  kWBwdDqAcc = 0x412,
  kWBwdMisaligned = 0x5A1,
};

// The usual dK / dV epilogue: this thread's row of the TMEM accumulator at
// column `tcol`, times `mul`, rounded to bf16 into a staging tile in shared
// memory laid out as the TMA writes it (64-column sub-tiles `sub_stride`
// bytes apart, 128-byte rows in the 128-byte swizzle, row `srow` of the
// tile; a warp's 32 rows form one [32 x 64] box per sub-tile), from where
// the warp's TMA stores send whole lines to global memory.  Per-thread
// 16-byte stores of rows 2d bytes apart (the earlier form) kept the
// load/store pipe busy for thousands of cycles per item and delayed the next
// item's first P^T behind them.
template <int D>
__device__ __forceinline__ void kv_epilogue_stage(uint32_t tcol, uint8_t* tile,
                                                  uint32_t sub_stride,
                                                  uint32_t srow, float mul) {
#pragma unroll 1
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t v[32];
    tmem_ld32(tcol + ch * 32, v);
    tmem_wait_ld();
    reg_fence32(v);
    uint8_t* sub = tile + (ch >> 1) * sub_stride;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t col = (uint32_t)((ch & 1) * 32 + k * 8);
      *reinterpret_cast<uint4*>(sub + sw128_offset(srow, col)) = make_uint4(
          pack_bf16(__uint_as_float(v[8 * k + 0]) * mul, __uint_as_float(v[8 * k + 1]) * mul),
          pack_bf16(__uint_as_float(v[8 * k + 2]) * mul, __uint_as_float(v[8 * k + 3]) * mul),
          pack_bf16(__uint_as_float(v[8 * k + 4]) * mul, __uint_as_float(v[8 * k + 5]) * mul),
          pack_bf16(__uint_as_float(v[8 * k + 6]) * mul, __uint_as_float(v[8 * k + 7]) * mul));
    }
  }
}

// Row `krow` of dK or dV (key/value head bkv) from the TMEM accumulator at
// column `tcol` (this thread's lane), times `mul`, added in fp32 into `acc`
// (vector atomics; rounded later by the post kernel): the epilogue when the
// group's query heads are split over several blocks.  Rows at or past `len`
// (the sequence's length) are not written.
template <int D>
__device__ __forceinline__ void kv_epilogue_atomic(uint32_t tcol, float* acc,
                                                   int bkv, int krow, int N,
                                                   int len, float mul) {
  const bool valid = krow < len;
  const size_t row = (size_t)bkv * N + (valid ? krow : 0);
#pragma unroll 1
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t v[32];
    tmem_ld32(tcol + ch * 32, v);
    tmem_wait_ld();
    reg_fence32(v);
    if (!valid) continue;
    float4* dst = reinterpret_cast<float4*>(acc + row * D + ch * 32);
#pragma unroll
    for (int v4 = 0; v4 < 8; ++v4)
      atomicAdd(dst + v4, make_float4(__uint_as_float(v[4 * v4]) * mul,
                                      __uint_as_float(v[4 * v4 + 1]) * mul,
                                      __uint_as_float(v[4 * v4 + 2]) * mul,
                                      __uint_as_float(v[4 * v4 + 3]) * mul));
  }
}

// One work item of the main kernel: key tile j of key/value head bkv (one
// split of its query heads when the group is split), visiting nq (query head,
// query tile) pairs: query heads qh0 .. qh0 + hpb - 1, each over query tiles
// i_lo .. i_hi (the tiles whose band reaches key tile j).
struct BwdItem {
  int bkv, j, qh0, i_lo, i_hi, nq, len;
};

// Work item w in the schedule order.  Blocks resident together share a few
// key/value heads, so their Q/dO tiles and dQ accumulator rows stay in L2;
// causal key tile 0 (the most query tiles) of each head comes first.
//
// A block owns key tile j of key/value head bkv and visits, for each of the
// H / Hkv query heads that read that head, the query tiles whose band
// reaches tile j (query i sees key k when k <= i if causal and |i - k| <=
// window if a window is set); iteration `it` is query head it / nq_head of
// the group and query tile i_lo + it % nq_head.
//
// With many query heads per key/value head (multi-query attention) one item
// per (key/value head, key tile) is too coarse: the group's query heads are
// then dealt to nsplit items of hpb heads each, whose partial dK_j, dV_j are
// summed in fp32 (dk_acc, dv_acc) and rounded afterwards.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ BwdItem bwd_item(int w, int n_tiles, const BwdArgs& a) {
  BwdItem itm;
  const TileSlot slot = grouped_slot(w, n_tiles, a.BHkv * a.nsplit, a.group);
  itm.bkv = slot.bh / a.nsplit;
  const int split = slot.bh - itm.bkv * a.nsplit;
  itm.j = slot.tile;
  const int qgroup = a.H / a.Hkv;
  itm.qh0 = (itm.bkv / a.Hkv) * a.H + (itm.bkv % a.Hkv) * qgroup + split * a.hpb;
  // With per-sequence lengths (the VARLEN instantiations; the others keep
  // none of this arithmetic) only the sequence's own tiles count: a key tile
  // at or past its end gives the item no work (nq = 0).
  itm.len = VARLEN ? seq_len_of(a.seq_lens, itm.bkv / a.Hkv, a.N) : a.N;
  const int tiles_b = VARLEN ? (itm.len + kTile - 1) / kTile : n_tiles;
  const long long k0 = (long long)itm.j * kTile, k1 = k0 + kTile - 1;
  itm.i_lo = CAUSAL ? itm.j : ((a.window >= 0 && k0 > a.window)
                                   ? (int)((k0 - a.window) / kTile) : 0);
  itm.i_hi = tiles_b - 1;
  if (a.window >= 0) {
    const long long h = (k1 + a.window) / kTile;
    if (h < itm.i_hi) itm.i_hi = (int)h;
  }
  itm.nq = (!VARLEN || (itm.j < tiles_b && itm.i_hi >= itm.i_lo))
               ? a.hpb * (itm.i_hi - itm.i_lo + 1) : 0;
  return itm;
}

// Work items are handed out dynamically: block b starts with item b and then
// takes the next unclaimed one from a counter in the workspace (zeroed by the
// pre kernel), so blocks that drew light items take more of them and all
// finish together.  Within a head group the items come heaviest first, and
// the last items of the whole order are the lightest.  The block's producer
// thread claims the items and publishes each in a two-slot ring in shared
// memory, which the other roles read in the same order.

// Item t of this block as published by the producer (n_items or more: none
// left).  Every thread of the calling warp waits and reads; one arrives.
template <bool kWarp>
__device__ __forceinline__ bool sched_take(BwdBars* bars, int t, const WaitCtl& wc,
                                           uint32_t where, int& w) {
  const int sl = t & 1;
  const uint32_t par = (uint32_t)(t >> 1) & 1u;
  const bool ok = kWarp ? wait_bar_warp(&bars->sched_full[sl], par, wc, where)
                        : wait_bar(&bars->sched_full[sl], par, wc, where);
  if (!ok) return false;
  w = *reinterpret_cast<volatile int*>(&bars->sched_item[sl]);
  if (kWarp) warp_arrive(&bars->sched_empty[sl]);
  else mbar_arrive(&bars->sched_empty[sl]);
  return true;
}

// Walks (query head, query tile) in iteration order without divisions.
struct QCursor {
  int bh, i;
};
__device__ __forceinline__ void q_next(QCursor& c, const BwdItem& itm) {
  if (++c.i > itm.i_hi) {
    c.i = itm.i_lo;
    ++c.bh;
  }
}

// Persistent: one block per SM takes work items one after another.  The
// barrier phases run on across items (`g` counts the block's query-tile
// iterations, `t` its items), so the next item's V, first Q and
// dO tiles load while the current one finishes, its K as soon as the last
// MMA reading K_j is done, and its first S^T / dP^T overlap the read-out of
// the current dK_j, dV_j.
template <int D, bool CAUSAL, bool VARLEN, bool HOOK>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq,
                    const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv,
                    const BwdArgs a) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (L::kSlack > 0) ? align1024(smem_raw) : smem_raw;
  auto* bars = reinterpret_cast<BwdBars*>(smem + L::kBarOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const int n_items = a.BHkv * a.nsplit * n_tiles;

  if (threadIdx.x == 0) {
    uint32_t stop = *reinterpret_cast<volatile unsigned int*>(&a.st->abort);
    if ((smem_addr(smem) & 1023u) != 0) {
      atomicCAS(&a.st->status, 0u, (unsigned)FA_ERR_UNSUPPORTED);
      atomicExch(&a.st->where, kWBwdMisaligned);
      stop = 1;
    }
    bars->abort = stop;
    mbar_init(&bars->k_full, 1);
    mbar_init(&bars->v_full, 1);
    mbar_init(&bars->k_empty, 1);
    mbar_init(&bars->v_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    mbar_init(&bars->do_full, 1);
    mbar_init(&bars->do_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 4);    // one arrival per warp
    mbar_init(&bars->ds_full, 4);   // one arrival per warp
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 4);   // one arrival per warp
    mbar_init(&bars->ds_free, 1);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->acc_free, 8);  // dK by warps 0-3, dV by warps 4-7
    mbar_init(&bars->mma_done, 1);
    for (int sl = 0; sl < 2; ++sl) {
      mbar_init(&bars->sched_full[sl], 1);
      mbar_init(&bars->sched_empty[sl], 9);  // MMA thread + 8 warps
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
  uint8_t* const k_s = smem + L::kKOff;
  uint8_t* const v_s = smem + L::kVOff;
  uint8_t* const do_s = smem + L::kDOOff;
  uint8_t* const ds_s = smem + L::kDSOff;
  uint8_t* const stg_s = smem + L::kStgOff;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0 && run) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      prefetch_tmap(&tm_dq);
      prefetch_tmap(&tm_dk);
      prefetch_tmap(&tm_dv);
      // Parity of the last load issued into each buffer (-1: none), so that
      // a stopping block can wait for its copies in flight.
      int k_par = -1, v_par = -1, q_par[2] = {-1, -1}, do_par = -1;
      bool ok = true;
      uint32_t g = 0;
      int w = (int)blockIdx.x;
      for (int t = 0; ok; ++t) {
        // Claim the next item with work (with per-sequence lengths some have
        // none) and publish it; n_items or more tells the others to stop.
        if (t > 0) w = (int)gridDim.x + (int)atomicAdd(a.work_next, 1u);
        BwdItem itm;
        while (w < n_items) {
          itm = bwd_item<CAUSAL, VARLEN>(w, n_tiles, a);
          if (!VARLEN || itm.nq > 0) break;
          w = (int)gridDim.x + (int)atomicAdd(a.work_next, 1u);
        }
        ok = wait_bar<false, HOOK>(&bars->sched_empty[t & 1], ((uint32_t)(t >> 1) & 1u) ^ 1u, wc,
                      kWBwdProdSched);
        if (!ok) break;
        *reinterpret_cast<volatile int*>(&bars->sched_item[t & 1]) = w;
        mbar_arrive(&bars->sched_full[t & 1]);
        if (w >= n_items) break;
        // V_j as soon as the previous item's last dP^T has read its V.
        if (t > 0) ok = wait_bar<false, HOOK>(&bars->v_empty, (uint32_t)(t - 1) & 1u, wc, kWBwdProdVEmpty);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->v_full, L::kTileBytes);
#pragma unroll
        for (int sb = 0; sb < L::kSub; ++sb)
          tma_load_3d(v_s + sb * kSubTileBytes, &tm_v, &bars->v_full, sb * 64,
                      itm.j * kTile, itm.bkv);
        v_par = t & 1;
        QCursor cur{itm.qh0, itm.i_lo};
        for (int it = 0; it < itm.nq; ++it, ++g, q_next(cur, itm)) {
          const int i = cur.i, bh = cur.bh;
          const int stage = (int)(g & 1u);
          const uint32_t sp = (g >> 1) & 1u;
          // Q_i, LSE2_i, D_i into Q stage g % 2
          ok = wait_bar<false, HOOK>(&bars->q_empty[stage], sp ^ 1u, wc, kWBwdProdQEmpty);
          if (!ok) break;
          uint8_t* qs = smem + L::kQOff + stage * L::kQStageBytes;
          mbar_arrive_expect_tx(&bars->q_full[stage], L::kTileBytes + 2 * kTile * 4);
#pragma unroll
          for (int sb = 0; sb < L::kSub; ++sb)
            tma_load_3d(qs + sb * kSubTileBytes, &tm_q, &bars->q_full[stage],
                        sb * 64, i * kTile, bh);
          const size_t row0 = (size_t)bh * a.N_pad + (size_t)i * kTile;
          bulk_load(qs + L::kTileBytes, a.lse2 + row0, kTile * 4, &bars->q_full[stage]);
          bulk_load(qs + L::kTileBytes + kTile * 4, a.ddot + row0, kTile * 4,
                    &bars->q_full[stage]);
          q_par[stage] = (int)sp;
          // dO_i into the single dO buffer
          ok = wait_bar<false, HOOK>(&bars->do_empty, (g & 1u) ^ 1u, wc, kWBwdProdDoEmpty);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars->do_full, L::kTileBytes);
#pragma unroll
          for (int sb = 0; sb < L::kSub; ++sb)
            tma_load_3d(do_s + sb * kSubTileBytes, &tm_do, &bars->do_full,
                        sb * 64, i * kTile, bh);
          do_par = (int)(g & 1u);
          if (it == 0) {
            // K_j once the previous item's last MMA reading K is done (its
            // first Q and dO are already on their way).
            if (t > 0) ok = wait_bar<false, HOOK>(&bars->k_empty, (uint32_t)(t - 1) & 1u, wc, kWBwdProdKEmpty);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars->k_full, L::kTileBytes);
#pragma unroll
            for (int sb = 0; sb < L::kSub; ++sb)
              tma_load_3d(k_s + sb * kSubTileBytes, &tm_k, &bars->k_full,
                          sb * 64, itm.j * kTile, itm.bkv);
            k_par = t & 1;
          }
        }
      }
      if (!ok) {
        if (k_par >= 0) drain_bar(&bars->k_full, (uint32_t)k_par, a.timeout_ns);
        if (v_par >= 0) drain_bar(&bars->v_full, (uint32_t)v_par, a.timeout_ns);
        for (int s = 0; s < 2; ++s)
          if (q_par[s] >= 0)
            drain_bar(&bars->q_full[s], (uint32_t)q_par[s], a.timeout_ns);
        if (do_par >= 0) drain_bar(&bars->do_full, (uint32_t)do_par, a.timeout_ns);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0 && run) {
      constexpr uint32_t id_st = idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_kv = idesc_bf16(128, D, false, true);
      constexpr uint32_t id_q = idesc_bf16(128, D, true, true);
      const uint32_t tS = tmem, tDP = tmem + 128;
      const uint32_t tDK = tmem + 256, tDV = tmem + 256 + D;
      // Operand descriptors, fixed for the block's lifetime (K-major: 16-wide
      // K steps 32 bytes apart within 128-byte rows, sub-tiles 16 KB apart;
      // MN-major: 16-row K steps 2048 bytes apart).
      const uint64_t k_km = sdesc_sw128(smem_addr(k_s), 16, 1024);
      const uint64_t k_mn = sdesc_sw128(smem_addr(k_s), kSubTileBytes, 1024);
      const uint64_t v_km = sdesc_sw128(smem_addr(v_s), 16, 1024);
      const uint64_t do_km = sdesc_sw128(smem_addr(do_s), 16, 1024);
      const uint64_t do_mn = sdesc_sw128(smem_addr(do_s), kSubTileBytes, 1024);
      const uint64_t ds_mn = sdesc_sw128(smem_addr(ds_s), kSubTileBytes, 1024);
      const uint64_t q_km0 = sdesc_sw128(smem_addr(smem + L::kQOff), 16, 1024);
      const uint64_t q_mn0 =
          sdesc_sw128(smem_addr(smem + L::kQOff), kSubTileBytes, 1024);
      auto q_km = [&](uint32_t gi) { return sdesc_adv(q_km0, (gi & 1u) * L::kQStageBytes); };
      auto q_mn = [&](uint32_t gi) { return sdesc_adv(q_mn0, (gi & 1u) * L::kQStageBytes); };
      auto kstep = [](int s) {  // K-major offset of 16-wide K step s
        return (uint32_t)((s >> 2) * kSubTileBytes + (s & 3) * 32);
      };
      // Software pipeline: S^T and dP^T of tile it+1 are issued around the
      // dK/dQ MMAs of tile it, so the P/dS warps work on tile it+1 while the
      // tensor core finishes tile it.  Per iteration the issue order is
      //   dV(it)  S^T(it+1)  dK(it)  dQ(it)  dP^T(it+1)
      // S^T(it+1) may overwrite P^T(it) because dV(it) precedes it in the
      // tensor core's in-order queue; the same holds across items.
      auto issue_st = [&](uint32_t gi) {  // S^T = K_j Q_i^T  [keys x queries]
        const uint64_t qd = q_km(gi);
#pragma unroll
        for (int s = 0; s < D / 16; ++s)
          mma_ss(tS, sdesc_adv(k_km, kstep(s)), sdesc_adv(qd, kstep(s)), id_st,
                 s > 0 ? 1u : 0u);
        mma_commit(&bars->s_full);
      };
      auto issue_dp = [&]() {  // dP^T = V_j dO_i^T  [keys x queries]
#pragma unroll
        for (int s = 0; s < D / 16; ++s)
          mma_ss(tDP, sdesc_adv(v_km, kstep(s)), sdesc_adv(do_km, kstep(s)),
                 id_st, s > 0 ? 1u : 0u);
        mma_commit(&bars->dp_full);
      };
      bool ok = true;
      uint32_t g = 0;
      for (int t = 0; ok; ++t) {
        int w;
        ok = sched_take<false>(bars, t, wc, kWBwdMmaSched, w);
        if (!ok || w >= n_items) break;
        const BwdItem itm = bwd_item<CAUSAL, VARLEN>(w, n_tiles, a);
        const int nq = itm.nq;
        const uint32_t tp = (uint32_t)t & 1u;
        // The item's first S^T and dP^T.  dP^T(0) reuses the columns of the
        // previous item's last dQ, which the drain warps must have read.
        ok = wait_bar<false, HOOK>(&bars->k_full, tp, wc, kWBwdMmaKV);
        if (ok) ok = wait_bar<false, HOOK>(&bars->q_full[g & 1u], (g >> 1) & 1u, wc, kWBwdMmaQ);
        if (!ok) break;
        tc_fence_after();
        issue_st(g);
        ok = wait_bar<false, HOOK>(&bars->v_full, tp, wc, kWBwdMmaKV);
        if (ok) ok = wait_bar<false, HOOK>(&bars->do_full, g & 1u, wc, kWBwdMmaDo);
        if (ok && g > 0) ok = wait_bar<false, HOOK>(&bars->dq_free, (g - 1u) & 1u, wc, kWBwdMmaDqFree);
        if (!ok) break;
        tc_fence_after();
        issue_dp();
        if (nq == 1) mma_commit(&bars->v_empty);   // V_j no longer read
        for (int it = 0; it < nq && ok; ++it) {
          const uint32_t gi = g + (uint32_t)it;
          const uint32_t par = gi & 1u;
          ok = wait_bar<false, HOOK>(&bars->p_full, par, wc, kWBwdMmaP);
          // dK, dV of the previous item must be out of TMEM before this
          // item's first products overwrite them.
          if (ok && it == 0 && t > 0)
            ok = wait_bar<false, HOOK>(&bars->acc_free, tp ^ 1u, wc, kWBwdMmaAccFree);
          if (!ok) break;
          tc_fence_after();
          // dV_j += P^T dO_i   [keys x d], K = queries; P^T from TMEM
#pragma unroll
          for (int s = 0; s < kTile / 16; ++s)
            mma_ts(tDV, tS + s * 8, sdesc_adv(do_mn, s * 2048), id_kv,
                   (it > 0 || s > 0) ? 1u : 0u);
          mma_commit(&bars->do_empty);   // dO_i no longer needed
          if (it + 1 < nq) {
            ok = wait_bar<false, HOOK>(&bars->q_full[(gi + 1u) & 1u], ((gi + 1u) >> 1) & 1u,
                          wc, kWBwdMmaQ);
            if (!ok) break;
            tc_fence_after();
            issue_st(gi + 1u);
          }
          ok = wait_bar<false, HOOK>(&bars->ds_full, par, wc, kWBwdMmaDs);
          if (!ok) break;
          tc_fence_after();
          // dK_j += dS^T Q_i   [keys x d], K = queries; dS^T from TMEM (bf16
          // pairs in the dP^T columns), Q read MN-major
          const uint64_t qmn = q_mn(gi);
#pragma unroll
          for (int s = 0; s < kTile / 16; ++s)
            mma_ts(tDK, tDP + s * 8, sdesc_adv(qmn, s * 2048), id_kv,
                   (it > 0 || s > 0) ? 1u : 0u);
          mma_commit(&bars->q_empty[gi & 1u]);   // Q_i, LSE2_i, D_i released
          // dQ_i = dS K_j   [queries x d], K = keys; dS read MN-major
#pragma unroll
          for (int s = 0; s < kTile / 16; ++s)
            mma_ss(tDP, sdesc_adv(ds_mn, s * 2048), sdesc_adv(k_mn, s * 2048), id_q,
                   s > 0 ? 1u : 0u);
          mma_commit(&bars->dq_full);
          mma_commit(&bars->ds_free);    // dS_i no longer read
          if (it + 1 < nq) {
            // dQ_it occupies the dP columns until the drain warps have read it.
            ok = wait_bar<false, HOOK>(&bars->dq_free, par, wc, kWBwdMmaDqFree);
            if (ok) ok = wait_bar<false, HOOK>(&bars->do_full, par ^ 1u, wc, kWBwdMmaDo);
            if (!ok) break;
            tc_fence_after();
            issue_dp();
            if (it + 2 == nq) mma_commit(&bars->v_empty);   // V_j no longer read
          }
        }
        if (!ok) break;
        mma_commit(&bars->k_empty);    // K_j no longer read
        mma_commit(&bars->acc_done);   // dK_j, dV_j complete
        g += (uint32_t)nq;
      }
      mma_commit(&bars->mma_done);
      drain_bar(&bars->mma_done, 0, a.timeout_ns);
    }
  } else if (warp < 4) {
    // -------------------------------------- P^T and dS^T (thread = key row)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                  // key row in tile j
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const float c = a.scale_log2;
    const uint64_t c2 = bcast2(c);
    bool ok = run;
    bool stg_pending = false;  // this warp's dK rows are being stored from dS
    uint32_t g = 0;
    for (int t = 0; ok; ++t) {
      int w;
      ok = sched_take<true>(bars, t, wc, kWBwdCmpSched, w);
      if (!ok || w >= n_items) break;
      const BwdItem itm = bwd_item<CAUSAL, VARLEN>(w, n_tiles, a);
      const int j = itm.j;
      // Band: query q (global) sees key k when dmin <= q - k <= dmax (INT_MIN
      // / INT_MAX: no bound); a tile pair needs the mask only if its offsets
      // reach outside [dmin, dmax].  Tile offsets fit in int because
      // N <= 2^30 and the window is below N.
      // With per-sequence lengths, key rows past the sequence's end hold real
      // (finite) data, so their P must be forced to zero: the tile that holds
      // the end takes the masked path, with no visible query for those rows.
      const bool key_in = j * kTile + r < itm.len;
      const bool tail = VARLEN && (j + 1) * kTile > itm.len;
      const int win = a.window;
      const int dmin = CAUSAL ? 0 : (win >= 0 ? -win : INT_MIN);
      const int dmax = win >= 0 ? win : INT_MAX;
      QCursor cur{itm.qh0, itm.i_lo};
      for (int it = 0; it < itm.nq && ok; ++it, q_next(cur, itm)) {
        const uint32_t gi = g + (uint32_t)it;
        const int i = cur.i;
        const int stage = (int)(gi & 1u);
        const uint32_t sp = (gi >> 1) & 1u;
        const uint32_t par = gi & 1u;
        ok = wait_bar_warp(&bars->q_full[stage], sp, wc, kWBwdCmpQ);
        if (!ok) break;
        // -LSE_i log2(e) and D_i of this Q tile's rows, in smem after Q_i
        const float* nlse2 = reinterpret_cast<const float*>(
            smem + L::kQOff + stage * L::kQStageBytes + L::kTileBytes);
        const float* dd = nlse2 + kTile;
        ok = wait_bar_warp(&bars->s_full, par, wc, kWBwdCmpS);
        if (!ok) break;
        tc_fence_after();
        // P^T = exp2(S^T c + LSE2) (LSE2 = -LSE log2 e; packed pairs), in two
        // halves of 64 queries so that only
        // half a row of S is live; P half h goes to TMEM columns [32h, 32h+32),
        // over S columns that have already been read.
        uint32_t pk[64];
        const int off0 = (i - j) * kTile;  // q - k where local q = local k
        const bool edge = tail ||
                          (dmin != INT_MIN && off0 - (kTile - 1) < dmin) ||
                          (dmax != INT_MAX && off0 + (kTile - 1) > dmax);
        // Local query index q is visible to key row r when q_lo <= q <= q_hi.
        int q_lo = 0, q_hi = kTile - 1;
        if (edge) {
          const long long base = off0 - r;  // q - k = base + local q
          if (dmin != INT_MIN)
            q_lo = (int)max(0ll, min((long long)kTile, dmin - base));
          if (dmax != INT_MAX)
            q_hi = (int)max(-1ll, min((long long)kTile - 1, dmax - base));
          if (VARLEN && !key_in) q_lo = kTile;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t s[64];
          tmem_ld32(tl + 64 * h, s);
          tmem_ld32(tl + 64 * h + 32, s + 32);
          tmem_wait_ld();
          reg_fence32(s);
          reg_fence32(s + 32);
#pragma unroll
          for (int e = 0; e < 64; e += 4) {
            const int q = 64 * h + e;
            const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + q);
            float x0, x1, x2, x3;
            fma2_bc(x0, x1, __uint_as_float(s[e + 0]), __uint_as_float(s[e + 1]),
                    c2, l4.x, l4.y);
            fma2_bc(x2, x3, __uint_as_float(s[e + 2]), __uint_as_float(s[e + 3]),
                    c2, l4.z, l4.w);
            pk[q / 2] = pack_bf16(ex2(x0), ex2(x1));
            pk[q / 2 + 1] = pack_bf16(ex2(x2), ex2(x3));
          }
          if (edge) {  // P of queries outside [q_lo, q_hi] is exactly 0
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int q = 64 * h + 2 * k;
              uint32_t keep = 0xffffffffu;
              if (q < q_lo || q > q_hi) keep &= 0xffff0000u;
              if (q + 1 < q_lo || q + 1 > q_hi) keep &= 0x0000ffffu;
              pk[32 * h + k] &= keep;
            }
          }
          tmem_st32(tl + 32 * h, pk + 32 * h);
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&bars->p_full);

        ok = wait_bar_warp(&bars->dp_full, par, wc, kWBwdCmpDp);
        if (ok && gi > 0) ok = wait_bar_warp(&bars->ds_free, par ^ 1u, wc, kWBwdCmpDsFree);
        if (!ok) break;
        if (stg_pending) {  // the TMA has read this warp's dK rows from dS
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          stg_pending = false;
        }
        tc_fence_after();
        // dS^T goes to smem (read MN-major as dS by the dQ MMA) and, packed to
        // bf16 pairs, into TMEM columns [128, 192) over dP^T values already
        // read (the dK MMA takes it from there as its A operand): chunk ch
        // (32 queries) fills columns 128 + 16 ch .. 128 + 16 ch + 15, which
        // held dP^T of chunk ch / 2, already loaded.
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t dp[32];
          tmem_ld32(tl + 128 + ch * 32, dp);
          tmem_wait_ld();
          reg_fence32(dp);
          uint32_t dsk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const int q = ch * 32 + e;
            const float4 d4 = *reinterpret_cast<const float4*>(dd + q);
            const uint32_t pa = pk[q / 2], pb = pk[q / 2 + 1];
            float ds0, ds1, ds2, ds3;
            mulsub2(ds0, ds1, bf16_lo(pa), bf16_hi(pa), __uint_as_float(dp[e + 0]),
                    __uint_as_float(dp[e + 1]), d4.x, d4.y);
            mulsub2(ds2, ds3, bf16_lo(pb), bf16_hi(pb), __uint_as_float(dp[e + 2]),
                    __uint_as_float(dp[e + 3]), d4.z, d4.w);
            dsk[e / 2] = pack_bf16(ds0, ds1);
            dsk[e / 2 + 1] = pack_bf16(ds2, ds3);
          }
          // Row r of dS^T, queries ch*32 .. ch*32+31, into the swizzled tile.
          uint8_t* sub = ds_s + (ch >> 1) * kSubTileBytes;
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {
            const uint32_t col = (uint32_t)((ch & 1) * 32 + gq * 8);
            *reinterpret_cast<uint4*>(sub + sw128_offset((uint32_t)r, col)) =
                make_uint4(dsk[4 * gq], dsk[4 * gq + 1], dsk[4 * gq + 2],
                           dsk[4 * gq + 3]);
          }
          tmem_st16(tl + 128 + ch * 16, dsk);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(&bars->ds_full);
      }
      if (!ok) break;
      // dK epilogue (rows = keys), then the columns are free for the next item
      ok = wait_bar_warp(&bars->acc_done, (uint32_t)t & 1u, wc, kWBwdCmpAcc);
      if (!ok) break;
      tc_fence_after();
      if (a.nsplit > 1) {
        kv_epilogue_atomic<D>(tl + 256, a.dk_acc, itm.bkv, j * kTile + r, a.N,
                              itm.len, a.scale);
        tc_fence_before();
        warp_arrive(&bars->acc_free);
      } else {
        // Staged in the dS tile: its last reader, the item's last dQ MMA, is
        // complete (acc_done follows it), and each warp owns its 32 rows
        // there.  The stores clip rows past N; rows past a sequence's end
        // hold zeros (no visible query) and are cleared again by the post
        // kernel.
        kv_epilogue_stage<D>(tl + 256, ds_s, kSubTileBytes, (uint32_t)r, a.scale);
        tc_fence_before();
        warp_arrive(&bars->acc_free);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int sb = 0; sb < L::kSub; ++sb)
            tma_store_3d(&tm_dk, ds_s + sb * kSubTileBytes + quarter * 32 * 128,
                         sb * 64, j * kTile + quarter * 32, itm.bkv);
          bulk_commit_group();
        }
        stg_pending = true;
      }
      g += (uint32_t)itm.nq;
    }
    if (lane == 0) bulk_wait_all();  // dK stores complete before exit
  } else if (warp < 8) {
    // ------------------------------------- dQ drain (thread = query row)
    // dQ_i leaves TMEM into registers (then the columns are released) and is
    // added into the fp32 accumulator by TMA reduce-add (whole 128-byte
    // lines at L2).  Each warp handles its own 32 rows independently: box by
    // box ([32 rows][32 fp32] = 4 KB in the 128-byte swizzle layout) through
    // two staging buffers of its own, rewriting a buffer only after the TMA
    // has read the box before the last one (bulk groups are per thread, and
    // lane 0 issues and waits on all of this warp's).
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    uint8_t* const stg_w = stg_s + quarter * 2 * L::kStgBoxBytes;
    constexpr int kBoxes = D / 32;
    int gb = 0;                                      // boxes staged so far
    bool stg_busy = false;  // both boxes hold dV rows being stored
    bool ok = run;
    uint32_t g = 0;
    for (int t = 0; ok; ++t) {
      int w;
      ok = sched_take<true>(bars, t, wc, kWBwdDqSched, w);
      if (!ok || w >= n_items) break;
      const BwdItem itm = bwd_item<CAUSAL, VARLEN>(w, n_tiles, a);
      QCursor cur{itm.qh0, itm.i_lo};
      for (int it = 0; it < itm.nq && ok; ++it, q_next(cur, itm)) {
        const uint32_t gi = g + (uint32_t)it;
        const int i = cur.i, bh = cur.bh;
        ok = wait_bar_warp(&bars->dq_full, gi & 1u, wc, kWBwdDqFull);
        if (!ok) break;
        tc_fence_after();
        uint32_t acc[D];
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) tmem_ld32(tl + 128 + ch * 32, acc + ch * 32);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) reg_fence32(acc + ch * 32);
        tc_fence_before();
        warp_arrive(&bars->dq_free);   // the dP/dQ columns may be reused now
#pragma unroll
        for (int b = 0; b < kBoxes; ++b, ++gb) {
          uint8_t* const buf = stg_w + (gb & 1) * L::kStgBoxBytes;
          if (stg_busy) {  // the dV stores have read both boxes
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            stg_busy = false;
          } else if (gb >= 2) {
            if (lane == 0) bulk_wait_read_allbut1();  // box gb-2 has been read
            __syncwarp();
          }
          uint8_t* dst = buf + lane * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            *reinterpret_cast<uint4*>(dst + ((k ^ (lane & 7)) * 16)) =
                make_uint4(acc[32 * b + 4 * k], acc[32 * b + 4 * k + 1],
                           acc[32 * b + 4 * k + 2], acc[32 * b + 4 * k + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&tm_dq, buf, b * 32, i * kTile + quarter * 32, bh);
            bulk_commit_group();
          }
        }
      }
      if (!ok) break;
      // dV epilogue (rows = keys), then the columns are free for the next item
      ok = wait_bar_warp(&bars->acc_done, (uint32_t)t & 1u, wc, kWBwdDqAcc);
      if (!ok) break;
      tc_fence_after();
      if (a.nsplit > 1) {
        kv_epilogue_atomic<D>(tl + 256 + D, a.dv_acc, itm.bkv, itm.j * kTile + r,
                              a.N, itm.len, 1.0f);
        tc_fence_before();
        warp_arrive(&bars->acc_free);
      } else {
        // Staged in this warp's two boxes once its dQ adds have read them.
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        kv_epilogue_stage<D>(tl + 256 + D, stg_w, L::kStgBoxBytes, (uint32_t)lane,
                             1.0f);
        tc_fence_before();
        warp_arrive(&bars->acc_free);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int sb = 0; sb < L::kSub; ++sb)
            tma_store_3d(&tm_dv, stg_w + sb * L::kStgBoxBytes, sb * 64,
                         itm.j * kTile + quarter * 32, itm.bkv);
          bulk_commit_group();
        }
        stg_busy = true;
      }
      g += (uint32_t)itm.nq;
    }
    if (lane == 0) bulk_wait_all();  // dQ adds and dV stores complete before exit
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Per-sequence lengths: work on a [heads_total, N, *] tensor in units of
// kChunkRows rows of one head, dealt over the grid's blocks; f(h, r0, r1, len)
// handles rows [r0, r1) of head h, whose sequence (batch entry h / heads)
// has length len.  One division per unit instead of one per row keeps these
// HBM-bound loops from being instruction-bound.
constexpr int kChunkRows = 64;
template <class F>
__device__ __forceinline__ void over_row_chunks(long long heads_total, int heads,
                                                int N, const int* seq_lens,
                                                F&& f) {
  const int chunks = (N + kChunkRows - 1) / kChunkRows;
  const long long units = heads_total * chunks;
  for (long long u = blockIdx.x; u < units; u += gridDim.x) {
    const long long h = u / chunks;
    const int r0 = (int)(u - h * chunks) * kChunkRows;
    const int r1 = r0 + kChunkRows < N ? r0 + kChunkRows : N;
    f(h, r0, r1, seq_len_of(seq_lens, (int)(h / heads), N));
  }
}

// Rows of a [heads_total, N, D] fp32 accumulator that lie inside their
// sequence -> 0.
template <int D>
__device__ __forceinline__ void zero_real_rows(float* acc_f, long long heads_total,
                                               int heads, int N,
                                               const int* seq_lens) {
  constexpr int kPerRow = D / 4;  // float4 per row
  float4* acc = reinterpret_cast<float4*>(acc_f);
  over_row_chunks(heads_total, heads, N, seq_lens,
                  [&](long long h, int r0, int r1, int len) {
    const int e = r1 < len ? r1 : len;
    if (e <= r0) return;
    float4* base = acc + ((size_t)h * N + r0) * kPerRow;
    const int n = (e - r0) * kPerRow;
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      base[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  });
}

// D_i = dO_i . O_i and LSE2_i = -LSE_i log2(e) for every padded row (one warp
// per row, four rows in flight per warp), clearing the dQ accumulator of each
// real row in the same pass (with per-sequence lengths, padding rows are
// never read: the post kernel writes zeros there); then the split groups'
// dK and dV accumulators.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a) {
  // The main kernel's work counter starts from zero on every call.
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.work_next = 0u;
  constexpr int kRows = 4;
  constexpr int kPer = D / 32;  // 4 (d=128) or 2 (d=64) elements per lane
  const int lane = threadIdx.x & 31;
  const long long warps_total = (long long)gridDim.x * (blockDim.x >> 5);
  const long long gwarp = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long rows = (long long)a.BH * a.N_pad;
  for (long long row0 = gwarp * kRows; row0 < rows; row0 += warps_total * kRows) {
    uint32_t ov[kRows][kPer / 2], dv[kRows][kPer / 2];
    bool valid[kRows];
    long long lrow[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      const long long row = row0 + k;
      const int bh = (int)(row / a.N_pad);
      const int q = (int)(row - (long long)bh * a.N_pad);
      valid[k] = row < rows &&
                 q < (a.seq_lens ? seq_len_of(a.seq_lens, bh / a.H, a.N) : a.N);
      lrow[k] = (long long)bh * a.N + q;
#pragma unroll
      for (int e = 0; e < kPer / 2; ++e) ov[k][e] = dv[k][e] = 0u;
      if (valid[k]) {
        const size_t base = (size_t)lrow[k] * D + lane * kPer;
        if constexpr (kPer == 4) {
          const uint2 o2 = *reinterpret_cast<const uint2*>(a.o + base);
          const uint2 d2 = *reinterpret_cast<const uint2*>(a.dout + base);
          ov[k][0] = o2.x; ov[k][1] = o2.y;
          dv[k][0] = d2.x; dv[k][1] = d2.y;
        } else {
          ov[k][0] = *reinterpret_cast<const uint32_t*>(a.o + base);
          dv[k][0] = *reinterpret_cast<const uint32_t*>(a.dout + base);
        }
        // The row's dQ accumulator is cleared in the same pass, so that the
        // writes overlap the reads instead of following them.
        float4* acc = reinterpret_cast<float4*>(a.dq_acc) + (size_t)lrow[k] * (D / 4);
        for (int c = lane; c < D / 4; c += 32) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      float dsum = 0.f;
#pragma unroll
      for (int e = 0; e < kPer / 2; ++e)
        dsum += bf16_lo(ov[k][e]) * bf16_lo(dv[k][e]) + bf16_hi(ov[k][e]) * bf16_hi(dv[k][e]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
      const long long row = row0 + k;
      if (lane == 0 && row < rows) {
        a.ddot[row] = valid[k] ? dsum : 0.f;
        a.lse2[row] = valid[k] ? -(a.lse[lrow[k]] * kLog2e) : -INFINITY;
      }
    }
  }
  if (a.nsplit > 1) {
    if (a.seq_lens) {
      // With per-sequence lengths only real rows are cleared: the post
      // kernel writes zeros on padding rows without reading them.
      zero_real_rows<D>(a.dk_acc, a.BHkv, a.Hkv, a.N, a.seq_lens);
      zero_real_rows<D>(a.dv_acc, a.BHkv, a.Hkv, a.N, a.seq_lens);
      return;
    }
    const long long m4 = (long long)a.BHkv * a.N * D / 4;
    float4* ak = reinterpret_cast<float4*>(a.dk_acc);
    float4* av = reinterpret_cast<float4*>(a.dv_acc);
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
         idx < m4; idx += (long long)gridDim.x * blockDim.x) {
      ak[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
      av[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// out = mul * acc -> bf16 over n8 groups of eight elements.
__device__ __forceinline__ void round_rows(const float* acc_f, __nv_bfloat16* out_b,
                                           long long n8, float mul) {
  const float4* acc = reinterpret_cast<const float4*>(acc_f);
  uint4* out = reinterpret_cast<uint4*>(out_b);
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n8;
       idx += (long long)gridDim.x * blockDim.x) {
    const float4 x = acc[2 * idx], y = acc[2 * idx + 1];
    out[idx] = make_uint4(pack_bf16(x.x * mul, x.y * mul),
                          pack_bf16(x.z * mul, x.w * mul),
                          pack_bf16(y.x * mul, y.y * mul),
                          pack_bf16(y.z * mul, y.w * mul));
  }
}

// Per-sequence lengths: out = mul * acc -> bf16 on the rows inside each
// sequence and 0 on the rows past its end (acc not read there), for a
// [heads_total, N, d] tensor; acc == nullptr: only the zeros are written.
__device__ __forceinline__ void round_rows_varlen(const float* acc_f,
                                                  __nv_bfloat16* out_b,
                                                  long long heads_total,
                                                  int heads, int N, int d,
                                                  float mul,
                                                  const int* seq_lens) {
  const int per_row = d / 8;  // groups of eight elements
  const float4* acc = reinterpret_cast<const float4*>(acc_f);
  uint4* out = reinterpret_cast<uint4*>(out_b);
  over_row_chunks(heads_total, heads, N, seq_lens,
                  [&](long long h, int r0, int r1, int len) {
    const int e = r1 < len ? r1 : (len > r0 ? len : r0);  // real rows [r0, e)
    const size_t base = ((size_t)h * N + r0) * per_row;
    const int n_real = (e - r0) * per_row, n_all = (r1 - r0) * per_row;
    if (acc) {
      for (int i = threadIdx.x; i < n_real; i += blockDim.x) {
        const float4 x = acc[2 * (base + i)], y = acc[2 * (base + i) + 1];
        out[base + i] = make_uint4(pack_bf16(x.x * mul, x.y * mul),
                                   pack_bf16(x.z * mul, x.w * mul),
                                   pack_bf16(y.x * mul, y.y * mul),
                                   pack_bf16(y.z * mul, y.w * mul));
      }
    }
    for (int i = n_real + threadIdx.x; i < n_all; i += blockDim.x)
      out[base + i] = make_uint4(0u, 0u, 0u, 0u);
  });
}

// dQ = scale * accumulator -> bf16, eight elements per thread per step; with
// split key/value groups also dK and dV (already scaled) -> bf16.  With
// per-sequence lengths the same row by row, padding rows of dQ, dK and dV
// set to zero without reading the accumulators there.
__global__ void __launch_bounds__(256) bwd_post_kernel(const BwdArgs a, int d) {
  if (a.seq_lens) {
    const bool split = a.nsplit > 1;
    round_rows_varlen(a.dq_acc, a.dq, a.BH, a.H, a.N, d, a.scale, a.seq_lens);
    round_rows_varlen(split ? a.dk_acc : nullptr, a.dk, a.BHkv, a.Hkv, a.N, d,
                      1.0f, a.seq_lens);
    round_rows_varlen(split ? a.dv_acc : nullptr, a.dv, a.BHkv, a.Hkv, a.N, d,
                      1.0f, a.seq_lens);
    return;
  }
  round_rows(a.dq_acc, a.dq, (long long)a.BH * a.N * d / 8, a.scale);
  if (a.nsplit > 1) {
    const long long m8 = (long long)a.BHkv * a.N * d / 8;
    round_rows(a.dk_acc, a.dk, m8, 1.0f);
    round_rows(a.dv_acc, a.dv, m8, 1.0f);
  }
}

template <int D, bool CAUSAL, bool VARLEN, bool HOOK = false>
cudaError_t launch_main_t(const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo,
                          const CUtensorMap& tdq, const CUtensorMap& tdk,
                          const CUtensorMap& tdv, const BwdArgs& a,
                          int grid_blocks, cudaStream_t stream) {
  using L = BwdLayout<D>;
  // The failure-path test hook has its own instantiation, for d = 128
  // without per-sequence lengths only.
  if constexpr (D == 128 && !VARLEN && !HOOK) {
    if (a.hook)
      return launch_main_t<D, CAUSAL, VARLEN, true>(tq, tk, tv, tdo, tdq, tdk,
                                                    tdv, a, grid_blocks, stream);
  }
  auto kern = bwd_main_kernel<D, CAUSAL, VARLEN, HOOK>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const long long n_items = (long long)a.BHkv * a.nsplit * n_tiles;
  const int blocks = n_items < grid_blocks ? (int)n_items : grid_blocks;
  kern<<<blocks, kBwdThreads, L::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq,
                                                        tdk, tdv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_pre(const BwdArgs& a, int d, int grid_blocks,
                           cudaStream_t stream) {
  if (d == 128)
    bwd_pre_kernel<128><<<grid_blocks, 256, 0, stream>>>(a);
  else
    bwd_pre_kernel<64><<<grid_blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tdq, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, const BwdArgs& a, int d,
                            bool causal, int grid_blocks, cudaStream_t stream) {
  const bool vl = a.seq_lens != nullptr;
  const int gb = grid_blocks;
  if (d == 128) {
    if (causal)
      return vl ? launch_main_t<128, true, true>(tq, tk, tv, tdo, tdq, tdk, tdv, a, gb, stream)
                : launch_main_t<128, true, false>(tq, tk, tv, tdo, tdq, tdk, tdv, a, gb, stream);
    return vl ? launch_main_t<128, false, true>(tq, tk, tv, tdo, tdq, tdk, tdv, a, gb, stream)
              : launch_main_t<128, false, false>(tq, tk, tv, tdo, tdq, tdk, tdv, a, gb, stream);
  }
  if (causal)
    return vl ? launch_main_t<64, true, true>(tq, tk, tv, tdo, tdq, tdk, tdv, a, gb, stream)
              : launch_main_t<64, true, false>(tq, tk, tv, tdo, tdq, tdk, tdv, a, gb, stream);
  return vl ? launch_main_t<64, false, true>(tq, tk, tv, tdo, tdq, tdk, tdv, a, gb, stream)
            : launch_main_t<64, false, false>(tq, tk, tv, tdo, tdq, tdk, tdv, a, gb, stream);
}

cudaError_t launch_bwd_post(const BwdArgs& a, int d, int grid_blocks,
                            cudaStream_t stream) {
  bwd_post_kernel<<<grid_blocks, 256, 0, stream>>>(a, d);
  return cudaGetLastError();
}

cudaError_t set_expire_site_bwd(uint32_t site) {
  return cudaMemcpyToSymbol(c_expire_site, &site, sizeof(site));
}

}  // namespace fa
