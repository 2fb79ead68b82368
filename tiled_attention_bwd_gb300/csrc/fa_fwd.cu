// fa_fwd.cu -- forward attention kernel for sm_103a.
//
// O = softmax(scale * Q K^T [+ causal mask]) V and LSE per row, computed
// tile by tile with an online softmax so the N x N scores never leave the SM
// ("RTX Flash Attention Implementation COMPLETE", "CUDA Kernel Design: Flash
// Attention Forward Kernel" and "Online Softmax Algorithm"; the TMA /
// warp-specialised pipeline of "GPU Performance Optimization Batch 1 --
// Design Spec", Item 3, sections "TMA" and "Warp Specialization").
//
// One thread block owns two 128-row Q tiles of one (batch, head) and streams
// the 128-row K/V tiles past them:
//   warp 8      TMA producer: Q0, Q1 once; K_j, V_j through a smem ring.
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM, then
//               O_t += P_t V_j with P_t read straight from TMEM.
//   warps 0-3   softmax for Q tile 0, warps 4-7 for Q tile 1; thread = row.
//               exp2 with the scale folded in, lazy rescaling of O (only when
//               the row max grows by more than 2^8), P written back to TMEM
//               as bf16 over the S columns it came from.
// While one softmax group works on its tile the tensor core runs the other
// tile's MMAs (ping-pong).  Causal blocks stop at the diagonal tile; only the
// diagonal (and a ragged last tile) is masked.
//
// TMEM columns (512 allocated): S0 [0,128) S1 [128,256) O0 [256,256+d)
// O1 [256+d, 256+2d).  P_t occupies the first 64 columns of S_t.
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

constexpr int kFwdThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: factor 256

template <int D>
struct FwdLayout {
  static constexpr int kSub = D / 64;             // 64-column sub-tiles
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kStages = (D == 128) ? 4 : 6;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // + align slack
};

template <int STAGES>
struct FwdBars {
  uint64_t q_full[2];
  uint64_t kv_full[STAGES];
  uint64_t kv_empty[STAGES];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
};

// Where-codes of bounded waits (recorded when a wait expires).
enum : uint32_t {
  kWFwdProdEmpty = 0x101,
  kWFwdMmaQ = 0x201,
  kWFwdMmaKV = 0x202,
  kWFwdMmaP = 0x203,
  kWFwdSmS = 0x301,
  kWFwdSmO = 0x302,
};

template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_addr,
                                         uint32_t k_addr) {
  constexpr uint32_t id = idesc_bf16(128, 128, false, false);
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    const uint32_t off = (s >> 2) * kSubTileBytes + (s & 3) * 32;
    mma_ss(d_tmem, sdesc_sw128(q_addr + off, 16, 1024),
           sdesc_sw128(k_addr + off, 16, 1024), id, s > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem,
                                         uint32_t v_addr, bool accumulate) {
  constexpr uint32_t id = idesc_bf16(128, D, false, true);
#pragma unroll
  for (int s = 0; s < kTile / 16; ++s) {
    mma_ts(o_tmem, p_tmem + s * 8,
           sdesc_sw128(v_addr + s * 2048, kSubTileBytes, 1024), id,
           (accumulate || s > 0) ? 1u : 0u);
  }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = FwdLayout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  auto* bars = reinterpret_cast<FwdBars<S>*>(smem + L::kBarOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const int n_pairs = (n_tiles + 1) / 2;
  const TileSlot slot = grouped_slot((int)blockIdx.x, n_pairs, a.BH, a.group);
  const int bh = slot.bh;
  // Causal: the heaviest (last) pair of each head is scheduled first.
  const int pair = CAUSAL ? (n_pairs - 1 - slot.tile) : slot.tile;
  const int qt0 = 2 * pair, qt1 = 2 * pair + 1;
  const int nkv0 = CAUSAL ? qt0 + 1 : n_tiles;
  const int nkv1 = (qt1 < n_tiles) ? (CAUSAL ? qt1 + 1 : n_tiles) : 0;
  const int nkv = nkv0 > nkv1 ? nkv0 : nkv1;

  if (threadIdx.x == 0) {
    bars->abort = *reinterpret_cast<volatile unsigned int*>(&a.st->abort);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 4);   // one arrival per warp
      mbar_init(&bars->o_done[t], 1);
    }
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->mma_done, 1);
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

  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0 && run) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(&bars->q_full[0], L::kTileBytes);
#pragma unroll
      for (int sb = 0; sb < L::kSub; ++sb)
        tma_load_3d(smem + L::kQOff + sb * kSubTileBytes, &tm_q,
                    &bars->q_full[0], sb * 64, qt0 * kTile, bh);
      if (nkv1 > 0) {
        mbar_arrive_expect_tx(&bars->q_full[1], L::kTileBytes);
#pragma unroll
        for (int sb = 0; sb < L::kSub; ++sb)
          tma_load_3d(smem + L::kQOff + L::kTileBytes + sb * kSubTileBytes,
                      &tm_q, &bars->q_full[1], sb * 64, qt1 * kTile, bh);
      }
      int last_par[S];
#pragma unroll
      for (int s = 0; s < S; ++s) last_par[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int j = 0; j < nkv && ok; ++j) {
        for (int w = 0; w < 2; ++w) {  // 0: K_j, 1: V_j
          ok = wait_bar(&bars->kv_empty[stage], phase ^ 1u, wc, kWFwdProdEmpty);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars->kv_full[stage], L::kTileBytes);
          const CUtensorMap* m = w ? &tm_v : &tm_k;
#pragma unroll
          for (int sb = 0; sb < L::kSub; ++sb)
            tma_load_3d(smem + L::kKVOff + stage * L::kTileBytes +
                            sb * kSubTileBytes,
                        m, &bars->kv_full[stage], sb * 64, j * kTile, bh);
          last_par[stage] = (int)phase;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Stopping: let every copy this thread started land before exit.
        drain_bar(&bars->q_full[0], 0, a.timeout_ns);
        if (nkv1 > 0) drain_bar(&bars->q_full[1], 0, a.timeout_ns);
        for (int s = 0; s < S; ++s)
          if (last_par[s] >= 0)
            drain_bar(&bars->kv_full[s], (uint32_t)last_par[s], a.timeout_ns);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0 && run) {
      const uint32_t q_addr0 = smem_addr(smem + L::kQOff);
      const uint32_t q_addr1 = q_addr0 + L::kTileBytes;
      const uint32_t kv_addr = smem_addr(smem + L::kKVOff);
      const uint32_t tS0 = tmem, tS1 = tmem + 128;
      const uint32_t tO0 = tmem + 256, tO1 = tmem + 256 + D;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = wait_bar(&bars->q_full[0], 0, wc, kWFwdMmaQ);
      if (ok && nkv1 > 0) ok = wait_bar(&bars->q_full[1], 0, wc, kWFwdMmaQ);
      // K_0
      int k_stage = stage;
      if (ok) ok = wait_bar(&bars->kv_full[stage], phase, wc, kWFwdMmaKV);
      if (++stage == S) { stage = 0; phase ^= 1u; }
      if (ok) {
        tc_fence_after();
        issue_qk<D>(tS0, q_addr0, kv_addr + k_stage * L::kTileBytes);
        mma_commit(&bars->s_full[0]);
        if (nkv1 > 0) {
          issue_qk<D>(tS1, q_addr1, kv_addr + k_stage * L::kTileBytes);
          mma_commit(&bars->s_full[1]);
        }
        mma_commit(&bars->kv_empty[k_stage]);
      }
      for (int j = 0; j < nkv && ok; ++j) {
        const int v_stage = stage;
        ok = wait_bar(&bars->kv_full[stage], phase, wc, kWFwdMmaKV);
        if (++stage == S) { stage = 0; phase ^= 1u; }
        if (!ok) break;
        tc_fence_after();
        const uint32_t v_addr = kv_addr + v_stage * L::kTileBytes;
        if (j < nkv0) {
          ok = wait_bar(&bars->p_full[0], (uint32_t)(j & 1), wc, kWFwdMmaP);
          if (!ok) break;
          tc_fence_after();
          issue_pv<D>(tO0, tS0, v_addr, j > 0);
        }
        int kn_stage = -1;
        if (j + 1 < nkv) {
          kn_stage = stage;
          ok = wait_bar(&bars->kv_full[stage], phase, wc, kWFwdMmaKV);
          if (++stage == S) { stage = 0; phase ^= 1u; }
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t kn_addr = kv_addr + (kn_stage < 0 ? 0 : kn_stage) * L::kTileBytes;
        if (j + 1 < nkv0) {
          issue_qk<D>(tS0, q_addr0, kn_addr);
          mma_commit(&bars->s_full[0]);
        } else if (j == nkv0 - 1) {
          mma_commit(&bars->o_done[0]);
        }
        if (j < nkv1) {
          ok = wait_bar(&bars->p_full[1], (uint32_t)(j & 1), wc, kWFwdMmaP);
          if (!ok) break;
          tc_fence_after();
          issue_pv<D>(tO1, tS1, v_addr, j > 0);
        }
        mma_commit(&bars->kv_empty[v_stage]);
        if (j + 1 < nkv1) {
          issue_qk<D>(tS1, q_addr1, kn_addr);
          mma_commit(&bars->s_full[1]);
        } else if (j == nkv1 - 1) {
          mma_commit(&bars->o_done[1]);
        }
        if (kn_stage >= 0) mma_commit(&bars->kv_empty[kn_stage]);
      }
      // Every MMA issued above must finish before TMEM is released.
      mma_commit(&bars->mma_done);
      drain_bar(&bars->mma_done, 0, a.timeout_ns);
    }
  } else {
    // ------------------------------------------------- softmax (thread = row)
    const int t = warp >> 2, quarter = warp & 3;
    const int nkv_t = t ? nkv1 : nkv0;
    if (run && nkv_t > 0) {
      const int qrow = (2 * pair + t) * kTile + quarter * 32 + lane;
      const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
      const uint32_t tS = tl + t * 128;
      const uint32_t tO = tl + 256 + t * D;
      const float c = a.scale_log2;
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < nkv_t; ++j) {
        if (!wait_bar_warp(&bars->s_full[t], (uint32_t)(j & 1), wc, kWFwdSmS)) {
          ok = false;
          break;
        }
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
        // Mask: the diagonal tile (causal) or keys past N (ragged last tile).
        const bool masked_tile = (j == nkv_t - 1) && (CAUSAL || (a.N & (kTile - 1)));
        float mx = -INFINITY;
        if (masked_tile) {
          const int lim = (CAUSAL ? qrow : a.N - 1) - j * kTile;
#pragma unroll
          for (int e = 0; e < 128; ++e) {
            if (e > lim) s[e] = __float_as_uint(-INFINITY);
            mx = fmaxf(mx, __uint_as_float(s[e]));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 128; ++e) mx = fmaxf(mx, __uint_as_float(s[e]));
        }
        const float m_tile = mx * c;
        // Lazy rescale: keep the reference max until the row max exceeds it
        // by more than the threshold; exp2(x - m_ref) <= 2^8 meanwhile.
        const bool bump = m_tile > m_ref + kRescaleThreshold;
        float alpha = 1.f;
        if (bump) {
          alpha = ex2(m_ref - m_tile);
          m_ref = m_tile;
        }
        l *= alpha;
        if (j > 0 && __any_sync(0xffffffffu, bump)) {
          // O_t holds P V for tiles < j (the S_t(j) commit came after them).
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
        const float neg_m = -m_ref;
        uint32_t pk[64];
        float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
        for (int e = 0; e < 128; e += 4) {
          const float p0 = ex2(fmaf(__uint_as_float(s[e + 0]), c, neg_m));
          const float p1 = ex2(fmaf(__uint_as_float(s[e + 1]), c, neg_m));
          const float p2 = ex2(fmaf(__uint_as_float(s[e + 2]), c, neg_m));
          const float p3 = ex2(fmaf(__uint_as_float(s[e + 3]), c, neg_m));
          l0 += p0;
          l1 += p1;
          l2 += p2;
          l3 += p3;
          pk[e / 2] = pack_bf16(p0, p1);
          pk[e / 2 + 1] = pack_bf16(p2, p3);
        }
        l += (l0 + l1) + (l2 + l3);
        tmem_st32(tS + 0, pk);
        tmem_st32(tS + 32, pk + 32);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&bars->p_full[t]);
      }
      if (ok) ok = wait_bar_warp(&bars->o_done[t], 0, wc, kWFwdSmO);
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.0f / l;
        const bool valid = qrow < a.N;
        __nv_bfloat16* orow = a.o + ((size_t)bh * a.N + (valid ? qrow : 0)) * D;
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
            uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2],
                                   pk[4 * v4 + 3]);
          }
        }
        if (valid) a.lse[(size_t)bh * a.N + qrow] = (m_ref + lg2(l)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const FwdArgs& a, int BH,
                         cudaStream_t stream) {
  using L = FwdLayout<D>;
  auto kern = fwd_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const int n_pairs = (n_tiles + 1) / 2;
  dim3 grid((unsigned)(BH * n_pairs));
  kern<<<grid, kFwdThreads, L::kSmemBytes, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdArgs& a, int BH, int d,
                       bool causal, cudaStream_t stream) {
  if (d == 128)
    return causal ? launch_fwd_t<128, true>(tq, tk, tv, a, BH, stream)
                  : launch_fwd_t<128, false>(tq, tk, tv, a, BH, stream);
  return causal ? launch_fwd_t<64, true>(tq, tk, tv, a, BH, stream)
                : launch_fwd_t<64, false>(tq, tk, tv, a, BH, stream);
}

}  // namespace fa
