// fa_launch.h -- internal interface between the host layer (fa_api.cu) and
// the kernel translation units (fa_fwd.cu, fa_bwd.cu).  Not part of the ABI.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fa {

struct DevState;

struct FwdArgs {
  __nv_bfloat16* o;     // [BH, N, d]
  int o_wide;           // 1: o is 32-byte aligned (rows leave in 32-byte stores)
  float* lse;           // [BH, N]
  int BH;               // batch x query heads
  int N;
  int H;                // query heads per batch entry
  int Hkv;              // key/value heads per batch entry (divides H)
  int window;           // band half-width in keys, < 0: none
  int group;            // heads per scheduling group
  float scale_log2;     // scale * log2(e): scores enter exp2 directly
  // Per-sequence lengths ([B] int32, device) or null: batch entry b attends
  // over its first seq_lens[b] rows only.
  const int* seq_lens;
  // With lengths: 1 when the kernel builds its balanced item table in shared
  // memory (set by the launcher when the table fits), else 0.
  int sched;
  // FP8 path only: per-16-row-block scales of the E4M3 Q and K,
  // [BH or BHkv][n_sblk] with n_sblk = N rounded up to 128, over 16.
  const float* q_scale;
  const float* k_scale;
  int n_sblk;
  // 1: blocks claim items from this call's work counter (a slot of a
  // zero-initialised ring, with its count of finished blocks; the last
  // block resets both); 0: items are dealt in alternating rounds.  Calls
  // with a window always use 0.
  int dynamic;
  // 1: each work item is one Q tile instead of a pair (set when a problem
  // has fewer pairs than SMs; never with per-sequence lengths).
  int single;
  unsigned int* work_next;
  unsigned int* work_done;
  int hook;           // 1: run the failure-path test hook instantiation
  DevState* st;
  uint64_t timeout_ns;
};

struct BwdArgs {
  const __nv_bfloat16* o;     // [BH, N, d]
  const __nv_bfloat16* dout;  // [BH, N, d]
  const float* lse;           // [BH, N]
  float* dq_acc;              // [BH, N, d]  fp32 workspace
  float* ddot;                // [BH, N_pad] D_i = dO_i . O_i  (0 past N)
  float* lse2;                // [BH, N_pad] -LSE_i * log2(e)  (-inf past N)
  __nv_bfloat16* dq;          // [BH, N, d]
  __nv_bfloat16* dk;          // [BHkv, N, d]
  __nv_bfloat16* dv;          // [BHkv, N, d]
  float* dk_acc;              // [BHkv, N, d] fp32, used when nsplit > 1
  float* dv_acc;              // [BHkv, N, d] fp32, used when nsplit > 1
  int BH;                     // batch x query heads
  int BHkv;                   // batch x key/value heads
  int H;                      // query heads per batch entry
  int Hkv;                    // key/value heads per batch entry (divides H)
  int window;                 // band half-width in keys, < 0: none
  const int* seq_lens;        // [B] int32 per-sequence lengths, or null
  int hpb;                    // query heads per block (divides H / Hkv)
  int nsplit;                 // blocks per (key/value head, key tile)
  int N;
  int N_pad;                  // N rounded up to a multiple of 128
  int group;                  // key/value heads per scheduling group
  float scale;
  float scale_log2;
  unsigned int* work_next;    // main kernel's work counter (workspace)
  int hook;                   // 1: run the failure-path test hook instantiation
  DevState* st;
  uint64_t timeout_ns;
};

// Each returns the launch error (cudaSuccess on success).  `to` maps O
// ([BH, N, d] bf16, boxes of 32 rows x 64 columns, 128-byte swizzle) for the
// kernels that store O by TMA.
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to,
                       const FwdArgs& a, int BH, int d, bool causal,
                       int grid_blocks, cudaStream_t stream);
// FP8 forward: tq, tk are E4M3 tensor maps (one byte per element, rows of
// 128 bytes: at d = 64 the upper half of each row is zero), tv the bf16 V
// map; d = 64 or 128.
cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to,
                           const FwdArgs& a, int BH, int d, bool causal,
                           int grid_blocks, cudaStream_t stream);
// E4M3 codes and per-16-row-block scales of a bf16 [BH, N, d] tensor
// (d = 64 or 128); scales has BH * n_sblk entries, 1 for blocks past N.
// Code rows are `pitch` bytes apart (>= d), bytes d .. pitch - 1 zero.
cudaError_t launch_quant_e4m3(const __nv_bfloat16* x, uint8_t* codes,
                              float* scales, int BH, int N, int d, int n_sblk,
                              int pitch, int grid_blocks, cudaStream_t stream);
cudaError_t launch_bwd_pre(const BwdArgs& a, int d, int grid_blocks,
                           cudaStream_t stream);
// Persistent: min(work items, grid_blocks) blocks, one per SM.
cudaError_t launch_bwd_main(const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tdq, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, const BwdArgs& a, int d,
                            bool causal, int grid_blocks, cudaStream_t stream);
cudaError_t launch_bwd_post(const BwdArgs& a, int d, int grid_blocks,
                            cudaStream_t stream);
cudaError_t launch_expire_wait(DevState* st, uint64_t timeout_ns,
                               cudaStream_t stream);
// The failure-path test hook of the forward / backward kernels (the site
// whose waits expire at once, 0 for none), for the current device.
// Synchronous; call only while no kernel of the library runs.
cudaError_t set_expire_site_fwd(uint32_t site);
cudaError_t set_expire_site_bwd(uint32_t site);

}  // namespace fa
