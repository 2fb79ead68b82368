// fa_common.cuh -- pieces shared by the forward and backward kernels:
// the device status record, bounded pipeline waits, tile geometry.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "fa.h"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int kTile = 128;            // rows of a Q tile and of a K/V tile
constexpr int kSwizzleBytes = 128;    // width of one swizzled smem row
constexpr int kSubTileBytes = kTile * kSwizzleBytes;  // 128 rows x 64 bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// One per GPU, in device memory owned by the library.  `status` keeps the
// first error code, `abort` tells every running block to stop at its next
// wait, `where` records which wait expired (role * 256 + site).
struct DevState {
  unsigned int status;
  unsigned int abort;
  unsigned int where;
  unsigned int blocks_aborted;
};

// Everything a bounded wait needs.
struct WaitCtl {
  DevState* st;
  uint32_t* cta_abort;  // shared-memory flag: this block is stopping
  uint64_t timeout_ns;
};

// Failure-path test hook.  In the kernel instantiations compiled with it
// (kHook), a wait whose where-code equals c_expire_site and whose barrier
// is not complete at its first test behaves as if its time limit had
// passed: it records the timeout and stops the grid like a real one.  The
// production instantiations carry none of it: even on the slow path alone
// the test cost about 1% of the backward.  One copy of the site per
// translation unit, set by the host between launches (set_expire_site_*);
// 0 (the default) matches none.
static __constant__ uint32_t c_expire_site;

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}

__device__ __forceinline__ void raise_abort(const WaitCtl& c, uint32_t where) {
  atomicCAS(&c.st->status, 0u, (unsigned)FA_ERR_DEVICE_TIMEOUT);
  atomicExch(&c.st->where, where);
  atomicExch(&c.st->abort, 1u);
  atomicAdd(&c.st->blocks_aborted, 1u);
  *reinterpret_cast<volatile uint32_t*>(c.cta_abort) = 1u;
}

// Longest a polling thread sleeps in one try_wait before it looks at the
// abort flags and the clock again (it wakes as soon as the phase completes).
constexpr uint32_t kPollHintNs = 100000;

// Wait for the phase of `bar` with the given parity.  Returns false (and
// never blocks longer than the time limit) if the wait expired here or the
// block / grid is already stopping.
template <bool kHook>
__device__ __forceinline__ bool wait_bar_poll(uint64_t* bar, uint32_t parity,
                                              const WaitCtl& c, uint32_t where) {
  // Test hook (a real wait only): skip the polling, take the timeout path.
  const bool hook = kHook && c_expire_site == where;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = hook ? 64 : 0; i < 64; ++i)
      if (mbar_try_wait_hint(bar, parity, kPollHintNs)) return true;
    if (ld_volatile_u32(c.cta_abort)) return false;
    if (*reinterpret_cast<volatile unsigned int*>(&c.st->abort)) {
      *reinterpret_cast<volatile uint32_t*>(c.cta_abort) = 1u;
      return false;
    }
    if (hook || global_timer_ns() - t0 > c.timeout_ns) {
      raise_abort(c, where);
      return false;
    }
  }
}

// Out-of-line copy of the polling loop, which keeps the waits of kernels
// compiled at one register count small.  Kernels that change their register
// count per warpgroup (setmaxnreg) cannot call functions and use the inline
// form (kInline = true).
template <bool kHook>
static __device__ __noinline__ bool wait_bar_slow(uint64_t* bar,
                                                   uint32_t parity,
                                                   WaitCtl c, uint32_t where) {
  return wait_bar_poll<kHook>(bar, parity, c, where);
}

template <bool kInline = false, bool kHook = false>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity,
                                         const WaitCtl& c, uint32_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  if constexpr (kInline) return wait_bar_poll<kHook>(bar, parity, c, where);
  else return wait_bar_slow<kHook>(bar, parity, c, where);
}

// Drain wait used only while a block is stopping: waits for an in-flight copy
// or MMA (which complete on their own) with a time limit, ignoring the abort
// flags.  Returns false if even that expired.
__device__ __forceinline__ bool drain_bar_poll(uint64_t* bar, uint32_t parity,
                                               uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
  return true;
}
static __device__ __noinline__ bool drain_bar_slow(uint64_t* bar,
                                                    uint32_t parity,
                                                    uint64_t timeout_ns) {
  return drain_bar_poll(bar, parity, timeout_ns);
}
template <bool kInline = false>
__device__ __forceinline__ bool drain_bar(uint64_t* bar, uint32_t parity,
                                          uint64_t timeout_ns) {
  if constexpr (kInline) return drain_bar_poll(bar, parity, timeout_ns);
  else return drain_bar_slow(bar, parity, timeout_ns);
}

// Warp-uniform wait: every lane waits (a single polling lane with the rest
// parked was measured markedly slower), and the warp proceeds only if all
// lanes saw the phase complete, so warp-collective tcgen05 loads/stores are
// never executed by a partial warp.
template <bool kInline = false>
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity,
                                              const WaitCtl& c,
                                              uint32_t where) {
  bool ok = wait_bar<kInline>(bar, parity, c, where);
  return __all_sync(0xffffffffu, ok);
}

// Warp-collective arrive: the warp synchronises (ordering every lane's
// earlier writes before lane 0's release) and lane 0 arrives once.  Barriers
// fed this way count warps, not threads.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Block scheduling.  Heads are taken in groups of `group` heads, sized on
// the host so one group's K/V (forward) or Q/dO/dQ rows (backward) fit in L2.
// Within a group the tile index is slow and the head fast, so the blocks
// that are resident together share few heads, and (with tile 0 the
// heaviest) the longest blocks of a group start first.
struct TileSlot {
  int bh;
  int tile;
};
__device__ __forceinline__ TileSlot grouped_slot(int linear, int n_tiles,
                                                 int BH, int group) {
  const int per_group = group * n_tiles;
  const int g = linear / per_group;
  const int r = linear - g * per_group;
  const int rest = BH - g * group;
  const int heads = rest < group ? rest : group;
  const int t = r / heads;
  return TileSlot{g * group + (r - t * heads), t};
}

// Aligns the dynamic shared memory base to 1024 bytes (128-byte swizzle atoms).
// Length of batch entry b's sequence: N without per-sequence lengths, else
// seq_lens[b] clamped to [0, N] (an out-of-range length cannot send a tile
// past the tensor).
__device__ __forceinline__ int seq_len_of(const int* seq_lens, int b, int N) {
  if (!seq_lens) return N;
  const int l = seq_lens[b];
  return l < 0 ? 0 : (l > N ? N : l);
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return reinterpret_cast<uint8_t*>((a + 1023) & ~uintptr_t(1023));
}

// Byte offset of bf16 element (row, col) inside a [128 x 64] tile stored with
// the 128-byte swizzle (16-byte chunk index XOR row % 8), as TMA writes it.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col) {
  uint32_t chunk = (col >> 3) ^ (row & 7u);
  return row * 128u + chunk * 16u + (col & 7u) * 2u;
}

}  // namespace fa
