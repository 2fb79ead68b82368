// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// checks, TMA descriptor encoding, launch sequencing, the per-GPU device
// status record, and the wait-expiry self-test kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_common.cuh"
#include "fa_launch.h"

namespace {

__device__ fa::DevState g_dev_state;  // zero-initialised at module load
// Work counters of forward calls: (next item, finished blocks) per slot,
// zero-initialised; each call takes the next slot and its last block sets
// the pair back to zero.  Calls more than kFwdSchedSlots apart may reuse a
// slot only after the earlier one has finished.
constexpr unsigned kFwdSchedSlots = 64;
__device__ unsigned int g_fwd_sched[kFwdSchedSlots][2];

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s
std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};

uint64_t kernel_timeout() { return g_timeout_ns.load(); }
// Set while the failure-path test hook has a site: launches then use the
// instantiations compiled with the hook.
std::atomic<bool> g_hook_on{false};

constexpr int kMaxDevices = 64;
constexpr int kMaxN = 1 << 30;  // keeps every row index inside int

struct DeviceCtx {
  bool ready = false;
  fa::DevState* state = nullptr;
  unsigned int* fwd_sched = nullptr;  // device address of g_fwd_sched
  std::atomic<unsigned> fwd_slot{0};
  int sm_count = 0;
};
DeviceCtx g_ctx[kMaxDevices];
std::mutex g_ctx_mu;

thread_local uint32_t g_last_where = 0;  // site of the last reported failure
thread_local cudaEvent_t g_ev_before_main = nullptr;
thread_local cudaEvent_t g_ev_after_main = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// Per-device set-up: device address of the status record, SM count.
fa_status device_ctx(DeviceCtx** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_ctx_mu);
  DeviceCtx& c = g_ctx[dev];
  if (!c.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_state) != cudaSuccess) return FA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
      return FA_ERR_CUDA;
    void* ps = nullptr;
    if (cudaGetSymbolAddress(&ps, g_fwd_sched) != cudaSuccess) return FA_ERR_CUDA;
    c.state = static_cast<fa::DevState*>(p);
    c.fwd_sched = static_cast<unsigned int*>(ps);
    c.sm_count = sms;
    c.ready = true;
  }
  *out = &c;
  return FA_OK;
}

// The work counter slot of one forward call.
void fwd_sched_slot(DeviceCtx* ctx, fa::FwdArgs& a) {
  const unsigned slot = ctx->fwd_slot.fetch_add(1u) % kFwdSchedSlots;
  a.work_next = ctx->fwd_sched + 2 * slot;
  a.work_done = a.work_next + 1;
}

// Schedule of the forward.  When every head's K and V (4 d bytes per row
// and head) fit in L2 together, or a window is set (a band's K and V stay in
// L2 anyway), one group of all heads, dealt in alternating rounds (measured
// best there: the last items are the lightest of all).  Otherwise groups of
// as many heads as keep their K and V within a share of L2, with items
// claimed dynamically (a separate kernel instantiation) so that the groups
// cost no balance.
void fwd_schedule(int BH, int N, int d, fa::FwdArgs& a) {
  constexpr size_t kAll = 96u << 20, kBudget = 48u << 20;
  const size_t per_head = (size_t)4 * N * d;
  // (With per-sequence lengths the call always runs with a window, N - 1
  // at widest, so it takes this branch too.)
  if (a.window >= 0 || per_head * (size_t)BH <= kAll) {
    a.group = BH;
    a.dynamic = 0;
    return;
  }
  size_t g = per_head ? kBudget / per_head : (size_t)BH;
  if (g < 1) g = 1;
  if (g > (size_t)BH) g = (size_t)BH;
  a.group = (int)g;
  a.dynamic = 1;
}

// Forward work items of one Q tile instead of two when a problem has fewer
// pairs of Q tiles than SMs (then most SMs would idle); the two tiles of a
// pair share their K/V loads, so pairs stay the unit otherwise.  The
// kernels with per-sequence lengths keep pairs (their balanced item table
// counts pairs).
int single_tile_items(int BH, int N, int sm_count, bool lengths) {
  const long long pairs = (long long)BH * (((N + fa::kTile - 1) / fa::kTile + 1) / 2);
  return (!lengths && pairs < sm_count) ? 1 : 0;
}

fa_status encode_fn(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!g_encode) return FA_ERR_CUDA;
  *fn = g_encode;
  return FA_OK;
}

// 3-D view [BH][N][d] of a bf16 [B,H,N,d] tensor; box = `box_rows` rows x 64
// columns (128 bytes, the swizzle width).  Rows past N read as zeros.
fa_status make_tile_map(CUtensorMap* m, const void* base, int BH, int N,
                        int d, int box_rows = fa::kTile) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  fa_status s = encode_fn(&fn);
  if (s != FA_OK) return s;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 3-D view [BH][N][d] of the fp32 dQ accumulator; box = 32 rows x 32
// columns (128 bytes), 128-byte swizzle: one drain warp's rows of one
// 32-column group.  Reduce-adds clip rows past N.
fa_status make_acc_map(CUtensorMap* m, const void* base, int BH, int N,
                       int d) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  fa_status s = encode_fn(&fn);
  if (s != FA_OK) return s;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * d * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 3-D view [BH][N][row_bytes] of an E4M3 tensor (one byte per element);
// box = 128 rows x 128 bytes, 128-byte swizzle.  Rows past N read as zeros.
fa_status make_fp8_map(CUtensorMap* m, const void* base, int BH, int N,
                       int d) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  fa_status s = encode_fn(&fn);
  if (s != FA_OK) return s;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)N * d};
  cuuint32_t box[3] = {128, (cuuint32_t)fa::kTile, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Shared shape/scalar checks.  *empty is set for a problem with no elements.
fa_status check_shape(int B, int H, int N, int d, int causal, float scale,
                      bool* empty) {
  *empty = false;
  if (B < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return FA_ERR_INVALID_ARG;
  if (d <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H > INT_MAX) return FA_ERR_UNSUPPORTED;
  if (N > kMaxN) return FA_ERR_UNSUPPORTED;
  // One block per (head, 128-row tile) must fit a 31-bit grid.
  if ((long long)B * H * ((N + fa::kTile - 1) / fa::kTile) > INT_MAX)
    return FA_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) *empty = true;
  return FA_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Checks of the grouped-head / window arguments on top of check_shape.
// H query heads share Hkv key/value heads (Hkv divides H); window < 0 means
// no band.  A window of N - 1 or more hides nothing and is returned as -1.
fa_status check_ext(int H, int Hkv, int N, int window, int* window_out) {
  if (Hkv < 0) return FA_ERR_INVALID_ARG;
  if (H > 0 && (Hkv == 0 || Hkv > H || H % Hkv != 0)) return FA_ERR_INVALID_ARG;
  *window_out = (window < 0 || (long long)window >= (long long)N - 1) ? -1 : window;
  return FA_OK;
}

// Heads per scheduling group: as many heads as keep `bytes_per_head` of
// re-read data within an L2 budget, at least one.
int heads_per_group(int BH, size_t bytes_per_head) {
  constexpr size_t kL2Budget = 32u << 20;
  size_t g = bytes_per_head ? kL2Budget / bytes_per_head : (size_t)BH;
  if (g < 1) g = 1;
  if (g > (size_t)BH) g = (size_t)BH;
  return (int)g;
}

// Query heads per backward block: the largest divisor of the group size
// H / Hkv not above kMaxHeadsPerBlock.  A larger group is split over
// several blocks per (key/value head, key tile), which then sum dK, dV in
// fp32 workspace.
constexpr int kMaxHeadsPerBlock = 8;
int heads_per_block(int qgroup) {
  for (int h = qgroup < kMaxHeadsPerBlock ? qgroup : kMaxHeadsPerBlock; h > 1; --h)
    if (qgroup % h == 0) return h;
  return 1;
}

struct WsLayout {
  size_t dq_acc_off, ddot_off, lse2_off, sched_off, dk_acc_off, dv_acc_off, total;
  int hpb, nsplit;
};

// dQacc [B,H,N,d] | D [B*H, N_pad] | LSE2 [B*H, N_pad] | the main kernel's
// work counter (256 bytes) (| dKacc, dVacc [B,Hkv,N,d] when the group is
// split), each 256-byte aligned.
WsLayout ws_layout(int B, int H, int Hkv, int N, int d) {
  const size_t BH = (size_t)B * H, BHkv = (size_t)B * Hkv;
  const size_t n_pad = align_up((size_t)N, fa::kTile);
  WsLayout w;
  const int qgroup = Hkv > 0 ? H / Hkv : 1;
  w.hpb = heads_per_block(qgroup);
  w.nsplit = qgroup / w.hpb;
  w.dq_acc_off = 0;
  w.ddot_off = align_up(BH * N * d * sizeof(float), 256);
  w.lse2_off = w.ddot_off + align_up(BH * n_pad * sizeof(float), 256);
  w.sched_off = w.lse2_off + align_up(BH * n_pad * sizeof(float), 256);
  w.dk_acc_off = w.sched_off + 256;
  const size_t kv_acc = w.nsplit > 1 ? align_up(BHkv * N * d * sizeof(float), 256) : 0;
  w.dv_acc_off = w.dk_acc_off + kv_acc;
  w.total = w.dv_acc_off + kv_acc;
  return w;
}

// Scale blocks (16 rows) per head, counted over N rounded up to 128.
int scale_blocks(int N) { return (int)(align_up((size_t)N, fa::kTile) / 16); }

struct Fp8Layout {
  size_t q8_off, k8_off, sq_off, sk_off, total;
};

// E4M3 rows of the FP8 forward: 128 bytes whatever d (d = 64 rows carry 64
// zero bytes, so that Q K^T is the d = 128 product).
constexpr int kFp8RowBytes = 128;

// E4M3 Q | E4M3 K (B*H*N rows of kFp8RowBytes each) | Q scales | K scales
// ([B*H][scale_blocks(N)] float32), each 256-byte aligned.
Fp8Layout fp8_layout(int B, int H, int N, int /*d*/) {
  const size_t BH = (size_t)B * H;
  Fp8Layout w;
  w.q8_off = 0;
  w.k8_off = align_up(BH * N * kFp8RowBytes, 256);
  w.sq_off = w.k8_off + align_up(BH * N * kFp8RowBytes, 256);
  w.sk_off = w.sq_off + align_up(BH * scale_blocks(N) * sizeof(float), 256);
  w.total = w.sk_off + align_up(BH * scale_blocks(N) * sizeof(float), 256);
  return w;
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
  }
  return "FA_ERR_UNKNOWN";
}

void fa_debug_expire_at(uint32_t site) {
  (void)fa::set_expire_site_fwd(site);
  (void)fa::set_expire_site_bwd(site);
  g_hook_on.store(site != 0);
}

void fa_set_wait_timeout_ns(uint64_t ns) {
  g_timeout_ns.store(ns == 0 ? kDefaultTimeoutNs : ns);
}

}  // extern "C"

namespace {

fa_status fwd_impl(const void* q, const void* k, const void* v, void* o,
                   float* lse, const int* seq_lens, int B, int H, int Hkv,
                   int N, int d, int causal, int window, float scale,
                   void* stream) {
  bool empty = false;
  fa_status s = check_shape(B, H, N, d, causal, scale, &empty);
  if (s != FA_OK) return s;
  int win = -1;
  if ((s = check_ext(H, Hkv, N, window, &win)) != FA_OK || empty) return s;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  DeviceCtx* ctx = nullptr;
  if ((s = device_ctx(&ctx)) != FA_OK) return s;
  const int BH = B * H, BHkv = B * Hkv;
  CUtensorMap tq, tk, tv;
  if ((s = make_tile_map(&tq, q, BH, N, d)) != FA_OK) return s;
  if ((s = make_tile_map(&tk, k, BHkv, N, d)) != FA_OK) return s;
  if ((s = make_tile_map(&tv, v, BHkv, N, d)) != FA_OK) return s;
  CUtensorMap to;  // O, stored by TMA in 32-row boxes
  if ((s = make_tile_map(&to, o, BH, N, d, 32)) != FA_OK) return s;
  fa::FwdArgs a{};
  a.o = static_cast<__nv_bfloat16*>(o);
  a.o_wide = aligned(o, 32) ? 1 : 0;
  a.lse = lse;
  a.BH = BH;
  a.N = N;
  a.H = H;
  a.Hkv = Hkv;
  // Only the windowed forward kernels read per-sequence lengths; a window
  // of N - 1 hides no key, so a call with lengths and no window runs there.
  a.window = (seq_lens && win < 0) ? N - 1 : win;
  a.seq_lens = seq_lens;
  fwd_schedule(BH, N, d, a);
  a.single = single_tile_items(BH, N, ctx->sm_count, seq_lens != nullptr);
  a.scale_log2 = scale * fa::kLog2e;
  a.st = ctx->state;
  a.timeout_ns = kernel_timeout();
  a.hook = g_hook_on.load() ? 1 : 0;
  fwd_sched_slot(ctx, a);
  cudaError_t e = fa::launch_fwd(tq, tk, tv, to, a, BH, d, causal != 0,
                                 ctx->sm_count, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

fa_status fa_fwd_ext(const void* q, const void* k, const void* v, void* o,
                     float* lse, int B, int H, int Hkv, int N, int d,
                     int causal, int window, float scale, void* stream) {
  return fwd_impl(q, k, v, o, lse, nullptr, B, H, Hkv, N, d, causal, window,
                  scale, stream);
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o,
                        float* lse, const int* seq_lens, int B, int H, int Hkv,
                        int N, int d, int causal, int window, float scale,
                        void* stream) {
  if (B > 0 && (!seq_lens || !aligned(seq_lens, 4))) return FA_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, seq_lens, B, H, Hkv, N, d, causal, window,
                  scale, stream);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o,
                 float* lse, int B, int H, int N, int d, int causal,
                 float scale, void* stream) {
  return fwd_impl(q, k, v, o, lse, nullptr, B, H, H, N, d, causal, -1, scale,
                  stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  bool empty = false;
  if (check_shape(B, H, N, d, 0, 1.0f, &empty) != FA_OK || empty) return 0;
  return ws_layout(B, H, H, N, d).total;
}

size_t fa_bwd_ext_workspace_size(int B, int H, int Hkv, int N, int d) {
  bool empty = false;
  int win = -1;
  if (check_shape(B, H, N, d, 0, 1.0f, &empty) != FA_OK || empty) return 0;
  if (check_ext(H, Hkv, N, -1, &win) != FA_OK) return 0;
  return ws_layout(B, H, Hkv, N, d).total;
}

}  // extern "C"

namespace {

// Records a measurement event on `st`: as an external event node while the
// stream is being captured into a CUDA graph (so that every run of the graph
// records it), as a plain record otherwise.
cudaError_t record_phase_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
             : cudaEventRecord(ev, st);
}

fa_status bwd_impl(const void* q, const void* k, const void* v,
                   const void* o, const float* lse, const void* dout,
                   void* dq, void* dk, void* dv, const int* seq_lens,
                   void* workspace, size_t workspace_bytes, int B, int H,
                   int Hkv, int N, int d, int causal, int window, float scale,
                   void* stream) {
  bool empty = false;
  fa_status s = check_shape(B, H, N, d, causal, scale, &empty);
  if (s != FA_OK) return s;
  int win = -1;
  if ((s = check_ext(H, Hkv, N, window, &win)) != FA_OK || empty) return s;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv)
    return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(o, 16) || !aligned(dout, 16) || !aligned(dq, 16) ||
      !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(B, H, Hkv, N, d);
  if (!workspace || !aligned(workspace, 16) || workspace_bytes < w.total)
    return FA_ERR_WORKSPACE;
  DeviceCtx* ctx = nullptr;
  if ((s = device_ctx(&ctx)) != FA_OK) return s;
  const int BH = B * H, BHkv = B * Hkv;
  char* ws = static_cast<char*>(workspace);
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  if ((s = make_tile_map(&tq, q, BH, N, d)) != FA_OK) return s;
  if ((s = make_tile_map(&tk, k, BHkv, N, d)) != FA_OK) return s;
  if ((s = make_tile_map(&tv, v, BHkv, N, d)) != FA_OK) return s;
  if ((s = make_tile_map(&tdo, dout, BH, N, d)) != FA_OK) return s;
  // dK, dV leave the main kernel in [32 rows x 64 columns] boxes, one per
  // warp and 64-column half.
  if ((s = make_tile_map(&tdk, dk, BHkv, N, d, 32)) != FA_OK) return s;
  if ((s = make_tile_map(&tdv, dv, BHkv, N, d, 32)) != FA_OK) return s;
  if ((s = make_acc_map(&tdq, ws + w.dq_acc_off, BH, N, d)) != FA_OK) return s;
  fa::BwdArgs a{};
  a.o = static_cast<const __nv_bfloat16*>(o);
  a.dout = static_cast<const __nv_bfloat16*>(dout);
  a.lse = lse;
  a.dq_acc = reinterpret_cast<float*>(ws + w.dq_acc_off);
  a.ddot = reinterpret_cast<float*>(ws + w.ddot_off);
  a.lse2 = reinterpret_cast<float*>(ws + w.lse2_off);
  a.dq = static_cast<__nv_bfloat16*>(dq);
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.dk_acc = reinterpret_cast<float*>(ws + w.dk_acc_off);
  a.work_next = reinterpret_cast<unsigned int*>(ws + w.sched_off);
  a.dv_acc = reinterpret_cast<float*>(ws + w.dv_acc_off);
  a.hpb = w.hpb;
  a.nsplit = w.nsplit;
  a.seq_lens = seq_lens;
  a.BH = BH;
  a.BHkv = BHkv;
  a.H = H;
  a.Hkv = Hkv;
  a.window = win;
  a.N = N;
  a.N_pad = (int)align_up((size_t)N, fa::kTile);
  // Re-read per block row of the schedule (a key/value head, or one split
  // of its query heads): Q and dO (bf16) and the fp32 dQ accumulator of its
  // query heads.
  a.group = heads_per_group(BHkv * w.nsplit, (size_t)8 * N * d * w.hpb);
  a.scale = scale;
  a.scale_log2 = scale * fa::kLog2e;
  a.st = ctx->state;
  a.timeout_ns = kernel_timeout();
  a.hook = g_hook_on.load() ? 1 : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int elem_blocks = ctx->sm_count * 8;
  cudaError_t e = fa::launch_bwd_pre(a, d, elem_blocks, st);
  if (e == cudaSuccess && g_ev_before_main)
    e = record_phase_event(g_ev_before_main, st);
  if (e == cudaSuccess)
    e = fa::launch_bwd_main(tq, tk, tv, tdo, tdq, tdk, tdv, a, d, causal != 0,
                            ctx->sm_count, st);
  if (e == cudaSuccess && g_ev_after_main)
    e = record_phase_event(g_ev_after_main, st);
  if (e == cudaSuccess) e = fa::launch_bwd_post(a, d, elem_blocks, st);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

fa_status fa_bwd_ext(const void* q, const void* k, const void* v,
                     const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, int B, int H, int Hkv, int N,
                     int d, int causal, int window, float scale,
                     void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, nullptr, workspace,
                  workspace_bytes, B, H, Hkv, N, d, causal, window, scale,
                  stream);
}

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* dout,
                        void* dq, void* dk, void* dv, const int* seq_lens,
                        void* workspace, size_t workspace_bytes, int B, int H,
                        int Hkv, int N, int d, int causal, int window,
                        float scale, void* stream) {
  if (B > 0 && (!seq_lens || !aligned(seq_lens, 4))) return FA_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, seq_lens, workspace,
                  workspace_bytes, B, H, Hkv, N, d, causal, window, scale,
                  stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dout, void* dq, void* dk,
                 void* dv, void* workspace, size_t workspace_bytes, int B,
                 int H, int N, int d, int causal, float scale, void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, nullptr, workspace,
                  workspace_bytes, B, H, H, N, d, causal, -1, scale, stream);
}

size_t fa_fwd_fp8_workspace_size(int B, int H, int N, int d) {
  bool empty = false;
  if (check_shape(B, H, N, d, 0, 1.0f, &empty) != FA_OK || empty) return 0;
  return fp8_layout(B, H, N, d).total;
}

fa_status fa_quantize_e4m3(const void* x, void* codes, float* scales, int BH,
                           int N, int d, void* stream) {
  bool empty = false;
  fa_status s = check_shape(1, BH, N, d, 0, 1.0f, &empty);
  if (s != FA_OK || empty) return s;
  if (!x || !codes || !scales) return FA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4))
    return FA_ERR_INVALID_ARG;
  DeviceCtx* ctx = nullptr;
  if ((s = device_ctx(&ctx)) != FA_OK) return s;
  cudaError_t e = fa::launch_quant_e4m3(
      static_cast<const __nv_bfloat16*>(x), static_cast<uint8_t*>(codes),
      scales, BH, N, d, scale_blocks(N), d, ctx->sm_count * 8,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o,
                     float* lse, void* workspace, size_t workspace_bytes,
                     int B, int H, int N, int d, int causal, float scale,
                     void* stream) {
  bool empty = false;
  fa_status s = check_shape(B, H, N, d, causal, scale, &empty);
  if (s != FA_OK || empty) return s;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  const Fp8Layout w = fp8_layout(B, H, N, d);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < w.total)
    return FA_ERR_WORKSPACE;
  DeviceCtx* ctx = nullptr;
  if ((s = device_ctx(&ctx)) != FA_OK) return s;
  const int BH = B * H;
  char* ws = static_cast<char*>(workspace);
  uint8_t* q8 = reinterpret_cast<uint8_t*>(ws + w.q8_off);
  uint8_t* k8 = reinterpret_cast<uint8_t*>(ws + w.k8_off);
  float* sq = reinterpret_cast<float*>(ws + w.sq_off);
  float* sk = reinterpret_cast<float*>(ws + w.sk_off);
  CUtensorMap tq, tk, tv;
  if ((s = make_fp8_map(&tq, q8, BH, N, kFp8RowBytes)) != FA_OK) return s;
  if ((s = make_fp8_map(&tk, k8, BH, N, kFp8RowBytes)) != FA_OK) return s;
  if ((s = make_tile_map(&tv, v, BH, N, d)) != FA_OK) return s;
  CUtensorMap to;  // O (the FP8 kernels store it from registers)
  if ((s = make_tile_map(&to, o, BH, N, d, 32)) != FA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int nsb = scale_blocks(N);
  cudaError_t e = fa::launch_quant_e4m3(static_cast<const __nv_bfloat16*>(q),
                                        q8, sq, BH, N, d, nsb, kFp8RowBytes,
                                        ctx->sm_count * 8, st);
  if (e == cudaSuccess)
    e = fa::launch_quant_e4m3(static_cast<const __nv_bfloat16*>(k), k8, sk, BH,
                              N, d, nsb, kFp8RowBytes, ctx->sm_count * 8, st);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  fa::FwdArgs a{};
  a.o = static_cast<__nv_bfloat16*>(o);
  a.o_wide = aligned(o, 32) ? 1 : 0;
  a.lse = lse;
  a.BH = BH;
  a.N = N;
  a.H = H;
  a.Hkv = H;
  a.window = -1;
  fwd_schedule(BH, N, d, a);
  a.single = single_tile_items(BH, N, ctx->sm_count, false);
  a.scale_log2 = scale * fa::kLog2e;
  a.q_scale = sq;
  a.k_scale = sk;
  a.n_sblk = nsb;
  a.st = ctx->state;
  a.timeout_ns = kernel_timeout();
  a.hook = g_hook_on.load() ? 1 : 0;
  fwd_sched_slot(ctx, a);
  e = fa::launch_fwd_fp8(tq, tk, tv, to, a, BH, d, causal != 0, ctx->sm_count, st);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

void fa_bwd_set_phase_events(void* before_main, void* after_main) {
  g_ev_before_main = static_cast<cudaEvent_t>(before_main);
  g_ev_after_main = static_cast<cudaEvent_t>(after_main);
}

fa_status fa_check_device_status(void* stream) {
  DeviceCtx* ctx = nullptr;
  fa_status s = device_ctx(&ctx);
  if (s != FA_OK) return s;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  fa::DevState h{};
  if (cudaMemcpy(&h, ctx->state, sizeof(h), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  g_last_where = 0;
  if (h.status == 0 && h.abort == 0) return FA_OK;
  g_last_where = h.where;
  if (cudaMemset(ctx->state, 0, sizeof(fa::DevState)) != cudaSuccess)
    return FA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  return h.status != 0 ? static_cast<fa_status>(h.status)
                       : FA_ERR_DEVICE_TIMEOUT;
}

uint32_t fa_last_failure_site(void) { return g_last_where; }

fa_status fa_debug_expire_wait(void* stream) {
  DeviceCtx* ctx = nullptr;
  fa_status s = device_ctx(&ctx);
  if (s != FA_OK) return s;
  cudaError_t e = fa::launch_expire_wait(ctx->state, kernel_timeout(),
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
// ---------------------------------------------------------------------------
// Backward pass without any device allocation by the caller or the library.
//
// Some callers cannot obtain device memory at the point where they run the
// backward pass: code that owns no allocator (a plug-in handed only the
// tensors), serving or training loops that reserve all memory up front and
// forbid allocation on the hot path, and code that must not call cudaMalloc
// because it synchronises the device.  For them the workspace lives in a
// fixed array in device memory that every GPU which loads this library keeps
// until the process exits.
//
// On the first call on a device (with that device current) the array's
// device address is looked up once with cudaGetSymbolAddress; make that first
// call before any stream capture.  All calls share the array: two calls whose
// kernels overlap on the GPU (different streams, or other threads) race on
// it.  Nothing in it needs to start at zero across calls: the pre kernel
// rewrites every part the backward reads (D, LSE*log2e, and a zeroed dQ
// accumulator) on every call.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
void* g_noalloc_addr[kMaxDevices] = {};
std::mutex g_noalloc_mu;
}  // namespace

extern "C" size_t fa_bwd_noalloc_max_workspace(void) { return kNoAllocScratchBytes; }

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v,
                                    const void* o, const float* lse,
                                    const void* dout, void* dq, void* dk,
                                    void* dv, int B, int H, int N, int d,
                                    int causal, float scale, void* stream) {
  bool empty = false;
  fa_status s = check_shape(B, H, N, d, causal, scale, &empty);
  if (s != FA_OK || empty) return s;
  if (ws_layout(B, H, H, N, d).total > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return FA_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
        return FA_ERR_CUDA;
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, scratch,
                kNoAllocScratchBytes, B, H, N, d, causal, scale, stream);
}

// ---------------------------------------------------------------------------
// Training step on host-resident tensors, pipelined by chunks of heads.
//
// Heads are independent, so the step runs chunk by chunk (flat head index
// over B*H; each chunk is one contiguous block of every [B,H,N,d] tensor):
// the inputs of chunk c+1 are copied in on one stream while chunk c computes
// on the caller's stream and the outputs of chunk c-1 are copied out on a
// third, so both copy directions overlap each other and the kernels.  Three
// device slots (inputs, outputs, backward workspace of one chunk each) rotate
// over the chunks; a slot is refilled only after the outputs it held have
// been copied out.
namespace fa {
namespace {

constexpr int kSlots = 3;
// Copy streams per direction (two were measured no faster: the host link,
// not the number of copy engines, limits the copies).
constexpr int kCopyStreams = 1;

struct HostPipe {
  bool ready = false;
  cudaStream_t h2d[kCopyStreams] = {}, d2h[kCopyStreams] = {};
  cudaEvent_t start = nullptr;
  cudaEvent_t in_done[kSlots][kCopyStreams] = {}, comp_done[kSlots] = {},
              out_done[kSlots][kCopyStreams] = {}, end[kCopyStreams] = {};
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

fa_status host_pipe(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe& p = g_pipe[dev];
  if (!p.ready) {
    const unsigned fl = cudaEventDisableTiming;
    if (cudaEventCreateWithFlags(&p.start, fl) != cudaSuccess) return FA_ERR_CUDA;
    for (int c = 0; c < kCopyStreams; ++c)
      if (cudaStreamCreateWithFlags(&p.h2d[c], cudaStreamNonBlocking) != cudaSuccess ||
          cudaStreamCreateWithFlags(&p.d2h[c], cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.end[c], fl) != cudaSuccess)
        return FA_ERR_CUDA;
    for (int i = 0; i < kSlots; ++i) {
      if (cudaEventCreateWithFlags(&p.comp_done[i], fl) != cudaSuccess)
        return FA_ERR_CUDA;
      for (int c = 0; c < kCopyStreams; ++c)
        if (cudaEventCreateWithFlags(&p.in_done[i][c], fl) != cudaSuccess ||
            cudaEventCreateWithFlags(&p.out_done[i][c], fl) != cudaSuccess)
          return FA_ERR_CUDA;
    }
    p.ready = true;
  }
  *out = &p;
  return FA_OK;
}

struct SlotLayout {
  size_t tensor, lse, ws, total;  // bytes: one [ch,N,d] bf16 tensor, ...
};

// One slot: q, k, v, dO, O, dQ, dK, dV ([ch,N,d] bf16 each), LSE, and the
// backward workspace of ch heads, each 256-byte aligned.
SlotLayout slot_layout(int ch, int N, int d) {
  SlotLayout s;
  s.tensor = align_up((size_t)ch * N * d * 2, 256);
  s.lse = align_up((size_t)ch * N * 4, 256);
  s.ws = align_up(ws_layout(1, ch, ch, N, d).total, 256);
  s.total = 8 * s.tensor + s.lse + s.ws;
  return s;
}

int chunk_heads_or_default(int BH, int chunk_heads) {
  if (chunk_heads > 0) return chunk_heads < BH ? chunk_heads : BH;
  const int c = (BH + 15) / 16;  // about sixteen chunks (measured best)
  return c > 0 ? c : 1;
}

}  // namespace
}  // namespace fa

extern "C" size_t fa_step_host_scratch_size(int B, int H, int N, int d,
                                            int chunk_heads) {
  bool empty = false;
  if (check_shape(B, H, N, d, 0, 1.0f, &empty) != FA_OK || empty) return 0;
  const int ch = fa::chunk_heads_or_default(B * H, chunk_heads);
  return (size_t)fa::kSlots * fa::slot_layout(ch, N, d).total;
}

extern "C" fa_status fa_step_host(const void* q, const void* k, const void* v,
                                  const void* dout, void* o, float* lse,
                                  void* dq, void* dk, void* dv, void* scratch,
                                  size_t scratch_bytes, int B, int H, int N,
                                  int d, int causal, float scale,
                                  int chunk_heads, void* stream) {
  bool empty = false;
  fa_status s = check_shape(B, H, N, d, causal, scale, &empty);
  if (s != FA_OK || empty) return s;
  if (chunk_heads < 0) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !dout || !o || !lse || !dq || !dk || !dv)
    return FA_ERR_INVALID_ARG;
  const int BH = B * H;
  const int ch = fa::chunk_heads_or_default(BH, chunk_heads);
  const fa::SlotLayout L = fa::slot_layout(ch, N, d);
  if (!scratch || !aligned(scratch, 256) ||
      scratch_bytes < (size_t)fa::kSlots * L.total)
    return FA_ERR_WORKSPACE;
  fa::HostPipe* p = nullptr;
  if ((s = fa::host_pipe(&p)) != FA_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // Everything already on the caller's stream comes first.
  if (cudaEventRecord(p->start, cs) != cudaSuccess) return FA_ERR_CUDA;
  for (int c = 0; c < fa::kCopyStreams; ++c)
    if (cudaStreamWaitEvent(p->h2d[c], p->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(p->d2h[c], p->start, 0) != cudaSuccess)
      return FA_ERR_CUDA;
  const size_t row_bytes = (size_t)N * d * 2;  // one head of one tensor
  const int n_chunks = (BH + ch - 1) / ch;
  const void* in_h[4] = {q, k, v, dout};
  void* out_h[4] = {o, dq, dk, dv};
  for (int c = 0; c < n_chunks; ++c) {
    const int slot = c % fa::kSlots;
    const int h0 = c * ch;
    const int hc = BH - h0 < ch ? BH - h0 : ch;
    char* base = static_cast<char*>(scratch) + (size_t)slot * L.total;
    char* t[8];
    for (int i = 0; i < 8; ++i) t[i] = base + (size_t)i * L.tensor;
    float* lse_d = reinterpret_cast<float*>(base + 8 * L.tensor);
    void* ws_d = base + 8 * L.tensor + L.lse;
    const size_t bytes = (size_t)hc * row_bytes;
    // inputs of chunk c, tensor i on copy stream i % kCopyStreams, after the
    // slot's previous outputs have left
    for (int cc = 0; cc < fa::kCopyStreams; ++cc)
      if (c >= fa::kSlots)
        for (int dc = 0; dc < fa::kCopyStreams; ++dc)
          if (cudaStreamWaitEvent(p->h2d[cc], p->out_done[slot][dc], 0) != cudaSuccess)
            return FA_ERR_CUDA;
    for (int i = 0; i < 4; ++i)
      if (cudaMemcpyAsync(t[i], static_cast<const char*>(in_h[i]) + (size_t)h0 * row_bytes,
                          bytes, cudaMemcpyHostToDevice,
                          p->h2d[i % fa::kCopyStreams]) != cudaSuccess)
        return FA_ERR_CUDA;
    for (int cc = 0; cc < fa::kCopyStreams; ++cc)
      if (cudaEventRecord(p->in_done[slot][cc], p->h2d[cc]) != cudaSuccess ||
          cudaStreamWaitEvent(cs, p->in_done[slot][cc], 0) != cudaSuccess)
        return FA_ERR_CUDA;
    // compute on the caller's stream
    if ((s = fa_fwd(t[0], t[1], t[2], t[4], lse_d, 1, hc, N, d, causal, scale,
                    stream)) != FA_OK)
      return s;
    if ((s = fa_bwd(t[0], t[1], t[2], t[4], lse_d, t[3], t[5], t[6], t[7],
                    ws_d, L.ws, 1, hc, N, d, causal, scale, stream)) != FA_OK)
      return s;
    if (cudaEventRecord(p->comp_done[slot], cs) != cudaSuccess) return FA_ERR_CUDA;
    for (int cc = 0; cc < fa::kCopyStreams; ++cc)
      if (cudaStreamWaitEvent(p->d2h[cc], p->comp_done[slot], 0) != cudaSuccess)
        return FA_ERR_CUDA;
    // outputs of chunk c
    for (int i = 0; i < 4; ++i)
      if (cudaMemcpyAsync(static_cast<char*>(out_h[i]) + (size_t)h0 * row_bytes,
                          t[4 + i], bytes, cudaMemcpyDeviceToHost,
                          p->d2h[i % fa::kCopyStreams]) != cudaSuccess)
        return FA_ERR_CUDA;
    if (cudaMemcpyAsync(lse + (size_t)h0 * N, lse_d, (size_t)hc * N * 4,
                        cudaMemcpyDeviceToHost, p->d2h[0]) != cudaSuccess)
      return FA_ERR_CUDA;
    for (int cc = 0; cc < fa::kCopyStreams; ++cc)
      if (cudaEventRecord(p->out_done[slot][cc], p->d2h[cc]) != cudaSuccess)
        return FA_ERR_CUDA;
  }
  // Later work on the caller's stream sees every output on the host.
  for (int c = 0; c < fa::kCopyStreams; ++c)
    if (cudaEventRecord(p->end[c], p->d2h[c]) != cudaSuccess ||
        cudaStreamWaitEvent(cs, p->end[c], 0) != cudaSuccess)
      return FA_ERR_CUDA;
  return FA_OK;
}

namespace fa {

// One thread waits, with the configured limit, on a barrier whose single
// expected arrival never happens; the wait expires and records the timeout.
__global__ void expire_wait_kernel(DevState* st, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t cta_abort;
  if (threadIdx.x == 0) {
    cta_abort = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl wc{st, &cta_abort, timeout_ns};
    (void)wait_bar(&bar, 0, wc, 0x7E57u);
  }
}

cudaError_t launch_expire_wait(DevState* st, uint64_t timeout_ns,
                               cudaStream_t stream) {
  expire_wait_kernel<<<1, 32, 0, stream>>>(st, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fa
