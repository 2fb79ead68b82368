/*
 * fa.h -- C ABI of the GB300 (sm_103a) tiled attention library, libfa.so.
 *
 * The library computes exact scaled-dot-product attention and its training
 * backward pass, tile by tile with an online softmax, so that the N x N score
 * matrix never reaches device memory:
 *
 *   forward(q, k, v, causal, scale) -> output, lse
 *   backward(dout, q, k, v, output, lse, causal, scale) -> dq, dk, dv
 *
 * which is the interface of "RTX Flash Attention Implementation COMPLETE",
 * section "Usage Examples" (basic forward pass; training with backward pass),
 * with tensors laid out as [batch, heads, seq_len, head_dim].  The operation
 * itself is O = softmax(scale * Q K^T [+ causal mask]) V with the online
 * softmax of the same page's "Online Softmax Algorithm" section (running max
 * m, running sum l); the backward recomputes P from the saved LSE, as in
 * "GPU Performance Optimization Batch 1 -- Design Spec", Item 3
 * ("FlashAttention-3 Blackwell"), backward paragraph.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors q, k, v, o, dout, dq, dk, dv are contiguous row-major bfloat16
 *    arrays of shape [B, H, N, d] in device memory (element (b,h,i,t) at
 *    ((b*H + h)*N + i)*d + t).  Their base addresses must be 16-byte aligned;
 *    where the forward stores O from registers (problems whose K and V fit
 *    in L2, without a window), a 32-byte-aligned o is written in whole
 *    32-byte sectors (faster, same values).
 *  - lse is a contiguous float32 array [B, H, N] in device memory holding the
 *    natural-log log-sum-exp of each row's scaled scores:
 *    lse[b,h,i] = ln sum_j exp(scale * q_i . k_j) over the visible keys j.
 *    4-byte alignment is enough.
 *  - causal = 1 lets query i see keys j <= i (equal query and key lengths);
 *    causal = 0 lets every query see every key.
 *  - scale multiplies Q K^T before the mask and the softmax; it must be finite
 *    and > 0 (usually 1/sqrt(d)).
 *  - Supported: d in {64, 128}; 1 <= N <= 2^30 of any size (tiles past N
 *    are masked); B, H >= 1 with B*H <= INT_MAX.  B, H or N equal to 0 is
 *    an empty problem: the call returns FA_OK and touches nothing (pointers
 *    may then be NULL).
 *  - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every compute entry point is asynchronous on that stream:
 *    FA_OK means the kernels were launched.  A failure detected on the device
 *    (a pipeline wait that ran past its time limit) is reported later by
 *    fa_check_device_status().
 *  - Memory: all tensors and the workspace belong to the caller.  The library
 *    allocates no device memory per call; it keeps one small device status
 *    record per GPU for the lifetime of the process.
 *  - Errors: invalid arguments are rejected on the host before anything is
 *    launched (FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED); a failing CUDA call
 *    returns FA_ERR_CUDA.  No entry point aborts the process.
 *  - The device must be an sm_103a (GB300-class) GPU; kernels are compiled
 *    for that target only.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size or scale */
  FA_ERR_UNSUPPORTED = 2,     /* valid but not implemented (e.g. d = 96)    */
  FA_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed          */
  FA_ERR_DEVICE_TIMEOUT = 4,  /* a kernel's bounded pipeline wait expired   */
  FA_ERR_WORKSPACE = 5        /* workspace missing or smaller than needed   */
} fa_status;

/*
 * Forward pass.
 *   q, k, v : in,  bf16 [B,H,N,d]
 *   o       : out, bf16 [B,H,N,d]   o_i = sum_j softmax_j(scale q_i.k_j) v_j
 *   lse     : out, fp32 [B,H,N]     natural-log log-sum-exp per row
 * o and lse may not alias the inputs.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o,
                 float* lse, int B, int H, int N, int d, int causal,
                 float scale, void* stream);

/*
 * Bytes of device workspace fa_bwd needs for this shape: an fp32 dQ
 * accumulator [B,H,N,d] followed by two fp32 per-row vectors
 * (D_i = dO_i . O_i and -LSE_i * log2(e)) padded to whole 128-row tiles and
 * a 256-byte counter that hands the work out to the thread blocks.
 * The accumulator is where the backward's dQ contributions of all key tiles
 * meet ("RTX Flash Attention Implementation COMPLETE", "Flash Attention
 * Backward Kernel": atomic memory operations for the gradient updates, read
 * here as additions in fp32), and D_i is the row term of the
 * recomputation from the saved LSE ("GPU Performance Optimization Batch 1 --
 * Design Spec", Item 3, backward paragraph).  The caller owns the memory, as
 * the page's usage example owns its tensors ("Usage Examples").
 * Returns 0 for an empty problem or unsupported d.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass.
 *   q, k, v   : in,  bf16 [B,H,N,d]  the forward's inputs
 *   o, lse    : in,  bf16 [B,H,N,d] / fp32 [B,H,N]  the forward's outputs
 *   dout      : in,  bf16 [B,H,N,d]  dL/dO
 *   dq, dk, dv: out, bf16 [B,H,N,d]  dL/dQ, dL/dK, dL/dV
 *   workspace : device scratch of at least fa_bwd_workspace_size() bytes,
 *               16-byte aligned, owned by the caller; its contents on entry
 *               do not matter and on return are unspecified.
 * dQ is accumulated in fp32 across key tiles, then scaled and rounded once.
 * Calls that share a workspace must not overlap in time (same stream is fine).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dout, void* dq, void* dk,
                 void* dv, void* workspace, size_t workspace_bytes, int B,
                 int H, int N, int d, int causal, float scale, void* stream);

/*
 * Grouped-query / multi-query attention and sliding-window attention, the
 * variants listed under "Advanced Features (Future)" of "RTX Flash Attention
 * Implementation COMPLETE" ("Multi-Query Attention: grouped query attention
 * variants"; "Sliding Window: local attention").  Same operation and
 * conventions as fa_fwd / fa_bwd, except:
 *   - k, v (and dk, dv) have Hkv heads: bf16 [B,Hkv,N,d].  Query head h of a
 *     batch entry reads key/value head h / (H / Hkv).  Hkv must divide H
 *     (1 <= Hkv <= H); Hkv = 1 is multi-query attention, Hkv = H the plain
 *     operation.  dk and dv are summed over the H / Hkv query heads that
 *     share each key/value head.
 *   - window >= 0 limits query i to keys j with |i - j| <= window (and
 *     j <= i when causal = 1); window < 0 means no limit.  A window of N - 1
 *     or more hides nothing.  The pages' "global tokens" are not defined
 *     there and are not part of this operation.
 *   - lse, o, dout, dq keep the query heads: [B,H,N] / [B,H,N,d].
 * fa_bwd_ext needs fa_bwd_ext_workspace_size(B, H, Hkv, N, d) bytes of
 * workspace (equal to fa_bwd_workspace_size(B, H, N, d) for Hkv = H).
 * H % Hkv != 0, Hkv < 1 or Hkv > H (for H >= 1) is FA_ERR_INVALID_ARG.
 * fa_fwd and fa_bwd are these calls with Hkv = H and window = -1.
 */
fa_status fa_fwd_ext(const void* q, const void* k, const void* v, void* o,
                     float* lse, int B, int H, int Hkv, int N, int d,
                     int causal, int window, float scale, void* stream);

/*
 * Bytes of device workspace fa_bwd_ext needs: the fa_bwd workspace plus,
 * when more than 8 query heads share a key/value head (their backward is
 * then split over several blocks), two fp32 [B,Hkv,N,d] accumulators for dK
 * and dV.  Returns 0 for an empty problem, unsupported d or invalid Hkv.
 */
size_t fa_bwd_ext_workspace_size(int B, int H, int Hkv, int N, int d);

fa_status fa_bwd_ext(const void* q, const void* k, const void* v,
                     const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, int B, int H, int Hkv, int N,
                     int d, int causal, int window, float scale,
                     void* stream);

/*
 * Per-sequence lengths over a padded batch: the "variable sequence lengths"
 * that "GPU Performance Optimization Batch 1 -- Design Spec", Item 1 ("CUDA
 * Graphs", Constraint) names as the product of dynamic padding.  Same
 * operation, arguments and workspace as fa_fwd_ext / fa_bwd_ext, plus
 *   - seq_lens: device int32 [B], 4-byte aligned, owned by the caller and
 *     read by the kernels on `stream` (it may change between calls, or
 *     between replays of a captured graph, without changing any shape).
 *     Batch entry b is the plain operation on its first L_b = seq_lens[b]
 *     rows of q, k, v, o, dout (every head of the entry): queries i < L_b
 *     see keys j < L_b only, with the causal and window rules on top.
 *     Lengths are clamped to [0, N]; L_b = 0 is an empty sequence.
 *   - Rows at or past L_b are padding.  Their q, k, v, dout must be finite
 *     (they multiply exact zeros); fa_fwd_varlen leaves o and lse there
 *     unwritten; fa_bwd_varlen sets dq, dk, dv there to zero and never reads
 *     o or lse there.
 *   - seq_lens NULL or misaligned (with B > 0): FA_ERR_INVALID_ARG.
 */
fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o,
                        float* lse, const int* seq_lens, int B, int H, int Hkv,
                        int N, int d, int causal, int window, float scale,
                        void* stream);

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* dout,
                        void* dq, void* dk, void* dv, const int* seq_lens,
                        void* workspace, size_t workspace_bytes, int B, int H,
                        int Hkv, int N, int d, int causal, int window,
                        float scale, void* stream);

/*
 * FP8 forward: the optional FP8 path of "GPU Performance Optimization Batch
 * 1 -- Design Spec", Item 3 ("FlashAttention-3 Blackwell"): before the
 * Q K^T product, Q and K are quantised to E4M3 block by block, each block
 * with its own scale, and the product runs on the FP8 tensor cores.
 *   - Blocks are 16 rows by the whole head dimension of one head:
 *     scale = amax / 448 in float32 (1 for an all-zero block), code = E4M3
 *     round-to-nearest-even of x / scale (IEEE float32 division), saturating
 *     at +-448.  A block spans the head dimension because a scale that
 *     varied along the contraction could not be applied after the product.
 *   - S = (Q8 K8^T) * sq_i * sk_j is accumulated in fp32; softmax, P (bf16)
 *     and O = P V (bf16 V) are as in fa_fwd.  Results therefore differ from
 *     fa_fwd by the quantisation of Q and K.
 *   - Same arguments as fa_fwd plus a workspace of
 *     fa_fwd_fp8_workspace_size(B, H, N, d) bytes (E4M3 copies of Q and K
 *     and their scales), 256-byte aligned, owned by the caller.
 *   - d = 64 or 128.  The E4M3 copies have rows of 128 bytes; at d = 64 the
 *     upper 64 bytes of each row are zero, so Q K^T runs as the d = 128
 *     product and P V as the d = 64 one.
 */
size_t fa_fwd_fp8_workspace_size(int B, int H, int N, int d);
fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o,
                     float* lse, void* workspace, size_t workspace_bytes,
                     int B, int H, int N, int d, int causal, float scale,
                     void* stream);

/*
 * The quantisation step of fa_fwd_fp8 on its own: x bf16 [BH, N, d]
 * (d = 64 or 128) -> codes E4M3 bytes [BH, N, d] and scales float32
 * [BH, 8 * ceil(N / 128)] (one per 16-row block; blocks that start at or
 * past N get scale 1).  x and codes 16-byte aligned; asynchronous on stream.
 */
fa_status fa_quantize_e4m3(const void* x, void* codes, float* scales, int BH,
                           int N, int d, void* stream);

/*
 * One training step of attention on tensors in HOST memory: copies q, k, v,
 * dout to the device, runs the forward and the backward, and copies o, lse,
 * dq, dk, dv back -- the same results as fa_fwd + fa_bwd on device copies.
 *   - q, k, v, dout, o, dq, dk, dv: host bf16 [B,H,N,d]; lse: host fp32
 *     [B,H,N].  Page-locked (pinned) host memory lets the copies run
 *     asynchronously and overlap; pageable memory works but serialises.
 *   - The B*H heads are processed in chunks of chunk_heads (0: about a
 *     sixteenth of them): the inputs of the next chunk are copied in and the
 *     outputs of the previous one copied out on two streams of the library
 *     while the current chunk computes on `stream`, so the copies in both
 *     directions overlap each other and the kernels.
 *   - scratch: device memory of fa_step_host_scratch_size(B, H, N, d,
 *     chunk_heads) bytes, 256-byte aligned, owned by the caller (three
 *     rotating chunk slots of tensors and workspace).
 *   - Asynchronous: the step is ordered after earlier work on `stream`, and
 *     work submitted to `stream` afterwards (including a synchronisation of
 *     it) sees every output in host memory.  Calls on one device must not
 *     overlap each other (they share the library's copy streams).
 */
size_t fa_step_host_scratch_size(int B, int H, int N, int d, int chunk_heads);
fa_status fa_step_host(const void* q, const void* k, const void* v,
                       const void* dout, void* o, float* lse, void* dq,
                       void* dk, void* dv, void* scratch, size_t scratch_bytes,
                       int B, int H, int N, int d, int causal, float scale,
                       int chunk_heads, void* stream);

/*
 * Synchronises `stream`, then reports (and clears) the device status record
 * of the current GPU: FA_ERR_DEVICE_TIMEOUT if any kernel of this library
 * gave up on a pipeline wait since the last check, FA_ERR_CUDA if the stream
 * reported an error, else FA_OK.  This is the error reporting of
 * "RTX Flash Attention Implementation COMPLETE", "Complete Rust Integration"
 * ("Error Handling: comprehensive error reporting and recovery") for work
 * that runs asynchronously: a failure inside a kernel is recorded on the
 * device and read here, after which the library is usable again.
 */
fa_status fa_check_device_status(void* stream);

/*
 * Time limit, in nanoseconds, of every pipeline wait inside the kernels
 * launched after this call (default 2e9 = 2 s).  A wait that runs past it
 * records FA_ERR_DEVICE_TIMEOUT,
 * stops its thread block cleanly (in-flight copies drained, tensor memory
 * released) and makes the other blocks of the grid stop at their next wait.
 * Values of 0 restore the default.
 */
void fa_set_wait_timeout_ns(uint64_t ns);

/*
 * Test hook of the failure path, for the current device.  Until called
 * again with 0, every pipeline wait at `site` inside the forward and
 * backward kernels launched after this call that finds its barrier not yet
 * complete (a real wait) behaves as if its time limit had passed: it
 * records FA_ERR_DEVICE_TIMEOUT with that
 * site, and its block and the rest of the grid stop exactly as after a real
 * timeout (nothing is faulted, trapped or left hanging).  A site is a
 * where-code, role * 256 + n:
 *   forward:  0x101 producer waiting for a K/V ring slot, 0x102 producer
 *             waiting for a Q buffer, 0x103 producer waiting to publish a
 *             claimed item; 0x201 MMA thread waiting for Q, 0x202 for K/V,
 *             0x203 for P, 0x204 for the next item; 0x301 softmax waiting
 *             for S, 0x302 for the finished O, 0x303 for the next item.
 *   backward: 0x111 producer waiting for a Q stage, 0x112 for the dO
 *             buffer, 0x113 for the K buffer, 0x114 for the V buffer, 0x115
 *             to publish an item; 0x211 MMA thread waiting for K/V, 0x212
 *             Q, 0x213 the dQ read-out, 0x214 P, 0x215 dS, 0x216 dO, 0x217
 *             the dK/dV read-out, 0x218 the next item; 0x311 P/dS warps
 *             waiting for Q, 0x312 S, 0x313 dP, 0x314 the dS buffer, 0x315
 *             the finished dK, 0x316 the next item; 0x411 dQ drain waiting
 *             for dQ, 0x412 the finished dV, 0x413 the next item.
 * While a site is set, forward and backward calls with d = 128 and no
 * window, lengths or FP8 run kernel instantiations compiled with the hook
 * (the same source; the ones used otherwise carry no trace of it, since
 * even a test on the slow path of each wait cost about 1%); other calls
 * ignore it.  The call is synchronous (it writes a constant in device
 * memory): make it only while no kernel of this library is running on the
 * device.
 * The pages have no counterpart; this exists so that the failure handling
 * of the real kernels can be tested without harming the GPU.
 */
void fa_debug_expire_at(uint32_t site);

/*
 * Site (where-code, as listed at fa_debug_expire_at) of the failure that the
 * last fa_check_device_status call of the calling thread reported; 0 if that
 * call reported none.
 */
uint32_t fa_last_failure_site(void);

/*
 * Launches one small kernel whose thread waits, with the configured time
 * limit, on a pipeline barrier that nothing ever signals, so that the wait
 * runs out and the failure path of every kernel (status record, clean exit)
 * can be exercised without harming the GPU.  Used by the test suite; expect
 * fa_check_device_status() to return FA_ERR_DEVICE_TIMEOUT afterwards.
 */
fa_status fa_debug_expire_wait(void* stream);

/*
 * Measurement hook.  Until called again, every fa_bwd on the calling thread
 * records the caller-owned CUDA events `before_main` and `after_main`
 * (cudaEvent_t passed as void*) on its stream immediately before and after
 * the launch of its main kernel (the one running the tensor-core work), so
 * the caller can time that kernel alone.  While the stream is being
 * captured into a CUDA graph they are recorded as external events
 * (cudaEventRecordExternal), so the graph records them each time it runs.
 * NULL, NULL turns it off.
 */
void fa_bwd_set_phase_events(void* before_main, void* after_main);

/*
 * Backward pass for callers that cannot allocate device memory.  (The pages
 * have no counterpart: this entry point exists for callers of this library.)
 *
 * Same arguments and results as fa_bwd, without the workspace: a plug-in
 * that is handed only the tensors and owns no allocator, a serving or
 * training loop that reserves all memory up front and forbids allocation on
 * its hot path, or code that must not call cudaMalloc because it synchronises
 * the device can still run the backward pass.  The scratch is a fixed
 * 64 MiB array in device memory (fa_bwd_noalloc_max_workspace()), held by
 * every GPU that loads the library until the process exits; neither the
 * caller nor the library allocates anything per call.
 *   - Shapes whose fa_bwd_workspace_size() exceeds that maximum are rejected
 *     with FA_ERR_WORKSPACE before anything is launched.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address once; make that first call before any stream
 *     capture.
 *   - Every call shares the one array, so calls whose kernels overlap on the
 *     GPU (other streams, other host threads) race on it.  Its contents
 *     from a previous call do not matter: each call rewrites what it reads.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout,
                         void* dq, void* dk, void* dv, int B, int H, int N,
                         int d, int causal, float scale, void* stream);

/* Size in bytes of the fixed scratch array used by fa_bwd_noalloc. */
size_t fa_bwd_noalloc_max_workspace(void);

/*
 * Human-readable name of a status code (static storage, never NULL), the
 * reporting half of the same page's "Error Handling" item.
 */
const char* fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
