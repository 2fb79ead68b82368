"""Python binding of libfa.so (argument marshalling only).

Every function here checks tensor shapes/dtypes/devices, then passes raw
device pointers and the current CUDA stream to the C ABI of ``include/fa.h``.
All arithmetic runs in the library's CUDA kernels; there is no fallback.  If
the library has not been built, loading it raises immediately.

Names mirror the C ABI: ``fa_fwd``, ``fa_bwd``, ``fa_bwd_workspace_size``,
``fa_check_device_status``, ``fa_set_wait_timeout_ns``,
``fa_debug_expire_wait``, ``fa_debug_expire_at``, ``fa_last_failure_site``,
``fa_bwd_set_phase_events``, ``fa_status_string``.
"""
import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libfa.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fa.h")

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED",
                3: "FA_ERR_CUDA", 4: "FA_ERR_DEVICE_TIMEOUT",
                5: "FA_ERR_WORKSPACE"}

_lib = None


class FAError(RuntimeError):
    """A non-OK status from libfa.so."""

    def __init__(self, where, status):
        self.status = int(status)
        super().__init__("%s failed: %s (%d)" % (
            where, STATUS_NAMES.get(self.status, "FA_ERR_UNKNOWN"),
            self.status))


def load_library():
    """Load the in-tree libfa.so (once).  Raises if it is missing: there is
    no other compute path."""
    global _lib
    if _lib is None:
        _lib = open_library(LIB_PATH)
    return _lib


def open_library(path: str):
    """Open a libfa.so at `path` and declare its C signatures."""
    if not os.path.exists(path):
        raise RuntimeError(
            "libfa.so not found at %s; build it with "
            "`python -m tiled_attention_bwd_gb300.build`" % path)
    lib = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.fa_fwd.restype = i
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                           ctypes.c_size_t, i, i, i, i, i, f, vp]
    lib.fa_bwd.restype = i
    lib.fa_fwd_ext.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.fa_fwd_ext.restype = i
    lib.fa_bwd_ext.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                               ctypes.c_size_t, i, i, i, i, i, i, i, f, vp]
    lib.fa_bwd_ext.restype = i
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                  i, f, vp]
    lib.fa_fwd_varlen.restype = i
    lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                  ctypes.c_size_t, i, i, i, i, i, i, i, f, vp]
    lib.fa_bwd_varlen.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                               i, i, i, i, i, f, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_fwd_fp8_workspace_size.argtypes = [i, i, i, i]
    lib.fa_fwd_fp8_workspace_size.restype = ctypes.c_size_t
    lib.fa_quantize_e4m3.argtypes = [vp, vp, vp, i, i, i, vp]
    lib.fa_quantize_e4m3.restype = i
    lib.fa_step_host_scratch_size.argtypes = [i, i, i, i, i]
    lib.fa_step_host_scratch_size.restype = ctypes.c_size_t
    lib.fa_step_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                 ctypes.c_size_t, i, i, i, i, i, f, i, vp]
    lib.fa_step_host.restype = i
    lib.fa_bwd_ext_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_bwd_ext_workspace_size.restype = ctypes.c_size_t
    lib.fa_check_device_status.argtypes = [vp]
    lib.fa_check_device_status.restype = i
    lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.fa_set_wait_timeout_ns.restype = None
    lib.fa_debug_expire_wait.argtypes = [vp]
    lib.fa_debug_expire_wait.restype = i
    lib.fa_debug_expire_at.argtypes = [ctypes.c_uint32]
    lib.fa_debug_expire_at.restype = None
    lib.fa_last_failure_site.argtypes = []
    lib.fa_last_failure_site.restype = ctypes.c_uint32
    lib.fa_bwd_set_phase_events.argtypes = [vp, vp]
    lib.fa_bwd_set_phase_events.restype = None
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                   i, i, i, i, i, f, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_noalloc_max_workspace.argtypes = []
    lib.fa_bwd_noalloc_max_workspace.restype = ctypes.c_size_t
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    return lib


def header_functions(path: str = HEADER_PATH):
    """Names of the functions declared in include/fa.h."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def _check(where, status):
    if status != FA_OK:
        raise FAError(where, status)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream_handle(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_qkv(name, t, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4:
        raise ValueError("%s must be a 4-D bf16 CUDA tensor [B,H,N,d]" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (
            name, tuple(t.shape), tuple(shape)))


def _check_lse(lse, B, H, N):
    if not isinstance(lse, torch.Tensor) or lse.dtype != torch.float32 \
            or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B,H,N]")


def _lse_buffer(lse, B, H, N, device):
    """A forward's LSE output: the caller's tensor (checked) or a new one."""
    if lse is None:
        return torch.empty((B, H, N), dtype=torch.float32, device=device)
    _check_lse(lse, B, H, N)
    return lse


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_set_wait_timeout_ns(ns: int) -> None:
    load_library().fa_set_wait_timeout_ns(int(ns))


def fa_check_device_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the status code."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    return int(load_library().fa_check_device_status(_stream_handle(dev)))


def fa_debug_expire_at(site: int) -> None:
    """Make every pipeline wait at `site` (a where-code, see include/fa.h) in
    later launches behave as if its time limit had passed; 0 turns it off."""
    load_library().fa_debug_expire_at(int(site))


def fa_last_failure_site() -> int:
    """Where-code of the failure the last fa_check_device_status call on this
    thread reported (0: none)."""
    return int(load_library().fa_last_failure_site())


def fa_debug_expire_wait(device=None) -> None:
    dev = torch.device("cuda") if device is None else torch.device(device)
    _check("fa_debug_expire_wait",
           load_library().fa_debug_expire_wait(_stream_handle(dev)))


def fa_bwd_set_phase_events(before_main=None, after_main=None) -> None:
    """Have later fa_bwd calls record these torch.cuda.Event objects around
    their main kernel (None, None turns it off)."""
    def handle(ev):
        if ev is None:
            return None
        return ctypes.c_void_p(ev.cuda_event)
    load_library().fa_bwd_set_phase_events(handle(before_main),
                                           handle(after_main))


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa_bwd_workspace_size(B, H, N, d))


def fa_fwd(q, k, v, causal: bool, scale: float, out=None, lse=None):
    """Forward pass.  Returns (O bf16 [B,H,N,d], LSE fp32 [B,H,N])."""
    lib = load_library()
    _check_qkv("q", q)
    _check_qkv("k", k, q.shape)
    _check_qkv("v", v, q.shape)
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check_qkv("out", out, q.shape)
    lse = _lse_buffer(lse, B, H, N, q.device)
    with torch.cuda.device(q.device):
        _check("fa_fwd", lib.fa_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
            int(bool(causal)), float(scale), _stream_handle(q.device)))
    return out, lse


def fa_bwd(q, k, v, o, lse, dout, causal: bool, scale: float, dq=None,
           dk=None, dv=None, workspace=None):
    """Backward pass.  Returns (dQ, dK, dV), bf16 [B,H,N,d] each."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_qkv(name, t, q.shape)
    B, H, N, d = q.shape
    _check_lse(lse, B, H, N)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, q.shape)
    need = fa_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8,
                                device=q.device)
    with torch.cuda.device(q.device):
        _check("fa_bwd", lib.fa_bwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
            workspace.numel() * workspace.element_size(), B, H, N, d,
            int(bool(causal)), float(scale), _stream_handle(q.device)))
    return dq, dk, dv


def fa_bwd_ext_workspace_size(B: int, H: int, Hkv: int, N: int,
                              d: int) -> int:
    return int(load_library().fa_bwd_ext_workspace_size(B, H, Hkv, N, d))


def _check_ext_shapes(q, k):
    """[B,H,N,d] queries, [B,Hkv,N,d] keys/values with Hkv dividing H
    (shapes only; dtype, device and layout are checked by _check_qkv)."""
    for name, t in (("q", q), ("k", k)):
        if not isinstance(t, torch.Tensor) or t.dim() != 4:
            raise ValueError("%s must be a 4-D tensor" % name)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, N, d) or Hkv < 1 or H % Hkv != 0:
        raise ValueError("k has shape %s; expected [B,Hkv,N,d] = [%d,Hkv,%d,%d]"
                         " with Hkv dividing H = %d" % (tuple(k.shape), B, N,
                                                        d, H))
    return B, H, Hkv, N, d


def _ext_forward_buffers(q, k, v, out, lse):
    """Checks of the grouped-head forward's tensors; returns the sizes and
    the output buffers (allocated when not given)."""
    B, H, Hkv, N, d = _check_ext_shapes(q, k)
    _check_qkv("q", q)
    _check_qkv("k", k, (B, Hkv, N, d))
    _check_qkv("v", v, (B, Hkv, N, d))
    if out is None:
        out = torch.empty_like(q)
    _check_qkv("out", out, q.shape)
    return (B, H, Hkv, N, d), out, _lse_buffer(lse, B, H, N, q.device)


def _ext_backward_buffers(q, k, v, o, lse, dout, dq, dk, dv, workspace):
    """Checks of the grouped-head backward's tensors; returns the sizes, the
    gradient buffers and the workspace (allocated when not given)."""
    B, H, Hkv, N, d = _check_ext_shapes(q, k)
    _check_qkv("q", q)
    for name, t in (("k", k), ("v", v)):
        _check_qkv(name, t, (B, Hkv, N, d))
    for name, t in (("o", o), ("dout", dout)):
        _check_qkv(name, t, q.shape)
    _check_lse(lse, B, H, N)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_qkv("dq", dq, q.shape)
    for name, t in (("dk", dk), ("dv", dv)):
        _check_qkv(name, t, (B, Hkv, N, d))
    if workspace is None:
        need = fa_bwd_ext_workspace_size(B, H, Hkv, N, d)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8,
                                device=q.device)
    return (B, H, Hkv, N, d), (dq, dk, dv), workspace


def fa_fwd_ext(q, k, v, causal: bool, scale: float, window: int = -1,
               out=None, lse=None):
    """Forward pass with Hkv = k.shape[1] key/value heads shared by the
    query heads (grouped / multi-query attention) and an optional sliding
    window (|i - j| <= window; < 0: none).  Returns (O, LSE)."""
    lib = load_library()
    dims, out, lse = _ext_forward_buffers(q, k, v, out, lse)
    with torch.cuda.device(q.device):
        _check("fa_fwd_ext", lib.fa_fwd_ext(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), *dims,
            int(bool(causal)), int(window), float(scale),
            _stream_handle(q.device)))
    return out, lse


def fa_bwd_ext(q, k, v, o, lse, dout, causal: bool, scale: float,
               window: int = -1, dq=None, dk=None, dv=None, workspace=None):
    """Backward of fa_fwd_ext.  Returns (dQ [B,H,N,d], dK, dV [B,Hkv,N,d]);
    dK and dV are summed over the query heads sharing each K/V head."""
    lib = load_library()
    dims, (dq, dk, dv), workspace = _ext_backward_buffers(
        q, k, v, o, lse, dout, dq, dk, dv, workspace)
    with torch.cuda.device(q.device):
        _check("fa_bwd_ext", lib.fa_bwd_ext(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
            workspace.numel() * workspace.element_size(), *dims,
            int(bool(causal)), int(window), float(scale),
            _stream_handle(q.device)))
    return dq, dk, dv


def _check_seq_lens(seq_lens, B, device):
    if not isinstance(seq_lens, torch.Tensor) or seq_lens.dtype != torch.int32 \
            or tuple(seq_lens.shape) != (B,) or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be a contiguous int32 tensor [B] = [%d]"
                         % B)
    if seq_lens.device != device:
        raise ValueError("seq_lens is on %s, the inputs on %s"
                         % (seq_lens.device, device))


def fa_fwd_varlen(q, k, v, seq_lens, causal: bool, scale: float,
                  window: int = -1, out=None, lse=None):
    """fa_fwd_ext over a padded batch: batch entry b attends over its first
    seq_lens[b] rows only (int32 [B] on the inputs' device, clamped to
    [0, N]).  Rows past a sequence's end of the returned O and LSE are left
    as they were (unwritten).  Returns (O, LSE)."""
    lib = load_library()
    dims, out, lse = _ext_forward_buffers(q, k, v, out, lse)
    _check_seq_lens(seq_lens, dims[0], q.device)
    with torch.cuda.device(q.device):
        _check("fa_fwd_varlen", lib.fa_fwd_varlen(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(seq_lens),
            *dims, int(bool(causal)), int(window), float(scale),
            _stream_handle(q.device)))
    return out, lse


def fa_bwd_varlen(q, k, v, o, lse, dout, seq_lens, causal: bool,
                  scale: float, window: int = -1, dq=None, dk=None, dv=None,
                  workspace=None):
    """Backward of fa_fwd_varlen.  Returns (dQ [B,H,N,d], dK, dV [B,Hkv,N,d])
    with every row past its sequence's end set to zero."""
    lib = load_library()
    dims, (dq, dk, dv), workspace = _ext_backward_buffers(
        q, k, v, o, lse, dout, dq, dk, dv, workspace)
    _check_seq_lens(seq_lens, dims[0], q.device)
    with torch.cuda.device(q.device):
        _check("fa_bwd_varlen", lib.fa_bwd_varlen(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(seq_lens), _ptr(workspace),
            workspace.numel() * workspace.element_size(), *dims,
            int(bool(causal)), int(window), float(scale),
            _stream_handle(q.device)))
    return dq, dk, dv


def fa_fwd_fp8_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa_fwd_fp8_workspace_size(B, H, N, d))


def fa_fwd_fp8(q, k, v, causal: bool, scale: float, out=None, lse=None,
               workspace=None):
    """FP8 forward: Q and K quantised to E4M3 per 16-row block, Q K^T on
    the FP8 tensor cores.  Returns (O bf16 [B,H,N,d], LSE fp32 [B,H,N])."""
    lib = load_library()
    _check_qkv("q", q)
    _check_qkv("k", k, q.shape)
    _check_qkv("v", v, q.shape)
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check_qkv("out", out, q.shape)
    lse = _lse_buffer(lse, B, H, N, q.device)
    if workspace is None:
        need = fa_fwd_fp8_workspace_size(B, H, N, d)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8,
                                device=q.device)
    with torch.cuda.device(q.device):
        _check("fa_fwd_fp8", lib.fa_fwd_fp8(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace),
            workspace.numel() * workspace.element_size(), B, H, N, d,
            int(bool(causal)), float(scale), _stream_handle(q.device)))
    return out, lse


def fa_quantize_e4m3(x):
    """E4M3 codes (uint8, same shape) and per-16-row-block scales (fp32
    [..., 8 * ceil(N / 128)]) of a bf16 [..., N, d] CUDA tensor."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 \
            or not x.is_cuda or x.dim() < 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 CUDA tensor [..., N, d]")
    *lead, N, d = x.shape
    BH = 1
    for n in lead:
        BH *= n
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty((*lead, 8 * ((N + 127) // 128)), dtype=torch.float32,
                         device=x.device)
    with torch.cuda.device(x.device):
        _check("fa_quantize_e4m3", lib.fa_quantize_e4m3(
            _ptr(x), _ptr(codes), _ptr(scales), BH, N, d,
            _stream_handle(x.device)))
    return codes, scales


def fa_step_host_scratch_size(B: int, H: int, N: int, d: int,
                              chunk_heads: int = 0) -> int:
    return int(load_library().fa_step_host_scratch_size(B, H, N, d,
                                                        chunk_heads))


def fa_step_host(q, k, v, dout, causal: bool, scale: float, o, lse, dq, dk,
                 dv, scratch=None, chunk_heads: int = 0, device=None):
    """Forward + backward on HOST tensors (bf16 [B,H,N,d]; lse fp32
    [B,H,N]; pinned memory for overlap), pipelined by chunks of heads on
    `device`.  Outputs are written into o, lse, dq, dk, dv; the call is
    asynchronous on the device's current stream."""
    lib = load_library()
    dev = torch.device("cuda") if device is None else torch.device(device)
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout), ("o", o),
                    ("dq", dq), ("dk", dk), ("dv", dv)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or \
                t.dtype != torch.bfloat16 or t.dim() != 4 or \
                not t.is_contiguous() or tuple(t.shape) != tuple(q.shape):
            raise ValueError("%s must be a contiguous bf16 host tensor of "
                             "q's shape" % name)
    B, H, N, d = q.shape
    if lse.is_cuda or lse.dtype != torch.float32 or \
            tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 host tensor [B,H,N]")
    if scratch is None:
        need = fa_step_host_scratch_size(B, H, N, d, chunk_heads)
        scratch = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check("fa_step_host", lib.fa_step_host(
            _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(o), _ptr(lse),
            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(scratch),
            scratch.numel() * scratch.element_size(), B, H, N, d,
            int(bool(causal)), float(scale), int(chunk_heads),
            _stream_handle(dev)))
    return o, lse, dq, dk, dv


def fa_bwd_noalloc_max_workspace() -> int:
    return int(load_library().fa_bwd_noalloc_max_workspace())


def fa_bwd_noalloc(q, k, v, o, lse, dout, causal: bool, scale: float, dq,
                   dk, dv):
    """Backward pass through the entry point that allocates nothing: the
    caller passes preallocated dq, dk, dv and the library uses its fixed
    device scratch array instead of a workspace."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout),
                    ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, q.shape)
    B, H, N, d = q.shape
    _check_lse(lse, B, H, N)
    with torch.cuda.device(q.device):
        _check("fa_bwd_noalloc", lib.fa_bwd_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
            _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)),
            float(scale), _stream_handle(q.device)))
    return dq, dk, dv
