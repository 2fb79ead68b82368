"""The C-ABI library on the host (CPU only, no GPU calls).

Checks that libfa.so builds for sm_103a, loads, exports every function that
include/fa.h declares, and rejects bad arguments on the host before anything
would reach a GPU.  Every call here returns before the library's first CUDA
runtime call.
"""
import ctypes
import json
import subprocess

import pytest

from tiled_attention_bwd_gb300 import build as fa_build
from tiled_attention_bwd_gb300 import fa

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 5


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load_library()


def test_header_declares_the_expected_entry_points():
    names = fa.header_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size",
              "fa_fwd_ext", "fa_bwd_ext", "fa_bwd_ext_workspace_size",
              "fa_fwd_varlen", "fa_bwd_varlen",
              "fa_fwd_fp8", "fa_fwd_fp8_workspace_size", "fa_quantize_e4m3",
              "fa_check_device_status", "fa_status_string",
              "fa_set_wait_timeout_ns", "fa_debug_expire_wait",
              "fa_debug_expire_at", "fa_last_failure_site"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in fa.header_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_library_targets_sm103a(lib):
    # The flags the build recorded next to the library: one target,
    # sm_103a, for every object and for the link.
    with open(fa_build.FLAGS) as f:
        flags = json.load(f)
    for step in ("compile", "link"):
        args = flags[step]
        targets = [args[i + 1] for i, a in enumerate(args)
                   if a in ("-gencode", "-arch", "--gpu-architecture")]
        assert targets == ["arch=compute_103a,code=sm_103a"], (step, targets)


def test_missing_library_fails_loudly():
    with pytest.raises(RuntimeError):
        fa.open_library("/nonexistent/libfa.so")


def test_status_strings(lib):
    for code, name in fa.STATUS_NAMES.items():
        assert lib.fa_status_string(code).decode() == name
    assert lib.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"


def _fwd(lib, q=16, k=16, v=16, o=16, lse=16, B=1, H=1, N=128, d=128,
         causal=0, scale=0.125):
    p = lambda x: ctypes.c_void_p(x) if x else None
    return lib.fa_fwd(p(q), p(k), p(v), p(o), p(lse), B, H, N, d, causal,
                      scale, None)


def _bwd(lib, ptr=16, ws=16, ws_bytes=1 << 40, B=1, H=1, N=128, d=128,
         causal=0, scale=0.125, lse=16):
    p = lambda x: ctypes.c_void_p(x) if x else None
    return lib.fa_bwd(p(ptr), p(ptr), p(ptr), p(ptr), p(lse), p(ptr), p(ptr),
                      p(ptr), p(ptr), p(ws), ws_bytes, B, H, N, d, causal,
                      scale, None)


def test_forward_argument_checks(lib):
    assert _fwd(lib, d=96) == UNSUPPORTED
    assert _fwd(lib, d=256) == UNSUPPORTED
    assert _fwd(lib, d=0) == INVALID
    assert _fwd(lib, scale=0.0) == INVALID
    assert _fwd(lib, scale=-1.0) == INVALID
    assert _fwd(lib, scale=float("inf")) == INVALID
    assert _fwd(lib, scale=float("nan")) == INVALID
    assert _fwd(lib, causal=2) == INVALID
    assert _fwd(lib, B=-1) == INVALID
    assert _fwd(lib, N=(1 << 30) + 1) == UNSUPPORTED
    assert _fwd(lib, q=0) == INVALID            # null pointer
    assert _fwd(lib, lse=0) == INVALID
    assert _fwd(lib, q=24) == INVALID           # not 16-byte aligned
    assert _fwd(lib, o=8) == INVALID
    assert _fwd(lib, lse=18) == INVALID         # not 4-byte aligned


def test_empty_problems_are_no_ops(lib):
    # No element to compute: FA_OK without touching (here: null) pointers.
    assert _fwd(lib, q=0, k=0, v=0, o=0, lse=0, N=0) == OK
    assert _fwd(lib, q=0, k=0, v=0, o=0, lse=0, B=0) == OK
    assert _bwd(lib, ptr=0, ws=0, ws_bytes=0, lse=0, H=0) == OK
    assert lib.fa_bwd_workspace_size(0, 4, 128, 128) == 0


def test_backward_argument_checks(lib):
    assert _bwd(lib, d=80) == UNSUPPORTED
    assert _bwd(lib, scale=0.0) == INVALID
    assert _bwd(lib, ptr=0) == INVALID
    assert _bwd(lib, ptr=40) == INVALID
    assert _bwd(lib, ws=0) == WORKSPACE
    assert _bwd(lib, ws=8) == WORKSPACE
    need = lib.fa_bwd_workspace_size(1, 1, 128, 128)
    assert _bwd(lib, ws_bytes=need - 1) == WORKSPACE


def _align(x, a=256):
    return (x + a - 1) // a * a


@pytest.mark.parametrize("B,H,N,d", [(2, 8, 512, 64), (4, 64, 4096, 128),
                                     (1, 1, 1, 64), (3, 5, 333, 128)])
def test_workspace_size(lib, B, H, N, d):
    n_pad = _align(N, 128)
    # dQ accumulator, D and -LSE log2(e) per padded row, the work counter
    expect = (_align(B * H * N * d * 4) + 2 * _align(B * H * n_pad * 4) + 256)
    assert lib.fa_bwd_workspace_size(B, H, N, d) == expect
    assert fa.fa_bwd_workspace_size(B, H, N, d) == expect


def _fwd_ext(lib, ptr=16, lse=16, B=1, H=4, Hkv=2, N=128, d=128, causal=0,
             window=-1, scale=0.125):
    p = lambda x: ctypes.c_void_p(x) if x else None
    return lib.fa_fwd_ext(p(ptr), p(ptr), p(ptr), p(ptr), p(lse), B, H, Hkv,
                          N, d, causal, window, scale, None)


def _bwd_ext(lib, ptr=16, ws=16, ws_bytes=1 << 40, B=1, H=4, Hkv=2, N=128,
             d=128, causal=0, window=-1, scale=0.125, lse=16):
    p = lambda x: ctypes.c_void_p(x) if x else None
    return lib.fa_bwd_ext(p(ptr), p(ptr), p(ptr), p(ptr), p(lse), p(ptr),
                          p(ptr), p(ptr), p(ptr), p(ws), ws_bytes, B, H, Hkv,
                          N, d, causal, window, scale, None)


def test_grouped_head_argument_checks(lib):
    for call in (_fwd_ext, _bwd_ext):
        assert call(lib, Hkv=0) == INVALID        # no key/value head
        assert call(lib, Hkv=-1) == INVALID
        assert call(lib, H=4, Hkv=3) == INVALID   # does not divide H
        assert call(lib, H=4, Hkv=8) == INVALID   # more K/V than query heads
        assert call(lib, d=96) == UNSUPPORTED
        assert call(lib, scale=0.0) == INVALID
        assert call(lib, causal=2) == INVALID
        assert call(lib, ptr=0) == INVALID
        assert call(lib, ptr=24) == INVALID
        # Empty problems are no-ops whatever the window.
        assert call(lib, ptr=0, lse=0, N=0, window=5) == OK
        assert call(lib, ptr=0, lse=0, H=0, Hkv=0) == OK
    assert _bwd_ext(lib, ws=0) == WORKSPACE
    need = lib.fa_bwd_ext_workspace_size(1, 4, 2, 128, 128)
    assert _bwd_ext(lib, ws_bytes=need - 1) == WORKSPACE


@pytest.mark.parametrize("B,H,Hkv,N,d", [(4, 64, 64, 4096, 128),
                                         (4, 64, 8, 4096, 128),
                                         (4, 64, 1, 4096, 128),
                                         (2, 12, 1, 333, 64),
                                         (1, 16, 2, 1000, 128)])
def test_grouped_workspace_size(lib, B, H, Hkv, N, d):
    n_pad = _align(N, 128)
    base = _align(B * H * N * d * 4) + 2 * _align(B * H * n_pad * 4) + 256
    g = H // Hkv
    hpb = max(h for h in range(1, min(g, 8) + 1) if g % h == 0)
    extra = 2 * _align(B * Hkv * N * d * 4) if g // hpb > 1 else 0
    assert lib.fa_bwd_ext_workspace_size(B, H, Hkv, N, d) == base + extra
    if Hkv == H:
        assert lib.fa_bwd_workspace_size(B, H, N, d) == base
    assert lib.fa_bwd_ext_workspace_size(B, H, 3, N, d) == 0 or H % 3 == 0
    assert lib.fa_bwd_ext_workspace_size(0, H, Hkv, N, d) == 0


def test_python_binding_checks_grouped_shapes():
    import torch
    q = torch.zeros((1, 4, 8, 64), dtype=torch.bfloat16)
    k = torch.zeros((1, 3, 8, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa._check_ext_shapes(q, k)     # 3 does not divide 4
    k = torch.zeros((1, 2, 9, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa._check_ext_shapes(q, k)     # sequence lengths differ
    k = torch.zeros((1, 2, 8, 64), dtype=torch.bfloat16)
    assert fa._check_ext_shapes(q, k) == (1, 4, 2, 8, 64)


def _fwd_varlen(lib, ptr=16, lse=16, sl=16, B=2, H=4, Hkv=2, N=128, d=128,
                causal=0, window=-1, scale=0.125):
    p = lambda x: ctypes.c_void_p(x) if x else None
    return lib.fa_fwd_varlen(p(ptr), p(ptr), p(ptr), p(ptr), p(lse), p(sl), B,
                             H, Hkv, N, d, causal, window, scale, None)


def _bwd_varlen(lib, ptr=16, ws=16, ws_bytes=1 << 40, sl=16, B=2, H=4, Hkv=2,
                N=128, d=128, causal=0, window=-1, scale=0.125, lse=16):
    p = lambda x: ctypes.c_void_p(x) if x else None
    return lib.fa_bwd_varlen(p(ptr), p(ptr), p(ptr), p(ptr), p(lse), p(ptr),
                             p(ptr), p(ptr), p(ptr), p(sl), p(ws), ws_bytes, B,
                             H, Hkv, N, d, causal, window, scale, None)


def test_varlen_argument_checks(lib):
    for call in (_fwd_varlen, _bwd_varlen):
        assert call(lib, sl=0) == INVALID          # lengths are required
        assert call(lib, sl=18) == INVALID         # not 4-byte aligned
        assert call(lib, ptr=0) == INVALID
        assert call(lib, H=4, Hkv=3) == INVALID
        assert call(lib, scale=0.0) == INVALID
        assert call(lib, d=96) == UNSUPPORTED
        # Empty problems are no-ops; with B = 0 there are no lengths to read.
        assert call(lib, ptr=0, lse=0, sl=0, B=0) == OK
        assert call(lib, ptr=0, lse=0, N=0) == OK
    assert _bwd_varlen(lib, ws=0) == WORKSPACE
    need = lib.fa_bwd_ext_workspace_size(2, 4, 2, 128, 128)
    assert _bwd_varlen(lib, ws_bytes=need - 1) == WORKSPACE


def test_python_binding_checks_seq_lens():
    import torch
    good = torch.zeros(3, dtype=torch.int32)
    fa._check_seq_lens(good, 3, good.device)
    for bad in (torch.zeros(3, dtype=torch.int64),      # wrong dtype
                torch.zeros(4, dtype=torch.int32),      # wrong length
                torch.zeros((3, 1), dtype=torch.int32),
                torch.zeros(6, dtype=torch.int32)[::2],  # not contiguous
                [1, 2, 3]):                              # not a tensor
        with pytest.raises(ValueError):
            fa._check_seq_lens(bad, 3, good.device)
    with pytest.raises(ValueError):
        fa._check_seq_lens(good, 3, torch.device("meta"))


def _fwd_fp8(lib, ptr=256, lse=16, ws=256, ws_bytes=1 << 40, B=1, H=1, N=128,
             d=128, causal=0, scale=0.125):
    p = lambda x: ctypes.c_void_p(x) if x else None
    return lib.fa_fwd_fp8(p(ptr), p(ptr), p(ptr), p(ptr), p(lse), p(ws),
                          ws_bytes, B, H, N, d, causal, scale, None)


def test_fp8_forward_argument_checks(lib):
    assert _fwd_fp8(lib, d=96) == UNSUPPORTED
    assert _fwd_fp8(lib, scale=0.0) == INVALID
    assert _fwd_fp8(lib, ptr=0) == INVALID
    assert _fwd_fp8(lib, ptr=24) == INVALID
    assert _fwd_fp8(lib, ws=0) == WORKSPACE
    assert _fwd_fp8(lib, ws=16) == WORKSPACE          # not 256-byte aligned
    need = lib.fa_fwd_fp8_workspace_size(1, 1, 128, 128)
    assert _fwd_fp8(lib, ws_bytes=need - 1) == WORKSPACE
    assert _fwd_fp8(lib, ptr=0, lse=0, ws=0, ws_bytes=0, N=0) == OK
    p = lambda x: ctypes.c_void_p(x) if x else None
    assert lib.fa_quantize_e4m3(p(16), p(16), p(16), 2, 100, 96, None) == UNSUPPORTED
    assert lib.fa_quantize_e4m3(p(0), p(16), p(16), 2, 100, 128, None) == INVALID
    assert lib.fa_quantize_e4m3(p(0), p(0), p(0), 2, 0, 128, None) == OK


@pytest.mark.parametrize("B,H,N,d", [(4, 64, 4096, 128), (1, 3, 333, 128),
                                     (2, 2, 1, 128), (2, 8, 512, 64),
                                     (1, 3, 333, 64)])
def test_fp8_workspace_size(lib, B, H, N, d):
    nsb = 8 * ((N + 127) // 128)
    # E4M3 rows are 128 bytes at either d (zero-padded at d = 64)
    expect = 2 * _align(B * H * N * 128) + 2 * _align(B * H * nsb * 4)
    assert lib.fa_fwd_fp8_workspace_size(B, H, N, d) == expect
    assert lib.fa_fwd_fp8_workspace_size(B, H, N, 96) == 0


def _step_host(lib, ptr=256, scratch=256, scratch_bytes=1 << 40, B=2, H=8,
               N=512, d=128, causal=1, scale=0.125, chunk=0):
    p = lambda x: ctypes.c_void_p(x) if x else None
    return lib.fa_step_host(p(ptr), p(ptr), p(ptr), p(ptr), p(ptr), p(ptr),
                            p(ptr), p(ptr), p(ptr), p(scratch), scratch_bytes,
                            B, H, N, d, causal, scale, chunk, None)


@pytest.mark.parametrize("B,H,N,d,chunk", [(2, 8, 512, 128, 0),
                                          (2, 8, 512, 128, 5),
                                          (1, 3, 333, 64, 1),
                                          (1, 4, 256, 128, 100),
                                          (4, 64, 4096, 128, 0)])
def test_step_host_scratch_size(lib, B, H, N, d, chunk):
    # Three rotating slots; each holds eight [ch,N,d] bf16 tensors, the LSE
    # rows and the backward workspace of ch heads, each 256-byte aligned.
    BH = B * H
    ch = min(chunk, BH) if chunk > 0 else (BH + 15) // 16
    slot = (8 * _align(ch * N * d * 2) + _align(ch * N * 4)
            + _align(lib.fa_bwd_workspace_size(1, ch, N, d)))
    assert lib.fa_step_host_scratch_size(B, H, N, d, chunk) == 3 * slot
    assert lib.fa_step_host_scratch_size(0, H, N, d, chunk) == 0
    assert lib.fa_step_host_scratch_size(B, H, N, 96, chunk) == 0


def test_step_host_argument_checks(lib):
    assert _step_host(lib, chunk=-1) == INVALID
    assert _step_host(lib, ptr=0) == INVALID
    assert _step_host(lib, scale=0.0) == INVALID
    assert _step_host(lib, d=96) == UNSUPPORTED
    assert _step_host(lib, scratch=0) == WORKSPACE
    assert _step_host(lib, scratch=128) == WORKSPACE      # not 256-aligned
    need = lib.fa_step_host_scratch_size(2, 8, 512, 128, 0)
    assert _step_host(lib, scratch_bytes=need - 1) == WORKSPACE
    assert _step_host(lib, ptr=0, scratch=0, N=0) == OK   # empty problem


def test_phase_events_can_be_cleared(lib):
    # Null events turn the recording off; nothing is launched.
    lib.fa_bwd_set_phase_events(None, None)
