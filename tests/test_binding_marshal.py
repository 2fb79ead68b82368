"""The Python binding passes arguments to the C ABI in the order and with
the values include/fa.h declares (CPU only: the library is replaced by a
recorder, so no kernel runs).

Checked for the grouped-head and per-sequence-length entry points: sizes
(B, H, Hkv, N, d), flags, window, scale, the pointers of the caller's
tensors, and the workspace size; and that a backward without an LSE
tensor is refused rather than given a fresh (uninitialised) one.
"""
import contextlib

import pytest
import torch

from tiled_attention_bwd_gb300 import fa


class Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if name == "fa_bwd_ext_workspace_size":
            return lambda *a: 4096
        def call(*args):
            self.calls.append((name, args))
            return 0
        return call


@pytest.fixture
def rec(monkeypatch):
    r = Recorder()
    monkeypatch.setattr(fa, "load_library", lambda: r)
    monkeypatch.setattr(fa, "_check_qkv", lambda *a, **k: None)
    monkeypatch.setattr(fa, "_stream_handle", lambda dev: "stream")
    monkeypatch.setattr(torch.cuda, "device", lambda dev: contextlib.nullcontext())
    return r


def ptr(t):
    return t.data_ptr()


def tensors(B=2, H=4, Hkv=2, N=40, d=64):
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16)
    k = torch.zeros((B, Hkv, N, d), dtype=torch.bfloat16)
    v = torch.zeros((B, Hkv, N, d), dtype=torch.bfloat16)
    return q, k, v


def values(args):
    return [a.value if hasattr(a, "value") else a for a in args]


def test_forward_calls(rec):
    q, k, v = tensors()
    lens = torch.tensor([40, 7], dtype=torch.int32)
    o, lse = fa.fa_fwd_ext(q, k, v, True, 0.25, 9)
    o2, lse2 = fa.fa_fwd_varlen(q, k, v, lens, False, 0.5, -1)
    (n1, a1), (n2, a2) = rec.calls
    assert n1 == "fa_fwd_ext" and n2 == "fa_fwd_varlen"
    assert values(a1) == [ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse),
                          2, 4, 2, 40, 64, 1, 9, 0.25, "stream"]
    assert values(a2) == [ptr(q), ptr(k), ptr(v), ptr(o2), ptr(lse2),
                          ptr(lens), 2, 4, 2, 40, 64, 0, -1, 0.5, "stream"]
    assert o.shape == q.shape and lse.shape == (2, 4, 40)
    assert lse.dtype == torch.float32


def test_backward_calls(rec):
    q, k, v = tensors()
    lens = torch.tensor([3, 40], dtype=torch.int32)
    o, do = torch.zeros_like(q), torch.zeros_like(q)
    lse = torch.zeros((2, 4, 40), dtype=torch.float32)
    g = fa.fa_bwd_ext(q, k, v, o, lse, do, False, 0.125, 5)
    g2 = fa.fa_bwd_varlen(q, k, v, o, lse, do, lens, True, 0.125)
    (n1, a1), (n2, a2) = rec.calls
    assert n1 == "fa_bwd_ext" and n2 == "fa_bwd_varlen"
    a1, a2 = values(a1), values(a2)
    assert a1[:9] == [ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(do),
                      ptr(g[0]), ptr(g[1]), ptr(g[2])]
    assert a1[10:] == [4096, 2, 4, 2, 40, 64, 0, 5, 0.125, "stream"]
    assert a2[:10] == [ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(do),
                       ptr(g2[0]), ptr(g2[1]), ptr(g2[2]), ptr(lens)]
    assert a2[11:] == [4096, 2, 4, 2, 40, 64, 1, -1, 0.125, "stream"]
    assert g[1].shape == k.shape and g[0].shape == q.shape


def test_backward_requires_an_lse(rec):
    q, k, v = tensors()
    o = torch.zeros_like(q)
    lens = torch.tensor([3, 40], dtype=torch.int32)
    with pytest.raises(ValueError):
        fa.fa_bwd_ext(q, k, v, o, None, o, True, 0.1)
    with pytest.raises(ValueError):
        fa.fa_bwd_varlen(q, k, v, o, None, o, lens, True, 0.1)
    with pytest.raises(ValueError):     # wrong LSE shape
        fa.fa_bwd_ext(q, k, v, o, torch.zeros((2, 4, 39)), o, True, 0.1)
    with pytest.raises(ValueError):     # lengths of the wrong batch size
        fa.fa_fwd_varlen(q, k, v, lens[:1], True, 0.1)
    assert rec.calls == []
