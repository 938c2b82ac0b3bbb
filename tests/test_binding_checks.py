"""The Python binding's argument checks, on the CPU.

Every binding checks dtypes and shapes before it hands pointers to the
library, so that a short tensor raises instead of being read past its end on
the device.  Here the CUDA-tensor check, the stream and the library are
replaced by stand-ins, so the checks run without a GPU: valid calls must
reach the library, and every mismatched shape must raise ValueError.
"""
import contextlib
import ctypes

import pytest
import torch

import sampling_online_softmax_gb300 as sv


@pytest.fixture
def fake(monkeypatch):
    calls = []

    class FakeLib:
        def __getattr__(self, name):
            def f(*args):
                calls.append(name)
                return 64 if name.startswith("spec_workspace_bytes") else 0
            return f

    lib = FakeLib()
    monkeypatch.setattr(sv, "load_library", lambda: lib)

    def cpu_cuda(t, name, dtype=None):
        if t is not None and dtype is not None and t.dtype != dtype:
            raise TypeError(name)
        return t

    monkeypatch.setattr(sv, "_cuda", cpu_cuda)
    monkeypatch.setattr(sv, "_stream_handle", lambda dev, stream: (ctypes.c_void_p(0), None))
    monkeypatch.setattr(sv, "_workspace", lambda dev, s, n: torch.zeros(max(n, 256), dtype=torch.uint8))
    monkeypatch.setattr(torch.cuda, "device", lambda d: contextlib.nullcontext())
    monkeypatch.setattr(torch.cuda, "stream", lambda s: contextlib.nullcontext())
    return calls


B, K, V, N = 3, 2, 50, 6
i32 = torch.int32


def test_linear(fake):
    t, d = torch.zeros((B, K + 1, V)), torch.zeros((B, K, V))
    tok, ua, ub = torch.zeros((B, K), dtype=i32), torch.zeros((B, K)), torch.zeros(B)
    sv.spec_verify_linear(t, d, tok, ua, ub, 1.0)
    assert "spec_verify_linear" in fake
    for kw in (dict(draft=torch.zeros((B, K + 1, V))), dict(tok=torch.zeros((B, K + 1), dtype=i32)),
               dict(ua=torch.zeros((B, K + 1))), dict(ub=torch.zeros(B + 1))):
        with pytest.raises(ValueError):
            sv.spec_verify_linear(t, kw.get("draft", d), kw.get("tok", tok), kw.get("ua", ua), kw.get("ub", ub), 1.0)


def test_extra_token_alone(fake):
    t, d, ub = torch.zeros((B, K + 1, V)), torch.zeros((B, K, V)), torch.zeros(B)
    sv.spec_sample_bonus(t, d, torch.zeros(B, dtype=i32), ub, 1.0)
    assert "spec_sample_bonus" in fake
    with pytest.raises(ValueError):
        sv.spec_sample_bonus(t, d, torch.zeros(B + 1, dtype=i32), ub, 1.0)
    with pytest.raises(ValueError):
        sv.spec_sample_bonus(t, d, torch.zeros(B, dtype=i32), torch.zeros(B - 1), 1.0)


def test_trees(fake):
    t, par, nt, u = torch.zeros((B, N, V)), torch.zeros(N, dtype=i32), torch.zeros((B, N), dtype=i32), torch.zeros((B, N))
    sv.spec_verify_tree(t, par, nt, 3)
    sv.spec_verify_tree_sample(t, par, nt, u, 1.0, 3)
    assert "spec_verify_tree" in fake and "spec_verify_tree_sample" in fake
    with pytest.raises(ValueError):
        sv.spec_verify_tree(t, torch.zeros(N + 1, dtype=i32), nt, 3)
    for p2, n2, u2 in ((par, torch.zeros((B, N + 1), dtype=i32), u), (par, nt, torch.zeros((B, N - 1)))):
        with pytest.raises(ValueError):
            sv.spec_verify_tree_sample(t, p2, n2, u2, 1.0, 3)


def test_rows_and_mask(fake):
    x = torch.zeros((B, V))
    sv.spec_sample_rows(x, torch.zeros(B), 1.0)
    sv.spec_sample_rows(x, None, 0.0)
    sv.spec_tree_mask(torch.zeros(N, dtype=i32))
    assert "spec_sample_rows" in fake and "spec_tree_mask" in fake
    with pytest.raises(ValueError):
        sv.spec_sample_rows(x, torch.zeros(B + 2), 1.0)
    with pytest.raises(TypeError):
        sv.spec_sample_rows(x, torch.zeros(B, dtype=torch.float64), 1.0)
