"""The Python binding's argument checks, on the CPU.

Every binding checks dtypes and shapes before it hands pointers to the
library, so that a short tensor raises instead of being read past its end on
the device.  Here the CUDA-tensor check, the stream and the library are
replaced by stand-ins, so the checks run without a GPU: valid calls must
reach the library, and every mismatched shape must raise ValueError.  Outputs the
caller passes in (`out=`, `status=`, `workspace=`) are checked the same way:
a short output would be written past its end on the device.
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

    def cpu_cuda(t, name, dtype=None, device=None):
        if t is None:
            return None
        if device is not None and t.device != device:
            raise ValueError(name)
        if dtype is not None and t.dtype != dtype:
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


def _linear_args():
    return (torch.zeros((B, K + 1, V)), torch.zeros((B, K, V)), torch.zeros((B, K), dtype=i32),
            torch.zeros((B, K)), torch.zeros(B))


def _linear_out(**over):
    out = dict(accept_len=torch.zeros(B, dtype=i32), out_tokens=torch.zeros((B, K + 1), dtype=i32),
               num_emitted=torch.zeros(B, dtype=i32))
    out.update(over)
    return out


def test_linear_outputs_passed_in_are_checked(fake):
    args = _linear_args()
    st = torch.zeros(1, dtype=i32)
    sv.spec_verify_linear(*args, 1.0, out=_linear_out(), status=st)
    sv.spec_verify_linear_static(*args, 1.0, out=_linear_out(), status=st)
    assert "spec_verify_linear_static" in fake
    bad = [dict(accept_len=torch.zeros(B - 1, dtype=i32)), dict(out_tokens=torch.zeros((B, K), dtype=i32)),
           dict(num_emitted=torch.zeros(B + 1, dtype=i32)), dict(probs=torch.zeros((B, K, 2))),
           dict(out_tokens=None)]
    for over in bad:
        out = _linear_out(**over)
        if over.get("out_tokens", 0) is None:
            del out["out_tokens"]
        for f in (sv.spec_verify_linear, sv.spec_verify_linear_static):
            with pytest.raises(ValueError):
                f(*args, 1.0, out=dict(out), status=st)
    with pytest.raises(TypeError):
        sv.spec_verify_linear(*args, 1.0, out=_linear_out(accept_len=torch.zeros(B, dtype=torch.int64)), status=st)
    for f in (sv.spec_verify_linear, sv.spec_verify_linear_static):
        with pytest.raises(ValueError):
            f(*args, 1.0, out=_linear_out(), status=torch.zeros(0, dtype=i32))
    with pytest.raises(ValueError):
        sv.spec_verify_linear_static(*args, 1.0, out=_linear_out(), status=None)
    with pytest.raises(ValueError):
        sv.spec_verify_linear(*args, 1.0, workspace=torch.zeros(8, dtype=torch.uint8))


def test_inputs_and_outputs_on_another_device_are_refused(fake):
    """Every tensor must sit on the logits' device (here: a meta tensor stands for another device)."""
    t, d, tok, ua, ub = _linear_args()
    other = dict(tok=tok.to("meta"), ua=ua.to("meta"), ub=ub.to("meta"), d=d.to("meta"))
    for k in other:
        a = dict(d=d, tok=tok, ua=ua, ub=ub)
        a[k] = other[k]
        with pytest.raises(ValueError):
            sv.spec_verify_linear(t, a["d"], a["tok"], a["ua"], a["ub"], 1.0)
    with pytest.raises(ValueError):
        sv.spec_verify_linear(t, d, tok, ua, ub, 1.0, out=_linear_out(num_emitted=torch.zeros(B, dtype=i32,
                                                                                                device="meta")))


def test_other_outputs_passed_in_are_checked(fake):
    t, d, ub = torch.zeros((B, K + 1, V)), torch.zeros((B, K, V)), torch.zeros(B)
    with pytest.raises(ValueError):
        sv.spec_sample_bonus(t, d, torch.zeros(B, dtype=i32), ub, 1.0, out=torch.zeros(B - 1, dtype=i32))
    tt, par, nt = torch.zeros((B, N, V)), torch.zeros(N, dtype=i32), torch.zeros((B, N), dtype=i32)
    good = dict(path_nodes=torch.zeros((B, 4), dtype=i32), path_len=torch.zeros(B, dtype=i32),
                out_tokens=torch.zeros((B, 4), dtype=i32))
    sv.spec_verify_tree(tt, par, nt, 3, out=dict(good))
    for k, shape in (("path_nodes", (B, 3)), ("path_len", (B + 1,)), ("out_tokens", (B, 5))):
        out = dict(good)
        out[k] = torch.zeros(shape, dtype=i32)
        with pytest.raises(ValueError):
            sv.spec_verify_tree(tt, par, nt, 3, out=out)
        with pytest.raises(ValueError):
            sv.spec_verify_tree_sample(tt, par, nt, torch.zeros((B, N)), 1.0, 3, out=out)
    with pytest.raises(ValueError):
        sv.spec_sample_rows(torch.zeros((B, V)), torch.zeros(B), 1.0, out=dict(tokens=torch.zeros(B + 1, dtype=i32)))
    with pytest.raises(ValueError):
        sv.spec_tree_mask(torch.zeros(N, dtype=i32), out=dict(mask=torch.zeros((N, 2), dtype=i32),
                                                             depth=torch.zeros(N, dtype=i32)))


def test_mtp_plug(fake):
    inp, ot, ne = torch.zeros((B, K + 1), dtype=i32), torch.zeros((B, K + 1), dtype=i32), torch.zeros(B, dtype=i32)
    sv.spec_mtp_plug(inp, ot, ne, 0, torch.zeros(B, dtype=i32))
    sv.spec_mtp_plug(inp, ot, ne, 0, None, in_place=True)
    assert "spec_mtp_plug" in fake
    for a in ((inp, torch.zeros((B, K), dtype=i32), ne, None), (inp, ot, torch.zeros(B + 1, dtype=i32), None),
              (inp, ot, ne, torch.zeros(B - 1, dtype=i32))):
        with pytest.raises(ValueError):
            sv.spec_mtp_plug(*a)
    with pytest.raises(ValueError):
        sv.spec_mtp_plug(inp, ot, ne, out=torch.zeros((B, K), dtype=i32))
    with pytest.raises(TypeError):
        sv.spec_mtp_plug(inp, ot, ne.to(torch.int64))
