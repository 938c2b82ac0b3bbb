"""spec_verify_linear_static: the linear verify on the library's built-in
workspace, compared with spec_verify_linear on the same inputs.

The file name sorts last so that these tests also run after every other test
in one session (the built-in workspace then holds whatever earlier calls left
on the device); each test passes on its own as well.
"""
import ctypes

import pytest
import torch

import sampling_online_softmax_gb300 as sv
from sampling_online_softmax_gb300 import build as sv_build
from workloads import make_linear

PROB_ATOL = 1e-5
FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: the host checks fail first


@pytest.fixture(scope="module")
def lib():
    sv_build.build()
    return sv.load_library()


def _static(lib, B, K, V, dtype=1, T=1.0, ub=FAKE, ws_probs=None):
    return lib.spec_verify_linear_static(FAKE, FAKE, dtype, B, K, V, FAKE, FAKE, ub, T, FAKE, FAKE, FAKE, ws_probs,
                                         FAKE, None)


def test_static_limit_is_declared_and_checked_on_the_host(lib):
    limit = 16 << 20
    assert sv.spec_workspace_bytes_linear(64, 4, 128256, sv.SPEC_BF16) <= limit
    big = sv.spec_workspace_bytes_linear(4096, 8, 256000, sv.SPEC_BF16)
    assert big > limit
    assert _static(lib, 4096, 8, 256000) == sv.SPEC_ERR_WORKSPACE
    msg = lib.spec_last_error().decode()
    assert str(big) in msg and str(limit) in msg
    # argument errors come before the size check; an empty batch is a no-op
    assert _static(lib, 2, 3, 100, dtype=7) == sv.SPEC_ERR_INVALID_ARG
    assert _static(lib, 2, 3, 100, T=float("nan")) == sv.SPEC_ERR_INVALID_ARG
    assert _static(lib, 0, 3, 100) == sv.SPEC_OK


def _outputs(B, K, dev, probs):
    out = dict(accept_len=torch.full((B,), -7, dtype=torch.int32, device=dev),
               out_tokens=torch.full((B, K + 1), -7, dtype=torch.int32, device=dev),
               num_emitted=torch.full((B,), -7, dtype=torch.int32, device=dev))
    if probs:
        out["probs"] = torch.full((B, K, 3), -7.0, dtype=torch.float32, device=dev)
    return out, torch.zeros(1, dtype=torch.int32, device=dev)


def _host(r):
    return {k: v.cpu() for k, v in r.items()}


def _same(a, b):
    for k in ("accept_len", "out_tokens", "num_emitted", "status"):
        assert torch.equal(a[k], b[k]), k
    if "probs" in a:
        assert torch.allclose(a["probs"], b["probs"], rtol=0.0, atol=PROB_ATOL)


@pytest.mark.gpu
@pytest.mark.parametrize("number,T,shape", [
    (2, 0.7, None),                # draft/target pair at full size: B=64, K=4, V=128256, bf16
    (1, 0.0, None),                # greedy
    (1, 1.0, (5, 3, 5003)),        # ragged vocabulary, rows not 16-byte aligned
])
def test_static_matches_workspace_entry_point_twice_in_a_row(number, T, shape):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    kw = {} if shape is None else dict(B=shape[0], K=shape[1], V=shape[2])
    d = make_linear(number, T, device="cuda", **kw)
    draft = d["draft"] if T > 0 else None
    ref = sv.spec_verify_linear(d["target"], draft, d["draft_tokens"], d["u_accept"], d["u_bonus"], T,
                                probs=T > 0)
    torch.cuda.synchronize()
    ref = _host(ref)
    B, K = d["draft_tokens"].shape
    outs = [_outputs(B, K, "cuda", T > 0) for _ in range(2)]
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    for out, status in outs:  # two calls in a row on one stream, no sync between them
        sv.spec_verify_linear_static(d["target"], draft, d["draft_tokens"], d["u_accept"], d["u_bonus"], T,
                                     out=out, status=status)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before
    for out, status in outs:
        got = _host(out)
        assert int(got["status"][0]) == 0
        _same(got, ref)


@pytest.mark.gpu
def test_static_after_a_larger_shape_and_on_a_side_stream():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    big = make_linear(1, 1.0, device="cuda", B=40, K=6, V=32000)
    small = make_linear(1, 1.0, device="cuda", B=3, K=2, V=777)
    s = torch.cuda.Stream()
    results = []
    for d in (big, small, big):
        B, K = d["draft_tokens"].shape
        out, status = _outputs(B, K, "cuda", True)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            sv.spec_verify_linear_static(d["target"], d["draft"], d["draft_tokens"], d["u_accept"], d["u_bonus"],
                                         1.0, out=out, status=status, stream=s)
        results.append((d, out))
    torch.cuda.synchronize()
    for d, out in results:
        ref = sv.spec_verify_linear(d["target"], d["draft"], d["draft_tokens"], d["u_accept"], d["u_bonus"], 1.0,
                                    probs=True)
        torch.cuda.synchronize()
        _same(_host(out), _host(ref))
