"""A bounded wait that runs out: the status bit, the cleared workspace, and a
correct next call on the same workspace.

The library's kernels never trap: every wait on a value another warp publishes
gives up after a bounded number of polls, sets SPEC_DEV_TIMEOUT, and the call's
last CTA then clears the whole workspace.  To make a wait run out without
faulting or hanging anything, these tests build a separate copy of the
library with SPEC_TEST_HOOKS (an extra entry point, spec_test_set_withhold,
that makes the kernel skip publishing one unit's first partial -- a value that
nothing else will ever set) and a short spin limit, so the finisher that waits
for it gives up after about a millisecond.  The product library has neither.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from sampling_online_softmax_gb300 import build as sv_build
from workloads import make_linear

pytestmark = pytest.mark.gpu

HOOKS_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libspecverify_hooks.so")
DEV_TIMEOUT = 4
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def hooks():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    os.makedirs(os.path.dirname(HOOKS_LIB), exist_ok=True)
    sv_build.build(out=HOOKS_LIB, extra_flags=["-DSPEC_TEST_HOOKS", "-DSPEC_SPIN_LIMIT=16384"])
    lib = ctypes.CDLL(HOOKS_LIB)
    i32, u64 = ctypes.c_int, ctypes.c_size_t
    lib.spec_verify_linear.argtypes = [P, P, i32, i32, i32, i32, P, P, P, ctypes.c_float, P, P, P, P, P, P, u64, P]
    lib.spec_verify_linear.restype = i32
    lib.spec_workspace_bytes_linear.argtypes = [i32, i32, i32, i32]
    lib.spec_workspace_bytes_linear.restype = u64
    lib.spec_test_set_withhold.argtypes = [i32]
    lib.spec_test_set_withhold.restype = None
    lib.spec_last_error.restype = ctypes.c_char_p
    yield lib
    lib.spec_test_set_withhold(-1)


def to_oracle(t):
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _call(lib, d, T, ws, B, K, V):
    out = dict(accept_len=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
               out_tokens=torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda"),
               num_emitted=torch.full((B,), -7, dtype=torch.int32, device="cuda"),
               probs=torch.zeros((B, K, 3), dtype=torch.float32, device="cuda"),
               status=torch.zeros(1, dtype=torch.int32, device="cuda"))
    dt = 0 if d["target"].dtype == torch.float32 else 1
    draft = d["draft"] if T > 0 else None
    ptr = lambda t: None if t is None else P(t.data_ptr())  # noqa: E731
    st = lib.spec_verify_linear(ptr(d["target"]), ptr(draft), dt, B, K, V, ptr(d["draft_tokens"]),
                                ptr(d["u_accept"]), ptr(d["u_bonus"]), ctypes.c_float(T), ptr(out["accept_len"]),
                                ptr(out["out_tokens"]), ptr(out["num_emitted"]), ptr(out["probs"] if T > 0 else None),
                                ptr(out["status"]), ptr(ws), ws.numel(), P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.spec_last_error()
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("T,dtype_number", [(0.8, 2), (0.0, 2), (1.0, 1)])
def test_wait_that_runs_out_reports_clears_and_recovers(hooks, T, dtype_number):
    B, K, V = 6, 3, 5003
    d = make_linear(dtype_number, T, device="cuda", B=B, K=K, V=V, seed=77)
    ws = torch.zeros(hooks.spec_workspace_bytes_linear(B, K, V, 0 if dtype_number == 1 else 1) + 4096,
                     dtype=torch.uint8, device="cuda")
    # 1: unit (b=1, position 1) never publishes its first partial; its finisher's wait runs out
    hooks.spec_test_set_withhold(1 * (K + 1) + 1)
    g = _call(hooks, d, T, ws, B, K, V)
    hooks.spec_test_set_withhold(-1)
    assert int(g["status"][0]) & DEV_TIMEOUT, "the withheld partial should have timed out"
    assert int(ws.count_nonzero()) == 0, "a timed-out call must leave the workspace zeroed"
    # 2: the next call on the same workspace is exact again
    g = _call(hooks, d, T, ws, B, K, V)
    assert int(g["status"][0]) == 0
    assert int(ws.count_nonzero()) == 0
    o = oracle.verify_linear(to_oracle(d["target"]), to_oracle(d["draft"]) if T > 0 else None,
                             to_oracle(d["draft_tokens"]), to_oracle(d["u_accept"]), to_oracle(d["u_bonus"]), T)
    if T == 0:
        g.pop("probs")
    rep = compare.compare_linear(g, o, to_oracle(d["u_accept"]), to_oracle(d["u_bonus"]), T)
    assert rep.ok, rep.failures[:5]
