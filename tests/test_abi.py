"""The C ABI library builds, loads and exports every declared symbol; host-side
argument checks return their documented status without touching a GPU."""
import ctypes
import os
import re

import pytest

import sampling_online_softmax_gb300 as sv
from sampling_online_softmax_gb300 import build as sv_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    sv_build.build()
    return sv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("spec_verify_linear", "spec_sample_bonus", "spec_verify_tree", "spec_status_string",
              "spec_last_error", "spec_workspace_bytes_linear", "spec_workspace_bytes_bonus",
              "spec_workspace_bytes_tree"):
        assert n in names


def test_header_is_plain_c(tmp_path):
    """The boundary is a C ABI: the header compiles as strict C99, with every entry point taken by address."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    names = [n for n in declared_functions()]
    src = tmp_path / "abi.c"
    src.write_text('#include "spec_verify.h"\ntypedef void (*fn)(void);\nint main(void) {\n  const fn f[] = {' +
                   ", ".join("(fn)&%s" % n for n in names) + '};\n  return f[0] == 0;\n}\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.dirname(HEADER),
                        "-fsyntax-only", str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(sv.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_only_the_declared_entry_points_are_exported(lib):
    """The library is built with hidden visibility: its exported spec_* symbols are
    exactly the header's functions (no C++ internals a second copy could bind to)."""
    import shutil
    import subprocess
    if shutil.which("nm") is None:
        pytest.skip("no nm")
    r = subprocess.run(["nm", "-D", "--defined-only", sv.LIB_PATH], capture_output=True, text=True, check=True)
    exported = sorted({ln.split()[-1] for ln in r.stdout.splitlines() if ln.split()[-1].startswith("spec_")})
    assert exported == declared_functions()
    assert not [ln for ln in r.stdout.splitlines() if "_ZN4spec" in ln]


def test_status_strings(lib):
    for code in range(5):
        s = lib.spec_status_string(code).decode()
        assert s.startswith("SPEC_")
    assert "unknown" in lib.spec_status_string(99).decode()


def test_workspace_sizes(lib):
    assert sv.spec_workspace_bytes_linear(0, 4, 1000, sv.SPEC_F32) == 0
    assert sv.spec_workspace_bytes_linear(4, 4, 0, sv.SPEC_F32) == 0
    assert sv.spec_workspace_bytes_linear(4, 4, 1000, 9) == 0
    a = sv.spec_workspace_bytes_linear(64, 4, 128256, sv.SPEC_BF16)
    # counters, accept bits, values, and 8-byte partials for 16 KB slices of every row
    slices = -(-128256 * 2 // 16384)
    assert a >= 64 * 5 * 4 + 64 * 4 * 4 + 64 * 5 * 4 + 64 * 5 * 2 * slices * 8 and a % 16 == 0
    assert sv.spec_workspace_bytes_linear(128, 4, 128256, sv.SPEC_BF16) > a
    assert sv.spec_workspace_bytes_linear(64, 4, 128256, sv.SPEC_F32) > a      # twice the slices
    t = sv.spec_workspace_bytes_tree(16, 64, 32000, sv.SPEC_F32)
    assert t >= 16 * 64 * 4 * 2
    assert sv.spec_workspace_bytes_tree(16, 0, 32000, sv.SPEC_F32) == 0
    assert sv.spec_workspace_bytes_bonus(8, 1000, sv.SPEC_BF16) > 0


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every case below fails on the host


def _linear(lib, **kw):
    args = dict(target=FAKE, draft=FAKE, dtype=1, B=2, K=3, V=100, tokens=FAKE, u=FAKE, ub=FAKE, T=1.0,
                al=FAKE, ot=FAKE, ne=FAKE, probs=None, st=FAKE, ws=FAKE, wsb=1 << 20, stream=None)
    args.update(kw)
    return lib.spec_verify_linear(args["target"], args["draft"], args["dtype"], args["B"], args["K"], args["V"],
                                  args["tokens"], args["u"], args["ub"], args["T"], args["al"], args["ot"],
                                  args["ne"], args["probs"], args["st"], args["ws"], args["wsb"], args["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(dtype=7), sv.SPEC_ERR_INVALID_ARG),
    (dict(B=-1), sv.SPEC_ERR_INVALID_ARG),
    (dict(K=-1), sv.SPEC_ERR_INVALID_ARG),
    (dict(V=0), sv.SPEC_ERR_INVALID_ARG),
    (dict(T=float("nan")), sv.SPEC_ERR_INVALID_ARG),
    (dict(T=-0.5), sv.SPEC_ERR_INVALID_ARG),
    (dict(T=float("inf")), sv.SPEC_ERR_INVALID_ARG),
    (dict(T=1e-45), sv.SPEC_ERR_INVALID_ARG),          # log2(e)/T overflows float
    (dict(target=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(target=ctypes.c_void_p(0x10001)), sv.SPEC_ERR_INVALID_ARG),  # misaligned bf16
    (dict(draft=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(u=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(tokens=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(al=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(st=None), sv.SPEC_ERR_INVALID_ARG),
    (dict(ot=None), sv.SPEC_ERR_INVALID_ARG),            # required with u_bonus
    (dict(ws=None), sv.SPEC_ERR_WORKSPACE),
    (dict(wsb=16), sv.SPEC_ERR_WORKSPACE),
    (dict(ws=ctypes.c_void_p(0x10008)), sv.SPEC_ERR_WORKSPACE),
    (dict(B=0), sv.SPEC_OK),                             # empty batch: nothing to do
])
def test_linear_host_validation(lib, kw, expect):
    assert _linear(lib, **kw) == expect
    if expect != sv.SPEC_OK:
        assert lib.spec_last_error().decode() != ""


def test_greedy_needs_no_draft(lib):
    # greedy with a null draft and null uniforms passes validation up to the workspace check
    assert _linear(lib, T=0.0, draft=None, u=None, ws=None) == sv.SPEC_ERR_WORKSPACE


def test_bonus_and_tree_host_validation(lib):
    f = lib.spec_sample_bonus
    W = 1 << 20
    assert f(FAKE, FAKE, 1, -1, 2, 10, FAKE, FAKE, 1.0, FAKE, FAKE, FAKE, W, None) == sv.SPEC_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 1, 2, 2, 10, None, FAKE, 1.0, FAKE, FAKE, FAKE, W, None) == sv.SPEC_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 1, 2, 2, 10, FAKE, None, 1.0, FAKE, FAKE, FAKE, W, None) == sv.SPEC_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 1, 2, 2, 10, FAKE, FAKE, 1.0, FAKE, FAKE, None, W, None) == sv.SPEC_ERR_WORKSPACE
    assert f(FAKE, FAKE, 1, 0, 2, 10, FAKE, FAKE, 1.0, FAKE, FAKE, FAKE, W, None) == sv.SPEC_OK
    t = lib.spec_verify_tree
    assert t(FAKE, 0, 2, 0, 10, FAKE, FAKE, 3, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert t(FAKE, 0, 2, 5, 10, FAKE, FAKE, -1, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert t(FAKE, 0, 2, 5, 10, None, FAKE, 3, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == sv.SPEC_ERR_INVALID_ARG
    assert t(FAKE, 0, 2, 5, 10, FAKE, FAKE, 3, FAKE, FAKE, FAKE, FAKE, None, 1 << 20, None) == sv.SPEC_ERR_WORKSPACE
    assert t(FAKE, 0, 0, 5, 10, FAKE, FAKE, 3, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == sv.SPEC_OK


def test_sample_rows_host_validation(lib):
    f = lib.spec_sample_rows
    W = 1 << 20
    assert f(FAKE, 1, -1, 10, FAKE, 1.0, FAKE, FAKE, FAKE, W, None) == sv.SPEC_ERR_INVALID_ARG
    assert f(FAKE, 1, 4, 0, FAKE, 1.0, FAKE, FAKE, FAKE, W, None) == sv.SPEC_ERR_INVALID_ARG
    assert f(FAKE, 1, 4, 10, None, 1.0, FAKE, FAKE, FAKE, W, None) == sv.SPEC_ERR_INVALID_ARG   # sampling needs u
    assert f(FAKE, 1, 4, 10, FAKE, -1.0, FAKE, FAKE, FAKE, W, None) == sv.SPEC_ERR_INVALID_ARG
    assert f(FAKE, 1, 4, 10, FAKE, 1.0, None, FAKE, FAKE, W, None) == sv.SPEC_ERR_INVALID_ARG
    assert f(FAKE, 1, 4, 10, None, 0.0, FAKE, FAKE, None, W, None) == sv.SPEC_ERR_WORKSPACE  # greedy: no u
    assert f(FAKE, 1, 0, 10, FAKE, 1.0, FAKE, FAKE, FAKE, W, None) == sv.SPEC_OK
    assert sv.spec_workspace_bytes_rows(8, 1000, sv.SPEC_BF16) > 0
    assert sv.spec_workspace_bytes_rows(0, 1000, sv.SPEC_BF16) == 0
    # the extra-token-alone call still needs its lengths
    assert lib.spec_sample_bonus(FAKE, FAKE, 1, 2, 2, 10, None, FAKE, 1.0, FAKE, FAKE, FAKE, W, None) == \
        sv.SPEC_ERR_INVALID_ARG


def test_tree_mask_host_validation(lib):
    f = lib.spec_tree_mask
    assert f(FAKE, 0, FAKE, FAKE, FAKE, None) == sv.SPEC_ERR_INVALID_ARG
    assert f(FAKE, 16385, FAKE, FAKE, FAKE, None) == sv.SPEC_ERR_UNSUPPORTED
    assert f(None, 10, FAKE, FAKE, FAKE, None) == sv.SPEC_ERR_INVALID_ARG
    assert f(FAKE, 10, FAKE, None, FAKE, None) == sv.SPEC_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(0x10002), 10, FAKE, FAKE, FAKE, None) == sv.SPEC_ERR_INVALID_ARG   # misaligned


def test_mtp_plug_host_validation(lib):
    f = lib.spec_mtp_plug
    OTHER = ctypes.c_void_p(0x20000)

    def call(inp=FAKE, B=4, K=1, ot=OTHER, ne=FAKE, nxt=FAKE, lens=FAKE, st=FAKE):
        return f(inp, B, K, ot, ne, 0, nxt, lens, st, None)
    assert call(B=-1) == sv.SPEC_ERR_INVALID_ARG
    assert call(K=-1) == sv.SPEC_ERR_INVALID_ARG
    assert call(B=0) == sv.SPEC_OK
    for kw in (dict(inp=None), dict(ot=None), dict(ne=None), dict(nxt=None), dict(st=None)):
        assert call(**kw) == sv.SPEC_ERR_INVALID_ARG
    assert call(nxt=OTHER) == sv.SPEC_ERR_INVALID_ARG                  # next_tokens must not be out_tokens
    assert call(lens=ctypes.c_void_p(0x10002)) == sv.SPEC_ERR_INVALID_ARG  # misaligned
    assert call(B=1 << 30, K=8) == sv.SPEC_ERR_UNSUPPORTED


def test_tree_sample_host_validation(lib):
    t = lib.spec_verify_tree_sample
    W = 1 << 20

    def call(B=2, N=5, V=10, u=FAKE, T=1.0, D=3, ws=FAKE, wsb=W):
        return t(FAKE, 0, B, N, V, FAKE, FAKE, u, T, D, FAKE, FAKE, FAKE, FAKE, ws, wsb, None)
    assert call(T=0.0) == sv.SPEC_ERR_INVALID_ARG          # sampling needs T > 0
    assert call(T=float("nan")) == sv.SPEC_ERR_INVALID_ARG
    assert call(u=None) == sv.SPEC_ERR_INVALID_ARG
    assert call(N=0) == sv.SPEC_ERR_INVALID_ARG
    assert call(D=-1) == sv.SPEC_ERR_INVALID_ARG
    assert call(ws=None) == sv.SPEC_ERR_WORKSPACE
    need = sv.spec_workspace_bytes_tree_sample(2, 5, 10, sv.SPEC_F32)
    assert call(wsb=need - 16) == sv.SPEC_ERR_WORKSPACE
    assert call(B=0) == sv.SPEC_OK
    # one draw entry and its chunk sums per node: more than the greedy walk needs
    assert need > sv.spec_workspace_bytes_tree(2, 5, 10, sv.SPEC_F32)
    assert sv.spec_workspace_bytes_tree_sample(0, 5, 10, sv.SPEC_F32) == 0


def test_binding_refuses_cpu_tensors(lib):
    import torch
    t = torch.zeros((1, 2, 8))
    with pytest.raises(ValueError):
        sv.spec_verify_linear(t, t[:, :1], torch.zeros((1, 1), dtype=torch.int32), torch.zeros((1, 1)),
                              torch.zeros(1), 1.0)
