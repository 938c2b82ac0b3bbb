"""CPU oracle for the speculative-decoding verify-and-sample step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library: the arithmetic lives in ``spec_oracle.c`` (plain C,
float64, one sequential loop per row), compiled here with gcc, and this module
only marshals numpy arrays into it.

The functions follow "Beschleunigung von Sonar durch Spekulation" (Perplexity),
sections "Spekulatives Decoding" and "Ziel-Entwurf", with the acceptance rule of
the method that page cites ("Fast Inference from Transformers via Speculative
Decoding"), and section 三 (Attention Tree) of the "Speculative-Decoding /
Medusa" blog for the tree walk.  The header of ``spec_oracle.c`` lists every
reading taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F32 = 0
BF16 = 1
FLAG_ZERO_RESIDUAL = 1
FLAG_BAD_TOKEN = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (OpenMP over sequences) and return the .so path."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    P = ctypes.c_void_p
    i32 = ctypes.c_int
    lib.oracle_verify_linear.argtypes = [P, P, i32, i32, i32, i32, P, P, P, ctypes.c_float,
                                         P, P, P, P, P, P]
    lib.oracle_verify_linear.restype = i32
    lib.oracle_sample_bonus.argtypes = [P, P, i32, i32, i32, i32, P, P, ctypes.c_float,
                                        P, P, P]
    lib.oracle_sample_bonus.restype = i32
    lib.oracle_verify_tree.argtypes = [P, i32, i32, i32, i32, P, P, i32, P, P, P]
    lib.oracle_verify_tree.restype = i32
    lib.oracle_verify_tree_sample.argtypes = [P, i32, i32, i32, i32, P, P, P, ctypes.c_float, i32,
                                              P, P, P, P]
    lib.oracle_verify_tree_sample.restype = i32
    lib.oracle_sample_rows.argtypes = [P, i32, i32, i32, P, ctypes.c_float, P, P]
    lib.oracle_sample_rows.restype = i32
    lib.oracle_tree_mask.argtypes = [P, i32, P, P]
    lib.oracle_tree_mask.restype = i32
    lib.oracle_mtp_plug.argtypes = [P, i32, i32, P, P, ctypes.c_int32, P, P]
    lib.oracle_mtp_plug.restype = i32
    lib.oracle_build_sparse_tree.argtypes = [P, i32, i32, i32, P, P, P, P, P]
    lib.oracle_build_sparse_tree.restype = i32
    lib.oracle_threads.argtypes = [i32]
    lib.oracle_threads.restype = i32
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.  A path loads that build."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def threads(n: int = 0, lib=None) -> int:
    """Set (n > 0) and return the number of OpenMP threads the oracle uses."""
    return (lib or load()).oracle_threads(int(n))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    """numpy float32 -> (array, F32); numpy uint16 holding bf16 bits -> (array, BF16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError("oracle logits must be float32 or uint16 (bf16 bits), got %s" % a.dtype)


def verify_linear(target, draft, draft_tokens, u_accept, u_bonus, temperature, lib=None):
    """Linear verify.  target [B, K+1, V], draft [B, K, V] (None allowed when
    temperature == 0), draft_tokens [B, K] int32, u_accept [B, K] float32,
    u_bonus [B] float32 or None.  Returns a dict of numpy arrays."""
    lib = lib or load()
    target, dt = _logits(target)
    B, K1, V = target.shape
    K = K1 - 1
    if draft is not None:
        draft, dd = _logits(draft)
        assert dd == dt and draft.shape == (B, K, V)
    tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, K)
    ua = None if u_accept is None else np.ascontiguousarray(u_accept, dtype=np.float32).reshape(B, K)
    ub = None if u_bonus is None else np.ascontiguousarray(u_bonus, dtype=np.float32).reshape(B)
    out = dict(
        accept_len=np.zeros(B, np.int32),
        out_tokens=np.zeros((B, K + 1), np.int32),
        num_emitted=np.zeros(B, np.int32),
        probs=np.zeros((B, K, 3), np.float64),
        bonus_cdf=np.zeros((B, 2), np.float64),
        flags=np.zeros(B, np.uint32),
    )
    rc = lib.oracle_verify_linear(
        _ptr(target), _ptr(draft), dt, B, K, V, _ptr(tokens), _ptr(ua), _ptr(ub),
        ctypes.c_float(temperature), _ptr(out["accept_len"]), _ptr(out["out_tokens"]),
        _ptr(out["num_emitted"]), _ptr(out["probs"]), _ptr(out["bonus_cdf"]), _ptr(out["flags"]))
    if rc != 0:
        raise ValueError("oracle_verify_linear rejected its arguments")
    return out


def sample_bonus(target, draft, accept_len, u_bonus, temperature, lib=None):
    """The extra token alone at row accept_len[b] of each sequence."""
    lib = lib or load()
    target, dt = _logits(target)
    B, K1, V = target.shape
    K = K1 - 1
    if draft is not None:
        draft, dd = _logits(draft)
        assert dd == dt and draft.shape == (B, K, V)
    al = np.ascontiguousarray(accept_len, dtype=np.int32).reshape(B)
    ub = None if u_bonus is None else np.ascontiguousarray(u_bonus, dtype=np.float32).reshape(B)
    out = dict(bonus_token=np.zeros(B, np.int32), bonus_cdf=np.zeros((B, 2), np.float64),
               flags=np.zeros(B, np.uint32))
    rc = lib.oracle_sample_bonus(_ptr(target), _ptr(draft), dt, B, K, V, _ptr(al), _ptr(ub),
                                 ctypes.c_float(temperature), _ptr(out["bonus_token"]),
                                 _ptr(out["bonus_cdf"]), _ptr(out["flags"]))
    if rc != 0:
        raise ValueError("oracle_sample_bonus rejected its arguments")
    return out


def verify_tree(target, parents, node_tokens, max_depth, lib=None):
    """Greedy tree verify.  target [B, N, V], parents [N], node_tokens [B, N]."""
    lib = lib or load()
    target, dt = _logits(target)
    B, N, V = target.shape
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(N)
    tok = np.ascontiguousarray(node_tokens, dtype=np.int32).reshape(B, N)
    out = dict(path_nodes=np.zeros((B, max_depth + 1), np.int32),
               path_len=np.zeros(B, np.int32),
               out_tokens=np.zeros((B, max_depth + 1), np.int32))
    rc = lib.oracle_verify_tree(_ptr(target), dt, B, N, V, _ptr(par), _ptr(tok), int(max_depth),
                                _ptr(out["path_nodes"]), _ptr(out["path_len"]),
                                _ptr(out["out_tokens"]))
    if rc != 0:
        raise ValueError("oracle_verify_tree rejected its arguments")
    return out


def verify_tree_sample(target, parents, node_tokens, u_nodes, temperature, max_depth, lib=None):
    """Tree verify in sampling mode.  target [B, N, V], parents [N], node_tokens [B, N],
    u_nodes [B, N] (the uniform of the target's draw at each node), temperature > 0.
    node_cdf [B, N, 2] is every node's draw as its normalised cumulative interval."""
    lib = lib or load()
    target, dt = _logits(target)
    B, N, V = target.shape
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(N)
    tok = np.ascontiguousarray(node_tokens, dtype=np.int32).reshape(B, N)
    un = np.ascontiguousarray(u_nodes, dtype=np.float32).reshape(B, N)
    out = dict(path_nodes=np.zeros((B, max_depth + 1), np.int32),
               path_len=np.zeros(B, np.int32),
               out_tokens=np.zeros((B, max_depth + 1), np.int32),
               node_cdf=np.zeros((B, N, 2), np.float64))
    rc = lib.oracle_verify_tree_sample(_ptr(target), dt, B, N, V, _ptr(par), _ptr(tok), _ptr(un),
                                       float(temperature), int(max_depth), _ptr(out["path_nodes"]),
                                       _ptr(out["path_len"]), _ptr(out["out_tokens"]), _ptr(out["node_cdf"]))
    if rc != 0:
        raise ValueError("oracle_verify_tree_sample rejected its arguments")
    return out


def sample_rows(logits, u, temperature, lib=None):
    """One token per row of logits [B, V]: a draw from softmax(l / T) at u [B], or argmax when T == 0.
    Returns dict(tokens [B], cdf [B, 2])."""
    lib = lib or load()
    logits, dt = _logits(logits)
    B, V = logits.shape
    uu = None if u is None else np.ascontiguousarray(u, dtype=np.float32).reshape(B)
    if temperature > 0 and uu is None:
        raise ValueError("sampling needs u")
    out = dict(tokens=np.zeros(B, np.int32), cdf=np.zeros((B, 2), np.float64))
    rc = lib.oracle_sample_rows(_ptr(logits), dt, B, V, _ptr(uu) if uu is not None else None, float(temperature),
                                _ptr(out["tokens"]), _ptr(out["cdf"]))
    if rc != 0:
        raise ValueError("oracle_sample_rows rejected its arguments")
    return out


def tree_mask(parents, lib=None):
    """Ancestor-or-self bitmask [N, ceil(N/32)] uint32 and depth [N] of a parent array.
    Returns dict(mask, depth, bad) (bad: some parent was not an earlier node)."""
    lib = lib or load()
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(-1)
    N = len(par)
    W = (N + 31) // 32
    out = dict(mask=np.zeros((N, W), np.uint32), depth=np.zeros(N, np.int32))
    rc = lib.oracle_tree_mask(_ptr(par), N, _ptr(out["mask"]), _ptr(out["depth"]))
    if rc == 1:
        raise ValueError("oracle_tree_mask rejected its arguments")
    out["bad"] = rc == 2
    return out


def mask_bits(mask, N):
    """The bitmask as a dense [N, N] 0/1 array."""
    bits = np.unpackbits(np.ascontiguousarray(mask).view(np.uint8), axis=1, bitorder="little")
    return bits[:, :N]


def mtp_plug(in_tokens, out_tokens, num_emitted, pad=0, seq_lens=None, lib=None):
    """MTP token plug-in: the draft's next input tokens from the target's input
    tokens [B, K+1] and a linear verify's out_tokens [B, K+1] and num_emitted [B].
    Returns dict(next_tokens [B, K+1], seq_lens [B] or None, bad)."""
    lib = lib or load()
    inp = np.ascontiguousarray(in_tokens, dtype=np.int32)
    B, W = inp.shape
    ot = np.ascontiguousarray(out_tokens, dtype=np.int32).reshape(B, W)
    ne = np.ascontiguousarray(num_emitted, dtype=np.int32).reshape(B)
    nxt = np.zeros((B, W), np.int32)
    sl = None if seq_lens is None else np.array(seq_lens, dtype=np.int32).reshape(B)
    rc = lib.oracle_mtp_plug(_ptr(inp), B, W - 1, _ptr(ot), _ptr(ne), int(pad), _ptr(nxt), _ptr(sl))
    if rc == 1:
        raise ValueError("oracle_mtp_plug rejected its arguments")
    return dict(next_tokens=nxt, seq_lens=sl, bad=rc == 2)


def build_sparse_tree(accuracy, n_nodes, lib=None):
    """Greedy sparse candidate tree from an accuracy table [K, S] (a_k^(i) at [k-1, i-1]) with
    n_nodes nodes (root included; fewer when the full tree is smaller).
    Returns dict(parents, depth, rank, expected_len)."""
    lib = lib or load()
    acc = np.ascontiguousarray(accuracy, dtype=np.float64)
    K, S = acc.shape
    par = np.zeros(n_nodes, np.int32)
    dep = np.zeros(n_nodes, np.int32)
    rk = np.zeros(n_nodes, np.int32)
    nb = ctypes.c_int(0)
    el = ctypes.c_double(0.0)
    rc = lib.oracle_build_sparse_tree(_ptr(acc), K, S, int(n_nodes), _ptr(par), _ptr(dep), _ptr(rk),
                                      ctypes.byref(nb), ctypes.byref(el))
    if rc != 0:
        raise ValueError("oracle_build_sparse_tree rejected its arguments")
    n = nb.value
    return dict(parents=par[:n], depth=dep[:n], rank=rk[:n], expected_len=el.value)
