"""Speculative-decoding verify-and-sample step for NVIDIA GB300 (sm_103a).

Python binding of ``libspecverify.so`` (C ABI in ``include/spec_verify.h``).
This module only marshals arguments: it allocates outputs and the workspace
with PyTorch, passes raw device pointers and the current CUDA stream, and
raises ``SpecError`` on a non-OK status.  Every step of the computation runs in
the library's CUDA kernels; there is no fallback, and importing the functions
fails loudly when the library has not been built.

Entry points (same names as the C ABI):
  spec_verify_linear   accept/reject K draft tokens per sequence and draw the
                       extra token ("Beschleunigung von Sonar durch Spekulation",
                       sections "Spekulatives Decoding" and "Ziel-Entwurf")
  spec_sample_bonus    the extra token alone, given accept_len
  spec_verify_tree     greedy walk of a Medusa candidate tree
                       ("Speculative-Decoding / Medusa", section 三)
  spec_verify_tree_sample  the same walk with the target's choice drawn at
                       every node (the section's sampled variant)
  spec_sample_rows     one token per row (the draft side's next token)
  spec_tree_mask       the tree attention mask (ancestor bits) and depths
  spec_build_sparse_tree  the greedy sparse candidate tree from per-head top-i
                       accuracies (the blog's section 四; host code)
  spec_mtp_plug        the MTP draft layer's next input tokens from a verify's
                       outputs, and the advanced lengths, on the device
                       ("Beschleunigung von Sonar durch Spekulation", sections
                       "MTP" and "MTP-Zeitplan für ein einzelnes Token")
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_UNSUPPORTED = 2
SPEC_ERR_CUDA = 3
SPEC_ERR_WORKSPACE = 4

SPEC_F32 = 0
SPEC_BF16 = 1

DEV_BAD_TOKEN = 1
DEV_NONFINITE = 2
DEV_TIMEOUT = 4
DEV_ZERO_RESIDUAL = 8
DEV_BAD_TREE = 16
DEV_BAD_LENGTH = 32


class SpecError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__("%s (%s)" % (detail, _status_name(status)))
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library():
    """Load libspecverify.so; raises ImportError if it was not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError("libspecverify.so is not built (run __graft_entry__.build() or "
                              "python -m sampling_online_softmax_gb300.build)")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, u64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
        lib.spec_workspace_bytes_linear.argtypes = [i32, i32, i32, i32]
        lib.spec_workspace_bytes_linear.restype = u64
        lib.spec_workspace_bytes_bonus.argtypes = [i32, i32, i32]
        lib.spec_workspace_bytes_bonus.restype = u64
        lib.spec_workspace_bytes_tree.argtypes = [i32, i32, i32, i32]
        lib.spec_workspace_bytes_tree.restype = u64
        lib.spec_workspace_bytes_tree_sample.argtypes = [i32, i32, i32, i32]
        lib.spec_workspace_bytes_rows.argtypes = [i32, i32, i32]
        lib.spec_workspace_bytes_rows.restype = u64
        lib.spec_sample_rows.argtypes = [P, i32, i32, i32, P, f32, P, P, P, u64, P]
        lib.spec_sample_rows.restype = i32
        lib.spec_tree_mask.argtypes = [P, i32, P, P, P, P]
        lib.spec_tree_mask.restype = i32
        lib.spec_build_sparse_tree.argtypes = [P, i32, i32, i32, P, P, P, P, P]
        lib.spec_build_sparse_tree.restype = i32
        lib.spec_mtp_plug.argtypes = [P, i32, i32, P, P, ctypes.c_int32, P, P, P, P]
        lib.spec_mtp_plug.restype = i32
        lib.spec_workspace_bytes_tree_sample.restype = u64
        lib.spec_verify_linear.argtypes = [P, P, i32, i32, i32, i32, P, P, P, f32, P, P, P, P, P, P, u64, P]
        lib.spec_verify_linear.restype = i32
        lib.spec_verify_linear_static.argtypes = [P, P, i32, i32, i32, i32, P, P, P, f32, P, P, P, P, P, P]
        lib.spec_verify_linear_static.restype = i32
        lib.spec_sample_bonus.argtypes = [P, P, i32, i32, i32, i32, P, P, f32, P, P, P, u64, P]
        lib.spec_sample_bonus.restype = i32
        lib.spec_verify_tree.argtypes = [P, i32, i32, i32, i32, P, P, i32, P, P, P, P, P, u64, P]
        lib.spec_verify_tree.restype = i32
        lib.spec_verify_tree_sample.argtypes = [P, i32, i32, i32, i32, P, P, P, f32, i32, P, P, P, P, P, u64, P]
        lib.spec_verify_tree_sample.restype = i32
        lib.spec_status_string.argtypes = [i32]
        lib.spec_status_string.restype = ctypes.c_char_p
        lib.spec_last_error.argtypes = []
        lib.spec_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _status_name(status: int) -> str:
    try:
        return load_library().spec_status_string(int(status)).decode()
    except ImportError:
        return "status %d" % status


def _check(status: int):
    if status != SPEC_OK:
        raise SpecError(status, load_library().spec_last_error().decode() or "call failed")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError("logits must be float32 or bfloat16, got %s" % t.dtype)


def _cuda(t, name, dtype=None, device=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, the logits on %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def _outputs(out, shapes, device):
    """Check caller-provided output tensors: every name present, int32/float32 as
    given, on `device`, contiguous, with exactly the shape the kernel writes."""
    for name, (shape, dtype) in shapes.items():
        t = out.get(name)
        if t is None:
            raise ValueError("out[%r] is missing" % name)
        _cuda(t, "out[%r]" % name, dtype, device)
        if tuple(t.shape) != tuple(shape):
            raise ValueError("out[%r] must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return out


def _status(status, device, stream):
    if status is None:
        with torch.cuda.stream(stream):
            return torch.zeros(1, dtype=torch.int32, device=device)
    _cuda(status, "status", torch.int32, device)
    if status.numel() < 1:
        raise ValueError("status must hold at least one int32")
    return status


def _ws(workspace, nbytes, device, stream):
    if workspace is None:
        return _workspace(device, stream, nbytes)
    _cuda(workspace, "workspace", None, device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError("workspace needs %d bytes" % nbytes)
    return workspace


def _tree_shapes(parents, node_tokens, B, N):
    if parents.numel() != N:
        raise ValueError("parents must hold N = %d entries" % N)
    if tuple(node_tokens.shape) != (B, N):
        raise ValueError("node_tokens must be [B, N]")


def _tree_inputs(target, parents, node_tokens):
    """Check the inputs of a tree verify; returns (B, N, V, device)."""
    _cuda(target, "target")
    if target.dim() != 3:
        raise ValueError("target must be [B, N, V]")
    B, N, V = target.shape
    dev = target.device
    if parents is None or node_tokens is None:
        raise ValueError("parents and node_tokens are required")
    _cuda(parents, "parents", torch.int32, dev)
    _cuda(node_tokens, "node_tokens", torch.int32, dev)
    _tree_shapes(parents, node_tokens, B, N)
    return B, N, V, dev


def _tree_outputs(out, B, D, dev):
    if D < 0:
        raise ValueError("max_depth must be >= 0")
    if out is None:
        out = dict(path_nodes=torch.empty((B, D + 1), dtype=torch.int32, device=dev),
                   path_len=torch.empty(B, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty((B, D + 1), dtype=torch.int32, device=dev))
    return _outputs(out, {"path_nodes": ((B, D + 1), torch.int32), "path_len": ((B,), torch.int32),
                          "out_tokens": ((B, D + 1), torch.int32)}, dev)


def _stream_handle(device, stream):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream), s


# one zero-filled workspace per (device, stream), grown on demand; every call
# leaves it zero-filled again, so it is cleared only when allocated
_ws_cache = {}
_ws_lock = threading.Lock()


def _workspace(device, stream, nbytes):
    key = (device.index, stream.cuda_stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            with torch.cuda.stream(stream):
                ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
        return ws


def _dtype_arg(dtype) -> int:
    if isinstance(dtype, torch.dtype):
        return SPEC_F32 if dtype == torch.float32 else SPEC_BF16
    return int(dtype)


def spec_workspace_bytes_linear(B: int, K: int, V: int, dtype) -> int:
    return int(load_library().spec_workspace_bytes_linear(int(B), int(K), int(V), _dtype_arg(dtype)))


def spec_workspace_bytes_bonus(B: int, V: int, dtype) -> int:
    return int(load_library().spec_workspace_bytes_bonus(int(B), int(V), _dtype_arg(dtype)))


def spec_workspace_bytes_tree(B: int, N: int, V: int, dtype) -> int:
    return int(load_library().spec_workspace_bytes_tree(int(B), int(N), int(V), _dtype_arg(dtype)))


def spec_workspace_bytes_rows(B: int, V: int, dtype) -> int:
    return int(load_library().spec_workspace_bytes_rows(int(B), int(V), _dtype_arg(dtype)))


def spec_workspace_bytes_tree_sample(B: int, N: int, V: int, dtype) -> int:
    return int(load_library().spec_workspace_bytes_tree_sample(int(B), int(N), int(V), _dtype_arg(dtype)))


def _linear_inputs(target, draft, draft_tokens, u_accept, u_bonus):
    """Check the inputs of a linear verify; returns (B, K, V, device)."""
    _cuda(target, "target")
    if target.dim() != 3:
        raise ValueError("target must be [B, K+1, V]")
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    _cuda(draft, "draft", None, dev)
    _cuda(draft_tokens, "draft_tokens", torch.int32, dev)
    _cuda(u_accept, "u_accept", torch.float32, dev)
    _cuda(u_bonus, "u_bonus", torch.float32, dev)
    if draft is not None and (draft.dtype != target.dtype or tuple(draft.shape) != (B, K, V)):
        raise ValueError("draft must match target's dtype with shape [B, K, V]")
    if draft_tokens is not None and tuple(draft_tokens.shape) != (B, K):
        raise ValueError("draft_tokens must be [B, K]")
    if u_accept is not None and tuple(u_accept.shape) != (B, K):
        raise ValueError("u_accept must be [B, K]")
    if u_bonus is not None and tuple(u_bonus.shape) != (B,):
        raise ValueError("u_bonus must be [B]")
    return B, K, V, dev


def _linear_outputs(out, B, K, dev):
    shapes = {"accept_len": ((B,), torch.int32), "out_tokens": ((B, K + 1), torch.int32),
              "num_emitted": ((B,), torch.int32)}
    if out.get("probs") is not None:
        shapes["probs"] = ((B, K, 3), torch.float32)
    return _outputs(out, shapes, dev)


def spec_verify_linear(target, draft, draft_tokens, u_accept, u_bonus, temperature, *,
                       probs: bool = False, status=None, out=None, workspace=None, stream=None):
    """Verify K draft tokens per sequence; returns a dict of device tensors.

    target [B, K+1, V] and draft [B, K, V] (float32 or bfloat16; draft may be
    None in greedy mode), draft_tokens [B, K] int32, u_accept [B, K] float32,
    u_bonus [B] float32 or None (no extra token), temperature >= 0 (0: greedy).
    Result: accept_len [B], out_tokens [B, K+1], num_emitted [B], status [1]
    (SPEC_DEV_* bits, int32), and probs [B, K, 3] when requested.
    """
    lib = load_library()
    B, K, V, dev = _linear_inputs(target, draft, draft_tokens, u_accept, u_bonus)
    h, s = _stream_handle(dev, stream)
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   out_tokens=torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                   num_emitted=torch.empty(B, dtype=torch.int32, device=dev))
        if probs:
            out["probs"] = torch.empty((B, K, 3), dtype=torch.float32, device=dev)
    _linear_outputs(out, B, K, dev)
    status = _status(status, dev, s)
    out["status"] = status
    nbytes = spec_workspace_bytes_linear(B, K, V, target.dtype)
    ws = _ws(workspace, nbytes, dev, s)
    with torch.cuda.device(dev):
        st = lib.spec_verify_linear(
            _ptr(target), _ptr(draft), _dtype_code(target), B, K, V, _ptr(draft_tokens), _ptr(u_accept),
            _ptr(u_bonus), float(temperature), _ptr(out["accept_len"]), _ptr(out["out_tokens"]),
            _ptr(out["num_emitted"]), _ptr(out.get("probs")), _ptr(status), _ptr(ws), ws.numel(), h)
    _check(st)
    return out


def spec_verify_linear_static(target, draft, draft_tokens, u_accept, u_bonus, temperature, *, out, status,
                              stream=None):
    """spec_verify_linear on the library's built-in per-device workspace.

    For callers that must not allocate device memory during the step: nothing
    is allocated here either, so `out` (accept_len, out_tokens, num_emitted and
    optionally probs, as returned by spec_verify_linear) and `status` (int32 [1],
    zeroed by the caller) must be passed in.  Calls that may overlap in time
    share the one workspace and race; keep them on one stream.
    """
    lib = load_library()
    B, K, V, dev = _linear_inputs(target, draft, draft_tokens, u_accept, u_bonus)
    _linear_outputs(out, B, K, dev)
    if status is None:
        raise ValueError("status must be passed in (nothing is allocated here)")
    _cuda(status, "status", torch.int32, dev)
    if status.numel() < 1:
        raise ValueError("status must hold at least one int32")
    h, _ = _stream_handle(dev, stream)
    with torch.cuda.device(dev):
        st = lib.spec_verify_linear_static(
            _ptr(target), _ptr(draft), _dtype_code(target), B, K, V, _ptr(draft_tokens), _ptr(u_accept),
            _ptr(u_bonus), float(temperature), _ptr(out["accept_len"]), _ptr(out["out_tokens"]),
            _ptr(out["num_emitted"]), _ptr(out.get("probs")), _ptr(status), h)
    _check(st)
    out["status"] = status
    return out


def spec_sample_bonus(target, draft, accept_len, u_bonus, temperature, *, status=None, out=None, workspace=None,
                      stream=None):
    """The extra token alone at row accept_len[b]; returns dict(bonus_token [B], status [1])."""
    lib = load_library()
    _cuda(target, "target")
    if target.dim() != 3:
        raise ValueError("target must be [B, K+1, V]")
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    _cuda(draft, "draft", None, dev)
    _cuda(accept_len, "accept_len", torch.int32, dev)
    _cuda(u_bonus, "u_bonus", torch.float32, dev)
    if draft is not None and (draft.dtype != target.dtype or tuple(draft.shape) != (B, K, V)):
        raise ValueError("draft must match target's dtype with shape [B, K, V]")
    if accept_len is not None and tuple(accept_len.shape) != (B,):
        raise ValueError("accept_len must be [B]")
    if u_bonus is not None and tuple(u_bonus.shape) != (B,):
        raise ValueError("u_bonus must be [B]")
    h, s = _stream_handle(dev, stream)
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=dev)
    _outputs(dict(bonus_token=out), {"bonus_token": ((B,), torch.int32)}, dev)
    status = _status(status, dev, s)
    nbytes = spec_workspace_bytes_bonus(B, V, target.dtype)
    ws = _ws(workspace, nbytes, dev, s)
    with torch.cuda.device(dev):
        st = lib.spec_sample_bonus(_ptr(target), _ptr(draft), _dtype_code(target), B, K, V, _ptr(accept_len),
                                   _ptr(u_bonus), float(temperature), _ptr(out), _ptr(status), _ptr(ws),
                                   ws.numel(), h)
    _check(st)
    return dict(bonus_token=out, status=status)


def spec_verify_tree(target, parents, node_tokens, max_depth, *, status=None, out=None, workspace=None,
                     stream=None):
    """Greedy tree walk; returns dict(path_nodes, path_len, out_tokens, status)."""
    lib = load_library()
    B, N, V, dev = _tree_inputs(target, parents, node_tokens)
    h, s = _stream_handle(dev, stream)
    D = int(max_depth)
    out = _tree_outputs(out, B, D, dev)
    status = _status(status, dev, s)
    out["status"] = status
    nbytes = spec_workspace_bytes_tree(B, N, V, target.dtype)
    ws = _ws(workspace, nbytes, dev, s)
    with torch.cuda.device(dev):
        st = lib.spec_verify_tree(_ptr(target), _dtype_code(target), B, N, V, _ptr(parents), _ptr(node_tokens), D,
                                  _ptr(out["path_nodes"]), _ptr(out["path_len"]), _ptr(out["out_tokens"]),
                                  _ptr(status), _ptr(ws), ws.numel(), h)
    _check(st)
    return out


def spec_verify_tree_sample(target, parents, node_tokens, u_nodes, temperature, max_depth, *, status=None,
                            out=None, workspace=None, stream=None):
    """Tree walk with the target's choice drawn at every node (u_nodes [B, N] fp32);
    returns dict(path_nodes, path_len, out_tokens, status)."""
    lib = load_library()
    B, N, V, dev = _tree_inputs(target, parents, node_tokens)
    if u_nodes is None:
        raise ValueError("u_nodes is required")
    _cuda(u_nodes, "u_nodes", torch.float32, dev)
    if tuple(u_nodes.shape) != (B, N):
        raise ValueError("u_nodes must be [B, N]")
    h, s = _stream_handle(dev, stream)
    D = int(max_depth)
    out = _tree_outputs(out, B, D, dev)
    status = _status(status, dev, s)
    out["status"] = status
    nbytes = spec_workspace_bytes_tree_sample(B, N, V, target.dtype)
    ws = _ws(workspace, nbytes, dev, s)
    with torch.cuda.device(dev):
        st = lib.spec_verify_tree_sample(_ptr(target), _dtype_code(target), B, N, V, _ptr(parents),
                                         _ptr(node_tokens), _ptr(u_nodes), float(temperature), D,
                                         _ptr(out["path_nodes"]), _ptr(out["path_len"]), _ptr(out["out_tokens"]),
                                         _ptr(status), _ptr(ws), ws.numel(), h)
    _check(st)
    return out


def spec_sample_rows(logits, u, temperature, *, status=None, out=None, workspace=None, stream=None):
    """One token per row of logits [B, V]: a draw from softmax(l / T) at u [B] (float32), or the
    argmax when temperature == 0 (u may be None); returns dict(tokens [B], status)."""
    lib = load_library()
    _cuda(logits, "logits")
    if logits.dim() != 2:
        raise ValueError("logits must be [B, V]")
    B, V = logits.shape
    dev = logits.device
    _cuda(u, "u", torch.float32, dev)
    if u is not None and tuple(u.shape) != (B,):
        raise ValueError("u must be [B]")
    h, s = _stream_handle(dev, stream)
    if out is None:
        out = dict(tokens=torch.empty(B, dtype=torch.int32, device=dev))
    _outputs(out, {"tokens": ((B,), torch.int32)}, dev)
    status = _status(status, dev, s)
    out["status"] = status
    nbytes = spec_workspace_bytes_rows(B, V, logits.dtype)
    ws = _ws(workspace, nbytes, dev, s)
    with torch.cuda.device(dev):
        st = lib.spec_sample_rows(_ptr(logits), _dtype_code(logits), B, V, _ptr(u), float(temperature),
                                  _ptr(out["tokens"]), _ptr(status), _ptr(ws), ws.numel(), h)
    _check(st)
    return out


def spec_tree_mask(parents, *, status=None, out=None, stream=None):
    """Tree attention mask of a parent array [N] (int32, CUDA): returns dict(mask [N, ceil(N/32)]
    (int32 words holding uint32 bits: bit j % 32 of word j // 32 of row i is set iff node j is node
    i or an ancestor), depth [N], status)."""
    lib = load_library()
    _cuda(parents, "parents", torch.int32)
    N = parents.numel()
    dev = parents.device
    h, s = _stream_handle(dev, stream)
    W = (N + 31) // 32
    if out is None:
        out = dict(mask=torch.empty((N, W), dtype=torch.int32, device=dev),
                   depth=torch.empty(N, dtype=torch.int32, device=dev))
    _outputs(out, {"mask": ((N, W), torch.int32), "depth": ((N,), torch.int32)}, dev)
    status = _status(status, dev, s)
    out["status"] = status
    with torch.cuda.device(dev):
        st = lib.spec_tree_mask(_ptr(parents), N, _ptr(out["mask"]), _ptr(out["depth"]), _ptr(status), h)
    _check(st)
    return out


def spec_mtp_plug(in_tokens, out_tokens, num_emitted, pad=0, seq_lens=None, *, in_place=False, out=None,
                  status=None, stream=None):
    """The MTP draft layer's next input tokens [B, K+1]: in_tokens shifted left by one, with
    the verify's emitted tokens (out_tokens [B, K+1], num_emitted [B]) in their places and
    `pad` at the end; seq_lens [B] (int32, optional) grows by num_emitted in place.
    in_place=True writes into in_tokens.  Returns dict(next_tokens, seq_lens, status)."""
    lib = load_library()
    _cuda(in_tokens, "in_tokens", torch.int32)
    if in_tokens.dim() != 2:
        raise ValueError("in_tokens must be [B, K+1]")
    B, W = in_tokens.shape
    dev = in_tokens.device
    _cuda(out_tokens, "out_tokens", torch.int32, dev)
    _cuda(num_emitted, "num_emitted", torch.int32, dev)
    _cuda(seq_lens, "seq_lens", torch.int32, dev)
    if out_tokens is None or tuple(out_tokens.shape) != (B, W):
        raise ValueError("out_tokens must be [B, K+1]")
    if num_emitted is None or tuple(num_emitted.shape) != (B,):
        raise ValueError("num_emitted must be [B]")
    if seq_lens is not None and tuple(seq_lens.shape) != (B,):
        raise ValueError("seq_lens must be [B]")
    h, s = _stream_handle(dev, stream)
    if in_place:
        nxt = in_tokens
    else:
        nxt = out if out is not None else torch.empty((B, W), dtype=torch.int32, device=dev)
        _outputs(dict(next_tokens=nxt), {"next_tokens": ((B, W), torch.int32)}, dev)
    status = _status(status, dev, s)
    with torch.cuda.device(dev):
        st = lib.spec_mtp_plug(_ptr(in_tokens), B, W - 1, _ptr(out_tokens), _ptr(num_emitted), int(pad), _ptr(nxt),
                               _ptr(seq_lens), _ptr(status), h)
    _check(st)
    return dict(next_tokens=nxt, seq_lens=seq_lens, status=status)


def spec_build_sparse_tree(accuracy, n_nodes):
    """Greedy sparse candidate tree (host): accuracy [K, S] (a_k^(i) at [k-1, i-1], numpy or
    a CPU tensor, values in [0, 1]) and the node count wanted (root included).  Returns
    dict(parents, depth, rank) as int32 numpy arrays of the nodes built, and expected_len."""
    import numpy as np
    lib = load_library()
    acc = np.ascontiguousarray(np.asarray(accuracy, dtype=np.float64))
    if acc.ndim != 2:
        raise ValueError("accuracy must be [K, S]")
    K, S = acc.shape
    n = int(n_nodes)
    par, dep, rk = (np.zeros(max(n, 1), np.int32) for _ in range(3))
    nb, el = ctypes.c_int(0), ctypes.c_double(0.0)
    st = lib.spec_build_sparse_tree(acc.ctypes.data_as(ctypes.c_void_p), K, S, n,
                                    par.ctypes.data_as(ctypes.c_void_p), dep.ctypes.data_as(ctypes.c_void_p),
                                    rk.ctypes.data_as(ctypes.c_void_p), ctypes.byref(nb), ctypes.byref(el))
    _check(st)
    m = nb.value
    return dict(parents=par[:m].copy(), depth=dep[:m].copy(), rank=rk[:m].copy(), expected_len=el.value)
