"""Seeded synthetic inputs for the verify-and-sample step.

This module is shared by the tests, the benchmark and the smoke check.  It
holds none of the verify step's arithmetic: it draws logits, draft tokens and
uniforms, and nothing here computes an acceptance test, a softmax ratio or a
residual.  Draft tokens stand in for the draft model's own sampler: in sampling
mode they are drawn from softmax(draft / T) with the Gumbel-max construction
(argmax of draft / T + Gumbel noise, which is an exact draw from that
softmax), in greedy mode they are argmax(draft).

Workloads (sizes and distributions; the pages give none of their own for this
step, so these stand in for the draft-target, MTP, Medusa and large-batch
settings that "Beschleunigung von Sonar durch Spekulation" and the
"Speculative-Decoding / Medusa" blog describe):

  linear_small   B=4,   K=4, V=32000  fp32  target ~N(0,3^2); draft = target + N(0,1)
  draft_target   B=64,  K=4, V=128256 bf16  target ~N(0,4^2), 5 % of rows get one
                 random token +12; draft = 0.8 * target + N(0,1.5^2); T = 0.7
  mtp_single     B=256, K=1, V=129280 bf16  target [B,2,V] ~N(0,4^2) (2*B scored
                 tokens); draft = target row 0 + N(0,2^2); greedy and T = 1
  medusa_tree    B=16,  N=64 nodes, V=32000 fp32 target ~N(0,3^2); 64-node tree
                 built from a_k^(i) = 0.6 * 0.8^k * 0.5^i; node tokens drawn per head
  stress         B=512, K=8, V=152064 bf16  target ~N(0,5^2), 30 % of rows get one
                 logit +20; draft = target + N(0,1); T = 0.7

Every array is drawn from one torch.Generator seeded with 1000 + workload number,
on the device the caller names, in a fixed order and in fixed-size batches of
sequences, so the same (workload, device, sizes) always gives the same bytes.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import medusa_tree  # noqa: F401  (re-exported)


@dataclasses.dataclass(frozen=True)
class Workload:
    number: int
    name: str
    kind: str           # "linear" or "tree"
    B: int
    K: int              # draft positions (linear) or heads (tree depth)
    V: int
    dtype: str          # "f32" or "bf16"
    temperatures: tuple
    N: int = 0          # tree nodes including the root
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def logits_bytes(self, temperature: float) -> int:
        """Bytes of logits one verify call reads (each logit once)."""
        eb = 4 if self.dtype == "f32" else 2
        if self.kind == "tree":
            return self.B * self.N * self.V * eb
        rows = self.K + 1 + (self.K if temperature > 0 else 0)
        return self.B * rows * self.V * eb


WORKLOADS = {
    1: Workload(1, "linear_small", "linear", 4, 4, 32000, "f32", (1.0, 0.0), seed=1001),
    2: Workload(2, "draft_target", "linear", 64, 4, 128256, "bf16", (0.7,), seed=1002),
    3: Workload(3, "mtp_single", "linear", 256, 1, 129280, "bf16", (0.0, 1.0), seed=1003),
    4: Workload(4, "medusa_tree", "tree", 16, 4, 32000, "f32", (0.0,), N=64, seed=1004),
    5: Workload(5, "stress", "linear", 512, 8, 152064, "bf16", (0.7,), seed=1005),
}

# sequences generated per batch (fixed, so the bytes do not depend on memory)
_GEN_BATCH = 16


def _gumbel_argmax(logits_f32: torch.Tensor, temperature: float, gen: torch.Generator) -> torch.Tensor:
    """One exact draw from softmax(logits / T) per row via the Gumbel-max construction."""
    u = torch.rand(logits_f32.shape, generator=gen, device=logits_f32.device, dtype=torch.float64)
    u = u.clamp_(min=1e-300)
    g = -torch.log(-torch.log(u))
    return torch.argmax(logits_f32.double() / temperature + g, dim=-1).to(torch.int32)


def _linear_rows(w: Workload, b: int, K: int, V: int, gen, device):
    """Target [b, K+1, V] and draft [b, K, V] (float32) for one batch of sequences."""
    if w.number == 1:
        t = 3.0 * torch.randn((b, K + 1, V), generator=gen, device=device)
        d = t[:, :K] + torch.randn((b, K, V), generator=gen, device=device)
    elif w.number == 2:
        t = 4.0 * torch.randn((b, K + 1, V), generator=gen, device=device)
        spike = torch.rand((b, K + 1), generator=gen, device=device) < 0.05
        tok = torch.randint(0, V, (b, K + 1), generator=gen, device=device)
        t.scatter_add_(2, tok.unsqueeze(-1), 12.0 * spike.unsqueeze(-1).float())
        d = 0.8 * t[:, :K] + 1.5 * torch.randn((b, K, V), generator=gen, device=device)
    elif w.number == 3:
        t = 4.0 * torch.randn((b, K + 1, V), generator=gen, device=device)
        d = t[:, :K] + 2.0 * torch.randn((b, K, V), generator=gen, device=device)
    elif w.number == 5:
        t = 5.0 * torch.randn((b, K + 1, V), generator=gen, device=device)
        spike = torch.rand((b, K + 1), generator=gen, device=device) < 0.30
        tok = torch.randint(0, V, (b, K + 1), generator=gen, device=device)
        t.scatter_add_(2, tok.unsqueeze(-1), 20.0 * spike.unsqueeze(-1).float())
        d = t[:, :K] + torch.randn((b, K, V), generator=gen, device=device)
    else:
        raise ValueError("workload %d is not a linear workload" % w.number)
    return t, d


def make_linear(number: int, temperature: float, device="cpu", B: int | None = None,
                K: int | None = None, V: int | None = None, seed: int | None = None):
    """Inputs of one linear-verify workload, optionally with smaller B / K / V.

    Returns dict(target [B,K+1,V], draft [B,K,V], draft_tokens [B,K] int32,
    u_accept [B,K] float32, u_bonus [B] float32, temperature) on ``device``;
    logits in the workload's dtype.
    """
    w = WORKLOADS[number]
    B = w.B if B is None else B
    K = w.K if K is None else K
    V = w.V if V is None else V
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    target = torch.empty((B, K + 1, V), dtype=w.torch_dtype, device=device)
    draft = torch.empty((B, K, V), dtype=w.torch_dtype, device=device)
    tokens = torch.empty((B, K), dtype=torch.int32, device=device)
    for b0 in range(0, B, _GEN_BATCH):
        nb = min(_GEN_BATCH, B - b0)
        t, d = _linear_rows(w, nb, K, V, gen, device)
        target[b0:b0 + nb] = t.to(w.torch_dtype)
        draft[b0:b0 + nb] = d.to(w.torch_dtype)
        if K > 0:
            dq = draft[b0:b0 + nb].float()   # the draft the verifier sees
            if temperature > 0:
                tokens[b0:b0 + nb] = _gumbel_argmax(dq, temperature, gen)
            else:
                tokens[b0:b0 + nb] = torch.argmax(dq, dim=-1).to(torch.int32)
        del t, d
    u_accept = torch.rand((B, K), generator=gen, device=device, dtype=torch.float32)
    u_bonus = torch.rand((B,), generator=gen, device=device, dtype=torch.float32)
    return dict(target=target, draft=draft, draft_tokens=tokens, u_accept=u_accept,
                u_bonus=u_bonus, temperature=float(temperature))


def make_tree(number: int = 4, device="cpu", B: int | None = None, V: int | None = None,
              seed: int | None = None, n_nodes: int | None = None):
    """Inputs of the Medusa tree workload.

    The tree is the greedy sparse tree of ``medusa_tree.build_sparse_tree``
    (root + n_nodes-1 candidates).  For every sequence and every node with
    children, one "correct" rank r is drawn with P(r = i) = a_k^(i) (k = depth
    of the children), else none; the child of rank r, if the tree holds it,
    carries argmax(target row of the parent), and its siblings carry distinct
    random tokens different from that argmax.
    Returns dict(target [B,N,V], parents [N] int32, node_tokens [B,N] int32,
    max_depth, tree) on ``device``.
    """
    w = WORKLOADS[number]
    B = w.B if B is None else B
    V = w.V if V is None else V
    n_nodes = w.N if n_nodes is None else n_nodes
    device = torch.device(device)
    tree = medusa_tree.build_sparse_tree(w.K, 8, n_nodes, medusa_tree.synthetic_accuracy)
    N = len(tree.parents)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    target = 3.0 * torch.randn((B, N, V), generator=gen, device=device)
    target = target.to(w.torch_dtype)
    am = torch.argmax(target.float(), dim=-1).cpu().numpy()      # [B, N]
    # host-side draws for the tokens (small), from a numpy generator seeded alike
    rng = np.random.default_rng((w.seed if seed is None else seed) + 7919)
    tokens = np.zeros((B, N), dtype=np.int32)
    children = tree.children()
    if max(len(ch) for ch in children) + 1 > V:
        raise ValueError("V = %d is too small for distinct sibling tokens (fan-out %d)"
                         % (V, max(len(ch) for ch in children)))
    for n in range(N):
        ch = children[n]
        if not ch:
            continue
        k = tree.depth[n] + 1
        cum = np.cumsum([medusa_tree.synthetic_accuracy(k, i) for i in range(1, 9)])
        u = rng.random(B)
        r = np.where(u < cum[-1], np.searchsorted(cum, u, side="right") + 1, 0)
        for b in range(B):
            want = int(am[b, n])
            used = {want}
            for c in ch:
                if tree.rank[c] == r[b]:
                    tokens[b, c] = want
                else:
                    t = int(rng.integers(0, V))
                    while t in used:
                        t = int(rng.integers(0, V))
                    used.add(t)
                    tokens[b, c] = t
    return dict(target=target, parents=torch.tensor(tree.parents, dtype=torch.int32, device=device),
                node_tokens=torch.from_numpy(tokens).to(device), max_depth=max(tree.depth), tree=tree)
