"""Parity rules between the GPU library's outputs and the oracle's.

TEST INFRASTRUCTURE ONLY (used by tests/, the smoke check and nothing else).

Integer outputs -- accepted lengths, emitted tokens, tree paths -- must be
equal, with one allowance for sampling mode: where the oracle's float64 value
and the GPU's fp32 value sit on opposite sides of a decision because the
uniform lies within NEAR_TIE of it, the case is counted as a near tie and the
rest of that sequence is not compared.  The two decisions are
  * acceptance: |u_i - min(1, p_i/q_i)| < NEAR_TIE at the first position where
    GPU and oracle disagree;
  * inverse CDF: |u_b - C/W| < NEAR_TIE at either end of the oracle's chosen
    token's cumulative interval.
Probabilities p_i(x_i), q_i(x_i), min(1, ratio) must agree within PROB_ATOL.
"""
from __future__ import annotations

import dataclasses

import numpy as np

NEAR_TIE = 1e-6
PROB_ATOL = 1e-5

# Every report made in this process, with the label the caller set (the test
# session prints them, so near ties are reported, not only counted).
LOG = []
LABEL = [""]


def _logged(rep, kind):
    LOG.append((LABEL[0], kind, rep))
    return rep


@dataclasses.dataclass
class ParityReport:
    sequences: int = 0
    exact: int = 0
    accept_ties: int = 0
    bonus_ties: int = 0
    max_prob_err: float = 0.0
    failures: list = dataclasses.field(default_factory=list)

    @property
    def ok(self) -> bool:
        return not self.failures

    def summary(self) -> str:
        return ("%d sequences: %d exact, %d acceptance near-ties, %d inverse-CDF near-ties, "
                "max |prob err| %.2e, %d failures" % (self.sequences, self.exact, self.accept_ties,
                                                      self.bonus_ties, self.max_prob_err, len(self.failures)))


def compare_linear(gpu: dict, ora: dict, u_accept, u_bonus, temperature: float, check_probs=True) -> ParityReport:
    """gpu: numpy arrays accept_len, out_tokens, num_emitted (and probs); ora: oracle.verify_linear output."""
    rep = ParityReport()
    B = len(ora["accept_len"])
    rep.sequences = B
    K = ora["out_tokens"].shape[1] - 1
    u_accept = None if u_accept is None else np.asarray(u_accept, np.float64).reshape(B, K)
    u_bonus = None if u_bonus is None else np.asarray(u_bonus, np.float64).reshape(B)
    if temperature > 0 and check_probs and "probs" in gpu and K > 0:
        err = np.abs(gpu["probs"].astype(np.float64) - ora["probs"])
        rep.max_prob_err = float(err.max())
        bad = np.argwhere(err > PROB_ATOL)
        for b, i, k in bad[:10]:
            rep.failures.append("b=%d i=%d %s: gpu %.9g oracle %.9g" % (
                b, i, ("p", "q", "thr")[k], gpu["probs"][b, i, k], ora["probs"][b, i, k]))
    for b in range(B):
        jg, jo = int(gpu["accept_len"][b]), int(ora["accept_len"][b])
        if temperature == 0:
            same = (jg == jo and np.array_equal(gpu["out_tokens"][b], ora["out_tokens"][b])
                    and gpu["num_emitted"][b] == ora["num_emitted"][b])
            if same:
                rep.exact += 1
            else:
                rep.failures.append("b=%d greedy: gpu j=%d %s, oracle j=%d %s" % (
                    b, jg, list(gpu["out_tokens"][b]), jo, list(ora["out_tokens"][b])))
            continue
        if jg != jo:
            i = min(jg, jo)          # first position where the decisions differ
            thr = ora["probs"][b, i, 2]
            if abs(u_accept[b, i] - thr) < NEAR_TIE:
                rep.accept_ties += 1
            else:
                rep.failures.append("b=%d: gpu j=%d oracle j=%d, u=%.9g thr=%.9g" % (b, jg, jo, u_accept[b, i], thr))
            continue
        if gpu["num_emitted"][b] != ora["num_emitted"][b]:
            rep.failures.append("b=%d num_emitted %d vs %d" % (b, gpu["num_emitted"][b], ora["num_emitted"][b]))
            continue
        if np.array_equal(gpu["out_tokens"][b], ora["out_tokens"][b]):
            rep.exact += 1
            continue
        if not np.array_equal(gpu["out_tokens"][b, :jo], ora["out_tokens"][b, :jo]) or \
                not np.array_equal(gpu["out_tokens"][b, jo + 1:], ora["out_tokens"][b, jo + 1:]):
            rep.failures.append("b=%d tokens differ outside the extra token" % b)
            continue
        lo, hi = ora["bonus_cdf"][b]
        if u_bonus is not None and (abs(u_bonus[b] - lo) < NEAR_TIE or abs(u_bonus[b] - hi) < NEAR_TIE):
            rep.bonus_ties += 1
        else:
            rep.failures.append("b=%d extra token gpu %d oracle %d (u_b=%.9g, interval [%.9g, %.9g))" % (
                b, gpu["out_tokens"][b, jo], ora["out_tokens"][b, jo], u_bonus[b], lo, hi))
    return _logged(rep, "linear")


def compare_bonus(gpu_tokens, ora: dict, u_bonus, temperature: float) -> ParityReport:
    rep = ParityReport()
    gpu_tokens = np.asarray(gpu_tokens)
    rep.sequences = len(gpu_tokens)
    for b, g in enumerate(gpu_tokens):
        o = ora["bonus_token"][b]
        if g == o:
            rep.exact += 1
        elif temperature > 0 and (abs(u_bonus[b] - ora["bonus_cdf"][b, 0]) < NEAR_TIE
                                  or abs(u_bonus[b] - ora["bonus_cdf"][b, 1]) < NEAR_TIE):
            rep.bonus_ties += 1
        else:
            rep.failures.append("b=%d extra token gpu %d oracle %d" % (b, g, o))
    return _logged(rep, "extra token")


def compare_tree(gpu: dict, ora: dict) -> ParityReport:
    rep = ParityReport()
    B = len(ora["path_len"])
    rep.sequences = B
    for b in range(B):
        if (gpu["path_len"][b] == ora["path_len"][b] and np.array_equal(gpu["path_nodes"][b], ora["path_nodes"][b])
                and np.array_equal(gpu["out_tokens"][b], ora["out_tokens"][b])):
            rep.exact += 1
        else:
            rep.failures.append("b=%d tree: gpu len %d nodes %s tokens %s; oracle len %d nodes %s tokens %s" % (
                b, gpu["path_len"][b], list(gpu["path_nodes"][b]), list(gpu["out_tokens"][b]),
                ora["path_len"][b], list(ora["path_nodes"][b]), list(ora["out_tokens"][b])))
    return _logged(rep, "tree")


def _diverging_node(gp, op, tokens_equal_on_path):
    """The node whose draw decided where two sampled walks part: the last node the
    two root paths share (if the paths differ), else the last node (if only the
    extra token, the draw at the last node, differs)."""
    common = 0
    while common < min(len(gp), len(op)) and gp[common] == op[common]:
        common += 1
    if len(gp) == len(op) == common and tokens_equal_on_path:
        return gp[-1]
    return gp[common - 1] if common > 0 else 0


def compare_tree_sample(gpu: dict, ora: dict, u_nodes) -> ParityReport:
    """Sampled tree walk: paths and tokens equal, except where the walks part at a
    node whose uniform lies within NEAR_TIE of an end of that node's draw interval
    in the oracle (counted as a tie).  Only that first diverging node is tested."""
    rep = ParityReport()
    u_nodes = np.asarray(u_nodes, np.float64)
    B = len(ora["path_len"])
    rep.sequences = B
    for b in range(B):
        if (gpu["path_len"][b] == ora["path_len"][b] and np.array_equal(gpu["path_nodes"][b], ora["path_nodes"][b])
                and np.array_equal(gpu["out_tokens"][b], ora["out_tokens"][b])):
            rep.exact += 1
            continue
        gl, ol = int(gpu["path_len"][b]), int(ora["path_len"][b])
        gp = [int(n) for n in gpu["path_nodes"][b][:gl + 1]]
        op = [int(n) for n in ora["path_nodes"][b][:ol + 1]]
        same_path_tokens = gl == ol and np.array_equal(gpu["out_tokens"][b][:gl], ora["out_tokens"][b][:ol])
        n = _diverging_node(gp, op, same_path_tokens)
        lo, hi = ora["node_cdf"][b, n]
        if min(abs(u_nodes[b, n] - lo), abs(u_nodes[b, n] - hi)) < NEAR_TIE:
            rep.bonus_ties += 1
        else:
            rep.failures.append("b=%d sampled tree: gpu len %d nodes %s tokens %s; oracle len %d nodes %s tokens %s "
                                "(walks part at node %d, u=%.9g, interval [%.9g, %.9g))" % (
                                    b, gl, gp, list(gpu["out_tokens"][b]), ol, op, list(ora["out_tokens"][b]),
                                    n, u_nodes[b, n], lo, hi))
    return _logged(rep, "sampled tree")


def compare_rows(gpu_tokens, ora: dict, u, temperature: float) -> ParityReport:
    """One token per row: equal, except a sampled token whose uniform lies within NEAR_TIE
    of either end of the oracle's interval (counted as a tie)."""
    rep = ParityReport()
    gpu_tokens = np.asarray(gpu_tokens)
    rep.sequences = len(gpu_tokens)
    for b, g in enumerate(gpu_tokens):
        o = ora["tokens"][b]
        if g == o:
            rep.exact += 1
        elif temperature > 0 and u is not None and (abs(float(u[b]) - ora["cdf"][b, 0]) < NEAR_TIE
                                                     or abs(float(u[b]) - ora["cdf"][b, 1]) < NEAR_TIE):
            rep.bonus_ties += 1
        else:
            rep.failures.append("b=%d row token gpu %d oracle %d" % (b, g, o))
    return _logged(rep, "rows")
