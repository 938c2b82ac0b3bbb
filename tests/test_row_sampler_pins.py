"""Pins of the oracle's one-token-per-row sampler.

The draft side chooses its next draft token from its own logits ("Beschleunigung
von Sonar durch Spekulation", section "Ziel-Entwurf": the draft proposes tokens
that the target then scores; the cited "Fast Inference from Transformers via
Speculative Decoding" draws each draft token from the draft's distribution q).
A draw from softmax(l / T) by inverse CDF with the row's uniform, or the
argmax (lowest index) in greedy mode.

The pins fix it against what the mathematics fixes:
  - over a fine grid of uniforms, each token is drawn with frequency equal to
    its temperature-softmax probability;
  - T == 0 is numpy's argmax (first maximum);
  - dividing the temperature by two equals doubling the logits (both exact
    in binary floating point), so the draws agree at every uniform;
  - bf16 rows decode to the fp32 values they represent.
"""
import numpy as np
import pytest

import oracle


def _softmax64(row, T):
    x = row.astype(np.float64) / T
    e = np.exp(x - x.max())
    return e / e.sum()


def check_frequencies(lib, V=6, T=0.8, M=24000, seed=11):
    rng = np.random.default_rng(seed)
    row = (rng.standard_normal(V) * 2.0).astype(np.float32)
    logits = np.broadcast_to(row, (M, V)).copy()
    u = ((np.arange(M) + 0.5) / M).astype(np.float32)
    r = oracle.sample_rows(logits, u, T, lib=lib)
    counts = np.bincount(r["tokens"], minlength=V)
    p = _softmax64(row, T)
    assert np.all(np.abs(counts / M - p) <= 1.0 / M + 1e-6), (counts / M, p)


def check_greedy_is_argmax(lib, seed=12):
    rng = np.random.default_rng(seed)
    logits = rng.integers(-3, 4, (300, 17)).astype(np.float32)     # many ties
    r = oracle.sample_rows(logits, None, 0.0, lib=lib)
    np.testing.assert_array_equal(r["tokens"], logits.argmax(-1))


def check_temperature_scaling(lib, seed=13):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((500, 40)).astype(np.float32)
    u = rng.random(500).astype(np.float32)
    a = oracle.sample_rows(logits, u, 0.5, lib=lib)
    b = oracle.sample_rows(2.0 * logits, u, 1.0, lib=lib)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    c = oracle.sample_rows(logits, u, 1.0, lib=lib)
    assert (a["tokens"] != c["tokens"]).any()      # the temperature matters


def test_frequencies_follow_softmax(oracle_lib):
    check_frequencies(oracle_lib)


@pytest.mark.parametrize("V,T", [(3, 0.3), (9, 2.5)])
def test_frequencies_other_shapes(oracle_lib, V, T):
    check_frequencies(oracle_lib, V=V, T=T, M=9000, seed=V)


def test_greedy_is_argmax(oracle_lib):
    check_greedy_is_argmax(oracle_lib)


def test_temperature_scaling(oracle_lib):
    check_temperature_scaling(oracle_lib)


def test_bf16_rows_decode_to_their_values(oracle_lib):
    rng = np.random.default_rng(14)
    f = rng.standard_normal((200, 33)).astype(np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)             # truncate to bf16
    exact = (bits.astype(np.uint32) << 16).view(np.float32)
    u = rng.random(200).astype(np.float32)
    a = oracle.sample_rows(bits, u, 0.7, lib=oracle_lib)
    b = oracle.sample_rows(exact, u, 0.7, lib=oracle_lib)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])


def test_cdf_brackets_the_uniform(oracle_lib):
    rng = np.random.default_rng(15)
    logits = rng.standard_normal((100, 50)).astype(np.float32)
    u = rng.random(100).astype(np.float32)
    r = oracle.sample_rows(logits, u, 1.2, lib=oracle_lib)
    assert np.all(r["cdf"][:, 0] <= u) and np.all(u < r["cdf"][:, 1])
