"""Pins for the oracle's merged embedding lookup and merged LM head (CPU only).

Optimized Parler TTS, "Analysis and improvements", other optimizations: the LM
head evaluated on the last position only, the nine codebook heads merged into
one weight matrix, and the nine embedding lookups merged into one.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_self_gb300 import workloads as W


def bits_of(x):
    return W.bits(torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16))


def vals(b):
    return torch.from_numpy(b.astype(np.int16)).view(torch.bfloat16).double().numpy()


def test_embedding_of_one_hot_tables():
    # Table rows are one-hot in d: the sum marks exactly which rows were gathered.
    C, V, Dm = 3, 5, 15
    tab = np.zeros((C * V, Dm), np.float32)
    for r in range(C * V):
        tab[r, r] = 1.0
    tokens = np.array([[0, 4, 2], [1, 1, 1]], np.int32)
    out = oracle.embed_tokens(tokens, bits_of(tab), V)
    expect = np.zeros((2, Dm))
    for b in range(2):
        for c in range(C):
            expect[b, c * V + tokens[b, c]] += 1.0
    assert np.array_equal(out, expect)


def test_embedding_matches_numpy_gather_sum():
    rng = np.random.default_rng(1)
    C, V, Dm, B = 9, 1088, 64, 4
    tab = bits_of(rng.normal(size=(C * V, Dm)))
    tokens = rng.integers(0, V, size=(B, C)).astype(np.int32)
    out = oracle.embed_tokens(tokens, tab, V)
    tv = vals(tab)
    ref = np.stack([sum(tv[c * V + tokens[b, c]] for c in range(C)) for b in range(B)])
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # codebook offsets matter: the same token id in two codebooks picks two different rows
    t2 = np.zeros((1, C), np.int32)
    o2 = oracle.embed_tokens(t2, tab, V)
    assert np.abs(o2[0] - C * tv[0]).max() > 1e-3


def test_embedding_rejects_out_of_range_tokens():
    tab = bits_of(np.zeros((2 * 4, 8)))
    with pytest.raises(ValueError):
        oracle.embed_tokens(np.array([[0, 4]], np.int32), tab, 4)
    with pytest.raises(ValueError):
        oracle.embed_tokens(np.array([[-1, 0]], np.int32), tab, 4)


def test_lm_head_matches_float64_matmul():
    rng = np.random.default_rng(2)
    B, K, N = 3, 96, 40
    h, w = bits_of(rng.normal(size=(B, K))), bits_of(rng.normal(size=(N, K)) * 0.05)
    out = oracle.lm_head(h, w)
    np.testing.assert_allclose(out, vals(h) @ vals(w).T, rtol=1e-13, atol=1e-13)


def test_lm_head_unit_rows_select_hidden_entries():
    rng = np.random.default_rng(3)
    B, K = 2, 32
    h = bits_of(rng.normal(size=(B, K)))
    Wm = np.zeros((K, K), np.float32)
    perm = rng.permutation(K)
    Wm[np.arange(K), perm] = 1.0                      # row n picks hidden[:, perm[n]]
    out = oracle.lm_head(h, bits_of(Wm))
    assert np.array_equal(out, vals(h)[:, perm])
    # a transposed weight (W[k][n] instead of W[n][k]) gives the inverse permutation instead
    out_t = oracle.lm_head(h, bits_of(Wm.T.copy()))
    assert not np.array_equal(out_t, out)
