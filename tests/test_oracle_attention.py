"""Pins for the oracle's attention and KV append (CPU only, no GPU).

Each check is fixed by mathematics or by a library routine the oracle does not
call, chosen so that a dropped scale, a wrong softmax axis, a transposed
operand, an off-by-one in the valid length or a wrong paged address fails at
least one of them.

Definition pinned (Optimized Parler TTS, "Analysis and improvements": static
caches for causal and cross attention, the kernel reading the valid length
only): o = sum_j softmax_j(scale * q.k_j) v_j over the valid keys j < L.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_attention_self_gb300 import workloads as W

D = 64
SCALE = 1.0 / math.sqrt(D)


def bf16_bits(x) -> np.ndarray:
    return W.bits(torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16))


def bf16_vals(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(b.astype(np.int16)).view(torch.bfloat16).float().double().numpy()


def rand_bits(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return W.bits(torch.randn(shape, generator=g).to(torch.bfloat16))


def test_bf16_decode_exact():
    # bf16 -> binary32 is exact: 1.0 = 0x3F80, -2.5 = 0xC020, smallest normal 2^-126 = 0x0080.
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC020) == -2.5
    assert oracle.bf16_to_double(0x0080) == 2.0 ** -126
    assert math.isnan(oracle.bf16_to_double(W.BF16_NAN_BITS))


def test_uniform_keys_give_mean_of_values():
    # All keys equal -> all scores equal -> p_j = 1/L -> o = mean of the valid values.
    L = 37
    q = rand_bits((D,), 1)
    k = np.tile(rand_bits((1, D), 2), (L, 1))
    v = rand_bits((L, D), 3)
    out, psum = oracle.attend(q, k, v, SCALE)
    np.testing.assert_allclose(out, bf16_vals(v).mean(axis=0), rtol=0, atol=1e-12)
    assert abs(psum - 1.0) < 1e-12


def test_zero_scale_gives_mean_of_values():
    L = 50
    q, k, v = rand_bits((D,), 4), rand_bits((L, D), 5), rand_bits((L, D), 6)
    out, _ = oracle.attend(q, k, v, 0.0)
    np.testing.assert_allclose(out, bf16_vals(v).mean(axis=0), rtol=0, atol=1e-12)


def test_single_key_returns_its_value_exactly():
    q, k, v = rand_bits((D,), 7), rand_bits((1, D), 8), rand_bits((1, D), 9)
    out, psum = oracle.attend(q, k, v, SCALE)
    assert np.array_equal(out, bf16_vals(v)[0])
    assert psum == 1.0


def test_dominant_key_selects_its_value():
    # q = 8 e_0; key 5 = 8 e_0 (score 64*scale*... = 8), others 0 -> weight of key 5 = 1/(1+(L-1)e^-8)
    L = 12
    qv = np.zeros(D, np.float32); qv[0] = 8.0
    kv = np.zeros((L, D), np.float32); kv[5, 0] = 8.0
    v = rand_bits((L, D), 10)
    out, _ = oracle.attend(bf16_bits(qv), bf16_bits(kv), v, SCALE)
    s = 8.0 * 8.0 * SCALE
    w5 = 1.0 / (1.0 + (L - 1) * math.exp(-s))
    vv = bf16_vals(v)
    expect = w5 * vv[5] + (1 - w5) * (vv.sum(axis=0) - vv[5]) / (L - 1)
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-12)


def test_two_keys_logistic_closed_form():
    # Two keys: p_0 = sigmoid(s_0 - s_1).
    q, k, v = rand_bits((D,), 11), rand_bits((2, D), 12), rand_bits((2, D), 13)
    qf, kf, vf = bf16_vals(q), bf16_vals(k), bf16_vals(v)
    s0, s1 = SCALE * float(qf @ kf[0]), SCALE * float(qf @ kf[1])
    p0 = 0.5 * (1.0 + math.tanh((s0 - s1) / 2.0))
    out, _ = oracle.attend(q, k, v, SCALE)
    np.testing.assert_allclose(out, p0 * vf[0] + (1 - p0) * vf[1], rtol=0, atol=1e-12)


@pytest.mark.parametrize("L", [1, 5, 64, 333])
def test_matches_torch_sdpa_float64(L):
    # Library cross-check: torch's scaled_dot_product_attention in float64 on the CPU.
    q, k, v = rand_bits((D,), 20 + L), rand_bits((L, D), 30 + L), rand_bits((L, D), 40 + L)
    out, psum = oracle.attend(q, k, v, SCALE)
    qt, kt, vt = (torch.from_numpy(bf16_vals(a)) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qt.view(1, 1, 1, D), kt.view(1, 1, L, D),
                                                           vt.view(1, 1, L, D), scale=SCALE).view(D).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    assert abs(psum - 1.0) < 1e-12


def test_scale_matters_against_sdpa_default():
    # The default scale is 1/sqrt(D); SDPA's default is the same, a different scale is not.
    L = 40
    q, k, v = rand_bits((D,), 50), rand_bits((L, D), 51), rand_bits((L, D), 52)
    qt, kt, vt = (torch.from_numpy(bf16_vals(a)) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qt.view(1, 1, 1, D), kt.view(1, 1, L, D),
                                                           vt.view(1, 1, L, D)).view(D).numpy()
    out, _ = oracle.attend(q, k, v, oracle.default_scale(D))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    out2, _ = oracle.attend(q, k, v, 1.0)
    assert np.abs(out2 - ref).max() > 1e-3


def test_contiguous_reads_only_valid_length():
    # NaN past seq_len: any read beyond the valid range would make the output NaN.
    w = W.make_workload(1)
    cache = W.make_self_cache(w, 0, filled_len=w.seq_len)
    q = W.bits(W.make_step_inputs(w, 0)[0])
    out = oracle.attn_contiguous(q, W.bits(cache.k), W.bits(cache.v), w.seq_len, SCALE)
    assert np.isfinite(out).all()
    L = int(w.seq_len[0])
    qt = torch.from_numpy(bf16_vals(q)).view(1, 16, 1, D)
    kt = torch.from_numpy(bf16_vals(W.bits(cache.k)[:, :, :L]))
    vt = torch.from_numpy(bf16_vals(W.bits(cache.v)[:, :, :L]))
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=SCALE).view(1, 16, D).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_paged_equals_contiguous_with_shuffled_table():
    # The same logical sequences laid out contiguously and in a shuffled block pool give the same output.
    B, H, bs = 3, 4, 16
    lens = np.array([1, 17, 50], np.int32)
    mb = 4
    g = torch.Generator().manual_seed(60)
    kc = torch.randn((B, H, mb * bs, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, H, mb * bs, D), generator=g).to(torch.bfloat16)
    q = torch.randn((B, H, D), generator=g).to(torch.bfloat16)
    for b in range(B):
        kc[b, :, lens[b]:] = float("nan")
        vc[b, :, lens[b]:] = float("nan")
    nblk = (lens + bs - 1) // bs
    NB = int(nblk.sum()) + 3
    perm = np.random.default_rng(61).permutation(NB)
    table = np.full((B, mb), -1, np.int32)
    kp = torch.full((NB, H, bs, D), float("nan"), dtype=torch.bfloat16)
    vp = kp.clone()
    off = 0
    for b in range(B):
        for j in range(nblk[b]):
            blk = int(perm[off]); off += 1
            table[b, j] = blk
            kp[blk] = kc[b, :, j * bs:(j + 1) * bs]
            vp[blk] = vc[b, :, j * bs:(j + 1) * bs]
    oc = oracle.attn_contiguous(W.bits(q), W.bits(kc), W.bits(vc), lens, SCALE)
    op = oracle.attn_paged(W.bits(q), W.bits(kp), W.bits(vp), table, lens, SCALE)
    assert np.array_equal(oc, op)
    # swapping two full blocks of a row only permutes (k, v) pairs: invariant up to rounding
    sw = table.copy(); sw[2, [0, 1]] = sw[2, [1, 0]]
    osw = oracle.attn_paged(W.bits(q), W.bits(kp), W.bits(vp), sw, lens, SCALE)
    np.testing.assert_allclose(osw[2], oc[2], rtol=0, atol=1e-12)
    # swapping a full block with the partial last block reads unfilled (NaN) slots
    bad = table.copy(); bad[2, [0, 3]] = bad[2, [3, 0]]
    ob = oracle.attn_paged(W.bits(q), W.bits(kp), W.bits(vp), bad, lens, SCALE)
    assert np.isnan(ob[2]).all()
    assert np.array_equal(ob[:2], oc[:2])


def test_permutation_of_key_value_pairs_is_invariant():
    L = 29
    q, k, v = rand_bits((D,), 70), rand_bits((L, D), 71), rand_bits((L, D), 72)
    perm = np.random.default_rng(73).permutation(L)
    a, _ = oracle.attend(q, k, v, SCALE)
    b, _ = oracle.attend(q, k[perm].copy(), v[perm].copy(), SCALE)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    # permuting keys alone (a transposed / mismatched pairing) does change it
    c, _ = oracle.attend(q, k[perm].copy(), v, SCALE)
    assert np.abs(a - c).max() > 1e-4


def test_paged_rejects_table_entry_outside_pool():
    q = rand_bits((1, 1, D), 80)
    kp = rand_bits((2, 1, 16, D), 81)
    with pytest.raises(ValueError):
        oracle.attn_paged(q, kp, kp, np.array([[5]], np.int32), np.array([3], np.int32), SCALE)


def test_append_contiguous_round_trip():
    B, H, cap = 2, 3, 8
    k = rand_bits((B, H, cap, D), 90); v = rand_bits((B, H, cap, D), 91)
    k0, v0 = k.copy(), v.copy()
    kn, vn = rand_bits((B, H, D), 92), rand_bits((B, H, D), 93)
    pos = np.array([0, 7], np.int32)
    oracle.kv_append_contiguous(k, v, kn, vn, pos)
    for b in range(B):
        assert np.array_equal(k[b, :, pos[b]], kn[b]) and np.array_equal(v[b, :, pos[b]], vn[b])
        mask = np.ones(cap, bool); mask[pos[b]] = False
        assert np.array_equal(k[b][:, mask], k0[b][:, mask]) and np.array_equal(v[b][:, mask], v0[b][:, mask])


def test_append_paged_round_trip():
    B, H, NB = 2, 3, 5
    kp = rand_bits((NB, H, 16, D), 94); vp = rand_bits((NB, H, 16, D), 95)
    k0 = kp.copy()
    table = np.array([[3, 1], [4, -1]], np.int32)
    kn, vn = rand_bits((B, H, D), 96), rand_bits((B, H, D), 97)
    pos = np.array([19, 0], np.int32)
    oracle.kv_append_paged(kp, vp, table, kn, vn, pos)
    assert np.array_equal(kp[1, :, 3], kn[0]) and np.array_equal(vp[1, :, 3], vn[0])
    assert np.array_equal(kp[4, :, 0], kn[1]) and np.array_equal(vp[4, :, 0], vn[1])
    diff = (kp != k0).any(axis=(1, 3))
    assert set(map(tuple, np.argwhere(diff))) == {(1, 3), (4, 0)}


def test_append_then_attend_sees_new_key():
    # Causal decode reading: the query attends every valid key including the one appended this step.
    w = W.make_workload(1)
    cache = W.make_self_cache(w, 0)                 # slot L-1 holds NaN until the append
    q, _, kn, vn = W.make_step_inputs(w, 0)
    k, v = W.bits(cache.k).copy(), W.bits(cache.v).copy()
    pos = w.seq_len - 1
    before = oracle.attn_contiguous(W.bits(q), k, v, w.seq_len, SCALE)
    assert np.isnan(before).all()
    oracle.kv_append_contiguous(k, v, W.bits(kn), W.bits(vn), pos)
    after = oracle.attn_contiguous(W.bits(q), k, v, w.seq_len, SCALE)
    assert np.isfinite(after).all()


def test_row_entry_points_equal_the_batch_ones():
    # The per-row oracle calls (used for sampled checks at full size) must give, row by row, exactly what
    # the pinned batch calls give.
    rng = np.random.default_rng(31)
    B, H, D, cap = 3, 2, 64, 40
    lens = np.array([1, 17, 40], np.int32)
    gen = torch.Generator().manual_seed(32)
    q = W.bits(torch.randn((B, H, D), generator=gen).to(torch.bfloat16))
    k = W.bits(torch.randn((B, H, cap, D), generator=gen).to(torch.bfloat16))
    v = W.bits(torch.randn((B, H, cap, D), generator=gen).to(torch.bfloat16))
    batch = oracle.attn_contiguous(q, k, v, lens, 0.125)
    for b in range(B):
        for h in range(H):
            row = oracle.attn_contiguous_row(q[b, h], np.ascontiguousarray(k[b, h]), np.ascontiguousarray(v[b, h]),
                                             int(lens[b]), 0.125)
            assert np.array_equal(row, batch[b, h])
    NB = 9
    table = rng.permutation(NB)[:B * 3].reshape(B, 3).astype(np.int32)
    kp = W.bits(torch.randn((NB, H, 16, D), generator=gen).to(torch.bfloat16))
    vp = W.bits(torch.randn((NB, H, 16, D), generator=gen).to(torch.bfloat16))
    pbatch = oracle.attn_paged(q, kp, vp, table, lens, 0.125)
    for b in range(B):
        for h in range(H):
            row = oracle.attn_paged_row(q[b, h], kp, vp, table[b], h, int(lens[b]), 0.125)
            assert np.array_equal(row, pbatch[b, h])
