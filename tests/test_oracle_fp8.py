"""Pins for the oracle's FP8 E4M3 KV cache (CPU only).

E4M3 per the OCP 8-bit floating point specification: the decode table is
checked against the format's defining values, the encoder against its
definition (nearest value, ties to the even code, saturation to 448), and the
fp8-cache attention against the bf16 oracle on values E4M3 holds exactly.
"""
import math

import numpy as np
import torch

import oracle
from decode_attention_self_gb300 import workloads as W


def test_e4m3_decode_defining_values():
    assert oracle.e4m3_to_double(0x00) == 0.0
    assert oracle.e4m3_to_double(0x80) == 0.0 and math.copysign(1, oracle.e4m3_to_double(0x80)) == -1
    assert oracle.e4m3_to_double(0x38) == 1.0            # exponent 7 = bias
    assert oracle.e4m3_to_double(0x7E) == 448.0          # largest finite
    assert oracle.e4m3_to_double(0xFE) == -448.0
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_to_double(0x07) == 7 * 2.0 ** -9  # largest subnormal
    assert math.isnan(oracle.e4m3_to_double(0x7F)) and math.isnan(oracle.e4m3_to_double(0xFF))
    vals = [oracle.e4m3_to_double(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))     # codes 0..126 increase strictly


def test_e4m3_encode_round_trip_ties_and_saturation():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.double_to_e4m3(oracle.e4m3_to_double(c)) == c
    # halfway between 1.0 (0x38, even) and 1.125 (0x39, odd) -> even
    assert oracle.double_to_e4m3(1.0625) == 0x38
    # halfway between 1.125 (0x39) and 1.25 (0x3A) -> 0x3A (even)
    assert oracle.double_to_e4m3(1.1875) == 0x3A
    assert oracle.double_to_e4m3(1.0625 + 1e-9) == 0x39
    assert oracle.double_to_e4m3(447.9) == 0x7E and oracle.double_to_e4m3(1e6) == 0x7E
    assert oracle.double_to_e4m3(-1e6) == 0xFE
    assert oracle.double_to_e4m3(2.0 ** -10) == 0x00          # tie between 0 and the smallest subnormal
    assert oracle.double_to_e4m3(2.0 ** -10 * 1.01) == 0x01
    assert oracle.double_to_e4m3(float("nan")) == 0x7F
    assert oracle.double_to_e4m3(-0.0) == 0x80


def _exact_e4m3_values(rng, shape):
    codes = rng.integers(0, 0x7E, size=shape).astype(np.uint8) | (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)
    return codes, np.vectorize(oracle.e4m3_to_double)(codes)


def test_fp8_attention_equals_bf16_attention_on_exact_values():
    # Values that both bf16 and e4m3 hold exactly: the two oracles must agree to rounding.
    rng = np.random.default_rng(0)
    B, H, L, D = 2, 3, 40, 64
    kc, kf = _exact_e4m3_values(rng, (B, H, L, D))
    vc, vf = _exact_e4m3_values(rng, (B, H, L, D))
    # e4m3 values have at most 4 significant bits, so bf16 (8 bits) holds them exactly
    q = W.bits(torch.randn((B, H, D), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16))
    lens = np.array([40, 7], np.int32)
    ks, vs = 0.5, 0.25                                          # powers of two: scaling stays exact
    a = oracle.attn_fp8_contiguous(q, kc, vc, lens, 0.125 / 16, ks, vs)
    kb2 = W.bits(torch.from_numpy(kf * ks).float().to(torch.bfloat16))
    vb2 = W.bits(torch.from_numpy(vf * vs).float().to(torch.bfloat16))
    b = oracle.attn_contiguous(q, kb2, vb2, lens, 0.125 / 16)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_fp8_append_quantizes_with_division_then_rounding():
    rng = np.random.default_rng(2)
    B, H, D, cap = 2, 2, 64, 8
    kn = W.bits(torch.randn((B, H, D), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16))
    vn = W.bits(torch.randn((B, H, D), generator=torch.Generator().manual_seed(4)).to(torch.bfloat16))
    k = np.zeros((B, H, cap, D), np.uint8)
    v = np.zeros((B, H, cap, D), np.uint8)
    pos = np.array([0, 5], np.int32)
    ks, vs = 0.02, 0.03
    oracle.kv_append_fp8_contiguous(k, v, kn, vn, pos, ks, vs)
    kf = torch.from_numpy(kn.astype(np.int16)).view(torch.bfloat16).float().numpy()
    for b in range(B):
        for h in range(H):
            for e in range(D):
                x = np.float32(kf[b, h, e]) / np.float32(ks)   # binary32 division
                assert k[b, h, pos[b], e] == oracle.double_to_e4m3(float(x))
    # dequantised values are within half an e4m3 step (relative 2^-4) of the scaled inputs, or saturated
    deq = np.vectorize(oracle.e4m3_to_double)(k[np.arange(B), :, pos]) * ks
    np.testing.assert_allclose(deq, kf, rtol=2 ** -4, atol=2 ** -10 * ks)


def test_fp8_paged_equals_contiguous():
    rng = np.random.default_rng(5)
    B, H, D = 2, 2, 64
    lens = np.array([20, 33], np.int32)
    kc, _ = _exact_e4m3_values(rng, (B, H, 48, D))
    vc, _ = _exact_e4m3_values(rng, (B, H, 48, D))
    q = W.bits(torch.randn((B, H, D), generator=torch.Generator().manual_seed(6)).to(torch.bfloat16))
    NB = 8
    perm = rng.permutation(NB)
    table = np.full((B, 3), -1, np.int32)
    kp = np.zeros((NB, H, 16, D), np.uint8)
    vp = np.zeros((NB, H, 16, D), np.uint8)
    i = 0
    for b in range(B):
        for j in range(3):
            table[b, j] = perm[i]
            kp[perm[i]] = kc[b, :, 16 * j:16 * j + 16]
            vp[perm[i]] = vc[b, :, 16 * j:16 * j + 16]
            i += 1
    a = oracle.attn_fp8_contiguous(q, kc, vc, lens, 0.125, 0.1, 0.2)
    b_ = oracle.attn_fp8_paged(q, kp, vp, table, lens, 0.125, 0.1, 0.2)
    assert np.array_equal(a, b_)


def test_fp8_paged_append_writes_the_contiguous_codes_at_the_logical_slot():
    # The paged append must write, at block table[b][pos/16], slot pos % 16, the same codes the (pinned)
    # contiguous append writes at position pos, and leave every other slot of the pool untouched.
    rng = np.random.default_rng(7)
    B, H, D, bs, NB = 3, 2, 64, 16, 7
    kn = W.bits(torch.randn((B, H, D), generator=torch.Generator().manual_seed(8)).to(torch.bfloat16))
    vn = W.bits(torch.randn((B, H, D), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16))
    pos = np.array([0, 17, 31], np.int32)
    table = rng.permutation(NB)[:B * 2].reshape(B, 2).astype(np.int32)
    kp = rng.integers(0, 0x7F, size=(NB, H, bs, D), dtype=np.uint8)
    vp = rng.integers(0, 0x7F, size=(NB, H, bs, D), dtype=np.uint8)
    kp0, vp0 = kp.copy(), vp.copy()
    ks, vs = 0.05, 0.07
    oracle.kv_append_fp8_paged(kp, vp, table, kn, vn, pos, ks, vs)
    kc = np.zeros((B, H, 32, D), np.uint8)
    vc = np.zeros((B, H, 32, D), np.uint8)
    oracle.kv_append_fp8_contiguous(kc, vc, kn, vn, pos, ks, vs)
    written = np.zeros((NB, bs), bool)
    for b in range(B):
        blk, slot = table[b, pos[b] // bs], pos[b] % bs
        assert np.array_equal(kp[blk, :, slot], kc[b, :, pos[b]])
        assert np.array_equal(vp[blk, :, slot], vc[b, :, pos[b]])
        written[blk, slot] = True
    untouched = ~written
    assert np.array_equal(kp.transpose(0, 2, 1, 3)[untouched], kp0.transpose(0, 2, 1, 3)[untouched])
    assert np.array_equal(vp.transpose(0, 2, 1, 3)[untouched], vp0.transpose(0, 2, 1, 3)[untouched])
