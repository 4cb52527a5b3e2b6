"""GPU parity at the size limits of the C ABI, against the oracle.

The decode-step calls (Optimized Parler TTS: the static and paged caches of
"Analysis and improvements" and "Future work" item 1, the fused sampler of
"Future work" item 2, the merged embedding of the other optimizations) at the
largest batch each call's grid takes (65,535 rows; 32,767 for the fused layer,
whose self and cross rows share one grid dimension), at rows of 131,072 keys
(each row cut over a full 8-CTA cluster, 1,024 keys per warp), and with 1,024
heads.  One past each batch limit is refused on the host.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_self_gb300 import workloads as W
from tests.parity import assert_attn_close, assert_probs_match, assert_tokens_match, default_scale

pytestmark = pytest.mark.gpu
D = 64


@pytest.fixture(scope="module")
def api(cuda_device):
    from decode_attention_self_gb300 import api as _api

    return _api


def workload(layout, lens, cap, H, seed, enc=None):
    B = len(lens)
    lens = np.asarray(lens, np.int32)
    enc = lens if enc is None else np.asarray(enc, np.int32)
    return W.Workload(600 + seed, "limits", 1, B, layout, lens, cap, enc, int(enc.max()), 1.0, 1, 1.0,
                      np.zeros(B, np.uint64), np.zeros(B, np.int32), H=H)


def dev_cache(api, c, dev):
    return api.KVCache(c.k.to(dev), c.v.to(dev), c.block_table.to(dev) if c.block_table is not None else None)


def oracle_self(w, c, q):
    s = default_scale(D)
    if c.layout == "contiguous":
        return oracle.attn_contiguous(W.bits(q), W.bits(c.k), W.bits(c.v), w.seq_len, s)
    return oracle.attn_paged(W.bits(q), W.bits(c.k), W.bits(c.v), c.block_table.numpy(), w.seq_len, s)


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_self_attention_at_the_batch_limit(api, cuda_device, layout):
    dev = cuda_device
    rng = np.random.default_rng(1)
    w = workload(layout, rng.integers(1, 40, size=65535, endpoint=True), 40, 1, 1)
    c = W.make_self_cache(w, 0, filled_len=w.seq_len)
    q = W.randn_bf16((w.B, 1, D), "cpu", 601, 1)
    out = torch.empty((w.B, 1, D), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_decode_self_attn(q.to(dev), dev_cache(api, c, dev), torch.from_numpy(w.seq_len).to(dev), out,
                            max_seq_len_hint=40, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(out, oracle_self(w, c, q), f"B=65535 {layout}")
    with pytest.raises(api.DrError) as e:
        api.dr_decode_self_attn(torch.zeros((65536, 1, D), dtype=torch.bfloat16, device=dev), dev_cache(api, c, dev),
                                torch.ones(65536, dtype=torch.int32, device=dev),
                                torch.empty((65536, 1, D), dtype=torch.float32, device=dev))
    assert e.value.status == api.DR_ERR_INVALID_ARG


def test_fused_layer_at_the_batch_limit(api, cuda_device):
    dev = cuda_device
    rng = np.random.default_rng(2)
    B = 32767
    w = workload("paged", rng.integers(1, 24, size=B, endpoint=True), 24, 1, 2,
                 enc=rng.integers(1, 24, size=B, endpoint=True))
    c = W.make_self_cache(w, 0)                                  # slot seq_len - 1 is written by the launch
    q, qx, kn, vn = W.make_step_inputs(w, 0)
    kx, vx = W.make_cross_kv(w, 0)
    kv = dev_cache(api, c, dev)
    out = torch.empty((B, 1, D), dtype=torch.float32, device=dev)
    outx = torch.empty_like(out)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_decode_layer(q.to(dev), kv, kn.to(dev), vn.to(dev), torch.from_numpy(w.seq_len).to(dev), qx.to(dev),
                        kx.to(dev), vx.to(dev), torch.from_numpy(w.enc_len).to(dev), out, outx, max_seq_len_hint=24,
                        err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kh, vh = W.bits(c.k).copy(), W.bits(c.v).copy()
    table = c.block_table.numpy()
    oracle.kv_append_paged(kh, vh, table, W.bits(kn), W.bits(vn), w.seq_len - 1)
    assert np.array_equal(W.bits(kv.k), kh) and np.array_equal(W.bits(kv.v), vh)
    s = default_scale(D)
    assert_attn_close(out, oracle.attn_paged(W.bits(q), kh, vh, table, w.seq_len, s), "fused self, B=32767")
    assert_attn_close(outx, oracle.attn_contiguous(W.bits(qx), W.bits(kx), W.bits(vx), w.enc_len, s),
                      "fused cross, B=32767")
    with pytest.raises(api.DrError) as e:                        # one more row than the grid takes
        z = torch.zeros((B + 1, 1, D), dtype=torch.bfloat16, device=dev)
        ones = torch.ones(B + 1, dtype=torch.int32, device=dev)
        api.dr_decode_layer(z, kv, z, z, ones, z, torch.zeros((B + 1, 1, 1, D), dtype=torch.bfloat16, device=dev),
                            torch.zeros((B + 1, 1, 1, D), dtype=torch.bfloat16, device=dev), ones,
                            torch.empty((B + 1, 1, D), dtype=torch.float32, device=dev),
                            torch.empty((B + 1, 1, D), dtype=torch.float32, device=dev))
    assert e.value.status == api.DR_ERR_INVALID_ARG


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_rows_of_131072_keys(api, cuda_device, layout):
    # 131,072 keys in 8 CTAs of 16,384 keys: 256 tiles per warp; the paged pool holds 14,506 blocks
    dev = cuda_device
    w = workload(layout, [131072, 100000], 131072, 2, 3)
    c = W.make_self_cache(w, 0, filled_len=w.seq_len)
    q = W.randn_bf16((w.B, 2, D), "cpu", 603, 1)
    out = torch.empty((w.B, 2, D), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_decode_self_attn(q.to(dev), dev_cache(api, c, dev), torch.from_numpy(w.seq_len).to(dev), out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(out, oracle_self(w, c, q), f"131072 keys {layout}")


def test_1024_heads(api, cuda_device):
    dev = cuda_device
    w = workload("paged", [100, 17, 1], 128, 1024, 4)
    c = W.make_self_cache(w, 0, filled_len=w.seq_len)
    q = W.randn_bf16((w.B, 1024, D), "cpu", 604, 1)
    out = torch.empty((w.B, 1024, D), dtype=torch.bfloat16, device=dev)
    api.dr_decode_self_attn(q.to(dev), dev_cache(api, c, dev), torch.from_numpy(w.seq_len).to(dev), out)
    torch.cuda.synchronize()
    assert_attn_close(out, oracle_self(w, c, q), "H=1024")


def test_append_at_the_batch_limit(api, cuda_device):
    dev = cuda_device
    rng = np.random.default_rng(5)
    w = workload("paged", rng.integers(1, 32, size=65535, endpoint=True), 32, 1, 5)
    c = W.make_self_cache(w, 0)
    _, _, kn, vn = W.make_step_inputs(w, 0)
    kv = dev_cache(api, c, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_kv_append(kv, kn.to(dev), vn.to(dev), torch.from_numpy(w.seq_len - 1).to(dev), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kh, vh = W.bits(c.k).copy(), W.bits(c.v).copy()
    oracle.kv_append_paged(kh, vh, c.block_table.numpy(), W.bits(kn), W.bits(vn), w.seq_len - 1)
    assert np.array_equal(W.bits(kv.k), kh) and np.array_equal(W.bits(kv.v), vh)


def test_sampler_at_the_batch_limit(api, cuda_device):
    dev = cuda_device
    B, C, V = 65535, 1, 64
    rng = np.random.default_rng(6)
    logits = (rng.normal(size=(B, C, V)) * 3).astype(np.float32)
    seeds = rng.integers(0, 2 ** 63, size=B, dtype=np.uint64)
    steps = rng.integers(0, 3, size=B).astype(np.int32)            # step 0 pads codebook 0
    lg = torch.from_numpy(logits).to(dev)
    sd = torch.from_numpy(seeds.view(np.int64)).to(dev)
    st = torch.from_numpy(steps).to(dev)
    tok = torch.full((B, C), -7, dtype=torch.int32, device=dev)
    pr = torch.full((B, C, V), -1.0, dtype=torch.float32, device=dev)
    api.dr_sample_topk_delayed(lg, 0.8, 8, sd, st, 1024, tok, pr)
    torch.cuda.synchronize()
    ref = oracle.sample(logits, 0.8, 8, seeds, steps, 1024, want_probs=True)
    assert_tokens_match(tok, ref, "tokens, B=65535")
    assert_probs_match(pr, ref, "probs, B=65535")
    with pytest.raises(api.DrError) as e:                        # the grid holds 65,535 rows
        api.dr_sample_topk_delayed(torch.zeros((B + 1, C, V), device=dev), 0.8, 8,
                                   torch.zeros(B + 1, dtype=torch.int64, device=dev),
                                   torch.zeros(B + 1, dtype=torch.int32, device=dev), 1024,
                                   torch.empty((B + 1, C), dtype=torch.int32, device=dev))
    assert e.value.status == api.DR_ERR_UNSUPPORTED


def test_embedding_at_the_batch_limit(api, cuda_device):
    dev = cuda_device
    B, C, V, Dm = 65535, 9, 40, 64
    rng = np.random.default_rng(7)
    tokens = rng.integers(0, V, size=(B, C)).astype(np.int32)
    table = W.randn_bf16((C * V, Dm), "cpu", 607, 1)
    out = torch.empty((B, Dm), dtype=torch.float32, device=dev)
    api.dr_embed_tokens(torch.from_numpy(tokens).to(dev), table.to(dev), V, out)
    torch.cuda.synchronize()
    ref = oracle.embed_tokens(tokens, W.bits(table), V)
    # an fp32 sum of nine bf16 values in codebook order: within 9 u sum |x| of the float64 sum (u = 2^-24)
    tv = np.abs(table.double().numpy())
    mag = sum(tv[c * V + tokens[:, c]] for c in range(C))
    assert (np.abs(out.cpu().numpy() - ref) <= C * 2.0 ** -24 * mag + 1e-30).all()
