"""GPU parity of the FP8 E4M3 KV cache: the quantising append bit for bit, and
self-attention / the fused layer over an e4m3 cache within the attention
tolerance of the oracle's fp8 attention (key = code * k_scale, value = code *
v_scale, decoded exactly; only the fp32 accumulation differs)."""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_self_gb300 import workloads as W
from tests.parity import assert_attn_close, default_scale

pytestmark = pytest.mark.gpu
D = 64


@pytest.fixture(scope="module")
def api(cuda_device):
    from decode_attention_self_gb300 import api as _api

    return _api


def dev_cache(api, c, dev):
    return api.KVCache(c.k.to(dev), c.v.to(dev), c.block_table.to(dev) if c.block_table is not None else None,
                       c.k_scale, c.v_scale)


def codes(t):
    return t.detach().cpu().numpy().astype(np.uint8)


def ragged(layout, lens, cap, seed, filled=None):
    B = len(lens)
    w = W.Workload(300 + seed, "fp8", 1, B, layout, np.array(lens, np.int32), cap, np.array(lens, np.int32), cap, 1.0,
                   1, 1.0, np.zeros(B, np.uint64), np.zeros(B, np.int32))
    return w, W.make_self_cache_fp8(w, seed, filled_len=filled)


def oracle_fp8(w, c, q, lens=None):
    lens = w.seq_len if lens is None else lens
    s = default_scale(D)
    if c.layout == "contiguous":
        return oracle.attn_fp8_contiguous(W.bits(q), codes(c.k), codes(c.v), lens, s, c.k_scale, c.v_scale)
    return oracle.attn_fp8_paged(W.bits(q), codes(c.k), codes(c.v), c.block_table.numpy(), lens, s, c.k_scale,
                                 c.v_scale)


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_fp8_append_bit_exact(api, cuda_device, layout):
    dev = cuda_device
    w, c = ragged(layout, [1, 17, 64, 200], 256, 1)
    _, _, kn, vn = W.make_step_inputs(w, 1)
    kn = (kn.float() * 3).to(torch.bfloat16)                  # exercise the saturation at +-448 * scale too
    kv = dev_cache(api, c, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_kv_append(kv, kn.to(dev), vn.to(dev), torch.from_numpy(w.seq_len - 1).to(dev), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kh, vh = codes(c.k).copy(), codes(c.v).copy()
    if layout == "contiguous":
        oracle.kv_append_fp8_contiguous(kh, vh, W.bits(kn), W.bits(vn), w.seq_len - 1, c.k_scale, c.v_scale)
    else:
        oracle.kv_append_fp8_paged(kh, vh, c.block_table.numpy(), W.bits(kn), W.bits(vn), w.seq_len - 1, c.k_scale,
                                   c.v_scale)
    assert np.array_equal(codes(kv.k), kh) and np.array_equal(codes(kv.v), vh)


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("hint", [0, 64])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fp8_self_attention(api, cuda_device, layout, hint, out_dtype):
    dev = cuda_device
    lens = [1, 2, 15, 16, 17, 63, 100, 255, 256]
    w, c = ragged(layout, lens, 256, 2, filled=np.array(lens, np.int32))
    q = W.randn_bf16((w.B, 16, D), "cpu", 302, 1)
    out = torch.empty((w.B, 16, D), dtype=out_dtype, device=dev)
    api.dr_decode_self_attn(q.to(dev), dev_cache(api, c, dev), torch.from_numpy(w.seq_len).to(dev), out,
                            max_seq_len_hint=hint)
    assert_attn_close(out, oracle_fp8(w, c, q), f"fp8 {layout} hint {hint}")


# ceil(6 * 152 / (16 B)) CTAs per row (at most 8); an e4m3 row of 1024 keys is 128 KiB, under one CTA's share.
FP8_SPLIT_BATCHES = {8: 8, 9: 7, 10: 6, 12: 5, 15: 4, 20: 3, 29: 2, 57: 1}


@pytest.mark.parametrize("B", sorted(FP8_SPLIT_BATCHES))
def test_fp8_every_split_count(api, cuda_device, B):
    S = FP8_SPLIT_BATCHES[B]
    assert api.dr_plan_splits(B, 16, 1024, api.DR_KV_FP8_E4M3, 152) == S
    dev = cuda_device
    rng = np.random.default_rng(400 + B)
    # ragged rows, with short rows that leave some CTAs of their cluster without a tile
    lens = [1024, 1, 16, 17] + [int(x) for x in rng.integers(1, 1024, size=B - 4, endpoint=True)]
    w, c = ragged("paged", lens, 1024, 40 + B, filled=np.array(lens, np.int32))
    q = W.randn_bf16((w.B, 16, D), "cpu", 303, B)
    out = torch.empty((w.B, 16, D), dtype=torch.float32, device=dev)
    api.dr_decode_self_attn(q.to(dev), dev_cache(api, c, dev), torch.from_numpy(w.seq_len).to(dev), out,
                            max_seq_len_hint=1024)
    assert_attn_close(out, oracle_fp8(w, c, q), f"fp8 B={B}, {S} CTAs per row")


@pytest.mark.parametrize("index", [2, 4, 5])
def test_fp8_fused_layer_workloads(api, cuda_device, index):
    dev = cuda_device
    w = W.make_workload(index)
    c = W.make_self_cache_fp8(w, 4)
    q, qx, kn, vn = W.make_step_inputs(w, 4)
    kx, vx = W.make_cross_kv(w, 4)
    kv = dev_cache(api, c, dev)
    out = torch.empty((w.B, w.H, D), dtype=torch.float32, device=dev)
    outx = torch.empty_like(out)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_decode_layer(q.to(dev), kv, kn.to(dev), vn.to(dev), torch.from_numpy(w.seq_len).to(dev), qx.to(dev),
                        kx.to(dev), vx.to(dev), torch.from_numpy(w.enc_len).to(dev), out, outx,
                        max_seq_len_hint=int(w.seq_len.max()), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kh, vh = codes(c.k).copy(), codes(c.v).copy()
    if c.layout == "contiguous":
        oracle.kv_append_fp8_contiguous(kh, vh, W.bits(kn), W.bits(vn), w.seq_len - 1, c.k_scale, c.v_scale)
        ref = oracle.attn_fp8_contiguous(W.bits(q), kh, vh, w.seq_len, default_scale(D), c.k_scale, c.v_scale)
    else:
        t = c.block_table.numpy()
        oracle.kv_append_fp8_paged(kh, vh, t, W.bits(kn), W.bits(vn), w.seq_len - 1, c.k_scale, c.v_scale)
        ref = oracle.attn_fp8_paged(W.bits(q), kh, vh, t, w.seq_len, default_scale(D), c.k_scale, c.v_scale)
    assert np.array_equal(codes(kv.k), kh) and np.array_equal(codes(kv.v), vh)
    assert_attn_close(out, ref, f"fp8 fused self, workload {index}")
    assert_attn_close(outx, oracle.attn_contiguous(W.bits(qx), W.bits(kx), W.bits(vx), w.enc_len, default_scale(D)),
                      f"fused cross next to an fp8 self cache, workload {index}")


def test_fp8_separate_calls_equal_fused(api, cuda_device):
    dev = cuda_device
    w, c = ragged("paged", [500, 1000, 37, 4000], 4096, 5)
    q, qx, kn, vn = W.make_step_inputs(w, 5)
    kx, vx = W.make_cross_kv(w, 5)
    seq = torch.from_numpy(w.seq_len).to(dev)
    kv1, kv2 = dev_cache(api, c, dev), dev_cache(api, c, dev)
    o1 = torch.empty((w.B, 16, D), dtype=torch.float32, device=dev)
    o2, ox = torch.empty_like(o1), torch.empty_like(o1)
    api.dr_kv_append(kv1, kn.to(dev), vn.to(dev), torch.from_numpy(w.seq_len - 1).to(dev))
    api.dr_decode_self_attn(q.to(dev), kv1, seq, o1, max_seq_len_hint=4096)
    api.dr_decode_layer(q.to(dev), kv2, kn.to(dev), vn.to(dev), seq, qx.to(dev), kx.to(dev), vx.to(dev),
                        torch.from_numpy(w.enc_len).to(dev), o2, ox, max_seq_len_hint=4096)
    torch.cuda.synchronize()
    assert torch.equal(kv1.k, kv2.k) and torch.equal(kv1.v, kv2.v)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_fp8_fused_layer_edge_lengths(api, cuda_device, layout):
    # the fused append quantises this step's key inside the attention launch: lengths at and around the 16-key
    # tile edges, a row of one key, the capacity, and description lengths around the packing threshold
    dev = cuda_device
    lens = np.array([1, 2, 16, 17, 64, 255, 256], np.int32)
    enc_len = np.array([1, 300, 16, 17, 5, 299, 100], np.int32)
    B = len(lens)
    w = W.Workload(320, "fp8 edge", 1, B, layout, lens, 256, enc_len, 300, 1.0, 1, 1.0, np.zeros(B, np.uint64),
                   np.zeros(B, np.int32))
    c = W.make_self_cache_fp8(w, 0)
    q, qx, kn, vn = W.make_step_inputs(w, 0)
    kx, vx = W.make_cross_kv(w, 0)
    s = default_scale(D)
    refx = oracle.attn_contiguous(W.bits(qx), W.bits(kx), W.bits(vx), enc_len, s)
    for hint in (0, 64):
        kv = dev_cache(api, c, dev)
        out = torch.empty((B, 16, D), dtype=torch.bfloat16, device=dev)
        outx = torch.empty_like(out)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        api.dr_decode_layer(q.to(dev), kv, kn.to(dev), vn.to(dev), torch.from_numpy(lens).to(dev), qx.to(dev),
                            kx.to(dev), vx.to(dev), torch.from_numpy(enc_len).to(dev), out, outx,
                            max_seq_len_hint=hint, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        kh, vh = codes(c.k).copy(), codes(c.v).copy()
        if layout == "contiguous":
            oracle.kv_append_fp8_contiguous(kh, vh, W.bits(kn), W.bits(vn), lens - 1, c.k_scale, c.v_scale)
            ref = oracle.attn_fp8_contiguous(W.bits(q), kh, vh, lens, s, c.k_scale, c.v_scale)
        else:
            t = c.block_table.numpy()
            oracle.kv_append_fp8_paged(kh, vh, t, W.bits(kn), W.bits(vn), lens - 1, c.k_scale, c.v_scale)
            ref = oracle.attn_fp8_paged(W.bits(q), kh, vh, t, lens, s, c.k_scale, c.v_scale)
        assert np.array_equal(codes(kv.k), kh) and np.array_equal(codes(kv.v), vh), f"codes, hint {hint}"
        assert_attn_close(out, ref, f"fp8 fused self {layout} hint {hint}")
        assert_attn_close(outx, refx, f"fused cross {layout} hint {hint}")


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_fp8_wide_clusters_for_few_long_rows(api, cuda_device, layout):
    # batch 1, e4m3 rows of 2048 keys or more: one non-portable cluster of 16 CTAs per row
    assert api.dr_plan_splits(1, 16, 4096, api.DR_KV_FP8_E4M3, 152) == 16
    dev = cuda_device
    lens = [3500]
    w, c = ragged(layout, lens, 4096, 77, filled=np.array(lens, np.int32))
    q = W.randn_bf16((1, 16, D), "cpu", 304, 1)
    out = torch.empty((1, 16, D), dtype=torch.float32, device=dev)
    api.dr_decode_self_attn(q.to(dev), dev_cache(api, c, dev), torch.from_numpy(w.seq_len).to(dev), out,
                            max_seq_len_hint=4096)
    assert_attn_close(out, oracle_fp8(w, c, q), f"fp8 {layout} 16 CTAs per row")
