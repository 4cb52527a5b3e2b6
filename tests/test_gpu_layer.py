"""GPU parity of dr_decode_layer (append + self-attention + cross-attention in one launch).

The fused launch must equal the three separate calls it replaces: the cache
after it bit for bit, the self-attention bit for bit (same split plan, same
arithmetic), and both attention outputs within tolerance of the oracle.
"""
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


def dev_cache(api, cache, dev):
    return api.KVCache(cache.k.to(dev), cache.v.to(dev),
                       cache.block_table.to(dev) if cache.block_table is not None else None)


_HOST = {}


def host_layer(index):
    if index not in _HOST:
        w = W.make_workload(index)
        cache = W.make_self_cache(w, 3)
        _HOST[index] = (w, cache, W.make_step_inputs(w, 3), W.make_cross_kv(w, 3))
    return _HOST[index]


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_fused_layer_matches_oracle_and_separate_calls(api, cuda_device, index):
    dev = cuda_device
    w, cache, (q, qx, kn, vn), (kx, vx) = host_layer(index)
    seq = torch.from_numpy(w.seq_len).to(dev)
    enc = torch.from_numpy(w.enc_len).to(dev)
    pos = torch.from_numpy(w.seq_len - 1).to(dev)
    hint = int(w.seq_len.max())
    qd, qxd, knd, vnd, kxd, vxd = (t.to(dev) for t in (q, qx, kn, vn, kx, vx))
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    kv_f = dev_cache(api, cache, dev)
    out_f = torch.empty((w.B, w.H, D), dtype=torch.float32, device=dev)
    outx_f = torch.empty_like(out_f)
    api.dr_decode_layer(qd, kv_f, knd, vnd, seq, qxd, kxd, vxd, enc, out_f, outx_f, max_seq_len_hint=hint,
                        err_flag=err)

    kv_s = dev_cache(api, cache, dev)
    out_s = torch.empty_like(out_f)
    api.dr_kv_append(kv_s, knd, vnd, pos, err_flag=err)
    api.dr_decode_self_attn(qd, kv_s, seq, out_s, max_seq_len_hint=hint, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bits16 = lambda t: t.view(torch.int16)                            # NaN padding: compare bit patterns
    assert torch.equal(bits16(kv_f.k), bits16(kv_s.k)) and torch.equal(bits16(kv_f.v), bits16(kv_s.v))
    assert torch.equal(out_f, out_s)

    scale = default_scale(D)
    kh, vh = W.bits(cache.k).copy(), W.bits(cache.v).copy()
    if cache.layout == "contiguous":
        oracle.kv_append_contiguous(kh, vh, W.bits(kn), W.bits(vn), w.seq_len - 1)
        ref = oracle.attn_contiguous(W.bits(q), kh, vh, w.seq_len, scale)
    else:
        t = cache.block_table.numpy()
        oracle.kv_append_paged(kh, vh, t, W.bits(kn), W.bits(vn), w.seq_len - 1)
        ref = oracle.attn_paged(W.bits(q), kh, vh, t, w.seq_len, scale)
    assert np.array_equal(W.bits(kv_f.k), kh) and np.array_equal(W.bits(kv_f.v), vh)
    assert_attn_close(out_f, ref, f"fused self-attention, workload {index}")
    refx = oracle.attn_contiguous(W.bits(qx), W.bits(kx), W.bits(vx), w.enc_len, scale)
    assert_attn_close(outx_f, refx, f"fused cross-attention, workload {index}")


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_fused_layer_edge_lengths_bf16(api, cuda_device, layout):
    dev = cuda_device
    lens = np.array([1, 2, 16, 17, 64, 255, 256], np.int32)
    enc_len = np.array([1, 300, 16, 17, 5, 299, 100], np.int32)
    B = len(lens)
    w = W.Workload(120, "edge", 1, B, layout, lens, 256, enc_len, 300, 1.0, 1, 1.0, np.zeros(B, np.uint64),
                   np.zeros(B, np.int32))
    cache = W.make_self_cache(w, 0)
    q, qx, kn, vn = W.make_step_inputs(w, 0)
    kx, vx = W.make_cross_kv(w, 0)
    kv = dev_cache(api, cache, dev)
    out = torch.empty((B, 16, D), dtype=torch.bfloat16, device=dev)
    outx = torch.empty_like(out)
    for hint in (0, 64):
        api.dr_decode_layer(q.to(dev), kv, kn.to(dev), vn.to(dev), torch.from_numpy(lens).to(dev), qx.to(dev),
                            kx.to(dev), vx.to(dev), torch.from_numpy(enc_len).to(dev), out, outx,
                            max_seq_len_hint=hint)
        torch.cuda.synchronize()
        kh, vh = W.bits(cache.k).copy(), W.bits(cache.v).copy()
        if layout == "contiguous":
            oracle.kv_append_contiguous(kh, vh, W.bits(kn), W.bits(vn), lens - 1)
            ref = oracle.attn_contiguous(W.bits(q), kh, vh, lens, default_scale(D))
        else:
            t = cache.block_table.numpy()
            oracle.kv_append_paged(kh, vh, t, W.bits(kn), W.bits(vn), lens - 1)
            ref = oracle.attn_paged(W.bits(q), kh, vh, t, lens, default_scale(D))
        assert_attn_close(out, ref, f"{layout} hint {hint}")
        refx = oracle.attn_contiguous(W.bits(qx), W.bits(kx), W.bits(vx), enc_len, default_scale(D))
        assert_attn_close(outx, refx, f"{layout} cross hint {hint}")


def test_fused_layer_invalid_length_skips_the_append(api, cuda_device):
    dev = cuda_device
    w = W.Workload(121, "edge", 1, 2, "contiguous", np.array([10, 10], np.int32), 32, np.array([4, 4], np.int32), 8,
                   1.0, 1, 1.0, np.zeros(2, np.uint64), np.zeros(2, np.int32))
    cache = W.make_self_cache(w, 0, filled_len=np.array([10, 32], np.int32))
    q, qx, kn, vn = W.make_step_inputs(w, 0)
    kx, vx = W.make_cross_kv(w, 0)
    kv = dev_cache(api, cache, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((2, 16, D), dtype=torch.float32, device=dev)
    outx = torch.empty_like(out)
    seq = torch.tensor([10, 99], dtype=torch.int32, device=dev)       # row 1 past the 32-key capacity
    api.dr_decode_layer(q.to(dev), kv, kn.to(dev), vn.to(dev), seq, qx.to(dev), kx.to(dev), vx.to(dev),
                        torch.from_numpy(w.enc_len).to(dev), out, outx, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1 and int(err.item()) & 4
    kb = W.bits(kv.k)
    assert np.array_equal(kb[1], W.bits(cache.k)[1])                  # row 1 untouched
    assert np.array_equal(kb[0, :, 9], W.bits(kn)[0])                 # row 0 appended at slot 9
    ref1 = oracle.attn_contiguous(W.bits(q)[1:], W.bits(cache.k)[1:], W.bits(cache.v)[1:], np.array([32]),
                                  default_scale(D))
    assert_attn_close(out[1:], ref1)


@pytest.mark.parametrize("B,self_len,enc_max", [(5, 1000, 64), (3, 3000, 40), (9, 600, 1500)])
def test_fused_layer_cross_row_layouts(api, cuda_device, B, self_len, enc_max):
    # Short description rows are packed one per CTA (with an idle tail when B is not a multiple of the
    # cluster size); long ones are split across the cluster like the self rows.
    dev = cuda_device
    rng = np.random.default_rng(B)
    lens = rng.integers(self_len // 2, self_len, size=B, endpoint=True).astype(np.int32)
    enc_len = rng.integers(1, enc_max, size=B, endpoint=True).astype(np.int32)
    w = W.Workload(130 + B, "layouts", 1, B, "paged", lens, 4096, enc_len, enc_max, 1.0, 1, 1.0,
                   np.zeros(B, np.uint64), np.zeros(B, np.int32))
    s_self = api.dr_plan_splits(B, 16, int(lens.max()), api.DR_KV_BF16, 152)
    s_cross = api.dr_plan_splits(B, 16, enc_max, api.DR_KV_BF16, 152)
    cache = W.make_self_cache(w, 0)
    q, qx, kn, vn = W.make_step_inputs(w, 0)
    kx, vx = W.make_cross_kv(w, 0)
    kv = dev_cache(api, cache, dev)
    out = torch.empty((B, 16, D), dtype=torch.float32, device=dev)
    outx = torch.empty_like(out)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_decode_layer(q.to(dev), kv, kn.to(dev), vn.to(dev), torch.from_numpy(lens).to(dev), qx.to(dev), kx.to(dev),
                        vx.to(dev), torch.from_numpy(enc_len).to(dev), out, outx, max_seq_len_hint=int(lens.max()),
                        err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kh, vh = W.bits(cache.k).copy(), W.bits(cache.v).copy()
    t = cache.block_table.numpy()
    oracle.kv_append_paged(kh, vh, t, W.bits(kn), W.bits(vn), lens - 1)
    assert_attn_close(out, oracle.attn_paged(W.bits(q), kh, vh, t, lens, default_scale(D)),
                      f"self (splits {s_self})")
    assert_attn_close(outx, oracle.attn_contiguous(W.bits(qx), W.bits(kx), W.bits(vx), enc_len, default_scale(D)),
                      f"cross (standalone plan {s_cross}, self plan {s_self})")


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("L,enc_max", [(2048, 64), (2050, 3000), (4096, 700)])
def test_fused_layer_wide_clusters(api, cuda_device, layout, L, enc_max):
    # Batch 1 with a self row of 2048 keys or more: 16 CTAs per row in one non-portable cluster; the description
    # rows are either packed 16 to a cluster (64 keys) or split 16 ways like the self rows (3000 keys).  The
    # appended key opens a new tile (2050) or fills the cache's last slot (4096).  The fused launch equals the
    # separate calls bit for bit (cache and self-attention) and the oracle within tolerance.
    dev = cuda_device
    assert api.dr_plan_splits(1, 16, L, api.DR_KV_BF16, 152) == 16
    lens = np.array([L], np.int32)
    enc_len = np.array([enc_max - 7], np.int32)
    w = W.Workload(121, "wide", 1, 1, layout, lens, 4096, enc_len, enc_max, 1.0, 1, 1.0, np.zeros(1, np.uint64),
                   np.zeros(1, np.int32))
    cache = W.make_self_cache(w, L % 97)
    q, qx, kn, vn = W.make_step_inputs(w, 1)
    kx, vx = W.make_cross_kv(w, 1)
    seq, enc = torch.from_numpy(lens).to(dev), torch.from_numpy(enc_len).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kv_f, kv_s = dev_cache(api, cache, dev), dev_cache(api, cache, dev)
    out_f = torch.empty((1, 16, D), dtype=torch.float32, device=dev)
    outx_f, out_s, outx_s = torch.empty_like(out_f), torch.empty_like(out_f), torch.empty_like(out_f)
    qd, qxd, knd, vnd, kxd, vxd = (t.to(dev) for t in (q, qx, kn, vn, kx, vx))
    api.dr_decode_layer(qd, kv_f, knd, vnd, seq, qxd, kxd, vxd, enc, out_f, outx_f, max_seq_len_hint=L, err_flag=err)
    api.dr_kv_append(kv_s, knd, vnd, seq - 1, err_flag=err)
    api.dr_decode_self_attn(qd, kv_s, seq, out_s, max_seq_len_hint=L, err_flag=err)
    api.dr_decode_cross_attn(qxd, kxd, vxd, enc, outx_s, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # bit patterns: the slots past the valid keys hold NaN
    assert np.array_equal(W.bits(kv_f.k), W.bits(kv_s.k)) and np.array_equal(W.bits(kv_f.v), W.bits(kv_s.v))
    assert torch.equal(out_f, out_s)
    kh, vh = W.bits(cache.k).copy(), W.bits(cache.v).copy()
    if layout == "contiguous":
        oracle.kv_append_contiguous(kh, vh, W.bits(kn), W.bits(vn), lens - 1)
        ref = oracle.attn_contiguous(W.bits(q), kh, vh, lens, default_scale(D))
    else:
        t = cache.block_table.numpy()
        oracle.kv_append_paged(kh, vh, t, W.bits(kn), W.bits(vn), lens - 1)
        ref = oracle.attn_paged(W.bits(q), kh, vh, t, lens, default_scale(D))
    assert np.array_equal(W.bits(kv_f.k), kh) and np.array_equal(W.bits(kv_f.v), vh)
    assert_attn_close(out_f, ref, f"self, {layout} L={L}")
    refx = oracle.attn_contiguous(W.bits(qx), W.bits(kx), W.bits(vx), enc_len, default_scale(D))
    assert_attn_close(outx_f, refx, f"cross, {layout} L={L}")
    assert_attn_close(outx_s, refx, f"standalone cross, {layout} L={L}")
