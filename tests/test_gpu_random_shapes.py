"""Randomised parity sweep over launch shapes (GPU against the oracle).

Every call here goes through the same arithmetic, but the launcher picks the
kernel variant (whole grid resident or streaming), the cluster width (1-8 CTAs
per row, or 16 for a few long rows), packed or split description rows and
the cluster-merge form from the batch, the heads, the length bound and the
device.  Seeded random shapes cross those boundaries: batch 1..40, 1..19
heads, capacities 64..4096, uniform / full / few-long-among-short length
mixes, both layouts, bf16 and e4m3 caches, the fused layer or the three
separate calls, and several length hints.  Each must match the oracle within
the attention tolerance, with no device error flag.
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


def random_shape(seed):
    r = np.random.default_rng([77, seed])
    B = int(r.choice([1, 1, 2, 3, 5, 8, 12, 19, 32, 40]))
    H = int(r.choice([1, 2, 4, 16, 16, 19]))
    cap = int(r.choice([64, 200, 1024, 2048, 4096]))
    while B > 1 and B * H * cap > 1 << 19:   # keeps the host-side cache and the oracle small
        B //= 2
    mode = int(r.integers(0, 3))
    if mode == 0:
        lens = r.integers(1, cap, size=B, endpoint=True)
    elif mode == 1:
        lens = np.full(B, cap)
    else:
        lens = np.where(r.random(B) < 0.25, cap, r.integers(1, max(2, cap // 16), size=B, endpoint=True))
    enc_max = int(r.choice([16, 64, 300, 1024, 3000]))
    return dict(B=B, H=H, cap=cap, lens=lens.astype(np.int32), layout=str(r.choice(["contiguous", "paged"])),
                fp8=bool(r.random() < 0.3), fused=bool(r.random() < 0.5),
                hint=int(r.choice([0, int(lens.max()), cap])), enc_max=enc_max,
                enc=r.integers(1, enc_max, size=B, endpoint=True).astype(np.int32))


@pytest.mark.parametrize("seed", range(48))
def test_random_shape_matches_the_oracle(api, cuda_device, seed):
    s = random_shape(seed)
    dev, B, H, lens, enc = cuda_device, s["B"], s["H"], s["lens"], s["enc"]
    w = W.Workload(400 + seed, "random", 1, B, s["layout"], lens, s["cap"], enc, s["enc_max"], 1.0, 1, 1.0,
                   np.zeros(B, np.uint64), np.zeros(B, np.int32), H=H)
    cache = (W.make_self_cache_fp8 if s["fp8"] else W.make_self_cache)(w, seed)   # slot len-1 filled by the append
    q, qx, kn, vn = W.make_step_inputs(w, seed)
    kx, vx = W.make_cross_kv(w, seed)
    kv = api.KVCache(cache.k.to(dev), cache.v.to(dev),
                     cache.block_table.to(dev) if cache.block_table is not None else None, cache.k_scale, cache.v_scale)
    seq, encd = torch.from_numpy(lens).to(dev), torch.from_numpy(enc).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    outx = torch.empty_like(out)
    qd, qxd, knd, vnd, kxd, vxd = (t.to(dev) for t in (q, qx, kn, vn, kx, vx))
    if s["fused"]:
        api.dr_decode_layer(qd, kv, knd, vnd, seq, qxd, kxd, vxd, encd, out, outx, max_seq_len_hint=s["hint"],
                            err_flag=err)
    else:
        api.dr_kv_append(kv, knd, vnd, seq - 1, err_flag=err)
        api.dr_decode_self_attn(qd, kv, seq, out, max_seq_len_hint=s["hint"], err_flag=err)
        api.dr_decode_cross_attn(qxd, kxd, vxd, encd, outx, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, s

    sc = default_scale(D)
    table = cache.block_table.numpy() if cache.block_table is not None else None
    if s["fp8"]:
        kh, vh = cache.k.numpy().astype(np.uint8).copy(), cache.v.numpy().astype(np.uint8).copy()
        if table is None:
            oracle.kv_append_fp8_contiguous(kh, vh, W.bits(kn), W.bits(vn), lens - 1, cache.k_scale, cache.v_scale)
            ref = oracle.attn_fp8_contiguous(W.bits(q), kh, vh, lens, sc, cache.k_scale, cache.v_scale)
        else:
            oracle.kv_append_fp8_paged(kh, vh, table, W.bits(kn), W.bits(vn), lens - 1, cache.k_scale, cache.v_scale)
            ref = oracle.attn_fp8_paged(W.bits(q), kh, vh, table, lens, sc, cache.k_scale, cache.v_scale)
    else:
        kh, vh = W.bits(cache.k).copy(), W.bits(cache.v).copy()
        if table is None:
            oracle.kv_append_contiguous(kh, vh, W.bits(kn), W.bits(vn), lens - 1)
            ref = oracle.attn_contiguous(W.bits(q), kh, vh, lens, sc)
        else:
            oracle.kv_append_paged(kh, vh, table, W.bits(kn), W.bits(vn), lens - 1)
            ref = oracle.attn_paged(W.bits(q), kh, vh, table, lens, sc)
    what = ", ".join(f"{k}={v if not isinstance(v, np.ndarray) else v[:6].tolist()}" for k, v in s.items())
    assert_attn_close(out, ref, "self: " + what)
    assert_attn_close(outx, oracle.attn_contiguous(W.bits(qx), W.bits(kx), W.bits(vx), enc, sc), "cross: " + what)
    # the append wrote exactly the new rows
    got_k = kv.k.cpu().numpy() if s["fp8"] else W.bits(kv.k)
    assert np.array_equal(got_k.astype(kh.dtype), kh)
