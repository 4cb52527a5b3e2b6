"""GPU checks of dr_kv_append: bit-exact cache contents against the oracle's append, and
device-side errors (position past the capacity, unmapped paged block) flagged without a write."""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_self_gb300 import workloads as W

pytestmark = pytest.mark.gpu
D = 64


@pytest.fixture(scope="module")
def api(cuda_device):
    from decode_attention_self_gb300 import api as _api

    return _api


def case(layout, lens, cap, H=16, seed=0):
    B = len(lens)
    w = W.Workload(140 + seed, "append", 1, B, layout, np.array(lens, np.int32), cap, np.array(lens, np.int32), cap,
                   1.0, 1, 1.0, np.zeros(B, np.uint64), np.zeros(B, np.int32), H=H)
    cache = W.make_self_cache(w, seed)
    _, _, kn, vn = W.make_step_inputs(w, seed)
    return w, cache, kn, vn


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("H", [1, 16, 33])
def test_append_bit_exact(api, cuda_device, layout, H):
    dev = cuda_device
    w, cache, kn, vn = case(layout, [1, 16, 17, 200, 256], 256, H=H, seed=H)
    kv = api.KVCache(cache.k.to(dev), cache.v.to(dev),
                     cache.block_table.to(dev) if cache.block_table is not None else None)
    pos = w.seq_len - 1
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_kv_append(kv, kn.to(dev), vn.to(dev), torch.from_numpy(pos).to(dev), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kh, vh = W.bits(cache.k).copy(), W.bits(cache.v).copy()
    if layout == "contiguous":
        oracle.kv_append_contiguous(kh, vh, W.bits(kn), W.bits(vn), pos)
    else:
        oracle.kv_append_paged(kh, vh, cache.block_table.numpy(), W.bits(kn), W.bits(vn), pos)
    assert np.array_equal(W.bits(kv.k), kh) and np.array_equal(W.bits(kv.v), vh)


def test_append_position_out_of_range_is_flagged_and_skipped(api, cuda_device):
    dev = cuda_device
    w, cache, kn, vn = case("contiguous", [10, 10, 10], 32, seed=50)
    kv = api.KVCache(cache.k.to(dev), cache.v.to(dev))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pos = torch.tensor([3, 32, -1], dtype=torch.int32, device=dev)       # rows 1 and 2 are invalid
    api.dr_kv_append(kv, kn.to(dev), vn.to(dev), pos, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 4
    kb = W.bits(kv.k)
    ref = W.bits(cache.k)
    assert np.array_equal(kb[0, :, 3], W.bits(kn)[0])
    assert np.array_equal(kb[1:], ref[1:])


def test_append_to_unmapped_block_is_flagged_and_skipped(api, cuda_device):
    dev = cuda_device
    w, cache, kn, vn = case("paged", [20, 40], 64, seed=51)
    table = cache.block_table.clone()
    table[1, 2] = -1                                                     # row 1's position 39 has no block
    kv = api.KVCache(cache.k.to(dev), cache.v.to(dev), table.to(dev))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_kv_append(kv, kn.to(dev), vn.to(dev), torch.tensor([19, 39], dtype=torch.int32, device=dev), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 4
    kh = W.bits(cache.k).copy()
    vh = W.bits(cache.v).copy()
    t = cache.block_table.numpy()
    oracle.kv_append_paged(kh, vh, t[:1], W.bits(kn)[:1], W.bits(vn)[:1], np.array([19]))
    assert np.array_equal(W.bits(kv.k), kh)
