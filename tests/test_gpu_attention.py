"""GPU parity of dr_decode_self_attn / dr_decode_cross_attn against the oracle.

Single-query attention over the valid part of a static or paged cache
(Optimized Parler TTS, "Analysis and improvements" and "Future work" item 1)
and over the description encoder's keys and values (architecture overview).
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


def to_dev(cache: W.SelfCache, dev):
    from decode_attention_self_gb300 import api as _api

    return _api.KVCache(cache.k.to(dev), cache.v.to(dev),
                        cache.block_table.to(dev) if cache.block_table is not None else None)


def oracle_self(w, cache, q, scale, lens=None):
    lens = w.seq_len if lens is None else lens
    if cache.layout == "contiguous":
        return oracle.attn_contiguous(W.bits(q), W.bits(cache.k), W.bits(cache.v), lens, scale)
    return oracle.attn_paged(W.bits(q), W.bits(cache.k), W.bits(cache.v), cache.block_table.numpy(), lens, scale)


# ---------------------------------------------------------------------------
# the five workloads: append + self-attention + cross-attention of one layer
# ---------------------------------------------------------------------------
_HOST = {}


def host_layer(index):
    """Seeded host inputs of one layer of workload `index` (generated once per module)."""
    if index not in _HOST:
        w = W.make_workload(index)
        layer = 0 if index != 2 else 7
        cache = W.make_self_cache(w, layer)                   # slot seq_len-1 is NaN until the append
        _HOST[index] = (w, cache, W.make_step_inputs(w, layer), W.make_cross_kv(w, layer))
    return _HOST[index]


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_workload_layer_parity(api, cuda_device, index, out_dtype):
    dev = cuda_device
    w, cache, (q, qx, kn, vn), (kx, vx) = host_layer(index)
    kv = to_dev(cache, dev)
    pos = torch.from_numpy(w.seq_len - 1).to(dev)
    seq = torch.from_numpy(w.seq_len).to(dev)
    enc = torch.from_numpy(w.enc_len).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out_s = torch.empty((w.B, w.H, D), dtype=out_dtype, device=dev)
    out_x = torch.empty_like(out_s)
    api.dr_kv_append(kv, kn.to(dev), vn.to(dev), pos, err_flag=err)
    api.dr_decode_self_attn(q.to(dev), kv, seq, out_s, max_seq_len_hint=int(w.seq_len.max()), err_flag=err)
    api.dr_decode_cross_attn(qx.to(dev), kx.to(dev), vx.to(dev), enc, out_x, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    scale = default_scale(D)
    kh, vh = W.bits(cache.k).copy(), W.bits(cache.v).copy()
    if cache.layout == "contiguous":
        oracle.kv_append_contiguous(kh, vh, W.bits(kn), W.bits(vn), w.seq_len - 1)
        ref_s = oracle.attn_contiguous(W.bits(q), kh, vh, w.seq_len, scale)
    else:
        table = cache.block_table.numpy()
        oracle.kv_append_paged(kh, vh, table, W.bits(kn), W.bits(vn), w.seq_len - 1)
        ref_s = oracle.attn_paged(W.bits(q), kh, vh, table, w.seq_len, scale)
    ref_x = oracle.attn_contiguous(W.bits(qx), W.bits(kx), W.bits(vx), w.enc_len, scale)
    assert_attn_close(out_s, ref_s, f"self-attention, workload {index}")
    assert_attn_close(out_x, ref_x, f"cross-attention, workload {index}")
    # the append wrote exactly the new rows (bit-exact cache contents)
    assert np.array_equal(W.bits(kv.k), kh) and np.array_equal(W.bits(kv.v), vh)


# ---------------------------------------------------------------------------
# edge cases: lengths around tile boundaries, capacity, every split count
# ---------------------------------------------------------------------------
LENS = [1, 2, 15, 16, 17, 31, 33, 63, 64, 65, 100, 255, 256]


def ragged_case(layout, lens, cap, H=16, seed=0):
    w = W.Workload(100 + seed, "edge", 1, len(lens), layout, np.array(lens, np.int32), cap,
                   np.array(lens, np.int32), cap, 1.0, 1, 1.0, np.zeros(len(lens), np.uint64),
                   np.zeros(len(lens), np.int32), H=H)
    cache = W.make_self_cache(w, seed, filled_len=w.seq_len)
    q = W.randn_bf16((w.B, H, D), "cpu", 100 + seed, 9)
    return w, cache, q


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("hint", [0, 64, 256, 1024])
def test_ragged_lengths_and_split_counts(api, cuda_device, layout, hint):
    w, cache, q = ragged_case(layout, LENS, 256)
    kv = to_dev(cache, cuda_device)
    out = torch.empty((w.B, w.H, D), dtype=torch.float32, device=cuda_device)
    api.dr_decode_self_attn(q.to(cuda_device), kv, torch.from_numpy(w.seq_len).to(cuda_device), out,
                            max_seq_len_hint=hint)
    assert_attn_close(out, oracle_self(w, cache, q, default_scale(D)), f"{layout} hint {hint}")


# Batch sizes whose 16-head rows give each split count for a 1024-key bound on 152 SMs: the plan asks for
# ceil(6 * 152 / (16 B)) CTAs per row (at most 8), and 256 KiB per CTA needs only one.
SPLIT_BATCHES = {8: 8, 9: 7, 10: 6, 12: 5, 15: 4, 20: 3, 29: 2, 57: 1}


@pytest.mark.parametrize("B", sorted(SPLIT_BATCHES))
def test_every_split_count(api, cuda_device, B):
    S = SPLIT_BATCHES[B]
    assert api.dr_plan_splits(B, 16, 1024, api.DR_KV_BF16, 152) == S
    rng = np.random.default_rng(B)
    # ragged rows, with short rows that leave some CTAs of their cluster without a tile
    lens = [1024, 1, 16, 17] + [int(x) for x in rng.integers(1, 1024, size=B - 4, endpoint=True)]
    w, cache, q = ragged_case("paged", lens, 1024, seed=20 + B)
    kv = to_dev(cache, cuda_device)
    out = torch.empty((w.B, w.H, D), dtype=torch.float32, device=cuda_device)
    api.dr_decode_self_attn(q.to(cuda_device), kv, torch.from_numpy(w.seq_len).to(cuda_device), out,
                            max_seq_len_hint=1024)
    assert_attn_close(out, oracle_self(w, cache, q, default_scale(D)), f"B={B}, {S} CTAs per row")


@pytest.mark.parametrize("mode", ["growing", "peaked", "zero_query", "huge"])
def test_extreme_score_ranges(api, cuda_device, mode):
    # growing: each key scores ~0.7 above the previous one in the log2 domain (~11 per 16-key tile, more than
    #   the kernel's rescale slack of 8), so the running maximum moves and the state is rescaled tile after tile;
    # peaked: one key of each row dominates the others by thousands;
    # zero_query: every score is 0, so the output is the mean of the values;
    # huge: scores in the thousands with both signs (most weights underflow to zero).
    lens = [1, 40, 700, 3000]
    w, cache, q = ragged_case("contiguous", lens, 3072, seed=61)
    gen = torch.Generator().manual_seed(62)
    u = torch.randn(D, generator=gen)
    u = u / u.norm()
    k = cache.k.float()
    qf = q.float()
    if mode == "growing":
        c = torch.arange(3072, dtype=torch.float32) / 2.0            # q.k grows by 4 per key: 0.5 after x 1/8
        k = 0.1 * k + c.view(1, 1, -1, 1) * u.view(1, 1, 1, -1)
        qf = 8.0 * u.expand_as(qf).clone()
    elif mode == "peaked":
        k = 0.1 * k
        for b, L in enumerate(lens):
            k[b, :, (L - 1) // 2] = 300.0 * u
        qf = 8.0 * u.expand_as(qf).clone()
    elif mode == "zero_query":
        qf = torch.zeros_like(qf)
    else:
        k = 40.0 * k
        qf = 40.0 * qf
    cache.k = k.to(torch.bfloat16)
    q = qf.to(torch.bfloat16)
    kv = to_dev(cache, cuda_device)
    out = torch.empty((w.B, w.H, D), dtype=torch.float32, device=cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    api.dr_decode_self_attn(q.to(cuda_device), kv, torch.from_numpy(w.seq_len).to(cuda_device), out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle_self(w, cache, q, default_scale(D))
    if mode == "zero_query":   # the plain mean, independently of the oracle
        vv = cache.v.double().numpy()
        for b, L in enumerate(lens):
            np.testing.assert_allclose(ref[b], vv[b, :, :L].mean(axis=1), rtol=0, atol=1e-12)
    assert_attn_close(out, ref, f"scores {mode}")


@pytest.mark.parametrize("L", [1, 17, 1000, 4095, 4096])
def test_batch1_long_rows(api, cuda_device, L):
    w, cache, q = ragged_case("contiguous", [L], 4096, seed=3)
    kv = to_dev(cache, cuda_device)
    out = torch.empty((1, 16, D), dtype=torch.float32, device=cuda_device)
    api.dr_decode_self_attn(q.to(cuda_device), kv, torch.from_numpy(w.seq_len).to(cuda_device), out)
    assert_attn_close(out, oracle_self(w, cache, q, default_scale(D)), f"L={L}")


def test_other_head_counts_and_scale(api, cuda_device):
    for H in (1, 3, 40):
        w, cache, q = ragged_case("paged", [5, 70, 129], 160, H=H, seed=H)
        kv = to_dev(cache, cuda_device)
        out = torch.empty((w.B, H, D), dtype=torch.float32, device=cuda_device)
        api.dr_decode_self_attn(q.to(cuda_device), kv, torch.from_numpy(w.seq_len).to(cuda_device), out, scale=0.3)
        assert_attn_close(out, oracle_self(w, cache, q, 0.3), f"H={H}")


def test_paged_equals_contiguous_bitwise(api, cuda_device):
    # Same logical rows, same split plan: the kernel's reduction order depends only on the tile
    # partition, so the paged layout with a shuffled table must reproduce the contiguous result bit for bit.
    lens = [7, 16, 100, 255, 256, 33]
    wc, cc, q = ragged_case("contiguous", lens, 256, seed=5)
    wp = W.Workload(105, "edge", 1, len(lens), "paged", wc.seq_len, 256, wc.seq_len, 256, 1.0, 1, 1.0,
                    wc.seeds, wc.steps)
    table, NB = W.make_block_table(wp, "cpu", 5)
    kp = torch.full((NB, 16, 16, D), float("nan"), dtype=torch.bfloat16)
    vp = kp.clone()
    for b, L in enumerate(lens):
        for j in range((L + 15) // 16):
            kp[table[b, j]] = cc.k[b, :, 16 * j:16 * j + 16]
            vp[table[b, j]] = cc.v[b, :, 16 * j:16 * j + 16]
    from decode_attention_self_gb300 import api as _api
    dev = cuda_device
    kvc = _api.KVCache(cc.k.to(dev), cc.v.to(dev))
    kvp = _api.KVCache(kp.to(dev), vp.to(dev), table.to(dev))
    seq = torch.from_numpy(wc.seq_len).to(dev)
    oc = torch.empty((len(lens), 16, D), dtype=torch.float32, device=dev)
    op = torch.empty_like(oc)
    for hint in (0, 64, 256):
        api.dr_decode_self_attn(q.to(dev), kvc, seq, oc, max_seq_len_hint=hint)
        api.dr_decode_self_attn(q.to(dev), kvp, seq, op, max_seq_len_hint=hint)
        torch.cuda.synchronize()
        assert torch.equal(oc, op), f"hint {hint}"


def test_deterministic_and_batch_position_invariant(api, cuda_device):
    lens = [300, 12, 1024, 77, 513, 5, 1000, 64] * 5          # 40 rows: the split plan is set by the length
    w, cache, q = ragged_case("paged", lens, 1024, seed=7)
    dev = cuda_device
    kv = to_dev(cache, dev)
    seq = torch.from_numpy(w.seq_len).to(dev)
    o1 = torch.empty((w.B, 16, D), dtype=torch.float32, device=dev)
    o2 = torch.empty_like(o1)
    api.dr_decode_self_attn(q.to(dev), kv, seq, o1)
    api.dr_decode_self_attn(q.to(dev), kv, seq, o2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    perm = torch.from_numpy(np.random.default_rng(8).permutation(w.B))
    kvp = type(kv)(kv.k, kv.v, kv.block_table[perm.to(dev)].contiguous())
    o3 = torch.empty_like(o1)
    api.dr_decode_self_attn(q[perm].contiguous().to(dev), kvp, seq[perm.to(dev)].contiguous(), o3)
    torch.cuda.synchronize()
    assert torch.equal(o3, o1[perm.to(dev)])


def test_cross_attention_ragged_lengths(api, cuda_device):
    B, H, Lc = 6, 16, 300
    enc_len = np.array([1, 16, 17, 150, 299, 300], np.int32)
    w = W.Workload(110, "cross", 1, B, "contiguous", enc_len, Lc, enc_len, Lc, 1.0, 1, 1.0, np.zeros(B, np.uint64),
                   np.zeros(B, np.int32))
    kx, vx = W.make_cross_kv(w, 0)
    q = W.randn_bf16((B, H, D), "cpu", 110, 1)
    dev = cuda_device
    for out_dtype in (torch.float32, torch.bfloat16):
        out = torch.empty((B, H, D), dtype=out_dtype, device=dev)
        api.dr_decode_cross_attn(q.to(dev), kx.to(dev), vx.to(dev), torch.from_numpy(enc_len).to(dev), out)
        ref = oracle.attn_contiguous(W.bits(q), W.bits(kx), W.bits(vx), enc_len, default_scale(D))
        assert_attn_close(out, ref, f"cross {out_dtype}")


# ---------------------------------------------------------------------------
# device-side errors: flagged, clamped or skipped, never a trap
# ---------------------------------------------------------------------------
def test_length_above_capacity_is_clamped_and_flagged(api, cuda_device):
    w, cache, q = ragged_case("contiguous", [64, 64], 64, seed=9)
    dev = cuda_device
    kv = to_dev(cache, dev)
    seq = torch.tensor([64, 500], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((2, 16, D), dtype=torch.float32, device=dev)
    api.dr_decode_self_attn(q.to(dev), kv, seq, out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    assert_attn_close(out, oracle_self(w, cache, q, default_scale(D), lens=np.array([64, 64], np.int32)))


def test_zero_length_row_outputs_zeros_and_is_flagged(api, cuda_device):
    w, cache, q = ragged_case("contiguous", [10, 10], 64, seed=10)
    dev = cuda_device
    kv = to_dev(cache, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.full((2, 16, D), 7.0, dtype=torch.float32, device=dev)
    api.dr_decode_self_attn(q.to(dev), kv, torch.tensor([10, 0], dtype=torch.int32, device=dev), out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    assert torch.count_nonzero(out[1]) == 0
    assert_attn_close(out[0:1], oracle_self(w, cache, q, default_scale(D))[0:1])


def test_block_id_outside_pool_is_skipped_and_flagged(api, cuda_device):
    w, cache, q = ragged_case("paged", [40], 64, seed=11)
    dev = cuda_device
    table = cache.block_table.clone()
    table[0, 1] = cache.num_blocks + 1000          # never dereferenced: the kernel checks it first
    from decode_attention_self_gb300 import api as _api
    kv = _api.KVCache(cache.k.to(dev), cache.v.to(dev), table.to(dev))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((1, 16, D), dtype=torch.float32, device=dev)
    api.dr_decode_self_attn(q.to(dev), kv, torch.tensor([40], dtype=torch.int32, device=dev), out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 2
    # keys 16..31 were skipped: the result is attention over keys 0..15 and 32..39
    kb, vb = W.bits(cache.k), W.bits(cache.v)
    t = cache.block_table.numpy()[0]
    keep = [(t[j // 16], j % 16) for j in list(range(16)) + list(range(32, 40))]
    ref = np.zeros((1, 16, D))
    for h in range(16):
        ks = np.stack([kb[blk, h, s] for blk, s in keep])
        vs = np.stack([vb[blk, h, s] for blk, s in keep])
        ref[0, h] = oracle.attend(W.bits(q)[0, h], ks, vs, default_scale(D))[0]
    assert_attn_close(out, ref)


def test_calls_capture_into_a_cuda_graph(api, cuda_device):
    w, cache, q = ragged_case("paged", [33, 200, 256], 256, seed=12)
    dev = cuda_device
    kv = to_dev(cache, dev)
    seq = torch.from_numpy(w.seq_len).to(dev)
    qd = q.to(dev)
    out_e = torch.empty((w.B, 16, D), dtype=torch.float32, device=dev)
    out_g = torch.empty_like(out_e)
    api.dr_decode_self_attn(qd, kv, seq, out_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            api.dr_decode_self_attn(qd, kv, seq, out_g)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_e, out_g)


def test_two_streams_at_once_give_the_single_stream_bits(api, cuda_device):
    # The library holds no state between calls, so two problems launched on two streams, interleaved and free
    # to run at the same time, give the bits each gives alone.  One problem is small (its whole grid is
    # resident: the pipelined variant, clusters of 8), the other large (2 CTAs per row, 1280 CTAs: the
    # streaming variant, whose split rows merge on an mbarrier).
    dev = cuda_device
    rng = np.random.default_rng(41)
    small = ragged_case("paged", [1500, 300], 2048, seed=41)
    large = ragged_case("contiguous", [int(x) for x in rng.integers(256, 1024, size=40)], 1024, seed=42)
    bf16 = api.DR_KV_BF16
    assert api.dr_plan_splits(2, 16, 2048, bf16, 152) == 8 and api.dr_plan_splits(40, 16, 1024, bf16, 152) == 2
    cases = []
    for w, cache, q in (small, large):
        cases.append((w, cache, q, q.to(dev), to_dev(cache, dev), torch.from_numpy(w.seq_len).to(dev)))
    alone = []
    for w, _, _, qd, kv, seq in cases:
        o = torch.empty((w.B, 16, D), dtype=torch.float32, device=dev)
        api.dr_decode_self_attn(qd, kv, seq, o)
        alone.append(o)
    torch.cuda.synchronize()
    reps = 6
    outs = [[torch.empty_like(o) for _ in range(reps)] for o in alone]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for it in range(reps):
        for i, (_, _, _, qd, kv, seq) in enumerate(cases):
            api.dr_decode_self_attn(qd, kv, seq, outs[i][it], stream=streams[i])
    torch.cuda.synchronize()
    for i in range(2):
        for it in range(reps):
            assert torch.equal(outs[i][it], alone[i]), (i, it)
    for (w, cache, q, *_), o in zip(cases, alone):
        assert_attn_close(o, oracle_self(w, cache, q, default_scale(D)))


def test_row_result_independent_of_batch_and_kernel_variant(api, cuda_device):
    # A row alone (B=1: the whole grid is resident, the pipelined variant runs) and the same row inside a
    # batch of 8 (1024 CTAs, more than 4 per SM: the streaming variant runs) share the split plan (8 CTAs
    # per row for a 2000-key bound), and the two variants do the same arithmetic in the same order: the
    # outputs must be bit-identical.
    from decode_attention_self_gb300 import api as _api
    dev = cuda_device
    lens = [2000] + [int(x) for x in np.random.default_rng(13).integers(1000, 2000, size=7)]
    w, cache, q = ragged_case("paged", lens, 2048, seed=13)
    bf16 = api.DR_KV_BF16
    assert api.dr_plan_splits(1, 16, 2000, bf16, 152) == api.dr_plan_splits(8, 16, 2000, bf16, 152) == 8
    kv = to_dev(cache, dev)
    seq = torch.from_numpy(w.seq_len).to(dev)
    big = torch.empty((w.B, 16, D), dtype=torch.float32, device=dev)
    api.dr_decode_self_attn(q.to(dev), kv, seq, big, max_seq_len_hint=2000)
    one_kv = _api.KVCache(kv.k, kv.v, kv.block_table[:1].contiguous())
    one = torch.empty((1, 16, D), dtype=torch.float32, device=dev)
    api.dr_decode_self_attn(q[:1].contiguous().to(dev), one_kv, seq[:1].contiguous(), one, max_seq_len_hint=2000)
    torch.cuda.synchronize()
    assert torch.equal(one[0], big[0])
    assert_attn_close(big[:2], oracle_self(w, cache, q, default_scale(D))[:2])


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("L", [2047, 2048, 3001, 4096])
def test_wide_clusters_for_few_long_rows(api, cuda_device, layout, L):
    # Batch 1 with rows of 2048 keys or more: 16 CTAs per row, one non-portable cluster, 16 state slots in
    # rank 0.  Rows shorter than the bound leave the last CTAs of their cluster without a tile.
    bf16 = api.DR_KV_BF16
    assert api.dr_plan_splits(1, 16, L, bf16, 152) == 16
    dev = cuda_device
    w, cache, q = ragged_case(layout, [L], 4096, seed=40 + L % 7)
    kv = to_dev(cache, dev)
    seq = torch.from_numpy(w.seq_len).to(dev)
    out = torch.empty((1, 16, D), dtype=torch.float32, device=dev)
    for hint in (L, 4096):
        api.dr_decode_self_attn(q.to(dev), kv, seq, out, max_seq_len_hint=hint)
        assert_attn_close(out, oracle_self(w, cache, q, default_scale(D)), f"{layout} L={L} hint {hint}")
    # and the same row as a description row (dr_decode_cross_attn plans its rows the same way)
    xk, xv = cache.k, cache.v
    if layout == "contiguous":
        api.dr_decode_cross_attn(q.to(dev), xk.to(dev), xv.to(dev), seq, out)
        assert_attn_close(out, oracle_self(w, cache, q, default_scale(D)), f"cross L={L}")


def test_wide_clusters_paged_equals_contiguous_bitwise(api, cuda_device):
    # the 16-CTA split partitions the row by tiles exactly as the 8-CTA one does: the paged layout with a
    # shuffled table reproduces the contiguous result bit for bit
    dev = cuda_device
    lens = [3001]
    wc, cc, q = ragged_case("contiguous", lens, 4096, seed=6)
    wp = W.Workload(106, "edge", 1, 1, "paged", wc.seq_len, 4096, wc.seq_len, 4096, 1.0, 1, 1.0, wc.seeds, wc.steps)
    table, NB = W.make_block_table(wp, "cpu", 6)
    kp = torch.full((NB, 16, 16, D), float("nan"), dtype=torch.bfloat16)
    vp = kp.clone()
    for j in range((lens[0] + 15) // 16):
        kp[table[0, j]] = cc.k[0, :, 16 * j:16 * j + 16]
        vp[table[0, j]] = cc.v[0, :, 16 * j:16 * j + 16]
    from decode_attention_self_gb300 import api as _api
    kvc = _api.KVCache(cc.k.to(dev), cc.v.to(dev))
    kvp = _api.KVCache(kp.to(dev), vp.to(dev), table.to(dev))
    seq = torch.from_numpy(wc.seq_len).to(dev)
    oc = torch.empty((1, 16, D), dtype=torch.float32, device=dev)
    op = torch.empty_like(oc)
    assert api.dr_plan_splits(1, 16, 4096, api.DR_KV_BF16, 152) == 16
    api.dr_decode_self_attn(q.to(dev), kvc, seq, oc, max_seq_len_hint=4096)
    api.dr_decode_self_attn(q.to(dev), kvp, seq, op, max_seq_len_hint=4096)
    torch.cuda.synchronize()
    assert torch.equal(oc, op)


def test_cluster_merge_wait_that_runs_out(api, cuda_device):
    # Test hook: CTA 1 of row 5 (b=0, h=5) never sends its state to the row's rank 0, whose bounded wait for it
    # gives up after about 2 s.  DR_ERRF_TIMEOUT is set, that row's output stays unwritten, every other row is
    # right, and the next ordinary call on the same context is right everywhere.  Batch 32 of 2048 keys:
    # 2 CTAs per row, 1024 CTAs, the streaming variant whose split rows merge through that wait.
    dev = cuda_device
    lens = [2048] * 32
    w, cache, q = ragged_case("paged", lens, 2048, seed=31)
    assert api.dr_plan_splits(32, 16, 2048, api.DR_KV_BF16, 152) == 2
    kv = to_dev(cache, dev)
    seq = torch.from_numpy(w.seq_len).to(dev)
    ref = oracle_self(w, cache, q, default_scale(D))
    out = torch.full((w.B, 16, D), float("nan"), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_decode_self_attn_stall_test(q.to(dev), kv, seq, out, 5, max_seq_len_hint=2048, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & api.DR_ERRF_TIMEOUT
    got = out.cpu().numpy()
    assert np.isnan(got[0, 5]).all()
    keep = np.ones((w.B, 16), bool)
    keep[0, 5] = False
    assert (np.abs(got[keep] - ref[keep]) <= 2e-3).all()
    err.zero_()
    api.dr_decode_self_attn(q.to(dev), kv, seq, out, max_seq_len_hint=2048, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(out, ref, "after the wait that ran out")
