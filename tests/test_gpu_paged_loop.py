"""A batch decoding several consecutive steps through the whole path, the way a
decoder uses it: per step and layer one fused launch (append at the row's
position, self-attention, cross-attention), then the sampler with the device
step counter advancing, then the merged embedding lookup of the drawn tokens
(the next step's input).  Rows start at different lengths in a paged cache
(e4m3 for some layers, bf16 for others); nothing is synchronised with the
host between steps.  Every step's tokens, every layer's attention at the last
step and the final caches are compared with the oracle."""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_self_gb300 import workloads as W
from tests.parity import assert_attn_close, assert_tokens_match, default_scale

pytestmark = pytest.mark.gpu
D, H, C, V = 64, 16, 9, 1088


def test_paged_batch_decode_loop(cuda_device):
    from decode_attention_self_gb300 import api

    dev = cuda_device
    B, layers, steps, T, k, pad = 6, 3, 12, 0.8, 40, 1024
    start = np.array([1, 15, 16, 100, 499, 1023], np.int32)          # keys already cached per row
    final = start + steps
    w = W.Workload(400, "loop", layers, B, "paged", final, 1040, np.array([5, 60, 33, 256, 1, 77], np.int32), 256,
                   T, k, 3.0, np.arange(B, dtype=np.uint64) * 3 + 1, np.array([0, 2, 8, 9, 30, 3], np.int32))
    fp8_layer = [False, True, False]
    caches, hosts = [], []
    for l in range(layers):
        c = (W.make_self_cache_fp8 if fp8_layer[l] else W.make_self_cache)(w, l, filled_len=start)
        hosts.append(c)
        caches.append(api.KVCache(c.k.to(dev), c.v.to(dev), c.block_table.to(dev), c.k_scale, c.v_scale))
    cross = [W.make_cross_kv(w, l) for l in range(layers)]
    qs = [[W.make_step_inputs(w, l, step_key=t) for l in range(layers)] for t in range(steps)]
    logits = [W.make_logits(w, step_key=t) for t in range(steps)]
    emb_table = W.randn_bf16((C * V, 128), "cpu", 400, 9)

    seq = torch.from_numpy(start + 1).to(dev)                         # length after this step's append
    one = torch.ones(B, dtype=torch.int32, device=dev)
    enc = torch.from_numpy(w.enc_len).to(dev)
    step = torch.from_numpy(w.steps.copy()).to(dev)
    seeds = torch.from_numpy(w.seeds.view(np.int64)).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    tokens = torch.empty((steps, B, C), dtype=torch.int32, device=dev)
    outs = torch.empty((layers, 2, B, H, D), dtype=torch.float32, device=dev)
    emb = torch.empty((steps, B, 128), dtype=torch.float32, device=dev)
    cross_d = [(kx.to(dev), vx.to(dev)) for kx, vx in cross]
    emb_d = emb_table.to(dev)
    lg_d = [x.to(dev) for x in logits]
    qs_d = [[tuple(t.to(dev) for t in qs[s][l]) for l in range(layers)] for s in range(steps)]
    for s in range(steps):
        for l in range(layers):
            q, qx, kn, vn = qs_d[s][l]
            api.dr_decode_layer(q, caches[l], kn, vn, seq, qx, cross_d[l][0], cross_d[l][1], enc, outs[l, 0],
                                outs[l, 1], max_seq_len_hint=1040, err_flag=err)
        api.dr_sample_topk_delayed(lg_d[s], T, k, seeds, step, pad, tokens[s], advance=True)
        api.dr_embed_tokens(tokens[s], emb_d, V, emb[s], err_flag=err)
        seq += one                                                    # the caller's position bookkeeping
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(step.cpu().numpy(), w.steps + steps)

    # oracle replay
    scale = default_scale(D)
    kh = [W.bits(c.k).copy() if not fp8_layer[l] else c.k.numpy().copy() for l, c in enumerate(hosts)]
    vh = [W.bits(c.v).copy() if not fp8_layer[l] else c.v.numpy().copy() for l, c in enumerate(hosts)]
    tables = [c.block_table.numpy() for c in hosts]
    got_tok = tokens.cpu().numpy()
    for s in range(steps):
        lens = start + 1 + s
        for l in range(layers):
            q, qx, kn, vn = qs[s][l]
            c = hosts[l]
            if fp8_layer[l]:
                oracle.kv_append_fp8_paged(kh[l], vh[l], tables[l], W.bits(kn), W.bits(vn), lens - 1, c.k_scale,
                                           c.v_scale)
            else:
                oracle.kv_append_paged(kh[l], vh[l], tables[l], W.bits(kn), W.bits(vn), lens - 1)
        ref = oracle.sample(logits[s].numpy(), T, k, w.seeds, w.steps + s, pad)
        assert_tokens_match(got_tok[s], ref, f"tokens at step {s}")
        # next-step input from the oracle's tokens, on the rows whose draws all matched
        ref_emb = oracle.embed_tokens(ref["tokens"], W.bits(emb_table), V)
        same = (got_tok[s] == ref["tokens"]).all(axis=1)
        np.testing.assert_allclose(emb[s].cpu().numpy()[same], ref_emb[same], rtol=0, atol=1e-4)
    lens = start + steps
    for l in range(layers):
        q, qx, _, _ = qs[steps - 1][l]
        c = hosts[l]
        if fp8_layer[l]:
            ref_s = oracle.attn_fp8_paged(W.bits(q), kh[l], vh[l], tables[l], lens, scale, c.k_scale, c.v_scale)
            assert np.array_equal(caches[l].k.cpu().numpy(), kh[l]) and np.array_equal(caches[l].v.cpu().numpy(), vh[l])
        else:
            ref_s = oracle.attn_paged(W.bits(q), kh[l], vh[l], tables[l], lens, scale)
            assert np.array_equal(W.bits(caches[l].k), kh[l]) and np.array_equal(W.bits(caches[l].v), vh[l])
        assert_attn_close(outs[l, 0], ref_s, f"self-attention layer {l} at the last step")
        ref_x = oracle.attn_contiguous(W.bits(qx), W.bits(cross[l][0]), W.bits(cross[l][1]), w.enc_len, scale)
        assert_attn_close(outs[l, 1], ref_x, f"cross-attention layer {l} at the last step")
