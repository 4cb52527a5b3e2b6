"""The long-output workload end to end: 2048 consecutive decode steps of a
24-layer decoder at batch 1 (Optimized Parler TTS, "Speeding up Parler TTS
decoder": 2048 tokens decoded from a 64-token input).

Each step t appends k/v at position t of every layer's 4096-slot static
cache, attends t+1 keys, attends the 64 description keys, and samples nine
codebooks at step t (the device step counter advances inside the sampler, so
no host synchronisation is needed between steps).  Every step's tokens are
compared with the oracle; attention outputs of every layer are compared at
steps 0, 1, 15, 16, 17, 1023 and 2047.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_self_gb300 import workloads as W
from tests.parity import assert_attn_close, assert_tokens_match, default_scale

pytestmark = pytest.mark.gpu

CHECK_STEPS = (0, 1, 15, 16, 17, 1023, 2047)


def test_long_output_2048_steps(cuda_device):
    from decode_attention_self_gb300 import api

    dev = cuda_device
    w = W.make_workload(3)
    T, Lyr, H, D, cap = w.n_steps, w.layers, w.H, w.D, w.cap
    scale = default_scale(D)

    # host streams (seeded), then one copy each to the device
    q_h = [W.randn_bf16((T, 1, H, D), "cpu", 3, l, 40) for l in range(Lyr)]
    qx_h = [W.randn_bf16((T, 1, H, D), "cpu", 3, l, 41) for l in range(Lyr)]
    kn_h = [W.randn_bf16((T, 1, H, D), "cpu", 3, l, 42) for l in range(Lyr)]
    vn_h = [W.randn_bf16((T, 1, H, D), "cpu", 3, l, 43) for l in range(Lyr)]
    cross_h = [W.make_cross_kv(w, l) for l in range(Lyr)]
    logits_h = torch.stack([W.make_logits(w, step_key=t) for t in range(T)])       # [T, 1, 9, 1088]

    q_d = [x.to(dev) for x in q_h]
    qx_d = [x.to(dev) for x in qx_h]
    kn_d = [x.to(dev) for x in kn_h]
    vn_d = [x.to(dev) for x in vn_h]
    cross_d = [(k.to(dev), v.to(dev)) for k, v in cross_h]
    logits_d = logits_h.to(dev)
    caches = [api.KVCache(torch.full((1, H, cap, D), float("nan"), dtype=torch.bfloat16, device=dev),
                          torch.full((1, H, cap, D), float("nan"), dtype=torch.bfloat16, device=dev))
              for _ in range(Lyr)]
    positions = torch.arange(T, dtype=torch.int32, device=dev)
    lengths = torch.arange(1, T + 1, dtype=torch.int32, device=dev)
    enc = torch.from_numpy(w.enc_len).to(dev)
    seeds = torch.from_numpy(w.seeds.view(np.int64)).to(dev)
    step = torch.zeros(1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out_s = torch.empty((Lyr, 1, H, D), dtype=torch.float32, device=dev)
    out_x = torch.empty_like(out_s)
    tokens = torch.empty((T, 1, w.C), dtype=torch.int32, device=dev)
    saved = {}

    for t in range(T):
        for l in range(Lyr):
            api.dr_kv_append(caches[l], kn_d[l][t], vn_d[l][t], positions[t:t + 1], err_flag=err)
            api.dr_decode_self_attn(q_d[l][t], caches[l], lengths[t:t + 1], out_s[l], err_flag=err)
            api.dr_decode_cross_attn(qx_d[l][t], cross_d[l][0], cross_d[l][1], enc, out_x[l], err_flag=err)
        api.dr_sample_topk_delayed(logits_d[t], w.temperature, w.top_k, seeds, step, w.pad_id, tokens[t],
                                   advance=True)
        if t in CHECK_STEPS:
            saved[t] = (out_s.cpu(), out_x.cpu())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert int(step.item()) == T

    # tokens of every step
    got = tokens.cpu().numpy()
    for t in range(T):
        ref = oracle.sample(logits_h[t].numpy(), w.temperature, w.top_k, w.seeds, np.array([t], np.int32), w.pad_id)
        assert_tokens_match(got[t], ref, f"tokens at step {t}")
        assert ((got[t, 0] == w.pad_id) | (np.arange(w.C) < t)).all()

    # attention of every layer at the sampled steps
    for t in CHECK_STEPS:
        gs, gx = saved[t]
        for l in range(Lyr):
            ks, vs = W.bits(kn_h[l][: t + 1, 0]), W.bits(vn_h[l][: t + 1, 0])     # [t+1, H, D]
            qb, qxb = W.bits(q_h[l][t, 0]), W.bits(qx_h[l][t, 0])
            kx, vx = W.bits(cross_h[l][0][0]), W.bits(cross_h[l][1][0])          # [H, Lc, D]
            ref_s = np.stack([oracle.attend(qb[h], np.ascontiguousarray(ks[:, h]), np.ascontiguousarray(vs[:, h]),
                                            scale)[0] for h in range(H)])
            ref_x = np.stack([oracle.attend(qxb[h], np.ascontiguousarray(kx[h, :64]), np.ascontiguousarray(vx[h, :64]),
                                            scale)[0] for h in range(H)])
            assert_attn_close(gs[l, 0], ref_s, f"self-attention layer {l} step {t}")
            assert_attn_close(gx[l, 0], ref_x, f"cross-attention layer {l} step {t}")
