"""GPU parity of dr_embed_tokens and dr_lm_head against the oracle, and of the
chain LM head -> fused sampler (Optimized Parler TTS, "Analysis and
improvements", other optimizations items 1-3).

Tolerances derived from the arithmetic:
  embedding, fp32 out : C fp32 additions -> |err| <= C * 2^-24 * sum_c |e_c| (+ bf16 half-ulp for bf16 out)
  LM head             : a K-term fp32 sum in any order, rounded to nearest or truncated (the tensor-core
                        path's internal order and rounding are not specified)
                        -> |err| <= (K - 1) * 2^-23 * sum_k |h_k w_k|
  LM head -> sampler  : the logits differ from the oracle's by at most that bound, so draws and top-k
                        boundaries closer than 1e-3 (after dividing by T) are not compared.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_self_gb300 import workloads as W

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


@pytest.fixture(scope="module")
def api(cuda_device):
    from decode_attention_self_gb300 import api as _api

    return _api


def vals(b):
    return torch.from_numpy(b.astype(np.int16)).view(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("B,C", [(1, 9), (5, 9), (128, 9), (3, 16), (130, 16), (2, 1)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_embed_tokens(api, cuda_device, B, C, out_dtype):
    # C = 16 is the largest codebook count the call accepts: every one of the 16 rows enters the sum
    dev = cuda_device
    V, Dm = 1088, 1024
    table = W.randn_bf16((C * V, Dm), "cpu", 200, C)
    tokens = torch.from_numpy(np.random.default_rng(B + 1000 * C).integers(0, V, size=(B, C)).astype(np.int32))
    out = torch.empty((B, Dm), dtype=out_dtype, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_embed_tokens(tokens.to(dev), table.to(dev), V, out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.embed_tokens(tokens.numpy(), W.bits(table), V)
    tv = np.abs(vals(W.bits(table)))
    mag = np.stack([sum(tv[c * V + int(tokens[b, c])] for c in range(C)) for b in range(B)])
    tol = C * U * mag + (2.0 ** -8 * np.abs(ref) if out_dtype == torch.bfloat16 else 0)
    assert (np.abs(out.float().cpu().numpy() - ref) <= tol + 1e-30).all()


def test_embed_more_than_16_codebooks_is_refused(api, cuda_device):
    dev = cuda_device
    C, V, Dm = 17, 8, 64
    table = torch.zeros((C * V, Dm), dtype=torch.bfloat16, device=dev)
    tokens = torch.zeros((2, C), dtype=torch.int32, device=dev)
    out = torch.full((2, Dm), 7.0, dtype=torch.float32, device=dev)
    with pytest.raises(RuntimeError, match="unsupported"):
        api.dr_embed_tokens(tokens, table, V, out)
    torch.cuda.synchronize()
    assert (out == 7.0).all()                     # nothing was enqueued


def test_embed_invalid_token_is_left_out_and_flagged(api, cuda_device):
    dev = cuda_device
    C, V, Dm = 3, 16, 64
    table = W.randn_bf16((C * V, Dm), "cpu", 201, 1)
    tokens = torch.tensor([[1, 99, 2], [0, 5, -3]], dtype=torch.int32)
    out = torch.empty((2, Dm), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_embed_tokens(tokens.to(dev), table.to(dev), V, out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 8
    # reference: the same sum with the offending codebook's contribution removed (its rows zeroed)
    tb = W.bits(table).copy()
    tk = tokens.numpy().copy()
    ref = np.zeros((2, Dm))
    for b in range(2):
        t2, tb2 = tk[b:b + 1].copy(), tb.copy()
        for c in range(C):
            if not 0 <= t2[0, c] < V:
                tb2[c * V:(c + 1) * V] = 0
                t2[0, c] = 0
        ref[b] = oracle.embed_tokens(t2, tb2, V)[0]
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=0, atol=1e-5)


@pytest.mark.parametrize("B,K", [
    (1, 1024), (3, 1024), (2, 256), (2, 512), (2, 2048),          # CUDA cores (batch < 4)
    (4, 1024), (15, 1024), (16, 1024), (17, 1024), (32, 2048),    # tensor cores, K split over a 2-CTA cluster
    (33, 1024), (64, 256), (80, 512), (100, 1024), (128, 1024),   # tensor cores, the batch cut in two tiles
    (200, 2048), (256, 768), (300, 1024), (513, 512)])            # tensor cores, several batch tiles
def test_lm_head(api, cuda_device, B, K):
    dev = cuda_device
    C, V, ldv = 9, 1088, 1096
    hidden = W.randn_bf16((B, K), "cpu", 202, B, K)
    Wt = (torch.randn((C * V, K), generator=torch.Generator().manual_seed(K)) * (3.0 / K ** 0.5)).to(torch.bfloat16)
    logits = torch.full((B, C, ldv), float("nan"), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_lm_head(hidden.to(dev), Wt.to(dev), C, logits, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.lm_head(W.bits(hidden), W.bits(Wt)).reshape(B, C, V)
    mag = (np.abs(vals(W.bits(hidden))) @ np.abs(vals(W.bits(Wt))).T).reshape(B, C, V)
    got = logits.cpu().numpy()
    assert np.isnan(got[:, :, V:]).all()                     # padding columns untouched
    assert (np.abs(got[:, :, :V] - ref) <= (K - 1) * 2 * U * mag + 1e-30).all()


def test_lm_head_more_slabs_than_sms(api, cuda_device):
    # 16 codebooks of 2048: 256 weight slabs of 128 rows, more than the SMs, so a batch of 64 stays one tile
    # (no batch split) and the grid runs at two CTAs per SM.
    dev = cuda_device
    B, K, C, V = 64, 512, 16, 2048
    hidden = W.randn_bf16((B, K), "cpu", 204, B, K)
    Wt = (torch.randn((C * V, K), generator=torch.Generator().manual_seed(9)) * (3.0 / K ** 0.5)).to(torch.bfloat16)
    logits = torch.full((B, C, V), float("nan"), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_lm_head(hidden.to(dev), Wt.to(dev), C, logits, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.lm_head(W.bits(hidden), W.bits(Wt)).reshape(B, C, V)
    mag = (np.abs(vals(W.bits(hidden))) @ np.abs(vals(W.bits(Wt))).T).reshape(B, C, V)
    assert (np.abs(logits.cpu().numpy() - ref) <= (K - 1) * 2 * U * mag + 1e-30).all()


def test_lm_head_feeding_the_sampler(api, cuda_device):
    dev = cuda_device
    B, K, C, V, T, k = 4, 1024, 9, 1088, 0.9, 50
    hidden = W.randn_bf16((B, K), "cpu", 203, 1)
    Wt = (torch.randn((C * V, K), generator=torch.Generator().manual_seed(5)) * (3.0 / K ** 0.5)).to(torch.bfloat16)
    logits = torch.empty((B, C, V), dtype=torch.float32, device=dev)
    seeds = np.arange(B, dtype=np.uint64) + 7
    steps = np.array([3, 9, 20, 50], np.int32)
    tokens = torch.empty((B, C), dtype=torch.int32, device=dev)
    probs = torch.empty((B, C, V), dtype=torch.float32, device=dev)
    api.dr_lm_head(hidden.to(dev), Wt.to(dev), C, logits)
    api.dr_sample_topk_delayed(logits, T, k, torch.from_numpy(seeds.view(np.int64)).to(dev),
                               torch.from_numpy(steps).to(dev), 1024, tokens, probs)
    torch.cuda.synchronize()
    ref_logits = oracle.lm_head(W.bits(hidden), W.bits(Wt)).reshape(B, C, V).astype(np.float32)
    ref = oracle.sample(ref_logits, T, k, seeds, steps, 1024, want_probs=True)
    got_t = tokens.cpu().numpy()
    cmp = ref["margins"] >= 1e-3
    assert cmp.sum() > 20 and (got_t[cmp] == ref["tokens"][cmp]).all()
    # top-k sets, except rows whose k-th / (k+1)-th scaled logits are closer than 1e-3
    x = ref_logits / np.float32(T)
    srt = -np.sort(-x, axis=2)
    clear = (srt[:, :, k - 1] - srt[:, :, k]) >= 1e-3
    sup_g, sup_r = probs.cpu().numpy() != 0, ref["probs"] != 0
    for b in range(B):
        for c in range(C):
            if clear[b, c] and steps[b] > c:
                assert np.array_equal(sup_g[b, c], sup_r[b, c]), (b, c)


@pytest.mark.parametrize("B", [16, 128])   # K split over a 2-CTA cluster; two batch tiles, K whole
def test_lm_head_wait_that_runs_out(api, cuda_device, B):
    # Test hook: the CTAs of weight slab 5 (logit rows 640..767) never load their first K chunk, so their bounded
    # pipeline wait gives up after about 2 s.  DR_ERRF_TIMEOUT is set, those logits stay unwritten, every other
    # logit is right, and the next ordinary call on the same context is right everywhere.
    dev = cuda_device
    K, C, V = 1024, 9, 1088
    hidden = W.randn_bf16((B, K), "cpu", 205, B)
    Wt = (torch.randn((C * V, K), generator=torch.Generator().manual_seed(11)) * (3.0 / K ** 0.5)).to(torch.bfloat16)
    ref = oracle.lm_head(W.bits(hidden), W.bits(Wt))
    mag = np.abs(vals(W.bits(hidden))) @ np.abs(vals(W.bits(Wt))).T
    tol = (K - 1) * 2 * U * mag + 1e-30
    hd, wd = hidden.to(dev), Wt.to(dev)
    logits = torch.full((B, C, V), float("nan"), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dr_lm_head_stall_test(hd, wd, C, logits, 5, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & api.DR_ERRF_TIMEOUT
    got = logits.cpu().numpy().reshape(B, C * V)
    stalled = np.zeros(C * V, bool)
    stalled[640:768] = True
    assert np.isnan(got[:, stalled]).all()
    assert (np.abs(got[:, ~stalled] - ref[:, ~stalled]) <= tol[:, ~stalled]).all()
    err.zero_()
    api.dr_lm_head(hd, wd, C, logits, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert (np.abs(logits.cpu().numpy().reshape(B, C * V) - ref) <= tol).all()
