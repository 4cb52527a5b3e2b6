"""GPU parity of dr_sample_topk_delayed against the oracle.

The fused sampler (Optimized Parler TTS, "Future work" item 2: temperature,
top-k and softmax in one kernel; the nine codebooks under the delayed pattern,
architecture overview): tokens bit-exact outside the Gumbel-margin exclusion,
top-k sets bit-exact (ties to the lower index), probabilities within fp32
tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_self_gb300 import workloads as W
from tests.parity import assert_probs_match, assert_tokens_match

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_device):
    from decode_attention_self_gb300 import api as _api

    return _api


def run_gpu(api, dev, logits, T, k, seeds, steps, pad_id, V=None, want_probs=True, advance=False):
    B, C, ldv = logits.shape
    V = ldv if V is None else V
    lg = torch.as_tensor(logits).to(dev)
    sd = torch.from_numpy(np.asarray(seeds, np.uint64).view(np.int64)).to(dev)
    st = torch.from_numpy(np.asarray(steps, np.int32).copy()).to(dev)
    tok = torch.full((B, C), -7, dtype=torch.int32, device=dev)
    pr = torch.full((B, C, V), -1.0, dtype=torch.float32, device=dev) if want_probs else None
    api.dr_sample_topk_delayed(lg, T, k, sd, st, pad_id, tok, pr, V=V, advance=advance)
    torch.cuda.synchronize()
    return tok, pr, st


def check(api, dev, logits, T, k, seeds, steps, pad_id, V=None):
    x = np.asarray(logits, np.float32)
    tok, pr, _ = run_gpu(api, dev, x, T, k, seeds, steps, pad_id, V=V)
    ref = oracle.sample(x, T, k, seeds, steps, pad_id, V=V, want_probs=True)
    n_cmp, n_excl = assert_tokens_match(tok, ref)
    assert_probs_match(pr, ref)
    return n_cmp, n_excl


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_workload_sampler_parity(api, cuda_device, index):
    w = W.make_workload(index)
    logits = W.make_logits(w).numpy()
    n_cmp, n_excl = check(api, cuda_device, logits, w.temperature, w.top_k, w.seeds, w.steps, w.pad_id, V=w.V)
    assert n_cmp > 0 and n_excl <= max(1, n_cmp // 100)


def test_many_steps_and_seeds(api, cuda_device):
    rng = np.random.default_rng(1)
    B = 64
    logits = (rng.normal(size=(B, 9, 1088)) * 3).astype(np.float32)
    seeds = rng.integers(0, 2 ** 63, size=B, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    steps = rng.integers(0, 5000, size=B).astype(np.int32)
    check(api, cuda_device, logits, 1.0, 50, seeds, steps, 1024)


@pytest.mark.parametrize("V", [1, 5, 64, 65, 256, 257, 512, 513, 1088, 1089, 2048])
def test_vocab_sizes(api, cuda_device, V):
    rng = np.random.default_rng(V)
    logits = (rng.normal(size=(3, 9, V)) * 2).astype(np.float32)
    for k in sorted({1, min(V, 7), min(V, 50), V}):
        check(api, cuda_device, logits, 0.9, k, np.array([5, 6, 7], np.uint64), np.array([9, 9, 9], np.int32), 3)


@pytest.mark.parametrize("C", [1, 4, 9, 16])
def test_codebook_counts(api, cuda_device, C):
    rng = np.random.default_rng(C)
    logits = (rng.normal(size=(2, C, 300)) * 3).astype(np.float32)
    check(api, cuda_device, logits, 1.3, 20, np.array([1, 2], np.uint64), np.array([C + 1, C // 2], np.int32), 7)


def test_row_stride_padding_is_never_read(api, cuda_device):
    rng = np.random.default_rng(2)
    x = np.full((4, 9, 1096), np.nan, np.float32)
    x[:, :, :1088] = rng.normal(size=(4, 9, 1088)) * 3
    check(api, cuda_device, x, 1.0, 50, np.arange(4, dtype=np.uint64), np.full(4, 20, np.int32), 1024, V=1088)


def test_planted_ties_at_the_topk_boundary(api, cuda_device):
    rng = np.random.default_rng(3)
    B, V, k = 16, 1088, 250
    x = (rng.normal(size=(B, 9, V)) * 5).astype(np.float32)
    for b in range(B):
        for c in range(9):
            row = x[b, c]
            kth = np.argsort(-row, kind="stable")[k - 1]
            idx = rng.choice(V, size=20, replace=False)
            row[idx] = row[kth]                        # 21 entries share the boundary value
    check(api, cuda_device, x, 0.7, k, np.arange(B, dtype=np.uint64) + 99, np.full(B, 15, np.int32), 1024)


@pytest.mark.parametrize("k", [1, 2, 7, 50, 250, 1000, 1088])
def test_few_distinct_values(api, cuda_device, k):
    # Logits drawn from 12 distinct values, two of them equal in their first 16 bits: the bin of the
    # top_k-th key often holds many equal keys, so the radix select ends at different passes, both with
    # the bin kept whole and with the equal keys ranked by index.
    rng = np.random.default_rng(k)
    vals = np.array([-3.5, -1.25, -1.0, -0.5, 0.0, 0.125, 0.5, 1.0, 1.5, 2.0, 2.0078125, 4.0], np.float32)
    logits = vals[rng.integers(0, len(vals), size=(6, 9, 1088))]
    check(api, cuda_device, logits, 1.0, k, np.arange(6, dtype=np.uint64) + 11, np.full(6, 20, np.int32), 1024)


@pytest.mark.parametrize("k", [1, 7, 20, 40])
def test_signed_zeros_tie_by_index(api, cuda_device, k):
    # -0.0 and +0.0 are equal values: at the top-k boundary they tie and the lower index wins, whatever the
    # sign bit (the kernel's order keys must not separate them).
    rng = np.random.default_rng(70 + k)
    vals = np.array([-0.0, 0.0, -0.0, 0.0, 1.0, -1.0, -np.inf], np.float32)
    logits = vals[rng.choice(len(vals), size=(4, 9, 64), p=[0.3, 0.3, 0.15, 0.15, 0.04, 0.04, 0.02])]
    check(api, cuda_device, logits, 1.0, k, np.arange(4, dtype=np.uint64) + 3, np.full(4, 20, np.int32), 63)


def test_all_equal_logits_take_the_first_k(api, cuda_device):
    x = np.zeros((2, 9, 1088), np.float32)
    tok, pr, _ = run_gpu(api, cuda_device, x, 1.0, 50, np.array([1, 2], np.uint64), np.array([20, 20], np.int32), 5)
    support = (pr.cpu().numpy() != 0)
    assert (support[:, :, :50]).all() and not support[:, :, 50:].any()
    check(api, cuda_device, x, 1.0, 50, np.array([1, 2], np.uint64), np.array([20, 20], np.int32), 5)


def test_negative_infinity_logits(api, cuda_device):
    rng = np.random.default_rng(4)
    x = (rng.normal(size=(3, 9, 200)) * 2).astype(np.float32)
    x[0, :, :] = -np.inf                               # whole rows -inf: the lowest index of the set
    x[1, :, 150:] = -np.inf                            # k larger than the finite count
    x[2, :, ::3] = -np.inf
    check(api, cuda_device, x, 1.0, 170, np.array([1, 2, 3], np.uint64), np.full(3, 12, np.int32), 9)
    check(api, cuda_device, x, 1.0, 1, np.array([1, 2, 3], np.uint64), np.full(3, 12, np.int32), 9)


def test_k1_is_argmax(api, cuda_device):
    rng = np.random.default_rng(5)
    x = rng.integers(-4, 4, size=(8, 9, 1088)).astype(np.float32)   # many exact ties
    tok, _, _ = run_gpu(api, cuda_device, x, 1.0, 1, np.arange(8, dtype=np.uint64), np.full(8, 50, np.int32), 0)
    assert np.array_equal(tok.cpu().numpy(), x.argmax(axis=2))


@pytest.mark.parametrize("step", list(range(0, 11)))
def test_delay_pattern(api, cuda_device, step):
    rng = np.random.default_rng(step)
    x = (rng.normal(size=(2, 9, 1088)) * 3).astype(np.float32)
    x[:, :, 1024] = -np.inf
    tok, pr, _ = run_gpu(api, cuda_device, x, 1.0, 50, np.array([0, 1], np.uint64), np.array([step, step], np.int32),
                         1024)
    t = tok.cpu().numpy()
    for c in range(9):
        assert ((t[:, c] == 1024) == (step <= c)).all()
        if step <= c:
            assert (pr[:, c].cpu().numpy() == 0).all()
    check(api, cuda_device, x, 1.0, 50, np.array([0, 1], np.uint64), np.array([step, step], np.int32), 1024)


def test_advance_flag_increments_step_once_per_call(api, cuda_device):
    rng = np.random.default_rng(6)
    B = 5
    x = (rng.normal(size=(B, 9, 1088)) * 3).astype(np.float32)
    steps0 = np.array([0, 3, 8, 9, 100], np.int32)
    seeds = np.arange(B, dtype=np.uint64)
    dev = cuda_device
    lg = torch.from_numpy(x).to(dev)
    sd = torch.from_numpy(seeds.view(np.int64)).to(dev)
    st = torch.from_numpy(steps0.copy()).to(dev)
    tok = torch.empty((B, 9), dtype=torch.int32, device=dev)
    for it in range(3):
        api.dr_sample_topk_delayed(lg, 1.0, 50, sd, st, 1024, tok, advance=True)
        torch.cuda.synchronize()
        ref = oracle.sample(x, 1.0, 50, seeds, steps0 + it, 1024)
        assert_tokens_match(tok, ref)
        assert np.array_equal(st.cpu().numpy(), steps0 + it + 1)


@pytest.mark.parametrize("V", [5, 257, 1088, 2048])
def test_large_grid(api, cuda_device, V):
    # 128 rows x 9 codebooks: more CTAs than the GPU holds at once at 256 threads, so the sampler runs
    # 128-thread CTAs (each thread keeps twice the keys).  Half the rows draw from few distinct values, so
    # the top-k boundary ties and the radix select ends at different passes.
    rng = np.random.default_rng(300 + V)
    B = 128
    x = (rng.normal(size=(B, 9, V)) * 3).astype(np.float32)
    vals = np.array([-2.0, -0.5, 0.0, 0.5, 1.0, 1.0078125, 3.0], np.float32)
    x[::2] = vals[rng.integers(0, len(vals), size=(B // 2, 9, V))]
    steps = rng.integers(0, 12, size=B).astype(np.int32)
    for k in sorted({1, min(V, 50), min(V, 250), V}):
        check(api, cuda_device, x, 0.8, k, np.arange(B, dtype=np.uint64) + 5, steps, V - 1)


def test_advance_flag_large_grid(api, cuda_device):
    rng = np.random.default_rng(7)
    B = 128
    x = (rng.normal(size=(B, 9, 1088)) * 3).astype(np.float32)
    steps0 = rng.integers(0, 20, size=B).astype(np.int32)
    seeds = np.arange(B, dtype=np.uint64) + 1
    dev = cuda_device
    lg = torch.from_numpy(x).to(dev)
    sd = torch.from_numpy(seeds.view(np.int64)).to(dev)
    st = torch.from_numpy(steps0.copy()).to(dev)
    tok = torch.empty((B, 9), dtype=torch.int32, device=dev)
    for it in range(2):
        api.dr_sample_topk_delayed(lg, 1.0, 50, sd, st, 1024, tok, advance=True)
        torch.cuda.synchronize()
        ref = oracle.sample(x, 1.0, 50, seeds, steps0 + it, 1024)
        assert_tokens_match(tok, ref)
        assert np.array_equal(st.cpu().numpy(), steps0 + it + 1)


def test_deterministic(api, cuda_device):
    w = W.make_workload(5)
    x = W.make_logits(w).numpy()
    a, pa, _ = run_gpu(api, cuda_device, x, w.temperature, w.top_k, w.seeds, w.steps, w.pad_id)
    b, pb, _ = run_gpu(api, cuda_device, x, w.temperature, w.top_k, w.seeds, w.steps, w.pad_id)
    assert torch.equal(a, b) and torch.equal(pa, pb)


@pytest.mark.parametrize("C", [1, 2, 16])
def test_advance_flag_every_cluster_shape(api, cuda_device, C):
    # DR_SAMPLE_ADVANCE makes each row's C codebook CTAs one cluster: none for C = 1, two CTAs, and a
    # non-portable cluster of 16
    rng = np.random.default_rng(40 + C)
    B = 6
    x = (rng.normal(size=(B, C, 700)) * 3).astype(np.float32)
    steps0 = np.array([0, 1, C - 1, C, C + 5, 1000], np.int32)
    seeds = np.arange(B, dtype=np.uint64) * np.uint64(977) + np.uint64(3)
    dev = cuda_device
    lg = torch.from_numpy(x).to(dev)
    sd = torch.from_numpy(seeds.view(np.int64)).to(dev)
    st = torch.from_numpy(steps0.copy()).to(dev)
    tok = torch.empty((B, C), dtype=torch.int32, device=dev)
    for it in range(3):
        api.dr_sample_topk_delayed(lg, 1.1, 30, sd, st, 700, tok, advance=True)
        torch.cuda.synchronize()
        ref = oracle.sample(x, 1.1, 30, seeds, steps0 + it, 700)
        assert_tokens_match(tok, ref, f"C={C} call {it}")
        assert np.array_equal(st.cpu().numpy(), steps0 + it + 1)


def test_positive_infinity_and_a_tiny_temperature(api, cuda_device):
    # x = logit / T at +inf (an infinite logit, or T so small that the division overflows): the +inf entries
    # lead the top-k set (ties to the lower index) and each perturbed score x - log(-log u) of them is +inf,
    # so the token is the lowest-index +inf entry; the probabilities are undefined there and not compared.
    dev = cuda_device
    rng = np.random.default_rng(50)
    B, C, V = 4, 9, 300
    x = (rng.normal(size=(B, C, V)) * 3).astype(np.float32)
    for b in range(B):
        for c in range(C):
            x[b, c, rng.choice(V, size=1 + (b + c) % 4, replace=False)] = np.inf
    seeds, steps = np.arange(B, dtype=np.uint64), np.full(B, 20, np.int32)
    first_inf = np.argmax(np.isinf(x) & (x > 0), axis=2)
    for k in (1, 2, 50, V):
        tok, _, _ = run_gpu(api, dev, x, 1.0, k, seeds, steps, 1024, want_probs=False)
        ref = oracle.sample(x, 1.0, k, seeds, steps, 1024)
        assert np.array_equal(tok.cpu().numpy(), first_inf) and np.array_equal(ref["tokens"], first_inf), k
    # a subnormal temperature: y / T overflows to +-inf for every |y| above 3.4e38 * T (binary32 division)
    T = np.float32(1e-44)
    y = rng.normal(size=(B, C, V)).astype(np.float32)
    with np.errstate(over="ignore"):
        xs = y / T
    assert (np.isinf(xs) & (xs > 0)).any(axis=2).all()
    first = np.argmax(np.isinf(xs) & (xs > 0), axis=2)
    tok, _, _ = run_gpu(api, dev, y, float(T), 50, seeds, steps, 1024, want_probs=False)
    ref = oracle.sample(y, float(T), 50, seeds, steps, 1024)
    assert np.array_equal(tok.cpu().numpy(), first) and np.array_equal(ref["tokens"], first)


@pytest.mark.parametrize("k", [1, 3, 50])
def test_nan_logits_token_stays_in_range(api, cuda_device, k):
    # NaN logits have no defined draw (the oracle refuses them), but the token must stay inside [0, V): a NaN
    # order key sorts above +inf, so with top_k = 1 the kept set can be a NaN entry alone, and then every
    # perturbed score of the set is NaN.
    rng = np.random.default_rng(80 + k)
    B, C, V = 3, 9, 300
    x = (rng.normal(size=(B, C, V)) * 3).astype(np.float32)
    x[0, :, 17] = np.nan                               # one NaN per row
    x[1, :, ::50] = np.nan                             # several
    x[2, :, :] = np.nan                                # all of them
    tok, _, _ = run_gpu(api, cuda_device, x, 1.0, k, np.arange(B, dtype=np.uint64), np.full(B, 20, np.int32),
                        1024, want_probs=False)
    t = tok.cpu().numpy()
    assert ((t >= 0) & (t < V)).all(), t


@pytest.mark.parametrize("k", [1, 13, 50, 64, 70])
def test_order_keys_across_every_float_class(api, cuda_device, k):
    # The radix select orders the logits through a float -> uint32 key map.  Here 64 entries of each row lie in
    # [0.5, 30] and the rest are random bit patterns of every other class -- negative values of every exponent,
    # -inf, subnormals of both signs, +-0 and tiny positives -- so the first radix pass sees keys in every bin.
    # The top 64 are the band; k = 70 takes six more from the background's largest, which are planted tiny
    # non-negative values (zeros and subnormals, so also ties), and stay within fp32's exp range of the maximum.
    rng = np.random.default_rng(90 + k)
    B, C, V = 4, 9, 1088
    bits = rng.integers(0, 2 ** 32, size=(B, C, V), dtype=np.uint64).astype(np.uint32)
    bg = bits.view(np.float32).copy()
    bad = ~np.isfinite(bg) | (bg > 1e-30)
    bg[bad] = -np.abs(np.where(np.isnan(bg[bad]), 1.0, bg[bad]))        # background: every float <= 1e-30
    x = bg
    for b in range(B):
        for c in range(C):
            pos = rng.choice(V, size=64 + 10 + 3, replace=False)
            x[b, c, pos[:64]] = rng.uniform(0.5, 30.0, size=64).astype(np.float32)
            x[b, c, pos[64:74]] = np.array([0.0, -0.0, 0.0, 1e-45, 3e-39, 1e-38, 1e-40, -0.0, 0.0, 2e-45],
                                           np.float32)
            x[b, c, pos[74:]] = -np.inf
    assert np.isfinite(x[x > 0]).all() and not np.isnan(x).any()
    check(api, cuda_device, x, 1.0, k, np.arange(B, dtype=np.uint64) + 3, np.full(B, 20, np.int32), 5)
