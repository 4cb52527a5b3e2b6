"""Seeded synthetic inputs for the decode-step workloads.

This module only draws random numbers and lays them out; it holds none of the
decode step's arithmetic.  Both the CUDA library's tests/bench and the CPU
oracle take their inputs from here, so the two sides see identical bits.

Recipe (all seeded, no trained weights, no dataset):
  * q, k, v (self and cross) ~ N(0, 1) drawn in float32, rounded to bf16 (RNE);
  * every cache slot that is not valid (past a row's length, spare paged
    blocks, the slot the step's append will fill) holds bf16 NaN (0x7FC0),
    so a read outside the valid range poisons the output;
  * paged caches use block size 16 and a seeded random permutation of the
    pool's blocks; table entries past a row's last block are -1;
  * logits ~ N(0, sigma^2) in float32; the stress workload plants exact ties,
    two of them on the row's top_k-th largest value.

The five workloads follow the decode step of a Parler-TTS / MusicGen decoder
(16 heads x head_dim 64, 9 codebooks x 1088 logits):
  1  one layer, B=1, self length 64 in a 2048-slot static cache, cross 64;
  2  24 layers, B=1, self 1024 of 4096, cross 1024 (long description);
  3  24 layers, B=1, 2048 consecutive steps, cross 64 (long output);
  4  24 layers, B=32 ragged, paged, self U{64..2048}, cross U{32..512};
  5  24 layers, B=128 ragged, paged, self U{512..4096}, cross 256, ties.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

H_DEFAULT = 16
D_DEFAULT = 64
BLOCK = 16
BF16_NAN_BITS = 0x7FC0


@dataclasses.dataclass
class Workload:
    """Shapes and per-row parameters of one decode-step workload (host arrays)."""

    index: int
    name: str
    layers: int
    B: int
    layout: str                 # "contiguous" or "paged" (self-attention cache)
    seq_len: np.ndarray         # [B] int32, valid self-attention keys after this step's append
    cap: int                    # keys one row of the self cache can hold
    enc_len: np.ndarray         # [B] int32, description (cross) length of each row
    Lc_max: int                 # capacity of the cross K/V rows
    temperature: float
    top_k: int
    logit_std: float
    seeds: np.ndarray           # [B] uint64 Philox seeds
    steps: np.ndarray           # [B] int32 decode step of each row
    H: int = H_DEFAULT
    D: int = D_DEFAULT
    C: int = 9
    V: int = 1088
    ldv: int = 1088
    pad_id: int = 1024
    ties: bool = False
    n_steps: int = 1            # consecutive steps the workload describes (workload 3: 2048)

    @property
    def max_blocks(self) -> int:
        return (self.cap + BLOCK - 1) // BLOCK

    def self_kv_bytes(self) -> int:
        """Valid K+V bytes one self-attention layer reads: 2 tensors x H x L_b x D x 2 B."""
        return int(2 * self.H * self.D * 2 * int(self.seq_len.astype(np.int64).sum()))

    def cross_kv_bytes(self) -> int:
        return int(2 * self.H * self.D * 2 * int(self.enc_len.astype(np.int64).sum()))


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(list(key))


def make_workload(index: int) -> Workload:
    """The host-side description of workload `index` (1..5)."""
    if index == 1:
        return Workload(1, "1 layer, batch 1, self 64 of 2048 (contiguous), cross 64", 1, 1, "contiguous",
                        np.array([64], np.int32), 2048, np.array([64], np.int32), 64, 1.0, 50, 3.0,
                        np.array([0], np.uint64), np.array([5], np.int32))
    if index == 2:
        return Workload(2, "24 layers, batch 1, self 1024 of 4096 (contiguous), cross 1024 (long input)", 24, 1,
                        "contiguous", np.array([1024], np.int32), 4096, np.array([1024], np.int32), 1024, 1.0, 50,
                        3.0, np.array([0], np.uint64), np.array([100], np.int32))
    if index == 3:
        return Workload(3, "24 layers, batch 1, 2048 consecutive steps in a 4096 cache, cross 64 (long output)", 24,
                        1, "contiguous", np.array([2048], np.int32), 4096, np.array([64], np.int32), 64, 1.0, 50,
                        3.0, np.array([0], np.uint64), np.array([2047], np.int32), n_steps=2048)
    if index == 4:
        r = _rng(4, 0)
        B = 32
        return Workload(4, "24 layers, batch 32 ragged, paged bs16 self U{64..2048}, cross U{32..512}", 24, B, "paged",
                        r.integers(64, 2048, size=B, endpoint=True).astype(np.int32), 2048,
                        r.integers(32, 512, size=B, endpoint=True).astype(np.int32), 512, 0.9, 50, 3.0,
                        np.zeros(B, np.uint64), r.integers(0, 20, size=B, endpoint=True).astype(np.int32))
    if index == 5:
        r = _rng(5, 0)
        B = 128
        return Workload(5, "24 layers, batch 128 ragged, paged bs16 self U{512..4096}, cross 256, ties", 24, B,
                        "paged", r.integers(512, 4096, size=B, endpoint=True).astype(np.int32), 4096,
                        np.full(B, 256, np.int32), 256, 0.7, 250, 5.0,
                        (np.uint64(0x5EED0000) + np.arange(B, dtype=np.uint64)),
                        r.integers(0, 20, size=B, endpoint=True).astype(np.int32), ties=True)
    raise ValueError(f"unknown workload {index}")


# --------------------------------------------------------------------------
# tensor generation
# --------------------------------------------------------------------------
def _gen(device, *key: int) -> torch.Generator:
    g = torch.Generator(device=device)
    s = 0
    for k in key:
        s = (s * 1_000_003 + int(k)) % (2 ** 61 - 1)
    g.manual_seed(s)
    return g


def randn_bf16(shape, device, *key: int) -> torch.Tensor:
    """N(0,1) float32 draws rounded to bf16, seeded by `key`."""
    return torch.randn(shape, generator=_gen(device, *key), device=device, dtype=torch.float32).to(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its uint16 bit patterns as a host numpy array (for the oracle)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@dataclasses.dataclass
class SelfCache:
    layout: str
    k: torch.Tensor             # contiguous [B,H,cap,D] or paged [NB,H,16,D]; bf16, or uint8 e4m3 codes
    v: torch.Tensor
    cap: int
    block_table: torch.Tensor | None = None   # [B, max_blocks] int32
    num_blocks: int = 0
    k_scale: float = 1.0        # e4m3 caches: key = code * k_scale
    v_scale: float = 1.0


E4M3_NAN_CODE = 0x7F
FP8_SCALE = 1.0 / 64.0


def to_e4m3_codes(t: torch.Tensor, scale: float, invalid: torch.Tensor | None = None) -> torch.Tensor:
    """Seeded e4m3 codes for a synthetic fp8 cache: torch's own float8 conversion of t / scale
    (clamped to the format's +-448), as uint8; `invalid` slots get the NaN code 0x7F."""
    codes = (t.float() / scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    if invalid is not None:
        codes = codes.masked_fill(invalid, E4M3_NAN_CODE)
    return codes


def make_self_cache_fp8(w: Workload, layer: int, device="cpu", filled_len: np.ndarray | None = None,
                        k_scale: float = FP8_SCALE, v_scale: float = FP8_SCALE) -> SelfCache:
    """The bf16 cache of make_self_cache, held as e4m3 codes (NaN code past the valid keys)."""
    c = make_self_cache(w, layer, device, filled_len)
    k = to_e4m3_codes(torch.nan_to_num(c.k.float(), nan=0.0), k_scale, torch.isnan(c.k))
    v = to_e4m3_codes(torch.nan_to_num(c.v.float(), nan=0.0), v_scale, torch.isnan(c.v))
    return SelfCache(c.layout, k, v, c.cap, c.block_table, c.num_blocks, k_scale, v_scale)


def make_block_table(w: Workload, device="cpu", key: int = 0):
    """Seeded shuffled block table for w.seq_len (block size 16) and the pool size."""
    nblk = (w.seq_len.astype(np.int64) + BLOCK - 1) // BLOCK
    NB = int(nblk.sum()) + 64
    r = _rng(w.index, 77, key)
    perm = r.permutation(NB).astype(np.int32)
    table = np.full((w.B, w.max_blocks), -1, np.int32)
    off = 0
    for b in range(w.B):
        table[b, : nblk[b]] = perm[off: off + nblk[b]]
        off += int(nblk[b])
    return torch.from_numpy(table).to(device), NB


def make_self_cache(w: Workload, layer: int, device="cpu", filled_len: np.ndarray | None = None) -> SelfCache:
    """Self-attention cache of one layer: keys 0..filled_len[b]-1 ~ N(0,1), the rest NaN.

    By default filled_len = seq_len - 1: the step's append fills slot seq_len-1.
    """
    fl = (w.seq_len - 1) if filled_len is None else np.asarray(filled_len, np.int32)
    H, D = w.H, w.D
    if w.layout == "contiguous":
        k = randn_bf16((w.B, H, w.cap, D), device, w.index, layer, 1)
        v = randn_bf16((w.B, H, w.cap, D), device, w.index, layer, 2)
        pos = torch.arange(w.cap, device=device).view(1, 1, w.cap, 1)
        invalid = pos >= torch.from_numpy(fl.astype(np.int64)).to(device).view(w.B, 1, 1, 1)
        k.masked_fill_(invalid, float("nan"))
        v.masked_fill_(invalid, float("nan"))
        return SelfCache("contiguous", k, v, w.cap)
    table, NB = make_block_table(w, device, layer)
    k = randn_bf16((NB, H, BLOCK, D), device, w.index, layer, 1)
    v = randn_bf16((NB, H, BLOCK, D), device, w.index, layer, 2)
    # slot validity: table entry j of row b holds keys 16j .. 16j+15 of that row
    tab = table.cpu().numpy()
    valid_np = np.zeros((NB, BLOCK), dtype=bool)
    for b in range(w.B):
        for j in range(ceil_div(int(fl[b]), BLOCK)):
            valid_np[tab[b, j], : min(BLOCK, int(fl[b]) - BLOCK * j)] = True
    valid = torch.from_numpy(valid_np).to(device)
    inv = ~valid.view(NB, 1, BLOCK, 1)
    k.masked_fill_(inv, float("nan"))
    v.masked_fill_(inv, float("nan"))
    return SelfCache("paged", k, v, w.cap, table.to(torch.int32), NB)


def make_step_inputs(w: Workload, layer: int, device="cpu", step_key: int = 0):
    """Per-layer per-step activations: q (self), q (cross), k_new, v_new, each [B,H,D] bf16."""
    shp = (w.B, w.H, w.D)
    return (randn_bf16(shp, device, w.index, layer, 10, step_key), randn_bf16(shp, device, w.index, layer, 11, step_key),
            randn_bf16(shp, device, w.index, layer, 12, step_key), randn_bf16(shp, device, w.index, layer, 13, step_key))


def make_cross_kv(w: Workload, layer: int, device="cpu"):
    """Description-encoder keys/values [B,H,Lc_max,D] bf16, NaN past enc_len."""
    shp = (w.B, w.H, w.Lc_max, w.D)
    k = randn_bf16(shp, device, w.index, layer, 20)
    v = randn_bf16(shp, device, w.index, layer, 21)
    pos = torch.arange(w.Lc_max, device=device).view(1, 1, -1, 1)
    invalid = pos >= torch.from_numpy(w.enc_len.astype(np.int64)).to(device).view(-1, 1, 1, 1)
    k.masked_fill_(invalid, float("nan"))
    v.masked_fill_(invalid, float("nan"))
    return k, v


def make_logits(w: Workload, device="cpu", step_key: int = 0) -> torch.Tensor:
    """[B, C, ldv] float32 logits ~ N(0, logit_std^2); columns V..ldv-1 hold NaN.

    With w.ties: in each (b, c) row eleven entries are overwritten with the value
    of another entry of the same row, two of them with the row's top_k-th
    largest value, so the top-k boundary itself is tied.
    """
    g = _gen("cpu", w.index, 30, step_key)
    x = torch.randn((w.B, w.C, w.ldv), generator=g, dtype=torch.float32) * w.logit_std
    if w.ldv > w.V:
        x[:, :, w.V:] = float("nan")
    if w.ties:
        r = _rng(w.index, 31, step_key)
        xr = x[:, :, : w.V].reshape(-1, w.V)
        for row in range(xr.shape[0]):
            vals = xr[row]
            order = torch.argsort(vals, descending=True, stable=True)
            kth = int(order[w.top_k - 1])
            cand = r.choice(np.setdiff1d(np.arange(w.V), [kth]), size=11, replace=False)
            vals[cand[:2]] = float(vals[kth])
            src = r.integers(0, w.V, size=9)
            vals[cand[2:]] = vals[src].clone()
    return x.to(device)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["Workload", "make_workload", "make_self_cache", "make_self_cache_fp8", "to_e4m3_codes", "make_step_inputs", "make_cross_kv", "make_logits",
           "make_block_table", "bits", "randn_bf16", "SelfCache", "BLOCK", "BF16_NAN_BITS", "ceil_div"]
