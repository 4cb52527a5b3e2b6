"""ctypes wrapper around the plain C oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
baseline leg may import this package; the product library never does.

Arrays cross as numpy arrays: bf16 tensors as ``uint16`` bit patterns, lengths
and tables as ``int32``, logits as ``float32``, results as ``float64``.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np

from .build import build as _build

_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(_build())
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_attend.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_double, _f64p, _f64p]
        L.oracle_attend.restype = None
        L.oracle_attn_contiguous.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, _i32p, ctypes.c_double, _f64p]
        L.oracle_attn_contiguous.restype = None
        L.oracle_attn_contiguous_row.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                                 _f64p]
        L.oracle_attn_contiguous_row.restype = None
        L.oracle_attn_paged_row.argtypes = [_u16p, _u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, _f64p]
        L.oracle_attn_paged_row.restype = ctypes.c_int
        L.oracle_attn_paged.argtypes = [_u16p, _u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_double, _f64p]
        L.oracle_attn_paged.restype = ctypes.c_int
        L.oracle_kv_append_contiguous.argtypes = [_u16p, _u16p, _u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_int]
        L.oracle_kv_append_contiguous.restype = None
        L.oracle_kv_append_paged.argtypes = [_u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int, _u16p, _u16p, _i32p,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.oracle_kv_append_paged.restype = None
        L.oracle_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        L.oracle_philox4x32_10.restype = None
        L.oracle_uniform.argtypes = [ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
        L.oracle_uniform.restype = ctypes.c_double
        L.oracle_sample_row.argtypes = [_f32p, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_uint64,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _i32p, _f64p,
                                        _f64p, _i32p]
        L.oracle_sample_row.restype = ctypes.c_int
        L.oracle_sample.argtypes = [_f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                    ctypes.c_int, _u64p, _i32p, ctypes.c_int32, _i32p, _f64p, _f64p, _i32p]
        L.oracle_sample.restype = ctypes.c_int
        L.oracle_embed_tokens.argtypes = [_i32p, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64p]
        L.oracle_embed_tokens.restype = ctypes.c_int
        L.oracle_lm_head.argtypes = [_u16p, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64p]
        L.oracle_lm_head.restype = None
        _u8p = ctypes.POINTER(ctypes.c_uint8)
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_double.restype = ctypes.c_double
        L.oracle_double_to_e4m3.argtypes = [ctypes.c_double]
        L.oracle_double_to_e4m3.restype = ctypes.c_uint8
        L.oracle_kv_append_fp8_contiguous.argtypes = [_u8p, _u8p, _u16p, _u16p, _i32p, ctypes.c_int, ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_float]
        L.oracle_kv_append_fp8_contiguous.restype = None
        L.oracle_kv_append_fp8_paged.argtypes = [_u8p, _u8p, _i32p, ctypes.c_int, ctypes.c_int, _u16p, _u16p, _i32p,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                                 ctypes.c_float]
        L.oracle_kv_append_fp8_paged.restype = None
        L.oracle_attn_fp8_contiguous.argtypes = [_u16p, _u8p, _u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, _i32p, ctypes.c_double, ctypes.c_double,
                                                 ctypes.c_double, _f64p]
        L.oracle_attn_fp8_contiguous.restype = None
        L.oracle_attn_fp8_paged.argtypes = [_u16p, _u8p, _u8p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_double,
                                            ctypes.c_double, ctypes.c_double, _f64p]
        L.oracle_attn_fp8_paged.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray, ty):
    assert a.flags.c_contiguous, "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ty)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(bits)


def attend(q, keys, values, scale):
    """Attention of one query q[D] over keys/values [n, D] (bf16 bits). Returns (out[D], sum of p)."""
    q, keys, values = _u16(q), _u16(keys), _u16(values)
    D = q.shape[-1]
    n = keys.shape[0] if keys.ndim == 2 else 0
    out = np.zeros(D, np.float64)
    ps = np.zeros(1, np.float64)
    lib().oracle_attend(_p(q, _u16p), _p(keys, _u16p), _p(values, _u16p), n, D, scale, _p(out, _f64p), _p(ps, _f64p))
    return out, float(ps[0])


def attn_contiguous(q, k, v, seq_len, scale):
    """q [B,H,D]; k, v [B,H,max_len,D] (bf16 bits); seq_len [B]. Returns [B,H,D] float64."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, H, max_len, D = k.shape
    sl = _i32(seq_len)
    out = np.zeros((B, H, D), np.float64)
    lib().oracle_attn_contiguous(_p(q, _u16p), _p(k, _u16p), _p(v, _u16p), B, H, D, max_len, _p(sl, _i32p), scale,
                                 _p(out, _f64p))
    return out


def attn_contiguous_row(q_row, k_row, v_row, n, scale):
    """One (b,h) row: q_row [D]; k_row, v_row [>=n, D]. Returns [D] float64."""
    q_row, k_row, v_row = _u16(q_row), _u16(k_row), _u16(v_row)
    D = q_row.shape[-1]
    out = np.zeros(D, np.float64)
    lib().oracle_attn_contiguous_row(_p(q_row, _u16p), _p(k_row, _u16p), _p(v_row, _u16p), D, int(n), scale,
                                     _p(out, _f64p))
    return out


def attn_paged(q, k_pool, v_pool, block_table, seq_len, scale, block_size=16):
    """q [B,H,D]; pools [NB,H,bs,D]; block_table [B,max_blocks]; seq_len [B]. Returns [B,H,D] float64."""
    q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
    bt = _i32(block_table)
    sl = _i32(seq_len)
    B, H, D = q.shape
    NB = k_pool.shape[0]
    out = np.zeros((B, H, D), np.float64)
    rc = lib().oracle_attn_paged(_p(q, _u16p), _p(k_pool, _u16p), _p(v_pool, _u16p), _p(bt, _i32p), bt.shape[1], NB,
                                 block_size, B, H, D, _p(sl, _i32p), scale, _p(out, _f64p))
    if rc:
        raise ValueError("block table entry outside the pool")
    return out


def attn_paged_row(q_row, k_pool, v_pool, table_row, h, n, scale, block_size=16):
    q_row, k_pool, v_pool = _u16(q_row), _u16(k_pool), _u16(v_pool)
    tr = _i32(table_row)
    NB, H, _, D = k_pool.shape
    out = np.zeros(D, np.float64)
    rc = lib().oracle_attn_paged_row(_p(q_row, _u16p), _p(k_pool, _u16p), _p(v_pool, _u16p), _p(tr, _i32p), NB,
                                     block_size, H, int(h), D, int(n), scale, _p(out, _f64p))
    if rc:
        raise ValueError("block table entry outside the pool")
    return out


def kv_append_contiguous(k, v, k_new, v_new, pos):
    """In-place append into host caches k, v [B,H,max_len,D] (uint16, C-contiguous)."""
    k_new, v_new = _u16(k_new), _u16(v_new)
    B, H, max_len, D = k.shape
    ps = _i32(pos)
    lib().oracle_kv_append_contiguous(_p(k, _u16p), _p(v, _u16p), _p(k_new, _u16p), _p(v_new, _u16p), _p(ps, _i32p),
                                      B, H, D, max_len)


def kv_append_paged(k_pool, v_pool, block_table, k_new, v_new, pos, block_size=16):
    k_new, v_new = _u16(k_new), _u16(v_new)
    bt = _i32(block_table)
    ps = _i32(pos)
    B, H, D = k_new.shape
    lib().oracle_kv_append_paged(_p(k_pool, _u16p), _p(v_pool, _u16p), _p(bt, _i32p), bt.shape[1], block_size,
                                 _p(k_new, _u16p), _p(v_new, _u16p), _p(ps, _i32p), B, H, D)


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_p(c, _u32p), _p(k, _u32p), _p(out, _u32p))
    return out


def uniform(seed, b, c, step, i):
    return lib().oracle_uniform(int(seed), int(b), int(c), int(step), int(i))


def sample_row(logits_row, temperature, top_k, seed, b, c, step, pad_id, want_probs=False, want_topk=False):
    """One (b,c) row. Returns dict(token, margin, probs|None, topk|None)."""
    x = np.ascontiguousarray(logits_row, dtype=np.float32)
    V = x.shape[0]
    tok = np.zeros(1, np.int32)
    mar = np.zeros(1, np.float64)
    probs = np.zeros(V, np.float64) if want_probs else None
    topk = np.zeros(top_k, np.int32) if want_topk else None
    rc = lib().oracle_sample_row(_p(x, _f32p), V, temperature, top_k, int(seed), b, c, step, pad_id,
                                 _p(tok, _i32p), _p(mar, _f64p), _p(probs, _f64p) if probs is not None else None,
                                 _p(topk, _i32p) if topk is not None else None)
    if rc:
        raise ValueError("invalid sampler input")
    return dict(token=int(tok[0]), margin=float(mar[0]), probs=probs, topk=topk)


def sample(logits, temperature, top_k, seeds, steps, pad_id, V=None, want_probs=False, want_topk=False):
    """logits [B,C,ldv] float32; seeds [B] uint64; steps [B]. Returns dict of arrays."""
    x = np.ascontiguousarray(logits, dtype=np.float32)
    B, C, ldv = x.shape
    V = ldv if V is None else V
    sd = np.ascontiguousarray(seeds, dtype=np.uint64)
    st = _i32(steps)
    tokens = np.zeros((B, C), np.int32)
    margins = np.zeros((B, C), np.float64)
    probs = np.zeros((B, C, V), np.float64) if want_probs else None
    topk = np.zeros((B, C, top_k), np.int32) if want_topk else None
    rc = lib().oracle_sample(_p(x, _f32p), B, C, V, ldv, temperature, top_k, _p(sd, _u64p), _p(st, _i32p), pad_id,
                             _p(tokens, _i32p), _p(margins, _f64p),
                             _p(probs, _f64p) if probs is not None else None,
                             _p(topk, _i32p) if topk is not None else None)
    if rc:
        raise ValueError("invalid sampler input")
    return dict(tokens=tokens, margins=margins, probs=probs, topk=topk)


def embed_tokens(tokens, table, V):
    """tokens [B,C] int; table [C*V, Dm] bf16 bits. Returns [B, Dm] float64 (sum of the C embeddings)."""
    tk = _i32(tokens)
    tb = _u16(table)
    B, C = tk.shape
    Dm = tb.shape[1]
    out = np.zeros((B, Dm), np.float64)
    if lib().oracle_embed_tokens(_p(tk, _i32p), _p(tb, _u16p), B, C, V, Dm, _p(out, _f64p)):
        raise ValueError("token outside the vocabulary")
    return out


def lm_head(hidden, W):
    """hidden [B,K], W [N,K] (bf16 bits). Returns [B,N] float64 logits."""
    h, w = _u16(hidden), _u16(W)
    B, K = h.shape
    N = w.shape[0]
    out = np.zeros((B, N), np.float64)
    lib().oracle_lm_head(_p(h, _u16p), _p(w, _u16p), B, K, N, _p(out, _f64p))
    return out


_u8p = ctypes.POINTER(ctypes.c_uint8)


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint8, a.dtype
    return a


def e4m3_to_double(code: int) -> float:
    return lib().oracle_e4m3_to_double(int(code))


def double_to_e4m3(x: float) -> int:
    return int(lib().oracle_double_to_e4m3(float(x)))


def kv_append_fp8_contiguous(k, v, k_new, v_new, pos, k_scale, v_scale):
    """In-place quantising append into host fp8 caches k, v [B,H,max_len,D] (uint8 codes)."""
    k_new, v_new = _u16(k_new), _u16(v_new)
    B, H, max_len, D = k.shape
    ps = _i32(pos)
    lib().oracle_kv_append_fp8_contiguous(_p(k, _u8p), _p(v, _u8p), _p(k_new, _u16p), _p(v_new, _u16p),
                                          _p(ps, _i32p), B, H, D, max_len, k_scale, v_scale)


def kv_append_fp8_paged(k_pool, v_pool, block_table, k_new, v_new, pos, k_scale, v_scale, block_size=16):
    k_new, v_new = _u16(k_new), _u16(v_new)
    bt = _i32(block_table)
    ps = _i32(pos)
    B, H, D = k_new.shape
    lib().oracle_kv_append_fp8_paged(_p(k_pool, _u8p), _p(v_pool, _u8p), _p(bt, _i32p), bt.shape[1], block_size,
                                     _p(k_new, _u16p), _p(v_new, _u16p), _p(ps, _i32p), B, H, D, k_scale, v_scale)


def attn_fp8_contiguous(q, k, v, seq_len, scale, k_scale, v_scale):
    q, k, v = _u16(q), _u8(k), _u8(v)
    B, H, max_len, D = k.shape
    sl = _i32(seq_len)
    out = np.zeros((B, H, D), np.float64)
    lib().oracle_attn_fp8_contiguous(_p(q, _u16p), _p(k, _u8p), _p(v, _u8p), B, H, D, max_len, _p(sl, _i32p), scale,
                                     k_scale, v_scale, _p(out, _f64p))
    return out


def attn_fp8_paged(q, k_pool, v_pool, block_table, seq_len, scale, k_scale, v_scale, block_size=16):
    q, k_pool, v_pool = _u16(q), _u8(k_pool), _u8(v_pool)
    bt = _i32(block_table)
    sl = _i32(seq_len)
    B, H, D = q.shape
    out = np.zeros((B, H, D), np.float64)
    rc = lib().oracle_attn_fp8_paged(_p(q, _u16p), _p(k_pool, _u8p), _p(v_pool, _u8p), _p(bt, _i32p), bt.shape[1],
                                     k_pool.shape[0], block_size, B, H, D, _p(sl, _i32p), scale, k_scale, v_scale,
                                     _p(out, _f64p))
    if rc:
        raise ValueError("block table entry outside the pool")
    return out
