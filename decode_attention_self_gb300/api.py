"""Thin ctypes binding of libdecoderattn.so (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks that the torch tensors it is given are CUDA,
contiguous and of the right dtype, and passes their device pointers, sizes and
the current CUDA stream through the C ABI declared in include/dr_api.h.
PyTorch only provides device memory and streams.

Importing this module loads the library and fails loudly if it is missing:
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdecoderattn.so")

DR_OK, DR_ERR_INVALID_ARG, DR_ERR_UNSUPPORTED, DR_ERR_CUDA = 0, 1, 2, 3
DR_KV_CONTIGUOUS, DR_KV_PAGED = 0, 1
DR_BF16, DR_F32 = 0, 1
DR_KV_BF16, DR_KV_FP8_E4M3 = 0, 1
DR_ERRF_SEQ_LEN, DR_ERRF_BLOCK_ID, DR_ERRF_POS, DR_ERRF_TOKEN, DR_ERRF_TIMEOUT = 1, 2, 4, 8, 16
DR_SAMPLE_ADVANCE = 1

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
_lib = ctypes.CDLL(LIB_PATH)


class dr_kv_cache(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int32), ("max_len", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


_vp, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_lib.dr_kv_append.argtypes = [ctypes.POINTER(dr_kv_cache), _vp, _vp, _vp, _i, _i, _i, _vp, _vp]
_lib.dr_decode_self_attn.argtypes = [_vp, ctypes.POINTER(dr_kv_cache), _vp, _i, _i, _i, _i, _f, _vp, _i, _vp, _vp]
_lib.dr_decode_cross_attn.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _vp, _i, _vp, _vp]
_lib.dr_decode_layer.argtypes = [_vp, ctypes.POINTER(dr_kv_cache), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                                 _i, _f, _vp, _vp, _i, _vp, _vp]
_lib.dr_sample_topk_delayed.argtypes = [_vp, _i, _i, _i, _i, _f, _i, _vp, _vp, ctypes.c_int32, _vp, _vp, _i, _vp]
_lib.dr_embed_tokens.argtypes = [_vp, _vp, _i, _i, _i, _i, _vp, _i, _vp, _vp]
_lib.dr_lm_head.argtypes = [_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp]
_lib.dr_lm_head_stall_test.argtypes = [_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _i, _vp]
_lib.dr_decode_self_attn_stall_test.argtypes = [_vp, ctypes.POINTER(dr_kv_cache), _vp, _i, _i, _i, _i, _f, _vp, _i, _vp,
                                                _i, _vp]
_lib.dr_plan_splits.argtypes = [_i, _i, _i, _i, _i]
_lib.dr_plan_splits.restype = _i
_lib.dr_status_string.argtypes = [_i]
_lib.dr_status_string.restype = ctypes.c_char_p
for _fn in ("dr_kv_append", "dr_decode_self_attn", "dr_decode_cross_attn", "dr_decode_layer",
            "dr_sample_topk_delayed", "dr_embed_tokens", "dr_lm_head", "dr_lm_head_stall_test",
            "dr_decode_self_attn_stall_test"):
    getattr(_lib, _fn).restype = _i


class DrError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {dr_status_string(status)} (status {status})")
        self.status = status


def dr_status_string(status: int) -> str:
    return _lib.dr_status_string(int(status)).decode()


def dr_plan_splits(B: int, H: int, max_len: int, kv_dtype: int, num_sms: int) -> int:
    return int(_lib.dr_plan_splits(B, H, max_len, kv_dtype, num_sms))


def _check(fn: str, status: int):
    if status != DR_OK:
        raise DrError(fn, status)


def _ptr(t: torch.Tensor | None, dtype: torch.dtype | None = None, name: str = "tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


@dataclasses.dataclass
class KVCache:
    """One layer's self-attention cache (device tensors owned by the caller).

    contiguous: k, v [B, H, max_len, D] bf16, or uint8 e4m3 codes with k_scale/v_scale.
    paged:      k, v [num_blocks, H, 16, D] (same element formats) and block_table [B, max_blocks] int32.
    """

    k: torch.Tensor
    v: torch.Tensor
    block_table: torch.Tensor | None = None
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def fp8(self) -> bool:
        return self.k.dtype == torch.uint8

    @property
    def paged(self) -> bool:
        return self.block_table is not None

    @property
    def capacity(self) -> int:
        return self.block_table.shape[1] * self.k.shape[2] if self.paged else self.k.shape[2]

    def as_c(self) -> dr_kv_cache:
        c = dr_kv_cache()
        dt = torch.uint8 if self.fp8 else torch.bfloat16
        c.k = _ptr(self.k, dt, "cache.k")
        c.v = _ptr(self.v, dt, "cache.v")
        c.kv_dtype = DR_KV_FP8_E4M3 if self.fp8 else DR_KV_BF16
        c.k_scale = float(self.k_scale)
        c.v_scale = float(self.v_scale)
        if self.paged:
            c.layout = DR_KV_PAGED
            c.block_size = self.k.shape[2]
            c.num_blocks = self.k.shape[0]
            c.max_blocks_per_seq = self.block_table.shape[1]
            c.block_table = _ptr(self.block_table, torch.int32, "cache.block_table")
        else:
            c.layout = DR_KV_CONTIGUOUS
            c.max_len = self.k.shape[2]
        return c


def dr_kv_append(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, pos: torch.Tensor,
                 err_flag: torch.Tensor | None = None, stream=None) -> None:
    """Write k_new, v_new [B, H, D] bf16 at position pos[b] (int32 [B]) of every row."""
    B, H, D = k_new.shape
    c = cache.as_c()
    _check("dr_kv_append", _lib.dr_kv_append(ctypes.byref(c), _ptr(k_new, torch.bfloat16, "k_new"),
                                             _ptr(v_new, torch.bfloat16, "v_new"), _ptr(pos, torch.int32, "pos"),
                                             B, H, D, _ptr(err_flag, torch.int32, "err_flag"), _stream(stream)))


def dr_decode_self_attn(q: torch.Tensor, cache: KVCache, seq_len: torch.Tensor, out: torch.Tensor,
                        max_seq_len_hint: int = 0, scale: float = 0.0, err_flag: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """out[b,h] = softmax(scale q[b,h].K[b,h,:seq_len[b]]) V[b,h,:seq_len[b]] (out bf16 or float32)."""
    B, H, D = q.shape
    c = cache.as_c()
    od = DR_F32 if out.dtype == torch.float32 else DR_BF16
    _check("dr_decode_self_attn",
           _lib.dr_decode_self_attn(_ptr(q, torch.bfloat16, "q"), ctypes.byref(c), _ptr(seq_len, torch.int32, "seq_len"),
                                    B, H, D, int(max_seq_len_hint), float(scale), _ptr(out, None, "out"), od,
                                    _ptr(err_flag, torch.int32, "err_flag"), _stream(stream)))
    return out


def dr_decode_self_attn_stall_test(q: torch.Tensor, cache: KVCache, seq_len: torch.Tensor, out: torch.Tensor,
                                   stall_row: int, max_seq_len_hint: int = 0, scale: float = 0.0,
                                   err_flag: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Test hook: dr_decode_self_attn with row stall_row's cluster merge left waiting until its bound runs out."""
    B, H, D = q.shape
    c = cache.as_c()
    od = DR_F32 if out.dtype == torch.float32 else DR_BF16
    _check("dr_decode_self_attn_stall_test",
           _lib.dr_decode_self_attn_stall_test(_ptr(q, torch.bfloat16, "q"), ctypes.byref(c),
                                               _ptr(seq_len, torch.int32, "seq_len"), B, H, D, int(max_seq_len_hint),
                                               float(scale), _ptr(out, None, "out"), od,
                                               _ptr(err_flag, torch.int32, "err_flag"), int(stall_row),
                                               _stream(stream)))
    return out


def dr_decode_cross_attn(q: torch.Tensor, k_enc: torch.Tensor, v_enc: torch.Tensor, enc_len: torch.Tensor,
                         out: torch.Tensor, scale: float = 0.0, err_flag: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """Attention of q [B,H,D] over k_enc, v_enc [B,H,Lc_max,D] limited to enc_len[b] keys."""
    B, H, D = q.shape
    Lc_max = k_enc.shape[2]
    od = DR_F32 if out.dtype == torch.float32 else DR_BF16
    _check("dr_decode_cross_attn",
           _lib.dr_decode_cross_attn(_ptr(q, torch.bfloat16, "q"), _ptr(k_enc, torch.bfloat16, "k_enc"),
                                     _ptr(v_enc, torch.bfloat16, "v_enc"), _ptr(enc_len, torch.int32, "enc_len"),
                                     B, H, D, Lc_max, float(scale), _ptr(out, None, "out"), od,
                                     _ptr(err_flag, torch.int32, "err_flag"), _stream(stream)))
    return out


def dr_decode_layer(q: torch.Tensor, cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, seq_len: torch.Tensor,
                    q_cross: torch.Tensor, k_enc: torch.Tensor, v_enc: torch.Tensor, enc_len: torch.Tensor,
                    out: torch.Tensor, out_cross: torch.Tensor, max_seq_len_hint: int = 0, scale: float = 0.0,
                    err_flag: torch.Tensor | None = None, stream=None) -> None:
    """One launch: append k_new, v_new at seq_len-1, self-attention over seq_len keys, cross-attention."""
    B, H, D = q.shape
    if out_cross.dtype != out.dtype:
        raise ValueError("out and out_cross must have the same dtype")
    c = cache.as_c()
    od = DR_F32 if out.dtype == torch.float32 else DR_BF16
    _check("dr_decode_layer",
           _lib.dr_decode_layer(_ptr(q, torch.bfloat16, "q"), ctypes.byref(c), _ptr(k_new, torch.bfloat16, "k_new"),
                                _ptr(v_new, torch.bfloat16, "v_new"), _ptr(seq_len, torch.int32, "seq_len"),
                                _ptr(q_cross, torch.bfloat16, "q_cross"), _ptr(k_enc, torch.bfloat16, "k_enc"),
                                _ptr(v_enc, torch.bfloat16, "v_enc"), _ptr(enc_len, torch.int32, "enc_len"),
                                k_enc.shape[2], B, H, D, int(max_seq_len_hint), float(scale), _ptr(out, None, "out"),
                                _ptr(out_cross, None, "out_cross"), od, _ptr(err_flag, torch.int32, "err_flag"),
                                _stream(stream)))


def dr_sample_topk_delayed(logits: torch.Tensor, temperature: float, top_k: int, seeds: torch.Tensor,
                           step: torch.Tensor, pad_id: int, tokens: torch.Tensor, probs: torch.Tensor | None = None,
                           V: int | None = None, advance: bool = False, stream=None) -> torch.Tensor:
    """tokens [B,C] int32 from logits [B,C,ldv] float32; seeds [B] int64 (uint64 bits); step [B] int32."""
    B, C, ldv = logits.shape
    V = ldv if V is None else V
    if seeds.dtype not in (torch.int64, torch.uint64):
        raise ValueError("seeds must be a 64-bit integer tensor")
    _check("dr_sample_topk_delayed",
           _lib.dr_sample_topk_delayed(_ptr(logits, torch.float32, "logits"), B, C, V, ldv, float(temperature),
                                       int(top_k), _ptr(seeds, None, "seeds"), _ptr(step, torch.int32, "step"),
                                       int(pad_id), _ptr(tokens, torch.int32, "tokens"),
                                       _ptr(probs, torch.float32, "probs"), DR_SAMPLE_ADVANCE if advance else 0,
                                       _stream(stream)))
    return tokens


def dr_embed_tokens(tokens: torch.Tensor, table: torch.Tensor, V: int, out: torch.Tensor,
                    err_flag: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[b] = sum_c table[c*V + tokens[b,c]]; tokens [B,C] int32, table [C*V, Dm] bf16, out [B,Dm]."""
    B, C = tokens.shape
    Dm = table.shape[1]
    od = DR_F32 if out.dtype == torch.float32 else DR_BF16
    _check("dr_embed_tokens",
           _lib.dr_embed_tokens(_ptr(tokens, torch.int32, "tokens"), _ptr(table, torch.bfloat16, "table"), B, C, V, Dm,
                                _ptr(out, None, "out"), od, _ptr(err_flag, torch.int32, "err_flag"), _stream(stream)))
    return out


def dr_lm_head(hidden: torch.Tensor, W: torch.Tensor, C: int, logits: torch.Tensor,
               err_flag: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """logits [B,C,ldv] float32 from hidden [B,K] bf16 and merged heads W [C*V, K] bf16 (V = W rows / C)."""
    B, K = hidden.shape
    V = W.shape[0] // C
    ldv = logits.shape[2]
    _check("dr_lm_head",
           _lib.dr_lm_head(_ptr(hidden, torch.bfloat16, "hidden"), _ptr(W, torch.bfloat16, "W"), B, K, C, V, ldv,
                           _ptr(logits, torch.float32, "logits"), _ptr(err_flag, torch.int32, "err_flag"),
                           _stream(stream)))
    return logits


def dr_lm_head_stall_test(hidden: torch.Tensor, W: torch.Tensor, C: int, logits: torch.Tensor, stall_slab: int,
                          err_flag: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Test hook: dr_lm_head with the CTAs of weight slab `stall_slab` made to time out (see dr_api.h)."""
    B, K = hidden.shape
    V = W.shape[0] // C
    ldv = logits.shape[2]
    _check("dr_lm_head_stall_test",
           _lib.dr_lm_head_stall_test(_ptr(hidden, torch.bfloat16, "hidden"), _ptr(W, torch.bfloat16, "W"), B, K, C, V,
                                      ldv, _ptr(logits, torch.float32, "logits"),
                                      _ptr(err_flag, torch.int32, "err_flag"), int(stall_slab), _stream(stream)))
    return logits


def loaded_library_path() -> str:
    return LIB_PATH
