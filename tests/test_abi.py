"""The C-ABI library loads without a GPU, exports every symbol include/dr_api.h
declares, and rejects host-checkable mistakes before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dr_api.h")


@pytest.fixture(scope="module")
def lib():
    from decode_attention_self_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:dr_status|int|const char\s*\*)\s*(dr_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_decode_step_entry_points():
    names = declared_functions()
    for n in ("dr_kv_append", "dr_decode_self_attn", "dr_decode_cross_attn", "dr_sample_topk_delayed",
              "dr_status_string", "dr_plan_splits"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in dr_api.h but not exported"


def test_library_is_built_for_sm_103a_only():
    from decode_attention_self_gb300 import build

    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    lib.dr_status_string.restype = ctypes.c_char_p
    assert lib.dr_status_string(0) == b"ok"
    assert lib.dr_status_string(1) == b"invalid argument"
    assert lib.dr_status_string(2) == b"unsupported shape"
    assert lib.dr_status_string(3) == b"CUDA launch failed"


class Cache(ctypes.Structure):
    _fields_ = [("layout", ctypes.c_int32), ("max_len", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


FAKE = 0x10000   # a 16-byte aligned non-null address; never dereferenced on the host


def test_host_validation_rejects_before_any_launch(lib):
    c = Cache(0, 2048, 0, 0, 0, 0, FAKE, FAKE, None)
    cp = ctypes.byref(c)
    vp = ctypes.c_void_p
    # D != 64 is unsupported
    assert lib.dr_kv_append(cp, vp(FAKE), vp(FAKE), vp(FAKE), 1, 16, 32, None, None) == 2
    # null k_new
    assert lib.dr_kv_append(cp, None, vp(FAKE), vp(FAKE), 1, 16, 64, None, None) == 1
    # misaligned q
    assert lib.dr_decode_self_attn(vp(FAKE + 2), cp, vp(FAKE), 1, 16, 64, 0, ctypes.c_float(0), vp(FAKE), 0, None,
                                   None) == 1
    # bad batch / heads
    assert lib.dr_decode_self_attn(vp(FAKE), cp, vp(FAKE), 0, 16, 64, 0, ctypes.c_float(0), vp(FAKE), 0, None,
                                   None) == 1
    # paged with block size 32 is unsupported; paged without a table is invalid
    cpg = Cache(1, 0, 32, 10, 4, 0, FAKE, FAKE, FAKE)
    assert lib.dr_decode_self_attn(vp(FAKE), ctypes.byref(cpg), vp(FAKE), 1, 16, 64, 0, ctypes.c_float(0), vp(FAKE),
                                   0, None, None) == 2
    cpn = Cache(1, 0, 16, 10, 4, 0, FAKE, FAKE, None)
    assert lib.dr_decode_self_attn(vp(FAKE), ctypes.byref(cpn), vp(FAKE), 1, 16, 64, 0, ctypes.c_float(0), vp(FAKE),
                                   0, None, None) == 1
    # unknown layout, unknown KV format, e4m3 cache without positive scales
    assert lib.dr_decode_self_attn(vp(FAKE), ctypes.byref(Cache(7, 16, 0, 0, 0, 0, FAKE, FAKE, None)), vp(FAKE), 1,
                                   16, 64, 0, ctypes.c_float(0), vp(FAKE), 0, None, None) == 1
    assert lib.dr_decode_self_attn(vp(FAKE), ctypes.byref(Cache(0, 16, 0, 0, 0, 5, FAKE, FAKE, None)), vp(FAKE), 1,
                                   16, 64, 0, ctypes.c_float(0), vp(FAKE), 0, None, None) == 1
    assert lib.dr_decode_self_attn(vp(FAKE), ctypes.byref(Cache(0, 16, 0, 0, 0, 1, FAKE, FAKE, None, 0.0, 1.0)),
                                   vp(FAKE), 1, 16, 64, 0, ctypes.c_float(0), vp(FAKE), 0, None, None) == 1
    assert lib.dr_kv_append(ctypes.byref(Cache(0, 16, 0, 0, 0, 1, FAKE, FAKE, None, 1.0, float("inf"))), vp(FAKE),
                            vp(FAKE), vp(FAKE), 1, 16, 64, None, None) == 1
    # cross attention: Lc_max < 1, bad out dtype, NaN scale
    assert lib.dr_decode_cross_attn(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1, 16, 64, 0, ctypes.c_float(0),
                                    vp(FAKE), 0, None, None) == 1
    assert lib.dr_decode_cross_attn(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1, 16, 64, 8, ctypes.c_float(0),
                                    vp(FAKE), 5, None, None) == 1
    assert lib.dr_decode_cross_attn(vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 1, 16, 64, 8,
                                    ctypes.c_float(float("nan")), vp(FAKE), 0, None, None) == 1


def test_sampler_validation(lib):
    vp, f = ctypes.c_void_p, ctypes.c_float
    args = lambda B=1, C=9, V=1088, ldv=1088, T=1.0, k=50, flags=0: (
        vp(FAKE), B, C, V, ldv, f(T), k, vp(FAKE), vp(FAKE), 1024, vp(FAKE), None, flags, None)
    assert lib.dr_sample_topk_delayed(*args(k=0)) == 1
    assert lib.dr_sample_topk_delayed(*args(k=1089)) == 1
    assert lib.dr_sample_topk_delayed(*args(T=0.0)) == 1
    assert lib.dr_sample_topk_delayed(*args(T=-1.0)) == 1
    assert lib.dr_sample_topk_delayed(*args(T=float("inf"))) == 1
    assert lib.dr_sample_topk_delayed(*args(ldv=1000)) == 1
    assert lib.dr_sample_topk_delayed(*args(C=17)) == 2
    assert lib.dr_sample_topk_delayed(*args(V=4096, ldv=4096, k=5)) == 2
    assert lib.dr_sample_topk_delayed(*args(flags=2)) == 1
    assert lib.dr_sample_topk_delayed(*args(B=0)) == 1
    assert lib.dr_sample_topk_delayed(*args(B=65536)) == 2      # the grid holds one batch row per y index
    assert lib.dr_sample_topk_delayed(vp(FAKE), 1, 9, 1088, 1088, f(1.0), 50, None, vp(FAKE), 1024, vp(FAKE), None, 0,
                                      None) == 1


def test_embedding_validation(lib):
    # the merged embedding lookup keeps one token per codebook on chip, for up to 16 codebooks: a 17th is refused
    # before anything is enqueued rather than left out of the sum
    vp = ctypes.c_void_p
    call = lambda B=2, C=9, V=1088, Dm=1024, od=0, tok=FAKE, table=FAKE, out=FAKE: lib.dr_embed_tokens(
        vp(tok) if tok else None, vp(table) if table else None, B, C, V, Dm, vp(out) if out else None, od, None, None)
    assert call(C=17) == 2
    assert call(C=64) == 2
    assert call(C=0) == 1
    assert call(B=0) == 1
    assert call(V=0) == 1
    assert call(Dm=12) == 1                       # not a multiple of 8
    assert call(od=5) == 1
    assert call(tok=0) == 1
    assert call(table=FAKE + 8) == 1              # table must be 16-byte aligned


def test_self_attn_stall_hook_validation(lib):
    # the row must exist; the check comes before anything needs a device
    c = Cache(0, 2048, 0, 0, 0, 0, FAKE, FAKE, None)
    vp = ctypes.c_void_p
    call = lambda row, B=2: lib.dr_decode_self_attn_stall_test(vp(FAKE), ctypes.byref(c), vp(FAKE), B, 16, 64, 0,
                                                               ctypes.c_float(0), vp(FAKE), 0, None, row, None)
    assert call(-1) == 1
    assert call(32) == 1
    assert call(0, B=0) == 1


def test_split_plan(lib):
    # split count per (b, h) row: one cluster of at most 8 CTAs, >= 64 keys each, <= 256 KiB of K+V each at
    # the longest row, and at least 6 CTAs per SM of a 152-SM GPU when the rows alone are fewer.
    plan = lib.dr_plan_splits
    BF16, E4M3 = 0, 1
    assert plan(128, 16, 4096, BF16, 152) == 4    # 4096 keys x 256 B = 1 MiB per row: 4 CTAs
    assert plan(128, 16, 4096, E4M3, 152) == 2    # 128 B per key: 2 CTAs
    assert plan(32, 16, 2048, BF16, 152) == 2     # 512 rows: 2 CTAs each cover 6 x 152 = 912
    assert plan(16, 16, 1024, BF16, 152) == 4     # 256 rows: ceil(912 / 256) = 4
    assert plan(1, 16, 1024, BF16, 152) == 8      # batch 1: fill the GPU, capped by the cluster size
    assert plan(1, 16, 64, BF16, 152) == 1        # a 64-key row is one CTA
    assert plan(1, 16, 200, BF16, 152) == 4       # 13 tiles, at least 4 per CTA: ceil(13 / 4) = 4 CTAs
    # a few long rows: 16 CTAs per row (a non-portable cluster) when 8 would take >= 16 tiles each and
    # 16 per row is at most 2 CTAs per SM
    assert plan(1, 16, 2048, BF16, 152) == 16
    assert plan(1, 16, 4096, E4M3, 152) == 16
    assert plan(1, 19, 2048, BF16, 152) == 16     # 304 CTAs on 152 SMs
    assert plan(1, 20, 2048, BF16, 152) == 8      # 320: more than 2 per SM
    assert plan(1, 16, 2000, BF16, 152) == 8      # 125 tiles: fewer than 16 per CTA at 8 CTAs
    assert plan(2, 16, 4096, BF16, 152) == 8
    assert plan(128, 16, 4096, 7, 152) == 1       # unknown storage type
    assert plan(0, 16, 4096, BF16, 152) == 1


def test_lm_head_stall_hook_validation(lib):
    # the test hook applies to the tensor-core head (batch >= 4) and to a slab that exists: ceil(9 * 1088 / 128) = 77
    vp = ctypes.c_void_p
    call = lambda B=8, slab=0: lib.dr_lm_head_stall_test(vp(FAKE), vp(FAKE), B, 1024, 9, 1088, 1088, vp(FAKE), None,
                                                       slab, None)
    assert call(B=3) == 2
    assert call(slab=-1) == 1
    assert call(slab=77) == 1


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++11")])
def test_header_compiles_alone_as_strict_c_and_cpp(lang, std):
    import shutil
    import subprocess

    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    flags = ["-Wall", "-Wextra", "-Werror"] + (["-pedantic"] if lang == "c" else [])
    subprocess.run([cc, std, *flags, "-fsyntax-only", "-x", lang, HEADER], check=True)


def test_plain_c_program_links_and_calls_the_library(lib, tmp_path):
    # A C99 program that includes only dr_api.h, takes every entry point as a C function pointer and calls the
    # two host-only ones: the ABI is usable from C without any C++ or CUDA header.
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no host compiler")
    from decode_attention_self_gb300 import build

    pkg = os.path.dirname(build.LIB)
    src = tmp_path / "use_dr_api.c"
    entry = ", ".join(f"(fn){n}" for n in declared_functions())
    src.write_text('#include <stdio.h>\n#include "dr_api.h"\ntypedef void (*fn)(void);\n'
                   f"int main(void) {{\n    fn all[] = {{{entry}}};\n"
                   '    printf("%s %d %d\\n", dr_status_string(DR_OK), dr_plan_splits(128, 16, 4096, DR_KV_BF16, 152),\n'
                   "           (int)(sizeof all / sizeof all[0]));\n    return 0;\n}\n")
    exe = tmp_path / "use_dr_api"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.dirname(HEADER),
                    str(src), "-L", pkg, "-ldecoderattn", f"-Wl,-rpath,{pkg}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert out == ["ok", "4", str(len(declared_functions()))]
