"""The C-ABI library on the host (no GPU): it loads, exports every symbol the
headers declare, and rejects bad arguments before making any CUDA call.

Every call here returns from host-side validation (or from num_tokens == 0)
before the library touches the CUDA runtime, so fake pointers are safe."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import norm_activation_fp8_gb300 as vg
from norm_activation_fp8_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, NULL, SHAPE, ALIGN, MODE, GROUP = 0, 1, 2, 3, 4, 5
A = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return vg.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(vg_\w+)\s*\(", text))
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert {"vg_fused_add_rms_norm_fp8", "vg_silu_mul_fp8"} <= names
    assert {"vg_fused_mla_dual_rms_norm", "vg_fused_mla_dual_rms_norm_per_token_quant",
            "vg_fused_add_rms_norm_pad", "vg_fused_qk_norm_rope"} <= names
    assert names == set(vg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(vg_\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None
    assert lib.vg_abi_version() == 3


def test_status_strings(lib):
    for s in range(8):
        assert lib.vg_status_string(s)
    assert lib.vg_status_string(0) == b"ok"


def norm(lib, q=A, r_out=A, scale=A, x=A, res=A, w=A, T=4, H=1024, eps=1e-5, mode=0, G=128):
    return lib.vg_fused_add_rms_norm_fp8(q, r_out, scale, x, res, w, T, H, ctypes.c_float(eps),
                                         mode, G, None)


def silu(lib, q=A, scale=A, gu=A, T=4, I=1024, mode=0, G=128):
    return lib.vg_silu_mul_fp8(q, scale, gu, T, I, mode, G, None)


@pytest.mark.parametrize("fn", [norm, silu])
def test_bad_mode(lib, fn):
    assert fn(lib, mode=3) == MODE
    assert fn(lib, mode=-1) == MODE


@pytest.mark.parametrize("fn,key", [(norm, "H"), (silu, "I")])
def test_bad_shape(lib, fn, key):
    for n in (0, 4, 12, 1030, 32776, 65536):
        assert fn(lib, **{key: n}) == SHAPE, n
    assert fn(lib, T=-1) == SHAPE
    assert fn(lib, T=2 ** 31) == SHAPE


@pytest.mark.parametrize("fn,key", [(norm, "H"), (silu, "I")])
def test_bad_group(lib, fn, key):
    assert fn(lib, mode=2, G=32) == GROUP
    assert fn(lib, mode=2, G=256) == GROUP
    assert fn(lib, mode=2, G=0) == GROUP
    assert fn(lib, mode=2, G=128, **{key: 1088}) == GROUP  # 1088 = 8.5 * 128
    # group_size is ignored outside per-group mode (T = 0 stops before launch)
    assert fn(lib, mode=0, G=7, T=0) == OK


@pytest.mark.parametrize("fn", [norm, silu])
def test_zero_tokens_is_ok_without_pointers(lib, fn):
    if fn is norm:
        assert norm(lib, q=None, r_out=None, scale=None, x=None, res=None, w=None, T=0) == OK
    else:
        assert silu(lib, q=None, scale=None, gu=None, T=0) == OK


def test_null_pointers(lib):
    for k in ("q", "scale", "x", "w"):
        assert norm(lib, **{k: None}) == NULL, k
    assert norm(lib, res=None) == NULL          # residual_out without residual
    assert norm(lib, r_out=None) == NULL        # residual without residual_out
    for k in ("q", "scale", "gu"):
        assert silu(lib, **{k: None}) == NULL, k


def test_misaligned(lib):
    for k in ("q", "r_out", "x", "res", "w"):
        assert norm(lib, **{k: A + 8}) == ALIGN, k
    assert norm(lib, scale=A + 2) == ALIGN
    assert silu(lib, q=A + 4) == ALIGN
    assert silu(lib, gu=A + 8) == ALIGN
    assert silu(lib, scale=A + 1) == ALIGN


def test_binding_rejects_cpu_tensors(lib):
    import torch
    x = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        vg.vg_silu_mul_fp8(torch.zeros(2, 32, dtype=torch.uint8), torch.ones(1), x, 0)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        vg.load(str(tmp_path / "absent.so"))


def test_device_status_rejects_null(lib):
    assert lib.vg_device_status(None, 0) == NULL


def mla(lib, q=A, kv=A, qc=A, qs=2112, qw=A, kc=A, ks=2112, kw=A, T=4, qd=1536, kd=512):
    return lib.vg_fused_mla_dual_rms_norm(q, kv, qc, qs, qw, kc, ks, kw, T, qd, kd,
                                          ctypes.c_float(1e-6), ctypes.c_float(1e-6), None)


def mla8(lib, q8=A, s=A, kv=A, qc=A, qs=2112, qw=A, kc=A, ks=2112, kw=A, T=4, qd=1536, kd=512):
    return lib.vg_fused_mla_dual_rms_norm_per_token_quant(q8, s, kv, qc, qs, qw, kc, ks, kw, T, qd,
                                                          kd, ctypes.c_float(1e-6),
                                                          ctypes.c_float(1e-6), None)


@pytest.mark.parametrize("fn", [mla, mla8])
def test_mla_bad_shape(lib, fn):
    for qd in (0, 4, 12, 32776):
        assert fn(lib, qd=qd, qs=40000) == SHAPE, qd
    for kd in (0, 1030, 65536):
        assert fn(lib, kd=kd, ks=70000) == SHAPE, kd
    assert fn(lib, qs=1528) == SHAPE          # stride below the row length
    assert fn(lib, ks=2116) == SHAPE          # stride not a multiple of 8
    assert fn(lib, T=-1) == SHAPE
    assert fn(lib, T=2 ** 31) == SHAPE


def test_mla_null_pointers(lib):
    for k in ("q", "kv", "qc", "qw", "kc", "kw"):
        assert mla(lib, **{k: None}) == NULL, k
    for k in ("q8", "s", "kv", "qc", "qw", "kc", "kw"):
        assert mla8(lib, **{k: None}) == NULL, k
    assert mla(lib, q=None, kv=None, qc=None, qw=None, kc=None, kw=None, T=0) == OK
    assert mla8(lib, q8=None, s=None, kv=None, qc=None, qw=None, kc=None, kw=None, T=0) == OK


def test_mla_misaligned(lib):
    for k in ("q", "kv", "qc", "qw", "kc", "kw"):
        assert mla(lib, **{k: A + 8}) == ALIGN, k
    assert mla8(lib, q8=A + 4) == ALIGN
    assert mla8(lib, s=A + 2) == ALIGN


def test_binding_mla_rejects_strided_columns(lib):
    import torch
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        vg.vg_fused_mla_dual_rms_norm(None, None, x, None, x, None, 1e-6, 1e-6)


def pad(lib, out=A, r_out=A, x=A, res=A, w=A, T=4, H=2880, Hp=3072, eps=1e-6):
    return lib.vg_fused_add_rms_norm_pad(out, r_out, x, res, w, T, H, Hp, ctypes.c_float(eps), None)


def test_pad_validation(lib):
    for H in (0, 4, 12, 32776):
        assert pad(lib, H=H, Hp=70000) == SHAPE, H
    assert pad(lib, Hp=2872) == SHAPE        # padded below hidden
    assert pad(lib, Hp=3076) == SHAPE        # not a multiple of 8
    assert pad(lib, Hp=65544) == SHAPE       # wider than 2 * VG_MAX_ROW
    assert pad(lib, T=-1) == SHAPE
    for k in ("out", "x", "w"):
        assert pad(lib, **{k: None}) == NULL, k
    assert pad(lib, res=None) == NULL
    assert pad(lib, r_out=None) == NULL
    assert pad(lib, out=None, r_out=None, x=None, res=None, w=None, T=0) == OK
    for k in ("out", "r_out", "x", "res", "w"):
        assert pad(lib, **{k: A + 8}) == ALIGN, k


def qk(lib, qkv=A, qw=A, kw=A, cache=A, pos=A, T=4, hq=32, hkv=8, D=128, maxp=4096, neox=1):
    return lib.vg_fused_qk_norm_rope(qkv, qw, kw, cache, pos, T, hq, hkv, D, maxp,
                                     ctypes.c_float(1e-6), neox, None)


def test_qk_validation(lib):
    for D in (0, 32, 96, 512):
        assert qk(lib, D=D) == SHAPE, D
    assert qk(lib, hq=0, hkv=0) == SHAPE
    assert qk(lib, hq=-1) == SHAPE
    assert qk(lib, hq=4000, hkv=100) == SHAPE   # more than 4096 heads in a row
    assert qk(lib, maxp=0) == SHAPE
    assert qk(lib, T=-1) == SHAPE
    for k in ("qkv", "qw", "kw", "cache", "pos"):
        assert qk(lib, **{k: None}) == NULL, k
    assert qk(lib, qkv=None, qw=None, kw=None, cache=None, pos=None, T=0) == OK
    for k in ("qkv", "qw", "kw", "cache"):
        assert qk(lib, **{k: A + 8}) == ALIGN, k
    assert qk(lib, pos=A + 4) == ALIGN


def nf_norm(lib, q4=A, sf=A, r_out=A, x=A, res=A, w=A, gs=A, T=4, H=4096):
    return lib.vg_fused_add_rms_norm_nvfp4(q4, sf, r_out, x, res, w, gs, T, H,
                                           ctypes.c_float(1e-6), None)


def nf_silu(lib, q4=A, sf=A, gu=A, gs=A, T=4, I=4096):
    return lib.vg_silu_mul_nvfp4(q4, sf, gu, gs, T, I, None)


def test_nvfp4_validation(lib):
    # row length: a multiple of 16 within [16, VG_MAX_ROW]
    for n in (0, 8, 24, 4104, 32784):
        assert nf_norm(lib, H=n) == SHAPE, n
        assert nf_silu(lib, I=n) == SHAPE, n
    assert nf_norm(lib, T=-1) == SHAPE
    assert nf_silu(lib, T=-1) == SHAPE
    for k in ("q4", "sf", "x", "w", "gs"):
        assert nf_norm(lib, **{k: None}) == NULL, k
    assert nf_norm(lib, res=None) == NULL
    assert nf_norm(lib, r_out=None) == NULL
    for k in ("q4", "sf", "gu", "gs"):
        assert nf_silu(lib, **{k: None}) == NULL, k
    assert nf_norm(lib, q4=None, sf=None, r_out=None, x=None, res=None, w=None, gs=None,
                   T=0) == OK
    assert nf_silu(lib, q4=None, sf=None, gu=None, gs=None, T=0) == OK
    for k in ("q4", "r_out", "x", "res", "w"):
        assert nf_norm(lib, **{k: A + 8}) == ALIGN, k
    assert nf_norm(lib, gs=A + 2) == ALIGN
    for k in ("q4", "gu"):
        assert nf_silu(lib, **{k: A + 8}) == ALIGN, k
    assert nf_silu(lib, gs=A + 2) == ALIGN


def test_header_is_plain_c():
    """The boundary header compiles as C99 and as C++ on its own (no CUDA or
    torch types in the signatures)."""
    import shutil
    h = os.path.join(ROOT, "include", "vg_fused.h")
    for cc, lang, std in (("gcc", "c", "-std=c99"), ("g++", "c++", "-std=c++11")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not available")
        subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-x", lang, h],
                       check=True, capture_output=True)
