"""Device bounds checks, in a test-only debug build of the library.

The debug copy (VG_DEBUG_CHECKS) checks every global store, and the source
of every bulk copy, against the extent of the tensor it touches; an access
outside is skipped and reported as VG_DEVICE_OUT_OF_BOUNDS, so an indexing
mistake shows up as a status flag instead of a fault or overwritten memory.

(1) On every entry point and launch form the debug copy writes exactly the
product library's outputs and reports nothing: no kernel computes an address
outside its tensors.  (2) A copy that reports every tensor one row short
flags the last row's accesses, skips them and leaves every other row as the
product library writes it; the context stays usable.  Nothing here faults.
"""
import numpy as np
import pytest

import gen
import parity
import norm_activation_fp8_gb300 as vg
from norm_activation_fp8_gb300 import build

pytestmark = pytest.mark.gpu

PT, PG, ST = gen.PER_TOKEN, gen.PER_GROUP, gen.STATIC
OPT = gen.UE8M0 | gen.COL_MAJOR


def _norm(T, H, mode, G=128):
    d = gen.norm_inputs(T, H, seed=T + H)
    return lambda: parity.gpu_norm(d["x"], d["residual"], d["weight"], 1e-5, mode, G, scale=0.05)


def _silu(T, I, mode, G=128):
    d = gen.silu_inputs(T, I, seed=T + I)
    return lambda: parity.gpu_silu(d["gate_up"], mode, G, scale=0.1)


def _mla(T, fp8, q_dim=gen.MLA_Q_DIM, kv_dim=gen.MLA_KV_DIM):
    d = gen.mla_inputs(T, q_dim, kv_dim, seed=T)
    return lambda: parity.gpu_mla(d["q_c"], d["q_weight"], d["kv_c"], d["kv_weight"], 1e-6, 1e-6, fp8)


def _pad(T):
    d = gen.norm_inputs(T, 2880, seed=T)
    return lambda: parity.gpu_pad(d["x"], d["residual"], d["weight"], 1e-5, 3072)


def _nvfp4_norm(T, H):
    d = gen.norm_inputs(T, H, seed=T + H)
    return lambda: parity.gpu_nvfp4_norm(d["x"], d["residual"], d["weight"], 1e-5, 168.0)


def _nvfp4_silu(T, I):
    d = gen.silu_inputs(T, I, seed=T + I)
    return lambda: parity.gpu_nvfp4_silu(d["gate_up"], 168.0)


def _qk(T):
    d = gen.qk_inputs(T, 32, 8, 128, 4096, seed=T)
    return lambda: {"qkv": parity.gpu_qk(d, 32, 8, 128, 1e-6, True)}


# every kernel and launch form: register and persistent norms (128- and
# 256-thread rows), scale options, NVFP4, padding; SiLU row segments (three
# and four CTAs per SM), per-token register and pipelined; MLA warp-group,
# warp and staged warp kernels; QK norm + RoPE
CASES = {
    "norm-static-64x4096": _norm(64, 4096, ST),
    "norm-token-256x4096": _norm(256, 4096, PT),
    "norm-group-1000x4096-tma": _norm(1000, 4096, PG),
    "norm-token-700x8192-tma": _norm(700, 8192, PT),
    "norm-group-ue8m0-colmajor-700x8192": _norm(700, 8192, PG | OPT),
    "norm-nvfp4-700x8192": _nvfp4_norm(700, 8192),
    "norm-pad-700x2880": _pad(700),
    "silu-static-300x14336": _silu(300, 14336, ST),
    "silu-static-400x14336-dense": _silu(400, 14336, ST),
    "silu-group-64x14336": _silu(64, 14336, PG),
    "silu-group-400x14336-dense": _silu(400, 14336, PG),
    "silu-token-256x14336": _silu(256, 14336, PT),
    "silu-token-400x14336-tma": _silu(400, 14336, PT),
    "silu-group-ue8m0-colmajor-400x14336": _silu(400, 14336, PG | OPT),
    "silu-nvfp4-400x14336": _nvfp4_silu(400, 14336),
    "mla-bf16-64": _mla(64, False),
    "mla-fp8-2048-wave": _mla(2048, True),
    "mla-fp8-2100-registers-wave": _mla(2100, True, 1024, 512),
    "mla-bf16-5000-registers": _mla(5000, False, 1024, 512),
    "mla-bf16-7400-staged": _mla(7400, False),
    "mla-fp8-7400-staged": _mla(7400, True),
    "qk-neox-64": _qk(64),
}


def _outputs(run, lib, monkeypatch):
    with monkeypatch.context() as m:
        m.setattr(vg, "_lib", lib)
        vg.vg_device_status(reset=True)
        out = run()
        return out, vg.vg_device_status(reset=True)


@pytest.mark.parametrize("case", sorted(CASES))
def test_debug_build_matches_and_reports_nothing(case, monkeypatch):
    product = vg.load()
    debug = vg.load(build.build_debug())
    want, st0 = _outputs(CASES[case], product, monkeypatch)
    got, st = _outputs(CASES[case], debug, monkeypatch)
    assert st0 == 0 and st == 0, (st0, st)
    for k, v in want.items():
        if v is not None:
            assert np.array_equal(got[k], v), k


SHRUNK = ["norm-token-256x4096", "norm-group-1000x4096-tma", "silu-token-400x14336-tma",
          "silu-group-400x14336-dense", "silu-static-400x14336-dense", "mla-fp8-7400-staged",
          "mla-fp8-2048-wave", "mla-bf16-5000-registers", "qk-neox-64"]


@pytest.mark.parametrize("case", SHRUNK)
def test_out_of_range_accesses_are_flagged_and_skipped(case, monkeypatch):
    product = vg.load()
    shrunk = vg.load(build.build_debug(shrunk=True))
    want, _ = _outputs(CASES[case], product, monkeypatch)
    got, st = _outputs(CASES[case], shrunk, monkeypatch)
    assert st & vg.DEVICE_OUT_OF_BOUNDS, st
    for k, v in want.items():
        if v is None or v.ndim < 2:
            continue
        assert np.array_equal(got[k][:-1], v[:-1]), k  # every row but the last as usual
    # the context is still good, and the product library reports nothing
    again, st2 = _outputs(CASES[case], product, monkeypatch)
    assert st2 == 0
    for k, v in want.items():
        if v is not None:
            assert np.array_equal(again[k], v), k
