"""Every point of the widened sweeps (MLA dual norm, padded norm, QK norm +
RoPE, NVFP4, per-group scale options) against the oracle, in the launch
configuration bench.py --sweep times: the GPU runs the whole point; points
above 64 Mi elements are checked on 192 sampled rows (first, last and random
ones; rows are independent), the rest on every row."""
import numpy as np
import pytest

import gen
import parity

pytestmark = pytest.mark.gpu


def _rows(T, n):
    if T * n <= 64 * 2 ** 20:
        return None
    rng = np.random.default_rng(0)
    return np.array(sorted(set(rng.choice(T, 188, replace=False).tolist()) | {0, 1, T - 2, T - 1}))


def _sel(a, rows):
    return a if rows is None or a is None else a[rows]


POINTS = (gen.mla_workloads() + gen.pad_workloads() + gen.qk_workloads() + gen.nvfp4_workloads()
          + gen.group_option_workloads())


@pytest.mark.parametrize("w", POINTS, ids=lambda w: w.name)
def test_widened_sweep_point(w):
    d = w.inputs()
    if w.op == "mla":
        fp8 = w.mode == gen.PER_TOKEN
        g = parity.gpu_mla(d["q_c"], d["q_weight"], d["kv_c"], d["kv_weight"], w.eps, w.eps, fp8)
        rows = _rows(w.T, w.n + w.n2)
        o = parity.oracle_mla(_sel(d["q_c"], rows), d["q_weight"], _sel(d["kv_c"], rows),
                              d["kv_weight"], w.eps, w.eps, fp8)
        parity.check_mla({k: _sel(v, rows) for k, v in g.items()}, o, fp8)
    elif w.op == "pad":
        g = parity.gpu_pad(d["x"], d["residual"], d["weight"], w.eps, w.n2)
        rows = _rows(w.T, w.n)
        o = parity.oracle_pad(_sel(d["x"], rows), _sel(d["residual"], rows), d["weight"], w.eps, w.n2)
        parity.check_pad({k: _sel(v, rows) for k, v in g.items()}, o)
    elif w.op == "qk":
        neox = w.mode == 1
        qkv_in = d["qkv"]
        g = parity.gpu_qk(d, w.hq, w.hkv, w.n, w.eps, neox)
        rows = _rows(w.T, qkv_in.shape[1])
        sub = dict(d, qkv=_sel(qkv_in, rows), positions=_sel(d["positions"], rows))
        o = parity.oracle_qk(sub, w.hq, w.hkv, w.n, w.eps, neox)
        parity.check_qk(_sel(g, rows), o, sub["qkv"], w.hq, w.hkv, w.n)
    elif w.op == "norm4":
        g = parity.gpu_nvfp4_norm(d["x"], d["residual"], d["weight"], w.eps, w.static_scale)
        rows = _rows(w.T, w.n)
        o = parity.oracle_nvfp4_norm(_sel(d["x"], rows), _sel(d["residual"], rows), d["weight"],
                                     w.eps, w.static_scale)
        parity.check_nvfp4(g, o, rows=rows)
    elif w.op == "silu4":
        g = parity.gpu_nvfp4_silu(d["gate_up"], w.static_scale)
        rows = _rows(w.T, w.n)
        o = parity.oracle_nvfp4_silu(_sel(d["gate_up"], rows), w.static_scale)
        parity.check_nvfp4(g, o, rows=rows)
    elif w.op == "norm":
        mode = w.mode | w.flags
        g = parity.gpu_norm(d["x"], d["residual"], d["weight"], w.eps, mode, w.group_size)
        rows = _rows(w.T, w.n)
        o = parity.oracle_norm(_sel(d["x"], rows), _sel(d["residual"], rows), d["weight"], w.eps,
                               mode, w.group_size)
        parity.check_norm(g, o, w.mode, rows=rows)
    else:
        mode = w.mode | w.flags
        g = parity.gpu_silu(d["gate_up"], mode, w.group_size)
        rows = _rows(w.T, w.n)
        o = parity.oracle_silu(_sel(d["gate_up"], rows), mode, w.group_size)
        parity.check_silu(g, o, w.mode, rows=rows)
