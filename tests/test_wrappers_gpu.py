"""The allocating PyTorch wrappers (fused_add_rms_norm_fp8, silu_mul_fp8,
fused_add_rms_norm_pad, the NVFP4 pair) against the oracle: they pass bf16
tensors through the C ABI, allocate outputs of the right shape and dtype,
update the residual in place when asked, and return the same results as the
raw calls' parity tests require."""
import numpy as np
import pytest

import gen
import parity
import norm_activation_fp8_gb300 as vg

pytestmark = pytest.mark.gpu

OPT = vg.UE8M0 | vg.COLUMN_MAJOR


def _bf16(torch, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _scales(s, mode, T, n, G):
    a = s.cpu().numpy()
    if mode & vg.COLUMN_MAJOR:
        return np.ascontiguousarray(a.reshape(n // G, -1)[:, :T].T)
    return a.reshape(-1) if (mode & 0xFF) != vg.PER_GROUP else a.reshape(T, n // G)


@pytest.mark.parametrize("inplace", [True, False], ids=["in-place", "out-of-place"])
@pytest.mark.parametrize("mode,G", [(vg.STATIC, 128), (vg.PER_TOKEN, 128), (vg.PER_GROUP, 128),
                                    (vg.PER_GROUP, 64), (vg.PER_GROUP | OPT, 128)],
                         ids=["static", "per-token", "per-group128", "per-group64", "ue8m0-colmajor"])
def test_fused_add_rms_norm_fp8_wrapper(mode, G, inplace):
    import torch
    T, H = 333, 4096
    d = gen.norm_inputs(T, H, seed=11)
    x, res, w = _bf16(torch, d["x"]), _bf16(torch, d["residual"]), _bf16(torch, d["weight"])
    scale = torch.tensor([0.05], dtype=torch.float32, device="cuda") if mode == vg.STATIC else None
    res_before = res.clone()
    q, s, r_out = vg.fused_add_rms_norm_fp8(x, res, w, 1e-5, mode, G, scale=scale, inplace=inplace)
    torch.cuda.synchronize()
    assert q.dtype == torch.float8_e4m3fn and tuple(q.shape) == (T, H)
    assert (r_out is res) == inplace
    if not inplace:
        assert torch.equal(res, res_before)
    o = parity.oracle_norm(d["x"], d["residual"], d["weight"], 1e-5, mode, G, scale=0.05)
    g = {"q": q.view(torch.uint8).cpu().numpy(), "scale": _scales(s, mode, T, H, G),
         "residual_out": r_out.view(torch.int16).cpu().numpy().view(np.uint16)}
    parity.check_norm(g, o, mode)


def test_fused_add_rms_norm_fp8_wrapper_without_residual():
    import torch
    T, H = 64, 2048
    d = gen.norm_inputs(T, H, seed=12)
    q, s, r_out = vg.fused_add_rms_norm_fp8(_bf16(torch, d["x"]), None, _bf16(torch, d["weight"]),
                                           1e-6, vg.PER_TOKEN)
    torch.cuda.synchronize()
    assert r_out is None
    o = parity.oracle_norm(d["x"], None, d["weight"], 1e-6, vg.PER_TOKEN)
    parity.check_norm({"q": q.view(torch.uint8).cpu().numpy(), "scale": s.cpu().numpy(),
                       "residual_out": None}, o, vg.PER_TOKEN)


@pytest.mark.parametrize("mode,G", [(vg.STATIC, 128), (vg.PER_TOKEN, 128), (vg.PER_GROUP, 128),
                                    (vg.PER_GROUP | OPT, 128)],
                         ids=["static", "per-token", "per-group128", "ue8m0-colmajor"])
def test_silu_mul_fp8_wrapper(mode, G):
    import torch
    T, I = 400, 14336
    d = gen.silu_inputs(T, I, seed=13)
    scale = torch.tensor([0.1], dtype=torch.float32, device="cuda") if mode == vg.STATIC else None
    q, s = vg.silu_mul_fp8(_bf16(torch, d["gate_up"]), mode, G, scale=scale)
    torch.cuda.synchronize()
    assert q.dtype == torch.float8_e4m3fn and tuple(q.shape) == (T, I)
    o = parity.oracle_silu(d["gate_up"], mode, G, scale=0.1)
    parity.check_silu({"q": q.view(torch.uint8).cpu().numpy(), "scale": _scales(s, mode, T, I, G)},
                      o, mode)


def test_fused_add_rms_norm_pad_wrapper():
    import torch
    T, H, P = 300, 2880, 3072
    d = gen.norm_inputs(T, H, seed=14)
    res = _bf16(torch, d["residual"])
    out, r_out = vg.fused_add_rms_norm_pad(_bf16(torch, d["x"]), res, _bf16(torch, d["weight"]),
                                           1e-5, P)
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == (T, P) and r_out is res
    o = parity.oracle_pad(d["x"], d["residual"], d["weight"], 1e-5, P)
    parity.check_pad({"out": out.view(torch.int16).cpu().numpy().view(np.uint16),
                      "residual_out": r_out.view(torch.int16).cpu().numpy().view(np.uint16)}, o)


def test_nvfp4_wrappers():
    import torch
    gs = torch.tensor([168.0], dtype=torch.float32, device="cuda")
    T, H = 300, 8192
    d = gen.norm_inputs(T, H, seed=15)
    q4, sf, r_out = vg.fused_add_rms_norm_nvfp4(_bf16(torch, d["x"]), _bf16(torch, d["residual"]),
                                                _bf16(torch, d["weight"]), 1e-5, gs)
    torch.cuda.synchronize()
    assert tuple(q4.shape) == (T, H // 2) and tuple(sf.shape) == (T, H // 16)
    o = parity.oracle_nvfp4_norm(d["x"], d["residual"], d["weight"], 1e-5, 168.0)
    parity.check_nvfp4({"q4": q4.cpu().numpy(), "sf": sf.view(torch.uint8).cpu().numpy(),
                        "residual_out": r_out.view(torch.int16).cpu().numpy().view(np.uint16)}, o)
    I = 14336
    ds = gen.silu_inputs(T, I, seed=16)
    q4, sf = vg.silu_mul_nvfp4(_bf16(torch, ds["gate_up"]), gs)
    torch.cuda.synchronize()
    assert tuple(q4.shape) == (T, I // 2) and tuple(sf.shape) == (T, I // 16)
    o = parity.oracle_nvfp4_silu(ds["gate_up"], 168.0)
    parity.check_nvfp4({"q4": q4.cpu().numpy(), "sf": sf.view(torch.uint8).cpu().numpy()}, o)
