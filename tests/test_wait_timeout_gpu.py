"""A bounded wait that runs out is reported, and the context stays usable.

A test-only copy of the library (built with VG_TEST_FORCE_WAIT_TIMEOUT and a
4096-poll limit) makes every CTA of the pipelined kernels also wait, after its
first stage wait, on a shared-memory barrier that nothing arrives on.  That
wait gives up, the CTA leaves its loop at the next barrier, records
VG_DEVICE_WAIT_TIMEOUT, waits (bounded) for its real copies, which do
complete, and returns.  No fault, trap or hang is involved."""
import ctypes

import numpy as np
import pytest

import gen
import parity
import norm_activation_fp8_gb300 as vg
from norm_activation_fp8_gb300 import build

pytestmark = pytest.mark.gpu


def _status(lib, reset):
    flags = ctypes.c_uint32(0)
    assert lib.vg_device_status(ctypes.byref(flags), 1 if reset else 0) == 0
    return flags.value


def test_forced_wait_timeout_is_reported_and_context_survives():
    import torch
    lib = vg.load(build.build_wait_test())  # its own copy, with its own status word
    dev = "cuda"
    _status(lib, reset=True)
    # the pipelined dynamic norm (T >= 4 rows per SM, H >= 2048) ...
    T, H = 4096, 4096
    d = gen.norm_inputs(T, H, seed=2)
    x = torch.from_numpy(d["x"].view(np.int16)).to(dev)
    r = torch.from_numpy(d["residual"].view(np.int16)).to(dev)
    w = torch.from_numpy(d["weight"].view(np.int16)).to(dev)
    q = torch.empty(T, H, dtype=torch.uint8, device=dev)
    s = torch.empty(T, dtype=torch.float32, device=dev)
    st = lib.vg_fused_add_rms_norm_fp8(q.data_ptr(), r.data_ptr(), s.data_ptr(), x.data_ptr(),
                                       r.data_ptr(), w.data_ptr(), T, H, ctypes.c_float(1e-5),
                                       vg.PER_TOKEN, 128, None)
    assert st == 0
    torch.cuda.synchronize()
    assert _status(lib, reset=True) & vg.DEVICE_WAIT_TIMEOUT
    assert _status(lib, reset=False) == 0  # the reset cleared it
    # ... and the pipelined per-token SiLU (two half-row stages)
    T, I = 1024, 14336
    gu = torch.from_numpy(gen.silu_inputs(T, I, seed=3)["gate_up"].view(np.int16)).to(dev)
    q = torch.empty(T, I, dtype=torch.uint8, device=dev)
    s = torch.empty(T, dtype=torch.float32, device=dev)
    st = lib.vg_silu_mul_fp8(q.data_ptr(), s.data_ptr(), gu.data_ptr(), T, I, vg.PER_TOKEN, 128,
                             None)
    assert st == 0
    torch.cuda.synchronize()
    assert _status(lib, reset=True) & vg.DEVICE_WAIT_TIMEOUT

    # the context is still good: the product library runs the same shapes and
    # matches the oracle, and its own status word never saw a timeout
    vg.vg_device_status(reset=True)
    d = gen.norm_inputs(1024, 4096, seed=4)
    g = parity.gpu_norm(d["x"], d["residual"], d["weight"], 1e-5, vg.PER_TOKEN, 128)
    o = parity.oracle_norm(d["x"], d["residual"], d["weight"], 1e-5, vg.PER_TOKEN, 128)
    parity.check_norm(g, o, vg.PER_TOKEN)
    gs = parity.gpu_silu(gen.silu_inputs(700, 14336, seed=5)["gate_up"], vg.PER_TOKEN)
    os_ = parity.oracle_silu(gen.silu_inputs(700, 14336, seed=5)["gate_up"], vg.PER_TOKEN)
    parity.check_silu(gs, os_, vg.PER_TOKEN)
    assert vg.vg_device_status() == 0
