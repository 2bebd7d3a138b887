"""Back-to-back dependent calls on one stream, with no host synchronisation
between them (GPU).

The register kernels are launched with programmatic dependent launch: a
grid may start while the previous kernel in the stream drains, and waits
for it (griddepcontrol.wait) before touching memory.  Here every call reads
what the call before it wrote: a chain of in-place norm calls on one
residual buffer, then a torch kernel that builds gate_up from the final
residual, then the SiLU call on it.  The chain runs eagerly and captured in
a CUDA graph, and must equal the oracle applied in the same order.
"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import parity

pytestmark = pytest.mark.gpu

STATIC, PER_TOKEN, PER_GROUP = 0, 1, 2
CHAIN = 4


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from norm_activation_fp8_gb300 import build
    build.build()
    import norm_activation_fp8_gb300 as vg
    vg.load()


def _oracle_chain(xs, res0, w, mode, G):
    res = res0
    outs = []
    for x in xs:
        o = parity.oracle_norm(x, res, w, 1e-5, mode, G, scale=0.05)
        outs.append(o)
        res = o["residual_out"]
    gu = np.concatenate([res, xs[0]], axis=1)  # gate = final residual, up = x_0
    return outs, res, parity.oracle_silu(gu, mode, G, scale=0.1)


class _Chain:
    """Device buffers of one chain: CHAIN norm calls on one residual, then a
    torch-built gate_up and the SiLU call."""

    def __init__(self, torch, xs, res0, w, mode, G):
        T, H = res0.shape
        dev = "cuda"
        self.torch, self.mode, self.G, self.T, self.H = torch, mode, G, T, H
        self.xs = [torch.from_numpy(x.view(np.int16)).to(dev) for x in xs]
        self.res0 = torch.from_numpy(res0.view(np.int16)).to(dev)
        self.res = torch.empty_like(self.res0)
        self.w = torch.from_numpy(w.view(np.int16)).to(dev)
        self.qs = [torch.empty((T, H), dtype=torch.uint8, device=dev) for _ in xs]
        self.ss = [self._scale(T, H) for _ in xs]
        self.gu = torch.empty((T, 2 * H), dtype=torch.int16, device=dev)
        self.q_act = torch.empty((T, H), dtype=torch.uint8, device=dev)
        self.s_act = self._scale(T, H, 0.1)

    def _scale(self, T, n, static=0.05):
        torch = self.torch
        if self.mode == STATIC:
            return torch.full((1,), static, dtype=torch.float32, device="cuda")
        if self.mode == PER_TOKEN:
            return torch.empty((T,), dtype=torch.float32, device="cuda")
        return torch.empty((T, n // self.G), dtype=torch.float32, device="cuda")

    def run(self):
        import norm_activation_fp8_gb300 as vg
        self.res.copy_(self.res0)
        for x, q, s in zip(self.xs, self.qs, self.ss):
            vg.vg_fused_add_rms_norm_fp8(q, self.res, s, x, self.res, self.w, 1e-5, self.mode,
                                         self.G)
        # a torch kernel writes gate_up from what the last norm call wrote
        self.gu[:, :self.H].copy_(self.res)
        self.gu[:, self.H:].copy_(self.xs[0])
        vg.vg_silu_mul_fp8(self.q_act, self.s_act, self.gu, self.mode, self.G)

    def check(self, outs, res, act):
        for k, o in enumerate(outs):
            g = {"q": self.qs[k].cpu().numpy(), "scale": self.ss[k].cpu().numpy().reshape(
                o["scale"].shape)}
            # each call's residual_out is the next call's input: only the
            # final one is still in the buffer
            parity.check_norm(g, dict(o, residual_out=None), self.mode)
        parity.compare_exact(self.res.cpu().numpy().view(np.uint16), res, "final residual")
        g = {"q": self.q_act.cpu().numpy(), "scale": self.s_act.cpu().numpy().reshape(
            act["scale"].shape)}
        parity.check_silu(g, act, self.mode)

    def clear_outputs(self):
        for q in self.qs + [self.q_act]:
            q.fill_(0xAA)
        if self.mode != STATIC:
            for s in self.ss + [self.s_act]:
                s.fill_(-1.0)


@pytest.mark.parametrize("mode,G", [(STATIC, 128), (PER_TOKEN, 128), (PER_GROUP, 128)],
                         ids=["static", "per_token", "per_group"])
@pytest.mark.parametrize("T", [64, 1024], ids=["register", "pipelined"])
def test_dependent_chain_eager_and_graph(T, mode, G):
    import torch
    H = 4096
    xs = [gen.norm_inputs(T, H, seed=40 + k)["x"] for k in range(CHAIN)]
    res0 = gen.norm_inputs(T, H, seed=50)["residual"]
    w = gen.norm_inputs(T, H, seed=50)["weight"]
    outs, res, act = _oracle_chain(xs, res0, w, mode, G)
    ch = _Chain(torch, xs, res0, w, mode, G)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ch.run()  # eager: no synchronisation inside the chain
    torch.cuda.synchronize()
    ch.check(outs, res, act)

    ch.clear_outputs()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        ch.run()
    ch.clear_outputs()
    torch.cuda.synchronize()
    for _ in range(2):  # replays start from the pristine residual each time
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        ch.check(outs, res, act)
        ch.clear_outputs()
        torch.cuda.synchronize()
