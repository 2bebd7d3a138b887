"""Each kernel asks its first input rows into L2 before it waits on the
previous grid (programmatic dependent launch).  These chains make the
previous kernel in the stream WRITE exactly those rows, with no host
synchronisation in between, so a prefetch races the writes it must not
overtake: QK norm + RoPE twice in place on one buffer; a torch kernel that
rewrites the MLA dual norm's projected tensor (or the SiLU's gate_up) right
before each call.  Run eagerly and in a CUDA graph, every chain must equal
the same calls with a device synchronisation between them, bit for bit.
(Each call's parity against the oracle is covered elsewhere.)"""
from __future__ import annotations

import numpy as np
import pytest

import gen
import norm_activation_fp8_gb300 as vg

pytestmark = pytest.mark.gpu


def _run_both_ways(torch, build, run, outputs):
    """run(sync) issues the chain (with a synchronisation between calls when
    sync is True); returns the outputs of the synchronised run, of an eager
    run without synchronisation, and of two replays of a graph of it."""
    stream = torch.cuda.Stream()
    results = []
    for mode in ("sync", "eager", "graph"):
        build()
        torch.cuda.synchronize()
        if mode == "graph":
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run(False)
            for _ in range(2):
                build()
                torch.cuda.synchronize()
                with torch.cuda.stream(stream):
                    g.replay()
                torch.cuda.synchronize()
                results.append([o.clone() for o in outputs()])
        else:
            with torch.cuda.stream(stream):
                run(mode == "sync")
            torch.cuda.synchronize()
            results.append([o.clone() for o in outputs()])
    ref = results[0]
    for res in results[1:]:
        for a, b in zip(ref, res):
            assert torch.equal(a, b)


@pytest.mark.parametrize("T", [1, 64, 1000], ids=["decode", "register", "many"])
def test_qk_norm_rope_twice_in_place(T):
    import torch
    d = gen.qk_inputs(T, 32, 8, 128, 4096, seed=T)
    dev = "cuda"
    src = torch.from_numpy(d["qkv"].view(np.int16)).to(dev)
    qkv = torch.empty_like(src)
    qw = torch.from_numpy(d["q_weight"].view(np.int16)).to(dev)
    kw = torch.from_numpy(d["k_weight"].view(np.int16)).to(dev)
    cache = torch.from_numpy(d["cos_sin_cache"]).to(dev)
    pos = torch.from_numpy(d["positions"]).to(dev)

    def run(sync):
        for _ in range(2):
            vg.vg_fused_qk_norm_rope(qkv, qw, kw, cache, pos, 32, 8, 128, 1e-6, True)
            if sync:
                torch.cuda.synchronize()

    _run_both_ways(torch, lambda: qkv.copy_(src), run, lambda: [qkv])


@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "fp8"])
@pytest.mark.parametrize("T", [64, 2048, 7400], ids=["group", "warp-wave", "warp"])
def test_mla_after_a_rewrite_of_its_input(T, fp8):
    import torch
    q_dim, kv_dim, rope = gen.MLA_Q_DIM, gen.MLA_KV_DIM, 64
    dev = "cuda"
    d0 = gen.mla_inputs(T, q_dim, kv_dim, seed=T)
    d1 = gen.mla_inputs(T, q_dim, kv_dim, seed=T + 1)

    def proj(d):
        p = np.zeros((T, q_dim + kv_dim + rope), np.uint16)
        p[:, :q_dim], p[:, q_dim:q_dim + kv_dim] = d["q_c"], d["kv_c"]
        return torch.from_numpy(p.view(np.int16)).to(dev)

    srcs = [proj(d0), proj(d1)]
    pt = torch.empty_like(srcs[0])
    qc, kc = pt[:, :q_dim], pt[:, q_dim:q_dim + kv_dim]
    qw = torch.from_numpy(d0["q_weight"].view(np.int16)).to(dev)
    kw = torch.from_numpy(d0["kv_weight"].view(np.int16)).to(dev)
    outs = []
    for _ in srcs:
        kv = torch.empty((T, kv_dim), dtype=torch.int16, device=dev)
        q = torch.empty((T, q_dim), dtype=torch.uint8 if fp8 else torch.int16, device=dev)
        s = torch.empty((T,), dtype=torch.float32, device=dev) if fp8 else None
        outs.append((q, s, kv))

    def run(sync):
        for src, (q, s, kv) in zip(srcs, outs):
            pt.copy_(src)  # a torch kernel writes the rows the next call prefetches
            if fp8:
                vg.vg_fused_mla_dual_rms_norm_per_token_quant(q, s, kv, qc, qw, kc, kw, 1e-6, 1e-6)
            else:
                vg.vg_fused_mla_dual_rms_norm(q, kv, qc, qw, kc, kw, 1e-6, 1e-6)
            if sync:
                torch.cuda.synchronize()

    def outputs():
        return [t for o in outs for t in o if t is not None]

    _run_both_ways(torch, lambda: [t.fill_(0) for t in outputs()], run, outputs)


@pytest.mark.parametrize("mode", [gen.STATIC, gen.PER_GROUP, gen.PER_TOKEN], ids=["static", "per_group", "per_token"])
@pytest.mark.parametrize("T", [64, 400], ids=["register", "dense"])
def test_silu_after_a_rewrite_of_its_input(T, mode):
    import torch
    I = 14336
    dev = "cuda"
    srcs = [torch.from_numpy(gen.silu_inputs(T, I, seed=T + k)["gate_up"].view(np.int16)).to(dev)
            for k in range(2)]
    gu = torch.empty_like(srcs[0])
    static = torch.full((1,), 0.1, dtype=torch.float32, device=dev)  # an input, not rewritten
    outs = []
    for _ in srcs:
        q = torch.empty((T, I), dtype=torch.uint8, device=dev)
        s = static if mode == gen.STATIC else torch.empty(
            (T,) if mode == gen.PER_TOKEN else (T, I // 128), dtype=torch.float32, device=dev)
        outs.append((q, s))

    def run(sync):
        for src, (q, s) in zip(srcs, outs):
            gu.copy_(src)
            vg.vg_silu_mul_fp8(q, s, gu, mode, 128)
            if sync:
                torch.cuda.synchronize()

    def outputs():
        return [t for o in outs for t in o if t is not static]

    _run_both_ways(torch, lambda: [t.fill_(0) for t in outputs()], run, outputs)
