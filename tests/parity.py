"""Parity helpers: run the oracle (row-parallel) and the CUDA path on the same
seeded bytes, and compare them with the tolerance the benchmark spec fixes:

  residual_out  bf16, bit-exact
  bf16 norm outputs (MLA dual norm, padded norm): bit-exact (the kernels
                round the exact product)
  bf16 QK norm + RoPE outputs: compare_bf16 (one ulp, only within 2^-19 of
                a bf16 midpoint, at most 0.1 % of the elements)
  scale         |s_gpu - s_oracle| <= 1e-6 * |s_oracle|
  q             identical codes, except codes adjacent in value (1 ULP, same
                sign) where the oracle's pre-rounding value v = y/s lies
                within 1e-3 relative of the midpoint of the two codes; such
                flips may be at most 0.01 % of the elements; wherever
                |v| >= 448 (saturation) the codes agree exactly.
  NVFP4         block scale codes bit-exact; E2M1 element codes under the
                same rule (adjacent codes near a midpoint, at most 0.01 %,
                exact wherever |v| >= 6)
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import exact
import oracle

SCALE_RTOL = 1e-6
MIDPOINT_RTOL = 1e-3
FLIP_FRACTION = 1e-4

_E4M3_MAG = exact.E4M3_POS_F64  # magnitude of codes 0x00..0x7E


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


def _blocks(rows, nblk):
    step = max(1, (rows + nblk - 1) // nblk)
    return [(r, min(rows, r + step)) for r in range(0, rows, step)]


# ------------------------------------------------------------------ oracle

def _oracle_mode(mode):
    """The oracle runs a mode's arithmetic with row-major scales; the layout
    itself is pinned in the oracle's own tests."""
    return mode & ~COL_MAJOR


def oracle_norm(x, residual, weight, eps, mode, group_size=128, scale=None, want_v=True):
    """The oracle over all rows of x, split into row blocks run in threads
    (rows are independent; the oracle releases the GIL in its C code)."""
    T, H = x.shape
    out = {"q": np.empty((T, H), np.uint8),
           "residual_out": None if residual is None else np.empty((T, H), np.uint16),
           "v": np.empty((T, H), np.float64) if want_v else None}
    base = mode & 0xFF
    mode = _oracle_mode(mode)
    if base == 0:
        out["scale"] = np.array([np.float32(scale)], np.float32)
    elif base == 1:
        out["scale"] = np.empty((T,), np.float32)
    else:
        out["scale"] = np.empty((T, H // group_size), np.float32)

    def work(b):
        r0, r1 = b
        o = oracle.fused_add_rms_norm_fp8(x[r0:r1], None if residual is None else residual[r0:r1],
                                          weight, eps, mode, group_size, scale=scale,
                                          want_v=want_v)
        out["q"][r0:r1] = o["q"]
        if residual is not None:
            out["residual_out"][r0:r1] = o["residual_out"]
        if want_v:
            out["v"][r0:r1] = o["v"]
        if mode != 0:
            out["scale"][r0:r1] = o["scale"]

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, _blocks(T, 4 * _threads())))
    return out


def oracle_silu(gate_up, mode, group_size=128, scale=None, want_v=True):
    T, two_i = gate_up.shape
    I = two_i // 2
    out = {"q": np.empty((T, I), np.uint8), "v": np.empty((T, I), np.float64) if want_v else None}
    base = mode & 0xFF
    mode = _oracle_mode(mode)
    if base == 0:
        out["scale"] = np.array([np.float32(scale)], np.float32)
    elif base == 1:
        out["scale"] = np.empty((T,), np.float32)
    else:
        out["scale"] = np.empty((T, I // group_size), np.float32)

    def work(b):
        r0, r1 = b
        o = oracle.silu_mul_fp8(gate_up[r0:r1], mode, group_size, scale=scale, want_v=want_v)
        out["q"][r0:r1] = o["q"]
        if want_v:
            out["v"][r0:r1] = o["v"]
        if mode != 0:
            out["scale"][r0:r1] = o["scale"]

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, _blocks(T, 4 * _threads())))
    return out


def oracle_nvfp4_norm(x, residual, weight, eps, gs, want_v=True):
    T, H = x.shape
    out = {"q4": np.empty((T, H // 2), np.uint8), "sf": np.empty((T, H // 16), np.uint8),
           "residual_out": None if residual is None else np.empty((T, H), np.uint16),
           "v": np.empty((T, H), np.float64) if want_v else None}

    def work(b):
        r0, r1 = b
        o = oracle.fused_add_rms_norm_nvfp4(x[r0:r1], None if residual is None else residual[r0:r1],
                                            weight, eps, gs, want_v=want_v)
        for k in ("q4", "sf", "residual_out", "v"):
            if out[k] is not None:
                out[k][r0:r1] = o[k]

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, _blocks(T, 4 * _threads())))
    return out


def oracle_nvfp4_silu(gate_up, gs, want_v=True):
    T, two_i = gate_up.shape
    I = two_i // 2
    out = {"q4": np.empty((T, I // 2), np.uint8), "sf": np.empty((T, I // 16), np.uint8),
           "v": np.empty((T, I), np.float64) if want_v else None}

    def work(b):
        r0, r1 = b
        o = oracle.silu_mul_nvfp4(gate_up[r0:r1], gs, want_v=want_v)
        for k in ("q4", "sf", "v"):
            if out[k] is not None:
                out[k][r0:r1] = o[k]

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, _blocks(T, 4 * _threads())))
    return out


# ------------------------------------------------------------------ compare

class ParityError(AssertionError):
    pass


def compare_codes(q_gpu, q_orc, v_orc, what="q"):
    """Applies the FP8 code rule; returns statistics, raises ParityError."""
    q_gpu = np.asarray(q_gpu, np.uint8).reshape(-1)
    q_orc = np.asarray(q_orc, np.uint8).reshape(-1)
    v = np.asarray(v_orc, np.float64).reshape(-1)
    n = q_orc.size
    diff = np.flatnonzero(q_gpu != q_orc)
    stats = {"elements": n, "mismatch": int(diff.size), "flips": 0, "max_flip_rel_dist": 0.0}
    if diff.size == 0:
        return stats
    a, b, vv = q_gpu[diff], q_orc[diff], v[diff]
    same_sign = (a & 0x80) == (b & 0x80)
    ma, mb = (a & 0x7F).astype(np.int32), (b & 0x7F).astype(np.int32)
    adjacent = same_sign & (np.abs(ma - mb) == 1) & (ma <= 0x7E) & (mb <= 0x7E)
    bad = ~adjacent
    mid = np.zeros_like(vv)
    ok = adjacent
    mid[ok] = (_E4M3_MAG[ma[ok]] + _E4M3_MAG[mb[ok]]) / 2.0
    rel = np.full_like(vv, np.inf)
    rel[ok] = np.abs(np.abs(vv[ok]) - mid[ok]) / mid[ok]
    bad |= rel > MIDPOINT_RTOL
    bad |= np.abs(vv) >= 448.0
    if np.any(bad):
        i = diff[np.flatnonzero(bad)[:8]]
        raise ParityError(f"{what}: {int(bad.sum())} codes outside tolerance, e.g. "
                          + ", ".join(f"[{k}] gpu={q_gpu[k]:#04x} oracle={q_orc[k]:#04x} v={v[k]!r}"
                                      for k in i))
    stats["flips"] = int(diff.size)
    stats["max_flip_rel_dist"] = float(rel.max())
    if diff.size > FLIP_FRACTION * n:
        raise ParityError(f"{what}: {diff.size} near-midpoint flips in {n} elements "
                          f"(> {FLIP_FRACTION:.2%})")
    return stats


def compare_scales(s_gpu, s_orc, what="scale"):
    """Finite scales within 1e-6 relative; a non-finite oracle scale (an
    infinite amax) must be the same non-finite value."""
    s_gpu = np.asarray(s_gpu, np.float32).astype(np.float64).reshape(-1)
    s_orc = np.asarray(s_orc, np.float32).astype(np.float64).reshape(-1)
    if s_gpu.shape != s_orc.shape:
        raise ParityError(f"{what}: shape {s_gpu.shape} != {s_orc.shape}")
    fin = np.isfinite(s_orc)
    odd = ~fin & ~((s_gpu == s_orc) | (np.isnan(s_gpu) & np.isnan(s_orc)))
    if np.any(odd) or np.any(fin & ~np.isfinite(s_gpu)):
        i = np.flatnonzero(odd | (fin & ~np.isfinite(s_gpu)))[:8]
        raise ParityError(f"{what}: non-finite scales differ, e.g. "
                          + ", ".join(f"[{k}] {s_gpu[k]!r} vs {s_orc[k]!r}" for k in i))
    s_gpu, s_orc = s_gpu[fin], s_orc[fin]
    err = np.abs(s_gpu - s_orc)
    bad = err > SCALE_RTOL * np.abs(s_orc)
    if np.any(bad):
        i = np.flatnonzero(bad)[:8]
        raise ParityError(f"{what}: {int(bad.sum())} scales off by > 1e-6 relative, e.g. "
                          + ", ".join(f"[{k}] {s_gpu[k]!r} vs {s_orc[k]!r}" for k in i))
    rel = err / np.maximum(np.abs(s_orc), 1e-300)
    return {"max_scale_rel_err": float(rel.max()) if rel.size else 0.0}


BF16_MIDPOINT_RTOL = 2.0 ** -19
BF16_FLIP_FRACTION = 1e-3


def compare_bf16(g, o, v, what="bf16"):
    """bf16 outputs of an fp32 path whose pre-rounding error is below 2^-20
    relative: identical to the oracle's, except adjacent codes (same sign,
    one ulp) where the oracle's fp64 value v lies within 2^-19 relative of
    the midpoint of the two; such flips at most 0.1 % of the elements."""
    g = np.asarray(g, np.uint16).reshape(-1)
    o = np.asarray(o, np.uint16).reshape(-1)
    v = np.asarray(v, np.float64).reshape(-1)
    diff = np.flatnonzero(g != o)
    if diff.size == 0:
        return {"elements": g.size, "flips": 0}
    a, b, vv = g[diff].astype(np.int64), o[diff].astype(np.int64), v[diff]
    same_sign = (a & 0x8000) == (b & 0x8000)
    adjacent = same_sign & (np.abs((a & 0x7FFF) - (b & 0x7FFF)) == 1)
    va = exact.bf16_bits_to_f64(a.astype(np.uint16))
    vb = exact.bf16_bits_to_f64(b.astype(np.uint16))
    mid = (va + vb) / 2.0
    with np.errstate(invalid="ignore", divide="ignore"):
        rel = np.abs(vv - mid) / np.abs(mid)
    bad = ~adjacent | ~(rel <= BF16_MIDPOINT_RTOL)
    if np.any(bad):
        i = diff[np.flatnonzero(bad)[:8]]
        raise ParityError(f"{what}: {int(bad.sum())} values outside tolerance, e.g. "
                          + ", ".join(f"[{k}] gpu={g[k]:#06x} oracle={o[k]:#06x} v={v[k]!r}" for k in i))
    if diff.size > BF16_FLIP_FRACTION * g.size:
        raise ParityError(f"{what}: {diff.size} near-midpoint flips in {g.size} elements")
    return {"elements": g.size, "flips": int(diff.size), "max_rel": float(rel.max())}


_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def unpack_e2m1(q4):
    """[T, n/2] packed bytes -> [T, n] E2M1 codes (column 2i = low nibble)."""
    q4 = np.asarray(q4, np.uint8)
    out = np.empty(q4.shape[:-1] + (2 * q4.shape[-1],), np.uint8)
    out[..., 0::2] = q4 & 0xF
    out[..., 1::2] = q4 >> 4
    return out


def compare_e2m1(q4_gpu, q4_orc, v_orc, what="q4"):
    """The code rule for E2M1: identical codes, except codes adjacent in value
    (same sign) where the oracle's v lies within 1e-3 relative of their
    midpoint, at most 0.01 % of the elements; exact wherever |v| >= 6."""
    a = unpack_e2m1(q4_gpu).reshape(-1)
    b = unpack_e2m1(q4_orc).reshape(-1)
    v = np.asarray(v_orc, np.float64).reshape(-1)
    diff = np.flatnonzero(a != b)
    stats = {"elements": b.size, "flips": int(diff.size)}
    if diff.size == 0:
        return stats
    ca, cb, vv = a[diff], b[diff], v[diff]
    ma, mb = (ca & 7).astype(np.int32), (cb & 7).astype(np.int32)
    adjacent = ((ca & 8) == (cb & 8)) & (np.abs(ma - mb) == 1)
    mid = (_E2M1_MAG[ma] + _E2M1_MAG[mb]) / 2.0
    rel = np.where(adjacent, np.abs(np.abs(vv) - mid) / np.maximum(mid, 1e-300), np.inf)
    bad = ~adjacent | (rel > MIDPOINT_RTOL) | (np.abs(vv) >= 6.0)
    if np.any(bad):
        k = diff[np.flatnonzero(bad)[:8]]
        raise ParityError(f"{what}: {int(bad.sum())} codes outside tolerance, e.g. "
                          + ", ".join(f"[{j}] gpu={a[j]:#x} oracle={b[j]:#x} v={v[j]!r}" for j in k))
    if diff.size > FLIP_FRACTION * b.size:
        raise ParityError(f"{what}: {diff.size} near-midpoint flips in {b.size} elements")
    stats["max_flip_rel_dist"] = float(rel.max())
    return stats


def check_nvfp4(gpu, orc, rows=None):
    """gpu/orc: dicts with q4, sf (and residual_out, orc['v'])."""
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    compare_exact(sel(gpu["sf"]), orc["sf"], "block_scale")
    stats = compare_e2m1(sel(gpu["q4"]), orc["q4"], orc["v"])
    if orc.get("residual_out") is not None:
        compare_exact(sel(gpu["residual_out"]), orc["residual_out"], "residual_out")
    return stats


def compare_exact(a, b, what):
    a = np.asarray(a)
    b = np.asarray(b)
    if a.shape != b.shape or not np.array_equal(a, b):
        d = np.flatnonzero(a.reshape(-1) != b.reshape(-1)) if a.shape == b.shape else []
        raise ParityError(f"{what}: not bit-exact ({len(d)} differ, first {list(d[:5])})")


def compare_bf16_exact(a, b, what):
    """bf16 bit patterns equal, where a NaN matches any NaN (IEEE fixes no
    NaN payload: the GPU's conversion returns its canonical NaN)."""
    a = np.asarray(a, np.uint16)
    b = np.asarray(b, np.uint16)
    if a.shape != b.shape:
        raise ParityError(f"{what}: shape {a.shape} != {b.shape}")

    def nan(v):
        return ((v & 0x7F80) == 0x7F80) & ((v & 0x7F) != 0)
    diff = (a != b) & ~(nan(a) & nan(b))
    if np.any(diff):
        d = np.flatnonzero(diff.reshape(-1))
        raise ParityError(f"{what}: not bit-exact ({d.size} differ, first {list(d[:5])})")


def check_norm(gpu, orc, mode, rows=None):
    """gpu/orc: dicts with q, residual_out, scale (and orc['v']).  ``rows``
    restricts the GPU side to sampled rows (the oracle ran on those rows)."""
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    stats = compare_codes(sel(gpu["q"]), orc["q"], orc["v"])
    if orc.get("residual_out") is not None:
        compare_bf16_exact(sel(gpu["residual_out"]), orc["residual_out"], "residual_out")
    if mode != 0:
        stats.update(compare_scales(sel(gpu["scale"]), orc["scale"]))
    return stats


def check_silu(gpu, orc, mode, rows=None):
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    stats = compare_codes(sel(gpu["q"]), orc["q"], orc["v"])
    if mode != 0:
        stats.update(compare_scales(sel(gpu["scale"]), orc["scale"]))
    return stats


def oracle_mla(q_c, q_weight, kv_c, kv_weight, eps_q, eps_kv, q_fp8):
    """The oracle's MLA dual norm over row blocks run in threads."""
    T = q_c.shape[0]
    parts = [None] * T
    blocks = _blocks(T, _threads())

    def work(i):
        r0, r1 = blocks[i]
        parts[i] = oracle.mla_dual_rms_norm(q_c[r0:r1], q_weight, kv_c[r0:r1], kv_weight,
                                            eps_q, eps_kv, q_fp8=q_fp8)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(len(blocks))))
    parts = [p for p in parts if p is not None]
    if not parts:
        return None
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}


def oracle_pad(x, residual, weight, eps, padded):
    """The oracle's padded norm over row blocks run in threads."""
    T, H = x.shape
    out = {"out": np.empty((T, padded), np.uint16),
           "residual_out": None if residual is None else np.empty((T, H), np.uint16)}
    blocks = _blocks(T, _threads())

    def work(b):
        r0, r1 = b
        o = oracle.fused_add_rms_norm_pad(x[r0:r1], None if residual is None else residual[r0:r1],
                                          weight, eps, padded, want_y=False)
        out["out"][r0:r1] = o["out"]
        if residual is not None:
            out["residual_out"][r0:r1] = o["residual_out"]

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, blocks))
    return out


def check_pad(gpu, orc):
    """The padded bf16 rows (tail included) and residual_out, bit-exact."""
    compare_exact(gpu["out"], orc["out"], "out")
    if orc["residual_out"] is not None:
        compare_exact(gpu["residual_out"], orc["residual_out"], "residual_out")


def oracle_qk(d, hq, hkv, head_dim, eps, neox):
    """The oracle's QK norm + RoPE over token blocks run in threads: (qkv
    after, the fp64 pre-rounding values of the Q and K heads)."""
    qkv = d["qkv"]
    T = qkv.shape[0]
    out = np.empty_like(qkv)
    o = np.empty((T, (hq + hkv) * head_dim), np.float64)
    blocks = _blocks(T, _threads())

    def work(b):
        r0, r1 = b
        r = oracle.qk_norm_rope(qkv[r0:r1], d["q_weight"], d["k_weight"], d["cos_sin_cache"],
                                d["positions"][r0:r1], hq, hkv, head_dim, eps, neox)
        out[r0:r1] = r["qkv"]
        o[r0:r1] = r["o"]

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, blocks))
    return out, o


def check_qk(g, orc, qkv_in, hq, hkv, head_dim):
    """Q and K heads under the bf16 tolerance; V columns untouched."""
    out, o = orc
    n = (hq + hkv) * head_dim
    stats = compare_bf16(g[:, :n], out[:, :n], o, "qk heads")
    compare_exact(g[:, n:], qkv_in[:, n:], "v heads")
    return stats


def check_mla(gpu, orc, q_fp8):
    """kv (and a bf16 q) bit-exact; an fp8 q under the code rule, its
    per-token scales within 1e-6."""
    compare_exact(gpu["kv"], orc["kv"], "kv_normed")
    if not q_fp8:
        compare_exact(gpu["q"], orc["q"], "q_normed")
        return {}
    stats = compare_codes(gpu["q_fp8"], orc["q_fp8"], orc["q_v"], "q_fp8")
    stats.update(compare_scales(gpu["q_scale"], orc["q_scale"], "q_scale"))
    return stats


# --------------------------------------------------------------- GPU side

GUARD = 256  # sentinel bytes before and after every GPU output


def _guarded(torch, nbytes, device):
    buf = torch.full((nbytes + 2 * GUARD,), 0xAA, dtype=torch.uint8, device=device)
    return buf, buf[GUARD:GUARD + nbytes]


def _check_guards(buf, nbytes, what):
    host = buf.cpu().numpy()
    if not (np.all(host[:GUARD] == 0xAA) and np.all(host[GUARD + nbytes:] == 0xAA)):
        raise ParityError(f"{what}: write outside the output buffer")


UE8M0, COL_MAJOR = 0x100, 0x200


def _scale_buffer(torch, mode, T, n, group_size, scale, device):
    """The guarded scale tensor for a mode (flags included): [1] static
    (filled), [T] per-token, [T, n/G] per-group, or [n/G, T4] column-major,
    whose padding columns keep the 0xAA guard pattern."""
    base = mode & 0xFF
    if base == 0:
        sbuf, sraw = _guarded(torch, 4, device)
        s = sraw.view(torch.float32)
        s.fill_(float(np.float32(scale)))
        return sbuf, s
    if base == 1:
        ns = T
    elif mode & COL_MAJOR:
        ns = (n // group_size) * ((T + 3) // 4 * 4)
    else:
        ns = T * (n // group_size)
    sbuf, sraw = _guarded(torch, 4 * ns, device)
    return sbuf, sraw.view(torch.float32)


def _scales_row_major(s, mode, T, n, group_size):
    """Scales as the oracle's row-major [T, n/G] (or [T] / [1]); a
    column-major buffer must hold the guard pattern in its padding columns."""
    base = mode & 0xFF
    a = s.cpu().numpy()
    if base == 0:
        return a
    if base == 1:
        return a.reshape(T)
    g = n // group_size
    if mode & COL_MAJOR:
        t4 = (T + 3) // 4 * 4
        a = a.reshape(g, t4)
        pad = a[:, T:].view(np.uint32)
        if not np.all(pad == 0xAAAAAAAA):
            raise ParityError("scale: column-major padding columns were written")
        return np.ascontiguousarray(a[:, :T].T)
    return a.reshape(T, g)


def gpu_norm(x, residual, weight, eps, mode, group_size=128, scale=None, inplace=True,
             device="cuda"):
    """Runs the CUDA path through the C ABI on numpy bf16-bit inputs; outputs
    sit between guard bands pre-filled with 0xAA, checked afterwards."""
    import torch
    import norm_activation_fp8_gb300 as vg
    T, H = x.shape
    xt = torch.from_numpy(x.view(np.int16)).to(device)
    wt = torch.from_numpy(np.ascontiguousarray(weight).view(np.int16)).to(device)
    qbuf, q = _guarded(torch, T * H, device)
    rt = rbuf = r_out = None
    if residual is not None:
        if inplace:
            rbuf, rraw = _guarded(torch, T * H * 2, device)
            rt = rraw.view(torch.int16).view(T, H)
            rt.copy_(torch.from_numpy(residual.view(np.int16)))
            r_out = rt
        else:
            rt = torch.from_numpy(residual.view(np.int16)).to(device)
            rbuf, rraw = _guarded(torch, T * H * 2, device)
            r_out = rraw.view(torch.int16).view(T, H)
    sbuf, s = _scale_buffer(torch, mode, T, H, group_size, scale, device)
    vg.vg_fused_add_rms_norm_fp8(q.view(T, H), r_out, s, xt, rt, wt, eps, mode, group_size)
    torch.cuda.synchronize()
    _check_guards(qbuf, T * H, "q")
    _check_guards(sbuf, s.numel() * 4, "scale")
    out = {"q": q.view(T, H).cpu().numpy(), "scale": _scales_row_major(s, mode, T, H, group_size)}
    if residual is not None:
        _check_guards(rbuf, T * H * 2, "residual_out")
        out["residual_out"] = r_out.cpu().numpy().view(np.uint16)
    else:
        out["residual_out"] = None
    return out


def gpu_silu(gate_up, mode, group_size=128, scale=None, device="cuda"):
    import torch
    import norm_activation_fp8_gb300 as vg
    T, two_i = gate_up.shape
    I = two_i // 2
    gt = torch.from_numpy(gate_up.view(np.int16)).to(device)
    qbuf, q = _guarded(torch, T * I, device)
    sbuf, s = _scale_buffer(torch, mode, T, I, group_size, scale, device)
    vg.vg_silu_mul_fp8(q.view(T, I), s, gt, mode, group_size)
    torch.cuda.synchronize()
    _check_guards(qbuf, T * I, "q")
    _check_guards(sbuf, s.numel() * 4, "scale")
    return {"q": q.view(T, I).cpu().numpy(), "scale": _scales_row_major(s, mode, T, I, group_size)}


def gpu_mla(q_c, q_weight, kv_c, kv_weight, eps_q, eps_kv, q_fp8, rope=64, q_pad=None,
            kv_pad=None, device="cuda"):
    """The CUDA MLA dual norm on numpy bf16-bit inputs.  By default q_c and
    kv_c are column slices of one projected [T, q_dim + kv_dim + rope]
    device tensor, as in the model; with q_pad / kv_pad each side is its own
    tensor whose rows are padded by that many elements (another stride).
    Outputs sit between 0xAA guard bands, checked afterwards."""
    import torch
    import norm_activation_fp8_gb300 as vg
    T, q_dim = q_c.shape
    kv_dim = kv_c.shape[1]
    if q_pad is None and kv_pad is None:
        proj = np.zeros((T, q_dim + kv_dim + rope), np.uint16)
        proj[:, :q_dim] = q_c
        proj[:, q_dim:q_dim + kv_dim] = kv_c
        pt = torch.from_numpy(proj.view(np.int16)).to(device)
        qt, kt = pt[:, :q_dim], pt[:, q_dim:q_dim + kv_dim]
    else:
        def padded(a, pad):
            buf = np.full((T, a.shape[1] + (pad or 0)), 0x7FC0, np.uint16)  # NaN padding
            buf[:, :a.shape[1]] = a
            return torch.from_numpy(buf.view(np.int16)).to(device)[:, :a.shape[1]]
        qt, kt = padded(q_c, q_pad), padded(kv_c, kv_pad)
    qw = torch.from_numpy(np.ascontiguousarray(q_weight).view(np.int16)).to(device)
    kw = torch.from_numpy(np.ascontiguousarray(kv_weight).view(np.int16)).to(device)
    kbuf, kraw = _guarded(torch, T * kv_dim * 2, device)
    kv_out = kraw.view(torch.int16).view(T, kv_dim)
    out = {}
    if q_fp8:
        qbuf, qraw = _guarded(torch, T * q_dim, device)
        sbuf, sraw = _guarded(torch, 4 * T, device)
        vg.vg_fused_mla_dual_rms_norm_per_token_quant(qraw.view(T, q_dim), sraw.view(torch.float32),
                                                      kv_out, qt, qw, kt, kw, eps_q, eps_kv)
        torch.cuda.synchronize()
        _check_guards(qbuf, T * q_dim, "q_fp8")
        _check_guards(sbuf, 4 * T, "q_scale")
        out["q_fp8"] = qraw.view(T, q_dim).cpu().numpy()
        out["q_scale"] = sraw.view(torch.float32).cpu().numpy()
    else:
        qbuf, qraw = _guarded(torch, T * q_dim * 2, device)
        q_out = qraw.view(torch.int16).view(T, q_dim)
        vg.vg_fused_mla_dual_rms_norm(q_out, kv_out, qt, qw, kt, kw, eps_q, eps_kv)
        torch.cuda.synchronize()
        _check_guards(qbuf, T * q_dim * 2, "q_normed")
        out["q"] = q_out.cpu().numpy().view(np.uint16)
    _check_guards(kbuf, T * kv_dim * 2, "kv_normed")
    out["kv"] = kv_out.cpu().numpy().view(np.uint16)
    return out


def gpu_pad(x, residual, weight, eps, padded, inplace=True, device="cuda"):
    """The CUDA padded norm on numpy bf16-bit inputs; outputs between 0xAA
    guard bands (the padded tail starts as 0xAA too, so it must be written)."""
    import torch
    import norm_activation_fp8_gb300 as vg
    T, H = x.shape
    xt = torch.from_numpy(x.view(np.int16)).to(device)
    wt = torch.from_numpy(np.ascontiguousarray(weight).view(np.int16)).to(device)
    obuf, oraw = _guarded(torch, T * padded * 2, device)
    out = oraw.view(torch.int16).view(T, padded)
    rt = rbuf = r_out = None
    if residual is not None:
        rbuf, rraw = _guarded(torch, T * H * 2, device)
        if inplace:
            rt = rraw.view(torch.int16).view(T, H)
            rt.copy_(torch.from_numpy(residual.view(np.int16)))
            r_out = rt
        else:
            rt = torch.from_numpy(residual.view(np.int16)).to(device)
            r_out = rraw.view(torch.int16).view(T, H)
    vg.vg_fused_add_rms_norm_pad(out, r_out, xt, rt, wt, eps)
    torch.cuda.synchronize()
    _check_guards(obuf, T * padded * 2, "out")
    res = {"out": out.cpu().numpy().view(np.uint16), "residual_out": None}
    if residual is not None:
        _check_guards(rbuf, T * H * 2, "residual_out")
        res["residual_out"] = r_out.cpu().numpy().view(np.uint16)
    return res


def gpu_qk(d, hq, hkv, head_dim, eps, neox, device="cuda"):
    """The CUDA QK norm + RoPE on numpy inputs; qkv (updated in place) sits
    between 0xAA guard bands, checked afterwards.  Returns qkv after."""
    import torch
    import norm_activation_fp8_gb300 as vg
    qkv = d["qkv"]
    T, row = qkv.shape
    qbuf, qraw = _guarded(torch, T * row * 2, device)
    qt = qraw.view(torch.int16).view(T, row)
    qt.copy_(torch.from_numpy(qkv.view(np.int16)))
    qw = torch.from_numpy(d["q_weight"].view(np.int16)).to(device)
    kw = torch.from_numpy(d["k_weight"].view(np.int16)).to(device)
    cache = torch.from_numpy(d["cos_sin_cache"]).to(device)
    pos = torch.from_numpy(d["positions"]).to(device)
    vg.vg_fused_qk_norm_rope(qt, qw, kw, cache, pos, hq, hkv, head_dim, eps, neox)
    torch.cuda.synchronize()
    _check_guards(qbuf, T * row * 2, "qkv")
    return qt.cpu().numpy().view(np.uint16)


def _gs_tensor(torch, gs, device):
    return torch.tensor([float(np.float32(gs))], dtype=torch.float32, device=device)


def gpu_nvfp4_norm(x, residual, weight, eps, gs, inplace=True, device="cuda"):
    """The NVFP4 norm through the C ABI, outputs between guard bands."""
    import torch
    import norm_activation_fp8_gb300 as vg
    T, H = x.shape
    xt = torch.from_numpy(x.view(np.int16)).to(device)
    wt = torch.from_numpy(np.ascontiguousarray(weight).view(np.int16)).to(device)
    qbuf, q4 = _guarded(torch, T * H // 2, device)
    fbuf, sf = _guarded(torch, T * H // 16, device)
    rt = rbuf = r_out = None
    if residual is not None:
        rbuf, rraw = _guarded(torch, T * H * 2, device)
        r_out = rraw.view(torch.int16).view(T, H)
        if inplace:
            r_out.copy_(torch.from_numpy(residual.view(np.int16)))
            rt = r_out
        else:
            rt = torch.from_numpy(residual.view(np.int16)).to(device)
    vg.vg_fused_add_rms_norm_nvfp4(q4.view(T, H // 2), sf.view(T, H // 16), r_out, xt, rt, wt,
                                   _gs_tensor(torch, gs, device), eps)
    torch.cuda.synchronize()
    _check_guards(qbuf, T * H // 2, "q4")
    _check_guards(fbuf, T * H // 16, "block_scale")
    out = {"q4": q4.view(T, H // 2).cpu().numpy(), "sf": sf.view(T, H // 16).cpu().numpy(),
           "residual_out": None}
    if residual is not None:
        _check_guards(rbuf, T * H * 2, "residual_out")
        out["residual_out"] = r_out.cpu().numpy().view(np.uint16)
    return out


def gpu_nvfp4_silu(gate_up, gs, device="cuda"):
    import torch
    import norm_activation_fp8_gb300 as vg
    T, two_i = gate_up.shape
    I = two_i // 2
    gt = torch.from_numpy(gate_up.view(np.int16)).to(device)
    qbuf, q4 = _guarded(torch, T * I // 2, device)
    fbuf, sf = _guarded(torch, T * I // 16, device)
    vg.vg_silu_mul_nvfp4(q4.view(T, I // 2), sf.view(T, I // 16), gt, _gs_tensor(torch, gs, device))
    torch.cuda.synchronize()
    _check_guards(qbuf, T * I // 2, "q4")
    _check_guards(fbuf, T * I // 16, "block_scale")
    return {"q4": q4.view(T, I // 2).cpu().numpy(), "sf": sf.view(T, I // 16).cpu().numpy()}
