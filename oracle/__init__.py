"""Plain fp64 CPU oracle for fused residual-add + RMSNorm -> FP8 and
SiLU-and-mul -> FP8 (numpy front end over ``oracle.c``).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product
package never imports it and shares no code with it.

What each function computes is documented in ``oracle.c`` with the passages
it follows ("Fusion torch.compile passes", sections "RMSNorm + Quantization
(fuse_norm_quant)", "SiLU+Mul + Quantization (fuse_act_quant)" (FP8, and FP4 as
NVIDIA's NVFP4), "MLA Dual
RMSNorm (fuse_mla_dual_rms_norm)", "RMSNorm + Padding (fuse_act_padding)" and
"QK Norm + RoPE (enable_qk_norm_rope_fusion)"; OCP OFP8 for the E4M3 format).

Parity status per function (each pin lives in ``tests/test_oracle_pins.py``):
  bf16 / e4m3 codecs ........ pinned (spec points, exhaustive round trips,
                              brute-force nearest value)
  fused_add_rms_norm_fp8 .... pinned (closed forms, invariants, library
                              bf16 add, exact-arithmetic brute force)
  silu_mul_fp8 .............. pinned (closed forms, library sigmoid,
                              exact-arithmetic brute force)
  rms_norm_bf16 ............. pinned (closed forms, invariants,
                              exact-arithmetic brute force)
  mla_dual_rms_norm ......... the two pinned norms above, side by side
  fused_add_rms_norm_pad .... pinned (zero tail, bf16 rms_norm on the
                              stored residual, library bf16 add)
  per-group UE8M0 / column-major scales ... pinned (powers of two that
                              bracket amax/448, exact rationals, the
                              transposed layout of the row-major scales)
  e2m1 codec, NVFP4 quant ... pinned (all 16 codes, exhaustive nearest
                              value, block scales and codes against exact
                              rationals, packing)
  qk_norm_rope .............. pinned (identity and quarter-turn rotations
                              against the pinned bf16 rms_norm, V untouched,
                              neox/gptj by permutation, exact rationals)
  NaN / Inf inputs, FP8 norm and SiLU ... pinned (the IEEE consequences:
                              NaN rows, an infinite residual, silu(-inf),
                              saturation under a static scale, against
                              values fixed by that reading)
  NaN / Inf in the NVFP4, padded, MLA and QK paths ... parity unpinned
                              (no workload contains them)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

STATIC, PER_TOKEN, PER_GROUP = 0, 1, 2
UE8M0, COL_MAJOR = 0x100, 0x200  # per-group options, or-ed into the mode

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()


def compile_source(src: str, out: str) -> str:
    """Compile one C source file into a shared library with the oracle's flags."""
    tmp = out + f".tmp{os.getpid()}"
    cc = os.environ.get("CC", "gcc")
    subprocess.check_call([cc, *_CFLAGS, "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, no GPU needed)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle's shared library."""
    lib = ctypes.CDLL(path or build())
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.orc_fused_add_rms_norm_fp8.argtypes = [P, P, P, P, P, P, P, i64, i64,
                                               ctypes.c_float, ctypes.c_int, i64]
    lib.orc_fused_add_rms_norm_fp8.restype = ctypes.c_int
    lib.orc_silu_mul_fp8.argtypes = [P, P, P, P, i64, i64, ctypes.c_int, i64]
    lib.orc_silu_mul_fp8.restype = ctypes.c_int
    lib.orc_rms_norm_bf16.argtypes = [P, P, P, P, i64, i64, ctypes.c_float]
    lib.orc_rms_norm_bf16.restype = ctypes.c_int
    lib.orc_fused_add_rms_norm_pad.argtypes = [P, P, P, P, P, P, i64, i64, i64, ctypes.c_float]
    lib.orc_fused_add_rms_norm_pad.restype = ctypes.c_int
    lib.orc_qk_norm_rope.argtypes = [P, P, P, P, P, P, i64, i64, i64, i64, i64, ctypes.c_float,
                                     ctypes.c_int]
    lib.orc_qk_norm_rope.restype = ctypes.c_int
    lib.orc_fused_add_rms_norm_nvfp4.argtypes = [P, P, P, P, P, P, P, ctypes.c_float, i64, i64,
                                                 ctypes.c_float]
    lib.orc_fused_add_rms_norm_nvfp4.restype = ctypes.c_int
    lib.orc_silu_mul_nvfp4.argtypes = [P, P, P, P, ctypes.c_float, i64, i64]
    lib.orc_silu_mul_nvfp4.restype = ctypes.c_int
    for name in ("orc_bf16_decode_n", "orc_bf16_encode_n",
                 "orc_e4m3_decode_n", "orc_e4m3_encode_n",
                 "orc_e2m1_decode_n", "orc_e2m1_encode_n"):
        getattr(lib, name).argtypes = [P, P, i64]
        getattr(lib, name).restype = None
    lib.orc_amax_floor.argtypes = []
    lib.orc_amax_floor.restype = ctypes.c_double
    return lib


class Oracle:
    """The oracle's functions bound to one loaded copy of its library (the
    tests also load deliberately broken copies to show the pins catch them)."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib

    # -------------------------------------------------------------- codecs
    def bf16_decode(self, bits) -> np.ndarray:
        b = _u16(bits)
        out = np.empty(b.shape, np.float64)
        self.lib.orc_bf16_decode_n(_ptr(out), _ptr(b), b.size)
        return out

    def bf16_encode(self, values) -> np.ndarray:
        v = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(v.shape, np.uint16)
        self.lib.orc_bf16_encode_n(_ptr(out), _ptr(v), v.size)
        return out

    def e4m3_decode(self, codes) -> np.ndarray:
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(c.shape, np.float64)
        self.lib.orc_e4m3_decode_n(_ptr(out), _ptr(c), c.size)
        return out

    def e4m3_encode(self, values) -> np.ndarray:
        v = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(v.shape, np.uint8)
        self.lib.orc_e4m3_encode_n(_ptr(out), _ptr(v), v.size)
        return out

    def e2m1_decode(self, codes) -> np.ndarray:
        c = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(c.shape, np.float64)
        self.lib.orc_e2m1_decode_n(_ptr(out), _ptr(c), c.size)
        return out

    def e2m1_encode(self, values) -> np.ndarray:
        v = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(v.shape, np.uint8)
        self.lib.orc_e2m1_encode_n(_ptr(out), _ptr(v), v.size)
        return out

    def amax_floor(self) -> float:
        """A_MIN, the floor on a dynamic amax (the fp32 number nearest 1e-10)."""
        return float(self.lib.orc_amax_floor())

    # ----------------------------------------------------------------- ops
    def fused_add_rms_norm_fp8(self, x, residual, weight, eps: float, mode: int,
                               group_size: int = 128, scale=None, want_v: bool = True):
        """fused_add_rms_norm(x, residual) -> quant_fp8, or with ``residual``
        None the plain rms_norm(x) -> quant_fp8 variant.

        x, residual: uint16 bf16 bits [T, H]; weight: uint16 [H].
        Returns dict(q uint8 [T,H], residual_out uint16 [T,H] or None,
        scale float32 ([1] static / [T] / [T,H/G]), v float64 [T,H] = y/s)."""
        x = _u16(x)
        T, H = x.shape
        w = _u16(weight).reshape(H)
        res = None if residual is None else _u16(residual).reshape(T, H)
        q = np.empty((T, H), np.uint8)
        r_out = None if res is None else np.empty((T, H), np.uint16)
        s = _scale_buffer(mode, T, H, group_size, scale)
        v = np.empty((T, H), np.float64) if want_v else None
        rc = self.lib.orc_fused_add_rms_norm_fp8(
            _ptr(q), _ptr(r_out), _ptr(s), _ptr(v), _ptr(x), _ptr(res), _ptr(w),
            T, H, ctypes.c_float(eps), mode, group_size)
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (rc={rc})")
        return {"q": q, "residual_out": r_out, "scale": s, "v": v}

    def silu_mul_fp8(self, gate_up, mode: int, group_size: int = 128, scale=None,
                     want_v: bool = True):
        """silu_and_mul(gate_up) -> quant_fp8.

        gate_up: uint16 bf16 bits [T, 2I], gate = columns [0, I), up = [I, 2I).
        Returns dict(q uint8 [T,I], scale, v float64 [T,I])."""
        gu = _u16(gate_up)
        T, two_i = gu.shape
        if two_i % 2:
            raise ValueError("gate_up must have an even number of columns")
        I = two_i // 2
        q = np.empty((T, I), np.uint8)
        s = _scale_buffer(mode, T, I, group_size, scale)
        v = np.empty((T, I), np.float64) if want_v else None
        rc = self.lib.orc_silu_mul_fp8(_ptr(q), _ptr(s), _ptr(v), _ptr(gu), T, I, mode,
                                       group_size)
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (rc={rc})")
        return {"q": q, "scale": s, "v": v}


    def fused_add_rms_norm_nvfp4(self, x, residual, weight, eps: float, global_scale: float,
                                 want_v: bool = True):
        """fused_add_rms_norm(x, residual) -> NVFP4 (residual None: the plain
        variant).  Returns dict(q4 uint8 [T,H/2] (column 2i in the low
        nibble), sf uint8 [T,H/16] E4M3 block codes, residual_out, v)."""
        x = _u16(x)
        T, H = x.shape
        w = _u16(weight).reshape(H)
        res = None if residual is None else _u16(residual).reshape(T, H)
        q4 = np.empty((T, H // 2), np.uint8)
        sf = np.empty((T, H // 16), np.uint8)
        r_out = None if res is None else np.empty((T, H), np.uint16)
        v = np.empty((T, H), np.float64) if want_v else None
        rc = self.lib.orc_fused_add_rms_norm_nvfp4(_ptr(q4), _ptr(sf), _ptr(r_out), _ptr(v), _ptr(x),
                                                   _ptr(res), _ptr(w), ctypes.c_float(global_scale),
                                                   T, H, ctypes.c_float(eps))
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (rc={rc})")
        return {"q4": q4, "sf": sf, "residual_out": r_out, "v": v}

    def silu_mul_nvfp4(self, gate_up, global_scale: float, want_v: bool = True):
        """silu_and_mul(gate_up) -> NVFP4.  Returns dict(q4 [T,I/2], sf [T,I/16], v)."""
        gu = _u16(gate_up)
        T, two_i = gu.shape
        I = two_i // 2
        q4 = np.empty((T, I // 2), np.uint8)
        sf = np.empty((T, I // 16), np.uint8)
        v = np.empty((T, I), np.float64) if want_v else None
        rc = self.lib.orc_silu_mul_nvfp4(_ptr(q4), _ptr(sf), _ptr(v), _ptr(gu),
                                         ctypes.c_float(global_scale), T, I)
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (rc={rc})")
        return {"q4": q4, "sf": sf, "v": v}

    def rms_norm_bf16(self, x, weight, eps: float, want_y: bool = True):
        """rms_norm(x, weight, eps) with the output rounded once to bf16.

        x: uint16 bf16 bits [T, H]; weight: uint16 [H].
        Returns dict(out uint16 [T,H], y float64 [T,H] before rounding)."""
        x = _u16(x)
        T, H = x.shape
        w = _u16(weight).reshape(H)
        out = np.empty((T, H), np.uint16)
        y = np.empty((T, H), np.float64) if want_y else None
        rc = self.lib.orc_rms_norm_bf16(_ptr(out), _ptr(y), _ptr(x), _ptr(w), T, H,
                                        ctypes.c_float(eps))
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (rc={rc})")
        return {"out": out, "y": y}

    def fused_add_rms_norm_pad(self, x, residual, weight, eps: float, padded: int,
                               want_y: bool = True):
        """fused_add_rms_norm(x, residual) with a bf16 output padded to
        ``padded`` columns (zeros after the first H), or with ``residual``
        None the plain rms_norm(x) variant.

        Returns dict(out uint16 [T,padded], residual_out uint16 [T,H] or None,
        y float64 [T,H] before rounding)."""
        x = _u16(x)
        T, H = x.shape
        w = _u16(weight).reshape(H)
        res = None if residual is None else _u16(residual).reshape(T, H)
        out = np.empty((T, padded), np.uint16)
        r_out = None if res is None else np.empty((T, H), np.uint16)
        y = np.empty((T, H), np.float64) if want_y else None
        rc = self.lib.orc_fused_add_rms_norm_pad(_ptr(out), _ptr(r_out), _ptr(y), _ptr(x),
                                                 _ptr(res), _ptr(w), T, H, padded,
                                                 ctypes.c_float(eps))
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (rc={rc})")
        return {"out": out, "residual_out": r_out, "y": y}

    def qk_norm_rope(self, qkv, q_weight, k_weight, cos_sin_cache, positions, num_q_heads: int,
                     num_kv_heads: int, head_dim: int, eps: float, is_neox: bool = True,
                     want_o: bool = True):
        """fused_qk_norm_rope on a copy of qkv (uint16 bf16 bits
        [T, (Hq + 2 Hkv) * D]); cos_sin_cache float32 [max_pos, D];
        positions int64 [T].  Returns dict(qkv uint16 (V columns unchanged),
        o float64 [T, (Hq + Hkv) * D] before rounding)."""
        out = _u16(qkv).copy()
        T = out.shape[0]
        cache = np.ascontiguousarray(cos_sin_cache, dtype=np.float32)
        pos = np.ascontiguousarray(positions, dtype=np.int64).reshape(T)
        o = np.empty((T, (num_q_heads + num_kv_heads) * head_dim), np.float64) if want_o else None
        rc = self.lib.orc_qk_norm_rope(_ptr(out), _ptr(o), _ptr(_u16(q_weight)), _ptr(_u16(k_weight)),
                                       _ptr(cache), _ptr(pos), T, num_q_heads, num_kv_heads,
                                       head_dim, cache.shape[0], ctypes.c_float(eps),
                                       1 if is_neox else 0)
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (rc={rc})")
        return {"qkv": out, "o": o}

    def mla_dual_rms_norm(self, q_c, q_weight, kv_c, kv_weight, eps_q: float,
                          eps_kv: float, q_fp8: bool = False, want_v: bool = True):
        """fused_mla_dual_rms_norm: the two norms of the unfused MLA graph,
        side by side.  q_normed = rms_norm(q_c, q_weight, eps_q) and
        kv_normed = rms_norm(kv_c, kv_weight, eps_kv), both bf16.  With
        ``q_fp8`` (fused_mla_dual_rms_norm_per_token_quant) the q side is the
        plain rms_norm -> dynamic per-token FP8 of fuse_norm_quant instead.

        Returns dict(kv uint16 [T,kv_dim], kv_y, and either q uint16 [T,q_dim]
        with q_y, or q_fp8 uint8 [T,q_dim], q_scale float32 [T], q_v)."""
        kv = self.rms_norm_bf16(kv_c, kv_weight, eps_kv, want_y=want_v)
        out = {"kv": kv["out"], "kv_y": kv["y"]}
        if q_fp8:
            q = self.fused_add_rms_norm_fp8(q_c, None, q_weight, eps_q, PER_TOKEN, want_v=want_v)
            out.update(q_fp8=q["q"], q_scale=q["scale"], q_v=q["v"])
        else:
            q = self.rms_norm_bf16(q_c, q_weight, eps_q, want_y=want_v)
            out.update(q=q["out"], q_y=q["y"])
        return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


def _scale_buffer(mode: int, rows: int, n: int, group_size: int, scale):
    if mode & COL_MAJOR and mode & 0xFF == PER_GROUP:
        if group_size <= 0 or n % group_size:
            raise ValueError("per-group mode needs a group size dividing the row")
        # [n/G, T4]; the padding columns keep this sentinel (never written)
        return np.full((n // group_size, (rows + 3) // 4 * 4), -1.0, np.float32)
    mode &= 0xFF
    if mode == STATIC:
        if scale is None:
            raise ValueError("static mode needs the fp32 scale")
        return np.array([np.asarray(scale, np.float32).reshape(-1)[0]], np.float32)
    if mode == PER_TOKEN:
        return np.zeros((rows,), np.float32)
    if mode == PER_GROUP:
        if group_size <= 0 or n % group_size:
            raise ValueError("per-group mode needs a group size dividing the row")
        return np.zeros((rows, n // group_size), np.float32)
    raise ValueError(f"bad scale mode {mode}")


def default() -> Oracle:
    """The oracle built from ``oracle.c`` as committed."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(load_library())
    return _default


_default = None


def bf16_decode(bits):
    return default().bf16_decode(bits)


def bf16_encode(values):
    return default().bf16_encode(values)


def e4m3_decode(codes):
    return default().e4m3_decode(codes)


def e4m3_encode(values):
    return default().e4m3_encode(values)


def amax_floor():
    return default().amax_floor()


def fused_add_rms_norm_fp8(*args, **kwargs):
    return default().fused_add_rms_norm_fp8(*args, **kwargs)


def silu_mul_fp8(*args, **kwargs):
    return default().silu_mul_fp8(*args, **kwargs)


def rms_norm_bf16(*args, **kwargs):
    return default().rms_norm_bf16(*args, **kwargs)


def mla_dual_rms_norm(*args, **kwargs):
    return default().mla_dual_rms_norm(*args, **kwargs)


def fused_add_rms_norm_pad(*args, **kwargs):
    return default().fused_add_rms_norm_pad(*args, **kwargs)


def qk_norm_rope(*args, **kwargs):
    return default().qk_norm_rope(*args, **kwargs)


def fused_add_rms_norm_nvfp4(*args, **kwargs):
    return default().fused_add_rms_norm_nvfp4(*args, **kwargs)


def silu_mul_nvfp4(*args, **kwargs):
    return default().silu_mul_nvfp4(*args, **kwargs)


def e2m1_decode(codes):
    return default().e2m1_decode(codes)


def e2m1_encode(values):
    return default().e2m1_encode(values)
