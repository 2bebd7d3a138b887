"""Fused residual-add + RMSNorm -> FP8 and SiLU-and-mul -> FP8 on GB300.

Thin Python binding over the C ABI of ``libvg_fused.so`` (declared in
``include/vg_fused.h``).  Every step of both ops runs in the library's CUDA
kernels; this module only marshals arguments: it checks dtypes, devices and
contiguity of torch tensors, passes their device pointers and the current
CUDA stream, and turns a non-zero status into ``VgError``.  There is no CPU
fallback: if the library has not been built, every call raises.

Entry points (same names and argument order as the C ABI):
  vg_fused_add_rms_norm_fp8(q, residual_out, scale, x, residual, weight,
                            eps, mode, group_size=128, stream=None)
  vg_silu_mul_fp8(q, scale, gate_up, mode, group_size=128, stream=None)
  vg_fused_add_rms_norm_pad(out, residual_out, x, residual, weight, eps, stream=None)
  vg_fused_qk_norm_rope(qkv, q_weight, k_weight, cos_sin_cache, positions,
                        num_q_heads, num_kv_heads, head_dim, eps, is_neox=True, stream=None)
  vg_fused_mla_dual_rms_norm(q_out, kv_out, q_c, q_weight, kv_c, kv_weight,
                             eps_q, eps_kv, stream=None)
  vg_fused_mla_dual_rms_norm_per_token_quant(q_fp8, q_scale, kv_out, q_c,
                             q_weight, kv_c, kv_weight, eps_q, eps_kv, stream=None)
  (the MLA inputs may be column-slice views: their row stride is passed on)
  vg_fused_add_rms_norm_nvfp4(q4, block_scale, residual_out, x, residual, weight,
                              global_scale, eps, stream=None)
  vg_silu_mul_nvfp4(q4, block_scale, gate_up, global_scale, stream=None)
Convenience wrappers that allocate the outputs with torch:
  fused_add_rms_norm_fp8(x, residual, weight, eps, mode, ...)
  silu_mul_fp8(gate_up, mode, ...)
  fused_add_rms_norm_pad(x, residual, weight, eps, padded_hidden, ...)
  mla_dual_rms_norm(q_c, q_weight, kv_c, kv_weight, eps_q, eps_kv, q_fp8=False)
  fused_add_rms_norm_nvfp4(x, residual, weight, eps, global_scale, ...)
  silu_mul_nvfp4(gate_up, global_scale, ...)
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

STATIC, PER_TOKEN, PER_GROUP = 0, 1, 2
UE8M0, COLUMN_MAJOR = 0x100, 0x200  # per-group options, or-ed into the mode
MAX_ROW = 32768

STATUS_NAMES = {
    0: "VG_OK", 1: "VG_ERR_NULL_PTR", 2: "VG_ERR_BAD_SHAPE", 3: "VG_ERR_MISALIGNED",
    4: "VG_ERR_BAD_MODE", 5: "VG_ERR_BAD_GROUP", 6: "VG_ERR_UNSUPPORTED_DEVICE", 7: "VG_ERR_CUDA",
}

EXPORTED_SYMBOLS = ("vg_fused_add_rms_norm_fp8", "vg_silu_mul_fp8", "vg_fused_add_rms_norm_pad",
                    "vg_fused_mla_dual_rms_norm", "vg_fused_qk_norm_rope",
                    "vg_fused_mla_dual_rms_norm_per_token_quant", "vg_fused_add_rms_norm_nvfp4",
                    "vg_silu_mul_nvfp4", "vg_device_status",
                    "vg_status_string", "vg_abi_version")
DEVICE_WAIT_TIMEOUT = 1
DEVICE_BAD_POSITION = 2
DEVICE_OUT_OF_BOUNDS = 4  # debug builds (VG_DEBUG_CHECKS) only

_lock = threading.Lock()
_lib = None


class VgError(RuntimeError):
    """A non-zero vg_status returned by the library."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (built by ``build.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or os.environ.get("VG_FUSED_LIB", LIB_PATH)
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library {p} is missing: build it with "
                "`python -m norm_activation_fp8_gb300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(p)
        P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        lib.vg_fused_add_rms_norm_fp8.argtypes = [P, P, P, P, P, P, i64, i64, ctypes.c_float,
                                                  i32, i32, P]
        lib.vg_fused_add_rms_norm_fp8.restype = ctypes.c_int
        lib.vg_silu_mul_fp8.argtypes = [P, P, P, i64, i64, i32, i32, P]
        lib.vg_silu_mul_fp8.restype = ctypes.c_int
        f32 = ctypes.c_float
        lib.vg_fused_add_rms_norm_pad.argtypes = [P, P, P, P, P, i64, i64, i64, f32, P]
        lib.vg_fused_qk_norm_rope.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i64, f32, i32, P]
        lib.vg_fused_qk_norm_rope.restype = ctypes.c_int
        lib.vg_fused_add_rms_norm_pad.restype = ctypes.c_int
        lib.vg_fused_mla_dual_rms_norm.argtypes = [P, P, P, i64, P, P, i64, P, i64, i64, i64,
                                                   f32, f32, P]
        lib.vg_fused_mla_dual_rms_norm.restype = ctypes.c_int
        lib.vg_fused_mla_dual_rms_norm_per_token_quant.argtypes = [P, P, P, P, i64, P, P, i64, P,
                                                                   i64, i64, i64, f32, f32, P]
        lib.vg_fused_mla_dual_rms_norm_per_token_quant.restype = ctypes.c_int
        lib.vg_fused_add_rms_norm_nvfp4.argtypes = [P, P, P, P, P, P, P, i64, i64, f32, P]
        lib.vg_fused_add_rms_norm_nvfp4.restype = ctypes.c_int
        lib.vg_silu_mul_nvfp4.argtypes = [P, P, P, P, i64, i64, P]
        lib.vg_silu_mul_nvfp4.restype = ctypes.c_int
        lib.vg_status_string.argtypes = [ctypes.c_int]
        lib.vg_status_string.restype = ctypes.c_char_p
        lib.vg_abi_version.argtypes = []
        lib.vg_abi_version.restype = i32
        lib.vg_device_status.argtypes = [P, i32]
        lib.vg_device_status.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().vg_status_string(status).decode()


def _check(status: int):
    if status != 0:
        raise VgError(status, status_string(status))


# ----------------------------------------------------------- marshalling

def _ptr(t, dtypes, name):
    """Device pointer of a torch tensor (or pass an int pointer / None)."""
    if t is None or isinstance(t, int):
        return t
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, an int pointer or None")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtypes():
    import torch
    bf16 = (torch.bfloat16, torch.int16, torch.uint16)
    fp8 = (torch.float8_e4m3fn, torch.uint8, torch.int8)
    return bf16, fp8, (torch.float32,)


def _rows(t, name):
    if isinstance(t, int) or t is None:
        raise ValueError(f"{name}: shapes cannot be taken from a raw pointer; pass num_tokens")
    if t.dim() != 2:
        raise ValueError(f"{name}: expected a 2-D [T, n] tensor")
    return t.shape[0], t.shape[1]


def vg_fused_add_rms_norm_fp8(q, residual_out, scale, x, residual, weight, eps: float,
                              mode: int, group_size: int = 128, stream=None,
                              num_tokens: int | None = None, hidden: int | None = None):
    """Residual add + RMSNorm -> FP8 through the C ABI (outputs preallocated).

    q [T,H] fp8/uint8; residual_out [T,H] bf16 (may be ``residual`` itself)
    or None with residual None; scale fp32 ([1] static input, [T] or
    [T,H/G] output); x [T,H] bf16; residual [T,H] bf16 or None; weight [H]."""
    bf16, fp8, f32 = _dtypes()
    if num_tokens is None or hidden is None:
        num_tokens, hidden = _rows(x, "x")
    st = load().vg_fused_add_rms_norm_fp8(
        _ptr(q, fp8, "q"), _ptr(residual_out, bf16, "residual_out"), _ptr(scale, f32, "scale"),
        _ptr(x, bf16, "x"), _ptr(residual, bf16, "residual"), _ptr(weight, bf16, "weight"),
        num_tokens, hidden, ctypes.c_float(eps), mode, group_size, _stream(stream))
    _check(st)


def vg_silu_mul_fp8(q, scale, gate_up, mode: int, group_size: int = 128, stream=None,
                    num_tokens: int | None = None, inter: int | None = None):
    """SiLU(gate) * up -> FP8 through the C ABI (outputs preallocated).

    q [T,I] fp8/uint8; scale fp32 ([1] static input, [T] or [T,I/G]
    output); gate_up [T,2I] bf16 with gate = columns [0,I), up = [I,2I)."""
    bf16, fp8, f32 = _dtypes()
    if num_tokens is None or inter is None:
        num_tokens, two_i = _rows(gate_up, "gate_up")
        if two_i % 2:
            raise ValueError("gate_up must have an even number of columns")
        inter = two_i // 2
    st = load().vg_silu_mul_fp8(_ptr(q, fp8, "q"), _ptr(scale, f32, "scale"),
                                _ptr(gate_up, bf16, "gate_up"), num_tokens, inter, mode,
                                group_size, _stream(stream))
    _check(st)


def vg_fused_add_rms_norm_pad(out, residual_out, x, residual, weight, eps: float, stream=None,
                              num_tokens: int | None = None, hidden: int | None = None,
                              padded_hidden: int | None = None):
    """Residual add + RMSNorm into a padded bf16 row through the C ABI.

    out [T, padded] bf16 (columns >= H come back zero); residual_out [T,H]
    (may be ``residual`` itself) or None with residual None; x [T,H]; weight [H]."""
    bf16, _, _ = _dtypes()
    if num_tokens is None or hidden is None:
        num_tokens, hidden = _rows(x, "x")
    if padded_hidden is None:
        padded_hidden = _rows(out, "out")[1]
    _check(load().vg_fused_add_rms_norm_pad(
        _ptr(out, bf16, "out"), _ptr(residual_out, bf16, "residual_out"), _ptr(x, bf16, "x"),
        _ptr(residual, bf16, "residual"), _ptr(weight, bf16, "weight"), num_tokens, hidden,
        padded_hidden, ctypes.c_float(eps), _stream(stream)))


def vg_fused_qk_norm_rope(qkv, q_weight, k_weight, cos_sin_cache, positions, num_q_heads: int,
                          num_kv_heads: int, head_dim: int, eps: float, is_neox: bool = True,
                          stream=None):
    """Per-head QK RMSNorm + rotary embedding, in place on qkv
    [T, (Hq + 2 Hkv) * D] bf16; cos_sin_cache fp32 [max_pos, D]; positions
    int64 [T]."""
    import torch
    bf16, _, f32 = _dtypes()
    T = _rows(qkv, "qkv")[0]
    max_pos = _rows(cos_sin_cache, "cos_sin_cache")[0]
    _check(load().vg_fused_qk_norm_rope(
        _ptr(qkv, bf16, "qkv"), _ptr(q_weight, bf16, "q_weight"), _ptr(k_weight, bf16, "k_weight"),
        _ptr(cos_sin_cache, f32, "cos_sin_cache"), _ptr(positions, (torch.int64,), "positions"),
        T, num_q_heads, num_kv_heads, head_dim, max_pos, ctypes.c_float(eps),
        1 if is_neox else 0, _stream(stream)))


def _rows_ptr(t, name):
    """(device pointer, row stride in elements, rows, columns) of a 2-D bf16
    CUDA tensor whose rows are contiguous (a column slice is fine)."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    bf16, _, _ = _dtypes()
    if t.dtype not in bf16:
        raise TypeError(f"{name}: dtype {t.dtype} not in {bf16}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (there is no CPU path)")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name}: expected a 2-D [T, n] tensor with contiguous rows")
    return t.data_ptr(), t.stride(0), t.shape[0], t.shape[1]


def vg_fused_mla_dual_rms_norm(q_out, kv_out, q_c, q_weight, kv_c, kv_weight, eps_q: float,
                               eps_kv: float, stream=None):
    """MLA dual RMSNorm through the C ABI: q_out = bf16(rms_norm(q_c)),
    kv_out = bf16(rms_norm(kv_c)) in one launch (outputs preallocated,
    dense bf16; q_c / kv_c may be column slices of one projected tensor)."""
    bf16, _, _ = _dtypes()
    qp, qs, T, q_dim = _rows_ptr(q_c, "q_c")
    kp, ks, T2, kv_dim = _rows_ptr(kv_c, "kv_c")
    if T2 != T:
        raise ValueError("q_c and kv_c must have the same number of rows")
    _check(load().vg_fused_mla_dual_rms_norm(
        _ptr(q_out, bf16, "q_out"), _ptr(kv_out, bf16, "kv_out"), qp, qs,
        _ptr(q_weight, bf16, "q_weight"), kp, ks, _ptr(kv_weight, bf16, "kv_weight"),
        T, q_dim, kv_dim, ctypes.c_float(eps_q), ctypes.c_float(eps_kv), _stream(stream)))


def vg_fused_mla_dual_rms_norm_per_token_quant(q_fp8, q_scale, kv_out, q_c, q_weight, kv_c,
                                               kv_weight, eps_q: float, eps_kv: float,
                                               stream=None):
    """The per-token-quant variant: q to FP8 with q_scale [T] fp32, kv bf16."""
    bf16, fp8, f32 = _dtypes()
    qp, qs, T, q_dim = _rows_ptr(q_c, "q_c")
    kp, ks, T2, kv_dim = _rows_ptr(kv_c, "kv_c")
    if T2 != T:
        raise ValueError("q_c and kv_c must have the same number of rows")
    _check(load().vg_fused_mla_dual_rms_norm_per_token_quant(
        _ptr(q_fp8, fp8, "q_fp8"), _ptr(q_scale, f32, "q_scale"), _ptr(kv_out, bf16, "kv_out"),
        qp, qs, _ptr(q_weight, bf16, "q_weight"), kp, ks, _ptr(kv_weight, bf16, "kv_weight"),
        T, q_dim, kv_dim, ctypes.c_float(eps_q), ctypes.c_float(eps_kv), _stream(stream)))


def vg_fused_add_rms_norm_nvfp4(q4, block_scale, residual_out, x, residual, weight,
                                global_scale, eps: float, stream=None,
                                num_tokens: int | None = None, hidden: int | None = None):
    """Residual add + RMSNorm -> NVFP4 through the C ABI (outputs preallocated).

    q4 [T,H/2] uint8 (two E2M1 codes a byte, column 2i in the low nibble);
    block_scale [T,H/16] uint8 E4M3 codes; residual_out as for the FP8 op;
    global_scale fp32 [1] on the device."""
    import torch
    bf16, fp8, f32 = _dtypes()
    u8 = (torch.uint8,)
    if num_tokens is None or hidden is None:
        num_tokens, hidden = _rows(x, "x")
    _check(load().vg_fused_add_rms_norm_nvfp4(
        _ptr(q4, u8, "q4"), _ptr(block_scale, fp8, "block_scale"),
        _ptr(residual_out, bf16, "residual_out"), _ptr(x, bf16, "x"),
        _ptr(residual, bf16, "residual"), _ptr(weight, bf16, "weight"),
        _ptr(global_scale, f32, "global_scale"), num_tokens, hidden, ctypes.c_float(eps),
        _stream(stream)))


def vg_silu_mul_nvfp4(q4, block_scale, gate_up, global_scale, stream=None,
                      num_tokens: int | None = None, inter: int | None = None):
    """SiLU(gate) * up -> NVFP4 through the C ABI: q4 [T,I/2] uint8,
    block_scale [T,I/16] E4M3 codes, gate_up [T,2I] bf16, global_scale fp32
    [1] on the device."""
    import torch
    bf16, fp8, f32 = _dtypes()
    if num_tokens is None or inter is None:
        num_tokens, two_i = _rows(gate_up, "gate_up")
        if two_i % 2:
            raise ValueError("gate_up must have an even number of columns")
        inter = two_i // 2
    _check(load().vg_silu_mul_nvfp4(
        _ptr(q4, (torch.uint8,), "q4"), _ptr(block_scale, fp8, "block_scale"),
        _ptr(gate_up, bf16, "gate_up"), _ptr(global_scale, f32, "global_scale"), num_tokens,
        inter, _stream(stream)))


def vg_device_status(reset: bool = False) -> int:
    """Flags the library's kernels left on the current device
    (DEVICE_WAIT_TIMEOUT: a bounded wait gave up; that call's outputs are
    not valid).  Synchronous."""
    flags = ctypes.c_uint32(0)
    _check(load().vg_device_status(ctypes.byref(flags), 1 if reset else 0))
    return flags.value


# ------------------------------------------------- allocating wrappers

def _scale_out(mode, T, n, group_size, scale, device):
    import torch
    if mode & COLUMN_MAJOR:
        return torch.empty((n // group_size, (T + 3) // 4 * 4), dtype=torch.float32, device=device)
    mode &= 0xFF
    if mode == STATIC:
        if scale is None:
            raise ValueError("static mode needs a scale tensor")
        return scale
    if mode == PER_TOKEN:
        return torch.empty((T,), dtype=torch.float32, device=device)
    return torch.empty((T, n // group_size), dtype=torch.float32, device=device)


def fused_add_rms_norm_fp8(x, residual, weight, eps: float, mode: int, group_size: int = 128,
                           scale=None, inplace: bool = True, stream=None):
    """Returns (q float8_e4m3fn [T,H], scale, residual_out).  With
    ``inplace`` the residual is updated in place, as the fused op does."""
    import torch
    T, H = x.shape
    q = torch.empty((T, H), dtype=torch.float8_e4m3fn, device=x.device)
    s = _scale_out(mode, T, H, group_size, scale, x.device)
    r_out = None
    if residual is not None:
        r_out = residual if inplace else torch.empty_like(residual)
    vg_fused_add_rms_norm_fp8(q, r_out, s, x, residual, weight, eps, mode, group_size, stream)
    return q, s, r_out


def silu_mul_fp8(gate_up, mode: int, group_size: int = 128, scale=None, stream=None):
    """Returns (q float8_e4m3fn [T,I], scale)."""
    import torch
    T, two_i = gate_up.shape
    q = torch.empty((T, two_i // 2), dtype=torch.float8_e4m3fn, device=gate_up.device)
    s = _scale_out(mode, T, two_i // 2, group_size, scale, gate_up.device)
    vg_silu_mul_fp8(q, s, gate_up, mode, group_size, stream)
    return q, s


def mla_dual_rms_norm(q_c, q_weight, kv_c, kv_weight, eps_q: float, eps_kv: float,
                      q_fp8: bool = False, stream=None):
    """Returns (q_normed bf16 [T,q_dim], kv_normed bf16 [T,kv_dim]), or with
    ``q_fp8`` (q float8_e4m3fn [T,q_dim], q_scale fp32 [T], kv_normed)."""
    import torch
    T, q_dim = q_c.shape
    kv = torch.empty((T, kv_c.shape[1]), dtype=kv_c.dtype, device=kv_c.device)
    if q_fp8:
        q = torch.empty((T, q_dim), dtype=torch.float8_e4m3fn, device=q_c.device)
        s = torch.empty((T,), dtype=torch.float32, device=q_c.device)
        vg_fused_mla_dual_rms_norm_per_token_quant(q, s, kv, q_c, q_weight, kv_c, kv_weight,
                                                   eps_q, eps_kv, stream)
        return q, s, kv
    q = torch.empty((T, q_dim), dtype=q_c.dtype, device=q_c.device)
    vg_fused_mla_dual_rms_norm(q, kv, q_c, q_weight, kv_c, kv_weight, eps_q, eps_kv, stream)
    return q, kv


def fused_add_rms_norm_pad(x, residual, weight, eps: float, padded_hidden: int,
                           inplace: bool = True, stream=None):
    """Returns (out bf16 [T, padded_hidden], residual_out)."""
    import torch
    T, H = x.shape
    out = torch.empty((T, padded_hidden), dtype=x.dtype, device=x.device)
    r_out = None
    if residual is not None:
        r_out = residual if inplace else torch.empty_like(residual)
    vg_fused_add_rms_norm_pad(out, r_out, x, residual, weight, eps, stream)
    return out, r_out


def fused_add_rms_norm_nvfp4(x, residual, weight, eps: float, global_scale, inplace: bool = True,
                             stream=None):
    """Returns (q4 uint8 [T,H/2], block_scale float8_e4m3fn [T,H/16],
    residual_out); global_scale is an fp32 [1] device tensor."""
    import torch
    T, H = x.shape
    q4 = torch.empty((T, H // 2), dtype=torch.uint8, device=x.device)
    sf = torch.empty((T, H // 16), dtype=torch.float8_e4m3fn, device=x.device)
    r_out = None
    if residual is not None:
        r_out = residual if inplace else torch.empty_like(residual)
    vg_fused_add_rms_norm_nvfp4(q4, sf, r_out, x, residual, weight, global_scale, eps, stream)
    return q4, sf, r_out


def silu_mul_nvfp4(gate_up, global_scale, stream=None):
    """Returns (q4 uint8 [T,I/2], block_scale float8_e4m3fn [T,I/16])."""
    import torch
    T, two_i = gate_up.shape
    q4 = torch.empty((T, two_i // 4), dtype=torch.uint8, device=gate_up.device)
    sf = torch.empty((T, two_i // 32), dtype=torch.float8_e4m3fn, device=gate_up.device)
    vg_silu_mul_nvfp4(q4, sf, gate_up, global_scale, stream)
    return q4, sf
