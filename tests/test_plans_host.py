"""Launch plans, on the host (no GPU): the plan each entry point picks covers
every row and every 16-byte chunk of a row with a kernel instance that
exists, within that instance's thread limit.

The plan functions are the library's own (vg::plan_* in vg_fused.cu), called
through their C++ symbols; the structs below mirror launch.h field by field.
Each kernel maps work to threads as follows, and each test checks the plan
against that map over sweeps of token counts (around every plan switch),
row widths and SM counts:
  register norm / SiLU kernels: thread i of a row owns chunks i + k * ntr,
    k < vpt; a CTA holds rpc rows (CTA b: rows b * rpc ..); a SiLU row
    segment s starts at chunk s * ntr * vpt;
  persistent kernels: CTA b takes rows b, b + grid, ...; a row's chunks are
    block * vpt wide (the SiLU's in nseg segments of vpt / nseg a thread);
  MLA warp kernel: eight warps a CTA, warp w of CTA b on token b * 8 + w, or
    b + w * grid when the plan deals a single wave; MLA warp-group kernel:
    thr[side] threads a row, vpt chunks each, rpc tokens a CTA.
Parity of every plan branch against the oracle is tested on the GPU."""
import ctypes

import numpy as np
import pytest

import norm_activation_fp8_gb300 as vg
from norm_activation_fp8_gb300 import build

STATIC, PER_TOKEN, PER_GROUP, NVFP4 = 0, 1, 2, 5
TMA_MAX_SMEM = 227 * 1024  # kTmaMaxSmem
SMS = [152, 148, 132, 16, 2, 1]


class RowPlan(ctypes.Structure):
    _fields_ = [("vpt", ctypes.c_int), ("ntr", ctypes.c_int), ("rpc", ctypes.c_int),
                ("grid", ctypes.c_int64), ("segs", ctypes.c_int), ("dense", ctypes.c_bool)]


class TmaPlan(ctypes.Structure):
    _fields_ = [("vpt", ctypes.c_int), ("block", ctypes.c_int), ("stages", ctypes.c_int),
                ("grid", ctypes.c_int64), ("smem", ctypes.c_size_t)]


class SiluTmaPlan(ctypes.Structure):
    _fields_ = [("vpt", ctypes.c_int), ("block", ctypes.c_int), ("nseg", ctypes.c_int),
                ("grid", ctypes.c_int64), ("smem", ctypes.c_size_t)]


class MlaPlan(ctypes.Structure):
    _fields_ = [("spread", ctypes.c_bool), ("vpt", ctypes.c_int), ("thr", ctypes.c_int * 2),
                ("rpc", ctypes.c_int), ("block", ctypes.c_int), ("grid", ctypes.c_int64)]


@pytest.fixture(scope="module")
def plans():
    build.build()
    lib = vg.load()
    i64, i32, b = ctypes.c_int64, ctypes.c_int, ctypes.c_bool

    def fn(name, restype, *argtypes):
        f = getattr(lib, name)
        f.restype, f.argtypes = restype, list(argtypes)
        return f

    return {
        "rows": fn("_ZN2vg9plan_rowsEliii", RowPlan, i64, i32, i32, i32),
        "silu": fn("_ZN2vg9plan_siluEliii", RowPlan, i64, i32, i32, i32),
        "silu_tma": fn("_ZN2vg19plan_silu_tma_tokenEliiiPNS_11SiluTmaPlanE", b, i64, i32, i32,
                       i32, ctypes.POINTER(SiluTmaPlan)),
        "norm_tma": fn("_ZN2vg13plan_norm_tmaElibiiiPNS_7TmaPlanE", b, i64, i32, b, i32, i32, i32,
                       ctypes.POINTER(TmaPlan)),
        "mla": fn("_ZN2vg8plan_mlaEliibi", MlaPlan, i64, i32, i32, b, i32),
        "norm_smem": fn("_ZN2vg19norm_tma_smem_bytesEibiiii", ctypes.c_size_t, i32, b, i32, i32,
                        i32, i32),
        "silu_smem": fn("_ZN2vg25silu_tma_token_smem_bytesEii", ctypes.c_size_t, i32, i32),
    }


def token_counts(sms):
    """1..40, and k * sms - 1, k * sms, k * sms + 1 for every multiple the
    plans switch at (2, 4, 10, 13, 32, 40 rows per SM and more)."""
    ts = set(range(1, 41))
    for k in (1, 2, 3, 4, 8, 10, 12, 13, 16, 20, 32, 40, 41, 64, 128, 160, 320):
        for d in (-1, 0, 1):
            if k * sms + d >= 1:
                ts.add(k * sms + d)
    ts |= {4096, 16384, 32768, 65536, 1 << 20}
    return sorted(ts)


def widths():
    """Chunk counts (row width / 8): every count up to 160, the workloads'
    widths and seeded random ones, up to 32768 columns."""
    rng = np.random.default_rng(7)
    n = set(range(1, 161)) | {192, 256, 360, 384, 448, 512, 896, 1024, 1536, 1792, 2048, 3584,
                              4096}
    n |= set(int(v) for v in rng.integers(1, 4097, 40))
    return sorted(n)


def check_row_cover(p, T, nch, limit):
    assert p.vpt in (1, 2, 4, 8), p.vpt
    assert p.ntr % 32 == 0 and 32 <= p.ntr
    assert p.rpc >= 1 and p.ntr * p.rpc <= limit, (p.ntr, p.rpc)
    assert p.grid * p.rpc >= T and (p.grid - 1) * p.rpc < T, (p.grid, p.rpc, T)
    assert p.segs >= 1
    seg = p.ntr * p.vpt  # chunks a segment (a whole row when segs == 1)
    assert p.segs * seg >= nch and (p.segs - 1) * seg < nch, (p.segs, seg, nch)


@pytest.mark.parametrize("sms", SMS)
def test_norm_register_plan(plans, sms):
    for T in token_counts(sms):
        for nch in widths():
            for min_vpt in (2, 4):  # FP8 modes and padding; NVFP4
                p = plans["rows"](T, nch, min_vpt, sms)
                check_row_cover(p, T, nch, 512)
                assert p.segs == 1 and not p.dense
                assert p.ntr <= 512


@pytest.mark.parametrize("sms", SMS)
def test_silu_register_plan(plans, sms):
    for T in token_counts(sms):
        for nch in widths():
            for mode in (STATIC, PER_TOKEN, PER_GROUP):
                p = plans["silu"](T, nch, mode, sms)
                assert p.vpt in (1, 2, 4)  # the SiLU instances
                if mode == PER_TOKEN:
                    # the row's amax needs the row in one CTA (up to 1024 threads)
                    check_row_cover(p, T, nch, 1024)
                    assert p.segs == 1 and not p.dense
                else:
                    check_row_cover(p, T, nch, 512)
                    if nch > 64:
                        assert p.ntr <= 448
                    if p.dense:  # the four-CTA instances exist for two chunks a thread or fewer
                        assert p.vpt <= 2 and T >= 2 * sms


@pytest.mark.parametrize("sms", SMS)
def test_silu_persistent_token_plan(plans, sms):
    out = SiluTmaPlan()
    for T in token_counts(sms):
        for nch in widths():
            for mode in (STATIC, PER_TOKEN, PER_GROUP):
                if not plans["silu_tma"](T, nch, mode, sms, ctypes.byref(out)):
                    continue
                assert mode == PER_TOKEN and T >= 2 * sms
                p = out
                assert p.nseg in (1, 2) and nch % p.nseg == 0
                assert p.block % 32 == 0 and 32 <= p.block <= 1024
                assert p.block * (p.vpt // p.nseg) >= nch // p.nseg
                assert 1 <= p.grid <= T
                need = plans["silu_smem"](nch * 8, p.nseg)
                assert need <= TMA_MAX_SMEM - 1024 and p.smem <= TMA_MAX_SMEM


@pytest.mark.parametrize("sms", SMS)
def test_norm_persistent_plan(plans, sms):
    out = TmaPlan()
    for T in token_counts(sms):
        for nch in widths():
            H = nch * 8
            for mode, group in ((STATIC, 0), (PER_TOKEN, 0), (PER_GROUP, 128), (PER_GROUP, 64),
                                (NVFP4, 16)):
                if group and H % group:
                    continue
                slots = H // group if group else 1
                for res in (True, False):
                    if not plans["norm_tma"](T, H, res, mode, slots, sms, ctypes.byref(out)):
                        continue
                    p = out
                    assert mode != STATIC and T >= 4 * sms
                    assert p.vpt in (2, 4, 8) and p.stages >= 1
                    assert p.block % 32 == 0 and 32 <= p.block <= 512
                    assert p.block * p.vpt >= nch
                    assert 1 <= p.grid <= T
                    need = plans["norm_smem"](H, res, p.stages, p.block, p.vpt, slots)
                    assert need <= TMA_MAX_SMEM and p.smem >= 0


MLA_WIDTHS = [(192, 64), (128, 64), (128, 127), (1, 1), (31, 225), (160, 96), (125, 50),
              (193, 64), (192, 65), (224, 64), (512, 256), (1024, 1024), (4096, 4096), (193, 65)]


@pytest.mark.parametrize("sms", SMS)
def test_mla_plan(plans, sms):
    for T in token_counts(sms):
        for nq, nkv in MLA_WIDTHS:
            for fp8 in (False, True):
                p = plans["mla"](T, nq, nkv, fp8, sms)
                warp = (nq + 31) // 32 + (nkv + 31) // 32 <= 8 and T >= 13 * sms
                if warp:
                    # one warp a token, eight warps a CTA; DeepSeek's widths
                    # run the staged instance (five CTAs a SM), others four
                    assert p.vpt == 0 and p.block == 256 and p.rpc == 8
                    wave = sms * (5 if (nq, nkv) == (192, 64) else 4)
                    assert p.spread == (T < 8 * wave)
                    if p.spread:
                        assert p.grid == wave and 8 * p.grid >= T
                    else:
                        assert p.grid == (T + 7) // 8
                    continue
                assert not p.spread and p.vpt in (1, 2, 4, 8)
                for side, n in enumerate((nq, nkv)):
                    assert p.thr[side] % 32 == 0 and p.thr[side] * p.vpt >= n
                per_tok = p.thr[0] + p.thr[1]
                assert p.block == p.rpc * per_tok
                assert p.block <= (1024 if p.vpt == 8 else 512)
                assert p.grid * p.rpc >= T and (p.grid - 1) * p.rpc < T
