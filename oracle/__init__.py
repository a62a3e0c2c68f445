"""fp64 CPU oracle for paged-KV decode attention and MLA paged causal prefill.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the product package.
The arithmetic lives in ``oracle.c`` (plain C, double precision); this module
only compiles it with gcc and marshals numpy arrays through ctypes.

Every function computes its definition directly (see the comments in
``oracle.c``, each citing the page and the function or section it follows).
Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force on tiny inputs, library routines, closed forms and invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

STATUS_OK, STATUS_INVALID, STATUS_BAD_TABLE = 0, 1, 5
F16, BF16, FP8_E4M3 = 0, 1, 2
NHD, VLLM = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (portable flags, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, d, p = ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.oracle_widen.argtypes = [ctypes.c_uint16, i]
            lib.oracle_widen.restype = d
            lib.oracle_widen8.argtypes = [ctypes.c_uint8]
            lib.oracle_widen8.restype = d
            lib.oracle_decode.argtypes = [i] * 12 + [p] * 5 + [d, d, d, p, i, i, p, p, p]
            lib.oracle_decode.restype = i
            lib.oracle_decode_partials.argtypes = [i] * 12 + [p] * 5 + [d, d, d, p, i, i, i, i, p, p, p, p]
            lib.oracle_decode_partials.restype = i
            lib.oracle_combine.argtypes = [i, i, i, i, i, p, p, p, p, i, i, p]
            lib.oracle_combine.restype = i
            lib.oracle_mla.argtypes = [i] * 6 + [p] * 7 + [d, i, i, p, p, p]
            lib.oracle_mla.restype = i
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__("oracle status %d" % status)
        self.status = status


def widen(bits: int, dtype: int) -> float:
    """Exact value of one fp16 (dtype=0) or bf16 (dtype=1) bit pattern."""
    return _load().oracle_widen(int(bits) & 0xFFFF, int(dtype))


def widen8(bits: int) -> float:
    """Exact value of one FP8 E4M3 bit pattern."""
    return _load().oracle_widen8(int(bits) & 0xFF)


def q_len_of(case) -> int:
    """Query tokens per sequence: q is [B][Hq][D] (one) or [B][q_len][Hq][D]."""
    return int(case.get("q_len", 1))


def _decode_common(case):
    kv_dtype = case.get("kv_dtype", case["dtype"])
    q_len = q_len_of(case)
    assert case["q"].size == case["B"] * q_len * case["Hq"] * case["D"]
    kv_np = np.uint8 if kv_dtype == FP8_E4M3 else np.uint16
    q = _c(case["q"], np.uint16)
    k = _c(case["k_cache"], kv_np)
    v = _c(case["v_cache"], kv_np)
    table = _c(case["block_table"], np.int32)
    ctx = _c(case["context_lens"], np.int32)
    dims = [case["B"], case["Hq"], case["Hkv"], case["D"], case["block_size"],
            table.shape[1] if table.ndim == 2 else 0, case["num_blocks"],
            case["dtype"], case["layout"], case.get("x", 8), kv_dtype, q_len]
    scales = [float(case["scale"]), float(case.get("k_scale", 1.0)), float(case.get("v_scale", 1.0))]
    alibi = case.get("alibi_slopes")
    if alibi is not None:
        alibi = _c(alibi, np.float64)
        assert alibi.shape == (case["Hq"],)
    return dims, (q, k, v, table, ctx), scales, alibi


def decode(case, b_lo: int = 0, b_hi: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """fp64 attention output shaped like q: [B][Hq][D], or [B][q_len][Hq][D] with
    several query tokens (only sequences b in [b_lo, b_hi) are filled)."""
    dims, arrs, scales, alibi = _decode_common(case)
    B, D = case["B"], case["D"]
    b_hi = B if b_hi is None else b_hi
    if out is None:
        out = np.full(case["q"].shape, np.nan)
    maxn = int(max(1, int(np.max(arrs[4][b_lo:b_hi], initial=1))))
    sbuf = np.zeros(maxn)
    acc = np.zeros(D)
    st = _load().oracle_decode(*dims, *[_ptr(a) for a in arrs], *scales, None if alibi is None else _ptr(alibi),
                               b_lo, b_hi, _ptr(out), _ptr(sbuf), _ptr(acc))
    if st:
        raise OracleError(st)
    return out


def decode_partials(case, P: int, NS: int, b_lo: int = 0, b_hi: int | None = None):
    """Split-mode partials (m, l, acc) with split s = tokens [s*P, min((s+1)*P, n)),
    cut at each query's causal window; leading dimensions those of q without D."""
    dims, arrs, scales, alibi = _decode_common(case)
    B, D = case["B"], case["D"]
    b_hi = B if b_hi is None else b_hi
    lead = case["q"].shape[:-1]
    pm = np.full(lead + (NS,), np.nan)
    pl = np.full(lead + (NS,), np.nan)
    pacc = np.full(lead + (NS, D), np.nan)
    sbuf = np.zeros(max(1, P))
    st = _load().oracle_decode_partials(*dims, *[_ptr(a) for a in arrs], *scales,
                                        None if alibi is None else _ptr(alibi), int(P), int(NS), b_lo, b_hi,
                                        _ptr(pm), _ptr(pl), _ptr(pacc), _ptr(sbuf))
    if st:
        raise OracleError(st)
    return pm, pl, pacc


def combine(context_lens, pm, pl, pacc) -> np.ndarray:
    """Log-sum-exp combine of split partials ([B][Hq][NS][D] or [B][q_len][Hq][NS][D])
    into the output ([B][Hq][D] or [B][q_len][Hq][D])."""
    ctx = _c(context_lens, np.int32)
    pm, pl, pacc = _c(pm, np.float64), _c(pl, np.float64), _c(pacc, np.float64)
    if pacc.ndim == 4:
        B, Hq, NS, D = pacc.shape
        q_len = 1
    else:
        B, q_len, Hq, NS, D = pacc.shape
    out = np.full(pacc.shape[:-2] + (D,), np.nan)
    st = _load().oracle_combine(B, q_len, Hq, D, NS, _ptr(ctx), _ptr(pm), _ptr(pl), _ptr(pacc), 0, B, _ptr(out))
    if st:
        raise OracleError(st)
    return out


def mla(case, t_lo: int = 0, t_hi: int | None = None, out=None, lse=None):
    """fp64 MLA paged causal prefill: (out [total_q][H][Dc], lse base 2 [total_q][H])."""
    qn = _c(case["q_nope"], np.uint16)
    qp = _c(case["q_pe"], np.uint16)
    ckv = _c(case["ckv_cache"], np.uint16)
    kpe = _c(case["kpe_cache"], np.uint16)
    qo = _c(case["qo_indptr"], np.int32)
    kvp = _c(case["kv_indptr"], np.int32)
    kvi = _c(case["kv_indices"], np.int32)
    T, H, Dc = qn.shape
    Dr = qp.shape[2]
    t_hi = T if t_hi is None else t_hi
    if out is None:
        out = np.full((T, H, Dc), np.nan)
    if lse is None:
        lse = np.full((T, H), np.nan)
    maxkv = int(max(1, int(np.max(np.diff(kvp), initial=1))))
    sbuf = np.zeros(maxkv)
    st = _load().oracle_mla(T, H, Dc, Dr, len(qo) - 1, ckv.shape[0],
                            _ptr(qn), _ptr(qp), _ptr(ckv), _ptr(kpe), _ptr(qo), _ptr(kvp), _ptr(kvi),
                            float(case["sm_scale"]), t_lo, t_hi, _ptr(out), _ptr(lse), _ptr(sbuf))
    if st:
        raise OracleError(st)
    return out, lse
