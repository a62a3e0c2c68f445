"""The fp64 oracle over a whole problem, on every host core.

Full-size parity tests compare every output row of the CUDA path with the
oracle.  The oracle is single-threaded C called through ctypes, which drops
the GIL for the duration of each call, so a thread pool over sequences
(decode) or over blocks of query tokens (MLA) runs it on all cores.  Work is
handed out longest first so one long sequence does not finish last.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle


def _threads() -> int:
    return max(1, os.cpu_count() or 1)


def decode_all(case) -> np.ndarray:
    """oracle.decode for every sequence of `case`; shaped like q."""
    ref = np.full(case["q"].shape, np.nan)
    order = np.argsort(-np.asarray(case["context_lens"], dtype=np.int64), kind="stable")
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(lambda b: oracle.decode(case, int(b), int(b) + 1, out=ref), order))
    return ref


def mla_all(case, block: int = 8):
    """oracle.mla for every query token of `case`: (out, lse)."""
    T = int(case["total_q"])
    out = np.full((T, case["H"], case["Dc"]), np.nan)
    lse = np.full((T, case["H"]), np.nan)
    # cost of a token ~ the keys it sees: later tokens of longer sequences first
    qo, kvp = case["qo_indptr"], case["kv_indptr"]
    starts = []
    for b in range(len(qo) - 1):
        q_len, kv_len = int(qo[b + 1] - qo[b]), int(kvp[b + 1] - kvp[b])
        for i0 in range(0, q_len, block):
            starts.append((kv_len - q_len + i0, int(qo[b]) + i0, min(int(qo[b + 1]), int(qo[b]) + i0 + block)))
    starts.sort(reverse=True)
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(lambda s: oracle.mla(case, s[1], s[2], out=out, lse=lse), starts))
    return out, lse
