"""ctypes binding of libpkv (include/pkv.h), same function names.

Argument marshalling only: device tensors are passed as raw pointers, shapes
as integers, and the caller's current CUDA stream is used unless one is given.
No computation happens here; a missing library raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")
_lib = None

PKV_OK, PKV_INVALID_ARG, PKV_UNSUPPORTED, PKV_WORKSPACE_TOO_SMALL, PKV_CUDA_ERROR, PKV_BAD_BLOCK_TABLE = range(6)
PKV_F16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2
PKV_KV_AS_Q = 0
PKV_DECODE_DEVICE_PLAN = 1
PKV_DECODE_PLAN_READY = 2
PKV_LAYOUT_NHD, PKV_LAYOUT_VLLM = 0, 1

FUNCTIONS = [
    "pkv_status_string", "pkv_version", "pkv_plan_splits", "pkv_decode_workspace_size",
    "pkv_paged_decode_attention", "pkv_decode_partials", "pkv_combine", "pkv_validate_block_table",
    "pkv_paged_decode_attention_static", "pkv_static_scratch_error", "pkv_mla_workspace_size",
    "pkv_mla_paged_prefill", "pkv_set_stress_delay",
]
PKV_STATIC_SCRATCH_BYTES = 32 << 20


class pkv_decode_desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
                ("block_size", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int), ("num_blocks", ctypes.c_int),
                ("max_context_len", ctypes.c_int), ("sum_context_len", ctypes.c_longlong),
                ("dtype", ctypes.c_int), ("layout", ctypes.c_int), ("x_pack", ctypes.c_int),
                ("kv_dtype", ctypes.c_int), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
                ("q_len", ctypes.c_int)]


class pkv_decode_opts(ctypes.Structure):
    _fields_ = [("partition_tokens", ctypes.c_int), ("num_splits", ctypes.c_int), ("flags", ctypes.c_int),
                ("phase1_event_start", ctypes.c_void_p), ("phase1_event_stop", ctypes.c_void_p),
                ("alibi_slopes", ctypes.c_void_p)]


class pkv_mla_desc(ctypes.Structure):
    _fields_ = [("total_q", ctypes.c_int), ("num_heads", ctypes.c_int), ("d_ckv", ctypes.c_int),
                ("d_kpe", ctypes.c_int), ("batch", ctypes.c_int), ("num_pages", ctypes.c_int),
                ("nnz", ctypes.c_int), ("max_kv_len", ctypes.c_int)]


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__("%s failed: %s (%d)" % (fn, status_string(status), status))
        self.status = status


def load():
    """Load libpkv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libpkv.so is missing at %s: run __graft_entry__.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    D, O = ctypes.POINTER(pkv_decode_desc), ctypes.POINTER(pkv_decode_opts)
    lib.pkv_status_string.argtypes = [I]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_version.argtypes = []
    lib.pkv_version.restype = I
    lib.pkv_plan_splits.argtypes = [D, O, I, ctypes.POINTER(I), ctypes.POINTER(I)]
    lib.pkv_decode_workspace_size.argtypes = [D, O, I, ctypes.POINTER(SZ)]
    lib.pkv_paged_decode_attention.argtypes = [D, O, P, P, P, P, P, ctypes.c_float, P, P, SZ, P]
    lib.pkv_decode_partials.argtypes = [D, O, P, P, P, P, P, ctypes.c_float, P, P, P, I,
                                        ctypes.POINTER(I), ctypes.POINTER(I), P]
    lib.pkv_combine.argtypes = [D, I, I, P, P, P, P, P, P]
    lib.pkv_validate_block_table.argtypes = [D, P, P, P, P]
    lib.pkv_paged_decode_attention_static.argtypes = [D, O, P, P, P, P, P, ctypes.c_float, P, P]
    lib.pkv_static_scratch_error.argtypes = [P, P]
    lib.pkv_set_stress_delay.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
    lib.pkv_mla_workspace_size.argtypes = [ctypes.POINTER(pkv_mla_desc), ctypes.POINTER(SZ)]
    lib.pkv_mla_paged_prefill.argtypes = [ctypes.POINTER(pkv_mla_desc), P, P, P, P, P, P, P, ctypes.c_float,
                                          P, P, P, SZ, P]
    for f in FUNCTIONS[2:]:
        getattr(lib, f).restype = I
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def _check(fn: str, st: int) -> None:
    if st != PKV_OK:
        raise PkvError(fn, st)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_desc(B, Hq, Hkv, D, block_size, max_blocks_per_seq, num_blocks, max_context_len, sum_context_len,
              dtype, layout=PKV_LAYOUT_NHD, x_pack=8, kv_dtype=PKV_KV_AS_Q, k_scale=1.0,
              v_scale=1.0, q_len=1) -> pkv_decode_desc:
    return pkv_decode_desc(int(B), int(Hq), int(Hkv), int(D), int(block_size), int(max_blocks_per_seq),
                           int(num_blocks), int(max_context_len), int(sum_context_len), int(dtype), int(layout),
                           int(x_pack), int(kv_dtype), float(k_scale), float(v_scale), int(q_len))


def make_opts(partition_tokens=0, num_splits=0, event_start=None, event_stop=None,
              alibi_slopes=None, device_plan=False, plan_ready=False, flags=None) -> pkv_decode_opts:
    """alibi_slopes: a device fp32 tensor [Hq] (kept alive by the caller) or None.
    device_plan: plan the splits on the device (PKV_DECODE_DEVICE_PLAN); plan_ready: reuse the
    plan an earlier device-planned call left in the workspace; flags: raw flag word."""
    ev = lambda e: None if e is None else (e if isinstance(e, int) else e.cuda_event)
    if flags is None:
        flags = (PKV_DECODE_DEVICE_PLAN if device_plan or plan_ready else 0) | (PKV_DECODE_PLAN_READY if plan_ready else 0)
    return pkv_decode_opts(int(partition_tokens), int(num_splits), int(flags), ev(event_start), ev(event_stop),
                           _ptr(alibi_slopes))


def _opt_ref(opts):
    return None if opts is None else ctypes.byref(opts)


def pkv_version() -> int:
    return load().pkv_version()


def pkv_plan_splits(desc, opts=None, num_sms: int = 0):
    """(num_splits, partition_tokens) of the split planner."""
    ns, P = ctypes.c_int(0), ctypes.c_int(0)
    _check("pkv_plan_splits", load().pkv_plan_splits(ctypes.byref(desc), _opt_ref(opts), int(num_sms),
                                                     ctypes.byref(ns), ctypes.byref(P)))
    return ns.value, P.value


def pkv_decode_workspace_size(desc, opts=None, num_sms: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check("pkv_decode_workspace_size", load().pkv_decode_workspace_size(ctypes.byref(desc), _opt_ref(opts),
                                                                         int(num_sms), ctypes.byref(n)))
    return n.value


def pkv_paged_decode_attention(desc, q, k_cache, v_cache, block_table, context_lens, scale, out, workspace,
                               workspace_bytes=None, opts=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("pkv_paged_decode_attention", load().pkv_paged_decode_attention(
        ctypes.byref(desc), _opt_ref(opts), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(context_lens), float(scale), _ptr(out), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def pkv_decode_partials(desc, q, k_cache, v_cache, block_table, context_lens, scale, part_acc, part_m, part_l,
                        num_splits_capacity, opts=None, stream=None):
    """Runs phase 1 alone; returns (partition_tokens, num_splits)."""
    P, ns = ctypes.c_int(0), ctypes.c_int(0)
    _check("pkv_decode_partials", load().pkv_decode_partials(
        ctypes.byref(desc), _opt_ref(opts), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(context_lens), float(scale), _ptr(part_acc), _ptr(part_m), _ptr(part_l), int(num_splits_capacity),
        ctypes.byref(P), ctypes.byref(ns), _stream(stream)))
    return P.value, ns.value


def pkv_combine(desc, partition_tokens, num_splits, context_lens, part_acc, part_m, part_l, out,
                stream=None) -> None:
    _check("pkv_combine", load().pkv_combine(ctypes.byref(desc), int(partition_tokens), int(num_splits),
                                             _ptr(context_lens), _ptr(part_acc), _ptr(part_m), _ptr(part_l),
                                             _ptr(out), _stream(stream)))


def pkv_paged_decode_attention_static(desc, q, k_cache, v_cache, block_table, context_lens, scale, out,
                                      opts=None, stream=None) -> None:
    """Decode step with the library's static device scratch (allocates nothing)."""
    _check("pkv_paged_decode_attention_static", load().pkv_paged_decode_attention_static(
        ctypes.byref(desc), _opt_ref(opts), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(context_lens), float(scale), _ptr(out), _stream(stream)))


def pkv_static_scratch_error(dst, stream=None) -> None:
    """Copies the static scratch's error word into dst (4 bytes, device or host memory)."""
    _check("pkv_static_scratch_error", load().pkv_static_scratch_error(_ptr(dst), _stream(stream)))


def pkv_set_stress_delay(producer_delay_ns: int, consumer_delay_ns: int = 0) -> None:
    """Producer / consumer pauses (ns) in later calls; 0 turns each off (race testing)."""
    _check("pkv_set_stress_delay", load().pkv_set_stress_delay(int(producer_delay_ns), int(consumer_delay_ns)))


def make_mla_desc(total_q, batch, num_pages, nnz, num_heads=16, d_ckv=512, d_kpe=64, max_kv_len=0) -> pkv_mla_desc:
    return pkv_mla_desc(int(total_q), int(num_heads), int(d_ckv), int(d_kpe), int(batch), int(num_pages),
                        int(nnz), int(max_kv_len))


def pkv_mla_workspace_size(desc) -> int:
    n = ctypes.c_size_t(0)
    _check("pkv_mla_workspace_size", load().pkv_mla_workspace_size(ctypes.byref(desc), ctypes.byref(n)))
    return n.value


def pkv_mla_paged_prefill(desc, q_nope, q_pe, ckv_cache, kpe_cache, qo_indptr, kv_indptr, kv_indices, sm_scale,
                          out, lse, workspace, workspace_bytes=None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("pkv_mla_paged_prefill", load().pkv_mla_paged_prefill(
        ctypes.byref(desc), _ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache), _ptr(qo_indptr),
        _ptr(kv_indptr), _ptr(kv_indices), float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        int(workspace_bytes), _stream(stream)))


def pkv_validate_block_table(desc, block_table, context_lens, err_word, stream=None) -> None:
    _check("pkv_validate_block_table", load().pkv_validate_block_table(
        ctypes.byref(desc), _ptr(block_table), _ptr(context_lens), _ptr(err_word), _stream(stream)))


def raw_status(fn: str, *args) -> int:
    """Calls a C-ABI function with raw arguments and returns its status (tests of the error paths)."""
    return getattr(load(), fn)(*args)
