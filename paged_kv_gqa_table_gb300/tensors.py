"""Device-memory plumbing around the C ABI: uploads synthetic cases into torch
CUDA tensors, sizes workspaces and wraps the calls with torch-allocated
outputs.  Nothing here computes attention; every step runs in libpkv."""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from . import synth

TORCH_DTYPE = {synth.F16: torch.float16, synth.BF16: torch.bfloat16}


def bits_to_torch(bits: np.ndarray, dtype: int, device, pin: bool = False) -> torch.Tensor:
    """uint16 bit patterns -> torch fp16/bf16 tensor (on `device`, or pinned host memory)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH_DTYPE[dtype])
    if device == "cpu":
        return t.pin_memory() if pin else t
    return t.to(device)


def int_to_torch(a: np.ndarray, device, pin: bool = False) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))
    if device == "cpu":
        return t.pin_memory() if pin else t
    return t.to(device)


def fp8_kv(case: dict) -> bool:
    return case.get("kv_dtype", case["dtype"]) == synth.FP8_E4M3


def decode_desc(case: dict) -> B.pkv_decode_desc:
    ctx = case["context_lens"]
    kv = dict(kv_dtype=B.PKV_FP8_E4M3, k_scale=case["k_scale"], v_scale=case["v_scale"]) if fp8_kv(case) else {}
    return B.make_desc(case["B"], case["Hq"], case["Hkv"], case["D"], case["block_size"],
                       case["block_table"].shape[1], case["num_blocks"], int(np.max(ctx, initial=0)),
                       int(np.sum(ctx, dtype=np.int64)), case["dtype"], case["layout"], case.get("x", 8), **kv,
                       q_len=case.get("q_len", 1))


def cache_to_torch(bits: np.ndarray, case: dict, device) -> torch.Tensor:
    """A KV cache array: fp16/bf16 bits as that dtype, FP8 E4M3 bits as uint8."""
    if fp8_kv(case):
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).to(device)
    return bits_to_torch(bits, case["dtype"], device)


def upload_decode_case(case: dict, device="cuda") -> dict:
    dt = case["dtype"]
    return dict(q=bits_to_torch(case["q"], dt, device), k_cache=cache_to_torch(case["k_cache"], case, device),
                v_cache=cache_to_torch(case["v_cache"], case, device),
                block_table=int_to_torch(case["block_table"], device),
                context_lens=int_to_torch(case["context_lens"], device))


def _aligned_zeros(n: int, device) -> torch.Tensor:
    ws = torch.zeros((n + 255) // 256 * 256 + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def workspace_for(desc, opts=None, device="cuda") -> torch.Tensor:
    """Zeroed, 256-byte-aligned decode workspace of pkv_decode_workspace_size bytes."""
    return _aligned_zeros(B.pkv_decode_workspace_size(desc, opts), device)


def mla_workspace_for(desc, device="cuda") -> torch.Tensor:
    """Zeroed, 256-byte-aligned MLA workspace of pkv_mla_workspace_size bytes."""
    return _aligned_zeros(B.pkv_mla_workspace_size(desc), device)


def paged_decode_attention(case: dict, dev: dict | None = None, opts=None, out=None, workspace=None,
                           stream=None) -> torch.Tensor:
    """Runs the full decode path on a synthetic case; returns out shaped like q
    ([B][Hq][D], or [B][q_len][Hq][D]) on the device."""
    dev = dev if dev is not None else upload_decode_case(case)
    desc = decode_desc(case)
    if out is None:
        out = torch.empty(case["q"].shape, dtype=TORCH_DTYPE[case["dtype"]], device=dev["q"].device)
    if workspace is None:
        workspace = workspace_for(desc, opts, device=dev["q"].device)
    B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                 dev["context_lens"], case["scale"], out, workspace, opts=opts, stream=stream)
    return out


def decode_partials(case: dict, dev: dict | None = None, opts=None, capacity: int | None = None):
    """Phase 1 alone; returns (P, NS, m, l, acc) as float64 numpy arrays with NS columns
    (leading dimensions those of q without D)."""
    dev = dev if dev is not None else upload_decode_case(case)
    desc = decode_desc(case)
    ns, P = B.pkv_plan_splits(desc, opts)
    cap = capacity if capacity is not None else ns
    d = dev["q"].device
    lead, D = tuple(case["q"].shape[:-1]), case["D"]
    acc = torch.full(lead + (cap, D), float("nan"), dtype=torch.float32, device=d)
    m = torch.full(lead + (cap,), float("nan"), dtype=torch.float32, device=d)
    l = torch.full(lead + (cap,), float("nan"), dtype=torch.float32, device=d)
    P2, ns2 = B.pkv_decode_partials(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                    dev["context_lens"], case["scale"], acc, m, l, cap, opts=opts)
    torch.cuda.synchronize()
    return P2, ns2, m.double().cpu().numpy(), l.double().cpu().numpy(), acc.double().cpu().numpy()


def mla_desc(case: dict, replay: bool = True) -> B.pkv_mla_desc:
    """The call's description; replay=True passes the longest kv_len as max_kv_len (S once per
    row tile, the second output half replayed from the first's softmax weights)."""
    kv = np.asarray(case["kv_indptr"], dtype=np.int64)
    max_kv = int(np.max(kv[1:] - kv[:-1], initial=0)) if replay else 0
    return B.make_mla_desc(case["total_q"], case["batch"], case["num_pages"], int(kv[-1]),
                           case["H"], case["Dc"], case["Dr"], max_kv_len=max_kv)


def upload_mla_case(case: dict, device="cuda") -> dict:
    bf = synth.BF16
    return dict(q_nope=bits_to_torch(case["q_nope"], bf, device), q_pe=bits_to_torch(case["q_pe"], bf, device),
                ckv_cache=bits_to_torch(case["ckv_cache"], bf, device),
                kpe_cache=bits_to_torch(case["kpe_cache"], bf, device),
                qo_indptr=int_to_torch(case["qo_indptr"], device), kv_indptr=int_to_torch(case["kv_indptr"], device),
                kv_indices=int_to_torch(case["kv_indices"], device))


def mla_paged_prefill(case: dict, dev: dict | None = None, out=None, lse=None, workspace=None, stream=None,
                      desc=None):
    """Runs the MLA prefill on a synthetic case; returns (out [T][H][Dc] bf16, lse [T][H] fp32) on the device."""
    dev = dev if dev is not None else upload_mla_case(case)
    d = dev["q_nope"].device
    T, H, Dc = case["total_q"], case["H"], case["Dc"]
    desc = desc if desc is not None else mla_desc(case)
    if out is None:
        out = torch.empty((T, H, Dc), dtype=torch.bfloat16, device=d)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=d)
    if workspace is None:
        workspace = mla_workspace_for(desc, device=d)
    B.pkv_mla_paged_prefill(desc, dev["q_nope"], dev["q_pe"], dev["ckv_cache"], dev["kpe_cache"],
                            dev["qo_indptr"], dev["kv_indptr"], dev["kv_indices"], case["sm_scale"], out, lse,
                            workspace, stream=stream)
    return out, lse
