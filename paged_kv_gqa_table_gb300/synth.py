"""Seeded synthetic inputs for paged decode attention and MLA paged prefill.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so the CUDA path and the CPU oracle can both be fed from
it.  Values are N(0, 1) float32 draws rounded to nearest-even into fp16 or bf16
bit patterns (uint16 arrays); context lengths are uniform integers (inclusive);
physical pages are a random permutation of the pool; block-table entries past
a sequence's last page are -1 (the "unallocated" marker of the flash-decode
post's block_table).  Every stream is derived from (seed, stream id, chunk),
so results do not depend on thread count or chunking.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

F16, BF16, FP8_E4M3 = 0, 1, 2
NHD, VLLM = 0, 1
NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0, FP8_E4M3: 0x7F}
_CHUNK = 1 << 24
_STREAM_LENS, _STREAM_PAGES, _STREAM_Q, _STREAM_K, _STREAM_V = 1, 2, 3, 4, 5
_STREAM_QPE, _STREAM_KPE = 6, 7


def _rng(seed: int, *ids: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *map(int, ids)])))


def f32_to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float32 values to nearest-even fp16 / bf16, returned as uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


# The 127 non-negative finite FP8 E4M3 values in bit order (0x00 .. 0x7E), as
# float64: exponent field e (bias 7) and 3 fraction bits f, e = 0 subnormal.
_E4M3_POS = np.array([(f / 8.0) * 2.0 ** -6 if (b >> 3) == 0 else (1 + f / 8.0) * 2.0 ** ((b >> 3) - 7)
                      for b in range(0x7F) for f in [b & 7]], dtype=np.float64)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round values to nearest-even FP8 E4M3 (saturating at +-448), as uint8 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), _E4M3_POS[-1])
    hi = np.clip(np.searchsorted(_E4M3_POS, a), 0, len(_E4M3_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return code | (np.signbit(x).astype(np.uint8) << 7)


def bits_to_f32(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Widen fp16 / bf16 bit patterns to float32 (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def normal_bits(seed: int, stream: int, n: int, dtype: int, threads: int = 8, fp8_scale: float = 1.0) -> np.ndarray:
    """n N(0,1) samples as fp16/bf16 bits (uint16), or as FP8 E4M3 bits (uint8) of
    sample / fp8_scale, drawn chunk by chunk from independent streams."""
    out = np.empty(n, dtype=np.uint8 if dtype == FP8_E4M3 else np.uint16)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        x = _rng(seed, stream, c).standard_normal(hi - lo, dtype=np.float32)
        if dtype == FP8_E4M3:
            out[lo:hi] = f32_to_e4m3_bits(x / np.float32(fp8_scale))
        else:
            out[lo:hi] = f32_to_bits(x, dtype)

    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(max(1, min(threads, nchunks))) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def assign_pages(seed: int, pages_per_seq: np.ndarray, max_blocks_per_seq: int, slack_pages: int = 0):
    """Random physical page ids for each sequence's logical blocks.

    Returns (block_table int32 [B][max_blocks_per_seq], num_blocks, unused page ids).
    """
    B = len(pages_per_seq)
    total = int(np.sum(pages_per_seq))
    nb = total + int(slack_pages)
    perm = _rng(seed, _STREAM_PAGES).permutation(nb).astype(np.int32)
    table = np.full((B, max_blocks_per_seq), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        p = int(pages_per_seq[b])
        table[b, :p] = perm[off:off + p]
        off += p
    return table, nb, perm[total:]


def decode_case(seed: int, B: int, Hq: int, Hkv: int, D: int, block_size: int, dtype: int,
                layout: int = NHD, context_lens=None, ctx_range=None, max_blocks_per_seq=None,
                slack_pages: int = 0, poison: bool = False, scale: float | None = None,
                x: int = 8, kv_dtype: int | None = None, k_scale: float = 1.0 / 16,
                v_scale: float = 1.0 / 16, q_len: int = 1) -> dict:
    """One paged GQA decode problem: q_len query tokens per sequence, the last
    q_len of its context (q [B][Hq][D] for one, [B][q_len][Hq][D] for several).

    Layouts: NHD k/v_cache [num_blocks][Hkv][block_size][D]; VLLM key_cache
    [num_blocks][Hkv][D/x][block_size][x], value_cache [num_blocks][Hkv][D][block_size].
    kv_dtype=FP8_E4M3 (NHD only) stores the caches as FP8 E4M3 bits of
    N(0,1) / k_scale and N(0,1) / v_scale (uint8); q stays fp16/bf16.
    poison=True writes NaN into every slot no query may read: the tail slots of
    each sequence's last page and all slack pages.
    """
    kv_dtype = dtype if kv_dtype is None else kv_dtype
    if context_lens is None:
        lo, hi = ctx_range
        context_lens = _rng(seed, _STREAM_LENS).integers(lo, hi + 1, size=B)
    ctx = np.asarray(context_lens, dtype=np.int32).reshape(B)
    pages = (ctx.astype(np.int64) + block_size - 1) // block_size
    mbps = int(max_blocks_per_seq) if max_blocks_per_seq is not None else int(max(1, pages.max(initial=1)))
    table, nb, unused = assign_pages(seed, pages, mbps, slack_pages)
    q = normal_bits(seed, _STREAM_Q, B * q_len * Hq * D, dtype)
    q = q.reshape(B, Hq, D) if q_len == 1 else q.reshape(B, q_len, Hq, D)
    n_kv = nb * Hkv * block_size * D
    k = normal_bits(seed, _STREAM_K, n_kv, kv_dtype, fp8_scale=k_scale)
    v = normal_bits(seed, _STREAM_V, n_kv, kv_dtype, fp8_scale=v_scale)
    if layout == NHD:
        k = k.reshape(nb, Hkv, block_size, D)
        v = v.reshape(nb, Hkv, block_size, D)
    else:
        k = k.reshape(nb, Hkv, D // x, block_size, x)
        v = v.reshape(nb, Hkv, D, block_size)
    case = dict(B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size, dtype=dtype, layout=layout, x=x,
                num_blocks=nb, q=q, k_cache=k, v_cache=v, block_table=table, context_lens=ctx,
                scale=float(scale if scale is not None else 1.0 / math.sqrt(D)), unused_pages=unused)
    if kv_dtype != dtype:
        case.update(kv_dtype=kv_dtype, k_scale=float(k_scale), v_scale=float(v_scale))
    if q_len != 1:
        case["q_len"] = int(q_len)
    if poison:
        poison_decode_case(case)
    return case


def poison_decode_case(case: dict) -> None:
    """Fill unread KV slots (last-page tails, unused pages) with NaN, in place."""
    nan = NAN_BITS[case.get("kv_dtype", case["dtype"])]
    BS, k, v = case["block_size"], case["k_cache"], case["v_cache"]
    vllm = case["layout"] == VLLM
    for p in case["unused_pages"]:
        k[p] = nan
        v[p] = nan
    for b, n in enumerate(case["context_lens"]):
        n = int(n)
        if n % BS == 0:
            continue
        p = case["block_table"][b, n // BS]
        o = n % BS
        if vllm:
            k[p, :, :, o:, :] = nan
            v[p, :, :, o:] = nan
        else:
            k[p, :, o:, :] = nan
            v[p, :, o:, :] = nan


def relabel_pages(case: dict, seed: int) -> dict:
    """Same logical problem with the physical pages permuted (pool and table rewritten)."""
    nb = case["num_blocks"]
    perm = _rng(seed, 99).permutation(nb)        # old page p moves to perm[p]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(nb)
    new = dict(case)
    new["k_cache"] = case["k_cache"][inv].copy()
    new["v_cache"] = case["v_cache"][inv].copy()
    t = case["block_table"]
    new["block_table"] = np.where(t >= 0, perm[np.maximum(t, 0)], -1).astype(np.int32)
    new["unused_pages"] = perm[case["unused_pages"]]
    return new


def mla_case(seed: int, batch: int, q_len_range, prefix_range, H: int = 16, Dc: int = 512,
             Dr: int = 64, sm_scale: float | None = None, q_lens=None, prefixes=None,
             slack_pages: int = 0, poison: bool = False) -> dict:
    """One MLA paged causal prefill problem with page_size 1 (bf16).

    Sequence b has q_len_b query tokens and kv_len_b = prefix_b + q_len_b cached
    rows; kv_indices lists a random permutation of the pool.
    """
    r = _rng(seed, _STREAM_LENS)
    if q_lens is None:
        q_lens = r.integers(q_len_range[0], q_len_range[1] + 1, size=batch)
    if prefixes is None:
        prefixes = r.integers(prefix_range[0], prefix_range[1] + 1, size=batch)
    q_lens = np.asarray(q_lens, dtype=np.int64).reshape(batch)
    prefixes = np.asarray(prefixes, dtype=np.int64).reshape(batch)
    kv_lens = q_lens + prefixes
    qo = np.zeros(batch + 1, dtype=np.int32)
    kvp = np.zeros(batch + 1, dtype=np.int32)
    qo[1:] = np.cumsum(q_lens)
    kvp[1:] = np.cumsum(kv_lens)
    nnz = int(kvp[-1])
    npages = nnz + int(slack_pages)
    perm = _rng(seed, _STREAM_PAGES).permutation(npages).astype(np.int32)
    kv_indices = perm[:nnz].copy()
    T = int(qo[-1])
    case = dict(
        batch=batch, H=H, Dc=Dc, Dr=Dr, total_q=T, num_pages=npages,
        q_nope=normal_bits(seed, _STREAM_Q, T * H * Dc, BF16).reshape(T, H, Dc),
        q_pe=normal_bits(seed, _STREAM_QPE, T * H * Dr, BF16).reshape(T, H, Dr),
        ckv_cache=normal_bits(seed, _STREAM_K, npages * Dc, BF16).reshape(npages, 1, Dc),
        kpe_cache=normal_bits(seed, _STREAM_KPE, npages * Dr, BF16).reshape(npages, 1, Dr),
        qo_indptr=qo, kv_indptr=kvp, kv_indices=kv_indices,
        sm_scale=float(sm_scale if sm_scale is not None else 1.0 / math.sqrt(192.0)),
        unused_pages=perm[nnz:],
    )
    if poison:
        for p in case["unused_pages"]:
            case["ckv_cache"][p] = NAN_BITS[BF16]
            case["kpe_cache"][p] = NAN_BITS[BF16]
    return case


# Named workloads (shapes and distributions of the pages' problem statement).
WORKLOADS = {
    "tiny": dict(B=2, Hq=4, Hkv=2, D=64, block_size=16, dtype=F16, layout=NHD,
                 context_lens=[37, 100], slack_pages=6, max_blocks_per_seq=8),
    "llama3_8b_decode": dict(B=64, Hq=32, Hkv=8, D=128, block_size=16, dtype=BF16, layout=NHD,
                             ctx_range=(1, 4096), max_blocks_per_seq=256),
    "long_context_decode": dict(B=4, Hq=32, Hkv=8, D=128, block_size=16, dtype=BF16, layout=NHD,
                                ctx_range=(32768, 131072), max_blocks_per_seq=8192),
    "gqa6_d256_vllm_decode": dict(B=128, Hq=24, Hkv=4, D=256, block_size=16, dtype=F16, layout=VLLM,
                                  ctx_range=(512, 8192), max_blocks_per_seq=512),
    # the Llama-3-8B-shaped step with an FP8 E4M3 KV cache (K, V = N(0,1) / 16 stored, scales 1/16)
    "llama3_8b_decode_fp8": dict(B=64, Hq=32, Hkv=8, D=128, block_size=16, dtype=BF16, layout=NHD,
                                 ctx_range=(1, 4096), max_blocks_per_seq=256, kv_dtype=FP8_E4M3),
    # the Llama-3-8B-shaped step verifying 4 tokens per sequence (speculative decoding: the last
    # 4 cached positions of each context are queries, bottom-right causal); same lengths and pages
    "llama3_8b_spec_decode_q4": dict(B=64, Hq=32, Hkv=8, D=128, block_size=16, dtype=BF16, layout=NHD,
                                     ctx_range=(1, 4096), max_blocks_per_seq=256, q_len=4),
}
MLA_WORKLOADS = {
    "mla_prefill_h16": dict(batch=8, q_len_range=(64, 512), prefix_range=(0, 2048)),
}


def kv_bytes(case: dict) -> int:
    """Algorithmic KV bytes of one decode step: live tokens x Hkv x D x (K and V) x element bytes
    (2 for fp16/bf16 caches, 1 for FP8 E4M3)."""
    e = 1 if case.get("kv_dtype", case["dtype"]) == FP8_E4M3 else 2
    return int(np.sum(case["context_lens"], dtype=np.int64)) * case["Hkv"] * case["D"] * 2 * e
