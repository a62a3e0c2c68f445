"""Pins for the fp64 oracle: each check comes from outside the oracle itself.

* widening of fp16/bf16 bits vs numpy's own conversions (all 65536 patterns);
* hand-derived closed-form cases (tests/golden/hand_cases.json);
* brute force: de-paged dense softmax attention written with numpy, and
  torch's CPU fp64 scaled_dot_product_attention (a library routine);
* invariants: page relabelling, poisoned unread slots, constant V, n = 1,
  identical K rows, q = 0, split-then-combine = unsplit;
* planted mistakes: mutated copies of oracle.c must fail the pins above.
"""
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from paged_kv_gqa_table_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def widen_np(bits, dtype):
    return synth.bits_to_f32(bits, dtype).astype(np.float64)


def depage_dense(case, b):
    """Dense K, V [n][Hkv][D] of sequence b, gathered with numpy reshapes."""
    n, BS, D, Hkv, dt = int(case["context_lens"][b]), case["block_size"], case["D"], case["Hkv"], case["dtype"]
    pages = case["block_table"][b, : (n + BS - 1) // BS]
    k = case["k_cache"][pages]
    v = case["v_cache"][pages]
    if case["layout"] == synth.VLLM:
        # [P][Hkv][D/x][BS][x] -> [P][BS][Hkv][D];  [P][Hkv][D][BS] -> [P][BS][Hkv][D]
        k = k.transpose(0, 3, 1, 2, 4).reshape(len(pages), BS, Hkv, D)
        v = v.transpose(0, 3, 1, 2)
    else:
        k = k.transpose(0, 2, 1, 3)
        v = v.transpose(0, 2, 1, 3)
    k = widen_np(k.reshape(-1, Hkv, D)[:n], dt)
    v = widen_np(v.reshape(-1, Hkv, D)[:n], dt)
    return k, v


def brute_force_decode(case):
    B, Hq, Hkv, D = case["B"], case["Hq"], case["Hkv"], case["D"]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    q = widen_np(case["q"], case["dtype"])
    for b in range(B):
        n = int(case["context_lens"][b])
        if n == 0:
            continue
        k, v = depage_dense(case, b)
        for h in range(Hq):
            s = case["scale"] * (k[:, h // G, :] @ q[b, h])
            w = np.exp(s - s.max())
            out[b, h] = (w / w.sum()) @ v[:, h // G, :]
    return out


SMALL_CASES = [
    dict(B=2, Hq=4, Hkv=2, D=64, block_size=16, dtype=synth.F16, layout=synth.NHD,
         context_lens=[37, 100], slack_pages=6, max_blocks_per_seq=8),
    dict(B=3, Hq=6, Hkv=1, D=16, block_size=4, dtype=synth.BF16, layout=synth.NHD,
         context_lens=[0, 1, 9], slack_pages=2),
    dict(B=3, Hq=6, Hkv=2, D=16, block_size=4, dtype=synth.F16, layout=synth.VLLM,
         context_lens=[5, 12, 3], slack_pages=3),
    dict(B=2, Hq=3, Hkv=3, D=8, block_size=2, dtype=synth.BF16, layout=synth.VLLM,
         context_lens=[7, 4]),
]


def test_widen_fp16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.widen(b, oracle.F16) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_widen_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([oracle.widen(int(b), oracle.BF16) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_widen_e4m3_all_patterns():
    # FP8 E4M3 ("e4m3fn"): against torch's float8_e4m3fn conversion.
    torch = pytest.importorskip("torch")
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.widen8(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def _fp8_case(seed, **kw):
    base = dict(B=4, Hq=8, Hkv=2, D=32, block_size=16, dtype=synth.BF16, ctx_range=(1, 70),
                kv_dtype=synth.FP8_E4M3, k_scale=1.0 / 16, v_scale=1.0 / 16, slack_pages=3)
    base.update(kw)
    return synth.decode_case(seed=seed, **base)


def _fp8_as_bf16(case):
    """The same problem with the caches rewritten as bf16 bits of scale * fp8 value
    (exact: E4M3 values times a power of two fit bf16), via torch's conversions."""
    torch = pytest.importorskip("torch")
    def conv(bits, sc):
        v = torch.from_numpy(np.ascontiguousarray(bits)).view(torch.float8_e4m3fn).to(torch.float32) * sc
        return v.to(torch.bfloat16).view(torch.uint16).numpy().astype(np.uint16)
    new = {k: v for k, v in case.items() if k not in ("kv_dtype", "k_scale", "v_scale")}
    new["k_cache"] = conv(case["k_cache"], case["k_scale"])
    new["v_cache"] = conv(case["v_cache"], case["v_scale"])
    return new


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fp8_cache_decode_equals_bf16_decode_of_the_same_values(seed):
    case = _fp8_case(seed)
    got = oracle.decode(case)
    ref = oracle.decode(_fp8_as_bf16(case))
    assert np.array_equal(got, ref)
    P = 32
    NS = -(-int(case["context_lens"].max()) // P)
    for a, b in zip(oracle.decode_partials(case, P, NS), oracle.decode_partials(_fp8_as_bf16(case), P, NS)):
        assert np.array_equal(a, b)


def test_fp8_scales_act_as_stated():
    # k_scale multiplies every score, v_scale the output (closed forms).
    a = _fp8_case(5)
    b = dict(a, k_scale=a["k_scale"] * 2.0)
    c = dict(a, scale=a["scale"] * 2.0)
    assert np.allclose(oracle.decode(b), oracle.decode(c), rtol=1e-12, atol=1e-14)
    d = dict(a, v_scale=a["v_scale"] * 3.0)
    assert np.allclose(oracle.decode(d), 3.0 * oracle.decode(a), rtol=1e-12, atol=1e-14)


def _golden_scale(s):
    return {"ln3": math.log(3.0), "ln2/2": math.log(2.0) / 2, "ln2": math.log(2.0)}[s] if isinstance(s, str) else s


def _golden_decode_case(g):
    B, Hq, Hkv, D, BS, NB = g["B"], g["Hq"], g["Hkv"], g["D"], g["block_size"], g["num_blocks"]
    k = np.full((NB, Hkv, BS, D), 7.0, np.float32)
    v = np.full((NB, Hkv, BS, D), 7.0, np.float32)
    for p, rows in g["page_tokens"].items():
        k[int(p), 0] = rows["K"]
        v[int(p), 0] = rows["V"]
    enc = lambda a: synth.f32_to_bits(np.asarray(a, np.float32), synth.F16)
    return dict(B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=BS, dtype=synth.F16, layout=synth.NHD, x=8,
                num_blocks=NB, q=enc(g["q"]).reshape(B, Hq, D), k_cache=enc(k), v_cache=enc(v),
                block_table=np.array(g["block_table"], np.int32), context_lens=np.array(g["context_lens"], np.int32),
                scale=_golden_scale(g["scale"]))


@pytest.mark.parametrize("name", ["decode_two_tokens", "decode_gqa_two_heads"])
def test_golden_decode(name):
    g = json.load(open(GOLDEN))[name]
    case = _golden_decode_case(g)
    out = oracle.decode(case)
    np.testing.assert_allclose(out.reshape(-1, case["D"]), np.array(g["out"]), rtol=0, atol=1e-14)
    if "split_P" in g:
        pm, pl, pacc = oracle.decode_partials(case, g["split_P"], 2)
        ref_m = [_golden_scale(x) for x in g["partials"]["m"]]
        np.testing.assert_allclose(pm.reshape(-1), ref_m, atol=1e-15)
        np.testing.assert_allclose(pl.reshape(-1), g["partials"]["l"], atol=1e-15)
        np.testing.assert_allclose(pacc.reshape(2, -1), g["partials"]["acc"], atol=1e-15)
        np.testing.assert_allclose(oracle.combine(case["context_lens"], pm, pl, pacc).reshape(-1, case["D"]),
                                   np.array(g["out"]), atol=1e-14)


def test_golden_mla():
    g = json.load(open(GOLDEN))["mla_causal_two_queries"]
    NP, Dc, Dr = g["num_pages"], g["Dc"], g["Dr"]
    ckv = np.full((NP, 1, Dc), 5.0, np.float32)
    kpe = np.full((NP, 1, Dr), 5.0, np.float32)
    for p, r in g["rows"].items():
        ckv[int(p), 0] = r["ckv"]
        kpe[int(p), 0] = r["kpe"]
    enc = lambda a: synth.f32_to_bits(np.asarray(a, np.float32), synth.BF16)
    case = dict(q_nope=enc(g["q_nope"]), q_pe=enc(g["q_pe"]), ckv_cache=enc(ckv), kpe_cache=enc(kpe),
                qo_indptr=np.array(g["qo_indptr"]), kv_indptr=np.array(g["kv_indptr"]),
                kv_indices=np.array(g["kv_indices"]), sm_scale=_golden_scale(g["sm_scale"]))
    out, lse = oracle.mla(case)
    np.testing.assert_allclose(out, np.array(g["out"]), atol=1e-14)
    np.testing.assert_allclose(lse, np.array(g["lse"]), atol=1e-14)


@pytest.mark.parametrize("idx", range(len(SMALL_CASES)))
def test_decode_vs_numpy_brute_force(idx):
    case = synth.decode_case(seed=idx, **SMALL_CASES[idx])
    np.testing.assert_allclose(oracle.decode(case), brute_force_decode(case), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("idx", range(len(SMALL_CASES)))
def test_decode_vs_torch_sdpa(idx):
    torch = pytest.importorskip("torch")
    case = synth.decode_case(seed=100 + idx, **SMALL_CASES[idx])
    G = case["Hq"] // case["Hkv"]
    q = widen_np(case["q"], case["dtype"])
    ref = np.zeros((case["B"], case["Hq"], case["D"]))
    for b in range(case["B"]):
        if case["context_lens"][b] == 0:
            continue
        k, v = depage_dense(case, b)
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)   # [Hq][n][D]
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
        qt = torch.from_numpy(q[b]).unsqueeze(1)                              # [Hq][1][D]
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=case["scale"])
        ref[b] = o[:, 0, :].numpy()
    np.testing.assert_allclose(oracle.decode(case), ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_alibi_decode_vs_torch_sdpa_with_additive_mask(idx):
    # ALiBi as the additive float mask slope_h * (t - (n - 1)) of torch's SDPA.
    torch = pytest.importorskip("torch")
    case = synth.decode_case(seed=200 + idx, **SMALL_CASES[idx])
    slopes = np.float32(2.0) ** -np.arange(1, case["Hq"] + 1, dtype=np.float32) * np.float32(3.0)
    case["alibi_slopes"] = slopes
    G = case["Hq"] // case["Hkv"]
    q = widen_np(case["q"], case["dtype"])
    ref = np.zeros((case["B"], case["Hq"], case["D"]))
    for b in range(case["B"]):
        n = int(case["context_lens"][b])
        if n == 0:
            continue
        k, v = depage_dense(case, b)
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
        qt = torch.from_numpy(q[b]).unsqueeze(1)
        bias = torch.from_numpy(slopes.astype(np.float64))[:, None, None] * (torch.arange(n, dtype=torch.float64) - (n - 1))
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=bias, scale=case["scale"])
        ref[b] = o[:, 0, :].numpy()
    np.testing.assert_allclose(oracle.decode(case), ref, rtol=1e-10, atol=1e-12)


def test_alibi_geometric_closed_form():
    # q = 0 leaves only the bias: weights rho^j over distances j = n-1-t with
    # rho = e^-s.  With V_t = t (every element), out = (n-1) - E[j], and
    # E[j] = rho (1 - n rho^(n-1) + (n-1) rho^n) / ((1 - rho)(1 - rho^n)).
    n_list = [1, 2, 5, 37, 100]
    case = synth.decode_case(seed=3, B=len(n_list), Hq=2, Hkv=1, D=16, block_size=16, dtype=synth.BF16,
                             context_lens=n_list)
    case["q"] = np.zeros_like(case["q"])
    v = np.zeros(case["v_cache"].shape, np.float32)
    for b, n in enumerate(n_list):
        for t in range(n):
            v[case["block_table"][b, t // 16], 0, t % 16, :] = t
    case["v_cache"] = synth.f32_to_bits(v, synth.BF16).reshape(case["v_cache"].shape)
    s_h = [0.25, 1.5]
    case["alibi_slopes"] = np.array(s_h, np.float32)
    out = oracle.decode(case)
    for b, n in enumerate(n_list):
        for h, sl in enumerate(s_h):
            rho = math.exp(-sl)
            ej = 0.0 if n == 1 else rho * (1 - n * rho ** (n - 1) + (n - 1) * rho ** n) / ((1 - rho) * (1 - rho ** n))
            np.testing.assert_allclose(out[b, h], (n - 1) - ej, rtol=1e-12, atol=1e-12)


def test_relabel_pages_is_bit_identical():
    case = synth.decode_case(seed=7, **SMALL_CASES[2])
    moved = synth.relabel_pages(case, seed=3)
    assert not np.array_equal(moved["block_table"], case["block_table"])
    assert np.array_equal(oracle.decode(case), oracle.decode(moved))


@pytest.mark.parametrize("idx", [0, 2])
def test_poisoned_unread_slots_change_nothing(idx):
    clean = synth.decode_case(seed=11, **SMALL_CASES[idx])
    dirty = synth.decode_case(seed=11, poison=True, **SMALL_CASES[idx])
    assert np.array_equal(oracle.decode(clean), oracle.decode(dirty))


def _with_values(case, k=None, v=None, q=None):
    c = dict(case)
    if k is not None:
        c["k_cache"] = np.full_like(case["k_cache"], k)
    if v is not None:
        c["v_cache"] = np.full_like(case["v_cache"], v)
    if q is not None:
        c["q"] = np.full_like(case["q"], q)
    return c


def test_constant_v_rows_give_the_constant():
    case = synth.decode_case(seed=1, **SMALL_CASES[0])
    c = _with_values(case, v=0x4500)          # fp16 5.0
    out = oracle.decode(c)
    np.testing.assert_allclose(out, 5.0, rtol=1e-15)


def test_identical_k_rows_and_zero_q_give_mean_v():
    case = synth.decode_case(seed=2, **SMALL_CASES[2])
    for c in (_with_values(case, k=0x3C00), _with_values(case, q=0)):
        out = oracle.decode(c)
        for b in range(case["B"]):
            n = int(case["context_lens"][b])
            _, v = depage_dense(case, b)
            G = case["Hq"] // case["Hkv"]
            for h in range(case["Hq"]):
                np.testing.assert_allclose(out[b, h], v[:, h // G, :].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_context_len_one_gives_first_v_row():
    case = synth.decode_case(seed=5, **dict(SMALL_CASES[1], context_lens=[1, 1, 1]))
    out = oracle.decode(case)
    G = case["Hq"] // case["Hkv"]
    for b in range(case["B"]):
        _, v = depage_dense(case, b)
        for h in range(case["Hq"]):
            assert np.array_equal(out[b, h], v[0, h // G])


def test_empty_context_gives_zeros():
    case = synth.decode_case(seed=5, **dict(SMALL_CASES[1], context_lens=[0, 3, 0]))
    out = oracle.decode(case)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)


@pytest.mark.parametrize("P", [4, 8, 28, 512])
def test_split_then_combine_equals_unsplit(P):
    case = synth.decode_case(seed=9, **dict(SMALL_CASES[1], context_lens=[0, 1, 37],
                                            max_blocks_per_seq=10))
    NS = max(1, -(-37 // P)) + 2            # two always-empty splits at the end
    pm, pl, pacc = oracle.decode_partials(case, P, NS)
    for b in range(case["B"]):
        n = int(case["context_lens"][b])
        for s in range(NS):
            if s * P >= n:
                assert np.all(pm[b, :, s] == -np.inf) and np.all(pl[b, :, s] == 0)
                assert np.all(pacc[b, :, s] == 0)
    np.testing.assert_allclose(oracle.combine(case["context_lens"], pm, pl, pacc), oracle.decode(case),
                               rtol=1e-12, atol=1e-14)


def test_bad_table_and_bad_shapes_are_rejected():
    case = synth.decode_case(seed=3, **SMALL_CASES[0])
    bad = dict(case)
    bad["block_table"] = case["block_table"].copy()
    bad["block_table"][1, 2] = -1                        # inside the live range of sequence 1
    with pytest.raises(oracle.OracleError) as e:
        oracle.decode(bad)
    assert e.value.status == oracle.STATUS_BAD_TABLE
    bad["block_table"] = case["block_table"].copy()
    bad["block_table"][0, 0] = case["num_blocks"]        # past the pool
    with pytest.raises(oracle.OracleError):
        oracle.decode(bad)
    long_ctx = dict(case, context_lens=np.array([37, 8 * 16 + 1], np.int32))
    with pytest.raises(oracle.OracleError) as e:
        oracle.decode(long_ctx)
    assert e.value.status == oracle.STATUS_INVALID
    with pytest.raises(oracle.OracleError):
        oracle.decode(dict(case, Hkv=3))
    # entries past the live range are never read, whatever their value
    ok = dict(case)
    ok["block_table"] = case["block_table"].copy()
    ok["block_table"][0, 5:] = 12345
    assert np.array_equal(oracle.decode(ok), oracle.decode(case))


# ------------------------------------------------- multi-token decode ----
#
# q_len query tokens per sequence are its last q_len positions: query i sits at
# pos = n - q_len + i and sees keys t <= pos (the MLA page's bottom-right causal
# rule on the decode cache layouts); an empty window gives a zero row.

MT_CASES = [
    dict(B=4, Hq=4, Hkv=2, D=16, block_size=4, dtype=synth.F16, layout=synth.NHD, q_len=3,
         context_lens=[0, 2, 3, 13], slack_pages=2),
    dict(B=3, Hq=6, Hkv=2, D=16, block_size=4, dtype=synth.BF16, layout=synth.VLLM, q_len=5,
         context_lens=[5, 12, 9]),
    dict(B=2, Hq=3, Hkv=1, D=8, block_size=2, dtype=synth.BF16, layout=synth.NHD, q_len=2,
         context_lens=[7, 1], kv_dtype=synth.FP8_E4M3),
]


def _dense_q(case):
    """Queries as fp64 [B][q_len][Hq][D]."""
    q = widen_np(case["q"], case["dtype"])
    return q.reshape(case["B"], case.get("q_len", 1), case["Hq"], case["D"])


def _dense_kv(case, b):
    """Dense K, V [n][Hkv][D] of sequence b for 16-bit or FP8 caches (scales applied)."""
    if case.get("kv_dtype", case["dtype"]) == synth.FP8_E4M3:
        c = _fp8_as_bf16(case)
        return depage_dense(c, b)
    return depage_dense(case, b)


def brute_force_multi_token(case, P=None, NS=None):
    """numpy restatement: output [B][q_len][Hq][D]; with P, NS also the split
    partials (m, l, acc) of each query's window cut into [s*P, (s+1)*P)."""
    B, Hq, Hkv, D = case["B"], case["Hq"], case["Hkv"], case["D"]
    ql, G = case.get("q_len", 1), Hq // Hkv
    slopes = case.get("alibi_slopes")
    q = _dense_q(case)
    out = np.zeros((B, ql, Hq, D))
    parts = None
    if P is not None:
        parts = (np.full((B, ql, Hq, NS), -np.inf), np.zeros((B, ql, Hq, NS)), np.zeros((B, ql, Hq, NS, D)))
    for b in range(B):
        n = int(case["context_lens"][b])
        if n == 0:
            continue
        k, v = _dense_kv(case, b)
        for i in range(ql):
            pos = n - ql + i
            if pos < 0:
                continue
            t = np.arange(pos + 1)
            for h in range(Hq):
                s = case["scale"] * (k[: pos + 1, h // G, :] @ q[b, i, h])
                if slopes is not None:
                    s = s + float(slopes[h]) * (t - pos)
                w = np.exp(s - s.max())
                out[b, i, h] = (w / w.sum()) @ v[: pos + 1, h // G, :]
                if parts is not None:
                    for sp in range(NS):
                        sel = (t >= sp * P) & (t < (sp + 1) * P)
                        if sel.any():
                            m = s[sel].max()
                            e = np.exp(s[sel] - m)
                            parts[0][b, i, h, sp] = m
                            parts[1][b, i, h, sp] = e.sum()
                            parts[2][b, i, h, sp] = e @ v[: pos + 1][sel][:, h // G, :]
    return out, parts


@pytest.mark.parametrize("idx", range(len(MT_CASES)))
def test_multi_token_decode_vs_numpy_brute_force(idx):
    case = synth.decode_case(seed=300 + idx, **MT_CASES[idx])
    assert case["q"].shape == (case["B"], case["q_len"], case["Hq"], case["D"])
    np.testing.assert_allclose(oracle.decode(case), brute_force_multi_token(case)[0], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("idx", range(len(MT_CASES)))
def test_multi_token_decode_vs_torch_sdpa_bottom_right_mask(idx):
    # torch's is_causal is top-left aligned when q_len != n, so the mask is
    # spelled out: query i may see key t iff t <= n - q_len + i.
    torch = pytest.importorskip("torch")
    case = synth.decode_case(seed=310 + idx, **MT_CASES[idx])
    ql, G = case["q_len"], case["Hq"] // case["Hkv"]
    q = _dense_q(case)
    ref = np.zeros_like(q)
    for b in range(case["B"]):
        n = int(case["context_lens"][b])
        if n == 0:
            continue
        k, v = _dense_kv(case, b)
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)     # [Hq][n][D]
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
        qt = torch.from_numpy(q[b]).permute(1, 0, 2)                              # [Hq][q_len][D]
        allowed = torch.arange(n)[None, :] <= (n - ql + torch.arange(ql))[:, None]  # [q_len][n]
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=allowed, scale=case["scale"])
        o = o.permute(1, 0, 2).numpy().copy()
        o[~allowed.any(dim=1).numpy()] = 0.0                                       # empty windows: zero rows
        ref[b] = o
    np.testing.assert_allclose(oracle.decode(case), ref, rtol=1e-10, atol=1e-12)


def test_multi_token_alibi_vs_torch_sdpa_with_additive_mask():
    torch = pytest.importorskip("torch")
    case = synth.decode_case(seed=320, **MT_CASES[1])
    slopes = np.float32(2.0) ** -np.arange(1, case["Hq"] + 1, dtype=np.float32) * np.float32(5.0)
    case["alibi_slopes"] = slopes
    ql, G = case["q_len"], case["Hq"] // case["Hkv"]
    q = _dense_q(case)
    ref = np.zeros_like(q)
    for b in range(case["B"]):
        n = int(case["context_lens"][b])
        k, v = _dense_kv(case, b)
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
        qt = torch.from_numpy(q[b]).permute(1, 0, 2)
        rel = torch.arange(n, dtype=torch.float64)[None, :] - (n - ql + torch.arange(ql, dtype=torch.float64))[:, None]
        bias = torch.from_numpy(slopes.astype(np.float64))[:, None, None] * rel            # [Hq][q_len][n]
        bias = bias.masked_fill(rel > 0, -math.inf)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=bias, scale=case["scale"])
        ref[b] = o.permute(1, 0, 2).numpy()
    np.testing.assert_allclose(oracle.decode(case), ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("idx", range(len(MT_CASES)))
def test_each_query_token_equals_plain_decode_of_its_prefix(idx):
    # Query i of a q_len case is the one-token decode of the first n - q_len + i + 1 tokens.
    case = synth.decode_case(seed=330 + idx, **MT_CASES[idx])
    out = oracle.decode(case)
    ql = case["q_len"]
    for i in range(ql):
        single = dict(case, q=np.ascontiguousarray(case["q"][:, i]),
                      context_lens=np.maximum(case["context_lens"] - ql + i + 1, 0).astype(np.int32))
        single.pop("q_len")
        assert np.array_equal(out[:, i], oracle.decode(single))


@pytest.mark.parametrize("P", [2, 4, 8])
def test_multi_token_partials_vs_numpy_brute_force(P):
    # Fixes ALiBi's reference point in m: the bias is zero at each query's own position.
    case = synth.decode_case(seed=340, **MT_CASES[0])
    case["alibi_slopes"] = np.array([0.5, 0.25, 1.0, 2.0], np.float32)
    NS = -(-13 // P) + 1
    pm, pl, pacc = oracle.decode_partials(case, P, NS)
    _, (bm, bl, bacc) = brute_force_multi_token(case, P, NS)
    assert np.array_equal(pm == -np.inf, bm == -np.inf)
    fin = bm > -np.inf
    np.testing.assert_allclose(pm[fin], bm[fin], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(pl, bl, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(pacc, bacc, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("P", [2, 4, 8, 16])
@pytest.mark.parametrize("idx", [0, 1])
def test_multi_token_split_then_combine_equals_unsplit(P, idx):
    # case 0 holds sequences shorter than q_len (empty windows, all-sentinel rows)
    case = synth.decode_case(seed=350, **MT_CASES[idx])
    NS = -(-int(case["context_lens"].max()) // P) + 1
    pm, pl, pacc = oracle.decode_partials(case, P, NS)
    np.testing.assert_allclose(oracle.combine(case["context_lens"], pm, pl, pacc), oracle.decode(case),
                               rtol=1e-12, atol=1e-14)


def test_multi_token_rejects_bad_q_len():
    case = synth.decode_case(seed=360, **MT_CASES[0])
    with pytest.raises(oracle.OracleError) as e:
        oracle.decode(dict(case, q_len=0, q=case["q"][:, :0]))
    assert e.value.status == oracle.STATUS_INVALID


# ---------------------------------------------------------------- MLA ----

MLA_SMALL = [
    dict(batch=3, q_len_range=(1, 5), prefix_range=(0, 7), H=2, Dc=16, Dr=8, slack_pages=3),
    dict(batch=2, q_len_range=(1, 1), prefix_range=(3, 9), H=3, Dc=8, Dr=4),
    dict(batch=2, q_len_range=(4, 9), prefix_range=(0, 0), H=2, Dc=8, Dr=8, sm_scale=1.0),
]


def brute_force_mla(case):
    qn = widen_np(case["q_nope"], synth.BF16)
    qp = widen_np(case["q_pe"], synth.BF16)
    ckv = widen_np(case["ckv_cache"], synth.BF16)[:, 0, :]
    kpe = widen_np(case["kpe_cache"], synth.BF16)[:, 0, :]
    qo, kvp, kvi = case["qo_indptr"], case["kv_indptr"], case["kv_indices"]
    T, H, Dc = qn.shape
    out = np.zeros((T, H, Dc))
    lse = np.full((T, H), -np.inf)
    for b in range(len(qo) - 1):
        rows = kvi[kvp[b]:kvp[b + 1]]
        K = np.concatenate([ckv[rows], kpe[rows]], axis=1)
        q_len, kv_len = qo[b + 1] - qo[b], kvp[b + 1] - kvp[b]
        for i in range(q_len):
            t = qo[b] + i
            vis = np.arange(kv_len) <= (kv_len - q_len) + i
            Q = np.concatenate([qn[t], qp[t]], axis=1)           # [H][Dc+Dr]
            logits = case["sm_scale"] * (Q @ K.T)                 # [H][kv_len]
            logits[:, ~vis] = -np.inf
            mx = logits.max(axis=1, keepdims=True)
            w = np.exp(logits - mx)
            out[t] = (w / w.sum(axis=1, keepdims=True)) @ ckv[rows]
            lse[t] = np.log2(np.exp(logits).sum(axis=1))
    return out, lse


@pytest.mark.parametrize("idx", range(len(MLA_SMALL)))
def test_mla_vs_numpy_brute_force(idx):
    case = synth.mla_case(seed=idx, **MLA_SMALL[idx])
    out, lse = oracle.mla(case)
    ref_out, ref_lse = brute_force_mla(case)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("idx", range(len(MLA_SMALL)))
def test_mla_vs_torch_sdpa_causal_mqa(idx):
    """MLA is causal MQA with K = [ckv; kpe], Q = [q_nope; q_pe] and V = ckv."""
    torch = pytest.importorskip("torch")
    case = synth.mla_case(seed=50 + idx, **MLA_SMALL[idx])
    qn = torch.from_numpy(widen_np(case["q_nope"], synth.BF16))
    qp = torch.from_numpy(widen_np(case["q_pe"], synth.BF16))
    ckv = torch.from_numpy(widen_np(case["ckv_cache"], synth.BF16))[:, 0]
    kpe = torch.from_numpy(widen_np(case["kpe_cache"], synth.BF16))[:, 0]
    qo, kvp, kvi = case["qo_indptr"], case["kv_indptr"], torch.from_numpy(case["kv_indices"].astype(np.int64))
    out, _ = oracle.mla(case)
    for b in range(len(qo) - 1):
        rows = kvi[kvp[b]:kvp[b + 1]]
        K = torch.cat([ckv[rows], kpe[rows]], dim=1)[None]                 # [1][kv][576]
        V = ckv[rows][None]
        Q = torch.cat([qn[qo[b]:qo[b + 1]], qp[qo[b]:qo[b + 1]]], dim=2).permute(1, 0, 2)  # [H][q][Dq]
        q_len, kv_len = qo[b + 1] - qo[b], kvp[b + 1] - kvp[b]
        mask = torch.arange(kv_len)[None, :] <= (kv_len - q_len) + torch.arange(q_len)[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(Q, K.expand(Q.shape[0], -1, -1),
                                                             V.expand(Q.shape[0], -1, -1),
                                                             attn_mask=mask, scale=case["sm_scale"])
        np.testing.assert_allclose(out[qo[b]:qo[b + 1]], o.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_mla_zero_query_gives_uniform_weights():
    case = synth.mla_case(seed=4, **MLA_SMALL[0])
    case["q_nope"] = np.zeros_like(case["q_nope"])
    case["q_pe"] = np.zeros_like(case["q_pe"])
    out, lse = oracle.mla(case)
    ckv = widen_np(case["ckv_cache"], synth.BF16)[:, 0, :]
    qo, kvp, kvi = case["qo_indptr"], case["kv_indptr"], case["kv_indices"]
    for b in range(len(qo) - 1):
        q_len, kv_len = qo[b + 1] - qo[b], kvp[b + 1] - kvp[b]
        for i in range(q_len):
            cnt = kv_len - q_len + i + 1
            np.testing.assert_allclose(lse[qo[b] + i], np.log2(cnt), atol=1e-14)
            np.testing.assert_allclose(out[qo[b] + i], np.broadcast_to(ckv[kvi[kvp[b]:kvp[b] + cnt]].mean(0),
                                                                        out[qo[b] + i].shape), rtol=1e-12, atol=1e-14)


def test_mla_lse_normalises_the_weights():
    case = synth.mla_case(seed=6, **MLA_SMALL[0])
    _, lse = oracle.mla(case)
    qn = widen_np(case["q_nope"], synth.BF16)
    qp = widen_np(case["q_pe"], synth.BF16)
    ckv = widen_np(case["ckv_cache"], synth.BF16)[:, 0, :]
    kpe = widen_np(case["kpe_cache"], synth.BF16)[:, 0, :]
    qo, kvp, kvi = case["qo_indptr"], case["kv_indptr"], case["kv_indices"]
    for b in range(len(qo) - 1):
        q_len, kv_len = qo[b + 1] - qo[b], kvp[b + 1] - kvp[b]
        for i in range(q_len):
            t = qo[b] + i
            rows = kvi[kvp[b]:kvp[b] + kv_len - q_len + i + 1]
            logit = case["sm_scale"] * (qn[t] @ ckv[rows].T + qp[t] @ kpe[rows].T)
            np.testing.assert_allclose(np.sum(2.0 ** (logit * math.log2(math.e) - lse[t][:, None]), axis=1), 1.0,
                                       atol=1e-12)


def test_mla_empty_kv_and_bad_indices():
    case = synth.mla_case(seed=8, batch=2, q_len_range=(2, 2), prefix_range=(0, 0), H=2, Dc=8, Dr=4,
                          q_lens=[2, 0], prefixes=[1, 0])
    out, lse = oracle.mla(case)
    assert np.all(np.isfinite(lse))
    # a sequence with kv_len = 0 but q_len > 0: zeros and -inf
    c2 = dict(case, kv_indptr=np.array([0, 3, 3], np.int32), qo_indptr=np.array([0, 1, 2], np.int32))
    out, lse = oracle.mla(c2)
    assert np.all(out[1] == 0) and np.all(lse[1] == -np.inf)
    bad = dict(case, kv_indices=case["kv_indices"].copy())
    bad["kv_indices"][0] = case["num_pages"]
    with pytest.raises(oracle.OracleError) as e:
        oracle.mla(bad)
    assert e.value.status == oracle.STATUS_BAD_TABLE


# ------------------------------------------------------- planted mistakes ----

MUTANTS = [
    ("grouping", "int g = h / G;", "int g = h % a->Hkv;"),
    ("scale dropped", "return a->scale * s;", "return s;"),
    ("vllm x-pack swapped", "* BS + o) * x + d % x;", "* BS + o) * x + d / x % x;"),
    ("vllm value transposed", "* D + d) * BS + o;", "* BS + o) * D + d;"),
    ("combine weight dropped", "L += f * l[s];", "L += l[s];"),
    ("max not subtracted", "double w = exp(sbuf[t - t0] - m);", "double w = exp(sbuf[t - t0]);"),
    ("causal top-left", "int pos = (kv_len - q_len) + (t - qo_indptr[b]);", "int pos = (t - qo_indptr[b]);"),
    ("lse natural log", "lse[(size_t)t * H + h] = (m + log(z)) / log(2.0);", "lse[(size_t)t * H + h] = (m + log(z));"),
    ("kpe term dropped", "s += bf16_bits_to_double(qp[d])", "s += 0 * bf16_bits_to_double(qp[d])"),
    ("bf16 exponent bias", "v = ldexp((double)(f + 128), e - 134);", "v = ldexp((double)(f + 128), e - 133);"),
    ("e4m3 exponent bias", "v = ldexp((double)(f + 8), e - 10);", "v = ldexp((double)(f + 8), e - 9);"),
    ("e4m3 subnormal scale", "v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    ("fp8 k_scale dropped", "cache_value(a, a->k, k_index(a->layout, a->Hkv, a->BS, a->D, a->x, p, g, o, d), a->k_scale)",
     "cache_value(a, a->k, k_index(a->layout, a->Hkv, a->BS, a->D, a->x, p, g, o, d), 1.0)"),
    ("fp8 v_scale dropped", "a->v_scale);\n}", "1.0);\n}"),
    ("alibi sign flipped", "a->alibi[h] * (double)(t - pos);", "a->alibi[h] * (double)(pos - t);"),
    ("alibi dropped", "if (a->alibi) sbuf[t - t0] += a->alibi[h] * (double)(t - pos);", "(void)pos;"),
    ("alibi from the last position", "int pos = seq_len(a, b) - a->q_len + i;", "int pos = seq_len(a, b) - 1;"),
    ("decode window one short", "return n - q_len + i + 1;", "return n - q_len + i;"),
    ("decode window top-left", "return n - q_len + i + 1;", "return i + 1;"),
    ("query token ignored", "(((size_t)b * a->q_len + i) * a->Hq + h) * a->D + d]",
     "(((size_t)b * a->q_len + 0) * a->Hq + h) * a->D + d]"),
    ("combine window ignored", "if (window_end(ctx[b], q_len, i) <= 0) {", "if (ctx[b] == 0) {"),
]


def _mutant(tmp_path, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(old) == 1, old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "mutant.so"
    subprocess.check_call(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-o", str(so), str(path), "-lm"])
    return str(so)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistakes_are_caught(tmp_path, monkeypatch, name, old, new):
    so = _mutant(tmp_path, old, new)
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "build", lambda force=False: so)
    failures = 0
    for fn in (lambda: test_decode_vs_numpy_brute_force(2), lambda: test_decode_vs_numpy_brute_force(0),
               lambda: test_split_then_combine_equals_unsplit(8), lambda: test_mla_vs_numpy_brute_force(0),
               test_widen_bf16_all_patterns, test_widen_e4m3_all_patterns,
               lambda: test_fp8_cache_decode_equals_bf16_decode_of_the_same_values(0),
               test_alibi_geometric_closed_form, lambda: test_multi_token_decode_vs_numpy_brute_force(0),
               lambda: test_multi_token_partials_vs_numpy_brute_force(4),
               lambda: test_multi_token_split_then_combine_equals_unsplit(4, 0)):
        try:
            fn()
        except (AssertionError, oracle.OracleError):
            failures += 1
    monkeypatch.setattr(oracle, "_lib", None)
    assert failures > 0, "mutant %r passed every pin" % name
