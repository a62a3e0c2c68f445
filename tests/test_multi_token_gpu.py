"""GPU parity of multi-token (speculative) paged decode against the fp64 oracle.

q_len query tokens per sequence are its last q_len cached positions: token i
sits at n - q_len + i and attends keys up to its own position (the MLA page's
bottom-right causal rule on the decode cache layouts); an empty window gives a
zero row.  Every call goes through the C ABI; tolerances are the decode bars
(max |diff| <= 4e-3 fp16, <= 1.6e-2 bf16; partial LSE within 1e-3).

The cases cover one and several row tiles (G * q_len query rows, 16 per CTA,
8 for D = 256), both cache layouts and FP8 caches, windows that end inside a
page, inside a split and before the context starts (n < q_len), and groups of
any size at q_len = 1.
"""
import numpy as np
import pytest

import oracle
from paged_kv_gqa_table_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TOL = {synth.F16: 4e-3, synth.BF16: 1.6e-2}


def _tensors():
    from paged_kv_gqa_table_gb300 import tensors
    return tensors


def _binding():
    from paged_kv_gqa_table_gb300 import binding
    return binding


def gpu_out(case, opts=None):
    out = _tensors().paged_decode_attention(case, opts=opts)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def check(case, got):
    ref = oracle.decode(case)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), "non-finite output"
    worst = float(np.max(np.abs(got - ref), initial=0.0))
    assert worst <= TOL[case["dtype"]], "max |diff| %.3g over tolerance" % worst
    return ref


def lens_for(q_len, P):
    """Context lengths around every boundary the causal windows can cross."""
    base = [0, 1, q_len - 1, q_len, q_len + 1, 15, 16, 17, 16 + q_len, 200, 1000]
    if P:
        base += [P - 1, P, P + 1, P + q_len - 1, 2 * P + 3]
    return sorted({max(0, n) for n in base})


# (layout, dtype, D, G, q_len, kv8, P): row tiles = ceil(G * q_len / (16, or 8 for D = 256 or <= 8 rows))
MT_CASES = [
    (synth.NHD, synth.BF16, 128, 4, 4, False, 0),      # 16 rows: one full tile (Llama-3-8B heads)
    (synth.NHD, synth.F16, 64, 2, 3, False, 48),       # 6 rows, small splits
    (synth.VLLM, synth.F16, 256, 6, 2, False, 256),    # 12 rows, D = 256: two tiles of 8
    (synth.VLLM, synth.BF16, 128, 8, 4, False, 0),     # 32 rows: two tiles
    (synth.NHD, synth.BF16, 128, 4, 8, True, 0),       # FP8 cache, fragments straight from the ring
    (synth.NHD, synth.F16, 64, 4, 5, True, 64),        # FP8 cache, D = 64 staging path, 20 rows
    (synth.NHD, synth.BF16, 128, 1, 7, False, 32),     # no grouping, 7 rows
    (synth.NHD, synth.BF16, 128, 32, 2, False, 0),     # 64 rows: four tiles
    (synth.NHD, synth.F16, 256, 2, 16, True, 0),       # FP8 D = 256, 32 rows
]


@pytest.mark.parametrize("layout,dtype,D,G,q_len,kv8,P", MT_CASES)
def test_multi_token_matches_oracle(layout, dtype, D, G, q_len, kv8, P):
    B = _binding()
    extra = dict(kv_dtype=synth.FP8_E4M3) if kv8 else {}
    lens = lens_for(q_len, P)
    case = synth.decode_case(seed=500 + D + G + q_len, B=len(lens), Hq=2 * G, Hkv=2, D=D, block_size=16,
                             dtype=dtype, layout=layout, context_lens=lens, max_blocks_per_seq=80, slack_pages=4,
                             poison=True, q_len=q_len, **extra)
    got = gpu_out(case, B.make_opts(partition_tokens=P) if P else None)
    check(case, got)
    for b, n in enumerate(lens):
        for i in range(q_len):
            if n - q_len + i < 0:
                assert np.all(got[b, i] == 0.0), (n, i)


@pytest.mark.parametrize("layout,dtype,D,G", [(synth.NHD, synth.BF16, 128, 32), (synth.VLLM, synth.F16, 64, 24),
                                              (synth.NHD, synth.F16, 256, 12)])
def test_one_token_groups_beyond_one_tile(layout, dtype, D, G):
    # q_len = 1 with more heads per KV head than one CTA holds: the one-token kernel over row tiles
    lens = [0, 1, 17, 513, 1000]
    case = synth.decode_case(seed=520 + G, B=len(lens), Hq=G, Hkv=1, D=D, block_size=16, dtype=dtype,
                             layout=layout, context_lens=lens, max_blocks_per_seq=64, poison=True)
    check(case, gpu_out(case))


def _slopes(Hq):
    return (2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq)).astype(np.float32)


@pytest.mark.parametrize("kv8", [False, True])
def test_multi_token_with_alibi(kv8):
    B = _binding()
    extra = dict(kv_dtype=synth.FP8_E4M3) if kv8 else {}
    case = synth.decode_case(seed=530, B=9, Hq=8, Hkv=2, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, ctx_range=(0, 1500), max_blocks_per_seq=100, poison=True,
                             q_len=5, **extra)
    case["alibi_slopes"] = _slopes(8)
    slopes = torch.from_numpy(case["alibi_slopes"]).cuda()
    check(case, gpu_out(case, B.make_opts(partition_tokens=256, alibi_slopes=slopes)))


@pytest.mark.parametrize("P", [16, 64, 512])
def test_multi_token_partials_match_oracle(P):
    # Phase 1 alone: per (b, i, h, s) partial of the split's tokens inside query i's window;
    # sentinels where that range is empty (windows ending before the split, n < q_len).
    T, B = _tensors(), _binding()
    case = synth.decode_case(seed=540, B=6, Hq=8, Hkv=2, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, context_lens=[0, 2, 16, 67, 512, 1100], max_blocks_per_seq=80,
                             poison=True, q_len=4)
    case["alibi_slopes"] = _slopes(8)
    slopes = torch.from_numpy(case["alibi_slopes"]).cuda()
    P2, ns, m, l, acc = T.decode_partials(case, opts=B.make_opts(partition_tokens=P, alibi_slopes=slopes))
    assert P2 == P and ns == -(-1100 // P)
    rm, rl, racc = oracle.decode_partials(case, P, ns)
    sentinel = rm == -np.inf
    assert np.all(m[sentinel] == -np.inf) and np.all(l[sentinel] == 0) and np.all(acc[sentinel] == 0)
    live = ~sentinel
    assert np.all(np.isfinite(m[live])) and np.all(l[live] > 0)
    np.testing.assert_allclose(m[live] + np.log(l[live]), rm[live] + np.log(rl[live]), rtol=0, atol=1e-3)
    np.testing.assert_allclose(acc[live] / l[live][..., None], racc[live] / rl[live][..., None], rtol=0,
                               atol=TOL[synth.BF16])


def test_multi_token_combine_of_oracle_partials():
    B, T = _binding(), _tensors()
    case = synth.decode_case(seed=550, B=5, Hq=4, Hkv=2, D=64, block_size=16, dtype=synth.F16,
                             layout=synth.NHD, context_lens=[0, 1, 3, 77, 400], max_blocks_per_seq=32, q_len=3)
    P = 32
    ns = 400 // P + 2
    rm, rl, racc = oracle.decode_partials(case, P, ns)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    out = torch.full(case["q"].shape, float("nan"), dtype=torch.float16, device="cuda")
    ctx = torch.from_numpy(case["context_lens"]).cuda()
    B.pkv_combine(T.decode_desc(case), P, ns, ctx, dev(racc), dev(rm), dev(rl), out)
    torch.cuda.synchronize()
    check(case, out.double().cpu().numpy())


def test_multi_token_graph_replay_with_changed_lengths():
    # Captured once with the capacity as the host bound; replays see new context lengths.
    B, T = _binding(), _tensors()
    cap = 40 * 16
    case = synth.decode_case(seed=560, B=8, Hq=16, Hkv=4, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, context_lens=[cap] * 8, max_blocks_per_seq=40, q_len=4)
    dev = T.upload_decode_case(case)
    desc = T.decode_desc(case)
    out = torch.empty(case["q"].shape, dtype=torch.bfloat16, device="cuda")
    ws = T.workspace_for(desc)
    run = lambda: B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                               dev["context_lens"], case["scale"], out, ws)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    rng = np.random.default_rng(3)
    for trial in range(3):
        lens = rng.integers(0, cap + 1, size=8).astype(np.int32)
        lens[trial] = trial + 1                      # shorter than q_len: partly empty windows
        dev["context_lens"].copy_(torch.from_numpy(lens))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        check(dict(case, context_lens=lens), out.double().cpu().numpy())


def test_speculative_workload_full_size_every_row():
    """The benchmark's 4-token workload at full size in the benchmark's launch
    configuration; every sequence, query token and head checked against the
    oracle."""
    from oracle_threads import decode_all
    case = synth.decode_case(seed=0, **synth.WORKLOADS["llama3_8b_spec_decode_q4"])
    got = gpu_out(case)
    assert np.all(np.isfinite(got))
    ref = decode_all(case)
    worst = float(np.max(np.abs(got - ref)))
    assert worst <= TOL[case["dtype"]], worst
