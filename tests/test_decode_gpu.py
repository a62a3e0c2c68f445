"""GPU parity of paged GQA decode (phase 1 + combine) against the fp64 oracle.

Every call goes through the C ABI (libpkv) via the ctypes binding.  Tolerances
are the stated bars on outputs: max |diff| <= 4e-3 for fp16 and <= 1.6e-2 for
bf16, against the unrounded fp64 oracle.  Partials compare lse_s = m_s + ln l_s
within 1e-3 and acc_s / l_s within the output tolerance.
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
    T = _tensors()
    out = T.paged_decode_attention(case, opts=opts)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def check_rows(case, got, b_idx, err_out=None):
    ref = np.full(got.shape, np.nan)
    for b in b_idx:
        oracle.decode(case, b, b + 1, out=ref)
    diff = np.abs(got[b_idx] - ref[b_idx])
    assert np.all(np.isfinite(got[b_idx])), "non-finite output"
    worst = float(diff.max(initial=0.0))
    assert worst <= TOL[case["dtype"]], "max |diff| %.3g over tolerance" % worst
    return worst


def _case(seed, **kw):
    return synth.decode_case(seed=seed, **kw)


# ------------------------------------------------------------------ tiny ----

@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4])
def test_tiny_workload(seed):
    case = _case(seed, poison=True, **synth.WORKLOADS["tiny"])
    check_rows(case, gpu_out(case), list(range(case["B"])))


# ---------------------------------------------------- shapes and edge cases ----

SHAPES = []
for layout in (synth.NHD, synth.VLLM):
    for dtype in (synth.F16, synth.BF16):
        for D in (64, 128, 256):
            for G in (1, 2, 4, 6, 8, 16):
                if G > 8 and D > 128:
                    continue
                SHAPES.append((layout, dtype, D, G))


@pytest.mark.parametrize("layout,dtype,D,G", SHAPES)
def test_shapes_and_edge_lengths(layout, dtype, D, G):
    Hkv = 2
    lens = [0, 1, 15, 16, 17, 200, 512, 513, 1000]
    case = _case(7 * D + G, B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=D, block_size=16, dtype=dtype, layout=layout,
                 context_lens=lens, slack_pages=5, max_blocks_per_seq=70, poison=True)
    got = gpu_out(case)
    check_rows(case, got, list(range(case["B"])))
    assert np.all(got[0] == 0.0)


@pytest.mark.parametrize("opts", [dict(partition_tokens=16), dict(partition_tokens=48), dict(partition_tokens=512),
                                  dict(num_splits=7), dict(num_splits=1), dict(partition_tokens=4096)])
@pytest.mark.parametrize("layout", [synth.NHD, synth.VLLM])
def test_forced_splits(opts, layout):
    B = _binding()
    case = _case(11, B=5, Hq=8, Hkv=2, D=128, block_size=16, dtype=synth.BF16, layout=layout,
                 context_lens=[3, 700, 1, 1024, 333], max_blocks_per_seq=64, slack_pages=2, poison=True)
    got = gpu_out(case, B.make_opts(**opts))
    check_rows(case, got, list(range(case["B"])))


def test_all_contexts_empty_with_an_empty_pool():
    # no page in the pool: null caches are accepted and every row is zero
    B, T = _binding(), _tensors()
    case = _case(6, B=3, Hq=8, Hkv=2, D=128, block_size=16, dtype=synth.BF16, layout=synth.NHD,
                 context_lens=[0, 0, 0], max_blocks_per_seq=4)
    assert case["num_blocks"] == 0
    dev = T.upload_decode_case(case)
    out = torch.full(case["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    desc = T.decode_desc(case)
    B.pkv_paged_decode_attention(desc, dev["q"], None, None, dev["block_table"], dev["context_lens"],
                                 case["scale"], out, T.workspace_for(desc))
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_all_contexts_empty():
    case = _case(5, B=3, Hq=4, Hkv=1, D=64, block_size=16, dtype=synth.F16, layout=synth.NHD,
                 context_lens=[0, 0, 0], max_blocks_per_seq=2, slack_pages=2)
    got = gpu_out(case)
    assert np.all(got == 0.0)


# ---------------------------------------------------------- invariants ----

def test_relabelled_pages_are_bit_identical_on_gpu():
    case = _case(21, B=6, Hq=16, Hkv=4, D=128, block_size=16, dtype=synth.BF16, layout=synth.NHD,
                 ctx_range=(1, 900), max_blocks_per_seq=64, slack_pages=9)
    moved = synth.relabel_pages(case, seed=5)
    a, b = gpu_out(case), gpu_out(moved)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("layout", [synth.NHD, synth.VLLM])
def test_poisoned_unread_slots_are_bit_identical_on_gpu(layout):
    kw = dict(B=6, Hq=12, Hkv=2, D=256 if layout == synth.VLLM else 128, block_size=16, dtype=synth.F16,
              layout=layout, ctx_range=(1, 700), max_blocks_per_seq=64, slack_pages=4)
    clean = _case(31, **kw)
    dirty = _case(31, poison=True, **kw)
    assert np.array_equal(gpu_out(clean), gpu_out(dirty))


def test_constant_v_rows_give_the_constant_on_gpu():
    case = _case(3, B=4, Hq=8, Hkv=2, D=128, block_size=16, dtype=synth.F16, layout=synth.NHD,
                 context_lens=[1, 17, 600, 1500], max_blocks_per_seq=100)
    case["v_cache"] = np.full_like(case["v_cache"], 0x4500)   # 5.0
    got = gpu_out(case)
    assert np.max(np.abs(got - 5.0)) <= TOL[synth.F16]


# ------------------------------------------------------------- layered ----

@pytest.mark.parametrize("layout,dtype,D,G,P", [(synth.NHD, synth.BF16, 128, 4, 64), (synth.NHD, synth.F16, 64, 2, 48),
                                               (synth.VLLM, synth.F16, 256, 6, 512), (synth.VLLM, synth.BF16, 128, 16, 32)])
def test_phase1_partials_match_oracle_split_mode(layout, dtype, D, G, P):
    T, B = _tensors(), _binding()
    case = _case(41, B=4, Hq=2 * G, Hkv=2, D=D, block_size=16, dtype=dtype, layout=layout,
                 context_lens=[0, 5, 130, 1100], max_blocks_per_seq=80, slack_pages=3, poison=True)
    P2, ns, m, l, acc = T.decode_partials(case, opts=B.make_opts(partition_tokens=P), capacity=None)
    assert P2 == P and ns == -(-1100 // P)
    rm, rl, racc = oracle.decode_partials(case, P, ns)
    sentinel = rm == -np.inf
    assert np.all(m[sentinel] == -np.inf) and np.all(l[sentinel] == 0) and np.all(acc[sentinel] == 0)
    live = ~sentinel
    np.testing.assert_allclose(m[live] + np.log(l[live]), rm[live] + np.log(rl[live]), rtol=0, atol=1e-3)
    np.testing.assert_allclose(acc[live] / l[live][..., None], racc[live] / rl[live][..., None], rtol=0, atol=TOL[dtype])


@pytest.mark.parametrize("dtype,D,P", [(synth.BF16, 128, 64), (synth.F16, 64, 64), (synth.F16, 256, 64),
                                       (synth.BF16, 128, 16), (synth.F16, 64, 16)])
def test_combine_of_oracle_partials(dtype, D, P):
    """Phase 2 fed the oracle's partials; P = 16 gives 66 splits (the many-split variant)."""
    B = _binding()
    T = _tensors()
    case = _case(43, B=5, Hq=4, Hkv=2, D=D, block_size=16, dtype=dtype, layout=synth.NHD,
                 context_lens=[0, 1, 77, 400, 1024], max_blocks_per_seq=64)
    ns = 1024 // P + 2
    rm, rl, racc = oracle.decode_partials(case, P, ns)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    out = torch.empty((case["B"], case["Hq"], D), dtype=T.TORCH_DTYPE[dtype], device="cuda")
    ctx = torch.from_numpy(case["context_lens"]).cuda()
    B.pkv_combine(T.decode_desc(case), P, ns, ctx, dev(racc), dev(rm), dev(rl), out)
    torch.cuda.synchronize()
    check_rows(case, out.double().cpu().numpy(), list(range(case["B"])))


# ---------------------------------------------------------- validator ----

def test_validator_flags_bad_tables_without_faulting():
    B, T = _binding(), _tensors()
    case = _case(51, B=3, Hq=4, Hkv=2, D=64, block_size=16, dtype=synth.F16, layout=synth.NHD,
                 context_lens=[40, 16, 0], max_blocks_per_seq=4, slack_pages=1)
    desc = T.decode_desc(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = T.upload_decode_case(case)
    B.pkv_validate_block_table(desc, dev["block_table"], dev["context_lens"], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bad = case["block_table"].copy()
    bad[0, 1] = -1                     # live entry of sequence 0
    bad[1, 3] = 10 ** 6                # past sequence 1's live range: not inspected
    dev_bad = torch.from_numpy(bad).cuda()
    B.pkv_validate_block_table(desc, dev_bad, dev["context_lens"], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 2
    # the decode itself stays in bounds on the same bad table (result unspecified)
    case_bad = dict(case, block_table=bad)
    out = gpu_out(case_bad)
    assert out.shape == (3, 4, 64)
    err.zero_()
    ctx_bad = torch.tensor([40, 65, 0], dtype=torch.int32, device="cuda")   # 65 > 4 pages * 16
    B.pkv_validate_block_table(desc, dev["block_table"], ctx_bad, err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1


# ------------------------------------------------- full-size workloads ----

FULL = ["llama3_8b_decode", "long_context_decode", "gqa6_d256_vllm_decode", "llama3_8b_decode_fp8"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads_every_row(name):
    """The benchmark's workloads at full size, in the launch configuration the
    benchmark times (default plan): every output row (all sequences, all query
    heads, all D columns) checked against the oracle."""
    from oracle_threads import decode_all
    case = synth.decode_case(seed=0, **synth.WORKLOADS[name])
    got = gpu_out(case)
    assert np.all(np.isfinite(got))
    ref = decode_all(case)
    assert np.all(np.isfinite(ref))
    worst = float(np.max(np.abs(got - ref)))
    assert worst <= TOL[case["dtype"]], worst


# ------------------------------------------------------------ FP8 caches ----

FP8_CASES = [
    (synth.BF16, 128, 4, (1, 3000), 0),      # Llama-3-8B-shaped heads, planner
    (synth.F16, 128, 4, (0, 700), 64),       # fp16 queries, empty contexts, small splits
    (synth.BF16, 64, 8, (1, 500), 0),
    (synth.F16, 256, 6, (17, 1200), 256),    # D = 256
    (synth.BF16, 128, 16, (1, 900), 128),    # two head tiles
]


@pytest.mark.parametrize("dtype,D,G,ctx,P", FP8_CASES)
def test_fp8_kv_cache_matches_oracle(dtype, D, G, ctx, P):
    B = _binding()
    case = _case(21, B=19, Hq=2 * G, Hkv=2, D=D, block_size=16, dtype=dtype, layout=synth.NHD, ctx_range=ctx,
                 max_blocks_per_seq=200, kv_dtype=synth.FP8_E4M3, k_scale=0.05, v_scale=0.07, slack_pages=5,
                 poison=True)
    got = gpu_out(case, B.make_opts(partition_tokens=P) if P else None)
    check_rows(case, got, list(range(case["B"])))


def test_fp8_poisoned_unread_slots_are_bit_identical():
    kw = dict(B=11, Hq=16, Hkv=4, D=128, block_size=16, dtype=synth.BF16, layout=synth.NHD, ctx_range=(1, 600),
              kv_dtype=synth.FP8_E4M3, slack_pages=9)
    clean = gpu_out(_case(22, **kw))
    dirty = gpu_out(_case(22, poison=True, **kw))
    assert np.array_equal(clean, dirty)


def test_fp8_partials_match_oracle():
    B = _binding()
    T = _tensors()
    case = _case(23, B=9, Hq=8, Hkv=2, D=128, block_size=16, dtype=synth.F16, layout=synth.NHD,
                 ctx_range=(0, 900), kv_dtype=synth.FP8_E4M3, k_scale=0.03, v_scale=0.1)
    dev = T.upload_decode_case(case)
    NS_cap = 8
    acc = torch.empty((9, 8, NS_cap, 128), device="cuda")
    m = torch.empty((9, 8, NS_cap), device="cuda")
    l = torch.empty((9, 8, NS_cap), device="cuda")
    P, ns = B.pkv_decode_partials(T.decode_desc(case), dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                  dev["context_lens"], case["scale"], acc, m, l, NS_cap,
                                  opts=B.make_opts(partition_tokens=128))
    torch.cuda.synchronize()
    pm, pl, pacc = oracle.decode_partials(case, P, ns)
    gm, gl, gacc = m.cpu().numpy()[:, :, :ns], l.cpu().numpy()[:, :, :ns], acc.cpu().numpy()[:, :, :ns]
    live = pl > 0
    assert np.array_equal(live, gl > 0)
    assert np.all(np.isneginf(gm[~live]))
    lse_g, lse_r = gm[live] + np.log(gl[live]), pm[live] + np.log(pl[live])
    assert np.max(np.abs(lse_g - lse_r)) <= 1e-3
    assert np.max(np.abs(gacc[live] / gl[live][:, None] - pacc[live] / pl[live][:, None])) <= TOL[synth.F16]


def test_fp8_with_bf16_queries_beyond_the_fp16_range():
    # bf16 queries up to ~2^22 (scaled by 2^20) with the score scale reduced by
    # the same factor: same attention, but the queries only fit fp16 after the
    # kernel's power-of-two down-scaling.
    case = _case(24, B=6, Hq=8, Hkv=2, D=128, block_size=16, dtype=synth.BF16, layout=synth.NHD,
                 ctx_range=(20, 400), kv_dtype=synth.FP8_E4M3)
    qf = synth.bits_to_f32(case["q"], synth.BF16) * np.float32(2.0 ** 20)
    case["q"] = synth.f32_to_bits(qf, synth.BF16).reshape(case["q"].shape)
    case["scale"] = case["scale"] * 2.0 ** -20
    got = gpu_out(case)
    assert np.all(np.isfinite(got))
    check_rows(case, got, list(range(case["B"])))


# ------------------------------------------------------------------ ALiBi ----

def _slopes(Hq):
    # the usual geometric ALiBi slopes 2^(-8 i / Hq), i = 1..Hq
    return (2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq)).astype(np.float32)


@pytest.mark.parametrize("layout,dtype,D,G,kv8,P", [
    (synth.NHD, synth.BF16, 128, 4, False, 0),
    (synth.VLLM, synth.F16, 256, 6, False, 256),
    (synth.NHD, synth.F16, 64, 8, False, 64),
    (synth.NHD, synth.BF16, 128, 16, False, 128),
    (synth.NHD, synth.BF16, 128, 4, True, 0),
    (synth.NHD, synth.F16, 256, 2, True, 256),
])
def test_alibi_matches_oracle(layout, dtype, D, G, kv8, P):
    B = _binding()
    extra = dict(kv_dtype=synth.FP8_E4M3) if kv8 else {}
    case = _case(31, B=13, Hq=2 * G, Hkv=2, D=D, block_size=16, dtype=dtype, layout=layout, ctx_range=(0, 1800),
                 max_blocks_per_seq=128, poison=True, **extra)
    case["alibi_slopes"] = _slopes(case["Hq"])
    slopes = torch.from_numpy(case["alibi_slopes"]).cuda()
    got = gpu_out(case, B.make_opts(partition_tokens=P, alibi_slopes=slopes))
    check_rows(case, got, list(range(case["B"])))
    # and it is a different problem: without the slopes the output changes
    plain = gpu_out(case, B.make_opts(partition_tokens=P))
    assert not np.allclose(plain, got)


def test_alibi_partials_match_oracle():
    B = _binding()
    T = _tensors()
    case = _case(32, B=7, Hq=8, Hkv=2, D=128, block_size=16, dtype=synth.BF16, layout=synth.NHD,
                 ctx_range=(1, 700))
    case["alibi_slopes"] = _slopes(8)
    dev = T.upload_decode_case(case)
    slopes = torch.from_numpy(case["alibi_slopes"]).cuda()
    acc = torch.empty((7, 8, 8, 128), device="cuda")
    m = torch.empty((7, 8, 8), device="cuda")
    l = torch.empty((7, 8, 8), device="cuda")
    P, ns = B.pkv_decode_partials(T.decode_desc(case), dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                  dev["context_lens"], case["scale"], acc, m, l, 8,
                                  opts=B.make_opts(partition_tokens=96, alibi_slopes=slopes))
    torch.cuda.synchronize()
    pm, pl, pacc = oracle.decode_partials(case, P, ns)
    gm, gl, gacc = m.cpu().numpy()[:, :, :ns], l.cpu().numpy()[:, :, :ns], acc.cpu().numpy()[:, :, :ns]
    live = pl > 0
    assert np.array_equal(live, gl > 0)
    assert np.max(np.abs((gm[live] + np.log(gl[live])) - (pm[live] + np.log(pl[live])))) <= 1e-3
    assert np.max(np.abs(gacc[live] / gl[live][:, None] - pacc[live] / pl[live][:, None])) <= TOL[synth.BF16]


# ---------------------------------------------------------- CUDA graphs ----

@pytest.mark.parametrize("kv8", [False, True])
def test_decode_step_replays_in_a_cuda_graph(kv8):
    """One call captured into a CUDA graph (phase 1, and the combine as its
    programmatic dependent) replays correctly after context_lens change on the
    device: the plan only needs host-known upper bounds (here the block-table
    capacity), so the captured grid covers every replay."""
    B = _binding()
    T = _tensors()
    cap = 80 * 16
    extra = dict(kv_dtype=synth.FP8_E4M3) if kv8 else {}
    case = _case(41, B=12, Hq=16, Hkv=4, D=128, block_size=16, dtype=synth.BF16, layout=synth.NHD,
                 context_lens=[cap] * 12, max_blocks_per_seq=80, **extra)
    dev = T.upload_decode_case(case)
    desc = T.decode_desc(case)            # max_context_len = cap, sum = 12 * cap: bounds for any replay
    out = torch.empty((12, 16, 128), dtype=torch.bfloat16, device="cuda")
    ws = T.workspace_for(desc)
    run = lambda: B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                               dev["context_lens"], case["scale"], out, ws)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run()                             # first call on the device: kernel attributes, outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    rng = np.random.default_rng(7)
    for trial in range(3):
        lens = rng.integers(0, cap + 1, size=12).astype(np.int32)
        lens[trial] = 0
        dev["context_lens"].copy_(torch.from_numpy(lens))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        sub = dict(case, context_lens=lens)
        check_rows(sub, out.double().cpu().numpy(), list(range(12)))


def test_million_token_context():
    # One sequence of 1,000,003 tokens beside a short one: 1,954 splits of 512 tokens merged by the
    # wide combine, a block-table row of 62,501 pages (a random permutation of the pool), and the
    # unread tail slots poisoned.  Host plan and device plan (exact bounds: the same items, so the
    # same bits) against the oracle on both rows.
    B, T = _binding(), _tensors()
    case = _case(31, B=2, Hq=8, Hkv=1, D=128, block_size=16, dtype=synth.BF16, layout=synth.NHD,
                 context_lens=[1_000_003, 777], max_blocks_per_seq=62_501, slack_pages=3, poison=True)
    desc = T.decode_desc(case)
    assert B.pkv_plan_splits(desc) == (1954, 512)
    dev = T.upload_decode_case(case)
    outs = []
    for opts in (None, B.make_opts(device_plan=True)):
        out = T.paged_decode_attention(case, dev=dev, opts=opts)
        torch.cuda.synchronize()
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
    check_rows(case, outs[0].double().cpu().numpy(), [0, 1])
