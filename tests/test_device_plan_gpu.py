"""GPU tests of the device plan (PKV_DECODE_DEVICE_PLAN).

Every CTA of phase 1 reads context_lens on the device, applies the planner
rule to the actual longest and total context and finds its own non-empty
(sequence, KV head, row tile, split) items: the CTAs of a fixed grid take them
in turn.  With exact host bounds the device makes
the host's plan, so the outputs must be bit-identical to the host-planned call;
with capacity bounds (what a captured CUDA graph needs) the outputs must match
the oracle within the decode tolerances.
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


def run(case, desc, opts, dev=None):
    B, T = _binding(), _tensors()
    dev = dev if dev is not None else T.upload_decode_case(case)
    out = torch.full(case["q"].shape, float("nan"), dtype=T.TORCH_DTYPE[case["dtype"]], device="cuda")
    ws = T.workspace_for(desc, opts)
    B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                 dev["context_lens"], case["scale"], out, ws, opts=opts)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "device error word set"
    return out


def loose(case, desc):
    """The description with capacity bounds: every context may reach the table's capacity."""
    cap = case["block_table"].shape[1] * case["block_size"]
    desc.max_context_len = cap
    desc.sum_context_len = case["B"] * cap
    return desc


def check(case, got):
    ref = oracle.decode(case)
    got = got.double().cpu().numpy()
    assert np.all(np.isfinite(got)), "non-finite output"
    worst = float(np.max(np.abs(got - ref), initial=0.0))
    assert worst <= TOL[case["dtype"]], "max |diff| %.3g over tolerance" % worst


CASES = [
    dict(B=64, Hq=32, Hkv=8, D=128, dtype=synth.BF16, layout=synth.NHD, ctx_range=(1, 4096)),
    dict(B=16, Hq=24, Hkv=4, D=256, dtype=synth.F16, layout=synth.VLLM, ctx_range=(0, 3000)),
    dict(B=32, Hq=32, Hkv=8, D=128, dtype=synth.BF16, layout=synth.NHD, ctx_range=(1, 2500),
         kv_dtype=synth.FP8_E4M3),
    dict(B=32, Hq=32, Hkv=8, D=128, dtype=synth.BF16, layout=synth.NHD, ctx_range=(0, 2500), q_len=4),
    dict(B=24, Hq=64, Hkv=4, D=128, dtype=synth.BF16, layout=synth.NHD, ctx_range=(1, 3000)),
]


@pytest.mark.parametrize("idx", range(len(CASES)))
@pytest.mark.parametrize("opt", [dict(), dict(partition_tokens=96), dict(num_splits=5)])
def test_exact_bounds_give_the_host_plan_bit_for_bit(idx, opt):
    B, T = _binding(), _tensors()
    case = synth.decode_case(seed=600 + idx, block_size=16, max_blocks_per_seq=256, **CASES[idx])
    dev = T.upload_decode_case(case)
    desc = T.decode_desc(case)
    host = run(case, desc, B.make_opts(**opt), dev)
    devp = run(case, desc, B.make_opts(device_plan=True, **opt), dev)
    assert torch.equal(host, devp)


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_capacity_bounds_match_the_oracle(idx):
    B, T = _binding(), _tensors()
    case = synth.decode_case(seed=610 + idx, block_size=16, max_blocks_per_seq=300, poison=True, **CASES[idx])
    desc = loose(case, T.decode_desc(case))
    check(case, run(case, desc, B.make_opts(device_plan=True)))


def test_items_beyond_the_grid_are_taken_in_turns():
    # 16-token partitions: ~24k items for a grid of 24 CTAs per SM, so every CTA takes several.
    B, T = _binding(), _tensors()
    case = synth.decode_case(seed=620, B=16, Hq=32, Hkv=8, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, ctx_range=(2000, 4096), max_blocks_per_seq=256)
    dev = T.upload_decode_case(case)
    desc = T.decode_desc(case)
    host = run(case, desc, B.make_opts(partition_tokens=16), dev)
    devp = run(case, desc, B.make_opts(partition_tokens=16, device_plan=True), dev)
    assert torch.equal(host, devp)
    rows = [0, 7, 15]
    ref = np.full(case["q"].shape, np.nan)
    for b in rows:
        oracle.decode(case, b, b + 1, out=ref)
    assert np.max(np.abs(devp.double().cpu().numpy()[rows] - ref[rows])) <= TOL[synth.BF16]


@pytest.mark.parametrize("q_len,kv8", [(1, False), (1, True), (4, False)])
def test_graph_replay_with_capacity_bounds(q_len, kv8):
    """Captured once with capacity bounds; replays see new context lengths.  The
    short-context replays make the device planner raise the partition so that
    the splits fit the workspace's split count; the all-empty replay lists only
    the zero-row items."""
    B, T = _binding(), _tensors()
    cap = 80 * 16
    extra = dict(kv_dtype=synth.FP8_E4M3) if kv8 else {}
    case = synth.decode_case(seed=630, B=12, Hq=16, Hkv=4, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, context_lens=[cap] * 12, max_blocks_per_seq=80, q_len=q_len, **extra)
    dev = T.upload_decode_case(case)
    desc = T.decode_desc(case)                       # bounds: cap and 12 * cap
    opts = B.make_opts(device_plan=True)
    out = torch.empty(case["q"].shape, dtype=torch.bfloat16, device="cuda")
    ws = T.workspace_for(desc, opts)
    run_ = lambda: B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                                dev["context_lens"], case["scale"], out, ws, opts=opts)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run_()
    rng = np.random.default_rng(5)
    trials = [rng.integers(0, cap + 1, size=12), np.full(12, cap), np.zeros(12), rng.integers(0, 40, size=12)]
    for lens in trials:
        lens = lens.astype(np.int32)
        dev["context_lens"].copy_(torch.from_numpy(lens))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        check(dict(case, context_lens=lens), out)
    assert int(ws[:4].view(torch.int32).item()) == 0


def test_device_plan_header():
    # Header words 4..5, written by phase 1: partition, splits of the longest context.
    B, T = _binding(), _tensors()
    lens = [0, 1, 700, 1024, 1025, 300]
    case = synth.decode_case(seed=640, B=6, Hq=8, Hkv=2, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, context_lens=lens, max_blocks_per_seq=128)
    desc = loose(case, T.decode_desc(case))          # bounds 2048 / 12288: host plan 512, 4 splits
    opts = B.make_opts(partition_tokens=512, device_plan=True)
    dev = T.upload_decode_case(case)
    out = torch.empty(case["q"].shape, dtype=torch.bfloat16, device="cuda")
    ws = T.workspace_for(desc, opts)
    B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                 dev["context_lens"], case["scale"], out, ws, opts=opts)
    torch.cuda.synchronize()
    hdr = ws[16:24].view(torch.int32).cpu().tolist()
    assert hdr == [512, 3]
    check(case, out)


def test_more_sequences_than_one_scan_chunk():
    # 2500 sequences: each phase-1 CTA walks them 32 at a time to its items (later chunks reload their
    # lengths from global memory); many empty and one-page contexts.
    B, T = _binding(), _tensors()
    case = synth.decode_case(seed=650, B=2500, Hq=8, Hkv=2, D=64, block_size=16, dtype=synth.F16,
                             layout=synth.NHD, ctx_range=(0, 90), max_blocks_per_seq=8)
    dev = T.upload_decode_case(case)
    desc = T.decode_desc(case)
    for opt in (dict(), dict(partition_tokens=32)):
        host = run(case, desc, B.make_opts(**opt), dev)
        devp = run(case, desc, B.make_opts(device_plan=True, **opt), dev)
        assert torch.equal(host, devp)
    rows = [0, 1023, 1024, 1500, 2047, 2048, 2499]
    ref = np.full(case["q"].shape, np.nan)
    for b in rows:
        oracle.decode(case, b, b + 1, out=ref)
    got = run(case, loose(case, T.decode_desc(case)), B.make_opts(device_plan=True), dev).double().cpu().numpy()
    assert np.max(np.abs(got[rows] - ref[rows])) <= TOL[synth.F16]


@pytest.mark.parametrize("q_len", [1, 4])
def test_plan_made_once_reused_by_later_layers(q_len):
    # Three "layers" of one decode step share context_lens and the block table: the first call
    # plans on the device, the next two reuse its plan (PKV_DECODE_PLAN_READY) with their own
    # queries and caches.
    B, T = _binding(), _tensors()
    base = synth.decode_case(seed=660, B=20, Hq=16, Hkv=4, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, ctx_range=(0, 1500), max_blocks_per_seq=100, q_len=q_len)
    layers = [base]
    for i in (1, 2):
        new = lambda stream, a: synth.normal_bits(661 + i, stream, a.size, synth.BF16).reshape(a.shape)
        layers.append(dict(base, q=new(3, base["q"]), k_cache=new(4, base["k_cache"]),
                           v_cache=new(5, base["v_cache"])))
    desc = loose(base, T.decode_desc(base))
    plan, reuse = B.make_opts(device_plan=True), B.make_opts(plan_ready=True)
    ws = T.workspace_for(desc, plan)
    outs = []
    for i, c in enumerate(layers):
        dev = T.upload_decode_case(c)
        out = torch.full(c["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                     dev["context_lens"], c["scale"], out, ws, opts=plan if i == 0 else reuse)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    for c, out in zip(layers, outs):
        check(c, out)


def _call(case, desc, opts, dev, ws, out):
    B = _binding()
    B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                 dev["context_lens"], case["scale"], out, ws, opts=opts)


REUSE_CASES = CASES + [
    # more sequences than the planner keeps in registers (its walk from memory writes the table)
    dict(B=300, Hq=8, Hkv=2, D=64, dtype=synth.F16, layout=synth.NHD, ctx_range=(0, 400)),
]


@pytest.mark.parametrize("idx", range(len(REUSE_CASES)))
@pytest.mark.parametrize("bounds", ["exact", "capacity"])
@pytest.mark.parametrize("opt", [dict(), dict(partition_tokens=32)])
def test_reused_plan_is_bit_identical_to_planning(idx, bounds, opt):
    # A call with PKV_DECODE_PLAN_READY takes its items from the split table the planning call
    # left in the workspace: the same items, so the same bits; a second reuse finds the table
    # unchanged.
    B, T = _binding(), _tensors()
    case = synth.decode_case(seed=670 + idx, block_size=16, max_blocks_per_seq=256, **REUSE_CASES[idx])
    dev = T.upload_decode_case(case)
    desc = T.decode_desc(case)
    if bounds == "capacity":
        desc = loose(case, desc)
    plan, reuse = B.make_opts(device_plan=True, **opt), B.make_opts(plan_ready=True, **opt)
    ws = T.workspace_for(desc, plan)
    outs = []
    for opts in (plan, reuse, reuse):
        out = torch.full(case["q"].shape, float("nan"), dtype=T.TORCH_DTYPE[case["dtype"]], device="cuda")
        _call(case, desc, opts, dev, ws, out)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    check(case, outs[1])


def test_split_table_contents():
    # Header word 6 holds the plan's split count; entry g of the table (after the partials) is
    # {sequence, split, clamped context, 0} for the g-th split in (sequence, split) order.
    B, T = _binding(), _tensors()
    lens = [0, 1, 700, 1024, 1025, 300]
    case = synth.decode_case(seed=641, B=6, Hq=8, Hkv=2, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, context_lens=lens, max_blocks_per_seq=128)
    desc = loose(case, T.decode_desc(case))          # bounds 2048: 4 splits of 512 per sequence
    opts = B.make_opts(partition_tokens=512, device_plan=True)
    ns, P = B.pkv_plan_splits(desc, opts)
    dev = T.upload_decode_case(case)
    out = torch.empty(case["q"].shape, dtype=torch.bfloat16, device="cuda")
    ws = T.workspace_for(desc, opts)
    _call(case, desc, opts, dev, ws, out)
    torch.cuda.synchronize()
    want = [(b, s, n) for b, n in enumerate(lens) for s in range(max(1, -(-n // 512)))]
    assert ws[16:28].view(torch.int32).cpu().tolist() == [512, 3, len(want)]
    tab_bytes = (6 * ns * 16 + 255) // 256 * 256
    tab = ws[ws.numel() - tab_bytes:].view(torch.int32).view(-1, 4).cpu().numpy()
    assert [tuple(int(v) for v in row[:3]) for row in tab[:len(want)]] == want
    assert np.all(tab[:len(want), 3] == 0)


def test_reuse_without_a_plan_is_reported():
    # The flag states that the workspace holds this problem's plan.  A workspace that holds none
    # (a header of all ones) sets error bit 1 and reads nothing else of it; a table whose entries
    # are out of range (all ones after a real plan) sets it too and skips those items.  Either way
    # no memory outside the arguments is touched, and the next planning call is correct.
    B, T = _binding(), _tensors()
    case = synth.decode_case(seed=642, B=16, Hq=32, Hkv=8, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, ctx_range=(16, 3000), max_blocks_per_seq=256)
    desc = T.decode_desc(case)
    plan, reuse = B.make_opts(device_plan=True), B.make_opts(plan_ready=True)
    ns, _ = B.pkv_plan_splits(desc, plan)
    dev = T.upload_decode_case(case)
    out = torch.zeros(case["q"].shape, dtype=torch.bfloat16, device="cuda")
    ws = T.workspace_for(desc, plan)
    ws.fill_(0xFF)
    ws[:4].zero_()
    _call(case, desc, reuse, dev, ws, out)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 2
    tab_bytes = (case["B"] * ns * 16 + 255) // 256 * 256
    ws[:4].zero_()
    _call(case, desc, plan, dev, ws, out)
    ws[ws.numel() - tab_bytes:].fill_(0xFF)
    _call(case, desc, reuse, dev, ws, out)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 2
    # A partition that is not a page multiple is refused; one near 2^31 fails the entries whose
    # last key or page index would overflow (every context here is longer than 15 tokens).
    assert min(case["context_lens"]) > 15
    for bad_p in (17, 0x7FFFFFF0):
        ws[:4].zero_()
        _call(case, desc, plan, dev, ws, out)
        ws[16:20].view(torch.int32).fill_(bad_p)
        _call(case, desc, reuse, dev, ws, out)
        torch.cuda.synchronize()
        assert int(ws[:4].view(torch.int32).item()) == 2, bad_p
    ws[:4].zero_()
    _call(case, desc, plan, dev, ws, out)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    check(case, out)
