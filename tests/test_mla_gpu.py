"""GPU parity of the MLA paged causal prefill (tcgen05 path) against the fp64 oracle.

Calls go through the C ABI.  Bars: bf16 output max |diff| <= 1.6e-2, base-2
LSE max |diff| <= 1e-3 (absolute), both against the unrounded fp64 oracle.
"""
import numpy as np
import pytest

import oracle
from paged_kv_gqa_table_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TOL_OUT, TOL_LSE = 1.6e-2, 1e-3


def gpu_mla(case, replay=True):
    """replay=True (the default of tensors.mla_desc) passes max_kv_len: S once per row tile,
    the second output half computed from the first's exported softmax weights."""
    from paged_kv_gqa_table_gb300 import tensors
    out, lse = tensors.mla_paged_prefill(case, desc=tensors.mla_desc(case, replay=replay))
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def check(case, got_out, got_lse, tokens=None):
    T = case["total_q"]
    tokens = list(range(T)) if tokens is None else tokens
    ref_out = np.full(got_out.shape, np.nan)
    ref_lse = np.full(got_lse.shape, np.nan)
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(8) as ex:
        list(ex.map(lambda t: oracle.mla(case, t, t + 1, out=ref_out, lse=ref_lse), tokens))
    o, l = got_out[tokens], got_lse[tokens]
    ro, rl = ref_out[tokens], ref_lse[tokens]
    assert np.all(np.isfinite(o)), "non-finite output"
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(l), fin)
    assert np.all(l[~fin] == rl[~fin])
    err_o = float(np.max(np.abs(o - ro), initial=0.0))
    err_l = float(np.max(np.abs(l[fin] - rl[fin]), initial=0.0))
    assert err_o <= TOL_OUT, "out max |diff| %.3g" % err_o
    assert err_l <= TOL_LSE, "lse max |diff| %.3g" % err_l
    return err_o, err_l


SMALL = [
    dict(batch=3, q_len_range=(1, 20), prefix_range=(0, 300), slack_pages=7),
    dict(batch=2, q_len_range=(8, 8), prefix_range=(120, 136), slack_pages=3),
    dict(batch=4, q_len_range=(1, 1), prefix_range=(0, 700)),
    dict(batch=2, q_len_range=(33, 70), prefix_range=(0, 0), sm_scale=1.0),
    dict(batch=2, q_len_range=(100, 140), prefix_range=(250, 270), sm_scale=1.0 / 24.0),
]


@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_mla_small_cases(idx):
    case = synth.mla_case(seed=idx, poison=True, **SMALL[idx])
    check(case, *gpu_mla(case))


def test_mla_empty_sequences():
    # q_len = 0 in the middle, and a sequence whose KV is empty (out 0, lse -inf)
    case = synth.mla_case(seed=3, batch=3, q_len_range=(1, 1), prefix_range=(0, 0), q_lens=[5, 0, 9],
                          prefixes=[30, 0, 200])
    check(case, *gpu_mla(case))
    empty = synth.mla_case(seed=4, batch=2, q_len_range=(1, 1), prefix_range=(0, 0), q_lens=[3, 4],
                           prefixes=[10, 0])
    empty["kv_indptr"] = np.array([0, 13, 13], np.int32)          # second sequence: 4 queries, no KV
    empty["kv_indices"] = empty["kv_indices"][:13].copy()
    out, lse = gpu_mla(empty)
    assert np.all(out[3:] == 0) and np.all(lse[3:] == -np.inf)
    check(empty, out, lse)


def test_mla_zero_query_closed_form():
    case = synth.mla_case(seed=9, batch=2, q_len_range=(20, 40), prefix_range=(100, 300))
    case["q_nope"] = np.zeros_like(case["q_nope"])
    case["q_pe"] = np.zeros_like(case["q_pe"])
    out, lse = gpu_mla(case)
    qo, kvp = case["qo_indptr"], case["kv_indptr"]
    for b in range(2):
        q_len, kv_len = qo[b + 1] - qo[b], kvp[b + 1] - kvp[b]
        for i in range(q_len):
            assert np.max(np.abs(lse[qo[b] + i] - np.log2(kv_len - q_len + i + 1))) <= TOL_LSE
    check(case, out, lse)


def test_mla_relabelled_pages_are_bit_identical():
    case = synth.mla_case(seed=12, batch=3, q_len_range=(10, 30), prefix_range=(50, 400), slack_pages=11)
    a = gpu_mla(case)
    perm = np.random.default_rng(5).permutation(case["num_pages"])   # page p moves to perm[p]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    moved = dict(case, ckv_cache=case["ckv_cache"][inv].copy(), kpe_cache=case["kpe_cache"][inv].copy(),
                 kv_indices=perm[case["kv_indices"]].astype(np.int32))
    b = gpu_mla(moved)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_mla_full_size_workload_every_token():
    """The benchmark's MLA workload at full size: every query token and head
    (output and LSE) checked against the oracle."""
    from oracle_threads import mla_all
    case = synth.mla_case(seed=0, **synth.MLA_WORKLOADS["mla_prefill_h16"])
    out, lse = gpu_mla(case)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    ref_out, ref_lse = mla_all(case)
    err_o = float(np.max(np.abs(out - ref_out)))
    err_l = float(np.max(np.abs(lse - ref_lse)))
    assert err_o <= TOL_OUT, "out max |diff| %.3g" % err_o
    assert err_l <= TOL_LSE, "lse max |diff| %.3g" % err_l


@pytest.mark.parametrize("seed", [0, 1])
def test_mla_non_finite_rows_stay_in_their_sequence(seed):
    """NaN in every cached row of the middle sequence of three: the other two
    sequences' outputs and LSEs match the oracle element by element (their
    128-key blocks never reach the middle sequence's rows); the middle
    sequence's own rows are not checked."""
    case = synth.mla_case(seed=40 + seed, batch=3, q_len_range=(1, 1), prefix_range=(0, 0),
                          q_lens=[37, 20, 45], prefixes=[50 + 60 * seed, 90, 200])
    kvp, qo = case["kv_indptr"], case["qo_indptr"]
    clean = synth.mla_case(seed=40 + seed, batch=3, q_len_range=(1, 1), prefix_range=(0, 0),
                           q_lens=[37, 20, 45], prefixes=[50 + 60 * seed, 90, 200])
    for r in case["kv_indices"][kvp[1]:kvp[2]]:
        case["ckv_cache"][r] = synth.NAN_BITS[synth.BF16]
        case["kpe_cache"][r] = synth.NAN_BITS[synth.BF16]
    out, lse = gpu_mla(case)
    ref_out, ref_lse = oracle.mla(clean)
    keep = np.r_[qo[0]:qo[1], qo[2]:qo[3]]
    assert np.all(np.isfinite(out[keep])) and np.all(np.isfinite(lse[keep]))
    assert float(np.max(np.abs(out[keep] - ref_out[keep]))) <= TOL_OUT
    assert float(np.max(np.abs(lse[keep] - ref_lse[keep]))) <= TOL_LSE


def _run_with(case, nnz=None, fill=None, max_kv_len=None):
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import tensors
    desc = tensors.mla_desc(case)
    if nnz is not None:
        desc.nnz = int(nnz)
    if max_kv_len is not None:
        desc.max_kv_len = int(max_kv_len)
    ws = tensors.mla_workspace_for(desc)
    if fill is not None:
        ws[256:].fill_(fill)           # leave the error header zeroed
    out, lse = tensors.mla_paged_prefill(case, workspace=ws, desc=desc)
    torch.cuda.synchronize()
    err = int(ws[:4].view(torch.int32).item())
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), err


def test_mla_workspace_contents_do_not_matter():
    # 0xFF bytes are NaN in bf16: every staged row the kernel reads must have
    # been written by this call, including the zero rows past the last key.
    case = synth.mla_case(seed=21, batch=3, q_len_range=(5, 140), prefix_range=(0, 260), slack_pages=5)
    out, lse, err = _run_with(case, fill=0xFF)
    assert err == 0
    check(case, out, lse)
    # an upper bound for nnz (more rows than kv_indptr[batch]) gives the same bits
    out2, lse2, err2 = _run_with(case, nnz=int(case["kv_indptr"][-1]) + 1000, fill=0xFF)
    assert err2 == 0
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_mla_short_nnz_is_reported():
    # nnz below kv_indptr[batch]: keys past it are not staged (their boxes read
    # TMA zero fill), the call completes and error bit 1 is set.
    case = synth.mla_case(seed=22, batch=2, q_len_range=(20, 40), prefix_range=(100, 200))
    out, lse, err = _run_with(case, nnz=int(case["kv_indptr"][-1]) // 2)
    assert err == 2
    assert out.shape == (case["total_q"], 16, 512)


@pytest.mark.parametrize("i", range(30))
def test_mla_random_case_matches_oracle(i):
    """Seeded random batches: empty and single-token queries, row tiles cut at 8
    tokens, prefixes around the 128-key block edge, slack pages poisoned."""
    import random
    r = random.Random(9000 + i)
    batch = r.randint(1, 5)
    q_lens = [r.choice([0, 1, r.randint(1, 70), 8, 9, 16]) for _ in range(batch)]
    prefixes = [r.choice([0, r.randint(0, 300), 127, 128, 129]) for _ in range(batch)]
    case = synth.mla_case(seed=i, batch=batch, q_len_range=(1, 1), prefix_range=(0, 0), q_lens=q_lens,
                          prefixes=prefixes, slack_pages=r.randint(0, 5), poison=True)
    if case["total_q"] == 0:
        pytest.skip("no query token")
    check(case, *gpu_mla(case))


REPLAY_CASES = SMALL + [dict(batch=3, q_len_range=(40, 200), prefix_range=(300, 1500), slack_pages=4)]


@pytest.mark.parametrize("idx", range(len(REPLAY_CASES)))
def test_mla_replay_is_bit_identical_to_computing_s_twice(idx):
    """With max_kv_len, the second 256 output columns come from the first half's
    exported softmax weights, rescale factors and row sums instead of a second
    S = Q.K^T; the arithmetic is the one the second half's own task did, so the
    outputs and LSEs equal those of the call without the bound bit for bit."""
    case = synth.mla_case(seed=50 + idx, poison=True, **REPLAY_CASES[idx])
    a = gpu_mla(case, replay=False)
    b = gpu_mla(case, replay=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    check(case, *b)


def test_mla_replay_full_size_is_bit_identical():
    case = synth.mla_case(seed=0, **synth.MLA_WORKLOADS["mla_prefill_h16"])
    a = gpu_mla(case, replay=False)
    b = gpu_mla(case, replay=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_mla_export_overflow_is_reported():
    """max_kv_len below the longest kv_len: the export does not fit the
    workspace; error bit 2 is set, nothing outside the workspace is touched,
    and the first 256 output columns and the LSEs still match the oracle."""
    case = synth.mla_case(seed=23, batch=3, q_len_range=(30, 60), prefix_range=(400, 900))
    out, lse, err = _run_with(case, max_kv_len=100, fill=0xFF)
    assert err == 4
    T = case["total_q"]
    ref_out, ref_lse = np.full(out.shape, np.nan), np.full(lse.shape, np.nan)
    oracle.mla(case, 0, T, out=ref_out, lse=ref_lse)
    assert float(np.max(np.abs(out[:, :, :256] - ref_out[:, :, :256]))) <= TOL_OUT
    assert float(np.max(np.abs(lse - ref_lse))) <= TOL_LSE


@pytest.mark.parametrize("i", range(10))
def test_mla_replay_random_cases_are_bit_identical(i):
    """Seeded random batches (as test_mla_random_case_matches_oracle draws
    them): the replayed second half equals the two-task result bit for bit,
    and both match the oracle."""
    import random
    r = random.Random(7000 + i)
    batch = r.randint(1, 5)
    q_lens = [r.choice([0, 1, r.randint(1, 70), 8, 9, 16, 17]) for _ in range(batch)]
    prefixes = [r.choice([0, r.randint(0, 600), 127, 128, 129, 255, 256]) for _ in range(batch)]
    case = synth.mla_case(seed=100 + i, batch=batch, q_len_range=(1, 1), prefix_range=(0, 0), q_lens=q_lens,
                          prefixes=prefixes, slack_pages=r.randint(0, 5), poison=True)
    if case["total_q"] == 0:
        pytest.skip("no query token")
    a = gpu_mla(case, replay=False)
    b = gpu_mla(case, replay=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    check(case, *b)


def test_mla_long_sequence_shares_the_last_task_bin():
    """A 300,000-key prefix: both of its row tiles hold 2,344 key blocks of 128,
    above the 2,047 at which the task builder's block-count bins stop being
    distinct, and its export spans 2,345 blocks per row tile.  The replayed
    second half equals the two-task result bit for bit; every token of a short
    sequence beside it, and sampled (token, head) pairs at the long sequence's
    row-tile edges, match the oracle.  Heads are independent in the method, so
    one head of a token is the oracle run on the query sliced to that head."""
    case = synth.mla_case(seed=61, batch=2, q_len_range=(1, 1), prefix_range=(0, 0), q_lens=[24, 40],
                          prefixes=[300_000, 1_000], slack_pages=5, poison=True)
    a = gpu_mla(case, replay=False)
    b = gpu_mla(case, replay=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    got_out, got_lse = b
    check(case, got_out, got_lse, tokens=list(range(24, 64)))
    pairs = [(0, 0), (0, 11), (15, 4), (16, 15), (23, 7), (23, 8)]

    def one(th):
        t, h = th
        sub = dict(case, H=1, q_nope=np.ascontiguousarray(case["q_nope"][:, h:h + 1]),
                   q_pe=np.ascontiguousarray(case["q_pe"][:, h:h + 1]))
        o, l = oracle.mla(sub, t, t + 1, out=np.full((case["total_q"], 1, 512), np.nan),
                          lse=np.full((case["total_q"], 1), np.nan))
        return o[t, 0], l[t, 0]
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(len(pairs)) as ex:
        refs = list(ex.map(one, pairs))
    for (t, h), (ro, rl) in zip(pairs, refs):
        assert float(np.max(np.abs(got_out[t, h] - ro))) <= TOL_OUT, (t, h)
        assert abs(float(got_lse[t, h]) - float(rl)) <= TOL_LSE, (t, h)


def test_mla_batch_of_600_sequences():
    """600 sequences: the task builder's scans over the batch (256 sequences per pass, carried
    across passes), its tile loops and its export-block scan all take several passes.  Query
    lengths include 0 and the 16-token tile edges, prefixes 0 and the 128-key block edges.  The
    replay equals the two-task result bit for bit; the first and last token of every sequence
    match the oracle."""
    import random
    r = random.Random(8600)
    batch = 600
    q_lens = [r.choice([0, 1, 5, 16, 17, 40]) for _ in range(batch)]
    prefixes = [r.choice([0, 1, 127, 128, 300]) for _ in range(batch)]
    case = synth.mla_case(seed=86, batch=batch, q_len_range=(1, 1), prefix_range=(0, 0), q_lens=q_lens,
                          prefixes=prefixes, slack_pages=9, poison=True)
    a = gpu_mla(case, replay=False)
    b = gpu_mla(case, replay=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    qo = case["qo_indptr"]
    tokens = sorted({int(t) for i in range(batch) if qo[i + 1] > qo[i] for t in (qo[i], qo[i + 1] - 1)})
    check(case, *b, tokens=tokens)


def test_mla_one_long_query_sequence():
    """One sequence of 4,096 query tokens over a 100-key prefix: 256 row tiles of one sequence
    whose block counts run from 1 to 33, so the causal diagonal crosses every position inside a
    key block.  The replay equals the two-task result bit for bit; tokens at row-tile edges and
    at key-block edges match the oracle."""
    case = synth.mla_case(seed=87, batch=1, q_len_range=(1, 1), prefix_range=(0, 0), q_lens=[4096],
                          prefixes=[100], slack_pages=4, poison=True)
    a = gpu_mla(case, replay=False)
    b = gpu_mla(case, replay=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # token t sees keys 0 .. 100 + t: edges of 16-token tiles and of 128-key blocks
    tokens = sorted({0, 1, 15, 16, 27, 28, 155, 156, 2047, 2048, 4080, 4095} |
                    {128 * k - 101 for k in range(1, 33)} | {128 * k - 100 for k in range(1, 33)})
    check(case, *b, tokens=[t for t in tokens if 0 <= t < 4096])
