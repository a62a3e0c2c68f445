"""GPU tests of head pairs: FP8 caches at D = 128 whose query rows per KV head
(G * q_len) fill at most half a column tile run one CTA per pair of adjacent KV
heads, both heads' page slices in one ring stage.  Each query column takes its
scores from its own head's keys and adds only its own head's P.V product, so
the outputs must be bit-identical to running every KV head as a problem of its
own (one KV head: the one-head kernel), and within the decode tolerances of the
fp64 oracle.  Calls go through the C ABI.
"""
import numpy as np
import pytest

import oracle
from paged_kv_gqa_table_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TOL = {synth.F16: 4e-3, synth.BF16: 1.6e-2}


def run(case, P=0, alibi=None):
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import tensors
    slopes = torch.from_numpy(alibi).cuda() if alibi is not None else None
    out = tensors.paged_decode_attention(case, opts=B.make_opts(partition_tokens=P, alibi_slopes=slopes))
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def one_head(case, h):
    """KV head h of the case as a problem of its own (its G query heads, its cache slices)."""
    G = case["Hq"] // case["Hkv"]
    return dict(case, Hq=G, Hkv=1, q=np.ascontiguousarray(case["q"][..., h * G:(h + 1) * G, :]),
                k_cache=np.ascontiguousarray(case["k_cache"][:, h:h + 1]),
                v_cache=np.ascontiguousarray(case["v_cache"][:, h:h + 1]))


def slopes_for(Hq):
    return (2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq)).astype(np.float32)


# (G, q_len, Hkv, query dtype, ALiBi): every shape with G * q_len <= 4, including
# pairs that leave columns empty (G * q_len = 1 or 3)
SHAPES = [(4, 1, 2, synth.BF16, False), (4, 1, 4, synth.F16, False), (2, 2, 2, synth.F16, False),
          (1, 4, 2, synth.BF16, True), (3, 1, 6, synth.BF16, False), (1, 1, 2, synth.F16, False),
          (2, 1, 4, synth.BF16, True), (1, 3, 2, synth.BF16, False)]


@pytest.mark.parametrize("idx", range(len(SHAPES)))
@pytest.mark.parametrize("P", [64, 0])
def test_pairs_bit_identical_to_single_heads_and_match_oracle(idx, P):
    G, q_len, Hkv, dtype, alibi = SHAPES[idx]
    case = synth.decode_case(seed=700 + idx, B=7, Hq=G * Hkv, Hkv=Hkv, D=128, block_size=16, dtype=dtype,
                             layout=synth.NHD, context_lens=[0, 1, 17, 300, 513, 1000, 64],
                             max_blocks_per_seq=70, slack_pages=5, poison=True, q_len=q_len,
                             kv_dtype=synth.FP8_E4M3, k_scale=0.05, v_scale=0.08)
    slopes = slopes_for(case["Hq"]) if alibi else None
    if alibi:
        case["alibi_slopes"] = slopes
    if P == 0:
        from paged_kv_gqa_table_gb300 import binding as B
        from paged_kv_gqa_table_gb300 import tensors
        _, P = B.pkv_plan_splits(tensors.decode_desc(case))   # the one-head problems get the same partition
    got = run(case, P, slopes)
    for h in range(Hkv):
        sub = one_head(case, h)
        ref = run(sub, P, slopes[h * G:(h + 1) * G].copy() if alibi else None)
        assert np.array_equal(got[..., h * G:(h + 1) * G, :], ref), "head %d differs from its one-head run" % h
    want = oracle.decode(case)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - want)) <= TOL[dtype]


def test_pairs_partials_match_oracle():
    # the layered entry point under head pairs: 2 query tokens of a G = 2 group with ALiBi
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import tensors
    case = synth.decode_case(seed=720, B=5, Hq=8, Hkv=4, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, context_lens=[0, 3, 200, 700, 129], max_blocks_per_seq=50,
                             q_len=2, kv_dtype=synth.FP8_E4M3)
    slopes = slopes_for(8)
    case["alibi_slopes"] = slopes
    dev = tensors.upload_decode_case(case)
    NS_cap = 12
    acc = torch.empty((5, 2, 8, NS_cap, 128), device="cuda")
    m = torch.empty((5, 2, 8, NS_cap), device="cuda")
    l = torch.empty((5, 2, 8, NS_cap), device="cuda")
    P, ns = B.pkv_decode_partials(tensors.decode_desc(case), dev["q"], dev["k_cache"], dev["v_cache"],
                                  dev["block_table"], dev["context_lens"], case["scale"], acc, m, l, NS_cap,
                                  opts=B.make_opts(partition_tokens=64,
                                                   alibi_slopes=torch.from_numpy(slopes).cuda()))
    torch.cuda.synchronize()
    pm, pl, pacc = oracle.decode_partials(case, P, ns)
    gm, gl, gacc = m.cpu().numpy()[..., :ns], l.cpu().numpy()[..., :ns], acc.cpu().numpy()[..., :ns, :]
    live = pl > 0
    assert np.array_equal(live, gl > 0)
    assert np.all(np.isneginf(gm[~live])) and np.all(gl[~live] == 0) and np.all(gacc[~live] == 0)
    assert np.max(np.abs((gm[live] + np.log(gl[live])) - (pm[live] + np.log(pl[live])))) <= 1e-3
    assert np.max(np.abs(gacc[live] / gl[live][:, None] - pacc[live] / pl[live][:, None])) <= TOL[synth.BF16]


def test_odd_kv_heads_and_wide_groups_keep_one_head_per_cta():
    # Hkv = 3 (no pairing) and G * q_len = 8 (a full tile per head): the one-head kernel, within tolerance
    for kw in (dict(Hq=12, Hkv=3, q_len=1), dict(Hq=16, Hkv=2, q_len=1), dict(Hq=8, Hkv=2, q_len=2)):
        case = synth.decode_case(seed=730, B=4, D=128, block_size=16, dtype=synth.BF16, layout=synth.NHD,
                                 context_lens=[5, 400, 0, 1029], max_blocks_per_seq=70,
                                 kv_dtype=synth.FP8_E4M3, **kw)
        got = run(case, 128)
        assert np.max(np.abs(got - oracle.decode(case))) <= TOL[synth.BF16]
