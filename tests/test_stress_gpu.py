"""Parity under perturbed timing (pkv_set_stress_delay).

Every kernel of the library orders its consumers after their data with
barriers.  A wait that relies on timing instead -- for instance a parity wait
on a barrier that can run two phases behind the expected one -- passes the
ordinary parity tests as long as every role runs at its usual pace, and fails
once one of them is slow.  These tests slow the copy producers (a pause after
each issued page, Q chunk or key slot) or the consumers (decode consumer warps
after each page; the MLA MMA thread after each ring slot and its softmax warps
after each key block) and compare the results with the fp64 oracle: the MLA
prefill kernel's task epilogue once had such a wait, and a run with a slowed
producer made every small MLA case fail.
"""
import numpy as np
import pytest

from paged_kv_gqa_table_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TOL = {synth.F16: 4e-3, synth.BF16: 1.6e-2}


@pytest.fixture
def stress():
    from paged_kv_gqa_table_gb300 import binding as B
    def set_delay(producer_ns, consumer_ns):
        B.pkv_set_stress_delay(producer_ns, consumer_ns)
    yield set_delay
    B.pkv_set_stress_delay(0, 0)


MLA_CASES = [
    dict(batch=3, q_len_range=(1, 20), prefix_range=(0, 300), slack_pages=7),
    dict(batch=2, q_len_range=(8, 8), prefix_range=(120, 136), slack_pages=3),
    dict(batch=2, q_len_range=(100, 140), prefix_range=(250, 270), sm_scale=1.0 / 24.0),
    dict(batch=4, q_len_range=(20, 60), prefix_range=(300, 700)),
]


@pytest.mark.parametrize("delays", [(300, 0), (2000, 0), (0, 1000)])
@pytest.mark.parametrize("idx", range(len(MLA_CASES)))
def test_mla_parity_with_slow_roles(stress, idx, delays):
    from paged_kv_gqa_table_gb300 import tensors as T
    import oracle
    stress(*delays)
    case = synth.mla_case(seed=40 + idx, poison=True, **MLA_CASES[idx])
    desc = T.mla_desc(case)
    ws = T.mla_workspace_for(desc)
    out, lse = T.mla_paged_prefill(case, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "device error word set"
    ro, rl = oracle.mla(case)
    got, gl = out.double().cpu().numpy(), lse.double().cpu().numpy()
    assert float(np.max(np.abs(got - ro))) <= TOL[synth.BF16]
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(gl), fin)
    assert float(np.max(np.abs(gl[fin] - rl[fin]), initial=0.0)) <= 1e-3


DECODE_CASES = [
    dict(B=16, Hq=32, Hkv=8, D=128, dtype=synth.BF16, layout=synth.NHD, ctx_range=(1, 3000)),
    dict(B=12, Hq=24, Hkv=4, D=256, dtype=synth.F16, layout=synth.VLLM, ctx_range=(0, 2500)),
    dict(B=16, Hq=32, Hkv=8, D=128, dtype=synth.BF16, layout=synth.NHD, ctx_range=(1, 3000),
         kv_dtype=synth.FP8_E4M3),
    dict(B=12, Hq=32, Hkv=8, D=128, dtype=synth.BF16, layout=synth.NHD, ctx_range=(0, 2500), q_len=4),
]


@pytest.mark.parametrize("delays", [(1000, 0), (0, 1000)])
@pytest.mark.parametrize("device_plan", [False, True])
@pytest.mark.parametrize("idx", range(len(DECODE_CASES)))
def test_decode_parity_with_slow_roles(stress, idx, device_plan, delays):
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import tensors as T
    import oracle
    stress(*delays)
    case = synth.decode_case(seed=70 + idx, block_size=16, max_blocks_per_seq=200, poison=True,
                             **DECODE_CASES[idx])
    opts = B.make_opts(device_plan=True) if device_plan else None
    desc = T.decode_desc(case)
    ws = T.workspace_for(desc, opts)
    dev = T.upload_decode_case(case)
    out = torch.full(case["q"].shape, float("nan"), dtype=T.TORCH_DTYPE[case["dtype"]], device="cuda")
    B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                 dev["context_lens"], case["scale"], out, ws, opts=opts)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "device error word set"
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert float(np.max(np.abs(got - oracle.decode(case)))) <= TOL[case["dtype"]]
