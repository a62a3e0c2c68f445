"""The decode entry point that allocates nothing (pkv_paged_decode_attention_static).

It exists for callers that may not allocate device memory when they run a
decode step (a plugin's enqueue hook, an engine with a fixed memory pool, a
latency-critical loop).  It keeps the decode step's scratch (error word and
split partials) in the library's own static device array instead of a
caller workspace.  These tests call it through the C ABI and compare it with
the fp64 oracle and with the workspace entry point on the same inputs, twice
in a row with different problems (the array keeps the previous call's
contents, which must not matter), within the tolerance the parity tests use.
The file is named to be collected last.
"""
import numpy as np
import pytest

from paged_kv_gqa_table_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TOL = {synth.F16: 4e-3, synth.BF16: 1.6e-2}


def _run_both(case, opts=None):
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import tensors as T
    dev = T.upload_decode_case(case)
    desc = T.decode_desc(case)
    ref = T.paged_decode_attention(case, dev=dev, opts=opts)
    out = torch.full_like(ref, float("nan"))
    B.pkv_paged_decode_attention_static(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                        dev["context_lens"], case["scale"], out, opts=opts)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), ref.double().cpu().numpy()


def _static_call(case, opts=None):
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import tensors as T
    dev = T.upload_decode_case(case)
    out = torch.full(case["q"].shape, float("nan"), dtype=torch.bfloat16 if case["dtype"] == synth.BF16
                     else torch.float16, device="cuda")
    B.pkv_paged_decode_attention_static(T.decode_desc(case), dev["q"], dev["k_cache"], dev["v_cache"],
                                        dev["block_table"], dev["context_lens"], case["scale"], out, opts=opts)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def test_static_scratch_matches_oracle_and_workspace_entry_point_twice():
    from paged_kv_gqa_table_gb300 import binding as B
    import oracle
    # Both calls need scratch: their sequences are split, so the split
    # partials live in the static array (default plan first, then fixed
    # 512-token partitions).
    first = synth.decode_case(seed=0, B=16, Hq=32, Hkv=8, D=128, block_size=16, dtype=synth.BF16,
                              layout=synth.NHD, ctx_range=(1, 4096), max_blocks_per_seq=256)
    second = synth.decode_case(seed=1, B=24, Hq=24, Hkv=4, D=256, block_size=16, dtype=synth.F16,
                               layout=synth.VLLM, ctx_range=(600, 3000), max_blocks_per_seq=200)
    for case, opts in ((first, None), (second, B.make_opts(partition_tokens=512))):
        got, ref = _run_both(case, opts)
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - oracle.decode(case)))) <= TOL[case["dtype"]]
        assert float(np.max(np.abs(got - ref))) <= TOL[case["dtype"]]


def test_static_scratch_refuses_problems_that_do_not_fit():
    from paged_kv_gqa_table_gb300 import binding as B
    # 256 sequences x 64 heads x 256 fixed partitions of fp32 partials is far beyond 32 MiB
    desc = B.make_desc(256, 64, 8, 128, 16, 8192, 300000, 131072, 256 * 131072, synth.BF16)
    opts = B.make_opts(partition_tokens=512)
    assert B.pkv_decode_workspace_size(desc, opts) > B.PKV_STATIC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.PkvError) as e:
        B.pkv_paged_decode_attention_static(desc, dummy, dummy, dummy, dummy, dummy, 0.1, dummy, opts=opts)
    assert e.value.status == B.PKV_WORKSPACE_TOO_SMALL


def test_static_scratch_keeps_a_device_plan_for_reuse():
    # A device-planned call (PKV_DECODE_DEVICE_PLAN), then one that states the plan is
    # ready (PKV_DECODE_PLAN_READY) with new queries: both match the oracle.
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import tensors as T
    import oracle
    case = synth.decode_case(seed=3, B=12, Hq=16, Hkv=4, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, ctx_range=(1, 2000), max_blocks_per_seq=128)
    second = dict(case, q=synth.normal_bits(4, 3, case["q"].size, synth.BF16).reshape(case["q"].shape))
    desc = T.decode_desc(case)
    for c, opts in ((case, B.make_opts(device_plan=True)), (second, B.make_opts(plan_ready=True))):
        dev = T.upload_decode_case(c)
        out = torch.full(c["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        B.pkv_paged_decode_attention_static(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                            dev["context_lens"], c["scale"], out, opts=opts)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - oracle.decode(c)))) <= TOL[synth.BF16]


def test_static_scratch_refuses_a_plan_another_call_replaced():
    # A device plan made by one static call, then a static call of another
    # problem (its partials overwrite the array): reusing the first plan is
    # refused on the host; planning again works and matches the oracle.
    from paged_kv_gqa_table_gb300 import binding as B
    import oracle
    case = synth.decode_case(seed=5, B=12, Hq=16, Hkv=4, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, ctx_range=(1, 2000), max_blocks_per_seq=128)
    other = synth.decode_case(seed=6, B=20, Hq=32, Hkv=8, D=128, block_size=16, dtype=synth.BF16,
                              layout=synth.NHD, ctx_range=(100, 3000), max_blocks_per_seq=200)
    got = _static_call(case, B.make_opts(device_plan=True))
    assert float(np.max(np.abs(got - oracle.decode(case)))) <= TOL[synth.BF16]
    got = _static_call(other)
    assert float(np.max(np.abs(got - oracle.decode(other)))) <= TOL[synth.BF16]
    with pytest.raises(B.PkvError) as e:
        _static_call(case, B.make_opts(plan_ready=True))
    assert e.value.status == B.PKV_INVALID_ARG
    got = _static_call(case, B.make_opts(device_plan=True))
    got2 = _static_call(case, B.make_opts(plan_ready=True))
    for g in (got, got2):
        assert float(np.max(np.abs(g - oracle.decode(case)))) <= TOL[synth.BF16]


def test_static_scratch_error_word_reads_back_and_survives_rejected_calls():
    # The error word of the last static call is readable without allocating
    # in the library; a call rejected by the argument checks touches nothing.
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import tensors as T
    import oracle
    case = synth.decode_case(seed=7, B=8, Hq=32, Hkv=8, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, ctx_range=(1, 3000), max_blocks_per_seq=200)
    got = _static_call(case)
    assert float(np.max(np.abs(got - oracle.decode(case)))) <= TOL[synth.BF16]
    word = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    B.pkv_static_scratch_error(word)
    torch.cuda.synchronize()
    assert int(word.item()) == 0
    dev = T.upload_decode_case(case)
    out = torch.empty(case["q"].shape, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.PkvError) as e:   # q missing: refused before anything is enqueued
        B.pkv_paged_decode_attention_static(T.decode_desc(case), None, dev["k_cache"], dev["v_cache"],
                                            dev["block_table"], dev["context_lens"], case["scale"], out)
    assert e.value.status == B.PKV_INVALID_ARG
    host = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    B.pkv_static_scratch_error(host)
    torch.cuda.synchronize()
    assert int(host.item()) == 0
