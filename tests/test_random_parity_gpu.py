"""Randomised GPU parity: seeded random small decode problems over every feature
combination -- head dim, layout, dtype, FP8 caches, group size, query tokens per
sequence, ALiBi, forced partitions or split counts, the device plan with exact or
capacity bounds, empty and full contexts -- each checked against the fp64 oracle
(max |diff| <= 4e-3 fp16, <= 1.6e-2 bf16) with the device error word clear.
"""
import random

import numpy as np
import pytest

import oracle
from paged_kv_gqa_table_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TOL = {synth.F16: 4e-3, synth.BF16: 1.6e-2}


def draw(i):
    r = random.Random(7000 + i)
    D = r.choice([64, 128, 256])
    layout = r.choice([synth.NHD, synth.NHD, synth.VLLM])
    cfg = dict(D=D, layout=layout, dtype=r.choice([synth.F16, synth.BF16]),
               kv8=layout == synth.NHD and r.random() < 0.3, Hkv=r.choice([1, 2, 3, 4]),
               G=r.choice([1, 2, 3, 4, 5, 6, 8, 12, 16, 20, 32]), q_len=r.choice([1, 1, 1, 2, 3, 4, 5, 8]),
               B=r.randint(1, 6), mbps=r.randint(1, 24))
    cfg["lens"] = [min(cfg["mbps"] * 16, r.choice([0, 1, r.randint(0, cfg["mbps"] * 16), cfg["mbps"] * 16,
                                                   r.randint(0, 40)])) for _ in range(cfg["B"])]
    cfg.update(alibi=r.random() < 0.3, P=r.choice([0, 0, 0, 16, 48, 64, 128, 512]), ns=r.choice([0, 0, 0, 3]),
               device_plan=r.random() < 0.3, slack=r.randint(0, 4))
    cfg["loose"] = cfg["device_plan"] and r.random() < 0.7
    return cfg


@pytest.mark.parametrize("i", range(120))
def test_random_case_matches_oracle(i):
    from paged_kv_gqa_table_gb300 import binding as B, tensors as T
    c = draw(i)
    extra = dict(kv_dtype=synth.FP8_E4M3) if c["kv8"] else {}
    case = synth.decode_case(seed=i, B=c["B"], Hq=c["G"] * c["Hkv"], Hkv=c["Hkv"], D=c["D"], block_size=16,
                             dtype=c["dtype"], layout=c["layout"], context_lens=c["lens"],
                             max_blocks_per_seq=c["mbps"], slack_pages=c["slack"], poison=True, q_len=c["q_len"],
                             **extra)
    desc = T.decode_desc(case)
    if c["loose"]:
        if case["num_blocks"] == 0:
            pytest.skip("a positive context bound on an empty pool is an argument error")
        desc.max_context_len = c["mbps"] * 16
        desc.sum_context_len = c["B"] * c["mbps"] * 16
    slopes = None
    if c["alibi"]:
        Hq = c["G"] * c["Hkv"]
        case["alibi_slopes"] = (2.0 ** (-8.0 * np.arange(1, Hq + 1) / Hq)).astype(np.float32)
        slopes = torch.from_numpy(case["alibi_slopes"]).cuda()
    opts = B.make_opts(partition_tokens=c["P"], num_splits=0 if c["P"] else c["ns"], alibi_slopes=slopes,
                       device_plan=c["device_plan"])
    dev = T.upload_decode_case(case)
    out = torch.full(case["q"].shape, float("nan"), dtype=T.TORCH_DTYPE[c["dtype"]], device="cuda")
    ws = T.workspace_for(desc, opts)
    B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                 dev["context_lens"], case["scale"], out, ws, opts=opts)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "device error word set"
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got)), c
    worst = float(np.max(np.abs(got - oracle.decode(case)), initial=0.0))
    assert worst <= TOL[c["dtype"]], (worst, c)
