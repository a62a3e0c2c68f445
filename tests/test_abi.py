"""Host-side tests of the C ABI (no GPU needed): the library loads, exports
every function include/pkv.h declares, plans splits by its documented rule
(checked against an independent restatement), sizes workspaces, and rejects
bad arguments before launching anything."""
import ctypes
import os
import random
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from paged_kv_gqa_table_gb300 import binding, build
    if not os.path.exists(binding.LIB_PATH):
        build.build()
    binding.load()
    return binding


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(pkv_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_library_exports_every_declared_function(B):
    names = declared_functions()
    assert "pkv_paged_decode_attention" in names and len(names) >= 8
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(B.FUNCTIONS) <= set(names)


def test_version_and_status_strings(B):
    assert B.pkv_version() == 9
    assert B.status_string(0) == "ok"
    assert B.status_string(5) == "bad block table"
    assert B.status_string(99) == "unknown status"


def test_stress_delay_accepts_its_range_on_the_host(B):
    # a host setting only: no GPU is touched; the value is left at 0 (off)
    B.pkv_set_stress_delay(1000000, 1000000)
    B.pkv_set_stress_delay(0, 0)
    for bad in ((1000001, 0), (0, 1000001)):
        with pytest.raises(B.PkvError) as e:
            B.pkv_set_stress_delay(*bad)
        assert e.value.status == B.PKV_INVALID_ARG


def desc(lib, **kw):
    base = dict(B=64, Hq=32, Hkv=8, D=128, block_size=16, max_blocks_per_seq=256, num_blocks=9000,
                max_context_len=4096, sum_context_len=131072, dtype=1, layout=0, x_pack=8)
    base.update(kw)
    return lib.make_desc(**base)


def ref_rows_per_cta(d):
    """Query rows per CTA of the documented column tiling: 16, or 8 for D = 256 or <= 8 rows."""
    R = d.Hq // d.Hkv * d.q_len
    return 16 if (R > 8 and d.D <= 128) else 8


def ref_row_tiles(d):
    return -(-(d.Hq // d.Hkv * d.q_len) // ref_rows_per_cta(d))


def ref_heads_per_cta(d):
    """2 for the documented head pairs (FP8, D = 128, even Hkv, <= 4 query rows per KV head), else 1."""
    pair = d.kv_dtype == 2 and d.D == 128 and d.Hkv % 2 == 0 and 2 * (d.Hq // d.Hkv) * d.q_len <= 8
    return 2 if pair else 1


def ref_plan(d, num_sms, P_forced=0, ns_forced=0):
    """Independent restatement of the planner's documented rule."""
    bs = d.block_size
    up = lambda a: -(-a // bs) * bs
    if P_forced:
        P = P_forced
    elif ns_forced:
        P = up(-(-max(d.max_context_len, 1) // ns_forced))
    else:
        P = up(min(max(d.max_context_len, 1), 512 * ref_rows_per_cta(d) // 8 * ref_heads_per_cta(d)))
        while P > 4 * bs and d.Hkv * ref_row_tiles(d) * -(-max(d.sum_context_len, 1) // P) < 6 * num_sms:
            P = max(4 * bs, up(P // 2))
    return max(1, -(-d.max_context_len // P)), P


def test_plan_matches_the_documented_rule(B):
    rng = random.Random(0)
    for _ in range(2000):
        Hkv = rng.choice([1, 2, 4, 8])
        Bn = rng.randint(1, 300)
        mbps = rng.randint(1, 9000)
        maxn = rng.randint(0, mbps * 16)
        s = rng.randint(maxn, max(maxn, maxn * Bn))
        d = desc(B, B=Bn, Hkv=Hkv, Hq=Hkv * rng.choice([1, 2, 4, 6, 8, 12, 32]), D=rng.choice([64, 128, 256]),
                 max_blocks_per_seq=mbps, max_context_len=maxn, sum_context_len=s,
                 q_len=rng.choice([1, 1, 2, 3, 4, 8]), kv_dtype=rng.choice([0, 2]))
        sms = rng.choice([1, 76, 148, 152])
        mode = rng.randint(0, 2)
        if mode == 0:
            assert B.pkv_plan_splits(d, None, sms) == ref_plan(d, sms)
        elif mode == 1:
            P = 16 * rng.randint(1, 300)
            assert B.pkv_plan_splits(d, B.make_opts(partition_tokens=P), sms) == ref_plan(d, sms, P_forced=P)
        else:
            k = rng.randint(1, 400)
            assert B.pkv_plan_splits(d, B.make_opts(num_splits=k), sms) == ref_plan(d, sms, ns_forced=k)


def test_named_workload_plans(B):
    # 152 SMs: the decode workloads split into 512-token partitions.
    assert B.pkv_plan_splits(desc(B), None, 152) == (8, 512)
    long_ctx = desc(B, B=4, max_blocks_per_seq=8192, max_context_len=131072, sum_context_len=4 * 81920)
    assert B.pkv_plan_splits(long_ctx, None, 152) == (256, 512)
    # the FP8 variant of the default runs head pairs: 512 tokens per KV head of the CTA
    assert B.pkv_plan_splits(desc(B, kv_dtype=2), None, 152) == (4, 1024)
    # ... but not with an odd KV head count or a full column tile per KV head
    assert B.pkv_plan_splits(desc(B, kv_dtype=2, Hkv=1, Hq=4), None, 152)[1] < 1024
    assert B.pkv_plan_splits(desc(B, kv_dtype=2, q_len=2), None, 152) == (8, 512)
    tiny = desc(B, B=2, Hq=4, Hkv=2, D=64, max_blocks_per_seq=8, num_blocks=16, max_context_len=100,
                sum_context_len=137, dtype=0)
    assert B.pkv_plan_splits(tiny, None, 152) == (2, 64)


def test_workspace_size(B):
    al = lambda x: (x + 255) // 256 * 256
    d = desc(B)
    # header | m, l [B][Hq][NS] | acc [B][Hq][NS][D]
    ns, P = B.pkv_plan_splits(d, None, 152)
    rows = 64 * 32 * ns
    assert B.pkv_decode_workspace_size(d, None, 152) == 256 + 2 * al(rows * 4) + al(rows * 128 * 4)
    single = B.make_opts(num_splits=1)
    assert B.pkv_decode_workspace_size(d, single, 152) == 256
    # several query tokens: m, l [B][q_len][Hq][NS], acc [B][q_len][Hq][NS][D]
    d4 = desc(B, q_len=4)
    ns, P = B.pkv_plan_splits(d4, None, 152)
    rows = 64 * 4 * 32 * ns
    assert ns > 1 and B.pkv_decode_workspace_size(d4, None, 152) == 256 + 2 * al(rows * 4) + al(rows * 128 * 4)


@pytest.mark.parametrize("field,value,status", [
    ("Hkv", 3, 1), ("Hq", 0, 1), ("D", 96, 2), ("block_size", 32, 2), ("dtype", 7, 1), ("layout", 2, 1),
    ("max_context_len", 256 * 16 + 1, 1), ("B", -1, 1), ("num_blocks", 0, 1), ("sum_context_len", -5, 1),
    ("q_len", 0, 1), ("q_len", -2, 1), ("q_len", 1 << 27, 2),
])
def test_bad_descriptions_are_rejected(B, field, value, status):
    d = desc(B, **{field: value})
    with pytest.raises(B.PkvError) as e:
        B.pkv_plan_splits(d, None, 152)
    assert e.value.status == status


def test_device_plan_options(B):
    al = lambda x: (x + 255) // 256 * 256
    d = desc(B)
    ns, P = B.pkv_plan_splits(d, None, 152)
    plain = B.pkv_decode_workspace_size(d, None, 152)
    # phase 1 plans on the device itself: the workspace is that of the bounds' host plan, plus the
    # split table the plan is kept in for the calls that reuse it (16 bytes per sequence and split)
    dev = B.pkv_decode_workspace_size(d, B.make_opts(device_plan=True), 152)
    assert dev == plain + al(d.B * ns * 16)
    assert B.pkv_decode_workspace_size(d, B.make_opts(plan_ready=True), 152) == dev
    assert B.pkv_plan_splits(d, B.make_opts(device_plan=True), 152) == (ns, P)
    assert B.pkv_plan_splits(d, B.make_opts(plan_ready=True), 152) == (ns, P)   # flags 3
    assert B.make_opts(plan_ready=True).flags == B.PKV_DECODE_DEVICE_PLAN | B.PKV_DECODE_PLAN_READY
    for bad in (2, 4, 6, 1 << 30, -1):   # 2: plan reuse without the device plan
        with pytest.raises(B.PkvError) as e:
            B.pkv_plan_splits(d, B.make_opts(flags=bad), 152)
        assert e.value.status == B.PKV_INVALID_ARG
    # phase 1 alone keeps the host plan's partial layout
    st = B.raw_status("pkv_decode_partials", ctypes.byref(d), ctypes.byref(B.make_opts(device_plan=True)),
                      None, None, None, None, None, ctypes.c_float(0.1), None, None, None, 8, None, None, None)
    assert st == B.PKV_UNSUPPORTED


def test_large_groups_take_row_tiles(B):
    # Any group size plans: its query rows are covered by several CTAs.
    assert B.pkv_plan_splits(desc(B, Hq=8 * 17), None, 152) == ref_plan(desc(B, Hq=8 * 17), 152)
    assert B.pkv_plan_splits(desc(B, Hq=8 * 12, D=256), None, 152) == ref_plan(desc(B, Hq=8 * 12, D=256), 152)
    mqa = desc(B, Hq=64, Hkv=1, q_len=3)
    assert ref_row_tiles(mqa) == 12 and B.pkv_plan_splits(mqa, None, 152) == ref_plan(mqa, 152)
    # 16 query rows per CTA start from 1024-token partitions: the 4-token Llama-3-shaped step
    assert B.pkv_plan_splits(desc(B, q_len=4), None, 152) == (4, 1024)
    with pytest.raises(B.PkvError) as e:
        B.pkv_plan_splits(desc(B, layout=1, x_pack=4), None, 152)
    assert e.value.status == 1


def test_pointer_checks_happen_before_any_launch(B):
    d = desc(B)
    P = ctypes.c_void_p
    good = 1 << 20       # aligned fake addresses: the calls must fail before using them
    args = lambda **kw: [kw.get(k, good) for k in ("q", "k", "v", "t", "c")]
    for bad in (dict(q=None), dict(k=good + 8), dict(v=None), dict(t=good + 2), dict(c=None)):
        q, k, v, t, c = args(**bad)
        st = B.raw_status("pkv_paged_decode_attention", ctypes.byref(d), None, q, k, v, t, c,
                          ctypes.c_float(0.1), good, good, 1 << 30, None)
        assert st == B.PKV_INVALID_ARG, bad
    st = B.raw_status("pkv_paged_decode_attention", ctypes.byref(d), None, good, good, good, good, good,
                      ctypes.c_float(0.1), good + 4, good, 1 << 30, None)
    assert st == B.PKV_INVALID_ARG       # misaligned out
    st = B.raw_status("pkv_paged_decode_attention", ctypes.byref(d), None, good, good, good, good, good,
                      ctypes.c_float(float("nan")), good, good, 1 << 30, None)
    assert st == B.PKV_INVALID_ARG       # non-finite scale
    st = B.raw_status("pkv_paged_decode_attention", None, None, good, good, good, good, good,
                      ctypes.c_float(0.1), good, good, 1 << 30, None)
    assert st == B.PKV_INVALID_ARG
    # partial arrays and combine arguments
    st = B.raw_status("pkv_combine", ctypes.byref(d), 500, 9, good, good, good, good, good, None)
    assert st == B.PKV_INVALID_ARG       # 500 is not a multiple of the page size
    st = B.raw_status("pkv_combine", ctypes.byref(d), 512, 7, good, good, good, good, good, None)
    assert st == B.PKV_INVALID_ARG       # 7 splits of 512 cannot cover 4096 tokens
    st = B.raw_status("pkv_validate_block_table", ctypes.byref(d), good, good, None, None)
    assert st == B.PKV_INVALID_ARG
    # an empty pool (every context empty) may come without caches, a column-less table without a table
    empty = desc(B, num_blocks=0, max_context_len=0, sum_context_len=0, max_blocks_per_seq=0)
    st = B.raw_status("pkv_paged_decode_attention", ctypes.byref(empty), None, good, None, None, None, good,
                      ctypes.c_float(0.1), good, good, 1 << 30, None)
    assert st != B.PKV_INVALID_ARG       # (no GPU here: the launch itself reports a CUDA error)
    with_pool = desc(B, max_context_len=0, sum_context_len=0)
    st = B.raw_status("pkv_paged_decode_attention", ctypes.byref(with_pool), None, good, None, good, good, good,
                      ctypes.c_float(0.1), good, good, 1 << 30, None)
    assert st == B.PKV_INVALID_ARG       # a pool was described: its caches are required


def test_empty_batch_is_a_no_op(B):
    d = desc(B, B=0, max_context_len=0, sum_context_len=0)
    st = B.raw_status("pkv_paged_decode_attention", ctypes.byref(d), None, None, None, None, None, None,
                      ctypes.c_float(0.1), None, None, 0, None)
    assert st == B.PKV_OK


def test_mla_workspace_size_and_argument_checks(B):
    al = lambda x: (x + 255) // 256 * 256
    # header | work list (one 16-byte entry per 16-token row tile and output
    # half) | per-sequence first tile (batch + 1 ints) and first staged row |
    # staged rows: every sequence's keys start on a multiple of 128 rows, so
    # room for nnz rows plus at most 127 zero rows per sequence (none without keys)
    for nnz, batch in ((0, 8), (1, 1), (8070, 8), (123457, 300)):
        d = B.make_mla_desc(2866, batch, 9000, nnz)
        rows = nnz + 128 * batch if nnz > 0 else 0
        tasks = 2 * ((2866 + 15) // 16 + batch)
        want = 256 + al(tasks * 16) + al((batch + 1) * 4) + al(batch * 4) + al(rows * 1152)
        assert B.pkv_mla_workspace_size(d) == want
        # with a max_kv_len bound: per row tile an export base and 1 KB of row sums,
        # per possible exported key block 64 KB of P, 1 KB of factors, 16 flag bytes
        for max_kv in (1, 128, 129, 2124):
            e = tasks // 2 * ((max_kv + 127) // 128)
            want_r = want + al(tasks // 2 * 4) + al(e * 65536) + al(e * 1024) + al(e * 16) + al(tasks // 2 * 1024)
            assert B.pkv_mla_workspace_size(B.make_mla_desc(2866, batch, 9000, nnz, max_kv_len=max_kv)) == want_r
    for bad in (dict(nnz=-1), dict(total_q=-1), dict(num_pages=-3), dict(max_kv_len=-1)):
        kw = dict(total_q=100, batch=2, num_pages=50, nnz=40)
        kw.update(bad)
        with pytest.raises(B.PkvError) as e:
            B.pkv_mla_workspace_size(B.make_mla_desc(**kw))
        assert e.value.status == B.PKV_INVALID_ARG
    with pytest.raises(B.PkvError) as e:
        B.pkv_mla_workspace_size(B.make_mla_desc(100, 2, 50, 40, num_heads=8))
    assert e.value.status == B.PKV_UNSUPPORTED
    d = B.make_mla_desc(100, 2, 50, 40)
    need = B.pkv_mla_workspace_size(d)
    good = 1 << 20
    args = lambda ws, n: [ctypes.byref(d), good, good, good, good, good, good, good, ctypes.c_float(0.1), good, good,
                          ws, n, None]
    assert B.raw_status("pkv_mla_paged_prefill", *args(good, need - 1)) == B.PKV_WORKSPACE_TOO_SMALL
    assert B.raw_status("pkv_mla_paged_prefill", *args(good + 128, need)) == B.PKV_INVALID_ARG   # misaligned
    assert B.raw_status("pkv_mla_paged_prefill", *args(None, need)) == B.PKV_INVALID_ARG


def test_library_exports_only_the_declared_functions(B):
    # Built with hidden visibility: any other exported symbol (a template's
    # static "attribute already set" flag, say) would be shared with a second
    # copy of the library loaded in the same process.
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set()
    for line in out.splitlines():
        parts = line.split()
        if len(parts) == 3 and parts[1] in "TtDdBbRrVvWwu":
            exported.add(parts[2])
    ours = {n for n in exported if not n.startswith("_")}
    assert ours == set(declared_functions()), sorted(ours ^ set(declared_functions()))
    assert not any(parts.split()[1] == "u" for parts in out.splitlines() if len(parts.split()) == 3)


def test_fp8_descriptions(B):
    base = dict(B=8, Hq=32, Hkv=8, D=128, block_size=16, max_blocks_per_seq=64, num_blocks=500,
                max_context_len=1000, sum_context_len=8000, dtype=1)
    ok = B.make_desc(**base, kv_dtype=B.PKV_FP8_E4M3, k_scale=0.1, v_scale=0.2)
    assert B.pkv_plan_splits(ok, None, 152) == B.pkv_plan_splits(B.make_desc(**base), None, 152)
    assert B.pkv_decode_workspace_size(ok, None, 152) == B.pkv_decode_workspace_size(B.make_desc(**base), None, 152)
    for kw, status in ((dict(kv_dtype=3), B.PKV_INVALID_ARG), (dict(kv_dtype=1), B.PKV_INVALID_ARG),
                       (dict(kv_dtype=2, k_scale=0.0, v_scale=1.0), B.PKV_INVALID_ARG),
                       (dict(kv_dtype=2, k_scale=1.0, v_scale=float("nan")), B.PKV_INVALID_ARG),
                       (dict(kv_dtype=2, k_scale=1.0, v_scale=1.0, layout=1), B.PKV_UNSUPPORTED)):
        with pytest.raises(B.PkvError) as e:
            B.pkv_plan_splits(B.make_desc(**{**base, **kw}), None, 152)
        assert e.value.status == status, kw


def test_misaligned_alibi_slopes_are_rejected(B):
    d = desc(B)
    good = 1 << 20
    opts = B.pkv_decode_opts(0, 0, 0, None, None, good + 2)
    st = B.raw_status("pkv_paged_decode_attention", ctypes.byref(d), ctypes.byref(opts), good, good, good, good, good,
                      ctypes.c_float(0.1), good, good, 1 << 30, None)
    assert st == B.PKV_INVALID_ARG


def test_device_planner_condition_equals_the_host_rule():
    # The device plan tests "enough work items" as sum > (ceil(target / (Hkv*RT)) - 1) * P
    # instead of the host's Hkv * RT * ceil(sum / P) >= target (no 64-bit division on the
    # device); the two must agree for every operand, and so must its overflow-safe ceilings.
    rng = random.Random(1)
    cdiv = lambda a, b: (a - 1) // b + 1 if a > 0 else 0
    for _ in range(200000):
        hr = rng.choice([1, 2, 4, 8, 12, 64, 1000]) * rng.randint(1, 3)
        P = 16 * rng.randint(4, 4096)
        target = 6 * rng.choice([1, 76, 148, 152, 160])
        s = rng.choice([rng.randint(1, 10 ** 4), rng.randint(1, 10 ** 8), rng.randint(1, 10 ** 12)])
        host = hr * -(-s // P) >= target
        need = -(-target // hr)
        assert host == (s > (need - 1) * P), (hr, P, target, s)
        n, k = rng.randint(0, 2 ** 31 - 1), rng.randint(1, 2 ** 20)
        assert cdiv(n, k) == -(-n // k)
