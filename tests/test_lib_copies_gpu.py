"""Two copies of libpkv in one process keep separate state.

Each launcher raises its kernel's dynamic shared-memory limit once per device
and remembers that in a static flag; if that flag were an exported symbol the
dynamic linker would share it between the copies and the second copy would
launch a kernel whose limit was never raised (a launch error for phase 1 of a
D=128 problem, which needs more than 48 KB).  Both copies must give the same
bits.
"""
import ctypes
import shutil

import numpy as np
import pytest

from paged_kv_gqa_table_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def test_second_copy_of_the_library_launches(tmp_path):
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import tensors as T
    case = synth.decode_case(seed=5, B=8, Hq=32, Hkv=8, D=128, block_size=16, dtype=synth.BF16,
                             layout=synth.NHD, ctx_range=(100, 2000), max_blocks_per_seq=128)
    first = T.paged_decode_attention(case).cpu()
    copy = tmp_path / "libpkv_copy.so"
    shutil.copyfile(B.LIB_PATH, copy)
    saved_path, saved_lib = B.LIB_PATH, B._lib
    try:
        B.LIB_PATH, B._lib = str(copy), None
        lib = B.load()
        assert ctypes.cast(lib.pkv_version, ctypes.c_void_p).value != \
            ctypes.cast(saved_lib.pkv_version, ctypes.c_void_p).value
        second = T.paged_decode_attention(case).cpu()
        torch.cuda.synchronize()
    finally:
        B.LIB_PATH, B._lib = saved_path, saved_lib
    assert torch.equal(first.view(torch.int16), second.view(torch.int16))
