"""The C ABI: the library loads, exports every declared symbol, and its
host-only logic behaves, all without a GPU (no compute call is made)."""

import ctypes
import os
import re

import pytest

from oracle import protocol as oproto
from tp_allreduce_persistent_b300 import build, llar

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "llar.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(llar_\w+)\s*\(", text, flags=re.M)))


def test_library_builds_and_exports_every_declared_symbol():
    build.build()
    names = declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(llar.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the Python binding wraps each of them under the same name
    assert all(hasattr(llar, n) for n in names if n != "llar_strerror")


def test_speed_of_light_formula_matches_page_numbers():
    # 2 x 0.306 us (L2 round trip) + 0.792 us (remote write) = 1.404 us on two GB200s
    assert abs(llar.llar_sol_bound_us(0.306, 0.792) - 1.404) < 1e-12


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_layout_constants(dtype):
    e = {"fp32": 4, "fp16": 2, "bf16": 2}[dtype]
    lb, pl, st = llar.llar_layout("ll", dtype, 4, 8192)
    assert (lb, pl * e) == (16, 8) and st == 2 * oproto.ll_staging_bytes(8192 * e)
    lb, pl, st = llar.llar_layout("ll128", dtype, 8, 1 << 20)
    assert lb == 128 and pl == oproto.ll128_payload_elems(dtype)
    assert st == 2 * oproto.ll128_round_staging_bytes(1 << 20, 8, dtype)
    lb, pl, st = llar.llar_layout("sentinel", dtype, 8, 32768)
    assert lb == 16 and pl * e == 16 and st == 2 * 8 * 8192


def test_protocol_selection_is_monotone_in_size():
    order = ["ll", "sentinel", "ll128", "fixed_oneshot", "fixed_twoshot"]
    last = 0
    for nbytes in [16, 4096, 16384, 65536, 1 << 18, 1 << 20, 1 << 22, 1 << 26]:
        p = llar.llar_select_protocol(8, "bf16", nbytes // 2)
        assert p in order
        assert order.index(p) >= last
        last = order.index(p)
    assert llar.llar_select_protocol(8, "bf16", 8192) == "ll"


def test_argument_checks_without_device():
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_init(1, "bf16", 1024)
    assert ei.value.code == llar.ERR_INVALID
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_init(9, "bf16", 1024)
    assert ei.value.code == llar.ERR_INVALID
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_init(4, 7, 1024)
    assert ei.value.code == llar.ERR_INVALID
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_set_launch(2, 48)
    assert ei.value.code == llar.ERR_INVALID
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_debug_inject(0, 9)
    assert ei.value.code == llar.ERR_INVALID
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_allreduce([0] * 4, [0] * 4, 16, "ll", stream=0)
    assert ei.value.code == llar.ERR_NOT_INIT
    assert llar.llar_get_status()[0] == llar.ERR_NOT_INIT
    assert llar.strerror(llar.ERR_TIMEOUT) == "a device-side wait timed out"


def test_init_without_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_init(8, "bf16", 1 << 20)
    assert ei.value.code == llar.ERR_CUDA
    llar.llar_set_launch(0, 0)
