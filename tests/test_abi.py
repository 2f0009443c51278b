"""The C ABI: the library loads, exports every declared symbol, and its
host-only logic behaves, all without a GPU (no compute call is made)."""

import ctypes
import os
import re

import pytest

from oracle import protocol as oproto
from tp_allreduce_persistent_b300 import build, llar

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", n) for n in sorted(os.listdir(os.path.join(ROOT, "include")))
           if n.endswith(".h")]


def declared_functions():
    names = set()
    for path in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names |= set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(llar_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


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
    # the direct-AllGather variant: the same lines, three slots, no LL copy
    lb, pl, st = llar.llar_layout("ll128_direct", dtype, 8, 1 << 20)
    assert lb == 128 and pl == oproto.ll128_payload_elems(dtype)
    assert st == 3 * oproto.ll128_round_staging_bytes(1 << 20, 8, dtype)
    lb, pl, st = llar.llar_layout("sentinel", dtype, 8, 32768)
    # published once per rank: a ring of 32 slots of the 64 KiB default chunk, one tail word per vector
    assert lb == 16 and pl * e == 16 and st == 32 * 65536 + 65536 // 16 * 8


@pytest.mark.parametrize("n", range(2, 9))
def test_protocol_selection_per_rank_count(n):
    # one AllReduce per launch: LL / direct one-shot / direct two-shot
    # thresholds in KiB per rank (ll_max 0: LL never)
    kib = 512  # bf16 elements per KiB
    ll_max, one_max = {2: (0, 1024), 3: (0, 1024), 4: (64, 256), 5: (0, 128), 6: (0, 64),
                       7: (32, 32), 8: (32, 32)}[n]
    order = ["ll", "fixed_oneshot", "fixed_twoshot"]
    last = 0
    for k in (2, 4, 8, 16, 32, 33, 64, 65, 128, 129, 256, 257, 512, 513, 1024, 1025, 4096):
        p = llar.llar_select_protocol(n, "bf16", k * kib)
        expect = "ll" if k <= ll_max else ("fixed_oneshot" if k <= one_max else "fixed_twoshot")
        assert p == expect, (n, k, p)
        assert order.index(p) >= last
        last = order.index(p)
    # the rule is in bytes: fp32 reaches each threshold at half the elements
    if ll_max:
        assert llar.llar_select_protocol(n, "fp32", (ll_max * 1024) // 4) == "ll"
        assert llar.llar_select_protocol(n, "fp32", (ll_max * 1024) // 4 + 1) != "ll"
    assert llar.llar_select_protocol(n, "fp32", (one_max * 1024) // 4 + 1) == "fixed_twoshot"


def test_protocol_selection_is_monotone_in_size():
    order = ["ll", "sentinel", "ll128", "fixed_oneshot", "fixed_twoshot"]
    last = 0
    for nbytes in [16, 4096, 16384, 65536, 1 << 18, 1 << 20, 1 << 22, 1 << 26]:
        p = llar.llar_select_protocol(8, "bf16", nbytes // 2)
        assert p in order
        assert order.index(p) >= last
        last = order.index(p)
    assert llar.llar_select_protocol(8, "bf16", 8192) == "ll"


def test_host_memory_protocol_selection():
    # host buffers read across the bus: LL up to 4 KiB per rank, the
    # direct-read two-shot above, for every rank count and dtype (in bytes)
    for n in range(2, 9):
        for dtype, e in (("bf16", 2), ("fp16", 2), ("fp32", 4)):
            assert llar.llar_select_protocol_host(n, dtype, 16 // e) == "ll"
            assert llar.llar_select_protocol_host(n, dtype, 4096 // e) == "ll"
            assert llar.llar_select_protocol_host(n, dtype, 4096 // e + 1) == "fixed_twoshot"
            assert llar.llar_select_protocol_host(n, dtype, (1 << 20) // e) == "fixed_twoshot"
    assert llar.llar_select_protocol_host(1, "bf16", 8192) == "auto"
    assert llar.lib().llar_select_protocol_host(8, 7, 8192) == llar.PROTOCOLS["auto"]  # no such dtype


def test_persistent_protocol_selection():
    # one AllReduce per launch: the single-call rule
    for n in range(2, 9):
        for kib in (4, 64, 512, 1024):
            count = kib * 512
            assert llar.llar_select_protocol_iters(n, "bf16", count, 1) == llar.llar_select_protocol(n, "bf16", count)
    # chains: LL up to the 1 MiB LL capacity (7-8 ranks: up to 512 KiB), then the two-shot
    for n in range(2, 9):
        for kib in (1, 64, 256, 512, 513, 1024, 1025, 4096):
            count = kib * 512
            ll = kib <= 1024 and (n <= 6 or kib <= 512)
            want = "ll" if ll else "fixed_twoshot"
            assert llar.llar_select_protocol_iters(n, "bf16", count, 160, True) == want, (n, kib)
    # independent back to back: LL up to 256 KiB (2 ranks), 128 KiB (3-4), 64 KiB (5-8),
    # the one-shot up to 1 MiB (2-3), 512 KiB (4), 256 KiB (5), then the two-shot
    loop = {2: (256, 1024), 3: (128, 1024), 4: (128, 512), 5: (64, 256), 6: (64, 64), 7: (64, 64), 8: (64, 64)}
    for n in range(2, 9):
        for kib in (16, 33, 64, 65, 128, 129, 256, 257, 512, 513, 1024, 1025):
            ll_max, one_max = loop[n]
            want = "ll" if kib <= ll_max else ("fixed_oneshot" if kib <= one_max else "fixed_twoshot")
            assert llar.llar_select_protocol_iters(n, "bf16", kib * 512, 200, False) == want, (n, kib)
    assert llar.llar_select_protocol_iters(8, "bf16", 8192, 0) == "auto"
    # with nondeterministic protocols allowed, chains take LL128 direct where measured fastest
    for n in range(2, 9):
        for kib in (128, 256, 512, 1024):
            count = kib * 512
            got = llar.llar_select_protocol_iters(n, "bf16", count, 160, True, True)
            atomic = n >= 5 and (kib >= 512 or (n == 8 and kib >= 256)) and (n <= 6 or kib <= 512)
            want = "ll128_direct" if atomic else llar.llar_select_protocol_iters(n, "bf16", count, 160, True)
            assert got == want, (n, kib)
            # never for independent AllReduces or single calls
            assert llar.llar_select_protocol_iters(n, "bf16", count, 200, False, True) != "ll128_direct"
            assert llar.llar_select_protocol_iters(n, "bf16", count, 1, True, True) != "ll128_direct"
    with pytest.raises(llar.LlarError):
        llar.llar_set_auto_nondeterministic(True)  # needs a context


def test_segment_protocol_selection():
    # the direct copies for both halves at every size and rank count, whole
    # 16-byte vector segments or ragged ones
    for n in range(2, 9):
        for kib in (1, 16, 64, 65, 1024):
            for dtype, e in (("bf16", 2), ("fp32", 4)):
                for count in (kib * 1024 // e, kib * 1024 // e - 1, kib * 1024 // e - 8 * n + 3):
                    assert llar.llar_select_protocol_segment(True, n, dtype, count) == "fixed_oneshot"
                    assert llar.llar_select_protocol_segment(False, n, dtype, count) == "fixed_oneshot", (n, count)
    assert llar.llar_select_protocol_segment(True, 9, "bf16", 8) == "auto"


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
    # the host-buffer table belongs to a context
    for call in (lambda: llar.llar_host_register(4096, 64), lambda: llar.llar_host_unregister(4096)):
        with pytest.raises(llar.LlarError) as ei:
            call()
        assert ei.value.code == llar.ERR_NOT_INIT
    # so does the placed speed-of-light probe (it takes the last launch's shape)
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_sol_probe_placed()
    assert ei.value.code == llar.ERR_NOT_INIT
    # an unknown protocol value
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_debug_launch_shape(8, "bf16", 8192, 7)
    assert ei.value.code == llar.ERR_INVALID
    assert llar.strerror(llar.ERR_TIMEOUT) == "a device-side wait timed out"


def test_init_without_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_init(8, "bf16", 1 << 20)
    assert ei.value.code == llar.ERR_CUDA
    llar.llar_set_launch(0, 0)


def test_llbuffer_descriptor_layout_matches_c():
    """The ctypes mirror of llar_llbuffer has the C compiler's offsets and size."""
    import shutil
    import subprocess
    import tempfile
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    fields = [f for f, _ in llar.LLBufferDesc._fields_]
    src = "#include <stdio.h>\n#include <stddef.h>\n#include \"llar_llbuffer.h\"\nint main(void){\n"
    src += 'printf("%zu\\n", sizeof(llar_llbuffer));\n'
    for f in fields:
        src += f'printf("%zu\\n", offsetof(llar_llbuffer, {f}));\n'
    src += 'printf("%zu %zu\\n", sizeof(llar_llbuffer_status), offsetof(llar_llbuffer_status, epoch));\n'
    src += "return 0;}\n"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(src)
        subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()
    want = [ctypes.sizeof(llar.LLBufferDesc)] + [getattr(llar.LLBufferDesc, f).offset for f in fields]
    want += [ctypes.sizeof(llar.LLBufferStatus), llar.LLBufferStatus.epoch.offset]
    assert [int(x) for x in got] == want


def test_llbuffer_argument_checks_without_device():
    for n, b in [(1, 1024), (9, 1024), (4, 0), (4, (1 << 30) + 1)]:
        with pytest.raises(llar.LlarError) as ei:
            llar.LLBuffer(n, b)
        assert ei.value.code == llar.ERR_INVALID
    desc = llar.LLBufferDesc()  # never created
    assert llar.lib().llar_llbuffer_destroy(ctypes.byref(desc)) == llar.ERR_INVALID
    assert llar.lib().llar_llbuffer_get_status(ctypes.byref(desc), None, None) == llar.ERR_INVALID
    pp = (ctypes.c_void_p * 8)()
    assert llar.lib().llar_llbuffer_allreduce(ctypes.byref(desc), pp, pp, 16, 0, 1, 1, None) == llar.ERR_INVALID
    # the plain GEMV checks its shape before touching the device
    assert llar.lib().llar_linear_partials(pp, pp, pp, 2, 17, 8, 8, 2, None) == llar.ERR_INVALID  # M > 16
    assert llar.lib().llar_linear_partials(pp, pp, pp, 2, 1, 8, 12, 2, None) == llar.ERR_INVALID  # H % 8
    import torch
    if not torch.cuda.is_available():
        with pytest.raises(llar.LlarError) as ei:
            llar.LLBuffer(2, 1024)
        assert ei.value.code == llar.ERR_CUDA


def test_device_header_links_into_several_translation_units():
    """Two .cu files of one program both include the device header."""
    import shutil
    import subprocess
    import tempfile
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    src = ('#include "llar_llbuffer.cuh"\n'
           '__global__ void k_%s(llar_llbuffer b) { llb::u64 d; llb::ll_wait(b, 0, 1, 1, 0, d); }\n')
    with tempfile.TemporaryDirectory() as d:
        files = []
        for name in ("a", "b"):
            path = os.path.join(d, name + ".cu")
            open(path, "w").write(src % name)
            files.append(path)
        main = os.path.join(d, "main.cu")
        open(main, "w").write("int main() { return 0; }\n")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-I", os.path.join(ROOT, "include"),
                        *files, main, "-o", os.path.join(d, "prog")], check=True, capture_output=True)
