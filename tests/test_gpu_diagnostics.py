"""The measurement helpers behind the bench's latency evidence.

llar_sol_probe_placed: the speed of light (2 x L2 round trip + one remote
write, "Every Microsecond Matters", summary page) over the CTAs that a
launch of the last AllReduce's shape places: every pair of CTAs that
exchange data is measured once (G x N (N - 1) / 2 pairs), and the result is
the bound at the worst pair.

llar_debug_poll_stats: the poll-counting build of the library counts every
polling round; in the regular build the call reports LLAR_ERR_UNSUPPORTED.
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from tp_allreduce_persistent_b300 import build as libbuild
from tp_allreduce_persistent_b300 import inputs, llar

from gpu_util import context, device_inputs, filled_outputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_poll_stats_unsupported_in_the_regular_build():
    # no device work: the regular build answers before any CUDA call
    if os.environ.get("LLAR_LIBRARY"):
        pytest.skip("another build of the library is selected")
    with pytest.raises(llar.LlarError) as ei:
        llar.llar_debug_poll_stats()
    assert ei.value.code == llar.ERR_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("n", [8, 5])
def test_placed_probe_measures_every_exchanging_pair(n):
    count = 8192
    x = inputs.normal(n, count, "bf16", seed=3, scale=0.02)
    with context(n, "bf16", count * 2):
        with pytest.raises(llar.LlarError) as ei:
            llar.llar_sol_probe_placed()  # no AllReduce launched yet
        assert ei.value.code == llar.ERR_INVALID
        ins = device_inputs(x)
        outs = filled_outputs(n, count, "bf16")
        llar.llar_allreduce(ins, outs, count, "ll")
        torch.cuda.synchronize()
        _, G, _, _ = llar.llar_last_launch()
        l2, wr, sol, pairs = llar.llar_sol_probe_placed()
        med_l2, med_wr, med_sol = llar.llar_sol_probe()
    assert pairs == G * n * (n - 1) // 2
    assert 0.02 < l2 < 5.0 and 0.02 < wr < 50.0
    assert abs(sol - (2 * l2 + wr)) < 1e-9
    assert l2 >= 0.5 * med_l2  # the worst placed SM is not far below the median SM


POLL_SCRIPT = r"""
import json, sys, torch
sys.path.insert(0, {root!r})
from tp_allreduce_persistent_b300 import inputs, llar
n, count = 8, 8192
x = inputs.normal(n, count, "bf16", seed=5, scale=0.02, exclude_sentinel=True)
out = {{}}
for proto in ("ll", "sentinel", "ll128"):
    llar.llar_init(n, "bf16", count * 2)
    ins = [x[r].cuda() for r in range(n)]
    outs = [torch.empty_like(t) for t in ins]
    llar.llar_allreduce_iters(ins, outs, count, proto, 5)
    llar.llar_debug_poll_stats(reset=True)
    llar.llar_allreduce_iters(ins, outs, count, proto, 50)
    out[proto] = llar.llar_debug_poll_stats(reset=True)
    assert llar.llar_get_status()[0] == llar.OK
    llar.llar_destroy()
print(json.dumps(out))
"""


@pytest.mark.gpu
def test_poll_counting_build_counts_every_awaited_line():
    lib = libbuild.POLLS_LIB
    if not os.path.exists(lib):
        pytest.fail(f"{lib} is missing: python -m tp_allreduce_persistent_b300.build --poll-stats")
    env = dict(os.environ, LLAR_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", POLL_SCRIPT.format(root=ROOT)], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    counts = json.loads(r.stdout.strip().splitlines()[-1])
    n, words, vecs = 8, 8192 * 2 // 8, 8192 * 2 // 16
    # LL: every rank waits for every peer's line of every word, every iteration
    rounds, loads, waits, awaited = counts["ll"]
    assert awaited == 50 * n * (n - 1) * words
    assert waits == 50 * n * words and loads >= awaited and rounds >= waits
    # sentinel (published once): every rank waits for every peer's vector of
    # every chunk, and once per launch for every peer's tail word
    rounds, loads, waits, awaited = counts["sentinel"]
    assert awaited == 50 * n * (n - 1) * vecs + n * (n - 1) * vecs
    assert loads >= awaited and rounds >= waits
    rounds, loads, waits, awaited = counts["ll128"]
    assert waits > 0 and loads >= awaited > 0


@pytest.mark.gpu
@pytest.mark.parametrize("force", ["0", "2", None])
def test_ll_placement_either_way_gives_the_oracle(force, monkeypatch):
    # llar_init times LL with and without clusters of N blocks and keeps the
    # faster for long launches; LLAR_CLUSTER forces either. The sums are
    # fixed-order, so every placement must give the oracle's bits.
    from oracle import allreduce as orc
    if force is None:
        monkeypatch.delenv("LLAR_CLUSTER", raising=False)
    else:
        monkeypatch.setenv("LLAR_CLUSTER", force)
    n, count, iters = 8, 8192, 20
    x = inputs.normal(n, count, "bf16", seed=11, scale=0.02, iters=iters)
    with context(n, "bf16", count * 2):
        placed = llar.llar_ll_placement()
        assert placed in (0, 1)
        if force is not None:
            assert placed == (1 if force == "2" else 0)
        from gpu_util import allreduce_iters
        got = allreduce_iters(x, "bf16", "ll", iters)
    assert np.array_equal(got, orc.allreduce_iters(inputs.bits_of(x), iters, "bf16"))
