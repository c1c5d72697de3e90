"""The oracle's all-core build (the same source compiled with OpenMP, used
only to time the oracle on every host core) gives exactly the plain build's
results: its parallel loops run over tokens (dispatch, combine) or experts
(low-latency dispatch) whose output rows are disjoint."""
import numpy as np
import pytest

import epinputs as ei
import oracle


@pytest.fixture()
def both():
    def run(fn):
        oracle.use_all_cores(False)
        a = fn()
        if not oracle.use_all_cores(True):
            pytest.skip("no OpenMP build on this host")
        try:
            assert oracle.threads() >= 1
            b = fn()
        finally:
            oracle.use_all_cores(False)
        return a, b
    return run


def _same(a, b):
    if isinstance(a, dict):
        assert a.keys() == b.keys()
        for k in a:
            _same(a[k], b[k])
    elif isinstance(a, (tuple, list)):
        for u, v in zip(a, b):
            _same(u, v)
    elif isinstance(a, np.ndarray):
        assert np.array_equal(a, b)
    else:
        assert a == b


@pytest.mark.parametrize("c,fp8", [(3, True), (4, False), (5, True)])
def test_dispatch_and_combine_identical(both, c, fp8):
    cfg = ei.WORKLOADS[c].scaled(N=300, H=512)
    d = ei.make_inputs(cfg, seed=7)

    def step():
        lay = oracle.layout(d["topk_idx"], cfg.E, cfg.R)
        o = oracle.dispatch(d["x"], d["topk_idx"], d["topk_weights"], cfg.E, cfg.R, fp8, lay=lay)
        y = d["x"][np.arange(o["exp_x"].shape[0]) % cfg.N]
        return o, oracle.combine(y, lay["expert_slot"], d["topk_weights"])
    a, b = both(step)
    _same(a, b)


@pytest.mark.parametrize("c", [1, 2])
def test_low_latency_identical(both, c):
    base = ei.WORKLOADS[c]
    cfg = base.scaled(N=base.R * 4, H=256, T=8)
    d = ei.make_inputs(cfg, seed=8)
    a, b = both(lambda: oracle.ll_dispatch(d["x"], d["topk_idx"], cfg.E, cfg.R, cfg.T, cfg.fp8))
    _same(a, b)
