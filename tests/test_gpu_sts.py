"""The STS calibration fit on the GPU against the oracle.

Parity rule: the chosen grid temperature of every position is bit-exact up to
the first position the oracle calls too close (its best and second-best ECE
within STS_MARGIN; a different choice there changes every later position), and
the ECE of each compared position agrees within STS_ECE_TOL. The GPU forms the
running products in fp32, so a sample can fall into the neighbouring bin when
it lies within fp32 rounding of a bin edge; that moves an ECE by at most
2/N, hence the tolerances.
"""

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_head_gb300 import binding, build
from speculative_decoding_head_gb300.workloads import STS_SETS, make_sts_inputs, sts_grid

pytestmark = pytest.mark.gpu

STS_MARGIN = 1e-4
STS_ECE_TOL = 5e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _compare(raw, cstar, grid, M):
    T, ece, st = binding.sts_fit(raw.cuda(), cstar.cuda(), grid.cuda(), M)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    oT, oe, om = oracle.sts_fit(raw.numpy(), cstar.numpy(), grid.numpy(), M)
    T, ece = T.cpu().numpy(), ece.cpu().numpy()
    compared = 0
    for k in range(len(oT)):
        if om[k] < STS_MARGIN:
            break
        assert T[k] == oT[k], (k, T[k], oT[k], om[k])
        assert abs(ece[k] - oe[k]) <= STS_ECE_TOL, (k, ece[k], oe[k])
        compared += 1
    return compared


@pytest.mark.parametrize("name", list(STS_SETS))
def test_sts_parity(name):
    c = STS_SETS[name]
    inp = make_sts_inputs(c["N"], c["gamma"], c["seed"])
    assert _compare(inp["raw"], inp["cstar"], sts_grid(c["G"]), c["M"]) == c["gamma"]


def test_sts_recovers_generating_temperatures_and_bin_counts():
    rng = np.random.default_rng(11)
    N, g = 50000, 3
    raw = rng.normal(1.0, 1.5, (N, g)).astype(np.float32)
    grid = sts_grid(30)
    Tstar = grid.numpy()[[5, 14, 22]]
    cstar = (1.0 / (1.0 + np.exp(-raw.astype(np.float64) / Tstar.astype(np.float64)))).astype(np.float32)
    raw_t, cstar_t = torch.from_numpy(raw), torch.from_numpy(cstar)
    for M in (1, 7, 15, 32):
        T, ece, st = binding.sts_fit(raw_t.cuda(), cstar_t.cuda(), grid.cuda(), M)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(T.cpu().numpy(), Tstar), (M, T)
        assert ece.cpu().numpy().max() < 1e-6
    assert _compare(raw_t, cstar_t, grid, 15) == g


def test_sts_bad_grid_is_reported():
    inp = make_sts_inputs(1000, 2, 7)
    grid = sts_grid(10).clone()
    grid[3] = -1.0
    T, ece, st = binding.sts_fit(inp["raw"].cuda(), inp["cstar"].cuda(), grid.cuda(), 15)
    torch.cuda.synchronize()
    assert int(st.item()) == 6          # DSPARK_ERANGE
    with pytest.raises(binding.DsparkError):
        binding.sts_fit(inp["raw"].cuda(), inp["cstar"].cuda(), grid.cuda(), 33)   # more bins than supported
