"""Step a6's arithmetic on its own: the expert kernel's SiLU(gate) * up (a
hardware base-2 exponential and a Newton-Raphson reciprocal), evaluated on the
device through moe_selftest_silu and compared with float64 SiLU(g) * u =
g u / (1 + e^-g) over the whole range of g the layer can produce."""
import numpy as np
import pytest
import torch

import expert_ffn_layer_gb300 as moe

pytestmark = pytest.mark.gpu

# relative error bound where the result is a normal float well above underflow
REL_BOUND = 1e-5
# below g = -83 the exponential's argument is capped at 120: the result is then
# at most |g u| 2^-119 (the true value is below 1e-34 there)
G_CAP = -83.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _device_silu(g32: np.ndarray, u32: np.ndarray) -> np.ndarray:
    g = torch.from_numpy(g32).cuda()
    u = torch.from_numpy(u32).cuda()
    out = torch.full_like(g, float("nan"))
    moe.moe_selftest_silu(g, u, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _reference(g32, u32):
    g, u = g32.astype(np.float64), u32.astype(np.float64)
    with np.errstate(over="ignore"):
        return g * u / (1.0 + np.exp(-g))


def test_silu_mul_error_bound_over_the_range():
    rng = np.random.default_rng(17)
    special = np.array([0.0, -0.0, 1.0, -1.0, 1e-30, -1e-30, 1e-6, -1e-6, 0.5, -0.5, 20.0, -20.0, 60.0, -60.0,
                        88.0, 100.0, 120.0, -82.9, -83.0, -83.2, -87.0, -100.0, -119.9, -120.0])
    g = np.concatenate([np.linspace(-120.0, 120.0, 2_400_001), special, rng.normal(0.0, 3.0, 200_000),
                        rng.uniform(-120.0, 120.0, 200_000)]).astype(np.float32)
    for u in (np.ones_like(g), rng.normal(0.0, 2.0, g.size).astype(np.float32)):
        got = _device_silu(g, u).astype(np.float64)
        ref = _reference(g, u)
        assert np.isfinite(got).all()
        big = g >= G_CAP
        rel = np.abs(got[big] - ref[big]) / np.maximum(np.abs(ref[big]), 1e-300)
        nz = ref[big] != 0
        assert rel[nz].max() <= REL_BOUND, f"max rel err {rel[nz].max():.3e} at g={g[big][nz][rel[nz].argmax()]}"
        assert (got[big][~nz] == 0).all()
        # the capped tail: tiny, and no larger than the cap allows
        tail = ~big
        lim = np.abs(g[tail].astype(np.float64) * u[tail]) * 2.0 ** -119
        assert (np.abs(got[tail]) <= lim).all() and (np.abs(got[tail] - ref[tail]) <= lim).all()
        # SiLU(0) * u is exactly zero
        assert (got[g == 0] == 0).all()
