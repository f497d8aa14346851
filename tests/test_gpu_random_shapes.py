"""The whole path on seeded random small layers: token counts down to one,
widths down to a single 16-byte vector, one expert up to 64, any k <= E,
random skew and retention, dead experts.  Every case is checked against the
fp64 oracle like the fixed parity cases (bit-exact integer work and
compaction, scores within 1e-5, GEMMs within 5e-3 per expert)."""

from fractions import Fraction

import numpy as np
import pytest

from gpu_common import built_library, custom_inputs, need_gpu
from test_gpu_parity import full_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    built_library()


def _cases(n=20, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.integers(1, 65))
        k = int(rng.integers(1, min(E, 8) + 1))
        T = int(rng.choice([1, 7, int(rng.integers(8, 400)), int(rng.integers(8, 400)), int(rng.integers(400, 3000))]))
        h = 8 * int(rng.integers(1, 97))
        I = 8 * int(rng.integers(1, 97))
        s = float(rng.choice([0.0, 0.5, 1.0, 1.6]))
        rho = Fraction(int(rng.integers(1, 5)), 4)
        dead = int(rng.integers(1, min(4, E - k) + 1)) if E - k >= 2 and i % 3 == 0 else 0
        out.append(dict(T=T, E=E, k=k, h=h, I=I, s=s, rho=rho, seed=100 + i, dead=dead))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"T{c['T']}_E{c['E']}_k{c['k']}_h{c['h']}_I{c['I']}")
def test_random_layer(case):
    full_check(custom_inputs(**case))


@pytest.mark.parametrize("T,E,k,h,I", [(300, 5, 2, 8, 8), (1, 1, 1, 8, 16), (64, 2, 2, 16, 8)])
def test_minimal_widths(T, E, k, h, I):
    # one 16-byte vector per row of g or phi: the smallest rows every kernel must handle
    full_check(custom_inputs(T=T, E=E, k=k, h=h, I=I, s=0.0, rho=Fraction(3, 4), seed=7 + T))
