"""Randomised parity: seeded draws of shapes across the supported space, each
step (new tokens written, then the decode: pa_decode_append) against the
oracle (scatter, then fp64 attention over the updated cache). The draws and
the checks are in pa_random_draws."""
import pytest

import pa_random_draws

pytestmark = pytest.mark.gpu

NUM_DRAWS = 64


@pytest.mark.parametrize("seed", range(NUM_DRAWS))
def test_random_shape_step(seed):
    pa_random_draws.run_draw(seed)
