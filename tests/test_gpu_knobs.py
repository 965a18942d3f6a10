"""The decode tuning knobs, each in a child process (they are read once per
process), on the first seeded draws of the randomised parity test: each
step (new tokens written, then the decode) against the oracle, caches bit
for bit. A knob changes how the work is cut and launched, never the result
beyond the stated bound."""
import json
import os
import subprocess
import sys

if __name__ == "__main__":   # the child process: the repo root and tests/, as conftest gives pytest
    here = os.path.dirname(os.path.abspath(__file__))
    sys.path[:0] = [os.path.dirname(here), here]

import pytest

pytestmark = pytest.mark.gpu

DRAWS = 12

KNOBS = {
    "no_pdl": {"PA_PDL": "0"},                       # plain launches, no programmatic dependent launch
    "simt": {"PA_DECODE_KERNEL": "simt"},            # the CUDA-core kernel for 16-bit caches too
    "one_head_per_cta": {"PA_DECODE_HEADS": "1"},
    "two_heads_per_cta": {"PA_DECODE_HEADS": "2"},
    "six_ctas_per_sm": {"PA_DECODE_CTAS_PER_SM": "6"},
    "smallest_ring": {"PA_DECODE_RING_KB": "16"},    # one stage per ring
    "largest_ring": {"PA_DECODE_RING_KB": "200"},
    "never_balanced": {"PA_DECODE_BALANCE": "0"},
}


def child():
    import torch
    import pa_random_draws
    for seed in range(DRAWS):
        pa_random_draws.run_draw(seed)
    torch.cuda.synchronize()
    print(json.dumps({"draws": DRAWS}))


@pytest.mark.parametrize("knob", sorted(KNOBS))
def test_decode_under_knob(knob):
    env = dict(os.environ, **KNOBS[knob])
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "child"], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    assert json.loads(r.stdout.strip().splitlines()[-1])["draws"] == DRAWS


if __name__ == "__main__" and sys.argv[1:] == ["child"]:
    child()
