"""Ragged-balanced decode: the batch's 16-token tiles cut into equal ranges per
CTA on the device, pieces of sequences that straddle two ranges merged by
log-sum-exp. Parity with the fp64 oracle ("What Does PagedAttention Actually
Optimize?", section 8: the result is softmax(scale q K^T) V whatever the
split), both where pa_decode picks it by itself (many sequences) and, in a
child process with PA_DECODE_BALANCE=1, on small batches that exercise
every corner: CTAs whose range spans several sequences, sequences spread
over many CTAs, empty sequences, more CTAs than tiles, lengths past the
host bound."""
import json
import os
import subprocess
import sys

if __name__ == "__main__":   # the child process: the repo root, as conftest gives pytest
    sys.path[:0] = [os.path.dirname(os.path.dirname(os.path.abspath(__file__)))]

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import ATOL, DeviceBatch, make_workspace, max_err, oracle_step, run_step

pytestmark = pytest.mark.gpu


def ragged_batch(name, lens, hq, hkv, d, bs, seed, max_blocks=None):
    need = sum(workloads.cdiv(int(n), bs) for n in lens)
    return workloads.make_batch(name, lens, hq, hkv, d, bs, need + 11, True, seed_values=seed,
                                seed_blocks=seed + 1, max_blocks=max_blocks)


@pytest.mark.parametrize("case", [
    # B, length range, Hq, Hkv, D, block size
    (128, (0, 700), 32, 8, 128, 16),
    (160, (1, 300), 32, 8, 128, 32),
    (240, (0, 200), 16, 4, 64, 16),
    (400, (1, 90), 32, 8, 128, 64),
])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_balanced_is_chosen_for_many_sequences(case, out_dtype):
    B, (lo, hi), hq, hkv, d, bs = case
    rng = np.random.default_rng(B + bs)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    lens[::17] = 0            # a few empty sequences
    lens[5] = hi              # the bound is reached
    batch = ragged_batch("bal", lens, hq, hkv, d, bs, seed=B)
    batch.new_pos = np.where(lens > 0, lens - 1, -1).astype(np.int32)   # scatter only into live sequences
    plan = pa.pa_decode_plan(B, hq, hkv, d, bs, int(lens.max()), pa.PA_BF16, with_workspace=True)
    assert plan["balanced"] == 1 and plan["kernel_launches"] == 2
    db = DeviceBatch(batch)
    ws = make_workspace(batch)
    ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device="cuda"))   # needs no initialisation
    out = run_step(db, workspace=ws, out_dtype=out_dtype)
    want, _, _ = oracle_step(batch)
    g = out.float().cpu().numpy().astype(np.float64)
    tol = ATOL + (np.abs(want) * 2.0 ** -8 if out_dtype == torch.bfloat16 else 0.0)
    assert np.all(np.isfinite(g)) and np.all(np.abs(g - want) <= tol)
    assert np.all(g[lens == 0] == 0)
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0


def test_balanced_off_without_workspace_or_with_few_sequences():
    assert pa.pa_decode_plan(64, 32, 8, 128, 16, 4096, pa.PA_BF16, with_workspace=False)["balanced"] == 0
    assert pa.pa_decode_plan(16, 32, 8, 128, 16, 4164, pa.PA_BF16, with_workspace=True)["balanced"] == 0
    assert pa.pa_decode_plan(64, 32, 8, 128, 8, 4096, pa.PA_BF16, with_workspace=True)["balanced"] == 0


# ---------------------------------------------------------------------------
# forced on small batches (child process: the switch is read once per process)
# ---------------------------------------------------------------------------
FORCED = [
    # lens, Hq, Hkv, D, block size, max_context_len (None: the longest)
    ((25, 47, 12), 4, 4, 64, 16, None),                 # more CTAs than tiles
    ((0, 1, 0, 33, 500, 16, 17), 8, 2, 128, 16, None),  # empty sequences, one-tile sequences
    ((3000, 5, 2900, 40), 32, 8, 128, 32, None),        # long sequences spread over many CTAs
    ((700, 300, 129, 64, 1), 64, 2, 128, 64, None),     # G = 32: two head tiles
    ((400, 333, 250), 24, 12, 64, 16, None),            # 12 KV heads: groups of 6
    ((900, 100, 650), 8, 2, 128, 128, 600),             # lengths past the host bound are cut
    ((1,) * 40 + (4000,), 16, 4, 128, 16, None),        # one long sequence among many short
    ((0, 0, 0), 8, 2, 128, 16, 64),                     # no tile at all: zeros only
    ((300, 900, 1, 513, 256), 8, 2, 128, 256, None),    # the largest blocks: 16 tiles per block
]


def child_main():
    results = []
    for i, (lens, hq, hkv, d, bs, mcl) in enumerate(FORCED):
        lens = np.asarray(lens, np.int32)
        batch = ragged_batch("forced", lens, hq, hkv, d, bs, seed=300 + i,
                             max_blocks=None if lens.max() > 0 else workloads.cdiv(mcl, bs))
        batch.new_pos = np.full(len(lens), -1, np.int32)
        bound = int(lens.max()) if mcl is None else mcl
        plan = pa.pa_decode_plan(len(lens), hq, hkv, d, bs, bound, pa.PA_BF16, with_workspace=True)
        db = DeviceBatch(batch)
        ws = make_workspace(batch, max_context_len=bound)
        ws.fill_(0xFF)   # the workspace needs no initialisation
        want = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                      np.minimum(lens, bound), batch.scale)
        errs = []
        for _ in range(3):   # the same workspace again: nothing left by one call leaks into the next
            out = torch.full((len(lens), hq, d), 5.0, dtype=torch.float32, device="cuda")
            pa.pa_decode(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens, bound,
                         batch.scale, workspace=ws)
            errs.append(max_err(out, want))
        torch.cuda.synchronize()
        results.append({"case": i, "balanced": plan["balanced"], "err": max(errs),
                        "status": pa.pa_device_status(clear=True)})
    print(json.dumps(results))


def test_balanced_forced_small_batches():
    env = dict(os.environ, PA_DECODE_BALANCE="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "child"], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    results = json.loads(r.stdout.strip().splitlines()[-1])
    assert len(results) == len(FORCED)
    for res in results:
        assert res["balanced"] == 1, res
        assert res["status"] == 0, res
        assert res["err"] <= ATOL, res


if __name__ == "__main__" and sys.argv[1:] == ["child"]:
    child_main()
