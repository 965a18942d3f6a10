"""Randomised parity of the shared-prefix decode (pa_decode_shared_prefix):
seeded draws across its supported space, each against the oracle, which is
plain paged attention over the same block tables ("PagedAttention: KV cache
virtual memory", "Copy-on-write: when two requests share a prefix": shared
blocks change where K and V sit, not what attention computes).

Each draw picks the batch size, the GQA ratio (up to 128 query heads per KV
head, the tcgen05 pass's largest row group), the KV heads, head_dim, the block
size (8 to 256), how many leading blocks are shared (none included), the
lengths past them (empty ones included), the element type and the output
type. The draw is recorded in the failure message.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import ATOL, DeviceBatch

pytestmark = pytest.mark.gpu

NUM_DRAWS = 40
ORACLE_BUDGET = 2.5e7   # rows x tokens the fp64 oracle is given per draw


def draw(seed):
    rng = np.random.default_rng(40_000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([g for g in (1, 2, 3, 4, 6, 8, 16, 32, 64, 128) if g * hkv <= 128]))
    d = int(rng.choice([64, 128]))
    bs = int(rng.choice([8, 16, 32, 64, 128, 256]))
    nsh = int(rng.integers(0, max(1, 3000 // bs) + 1))
    hi = int(rng.choice([0, 16, 300, 2000]))
    b = int(rng.integers(1, 101))
    max_ctx = nsh * bs + hi
    b = max(1, min(b, int(ORACLE_BUDGET // max(1, hkv * group * max(max_ctx, 1)))))
    suffix = rng.integers(0, hi + 1, size=b)
    suffix[rng.random(b) < 0.1] = 0
    kind = str(rng.choice(["bf16", "f16"]))
    out_kind = str(rng.choice(["f32", "same"]))
    return dict(nsh=nsh, suffix=suffix.astype(np.int64), hq=hkv * group, hkv=hkv, d=d, bs=bs, kind=kind,
                out_kind=out_kind)


@pytest.mark.parametrize("seed", range(NUM_DRAWS))
def test_random_shared_prefix(seed):
    c = draw(seed)
    batch = workloads.shared_prefix_batch("rp", c["nsh"], c["suffix"], c["hq"], c["hkv"], c["d"], c["bs"],
                                          seed_values=50_000 + seed, seed_blocks=60_000 + seed,
                                          f16=c["kind"] == "f16")
    db = DeviceBatch(batch)
    n = pa.pa_decode_shared_prefix_workspace_size(batch.num_seqs, c["hq"], c["hkv"], c["d"], c["bs"],
                                                  batch.max_context_len, c["nsh"])
    ws = torch.full((max(n, 1),), 0xFF, dtype=torch.uint8, device="cuda")   # no initialisation needed
    out_dtype = torch.float32 if c["out_kind"] == "f32" else db.k_cache.dtype
    out = torch.full((batch.num_seqs, c["hq"], c["d"]), float("nan"), dtype=out_dtype, device="cuda")
    pa.pa_decode_shared_prefix(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                               batch.max_context_len, c["nsh"], batch.scale, ws)
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0, c
    want = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                  batch.context_lens, batch.scale)
    g = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), c
    # a 16-bit output adds at most half an ulp of its type
    rel = {torch.float32: 0.0, torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}[out_dtype]
    bad = np.abs(g - want) > ATOL + np.abs(want) * rel
    assert not bad.any(), (c, float(np.max(np.abs(g - want))))
