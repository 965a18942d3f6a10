"""Seeded draws of decode shapes across the supported space, and one decode
step (new tokens written, then the decode: pa_decode_append) on a draw,
checked against the oracle (scatter, then fp64 attention over the updated
cache). Shared by the randomised parity test and the knob tests.

Each draw picks the batch size, ragged lengths (empty and one-token contexts
included), the GQA ratio, head_dim, block size, element type, whether a
workspace is passed, and the output type. Caches must match bit for bit and
the output within the bound; the plan pa_decode_plan reports is recorded in
the failure message so that a failing draw names the path it took.
"""
import numpy as np
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import ATOL, DeviceBatch, make_workspace, to_host_bits


def draw(seed):
    rng = np.random.default_rng(10_000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8, 12]))
    group = int(rng.choice([1, 2, 3, 4, 6, 8, 16, 32]))
    d = int(rng.choice([64, 128]))
    kind = str(rng.choice(["bf16", "bf16", "f16", "f32"]))
    bs = int(rng.choice([1, 2, 4, 8, 12, 16, 32, 64, 128, 256] if kind != "f32" else [8, 12, 16, 32]))
    b = int(rng.integers(1, 40))
    hi = int(rng.choice([64, 700, 3000, 9000]))
    lens = rng.integers(0, hi + 1, size=b)
    lens[rng.random(b) < 0.1] = 0
    lens[rng.random(b) < 0.1] = 1
    use_ws = bool(rng.random() < 0.7)
    out_kind = str(rng.choice(["f32", "f32", "same"]))
    return dict(lens=lens.astype(np.int32), hq=hkv * group, hkv=hkv, d=d, bs=bs, kind=kind, use_ws=use_ws,
                out_kind=out_kind)


def run_draw(seed):
    c = draw(seed)
    lens, hq, hkv, d, bs, kind = c["lens"], c["hq"], c["hkv"], c["d"], c["bs"], c["kind"]
    need = sum(workloads.cdiv(int(n), bs) for n in lens)
    batch = workloads.make_batch("rand", lens, hq, hkv, d, bs, need + 7, kind == "bf16", seed_values=20_000 + seed,
                                 seed_blocks=30_000 + seed, f16=kind == "f16")
    batch.new_pos = np.where(lens > 0, lens - 1, -1).astype(np.int32)
    mcl = max(1, int(lens.max()))
    kv_dtype = {"bf16": pa.PA_BF16, "f16": pa.PA_F16, "f32": pa.PA_F32}[kind]
    plan = pa.pa_decode_plan(len(lens), hq, hkv, d, bs, mcl, kv_dtype=kv_dtype, with_workspace=c["use_ws"])
    db = DeviceBatch(batch)
    ws = make_workspace(batch, max_context_len=mcl) if c["use_ws"] else None
    out_dtype = torch.float32 if c["out_kind"] == "f32" else db.k_cache.dtype
    out = torch.full((len(lens), hq, d), float("nan"), dtype=out_dtype, device="cuda")
    pa.pa_decode_append(out, db.query, db.new_key, db.new_value, db.k_cache, db.v_cache, db.block_tables,
                        db.context_lens, mcl, batch.scale, workspace=ws)
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0, (c, plan)

    k, v = batch.k_cache.copy(), batch.v_cache.copy()
    seqs = np.arange(len(lens))
    live = lens > 0
    slots = oracle.slot_mapping(batch.block_tables, seqs[live], lens[live] - 1, bs)
    oracle.reshape_and_cache(k, v, batch.new_key[live], batch.new_value[live], slots)
    want = oracle.paged_attention(batch.query, k, v, batch.block_tables, lens, batch.scale)
    assert np.array_equal(to_host_bits(db.k_cache), k) and np.array_equal(to_host_bits(db.v_cache), v), (c, plan)
    g = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), (c, plan)
    # a 16-bit output adds at most half an ulp of its type
    rel = {torch.float32: 0.0, torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}[out_dtype]
    bad = np.abs(g - want) > ATOL + np.abs(want) * rel
    assert not bad.any(), (c, plan, float(np.max(np.abs(g - want))))
