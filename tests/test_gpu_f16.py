"""fp16 query and caches ("What Does PagedAttention Actually Optimize?",
section 2: fp16 and bf16 are both two bytes a value) through every path:
per-partition and cluster decode at every load mode, split-K and merge, the
ragged-balanced decode, the contiguous baseline, the shared-prefix passes,
the scatter and the block copy. Parity with the fp64 oracle on the same
fp16 values (widened exactly); bit-exact for the copies."""
import os
import subprocess
import sys

if __name__ == "__main__":   # the child process: the repo root, as conftest gives pytest
    sys.path[:0] = [os.path.dirname(os.path.dirname(os.path.abspath(__file__)))]

import json

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import ATOL, DeviceBatch, make_workspace, max_err, oracle_step, run_step, to_dev

pytestmark = pytest.mark.gpu


def clean():
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0


def f16_batch(name, lens, hq, hkv, d, bs, seed, extra=13):
    need = sum(workloads.cdiv(int(n), bs) for n in lens)
    return workloads.make_batch(name, lens, hq, hkv, d, bs, need + extra, False, seed_values=seed,
                                seed_blocks=seed + 1, f16=True)


CASES = [
    # lens, Hq, Hkv, D, block size
    ((1, 2, 15, 16, 17, 100, 333), 8, 2, 128, 16),
    ((1, 7, 8, 9, 64, 250), 16, 4, 128, 8),         # two blocks per tile
    ((19, 90, 300), 8, 2, 128, 4),                  # one bulk copy per token row
    ((3, 50, 129), 8, 8, 64, 1),
    ((1, 31, 32, 33, 700), 32, 8, 128, 32),
    ((50, 260), 64, 2, 128, 16),                    # G = 32: two head tiles
    ((5, 600), 12, 3, 128, 128),
    ((40, 90), 8, 2, 64, 12),                       # not a power of two: CUDA-core kernel
    ((3000, 4000), 16, 4, 128, 16),                 # a wide split: merge kernel
    ((5, 700), 8, 2, 128, 256),                     # the largest blocks
    ((2, 33, 250), 8, 2, 64, 2),                    # blocks of 2: one bulk copy per token row
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("use_ws", [False, True])
def test_f16_decode(case, use_ws):
    lens, hq, hkv, d, bs = CASES[case]
    batch = f16_batch("f16", lens, hq, hkv, d, bs, seed=700 + case)
    db = DeviceBatch(batch)
    assert db.k_cache.dtype == torch.float16
    out = run_step(db, workspace=make_workspace(batch) if use_ws else None)
    want, k_want, v_want = oracle_step(batch)
    assert np.array_equal(db.k_cache.cpu().numpy().view(np.uint16), k_want.view(np.uint16))
    assert np.array_equal(db.v_cache.cpu().numpy().view(np.uint16), v_want.view(np.uint16))
    assert max_err(out, want) <= ATOL
    clean()


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_f16_output_types(out_dtype):
    batch = f16_batch("f16out", (100, 513), 32, 8, 128, 16, seed=720)
    out = run_step(DeviceBatch(batch), workspace=make_workspace(batch), out_dtype=out_dtype)
    want, _, _ = oracle_step(batch)
    ulp = 2.0 ** -11 if out_dtype == torch.float16 else 2.0 ** -8   # half an ulp, relative
    g = out.float().cpu().numpy()
    assert np.all(np.abs(g - want) <= ATOL + np.abs(want) * ulp)
    # an fp16 output from bf16 inputs too
    bb = workloads.make_batch("bf16in", (100, 513), 32, 8, 128, 16, 80, True, seed_values=721)
    o2 = run_step(DeviceBatch(bb), workspace=make_workspace(bb), out_dtype=torch.float16)
    w2, _, _ = oracle_step(bb)
    assert np.all(np.abs(o2.float().cpu().numpy() - w2) <= ATOL + np.abs(w2) * 2.0 ** -11)
    clean()


def test_f16_splitk_and_merge():
    lens = (1, 100, 511, 512, 513, 1500)
    hq, hkv, d, bs, ps = 16, 4, 128, 16, 48
    batch = f16_batch("f16sk", lens, hq, hkv, d, bs, seed=730)
    db = DeviceBatch(batch)
    P = workloads.cdiv(max(lens), ps)
    tmp = torch.empty((len(lens), hq, P, d), dtype=torch.float32, device="cuda")
    ml = torch.empty((len(lens), hq, P), dtype=torch.float32, device="cuda")
    es = torch.empty((len(lens), hq, P), dtype=torch.float32, device="cuda")
    pa.pa_decode_splitk(tmp, ml, es, ps, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                        max(lens), batch.scale)
    out = torch.empty((len(lens), hq, d), dtype=torch.float16, device="cuda")
    pa.pa_lse_merge(out, tmp, ml, es, db.context_lens, ps)
    want = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                  batch.context_lens, batch.scale)
    assert np.all(np.abs(out.float().cpu().numpy() - want) <= ATOL + np.abs(want) * 2.0 ** -11)
    clean()


def test_f16_balanced():
    rng = np.random.default_rng(740)
    lens = rng.integers(0, 700, size=160).astype(np.int32)
    batch = f16_batch("f16bal", lens, 32, 8, 128, 16, seed=741)
    batch.new_pos = np.where(lens > 0, lens - 1, -1).astype(np.int32)
    assert pa.pa_decode_plan(160, 32, 8, 128, 16, int(lens.max()), pa.PA_F16, with_workspace=True)["balanced"]
    out = run_step(DeviceBatch(batch), workspace=make_workspace(batch))
    want, _, _ = oracle_step(batch)
    assert max_err(out, want) <= ATOL
    clean()


def test_f16_contiguous():
    cb = workloads.contiguous("f16c", (0, 1, 15, 333, 250), 32, 8, 128, 333, tail_nan=True, f16=True)
    q, k, v, lens = to_dev(cb.query), to_dev(cb.k), to_dev(cb.v), to_dev(cb.context_lens)
    out = torch.empty((cb.num_seqs, cb.num_heads, cb.head_dim), dtype=torch.float32, device="cuda")
    pa.pa_decode_contiguous(out, q, k, v, lens, cb.max_context_len, cb.scale)
    B, L = cb.num_seqs, cb.max_seq_len
    tables = (np.arange(B)[:, None] * L + np.arange(L)[None, :]).astype(np.int32)
    want = oracle.paged_attention(cb.query, cb.k.reshape(B * L, 1, 8, 128), cb.v.reshape(B * L, 1, 8, 128),
                                  tables, cb.context_lens, cb.scale)
    assert max_err(out, want) <= ATOL
    clean()


def shared_prefix_case(seed):
    return workloads.shared_prefix_batch("f16sp", 24, (5, 60, 3, 0, 130), 32, 8, 128, 16, seed_values=seed,
                                         f16=True)


def run_shared(batch, nsh):
    db = DeviceBatch(batch)
    n = pa.pa_decode_shared_prefix_workspace_size(batch.num_seqs, batch.num_heads, batch.num_kv_heads,
                                                  batch.head_dim, batch.block_size, batch.max_context_len, nsh)
    ws = torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty((batch.num_seqs, batch.num_heads, batch.head_dim), dtype=torch.float32, device="cuda")
    pa.pa_decode_shared_prefix(out, db.query, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                               batch.max_context_len, nsh, batch.scale, ws)
    return out


def test_f16_shared_prefix_tcgen05():
    batch = shared_prefix_case(750)
    want = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                  batch.context_lens, batch.scale)
    for nsh in (24, 7):
        assert max_err(run_shared(batch, nsh), want) <= ATOL
    clean()


def child_prefix_mma():
    batch = shared_prefix_case(751)
    want = oracle.paged_attention(batch.query, batch.k_cache, batch.v_cache, batch.block_tables,
                                  batch.context_lens, batch.scale)
    errs = [max_err(run_shared(batch, nsh), want) for nsh in (24, 7)]
    torch.cuda.synchronize()
    print(json.dumps({"errs": errs, "status": pa.pa_device_status(clear=True)}))


def test_f16_shared_prefix_mma_sync():
    env = dict(os.environ, PA_PREFIX_KERNEL="mma")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "child"], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["status"] == 0 and max(res["errs"]) <= ATOL, res


def test_f16_scatter_and_copy_bit_exact():
    rng = np.random.default_rng(760)
    nb, bs, hkv, d, T = 60, 16, 8, 128, 97
    k = rng.standard_normal((nb, bs, hkv, d)).astype(np.float16)
    v = rng.standard_normal((nb, bs, hkv, d)).astype(np.float16)
    key = rng.standard_normal((T, hkv, d)).astype(np.float16)
    val = rng.standard_normal((T, hkv, d)).astype(np.float16)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[::9] = -1
    kd, vd = to_dev(k), to_dev(v)
    pa.pa_reshape_and_cache(to_dev(key), to_dev(val), kd, vd, torch.from_numpy(slots).cuda())
    oracle.reshape_and_cache(k, v, key, val, slots)
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:20], perm[20:40]], axis=1).astype(np.int64)
    pa.pa_copy_blocks(kd, vd, torch.from_numpy(pairs).cuda())
    oracle.copy_blocks(k, v, pairs)
    assert np.array_equal(kd.cpu().numpy().view(np.uint16), k.view(np.uint16))
    assert np.array_equal(vd.cpu().numpy().view(np.uint16), v.view(np.uint16))
    clean()


if __name__ == "__main__" and sys.argv[1:] == ["child"]:
    child_prefix_mma()
