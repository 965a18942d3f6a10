"""Pins for the oracle's paged decode attention, split partitions and merge.

The pages print no numeric attention output, so the oracle is pinned to what
they and the mathematics fix:
  * paging does not change the result ("PagedAttention: KV cache virtual
    memory", section "Misconceptions"; "What Does PagedAttention Actually
    Optimize?", section 8): the paged oracle must equal torch's
    scaled_dot_product_attention (fp64, CPU) run on the dense, contiguous
    K and V the pool was built from -- the pool is made here by reshaping the
    dense arrays into blocks and scattering whole blocks to random pool
    positions, with the unused tail slots filled with NaN;
  * a random re-placement of the physical blocks leaves the output bitwise
    unchanged;
  * closed forms: one token returns its V; equal keys return the mean of V;
    V = 1 returns 1 (the weights sum to one); scale 0 returns the mean of V;
    one dominant key returns its V;
  * partitions: each partition is attention over its own tokens; its max and
    sum give torch.logsumexp of its scores; merging gives the whole-context
    result.
A mutation test plants plausible mistakes in a copy of the oracle's C source
and checks that these pins catch every one.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import bf16_round, bf16_to_f32

NAN_BF16 = np.uint16(0x7FC0)


def paged_from_dense(dense_k, dense_v, block_size, num_blocks, rng, bf16):
    """Pool + tables from per-sequence dense [len, Hkv, D] arrays, by reshape
    into whole blocks and random placement; tail slots are NaN."""
    B = len(dense_k)
    hkv, d = dense_k[0].shape[1:]
    dt = np.uint16 if bf16 else np.float32
    nan = NAN_BF16 if bf16 else np.float32(np.nan)
    kpool = np.full((num_blocks, block_size, hkv, d), nan, dtype=dt)
    vpool = np.full_like(kpool, nan)
    nblk = [-(-x.shape[0] // block_size) for x in dense_k]
    tables = np.zeros((B, max(1, max(nblk))), dtype=np.int32)
    perm = rng.permutation(num_blocks)
    pos = 0
    for b in range(B):
        n = nblk[b]
        if n == 0:
            continue
        padded_k = np.full((n * block_size, hkv, d), nan, dtype=dt)
        padded_v = np.full_like(padded_k, nan)
        padded_k[:dense_k[b].shape[0]] = dense_k[b]
        padded_v[:dense_v[b].shape[0]] = dense_v[b]
        ids = perm[pos:pos + n]
        pos += n
        kpool[ids] = padded_k.reshape(n, block_size, hkv, d)
        vpool[ids] = padded_v.reshape(n, block_size, hkv, d)
        tables[b, :n] = ids
    return kpool, vpool, tables


def widen(x, bf16):
    return (bf16_to_f32(x) if bf16 else np.asarray(x, dtype=np.float32)).astype(np.float64)


def sdpa_reference(q, K, V, scale):
    """torch SDPA in fp64: q [Hq, D], K/V [len, Hkv, D] -> [Hq, D]."""
    Hq = q.shape[0]
    G = Hq // K.shape[1]
    k = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0)
    v = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0)
    qt = torch.from_numpy(q)[:, None, :]
    return F.scaled_dot_product_attention(qt, k, v, scale=scale)[:, 0, :].numpy()


def make_case(lens, Hq, Hkv, D, bs, bf16, seed, num_blocks=None):
    rng = np.random.default_rng(seed)
    dt_draw = lambda shape: (bf16_round(rng.standard_normal(shape, dtype=np.float32)) if bf16
                             else rng.standard_normal(shape, dtype=np.float32))
    dense_k = [dt_draw((n, Hkv, D)) for n in lens]
    dense_v = [dt_draw((n, Hkv, D)) for n in lens]
    q = dt_draw((len(lens), Hq, D))
    need = sum(-(-n // bs) for n in lens)
    nb = num_blocks or need + 7
    kpool, vpool, tables = paged_from_dense(dense_k, dense_v, bs, nb, rng, bf16)
    return dict(q=q, dense_k=dense_k, dense_v=dense_v, kpool=kpool, vpool=vpool, tables=tables,
                lens=np.asarray(lens, np.int32), bf16=bf16, scale=1.0 / np.sqrt(D), bs=bs)


CASES = [
    # lens, Hq, Hkv, D, block_size, bf16
    ((1, 15, 16, 17, 33), 4, 4, 64, 16, False),
    ((25, 47, 12), 4, 4, 64, 16, False),
    ((5, 31, 64, 70), 8, 2, 64, 8, True),
    ((40, 7), 8, 1, 128, 4, True),
    ((100, 3, 65), 12, 4, 128, 32, True),
]


# ---------------------------------------------------------------------------
# pins, written as functions of the oracle entry points so that the mutation
# test can run them against a planted-mistake build
# ---------------------------------------------------------------------------
def pin_contiguous_sdpa(lib=None):
    for i, (lens, Hq, Hkv, D, bs, bf16) in enumerate(CASES):
        c = make_case(lens, Hq, Hkv, D, bs, bf16, seed=1000 + i)
        out = oracle.paged_attention(c["q"], c["kpool"], c["vpool"], c["tables"], c["lens"],
                                     c["scale"], nthreads=2, lib=lib)
        q64 = widen(c["q"], bf16)
        for b, n in enumerate(lens):
            ref = sdpa_reference(q64[b], widen(c["dense_k"][b], bf16), widen(c["dense_v"][b], bf16),
                                 c["scale"])
            assert np.allclose(out[b], ref, rtol=0, atol=1e-12), (i, b)


def pin_permutation_invariance(lib=None):
    lens, Hq, Hkv, D, bs, bf16 = CASES[2]
    a = make_case(lens, Hq, Hkv, D, bs, bf16, seed=7, num_blocks=64)
    rng = np.random.default_rng(99)
    kpool, vpool, tables = paged_from_dense(a["dense_k"], a["dense_v"], bs, 64, rng, bf16)
    o1 = oracle.paged_attention(a["q"], a["kpool"], a["vpool"], a["tables"], a["lens"], a["scale"], lib=lib)
    o2 = oracle.paged_attention(a["q"], kpool, vpool, tables, a["lens"], a["scale"], lib=lib)
    assert not np.array_equal(a["tables"], tables)
    assert np.array_equal(o1, o2)


def pin_closed_forms(lib=None):
    rng = np.random.default_rng(5)
    Hq, Hkv, D, bs = 6, 3, 64, 8
    # one token: softmax of a single score is 1, the output is that V exactly
    dk = [rng.standard_normal((1, Hkv, D)).astype(np.float32)]
    dv = [rng.standard_normal((1, Hkv, D)).astype(np.float32)]
    kp, vp, tb = paged_from_dense(dk, dv, bs, 4, rng, False)
    q = rng.standard_normal((1, Hq, D)).astype(np.float32)
    out = oracle.paged_attention(q, kp, vp, tb, [1], 0.125, lib=lib)
    for h in range(Hq):
        assert np.array_equal(out[0, h], dv[0][0, h // 2].astype(np.float64))
    # equal keys: uniform weights, the output is the mean of V
    n = 37
    key = rng.standard_normal((1, Hkv, D)).astype(np.float32)
    dk = [np.repeat(key, n, axis=0)]
    dv = [rng.standard_normal((n, Hkv, D)).astype(np.float32)]
    kp, vp, tb = paged_from_dense(dk, dv, bs, 16, rng, False)
    out = oracle.paged_attention(q, kp, vp, tb, [n], 0.125, lib=lib)
    mean_v = dv[0].astype(np.float64).mean(axis=0)
    for h in range(Hq):
        assert np.allclose(out[0, h], mean_v[h // 2], rtol=0, atol=1e-12)
    # scale 0: uniform weights as well
    dk = [rng.standard_normal((n, Hkv, D)).astype(np.float32)]
    kp, vp, tb = paged_from_dense(dk, dv, bs, 16, rng, False)
    out = oracle.paged_attention(q, kp, vp, tb, [n], 0.0, lib=lib)
    for h in range(Hq):
        assert np.allclose(out[0, h], mean_v[h // 2], rtol=0, atol=1e-12)
    # V = 1 everywhere: the output is the sum of the weights, i.e. 1
    ones = [np.ones((n, Hkv, D), np.float32)]
    kp, vp, tb = paged_from_dense(dk, ones, bs, 16, rng, False)
    out = oracle.paged_attention(q, kp, vp, tb, [n], 0.125, lib=lib)
    assert np.allclose(out, 1.0, rtol=0, atol=1e-14)
    # one dominant key: its weight is 1 to double precision
    dk = [rng.standard_normal((n, Hkv, D)).astype(np.float32) * 0.01]
    j = 11
    dk[0][j] = 0
    qd = np.zeros((1, Hq, D), np.float32)
    qd[0, :, 0] = 100.0
    dk[0][j, :, 0] = 100.0
    kp, vp, tb = paged_from_dense(dk, dv, bs, 16, rng, False)
    out = oracle.paged_attention(qd, kp, vp, tb, [n], 1.0, lib=lib)
    for h in range(Hq):
        assert np.allclose(out[0, h], dv[0][j, h // 2], rtol=0, atol=1e-12)


def pin_partitions_and_merge(lib=None):
    lens, Hq, Hkv, D, bs = (70, 33, 8, 1), 8, 2, 64, 8
    c = make_case(lens, Hq, Hkv, D, bs, True, seed=31)
    ps, P = 16, 5
    po, pm, psum = oracle.paged_attention_partitions(c["q"], c["kpool"], c["vpool"], c["tables"],
                                                     c["lens"], c["scale"], ps, P, lib=lib)
    q64 = widen(c["q"], True)
    for b, n in enumerate(lens):
        K = widen(c["dense_k"][b], True)
        V = widen(c["dense_v"][b], True)
        for p in range(P):
            t0, t1 = p * ps, min(n, (p + 1) * ps)
            if t1 <= t0:
                assert np.all(po[b, :, p] == 0) and np.all(psum[b, :, p] == 0)
                assert np.all(np.isneginf(pm[b, :, p]))
                continue
            ref = sdpa_reference(q64[b], K[t0:t1], V[t0:t1], c["scale"])
            assert np.allclose(po[b, :, p], ref, rtol=0, atol=1e-12)
            G = Hq // Hkv
            for h in range(Hq):
                s = torch.from_numpy(K[t0:t1, h // G] @ q64[b, h] * c["scale"])
                lse = torch.logsumexp(s, 0).item()
                assert abs(pm[b, h, p] + np.log(psum[b, h, p]) - lse) < 1e-12
    merged = oracle.lse_merge(po, pm, psum, lib=lib)
    full = oracle.paged_attention(c["q"], c["kpool"], c["vpool"], c["tables"], c["lens"], c["scale"], lib=lib)
    assert np.allclose(merged, full, rtol=0, atol=1e-12)


PINS = [pin_contiguous_sdpa, pin_permutation_invariance, pin_closed_forms, pin_partitions_and_merge]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin()


def test_oracle_rejects_block_outside_pool():
    c = make_case((20,), 2, 2, 64, 16, False, seed=3)
    tables = c["tables"].copy()
    tables[0, 1] = c["kpool"].shape[0]
    with pytest.raises(ValueError):
        oracle.paged_attention(c["q"], c["kpool"], c["vpool"], tables, c["lens"], c["scale"])


def test_oracle_ignores_table_entries_past_the_context():
    c = make_case((20,), 2, 2, 64, 16, False, seed=4)
    tables = np.concatenate([c["tables"], np.full((1, 3), 10**6, np.int32)], axis=1)
    a = oracle.paged_attention(c["q"], c["kpool"], c["vpool"], c["tables"], c["lens"], c["scale"])
    b = oracle.paged_attention(c["q"], c["kpool"], c["vpool"], tables, c["lens"], c["scale"])
    assert np.array_equal(a, b)


# ---------------------------------------------------------------------------
# planted mistakes: every one must be caught by at least one pin
# ---------------------------------------------------------------------------
MUTATIONS = {
    "dropped_scale": ("        s *= scale;\n", "        (void)scale;\n"),
    "wrong_kv_head": ("* num_kv_heads + g) * (int64_t)head_dim;",
                      "* num_kv_heads + 0) * (int64_t)head_dim;"),
    "interleaved_gqa": ("for (int h = g * group; h < (g + 1) * group; ++h) {",
                        "for (int h = g; h < num_heads; h += num_kv_heads) {"),
    "reversed_offset": ("int offset = t % block_size;",
                        "int offset = block_size - 1 - t % block_size;"),
    "logical_off_by_one": ("int logical = t / block_size;",
                           "int logical = (t + 1) / block_size < max_logical ? (t + 1) / block_size : t / block_size;"),
    "unnormalised": ("double p = exp(score[t - t0] - m) / l;", "double p = exp(score[t - t0] - m);"),
    "merge_ignores_sums": ("double w = sm[p] * exp(mx[p] - M);", "double w = exp(mx[p] - M);"),
    "partition_off_by_one": ("int t0 = partition_size > 0 ? p * partition_size : 0;",
                             "int t0 = partition_size > 0 ? (p > 0 ? p * partition_size - 1 : 0) : 0;"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "paged_attention.c")).read()
    assert src.count(old) == 1, name
    mutated = src.replace(old, new)
    if name == "logical_off_by_one":
        mutated = mutated.replace("    for (int t = 0; t < len; ++t) {\n        int logical",
                                  "    int max_logical = (len + block_size - 1) / block_size;\n"
                                  "    for (int t = 0; t < len; ++t) {\n        int logical", 1)
    c = tmp_path / f"{name}.c"
    c.write_text(mutated)
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"],
                   check=True)
    return oracle.load_library(str(so))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(tmp_path, name):
    old, new = MUTATIONS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    caught = []
    for pin in PINS:
        try:
            pin(lib=lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {name}"


def test_oracle_fp16_inputs():
    """fp16 caches and queries are widened exactly ("What Does PagedAttention
    Actually Optimize?", section 2: fp16 and bf16 both two bytes a value).
    Pinned two ways: a one-token context returns its V row, bit for bit, at
    the edges of the fp16 range; and a random fp16 batch through the paged
    pool equals torch SDPA on the dense, widened arrays."""
    edge = np.array([65504.0, -65504.0, 2.0 ** -14, 2.0 ** -24, -0.0, 1.0 / 3.0, -2.5, 1.0], np.float16)
    hkv, d, bs = 1, 64, 16
    v = np.zeros((4, bs, hkv, d), np.float16)
    k = np.zeros_like(v)
    v[2, 0, 0, :8] = edge
    v[2, 0, 0, 8:] = np.float16(0.75)
    k[2, 0, 0, :] = np.float16(0.5)
    q = np.full((1, 2, d), np.float16(-1.25), np.float16)
    out = oracle.paged_attention(q, k, v, np.array([[2]], np.int32), np.array([1], np.int32), 0.125)
    for h in range(2):
        assert np.array_equal(out[0, h], v[2, 0, 0].astype(np.float64))

    rng = np.random.default_rng(31)
    lens = [37, 5, 64]
    hq, hkv, d, bs = 8, 2, 64, 16
    dk = [rng.standard_normal((n, hkv, d)).astype(np.float16) for n in lens]
    dv = [rng.standard_normal((n, hkv, d)).astype(np.float16) for n in lens]
    q = rng.standard_normal((len(lens), hq, d)).astype(np.float16)
    kpool = np.zeros((12, bs, hkv, d), np.float16)
    vpool = np.zeros_like(kpool)
    tables = np.zeros((len(lens), 4), np.int32)
    perm = rng.permutation(12)
    pos = 0
    for b, n in enumerate(lens):
        nb = -(-n // bs)
        for j in range(nb):
            rows = slice(j * bs, min(n, (j + 1) * bs))
            kpool[perm[pos], :rows.stop - rows.start] = dk[b][rows]
            vpool[perm[pos], :rows.stop - rows.start] = dv[b][rows]
            tables[b, j] = perm[pos]
            pos += 1
    out = oracle.paged_attention(q, kpool, vpool, tables, np.array(lens, np.int32), d ** -0.5)
    for b, n in enumerate(lens):
        want = sdpa_reference(q[b].astype(np.float64), dk[b].astype(np.float64), dv[b].astype(np.float64),
                              d ** -0.5)
        assert np.max(np.abs(out[b] - want)) < 1e-12
