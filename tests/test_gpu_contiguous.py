"""Decode over a contiguous (unpaged) cache, the baseline paging is measured
against ("Paged Attention: Virtual Memory for the KV Cache", "What paging
costs"): parity with the fp64 oracle, and bit-for-bit equality with paged
decode over the same values ("PagedAttention: KV cache virtual memory",
"Misconceptions": the layout changes how K and V are fetched, not the
result)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import ATOL, max_err, to_dev

pytestmark = pytest.mark.gpu


def oracle_contiguous(cb):
    """The oracle over the contiguous cache read as a pool of one-token
    blocks: sequence b's token t is block b * max_seq_len + t."""
    B, L = cb.num_seqs, cb.max_seq_len
    k = cb.k.reshape(B * L, 1, cb.num_kv_heads, cb.head_dim)
    v = cb.v.reshape(B * L, 1, cb.num_kv_heads, cb.head_dim)
    tables = (np.arange(B, dtype=np.int64)[:, None] * L + np.arange(L)[None, :]).astype(np.int32)
    return oracle.paged_attention(cb.query, k, v, tables, cb.context_lens, cb.scale)


def workspace_for(cb):
    n = pa.pa_decode_workspace_size(cb.num_seqs, cb.num_heads, cb.num_kv_heads, cb.head_dim, 16,
                                    cb.max_context_len)
    return torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda")


def run_contiguous(cb, workspace=None, out_dtype=torch.float32, max_context_len=None):
    q, k, v, lens = to_dev(cb.query), to_dev(cb.k), to_dev(cb.v), to_dev(cb.context_lens)
    out = torch.empty((cb.num_seqs, cb.num_heads, cb.head_dim), dtype=out_dtype, device="cuda")
    mcl = cb.max_context_len if max_context_len is None else max_context_len
    pa.pa_decode_contiguous(out, q, k, v, lens, mcl, cb.scale, workspace=workspace)
    torch.cuda.synchronize()
    assert pa.pa_device_status(clear=True) == 0
    return out


CONTIG = [
    # lens, Hq, Hkv, D, max_seq_len
    ((0, 1, 15, 16, 17, 100), 8, 2, 128, 100),
    ((1, 333, 250), 32, 8, 128, 333),       # rows per sequence not a multiple of 16
    ((5, 40, 129), 4, 4, 64, 130),          # G = 1
    ((3, 77, 300), 16, 1, 64, 301),         # G = 16
    ((50, 260), 64, 2, 128, 270),           # G = 32: two head tiles
    ((33, 200, 17), 24, 12, 128, 200),      # 12 KV heads
    ((700, 1, 2048), 16, 4, 128, 2049),     # split contexts
]


@pytest.mark.parametrize("case", range(len(CONTIG)))
@pytest.mark.parametrize("use_ws", [False, True])
def test_contiguous_small(case, use_ws):
    lens, Hq, Hkv, D, L = CONTIG[case]
    cb = workloads.contiguous("contig", lens, Hq, Hkv, D, L, tail_nan=True, seed_values=700 + case)
    out = run_contiguous(cb, workspace_for(cb) if use_ws else None)
    err = max_err(out, oracle_contiguous(cb))
    assert err <= ATOL, err


def test_contiguous_bf16_output_and_short_max_context():
    cb = workloads.contiguous("contig", (90, 33, 64), 16, 4, 128, 96, seed_values=731)
    want = oracle_contiguous(cb)
    out = run_contiguous(cb, out_dtype=torch.bfloat16)
    g = out.float().cpu().numpy()
    # rounding the output to bf16 adds at most half an ulp: 2^-8 relative
    assert np.all(np.abs(g - want) <= ATOL + np.abs(want) * 2.0 ** -8)
    # a host bound below the longest length attends to that many tokens only
    cb2 = workloads.contiguous("contig", (90, 33, 64), 16, 4, 128, 96, seed_values=731)
    cb2.context_lens = np.minimum(cb2.context_lens, 40).astype(np.int32)
    out2 = run_contiguous(cb2, max_context_len=40)
    assert max_err(out2, oracle_contiguous(cb2)) <= ATOL


def test_contiguous_refuses_bad_arguments():
    cb = workloads.contiguous("contig", (10,), 8, 2, 128, 16, seed_values=732)
    q, k, v, lens = to_dev(cb.query), to_dev(cb.k), to_dev(cb.v), to_dev(cb.context_lens)
    out = torch.empty((1, 8, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(pa.PAError):          # max_context_len above the reservation
        pa.pa_decode_contiguous(out, q, k, v, lens, 17, cb.scale)
    k32 = k.float()
    with pytest.raises(pa.PAError):          # fp32 caches: tensor-core kernel only
        pa.pa_decode_contiguous(out, q.float(), k32, k32, lens, 10, cb.scale)


@pytest.mark.parametrize("use_ws", [False, True])
def test_contiguous_equals_paged_bitwise(use_ws):
    """The same rows as a contiguous cache and as 16-token blocks scattered
    over a pool by a seeded permutation: the outputs are identical."""
    lens = (4164, 4164, 4164, 4164, 1000, 17)
    B, L, Hq, Hkv, D = len(lens), 4176, 32, 8, 128
    cb = workloads.contiguous("eq", lens, Hq, Hkv, D, L, seed_values=733)
    nblk = L // 16
    perm = np.random.default_rng(734).permutation(B * nblk)
    pk = np.empty((B * nblk, 16, Hkv, D), dtype=np.uint16)
    pv = np.empty_like(pk)
    pk[perm] = cb.k.reshape(B * nblk, 16, Hkv, D)
    pv[perm] = cb.v.reshape(B * nblk, 16, Hkv, D)
    tables = perm.reshape(B, nblk).astype(np.int32)
    ws = workspace_for(cb) if use_ws else None
    out_c = run_contiguous(cb, ws)
    q, lens_d = to_dev(cb.query), to_dev(cb.context_lens)
    out_p = torch.empty_like(out_c)
    pa.pa_decode(out_p, q, to_dev(pk), to_dev(pv), to_dev(tables), lens_d, cb.max_context_len, cb.scale,
                 workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out_c, out_p)
    assert max_err(out_c, oracle_contiguous(cb)) <= ATOL


@pytest.mark.parametrize("shape", ["qwen3", "long"])
def test_contiguous_full_size(shape):
    """The bench's contiguous baselines: 16 x 4,164 tokens (Hq 32) and
    4 x 32,768 tokens (Hq 64), Hkv 8, D 128, with the bench's workspace."""
    if shape == "qwen3":
        cb = workloads.contiguous("qwen3", [4164] * 16, 32, 8, 128, 4164, seed_values=735)
    else:
        cb = workloads.contiguous("long", [32768] * 4, 64, 8, 128, 32768, seed_values=736)
    out = run_contiguous(cb, workspace_for(cb))
    assert max_err(out, oracle_contiguous(cb)) <= ATOL
