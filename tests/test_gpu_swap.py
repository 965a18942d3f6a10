"""Block swap between the GPU cache and a page-locked CPU pool (pa_swap_blocks)
and a whole preemption round trip through the block manager: bytes are moved
exactly, and decode after swapping back in equals decode before
("PagedAttention, explained.", procedure steps 7-8)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_121_gb300 as pa
import workloads
from gpu_cases import ATOL, max_err, to_dev, to_host_bits

pytestmark = pytest.mark.gpu


def pinned_like(a: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else a.copy())
    t = t.pin_memory()
    return t.view(torch.bfloat16) if a.dtype == np.uint16 else t


@pytest.mark.parametrize("bs,dtype", [(16, "bf16"), (32, "f32"), (8, "bf16")])
@pytest.mark.parametrize("mapping_on_host", [False, True])
def test_swap_blocks_bit_exact(bs, dtype, mapping_on_host):
    rng = np.random.default_rng(bs)
    shape_g, shape_h = (40, bs, 4, 64), (24, bs, 4, 64)
    if dtype == "bf16":
        gk, gv = (rng.integers(0, 2**16, size=shape_g, dtype=np.uint16) for _ in range(2))
        hk, hv = (rng.integers(0, 2**16, size=shape_h, dtype=np.uint16) for _ in range(2))
    else:
        gk, gv = (rng.standard_normal(shape_g).astype(np.float32) for _ in range(2))
        hk, hv = (rng.standard_normal(shape_h).astype(np.float32) for _ in range(2))
    dgk, dgv = to_dev(gk), to_dev(gv)
    phk, phv = pinned_like(hk), pinned_like(hv)
    out_pairs = np.array([[3, 0], [39, 5], [0, 23], [17, 11], [40, 2], [-1, 3], [5, 24]], np.int64)
    m = torch.from_numpy(out_pairs)
    m = m.pin_memory() if mapping_on_host else m.cuda()
    pa.pa_swap_blocks(phk, phv, dgk, dgv, m)              # GPU -> CPU
    torch.cuda.synchronize()
    oracle.swap_blocks(hk, hv, gk, gv, out_pairs)
    assert np.array_equal(to_host_bits(phk) if dtype == "bf16" else phk.numpy(), hk)
    assert np.array_equal(to_host_bits(phv) if dtype == "bf16" else phv.numpy(), hv)
    in_pairs = np.array([[0, 1], [5, 2], [23, 38], [11, 7]], np.int64)
    m2 = torch.from_numpy(in_pairs)
    m2 = m2.pin_memory() if mapping_on_host else m2.cuda()
    pa.pa_swap_blocks(dgk, dgv, phk, phv, m2)            # CPU -> GPU
    torch.cuda.synchronize()
    oracle.swap_blocks(gk, gv, hk, hv, in_pairs)
    assert np.array_equal(to_host_bits(dgk) if dtype == "bf16" else dgk.cpu().numpy(), gk)
    assert np.array_equal(to_host_bits(dgv) if dtype == "bf16" else dgv.cpu().numpy(), gv)


def test_swap_blocks_refuses_pageable_host_memory():
    k = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    pageable = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16)
    m = torch.tensor([[0, 1]], dtype=torch.int64, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_swap_blocks(pageable, pageable, k, k, m)
    assert e.value.status == pa.PA_ERR_INVALID_ARG


def test_preemption_round_trip_through_the_block_manager():
    """Beams sharing a prompt are evicted together to the CPU pool, their GPU
    blocks reused and overwritten by another request, then brought back into
    fresh blocks: decode afterwards is bit-for-bit the decode before."""
    bs, hq, hkv, d, nb = 16, 32, 8, 128, 96
    bm = pa.BlockManager(nb, bs)
    bm.enable_swap(64)
    model = oracle.BlockManagerModel(nb, bs)
    model.enable_swap(64)
    rng = np.random.default_rng(11)
    kd = torch.zeros((nb, bs, hkv, d), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros_like(kd)
    k_h = np.zeros((nb, bs, hkv, d), np.uint16)
    v_h = np.zeros_like(k_h)

    def write(seq, n):
        """Append n tokens of random K/V to seq (copy-on-write first)."""
        pairs, slots = [], []
        for _ in range(n):
            slot, src, dst = bm.append_slot(seq)
            assert (slot, src, dst) == model.append_slot(seq)
            if src >= 0:
                pairs.append((src, dst))
            slots.append(slot)
        if pairs:
            pm = np.array(pairs, np.int64)
            pa.pa_copy_blocks(kd, vd, torch.from_numpy(pm).cuda())
            oracle.copy_blocks(k_h, v_h, pm)
        kk = workloads.bf16_round(rng.standard_normal((n, hkv, d)).astype(np.float32))
        vv = workloads.bf16_round(rng.standard_normal((n, hkv, d)).astype(np.float32))
        sl = np.array(slots, np.int64)
        pa.pa_reshape_and_cache(to_dev(kk), to_dev(vv), kd, vd, torch.from_numpy(sl).cuda())
        oracle.reshape_and_cache(k_h, v_h, kk, vv, sl)

    bm.allocate(0, 0)
    model.allocate(0, 0)
    write(0, 300)                                    # the prompt
    for s in (1, 2):
        bm.fork(0, s)
        model.fork(0, s)
    for s in (0, 1, 2):
        write(s, 40 + 7 * s)                         # each beam's own tokens
    beams = [0, 1, 2]
    query = workloads.bf16_round(rng.standard_normal((3, hq, d)).astype(np.float32))

    def decode():
        tables = np.zeros((3, max(len(bm.block_table(s)) for s in beams)), np.int32)
        for i, s in enumerate(beams):
            t = bm.block_table(s)
            tables[i, :len(t)] = t
        lens = np.array([bm.num_tokens(s) for s in beams], np.int32)
        out = torch.empty((3, hq, d), dtype=torch.float32, device="cuda")
        n = pa.pa_decode_workspace_size(3, hq, hkv, d, bs, int(lens.max()))
        pa.pa_decode(out, to_dev(query), kd, vd, to_dev(tables), to_dev(lens), int(lens.max()),
                     1.0 / np.sqrt(d), workspace=torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda"))
        want = oracle.paged_attention(query, k_h, v_h, tables, lens, 1.0 / np.sqrt(d))
        return out, want

    before, want_before = decode()
    assert max_err(before, want_before) <= ATOL
    hk = torch.zeros((64, bs, hkv, d), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    ok_h = np.zeros((64, bs, hkv, d), np.uint16)          # the oracle's CPU pool
    ov_h = np.zeros_like(ok_h)
    pairs = bm.swap_out(beams)
    assert [tuple(p) for p in pairs.tolist()] == model.swap_out(beams)
    pa.pa_swap_blocks(hk, hv, kd, vd, torch.from_numpy(pairs).cuda())
    oracle.swap_blocks(ok_h, ov_h, k_h, v_h, pairs)
    torch.cuda.synchronize()
    assert np.array_equal(to_host_bits(hk), ok_h) and np.array_equal(to_host_bits(hv), ov_h)
    # another request takes (and overwrites) the freed GPU blocks
    bm.allocate(9, 0)
    model.allocate(9, 0)
    write(9, 16 * 20)
    bm.free(9)
    model.free_seq(9)
    back = bm.swap_in(beams)
    assert [tuple(p) for p in back.tolist()] == model.swap_in(beams)
    pa.pa_swap_blocks(kd, vd, hk, hv, torch.from_numpy(back).cuda())
    oracle.swap_blocks(k_h, v_h, ok_h, ov_h, back)
    after, want_after = decode()
    assert torch.equal(before, after)                # same values in logical order: same result
    assert max_err(after, want_after) <= ATOL
    assert np.array_equal(to_host_bits(kd), k_h) and np.array_equal(to_host_bits(vd), v_h)
