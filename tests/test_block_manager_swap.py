"""CPU tests of the host block manager's swapping and of beam-search style
sharing, against the oracle's list model ("PagedAttention, explained.",
procedure steps 6-8: reference-counted sharing among the beams of a request,
copy-on-write, eviction of a request's blocks all at once -- sharing
sequences together -- to CPU memory and back)."""
import numpy as np
import pytest

import oracle
import paged_kv_cache_121_gb300 as pa


def compare(bm, model, live):
    for s in live:
        assert bm.block_table(s) == model.block_table(s)
        assert bm.num_tokens(s) == model.num_tokens(s)
        assert bm.is_swapped(s) == (s in model.swapped)
    assert bm.free_list() == model.free
    st = bm.stats()
    for k, v in model.stats().items():
        assert st[k] == v, k
    for b in range(model.num_blocks):
        assert bm.refcount(b) == model.refcount[b]
    if model.host_free is not None:
        sw = bm.swap_stats()
        assert sw["free_host_blocks"] == len(model.host_free)
        assert sw["swapped_seqs"] == len(model.swapped)


def expect_same(model_call, bm_call):
    """Run the model's operation, then the library's; both succeed with the
    same result or fail with the matching status."""
    try:
        want = model_call()
    except oracle.OutOfBlocks:
        with pytest.raises(pa.PAError) as e:
            bm_call()
        assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
        return None, False
    except ValueError:
        with pytest.raises(pa.PAError) as e:
            bm_call()
        assert e.value.status == pa.PA_ERR_INVALID_ARG
        return None, False
    got = bm_call()
    return (want, got), True


@pytest.mark.parametrize("seed", range(6))
def test_swap_matches_model_on_random_ops(seed):
    rng = np.random.default_rng(1000 + seed)
    nb, bs, nh = int(rng.integers(10, 40)), int(rng.choice([1, 4, 16])), int(rng.integers(4, 40))
    bm = pa.BlockManager(nb, bs)
    model = oracle.BlockManagerModel(nb, bs)
    bm.enable_swap(nh)
    model.enable_swap(nh)
    live, next_id = [], 100
    for _ in range(500):
        op = rng.choice(["alloc", "append", "append", "fork", "free", "out", "out", "in", "in"])
        if op == "alloc" or not live:
            n = int(rng.integers(0, 3 * bs + 2))
            r, ok = expect_same(lambda: model.allocate(next_id, n), lambda: bm.allocate(next_id, n))
            if ok:
                live.append(next_id)
            next_id += 1
        elif op == "append":
            s = int(rng.choice(live))
            r, ok = expect_same(lambda: model.append_slot(s), lambda: bm.append_slot(s))
            if ok:
                assert r[0] == r[1]
        elif op == "fork":
            s = int(rng.choice(live))
            r, ok = expect_same(lambda: model.fork(s, next_id), lambda: bm.fork(s, next_id))
            if ok:
                live.append(next_id)
            next_id += 1
        elif op == "free":
            s = int(rng.choice(live))
            model.free_seq(s)
            bm.free(s)
            live.remove(s)
        else:
            k = int(rng.integers(1, min(4, len(live)) + 1))
            group = [int(x) for x in rng.choice(live, size=k, replace=False)]
            if op == "out":
                r, ok = expect_same(lambda: model.swap_out(group), lambda: bm.swap_out(group))
            else:
                r, ok = expect_same(lambda: model.swap_in(group), lambda: bm.swap_in(group))
            if ok:
                assert [tuple(p) for p in r[1].tolist()] == r[0]
        compare(bm, model, live)


def test_swap_out_and_back_keeps_the_sharing_pattern():
    """Three beams sharing a 3-block prompt and each owning one block: the
    group moves out as 6 distinct blocks, the GPU pool gets them back, and
    swapping in restores the same sharing with fresh GPU blocks."""
    bs = 4
    bm = pa.BlockManager(16, bs)
    bm.enable_swap(8)
    bm.allocate(0, 12)                     # 3 full blocks
    bm.fork(0, 1)
    bm.fork(0, 2)
    for s in (0, 1, 2):
        bm.append_slot(s)                  # each beam's first private block
    before = {s: bm.block_table(s) for s in (0, 1, 2)}
    free_before = bm.stats()["free_blocks"]
    with pytest.raises(pa.PAError) as e:   # beam 0 alone shares the prompt with 1 and 2
        bm.swap_out([0])
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    pairs = bm.swap_out([0, 1, 2])
    assert pairs.shape == (6, 2)
    assert pairs[:, 0].tolist() == before[0] + [before[1][3], before[2][3]]
    assert pairs[:, 1].tolist() == list(range(6))   # CPU ids from the front of their queue
    assert bm.stats()["free_blocks"] == free_before + 6
    assert bm.block_table(1) == [0, 1, 2, 4]
    with pytest.raises(pa.PAError):
        bm.append_slot(1)                  # swapped out: no growth
    back = bm.swap_in([2, 1, 0])
    assert back.shape == (6, 2)
    after = {s: bm.block_table(s) for s in (0, 1, 2)}
    for s in (0, 1, 2):                    # the prompt blocks are shared again, privates private
        assert after[s][:3] == after[0][:3]
    assert len({after[s][3] for s in (0, 1, 2)}) == 3
    assert all(bm.refcount(b) == 3 for b in after[0][:3])
    assert bm.swap_stats() == {"host_blocks": 8, "free_host_blocks": 8, "swapped_seqs": 0}


# The beams-and-prompt case above worked out by hand from the rules on the
# pages ("PagedAttention, explained.", procedure steps 7-8: a request's blocks
# go out together; "Paged Attention: Virtual Memory for the KV Cache", "Inside
# vLLM: the block pool": allocation pops the free queue's front, freed blocks
# go back to its front). Pool of 16 with the null block reserved: queue 1..15.
#   allocate(0, 12) -> [1, 2, 3]; forks share them; each beam's append takes
#   the next block: beams 0/1/2 = [1,2,3,4] / [1,2,3,5] / [1,2,3,6].
#   swap_out([0, 1, 2]): distinct blocks in order of first appearance
#   1,2,3,4,5,6 -> CPU 0..5; beam 1 reads [0, 1, 2, 4].
#   swap_in([2, 1, 0]): first appearance over beams 2, 1, 0 is CPU 0,1,2,5,4,3;
#   GPU blocks 1..6 come back off the queue front in that order.
HAND_SWAP_OUT = [(1, 0), (2, 1), (3, 2), (4, 3), (5, 4), (6, 5)]
HAND_SWAP_IN = [(0, 1), (1, 2), (2, 3), (5, 4), (4, 5), (3, 6)]
HAND_TABLES_AFTER = {0: [1, 2, 3, 6], 1: [1, 2, 3, 5], 2: [1, 2, 3, 4]}


def _beams(mgr):
    mgr.enable_swap(8)
    mgr.allocate(0, 12)
    mgr.fork(0, 1)
    mgr.fork(0, 2)
    for s in (0, 1, 2):
        mgr.append_slot(s)


def test_swap_model_matches_hand_worked_case():
    """The oracle's block-manager model on the case worked out by hand."""
    model = oracle.BlockManagerModel(16, 4)
    _beams(model)
    assert [model.block_table(s) for s in (0, 1, 2)] == [[1, 2, 3, 4], [1, 2, 3, 5], [1, 2, 3, 6]]
    with pytest.raises(ValueError):
        model.swap_out([0])                # shares the prompt with beams 1 and 2
    assert model.swap_out([0, 1, 2]) == HAND_SWAP_OUT
    assert model.block_table(1) == [0, 1, 2, 4]
    assert model.stats()["free_blocks"] == 15 and model.free[:6] == [1, 2, 3, 4, 5, 6]
    with pytest.raises(ValueError):
        model.append_slot(1)
    assert model.swap_in([2, 1, 0]) == HAND_SWAP_IN
    assert {s: model.block_table(s) for s in (0, 1, 2)} == HAND_TABLES_AFTER
    assert all(model.refcount[b] == 3 for b in (1, 2, 3))
    assert model.host_free == [0, 1, 2, 5, 4, 3, 6, 7]


def test_swap_libpa_matches_hand_worked_case():
    bm = pa.BlockManager(16, 4)
    _beams(bm)
    assert bm.swap_out([0, 1, 2]).tolist() == [list(p) for p in HAND_SWAP_OUT]
    assert bm.swap_in([2, 1, 0]).tolist() == [list(p) for p in HAND_SWAP_IN]
    assert {s: bm.block_table(s) for s in (0, 1, 2)} == HAND_TABLES_AFTER


def test_swap_is_all_or_nothing():
    bm = pa.BlockManager(10, 4)
    bm.enable_swap(2)
    bm.allocate(0, 12)                     # 3 blocks, CPU pool holds 2
    free = bm.free_list()
    with pytest.raises(pa.PAError) as e:
        bm.swap_out([0])
    assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
    assert bm.free_list() == free and not bm.is_swapped(0)
    bm2 = pa.BlockManager(10, 4)
    with pytest.raises(pa.PAError):        # no CPU pool
        bm2.swap_out([0])


def test_beam_search_sharing_matches_model():
    """Beam search over a shared prompt: every step each live beam appends a
    token (copy-on-write of its shared last block), then half the beams are
    pruned and the survivors fork. Counts, copies and the final release of
    every block agree with the model."""
    rng = np.random.default_rng(7)
    bs, nb, width = 4, 64, 6
    bm = pa.BlockManager(nb, bs)
    model = oracle.BlockManagerModel(nb, bs)
    bm.allocate(0, 10)
    model.allocate(0, 10)
    beams, next_id, cow = [0], 1, 0
    for b in range(1, width):
        bm.fork(0, b)
        model.fork(0, b)
        beams.append(b)
    next_id = width
    for step in range(12):
        for b in beams:
            got, want = bm.append_slot(b), model.append_slot(b)
            assert got == want
            cow += got[1] >= 0
        keep = sorted(int(x) for x in rng.choice(beams, size=width // 2, replace=False))
        for b in beams:
            if b not in keep:
                bm.free(b)
                model.free_seq(b)
        beams = list(keep)
        for b in keep:                      # each survivor spawns one child
            bm.fork(b, next_id)
            model.fork(b, next_id)
            beams.append(next_id)
            next_id += 1
        compare(bm, model, beams)
    assert bm.stats()["cow_copies"] == cow == model.cow_copies
    assert cow > 0
    for b in beams:
        bm.free(b)
        model.free_seq(b)
    assert bm.stats()["free_blocks"] == nb - 1 and bm.stats()["used_blocks"] == 0
    assert bm.free_list() == model.free


def test_oracle_swap_blocks_round_trip_and_skips():
    """The oracle's block swap: out and back restores every byte; a pair
    naming a block outside its pool moves nothing; other blocks are untouched."""
    rng = np.random.default_rng(3)
    gk = rng.integers(0, 2**16, size=(9, 4, 2, 8), dtype=np.uint16)
    gv = rng.integers(0, 2**16, size=(9, 4, 2, 8), dtype=np.uint16)
    hk, hv = np.zeros((5, 4, 2, 8), np.uint16), np.zeros((5, 4, 2, 8), np.uint16)
    pairs = [(7, 0), (2, 1), (4, 2), (8, 9), (-1, 3)]        # the last two are skipped
    oracle.swap_blocks(hk, hv, gk, gv, pairs)
    assert np.array_equal(hk[:3], gk[[7, 2, 4]]) and np.array_equal(hv[:3], gv[[7, 2, 4]])
    assert not hk[3:].any() and not hv[3:].any()
    k0, v0 = gk.copy(), gv.copy()
    gk[[7, 2, 4]] = 0
    gv[[7, 2, 4]] = 0
    oracle.swap_blocks(gk, gv, hk, hv, [(0, 7), (1, 2), (2, 4)])
    assert np.array_equal(gk, k0) and np.array_equal(gv, v0)
