"""CPU tests of libpa: it loads, exports every symbol include/pa.h declares,
rejects bad arguments on the host before any launch, and its host block
manager and slot map agree with the oracle (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import paged_kv_cache_121_gb300 as pa
from paged_kv_cache_121_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    names = declared_symbols()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding declares a signature for each of them
    assert set(names) == set(_lib.SIGNATURES), set(names) ^ set(_lib.SIGNATURES)


def test_status_strings_and_version():
    lib = _lib.load()
    assert lib.pa_abi_version() == 2
    for code in range(8):
        assert lib.pa_status_string(code)
    assert lib.pa_status_string(99) == b"unknown status"


def test_host_argument_checks_return_before_launch():
    lib = _lib.load()
    s = None
    # decode: bad head_dim, bad GQA ratio, context longer than the table
    args = dict(out=None, out_dtype=0, query=None, q_dtype=0, k=None, v=None, kv_dtype=0, bt=None,
                cl=None, B=1, Hq=4, Hkv=4, D=64, BS=16, maxb=2, nb=8, maxctx=20, scale=0.125)

    def decode(**kw):
        a = dict(args, **kw)
        return lib.pa_decode(a["out"], a["out_dtype"], a["query"], a["q_dtype"], a["k"], a["v"],
                             a["kv_dtype"], a["bt"], a["cl"], a["B"], a["Hq"], a["Hkv"], a["D"],
                             a["BS"], a["maxb"], a["nb"], a["maxctx"], a["scale"], None, 0, s)

    assert decode(D=96) == pa.PA_ERR_UNSUPPORTED
    assert decode(Hq=6, Hkv=4) == pa.PA_ERR_INVALID_ARG
    assert decode(maxctx=33) == pa.PA_ERR_INVALID_ARG
    assert decode(q_dtype=0, kv_dtype=1) == pa.PA_ERR_UNSUPPORTED
    assert decode(out_dtype=7) == pa.PA_ERR_INVALID_ARG
    assert decode(scale=float("nan")) == pa.PA_ERR_INVALID_ARG
    assert decode(B=0) == pa.PA_OK                     # nothing to do
    assert decode() == pa.PA_ERR_INVALID_ARG           # null pointers
    # split-K: partition size must be a multiple of the block size
    assert lib.pa_decode_splitk(None, None, None, 24, None, 1, None, None, 1, None, None, 1, 4, 4,
                                64, 16, 2, 8, 20, 0.1, s) == pa.PA_ERR_INVALID_ARG
    # scatter / copy: nothing to do is fine, null pointers are not
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, 8, 16, 4, 64, 1, s) == pa.PA_OK
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 3, 8, 16, 4, 64, 1, s) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_copy_blocks(None, None, None, 0, 8, 16, 4, 64, 1, s) == pa.PA_OK
    assert lib.pa_copy_blocks(None, None, None, 2, 8, 16, 4, 64, 1, s) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_lse_merge(None, 0, None, None, None, None, 2, 4, 64, 0, 512, s) == pa.PA_ERR_INVALID_ARG


def test_slot_mapping_matches_oracle():
    rng = np.random.default_rng(11)
    B, maxb, bs = 5, 9, 16
    tables = rng.integers(0, 1000, size=(B, maxb)).astype(np.int32)
    seq = rng.integers(0, B, size=200).astype(np.int32)
    pos = rng.integers(-3, maxb * bs, size=200).astype(np.int32)
    got = pa.pa_compute_slot_mapping(tables, seq, pos, bs)
    want = oracle.slot_mapping(tables, seq, pos, bs)
    assert np.array_equal(got, want)
    with pytest.raises(pa.PAError):
        pa.pa_compute_slot_mapping(tables, [0], [maxb * bs], bs)


def _compare(bm, model, seqs):
    for s in seqs:
        assert bm.block_table(s) == model.block_table(s)
        assert bm.num_tokens(s) == model.num_tokens(s)
    assert bm.free_list() == model.free
    st = bm.stats()
    for k, v in model.stats().items():
        assert st[k] == v, k
    for b in range(model.num_blocks):
        assert bm.refcount(b) == model.refcount[b]


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_block_manager_matches_model_on_random_ops(seed):
    rng = np.random.default_rng(seed)
    nb, bs = int(rng.integers(8, 40)), int(rng.choice([1, 4, 16]))
    reserve = bool(seed % 2)
    bm = pa.BlockManager(nb, bs, reserve_null_block=reserve)
    model = oracle.BlockManagerModel(nb, bs, reserve_null_block=reserve)
    live = []
    next_id = 100
    for _ in range(400):
        op = rng.choice(["alloc", "append", "append", "append", "fork", "free"])
        if op == "alloc" or not live:
            n = int(rng.integers(0, 3 * bs + 2))
            try:
                model.allocate(next_id, n)
                ok = True
            except oracle.OutOfBlocks:
                ok = False
            if ok:
                bm.allocate(next_id, n)
                live.append(next_id)
            else:
                with pytest.raises(pa.PAError) as e:
                    bm.allocate(next_id, n)
                assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
            next_id += 1
        elif op == "append":
            s = int(rng.choice(live))
            try:
                want = model.append_slot(s)
            except oracle.OutOfBlocks:
                with pytest.raises(pa.PAError) as e:
                    bm.append_slot(s)
                assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
                continue
            assert bm.append_slot(s) == want
        elif op == "fork":
            s = int(rng.choice(live))
            model.fork(s, next_id)
            bm.fork(s, next_id)
            live.append(next_id)
            next_id += 1
        else:
            s = int(rng.choice(live))
            model.free_seq(s)
            bm.free(s)
            live.remove(s)
        _compare(bm, model, live)


def test_block_manager_pages_examples(golden):
    g = golden["incremental_fill"]
    bm = pa.BlockManager(32, 4, free_order=g["free_list"])
    bm.allocate(7, 6)
    assert bm.block_table(7) == g["table_after_prefill"]
    for _ in range(3):
        bm.append_slot(7)
    assert bm.block_table(7) == g["table_after_third_block"]
    bm.free(7)
    assert bm.free_list()[:3] == g["returned_on_finish"]
    c = golden["cow_clone"]
    bm = pa.BlockManager(8, 16, reserve_null_block=False)
    bm.allocate(0, 20)
    bm.fork(0, 1)
    slot, src, dst = bm.append_slot(1)
    assert [src, dst] == c["pair"] and bm.block_table(1) == c["writer_table_after"]
    assert bm.block_table(0) == c["other_table_after"]


def test_block_manager_errors():
    bm = pa.BlockManager(4, 16)
    with pytest.raises(pa.PAError) as e:
        bm.append_slot(5)
    assert e.value.status == pa.PA_ERR_NOT_FOUND
    bm.allocate(1, 16)
    with pytest.raises(pa.PAError) as e:
        bm.allocate(1, 1)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    with pytest.raises(pa.PAError) as e:
        bm.allocate(2, 100)
    assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
    assert bm.stats()["free_blocks"] == 2   # unchanged by the failed call
    with pytest.raises(pa.PAError):
        pa.BlockManager(4, 16, free_order=[1, 1])


def test_wait_timeout_check_rejects_bad_limits_before_launch():
    lib = _lib.load()
    assert lib.pa_check_wait_timeout(0, None) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_check_wait_timeout(2000001, None) == pa.PA_ERR_INVALID_ARG
