"""pa_decode_plan: the host-side description of how pa_decode runs a problem
(kernel, context split, merge, launches) agrees with what the workspace
query reports and with the kernels' constraints."""
import pytest

import paged_kv_cache_121_gb300 as pa

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, Hq, Hkv, D, block_size, max_context_len
    (16, 32, 8, 128, 16, 4164),     # Qwen3-8B layer
    (4, 64, 8, 128, 16, 32768),     # long context
    (64, 32, 8, 128, 16, 4096),     # GQA batch
    (16, 32, 8, 128, 8, 4164),
    (16, 32, 8, 128, 128, 4164),
    (3, 8, 2, 64, 4, 500),          # blocks of 4: tensor cores, rows copied by cp.async
    (16, 32, 8, 128, 1, 4164),      # blocks of 1
    (3, 8, 2, 64, 12, 500),         # block size not a power of two: CUDA-core kernel
    (1, 8, 8, 128, 16, 1),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("with_ws", [True, False])
def test_plan_is_consistent(shape, with_ws):
    B, hq, hkv, d, bs, mcl = shape
    p = pa.pa_decode_plan(B, hq, hkv, d, bs, mcl, pa.PA_BF16, with_workspace=with_ws)
    assert p["tensor_cores"] == (1 if bs & (bs - 1) == 0 else 0)
    assert hkv % p["heads_per_cta"] == 0
    assert p["num_splits"] >= 1
    if p["balanced"]:
        # equal tile ranges cut on the device: decode + merge through the workspace
        assert with_ws and p["tensor_cores"] and bs >= 16 and not p["cluster_merge"]
        assert p["partition_tokens"] == 0 and p["kernel_launches"] == 2
        assert 0 < p["workspace_bytes"] <= pa.pa_decode_workspace_size(B, hq, hkv, d, bs, mcl)
        return
    # the partitions cover the context, and none is empty by construction
    assert p["num_splits"] * p["partition_tokens"] >= mcl
    assert (p["num_splits"] - 1) * p["partition_tokens"] < max(mcl, 1) or p["cluster_merge"]
    if p["tensor_cores"]:
        assert p["partition_tokens"] % 16 == 0          # whole 16-token tiles
    else:
        assert p["partition_tokens"] % bs == 0          # whole blocks
    if p["cluster_merge"]:
        assert 2 <= p["num_splits"] <= 8
        assert p["kernel_launches"] == 1 and p["workspace_bytes"] == 0
    elif p["num_splits"] > 1:
        assert with_ws
        assert p["kernel_launches"] == 2
        assert 0 < p["workspace_bytes"] <= pa.pa_decode_workspace_size(B, hq, hkv, d, bs, mcl)
    else:
        assert p["kernel_launches"] == 1 and p["workspace_bytes"] == 0


def test_plan_headline_shapes():
    """The Qwen3 layer is split within a cluster (one launch, no workspace);
    the long context needs the workspace and the merge kernel."""
    q = pa.pa_decode_plan(16, 32, 8, 128, 16, 4164)
    assert q["tensor_cores"] == 1 and q["cluster_merge"] == 1 and q["kernel_launches"] == 1
    lc = pa.pa_decode_plan(4, 64, 8, 128, 16, 32768)
    assert lc["kernel_launches"] == 2 and lc["num_splits"] > 8
    lc0 = pa.pa_decode_plan(4, 64, 8, 128, 16, 32768, with_workspace=False)
    assert lc0["cluster_merge"] == 1 and lc0["num_splits"] == 8


def test_plan_refuses_bad_shapes():
    with pytest.raises(pa.PAError):
        pa.pa_decode_plan(4, 30, 8, 128, 16, 100)      # Hq % Hkv != 0
    with pytest.raises(pa.PAError):
        pa.pa_decode_plan(4, 32, 8, 96, 16, 100)       # head_dim 96
