"""moe_dispatch_noalloc: the dispatch step for callers that cannot allocate
device memory (for example a plugin that is handed only its input and output
pointers, or a serving loop whose memory another allocator reserved at
start-up).  It keeps its scratch state in a fixed array inside the library
instead of a caller workspace.  These checks call it through the C ABI and
compare every output with moe_dispatch's on the same inputs, twice in a row
(the second call finds the first call's leftovers in the shared array), then
with a different shape.  The file name makes pytest collect it last."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
KEYS = ["xp", "row_token", "slot_row", "expert_counts", "expert_offsets", "rank_counts",
        "rank_splits", "n_dropped"]


def _outputs(cfg, dtype):
    rows = max(moe.moe_max_rows(cfg), 1)
    i32 = dict(dtype=torch.int32, device=DEV)
    return dict(xp=torch.zeros((rows, cfg.d), dtype=dtype, device=DEV),
                row_token=torch.full((rows,), -5, **i32),
                slot_row=torch.full((cfg.T, cfg.k), -9, **i32),
                expert_counts=torch.full((cfg.E,), -1, **i32),
                expert_offsets=torch.full((cfg.E + 1,), -1, **i32),
                rank_counts=torch.full((cfg.R,), -1, **i32),
                rank_splits=torch.full((cfg.R, cfg.R), -1, **i32),
                n_dropped=torch.full((1,), -1, **i32))


def _with_workspace(cfg, x, idx):
    o = _outputs(cfg, x.dtype)
    ws = moe.alloc_workspace(cfg)
    moe.moe_dispatch(cfg, x, idx, o["xp"], o["row_token"], o["slot_row"], o["expert_counts"],
                     o["expert_offsets"], o["rank_counts"], o["rank_splits"], o["n_dropped"], ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    return o


def _without_workspace(cfg, x, idx, with_status=True):
    o = _outputs(cfg, x.dtype)
    status = torch.zeros(1, dtype=torch.int32, device=DEV) if with_status else None
    moe.moe_dispatch_noalloc(cfg, x, idx, o["xp"], o["row_token"], o["slot_row"],
                             o["expert_counts"], o["expert_offsets"], o["rank_counts"],
                             o["rank_splits"], o["n_dropped"], status)
    torch.cuda.synchronize()
    if with_status:
        assert int(status.item()) == 0
    return o


def _case(T, d, E, k, R, cf, seed):
    cfg = moe.make_config(T, d, E, k, R, 0, 0, "bf16", "softmax", True, cf, 0, "identity")
    idx = W.random_topk(T, E, k, seed=seed, skew=1.2).to(DEV)
    x = W._grid_int((T, d), -8, 8, 8.0, W._gen(seed, DEV), DEV).to(torch.bfloat16)
    return cfg, x, idx


def test_noalloc_dispatch_matches_dispatch_two_calls_in_a_row():
    cfg, x, idx = _case(5000, 256, 64, 4, 8, 1.1, seed=21)
    ref = _with_workspace(cfg, x, idx)
    assert int(ref["n_dropped"].item()) > 0
    for _ in range(2):
        got = _without_workspace(cfg, x, idx)
        rows = int(ref["expert_offsets"][-1].item())
        for key in KEYS:
            a, b = got[key], ref[key]
            if key in ("xp", "row_token"):
                a, b = a[:rows], b[:rows]
            assert torch.equal(a, b), key
    # a different shape after the first one: nothing carries over
    cfg2, x2, idx2 = _case(777, 128, 16, 2, 4, 0.0, seed=5)
    ref2 = _with_workspace(cfg2, x2, idx2)
    got2 = _without_workspace(cfg2, x2, idx2)
    for key in KEYS:
        assert torch.equal(got2[key], ref2[key]), key


def test_noalloc_dispatch_without_a_status_word():
    """device_status may be NULL: the kernels then keep their status bits in
    the library's own array, and the outputs are unchanged."""
    cfg, x, idx = _case(3000, 192, 32, 2, 4, 1.25, seed=9)
    ref = _with_workspace(cfg, x, idx)
    for _ in range(2):
        got = _without_workspace(cfg, x, idx, with_status=False)
        rows = int(ref["expert_offsets"][-1].item())
        for key in KEYS:
            a, b = got[key], ref[key]
            if key in ("xp", "row_token"):
                a, b = a[:rows], b[:rows]
            assert torch.equal(a, b), key


def test_noalloc_dispatch_rejects_shapes_beyond_its_scratch():
    cfg = moe.make_config(131072, 64, 256, 8, 8, 0, 0, "bf16", "softmax", True, 0.0, 0,
                          "identity")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_dispatch_noalloc(cfg, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000,
                                 0x8000, None, 0x9000)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
