"""GPU parity of Step 2 (Dispatch) against the oracle: counts, offsets,
receive counts, send counts, slot rows, row tokens, drops and the permuted
rows, all bit for bit.  Expert choices come from the seeded generator, so
the same input drives both sides."""
import json
import os

import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, run_dispatch

pytestmark = pytest.mark.gpu


def _cfg(T, d, E, k, R, capacity_factor=0.0, capacity=0, dtype="bf16"):
    return moe.make_config(T, d, E, k, R, 0, 0, dtype, "softmax", True, capacity_factor, capacity,
                           "identity")


def _compare(cfg, x, idx, out, check_xp_full=True):
    C = oracle.capacity(cfg.T, cfg.k, cfg.E, cfg.capacity_factor, cfg.capacity)
    ref = oracle.dispatch(idx, cfg.E, cfg.R, C)
    assert out["status"] == 0
    assert torch.equal(out["expert_counts"].cpu(), ref["expert_counts"])
    assert torch.equal(out["expert_offsets"].cpu(), ref["expert_offsets"])
    assert torch.equal(out["rank_counts"].cpu(), ref["rank_counts"])
    if out["rank_splits"] is not None:
        assert torch.equal(out["rank_splits"].cpu(), ref["rank_splits"])
    assert torch.equal(out["slot_row"].cpu(), ref["slot_row"])
    assert int(out["n_dropped"].item()) == ref["n_dropped"]
    rows = ref["rows"]
    assert torch.equal(out["row_token"][:rows].cpu(), ref["row_token"])
    if check_xp_full:
        xp_ref = oracle.permute(x.cpu(), ref["slot_row"], rows)
        assert torch.equal(out["xp"][:rows].cpu().view(torch.int16 if x.dtype == torch.bfloat16
                                                       else torch.int32),
                           xp_ref.view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32))
    else:
        # bytes of every kept row equal its token's row (checked on the device)
        rt = out["row_token"][:rows].long()
        assert torch.equal(out["xp"][:rows], x[rt])
    return ref


@pytest.mark.parametrize("T,d,E,k,R,cf,cap,skew", [
    (1, 64, 4, 2, 2, 0.0, 0, 0.0),
    (31, 64, 8, 2, 4, 0.0, 0, 0.0),
    (32, 128, 8, 2, 4, 0.0, 0, 0.0),
    (33, 128, 8, 2, 4, 0.0, 0, 0.0),
    (1000, 256, 64, 1, 8, 1.25, 0, 1.1),
    (777, 64, 16, 4, 8, 1.0, 0, 1.5),
    (4099, 512, 256, 8, 8, 0.0, 0, 0.0),
    (4099, 512, 256, 8, 8, 1.0, 0, 1.5),
    (5000, 64, 8, 8, 1, 0.0, 0, 0.0),     # k = E: every expert takes every token
    (2048, 64, 32, 3, 32, 0.0, 7, 0.5),   # 32 virtual ranks, explicit capacity
    (257, 64, 3, 1, 3, 0.0, 0, 0.0),      # odd expert count
    (100, 64, 1, 1, 1, 0.0, 0, 0.0),      # a single expert
    (100, 64, 1, 1, 1, 0.0, 10, 0.0),     # a single expert keeping its first 10 tokens
    # few token blocks with long rows: each block's row copies split over column chunks
    (300, 7168, 256, 8, 8, 0.0, 0, 0.5),
    (129, 4096, 8, 2, 8, 0.0, 0, 0.0),
    (200, 2048, 16, 4, 8, 1.0, 0, 1.0),
])
def test_dispatch_matches_oracle(T, d, E, k, R, cf, cap, skew):
    cfg = _cfg(T, d, E, k, R, cf, cap)
    idx = W.random_topk(T, E, k, seed=T + 3 * E + k, skew=skew)
    x = W._grid_int((T, d), -8, 8, 8.0, W._gen(T, "cpu"), "cpu").to(torch.bfloat16).to(DEV)
    out = run_dispatch(cfg, x, idx)
    _compare(cfg, x, idx, out)


def test_dispatch_no_tokens_writes_zero_metadata():
    cfg = _cfg(0, 64, 8, 2, 4)
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device=DEV)
    out = run_dispatch(cfg, x, torch.zeros((0, 2), dtype=torch.int32))
    assert out["status"] == 0
    for key in ("expert_counts", "expert_offsets", "rank_counts", "rank_splits", "n_dropped"):
        assert torch.all(out[key] == 0), key


def test_dispatch_fp32_long_rows_in_column_chunks():
    cfg = _cfg(90, 3072, 8, 2, 4, dtype="f32")
    idx = W.random_topk(90, 8, 2, seed=11, skew=0.7)
    x = W._grid_int((90, 3072), -8, 8, 8.0, W._gen(11, "cpu"), "cpu").to(DEV)
    _compare(cfg, x, idx, run_dispatch(cfg, x, idx))


def test_dispatch_fp32_rows():
    cfg = _cfg(999, 36, 8, 2, 4, dtype="f32")
    idx = W.random_topk(999, 8, 2, seed=1)
    x = torch.randn(999, 36).to(DEV)
    _compare(cfg, x, idx, run_dispatch(cfg, x, idx))


def test_dispatch_capacity_example():
    """ai360xpert capacity example: capacity 100, 150 routed -> the first 100
    (token order) kept, the last 50 dropped."""
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "capacity_example.json")))
    T = g["routed"]
    cfg = _cfg(T, 64, 2, 1, 1, capacity=g["capacity"])
    idx = torch.zeros((T, 1), dtype=torch.int32)
    x = torch.arange(T * 64, dtype=torch.float32).view(T, 64).to(torch.bfloat16).to(DEV)
    out = run_dispatch(cfg, x, idx)
    _compare(cfg, x, idx, out)
    assert int(out["n_dropped"].item()) == g["dropped"]
    sr = out["slot_row"].cpu().flatten()
    assert sr[:100].tolist() == list(range(100)) and (sr[100:] == -1).all()


def test_dispatch_without_rank_splits_and_twice_in_a_row():
    cfg = _cfg(3000, 64, 16, 2, 4, 1.1)
    idx = W.random_topk(3000, 16, 2, seed=5, skew=1.0)
    x = W._grid_int((3000, 64), -8, 8, 8.0, W._gen(2, "cpu"), "cpu").to(torch.bfloat16).to(DEV)
    ws = moe.alloc_workspace(cfg)
    a = run_dispatch(cfg, x, idx, rank_splits=False, ws=ws)
    b = run_dispatch(cfg, x, idx, rank_splits=True, ws=ws)
    _compare(cfg, x, idx, a)
    _compare(cfg, x, idx, b)


def test_dispatch_bad_index_sets_status():
    """An out-of-range expert index is caught by the kernels' own checks: the
    status word reports it and the assignment is treated as dropped."""
    cfg = _cfg(64, 64, 8, 2, 4)
    idx = W.random_topk(64, 8, 2, seed=9)
    idx[5, 1] = 8
    idx[7, 0] = -3
    x = torch.zeros((64, 64), dtype=torch.bfloat16, device=DEV)
    out = run_dispatch(cfg, x, idx)
    assert out["status"] & moe.MOE_DEV_BAD_INDEX
    assert int(out["slot_row"][5, 1]) == -1 and int(out["slot_row"][7, 0]) == -1


@pytest.mark.parametrize("T,s", [(131072, 1.5), (65536, 0.0)])
def test_dispatch_sweep_full_size(T, s):
    """The largest sweep points: T*k up to 1M assignments, E=256, d=7168."""
    E, k, R, d = 256, 8, 8, 7168
    cfg = _cfg(T, d, E, k, R, 1.25 if s > 0 else 0.0)
    idx = W.random_topk(T, E, k, seed=T, skew=s)
    x = W._grid_int((T, d), -8, 8, 8.0, W._gen(1, DEV), DEV).to(torch.bfloat16)
    out = run_dispatch(cfg, x, idx)
    _compare(cfg, x, idx, out, check_xp_full=False)


def test_dispatch_deterministic():
    cfg = _cfg(20000, 128, 64, 4, 8, 1.2)
    idx = W.random_topk(20000, 64, 4, seed=3, skew=1.2)
    x = W._grid_int((20000, 128), -8, 8, 8.0, W._gen(4, DEV), DEV).to(torch.bfloat16)
    a = run_dispatch(cfg, x, idx)
    b = run_dispatch(cfg, x, idx)
    for key in ["slot_row", "row_token", "expert_offsets", "xp", "rank_splits"]:
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("T,E,k", [(3000, 16, 2), (4099, 256, 8)])
def test_dispatch_launch_count(T, E, k):
    """One moe_dispatch call enqueues three kernels (count, scan, place), as the
    library's own launch counter reports."""
    cfg = _cfg(T, 256, E, k, 8)
    idx = W.random_topk(T, E, k, seed=T + E, skew=0.8)
    x = W._grid_int((T, 256), -8, 8, 8.0, W._gen(T, "cpu"), "cpu").to(torch.bfloat16).to(DEV)
    n0 = moe.moe_launch_count()
    out = run_dispatch(cfg, x, idx)
    assert moe.moe_launch_count() - n0 == 3
    _compare(cfg, x, idx, out)
