"""C-ABI checks that need no GPU: the library loads, exports every function
include/moe.h declares, and its host-side logic (validation, capacity,
workspace sizing, status strings) behaves as documented.  No compute call is
made here."""
import ctypes
import math
import os
import re
import subprocess

import pytest

import expert_dispatch_top_b300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z_]+)\s*\(", src,
                       flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ["moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_layer_forward",
              "moe_workspace_size", "moe_status_string", "moe_read_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = moe.library()
    for n in _declared_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T (moe_[a-z_]+)$", out, flags=re.M))
    assert set(_declared_functions()) <= exported


def test_status_strings():
    for s in range(7):
        assert moe.status_string(s).startswith("MOE_")
    assert "unknown" in moe.status_string(99)


def _cfg(**kw):
    base = dict(T=4096, d=512, E=8, k=2, R=4, d_ff=1024, dtype="f32", score="softmax",
                act="gelu")
    base.update(kw)
    return moe.make_config(**base)


def test_struct_layout_matches_header():
    assert ctypes.sizeof(moe.moe_config) == 15 * 4
    assert ctypes.sizeof(moe.moe_buffers) == 14 * 8


@pytest.mark.parametrize("kw,status", [
    (dict(), moe.MOE_OK),
    (dict(k=0), moe.MOE_ERR_INVALID_ARG),
    (dict(k=9, E=16, R=4), moe.MOE_ERR_INVALID_ARG),
    (dict(k=5, E=4, R=4), moe.MOE_ERR_INVALID_ARG),
    (dict(E=257, R=1), moe.MOE_ERR_INVALID_ARG),
    (dict(E=12, R=8), moe.MOE_ERR_INVALID_ARG),
    (dict(R=64, E=256), moe.MOE_ERR_INVALID_ARG),
    (dict(d=6), moe.MOE_ERR_INVALID_ARG),                 # fp32 row not 16-byte multiple
    (dict(d=520, dtype="bf16"), moe.MOE_ERR_UNSUPPORTED),  # tensor-core path wants d % 64
    (dict(d=516), moe.MOE_OK),                             # fp32 path takes d % 4
    (dict(d_ff=0), moe.MOE_ERR_INVALID_ARG),
    (dict(d_ff=0, act="identity"), moe.MOE_OK),
    (dict(n_shared=1, act="identity", d_ff=0), moe.MOE_ERR_INVALID_ARG),
    (dict(n_shared=2), moe.MOE_ERR_INVALID_ARG),
    (dict(T=0), moe.MOE_OK),
    (dict(T=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(T=1 << 28, k=4, E=8), moe.MOE_ERR_INVALID_ARG),  # T*k >= 2^30
    (dict(capacity=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(max_ranks=2), moe.MOE_OK),
    (dict(max_ranks=5), moe.MOE_ERR_INVALID_ARG),                    # more than R
    (dict(max_ranks=1, k=3), moe.MOE_ERR_INVALID_ARG),               # 1 rank x 2 experts < k
])
def test_check_config(kw, status):
    assert moe.moe_check_config(_cfg(**kw)) == status


def test_capacity_and_max_rows():
    # explicit capacity, factor, none
    assert moe.moe_capacity(_cfg(capacity=100)) == 100
    assert moe.moe_capacity(_cfg(capacity_factor=1.25)) == math.ceil(1.25 * 4096 * 2 / 8)
    assert moe.moe_capacity(_cfg()) == -1
    assert moe.moe_max_rows(_cfg()) == 4096 * 2
    assert moe.moe_max_rows(_cfg(capacity=100)) == 8 * 100
    assert moe.moe_max_rows(_cfg(capacity=5000)) == 4096 * 2
    sw = moe.make_config(32768, 1024, 64, 1, 8, 4096, dtype="bf16", act="gelu",
                         capacity_factor=1.25, renorm=False)
    assert moe.moe_capacity(sw) == 640
    assert moe.moe_max_rows(sw) == min(32768, 64 * 640)
    tight = moe.make_config(32768, 1024, 64, 1, 8, 4096, dtype="bf16", act="gelu", capacity=300)
    assert moe.moe_max_rows(tight) == 64 * 300


def test_workspace_size():
    c = _cfg()
    n = moe.moe_workspace_size(c)
    assert n > 0 and n % 256 == 0
    # metadata arrays of the whole-layer call fit inside
    assert n >= 3 * 4096 * 2 * 4 + 4096 * 2 * 4
    assert moe.moe_workspace_size(_cfg(k=0)) == 0
    big = moe.make_config(131072, 7168, 256, 8, 8, 0, act="identity", score="sigmoid")
    assert moe.moe_workspace_size(big) > 131072 // 32 * 256 * 8


def test_workspace_holds_the_tf32_split_of_fp32_experts():
    """fp32 experts whose d and d_ff are multiples of 16 run on the tensor cores
    from tf32 high / low parts kept in the workspace: 2 x 4 bytes per element of
    the expert rows and of both weight stacks, 4 bytes per element of h (the
    high part of h lives in the caller's h); other shapes, bf16 and identity
    experts keep none."""
    T, d, E, k, f = 4096, 512, 8, 2, 1024
    split = 2 * 4 * (T * k * d + E * f * d + E * d * f) + 4 * T * k * f
    base = moe.moe_workspace_size(_cfg(d_ff=1028))  # FFMA shape: no split sections
    n = moe.moe_workspace_size(_cfg())
    assert n - base >= split and n - base < split + 8 * 256
    swiglu = moe.moe_workspace_size(_cfg(act="swiglu")) - moe.moe_workspace_size(_cfg(act="swiglu", d_ff=1028))
    assert swiglu >= split + 2 * 4 * E * f * d  # the gate rows double W_up
    for kw in (dict(dtype="bf16"), dict(act="identity", d_ff=0)):
        assert moe.moe_workspace_size(_cfg(**kw)) < split


def test_invalid_calls_fail_before_any_launch():
    """Argument errors come back synchronously, with no GPU touched."""
    c = _cfg()
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route(c, None, None, None, None, None, None, None, stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route(_cfg(k=0), None, None, None, None, None, None, None, stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    # misaligned pointer
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route(c, 0x1008 + 4, 0x2000, None, None, 0x3000, 0x4000, None, stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    # selection-only bias needs sigmoid scores
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route(c, 0x1000, 0x2000, None, 0x5000, 0x3000, 0x4000, 0x6000, stream=0)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    # the route needs a workspace (its status word)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route(c, 0x1000, 0x2000, None, None, 0x3000, 0x4000, None, stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as e:
        moe.moe_dispatch(c, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, None, 0x7000, 0x8000, None,
                         0x9000, 0xa000, stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as e:
        moe.moe_combine(_cfg(add_residual=True), 0x1000, 0x2000, 0x3000, None, None, 0x4000,
                        stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_forward(c, 0x1000, 0x2000, None, None, 0x3000, 0x4000, None, None,
                              moe.moe_buffers(), 0x5000, 0x6000, stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoeError) as e:
        moe.moe_read_device_status(None, stream=0)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG


def test_empty_batch_is_a_noop():
    c = _cfg(T=0)
    moe.moe_route(c, None, None, None, None, None, None, None, stream=0)
    moe.moe_combine(c, None, None, None, None, None, None, stream=0)


def test_backward_scratch_size():
    bf = _cfg(dtype="bf16", act="swiglu", d=512, d_ff=1024)
    full = moe.moe_expert_ffn_backward_scratch_size(bf, True)
    dgrad = moe.moe_expert_ffn_backward_scratch_size(bf, False)
    assert full > dgrad > 0 and full % 256 == 0 and dgrad % 256 == 0
    assert moe.moe_expert_ffn_backward_scratch_size(_cfg(k=0), True) == 0
    assert moe.moe_expert_ffn_backward_scratch_size(_cfg(act="identity", d_ff=0), True) == 0
    # more tokens, more scratch
    assert moe.moe_expert_ffn_backward_scratch_size(_cfg(dtype="bf16", act="swiglu", T=8192), True) \
        > moe.moe_expert_ffn_backward_scratch_size(_cfg(dtype="bf16", act="swiglu", T=4096), True)


def test_backward_and_hooks_reject_bad_arguments_before_any_launch():
    lib = moe.library()
    c = _cfg(dtype="bf16", act="swiglu")
    need = moe.moe_expert_ffn_backward_scratch_size(c, True)

    def ffn_bwd(cfg, scratch, nbytes, d_w_up=0x7000, ws=0x9000):
        return lib.moe_expert_ffn_backward(ctypes.byref(cfg), 0x1000, 0x2000, 0x3000, 0x4000,
                                           0x5000, 0x6000, d_w_up, 0x8000, scratch,
                                           ctypes.c_size_t(nbytes), ws, None)
    assert ffn_bwd(c, 0x10000, need - 256) == moe.MOE_ERR_INVALID_ARG      # scratch too small
    assert ffn_bwd(c, 0x10000 + 16, need) == moe.MOE_ERR_INVALID_ARG       # not 256-byte aligned
    assert ffn_bwd(c, 0x10000, need, ws=None) == moe.MOE_ERR_INVALID_ARG   # no status word
    assert ffn_bwd(c, 0x10000, need, d_w_up=0x7004) == moe.MOE_ERR_INVALID_ARG  # misaligned dW
    ident = _cfg(act="identity", d_ff=0)
    assert ffn_bwd(ident, 0, 0) == moe.MOE_ERR_INVALID_ARG   # identity experts have no weights
    # failure-detection hook: K block in range, bounded limit, bf16 experts only
    for kb, us in ((-1, 1000), (512 // 64, 1000), (0, 0), (0, 4000001)):
        assert lib.moe_test_expert_ffn_stall(ctypes.byref(c), 0x1000, 0x2000, 0x3000, 0x4000, kb,
                                             us, 0x9000, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_test_expert_ffn_stall(ctypes.byref(_cfg()), 0x1000, 0x2000, 0x3000, 0x4000, 0,
                                         1000, 0x9000, None) == moe.MOE_ERR_UNSUPPORTED
    # balancing step: the step size must be finite and non-negative
    for gamma in (-1e-3, float("inf"), float("nan")):
        assert lib.moe_update_sel_bias(ctypes.byref(c), 0x1000, 0x2000, ctypes.c_float(gamma),
                                       None) == moe.MOE_ERR_INVALID_ARG


def test_noalloc_dispatch_rejects_shapes_beyond_its_array():
    lib = moe.library()
    big = moe.make_config(131072, 7168, 256, 8, 8, 0, act="identity", score="sigmoid")
    st = lib.moe_dispatch_noalloc(ctypes.byref(big), 0x1000, 0x2000, 0x3000, 0x4000, 0x5000,
                                  0x6000, 0x7000, 0x8000, 0x9000, 0xa000, None, None)
    assert st == moe.MOE_ERR_INVALID_ARG


def _layer_args(cfg, **over):
    """Aligned stand-in device addresses for every moe_layer_forward argument
    (never dereferenced: each case below must fail its checks first)."""
    a = dict(x=0x10000, w_router=0x20000, logit_bias=None, sel_bias=None, w_up=0x30000,
             w_down=0x40000, shared_up=None, shared_down=None, y=0x50000, ws=0x60000)
    b = dict(xp=0x70000, h=0x80000, yp=0x90000, shared_h=None, shared_out=None)
    if cfg.n_shared:
        a.update(shared_up=0xa0000, shared_down=0xb0000)
        b.update(shared_h=0xc0000, shared_out=0xd0000)
    for key, v in over.items():
        (a if key in a else b)[key] = v
    buf = moe.moe_buffers(**b)
    lib = moe.library()
    return lib.moe_layer_forward(ctypes.byref(cfg), a["x"], a["w_router"], a["logit_bias"],
                                 a["sel_bias"], a["w_up"], a["w_down"], a["shared_up"],
                                 a["shared_down"], ctypes.byref(buf), a["y"], a["ws"], None)


@pytest.mark.parametrize("dtype,act,n_shared", [("bf16", "swiglu", 1), ("bf16", "gelu", 0),
                                                ("f32", "gelu", 0)])
def test_layer_forward_rejects_every_argument_error_before_any_launch(dtype, act, n_shared):
    """moe_layer_forward checks the arguments of all four steps before its
    first launch.  On this GPU-less host a launch that went out would fail as
    MOE_ERR_CUDA; each bad argument must instead come back as
    MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED."""
    import torch
    c = _cfg(dtype=dtype, act=act, n_shared=n_shared, score="sigmoid" if n_shared else "softmax")
    bad = [dict(w_up=None), dict(w_down=None), dict(w_up=0x30008), dict(yp=0x90008),
           dict(h=0x80004), dict(y=0x50008), dict(xp=None), dict(ws=0x60008),
           dict(w_router=None), dict(logit_bias=0x1002)]
    if n_shared:
        bad += [dict(shared_up=None), dict(shared_out=0xd0008), dict(shared_h=None)]
    launches = moe.moe_launch_count()
    for over in bad:
        assert _layer_args(c, **over) == moe.MOE_ERR_INVALID_ARG, over
    # the library's own launch counter agrees: nothing was enqueued
    assert moe.moe_launch_count() == launches
    # a selection-only bias with softmax scores is a valid call this library does not run
    if not n_shared:
        assert _layer_args(c, sel_bias=0x1000) == moe.MOE_ERR_UNSUPPORTED
    # bf16 expert GEMMs take d and d_ff in multiples of 64
    if dtype == "bf16":
        assert _layer_args(_cfg(dtype=dtype, act=act, d=72)) == moe.MOE_ERR_UNSUPPORTED
        assert _layer_args(_cfg(dtype=dtype, act=act, d_ff=1000)) == moe.MOE_ERR_UNSUPPORTED
    if not torch.cuda.is_available():
        # control: with every argument valid the call gets as far as a launch,
        # which fails here for want of a device
        assert _layer_args(c) == moe.MOE_ERR_CUDA


def test_release_and_checked_builds_say_which_they_are():
    assert moe.library().moe_build_checked() == 0
    child = ("import sys; sys.path.insert(0, sys.argv[1]); import expert_dispatch_top_b300 as m; "
             "print(m.LIB_PATH); print(m.moe_build_checked())")
    r = subprocess.run(["python", "-c", child, ROOT], capture_output=True, text=True,
                       env=dict(os.environ, MOE_B300_CHECKED="1"), timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    path, flag = r.stdout.strip().splitlines()[-2:]
    assert path.endswith("libmoe_b300_checked.so") and flag == "True"


def test_route_backward_rejects_bad_arguments_before_any_launch():
    lib = moe.library()
    c = _cfg(dtype="bf16", act="swiglu")

    def call(x=0x1000, w=0x2000, lb=None, idx=0x3000, dg=0x4000, dl=0x5000, dx=0x6000, dw=0x7000,
             dlb=None):
        return lib.moe_route_backward(ctypes.byref(c), x, w, lb, idx, dg, dl, dx, dw, dlb, None)
    assert call(dl=None) == moe.MOE_ERR_INVALID_ARG          # d_logits is required
    assert call(x=None) == moe.MOE_ERR_INVALID_ARG
    assert call(dx=0x6008) == moe.MOE_ERR_INVALID_ARG        # misaligned dx
    assert call(idx=0x3002) == moe.MOE_ERR_INVALID_ARG       # misaligned topk_idx
    assert lib.moe_route_backward(ctypes.byref(_cfg(k=0)), 0x1000, 0x2000, None, 0x3000, 0x4000,
                                  0x5000, None, None, None, None) == moe.MOE_ERR_INVALID_ARG


def test_layer_forward_host_checks_before_its_first_copy():
    """moe_layer_forward_host runs the layer's argument checks before it
    enqueues the input copy: on this GPU-less host a copy that went out would
    fail as MOE_ERR_CUDA, an argument error comes back as MOE_ERR_INVALID_ARG."""
    import torch
    lib = moe.library()
    c = _cfg(dtype="bf16", act="swiglu")
    host = (ctypes.c_uint8 * 64)()
    buf = moe.moe_buffers(xp=0x70000, h=0x80000, yp=0x90000)

    def call(x_host=ctypes.addressof(host), y_host=ctypes.addressof(host), w_up=0x30000,
             x_dev=0x10000, y_dev=0x50000):
        return lib.moe_layer_forward_host(ctypes.byref(c), x_host, x_dev, 0x20000, None, None,
                                          w_up, 0x40000, None, None, ctypes.byref(buf), y_dev,
                                          y_host, 0x60000, None)
    assert call(y_host=None) == moe.MOE_ERR_INVALID_ARG
    assert call(x_dev=None) == moe.MOE_ERR_INVALID_ARG
    assert call(w_up=None) == moe.MOE_ERR_INVALID_ARG          # a layer argument
    assert call(y_dev=0x50008) == moe.MOE_ERR_INVALID_ARG       # misaligned staging y
    if not torch.cuda.is_available():
        assert call() == moe.MOE_ERR_CUDA                        # valid: gets as far as the copy
