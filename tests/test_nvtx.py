"""Every C-ABI call opens an NVTX range named after it and closes it, even
when it returns an argument error before launching anything.  Checked
without a GPU through a small NVTX injection library (tests/native) that
records the ranges: calls that fail their argument checks touch no device."""
import ctypes
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "native", "nvtx_recorder.c")

CHILD = r'''
import ctypes, sys
sys.path.insert(0, sys.argv[1])
import expert_dispatch_top_b300 as moe
rec = ctypes.CDLL(sys.argv[2])
rec.recorded_names.restype = ctypes.c_char_p
lib = moe.library()
cfg = moe.make_config(64, 128, 8, 2, 4, 64, dtype="bf16", act="swiglu")
st = [lib.moe_route(ctypes.byref(cfg), None, None, None, None, None, None, None, None),
      lib.moe_dispatch(ctypes.byref(cfg), *([None] * 12)),
      lib.moe_combine(ctypes.byref(cfg), *([None] * 7)),
      lib.moe_expert_ffn(ctypes.byref(cfg), *([None] * 13)),
      lib.moe_layer_forward(ctypes.byref(cfg), *([None] * 8), None, None, None, None),
      lib.moe_dispatch_noalloc(ctypes.byref(cfg), *([None] * 12))]
print(",".join(str(s) for s in st))
print(rec.recorded_names().decode().strip().replace("\n", ","))
print(rec.recorded_pops(), rec.recorded_depth())
'''


def test_each_call_opens_and_closes_its_nvtx_range(tmp_path):
    so = str(tmp_path / "libnvtx_recorder.so")
    subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", "-I", "/usr/local/cuda/include", SRC,
                           "-o", so])
    env = dict(os.environ, NVTX_INJECTION64_PATH=so)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, so], capture_output=True, text=True,
                       env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    status, names, counts = r.stdout.strip().splitlines()[-3:]
    assert set(status.split(",")) == {"1"}          # every call: MOE_ERR_INVALID_ARG
    assert names.split(",") == ["moe_route", "moe_dispatch", "moe_combine", "moe_expert_ffn",
                                "moe_layer_forward", "moe_dispatch_noalloc"]
    assert counts.split() == ["6", "0"]              # six pops, nothing left open
