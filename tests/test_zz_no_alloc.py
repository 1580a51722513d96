"""The layer entry point that needs no workspace from the caller.

Callers such as a serving engine that owns all of HBM, or a plugin interface
with no allocator, cannot hand the library scratch memory; for them
moe_lora_layer_noalloc keeps its intermediates in a library-held device array.
This file is collected last so that a failure here cannot stop the rest of the
GPU suite from running first. It calls the entry point through the C ABI and
checks it against moe_lora_layer on two calls in a row (different shapes, so a
stale array from the first call cannot hide in the second).
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from workloads import make_workload_inputs, make_layer_inputs

from gpu_util import LAYER_RTOL, assert_close, dev, need_gpu

pytestmark = pytest.mark.gpu

_P, _I = ctypes.c_void_p, ctypes.c_int


def _noalloc_fn(lib):
    fn = lib.moe_lora_layer_noalloc
    fn.restype = _I
    fn.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _I, _P,
                   _I, _P, _P]
    return fn


def _p(t):
    return None if t is None else t.data_ptr()


def test_noalloc_matches_layer_on_two_calls():
    m = need_gpu()
    fn = _noalloc_fn(m.lib())
    stream = torch.cuda.current_stream().cuda_stream
    cases = [make_workload_inputs("tiny"),
             make_layer_inputs(T=37, H=192, I=160, E=6, k=3, L=3, r=16, seed=5, lora_std=None)]
    for inp in cases:
        x, W1, W2 = dev(inp.x), dev(inp.W1), dev(inp.W2)
        lg, ta = dev(inp.logits), dev(inp.token_adapter)
        A1, B1, A2, B2 = dev(inp.A1), dev(inp.B1), dev(inp.A2), dev(inp.B2)
        y_ref = m.moe_lora_layer(x, W1, W2, logits=lg, k=inp.k, token_adapter=ta, A1=A1, B1=B1,
                                 A2=A2, B2=B2, y_fp32=True)
        y = torch.full((inp.T, inp.H), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.full((1,), 0xFF, dtype=torch.int32, device="cuda")
        st = fn(_p(x), _p(lg), None, None, _p(ta), inp.T, inp.H, inp.I, inp.E, inp.k, _p(W1),
                _p(W2), _p(A1), _p(B1), _p(A2), _p(B2), inp.L, inp.r, _p(y), 1, _p(err), stream)
        assert st == 0, m.status_string(st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(y.cpu(), y_ref.cpu().double().numpy(), LAYER_RTOL, f"noalloc T={inp.T}")
        # and against the oracle itself
        ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
        ref = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter, inp.A1,
                                    inp.B1, inp.A2, inp.B2)
        assert_close(y.cpu(), ref, LAYER_RTOL, f"noalloc vs oracle T={inp.T}")


def test_noalloc_reports_device_errors_per_call():
    """err_out receives the call's device error word: a caller-routed expert id out of
    range sets the expert bit (the slot is dropped, not trapped on); the next clean call
    clears it, because each call starts from a clear word in the shared array."""
    m = need_gpu()
    fn = _noalloc_fn(m.lib())
    stream = torch.cuda.current_stream().cuda_stream
    inp = make_layer_inputs(T=12, H=128, I=64, E=4, k=2, L=2, r=8, seed=7, lora_std=None)
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    bad = ids.copy()
    bad[5, 1] = inp.E  # out of range
    x, W1, W2, ta = dev(inp.x), dev(inp.W1), dev(inp.W2), dev(inp.token_adapter)
    A1, B1, A2, B2 = dev(inp.A1), dev(inp.B1), dev(inp.A2), dev(inp.B2)
    w_d = dev(torch.as_tensor(w, dtype=torch.float32))
    y = torch.empty((inp.T, inp.H), dtype=torch.float32, device="cuda")
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    for ids_in, expect in ((bad, 0x1), (ids, 0), (bad, 0x1), (ids, 0)):
        ids_d = dev(torch.as_tensor(ids_in, dtype=torch.int32))
        err.fill_(0x7F)
        st = fn(_p(x), None, _p(ids_d), _p(w_d), _p(ta), inp.T, inp.H, inp.I, inp.E, inp.k,
                _p(W1), _p(W2), _p(A1), _p(B1), _p(A2), _p(B2), inp.L, inp.r, _p(y), 1,
                _p(err), stream)
        assert st == 0, m.status_string(st)
        torch.cuda.synchronize()
        assert int(err.item()) == expect
    ref = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter, inp.A1,
                                inp.B1, inp.A2, inp.B2)
    assert_close(y.cpu(), ref, LAYER_RTOL, "noalloc after a flagged call")


def test_noalloc_after_device_reset_in_fresh_process():
    """A caller may destroy and re-create its CUDA context (cudaDeviceReset); the array's
    device address changes with the context and the entry point must look it up again.
    Run in a child process (torch's device state would not survive the reset): two
    rounds of moe_lora_layer_noalloc against moe_lora_layer, a reset in between."""
    m = need_gpu()
    child = os.path.join(os.path.dirname(os.path.abspath(__file__)), "noalloc_reset_child.py")
    p = subprocess.run([sys.executable, child, m.LIB_PATH], capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0 and p.stdout.strip().endswith("ok"), p.stdout + p.stderr


def test_noalloc_rejects_shapes_beyond_its_array():
    m = need_gpu()
    fn = _noalloc_fn(m.lib())
    big = 0x100000  # aligned stand-in pointers: the call must reject the shape before use
    st = fn(big, big, None, None, big, 4096, 2880, 2880, 32, 4, big, big, big, big, big, big,
            16, 16, big, 0, None, torch.cuda.current_stream().cuda_stream)
    assert st == 4  # MOE_LORA_ERR_WORKSPACE_TOO_SMALL
