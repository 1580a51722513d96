"""Failure detection on the GPU without a fault: a bounded device wait that runs out.

Every mbarrier wait in the grouped GEMMs (and in the short-K shrink) gives up after a
wall-time limit, records MOE_LORA_DEVERR_TIMEOUT in the sticky error word, drains its
CTA's copies and tensor-core work, frees its tensor memory and exits; a CTA pair (the
fused GEMM at 256-row token tiles) also mirrors the abort into the other CTA and meets
it at cluster barriers before either frees anything. The test makes the
main waits give up at their first unsuccessful poll (wait_limit_ns < 0), reads the
status through moe_lora_get_error, then clears the word and checks that the next normal
call on the same workspace matches the oracle: the context stays usable.
"""
import ctypes

import pytest
import torch

import oracle
from workloads import make_layer_inputs

from gpu_util import LAYER_RTOL, assert_close, dev, need_gpu

pytestmark = pytest.mark.gpu

ERR_TIMEOUT = 5
DEVERR_TIMEOUT = 0x4


@pytest.mark.parametrize("expand_mode", [0, 1])
@pytest.mark.parametrize("shape", ["small", "many_adapters", "cta_pairs"])
def test_bounded_waits_give_up_and_recover(expand_mode, shape):
    m = need_gpu()
    if shape == "small":
        kw = dict(T=16, H=256, I=128, E=4, k=2, L=2, r=16)
    elif shape == "many_adapters":  # many short LoRA blocks and K <= 832: the down shrink
        kw = dict(T=256, H=256, I=128, E=64, k=8, L=32, r=32, adapters="zipf1.1")  # stages A
    else:  # 256-row token tiles: the fused chain's GEMMs run on CTA pairs (cluster barriers,
        kw = dict(T=800, H=256, I=128, E=3, k=2, L=2, r=16)  # copies on the leader's barriers)
    inp = make_layer_inputs(seed=41, lora_std=None, **kw)
    lora = dict(A1=dev(inp.A1), B1=dev(inp.B1), A2=dev(inp.A2), B2=dev(inp.B2))
    args = (dev(inp.x), dev(inp.W1), dev(inp.W2))
    ws = m.new_workspace(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r)
    lg, ta = dev(inp.logits), dev(inp.token_adapter)
    m.moe_lora_layer(*args, logits=lg, k=inp.k, token_adapter=ta, y_fp32=True, workspace=ws,
                     expand_mode=expand_mode, wait_limit_ns=-1, **lora)
    torch.cuda.synchronize()
    word = ctypes.c_uint32(0)
    st = m.lib().moe_lora_get_error(ws.data_ptr(), torch.cuda.current_stream().cuda_stream,
                                    ctypes.byref(word))
    assert st == ERR_TIMEOUT and word.value & DEVERR_TIMEOUT, (st, word.value)
    m.clear_error(ws)
    y = m.moe_lora_layer(*args, logits=lg, k=inp.k, token_adapter=ta, y_fp32=True, workspace=ws,
                         expand_mode=expand_mode, **lora)
    torch.cuda.synchronize()
    assert m.get_error(ws) == 0
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    tok = slice(0, 32)
    ref = oracle.moe_lora_layer(inp.x[tok], inp.W1, inp.W2, ids[tok], w[tok],
                                inp.token_adapter[tok], inp.A1, inp.B1, inp.A2, inp.B2)
    assert_close(y.cpu()[tok], ref, LAYER_RTOL, f"after recovery ({shape}, mode {expand_mode})")
