"""The bounded waits of the expert FFN kernels, made to run out on purpose with a tiny budget
(bre_set_ffn_wait_limit): the call returns, BRE_DEVERR_TIMEOUT is set in dev_err after
synchronisation (strix-llama.cpp issue, ROCm cached-expert notes: runtime errors surface after
synchronisation, never as a trap), and the next call on the same workspace, with the default
budget, is bit-identical to a clean one.  Each kernel that gives up still waits (with the
default budget) for the copies and tensor-core operations it has in flight before it exits.
Covers the decode path (T = 8, V4.1 shape) and the grouped-GEMM path (T = 64, d = 512)."""
import pytest
import torch

from bit_routed_expert_gb300 import _lib, synth
from helpers import device_layer

pytestmark = pytest.mark.gpu

SEED = 1


@pytest.mark.parametrize("shape,T", [(synth.V41, 8), (synth.TINY, 64)])
def test_ffn_wait_budget_runs_out_then_next_call_is_clean(cuda_dev, shape, T):
    L = _lib.load()
    layer = device_layer(SEED, 0, shape, T, cuda_dev)
    x = synth.x_bf16(SEED, 0, 70, T, shape.d).to(cuda_dev)
    ref, _ = layer.forward(x)
    ref = ref.clone()
    torch.cuda.synchronize()
    assert int(layer.dev_err) == 0
    try:
        assert L.bre_set_ffn_wait_limit(1) == _lib.BRE_OK
        layer.forward(x)
        torch.cuda.synchronize()
    finally:
        assert L.bre_set_ffn_wait_limit(0) == _lib.BRE_OK
    assert int(layer.dev_err) & _lib.BRE_DEVERR_TIMEOUT
    layer.dev_err.zero_()
    again, _ = layer.forward(x)
    torch.cuda.synchronize()
    assert int(layer.dev_err) == 0
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))


def test_ffn_wait_limit_rejects_negative():
    L = _lib.load()
    assert L.bre_set_ffn_wait_limit(-1) == _lib.BRE_ERR_ARG
