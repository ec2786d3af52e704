"""moe_route_static: the router entry point that allocates nothing (its scratch is a fixed
array inside the library), for callers that cannot allocate device memory -- serving loops that
must not call cudaMalloc on the hot path, or integrations handed only pre-allocated buffers.

Checked through the C ABI against moe_route (the workspace variant) on two calls in a row, and
against the oracle's router; the router's bar is bit-exact ids and weights.  The shapes reach
both router kernels through the fixed array: the small-batch cluster kernel (T <= 32, up to
E = 1024 at the array's size limit) and the tiled-logits + top-k kernels (T > 32).  Kept in a
file that is collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_routed_expert_gb300 import _lib, api, synth

pytestmark = pytest.mark.gpu


def _static_route(L, x, w_r, bias, k):
    T, d = x.shape
    E = w_r.shape[1]
    ids = torch.full((T, k), -7, dtype=torch.int32, device=x.device)
    w = torch.full((T, k), -1.0, dtype=torch.float32, device=x.device)
    rc = L.moe_route_static(_lib.ptr(x), _lib.ptr(w_r), _lib.ptr(bias), T, d, E, k, _lib.ptr(ids), _lib.ptr(w),
                            _lib.stream_handle())
    assert rc == _lib.BRE_OK, L.bre_status_string(rc)
    return ids, w


def _check_against_oracle(x, w_r, b, k, ids, w):
    ids_o, w_o = oracle.route(x.cpu(), w_r.cpu(), b.cpu(), k)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), np.asarray(w_o, dtype=np.float32).view(np.uint32))


def test_route_static_matches_workspace_route(cuda_dev):
    L = _lib.load()
    shape = synth.V41
    w_r = synth.router_weight(1, 0, shape.d, shape.E).to(cuda_dev)
    b = synth.route_bias(1, 0, shape.E, shape.bias_half_width).to(cuda_dev)
    for call, T in enumerate((8, 5)):             # two calls in a row, different batches
        x = synth.x_bf16(1, 0, 300 + call, T, shape.d).to(cuda_dev)
        ids_s, w_s = _static_route(L, x, w_r, b, shape.k)
        ids_r, w_r_out = api.moe_route(x, w_r, b, shape.k)
        torch.cuda.synchronize()
        assert torch.equal(ids_s, ids_r)
        assert torch.equal(w_s.view(torch.int32), w_r_out.view(torch.int32))
        _check_against_oracle(x, w_r, b, shape.k, ids_s, w_s)


@pytest.mark.parametrize("T,d,E", [(64, 4096, 384), (32, 512, 1024), (33, 256, 992)])
def test_route_static_both_kernels_at_the_size_limit(cuda_dev, T, d, E):
    """T = 64 at E = 384 runs the tiled-logits kernels through the array; T = 32 at E = 1024 is
    the small-batch kernel at its largest workspace (T * E = BRE_ROUTE_STATIC_MAX_TE); T = 33 at
    E = 992 is the tiled path just past the small-batch limit."""
    L = _lib.load()
    k = 6
    w_r = synth.router_weight(2, 0, d, E).to(cuda_dev)
    b = synth.route_bias(2, 0, E, 0.5).to(cuda_dev)
    for call in range(2):
        x = synth.x_bf16(2, 0, 400 + call, T, d).to(cuda_dev)
        ids_s, w_s = _static_route(L, x, w_r, b, k)
        ids_r, w_r_out = api.moe_route(x, w_r, b, k)
        torch.cuda.synchronize()
        assert torch.equal(ids_s, ids_r)
        assert torch.equal(w_s.view(torch.int32), w_r_out.view(torch.int32))
        _check_against_oracle(x, w_r, b, k, ids_s, w_s)


def test_route_static_rejects_sizes_beyond_its_scratch(cuda_dev):
    L = _lib.load()
    T, d, E, k = 64, 64, 1024, 6                  # T * E = 65536 > the fixed maximum
    x = torch.zeros((T, d), dtype=torch.bfloat16, device=cuda_dev)
    w_r = torch.zeros((d, E), dtype=torch.float32, device=cuda_dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=cuda_dev)
    w = torch.empty((T, k), dtype=torch.float32, device=cuda_dev)
    rc = L.moe_route_static(_lib.ptr(x), _lib.ptr(w_r), None, T, d, E, k, _lib.ptr(ids), _lib.ptr(w),
                            _lib.stream_handle())
    assert rc == _lib.BRE_ERR_WORKSPACE
