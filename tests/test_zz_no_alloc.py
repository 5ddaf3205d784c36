"""instant_grad_x_static (the input gradient with g_hat_x in the library's
fixed device array) agrees with instant_grad_x on the same inputs, call after
call, without any device allocation by the caller.

Collected last so that it also runs after every other GPU test in the same
process; it passes alone in a fresh process as well."""

import ctypes

import numpy as np
import pytest

import oracle as O
from gpu_util import (assert_parity, nan_like, orthonormal_rows, rng, stored, to_dev, to_np, tol,
                      torch_or_skip)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


CASES = [
    # dtype, B, L, Cx, Cy, Ry
    ("bf16", 32, 512, 768, 768, 8),      # BERT-base block: instant_grad_x takes its fused kernel
    ("bf16", 3, 200, 136, 264, 5),       # ragged tiles on every axis
    ("bf16", 4, 256, 256, 3072, 16),     # long contraction: instant_grad_x uses the same two kernels
    ("f32", 2, 72, 40, 48, 4),
]


def _inputs(torch, dtype, B, L, Cx, Cy, Ry, seed):
    g = rng(seed)
    host = (stored(g.standard_normal((B * Ry, Cy)), dtype),
            stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), dtype),
            stored(orthonormal_rows(g, Ry, L), dtype))
    return tuple(to_dev(a) for a in host), host


@pytest.mark.parametrize("dtype,B,L,Cx,Cy,Ry", CASES)
def test_static_scratch_matches_grad_x(torch, dtype, B, L, Cx, Cy, Ry):
    from rank_compressed_backprop_gb300 import api

    (Sq, w, Q), (Sq_h, w_h, Q_h) = _inputs(torch, dtype, B, L, Cx, Cy, Ry, 9100 + B + Ry)
    tdt = Sq.dtype
    ws = torch.empty(max(api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, tdt), 16), dtype=torch.uint8,
                     device="cuda")
    ref = nan_like(torch, (B, L, Cx), tdt)
    api.grad_x(Sq, w, Q, ref, ws)
    first = torch.full((B, L, Cx), float("nan"), dtype=tdt, device="cuda")
    second = torch.full((B, L, Cx), float("nan"), dtype=tdt, device="cuda")
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved())
    api.grad_x_static(Sq, w, Q, first)
    api.grad_x_static(Sq, w, Q, second)
    torch.cuda.synchronize()
    assert (torch.cuda.memory_allocated(), torch.cuda.memory_reserved()) == before
    from rank_compressed_backprop_gb300 import _lib

    assert _lib.lib().instant_device_status(1, None) == 0
    r = to_np(ref)
    oracle = O.grad_x(O.decode(Sq_h).reshape(B, Ry, Cy), w_h, Q_h)
    assert_parity(r, oracle, tol(dtype), "grad_x vs oracle")
    for out in (first, second):
        o = to_np(out)
        assert_parity(o, r, tol(dtype), "grad_x_static vs grad_x")
        assert_parity(o, oracle, tol(dtype), "grad_x_static vs oracle")
    # the two calls in a row run the same kernels on the same inputs
    assert torch.equal(first, second)


def test_static_scratch_rejects_a_misaligned_output_before_launching(torch):
    from rank_compressed_backprop_gb300._lib import lib

    B, L, Cx, Cy, Ry = 2, 64, 256, 256, 8
    (Sq, w, Q), _ = _inputs(torch, "bf16", B, L, Cx, Cy, Ry, 9200)
    buf = torch.full((B * L * Cx + 8,), 3.0, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    n0 = lib().instant_launch_count()
    st = lib().instant_grad_x_static(ctypes.c_void_p(Sq.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                     ctypes.c_void_p(Q.data_ptr()),
                                     ctypes.c_void_p(buf.data_ptr() + 2),   # 2 bytes off
                                     B, L, Cx, Cy, Ry, 1, None)
    assert st == 4                                                     # INSTANT_ERR_ALIGN
    assert lib().instant_launch_count() == n0
    torch.cuda.synchronize()
    assert bool((buf == 3.0).all())


def test_static_scratch_rejects_sizes_beyond_the_array(torch):
    from rank_compressed_backprop_gb300 import api
    from rank_compressed_backprop_gb300._lib import GRAD_X_STATIC_SCRATCH_BYTES, lib

    B, L, Cy, Ry = 64, 128, 64, 64
    Cx = 1024 + 8                         # B*Ry*Cx*2 just past the 8 MiB array
    assert api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, torch.bfloat16) > GRAD_X_STATIC_SCRATCH_BYTES
    Sq = torch.zeros(B * Ry, Cy, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(Cy, Cx, dtype=torch.bfloat16, device="cuda")
    Q = torch.zeros(Ry, L, dtype=torch.bfloat16, device="cuda")
    gx = torch.full((B, L, Cx), 3.0, dtype=torch.bfloat16, device="cuda")
    n0 = lib().instant_launch_count()
    with pytest.raises(ValueError, match="fixed array"):
        api.grad_x_static(Sq, w, Q, gx)
    assert lib().instant_launch_count() == n0
    st = lib().instant_grad_x_static(ctypes.c_void_p(Sq.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                     ctypes.c_void_p(Q.data_ptr()), ctypes.c_void_p(gx.data_ptr()),
                                     B, L, Cx, Cy, Ry, 1, None)
    assert st == 5
    torch.cuda.synchronize()
    assert bool((gx == 3.0).all())
    # exactly at the limit is accepted
    Cx = 1024
    assert api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, torch.bfloat16) == GRAD_X_STATIC_SCRATCH_BYTES
    w = torch.zeros(Cy, Cx, dtype=torch.bfloat16, device="cuda")
    gx = torch.full((B, L, Cx), 3.0, dtype=torch.bfloat16, device="cuda")
    api.grad_x_static(Sq, w, Q, gx)
    torch.cuda.synchronize()
    assert bool((gx == 0).all())
