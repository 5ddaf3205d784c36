"""The C-ABI library builds, loads and exports every entry point of
include/instant.h; host-side validation answers without touching a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "instant.h")


@pytest.fixture(scope="module")
def L():
    from rank_compressed_backprop_gb300.build import build

    build()
    from rank_compressed_backprop_gb300._lib import lib

    return lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(instant_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_six_calls():
    names = declared_functions()
    for n in ["instant_compress_act", "instant_project_grad", "instant_grad_w",
              "instant_grad_x", "instant_calib_accumulate", "instant_calib_solve"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_functions():
        assert hasattr(L, n), n


def test_version_and_status_strings(L):
    assert L.instant_version() == 100
    for s in range(10):
        assert L.instant_status_string(s)
    assert L.instant_status_string(0) == b"ok"


def test_validation_without_gpu(L):
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: validation returns first
    null = ctypes.c_void_p(0)
    # bad dtype
    assert L.instant_compress_act(fake, fake, fake, 1, 8, 8, 4, 7, null) == 3
    # null pointer
    assert L.instant_compress_act(null, fake, fake, 1, 8, 8, 4, 1, null) == 1
    # bad shape: rank out of range
    assert L.instant_compress_act(fake, fake, fake, 1, 8, 8, 65, 1, null) == 2
    assert L.instant_project_grad(fake, fake, fake, fake, 1, 8, 8, 100, 100, 1, null) == 2
    # misaligned bf16 pointer / row pitch not a multiple of 8 elements
    odd = ctypes.c_void_p(0x1002)
    assert L.instant_project_grad(odd, fake, fake, fake, 1, 8, 64, 4, 4, 1, null) == 4
    assert L.instant_project_grad(fake, fake, fake, fake, 1, 8, 60, 4, 4, 1, null) == 4
    assert L.instant_grad_w(fake, fake, fake, 0, 2, 4, 60, 64, 1, null) == 4
    # workspace too small
    need = L.instant_grad_x_workspace_bytes(4, 64, 256, 256, 8, 1)
    assert need > 0
    assert L.instant_grad_x(fake, fake, fake, fake, fake, need - 1, 4, 64, 256, 256, 8, 1, null) == 5
    assert L.instant_calib_accumulate(fake, fake, 1, 9000, 8, 1, null) == 2


def test_static_grad_x_checks_alignment_before_any_launch(L):
    """instant_grad_x_static: a misaligned bf16 gx (or a row pitch that is not
    a multiple of 8) is reported before anything is launched, and before the
    call touches the device at all."""
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1002)
    null = ctypes.c_void_p(0)
    n0 = L.instant_launch_count()
    assert L.instant_grad_x_static(fake, fake, fake, odd, 4, 64, 256, 256, 8, 1, null) == 4
    assert L.instant_grad_x_static(odd, fake, fake, fake, 4, 64, 256, 256, 8, 1, null) == 4
    assert L.instant_grad_x_static(fake, odd, fake, fake, 4, 64, 256, 256, 8, 1, null) == 4
    assert L.instant_grad_x_static(fake, fake, fake, fake, 4, 64, 252, 256, 8, 1, null) == 4
    assert L.instant_grad_x_static(fake, fake, fake, fake, 4, 64, 256, 252, 8, 1, null) == 4
    assert L.instant_launch_count() == n0


def test_calib_solve_validation_without_gpu(L):
    from rank_compressed_backprop_gb300._lib import CalibParams

    fake = ctypes.c_void_p(0x1000)
    null = ctypes.c_void_p(0)
    k, R = ctypes.c_int(), ctypes.c_int()
    s = ctypes.c_float()
    prm = CalibParams(0.95, 2, 0, 1, 0, 0.0)
    need = L.instant_calib_workspace_bytes(512, 16)
    assert need > 0
    args = lambda n, Lr, rcap, ws_bytes, p=prm: L.instant_calib_solve(  # noqa: E731
        fake, n, Lr, ctypes.byref(p), fake, rcap, 1, ctypes.byref(k), ctypes.byref(R),
        ctypes.byref(s), None, None, fake, ws_bytes, null)
    assert args(0, 512, 16, need) == 1           # no samples
    assert args(8, 512, 200, need) == 2          # r_cap beyond the block limit
    assert args(8, 512, 16, need - 1) == 5       # workspace too small
    bad = CalibParams(1.5, 2, 0, 1, 0, 0.0)
    assert args(8, 512, 16, need, bad) == 1      # eps out of (0, 1]
    over = CalibParams(0.95, 2, 32, 1, 0, 0.0)
    assert args(8, 512, 16, need, over) == 2     # imposed rank beyond r_cap


def test_workspace_sizes_follow_the_plan(L):
    # the workspace holds g_hat_x [B*Ry, Cx] in the step's dtype (split-K is
    # reduced on chip, so it does not grow the workspace)
    f32 = L.instant_grad_x_workspace_bytes(1, 64, 64, 64, 4, 0)
    assert f32 == 1 * 4 * 64 * 4
    b2 = L.instant_grad_x_workspace_bytes(32, 512, 768, 768, 8, 1)
    assert b2 == 32 * 8 * 768 * 2


def test_python_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    from rank_compressed_backprop_gb300 import api

    x = torch.zeros(1, 8, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.compress_act(x, torch.zeros(4, 8, dtype=torch.bfloat16),
                         torch.zeros(1, 4, 8, dtype=torch.bfloat16))


def test_empty_extents_are_rejected_without_gpu(L):
    fake = ctypes.c_void_p(0x1000)
    null = ctypes.c_void_p(0)
    for B, Lr, C in ((0, 8, 64), (1, 0, 64), (1, 8, 0)):
        assert L.instant_compress_act(fake, fake, fake, B, Lr, C, 4, 1, null) == 2
        assert L.instant_project_grad(fake, fake, fake, fake, B, Lr, C, 4, 4, 1, null) == 2
        assert L.instant_calib_accumulate(fake, fake, B, Lr, C, 1, null) == 2
        assert L.instant_grad_x(fake, fake, fake, fake, fake, 1 << 20, B, Lr, C, 64, 4, 1, null) == 2
        assert L.instant_grad_w_x(fake, fake, fake, 0, fake, fake, fake, fake, fake, 1 << 20,
                                  B, Lr, C, 64, 4, 4, 1, null) == 2
        assert L.instant_grad_x_static(fake, fake, fake, fake, B, Lr, C, 64, 4, 1, null) == 2
    assert L.instant_grad_w(fake, fake, fake, 0, 0, 4, 64, 64, 1, null) == 2
    e2, n2 = ctypes.c_double(), ctypes.c_double()
    assert L.instant_reconstruction_error(fake, fake, fake, 0, 8, 64, 4, 1, ctypes.byref(e2),
                                          ctypes.byref(n2), fake, 16, null) == 2
    assert L.instant_reconstruction_error(fake, fake, fake, 1, 8, 64, 4, 1, ctypes.byref(e2),
                                          ctypes.byref(n2), fake, 8, null) == 5


def test_batch_solve_validation_without_gpu(L):
    from rank_compressed_backprop_gb300._lib import CalibParams, CalibProblem

    assert L.instant_calib_batch_workspace_bytes(512, 2) >= 2 * L.instant_calib_workspace_bytes(512, 8)
    assert L.instant_calib_batch_workspace_bytes(0, 2) == 0
    assert L.instant_calib_solve_batch(None, 1, 64, 1, ctypes.c_void_p(0x1000), 1 << 30, None) == 1
    arr = (CalibProblem * 2)()
    for i in range(2):
        arr[i] = CalibProblem(0x1000 + 4096 * i, 4, CalibParams(0.95, 0, 8, 1, 0, 0.0, 0),
                              0x100000 + 4096 * i, 8, None, 0, 0, 0.0, 0.0, -1)
    fake = ctypes.c_void_p(0x200000)
    assert L.instant_calib_solve_batch(arr, 0, 64, 1, fake, 1 << 30, None) == 1
    need = L.instant_calib_batch_workspace_bytes(64, 2)
    assert L.instant_calib_solve_batch(arr, 2, 64, 1, fake, need - 1, None) == 5
    assert [arr[i].status for i in range(2)] == [5, 5]
    arr[1].prm.r_override = 9                 # beyond r_cap
    assert L.instant_calib_solve_batch(arr, 2, 64, 1, fake, need, None) == 2
    assert [arr[i].status for i in range(2)] == [2, 2]
    arr[1].prm.r_override = 8
    assert L.instant_calib_solve_batch(arr, 2, 64, 7, fake, need, None) == 3   # dtype


def test_backward_validation_without_gpu(L):
    fake = ctypes.c_void_p(0x1000)
    need = L.instant_backward_workspace_bytes(32, 512, 768, 768, 8, 1)
    assert need >= 256 + L.instant_grad_x_workspace_bytes(32, 512, 768, 768, 8, 1)
    args = lambda B=32, Lr=512, Cx=768, Cy=768, Rx=8, Ry=8, dt=1, ws_bytes=need, ws=fake: (  # noqa: E731
        fake, fake, fake, fake, fake, fake, fake, 0, fake, ws, ws_bytes, B, Lr, Cx, Cy, Rx, Ry, dt,
        None)
    assert L.instant_backward(*args(dt=7)) == 3
    assert L.instant_backward(*args(B=0)) == 2
    assert L.instant_backward(*args(Lr=0)) == 2
    assert L.instant_backward(*args(Rx=70, Ry=64)) == 2
    assert L.instant_backward(*args(Ry=65)) == 2
    assert L.instant_backward(*args(ws_bytes=need - 1)) == 5
    assert L.instant_backward(*args(ws=ctypes.c_void_p(0x1008))) == 4
    assert L.instant_backward(*args(Cx=764)) == 4            # Cx % 8 != 0 for bf16


def test_accumulate_batch_validation_without_gpu(L):
    from rank_compressed_backprop_gb300._lib import AccumulateItem

    items = (AccumulateItem * 2)(AccumulateItem(0x1000, 0x2000, 4, 64),
                                 AccumulateItem(0x3000, 0x4000, 4, 128))
    assert L.instant_calib_accumulate_batch(None, 1, 64, 1, None) == 1
    assert L.instant_calib_accumulate_batch(items, 0, 64, 1, None) == 1
    assert L.instant_calib_accumulate_batch(items, 2, 64, 7, None) == 3
    assert L.instant_calib_accumulate_batch(items, 2, 0, 1, None) == 2
    assert L.instant_calib_accumulate_batch(items, 2, 8193, 1, None) == 2
    items[1].B = 0
    assert L.instant_calib_accumulate_batch(items, 2, 64, 1, None) == 2
    items[1].B = 4
    items[1].Cdim = 60                      # not a multiple of 8 for bf16
    assert L.instant_calib_accumulate_batch(items, 2, 64, 1, None) == 4
    items[1].Cdim = 128
    items[1].t = 0x3008                     # misaligned
    assert L.instant_calib_accumulate_batch(items, 2, 64, 1, None) == 4
    items[1].t = None
    assert L.instant_calib_accumulate_batch(items, 2, 64, 1, None) == 1
