"""Host threads calling the library at once, each on its own stream, with
configurations whose launch parameters (shared memory sizes, residency counts)
are planned and cached on first use: every result still matches the oracle."""

import threading

import numpy as np
import pytest

import oracle as O
from gpu_util import assert_parity, nan_like, orthonormal_rows, rng, stored, to_dev, to_np, torch_or_skip

pytestmark = pytest.mark.gpu


def test_threads_plan_and_launch_together():
    torch = torch_or_skip()
    from rank_compressed_backprop_gb300 import api

    # (B, L, Cx, Cy, Ry): short and long token axes, both Q^T paths
    shapes = [(6, 49, 192, 64, 16), (4, 512, 256, 64, 16), (3, 300, 264, 136, 8),
              (5, 130, 136, 72, 8)]
    cases = []
    for i, (B, L, Cx, Cy, Ry) in enumerate(shapes):
        g = rng(5200 + i)
        Sq = stored(g.standard_normal((B * Ry, Cy)), "bf16")
        w = stored(g.standard_normal((Cy, Cx)) / np.sqrt(Cy), "bf16")
        Q = stored(orthonormal_rows(g, Ry, L), "bf16")
        t = stored(g.standard_normal((B, L, Cy)), "bf16")
        PQ = stored(orthonormal_rows(g, 2 * Ry, L), "bf16")
        cases.append((B, L, Cx, Cy, Ry, Sq, w, Q, t, PQ))
    outs = [None] * len(cases)
    errors = []

    def work(k):
        try:
            B, L, Cx, Cy, Ry, Sq, w, Q, t, PQ = cases[k]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                gx = nan_like(torch, (B, L, Cx), torch.bfloat16)
                Sx = nan_like(torch, (B * Ry, Cy), torch.bfloat16)
                S2 = nan_like(torch, (B * Ry, Cy), torch.bfloat16)
                ws = torch.empty(api.grad_x_workspace_bytes(B, L, Cx, Cy, Ry, torch.bfloat16),
                                 dtype=torch.uint8, device="cuda")
                dSq, dw, dQ, dt, dPQ = (to_dev(a) for a in (Sq, w, Q, t, PQ))
                for _ in range(3):
                    api.grad_x_core(dSq, dw, ws, B, stream=s)
                    api.expand(dQ, gx, ws, Cy, stream=s)
                    api.project_grad(dt, dPQ, Sx, S2, Ry, Ry, stream=s)
                s.synchronize()
            outs[k] = (gx, Sx, S2)
        except Exception as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(len(cases))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for (B, L, Cx, Cy, Ry, Sq, w, Q, t, PQ), (gx, Sx, S2) in zip(cases, outs):
        ref = O.grad_x(O.decode(Sq).reshape(B, Ry, Cy), w, Q)
        assert_parity(to_np(gx), ref, 2e-2, "g_x")
        r0, r1 = O.project_grad(t, PQ[:Ry], PQ[Ry:])
        assert_parity(to_np(Sx).reshape(B, Ry, Cy), r0, 2e-2, "Sx")
        assert_parity(to_np(S2).reshape(B, Ry, Cy), r1, 2e-2, "Sq")
    assert api.device_status() == 0
