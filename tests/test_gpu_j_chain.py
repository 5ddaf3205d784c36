"""A projection whose input the preceding launch has just written.

Projection CTAs prefetch their input tile into L2 before they wait for the
preceding kernel (programmatic dependent launch).  That is only correct
because L2 is the point of coherence: lines fetched early are updated by the
predecessor's later writes, and the real loads come after the wait.  This
test chains compress_act launches so that each reads the output of the one
before (x_hat has the shape of an input when Rx = L), eagerly and as a CUDA
graph, and compares every link with the oracle on the stored bf16 values."""

import numpy as np
import pytest

import oracle as O
from gpu_util import assert_parity, orthonormal_rows, rel, rng, stored, to_dev, to_np, torch_or_skip

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_or_skip()


@pytest.mark.parametrize("graph", [False, True])
def test_projection_reads_what_its_predecessor_wrote(torch, graph):
    from rank_compressed_backprop_gb300 import api

    g = rng(9300 + int(graph))
    B, L, C = 16, 64, 768                       # x_hat [B, L, C] when Rx = L
    links = 6
    x0 = stored(g.standard_normal((B, L, C)), "bf16")
    # an orthonormal P keeps the values bounded along the chain
    P = stored(orthonormal_rows(g, L, L), "bf16")
    bufs = [to_dev(x0)] + [torch.full((B, L, C), float("nan"), dtype=torch.bfloat16, device="cuda")
                           for _ in range(links)]
    Pd = to_dev(P)

    def chain():
        for i in range(links):
            api.compress_act(bufs[i], Pd, bufs[i + 1])

    if graph:
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cs):
            with torch.cuda.graph(gr, stream=cs):
                chain()
        torch.cuda.current_stream().wait_stream(cs)
        for b in bufs[1:]:
            b.fill_(float("nan"))
        for _ in range(3):
            gr.replay()
    else:
        chain()
    torch.cuda.synchronize()
    cur = x0
    for i in range(links):
        want = O.compress_act(cur, P)                 # fp64 from the stored bits
        got = to_np(bufs[i + 1])
        assert_parity(got, want, 2e-2, f"link {i}")
        cur = stored(got, "bf16")                     # the next link reads the stored values
    assert api.device_status() == 0
