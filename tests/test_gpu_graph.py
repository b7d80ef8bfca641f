"""Chained calls through a captured CUDA graph give the same bits as eager
calls.  The hot-path kernels start while their predecessor drains
(programmatic dependent launch) and wait for it before any global access;
here every call reads the previous call's output (layer 2's queries are
layer 1's O, layer 1's upstream gradient is layer 2's dQ), so a missing wait
would show as a difference between replays and the eager run."""
import pytest

import oracle as o
import sfa_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sfa(sfa_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import static_offset_sparse_gb300 as s

    return s


def _two_layers(sfa, x1, x2, fwd, bwd):
    """Layer 2 reads layer 1's output as its queries; layer 1's backward takes
    layer 2's dQ as its upstream gradient."""
    O1, L1 = fwd(x1["q"], x1["k"], x1["v"])
    O2, L2 = fwd(O1, x2["k"], x2["v"])
    g2 = bwd(O1, x2["k"], x2["v"], O2, L2, x2["do"])
    g1 = bwd(x1["q"], x1["k"], x1["v"], O1, L1, g2[0])
    return (O1, L1, O2, L2) + tuple(g2) + tuple(g1)


def _check_graph_matches_eager(sfa, x1, x2, fwd, bwd):
    import torch

    d1 = {n: t.cuda() for n, t in x1.items()}
    d2 = {n: t.cuda() for n, t in x2.items()}
    eager = _two_layers(sfa, d1, d2, fwd, bwd)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up on the capture stream
        _two_layers(sfa, d1, d2, fwd, bwd)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = _two_layers(sfa, d1, d2, fwd, bwd)
    for _ in range(3):
        for t in out:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert sfa.get_device_status() == 0
        for a, b in zip(eager, out):
            assert torch.equal(a, b)


def test_rung_path_graph_matches_eager(sfa):
    """Interpolated path, 8/2 heads (rung kernels, rotated keys in each call)."""
    base = o.fib_offsets(15)
    x1 = si.make_qkvdo(2, 512, 8, 2, 64, "bf16", seed=71)
    x2 = si.make_qkvdo(2, 512, 8, 2, 64, "bf16", seed=72)
    fwd = lambda q, k, v: sfa.forward(q, k, v, W=8, alpha=1.13, base=base)  # noqa: E731
    bwd = lambda q, k, v, O, L, dO: sfa.backward(q, k, v, O, L, dO, W=8, alpha=1.13,  # noqa: E731
                                                 base=base)
    _check_graph_matches_eager(sfa, x1, x2, fwd, bwd)


def test_band_path_graph_matches_eager(sfa):
    """Christoffel 128/1024 offsets, 4/4 heads (band kernels)."""
    dist = o.christoffel_offsets(128, 1024, include_zero=True)
    assert sfa.band_plan(dist, 2048, 1)[0] == 8
    x1 = si.make_qkvdo(1, 2048, 4, 4, 64, "bf16", seed=73)
    x2 = si.make_qkvdo(1, 2048, 4, 4, 64, "bf16", seed=74)
    fwd = lambda q, k, v: sfa.forward_int(q, k, v, dist=dist)  # noqa: E731
    bwd = lambda q, k, v, O, L, dO: sfa.backward_int(q, k, v, O, L, dO, dist=dist)  # noqa: E731
    _check_graph_matches_eager(sfa, x1, x2, fwd, bwd)
