"""dyra_linear_forward_static: the forward for callers that cannot allocate device memory
(for example code running inside a custom allocator, or a serving process whose device
memory is fixed at start-up), which takes its scratch from a static array in the library.

The file name sorts last, so a run that stops at its first failure has run every other test
before this one. Each case compares the static-scratch forward with dyra_linear_forward on
the same layer and inputs, on two calls in a row with different inputs (the array keeps
the previous call's contents, so the second call checks that nothing stale leaks in)."""
import numpy as np
import pytest

import workloads as WL
from gpu_util import make_layer, rel, to_device, to_host, tol, weights_and_prep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import input_adaptive_rank_dyra_b300 as dy
    dy.load()
    yield


@pytest.mark.parametrize("name,batch", [("c2", 4), ("c1", 1)])
def test_static_forward_matches_workspace_forward_twice(name, batch):
    import torch
    import input_adaptive_rank_dyra_b300 as dy
    cfg = WL.reduced(WL.get_config(name), batch=2 * batch)
    W, b, prep = weights_and_prep(name)
    X = WL.make_inputs(cfg)
    layer = make_layer(cfg, prep, W, b)
    outs = []
    for call in range(2):
        Xd = to_device(X[call * batch:(call + 1) * batch], cfg.dtype)
        Y_ref = dy.linear_forward(layer, Xd)
        Y_static = dy.linear_forward_static(layer, Xd)
        torch.cuda.synchronize()
        a, r_ = to_host(Y_static), to_host(Y_ref)
        assert np.all(np.isfinite(a))
        assert rel(a, r_) <= tol(cfg), f"call {call}: {rel(a, r_):.3e}"
        outs.append(a)
    assert rel(outs[0], outs[1]) > tol(cfg)   # two different inputs, two different outputs


def test_static_forward_rejects_oversize_without_launching():
    import torch
    import input_adaptive_rank_dyra_b300 as dy
    cfg = WL.get_config("c2")
    W, b, prep = weights_and_prep("c2")
    layer = make_layer(cfg, prep, W, b)
    batch = 128
    need = layer.workspace_size(batch, cfg.n)
    assert need > 32 * 1024 * 1024
    X = torch.zeros((batch, cfg.n, cfg.d), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((batch, cfg.n, cfg.m), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dy.DyraError) as err:
        dy.linear_forward_static(layer, X, Y)
    assert err.value.status == 7          # DYRA_ERR_WORKSPACE
    assert "static" in str(err.value)
    torch.cuda.synchronize()
    assert bool((Y == 7.0).all())         # nothing was launched
