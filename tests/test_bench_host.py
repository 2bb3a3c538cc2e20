"""bench.py's host-side accounting, on the CPU: the per-kernel algorithmic FLOPs of a forward
add up to the layer's FLOP model, and the recorded DRAM traffic file is well formed."""
import os
import re

import pytest

import bench
import workloads as WL

MAIN = ("xproj_static_L", "residual_product", "fused_output")


@pytest.mark.parametrize("name", ["c2", "c3_fc1", "c3_fc2", "c5"])
def test_kernel_flops_add_up_to_the_layer_model(name):
    """xproj (X [U | P]), the Gram GEMM (L^T L, L^T X), the residual product and the output
    GEMM are exactly the layer model's terms; the fused solve adds the inversion (2 r^3) and
    the apply (2 r^2 d) per sample on top."""
    cfg = WL.get_config(name)
    B, d, r = cfg.batch, cfg.d, cfg.r
    main = sum(bench.kernel_work(cfg, k)[0] for k in MAIN)
    gram = bench.kernel_work(cfg, "cg_c_gram")[0]
    assert main + gram == pytest.approx(bench.layer_flops(cfg), rel=1e-12)
    fused = bench.kernel_work(cfg, "cg_solve")[0]
    assert fused - gram == pytest.approx(B * (2.0 * r ** 3 + 2.0 * r * r * d), rel=1e-12)


def test_als_adds_the_l_update_terms():
    """t = 2 adds one L-update (R R^T, W_res R^T, the apply of (R R^T)^-1, X P) and one more
    R-update to the t = 1 model."""
    cfg = WL.get_config("c2")
    cfg2 = bench.bench_config("c2_t2")
    B, n, d, m, r = cfg.batch, cfg.n, cfg.d, cfg.m, cfg.r
    l_update = 2.0 * r * r * m + 2.0 * d * m * r + 2.0 * r * r * d + 2.0 * n * d * r
    r_update = 2.0 * n * r * r + 2.0 * n * r * d + 2.0 * r * d * m
    assert bench.layer_flops(cfg2) - bench.layer_flops(cfg) == pytest.approx(
        B * (l_update + r_update), rel=1e-12)


def test_recorded_traffic_file_is_well_formed():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")
    lines = [l for l in open(path) if l.strip() and not l.startswith("#")]
    assert lines
    workloads = {WL.get_config(c).name for c in WL.CONFIGS}
    for line in lines:
        wl, kernel, nbytes, h = line.split()
        assert wl in workloads, wl
        assert int(nbytes) > 0
        assert re.fullmatch(r"[0-9a-f]{12}", h), h
        # a record whose hash is the kernel's current one is the figure bench.py reports
        if h == bench.kernel_source_hash(kernel):
            assert bench.recorded_traffic(wl, kernel) == float(nbytes)
