"""The cluster engine (a row split across a thread-block cluster) against the
fp64 oracle: chosen by default for aligned rows longer than one CTA's tile,
and forced onto short rows to cover every cluster size, both weight-gradient
modes and the fused-add variant."""
import pytest
import torch

from rmsnorm_backward_bwd_gb300 import native
from rmsnorm_backward_bwd_gb300.synth import Case

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_options():
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)
    yield
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)


def _run(case):
    ex = parity.expected_bwd(case)
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    parity.check_bwd(ex, dx, dw, dw32, tag=" [%s]" % plan)
    return plan, (dx, dw, dw32)


@pytest.mark.parametrize("M,N,dt,csize", [(64, 16392, "bf16", 2), (24, 32768, "bf16", 2),
                                          (12, 65536, "bf16", 4), (5, 131072, "bf16", 8),
                                          (3, 262144, "bf16", 16), (16, 16384, "f32", 2),
                                          (7, 24576, "f16", 2), (4, 60000, "f32", 8)],
                         ids=lambda v: str(v))
@pytest.mark.parametrize("fused", [False, True])
def test_long_rows_take_the_cluster_engine(M, N, dt, csize, fused):
    plan, _ = _run(Case("cluster %s M=%d N=%d" % (dt, M, N), M, N, dt, fused=fused,
                        with_dres=fused))
    assert "engine=cluster" in plan and "csize=%d" % csize in plan, plan


@pytest.mark.parametrize("csize", [2, 4, 8, 16])
@pytest.mark.parametrize("mode", [1, 2])
def test_forced_cluster_sizes_on_short_rows(csize, mode):
    native.set_option(native.OPT_BWD_ENGINE, 3)
    native.set_option(native.OPT_CLUSTER_SIZE, csize)
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    plan, _ = _run(Case("cluster bf16 M=300 N=4096", 300, 4096, "bf16", seed=csize))
    assert "csize=%d" % csize in plan and ("atomic" if mode == 2 else "scratch") in plan, plan


@pytest.mark.parametrize("cpt,stages", [(1, 2), (2, 3), (4, 2), (4, 4)])
def test_cluster_tile_options(cpt, stages):
    native.set_option(native.OPT_BWD_ENGINE, 3)
    native.set_option(native.OPT_CLUSTER_SIZE, 2)
    native.set_option(native.OPT_CHUNKS_PER_THREAD, cpt)
    native.set_option(native.OPT_STAGES, stages)
    plan, _ = _run(Case("cluster f16 M=99 N=8192", 99, 8192, "f16", fused=True, with_dres=True))
    assert "cpt=%d" % cpt in plan and "stages=%d" % stages in plan, plan


def test_fewer_rows_than_clusters():
    plan, _ = _run(Case("cluster bf16 M=3 N=65536", 3, 65536, "bf16"))
    assert "clusters=3" in plan, plan


def test_cluster_scratch_mode_is_repeatable():
    native.set_option(native.OPT_DWEIGHT_MODE, 1)
    case = Case("cluster bf16 M=200 N=32768", 200, 32768, "bf16")
    ex = parity.expected_bwd(case)
    a = parity.run_gpu_bwd(ex)
    b = parity.run_gpu_bwd(ex)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    parity.check_bwd(ex, *a)


def test_cluster_grid_cap():
    native.set_option(native.OPT_GRID, 8)
    plan, _ = _run(Case("cluster bf16 M=50 N=32768", 50, 32768, "bf16"))
    assert "clusters=4" in plan, plan


def test_forced_cluster_refuses_unaligned_rows():
    native.set_option(native.OPT_BWD_ENGINE, 3)
    ex = parity.expected_bwd(Case("cluster bf16 M=4 N=4099", 4, 4099, "bf16"))
    with pytest.raises(native.RNError, match="cluster engine cannot take"):
        parity.run_gpu_bwd(ex)
