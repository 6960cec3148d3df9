"""The backward on side streams and inside CUDA graphs.

The library launches only on the caller's stream and allocates nothing; the
binding keeps one workspace per (device, stream). So two streams may run
backwards at once, and a call made once outside capture (first-call setup:
device queries and kernel attributes) can then be captured into a CUDA graph
and replayed.
"""
import pytest
import torch

import parity
import rmsnorm_backward_bwd_gb300 as rn
from rmsnorm_backward_bwd_gb300 import native, ops
from rmsnorm_backward_bwd_gb300.synth import Case

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_options():
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)
    yield


def _device_inputs(ex):
    t = dict(x=ex.x.cuda(), g=ex.gamma.cuda(), dy=ex.dy.cuda(), rstd=ex.rstd.cuda())
    if ex.case.fused and ex.dres is not None:
        t["dres"] = ex.dres.cuda()
    return t


@pytest.mark.parametrize("mode", [1, 2])
def test_two_streams_concurrently(mode):
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    exs = [parity.expected_bwd(Case("s%d" % i, 2048, 4096, "bf16", seed=i)) for i in range(2)]
    ins = [_device_inputs(ex) for ex in exs]
    streams = [torch.cuda.Stream() for _ in exs]
    torch.cuda.synchronize()
    outs = []
    for _ in range(3):   # several rounds so the two streams overlap
        outs = []
        for st, t in zip(streams, ins):
            with torch.cuda.stream(st):
                outs.append(rn.rmsnorm_bwd(t["x"], t["g"], t["dy"], t["rstd"]))
    torch.cuda.synchronize()
    for ex, (dx, dw, dw32) in zip(exs, outs):
        parity.check_bwd(ex, dx, dw, dw32)


@pytest.mark.parametrize("case", [Case("graph plain", 1024, 4096, "bf16"),
                                  Case("graph fused", 512, 3000, "f32", fused=True, with_dres=True),
                                  Case("graph long rows", 8, 32768, "bf16")],
                         ids=lambda c: c.name)
@pytest.mark.parametrize("mode", [1, 2])
def test_backward_captured_in_a_cuda_graph(case, mode):
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    ex = parity.expected_bwd(case)
    t = _device_inputs(ex)
    x, g, dy, rstd = t["x"], t["g"], t["dy"], t["rstd"]
    dx = torch.empty_like(x)
    dw32 = torch.empty(case.N, dtype=torch.float32, device="cuda")
    dw = torch.empty(case.N, dtype=x.dtype, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ws = rn.bwd_workspace(case.M, case.N, x.dtype, x.device)

        def call():
            if case.fused:
                rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, t.get("dres"), dx=dx, dweight_f32=dw32,
                                         dweight=dw, workspace=ws)
            else:
                rn.rmsnorm_bwd(x, g, dy, rstd, dx=dx, dweight_f32=dw32, dweight=dw, workspace=ws)
        call()   # first call outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        call()
    for buf in (dx, dw32, dw):
        buf.fill_(7)          # replays must rewrite every output
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    parity.check_bwd(ex, dx, dw, dw32)


def test_graph_keeps_its_workspace_after_the_cache_grows():
    """A graph captured on a stream whose cached workspace then grows (a wider
    call on the same stream) must still own its buffer: the binding keeps the
    smaller workspace allocated, so no later tensor is placed under the
    graph's scratch writes."""
    native.set_option(native.OPT_DWEIGHT_MODE, 1)      # scratch: the partials live in the workspace
    ex = parity.expected_bwd(Case("graph ws small", 512, 1024, "bf16"))
    t = _device_inputs(ex)
    x, g, dy, rstd = t["x"], t["g"], t["dy"], t["rstd"]
    dx = torch.empty_like(x)
    dw32 = torch.empty(1024, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        rn.rmsnorm_bwd(x, g, dy, rstd, dx=dx, dweight_f32=dw32)   # caches this stream's workspace
        small_ws_bytes = ops._ws_bytes(512, 1024, native.RN_BF16, 0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        rn.rmsnorm_bwd(x, g, dy, rstd, dx=dx, dweight_f32=dw32)
    # a wider call on the same stream replaces the cached workspace
    wide = parity.expected_bwd(Case("graph ws wide", 64, 8192, "bf16"))
    tw = _device_inputs(wide)
    with torch.cuda.stream(side):
        rn.rmsnorm_bwd(tw["x"], tw["g"], tw["dy"], tw["rstd"])
    torch.cuda.synchronize()
    # tensors of the small workspace's size: the allocator would hand them its block if freed
    canaries = [torch.full((small_ws_bytes,), 0x5A, dtype=torch.uint8, device="cuda")
                for _ in range(4)]
    dx.fill_(7)
    graph.replay()
    torch.cuda.synchronize()
    parity.check_bwd(ex, dx, None, dw32)
    for c in canaries:
        assert bool((c == 0x5A).all()), "a graph replay wrote into a later tensor"


@pytest.mark.parametrize("mode", [1, 2])
def test_staged_kernels_captured_in_a_cuda_graph(mode):
    """The staged phase-class kernels (mbarriers initialised by every launch)
    replayed from a CUDA graph: the RMSNorm backward and the three forwards on
    rows that are not 16-byte multiples; every replay rewrites every output and
    matches the eager call bit for bit."""
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    ex = parity.expected_bwd(Case("graph staged", 2048, 4095, "bf16", fused=True, with_dres=True,
                                  seed=81))
    t = _device_inputs(ex)
    x, g, dy, rstd, dres = t["x"], t["g"], t["dy"], t["rstd"], t["dres"]
    outs = {k: torch.empty_like(x) for k in ("dx", "y", "lny")}
    dw32 = torch.empty(4095, dtype=torch.float32, device="cuda")
    dw = torch.empty(4095, dtype=x.dtype, device="cuda")
    st1 = {k: torch.empty(2048, dtype=torch.float32, device="cuda") for k in ("rstd", "mean", "lrstd")}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ws = rn.bwd_workspace(2048, 4095, x.dtype, x.device)

        def call():
            rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres, dx=outs["dx"], dweight_f32=dw32,
                                     dweight=dw, workspace=ws)
            rn.rmsnorm_fwd(x, g, 1e-6, y=outs["y"], rstd=st1["rstd"])
            rn.layernorm_fwd(x, g, g, 1e-5, y=outs["lny"], mean=st1["mean"], rstd=st1["lrstd"])
        call()   # first call outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert "staged" in native.last_plan(), native.last_plan()
    eager = {k: v.clone() for k, v in list(outs.items()) + list(st1.items())}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        call()
    for _ in range(2):
        for buf in list(outs.values()) + list(st1.values()) + [dw32, dw]:
            buf.fill_(7)      # every replay must rewrite every output
        graph.replay()
        torch.cuda.synchronize()
        for k, v in list(outs.items()) + list(st1.items()):
            assert torch.equal(v, eager[k]), k   # dx, y and the statistics are deterministic
        parity.check_bwd(ex, outs["dx"], dw, dw32)
    assert native.take_device_status() == 0
