"""The kernel count that the benchmark reports as gpu_launches comes from
MoELayerStep.launches() / ChunkedLayerStep.launches().  Here the CUDA
profiler's kernel records of one eager pass over a stream's layers are
counted and compared with that figure, for every way the layer step can be
put together: the fused front (with and without the prediction), the
separate calls, the gather FFN, the combine in GEMM2's epilogue, physical
replica copies, SwiGLU, experts too large for the fused FFN kernel, and the
chunked step."""
import dataclasses
import re

import pytest

from moe_expert_routing_02_b300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
import moe_expert_routing_02_b300 as M  # noqa: E402
from moe_expert_routing_02_b300.layer import ChunkedLayerStep, MoELayerStep  # noqa: E402

# namespaces of the library's kernels
LIB_NS = {"front", "route", "stats", "replicate", "dispatch", "ffn", "ffn2", "ffn3", "ffn_small", "ffn_wg",
          "combine", "replica_copy", "bwd"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from moe_expert_routing_02_b300 import _build
    _build.build()
    M.lib()


def _namespace(name: str) -> str:
    """Outer namespace of a kernel record's name, demangled
    ('void front::route_count_kernel<2, true>(front::Args)') or mangled
    ('_ZN5front18route_count_kernel...')."""
    m = re.match(r"_ZN(\d+)", name)
    if m:
        n = int(m.group(1))
        start = m.end()
        return name[start:start + n]
    fn = name.split("(")[0].split("<")[0].strip()
    if fn.startswith("void "):
        fn = fn[5:]
    return fn.split("::")[0] if "::" in fn else ""


def test_namespace_parser():
    assert _namespace("void front::route_count_kernel<2, true>(front::Args)") == "front"
    assert _namespace("void ffn3::ffn_fused_kernel<(ffn::Epi)0>(CUtensorMap, ffn::Params)") == "ffn3"
    assert _namespace("_ZN9ffn_small12small_kernelILN3ffn3EpiE0EEEvNS1_6ParamsE") == "ffn_small"
    assert _namespace("Memset (Device)") == ""
    assert _namespace("void at::native::vectorized_elementwise_kernel<4>(int)") == "at"


def _count_kernels(body):
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CPU, ProfilerActivity.CUDA]) as prof:
        body()
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    ours = [n for n in names if _namespace(n) in LIB_NS]
    return len(ours), ours


def _layer_inputs(c, physical=False):
    lgs = [torch.from_numpy(l).cuda() for l in W.make_layer_logits(c, 0)]
    xs = [W.make_x(c, 0, j, device="cuda") for j in range(c.L)]
    ws = [W.make_weights(c, j, device="cuda") for j in range(c.L)]
    if physical:
        ws = [MoELayerStep.replica_buffers(w) for w in ws]
    outs = [torch.empty((c.T, c.H), dtype=torch.bfloat16, device="cuda") for _ in range(c.L)]
    return lgs, xs, ws, outs


CASES = [
    # (workload, overrides, MoELayerStep options, predict)
    ("moe_gpt_stream", {"T": 2048, "L": 3}, {}, True),
    ("moe_gpt_stream", {"T": 2048, "L": 3}, {}, False),
    ("moe_gpt_stream", {"T": 2048, "L": 3}, {"fused": False}, True),
    ("moe_gpt_stream", {"T": 2048, "L": 3}, {"fused": False}, False),
    ("moe_gpt_stream", {"T": 2048, "L": 2}, {"gather": True}, True),
    ("moe_gpt_stream", {"T": 2048, "L": 2}, {"fuse_combine": True}, True),
    ("moe_gpt_stream", {"T": 2048, "L": 2}, {"fuse_combine": True, "fused": False}, True),
    ("moe_gpt_stream", {"T": 2048, "L": 2}, {"physical_replicas": True}, True),
    ("moe_gpt_stream", {"T": 2048, "L": 2, "F": 8192}, {}, True),   # 32 MB experts: two-launch FFN
    ("tiny", {"act": "swiglu"}, {}, True),
    ("tiny", {"act": "swiglu"}, {"fused": False, "small_group_threshold": 0}, True),
]


@pytest.mark.parametrize("name,over,opts,predict", CASES)
def test_layer_step_launch_count(name, over, opts, predict):
    c = dataclasses.replace(W.config_by_name(name), **over)
    st = M.MoEStats(c.L, c.E, c.window)
    step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, st, **opts)
    lgs, xs, ws, outs = _layer_inputs(c, physical=opts.get("physical_replicas", False))

    def body():
        for j in range(c.L):
            step.run(0, j, lgs[j], xs[j], ws[j], outs[j], predict=predict)

    body()  # first pass: one-time set-up outside the profiled region
    torch.cuda.synchronize()
    M.moe_check()
    got, names = _count_kernels(body)
    M.moe_check()
    want = sum(step.launches(j, c.L, predict=predict) for j in range(c.L))
    assert got == want, (want, names)


def test_chunked_step_launch_count():
    c = dataclasses.replace(W.config_by_name("moe_gpt_stream"), T=2048, L=2)
    st = M.MoEStats(c.L, c.E, c.window)
    step = ChunkedLayerStep(c.T, c.E, c.k, c.H, c.F, c.act, st, chunks=2)
    lgs, xs, ws, outs = _layer_inputs(c)

    def body():
        for j in range(c.L):
            step.run(0, j, lgs[j], xs[j], ws[j], outs[j])
        torch.cuda.synchronize()

    body()
    M.moe_check()
    got, names = _count_kernels(body)
    M.moe_check()
    want = sum(step.launches(j, c.L) for j in range(c.L))
    assert got == want, (want, names)


@pytest.mark.parametrize("T", [2048, 16384, 200000])
def test_front_launch_count_one_launch_option(T):
    """With MOE_OPT_FRONT_ONE_LAUNCH on, the front is one kernel where all its
    blocks fit on the device (two past that); the count the layer step reports
    follows the library's own answer, checked against the profiler."""
    c = dataclasses.replace(W.config_by_name("moe_gpt_stream"), T=T, L=2, H=64, F=128)
    M.moe_set_option(M.MOE_OPT_FRONT_ONE_LAUNCH, 1)
    try:
        st = M.MoEStats(c.L, c.E, c.window)
        step = MoELayerStep(c.T, c.E, c.k, c.H, c.F, c.act, st)
        lgs, xs, ws, outs = _layer_inputs(c)

        def body():
            for j in range(c.L):
                step.run(0, j, lgs[j], xs[j], ws[j], outs[j])

        body()
        torch.cuda.synchronize()
        M.moe_check()
        got, names = _count_kernels(body)
        M.moe_check()
        want = sum(step.launches(j, c.L) for j in range(c.L))
        assert got == want, (want, names)
        assert M.moe_layer_front_launches(T, c.E, c.k) == (1 if T <= 16384 else 2)
    finally:
        M.moe_set_option(M.MOE_OPT_FRONT_ONE_LAUNCH, 0)
