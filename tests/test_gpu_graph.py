"""The stateless fills inside a captured CUDA graph.

Every fill below is a pure function of (seed, counter) with no device state
of the library, so a stream capture records its kernels like any other
launch and each replay writes the same values: the oracle's.  (The f64
ziggurat keeps per-device miss lists and is not part of this capture.)"""
import numpy as np
import pytest

from dropout_lowbias32_hash32_gb300 import workloads

pytestmark = pytest.mark.gpu
U32 = 1 << 32


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def test_fills_replay_from_a_cuda_graph(torch, orc):
    import dropout_lowbias32_hash32_gb300 as rng
    n, first = 3 * 65536 + 7, U32 - 1000  # several blocks, a ragged tail, counters that wrap
    dev = torch.device("cuda")
    x_host = workloads.dropout_x(n)
    x = torch.from_numpy(x_host).to(dev)
    outs = {
        "u32": torch.empty(n, dtype=torch.int32, device=dev),
        "f64": torch.empty(n, dtype=torch.float64, device=dev),
        "u64_below": torch.empty(n, dtype=torch.int64, device=dev),
        "normal_f32": torch.empty(n, dtype=torch.float32, device=dev),
        "exponential_f32": torch.empty(n, dtype=torch.float32, device=dev),
        "dropout": torch.empty(n, dtype=torch.float32, device=dev),
    }

    def step():
        rng.rng_fill_u32(5, first, outs["u32"])
        rng.rng_fill_f64(5, first, outs["f64"])
        rng.rng_fill_u64_below(6, first, 1000, outs["u64_below"])
        rng.rng_fill_normal_f32(7, first, outs["normal_f32"])
        rng.rng_fill_exponential_f32(8, first, outs["exponential_f32"])
        rng.rng_dropout_fwd(x, outs["dropout"], 0.25, 9, first)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture, as torch recommends
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    launches = rng.rng_debug_launch_count()
    with torch.cuda.graph(graph):
        step()
    assert rng.rng_debug_launch_count() - launches == 6  # recorded, one kernel per fill
    for o in outs.values():
        o.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()

    def host(t):
        return t.cpu().numpy()

    assert np.array_equal(host(outs["u32"]).view(np.uint32), orc.fill_u32(5, first, n))
    assert np.array_equal(host(outs["f64"]).view(np.uint64), orc.fill_f64(5, first, n).view(np.uint64))
    assert np.array_equal(host(outs["u64_below"]).view(np.uint64), orc.fill_u64_below(6, first, 1000, n))
    z = host(outs["normal_f32"]).astype(np.float64)
    ref = orc.fill_randn(7, first, n)
    assert np.max(np.abs(z - ref) / (1 + np.abs(ref))) <= 4e-6
    assert np.array_equal(host(outs["exponential_f32"]).view(np.uint32),
                          orc.fill_exponential_f32_own(8, first, n).view(np.uint32))
    assert np.array_equal(host(outs["dropout"]).view(np.uint32), orc.dropout(x_host, 0.25, 9, first).view(np.uint32))

    # a replay after the input changed reads the new input (the mask is regenerated, not stored)
    x2_host = workloads.dropout_dy(n)
    x.copy_(torch.from_numpy(x2_host))
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host(outs["dropout"]).view(np.uint32), orc.dropout(x2_host, 0.25, 9, first).view(np.uint32))
