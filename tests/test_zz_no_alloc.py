"""nvfp4_quantize_noalloc, the entry point for callers that cannot allocate
device memory (an engine that owns all of HBM through its own arena, or a
thread that may not risk cudaMalloc/cudaFree blocking the device): it keeps
its scratch in a static array inside the library instead of a workspace.

Called through the C ABI (ctypes) and compared with nvfp4_quantize, which
takes a workspace, and with the oracle, on calls in a row through each of
the quantize's kernel paths: no call may see what the one before it left in
the shared scratch.  Quantize results are bit-exact, the tolerance every
quantize test here uses.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantize_block_scaled_gb300 import build as b
    b.build()
    import quantize_block_scaled_gb300 as nv
    nv.lib()
    return nv


def noalloc_quantize(nv, xd):
    rows, cols = xd.shape
    q = torch.empty(rows, cols // 2, dtype=torch.uint8, device="cuda")
    sf = torch.empty(rows, cols // 16, dtype=torch.uint8, device="cuda")
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    rc = nv.lib().nvfp4_quantize_noalloc(
        P(xd.data_ptr()), rows, cols, xd.stride(0), P(q.data_ptr()), P(sf.data_ptr()),
        P(gs.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, nv.lib().nvfp4_status_string(rc)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy(), gs.cpu().numpy()


def _scaled(x_bits, factor):
    """bf16 bits of the values of x_bits times factor (scaled as floats)."""
    return workloads.bf16_bits(workloads.bf16_to_f32(x_bits) * np.float32(factor))


# One input per kernel path nvfp4_quantize takes (one cluster up to 512 KB,
# one cooperative grid up to the SMs' shared memory, two kernels beyond),
# each followed by one with smaller values, so that a maximum left behind in
# the shared scratch by the call before would change the global scale.
CASES = [
    ("cluster", lambda: workloads.quantize_input(12, seed=43)),
    ("cluster, smaller", lambda: _scaled(workloads.quantize_input(12, seed=44), 0.25)),
    ("cooperative", lambda: workloads.quantize_input(256, seed=41)),
    ("cooperative, smaller", lambda: _scaled(workloads.quantize_input(37, seed=42), 0.25)),
    ("two kernels", lambda: workloads.quantize_input(2200, seed=45)),
    ("two kernels, smaller", lambda: _scaled(workloads.quantize_input(2200, seed=46), 0.25)),
]


def test_noalloc_matches_workspace_path_and_oracle(nv):
    ws = nv.workspace()
    for what, make in CASES:
        x = make()
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        got = noalloc_quantize(nv, xd)
        rq, rsf, rgs = nv.quantize(xd, ws)
        torch.cuda.synchronize()
        assert got[2].view(np.uint32)[0] == rgs.cpu().numpy().view(np.uint32)[0], what
        assert np.array_equal(got[1], rsf.cpu().numpy()), what
        assert np.array_equal(got[0], rq.cpu().numpy()), what
        oq, osf, ogs = oracle.quantize(x)
        assert got[2].view(np.uint32)[0] == np.float32(ogs).view(np.uint32), what
        assert np.array_equal(got[1], osf) and np.array_equal(got[0], oq), what


def test_noalloc_rejects_bad_arguments(nv):
    P = ctypes.c_void_p
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    # cols not a multiple of 16: refused before any launch
    rc = nv.lib().nvfp4_quantize_noalloc(P(gs.data_ptr()), 1, 24, 24, P(gs.data_ptr()),
                                         P(gs.data_ptr()), P(gs.data_ptr()), None)
    assert rc == 2
