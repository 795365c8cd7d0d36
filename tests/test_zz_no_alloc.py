"""The allocation-free prefill matmul (bitnet_i2s_matmul_noalloc), through the C ABI.

It is meant for callers that may not allocate device memory, such as a plugin whose host
framework owns all device memory, or a loop where cudaMalloc would synchronise the device.
It must give the same result as bitnet_i2s_matmul_ws with a caller-provided workspace, and
the oracle's, on consecutive calls that reuse the library's shared scratch array; problems
whose workspace is exactly the 64 MiB of the scratch must run, and one 256-byte step more
must be refused. This file is collected last so that a stop-at-first-failure run has run
every other test before it.
"""
import numpy as np
import pytest
import torch

import oracle
from ternary_weight_gb300 import _build, binding, workloads

pytestmark = pytest.mark.gpu

REL_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    _build.build()
    binding.lib()


def _inputs(M, N, K, seed):
    x = torch.from_numpy(workloads.activations(M, K, seed, "bf16").view(np.int16)).cuda().view(torch.bfloat16)
    wp = binding.pack_i2s(torch.from_numpy(workloads.ternary_weights(N, K, seed + 1)).cuda())
    xq, s, rs = binding.quant_act(x)
    return xq, s, rs, wp, workloads.weight_scale(N, K, seed + 2)


def _close(a, b):
    a64, b64 = a.double(), b.double()
    return bool(torch.all((a64 - b64).abs() <= REL_TOL * b64.abs()))


def _oracle_check(xq, s, wp, ws, acc, out):
    o_out, o_acc = oracle.ternary_matmul(xq.cpu().numpy(), s.cpu().numpy(), wp.cpu().numpy(), ws,
                                         nthreads=oracle.default_threads())
    assert np.array_equal(acc.cpu().numpy(), o_acc)
    assert _close(out, torch.from_numpy(o_out).cuda())


def test_noalloc_matches_workspace_path_on_two_calls_in_a_row():
    for (M, N, K, seed) in ((200, 1000, 2560, 950), (512, 2560, 6912, 960)):
        xq, s, rs, wp, ws = _inputs(M, N, K, seed)
        acc_ref = torch.empty((M, N), dtype=torch.int32, device="cuda")
        ref = binding.i2s_matmul_ws(xq, s, rs, wp, ws, acc_out=acc_ref)
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        got = binding.i2s_matmul_noalloc(xq, s, rs, wp, ws, acc_out=acc)
        torch.cuda.synchronize()
        assert torch.equal(acc, acc_ref)
        assert _close(got, ref)
        _oracle_check(xq, s, wp, ws, acc, got)
    assert binding.last_device_error() == 0


def test_noalloc_at_exactly_the_scratch_size_and_one_step_beyond():
    """K = 128: the workspace is 256 (M + N) bytes, so M + N = 2^18 fills the 64 MiB exactly and
    must run (and match the oracle); one more weight row needs 256 bytes more and is refused."""
    M, K = 128, 128
    N = (1 << 18) - M
    assert binding.workspace_size(M, N, K) == 64 << 20
    assert binding.workspace_size(M, N + 1, K) == (64 << 20) + 256
    xq, s, rs, wp, ws = _inputs(M, N + 1, K, 970)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    got = binding.i2s_matmul_noalloc(xq, s, rs, wp[:N], ws, acc_out=acc)
    torch.cuda.synchronize()
    _oracle_check(xq, s, wp[:N], ws, acc, got)
    with pytest.raises(binding.BitnetError) as e:
        binding.i2s_matmul_noalloc(xq, s, rs, wp, ws)
    assert e.value.status == binding.BITNET_EINVAL
    assert binding.last_device_error() == 0


def test_noalloc_refuses_problems_beyond_its_scratch():
    M, N, K = 4096, 2560, 6912  # needs about 92 MB of workspace, more than the 64 MiB scratch
    xq = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    s = torch.ones(M, device="cuda")
    rs = torch.zeros(M, dtype=torch.int32, device="cuda")
    wp = torch.zeros((N, K // 4), dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.BitnetError) as e:
        binding.i2s_matmul_noalloc(xq, s, rs, wp, 1.0)
    assert e.value.status == binding.BITNET_EINVAL
