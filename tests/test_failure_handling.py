"""Failure handling on the GPU without a GPU fault: a bounded device wait that runs out.

Every mbarrier wait in the library's kernels is bounded. When one runs out, the kernel records
BITNET_ETIMEOUT in its device error word, stops, waits (bounded) for its own bulk copies in
flight, and returns; bitnet_last_device_error reports and clears the word. The self-test kernel
takes that path on purpose: it waits on a barrier nothing arrives on, with a small poll limit,
while a real bulk copy is in flight. No trap, fault or endless loop is involved.
"""
import numpy as np
import pytest
import torch

import oracle
from ternary_weight_gb300 import _build, binding, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    _build.build()
    binding.lib()
    assert binding.last_device_error() == 0  # start clean


@pytest.mark.parametrize("nbytes,polls", [(16, 1), (4096, 64), (16384, 1000)])
def test_bounded_wait_runs_out_and_is_reported(nbytes, polls):
    words = np.random.default_rng(nbytes).integers(0, 2 ** 32, nbytes // 4, dtype=np.uint64).astype(np.uint32)
    src = torch.from_numpy(words.view(np.int32)).cuda()
    report = binding.selftest_wait_timeout(src, polls)
    torch.cuda.synchronize()
    gave_up, landed, wsum = (int(v) & 0xFFFFFFFF for v in report.cpu().numpy())
    assert gave_up == 1, "the wait on a barrier nothing arrives on did not give up"
    assert landed == 1, "the copy in flight was not waited for before the kernel returned"
    assert wsum == int(words.astype(np.uint64).sum()) & 0xFFFFFFFF, "the copied bytes differ from the source"
    assert binding.last_device_error() == binding.BITNET_ETIMEOUT
    # the word was read and cleared: a second read is clean
    assert binding.last_device_error() == 0


def test_next_call_after_a_timeout_is_clean_and_exact():
    src = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    binding.selftest_wait_timeout(src, 8)
    assert binding.last_device_error() == binding.BITNET_ETIMEOUT
    M, N, K = 3, 1000, 2560
    wp_np = workloads.random_packed_bytes(N, K, 31)
    xq_np = workloads.random_int8(M, K, 32)
    s_np = np.array([0.5, 3.0, 70.0], np.float32)
    rs_np = xq_np.astype(np.int64).sum(axis=1).astype(np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    out = binding.i2s_matmul(dev(xq_np), dev(s_np), dev(rs_np), dev(wp_np), 0.02, acc_out=acc)
    torch.cuda.synchronize()
    o_out, o_acc = oracle.ternary_matmul(xq_np, s_np, wp_np, 0.02)
    assert np.array_equal(acc.cpu().numpy(), o_acc)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), o_out.view(np.uint32))
    assert binding.last_device_error() == 0


def test_selftest_rejects_bad_arguments_on_host():
    src = torch.zeros(64, dtype=torch.uint8, device="cuda")
    lib = binding.lib()
    rep = torch.zeros(3, dtype=torch.int32, device="cuda")
    for nbytes, polls, status in ((0, 1, -1), (20, 1, -1), (16400, 1, -1), (64, 0, -1), (64, (1 << 20) + 1, -1)):
        assert lib.bitnet_selftest_wait_timeout(src.data_ptr(), nbytes, polls, rep.data_ptr(), None) == status
    assert lib.bitnet_selftest_wait_timeout(src.data_ptr() + 8, 16, 1, rep.data_ptr(), None) == -2
    assert binding.last_device_error() == 0
