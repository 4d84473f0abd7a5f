"""The bounded-wait failure path on the GPU, made to happen on purpose.

Every mbarrier wait in the kernels gives up after a cycle limit; a wait that
gives up sets the workspace status word and an abort flag, every role of the
CTA leaves its loop, the copies already started are waited for, and the CTA
exits.  The test hook affqmm_test_fault_wait makes the decode kernel's
consumer warps first wait, for a short limit, on a barrier that nothing
completes: the wait runs out on every CTA.  Nothing faults or hangs; the host
then reads AFFQMM_E_TIMEOUT from the workspace, and the same context and
workspace serve the next normal call, which must match the oracle.
"""
import pytest
import torch

from group_affine_bit_gb300 import api, build, synth
from helpers import assert_within_tolerance, u16

pytestmark = pytest.mark.gpu

LIMIT_CYCLES = 1 << 20   # about half a millisecond of SM clock


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return api.lib()


@pytest.mark.parametrize("M,N,K", [(2, 512, 1024), (16, 200, 21504)])
def test_wait_runs_out_then_next_call_is_correct(orc, M, N, K):
    bits, group = 4, 64
    x, codes, s, b = synth.problem(bits, group, M, N, K, seed=900 + M)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    xd = x.cuda()
    ws = api.Workspace()
    api.test_fault_wait(LIMIT_CYCLES)
    try:
        api.run(w, xd, workspace=ws)
        torch.cuda.synchronize()
    finally:
        api.test_fault_wait(0)
    assert api.STATUS_NAMES[api.workspace_status(ws.buf)] == "AFFQMM_E_TIMEOUT"
    torch.cuda.synchronize()
    assert int(ws.buf[:api.WORKSPACE_ZEROED].count_nonzero()) == 0, "status word and counters not cleared"
    # the context and the workspace are usable again
    y = api.run(w, xd, workspace=ws)
    torch.cuda.synchronize()
    assert api.workspace_status(ws.buf) == 0
    y_ref = orc.qmm(bits, group, u16(x), codes.numpy(), u16(s), u16(b), nthreads=8)
    assert_within_tolerance(y, y_ref, f"after a timeout M={M} N={N} K={K}")


def test_fault_wait_refuses_negative():
    with pytest.raises(api.AffqmmError) as ei:
        api.test_fault_wait(-1)
    assert ei.value.name == "AFFQMM_E_ARG"
