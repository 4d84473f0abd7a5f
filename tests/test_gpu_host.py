"""affqmm_run_host: x uploaded from host memory, the projection, y read back
-- one C call -- must give affqmm_run's bits (decode rows, prompt rows, a
ragged shape and the K = 0 case), and the oracle's values within tolerance."""
import pytest
import torch

from group_affine_bit_gb300 import api, build, synth
from helpers import assert_within_tolerance, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return api.lib()


# (bits, group, M, N, K, seed): one decode row, a few decode rows on a ragged
# shape, and prompt rows
CASES = [(4, 64, 1, 1024, 3840, 31), (5, 32, 3, 300, 640, 32), (4, 64, 40, 512, 1024, 33)]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("bits,group,M,N,K,seed", CASES)
def test_run_host_equals_run(orc, bits, group, M, N, K, seed, pinned):
    """Page-locked host buffers take the transfer kernels, pageable ones the
    driver's copies: the same bits either way."""
    x, codes, s, b = synth.problem(bits, group, M, N, K, seed)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    y_dev_ref = api.run(w, x.cuda(), workspace=api.Workspace())
    x_host = x.contiguous().pin_memory() if pinned else x.contiguous().clone()
    y_host = torch.empty(M, N, dtype=torch.bfloat16)
    if pinned:
        y_host = y_host.pin_memory()
    x_dev = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    y_dev = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    api.run_host(w, x_host, y_host, x_dev, y_dev, workspace=api.Workspace())
    torch.cuda.synchronize()
    what = f"run_host ({'page-locked' if pinned else 'pageable'}) {bits}b g{group} M={M} N={N} K={K}"
    assert torch.equal(y_host.view(torch.int16), y_dev_ref.cpu().view(torch.int16)), f"{what}: differs from affqmm_run"
    y_ref = orc.qmm(bits, group, u16(x), codes.numpy(), u16(s), u16(b))
    assert_within_tolerance(y_host, y_ref, what)


def test_run_host_empty_depth_writes_zeros():
    w = api.pack(torch.zeros(64, 0, dtype=torch.uint8, device="cuda"), torch.zeros(64, 0, dtype=torch.bfloat16, device="cuda"),
                 torch.zeros(64, 0, dtype=torch.bfloat16, device="cuda"), 4, 64)
    x_host = torch.empty(2, 0, dtype=torch.bfloat16).pin_memory()
    y_host = torch.full((2, 64), 7.0, dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty(2, 0, dtype=torch.bfloat16, device="cuda")
    y_dev = torch.full((2, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    api.run_host(w, x_host, y_host, x_dev, y_dev)
    torch.cuda.synchronize()
    assert not bool(y_host.float().abs().max())


def test_run_host_back_to_back_calls_reuse_the_staging_buffers(orc):
    """Consecutive calls on one stream with the same staging buffers and
    different host inputs: each call's upload waits for the previous call's
    projection, so every output is that call's own."""
    bits, group, M, N, K = 4, 64, 2, 640, 1024
    xs, ys, ws = [], [], []
    for i in range(3):
        x, codes, s, b = synth.problem(bits, group, M, N, K, 50 + i)
        xs.append(x)
        ws.append((api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group), codes, s, b))
    x_dev = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    y_dev = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    hosts = [x.contiguous().pin_memory() for x in xs]
    outs = [torch.empty(M, N, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    work = api.Workspace()
    for _ in range(2):
        for i in range(3):
            api.run_host(ws[i][0], hosts[i], outs[i], x_dev, y_dev, workspace=work)
    torch.cuda.synchronize()
    for i in range(3):
        w, codes, s, b = ws[i]
        ref = api.run(w, xs[i].cuda(), workspace=api.Workspace()).cpu()
        assert torch.equal(outs[i].view(torch.int16), ref.view(torch.int16)), f"call {i} differs"
