"""Parity of the tcgen05 prompt path (M >= 17, chunks of 128 rows) with the
CPU oracle, through the C ABI."""
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


def run_case(orc, bits, group, M, N, K, seed, nthreads=16):
    x, codes, s, b = synth.problem(bits, group, M, N, K, seed)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    ws = api.Workspace()
    y = api.run(w, x.cuda(), workspace=ws)
    torch.cuda.synchronize()
    assert api.workspace_status(ws.buf) == 0
    y_ref = orc.qmm(bits, group, u16(x), codes.numpy(), u16(s), u16(b), nthreads=nthreads)
    assert_within_tolerance(y, y_ref, f"M={M} N={N} K={K} {bits}b g{group}")
    assert int(ws.buf[:api.WORKSPACE_ZEROED].count_nonzero()) == 0, "counters not left zeroed"
    return w, x, y


@pytest.mark.parametrize("M", [17, 31, 64, 100, 127, 128])
@pytest.mark.parametrize("N,K", [(256, 128), (300, 384), (1000, 640), (4096, 2048)])
def test_prompt_shapes(orc, M, N, K):
    run_case(orc, 4, 64, M, N, K, seed=M + N + K)


@pytest.mark.parametrize("M", [129, 200, 256, 300])
def test_prompt_more_than_one_chunk(orc, M):
    run_case(orc, 4, 64, M, 640, 1024, seed=M)


@pytest.mark.parametrize("bits,group", [(b, g) for b in (2, 3, 4, 5, 6, 8) for g in (32, 64, 128)])
def test_prompt_all_widths(orc, bits, group):
    K = 512 + (group if group < 128 else 0)
    run_case(orc, bits, group, 128, 520, K, seed=bits * 10 + group)


def test_prompt_one_hot_rows_reproduce_weight_columns():
    bits, group, N, K, M = 4, 64, 700, 1024, 128
    _, codes, s, b = synth.problem(bits, group, 1, N, K, seed=78)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
    W = api.dequant(w).float()
    g = torch.Generator().manual_seed(5)
    ks = torch.randint(0, K, (M,), generator=g)
    js = torch.randint(-3, 4, (M,), generator=g)
    x = torch.zeros(M, K)
    x[torch.arange(M), ks] = 2.0 ** js.float()
    y = api.run(w, x.to(torch.bfloat16).cuda())
    want = (W[:, ks.cuda()].T * (2.0 ** js.float().cuda())[:, None]).to(torch.bfloat16)
    assert torch.equal(y.view(torch.int16), want.view(torch.int16))


def test_prompt_deterministic_and_stacked_equals_separate(orc):
    bits, group, K, M = 4, 64, 2048, 128
    g = synth.generator(91)
    xc = synth.activations(M, K, g)
    x = xc.cuda()
    ws_list, singles, tables = [], [], []
    for N in (3000, 700, 5376):
        codes, s, b = synth.affine_table(bits, group, N, K, g)
        w = api.pack(codes.cuda(), s.cuda(), b.cuda(), bits, group)
        ws_list.append(w)
        tables.append((codes, s, b))
        singles.append(api.run(w, x))
    again = [api.run(w, x) for w in ws_list]
    for a, c in zip(singles, again):
        assert torch.equal(a.view(torch.int16), c.view(torch.int16))
    ys = api.run_stacked(ws_list, x)
    for i, (a, c, (codes, s, b)) in enumerate(zip(ys, singles, tables)):
        assert torch.equal(a.view(torch.int16), c.view(torch.int16))
        y_ref = orc.qmm(bits, group, u16(xc), codes.numpy(), u16(s), u16(b), nthreads=16)
        assert_within_tolerance(a, y_ref, f"stacked prompt projection {i}")


@pytest.mark.parametrize("name", ["qkv", "o", "gate_up", "down"])
def test_prompt_chunk_layer_shapes_full(orc, name):
    """The prompt-chunk workload's projection shapes at full size (M = 128),
    every output against the oracle (the tolerance's rms over whole rows)."""
    N, K = synth.DECODER_LAYER_SHAPES[name]
    c = synth.PROMPT_CHUNK
    seed = synth.step_seed(c["seed"], 0, list(synth.DECODER_LAYER_SHAPES).index(name))
    x, codes, s, b = synth.problem(c["bits"], c["group"], c["M"], N, K, seed)
    w = api.pack(codes.cuda(), s.cuda(), b.cuda(), c["bits"], c["group"])
    y = api.run(w, x.cuda())
    torch.cuda.synchronize()
    threads = max(1, min(16, len(__import__("os").sched_getaffinity(0))))
    y_ref = orc.qmm(c["bits"], c["group"], u16(x), codes.numpy(), u16(s), u16(b), nthreads=threads)
    assert_within_tolerance(y, y_ref, f"prompt chunk {name}")
