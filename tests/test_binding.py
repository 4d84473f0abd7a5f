"""The Python binding without a GPU: it computes nothing itself, so it must
refuse host tensors where the C ABI wants device memory, and fail loudly
(ImportError) when libaffqmm.so is missing -- there is no CPU fallback."""
import pytest
import torch

from group_affine_bit_gb300 import api, build


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return api.lib()


def _w(N=64, K=128):
    return api.PackedWeight(4, 64, N, K, torch.zeros(16, dtype=torch.uint8))


def test_device_entry_points_refuse_host_activations():
    x = torch.zeros(1, 128, dtype=torch.bfloat16)
    for fn in (api.run, api.run_exact):
        with pytest.raises(ValueError):
            fn(_w(), x)
    with pytest.raises(ValueError):
        api.run_stacked([_w(), _w()], x)
    with pytest.raises(ValueError):
        api.embed_rows(_w(), torch.zeros(4, dtype=torch.int32))


def test_activations_must_match_the_weight():
    with pytest.raises(ValueError):
        api.run(_w(K=128), torch.zeros(1, 256, dtype=torch.bfloat16))   # wrong K (refused before any device use)
    with pytest.raises(ValueError):
        api.run(_w(), torch.zeros(1, 128, dtype=torch.float32))


def test_host_call_refuses_device_staging_on_the_host():
    x = torch.zeros(1, 128, dtype=torch.bfloat16)
    y = torch.zeros(1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.run_host(_w(), x, y, x, y)          # staging buffers must be CUDA tensors
    with pytest.raises(ValueError):
        api.run_host(_w(), x, torch.zeros(1, 32, dtype=torch.bfloat16), x, y)   # y of the wrong width


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(api, "LIB_PATH", str(tmp_path / "libaffqmm.so"))
    monkeypatch.setattr(api, "_lib", None)
    with pytest.raises(ImportError):
        api.lib()
    with pytest.raises(ImportError):
        api.strerror(0)
