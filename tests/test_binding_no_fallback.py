"""The Python binding has no CPU path: host tensors are refused before any call, and
a missing library is an error, not a fallback (host only)."""
import pytest
import torch

from bit_asymmetric_kv_gb300 import kivi


def test_host_tensors_are_refused():
    k = torch.zeros(1, 1, 32, 128, dtype=torch.float16)
    with pytest.raises(TypeError, match="CUDA float16"):
        kivi.kivi_quantize_prefill(None, k, k)
    with pytest.raises(TypeError, match="CUDA float16"):
        kivi.kivi_append_token(None, k[:, :, 0], k[:, :, 0])
    with pytest.raises(TypeError, match="CUDA float16"):
        kivi.kivi_decode_attention(None, k[:, :, 0], 1.0)


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(kivi, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(kivi, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        kivi.lib()
