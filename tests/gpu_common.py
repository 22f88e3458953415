"""Fixtures shared by the GPU tests (imported by test modules)."""
import pytest

torch = pytest.importorskip("torch")


def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def status_ok():
    import io_aware_exact_15_gb300 as fa
    torch.cuda.synchronize()
    st = fa.fa_get_device_status()
    assert st == fa.FA_OK, f"device status {fa.fa_status_string(st)}"
